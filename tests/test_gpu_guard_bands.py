"""Guard bands around every output buffer of every entry point (race and bounds checks).

Each output (and each backward workspace) is placed inside a larger device buffer whose
margins and interior start as a NaN bit pattern.  After the call: the margins must be
untouched (no tail tile wrote past the end of a buffer or before its start, e.g. into a
neighbouring allocation), and the interior must hold the oracle's values (no element
left unwritten).  The sizes are ragged, so the last query and key tiles are partial
and the 16-bit rows at head sizes that are not 32, 64 or 128 end inside a kernel tile.

Reference for the stores guarded here: "vision-rs 0.1.1 flash_attn2.rs" (one output
row per program in the forward and both backward kernels) and
"vision_rs/models/yolo/kernels/attention/psa.rs" (the rearrangements and their
adjoints, psa_fa2_backward).
"""
import math

import numpy as np
import pytest

from attention_fa2_forward_02_gb300 import binding, synth
from oracle import attention as A
from oracle import psa as P
from tests import gpu_util as G
from tests.tolerance import check_16bit, check_f32, check_lse

pytestmark = pytest.mark.gpu

BH, N_Q, N_K = 2, 333, 250
CODES = {"bf16": binding.DTYPE_BF16, "f16": binding.DTYPE_F16}


def _forward(tag, d, dtype, bh=BH, n_q=N_Q, n_k=N_K):
    torch = G.require_gpu()
    q, k, v = G.inputs(tag, bh, n_q, n_k, d, dtype)
    qd, kd, vd = (G.to_device(x, dtype) for x in (q, k, v))
    o = G.guarded((bh, n_q, d), dtype)
    lse = G.Guarded((bh, n_q), torch.float32)
    scale = 1 / math.sqrt(d)
    binding.fa2_forward(qd, kd, vd, o.t, lse.t, scale)
    binding.fa2_device_status()
    return (q, k, v), (qd, kd, vd), o, lse, scale


@pytest.mark.parametrize("d,dtype", [(40, "bf16"), (64, "f16"), (64, "bf16"), (128, "bf16"), (40, "f32"), (7, "f32")])
def test_forward_outputs_fenced(d, dtype):
    (q, k, v), _, o, lse, scale = _forward(f"guard/fwd/{d}/{dtype}", d, dtype)
    o.assert_intact("O")
    lse.assert_intact("LSE")
    w = lambda x: synth.widen(x, dtype) if dtype != "f32" else x.astype(np.float64)  # noqa: E731
    o_ref, l_ref = A.forward(w(q), w(k), w(v), scale)
    if dtype == "f32":
        check_f32(G.to_f64(o.t), o_ref, "O")
        check_f32(G.to_f64(lse.t), l_ref, "LSE")
    else:
        check_16bit(G.to_f64(o.t), o_ref, "O")
        check_lse(G.to_f64(lse.t), l_ref)


def _backward_inputs(tag, d, dtype, bh=BH):
    (q, k, v), (qd, kd, vd), o, lse, scale = _forward(tag, d, dtype, bh)
    d_o = synth.tensor(tag + "/do", (bh, N_Q, d), dtype)
    dod = G.to_device(d_o, dtype)
    w = lambda x: synth.widen(x, dtype)  # noqa: E731
    ref = A.backward(w(q), w(k), w(v), w(d_o), scale)
    return (qd, kd, vd, o.t, dod, lse.t), ref, scale


def _grads(d, dtype, bh=BH):
    return G.guarded((bh, N_Q, d), dtype), G.guarded((bh, N_K, d), dtype), G.guarded((bh, N_K, d), dtype)


def _check_grads(grads, ref, what):
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        g.assert_intact(f"{what} {name}")
        check_16bit(G.to_f64(g.t), r, f"{what} {name}")


@pytest.mark.parametrize("d,dtype,bh", [(40, "bf16", 80), (64, "bf16", 80), (64, "f16", BH), (128, "bf16", BH),
                                         (128, "f16", BH)])
def test_backward_outputs_and_workspace_fenced(d, dtype, bh):
    """fa2_backward: the one-pass kernel with its float32 dQ accumulator (head size <= 64 with
    80 heads, more than 74 key tiles in all) and the two passes in one grid (head size > 64,
    or too few key tiles); the workspace is fenced at exactly fa2_backward_workspace_size
    bytes."""
    torch = G.require_gpu()
    (qd, kd, vd, o, dod, lse), ref, scale = _backward_inputs(f"guard/bwd/{d}/{dtype}/{bh}", d, dtype, bh)
    grads = _grads(d, dtype, bh)
    ws = G.Guarded((binding.fa2_backward_workspace_size(bh, N_Q, N_K, d, CODES[dtype]),), torch.uint8)
    binding.fa2_backward(qd, kd, vd, o, dod, lse, *(g.t for g in grads), ws.t, scale)
    binding.fa2_device_status()
    ws.assert_intact("workspace")
    _check_grads(grads, ref, "fa2_backward")


@pytest.mark.parametrize("d,dtype", [(40, "bf16"), (64, "f16"), (128, "bf16")])
def test_backward_stages_fenced(d, dtype):
    """fa2_backward_preprocess, then _dkdv + _dq, and again _passes, from the smaller
    two-pass workspace (8 bytes per padded query row), fenced at exactly that size."""
    torch = G.require_gpu()
    (qd, kd, vd, o, dod, lse), ref, scale = _backward_inputs(f"guard/stages/{d}/{dtype}", d, dtype)
    n_q_pad = -(-N_Q // 128) * 128
    ws = G.Guarded((8 * BH * n_q_pad,), torch.uint8)
    binding.fa2_backward_preprocess(o, dod, lse, ws.t, N_K)
    staged = _grads(d, dtype)
    binding.fa2_backward_dkdv(qd, kd, vd, dod, ws.t, staged[1].t, staged[2].t, scale)
    binding.fa2_backward_dq(qd, kd, vd, dod, ws.t, staged[0].t, scale)
    one_grid = _grads(d, dtype)
    binding.fa2_backward_passes(qd, kd, vd, dod, ws.t, *(g.t for g in one_grid), scale)
    binding.fa2_device_status()
    ws.assert_intact("two-pass workspace")
    _check_grads(staged, ref, "stages")
    _check_grads(one_grid, ref, "fa2_backward_passes")


@pytest.mark.parametrize("kd,dtype", [(24, "f16"), (32, "f16"), (64, "bf16")])
def test_psa_attention_outputs_fenced(kd, dtype):
    """psa_fa2_forward's o_lo, o_hi and lse, then psa_fa2_backward's d_packed and workspace."""
    torch = G.require_gpu()
    bh, n = 3, 333
    tag = f"guard/psa/{kd}/{dtype}"
    packed = synth.tensor(tag + "/packed", (4, bh, n, kd), dtype)
    d_lo = synth.tensor(tag + "/dlo", (bh, n, kd), dtype)
    d_hi = synth.tensor(tag + "/dhi", (bh, n, kd), dtype)
    pd = G.to_device(packed, dtype)
    o_lo, o_hi = G.guarded((bh, n, kd), dtype), G.guarded((bh, n, kd), dtype)
    lse = G.Guarded((bh, n), torch.float32)
    scale = 1 / math.sqrt(kd)
    binding.psa_fa2_forward(pd, o_lo.t, o_hi.t, lse.t, scale)
    d_packed = G.guarded((4, bh, n, kd), dtype)
    ws = G.Guarded((8 * bh * (-(-n // 128) * 128),), torch.uint8)
    binding.psa_fa2_backward(pd, o_lo.t, o_hi.t, G.to_device(d_lo, dtype), G.to_device(d_hi, dtype), lse.t, d_packed.t,
                             ws.t, scale)
    binding.fa2_device_status()
    for name, g in (("O_lo", o_lo), ("O_hi", o_hi), ("LSE", lse), ("d_packed", d_packed), ("workspace", ws)):
        g.assert_intact(name)
    w = synth.widen(packed, dtype)
    r_lo, r_lse = A.forward(w[0], w[1], w[2], scale)
    r_hi, _ = A.forward(w[0], w[1], w[3], scale)
    check_16bit(G.to_f64(o_lo.t), r_lo, "O_lo")
    check_16bit(G.to_f64(o_hi.t), r_hi, "O_hi")
    check_lse(G.to_f64(lse.t), r_lse)
    want = A.psa_backward(w, synth.widen(d_lo, dtype), synth.widen(d_hi, dtype), scale)
    got = G.to_f64(d_packed.t)
    for s, name in enumerate(("dQ_lo+dQ_hi", "dK_lo+dK_hi", "dV_lo", "dV_hi")):
        check_16bit(got[s], want[s], name)


def _words(t):
    import torch
    if t.element_size() == 4:
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _raw(words, dtype):
    import torch
    if dtype == "f32":
        return torch.from_numpy(words.view(np.int32).copy()).view(torch.float32).cuda()
    return torch.from_numpy(words.view(np.int16).copy()).view(torch.bfloat16 if dtype == "bf16" else torch.float16).cuda()


def _patterns(tag, shape, dtype):
    w16 = synth.counter_u16(tag, shape)
    if dtype == "f32":
        return (synth.counter_u16(tag + "/hi", shape).astype(np.uint32) << np.uint32(16)) | w16.astype(np.uint32)
    return w16


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("B,nh,kd,H,W", [(8, 4, 32, 20, 20), (421, 5, 24, 8, 13), (3, 1, 8, 3, 5)])
def test_psa_rearrangements_fenced(dtype, B, nh, kd, H, W):
    """psa_pack_qkv, psa_merge_attn_nchw, psa_extract_v_nchw and the three adjoints (the
    shared-memory tile at the smaller shapes, the register transpose at B=421 for 16-bit
    data): margins untouched, contents bit-exact against the oracle's index maps."""
    G.require_gpu()
    tag = f"guard/rearr/{dtype}/{B}/{nh}/{kd}/{H}/{W}"
    bh, n, c = B * nh, H * W, nh * 2 * kd
    qkv = _patterns(tag + "/qkv", (B, nh * 4 * kd, H, W), dtype)
    qkv_d = _raw(qkv, dtype).view(qkv.shape)
    packed = G.guarded((4, bh, n, kd), dtype)
    binding.psa_pack_qkv(qkv_d, packed.t, nh)
    lo, hi = _patterns(tag + "/lo", (bh, n, kd), dtype), _patterns(tag + "/hi", (bh, n, kd), dtype)
    merged = G.guarded((B, c, H, W), dtype)
    binding.psa_merge_attn_nchw(_raw(lo, dtype).view(lo.shape), _raw(hi, dtype).view(hi.shape), merged.t, nh)
    v = G.guarded((B, c, H, W), dtype)
    binding.psa_extract_v_nchw(qkv_d, v.t, nh)
    d_packed = _patterns(tag + "/dpacked", (4, bh, n, kd), dtype)
    d_qkv = G.guarded(qkv.shape, dtype)
    binding.psa_pack_qkv_backward(_raw(d_packed, dtype).view(d_packed.shape), d_qkv.t, nh)
    d_merged = _patterns(tag + "/dmerged", (B, c, H, W), dtype)
    d_lo = G.guarded((bh, n, kd), dtype)
    d_hi = G.guarded((bh, n, kd), dtype)
    binding.psa_merge_attn_backward(_raw(d_merged, dtype).view(d_merged.shape), d_lo.t, d_hi.t, nh)
    binding.fa2_device_status()
    for name, g in (("packed", packed), ("merged", merged), ("v", v), ("d_qkv", d_qkv), ("d_lo", d_lo),
                    ("d_hi", d_hi)):
        g.assert_intact(name)
    assert np.array_equal(_words(packed.t).reshape(4, bh, n, kd), P.pack_qkv(qkv, nh))
    assert np.array_equal(_words(merged.t).reshape(B, c, H, W), P.merge_attn_nchw(lo, hi, B, nh, H, W))
    assert np.array_equal(_words(v.t).reshape(B, c, H, W), P.extract_v_nchw(qkv, nh))
    assert np.array_equal(_words(d_qkv.t).reshape(qkv.shape), P.pack_qkv_backward(d_packed, B, nh, H, W))
    want_lo, want_hi = P.merge_attn_backward(d_merged, nh)
    assert np.array_equal(_words(d_lo.t).reshape(want_lo.shape), want_lo)
    assert np.array_equal(_words(d_hi.t).reshape(want_hi.shape), want_hi)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("B,nh,kd,H,W", [(8, 4, 32, 20, 20), (421, 5, 24, 8, 13)])
def test_psa_extract_v_backward_fenced(dtype, B, nh, kd, H, W):
    """psa_extract_v_backward reads and writes d_qkv in place: its margins stay untouched and
    the result is the oracle's exact sum rounded once."""
    G.require_gpu()
    tag = f"guard/evb/{dtype}/{B}/{nh}/{kd}"
    d_packed = synth.tensor(tag + "/dpacked", (4, B * nh, H * W, kd), dtype)
    d_v = synth.tensor(tag + "/dv", (B, nh * 2 * kd, H, W), dtype)
    d_qkv = G.guarded((B, nh * 4 * kd, H, W), dtype)
    binding.psa_pack_qkv_backward(G.to_device(d_packed, dtype), d_qkv.t, nh)
    binding.psa_extract_v_backward(G.to_device(d_v, dtype), d_qkv.t, nh)
    binding.fa2_device_status()
    d_qkv.assert_intact("d_qkv")
    want = P.extract_v_backward(d_v, P.pack_qkv_backward(d_packed, B, nh, H, W), nh, dtype)
    assert np.array_equal(_words(d_qkv.t).reshape(want.shape), want.view(np.uint16))
