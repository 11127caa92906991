"""GPU parity of the PSA rearrangement passes (bit-exact) and of the C2PSA attention pipeline."""
import math

import numpy as np
import pytest

from attention_fa2_forward_02_gb300 import binding, synth
from oracle import attention as A
from oracle import psa as P
from tests import gpu_util as G
from tests.tolerance import check_16bit

pytestmark = pytest.mark.gpu


def _raw_tensor(words, dtype):
    """Raw words as a CUDA tensor whose bits are exactly `words`."""
    import torch
    if dtype == "f32":
        return torch.from_numpy(words.view(np.int32).copy()).view(torch.float32).cuda()
    t = torch.from_numpy(words.view(np.int16).copy())
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).cuda()


def _words(t, dtype):
    import torch
    if dtype == "f32":
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _patterns(tag, shape, dtype):
    w16 = synth.counter_u16(tag, shape)
    if dtype == "f32":
        hi = synth.counter_u16(tag + "/hi", shape).astype(np.uint32)
        return (hi << np.uint32(16)) | w16.astype(np.uint32)
    return w16


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("B,nh,kd,H,W", [(8, 4, 32, 20, 20), (2, 2, 16, 5, 7), (1, 3, 8, 1, 1), (3, 1, 64, 9, 16)])
def test_pack_merge_bit_exact(dtype, B, nh, kd, H, W):
    G.require_gpu()
    qkv = _patterns(f"psa/{dtype}/{B}/{nh}/{kd}/{H}/{W}", (B, nh * 4 * kd, H, W), dtype)
    qkv_d = _raw_tensor(qkv, dtype)
    packed = _raw_tensor(np.zeros(qkv.size, dtype=qkv.dtype), dtype)
    binding.psa_pack_qkv(qkv_d, packed, nh)
    got = _words(packed, dtype).reshape(4, B * nh, H * W, kd)
    assert np.array_equal(got, P.pack_qkv(qkv, nh))
    # merge the V_lo / V_hi sections back: the V channels of QKV, bit for bit
    out = _raw_tensor(np.zeros((B, nh * 2 * kd, H, W), dtype=qkv.dtype), dtype).view(B, nh * 2 * kd, H, W)
    sec = packed.view(4, B * nh, H * W, kd)
    binding.psa_merge_attn_nchw(sec[2], sec[3], out, nh)
    binding.fa2_device_status()
    merged = _words(out, dtype).reshape(B, nh * 2 * kd, H, W)
    assert np.array_equal(merged, P.merge_attn_nchw(got[2], got[3], B, nh, H, W))
    assert np.array_equal(merged, P.extract_v_nchw(qkv, nh))


def test_merge_independent_inputs():
    G.require_gpu()
    B, nh, kd, H, W = 2, 3, 32, 6, 10
    lo = synth.counter_u16("merge/lo", (B * nh, H * W, kd))
    hi = synth.counter_u16("merge/hi", (B * nh, H * W, kd))
    out = _raw_tensor(np.zeros((B, nh * 2 * kd, H, W), dtype=np.uint16), "f16").view(B, nh * 2 * kd, H, W)
    binding.psa_merge_attn_nchw(_raw_tensor(lo, "f16").view(B * nh, H * W, kd), _raw_tensor(hi, "f16").view(B * nh, H * W, kd), out, nh)
    binding.fa2_device_status()
    assert np.array_equal(_words(out, "f16").reshape(B, nh * 2 * kd, H, W), P.merge_attn_nchw(lo, hi, B, nh, H, W))


def test_c2psa_pipeline():
    """YOLO C2PSA block: QKV [8, 512, 20, 20] fp16, num_heads 4, KEY_DIM 32: pack, two
    attention calls (V_lo, V_hi) with HEAD_DIM 32 on N = 400 tokens, merge to [8, 256, 20, 20]."""
    torch = G.require_gpu()
    B, nh, kd, H, W = 8, 4, 32, 20, 20
    n, bh = H * W, B * nh
    qkv = synth.tensor("config/c2psa/qkv", (B, nh * 4 * kd, H, W), "f16")
    qkv_d = G.to_device(qkv, "f16")
    packed = torch.empty((4, bh, n, kd), dtype=torch.float16, device="cuda")
    binding.psa_pack_qkv(qkv_d, packed, nh)
    o_lo = torch.empty((bh, n, kd), dtype=torch.float16, device="cuda")
    o_hi = torch.empty_like(o_lo)
    lse_lo = torch.empty((bh, n), dtype=torch.float32, device="cuda")
    lse_hi = torch.empty_like(lse_lo)
    scale = 1.0 / math.sqrt(kd)
    binding.fa2_forward(packed[0], packed[1], packed[2], o_lo, lse_lo, scale)
    binding.fa2_forward(packed[0], packed[1], packed[3], o_hi, lse_hi, scale)
    out = torch.empty((B, nh * 2 * kd, H, W), dtype=torch.float16, device="cuda")
    binding.psa_merge_attn_nchw(o_lo, o_hi, out, nh)
    binding.fa2_device_status()
    # oracle pipeline
    pk = synth.widen(P.pack_qkv(qkv, nh), "f16")
    r_lo, _ = A.forward(pk[0], pk[1], pk[2], scale)
    r_hi, _ = A.forward(pk[0], pk[1], pk[3], scale)
    ref = P.merge_attn_nchw(r_lo, r_hi, B, nh, H, W)
    check_16bit(G.to_f64(out), ref, "merged attention output")


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("B,nh,kd,H,W", [(8, 4, 32, 20, 20), (2, 2, 16, 5, 7), (1, 3, 2, 1, 3)])
def test_extract_v_and_adjoints_bit_exact(dtype, B, nh, kd, H, W):
    """psa_extract_v_nchw, psa_pack_qkv_backward and psa_merge_attn_backward move words exactly."""
    import torch
    G.require_gpu()
    tag = f"psa_adj/{dtype}/{B}/{nh}/{kd}/{H}/{W}"
    qkv = _patterns(tag + "/qkv", (B, nh * 4 * kd, H, W), dtype)
    v = _raw_tensor(np.zeros((B, nh * 2 * kd, H, W), dtype=qkv.dtype), dtype).view(B, nh * 2 * kd, H, W)
    binding.psa_extract_v_nchw(_raw_tensor(qkv, dtype).view(qkv.shape), v, nh)
    d_packed = _patterns(tag + "/dpacked", (4, B * nh, H * W, kd), dtype)
    d_qkv = _raw_tensor(np.zeros(qkv.shape, dtype=qkv.dtype), dtype).view(qkv.shape)
    binding.psa_pack_qkv_backward(_raw_tensor(d_packed, dtype), d_qkv, nh)
    d_merged = _patterns(tag + "/dmerged", (B, nh * 2 * kd, H, W), dtype)
    d_lo = _raw_tensor(np.zeros((B * nh, H * W, kd), dtype=qkv.dtype), dtype).view(B * nh, H * W, kd)
    d_hi = torch.empty_like(d_lo)
    binding.psa_merge_attn_backward(_raw_tensor(d_merged, dtype).view(d_merged.shape), d_lo, d_hi, nh)
    binding.fa2_device_status()
    assert np.array_equal(_words(v, dtype).reshape(v.shape), P.extract_v_nchw(qkv, nh))
    assert np.array_equal(_words(d_qkv, dtype).reshape(qkv.shape), P.pack_qkv_backward(d_packed, B, nh, H, W))
    want_lo, want_hi = P.merge_attn_backward(d_merged, nh)
    assert np.array_equal(_words(d_lo, dtype).reshape(want_lo.shape), want_lo)
    assert np.array_equal(_words(d_hi, dtype).reshape(want_hi.shape), want_hi)



@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("B,nh,kd,H,W", [(128, 4, 32, 20, 20), (421, 5, 24, 8, 13)])
def test_large_rearrangements_bit_exact(dtype, B, nh, kd, H, W):
    """Batches large enough for the one-thread-per-8x8-block transpose on every one of the
    four rearrangements (pack, merge and their adjoints); the second shape leaves a partial
    last block of threads and head sizes that are not powers of two."""
    G.require_gpu()
    tag = f"psa_big/{dtype}/{B}/{nh}/{kd}/{H}/{W}"
    bh, n = B * nh, H * W
    qkv = _patterns(tag + "/qkv", (B, nh * 4 * kd, H, W), dtype)
    packed = G.empty((4, bh, n, kd), dtype)
    binding.psa_pack_qkv(_raw_tensor(qkv, dtype).view(qkv.shape), packed, nh)
    lo = _patterns(tag + "/lo", (bh, n, kd), dtype)
    hi = _patterns(tag + "/hi", (bh, n, kd), dtype)
    merged = G.empty((B, nh * 2 * kd, H, W), dtype)
    binding.psa_merge_attn_nchw(_raw_tensor(lo, dtype).view(lo.shape), _raw_tensor(hi, dtype).view(hi.shape), merged, nh)
    d_qkv = G.empty(qkv.shape, dtype)
    d_packed = _patterns(tag + "/dpacked", (4, bh, n, kd), dtype)
    binding.psa_pack_qkv_backward(_raw_tensor(d_packed, dtype).view(d_packed.shape), d_qkv, nh)
    d_merged = _patterns(tag + "/dmerged", (B, nh * 2 * kd, H, W), dtype)
    d_lo, d_hi = G.empty((bh, n, kd), dtype), G.empty((bh, n, kd), dtype)
    binding.psa_merge_attn_backward(_raw_tensor(d_merged, dtype).view(d_merged.shape), d_lo, d_hi, nh)
    binding.fa2_device_status()
    assert np.array_equal(_words(packed, dtype).reshape(4, bh, n, kd), P.pack_qkv(qkv, nh))
    assert np.array_equal(_words(merged, dtype).reshape(merged.shape), P.merge_attn_nchw(lo, hi, B, nh, H, W))
    assert np.array_equal(_words(d_qkv, dtype).reshape(qkv.shape), P.pack_qkv_backward(d_packed, B, nh, H, W))
    want_lo, want_hi = P.merge_attn_backward(d_merged, nh)
    assert np.array_equal(_words(d_lo, dtype).reshape(want_lo.shape), want_lo)
    assert np.array_equal(_words(d_hi, dtype).reshape(want_hi.shape), want_hi)

@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("B,nh,kd,H,W", [(8, 4, 32, 20, 20), (3, 1, 8, 3, 5)])
def test_extract_v_backward_accumulates_exactly(dtype, B, nh, kd, H, W):
    """d_qkv from psa_pack_qkv_backward, then psa_extract_v_backward adds d_v into its V channels:
    bit-exact against the oracle's exact sum rounded once to the storage type."""
    G.require_gpu()
    tag = f"psa_evb/{dtype}/{B}/{nh}/{kd}"
    d_packed = synth.tensor(tag + "/dpacked", (4, B * nh, H * W, kd), dtype)
    d_v = synth.tensor(tag + "/dv", (B, nh * 2 * kd, H, W), dtype)
    d_qkv = G.empty((B, nh * 4 * kd, H, W), dtype)
    binding.psa_pack_qkv_backward(G.to_device(d_packed, dtype), d_qkv, nh)
    binding.psa_extract_v_backward(G.to_device(d_v, dtype), d_qkv, nh)
    binding.fa2_device_status()
    want = P.extract_v_backward(d_v, P.pack_qkv_backward(d_packed, B, nh, H, W), nh, dtype)
    assert np.array_equal(_words(d_qkv, dtype).reshape(want.shape), want.view(np.uint32 if dtype == "f32" else np.uint16))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("bh,n,kd", [(32, 400, 32), (3, 129, 32), (2, 300, 64), (1, 1, 32), (2, 520, 64)])
def test_psa_fa2_forward_vs_oracle(dtype, bh, n, kd):
    """One pass over the scores, applied to V_lo and V_hi: each output against the oracle's attention."""
    torch = G.require_gpu()
    packed = synth.tensor(f"psa_fused/{dtype}/{bh}/{n}/{kd}", (4, bh, n, kd), dtype)
    pd = G.to_device(packed, dtype)
    o_lo, o_hi = G.empty((bh, n, kd), dtype), G.empty((bh, n, kd), dtype)
    lse = torch.empty((bh, n), dtype=torch.float32, device="cuda")
    scale = 1 / math.sqrt(kd)
    binding.psa_fa2_forward(pd, o_lo, o_hi, lse, scale)
    binding.fa2_device_status()
    w = synth.widen(packed, dtype)
    r_lo, r_lse = A.forward(w[0], w[1], w[2], scale)
    r_hi, _ = A.forward(w[0], w[1], w[3], scale)
    check_16bit(G.to_f64(o_lo), r_lo, "O_lo")
    check_16bit(G.to_f64(o_hi), r_hi, "O_hi")
    from tests.tolerance import check_lse
    check_lse(G.to_f64(lse), r_lse)


def test_psa_fa2_forward_equals_two_calls():
    """The fused call and the two separate fa2_forward calls agree to rounding (same scores, same P)."""
    torch = G.require_gpu()
    bh, n, kd = 32, 400, 32
    packed = synth.tensor("psa_fused/two_calls", (4, bh, n, kd), "f16")
    pd = G.to_device(packed, "f16")
    fo = [G.empty((bh, n, kd), "f16") for _ in range(2)]
    lse = torch.empty((bh, n), dtype=torch.float32, device="cuda")
    binding.psa_fa2_forward(pd, fo[0], fo[1], lse, 1 / math.sqrt(kd))
    so = [G.empty((bh, n, kd), "f16") for _ in range(2)]
    sl = torch.empty_like(lse)
    for i, sec in enumerate((2, 3)):
        binding.fa2_forward(pd[0], pd[1], pd[sec], so[i], sl, 1 / math.sqrt(kd))
    binding.fa2_device_status()
    for a, b in zip(fo, so):
        assert float((a.float() - b.float()).abs().max()) <= 2e-3
    assert float((lse - sl).abs().max()) <= 1e-5


def _psa_fwd_bwd(packed, d_lo, d_hi, dtype, scale):
    torch = G.require_gpu()
    _, bh, n, kd = packed.shape
    pd = G.to_device(packed, dtype)
    o_lo, o_hi = G.empty((bh, n, kd), dtype), G.empty((bh, n, kd), dtype)
    lse = torch.empty((bh, n), dtype=torch.float32, device="cuda")
    binding.psa_fa2_forward(pd, o_lo, o_hi, lse, scale)
    d_packed = G.empty(packed.shape, dtype)
    code = {"bf16": binding.DTYPE_BF16, "f16": binding.DTYPE_F16}[dtype]
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n, n, kd, code), dtype=torch.uint8, device="cuda")
    binding.psa_fa2_backward(pd, o_lo, o_hi, G.to_device(d_lo, dtype), G.to_device(d_hi, dtype), lse, d_packed, ws, scale)
    binding.fa2_device_status()
    return d_packed


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("bh,n,kd", [(32, 400, 32), (3, 129, 32), (2, 300, 64), (1, 1, 32)])
def test_psa_fa2_backward_vs_oracle(dtype, bh, n, kd):
    """Sections of d_packed: dQ_lo + dQ_hi, dK_lo + dK_hi, dV_lo, dV_hi against the oracle."""
    tag = f"psa_bwd/{dtype}/{bh}/{n}/{kd}"
    packed = synth.tensor(tag + "/packed", (4, bh, n, kd), dtype)
    d_lo = synth.tensor(tag + "/dlo", (bh, n, kd), dtype)
    d_hi = synth.tensor(tag + "/dhi", (bh, n, kd), dtype)
    scale = 1 / math.sqrt(kd)
    got = G.to_f64(_psa_fwd_bwd(packed, d_lo, d_hi, dtype, scale))
    w = lambda x: synth.widen(x, dtype)  # noqa: E731
    want = A.psa_backward(w(packed), w(d_lo), w(d_hi), scale)
    for s, name in enumerate(("dQ_lo+dQ_hi", "dK_lo+dK_hi", "dV_lo", "dV_hi")):
        check_16bit(got[s], want[s], name)


def test_c2psa_training_chain():
    """The whole C2PSA attention step and its gradient, fp16, QKV [8, 512, 20, 20], 4 heads, KEY_DIM 32:
    pack -> fused attention -> merge; then merge^T -> fused attention backward -> pack^T, plus a
    gradient arriving at the extracted V (extract_v^T adds it into d_qkv)."""
    torch = G.require_gpu()
    B, nh, kd, H, W = 8, 4, 32, 20, 20
    n, bh, c = H * W, B * nh, nh * 2 * kd
    qkv = synth.tensor("c2psa_train/qkv", (B, nh * 4 * kd, H, W), "f16")
    d_out = synth.tensor("c2psa_train/dout", (B, c, H, W), "f16")
    d_vpe = synth.tensor("c2psa_train/dvpe", (B, c, H, W), "f16")
    scale = 1 / math.sqrt(kd)
    qkv_d = G.to_device(qkv, "f16")
    packed = G.empty((4, bh, n, kd), "f16")
    binding.psa_pack_qkv(qkv_d, packed, nh)
    o_lo, o_hi = G.empty((bh, n, kd), "f16"), G.empty((bh, n, kd), "f16")
    lse = torch.empty((bh, n), dtype=torch.float32, device="cuda")
    binding.psa_fa2_forward(packed, o_lo, o_hi, lse, scale)
    d_lo, d_hi = G.empty((bh, n, kd), "f16"), G.empty((bh, n, kd), "f16")
    binding.psa_merge_attn_backward(G.to_device(d_out, "f16"), d_lo, d_hi, nh)
    d_packed = G.empty((4, bh, n, kd), "f16")
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n, n, kd, binding.DTYPE_F16), dtype=torch.uint8,
                     device="cuda")
    binding.psa_fa2_backward(packed, o_lo, o_hi, d_lo, d_hi, lse, d_packed, ws, scale)
    d_qkv = G.empty(qkv.shape, "f16")
    binding.psa_pack_qkv_backward(d_packed, d_qkv, nh)
    binding.psa_extract_v_backward(G.to_device(d_vpe, "f16"), d_qkv, nh)
    binding.fa2_device_status()
    # oracle chain in float64
    pk = synth.widen(P.pack_qkv(qkv, nh), "f16")
    g_lo, g_hi = P.merge_attn_backward(synth.widen(d_out, "f16"), nh)
    g_packed = A.psa_backward(pk, g_lo, g_hi, scale)
    want = P.pack_qkv_backward(g_packed, B, nh, H, W)
    for h in range(nh):
        want[:, h * 4 * kd + 2 * kd:(h + 1) * 4 * kd] += synth.widen(d_vpe, "f16")[:, h * 2 * kd:(h + 1) * 2 * kd]
    check_16bit(G.to_f64(d_qkv), want, "d_qkv")
