"""Attention on tensors of more than 2^31 elements, checked exactly through repeated keys.

With N_k = c * P keys in which key j is a copy of key j mod P, every softmax row weighs the
c copies of a key alike, so the problem reduces to the one over the P distinct keys
(flash_attn2.rs, `flash_attention2_forward` / `_backward_dkv` / `_backward_dq`, with every
sum over keys grouped by copy): O and dQ are the P-key problem's, LSE is its LSE + ln c, and
dK, dV of key j are the P-key problem's dK, dV of key j mod P divided by c (the oracle pin
`test_repeated_keys_reduce_to_the_distinct_ones`). The float64 oracle solves the P-key
problem; the kernels run all N_k keys. P = 1000 is not a multiple of the tile size, so every
key tile holds a different mix of the P keys, and every copy of a key must come out with
the same dK and dV row bit for bit."""
import math

import numpy as np
import pytest

from attention_fa2_forward_02_gb300 import binding, synth
from oracle import attention as A
from tests import gpu_util as G
from tests.split_rules import balanced_ranges, fwd_key_splits
from tests.tolerance import check_16bit, check_16bit_grad, check_16bit_long, check_lse

pytestmark = pytest.mark.gpu

P, D, N_Q = 1000, 128, 200


def _run(tag, bh, copies):
    """Forward and backward on `bh` heads of P * copies repeated keys; host copies of the
    P-key inputs and the device outputs."""
    torch = G.require_gpu()
    n_k = P * copies
    scale = 1 / math.sqrt(D)
    q = synth.tensor(f"{tag}/q", (bh, N_Q, D), "bf16")
    kp = synth.tensor(f"{tag}/k", (bh, P, D), "bf16")
    vp = synth.tensor(f"{tag}/v", (bh, P, D), "bf16")
    d_o = synth.tensor(f"{tag}/do", (bh, N_Q, D), "bf16")
    qd, dod = G.to_device(q, "bf16"), G.to_device(d_o, "bf16")
    kd = G.to_device(kp, "bf16").repeat(1, copies, 1)  # key j is key j mod P
    vd = G.to_device(vp, "bf16").repeat(1, copies, 1)
    o = G.empty((bh, N_Q, D), "bf16")
    lse = torch.empty((bh, N_Q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    dq, dk, dv = G.empty((bh, N_Q, D), "bf16"), G.empty((bh, n_k, D), "bf16"), G.empty((bh, n_k, D), "bf16")
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, N_Q, n_k, D, binding.DTYPE_BF16), dtype=torch.uint8,
                     device="cuda")
    binding.fa2_backward(qd, kd, vd, o, dod, lse, dq, dk, dv, ws, scale)
    binding.fa2_device_status()
    for name, g in (("dK", dk), ("dV", dv)):
        for b in range(bh):
            rows = g[b].view(copies, P, D)
            for c0 in range(0, copies, 2048):
                part = rows[c0:c0 + 2048]
                assert torch.equal(part, rows[:1].expand_as(part)), f"{name} head {b}: copies {c0}.. differ"
    return (q, kp, vp, d_o), (o, lse, dq, dk, dv), scale


def _reference(inputs, outputs, scale, b, copies):
    """The oracle's P-key problem for head b, its backward from the stored O and LSE that the
    kernels read, and the device outputs of that head in float64."""
    q, kp, vp, d_o = (synth.widen(x[b:b + 1], "bf16") for x in inputs)
    o, lse, dq, dk, dv = outputs
    o_got, l_got = G.to_f64(o[b:b + 1]), G.to_f64(lse[b:b + 1])
    o_ref, l_ref = A.forward(q, kp, vp, scale)
    grads = A.backward_slice(q, kp, vp, d_o, scale, 0, row_chunk=256, o=o_got, lse=l_got - math.log(copies),
                             rounding_scales=True)
    weighted = A.probabilities(q, kp, scale)[0] @ np.abs(vp[0])  # sum_j P_ij |v_jd|
    got = (o_got[0], l_got[0], G.to_f64(dq[b]), copies * G.to_f64(dk[b, :P]), copies * G.to_f64(dv[b, :P]))
    return got, (o_ref[0], l_ref[0] + math.log(copies)), grads, weighted


def test_heads_past_2_31_elements():
    """130 heads of 131,000 keys: K, V, dK and dV hold 2.18e9 elements; byte offsets cross
    2^31 inside head 64, element offsets cross 2^31 (byte offsets 2^32) inside head 128, and
    head 129 lies wholly past both; every head ends in a partial key tile (131,000 mod
    128 = 56). Heads 0, 64, 128, 129 against the oracle at the usual bars; every copy of
    every key bit-identical in dK and dV."""
    bh, copies = 130, 131
    per_head = P * copies * D
    assert 64 * per_head * 2 < 2 ** 31 < 65 * per_head * 2 and 128 * per_head < 2 ** 31 < 129 * per_head
    inputs, outputs, scale = _run("large/heads", bh, copies)
    for b in (0, 64, 128, 129):
        (o, lse, dq, dk_c, dv_c), (o_ref, l_ref), g, _ = _reference(inputs, outputs, scale, b, copies)
        check_16bit(o, o_ref, f"O head {b}")
        check_lse(lse, l_ref, f"LSE head {b}")
        check_16bit_grad(dq, g[0], g[3] / math.sqrt(copies), "bf16", f"dQ head {b}")
        check_16bit_grad(dk_c, g[1], g[4], "bf16", f"dK x c head {b}")
        check_16bit_grad(dv_c, g[2], g[5], "bf16", f"dV x c head {b}")


def test_one_head_of_16m_keys():
    """One head of 16,778,000 keys (2.15e9 elements in K, V, dK, dV; a partial last key tile,
    N_k mod 128 = 16). The forward's query-tile pair is shared by a cluster of 16 CTAs, each
    adding 8,192 or 8,193 of the 131,079 key tiles into its float32 O and row sums, so O is held to
    the bar for float32 accumulation over that many additions (check_16bit_long: the 2e-2
    absolute bar, and 2e-2 max|ref| + n 2^-24 sum_j P_ij |v_j| per element); LSE, and the
    gradients (dQ summed in the split dQ pass's key ranges, dK and dV over the 200 queries)
    at the usual bars."""
    copies = 16778
    n_k = P * copies
    assert n_k * D > 2 ** 31 and n_k % 128 == 16
    inputs, outputs, scale = _run("large/long", 1, copies)
    (o, lse, dq, dk_c, dv_c), (o_ref, l_ref), g, weighted = _reference(inputs, outputs, scale, 0, copies)
    n_kt, ranges = (n_k + 127) // 128, fwd_key_splits(1, N_Q, n_k, D)
    assert ranges == 16
    longest = max(hi - lo for lo, hi in balanced_ranges(n_kt, ranges))
    check_16bit_long(o, o_ref, weighted, longest, "O")
    check_lse(lse, l_ref, "LSE")
    check_16bit_grad(dq, g[0], g[3] / math.sqrt(copies), "bf16", "dQ")
    check_16bit_grad(dk_c, g[1], g[4], "bf16", "dK x c")
    check_16bit_grad(dv_c, g[2], g[5], "bf16", "dV x c")
