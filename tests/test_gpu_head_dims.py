"""Head dimensions other than 32 / 64 / 128 (any multiple of 8 up to 128).

The pages' builders accept any head_dim (the vyre unit tests use 7, 8 and 16);
the kernels run at the next of 32, 64, 128 with the extra columns read as zeros
and never stored.  Forward and backward against the float64 oracle.
"""
import math

import numpy as np
import pytest

from attention_fa2_forward_02_gb300 import binding, synth
from oracle import attention as A
from tests import gpu_util as G
from tests.tolerance import check_16bit, check_f32, check_lse

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [8, 16, 24, 40, 48, 56, 72, 96, 120])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("bh", [2, 50])
def test_forward_backward_any_head_dim(d, dtype, bh):
    """Two heads (the backward's two passes at every head size) and 50 heads of 3 key tiles
    (150 in all: the one-pass backward up to head size 64)."""
    torch = G.require_gpu()
    n_q, n_k = 200, 333
    tag = f"hd/{dtype}/{d}/{bh}"
    q, k, v = G.inputs(tag, bh, n_q, n_k, d, dtype)
    d_o = synth.tensor(tag + "/do", (bh, n_q, d), dtype)
    scale = 1 / math.sqrt(d)
    qd, kd, vd, dod = (G.to_device(x, dtype) for x in (q, k, v, d_o))
    o = G.empty((bh, n_q, d), dtype)
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    dq, dk, dv = G.empty((bh, n_q, d), dtype), G.empty((bh, n_k, d), dtype), G.empty((bh, n_k, d), dtype)
    code = {"bf16": binding.DTYPE_BF16, "f16": binding.DTYPE_F16}[dtype]
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n_q, n_k, d, code), dtype=torch.uint8, device="cuda")
    binding.fa2_backward(qd, kd, vd, o, dod, lse, dq, dk, dv, ws, scale)
    binding.fa2_device_status()
    w = lambda x: synth.widen(x, dtype)  # noqa: E731
    o_ref, l_ref = A.forward(w(q), w(k), w(v), scale)
    check_16bit(G.to_f64(o), o_ref, "O")
    check_lse(G.to_f64(lse), l_ref)
    rq, rk, rv = A.backward(w(q), w(k), w(v), w(d_o), scale)
    check_16bit(G.to_f64(dq), rq, "dQ")
    check_16bit(G.to_f64(dk), rk, "dK")
    check_16bit(G.to_f64(dv), rv, "dV")


@pytest.mark.parametrize("d", [1, 3, 7, 8, 16, 48, 100, 104, 127])
def test_forward_f32_any_head_dim(d):
    torch = G.require_gpu()
    bh, n_q, n_k = 2, 64, 90
    q, k, v = G.inputs(f"hd32/{d}", bh, n_q, n_k, d, "f32")
    qd, kd, vd = (G.to_device(x, "f32") for x in (q, k, v))
    o = G.empty((bh, n_q, d), "f32")
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, 1 / math.sqrt(d))
    binding.fa2_device_status()
    o_ref, l_ref = A.forward(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), 1 / math.sqrt(d))
    check_f32(G.to_f64(o), o_ref, "O")
    check_f32(G.to_f64(lse), l_ref, "LSE")


@pytest.mark.parametrize("kd", [16, 48])
def test_psa_fused_pair_other_key_dims(kd):
    torch = G.require_gpu()
    bh, n = 4, 150
    packed = synth.tensor(f"hd_psa/{kd}", (4, bh, n, kd), "bf16")
    d_lo = synth.tensor(f"hd_psa/{kd}/dlo", (bh, n, kd), "bf16")
    d_hi = synth.tensor(f"hd_psa/{kd}/dhi", (bh, n, kd), "bf16")
    scale = 1 / math.sqrt(kd)
    pd = G.to_device(packed, "bf16")
    o_lo, o_hi = G.empty((bh, n, kd), "bf16"), G.empty((bh, n, kd), "bf16")
    lse = torch.empty((bh, n), dtype=torch.float32, device="cuda")
    binding.psa_fa2_forward(pd, o_lo, o_hi, lse, scale)
    d_packed = G.empty(packed.shape, "bf16")
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n, n, kd, binding.DTYPE_BF16), dtype=torch.uint8,
                     device="cuda")
    binding.psa_fa2_backward(pd, o_lo, o_hi, G.to_device(d_lo, "bf16"), G.to_device(d_hi, "bf16"), lse, d_packed, ws,
                             scale)
    binding.fa2_device_status()
    w = synth.widen(packed, "bf16")
    check_16bit(G.to_f64(o_lo), A.forward(w[0], w[1], w[2], scale)[0], "O_lo")
    check_16bit(G.to_f64(o_hi), A.forward(w[0], w[1], w[3], scale)[0], "O_hi")
    want = A.psa_backward(w, synth.widen(d_lo, "bf16"), synth.widen(d_hi, "bf16"), scale)
    got = G.to_f64(d_packed)
    for s in range(4):
        check_16bit(got[s], want[s], f"d_packed section {s}")
