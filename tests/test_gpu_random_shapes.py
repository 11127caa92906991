"""Forward and backward on seeded random shapes, against the float64 oracle.

The library picks its kernels from the sizes alone: the forward's key ranges in a cluster
for few query tiles and many keys, the one-pass backward or the two passes, the dQ pass's
key ranges and the dK/dV pass's query ranges in a cluster. Shapes drawn log-uniformly
(heads up to 120, 1 to 40000 queries and keys, head sizes 8 to 128 in either 16-bit type)
reach every one of those choices and the edges between them, single rows and ragged tails
included; the mirrors of the choices below show which each shape takes, and the draw
covers them all. O and LSE of the first and last heads, and their gradients at the
elementwise bound (from the stored O and LSE the backward reads), against the oracle.
"""
import math
import random

import numpy as np
import pytest

from attention_fa2_forward_02_gb300 import binding, synth
from oracle import attention as A
from tests import gpu_util as G
from tests.split_rules import dkdv_tiles_per_cta, dkv_query_splits, dq_key_splits, fwd_key_splits, one_pass
from tests.tolerance import check_16bit, check_16bit_grad, check_lse

pytestmark = pytest.mark.gpu


def _draw(count=24, seed=2026):
    rng = random.Random(seed)
    shapes = []
    while len(shapes) < count:
        d = rng.choice([8, 16, 24, 32, 40, 48, 56, 64, 72, 96, 112, 128])
        bh = int(math.exp(rng.uniform(0, math.log(120))))
        n_q = int(math.exp(rng.uniform(0, math.log(40000))))
        n_k = int(math.exp(rng.uniform(0, math.log(40000))))
        if n_q * n_k > 3e6 or bh * n_q * n_k * d > 2e9:  # keeps the oracle's share to seconds
            continue
        shapes.append((bh, n_q, n_k, d, rng.choice(["bf16", "f16"])))
    return shapes


SHAPES = _draw()


def test_the_draw_reaches_every_kernel_choice():
    two = [s for s in SHAPES if not one_pass(s[0], s[2], s[3])]
    assert any(fwd_key_splits(*s[:4]) > 1 for s in SHAPES)
    assert any(one_pass(s[0], s[2], s[3]) for s in SHAPES) and two
    assert {2, 4, 8} <= {dkv_query_splits(*s[:4]) for s in two}
    assert any(dq_key_splits(*s[:3]) > 1 and dkv_query_splits(*s[:4]) == 1 for s in two)
    assert any(s[1] == 1 for s in SHAPES) and any(s[2] <= 2 for s in SHAPES)


@pytest.mark.parametrize("bh,n_q,n_k,d,dtype", SHAPES)
def test_random_shape_vs_oracle(bh, n_q, n_k, d, dtype):
    torch = G.require_gpu()
    tag = f"rand/{bh}/{n_q}/{n_k}/{d}/{dtype}"
    q, k, v = G.inputs(tag, bh, n_q, n_k, d, dtype)
    d_o = synth.tensor(tag + "/do", (bh, n_q, d), dtype)
    scale = 1 / math.sqrt(d)
    qd, kd, vd, dod = (G.to_device(x, dtype) for x in (q, k, v, d_o))
    o = G.empty((bh, n_q, d), dtype)
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    assert binding.fa2_last_launch_info()["fwd_key_ranges"] == fwd_key_splits(bh, n_q, n_k, d)
    grads = [G.empty(x.shape, dtype) for x in (q, k, v)]
    code = {"bf16": binding.DTYPE_BF16, "f16": binding.DTYPE_F16}[dtype]
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n_q, n_k, d, code), dtype=torch.uint8, device="cuda")
    binding.fa2_backward(qd, kd, vd, o, dod, lse, *grads, ws, scale)
    # the kernels the library chose are the ones the size rules give
    info = binding.fa2_last_launch_info()
    if one_pass(bh, n_k, d):
        expect = (1, 1, 1, 0)
    else:
        qs = dkv_query_splits(bh, n_q, n_k, d)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        expect = (0, qs, dq_key_splits(bh, n_q, n_k), 0 if qs > 1 else dkdv_tiles_per_cta(bh, n_q, n_k, sms))
    assert (info["bwd_one_pass"], info["bwd_dkv_query_ranges"], info["bwd_dq_key_ranges"],
            info["bwd_key_tiles_per_cta"]) == expect
    binding.fa2_device_status()
    o_st, l_st = G.to_f64(o), G.to_f64(lse)
    dq, dk, dv = (G.to_f64(g) for g in grads)
    w = lambda x: synth.widen(x, dtype)  # noqa: E731
    for b in sorted({0, bh - 1}):
        o_ref, l_ref = A.forward(w(q[b:b + 1]), w(k[b:b + 1]), w(v[b:b + 1]), scale)
        check_16bit(o_st[b], o_ref[0], f"O head {b}")
        check_lse(l_st[b], l_ref[0], f"LSE head {b}")
        rq, rk, rv, sq, sk, sv = A.backward_slice(w(q), w(k), w(v), w(d_o), scale, b, row_chunk=512, o=o_st,
                                                  lse=l_st, rounding_scales=True)
        check_16bit_grad(dq[b], rq, sq, dtype, f"dQ head {b}")
        check_16bit_grad(dk[b], rk, sk, dtype, f"dK head {b}")
        check_16bit_grad(dv[b], rv, sv, dtype, f"dV head {b}")
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))
