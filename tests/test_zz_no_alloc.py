"""fa2_backward_noalloc: the backward for callers that cannot allocate device memory.

Such callers (code whose device memory belongs to a host framework's pool, or a
service with a memory budget fixed at start-up) cannot hand fa2_backward a
workspace; this entry point takes it from the library's fixed device scratch
instead.  The test calls it through the C ABI twice in a row, on two different
problems, and checks each result against fa2_backward with a caller-owned
workspace: bit for bit where that computation is deterministic (every gradient at
head size 128, dK and dV at 64), within the parity bar the other GPU tests use for
the one-pass dQ, whose float32 sums land in any order.  It also checks that a
problem needing more than the fixed scratch is refused without a launch, and that
a problem whose dQ pass is split over key ranges (partial sums in the scratch)
matches fa2_backward bit for bit.

The file name makes pytest collect it last.
"""
import ctypes
import math

import pytest

from attention_fa2_forward_02_gb300 import binding, synth
from tests import gpu_util as G
from tests.tolerance import check_16bit

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 7


def _problem(tag, bh, n_q, n_k, d, dtype):
    torch = G.require_gpu()
    q, k, v = G.inputs(tag, bh, n_q, n_k, d, dtype)
    d_o = synth.tensor(tag + "/do", (bh, n_q, d), dtype)
    qd, kd, vd, dod = (G.to_device(x, dtype) for x in (q, k, v, d_o))
    scale = 1 / math.sqrt(d)
    o = G.empty((bh, n_q, d), dtype)
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    return qd, kd, vd, o, dod, lse, scale


def _with_workspace(qd, kd, vd, o, dod, lse, scale):
    torch = G.require_gpu()
    bh, n_q, d = qd.shape
    code = binding.DTYPE_BF16 if qd.dtype == torch.bfloat16 else binding.DTYPE_F16
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n_q, kd.shape[1], d, code), dtype=torch.uint8,
                     device="cuda")
    grads = [torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)]
    binding.fa2_backward(qd, kd, vd, o, dod, lse, *grads, ws, scale)
    return grads


def test_noalloc_matches_backward_on_two_calls_in_a_row():
    """Head size 128 runs the deterministic two passes, so the result must equal
    fa2_backward's bit for bit; head size 64 runs the one-pass kernel, whose dQ sums land
    in any order, so dQ is compared within the parity bar (dK and dV bit for bit).
    The outputs sit between guard bands that must stay untouched."""
    torch = G.require_gpu()
    # 80 heads of 3 key tiles at head size 64: enough key tiles for the one-pass kernel
    problems = [("noalloc/a", 3, 700, 520, 128, "bf16"), ("noalloc/b", 80, 129, 300, 64, "f16")]
    results = []
    for tag, bh, n_q, n_k, d, dtype in problems:
        args = _problem(tag, bh, n_q, n_k, d, dtype)
        got = [G.Guarded(tuple(x.shape), x.dtype) for x in args[:3]]
        binding.fa2_backward_noalloc(*args[:6], *(g.t for g in got), args[6])
        results.append((d, args, got))
    binding.fa2_device_status()
    for d, args, got in results:
        want = _with_workspace(*args)
        torch.cuda.synchronize()
        for name, a, b in zip(("dQ", "dK", "dV"), got, want):
            a.assert_intact(f"fa2_backward_noalloc {name}")
            if d > 64 or name != "dQ":
                assert torch.equal(a.t, b), f"fa2_backward_noalloc {name} differs from fa2_backward (head size {d})"
            else:
                check_16bit(G.to_f64(a.t), G.to_f64(b), f"fa2_backward_noalloc {name}")


def test_noalloc_two_pass_when_the_accumulator_does_not_fit():
    """8 heads x 4096 query rows x 1280 keys, head_dim 64: the one-pass workspace (8.65 MB
    with its dQ accumulator) exceeds the fixed 8 MiB scratch, the two-pass one (256 KiB)
    fits. (With fewer keys the shape would leave the one-pass kernel anyway: its dK/dV pass
    would split the queries over clusters, which the two passes do.)"""
    torch = G.require_gpu()
    bh, n_q, n_k, d = 8, 4096, 1280, 64
    assert binding.fa2_backward_workspace_size(bh, n_q, n_k, d, binding.DTYPE_BF16) > 8 << 20
    args = _problem("noalloc/c", bh, n_q, n_k, d, "bf16")
    got = [torch.empty_like(args[0]), torch.empty_like(args[1]), torch.empty_like(args[2])]
    binding.fa2_backward_noalloc(*args[:6], *got, args[6])
    binding.fa2_device_status()
    want = _with_workspace(*args)
    torch.cuda.synchronize()
    for name, a, b in zip(("dQ", "dK", "dV"), got, want):
        check_16bit(G.to_f64(a), G.to_f64(b), f"fa2_backward_noalloc (two-pass) {name}")


def test_noalloc_refuses_problems_beyond_its_scratch():
    torch = G.require_gpu()
    t = torch.empty((1, 128, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 128), dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(t.data_ptr())
    # 64 heads x 32768 query rows need 16 MiB of workspace: refused before anything is launched
    st = binding.library().fa2_backward_noalloc(p, p, p, p, p, ctypes.c_void_p(lse.data_ptr()), p, p, p,
                                                64, 32768, 128, 128, binding.DTYPE_BF16, 0.088, None)
    assert st == SCRATCH_LIMIT
    binding.fa2_device_status()


def test_noalloc_with_the_split_dq_pass():
    """Two heads of one query tile and 4096 keys at head size 128: fa2_backward splits the dQ
    pass into key ranges whose float32 partial sums live in the workspace; from the fixed
    scratch, fa2_backward_noalloc does the same and must equal fa2_backward bit for bit."""
    torch = G.require_gpu()
    bh, n_q, n_k, d = 2, 128, 4096, 128
    ws_bytes = binding.fa2_backward_workspace_size(bh, n_q, n_k, d, binding.DTYPE_BF16)
    assert ws_bytes > 8 * bh * 128  # the partial sums are part of it
    args = _problem("noalloc/split", bh, n_q, n_k, d, "bf16")
    got = [G.Guarded(tuple(x.shape), x.dtype) for x in args[:3]]
    binding.fa2_backward_noalloc(*args[:6], *(g.t for g in got), args[6])
    binding.fa2_device_status()
    want = _with_workspace(*args)
    torch.cuda.synchronize()
    for name, a, b in zip(("dQ", "dK", "dV"), got, want):
        a.assert_intact(f"fa2_backward_noalloc {name}")
        assert torch.equal(a.t, b), f"fa2_backward_noalloc {name} differs from fa2_backward"
