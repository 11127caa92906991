"""GPU parity of fa2_backward (dQ, dK, dV) against the float64 oracle, through the C ABI."""
import math

import numpy as np
import pytest

from attention_fa2_forward_02_gb300 import binding, synth
from oracle import attention as A
from tests import gpu_util as G
from tests.split_rules import dkv_query_splits, dq_key_splits, one_pass
from tests.tolerance import check_reordered_sum, check_16bit, check_16bit_grad, check_lse

pytestmark = pytest.mark.gpu


def run_fwd_bwd(q, k, v, d_o, dtype, scale):
    """GPU forward (O, LSE), then GPU backward from them, as a training step would."""
    torch = G.require_gpu()
    bh, n_q, d = q.shape
    n_k = k.shape[1]
    qd, kd, vd, dod = (G.to_device(x, dtype) for x in (q, k, v, d_o))
    o = G.empty((bh, n_q, d), dtype)
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    dq, dk, dv = G.empty((bh, n_q, d), dtype), G.empty((bh, n_k, d), dtype), G.empty((bh, n_k, d), dtype)
    code = {"bf16": binding.DTYPE_BF16, "f16": binding.DTYPE_F16}[dtype]
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n_q, n_k, d, code), dtype=torch.uint8, device="cuda")
    binding.fa2_backward(qd, kd, vd, o, dod, lse, dq, dk, dv, ws, scale)
    binding.fa2_device_status()
    return G.to_f64(dq), G.to_f64(dk), G.to_f64(dv)


SHAPES = [(2, 300, 400), (1, 1, 1), (3, 129, 129), (1, 520, 77), (2, 64, 1000), (1, 256, 256)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("bh,n_q,n_k", SHAPES)
def test_backward_vs_oracle(dtype, d, bh, n_q, n_k):
    tag = f"bwd/{dtype}/{d}/{bh}/{n_q}/{n_k}"
    q, k, v = G.inputs(tag, bh, n_q, n_k, d, dtype)
    d_o = synth.tensor(tag + "/do", (bh, n_q, d), dtype)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = run_fwd_bwd(q, k, v, d_o, dtype, scale)
    w = lambda x: synth.widen(x, dtype)
    rq, rk, rv = A.backward(w(q), w(k), w(v), w(d_o), scale)
    check_16bit(dq, rq, "dQ")
    check_16bit(dk, rk, "dK")
    check_16bit(dv, rv, "dV")


# many heads, so that head sizes up to 64 take the one-pass kernel; ragged query and key tails
ONE_PASS_SHAPES = [(80, 300, 150), (160, 129, 77), (75, 64, 1000), (96, 1, 129)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [32, 40, 64])
@pytest.mark.parametrize("bh,n_q,n_k", ONE_PASS_SHAPES)
def test_backward_one_pass_vs_oracle(dtype, d, bh, n_q, n_k):
    """The one-pass kernel (head size <= 64, more than 74 key tiles in all) on ragged shapes."""
    assert one_pass(bh, n_k, d)
    tag = f"bwd1p/{dtype}/{d}/{bh}/{n_q}/{n_k}"
    q, k, v = G.inputs(tag, bh, n_q, n_k, d, dtype)
    d_o = synth.tensor(tag + "/do", (bh, n_q, d), dtype)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = run_fwd_bwd(q, k, v, d_o, dtype, scale)
    w = lambda x: synth.widen(x, dtype)  # noqa: E731
    rq, rk, rv = A.backward(w(q), w(k), w(v), w(d_o), scale)
    check_16bit(dq, rq, "dQ")
    check_16bit(dk, rk, "dK")
    check_16bit(dv, rv, "dV")


def test_backward_gradient_identities():
    """sum_j dV_j = sum_i dO_i and sum_j dK_j = 0 (the rows of P sum to one) on the GPU result."""
    bh, n, d = 2, 384, 64
    q, k, v = G.inputs("bwd/identities", bh, n, n, d, "bf16")
    d_o = synth.tensor("bwd/identities/do", (bh, n, d), "bf16")
    dq, dk, dv = run_fwd_bwd(q, k, v, d_o, "bf16", 1 / math.sqrt(d))
    do64 = synth.widen(d_o, "bf16")
    assert np.max(np.abs(dv.sum(axis=1) - do64.sum(axis=1))) <= 0.05 * np.max(np.abs(do64.sum(axis=1)))
    assert np.max(np.abs(dk.sum(axis=1))) <= 0.02 * np.max(np.abs(dk)) * math.sqrt(n)


def test_backward_full_size_whole_heads():
    """bf16 forward+backward, B=2 H=16 (BH=32), N=8192, d=128: every dQ/dK/dV row of two heads
    against the oracle's chunked per-head backward."""
    bh, n, d = 32, 8192, 128
    q, k, v = G.inputs("config/fwdbwd_d128", bh, n, n, d, "bf16")
    d_o = synth.tensor("config/fwdbwd_d128/do", (bh, n, d), "bf16")
    scale = 1 / math.sqrt(d)
    dq, dk, dv = run_fwd_bwd(q, k, v, d_o, "bf16", scale)
    w = lambda x: synth.widen(x, "bf16")
    for b in (0, 31):
        rq, rk, rv = A.backward_slice(w(q[b:b + 1]), w(k[b:b + 1]), w(v[b:b + 1]), w(d_o[b:b + 1]), scale, 0)
        check_16bit(dq[b], rq, f"dQ head {b}")
        check_16bit(dk[b], rk, f"dK head {b}")
        check_16bit(dv[b], rv, f"dV head {b}")



def test_backward_full_size_d64_whole_heads():
    """bf16 forward+backward, B=4 H=16 (BH=64), N=4096, d=64 (the one-pass backward with the
    float32 dQ accumulator): every dQ/dK/dV row of the first and last heads against the oracle."""
    bh, n, d = 64, 4096, 64
    q, k, v = G.inputs("config/fwdbwd_d64", bh, n, n, d, "bf16")
    d_o = synth.tensor("config/fwdbwd_d64/do", (bh, n, d), "bf16")
    scale = 1 / math.sqrt(d)
    dq, dk, dv = run_fwd_bwd(q, k, v, d_o, "bf16", scale)
    w = lambda x: synth.widen(x, "bf16")
    for b in (0, bh - 1):
        rq, rk, rv = A.backward_slice(w(q[b:b + 1]), w(k[b:b + 1]), w(v[b:b + 1]), w(d_o[b:b + 1]), scale, 0)
        check_16bit(dq[b], rq, f"dQ head {b}")
        check_16bit(dk[b], rk, f"dK head {b}")
        check_16bit(dv[b], rv, f"dV head {b}")


def test_backward_cross_attention_peaked_whole_heads():
    """B=1 H=32, N_q=1024 vs N_k=32768, d=128, K scaled by 8 (peaked rows; the one-grid passes
    kernel puts its dQ CTAs first at this shape).  The backward reads a stored O and LSE: for the
    two checked heads those are the oracle's (O rounded to bfloat16, LSE to float32), the same
    ones the oracle's backward reads, so that both sides form the same D; the other heads keep
    the GPU forward's.  Two runs give bit-identical gradients, and every dQ/dK/dV element of
    heads 0 and 31 is within 2e-2 + u|ref| + 8u R of the oracle (tests/tolerance.py)."""
    torch = G.require_gpu()
    bh, n_q, n_k, d = 32, 1024, 32768, 128
    q, k, v = G.inputs("config/cross_k8", bh, n_q, n_k, d, "bf16", k_scale=8.0)
    d_o = synth.tensor("config/cross_k8/do", (bh, n_q, d), "bf16")
    scale = 1 / math.sqrt(d)
    w = lambda x: synth.widen(x, "bf16")
    qd, kd, vd, dod = (G.to_device(x, "bf16") for x in (q, k, v, d_o))
    o = G.empty((bh, n_q, d), "bf16")
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    heads = (0, bh - 1)
    stored = {}
    for b in heads:
        o_ref = np.empty((n_q, d))
        l_ref = np.empty(n_q)
        for r0 in range(0, n_q, 128):
            rows = np.arange(r0, r0 + 128)
            o_ref[rows], l_ref[rows] = A.forward_rows(w(q[b:b + 1]), w(k[b:b + 1]), w(v[b:b + 1]), scale, 0, rows)
        o_st = synth.to_storage(o_ref[None], "bf16")
        l_st = l_ref.astype(np.float32)
        o[b] = G.to_device(o_st, "bf16")[0]
        lse[b] = torch.from_numpy(l_st).cuda()
        stored[b] = (synth.widen(o_st, "bf16"), l_st.astype(np.float64)[None])
    code = binding.DTYPE_BF16
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n_q, n_k, d, code), dtype=torch.uint8, device="cuda")
    runs = []
    for _ in range(2):
        grads = [G.empty(x.shape, "bf16") for x in (q, k, v)]
        binding.fa2_backward(qd, kd, vd, o, dod, lse, *grads, ws, scale)
        binding.fa2_device_status()
        runs.append([G.to_f64(g) for g in grads])
    for name, a, b in zip(("dQ", "dK", "dV"), *runs):
        assert np.array_equal(a, b), f"{name} differs between two runs"
    dq, dk, dv = runs[0]
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))
    for b in heads:
        o_st, l_st = stored[b]
        rq, rk, rv, sq, sk, sv = A.backward_slice(w(q[b:b + 1]), w(k[b:b + 1]), w(v[b:b + 1]), w(d_o[b:b + 1]), scale,
                                                  0, row_chunk=256, o=o_st, lse=l_st, rounding_scales=True)
        check_16bit_grad(dq[b], rq, sq, "bf16", f"dQ head {b}")
        check_16bit_grad(dk[b], rk, sk, "bf16", f"dK head {b}")
        check_16bit_grad(dv[b], rv, sv, "bf16", f"dV head {b}")


def _stages(qd, kd, vd, o, dod, lse, scale, ws, dtype):
    """The two-pass backward through its three stage entry points."""
    staged = [G.empty(tuple(x.shape), dtype) for x in (qd, kd, vd)]
    binding.fa2_backward_preprocess(o, dod, lse, ws, kd.shape[1])
    binding.fa2_backward_dkdv(qd, kd, vd, dod, ws, staged[1], staged[2], scale)
    binding.fa2_backward_dq(qd, kd, vd, dod, ws, staged[0], scale)
    return staged


@pytest.mark.parametrize("d,dtype", [(64, "f16"), (128, "bf16")])
def test_backward_stages_vs_oracle_and_whole(d, dtype):
    """fa2_backward_preprocess + _dkdv + _dq (the pages' two-pass structure, from the smaller
    two-pass workspace) against the oracle and bit-reproducible from run to run; equal to
    fa2_backward bit for bit where that takes the same two passes (head_dim > 64, or too few
    key tiles for the one-pass kernel), within the parity bar of its one-pass result
    otherwise (40 heads here at head size 64)."""
    torch = G.require_gpu()
    bh, n_q, n_k = (40 if d <= 64 else 2), 333, 250
    q, k, v = G.inputs(f"bwd/stages/{d}", bh, n_q, n_k, d, dtype)
    d_o = synth.tensor(f"bwd/stages/{d}/do", (bh, n_q, d), dtype)
    qd, kd, vd, dod = (G.to_device(x, dtype) for x in (q, k, v, d_o))
    scale = 1 / math.sqrt(d)
    o = G.empty((bh, n_q, d), dtype)
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    code = {"bf16": binding.DTYPE_BF16, "f16": binding.DTYPE_F16}[dtype]
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n_q, n_k, d, code), dtype=torch.uint8, device="cuda")
    whole = [G.empty(x.shape, dtype) for x in (q, k, v)]
    binding.fa2_backward(qd, kd, vd, o, dod, lse, *whole, ws, scale)
    small = torch.empty(8 * bh * 384, dtype=torch.uint8, device="cuda")  # D and LSE2 only
    assert one_pass(bh, n_k, d) == (d <= 64)
    staged = _stages(qd, kd, vd, o, dod, lse, scale, small, dtype)
    again = _stages(qd, kd, vd, o, dod, lse, scale, small, dtype)
    one_grid = [G.empty(tuple(x.shape), dtype) for x in (qd, kd, vd)]
    binding.fa2_backward_preprocess(o, dod, lse, small, n_k)
    binding.fa2_backward_passes(qd, kd, vd, dod, small, *one_grid, scale)
    binding.fa2_device_status()
    for name, a, b in zip(("dQ", "dK", "dV"), staged, one_grid):
        assert torch.equal(a, b), f"fa2_backward_passes {name} differs from _dkdv + _dq"
    w = lambda x: synth.widen(x, dtype)
    ref = A.backward(w(q), w(k), w(v), w(d_o), scale)
    for name, a, b, c, r in zip(("dQ", "dK", "dV"), staged, whole, again, ref):
        check_16bit(G.to_f64(a), r, f"two-pass {name}")
        assert torch.equal(a, c), f"two-pass {name} not reproducible"
        if not one_pass(bh, n_k, d):
            assert torch.equal(a, b), f"fa2_backward {name} differs from its stages"
        else:
            check_16bit(G.to_f64(a), G.to_f64(b), f"two-pass vs one-pass {name}")


@pytest.mark.parametrize("d", [64, 128])
def test_backward_reproducibility(d):
    """head_dim > 64 (two passes): every gradient is bit-reproducible.  head_dim <= 64 (one
    pass): dK and dV are; dQ is a float32 sum of per-key-tile partial sums added in arrival
    order, so two runs may differ by the reordering of that sum (`check_reordered_sum`: one
    unit in the last place of the 16-bit result, plus 2^-16 of the largest |dQ| where the
    partials cancel) (80 heads at head size 64, for the one-pass kernel)."""
    bh, n = (80 if d <= 64 else 2), 300
    assert one_pass(bh, n, d) == (d <= 64)
    q, k, v = G.inputs(f"bwd/det/{d}", bh, n, n, d, "bf16")
    d_o = synth.tensor(f"bwd/det/{d}/do", (bh, n, d), "bf16")
    a = run_fwd_bwd(q, k, v, d_o, "bf16", 1 / math.sqrt(d))
    b = run_fwd_bwd(q, k, v, d_o, "bf16", 1 / math.sqrt(d))
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    if d > 64:
        assert np.array_equal(a[0], b[0])
    check_reordered_sum(a[0], b[0])


@pytest.mark.parametrize("d", [64, 128])
def test_backward_far_negative_scores_with_a_partial_key_tile(d):
    """Every score near -110 (LSE near -105): a padded key of the last, partial key tile has
    score 0 and probability exp(0 - LSE), beyond float32; the kernels must keep it out of
    dQ (one-pass head size 64 with its 80 heads, two-pass 128) and stay finite. The keys sit
    near -6.9 in every column and sum_j dS_ij = 0, so dQ is a small difference of large
    terms: the elementwise bound with the rounding scale of its last product, from the
    stored O and LSE the kernels read (tests/tolerance.py)."""
    torch = G.require_gpu()
    bh, n_q, n_k = (80 if d <= 64 else 1), 150, 200
    assert one_pass(bh, n_k, d) == (d <= 64)
    scale = 1 / math.sqrt(d)
    q = synth.to_storage(np.full((bh, n_q, d), 2.0), "bf16")
    k_base = -110.0 / (2.0 * d * scale)
    k = synth.to_storage(k_base + 0.5 * synth.normal(synth.BASE_SEED, f"bwd/farneg/{d}/k", bh * n_k * d).reshape(bh, n_k, d),
                         "bf16")
    v = synth.tensor(f"bwd/farneg/{d}/v", (bh, n_k, d), "bf16")
    d_o = synth.tensor(f"bwd/farneg/{d}/do", (bh, n_q, d), "bf16")
    qd, kd, vd, dod = (G.to_device(x, "bf16") for x in (q, k, v, d_o))
    o = G.empty((bh, n_q, d), "bf16")
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    grads = [G.empty(x.shape, "bf16") for x in (q, k, v)]
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n_q, n_k, d, binding.DTYPE_BF16), dtype=torch.uint8,
                     device="cuda")
    binding.fa2_backward(qd, kd, vd, o, dod, lse, *grads, ws, scale)
    binding.fa2_device_status()
    dq, dk, dv = (G.to_f64(g) for g in grads)
    for x in (dq, dk, dv):
        assert np.all(np.isfinite(x))
    w = lambda x: synth.widen(x, "bf16")  # noqa: E731
    _, lse_exact = A.forward(w(q[:1]), w(k[:1]), w(v[:1]), scale)
    assert np.max(lse_exact) < -89  # exp(-LSE) overflows float32: the regime this test is about
    o_st, l_st = G.to_f64(o), G.to_f64(lse)
    for b in range(bh):
        rq, rk, rv, sq, sk, sv = A.backward_slice(w(q), w(k), w(v), w(d_o), scale, b, o=o_st, lse=l_st,
                                                  rounding_scales=True)
        check_16bit_grad(dq[b], rq, sq, "bf16", f"dQ head {b}")
        check_16bit_grad(dk[b], rk, sk, "bf16", f"dK head {b}")
        check_16bit_grad(dv[b], rv, sv, "bf16", f"dV head {b}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("n_q,n_k", [
    (505, 1147),   # 4 query tiles: 8 key tiles per dK/dV CTA, 9 key tiles -> CTAs of 8 and 1
    (100, 333),    # 1 query tile: 3 key tiles in one CTA (K and V freed right after the first products)
    (200, 2100),   # 2 query tiles: 17 key tiles -> CTAs of 8, 8 and 1
    (100, 4096),   # 1 query tile, 32 key tiles: dQ CTAs first, then 4 dK/dV CTAs of 8 key tiles
])
def test_backward_passes_over_several_key_tiles_equal_the_stages(n_q, n_k, d, dtype):
    """The one-grid passes kernel runs a head's dK/dV in CTAs of several consecutive key tiles
    when the head has few query tiles (at every head size: fa2_backward_passes, and at head
    sizes up to 64 the two-pass fallback of fa2_backward_noalloc); its gradients equal, bit for
    bit, those of the stage entry points (one key tile per dK/dV CTA), and the oracle's.
    The launch takes fewer key tiles per CTA when that would leave fewer dK/dV CTAs than
    SMs, so each shape runs with enough heads to keep the counts in the comments."""
    torch = G.require_gpu()
    n_qt, n_kt = -(-n_q // 128), -(-n_k // 128)
    m = min(8, -(-32 // n_qt))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    bh = max(2, -(-sms // -(-n_kt // m)))
    tag = f"bwd/multikt/{n_q}/{n_k}/{d}/{dtype}"
    q, k, v = G.inputs(tag, bh, n_q, n_k, d, dtype)
    d_o = synth.tensor(tag + "/do", (bh, n_q, d), dtype)
    qd, kd, vd, dod = (G.to_device(x, dtype) for x in (q, k, v, d_o))
    scale = 1 / math.sqrt(d)
    o = G.empty((bh, n_q, d), dtype)
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    code = {"bf16": binding.DTYPE_BF16, "f16": binding.DTYPE_F16}[dtype]
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n_q, n_k, d, code), dtype=torch.uint8, device="cuda")
    staged = _stages(qd, kd, vd, o, dod, lse, scale, ws, dtype)
    one_grid = [G.empty(tuple(x.shape), dtype) for x in (qd, kd, vd)]
    binding.fa2_backward_passes(qd, kd, vd, dod, ws, *one_grid, scale)
    binding.fa2_device_status()
    for name, a, b in zip(("dQ", "dK", "dV"), staged, one_grid):
        assert torch.equal(a, b), f"fa2_backward_passes {name} differs from _dkdv + _dq"
    w = lambda x: synth.widen(x, dtype)
    for b in (0, bh - 1):
        ref = A.backward(w(q[b:b + 1]), w(k[b:b + 1]), w(v[b:b + 1]), w(d_o[b:b + 1]), scale)
        for name, a, r in zip(("dQ", "dK", "dV"), one_grid, ref):
            check_16bit(G.to_f64(a[b]), r[0], f"one-grid {name} of head {b}")


@pytest.mark.parametrize("bh,n_q,n_k,d,dtype", [
    (2, 128, 4096, 128, "bf16"),   # 2 dQ CTAs of 32 key tiles unsplit: 4 ranges of 8
    (3, 200, 2500, 128, "f16"),    # ragged keys (20 key tiles, the last partial): 2 ranges of 10
    (1, 300, 8192, 128, "bf16"),   # 3 query tiles x 8 ranges of 8 key tiles
    (2, 100, 3000, 64, "bf16"),    # head size 64 through the stage entry points: 3 ranges of 8 key tiles
])
def test_backward_split_dq_pass(bh, n_q, n_k, d, dtype):
    """Few query tiles per head and many keys: the dQ pass divides each query tile's keys into
    ranges whose CTAs write float32 partial sums, added in range order by a last kernel, when
    the workspace holds them (fa2_backward_workspace_size bytes).  The gradients are
    bit-reproducible, equal bit for bit between fa2_backward_passes and the stages given the
    same workspace, within the parity bar of the unsplit pass (a workspace without room for
    the partial sums) and of the oracle; nothing is written outside dq, dk, dv or the
    workspace."""
    torch = G.require_gpu()
    splits = dq_key_splits(bh, n_q, n_k)
    assert splits >= 2
    tag = f"bwd/split/{bh}/{n_q}/{n_k}/{d}/{dtype}"
    q, k, v = G.inputs(tag, bh, n_q, n_k, d, dtype)
    d_o = synth.tensor(tag + "/do", (bh, n_q, d), dtype)
    qd, kd, vd, dod = (G.to_device(x, dtype) for x in (q, k, v, d_o))
    scale = 1 / math.sqrt(d)
    o = G.empty((bh, n_q, d), dtype)
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    n_q_pad = -(-n_q // 128) * 128
    hd = 32 if d <= 32 else (64 if d <= 64 else 128)
    ws_bytes = 8 * bh * n_q_pad + splits * bh * n_q_pad * hd * 4
    if d > 64:
        code = {"bf16": binding.DTYPE_BF16, "f16": binding.DTYPE_F16}[dtype]
        assert binding.fa2_backward_workspace_size(bh, n_q, n_k, d, code) == ws_bytes
    ws = G.Guarded((ws_bytes,), torch.uint8)
    runs = []
    for _ in range(2):
        grads = [G.guarded(tuple(x.shape), dtype) for x in (qd, kd, vd)]
        binding.fa2_backward_preprocess(o, dod, lse, ws.t, n_k)
        binding.fa2_backward_passes(qd, kd, vd, dod, ws.t, *(g.t for g in grads), scale)
        runs.append(grads)
    staged = _stages(qd, kd, vd, o, dod, lse, scale, ws.t, dtype)
    small = torch.empty(8 * bh * n_q_pad, dtype=torch.uint8, device="cuda")  # no room for partial sums
    unsplit = _stages(qd, kd, vd, o, dod, lse, scale, small, dtype)
    binding.fa2_device_status()
    ws.assert_intact("workspace")
    for name, a, b, c in zip(("dQ", "dK", "dV"), runs[0], runs[1], staged):
        a.assert_intact(name)
        assert torch.equal(a.t, b.t), f"{name} differs between two runs"
        assert torch.equal(a.t, c), f"fa2_backward_passes {name} differs from the stages"
    check_16bit(G.to_f64(runs[0][0].t), G.to_f64(unsplit[0]), "split dQ against the unsplit pass")
    for name, a, u in zip(("dK", "dV"), runs[0][1:], unsplit[1:]):
        assert torch.equal(a.t, u), f"{name} depends on the dQ split"
    w = lambda x: synth.widen(x, dtype)  # noqa: E731
    ref = A.backward(w(q), w(k), w(v), w(d_o), scale)
    for name, a, r in zip(("dQ", "dK", "dV"), runs[0], ref):
        check_16bit(G.to_f64(a.t), r, f"{name} (dQ pass in {splits} key ranges)")


# (bh, n_q, n_k): many queries, few key tiles; 16 / 8 / 4 / 2 query ranges (8 for the first at
# head size 32; the second has 8 query tiles per range at most, below the 16 a cluster of 16 needs)
DKV_SPLIT_SHAPES = [(2, 32768, 128), (4, 16384, 256), (5, 10200, 600), (40, 2100, 100)]


def test_backward_split_shapes_take_every_cluster_size():
    assert {dkv_query_splits(*s, d) for s in DKV_SPLIT_SHAPES for d in (32, 128)} == {2, 4, 8, 16}


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [32, 40, 64, 72, 128])
@pytest.mark.parametrize("bh,n_q,n_k", DKV_SPLIT_SHAPES)
def test_backward_dkdv_query_ranges_in_a_cluster(dtype, d, bh, n_q, n_k):
    """Queries far outnumbering the keys of few heads: the dK/dV pass splits each key tile's
    queries over a cluster of CTAs that add their dK and dV in distributed shared memory
    (every head size then takes the two passes). dQ, dK, dV against the oracle; two runs
    bit-identical; nothing written outside the gradients."""
    torch = G.require_gpu()
    assert dkv_query_splits(bh, n_q, n_k, d) > 1
    tag = f"bwdsplitq/{dtype}/{d}/{bh}/{n_q}/{n_k}"
    q, k, v = G.inputs(tag, bh, n_q, n_k, d, dtype)
    d_o = synth.tensor(tag + "/do", (bh, n_q, d), dtype)
    scale = 1 / math.sqrt(d)
    qd, kd, vd, dod = (G.to_device(x, dtype) for x in (q, k, v, d_o))
    o = G.empty((bh, n_q, d), dtype)
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    code = {"bf16": binding.DTYPE_BF16, "f16": binding.DTYPE_F16}[dtype]
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n_q, n_k, d, code), dtype=torch.uint8, device="cuda")
    runs = []
    for _ in range(2):
        grads = [G.guarded(tuple(x.shape), dtype) for x in (q, k, v)]
        binding.fa2_backward(qd, kd, vd, o, dod, lse, *(g.t for g in grads), ws, scale)
        info = binding.fa2_last_launch_info()
        assert (info["bwd_one_pass"], info["bwd_dkv_query_ranges"], info["bwd_dq_key_ranges"],
                info["bwd_key_tiles_per_cta"]) == (0, dkv_query_splits(bh, n_q, n_k, d), dq_key_splits(bh, n_q, n_k), 0)
        binding.fa2_device_status()
        for name, g in zip(("dQ", "dK", "dV"), grads):
            g.assert_intact(name)
        runs.append([g.t.clone() for g in grads])
    for name, a, b in zip(("dQ", "dK", "dV"), *runs):
        assert torch.equal(a, b), f"{name} differs between two runs"
    # dK and dV sum over up to 32768 queries (|dK| ~ 10, where a bfloat16 step is 0.04): the
    # elementwise gradient bound, from the stored O and LSE the kernels read
    w = lambda x: synth.widen(x, dtype)  # noqa: E731
    o_st, l_st = G.to_f64(o), G.to_f64(lse)
    got = [G.to_f64(g) for g in runs[0]]
    for b in range(bh):
        rq, rk, rv, sq, sk, sv = A.backward_slice(w(q), w(k), w(v), w(d_o), scale, b, row_chunk=4096, o=o_st,
                                                  lse=l_st, rounding_scales=True)
        check_16bit_grad(got[0][b], rq, sq, dtype, f"dQ head {b}")
        check_16bit_grad(got[1][b], rk, sk, dtype, f"dK head {b}")
        check_16bit_grad(got[2][b], rv, sv, dtype, f"dV head {b}")
    if d == 128 and dtype == "bf16":  # the stage entry points take the same split, bit for bit
        staged = _stages(qd, kd, vd, o, dod, lse, scale, ws, dtype)
        for name, a, b in zip(("dQ", "dK", "dV"), runs[0], staged):
            assert torch.equal(a, b), f"{name}: stages differ from fa2_backward"


@pytest.mark.parametrize("d", [64, 128])
def test_the_most_heads_a_call_takes(d):
    """B·H = 65535, the largest the entry points accept (the kernels take the head from the
    grid's y index, whose limit that is), of 3 queries and 5 keys: forward and backward (at
    head size 64 the one-pass kernel, its float32 dQ accumulator 2.1 GB of workspace; at 128
    the two passes in one grid). The first, a middle and the last head against the oracle."""
    torch = G.require_gpu()
    bh, n_q, n_k = 65535, 3, 5
    tag = f"bwd/maxheads/{d}"
    q, k, v = G.inputs(tag, bh, n_q, n_k, d, "bf16")
    d_o = synth.tensor(tag + "/do", (bh, n_q, d), "bf16")
    qd, kd, vd, dod = (G.to_device(x, "bf16") for x in (q, k, v, d_o))
    scale = 1 / math.sqrt(d)
    o = G.empty((bh, n_q, d), "bf16")
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    grads = [G.empty(tuple(x.shape), "bf16") for x in (q, k, v)]
    ws = torch.empty(binding.fa2_backward_workspace_size(bh, n_q, n_k, d, binding.DTYPE_BF16), dtype=torch.uint8,
                     device="cuda")
    binding.fa2_backward(qd, kd, vd, o, dod, lse, *grads, ws, scale)
    assert binding.fa2_last_launch_info()["bwd_one_pass"] == (1 if one_pass(bh, n_k, d) else 0) == (d <= 64)
    binding.fa2_device_status()
    w = lambda x: synth.widen(x, "bf16")  # noqa: E731
    o_st, l_st = G.to_f64(o), G.to_f64(lse)
    dq, dk, dv = (G.to_f64(g) for g in grads)
    for b in (0, bh // 2, bh - 1):
        one = slice(b, b + 1)
        o_ref, l_ref = A.forward(w(q[one]), w(k[one]), w(v[one]), scale)
        check_16bit(o_st[b], o_ref[0], f"O head {b}")
        check_lse(l_st[b], l_ref[0], f"LSE head {b}")
        rq, rk, rv, sq, sk, sv = A.backward_slice(w(q[one]), w(k[one]), w(v[one]), w(d_o[one]), scale, 0,
                                                  o=o_st[one], lse=l_st[one], rounding_scales=True)
        check_16bit_grad(dq[b], rq, sq, "bf16", f"dQ head {b}")
        check_16bit_grad(dk[b], rk, sk, "bf16", f"dK head {b}")
        check_16bit_grad(dv[b], rv, sv, "bf16", f"dV head {b}")
