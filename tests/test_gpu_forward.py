"""GPU parity of fa2_forward against the float64 oracle, through the C ABI."""
import math

import numpy as np
import pytest

from attention_fa2_forward_02_gb300 import binding, synth
from oracle import attention as A
from tests import gpu_util as G
from tests.golden.load import load
from tests.split_rules import fwd_key_splits
from tests.tolerance import check_16bit, check_f32, check_lse

pytestmark = pytest.mark.gpu


def run_forward(q, k, v, dtype, scale):
    torch = G.require_gpu()
    bh, n_q, d = q.shape
    qd, kd, vd = G.to_device(q, dtype), G.to_device(k, dtype), G.to_device(v, dtype)
    o = G.empty((bh, n_q, d), dtype)
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    binding.fa2_device_status()
    return G.to_f64(o), G.to_f64(lse)


SHAPES = [
    (2, 300, 400),    # ragged query and key tails, several tiles
    (1, 1, 1),        # a single query and a single key
    (3, 129, 129),    # one past a tile
    (2, 256, 128),    # exactly two query tiles, one key tile
    (1, 520, 77),     # key length below one tile
    (2, 64, 1000),    # queries below one tile, many key tiles
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("bh,n_q,n_k", SHAPES)
def test_forward_tensor_core_vs_oracle(dtype, d, bh, n_q, n_k):
    q, k, v = G.inputs(f"fwd/{dtype}/{d}/{bh}/{n_q}/{n_k}", bh, n_q, n_k, d, dtype)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_forward(q, k, v, dtype, scale)
    o_ref, lse_ref = A.forward(synth.widen(q, dtype), synth.widen(k, dtype), synth.widen(v, dtype), scale)
    check_16bit(o, o_ref, "O")
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("bh,n_q,n_k", [(2, 64, 64), (1, 37, 91), (1, 1, 1)])
def test_forward_f32_vs_oracle(d, bh, n_q, n_k):
    q, k, v = G.inputs(f"fwd32/{d}/{bh}/{n_q}/{n_k}", bh, n_q, n_k, d, "f32")
    scale = 1.0 / math.sqrt(d)
    o, lse = run_forward(q, k, v, "f32", scale)
    o_ref, lse_ref = A.forward(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), scale)
    check_f32(o, o_ref, "O")
    check_f32(lse, lse_ref, "LSE")


def test_forward_tiny_fp32_config():
    """BH=2 (B=1, H=2), N_q=N_k=64, HEAD_DIM=32, float32, scale 1/sqrt(32)."""
    q, k, v = G.inputs("config/tiny_fp32", 2, 64, 64, 32, "f32")
    o, lse = run_forward(q, k, v, "f32", 1 / math.sqrt(32))
    o_ref, lse_ref = A.forward(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), 1 / math.sqrt(32))
    check_f32(o, o_ref, "O")
    check_f32(lse, lse_ref, "LSE")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_forward_page_worked_example(dtype):
    """The single-key example of the vyre-libs unit tests, head_dim zero-padded to 32.

    Zero columns add nothing to q.k, and zero V columns only add zero output
    columns, so the first four outputs must be V itself and LSE = 12.5.
    """
    g = load("seq_len_one.txt")
    pad = lambda x: np.pad(np.array(x, dtype=np.float64).reshape(1, 1, 4), ((0, 0), (0, 0), (0, 28)))
    q, k, v = (synth.to_storage(pad(g[n]), dtype) for n in ("q", "k", "v"))
    o, lse = run_forward(q, k, v, dtype, g["scale"])
    assert np.array_equal(o[0, 0, :4], np.array(g["o"])) and np.all(o[0, 0, 4:] == 0)
    assert abs(lse[0, 0] - g["lse"]) <= 1e-5


def test_forward_constant_rows_example_at_its_own_head_dim():
    """The constant-input example exactly as the page's unit test states it: N = 5,
    head_dim 7 (float32, the only type whose rows need not be 16-byte multiples)."""
    g = load("constant_rows.txt")
    n, d = int(g["n_q"]), int(g["head_dim"])
    q, k, v = (np.full((1, n, d), g[f"fill_{x}"], dtype=np.float32) for x in ("q", "k", "v"))
    o, lse = run_forward(q, k, v, "f32", g["scale"])
    assert np.all(o == g["fill_o"])
    assert np.max(np.abs(lse - g["lse"])) <= 1e-5


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_forward_constant_rows_example(dtype):
    """The constant-input example (q=1, k=0.5, v=2) at GPU head_dim 32 and several tiles of rows."""
    n, d = 300, 32
    q = synth.to_storage(np.full((1, n, d), 1.0), dtype)
    k = synth.to_storage(np.full((1, n, d), 0.5), dtype)
    v = synth.to_storage(np.full((1, n, d), 2.0), dtype)
    scale = 1 / math.sqrt(d)
    o, lse = run_forward(q, k, v, dtype, scale)
    assert np.all(o == 2.0)
    assert np.max(np.abs(lse - (math.log(n) + d * 0.5 * scale))) <= 1e-4


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_forward_invariants(dtype):
    """Constant V gives that constant; identical key rows give mean(V) and LSE = ln N_k + scale q.k."""
    bh, n_q, n_k, d = 2, 200, 333, 64
    q, k, v = G.inputs(f"inv/{dtype}", bh, n_q, n_k, d, dtype)
    scale = 1 / math.sqrt(d)
    vc = synth.to_storage(np.full((bh, n_k, d), -1.25), dtype)
    o, _ = run_forward(q, k, vc, dtype, scale)
    assert np.max(np.abs(o + 1.25)) <= 1e-2
    krow = k[:, :1]
    ks = np.repeat(krow, n_k, axis=1)
    o, lse = run_forward(q, ks, v, dtype, scale)
    check_16bit(o, np.broadcast_to(synth.widen(v, dtype).mean(axis=1, keepdims=True), o.shape), "O (identical keys)")
    want = math.log(n_k) + scale * np.einsum("bid,bd->bi", synth.widen(q, dtype), synth.widen(krow, dtype)[:, 0])
    check_lse(lse, want, "LSE (identical keys)")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_forward_rising_scores_rescale_often(dtype, d):
    """Keys scaled up along the sequence (by 1 + 3 j / 128 for key j), so that each key tile's
    row maximum exceeds the previous one by more than the rescale threshold: the O / l
    rescale of the online softmax runs at nearly every tile, which the N(0, 1) inputs of
    the other tests rarely reach."""
    bh, n_q, n_k = 2, 300, 1000
    q = synth.tensor(f"rise/{d}/q", (bh, n_q, d), dtype)
    ramp = 1.0 + 3.0 * np.arange(n_k, dtype=np.float64) / 128.0
    k = synth.to_storage(synth.normal(synth.BASE_SEED, f"rise/{d}/k", bh * n_k * d).reshape(bh, n_k, d)
                         * ramp[None, :, None], dtype)
    v = synth.tensor(f"rise/{d}/v", (bh, n_k, d), dtype)
    scale = 1 / math.sqrt(d)
    w = lambda x: synth.widen(x, dtype)
    # the regime: tile maxima (log2 units) rise by more than the threshold of 8 on average
    s2 = np.einsum("bid,bjd->bij", w(q), w(k)) * scale / math.log(2.0)
    tile_max = np.stack([s2[:, :, j:j + 128].max(axis=2) for j in range(0, n_k, 128)], axis=2)
    assert np.mean(np.diff(tile_max, axis=2)) > 8.0
    o, lse = run_forward(q, k, v, dtype, scale)
    o_ref, lse_ref = A.forward(w(q), w(k), w(v), scale)
    check_16bit(o, o_ref, "O (rising scores)")
    check_lse(lse, lse_ref, "LSE (rising scores)")


def test_forward_deterministic_and_in_bounds():
    """Two runs agree bit for bit, and nothing is written outside O and LSE (guard bands)."""
    torch = G.require_gpu()
    bh, n_q, n_k, d = 3, 300, 200, 128
    q, k, v = G.inputs("canary", bh, n_q, n_k, d, "bf16")
    qd, kd, vd = (G.to_device(x, "bf16") for x in (q, k, v))
    guard = 4096
    o_buf = torch.full((bh * n_q * d + 2 * guard,), -7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((bh * n_q + 2 * guard,), -7.0, dtype=torch.float32, device="cuda")
    o = o_buf[guard:guard + bh * n_q * d].view(bh, n_q, d)
    lse = l_buf[guard:guard + bh * n_q].view(bh, n_q)
    binding.fa2_forward(qd, kd, vd, o, lse, 1 / math.sqrt(d))
    first = (o.clone(), lse.clone())
    binding.fa2_forward(qd, kd, vd, o, lse, 1 / math.sqrt(d))
    binding.fa2_device_status()
    assert torch.equal(first[0], o) and torch.equal(first[1], lse)
    assert torch.all(o_buf[:guard] == -7.0) and torch.all(o_buf[-guard:] == -7.0)
    assert torch.all(l_buf[:guard] == -7.0) and torch.all(l_buf[-guard:] == -7.0)


def _whole_heads(tag, bh, n_q, n_k, d, k_scale, heads, row_chunk=512):
    """GPU forward of the whole problem; every row of O and LSE of the listed heads against
    the oracle, element by element (the oracle runs on chunks of query rows to bound its memory)."""
    torch = G.require_gpu()
    q, k, v = G.inputs(tag, bh, n_q, n_k, d, "bf16", k_scale=k_scale)
    scale = 1 / math.sqrt(d)
    qd, kd, vd = (G.to_device(x, "bf16") for x in (q, k, v))
    o = G.empty((bh, n_q, d), "bf16")
    lse = torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, scale)
    binding.fa2_device_status()
    o_all, lse_all = G.to_f64(o), G.to_f64(lse)
    assert np.all(np.isfinite(o_all)) and np.all(np.isfinite(lse_all))
    for b in heads:
        w = lambda x: synth.widen(x[b:b + 1], "bf16")  # noqa: E731
        qb, kb, vb = w(q), w(k), w(v)
        o_ref = np.empty((n_q, d))
        l_ref = np.empty(n_q)
        for r0 in range(0, n_q, row_chunk):
            rows = np.arange(r0, min(n_q, r0 + row_chunk))
            o_ref[rows], l_ref[rows] = A.forward_rows(qb, kb, vb, scale, 0, rows)
        check_16bit(o_all[b], o_ref, f"O of head {b}")
        check_lse(lse_all[b], l_ref, f"LSE of head {b}")


def test_forward_full_size_d64_whole_heads():
    """Non-causal bf16 forward, B=4 H=16 (BH=64), N=4096, d=64: every row of O and LSE of the
    first and last heads against the oracle."""
    _whole_heads("config/fwd_d64", 64, 4096, 4096, 64, 1.0, [0, 63])


def test_forward_full_size_d128_whole_heads():
    """bf16 forward, B=2 H=16 (BH=32), N=8192, d=128: every row of O and LSE of the first and
    last heads against the oracle."""
    _whole_heads("config/fwdbwd_d128", 32, 8192, 8192, 128, 1.0, [0, 31])


def test_forward_cross_attention_peaked_whole_heads():
    """B=1 H=32, N_q=1024 vs N_k=32768, d=128, K scaled by 8 (peaked rows): every row of O and
    LSE of the first and last heads against the oracle."""
    _whole_heads("config/cross_k8", 32, 1024, 32768, 128, 8.0, [0, 31], row_chunk=128)


# (bh, n_q, n_k): a query row alone, ragged query and key tails; 16 / 4 / 2 / 4 ranges (8 for
# the first at head size 32: a CTA's 2-column share would not make a 16-byte group)
SPLIT_SHAPES = [(2, 128, 32768), (1, 300, 5000), (3, 200, 2100), (2, 1, 4096)]


def test_forward_split_shapes_take_every_cluster_size():
    sizes = {fwd_key_splits(bh, n_q, n_k, d) for bh, n_q, n_k in SPLIT_SHAPES for d in (32, 128)}
    assert sizes == {2, 4, 8, 16}


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("d", [32, 40, 64, 72, 128])
@pytest.mark.parametrize("bh,n_q,n_k", SPLIT_SHAPES)
def test_forward_key_ranges_in_a_cluster(dtype, d, bh, n_q, n_k):
    """Few query tiles, many keys: the CTAs of a cluster each take a key range of a query-tile
    pair and combine (O, m, l) through distributed shared memory. Every element of O and LSE
    against the oracle; two runs bit-identical; nothing written outside O and LSE."""
    torch = G.require_gpu()
    assert fwd_key_splits(bh, n_q, n_k, d) > 1
    q, k, v = G.inputs(f"fwdsplit/{dtype}/{d}/{bh}/{n_q}/{n_k}", bh, n_q, n_k, d, dtype)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = (G.to_device(x, dtype) for x in (q, k, v))
    runs = []
    for _ in range(2):
        o = G.guarded((bh, n_q, d), dtype)
        lse = G.guarded((bh, n_q), "f32")
        binding.fa2_forward(qd, kd, vd, o.t, lse.t, scale)
        # the library launched the cluster the size rule gives (a GB300 holds every size)
        assert binding.fa2_last_launch_info()["fwd_key_ranges"] == fwd_key_splits(bh, n_q, n_k, d)
        binding.fa2_device_status()
        o.assert_intact("O")
        lse.assert_intact("LSE")
        runs.append((o.t.clone(), lse.t.clone()))
    assert torch.equal(runs[0][0], runs[1][0]) and torch.equal(runs[0][1], runs[1][1])
    o_ref, lse_ref = A.forward(synth.widen(q, dtype), synth.widen(k, dtype), synth.widen(v, dtype), scale)
    check_16bit(G.to_f64(runs[0][0]), o_ref, "O")
    check_lse(G.to_f64(runs[0][1]), lse_ref)


def test_calls_from_other_host_threads():
    """The library works from host threads other than the one that first used CUDA (a thread
    with no current context makes the primary one current before encoding its tensor maps),
    and fa2_last_launch_info describes the calling thread's own calls: two threads, one
    launching a 4-CTA cluster split and one no split, each run a forward and a backward and
    read back their own choices; the outputs match those of the same calls on this thread."""
    import threading

    torch = G.require_gpu()
    shapes = {"split": (1, 300, 5000, 64), "plain": (4, 512, 512, 64)}
    assert fwd_key_splits(*shapes["split"]) == 4 and fwd_key_splits(*shapes["plain"]) == 1
    work = {}
    for name, (bh, n_q, n_k, d) in shapes.items():
        q, k, v = G.inputs(f"fwdthread/{name}", bh, n_q, n_k, d, "bf16")
        d_o = synth.tensor(f"fwdthread/{name}/do", (bh, n_q, d), "bf16")
        ins = [G.to_device(x, "bf16") for x in (q, k, v, d_o)]
        ws = torch.empty(binding.fa2_backward_workspace_size(bh, n_q, n_k, d, binding.DTYPE_BF16), dtype=torch.uint8,
                         device="cuda")
        work[name] = (ins, ws, (bh, n_q, n_k, d))

    def outputs(name):
        (qd, kd, vd, dod), ws, (bh, n_q, n_k, d) = work[name]
        o, lse = G.empty((bh, n_q, d), "bf16"), torch.empty((bh, n_q), dtype=torch.float32, device="cuda")
        binding.fa2_forward(qd, kd, vd, o, lse, 0.125)
        fwd = binding.fa2_last_launch_info()["fwd_key_ranges"]
        grads = [G.empty(tuple(x.shape), "bf16") for x in (qd, kd, vd)]
        binding.fa2_backward(qd, kd, vd, o, dod, lse, *grads, ws, 0.125)
        return fwd, binding.fa2_last_launch_info()["bwd_one_pass"], [o, lse, *grads]

    seen, errors, barrier = {}, [], threading.Barrier(2, timeout=60)

    def run(name):
        try:
            result = outputs(name)
            torch.cuda.synchronize()
        except Exception as e:  # reported below; the other thread must not wait for ever
            errors.append(f"{name}: {e}")
            result = None
        try:
            barrier.wait()  # both threads have launched before either compares
        except threading.BrokenBarrierError:
            pass
        seen[name] = result

    threads = [threading.Thread(target=run, args=(name,)) for name in shapes]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    binding.fa2_device_status()
    for name, want_fwd in (("split", 4), ("plain", 1)):
        fwd, bwd_one_pass, got = seen[name]
        assert fwd == want_fwd and bwd_one_pass == 0  # 1 or 4 heads of few key tiles: two passes
        _, _, here = outputs(name)
        binding.fa2_device_status()
        for a, b in zip(got, here):
            assert torch.equal(a, b), f"{name}: a worker thread's result differs from this thread's"


def test_forward_key_ranges_peaked_rows():
    """Keys scaled by 8 (peaked rows): the key ranges of a pair end with maxima far apart, so
    the combine's rescaling by 2^(m_r - M) carries the result. B·H = 2, N_q = 200, N_k = 33000,
    d = 128, sixteen ranges."""
    G.require_gpu()
    bh, n_q, n_k, d = 2, 200, 33000, 128
    assert fwd_key_splits(bh, n_q, n_k, d) == 16
    q, k, v = G.inputs("fwdsplit/peaked", bh, n_q, n_k, d, "bf16", k_scale=8.0)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_forward(q, k, v, "bf16", scale)
    o_ref, lse_ref = A.forward(synth.widen(q, "bf16"), synth.widen(k, "bf16"), synth.widen(v, "bf16"), scale)
    check_16bit(o, o_ref, "O")
    check_lse(lse, lse_ref)
