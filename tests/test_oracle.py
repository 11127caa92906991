"""Pins for the CPU oracle: it is checked against things other than itself.

* brute force on tiny inputs (pure-Python loops, no max shift, exact-sum fsum);
* the worked examples the pages print (tests/golden/);
* closed forms and invariants of softmax attention;
* library routines the special cases reduce to (scipy softmax / logsumexp);
* central finite differences of L = sum(O * dO) for every input element;
* element-by-element index loops for the PSA rearrangements;
* planted mistakes: mutated copies of the oracle must fail at least one pin.
"""
import math

import numpy as np
import pytest
from scipy import special

from oracle import attention as A
from oracle import psa as P
from tests.golden.load import load
from attention_fa2_forward_02_gb300 import synth


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# --------------------------------------------------------------------------- forward pins

def brute_forward(q, k, v, scale):
    """Independent formulation: exp of raw scores (no max shift), fsum, explicit loops."""
    bh, nq, d = q.shape
    nk = k.shape[1]
    o = np.zeros((bh, nq, v.shape[2]))
    lse = np.zeros((bh, nq))
    for b in range(bh):
        for i in range(nq):
            e = [math.exp(scale * math.fsum(q[b, i, t] * k[b, j, t] for t in range(d))) for j in range(nk)]
            z = math.fsum(e)
            lse[b, i] = math.log(z)
            for t in range(v.shape[2]):
                o[b, i, t] = math.fsum(e[j] * v[b, j, t] for j in range(nk)) / z
    return o, lse


def pin_brute(fwd):
    q, k, v = _rand((2, 3, 4), 1), _rand((2, 5, 4), 2), _rand((2, 5, 4), 3)
    o, lse = fwd(q, k, v, 0.5)
    ob, lb = brute_forward(q, k, v, 0.5)
    return np.allclose(o, ob, atol=1e-12, rtol=0) and np.allclose(lse, lb, atol=1e-12, rtol=0)


def pin_golden_one(fwd):
    g = load("seq_len_one.txt")
    q = np.array(g["q"]).reshape(1, 1, 4)
    k = np.array(g["k"]).reshape(1, 1, 4)
    v = np.array(g["v"]).reshape(1, 1, 4)
    o, lse = fwd(q, k, v, g["scale"])
    return np.array_equal(o.ravel(), np.array(g["o"])) and lse.ravel()[0] == g["lse"]


def pin_golden_const(fwd):
    g = load("constant_rows.txt")
    nq, nk, d = int(g["n_q"]), int(g["n_k"]), int(g["head_dim"])
    q = np.full((1, nq, d), g["fill_q"])
    k = np.full((1, nk, d), g["fill_k"])
    v = np.full((1, nk, d), g["fill_v"])
    o, lse = fwd(q, k, v, g["scale"])
    return np.allclose(o, g["fill_o"], atol=1e-14, rtol=0) and np.allclose(lse, g["lse"], atol=1e-13, rtol=0)


def pin_library_softmax(fwd):
    """N_q rows against scipy's softmax-weighted average and logsumexp."""
    q, k, v = _rand((3, 6, 8), 4), _rand((3, 9, 8), 5), _rand((3, 9, 5), 6)
    scale = 1 / math.sqrt(8)
    o, lse = fwd(q, k, v, scale)
    s = scale * np.einsum("bid,bjd->bij", q, k)
    w = special.softmax(s, axis=-1)
    return (np.allclose(o, np.einsum("bij,bjd->bid", w, v), atol=1e-13, rtol=0)
            and np.allclose(lse, special.logsumexp(s, axis=-1), atol=1e-13, rtol=0))


def pin_shift_invariance(fwd):
    """Adding u to every key row leaves O unchanged and moves LSE_i by scale*q_i.u."""
    q, k, v = _rand((2, 4, 6), 7), _rand((2, 7, 6), 8), _rand((2, 7, 6), 9)
    u = _rand((6,), 10)
    scale = 0.3
    o0, l0 = fwd(q, k, v, scale)
    o1, l1 = fwd(q, k + u, v, scale)
    return np.allclose(o0, o1, atol=1e-12, rtol=0) and np.allclose(l1 - l0, scale * (q @ u), atol=1e-12, rtol=0)


def pin_identical_keys(fwd):
    """Identical K rows: O = mean(V), LSE_i = ln N_k + scale*q_i.k."""
    q, v = _rand((2, 4, 6), 11), _rand((2, 9, 6), 12)
    krow = _rand((2, 1, 6), 13)
    k = np.repeat(krow, 9, axis=1)
    scale = 0.4
    o, lse = fwd(q, k, v, scale)
    want_l = math.log(9) + scale * np.einsum("bid,bd->bi", q, krow[:, 0])
    return (np.allclose(o, v.mean(axis=1, keepdims=True), atol=1e-13, rtol=0)
            and np.allclose(lse, want_l, atol=1e-13, rtol=0))


FORWARD_PINS = [pin_brute, pin_golden_one, pin_golden_const, pin_library_softmax,
                pin_shift_invariance, pin_identical_keys]


@pytest.mark.parametrize("pin", FORWARD_PINS, ids=lambda f: f.__name__)
def test_forward_pins(pin):
    assert pin(A.forward)


def test_forward_invariants_random():
    q, k, v = _rand((2, 33, 16), 20), _rand((2, 47, 16), 21), _rand((2, 47, 16), 22)
    scale = 0.25
    o, lse = A.forward(q, k, v, scale)
    s = A.scores(q, k, scale)
    # LSE_i lies in [max_j s_ij, max_j s_ij + ln N_k]
    mx = s.max(-1)
    assert np.all(lse >= mx - 1e-12) and np.all(lse <= mx + math.log(47) + 1e-12)
    # rows of P sum to one and P is non-negative
    p = A.probabilities(q, k, scale)
    assert np.allclose(p.sum(-1), 1.0, atol=1e-14) and np.all(p >= 0)
    # constant V gives that constant
    oc, _ = A.forward(q, k, np.full_like(v, -1.75), scale)
    assert np.allclose(oc, -1.75, atol=1e-14)
    # permuting keys and values together changes nothing
    perm = np.random.default_rng(3).permutation(47)
    op, lp = A.forward(q, k[:, perm], v[:, perm], scale)
    assert np.allclose(op, o, atol=1e-13) and np.allclose(lp, lse, atol=1e-13)
    # a single key passes V through with LSE equal to the score
    o1, l1 = A.forward(q, k[:, :1], v[:, :1], scale)
    assert np.allclose(o1, np.broadcast_to(v[:, :1], o1.shape), atol=1e-15)
    assert np.allclose(l1, s[:, :, 0], atol=1e-14)


def test_forward_page_fixtures_brute():
    """The trig / linear fixtures of the vyre-libs unit tests, oracle vs brute force."""
    n, d = 8, 16
    i = np.arange(n * d, dtype=np.float64)
    q = (np.sin(i * 0.13) - 0.5).reshape(1, n, d)
    k = (np.cos(i * 0.07) + 0.25).reshape(1, n, d)
    v = (np.sin(i * 0.19) * 2.0).reshape(1, n, d)
    o, lse = A.forward(q, k, v, 1 / math.sqrt(d))
    ob, lb = brute_forward(q, k, v, 1 / math.sqrt(d))
    assert np.allclose(o, ob, atol=1e-12) and np.allclose(lse, lb, atol=1e-12)
    for n, d, a, b, c in [(4, 8, (0.1, 0.0), (0.05, 0.2), (0.3, -0.1)), (5, 8, (0.11, 0.0), (0.06, 0.15), (0.25, -0.05))]:
        i = np.arange(n * d, dtype=np.float64)
        q = (i * a[0] + a[1]).reshape(1, n, d)
        k = (i * b[0] + b[1]).reshape(1, n, d)
        v = (i * c[0] + c[1]).reshape(1, n, d)
        o, lse = A.forward(q, k, v, 1 / math.sqrt(d))
        ob, lb = brute_forward(q, k, v, 1 / math.sqrt(d))
        assert np.allclose(o, ob, rtol=1e-12, atol=1e-12) and np.allclose(lse, lb, rtol=1e-13)


def test_forward_rows_matches_full():
    q, k, v = _rand((3, 20, 8), 30), _rand((3, 25, 8), 31), _rand((3, 25, 8), 32)
    o, lse = A.forward(q, k, v, 0.35)
    rows = [0, 7, 19]
    orow, lrow = A.forward_rows(q, k, v, 0.35, 2, rows)
    assert np.allclose(orow, o[2, rows], atol=1e-14) and np.allclose(lrow, lse[2, rows], atol=1e-14)


def test_forward_rejects_empty():
    with pytest.raises(ValueError):
        A.forward(np.zeros((1, 0, 4)), np.zeros((1, 3, 4)), np.zeros((1, 3, 4)), 1.0)


# --------------------------------------------------------------------------- backward pins

def _loss(q, k, v, d_o, scale):
    o, _ = A.forward(q, k, v, scale)
    return float(np.sum(o * d_o))


def pin_finite_differences(bwd):
    q, k, v, d_o = _rand((1, 3, 4), 40), _rand((1, 5, 4), 41), _rand((1, 5, 4), 42), _rand((1, 3, 4), 43)
    scale = 0.5
    dq, dk, dv = bwd(q, k, v, d_o, scale)
    h = 1e-6
    ok = True
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            fp = _loss(q, k, v, d_o, scale)
            x[idx] = old - h
            fm = _loss(q, k, v, d_o, scale)
            x[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        ok &= bool(np.allclose(g, num, rtol=1e-6, atol=1e-8))
    return ok


def pin_gradient_closed_forms(bwd):
    q, k, v, d_o = _rand((2, 6, 5), 50), _rand((2, 8, 5), 51), _rand((2, 8, 5), 52), _rand((2, 6, 5), 53)
    dq, dk, dv = bwd(q, k, v, d_o, 0.45)
    ok = np.allclose(dk.sum(axis=1), 0.0, atol=1e-12)          # sum_j dS_ij = 0 for every i
    ok &= np.allclose(dv.sum(axis=1), d_o.sum(axis=1), atol=1e-12)  # rows of P sum to one
    # a single key: O = v_0 does not depend on q or k
    dq1, dk1, dv1 = bwd(q, k[:, :1], v[:, :1], d_o, 0.45)
    ok &= np.allclose(dq1, 0, atol=1e-14) and np.allclose(dk1, 0, atol=1e-14)
    ok &= np.allclose(dv1[:, 0], d_o.sum(axis=1), atol=1e-13)
    return bool(ok)


BACKWARD_PINS = [pin_finite_differences, pin_gradient_closed_forms]


@pytest.mark.parametrize("pin", BACKWARD_PINS, ids=lambda f: f.__name__)
def test_backward_pins(pin):
    assert pin(A.backward)


def test_backward_slice_pinned():
    """The chunked per-head backward passes the same pins and matches row chunking of any size."""
    def sliced(q, k, v, d_o, scale):
        outs = [A.backward_slice(q, k, v, d_o, scale, b, row_chunk=2) for b in range(q.shape[0])]
        return tuple(np.stack([o[i] for o in outs]) for i in range(3))
    assert pin_finite_differences(sliced)
    assert pin_gradient_closed_forms(sliced)


def test_backward_slice_from_stored_outputs():
    """backward_slice with the stored O and LSE (what the page's backward kernels read):
    given the exact ones it reproduces the default; a stored LSE larger by c scales every
    gradient by exp(-c) (P = exp(s - LSE)); a stored O whose row sum D is larger by t moves
    dS by -t P, so dQ by -t scale P K and dK by -t scale P^T Q, and leaves dV."""
    q, k, v, d_o = _rand((2, 7, 5), 110), _rand((2, 9, 5), 111), _rand((2, 9, 5), 112), _rand((2, 7, 5), 113)
    scale = 0.41
    o, lse = A.forward(q, k, v, scale)
    for b in range(2):
        base = A.backward_slice(q, k, v, d_o, scale, b, row_chunk=3)
        same = A.backward_slice(q, k, v, d_o, scale, b, row_chunk=3, o=o, lse=lse)
        for x, y in zip(base, same):
            assert np.allclose(x, y, atol=1e-13)
        c = 0.7
        shifted = A.backward_slice(q, k, v, d_o, scale, b, row_chunk=4, o=o, lse=lse + c)
        for x, y in zip(base, shifted):
            assert np.allclose(y, x * math.exp(-c), atol=1e-13)
        t = 0.3
        o2 = o + t * d_o / np.sum(d_o * d_o, axis=-1, keepdims=True)  # D_i + t for every row
        moved = A.backward_slice(q, k, v, d_o, scale, b, row_chunk=2, o=o2, lse=lse)
        p = A.probabilities(q[b:b + 1], k[b:b + 1], scale)[0]
        assert np.allclose(moved[0], base[0] - t * scale * p @ k[b], atol=1e-12)
        assert np.allclose(moved[1], base[1] - t * scale * p.T @ q[b], atol=1e-12)
        assert np.allclose(moved[2], base[2], atol=1e-13)


def test_repeated_keys_reduce_to_the_distinct_ones():
    """Keys repeated c times (key j a copy of key j mod P): the oracle on all c*P keys gives
    the P-key O and dQ, the P-key LSE + ln c, and the P-key dK, dV over c for every copy,
    including the rounding scales (dQ's over sqrt(c)). The large-size GPU test checks the
    kernels through this reduction."""
    n_p, c = 7, 5
    q, d_o = _rand((1, 6, 4), 118), _rand((1, 6, 4), 119)
    kp, vp = _rand((1, n_p, 4), 120), _rand((1, n_p, 4), 121)
    k, v = np.tile(kp, (1, c, 1)), np.tile(vp, (1, c, 1))
    scale = 0.53
    o_p, l_p = A.forward(q, kp, vp, scale)
    o, lse = A.forward(q, k, v, scale)
    assert np.allclose(o, o_p, atol=1e-13) and np.allclose(lse, l_p + math.log(c), atol=1e-13)
    full = A.backward_slice(q, k, v, d_o, scale, 0, row_chunk=4, rounding_scales=True)
    red = A.backward_slice(q, kp, vp, d_o, scale, 0, row_chunk=4, rounding_scales=True)
    assert np.allclose(full[0], red[0], atol=1e-13)
    assert np.allclose(full[3], red[3] / math.sqrt(c), atol=1e-13)
    for j in range(n_p * c):
        for x, y in ((full[1], red[1]), (full[2], red[2]), (full[4], red[4]), (full[5], red[5])):
            assert np.allclose(c * x[j], y[j % n_p], atol=1e-13)


def test_backward_slice_rounding_scales_brute():
    """The root-sum-square scales of the last products, against explicit loops with fsum."""
    q, k, v, d_o = _rand((1, 4, 3), 114), _rand((1, 5, 3), 115), _rand((1, 5, 3), 116), _rand((1, 4, 3), 117)
    scale = 0.6
    o, lse = A.forward(q, k, v, scale)
    out = A.backward_slice(q, k, v, d_o, scale, 0, row_chunk=3, rounding_scales=True)
    assert len(out) == 6
    p = A.probabilities(q, k, scale)[0]
    dmat = A.bwd_preprocess(o, d_o)[0]
    ds = [[p[i, j] * (math.fsum(d_o[0, i, t] * v[0, j, t] for t in range(3)) - dmat[i]) for j in range(5)] for i in range(4)]
    for i in range(4):
        for c in range(3):
            want = scale * math.sqrt(math.fsum((ds[i][j] * k[0, j, c]) ** 2 for j in range(5)))
            assert abs(out[3][i, c] - want) <= 1e-12
    for j in range(5):
        for c in range(3):
            want_k = scale * math.sqrt(math.fsum((ds[i][j] * q[0, i, c]) ** 2 for i in range(4)))
            want_v = math.sqrt(math.fsum((p[i, j] * d_o[0, i, c]) ** 2 for i in range(4)))
            assert abs(out[4][j, c] - want_k) <= 1e-12 and abs(out[5][j, c] - want_v) <= 1e-12
    # the gradients themselves are the default ones
    for x, y in zip(out[:3], A.backward_slice(q, k, v, d_o, scale, 0)):
        assert np.allclose(x, y, atol=1e-14)


def test_psa_backward_finite_differences():
    """Gradient of L = sum(O_lo * dO_lo) + sum(O_hi * dO_hi) w.r.t. every element of the packed buffer."""
    packed = _rand((4, 1, 4, 3), 95)
    d_lo, d_hi = _rand((1, 4, 3), 96), _rand((1, 4, 3), 97)
    scale = 0.6

    def loss(pk):
        o_lo, _ = A.forward(pk[0], pk[1], pk[2], scale)
        o_hi, _ = A.forward(pk[0], pk[1], pk[3], scale)
        return float(np.sum(o_lo * d_lo) + np.sum(o_hi * d_hi))

    g = A.psa_backward(packed, d_lo, d_hi, scale)
    h = 1e-6
    num = np.zeros_like(packed)
    for idx in np.ndindex(packed.shape):
        old = packed[idx]
        packed[idx] = old + h
        fp = loss(packed)
        packed[idx] = old - h
        fm = loss(packed)
        packed[idx] = old
        num[idx] = (fp - fm) / (2 * h)
    assert np.allclose(g, num, rtol=1e-6, atol=1e-8)


def test_psa_backward_null_control():
    """With dO_hi = 0 the V_hi call contributes nothing: sections 0-2 are the plain backward of
    (Q, K, V_lo) and section 3 is zero; symmetrically with dO_lo = 0.  A version that let the
    hi call's gradient leak into section 2, or dropped the lo call's dQ / dK from the sums,
    fails one of the two."""
    packed = _rand((4, 2, 5, 3), 98)
    d_lo, d_hi = _rand((2, 5, 3), 99), _rand((2, 5, 3), 100)
    scale = 0.55
    g = A.psa_backward(packed, d_lo, np.zeros_like(d_hi), scale)
    dq, dk, dv = A.backward(packed[0], packed[1], packed[2], d_lo, scale)
    assert np.allclose(g[0], dq, atol=1e-14) and np.allclose(g[1], dk, atol=1e-14)
    assert np.allclose(g[2], dv, atol=1e-14) and np.all(g[3] == 0)
    g = A.psa_backward(packed, np.zeros_like(d_lo), d_hi, scale)
    dq, dk, dv = A.backward(packed[0], packed[1], packed[3], d_hi, scale)
    assert np.allclose(g[0], dq, atol=1e-14) and np.allclose(g[1], dk, atol=1e-14)
    assert np.all(g[2] == 0) and np.allclose(g[3], dv, atol=1e-14)


def test_preprocess_loop():
    o, d_o = _rand((2, 3, 5), 60), _rand((2, 3, 5), 61)
    want = np.array([[math.fsum(o[b, i, t] * d_o[b, i, t] for t in range(5)) for i in range(3)] for b in range(2)])
    assert np.allclose(A.bwd_preprocess(o, d_o), want, atol=1e-15)


# --------------------------------------------------------------------------- planted mistakes

def _mut_no_scale(q, k, v, scale):
    return A.forward(q, k, v, 1.0)


def _mut_lse_without_max(q, k, v, scale):
    o, lse = A.forward(q, k, v, scale)
    return o, lse - A.scores(q, k, scale).max(-1)


def _mut_transposed_value(q, k, v, scale):
    o, lse = A.forward(q, k, v, scale)
    return o[..., ::-1], lse


def _mut_log2(q, k, v, scale):
    o, lse = A.forward(q, k, v, scale)
    return o, lse / math.log(2)


def _mut_k_dim_swap(q, k, v, scale):
    return A.forward(q, k[..., ::-1], v, scale)


@pytest.mark.parametrize("mutant", [_mut_no_scale, _mut_lse_without_max, _mut_transposed_value, _mut_log2, _mut_k_dim_swap],
                         ids=lambda f: f.__name__)
def test_forward_mutants_fail_a_pin(mutant):
    assert not all(pin(mutant) for pin in FORWARD_PINS)


def _bmut_sign(q, k, v, d_o, scale):
    dq, dk, dv = A.backward(q, k, v, d_o, scale)
    return dq, -dk, dv


def _bmut_no_d(q, k, v, d_o, scale):
    o, lse = A.forward(q, k, v, scale)
    p = np.exp(A.scores(q, k, scale) - lse[..., None])
    ds = p * (d_o @ np.swapaxes(v, -1, -2))
    return scale * ds @ k, scale * np.swapaxes(ds, -1, -2) @ q, np.swapaxes(p, -1, -2) @ d_o


def _bmut_missing_scale(q, k, v, d_o, scale):
    dq, dk, dv = A.backward(q, k, v, d_o, scale)
    return dq / scale, dk, dv


def _bmut_dv_untransposed(q, k, v, d_o, scale):
    dq, dk, dv = A.backward(q, k, v, d_o, scale)
    o, lse = A.forward(q, k, v, scale)
    return dq, dk, dv[:, ::-1]


@pytest.mark.parametrize("mutant", [_bmut_sign, _bmut_no_d, _bmut_missing_scale, _bmut_dv_untransposed],
                         ids=lambda f: f.__name__)
def test_backward_mutants_fail_a_pin(mutant):
    assert not all(pin(mutant) for pin in BACKWARD_PINS)


# --------------------------------------------------------------------------- PSA pins

def _brute_pack(qkv, nh):
    b_, qkv_h, hh, ww = qkv.shape
    kd = qkv_h // (4 * nh)
    out = np.zeros((4, b_ * nh, hh * ww, kd), dtype=qkv.dtype)
    for s in range(4):
        for bh in range(b_ * nh):
            for n in range(hh * ww):
                for dd in range(kd):
                    b, h = divmod(bh, nh)
                    out[s, bh, n, dd] = qkv[b, h * 4 * kd + s * kd + dd, n // ww, n % ww]
    return out


def _brute_merge(lo, hi, b_, nh, hh, ww):
    kd = lo.shape[2]
    out = np.zeros((b_, nh * 2 * kd, hh, ww), dtype=lo.dtype)
    for bh in range(b_ * nh):
        for n in range(hh * ww):
            for dd in range(kd):
                b, h = divmod(bh, nh)
                out[b, h * 2 * kd + dd, n // ww, n % ww] = lo[bh, n, dd]
                out[b, h * 2 * kd + kd + dd, n // ww, n % ww] = hi[bh, n, dd]
    return out


@pytest.mark.parametrize("b_,nh,kd,hh,ww", [(2, 2, 4, 3, 5), (1, 3, 2, 1, 1), (3, 1, 8, 2, 7)])
def test_psa_pack_merge_brute(b_, nh, kd, hh, ww):
    qkv = synth.counter_u16("pin_qkv", (b_, nh * 4 * kd, hh, ww))
    packed = P.pack_qkv(qkv, nh)
    assert packed.dtype == np.uint16 and np.array_equal(packed, _brute_pack(qkv, nh))
    lo = synth.counter_u16("pin_lo", (b_ * nh, hh * ww, kd))
    hi = synth.counter_u16("pin_hi", (b_ * nh, hh * ww, kd))
    merged = P.merge_attn_nchw(lo, hi, b_, nh, hh, ww)
    assert np.array_equal(merged, _brute_merge(lo, hi, b_, nh, hh, ww))
    # round trip: merging the V_lo / V_hi sections of a pack gives the V channels of QKV
    rt = P.merge_attn_nchw(packed[2], packed[3], b_, nh, hh, ww)
    assert np.array_equal(rt, P.extract_v_nchw(qkv, nh))
    ev = np.zeros_like(rt)
    for b in range(b_):
        for h in range(nh):
            for dd in range(kd):
                ev[b, h * 2 * kd + dd] = qkv[b, h * 4 * kd + 2 * kd + dd]
                ev[b, h * 2 * kd + kd + dd] = qkv[b, h * 4 * kd + 3 * kd + dd]
    assert np.array_equal(rt, ev)


def test_psa_adjoints():
    """<pack(x), y> = <x, pack^T(y)> and the same for merge (dot-product test)."""
    b_, nh, kd, hh, ww = 2, 3, 4, 3, 2
    x = _rand((b_, nh * 4 * kd, hh, ww), 70)
    y = _rand((4, b_ * nh, hh * ww, kd), 71)
    assert np.isclose(np.sum(P.pack_qkv(x, nh) * y), np.sum(x * P.pack_qkv_backward(y, b_, nh, hh, ww)), rtol=1e-12)
    lo, hi = _rand((b_ * nh, hh * ww, kd), 72), _rand((b_ * nh, hh * ww, kd), 73)
    g = _rand((b_, nh * 2 * kd, hh, ww), 74)
    dlo, dhi = P.merge_attn_backward(g, nh)
    assert np.isclose(np.sum(P.merge_attn_nchw(lo, hi, b_, nh, hh, ww) * g), np.sum(lo * dlo) + np.sum(hi * dhi), rtol=1e-12)


def test_psa_adjoint_maps_brute():
    """pack^T and merge^T as element loops on raw 16-bit words; extract_v^T on exact values."""
    b_, nh, kd, hh, ww = 2, 2, 4, 3, 5
    n = hh * ww
    d_packed = synth.counter_u16("pin/dpacked", (4, b_ * nh, n, kd))
    got = P.pack_qkv_backward(d_packed, b_, nh, hh, ww)
    assert got.dtype == np.uint16
    for s in range(4):
        for bh in range(b_ * nh):
            b, h = divmod(bh, nh)
            for t in range(n):
                for dd in range(kd):
                    assert got[b, h * 4 * kd + s * kd + dd, t // ww, t % ww] == d_packed[s, bh, t, dd]
    d_merged = synth.counter_u16("pin/dmerged", (b_, nh * 2 * kd, hh, ww))
    d_lo, d_hi = P.merge_attn_backward(d_merged, nh)
    for bh in range(b_ * nh):
        b, h = divmod(bh, nh)
        for t in range(n):
            for dd in range(kd):
                assert d_lo[bh, t, dd] == d_merged[b, h * 2 * kd + dd, t // ww, t % ww]
                assert d_hi[bh, t, dd] == d_merged[b, h * 2 * kd + kd + dd, t // ww, t % ww]
    # extract_v^T: exact sums of small integers survive every rounding, other channels untouched
    qkv = np.arange(b_ * nh * 4 * kd * n, dtype=np.float64).reshape(b_, nh * 4 * kd, hh, ww) % 7
    dv = (np.arange(b_ * nh * 2 * kd * n, dtype=np.float64).reshape(b_, nh * 2 * kd, hh, ww) % 5) - 2
    for dt in ("f32", "f16", "bf16"):
        store = (lambda x: P._round_f64(x, dt))
        out = P._words_to_f64(P.extract_v_backward(store(dv), store(qkv), nh, dt), dt)
        want = qkv.copy()
        for b in range(b_):
            for h in range(nh):
                for t in range(2 * kd):
                    want[b, h * 4 * kd + 2 * kd + t] += dv[b, h * 2 * kd + t]
        assert np.array_equal(out, want)


def test_psa_extract_v_backward_is_the_adjoint():
    """<extract_v(x), y> = <x, extract_v^T(y)> on exact values (extract_v^T applied to a zero d_qkv)."""
    b_, nh, kd, hh, ww = 2, 3, 2, 2, 3
    x = _rand((b_, nh * 4 * kd, hh, ww), 80)
    y = _rand((b_, nh * 2 * kd, hh, ww), 81)
    lhs = np.sum(P.extract_v_nchw(x, nh) * y)
    back = np.zeros_like(x)
    for h in range(nh):
        back[:, h * 4 * kd + 2 * kd:(h + 1) * 4 * kd] += y[:, h * 2 * kd:(h + 1) * 2 * kd]
    assert np.isclose(lhs, np.sum(x * back), rtol=1e-12)
    # the oracle's accumulating adjoint in float32 storage agrees to float32 rounding
    got = P.extract_v_backward(y.astype(np.float32), np.zeros_like(x, dtype=np.float32), nh, "f32")
    assert np.allclose(got, back, atol=1e-6)


def test_psa_rejects_bad_channels():
    with pytest.raises(ValueError):
        P.pack_qkv(np.zeros((1, 10, 2, 2), np.uint16), 1)


# --------------------------------------------------------------------------- the generator itself

def test_synth_is_deterministic_and_normal():
    a = synth.normal(7, "x", 200001)
    b = synth.normal(7, "x", 200001)
    assert np.array_equal(a, b)
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1) < 0.01
    # counter based: a prefix is the prefix of a longer draw
    assert np.array_equal(synth.normal(7, "x", 1001), a[:1001])
    assert not np.array_equal(synth.normal(7, "y", 1000), a[:1000])


def test_bf16_rounding():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f64(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa wins (1.0); 1 + 3*2^-8 rounds up
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2 ** -6 and back[3] == -2.5
    assert np.all(np.abs(back[:4] - x[:4]) <= np.abs(x[:4]) * 2 ** -8)


# --------------------------------------------------------------------------- the parity bar itself

def test_tolerance_rejects_null_output():
    """A zeroed output must fail the 16-bit bar even where |O| ~ 1e-2 (the full-size regime)."""
    from tests.tolerance import check_16bit
    ref = _rand((64, 32), 90, scale=1e-2)
    with pytest.raises(AssertionError):
        check_16bit(np.zeros_like(ref), ref)
    with pytest.raises(AssertionError):
        check_16bit(ref * 0.9, ref)
    check_16bit(ref + 1e-5, ref)


def _peaked_backward_case(seed):
    """A small peaked problem (keys scaled by 8), its stored O / LSE, the oracle's gradients and
    rounding scales, and an emulation of the 16-bit backward on the same stored O / LSE: dS and
    P rounded to bfloat16 before their products, float64 sums, outputs rounded to bfloat16."""
    bh, nq, nk, d = 1, 96, 600, 32
    q = synth.to_storage(_rand((bh, nq, d), seed), "bf16")
    k = synth.to_storage(8.0 * _rand((bh, nk, d), seed + 1), "bf16")
    v = synth.to_storage(_rand((bh, nk, d), seed + 2), "bf16")
    d_o = synth.to_storage(_rand((bh, nq, d), seed + 3), "bf16")
    w = lambda x: synth.widen(x, "bf16")  # noqa: E731
    bfr = lambda x: synth.widen(synth.to_storage(x, "bf16"), "bf16")  # noqa: E731
    scale = 1 / math.sqrt(d)
    o, lse = A.forward(w(q), w(k), w(v), scale)
    o = bfr(o)
    lse = lse.astype(np.float32).astype(np.float64)
    ref = A.backward_slice(w(q), w(k), w(v), w(d_o), scale, 0, o=o, lse=lse, rounding_scales=True)
    qb, kb, vb, dob = w(q)[0], w(k)[0], w(v)[0], w(d_o)[0]
    p = np.exp(scale * qb @ kb.T - lse[0][:, None])
    ds = bfr(p * (dob @ vb.T - np.sum(o[0] * dob, axis=-1, keepdims=True)))
    emu = (bfr(scale * ds @ kb), bfr(scale * ds.T @ qb), bfr(bfr(p).T @ dob))
    return ref, emu


def test_gradient_tolerance_accepts_the_16bit_arithmetic():
    """The bound accepts what rounding dS / P and the outputs to bfloat16 does to the gradients
    of peaked rows, including dQ, whose terms cancel; a bound of 2e-2 + 2^-7 |ref| would not."""
    from tests.tolerance import check_16bit_grad
    ref, emu = _peaked_backward_case(120)
    for g, r, rss in zip(emu, ref[:3], ref[3:]):
        check_16bit_grad(g, r, rss)
    assert np.max(np.abs(ref[0])) > 1.0  # peaked: gradients well above the fixed bar
    assert np.any(np.abs(emu[0] - ref[0]) > 2e-2 + 2.0 ** -7 * np.abs(ref[0]))


def test_gradient_tolerance_accepts_cancelling_terms():
    """Keys near -6.9 in every column (all scores far below zero): sum_j dS_ij = 0, so dQ is a
    small difference of terms about 7 times larger. The 16-bit emulation (dS, P and the outputs
    rounded to bfloat16) passes the bound, whose RMS guard includes u RMS(R); its RMS error is
    above 2^-6 RMS(ref) alone."""
    from tests.tolerance import check_16bit_grad
    bh, nq, nk, d = 1, 96, 300, 64
    scale = 1 / math.sqrt(d)
    rng = np.random.default_rng(123)
    q = synth.to_storage(np.full((bh, nq, d), 2.0) + 0.1 * rng.standard_normal((bh, nq, d)), "bf16")
    k = synth.to_storage(-110.0 / (2.0 * d * scale) + 0.5 * rng.standard_normal((bh, nk, d)), "bf16")
    v = synth.to_storage(rng.standard_normal((bh, nk, d)), "bf16")
    d_o = synth.to_storage(rng.standard_normal((bh, nq, d)), "bf16")
    w = lambda x: synth.widen(x, "bf16")  # noqa: E731
    bfr = lambda x: synth.widen(synth.to_storage(x, "bf16"), "bf16")  # noqa: E731
    o, lse = A.forward(w(q), w(k), w(v), scale)
    o = bfr(o)
    lse = lse.astype(np.float32).astype(np.float64)
    rq, rk, rv, sq, sk, sv = A.backward_slice(w(q), w(k), w(v), w(d_o), scale, 0, o=o, lse=lse, rounding_scales=True)
    qb, kb, vb, dob = w(q)[0], w(k)[0], w(v)[0], w(d_o)[0]
    p = np.exp(scale * qb @ kb.T - lse[0][:, None])
    ds = bfr(p * (dob @ vb.T - np.sum(o[0] * dob, axis=-1, keepdims=True)))
    emu_dq = bfr(scale * ds @ kb)
    check_16bit_grad(emu_dq, rq, sq, "bf16", "emulated dQ")
    check_16bit_grad(bfr(scale * ds.T @ qb), rk, sk, "bf16", "emulated dK")
    check_16bit_grad(bfr(bfr(p).T @ dob), rv, sv, "bf16", "emulated dV")
    rms = lambda x: math.sqrt(float(np.mean(x ** 2)))  # noqa: E731
    assert rms(emu_dq - rq) > 2.0 ** -6 * rms(rq)


def test_gradient_tolerance_on_an_identically_zero_result():
    """One key: dS = P (dP - D) = 0 up to rounding, so dQ and dK vanish and so do their
    rounding scales; the RMS guard still allows 1e-5 (the kernels' D and dP, summed in
    different orders, leave noise near 1e-6) and rejects 1e-4."""
    from tests.tolerance import check_16bit_grad
    q, k, v, d_o = _rand((1, 5, 8), 124), _rand((1, 1, 8), 125), _rand((1, 1, 8), 126), _rand((1, 5, 8), 127)
    rq, rk, rv, sq, sk, sv = A.backward_slice(q, k, v, d_o, 0.3, 0, rounding_scales=True)
    assert max(np.max(np.abs(rq)), np.max(np.abs(rk)), np.max(sq), np.max(sk)) < 1e-12
    check_16bit_grad(rq + 2e-6, rq, sq, "bf16", "dQ with noise")
    with pytest.raises(AssertionError):
        check_16bit_grad(rq + 1e-4, rq, sq, "bf16", "dQ off by 1e-4")
    check_16bit_grad(rv, rv, sv, "bf16", "dV")  # not zero: the usual bound


def test_gradient_tolerance_rejects_errors():
    """Zeroed, 10 %-scaled or biased gradients fail (the RMS guard), and so do a few single
    elements off by 0.1 or by 5 %, although the rest of the array is exact."""
    from tests.tolerance import check_16bit_grad
    ref, emu = _peaked_backward_case(121)
    dq, rss = ref[0], ref[3]
    for bad in (np.zeros_like(dq), dq * 0.9, dq + 0.05 * np.std(dq)):
        with pytest.raises(AssertionError):
            check_16bit_grad(bad, dq, rss)
    allowed = 2e-2 + 2.0 ** -8 * np.abs(dq) + 8 * 2.0 ** -8 * rss
    small = np.argsort(allowed, axis=None)[:3]            # the three tightest elements
    bad = emu[0].copy()
    bad.flat[small] += 0.1
    with pytest.raises(AssertionError):
        check_16bit_grad(bad, dq, rss)
    big = np.unravel_index(int(np.argmax(np.abs(dq) / allowed)), dq.shape)
    bad = emu[0].copy()
    bad[big] = dq[big] * 1.05
    assert abs(bad[big] - dq[big]) > allowed[big]           # a 5 % error there is beyond its allowance
    with pytest.raises(AssertionError):
        check_16bit_grad(bad, dq, rss)


def test_long_accumulation_bound():
    """Recursive float32 summation that truncates each partial sum toward zero (as the
    O accumulator's additions behave over very many key tiles) drifts linearly with the
    number of additions: over 20,000 additions its error stays under n 2^-24 sum|x| and is
    far above the random-walk size sqrt(n) 2^-24 sum|x|. check_16bit_long accepts an error
    within 2e-2 max|ref| + n 2^-24 sum|x| per element and rejects one past it."""
    from tests.tolerance import check_16bit_long
    rng = np.random.default_rng(122)
    x = (rng.standard_normal(20000) * 0.01 + 0.004).astype(np.float32)
    acc = np.float32(0.0)
    for xi in x:
        exact = float(acc) + float(xi)
        r = np.float32(exact)
        if abs(float(r)) > abs(exact):
            r = np.nextafter(r, np.float32(0.0))
        acc = r
    err = abs(float(acc) - math.fsum(float(t) for t in x))
    total = math.fsum(abs(float(t)) for t in x)
    n = len(x)
    assert err <= n * 2.0 ** -24 * total
    assert err > 20 * math.sqrt(n) * 2.0 ** -24 * total
    ref = np.linspace(-0.3, 0.3, 64).reshape(4, 16)
    weighted = np.full_like(ref, 0.8)
    slack = 131079 * 2.0 ** -24 * 0.8
    check_16bit_long(ref + 0.9 * (2e-2 * 0.3 + slack), ref, weighted, 131079, "within")
    with pytest.raises(AssertionError):
        check_16bit_long(ref + 1.1 * (2e-2 * 0.3 + slack), ref, weighted, 131079, "past")
    with pytest.raises(AssertionError):
        check_16bit_long(ref + 1.1 * 2e-2 * 0.3, ref, weighted, 0, "no additions")
