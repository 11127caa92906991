"""The parity bar for floating-point outputs, in one place.

Attention outputs (O, dQ, dK, dV) computed from 16-bit inputs with float32
accumulation must be within 2e-2 absolute of the float64 oracle AND within
2e-2 * max|oracle| (the second bound keeps the check meaningful when the
outputs themselves are ~1e-2, where a zero output would pass a bare 2e-2).
The float32 path: 1e-4 absolute.  LSE: 1e-3 absolute.

Gradients of peaked score rows (keys scaled by 8: |dQ| up to ~30) are checked element
by element against what the arithmetic itself can move them by (`check_16bit_grad`):

    |got - ref| <= 2e-2 + u |ref| + 8 u R,

u the unit roundoff of the 16-bit type (2^-8 bfloat16, 2^-11 float16).  The terms:
2e-2 the fixed bar; u |ref| the rounding of the 16-bit output; 8 u R the rounding of
the 16-bit operand of the gradient's last product (dS for dQ and dK, P for dV), each
term of that sum moved by at most u relative.  R = sqrt(sum of the squared terms) comes
from the oracle (`backward_slice(..., rounding_scales=True)`).  The roundings are
bounded and independent, so by Hoeffding's inequality their sum exceeds 8 u R with
probability below 2 exp(-32) per element; a worst-case bound (u times the sum of the
absolute terms) would be looser by about the square root of the number of keys with
weight.  dQ needs the R term: its terms cancel (sum_j dS_ij = 0), so with keys scaled
by 8 its rounding error is a few percent of a small result, above any fixed fraction
of |ref|.  The test feeds both sides the same stored O and LSE, so that D (from the
16-bit O) agrees: dQ also amplifies an error in D by scale * sum_j P_ij k_j, and no
16-bit O pins D closer than about 2^-8 * sum_d |O_d dO_d|.  An RMS guard on top makes a
scaled, biased or zeroed gradient fail even where each element would pass: RMS error <=
2^-6 * RMS of the oracle + u * RMS(R). The second term is the size of the same operand
roundings over the array (each element's rounding error has a spread of at most u R):
where the terms of a gradient cancel (keys far from zero in every column, sum_j dS_ij =
0) R is much larger than the result, and the roundings alone exceed 2^-6 of its RMS.

Outputs summed over very many key tiles in one float32 accumulator (`check_16bit_long`):
the forward adds one key tile's P V at a time into O (and its row sums into l), so
recursive summation over n tiles can move O_id by up to n * 2^-24 * sum_j P_ij |v_jd|
(the standard bound, (n - 1) u times the sum of the absolute terms, for float32 u), and
the additions that follow the tensor core's accumulation do approach it. That term
is about 1.5e-5 at 256 key tiles; over 131,079 of them (16.8M keys) it reaches about
0.8 % of the absolute weighted sum. The relative bound then becomes
2e-2 * max|ref| + n * 2^-24 * sum_j P_ij |v_jd|, elementwise; the 2e-2 absolute bar stays.
"""
import numpy as np

ABS_16 = 2e-2
REL_16 = 2e-2
ABS_F32 = 1e-4
ABS_LSE = 1e-3
RMS_16 = 2.0 ** -6
UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}
ROUNDING_SIGMAS = 8.0         # Hoeffding: P(sum of roundings > 8 u R) < 2 exp(-32)


def attention_error(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    return err, scale


ZERO_REF_ABS = 1e-5  # when the exact result is identically zero (e.g. dQ, dK with one key)


def check_16bit(got, ref, what="output"):
    err, scale = attention_error(got, ref)
    bound = REL_16 * scale if scale > 0 else ZERO_REF_ABS
    ok = np.all(np.isfinite(got)) and err <= ABS_16 and err <= bound
    assert ok, f"{what}: max|err| = {err:.3e}, max|ref| = {scale:.3e} (bounds {ABS_16} and {REL_16}*max|ref|)"


def check_16bit_long(got, ref, abs_weighted, n_adds, what="output"):
    """The 16-bit bar for an output accumulated over n_adds key tiles in float32:
    max|err| <= 2e-2, and elementwise |err| <= 2e-2 * max|ref| + n_adds * 2^-24 * abs_weighted,
    abs_weighted = sum_j P_ij |v_jd| from the oracle."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err, scale = attention_error(got, ref)
    allowed = REL_16 * scale + n_adds * 2.0 ** -24 * np.asarray(abs_weighted, dtype=np.float64)
    excess = np.abs(got - ref) - allowed
    ok = np.all(np.isfinite(got)) and err <= ABS_16 and np.all(excess <= 0)
    worst = int(np.argmax(excess)) if excess.size else 0
    assert ok, (f"{what}: max|err| = {err:.3e} (bar {ABS_16}); worst element exceeds its bound "
                f"{allowed.flat[worst]:.3e} by {excess.flat[worst]:.3e}")


def check_f32(got, ref, what="output"):
    err, _ = attention_error(got, ref)
    assert np.all(np.isfinite(got)) and err <= ABS_F32, f"{what}: max|err| = {err:.3e} > {ABS_F32}"


def check_lse(got, ref, what="lse"):
    err, _ = attention_error(got, ref)
    assert np.all(np.isfinite(got)) and err <= ABS_LSE, f"{what}: max|err| = {err:.3e} > {ABS_LSE}"


def check_16bit_grad(got, ref, rss, dtype="bf16", what="gradient"):
    """Elementwise |got - ref| <= 2e-2 + u |ref| + 8 u rss, plus the RMS guard; rss is the
    oracle's root-sum-square of the terms of the gradient's last product. The RMS guard
    allows at least 1e-5 (the bar for an exactly zero result, as in check_16bit)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rss = np.asarray(rss, dtype=np.float64)
    u = UNIT_ROUNDOFF[dtype]
    diff = np.abs(got - ref)
    allowed = ABS_16 + u * np.abs(ref) + ROUNDING_SIGMAS * u * rss
    rms_err = float(np.sqrt(np.mean((got - ref) ** 2))) if ref.size else 0.0
    rms_ref = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    rms_rss = float(np.sqrt(np.mean(rss ** 2))) if ref.size else 0.0
    # at least the zero-result bar: an exactly zero gradient (dQ, dK with one key) has
    # RMS(ref) = RMS(R) = 0, and the kernels leave rounding noise near 1e-6 there
    rms_bound = max(RMS_16 * rms_ref + u * rms_rss, ZERO_REF_ABS)
    finite = bool(np.all(np.isfinite(got)))
    over = diff > allowed if finite else np.ones(ref.shape, dtype=bool)
    ok = finite and not np.any(over) and rms_err <= rms_bound
    if not ok:
        worst = np.unravel_index(int(np.argmax(diff - allowed)), ref.shape) if ref.size and finite else ()
        detail = (f"worst element {worst}: got {got[worst]:.5g}, ref {ref[worst]:.5g}, allowed {allowed[worst]:.3e}; "
                  if worst else "")
        raise AssertionError(f"{what}: {int(np.sum(over))} element(s) beyond 2e-2 + u|ref| + 8u*rss; {detail}"
                             f"RMS err = {rms_err:.3e} (bound {rms_bound:.3e}), finite = {finite}")


# Run-to-run agreement of the one-pass backward's dQ (not parity with the oracle): each
# element is a float32 sum of per-key-tile partial sums added in whatever order the CTAs
# reach the accumulator, then rounded to the 16-bit type. Two orders can differ by the
# reordering error of the float32 sum, about (key tiles) 2^-24 times the partials' size, and
# that can move the rounded result by one unit of its last place, or by more where the
# partials cancel to a small result. The bound: one unit of the 16-bit type at the larger of
# the two (2^-7 relative for bfloat16) plus 2^-16 of the tensor's largest magnitude.
def check_reordered_sum(a, b, what="dQ"):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    bound = np.maximum(np.abs(a), np.abs(b)) * 2.0 ** -7 + 2.0 ** -16 * max(float(np.max(np.abs(a))), 1e-30)
    excess = np.abs(a - b) - bound
    if not np.all(excess <= 0):
        i = np.unravel_index(int(np.argmax(excess)), excess.shape)
        raise AssertionError(f"{what}: runs differ by {abs(a[i] - b[i]):.3e} at {i} (bound {bound[i]:.3e})")
