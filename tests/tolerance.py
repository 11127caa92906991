"""The parity bar for floating-point outputs, in one place.

Attention outputs (O, dQ, dK, dV) computed from 16-bit inputs with float32
accumulation must be within 2e-2 absolute of the float64 oracle AND within
2e-2 * max|oracle| (the second bound keeps the check meaningful when the
outputs themselves are ~1e-2, where a zero output would pass a bare 2e-2).
The float32 path: 1e-4 absolute.  LSE: 1e-3 absolute.

Gradients larger than 1 (peaked score rows, e.g. keys scaled by 8, give |dQ| ~ 30)
cannot meet a fixed 2e-2: a 16-bit output's own rounding is 2^-9 of its value, 0.06
at 30.  For them the bound is 2e-2 * max(1, max|oracle|), the same as above
wherever max|oracle| <= 1, plus an RMS guard (RMS error <= 2^-6 * RMS of the
oracle) so that the wider bound cannot hide a systematic error.
"""
import numpy as np

ABS_16 = 2e-2
REL_16 = 2e-2
ABS_F32 = 1e-4
ABS_LSE = 1e-3
RMS_16 = 2.0 ** -6


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


def check_f32(got, ref, what="output"):
    err, _ = attention_error(got, ref)
    assert np.all(np.isfinite(got)) and err <= ABS_F32, f"{what}: max|err| = {err:.3e} > {ABS_F32}"


def check_lse(got, ref, what="lse"):
    err, _ = attention_error(got, ref)
    assert np.all(np.isfinite(got)) and err <= ABS_LSE, f"{what}: max|err| = {err:.3e} > {ABS_LSE}"


def check_16bit_grad(got, ref, what="gradient"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err, scale = attention_error(got, ref)
    bound = REL_16 * max(1.0, scale)
    rms_err = float(np.sqrt(np.mean((got - ref) ** 2)))
    rms_ref = float(np.sqrt(np.mean(ref ** 2)))
    ok = np.all(np.isfinite(got)) and err <= bound and rms_err <= RMS_16 * rms_ref
    assert ok, (f"{what}: max|err| = {err:.3e} (bound {bound:.3e}), RMS err = {rms_err:.3e} "
                f"(bound {RMS_16 * rms_ref:.3e}), max|ref| = {scale:.3e}")
