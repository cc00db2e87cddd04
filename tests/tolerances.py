"""Acceptance bounds of the GPU path against the oracle.

MATCH:  |gpu - oracle| <= 2 ulps (of the activation dtype) of the oracle value
        + 1e-3, elementwise; the stored gate/up projections (debug variants)
        equal the oracle's on at least 99.9 % of elements for bf16.
F32:    |gpu - oracle| <= 1e-3 + 8e-3 * |oracle|, elementwise.
Integer and byte results are compared bit for bit.

f16 activations (the bounds are stated for bf16; these are the readings for
f16): the ulp bounds are f16 ulps, and the exact-projection rate is 99 %.  The
f32 accumulator's error is the same whatever the output dtype, but f16's
rounding grid is 8 times finer than bf16's, so the same error moves about 8
times as many sums across a rounding boundary (the bf16 rate of 99.9 % scales
to about 99.2 %).
"""
from __future__ import annotations

import numpy as np

MATCH_ULPS = 2
ABS_TOL = 1e-3
F32_RTOL = 8e-3
EXACT_FRACTION = {"bf16": 0.999, "f16": 0.99}


def bf16_to_f64(h) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits, subnormal floor)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.where(a > 0, np.exp2(e - 7.0), 2.0 ** -133)


def f16_to_f64(h) -> np.ndarray:
    return np.asarray(h, dtype=np.uint16).view(np.float16).astype(np.float64)


def f16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of binary16 numbers at |v| (11 significant bits, subnormal floor)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -14.0)
    return np.where(a > 0, np.exp2(e - 10.0), 2.0 ** -24)


TO_F64 = {"bf16": bf16_to_f64, "f16": f16_to_f64}
ULP = {"bf16": bf16_ulp, "f16": f16_ulp}


def _summary(gpu, ref, bound):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    same = (gpu == ref) | (np.isnan(gpu) & np.isnan(ref))      # also equal infinities
    with np.errstate(invalid="ignore"):
        err = np.where(same, 0.0, np.abs(gpu - ref))
    err = np.where(np.isnan(err), np.inf, err)
    bad = ~(err <= bound)
    n_bad = int(bad.sum())
    info = {"n": int(gpu.size), "n_bad": n_bad, "max_err": float(err.max()) if err.size else 0.0}
    if n_bad:
        idx = np.argwhere(bad.reshape(np.shape(gpu)) if np.ndim(gpu) else bad)[:5]
        info["first_bad"] = [(tuple(int(t) for t in i), float(np.asarray(gpu).reshape(np.shape(gpu))[tuple(i)]),
                              float(np.asarray(ref).reshape(np.shape(ref))[tuple(i)])) for i in idx]
    return n_bad == 0, info


def check_match(gpu_bits, oracle_bits, dtype="bf16"):
    gpu, ref = TO_F64[dtype](gpu_bits), TO_F64[dtype](oracle_bits)
    return _summary(gpu, ref, MATCH_ULPS * ULP[dtype](ref) + ABS_TOL)


def check_f32(gpu_bits, oracle_bits, dtype="bf16"):
    gpu, ref = TO_F64[dtype](gpu_bits), TO_F64[dtype](oracle_bits)
    return _summary(gpu, ref, ABS_TOL + F32_RTOL * np.abs(ref))


def exact_fraction(gpu_bits, oracle_bits) -> float:
    a = np.asarray(gpu_bits, dtype=np.uint16)
    b = np.asarray(oracle_bits, dtype=np.uint16)
    return float((a == b).mean()) if a.size else 1.0


def check_match_with_projections(h_gpu, g_gpu, u_gpu, h_ref, g_ref, u_ref, epilogue, dtype="bf16", exact=None,
                                 bounds=None):
    """MATCH check that accounts for the projections' rounding.

    The GPU accumulates in f32, in another order than the oracle's f64 sum, so
    on a few elements the stored gate or up rounds to the neighbouring value;
    both results are correct.  What is unique is checked:
      * the stored projections (debug variants) equal the oracle's on >= 99.9 %
        of elements; elsewhere each must be a correct rounding of a value within
        the f32 accumulation bound of the exact sum (`exact` = (g64, u64),
        `bounds` = (bound_g, bound_u); without them: within 1 ulp + 1e-3);
      * where both projections equal the oracle's, hidden is within the MATCH
        bound (2 ulps + 1e-3) of the oracle's hidden;
      * elsewhere hidden is within the MATCH bound of the oracle's MATCH
        epilogue applied to the GPU's own (validated) projections;
      * the plain MATCH bound against the oracle's hidden is checked on every
        element: elements past it must be among those whose projections
        flipped, and their count and largest error (in ulps) are reported.  (A
        one-ulp change of the gate g moves silu(g) by about |1/g + 1 - sigma(g)|
        ulps relative, so for g << 0 hidden moves by about |g| of its ulps;
        the epilogue check above is what bounds those elements.)"""
    h_gpu, g_gpu, u_gpu = (np.asarray(a, dtype=np.uint16) for a in (h_gpu, g_gpu, u_gpu))
    h_ref, g_ref, u_ref = (np.asarray(a, dtype=np.uint16) for a in (h_ref, g_ref, u_ref))
    eg, eu = exact if exact is not None else (None, None)
    bg, bu = bounds if bounds is not None else (None, None)
    ok_g, info_g = check_projection(g_gpu, g_ref, dtype, exact=eg, bound=bg)
    ok_u, info_u = check_projection(u_gpu, u_ref, dtype, exact=eu, bound=bu)
    same = (g_gpu == g_ref) & (u_gpu == u_ref)
    ok_same, info_same = check_match(h_gpu[same], h_ref[same], dtype)
    alt = epilogue(g_gpu[~same], u_gpu[~same]) if (~same).any() else np.zeros(0, np.uint16)
    ok_alt, info_alt = check_match(h_gpu[~same], alt, dtype)
    # the plain bound on every element
    gpu, ref = TO_F64[dtype](h_gpu), TO_F64[dtype](h_ref)
    with np.errstate(invalid="ignore"):
        err = np.abs(gpu - ref)
    past = ~(err <= MATCH_ULPS * ULP[dtype](ref) + ABS_TOL) & ~((gpu == ref) | (np.isnan(gpu) & np.isnan(ref)))
    ok_plain = not (past & same).any()
    plain = {"n": int(h_gpu.size), "past_plain_bound": int(past.sum()),
             "max_ulps_past": float(((err - ABS_TOL) / ULP[dtype](ref))[past].max()) if past.any() else 0.0}
    info = {"gate": info_g, "up": info_u, "agreeing": info_same, "flipped": info_alt, "plain": plain,
            "flipped_fraction": float((~same).mean()) if same.size else 0.0}
    return ok_g and ok_u and ok_same and ok_alt and ok_plain, info


MIN_RATE_SAMPLE = 10_000


def check_projection(gpu_bits, oracle_bits, dtype="bf16", exact=None, bound=None):
    """Stored gate/up projection: bit-identical to the correctly rounded sum
    on >= 99.9 % of elements (a rate, enforced on samples of at least
    MIN_RATE_SAMPLE elements: a handful of elements cannot resolve a 0.1 %
    rate; smaller samples report it), and everywhere a valid result:
      * with the exact sums and their accumulation bound: a correct rounding of
        some value within `bound` of `exact`, |gpu - exact| <= bound + ulp/2;
      * without them: within 1 ulp + 1e-3 of the oracle's rounded value (the
        absolute term covers sums that cancel to near zero)."""
    frac = exact_fraction(gpu_bits, oracle_bits)
    gpu, ref = TO_F64[dtype](gpu_bits), TO_F64[dtype](oracle_bits)
    if exact is None:
        ok_close, info = _summary(gpu, ref, ULP[dtype](ref) + ABS_TOL)
    else:
        exact = np.asarray(exact, dtype=np.float64).reshape(np.shape(gpu))
        bound = np.asarray(bound, dtype=np.float64).reshape(np.shape(gpu))
        ok_close, info = _summary(gpu, exact, bound + 0.5 * ULP[dtype](gpu))
        diff = np.asarray(gpu) != np.asarray(ref)
        if diff.any():
            # how far the flipped ones sit from the midpoint, in units of the bound
            mid = 0.5 * (gpu + ref)
            info["flipped_max_dist_over_bound"] = float((np.abs(exact - mid) / bound)[diff].max())
    info["exact_fraction"] = frac
    rate_ok = frac >= EXACT_FRACTION[dtype] or np.size(gpu_bits) < MIN_RATE_SAMPLE
    return (rate_ok and ok_close), info
