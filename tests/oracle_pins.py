"""Checks that pin the CPU oracle to facts outside itself.

Each check takes an ``oracle.OracleLib`` so that the same battery can be run
against the real oracle (tests/test_oracle_pins.py) and against copies with a
planted mistake (tests/test_oracle_mutants.py), which must fail at least one.

Independent references used here, none of which is the oracle's own code:
  * the library float32 -> bf16 and float32 -> binary16 casts (torch), which
    round to nearest even, and numpy's float16 type for decoding binary16;
  * "round to odd" to binary32 followed by that library cast, which gives the
    correctly rounded bf16 of any double because binary32 keeps more than two
    extra bits (Boldo and Melquiond, "Emulation of FMA and correctly rounded
    sums: proved algorithms using rounding to odd", IEEE TC 2008);
  * exact rational arithmetic (fractions.Fraction) for dequantisation and sums;
  * numpy int64 matmul for the integer special case;
  * values worked by hand (tests/golden/hand_2x8.json).
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

from quantized_swiglu_mlp_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
MATCH, F32, DEBUG_GATE, DEBUG_UP = 0, 1, 2, 3


# ----------------------------------------------------------- references ----

def lib_bf16_bits(v32: np.ndarray) -> np.ndarray:
    """Library cast float32 -> bf16 (round to nearest even), as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def round_to_odd_f32(v: float) -> np.float32:
    f = np.float32(v)
    if float(f) == v or not math.isfinite(v):
        return f
    bits = f.view(np.uint32)
    if bits & 1:
        return f
    # f was rounded to an even neighbour: step to the odd neighbour on v's side
    return np.nextafter(f, np.float32(math.copysign(math.inf, v - float(f))), dtype=np.float32)


def ref_bf16(v: float) -> int:
    """Correctly rounded bf16 of a double via round-to-odd + library cast."""
    return int(lib_bf16_bits(np.array([round_to_odd_f32(float(v))], dtype=np.float32))[0])


def bf16_val(h: int) -> float:
    return float(np.array([h << 16], dtype=np.uint32).view(np.float32)[0])


def lib_f16_bits(v32: np.ndarray) -> np.ndarray:
    """Library cast float32 -> IEEE binary16 (round to nearest even), as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32))
    return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)


def ref_f16(v: float) -> int:
    """Correctly rounded binary16 of a double: round to odd in binary32 (13 spare
    bits), then the library cast."""
    return int(lib_f16_bits(np.array([round_to_odd_f32(float(v))], dtype=np.float32))[0])


def f16_val(h: int) -> float:
    return float(np.array([h], dtype=np.uint16).view(np.float16)[0])


REF = {"bf16": (ref_bf16, bf16_val), "f16": (ref_f16, f16_val)}


def ref_round(v: float) -> float:
    return bf16_val(ref_bf16(v))


def ref_codes_from_words(words, n, bits):
    """Unpack by string manipulation of the binary representation (LSB first)."""
    out = []
    pf = 32 // bits
    for w in words:
        s = format(int(w), "032b")[::-1]          # s[j] = bit j
        for c in range(pf):
            out.append(int(s[c * bits:(c + 1) * bits][::-1], 2))
    return out[:n]


def brute_force(case: inputs.Case, variant: int) -> np.ndarray:
    """Dequantise whole matrices with Fractions, then a triple loop (in the
    case's activation dtype)."""
    to_bits, val = REF[case.dtype]
    rnd = lambda v: val(to_bits(v))
    x = [[Fraction(val(int(h))) for h in row] for row in case.x]
    M, H, I = case.M, case.H, case.I

    def deq(qm: inputs.QuantMatrix):
        codes = [ref_codes_from_words(r, H, qm.bits) for r in qm.packed]
        W = []
        for i in range(I):
            row = []
            for k in range(H):
                s = Fraction(val(int(qm.scales[i, k // qm.gs])))
                b = Fraction(val(int(qm.biases[i, k // qm.gs])))
                row.append(Fraction(rnd(float(s * codes[i][k] + b))))
            W.append(row)
        return W

    Wg, Wu = deq(case.gate), deq(case.up)
    out = np.zeros((M, I), dtype=np.uint16)
    for m in range(M):
        for i in range(I):
            g = float(sum(x[m][k] * Wg[i][k] for k in range(H)))
            u = float(sum(x[m][k] * Wu[i][k] for k in range(H)))
            if variant == MATCH:
                gb, ub = rnd(g), rnd(u)
                sig = rnd(1.0 / (1.0 + math.exp(-gb)))
                silu = rnd(gb * sig)
                out[m, i] = to_bits(silu * ub)
            elif variant == F32:
                out[m, i] = to_bits(g * u / (1.0 + math.exp(-g)))
            elif variant == DEBUG_GATE:
                out[m, i] = to_bits(g)
            else:
                out[m, i] = to_bits(u)
    return out


# ------------------------------------------------------------ the pins -----

def pin_bf16_binary32(orc, n=20000, seed=0):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    bits[: n // 4] = (bits[: n // 4] & 0xFFFF0000) | 0x8000        # exact ties
    bits[n // 4: n // 2] = (bits[n // 4: n // 2] & 0xFFFF0000) | 0x7FFF
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) < np.float32(3.0e38))]
    got = orc.bf16_round_array(vals.astype(np.float64))
    want = lib_bf16_bits(vals)
    assert np.array_equal(got, want), "bf16 rounding disagrees with the library cast"


def pin_bf16_double(orc, n=5000, seed=1):
    rng = np.random.default_rng(seed)
    vals = []
    for _ in range(n):
        # a bf16 midpoint nudged by a few double ulps: binary32 would round it
        # to the midpoint itself, so a two-step rounding gives the wrong answer
        h = int(rng.integers(0x0080, 0x7F00))
        lo, hi = bf16_val(h), bf16_val(h + 1)
        mid = (lo + hi) / 2
        for d in (-3, -1, 1, 3):
            vals.append(math.copysign(1.0, rng.standard_normal()) * (mid + d * math.ulp(mid)))
    vals += [1e-40, -3e-39, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 3.3895313892515355e38,
             3.4e38, -1.0, 0.0, 65536.0 + 255.0]
    got = [orc.f64_to_bf16(v) for v in vals]
    want = [ref_bf16(v) for v in vals]
    assert got == want, "bf16 rounding of doubles is not a single correct rounding"


def pin_unpack(orc):
    assert list(orc.unpack(np.array([0x76543210], np.uint32), 8, 4)) == list(range(8))
    assert list(orc.unpack(np.array([0x89ABCDEF], np.uint32), 8, 4)) == list(range(15, 7, -1))
    assert list(orc.unpack(np.array([0x04030201], np.uint32), 4, 8)) == [1, 2, 3, 4]
    assert list(orc.unpack(np.array([0xE4], np.uint32), 4, 2)) == [0, 1, 2, 3]
    rng = np.random.default_rng(2)
    for bits in (2, 4, 8):
        codes = rng.integers(0, 1 << bits, size=(3, 64), dtype=np.uint8)
        words = inputs.pack_codes(codes, bits)
        got = orc.unpack(words.ravel(), codes.size, bits)
        assert np.array_equal(got, codes.ravel())
        assert ref_codes_from_words(words.ravel(), codes.size, bits) == list(codes.ravel())


def _hand_case():
    with open(os.path.join(GOLDEN, "hand_2x8.json")) as f:
        gd = json.load(f)

    def b16(vals):
        return lib_bf16_bits(np.asarray(vals, dtype=np.float32))

    gate = inputs.QuantMatrix(np.array(gd["wg_words"], np.uint32).reshape(2, 1),
                              b16(gd["sg"]).reshape(2, 1), b16(gd["bg"]).reshape(2, 1), 8, 4)
    up = inputs.QuantMatrix(np.array(gd["wu_words"], np.uint32).reshape(2, 1),
                            b16(gd["su"]).reshape(2, 1), b16(gd["bu"]).reshape(2, 1), 8, 4)
    x = b16(gd["x"]).reshape(2, 8)
    return gd, inputs.Case(x=x, gate=gate, up=up)


def pin_hand_example(orc):
    gd, case = _hand_case()
    out, g, u = orc.qswiglu(*case.oracle_args(), variant=MATCH, return_acc=True)
    assert np.array_equal(g, np.array(gd["g"])) and np.array_equal(u, np.array(gd["u"]))
    want = lib_bf16_bits(np.asarray(gd["match"], np.float32))
    assert np.array_equal(out, want), (out, want)
    out = orc.qswiglu(*case.oracle_args(), variant=F32)
    assert np.array_equal(out, lib_bf16_bits(np.asarray(gd["f32"], np.float32)))
    dg = orc.qswiglu(*case.oracle_args(), variant=DEBUG_GATE)
    du = orc.qswiglu(*case.oracle_args(), variant=DEBUG_UP)
    assert np.array_equal(dg, lib_bf16_bits(np.asarray(gd["g"], np.float32)))
    assert np.array_equal(du, lib_bf16_bits(np.asarray(gd["u"], np.float32)))
    # the unfused elementwise step on the stored bf16 projections, same values
    sm = orc.silu_mul(dg.ravel(), du.ravel(), MATCH).reshape(2, 2)
    assert np.array_equal(sm, lib_bf16_bits(np.asarray(gd["match"], np.float32)))
    # dequantised rows
    w = orc.dequant(case.gate.packed, case.gate.scales, case.gate.biases, 8, 8, 4)
    assert list(w[0]) == [-4, -3, -2, -1, 0, 1, 2, 3]
    assert list(w[1]) == [3.5, 3, 2.5, 2, 1.5, 1, 0.5, 0]


def pin_zero_input(orc):
    case = inputs.make_case(3, 128, 24, seed=3)
    case.x[:] = 0
    for v in (MATCH, F32, DEBUG_GATE, DEBUG_UP):
        out = orc.qswiglu(*case.oracle_args(), variant=v)
        assert np.all(out == 0), f"x=0 must give +0 (variant {v})"


def pin_integer_case(orc, seed=4):
    rng = np.random.default_rng(seed)
    M, H, I = 5, 96, 7
    for bits, gs in ((4, 32), (8, 32), (2, 96)):
        qg = rng.integers(0, 1 << bits, size=(I, H), dtype=np.uint8)
        qu = rng.integers(0, 1 << bits, size=(I, H), dtype=np.uint8)
        xi = rng.integers(-2, 3, size=(M, H))
        one = lib_bf16_bits(np.ones((I, H // gs), np.float32))
        zero = np.zeros((I, H // gs), np.uint16)
        case = inputs.Case(x=lib_bf16_bits(xi.astype(np.float32)),
                           gate=inputs.QuantMatrix(inputs.pack_codes(qg, bits), one, zero, gs, bits),
                           up=inputs.QuantMatrix(inputs.pack_codes(qu, bits), one, zero, gs, bits))
        g_int = xi.astype(np.int64) @ qg.astype(np.int64).T
        u_int = xi.astype(np.int64) @ qu.astype(np.int64).T
        dg = orc.qswiglu(*case.oracle_args(), variant=DEBUG_GATE)
        du = orc.qswiglu(*case.oracle_args(), variant=DEBUG_UP)
        assert np.array_equal(dg, lib_bf16_bits(g_int.astype(np.float32)))
        assert np.array_equal(du, lib_bf16_bits(u_int.astype(np.float32)))
        y = orc.qmm(case.x, case.gate.packed, one, zero, gs, bits)
        assert np.array_equal(y, lib_bf16_bits(g_int.astype(np.float32)))


def pin_brute_force(orc):
    cases = [
        inputs.make_case(2, 64, 3, bits_g=4, gs_g=32, seed=5),
        inputs.make_case(3, 64, 2, bits_g=8, gs_g=64, bits_u=4, gs_u=32, seed=6),
        inputs.make_case(1, 32, 4, bits_g=2, gs_g=32, bits_u=8, gs_u=32, seed=7,
                         scale_range=(0.05, 0.3)),
    ]
    for case in cases:
        for v in (MATCH, F32, DEBUG_GATE, DEBUG_UP):
            got = orc.qswiglu(*case.oracle_args(), variant=v)
            want = brute_force(case, v)
            assert np.array_equal(got, want), (case.meta, v, got, want)
        y = orc.qmm(case.x, case.up.packed, case.up.scales, case.up.biases, case.up.gs, case.up.bits)
        assert np.array_equal(y, brute_force(case, DEBUG_UP))


def pin_k_permutation(orc):
    """Permuting whole groups of K in x and both weights leaves g and u unchanged."""
    case = inputs.make_case(4, 256, 16, bits_g=4, gs_g=64, bits_u=8, gs_u=32, seed=8,
                            keep_codes=True)
    gs = 64
    perm_groups = np.random.default_rng(9).permutation(256 // gs)
    kperm = np.concatenate([np.arange(p * gs, (p + 1) * gs) for p in perm_groups])

    def permute(qm: inputs.QuantMatrix):
        codes = qm.codes[:, kperm]
        gperm = np.concatenate([np.arange(p * gs // qm.gs, (p + 1) * gs // qm.gs) for p in perm_groups])
        return inputs.QuantMatrix(inputs.pack_codes(codes, qm.bits), qm.scales[:, gperm].copy(),
                                  qm.biases[:, gperm].copy(), qm.gs, qm.bits)

    pc = inputs.Case(x=case.x[:, kperm].copy(), gate=permute(case.gate), up=permute(case.up))
    _, g0, u0 = orc.qswiglu(*case.oracle_args(), variant=MATCH, return_acc=True)
    _, g1, u1 = orc.qswiglu(*pc.oracle_args(), variant=MATCH, return_acc=True)
    assert np.allclose(g0, g1, rtol=1e-12, atol=1e-12) and np.allclose(u0, u1, rtol=1e-12, atol=1e-12)
    assert np.array_equal(orc.qswiglu(*case.oracle_args(), variant=F32),
                          orc.qswiglu(*pc.oracle_args(), variant=F32))


def pin_silu_values(orc):
    """Closed forms of the elementwise step: silu(0)=0, silu(g)->g for large g,
    silu(g) - silu(-g) = g, and sigmoid(0) = 1/2 exactly."""
    g = lib_bf16_bits(np.array([0.0, 0.0, 20.0, 40.0, -40.0, 2.0], np.float32))
    u = lib_bf16_bits(np.array([5.0, -3.0, 1.0, 2.0, 1.0, 1.0], np.float32))
    for v in (MATCH, F32):
        h = orc.silu_mul(g, u, v)
        vals = [bf16_val(int(t)) for t in h]
        assert vals[0] == 0.0 and vals[1] == 0.0
        assert vals[2] == 20.0 and vals[3] == 80.0
        assert abs(vals[4]) < 1e-15
        # silu(2) = 2 / (1 + e^-2) = 1.76159..
        assert abs(vals[5] - 2.0 / (1.0 + math.exp(-2.0))) <= 2 ** -7 * 2
    rng = np.random.default_rng(10)
    gv = rng.uniform(-6, 6, size=200).astype(np.float32)
    gp, gn = lib_bf16_bits(gv), lib_bf16_bits(-gv)
    one = lib_bf16_bits(np.ones(200, np.float32))
    hp = np.array([bf16_val(int(t)) for t in orc.silu_mul(gp, one, F32)])
    hn = np.array([bf16_val(int(t)) for t in orc.silu_mul(gn, one, F32)])
    gb = np.array([bf16_val(int(t)) for t in gp])
    assert np.allclose(hp - hn, gb, atol=2 ** -6 * (np.abs(gb) + 1))


def pin_silu_exhaustive(orc):
    """Every bf16 gate value in [-16, 16] (and a few u), against the step-by-step
    definition built from the reference rounding and the C library exp."""
    hs = np.arange(0, 0x10000, dtype=np.uint32)
    vals = (hs << 16).view(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= 16.0)
    g = hs[keep].astype(np.uint16)
    for uval in (1.0, -3.0, 0.3):
        u = lib_bf16_bits(np.full(g.shape, uval, np.float32))
        ub = bf16_val(int(u[0]))
        got_m = orc.silu_mul(g, u, MATCH)
        got_f = orc.silu_mul(g, u, F32)
        for j, h in enumerate(g[::3]):
            gv = bf16_val(int(h))
            sig = ref_round(1.0 / (1.0 + math.exp(-gv)))
            want_m = ref_bf16(ref_round(gv * sig) * ub)
            want_f = ref_bf16(gv * ub / (1.0 + math.exp(-gv)))
            assert got_m[3 * j] == want_m, (gv, uval)
            assert got_f[3 * j] == want_f, (gv, uval)


def pin_match_is_unfused(orc):
    """MATCH is defined as the unfused composition qmm, qmm, sigmoid, mul, mul."""
    case = inputs.make_case(5, 192, 40, bits_g=4, gs_g=64, bits_u=8, gs_u=32, seed=11)
    fused = orc.qswiglu(*case.oracle_args(), variant=MATCH)
    g = orc.qmm(case.x, case.gate.packed, case.gate.scales, case.gate.biases, 64, 4)
    u = orc.qmm(case.x, case.up.packed, case.up.scales, case.up.biases, 32, 8)
    assert np.array_equal(fused, orc.silu_mul(g, u, MATCH))


def pin_sampled_pairs(orc):
    case = inputs.make_case(6, 128, 30, seed=12)
    full = orc.qswiglu(*case.oracle_args(), variant=MATCH)
    pairs = np.array([[0, 0], [5, 29], [3, 17], [2, 2]])
    got = orc.qswiglu_pairs(*case.oracle_args(), MATCH, pairs)
    assert np.array_equal(got, full[pairs[:, 0], pairs[:, 1]])
    rows = orc.qswiglu(*case.oracle_args(), variant=MATCH, rows=[4, 1])
    assert np.array_equal(rows, full[[4, 1]])


# ---------------------------------------------------- f16 activations -----

def pin_f16_decode(orc):
    """Every binary16 bit pattern widens to numpy's float16 value."""
    hs = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    want = hs.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_f64(int(h)) for h in hs])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan])


def pin_f16_double(orc, n=4000, seed=13):
    """One correct rounding of doubles to binary16: midpoints nudged by a few
    double ulps, exact ties, the subnormal range and the overflow threshold."""
    rng = np.random.default_rng(seed)
    vals = []
    for _ in range(n):
        h = int(rng.integers(0x0001, 0x7BFF))
        lo, hi = f16_val(h), f16_val(h + 1)
        mid = (lo + hi) / 2
        sgn = math.copysign(1.0, rng.standard_normal())
        for d in (-3, -1, 0, 1, 3):
            vals.append(sgn * (mid + d * math.ulp(mid)))
    vals += [2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26, 2.0 ** -14 - 2.0 ** -25, 65504.0,
             65519.99, 65520.0, 65536.0, 1e6, -1e-9, 0.0, -0.0, 1.0 + 2.0 ** -11]
    got = [orc.f64_to_f16(v) for v in vals]
    want = [ref_f16(v) for v in vals]
    assert got == want, "binary16 rounding of doubles is not a single correct rounding"


def pin_f16_hand_example(orc):
    gd, case = _hand_case()
    with open(os.path.join(GOLDEN, "hand_2x8_f16.json")) as f:
        g16 = json.load(f)
    f16 = lambda vals: lib_f16_bits(np.asarray(vals, dtype=np.float32))
    q = lambda qm, s, b: inputs.QuantMatrix(qm.packed, f16(s).reshape(2, 1), f16(b).reshape(2, 1), 8, 4)
    c16 = inputs.Case(x=f16(gd["x"]).reshape(2, 8), gate=q(case.gate, gd["sg"], gd["bg"]),
                      up=q(case.up, gd["su"], gd["bu"]), dtype="f16")
    out, g, u = orc.qswiglu(*c16.oracle_args(), variant=MATCH, return_acc=True, dtype="f16")
    assert np.array_equal(g, np.array(gd["g"])) and np.array_equal(u, np.array(gd["u"]))
    assert np.array_equal(out, f16(g16["match"])), out
    assert np.array_equal(orc.qswiglu(*c16.oracle_args(), variant=F32, dtype="f16"), f16(g16["f32"]))
    dg = orc.qswiglu(*c16.oracle_args(), variant=DEBUG_GATE, dtype="f16")
    du = orc.qswiglu(*c16.oracle_args(), variant=DEBUG_UP, dtype="f16")
    sm = orc.silu_mul(dg.ravel(), du.ravel(), MATCH, dtype="f16").reshape(2, 2)
    assert np.array_equal(sm, f16(g16["match"]))
    # the same case read as bf16 gives the bf16 golden values: the dtype matters
    assert not np.array_equal(f16(g16["match"]), lib_bf16_bits(np.asarray(gd["match"], np.float32)))


def pin_f16_brute_force(orc):
    cases = [
        inputs.make_case(2, 64, 3, bits_g=4, gs_g=32, seed=14, dtype="f16"),
        inputs.make_case(2, 64, 2, bits_g=8, gs_g=64, bits_u=2, gs_u=32, seed=15, dtype="f16",
                         scale_range=(0.05, 0.3)),
    ]
    for case in cases:
        for v in (MATCH, F32, DEBUG_GATE, DEBUG_UP):
            got = orc.qswiglu(*case.oracle_args(), variant=v, dtype="f16")
            want = brute_force(case, v)
            assert np.array_equal(got, want), (case.meta, v, got, want)
        y = orc.qmm(case.x, case.gate.packed, case.gate.scales, case.gate.biases, case.gate.gs,
                    case.gate.bits, dtype="f16")
        assert np.array_equal(y, brute_force(case, DEBUG_GATE))
        w = orc.dequant(case.gate.packed, case.gate.scales, case.gate.biases, case.H, case.gate.gs,
                        case.gate.bits, dtype="f16")
        codes = np.array([ref_codes_from_words(r, case.H, case.gate.bits) for r in case.gate.packed])
        for i in range(case.I):
            for k in range(0, case.H, 7):
                s = f16_val(int(case.gate.scales[i, k // case.gate.gs]))
                b = f16_val(int(case.gate.biases[i, k // case.gate.gs]))
                assert w[i, k] == f16_val(ref_f16(float(Fraction(s) * int(codes[i, k]) + Fraction(b))))


def pin_f16_silu_exhaustive(orc):
    """Every binary16 gate value in [-16, 16] through the elementwise step,
    against the step-by-step definition in binary16."""
    hs = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    vals = hs.view(np.float16).astype(np.float64)
    g = hs[np.isfinite(vals) & (np.abs(vals) <= 16.0)]
    for uval in (1.0, -3.0, 0.3):
        u = lib_f16_bits(np.full(g.shape, uval, np.float32))
        ub = f16_val(int(u[0]))
        got_m = orc.silu_mul(g, u, MATCH, dtype="f16")
        got_f = orc.silu_mul(g, u, F32, dtype="f16")
        for j in range(0, g.size, 5):
            gv = f16_val(int(g[j]))
            sig = f16_val(ref_f16(1.0 / (1.0 + math.exp(-gv))))
            assert got_m[j] == ref_f16(f16_val(ref_f16(gv * sig)) * ub), (gv, uval)
            assert got_f[j] == ref_f16(gv * ub / (1.0 + math.exp(-gv))), (gv, uval)


# ------------------------------------------------- whole MLP, residual -----

def _mlp_case(M, H, I, Ho, dtype, seed):
    case = inputs.make_case(M, H, I, bits_g=4, gs_g=32, bits_u=8, gs_u=32, seed=seed, dtype=dtype)
    down = inputs.make_case(1, I, Ho, bits_g=4, gs_g=32, seed=seed + 100, dtype=dtype).gate
    h = inputs.make_x(M, Ho, seed=seed + 200, dtype=dtype)
    return case, down, h


def _brute_down(hidden_bits, down, h_bits, dtype):
    """y = T(h + hidden . Wd^T) with exact rational sums."""
    to_bits, val = REF[dtype]
    M, I = hidden_bits.shape
    Ho = down.packed.shape[0]
    codes = [ref_codes_from_words(r, I, down.bits) for r in down.packed]
    W = [[Fraction(val(to_bits(float(Fraction(val(int(down.scales[o, k // down.gs]))) * codes[o][k]
                                      + Fraction(val(int(down.biases[o, k // down.gs]))))))) for k in range(I)]
         for o in range(Ho)]
    y = np.zeros((M, Ho), dtype=np.uint16)
    for m in range(M):
        hid = [Fraction(val(int(t))) for t in hidden_bits[m]]
        for o in range(Ho):
            acc = sum(hid[k] * W[o][k] for k in range(I))
            if h_bits is not None:
                acc += Fraction(val(int(h_bits[m, o])))
            y[m, o] = to_bits(float(acc))
    return y


def pin_mlp_brute_force(orc):
    """The whole block against exact rational sums (bf16 and f16): hidden is
    the fused expansion, y = T(h + hidden . Wd^T) with one rounding."""
    for dtype, seed in (("bf16", 21), ("f16", 22)):
        case, down, h = _mlp_case(2, 64, 32, 5, dtype, seed)
        for v in (MATCH, F32):
            y, hidden = orc.mlp(case.x, h, *case.oracle_args()[1:], down.packed, down.scales, down.biases,
                                down.gs, down.bits, variant=v, dtype=dtype)
            assert np.array_equal(hidden, brute_force(case, v)), (dtype, v)
            assert np.array_equal(y, _brute_down(hidden, down, h, dtype)), (dtype, v)
        y0 = orc.qmm(case.x, case.gate.packed, case.gate.scales, case.gate.biases, case.gate.gs,
                     case.gate.bits, dtype=dtype, residual=None)
        assert np.array_equal(y0, brute_force(case, DEBUG_GATE))


def pin_mlp_zero_input(orc):
    """x = 0 gives hidden = 0 and y = h exactly; with no residual y = +0."""
    for dtype in ("bf16", "f16"):
        case, down, h = _mlp_case(3, 96, 64, 7, dtype, 23)
        case.x[:] = 0
        args = (*case.oracle_args()[1:], down.packed, down.scales, down.biases, down.gs, down.bits)
        y, hidden = orc.mlp(case.x, h, *args, variant=MATCH, dtype=dtype)
        assert np.all(hidden == 0) and np.array_equal(y, h)
        y, _ = orc.mlp(case.x, None, *args, variant=F32, dtype=dtype)
        assert np.all(y == 0)


ALL_PINS = [pin_bf16_binary32, pin_bf16_double, pin_unpack, pin_hand_example,
            pin_zero_input, pin_integer_case, pin_brute_force, pin_k_permutation,
            pin_silu_values, pin_silu_exhaustive, pin_match_is_unfused, pin_sampled_pairs,
            pin_f16_decode, pin_f16_double, pin_f16_hand_example, pin_f16_brute_force,
            pin_f16_silu_exhaustive, pin_mlp_brute_force, pin_mlp_zero_input]
