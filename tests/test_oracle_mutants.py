"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one (CPU only).  Each mutation is an exact text edit of
oracle/qsw_oracle.c; the edited copy is compiled into a temporary directory and
the whole pin battery is run against it."""
import pytest

import oracle
from tests import oracle_pins

MUTANTS = {
    "codes_msb_first": ("unsigned shift = (unsigned)((k % pf) * bits);",
                        "unsigned shift = (unsigned)((pf - 1 - k % pf) * bits);"),
    "bias_sign": ("sc * q + bi", "sc * q - bi"),
    "group_index": ("s[r * groups_per_row + k / gs]", "s[r * groups_per_row + (k / gs + 1) % groups_per_row]"),
    "sigmoid_sign": ("double sig = ract(1.0 / (1.0 + exp(-gb)), dt);", "double sig = ract(1.0 / (1.0 + exp(gb)), dt);"),
    "match_drops_silu_rounding": ("double silu = ract(gb * sig, dt);", "double silu = gb * sig;"),
    "match_drops_sigma_rounding": ("double sig = ract(1.0 / (1.0 + exp(-gb)), dt);",
                                   "double sig = 1.0 / (1.0 + exp(-gb));"),
    "f32_rounds_gate": ("case ORC_F32:        return f64_to_act(f32_epilogue(g, u, dt), dt);",
                        "case ORC_F32:        return f64_to_act(f32_epilogue(ract(g, dt), u, dt), dt);"),
    "ties_away": ("return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "return fl + 1.0;"),
    "bf16_one_bit_short": ("int ulp_exp = e - 7;", "int ulp_exp = e - 6;"),
    "up_uses_gate": ("double u = dot_f64(xd + j * H, wur, H);", "double u = dot_f64(xd + j * H, wgr, H);"),
    "dropped_term": ("for (int64_t k = 0; k < K; ++k) acc += xr[k] * wr[k];",
                     "for (int64_t k = 1; k < K; ++k) acc += xr[k] * wr[k];"),
    "silu_uses_up": ("return ract(silu * ub, dt);", "return ract(silu * gb, dt);"),
    "qmm_transposed": ("y[m * N + n] = f64_to_act(acc, dt);",
                       "y[(n % M) * N + (m + n / M) % N] = f64_to_act(acc, dt);"),
    "subnormal_spacing": ("if (ulp_exp < -133) ulp_exp = -133;", "if (ulp_exp < -126) ulp_exp = -126;"),
    "f16_one_bit_short": ("int ulp_exp = e - 10;", "int ulp_exp = e - 9;"),
    "f16_subnormal_spacing": ("if (ulp_exp < -24) ulp_exp = -24;", "if (ulp_exp < -14) ulp_exp = -14;"),
    "f16_exponent_bias": ("(uint16_t)((e + 15) << 10)", "(uint16_t)((e + 16) << 10)"),
    "f16_overflow_early": ("if (r >= 65536.0) return", "if (r >= 32768.0) return"),
    "f16_decode_bias": ("else a = ldexp((double)(1024 + fr), ex - 25);", "else a = ldexp((double)(1024 + fr), ex - 24);"),
    "residual_dropped": ("if (r) acc += act_to_f64(r[m * N + n], dt);", "(void)r;"),
    "residual_rounded_first": ("y[m * N + n] = f64_to_act(acc, dt);",
                               "y[m * N + n] = f64_to_act(r ? act_to_f64(f64_to_act(acc - act_to_f64(r[m * N + n], dt), dt), dt) + act_to_f64(r[m * N + n], dt) : acc, dt);"),
    "mlp_skips_silu": ("int rc = orc_qswiglu(x, M, H, I, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, variant, dt, hidden);",
                       "int rc = orc_qswiglu(x, M, H, I, wg, sg, bg, gs_g, bits_g, wu, su, bu, gs_u, bits_u, ORC_DEBUG_UP, dt, hidden);"),
    "dequant_ignores_dtype": ("out[r * K + k] = act_to_f64(f64_to_act(sc * q + bi, dt), dt);",
                              "out[r * K + k] = orc_bf16_to_f64(orc_f64_to_bf16(sc * q + bi));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    lib = oracle.OracleLib(oracle.build_variant(src.replace(old, new), str(tmp_path / f"{name}.so")))
    failures = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, IndexError):
            failures.append(pin.__name__)
    assert failures, f"no pin caught the planted mistake {name}"
