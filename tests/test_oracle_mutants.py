"""Planted mistakes in copies of the oracle (on the CPU): each must fail a pin.

Every mutant is a plausible slip -- a swapped nibble, a wrong offset or bias, a
transposed scale index, a dropped term, a lost sign, a missing router weight --
applied as a text edit to a temporary copy of oracle.c, which is compiled and
run through the same pins as the real oracle.
"""
import os

import pytest

import pins
from oracle import oracle

MUTANTS = {
    "int4_nibble_order": ("(i % 2 == 0) ? (b & 0x0F)", "(i % 2 == 1) ? (b & 0x0F)"),
    "int4_offset": ("(double)(code - 8)", "(double)(code - 7)"),
    "int3_offset": ("(double)(code - 4)", "(double)(code - 3)"),
    "int3_plane_b_bit_order": ("(i % 8)) & 1", "(7 - i % 8)) & 1"),
    "int3_plane_b_offset": ("w + O * (I / 4);", "w + O * (I / 8);"),
    "int3_plane_a_shift": ("(2 * (i % 4))) & 3", "(i % 4)) & 3"),
    "int8_unsigned": ("(int)(int8_t)w[o * I + i]", "(int)w[o * I + i]"),
    "e2m1_bias": ("ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e)"),
    "e2m1_no_sign": ("return sign ? -mag : mag;", "return mag;"),
    "e2m1_subnormal": ("(e == 0) ? 0.5 * m", "(e == 0) ? 1.0 * m"),
    "scale_first_group_only": ("scales[o * (I / gs) + i / gs]", "scales[o * (I / gs)]"),
    "int3_group_32": ("case ORACLE_INT3_G64: return 64;", "case ORACLE_INT3_G64: return 32;"),
    "mxfp4_group_64": ("case ORACLE_MXFP4_E8M0: return 32;", "case ORACLE_MXFP4_E8M0: return 64;"),
    "scale_group_mod": ("scales[o * (I / gs) + i / gs]", "scales[o * (I / gs) + i % (I / gs)]"),
    "gemv_dropped_term": ("for (long i = 0; i < I; i++)\n        acc +=", "for (long i = 1; i < I; i++)\n        acc +="),
    "gemv_token_ignored": ("y[t * O + o] = row_dot(fmt, gs, w, scales, O, I, o, x + t * I);",
                           "y[t * O + o] = row_dot(fmt, gs, w, scales, O, I, o, x);"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "gate_up_swapped": ("return oracle_silu(g) * u;", "return oracle_silu(u) * g;"),
    "clamp_up_one_sided": ("if (u < -limit) u = -limit;", "if (u < 0.0) u = 0.0;"),
    "clamp_gate_missing": ("if (g > limit) g = limit;", ""),
    "clamp_gate_both_sides": ("if (g > limit) g = limit;", "if (g > limit) g = limit;\n        if (g < -limit) g = -limit;"),
    "router_weight_dropped": ("out[t * ncols + j] += wr * z;", "out[t * ncols + j] += z;"),
    "down_transposed": ("oracle_weight(fmt, gs, de, dse, D, F, d, f)", "oracle_weight(fmt, gs, de, dse, F, D, f, d)"),
    "e8m0_bias": ("ldexp(1.0, e - 127)", "ldexp(1.0, e - 128)"),
    "e8m0_scales_as_f32": ("if (fmt == ORACLE_MXFP4_E8M0)\n        return", "if (fmt == -1)\n        return"),
    "int8_grouped_per_row": ("case ORACLE_INT8_ROW:\n    case ORACLE_INT4_ROW: return I;",
                             "case ORACLE_INT8_ROW:\n    case ORACLE_INT8_G:\n    case ORACLE_INT4_ROW: return I;"),
    "int4_row_no_offset": ("case ORACLE_INT4_ROW:\n    case ORACLE_INT4_G: return (double)(code - 8);",
                           "case ORACLE_INT4_G: return (double)(code - 8);\n    case ORACLE_INT4_ROW: return (double)code;"),
    "expert_rank_last_only": ("out[t * ncols + j] = 0.0;", "out[t * ncols + j] = 0.0 * out[t * ncols + j];"),
    "route_ties_high_index": ("key_scratch[e] > key_scratch[best]) best = e;", "key_scratch[e] >= key_scratch[best]) best = e;"),
    "route_renorm_over_all": ("if (renorm) {\n                for (long r = 0; r < k; r++) denom +=",
                              "if (0) {\n                for (long r = 0; r < k; r++) denom +="),
    "route_bias_in_weight": ("const double sg = oracle_sigmoid((double)l[ids[t * k + r]]);",
                             "const double sg = oracle_sigmoid((double)l[ids[t * k + r]]) + (double)bias[ids[t * k + r]];"),
    "route_sigmoid_sign": ("return 1.0 / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(z));"),
    "route_scale_dropped": ("wts[t * k + r] = scale * exp(", "wts[t * k + r] = exp("),
    "gemv_rows_unmapped": ("O, I, rows[j], x + t * I);", "O, I, j, x + t * I);"),
    "gate_up_rows_unmapped": ("F, D, rows[j], x + t * D);", "F, D, j, x + t * D);"),
    "expert_cols_unmapped": ("long d = cols ? cols[j] : j;", "long d = j;"),
    "expert_e8m0_scale_stride": ("long ssz = fmt == ORACLE_MXFP4_E8M0 ? 1 : (long)sizeof(float);",
                                 "long ssz = (long)sizeof(float);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(old) >= 1, f"mutation site of {name} not found"
    src = src.replace(old, new)
    if name == "expert_rank_last_only":
        # keep only the last rank: overwrite instead of accumulate
        src = src.replace("out[t * ncols + j] += wr * z;", "out[t * ncols + j] = wr * z;")
    path = os.path.join(tmp_path, f"{name}.c")
    open(path, "w").write(src)
    lib = oracle.compile_oracle(path, os.path.join(tmp_path, f"lib{name}.so"), openmp=False)
    orc = oracle.Oracle(lib)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
        except Exception as e:  # a crash of the mutant counts as caught too
            failed.append(f"{pin.__name__}:{type(e).__name__}")
    assert failed, f"mutant {name} passed every pin"
