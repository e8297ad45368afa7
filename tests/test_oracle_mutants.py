"""Plant plausible mistakes in copies of the oracle and check that the pins catch each.

Every mutant is a one-line change of ``oracle/oracle.c`` compiled into a temporary
library; the real oracle is never modified.  A mutant that no pin catches would mean
the pins cannot tell that mistake from the truth.
"""
import os
import subprocess

import pytest

import oracle
from oracle_cases import pin_battery

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "oracle.c")

MUTANTS = {
    # wrong GQA mapping: q-head h -> kv-head h mod Hkv instead of h / (Hq/Hkv)
    "gqa_modulo": ("int g = h / (num_q_heads / num_kv_heads);", "int g = h % num_kv_heads;"),
    # causal off-by-one: the diagonal key is not visible
    "causal_no_diagonal": ("int p = seq_lens[s] - q_len + i;                    /*",
                           "int p = seq_lens[s] - q_len + i - 1;                /*"),
    # chunk positions relative to the chunk instead of absolute
    "chunk_relative_positions": ("int p = seq_lens[s] - q_len + i;                    /*",
                                 "int p = i;                    /*"),
    # dropped softmax scale
    "no_scale": ("scores[j] = scale * dot;", "scores[j] = dot;"),
    # wrong sign in the exponent
    "exp_sign": ("scores[j] = exp(scores[j] - m);", "scores[j] = exp(m - scores[j]);"),
    # missing normalisation
    "no_normalise": ("for (int d = 0; d < head_dim; ++d) out_row[d] /= denom;", ""),
    # lse missing its log-sum term
    "lse_no_log": ("*lse_out = m + log(denom);", "*lse_out = m;"),
    # V gathered from the K pool (swapped operand)
    "v_from_k": ("out_row[d] += w * kv_elem(c->v_pool, c->v_codes, base, d, vs);",
                 "out_row[d] += w * kv_elem(c->k_pool, c->k_codes, base, d, vs);"),
    # pool read as [blocks][heads][slots][dim] instead of [blocks][slots][heads][dim]
    "pool_layout_transposed": (
        "return (((size_t)bt[j / c->block_size] * c->block_size + j % c->block_size) * c->num_kv_heads + g)",
        "return (((size_t)bt[j / c->block_size] * c->num_kv_heads + g) * c->block_size + j % c->block_size)"),
    # keys reversed inside a block
    "slot_reversed": (
        "return (((size_t)bt[j / c->block_size] * c->block_size + j % c->block_size) * c->num_kv_heads + g)",
        "return (((size_t)bt[j / c->block_size] * c->block_size + (c->block_size - 1 - j % c->block_size))"
        " * c->num_kv_heads + g)"),
    # E4M3 exponent bias 8 instead of 7
    "e4m3_bias": ("else v = ldexp(1.0 + m / 8.0, e - 7);", "else v = ldexp(1.0 + m / 8.0, e - 8);"),
    # E4M3 rounding by truncation instead of to nearest even
    "e4m3_truncate": ("double m = nearbyint(ldexp(a, 3 - e));", "double m = floor(ldexp(a, 3 - e));"),
    # 8-bit row scale for an int8-style range (127) instead of E4M3's 448
    "fp8_scale_range": ("float scale = amax > 0.0f ? amax / 448.0f : 1.0f;",
                        "float scale = amax > 0.0f ? amax / 127.0f : 1.0f;"),
    # scales read slot-major instead of [block][head][slot]
    "fp8_scale_layout": (
        "return (double)scales[((size_t)bt[j / c->block_size] * c->num_kv_heads + g) * c->block_size\n"
        "                          + (size_t)(j % c->block_size)];",
        "return (double)scales[((size_t)bt[j / c->block_size] * c->block_size + (size_t)(j % c->block_size))\n"
        "                          * c->num_kv_heads + g];"),
    # 8-bit append at the chunk-relative position
    "fp8_append_relative": ("int p = seq_lens[s] - q_len + i;\n            int blk", "int p = i;\n            int blk"),
    # projection with the weight read transposed ([hidden][n_out] instead of [n_out][hidden])
    "qkv_weight_transposed": ("bf16_to_double(w[(size_t)n * hidden + k]);",
                              "bf16_to_double(w[(size_t)k * n_out + n]);"),
    # projection ignores the requested rows
    "qkv_rows_ignored": ("const int t = rows ? rows[r] : r;", "const int t = r;"),
    # projection drops the last input element
    "qkv_dropped_term": ("for (int k = 0; k < hidden; ++k)\n            acc +=",
                         "for (int k = 0; k < hidden - 1; ++k)\n            acc +="),
    # bf16 rounding by truncation
    "bf16_truncate": ("if (frac > 0.5 || (frac == 0.5 && fmod(m, 2.0) != 0.0)) m += 1.0;", ""),
    # bf16 ties rounded away from zero instead of to even
    "bf16_ties_away": ("(frac == 0.5 && fmod(m, 2.0) != 0.0)", "(frac == 0.5)"),
    # bf16 subnormals with the normal quantum (8 significant bits all the way down)
    "bf16_no_subnormals": ("if (lo < -126) lo = -126;", ""),
    # rotary embedding: one sign of the rotation flipped
    "rope_sign": ("v[i] = lo * c - hi * s;", "v[i] = lo * c + hi * s;"),
    # rotary embedding: frequency exponent i / D instead of 2i / D
    "rope_frequency": ("pow(theta, -2.0 * i / head_dim)", "pow(theta, -1.0 * i / head_dim)"),
    # rotary embedding: adjacent dims paired (2i, 2i + 1) instead of (i, i + D/2)
    "rope_interleaved": ("const double lo = v[i], hi = v[i + half];\n                v[i] = lo * c - hi * s;\n"
                         "                v[i + half] = hi * c + lo * s;",
                         "const double lo = v[2 * i], hi = v[2 * i + 1];\n                v[2 * i] = lo * c - hi * s;\n"
                         "                v[2 * i + 1] = hi * c + lo * s;"),
    # rotary embedding at the chunk-relative position
    "rope_relative_position": ("pos[cu_q_lens[s] + i] = seq_lens[s] - q_len + i;", "pos[cu_q_lens[s] + i] = i;"),
    # QK-norm: eps left out of the square root
    "rms_no_eps": ("const double rms = sqrt(sum_sq / head_dim + eps);", "const double rms = sqrt(sum_sq / head_dim);"),
    # QK-norm: the sum of squares instead of their mean
    "rms_sum_not_mean": ("const double rms = sqrt(sum_sq / head_dim + eps);", "const double rms = sqrt(sum_sq + eps);"),
    # QK-norm: the mean square itself instead of its root
    "rms_no_sqrt": ("const double rms = sqrt(sum_sq / head_dim + eps);", "const double rms = sum_sq / head_dim + eps;"),
    # QK-norm: the gain read in reverse order
    "rms_gain_reversed": ("v[d] = bf16_to_double(gain[d]) * v[d] / rms;",
                          "v[d] = bf16_to_double(gain[head_dim - 1 - d]) * v[d] / rms;"),
    # QK-norm: every head normalised by the first head's root mean square
    "rms_first_head_only": ("for (int d = 0; d < head_dim; ++d) sum_sq += v[d] * v[d];",
                            "for (int d = 0; d < head_dim; ++d) sum_sq += v[d - h * head_dim] * v[d - h * head_dim];"),
    # append writes at the chunk-relative position
    "append_relative_position": ("int p = seq_lens[s] - q_len + i;            /* absolute position */",
                                 "int p = i;            /* absolute position */"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = src.replace(old, new)
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"{name}.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", str(c_path),
                    "-o", str(so_path), "-lm"], check=True)
    lib = oracle.load_library(str(so_path))
    failed = pin_battery(lib)
    assert failed, f"no pin caught the planted mistake {name}"


def test_unmutated_oracle_passes_battery():
    assert pin_battery(oracle._load()) == []
