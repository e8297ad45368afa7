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
    "v_from_k": ("out_row[d] += w * bf16_to_double(v_pool[base + d]);",
                 "out_row[d] += w * bf16_to_double(k_pool[base + d]);"),
    # pool read as [blocks][heads][slots][dim] instead of [blocks][slots][heads][dim]
    "pool_layout_transposed": (
        "size_t base = (((size_t)bt[j / block_size] * block_size + j % block_size) * num_kv_heads + g)\n"
        "                      * head_dim;\n        double dot",
        "size_t base = (((size_t)bt[j / block_size] * num_kv_heads + g) * block_size + j % block_size)\n"
        "                      * head_dim;\n        double dot"),
    # keys reversed inside a block
    "slot_reversed": (
        "size_t base = (((size_t)bt[j / block_size] * block_size + j % block_size) * num_kv_heads + g)\n"
        "                      * head_dim;\n        double dot",
        "size_t base = (((size_t)bt[j / block_size] * block_size + (block_size - 1 - j % block_size)) * num_kv_heads + g)\n"
        "                      * head_dim;\n        double dot"),
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
