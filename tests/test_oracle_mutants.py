"""Plant plausible mistakes in a copy of the oracle; every one must fail a pin.

Each mutant edits exactly one spot of ``oracle/ns_oracle.c`` (a dropped term,
a wrong sign, index or operand), is compiled on the CPU into a temp dir, and
is run against the full pin set of ``_pins.py``.  A mutant that no pin
catches would mean the pins do not fix that part of the oracle.
"""
import json
import os
import subprocess
import sys

import pytest

import _pins
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# A mutant may index outside its arrays and crash; each runs in a child
# process, and a crash counts as caught.
_CHILD = """
import json, sys
sys.path[:0] = [{root!r}, {here!r}]
import _pins, oracle
print(json.dumps(_pins.failing_pins(oracle.Oracle({lib!r}))))
"""


def _failing_pins_isolated(lib_path):
    code = _CHILD.format(root=ROOT, here=HERE, lib=lib_path)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return ["<crashed>"]
    return json.loads(r.stdout.strip().splitlines()[-1])

MUTANTS = {
    # Element decoding.
    "f16_exponent_bias": ("v = ldexp((double)(1024 + f), e - 25);",
                          "v = ldexp((double)(1024 + f), e - 24);"),
    "f16_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "bf16_exponent_bias": ("v = ldexp((double)(128 + f), e - 134);",
                           "v = ldexp((double)(128 + f), e - 133);"),
    "bf16_hidden_bit": ("v = ldexp((double)(128 + f), e - 134);",
                        "v = ldexp((double)(f), e - 134);"),
    # Append.
    "append_offset": ("int64_t offset = slot % block_size;",
                      "int64_t offset = (slot + 1) % block_size;"),
    "append_skips_negative_wrongly": ("if (slot < 0)\n            continue;",
                                      "if (slot <= 0)\n            continue;"),
    "append_head_stride": ("int64_t src = (t * num_kv_heads + h) * head_dim + d;",
                           "int64_t src = (t * num_kv_heads) * head_dim + d;"),
    "append_v_from_k": ("v_pool[dst] = v[src];", "v_pool[dst] = k[src];"),
    # Gather through the block table.
    "gqa_mapping_modulo": ("int h = j / group;", "int h = j % num_kv_heads;"),
    "k_offset_shift": (
        "const uint16_t *kr = k_pool + ((block * num_kv_heads + h) * block_size + p % block_size) * head_dim;",
        "const uint16_t *kr = k_pool + ((block * num_kv_heads + h) * block_size + (p + 1) % block_size) * head_dim;"),
    "k_layout_transposed": (
        "const uint16_t *kr = k_pool + ((block * num_kv_heads + h) * block_size + p % block_size) * head_dim;",
        "const uint16_t *kr = k_pool + ((h * num_blocks + block) * block_size + p % block_size) * head_dim;"),
    "v_read_from_k_pool": (
        "const uint16_t *vr = v_pool + ((block * num_kv_heads + h)",
        "const uint16_t *vr = k_pool + ((block * num_kv_heads + h)"),
    "v_block_index_off_by_one": (
        "int64_t block = block_tables[s * (int64_t)max_blocks_per_seq + p / block_size];\n            const uint16_t *vr",
        "int64_t block = block_tables[s * (int64_t)max_blocks_per_seq + (p + 1) / block_size];\n            const uint16_t *vr"),
    "table_row_stride": (
        "int64_t block = block_tables[s * (int64_t)max_blocks_per_seq + p / block_size];\n            if",
        "int64_t block = block_tables[s + p / block_size];\n            if"),
    "q_row_uses_kv_head": ("qv[d] = elem(dtype, q[(row * num_q_heads + j) * head_dim + d]);",
                           "qv[d] = elem(dtype, q[(row * num_q_heads + h) * head_dim + d]);"),
    # Scores and softmax.
    "scale_dropped": ("z[p] = scale * dot;", "z[p] = dot;"),
    "softmax_sign": ("z[p] = exp(z[p] - zmax);", "z[p] = exp(zmax - z[p]);"),
    "no_normalisation": ("double w = z[p] / denom;", "double w = z[p];"),
    # Query positions and the causal window.
    "causal_excludes_self": ("int64_t n_keys = row_pos[row] + 1;", "int64_t n_keys = row_pos[row];"),
    "causal_one_too_many": ("int64_t n_keys = row_pos[row] + 1;",
                            "int64_t n_keys = row_pos[row] + 1 + (row_pos[row] + 1 < context_lens[s]);"),
    "span_position_not_advanced": ("row_pos[first + i] = L - q_len + i;", "row_pos[first + i] = L - q_len;"),
}

def _source():
    with open(oracle.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    src = _source()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} must appear exactly once"
    mutant = oracle.build_variant(src.replace(old, new))
    bad = _failing_pins_isolated(mutant.path)
    assert bad, f"no pin catches mutant {name}"


def test_unmutated_copy_passes_every_pin():
    assert _failing_pins_isolated(oracle.build_variant(_source()).path) == []
