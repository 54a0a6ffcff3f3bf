"""Plant plausible mistakes in copies of the oracle; each must trip a pin.

A mutant is the oracle's C source with one textual change (a wrong index, a
dropped term, a swapped operand), compiled on the CPU into a temporary
library. The committed oracle is never modified.
"""
import json
import os
import subprocess
import sys

import pytest

from oracle import build as oracle_build

HERE = os.path.dirname(os.path.abspath(__file__))
REPO = os.path.dirname(HERE)

# Runs every pin against one mutant library in a child process, so that a
# mutant which reads out of bounds and crashes cannot take the test run down.
CHILD = """
import json, sys
sys.path[:0] = [{repo!r}, {tests!r}]
import oracle, oracle_pins
mut = oracle.Oracle({lib!r})
caught = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(mut)
    except Exception as exc:
        caught.append([pin.__name__, type(exc).__name__])
print(json.dumps(caught))
"""

MUTANTS = {
    "offset_uses_division": ("int64_t offset = pos % block_size;",
                             "int64_t offset = pos / block_size;"),
    "table_row_stride": ("block_tables[(int64_t)seq * max_blocks_per_seq + logical_block]",
                         "block_tables[(int64_t)seq * block_size + logical_block]"),
    "interleaved_groups": ("int qh = kv_head * group + j;", "int qh = j * n_kv_heads + kv_head;"),
    "scale_dropped": ("z[i] = scale * dot;\n        if (z[i] > zmax)\n            zmax = z[i];\n    }\n    double denom",
                      "z[i] = dot;\n        if (z[i] > zmax)\n            zmax = z[i];\n    }\n    double denom"),
    "values_from_keys": ("oracle_gather(v_cache, block_tables, max_blocks_per_seq, seq, length, kv_head,\n                      n_kv_heads, head_dim, block_size, dtype, V);\n        for (int j",
                         "oracle_gather(k_cache, block_tables, max_blocks_per_seq, seq, length, kv_head,\n                      n_kv_heads, head_dim, block_size, dtype, V);\n        for (int j"),
    "last_token_dropped": ("for (int i = 0; i < length; ++i) {\n        double dot",
                           "for (int i = 0; i < length - 1; ++i) {\n        double dot"),
    "exp_sign_flipped": ("z[i] = exp(z[i] - zmax);", "z[i] = exp(zmax - z[i]);"),
    "f16_bias_off_by_one": ("expo - 25", "expo - 24"),
    "bf16_wrong_half": ("uint32_t bits = (uint32_t)b << 16;", "uint32_t bits = (uint32_t)b << 15;"),
    "merge_drops_l": ("denom += w * l[p];", "denom += w;"),
    "merge_weight_sign": ("double w = exp(m[p] - M);", "double w = exp(M - m[p]);"),
    "append_row_offset": ("memcpy(k_cache + slot * row_bytes, k_rows + t * row_bytes",
                          "memcpy(k_cache + slot * row_bytes, k_rows + slot * row_bytes"),
    "padding_not_skipped": ("if (token_pos[t] < 0) {", "if (token_pos[t] < -1) {"),
    "copy_only_keys": ("        memcpy(v_cache + dst * block_bytes, v_cache + src * block_bytes, (size_t)block_bytes);\n", ""),
    "copy_direction_swapped": ("memcpy(k_cache + dst * block_bytes, k_cache + src * block_bytes",
                               "memcpy(k_cache + src * block_bytes, k_cache + dst * block_bytes"),
    "swap_destination_index": ("memcpy(dst_k + to * block_bytes, src_k + from * block_bytes",
                               "memcpy(dst_k + from * block_bytes, src_k + from * block_bytes"),
    "swap_bounds_one_pool": ("to < 0 || to >= dst_blocks", "to < 0 || to >= src_blocks"),
    "prefill_causal_exclusive": ("attend(qd, K, V, position + 1,", "attend(qd, K, V, position,"),
    "prefill_position_from_chunk_start": ("int position = length - rows + r;", "int position = r;"),
    "prefill_query_row_offset": ("((int64_t)(first + r) * n_q_heads + qh)",
                                 "((int64_t)r * n_q_heads + qh)"),
    "swap_only_keys": ("        memcpy(dst_v + to * block_bytes, src_v + from * block_bytes, (size_t)block_bytes);\n", ""),
}


def run_pins(src_text, tmp_dir):
    """Compile `src_text` as an oracle library and run every pin against it in
    the child harness; returns the finished process."""
    src = tmp_dir / "oracle_copy.c"
    src.write_text(src_text)
    lib = oracle_build.build(str(src), str(tmp_dir / "oracle_copy.so"))
    code = CHILD.format(repo=REPO, tests=HERE, lib=lib)
    return subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          timeout=300)


@pytest.fixture(scope="module")
def control(tmp_path_factory):
    """The unmutated source through the same compile step and child harness: it
    must exit 0 with no pin failing. Only then does a mutant's non-zero exit
    count as caught (an import error or a broken harness would otherwise make
    every mutant look caught)."""
    res = run_pins(open(oracle_build.SOURCE).read(), tmp_path_factory.mktemp("control"))
    assert res.returncode == 0, f"control run failed: {res.stderr[-2000:]}"
    caught = json.loads(res.stdout.strip().splitlines()[-1])
    assert caught == [], f"pins fail on the unmutated oracle: {caught}"
    return True


def test_control_passes_every_pin(control):
    assert control


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, control):
    old, new = MUTANTS[name]
    src = open(oracle_build.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique in the oracle source"
    res = run_pins(src.replace(old, new), tmp_path)
    if res.returncode != 0:
        # the mutant crashed or raised outside a pin (the control, run the same
        # way, exited 0): caught
        return
    caught = json.loads(res.stdout.strip().splitlines()[-1])
    assert caught, f"no pin caught mutant {name}"
