"""Each plausible mistake planted in a copy of the oracle's source (a dropped
term, a wrong sign or index, a transposed operand) must make at least one pin
fail.  The mistakes are planted in temporary copies only; the real oracle is
never modified.  CPU only."""
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, exact text in oracle.c, replacement)
MUTANTS = [
    ("drop_scale", "x[j] = scale * dot;", "x[j] = dot;"),
    ("gqa_modulo", "int32_t g = h / group;", "int32_t g = h % num_kv_heads;"),
    ("block_index_mod", "table_row[j / block_size]", "table_row[j % block_size]"),
    ("offset_div", "int64_t offset = j % block_size;", "int64_t offset = j / block_size;"),
    ("write_offset_div", "int64_t offset = slot % block_size;", "int64_t offset = slot / block_size;"),
    ("no_max_subtract", "x[j] = exp(x[j] - m);", "x[j] = exp(x[j]);"),
    ("flipped_sign", "x[j] = exp(x[j] - m);", "x[j] = exp(m - x[j]);"),
    ("no_normalise", "out[d] = acc / Z;", "out[d] = acc;"),
    ("drop_last_token", "for (int64_t j = 0; j < n; ++j) {\n        double dot",
     "for (int64_t j = 0; j < n - 1; ++j) {\n        double dot"),
    ("pool_transposed",
     "int64_t dst = ((block * num_kv_heads + g) * block_size + offset) * head_dim + d;",
     "int64_t dst = ((block * block_size + offset) * num_kv_heads + g) * head_dim + d;"),
    ("gather_transposed",
     "int64_t base = ((block * num_kv_heads + g) * block_size + offset) * head_dim;",
     "int64_t base = ((block * block_size + offset) * num_kv_heads + g) * head_dim;"),
    ("merge_unweighted_l", "L += parts_l[p] * exp(parts_m[p] - M);", "L += parts_l[p];"),
    ("merge_sign", "a += parts_acc[(int64_t)p * head_dim + d] * exp(parts_m[p] - M);",
     "a += parts_acc[(int64_t)p * head_dim + d] * exp(M - parts_m[p]);"),
    ("f16_bias", "expo - 25);", "expo - 24);"),
    ("f16_subnormal", "ldexp((double)frac, -24);", "ldexp((double)frac, -25);"),
    ("bf16_bias", "expo - 134);", "expo - 133);"),
    ("kv_bytes_no_two", "return (int64_t)2 * kv_heads", "return (int64_t)kv_heads"),
    ("blocks_off_by_one", "if (tok % block_size == 0)", "if (tok % block_size == 1)"),
    ("v_from_k", "V[j * head_dim + d] = to_double(v_pool[base + d], is_bf16);",
     "V[j * head_dim + d] = to_double(k_pool[base + d], is_bf16);"),
    ("q_index", "dot += q[d] * K[j * D + d];", "dot += q[0] * K[j * D + d];"),
    ("v_index", "acc += x[j] * V[j * D + d];", "acc += x[j] * V[d];"),
    ("skip_negative_as_bad", "if (slot < 0)\n            continue;", "if (slot < -1)\n            continue;"),
    ("accept_len_over_table", "if (n < 0 || n > (int64_t)max_blocks_per_seq * block_size) {",
     "if (n < 0) {"),
    ("accept_bad_block", "if (block < 0 || block >= num_blocks)", "if (block < 0)"),
    ("copy_only_k", "            v_pool[dst * per_block + e] = v_pool[src * per_block + e];",
     "            v_pool[dst * per_block + e] = v_pool[dst * per_block + e];"),
    ("copy_short", "        for (int64_t e = 0; e < per_block; ++e) {\n            k_pool[dst",
     "        for (int64_t e = 0; e < per_block - 1; ++e) {\n            k_pool[dst"),
    ("prefill_not_causal", "attend_rows(qv, K, V, pos + 1, head_dim, scale, x,",
     "attend_rows(qv, K, V, L, head_dim, scale, x,"),
    ("prefill_causal_off_by_one", "attend_rows(qv, K, V, pos + 1, head_dim, scale, x,",
     "attend_rows(qv, K, V, pos, head_dim, scale, x,"),
    ("prefill_position_base", "int64_t pos = L - C + j;", "int64_t pos = j;"),
    ("prefill_accepts_long_chunk", "int ok = C >= 0 && L >= C &&", "int ok = C >= 0 &&"),
    ("q8_gqa_modulo", "int32_t kv_head = h / group;", "int32_t kv_head = h % num_kv_heads;"),
    ("q8_no_127", "float d32 = amax / 127.0f;", "float d32 = amax / 128.0f;"),
    ("q8_floor", "float r = rintf(v / dq);", "float r = floorf(v / dq);"),
    ("q8_no_clamp", "c = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int)r);", "c = (int)r;"),
    ("q8_v_not_transposed", "v_codes[(slab * head_dim + d) * block_size + offset] = vc[d];",
     "v_codes[(slab * block_size + offset) * head_dim + d] = vc[d];"),
    ("q8_scale_group", "k_scales[(slab * block_size + offset) * ng + d / 32]",
     "k_scales[(slab * block_size + offset) * ng]"),
    ("f16_ties_away", "double q = rint((2.0 * m - 1.0) * 1024.0);",
     "double q = floor((2.0 * m - 1.0) * 1024.0 + 0.5);"),
    ("empty_not_zero", "if (n == 0) {\n        for (int32_t d = 0; d < D; ++d) out[d] = 0.0;",
     "if (n == 0) {\n        for (int32_t d = 0; d < D; ++d) out[d] = 1.0;"),
]


def test_mutation_sites_exist():
    src = open(SRC).read()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, f"mutation site of {name!r} must appear exactly once"


_RUNNER = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
o = oracle.load({lib!r})
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(o)
    except Exception:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = oracle.build(str(mutated), str(tmp_path / "libmutant.so"))
    # A mutant may write out of bounds, so the pins run in a child process;
    # a crash there also counts as the mistake being caught.
    here = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(here), tests=here, lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300)
    if r.returncode != 0:
        return
    line = [x for x in r.stdout.splitlines() if x.startswith("FAILED:")][-1]
    assert line != "FAILED:", f"no pin catches mutant {name}"
