"""The pins are strong enough: plausible mistakes planted in a copy of the
oracle source (on the CPU) each make at least one pin fail.

Each mutant is a textual edit of ``oracle/oracle.c`` compiled into a
temporary library; the real oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("gqa_modulo", "int j = h / group;", "int j = h % n_kv_heads;"),
    ("gqa_times", "int j = h / group;", "int j = (h * n_kv_heads) / n_q_heads / 2;"),
    ("row_reversed", "+ t % block_size) * head_dim", "+ (block_size - 1 - t % block_size)) * head_dim"),
    ("layout_head_major", "(((int64_t)block * n_kv_heads + j) * block_size",
     "(((int64_t)j * num_blocks + block) * block_size"),
    ("block_index_off_by_one", "+ t / block_size];", "+ (t + 1) / block_size];"),
    ("scale_dropped", "s[t - t_begin] = scale * dot;", "s[t - t_begin] = dot;"),
    ("dot_shifted", "g_f16[kt[k]];", "g_f16[kt[(k + 1) % head_dim]];"),
    ("v_from_k", "const uint16_t *vt = token_row(v_cache,", "const uint16_t *vt = token_row(k_cache,"),
    ("not_normalised", "double o = (l > 0.0) ? acc[k] / l : 0.0;", "double o = acc[k];"),
    ("lse_sign", "m + log(l) : -INFINITY", "m - log(l) : -INFINITY"),
    ("max_not_subtracted_in_l", "s[i] = exp(s[i] - m); l += s[i];", "s[i] = exp(s[i] - m); l += exp(s[i]);"),
    ("merge_unweighted", "denom += w * l[i];", "denom += l[i];"),
    ("merge_weight_sign", "double w = exp(m[i] - M);", "double w = exp(M - m[i]);"),
    ("f16_exponent", "expo - 25", "expo - 24"),
    ("f16_subnormal", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    ("encode_truncates", "double m = rint(ldexp(a, 10 - e));", "double m = floor(ldexp(a, 10 - e));"),
    ("append_offset", "int64_t offset = slot % block_size;", "int64_t offset = 0;"),
    ("append_keeps_negative", "if (slot < 0) continue;", "if (slot < -1) continue;"),
    ("e4m3_bias", "ldexp((double)(8 + frac), expo - 10)", "ldexp((double)(8 + frac), expo - 9)"),
    ("e4m3_truncates", "double m = rint(ldexp(a, 3 - e));", "double m = floor(ldexp(a, 3 - e));"),
    ("e4m3_no_saturation", "if (a >= 448.0) return (uint8_t)(sign | 0x7e);",
     "if (a >= 464.0) return 0x7f;"),
    ("e4m3_subnormal", "double m = rint(ldexp(a, 9));", "double m = rint(ldexp(a, 8));"),
    ("f8_quantize_multiplies", "volatile float y = x / scale;", "volatile float y = x * scale;"),
    ("f8_k_scale_dropped", "(g_e4m3[kt[k]] * k_scale)", "g_e4m3[kt[k]]"),
    ("f8_v_scale_dropped", "acc[k] += p * (g_e4m3[vt[k]] * v_scale);", "acc[k] += p * g_e4m3[vt[k]];"),
    ("multi_causal_one_past", "b, h, 0, pos + 1, &m, &l, acc);", "b, h, 0, pos + 2, &m, &l, acc);"),
    ("multi_no_causal_mask", "int pos = context_lens[b] - nq + (r - query_start[b]);",
     "int pos = context_lens[b] - 1;"),
    ("multi_position_from_start", "int pos = context_lens[b] - nq + (r - query_start[b]);",
     "int pos = r - query_start[b];"),
    ("multi_first_query_row", "rc = attend_range_qv(q + rh * head_dim,",
     "rc = attend_range_qv(q + ((int64_t)query_start[b] * n_q_heads + h) * head_dim,"),
    ("empty_range_bound", "for (int t = t_begin; t < t_end; ++t) {\n        const uint16_t *kt",
     "for (int t = t_begin; t < t_end - (t_end - t_begin > 1); ++t) {\n        const uint16_t *kt"),
]


def _build_mutant(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, f"{name}: pattern not found"
    mutated = text.replace(old, new, 1)
    src = tmp_path / f"{name}.c"
    src.write_text(mutated)
    out = tmp_path / f"{name}.so"
    oracle.build(force=True, src=str(src), out=str(out))
    return str(out)


_RUNNER = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, pins
lib = oracle.load({lib!r})
lib.pkvo_init()
for pin in pins.ALL_PINS:
    try:
        pin(lib)
    except (AssertionError, oracle.OracleError, ValueError, FloatingPointError, TypeError) as e:
        print("caught by", pin.__name__)
        sys.exit(3)
sys.exit(0)
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    path = _build_mutant(tmp_path, name, old, new)
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(tests_dir), tests=tests_dir, lib=path)
    # a separate process: a mutant that writes out of bounds may crash it,
    # which also counts as caught
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin"
