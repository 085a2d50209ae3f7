"""Planted mistakes in the oracle must each fail at least one pin (CPU only).

Each case copies oracle/pa_oracle.c, plants one plausible mistake by text
substitution (a dropped term, a wrong sign, a wrong index, a swapped operand),
compiles it with gcc into a temporary directory and runs every pin against it
in a child process. The unmodified oracle passes every pin (test_oracle.py);
each mutant must fail one. This is what shows the pins are strong enough to
stand in for a reference implementation the pages do not provide.
"""

import os
import subprocess
import sys
from pathlib import Path

import pytest

import oracle

HERE = Path(__file__).resolve().parent
SRC = Path(oracle.__file__).resolve().parent / "pa_oracle.c"

MUTATIONS = {
    "scale_dropped": ("s[t] = dot * scale;", "s[t] = dot;"),
    "exp_sign_flipped": ("s[t] = exp(s[t] - m);", "s[t] = exp(m - s[t]);"),
    "not_normalised": ("const double w = s[t] / denom;", "const double w = s[t];"),
    "gqa_interleaved": ("const int h = hq / group;", "const int h = hq % kv_heads;"),
    "causal_off_by_one": ("const int64_t visible = L - num_queries + i + 1;",
                          "const int64_t visible = L - num_queries + i;"),
    "no_causal_mask": ("const int64_t visible = L - num_queries + i + 1;",
                       "const int64_t visible = L;"),
    "query_row_from_kv_head": ("const int64_t qoff = (((int64_t)b * num_queries + i) * q_heads + hq) * head_dim;",
                               "const int64_t qoff = (((int64_t)b * num_queries + i) * q_heads + h) * head_dim;"),
    "k_and_v_swapped_in_gather": ("Vc[dst + d] = load_elem(v_cache, dtype, src + d);",
                                  "Vc[dst + d] = load_elem(k_cache, dtype, src + d);"),
    "block_row_from_next_block": (
        "const int32_t pb = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];",
        "const int32_t pb = block_tables[(int64_t)b * max_blocks_per_seq + (t / block_size + 1) % ((L + block_size - 1) / block_size)];"),
    "write_v_from_k": ("memcpy((char *)v_cache + dst * es, (const char *)v_new + src * es, row_bytes);",
                       "memcpy((char *)v_cache + dst * es, (const char *)k_new + src * es, row_bytes);"),
    "write_skips_last_head": ("for (int h = 0; h < kv_heads; ++h) {\n            const int64_t dst",
                              "for (int h = 0; h < kv_heads - 1; ++h) {\n            const int64_t dst"),
    "bf16_widened_wrong_half": ("uint32_t bits = ((uint32_t)((const uint16_t *)base)[index]) << 16;",
                                "uint32_t bits = ((uint32_t)((const uint16_t *)base)[index]) << 15;"),
    # int8 pool
    "q8_offset_127": ("return (uint8_t)((int)r + 128);", "return (uint8_t)((int)r + 127);"),
    "q8_floor_not_nearest": ("float r = rintf(x * inv);", "float r = floorf(x * inv);"),
    "q8_ties_away_from_zero": ("float r = rintf(x * inv);", "float r = roundf(x * inv);"),
    "q8_inverse_of_128": ("return maxabs == 0.0f ? 0.0f : 127.0f / maxabs; }", "return maxabs == 0.0f ? 0.0f : 128.0f / maxabs; }"),
    "q8_scale_over_128": ("return maxabs / 127.0f; }", "return maxabs / 128.0f; }"),
    "q8_dequant_without_offset": ("return (float)((int)byte - 128) * s; }", "return (float)((int)byte) * s; }"),
    "q8_k_scale_kept": ("ks[d] = q8_scale(m);", "(void)m;"),
    "q8_k_incoming_row_dropped": (
        "for (int d = 0; d < head_dim; ++d) x[r * head_dim + d] = q8_widen_bf16(src[d]);",
        "(void)src;"),
    "q8_v_row_from_k": ("const uint16_t *src = v_new + ((int64_t)j * kv_heads + h) * head_dim;",
                        "const uint16_t *src = k_new + ((int64_t)j * kv_heads + h) * head_dim;"),
    "q8_k_scale_per_row": ("for (int r = 0; r < block_size; ++r) {\n                    const float a = fabsf(x[r * head_dim + d]);",
                           "for (int r = 0; r < 1; ++r) {\n                    const float a = fabsf(x[r * head_dim + d]);"),
    "q8_v_scale_of_wrong_row": ("v_scale[blk * block_size + r] = q8_scale(m);",
                                "v_scale[blk * block_size + (r + 1) % block_size] = q8_scale(m);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    text = SRC.read_text()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "pa_oracle_mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.compile_oracle(src, tmp_path / "libmutant.so")
    env = dict(os.environ, OMP_NUM_THREADS="2")
    proc = subprocess.run([sys.executable, str(HERE / "oracle_pins.py"), str(lib)],
                          capture_output=True, text=True, env=env, timeout=600)
    assert proc.returncode != 0, f"mutant {name} passed every pin:\n{proc.stdout}\n{proc.stderr}"
    assert "FAILED" in proc.stdout, f"mutant {name} crashed instead of failing a pin:\n{proc.stderr[-2000:]}"
