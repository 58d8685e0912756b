"""The pins must catch plausible slips: each mutant below is a copy of the
oracle's C source with one mistake planted (on the CPU, in a temporary
directory); the pin suite, run against that mutant, has to fail."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pa_oracle.c")

MUTANTS = {
    "gqa_map_modulo": ("int kvh = h / group;", "int kvh = h % num_kv_heads;"),
    "scale_dropped": ("s[t] = scale * acc;", "s[t] = acc;"),
    "slot_uses_block_index": ("(size_t)(t % block_size) * row_stride", "(size_t)(t / block_size % block_size) * row_stride"),
    "values_read_from_keys": ("out[d] += w * pao_elem(v_cache", "out[d] += w * pao_elem(k_cache"),
    "no_max_subtraction": ("exp(s[t] - smax)", "exp(s[t])"),
    "exp_sign_flipped": ("exp(s[t] - smax)", "exp(smax - s[t])"),
    "minus_one_wraps": ("if (e < 0 || e >= num_blocks) return -1;",
                        "if (e < 0) e += num_blocks; if (e >= num_blocks) return -1;"),
    "half_exponent_bias": ("e - 25", "e - 24"),
    "bf16_shift": ("((uint32_t)h) << 16", "((uint32_t)h) << 15"),
    "no_normalisation": ("out[d] /= wsum;", "out[d] /= 1.0;"),
    "clamp_off_by_one": ("if (t > cap) t = cap;", "if (t > cap) t = cap - 1;"),
    "q_head_offset": ("((size_t)b * num_heads + h) * head_dim;", "((size_t)b * num_heads + kvh) * head_dim;"),
    "causal_off_by_one": ("int64_t n = T - q_len + i + 1; /* tokens 0 .. p */", "int64_t n = T - q_len + i; /* tokens 0 .. p */"),
    "append_slot_index": ("(size_t)(pos % block_size)) * row", "(size_t)(pos / block_size % block_size)) * row"),
    "append_values_from_keys": ("v_cache[dst + i] = v_new[", "v_cache[dst + i] = k_new["),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found"
    mutated = tmp_path / "pa_oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-o", str(lib), str(mutated), "-lm"],
                   check=True)
    env = dict(os.environ, PA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
