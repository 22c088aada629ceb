"""Plant plausible mistakes in a copy of the oracle and check that a pin fails.

Each mutation edits a copy of ``oracle/mla_oracle.c`` in a temporary directory,
compiles it, and runs the pins of ``pins.py`` against that build on the CPU.
A mutation that no pin notices would mean the pins leave that part of the
oracle unchecked.
"""
import os
import subprocess

import pytest

import pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "mla_oracle.c")

MUTATIONS = {
    "drop_rope_key_term": ("k[s->d_nope + e] = kr[e];", "k[s->d_nope + e] = 0.0 * kr[e];"),
    "drop_rope_query_term": (
        "memcpy(qq + d_nope, q_rope + (i * H + h) * (long)d_rope, sizeof(double) * (size_t)d_rope);",
        "memset(qq + d_nope, 0, sizeof(double) * (size_t)d_rope);"),
    "scale_without_rope_width": ("1.0 / sqrt((double)(d_nope + d_rope))",
                                 "1.0 / sqrt((double)(d_nope))"),
    "causal_sees_one_future_key": (
        "long n_keys = (long)q_pos[i] + 1;          /* causal: keys 0..p */",
        "long n_keys = (long)q_pos[i] + 1 + (q_pos[i] + 1 < s->S_max);"),
    "rotation_sign": ("*b = x0 * s + x1 * c;", "*b = -x0 * s + x1 * c;"),
    "frequency_exponent": ("pow(base, -2.0 * (double)i / (double)d)",
                           "pow(base, -1.0 * (double)i / (double)d)"),
    "half_split_paired_as_interleaved": ("rotate_pair(&v[i], &v[i + d / 2],",
                                         "rotate_pair(&v[2 * i], &v[2 * i + 1],"),
    "small_key_not_rotated": ("orc_rope_half(k, 1, 1, s->d_nope, &p, s->base);", "(void)p;"),
    "mlra_block_index": ("int g = h * s->d_nope + e, blk = g / sub_out_k, row = g % sub_out_k;",
                         "int g = h * s->d_nope + e, blk = g % s->L, row = g / s->L;"),
    "value_from_key_weights": ("v[e] = dot(s->W_UV + ((long)h * s->d_v + e) * s->r_kv, c, s->r_kv);",
                               "v[e] = dot(s->W_UK + ((long)h * s->d_v + e) * s->r_kv, c, s->r_kv);"),
    "absorbed_value_skips_last_key": ("for (long j = 0; j < n_keys; ++j) {\n            const double *cj = cache_lat + ((long)b * S_max + j) * r_kv;\n            for (int c = 0;",
                                      "for (long j = 0; j + 1 < n_keys; ++j) {\n            const double *cj = cache_lat + ((long)b * S_max + j) * r_kv;\n            for (int c = 0;"),
    "query_projection_skips_compression": ("orc_linear(c_q, T, r_q, W_UQ, H * d_nope, q_nope, n_threads);",
                                           "orc_linear(c_q, T, r_q, W_UQ, H * d_nope, q_nope, n_threads); q_nope[0] += 1.0;"),
}


def _first_failure(oracle_mod):
    for pin in pins.ALL_PINS:
        try:
            pin(oracle_mod)
        except (AssertionError, RuntimeError, ValueError) as e:
            return f"{pin.__name__}: {e}"[:200]
    return None


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(oracle_mod, tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"pattern for {name} not found in the oracle source"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", str(lib),
                    str(mutated), "-lm"], check=True)
    with oracle_mod.use_library(str(lib)):
        caught = _first_failure(oracle_mod)
    assert caught is not None, f"no pin notices mutation {name}"
