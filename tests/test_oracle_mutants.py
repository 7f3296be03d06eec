"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a private copy of the oracle's C
source (a dropped term, an off-by-one, a wrong operand or weight), builds it,
and requires that at least one pin in ``oracle_pins`` fails on it.  The real
oracle is never modified.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")

# (name, text in mla_oracle.c, replacement, which occurrence (0-based) or None for all)
MUTANTS = [
    ("mask_strict", "return j * D + r <= P;", "return j * D + r < P;", None),
    ("mask_off_by_one", "return j * D + r <= P;", "return j * D + r <= P + 1;", None),
    ("shard_owner", "if (p % D == r) ++n;", "if (p % D == (r + 1) % D) ++n;", None),
    ("rope_term_dropped", "acc += bf16_to_double(qp[e]) * bf16_to_double(row[KV_LORA_RANK + e]);", "acc += 0.0;",
     None),
    ("rope_sign", "acc += bf16_to_double(qp[e]) * bf16_to_double(row[KV_LORA_RANK + e]);",
     "acc -= bf16_to_double(qp[e]) * bf16_to_double(row[KV_LORA_RANK + e]);", None),
    ("nope_width", "for (int d = 0; d < KV_LORA_RANK; ++d)\n      acc +=",
     "for (int d = 0; d < KV_LORA_RANK - 1; ++d)\n      acc +=", None),
    ("no_scale", "s[k] = scale * acc;", "s[k] = acc;", None),
    ("lse_without_max", "double l = m + log(z);", "double l = log(z);", None),
    ("unnormalised_weights", "double p = exp(s[k] - l);", "double p = exp(s[k] - m);", None),
    ("value_width", "for (int d = 0; d < KV_LORA_RANK; ++d) out[d] += p",
     "for (int d = 0; d < KV_LORA_RANK - 1; ++d) out[d] += p", None),
    ("position_dense", "int64_t P = L - q_len + (t - qsl[b]);", "int64_t P = L - q_len + (t - qsl[b]) - 1;", 0),
    ("position_dcp", "int64_t P = L - q_len + (t - qsl[b]);", "int64_t P = L - q_len + (t - qsl[b]) - 1;", 1),
    ("position_kv8", "int64_t P = L - q_len + (t - qsl[b]);", "int64_t P = L - q_len + (t - qsl[b]) - 1;", 2),
    ("position_sparse", "int64_t P = L - q_len + (t - qsl[b]);", "int64_t P = L - q_len + (t - qsl[b]) + 1;", 3),
    ("page_offset", "return kv_cache + (page * page_size + j % page_size) * ROW_WIDTH;",
     "return kv_cache + (page * page_size + (j + 1) % page_size) * ROW_WIDTH;", None),
    ("sparse_future_kept", "if (p < 0 || p > P) continue;", "if (p < 0) continue;", None),
    ("sparse_valid_ignored", "e < valid[t] && e < K", "e < K", None),
    ("sparse_shard_filter", "if (p % D != r) continue;", "if (p % D == r) continue;", None),
    ("merge_counts_ignored", "int part = valid_counts ? valid_counts[r * T + t] > 0", "int part = valid_counts ? 1",
     None),
    ("merge_weight_max", "double w = exp(lses[(r * T + t) * H + h] - L);",
     "double w = exp(lses[(r * T + t) * H + h] - m);", None),
    ("merge_lse_without_max", "double L = m + log(z);", "double L = log(z);", None),
    ("e4m3_exponent_bias", "else v = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "else v = ldexp(1.0 + (double)m / 8.0, e - 8);", None),
    ("e4m3_subnormal_scale", "if (e == 0) v = ldexp((double)m, -9);", "if (e == 0) v = ldexp((double)m, -10);", None),
    ("e4m3_sign_dropped", "return sign ? -v : v;", "return v;", None),
    ("kv8_value_scale_dropped", "out[d] += p * (kv_scale * mla_oracle_e4m3_to_double(row[d]));",
     "out[d] += p * mla_oracle_e4m3_to_double(row[d]);", None),
    ("kv8_rope_term_dropped", "acc += bf16_to_double(qp[e]) *\n             (kv_scale", "acc += 0.0 *\n             (kv_scale",
     None),
    ("kv8_page_offset", "key_scratch[n++] = kv_cache + (page * page_size + j % page_size) * ROW_WIDTH;",
     "key_scratch[n++] = kv_cache + (page * page_size + (j + 1) % page_size) * ROW_WIDTH;", None),
    ("wuv_transposed", "acc += x[d] * bf16_to_double(w[d * V + v]);",
     "acc += x[d] * bf16_to_double(w[v * KV_LORA_RANK + d]);", None),
]


def _mutate(src, old, new, occ):
    assert old in src, old
    if occ is None:
        return src.replace(old, new)
    parts = src.split(old)
    assert len(parts) > occ + 1, (old, occ)
    return old.join(parts[:occ + 1]) + new + old.join(parts[occ + 1:])


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, occ):
    src = open(SRC).read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    c = tmp_path / "mutant.c"
    c.write_text(mutated)
    so = tmp_path / "mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"], check=True)
    lib = oracle.load(str(so))
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(lib)
        except AssertionError:
            failed.append(check.__name__)
            break
    assert failed, f"mutant {name} passed every pin"
