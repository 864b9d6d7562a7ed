"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/gqa_oracle.c`` (a dropped
term, a wrong index, an off-by-one bound, a wrong constant), compiles it with
gcc into a temporary library, points a fresh instance of the ``oracle`` wrapper
at it, and runs the pin tests of ``test_oracle_pins.py`` against that instance:
at least one pin must fail.  CPU only; nothing here touches the CUDA path.
"""
import importlib.util
import os
import subprocess

import numpy as np
import pytest

import test_oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gqa_oracle.c")
INIT = os.path.join(ROOT, "oracle", "__init__.py")

# (name, text in the oracle, planted replacement)
MUTATIONS = [
    ("head map h mod H_kv", "int kv = h / G; /* [AKL] p.15 §2 */", "int kv = h % c->H_kv;"),
    ("LSE without the max", "*lse = m + log(l);", "*lse = log(l);"),
    ("scale dropped", "s[j] = scale * acc;", "s[j] = acc;"),
    ("no normalisation by l", "double p = exp(s[j] - m) / l;", "double p = exp(s[j] - m);"),
    ("causal bound off by one", "attend_row(qrow, kh, vh, i + 1, d, c->scale, s,",
     "attend_row(qrow, kh, vh, i > 0 ? i : 1, d, c->scale, s,"),
    ("merge drops the running factor", "l_acc = a_acc * l_acc + a_s * l_s;",
     "l_acc = l_acc + a_s * l_s;"),
    ("split bound off by one", "if (hi > n) hi = n;", "if (hi > n) hi = n - 1;"),
    ("window one key short", "int64_t lo = (c->window >= 0 && a - c->window > 0) ? a - c->window : 0;",
     "int64_t lo = (c->window >= 0 && a - c->window + 1 > 0) ? a - c->window + 1 : 0;"),
    ("chunk anchored at the start", "int64_t q0 = L - c->T_q; /* absolute position of chunk row 0 */",
     "int64_t q0 = 0;"),
    ("page offset from the wrong term", "int64_t off = t % B_p;", "int64_t off = t / B_p % B_p;"),
    ("E4M3 bias 8", "v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("values read from the key head",
     "repeat_head(c->v, c->dtype, b, n, c->S_max, c->H_kv, d, kv, vh);\n  attend_row(qrow, kh, vh, n,",
     "repeat_head(c->k, c->dtype, b, n, c->S_max, c->H_kv, d, kv, vh);\n  attend_row(qrow, kh, vh, n,"),
]


def _golden_all(o):
    for case in pins._golden_cases():
        pins.test_golden_closed_forms(o, case)


PROBES = [
    _golden_all,
    pins.test_single_key_returns_that_value,
    pins.test_identical_keys_give_mean_of_values,
    pins.test_zero_query_is_uniform_over_visible_keys,
    pins.test_causal_row_zero_is_first_value,
    pins.test_gqa_equals_mha_with_repeated_kv_heads,
    lambda o: pins.test_split_then_merge_equals_unsplit(o, 3),
    pins.test_merge_is_commutative_and_has_identity,
    pins.test_brute_force_decimal_tiny_shapes,
    pins.test_three_pass_matches_online_forms,
    pins.test_prefill_row_equals_decode_on_its_prefix,
    pins.test_chunk_rows_are_the_tail_rows_of_the_full_prefill,
    pins.test_window_limits_and_closed_forms,
    lambda o: pins.test_paged_decode_equals_contiguous_decode(o, 4),
    pins.test_e4m3_decoding_matches_torch_for_every_code,
    pins.test_fp8_decode_equals_decode_of_the_dequantised_cache,
]


def _mutant(tmp_path, idx, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    path = tmp_path / f"mut{idx}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"libmut{idx}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", str(path),
                           "-o", str(lib), "-lm"])
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{idx}", INIT)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._LIB_PATH = str(lib)
    mod.build = lambda force=False: str(lib)
    return mod


def test_unmutated_oracle_passes_every_probe(oracle_mod):
    for probe in PROBES:
        probe(oracle_mod)


@pytest.mark.parametrize("idx", range(len(MUTATIONS)), ids=[m[0] for m in MUTATIONS])
def test_each_planted_mistake_is_caught(tmp_path, idx):
    name, old, new = MUTATIONS[idx]
    mod = _mutant(tmp_path, idx, old, new)
    caught = []
    for probe in PROBES:
        try:
            with np.errstate(all="ignore"):
                probe(mod)
        except AssertionError as e:  # a failed pin
            caught.append((getattr(probe, "__name__", "probe"), type(e).__name__))
    assert caught, f"no pin caught the planted mistake: {name}"
