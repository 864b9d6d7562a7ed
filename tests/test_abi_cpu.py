"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function the header declares, and rejects bad arguments before any
launch; the split and workspace arithmetic follows the header's formulas."""
import ctypes
import os
import re

import pytest

import gqa_attention_gb300 as g
from gqa_attention_gb300 import _binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "gqa_attn.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from gqa_attention_gb300 import build

    build.build()
    return g.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 10
    raw = ctypes.CDLL(_binding.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in gqa_attn.h but not exported"
    assert set(names) == set(_binding.SIGNATURES), "binding and header disagree"


def test_status_strings(lib):
    assert g.status_str(g.GQA_OK) == "GQA_OK"
    assert g.status_str(g.GQA_ERR_TIMEOUT) == "GQA_ERR_TIMEOUT"
    assert g.status_str(99) == "GQA_ERR_UNKNOWN"


@pytest.mark.parametrize("S_max,n_split", [(1024, 1), (1024, 4), (32768, 38), (131072, 64),
                                           (1, 1), (100, 7), (65, 2)])
def test_split_chunk_formula(lib, S_max, n_split):
    per = -(-S_max // n_split)
    assert g.gqa_attn_decode_split_chunk(S_max, n_split) == -(-per // 64) * 64
    assert g.gqa_attn_decode_split_chunk(0, 3) == 0


def test_workspace_bytes_formula(lib):
    B, H, d, n = 2, 64, 128, 38
    ml = B * H * n * 8
    assert g.gqa_attn_decode_workspace_bytes(B, H, d, n) == (ml + 255) // 256 * 256 + B * H * n * d * 4
    assert g.gqa_attn_decode_workspace_bytes(B, H, d, 1) == 0


def test_default_splits_are_bounded(lib):
    # no GPU here: the SM count falls back to a default; the chunk bounds hold
    for B, H_kv, S in [(1, 2, 1024), (1, 8, 32768), (8, 8, 131072), (64, 8, 64), (1, 1, 1)]:
        n = g.gqa_attn_decode_default_splits(B, H_kv, S, -1)
        assert 1 <= n <= max(1, -(-S // 128))
        assert n >= -(-S // 8192)
    assert g.gqa_attn_decode_default_splits(0, 8, 100, -1) == 1
    # an ordinal with no device behind it
    assert g.gqa_attn_decode_default_splits(1, 8, 32768, 4096) == 1


FAKE = 0x10000  # never dereferenced: every case below fails a host check first


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), g.GQA_ERR_INVALID_ARG),
    (dict(H_q=12, H_kv=8), g.GQA_ERR_INVALID_ARG),
    (dict(d=96), g.GQA_ERR_UNSUPPORTED),
    (dict(H_q=34, H_kv=2), g.GQA_ERR_UNSUPPORTED),      # G = 17 > 16
    (dict(n_split=0), g.GQA_ERR_INVALID_ARG),
    (dict(n_split=4, workspace=None), g.GQA_ERR_INVALID_ARG),
    (dict(B=0), g.GQA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), g.GQA_ERR_INVALID_ARG),
    (dict(q=FAKE + 2), g.GQA_ERR_INVALID_ARG),          # not 16-byte aligned
    (dict(n_split=4, workspace=FAKE + 16), g.GQA_ERR_INVALID_ARG),  # not 256-byte aligned
])
def test_decode_rejects_bad_arguments(lib, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, seq_lens=FAKE, B=1, S_max=64, H_q=8, H_kv=2, d=128,
             scale=0.1, n_split=1, workspace=None, out=FAKE, lse=FAKE)
    a.update(kw)
    st = g.gqa_attn_decode(a["q"], a["k"], a["v"], a["seq_lens"], a["B"], a["S_max"], a["H_q"],
                           a["H_kv"], a["d"], a["scale"], a["n_split"], a["workspace"], a["out"],
                           a["lse"], stream=0)
    assert st == status


def test_multi_token_row_limits_and_splits(lib):
    # d = 128 takes up to 128 rows per KV head (one tensor-core tile), d = 32/64
    # up to 64 (four mma.sync row groups); both fail before any launch
    assert g.gqa_attn_decode_multi(FAKE, FAKE, FAKE, FAKE, 1, 17, 64, 16, 2, 128, 0.1, 1, None,
                                   FAKE, FAKE, stream=0) == g.GQA_ERR_UNSUPPORTED  # 136 rows
    assert g.gqa_attn_decode_multi(FAKE, FAKE, FAKE, FAKE, 1, 9, 64, 16, 2, 64, 0.1, 1, None,
                                   FAKE, FAKE, stream=0) == g.GQA_ERR_UNSUPPORTED  # 72 rows, d = 64
    assert g.gqa_attn_decode_multi(FAKE, FAKE, FAKE, FAKE, 1, 65, 128, 2, 2, 128, 0.1, 1, None,
                                   FAKE, FAKE, stream=0) == g.GQA_ERR_INVALID_ARG  # T_q > 64
    # the tensor-core tile runs one CTA per SM: the plain decode's split count
    for B, T_q, H_q, H_kv, S in [(1, 8, 64, 8, 32768), (1, 16, 64, 8, 32768), (2, 3, 64, 8, 5000)]:
        assert g.gqa_attn_decode_multi_default_splits(B, T_q, H_q, H_kv, S, 128) == \
            g.gqa_attn_decode_default_splits(B, H_kv, S, -1)


def test_combine_and_prefill_reject_bad_arguments(lib):
    assert g.gqa_attn_decode_combine(None, 1, 8, 128, 2, FAKE, FAKE, stream=0) == g.GQA_ERR_INVALID_ARG
    assert g.gqa_attn_decode_combine(FAKE, 1, 8, 96, 2, FAKE, FAKE, stream=0) == g.GQA_ERR_UNSUPPORTED
    for d in (16, 96, 256):  # prefill serves d in {32, 64, 128}
        assert g.gqa_attn_prefill_causal(FAKE, FAKE, FAKE, 1, 128, 8, 2, d, 0.1, FAKE, FAKE,
                                         stream=0) == g.GQA_ERR_UNSUPPORTED
    assert g.gqa_attn_prefill_causal(FAKE, FAKE, FAKE, 1, 128, 8, 3, 128, 0.1, FAKE, FAKE,
                                     stream=0) == g.GQA_ERR_INVALID_ARG
    assert g.gqa_attn_prefill_causal(FAKE, None, FAKE, 1, 128, 8, 2, 128, 0.1, FAKE, FAKE,
                                     stream=0) == g.GQA_ERR_INVALID_ARG


def test_wait_limit_setter_round_trips(lib):
    old = g.gqa_set_wait_limit_ns(5_000_000)
    assert g.gqa_set_wait_limit_ns(old) == 5_000_000
    assert g.gqa_set_wait_limit_ns(old) == old


def test_trace_calls_are_unsupported_in_the_default_build(lib):
    """The default library records no trace: every diagnostics call says so
    without touching the GPU."""
    import numpy as np

    buf = np.zeros(64, dtype=np.uint64)
    assert g.gqa_trace_clear() == g.GQA_ERR_UNSUPPORTED
    assert g.gqa_trace_read(buf, buf.nbytes) == g.GQA_ERR_UNSUPPORTED
    assert g.gqa_trace_mma_rate(0, 1)[0] == g.GQA_ERR_UNSUPPORTED
    assert g.gqa_trace_prefill_read(buf, buf.nbytes) == g.GQA_ERR_UNSUPPORTED


def test_balanced_decode_counters_and_checks(lib):
    # two int32 words per (sequence, KV head)
    assert g.gqa_attn_decode_counter_bytes(3, 8) == 3 * 8 * 2 * 4
    assert g.gqa_attn_decode_counter_bytes(0, 8) == 0
    assert g.gqa_attn_decode_counter_bytes(2, -1) == 0
    # with several splits the counters are required and 4-byte aligned; both
    # checks fail before anything reaches the GPU
    args = (FAKE, FAKE, FAKE, FAKE, 1, 4096, 64, 8, 128, 0.1, 19, FAKE)
    assert g.gqa_attn_decode_balanced(*args, None, FAKE, FAKE, stream=0) == g.GQA_ERR_INVALID_ARG
    assert g.gqa_attn_decode_balanced(*args, FAKE + 2, FAKE, FAKE, stream=0) == \
        g.GQA_ERR_INVALID_ARG
    # the shared argument checks of gqa_attn_decode apply as well
    bad = (FAKE, FAKE, FAKE, FAKE, 1, 4096, 12, 8, 128, 0.1, 19, FAKE)  # H_q % H_kv != 0
    assert g.gqa_attn_decode_balanced(*bad, FAKE, FAKE, FAKE, stream=0) == g.GQA_ERR_INVALID_ARG
