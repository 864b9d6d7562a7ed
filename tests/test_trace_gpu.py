"""The trace build (-DGQA_TRACE=1) of the decode split kernel.

It must compute exactly what the default build computes (the trace only reads
clocks and waits for a phase's results before stamping it) and leave one sane
record per CTA: stamps in order, tile counts that match the split, phase cycles
that add up to at most the loop's.
"""
import math

import numpy as np
import pytest
import torch

import gqa_attention_gb300 as g
from gqa_attention_gb300 import _binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
WORDS = 64


@pytest.fixture(scope="module")
def libs(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_gb300 import build

    build.build()
    release = g.load()
    d = tmp_path_factory.mktemp("trace")
    path = build.build(extra_flags=["-DGQA_TRACE=1"], lib_path=str(d / "libgqa_attn_trace.so"),
                       build_dir=str(d / "obj"))
    saved = _binding._lib
    _binding._lib = None
    try:
        traced = _binding.load(path)
    finally:
        _binding._lib = saved
    yield release, traced
    _binding._lib = saved


def _with(handle, fn):
    saved = _binding._lib
    _binding._lib = handle
    try:
        out = fn()
        torch.cuda.synchronize()
        return out
    finally:
        _binding._lib = saved


def _records(handle, n_cta):
    buf = np.zeros(n_cta * WORDS, dtype=np.uint64)
    assert _with(handle, lambda: g.gqa_trace_read(buf, buf.nbytes)) == g.GQA_OK
    return buf.reshape(n_cta, WORDS)


@pytest.mark.parametrize("fp8", [False, True])
def test_trace_build_is_bit_identical_and_records_are_sane(libs, fp8):
    release, traced = libs
    B, H_q, H_kv, d, S, n = 1, 64, 8, 128, 8192, 19
    if fp8:
        host = inputs.decode_inputs_fp8(B, H_q, H_kv, d, S, seed=2)
        call = g.decode_fp8
    else:
        host = inputs.decode_inputs(B, H_q, H_kv, d, S, seed=2)
        call = g.decode
    args = [x.to(DEV) for x in host]
    outs = []
    for handle in (release, traced):
        if handle is traced:
            assert _with(handle, g.gqa_trace_clear) == g.GQA_OK
        outs.append(_with(handle, lambda: call(*args, n_split=n)))
    (o0, l0), (o1, l1) = outs
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)) and torch.equal(l0, l1)
    assert _with(traced, g.gqa_last_device_error) == g.GQA_OK

    rec = _records(traced, n * H_kv)
    chunk = g.gqa_attn_decode_split_chunk(S, n)
    tiles = [-(-(min(S, (s + 1) * chunk) - s * chunk) // 64) for s in range(n)]
    for r in rec:
        stamps = [int(x) for x in r[:5]]
        assert stamps[0] > 0 and stamps == sorted(stamps), stamps
        split = int(r[6])
        assert 0 <= split < n and int(r[7]) == tiles[split]
        warps = r[8:8 + 6 * 8].reshape(8, 6)
        used = warps[warps[:, 4] > 0]
        assert len(used) in (4, 8)
        # every tile is taken by one group of four warps
        assert int(used[:, 5].sum()) == 4 * tiles[split]
        for w in used:
            assert int(w[0] + w[1] + w[2] + w[3]) <= int(w[4])


def test_mma_rate_probe(libs):
    """The trace build's tcgen05.mma rate probe: every form reports a finite
    positive cost, N = 256 costs more per instruction than N = 128, and no
    form beats the nominal rate by more than clock-reading noise."""
    _, traced = libs
    rates = {}
    for form, nominal in ((0, 64), (1, 64), (2, 128), (3, 32), (4, 64), (5, 64)):
        st, cyc = _with(traced, lambda: g.gqa_trace_mma_rate(form, 64))
        assert st == g.GQA_OK, (form, st)
        assert math.isfinite(cyc) and cyc >= 0.95 * nominal, (form, cyc)
        rates[form] = cyc
    assert rates[2] > rates[0]
    for bad in ((-1, 8), (6, 8), (0, 0), (0, 1 << 17)):
        assert _with(traced, lambda: g.gqa_trace_mma_rate(*bad))[0] == g.GQA_ERR_INVALID_ARG


def test_prefill_trace_is_bit_identical_and_stamps_are_ordered(libs):
    """The trace build's causal prefill computes exactly what the default build
    computes, and each recorded tile's stamps follow the pipeline's order."""
    release, traced = libs
    S, H_q, H_kv, d = 2048, 16, 2, 128
    gen = torch.Generator().manual_seed(4)
    q, k, v = (torch.randn(1, S, h, d, generator=gen).to(torch.bfloat16).to(DEV)
               for h in (H_q, H_kv, H_kv))
    outs = []
    for handle in (release, traced):
        if handle is traced:
            assert _with(handle, g.gqa_trace_clear) == g.GQA_OK
        outs.append(_with(handle, lambda: g.prefill_causal(q, k, v)))
    (o0, l0), (o1, l1) = outs
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)) and torch.equal(l0, l1)
    buf = np.zeros(8 * 2 * 64 * 16, dtype=np.uint64)
    assert _with(traced, lambda: g.gqa_trace_prefill_read(buf, buf.nbytes)) == g.GQA_OK
    rec = buf.reshape(8, 2, 64, 16).astype(np.int64)
    # the heaviest items come first: every CTA's first item has all S / 128 tiles
    n = S // 128
    checked = 0
    for c in range(8):
        for x in range(2):
            for j in range(n):
                r = rec[c, x, j]
                assert (r[:14] > 0).all() or (j == n - 1 and (r[:14] > 0).sum() == 13), (c, x, j, r)
                assert r[0] <= r[8] <= r[9] <= r[10] <= r[4], (c, x, j, r)  # quarter 0's own order
                assert r[11] <= r[12] <= r[13] and r[12] >= max(r[4:8]), (c, x, j, r)
                if j + 1 < n:
                    assert r[13] <= r[14] <= min(rec[c, x, j + 1, 0:4]), (c, x, j, r)
                checked += 1
    assert checked == 8 * 2 * n
    assert _with(traced, lambda: g.gqa_trace_prefill_read(buf, buf.nbytes + 8)) == g.GQA_ERR_INVALID_ARG
