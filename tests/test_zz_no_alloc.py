"""The allocation-free decode entry point, through the C ABI.

gqa_attn_decode_noalloc() serves callers that cannot call cudaMalloc while
they decode (code inside a custom allocator's critical section, or a serving
process whose device memory pool is fixed up front); its split partials live
in a 16 MiB scratch array inside the library.  Its outputs are checked
against the regular two-stage decode and against the fp64 oracle, on two calls
in a row, and on a smaller call that follows a larger one (the scratch keeps
the previous call's contents).  This file is collected last so that a run
stopping at its first failure has already run every other test; it also
passes when run alone in a fresh process.
"""
import math

import pytest
import torch

import gqa_attention_gb300 as g
from gqa_attention_gb300 import inputs

from parity import MAX_DLSE, MAX_DO, MEAN_DO, assert_parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_gb300 import build

    build.build()
    g.load()
    yield
    assert g.gqa_last_device_error() == g.GQA_OK


def _close(a_out, a_lse, b_out, b_lse):
    do = (a_out.float() - b_out.float()).abs()
    dl = (a_lse - b_lse).abs()
    assert torch.isfinite(a_out.float()).all() and torch.isfinite(a_lse).all()
    assert do.max().item() <= MAX_DO and do.mean().item() <= MEAN_DO
    assert dl.max().item() <= MAX_DLSE


def _noalloc(q, k, v, sl, B, S_max, H_q, H_kv, d, scale, n_split):
    out = torch.full((B, H_q, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H_q), float("nan"), dtype=torch.float32, device=DEV)
    st = g.gqa_attn_decode_noalloc(q, k, v, sl, B, S_max, H_q, H_kv, d, scale, n_split, out, lse)
    assert st == g.GQA_OK
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("B,H_q,H_kv,d,S_max,lens,n_split", [
    (1, 64, 8, 128, 32768, None, 38),      # Llama3-70B decode shape, 38 splits
    (3, 16, 4, 64, 3000, [3000, 1, 1234], 7),
    (2, 8, 2, 32, 500, [500, 77], 1),       # no split: no scratch used
])
def test_noalloc_matches_two_stage_decode_and_oracle_twice(oracle_mod, B, H_q, H_kv, d, S_max,
                                                           lens, n_split):
    qh, kh, vh, slh = inputs.decode_inputs(B, H_q, H_kv, d, S_max, seed=21, seq_lens=lens)
    q, k, v, sl = (x.to(DEV) for x in (qh, kh, vh, slh))
    scale = 1 / math.sqrt(d)
    ref_out, ref_lse = g.decode(q, k, v, sl, scale=scale, n_split=n_split)
    orc_out, orc_lse = oracle_mod.decode(qh, kh, vh, slh, scale)
    for _ in range(2):  # the scratch keeps the previous call's contents
        out, lse = _noalloc(q, k, v, sl, B, S_max, H_q, H_kv, d, scale, n_split)
        _close(out, lse, ref_out, ref_lse)
        assert_parity(out, lse, orc_out, orc_lse, "noalloc vs oracle")


def test_noalloc_smaller_call_after_a_larger_one(oracle_mod):
    """A call with more rows and splits fills more of the scratch; the next,
    smaller call (other seed, other split count) must read only its own partials."""
    big = dict(B=4, H_q=32, H_kv=4, d=128, S_max=4096, lens=[4096, 3000, 17, 2048], n_split=48)
    small = dict(B=2, H_q=16, H_kv=2, d=128, S_max=2500, lens=[2500, 900], n_split=11)
    for cfg, seed in ((big, 5), (small, 6)):
        qh, kh, vh, slh = inputs.decode_inputs(cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["d"],
                                               cfg["S_max"], seed=seed, seq_lens=cfg["lens"])
        q, k, v, sl = (x.to(DEV) for x in (qh, kh, vh, slh))
        scale = 1 / math.sqrt(cfg["d"])
        out, lse = _noalloc(q, k, v, sl, cfg["B"], cfg["S_max"], cfg["H_q"], cfg["H_kv"],
                            cfg["d"], scale, cfg["n_split"])
        orc_out, orc_lse = oracle_mod.decode(qh, kh, vh, slh, scale)
        assert_parity(out, lse, orc_out, orc_lse, f"noalloc n_split={cfg['n_split']}")


def test_noalloc_allocates_no_device_memory():
    """After a first call on the device, further calls leave torch's allocator
    and the device's free memory untouched."""
    B, H_q, H_kv, d, S_max, n_split = 1, 64, 8, 128, 8192, 19
    q, k, v, sl = (x.to(DEV) for x in inputs.decode_inputs(B, H_q, H_kv, d, S_max, seed=3))
    out = torch.empty((B, H_q, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, H_q), dtype=torch.float32, device=DEV)
    args = (q, k, v, sl, B, S_max, H_q, H_kv, d, 1 / math.sqrt(d), n_split, out, lse)
    assert g.gqa_attn_decode_noalloc(*args) == g.GQA_OK  # first call: address look-up
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert g.gqa_attn_decode_noalloc(*args) == g.GQA_OK
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == torch_before
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before


def test_noalloc_rejects_partials_larger_than_its_scratch():
    B, H_q, d, n_split = 8, 64, 128, 64  # 8*64*64*(128*4) bytes of O partials > 16 MiB
    assert g.gqa_attn_decode_workspace_bytes(B, H_q, d, n_split) > 16 << 20
    x = torch.empty(16, dtype=torch.bfloat16, device=DEV)
    lens = torch.ones(B, dtype=torch.int32, device=DEV)
    st = g.gqa_attn_decode_noalloc(x, x, x, lens, B, 128, H_q, 8, d, 0.1, n_split, x,
                                   torch.empty(1, device=DEV))
    assert st == g.GQA_ERR_INVALID_ARG
