"""The allocation-free decode entry point against the regular two-stage decode.

gqa_attn_decode_noalloc() serves callers that cannot call cudaMalloc while
they decode (inside a graph capture, an allocator's critical section, or a
serving process with a fixed memory pool); its split partials live in a
16 MiB scratch array inside the library.  This file is collected last so that
a run stopping at its first failure has already run every other test; it also
passes when run alone in a fresh process.
"""
import math

import pytest
import torch

import gqa_attention_gb300 as g
from gqa_attention_gb300 import inputs

from parity import MAX_DLSE, MAX_DO, MEAN_DO

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


@pytest.mark.parametrize("B,H_q,H_kv,d,S_max,lens,n_split", [
    (1, 64, 8, 128, 32768, None, 38),      # Llama3-70B decode shape, default split count
    (3, 16, 4, 64, 3000, [3000, 1, 1234], 7),
    (2, 8, 2, 32, 500, [500, 77], 1),       # no split: no scratch used
])
def test_noalloc_matches_two_stage_decode_twice(B, H_q, H_kv, d, S_max, lens, n_split):
    q, k, v, sl = inputs.decode_inputs(B, H_q, H_kv, d, S_max, seed=21, seq_lens=lens)
    q, k, v, sl = (x.to(DEV) for x in (q, k, v, sl))
    scale = 1 / math.sqrt(d)
    ref_out, ref_lse = g.decode(q, k, v, sl, scale=scale, n_split=n_split)
    for _ in range(2):  # the scratch keeps the previous call's contents
        out = torch.full((B, H_q, d), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((B, H_q), float("nan"), dtype=torch.float32, device=DEV)
        st = g.gqa_attn_decode_noalloc(q, k, v, sl, B, S_max, H_q, H_kv, d, scale, n_split,
                                       out, lse)
        assert st == g.GQA_OK
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)


def test_noalloc_rejects_partials_larger_than_its_scratch():
    B, H_q, d, n_split = 8, 64, 128, 64  # 8*64*64*(128*4) bytes of O partials > 16 MiB
    assert g.gqa_attn_decode_workspace_bytes(B, H_q, d, n_split) > 16 << 20
    x = torch.empty(16, dtype=torch.bfloat16, device=DEV)
    lens = torch.ones(B, dtype=torch.int32, device=DEV)
    st = g.gqa_attn_decode_noalloc(x, x, x, lens, B, 128, H_q, 8, d, 0.1, n_split, x,
                                   torch.empty(1, device=DEV))
    assert st == g.GQA_ERR_INVALID_ARG
