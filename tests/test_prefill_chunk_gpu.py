"""GPU parity of chunked prefill (queries ending a cached sequence) and of the
sliding-window mask, against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import gqa_attention_gb300 as g
from gqa_attention_gb300 import inputs

from parity import assert_parity

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


def _chunk_inputs(B, T_q, S_max, H_q, H_kv, lens, seed, d=128):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T_q, H_q, d, generator=gen).to(torch.bfloat16)
    k = torch.randn(B, S_max, H_kv, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, S_max, H_kv, d, generator=gen).to(torch.bfloat16)
    for b, L in enumerate(lens):  # rows past each sequence must never be read
        k[b, L:] = float("nan")
        v[b, L:] = float("nan")
    return q, k, v, torch.tensor(lens, dtype=torch.int32)


def _gpu(q, k, v, lens, window):
    out, lse = g.prefill_chunk(q.to(DEV), k.to(DEV), v.to(DEV),
                               None if lens is None else lens.to(DEV), window=window)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("T_q,S_max,lens", [(1, 300, [300, 1]), (5, 300, [5, 299]),
                                             (128, 1000, [1000, 128]), (200, 1000, [777, 1000]),
                                             (300, 300, [300, 300])])
@pytest.mark.parametrize("window", [-1, 0, 1, 127, 128, 300])
def test_chunk_small_shapes(oracle_mod, T_q, S_max, lens, window):
    q, k, v, sl = _chunk_inputs(2, T_q, S_max, 8, 2, lens, seed=T_q + S_max + window)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(128), seq_lens=sl,
                                                 window=window)
    out, lse = _gpu(q, k, v, sl, window)
    assert_parity(out, lse, ref_o, ref_l, f"T_q={T_q} S_max={S_max} lens={lens} W={window}")


@pytest.mark.parametrize("d", [64, 32])
@pytest.mark.parametrize("T_q,S_max,lens", [(5, 300, [5, 299]), (200, 1000, [777, 1000]),
                                             (300, 300, [300, 300])])
@pytest.mark.parametrize("window", [-1, 0, 127, 300])
def test_chunk_small_head_dims(oracle_mod, T_q, S_max, lens, window, d):
    q, k, v, sl = _chunk_inputs(2, T_q, S_max, 8, 2, lens, seed=T_q + window + d, d=d)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(d), seq_lens=sl,
                                                 window=window)
    out, lse = _gpu(q, k, v, sl, window)
    assert_parity(out, lse, ref_o, ref_l, f"d={d} T_q={T_q} lens={lens} W={window}")


@pytest.mark.parametrize("d", [64, 32])
@pytest.mark.parametrize("n_part", [2, 3])
def test_chunk_split_parts_small_head_dims(oracle_mod, d, n_part):
    q, k, v, sl = _chunk_inputs(2, 200, 3000, 4, 2, [3000, 700], seed=11 + d, d=d)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(d), seq_lens=sl,
                                                 window=-1)
    out, lse = g.prefill_chunk(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV), n_part=n_part)
    torch.cuda.synchronize()
    assert_parity(out.cpu(), lse.cpu(), ref_o, ref_l, f"d={d} n_part={n_part}")


@pytest.mark.parametrize("H_q,H_kv", [(2, 2), (3, 1)])
def test_chunk_odd_groups(oracle_mod, H_q, H_kv):
    q, k, v, sl = _chunk_inputs(1, 130, 400, H_q, H_kv, [333], seed=3)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(128), seq_lens=sl,
                                                 window=100)
    out, lse = _gpu(q, k, v, sl, 100)
    assert_parity(out, lse, ref_o, ref_l, f"H_q={H_q} H_kv={H_kv}")


def test_chunk_without_lengths_is_the_causal_prefill_bit_for_bit():
    q, k, v = inputs.prefill_inputs(1, 700, 8, 2, 128, seed=6)
    a_o, a_l = g.prefill_causal(q.to(DEV), k.to(DEV), v.to(DEV))
    b_o, b_l = g.prefill_chunk(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(a_o.view(torch.int16), b_o.view(torch.int16))
    assert torch.equal(a_l, b_l)


def test_chunk_bad_length_gives_nan_and_error_word():
    q, k, v, sl = _chunk_inputs(2, 64, 256, 4, 2, [256, 100], seed=2)
    sl[1] = 63  # shorter than the chunk
    out, lse = _gpu(q, k, v, sl, -1)
    assert g.gqa_last_device_error() == g.GQA_ERR_INVALID_ARG
    assert torch.isnan(out[1].float()).all() and torch.isnan(lse[1]).all()
    assert torch.isfinite(out[0].float()).all()


def test_chunk_rejects_bad_host_arguments():
    x = torch.empty(16, dtype=torch.bfloat16, device=DEV)
    st = g.gqa_attn_prefill_chunk(x, x, x, None, 1, 300, 200, 8, 2, 128, 0.1, -1, x, x)
    assert st == g.GQA_ERR_INVALID_ARG  # T_q > S_max
    st = g.gqa_attn_prefill_chunk(x, x, x, None, 1, 10, 200, 8, 2, 96, 0.1, -1, x, x)
    assert st == g.GQA_ERR_UNSUPPORTED  # d not in {32, 64, 128}


def test_sliding_window_prefill_8k_sampled_rows(oracle_mod):
    cfg = inputs.LLAMA70B_PREFILL_8K
    q, k, v = inputs.prefill_inputs_for(cfg, seed=1)
    rows = inputs.sample_rows(cfg.S, 128, seed=1)
    W = 4096
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, cfg.scale, window=W, rows=rows)
    out, lse = _gpu(q, k, v, None, W)
    r = rows.numpy()
    assert_parity(out[:, r], lse[:, :, r], ref_o, ref_l, "window 4096 over 8K")


def test_chunk_2048_at_the_end_of_a_32k_cache_sampled_rows(oracle_mod):
    B, T_q, S_max, H_q, H_kv = 1, 2048, 32768, 64, 8
    gen = torch.Generator().manual_seed(9)
    q = torch.randn(B, T_q, H_q, 128, generator=gen).to(torch.bfloat16)
    k = torch.randn(B, S_max, H_kv, 128, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, S_max, H_kv, 128, generator=gen).to(torch.bfloat16)
    sl = torch.tensor([30000], dtype=torch.int32)
    rows = inputs.sample_rows(T_q, 64, seed=2)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(128), seq_lens=sl,
                                                 rows=rows)
    out, lse = _gpu(q, k, v, sl, -1)
    r = rows.numpy()
    assert_parity(out[:, r], lse[:, :, r], ref_o, ref_l, "chunk 2048 @ 30000")
    assert np.isfinite(lse.numpy()).all()


# ---- key-axis split of the work items (gqa_attn_prefill_chunk_split) ----

@pytest.mark.parametrize("T_q,S_max,lens", [(1, 300, [300, 1]), (200, 1000, [777, 1000]),
                                             (300, 2600, [2600, 300]), (130, 4000, [3000, 4000])])
@pytest.mark.parametrize("window", [-1, 0, 200])
@pytest.mark.parametrize("n_part", [2, 3, 8])
def test_split_parts_match_oracle(oracle_mod, T_q, S_max, lens, window, n_part):
    # n_part 8 over items of 1-3 key tiles leaves parts empty (the merge identity)
    q, k, v, sl = _chunk_inputs(2, T_q, S_max, 8, 2, lens, seed=T_q + n_part + window)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(128), seq_lens=sl,
                                                 window=window)
    out, lse = g.prefill_chunk(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV), window=window,
                               n_part=n_part)
    torch.cuda.synchronize()
    assert_parity(out.cpu(), lse.cpu(), ref_o, ref_l,
                  f"split n_part={n_part} T_q={T_q} S_max={S_max} W={window}")


def test_split_matches_unsplit_within_rounding():
    q, k, v, sl = _chunk_inputs(1, 512, 6000, 16, 2, [5900], seed=8)
    a_o, a_l = _gpu(q, k, v, sl, -1)
    b_o, b_l = g.prefill_chunk(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV), n_part=4)
    torch.cuda.synchronize()
    assert (a_o.float() - b_o.cpu().float()).abs().max().item() <= 2 ** -7
    assert (a_l - b_l.cpu()).abs().max().item() <= 1e-5


def test_split_bad_length_gives_nan_and_error_word():
    q, k, v, sl = _chunk_inputs(2, 64, 3000, 4, 2, [3000, 100], seed=4)
    sl[1] = 63  # shorter than the chunk
    out, lse = g.prefill_chunk(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV), n_part=3)
    torch.cuda.synchronize()
    assert g.gqa_last_device_error() == g.GQA_ERR_INVALID_ARG
    assert torch.isnan(out[1].float()).all() and torch.isnan(lse[1]).all()
    assert torch.isfinite(out[0].float()).all() and torch.isfinite(lse[0]).all()


def test_split_rejects_bad_host_arguments():
    x = torch.empty(4096, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    f = torch.empty(64, dtype=torch.float32, device=DEV)
    args = (x, x, x, None, 1, 10, 200, 8, 2, 128, 0.1, -1)
    assert g.gqa_attn_prefill_chunk_split(*args, 0, ws, x, f) == g.GQA_ERR_INVALID_ARG
    assert g.gqa_attn_prefill_chunk_split(*args, 9, ws, x, f) == g.GQA_ERR_INVALID_ARG
    assert g.gqa_attn_prefill_chunk_split(*args, 2, None, x, f) == g.GQA_ERR_INVALID_ARG
    assert g.gqa_attn_prefill_chunk_split(*args, 2, ws[1:], x, f) == g.GQA_ERR_INVALID_ARG
    assert g.gqa_attn_prefill_chunk_workspace_bytes(1, 10, 8, 128, 1) == 0
    rows = 10 * 8
    assert g.gqa_attn_prefill_chunk_workspace_bytes(1, 10, 8, 128, 2) == \
        (rows * 2 * 8 + 255) // 256 * 256 + rows * 2 * 128 * 4


def test_default_parts_split_few_long_items_only():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert g.gqa_attn_prefill_chunk_default_parts(1, 2048, 1024 * 2, 64, 8) >= 1
    assert g.gqa_attn_prefill_chunk_default_parts(1, 64, 1024, 64, 8) == 1  # short items
    p = g.gqa_attn_prefill_chunk_default_parts(1, 2048, 32768, 64, 8)
    items = 16 * 8 * 4
    eff = lambda P: (items * P / sms) / math.ceil(items * P / sms)  # noqa: E731
    assert eff(p) >= eff(1)


def test_split_chunk_2048_at_the_end_of_a_32k_cache_sampled_rows(oracle_mod):
    B, T_q, S_max, H_q, H_kv = 1, 2048, 32768, 64, 8
    gen = torch.Generator().manual_seed(19)
    q = torch.randn(B, T_q, H_q, 128, generator=gen).to(torch.bfloat16)
    k = torch.randn(B, S_max, H_kv, 128, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, S_max, H_kv, 128, generator=gen).to(torch.bfloat16)
    sl = torch.tensor([31000], dtype=torch.int32)
    rows = inputs.sample_rows(T_q, 64, seed=3)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(128), seq_lens=sl,
                                                 rows=rows)
    n_part = g.gqa_attn_prefill_chunk_default_parts(B, T_q, S_max, H_q, H_kv)
    out, lse = g.prefill_chunk(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV), n_part=n_part)
    torch.cuda.synchronize()
    r = rows.numpy()
    assert_parity(out.cpu()[:, r], lse.cpu()[:, :, r], ref_o, ref_l, f"split chunk n_part={n_part}")


@pytest.mark.parametrize("n_part", [1, 3])
def test_chunk_deterministic_across_runs(n_part):
    q, k, v, sl = _chunk_inputs(2, 300, 3000, 8, 2, [3000, 2000], seed=24)
    runs = []
    for _ in range(2):
        out, lse = g.prefill_chunk(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV), window=500,
                                   n_part=n_part)
        torch.cuda.synchronize()
        runs.append((out.cpu(), lse.cpu()))
    assert torch.equal(runs[0][0].view(torch.int16), runs[1][0].view(torch.int16))
    assert torch.equal(runs[0][1], runs[1][1])
