"""GPU parity of the multi-token decode (the last T_q positions of each sequence,
causal among themselves) against the fp64 oracle's chunk rows, and against the
chunked prefill path.  Cache rows past each sequence length hold NaN.  With
d = 128 and more than 16 query rows per KV head the tensor-core kernel runs;
otherwise the mma.sync row groups do."""
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


def _inputs(B, T_q, S_max, H_q, H_kv, d, lens, seed):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T_q, H_q, d, generator=gen).to(torch.bfloat16)
    k = torch.randn(B, S_max, H_kv, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, S_max, H_kv, d, generator=gen).to(torch.bfloat16)
    for b, L in enumerate(lens):  # rows past each sequence must never be read
        k[b, L:] = float("nan")
        v[b, L:] = float("nan")
    return q, k, v, torch.tensor(lens, dtype=torch.int32)


def _multi(q, k, v, sl, n_split):
    out, lse = g.decode_multi(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV), n_split=n_split)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("T_q,G", [(1, 8), (2, 8), (4, 4), (3, 5), (16, 1), (2, 1), (4, 8),
                                   (3, 7), (8, 8), (5, 12), (64, 1)])
@pytest.mark.parametrize("n_split", [1, 3, None])
def test_matches_oracle_chunk_rows(oracle_mod, d, T_q, G, n_split):
    H_kv = 2
    lens = [T_q, 700, 64 + T_q]  # the shortest legal sequence, a long one, a tile edge
    q, k, v, sl = _inputs(3, T_q, 700, G * H_kv, H_kv, d, lens, seed=7 * T_q + G + d)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(d), seq_lens=sl)
    out, lse = _multi(q, k, v, sl, n_split)
    # the oracle's chunk LSE is [B, H_q, T_q]; multi-token decode writes [B, T_q, H_q]
    assert_parity(out, lse.transpose(1, 2), ref_o, ref_l,
                  f"multi d={d} T_q={T_q} G={G} n_split={n_split}")


def test_matches_chunked_prefill():
    q, k, v, sl = _inputs(2, 2, 3000, 64, 8, 128, [3000, 1234], seed=5)
    m_o, m_l = _multi(q, k, v, sl, None)
    c_o, c_l = g.prefill_chunk(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV))
    torch.cuda.synchronize()
    assert (m_o.float() - c_o.cpu().float()).abs().max().item() <= 2 ** -7
    assert (m_l.transpose(1, 2) - c_l.cpu()).abs().max().item() <= 2e-5


def test_t_q_1_is_plain_decode_bit_for_bit():
    q, k, v, sl = inputs.decode_inputs(2, 16, 2, 128, 900, seed=3, seq_lens=[900, 77])
    for n_split in (1, 4):
        a_o, a_l = g.decode(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV), n_split=n_split)
        b_o, b_l = g.decode_multi(q[:, None].to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV),
                                  n_split=n_split)
        torch.cuda.synchronize()
        assert torch.equal(a_o.view(torch.int16), b_o[:, 0].view(torch.int16))
        assert torch.equal(a_l, b_l[:, 0])


def test_length_shorter_than_t_q_gives_nan_and_error_word():
    q, k, v, sl = _inputs(2, 4, 256, 8, 2, 64, [256, 3], seed=2)  # 3 < T_q
    out, lse = _multi(q, k, v, sl, 2)
    assert g.gqa_last_device_error() == g.GQA_ERR_INVALID_ARG
    assert torch.isnan(out[1].float()).all() and torch.isnan(lse[1]).all()
    assert torch.isfinite(out[0].float()).all() and torch.isfinite(lse[0]).all()


def test_rejects_bad_host_arguments():
    # every call below fails a host check before any launch
    x = torch.empty(4096, dtype=torch.bfloat16, device=DEV)
    t = torch.ones(2, dtype=torch.int32, device=DEV)
    f = torch.empty(64, dtype=torch.float32, device=DEV)
    # d = 64, T_q * G = 9 * 8 = 72 rows: more than four row groups of 16
    assert g.gqa_attn_decode_multi(x, x, x, t, 1, 9, 64, 16, 2, 64, 0.1, 1, None, x, f) == \
        g.GQA_ERR_UNSUPPORTED
    # d = 128, T_q * G = 17 * 8 = 136 rows: more than one tensor-core tile
    assert g.gqa_attn_decode_multi(x, x, x, t, 1, 17, 64, 16, 2, 128, 0.1, 1, None, x, f) == \
        g.GQA_ERR_UNSUPPORTED
    assert g.gqa_attn_decode_multi(x, x, x, t, 1, 0, 64, 8, 2, 128, 0.1, 1, None, x, f) == \
        g.GQA_ERR_INVALID_ARG
    assert g.gqa_attn_decode_multi(x, x, x, t, 1, 65, 64, 1, 1, 128, 0.1, 1, None, x, f) == \
        g.GQA_ERR_INVALID_ARG  # T_q > S_max (and > 16)
    assert g.gqa_attn_decode_multi(x, x, x, t, 1, 2, 64, 8, 2, 128, 0.1, 3, None, x, f) == \
        g.GQA_ERR_INVALID_ARG  # n_split > 1 without a workspace


@pytest.mark.parametrize("T_q,G,H_kv", [(9, 8, 2), (16, 8, 2), (32, 4, 2), (64, 2, 1), (2, 16, 2),
                                        (6, 3, 3), (40, 3, 1)])
@pytest.mark.parametrize("n_split", [1, 4, None])
def test_tensor_core_rows_match_oracle(oracle_mod, T_q, G, H_kv, n_split):
    """d = 128 with 17..128 query rows per KV head (one tensor-core tile): a
    sequence of exactly T_q tokens, a long one and one ending just past a
    128-key tile; cache rows past each length hold NaN."""
    lens = [T_q, 1000, 128 + T_q]
    q, k, v, sl = _inputs(3, T_q, 1000, G * H_kv, H_kv, 128, lens, seed=T_q * 31 + G)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(128), seq_lens=sl)
    out, lse = _multi(q, k, v, sl, n_split)
    assert_parity(out, lse.transpose(1, 2), ref_o, ref_l, f"tc T_q={T_q} G={G} n_split={n_split}")


def test_tensor_core_rows_match_chunked_prefill():
    q, k, v, sl = _inputs(2, 8, 3000, 64, 8, 128, [3000, 1234], seed=9)
    m_o, m_l = _multi(q, k, v, sl, None)
    c_o, c_l = g.prefill_chunk(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV))
    torch.cuda.synchronize()
    assert (m_o.float() - c_o.cpu().float()).abs().max().item() <= 2 ** -7
    assert (m_l.transpose(1, 2) - c_l.cpu()).abs().max().item() <= 2e-5


def test_tensor_core_length_shorter_than_t_q_gives_nan_and_error_word():
    q, k, v, sl = _inputs(2, 4, 512, 16, 2, 128, [512, 3], seed=4)  # 32 rows; 3 < T_q
    for n_split in (1, 3):
        out, lse = _multi(q, k, v, sl, n_split)
        assert g.gqa_last_device_error() == g.GQA_ERR_INVALID_ARG
        assert torch.isnan(out[1].float()).all() and torch.isnan(lse[1]).all()
        assert torch.isfinite(out[0].float()).all() and torch.isfinite(lse[0]).all()


def test_tensor_core_outputs_stay_inside_their_buffers():
    B, T_q, H_q, H_kv, d = 2, 8, 16, 2, 128
    q, k, v, sl = _inputs(B, T_q, 700, H_q, H_kv, d, [700, 9], seed=5)
    pad = 4096
    n = B * T_q * H_q
    out_buf = torch.full((n * d + 2 * pad,), 7.0, dtype=torch.bfloat16, device=DEV)
    lse_buf = torch.full((n + 2 * pad,), 7.0, dtype=torch.float32, device=DEV)
    out = out_buf[pad: pad + n * d].view(B, T_q, H_q, d)
    lse = lse_buf[pad: pad + n].view(B, T_q, H_q)
    g.decode_multi(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV), n_split=3, out=out, lse=lse)
    torch.cuda.synchronize()
    for buf, m in ((out_buf, n * d), (lse_buf, n)):
        assert (buf[:pad].float() == 7.0).all() and (buf[pad + m:].float() == 7.0).all()


@pytest.mark.parametrize("T_q", [2, 4, 8, 16])
def test_llama70b_verification_full_size(oracle_mod, T_q):
    """T_q query tokens ending a 32768-token Llama3-70B cache (G = 8: 8 T_q rows)."""
    q, k, v, sl = _inputs(1, T_q, 32768, 64, 8, 128, [32768], seed=11 + T_q)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(128), seq_lens=sl)
    out, lse = _multi(q, k, v, sl, None)
    assert_parity(out, lse.transpose(1, 2), ref_o, ref_l, f"multi T_q={T_q} llama70b 32K")
    assert np.isfinite(lse.numpy()).all()


def _paginate(k, v, page_size, seed, spare=3):
    """Scatter a contiguous cache [B, S, H, d] into shuffled pages; unused pages hold NaN."""
    B, S, H, d = k.shape
    nb = -(-S // page_size)
    n_pages = B * nb + spare
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(seed))
    kp = torch.full((n_pages, page_size, H, d), float("nan"), dtype=k.dtype)
    vp = torch.full_like(kp, float("nan"))
    table = torch.zeros(B, nb, dtype=torch.int32)
    for b in range(B):
        for j in range(nb):
            pg = int(perm[b * nb + j])
            lo, hi = j * page_size, min(S, (j + 1) * page_size)
            kp[pg, : hi - lo] = k[b, lo:hi]
            vp[pg, : hi - lo] = v[b, lo:hi]
            table[b, j] = pg
    return kp, vp, table


@pytest.mark.parametrize("page_size", [16, 64, 256])
@pytest.mark.parametrize("T_q,G", [(2, 8), (4, 4), (3, 2), (4, 8)])
def test_paged_multi_matches_oracle_and_contiguous(oracle_mod, page_size, T_q, G):
    H_kv = 2
    q, k, v, sl = _inputs(2, T_q, 1000, G * H_kv, H_kv, 128, [1000, 3 * T_q + 37],
                          seed=page_size + T_q)
    kp, vp, table = _paginate(k, v, page_size, seed=T_q)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(128), seq_lens=sl)
    n = g.paged_default_splits(2, H_kv, table.shape[1] * page_size, 128, page_size)
    out, lse = g.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV),
                              n_split=n)
    torch.cuda.synchronize()
    assert_parity(out.cpu(), lse.cpu().transpose(1, 2), ref_o, ref_l,
                  f"paged multi page={page_size} T_q={T_q} G={G}")
    c_o, c_l = _multi(q, k, v, sl, n)
    if T_q * G <= 16:  # both run the same mma.sync arithmetic
        assert torch.equal(out.cpu().view(torch.int16), c_o.view(torch.int16))
        assert torch.equal(lse.cpu(), c_l)
    else:  # the contiguous cache runs the tensor-core kernel: rounding only
        assert (out.cpu().float() - c_o.float()).abs().max().item() <= 2 ** -7
        assert (lse.cpu() - c_l).abs().max().item() <= 2e-5


@pytest.mark.parametrize("page_size", [16, 32, 128, 256])
@pytest.mark.parametrize("T_q,G", [(8, 8), (16, 8), (5, 4)])
def test_paged_tensor_core_rows_match_oracle_and_contiguous(oracle_mod, page_size, T_q, G):
    """d = 128 with more than 16 rows per KV head over a paged cache: each
    128-key tile arrives as one box per page; unused pages hold NaN."""
    H_kv = 2
    q, k, v, sl = _inputs(2, T_q, 1500, G * H_kv, H_kv, 128, [1500, 2 * T_q + 129],
                          seed=page_size + 3 * T_q)
    kp, vp, table = _paginate(k, v, page_size, seed=T_q + 1)
    ref_o, ref_l = oracle_mod.prefill_chunk_rows(q, k, v, 1 / math.sqrt(128), seq_lens=sl)
    for n_split in (1, 5):
        out, lse = g.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV),
                                  n_split=n_split)
        torch.cuda.synchronize()
        assert_parity(out.cpu(), lse.cpu().transpose(1, 2), ref_o, ref_l,
                      f"paged tc page={page_size} T_q={T_q} G={G} n_split={n_split}")
        c_o, c_l = _multi(q, k, v, sl, n_split)  # the same tiles, contiguous
        assert torch.equal(out.cpu().view(torch.int16), c_o.view(torch.int16))
        assert torch.equal(lse.cpu(), c_l)


def test_paged_tensor_core_bad_table_entry_gives_nan_and_error_word():
    q, k, v, sl = _inputs(2, 8, 512, 16, 2, 128, [512, 512], seed=8)  # 64 rows per KV head
    kp, vp, table = _paginate(k, v, 64, seed=2)
    table[1, 3] = kp.shape[0] + 5  # outside the pool
    out, lse = g.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), sl.to(DEV),
                              n_split=2)
    torch.cuda.synchronize()
    assert g.gqa_last_device_error() == g.GQA_ERR_INVALID_ARG
    assert torch.isnan(out[1].float()).all() and torch.isnan(lse[1]).all()
    assert torch.isfinite(out[0].float()).all() and torch.isfinite(lse[0]).all()


@pytest.mark.parametrize("T_q", [2, 8])  # mma.sync row group, tensor-core tile
def test_deterministic_across_runs(T_q):
    q, k, v, sl = _inputs(2, T_q, 3000, 64, 8, 128, [3000, 1500], seed=23 + T_q)
    a = _multi(q, k, v, sl, None)
    b = _multi(q, k, v, sl, None)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])
