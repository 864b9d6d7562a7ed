"""GPU parity of the balanced-split decode (gqa_attn_decode_balanced) against
the fp64 oracle.

Each split streams its own share of the tiles and then claims tail tiles from a
counter shared by the splits of its (sequence, KV head); the partials are merged
by the same combine kernel.  Besides parity, every test checks that the claim
counters are back at zero after each call, since the next call relies on it.
Cache rows past each sequence length hold NaN, so a tile claimed or masked
wrongly fails the finiteness check.
"""
import math

import numpy as np
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


def _dev(*xs):
    return [x.to(DEV) for x in xs]


def _balanced(q, k, v, lens, n_split, counters=None):
    B, H_q, d = q.shape
    H_kv = k.shape[2]
    if counters is None:
        counters = g.decode_counters(B, H_kv)
    out, lse = g.decode(*_dev(q, k, v, lens), n_split=n_split, counters=counters)
    torch.cuda.synchronize()
    assert int(counters.abs().sum()) == 0, "claim counters not returned to zero"
    return out, lse


def test_counter_bytes():
    assert g.gqa_attn_decode_counter_bytes(3, 8) == 3 * 8 * 2 * 4
    assert g.gqa_attn_decode_counter_bytes(0, 8) == 0
    assert g.gqa_attn_decode_counter_bytes(1, 0) == 0


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("G", [1, 8, 16])
@pytest.mark.parametrize("ctx", [1, 63, 65, 129, 1000, 5000])
def test_balanced_small_shapes(oracle_mod, d, G, ctx):
    H_kv = 2
    q, k, v, lens = inputs.decode_inputs(1, G * H_kv, H_kv, d, ctx, seed=ctx + 5 * G + d)
    ref_o, ref_l = oracle_mod.decode(q, k, v, lens, 1 / math.sqrt(d))
    counters = g.decode_counters(1, H_kv)
    # 19 splits over 2 tiles: most splits have no share and claim nothing
    for n_split in (2, 7, 19, 76):
        out, lse = _balanced(q, k, v, lens, n_split, counters)
        assert_parity(out, lse, ref_o, ref_l, f"d={d} G={G} ctx={ctx} n_split={n_split}")


@pytest.mark.parametrize("B,S_max,lens", [(3, 300, [1, 299, 300]), (4, 1000, [64, 65, 999, 128]),
                                          (2, 5000, [4097, 17]), (5, 2048, [2048, 1, 700, 64, 1500])])
def test_balanced_ragged_batches(oracle_mod, B, S_max, lens):
    q, k, v, sl = inputs.decode_inputs(B, 32, 4, 128, S_max, seed=B + 40, seq_lens=lens)
    ref_o, ref_l = oracle_mod.decode(q, k, v, sl, 1 / math.sqrt(128))
    counters = g.decode_counters(B, 4)
    for n_split in (2, 3, 16, 33):
        out, lse = _balanced(q, k, v, sl, n_split, counters)
        assert_parity(out, lse, ref_o, ref_l, f"lens={lens} n_split={n_split}")


@pytest.mark.parametrize("cfg", inputs.DECODE_CONFIGS, ids=lambda c: c.name)
def test_balanced_full_size_workloads(oracle_mod, cfg):
    """The decode workloads at full size with the default split count (8 splits
    for the tiny decode, whose default is unsplit)."""
    q, k, v, lens = inputs.decode_inputs_for(cfg, seed=0)
    ref_o, ref_l = oracle_mod.decode(q, k, v, lens, cfg.scale)
    n = g.gqa_attn_decode_default_splits(cfg.B, cfg.H_kv, cfg.S_max)
    out, lse = _balanced(q, k, v, lens, n if n > 1 else 8)
    assert_parity(out, lse, ref_o, ref_l, cfg.name)


def test_balanced_counters_serve_consecutive_calls(oracle_mod):
    """One counter array across calls with other inputs, lengths and split counts."""
    counters = g.decode_counters(2, 8)
    for seed, lens, n_split in ((1, [4096, 4096], 19), (2, [333, 4000], 7), (3, [4096, 64], 40)):
        q, k, v, sl = inputs.decode_inputs(2, 64, 8, 128, 4096, seed=seed, seq_lens=lens)
        ref_o, ref_l = oracle_mod.decode(q, k, v, sl, 1 / math.sqrt(128))
        out, lse = _balanced(q, k, v, sl, n_split, counters)
        assert_parity(out, lse, ref_o, ref_l, f"seed={seed} n_split={n_split}")


def test_balanced_matches_fixed_splits():
    """Same inputs: the balanced and the fixed splits agree to rounding."""
    q, k, v, lens = inputs.decode_inputs(1, 64, 8, 128, 32768, seed=12)
    a_o, a_l = g.decode(*_dev(q, k, v, lens), n_split=19)
    b_o, b_l = _balanced(q, k, v, lens, 19)
    assert (a_o.float() - b_o.float()).abs().max().item() <= 2 ** -7
    assert (a_l - b_l).abs().max().item() <= 1e-5


def test_balanced_partials_merge_to_the_oracle(oracle_mod):
    """The partials the balanced kernel leaves in the workspace: each is a valid
    (m, l, O) (l > 0 with finite O, or the empty identity), and merging them with
    the associative merge in fp64 gives the oracle's O and LSE."""
    B, H_q, H_kv, d, S_max, n_split = 2, 16, 2, 128, 2000, 9
    q, k, v, sl = inputs.decode_inputs(B, H_q, H_kv, d, S_max, seed=31, seq_lens=[2000, 300])
    tau = 1 / math.sqrt(d)
    ref_o, ref_l = oracle_mod.decode(q, k, v, sl, tau)
    ws = g.decode_workspace(B, H_q, d, n_split)
    counters = g.decode_counters(B, H_kv)
    out = torch.empty(B, H_q, d, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, H_q, dtype=torch.float32, device=DEV)
    st = g.gqa_attn_decode_balanced(*_dev(q, k, v, sl), B, S_max, H_q, H_kv, d, tau, n_split, ws,
                                    counters, out, lse)
    assert st == g.GQA_OK
    torch.cuda.synchronize()
    assert int(counters.abs().sum()) == 0
    ml, Og = g.split_workspace(ws, B, H_q, d, n_split)
    ml, Og = ml.cpu().double().numpy(), Og.cpu().double().numpy()
    m, l = ml[..., 0], ml[..., 1]
    live = ~np.isneginf(m)
    assert (l[live] > 0).all() and np.isfinite(Og[live]).all()
    assert (l[~live] == 0).all()
    M = np.where(live, m, -np.inf).max(axis=-1, keepdims=True)
    w = np.where(live, np.exp(np.where(live, m, 0.0) - M), 0.0)
    Lsum = (w * np.where(live, l, 0.0)).sum(-1)
    O = (w[..., None] * np.where(live[..., None], Og, 0.0)).sum(-2) / Lsum[..., None]
    # the parity bar (P is rounded to bf16 for the P V product on the GPU)
    assert np.abs(O - ref_o).max() <= MAX_DO and np.abs(O - ref_o).mean() <= MEAN_DO
    assert np.abs(M[..., 0] + np.log(Lsum) - ref_l).max() <= MAX_DLSE


def test_balanced_bad_seq_len_leaves_counters_at_zero(oracle_mod):
    q, k, v, lens = inputs.decode_inputs(2, 8, 2, 64, 1024, seed=1)
    lens[1] = 1025  # past S_max: caught on the device
    counters = g.decode_counters(2, 2)
    out, lse = _balanced(q, k, v, lens, 5, counters)
    assert g.gqa_last_device_error() == g.GQA_ERR_INVALID_ARG
    assert torch.isnan(out[1].float()).all() and torch.isnan(lse[1]).all()
    assert torch.isfinite(out[0].float()).all() and torch.isfinite(lse[0]).all()
    assert g.gqa_last_device_error() == g.GQA_OK
    lens[1] = 1000
    ref_o, ref_l = oracle_mod.decode(q, k, v, lens, 1 / math.sqrt(64))
    out, lse = _balanced(q, k, v, lens, 5, counters)
    assert_parity(out, lse, ref_o, ref_l, "after a bad length")


def test_balanced_argument_checks():
    q, k, v, lens = _dev(*inputs.decode_inputs(1, 8, 2, 64, 256, seed=2))
    ws = g.decode_workspace(1, 8, 64, 4)
    out = torch.empty(1, 8, 64, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(1, 8, dtype=torch.float32, device=DEV)
    tau = 1 / math.sqrt(64)
    assert g.gqa_attn_decode_balanced(q, k, v, lens, 1, 256, 8, 2, 64, tau, 4, ws, None, out,
                                      lse) == g.GQA_ERR_INVALID_ARG
    c = torch.zeros(8, dtype=torch.int32, device=DEV)
    assert g.gqa_attn_decode_balanced(q, k, v, lens, 1, 256, 8, 2, 64, tau, 4, ws,
                                      c[1:].data_ptr() + 2, out, lse) == g.GQA_ERR_INVALID_ARG
    # one split: the plain decode, counters unused
    assert g.gqa_attn_decode_balanced(q, k, v, lens, 1, 256, 8, 2, 64, tau, 1, None, None, out,
                                      lse) == g.GQA_OK
    torch.cuda.synchronize()

