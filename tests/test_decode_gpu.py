"""GPU parity of split-KV decode and the combine kernel against the fp64 oracle.

Calls go through the C ABI (ctypes binding).  Inputs come from the seeded
generators in ``gqa_attention_gb300.inputs``; cache rows past each sequence
length hold NaN, so any unmasked read of padding fails the finiteness check.
"""
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


def _run(q, k, v, lens, n_split, scale=None):
    qd, kd, vd, ld = (x.to(DEV) for x in (q, k, v, lens))
    out, lse = g.decode(qd, kd, vd, ld, scale=scale, n_split=n_split)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("G", [1, 4, 8, 16])
@pytest.mark.parametrize("ctx", [1, 2, 15, 63, 64, 65, 127, 129, 1000])
def test_small_shapes(oracle_mod, d, G, ctx):
    H_kv = 2
    q, k, v, lens = inputs.decode_inputs(1, G * H_kv, H_kv, d, ctx, seed=ctx + 7 * G + d)
    ref_o, ref_l = oracle_mod.decode(q, k, v, lens, 1 / math.sqrt(d))
    for n_split in (1, 2, 7, None):
        out, lse = _run(q, k, v, lens, n_split)
        assert_parity(out, lse, ref_o, ref_l, f"d={d} G={G} ctx={ctx} n_split={n_split}")


@pytest.mark.parametrize("B,S_max,lens", [(3, 300, [1, 299, 300]), (4, 1000, [64, 65, 999, 128]),
                                          (2, 5000, [4097, 17])])
def test_ragged_batches(oracle_mod, B, S_max, lens):
    q, k, v, sl = inputs.decode_inputs(B, 32, 4, 128, S_max, seed=B, seq_lens=lens)
    ref_o, ref_l = oracle_mod.decode(q, k, v, sl, 1 / math.sqrt(128))
    for n_split in (1, 3, 16, None):
        out, lse = _run(q, k, v, sl, n_split)
        assert_parity(out, lse, ref_o, ref_l, f"lens={lens} n_split={n_split}")


def test_partials_match_oracle_partials(oracle_mod):
    B, H_q, H_kv, d, S_max, n_split = 2, 16, 2, 128, 777, 5
    q, k, v, sl = inputs.decode_inputs(B, H_q, H_kv, d, S_max, seed=3, seq_lens=[777, 200])
    chunk = -(-(-(-S_max // n_split)) // 64) * 64  # ceil(S_max/n_split) rounded up to 64
    assert g.gqa_attn_decode_split_chunk(S_max, n_split) == chunk
    tau = 1 / math.sqrt(d)
    m, l, O = oracle_mod.decode_partials(q, k, v, sl, tau, n_split, chunk)
    ws = g.decode_workspace(B, H_q, d, n_split)
    out = torch.empty(B, H_q, d, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, H_q, dtype=torch.float32, device=DEV)
    st = g.gqa_attn_decode(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV), B, S_max, H_q, H_kv, d,
                           tau, n_split, ws, out, lse)
    assert st == g.GQA_OK
    torch.cuda.synchronize()
    ml, Og = g.split_workspace(ws, B, H_q, d, n_split)
    ml, Og = ml.cpu().double().numpy(), Og.cpu().double().numpy()
    empty = np.isneginf(m)
    assert (np.isneginf(ml[..., 0]) == empty).all()
    assert (ml[..., 1][empty] == 0).all()
    ne = ~empty
    # per-split LSE and normalised output (independent of the reference point
    # m), over the non-empty splits only (an empty split has l = 0)
    np.testing.assert_allclose(ml[..., 0][ne] + np.log(ml[..., 1][ne]), m[ne] + np.log(l[ne]),
                               atol=1e-3)
    np.testing.assert_allclose(Og[ne] / ml[..., 1][ne][:, None], O[ne] / l[ne][:, None], atol=1e-2)


def test_combine_merges_arbitrary_partials(oracle_mod):
    rng = np.random.default_rng(0)
    B, H_q, d, n_split = 2, 8, 64, 9
    m = rng.standard_normal((B, H_q, n_split)) * 4
    l = rng.uniform(0.5, 50, (B, H_q, n_split))
    O = rng.standard_normal((B, H_q, n_split, d)) * l[..., None]
    m[0, 0, :4] = -np.inf   # empty splits are skipped
    l[0, 0, :4] = 0
    O[0, 0, :4] = np.nan    # ... and their O is never read
    ws = g.decode_workspace(B, H_q, d, n_split)
    ml_v, O_v = g.split_workspace(ws, B, H_q, d, n_split)
    ml_v.copy_(torch.from_numpy(np.stack([m, l], -1)).float())
    O_v.copy_(torch.from_numpy(O).float())
    out = torch.empty(B, H_q, d, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, H_q, dtype=torch.float32, device=DEV)
    assert g.gqa_attn_decode_combine(ws, B, H_q, d, n_split, out, lse) == g.GQA_OK
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_mod.merge_partials(m.astype(np.float32).astype(np.float64),
                                             l.astype(np.float32).astype(np.float64),
                                             np.nan_to_num(O.astype(np.float32).astype(np.float64)))
    assert_parity(out, lse, ref_o, ref_l, "combine")


def test_deterministic_across_runs():
    q, k, v, lens = inputs.decode_inputs(1, 64, 8, 128, 4096, seed=11)
    a = _run(q, k, v, lens, None)
    b = _run(q, k, v, lens, None)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])


def test_outputs_stay_inside_their_buffers():
    B, H_q, H_kv, d = 2, 16, 2, 128
    q, k, v, lens = inputs.decode_inputs(B, H_q, H_kv, d, 700, seed=5, seq_lens=[700, 3])
    pad = 4096
    out_buf = torch.full((B * H_q * d + 2 * pad,), 7.0, dtype=torch.bfloat16, device=DEV)
    lse_buf = torch.full((B * H_q + 2 * pad,), 7.0, dtype=torch.float32, device=DEV)
    out = out_buf[pad: pad + B * H_q * d].view(B, H_q, d)
    lse = lse_buf[pad: pad + B * H_q].view(B, H_q)
    g.decode(q.to(DEV), k.to(DEV), v.to(DEV), lens.to(DEV), n_split=4, out=out, lse=lse)
    torch.cuda.synchronize()
    for buf, n in ((out_buf, B * H_q * d), (lse_buf, B * H_q)):
        assert (buf[:pad].float() == 7.0).all() and (buf[pad + n:].float() == 7.0).all()


def test_bad_seq_len_gives_nan_and_error_word():
    q, k, v, lens = inputs.decode_inputs(2, 8, 2, 64, 128, seed=1)
    lens[1] = 129  # past S_max: caught on the device
    for n_split in (1, 3):
        out, lse = _run(q, k, v, lens, n_split)
        assert g.gqa_last_device_error() == g.GQA_ERR_INVALID_ARG
        assert torch.isnan(out[1].float()).all() and torch.isnan(lse[1]).all()
        assert torch.isfinite(out[0].float()).all() and torch.isfinite(lse[0]).all()
    assert g.gqa_last_device_error() == g.GQA_OK


def test_wait_timeout_is_reported_and_context_survives(oracle_mod):
    assert g.gqa_selftest_wait_timeout(2_000_000) == g.GQA_OK  # 2 ms limit
    assert g.gqa_last_device_error() == g.GQA_ERR_TIMEOUT
    assert g.gqa_last_device_error() == g.GQA_OK  # cleared
    q, k, v, lens = inputs.decode_inputs(1, 8, 2, 32, 100, seed=2)
    out, lse = _run(q, k, v, lens, 2)
    ref_o, ref_l = oracle_mod.decode(q, k, v, lens, 1 / math.sqrt(32))
    assert_parity(out, lse, ref_o, ref_l, "after timeout")


@pytest.mark.parametrize("cfg", inputs.DECODE_CONFIGS, ids=lambda c: c.name)
def test_full_size_workloads(oracle_mod, cfg):
    """The three decode workloads at full size with the default split count."""
    q, k, v, lens = inputs.decode_inputs_for(cfg, seed=0)
    ref_o, ref_l = oracle_mod.decode(q, k, v, lens, cfg.scale)
    out, lse = _run(q, k, v, lens, None)
    assert_parity(out, lse, ref_o, ref_l, cfg.name)


@pytest.mark.parametrize("B,H_q,H_kv,d,n_split", [
    (1, 64, 8, 128, 19),    # 64 rows, <= 32 splits: column-per-warp combine
    (2, 16, 2, 128, 32),    # the largest split count it takes
    (2, 16, 2, 128, 33),    # one more: four warps of split groups (16 per round)
    (16, 64, 8, 128, 19),   # 1024 rows: more than four per SM, split groups of 8
    (16, 64, 8, 64, 40),    # many rows and splits
    (3, 8, 2, 32, 9),       # d = 32 on the column kernel
])
def test_combine_routes(oracle_mod, B, H_q, H_kv, d, n_split):
    """Every combine variant the launcher can pick, including empty splits."""
    S_max = 700
    lens = [S_max] + [1 + (97 * b) % S_max for b in range(1, B)]
    q, k, v, sl = inputs.decode_inputs(B, H_q, H_kv, d, S_max, seed=B + n_split, seq_lens=lens)
    ref_o, ref_l = oracle_mod.decode(q, k, v, sl, 1 / math.sqrt(d))
    out, lse = _run(q, k, v, sl, n_split)
    assert_parity(out, lse, ref_o, ref_l, f"B={B} d={d} n_split={n_split}")


@pytest.mark.parametrize("d", [32, 64])
@pytest.mark.parametrize("G,ctx", [(4, 5000), (8, 1024), (16, 131), (1, 3)])
def test_small_grid_and_full_grid_paths(oracle_mod, d, G, ctx):
    """The same sequence alone (2 CTAs, every CTA resident at once: the L2
    prefetch across the dependency wait is on) and as every member of a batch of
    160 (more CTAs than fit at once: the prefetch is off), against the oracle."""
    H_kv = 2
    q, k, v, lens = inputs.decode_inputs(1, G * H_kv, H_kv, d, ctx, seed=d + G + ctx)
    ref_o, ref_l = oracle_mod.decode(q, k, v, lens, 1 / math.sqrt(d))
    small_o, small_l = _run(q, k, v, lens, 1)  # 2 CTAs
    assert_parity(small_o, small_l, ref_o, ref_l, f"small grid d={d} G={G} ctx={ctx}")
    B = 160  # 320 CTAs: more than two per SM
    qb, kb, vb, lb = (x.expand(B, *x.shape[1:]).contiguous() for x in (q, k, v, lens))
    big_o, big_l = _run(qb, kb, vb, lb, 1)
    for b in (0, B - 1):
        assert_parity(big_o[b:b + 1], big_l[b:b + 1], ref_o, ref_l,
                      f"full grid d={d} G={G} ctx={ctx} b={b}")
