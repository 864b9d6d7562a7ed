"""GPU parity of the FP8 (E4M3, per-token scale) KV-cache decode, contiguous and
paged, against the fp64 oracle."""
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


def _dev(*xs):
    return [x.to(DEV) for x in xs]


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("G", [1, 8, 16])
@pytest.mark.parametrize("ctx", [1, 63, 65, 1000])
def test_fp8_small_shapes(oracle_mod, d, G, ctx):
    S_max = -(-ctx // 4) * 4
    q, k8, v8, ks, vs, lens = inputs.decode_inputs_fp8(1, 2 * G, 2, d, S_max, seed=ctx + G + d,
                                                       seq_lens=[ctx])
    ref_o, ref_l = oracle_mod.decode_fp8(q, k8, v8, ks, vs, lens, 1 / math.sqrt(d))
    for n_split in (1, 3, None):
        out, lse = g.decode_fp8(*_dev(q, k8, v8, ks, vs, lens), n_split=n_split)
        torch.cuda.synchronize()
        assert_parity(out, lse, ref_o, ref_l, f"fp8 d={d} G={G} ctx={ctx} n_split={n_split}")


def _paginate_fp8(k8, v8, ks, vs, page_size, seed):
    B, S, H, d = k8.shape
    nb = -(-S // page_size)
    n_pages = B * nb + 3
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(seed))
    kp = torch.full((n_pages, page_size, H, d), 0x7F, dtype=torch.uint8)  # NaN codes
    vp = kp.clone()
    ksp = torch.full((n_pages, page_size), float("nan"))
    vsp = ksp.clone()
    table = torch.zeros(B, nb, dtype=torch.int32)
    for b in range(B):
        for j in range(nb):
            p = int(perm[b * nb + j])
            lo, hi = j * page_size, min(S, (j + 1) * page_size)
            kp[p, : hi - lo], vp[p, : hi - lo] = k8[b, lo:hi], v8[b, lo:hi]
            ksp[p, : hi - lo], vsp[p, : hi - lo] = ks[b, lo:hi], vs[b, lo:hi]
            table[b, j] = p
    return kp, vp, ksp, vsp, table


@pytest.mark.parametrize("page_size", [16, 64, 128])
def test_fp8_paged(oracle_mod, page_size):
    q, k8, v8, ks, vs, lens = inputs.decode_inputs_fp8(3, 16, 2, 128, 1024, seed=page_size,
                                                       seq_lens=[1024, 3, 611])
    ref_o, ref_l = oracle_mod.decode_fp8(q, k8, v8, ks, vs, lens, 1 / math.sqrt(128))
    kp, vp, ksp, vsp, table = _paginate_fp8(k8, v8, ks, vs, page_size, seed=1)
    for n_split in (1, 4, None):
        out, lse = g.decode_fp8(*_dev(q, kp, vp, ksp, vsp, lens), n_split=n_split,
                                block_table=table.to(DEV))
        torch.cuda.synchronize()
        assert_parity(out, lse, ref_o, ref_l, f"paged fp8 {page_size} n_split={n_split}")


def test_fp8_rejects_unaligned_scale_rows():
    x = torch.empty(64, dtype=torch.uint8, device=DEV)
    f = torch.empty(64, dtype=torch.float32, device=DEV)
    lens = torch.ones(1, dtype=torch.int32, device=DEV)
    q = torch.empty(8, 128, dtype=torch.bfloat16, device=DEV)
    st = g.gqa_attn_decode_fp8(q, x, x, f, f, lens, 1, 6, 8, 2, 128, 0.1, 1, None, q, f)
    assert st == g.GQA_ERR_UNSUPPORTED  # S_max % 4 != 0


def test_fp8_llama70b_decode_full_size(oracle_mod):
    cfg = inputs.LLAMA70B_DECODE
    q, k8, v8, ks, vs, lens = inputs.decode_inputs_fp8(cfg.B, cfg.H_q, cfg.H_kv, cfg.d, cfg.S_max,
                                                       seed=0)
    ref_o, ref_l = oracle_mod.decode_fp8(q, k8, v8, ks, vs, lens, cfg.scale)
    out, lse = g.decode_fp8(*_dev(q, k8, v8, ks, vs, lens))
    torch.cuda.synchronize()
    assert_parity(out, lse, ref_o, ref_l, "fp8 llama70b")
    assert np.isfinite(lse.cpu().numpy()).all()


def test_fp8_deterministic_across_runs():
    """Same input, same split count: bit-identical O and LSE (fixed merge order)."""
    q, k8, v8, ks, vs, lens = inputs.decode_inputs_fp8(2, 64, 8, 128, 5000, seed=21,
                                                       seq_lens=[5000, 1234])
    runs = []
    for _ in range(2):
        out, lse = g.decode_fp8(*_dev(q, k8, v8, ks, vs, lens))
        torch.cuda.synchronize()
        runs.append((out.cpu(), lse.cpu()))
    assert torch.equal(runs[0][0].view(torch.int16), runs[1][0].view(torch.int16))
    assert torch.equal(runs[0][1], runs[1][1])


def test_fp8_llama70b_one_wave_two_consumer_groups(oracle_mod):
    """19 splits = 152 CTAs, at most one per SM: the kernel with two groups of
    consumer warps taking alternate tiles and the deep stage ring."""
    cfg = inputs.LLAMA70B_DECODE
    q, k8, v8, ks, vs, lens = inputs.decode_inputs_fp8(cfg.B, cfg.H_q, cfg.H_kv, cfg.d, cfg.S_max,
                                                       seed=4)
    ref_o, ref_l = oracle_mod.decode_fp8(q, k8, v8, ks, vs, lens, cfg.scale)
    args = _dev(q, k8, v8, ks, vs, lens)
    runs = []
    for _ in range(2):
        out, lse = g.decode_fp8(*args, n_split=19)
        torch.cuda.synchronize()
        assert_parity(out, lse, ref_o, ref_l, "fp8 llama70b, 19 splits")
        runs.append((out.cpu(), lse.cpu()))
    assert torch.equal(runs[0][0].view(torch.int16), runs[1][0].view(torch.int16))
    assert torch.equal(runs[0][1], runs[1][1])


@pytest.mark.parametrize("page_size", [16, 128])
def test_fp8_paged_one_wave_ragged_tail(oracle_mod, page_size):
    # 2 sequences x 8 KV heads x 9 splits = 144 CTAs (one wave); lengths leave
    # partial tiles and partial pages at the ends of splits
    B, H_q, H_kv, d, S_max = 2, 64, 8, 128, 4000
    q, k8, v8, ks, vs, lens = inputs.decode_inputs_fp8(B, H_q, H_kv, d, S_max, seed=8,
                                                       seq_lens=[4000, 2777])
    ref_o, ref_l = oracle_mod.decode_fp8(q, k8, v8, ks, vs, lens, 1 / math.sqrt(d))
    kp, vp, ksp, vsp, table = _paginate_fp8(k8, v8, ks, vs, page_size, seed=9)
    out, lse = g.decode_fp8(*_dev(q, kp, vp, ksp, vsp, lens), n_split=9,
                            block_table=table.to(DEV))
    torch.cuda.synchronize()
    assert_parity(out, lse, ref_o, ref_l, f"paged fp8 one wave, page {page_size}")
