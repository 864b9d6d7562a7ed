"""GPU parity of the paged-KV decode against the fp64 oracle and against the
contiguous decode on the same tokens."""
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


def _paginate(k, v, page_size, seed, spare=5):
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
            p = int(perm[b * nb + j])
            lo, hi = j * page_size, min(S, (j + 1) * page_size)
            kp[p, : hi - lo] = k[b, lo:hi]
            vp[p, : hi - lo] = v[b, lo:hi]
            table[b, j] = p
    return kp, vp, table


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("n_split", [1, 3, None])
def test_paged_matches_oracle_and_contiguous(oracle_mod, page_size, n_split):
    B, S_max, H_q, H_kv, d = 3, 1024, 16, 2, 128
    q, k, v, lens = inputs.decode_inputs(B, H_q, H_kv, d, S_max, seed=page_size,
                                         seq_lens=[1024, 1, 517])
    kp, vp, table = _paginate(k, v, page_size, seed=page_size)
    ref_o, ref_l = oracle_mod.decode_paged(q, kp, vp, table, lens, 1 / math.sqrt(d))
    if n_split is None:  # the paged default; the contiguous call below uses the same
        n_split = g.paged_default_splits(B, H_kv, table.shape[1] * page_size, d, page_size)
    out, lse = g.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), lens.to(DEV),
                              n_split=n_split)
    torch.cuda.synchronize()
    assert_parity(out, lse, ref_o, ref_l, f"page_size={page_size} n_split={n_split}")
    c_out, c_lse = g.decode(q.to(DEV), k.to(DEV), v.to(DEV), lens.to(DEV), n_split=n_split)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), c_out.view(torch.int16))  # same arithmetic
    assert torch.equal(lse, c_lse)


@pytest.mark.parametrize("d,G", [(32, 4), (64, 8), (128, 16)])
def test_paged_head_dims_and_groups(oracle_mod, d, G):
    q, k, v, lens = inputs.decode_inputs(2, 2 * G, 2, d, 300, seed=d, seq_lens=[300, 77])
    kp, vp, table = _paginate(k, v, 16, seed=d)
    ref_o, ref_l = oracle_mod.decode_paged(q, kp, vp, table, lens, 1 / math.sqrt(d))
    out, lse = g.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), lens.to(DEV),
                              n_split=2)
    torch.cuda.synchronize()
    assert_parity(out, lse, ref_o, ref_l, f"d={d} G={G}")


def test_paged_shared_prefix(oracle_mod):
    gen = torch.Generator().manual_seed(3)
    P, B_p, H_kv, d = 8, 16, 1, 128
    kp = torch.randn(P, B_p, H_kv, d, generator=gen).to(torch.bfloat16)
    vp = torch.randn(P, B_p, H_kv, d, generator=gen).to(torch.bfloat16)
    table = torch.tensor([[3, 1, 5, 7], [3, 1, 0, 2]], dtype=torch.int32)  # shared first 2 pages
    q = torch.randn(2, 4, d, generator=gen).to(torch.bfloat16)
    lens = torch.tensor([64, 40], dtype=torch.int32)
    ref_o, ref_l = oracle_mod.decode_paged(q, kp, vp, table, lens, 1 / math.sqrt(d))
    out, lse = g.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), lens.to(DEV))
    torch.cuda.synchronize()
    assert_parity(out, lse, ref_o, ref_l, "shared prefix")


def test_paged_bad_table_entry_gives_nan_and_error_word():
    q, k, v, lens = inputs.decode_inputs(2, 8, 2, 128, 256, seed=4)
    kp, vp, table = _paginate(k, v, 64, seed=1)
    table[1, 2] = kp.shape[0] + 7  # outside the pool
    out, lse = g.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), lens.to(DEV),
                              n_split=1)
    assert g.gqa_last_device_error() == g.GQA_ERR_INVALID_ARG
    assert torch.isnan(out[1].float()).all() and torch.isfinite(out[0].float()).all()


def test_paged_rejects_bad_host_arguments():
    x = torch.empty(64, dtype=torch.bfloat16, device=DEV)
    t = torch.zeros(4, dtype=torch.int32, device=DEV)
    args = dict(B=1, num_pages=4, page_size=24, max_blocks=4, H_q=8, H_kv=2, d=128)
    st = g.gqa_attn_decode_paged(x, x, x, t, t, args["B"], args["num_pages"], 24, 4, 8, 2, 128,
                                 0.1, 1, None, x, x)
    assert st == g.GQA_ERR_UNSUPPORTED  # page size not a power of two >= 16
    st = g.gqa_attn_decode_paged(x, x, x, None, t, 1, 4, 16, 4, 8, 2, 128, 0.1, 1, None, x, x)
    assert st == g.GQA_ERR_INVALID_ARG


@pytest.mark.parametrize("page_size", [16, 128])
def test_paged_llama70b_decode_full_size(oracle_mod, page_size):
    cfg = inputs.LLAMA70B_DECODE
    q, k, v, lens = inputs.decode_inputs_for(cfg, seed=0)
    kp, vp, table = _paginate(k, v, page_size, seed=7, spare=1)
    out, lse = g.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), lens.to(DEV))
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_mod.decode(q, k, v, lens, cfg.scale)
    assert_parity(out, lse, ref_o, ref_l, f"paged {page_size} llama70b")
    assert np.isfinite(lse.cpu().numpy()).all()


def test_paged_deterministic_across_runs():
    q, k, v, lens = inputs.decode_inputs(2, 64, 8, 128, 3000, seed=22, seq_lens=[3000, 777])
    kp, vp, table = _paginate(k, v, 16, seed=3)
    runs = []
    for _ in range(2):
        out, lse = g.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), lens.to(DEV))
        torch.cuda.synchronize()
        runs.append((out.cpu(), lse.cpu()))
    assert torch.equal(runs[0][0].view(torch.int16), runs[1][0].view(torch.int16))
    assert torch.equal(runs[0][1], runs[1][1])
