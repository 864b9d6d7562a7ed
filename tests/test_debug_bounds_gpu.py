"""The bounds-checking build against the default build.

A library compiled with -DGQA_DEBUG_BOUNDS=1 checks every computed global
store of every kernel against the extent of the buffer that the kernel's own
parameters describe (out and lse: B x T_q x H_q rows; the split workspace:
rows x n_split partials); an index outside it skips the store and sets the
bounds bit, which gqa_last_device_error() reports as GQA_ERR_CUDA.  Each path
below runs on both libraries with the same inputs: the checking build must
report no bounds bit, and its outputs must equal the default build's bit for
bit (the checks change no arithmetic).  Covered: plain decode at d = 32, 64,
128 with and without splits (split kernel, combine, cluster-fused variant),
paged decode, FP8 decode (contiguous and paged), multi-token decode on both
kernels (mma.sync rows and the tensor-core tile, contiguous and paged),
causal prefill, chunk prefill (one part and split into parts, windowed), and
the bad-length paths that write NaN rows.  The balanced-split decode, whose
tail claims depend on timing, is compared to rounding instead of bit for bit.
"""
import math

import pytest
import torch

import gqa_attention_gb300 as g
from gqa_attention_gb300 import _binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def libs(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_gb300 import build

    build.build()
    release = g.load()
    d = tmp_path_factory.mktemp("bounds")
    path = build.build(extra_flags=["-DGQA_DEBUG_BOUNDS=1"],
                       lib_path=str(d / "libgqa_attn_bounds.so"), build_dir=str(d / "obj"))
    saved = _binding._lib
    _binding._lib = None
    try:
        checking = _binding.load(path)
    finally:
        _binding._lib = saved
    assert checking is not release
    yield release, checking
    _binding._lib = saved


def _run(handle, fn):
    """Run fn() with the binding's calls going to `handle`; return (outputs, status)."""
    saved = _binding._lib
    _binding._lib = handle
    try:
        torch.manual_seed(0)
        outs = fn()
        torch.cuda.synchronize()
        return [o.clone() for o in outs], g.gqa_last_device_error()
    finally:
        _binding._lib = saved


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _compare(libs, fn, expect=g.GQA_OK):
    release, checking = libs
    a, st_a = _run(release, fn)
    b, st_b = _run(checking, fn)
    assert st_a == expect, g.status_str(st_a)
    assert st_b == expect, f"checking build: {g.status_str(st_b)}"
    for x, y in zip(a, b):
        assert torch.equal(_bits(x), _bits(y))


def _dev(*xs):
    return [x.to(DEV) for x in xs]


def _paginate(caches, S, page_size, seed, spare=3):
    """Shuffled pages of [B, S, ...] caches; unused pages hold NaN (0x7f for E4M3 codes)."""
    B = caches[0].shape[0]
    nb = -(-S // page_size)
    n_pages = B * nb + spare
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(seed))
    pools = [torch.full((n_pages, page_size, *c.shape[2:]),
                        0x7F if c.dtype == torch.uint8 else float("nan"), dtype=c.dtype)
             for c in caches]
    table = torch.zeros(B, nb, dtype=torch.int32)
    for b in range(B):
        for j in range(nb):
            p = int(perm[b * nb + j])
            lo, hi = j * page_size, min(S, (j + 1) * page_size)
            for pool, c in zip(pools, caches):
                pool[p, : hi - lo] = c[b, lo:hi]
            table[b, j] = p
    return pools, table


@pytest.mark.parametrize("d,G,n_split", [(128, 8, 1), (128, 8, 5), (128, 8, None), (64, 4, 3),
                                         (32, 2, 7), (128, 16, 4)])
def test_decode(libs, d, G, n_split):
    q, k, v, sl = _dev(*inputs.decode_inputs(3, 2 * G, 2, d, 1500, seed=d + G,
                                             seq_lens=[1500, 1, 777]))
    _compare(libs, lambda: g.decode(q, k, v, sl, n_split=n_split))


@pytest.mark.parametrize("d,G,n_split", [(128, 8, 5), (64, 4, 19), (32, 2, 3)])
def test_balanced_decode(libs, d, G, n_split):
    q, k, v, sl = _dev(*inputs.decode_inputs(3, 2 * G, 2, d, 1500, seed=d + G + 1,
                                             seq_lens=[1500, 1, 777]))
    ctr = g.decode_counters(3, 2)
    release, checking = libs
    a, st_a = _run(release, lambda: g.decode(q, k, v, sl, n_split=n_split, counters=ctr))
    b, st_b = _run(checking, lambda: g.decode(q, k, v, sl, n_split=n_split, counters=ctr))
    assert st_a == g.GQA_OK, g.status_str(st_a)
    assert st_b == g.GQA_OK, f"checking build: {g.status_str(st_b)}"
    assert int(ctr.abs().sum()) == 0
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2 ** -7
    assert (a[1] - b[1]).abs().max().item() <= 1e-4


def test_decode_fused(libs):
    q, k, v, sl = _dev(*inputs.decode_inputs(2, 64, 8, 128, 4000, seed=3, seq_lens=[4000, 5]))
    _compare(libs, lambda: g.decode_fused(q, k, v, sl))


@pytest.mark.parametrize("page_size", [16, 128])
def test_decode_paged(libs, page_size):
    q, k, v, sl = inputs.decode_inputs(3, 16, 2, 128, 1000, seed=page_size,
                                       seq_lens=[1000, 2, 555])
    (kp, vp), table = _paginate([k, v], 1000, page_size, seed=page_size)
    q, kp, vp, table, sl = _dev(q, kp, vp, table, sl)
    _compare(libs, lambda: g.decode_paged(q, kp, vp, table, sl))


@pytest.mark.parametrize("paged", [False, True])
def test_decode_fp8(libs, paged):
    q, k8, v8, ks, vs, sl = inputs.decode_inputs_fp8(3, 16, 2, 128, 1024, seed=5,
                                                     seq_lens=[1024, 3, 611])
    table = None
    if paged:
        (k8, v8, ks, vs), table = _paginate([k8, v8, ks, vs], 1024, 64, seed=2)
        table = table.to(DEV)
    q, k8, v8, ks, vs, sl = _dev(q, k8, v8, ks, vs, sl)
    for n_split in (1, 4, None):
        _compare(libs, lambda: g.decode_fp8(q, k8, v8, ks, vs, sl, n_split=n_split,
                                            block_table=table))


def _multi_inputs(B, T_q, H_q, H_kv, S_max, lens, seed):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T_q, H_q, 128, generator=gen).to(torch.bfloat16)
    k = torch.randn(B, S_max, H_kv, 128, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, S_max, H_kv, 128, generator=gen).to(torch.bfloat16)
    for b, L in enumerate(lens):
        k[b, L:] = float("nan")
        v[b, L:] = float("nan")
    return q, k, v, torch.tensor(lens, dtype=torch.int32)


@pytest.mark.parametrize("T_q,G", [(2, 4), (2, 8), (8, 8), (16, 8)])  # mma.sync rows, then tc
@pytest.mark.parametrize("n_split", [1, None])
def test_decode_multi(libs, T_q, G, n_split):
    q, k, v, sl = _dev(*_multi_inputs(2, T_q, 2 * G, 2, 1200, [1200, T_q + 40], seed=T_q + G))
    _compare(libs, lambda: g.decode_multi(q, k, v, sl, n_split=n_split))


@pytest.mark.parametrize("T_q,page_size", [(2, 16), (8, 16), (8, 128)])
def test_decode_paged_multi(libs, T_q, page_size):
    q, k, v, sl = _multi_inputs(2, T_q, 16, 2, 1000, [1000, 3 * T_q + 37], seed=page_size)
    (kp, vp), table = _paginate([k, v], 1000, page_size, seed=T_q)
    q, kp, vp, table, sl = _dev(q, kp, vp, table, sl)
    _compare(libs, lambda: g.decode_paged(q, kp, vp, table, sl))


@pytest.mark.parametrize("S", [128, 300, 1000])
@pytest.mark.parametrize("d", [128, 64, 32])
def test_prefill_causal(libs, S, d):
    q, k, v = _dev(*inputs.prefill_inputs(2, S, 16, 2, d, seed=S + d))
    _compare(libs, lambda: g.prefill_causal(q, k, v))


@pytest.mark.parametrize("d", [64, 32])
@pytest.mark.parametrize("n_part,window", [(1, -1), (3, 200)])
def test_prefill_chunk_small_head_dims(libs, d, n_part, window):
    gen = torch.Generator().manual_seed(d + n_part)
    q = torch.randn(2, 200, 16, d, generator=gen).to(torch.bfloat16)
    k = torch.randn(2, 1000, 2, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(2, 1000, 2, d, generator=gen).to(torch.bfloat16)
    q, k, v, sl = _dev(q, k, v, torch.tensor([777, 1000], dtype=torch.int32))
    _compare(libs, lambda: g.prefill_chunk(q, k, v, sl, window=window, n_part=n_part))


@pytest.mark.parametrize("n_part,window", [(1, -1), (3, -1), (2, 200)])
def test_prefill_chunk(libs, n_part, window):
    q, k, v, sl = _dev(*_multi_inputs(2, 200, 16, 2, 1000, [777, 1000], seed=n_part))
    _compare(libs, lambda: g.prefill_chunk(q, k, v, sl, window=window, n_part=n_part))


def test_bad_lengths_write_nan_rows_in_bounds(libs):
    """A length past the cache: NaN rows and GQA_ERR_INVALID_ARG, no bounds bit."""
    q, k, v, sl = _dev(*inputs.decode_inputs(2, 16, 2, 128, 600, seed=9, seq_lens=[600, 100]))
    sl[1] = 601
    for n_split in (1, 3):
        _compare(libs, lambda: g.decode(q, k, v, sl, n_split=n_split), expect=g.GQA_ERR_INVALID_ARG)
    qm, km, vm, slm = _dev(*_multi_inputs(2, 8, 16, 2, 600, [600, 100], seed=9))
    slm[0] = 700
    for n_split in (1, 3):
        _compare(libs, lambda: g.decode_multi(qm, km, vm, slm, n_split=n_split),
                 expect=g.GQA_ERR_INVALID_ARG)
    _compare(libs, lambda: g.prefill_chunk(qm, km, vm, slm, n_part=2), expect=g.GQA_ERR_INVALID_ARG)
