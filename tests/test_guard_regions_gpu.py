"""Guard regions around every output and workspace buffer (default build).

Each buffer handed to the library is the middle of a larger allocation whose
first and last 4 KiB hold a sentinel byte (0xA5).  After the call the
sentinels must be intact (no kernel wrote before or past its buffer) and no
element of out or lse may still hold the sentinel pattern (every output
element was written; a bf16 0xA5A5 or fp32 0xA5A5A5A5 is a magnitude near
3e-16 that these inputs cannot produce).  The split workspaces are checked at
their edges only: a split with no keys leaves its O rows unwritten by design.
"""
import pytest
import torch

import gqa_attention_gb300 as g
from gqa_attention_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096
SENT = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_gb300 import build

    build.build()
    g.load()
    yield
    assert g.gqa_last_device_error() == g.GQA_OK


class Guarded:
    """A buffer of `shape` x `dtype` (or `nbytes` raw bytes) inside sentinel guards."""

    def __init__(self, shape=None, dtype=torch.uint8, nbytes=None):
        esize = torch.empty((), dtype=dtype).element_size()
        n = nbytes if nbytes is not None else esize * int(torch.tensor(shape).prod())
        self.buf = torch.full((GUARD + n + GUARD,), SENT, dtype=torch.uint8, device=DEV)
        mid = self.buf[GUARD:GUARD + n]
        self.t = mid if nbytes is not None else mid.view(dtype).view(shape)

    def guards_intact(self):
        return bool((self.buf[:GUARD] == SENT).all()) and bool((self.buf[-GUARD:] == SENT).all())

    def fully_written(self):
        mid = self.buf[GUARD:-GUARD]
        w = self.t.element_size()
        words = mid.view(-1, w)
        return not bool((words == SENT).all(dim=1).any())


def _check(bufs, written):
    torch.cuda.synchronize()
    assert g.gqa_last_device_error() == g.GQA_OK
    for b in bufs:
        assert b.guards_intact()
    for b in written:
        assert b.fully_written()


def _decode_bufs(B, rows, H_q, d, n_split):
    out = Guarded(rows + (d,), torch.bfloat16)
    lse = Guarded(rows, torch.float32)
    ws = None
    if n_split > 1:
        ws = Guarded(nbytes=g.gqa_attn_decode_workspace_bytes(B, H_q, d, n_split))
    return out, lse, ws


@pytest.mark.parametrize("d,G,n_split", [(128, 8, 1), (128, 8, 6), (64, 4, 3), (32, 2, 5)])
def test_decode(d, G, n_split):
    B, H_q = 3, 2 * G
    q, k, v, sl = (x.to(DEV) for x in inputs.decode_inputs(B, H_q, 2, d, 1100, seed=d,
                                                           seq_lens=[1100, 1, 600]))
    out, lse, ws = _decode_bufs(B, (B, H_q), H_q, d, n_split)
    g.decode(q, k, v, sl, n_split=n_split, workspace=ws and ws.t, out=out.t, lse=lse.t)
    _check([b for b in (out, lse, ws) if b], [out, lse])


@pytest.mark.parametrize("T_q,G,n_split", [(2, 4, 3), (8, 8, 1), (8, 8, 4), (16, 8, 2)])
def test_decode_multi(T_q, G, n_split):
    B, H_q = 2, 2 * G
    gen = torch.Generator().manual_seed(T_q)
    q = torch.randn(B, T_q, H_q, 128, generator=gen).to(torch.bfloat16).to(DEV)
    k = torch.randn(B, 900, 2, 128, generator=gen).to(torch.bfloat16).to(DEV)
    v = torch.randn(B, 900, 2, 128, generator=gen).to(torch.bfloat16).to(DEV)
    sl = torch.tensor([900, T_q + 5], dtype=torch.int32, device=DEV)
    out, lse, ws = _decode_bufs(B * T_q, (B, T_q, H_q), H_q, 128, n_split)
    g.decode_multi(q, k, v, sl, n_split=n_split, workspace=ws and ws.t, out=out.t, lse=lse.t)
    _check([b for b in (out, lse, ws) if b], [out, lse])


def test_decode_fp8():
    q, k8, v8, ks, vs, sl = (x.to(DEV) for x in inputs.decode_inputs_fp8(
        2, 16, 2, 128, 1024, seed=3, seq_lens=[1024, 7]))
    out, lse, ws = _decode_bufs(2, (2, 16), 16, 128, 5)
    g.decode_fp8(q, k8, v8, ks, vs, sl, n_split=5, workspace=ws.t, out=out.t, lse=lse.t)
    _check([out, lse, ws], [out, lse])


def test_prefill_causal():
    q, k, v = (x.to(DEV) for x in inputs.prefill_inputs(2, 300, 16, 2, 128, seed=1))
    out = Guarded((2, 300, 16, 128), torch.bfloat16)
    lse = Guarded((2, 16, 300), torch.float32)
    g.prefill_causal(q, k, v, out=out.t, lse=lse.t)
    _check([out, lse], [out, lse])


@pytest.mark.parametrize("n_part", [1, 3])
def test_prefill_chunk(n_part):
    gen = torch.Generator().manual_seed(n_part)
    q = torch.randn(2, 150, 16, 128, generator=gen).to(torch.bfloat16).to(DEV)
    k = torch.randn(2, 800, 2, 128, generator=gen).to(torch.bfloat16).to(DEV)
    v = torch.randn(2, 800, 2, 128, generator=gen).to(torch.bfloat16).to(DEV)
    sl = torch.tensor([800, 333], dtype=torch.int32, device=DEV)
    out = Guarded((2, 150, 16, 128), torch.bfloat16)
    lse = Guarded((2, 16, 150), torch.float32)
    ws = None
    if n_part > 1:
        ws = Guarded(nbytes=g.gqa_attn_prefill_chunk_workspace_bytes(2, 150, 16, 128, n_part))
    g.prefill_chunk(q, k, v, sl, out=out.t, lse=lse.t, n_part=n_part, workspace=ws and ws.t)
    _check([b for b in (out, lse, ws) if b], [out, lse])
