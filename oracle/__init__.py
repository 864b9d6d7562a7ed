"""fp64 CPU oracle for grouped-query attention forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``gqa_attention_gb300``) never imports it, and the two share no code.

The arithmetic lives in ``gqa_oracle.c`` (plain C, fp64, libm exp/log); this
module only compiles it with gcc, marshals arrays and calls it.  What each entry
computes, with its sources:

* :func:`decode`: per (b, h) the three-pass safe softmax attention of the single
  query row over keys ``[0, seq_lens[b])`` ("Attention Kernel 계보" p.2 §1,
  p.3 §2, LSE p.3 §9), with query head h reading KV head ``h // (H_q // H_kv)``
  (p.15 §2) through an explicitly repeated KV head ("TileFoundry showcase",
  Stage0_Naive).
* :func:`prefill_causal_rows`: the same on chosen query rows of a causal prefill;
  row i sees keys ``[0, i]`` (p.13 §1).
* :func:`decode_partials`: per-split (m, l, O) with O unnormalised (p.4 §2, §8;
  p.18 §4 stage 1); empty splits are the identity (-inf, 0, 0) (p.4 §9).
* :func:`prefill_chunk_rows`: a chunk of T_q queries that are the last T_q
  tokens of each sequence (ADR-0060 §0.5.3 q_block_meta, §5.4): chunk row i of
  sequence b sits at position a = seq_lens[b] - T_q + i and sees keys
  a - window <= j <= a (the sliding window of p.13 §7; no lower bound when
  window < 0).
* :func:`decode_paged`: decode over a paged cache (p.17 §2-§4, p.18): token t
  of sequence b sits in page ``block_table[b][t // B_p]`` at offset
  ``t % B_p`` of the K and V pools ``[P, B_p, H_kv, d]``.
* :func:`decode_fp8`: decode over an FP8 (E4M3) cache with one scale per
  token (p.17 §7): key j is ``e4m3(k8[j]) * k_scale[j]``, likewise values.
* :func:`merge_partials`: the merge m = max, l = a_a l_a + a_b l_b,
  O = a_a O_a + a_b O_b folded over the splits, then O / l and m + ln l
  (p.4 §3, §8; p.18 §4 stage 2).

Inputs are CPU torch tensors (bfloat16 or float64) or numpy float64 arrays;
bf16 values are widened bit-exactly to fp64 inside the C code.  Outputs are
numpy float64 arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgqa_oracle.so")
_F64, _BF16 = 0, 1
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no target-specific flags)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P, I, D, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_int64
            lib.orc_decode.argtypes = [P, P, P, I, P, I, I, I, I, I, D, P, P, I]
            lib.orc_decode_partials.argtypes = [P, P, P, I, P, I, I, I, I, I, D, I, I, P, P, P, I]
            lib.orc_merge_partials.argtypes = [P, P, P, L, I, I, P, P]
            lib.orc_prefill_causal_rows.argtypes = [P, P, P, I, I, I, I, I, I, D, P, I, P, P, I]
            lib.orc_prefill_chunk_rows.argtypes = [P, P, P, I, P, I, I, I, I, I, I, D, I, P, I, P,
                                                   P, I]
            lib.orc_decode_paged.argtypes = [P, P, P, I, P, I, P, I, I, I, I, I, I, D, P, P, I]
            lib.orc_decode_fp8.argtypes = [P, I, P, P, P, P, P, I, I, I, I, I, D, P, P, I]
            lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_to_double.restype = ctypes.c_double
            for f in (lib.orc_decode, lib.orc_decode_partials, lib.orc_merge_partials,
                      lib.orc_prefill_causal_rows, lib.orc_prefill_chunk_rows,
                      lib.orc_decode_paged, lib.orc_decode_fp8):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _threads(nthreads):
    return int(nthreads) if nthreads else (os.cpu_count() or 1)


def _as_input(x):
    """Return (contiguous numpy array, dtype code) for a torch tensor or numpy array."""
    try:
        import torch  # noqa: F401  (only needed when torch tensors are passed)
        if isinstance(x, torch.Tensor):
            t = x.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), _BF16
            return t.to(torch.float64).numpy(), _F64
    except ImportError:
        pass
    a = np.ascontiguousarray(x)
    if a.dtype == np.uint16:
        return a, _BF16
    return np.ascontiguousarray(a, dtype=np.float64), _F64


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (code {rc})")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def decode(q, k, v, seq_lens, scale, nthreads=None):
    """q [B,H_q,d]; k,v [B,S_max,H_kv,d]; seq_lens [B] -> (out [B,H_q,d], lse [B,H_q])."""
    qa, qt = _as_input(q)
    ka, kt = _as_input(k)
    va, vt = _as_input(v)
    if not (qt == kt == vt):
        raise ValueError("q, k, v must share one dtype")
    B, H_q, d = qa.shape
    _, S_max, H_kv, d2 = ka.shape
    if d2 != d or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(B))
    out = np.empty((B, H_q, d))
    lse = np.empty((B, H_q))
    rc = _load().orc_decode(_ptr(qa), _ptr(ka), _ptr(va), qt, _ptr(sl), B, S_max, H_q, H_kv, d,
                            float(scale), _ptr(out), _ptr(lse), _threads(nthreads))
    _check(rc, "decode")
    return out, lse


def decode_partials(q, k, v, seq_lens, scale, n_split, chunk, nthreads=None):
    """Per-split partials: m, l [B,H_q,n_split]; O [B,H_q,n_split,d] (unnormalised)."""
    qa, qt = _as_input(q)
    ka, _ = _as_input(k)
    va, _ = _as_input(v)
    B, H_q, d = qa.shape
    _, S_max, H_kv, _ = ka.shape
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(B))
    m = np.empty((B, H_q, n_split))
    l = np.empty((B, H_q, n_split))
    O = np.empty((B, H_q, n_split, d))
    rc = _load().orc_decode_partials(_ptr(qa), _ptr(ka), _ptr(va), qt, _ptr(sl), B, S_max, H_q,
                                     H_kv, d, float(scale), int(n_split), int(chunk), _ptr(m),
                                     _ptr(l), _ptr(O), _threads(nthreads))
    _check(rc, "decode_partials")
    return m, l, O


def merge_partials(m, l, O):
    """m, l [..., n_split]; O [..., n_split, d] -> (out [..., d], lse [...])."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    O = np.ascontiguousarray(O, dtype=np.float64)
    lead = m.shape[:-1]
    n_split = m.shape[-1]
    d = O.shape[-1]
    R = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (d,))
    lse = np.empty(lead)
    rc = _load().orc_merge_partials(_ptr(m), _ptr(l), _ptr(O), R, n_split, d, _ptr(out), _ptr(lse))
    _check(rc, "merge_partials")
    return out, lse


def prefill_causal_rows(q, k, v, scale, rows=None, nthreads=None):
    """q [B,S,H_q,d]; k,v [B,S,H_kv,d]; rows: query positions (default all).

    Returns (out [B, n_rows, H_q, d], lse [B, H_q, n_rows]).
    """
    qa, qt = _as_input(q)
    ka, kt = _as_input(k)
    va, vt = _as_input(v)
    if not (qt == kt == vt):
        raise ValueError("q, k, v must share one dtype")
    B, S, H_q, d = qa.shape
    _, S2, H_kv, d2 = ka.shape
    if S2 != S or d2 != d or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    if rows is None:
        rows = np.arange(S, dtype=np.int64)
    ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    n_rows = ra.shape[0]
    out = np.empty((B, n_rows, H_q, d))
    lse = np.empty((B, H_q, n_rows))
    rc = _load().orc_prefill_causal_rows(_ptr(qa), _ptr(ka), _ptr(va), qt, B, S, H_q, H_kv, d,
                                         float(scale), _ptr(ra), n_rows, _ptr(out), _ptr(lse),
                                         _threads(nthreads))
    _check(rc, "prefill_causal_rows")
    return out, lse


def prefill_chunk_rows(q, k, v, scale, seq_lens=None, window=-1, rows=None, nthreads=None):
    """q [B,T_q,H_q,d]; k,v [B,S_max,H_kv,d]; seq_lens [B] (None: every sequence is S_max).

    Returns (out [B, n_rows, H_q, d], lse [B, H_q, n_rows]) for chunk rows `rows`
    (default all T_q rows).
    """
    qa, qt = _as_input(q)
    ka, kt = _as_input(k)
    va, vt = _as_input(v)
    if not (qt == kt == vt):
        raise ValueError("q, k, v must share one dtype")
    B, T_q, H_q, d = qa.shape
    _, S_max, H_kv, d2 = ka.shape
    if d2 != d or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    sl = None
    if seq_lens is not None:
        sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(B))
    if rows is None:
        rows = np.arange(T_q, dtype=np.int64)
    ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    n_rows = ra.shape[0]
    out = np.empty((B, n_rows, H_q, d))
    lse = np.empty((B, H_q, n_rows))
    rc = _load().orc_prefill_chunk_rows(_ptr(qa), _ptr(ka), _ptr(va), qt,
                                        _ptr(sl) if sl is not None else None, B, T_q, S_max, H_q,
                                        H_kv, d, float(scale), int(window), _ptr(ra), n_rows,
                                        _ptr(out), _ptr(lse), _threads(nthreads))
    _check(rc, "prefill_chunk_rows")
    return out, lse


def decode_paged(q, k_pool, v_pool, block_table, seq_lens, scale, nthreads=None):
    """q [B,H_q,d]; k_pool, v_pool [P,B_p,H_kv,d]; block_table [B,max_blocks]; seq_lens [B]."""
    qa, qt = _as_input(q)
    ka, kt = _as_input(k_pool)
    va, vt = _as_input(v_pool)
    if not (qt == kt == vt):
        raise ValueError("q, k, v must share one dtype")
    B, H_q, d = qa.shape
    P, B_p, H_kv, d2 = ka.shape
    if d2 != d or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    if bt.ndim != 2 or bt.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks]")
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(B))
    out = np.empty((B, H_q, d))
    lse = np.empty((B, H_q))
    rc = _load().orc_decode_paged(_ptr(qa), _ptr(ka), _ptr(va), qt, _ptr(bt), bt.shape[1],
                                  _ptr(sl), B, P, B_p, H_q, H_kv, d, float(scale), _ptr(out),
                                  _ptr(lse), _threads(nthreads))
    _check(rc, "decode_paged")
    return out, lse


def e4m3_to_double(code: int) -> float:
    """The oracle's decoding of one E4M3 byte."""
    return _load().orc_e4m3_to_double(int(code))


def decode_fp8(q, k8, v8, k_scale, v_scale, seq_lens, scale, nthreads=None):
    """q [B,H_q,d]; k8, v8 uint8 E4M3 codes [B,S_max,H_kv,d]; k_scale, v_scale [B,S_max]."""
    qa, qt = _as_input(q)
    k8a = np.ascontiguousarray(np.asarray(k8.cpu().numpy() if hasattr(k8, "cpu") else k8,
                                          dtype=np.uint8))
    v8a = np.ascontiguousarray(np.asarray(v8.cpu().numpy() if hasattr(v8, "cpu") else v8,
                                          dtype=np.uint8))
    ksa = np.ascontiguousarray(np.asarray(k_scale.cpu().numpy() if hasattr(k_scale, "cpu")
                                          else k_scale, dtype=np.float64))
    vsa = np.ascontiguousarray(np.asarray(v_scale.cpu().numpy() if hasattr(v_scale, "cpu")
                                          else v_scale, dtype=np.float64))
    B, H_q, d = qa.shape
    _, S_max, H_kv, d2 = k8a.shape
    if d2 != d or v8a.shape != k8a.shape or ksa.shape != (B, S_max) or vsa.shape != (B, S_max):
        raise ValueError("shape mismatch")
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(B))
    out = np.empty((B, H_q, d))
    lse = np.empty((B, H_q))
    rc = _load().orc_decode_fp8(_ptr(qa), qt, _ptr(k8a), _ptr(v8a), _ptr(ksa), _ptr(vsa), _ptr(sl),
                                B, S_max, H_q, H_kv, d, float(scale), _ptr(out), _ptr(lse),
                                _threads(nthreads))
    _check(rc, "decode_fp8")
    return out, lse
