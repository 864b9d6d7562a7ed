"""ctypes binding of libgqa_attn.so (declared in ``include/gqa_attn.h``).

Argument marshalling only: every step of the attention runs in the library's
CUDA kernels.  The functions named like the C entry points take torch CUDA
tensors (or raw integers for pointers) and return the C status code; the
helpers at the bottom allocate outputs with torch and raise on a bad status.
There is no CPU fallback: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgqa_attn.so")

GQA_OK, GQA_ERR_INVALID_ARG, GQA_ERR_UNSUPPORTED, GQA_ERR_CUDA, GQA_ERR_TIMEOUT = range(5)

#: Every symbol the header declares, with (restype, argtypes).
_P, _I, _F, _SZ, _U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64
SIGNATURES = {
    "gqa_status_str": (ctypes.c_char_p, [_I]),
    "gqa_version": (_I, []),
    "gqa_attn_decode_split_chunk": (_I, [_I, _I]),
    "gqa_attn_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "gqa_attn_decode_default_splits": (_I, [_I, _I, _I, _I]),
    "gqa_attn_decode": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P]),
    "gqa_attn_decode_combine": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "gqa_attn_decode_counter_bytes": (_SZ, [_I, _I]),
    "gqa_attn_decode_balanced": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P,
                                      _P]),
    "gqa_attn_decode_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P]),
    "gqa_attn_decode_paged": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P,
                                   _P, _P]),
    "gqa_attn_decode_fp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P,
                                 _P]),
    "gqa_attn_decode_paged_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                                       _I, _P, _P, _P, _P]),
    "gqa_attn_decode_multi": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P]),
    "gqa_attn_decode_multi_default_splits": (_I, [_I, _I, _I, _I, _I, _I]),
    "gqa_attn_decode_paged_multi": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                         _P, _P, _P, _P]),
    "gqa_attn_decode_fused_splits": (_I, [_I, _I, _I, _I]),
    "gqa_attn_decode_fused": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P]),
    "gqa_attn_prefill_causal": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P]),
    "gqa_attn_prefill_chunk": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P]),
    "gqa_attn_prefill_chunk_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "gqa_attn_prefill_chunk_default_parts": (_I, [_I, _I, _I, _I, _I]),
    "gqa_attn_prefill_chunk_split": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P,
                                          _P, _P, _P]),
    "gqa_last_device_error": (_I, [_P]),
    "gqa_trace_clear": (_I, []),
    "gqa_trace_read": (_I, [_P, _SZ]),
    "gqa_trace_mma_rate": (_I, [_I, _I, _P]),
    "gqa_trace_prefill_read": (_I, [_P, _SZ]),
    "gqa_set_wait_limit_ns": (_U64, [_U64]),
    "gqa_selftest_wait_timeout": (_I, [_U64, _P]),
}

_lock = threading.Lock()
_lib = None


class GQAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)}")


def load(path: str | None = None):
    """Load (building first if absent) and return the ctypes library handle."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                from . import build as _build  # compile in-tree; raises if nvcc fails
                _build.build()
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _device_index(x) -> int:
    """CUDA device ordinal of a tensor (-1, the current device, for anything else)."""
    dev = getattr(x, "device", None)
    return dev.index if getattr(dev, "type", None) == "cuda" and dev.index is not None else -1


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------- same-name entries --
def status_str(status: int) -> str:
    return load().gqa_status_str(int(status)).decode()


def gqa_attn_decode_split_chunk(S_max: int, n_split: int) -> int:
    return load().gqa_attn_decode_split_chunk(S_max, n_split)


def gqa_attn_decode_workspace_bytes(B: int, H_q: int, d: int, n_split: int) -> int:
    return load().gqa_attn_decode_workspace_bytes(B, H_q, d, n_split)


def gqa_attn_decode_default_splits(B: int, H_kv: int, S_max: int, device: int = -1) -> int:
    return load().gqa_attn_decode_default_splits(B, H_kv, S_max, device)


def gqa_attn_decode(q, k_cache, v_cache, seq_lens, B, S_max, H_q, H_kv, d, scale, n_split,
                    workspace, out, lse, stream=None) -> int:
    return load().gqa_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B, S_max,
                                  H_q, H_kv, d, scale, n_split, _ptr(workspace), _ptr(out),
                                  _ptr(lse), _stream(stream))


def gqa_attn_decode_combine(workspace, B, H_q, d, n_split, out, lse, stream=None) -> int:
    return load().gqa_attn_decode_combine(_ptr(workspace), B, H_q, d, n_split, _ptr(out),
                                          _ptr(lse), _stream(stream))


def gqa_attn_decode_counter_bytes(B: int, H_kv: int) -> int:
    return load().gqa_attn_decode_counter_bytes(B, H_kv)


def gqa_attn_decode_balanced(q, k_cache, v_cache, seq_lens, B, S_max, H_q, H_kv, d, scale,
                             n_split, workspace, counters, out, lse, stream=None) -> int:
    return load().gqa_attn_decode_balanced(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
                                           B, S_max, H_q, H_kv, d, scale, n_split,
                                           _ptr(workspace), _ptr(counters), _ptr(out), _ptr(lse),
                                           _stream(stream))


def gqa_attn_decode_multi(q, k_cache, v_cache, seq_lens, B, T_q, S_max, H_q, H_kv, d, scale,
                          n_split, workspace, out, lse, stream=None) -> int:
    return load().gqa_attn_decode_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B,
                                        T_q, S_max, H_q, H_kv, d, scale, n_split, _ptr(workspace),
                                        _ptr(out), _ptr(lse), _stream(stream))


def gqa_attn_decode_multi_default_splits(B, T_q, H_q, H_kv, S_max, d) -> int:
    return load().gqa_attn_decode_multi_default_splits(B, T_q, H_q, H_kv, S_max, d)


def gqa_attn_decode_paged_multi(q, k_pool, v_pool, block_table, seq_lens, B, T_q, num_pages,
                                page_size, max_blocks, H_q, H_kv, d, scale, n_split, workspace,
                                out, lse, stream=None) -> int:
    return load().gqa_attn_decode_paged_multi(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), _ptr(seq_lens), B, T_q, num_pages,
        page_size, max_blocks, H_q, H_kv, d, scale, n_split, _ptr(workspace), _ptr(out), _ptr(lse),
        _stream(stream))


def gqa_attn_decode_fused_splits(B, H_q, H_kv, d) -> int:
    return load().gqa_attn_decode_fused_splits(B, H_q, H_kv, d)


def gqa_attn_decode_fused(q, k_cache, v_cache, seq_lens, B, S_max, H_q, H_kv, d, scale, out, lse,
                          stream=None) -> int:
    return load().gqa_attn_decode_fused(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B,
                                        S_max, H_q, H_kv, d, scale, _ptr(out), _ptr(lse),
                                        _stream(stream))


def gqa_attn_decode_paged(q, k_pool, v_pool, block_table, seq_lens, B, num_pages, page_size,
                          max_blocks, H_q, H_kv, d, scale, n_split, workspace, out, lse,
                          stream=None) -> int:
    return load().gqa_attn_decode_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                        _ptr(seq_lens), B, num_pages, page_size, max_blocks, H_q,
                                        H_kv, d, scale, n_split, _ptr(workspace), _ptr(out),
                                        _ptr(lse), _stream(stream))


def gqa_attn_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, seq_lens, B, S_max, H_q, H_kv, d,
                        scale, n_split, workspace, out, lse, stream=None) -> int:
    return load().gqa_attn_decode_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                      _ptr(v_scale), _ptr(seq_lens), B, S_max, H_q, H_kv, d, scale,
                                      n_split, _ptr(workspace), _ptr(out), _ptr(lse),
                                      _stream(stream))


def gqa_attn_decode_paged_fp8(q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens, B,
                              num_pages, page_size, max_blocks, H_q, H_kv, d, scale, n_split,
                              workspace, out, lse, stream=None) -> int:
    return load().gqa_attn_decode_paged_fp8(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
                                            _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), B,
                                            num_pages, page_size, max_blocks, H_q, H_kv, d, scale,
                                            n_split, _ptr(workspace), _ptr(out), _ptr(lse),
                                            _stream(stream))


def gqa_attn_decode_noalloc(q, k_cache, v_cache, seq_lens, B, S_max, H_q, H_kv, d, scale, n_split,
                            out, lse, stream=None) -> int:
    return load().gqa_attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
                                          B, S_max, H_q, H_kv, d, scale, n_split, _ptr(out),
                                          _ptr(lse), _stream(stream))


def gqa_attn_prefill_causal(q, k, v, B, S, H_q, H_kv, d, scale, out, lse, stream=None) -> int:
    return load().gqa_attn_prefill_causal(_ptr(q), _ptr(k), _ptr(v), B, S, H_q, H_kv, d, scale,
                                          _ptr(out), _ptr(lse), _stream(stream))


def gqa_attn_prefill_chunk(q, k_cache, v_cache, seq_lens, B, T_q, S_max, H_q, H_kv, d, scale,
                           window, out, lse, stream=None) -> int:
    return load().gqa_attn_prefill_chunk(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B,
                                         T_q, S_max, H_q, H_kv, d, scale, int(window), _ptr(out),
                                         _ptr(lse), _stream(stream))


def gqa_attn_prefill_chunk_workspace_bytes(B, T_q, H_q, d, n_part) -> int:
    return load().gqa_attn_prefill_chunk_workspace_bytes(B, T_q, H_q, d, n_part)


def gqa_attn_prefill_chunk_default_parts(B, T_q, S_max, H_q, H_kv) -> int:
    return load().gqa_attn_prefill_chunk_default_parts(B, T_q, S_max, H_q, H_kv)


def gqa_attn_prefill_chunk_split(q, k_cache, v_cache, seq_lens, B, T_q, S_max, H_q, H_kv, d, scale,
                                 window, n_part, workspace, out, lse, stream=None) -> int:
    return load().gqa_attn_prefill_chunk_split(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B, T_q, S_max, H_q, H_kv, d, scale,
        int(window), int(n_part), _ptr(workspace), _ptr(out), _ptr(lse), _stream(stream))


def gqa_trace_clear() -> int:
    return load().gqa_trace_clear()


def gqa_trace_prefill_read(host, nbytes: int) -> int:
    """Copy the causal prefill's trace records into `host` (address or array)."""
    addr = host if isinstance(host, int) else (
        host.ctypes.data if hasattr(host, "ctypes") else host.data_ptr())
    return load().gqa_trace_prefill_read(addr, nbytes)


def gqa_trace_mma_rate(form: int, iters: int):
    """Return (status, SM cycles per tcgen05.mma of `form`) from the trace build."""
    out = ctypes.c_double(0.0)
    st = load().gqa_trace_mma_rate(int(form), int(iters), ctypes.addressof(out))
    return st, out.value


def gqa_trace_read(host, nbytes: int) -> int:
    """Copy trace records into `host` (an integer address, or a numpy/CPU array)."""
    addr = host if isinstance(host, int) else (
        host.ctypes.data if hasattr(host, "ctypes") else host.data_ptr())
    return load().gqa_trace_read(addr, nbytes)


def gqa_last_device_error(stream=None) -> int:
    return load().gqa_last_device_error(_stream(stream))


def gqa_set_wait_limit_ns(limit_ns: int) -> int:
    return load().gqa_set_wait_limit_ns(int(limit_ns))


def gqa_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    return load().gqa_selftest_wait_timeout(int(limit_ns), _stream(stream))


# ------------------------------------------------------------ torch helpers --
def _check(status: int, what: str):
    if status != GQA_OK:
        raise GQAError(status, what)


def decode_workspace(B, H_q, d, n_split, device="cuda"):
    """A workspace tensor for gqa_attn_decode (None when n_split == 1)."""
    import torch

    nbytes = gqa_attn_decode_workspace_bytes(B, H_q, d, n_split)
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def decode_counters(B, H_kv, device="cuda"):
    """Zeroed claim counters for gqa_attn_decode_balanced (int32 [B, H_kv, 2])."""
    import torch

    return torch.zeros((B, H_kv, 2), dtype=torch.int32, device=device)


def decode(q, k_cache, v_cache, seq_lens, scale=None, n_split=None, workspace=None, out=None,
           lse=None, stream=None, counters=None):
    """Split-KV decode + combine on CUDA tensors; returns (out bf16 [B,H_q,d], lse fp32 [B,H_q]).

    With ``counters`` (from decode_counters, reusable across calls) the splits
    are balanced (gqa_attn_decode_balanced)."""
    import torch

    B, H_q, d = q.shape
    _, S_max, H_kv, _ = k_cache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if n_split is None:
        n_split = gqa_attn_decode_default_splits(B, H_kv, S_max, _device_index(q))
    if out is None:
        out = torch.empty((B, H_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    if n_split > 1 and workspace is None:
        workspace = decode_workspace(B, H_q, d, n_split, q.device)
    if counters is None:
        _check(gqa_attn_decode(q, k_cache, v_cache, seq_lens, B, S_max, H_q, H_kv, d, scale,
                               n_split, workspace, out, lse, stream), "gqa_attn_decode")
    else:
        _check(gqa_attn_decode_balanced(q, k_cache, v_cache, seq_lens, B, S_max, H_q, H_kv, d,
                                        scale, n_split, workspace, counters, out, lse, stream),
               "gqa_attn_decode_balanced")
    if n_split > 1:
        _check(gqa_attn_decode_combine(workspace, B, H_q, d, n_split, out, lse, stream),
               "gqa_attn_decode_combine")
    return out, lse


def decode_multi(q, k_cache, v_cache, seq_lens, scale=None, n_split=None, workspace=None, out=None,
                 lse=None, stream=None):
    """Decode of the last T_q positions of each sequence (q [B, T_q, H_q, d]); returns
    (out bf16 [B, T_q, H_q, d], lse fp32 [B, T_q, H_q])."""
    import torch

    B, T_q, H_q, d = q.shape
    _, S_max, H_kv, _ = k_cache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if n_split is None:
        n_split = gqa_attn_decode_multi_default_splits(B, T_q, H_q, H_kv, S_max, d)
    if out is None:
        out = torch.empty((B, T_q, H_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, T_q, H_q), dtype=torch.float32, device=q.device)
    if n_split > 1 and workspace is None:
        workspace = decode_workspace(B * T_q, H_q, d, n_split, q.device)
    _check(gqa_attn_decode_multi(q, k_cache, v_cache, seq_lens, B, T_q, S_max, H_q, H_kv, d, scale,
                                 n_split, workspace, out, lse, stream), "gqa_attn_decode_multi")
    if n_split > 1:
        _check(gqa_attn_decode_combine(workspace, B * T_q, H_q, d, n_split, out, lse, stream),
               "gqa_attn_decode_combine")
    return out, lse


def decode_fused(q, k_cache, v_cache, seq_lens, scale=None, out=None, lse=None, stream=None):
    """Split-KV decode with the merge inside thread-block clusters (one launch, no workspace)."""
    import torch

    B, H_q, d = q.shape
    _, S_max, H_kv, _ = k_cache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    _check(gqa_attn_decode_fused(q, k_cache, v_cache, seq_lens, B, S_max, H_q, H_kv, d, scale, out,
                                 lse, stream), "gqa_attn_decode_fused")
    return out, lse


def paged_default_splits(B, H_kv, S_max, d, page_size):
    """Split count for the paged decode: the contiguous default, doubled for pages
    under 64 tokens (their smaller copies need two CTAs per SM in flight)."""
    n = gqa_attn_decode_default_splits(B, H_kv, S_max, -1)
    return 2 * n if page_size < 64 and n > 1 else n


def decode_paged(q, k_pool, v_pool, block_table, seq_lens, scale=None, n_split=None,
                 workspace=None, out=None, lse=None, stream=None):
    """Paged split-KV decode + combine on CUDA tensors; returns (out, lse).

    q [B, H_q, d] (out [B, H_q, d], lse [B, H_q]) or, for the last T_q positions of each
    sequence, q [B, T_q, H_q, d] (out [B, T_q, H_q, d], lse [B, T_q, H_q])."""
    import torch

    multi = q.dim() == 4
    if multi:
        B, T_q, H_q, d = q.shape
    else:
        (B, H_q, d), T_q = q.shape, 1
    P, B_p, H_kv, _ = k_pool.shape
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if n_split is None:
        n_split = paged_default_splits(B, H_kv, max_blocks * B_p, d, B_p)
    rows = (B, T_q, H_q) if multi else (B, H_q)
    if out is None:
        out = torch.empty(rows + (d,), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(rows, dtype=torch.float32, device=q.device)
    if n_split > 1 and workspace is None:
        workspace = decode_workspace(B * T_q, H_q, d, n_split, q.device)
    if multi:
        _check(gqa_attn_decode_paged_multi(q, k_pool, v_pool, block_table, seq_lens, B, T_q, P,
                                           B_p, max_blocks, H_q, H_kv, d, scale, n_split,
                                           workspace, out, lse, stream),
               "gqa_attn_decode_paged_multi")
    else:
        _check(gqa_attn_decode_paged(q, k_pool, v_pool, block_table, seq_lens, B, P, B_p,
                                     max_blocks, H_q, H_kv, d, scale, n_split, workspace, out, lse,
                                     stream), "gqa_attn_decode_paged")
    if n_split > 1:
        _check(gqa_attn_decode_combine(workspace, B * T_q, H_q, d, n_split, out, lse, stream),
               "gqa_attn_decode_combine")
    return out, lse


def decode_fp8(q, k8, v8, k_scale, v_scale, seq_lens, scale=None, n_split=None, workspace=None,
               out=None, lse=None, stream=None, block_table=None):
    """FP8-cache split-KV decode + combine (paged when block_table is given)."""
    import torch

    B, H_q, d = q.shape
    if block_table is None:
        _, S_max, H_kv, _ = k8.shape
    else:
        P, B_p, H_kv, _ = k8.shape
        S_max = block_table.shape[1] * B_p
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if n_split is None:  # the on-chip conversion wants three CTAs per SM
        n_split = 3 * gqa_attn_decode_default_splits(B, H_kv, S_max, _device_index(q))
    if out is None:
        out = torch.empty((B, H_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    if n_split > 1 and workspace is None:
        workspace = decode_workspace(B, H_q, d, n_split, q.device)
    if block_table is None:
        st = gqa_attn_decode_fp8(q, k8, v8, k_scale, v_scale, seq_lens, B, S_max, H_q, H_kv, d,
                                 scale, n_split, workspace, out, lse, stream)
    else:
        st = gqa_attn_decode_paged_fp8(q, k8, v8, k_scale, v_scale, block_table, seq_lens, B, P,
                                       B_p, block_table.shape[1], H_q, H_kv, d, scale, n_split,
                                       workspace, out, lse, stream)
    _check(st, "gqa_attn_decode_fp8")
    if n_split > 1:
        _check(gqa_attn_decode_combine(workspace, B, H_q, d, n_split, out, lse, stream),
               "gqa_attn_decode_combine")
    return out, lse


def prefill_causal(q, k, v, scale=None, out=None, lse=None, stream=None):
    """Causal prefill on CUDA tensors; returns (out bf16 [B,S,H_q,d], lse fp32 [B,H_q,S])."""
    import torch

    B, S, H_q, d = q.shape
    H_kv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, S, H_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H_q, S), dtype=torch.float32, device=q.device)
    _check(gqa_attn_prefill_causal(q, k, v, B, S, H_q, H_kv, d, scale, out, lse, stream),
           "gqa_attn_prefill_causal")
    return out, lse


def prefill_chunk(q, k_cache, v_cache, seq_lens=None, scale=None, window=-1, out=None, lse=None,
                  stream=None, n_part=None, workspace=None):
    """Chunk of T_q queries ending each sequence (optionally windowed); returns (out, lse).

    n_part None picks gqa_attn_prefill_chunk_default_parts; n_part > 1 splits each work
    item's key tiles into parts merged afterwards (workspace allocated when not given)."""
    import torch

    B, T_q, H_q, d = q.shape
    _, S_max, H_kv, _ = k_cache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, T_q, H_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H_q, T_q), dtype=torch.float32, device=q.device)
    if n_part is None:
        n_part = gqa_attn_prefill_chunk_default_parts(B, T_q, S_max, H_q, H_kv)
    if n_part == 1:
        _check(gqa_attn_prefill_chunk(q, k_cache, v_cache, seq_lens, B, T_q, S_max, H_q, H_kv, d,
                                      scale, window, out, lse, stream), "gqa_attn_prefill_chunk")
        return out, lse
    if workspace is None:
        nbytes = gqa_attn_prefill_chunk_workspace_bytes(B, T_q, H_q, d, n_part)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check(gqa_attn_prefill_chunk_split(q, k_cache, v_cache, seq_lens, B, T_q, S_max, H_q, H_kv, d,
                                        scale, window, n_part, workspace, out, lse, stream),
           "gqa_attn_prefill_chunk_split")
    return out, lse


def split_workspace(workspace, B, H_q, d, n_split):
    """Views (ml [B,H_q,n_split,2], O [B,H_q,n_split,d]) of a decode workspace tensor."""
    import torch

    ml_bytes = B * H_q * n_split * 8
    off = (ml_bytes + 255) // 256 * 256
    ml = workspace[:ml_bytes].view(torch.float32).view(B, H_q, n_split, 2)
    O = workspace[off: off + B * H_q * n_split * d * 4].view(torch.float32).view(B, H_q, n_split, d)
    return ml, O
