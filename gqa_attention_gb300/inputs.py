"""Seeded synthetic inputs for the grouped-query attention workloads.

This module holds shapes and random draws only, none of the attention
arithmetic.  Tests, the smoke check and the benchmark draw their inputs here;
the oracle and the CUDA path each receive the same tensors.

Recipe (all draws on a CPU ``torch.Generator`` seeded with ``seed``):

* decode: ``seq_lens`` first (ragged workloads: ``torch.randint(lo, hi + 1, (B,))``;
  otherwise every sequence is ``S_max`` long), then Q ``[B, H_q, d]``, then K
  ``[L_b, H_kv, d]`` for b = 0..B-1, then V in the same order; every draw is
  ``torch.randn`` in fp32 scaled by ``value_scale`` and rounded to bfloat16
  (round to nearest even).  Cache rows at or past ``seq_lens[b]`` are padding and
  hold NaN, so that any kernel reading them unmasked shows it.
* prefill: Q ``[B, S, H_q, d]``, K ``[B, S, H_kv, d]``, V ``[B, S, H_kv, d]`` in that
  order, ``randn * value_scale`` rounded to bfloat16.
* sampled query rows for the long prefill check: ``torch.randperm(S)`` on a
  generator seeded with ``seed + 7919``, first ``n`` entries, rows 0 and S-1
  always included.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    H_q: int
    H_kv: int
    d: int
    S_max: int
    ragged: tuple | None = None  # (lo, hi) inclusive range of seq_lens, or None
    value_scale: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    S: int
    H_q: int
    H_kv: int
    d: int
    value_scale: float = 1.0
    oracle_rows: int | None = None  # sampled rows per head for the oracle check

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads, by what they are.
TINY_DECODE = DecodeConfig("decode_b1_hq8_hkv2_d32_ctx1024", 1, 8, 2, 32, 1024)
LLAMA70B_DECODE = DecodeConfig("decode_llama70b_b1_ctx32768", 1, 64, 8, 128, 32768)
LLAMA70B_DECODE_RAGGED = DecodeConfig(
    "decode_llama70b_b8_ragged_ctx1024-131072", 8, 64, 8, 128, 131072, ragged=(1024, 131072)
)
LLAMA70B_PREFILL_8K = PrefillConfig("prefill_causal_llama70b_s8192", 1, 8192, 64, 8, 128)
PREFILL_64K = PrefillConfig(
    "prefill_causal_llama70b_s65536", 1, 65536, 64, 8, 128, value_scale=0.5, oracle_rows=256
)
DECODE_CONFIGS = (TINY_DECODE, LLAMA70B_DECODE, LLAMA70B_DECODE_RAGGED)
PREFILL_CONFIGS = (LLAMA70B_PREFILL_8K, PREFILL_64K)


def _randn_bf16(shape, g, value_scale):
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if value_scale != 1.0:
        x.mul_(value_scale)
    return x.to(torch.bfloat16)


def decode_inputs(B, H_q, H_kv, d, S_max, seed=0, seq_lens=None, ragged=None, value_scale=1.0):
    """Return CPU tensors (q bf16 [B,H_q,d], k, v bf16 [B,S_max,H_kv,d], seq_lens int32 [B])."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    if ragged is not None:
        lo, hi = ragged
        lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    elif seq_lens is not None:
        lens = torch.as_tensor(seq_lens, dtype=torch.int64).reshape(B)
    else:
        lens = torch.full((B,), S_max, dtype=torch.int64)
    if int(lens.min()) < 1 or int(lens.max()) > S_max:
        raise ValueError("seq_lens must lie in [1, S_max]")
    q = _randn_bf16((B, H_q, d), g, value_scale)
    k = torch.full((B, S_max, H_kv, d), float("nan"), dtype=torch.bfloat16)
    v = torch.full((B, S_max, H_kv, d), float("nan"), dtype=torch.bfloat16)
    for b in range(B):
        k[b, : int(lens[b])] = _randn_bf16((int(lens[b]), H_kv, d), g, value_scale)
    for b in range(B):
        v[b, : int(lens[b])] = _randn_bf16((int(lens[b]), H_kv, d), g, value_scale)
    return q, k, v, lens.to(torch.int32)


def quantize_e4m3_per_token(x):
    """Cache quantisation used to build FP8 inputs: x [B, S, H, d] fp32 -> (codes uint8
    [B, S, H, d], scale fp32 [B, S]) with scale = max |x| over (H, d) / 448, codes from
    torch's float8_e4m3fn rounding (round to nearest even).  A token whose values
    are all zero gets scale 1."""
    amax = x.abs().amax(dim=(2, 3))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (x / scale[:, :, None, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8), scale.to(torch.float32)


def decode_inputs_fp8(B, H_q, H_kv, d, S_max, seed=0, seq_lens=None, ragged=None):
    """Decode inputs with an E4M3 cache: (q bf16, k8, v8 uint8 [B,S_max,H_kv,d],
    k_scale, v_scale fp32 [B,S_max], seq_lens int32).  The same draws as
    decode_inputs (fp32 randn), quantised per token; codes and scales past each
    sequence end are NaN bytes (0x7f) and NaN scales."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    if ragged is not None:
        lo, hi = ragged
        lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    elif seq_lens is not None:
        lens = torch.as_tensor(seq_lens, dtype=torch.int64).reshape(B)
    else:
        lens = torch.full((B,), S_max, dtype=torch.int64)
    q = _randn_bf16((B, H_q, d), g, 1.0)
    k = torch.randn((B, S_max, H_kv, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, S_max, H_kv, d), generator=g, dtype=torch.float32)
    k8, ks = quantize_e4m3_per_token(k)
    v8, vs = quantize_e4m3_per_token(v)
    for b in range(B):
        L = int(lens[b])
        k8[b, L:] = 0x7F
        v8[b, L:] = 0x7F
        ks[b, L:] = float("nan")
        vs[b, L:] = float("nan")
    return q, k8, v8, ks, vs, lens.to(torch.int32)


def decode_inputs_for(cfg: DecodeConfig, seed=0):
    return decode_inputs(cfg.B, cfg.H_q, cfg.H_kv, cfg.d, cfg.S_max, seed=seed,
                         ragged=cfg.ragged, value_scale=cfg.value_scale)


def prefill_inputs(B, S, H_q, H_kv, d, seed=0, value_scale=1.0):
    """Return CPU tensors q bf16 [B,S,H_q,d]; k, v bf16 [B,S,H_kv,d]."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = _randn_bf16((B, S, H_q, d), g, value_scale)
    k = _randn_bf16((B, S, H_kv, d), g, value_scale)
    v = _randn_bf16((B, S, H_kv, d), g, value_scale)
    return q, k, v


def prefill_inputs_for(cfg: PrefillConfig, seed=0):
    return prefill_inputs(cfg.B, cfg.S, cfg.H_q, cfg.H_kv, cfg.d, seed=seed,
                          value_scale=cfg.value_scale)


def sample_rows(S, n, seed=0):
    """Sorted int64 query positions: n seeded rows of [0, S), always with 0 and S-1."""
    if n >= S:
        return torch.arange(S, dtype=torch.int64)
    g = torch.Generator(device="cpu").manual_seed(seed + 7919)
    rows = torch.randperm(S, generator=g)[:n].tolist()
    rows = set(rows[: max(n - 2, 0)]) | {0, S - 1}
    return torch.tensor(sorted(rows), dtype=torch.int64)
