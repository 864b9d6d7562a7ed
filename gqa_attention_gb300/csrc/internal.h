// internal.h -- parameter blocks and launchers shared between the C-ABI shim
// (api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gqa {

// Bits of the per-device error word.  kErrBounds is set only by a build with
// GQA_DEBUG_BOUNDS=1: a computed global store index outside its buffer.
enum : unsigned { kErrTimeout = 1u, kErrBadSeqLen = 2u, kErrBadPage = 4u, kErrBounds = 8u };

constexpr int kDecodeTile = 64;  // tokens per decode pipeline stage; split chunks are multiples

struct DecodeParams {
  const __nv_bfloat16* q;  // [B, T_q, H_q, d]
  const int32_t* seq_lens; // [B]
  int B, S_max, H_q, H_kv, G, d;
  // Query rows per sequence: the last T_q positions L - T_q .. L - 1, query
  // t seeing keys 0 .. L - T_q + t (1 for plain decode).  Row (b, t, h) is
  // (b * T_q + t) * H_q + h of out [B, T_q, H_q, d], lse and the workspace.
  // The T_q * G rows of a KV head come in n_rg groups of 16 (one mma M tile),
  // each its own CTA: grid x = split * n_rg + group.
  int T_q, n_rg;
  int n_split, chunk;
  float scale_log2;        // tau * log2(e)
  float2* ws_ml;           // [B, H_q, n_split]  (m in natural-log units, l)
  float* ws_O;             // [B, H_q, n_split, d]
  __nv_bfloat16* out;      // [B, H_q, d]      (n_split == 1)
  float* lse;              // [B, H_q]         (n_split == 1)
  unsigned* err;           // device error word
  uint64_t wait_ns;        // time limit of every pipeline wait
  // paged cache only: token t of sequence b is row page*page_size + t % page_size
  // of the pools, page = block_table[b * max_blocks + t / page_size]
  const int32_t* block_table;
  int max_blocks, page_size, num_pages;
  // Balanced splits (contiguous cache only): two int32 words per (sequence,
  // KV head), zero before the launch and zero again after it; null otherwise.
  int* tile_ctr;
  // Set by the launcher: K/V tiles each split CTA prefetches into L2 before
  // its dependency wait (0 = none; used only when the whole grid is resident
  // at once, so that the prefetch overlaps the previous kernel).
  int prefetch_tiles;
};

constexpr int kMaxPagesPerCta = 512;  // page indices a paged decode CTA stages in shared memory

struct CombineParams {
  const float2* ws_ml;
  const float* ws_O;
  int B, H_q, d, n_split;
  __nv_bfloat16* out;
  float* lse;
  unsigned* err;  // device error word (bounds bit of a checking build)
};

struct PrefillParams {
  int B, S, H_q, H_kv, G, d;  // S: query rows per sequence (T_q of a chunk)
  int S_kv;                   // key/value rows per sequence in k, v (S_max of a cache)
  const int32_t* seq_lens;    // [B] sequence lengths (chunk ends), or null: every one is S_kv
  int window;                 // sliding window W (keys a-W..a), or -1 for none
  float scale_log2;
  __nv_bfloat16* out;  // [B, S, H_q, d]
  float* lse;          // [B, H_q, S]
  unsigned* err;
  uint64_t wait_ns;
  // Chunk mode only: each item's key tiles are split into n_part parts run as
  // separate work units; a part writes its unnormalised (m in base-2 units, l)
  // and O for rows (b, i, h) -> (b * S + i) * H_q + h into the workspace, and
  // launch_prefill_merge folds the parts.  n_part = 1: no split, no workspace.
  int n_part;
  float2* ws_ml;  // [rows][n_part]
  float* ws_O;    // [rows][n_part][d]
};

// Byte offset of the O partials in a chunk-split prefill workspace.
inline size_t prefill_ws_O_offset(size_t rows, int n_part) {
  return (rows * n_part * sizeof(float2) + 255) / 256 * 256;
}

// Kernel launchers; each returns the launch status (cudaGetLastError).
cudaError_t launch_decode_split(const DecodeParams& p, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, cudaStream_t stream);
cudaError_t launch_decode_combine(const CombineParams& p, cudaStream_t stream);
// Split decode whose n_split (<= 16) CTAs per (KV head, sequence) form a
// cluster and merge in-cluster; probe = true only checks that such clusters
// can be resident on the current device.
cudaError_t launch_decode_fused(const DecodeParams& p, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, bool probe, cudaStream_t stream);
// Multi-token decode with all T_q * G (<= 128) rows of a KV head in one
// tcgen05.mma tile: d = 128, 128-key tiles (p.chunk a multiple of 128), Q
// through `tm_q` (q viewed as [B * T_q][H_q][d], box {64, G, T_q}), K/V boxes
// of 128 rows.  Same partial layout as launch_decode_split.
cudaError_t launch_decode_tc(const DecodeParams& p, const CUtensorMap& tm_q,
                             const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             cudaStream_t stream);
cudaError_t launch_decode_paged(const DecodeParams& p, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, cudaStream_t stream);
// E4M3 cache with per-token scales; paged when p.block_table is set.
cudaError_t launch_decode_fp8(const DecodeParams& p, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, const CUtensorMap& tm_ks,
                              const CUtensorMap& tm_vs, cudaStream_t stream);
cudaError_t launch_prefill_causal(const PrefillParams& p, const CUtensorMap& tm_q,
                                  const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                  int num_sms, cudaStream_t stream);
cudaError_t launch_prefill_chunk(const PrefillParams& p, const CUtensorMap& tm_q,
                                 const CUtensorMap& tm_k, const CUtensorMap& tm_v, int num_sms,
                                 cudaStream_t stream);
cudaError_t launch_prefill_merge(const PrefillParams& p, cudaStream_t stream);
// Trace build: zero the causal prefill's stamp records (no-op otherwise).
cudaError_t prefill_trace_clear();
cudaError_t launch_wait_selftest(unsigned* err, uint64_t limit_ns, cudaStream_t stream);

// Layout of the decode workspace: byte offset of the O partials.
inline size_t decode_ws_O_offset(int B, int H_q, int n_split) {
  size_t ml = (size_t)B * H_q * n_split * sizeof(float2);
  return (ml + 255) / 256 * 256;
}

}  // namespace gqa
