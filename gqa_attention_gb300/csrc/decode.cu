// decode.cu -- split-KV grouped-query decode (stage 1) and the log-sum-exp
// merge of the split partials (stage 2).
//
// Stage 1 follows the split-K decode of "Attention Kernel 계보" p.18 §4 with
// the GQA fold of p.15 §4/§7 and ADR-0060 §5.2: one CTA per (split, KV head,
// sequence) streams its split's K/V tiles once and serves all G query heads of
// the group, which sit in the M rows of the warp-level bf16 mma (G <= 16, rows
// past G are zero).  Softmax is the one-pass streaming (m, l, O) update of
// p.3 §5, in base-2 units with log2(e) folded into the scale (p.3 §8).  The four
// consumer warps take disjoint 16-token slices of every 64-token tile and are
// merged once at the end through shared memory (FA2 K-split, p.9 §5).  A fifth
// warp only issues TMA copies into a ring of NSTAGE shared-memory stages with
// full/empty mbarriers (p.10 §3); every wait has a time limit.
#include <type_traits>

#include "common.cuh"
#include "gqa_attn.h"
#include "internal.h"

// A build with GQA_TRACE=1 records where the split kernel's time goes: per CTA,
// globaltimer stamps (entry, release of the dependency wait, start and end of
// the tile loop, end of the epilogue) and the SM; per consumer warp, clock64
// cycles spent waiting for tiles, in Q K^T, in the softmax update, in P V and in
// the whole loop.  Phase boundaries wait for the phase's results (a register
// move of one of them), which perturbs the schedule a little; no arithmetic
// changes.  Other builds compile none of it.
#ifndef GQA_TRACE
#define GQA_TRACE 0
#endif

namespace gqa {
// One record of kTraceWords 64-bit words per CTA (linear block index), for the
// first kTraceCtas CTAs of the last launch: words 0-4 the stamps (ns), 5 the
// SM, 6 = split, 7 = tiles; from word 8, six words per consumer warp: wait,
// Q K^T, softmax, P V and loop cycles, and tiles the warp handled; words
// 56-58 the epilogue's phases and 59-61 the prologue's on thread 0 (cycles).
constexpr int kTraceCtas = 4096, kTraceWords = 64;
__device__ unsigned long long g_trace[GQA_TRACE ? kTraceCtas * kTraceWords : 1];

namespace {
constexpr bool kTrace = GQA_TRACE != 0;
__device__ __forceinline__ unsigned long long trace_clock() { return kTrace ? clock64() : 0ull; }
// Waits for `v` to be ready (a register move that reads it) in trace builds.
__device__ __forceinline__ void trace_ready(float& v) {
  if constexpr (kTrace) asm volatile("mov.b32 %0, %0;" : "+f"(v));
}

#ifndef GQA_SPLIT_PDL
#define GQA_SPLIT_PDL 1  // launch the split kernel as a programmatic dependent
#endif
#ifndef GQA_COMBINE_PDL
#define GQA_COMBINE_PDL 1  // launch the combine as a programmatic dependent of the split kernel
#endif

#ifndef GQA_DECODE_STAGES_FP8
#define GQA_DECODE_STAGES_FP8 4  // 16.5 KB each: three CTAs of four stages fit an SM
#endif
#ifndef GQA_DECODE_STAGES_FP8_ONE_WAVE
#define GQA_DECODE_STAGES_FP8_ONE_WAVE 8  // FP8, every CTA has an SM to itself
#endif
#ifndef GQA_FP8_ONE_WAVE_GROUPS
#define GQA_FP8_ONE_WAVE_GROUPS 2  // consumer groups of the one-wave FP8 CTAs
#endif

#ifndef GQA_DECODE_FUSED_STAGES_D128
#define GQA_DECODE_FUSED_STAGES_D128 3
#endif

#ifndef GQA_DECODE_STAGES_D128
#define GQA_DECODE_STAGES_D128 3  // 3 x 32 KB stages: two CTAs fit on one SM
#endif
#ifndef GQA_DECODE_STAGES_D128_ONE_WAVE
#define GQA_DECODE_STAGES_D128_ONE_WAVE 4  // when every CTA has an SM to itself
#endif

constexpr int kTile = kDecodeTile;  // tokens per stage
constexpr int kMaxClusterSplits = 16;
constexpr int kConsumerWarps = 4;   // 16 tokens each
// K/V bytes a split CTA may warm in L2 before its dependency wait, in whole
// tiles (at least one, at most kPrefetchMaxTiles).  Measured for the Llama3-70B
// decode at 32K (step = split + combine, median of three processes per depth):
// bf16 (32 KB tiles) 0/1/2/3/4/5/6/10/16 tiles 24.56/24.03/23.49/23.33/23.52/
// 23.64/23.77/24.10/24.51 us; E4M3 (17 KB tiles) best at 4-6 tiles
// (15.8-15.9 us), 17.9 us without.  A deeper prefetch fetches lines that this
// grid's own stream and the step's partials evict before use.
#ifndef GQA_PREFETCH_BYTES
#define GQA_PREFETCH_BYTES 98304
#endif
#ifndef GQA_PREFETCH_MAX_TILES
#define GQA_PREFETCH_MAX_TILES 6
#endif
constexpr int kPrefetchMaxTiles = GQA_PREFETCH_MAX_TILES;
static_assert(kPrefetchMaxTiles >= 0 && kPrefetchMaxTiles <= 32, "one tile per producer lane");
constexpr int prefetch_tiles(int stage_bytes) {
  return GQA_PREFETCH_BYTES / stage_bytes < 1 ? (kPrefetchMaxTiles > 0 ? 1 : 0)
         : GQA_PREFETCH_BYTES / stage_bytes > kPrefetchMaxTiles
             ? kPrefetchMaxTiles
             : GQA_PREFETCH_BYTES / stage_bytes;
}
constexpr int kThreads = (kConsumerWarps + 1) * 32;

// Balanced splits: each split CTA first streams a fixed share of about three
// quarters of its (sequence, KV head)'s tiles; the CTAs then claim the
// remaining tiles one at a time from a counter they share, so that a CTA that
// streams faster than its neighbours takes more of the tail.
constexpr int kStaticNum = 3, kStaticDen = 4;
// Tiles of a balanced split's own share for a sequence of L tokens.
__host__ __device__ __forceinline__ int balanced_static_tiles(int L, int n_split) {
  const long long n_t = (static_cast<long long>(L) + kTile - 1) / kTile;
  return static_cast<int>(n_t * kStaticNum / (static_cast<long long>(kStaticDen) * n_split));
}

template <int D>
struct DecodeLayout {
  static constexpr int kBox = D >= 64 ? 64 : D;            // elements per TMA box row
  static constexpr int kSpan = kBox * 2;                    // swizzle span (bytes)
  static constexpr int kChunksPerRow = kBox / 8;            // 16-byte chunks per box row
  static constexpr int kBlocks = D / kBox;                  // boxes per tile row
  static constexpr int kBlockBytes = kTile * kSpan;         // one box of a tile
  static constexpr int kTileBytes = kBlocks * kBlockBytes;  // K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;        // K + V
  // Shared-memory byte offset of (token row, 16-byte chunk along d) in a tile.
  __device__ static __forceinline__ uint32_t offset(int row, int chunk) {
    const int blk = chunk / kChunksPerRow;
    const int cc = chunk % kChunksPerRow;
    return blk * kBlockBytes + swizzle<kSpan>(row * kSpan + cc * 16);
  }
};

// FP8 cache stages: the E4M3 K and V tiles as TMA writes them (rows of D
// bytes, swizzled over min(D, 128) bytes) and the tile's per-token K and V
// scales.  Both are read straight into mma fragments and converted to f16 in
// registers (no f16 copy of the tile): a K fragment is 4 bytes of one key
// row; a V fragment is one byte of 4 key rows, gathered as 4-byte pieces of
// those rows and transposed with byte permutes.
// A tensor copy's shared-memory destination must be 128-byte aligned, so the
// scales of each h-row segment (h = page rows, at least 16) get their own
// 128-byte-aligned slot of round_up(4h, 128) bytes.
template <int D>
struct Fp8Layout {
  static constexpr int kTile8 = kTile * D;   // bytes of one E4M3 tile
  static constexpr int kScaleArea = 512;     // one tile's scales in up to 4 slots
  static constexpr int kOffV8 = kTile8;
  static constexpr int kOffKs = 2 * kTile8;
  static constexpr int kOffVs = 2 * kTile8 + kScaleArea;
  static constexpr int kTxBytes = 2 * kTile8 + 2 * kTile * 4;
  static constexpr int kStageBytes = (2 * kTile8 + 2 * kScaleArea + 1023) / 1024 * 1024;
  static constexpr int kSpan = D < 128 ? D : 128;  // swizzle span of an E4M3 row
  __host__ __device__ static constexpr int slot_bytes(int h) { return (h * 4 + 127) / 128 * 128; }
  // byte offset of token `col` (0..63) of a tile inside a scale area
  __device__ static __forceinline__ int scale_offset(int col, int h) {
    return (col / h) * slot_bytes(h) + (col % h) * 4;
  }
};

// FP8 key placement inside a warp's 16-key slice.  Logical key kappa (the
// order of the score and P fragments) sits in token row fp8_row(kappa) of the
// slice: the bit permutation (b3 b2 b1 b0) -> (b1 b3 b2 b0).  With 128-byte
// rows it puts the 8 rows of one K fragment load (kappa = 2g - (g & 1) + 2nt,
// g = 0..7) on 8 different swizzle phases, so those loads do not conflict in
// shared memory.  Any permutation is correct: scores, masks, scales and the
// V rows all go through the same map.
__device__ __forceinline__ int fp8_row(int kappa) {
  return ((kappa & 2) << 2) | ((kappa >> 2) << 1) | (kappa & 1);
}

// NW consecutive 32-bit words of row `row` of an E4M3 tile (rows of D bytes
// as TMA writes them, 16-byte chunks swizzled over min(D, 128) bytes) from
// byte b0 on; b0 is a multiple of 4 * min(NW, 4), so no load straddles a
// 16-byte chunk.
template <int D, int NW>
__device__ __forceinline__ void lds_fp8_words(const uint8_t* tile, int row, int b0,
                                              uint32_t (&w)[NW]) {
  constexpr int kSpan = Fp8Layout<D>::kSpan;
  if constexpr (NW >= 4) {
#pragma unroll
    for (int h = 0; h < NW / 4; ++h) {
      const uint4 v =
          *reinterpret_cast<const uint4*>(tile + swizzle<kSpan>(row * D + b0 + 16 * h));
      w[4 * h] = v.x;
      w[4 * h + 1] = v.y;
      w[4 * h + 2] = v.z;
      w[4 * h + 3] = v.w;
    }
  } else if constexpr (NW == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(tile + swizzle<kSpan>(row * D + b0));
    w[0] = v.x;
    w[1] = v.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(tile + swizzle<kSpan>(row * D + b0));
  }
}

// Shared-memory offset of a CTA's partial in the cluster merge: after the
// four warps' partials (mO, mML) of the final in-CTA merge.
template <int D>
constexpr int kClusterPartOff = (4 * 16 * D * 4 + 4 * 16 * 8 + 15) / 16 * 16;

template <int D, int NSTAGE, bool FP8>
constexpr int decode_smem_bytes() {
  return FP8 ? NSTAGE * Fp8Layout<D>::kStageBytes + 1024
             : NSTAGE * DecodeLayout<D>::kStageBytes + 1024;  // + alignment slack
}

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

// Online-softmax update of one query row held by a quad of lanes: x are this
// lane's 4 scores of the row in base-2 units (masked ones are -inf).  Returns
// the rescale factor for the row's O accumulators and writes exp2(x - m) to p.
__device__ __forceinline__ float online_update(float (&x)[4], float& m, float& l, float (&p)[4]) {
  const float mx = quad_max(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])));
  const float m_new = fmaxf(m, mx);
  const float ref = (m_new == -INFINITY) ? 0.f : m_new;  // no (-inf) - (-inf)
  const float alpha = ex2_approx(m - ref);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = ex2_approx(x[i] - ref);
  l = l * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
  m = m_new;
  return alpha;
}

// PAGED = true: the K/V cache is a pool of fixed-size pages reached through a
// block table ("Attention Kernel 계보" p.17 §2-§4, p.18 §5): the producer warp
// stages the CTA's page indices in shared memory once, then loads every page
// segment of a tile with its own TMA box.
// FP8 = true: the cache holds E4M3 codes with one fp32 scale per token
// ("Attention Kernel 계보" p.17 §7); the scales arrive with the tile and are
// applied in registers: score column j is multiplied by k_scale[j] and p_j by
// v_scale[j], so the mma sees the exact E4M3 values (converted to f16, with Q
// converted to f16 as well).
// CLUSTER = true: the n_split CTAs of one (KV head, sequence) form a thread-
// block cluster and merge their partials themselves: each CTA leaves its
// (m, l, O) in its own shared memory, and after a cluster barrier CTA `rank`
// folds slice `rank` of the G x D outputs over all n_split partials, read
// through distributed shared memory (the same associative merge as the
// combine kernel, p.4 of "Attention Kernel 계보").  No workspace, no second
// launch.
// Two CTAs per SM; three for the FP8 cache with G <= 8, whose sweep is bound
// by its per-tile integer work (E4M3 conversion, byte transposes) rather than
// by HBM, so it gains from more warps at 128 registers.
// NGRP = 2 (FP8 with one CTA per SM): two groups of four consumer warps take
// alternate tiles, so that each SM has two warps per scheduler to hide the
// latency of the per-tile E4M3 work; the eight warp partials are merged at
// the end as the four are otherwise.
// DYN = true (balanced splits, contiguous bf16 cache): split s first streams tiles
// s*n_s .. s*n_s + n_s - 1 of its (sequence, KV head), n_s =
// balanced_static_tiles(L, n_split); the tiles from n_split * n_s on form a
// pool that the producer warps of all n_split CTAs claim one tile at a time
// through p.tile_ctr[2 (b H_kv + kv)].  A split's partial then covers its
// share plus the tiles it claimed: the keys of a partial need not be
// contiguous, since the merge of "Attention Kernel 계보" p.4 is order-free.
// The producer writes each stage's first token next to the stage and ends
// the ring with a stage whose token is -1.  Every CTA that reaches the claims
// then counts itself out on p.tile_ctr[... + 1]; the last one returns both
// words to zero for the next call.
template <int D, bool ROWS16, int NSTAGE, bool PAGED, bool FP8, bool CLUSTER, int NGRP = 1,
          bool DYN = false>
__global__ void __launch_bounds__((kConsumerWarps * NGRP + 1) * 32,
                                  NGRP > 1 ? 1 : ((FP8 && !ROWS16) ? 3 : 2))
    gqa_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_ks,
                            const __grid_constant__ CUtensorMap tm_vs, const DecodeParams p) {
  static_assert(!(CLUSTER && (PAGED || FP8)), "the cluster merge serves the contiguous bf16 cache");
  static_assert(NGRP == 1 || (NGRP <= 3 && !CLUSTER), "several consumer groups: split CTAs only");
  static_assert(!DYN || (!PAGED && !FP8 && !CLUSTER && NGRP == 1),
                "balanced splits: a contiguous bf16 cache, one consumer group");
  constexpr int kCW = kConsumerWarps * NGRP;  // consumer warps
  constexpr int kThr = (kCW + 1) * 32;
  using Lay = DecodeLayout<D>;
  using F8 = Fp8Layout<D>;
  constexpr int kStageBytes = FP8 ? F8::kStageBytes : Lay::kStageBytes;
  constexpr int kTxBytes = FP8 ? F8::kTxBytes : Lay::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[NSTAGE];
  __shared__ __align__(8) uint64_t empty_bar[NSTAGE];
  __shared__ int abort_flag;
  __shared__ int bad_page;
  __shared__ int pages_sm[PAGED ? kMaxPagesPerCta : 1];
  __shared__ int stage_tok[DYN ? NSTAGE : 1];  // balanced splits: first token of each stage


  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);

  // (row groups of one split are neighbours in launch order, so their reads
  // of the same K/V tiles meet in L2)
  const int split = CLUSTER ? blockIdx.x : blockIdx.x / p.n_rg;
  const int rg = CLUSTER ? 0 : blockIdx.x % p.n_rg;
  const int kv = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long tr_entry = kTrace ? globaltimer_ns() : 0ull;
  const size_t tr_cta = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  unsigned long long* const tr_rec =
      (kTrace && tr_cta < (size_t)kTraceCtas) ? g_trace + tr_cta * kTraceWords : nullptr;
  const int G = p.G;
  const int h0 = kv * G;
  // mma row r (0..15) of row group rg is row x = 16 rg + r of the KV head:
  // query t = x / G of head h0 + x % G; rows past T_q * G are padding.
  const int R = min(16, p.T_q * G - 16 * rg);
  // x / G without an integer division: (x + 1/2) / G lies at least 1/32 from
  // the nearest integer (G <= 16), far more than the float error for x < 2^20.
  const float inv_g = 1.f / static_cast<float>(G);
  auto out_row = [&](int r) -> size_t {
    const int x = 16 * rg + r;
    const int tq = static_cast<int>((static_cast<float>(x) + 0.5f) * inv_g);
    return ((size_t)b * p.T_q + tq) * p.H_q + h0 + (x - tq * G);
  };
  const size_t n_rows = (size_t)p.B * p.T_q * p.H_q;  // rows of out, lse and the workspace
  // The ring's barriers touch shared memory only: they are set up while the
  // previous kernel finishes (the CTA barrier that publishes them comes
  // before the dependency wait as well).
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kConsumerWarps);
    }
    abort_flag = 0;
    bad_page = 0;
    fence_barrier_init();
  }
  // Launched as a programmatic dependent of the previous kernel in the stream:
  // no global memory is read or written before that kernel has completed.  While it
  // finishes, the producer warp of each split's first row group prefetches the
  // split's first K/V tiles into L2, one (tile, page segment) per lane.  The
  // extent comes from relaxed loads of seq_lens[b] and, for a paged cache, of
  // the page indices; they may see values from before the previous kernel's
  // writes and only aim the prefetch (an index outside the pool is skipped).
  // A prefetch hands no data to the kernel and L2 is where writes become
  // coherent, so it cannot expose stale values; at worst it fetches rows the
  // split will not use.
  if (p.prefetch_tiles > 0 && warp == kCW && rg == 0) {
    int L_hint;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(L_hint) : "l"(p.seq_lens + b));
    if (lane == 0) {
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
    }
    const int h = PAGED ? min(p.page_size, kTile) : kTile;  // rows per box
    const int subs = kTile / h;
    const int i = lane / subs, sub = lane % subs;
    // (a balanced split prefetches from its own share of the tiles)
    const int pchunk =
        DYN ? balanced_static_tiles(max(0, min(p.S_max, L_hint)), p.n_split) * kTile : p.chunk;
    const int tk = split * pchunk + i * kTile + sub * h;
    const int tp_end = min(min(p.S_max, L_hint), split * pchunk + pchunk);
    if (i < p.prefetch_tiles && tk < tp_end) {
      int row = b * p.S_max + tk, sc_x = tk, sc_y = b;
      bool ok = true;
      if constexpr (PAGED) {
        int pg;
        asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];"
                     : "=r"(pg)
                     : "l"(p.block_table + (size_t)b * p.max_blocks + tk / p.page_size));
        ok = pg >= 0 && pg < p.num_pages;
        row = pg * p.page_size + tk % p.page_size;
        sc_x = tk % p.page_size;
        sc_y = pg;
      }
      if (ok) {
        if constexpr (FP8) {
          tma_prefetch_l2_3d(&tm_k, 0, kv, row);
          tma_prefetch_l2_3d(&tm_v, 0, kv, row);
          tma_prefetch_l2_2d(&tm_ks, sc_x, sc_y);
          tma_prefetch_l2_2d(&tm_vs, sc_x, sc_y);
        } else {
#pragma unroll
          for (int blk = 0; blk < Lay::kBlocks; ++blk) {
            tma_prefetch_l2_3d(&tm_k, blk * Lay::kBox, kv, row);
            tma_prefetch_l2_3d(&tm_v, blk * Lay::kBox, kv, row);
          }
        }
      }
    }
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const unsigned long long tr_release = kTrace ? globaltimer_ns() : 0ull;
  const unsigned long long tp0 = trace_clock();
  int L = p.seq_lens[b];
  if constexpr (kTrace) asm volatile("mov.b32 %0, %0;" : "+r"(L));
  const unsigned long long tp1 = trace_clock();

  // ---- device-side argument check and empty splits (no pipeline needed) ----
  if (L < p.T_q || L > p.S_max || L < 1) {
    if (threadIdx.x == 0 && split == 0 && kv == 0 && rg == 0) atomicOr(p.err, kErrBadSeqLen);
    for (int e = threadIdx.x; e < R * D; e += kThr) {
      const int r = e / D, c = e % D;
      const size_t row = out_row(r);
      if (p.n_split == 1 || CLUSTER) {
        // (a cluster's CTAs all see the same length and all return here)
        if (CLUSTER && split != 0) continue;
        if (in_bounds(row * D + c, 1, n_rows * D, p.err)) p.out[row * D + c] = __float2bfloat16(NAN);
        if (c == 0 && in_bounds(row, 1, n_rows, p.err)) p.lse[row] = NAN;
      } else if (c == 0 && in_bounds(row * p.n_split + split, 1, n_rows * p.n_split, p.err)) {
        p.ws_ml[row * p.n_split + split] = make_float2(NAN, NAN);
      }
    }
    return;
  }
  // Balanced splits: the CTA's own share; the claimed tiles may lie anywhere
  // in [0, L), so the masks use the sequence end.
  const int n_static = DYN ? balanced_static_tiles(L, p.n_split) : 0;
  const int t0 = DYN ? split * n_static * kTile : split * p.chunk;
  if (!CLUSTER && !DYN && t0 >= L) {  // empty split: the merge identity (-inf, 0); O is not written
    for (int r = threadIdx.x; r < R; r += kThr)
      if (in_bounds(out_row(r) * p.n_split + split, 1, n_rows * p.n_split, p.err))
        p.ws_ml[out_row(r) * p.n_split + split] = make_float2(-INFINITY, 0.f);
    return;
  }
  // (in a cluster an empty split still takes part: no tiles, partial (-inf, 0, 0))
  const int t_end = DYN ? L : min(t0 + p.chunk, L);
  const int n_tiles = DYN ? n_static : (t_end > t0 ? (t_end - t0 + kTile - 1) / kTile : 0);

  const unsigned long long tp2 = trace_clock();

  // ------------------------------------------------------------ producer ----
  if (DYN && warp == kCW) {
    // Lane 0 runs the balanced producer: the CTA's own share, then claimed
    // tiles until the pool is empty, then the closing stage.
    if (lane == 0) {
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      // one row group per split: every K/V byte is read once
      const uint64_t kv_pol = l2_policy_evict_first();
      int* const ctr = p.tile_ctr + 2 * ((size_t)b * p.H_kv + kv);
      const int pool0 = p.n_split * n_static;
      const int n_pool = (L + kTile - 1) / kTile - pool0;  // >= 1: the share is below 3/4
      // Ring position i may be filled once the consumers have released
      // position i - NSTAGE (the abort flag is read only on the slow path).
      auto slot_free = [&](int i) -> bool {
        if (i < NSTAGE) return true;
        const uint32_t eb = smem_u32(&empty_bar[i % NSTAGE]), par = ((i / NSTAGE) - 1) & 1;
        if (mbar_try_wait(eb, par)) return true;
        if (*reinterpret_cast<volatile int*>(&abort_flag) || !mbar_wait(eb, par, p.wait_ns, p.err)) {
          *reinterpret_cast<volatile int*>(&abort_flag) = 1;
          return false;
        }
        return true;
      };
      // Ring position i takes the tile that starts at token tok.  The stage's
      // token is written before the barrier is armed (the arrive releases it
      // to the consumers' wait).
      auto load = [&](int i, int tok) {
        const int st = i % NSTAGE;
        stage_tok[st] = tok;
        const uint32_t fb = smem_u32(&full_bar[st]);
        mbar_arrive_expect_tx(fb, kTxBytes);
        const uint32_t dst_k = smem_base + st * kStageBytes;
        // (rows past the sequence end are masked by the consumers; past the
        // last sequence the copy fills zeros)
        const int row = b * p.S_max + tok;
#pragma unroll
        for (int blk = 0; blk < Lay::kBlocks; ++blk) {
          tma_load_3d(dst_k + blk * Lay::kBlockBytes, &tm_k, fb, blk * Lay::kBox, kv, row, kv_pol);
          tma_load_3d(dst_k + Lay::kTileBytes + blk * Lay::kBlockBytes, &tm_v, fb, blk * Lay::kBox,
                      kv, row, kv_pol);
        }
      };
      int issued = 0;
      bool live = true;
      for (; issued < n_static; ++issued) {
        if (!slot_free(issued)) {
          live = false;
          break;
        }
        load(issued, t0 + issued * kTile);
      }
      if (live) {
        int c = atomicAdd(ctr, 1);
        while (c < n_pool) {
          // the next claim travels while this tile waits for its slot
          const int c_next = atomicAdd(ctr, 1);
          if (!slot_free(issued)) {
            live = false;
            break;
          }
          load(issued, (pool0 + c) * kTile);
          ++issued;
          c = c_next;
        }
      }
      // (see the contiguous producer below on the trigger's placement)
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      // No copy may still target this CTA's shared memory when it exits.
      for (int i = max(0, issued - NSTAGE); i < issued; ++i)
        mbar_wait(smem_u32(&full_bar[i % NSTAGE]), (i / NSTAGE) & 1, p.wait_ns, p.err);
      // The closing stage: no copy, token -1.
      if (live && slot_free(issued)) {
        stage_tok[issued % NSTAGE] = -1;
        mbar_arrive(smem_u32(&full_bar[issued % NSTAGE]));
      }
      // Count this CTA out.  Each CTA's claims are performed before its count
      // (the fence orders them also when a claim's result went unused after
      // an abort), so the last count ends every claim of this launch and the
      // words can return to zero.
      __threadfence();
      if (atomicAdd(ctr + 1, 1) == p.n_split - 1) {
        atomicExch(ctr, 0);
        atomicExch(ctr + 1, 0);
      }
    }
    __syncwarp();
    return;
  }
  if (warp == kCW) {
    const int page0 = PAGED ? t0 / p.page_size : 0;
    if (PAGED) {
      // Stage the page indices of tokens [t0, t_end); an index outside the
      // pool is reported and replaced by 0 (the CTA's outputs become NaN).
      const int n_pages = (t_end - 1) / p.page_size - page0 + 1;
      const int32_t* row_table = p.block_table + (size_t)b * p.max_blocks;
      int bad = 0;
      for (int j = lane; j < n_pages; j += 32) {
        int pg = row_table[page0 + j];
        if (pg < 0 || pg >= p.num_pages) {
          bad = 1;
          pg = 0;
        }
        pages_sm[j] = pg;
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) {
        bad_page = 1;
        atomicOr(p.err, kErrBadPage);
      }
      __syncwarp();
    }
    if (lane == 0) {
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      if (FP8) {
        tma_prefetch_map(&tm_ks);
        tma_prefetch_map(&tm_vs);
      }
    }
    // The whole warp runs the tile loop: lane 0 takes the slot and arms its
    // barrier, then the copies are issued, by lane 0 for a contiguous cache
    // and by lane `sub` for page segment `sub` of a paged one (so that the
    // boxes of small pages are issued in parallel).  With one row group per
    // split each K/V byte is read once, so the copies are evict-first in L2;
    // several row groups read each tile through L2 and keep the default.
    const uint64_t kv_pol = p.n_rg == 1 ? l2_policy_evict_first() : l2_policy_evict_normal();
    int issued = 0;
    for (int i = 0; i < n_tiles; ++i) {
      const int st = i % NSTAGE;
      bool go = true;
      if (lane == 0 && i >= NSTAGE) {
        // A slot the consumers have released passes at once; the abort flag
        // (a consumer that gave up stops arriving) is read only on the slow path.
        const uint32_t eb = smem_u32(&empty_bar[st]), par = ((i / NSTAGE) - 1) & 1;
        if (!mbar_try_wait(eb, par) && (*reinterpret_cast<volatile int*>(&abort_flag) ||
                                        !mbar_wait(eb, par, p.wait_ns, p.err))) {
          *reinterpret_cast<volatile int*>(&abort_flag) = 1;
          go = false;
        }
      }
      if (lane == 0 && go) mbar_arrive_expect_tx(smem_u32(&full_bar[st]), kTxBytes);
      if (!__shfl_sync(0xffffffffu, go, 0)) break;  // (the barrier is armed before any copy)
      const uint32_t fb = smem_u32(&full_bar[st]);
      const uint32_t dst_k = smem_base + st * kStageBytes;
      const uint32_t dst_v = dst_k + Lay::kTileBytes;
      if constexpr (FP8) {
        // E4M3 rows (D bytes) and the per-token scales; page segments of
        // h rows when paged.  Rows past the end read as zeros (TMA fill).
        const int h = PAGED ? min(p.page_size, kTile) : kTile;
        const int sub = lane;
        if (sub < kTile / h) {
          const int tok = t0 + i * kTile + sub * h;
          int row, sc_x, sc_y;
          if (!PAGED) {
            row = b * p.S_max + tok;
            sc_x = tok;
            sc_y = b;
          } else if (tok < t_end) {
            const int pg = pages_sm[tok / p.page_size - page0];
            row = pg * p.page_size + tok % p.page_size;
            sc_x = tok % p.page_size;
            sc_y = pg;
          } else {
            row = p.num_pages * p.page_size;
            sc_x = 0;
            sc_y = p.num_pages;
          }
          tma_load_3d(dst_k + sub * h * D, &tm_k, fb, 0, kv, row, kv_pol);
          tma_load_3d(dst_k + F8::kOffV8 + sub * h * D, &tm_v, fb, 0, kv, row, kv_pol);
          tma_load_2d(dst_k + F8::kOffKs + sub * F8::slot_bytes(h), &tm_ks, fb, sc_x, sc_y,
                      kv_pol);
          tma_load_2d(dst_k + F8::kOffVs + sub * F8::slot_bytes(h), &tm_vs, fb, sc_x, sc_y,
                      kv_pol);
        }
      } else if (!PAGED) {
        if (lane == 0) {
          const int row = b * p.S_max + t0 + i * kTile;
#pragma unroll
          for (int blk = 0; blk < Lay::kBlocks; ++blk) {
            tma_load_3d(dst_k + blk * Lay::kBlockBytes, &tm_k, fb, blk * Lay::kBox, kv, row,
                        kv_pol);
            tma_load_3d(dst_v + blk * Lay::kBlockBytes, &tm_v, fb, blk * Lay::kBox, kv, row,
                        kv_pol);
          }
        }
      } else {
        // Boxes of h = min(page_size, 64) rows; a box wholly past the split
        // end reads rows past the pool (TMA fills them with zeros) so that
        // every stage still receives its full byte count.
        const int h = min(p.page_size, kTile);
        const int sub = lane;
        if (sub < kTile / h) {
          const int tok = t0 + i * kTile + sub * h;
          const int row = tok < t_end ? pages_sm[tok / p.page_size - page0] * p.page_size +
                                            tok % p.page_size
                                      : p.num_pages * p.page_size;
          const uint32_t off = sub * h * Lay::kSpan;
#pragma unroll
          for (int blk = 0; blk < Lay::kBlocks; ++blk) {
            tma_load_3d(dst_k + blk * Lay::kBlockBytes + off, &tm_k, fb, blk * Lay::kBox, kv, row,
                        kv_pol);
            tma_load_3d(dst_v + blk * Lay::kBlockBytes + off, &tm_v, fb, blk * Lay::kBox, kv, row,
                        kv_pol);
          }
        }
      }
      issued = i + 1;
    }
    if (lane == 0) {
      // Let the next kernel in the stream be scheduled once this CTA has
      // issued its last copy.  A following combine waits for this grid anyway;
      // a following split prefetches its first tiles into L2, which pays only
      // this late (earlier, this grid's own stream evicts them before use).
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      // No copy may still target this CTA's shared memory when it exits.
      for (int i = max(0, issued - NSTAGE); i < issued; ++i)
        mbar_wait(smem_u32(&full_bar[i % NSTAGE]), (i / NSTAGE) & 1, p.wait_ns, p.err);
    }
    __syncwarp();
    if constexpr (CLUSTER) {  // the consumers' two cluster barriers
      __syncwarp();
      cluster_sync();
      cluster_sync();
    }
    return;
  }

  // ------------------------------------------------------------ consumers ---
  const int g = lane >> 2, t = lane & 3;
  // 16-token slice of each tile this warp takes, and its group's tile parity
  const int ws = warp % kConsumerWarps, grp = warp / kConsumerWarps;
  // Q group as the A operand: rows = query heads h0..h0+G-1 (zero past G).
  uint32_t qa[D / 16][4];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
    const bool v0 = g < R, v1 = g + 8 < R;
    const size_t rb0 = v0 ? out_row(g) * (D / 2) : 0;
    const size_t rb1 = v1 ? out_row(g + 8) * (D / 2) : 0;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      // bf16: 32-bit word c holds columns (kk*16 + 2t, +1), word c + 4 holds
      // (kk*16 + 2t + 8, +1).  FP8: the k index of the fragment runs over d in
      // the order its K fragment is loaded: lane t holds bytes (D/4) t ..
      // (D/4) t + D/4 - 1 of a key row, 4 per k-step, so step kk takes words
      // (D/8) t + 2 kk and + 1 (columns (D/4) t + 4 kk .. + 3).
      const int c = FP8 ? (D / 8) * t + 2 * kk : kk * 8 + t;
      const int c2 = FP8 ? c + 1 : c + 4;
      qa[kk][0] = v0 ? q32[rb0 + c] : 0u;
      qa[kk][1] = v1 ? q32[rb1 + c] : 0u;
      qa[kk][2] = v0 ? q32[rb0 + c2] : 0u;
      qa[kk][3] = v1 ? q32[rb1 + c2] : 0u;
      if constexpr (FP8) {  // bf16 -> f16 (exact inside the f16 range)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 bv = *reinterpret_cast<const __nv_bfloat162*>(&qa[kk][e]);
          const float2 f = __bfloat1622float2(bv);
          qa[kk][e] = pack_f16x2(f.x, f.y);
        }
      }
    }
  }

  // FP8 with G <= 8 computes P V transposed, O^T = V^T P^T (M = d, N = the
  // 8 query rows, no padded rows): o[mt] is d-tile mt, only D/16 of them.
  // Otherwise o[n] is n-tile n of O (M = query rows, N = d).
  constexpr bool TPV = FP8 && !ROWS16;
  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;

  // ldmatrix lane roles.  K (non-transposed): matrix mi = lane/8 covers tokens
  // (mi/2)*8.. and d-chunk (mi%2); V (transposed): tokens (mi%2)*8.., chunk mi/2.
  const int k_row = ws * 16 + ((lane >> 4) << 3) + (lane & 7);
  const int k_chk = (lane >> 3) & 1;
  const int v_row = ws * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
  const int v_chk = lane >> 4;
  // FP8 (see fp8_row): tile rows of this lane's K fragments (n-tiles 0, 1)
  // and of its V gathers (logical keys 4t .. 4t + 3).
  const int k8_row0 = ws * 16 + fp8_row(2 * g - (g & 1));
  const int k8_row1 = ws * 16 + fp8_row(2 * g - (g & 1) + 2);
  int v8_row[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) v8_row[e] = ws * 16 + fp8_row(4 * t + e);

  // Key limits of rows g and g + 8 in this split: query t sees keys below
  // L - T_q + 1 + t (the split end t_end for plain decode).
  const int lim0 = min(t_end, L - p.T_q + 1 + (16 * rg + g) / G);
  const int lim1 = min(t_end, L - p.T_q + 1 + (16 * rg + g + 8) / G);
  const int lim_lo = min(lim0, lim1);

  bool aborted = false;
  if constexpr (kTrace) {
    float q_any = __uint_as_float(qa[0][0]);
    trace_ready(q_any);
    qa[0][0] = __float_as_uint(q_any);
  }
  const unsigned long long tp3 = trace_clock();
  const unsigned long long tr_loop0 = kTrace ? globaltimer_ns() : 0ull;
  unsigned long long tr_c[6] = {0, 0, 0, 0, trace_clock(), 0};  // wait, qk, softmax, pv, loop, tiles
  for (int i = grp; DYN || i < n_tiles; i += NGRP) {
    const int st = i % NSTAGE;
    const unsigned long long tc0 = trace_clock();
    // A stage that has landed passes at once; the abort flag is read only on
    // the slow path.
    const uint32_t fb = smem_u32(&full_bar[st]), par = (i / NSTAGE) & 1;
    bool ok = mbar_try_wait(fb, par);
    if (!ok) ok = *reinterpret_cast<volatile int*>(&abort_flag) == 0 && mbar_wait(fb, par, p.wait_ns, p.err);
    const unsigned long long tc1 = trace_clock();
    tr_c[0] += tc1 - tc0;
    tr_c[5] += 1;
    // Keep the warp converged for the warp-collective ldmatrix/mma below.
    if (!__all_sync(0xffffffffu, ok)) {
      *reinterpret_cast<volatile int*>(&abort_flag) = 1;
      aborted = true;
      break;
    }
    int tile_tok = t0 + i * kTile;
    if constexpr (DYN) {
      tile_tok = stage_tok[st];
      if (tile_tok < 0) break;  // the closing stage (the same value in every lane)
    }
    uint32_t kbase = smem_base + st * kStageBytes;
    uint32_t vbase = kbase + Lay::kTileBytes;
    const int tok0 = tile_tok + ws * 16;  // first token of this warp's slice
    float ksv[4], vsv[4];  // FP8: scales of this thread's 4 score columns
    if constexpr (FP8) {
      // Key order inside a warp's 16-key slice (FP8 only): the lane with
      // fragment column g of score tile nt holds logical key 2g - (g & 1) + 2 nt,
      // so lane (g, t) ends up with the scores of logical keys 4t .. 4t + 3,
      // which are the A-fragment k indices 2t, 2t + 1, 2t + 8, 2t + 9 of P V.
      // Logical key kappa is token row fp8_row(kappa) of the slice.
      const uint8_t* sc_sm = smem + st * kStageBytes;
      const int h = PAGED ? min(p.page_size, kTile) : kTile;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = v8_row[e];  // token of score column e of this lane
        const int off = F8::scale_offset(col, h);
        ksv[e] = *reinterpret_cast<const float*>(sc_sm + F8::kOffKs + off);
        vsv[e] = *reinterpret_cast<const float*>(sc_sm + F8::kOffVs + off);
      }
    }

    // S = Q K^T over this warp's 16 tokens (two n8 tiles).
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if constexpr (FP8) {
      // K fragments straight from the E4M3 rows: lane (g, t) loads bytes
      // (D/4) t .. + D/4 - 1 of its two key rows; word kk of a row becomes the
      // two f16 pairs of that row's k-step kk fragment.
      uint32_t kw[2][D / 16];
      lds_fp8_words<D, D / 16>(smem + st * kStageBytes, k8_row0, (D / 4) * t, kw[0]);
      lds_fp8_words<D, D / 16>(smem + st * kStageBytes, k8_row1, (D / 4) * t, kw[1]);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          mma_f16_16816(sacc[nt], qa[kk], e4m3x2_to_f16x2(kw[nt][kk]),
                        e4m3x2_to_f16x2(kw[nt][kk] >> 16));
    } else {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t b00, b01, b10, b11;
        ldsm_x4(kbase + Lay::offset(k_row, kk * 2 + k_chk), b00, b01, b10, b11);
        mma_bf16_16816(sacc[0], qa[kk], b00, b01);
        mma_bf16_16816(sacc[1], qa[kk], b10, b11);
      }
    }

    // Scores in base-2 units; tokens past the split end are masked by select.
    const bool partial = tok0 + 16 > lim_lo;
    trace_ready(sacc[0][0]);
    trace_ready(sacc[1][0]);
    const unsigned long long tc2 = trace_clock();
    tr_c[1] += tc2 - tc1;
    float x0[4], x1[4];  // row g (x0) and row g+8 (x1)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int tk = FP8 ? tok0 - ws * 16 + v8_row[2 * nt + c] : tok0 + nt * 8 + 2 * t + c;
        const bool ok0 = !partial || tk < lim0, ok1 = !partial || tk < lim1;
        const float sc = FP8 ? ksv[nt * 2 + c] * p.scale_log2 : p.scale_log2;
        x0[nt * 2 + c] = ok0 ? sacc[nt][c] * sc : -INFINITY;
        x1[nt * 2 + c] = ok1 ? sacc[nt][2 + c] * sc : -INFINITY;
        // p * v_scale = 0 past the split end (the scale there may be anything)
        if (FP8) vsv[nt * 2 + c] = (!partial || tk < t_end) ? vsv[nt * 2 + c] : 0.f;
      }
    }
    float p0[4], p1[4] = {0.f, 0.f, 0.f, 0.f};
    const float a0 = online_update(x0, m0, l0, p0);
    float a1 = 1.f;
    if (ROWS16) a1 = online_update(x1, m1, l1, p1);
    if constexpr (TPV) {
      // columns 2t, 2t + 1 of O^T are query rows 2t, 2t + 1, whose factors
      // live in lanes 8t and 8t + 4
      const float r0 = __shfl_sync(0xffffffffu, a0, 8 * t);
      const float r1 = __shfl_sync(0xffffffffu, a0, 8 * t + 4);
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        o[mt][0] *= r0;
        o[mt][1] *= r1;
        o[mt][2] *= r0;
        o[mt][3] *= r1;
      }
    } else {
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= a0;
        o[n][1] *= a0;
        if (ROWS16) {
          o[n][2] *= a1;
          o[n][3] *= a1;
        }
      }
    }
    // P as the A operand of P V (k = this warp's 16 tokens).
    trace_ready(p0[0]);
    trace_ready(o[0][0]);
    const unsigned long long tc3 = trace_clock();
    tr_c[2] += tc3 - tc2;
    uint32_t pa[4];
    if constexpr (FP8) {  // fold the value scales into P (f16)
      pa[0] = pack_f16x2(p0[0] * vsv[0], p0[1] * vsv[1]);
      pa[1] = pack_f16x2(p1[0] * vsv[0], p1[1] * vsv[1]);
      pa[2] = pack_f16x2(p0[2] * vsv[2], p0[3] * vsv[3]);
      pa[3] = pack_f16x2(p1[2] * vsv[2], p1[3] * vsv[3]);
    } else {
      pa[0] = pack_bf16x2(p0[0], p0[1]);
      pa[1] = pack_bf16x2(p1[0], p1[1]);
      pa[2] = pack_bf16x2(p0[2], p0[3]);
      pa[3] = pack_bf16x2(p1[2], p1[3]);
    }

    // Values of masked tokens may be anything (even NaN): zero them in the
    // B fragments so that 0 * V cannot produce NaN.
    uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
    if (partial) {
      // k indices 2t, 2t + 1 (vm0) and 2t + 8, 2t + 9 (vm1): keys tok0 + 2t ..
      // (FP8: logical keys 4t .. 4t + 3, in token rows v8_row[0..3])
      const int base = tok0 - ws * 16;
      const int ta = FP8 ? base + v8_row[0] : tok0 + 2 * t, tb = FP8 ? base + v8_row[1] : ta + 1;
      const int tc = FP8 ? base + v8_row[2] : tok0 + 2 * t + 8, td = FP8 ? base + v8_row[3] : tc + 1;
      vm0 = (ta < t_end ? 0x0000ffffu : 0u) | (tb < t_end ? 0xffff0000u : 0u);
      vm1 = (tc < t_end ? 0x0000ffffu : 0u) | (td < t_end ? 0xffff0000u : 0u);
    }
    if constexpr (FP8) {
      // n-tile n = 4J + jj, fragment column g is d = (D/8) g + n: lane (g, t)
      // loads bytes (D/8) g .. + D/8 - 1 of the rows of logical keys
      // 4t .. 4t + 3 (word J of each: d = (D/8) g + 4J ..) and transposes the
      // words J so that byte e of word jj is key 4t + e at d = (D/8) g + 4J + jj.
      const uint8_t* vraw = smem + st * kStageBytes + F8::kOffV8;
      uint32_t vw[4][D / 32];
#pragma unroll
      for (int e = 0; e < 4; ++e) lds_fp8_words<D, D / 32>(vraw, v8_row[e], (D / 8) * g, vw[e]);
      // Masking costs two ANDs per mma, so only the tile holding the split end
      // pays for it.
      auto pv = [&](auto masked) {
#pragma unroll
        for (int J = 0; J < D / 32; ++J) {
          const uint32_t lo01 = __byte_perm(vw[0][J], vw[1][J], 0x5140),
                         hi01 = __byte_perm(vw[0][J], vw[1][J], 0x7362);
          const uint32_t lo23 = __byte_perm(vw[2][J], vw[3][J], 0x5140),
                         hi23 = __byte_perm(vw[2][J], vw[3][J], 0x7362);
          const uint32_t x[4] = {__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo01, lo23, 0x7632),
                                 __byte_perm(hi01, hi23, 0x5410), __byte_perm(hi01, hi23, 0x7632)};
          if constexpr (TPV) {
            // d-tile mt = 2J + u: its rows g, g + 8 are d = (D/8) g + 4J + 2u
            // and + 1, i.e. words x[2u], x[2u + 1]; P^T is pa[0], pa[2]
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              uint32_t a[4] = {e4m3x2_to_f16x2(x[2 * u]), e4m3x2_to_f16x2(x[2 * u + 1]),
                               e4m3x2_to_f16x2(x[2 * u] >> 16), e4m3x2_to_f16x2(x[2 * u + 1] >> 16)};
              if constexpr (decltype(masked)::value) {
                a[0] &= vm0;
                a[1] &= vm0;
                a[2] &= vm1;
                a[3] &= vm1;
              }
              mma_f16_16816(o[2 * J + u], a, pa[0], pa[2]);
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              uint32_t b0 = e4m3x2_to_f16x2(x[jj]), b1 = e4m3x2_to_f16x2(x[jj] >> 16);
              if constexpr (decltype(masked)::value) {
                b0 &= vm0;
                b1 &= vm1;
              }
              mma_f16_16816(o[4 * J + jj], pa, b0, b1);
            }
          }
        }
      };
      if (partial)
        pv(std::true_type{});
      else
        pv(std::false_type{});
    } else {
#pragma unroll
      for (int jj = 0; jj < D / 16; ++jj) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_trans(vbase + Lay::offset(v_row, jj * 2 + v_chk), v0, v1, v2, v3);
        mma_bf16_16816(o[2 * jj], pa, v0 & vm0, v1 & vm1);
        mma_bf16_16816(o[2 * jj + 1], pa, v2 & vm0, v3 & vm1);
      }
    }
    trace_ready(o[0][0]);
    trace_ready(o[D / 16 - 1][3]);
    tr_c[3] += trace_clock() - tc3;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
  }
  (void)aborted;
  const unsigned long long tr_loop1 = kTrace ? globaltimer_ns() : 0ull;
  if (kTrace && tr_rec && lane == 0 && warp < 8) {
    tr_c[4] = trace_clock() - tr_c[4];
#pragma unroll
    for (int k = 0; k < 6; ++k) tr_rec[8 + 6 * warp + k] = tr_c[k];
  }

  l0 = quad_sum(l0);
  if (ROWS16) l1 = quad_sum(l1);

  // ------------------------------------------- merge the four warp partials --
  const unsigned long long te0 = trace_clock();
  named_bar_sync(1, kCW * 32);
  const unsigned long long te1 = trace_clock();
  const bool failed = *reinterpret_cast<volatile int*>(&abort_flag) != 0 ||
                      (PAGED && *reinterpret_cast<volatile int*>(&bad_page) != 0);
  float* mO = reinterpret_cast<float*>(smem);  // [warps][16][D]
  float2* mML = reinterpret_cast<float2*>(smem + kCW * 16 * D * 4);  // [warps][16]
  static_assert(kCW * 16 * D * 4 + kCW * 16 * 8 <=
                    NSTAGE * (FP8 ? Fp8Layout<D>::kStageBytes : DecodeLayout<D>::kStageBytes),
                "the warp partials reuse the stage ring");
  if (!failed) {
    if constexpr (TPV) {  // O^T d-tile mt = 2J + u: rows g, g + 8 are d = (D/8) g + 4J + 2u, + 1
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        const int d0 = (D / 8) * g + 4 * (mt >> 1) + 2 * (mt & 1);
        *reinterpret_cast<float2*>(&mO[(warp * 16 + 2 * t) * D + d0]) = make_float2(o[mt][0], o[mt][2]);
        *reinterpret_cast<float2*>(&mO[(warp * 16 + 2 * t + 1) * D + d0]) =
            make_float2(o[mt][1], o[mt][3]);
      }
    }
#pragma unroll
    for (int n = 0; n < (TPV ? 0 : D / 8); ++n) {
      if constexpr (FP8) {  // fragment column c of n-tile n is d = (D/8) c + n
        const int col = (D / 4) * t + n;
        mO[(warp * 16 + g) * D + col] = o[n][0];
        mO[(warp * 16 + g) * D + col + D / 8] = o[n][1];
        if (ROWS16) {
          mO[(warp * 16 + g + 8) * D + col] = o[n][2];
          mO[(warp * 16 + g + 8) * D + col + D / 8] = o[n][3];
        }
      } else {
        const int col = n * 8 + 2 * t;
        *reinterpret_cast<float2*>(&mO[(warp * 16 + g) * D + col]) = make_float2(o[n][0], o[n][1]);
        if (ROWS16)
          *reinterpret_cast<float2*>(&mO[(warp * 16 + g + 8) * D + col]) =
              make_float2(o[n][2], o[n][3]);
      }
    }
    if (t == 0) {
      mML[warp * 16 + g] = make_float2(m0, l0);
      if (ROWS16) mML[warp * 16 + g + 8] = make_float2(m1, l1);
    }
  }
  named_bar_sync(1, kCW * 32);
  const unsigned long long te2 = trace_clock();

  constexpr int V4 = D / 4;
  // Item e: row r = e / V4, columns 4 c4 .. 4 c4 + 3 of the merged partial.
  auto merge_item = [&](int e, bool live) {
    const int r = (e / V4) & 15, c4 = e % V4;
    const size_t row = out_row(r);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float M = -INFINITY, Lsum = 0.f;
    if (!failed) {
#pragma unroll
      for (int w = 0; w < kCW; ++w) M = fmaxf(M, mML[w * 16 + r].x);
      const float ref = (M == -INFINITY) ? 0.f : M;
#pragma unroll
      for (int w = 0; w < kCW; ++w) {
        const float2 ml = mML[w * 16 + r];
        const float a = ex2_approx(ml.x - ref);
        Lsum += a * ml.y;
        const float4 ow = *reinterpret_cast<const float4*>(&mO[(w * 16 + r) * D + c4 * 4]);
        acc.x += a * ow.x;
        acc.y += a * ow.y;
        acc.z += a * ow.z;
        acc.w += a * ow.w;
      }
    } else {
      M = NAN;
      Lsum = NAN;
      acc = make_float4(NAN, NAN, NAN, NAN);
    }
    if (!live) return;
    if constexpr (CLUSTER) {
      // this CTA's partial, kept for the cluster merge (m in base-2 units)
      float* cO = reinterpret_cast<float*>(smem + kClusterPartOff<D>);
      float2* cML = reinterpret_cast<float2*>(smem + kClusterPartOff<D> + 16 * D * 4);
      *reinterpret_cast<float4*>(&cO[r * D + c4 * 4]) = acc;
      if (c4 == 0) cML[r] = make_float2(M, Lsum);
    } else if (p.n_split == 1) {
      const float inv = 1.f / Lsum;
      uint2 packed;
      packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      if (in_bounds(row * D + c4 * 4, 4, n_rows * D, p.err))
        *reinterpret_cast<uint2*>(&p.out[row * D + c4 * 4]) = packed;
      if (c4 == 0 && in_bounds(row, 1, n_rows, p.err)) p.lse[row] = (M + log2f(Lsum)) * kLn2;
    } else {
      const size_t idx = row * p.n_split + split;
      if (in_bounds(idx * D + c4 * 4, 4, n_rows * p.n_split * D, p.err))
        *reinterpret_cast<float4*>(&p.ws_O[idx * D + c4 * 4]) = acc;
      if (c4 == 0 && in_bounds(idx, 1, n_rows * p.n_split, p.err))
        p.ws_ml[idx] = make_float2(M * kLn2, Lsum);
    }
  };
  if constexpr (FP8 && !ROWS16 && NGRP == 1) {
    // (three CTAs per SM at 128 registers: the rolled loop)
    for (int e = threadIdx.x; e < R * V4; e += kCW * 32) merge_item(e, true);
  } else {
    // A compile-time trip count (rows r < 16, and < 8 without ROWS16, keep
    // every shared-memory read in bounds), so that the items' loads overlap;
    // only the stores of items past R * V4 are skipped.
    constexpr int kMaxR = ROWS16 || CLUSTER ? 16 : 8;
    constexpr int kMergeIt = (kMaxR * V4 + kCW * 32 - 1) / (kCW * 32);
#pragma unroll
    for (int it = 0; it < kMergeIt; ++it) {
      const int e = threadIdx.x + it * kCW * 32;
      merge_item(e, e < R * V4);
    }
  }

  if (kTrace && tr_rec && threadIdx.x == 0) {
    tr_rec[56] = te1 - te0;            // waiting for the other consumer warps
    tr_rec[57] = te2 - te1;            // partials into shared memory
    tr_rec[58] = trace_clock() - te2;  // merge and global stores
    tr_rec[59] = tp1 - tp0;            // the sequence length read after the release
    tr_rec[60] = tp2 - tp1;            // the length checks before the roles start
    tr_rec[61] = tp3 - tp2;            // the query fragments
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    tr_rec[0] = tr_entry;
    tr_rec[1] = tr_release;
    tr_rec[2] = tr_loop0;
    tr_rec[3] = tr_loop1;
    tr_rec[4] = globaltimer_ns();
    tr_rec[5] = smid;
    tr_rec[6] = split;
    tr_rec[7] = n_tiles;
  }
  if constexpr (CLUSTER) {
    __syncwarp();
    cluster_sync();  // every partial of the cluster is in place
    const int C = p.n_split;
    const uint32_t rank = cluster_ctarank();
    const uint32_t cO = smem_base + kClusterPartOff<D>;
    const uint32_t cML = cO + 16 * D * 4;
    const int total = R * D, per = (total + C - 1) / C;
    for (int e = threadIdx.x; e < per; e += kConsumerWarps * 32) {
      const int idx = static_cast<int>(rank) * per + e;
      if (idx >= total) break;
      const int r = idx / D, c = idx % D;
      float2 ml[kMaxClusterSplits];
      float Mx = -INFINITY;
      bool bad = false;
#pragma unroll
      for (int q = 0; q < kMaxClusterSplits; ++q) {
        if (q >= C) break;
        ml[q] = ld_dsmem_f32x2(mapa_shared(cML + r * 8, q));
        bad |= isnan(ml[q].x) || isnan(ml[q].y);
        Mx = fmaxf(Mx, ml[q].x);
      }
      const float ref = (Mx == -INFINITY) ? 0.f : Mx;
      float Lt = 0.f, acc = 0.f;
#pragma unroll
      for (int q = 0; q < kMaxClusterSplits; ++q) {
        if (q >= C) break;
        if (ml[q].x == -INFINITY) continue;  // empty split: weight 0
        const float w = ex2_approx(ml[q].x - ref);
        Lt += w * ml[q].y;
        acc += w * ld_dsmem_f32(mapa_shared(cO + (r * D + c) * 4, q));
      }
      const bool poisoned = bad || !(Lt > 0.f);
      const size_t row = out_row(r);
      if (in_bounds(row * D + c, 1, n_rows * D, p.err))
        p.out[row * D + c] = __float2bfloat16(poisoned ? NAN : acc / Lt);
      if (c == 0 && in_bounds(row, 1, n_rows, p.err))
        p.lse[row] = poisoned ? NAN : (Mx + log2f(Lt)) * kLn2;
    }
    __syncwarp();
    cluster_sync();  // no CTA leaves while another may still read its partial
  }
}

// -------------------------------------------------------------- combine ----
// One CTA of four warps per (query head, sequence).  Warp w folds splits
// w, w+4, w+8, ... : each lane loads the (m, l) pair of every split it folds
// (a broadcast) and its D/32 columns of each O partial, all in one round of
// loads, then merges them; the four warp results are merged last.  The merge
// is the associative one of "Attention Kernel 계보" p.4, so the grouping does
// not change the result beyond rounding.  The kernel may start before the
// decode kernel ends (programmatic dependent launch); it reads nothing before
// griddepcontrol.wait.
// CHUNK = splits per warp per round of loads: 16, or 8 when every warp folds
// at most 8 splits, which halves the registers so that twice as many CTAs
// (rows) are resident at once.
constexpr int kCombineThreads = 128;
constexpr int kCombineWarps = kCombineThreads / 32;

template <int D, int CHUNK>
__global__ void __launch_bounds__(kCombineThreads, CHUNK == 8 ? 7 : 4)
    gqa_decode_combine_kernel(const CombineParams p) {
  constexpr int kCombineChunk = CHUNK;
  constexpr int VEC = D / 32;  // columns per lane
  __shared__ float s_m[kCombineWarps], s_l[kCombineWarps];
  __shared__ int s_bad[kCombineWarps];
  __shared__ __align__(16) float s_o[kCombineWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, b = blockIdx.y;
  const size_t row = (size_t)b * p.H_q + h;
  // A following split kernel may be scheduled now; it waits for this grid.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float2* ml = p.ws_ml + row * p.n_split;
  const float* O = p.ws_O + row * p.n_split * D + lane * VEC;

  float M = -INFINITY, L = 0.f, acc[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
  bool bad = false;
  for (int base = warp; base < p.n_split; base += kCombineWarps * kCombineChunk) {
    float2 mlv[kCombineChunk];
    float ov[kCombineChunk][VEC];
#pragma unroll
    for (int c = 0; c < kCombineChunk; ++c) {
      const int s = base + kCombineWarps * c;
      const bool in = s < p.n_split;
      mlv[c] = in ? ml[s] : make_float2(-INFINITY, 0.f);
      // this lane's VEC columns in one load: the workspace is 256-byte
      // aligned and a row of D floats is a multiple of 16 bytes
      if constexpr (VEC == 4) {
        const float4 w = in ? *reinterpret_cast<const float4*>(O + (size_t)s * D)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        ov[c][0] = w.x;
        ov[c][1] = w.y;
        ov[c][2] = w.z;
        ov[c][3] = w.w;
      } else if constexpr (VEC == 2) {
        const float2 w = in ? *reinterpret_cast<const float2*>(O + (size_t)s * D)
                            : make_float2(0.f, 0.f);
        ov[c][0] = w.x;
        ov[c][1] = w.y;
      } else {
        ov[c][0] = in ? O[(size_t)s * D] : 0.f;
      }
    }
    float cm = -INFINITY;
#pragma unroll
    for (int c = 0; c < kCombineChunk; ++c) {
      bad |= isnan(mlv[c].x) || isnan(mlv[c].y);
      cm = fmaxf(cm, mlv[c].x);
    }
    const float Mn = fmaxf(M, cm);
    const float ref = (Mn == -INFINITY) ? 0.f : Mn;
    const float a_old = (M == -INFINITY) ? 0.f : ex2_approx((M - ref) * kLog2e);
    L *= a_old;
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] *= a_old;
#pragma unroll
    for (int c = 0; c < kCombineChunk; ++c) {
      // an empty split (m = -inf) has weight 0 and its O (never written) is not used
      const bool live = mlv[c].x != -INFINITY;
      const float w = live ? ex2_approx((mlv[c].x - ref) * kLog2e) : 0.f;
      L += w * mlv[c].y;
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc[v] += live ? w * ov[c][v] : 0.f;
    }
    M = Mn;
  }
  if (lane == 0) {
    s_m[warp] = M;
    s_l[warp] = L;
    s_bad[warp] = bad;
  }
#pragma unroll
  for (int v = 0; v < VEC; ++v) s_o[warp][lane * VEC + v] = acc[v];
  __syncthreads();
  if (warp != 0) return;
  float Mt = -INFINITY;
  bool poisoned = false;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) {
    Mt = fmaxf(Mt, s_m[w]);
    poisoned |= s_bad[w] != 0;
  }
  const float ref = (Mt == -INFINITY) ? 0.f : Mt;
  float Lt = 0.f, tot[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) tot[v] = 0.f;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) {
    const float a = (s_m[w] == -INFINITY) ? 0.f : ex2_approx((s_m[w] - ref) * kLog2e);
    Lt += a * s_l[w];
#pragma unroll
    for (int v = 0; v < VEC; ++v) tot[v] += a * s_o[w][lane * VEC + v];
  }
  poisoned |= !(Lt > 0.f);  // every split empty, or NaN
  const float inv = poisoned ? NAN : 1.f / Lt;
  __nv_bfloat16* dst = p.out + row * D + lane * VEC;
  const size_t rows = (size_t)p.B * p.H_q;
  if (in_bounds(row * D + lane * VEC, VEC, rows * D, p.err)) {
#pragma unroll
    for (int v = 0; v < VEC; ++v) dst[v] = __float2bfloat16(tot[v] * inv);
  }
  if (lane == 0 && in_bounds(row, 1, rows, p.err)) p.lse[row] = poisoned ? NAN : Mt + logf(Lt);
}

// The same merge for at most kColsSplits splits and few rows: one warp per 32
// columns, one column per lane, each warp folding every split itself.  All
// loads are one round and no cross-warp merge follows, which shortens the
// dependent chain; the (m, l) loads are repeated by every warp (L1 hits).  It
// needs more registers than the kernel above, so it serves grids that fit on
// the GPU at once, four per SM (the Llama3-70B decode: 64 rows of 19 splits).
constexpr int kColsSplits = 32;

template <int D>
__global__ void __launch_bounds__(D, 4) gqa_decode_combine_cols_kernel(const CombineParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, b = blockIdx.y;
  const size_t row = (size_t)b * p.H_q + h;
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int col = warp * 32 + lane;
  const float2* ml = p.ws_ml + row * p.n_split;
  const float* O = p.ws_O + row * p.n_split * D + col;
  float2 mlv[kColsSplits];
  float ov[kColsSplits];
#pragma unroll
  for (int s = 0; s < kColsSplits; ++s) {
    const bool in = s < p.n_split;
    mlv[s] = in ? ml[s] : make_float2(-INFINITY, 0.f);
    ov[s] = in ? O[(size_t)s * D] : 0.f;
  }
  bool bad = false;
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < kColsSplits; ++s) {
    bad |= isnan(mlv[s].x) || isnan(mlv[s].y);
    M = fmaxf(M, mlv[s].x);
  }
  const float ref = (M == -INFINITY) ? 0.f : M;
  float L = 0.f, acc = 0.f;
#pragma unroll
  for (int s = 0; s < kColsSplits; ++s) {
    // an empty split (m = -inf) has weight 0 and its O (never written) is not used
    const bool live = mlv[s].x != -INFINITY;
    const float w = live ? ex2_approx((mlv[s].x - ref) * kLog2e) : 0.f;
    L += w * mlv[s].y;
    acc += live ? w * ov[s] : 0.f;
  }
  const bool poisoned = bad || !(L > 0.f);  // every split empty, or NaN
  const float inv = poisoned ? NAN : 1.f / L;
  const size_t rows = (size_t)p.B * p.H_q;
  if (in_bounds(row * D + col, 1, rows * D, p.err))
    p.out[row * D + col] = __float2bfloat16(acc * inv);
  if (col == 0 && in_bounds(row, 1, rows, p.err)) p.lse[row] = poisoned ? NAN : M + logf(L);
}

__global__ void gqa_wait_selftest_kernel(unsigned* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the wait must give up and flag a timeout.
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, limit_ns, err);
}

// Raises the dynamic shared-memory limit of `kern` once per device.
inline cudaError_t set_smem_attr_once(const void* kern, int smem, unsigned char* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;  // benign race: idempotent
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
  return e;
}

// CTAs of `kern` (`threads` threads, `smem` bytes) the current device holds at
// once, looked up once per device.
inline cudaError_t resident_ctas(const void* kern, int threads, int smem, int* cache, int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    *out = cache[dev];
    return cudaSuccess;
  }
  int per_sm = 0, sms = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  *out = per_sm * sms;
  if (dev >= 0 && dev < 64) cache[dev] = *out;  // benign race: idempotent
  return cudaSuccess;
}

template <int D, bool ROWS16, int NSTAGE, bool PAGED, bool FP8, int NGRP = 1, bool DYN = false>
cudaError_t launch_split(const DecodeParams& p_in, const CUtensorMap& tm_k,
                         const CUtensorMap& tm_v, const CUtensorMap& tm_ks,
                         const CUtensorMap& tm_vs, cudaStream_t stream) {
  constexpr int smem = decode_smem_bytes<D, NSTAGE, FP8>();
  constexpr int threads = (kConsumerWarps * NGRP + 1) * 32;
  auto kern = gqa_decode_split_kernel<D, ROWS16, NSTAGE, PAGED, FP8, false, NGRP, DYN>;
  static unsigned char done[64];
  static int resident[64];
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(kern), smem, done);
  if (e != cudaSuccess) return e;
  int fit = 0;
  e = resident_ctas(reinterpret_cast<const void*>(kern), threads, smem, resident, &fit);
  if (e != cudaSuccess) return e;
  DecodeParams p = p_in;
  // The L2 prefetch pays only when every CTA is resident while the previous
  // kernel drains; a CTA of a later wave would prefetch what it loads next.
  const long long ctas = (long long)p.n_split * p.n_rg * p.H_kv * p.B;
  constexpr int kPf =
      prefetch_tiles(FP8 ? Fp8Layout<D>::kTxBytes : DecodeLayout<D>::kStageBytes);
  p.prefetch_tiles = ctas <= fit ? kPf : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_split * p.n_rg, p.H_kv, p.B);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = GQA_SPLIT_PDL ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, tm_k, tm_v, tm_ks, tm_vs, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// SMs of the current device, looked up once per device.
inline cudaError_t sm_count(int* out) {
  static int cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    *out = cache[dev];
    return cudaSuccess;
  }
  e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && dev >= 0 && dev < 64) cache[dev] = *out;  // benign race: idempotent
  return e;
}

template <int D, bool PAGED, bool FP8, bool DYN = false>
cudaError_t launch_split_rows(const DecodeParams& p, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, const CUtensorMap& tm_ks,
                              const CUtensorMap& tm_vs, cudaStream_t stream) {
  constexpr int NSTAGE = FP8 ? GQA_DECODE_STAGES_FP8 : (D >= 128 ? GQA_DECODE_STAGES_D128 : 6);
  if constexpr (FP8) {
    // One CTA per SM: two consumer groups and a deep ring (the per-tile E4M3
    // conversions need more warps per SM than one group gives); otherwise
    // several single-group CTAs share each SM.
    constexpr int DEEP = GQA_DECODE_STAGES_FP8_ONE_WAVE;
    int sms = 0;
    cudaError_t e = sm_count(&sms);
    if (e != cudaSuccess) return e;
    if ((long long)p.n_split * p.n_rg * p.H_kv * p.B <= sms) {
      constexpr int NG = GQA_FP8_ONE_WAVE_GROUPS;
      if (p.T_q * p.G > 8)
        return launch_split<D, true, DEEP, PAGED, FP8, NG>(p, tm_k, tm_v, tm_ks, tm_vs, stream);
      return launch_split<D, false, DEEP, PAGED, FP8, NG>(p, tm_k, tm_v, tm_ks, tm_vs, stream);
    }
  }
  if constexpr (!FP8 && D >= 128) {
    // When the grid has at most one CTA per SM, a deeper ring (which leaves no
    // room for a second CTA) keeps more bytes in flight on each SM: measured
    // for Llama3-70B at 32K (152 CTAs), 23.3 -> 21.8 us for the split kernel;
    // with more CTAs than SMs two shallow rings per SM are faster.
    constexpr int DEEP = GQA_DECODE_STAGES_D128_ONE_WAVE;
    int sms = 0;
    cudaError_t e = sm_count(&sms);
    if (e != cudaSuccess) return e;
    if ((long long)p.n_split * p.n_rg * p.H_kv * p.B <= sms) {
      if (p.T_q * p.G > 8)
        return launch_split<D, true, DEEP, PAGED, FP8, 1, DYN>(p, tm_k, tm_v, tm_ks, tm_vs, stream);
      return launch_split<D, false, DEEP, PAGED, FP8, 1, DYN>(p, tm_k, tm_v, tm_ks, tm_vs, stream);
    }
  }
  if (p.T_q * p.G > 8)  // rows g + 8 are live (in the first row group at least)
    return launch_split<D, true, NSTAGE, PAGED, FP8, 1, DYN>(p, tm_k, tm_v, tm_ks, tm_vs, stream);
  return launch_split<D, false, NSTAGE, PAGED, FP8, 1, DYN>(p, tm_k, tm_v, tm_ks, tm_vs, stream);
}

template <bool PAGED, bool FP8, bool DYN = false>
cudaError_t launch_split_d(const DecodeParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const CUtensorMap& tm_ks, const CUtensorMap& tm_vs,
                           cudaStream_t stream) {
  switch (p.d) {
    case 32: return launch_split_rows<32, PAGED, FP8, DYN>(p, tm_k, tm_v, tm_ks, tm_vs, stream);
    case 64: return launch_split_rows<64, PAGED, FP8, DYN>(p, tm_k, tm_v, tm_ks, tm_vs, stream);
    case 128: return launch_split_rows<128, PAGED, FP8, DYN>(p, tm_k, tm_v, tm_ks, tm_vs, stream);
    default: return cudaErrorInvalidValue;
  }
}

// The cluster-merge launch: grid (C, H_kv, B) in clusters of (C, 1, 1), C =
// p.n_split.  `probe` only reports whether such clusters can be resident.
template <int D, bool ROWS16>
cudaError_t launch_fused(const DecodeParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                         bool probe, cudaStream_t stream) {
  constexpr int NSTAGE = D >= 128 ? GQA_DECODE_FUSED_STAGES_D128 : 6;
  constexpr int smem = decode_smem_bytes<D, NSTAGE, false>();
  static_assert(kClusterPartOff<D> + 16 * D * 4 + 16 * 8 <= NSTAGE * DecodeLayout<D>::kStageBytes,
                "the cluster partial fits in the stage buffers");
  auto kern = gqa_decode_split_kernel<D, ROWS16, NSTAGE, false, false, true>;
  static unsigned char done[64];
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(kern), smem, done);
  if (e != cudaSuccess) return e;
  if (p.n_split > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_split, p.H_kv, p.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.n_split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = GQA_SPLIT_PDL ? 2 : 1;
  if (probe) {
    int n = 0;
    cfg.numAttrs = 1;  // the cluster shape alone decides residency
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    return n >= 1 ? cudaSuccess : cudaErrorInvalidConfiguration;
  }
  e = cudaLaunchKernelEx(&cfg, kern, tm_k, tm_v, tm_k, tm_v, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, int CHUNK>
cudaError_t launch_comb(const CombineParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.H_q, p.B);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = GQA_COMBINE_PDL ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gqa_decode_combine_kernel<D, CHUNK>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_comb_cols(const CombineParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.H_q, p.B);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = GQA_COMBINE_PDL ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gqa_decode_combine_cols_kernel<D>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_split(const DecodeParams& p, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, cudaStream_t stream) {
  if (p.tile_ctr) {
    if (p.T_q != 1 || p.n_rg != 1 || p.n_split < 2) return cudaErrorInvalidValue;
    return launch_split_d<false, false, true>(p, tm_k, tm_v, tm_k, tm_v, stream);
  }
  return launch_split_d<false, false>(p, tm_k, tm_v, tm_k, tm_v, stream);
}

cudaError_t launch_decode_paged(const DecodeParams& p, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, cudaStream_t stream) {
  return launch_split_d<true, false>(p, tm_k, tm_v, tm_k, tm_v, stream);
}

cudaError_t launch_decode_fp8(const DecodeParams& p, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, const CUtensorMap& tm_ks,
                              const CUtensorMap& tm_vs, cudaStream_t stream) {
  if (p.block_table) return launch_split_d<true, true>(p, tm_k, tm_v, tm_ks, tm_vs, stream);
  return launch_split_d<false, true>(p, tm_k, tm_v, tm_ks, tm_vs, stream);
}

cudaError_t launch_decode_fused(const DecodeParams& p, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, bool probe, cudaStream_t stream) {
  if (p.n_split < 1 || p.n_split > kMaxClusterSplits) return cudaErrorInvalidValue;
  const bool rows16 = p.T_q * p.G > 8;
  switch (p.d) {
    case 32:
      return rows16 ? launch_fused<32, true>(p, tm_k, tm_v, probe, stream)
                    : launch_fused<32, false>(p, tm_k, tm_v, probe, stream);
    case 64:
      return rows16 ? launch_fused<64, true>(p, tm_k, tm_v, probe, stream)
                    : launch_fused<64, false>(p, tm_k, tm_v, probe, stream);
    case 128:
      return rows16 ? launch_fused<128, true>(p, tm_k, tm_v, probe, stream)
                    : launch_fused<128, false>(p, tm_k, tm_v, probe, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_combine(const CombineParams& p, cudaStream_t stream) {
  // Up to 32 splits over at most four rows per SM: the column kernel (one
  // round of loads, no cross-warp merge; measured 24.08 against 24.30 us for
  // the Llama3-70B decode step).  Otherwise the warp-per-split-group kernel.
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  if (p.n_split <= kColsSplits && (long long)p.B * p.H_q <= 4LL * sms) {
    switch (p.d) {
      case 32: return launch_comb_cols<32>(p, stream);
      case 64: return launch_comb_cols<64>(p, stream);
      case 128: return launch_comb_cols<128>(p, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  const bool small = p.n_split <= kCombineWarps * 8;  // one round of 8 per warp
  switch (p.d) {
    case 32: return small ? launch_comb<32, 8>(p, stream) : launch_comb<32, 16>(p, stream);
    case 64: return small ? launch_comb<64, 8>(p, stream) : launch_comb<64, 16>(p, stream);
    case 128: return small ? launch_comb<128, 8>(p, stream) : launch_comb<128, 16>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_wait_selftest(unsigned* err, uint64_t limit_ns, cudaStream_t stream) {
  gqa_wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace gqa

extern "C" gqa_status gqa_trace_clear(void) {
  if (!gqa::kTrace) return GQA_ERR_UNSUPPORTED;
  static unsigned long long zeros[gqa::kTraceCtas * gqa::kTraceWords];
  return cudaMemcpyToSymbol(gqa::g_trace, zeros, sizeof zeros) == cudaSuccess &&
                 gqa::prefill_trace_clear() == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

extern "C" gqa_status gqa_trace_read(void* host, size_t bytes) {
  if (!gqa::kTrace) return GQA_ERR_UNSUPPORTED;
  constexpr size_t total = sizeof(unsigned long long) * gqa::kTraceCtas * gqa::kTraceWords;
  if (!host || bytes > total) return GQA_ERR_INVALID_ARG;
  return cudaMemcpyFromSymbol(host, gqa::g_trace, bytes) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}
