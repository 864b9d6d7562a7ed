// prefill.cu -- causal grouped-query prefill on the fifth-generation tensor cores.
//
// What it computes (S_q = S_kv): for query row i of head h, O = softmax over
// keys j <= i of tau * q_i . k_j, times V, with h reading KV head floor(h / G)
// ("Attention Kernel 계보" p.2 §1, p.13 §1, p.15 §2).  The loop order is FA2's
// (p.8-p.9): a query tile stays resident while the key/value tiles stream past,
// the running (m, l, O) state is updated online and O is divided by l once.
//
// Work item = (sequence b, KV head, pair of query heads of that KV head's group,
// 128-row query tile).  The two query heads share every K/V tile the CTA loads
// (the GQA reuse of p.15 §4/§7), and their two softmaxes alternate with the
// tensor core: while one warpgroup turns S into P for its head, the tensor core
// runs the other head's P V and next Q K^T (the two-warpgroup ping-pong of p.11,
// here with tcgen05 and tensor memory instead of wgmma and registers).
// Causal block classes (p.13 §2-§4): key tiles past the query tile are never
// loaded; tiles fully below the diagonal run unmasked; only the diagonal tile
// is masked, by select.  Items are handed to persistent CTAs heaviest first in
// a snake order (p.13 §6).
//
// Roles (384 threads):
//   warp 0      TMA producer: Q pair once per item, then K_j, V_j through a
//               five-slot shared-memory ring.
//   warp 1      allocates tensor memory and issues every tcgen05.mma (the
//               whole warp runs the loop, one elected lane issues):
//               S_X = Q_X K_j^T and O_X += P_X V_j for X in {A, B}.
//   warps 2-3   idle.
//   warps 4-7   softmax + epilogue of head A (thread = one query row).
//   warps 8-11  softmax + epilogue of head B.
// Tensor memory (512 columns x 128 lanes, fp32): S_A | S_B (128 columns each)
// | O_A | O_B (DP columns each); P_X (bf16, two per column) overwrites the
// first 64 columns of S_X once S_X has been read, and is the tensor-memory A
// operand of O_X += P_X V.
// Shared memory: Q_A, Q_B and the K/V slots, every tile stored as DP/64
// halves of 128 rows x 128 bytes with the 128-byte swizzle.
//
// Head dimensions: DP = 128 serves d = 128 (five K/V slots of 32 KB); DP = 64
// serves d = 64 (ten slots of 16 KB) and d = 32, whose tiles are loaded as
// 64-element boxes over a 32-element-wide tensor: TMA fills columns 32..63 with
// zeros, which add nothing to Q K^T and give zero columns of O that are never
// stored.
//
// O is rescaled only when a row's running maximum grows by more than 2^8
// (base 2); p = 2^(x - m_ref) then stays <= 2^8, and because l and O always
// share the same reference m_ref, the final O / l is unchanged (p.3 §5 holds
// for any reference value, not only the running maximum).
#include <climits>

#include "gqa_attn.h"
#include "tcgen05.cuh"

#ifndef GQA_TRACE
#define GQA_TRACE 0
#endif

namespace gqa {

// A build with GQA_TRACE=1 records clock64 stamps of the causal kernel's
// pipeline: for the first work item of CTAs 0..7 and its first 64 key tiles,
// one record of 16 words per (CTA, head X of the pair, tile j), laid out
// [CTA][X][j][word]; see gqa_trace_prefill_read in the public header.
constexpr bool kPTrace = GQA_TRACE != 0;
constexpr int kPtCtas = 8, kPtTiles = 64, kPtWords = 16;
__device__ unsigned long long g_ptrace[kPTrace ? kPtCtas * 2 * kPtTiles * kPtWords : 1];

cudaError_t prefill_trace_clear() {
  if (!kPTrace) return cudaSuccess;
  static unsigned long long zeros[kPtCtas * 2 * kPtTiles * kPtWords];
  return cudaMemcpyToSymbol(g_ptrace, zeros, sizeof zeros);
}

namespace {

// Stamp word `w` of the record of (this CTA, head x, tile j) of the CTA's
// first item (k == 0); a no-op in other builds.
__device__ __forceinline__ void pt_stamp(int k, int x, int j, int w) {
  if constexpr (kPTrace) {
    if (k == 0 && blockIdx.x < kPtCtas && j < kPtTiles) {
      unsigned long long t;
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(t)::"memory");
      g_ptrace[((blockIdx.x * 2 + x) * kPtTiles + j) * kPtWords + w] = t;
    }
  }
}

constexpr int kPThreads = 384;
// Shared-memory layout for tiles of 128 rows x DP bf16 columns (DP = 64 or 128).
template <int DP>
struct PrefillLayout {
  static_assert(DP == 64 || DP == 128, "padded head width");
  static constexpr int kSlots = DP == 128 ? 5 : 10;         // K/V ring slots
  static constexpr int kHalves = DP / 64;                    // 128-byte-wide halves per tile
  static constexpr uint32_t kHalfB = 128u * 128u;            // 128 rows x 128 bytes
  static constexpr uint32_t kTileB = kHalves * kHalfB;       // one 128 x DP tile
  static constexpr uint32_t kOffQ = 0;                       // Q_A, Q_B
  static constexpr uint32_t kOffRing = 2 * kTileB;           // K/V slots
  static constexpr uint32_t kSmem = kOffRing + kSlots * kTileB + 1024;
};
constexpr float kRescaleLog2 = 8.f;
// Registers per thread: 168 at launch (384 threads, one CTA per SM); warps
// 0-3 (TMA, MMA, idle) give theirs up to the two softmax warpgroups.
constexpr int kRegsLaunch = 168, kRegsCtl = 88, kRegsSoftmax = 208;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= kPThreads * kRegsLaunch,
              "the register split must fit in the launch's registers");

struct Item {
  int b, kv, hp, qt, part;
};

// k-th item of this CTA: rounds of `grid` items, alternating direction, items
// ordered by descending query tile (the heaviest first); the parts of one
// split item are neighbours.
__device__ __forceinline__ bool item_of(int k, int n_items, int per_qt, int n_qt, int n_pairs,
                                        int H_kv, int n_part, Item& it) {
  const int grid = gridDim.x, cta = blockIdx.x;
  const int idx = k * grid + ((k & 1) ? (grid - 1 - cta) : cta);
  if (idx >= n_items) return false;
  it.qt = n_qt - 1 - idx / per_qt;
  int r = idx % per_qt;
  it.part = r % n_part;
  r /= n_part;
  it.hp = r % n_pairs;
  r /= n_pairs;
  it.kv = r % H_kv;
  it.b = r / H_kv;
  return true;
}

// Key tiles an item visits.  Causal prefill (GENERAL = false): tiles 0..qt.
// Chunk (GENERAL = true): the chunk is the last S rows of a sequence of L =
// seq_lens[b] tokens (ADR-0060 §0.5.3 q_block_meta, §5.4), so tile row r sits at
// absolute position a = (L - S) + 128 qt + r and sees keys a - W .. a; tiles
// wholly before the window or after the last row are never loaded.  A bad
// length is replaced by S (all accesses stay in bounds) and the rows get NaN.
struct Geom {
  int j0, n, q_off;
  bool bad;
};
constexpr int kLensSm = 256;  // sequence lengths kept in shared memory

template <bool GENERAL>
__device__ __forceinline__ Geom item_geom(const PrefillParams& p, const Item& it,
                                          const int* lens_sm) {
  Geom g;
  if (!GENERAL) {
    g.j0 = 0;
    g.n = it.qt + 1;
    g.q_off = 0;
    g.bad = false;
    return g;
  }
  int L = !p.seq_lens ? p.S_kv : it.b < kLensSm ? lens_sm[it.b] : p.seq_lens[it.b];
  g.bad = L < p.S || L > p.S_kv;
  if (g.bad) L = p.S;
  g.q_off = L - p.S;
  const int first = g.q_off + it.qt * 128;
  const int last = g.q_off + min(p.S, it.qt * 128 + 128) - 1;
  const int lo = p.window >= 0 ? max(0, first - p.window) : 0;
  g.j0 = lo / 128;
  g.n = last / 128 - g.j0 + 1;
  if (p.n_part > 1) {  // this part's share of the key tiles (possibly none)
    const int a = g.j0 + (it.part * g.n) / p.n_part;
    const int b = g.j0 + ((it.part + 1) * g.n) / p.n_part;
    g.j0 = a;
    g.n = b - a;
  }
  return g;
}

template <bool GENERAL, int DP>
__global__ void __launch_bounds__(kPThreads, 1)
    gqa_prefill_causal_kernel(const __grid_constant__ CUtensorMap tm_q,
                              const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using Lay = PrefillLayout<DP>;
  constexpr int kSlots = Lay::kSlots;
  constexpr uint32_t kTileB = Lay::kTileB, kHalfB = Lay::kHalfB;
  constexpr uint32_t kOffQ = Lay::kOffQ, kOffRing = Lay::kOffRing;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full, q_empty, drain;
  __shared__ __align__(8) uint64_t slot_full[kSlots], slot_empty[kSlots];
  __shared__ __align__(8) uint64_t s_full[2], p_ready[2], o_full[2], o_empty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  // every role derives each item's key range from seq_lens[b]: read it once
  __shared__ int lens_sm[GENERAL ? kLensSm : 1];

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_qt = (p.S + 127) / 128;
  const int n_pairs = (p.G + 1) / 2;
  const int per_qt = p.B * p.H_kv * n_pairs * p.n_part;
  const int n_items = n_qt * per_qt;
  const int n_rounds = (n_items + gridDim.x - 1) / gridDim.x;
  volatile int* abort_v = &abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&q_empty), 1);
    mbar_init(smem_u32(&drain), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_u32(&slot_full[s]), 1);
      mbar_init(smem_u32(&slot_empty[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&s_full[x]), 1);
      mbar_init(smem_u32(&p_ready[x]), 4);
      mbar_init(smem_u32(&o_full[x]), 1);
      mbar_init(smem_u32(&o_empty[x]), 4);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  if (GENERAL && p.seq_lens)
    for (int i = threadIdx.x; i < min(p.B, kLensSm); i += kPThreads) lens_sm[i] = p.seq_lens[i];
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  // A bounded wait that also gives up once another role has aborted.  A phase
  // that has already completed passes at once: the abort flag is read only on
  // the slow path, since a shared-memory load in front of every wait delays
  // the MMA warp's next issue (the tensor core queues about one instruction).
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait(smem_u32(bar), parity)) return true;
    if (*abort_v) return false;
    if (mbar_wait(smem_u32(bar), parity, p.wait_ns, p.err)) return true;
    *abort_v = 1;
    return false;
  };

  // The same, taken by every lane of a warp, with one agreed result.
  auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
    const bool ok = wait(bar, parity);
    return __all_sync(0xffffffffu, ok);
  };

  if (warp < 4) {
    regs_dec<kRegsCtl>();
    if (warp == 0) {
      // ------------------------------------------------------- TMA producer --
      if (lane == 0) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
        uint32_t ring = 0, q_iter = 0;
        bool ok = true;
        for (int k = 0; ok && k < n_rounds; ++k) {
          Item it;
          if (!item_of(k, n_items, per_qt, n_qt, n_pairs, p.H_kv, p.n_part, it)) continue;
          const bool pair = 2 * it.hp + 1 < p.G;
          const int hA = it.kv * p.G + 2 * it.hp;
          const Geom gm = item_geom<GENERAL>(p, it, lens_sm);
          if (GENERAL && gm.n == 0) continue;  // an empty part: nothing to load
          if (q_iter > 0 && !wait(&q_empty, (q_iter - 1) & 1)) break;
          const uint32_t qb = smem_u32(&q_full);
          mbar_arrive_expect_tx(qb, pair ? 2 * kTileB : kTileB);
          for (int dh = 0; dh < Lay::kHalves; ++dh) {
            tma_load_4d(sb + kOffQ + dh * kHalfB, &tm_q, qb, dh * 64, hA, it.qt * 128, it.b);
            if (pair)
              tma_load_4d(sb + kOffQ + kTileB + dh * kHalfB, &tm_q, qb, dh * 64, hA + 1,
                          it.qt * 128, it.b);
          }
          ++q_iter;
          const int n = gm.n;
          for (int j = 0; ok && j < n; ++j) {
            for (int t = 0; t < 2; ++t) {  // K_j then V_j
              const uint32_t slot = ring % kSlots;
              if (ring >= kSlots && !wait(&slot_empty[slot], ((ring / kSlots) - 1) & 1)) {
                ok = false;
                break;
              }
              const uint32_t fb = smem_u32(&slot_full[slot]);
              mbar_arrive_expect_tx(fb, kTileB);
              const CUtensorMap* m = t == 0 ? &tm_k : &tm_v;
              for (int dh = 0; dh < Lay::kHalves; ++dh)
                tma_load_4d(sb + kOffRing + slot * kTileB + dh * kHalfB, m, fb, dh * 64, it.kv,
                            (gm.j0 + j) * 128, it.b);
              ++ring;
            }
          }
        }
        // No copy may still target shared memory when the CTA exits.
        for (uint32_t r = ring > kSlots ? ring - kSlots : 0; r < ring; ++r)
          mbar_wait(smem_u32(&slot_full[r % kSlots]), (r / kSlots) & 1, p.wait_ns, p.err);
        if (q_iter > 0) mbar_wait(smem_u32(&q_full), (q_iter - 1) & 1, p.wait_ns, p.err);
      }
    } else if (warp == 1) {
      // ------------------------------------------------- MMA issuer (warp 1) --
      {
        constexpr uint32_t idS = instr_desc_bf16_f32(128, 128, false);
        constexpr uint32_t idPV = instr_desc_bf16_f32(128, DP, true);
        auto issue_s = [&](int x, uint32_t slot) {  // S_x = Q_x K^T, K = DP in steps of 16
          const uint32_t qa = sb + kOffQ + x * kTileB, kb = sb + kOffRing + slot * kTileB;
  #pragma unroll
          for (int kk = 0; kk < DP / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kHalfB + (kk & 3) * 32;
            tc_mma_ss(tmem + 128 * x, smem_desc_sw128(qa + off, 16, 1024),
                      smem_desc_sw128(kb + off, 16, 1024), idS, kk > 0);
          }
        };
        auto issue_pv = [&](int x, uint32_t slot, bool acc) {  // O_x (+)= P_x V, P_x in TMEM
          const uint32_t vb = sb + kOffRing + slot * kTileB;
  #pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_ts(tmem + 256 + DP * x, tmem + 128 * x + 8 * kk,
                      smem_desc_sw128(vb + kk * 2048, kHalfB, 1024), idPV, (acc || kk > 0) ? 1 : 0);
        };
        uint32_t ring = 0, q_iter = 0, pr_ph[2] = {0, 0}, oe_ph[2] = {0, 0};
        bool o_busy[2] = {false, false};
        bool ok = true;
        for (int k = 0; ok && k < n_rounds; ++k) {
          Item it;
          if (!item_of(k, n_items, per_qt, n_qt, n_pairs, p.H_kv, p.n_part, it)) continue;
          const bool pair = 2 * it.hp + 1 < p.G;
          const int nx = pair ? 2 : 1;
          const int n = item_geom<GENERAL>(p, it, lens_sm).n;
          if (GENERAL && n == 0) continue;  // an empty part: no work
          if (!wait_all(&q_full, q_iter & 1)) break;
          ++q_iter;
          uint32_t kslot = ring % kSlots;
          if (!wait_all(&slot_full[kslot], (ring / kSlots) & 1)) break;
          ++ring;
          tc_fence_after();
          for (int x = 0; x < nx; ++x) {
            issue_s(x, kslot);
            tc_commit(smem_u32(&s_full[x]));
          }
          tc_commit(smem_u32(&slot_empty[kslot]));
          if (n == 1) tc_commit(smem_u32(&q_empty));
          for (int j = 0; ok && j < n; ++j) {
            const uint32_t vslot = ring % kSlots;
            if (lane == 0) pt_stamp(k, 0, j, 15);
            if (!wait_all(&slot_full[vslot], (ring / kSlots) & 1)) {
              ok = false;
              break;
            }
            ++ring;
            const bool more = j + 1 < n;
            for (int x = 0; x < nx; ++x) {
              if (lane == 0) pt_stamp(k, x, j, 11);
              if (!wait_all(&p_ready[x], pr_ph[x])) {
                ok = false;
                break;
              }
              pr_ph[x] ^= 1;
              if (lane == 0) pt_stamp(k, x, j, 12);
              if (j == 0 && o_busy[x]) {  // the previous item's epilogue must have read O_x
                if (!wait_all(&o_empty[x], oe_ph[x])) {
                  ok = false;
                  break;
                }
                oe_ph[x] ^= 1;
                o_busy[x] = false;
              }
              tc_fence_after();
              issue_pv(x, vslot, j > 0);
              if (lane == 0) pt_stamp(k, x, j, 13);
              if (more) {
                if (x == 0) {
                  kslot = ring % kSlots;
                  if (!wait_all(&slot_full[kslot], (ring / kSlots) & 1)) {
                    ok = false;
                    break;
                  }
                  ++ring;
                  tc_fence_after();
                }
                issue_s(x, kslot);
                tc_commit(smem_u32(&s_full[x]));
                if (lane == 0) pt_stamp(k, x, j, 14);
              } else {
                tc_commit(smem_u32(&o_full[x]));
                o_busy[x] = true;
              }
            }
            if (!ok) break;
            tc_commit(smem_u32(&slot_empty[vslot]));
            if (more) {
              tc_commit(smem_u32(&slot_empty[kslot]));
              if (j + 2 == n) tc_commit(smem_u32(&q_empty));
            }
          }
        }
        // Every MMA issued here has completed (and every commit has landed)
        // before tensor memory is released.
        tc_commit(smem_u32(&drain));
        mbar_wait(smem_u32(&drain), 0, p.wait_ns, p.err);
        __syncwarp();
      }
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------ softmax + epilogue ----
    const int x = (warp - 4) >> 2;  // 0: head A, 1: head B
    const int quarter = warp & 3;   // tensor-memory lanes 32*quarter ..
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + 128 * x;
    const uint32_t tO = tmem + lane_base + 256 + DP * x;
    const int n_oc = p.d / 32;  // 32-column chunks of O that are stored
    const float c2 = p.scale_log2;
    uint32_t s_ph = 0, of_ph = 0;
    uint32_t ring_base = 0;  // ring position of this item's K_0 (chunk mode bookkeeping)
    bool alive = true;
    for (int k = 0; alive && k < n_rounds; ++k) {
      Item it;
      if (!item_of(k, n_items, per_qt, n_qt, n_pairs, p.H_kv, p.n_part, it)) continue;
      const bool pair = 2 * it.hp + 1 < p.G;
      if (x == 1 && !pair) continue;
      const int h = it.kv * p.G + 2 * it.hp + x;
      const Geom gm = item_geom<GENERAL>(p, it, lens_sm);
      const int n = gm.n;
      const int q_row = it.qt * 128 + r;
      const size_t ws_row = (static_cast<size_t>(it.b) * p.S + q_row) * p.H_q + h;
      const size_t n_rows = static_cast<size_t>(p.B) * p.S * p.H_q;  // rows of out, lse, workspace
      if (GENERAL && n == 0) {  // an empty part: the merge identity (-inf, 0)
        if (q_row < p.S && in_bounds(ws_row * p.n_part + it.part, 1, n_rows * p.n_part, p.err))
          p.ws_ml[ws_row * p.n_part + it.part] = make_float2(-INFINITY, 0.f);
        continue;
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        if (!wait_all(&s_full[x], s_ph)) {
          alive = false;
          break;
        }
        s_ph ^= 1;
        if (lane == 0) pt_stamp(k, x, j, quarter);
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        if (quarter == 0 && lane == 0) pt_stamp(k, x, j, 8);

        // Row maximum.  Diagonal tile: key column c is visible from row r iff
        // c <= r (select, only on this tile); other tiles are unmasked.
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (!GENERAL) {
          if (j == it.qt) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c > r) sr[c] = __float_as_uint(-INFINITY);
          }
        } else {
          // key 128*jt + c is visible from row r iff du + r - W <= c <= du + r
          const int du = gm.q_off + 128 * (it.qt - gm.j0 - j);
          const bool upper = du < 127;
          const bool lower = p.window >= 0 && du + 127 - p.window > 0;
          if (upper || lower) {
            const int hi = du + r, lo = p.window >= 0 ? du + r - p.window : INT_MIN;
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c > hi || c < lo) sr[c] = __float_as_uint(-INFINITY);
          }
        }
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            m4[t] = fmax3(m4[t], __uint_as_float(sr[c + 2 * t]), __uint_as_float(sr[c + 2 * t + 1]));
        }
        const float m_tile = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * c2;  // c2 > 0
        if constexpr (kPTrace) {  // stamp once the maximum is known
          float mt = m_tile;
          asm volatile("mov.b32 %0, %0;" : "+f"(mt));
          if (quarter == 0 && lane == 0) pt_stamp(k, x, j, 9);
        }
        float alpha = 1.f;
        bool rescale = false;
        // First tile (causal: key 0 is always visible), or, in chunk mode, no
        // visible key in this row so far (l and O are 0, nothing to rescale).
        if (GENERAL ? m_ref == -INFINITY : j == 0) {
          m_ref = m_tile;
        } else if (m_tile > m_ref + kRescaleLog2) {
          alpha = ex2_approx(m_ref - m_tile);
          m_ref = m_tile;
          rescale = true;
        }
        const float neg = (GENERAL && m_ref == -INFINITY) ? 0.f : -m_ref;

        // P = 2^(x c2 - m_ref), summed in fp32, and written as packed bf16 over
        // the first 64 columns of S_x: the A operand of the next P V.  The MMA
        // that overwrites S_x next is issued after that P V (tcgen05.mma
        // instructions of one thread execute in issue order).
        float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 16) {
          uint32_t pk[8];
#pragma unroll
          for (int g8 = 0; g8 < 16; g8 += 8) {
            float e[8];
#pragma unroll
            for (int t = 0; t < 8; t += 2)
              ffma2(e[t], e[t + 1], __uint_as_float(sr[c0 + g8 + t]),
                    __uint_as_float(sr[c0 + g8 + t + 1]), c2, c2, neg, neg);
#pragma unroll
            for (int t = 0; t < 8; ++t) e[t] = ex2_approx(e[t]);
            fadd2(sa0, sa1, sa0, sa1, e[0], e[1]);
            fadd2(sb0, sb1, sb0, sb1, e[2], e[3]);
            fadd2(sa0, sa1, sa0, sa1, e[4], e[5]);
            fadd2(sb0, sb1, sb0, sb1, e[6], e[7]);
#pragma unroll
            for (int t = 0; t < 4; ++t) pk[g8 / 2 + t] = pack_bf16x2(e[2 * t], e[2 * t + 1]);
          }
          tmem_st8(tS + c0 / 2, pk);
        }
        l = l * alpha + ((sa0 + sa1) + (sb0 + sb1));
        if constexpr (kPTrace) {  // stamp once the exponentials are summed
          float lt = l;
          asm volatile("mov.b32 %0, %0;" : "+f"(lt));
          if (quarter == 0 && lane == 0) pt_stamp(k, x, j, 10);
        }

        // O rows of this warp whose reference moved: O *= alpha.  O is stable:
        // the commit that signalled S also covered the previous P V; the next
        // P V is issued only after p_ready below.
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < n_oc; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
            reg_fence32(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + 32 * c, o);
          }
          tmem_wait_st();
        }

        // Chunk mode: cache rows at or past the sequence end may hold anything
        // (even NaN) and 0 * NaN would reach O through P V, so head A's
        // warps zero those rows of the last V tile before P is released (the
        // MMA issues head B's P V only after head A's).
        if (GENERAL && x == 0 && j == n - 1) {
          const int jt = gm.j0 + j;
          const int L_eff = gm.q_off + p.S;
          if (128 * jt + 127 >= L_eff) {
            const uint32_t pos = ring_base + 2 * j + 1;
            if (!wait_all(&slot_full[pos % kSlots], (pos / kSlots) & 1)) {
              alive = false;
              break;
            }
            if (128 * jt + r >= L_eff) {
              const uint32_t row = sb + kOffRing + (pos % kSlots) * kTileB + r * 128;
#pragma unroll
              for (int hh = 0; hh < Lay::kHalves; ++hh)
#pragma unroll
                for (int c16 = 0; c16 < 8; ++c16) st_shared_v4(row + hh * kHalfB + c16 * 16, 0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) pt_stamp(k, x, j, 4 + quarter);
        if (lane == 0) mbar_arrive(smem_u32(&p_ready[x]));
      }
      if (!alive) break;

      // Epilogue: O / l in bf16 and LSE = (m_ref + log2 l) * ln 2.
      if (!wait_all(&o_full[x], of_ph)) break;
      of_ph ^= 1;
      tc_fence_after();
      const float inv = (GENERAL && gm.bad) ? NAN : 1.f / l;
      const bool store = q_row < p.S;
      if (GENERAL && gm.bad && x == 0 && warp == 4 && lane == 0) atomicOr(p.err, kErrBadSeqLen);
      const bool split = GENERAL && p.n_part > 1;
      const int D = p.d;  // row width of out and of the O partials
#pragma unroll 1
      for (int c = 0; c < n_oc; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_wait_ld();
        reg_fence32(o);
        if (split && store && !in_bounds((ws_row * p.n_part + it.part) * D + 32 * c, 32,
                                         n_rows * p.n_part * D, p.err))
          continue;
        if (split && store) {  // this part's unnormalised O, fp32
          // (the workspace is 256-byte aligned, a partial row 4 D >= 128 bytes)
          float* d = p.ws_O + (ws_row * p.n_part + it.part) * D + 32 * c;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st_global_v8(d + 8 * v, o[8 * v], o[8 * v + 1], o[8 * v + 2], o[8 * v + 3], o[8 * v + 4],
                         o[8 * v + 5], o[8 * v + 6], o[8 * v + 7]);
        } else if (!split) {
          // Row r's 32 columns as four 16-byte units u[k] (columns 8k .. 8k+7).
          // A 4 x 4 transpose of units across each quad of lanes leaves lane
          // 4q + t with unit t of the quad's rows 4q .. 4q+3, so that every
          // store instruction writes 64 contiguous bytes of each of 8 rows.
          uint32_t u[4][4];
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
#pragma unroll
            for (int w = 0; w < 4; ++w)
              u[k4][w] = pack_bf16x2(__uint_as_float(o[8 * k4 + 2 * w]) * inv,
                                     __uint_as_float(o[8 * k4 + 2 * w + 1]) * inv);
          const int t = lane & 3;
#pragma unroll
          for (int w = 0; w < 4; ++w) {  // swap the off-diagonal 2 x 2 blocks (lanes t, t ^ 2)
            const uint32_t s0 = (t & 2) ? u[0][w] : u[2][w];
            const uint32_t s1 = (t & 2) ? u[1][w] : u[3][w];
            const uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 2);
            const uint32_t r1 = __shfl_xor_sync(0xffffffffu, s1, 2);
            if (t & 2) { u[0][w] = r0; u[1][w] = r1; } else { u[2][w] = r0; u[3][w] = r1; }
          }
#pragma unroll
          for (int w = 0; w < 4; ++w) {  // transpose each 2 x 2 block (lanes t, t ^ 1)
            const uint32_t s0 = (t & 1) ? u[0][w] : u[1][w];
            const uint32_t s1 = (t & 1) ? u[2][w] : u[3][w];
            const uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 1);
            const uint32_t r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
            if (t & 1) { u[0][w] = r0; u[2][w] = r1; } else { u[1][w] = r0; u[3][w] = r1; }
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) {  // u[v]: unit t of the quad's row v
            const int qrow = it.qt * 128 + quarter * 32 + (lane & ~3) + v;
            const size_t orow = (static_cast<size_t>(it.b) * p.S + qrow) * p.H_q + h;
            if (qrow < p.S && in_bounds(orow * D + 32 * c + 8 * t, 8, n_rows * D, p.err))
              *reinterpret_cast<uint4*>(p.out + orow * D + 32 * c + 8 * t) =
                  make_uint4(u[v][0], u[v][1], u[v][2], u[v][3]);
          }
        }
      }
      const size_t lse_at = (static_cast<size_t>(it.b) * p.H_q + h) * p.S + q_row;
      if (split && store && in_bounds(ws_row * p.n_part + it.part, 1, n_rows * p.n_part, p.err))
        p.ws_ml[ws_row * p.n_part + it.part] =
            gm.bad ? make_float2(NAN, NAN) : make_float2(m_ref, l);
      else if (!split && store && in_bounds(lse_at, 1, n_rows, p.err))
        p.lse[lse_at] = (GENERAL && gm.bad) ? NAN : (m_ref + log2f(l)) * kLn2;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&o_empty[x]));
      if (GENERAL) ring_base += 2 * n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool GENERAL, int DP>
cudaError_t launch_prefill_dp(const PrefillParams& p, const CUtensorMap& tm_q,
                              const CUtensorMap& tm_k, const CUtensorMap& tm_v, int num_sms,
                              cudaStream_t stream) {
  static unsigned char attr_done[64];
  constexpr uint32_t smem = PrefillLayout<DP>::kSmem;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  auto kern = gqa_prefill_causal_kernel<GENERAL, DP>;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = 1;
  }
  const long long n_items =
      (long long)((p.S + 127) / 128) * p.B * p.H_kv * ((p.G + 1) / 2) * (GENERAL ? p.n_part : 1);
  const int grid = (int)(n_items < num_sms ? n_items : num_sms);
  kern<<<grid, kPThreads, smem, stream>>>(tm_q, tm_k, tm_v, p);
  return cudaGetLastError();
}

// d = 128 on 128-wide tiles; d = 64 and d = 32 on 64-wide tiles (d = 32 zero-padded by TMA).
template <bool GENERAL>
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, int num_sms, cudaStream_t stream) {
  switch (p.d) {
    case 128: return launch_prefill_dp<GENERAL, 128>(p, tm_q, tm_k, tm_v, num_sms, stream);
    case 64:
    case 32: return launch_prefill_dp<GENERAL, 64>(p, tm_q, tm_k, tm_v, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Folds the n_part partials of every (b, i, h) row of a split chunk prefill
// (the associative merge of "Attention Kernel 계보" p.4): one warp per row,
// four of the row's d columns per lane (lanes past d / 4 only help with the
// weights).  A part whose rows saw no key is the identity (m = -inf, l = 0); a
// NaN partial (bad sequence length) makes the row NaN.
__global__ void __launch_bounds__(256) gqa_prefill_merge_kernel(const PrefillParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t rows = static_cast<size_t>(p.B) * p.S * p.H_q;
  const size_t row = static_cast<size_t>(blockIdx.x) * 8 + warp;
  if (row >= rows) return;
  const int P = p.n_part;
  const int D = p.d;
  const bool cols = lane * 4 < D;
  float M = -INFINITY;
  bool bad = false;
  for (int q = 0; q < P; ++q) {
    const float2 ml = p.ws_ml[row * P + q];
    bad |= isnan(ml.x) || isnan(ml.y);
    M = fmaxf(M, ml.x);
  }
  const float ref = (M == -INFINITY) ? 0.f : M;
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q = 0; q < P; ++q) {
    const float2 ml = p.ws_ml[row * P + q];
    if (ml.x == -INFINITY) continue;  // never written O is not read
    const float w = exp2f(ml.x - ref);
    L += w * ml.y;
    const float4 o = cols ? reinterpret_cast<const float4*>(p.ws_O + (row * P + q) * D)[lane]
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    acc.x += w * o.x;
    acc.y += w * o.y;
    acc.z += w * o.z;
    acc.w += w * o.w;
  }
  const bool poisoned = bad || !(L > 0.f);
  const float inv = poisoned ? NAN : 1.f / L;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  if (cols && in_bounds(row * D + lane * 4, 4, rows * D, p.err))
    reinterpret_cast<uint2*>(p.out + row * D)[lane] = packed;
  if (lane == 0) {
    const int h = static_cast<int>(row % p.H_q);
    const size_t bi = row / p.H_q;
    const int i = static_cast<int>(bi % p.S);
    const size_t b = bi / p.S;
    if (in_bounds((b * p.H_q + h) * p.S + i, 1, rows, p.err))
      p.lse[(b * p.H_q + h) * p.S + i] = poisoned ? NAN : (M + log2f(L)) * kLn2;
  }
}

}  // namespace

cudaError_t launch_prefill_merge(const PrefillParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.B * p.S * p.H_q;
  const long long blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  gqa_prefill_merge_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefill_causal(const PrefillParams& p, const CUtensorMap& tm_q,
                                  const CUtensorMap& tm_k, const CUtensorMap& tm_v, int num_sms,
                                  cudaStream_t stream) {
  return launch_prefill<false>(p, tm_q, tm_k, tm_v, num_sms, stream);
}

cudaError_t launch_prefill_chunk(const PrefillParams& p, const CUtensorMap& tm_q,
                                 const CUtensorMap& tm_k, const CUtensorMap& tm_v, int num_sms,
                                 cudaStream_t stream) {
  return launch_prefill<true>(p, tm_q, tm_k, tm_v, num_sms, stream);
}

}  // namespace gqa

extern "C" gqa_status gqa_trace_prefill_read(void* host, size_t bytes) {
  if (!gqa::kPTrace) return GQA_ERR_UNSUPPORTED;
  constexpr size_t total =
      sizeof(unsigned long long) * gqa::kPtCtas * 2 * gqa::kPtTiles * gqa::kPtWords;
  if (!host || bytes > total) return GQA_ERR_INVALID_ARG;
  return cudaMemcpyFromSymbol(host, gqa::g_ptrace, bytes) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

