// decode_tc.cu -- split-KV decode of many query rows per KV head on the
// fifth-generation tensor cores.
//
// What it computes: the multi-token decode of decode.cu.  The queries are the
// last T_q positions L - T_q .. L - 1 of each sequence (L = seq_lens[b]),
// query t sees keys 0 .. L - T_q + t, and the G query heads of a KV head read
// that head's K and V ("Attention Kernel 계보" p.2 §1, p.15 §2/§4; the chunk
// alignment of ADR-0060 §0.5.3 for short chunks).  The split-K decode of p.18
// §4: one CTA per (split, KV head, sequence) streams its split's keys once and
// leaves an unnormalised partial (m, l, O) per query row for the log-sum-exp
// merge of the combine kernel (p.4); with one split it writes O and LSE.
//
// Where decode.cu folds the T_q * G rows of a KV head into 16-row mma.sync
// tiles (one CTA per 16 rows, each re-reading K and V), this kernel puts all
// of them (up to 128) in the M rows of one tcgen05.mma tile, so every K/V
// tile is read once per split however many rows there are:
//   S_j = Q K_j^T       (M = 128 rows, N = 128 keys, K = d = 128; SS form)
//   O  += P_j V_j       (P_j bf16 in tensor memory; TS form)
// with FA2's loop order (p.8-p.9): Q stays in shared memory, K and V tiles of
// 128 keys stream through two three-slot rings, loaded in the order the tensor
// core consumes them (K_0, then K_{j+1}, V_j), so a K slot is refilled as soon
// as its S has been computed; (m, l, O) are updated online.  S is
// double-buffered in tensor memory: the tensor core computes S_{j+1} while the
// softmax warps turn S_j into P_j.
//
// Roles (192 threads):
//   warp 0      TMA producer: Q once, then the K and V tiles.
//   warp 1      allocates tensor memory and issues every tcgen05.mma.
//   warps 2-5   softmax + epilogue, thread = query row r = 32 (warp % 4) + lane
//               (tensor-memory lane r).
// Query row r of the tile is query t = r / G of head kv * G + r % G, the order
// in which the TMA box {d/2, G, T_q} of Q lands; rows r >= T_q * G are zero.
// Tensor memory (512 columns x 128 lanes, fp32): S_0 | S_1 | O; P_j (bf16, two
// per column) overwrites the first 64 columns of S_(j%2) once it has been read.
//
// O is rescaled only when a row's running maximum grows by more than 2^8
// (base 2), as in prefill.cu: l and O share one reference, so O / l holds.
//
// PAGED = true: the cache is a pool of fixed-size pages reached through a
// block table (p.17 §2-§4, p.18 §5); each 128-key tile arrives as boxes of
// min(page_size, 128) rows, one page each.  A page index outside the pool is
// reported and replaced by page 0, and the CTA's outputs become NaN.
#include "tcgen05.cuh"

namespace gqa {
namespace {

constexpr int kTcThreads = 192;
constexpr int kTcSlots = 3;                     // slots per ring (K and V)
#ifndef GQA_TC_PREFETCH_TILES
#define GQA_TC_PREFETCH_TILES 3  // 128-key tiles a CTA may warm in L2 before its dependency wait
#endif
static_assert(GQA_TC_PREFETCH_TILES >= 0 && GQA_TC_PREFETCH_TILES <= 32, "one tile per lane");
constexpr int kTcKeys = 128;                    // keys per ring stage
constexpr uint32_t kTileB = 128u * 128u * 2u;   // one 128 x 128 bf16 tile
constexpr uint32_t kHalfB = kTileB / 2;         // 128 rows x 128 bytes
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kTileB;              // K ring after Q
constexpr uint32_t kOffV = kOffK + kTcSlots * kTileB;  // then the V ring
constexpr uint32_t kTcSmem = kOffV + kTcSlots * kTileB + 1024;
constexpr uint32_t kColO = 256;                 // O after S_0, S_1
constexpr float kRescaleLog2 = 8.f;

template <bool PAGED>
__global__ void __launch_bounds__(kTcThreads, 1)
    gqa_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full, drain;
  __shared__ __align__(8) uint64_t k_full[kTcSlots], k_empty[kTcSlots], v_full[kTcSlots],
      v_empty[kTcSlots];
  __shared__ __align__(8) uint64_t s_full[2], p_ready[2], pv_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int bad_page;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, kv = blockIdx.y, b = blockIdx.z;
  const int G = p.G, rows = p.T_q * G;  // rows <= 128 (checked on the host)
  auto out_row = [&](int r) -> size_t {
    return ((size_t)b * p.T_q + r / G) * p.H_q + kv * G + r % G;
  };
  const size_t n_rows = (size_t)p.B * p.T_q * p.H_q;  // rows of out, lse and the workspace
  // NaN outputs of a row (one split), or its partial (m, l) alone (O is not read)
  auto write_nan_or_ml = [&](size_t row, float2 ml) {
    if (p.n_split == 1) {
      if (in_bounds(row * 128, 128, n_rows * 128, p.err))
        for (int c = 0; c < 128; ++c) p.out[row * 128 + c] = __float2bfloat16(NAN);
      if (in_bounds(row, 1, n_rows, p.err)) p.lse[row] = NAN;
    } else if (in_bounds(row * p.n_split + split, 1, n_rows * p.n_split, p.err)) {
      p.ws_ml[row * p.n_split + split] = ml;
    }
  };

  // Set-up that touches no global memory runs before the dependency wait.
  volatile int* abort_v = &abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&drain), 1);
    for (int s = 0; s < kTcSlots; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&s_full[x]), 1);
      mbar_init(smem_u32(&p_ready[x]), 4);
    }
    mbar_init(smem_u32(&pv_done), 1);
    abort_flag = 0;
    bad_page = 0;
    fence_barrier_init();
  }
  // Q rows past T_q * G are zero (their S, P and O rows are never stored, but
  // stay finite); the TMA box fills rows 0 .. rows - 1 only.
  for (int i = threadIdx.x; i < (128 - rows) * 16; i += kTcThreads) {
    const int r = rows + i / 16, c = i % 16;
    st_shared_v4(sb + kOffQ + (c >> 3) * kHalfB + r * 128 + (c & 7) * 16, 0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
    tc_fence_before();
  }
  // While the previous kernel finishes, the producer warp prefetches this
  // split's first K/V tiles into L2, one tile (paged: one page segment of a
  // tile) per lane; the launcher enables it when the whole grid is resident at
  // once.  The extent comes from a relaxed load of seq_lens[b] and, for a
  // paged cache, the rows from relaxed loads of the block table; they may see
  // values from before the previous kernel's writes and only aim the prefetch
  // (an index outside the pool is skipped).  A prefetch hands no data to the
  // kernel and L2 is where writes become coherent.
  if (warp == 0 && p.prefetch_tiles > 0) {
    const int h = PAGED ? min(p.page_size, kTcKeys) : kTcKeys;  // rows per box
    const int nb = kTcKeys / h;
    const int i = lane / nb, sub = lane % nb;
    int L_hint;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(L_hint) : "l"(p.seq_lens + b));
    const int tk = split * p.chunk + i * kTcKeys + sub * h;
    if (i < p.prefetch_tiles && tk < min(min(p.S_max, L_hint), split * p.chunk + p.chunk)) {
      int row = b * p.S_max + tk;
      bool ok = true;
      if constexpr (PAGED) {
        int pg;
        asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];"
                     : "=r"(pg)
                     : "l"(p.block_table + (size_t)b * p.max_blocks + tk / p.page_size));
        ok = pg >= 0 && pg < p.num_pages;
        row = pg * p.page_size + tk % p.page_size;
      }
      if (ok)
        for (int dh = 0; dh < 2; ++dh) {
          tma_prefetch_l2_3d(&tm_k, dh * 64, kv, row);
          tma_prefetch_l2_3d(&tm_v, dh * 64, kv, row);
        }
    }
  }

  // Launched as a programmatic dependent of the previous kernel in the
  // stream: nothing is read or written before that kernel has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int L = p.seq_lens[b];
  const bool bad = L < p.T_q || L > p.S_max;  // (L >= T_q >= 1 otherwise)
  const int t0 = split * p.chunk;
  const int t_end = bad ? 0 : min(t0 + p.chunk, L);
  const int n = t_end > t0 ? (t_end - t0 + kTcKeys - 1) / kTcKeys : 0;
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (bad || n == 0) {
    // A bad length: NaN outputs and the error bit.  An empty split: the merge
    // identity (-inf, 0); its O is not written.  (One split is never empty.)
    if (bad && threadIdx.x == 0 && split == 0 && kv == 0) atomicOr(p.err, kErrBadSeqLen);
    for (int r = threadIdx.x; r < rows; r += kTcThreads)
      write_nan_or_ml(out_row(r), bad ? make_float2(NAN, NAN) : make_float2(-INFINITY, 0.f));
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
    return;
  }

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

  if (warp == 0) {
    // ----------------------------------------------------------- TMA producer --
    // The whole warp runs the loop (so that the page indices of a tile are
    // read in parallel, one per lane); lane 0 arms each barrier before any
    // copy of its tile is issued.
    const uint32_t qb = smem_u32(&q_full);
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      mbar_arrive_expect_tx(qb, static_cast<uint32_t>(rows) * 256u);
      for (int dh = 0; dh < 2; ++dh)
        tma_load_3d(sb + kOffQ + dh * kHalfB, &tm_q, qb, dh * 64, kv * G, b * p.T_q);
    }
    // K_0, then K_{j+1} and V_j: the order in which the tensor core reads
    // them.  A tile's slot is refilled once the MMA that read it completed.
    int k_issued = 0, v_issued = 0;
    // Paged: boxes of h rows, one page each (h = page_size up to 128), box i
    // of a tile issued by lane i.  Each tile's page indices are read once,
    // two tiles ahead, so the reads are in flight while the producer waits for
    // a slot; K_j and V_j use the same boxes.  A box wholly past the split end
    // reads rows past the pool, which TMA fills with zeros, so that every tile
    // still receives its full bytes.
    const int h = PAGED ? min(p.page_size, kTcKeys) : kTcKeys;
    const int nb = kTcKeys / h;  // <= 8 (page_size >= 16)
    struct Box {
      int pg;
      bool has;
    };
    auto fetch = [&](int j) -> Box {  // this lane's page of tile j
      Box x;
      const int tok = t0 + j * kTcKeys + lane * h;
      x.has = PAGED && lane < nb && j < n && tok < t_end;
      x.pg = x.has ? p.block_table[(size_t)b * p.max_blocks + tok / p.page_size] : 0;
      return x;
    };
    // every K/V tile is read by this CTA alone, once: evict-first in L2
    const uint64_t kv_pol = l2_policy_evict_first();
    auto issue = [&](bool is_k, int j, Box x) -> bool {
      const int slot = j % kTcSlots;
      uint64_t* empty = is_k ? &k_empty[slot] : &v_empty[slot];
      if (j >= kTcSlots && !wait_all(empty, ((j / kTcSlots) - 1) & 1)) return false;
      const uint32_t fb = smem_u32(is_k ? &k_full[slot] : &v_full[slot]);
      const uint32_t dst = sb + (is_k ? kOffK : kOffV) + slot * kTileB;
      const CUtensorMap* map = is_k ? &tm_k : &tm_v;
      const int tok0 = t0 + j * kTcKeys;
      if constexpr (!PAGED) {
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, kTileB);
          for (int dh = 0; dh < 2; ++dh)
            tma_load_3d(dst + dh * kHalfB, map, fb, dh * 64, kv, b * p.S_max + tok0, kv_pol);
        }
      } else {
        const bool bad = x.has && (x.pg < 0 || x.pg >= p.num_pages);
        const int row = x.has ? (bad ? 0 : x.pg) * p.page_size + (tok0 + lane * h) % p.page_size
                              : p.num_pages * p.page_size;
        // a bad index is recorded before lane 0's arrive releases it
        if (__any_sync(0xffffffffu, bad) && lane == 0) {
          if (!*reinterpret_cast<volatile int*>(&bad_page)) atomicOr(p.err, kErrBadPage);
          *reinterpret_cast<volatile int*>(&bad_page) = 1;
        }
        if (lane == 0) mbar_arrive_expect_tx(fb, kTileB);
        __syncwarp();
        if (lane < nb)
          for (int dh = 0; dh < 2; ++dh)
            tma_load_3d(dst + dh * kHalfB + lane * h * 128, map, fb, dh * 64, kv, row, kv_pol);
      }
      return true;
    };
    Box box_j = fetch(0), box_j1 = fetch(1);  // tiles j and j + 1
    bool ok = issue(true, 0, box_j);
    if (ok) k_issued = 1;
    for (int j = 0; ok && j < n; ++j) {
      const Box box_j2 = fetch(j + 2);
      if (j + 1 < n) {
        ok = issue(true, j + 1, box_j1);
        if (!ok) break;
        k_issued = j + 2;
      }
      ok = issue(false, j, box_j);
      if (ok) v_issued = j + 1;
      box_j = box_j1;
      box_j1 = box_j2;
    }
    if (lane == 0) {
      // The next kernel in the stream may be scheduled now; it waits for this
      // grid before it reads anything.
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      // No copy may still target shared memory when the CTA exits.
      for (int j = max(0, k_issued - kTcSlots); j < k_issued; ++j)
        mbar_wait(smem_u32(&k_full[j % kTcSlots]), (j / kTcSlots) & 1, p.wait_ns, p.err);
      for (int j = max(0, v_issued - kTcSlots); j < v_issued; ++j)
        mbar_wait(smem_u32(&v_full[j % kTcSlots]), (j / kTcSlots) & 1, p.wait_ns, p.err);
      mbar_wait(qb, 0, p.wait_ns, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer --
    constexpr uint32_t idS = instr_desc_bf16_f32(128, 128, false);
    constexpr uint32_t idPV = instr_desc_bf16_f32(128, 128, true);
    auto issue_s = [&](int x, int slot) {  // S_x = Q K^T
      const uint32_t kb = sb + kOffK + slot * kTileB;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * kHalfB + (kk & 3) * 32;
        tc_mma_ss(tmem + 128 * x, smem_desc_sw128(sb + kOffQ + off, 16, 1024),
                  smem_desc_sw128(kb + off, 16, 1024), idS, kk > 0);
      }
    };
    auto issue_pv = [&](int x, int slot, bool acc) {  // O (+)= P_x V, P_x in tensor memory
      const uint32_t vb = sb + kOffV + slot * kTileB;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc_mma_ts(tmem + kColO, tmem + 128 * x + 8 * kk, smem_desc_sw128(vb + kk * 2048, kHalfB, 1024),
                  idPV, (acc || kk > 0) ? 1 : 0);
    };
    // P_j V_j once V_j has landed and the softmax has written P_j; then V_j's
    // slot is free.
    auto finish_tile = [&](int j) -> bool {
      if (!wait_all(&v_full[j % kTcSlots], (j / kTcSlots) & 1)) return false;
      if (!wait_all(&p_ready[j & 1], (j >> 1) & 1)) return false;
      tc_fence_after();
      issue_pv(j & 1, j % kTcSlots, j > 0);
      tc_commit(smem_u32(&pv_done));
      tc_commit(smem_u32(&v_empty[j % kTcSlots]));
      return true;
    };
    bool ok = wait_all(&q_full, 0);
    // Tensor-pipe order S_0, S_1, P_0 V_0, S_2, P_1 V_1, ...: S_{j+1} runs while
    // the softmax works on S_j.  S_j overwrites P_{j-2}, whose P V was issued
    // before it (the MMAs of one thread execute in issue order).
    for (int j = 0; ok && j < n; ++j) {
      const int slot = j % kTcSlots;
      if (!wait_all(&k_full[slot], (j / kTcSlots) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_s(j & 1, slot);
      tc_commit(smem_u32(&s_full[j & 1]));
      tc_commit(smem_u32(&k_empty[slot]));
      if (j > 0 && !finish_tile(j - 1)) ok = false;
    }
    if (ok) finish_tile(n - 1);
    // Every MMA issued here has completed (and every commit has landed)
    // before tensor memory is released.
    tc_commit(smem_u32(&drain));
    mbar_wait(smem_u32(&drain), 0, p.wait_ns, p.err);
    __syncwarp();
  } else {
    // ------------------------------------------------- softmax + epilogue --
    const int quarter = warp & 3;  // tensor-memory lanes 32 * quarter ..
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tO = tmem + lane_base + kColO;
    const float c2 = p.scale_log2;
    // Keys below `lim` are visible from this row: query t = r / G sees keys up
    // to L - T_q + t, and this split ends at t_end.  The bound shared by every
    // real row is lim_lo; tiles wholly below it need no mask.
    const int lim = r < rows ? min(t_end, L - p.T_q + 1 + r / G) : t_end;
    const int lim_lo = min(t_end, L - p.T_q + 1);
    float m_ref = -INFINITY, l = 0.f;
    bool alive = true;
    for (int j = 0; j < n; ++j) {
      const int x = j & 1;
      const uint32_t tS = tmem + lane_base + 128 * x;
      if (!wait_all(&s_full[x], (j >> 1) & 1)) {
        alive = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));

      const int tb = t0 + j * kTcKeys;  // key of column 0
      if (tb + kTcKeys > lim_lo) {
        const int vis = lim - tb;  // columns c < vis are visible
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= vis) sr[c] = __float_as_uint(-INFINITY);
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 128; c += 8) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          m4[u] = fmax3(m4[u], __uint_as_float(sr[c + 2 * u]), __uint_as_float(sr[c + 2 * u + 1]));
      }
      const float m_tile = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * c2;  // c2 > 0
      float alpha = 1.f;
      bool rescale = false;
      // No visible key in this row so far: l and O are 0, nothing to rescale.
      if (m_ref == -INFINITY) {
        m_ref = m_tile;
      } else if (m_tile > m_ref + kRescaleLog2) {
        alpha = ex2_approx(m_ref - m_tile);
        m_ref = m_tile;
        rescale = true;
      }
      const float neg = m_ref == -INFINITY ? 0.f : -m_ref;

      // P = 2^(x c2 - m_ref), summed in fp32, written as packed bf16 over the
      // first 64 columns of S_x: the A operand of P_j V_j.
      float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t pk[8];
#pragma unroll
        for (int g8 = 0; g8 < 16; g8 += 8) {
          float e[8];
#pragma unroll
          for (int u = 0; u < 8; u += 2)
            ffma2(e[u], e[u + 1], __uint_as_float(sr[c0 + g8 + u]), __uint_as_float(sr[c0 + g8 + u + 1]),
                  c2, c2, neg, neg);
#pragma unroll
          for (int u = 0; u < 8; ++u) e[u] = ex2_approx(e[u]);
          fadd2(sa0, sa1, sa0, sa1, e[0], e[1]);
          fadd2(sb0, sb1, sb0, sb1, e[2], e[3]);
          fadd2(sa0, sa1, sa0, sa1, e[4], e[5]);
          fadd2(sb0, sb1, sb0, sb1, e[6], e[7]);
#pragma unroll
          for (int u = 0; u < 4; ++u) pk[g8 / 2 + u] = pack_bf16x2(e[2 * u], e[2 * u + 1]);
        }
        tmem_st8(tS + c0 / 2, pk);
      }
      l = l * alpha + ((sa0 + sa1) + (sb0 + sb1));

      // P_{j-1} V_{j-1} has completed, so O is stable (P_j V_j is issued only
      // after p_ready below).  Every tile takes this wait, so the completions
      // of pv_done are consumed strictly in order.
      if (j > 0) {
        if (!wait_all(&pv_done, (j - 1) & 1)) {
          alive = false;
          break;
        }
        tc_fence_after();
      }
      // O rows of this warp whose reference moved: O *= alpha (never on the
      // first tile, where m_ref starts from -inf).
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_wait_ld();
          reg_fence32(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + 32 * c, o);
        }
      }

      // Cache rows at or past the split end may hold anything (even NaN: the
      // padding of a sequence, or the next sequence's rows), and 0 * NaN would
      // reach O through P V, so row r of this V tile is zeroed if it lies past
      // the end, once the tile has landed (it is refilled only after P_j V_j).
      if (tb + kTcKeys > t_end) {
        if (!wait_all(&v_full[j % kTcSlots], (j / kTcSlots) & 1)) {
          alive = false;
          break;
        }
        if (tb + r >= t_end) {
          const uint32_t vrow = sb + kOffV + (j % kTcSlots) * kTileB + r * 128;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16)
              st_shared_v4(vrow + hh * kHalfB + c16 * 16, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_ready[x]));
    }

    // Epilogue: the last P V, then O / l and LSE, or this split's partial.
    // Paged: a bad page index (recorded before the producer's arrive on the
    // last V tile, which this wait acquires) makes the outputs NaN.
    bool page_ok = true;
    if (PAGED && alive) {
      if (wait_all(&v_full[(n - 1) % kTcSlots], ((n - 1) / kTcSlots) & 1))
        page_ok = *reinterpret_cast<volatile int*>(&bad_page) == 0;
      else
        alive = false;
    }
    if (alive && page_ok && wait_all(&pv_done, (n - 1) & 1)) {
      tc_fence_after();
      const bool store = r < rows;
      const size_t row = store ? out_row(r) : 0;
      const bool one = p.n_split == 1;
      const float inv = 1.f / l;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_wait_ld();
        reg_fence32(o);
        if (!store) continue;
        const size_t at = (one ? row : row * p.n_split + split) * 128 + 32 * c;
        if (!in_bounds(at, 32, n_rows * (one ? 1 : p.n_split) * 128, p.err)) continue;
        if (one) {
          uint4* d4 = reinterpret_cast<uint4*>(p.out + row * 128 + 32 * c);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            d4[v] = w;
          }
        } else {
          // (the workspace is 256-byte aligned, a partial row 512 bytes)
          float* d = p.ws_O + (row * p.n_split + split) * 128 + 32 * c;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st_global_v8(d + 8 * v, o[8 * v], o[8 * v + 1], o[8 * v + 2], o[8 * v + 3], o[8 * v + 4],
                         o[8 * v + 5], o[8 * v + 6], o[8 * v + 7]);
        }
      }
      if (store) {
        if (one && in_bounds(row, 1, n_rows, p.err))
          p.lse[row] = (m_ref + log2f(l)) * kLn2;
        else if (!one && in_bounds(row * p.n_split + split, 1, n_rows * p.n_split, p.err))
          // m in natural-log units; a row with no visible key: (-inf, 0)
          p.ws_ml[row * p.n_split + split] = make_float2(m_ref * kLn2, l);
      }
    } else if (r < rows) {  // a wait gave up, or a bad page: this row's outputs are NaN
      write_nan_or_ml(out_row(r), make_float2(NAN, NAN));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeParams& p_in, const CUtensorMap& tm_q,
                             const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             cudaStream_t stream) {
  if (p_in.d != 128 || p_in.T_q * p_in.G > 128 || p_in.chunk % kTcKeys != 0)
    return cudaErrorInvalidValue;
  static unsigned char attr_done[64];
  static int sm_count[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(gqa_decode_tc_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gqa_decode_tc_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) {
      sm_count[dev] = sms;
      attr_done[dev] = 1;
    }
  }
  DecodeParams p = p_in;
  // One CTA per SM: the L2 prefetch pays only when every CTA is resident
  // while the previous kernel drains, and for a paged cache only with pages
  // of at least 64 tokens (T_q = 8, Llama3-70B 32K: 28.9 -> 26.5 us at page
  // 128, but 32.8 -> 34.3 us at page 16, whose 24 small boxes per CTA cost
  // more than they hide).
  const long long ctas = (long long)p.n_split * p.H_kv * p.B;
  const int sms = (dev >= 0 && dev < 64) ? sm_count[dev] : 0;
  const bool small_pages = p.block_table && p.page_size < 64;
  p.prefetch_tiles = (ctas <= sms && !small_pages) ? GQA_TC_PREFETCH_TILES : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_split, p.H_kv, p.B);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = p.block_table ? cudaLaunchKernelEx(&cfg, gqa_decode_tc_kernel<true>, tm_q, tm_k, tm_v, p)
                    : cudaLaunchKernelEx(&cfg, gqa_decode_tc_kernel<false>, tm_q, tm_k, tm_v, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gqa
