// api.cu -- the C ABI of libgqa_attn.so (declared in include/gqa_attn.h):
// argument checks, TMA tensor-map encoding, the per-device error word and the
// kernel launches.  Nothing here computes attention.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "gqa_attn.h"
#include "internal.h"

namespace {

// One error word per device (a module global is instantiated per context).
__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
std::atomic<uint64_t> g_wait_ns{2000000000ull};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

gqa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA; }

// Device pointer of the error word of the current device (looked up once).
gqa_status error_word(unsigned** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return GQA_ERR_CUDA;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_err_ptr[dev];
  return GQA_OK;
}

int num_sms_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_num_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 148;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

gqa_status get_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_encode) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f)
      return GQA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  *fn = g_encode;
  return GQA_OK;
}

// A tensor map of `rank` dims (innermost first); strides in bytes for dims 1.. .
gqa_status encode_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, int rank,
                      const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                      CUtensorMapSwizzle swz);

gqa_status encode_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swz) {
  return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides, box, swz);
}

gqa_status encode_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, int rank,
                      const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                      CUtensorMapSwizzle swz) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  gqa_status st = get_encoder(&enc);
  if (st != GQA_OK) return st;
  cuuint64_t gdim[5], gstr[4];
  cuuint32_t bdim[5], estr[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estr[i] = 1;
    if (i + 1 < rank) gstr[i] = strides[i];
  }
  CUresult r = enc(map, type, rank, const_cast<void*>(base), gdim,
                   gstr, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GQA_OK : GQA_ERR_INVALID_ARG;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool head_dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

// Query rows (T_q x G) a multi-token decode folds per KV head: four row groups
// of 16, each its own CTA; with d = 128, up to 128 rows in one tensor-core
// tile (used above 16 rows).
constexpr int kMaxMultiRows = 64;
constexpr int kMaxMultiRowsTc = 128;
bool multi_uses_tc(int T_q, int G, int d) { return d == 128 && T_q * G > 16; }

}  // namespace

extern "C" {

const char* gqa_status_str(int status) {
  switch (status) {
    case GQA_OK: return "GQA_OK";
    case GQA_ERR_INVALID_ARG: return "GQA_ERR_INVALID_ARG";
    case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED";
    case GQA_ERR_CUDA: return "GQA_ERR_CUDA";
    case GQA_ERR_TIMEOUT: return "GQA_ERR_TIMEOUT";
    default: return "GQA_ERR_UNKNOWN";
  }
}

int gqa_version(void) { return 100; }

int gqa_attn_decode_split_chunk(int S_max, int n_split) {
  if (S_max < 1 || n_split < 1) return 0;
  const long long per = ((long long)S_max + n_split - 1) / n_split;
  const long long t = gqa::kDecodeTile;
  return (int)((per + t - 1) / t * t);
}

size_t gqa_attn_decode_workspace_bytes(int B, int H_q, int d, int n_split) {
  if (B < 1 || H_q < 1 || d < 1 || n_split <= 1) return 0;
  return gqa::decode_ws_O_offset(B, H_q, n_split) + (size_t)B * H_q * n_split * d * sizeof(float);
}

int gqa_attn_decode_default_splits(int B, int H_kv, int S_max, int device) {
  if (B < 1 || H_kv < 1 || S_max < 1) return 1;
  int sms = 0;
  if (device < 0) {
    sms = num_sms_current_device();
  } else if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
             sms < 1) {
    cudaGetLastError();  // (a device that cannot be queried leaves no sticky error)
    return 1;
  }
  // Up to 1024 tokens one CTA streams the whole sequence: the combine launch
  // then costs more than the split saves (measured: d = 32, 1024 tokens, 6.1 us
  // unsplit against 9.0 us with 8 splits + combine; d = 128 about equal).
  if (S_max <= 1024) return 1;
  // About one CTA per SM (measured best for a single long sequence), with
  // splits of at least 128 tokens and at most 8192 tokens (ragged batches then
  // have enough CTAs to balance).
  const long long groups = (long long)B * H_kv;
  long long n = (sms + groups - 1) / groups;
  const long long most = (S_max + 127) / 128;
  const long long fill = (S_max + 8191) / 8192;
  if (n > most) n = most;
  if (n < fill) n = fill;
  if (n < 1) n = 1;
  if (n > 65535) n = 65535;
  return (int)n;
}

}  // extern "C"

namespace {

// Checks the decode arguments shared by the contiguous and the paged cache,
// encodes the K/V tensor maps (cache viewed as [rows][H_kv][d], boxes of
// box_rows token rows of one head, at most 64 elements / 128 bytes wide,
// swizzled for ldmatrix) and fills the kernel parameters.
gqa_status prepare_decode(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* seq_lens, int B, int S_max, long long rows, int box_rows,
                          int H_q, int H_kv, int d, float scale, int n_split, void* workspace,
                          void* out, float* lse, CUtensorMap* tm_k, CUtensorMap* tm_v,
                          gqa::DecodeParams* p, bool needs_workspace = true) {
  if (!q || !k_cache || !v_cache || !seq_lens || !out || !lse) return GQA_ERR_INVALID_ARG;
  if (B < 1 || S_max < 1 || H_q < 1 || H_kv < 1 || n_split < 1) return GQA_ERR_INVALID_ARG;
  if (B > 65535 || H_kv > 65535 || H_q % H_kv != 0) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (rows > 0x7fffffffLL || n_split > 0x7fffffff) return GQA_ERR_INVALID_ARG;
  if (!head_dim_ok(d) || H_q / H_kv > 16) return GQA_ERR_UNSUPPORTED;
  if (needs_workspace && n_split > 1 && !workspace) return GQA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(seq_lens, 4) || (workspace && !aligned(workspace, 256)))
    return GQA_ERR_INVALID_ARG;

  unsigned* err = nullptr;
  gqa_status st = error_word(&err);
  if (st != GQA_OK) return st;

  const int box_d = d >= 64 ? 64 : d;
  const uint64_t dims[3] = {(uint64_t)d, (uint64_t)H_kv, (uint64_t)rows};
  const uint64_t strides[2] = {(uint64_t)d * 2, (uint64_t)H_kv * d * 2};
  const uint32_t box[3] = {(uint32_t)box_d, 1u, (uint32_t)box_rows};
  const CUtensorMapSwizzle swz = box_d == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if ((st = encode_bf16(tm_k, k_cache, 3, dims, strides, box, swz)) != GQA_OK) return st;
  if ((st = encode_bf16(tm_v, v_cache, 3, dims, strides, box, swz)) != GQA_OK) return st;

  *p = gqa::DecodeParams{};
  p->q = static_cast<const __nv_bfloat16*>(q);
  p->seq_lens = seq_lens;
  p->T_q = 1;
  p->n_rg = 1;
  p->B = B;
  p->S_max = S_max;
  p->H_q = H_q;
  p->H_kv = H_kv;
  p->G = H_q / H_kv;
  p->d = d;
  p->n_split = n_split;
  p->chunk = gqa_attn_decode_split_chunk(S_max, n_split);
  p->scale_log2 = scale * 1.4426950408889634f;
  p->ws_ml = static_cast<float2*>(workspace);
  p->ws_O = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                 gqa::decode_ws_O_offset(B, H_q, n_split))
                      : nullptr;
  p->out = static_cast<__nv_bfloat16*>(out);
  p->lse = lse;
  p->err = err;
  p->wait_ns = g_wait_ns.load();
  return GQA_OK;
}

}  // namespace

extern "C" {

gqa_status gqa_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* seq_lens, int B, int S_max, int H_q, int H_kv, int d,
                           float scale, int n_split, void* workspace, void* out, float* lse,
                           gqa_stream_t stream) {
  CUtensorMap tm_k, tm_v;
  gqa::DecodeParams p;
  gqa_status st = prepare_decode(q, k_cache, v_cache, seq_lens, B, S_max, (long long)B * S_max,
                                 gqa::kDecodeTile, H_q, H_kv, d, scale, n_split, workspace, out,
                                 lse, &tm_k, &tm_v, &p);
  if (st != GQA_OK) return st;
  return cuda_status(gqa::launch_decode_split(p, tm_k, tm_v, reinterpret_cast<cudaStream_t>(stream)));
}

size_t gqa_attn_decode_counter_bytes(int B, int H_kv) {
  if (B < 1 || H_kv < 1) return 0;
  return (size_t)B * H_kv * 2 * sizeof(int32_t);
}

gqa_status gqa_attn_decode_balanced(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* seq_lens, int B, int S_max, int H_q, int H_kv,
                                    int d, float scale, int n_split, void* workspace,
                                    int32_t* counters, void* out, float* lse,
                                    gqa_stream_t stream) {
  if (n_split > 1 && (!counters || !aligned(counters, 4))) return GQA_ERR_INVALID_ARG;
  CUtensorMap tm_k, tm_v;
  gqa::DecodeParams p;
  gqa_status st = prepare_decode(q, k_cache, v_cache, seq_lens, B, S_max, (long long)B * S_max,
                                 gqa::kDecodeTile, H_q, H_kv, d, scale, n_split, workspace, out,
                                 lse, &tm_k, &tm_v, &p);
  if (st != GQA_OK) return st;
  if (n_split > 1) p.tile_ctr = counters;
  return cuda_status(gqa::launch_decode_split(p, tm_k, tm_v, reinterpret_cast<cudaStream_t>(stream)));
}

int gqa_attn_decode_multi_default_splits(int B, int T_q, int H_q, int H_kv, int S_max, int d) {
  if (B < 1 || T_q < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0) return 1;
  const int n = gqa_attn_decode_default_splits(B, H_kv, S_max, -1);
  const long long groups = (T_q * (long long)(H_q / H_kv) + 15) / 16;
  if (groups <= 1) return n;
  // The tensor-core kernel: one CTA per SM, K/V read once per split.
  if (multi_uses_tc(T_q, H_q / H_kv, d)) return n;
  // Several row groups: keep every CTA of a split resident at once (two per
  // SM), so the groups' reads of the same K/V tiles meet in L2 (measured for
  // Llama3-70B at 32K: 19 / 12 / 9 splits best for 2 / 3 / 4 groups).
  const long long fit = 2LL * num_sms_current_device() / ((long long)B * H_kv * groups);
  return (int)std::max(1LL, std::min((long long)n, fit));
}

gqa_status gqa_attn_decode_multi(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* seq_lens, int B, int T_q, int S_max, int H_q,
                                 int H_kv, int d, float scale, int n_split, void* workspace,
                                 void* out, float* lse, gqa_stream_t stream) {
  if (T_q < 1 || T_q > 64 || T_q > S_max) return GQA_ERR_INVALID_ARG;
  if (H_kv < 1 || H_q % H_kv != 0) return GQA_ERR_INVALID_ARG;
  const bool tc = multi_uses_tc(T_q, H_q / H_kv, d);
  if (T_q * (H_q / H_kv) > (tc ? kMaxMultiRowsTc : kMaxMultiRows)) return GQA_ERR_UNSUPPORTED;
  if ((long long)B * T_q > 65535) return GQA_ERR_INVALID_ARG;
  CUtensorMap tm_k, tm_v;
  gqa::DecodeParams p;
  gqa_status st = prepare_decode(q, k_cache, v_cache, seq_lens, B, S_max, (long long)B * S_max,
                                 tc ? 128 : gqa::kDecodeTile, H_q, H_kv, d, scale, n_split,
                                 workspace, out, lse, &tm_k, &tm_v, &p);
  if (st != GQA_OK) return st;
  if (tc) {
    // All T_q * G rows of a KV head in one tile: Q as [B * T_q][H_q][d], one
    // box of G heads x T_q queries per d half; 128-key splits.
    CUtensorMap tm_q;
    const uint64_t qdims[3] = {(uint64_t)d, (uint64_t)H_q, (uint64_t)B * T_q};
    const uint64_t qstrides[2] = {(uint64_t)d * 2, (uint64_t)H_q * d * 2};
    const uint32_t qbox[3] = {64u, (uint32_t)(H_q / H_kv), (uint32_t)T_q};
    if ((st = encode_bf16(&tm_q, q, 3, qdims, qstrides, qbox, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        GQA_OK)
      return st;
    p.T_q = T_q;
    p.n_rg = 1;
    const long long per = ((long long)S_max + n_split - 1) / n_split;
    p.chunk = (int)((per + 127) / 128 * 128);
    p.ws_O = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                  gqa::decode_ws_O_offset(B * T_q, H_q, n_split))
                       : nullptr;
    return cuda_status(
        gqa::launch_decode_tc(p, tm_q, tm_k, tm_v, reinterpret_cast<cudaStream_t>(stream)));
  }
  p.T_q = T_q;
  p.n_rg = (T_q * p.G + 15) / 16;
  if ((long long)n_split * p.n_rg > 0x7fffffffLL) return GQA_ERR_INVALID_ARG;
  // the partials are laid out for B * T_q rows of H_q heads
  p.ws_O = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                gqa::decode_ws_O_offset(B * T_q, H_q, n_split))
                     : nullptr;
  return cuda_status(gqa::launch_decode_split(p, tm_k, tm_v, reinterpret_cast<cudaStream_t>(stream)));
}

int gqa_attn_decode_fused_splits(int B, int H_q, int H_kv, int d) {
  if (B < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || !head_dim_ok(d) || H_q / H_kv > 16)
    return 0;
  // The largest cluster (16, else 8) whose CTAs can be resident together,
  // probed once per device and head shape class.
  static int cache[64][3][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const int di = d == 32 ? 0 : d == 64 ? 1 : 2, gi = H_q / H_kv > 8 ? 1 : 0;
  if (dev >= 0 && dev < 64 && cache[dev][di][gi] != 0) return cache[dev][di][gi] > 0 ? cache[dev][di][gi] : 0;
  int found = -1;
  for (int c : {16, 8}) {
    gqa::DecodeParams p{};
    p.B = 1;
    p.H_kv = 1;
    p.G = H_q / H_kv;
    p.d = d;
    p.n_split = c;
    CUtensorMap dummy{};
    if (gqa::launch_decode_fused(p, dummy, dummy, true, nullptr) == cudaSuccess) {
      found = c;
      break;
    }
    cudaGetLastError();  // clear a failed probe
  }
  if (dev >= 0 && dev < 64) cache[dev][di][gi] = found;
  return found > 0 ? found : 0;
}

gqa_status gqa_attn_decode_fused(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* seq_lens, int B, int S_max, int H_q, int H_kv,
                                 int d, float scale, void* out, float* lse, gqa_stream_t stream) {
  if (B < 1 || H_q < 1 || H_kv < 1) return GQA_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return GQA_ERR_INVALID_ARG;
  const int c = gqa_attn_decode_fused_splits(B, H_q, H_kv, d);
  if (c == 0) return GQA_ERR_UNSUPPORTED;
  CUtensorMap tm_k, tm_v;
  gqa::DecodeParams p;
  gqa_status st = prepare_decode(q, k_cache, v_cache, seq_lens, B, S_max, (long long)B * S_max,
                                 gqa::kDecodeTile, H_q, H_kv, d, scale, c, nullptr, out, lse,
                                 &tm_k, &tm_v, &p, /*needs_workspace=*/false);
  if (st != GQA_OK) return st;
  return cuda_status(
      gqa::launch_decode_fused(p, tm_k, tm_v, false, reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_attn_decode_paged_multi(const void* q, const void* k_pool, const void* v_pool,
                                       const int32_t* block_table, const int32_t* seq_lens, int B,
                                       int T_q, int num_pages, int page_size, int max_blocks,
                                       int H_q, int H_kv, int d, float scale, int n_split,
                                       void* workspace, void* out, float* lse,
                                       gqa_stream_t stream) {
  if (T_q < 1 || T_q > 64) return GQA_ERR_INVALID_ARG;
  if (H_kv < 1 || H_q % H_kv != 0) return GQA_ERR_INVALID_ARG;
  const bool tc = multi_uses_tc(T_q, H_q / H_kv, d);
  if (T_q * (H_q / H_kv) > (tc ? kMaxMultiRowsTc : kMaxMultiRows)) return GQA_ERR_UNSUPPORTED;
  if ((long long)B * T_q > 65535) return GQA_ERR_INVALID_ARG;
  if (!block_table || !aligned(block_table, 4)) return GQA_ERR_INVALID_ARG;
  if (num_pages < 1 || max_blocks < 1 || page_size < 1) return GQA_ERR_INVALID_ARG;
  if (page_size < 16 || (page_size & (page_size - 1)) != 0) return GQA_ERR_UNSUPPORTED;
  const long long S_max = (long long)max_blocks * page_size;
  const long long rows = (long long)num_pages * page_size;
  if (S_max > 0x7fffffffLL || rows > 0x7ffffffeLL) return GQA_ERR_INVALID_ARG;
  if (tc) {
    // All T_q * G rows of a KV head in one tensor-core tile; each 128-key tile
    // arrives as boxes of min(page_size, 128) rows, one page each.
    CUtensorMap tm_k, tm_v, tm_q;
    gqa::DecodeParams p;
    gqa_status st = prepare_decode(q, k_pool, v_pool, seq_lens, B, (int)S_max, rows,
                                   page_size < 128 ? page_size : 128, H_q, H_kv, d, scale,
                                   n_split, workspace, out, lse, &tm_k, &tm_v, &p);
    if (st != GQA_OK) return st;
    const uint64_t qdims[3] = {(uint64_t)d, (uint64_t)H_q, (uint64_t)B * T_q};
    const uint64_t qstrides[2] = {(uint64_t)d * 2, (uint64_t)H_q * d * 2};
    const uint32_t qbox[3] = {64u, (uint32_t)(H_q / H_kv), (uint32_t)T_q};
    if ((st = encode_bf16(&tm_q, q, 3, qdims, qstrides, qbox, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        GQA_OK)
      return st;
    p.block_table = block_table;
    p.max_blocks = max_blocks;
    p.page_size = page_size;
    p.num_pages = num_pages;
    p.T_q = T_q;
    p.n_rg = 1;
    const long long per = (S_max + n_split - 1) / n_split;
    p.chunk = (int)((per + 127) / 128 * 128);
    p.ws_O = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                  gqa::decode_ws_O_offset(B * T_q, H_q, n_split))
                       : nullptr;
    return cuda_status(
        gqa::launch_decode_tc(p, tm_q, tm_k, tm_v, reinterpret_cast<cudaStream_t>(stream)));
  }
  if (n_split >= 1) {
    const int chunk = gqa_attn_decode_split_chunk((int)S_max, n_split);
    if (chunk / page_size + 2 > gqa::kMaxPagesPerCta) return GQA_ERR_UNSUPPORTED;
  }
  CUtensorMap tm_k, tm_v;
  gqa::DecodeParams p;
  gqa_status st = prepare_decode(q, k_pool, v_pool, seq_lens, B, (int)S_max, rows,
                                 page_size < gqa::kDecodeTile ? page_size : gqa::kDecodeTile, H_q,
                                 H_kv, d, scale, n_split, workspace, out, lse, &tm_k, &tm_v, &p);
  if (st != GQA_OK) return st;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.page_size = page_size;
  p.num_pages = num_pages;
  p.T_q = T_q;
  p.n_rg = (T_q * p.G + 15) / 16;
  p.ws_O = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                gqa::decode_ws_O_offset(B * T_q, H_q, n_split))
                     : nullptr;
  return cuda_status(gqa::launch_decode_paged(p, tm_k, tm_v, reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_attn_decode_paged(const void* q, const void* k_pool, const void* v_pool,
                                 const int32_t* block_table, const int32_t* seq_lens, int B,
                                 int num_pages, int page_size, int max_blocks, int H_q, int H_kv,
                                 int d, float scale, int n_split, void* workspace, void* out,
                                 float* lse, gqa_stream_t stream) {
  return gqa_attn_decode_paged_multi(q, k_pool, v_pool, block_table, seq_lens, B, 1, num_pages,
                                     page_size, max_blocks, H_q, H_kv, d, scale, n_split,
                                     workspace, out, lse, stream);
}

}  // extern "C"

namespace {

// E4M3 cache maps: codes viewed as [rows][H_kv][d] bytes (boxes of box_rows rows
// of one head, swizzled over d bytes) and the per-token scales as [outer][inner] fp32.
gqa_status prepare_fp8_maps(const void* k8, const void* v8, const float* k_scale,
                            const float* v_scale, long long rows, int box_rows, int H_kv, int d,
                            int sc_inner, int sc_outer, CUtensorMap* tm_k, CUtensorMap* tm_v,
                            CUtensorMap* tm_ks, CUtensorMap* tm_vs) {
  if (!k8 || !v8 || !k_scale || !v_scale) return GQA_ERR_INVALID_ARG;
  if (!aligned(k8, 16) || !aligned(v8, 16) || !aligned(k_scale, 16) || !aligned(v_scale, 16))
    return GQA_ERR_INVALID_ARG;
  if ((sc_inner * 4) % 16 != 0) return GQA_ERR_UNSUPPORTED;
  const uint64_t dims[3] = {(uint64_t)d, (uint64_t)H_kv, (uint64_t)rows};
  const uint64_t strides[2] = {(uint64_t)d, (uint64_t)H_kv * d};
  const uint32_t box[3] = {(uint32_t)d, 1u, (uint32_t)box_rows};
  // rows of d bytes, swizzled over all of them (the kernel reads 4-byte pieces
  // of eight different rows per instruction without bank conflicts)
  const CUtensorMapSwizzle swz = d == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : d == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                           : CU_TENSOR_MAP_SWIZZLE_32B;
  gqa_status st;
  if ((st = encode_map(tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, k8, 3, dims, strides, box, swz)) !=
      GQA_OK)
    return st;
  if ((st = encode_map(tm_v, CU_TENSOR_MAP_DATA_TYPE_UINT8, v8, 3, dims, strides, box, swz)) !=
      GQA_OK)
    return st;
  const uint64_t sdims[2] = {(uint64_t)sc_inner, (uint64_t)sc_outer};
  const uint64_t sstr[1] = {(uint64_t)sc_inner * 4};
  const uint32_t sbox[2] = {(uint32_t)box_rows, 1u};
  if ((st = encode_map(tm_ks, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, k_scale, 2, sdims, sstr, sbox,
                       CU_TENSOR_MAP_SWIZZLE_NONE)) != GQA_OK)
    return st;
  return encode_map(tm_vs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, v_scale, 2, sdims, sstr, sbox,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

extern "C" {

gqa_status gqa_attn_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale,
                               const int32_t* seq_lens, int B, int S_max, int H_q, int H_kv,
                               int d, float scale, int n_split, void* workspace, void* out,
                               float* lse, gqa_stream_t stream) {
  CUtensorMap tm_k, tm_v, tm_ks, tm_vs;
  gqa::DecodeParams p;
  // the bf16 maps encoded here are replaced below; this runs the shared checks
  gqa_status st = prepare_decode(q, k_cache, v_cache, seq_lens, B, S_max, (long long)B * S_max,
                                 gqa::kDecodeTile, H_q, H_kv, d, scale, n_split, workspace, out,
                                 lse, &tm_k, &tm_v, &p);
  if (st != GQA_OK) return st;
  if ((st = prepare_fp8_maps(k_cache, v_cache, k_scale, v_scale, (long long)B * S_max,
                             gqa::kDecodeTile, H_kv, d, S_max, B, &tm_k, &tm_v, &tm_ks,
                             &tm_vs)) != GQA_OK)
    return st;
  return cuda_status(
      gqa::launch_decode_fp8(p, tm_k, tm_v, tm_ks, tm_vs, reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_attn_decode_paged_fp8(const void* q, const void* k_pool, const void* v_pool,
                                     const float* k_scale, const float* v_scale,
                                     const int32_t* block_table, const int32_t* seq_lens, int B,
                                     int num_pages, int page_size, int max_blocks, int H_q,
                                     int H_kv, int d, float scale, int n_split, void* workspace,
                                     void* out, float* lse, gqa_stream_t stream) {
  if (!block_table || !aligned(block_table, 4)) return GQA_ERR_INVALID_ARG;
  if (num_pages < 1 || max_blocks < 1 || page_size < 1) return GQA_ERR_INVALID_ARG;
  if (page_size < 16 || (page_size & (page_size - 1)) != 0) return GQA_ERR_UNSUPPORTED;
  const long long S_max = (long long)max_blocks * page_size;
  const long long rows = (long long)num_pages * page_size;
  if (S_max > 0x7fffffffLL || rows > 0x7ffffffeLL) return GQA_ERR_INVALID_ARG;
  if (n_split >= 1) {
    const int chunk = gqa_attn_decode_split_chunk((int)S_max, n_split);
    if (chunk / page_size + 2 > gqa::kMaxPagesPerCta) return GQA_ERR_UNSUPPORTED;
  }
  const int h = page_size < gqa::kDecodeTile ? page_size : gqa::kDecodeTile;
  CUtensorMap tm_k, tm_v, tm_ks, tm_vs;
  gqa::DecodeParams p;
  gqa_status st = prepare_decode(q, k_pool, v_pool, seq_lens, B, (int)S_max, rows, h, H_q, H_kv,
                                 d, scale, n_split, workspace, out, lse, &tm_k, &tm_v, &p);
  if (st != GQA_OK) return st;
  if ((st = prepare_fp8_maps(k_pool, v_pool, k_scale, v_scale, rows, h, H_kv, d, page_size,
                             num_pages, &tm_k, &tm_v, &tm_ks, &tm_vs)) != GQA_OK)
    return st;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.page_size = page_size;
  p.num_pages = num_pages;
  return cuda_status(
      gqa::launch_decode_fp8(p, tm_k, tm_v, tm_ks, tm_vs, reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_attn_decode_combine(const void* workspace, int B, int H_q, int d, int n_split,
                                   void* out, float* lse, gqa_stream_t stream) {
  if (!workspace || !out || !lse) return GQA_ERR_INVALID_ARG;
  if (B < 1 || H_q < 1 || n_split < 1 || B > 65535 || H_q > 65535) return GQA_ERR_INVALID_ARG;
  if (!head_dim_ok(d)) return GQA_ERR_UNSUPPORTED;
  if (!aligned(workspace, 256) || !aligned(out, 16) || !aligned(lse, 4)) return GQA_ERR_INVALID_ARG;
  unsigned* err = nullptr;
  const gqa_status st = error_word(&err);
  if (st != GQA_OK) return st;
  gqa::CombineParams p;
  p.ws_ml = static_cast<const float2*>(workspace);
  p.ws_O = reinterpret_cast<const float*>(static_cast<const char*>(workspace) +
                                          gqa::decode_ws_O_offset(B, H_q, n_split));
  p.B = B;
  p.H_q = H_q;
  p.d = d;
  p.n_split = n_split;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.err = err;
  return cuda_status(gqa::launch_decode_combine(p, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Shared checks and launch of the causal prefill kernel: S query rows per
// sequence against S_kv key rows (chunk: the queries end each sequence).
gqa_status run_prefill(bool chunk, const void* q, const void* k, const void* v,
                       const int32_t* seq_lens, int B, int S, int S_kv, int H_q, int H_kv, int d,
                       float scale, int window, int n_part, void* workspace, void* out, float* lse,
                       gqa_stream_t stream) {
  if (!q || !k || !v || !out || !lse) return GQA_ERR_INVALID_ARG;
  if (n_part < 1 || n_part > 8 || (n_part > 1 && (!chunk || !workspace))) return GQA_ERR_INVALID_ARG;
  if (workspace && !aligned(workspace, 256)) return GQA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || S_kv < S || H_q < 1 || H_kv < 1 || H_q % H_kv != 0)
    return GQA_ERR_INVALID_ARG;
  if (B > 65535 || H_q > 65535 || !std::isfinite(scale) || !(scale > 0.f))
    return GQA_ERR_INVALID_ARG;
  if ((long long)B * S * H_q > 0x7fffffffLL || (long long)B * S_kv > 0x7fffffffLL)
    return GQA_ERR_INVALID_ARG;
  if (!head_dim_ok(d)) return GQA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || (seq_lens && !aligned(seq_lens, 4)))
    return GQA_ERR_INVALID_ARG;
  unsigned* err = nullptr;
  gqa_status st = error_word(&err);
  if (st != GQA_OK) return st;

  // Q viewed as [B][S][H_q][d] with boxes of 128 rows of one head, 64 elements
  // wide (two boxes per 128-wide row), 128-byte swizzle; K and V likewise.  For
  // d = 32 the 64-element box is wider than the tensor: TMA fills elements
  // 32..63 with zeros, the padding the kernel's 64-wide tiles expect.
  const uint64_t dq[4] = {(uint64_t)d, (uint64_t)H_q, (uint64_t)S, (uint64_t)B};
  const uint64_t sq[3] = {(uint64_t)d * 2, (uint64_t)H_q * d * 2, (uint64_t)S * H_q * d * 2};
  const uint64_t dk[4] = {(uint64_t)d, (uint64_t)H_kv, (uint64_t)S_kv, (uint64_t)B};
  const uint64_t sk[3] = {(uint64_t)d * 2, (uint64_t)H_kv * d * 2, (uint64_t)S_kv * H_kv * d * 2};
  const uint32_t box[4] = {64u, 1u, 128u, 1u};
  CUtensorMap tm_q, tm_k, tm_v;
  if ((st = encode_bf16(&tm_q, q, 4, dq, sq, box, CU_TENSOR_MAP_SWIZZLE_128B)) != GQA_OK) return st;
  if ((st = encode_bf16(&tm_k, k, 4, dk, sk, box, CU_TENSOR_MAP_SWIZZLE_128B)) != GQA_OK) return st;
  if ((st = encode_bf16(&tm_v, v, 4, dk, sk, box, CU_TENSOR_MAP_SWIZZLE_128B)) != GQA_OK) return st;

  gqa::PrefillParams p;
  p.B = B;
  p.S = S;
  p.S_kv = S_kv;
  p.seq_lens = seq_lens;
  p.window = window < 0 ? -1 : window;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.G = H_q / H_kv;
  p.d = d;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.err = err;
  p.wait_ns = g_wait_ns.load();
  p.n_part = n_part;
  p.ws_ml = n_part > 1 ? static_cast<float2*>(workspace) : nullptr;
  p.ws_O = n_part > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                 gqa::prefill_ws_O_offset((size_t)B * S * H_q, n_part))
                      : nullptr;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int sms = num_sms_current_device();
  if (!chunk) return cuda_status(gqa::launch_prefill_causal(p, tm_q, tm_k, tm_v, sms, s));
  st = cuda_status(gqa::launch_prefill_chunk(p, tm_q, tm_k, tm_v, sms, s));
  if (st != GQA_OK || n_part == 1) return st;
  return cuda_status(gqa::launch_prefill_merge(p, s));
}

}  // namespace

extern "C" {

gqa_status gqa_attn_prefill_causal(const void* q, const void* k, const void* v, int B, int S,
                                   int H_q, int H_kv, int d, float scale, void* out, float* lse,
                                   gqa_stream_t stream) {
  return run_prefill(false, q, k, v, nullptr, B, S, S, H_q, H_kv, d, scale, -1, 1, nullptr, out, lse,
                     stream);
}

gqa_status gqa_attn_prefill_chunk(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* seq_lens, int B, int T_q, int S_max, int H_q,
                                  int H_kv, int d, float scale, int window, void* out, float* lse,
                                  gqa_stream_t stream) {
  return run_prefill(true, q, k_cache, v_cache, seq_lens, B, T_q, S_max, H_q, H_kv, d, scale,
                     window, 1, nullptr, out, lse, stream);
}

size_t gqa_attn_prefill_chunk_workspace_bytes(int B, int T_q, int H_q, int d, int n_part) {
  if (B < 1 || T_q < 1 || H_q < 1 || d < 1 || n_part <= 1) return 0;
  const size_t rows = (size_t)B * T_q * H_q;
  return gqa::prefill_ws_O_offset(rows, n_part) + rows * n_part * d * sizeof(float);
}

int gqa_attn_prefill_chunk_default_parts(int B, int T_q, int S_max, int H_q, int H_kv) {
  if (B < 1 || T_q < 1 || S_max < T_q || H_q < 1 || H_kv < 1 || H_q % H_kv != 0) return 1;
  // Split only long items (>= 16 key tiles if the chunk ends the cache), and
  // only when it evens out the last round of the persistent grid: the part
  // count P in 1..4 maximising x / ceil(x), x = items * P / SMs, must beat
  // P = 1 by at least 5% (a split costs a partial write, read and merge).
  if (S_max / 128 < 16) return 1;
  const long long items = (long long)((T_q + 127) / 128) * B * H_kv * ((H_q / H_kv + 1) / 2);
  const int sms = num_sms_current_device();
  auto eff = [&](int P) {
    const double x = (double)items * P / sms;
    return x / std::ceil(x);
  };
  int best = 1;
  for (int P = 2; P <= 4; ++P)
    if (eff(P) > eff(best) + 1e-9) best = P;
  return eff(best) >= eff(1) + 0.05 ? best : 1;
}

gqa_status gqa_attn_prefill_chunk_split(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* seq_lens, int B, int T_q, int S_max,
                                        int H_q, int H_kv, int d, float scale, int window,
                                        int n_part, void* workspace, void* out, float* lse,
                                        gqa_stream_t stream) {
  return run_prefill(true, q, k_cache, v_cache, seq_lens, B, T_q, S_max, H_q, H_kv, d, scale,
                     window, n_part, workspace, out, lse, stream);
}

gqa_status gqa_last_device_error(gqa_stream_t stream) {
  unsigned* err = nullptr;
  gqa_status st = error_word(&err);
  if (st != GQA_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GQA_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (word) {
    const unsigned zero = 0;
    if (cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return GQA_ERR_CUDA;
  }
  if (word & gqa::kErrBounds) return GQA_ERR_CUDA;  // bounds-checking builds: an internal fault
  if (word & gqa::kErrTimeout) return GQA_ERR_TIMEOUT;
  if (word & (gqa::kErrBadSeqLen | gqa::kErrBadPage)) return GQA_ERR_INVALID_ARG;
  return GQA_OK;
}

uint64_t gqa_set_wait_limit_ns(uint64_t limit_ns) {
  if (limit_ns < 1000) limit_ns = 1000;
  return g_wait_ns.exchange(limit_ns);
}

gqa_status gqa_selftest_wait_timeout(uint64_t limit_ns, gqa_stream_t stream) {
  unsigned* err = nullptr;
  gqa_status st = error_word(&err);
  if (st != GQA_OK) return st;
  if (limit_ns < 1000) limit_ns = 1000;
  return cuda_status(gqa::launch_wait_selftest(err, limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
