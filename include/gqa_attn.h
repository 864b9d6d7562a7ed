/*
 * gqa_attn.h -- C ABI of libgqa_attn.so: grouped-query fused attention forward
 * on one NVIDIA GB300 (sm_103a).
 *
 * The operation ("Attention Kernel 계보", p.2 §1 and p.15 §2): for query head h
 * of a group of G = H_q / H_kv query heads sharing KV head kv = floor(h / G),
 *     O_h = softmax(tau * q_h K_kv^T) V_kv,   LSE_h = ln sum_j exp(tau * q_h . k_j)
 * over the visible keys j, computed with the streaming (m, l, O) softmax of p.3
 * §5 so that the score matrix never reaches memory.  LSE is in natural-log units
 * of the scaled scores (p.3 §9).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers marked "device" are CUDA device pointers; the caller owns every
 *   buffer and keeps it alive until the stream work completes.  Tensors are
 *   dense, row-major, innermost index last, in the layouts given per call.
 *   bf16 = IEEE bfloat16 (2 bytes), fp32 = IEEE binary32.
 * - Every call is asynchronous on `stream` (NULL = legacy default stream) and
 *   never synchronises, except gqa_last_device_error().  The library allocates
 *   no memory per call; it keeps one 4-byte device error word per device,
 *   created on first use.
 * - Arguments that the host can check are checked before anything is launched;
 *   a failed check returns GQA_ERR_INVALID_ARG or GQA_ERR_UNSUPPORTED and leaves
 *   every output untouched.  A launch failure returns GQA_ERR_CUDA.
 * - Faults found on the device (a seq_lens entry out of range, a pipeline wait
 *   that exceeded its time limit) set bits in the device error word; the
 *   affected outputs are written as NaN and the call still returns GQA_OK.
 *   gqa_last_device_error() reports and clears them.
 * - Device pointers must be 16-byte aligned (tensor-memory-access copies).
 * - Thread safety: calls on different streams may run concurrently.  Shared
 *   state: the per-device error word, per-device values computed once and
 *   then only read (SM count, kernel attributes, cluster support), and the
 *   scratch array of gqa_attn_decode_noalloc (see there).
 *
 * Which call for which workload (measured on GB300, Llama3-70B heads, 32K cache)
 * -------------------------------------------------------------------------
 * - One new token per sequence, contiguous cache: gqa_attn_decode with
 *   gqa_attn_decode_default_splits, then gqa_attn_decode_combine (23.0-23.3 us
 *   per step; the split kernel streams K/V at 98-99% of the measured HBM rate).
 *   Several sequences of very different lengths: gqa_attn_decode_balanced
 *   (+ combine), whose splits share each sequence's last quarter of tiles.
 * - The same over a paged cache: gqa_attn_decode_paged (+ combine).
 * - An E4M3 cache with per-token scales: gqa_attn_decode_fp8 /
 *   gqa_attn_decode_paged_fp8 (+ combine) with 3x the default split count
 *   (15.8-16.3 us per step at 32K).
 * - A few new tokens per sequence (speculative verification, T_q <= 64):
 *   gqa_attn_decode_multi / gqa_attn_decode_paged_multi (+ combine with B * T_q
 *   rows); above 16 query rows per KV head at d = 128 they run on the tensor
 *   cores (T_q = 8: 25.5 us, against 397 us through the chunked prefill).
 * - A prompt: gqa_attn_prefill_causal (tensor cores, 86-87% of the measured
 *   dense bf16 rate at d = 128; d = 64 and 32 at about half and a quarter).
 * - A chunk of queries ending a cached sequence, optionally with a sliding
 *   window: gqa_attn_prefill_chunk, or gqa_attn_prefill_chunk_split for long
 *   keys and few query tiles.
 * - One launch without a workspace (small decodes): gqa_attn_decode_fused;
 *   without any caller buffer: gqa_attn_decode_noalloc.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* gqa_stream_t;

typedef enum gqa_status {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, bad seq_len on device */
  GQA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. head dim) */
  GQA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  GQA_ERR_TIMEOUT = 4      /* a device pipeline wait exceeded its time limit */
} gqa_status;

/* Static, human-readable name of a status code.  Never NULL. */
const char* gqa_status_str(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int gqa_version(void);

/* ------------------------------------------------------------------------
 * Split-KV decode ("Attention Kernel 계보", p.18 §4; ADR-0060 §5.1-§5.3)
 * ------------------------------------------------------------------------
 * One query token per sequence (T_q = 1) attends keys [0, seq_lens[b]) of a
 * padded cache.  The keys of each sequence are cut into n_split contiguous
 * splits of `chunk` tokens, chunk = gqa_attn_decode_split_chunk(S_max, n_split):
 * split s covers [s*chunk, min((s+1)*chunk, seq_lens[b])) and may be empty.
 *
 * Workspace (fp32, device, gqa_attn_decode_workspace_bytes() bytes, caller-
 * owned) holds one partial per (b, h, s):
 *   at byte 0:                 float2 ml[B][H_q][n_split] = (m_s, l_s)
 *   at byte round_up(B*H_q*n_split*8, 256):  float O[B][H_q][n_split][d]
 * with, over the keys j of split s and scaled scores x_j = tau * q_h . k_j,
 *   m_s = max_j x_j,  l_s = sum_j exp(x_j - m_s),  O_s = sum_j exp(x_j - m_s) v_j
 * (unnormalised; "Attention Kernel 계보", p.4 §2, §8).  An empty split is the
 * merge identity: m_s = -inf, l_s = 0, and its O_s is not written or read.
 */

/* Tokens per split for a cache of S_max positions cut n_split ways: ceil(S_max/
 * n_split) rounded up to a multiple of 64.  Returns 0 if an argument is < 1. */
int gqa_attn_decode_split_chunk(int S_max, int n_split);

/* Workspace bytes for gqa_attn_decode with n_split > 1; 0 if n_split == 1 or an
 * argument is < 1. */
size_t gqa_attn_decode_workspace_bytes(int B, int H_q, int d, int n_split);

/* Deterministic split count for a (B, H_kv, S_max) decode on CUDA device
 * `device` (its SM count; device < 0: the current device): 1 for S_max <= 1024
 * (one CTA per sequence and KV head; no combine needed), otherwise about one
 * CTA per SM, with splits of 128 to 8192 tokens.  The head dimension does not
 * enter.  Returns >= 1 (1 for invalid input or a device that cannot be
 * queried). */
int gqa_attn_decode_default_splits(int B, int H_kv, int S_max, int device);

/* Stage 1 of split-KV decode.
 *   q         device bf16 [B, H_q, d]           query (post-RoPE), read only
 *   k_cache   device bf16 [B, S_max, H_kv, d]   keys, read only
 *   v_cache   device bf16 [B, S_max, H_kv, d]   values, read only
 *   seq_lens  device int32 [B], 1 <= seq_lens[b] <= S_max (checked on device:
 *             a batch with a bad length gets NaN outputs and sets the
 *             GQA_ERR_INVALID_ARG bit of the error word)
 *   H_q % H_kv == 0, G = H_q / H_kv <= 16, d in {32, 64, 128}, scale finite > 0
 *   n_split   >= 1.  n_split == 1: writes out and lse directly, workspace unused
 *             (may be NULL).  n_split > 1: writes the workspace only; call
 *             gqa_attn_decode_combine() next on the same stream.
 *   out       device bf16 [B, H_q, d]     O = sum_j softmax_j v_j
 *   lse       device fp32 [B, H_q]        LSE = m + ln l
 * Keys past seq_lens[b] are never used: their cache rows may hold anything.
 * The kernel is launched as a programmatic dependent of the preceding kernel in
 * the stream: it may be scheduled early and then only prefetches the first K/V
 * tiles of each split into L2 (no data reaches the kernel); it reads and
 * writes nothing before that kernel has completed. */
gqa_status gqa_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* seq_lens, int B, int S_max, int H_q, int H_kv, int d,
                           float scale, int n_split, void* workspace, void* out, float* lse,
                           gqa_stream_t stream);

/* Stage 2 of split-KV decode: merges the n_split partials of each (b, h) with
 * the associative merge ("Attention Kernel 계보", p.4 §3-§9; p.18 §4 stage 2):
 *   M = max_s m_s,  L = sum_s e^(m_s - M) l_s,  O = sum_s e^(m_s - M) O_s / L,
 *   out = O (bf16), lse = M + ln L (fp32).
 * Splits with m_s = -inf contribute nothing.  If every split of a row is
 * empty the row is written as NaN.  Layouts as for gqa_attn_decode; the
 * workspace may also be filled by the caller in the documented format. */
gqa_status gqa_attn_decode_combine(const void* workspace, int B, int H_q, int d, int n_split,
                                   void* out, float* lse, gqa_stream_t stream);

/* Stage 1 of split-KV decode over a paged KV cache ("Attention Kernel 계보",
 * p.17 §2-§4 and p.18 §1-§5).  The cache is two pools of fixed-size pages,
 *   k_pool, v_pool  device bf16 [num_pages, page_size, H_kv, d]
 * and logical token t of sequence b is row t % page_size of page
 *   block_table[b * max_blocks + t / page_size]      (device int32 [B, max_blocks]).
 * page_size is a power of two >= 16; 1 <= seq_lens[b] <= max_blocks * page_size.
 * Splits, workspace, outputs and the follow-up gqa_attn_decode_combine() are
 * those of gqa_attn_decode() with S_max = max_blocks * page_size.  Pages may be
 * shared between sequences (read-only).  Only the table entries of tokens
 * < seq_lens[b] are read; an entry outside [0, num_pages) is reported through
 * the error word (GQA_ERR_INVALID_ARG) and makes that split's outputs NaN.
 * GQA_ERR_UNSUPPORTED if one split would span more than 510 pages (raise
 * n_split).  For pages shorter than 64 tokens each tile takes several small
 * copies; twice gqa_attn_decode_default_splits() (two CTAs per SM) measured
 * best there. */
gqa_status gqa_attn_decode_paged(const void* q, const void* k_pool, const void* v_pool,
                                 const int32_t* block_table, const int32_t* seq_lens, int B,
                                 int num_pages, int page_size, int max_blocks, int H_q, int H_kv,
                                 int d, float scale, int n_split, void* workspace, void* out,
                                 float* lse, gqa_stream_t stream);

/* Stage 1 of split-KV decode over an FP8 KV cache ("Attention Kernel 계보",
 * p.17 §7): keys and values are E4M3 codes (1 sign, 4 exponent bits with bias
 * 7, 3 mantissa bits; 0x7f/0xff are NaN) with one fp32 scale per token shared
 * by all KV heads; the key used is e4m3(k_cache[...]) * k_scale[b, t] (values
 * likewise).  The dequantisation is fused into the sweep: the codes are
 * converted exactly to f16 on chip, the key scale multiplies the score column
 * and the value scale multiplies p before the P V product.  Q is converted to
 * f16 for the Q K^T product, so |q| must stay below 65504.
 *   k_cache, v_cache  device uint8 [B, S_max, H_kv, d] (16-byte aligned)
 *   k_scale, v_scale  device fp32 [B, S_max] (16-byte aligned); S_max % 4 == 0
 *                     (else GQA_ERR_UNSUPPORTED)
 * Every other argument, the workspace and the follow-up combine are those of
 * gqa_attn_decode().  Codes and scales past seq_lens[b] are never used.  The
 * on-chip conversion favours several CTAs per SM: three times
 * gqa_attn_decode_default_splits() measured best (three CTAs per SM). */
gqa_status gqa_attn_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale,
                               const int32_t* seq_lens, int B, int S_max, int H_q, int H_kv,
                               int d, float scale, int n_split, void* workspace, void* out,
                               float* lse, gqa_stream_t stream);

/* The FP8 cache of gqa_attn_decode_fp8() in pages, as in gqa_attn_decode_paged():
 *   k_pool, v_pool    device uint8 [num_pages, page_size, H_kv, d]
 *   k_scale, v_scale  device fp32 [num_pages, page_size]: the scales of a page's
 *                     tokens stored with the page (its B_p per-token scalars)
 * and block_table, seq_lens, page_size, max_blocks as for the paged decode. */
gqa_status gqa_attn_decode_paged_fp8(const void* q, const void* k_pool, const void* v_pool,
                                     const float* k_scale, const float* v_scale,
                                     const int32_t* block_table, const int32_t* seq_lens, int B,
                                     int num_pages, int page_size, int max_blocks, int H_q,
                                     int H_kv, int d, float scale, int n_split, void* workspace,
                                     void* out, float* lse, gqa_stream_t stream);

/* Split-KV decode with balanced splits ("Attention Kernel 계보", p.18 §4: the
 * stage-1 / stage-2 split of the keys; the merge of p.4 §3-§9 does not depend
 * on which keys a partial holds).  Fixed splits end at different times: the
 * CTAs share the GPU's memory bandwidth unevenly, and the step waits for the
 * slowest.  Here split s first streams its own share, 64-token tiles
 * s*n_s .. s*n_s + n_s - 1 of its (sequence, KV head) with n_s =
 * floor(3 * ceil(seq_lens[b] / 64) / (4 * n_split)); the remaining tiles (about a
 * quarter) are then claimed one at a time by whichever split CTA of that
 * (sequence, KV head) has room for the next tile.  A partial therefore holds
 * a share of contiguous keys plus claimed tiles anywhere in the sequence.
 *   counters  device int32 [B, H_kv, 2], gqa_attn_decode_counter_bytes()
 *             bytes, 4-byte aligned, caller-owned.  All zero before the first
 *             call; every call returns them to zero by the time its kernel
 *             completes (also when a seq_lens entry is out of range or a wait
 *             timed out), so they can serve the next call as they are.  Calls
 *             that share one counter array must not overlap on the GPU.
 *             NULL or misaligned with n_split > 1: GQA_ERR_INVALID_ARG.
 * Every other argument, the workspace layout (one partial per split) and the
 * follow-up gqa_attn_decode_combine() are those of gqa_attn_decode().  The
 * result is that of gqa_attn_decode() up to rounding; since the claims depend
 * on timing, two calls on the same inputs may differ in the last bits.
 * n_split == 1 is exactly gqa_attn_decode() (counters unused, may be NULL).
 * Measured on GB300 (split + combine, Llama3-70B heads): the ragged batch of 8
 * sequences of 1K-128K tokens at 16 splits runs in 278.8 us against 283.1 us
 * with fixed splits, 2 sequences of 128K tokens in 150.9 against 156.2 us; the
 * single 32K sequence at 19 splits gains nothing (23.74 against 23.82 us), nor
 * do batches of 8K-32K sequences, so gqa_attn_decode, which is deterministic,
 * stays the choice there. */
size_t gqa_attn_decode_counter_bytes(int B, int H_kv);
gqa_status gqa_attn_decode_balanced(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* seq_lens, int B, int S_max, int H_q, int H_kv,
                                    int d, float scale, int n_split, void* workspace,
                                    int32_t* counters, void* out, float* lse,
                                    gqa_stream_t stream);

/* Split-KV decode that allocates nothing, for callers that cannot call
 * cudaMalloc when they decode: code running inside a custom allocator's
 * critical section (a nested allocation there would deadlock or recurse), or
 * a serving process whose device memory pool is fixed up front and may not
 * grow.  The pages have no counterpart of this entry point; it is a property
 * of this library's interface.
 *
 * Same arguments, layouts, checks and results as gqa_attn_decode() with the
 * same n_split followed by gqa_attn_decode_combine(), except that the split
 * partials live in a 16 MiB scratch array inside this library's device image
 * (present on every GPU that loads the library, until the process exits)
 * instead of a caller workspace.  The caller still passes q, the caches,
 * seq_lens, out and lse.
 *   - If gqa_attn_decode_workspace_bytes(B, H_q, d, n_split) exceeds 16 MiB
 *     (16777216 bytes) the call returns GQA_ERR_INVALID_ARG before any launch.
 *   - No cudaMalloc, cudaFree or other allocating call is made.  The first
 *     call with n_split > 1 on a device looks up the scratch array's device
 *     address (cudaGetSymbolAddress) with that device current and keeps it;
 *     make that first call before any stream capture.  The kept address is
 *     not valid after cudaDeviceReset() on that device: do not call this
 *     entry point on a device that was reset after its first call.
 *   - Devices with ordinal 64 or above return GQA_ERR_UNSUPPORTED (the
 *     library keeps one address per device for ordinals 0..63).
 *   - Every call shares the one array per device and it keeps the previous
 *     call's contents.  Nothing in it needs to start at zero: each call writes
 *     every partial that its combine reads.  Calls whose kernels overlap on the
 *     GPU (other streams, other host threads) race on the array: order them.
 *   - n_split == 1 uses no scratch and behaves exactly like gqa_attn_decode. */
gqa_status gqa_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* seq_lens, int B, int S_max, int H_q, int H_kv,
                                   int d, float scale, int n_split, void* out, float* lse,
                                   gqa_stream_t stream);

/* Diagnostics of a library built with -DGQA_TRACE=1 (the pages have no
 * counterpart; every other build returns GQA_ERR_UNSUPPORTED from both calls
 * and records nothing).  The split-KV decode kernel (gqa_attn_decode,
 * _paged, _fp8, _multi on the mma.sync rows) then keeps, for the first 4096
 * CTAs of its last launch (linear block index x + gridDim.x * (y + gridDim.y * z)),
 * one record of 64 64-bit words: 0-4 globaltimer stamps in ns (CTA entry,
 * release of the dependency wait, tile loop start, tile loop end, epilogue
 * end), 5 the SM, 6 the split, 7 the CTA's tiles; from word 8, six words per
 * consumer warp w (8 + 6w ..): clock64 cycles waiting for tiles, in Q K^T, in
 * the softmax update, in P V and in the whole loop, and the tiles the warp
 * handled; words 56-58: the epilogue's cycles on thread 0 waiting for the
 * other consumer warps, writing the warp partials to shared memory, and
 * merging them and storing the result; words 59-61: the prologue's cycles on
 * thread 0 after the dependency wait reading the sequence length, checking it
 * (the barriers are set up before the wait), and loading the query fragments.  CTAs that return before their tile
 * loop (empty splits, bad lengths) write no record.
 * gqa_trace_clear zeroes every record (synchronous); gqa_trace_read copies the
 * first `bytes` bytes (at most 4096 * 64 * 8) into `host` after the stream has
 * been synchronised by the caller.  GQA_ERR_INVALID_ARG for a null `host` or
 * too many bytes. */
gqa_status gqa_trace_clear(void);
gqa_status gqa_trace_read(void* host, size_t bytes);

/* Trace build only: clock64 stamps (SM cycles) of the causal prefill's pipeline
 * (gqa_attn_prefill_causal and the chunk kernels), for the first work item of
 * CTAs 0..7 of the last launch and that item's first 64 key tiles: records of
 * 16 64-bit words laid out [CTA 0..7][head X 0..1 of the pair][tile j 0..63].
 * Words 0-3: softmax warp of tensor-memory quarter q saw S_X(j) ready; 4-7:
 * quarter q released P_X(j); 8, 9, 10: quarter 0 had S in registers, the row
 * maximum, and the exponentials summed; 11, 12: the MMA warp started and
 * passed its wait for P_X(j); 13: it had issued O_X += P_X(j) V_j; 14: it had
 * issued and committed S_X(j + 1) (absent on the item's last tile); 15 (head A's
 * records only): it started waiting for V_j.  Unwritten words stay 0 after
 * gqa_trace_clear, which zeroes these records too.  GQA_ERR_INVALID_ARG for a
 * null `host` or more than 8 * 2 * 64 * 16 * 8 bytes. */
gqa_status gqa_trace_prefill_read(void* host, size_t bytes);

/* Trace build only: the issue rate of one tcgen05.mma form (M = 128, K = 16,
 * bf16 in, fp32 accumulate).  One CTA per SM issues `iters` rounds of
 * back-to-back instructions on zero operands from one converged warp; the
 * median over SMs of SM clock cycles per instruction is written to
 * *cycles_per_instruction (host memory).  Forms: 0 A and B in shared memory
 * (SS), N = 128; 1 A in tensor memory (TS), N = 128; 2 SS, N = 256; 3 SS,
 * N = 64; 4 TS, N = 128 with B MN-major; 5 the causal prefill's per-head step
 * (8 SS then 8 TS, N = 128, head and ring slot chosen at run time).  Nominal:
 * 32 cycles at N = 64, 64 at N = 128, 128 at N = 256 (8192 FLOP per clock per
 * SM).  Synchronous; uses the whole device.  GQA_ERR_INVALID_ARG for a null
 * pointer, a form outside 0..5 or iters outside 1..65536; GQA_ERR_TIMEOUT if
 * the final commit did not land within 2 s. */
gqa_status gqa_trace_mma_rate(int form, int iters, double* cycles_per_instruction);

/* ------------------------------------------------------------------------
 * Causal prefill ("Attention Kernel 계보", p.9 §4 and p.13 §1-§6)
 * ------------------------------------------------------------------------
 * S_q = S_kv = S; query row i sees keys j <= i.  Key tiles entirely above the
 * diagonal are never loaded; only diagonal tiles are masked.
 *   q     device bf16 [B, S, H_q, d]     read only
 *   k, v  device bf16 [B, S, H_kv, d]    read only
 *   H_q % H_kv == 0, d in {32, 64, 128}, S >= 1, B >= 1, scale finite > 0
 *   out   device bf16 [B, S, H_q, d]
 *   lse   device fp32 [B, H_q, S]
 * GQA_ERR_UNSUPPORTED for any other d.  d = 32 runs on the d = 64 tiles with
 * the unused columns zero (the same result, at the d = 64 cost). */
gqa_status gqa_attn_prefill_causal(const void* q, const void* k, const void* v, int B, int S,
                                   int H_q, int H_kv, int d, float scale, void* out, float* lse,
                                   gqa_stream_t stream);

/* Chunked prefill / multi-token decode with an optional sliding window
 * (ADR-0060 §0.5.3 q_block_meta {q_start, T_q} and §5.4; "Attention Kernel
 * 계보", p.13 §1 and §7).  The T_q queries of sequence b are its last T_q tokens:
 * with L_b = seq_lens[b] (the cache already holds their keys and values),
 * query row i sits at position a = L_b - T_q + i and sees keys j with
 * a - window <= j <= a (no lower bound when window < 0).  Key tiles wholly
 * outside every row's range are never loaded; tiles that cross a range edge
 * are masked by select.
 *   q         device bf16 [B, T_q, H_q, d]
 *   k_cache,
 *   v_cache   device bf16 [B, S_max, H_kv, d]; rows >= L_b are not read
 *   seq_lens  device int32 [B] with T_q <= L_b <= S_max, or NULL (every L_b =
 *             S_max).  A bad L_b is caught on the device: that sequence's
 *             rows are NaN and the GQA_ERR_INVALID_ARG error bit is set.
 *   H_q % H_kv == 0, d in {32, 64, 128}, 1 <= T_q <= S_max, scale finite > 0
 *   out       device bf16 [B, T_q, H_q, d]
 *   lse       device fp32 [B, H_q, T_q]
 * With seq_lens == NULL, T_q == S_max and window < 0 this is exactly
 * gqa_attn_prefill_causal(); window >= 0 with seq_lens == NULL and T_q ==
 * S_max is a sliding-window causal prefill. */
gqa_status gqa_attn_prefill_chunk(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* seq_lens, int B, int T_q, int S_max, int H_q,
                                  int H_kv, int d, float scale, int window, void* out, float* lse,
                                  gqa_stream_t stream);

/* Bytes of workspace gqa_attn_prefill_chunk_split needs: per (b, query row,
 * head) and part, the part's (m, l) pair (fp32) and its unnormalised O
 * (d fp32), the O partials at a 256-byte-aligned offset.  0 when n_part <= 1. */
size_t gqa_attn_prefill_chunk_workspace_bytes(int B, int T_q, int H_q, int d, int n_part);

/* A part count for gqa_attn_prefill_chunk_split on the current device: 1 (no
 * split) unless the work items are long (S_max >= 16 * 128) and splitting them
 * evens out the last round of the persistent grid; at most 4. */
int gqa_attn_prefill_chunk_default_parts(int B, int T_q, int S_max, int H_q, int H_kv);

/* gqa_attn_prefill_chunk with each work item's key tiles split into n_part
 * (1..8) contiguous parts that run as separate work units, so that few long
 * items still spread evenly over the SMs.  Each part keeps its unnormalised
 * (m, l, O) in `workspace` (device, 256-byte aligned, at least
 * gqa_attn_prefill_chunk_workspace_bytes(B, T_q, H_q, d, n_part) bytes); a
 * second launch merges the parts with the log-sum-exp merge ("Attention
 * Kernel 계보" p.4) into out and lse.  Same arguments, layouts, outputs and
 * errors as gqa_attn_prefill_chunk; n_part = 1 is exactly that call (workspace
 * unused).  GQA_ERR_INVALID_ARG for n_part outside 1..8 or a missing or
 * misaligned workspace with n_part > 1.  The result differs from the unsplit
 * one only by rounding. */
gqa_status gqa_attn_prefill_chunk_split(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* seq_lens, int B, int T_q, int S_max,
                                        int H_q, int H_kv, int d, float scale, int window,
                                        int n_part, void* workspace, void* out, float* lse,
                                        gqa_stream_t stream);

/* ------------------------------------------------------------------------
 * Multi-token decode
 * ------------------------------------------------------------------------ */

/* Decode of the last T_q positions of each sequence at once (speculative
 * verification, multi-token prediction): query t (0 <= t < T_q) of sequence b
 * sits at position L - T_q + t, L = seq_lens[b], and attends keys
 * 0 .. L - T_q + t of the cache (causal, aligned to the end of the sequence:
 * "Attention Kernel 계보" p.13 §1 with the chunk offset of ADR-0060 §5.4).
 * The T_q * G query rows of one KV head are folded into the M dimension of
 * the split-KV decode.  Up to 16 rows, and for d = 32 or 64 up to 64 rows in
 * groups of 16 (one mma.sync tile each, one CTA per group and split).  With
 * d = 128 and more than 16 rows, all rows (up to 128) form one tensor-core
 * tile, with one CTA per split reading each K/V tile once; its splits cover
 * 128-key multiples (ceil(S_max / n_split) rounded up to 128).
 * GQA_ERR_UNSUPPORTED for more rows, GQA_ERR_INVALID_ARG for T_q outside 1..64;
 * larger chunks go to gqa_attn_prefill_chunk.  q and out are bf16 [B, T_q, H_q, d],
 * lse fp32 [B, T_q, H_q] (natural log); the cache layout, splits and errors
 * are those of gqa_attn_decode, with the device check 1 <= T_q <= L <= S_max.
 * With n_split > 1 the partials go to `workspace`
 * (gqa_attn_decode_workspace_bytes(B * T_q, H_q, d, n_split) bytes) and
 * gqa_attn_decode_combine(workspace, B * T_q, H_q, d, n_split, out, lse)
 * merges them.  T_q = 1 is gqa_attn_decode. */
gqa_status gqa_attn_decode_multi(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* seq_lens, int B, int T_q, int S_max, int H_q,
                                 int H_kv, int d, float scale, int n_split, void* workspace,
                                 void* out, float* lse, gqa_stream_t stream);

/* Split count for gqa_attn_decode_multi on the current device: that of
 * gqa_attn_decode_default_splits when the T_q * G rows fit one group of 16 or
 * go to the tensor-core tile (d = 128); with more mma.sync groups, at most the
 * count that keeps all groups of all splits resident at once (two CTAs per
 * SM).  Returns >= 1. */
int gqa_attn_decode_multi_default_splits(int B, int T_q, int H_q, int H_kv, int S_max, int d);

/* gqa_attn_decode_multi over a paged cache: the cache, block table and page
 * rules of gqa_attn_decode_paged, the query rows, outputs, workspace and merge
 * of gqa_attn_decode_multi (including the tensor-core tile for more than 16
 * rows at d = 128, whose splits cover 128-key multiples and which needs no
 * page-count limit per split).  T_q = 1 is gqa_attn_decode_paged. */
gqa_status gqa_attn_decode_paged_multi(const void* q, const void* k_pool, const void* v_pool,
                                       const int32_t* block_table, const int32_t* seq_lens, int B,
                                       int T_q, int num_pages, int page_size, int max_blocks,
                                       int H_q, int H_kv, int d, float scale, int n_split,
                                       void* workspace, void* out, float* lse,
                                       gqa_stream_t stream);

/* ------------------------------------------------------------------------
 * Decode with the merge inside thread-block clusters
 * ------------------------------------------------------------------------ */

/* Number of KV splits gqa_attn_decode_fused uses on the current device for
 * this head shape: the largest cluster size (16, else 8) whose CTAs can be
 * resident together; 0 when the shape is unsupported (d not 32/64/128, G > 16,
 * H_q not a multiple of H_kv) or no such cluster fits. */
int gqa_attn_decode_fused_splits(int B, int H_q, int H_kv, int d);

/* The same computation as gqa_attn_decode followed by gqa_attn_decode_combine
 * (split-KV sweep, then the log-sum-exp merge of the split partials;
 * "Attention Kernel 계보" p.18 §4 and p.4), in one launch and without a
 * workspace.  The n_split = gqa_attn_decode_fused_splits(...) CTAs of one
 * (KV head, sequence) form a thread-block cluster; each keeps its partial
 * (m, l, O) in shared memory, and the cluster folds them through distributed
 * shared memory.  Arguments, layouts, outputs and error behaviour are those
 * of gqa_attn_decode with n_split = 1 (out [B, H_q, d] bf16, lse [B, H_q]
 * fp32, natural log; a bad seq_lens entry gives NaN rows and
 * GQA_ERR_INVALID_ARG from gqa_last_device_error).  GQA_ERR_UNSUPPORTED when
 * gqa_attn_decode_fused_splits returns 0.  Results differ from the two-kernel
 * path only by rounding (a different split count). */
gqa_status gqa_attn_decode_fused(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* seq_lens, int B, int S_max, int H_q, int H_kv,
                                 int d, float scale, void* out, float* lse, gqa_stream_t stream);

/* ------------------------------------------------------------------------
 * Diagnostics
 * ------------------------------------------------------------------------ */

/* Synchronises `stream`, reads and clears the current device's error word and
 * maps it to a status: GQA_ERR_TIMEOUT if a wait timed out, else
 * GQA_ERR_INVALID_ARG if a device-side argument check failed, else GQA_OK.
 * GQA_ERR_CUDA if the synchronisation itself failed, or, in a library built
 * with -DGQA_DEBUG_BOUNDS=1, if a kernel computed a global store index outside
 * the buffer its parameters describe (that store is skipped; this check
 * comes first).  The default build compiles those checks out. */
gqa_status gqa_last_device_error(gqa_stream_t stream);

/* Sets the time limit, in nanoseconds, of every device pipeline wait launched
 * afterwards from this process (default 2e9; values < 1000 are raised to 1000).
 * Returns the previous limit. */
uint64_t gqa_set_wait_limit_ns(uint64_t limit_ns);

/* Launches one CTA that waits on a pipeline barrier nothing will ever signal,
 * using the same bounded wait as the kernels, with a limit of `limit_ns`.  The
 * wait must give up, set the timeout bit and return; a following
 * gqa_last_device_error() then reports GQA_ERR_TIMEOUT.  Used to test the
 * failure path without hanging a GPU. */
gqa_status gqa_selftest_wait_timeout(uint64_t limit_ns, gqa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
