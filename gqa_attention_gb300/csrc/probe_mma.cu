// probe_mma.cu -- issue rate of tcgen05.mma forms (trace build only).
//
// A diagnostic behind the tensor-core kernels' design: one CTA per SM issues
// `iters` rounds of back-to-back tcgen05.mma of one form from a converged warp
// (zero operands, results discarded) and reads clock64 around them.  The host
// reports the median over SMs of SM cycles per instruction, to be set against
// the nominal rate of 8192 bf16 FLOP per clock per SM (M = 128, K = 16:
// 32 cycles at N = 64, 64 at N = 128, 128 at N = 256).  Every form is a
// template instance, so the issue loop is straight-line code: a runtime branch
// between the instructions slows the issue itself and the measurement with it.
// Built with -DGQA_TRACE=1 only; other builds return GQA_ERR_UNSUPPORTED.
#include <algorithm>
#include <vector>

#include "gqa_attn.h"
#include "tcgen05.cuh"

#ifndef GQA_TRACE
#define GQA_TRACE 0
#endif

namespace gqa {
namespace {

#if GQA_TRACE
constexpr int kProbeMaxSms = 512;
constexpr int kProbeForms = 6;
__device__ unsigned long long g_probe_cycles[kProbeMaxSms];
__device__ unsigned g_probe_err;

// Instructions per round of each form.
__host__ __device__ constexpr int probe_per_round(int form) { return form == 5 ? 16 : 8; }

// form 0: SS, N = 128      form 1: TS, N = 128 (A in tensor memory)
// form 2: SS, N = 256      form 3: SS, N = 64
// form 4: TS, N = 128, B MN-major (the P V form of the prefill)
// form 5: the causal prefill's step for one head: 8 SS (S = Q K^T) then 8 TS
//         (O += P V), head and ring slot chosen at run time as there.
template <int FORM>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int iters, uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tbase;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done), 1);
    fence_barrier_init();
  }
  // Operands: four 32 KB tiles of zeros (A at 0, B from 64 KB).
  for (int i = threadIdx.x; i < 4 * 32768 / 16; i += 128) st_shared_v4(sb + i * 16, 0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(&tbase), 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tbase;
  if (warp == 0) {
    constexpr int N = FORM == 2 ? 256 : FORM == 3 ? 64 : 128;
    constexpr uint32_t id = instr_desc_bf16_f32(128, N, FORM == 4);
    constexpr uint32_t idPV = instr_desc_bf16_f32(128, 128, true);
    const uint32_t A = sb, B = sb + 65536;
    const unsigned long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
      if constexpr (FORM == 5) {
        const int x = it & 1;
        const uint32_t slot = static_cast<uint32_t>(it) & 1u;
        const uint32_t qa = A + x * 32768, kb = B + slot * 32768;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          tc_mma_ss(tmem + 128 * x, smem_desc_sw128(qa + off, 16, 1024),
                    smem_desc_sw128(kb + off, 16, 1024), id, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_ts(tmem + 256 + 128 * x, tmem + 128 * x + 8 * kk,
                    smem_desc_sw128(kb + kk * 2048, 16384, 1024), idPV, 1);
      } else {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t acc = (kk > 0 || it > 0) ? 1u : 0u;
          if constexpr (FORM == 1)
            tc_mma_ts(tmem, tmem + 384 + 8 * kk, smem_desc_sw128(B + off, 16, 1024), id, acc);
          else if constexpr (FORM == 4)
            tc_mma_ts(tmem, tmem + 384 + 8 * kk, smem_desc_sw128(B + kk * 2048, 16384, 1024), id,
                      acc);
          else
            tc_mma_ss(tmem, smem_desc_sw128(A + off, 16, 1024), smem_desc_sw128(B + off, 16, 1024),
                      id, acc);
        }
      }
    }
    tc_commit(smem_u32(&done));
    const bool ok = mbar_wait(smem_u32(&done), 0, wait_ns, &g_probe_err);
    const unsigned long long t1 = clock64();
    if (threadIdx.x == 0 && blockIdx.x < kProbeMaxSms) g_probe_cycles[blockIdx.x] = ok ? t1 - t0 : 0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int FORM>
cudaError_t launch_mma_rate(int sms, int iters, uint64_t wait_ns) {
  // 4 x 32 KB operands, alignment slack, and enough more that one CTA fills an SM
  constexpr int smem = 4 * 32768 + 1024 + 40000;
  cudaError_t e = cudaFuncSetAttribute(mma_rate_kernel<FORM>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mma_rate_kernel<FORM><<<sms, 128, smem>>>(iters, wait_ns);
  return cudaGetLastError();
}
#endif

}  // namespace
}  // namespace gqa

extern "C" gqa_status gqa_trace_mma_rate(int form, int iters, double* cycles_per_instruction) {
#if GQA_TRACE
  using namespace gqa;
  if (!cycles_per_instruction || form < 0 || form >= kProbeForms || iters < 1 || iters > (1 << 16))
    return GQA_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GQA_ERR_CUDA;
  sms = std::min(sms, kProbeMaxSms);
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_probe_err, &zero, sizeof zero) != cudaSuccess) return GQA_ERR_CUDA;
  const uint64_t wait_ns = 2000000000ull;  // 2 s: far beyond any round count accepted here
  cudaError_t e;
  switch (form) {
    case 0: e = launch_mma_rate<0>(sms, iters, wait_ns); break;
    case 1: e = launch_mma_rate<1>(sms, iters, wait_ns); break;
    case 2: e = launch_mma_rate<2>(sms, iters, wait_ns); break;
    case 3: e = launch_mma_rate<3>(sms, iters, wait_ns); break;
    case 4: e = launch_mma_rate<4>(sms, iters, wait_ns); break;
    default: e = launch_mma_rate<5>(sms, iters, wait_ns); break;
  }
  if (e != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return GQA_ERR_CUDA;
  unsigned err = 0;
  std::vector<unsigned long long> cyc(sms);
  if (cudaMemcpyFromSymbol(&err, g_probe_err, sizeof err) != cudaSuccess ||
      cudaMemcpyFromSymbol(cyc.data(), g_probe_cycles, sizeof(unsigned long long) * sms) !=
          cudaSuccess)
    return GQA_ERR_CUDA;
  if (err != 0) return GQA_ERR_TIMEOUT;
  std::sort(cyc.begin(), cyc.end());
  *cycles_per_instruction =
      static_cast<double>(cyc[sms / 2]) / (static_cast<double>(iters) * probe_per_round(form));
  return GQA_OK;
#else
  (void)form;
  (void)iters;
  (void)cycles_per_instruction;
  return GQA_ERR_UNSUPPORTED;
#endif
}
