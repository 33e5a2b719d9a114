// Measurement kernel: the tensor core's rate for the UMMA shape of the attention
// kernels' score GEMM (M = N = 128, K = 16 per instruction, bf16 operands from 128-byte
// swizzled K-major shared-memory tiles, fp32 accumulate in TMEM), issued back to back by
// one thread per CTA with one CTA per SM.  It gives the tensor roof at the clock the
// kernels actually run, beside the library-GEMM peak the roofline fractions use.
#include <cuda_runtime.h>

#include "fa_kernels.h"
#include "ptx_sm103a.cuh"

namespace ta11 {
namespace probe {

constexpr int kRows = 128, kRowBytes = 128, kChunkBytes = kRows * kRowBytes;  // one 64-column chunk
constexpr int kChunks = 2;                                                      // K = 128 per group
constexpr int kTileBytes = kChunks * kChunkBytes;
// A and B tiles plus alignment room use 65 KB; 120 KB is reserved so that one CTA fits
// per SM and each SM's tensor core serves one issuing thread.
constexpr int kSmem = 120 * 1024;
static_assert(2 * kTileBytes + 1024 <= kSmem, "tiles fit");
constexpr uint32_t kIdesc = idesc_bf16(128, 128, false, false);
constexpr uint32_t kTmemCols = 128;

__device__ __forceinline__ uint32_t kmajor_off(int kk) {  // K step kk (16 elements) in a tile
  return (uint32_t)((kk * 16 / 64) * kChunkBytes + (kk * 16 % 64) * 2);
}

// `iters` groups of 8 UMMAs (K = 128) into one accumulator; the operand tiles are zeros
// (the rate does not depend on the data).  The wait for completion is bounded.
__global__ void __launch_bounds__(128, 1) umma_probe_kernel(int iters, unsigned long long limit_ns, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  for (int i = (int)threadIdx.x; i < 2 * kTileBytes / 16; i += (int)blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (threadIdx.x == 0) {
    const uint32_t sbase = smem_u32(smem);
    const uint64_t da = sdesc(sbase, 16, 8 * kRowBytes, umma_layout_for_swizzle(kRowBytes));
    const uint64_t db = sdesc(sbase + kTileBytes, 16, 8 * kRowBytes, umma_layout_for_swizzle(kRowBytes));
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < kChunks * 4; ++kk)
        umma_ss(tmem, desc_adv(da, kmajor_off(kk)), desc_adv(db, kmajor_off(kk)), kIdesc, (it | kk) ? 1u : 0u);
    }
    umma_commit(&bar);
    const WaitCtx wc{limit_ns, status, &abort_flag};
    if (!mbar_wait(&bar, 0, wc, 60)) {  // (status recorded) still let the UMMAs finish before TMEM is freed
      volatile int no_abort = 0;
      const WaitCtx w2{limit_ns, status, &no_abort};
      mbar_wait(&bar, 0, w2, 61);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace probe

cudaError_t launch_umma_probe(int n_ctas, int iters, unsigned long long limit_ns, unsigned* status,
                              cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(probe::umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       probe::kSmem);
  if (e != cudaSuccess) return e;
  probe::umma_probe_kernel<<<n_ctas, 128, probe::kSmem, st>>>(iters, limit_ns, status);
  return cudaGetLastError();
}

}  // namespace ta11
