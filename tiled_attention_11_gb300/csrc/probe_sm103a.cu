// Measurement library (libta11_probe.so, declared in probe.h): microbenchmarks of the
// roofs the attention kernels are judged against.  Not part of the attention library.
//   umma_probe_kernel  the tensor core's rate for the score GEMM's UMMA shape (M = N =
//                      128, K = 16, bf16 operands from 128-byte swizzled K-major shared
//                      memory, fp32 accumulate in TMEM), issued back to back by one thread
//                      per CTA, one CTA per SM: the tensor roof at the running clock.
//   ex2_probe_kernel   the special-function unit's exp2 rate (the softmax's third roof).
#include <cuda_runtime.h>

#include "probe.h"
#include "ptx_sm103a.cuh"

namespace {

__device__ unsigned g_probe_status[2];

constexpr int kRows = 128, kRowBytes = 128, kChunkBytes = kRows * kRowBytes;  // one 64-column chunk
constexpr int kChunks = 2;                                                      // K = 128 per group
constexpr int kTileBytes = kChunks * kChunkBytes;
// A and B tiles plus alignment room use 65 KB; 120 KB is reserved so that one CTA fits
// per SM and each SM's tensor core serves one issuing thread.
constexpr int kSmem = 120 * 1024;
static_assert(2 * kTileBytes + 1024 <= kSmem, "tiles fit");
constexpr uint32_t kIdesc = ta11::idesc_bf16(128, 128, false, false);
constexpr uint32_t kTmemCols = 128;

__device__ __forceinline__ uint32_t kmajor_off(int kk) {  // K step kk (16 elements) in a tile
  return (uint32_t)((kk * 16 / 64) * kChunkBytes + (kk * 16 % 64) * 2);
}

// `iters` groups of 8 UMMAs (K = 128) into one accumulator; the operand tiles are zeros
// (the rate does not depend on the data).  The wait for completion is bounded.
__global__ void __launch_bounds__(128, 1) umma_probe_kernel(int iters, unsigned long long limit_ns, unsigned* status) {
  using namespace ta11;
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

// Every thread runs 8 independent chains x <- 2^(-x) (values stay in [0.5, 1], no
// subnormals or overflow), so the exp2 pipe, not the chains' latency, sets the time.
// out[i] keeps the chains' sum so nothing is elided.
constexpr int kEx2Threads = 512, kEx2Chains = 8;
__global__ void __launch_bounds__(kEx2Threads) ex2_probe_kernel(float* out, int iters) {
  float x[kEx2Chains];
#pragma unroll
  for (int c = 0; c < kEx2Chains; ++c) x[c] = 0.03125f * (float)((threadIdx.x + c) & 31);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kEx2Chains; ++c) asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(x[c]) : "f"(-x[c]));
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kEx2Chains; ++c) s += x[c];
  out[(size_t)blockIdx.x * kEx2Threads + threadIdx.x] = s;
}

bool on_sm103() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return major == 10 && minor == 3;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" {

int ta11_probe_ex2(float* out, int n_blocks, int iters, cudaStream_t stream) {
  if (!out || n_blocks < 1 || n_blocks > 65535 || iters < 1 || iters > (1 << 20)) return 1;
  if (!aligned4(out)) return 3;
  if (!on_sm103()) return 5;
  ex2_probe_kernel<<<n_blocks, kEx2Threads, 0, stream>>>(out, iters);
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

int ta11_probe_umma(int n_ctas, int iters, unsigned long long limit_ns, cudaStream_t stream) {
  if (n_ctas < 1 || n_ctas > 65535 || iters < 1 || iters > (1 << 16)) return 1;
  if (!on_sm103()) return 5;
  void* st = nullptr;
  if (cudaGetSymbolAddress(&st, g_probe_status) != cudaSuccess) {
    cudaGetLastError();
    return 5;
  }
  if (cudaFuncSetAttribute(umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return 6;
  umma_probe_kernel<<<n_ctas, 128, kSmem, stream>>>(iters, limit_ns, static_cast<unsigned*>(st));
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

int ta11_probe_status(int reset) {
  if (!on_sm103()) return 5;
  unsigned h[2] = {0u, 0u};
  if (cudaMemcpyFromSymbol(h, g_probe_status, sizeof(h)) != cudaSuccess) {
    cudaGetLastError();
    return 6;
  }
  if (reset) {
    const unsigned z[2] = {0u, 0u};
    if (cudaMemcpyToSymbol(g_probe_status, z, sizeof(z)) != cudaSuccess) {
      cudaGetLastError();
      return 6;
    }
  }
  return (int)h[0];
}

}  // extern "C"
