// Per-tensor e4m3 quantisation of bf16 tensors for the FP8 forward ("FlashAttention技术演进全景图"
// §5.3 names FP8 as the quantised direction; the per-tensor scheme is the usual one):
//   amax = max |x|,  codes = e4m3(x * (448 / amax)) (round to nearest even, saturating),
//   descale = amax / 448 (both divisions IEEE fp32, so codes are fixed bit for bit),
// an all-zero tensor uses multiplier and descale 1.  HBM-bound: one read for amax, one
// read + 1-byte write for the codes; V is written transposed ([BH][D][ldt], keys
// innermost) through a shared-memory tile so both FP8 GEMMs read K-major operands.
#include <cuda_bf16.h>

#include "fa_kernels.h"
#include "ptx_sm103a.cuh"

namespace ta11 {
namespace quant {

__device__ __forceinline__ float absmax8(const uint4 w, float m) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  return m;
}

// Loads of 16 bytes, four independent ones in flight per thread (enough bytes in flight per
// SM to cover the HBM latency); read-only path.
__device__ __forceinline__ uint4 ld16(const uint4* p) { return __ldg(p); }

__global__ void __launch_bounds__(256) amax_kernel(const __nv_bfloat16* __restrict__ x, long long n,
                                                   unsigned* __restrict__ amax_bits) {
  // the quantise kernel that follows may be launched now; it waits for this grid's result
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  float m0 = 0.f, m1 = 0.f, m2 = 0.f, m3 = 0.f;
  const long long n8 = n / 8;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const uint4* x8 = reinterpret_cast<const uint4*>(x);
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    const uint4 a = ld16(x8 + i), b = ld16(x8 + i + stride), c = ld16(x8 + i + 2 * stride),
                d = ld16(x8 + i + 3 * stride);
    m0 = absmax8(a, m0);
    m1 = absmax8(b, m1);
    m2 = absmax8(c, m2);
    m3 = absmax8(d, m3);
  }
  for (; i < n8; i += stride) m0 = absmax8(ld16(x8 + i), m0);
  for (long long j = n8 * 8 + (long long)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
    m0 = fmaxf(m0, fabsf(__bfloat162float(x[j])));
  float m = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wm[8];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = wm[0];
    for (int w = 1; w < 8; ++w) b = fmaxf(b, wm[w]);
    atomicMax(amax_bits, __float_as_uint(b));  // non-negative floats order as their bits
  }
}

__device__ __forceinline__ float multiplier(float amax) { return amax > 0.f ? 448.f / amax : 1.f; }

__device__ __forceinline__ uint2 quant8(const uint4 w, float mult) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
  float f[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = __fmul_rn(v.x, mult);
    f[2 * i + 1] = __fmul_rn(v.y, mult);
  }
  return make_uint2(pack_e4m3x4(f[0], f[1], f[2], f[3]), pack_e4m3x4(f[4], f[5], f[6], f[7]));
}

__global__ void __launch_bounds__(256) quant_kernel(const __nv_bfloat16* __restrict__ x, long long n,
                                                    const float* __restrict__ amax, uint8_t* __restrict__ codes,
                                                    float* __restrict__ descale) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the amax grid has completed
  const float a = *amax;
  const float mult = multiplier(a);
  if (blockIdx.x == 0 && threadIdx.x == 0) *descale = a > 0.f ? a / 448.f : 1.f;
  const long long n8 = n / 8;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const uint4* x8 = reinterpret_cast<const uint4*>(x);
  uint2* c8 = reinterpret_cast<uint2*>(codes);
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    const uint4 a = ld16(x8 + i), b = ld16(x8 + i + stride), c = ld16(x8 + i + 2 * stride),
                d = ld16(x8 + i + 3 * stride);
    c8[i] = quant8(a, mult);
    c8[i + stride] = quant8(b, mult);
    c8[i + 2 * stride] = quant8(c, mult);
    c8[i + 3 * stride] = quant8(d, mult);
  }
  for (; i < n8; i += stride) c8[i] = quant8(ld16(x8 + i), mult);
  for (long long j = n8 * 8 + (long long)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    const uint32_t w = pack_e4m3x4(__fmul_rn(__bfloat162float(x[j]), mult), 0.f, 0.f, 0.f);
    codes[j] = (uint8_t)(w & 0xffu);
  }
}

// x [BH][N][D] bf16 -> codes_t [BH][D][ldt]: one block per (64-key slab, head).  A thread
// quantises the same 8 columns of 4 consecutive keys and writes, per column, the 4 codes
// as one 32-bit word of the transposed tile; tile rows are 72 bytes apart so the two
// column groups a warp writes fall on different banks.  Every byte of [0, ldt) of a row is
// written (keys past N as zero codes).
template <int D>
__global__ void __launch_bounds__(256) quant_t_kernel(const __nv_bfloat16* __restrict__ x, int N, int ldt,
                                                      const float* __restrict__ amax, uint8_t* __restrict__ codes_t,
                                                      float* __restrict__ descale) {
  constexpr int KEYS = 64, ROW = KEYS + 8;  // tile row stride (bytes)
  __shared__ __align__(16) uint8_t tile[D * ROW];  // [d][key]
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the amax grid has completed
  const float a = *amax;
  const float mult = multiplier(a);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *descale = a > 0.f ? a / 448.f : 1.f;
  const int bh = blockIdx.y;
  const int k0 = blockIdx.x * KEYS;
  const __nv_bfloat16* xs = x + ((size_t)bh * N + k0) * D;
  for (int e = threadIdx.x; e < (KEYS / 4) * (D / 8); e += blockDim.x) {
    const int j = e % (KEYS / 4), part = e / (KEYS / 4);  // keys 4j .. 4j+3, columns 8*part ..
    uint4 w[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int key = 4 * j + r;
      w[r] = k0 + key < N ? ld16(reinterpret_cast<const uint4*>(xs + (size_t)key * D) + part) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint2 c[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) c[r] = quant8(w[r], mult);  // (zero input -> zero codes)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int sh = 8 * (i & 3);
      uint32_t v = 0u;
#pragma unroll
      for (int r = 0; r < 4; ++r) v |= (((i < 4 ? c[r].x : c[r].y) >> sh) & 0xffu) << (8 * r);
      *reinterpret_cast<uint32_t*>(&tile[(part * 8 + i) * ROW + 4 * j]) = v;
    }
  }
  __syncthreads();
  uint8_t* out = codes_t + (size_t)bh * D * ldt + k0;
  for (int e = threadIdx.x; e < D * (KEYS / 16); e += blockDim.x) {
    const int d = e / (KEYS / 16), chunk = e % (KEYS / 16);
    if (k0 + chunk * 16 < N) {  // ldt >= N rounded up to 16, so whole 16-byte chunks fit
      const uint2* src = reinterpret_cast<const uint2*>(&tile[d * ROW + chunk * 16]);
      const uint2 lo = src[0], hi = src[1];
      *reinterpret_cast<uint4*>(out + (size_t)d * ldt + chunk * 16) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
  }
}

int grid_for(long long n8) {
  long long g = (n8 + 255) / 256;
  if (g > 152 * 8) g = 152 * 8;
  return g < 1 ? 1 : (int)g;
}

}  // namespace quant

cudaError_t launch_amax_bf16(const void* x, long long n, float* amax, cudaStream_t st) {
  quant::amax_kernel<<<quant::grid_for(n / 8 + 1), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), n,
                                                                  reinterpret_cast<unsigned*>(amax));
  return cudaGetLastError();
}

namespace quant {
// Launch on `st` as a programmatic dependent of the amax kernel before it: the grid may
// start while that one drains, and waits (griddepcontrol.wait) before it reads amax.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}
}  // namespace quant

cudaError_t launch_quant_e4m3(const void* x, long long n, const float* amax, void* codes, float* descale,
                              cudaStream_t st) {
  return quant::launch_dependent(quant::quant_kernel, dim3((unsigned)quant::grid_for(n / 8 + 1)), st,
                                 static_cast<const __nv_bfloat16*>(x), n, amax, static_cast<uint8_t*>(codes), descale);
}

cudaError_t launch_quant_e4m3_t(const void* x, int BH, int N, int D, int ldt, const float* amax, void* codes_t,
                                float* descale, cudaStream_t st) {
  dim3 grid((unsigned)((N + 63) / 64), (unsigned)BH);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  uint8_t* c = static_cast<uint8_t*>(codes_t);
  switch (D) {
    case 64: return quant::launch_dependent(quant::quant_t_kernel<64>, grid, st, xb, N, ldt, amax, c, descale);
    case 128: return quant::launch_dependent(quant::quant_t_kernel<128>, grid, st, xb, N, ldt, amax, c, descale);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ta11
