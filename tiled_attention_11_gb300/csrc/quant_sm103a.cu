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

// Up to three tensors per launch (grid.y selects one); amax_bits[y] receives its maximum.
struct Segs3 {
  const __nv_bfloat16* x0;
  const __nv_bfloat16* x1;
  const __nv_bfloat16* x2;
  long long n0, n1, n2;
};

__global__ void __launch_bounds__(256) amax_kernel(const Segs3 segs, unsigned* __restrict__ amax_bits) {
  // the quantise kernel that follows may be launched now; it waits for this grid's result
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int t = (int)blockIdx.y;
  const __nv_bfloat16* __restrict__ x = t == 0 ? segs.x0 : t == 1 ? segs.x1 : segs.x2;
  const long long n = t == 0 ? segs.n0 : t == 1 ? segs.n1 : segs.n2;
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
    atomicMax(amax_bits + t, __float_as_uint(b));  // non-negative floats order as their bits
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

// V^T slab: x [BH][N][D] bf16 -> codes_t [BH][D][ldt], one block of 256 threads per
// (128-key slab, head).  Thread item (part, g) holds columns 8*part .. 8*part+7 of keys
// 4g .. 4g+3; consecutive lanes take consecutive parts, so each load instruction of a warp
// reads whole key rows.  Per column the 4 codes go to shared memory as one 32-bit word of
// the transposed tile ([d][128 keys], 128 bytes a row), whose word index is XORed with
// swz(d) so that the 32 words a warp writes at once fall on 32 banks; each row then leaves
// as eight 16-byte stores (a warp writes four whole 128-byte row segments).  Keys at or past
// N load as zero and give zero codes; 16-byte chunks that start at or past N are not written
// (ldt >= N rounded up to 16, so written chunks stay inside the row).
template <int D>
struct VtSlab {
  static constexpr int KEYS = 128;
  static constexpr int P = D / 8;               // 16-byte column groups of a key row
  static constexpr int G = KEYS / 4;            // groups of 4 keys = 32-bit words of a tile row
  static constexpr int PER = P * G / 256;       // items per thread (2 at D = 128, 1 at D = 64)
  static_assert(P * G % 256 == 0, "items fill the block");
  __device__ static __forceinline__ int swz(int d) { return ((d >> 3) * (32 / P)) & 31; }

  uint4 w[PER][4];

  __device__ __forceinline__ void load(const __nv_bfloat16* __restrict__ x, int N, int bh, int k0) {
    const __nv_bfloat16* xs = x + ((size_t)bh * N + k0) * D;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = (int)threadIdx.x + 256 * u, part = e % P, g = e / P;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int key = 4 * g + r;
        w[u][r] = k0 + key < N ? ld16(reinterpret_cast<const uint4*>(xs + (size_t)key * D) + part)
                               : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }

  // tile: D * G words of shared memory; ends with the block's stores to codes_t
  __device__ __forceinline__ void finish(float mult, uint32_t* tile, int N, int ldt, uint8_t* __restrict__ codes_t,
                                         int bh, int k0) const {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = (int)threadIdx.x + 256 * u, part = e % P, g = e / P;
      uint2 c[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) c[r] = quant8(w[u][r], mult);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int sh = 8 * (i & 3), d = part * 8 + i;
        uint32_t v = 0u;
#pragma unroll
        for (int r = 0; r < 4; ++r) v |= (((i < 4 ? c[r].x : c[r].y) >> sh) & 0xffu) << (8 * r);
        tile[d * G + (g ^ swz(d))] = v;
      }
    }
    __syncthreads();
    uint8_t* out = codes_t + (size_t)bh * D * ldt + k0;
#pragma unroll
    for (int e = (int)threadIdx.x; e < D * (KEYS / 16); e += 256) {
      const int d = e / (KEYS / 16), ch = e % (KEYS / 16);
      if (k0 + ch * 16 < N) {
        const int s = swz(d);  // logical words 4ch+t sit at physical 4(ch ^ s/4) + (t ^ (s & 3))
        const uint4 ph = *reinterpret_cast<const uint4*>(&tile[d * G + 4 * (ch ^ (s >> 2))]);
        const uint4 lg = (s & 2) ? make_uint4(ph.z, ph.w, ph.x, ph.y) : ph;
        *reinterpret_cast<uint4*>(out + (size_t)d * ldt + ch * 16) = lg;
      }
    }
  }
};

template <int D>
__global__ void __launch_bounds__(256) quant_t_kernel(const __nv_bfloat16* __restrict__ x, int N, int ldt,
                                                      const float* __restrict__ amax, uint8_t* __restrict__ codes_t,
                                                      float* __restrict__ descale) {
  __shared__ __align__(16) uint32_t tile[D * VtSlab<D>::G];
  const int bh = blockIdx.y, k0 = blockIdx.x * VtSlab<D>::KEYS;
  VtSlab<D> sl;
  sl.load(x, N, bh, k0);  // x is not written by the amax grid: its loads may precede the wait
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the amax grid has completed
  const float a = *amax;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *descale = a > 0.f ? a / 448.f : 1.f;
  sl.finish(multiplier(a), tile, N, ldt, codes_t, bh, k0);
}

// Q, K and V of one attention call in one launch, after one amax launch over the three:
// blocks [0, n_vt) are V^T slabs, then Q and K in chunks of 2048 16-byte groups (32 KB of
// bf16 in, 16 KB of codes out per block, eight loads in flight per thread), so every block
// moves the same bytes.  Codes and descales equal the per-tensor kernels' bit for bit.
struct QkvArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  uint8_t* q8;
  uint8_t* k8;
  uint8_t* vt8;
  const float* amax;  // [3]: q, k, v
  float* descale;     // [3]
  long long nq8, nk8;  // 16-byte groups of q and k
  int BH, Nk, ldv, n_slabs, n_vt, n_qb;
};
constexpr int kChunkU = 8, kChunk = 256 * kChunkU;

template <int D>
__global__ void __launch_bounds__(256) quant_qkv_kernel(const QkvArgs a) {
  __shared__ __align__(16) uint32_t tile[D * VtSlab<D>::G];
  const int b = (int)blockIdx.x;
  if (b < a.n_vt) {
    const int bh = b / a.n_slabs, k0 = (b % a.n_slabs) * VtSlab<D>::KEYS;
    VtSlab<D> sl;
    sl.load(a.v, a.Nk, bh, k0);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the amax grid has completed
    if (b == 0 && threadIdx.x < 3) {
      const float m = a.amax[threadIdx.x];
      a.descale[threadIdx.x] = m > 0.f ? m / 448.f : 1.f;
    }
    sl.finish(multiplier(a.amax[2]), tile, a.Nk, a.ldv, a.vt8, bh, k0);
    return;
  }
  const bool is_q = b - a.n_vt < a.n_qb;
  const long long n8 = is_q ? a.nq8 : a.nk8;
  const uint4* x8 = reinterpret_cast<const uint4*>(is_q ? a.q : a.k);
  uint2* c8 = reinterpret_cast<uint2*>(is_q ? a.q8 : a.k8);
  const long long base = (long long)(is_q ? b - a.n_vt : b - a.n_vt - a.n_qb) * kChunk + threadIdx.x;
  uint4 w[kChunkU];
#pragma unroll
  for (int u = 0; u < kChunkU; ++u) {
    const long long i = base + 256 * u;
    w[u] = i < n8 ? ld16(x8 + i) : make_uint4(0u, 0u, 0u, 0u);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float mult = multiplier(a.amax[is_q ? 0 : 1]);
#pragma unroll
  for (int u = 0; u < kChunkU; ++u) {
    const long long i = base + 256 * u;
    if (i < n8) c8[i] = quant8(w[u], mult);
  }
}

int grid_for(long long n8) {
  long long g = (n8 + 255) / 256;
  if (g > 152 * 8) g = 152 * 8;
  return g < 1 ? 1 : (int)g;
}

}  // namespace quant

cudaError_t launch_amax_bf16(const void* x, long long n, float* amax, cudaStream_t st) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  const quant::Segs3 segs{xb, xb, xb, n, n, n};
  quant::amax_kernel<<<quant::grid_for(n / 8 + 1), 256, 0, st>>>(segs, reinterpret_cast<unsigned*>(amax));
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
  dim3 grid((unsigned)((N + 127) / 128), (unsigned)BH);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  uint8_t* c = static_cast<uint8_t*>(codes_t);
  switch (D) {
    case 64: return quant::launch_dependent(quant::quant_t_kernel<64>, grid, st, xb, N, ldt, amax, c, descale);
    case 128: return quant::launch_dependent(quant::quant_t_kernel<128>, grid, st, xb, N, ldt, amax, c, descale);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_quantize_qkv(const void* q, const void* k, const void* v, int BH, int Nq, int Nk, int D,
                                void* q8, void* k8, void* vt8, int ldv, float* amax, float* descale,
                                cudaStream_t st) {
  const long long nq = (long long)BH * Nq * D, nk = (long long)BH * Nk * D;
  const quant::Segs3 segs{static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                          static_cast<const __nv_bfloat16*>(v), nq, nk, nk};
  const long long nmax = nq > nk ? nq : nk;
  quant::amax_kernel<<<dim3((unsigned)quant::grid_for(nmax / 8 + 1), 3), 256, 0, st>>>(
      segs, reinterpret_cast<unsigned*>(amax));
  if (cudaGetLastError() != cudaSuccess) return cudaErrorLaunchFailure;
  quant::QkvArgs a{};
  a.q = segs.x0;
  a.k = segs.x1;
  a.v = segs.x2;
  a.q8 = static_cast<uint8_t*>(q8);
  a.k8 = static_cast<uint8_t*>(k8);
  a.vt8 = static_cast<uint8_t*>(vt8);
  a.amax = amax;
  a.descale = descale;
  a.nq8 = nq / 8;  // D is a multiple of 64: no elements past the last 16-byte group
  a.nk8 = nk / 8;
  a.BH = BH;
  a.Nk = Nk;
  a.ldv = ldv;
  const long long n_vt = (long long)((Nk + 127) / 128) * BH;
  const long long n_qb = (a.nq8 + quant::kChunk - 1) / quant::kChunk;
  const long long n_kb = (a.nk8 + quant::kChunk - 1) / quant::kChunk;
  const long long blocks = n_vt + n_qb + n_kb;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;  // (checked before any narrowing)
  a.n_slabs = (Nk + 127) / 128;
  a.n_vt = (int)n_vt;
  a.n_qb = (int)n_qb;
  const dim3 grid((unsigned)blocks);
  switch (D) {
    case 64: return quant::launch_dependent(quant::quant_qkv_kernel<64>, grid, st, a);
    case 128: return quant::launch_dependent(quant::quant_qkv_kernel<128>, grid, st, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ta11
