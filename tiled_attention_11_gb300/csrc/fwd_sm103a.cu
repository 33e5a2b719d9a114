// Forward pass of exact attention, tile by tile with an online softmax, for sm_103a.
//
// Method: "FlashAttention-2实现与优化：高效注意力机制详解" §3.1 (tiles of Q and K/V,
// running statistics (m, l, o_acc), m_new = max(m, rowmax S),
// l_new = e^(m-m_new) l + sum e^(S-m_new), o_acc = e^(m-m_new) o_acc + P V) and §3.2
// (one program per query tile, key-tile loop inside, O = o_acc / l, L = m + log l);
// the causal mask keeps key <= query on absolute indices (§4.3).  The scores are
// kept in base 2: with c = scale*log2(e), t = c*S, p = 2^(t - m2) and
// L = (m2 + log2 l) * ln 2, which is the same softmax.
//
// GB300 mapping (one CTA per (batch*head, 128-row query tile), 6 warps):
//   warp 0     TMA producer: Q once, then K_j / V_j through an NS-stage ring
//   warp 1     TMEM allocator and UMMA issuer (one thread):
//                S_j = Q K_j^T  -> TMEM (double-buffered, 128 fp32 columns each)
//                O  += P_j V_j  -> TMEM (P read from TMEM, aliasing S_j)
//   warps 2-5  softmax warpgroup, one thread per query row: TMEM -> registers,
//              mask (diagonal / ragged tiles only), online max / exp2 / sum,
//              P as bf16 back into TMEM, O rescale by alpha when the max moved,
//              and the epilogue O / l -> bf16, L.
// Every wait is bounded; a timeout records FA_ERR_TIMEOUT in the status word and
// the CTA drains its in-flight copies and MMAs before freeing TMEM.
#include "fa_kernels.h"
#include "ptx_sm103a.cuh"

namespace ta11 {
namespace fwd {

template <int D>
struct Cfg {
  static constexpr int BM = 128;                       // query rows per CTA
  static constexpr int BN = 128;                       // keys per tile
  static constexpr int CHUNK = D < 64 ? D : 64;        // elements per swizzled smem row
  static constexpr int NCHUNK = D / CHUNK;
  static constexpr int ROWB = CHUNK * 2;               // bytes per smem row == swizzle width
  static constexpr int CHUNK_BYTES = 128 * ROWB;
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr int NS = D <= 64 ? 4 : 2;           // K/V ring depth
  static constexpr uint32_t LAYOUT = umma_layout_for_swizzle(ROWB);
  static constexpr int TMEM_O = 256;
  static constexpr int TMEM_COLS = 512;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = TILE_BYTES;
  static constexpr int OFF_V = TILE_BYTES * (1 + NS);
  static constexpr int OFF_BAR = TILE_BYTES * (1 + 2 * NS);
  // barriers: q_full, k_full[NS], v_full[NS], kv_empty[NS], s_full[2], p_full[2], o_ready, drain
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 1;
  static constexpr int B_VF = 1 + NS;
  static constexpr int B_KVE = 1 + 2 * NS;
  static constexpr int B_SF = 1 + 3 * NS;
  static constexpr int B_PF = 3 + 3 * NS;
  static constexpr int B_O = 5 + 3 * NS;
  static constexpr int B_DRAIN = 6 + 3 * NS;
  static constexpr int NBAR = 7 + 3 * NS;
  static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 16;
  // At least ~120 KB so only one CTA (and one 512-column TMEM allocation) fits per SM.
  static constexpr int SMEM_ALLOC = (SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024) + 1024;
  static constexpr int THREADS = 192;
  static constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
  static_assert(TILE_BYTES % 1024 == 0, "tiles must keep 1024-byte alignment");
};

// K-major operand (rows of the tile x D contiguous): descriptor for the kk-th 16-wide K slice.
template <int D>
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
  using C = Cfg<D>;
  const int el = kk * 16;
  const uint32_t start = tile + (el / C::CHUNK) * C::CHUNK_BYTES + (el % C::CHUNK) * 2;
  return sdesc(start, 16, 8 * C::ROWB, C::LAYOUT);
}

// MN-major B operand (V: keys x D, D contiguous), kk-th slice of 16 keys.
template <int D>
__device__ __forceinline__ uint64_t desc_v(uint32_t tile, int kk) {
  using C = Cfg<D>;
  return sdesc(tile + kk * 16 * C::ROWB, C::CHUNK_BYTES, 8 * C::ROWB, C::LAYOUT);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, w, site));
}

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = (int)warp_id(), lane = (int)lane_id();
  // Query tiles of one head are adjacent in launch order, so the CTAs resident at
  // any moment share the K/V of a few heads in L2; within a head the heaviest
  // (causal) query tiles go first.
  const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;
  const int bh = blockIdx.y;
  const int q0 = qt * C::BM;
  const int nk_tiles = (p.Nk + C::BN - 1) / C::BN;
  const int n_kv = CAUSAL ? min(nk_tiles, qt + 1) : nk_tiles;
  const WaitCtx wc{p.wait_limit_ns, p.status, abort_flag};

  if (threadIdx.x == 0) {
    mbar_init(&bars[C::B_Q], 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bars[C::B_KF + s], 1);
      mbar_init(&bars[C::B_VF + s], 1);
      mbar_init(&bars[C::B_KVE + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[C::B_SF + b], 1);
      mbar_init(&bars[C::B_PF + b], 128);
    }
    mbar_init(&bars[C::B_O], 1);
    mbar_init(&bars[C::B_DRAIN], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&bars[C::B_Q], C::TILE_BYTES);
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_3d(smem + C::OFF_Q + c * C::CHUNK_BYTES, &tm_q, &bars[C::B_Q], c * C::CHUNK, q0, bh);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % C::NS;
        if (j >= C::NS && !mbar_wait(&bars[C::B_KVE + s], ((j / C::NS) - 1) & 1, wc, 1)) break;
        mbar_arrive_expect_tx(&bars[C::B_KF + s], C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(smem + C::OFF_K + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_k, &bars[C::B_KF + s],
                      c * C::CHUNK, j * C::BN, bh);
        mbar_arrive_expect_tx(&bars[C::B_VF + s], C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(smem + C::OFF_V + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_v, &bars[C::B_VF + s],
                      c * C::CHUNK, j * C::BN, bh);
        issued = j + 1;
      }
      if (*abort_flag) {
        // Let every copy already issued land before the CTA can exit.
        WaitCtx dw{p.wait_limit_ns, p.status, abort_flag};
        const int first = issued > C::NS ? issued - C::NS : 0;
        for (int j = first; j < issued; ++j) {
          const int s = j % C::NS;
          volatile int no_abort = 0;
          WaitCtx w2{dw.limit_ns, dw.status, &no_abort};
          mbar_wait(&bars[C::B_KF + s], (j / C::NS) & 1, w2, 20);
          mbar_wait(&bars[C::B_VF + s], (j / C::NS) & 1, w2, 21);
        }
        volatile int no_abort = 0;
        WaitCtx w2{dw.limit_ns, dw.status, &no_abort};
        mbar_wait(&bars[C::B_Q], 0, w2, 22);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- UMMA issuer
    if (lane == 0) {
      const uint32_t sQ = sbase + C::OFF_Q;
      if (mbar_wait(&bars[C::B_Q], 0, wc, 2)) {
        for (int j = 0; j <= n_kv; ++j) {
          if (j < n_kv) {
            const int s = j % C::NS;
            if (!mbar_wait(&bars[C::B_KF + s], (j / C::NS) & 1, wc, 3)) break;
            tc_fence_after();
            const uint32_t sK = sbase + C::OFF_K + s * C::TILE_BYTES;
            const uint32_t dS = tmem + (uint32_t)((j & 1) * 128);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              umma_ss(dS, desc_kmajor<D>(sQ, kk), desc_kmajor<D>(sK, kk), C::IDESC_S, kk > 0 ? 1u : 0u);
            umma_commit(&bars[C::B_SF + (j & 1)]);
          }
          if (j > 0) {
            const int jj = j - 1, s2 = jj % C::NS;
            if (!mbar_wait(&bars[C::B_PF + (jj & 1)], (jj >> 1) & 1, wc, 4)) break;
            if (!mbar_wait(&bars[C::B_VF + s2], (jj / C::NS) & 1, wc, 5)) break;
            tc_fence_after();
            const uint32_t sV = sbase + C::OFF_V + s2 * C::TILE_BYTES;
            const uint32_t aP = tmem + (uint32_t)((jj & 1) * 128);
#pragma unroll
            for (int kk = 0; kk < C::BN / 16; ++kk)
              umma_ts(tmem + C::TMEM_O, aP + kk * 8, desc_v<D>(sV, kk), C::IDESC_PV,
                      (jj > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&bars[C::B_KVE + s2]);
            umma_commit(&bars[C::B_O]);
          }
        }
      }
      // Every MMA issued so far must complete before TMEM is freed.
      umma_commit(&bars[C::B_DRAIN]);
      volatile int no_abort = 0;
      WaitCtx w2{p.wait_limit_ns, p.status, &no_abort};
      mbar_wait(&bars[C::B_DRAIN], 0, w2, 23);
    }
  } else {
    // ---------------------------------------------------------------- softmax warpgroup
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    const int q_idx = q0 + row;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      if (!warp_wait(&bars[C::B_SF + b], (j >> 1) & 1, wc, 6)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int g = 0; g < 4; ++g) tmem_ld32(t_lane + b * 128 + g * 32, s[g]);
      tmem_wait_ld(s[0]);
      reg_tie(s[1]);
      reg_tie(s[2]);
      reg_tie(s[3]);

      // Mask keys past Nk and (causal) keys after this row's query index.
      const bool need_mask = ((j + 1) * C::BN > p.Nk) || (CAUSAL && (j * C::BN + C::BN - 1 > q0));
      if (need_mask) {
        int lim = p.Nk - 1 - j * C::BN;  // last visible column of this tile
        if (CAUSAL) lim = min(lim, q_idx - j * C::BN);
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (g * 32 + c > lim) s[g][c] = __float_as_uint(-INFINITY);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int c = 0; c < 32; ++c) mx = fmaxf(mx, as_f(s[g][c]));
      const float m_new = fmaxf(m, mx * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m - m_use);
      float sum = 0.f;
      uint32_t pk[2][32];
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float p0 = ex2(fmaf(as_f(s[g][c]), sl2, -m_use));
          const float p1 = ex2(fmaf(as_f(s[g][c + 1]), sl2, -m_use));
          sum += p0 + p1;
          pk[g >> 1][(g & 1) * 16 + (c >> 1)] = pack_bf16(p0, p1);
        }
      l = l * alpha + sum;
      tmem_st32(t_lane + b * 128, pk[0]);
      tmem_st32(t_lane + b * 128 + 32, pk[1]);

      if (j > 0) {
        // PV(j-1) must have landed in O before it is rescaled.
        if (!warp_wait(&bars[C::B_O], (j - 1) & 1, wc, 7)) {
          ok = false;
          tmem_wait_st();
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int g = 0; g < D / 16; ++g) {
            uint32_t o[16];
            tmem_ld16(t_lane + C::TMEM_O + g * 16, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(as_f(o[c]) * alpha);
            tmem_st16(t_lane + C::TMEM_O + g * 16, o);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[C::B_PF + b]);
      m = m_new;
    }
    if (ok && warp_wait(&bars[C::B_O], (n_kv - 1) & 1, wc, 8)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)bh * p.Nq + q_idx) * D;
#pragma unroll
      for (int g = 0; g < D / 16; ++g) {
        uint32_t o[16];
        tmem_ld16(t_lane + C::TMEM_O + g * 16, o);
        tmem_wait_ld(o);
        uint4 w0, w1;
        w0.x = pack_bf16(as_f(o[0]) * inv_l, as_f(o[1]) * inv_l);
        w0.y = pack_bf16(as_f(o[2]) * inv_l, as_f(o[3]) * inv_l);
        w0.z = pack_bf16(as_f(o[4]) * inv_l, as_f(o[5]) * inv_l);
        w0.w = pack_bf16(as_f(o[6]) * inv_l, as_f(o[7]) * inv_l);
        w1.x = pack_bf16(as_f(o[8]) * inv_l, as_f(o[9]) * inv_l);
        w1.y = pack_bf16(as_f(o[10]) * inv_l, as_f(o[11]) * inv_l);
        w1.z = pack_bf16(as_f(o[12]) * inv_l, as_f(o[13]) * inv_l);
        w1.w = pack_bf16(as_f(o[14]) * inv_l, as_f(o[15]) * inv_l);
        if (q_idx < p.Nq) {
          reinterpret_cast<uint4*>(orow + g * 16)[0] = w0;
          reinterpret_cast<uint4*>(orow + g * 16)[1] = w1;
        }
      }
      if (q_idx < p.Nq) p.lse[(size_t)bh * p.Nq + q_idx] = (m + log2f(l)) * 0.69314718055994530942f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                     int BH, cudaStream_t st) {
  using C = Cfg<D>;
  auto kern = fwd_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.n_q_tiles, (unsigned)BH);
  kern<<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

// A kernel whose only job is a bounded wait on an mbarrier that nothing ever
// arrives on: it exercises the timeout path (status word, early return)
// without faulting or hanging the GPU.
__global__ void wait_probe_kernel(unsigned long long limit_ns, unsigned* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{limit_ns, status, &abort_flag};
  warp_wait(&bar, 0, wc, 99);
  __syncthreads();
}

}  // namespace fwd

cudaError_t launch_fwd(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int BH, cudaStream_t st) {
#define TA11_FWD_CASE(DD)                                                        \
  case DD:                                                                       \
    return causal ? fwd::launch_t<DD, true>(tq, tk, tv, p, BH, st)               \
                  : fwd::launch_t<DD, false>(tq, tk, tv, p, BH, st);
  switch (D) {
    TA11_FWD_CASE(16)
    TA11_FWD_CASE(32)
    TA11_FWD_CASE(64)
    TA11_FWD_CASE(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef TA11_FWD_CASE
}

cudaError_t launch_wait_probe(unsigned long long limit_ns, unsigned* status, cudaStream_t st) {
  fwd::wait_probe_kernel<<<1, 32, 0, st>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace ta11
