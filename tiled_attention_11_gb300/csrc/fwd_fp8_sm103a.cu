// FP8 (e4m3) forward of exact attention for sm_103a.
//
// Method: the tiled online-softmax forward of "FlashAttention-2实现与优化：高效注意力机制详解"
// §3.1/§3.2 (see fwd_sm103a.cu), on e4m3 inputs with per-tensor scales, the quantised
// direction named in "FlashAttention技术演进全景图" §5.3 (与量化训练结合, FP8).  Real
// values are descale * e4m3; S = Q K^T accumulates the e4m3 products exactly in fp32 on
// the tensor core (tcgen05 kind::f8f6f4) and the descales of Q and K join the softmax
// scale.  P is rounded to e4m3 for P V (the second fp8 GEMM); V's descale multiplies O.
//
// Precision choices:
//   * p = 2^(S*c - m + 4): the subtracted maximum m is refreshed when a row maximum
//     grows by more than 4 (base 2), so every p <= 2^8 < 448 (the e4m3 maximum) and
//     weights down to 2^-10 of the row maximum keep full e4m3 precision (not subnormal).
//   * O is divided by the sum of the e4m3-rounded weights P V actually used (each
//     32-key group summed in f16x2, exactly converted from e4m3, then in f32): a row
//     dominated by one key returns that key's V row up to bf16 rounding.  L uses the
//     unrounded sum.
//
// Layout: Q, K e4m3 [B*H][N][D] (D innermost); V given transposed, e4m3 [B*H][D][ldv]
// (keys innermost, ldv >= Nk, a multiple of 16), so both GEMMs read K-major shared-memory
// tiles.  O bf16 [B*H][Nq][D], L fp32 [B*H][Nq] (natural log of the scaled logits).
// CTA organisation as the bf16 forward: two 128-row query tiles ping-pong on the tensor
// core; warps 0-3 / 4-7 softmax, warp 8 TMA producer, warp 9 TMEM allocator + UMMA issuer.
// TMEM: S0 | S1 (128 fp32 columns each; P as e4m3 overwrites the first 32) | O0 | O1.
#include "fa_kernels.h"
#include "ptx_sm103a.cuh"

namespace ta11 {
namespace fwd8 {

template <int D>
struct Cfg {
  static constexpr int BM = 128;                       // query rows per tile
  static constexpr int BN = 128;                       // keys per tile
  static constexpr int ROWB = D;                       // bytes per Q / K smem row = swizzle width
  static constexpr int TILE_QK = 128 * D;              // Q or K tile bytes
  static constexpr int TILE_VT = D * 128;              // V^T tile: D rows of 128 keys
  static constexpr int NS = 4;                         // K / V ring depth
  static constexpr uint32_t LAYOUT_QK = umma_layout_for_swizzle(ROWB);
  static constexpr uint32_t LAYOUT_VT = umma_layout_for_swizzle(128);
  static constexpr int TMEM_S = 0;                     // + 128 * tile
  static constexpr int TMEM_O = 256;                   // + D * tile
  static constexpr int TMEM_COLS = 512;
  static constexpr int OFF_Q = 0;                      // 2 tiles
  static constexpr int OFF_K = 2 * TILE_QK;
  static constexpr int OFF_V = OFF_K + NS * TILE_QK;
  static constexpr int OFF_BAR = OFF_V + NS * TILE_VT;
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 2;
  static constexpr int B_VF = 2 + NS;
  static constexpr int B_KE = 2 + 2 * NS;
  static constexpr int B_VE = 2 + 3 * NS;
  static constexpr int B_SF = 2 + 4 * NS;
  static constexpr int B_PF = 4 + 4 * NS;
  static constexpr int B_O = 6 + 4 * NS;
  static constexpr int B_DRAIN = 8 + 4 * NS;
  // persistent kernel only: Q tile t free (the last S MMA of a unit that reads it is done);
  // work-unit ring slots full / empty; the answer of a launch-control request landed
  static constexpr int B_QE = 9 + 4 * NS;
  static constexpr int NU = 4;               // work-unit ring slots
  static constexpr int B_UF = 11 + 4 * NS;
  static constexpr int B_UE = B_UF + NU;
  static constexpr int B_CLC = B_UE + NU;
  static constexpr int NBAR = B_CLC + 1;
  static constexpr int OFF_CLC = OFF_BAR + ((NBAR * 8 + 16 + 15) / 16) * 16;  // 16-byte launch-control answer
  static constexpr int OFF_UNITS = OFF_CLC + 16;                               // NU x int2 work units
  static constexpr int SMEM_USED = OFF_UNITS + NU * 8;
  static constexpr int SMEM_ALLOC = (SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024) + 1024;
  static constexpr int THREADS = 320;
  static constexpr int W_PRODUCER = 8, W_MMA = 9;
  static constexpr uint32_t IDESC_S = idesc_e4m3(128, 128, false, false);
  static constexpr uint32_t IDESC_PV = idesc_e4m3(128, D, false, false);  // B = V^T, K-major
  static_assert(D == 64 || D == 128, "e4m3 rows of 64 or 128 bytes");
  static_assert(TILE_QK % 1024 == 0 && TILE_VT % 1024 == 0, "tiles keep 1024-byte alignment");
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

constexpr float kTau = 4.0f;     // base-2 growth of a row max that forces a rescale
constexpr float kOffset = 4.0f;  // p = 2^(t - m + kOffset): the row maximum maps to >= 16

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, w, site));
}

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

// One S tile (key tile j) of one query row: the masks, the lazily refreshed maximum, the
// weights as e4m3 into P's TMEM columns, the sums l and lr, and the rescale of O.
template <int D, bool CAUSAL>
__device__ __forceinline__ void softmax_tile(uint32_t t_s, uint32_t t_o, int j, int qt0, int q_idx, int Nk, float sl2,
                                             float& m, float& l, float& lr) {
  using C = Cfg<D>;
  uint32_t s[4][32];
#pragma unroll
  for (int g = 0; g < 4; ++g) tmem_ld32(t_s + g * 32, s[g]);
  tmem_wait_ld(s[0]);
  reg_tie(s[1]);
  reg_tie(s[2]);
  reg_tie(s[3]);

  // Mask keys past Nk and (causal) keys after this row's query index.
  const bool need_mask = ((j + 1) * C::BN > Nk) || (CAUSAL && (j * C::BN + C::BN - 1 > qt0));
  if (need_mask) {
    int lim = Nk - 1 - j * C::BN;  // last visible column of this tile
    if (CAUSAL) lim = min(lim, q_idx - j * C::BN);
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (g * 32 + c > lim) s[g][c] = __float_as_uint(-INFINITY);
  }
  float mx8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t* v = &s[i >> 1][(i & 1) * 16];
    float a = fmax3(as_f(v[0]), as_f(v[1]), as_f(v[2]));
#pragma unroll
    for (int e = 3; e < 15; e += 2) a = fmax3(a, as_f(v[e]), as_f(v[e + 1]));
    mx8[i] = fmaxf(a, as_f(v[15]));
  }
  const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
  const float mx2 = mx * sl2;
  float alpha = 1.f;
  if (mx2 > m + kTau) {  // also taken on the first tile, where m = -inf
    alpha = ex2(m - mx2);
    m = mx2;
  }
  // p = 2^(S*c - m + 4), four at a time into one word of e4m3; l sums p, lr the rounded p
  const uint64_t c2 = f2pack(sl2, sl2), nm2 = f2pack(kOffset - m, kOffset - m);
  uint64_t l2[2] = {0ull, 0ull};
  uint32_t pk[32];
  float lr_t = 0.f;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t h[8];  // f16x2 partial sums of the rounded weights of this 32-key group
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      float x0, x1, x2, x3;
      f2unpack(ffma2(f2pack(as_f(s[g][4 * w]), as_f(s[g][4 * w + 1])), c2, nm2), x0, x1);
      f2unpack(ffma2(f2pack(as_f(s[g][4 * w + 2]), as_f(s[g][4 * w + 3])), c2, nm2), x2, x3);
      const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
      l2[0] = fadd2(l2[0], f2pack(p0, p1));
      l2[1] = fadd2(l2[1], f2pack(p2, p3));
      const uint32_t word = pack_e4m3x4(p0, p1, p2, p3);
      pk[g * 8 + w] = word;
      uint32_t lo, hi;
      e4m3x4_to_f16x2(word, lo, hi);
      h[w] = hadd2(lo, hi);
    }
    const uint32_t h4 = hadd2(hadd2(hadd2(h[0], h[1]), hadd2(h[2], h[3])), hadd2(hadd2(h[4], h[5]), hadd2(h[6], h[7])));
    lr_t += f16x2_sum_f32(h4);
  }
  tmem_st32(t_s, pk);
  float la, lb, lc, ld;
  f2unpack(l2[0], la, lb);
  f2unpack(l2[1], lc, ld);
  l = l * alpha + ((la + lb) + (lc + ld));
  lr = lr * alpha + lr_t;

  // O holds P V up to tile j-1 (S_t(j) was issued after PV_t(j-1), so it has landed);
  // rescale the rows whose subtracted max moved.
  if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
    for (int g = 0; g < D / 16; ++g) {
      uint32_t o[16];
      tmem_ld16(t_o + g * 16, o);
      tmem_wait_ld(o);
#pragma unroll
      for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(as_f(o[c]) * alpha);
      tmem_st16(t_o + g * 16, o);
    }
  }
  tmem_wait_st();
}

// O row (TMEM columns from t_o) times mul, as bf16, to orow when valid.
template <int D>
__device__ __forceinline__ void store_o_row(uint32_t t_o, __nv_bfloat16* orow, bool valid, float mul) {
#pragma unroll
  for (int g = 0; g < D / 16; ++g) {
    uint32_t o[16];
    tmem_ld16(t_o + g * 16, o);
    tmem_wait_ld(o);
    if (valid) store16_bf16(orow + g * 16, o, mul);
  }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_vt, const Fp8FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = (int)warp_id(), lane = (int)lane_id();
  // heaviest (causal) query-tile pairs of a head first; pairs of one head adjacent
  const int pair = (int)gridDim.x - 1 - (int)blockIdx.x;
  const int bh = blockIdx.y;
  const int q0 = pair * 2 * C::BM;
  const int nk_tiles = (p.Nk + C::BN - 1) / C::BN;
  const int n_kv0 = CAUSAL ? min(nk_tiles, 2 * pair + 1) : nk_tiles;
  const int n_kv1 = CAUSAL ? min(nk_tiles, 2 * pair + 2) : nk_tiles;
  const WaitCtx wc{p.wait_limit_ns, p.status, abort_flag};

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars[C::B_Q + t], 1);
      mbar_init(&bars[C::B_SF + t], 1);
      mbar_init(&bars[C::B_PF + t], 128);
      mbar_init(&bars[C::B_O + t], 1);
    }
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bars[C::B_KF + s], 1);
      mbar_init(&bars[C::B_VF + s], 1);
      mbar_init(&bars[C::B_KE + s], 1);
      mbar_init(&bars[C::B_VE + s], 1);
    }
    mbar_init(&bars[C::B_DRAIN], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::W_MMA) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::W_PRODUCER) {
    // ---------------------------------------------------------------- TMA producer
    {
      if (lane == 0) tma_prefetch_desc(&tm_q);
      if (lane == 0) tma_prefetch_desc(&tm_k);
      if (lane == 0) tma_prefetch_desc(&tm_vt);
      for (int t = 0; t < 2; ++t) {
        mbar_arrive_expect_tx_w(&bars[C::B_Q + t], C::TILE_QK);
        tma_load_3d_w(smem + C::OFF_Q + t * C::TILE_QK, &tm_q, &bars[C::B_Q + t], 0, q0 + t * C::BM, bh);
      }
      int k_issued = 0, v_issued = 0;  // K and V tiles whose copies were started
      for (int j = 0; j < n_kv1; ++j) {
        const int s = j % C::NS;
        if (j >= C::NS && !mbar_wait_w(&bars[C::B_KE + s], ((j / C::NS) - 1) & 1, wc, 1)) break;
        mbar_arrive_expect_tx_w(&bars[C::B_KF + s], C::TILE_QK);
        tma_load_3d_w(smem + C::OFF_K + s * C::TILE_QK, &tm_k, &bars[C::B_KF + s], 0, j * C::BN, bh);
        k_issued = j + 1;
        if (j >= C::NS && !mbar_wait_w(&bars[C::B_VE + s], ((j / C::NS) - 1) & 1, wc, 1)) break;
        mbar_arrive_expect_tx_w(&bars[C::B_VF + s], C::TILE_VT);
        tma_load_3d_w(smem + C::OFF_V + s * C::TILE_VT, &tm_vt, &bars[C::B_VF + s], j * C::BN, 0, bh);
        v_issued = j + 1;
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        // Let every copy already started land before the CTA can exit: the last NS of
        // each ring, one per slot, so that each wait is on its slot's newest phase.
        volatile int no_abort = 0;
        const WaitCtx w2{p.wait_limit_ns, p.status, &no_abort};
        for (int j = k_issued > C::NS ? k_issued - C::NS : 0; j < k_issued; ++j)
          mbar_wait(&bars[C::B_KF + j % C::NS], (j / C::NS) & 1, w2, 20);
        for (int j = v_issued > C::NS ? v_issued - C::NS : 0; j < v_issued; ++j)
          mbar_wait(&bars[C::B_VF + j % C::NS], (j / C::NS) & 1, w2, 21);
        mbar_wait(&bars[C::B_Q], 0, w2, 22);
        mbar_wait(&bars[C::B_Q + 1], 0, w2, 22);
      }
    }
  } else if (warp == C::W_MMA) {
    // ---------------------------------------------------------------- UMMA issuer
    {
      // K-major descriptors for Q, the K ring and the V^T ring; a 32-byte K slice is a
      // 32-byte step inside the swizzled row.
      const uint64_t dq0 = sdesc(sbase + C::OFF_Q, 16, 8 * C::ROWB, C::LAYOUT_QK);
      const uint64_t dk0 = sdesc(sbase + C::OFF_K, 16, 8 * C::ROWB, C::LAYOUT_QK);
      const uint64_t dv0 = sdesc(sbase + C::OFF_V, 16, 8 * 128, C::LAYOUT_VT);
      auto issue_s = [&](int t, int slot) {  // S_t = Q_t K^T
        const uint64_t dq = desc_adv(dq0, (uint32_t)(t * C::TILE_QK));
        const uint64_t dk = desc_adv(dk0, (uint32_t)(slot * C::TILE_QK));
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)
          umma_ss_f8_w(tmem + C::TMEM_S + t * 128, desc_adv(dq, (uint32_t)(kk * 32)), desc_adv(dk, (uint32_t)(kk * 32)),
                     C::IDESC_S, kk > 0 ? 1u : 0u);
        umma_commit_w(&bars[C::B_SF + t]);
      };
      auto issue_pv = [&](int t, int slot, bool acc) {  // O_t (+)= P_t V  (A = P in TMEM, 4 per column)
        const uint64_t dv = desc_adv(dv0, (uint32_t)(slot * C::TILE_VT));
#pragma unroll
        for (int kk = 0; kk < C::BN / 32; ++kk)
          umma_ts_f8_w(tmem + C::TMEM_O + t * D, tmem + C::TMEM_S + t * 128 + kk * 8, desc_adv(dv, (uint32_t)(kk * 32)),
                     C::IDESC_PV, (acc || kk > 0) ? 1u : 0u);
        umma_commit_w(&bars[C::B_O + t]);
      };
      bool ok = mbar_wait_w(&bars[C::B_Q], 0, wc, 2) && mbar_wait_w(&bars[C::B_KF], 0, wc, 3);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        if ((ok = mbar_wait_w(&bars[C::B_Q + 1], 0, wc, 2))) {
          tc_fence_after();
          issue_s(1, 0);
          umma_commit_w(&bars[C::B_KE]);
        }
      }
      for (int j = 0; ok && j < n_kv1; ++j) {
        const int s = j % C::NS, s1 = (j + 1) % C::NS;
        if (!(ok = mbar_wait_w(&bars[C::B_VF + s], (j / C::NS) & 1, wc, 5))) break;
        const bool next_k = j + 1 < n_kv1;
        if (next_k && !(ok = mbar_wait_w(&bars[C::B_KF + s1], ((j + 1) / C::NS) & 1, wc, 3))) break;
        if (j < n_kv0) {
          if (!(ok = mbar_wait_w(&bars[C::B_PF], j & 1, wc, 4))) break;
          tc_fence_after();
          issue_pv(0, s, j > 0);
          if (j + 1 < n_kv0) issue_s(0, s1);
        }
        if (!(ok = mbar_wait_w(&bars[C::B_PF + 1], j & 1, wc, 4))) break;
        tc_fence_after();
        issue_pv(1, s, j > 0);
        umma_commit_w(&bars[C::B_VE + s]);
        if (next_k) {
          issue_s(1, s1);
          umma_commit_w(&bars[C::B_KE + s1]);
        }
      }
      // Every MMA issued so far must complete before TMEM is freed.
      umma_commit_w(&bars[C::B_DRAIN]);
      volatile int no_abort = 0;
      const WaitCtx w2{p.wait_limit_ns, p.status, &no_abort};
      mbar_wait(&bars[C::B_DRAIN], 0, w2, 23);
    }
  } else {
    // ---------------------------------------------------------------- softmax warpgroups
    const int t = warp >> 2;   // which query tile of the pair
    const int wq = warp & 3;   // TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    const int qt0 = q0 + t * C::BM;
    const int q_idx = qt0 + row;
    const int n_kv = t == 0 ? n_kv0 : n_kv1;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t t_s = t_lane + C::TMEM_S + t * 128;
    const uint32_t t_o = t_lane + C::TMEM_O + t * D;
    // the descales of Q and K join the softmax scale; V's multiplies O
    const float sl2 = p.scale_log2 * __ldg(p.q_descale) * __ldg(p.k_descale);
    const float v_descale = __ldg(p.v_descale);
    float m = -INFINITY, l = 0.f, lr = 0.f;  // m: max subtracted (base 2); l, lr: sums of p, e4m3(p)
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!warp_wait(&bars[C::B_SF + t], j & 1, wc, 6)) {
        ok = false;
        break;
      }
      tc_fence_after();
      softmax_tile<D, CAUSAL>(t_s, t_o, j, qt0, q_idx, p.Nk, sl2, m, l, lr);
      tc_fence_before();
      mbar_arrive(&bars[C::B_PF + t]);
    }
    if (ok && warp_wait(&bars[C::B_O + t], (n_kv - 1) & 1, wc, 8)) {
      tc_fence_after();
      store_o_row<D>(t_o, reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)bh * p.Nq + q_idx) * D, q_idx < p.Nq,
                     v_descale / lr);
      if (q_idx < p.Nq) p.lse[(size_t)bh * p.Nq + q_idx] = (m - kOffset + log2f(l)) * 0.69314718055994530942f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Persistent form of fwd_fp8_kernel (the bf16 forward's persistent kernel, on e4m3
// operands): the grid keeps one CTA per (query-tile pair, batch*head) in the same order,
// but a running CTA takes over the next CTA that has not started (cluster launch control)
// and its pipelines run on across units: Q tiles are reloaded once the unit's last S MMA
// reading them is done, ring positions and barrier phases count over all units, and the
// next unit's first S tiles are computed while the softmax warpgroups finish the current
// unit's epilogue.  Per-row arithmetic and key order are those of fwd_fp8_kernel.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    fwd_fp8_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_vt, const Fp8FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  void* clc_resp = smem + C::OFF_CLC;
  int2* units = reinterpret_cast<int2*>(smem + C::OFF_UNITS);

  const int warp = (int)warp_id(), lane = (int)lane_id();
  const int nk_tiles = (p.Nk + C::BN - 1) / C::BN;
  // key tiles of query tile t of pair `pair` (heaviest pairs of a head first: pair =
  // gridDim.x - 1 - x)
  auto n_keys = [&](int pair, int t) { return CAUSAL ? min(nk_tiles, 2 * pair + 1 + t) : nk_tiles; };
  // a published unit is a CTA index (x, y); lpt maps it to (pair rank, head), rank-major
  // within groups of p.lpt heads (all heads when p.lpt >= H)
  auto unit_map = [&](int2 u, int& rank, int& head) {
    rank = u.x;
    head = u.y;
    if (p.lpt) {
      const int gx = (int)gridDim.x, nh = (int)gridDim.y, gs0 = min(p.lpt, nh);
      const int lin = u.y * gx + u.x;
      const int grp = lin / (gs0 * gx), h0 = grp * gs0, gs = min(gs0, nh - h0);
      const int idx = lin - h0 * gx;
      rank = idx / gs;
      head = h0 + idx % gs;
    }
  };
  auto unit_rank = [&](int2 u) { int r, h; unit_map(u, r, h); return r; };
  auto unit_head = [&](int2 u) { int r, h; unit_map(u, r, h); return h; };
  const WaitCtx wc{p.wait_limit_ns, p.status, abort_flag};

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars[C::B_Q + t], 1);
      mbar_init(&bars[C::B_SF + t], 1);
      mbar_init(&bars[C::B_PF + t], 128);
      mbar_init(&bars[C::B_O + t], 1);
      mbar_init(&bars[C::B_QE + t], 1);
    }
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bars[C::B_KF + s], 1);
      mbar_init(&bars[C::B_VF + s], 1);
      mbar_init(&bars[C::B_KE + s], 1);
      mbar_init(&bars[C::B_VE + s], 1);
    }
    for (int u = 0; u < C::NU; ++u) {
      mbar_init(&bars[C::B_UF + u], 1);
      mbar_init(&bars[C::B_UE + u], 9);  // the issuing warp and one lane of each softmax warp
    }
    mbar_init(&bars[C::B_DRAIN], 1);
    mbar_init(&bars[C::B_CLC], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::W_MMA) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::W_PRODUCER) {
    // ---------------------------------------------------------------- scheduler + TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
    }
    int ux = (int)blockIdx.x, uy = (int)blockIdx.y;  // the unit to publish next (ux < 0: none)
    int jg = 0, k_issued = 0, v_issued = 0, q_units = 0;  // copies started (ring positions, Q pairs)
    bool asked = false;
    int n_asked = 0;
    for (int i = 0;; ++i) {
      const int us = i % C::NU;
      if (i >= C::NU && !mbar_wait_w(&bars[C::B_UE + us], ((i / C::NU) - 1) & 1, wc, 10)) break;
      units[us] = make_int2(ux, uy);
      mbar_arrive_w(&bars[C::B_UF + us]);
      if (ux < 0) break;
      // lpt: longest-first (rank-major) over all heads for causal launches of a few waves,
      // within groups of heads beyond
      int pr, bh;
      unit_map(make_int2(ux, uy), pr, bh);
      const int pair = (int)gridDim.x - 1 - pr, q0 = pair * 2 * C::BM;
      const int n_kv = n_keys(pair, 1);  // tile 1's walk contains tile 0's
      bool ok = true;
      for (int t = 0; t < 2 && ok; ++t) {  // Q_t is free once the last S MMA reading it is done
        if (i >= 1 && !(ok = mbar_wait_w(&bars[C::B_QE + t], (i - 1) & 1, wc, 11))) break;
        mbar_arrive_expect_tx_w(&bars[C::B_Q + t], C::TILE_QK);
        tma_load_3d_w(smem + C::OFF_Q + t * C::TILE_QK, &tm_q, &bars[C::B_Q + t], 0, q0 + t * C::BM, bh);
      }
      if (!ok) break;
      q_units = i + 1;
      for (int j = 0; j < n_kv && ok; ++j, ++jg) {
        const int s = jg % C::NS;
        if (jg >= C::NS && !(ok = mbar_wait_w(&bars[C::B_KE + s], ((jg / C::NS) - 1) & 1, wc, 1))) break;
        mbar_arrive_expect_tx_w(&bars[C::B_KF + s], C::TILE_QK);
        tma_load_3d_w(smem + C::OFF_K + s * C::TILE_QK, &tm_k, &bars[C::B_KF + s], 0, j * C::BN, bh);
        k_issued = jg + 1;
        if (jg >= C::NS && !(ok = mbar_wait_w(&bars[C::B_VE + s], ((jg / C::NS) - 1) & 1, wc, 1))) break;
        mbar_arrive_expect_tx_w(&bars[C::B_VF + s], C::TILE_VT);
        tma_load_3d_w(smem + C::OFF_V + s * C::TILE_VT, &tm_vt, &bars[C::B_VF + s], j * C::BN, 0, bh);
        v_issued = jg + 1;
      }
      if (!ok) break;
      // the next unit, asked for once this unit's last copies are started
      mbar_arrive_expect_tx_w(&bars[C::B_CLC], 16);
      clc_try_cancel_w(clc_resp, &bars[C::B_CLC]);
      asked = true;
      if (!mbar_wait_w(&bars[C::B_CLC], n_asked & 1, wc, 12)) break;
      asked = false;
      ++n_asked;
      int cx, cy;
      const bool taken = clc_taken(clc_resp, cx, cy);
      ux = (taken && cx >= 0 && cx < (int)gridDim.x && cy >= 0 && cy < (int)gridDim.y) ? cx : -1;
      uy = cy;
    }
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      // every copy already started lands before the CTA can exit: the newest phase of each
      // ring slot, the last Q pair and a pending launch-control answer
      volatile int no_abort = 0;
      const WaitCtx w2{p.wait_limit_ns, p.status, &no_abort};
      for (int j = k_issued > C::NS ? k_issued - C::NS : 0; j < k_issued; ++j)
        mbar_wait(&bars[C::B_KF + j % C::NS], (j / C::NS) & 1, w2, 20);
      for (int j = v_issued > C::NS ? v_issued - C::NS : 0; j < v_issued; ++j)
        mbar_wait(&bars[C::B_VF + j % C::NS], (j / C::NS) & 1, w2, 21);
      if (q_units > 0)
        for (int t = 0; t < 2; ++t) mbar_wait(&bars[C::B_Q + t], (q_units - 1) & 1, w2, 22);
      if (asked) mbar_wait(&bars[C::B_CLC], n_asked & 1, w2, 24);
    }
  } else if (warp == C::W_MMA) {
    // ---------------------------------------------------------------- UMMA issuer
    const uint64_t dq0 = sdesc(sbase + C::OFF_Q, 16, 8 * C::ROWB, C::LAYOUT_QK);
    const uint64_t dk0 = sdesc(sbase + C::OFF_K, 16, 8 * C::ROWB, C::LAYOUT_QK);
    const uint64_t dv0 = sdesc(sbase + C::OFF_V, 16, 8 * 128, C::LAYOUT_VT);
    auto issue_s = [&](int t, int slot) {  // S_t = Q_t K^T
      const uint64_t dq = desc_adv(dq0, (uint32_t)(t * C::TILE_QK));
      const uint64_t dk = desc_adv(dk0, (uint32_t)(slot * C::TILE_QK));
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk)
        umma_ss_f8_w(tmem + C::TMEM_S + t * 128, desc_adv(dq, (uint32_t)(kk * 32)), desc_adv(dk, (uint32_t)(kk * 32)),
                     C::IDESC_S, kk > 0 ? 1u : 0u);
      umma_commit_w(&bars[C::B_SF + t]);
    };
    auto issue_pv = [&](int t, int slot, bool acc) {  // O_t (+)= P_t V  (A = P in TMEM, 4 per column)
      const uint64_t dv = desc_adv(dv0, (uint32_t)(slot * C::TILE_VT));
#pragma unroll
      for (int kk = 0; kk < C::BN / 32; ++kk)
        umma_ts_f8_w(tmem + C::TMEM_O + t * D, tmem + C::TMEM_S + t * 128 + kk * 8, desc_adv(dv, (uint32_t)(kk * 32)),
                     C::IDESC_PV, (acc || kk > 0) ? 1u : 0u);
      umma_commit_w(&bars[C::B_O + t]);
    };
    int jg = 0;                // ring position of the unit's first key tile
    int npf[2] = {0, 0};       // P tiles consumed per query tile (phases of p_full)
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int us = i % C::NU;
      if (!(ok = mbar_wait_w(&bars[C::B_UF + us], (i / C::NU) & 1, wc, 13))) break;
      const int2 u = units[us];
      mbar_arrive_w(&bars[C::B_UE + us]);
      if (u.x < 0) break;
      const int pair = (int)gridDim.x - 1 - unit_rank(u);
      const int n_kv0 = n_keys(pair, 0), n_kv1 = n_keys(pair, 1);
      // the unit's first S tiles (their TMEM columns were last read by the previous unit's
      // P V, issued earlier by this warp)
      ok = mbar_wait_w(&bars[C::B_Q], i & 1, wc, 2) && mbar_wait_w(&bars[C::B_KF + jg % C::NS], (jg / C::NS) & 1, wc, 3);
      if (!ok) break;
      tc_fence_after();
      issue_s(0, jg % C::NS);
      if (n_kv0 == 1) umma_commit_w(&bars[C::B_QE]);
      if (!(ok = mbar_wait_w(&bars[C::B_Q + 1], i & 1, wc, 2))) break;
      tc_fence_after();
      issue_s(1, jg % C::NS);
      if (n_kv1 == 1) umma_commit_w(&bars[C::B_QE + 1]);
      umma_commit_w(&bars[C::B_KE + jg % C::NS]);
      for (int j = 0; ok && j < n_kv1; ++j) {
        const int pos = jg + j, s = pos % C::NS, s1 = (pos + 1) % C::NS;
        if (!(ok = mbar_wait_w(&bars[C::B_VF + s], (pos / C::NS) & 1, wc, 5))) break;
        const bool next_k = j + 1 < n_kv1;
        if (next_k && !(ok = mbar_wait_w(&bars[C::B_KF + s1], ((pos + 1) / C::NS) & 1, wc, 3))) break;
        if (j < n_kv0) {
          if (!(ok = mbar_wait_w(&bars[C::B_PF], npf[0] & 1, wc, 4))) break;
          ++npf[0];
          tc_fence_after();
          issue_pv(0, s, j > 0);
          if (j + 1 < n_kv0) {
            issue_s(0, s1);
            if (j + 2 == n_kv0) umma_commit_w(&bars[C::B_QE]);
          }
        }
        if (!(ok = mbar_wait_w(&bars[C::B_PF + 1], npf[1] & 1, wc, 4))) break;
        ++npf[1];
        tc_fence_after();
        issue_pv(1, s, j > 0);
        umma_commit_w(&bars[C::B_VE + s]);
        if (next_k) {
          issue_s(1, s1);
          if (j + 2 == n_kv1) umma_commit_w(&bars[C::B_QE + 1]);
          umma_commit_w(&bars[C::B_KE + s1]);
        }
      }
      jg += n_kv1;
    }
    // Every MMA issued so far must complete before TMEM is freed.
    umma_commit_w(&bars[C::B_DRAIN]);
    volatile int no_abort = 0;
    const WaitCtx w2{p.wait_limit_ns, p.status, &no_abort};
    mbar_wait(&bars[C::B_DRAIN], 0, w2, 23);
  } else {
    // ---------------------------------------------------------------- softmax warpgroups
    const int t = warp >> 2;   // which query tile of the pair
    const int wq = warp & 3;   // TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t t_s = t_lane + C::TMEM_S + t * 128;
    const uint32_t t_o = t_lane + C::TMEM_O + t * D;
    const float sl2 = p.scale_log2 * __ldg(p.q_descale) * __ldg(p.k_descale);
    const float v_descale = __ldg(p.v_descale);
    int ns = 0;  // S tiles of this query tile processed over all units (phases of s_full, o_done)
    bool ok = true;
    for (int i = 0;; ++i) {
      // the four warps agree to go on (a failed wait anywhere stops all of them together)
      const int us = i % C::NU;
      if (!named_bar_and(1 + t, 128, ok && warp_wait(&bars[C::B_UF + us], (i / C::NU) & 1, wc, 14))) break;
      const int2 u = units[us];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::B_UE + us]);
      if (u.x < 0) break;
      const int pair = (int)gridDim.x - 1 - unit_rank(u), bh = unit_head(u);
      const int qt0 = pair * 2 * C::BM + t * C::BM;
      const int q_idx = qt0 + row;
      const int n_kv = n_keys(pair, t);
      float m = -INFINITY, l = 0.f, lr = 0.f;
      for (int j = 0; j < n_kv; ++j, ++ns) {
        if (!warp_wait(&bars[C::B_SF + t], ns & 1, wc, 6)) {
          ok = false;
          break;
        }
        tc_fence_after();
        softmax_tile<D, CAUSAL>(t_s, t_o, j, qt0, q_idx, p.Nk, sl2, m, l, lr);
        tc_fence_before();
        mbar_arrive(&bars[C::B_PF + t]);
      }
      // epilogue; the next unit's P V overwrites O only after this tile's next P is ready
      const bool go = named_bar_and(1 + t, 128, ok && warp_wait(&bars[C::B_O + t], (ns - 1) & 1, wc, 8));
      if (go) {
        tc_fence_after();
        store_o_row<D>(t_o, reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)bh * p.Nq + q_idx) * D, q_idx < p.Nq,
                       v_descale / lr);
        if (q_idx < p.Nq) p.lse[(size_t)bh * p.Nq + q_idx] = (m - kOffset + log2f(l)) * 0.69314718055994530942f;
      }
      ok = ok && go;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt, const Fp8FwdParams& p,
                     int BH, cudaStream_t st) {
  using C = Cfg<D>;
  auto kern = p.persist ? fwd_fp8_persist_kernel<D, CAUSAL> : fwd_fp8_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((p.Nq + 2 * C::BM - 1) / (2 * C::BM)), (unsigned)BH);
  kern<<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(tq, tk, tvt, p);
  return cudaGetLastError();
}

}  // namespace fwd8

cudaError_t launch_fwd_fp8(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const Fp8FwdParams& p, int BH, cudaStream_t st) {
  switch (D) {
    case 64:
      return causal ? fwd8::launch_t<64, true>(tq, tk, tvt, p, BH, st) : fwd8::launch_t<64, false>(tq, tk, tvt, p, BH, st);
    case 128:
      return causal ? fwd8::launch_t<128, true>(tq, tk, tvt, p, BH, st)
                    : fwd8::launch_t<128, false>(tq, tk, tvt, p, BH, st);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace ta11
