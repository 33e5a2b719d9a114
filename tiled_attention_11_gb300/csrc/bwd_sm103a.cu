// Backward pass of exact attention for sm_103a: recompute P from the saved row
// logsumexp instead of storing it ("解释FlashAttention的显存优化原理" §2(2) 重计算;
// "FlashAttention技术演进全景图" §2.2 重计算机制; the forward saves (L, q, k, v, o),
// "FlashAttention-2实现与优化：高效注意力机制详解" §3.1).  The gradient formulas are the
// softmax Jacobian:  dV = P^T dO,  dP = dO V^T,  Dlt_i = rowsum(dO o O)_i,
// dS = P o (dP - Dlt),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Three kernels, in stream order:
//   prep     Dlt = rowsum(dO o O) (fp32), lse2 = L*log2(e) (+inf on padded rows),
//            dq_accum = 0.                                          (HBM-bound)
//   bwd      one CTA per (batch*head, 128-key tile); K_j, V_j stay in shared memory,
//            dK_j, dV_j accumulate in TMEM; 64-query tiles Q_i, dO_i stream through
//            a 3-stage TMA ring (causal: starting at the diagonal).  Per query tile, all on
//            tcgen05 (keys on the M=128 axis):
//              S^T  = K Q_i^T            -> TMEM   P^T = 2^(S^T c - lse2)  (compute WGs)
//              dP^T = V dO_i^T           -> TMEM   dS^T = P^T o (dP^T - Dlt) -> shared memory
//              dV  += P^T dO_i   (A = P^T from TMEM)
//              dK  += dS^T Q_i   (A = dS^T from shared memory)
//              dQ_i^T = K^T dS^T (A = K^T kept in TMEM, B = the same dS^T tile)
//                                   -> TMEM, into the S^T buffer dV has just consumed
//            Two warps issue the UMMAs: one the score GEMMs S^T, dP^T (which need only
//            loaded tiles and free TMEM), the other the gradient GEMMs dV, dQ^T, dK
//            (which wait for the compute warps).  The tensor core keeps almost no queue,
//            so a single issuing thread lets it run dry at every wait (~200 cycles each,
//            measured); with two, one feeds it while the other waits.  S^T / P^T is
//            double-buffered in TMEM so S(i+1) need not wait for dV(i); dQ_i^T reuses
//            step i's buffer, and S(i+2) waits until the dQ warpgroup has moved dQ_i^T
//            from TMEM to shared memory and added it into dq_accum (TMA bulk reduce-adds
//            of two 32-query halves, so the reduce reading one half overlaps the writes of
//            the other).  Shared-memory bandwidth is the limit (~270 KB per step against
//            128 B/cycle), which is why K^T is kept in TMEM.
//   convert  dq = bf16(dq_accum * scale).
#include "fa_kernels.h"
#include "ptx_sm103a.cuh"

namespace ta11 {
namespace bwd {

template <int D>
struct Cfg {
  static constexpr int BN = 128;                       // keys per CTA (UMMA M)
  static constexpr int BM = 64;                        // queries per inner step (UMMA N)
  static constexpr int CHUNK = D < 64 ? D : 64;
  static constexpr int NCHUNK = D / CHUNK;
  static constexpr int ROWB = CHUNK * 2;
  static constexpr uint32_t LAYOUT = umma_layout_for_swizzle(ROWB);
  static constexpr int K_CHUNK_BYTES = BN * ROWB;
  static constexpr int KV_TILE = BN * D * 2;
  static constexpr int Q_CHUNK_BYTES = BM * ROWB;
  static constexpr int Q_TILE = BM * D * 2;
  static constexpr int NS = D <= 64 ? 4 : 3;           // Q / dO / lse2 / Dlt ring depth
  // S^T / P^T / dQ^T TMEM buffers and dS^T shared-memory buffers: two at D = 128 (TMEM is
  // full), four at D <= 64, where the smaller accumulators leave room for two more and the
  // per-step chain (S^T -> P -> dS^T -> dQ^T -> drain -> S^T of the step NB later) spans
  // more steps (three measured 11-16% faster than two, four another 1%).  The
  // one-CTA-per-unit kernel uses the first two.
  static constexpr int NB = D <= 64 ? 4 : 2;
  static constexpr int DS_BYTES = BN * BM * 2;         // dS^T tile, bf16, 128-byte rows
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KV_TILE;
  static constexpr int OFF_Q = 2 * KV_TILE;
  static constexpr int OFF_DO = OFF_Q + NS * Q_TILE;
  static constexpr int OFF_DS = OFF_DO + NS * Q_TILE;
  static constexpr int OFF_LSE = OFF_DS + NB * DS_BYTES;
  static constexpr int OFF_DLT = OFF_LSE + NS * BM * 4;
  static constexpr int OFF_STG = OFF_DLT + NS * BM * 4;  // dQ_i staging, fp32 [BM][D]
  static constexpr int STG_BYTES = BM * D * 4;
  static constexpr int OFF_BAR = OFF_STG + STG_BYTES;
  // barriers ([2]: one per S^T/P^T TMEM buffer or dS^T smem buffer, where one side can
  // run two phases ahead of the other)
  static constexpr int B_KV = 0;
  static constexpr int B_QF = 1;             // [NS] Q, dO, lse2, Dlt stage loaded
  static constexpr int B_QE = 1 + NS;        // [NS] stage free (dK, its last reader, done)
  static constexpr int B_SF = 1 + 2 * NS;    // [NB] S^T in TMEM buffer b
  static constexpr int B_DPF = B_SF + NB;    // dP^T in TMEM
  static constexpr int B_PF = B_DPF + 1;     // [NB] P^T in TMEM buffer b (compute warps)
  // [2] dS^T in shared memory buffer b (compute warps).  One per buffer: dP^T(i+1) waits only
  // for the compute warps to have loaded dP^T(i), so they can publish dS^T(i) and dS^T(i+1)
  // before issuer B waits for dS^T(i); dS^T(i+2) needs dQ^T(i), which B issues after that wait.
  static constexpr int B_DSF = B_PF + NB;
  static constexpr int B_DQF = B_DSF + NB;   // [NB] dQ^T and dK MMAs of a step done: its dS^T smem buffer is free
  static constexpr int B_DQR = B_DQF + NB;   // [NB] dQ^T in TMEM buffer b, ready for the dQ warpgroup
  static constexpr int B_DQE = B_DQR + NB;   // [NB] dQ^T drained from TMEM buffer b (buffer free)
  static constexpr int B_KT = B_DQE + NB;    // K^T written into TMEM
  static constexpr int B_DPE = B_KT + 1;     // dP^T loaded by the compute warps (its TMEM columns free)
  static constexpr int B_DRAIN = B_DPE + 1;  // [2] one per issuing thread
  // persistent kernel only: K / V smem free (a unit's last S^T, dP^T done); K^T TMEM free (its
  // last dQ^T done); dK, dV drained from TMEM by the epilogue; work-unit ring full / empty;
  // the answer of a launch-control request landed
  static constexpr int B_KVE = B_DRAIN + 2;
  static constexpr int B_KTE = B_KVE + 1;
  static constexpr int B_ACCE = B_KTE + 1;
  static constexpr int NU = 4;               // work-unit ring slots
  static constexpr int B_UF = B_ACCE + 1;
  static constexpr int B_UE = B_UF + NU;
  static constexpr int B_CLC = B_UE + NU;
  static constexpr int NBAR = B_CLC + 1;
  static constexpr int OFF_CLC = OFF_BAR + ((NBAR * 8 + 16 + 15) / 16) * 16;  // 16-byte launch-control answer
  static constexpr int OFF_UNITS = OFF_CLC + 16;                               // NU x 32-byte work units
  static constexpr int SMEM_USED = OFF_UNITS + NU * 32;
  static constexpr int SMEM_ALLOC = (SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024) + 1024;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  // warps 0-3: dQ warpgroup, 4-11: two compute warpgroups, 12: TMA producer,
  // 13: UMMA issuer for S^T, dP^T (and TMEM allocator), 14: UMMA issuer for dV, dK, dQ^T
  static constexpr int THREADS = 480;
  static constexpr int W_PRODUCER = 12, W_MMA_A = 13, W_MMA_B = 14;
  // TMEM columns: S^T/P^T/dQ^T buffers 0 .. NB-1 | dP^T | K^T (bf16 pairs) | dV | dK
  static constexpr int T_S = 0, T_DP = NB * 64, T_KT = T_DP + 64, T_DV = T_KT + 64, T_DK = T_DV + D;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_S = idesc_bf16(128, BM, false, false);   // S^T, dP^T
  static constexpr uint32_t IDESC_KV = idesc_bf16(128, D, false, true);    // dV, dK (B MN-major)
  static constexpr uint32_t IDESC_DQ = idesc_bf16(128, BM, false, true);   // dQ^T (A = K^T in TMEM, B MN-major)
  static constexpr uint32_t IDESC_DQ2 = idesc_bf16(128, 2 * BM, false, true);  // dQ^T of two steps at once
  static_assert(Q_TILE % 1024 == 0 && KV_TILE % 1024 == 0 && OFF_STG % 128 == 0, "alignment");
  static_assert(T_DK + D <= TMEM_COLS, "TMEM budget");
};

// Byte offset of the kk-th 16-wide K slice of a K-major tile whose CHUNK-wide column
// blocks are `chunk_bytes` apart.
template <int D>
__host__ __device__ constexpr uint32_t koff(uint32_t chunk_bytes, int kk) {
  return (uint32_t)((kk * 16 / Cfg<D>::CHUNK) * chunk_bytes + (kk * 16 % Cfg<D>::CHUNK) * 2);
}
// Byte offset of the kk-th slice of 16 rows of an MN-major operand stored as rows of D.
template <int D>
__host__ __device__ constexpr uint32_t mnoff(int kk) { return (uint32_t)(kk * 16 * Cfg<D>::ROWB); }

// TMEM column of the packed bf16 A operand (P^T or dS^T) for the kk-th 16-query slice:
// queries 0..31 live in columns [0,16), queries 32..63 in [32,48).
__device__ __forceinline__ uint32_t a_col(int kk) { return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8); }

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, w, site));
}

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

template <int D, bool CAUSAL, bool VARLEN, bool LOCAL>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const BwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = (int)warp_id(), lane = (int)lane_id();
  // Key tiles of one head are adjacent in launch order, so resident CTAs share the
  // Q, dO and dq_accum of a few heads in L2; causal: low key tiles see the most
  // queries and go first.
  int kt = blockIdx.x;
  int chunk = -1;  // >= 0: this CTA covers query steps [chunk*split_q, (chunk+1)*split_q) only
  if (LOCAL && p.n_gk > 0) {
    const int n_split_ctas = p.n_gk * p.n_qsplit;
    if (kt < n_split_ctas) {
      chunk = kt % p.n_qsplit;
      kt = kt / p.n_qsplit;
    } else {
      kt = kt - n_split_ctas + p.n_gk;
    }
  }
  int bh = blockIdx.y;  // dense: batch * head; packed: head
  if (!VARLEN && !LOCAL && p.lpt) {
    // longest-first over all heads: key tile 0 of every head, then key tile 1, ...
    const int lin = (int)(blockIdx.y * gridDim.x + blockIdx.x);
    kt = lin / (int)gridDim.y;
    bh = lin % (int)gridDim.y;
  }
  // Packed batch: column x of the grid is a compact slot (slot_seq) of sequence b, whose
  // key tiles take its slots in order; a slot past the sequence's keys has nothing to do.
  int by = bh;
  if (VARLEN) {
    const int b = slot_seq(p.va.cu_k, p.va.B, p.va.total_k, 7, (int)blockIdx.x);
    by = b * p.va.H + bh;
    kt = (int)blockIdx.x - slot_base(p.va.cu_k, p.va.total_k, 7, b);
  }
  const int k0 = kt * C::BN;
  const SeqView sv = seq_view<VARLEN>(p.va, p.Nq, p.Nk, by);
  if (VARLEN && k0 >= sv.Nk) return;  // this sequence has fewer keys: nothing to do
  // TMA coordinates (dense maps [B*H][N][D]: y = row, z = bh; packed [total][H][D]: y = head,
  // z = token) and the first workspace row of this sequence
  const int qz_b = VARLEN ? sv.q_tok : bh, kz_b = VARLEN ? sv.k_tok : bh;
  auto ty = [&](int r) { return VARLEN ? sv.h : r; };
  auto tzq = [&](int r) { return VARLEN ? qz_b + r : qz_b; };
  auto tzk = [&](int r) { return VARLEN ? kz_b + r : kz_b; };
  const long long wrow0 = ws_row0(VARLEN, by, p.Nq_pad, sv);
  // Query steps (64 rows) that see a key of this tile: causal ones start at the diagonal;
  // with the local mask they are the global query steps [a, g) and the window steps [L, hi)
  // (every step when the tile holds a global key).
  const int n_qt = (sv.Nq + C::BM - 1) / C::BM;
  const int qlo = CAUSAL ? k0 : 0;  // first query that may see key k0
  TileSet qs = TileSet::make(qlo / C::BM, qlo / C::BM, qlo / C::BM, n_qt);
  if (LOCAL && k0 >= p.lm.n_glob) {
    const int ke = min(k0 + C::BN, sv.Nk) - 1;
    const int qmax = min(sv.Nq - 1, ke + p.lm.win_l);
    qs = TileSet::make(qlo / C::BM, (p.lm.n_glob + C::BM - 1) / C::BM, max(qlo, k0 - p.lm.win_r) / C::BM,
                       qmax >= 0 ? qmax / C::BM + 1 : 0);
  }
  if (LOCAL && chunk >= 0) {
    const int lo = chunk * p.split_q, hi = lo + p.split_q;
    qs = TileSet::make(max(qs.a, lo), min(qs.g, hi), max(qs.L, lo), min(qs.hi, hi));
  }
  const int n_it = qs.count();
  const WaitCtx wc{p.wait_limit_ns, p.status, abort_flag};

  if (threadIdx.x == 0) {
    mbar_init(&bars[C::B_KV], 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bars[C::B_QF + s], 1);
      mbar_init(&bars[C::B_QE + s], 1);
    }
    for (int b = 0; b < C::NB; ++b) {
      mbar_init(&bars[C::B_SF + b], 1);
      mbar_init(&bars[C::B_PF + b], 256);
      mbar_init(&bars[C::B_DSF + b], 256);
      mbar_init(&bars[C::B_DQF + b], 1);
      mbar_init(&bars[C::B_DQR + b], 1);
      mbar_init(&bars[C::B_DQE + b], 128);
    }
    mbar_init(&bars[C::B_DRAIN], 1);
    mbar_init(&bars[C::B_DRAIN + 1], 1);
    mbar_init(&bars[C::B_DPF], 1);
    mbar_init(&bars[C::B_KT], 128);
    mbar_init(&bars[C::B_DPE], 256);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::W_MMA_A) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::W_PRODUCER) {
    // ---------------------------------------------------------------- TMA producer
    if (n_it > 0) {
      if (lane == 0) tma_prefetch_desc(&tm_q);
      if (lane == 0) tma_prefetch_desc(&tm_k);
      if (lane == 0) tma_prefetch_desc(&tm_v);
      if (lane == 0) tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx_w(&bars[C::B_KV], 2 * C::KV_TILE);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_3d_w(smem + C::OFF_K + c * C::K_CHUNK_BYTES, &tm_k, &bars[C::B_KV], c * C::CHUNK, ty(k0), tzk(k0));
        tma_load_3d_w(smem + C::OFF_V + c * C::K_CHUNK_BYTES, &tm_v, &bars[C::B_KV], c * C::CHUNK, ty(k0), tzk(k0));
      }
      int issued = 0;
      for (int it = 0; it < n_it; ++it) {
        const int s = it % C::NS;
        const int i = qs.at(it);
        if (it >= C::NS && !mbar_wait_w(&bars[C::B_QE + s], ((it / C::NS) - 1) & 1, wc, 31)) break;
        mbar_arrive_expect_tx_w(&bars[C::B_QF + s], 2 * C::Q_TILE + 2 * C::BM * 4);
        for (int c = 0; c < C::NCHUNK; ++c) {
          tma_load_3d_w(smem + C::OFF_Q + s * C::Q_TILE + c * C::Q_CHUNK_BYTES, &tm_q, &bars[C::B_QF + s],
                      c * C::CHUNK, ty(i * C::BM), tzq(i * C::BM));
          tma_load_3d_w(smem + C::OFF_DO + s * C::Q_TILE + c * C::Q_CHUNK_BYTES, &tm_do, &bars[C::B_QF + s],
                      c * C::CHUNK, ty(i * C::BM), tzq(i * C::BM));
        }
        const size_t roff = (size_t)wrow0 + (size_t)i * C::BM;
        bulk_load_w(smem + C::OFF_LSE + s * C::BM * 4, p.lse2 + roff, C::BM * 4, &bars[C::B_QF + s]);
        bulk_load_w(smem + C::OFF_DLT + s * C::BM * 4, p.dlt + roff, C::BM * 4, &bars[C::B_QF + s]);
        issued = it + 1;
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        volatile int no_abort = 0;
        const WaitCtx w2{p.wait_limit_ns, p.status, &no_abort};
        mbar_wait(&bars[C::B_KV], 0, w2, 40);
        const int first = issued > C::NS ? issued - C::NS : 0;
        for (int it = first; it < issued; ++it)
          mbar_wait(&bars[C::B_QF + it % C::NS], (it / C::NS) & 1, w2, 41);
      }
    }
  } else if (warp == C::W_MMA_A) {
    // ---------------------------------------------------------------- UMMA issuer A: S^T, dP^T
    if (n_it > 0) {
      const uint64_t dK = sdesc(sbase + C::OFF_K, 16, 8 * C::ROWB, C::LAYOUT);       // K, K-major
      const uint64_t dV = sdesc(sbase + C::OFF_V, 16, 8 * C::ROWB, C::LAYOUT);       // V, K-major
      const uint64_t dQk = sdesc(sbase + C::OFF_Q, 16, 8 * C::ROWB, C::LAYOUT);      // Q stage 0, K-major
      const uint64_t dOk = sdesc(sbase + C::OFF_DO, 16, 8 * C::ROWB, C::LAYOUT);     // dO stage 0, K-major
      auto issue_s = [&](int it) {  // S^T(it) = K Q^T into TMEM buffer it & 1
        const uint64_t q = desc_adv(dQk, (uint32_t)((it % C::NS) * C::Q_TILE));
        const uint32_t d = tmem + C::T_S + (uint32_t)((it & 1) * 64);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_w(d, desc_adv(dK, koff<D>(C::K_CHUNK_BYTES, kk)), desc_adv(q, koff<D>(C::Q_CHUNK_BYTES, kk)),
                  C::IDESC_S, kk > 0 ? 1u : 0u);
        umma_commit_w(&bars[C::B_SF + (it & 1)]);
      };
      auto issue_dp = [&](int it) {  // dP^T(it) = V dO^T
        const uint64_t o = desc_adv(dOk, (uint32_t)((it % C::NS) * C::Q_TILE));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_w(tmem + C::T_DP, desc_adv(dV, koff<D>(C::K_CHUNK_BYTES, kk)), desc_adv(o, koff<D>(C::Q_CHUNK_BYTES, kk)),
                  C::IDESC_S, kk > 0 ? 1u : 0u);
        umma_commit_w(&bars[C::B_DPF]);
      };
      bool ok = mbar_wait_w(&bars[C::B_KV], 0, wc, 32) && mbar_wait_w(&bars[C::B_QF], 0, wc, 33);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int it = 0; ok && it < n_it; ++it) {
        // dP^T(it) overwrites dP^T(it-1) in TMEM once the compute warps have loaded it (its
        // stage is loaded: S^T(it) waited for it)
        if (it >= 1 && !(ok = mbar_wait_w(&bars[C::B_DPE], (it - 1) & 1, wc, 35))) break;
        tc_fence_after();
        issue_dp(it);
        // S^T(it+1) goes to the buffer that held P^T(it-1), then dQ^T(it-1): after the dQ
        // warpgroup drained it (which follows dV(it-1) and dQ^T(it-1) in issuer B's order)
        if (it + 1 < n_it) {
          const int s1 = (it + 1) % C::NS, b1 = (it + 1) & 1;
          if (!(ok = mbar_wait_w(&bars[C::B_QF + s1], ((it + 1) / C::NS) & 1, wc, 33))) break;
          if (it >= 1 && !(ok = mbar_wait_w(&bars[C::B_DQE + b1], ((it - 1) >> 1) & 1, wc, 49))) break;
          tc_fence_after();
          issue_s(it + 1);
        }
      }
      umma_commit_w(&bars[C::B_DRAIN]);
      volatile int no_abort = 0;
      const WaitCtx w2{p.wait_limit_ns, p.status, &no_abort};
      mbar_wait(&bars[C::B_DRAIN], 0, w2, 42);
    }
  } else if (warp == C::W_MMA_B) {
    // ---------------------------------------------------------------- UMMA issuer B: dV, dK, dQ^T
    if (n_it > 0) {
      const uint64_t dQm = sdesc(sbase + C::OFF_Q, C::Q_CHUNK_BYTES, 8 * C::ROWB, C::LAYOUT);   // MN-major
      const uint64_t dOm = sdesc(sbase + C::OFF_DO, C::Q_CHUNK_BYTES, 8 * C::ROWB, C::LAYOUT);  // MN-major
      const uint64_t dS0 = sdesc(sbase + C::OFF_DS, C::DS_BYTES, 1024, 2u);          // dS^T buffer 0, MN-major
      const uint64_t dSa = sdesc(sbase + C::OFF_DS, 16, 1024, 2u);                   // the same, K-major A
      bool ok = mbar_wait_w(&bars[C::B_KV], 0, wc, 32);
      for (int it = 0; ok && it < n_it; ++it) {
        const int s = it % C::NS, b = it & 1;
        const uint64_t qm = desc_adv(dQm, (uint32_t)(s * C::Q_TILE));
        const uint64_t om = desc_adv(dOm, (uint32_t)(s * C::Q_TILE));
        // dV += P^T dO_i once P^T(it) is in TMEM buffer b
        if (!(ok = mbar_wait_w(&bars[C::B_PF + b], (it >> 1) & 1, wc, 34))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          umma_ts_w(tmem + C::T_DV, tmem + C::T_S + (uint32_t)(b * 64) + a_col(kk), desc_adv(om, mnoff<D>(kk)),
                  C::IDESC_KV, (it > 0 || kk > 0) ? 1u : 0u);
        // dK += dS^T Q_i and dQ_i^T = K^T dS^T once dS^T is in shared memory buffer b (one
        // copy serves both: 128-byte swizzled rows of 64 queries per key are the K-major A
        // layout of dK and the MN-major B layout of dQ^T)
        if (!(ok = mbar_wait_w(&bars[C::B_DSF + b], (it >> 1) & 1, wc, 36))) break;
        if (it == 0 && !(ok = mbar_wait_w(&bars[C::B_KT], 0, wc, 47))) break;
        tc_fence_after();
        // dQ^T(it) first, into buffer b, which dV(it) (issued above: in-order) has finished
        // reading: the dQ warpgroup's drain of it gates S^T(it+2), so it starts as early as it can
        const uint64_t ds = desc_adv(dS0, (uint32_t)(b * C::DS_BYTES));
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          umma_ts_w(tmem + C::T_S + (uint32_t)(b * 64), tmem + C::T_KT + kk * 8, desc_adv(ds, (uint32_t)(kk * 16 * 128)),
                    C::IDESC_DQ, kk > 0 ? 1u : 0u);
        umma_commit_w(&bars[C::B_DQR + b]);
        const uint64_t dsa = desc_adv(dSa, (uint32_t)(b * C::DS_BYTES));
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          umma_ss_w(tmem + C::T_DK, desc_adv(dsa, (uint32_t)(kk * 32)), desc_adv(qm, mnoff<D>(kk)), C::IDESC_KV,
                    (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit_w(&bars[C::B_QE + s]);   // dK was the stage's last reader
        umma_commit_w(&bars[C::B_DQF + b]);  // dQ^T and dK have both read dS^T buffer b
      }
      umma_commit_w(&bars[C::B_DRAIN + 1]);
      volatile int no_abort = 0;
      const WaitCtx w2{p.wait_limit_ns, p.status, &no_abort};
      mbar_wait(&bars[C::B_DRAIN + 1], 0, w2, 42);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- compute warpgroups
    const int wg = (warp - 4) >> 2;  // 0: queries 0..31 of a tile (and dK), 1: queries 32..63 (and dV)
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // key row of the tile (also d for the dQ^T readout)
    const int key = k0 + row;
    const int col0 = wg * 32;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = p.scale_log2;
    uint8_t* sds_row_base = smem + C::OFF_DS + row * 128;
    bool ok = true;

    for (int it = 0; it < n_it && ok; ++it) {
      const int s = it % C::NS;
      const int i = qs.at(it);
      const uint32_t t_sb = (uint32_t)((it & 1) * 64);  // this step's S^T / P^T buffer
      if (!warp_wait(&bars[C::B_QF + s], (it / C::NS) & 1, wc, 38) ||
          !warp_wait(&bars[C::B_SF + (it & 1)], (it >> 1) & 1, wc, 39)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sreg[32];
      tmem_ld32(t_lane + C::T_S + t_sb + col0, sreg);
      tmem_wait_ld(sreg);
      const float* lse2 = reinterpret_cast<const float*>(smem + C::OFF_LSE + s * C::BM * 4) + col0;
      const float* dlt = reinterpret_cast<const float*>(smem + C::OFF_DLT + s * C::BM * 4) + col0;
      const int qb = i * C::BM + col0;  // query of column 0 of this warpgroup's half
      bool need_mask = (k0 + C::BN > sv.Nk) || (CAUSAL && (k0 + C::BN - 1 > qb));
      if (LOCAL)
        need_mask = need_mask || !(k0 + C::BN <= p.lm.n_glob || qb + 31 < p.lm.n_glob ||
                                   (k0 >= qb + 31 - p.lm.win_l && k0 + C::BN - 1 <= qb + p.lm.win_r));
      int lim = 1 << 30;  // columns c with q = qb + c < key are masked (causal)
      if (CAUSAL) lim = key - qb;
      const bool key_valid = key < sv.Nk;
      // local: for a non-global key, columns c >= gq (non-global queries) are visible only
      // inside the window key - win_r <= q <= key + win_l
      const bool kglob = !LOCAL || key < p.lm.n_glob;
      const int gq = p.lm.n_glob - qb, wlo = key - p.lm.win_r - qb, whi = key + p.lm.win_l - qb;
      float pv[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float x = ex2(fmaf(as_f(sreg[c]), sl2, -lse2[c]));
        if (need_mask && (!key_valid || (CAUSAL && c < lim))) x = 0.f;
        if (LOCAL && need_mask && !kglob && c >= gq && (c < wlo || c > whi)) x = 0.f;
        pv[c] = x;
      }
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) pk[c] = pack_bf16(pv[2 * c], pv[2 * c + 1]);
      tmem_st16(t_lane + C::T_S + t_sb + wg * 32, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[C::B_PF + (it & 1)]);

      if (!warp_wait(&bars[C::B_DPF], it & 1, wc, 43)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t dv[32];
      tmem_ld32(t_lane + C::T_DP + col0, dv);
      tmem_wait_ld(dv);
      tc_fence_before();
      mbar_arrive(&bars[C::B_DPE]);  // dP^T(it+1) may overwrite it now
      uint32_t dk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float d0 = pv[2 * c] * (as_f(dv[2 * c]) - dlt[2 * c]);
        const float d1 = pv[2 * c + 1] * (as_f(dv[2 * c + 1]) - dlt[2 * c + 1]);
        dk[c] = pack_bf16(d0, d1);
      }
      // dS^T row into shared memory (128-byte rows, 128B swizzle) for the dK and dQ^T MMAs,
      // once the dQ^T MMA two tiles back (issued after that tile's dK) has finished reading
      // this buffer.
      if (it >= 2 && !warp_wait(&bars[C::B_DQF + (it & 1)], ((it - 2) >> 1) & 1, wc, 44)) {
        ok = false;
        break;
      }
      uint8_t* dsrow = sds_row_base + (it & 1) * C::DS_BYTES;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int phys = (4 * wg + t) ^ (row & 7);
        *reinterpret_cast<uint4*>(dsrow + phys * 16) = make_uint4(dk[4 * t], dk[4 * t + 1], dk[4 * t + 2], dk[4 * t + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[C::B_DSF + (it & 1)]);
    }

    // epilogue: WG0 writes dK = scale * acc, WG1 writes dV; the last dQ commit covers both
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(wg == 0 ? p.dk : p.dv) +
                         (VARLEN ? ((size_t)(sv.k_tok + key) * p.va.H + sv.h) * D : ((size_t)bh * sv.Nk + key) * D);
    if (LOCAL && chunk >= 0) {
      // partial sums of a split global key tile: add (unscaled) into dkv_accum
      if (n_it > 0 && ok && warp_wait(&bars[C::B_DQF + ((n_it - 1) & 1)], ((n_it - 1) >> 1) & 1, wc, 45)) {
        tc_fence_after();
        float* acc = p.dkv_accum + (((size_t)bh * (p.n_gk * C::BN) + (size_t)row + (size_t)kt * C::BN) * 2 + wg) * D;
#pragma unroll
        for (int g = 0; g < D / 16; ++g) {
          uint32_t v[16];
          tmem_ld16(t_lane + (wg == 0 ? C::T_DK : C::T_DV) + g * 16, v);
          tmem_wait_ld(v);
          if (key < sv.Nk) {
#pragma unroll
            for (int c = 0; c < 16; c += 4)
              asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(acc + g * 16 + c), "f"(as_f(v[c])),
                           "f"(as_f(v[c + 1])), "f"(as_f(v[c + 2])), "f"(as_f(v[c + 3]))
                           : "memory");
          }
        }
      }
    } else if (n_it == 0) {
      if (key < sv.Nk) {
        for (int d = 0; d < D; d += 8) *reinterpret_cast<uint4*>(dst + d) = make_uint4(0, 0, 0, 0);
      }
    } else if (ok && warp_wait(&bars[C::B_DQF + ((n_it - 1) & 1)], ((n_it - 1) >> 1) & 1, wc, 45)) {
      tc_fence_after();
      const float mul = (wg == 0) ? p.scale : 1.f;
#pragma unroll
      for (int g = 0; g < D / 16; ++g) {
        uint32_t v[16];
        tmem_ld16(t_lane + (wg == 0 ? C::T_DK : C::T_DV) + g * 16, v);
        tmem_wait_ld(v);
        if (key < sv.Nk) store16_bf16(dst + g * 16, v, mul);
      }
    }
  } else {
    // ---------------------------------------------------------------- dQ warpgroup (warps 0-3)
    const int d = warp * 32 + lane;  // TMEM lane = row d of dQ^T
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
    float* stg = reinterpret_cast<float*>(smem + C::OFF_STG);
    // K^T into TMEM once per CTA: lane d holds K[key][d] for all 128 keys as bf16 pairs
    // (the A operand of dQ^T = K^T dS^T).  Lanes d >= D (D < 128) hold zeros.
    bool ok = n_it > 0 && named_bar_and(1, 128, warp_wait(&bars[C::B_KV], 0, wc, 48));
    if (ok) {
      const uint8_t* sK = smem + C::OFF_K;
      const int dc = d < D ? d : 0;
      const int chunk = dc / C::CHUNK, col = dc % C::CHUNK;
      const uint8_t* base = sK + chunk * C::K_CHUNK_BYTES + (col % 8) * 2;
      const int u = col / 8;
      uint32_t kt[2][32];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        uint32_t pr = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = 2 * c + h;  // key row of the swizzled K-major tile
          const int phys = u ^ ((r * C::ROWB >> 7) & (C::ROWB / 16 - 1));
          const uint32_t e = *reinterpret_cast<const uint16_t*>(base + r * C::ROWB + phys * 16);
          pr |= (d < D ? e : 0u) << (16 * h);
        }
        kt[c >> 5][c & 31] = pr;
      }
      tmem_st32(t_lane + C::T_KT, kt[0]);
      tmem_st32(t_lane + C::T_KT + 32, kt[1]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[C::B_KT]);
    }
    for (int it = 0; ok && it < n_it; ++it) {
      const int b = it & 1;
      // the four warps agree before any of them reaches the named barriers below
      if (!named_bar_and(1, 128, warp_wait(&bars[C::B_DQR + b], (it >> 1) & 1, wc, 46))) break;
      tc_fence_after();
      uint32_t v0[32], v1[32];
      tmem_ld32(t_lane + C::T_S + (uint32_t)(b * 64), v0);
      tmem_ld32(t_lane + C::T_S + (uint32_t)(b * 64) + 32, v1);
      tmem_wait_ld(v0);
      reg_tie(v1);
      tc_fence_before();
      mbar_arrive(&bars[C::B_DQE + b]);
      // two halves of 32 queries: a half is rewritten once the reduce that last read it is
      // done reading (bulk groups complete in order), so one half's read overlaps the other
      // half's writes
      float* gdst = p.dq_accum + ((size_t)wrow0 + (size_t)qs.at(it) * C::BM) * D;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        named_bar_sync(1, 128);
        if (d < D) {
#pragma unroll
          for (int c = 0; c < 32; ++c) stg[(h * 32 + c) * D + d] = as_f(h == 0 ? v0[c] : v1[c]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (threadIdx.x == 0) {
          bulk_reduce_add_f32(gdst + h * 32 * D, stg + h * 32 * D, C::STG_BYTES / 2);
          bulk_commit_group();
        }
      }
    }
    if (threadIdx.x == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA_A) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------
// Persistent form of bwd_kernel for the plain masks, dense or packed.  The grid still has
// one CTA per (128-key tile, batch*head) in the same order (packed: one per compact slot
// and head, see slot_seq), but a running CTA takes
// over the next CTA that has not started (cluster launch control) instead of exiting, and
// its pipelines run on across units: K / V of the next unit are loaded once the current
// unit's last S^T and dP^T and its K^T build have read the old ones, K^T is rebuilt in TMEM once the last
// dQ^T has read the old one, and the next unit's first score GEMMs run while the compute
// warps are still in the current unit's epilogue (its dK / dV accumulate from zero once
// that epilogue has read the old ones out of TMEM).  Step-indexed barrier phases count
// steps over all units (g = the unit's first global step + it); unit-indexed ones count
// units.  Roles, arithmetic and per-step order are those of bwd_kernel.  The producer
// resolves each CTA index into a unit (packed: passing over slots past a sequence's keys)
// and itself writes dK = dV = 0 for a key tile that no query step sees.
// ------------------------------------------------------------------------------------
// A unit as the producer publishes it: keys [k0, k0 + 128) of one (sequence, head).  Dense:
// z = batch*head, q_tok = k_tok = b = 0, nq = Nq, nk = Nk; packed: z = head, q_tok / k_tok
// the sequence's first tokens, nq / nk its lengths, b its index.  live = 0 ends the ring.
struct BwdUnit {
  int k0, z, q_tok, k_tok, nq, nk, b, live;  // b: packed, the sequence; local mask, the query
                                              // chunk of a split global key tile (-1: none)
};

// SPLIT (local mask only): the launch also holds the chunks of split global key tiles
template <int D, bool CAUSAL, bool VARLEN, bool LOCAL = false, bool SPLIT = false>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    bwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  void* clc_resp = smem + C::OFF_CLC;
  BwdUnit* units = reinterpret_cast<BwdUnit*>(smem + C::OFF_UNITS);

  const int warp = (int)warp_id(), lane = (int)lane_id();
  // query steps of a unit: causal ones start at the diagonal; a published unit has one at least
  auto first_step = [&](const BwdUnit& u) { return CAUSAL ? u.k0 / C::BM : 0; };
  auto n_steps = [&](const BwdUnit& u) { return (u.nq + C::BM - 1) / C::BM - first_step(u); };
  static_assert(!(LOCAL && VARLEN), "the local mask is dense only");
  static_assert(LOCAL || !SPLIT, "only the local mask splits key tiles");
  // local mask: bwd_kernel's step set of the unit's key tile, the global query steps [a, g)
  // then the window's steps [L, hi) (every step from the causal start when the tile holds a
  // global key); step it of the unit is query tile local_steps(u).at(it)
  auto local_steps = [&](const BwdUnit& u) -> TileSet {
    const int n_qt = (u.nq + C::BM - 1) / C::BM;
    const int qlo = CAUSAL ? u.k0 : 0;  // first query that may see key k0
    TileSet qs = TileSet::make(qlo / C::BM, qlo / C::BM, qlo / C::BM, n_qt);
    if (u.k0 >= p.lm.n_glob) {
      const int ke = min(u.k0 + C::BN, u.nk) - 1;
      const int qmax = min(u.nq - 1, ke + p.lm.win_l);
      qs = TileSet::make(qlo / C::BM, (p.lm.n_glob + C::BM - 1) / C::BM, max(qlo, u.k0 - p.lm.win_r) / C::BM,
                         qmax >= 0 ? qmax / C::BM + 1 : 0);
    }
    if (SPLIT && u.b >= 0) {  // a chunk of a split global key tile: its query steps only
      const int lo = u.b * p.split_q, hi = lo + p.split_q;
      qs = TileSet::make(max(qs.a, lo), min(qs.g, hi), max(qs.L, lo), min(qs.hi, hi));
    }
    return qs;
  };
  auto unit_steps = [&](const BwdUnit& u) -> int {
    if constexpr (LOCAL) return local_steps(u).count();
    else return n_steps(u);
  };
  // first workspace row of the unit's (sequence, head)
  auto wrow0 = [&](const BwdUnit& u) -> long long {
    return VARLEN ? (long long)u.z * p.Nq_pad + 64LL * ((u.q_tok + 63) / 64 + u.b) : (long long)u.z * p.Nq_pad;
  };
  const WaitCtx wc{p.wait_limit_ns, p.status, abort_flag};

  if (threadIdx.x == 0) {
    mbar_init(&bars[C::B_KV], 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bars[C::B_QF + s], 1);
      mbar_init(&bars[C::B_QE + s], 1);
    }
    for (int b = 0; b < C::NB; ++b) {
      mbar_init(&bars[C::B_SF + b], 1);
      mbar_init(&bars[C::B_PF + b], 256);
      mbar_init(&bars[C::B_DSF + b], 256);
      mbar_init(&bars[C::B_DQF + b], 1);
      mbar_init(&bars[C::B_DQR + b], 1);
      mbar_init(&bars[C::B_DQE + b], 128);
    }
    mbar_init(&bars[C::B_DRAIN], 1);
    mbar_init(&bars[C::B_DRAIN + 1], 1);
    mbar_init(&bars[C::B_DPF], 1);
    mbar_init(&bars[C::B_KT], 128);
    mbar_init(&bars[C::B_DPE], 256);
    mbar_init(&bars[C::B_KVE], 5);  // issuer A's commit and the 4 dQ warps (K^T built)
    mbar_init(&bars[C::B_KTE], 1);
    mbar_init(&bars[C::B_ACCE], 256);
    for (int u = 0; u < C::NU; ++u) {
      mbar_init(&bars[C::B_UF + u], 1);
      mbar_init(&bars[C::B_UE + u], 14);  // both issuing warps, the 8 compute warps, the 4 dQ warps
    }
    mbar_init(&bars[C::B_CLC], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::W_MMA_A) {
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
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
    }
    int ux = (int)blockIdx.x, uy = (int)blockIdx.y;  // the CTA index to work on next (ux < 0: none)
    int g0 = 0, issued = 0, kv_units = 0;  // the unit's first global step; steps / K,V pairs started
    bool asked = false;
    int n_asked = 0;
    // take over the next CTA of the grid that has not started (ux = -1: none is left)
    auto claim = [&]() -> bool {
      mbar_arrive_expect_tx_w(&bars[C::B_CLC], 16);
      clc_try_cancel_w(clc_resp, &bars[C::B_CLC]);
      asked = true;
      if (!mbar_wait_w(&bars[C::B_CLC], n_asked & 1, wc, 52)) return false;
      asked = false;
      ++n_asked;
      int cx, cy;
      const bool taken = clc_taken(clc_resp, cx, cy);
      ux = (taken && cx >= 0 && cx < (int)gridDim.x && cy >= 0 && cy < (int)gridDim.y) ? cx : -1;
      uy = cy;
      return true;
    };
    // the unit of CTA (ux, uy); false when it has nothing for the pipeline (packed: a slot past
    // its sequence's keys; either layout: a key tile no query sees, whose dK, dV rows get
    // zeros here)
    auto resolve = [&](BwdUnit& un) -> bool {
      un.live = 1;
      if (!VARLEN) {
        // lpt: units in longest-first order over all heads (key tile 0 of every head, then
        // key tile 1, ...), for causal launches of a few waves whose tail would otherwise be
        // one head's heaviest key tiles starting last
        int kt = ux, zz = uy, chunk = -1;
        if (SPLIT) {  // bwd_kernel's grid: the split global key tiles' chunks first
          const int n_split_ctas = p.n_gk * p.n_qsplit;
          if (kt < n_split_ctas) {
            chunk = kt % p.n_qsplit;
            kt = kt / p.n_qsplit;
          } else {
            kt = kt - n_split_ctas + p.n_gk;
          }
        }
        if (p.lpt) {  // rank-major within groups of p.lpt heads (all heads when p.lpt >= H)
          const int gx = (int)gridDim.x, nh = (int)gridDim.y, gs0 = min(p.lpt, nh);
          const int lin = uy * gx + ux;
          const int grp = lin / (gs0 * gx), h0 = grp * gs0, gs = min(gs0, nh - h0);
          const int idx = lin - h0 * gx;
          kt = idx / gs;
          zz = h0 + idx % gs;
        }
        un.k0 = kt * C::BN;
        un.z = zz;
        un.q_tok = un.k_tok = 0;
        un.b = SPLIT ? chunk : 0;
        un.nq = p.Nq;
        un.nk = p.Nk;
      } else {
        // lpt: slot-major over the heads (slot x of every head, then slot x + 1), so the
        // heaviest key tiles of a long sequence start while the other heads' work remains
        int sx = ux, hy = uy;
        if (p.lpt) {
          const int lin = uy * (int)gridDim.x + ux;
          sx = lin / (int)gridDim.y;
          hy = lin % (int)gridDim.y;
        }
        const int b = slot_seq(p.va.cu_k, p.va.B, p.va.total_k, 7, sx);
        const int kt = sx - slot_base(p.va.cu_k, p.va.total_k, 7, b);
        const SeqView sv = seq_view<true>(p.va, p.Nq, p.Nk, b * p.va.H + hy);
        if (kt * C::BN >= sv.Nk) return false;
        un.k0 = kt * C::BN;
        un.z = hy;
        un.q_tok = sv.q_tok;
        un.k_tok = sv.k_tok;
        un.nq = sv.Nq;
        un.nk = sv.Nk;
        un.b = b;
      }
      if (unit_steps(un) > 0) return true;
      if (SPLIT && un.b >= 0) return false;  // a chunk with no step adds nothing to dkv_accum
      const int r1 = min(un.k0 + C::BN, un.nk);
      for (int e = lane; e < (r1 - un.k0) * (D / 8); e += 32) {
        const int key = un.k0 + e / (D / 8);
        const size_t off = VARLEN ? ((size_t)(un.k_tok + key) * p.va.H + un.z) * D : ((size_t)un.z * p.Nk + key) * D;
        reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dk) + off)[e % (D / 8)] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dv) + off)[e % (D / 8)] = make_uint4(0, 0, 0, 0);
      }
      return false;
    };
    for (int u = 0;; ++u) {
      BwdUnit un;
      un.live = 0;
      bool ok = true;
      while (ux >= 0 && !resolve(un))
        if (!(ok = claim())) break;
      if (!ok) break;
      if (ux < 0) un.live = 0;
      const int us = u % C::NU;
      if (u >= C::NU && !mbar_wait_w(&bars[C::B_UE + us], ((u / C::NU) - 1) & 1, wc, 50)) break;
      units[us] = un;  // (every lane holds the same record)
      mbar_arrive_w(&bars[C::B_UF + us]);
      if (!un.live) break;
      const int k0 = un.k0, i0 = first_step(un), n_it = unit_steps(un);
      TileSet qs{};
      if constexpr (LOCAL) qs = local_steps(un);
      const long long w0 = wrow0(un);
      // TMA coordinates of row r: dense maps [B*H][N][D] (y = row, z = batch*head), packed
      // maps [total][H][D] (y = head, z = token)
      auto ty = [&](int r) { return VARLEN ? un.z : r; };
      auto tzq = [&](int r) { return VARLEN ? un.q_tok + r : un.z; };
      auto tzk = [&](int r) { return VARLEN ? un.k_tok + r : un.z; };
      // K / V: free once the previous unit's last S^T and dP^T and its K^T build have read them
      if (u >= 1 && !mbar_wait_w(&bars[C::B_KVE], (u - 1) & 1, wc, 51)) break;
      mbar_arrive_expect_tx_w(&bars[C::B_KV], 2 * C::KV_TILE);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_3d_w(smem + C::OFF_K + c * C::K_CHUNK_BYTES, &tm_k, &bars[C::B_KV], c * C::CHUNK, ty(k0), tzk(k0));
        tma_load_3d_w(smem + C::OFF_V + c * C::K_CHUNK_BYTES, &tm_v, &bars[C::B_KV], c * C::CHUNK, ty(k0), tzk(k0));
      }
      kv_units = u + 1;
      for (int it = 0; it < n_it; ++it) {
        const int g = g0 + it, s = g % C::NS, i = LOCAL ? qs.at(it) : i0 + it;
        if (g >= C::NS && !(ok = mbar_wait_w(&bars[C::B_QE + s], ((g / C::NS) - 1) & 1, wc, 31))) break;
        mbar_arrive_expect_tx_w(&bars[C::B_QF + s], 2 * C::Q_TILE + 2 * C::BM * 4);
        for (int c = 0; c < C::NCHUNK; ++c) {
          tma_load_3d_w(smem + C::OFF_Q + s * C::Q_TILE + c * C::Q_CHUNK_BYTES, &tm_q, &bars[C::B_QF + s],
                        c * C::CHUNK, ty(i * C::BM), tzq(i * C::BM));
          tma_load_3d_w(smem + C::OFF_DO + s * C::Q_TILE + c * C::Q_CHUNK_BYTES, &tm_do, &bars[C::B_QF + s],
                        c * C::CHUNK, ty(i * C::BM), tzq(i * C::BM));
        }
        const size_t roff = (size_t)w0 + (size_t)i * C::BM;
        bulk_load_w(smem + C::OFF_LSE + s * C::BM * 4, p.lse2 + roff, C::BM * 4, &bars[C::B_QF + s]);
        bulk_load_w(smem + C::OFF_DLT + s * C::BM * 4, p.dlt + roff, C::BM * 4, &bars[C::B_QF + s]);
        issued = g + 1;
      }
      if (!ok) break;
      g0 += n_it;
      // the next unit, asked for once this unit's last copies are started
      if (!claim()) break;
    }
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      volatile int no_abort = 0;
      const WaitCtx w2{p.wait_limit_ns, p.status, &no_abort};
      if (kv_units > 0) mbar_wait(&bars[C::B_KV], (kv_units - 1) & 1, w2, 40);
      for (int g = issued > C::NS ? issued - C::NS : 0; g < issued; ++g)
        mbar_wait(&bars[C::B_QF + g % C::NS], (g / C::NS) & 1, w2, 41);
      if (asked) mbar_wait(&bars[C::B_CLC], n_asked & 1, w2, 53);
    }
  } else if (warp == C::W_MMA_A) {
    // ---------------------------------------------------------------- UMMA issuer A: S^T, dP^T
    const uint64_t dK = sdesc(sbase + C::OFF_K, 16, 8 * C::ROWB, C::LAYOUT);       // K, K-major
    const uint64_t dV = sdesc(sbase + C::OFF_V, 16, 8 * C::ROWB, C::LAYOUT);       // V, K-major
    const uint64_t dQk = sdesc(sbase + C::OFF_Q, 16, 8 * C::ROWB, C::LAYOUT);      // Q stage 0, K-major
    const uint64_t dOk = sdesc(sbase + C::OFF_DO, 16, 8 * C::ROWB, C::LAYOUT);     // dO stage 0, K-major
    auto issue_s = [&](int g) {  // S^T(g) = K Q^T into TMEM buffer g % NB
      const uint64_t q = desc_adv(dQk, (uint32_t)((g % C::NS) * C::Q_TILE));
      const uint32_t d = tmem + C::T_S + (uint32_t)((g % C::NB) * 64);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        umma_ss_w(d, desc_adv(dK, koff<D>(C::K_CHUNK_BYTES, kk)), desc_adv(q, koff<D>(C::Q_CHUNK_BYTES, kk)),
                  C::IDESC_S, kk > 0 ? 1u : 0u);
      umma_commit_w(&bars[C::B_SF + g % C::NB]);
    };
    auto issue_dp = [&](int g) {  // dP^T(g) = V dO^T
      const uint64_t o = desc_adv(dOk, (uint32_t)((g % C::NS) * C::Q_TILE));
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        umma_ss_w(tmem + C::T_DP, desc_adv(dV, koff<D>(C::K_CHUNK_BYTES, kk)), desc_adv(o, koff<D>(C::Q_CHUNK_BYTES, kk)),
                  C::IDESC_S, kk > 0 ? 1u : 0u);
      umma_commit_w(&bars[C::B_DPF]);
    };
    // S^T(g) needs its stage loaded and its TMEM buffer drained of dQ^T(g-NB)
    auto s_ready = [&](int g) {
      return mbar_wait_w(&bars[C::B_QF + g % C::NS], (g / C::NS) & 1, wc, 33) &&
             (g < C::NB || mbar_wait_w(&bars[C::B_DQE + g % C::NB], ((g - C::NB) / C::NB) & 1, wc, 49));
    };
    int g0 = 0;
    bool ok = true;
    for (int u = 0; ok; ++u) {
      const int us = u % C::NU;
      if (!(ok = mbar_wait_w(&bars[C::B_UF + us], (u / C::NU) & 1, wc, 54))) break;
      const BwdUnit un = units[us];
      mbar_arrive_w(&bars[C::B_UE + us]);
      if (!un.live) break;
      const int n_it = unit_steps(un);
      if (!(ok = mbar_wait_w(&bars[C::B_KV], u & 1, wc, 32) && s_ready(g0))) break;
      tc_fence_after();
      issue_s(g0);
      for (int it = 0; ok && it < n_it; ++it) {
        const int g = g0 + it;
        // dP^T(g) overwrites dP^T(g-1) once the compute warps have loaded it
        if (g >= 1 && !(ok = mbar_wait_w(&bars[C::B_DPE], (g - 1) & 1, wc, 35))) break;
        tc_fence_after();
        issue_dp(g);
        if (it + 1 < n_it) {
          if (!(ok = s_ready(g + 1))) break;
          tc_fence_after();
          issue_s(g + 1);
        }
      }
      umma_commit_w(&bars[C::B_KVE]);  // this unit's last UMMA reads of K and V are done
      g0 += n_it;
    }
    umma_commit_w(&bars[C::B_DRAIN]);
    volatile int no_abort = 0;
    const WaitCtx w2{p.wait_limit_ns, p.status, &no_abort};
    mbar_wait(&bars[C::B_DRAIN], 0, w2, 42);
  } else if (warp == C::W_MMA_B) {
    // ---------------------------------------------------------------- UMMA issuer B: dV, dQ^T, dK
    const uint64_t dQm = sdesc(sbase + C::OFF_Q, C::Q_CHUNK_BYTES, 8 * C::ROWB, C::LAYOUT);   // MN-major
    const uint64_t dOm = sdesc(sbase + C::OFF_DO, C::Q_CHUNK_BYTES, 8 * C::ROWB, C::LAYOUT);  // MN-major
    const uint64_t dS0 = sdesc(sbase + C::OFF_DS, C::DS_BYTES, 1024, 2u);          // dS^T buffer 0, MN-major
    const uint64_t dSa = sdesc(sbase + C::OFF_DS, 16, 1024, 2u);                   // the same, K-major A
    int g0 = 0;
    bool ok = true;
    for (int u = 0; ok; ++u) {
      const int us = u % C::NU;
      if (!(ok = mbar_wait_w(&bars[C::B_UF + us], (u / C::NU) & 1, wc, 55))) break;
      const BwdUnit un = units[us];
      mbar_arrive_w(&bars[C::B_UE + us]);
      if (!un.live) break;
      const int n_it = unit_steps(un);
      // dV and dK start from zero: the previous unit's epilogue must have read them out
      if (u >= 1 && !(ok = mbar_wait_w(&bars[C::B_ACCE], (u - 1) & 1, wc, 56))) break;
      for (int it = 0; ok && it < n_it; ++it) {
        const int g = g0 + it, s = g % C::NS, b = g % C::NB, ph = (g / C::NB) & 1;
        const uint64_t qm = desc_adv(dQm, (uint32_t)(s * C::Q_TILE));
        const uint64_t om = desc_adv(dOm, (uint32_t)(s * C::Q_TILE));
        if (!(ok = mbar_wait_w(&bars[C::B_PF + b], ph, wc, 34))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          umma_ts_w(tmem + C::T_DV, tmem + C::T_S + (uint32_t)(b * 64) + a_col(kk), desc_adv(om, mnoff<D>(kk)),
                    C::IDESC_KV, (it > 0 || kk > 0) ? 1u : 0u);
        if (!(ok = mbar_wait_w(&bars[C::B_DSF + b], ph, wc, 36))) break;
        if (it == 0 && !(ok = mbar_wait_w(&bars[C::B_KT], u & 1, wc, 47))) break;
        tc_fence_after();
        // D = 64 (NB = 4): the dQ^T of an even step and the next step of the same unit run as
        // one N = 128 UMMA group over their two adjacent dS^T / TMEM buffers (an N = 64
        // group costs three quarters of an N = 128 one; 2-3% faster at D = 64, slower at
        // D <= 32); other steps run alone
        constexpr bool PAIRS = C::NB >= 4 && D == 64;
        const bool first_of_pair = PAIRS && (g & 1) == 0 && it + 1 < n_it;
        const bool second_of_pair = PAIRS && (g & 1) == 1 && it >= 1;
        if (!first_of_pair) {
          const int b0 = second_of_pair ? b - 1 : b;
          const uint64_t ds = desc_adv(dS0, (uint32_t)(b0 * C::DS_BYTES));
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)
            umma_ts_w(tmem + C::T_S + (uint32_t)(b0 * 64), tmem + C::T_KT + kk * 8,
                      desc_adv(ds, (uint32_t)(kk * 16 * 128)), second_of_pair ? C::IDESC_DQ2 : C::IDESC_DQ,
                      kk > 0 ? 1u : 0u);
          if (second_of_pair) umma_commit_w(&bars[C::B_DQR + b0]);
          umma_commit_w(&bars[C::B_DQR + b]);
        }
        const uint64_t dsa = desc_adv(dSa, (uint32_t)(b * C::DS_BYTES));
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          umma_ss_w(tmem + C::T_DK, desc_adv(dsa, (uint32_t)(kk * 32)), desc_adv(qm, mnoff<D>(kk)), C::IDESC_KV,
                    (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit_w(&bars[C::B_QE + s]);  // dK was the stage's last reader
        // dQ^T and dK have both read dS^T buffer b (a pair's first buffer is released with
        // the second, after their joint dQ^T)
        if (second_of_pair) umma_commit_w(&bars[C::B_DQF + b - 1]);
        if (!first_of_pair) umma_commit_w(&bars[C::B_DQF + b]);
      }
      umma_commit_w(&bars[C::B_KTE]);  // this unit's last read of K^T is done
      g0 += n_it;
    }
    umma_commit_w(&bars[C::B_DRAIN + 1]);
    volatile int no_abort = 0;
    const WaitCtx w2{p.wait_limit_ns, p.status, &no_abort};
    mbar_wait(&bars[C::B_DRAIN + 1], 0, w2, 42);
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- compute warpgroups
    const int wg = (warp - 4) >> 2;  // 0: queries 0..31 of a tile (and dK), 1: queries 32..63 (and dV)
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // key row of the tile
    const int col0 = wg * 32;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = p.scale_log2;
    uint8_t* sds_row_base = smem + C::OFF_DS + row * 128;
    int g0 = 0;
    bool ok = true;
    for (int u = 0;; ++u) {
      const int us = u % C::NU;
      if (!(ok = ok && warp_wait(&bars[C::B_UF + us], (u / C::NU) & 1, wc, 57))) break;
      const BwdUnit un = units[us];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::B_UE + us]);
      if (!un.live) break;
      const int k0 = un.k0, key = k0 + row, i0 = first_step(un), n_it = unit_steps(un);
      TileSet qs{};
      if constexpr (LOCAL) qs = local_steps(un);
      const int nk = VARLEN ? un.nk : p.Nk;  // (dense: the kernel parameter)
      for (int it = 0; it < n_it && ok; ++it) {
        const int g = g0 + it, s = g % C::NS, i = LOCAL ? qs.at(it) : i0 + it;
        const int b = g % C::NB, ph = (g / C::NB) & 1;
        const uint32_t t_sb = (uint32_t)(b * 64);  // this step's S^T / P^T buffer
        if (!warp_wait(&bars[C::B_QF + s], (g / C::NS) & 1, wc, 38) ||
            !warp_wait(&bars[C::B_SF + b], ph, wc, 39)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sreg[32];
        tmem_ld32(t_lane + C::T_S + t_sb + col0, sreg);
        tmem_wait_ld(sreg);
        const float* lse2 = reinterpret_cast<const float*>(smem + C::OFF_LSE + s * C::BM * 4) + col0;
        const float* dlt = reinterpret_cast<const float*>(smem + C::OFF_DLT + s * C::BM * 4) + col0;
        const int qb = i * C::BM + col0;  // query of column 0 of this warpgroup's half
        bool need_mask = (k0 + C::BN > nk) || (CAUSAL && (k0 + C::BN - 1 > qb));
        if (LOCAL)
          need_mask = need_mask || !(k0 + C::BN <= p.lm.n_glob || qb + 31 < p.lm.n_glob ||
                                     (k0 >= qb + 31 - p.lm.win_l && k0 + C::BN - 1 <= qb + p.lm.win_r));
        const int lim = CAUSAL ? key - qb : (1 << 30);  // columns c with q = qb + c < key are masked
        const bool key_valid = key < nk;
        // local: for a non-global key, columns c >= gq (non-global queries) are visible only
        // inside the window key - win_r <= q <= key + win_l
        const bool kglob = !LOCAL || key < p.lm.n_glob;
        const int gq = p.lm.n_glob - qb, wlo = key - p.lm.win_r - qb, whi = key + p.lm.win_l - qb;
        float pv[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float x = ex2(fmaf(as_f(sreg[c]), sl2, -lse2[c]));
          if (need_mask && (!key_valid || (CAUSAL && c < lim))) x = 0.f;
          if (LOCAL && need_mask && !kglob && c >= gq && (c < wlo || c > whi)) x = 0.f;
          pv[c] = x;
        }
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = pack_bf16(pv[2 * c], pv[2 * c + 1]);
        tmem_st16(t_lane + C::T_S + t_sb + wg * 32, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars[C::B_PF + b]);

        if (!warp_wait(&bars[C::B_DPF], g & 1, wc, 43)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t dv[32];
        tmem_ld32(t_lane + C::T_DP + col0, dv);
        tmem_wait_ld(dv);
        tc_fence_before();
        mbar_arrive(&bars[C::B_DPE]);  // dP^T(g+1) may overwrite it now
        uint32_t dk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float d0 = pv[2 * c] * (as_f(dv[2 * c]) - dlt[2 * c]);
          const float d1 = pv[2 * c + 1] * (as_f(dv[2 * c + 1]) - dlt[2 * c + 1]);
          dk[c] = pack_bf16(d0, d1);
        }
        // dS^T row into shared memory buffer g % NB once the dQ^T and dK MMAs of step g-NB
        // have read it
        if (g >= C::NB && !warp_wait(&bars[C::B_DQF + b], ((g - C::NB) / C::NB) & 1, wc, 44)) {
          ok = false;
          break;
        }
        uint8_t* dsrow = sds_row_base + b * C::DS_BYTES;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int phys = (4 * wg + t) ^ (row & 7);
          *reinterpret_cast<uint4*>(dsrow + phys * 16) = make_uint4(dk[4 * t], dk[4 * t + 1], dk[4 * t + 2], dk[4 * t + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[C::B_DSF + b]);
      }
      // epilogue: WG0 writes dK = scale * acc, WG1 writes dV, once the unit's last MMAs are
      // done; the accumulator is handed back to issuer B as soon as it is read out
      const int gl = g0 + n_it - 1;
      g0 += n_it;
      if (!(ok = ok && warp_wait(&bars[C::B_DQF + gl % C::NB], (gl / C::NB) & 1, wc, 45))) break;
      tc_fence_after();
      if (SPLIT && un.b >= 0) {
        // partial sums of a split global key tile: add (unscaled) into dkv_accum, as bwd_kernel
        float* acc = p.dkv_accum + (((size_t)un.z * (p.n_gk * C::BN) + (size_t)key) * 2 + wg) * D;
#pragma unroll
        for (int gg = 0; gg < D / 16; ++gg) {
          uint32_t v[16];
          tmem_ld16(t_lane + (wg == 0 ? C::T_DK : C::T_DV) + gg * 16, v);
          tmem_wait_ld(v);
          if (key < nk) {
#pragma unroll
            for (int c = 0; c < 16; c += 4)
              asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(acc + gg * 16 + c), "f"(as_f(v[c])),
                           "f"(as_f(v[c + 1])), "f"(as_f(v[c + 2])), "f"(as_f(v[c + 3]))
                           : "memory");
          }
        }
      } else {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(wg == 0 ? p.dk : p.dv) +
                             (VARLEN ? ((size_t)(un.k_tok + key) * p.va.H + un.z) * D : ((size_t)un.z * p.Nk + key) * D);
        const float mul = (wg == 0) ? p.scale : 1.f;
#pragma unroll
        for (int gg = 0; gg < D / 16; ++gg) {
          uint32_t v[16];
          tmem_ld16(t_lane + (wg == 0 ? C::T_DK : C::T_DV) + gg * 16, v);
          tmem_wait_ld(v);
          if (key < nk) store16_bf16(dst + gg * 16, v, mul);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[C::B_ACCE]);
    }
  } else {
    // ---------------------------------------------------------------- dQ warpgroup (warps 0-3)
    const int d = warp * 32 + lane;  // TMEM lane = row d of dQ^T
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
    float* stg = reinterpret_cast<float*>(smem + C::OFF_STG);
    int g0 = 0;
    bool ok = true;
    for (int u = 0;; ++u) {
      // the four warps agree before any of them reaches the named barriers below
      const int us = u % C::NU;
      if (!named_bar_and(1, 128, ok && warp_wait(&bars[C::B_UF + us], (u / C::NU) & 1, wc, 58))) break;
      const BwdUnit un = units[us];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::B_UE + us]);
      if (!un.live) break;
      const int i0 = first_step(un), n_it = unit_steps(un);
      TileSet qs{};
      if constexpr (LOCAL) qs = local_steps(un);
      const long long w0 = wrow0(un);
      // K^T into TMEM for this unit (lane d holds K[key][d] for all 128 keys as bf16 pairs,
      // lanes d >= D zeros) once K has landed and the previous unit's dQ^T MMAs are done
      ok = named_bar_and(1, 128, warp_wait(&bars[C::B_KV], u & 1, wc, 48) &&
                                     (u == 0 || warp_wait(&bars[C::B_KTE], (u - 1) & 1, wc, 59)));
      if (!ok) break;
      {
        const uint8_t* sK = smem + C::OFF_K;
        const int dc = d < D ? d : 0;
        const int chunk = dc / C::CHUNK, col = dc % C::CHUNK;
        const uint8_t* base = sK + chunk * C::K_CHUNK_BYTES + (col % 8) * 2;
        const int uu = col / 8;
        uint32_t ktr[2][32];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          uint32_t pr = 0;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int r = 2 * c + h;  // key row of the swizzled K-major tile
            const int phys = uu ^ ((r * C::ROWB >> 7) & (C::ROWB / 16 - 1));
            const uint32_t e = *reinterpret_cast<const uint16_t*>(base + r * C::ROWB + phys * 16);
            pr |= (d < D ? e : 0u) << (16 * h);
          }
          ktr[c >> 5][c & 31] = pr;
        }
        tc_fence_after();
        tmem_st32(t_lane + C::T_KT, ktr[0]);
        tmem_st32(t_lane + C::T_KT + 32, ktr[1]);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars[C::B_KT]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::B_KVE]);  // this warp's reads of K are done
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int g = g0 + it, b = g % C::NB;
        if (!(ok = named_bar_and(1, 128, warp_wait(&bars[C::B_DQR + b], (g / C::NB) & 1, wc, 46)))) break;
        tc_fence_after();
        uint32_t v0[32], v1[32];
        tmem_ld32(t_lane + C::T_S + (uint32_t)(b * 64), v0);
        tmem_ld32(t_lane + C::T_S + (uint32_t)(b * 64) + 32, v1);
        tmem_wait_ld(v0);
        reg_tie(v1);
        tc_fence_before();
        mbar_arrive(&bars[C::B_DQE + b]);
        float* gdst = p.dq_accum + ((size_t)w0 + (size_t)(LOCAL ? qs.at(it) : i0 + it) * C::BM) * D;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          named_bar_sync(1, 128);
          if (d < D) {
#pragma unroll
            for (int c = 0; c < 32; ++c) stg[(h * 32 + c) * D + d] = as_f(h == 0 ? v0[c] : v1[c]);
          }
          fence_proxy_async_smem();
          named_bar_sync(1, 128);
          if (threadIdx.x == 0) {
            bulk_reduce_add_f32(gdst + h * 32 * D, stg + h * 32 * D, C::STG_BYTES / 2);
            bulk_commit_group();
          }
        }
      }
      g0 += n_it;
    }
    if (threadIdx.x == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA_A) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------
// prep: Dlt = rowsum(dO o O), lse2 = L * log2(e) (+inf past Nq), dq_accum = 0, for the
// 64-row-padded workspace rows of one (sequence, head) per blockIdx.y.
// ------------------------------------------------------------------------------------
template <int D>
struct RowCfg {
  static constexpr int TPR = D / 8;          // threads per row, 8 bf16 each
  static constexpr int ROWS = 256 / TPR;     // rows per pass of a 256-thread block
  static constexpr int NSUB = ROWS < 64 ? 64 / ROWS : 1;  // passes per block
  static constexpr int ROWS_CTA = ROWS * NSUB;             // rows per block, a multiple of 64
};

template <int D, bool VARLEN>
__global__ void __launch_bounds__(256) prep_kernel(const PrepParams p) {
  using R = RowCfg<D>;
  constexpr int TPR = R::TPR;
  // dense: the last heads first (their O was written last, still in L2), so the first heads'
  // rows, which the main kernel takes first, are the ones left in L2 at the end
  const int bh = VARLEN ? (int)blockIdx.y : (int)gridDim.y - 1 - (int)blockIdx.y;
  const SeqView sv = seq_view<VARLEN>(p.va, p.Nq, p.Nq, bh);
  const int rows = VARLEN ? (sv.Nq + 63) / 64 * 64 : p.Nq_pad;  // padded rows of this sequence
  const int rb = blockIdx.x * R::ROWS_CTA;                       // first row of this block
  if (rb >= rows) return;  // (packed: a sequence shorter than the longest)
  const long long row0 = ws_row0(VARLEN, bh, p.Nq_pad, sv);
  const int part = threadIdx.x % TPR;
  // every pass's loads first, so NSUB 16-byte loads per tensor are in flight per thread
  uint4 a[R::NSUB], b[R::NSUB];
#pragma unroll
  for (int k = 0; k < R::NSUB; ++k) {
    const int r = rb + k * R::ROWS + threadIdx.x / TPR;
    a[k] = b[k] = make_uint4(0u, 0u, 0u, 0u);
    if (r < sv.Nq) {
      const size_t tok = VARLEN ? ((size_t)(sv.q_tok + r) * p.va.H + sv.h) : ((size_t)bh * sv.Nq + r);
      const size_t off = tok * D + part * 8;
      a[k] = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.o) + off);
      b[k] = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.dout) + off);
    }
  }
#pragma unroll
  for (int k = 0; k < R::NSUB; ++k) {
    const int r = rb + k * R::ROWS + threadIdx.x / TPR;
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[k]);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b[k]);
    float acc = 0.f;  // (zero words for rows past the sequence)
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 fa = __bfloat1622float2(a2[t]);
      const float2 fb = __bfloat1622float2(b2[t]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
#pragma unroll
    for (int w = TPR / 2; w >= 1; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (r < rows) {
      const size_t wr = (size_t)(row0 + r);
      float4* z = reinterpret_cast<float4*>(p.dq_accum + wr * D + part * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (part == 0) {
        p.dlt[wr] = acc;
        const size_t li = VARLEN ? (size_t)sv.h * p.va.total_q + sv.q_tok + r : (size_t)bh * sv.Nq + r;
        const float L = r < sv.Nq ? p.lse[li] : -INFINITY;  // -inf: the row sees no key
        p.lse2[wr] = L == -INFINITY ? INFINITY : L * 1.4426950408889634f;
      }
    }
  }
}

// ------------------------------------------------------------------------------------
// convert: dq = bf16(dq_accum * scale), rows < Nq of one (sequence, head) per blockIdx.y
// ------------------------------------------------------------------------------------
template <int D, bool VARLEN>
__global__ void __launch_bounds__(256) convert_kernel(const ConvParams p) {
  using R = RowCfg<D>;
  constexpr int TPR = R::TPR;
  // dense: the last heads first, whose dq_accum the main kernel touched last (still in L2)
  const int bh = VARLEN ? (int)blockIdx.y : (int)gridDim.y - 1 - (int)blockIdx.y;
  const SeqView sv = seq_view<VARLEN>(p.va, p.Nq, p.Nq, bh);
  const int rb = blockIdx.x * R::ROWS_CTA;
  if (rb >= sv.Nq) return;
  const int d = (threadIdx.x % TPR) * 8;
  const long long row0 = ws_row0(VARLEN, bh, p.Nq_pad, sv);
  float4 a[R::NSUB], b[R::NSUB];
#pragma unroll
  for (int k = 0; k < R::NSUB; ++k) {
    const int r = rb + k * R::ROWS + threadIdx.x / TPR;
    if (r < sv.Nq) {
      const float4* src = reinterpret_cast<const float4*>(p.dq_accum + (size_t)(row0 + r) * D + d);
      a[k] = src[0];
      b[k] = src[1];
    }
  }
#pragma unroll
  for (int k = 0; k < R::NSUB; ++k) {
    const int r = rb + k * R::ROWS + threadIdx.x / TPR;
    if (r < sv.Nq) {
      uint4 w;
      w.x = pack_bf16(a[k].x * p.scale, a[k].y * p.scale);
      w.y = pack_bf16(a[k].z * p.scale, a[k].w * p.scale);
      w.z = pack_bf16(b[k].x * p.scale, b[k].y * p.scale);
      w.w = pack_bf16(b[k].z * p.scale, b[k].w * p.scale);
      const size_t tok = VARLEN ? ((size_t)(sv.q_tok + r) * p.va.H + sv.h) : ((size_t)bh * sv.Nq + r);
      *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dq) + tok * D + d) = w;
    }
  }
}

// dK = scale * dk_accum, dV = dv_accum (bf16) for the rows of split global key tiles.
template <int D>
__global__ void __launch_bounds__(256) kv_convert_kernel(const KvConvertParams p) {
  constexpr int TPR = RowCfg<D>::TPR;
  const int bh = blockIdx.y;
  const int r = blockIdx.x * RowCfg<D>::ROWS + threadIdx.x / TPR;
  if (r >= p.n_rows || r >= p.Nk) return;
  const int d = (threadIdx.x % TPR) * 8;
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const float4* src = reinterpret_cast<const float4*>(p.dkv_accum + (((size_t)bh * p.n_rows + r) * 2 + m) * D + d);
    const float4 a = src[0], b = src[1];
    const float mul = m == 0 ? p.scale : 1.f;
    uint4 w;
    w.x = pack_bf16(a.x * mul, a.y * mul);
    w.y = pack_bf16(a.z * mul, a.w * mul);
    w.z = pack_bf16(b.x * mul, b.y * mul);
    w.w = pack_bf16(b.z * mul, b.w * mul);
    *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(m == 0 ? p.dk : p.dv) + ((size_t)bh * p.Nk + r) * D + d) = w;
  }
}

template <int D, bool CAUSAL, bool VARLEN, bool LOCAL = false>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                     const BwdParams& p, int BH, cudaStream_t st) {
  using C = Cfg<D>;
  auto kern = bwd_kernel<D, CAUSAL, VARLEN, LOCAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const int gx = (LOCAL && p.n_gk > 0) ? p.n_gk * p.n_qsplit + (p.n_k_tiles - p.n_gk) : p.n_k_tiles;
  // packed batch: compact slots of 128 keys (slot_seq), one grid row per head
  dim3 grid = VARLEN ? dim3((unsigned)((p.va.total_k >> 7) + p.va.B), (unsigned)p.va.H) : dim3((unsigned)gx, (unsigned)BH);
  kern<<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

template <int D, bool CAUSAL, bool VARLEN = false, bool LOCAL = false, bool SPLIT = false>
cudaError_t launch_persist_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                             const BwdParams& p, int BH, cudaStream_t st) {
  using C = Cfg<D>;
  auto kern = bwd_persist_kernel<D, CAUSAL, VARLEN, LOCAL, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const int gx = SPLIT ? p.n_gk * p.n_qsplit + (p.n_k_tiles - p.n_gk) : p.n_k_tiles;
  dim3 grid = VARLEN ? dim3((unsigned)((p.va.total_k >> 7) + p.va.B), (unsigned)p.va.H)
                     : dim3((unsigned)gx, (unsigned)BH);
  kern<<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t prep_t(const PrepParams& p, cudaStream_t st) {
  const int rows = p.va.cu_q ? (p.Nq + 63) / 64 * 64 : p.Nq_pad;  // varlen: padded maximum length
  dim3 grid((unsigned)((rows + RowCfg<D>::ROWS_CTA - 1) / RowCfg<D>::ROWS_CTA), (unsigned)p.BH);
  if (p.va.cu_q) prep_kernel<D, true><<<grid, 256, 0, st>>>(p);
  else prep_kernel<D, false><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t conv_t(const ConvParams& p, cudaStream_t st) {
  dim3 grid((unsigned)((p.Nq + RowCfg<D>::ROWS_CTA - 1) / RowCfg<D>::ROWS_CTA), (unsigned)p.BH);
  if (p.va.cu_q) convert_kernel<D, true><<<grid, 256, 0, st>>>(p);
  else convert_kernel<D, false><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace bwd

#define TA11_SWITCH_D(D, EXPR_T)       \
  switch (D) {                         \
    case 16: { constexpr int DD = 16; return EXPR_T; }   \
    case 32: { constexpr int DD = 32; return EXPR_T; }   \
    case 64: { constexpr int DD = 64; return EXPR_T; }   \
    case 128: { constexpr int DD = 128; return EXPR_T; } \
    default: return cudaErrorInvalidValue;               \
  }

cudaError_t launch_bwd(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, int BH, cudaStream_t st) {
  if (p.local && p.persist && p.n_gk > 0) {
    TA11_SWITCH_D(D, (causal ? bwd::launch_persist_t<DD, true, false, true, true>(tq, tk, tv, tdo, p, BH, st)
                             : bwd::launch_persist_t<DD, false, false, true, true>(tq, tk, tv, tdo, p, BH, st)))
  }
  if (p.local && p.persist) {
    TA11_SWITCH_D(D, (causal ? bwd::launch_persist_t<DD, true, false, true>(tq, tk, tv, tdo, p, BH, st)
                             : bwd::launch_persist_t<DD, false, false, true>(tq, tk, tv, tdo, p, BH, st)))
  }
  if (p.local) {
    TA11_SWITCH_D(D, (causal ? bwd::launch_t<DD, true, false, true>(tq, tk, tv, tdo, p, BH, st)
                             : bwd::launch_t<DD, false, false, true>(tq, tk, tv, tdo, p, BH, st)))
  }
  if (p.va.cu_q && p.persist) {
    TA11_SWITCH_D(D, (causal ? bwd::launch_persist_t<DD, true, true>(tq, tk, tv, tdo, p, BH, st)
                             : bwd::launch_persist_t<DD, false, true>(tq, tk, tv, tdo, p, BH, st)))
  }
  if (p.va.cu_q) {
    TA11_SWITCH_D(D, (causal ? bwd::launch_t<DD, true, true>(tq, tk, tv, tdo, p, BH, st)
                             : bwd::launch_t<DD, false, true>(tq, tk, tv, tdo, p, BH, st)))
  }
  if (p.persist) {
    TA11_SWITCH_D(D, (causal ? bwd::launch_persist_t<DD, true>(tq, tk, tv, tdo, p, BH, st)
                             : bwd::launch_persist_t<DD, false>(tq, tk, tv, tdo, p, BH, st)))
  }
  TA11_SWITCH_D(D, (causal ? bwd::launch_t<DD, true, false>(tq, tk, tv, tdo, p, BH, st)
                           : bwd::launch_t<DD, false, false>(tq, tk, tv, tdo, p, BH, st)))
}

cudaError_t launch_bwd_prep(int D, const PrepParams& p, cudaStream_t st) {
  TA11_SWITCH_D(D, bwd::prep_t<DD>(p, st))
}

cudaError_t launch_bwd_convert(int D, const ConvParams& p, cudaStream_t st) {
  TA11_SWITCH_D(D, bwd::conv_t<DD>(p, st))
}

template <int D>
cudaError_t kv_conv_t(const KvConvertParams& p, int BH, cudaStream_t st) {
  dim3 grid((unsigned)((p.n_rows + bwd::RowCfg<D>::ROWS - 1) / bwd::RowCfg<D>::ROWS), (unsigned)BH);
  bwd::kv_convert_kernel<D><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_kv_convert(int D, const KvConvertParams& p, int BH, cudaStream_t st) {
  TA11_SWITCH_D(D, kv_conv_t<DD>(p, BH, st))
}

}  // namespace ta11
