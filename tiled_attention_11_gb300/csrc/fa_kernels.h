// Parameters shared by the host launchers and the sm_103a attention kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ta11 {

// Variable-length batches: packed [total, H, D] tensors with per-sequence offsets
// cu[b] .. cu[b+1] (device int32, B+1 entries).  In that mode Nq / Nk hold the maximum
// sequence lengths, and every CTA derives its own sequence bounds (clamped to the packed
// extents, so inconsistent offsets can never make a kernel write outside its buffers).
struct VarlenArgs {
  const int* cu_q;      // null: dense [B,H,N,D] layout
  const int* cu_k;
  int H;                // heads
  int total_q, total_k; // packed token counts
  int B;                // sequences
};

// One (sequence, head) as seen by a CTA, for either layout.
struct SeqView {
  int Nq, Nk;           // this sequence's lengths
  int q_tok, k_tok;     // packed token index of row 0 (dense: 0)
  int h;                // head (varlen)
  int b;                // batch entry (varlen)
};

template <bool VARLEN>
__device__ __forceinline__ SeqView seq_view(const VarlenArgs& va, int Nq, int Nk, int by) {
  SeqView s;
  if (!VARLEN) {
    s.Nq = Nq; s.Nk = Nk; s.q_tok = 0; s.k_tok = 0; s.h = 0; s.b = 0;
    return s;
  }
  s.b = by / va.H;
  s.h = by % va.H;
  int qa = __ldg(va.cu_q + s.b), qe = __ldg(va.cu_q + s.b + 1);
  int ka = __ldg(va.cu_k + s.b), ke = __ldg(va.cu_k + s.b + 1);
  qa = max(0, min(qa, va.total_q));
  qe = max(qa, min(qe, va.total_q));
  ka = max(0, min(ka, va.total_k));
  ke = max(ka, min(ke, va.total_k));
  s.q_tok = qa;
  s.k_tok = ka;
  s.Nq = min(qe - qa, Nq);
  s.Nk = min(ke - ka, Nk);
  return s;
}

// Compact tile slots of a packed batch (one grid row per head): sequence b owns slots
// [f(b), f(b+1)) with f(b) = floor(cu[b] / 2^shift) + b.  That is at least
// ceil(len_b / 2^shift) slots (at most one more), f(B) = floor(total / 2^shift) + B in all,
// so a grid of f(B) columns launches at most B empty CTAs per head instead of one per
// tile of the longest sequence in every shorter one.
__device__ __forceinline__ int slot_base(const int* cu, int total, int shift, int b) {
  return (max(0, min(__ldg(cu + b), total)) >> shift) + b;
}

// The sequence of slot x: the largest b < B with f(b) <= x, found by 32-way probes of
// cu (one round of loads for B <= 32).  Every lane of a converged warp calls it and gets
// the answer.  cu must be nondecreasing; any other input still gives some b in [0, B).
__device__ __forceinline__ int slot_seq(const int* cu, int B, int total, int shift, int x) {
  const int lane = (int)(threadIdx.x & 31u);
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) >> 5;
    const int pos = lo + lane * step;
    const bool le = pos < hi && slot_base(cu, total, shift, pos) <= x;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    const int top = m ? 31 - __clz((int)m) : 0;
    lo += top * step;
    hi = min(lo + step, hi);
  }
  return lo;
}

// Local-window + global-token mask (absolute indices, top-left like the causal mask):
// key j is visible to query i iff j < Nk, (not causal or j <= i) and
// (i - win_l <= j <= i + win_r  or  j < n_glob  or  i < n_glob).  An unbounded side is
// stored as kUnbounded, so the comparisons need no special case and cannot overflow.
constexpr int kUnbounded = 1 << 29;
struct LocalMask {
  int win_l, win_r;     // window extents (kUnbounded: no limit)
  int n_glob;           // global tokens: the first n_glob queries and keys
};

// Tile indices [a, g) U [L, hi), ascending; make() orders and clips the bounds so the
// two parts are disjoint (g <= L) and count() is their total size.
struct TileSet {
  int a, g, L, hi;
  static __host__ __device__ __forceinline__ TileSet make(int a, int g, int L, int hi) {
    TileSet t;
    t.hi = hi > 0 ? hi : 0;
    t.a = a < 0 ? 0 : (a > t.hi ? t.hi : a);
    t.g = g < t.a ? t.a : (g > t.hi ? t.hi : g);
    t.L = L < t.g ? t.g : (L > t.hi ? t.hi : L);
    return t;
  }
  __host__ __device__ __forceinline__ int count() const { return (g - a) + (hi - L); }
  __host__ __device__ __forceinline__ int at(int n) const { return n < g - a ? a + n : L + (n - (g - a)); }
  __host__ __device__ __forceinline__ bool has(int x) const { return (x >= a && x < g) || (x >= L && x < hi); }
  // smallest member greater than x, or kNone
  static constexpr int kNone = 0x7fffffff;
  __host__ __device__ __forceinline__ int next(int x) const {
    int y = x + 1;
    if (y < a) y = a;
    if (y < g) return y;
    if (y < L) y = L;
    return y < hi ? y : kNone;
  }
};

struct FwdParams {
  void* o;              // bf16 [B,H,Nq,D] (varlen: [total_q,H,D])
  float* lse;           // fp32 [B,H,Nq] (varlen: [H,total_q]), natural log
  int Nq, Nk;           // lengths (varlen: maximum lengths)
  int n_q_tiles;        // ceil(Nq / 128)
  float scale_log2;     // scale * log2(e)
  unsigned long long wait_limit_ns;
  unsigned* status;     // device status word pair
  VarlenArgs va;
  LocalMask lm;         // used when `local` is set
  int local;            // 1: apply the local-window + global-token mask
  // Local mask, non-causal: the first n_gp query-tile pairs hold global query rows, which
  // see every key.  Each runs as n_split CTAs over key tiles [c*split_t, (c+1)*split_t)
  // that write partial results (the unnormalised O accumulator, and per row the
  // subtracted maximum m (base 2), the sum l and the sum of rounded weights lr);
  // fwd_combine merges them.  n_gp == 0: no split.
  int n_gp, n_split, split_t;
  float* part_o;        // [B*H][n_gp*256][n_split][D]
  float* part_ml;       // [B*H][n_gp*256][n_split][4]: m, l, lr, unused
  // Causal, dense layout, plain mask, launch of one wave: the sequential-tile kernel,
  // whose CTA `pair` holds query tiles pair and n_q_tiles-1-pair instead of 2*pair and
  // 2*pair+1, so every CTA walks about the same number of key tiles.
  int fold;
  // More units than one wave: the persistent kernel (a CTA takes over not-yet-started CTAs
  // of its grid instead of exiting).
  int persist;
  // persistent, causal: 0 claim units head by head; n > 0 rank-major (longest first) within
  // groups of n heads, over all heads when n >= H; packed layout: any n > 0 is slot-major
  // over all heads
  int lpt;
};

struct FwdCombineParams {
  const float* part_o;
  const float* part_ml;
  void* o;              // bf16 [B,H,Nq,D]
  float* lse;           // fp32 [B,H,Nq]
  int Nq, n_rows;       // n_rows = n_gp*256 (rows with partial records per head)
  int n_split;
};

// Backward workspace rows: dense, head bh owns rows [bh*Nq_pad, bh*Nq_pad + Nq_pad);
// varlen, head h owns Nq_pad rows (Nq_pad = 64*(ceil(total_q/64) + B)) and sequence b
// starts at row 64*(ceil(cu_q[b]/64) + b) of it: 64-row aligned, never overlapping.
__device__ __forceinline__ long long ws_row0(bool varlen, int bh, int Nq_pad, const SeqView& s) {
  if (!varlen) return (long long)bh * Nq_pad;
  return (long long)s.h * Nq_pad + 64LL * ((s.q_tok + 63) / 64 + s.b);
}

struct BwdParams {
  void* dk;             // bf16 [B,H,Nk,D] (varlen: [total_k,H,D])
  void* dv;
  float* dq_accum;      // fp32 workspace rows x D
  const float* lse2;    // fp32 workspace rows: lse * log2(e); +inf on padded rows
  const float* dlt;     // fp32 workspace rows: rowsum(dO o O); 0 on padded rows
  int Nq, Nk, Nq_pad;   // (varlen: maximum lengths, rows per head)
  int n_k_tiles;        // ceil(Nk / 128)
  float scale;          // softmax scale
  float scale_log2;     // scale * log2(e)
  unsigned long long wait_limit_ns;
  unsigned* status;
  VarlenArgs va;
  LocalMask lm;         // used when `local` is set
  int local;            // 1: apply the local-window + global-token mask
  // Local mask: the first n_gk key tiles hold global keys, which every (later) query sees.
  // Each runs as n_qsplit CTAs over query steps [c*split_q, (c+1)*split_q) that add their
  // partial dK, dV (fp32, unscaled) into dkv_accum; bwd_kv_convert writes them out.
  int n_gk, n_qsplit, split_q;
  float* dkv_accum;     // [B*H][n_gk*128][2][D] (zeroed before the launch)
  // More units than one wave: the persistent kernel (a CTA takes over not-yet-started CTAs
  // of its grid).
  int persist;
  // causal: 0 claim units head by head; n > 0 rank-major (longest first) within groups of
  // n heads, over all heads when n >= H (the one-CTA kernel: any n > 0 is over all heads);
  // packed layout, persistent: any n > 0 is slot-major over all heads
  int lpt;
};

struct KvConvertParams {
  const float* dkv_accum;
  void* dk;             // bf16 [B,H,Nk,D]
  void* dv;
  int Nk, n_rows;       // n_rows = n_gk*128
  float scale;
};

struct PrepParams {
  const void* o;        // bf16, layout as q
  const void* dout;     // bf16, layout as q
  const float* lse;     // fp32 [B,H,Nq] (varlen: [H,total_q])
  float* dq_accum;      // fp32 workspace rows x D (zeroed here)
  float* lse2;          // fp32 workspace rows
  float* dlt;           // fp32 workspace rows
  int BH, Nq, Nq_pad;   // (varlen: B*H, maximum Nq, rows per head)
  VarlenArgs va;
};

struct ConvParams {
  const float* dq_accum;  // fp32 workspace rows x D
  void* dq;               // bf16, layout as q
  int BH, Nq, Nq_pad;
  float scale;
  VarlenArgs va;
};

// FP8 forward: e4m3 Q, K [BH][N][D], V^T [BH][D][ldv]; descales are device scalars.
struct Fp8FwdParams {
  void* o;              // bf16 [B,H,Nq,D]
  float* lse;           // fp32 [B,H,Nq], natural log
  int Nq, Nk;
  float scale_log2;     // softmax scale * log2(e) (the Q and K descales are applied on top)
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  unsigned long long wait_limit_ns;
  unsigned* status;
  // more (query-tile pair, head) units than one wave: the persistent kernel
  int persist;
  // persistent, causal: 0 claim units head by head; n > 0 rank-major (longest first)
  // within groups of n heads, over all heads when n >= H
  int lpt;
};

// Host launchers (return cudaError_t of the launch).
// Launchers; p.va.cu_q != nullptr selects the variable-length layout, p.local the
// local-window + global-token mask (dense layout only).
// `to` maps O for the dense layout's bulk-store epilogue (unused by the packed layout).
cudaError_t launch_fwd(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdParams& p, int BH, cudaStream_t st);
cudaError_t launch_fwd_combine(int D, const FwdCombineParams& p, int BH, cudaStream_t st);
cudaError_t launch_bwd_prep(int D, const PrepParams& p, cudaStream_t st);
cudaError_t launch_bwd(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, int BH, cudaStream_t st);
cudaError_t launch_bwd_convert(int D, const ConvParams& p, cudaStream_t st);
cudaError_t launch_bwd_kv_convert(int D, const KvConvertParams& p, int BH, cudaStream_t st);
cudaError_t launch_fwd_fp8(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const Fp8FwdParams& p, int BH, cudaStream_t st);
// Per-tensor e4m3 quantisation: amax (device float, zeroed by the caller's stream
// order), then codes = e4m3(x * (448 / amax)) and descale = amax / 448.
cudaError_t launch_amax_bf16(const void* x, long long n, float* amax, cudaStream_t st);
cudaError_t launch_quant_e4m3(const void* x, long long n, const float* amax, void* codes, float* descale,
                              cudaStream_t st);
cudaError_t launch_quant_e4m3_t(const void* x, int BH, int N, int D, int ldt, const float* amax, void* codes_t,
                                float* descale, cudaStream_t st);
// Q, K (codes in place order) and V (codes transposed, [BH][D][ldv]) of one call: one amax
// launch over the three (amax[3], zeroed by the caller's stream order), one code launch.
cudaError_t launch_quantize_qkv(const void* q, const void* k, const void* v, int BH, int Nq, int Nk, int D,
                                void* q8, void* k8, void* vt8, int ldv, float* amax, float* descale,
                                cudaStream_t st);
cudaError_t launch_wait_probe(unsigned long long limit_ns, unsigned* status, cudaStream_t st);

}  // namespace ta11
