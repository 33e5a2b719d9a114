// Host side of the C ABI declared in include/fa.h: argument validation, TMA
// tensor-map encoding, kernel launches and the device status word.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <new>

#include "fa.h"
#include "fa_kernels.h"

namespace {

// Device-side status word pair: [0] = FA_OK or FA_ERR_TIMEOUT, [1] = wait site.
__device__ unsigned g_fa_status[2];

std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

// Forward kernel choice for the dense layout with plain masks beyond one wave: 1 the
// persistent kernel, 0 one CTA per unit (the persistent kernel's parity tests compare the two).
std::atomic<int> g_fwd_persist{1};
// The same choice for the main backward kernel.
std::atomic<int> g_bwd_persist{1};
// Longest-first claim order for causal persistent launches (over all heads up to eight
// waves, within groups of heads beyond).
std::atomic<int> g_lpt{1};
// Causal persistent launches of more than eight waves claim their units rank-major within
// groups of this many heads (0: head by head, heaviest unit of a head first).
// Measured on the B=4 H=32 N=4096 layer against head by head: forward 0.390 -> 0.364 ms with
// 16 heads (32: 0.367), backward main kernel 1.106 -> 1.077 ms with 8 or 16 (32: 1.095, its
// heads' Q, dO and dq_accum no longer fit in L2 together).
#ifndef TA11_FWD_CLAIM_GROUP
#define TA11_FWD_CLAIM_GROUP 16
#endif
#ifndef TA11_BWD_CLAIM_GROUP
#define TA11_BWD_CLAIM_GROUP 8
#endif
constexpr int kFwdClaimGroup = TA11_FWD_CLAIM_GROUP;
constexpr int kBwdClaimGroup = TA11_BWD_CLAIM_GROUP;
// Launches of up to eight waves: longest-first within groups of at most this many heads
// (the forward of B=4 H=16 N=4096 D=128 causal: 0.198 ms over all 64 heads, 0.190 with 16;
// launches of 16 heads or fewer are unaffected).
#ifndef TA11_SHORT_CLAIM_GROUP
#define TA11_SHORT_CLAIM_GROUP 16
#endif
constexpr long long kShortClaimGroup = TA11_SHORT_CLAIM_GROUP;
int short_group(size_t BH) { return (int)((long long)BH < kShortClaimGroup ? (long long)BH : kShortClaimGroup); }

// Optional events recorded around the main backward kernel (timing hook).
std::mutex g_ev_mu;
cudaEvent_t g_ev_begin = nullptr, g_ev_end = nullptr;

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::once_flag once;
  int ok = 0;               // 1: sm_103 and status word resolved
  unsigned* status = nullptr;
  int n_sm = 0;             // streaming multiprocessors
};
DeviceState g_dev[kMaxDevices];

// Resolve the current device: sm_103 check and the status word's device address.
int current_device(unsigned** status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_DEVICE;
  }
  DeviceState& s = g_dev[dev];
  std::call_once(s.once, [&]() {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    if (major != 10 || minor != 3) return;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    s.status = static_cast<unsigned*>(p);
    if (cudaDeviceGetAttribute(&s.n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    s.ok = 1;
  });
  if (!s.ok) return FA_ERR_DEVICE;
  *status = s.status;
  return FA_OK;
}

// SM count of the current device (after a successful current_device).
int current_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  return g_dev[dev].n_sm;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// 3-D bf16 tensor map over [BH][N][D] with a {chunk, box_rows, 1} box and the
// swizzle that matches a chunk row (32, 64 or 128 bytes).  Loads past N are
// zero-filled, so heads never read each other's rows.
bool make_map(CUtensorMap* m, const void* base, int D, int N, int BH, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int chunk = D < 64 ? D : 64;
  const CUtensorMapSwizzle sw = chunk == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                : chunk == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  cuuint32_t box[3] = {(cuuint32_t)chunk, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 tensor map over a packed [total][H][D] tensor: box {chunk, 1, box_rows}
// (rows of one head) lands in shared memory exactly like the dense box.
bool make_map_packed(CUtensorMap* m, const void* base, int D, int H, int total, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int chunk = D < 64 ? D : 64;
  const CUtensorMapSwizzle sw = chunk == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                : chunk == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)total};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {(cuuint32_t)chunk, 1, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D tensor map over 1-byte elements: dims {inner, rows, BH}, row stride `ld` bytes,
// box {inner (= the swizzle width, 64 or 128 bytes), box_rows, 1}.
bool make_map_u8(CUtensorMap* m, const void* base, int inner, int rows, int BH, long long ld, int box_inner,
                 int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const CUtensorMapSwizzle sw = box_inner == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)ld, (cuuint64_t)ld * rows};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Range {
  uintptr_t lo, hi;
};
Range rng(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return {a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

bool valid_d(int D) { return D == 16 || D == 32 || D == 64 || D == 128; }

// Longest sequence (and packed total) accepted.  The kernels index rows and tiles with
// 32-bit ints (row + tile size, tile counts, row + window extent), and an unbounded
// window side is stored as kUnbounded, which must reach past every row.
constexpr int kMaxLen = 1 << 29;
static_assert(kMaxLen <= ta11::kUnbounded, "an unbounded window must cover every row");
bool valid_len(int n) { return n >= 1 && n <= kMaxLen; }

// Shared size checks; returns FA_OK or a code.
int check_sizes(int B, int H, int Nq, int Nk, int D, float scale) {
  if (B < 1 || H < 1 || !valid_len(Nq) || !valid_len(Nk)) return FA_ERR_INVALID_ARG;
  if ((long long)B * H > 65535) return FA_ERR_INVALID_ARG;  // grid.y
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (!valid_d(D)) return FA_ERR_UNSUPPORTED_D;
  return FA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t dq_off, dlt_off, lse2_off, total;
  int Nq_pad;
};
WsLayout ws_layout(int B, int H, int Nq, int D) {
  WsLayout w;
  w.Nq_pad = ((Nq + 63) / 64) * 64;
  const size_t rows = (size_t)B * H * w.Nq_pad;
  w.dq_off = 0;
  w.dlt_off = round256(rows * D * 4);
  w.lse2_off = w.dlt_off + round256(rows * 4);
  w.total = w.lse2_off + round256(rows * 4);
  return w;
}

// Varlen workspace: per head 64*(ceil(total_q/64) + B) rows; sequence b starts at row
// 64*(ceil(cu_q[b]/64) + b) of its head (64-row aligned, never overlapping).
WsLayout ws_layout_varlen(int B, int H, int total_q, int D) {
  WsLayout w;
  w.Nq_pad = 64 * ((total_q + 63) / 64 + B);
  const size_t rows = (size_t)H * w.Nq_pad;
  w.dq_off = 0;
  w.dlt_off = round256(rows * D * 4);
  w.lse2_off = w.dlt_off + round256(rows * 4);
  w.total = w.lse2_off + round256(rows * 4);
  return w;
}

int check_varlen(int B, int H, int total_q, int total_k, int max_q, int max_k, int D, float scale) {
  if (B < 1 || H < 1 || !valid_len(total_q) || !valid_len(total_k) || !valid_len(max_q) || !valid_len(max_k))
    return FA_ERR_INVALID_ARG;
  if ((long long)B * H > 65535) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (!valid_d(D)) return FA_ERR_UNSUPPORTED_D;
  return FA_OK;
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace

extern "C" {

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "success";
    case FA_ERR_INVALID_ARG: return "invalid argument (null pointer, size, scale or overlapping buffers)";
    case FA_ERR_UNSUPPORTED_D: return "unsupported head dimension (D must be 16, 32, 64 or 128)";
    case FA_ERR_MISALIGNED: return "misaligned pointer (bf16 tensors need 16 bytes, lse 4 bytes)";
    case FA_ERR_WORKSPACE: return "backward workspace null, misaligned (256 bytes) or too small";
    case FA_ERR_DEVICE: return "no usable device: the current CUDA device must be sm_103 (GB300)";
    case FA_ERR_LAUNCH: return "kernel launch or TMA descriptor encoding failed";
    case FA_ERR_TIMEOUT: return "a kernel gave up a bounded wait (device status word)";
    case FA_ERR_SCRATCH_LIMIT: return "problem needs more than the 32 MiB fixed scratch of fa_bwd_noalloc";
    default: return "unknown status";
  }
}

void fa_set_wait_limit_ns(unsigned long long ns) { g_wait_limit_ns.store(ns ? ns : 1ull); }

int fa_set_fwd_persistent(int on) { return g_fwd_persist.exchange(on ? 1 : 0); }

int fa_set_bwd_persistent(int on) { return g_bwd_persist.exchange(on ? 1 : 0); }

size_t fa_bwd_workspace_size(int B, int H, int Nq, int Nk, int D) {
  if (check_sizes(B, H, Nq, Nk, D, 1.f) != FA_OK) return 0;
  return ws_layout(B, H, Nq, D).total;
}

}  // extern "C"

namespace {

// Mask arguments of the local-window entry points -> kernel form (negative: unbounded;
// global-token counts beyond both lengths change nothing and are clipped).
ta11::LocalMask local_mask(int Nq, int Nk, int window_left, int window_right, int n_global) {
  ta11::LocalMask m;
  m.win_l = (window_left < 0 || window_left >= ta11::kUnbounded) ? ta11::kUnbounded : window_left;
  m.win_r = (window_right < 0 || window_right >= ta11::kUnbounded) ? ta11::kUnbounded : window_right;
  const int nmax = Nq > Nk ? Nq : Nk;
  m.n_glob = n_global < 0 ? 0 : (n_global > nmax ? nmax : n_global);
  return m;
}

// Split of the global query rows' key range (local mask, non-causal, long key range):
// see FwdParams.  Everything zero when no split is needed.
struct FwdSplit {
  int n_gp = 0, n_split = 0, split_t = 0;
  size_t o_bytes = 0, ml_bytes = 0, total = 0;
};
constexpr int kSplitTiles = 16;  // key tiles per chunk: about one window CTA's work

FwdSplit fwd_split(int B, int H, int Nq, int Nk, int D, int causal, const ta11::LocalMask& m) {
  FwdSplit f;
  const int nk_tiles = (Nk + 127) / 128, n_pairs = (Nq + 255) / 256;
  if (causal || m.n_glob <= 0 || nk_tiles <= 2 * kSplitTiles) return f;
  f.n_gp = (m.n_glob + 255) / 256 < n_pairs ? (m.n_glob + 255) / 256 : n_pairs;
  f.split_t = kSplitTiles;
  f.n_split = (nk_tiles + kSplitTiles - 1) / kSplitTiles;
  const size_t recs = (size_t)B * H * f.n_gp * 256 * f.n_split;
  f.o_bytes = (recs * D * 4 + 255) / 256 * 256;
  f.ml_bytes = (recs * 16 + 255) / 256 * 256;
  f.total = f.o_bytes + f.ml_bytes;
  return f;
}

int fwd_dense(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk, int D,
              float scale, int causal, const ta11::LocalMask* lm, cudaStream_t stream, void* workspace = nullptr,
              size_t workspace_bytes = 0) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  int rc = check_sizes(B, H, Nq, Nk, D, scale);
  if (rc != FA_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_MISALIGNED;
  const size_t BH = (size_t)B * H;
  const Range rq = rng(q, BH * Nq * D * 2), rk = rng(k, BH * Nk * D * 2), rv = rng(v, BH * Nk * D * 2);
  const Range ro = rng(o, BH * Nq * D * 2), rl = rng(lse, BH * Nq * 4);
  for (Range out : {ro, rl})
    for (Range in : {rq, rk, rv})
      if (overlap(out, in)) return FA_ERR_INVALID_ARG;
  if (overlap(ro, rl)) return FA_ERR_INVALID_ARG;

  FwdSplit split;
  if (lm) {
    split = fwd_split(B, H, Nq, Nk, D, causal, *lm);
    if (split.n_gp > 0) {
      if (!workspace || !aligned(workspace, 256) || workspace_bytes < split.total) return FA_ERR_WORKSPACE;
      const Range rw = rng(workspace, split.total);
      for (Range r : {rq, rk, rv, ro, rl})
        if (overlap(rw, r)) return FA_ERR_INVALID_ARG;
    }
  }

  unsigned* status = nullptr;
  rc = current_device(&status);
  if (rc != FA_OK) return rc;

  CUtensorMap tq, tk, tv, to;
  if (!make_map(&tq, q, D, Nq, (int)BH, 128) || !make_map(&tk, k, D, Nk, (int)BH, 128) ||
      !make_map(&tv, v, D, Nk, (int)BH, 128) || !make_map(&to, o, D, Nq, (int)BH, 128))
    return FA_ERR_LAUNCH;
  ta11::FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_q_tiles = (Nq + 127) / 128;
  p.scale_log2 = scale * kLog2e;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.status = status;
  // Causal launches that fit in one wave are bound by their heaviest CTA: fold the pairs
  // (tile t with tile n-1-t) so that every CTA walks about the same number of key tiles.
  const long long n_ctas = (long long)BH * ((p.n_q_tiles + 1) / 2);
  p.fold = (!lm && causal && n_ctas <= current_sms()) ? 1 : 0;
  // persistent CTAs beyond one wave (with the local mask, split global rows' key chunks
  // included: the split is non-causal only)
  p.persist = (!p.fold && n_ctas > current_sms()) ? g_fwd_persist.load() : 0;
  // causal launches of up to eight waves: longest-first over all heads, so no head's
  // heaviest pairs start last (the layer's 13 waves keep head-by-head order for L2 locality)
  p.lpt = (!lm && p.persist && causal && g_lpt.load())
              ? (n_ctas <= 8LL * current_sms() ? short_group(BH) : kFwdClaimGroup) : 0;
  if (lm) {
    p.lm = *lm;
    p.local = 1;
    if (split.n_gp > 0) {
      p.n_gp = split.n_gp;
      p.n_split = split.n_split;
      p.split_t = split.split_t;
      p.part_o = static_cast<float*>(workspace);
      p.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + split.o_bytes);
    }
  }
  if (ta11::launch_fwd(D, causal != 0, tq, tk, tv, to, p, (int)BH, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  if (split.n_gp > 0) {
    ta11::FwdCombineParams cp{p.part_o, p.part_ml, o, lse, Nq, split.n_gp * 256, split.n_split};
    if (ta11::launch_fwd_combine(D, cp, (int)BH, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

// Split of the global key tiles' query range (local mask with global tokens, long query
// range): see BwdParams.  Everything zero when no split is needed.
struct BwdSplit {
  int n_gk = 0, n_qsplit = 0, split_q = 0;
  size_t bytes = 0;
};
constexpr int kSplitSteps = 32;  // 64-query steps per chunk

BwdSplit bwd_split(int B, int H, int Nq, int Nk, int D, const ta11::LocalMask& m) {
  BwdSplit f;
  const int nk_tiles = (Nk + 127) / 128, n_qt = (Nq + 63) / 64;
  if (m.n_glob <= 0 || n_qt <= 2 * kSplitSteps) return f;
  f.n_gk = (m.n_glob + 127) / 128 < nk_tiles ? (m.n_glob + 127) / 128 : nk_tiles;
  f.split_q = kSplitSteps;
  f.n_qsplit = (n_qt + kSplitSteps - 1) / kSplitSteps;
  f.bytes = ((size_t)B * H * f.n_gk * 128 * 2 * D * 4 + 255) / 256 * 256;
  return f;
}

int bwd_dense(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
              void* dk, void* dv, int B, int H, int Nq, int Nk, int D, float scale, int causal,
              const ta11::LocalMask* lm, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  int rc = check_sizes(B, H, Nq, Nk, D, scale);
  if (rc != FA_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return FA_ERR_MISALIGNED;
  const WsLayout w = ws_layout(B, H, Nq, D);
  const BwdSplit split = lm ? bwd_split(B, H, Nq, Nk, D, *lm) : BwdSplit{};
  const size_t ws_need = w.total + split.bytes;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < ws_need) return FA_ERR_WORKSPACE;
  const size_t BH = (size_t)B * H;
  const size_t nq_b = BH * Nq * D * 2, nk_b = BH * Nk * D * 2;
  const Range ins[] = {rng(q, nq_b), rng(k, nk_b), rng(v, nk_b), rng(o, nq_b), rng(lse, BH * Nq * 4), rng(dO, nq_b)};
  const Range outs[] = {rng(dq, nq_b), rng(dk, nk_b), rng(dv, nk_b), rng(workspace, ws_need)};
  for (int a = 0; a < 4; ++a) {
    for (const Range& in : ins)
      if (overlap(outs[a], in)) return FA_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlap(outs[a], outs[b])) return FA_ERR_INVALID_ARG;
  }

  unsigned* status = nullptr;
  rc = current_device(&status);
  if (rc != FA_OK) return rc;

  CUtensorMap tq, tk, tv, tdo;
  if (!make_map(&tq, q, D, Nq, (int)BH, 64) || !make_map(&tk, k, D, Nk, (int)BH, 128) ||
      !make_map(&tv, v, D, Nk, (int)BH, 128) || !make_map(&tdo, dO, D, Nq, (int)BH, 64))
    return FA_ERR_LAUNCH;

  char* ws = static_cast<char*>(workspace);
  float* dq_accum = reinterpret_cast<float*>(ws + w.dq_off);
  float* dlt = reinterpret_cast<float*>(ws + w.dlt_off);
  float* lse2 = reinterpret_cast<float*>(ws + w.lse2_off);

  ta11::PrepParams pp{o, dO, lse, dq_accum, lse2, dlt, (int)BH, Nq, w.Nq_pad, {}};  // dense: no varlen view
  if (ta11::launch_bwd_prep(D, pp, stream) != cudaSuccess) return FA_ERR_LAUNCH;

  ta11::BwdParams bp{};
  bp.dk = dk;
  bp.dv = dv;
  bp.dq_accum = dq_accum;
  bp.lse2 = lse2;
  bp.dlt = dlt;
  bp.Nq = Nq;
  bp.Nk = Nk;
  bp.Nq_pad = w.Nq_pad;
  bp.n_k_tiles = (Nk + 127) / 128;
  bp.scale = scale;
  bp.scale_log2 = scale * kLog2e;
  bp.wait_limit_ns = g_wait_limit_ns.load();
  bp.status = status;
  float* dkv_accum = nullptr;
  if (lm) {
    bp.lm = *lm;
    bp.local = 1;
    if (split.n_gk > 0) {
      dkv_accum = reinterpret_cast<float*>(ws + w.total);
      if (cudaMemsetAsync(dkv_accum, 0, split.bytes, stream) != cudaSuccess) return FA_ERR_LAUNCH;
      bp.n_gk = split.n_gk;
      bp.n_qsplit = split.n_qsplit;
      bp.split_q = split.split_q;
      bp.dkv_accum = dkv_accum;
    }
  }
  // persistent kernel: more CTAs than one wave.  It saves a fixed time per unit; with
  // D = 128 and more than 128 query steps per unit it measured about 1% slower than one CTA
  // per unit, so those keep one CTA per unit.  A window mask keeps units short whatever Nq
  // is (a split global key tile's chunks included).
  const bool short_units = lm || D < 128 || Nq <= 8192;
  bp.persist = (short_units && (long long)bp.n_k_tiles * BH > current_sms()) ? g_bwd_persist.load() : 0;
  // causal launches of a few waves (persistent or not): longest-first over all heads
  bp.lpt = (!lm && causal && g_lpt.load())
               ? ((long long)bp.n_k_tiles * BH <= 8LL * current_sms() ? short_group(BH)
                                                                         : (bp.persist ? kBwdClaimGroup : 0))
               : 0;
  cudaEvent_t ev_b = nullptr, ev_e = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_ev_mu);
    ev_b = g_ev_begin;
    ev_e = g_ev_end;
  }
  if (ev_b && ev_e && cudaEventRecord(ev_b, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  if (ta11::launch_bwd(D, causal != 0, tq, tk, tv, tdo, bp, (int)BH, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  if (ev_b && ev_e && cudaEventRecord(ev_e, stream) != cudaSuccess) return FA_ERR_LAUNCH;

  ta11::ConvParams cp{dq_accum, dq, (int)BH, Nq, w.Nq_pad, scale, {}};  // dense: no varlen view
  if (ta11::launch_bwd_convert(D, cp, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  if (split.n_gk > 0) {
    ta11::KvConvertParams kp{dkv_accum, dk, dv, Nk, split.n_gk * 128, scale};
    if (ta11::launch_bwd_kv_convert(D, kp, (int)BH, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk, int D,
           float scale, int causal, cudaStream_t stream) {
  return fwd_dense(q, k, v, o, lse, B, H, Nq, Nk, D, scale, causal, nullptr, stream);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
           void* dk, void* dv, int B, int H, int Nq, int Nk, int D, float scale, int causal, void* workspace,
           size_t workspace_bytes, cudaStream_t stream) {
  return bwd_dense(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, D, scale, causal, nullptr, workspace,
                   workspace_bytes, stream);
}

size_t fa_fwd_window_workspace_size(int B, int H, int Nq, int Nk, int D, int causal, int window_left,
                                    int window_right, int n_global) {
  if (check_sizes(B, H, Nq, Nk, D, 1.f) != FA_OK) return 0;
  return fwd_split(B, H, Nq, Nk, D, causal, local_mask(Nq, Nk, window_left, window_right, n_global)).total;
}

int fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                  int D, float scale, int causal, int window_left, int window_right, int n_global, void* workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
  const ta11::LocalMask m = local_mask(Nq, Nk, window_left, window_right, n_global);
  return fwd_dense(q, k, v, o, lse, B, H, Nq, Nk, D, scale, causal, &m, stream, workspace, workspace_bytes);
}

size_t fa_bwd_window_workspace_size(int B, int H, int Nq, int Nk, int D, int window_left, int window_right,
                                    int n_global) {
  if (check_sizes(B, H, Nq, Nk, D, 1.f) != FA_OK) return 0;
  return ws_layout(B, H, Nq, D).total + bwd_split(B, H, Nq, Nk, D, local_mask(Nq, Nk, window_left, window_right, n_global)).bytes;
}

int fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int D, float scale, int causal,
                  int window_left, int window_right, int n_global, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream) {
  const ta11::LocalMask m = local_mask(Nq, Nk, window_left, window_right, n_global);
  return bwd_dense(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, D, scale, causal, &m, workspace, workspace_bytes,
                   stream);
}

int fa_device_status(unsigned* site, int reset) {
  unsigned* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_LAUNCH;
  unsigned h[2] = {0, 0};
  if (cudaMemcpyFromSymbol(h, g_fa_status, sizeof(h)) != cudaSuccess) return FA_ERR_LAUNCH;
  if (site) *site = h[1];
  if (reset) {
    const unsigned z[2] = {0, 0};
    if (cudaMemcpyToSymbol(g_fa_status, z, sizeof(z)) != cudaSuccess) return FA_ERR_LAUNCH;
  }
  return h[0] == 0 ? FA_OK : (int)h[0];
}

void fa_set_bwd_main_events(cudaEvent_t begin, cudaEvent_t end) {
  std::lock_guard<std::mutex> lk(g_ev_mu);
  g_ev_begin = (begin && end) ? begin : nullptr;
  g_ev_end = (begin && end) ? end : nullptr;
}

int fa_wait_probe(unsigned long long limit_ns, cudaStream_t stream) {
  unsigned* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  return ta11::launch_wait_probe(limit_ns, status, stream) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // extern "C"

// ------------------------------------------------------------------------------------
// fa_graph_*: one fwd + bwd step captured into a CUDA graph.
// ------------------------------------------------------------------------------------
struct fa_graph_st {
  cudaGraphExec_t exec = nullptr;
};

extern "C" int fa_graph_create(const void* q, const void* k, const void* v, void* o, float* lse, const void* dO,
                               void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int D, float scale,
                               int causal, void* workspace, size_t workspace_bytes, fa_graph* out) {
  if (!out) return FA_ERR_INVALID_ARG;
  *out = nullptr;
  unsigned* status = nullptr;
  int rc = current_device(&status);  // one-time per-device set-up happens outside the capture
  if (rc != FA_OK) return rc;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  // An uncaptured call first: validates the arguments, loads the kernels and sets their
  // attributes, so the capture below records launches only.
  rc = fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, D, scale, causal, s);
  if (rc == FA_OK)
    rc = fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, D, scale, causal, workspace, workspace_bytes, s);
  if (rc == FA_OK && cudaStreamSynchronize(s) != cudaSuccess) rc = FA_ERR_LAUNCH;
  cudaGraph_t graph = nullptr;
  if (rc == FA_OK) {
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      rc = FA_ERR_LAUNCH;
    } else {
      rc = fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, D, scale, causal, s);
      if (rc == FA_OK)
        rc = fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, D, scale, causal, workspace, workspace_bytes, s);
      if (cudaStreamEndCapture(s, &graph) != cudaSuccess && rc == FA_OK) rc = FA_ERR_LAUNCH;
    }
  }
  cudaGraphExec_t exec = nullptr;
  if (rc == FA_OK && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) rc = FA_ERR_LAUNCH;
  if (graph) cudaGraphDestroy(graph);
  cudaStreamDestroy(s);
  if (rc != FA_OK) {
    cudaGetLastError();
    if (exec) cudaGraphExecDestroy(exec);
    return rc;
  }
  fa_graph g = new (std::nothrow) fa_graph_st;
  if (!g) {
    cudaGraphExecDestroy(exec);
    return FA_ERR_LAUNCH;
  }
  g->exec = exec;
  *out = g;
  return FA_OK;
}

extern "C" int fa_graph_launch(fa_graph g, cudaStream_t stream) {
  if (!g || !g->exec) return FA_ERR_INVALID_ARG;
  return cudaGraphLaunch(g->exec, stream) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

extern "C" void fa_graph_destroy(fa_graph g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  delete g;
}

// ------------------------------------------------------------------------------------
// fa_bwd_noalloc: the backward with its scratch in a fixed device array, for
// callers that cannot allocate device memory (see include/fa.h).
// ------------------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB, held by every device that loads the library

// File-scope device scratch.  In host code this name is only a host-side stand-in:
// its device address must be obtained with cudaGetSymbolAddress on each device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
  std::mutex mu;
  void* scratch = nullptr;  // device address of g_noalloc_scratch on this device (null: not looked up yet)
};
NoAllocDevice g_noalloc_dev[kMaxDevices];

// Set-up per device, run with that device current: the array's device address.  A
// failed lookup is not remembered, so a later call (outside a stream capture, say)
// tries again.
void* noalloc_scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  NoAllocDevice& s = g_noalloc_dev[dev];
  std::lock_guard<std::mutex> lk(s.mu);
  if (!s.scratch) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    s.scratch = ptr;
  }
  return s.scratch;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dO, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int D,
                              float scale, int causal, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  int rc = check_sizes(B, H, Nq, Nk, D, scale);
  if (rc != FA_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return FA_ERR_MISALIGNED;
  if (ws_layout(B, H, Nq, D).total > kNoAllocScratchBytes) return FA_ERR_SCRATCH_LIMIT;
  unsigned* status = nullptr;
  rc = current_device(&status);
  if (rc != FA_OK) return rc;
  void* ws = noalloc_scratch_for_current_device();
  if (!ws) return FA_ERR_DEVICE;
  // The same launch sequence as fa_bwd, with the fixed array as its workspace.  Its
  // preprocess kernel rewrites every scratch word the call reads (it zeroes dq_accum and
  // fills Dlt and L*log2(e)), so the previous call's contents never leak in.
  return bwd_dense(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, D, scale, causal, nullptr, ws,
                   kNoAllocScratchBytes, stream);
}

// ------------------------------------------------------------------------------------
// Variable-length batches: packed [total, H, D] tensors, sequences cu[b] .. cu[b+1].
// ------------------------------------------------------------------------------------
extern "C" int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                             const int* cu_seqlens_k, int B, int H, int total_q, int total_k, int max_seqlen_q,
                             int max_seqlen_k, int D, float scale, int causal, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse || !cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARG;
  int rc = check_varlen(B, H, total_q, total_k, max_seqlen_q, max_seqlen_k, D, scale);
  if (rc != FA_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
    return FA_ERR_MISALIGNED;
  const size_t tq_b = (size_t)total_q * H * D * 2, tk_b = (size_t)total_k * H * D * 2;
  const Range ins[] = {rng(q, tq_b), rng(k, tk_b), rng(v, tk_b), rng(cu_seqlens_q, (size_t)(B + 1) * 4),
                       rng(cu_seqlens_k, (size_t)(B + 1) * 4)};
  const Range ro = rng(o, tq_b), rl = rng(lse, (size_t)H * total_q * 4);
  for (const Range& in : ins)
    if (overlap(ro, in) || overlap(rl, in)) return FA_ERR_INVALID_ARG;
  if (overlap(ro, rl)) return FA_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  rc = current_device(&status);
  if (rc != FA_OK) return rc;
  CUtensorMap tq, tk, tv;
  if (!make_map_packed(&tq, q, D, H, total_q, 128) || !make_map_packed(&tk, k, D, H, total_k, 128) ||
      !make_map_packed(&tv, v, D, H, total_k, 128))
    return FA_ERR_LAUNCH;
  // (the packed layout stores O row by row: a bulk store of a tile would write past a
  // sequence's end into the next one; its O map argument is unused)
  ta11::FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.Nq = max_seqlen_q;
  p.Nk = max_seqlen_k;
  p.n_q_tiles = (max_seqlen_q + 127) / 128;
  p.scale_log2 = scale * kLog2e;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.status = status;
  p.va = ta11::VarlenArgs{cu_seqlens_q, cu_seqlens_k, H, total_q, total_k, B};
  // persistent CTAs beyond one wave (compact slots of 256 queries per head, see slot_seq)
  p.persist = ((long long)((total_q >> 8) + B) * H > current_sms()) ? g_fwd_persist.load() : 0;
  // causal packed batches: slot-major claim order over the heads, so a long sequence's
  // heaviest pairs do not start at the end of the launch for the last heads
  p.lpt = (p.persist && causal) ? g_lpt.load() : 0;
  return ta11::launch_fwd(D, causal != 0, tq, tk, tv, tq, p, B * H, stream) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

extern "C" size_t fa_bwd_varlen_workspace_size(int B, int H, int total_q, int max_seqlen_q, int D) {
  if (check_varlen(B, H, total_q, 1, max_seqlen_q, 1, D, 1.f) != FA_OK) return 0;
  return ws_layout_varlen(B, H, total_q, D).total;
}

extern "C" int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dO, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                             const int* cu_seqlens_k, int B, int H, int total_q, int total_k, int max_seqlen_q,
                             int max_seqlen_k, int D, float scale, int causal, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !cu_seqlens_q || !cu_seqlens_k)
    return FA_ERR_INVALID_ARG;
  int rc = check_varlen(B, H, total_q, total_k, max_seqlen_q, max_seqlen_k, D, scale);
  if (rc != FA_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) || !aligned(cu_seqlens_q, 4) ||
      !aligned(cu_seqlens_k, 4))
    return FA_ERR_MISALIGNED;
  const WsLayout w = ws_layout_varlen(B, H, total_q, D);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < w.total) return FA_ERR_WORKSPACE;
  const size_t tq_b = (size_t)total_q * H * D * 2, tk_b = (size_t)total_k * H * D * 2;
  const Range ins[] = {rng(q, tq_b), rng(k, tk_b), rng(v, tk_b), rng(o, tq_b), rng(lse, (size_t)H * total_q * 4),
                       rng(dO, tq_b), rng(cu_seqlens_q, (size_t)(B + 1) * 4), rng(cu_seqlens_k, (size_t)(B + 1) * 4)};
  const Range outs[] = {rng(dq, tq_b), rng(dk, tk_b), rng(dv, tk_b), rng(workspace, w.total)};
  for (int a = 0; a < 4; ++a) {
    for (const Range& in : ins)
      if (overlap(outs[a], in)) return FA_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlap(outs[a], outs[b])) return FA_ERR_INVALID_ARG;
  }
  unsigned* status = nullptr;
  rc = current_device(&status);
  if (rc != FA_OK) return rc;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_map_packed(&tq, q, D, H, total_q, 64) || !make_map_packed(&tk, k, D, H, total_k, 128) ||
      !make_map_packed(&tv, v, D, H, total_k, 128) || !make_map_packed(&tdo, dO, D, H, total_q, 64))
    return FA_ERR_LAUNCH;
  char* ws = static_cast<char*>(workspace);
  float* dq_accum = reinterpret_cast<float*>(ws + w.dq_off);
  float* dlt = reinterpret_cast<float*>(ws + w.dlt_off);
  float* lse2 = reinterpret_cast<float*>(ws + w.lse2_off);
  const ta11::VarlenArgs va{cu_seqlens_q, cu_seqlens_k, H, total_q, total_k, B};
  ta11::PrepParams pp{o, dO, lse, dq_accum, lse2, dlt, B * H, max_seqlen_q, w.Nq_pad, va};
  if (ta11::launch_bwd_prep(D, pp, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  ta11::BwdParams bp{};
  bp.dk = dk;
  bp.dv = dv;
  bp.dq_accum = dq_accum;
  bp.lse2 = lse2;
  bp.dlt = dlt;
  bp.Nq = max_seqlen_q;
  bp.Nk = max_seqlen_k;
  bp.Nq_pad = w.Nq_pad;
  bp.n_k_tiles = (max_seqlen_k + 127) / 128;
  bp.scale = scale;
  bp.scale_log2 = scale * kLog2e;
  bp.wait_limit_ns = g_wait_limit_ns.load();
  bp.status = status;
  bp.va = va;
  // persistent kernel beyond one wave of compact 128-key slots (slot_seq), as for the dense layout
  bp.persist = ((D < 128 || max_seqlen_q <= 8192) && (long long)((total_k >> 7) + B) * H > current_sms())
                   ? g_bwd_persist.load() : 0;
  bp.lpt = (bp.persist && causal) ? g_lpt.load() : 0;  // (as the forward: slot-major over the heads)
  if (ta11::launch_bwd(D, causal != 0, tq, tk, tv, tdo, bp, B * H, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  ta11::ConvParams cp{dq_accum, dq, B * H, max_seqlen_q, w.Nq_pad, scale, va};
  if (ta11::launch_bwd_convert(D, cp, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  return FA_OK;
}

// ------------------------------------------------------------------------------------
// FP8 (e4m3) forward and the per-tensor quantisation feeding it
// ------------------------------------------------------------------------------------
extern "C" int fa_quantize_e4m3(const void* x, long long n, void* codes, float* amax, float* descale,
                                cudaStream_t stream) {
  if (!x || !codes || !amax || !descale || n < 1) return FA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(amax, 4) || !aligned(descale, 4)) return FA_ERR_MISALIGNED;
  const Range rx = rng(x, (size_t)n * 2), rc = rng(codes, (size_t)n), ra = rng(amax, 4), rd = rng(descale, 4);
  if (overlap(rc, rx) || overlap(ra, rx) || overlap(rd, rx) || overlap(rc, ra) || overlap(rc, rd) || overlap(ra, rd))
    return FA_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  int rc_dev = current_device(&status);
  if (rc_dev != FA_OK) return rc_dev;
  if (cudaMemsetAsync(amax, 0, 4, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  if (ta11::launch_amax_bf16(x, n, amax, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  return ta11::launch_quant_e4m3(x, n, amax, codes, descale, stream) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

extern "C" int fa_quantize_e4m3_transposed(const void* x, int B, int H, int N, int D, int ldt, void* codes_t,
                                           float* amax, float* descale, cudaStream_t stream) {
  if (!x || !codes_t || !amax || !descale) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || !valid_len(N) || (long long)B * H > 65535 || ldt < N || ldt % 16 != 0)
    return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED_D;
  if (!aligned(x, 16) || !aligned(codes_t, 16) || !aligned(amax, 4) || !aligned(descale, 4)) return FA_ERR_MISALIGNED;
  const size_t BH = (size_t)B * H;
  const Range rx = rng(x, BH * N * D * 2), rc = rng(codes_t, BH * D * ldt), ra = rng(amax, 4), rd = rng(descale, 4);
  if (overlap(rc, rx) || overlap(ra, rx) || overlap(rd, rx) || overlap(rc, ra) || overlap(rc, rd) || overlap(ra, rd))
    return FA_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  int rc_dev = current_device(&status);
  if (rc_dev != FA_OK) return rc_dev;
  if (cudaMemsetAsync(amax, 0, 4, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  if (ta11::launch_amax_bf16(x, (long long)BH * N * D, amax, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  return ta11::launch_quant_e4m3_t(x, (int)BH, N, D, ldt, amax, codes_t, descale, stream) == cudaSuccess
             ? FA_OK
             : FA_ERR_LAUNCH;
}

extern "C" int fa_quantize_qkv_e4m3(const void* q, const void* k, const void* v, int B, int H, int Nq, int Nk,
                                    int D, void* q8, void* k8, void* vt8, int ldv, float* amax, float* descale,
                                    cudaStream_t stream) {
  if (!q || !k || !v || !q8 || !k8 || !vt8 || !amax || !descale) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || !valid_len(Nq) || !valid_len(Nk) || (long long)B * H > 65535 || ldv < Nk || ldv % 16 != 0)
    return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED_D;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q8, 16) || !aligned(k8, 16) ||
      !aligned(vt8, 16) || !aligned(amax, 4) || !aligned(descale, 4))
    return FA_ERR_MISALIGNED;
  const size_t BH = (size_t)B * H;
  const Range ins[] = {rng(q, BH * Nq * D * 2), rng(k, BH * Nk * D * 2), rng(v, BH * Nk * D * 2)};
  const Range outs[] = {rng(q8, BH * Nq * D), rng(k8, BH * Nk * D), rng(vt8, BH * D * ldv), rng(amax, 12),
                        rng(descale, 12)};
  for (int a = 0; a < 5; ++a) {
    for (const Range& in : ins)
      if (overlap(outs[a], in)) return FA_ERR_INVALID_ARG;
    for (int b = a + 1; b < 5; ++b)
      if (overlap(outs[a], outs[b])) return FA_ERR_INVALID_ARG;
  }
  unsigned* status = nullptr;
  int rc_dev = current_device(&status);
  if (rc_dev != FA_OK) return rc_dev;
  if (cudaMemsetAsync(amax, 0, 12, stream) != cudaSuccess) return FA_ERR_LAUNCH;
  return ta11::launch_quantize_qkv(q, k, v, (int)BH, Nq, Nk, D, q8, k8, vt8, ldv, amax, descale, stream) ==
                 cudaSuccess
             ? FA_OK
             : FA_ERR_LAUNCH;
}

extern "C" int fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, int ldv, const float* q_descale,
                          const float* k_descale, const float* v_descale, void* o, float* lse, int B, int H, int Nq,
                          int Nk, int D, float scale, int causal, cudaStream_t stream) {
  if (!q8 || !k8 || !vt8 || !q_descale || !k_descale || !v_descale || !o || !lse) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || !valid_len(Nq) || !valid_len(Nk) || (long long)B * H > 65535) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED_D;
  if (ldv < Nk || ldv % 16 != 0) return FA_ERR_INVALID_ARG;
  if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(vt8, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(q_descale, 4) || !aligned(k_descale, 4) || !aligned(v_descale, 4))
    return FA_ERR_MISALIGNED;
  const size_t BH = (size_t)B * H;
  const Range ins[] = {rng(q8, BH * Nq * D), rng(k8, BH * Nk * D), rng(vt8, BH * D * (size_t)ldv),
                       rng(q_descale, 4), rng(k_descale, 4), rng(v_descale, 4)};
  const Range ro = rng(o, BH * Nq * D * 2), rl = rng(lse, BH * Nq * 4);
  for (const Range& in : ins)
    if (overlap(ro, in) || overlap(rl, in)) return FA_ERR_INVALID_ARG;
  if (overlap(ro, rl)) return FA_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  CUtensorMap tq, tk, tv;
  if (!make_map_u8(&tq, q8, D, Nq, (int)BH, D, D, 128) || !make_map_u8(&tk, k8, D, Nk, (int)BH, D, D, 128) ||
      !make_map_u8(&tv, vt8, Nk, D, (int)BH, ldv, 128, D))
    return FA_ERR_LAUNCH;
  ta11::Fp8FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.Nq = Nq;
  p.Nk = Nk;
  p.scale_log2 = scale * kLog2e;
  p.q_descale = q_descale;
  p.k_descale = k_descale;
  p.v_descale = v_descale;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.status = status;
  // persistent CTAs beyond one wave; past 16384 queries per head the units are long enough
  // that one CTA per unit measured 1% faster
  p.persist = (Nq <= 16384 && (long long)((Nq + 255) / 256) * BH > current_sms()) ? g_fwd_persist.load() : 0;
  p.lpt = (p.persist && causal && g_lpt.load())
              ? ((long long)((Nq + 255) / 256) * BH <= 8LL * current_sms() ? short_group(BH) : kFwdClaimGroup)
              : 0;
  return ta11::launch_fwd_fp8(D, causal != 0, tq, tk, tv, p, (int)BH, stream) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// ------------------------------------------------------------------------------------
// One training step from pinned host buffers: copies in, forward, backward, copies out
// ------------------------------------------------------------------------------------
namespace {

struct StepLayout {
  size_t q, k, v, dO, o, lse, dq, dk, dv, ws, total;
};

StepLayout step_layout(int B, int H, int Nq, int Nk, int D) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t BH = (size_t)B * H, nq = up(BH * Nq * D * 2), nk = up(BH * Nk * D * 2), nl = up(BH * Nq * 4);
  StepLayout L{};
  size_t off = 0;
  L.q = off; off += nq;
  L.k = off; off += nk;
  L.v = off; off += nk;
  L.dO = off; off += nq;
  L.o = off; off += nq;
  L.lse = off; off += nl;
  L.dq = off; off += nq;
  L.dk = off; off += nk;
  L.dv = off; off += nk;
  L.ws = off; off += up(ws_layout(B, H, Nq, D).total);
  L.total = off;
  return L;
}

}  // namespace

extern "C" size_t fa_step_host_device_bytes(int B, int H, int Nq, int Nk, int D) {
  if (check_sizes(B, H, Nq, Nk, D, 1.f) != FA_OK) return 0;
  return step_layout(B, H, Nq, Nk, D).total;
}

extern "C" int fa_step_host(const void* q_h, const void* k_h, const void* v_h, const void* do_h, void* o_h,
                            float* lse_h, void* dq_h, void* dk_h, void* dv_h, void* dev, size_t dev_bytes, int B,
                            int H, int Nq, int Nk, int D, float scale, int causal, cudaStream_t stream) {
  if (!q_h || !k_h || !v_h || !do_h || !o_h || !lse_h || !dq_h || !dk_h || !dv_h || !dev) return FA_ERR_INVALID_ARG;
  int rc = check_sizes(B, H, Nq, Nk, D, scale);
  if (rc != FA_OK) return rc;
  const StepLayout L = step_layout(B, H, Nq, Nk, D);
  if (!aligned(dev, 256) || dev_bytes < L.total) return FA_ERR_WORKSPACE;
  unsigned* status = nullptr;
  rc = current_device(&status);
  if (rc != FA_OK) return rc;
  char* d = static_cast<char*>(dev);
  const size_t BH = (size_t)B * H, nq = BH * Nq * D * 2, nk = BH * Nk * D * 2, nl = BH * Nq * 4;
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  if (cudaMemcpyAsync(d + L.q, q_h, nq, h2d, stream) != cudaSuccess ||
      cudaMemcpyAsync(d + L.k, k_h, nk, h2d, stream) != cudaSuccess ||
      cudaMemcpyAsync(d + L.v, v_h, nk, h2d, stream) != cudaSuccess ||
      cudaMemcpyAsync(d + L.dO, do_h, nq, h2d, stream) != cudaSuccess)
    return FA_ERR_LAUNCH;
  rc = fa_fwd(d + L.q, d + L.k, d + L.v, d + L.o, reinterpret_cast<float*>(d + L.lse), B, H, Nq, Nk, D, scale,
              causal, stream);
  if (rc != FA_OK) return rc;
  rc = fa_bwd(d + L.q, d + L.k, d + L.v, d + L.o, reinterpret_cast<float*>(d + L.lse), d + L.dO, d + L.dq,
              d + L.dk, d + L.dv, B, H, Nq, Nk, D, scale, causal, d + L.ws, L.total - L.ws, stream);
  if (rc != FA_OK) return rc;
  if (cudaMemcpyAsync(o_h, d + L.o, nq, d2h, stream) != cudaSuccess ||
      cudaMemcpyAsync(lse_h, d + L.lse, nl, d2h, stream) != cudaSuccess ||
      cudaMemcpyAsync(dq_h, d + L.dq, nq, d2h, stream) != cudaSuccess ||
      cudaMemcpyAsync(dk_h, d + L.dk, nk, d2h, stream) != cudaSuccess ||
      cudaMemcpyAsync(dv_h, d + L.dv, nk, d2h, stream) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return FA_OK;
}
