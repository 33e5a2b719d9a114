/*
 * C ABI of the GB300 (sm_103a) tiled-attention library (libta11_fa.so).
 *
 * The library computes exact scaled-dot-product attention tile by tile with an
 * online softmax, forward and backward, on one GPU.  The method and its notation
 * follow the pages this library restates:
 *   [FA2-impl]  "FlashAttention-2实现与优化：高效注意力机制详解"
 *   [FA-hist]   "FlashAttention技术演进全景图"
 *   [FA-mem]    "解释FlashAttention的显存优化原理"
 *
 * Conventions shared by every call
 *   - Tensors are dense, contiguous, row-major [B, H, N, D] (D innermost) in
 *     bf16 (__nv_bfloat16); "void*" arguments are such bf16 device pointers.
 *     With H = 1 this is the [B, N, D] layout of [FA2-impl] §3.1/§3.2.
 *   - lse is fp32 [B, H, Nq]: the natural-log row logsumexp of the scaled
 *     scores, L_i = m_i + log(sum_j exp(S_ij - m_i)) ([FA2-impl] §3.1, L = m + log l).
 *   - Supported head dims: D in {16, 32, 64, 128}.  B, H, Nq, Nk >= 1;
 *     B*H <= 65535; Nq, Nk (and the packed totals and maximum lengths of the
 *     variable-length calls) <= 2^29.  scale must be finite and > 0
 *     (the usual value is 1/sqrt(D), [FA2-impl] §3.1).
 *   - causal != 0 keeps key j for query i iff j <= i on absolute indices
 *     (top-left alignment, [FA2-impl] §4.3), for any Nq, Nk.  Masked keys get
 *     exactly zero weight (the pages fill with -1e6; this library uses -inf).
 *   - Every device pointer must be non-null and 16-byte aligned (TMA); lse must
 *     be 4-byte aligned; the bwd workspace 256-byte aligned.  Output buffers
 *     may not overlap inputs or each other.
 *   - Ownership: the caller allocates and frees every buffer.  The library never
 *     allocates device memory and keeps no state between calls except the
 *     device status word below and a per-process wait limit.
 *   - Asynchrony: calls enqueue work on `stream` and return without
 *     synchronising.  A failed check returns its code and launches nothing.
 *     Launch errors are reported as FA_ERR_LAUNCH.
 *   - Thread safety: re-entrant; work on different streams is independent.
 *   - Device: the current CUDA device must be sm_103 (GB300); otherwise
 *     FA_ERR_DEVICE.  There is no CPU fallback.
 */
#ifndef TA11_FA_H_
#define TA11_FA_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad scale, overlapping buffers */
  FA_ERR_UNSUPPORTED_D = 2, /* D not in {16, 32, 64, 128} */
  FA_ERR_MISALIGNED = 3,    /* pointer alignment below the stated minimum */
  FA_ERR_WORKSPACE = 4,     /* bwd workspace null, misaligned or too small */
  FA_ERR_DEVICE = 5,        /* no CUDA device, or the current device is not sm_103 */
  FA_ERR_LAUNCH = 6,        /* a kernel launch or tensor-map encode failed */
  FA_ERR_TIMEOUT = 7,       /* a kernel gave up a bounded wait (see fa_device_status) */
  FA_ERR_SCRATCH_LIMIT = 8  /* fa_bwd_noalloc: problem needs more than its fixed scratch */
} fa_status;

/*
 * Forward: O = softmax(scale * Q K^T [masked]) V and the row logsumexp L.
 * [FA2-impl] §3.1 (forward(q, k, v, is_causal) returns o and saves (L, q, k, v, o))
 * and §3.2 (kernel arguments Q, K, V, O, L, N_QUERIES, N_KEYS, scale, D, IS_CAUSAL).
 *   q   [B,H,Nq,D] bf16 in      k, v [B,H,Nk,D] bf16 in
 *   o   [B,H,Nq,D] bf16 out     lse  [B,H,Nq]   fp32 out (natural log)
 * The N x N score matrix is never written to memory.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk, int D,
           float scale, int causal, cudaStream_t stream);

/*
 * Bytes of device workspace fa_bwd needs for these sizes (0 if they are invalid):
 * dq_accum fp32 [B*H, Nq_pad, D], Dlt fp32 [B*H, Nq_pad] and L*log2(e) fp32
 * [B*H, Nq_pad], with Nq_pad = 64*ceil(Nq/64), each segment 256-byte aligned.
 */
size_t fa_bwd_workspace_size(int B, int H, int Nq, int Nk, int D);

/*
 * Backward: given dO, computes dQ, dK, dV by recomputing P from lse instead of
 * storing it ([FA-mem] §2(2) recomputation; [FA-hist] §2.2; [FA2-impl] §7 lists the
 * backward as the next step).  Formulas: dV = P^T dO, dP = dO V^T,
 * Dlt_i = sum_d dO_id O_id, dS = P o (dP - Dlt), dQ = scale dS K, dK = scale dS^T Q.
 *   q, o, dO [B,H,Nq,D] bf16 in   k, v [B,H,Nk,D] bf16 in   lse [B,H,Nq] fp32 in
 *   dq [B,H,Nq,D], dk, dv [B,H,Nk,D] bf16 out
 *   workspace: >= fa_bwd_workspace_size(...) bytes of device memory, 256-byte
 *   aligned, owned by the caller, contents on entry ignored (overwritten).
 * o and lse must be the forward's outputs for the same q, k, v, scale, causal.
 * dQ adds every key tile's fp32 contribution in L2 (bulk reduce-adds) in no fixed order,
 * so it is not bitwise deterministic run to run; dK and dV (and fa_fwd's O, L) are.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
           void* dk, void* dv, int B, int H, int Nq, int Nk, int D, float scale, int causal, void* workspace,
           size_t workspace_bytes, cudaStream_t stream);

/* Static English description of a status code (never NULL). */
const char* fa_strerror(int status);

/*
 * Device status word: FA_OK, or FA_ERR_TIMEOUT once any kernel of this library
 * gave up a bounded wait on the current device.  Synchronises the device first.
 * *site (if non-null) receives the internal wait site of the first timeout.
 * reset != 0 clears the word afterwards.
 */
int fa_device_status(unsigned* site, int reset);

/* Per-process limit on every in-kernel wait, in nanoseconds (default 2e9). */
void fa_set_wait_limit_ns(unsigned long long ns);

/*
 * Schedule of the forward kernels (fa_fwd, fa_fwd_varlen, fa_fwd_fp8, fa_fwd_window, the
 * key chunks of its split global query rows included) when their (query-tile pair, head)
 * units are more than the SMs can hold at once (no counterpart on the pages; a scheduling
 * choice, not a change of the result):
 *   1 (default)  persistent CTAs: a CTA that finishes a unit takes over the next CTA of
 *                its grid that has not started, so one CTA's pipelines run on across
 *                units (the next unit's loads and first score GEMMs overlap the current
 *                unit's end);
 *   0            one CTA per unit.
 * Both compute every output bitwise the same.  Process-wide; returns the previous value.
 */
int fa_set_fwd_persistent(int on);

/*
 * The same choice for the backward's main kernel when its (key tile, head) units are more
 * than the SMs hold at once: fa_bwd and fa_bwd_varlen with D < 128 or at most 8192 queries
 * per head (where it measured faster), and fa_bwd_window (its split global key tiles'
 * chunks included, see fa_bwd_window_workspace_size).  1 (default) persistent CTAs whose
 * pipelines run on across units (the next unit's K / V loads and first score GEMMs overlap
 * the current unit's dK / dV epilogue), 0 one CTA per unit.  dK and dV are bitwise the same
 * either way, except the rows of split global key tiles (their chunks' fp32 partial sums
 * are added in no fixed order); dQ adds fp32 contributions in no fixed order, as fa_bwd
 * documents.
 * Process-wide; returns the previous value.
 */
int fa_set_bwd_persistent(int on);

/*
 * Self-test hook for the timeout path: launches a one-warp kernel that waits,
 * with the given limit, on a barrier nothing ever arrives on; it then records
 * FA_ERR_TIMEOUT in the status word and exits normally (no trap, no hang).
 */
int fa_wait_probe(unsigned long long limit_ns, cudaStream_t stream);

/*
 * Timing hook for measurement tools (no counterpart on the pages): while both
 * events are non-null, every fa_bwd records `begin` on its stream immediately
 * before launching its main tensor-core kernel and `end` immediately after it,
 * so cudaEventElapsedTime(begin, end) is that one kernel's duration.  The events
 * belong to the caller; pass NULL, NULL to stop recording.  Process-wide setting.
 */
void fa_set_bwd_main_events(cudaEvent_t begin, cudaEvent_t end);

/*
 * Local-window + global-token attention ([FA2-impl] §7: sparse attention combining local
 * windows and global tokens; [FA-mem] case 2: local blocks plus global key points for
 * 100K-token sequences), as an exact mask on absolute (top-left) indices: key j is visible
 * to query i iff
 *     j < Nk  and  (causal == 0 or j <= i)  and
 *     ( (window_left < 0 or j >= i - window_left) and (window_right < 0 or j <= i + window_right)
 *       or j < n_global or i < n_global )
 * A negative window bound is unbounded; n_global tokens (the first queries and keys) see
 * and are seen by every token (subject to the causal condition).  A query row with no
 * visible key gets O = 0 and L = -inf, and zero gradients.  Key tiles that no row of a
 * query tile can see are skipped, so the work grows with the window, not with Nk.
 * Layout, workspace (fa_bwd_workspace_size), ownership, asynchrony and errors as for
 * fa_fwd / fa_bwd.
 */
/* Without the causal condition the global query rows see every key; when the key range is
 * long (> 32 key tiles) their query tiles are split over chunks of 16 key tiles whose partial
 * results (unnormalised O, running maximum and sums) go to `workspace` and are merged by a
 * second kernel.  fa_fwd_window_workspace_size gives the bytes (0 when no split is needed;
 * workspace may then be null); workspace 256-byte aligned, caller-owned, FA_ERR_WORKSPACE
 * when missing or short. */
size_t fa_fwd_window_workspace_size(int B, int H, int Nq, int Nk, int D, int causal, int window_left,
                                    int window_right, int n_global);
int fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                  int D, float scale, int causal, int window_left, int window_right, int n_global, void* workspace,
                  size_t workspace_bytes, cudaStream_t stream);
/* Key tiles that hold global keys are seen by every (later) query; when the query range is
 * long (> 64 steps of 64 queries) they are split over chunks of 32 steps whose partial dK, dV
 * go to an fp32 area after the usual workspace and are written out by a final kernel.
 * fa_bwd_window_workspace_size gives the bytes (>= fa_bwd_workspace_size). */
size_t fa_bwd_window_workspace_size(int B, int H, int Nq, int Nk, int D, int window_left, int window_right,
                                    int n_global);
int fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int D, float scale, int causal,
                  int window_left, int window_right, int n_global, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream);

/*
 * One forward + backward step from host buffers: copies q, k, v, dO (host, bf16 [B,H,N,D];
 * pinned memory for asynchronous copies) into `dev`, runs fa_fwd and fa_bwd there and
 * copies o, lse, dq, dk, dv back to the host buffers, all asynchronously on `stream` (one
 * cudaMemcpyAsync per tensor).  `dev` (256-byte aligned, dev_bytes >=
 * fa_step_host_device_bytes(...)) holds the device copies and the backward workspace.
 * Host buffers must stay valid and untouched until the stream reaches the end of the
 * step.  Steps on different streams with separate `dev` buffers run concurrently, which
 * lets one step's copies overlap another's kernels.  Errors as for fa_fwd / fa_bwd;
 * FA_ERR_WORKSPACE for a missing, misaligned or short `dev`.
 */
size_t fa_step_host_device_bytes(int B, int H, int Nq, int Nk, int D);
int fa_step_host(const void* q_h, const void* k_h, const void* v_h, const void* do_h, void* o_h, float* lse_h,
                 void* dq_h, void* dk_h, void* dv_h, void* dev, size_t dev_bytes, int B, int H, int Nq, int Nk,
                 int D, float scale, int causal, cudaStream_t stream);

/*
 * FP8 (e4m3) forward with per-tensor scales ([FA-hist] §5.3 names FP8 quantisation as the
 * method's next direction).  e4m3 = 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
 * infinity, largest finite 448.  A tensor x is held as codes with one fp32 descale:
 * x ~= descale * e4m3(code).
 *
 * fa_quantize_e4m3: bf16 x[n] -> codes[n] (same element order), with
 *   amax = max|x|, codes = e4m3_rn_satfinite(x * (448 / amax)), descale = amax / 448
 *   (fp32 IEEE division and product: the codes are fixed bit for bit); an all-zero x uses
 *   multiplier and descale 1.  `amax` and `descale` are device floats written by the call
 *   (amax is zeroed first on `stream`).  x and codes 16-byte aligned.
 * fa_quantize_e4m3_transposed: bf16 [B,H,N,D] -> codes_t [B,H,D,ldt] (keys innermost, the
 *   layout fa_fwd_fp8 takes for V), same rule with one scale for the whole tensor;
 *   ldt >= N and a multiple of 16; bytes of a row past N may be left unwritten; D in {64, 128}.
 * fa_quantize_qkv_e4m3: the three quantisations fa_fwd_fp8 takes, in one call: q bf16
 *   [B,H,Nq,D] -> q8 and k bf16 [B,H,Nk,D] -> k8 as fa_quantize_e4m3, v bf16 [B,H,Nk,D] ->
 *   vt8 [B,H,D,ldv] as fa_quantize_e4m3_transposed (ldv >= Nk, a multiple of 16), with
 *   amax[3] and descale[3] (device floats, in the order q, k, v; amax zeroed first on
 *   `stream`).  Codes and descales are those of the three separate calls bit for bit; one
 *   amax pass reads the three tensors and one pass writes the three code tensors, so the
 *   call makes one memset and two kernel launches instead of three and six.  D in {64, 128};
 *   all tensors 16-byte aligned; no output may overlap an input or another output.
 * fa_fwd_fp8: O = softmax(scale * (qd*Q8)(kd*K8)^T) (vd*V8) and L as for fa_fwd, with
 *   q8, k8 e4m3 [B,H,N,D], vt8 e4m3 [B,H,D,ldv] (ldv >= Nk, multiple of 16), descales as
 *   device floats; O bf16 [B,H,Nq,D], L fp32 [B,H,Nq].  Both GEMMs run on e4m3 operands
 *   with fp32 accumulation; P is rounded to e4m3, so O carries ~2-3% relative error on
 *   diffuse rows (the e4m3 step is 2^-3 of a binade) and is exact up to bf16 rounding on a
 *   row dominated by one key.  D in {64, 128}; causal as for fa_fwd.
 * Ownership, asynchrony and error codes as for fa_fwd.
 */
int fa_quantize_e4m3(const void* x, long long n, void* codes, float* amax, float* descale, cudaStream_t stream);
int fa_quantize_e4m3_transposed(const void* x, int B, int H, int N, int D, int ldt, void* codes_t, float* amax,
                                float* descale, cudaStream_t stream);
int fa_quantize_qkv_e4m3(const void* q, const void* k, const void* v, int B, int H, int Nq, int Nk, int D, void* q8,
                         void* k8, void* vt8, int ldv, float* amax, float* descale, cudaStream_t stream);
int fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, int ldv, const float* q_descale,
               const float* k_descale, const float* v_descale, void* o, float* lse, int B, int H, int Nq, int Nk,
               int D, float scale, int causal, cudaStream_t stream);

/*
 * Variable-length ("ragged") batches ([FA2-impl] §7 names ragged inputs as the next step;
 * [FA-hist] §2.3 dynamic sequence lengths): B independent sequences packed back to back.
 *   q, o, dO, dq: [total_q, H, D] bf16;  k, v, dk, dv: [total_k, H, D] bf16 (D innermost)
 *   lse: [H, total_q] fp32 (natural log)
 *   cu_seqlens_q / cu_seqlens_k: device int32 [B + 1], non-decreasing, cu[0] = 0,
 *   cu[B] = total; sequence b owns tokens cu[b] .. cu[b+1]-1 of every head.
 *   max_seqlen_q / max_seqlen_k: upper bounds of the per-sequence lengths (grid size).
 * Each sequence is attended on its own (causal: top-left within the sequence). A
 * sequence with queries but no keys gets O = 0 and L = -inf (and zero gradients).
 * Offsets are read on the device and clamped to [0, total] and to the maximum lengths,
 * so inconsistent offsets cannot make a kernel touch memory outside the buffers.
 * Other conventions (alignment, ownership, asynchrony, errors) as for fa_fwd / fa_bwd.
 */
int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int B, int H, int total_q, int total_k, int max_seqlen_q,
                  int max_seqlen_k, int D, float scale, int causal, cudaStream_t stream);
/* Workspace bytes for fa_bwd_varlen: H * 64*(ceil(total_q/64) + B) rows of dq_accum (D fp32),
 * Dlt and L*log2(e), each segment 256-byte aligned (0 if the sizes are invalid). */
size_t fa_bwd_varlen_workspace_size(int B, int H, int total_q, int max_seqlen_q, int D);
int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                  int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int D, float scale, int causal,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * CUDA Graph of one forward + backward step ([FA-hist] §3.2 and §5.2: launch overhead
 * dominates short sequences, and a CUDA Graph removes it).  Captures fa_fwd followed by
 * fa_bwd for these exact buffers, sizes and flags into an instantiated graph; every
 * fa_graph_launch replays the four kernels on `stream` reading the buffers' current
 * contents.  The buffers must stay allocated (and unmoved) for the graph's lifetime.
 * Arguments are validated exactly as by fa_fwd / fa_bwd; on failure *out is NULL and
 * nothing is captured.  Capture uses a private stream; the caller's streams are not
 * touched.  Not thread-safe per handle.
 */
typedef struct fa_graph_st* fa_graph;
int fa_graph_create(const void* q, const void* k, const void* v, void* o, float* lse, const void* dO, void* dq,
                    void* dk, void* dv, int B, int H, int Nq, int Nk, int D, float scale, int causal,
                    void* workspace, size_t workspace_bytes, fa_graph* out);
int fa_graph_launch(fa_graph g, cudaStream_t stream);
void fa_graph_destroy(fa_graph g);

/*
 * Backward without any device allocation, for callers that cannot call
 * cudaMalloc or hand over a workspace: for example a process that must not
 * allocate device memory after start-up (its memory budget is fixed), or a
 * plug-in whose host framework owns the allocator and passes only input and
 * output buffers.  The pages have no counterpart of this call; it computes
 * exactly what fa_bwd computes, with the same arguments minus the workspace.
 *
 * Its scratch (dq_accum, Dlt, L*log2(e), laid out as fa_bwd's workspace) is a
 * fixed 32 MiB array in the library's device memory, which every GPU that
 * loads the library holds until the process exits.  Problems whose
 * fa_bwd_workspace_size(B, H, Nq, Nk, D) exceeds 32 MiB (33554432 bytes) are
 * rejected with FA_ERR_SCRATCH_LIMIT before anything is launched; that call is
 * the exact test.  The scratch holds (4*D + 8) bytes per query row with each
 * head's rows padded to a multiple of 64, so for D = 128 the limit is
 * B*H*64*ceil(Nq/64) <= 64512 padded rows (e.g. 1008 heads of up to 64 queries):
 * many short heads count as 64 rows each.
 *
 * The first call on a device looks up the array's device address (a set-up per
 * device, done with that device current); make that first call before any
 * stream capture.  A lookup that fails (FA_ERR_DEVICE) is not remembered: the
 * next call tries again.  All calls share the one array and the kernels
 * re-initialise what must start at zero, so calls that overlap on the GPU
 * (different streams, or different threads without ordering) race on it and
 * must be serialised by the caller.  Allocates nothing: no cudaMalloc,
 * cudaFree or allocating library routine.
 */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                   void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int D, float scale, int causal,
                   cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TA11_FA_H_ */
