/*
 * Measurement library libta11_probe.so: microbenchmark kernels used by the
 * benchmark's tables and the tests.  None of it is part of the attention library's
 * interface (include/fa.h); it exists to measure the roofs the attention kernels are
 * judged against.  Every call is asynchronous on `stream`; every pointer is a caller-owned
 * device pointer.  Return codes follow fa_status (0 = ok, 1 = invalid argument,
 * 3 = misaligned, 5 = no sm_103 device, 6 = launch failed).
 */
#ifndef TA11_PROBE_H
#define TA11_PROBE_H

#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * The special-function unit's exp2 rate.  n_blocks blocks of 512 threads; each thread
 * runs 8 independent chains x <- 2^(-x) of `iters` ex2.approx.ftz.f32 each, so one launch
 * performs n_blocks * 512 * 8 * iters of them.  `out` (n_blocks * 512 floats) receives
 * each thread's chain sum.  n_blocks in [1, 65535], iters in [1, 2^20].
 */
int ta11_probe_ex2(float* out, int n_blocks, int iters, cudaStream_t stream);

/*
 * The tensor core's rate for the attention kernels' score-GEMM UMMA shape (M = N = 128,
 * K = 16, bf16 operands from 128-byte swizzled K-major shared-memory tiles, fp32
 * accumulate in TMEM).  n_ctas CTAs (one per SM at most resident), each issuing `iters`
 * groups of 8 UMMAs back to back from one thread: n_ctas * iters * 8 * 2*128*128*16
 * FLOPs.  The completion wait is bounded by limit_ns; a timeout is recorded in the
 * library's status word (ta11_probe_status).  n_ctas in [1, 65535], iters in [1, 65536].
 */
int ta11_probe_umma(int n_ctas, int iters, unsigned long long limit_ns, cudaStream_t stream);

/* Status word of the probes' bounded waits: 0 or 7 (timeout); reset != 0 clears it. */
int ta11_probe_status(int reset);

#ifdef __cplusplus
}
#endif

#endif
