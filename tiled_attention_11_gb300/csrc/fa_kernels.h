// Parameters shared by the host launchers and the sm_103a attention kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ta11 {

struct FwdParams {
  void* o;              // bf16 [B,H,Nq,D]
  float* lse;           // fp32 [B,H,Nq], natural log
  int Nq, Nk;
  int n_q_tiles;        // ceil(Nq / 128)
  float scale_log2;     // scale * log2(e)
  unsigned long long wait_limit_ns;
  unsigned* status;     // device status word pair
};

struct BwdParams {
  void* dk;             // bf16 [B,H,Nk,D]
  void* dv;             // bf16 [B,H,Nk,D]
  float* dq_accum;      // fp32 [B*H, Nq_pad, D]
  const float* lse2;    // fp32 [B*H, Nq_pad]: lse * log2(e); +inf on padded rows
  const float* dlt;     // fp32 [B*H, Nq_pad]: rowsum(dO o O); 0 on padded rows
  int Nq, Nk, Nq_pad;
  int n_k_tiles;        // ceil(Nk / 128)
  float scale;          // softmax scale
  float scale_log2;     // scale * log2(e)
  unsigned long long wait_limit_ns;
  unsigned* status;
};

struct PrepParams {
  const void* o;        // bf16 [B,H,Nq,D]
  const void* dout;     // bf16 [B,H,Nq,D]
  const float* lse;     // fp32 [B,H,Nq]
  float* dq_accum;      // fp32 [B*H, Nq_pad, D] (zeroed here)
  float* lse2;          // fp32 [B*H, Nq_pad]
  float* dlt;           // fp32 [B*H, Nq_pad]
  int BH, Nq, Nq_pad;
};

struct ConvParams {
  const float* dq_accum;  // fp32 [B*H, Nq_pad, D]
  void* dq;               // bf16 [B,H,Nq,D]
  int BH, Nq, Nq_pad;
  float scale;
};

// Host launchers (return cudaError_t of the launch).
cudaError_t launch_fwd(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int BH, cudaStream_t st);
cudaError_t launch_bwd_prep(int D, const PrepParams& p, cudaStream_t st);
cudaError_t launch_bwd(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, int BH, cudaStream_t st);
cudaError_t launch_bwd_convert(int D, const ConvParams& p, cudaStream_t st);
cudaError_t launch_wait_probe(unsigned long long limit_ns, unsigned* status, cudaStream_t st);

}  // namespace ta11
