// Interface between the C-ABI translation unit and the kernel translation
// units.  Not part of the public boundary (that is include/fa.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fa_sched.h"

namespace fa {

struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // 3-D maps over [B*H][N][d] bf16, box 64 x 128 x 1, 128-byte swizzle
  float* o;                      // [B*H][N][d] fp32
  float* lse;                    // [B*H][N] fp32
  int n;                         // sequence length
  int d;                         // head dimension (64 or 128)
  int causal;
  float scale_log2;              // softmax scale * log2(e)
  SchedParams sched;
  int* status;                   // device status word (4 ints)
  unsigned long long wait_limit_ns;
  int stall_unit;                // testing: CTA 0 skips one K tile of its n-th unit (-1: never)
};

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);

struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // bf16 maps as for the forward pass
  const float* o;                       // forward output, fp32
  const float* lse;                     // forward log-sum-exp, fp32
  const uint16_t* dout;                 // dO, bf16 bits
  float* dq;
  float* dk;
  float* dv;
  float* delta;                         // D_i = rowsum(dO * O), [B*H][N]
  int heads;
  int n;
  int d;
  int causal;
  float scale;
  float scale_log2;
  int grid_kv;                          // CTAs of the dK/dV kernel
  int grid_q;                           // CTAs of the dQ kernel
  int grid_pre;                         // CTAs of the preprocess kernel
  SchedParams sched_kv;
  SchedParams sched_q;
  int* status;
  unsigned long long wait_limit_ns;
};

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);

// The three stages of launch_bwd, for callers that time or order them
// separately: 0 = preprocess (D'), 1 = dQ (corrects D), 2 = dK/dV.
cudaError_t launch_bwd_stage(const BwdArgs& a, int stage, cudaStream_t stream);

}  // namespace fa
