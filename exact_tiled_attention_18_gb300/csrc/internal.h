// Interface between the C-ABI translation unit and the kernel translation
// units.  Not part of the public boundary (that is include/fa.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "fa_sched.h"

namespace fa {

// One-time setup of a kernel on the current device, before its first launch
// there: checks the registers per thread it was compiled with (the kernels'
// warpgroup register splits assume that launch allocation; 0 skips the
// check) and raises its dynamic shared-memory limit.  `done` holds one bit
// per device already set up, so later launches skip both runtime calls.
template <typename Kernel>
cudaError_t setup_kernel_once(Kernel kern, int smem_bytes, int expect_regs, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ULL << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  if (expect_regs > 0) {
    cudaFuncAttributes fattr;
    e = cudaFuncGetAttributes(&fattr, kern);
    if (e != cudaSuccess) return e;
    if (fattr.numRegs != expect_regs) return cudaErrorInvalidConfiguration;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  done.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

// Sequence geometry: padded query/key lengths and optional per-sequence valid
// lengths (device arrays of B ints; null means all rows are valid).
struct SeqGeom {
  int nq, nk;
  const int* seqlens_q;
  const int* seqlens_k;
  int heads_per_batch;  // H: head index / H = sequence index
};

struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // 3-D maps over [B*H][Nq or Nk][d] bf16, box 64 x 128 x 1, 128-byte swizzle
  void* o;                       // [B*H][Nq][d] fp32, or bf16 when o_bf16
  float* lse;                    // [B*H][Nq] fp32
  int o_bf16;
  SeqGeom geom;
  int d;                         // head dimension (64 or 128)
  int causal;
  float scale_log2;              // softmax scale * log2(e)
  SchedParams sched;
  int* status;                   // device status word (4 ints)
  unsigned long long wait_limit_ns;
  int stall_unit;                // testing: CTA 0 skips one K tile of its n-th unit (-1: never)
  const uint16_t* bias;          // additive mask, bf16, or null; element (b, h, i, j) at
  long long bias_sb, bias_sh, bias_sq;  //   b * bias_sb + h * bias_sh + i * bias_sq + j
  // key splits (square fp32 forward only): splits > 1 divides every query
  // pair's key tiles into ranges of `chunk` tiles, one work unit each
  // (sched.units_per_head = pairs * splits); the partial results go to part,
  // [heads][splits][Nq][d] outputs then [heads][splits][Nq] log2-sum-exp,
  // and are merged into o and lse by launch_split_combine.
  int splits, chunk;
  float* part;
};

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);

// Additive mask on the scaled scores: bf16 element (b, h, i, j) at
// p + b*sb + h*sh + i*sq + j (strides in elements, 0 broadcasts).
struct BiasRef {
  const uint16_t* p;
  long long sb, sh, sq;
};

struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // bf16 maps as for the forward pass
  const void* o;                        // forward output, fp32 (or bf16 when o_bf16)
  int o_bf16;
  const float* lse;                     // forward log-sum-exp, fp32
  const uint16_t* dout;                 // dO, bf16 bits
  float* dq;
  float* dk;
  float* dv;
  float* delta;                         // D_i = rowsum(dO * O), [B*H][Nq]
  int heads;
  SeqGeom geom;
  int d;
  int causal;
  float scale;
  float scale_log2;
  int grid_kv;                          // CTAs of the dK/dV kernel
  int grid_q;                           // CTAs of the dQ kernel
  SchedParams sched_kv;
  SchedParams sched_q;
  int* status;
  unsigned long long wait_limit_ns;
  int stall_unit;                       // testing: CTA 0 skips one stage of its n-th unit (-1: never)
  BiasRef bias;                         // additive mask of the forward pass (p null: none)
};

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);

// FP8 forward (E4M3 q, k and v^T, d = 128, square): tm_q, tm_k over
// [B*H][N][128] bytes, tm_v over v^T [B*H][128][N] bytes; o fp32.
cudaError_t launch_fwd_fp8(const FwdArgs& a, cudaStream_t stream);

struct DecArgs {
  CUtensorMap tm_k, tm_v;  // 3-D maps over [B*H][Nk][d] bf16, box 64 x 64 x 1, 128-byte swizzle
  const uint16_t* q;       // [B*H][Nq][d] bf16
  float* o;                // [B*H][Nq][d] fp32
  float* lse;              // [B*H][Nq] fp32
  float* part;             // splits > 1: [B*H][splits][Nq][d] outputs, then [B*H][splits][Nq] log2-sum-exp
  SeqGeom geom;
  int heads;
  int d;
  int causal;
  float scale_log2;
  int splits;              // key splits per head (one CTA each)
  int chunk;               // keys per split, a multiple of 64
  int* status;
  unsigned long long wait_limit_ns;
  int stall_unit;          // testing: CTA n leaves its first stage unloaded (-1: never)
};

cudaError_t launch_decode(const DecArgs& a, cudaStream_t stream);

// Merges per-split normalised outputs and their log2-sum-exp (layout of
// DecArgs::part, `rows` = heads * nq rows) into o and lse (natural log).
cudaError_t launch_split_combine(const float* part, float* o, float* lse, int rows, int nq, int splits, int d,
                                 cudaStream_t stream);

// The stages of the two backward algorithms, for callers that time or order
// them separately.  Two-pass (launch_bwd): 0 = dQ (forms the row term D),
// 1 = dK/dV.  Single-pass (launch_bwd_single_pass): 2 = the row term D
// (and dQ set to zero), 3 = dK, dV and dQ accumulated into place.
cudaError_t launch_bwd_stage(const BwdArgs& a, int stage, cudaStream_t stream);
cudaError_t launch_bwd_single_pass(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_rowterm(const BwdArgs& a, cudaStream_t stream);

}  // namespace fa
