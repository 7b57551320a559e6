// Backward pass by recomputation.
//
// The forward pass keeps only O and the per-row log-sum-exp; the backward
// pass rebuilds the attention probabilities from Q, K and that LSE instead
// of storing the N x N matrices ("FlashAttention Interview Questions: IO
// Complexity, Tiling, and Numerical Stability", section "Why can
// recomputation help training?").  With P_ij = exp(s_ij - LSE_i):
//   dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,
//   dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
// (D_i = sum_j P_ij dP_ij equals rowsum(dO o O) because O = P V.)
//
// Two kernels, in stream order:
//   dq          one CTA per 128-query tile, sweeping its key tiles:
//               S = Q K^T, dP = dO V^T, dS (bf16) in TMEM, dQ += dS K;
//               a loader warp forms D' = rowsum(dO o O) one unit ahead, and
//               the kernel corrects D' to the exact row term (see the
//               kernel), so it runs before dkdv.
//   dkdv        one CTA per 128-key tile, sweeping the query tiles that
//               see it: S^T = K Q^T and dP^T = V dO^T on tcgen05 into TMEM,
//               P^T and dS^T computed by two warpgroups (thread = key row)
//               and written back to TMEM as bf16 (dS^T as a hi + lo pair),
//               then dV += P^T dO and dK += (dS^T hi + dS^T lo) Q with the A
//               operand read from TMEM.
// Every pipeline wait is bounded, as in the forward kernel.
#include <cuda_runtime.h>
#include <math_constants.h>

#include <type_traits>

#include "geom.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

enum BwdSite : int {
  SITE_KV_LOAD_KV = 11,
  SITE_KV_LOAD_QD = 12,
  SITE_KV_LD_EMPTY = 13,
  SITE_KV_MMA_KV = 14,
  SITE_KV_MMA_QD = 15,
  SITE_KV_MMA_PDS = 16,
  SITE_KV_EW_LD = 17,
  SITE_KV_EW_S = 18,
  SITE_KV_EW_ACC = 19,
  SITE_KV_EW_DP = 20,
  SITE_Q_LOAD_Q = 21,
  SITE_Q_LOAD_KV = 22,
  SITE_Q_MMA_Q = 23,
  SITE_Q_MMA_KV = 24,
  SITE_Q_MMA_DS = 25,
  SITE_Q_EW_S = 26,
  SITE_Q_EW_ACC = 27,
  SITE_Q_EW_XCH = 28,
  SITE_Q_EW_DP = 29,
  SITE_Q_MMA_P = 30,
  SITE_Q_EW_DD = 31,
  SITE_Q_DD_EMPTY = 32,
  SITE_KV_EW_DQ = 61,     // single pass: dQ share of the previous tile computed
  SITE_KV_EW_DSW = 62,    // single pass: the dS tile's buffer free to write
  SITE_KV_MMA_DQE = 63,   // single pass: dQ share read out (its columns free)
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& w, int site, int unit) {
  const bool ok = wait_bounded(bar, parity, w, site, unit);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

// Two-term bf16 split of a pair of fp32 values: hi keeps the top 16 bits of
// each value (truncation), lo is the exact remainder rounded to bf16, so
// hi + lo carries about 16 significant bits.  dS^T feeds the dK product
// this way: dK_j sums dS_ij q_i, and rows with large |q| (the long-context
// workload scales every 64th query by 10) amplify a plain bf16 rounding of
// dS past the gradient tolerance (dK error 0.155).  The dQ product sums
// dS_ij k_j over keys of ordinary size and takes dS rounded to bf16 (dQ
// error 8e-3 on that workload, against 2e-5 with the split, for one GEMM
// fewer per tile).
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const uint32_t u0 = __float_as_uint(x0), u1 = __float_as_uint(x1);
  hi = __byte_perm(u0, u1, 0x7632);  // top halves of both: truncation to bf16
  float r0, r1;
  f2_unpack(fsub2(f2_pack(x0, x1), f2_pack(__uint_as_float(u0 & 0xFFFF0000u), __uint_as_float(u1 & 0xFFFF0000u))),
            r0, r1);
  lo = pack_bf16x2(r0, r1);
}

__device__ __forceinline__ uint64_t f2_from(uint32_t a, uint32_t b) {
  return f2_pack(__uint_as_float(a), __uint_as_float(b));
}

// a pair of bf16 values (low half first) widened to an fp32 pair
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t u) {
  return f2_pack(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// Additive mask of one key for 64 consecutive queries q0.. (a column of the
// mask, stride sq elements), as bf16 pairs: queries q0..q0+31 in b0,
// q0+32..q0+63 in b1; 0 past query nq or without a column.  Across a warp
// (32 consecutive keys) each load is one contiguous 64-byte segment.
__device__ __forceinline__ void load_bias_column(const uint16_t* bcol, long long sq, int q0, int nq,
                                                 uint32_t (&b0)[16], uint32_t (&b1)[16]) {
  uint32_t h[64];
  if (bcol && q0 + 64 <= nq) {
    const uint16_t* p = bcol + q0 * sq;
#pragma unroll
    for (int c = 0; c < 64; ++c) h[c] = __ldg(p + c * sq);
  } else {
#pragma unroll
    for (int c = 0; c < 64; ++c) h[c] = (bcol && q0 + c < nq) ? __ldg(bcol + (q0 + c) * sq) : 0u;
  }
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    b0[e] = h[2 * e] | (h[2 * e + 1] << 16);
    b1[e] = h[32 + 2 * e] | (h[33 + 2 * e] << 16);
  }
}

// Additive mask of one query for 64 consecutive keys k0.. (part of a row),
// as bf16 pairs: keys k0..k0+31 in b0, k0+32..k0+63 in b1; 0 past key nk or
// without a row.  vec: the row starts on a 16-byte boundary (k0 is a
// multiple of 64, so then every load below is aligned).
__device__ __forceinline__ void load_bias_row(const uint16_t* brow, bool vec, int k0, int nk, uint32_t (&b0)[16],
                                              uint32_t (&b1)[16]) {
  if (vec && k0 + 64 <= nk) {
    const uint4* p = reinterpret_cast<const uint4*>(brow + k0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 x = __ldg(p + i), y = __ldg(p + 4 + i);
      b0[4 * i] = x.x, b0[4 * i + 1] = x.y, b0[4 * i + 2] = x.z, b0[4 * i + 3] = x.w;
      b1[4 * i] = y.x, b1[4 * i + 1] = y.y, b1[4 * i + 2] = y.z, b1[4 * i + 3] = y.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int c = k0 + 2 * e;
      const uint32_t lo = (brow && c < nk) ? __ldg(brow + c) : 0u;
      const uint32_t hi = (brow && c + 1 < nk) ? __ldg(brow + c + 1) : 0u;
      (e < 16 ? b0[e] : b1[e - 16]) = lo | (hi << 16);
    }
  }
}

// ------------------------------------------------------------------ dK / dV

// DQ: the single-pass variant, which also forms dQ_i += scale dS_ij k_j for
// every tile it visits and adds it into the fp32 dQ in global memory.  Its
// dS (bf16, [128 keys][128 queries], the 128-byte swizzled layout a TMA load
// of such a tile would give) is written to shared memory for that product:
// at d = 64 into a buffer of its own; at d = 128, where no 32 KB are left,
// over the dO tile of the current (Q, dO) stage once dV has read it (the
// stage is then released after the dQ product instead of after dK).
template <int D, bool DQ = false>
struct KvLayout {
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kStages = (D == 128) ? 2 : 4;  // (Q, dO) ring
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQdOff = 2 * kTileBytes;             // stage s: Q at +0, dO at +kTileBytes
  static constexpr bool kDsOwn = DQ && D == 64;             // dS tile in a buffer of its own
  static constexpr int kDsOff = kQdOff + kStages * 2 * kTileBytes;
  static constexpr int kLdOff = kDsOff + (kDsOwn ? kTileRows * kTileRows * 2 : 0);  // stage s: lse2[128], d[128]
  static constexpr int kBarOff = kLdOff + kStages * 1024;
  static constexpr int KV_FULL = 0;
  static constexpr int KV_EMPTY = 1;
  static constexpr int QD_FULL = 2;
  static constexpr int QD_EMPTY = QD_FULL + kStages;
  static constexpr int LD_FULL = QD_EMPTY + kStages;
  static constexpr int LD_EMPTY = LD_FULL + kStages;
  static constexpr int S_FULL = LD_EMPTY + kStages;  // S^T computed
  static constexpr int DP_FULL = S_FULL + 1;          // dP^T computed
  static constexpr int P_READY = DP_FULL + 1;    // P^T stored (one arrive per elementwise warp)
  static constexpr int DS_READY = P_READY + 1;   // dS^T hi/lo stored (and, DQ, the bf16 dS tile)
  static constexpr int ACC_FULL = DS_READY + 1;
  static constexpr int DV_DONE = ACC_FULL + 1;   // DQ: dV of the tile done (its dO tile may be overwritten)
  static constexpr int DQ_FULL = DV_DONE + 1;    // DQ: dQ share of the tile computed
  static constexpr int DQ_EMPTY = DQ_FULL + 1;   // DQ: dQ share read out (one arrive per elementwise warp)
  static constexpr int DS_FREE = DQ_EMPTY + 1;   // DQ, own buffer: the dQ product has read the dS tile
  static constexpr int DRAIN = DS_FREE + 1;
  static constexpr int kNumBars = DRAIN + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  // tensor memory columns; the dQ share has columns of its own at d = 64 and
  // reuses the dP^T columns at d = 128 (after dK has read dS^T from them)
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr uint32_t kColDQ = (D == 64) ? 256 + 2 * D : kColDP;
  static_assert(kSmemBytes <= 232448, "shared memory over the per-CTA limit");
};

// 12 warps: two elementwise warpgroups, then TMA (warp 8), MMA (warp 9), the
// LSE/D loader (warp 10) and an idle warp completing the third warpgroup.
// Launched at 168 registers a thread; the elementwise warpgroups take 184 and
// the third keeps 136 (2*128*184 + 128*136 = 384*168), enough for the MMA
// thread to hold its descriptors without spilling.
constexpr int kKvThreads = 384;
constexpr int kKvLaunchRegs = 168;
constexpr int kKvEwRegs = 184;
constexpr int kKvOtherRegs = 136;
static_assert(2 * 128 * kKvEwRegs + 128 * kKvOtherRegs <= kKvThreads * kKvLaunchRegs,
              "register split exceeds the launch allocation");

// The single-pass variant's dQ share of one key tile: each elementwise
// thread reads its query row's NC columns (lane = query row) out of tensor
// memory, the warp releases the columns, and the thread adds the values into
// the fp32 dQ row in global memory.  Every key tile adds its share, so the
// order of the sum (and its last bits) varies from run to run.
template <int NC>
__device__ __forceinline__ void dq_share_load(uint32_t taddr, uint32_t (&v)[NC / 32][32]) {
#pragma unroll
  for (int c = 0; c < NC / 32; ++c) tmem_ld32(taddr + 32 * c, v[c]);
  tmem_ld_wait();
}

template <int NC>
__device__ __forceinline__ void dq_share_add(float* dst, const uint32_t (&v)[NC / 32][32]) {
#pragma unroll
  for (int c = 0; c < NC / 32; ++c) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 32 * c + 4 * e),
                   "f"(__uint_as_float(v[c][4 * e])), "f"(__uint_as_float(v[c][4 * e + 1])),
                   "f"(__uint_as_float(v[c][4 * e + 2])), "f"(__uint_as_float(v[c][4 * e + 3]))
                   : "memory");
    }
  }
}

// Reads the pending dQ share (query tile pend_i of head pend_head) out of
// tensor memory, releases its columns to the MMA thread and adds it into dQ:
// warpgroup w takes columns [w d/2, (w+1) d/2) of its query rows.  No-op
// without a pending share.  Returns false if a wait gave up.
template <int D>
__device__ __forceinline__ bool dq_share_flush(uint32_t full_bar, uint32_t empty_bar, uint32_t& dqn,
                                               int& pend_head, int pend_i, int pend_lq, uint32_t taddr, float* dq,
                                               int nq, int r, int w, const WaitCtl& wc, int unit) {
  if (pend_head < 0) return true;
  const bool ok = wait_bounded(full_bar, dqn & 1, wc, SITE_KV_EW_DQ, unit);
  if (!__all_sync(0xffffffffu, ok)) return false;
  ++dqn;
  tc_fence_after();
  uint32_t v[D / 64][32];
  dq_share_load<D / 2>(taddr, v);
  tc_fence_before();
  mbar_arrive_warp(empty_bar);
  const int qrow = pend_i * kTileRows + r;
  if (qrow < pend_lq) dq_share_add<D / 2>(dq + (static_cast<size_t>(pend_head) * nq + qrow) * D + w * (D / 2), v);
  pend_head = -1;
  return true;
}

template <int D, bool CAUSAL, bool BIAS, bool DQ>
__global__ void __launch_bounds__(kKvThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const float* __restrict__ lse, const float* __restrict__ delta, float* __restrict__ dk,
                float* __restrict__ dv, float* __restrict__ dq, const SeqGeom geom, const float scale,
                const float scale_log2, const SchedParams sp, int* status, const unsigned long long limit_ns,
                const int stall_unit, const BiasRef bias) {
  using L = KvLayout<D, DQ>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kBarOff;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bars + 8 * L::KV_FULL, 1);
    mbar_init(bars + 8 * L::KV_EMPTY, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bars + 8 * (L::QD_FULL + s), 1);
      mbar_init(bars + 8 * (L::QD_EMPTY + s), 1);
      mbar_init(bars + 8 * (L::LD_FULL + s), 1);    // the loader warp
      mbar_init(bars + 8 * (L::LD_EMPTY + s), 8);   // one per elementwise warp
    }
    mbar_init(bars + 8 * L::S_FULL, 1);
    mbar_init(bars + 8 * L::DP_FULL, 1);
    mbar_init(bars + 8 * L::P_READY, 8);
    mbar_init(bars + 8 * L::DS_READY, 8);
    mbar_init(bars + 8 * L::ACC_FULL, 1);
    mbar_init(bars + 8 * L::DV_DONE, 1);
    mbar_init(bars + 8 * L::DQ_FULL, 1);
    mbar_init(bars + 8 * L::DQ_EMPTY, 8);
    mbar_init(bars + 8 * L::DS_FREE, 1);
    mbar_init(bars + 8 * L::DRAIN, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, status, limit_ns};
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  // shared-memory address of the bf16 dS tile of ring position qdpos (DQ)
  auto ds_tile = [&](uint32_t qdpos) -> uint32_t {
    return L::kDsOwn ? sbase + L::kDsOff : sbase + L::kQdOff + (qdpos % L::kStages) * 2 * L::kTileBytes + L::kTileBytes;
  };

  if (warp < 8) {
    // ------------------------------------------------ P^T and dS^T (thread = key row)
    regs_increase<kKvEwRegs>();
    const int w = warp >> 2;  // warpgroup: query columns [64 w, 64 w + 64)
    const int r = ((warp & 3) << 5) + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const float* ld_base = reinterpret_cast<const float*>(smem + L::kLdOff);
    uint32_t ldn = 0, sn = 0, an = 0;
    // DQ: dQ shares read out, dS tiles written; the tile whose dQ share is
    // still to be read (head, query tile; -1: none)
    uint32_t dqn = 0, dsn = 0;
    int pend_head = -1, pend_i = 0, pend_lq = 0;
    const uint32_t dq_cols = tmem + lane_off + L::kColDQ + w * (D / 2);
    SchedIter it = sched_begin(sp);
    int head, j;
    bool ok = true;
    while (ok && sched_next(it, sp, blockIdx.x, head, j)) {
      const HeadLen hl = head_len(geom, head);
      int i0, i1;
      key_tile_queries(hl, j, CAUSAL, i0, i1);
      const int unit = head * sp.units_per_head + j;
      // additive mask: this key's column, one element per query at stride sq
      const uint16_t* bcol = nullptr;
      if constexpr (BIAS) {
        const int bidx = head / geom.heads_per_batch;
        const int key = j * kTileRows + r;
        if (key < geom.nk)
          bcol = bias.p + bidx * bias.sb + (head - bidx * geom.heads_per_batch) * bias.sh + key;
      }
      for (int i = i0; i < i1; ++i) {
        // the mask of this key for the warpgroup's 64 queries, bf16 pairs
        // (fetched before the waits; 0 past the last query row)
        uint32_t bb0[BIAS ? 16 : 1], bb1[BIAS ? 16 : 1];
        if constexpr (BIAS) load_bias_column(bcol, bias.sq, i * kTileRows + 64 * w, geom.nq, bb0, bb1);
        const uint32_t ls = ldn % S;
        ok = warp_wait(BAR(L::LD_FULL + ls), (ldn / S) & 1, wc, SITE_KV_EW_LD, unit);
        if (!ok) break;
        // P^T needs only S^T: dP^T may still be in the tensor pipe
        const uint32_t sdp_parity = sn & 1;
        ok = warp_wait(BAR(L::S_FULL), sdp_parity, wc, SITE_KV_EW_S, unit);
        if (!ok) break;
        ++sn;
        tc_fence_after();
        const float* l2s = ld_base + ls * 256;
        const float* dds = l2s + 128;
        // key j*128 + r is hidden from query column c iff c < mlim
        const bool need_mask = CAUSAL && tile_crosses_diagonal(hl, i, j);
        const int mlim = r + (j - i) * kTileRows - hl.off;
        const uint64_t c2 = f2_pack(scale_log2, scale_log2);
        // Phase 1: P^T for 32 query columns starting at col0, kept in sr as fp32
        // bits and packed to bf16 in pk.  MASKED: a tile crossing the causal
        // boundary, where a key may come after the query.
        auto pchunk = [&](auto masked, uint32_t (&sr)[32], int col0, uint32_t (&pk)[16],
                          const uint32_t (&bh)[BIAS ? 16 : 1]) {
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            // l2s holds -LSE*log2(e) (-inf for padding and key-less queries)
            const float4 l4 = *reinterpret_cast<const float4*>(l2s + col0 + c);
            uint64_t t01 = f2_pack(l4.x, l4.y), t23 = f2_pack(l4.z, l4.w);
            if constexpr (BIAS) {
              // + bias * log2(e); a hidden key (-inf) gives p = 0
              t01 = ffma2(bf16x2_to_f2(bh[c / 2]), f2_pack(kLog2e, kLog2e), t01);
              t23 = ffma2(bf16x2_to_f2(bh[c / 2 + 1]), f2_pack(kLog2e, kLog2e), t23);
            }
            float p[4];
            f2_unpack(ffma2(f2_from(sr[c], sr[c + 1]), c2, t01), p[0], p[1]);
            f2_unpack(ffma2(f2_from(sr[c + 2], sr[c + 3]), c2, t23), p[2], p[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              p[e] = ex2_approx(p[e]);
              if (decltype(masked)::value && (col0 + c + e) < mlim) p[e] = 0.f;  // key after the query
              sr[c + e] = __float_as_uint(p[e]);
            }
            pk[c / 2] = pack_bf16x2(p[0], p[1]);
            pk[c / 2 + 1] = pack_bf16x2(p[2], p[3]);
          }
        };
        // Phase 2: dS^T = P^T o (dP^T - D), split into hk (hi) and lk (lo);
        // DQ: also scale * dS^T rounded to bf16 into the shared dS tile, this
        // thread's key row, queries [col0, col0 + 32) (four 16-byte chunks of
        // the 128-byte row of block w, swizzled by the row)
        const uint64_t sc2 = f2_pack(scale, scale);
        const bool key_live = j * kTileRows + r < hl.lk;
        auto dchunk = [&](const uint32_t (&pr)[32], uint32_t (&dr)[32], int col0, uint32_t (&hk)[16],
                          uint32_t (&lk)[16]) {
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(dds + col0 + c);
            if constexpr (!DQ) {
              float ds[4];
              f2_unpack(fmul2(f2_from(pr[c], pr[c + 1]), fsub2(f2_from(dr[c], dr[c + 1]), f2_pack(d4.x, d4.y))),
                        ds[0], ds[1]);
              f2_unpack(
                  fmul2(f2_from(pr[c + 2], pr[c + 3]), fsub2(f2_from(dr[c + 2], dr[c + 3]), f2_pack(d4.z, d4.w))),
                  ds[2], ds[3]);
              split_bf16x2(ds[0], ds[1], hk[c / 2], lk[c / 2]);
              split_bf16x2(ds[2], ds[3], hk[c / 2 + 1], lk[c / 2 + 1]);
            } else {
              uint64_t ds01 =
                  fmul2(f2_from(pr[c], pr[c + 1]), fsub2(f2_from(dr[c], dr[c + 1]), f2_pack(d4.x, d4.y)));
              uint64_t ds23 =
                  fmul2(f2_from(pr[c + 2], pr[c + 3]), fsub2(f2_from(dr[c + 2], dr[c + 3]), f2_pack(d4.z, d4.w)));
              float ds[4];
              f2_unpack(ds01, ds[0], ds[1]);
              f2_unpack(ds23, ds[2], ds[3]);
              split_bf16x2(ds[0], ds[1], hk[c / 2], lk[c / 2]);
              split_bf16x2(ds[2], ds[3], hk[c / 2 + 1], lk[c / 2 + 1]);
              float q0, q1, q2, q3;
              f2_unpack(fmul2(ds01, sc2), q0, q1);
              f2_unpack(fmul2(ds23, sc2), q2, q3);
              // the dP^T values just consumed make room for the packed pairs;
              // a key row past the sequence's valid length (not masked
              // without the causal rule) gives no dQ share
              dr[c] = key_live ? pack_bf16x2(q0, q1) : 0u;
              dr[c + 1] = key_live ? pack_bf16x2(q2, q3) : 0u;
            }
          }
          if constexpr (DQ) {
            const uint32_t row_base = ds_tile(ldn) + w * 16384 + r * 128;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t chunk = static_cast<uint32_t>(((col0 & 63) >> 3) + k);
              st_shared_v4(row_base + ((chunk ^ (r & 7)) << 4), dr[8 * k], dr[8 * k + 1], dr[8 * k + 4],
                           dr[8 * k + 5]);
            }
          }
        };
        // Column slice of this warpgroup: S^T [64w, 64w+64), dP^T likewise.
        // After use the slice holds P^T in S cols [64w, 64w+32) and dS^T hi
        // and lo in dP cols [64w, 64w+32) and [64w+32, 64w+64); every store
        // lands on columns this thread has already read.  P^T is published
        // first so the MMA thread can run dV += P^T dO, and then S^T of the
        // next query tile, while dS^T is still being computed.
        const uint32_t tS = tmem + lane_off + L::kColS + 64 * w;
        const uint32_t tD = tmem + lane_off + L::kColDP + 64 * w;
        {
          uint32_t s0[32], s1[32], d0[32], d1[32], pk[16], hk[16], lk[16];
          tmem_ld32(tS, s0);
          tmem_ld32(tS + 32, s1);
          tmem_ld_wait();
          if (need_mask) pchunk(std::true_type{}, s0, 64 * w, pk, bb0);
          else pchunk(std::false_type{}, s0, 64 * w, pk, bb0);
          tmem_st16(tS, pk);
          if (need_mask) pchunk(std::true_type{}, s1, 64 * w + 32, pk, bb1);
          else pchunk(std::false_type{}, s1, 64 * w + 32, pk, bb1);
          tmem_st16(tS + 16, pk);
          // publish P before taking dP, so that the GEMM reading P (and the
          // next tile's S behind it) queue up while dP is still running
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive_warp(BAR(L::P_READY));
          if constexpr (DQ) {
            // the previous tile's dQ share (computed while this tile's P ran)
            ok = dq_share_flush<D>(BAR(L::DQ_FULL), BAR(L::DQ_EMPTY), dqn, pend_head, pend_i, pend_lq, dq_cols, dq,
                                   geom.nq, r, w, wc, unit);
            if (!ok) break;
          }
          ok = warp_wait(BAR(L::DP_FULL), sdp_parity, wc, SITE_KV_EW_DP, unit);
          if (!ok) break;
          tc_fence_after();
          tmem_ld32(tD, d0);
          tmem_ld32(tD + 32, d1);
          if constexpr (DQ) {
            // the dS tile's buffer: free once the previous dQ product read it
            // (own buffer), or once dV has read the dO tile it overwrites
            ok = L::kDsOwn ? warp_wait(BAR(L::DS_FREE), (dsn & 1) ^ 1, wc, SITE_KV_EW_DSW, unit)
                           : warp_wait(BAR(L::DV_DONE), dsn & 1, wc, SITE_KV_EW_DSW, unit);
            ++dsn;
            tmem_ld_wait();
            if (!ok) break;
          } else {
            tmem_ld_wait();
          }
          dchunk(s0, d0, 64 * w, hk, lk);
          tmem_st16(tD, hk);
          tmem_st16(tD + 32, lk);
          dchunk(s1, d1, 64 * w + 32, hk, lk);
          tmem_st16(tD + 16, hk);
          tmem_st16(tD + 48, lk);
        }
        tmem_st_wait();
        tc_fence_before();
        if constexpr (DQ) fence_proxy_async_smem();  // the dS tile, for the tensor core
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(BAR(L::DS_READY));
          mbar_arrive(BAR(L::LD_EMPTY + ls));
        }
        ++ldn;
        if constexpr (DQ) {
          pend_head = head;
          pend_i = i;
          pend_lq = hl.lq;
        }
      }
      if (!ok) break;
      if constexpr (DQ) {
        ok = dq_share_flush<D>(BAR(L::DQ_FULL), BAR(L::DQ_EMPTY), dqn, pend_head, pend_i, pend_lq, dq_cols, dq,
                               geom.nq, r, w, wc, unit);
        if (!ok) break;
      }
      // epilogue: warpgroup 0 writes dV, warpgroup 1 writes scale * dK; key
      // rows past the valid length (and tiles no query sees) get zeros
      const int row = j * kTileRows + r;
      const bool valid = row < geom.nk;
      float* dst = (w == 0 ? dv : dk) + (static_cast<size_t>(head) * geom.nk + row) * D;
      if (i0 == i1) {
        if (valid) {
          const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
          for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(dst + c) = z;
        }
        continue;
      }
      ok = warp_wait(BAR(L::ACC_FULL), an & 1, wc, SITE_KV_EW_ACC, unit);
      if (!ok) break;
      ++an;
      tc_fence_after();
      const uint32_t col = (w == 0) ? L::kColDV : L::kColDK;
      const float mul = (w == 0) ? 1.0f : scale;
      // a padding key row may have met scores far above its queries' LSE:
      // select zeros rather than scale what it accumulated
      const bool live = row < hl.lk;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + col + 32 * c, v);
        tmem_ld_wait();
        if (!live) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        if (valid) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float4 o4;
            o4.x = __uint_as_float(v[4 * e + 0]) * mul;
            o4.y = __uint_as_float(v[4 * e + 1]) * mul;
            o4.z = __uint_as_float(v[4 * e + 2]) * mul;
            o4.w = __uint_as_float(v[4 * e + 3]) * mul;
            *reinterpret_cast<float4*>(dst + 32 * c + 4 * e) = o4;
          }
        }
      }
    }
  } else {
   regs_decrease<kKvOtherRegs>();
   if (warp == 8) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_keep = l2_policy_evict_last();
      const uint64_t pol_once = l2_policy_evict_first();
      uint32_t kvn = 0, qdpos = 0;
      SchedIter it = sched_begin(sp);
      int head, j;
      bool ok = true;
      while (ok && sched_next(it, sp, blockIdx.x, head, j)) {
        int i0, i1;
        key_tile_queries(head_len(geom, head), j, CAUSAL, i0, i1);
        if (i0 == i1) continue;
        const int unit = head * sp.units_per_head + j;
        ok = wait_bounded(BAR(L::KV_EMPTY), (kvn & 1) ^ 1, wc, SITE_KV_LOAD_KV, unit);
        if (!ok) break;
        ++kvn;
        mbar_arrive_expect_tx(BAR(L::KV_FULL), 2 * L::kTileBytes);
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb) {
          tma_load_3d_hint(sbase + L::kKOff + kb * 16384, &tm_k, BAR(L::KV_FULL), kb * 64, j * kTileRows, head,
                           pol_once);
          tma_load_3d_hint(sbase + L::kVOff + kb * 16384, &tm_v, BAR(L::KV_FULL), kb * 64, j * kTileRows, head,
                           pol_once);
        }
        for (int i = i0; i < i1; ++i) {
          const uint32_t s = qdpos % S, use = qdpos / S;
          ok = wait_bounded(BAR(L::QD_EMPTY + s), (use & 1) ^ 1, wc, SITE_KV_LOAD_QD, unit);
          if (!ok) break;
          if (blockIdx.x == 0 && static_cast<int>(kvn) - 1 == stall_unit && i == i0) {
            // testing hook: leave this (Q, dO) stage unloaded so the waits on
            // it run out and the kernel reports a timeout instead of hanging
            ++qdpos;
            continue;
          }
          mbar_arrive_expect_tx(BAR(L::QD_FULL + s), 2 * L::kTileBytes);
          const uint32_t qa = sbase + L::kQdOff + s * 2 * L::kTileBytes;
#pragma unroll
          for (int kb = 0; kb < D / 64; ++kb) {
            tma_load_3d_hint(qa + kb * 16384, &tm_q, BAR(L::QD_FULL + s), kb * 64, i * kTileRows, head, pol_keep);
            tma_load_3d_hint(qa + L::kTileBytes + kb * 16384, &tm_do, BAR(L::QD_FULL + s), kb * 64, i * kTileRows,
                             head, pol_keep);
          }
          ++qdpos;
        }
      }
      if (!ok) {
        if (kvn > 0) drain_wait(BAR(L::KV_FULL), (kvn - 1) & 1, limit_ns);
        for (uint32_t s = 0; s < static_cast<uint32_t>(S); ++s) {
          if (qdpos > s) {
            const uint32_t last = qdpos - 1 - ((qdpos - 1 - s) % S);
            drain_wait(BAR(L::QD_FULL + s), (last / S) & 1, limit_ns);
          }
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_acc = idesc_bf16_f32(128, D, false, true);
      // Descriptors built once; a stage or K step only moves the start-address
      // field (16-byte units), a plain add.  K-major views feed S^T and dP^T,
      // MN-major views (next 64-column block 16 KB away) feed dV and dK.
      constexpr uint32_t kTileUnits = L::kTileBytes >> 4;
      const SDesc kdesc = sdesc_sw128(sbase + L::kKOff, 16, 1024);
      const SDesc vdesc = sdesc_sw128(sbase + L::kVOff, 16, 1024);
      const SDesc qd_k0 = sdesc_sw128(sbase + L::kQdOff, 16, 1024);
      const SDesc qd_mn0 = sdesc_sw128(sbase + L::kQdOff, kTileRows * 128, 1024);
      auto q_k = [&](uint32_t pos) { return qd_k0 + (pos % S) * (2 * kTileUnits); };
      auto q_mn = [&](uint32_t pos) { return qd_mn0 + (pos % S) * (2 * kTileUnits); };
      // DQ: dQ_i += (scale dS) K, M = 128 queries, N = d, K = 128 keys; the
      // dS tile and K both MN-major (rows of 64 queries / d columns per key)
      constexpr uint32_t id_dq = idesc_bf16_f32(128, D, true, true);
      const SDesc k_mn = sdesc_sw128(sbase + L::kKOff, kTileRows * 128, 1024);
      uint32_t dq_issued = 0, dq_freed = 0;
      // waits until the elementwise warps have read every dQ share issued so
      // far out of tensor memory (at most one is outstanding)
      auto wait_dq_free = [&](int unit) -> bool {
        while (dq_freed < dq_issued) {
          if (!wait_bounded(BAR(L::DQ_EMPTY), dq_freed & 1, wc, SITE_KV_MMA_DQE, unit)) return false;
          ++dq_freed;
        }
        tc_fence_after();
        return true;
      };
      uint32_t kvn = 0, qdpos = 0, pn = 0;
      SchedIter it = sched_begin(sp);
      int head, j;
      bool ok = true;
      while (ok && sched_next(it, sp, blockIdx.x, head, j)) {
        int i0, i1;
        key_tile_queries(head_len(geom, head), j, CAUSAL, i0, i1);
        if (i0 == i1) continue;
        const int unit = head * sp.units_per_head + j;
        ok = wait_bounded(BAR(L::KV_FULL), kvn & 1, wc, SITE_KV_MMA_KV, unit);
        if (!ok) break;
        ++kvn;
        // S^T = K Q^T and dP^T = V dO^T of one query tile: M = 128 keys,
        // N = 128 queries, K = d
        auto issue_s = [&](SDesc qd) {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
            umma_ss(tmem + L::kColS, kdesc + off, qd + off, id_s, ks > 0 ? 1u : 0u);
          }
          umma_commit(BAR(L::S_FULL));
        };
        auto issue_dp = [&](SDesc dd) {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
            umma_ss(tmem + L::kColDP, vdesc + off, dd + off, id_s, ks > 0 ? 1u : 0u);
          }
          umma_commit(BAR(L::DP_FULL));
        };
        ok = wait_bounded(BAR(L::QD_FULL + qdpos % S), (qdpos / S) & 1, wc, SITE_KV_MMA_QD, unit);
        if (!ok) break;
        tc_fence_after();
        issue_s(q_k(qdpos));
        // DQ, d = 128: the dP^T columns hold the last dQ share until it is read
        if (DQ && L::kColDQ == L::kColDP && !wait_dq_free(unit)) {
          ok = false;
          break;
        }
        issue_dp(q_k(qdpos) + kTileUnits);
        // Per query tile i: dV += P^T dO once P^T is stored; then S^T of tile
        // i+1, which overwrites P^T(i) only after dV(i) has read it (the
        // tensor pipe runs in issue order), so the elementwise warps find
        // S^T(i+1) ready when they finish tile i; then dK += dS^T Q (hi and
        // lo, both in the dP^T columns); then dP^T of tile i+1, behind dK(i).
        // M = 128 keys, N = d, K = 128 queries; the warpgroup w's P^T sits in
        // S columns [64 w, 64 w + 32), its dS^T hi and lo in dP columns
        // [64 w, 64 w + 32) and [64 w + 32, 64 w + 64).
        for (int i = i0; i < i1; ++i) {
          const uint32_t s = qdpos % S;
          const SDesc qmn = q_mn(qdpos);
          const SDesc dmn = qmn + kTileUnits;
          ok = wait_bounded(BAR(L::P_READY), pn & 1, wc, SITE_KV_MMA_PDS, unit);
          if (!ok) break;
          tc_fence_after();
          const bool first = (i == i0);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t acol = 64 * (ks >> 2) + 8 * (ks & 3);
            umma_ts(tmem + L::kColDV, tmem + L::kColS + acol, dmn + static_cast<uint32_t>((ks * 2048) >> 4), id_acc,
                    (!first || ks > 0) ? 1u : 0u);
          }
          if constexpr (DQ) {
            if (!L::kDsOwn) umma_commit(BAR(L::DV_DONE));  // its dO tile becomes the dS tile
          }
          const bool more = i + 1 < i1;
          if (more) {
            ok = wait_bounded(BAR(L::QD_FULL + (qdpos + 1) % S), ((qdpos + 1) / S) & 1, wc, SITE_KV_MMA_QD, unit);
            if (!ok) break;
            tc_fence_after();
            issue_s(q_k(qdpos + 1));
          }
          ok = wait_bounded(BAR(L::DS_READY), pn & 1, wc, SITE_KV_MMA_PDS, unit);
          if (!ok) break;
          ++pn;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t acol = 64 * (ks >> 2) + 8 * (ks & 3);
            umma_ts(tmem + L::kColDK, tmem + L::kColDP + acol, qmn + static_cast<uint32_t>((ks * 2048) >> 4), id_acc,
                    (!first || ks > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {  // dS^T lo part
            const uint32_t acol = 32 + 64 * (ks >> 2) + 8 * (ks & 3);
            umma_ts(tmem + L::kColDK, tmem + L::kColDP + acol, qmn + static_cast<uint32_t>((ks * 2048) >> 4), id_acc,
                    1u);
          }
          if constexpr (DQ) {
            // this tile's dQ share (at d = 128 over the dP^T columns, which
            // the dK products above have read: the pipe runs in issue order)
            if (L::kColDQ != L::kColDP && !wait_dq_free(unit)) {
              ok = false;
              break;
            }
            const SDesc ds_mn = sdesc_sw128(ds_tile(qdpos), kTileRows * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t off = static_cast<uint32_t>((ks * 2048) >> 4);
              umma_ss(tmem + L::kColDQ, ds_mn + off, k_mn + off, id_dq, ks > 0 ? 1u : 0u);
            }
            umma_commit(BAR(L::DQ_FULL));
            ++dq_issued;
            if (L::kDsOwn) umma_commit(BAR(L::DS_FREE));
          }
          umma_commit(BAR(L::QD_EMPTY + s));
          ++qdpos;
          if (more) {
            if (DQ && L::kColDQ == L::kColDP && !wait_dq_free(unit)) {
              ok = false;
              break;
            }
            issue_dp(q_k(qdpos) + kTileUnits);
          }
        }
        if (!ok) break;
        umma_commit(BAR(L::ACC_FULL));
        umma_commit(BAR(L::KV_EMPTY));
      }
      umma_commit(BAR(L::DRAIN));
      drain_wait(BAR(L::DRAIN), 0, limit_ns);
    }
  } else if (warp == 10) {
    // ------------------------------------------- LSE / D rows of each query tile
    const float* lse_h = nullptr;
    uint32_t ldn = 0;
    float* ld_base = reinterpret_cast<float*>(smem + L::kLdOff);
    SchedIter it = sched_begin(sp);
    int head, j;
    bool ok = true;
    while (ok && sched_next(it, sp, blockIdx.x, head, j)) {
      const HeadLen hl = head_len(geom, head);
      int i0, i1;
      key_tile_queries(hl, j, CAUSAL, i0, i1);
      const int unit = head * sp.units_per_head + j;
      lse_h = lse + static_cast<size_t>(head) * geom.nq;
      const float* d_h = delta + static_cast<size_t>(head) * geom.nq;
      for (int i = i0; i < i1; ++i) {
        const uint32_t ls = ldn % S;
        ok = warp_wait(BAR(L::LD_EMPTY + ls), ((ldn / S) & 1) ^ 1, wc, SITE_KV_LD_EMPTY, unit);
        if (!ok) break;
        float* l2s = ld_base + ls * 256;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int idx = lane * 4 + t;
          const int q = i * kTileRows + idx;
          const float lv = q < hl.lq ? lse_h[q] : -CUDART_INF_F;
          const bool in = lv > -CUDART_INF_F;  // a valid query with at least one key
          l2s[idx] = in ? -lv * kLog2e : -CUDART_INF_F;
          l2s[128 + idx] = in ? d_h[q] : 0.f;
        }
        mbar_arrive_warp(BAR(L::LD_FULL + ls));
        ++ldn;
      }
    }
  }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ dQ

template <int D>
struct QLayout {
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kStages = (D == 128) ? 2 : 4;  // (K, V) ring
  static constexpr int kQOff = 0;
  static constexpr int kDoOff = kTileBytes;
  static constexpr int kKvOff = 2 * kTileBytes;  // stage s: K at +0, V at +kTileBytes
  static constexpr int kXchOff = kKvOff + kStages * 2 * kTileBytes;  // [2 units][2 warpgroups][128] fp32
  static constexpr int kDdOff = kXchOff + 2 * 2 * 128 * 4;            // [2 units][128] fp32 row terms D'
  static constexpr int kBarOff = kDdOff + 2 * 128 * 4;
  static constexpr int Q_FULL = 0;
  static constexpr int Q_EMPTY = 1;
  static constexpr int KV_FULL = 2;
  static constexpr int KV_EMPTY = KV_FULL + kStages;
  static constexpr int S_FULL = KV_EMPTY + kStages;  // S computed
  static constexpr int DP_FULL = S_FULL + 1;          // dP computed
  static constexpr int P_READY = DP_FULL + 1;         // P stored (one arrive per elementwise warp)
  static constexpr int DS_FULL = P_READY + 1;
  static constexpr int ACC_FULL = DS_FULL + 1;
  static constexpr int XCH = ACC_FULL + 1;
  static constexpr int DD_FULL = XCH + 1;       // 2 slots: D' of a unit written (two loader warps)
  static constexpr int DD_EMPTY = DD_FULL + 2;  // 2 slots: D' read (one arrive per elementwise warp)
  static constexpr int DRAIN = DD_EMPTY + 2;
  static constexpr int kNumBars = DRAIN + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  // S [0,128): after use P (bf16) in each warpgroup's first 32 columns;
  // dP [128,256): dS (bf16) in each warpgroup's first 32 columns;
  // dQ accumulator [256, 256+d); B = sum_j P_ij k_j accumulator [256+d, 256+2d).
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColB = 256 + D;
};

// 12 warps: two elementwise warpgroups, TMA (warp 8), MMA (warp 9) and the two
// row-term loaders (warps 10, 11) completing the third warpgroup.  Launched
// at 168 registers a thread: the elementwise warpgroups take 184, the third
// keeps 136.
constexpr int kQThreads = 384;
constexpr int kQLaunchRegs = 168;
constexpr int kQEwRegs = 184;
constexpr int kQOtherRegs = 136;
static_assert(2 * 128 * kQEwRegs + 128 * kQOtherRegs <= kQThreads * kQLaunchRegs,
              "register split exceeds the launch allocation");

template <int D, bool CAUSAL, bool BIAS>
__global__ void __launch_bounds__(kQThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const float* __restrict__ lse, const void* __restrict__ o, const uint16_t* __restrict__ dout,
              const int o_bf16, float* __restrict__ delta, float* __restrict__ dq, const SeqGeom geom,
              const float scale, const float scale_log2, const SchedParams sp, int* status,
              const unsigned long long limit_ns, const int stall_unit, const BiasRef bias) {
  using L = QLayout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kBarOff;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bars + 8 * L::Q_FULL, 1);
    mbar_init(bars + 8 * L::Q_EMPTY, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bars + 8 * (L::KV_FULL + s), 1);
      mbar_init(bars + 8 * (L::KV_EMPTY + s), 1);
    }
    mbar_init(bars + 8 * L::S_FULL, 1);
    mbar_init(bars + 8 * L::DP_FULL, 1);
    mbar_init(bars + 8 * L::P_READY, 8);
    mbar_init(bars + 8 * L::DS_FULL, 8);
    mbar_init(bars + 8 * L::ACC_FULL, 1);
    mbar_init(bars + 8 * L::XCH, 8);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bars + 8 * (L::DD_FULL + s), 2);  // the two loader warps
      mbar_init(bars + 8 * (L::DD_EMPTY + s), 8);
    }
    mbar_init(bars + 8 * L::DRAIN, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, status, limit_ns};
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };

  if (warp < 8) {
    // ------------------------------------------------- dS (thread = query row)
    regs_increase<kQEwRegs>();
    // The row term comes in as D'_i = rowsum(dO o O) (computed by the loader
    // warps one unit ahead) with O from the forward pass, whose P was rounded
    // to bf16 for the PV product.  The kernel sees every key of its rows, so
    // it also sums delta_i = sum_j dS'_ij = sum_j P_ij dP_ij - D'_i in fp32,
    // corrects its own product with
    // dQ = scale (sum_j dS'_ij k_j - delta_i sum_j P_ij k_j), and stores the
    // corrected D_i = D'_i + delta_i for the dK/dV kernel.
    const int w = warp >> 2;  // key columns [64 w, 64 w + 64)
    const int r = ((warp & 3) << 5) + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    float* xch = reinterpret_cast<float*>(smem + L::kXchOff);
    const float* dd_s = reinterpret_cast<const float*>(smem + L::kDdOff);
    uint32_t sn = 0, an = 0, ddn = 0;
    SchedIter it = sched_begin(sp);
    int head, i;
    bool ok = true;
    while (ok && sched_next(it, sp, blockIdx.x, head, i)) {
      const HeadLen hl = head_len(geom, head);
      const int nk = query_tile_keys(hl, i, CAUSAL);
      const int unit = head * sp.units_per_head + i;
      const int row = i * kTileRows + r;
      const bool valid = row < geom.nq;
      const size_t ridx = static_cast<size_t>(head) * geom.nq + row;
      float* dst = dq + ridx * D;
      if (nk == 0) {
        // padding rows, or rows that see no key: zero gradient and row term
        if (valid) {
          const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
          for (int c = w * (D / 2); c < (w + 1) * (D / 2); c += 4) *reinterpret_cast<float4*>(dst + c) = z;
          if (w == 0) delta[ridx] = 0.f;
        }
        continue;
      }
      const float lv = row < hl.lq ? lse[ridx] : -CUDART_INF_F;
      const bool has = lv > -CUDART_INF_F;  // a valid row with at least one key
      const float l2 = has ? lv * kLog2e : CUDART_INF_F;
      ok = warp_wait(BAR(L::DD_FULL + (ddn & 1)), (ddn >> 1) & 1, wc, SITE_Q_EW_DD, unit);
      if (!ok) break;
      const float dd = has ? dd_s[(ddn & 1) * 128 + r] : 0.f;
      mbar_arrive_warp(BAR(L::DD_EMPTY + (ddn & 1)));
      ++ddn;
      const float nl2 = -l2;
      const uint64_t c2 = f2_pack(scale_log2, scale_log2);
      const uint64_t nl2x2 = f2_pack(nl2, nl2);
      const uint64_t dd2 = f2_pack(dd, dd);
      float dsum = 0.f;  // this warpgroup's share of delta_i
      // additive mask: this row's keys (none for padding rows)
      const uint16_t* brow = nullptr;
      bool bvec = false;
      if constexpr (BIAS) {
        const int bidx = head / geom.heads_per_batch;
        if (row < hl.lq) {
          brow = bias.p + bidx * bias.sb + (head - bidx * geom.heads_per_batch) * bias.sh + row * bias.sq;
          bvec = (reinterpret_cast<uintptr_t>(brow) & 15) == 0;
        }
      }
      for (int jt = 0; jt < nk; ++jt) {
        // the mask of the warpgroup's 64 keys, fetched before the wait
        uint32_t bb0[BIAS ? 16 : 1], bb1[BIAS ? 16 : 1];
        if constexpr (BIAS) {
          load_bias_row(brow, bvec, jt * kTileRows + 64 * w, geom.nk, bb0, bb1);
          // the next key tile's 128 bytes of this row towards L2
          const int knext = (jt + 1) * kTileRows + 64 * w;
          if (brow && jt + 1 < nk && knext + 64 <= geom.nk) prefetch_l2(brow + knext);
        }
        // P needs only S: dP may still be in the tensor pipe
        const uint32_t sdp_parity = sn & 1;
        ok = warp_wait(BAR(L::S_FULL), sdp_parity, wc, SITE_Q_EW_S, unit);
        if (!ok) break;
        ++sn;
        tc_fence_after();
        const bool diag = CAUSAL && tile_crosses_diagonal(hl, i, jt);
        const bool tail = (jt == hl.nkt - 1) && ((hl.lk & (kTileRows - 1)) != 0);
        // number of eligible key columns of this tile for this row
        const bool need_mask = diag || tail;
        const int lim = need_mask ? ((CAUSAL ? min(row + hl.off + 1, hl.lk) : hl.lk) - jt * kTileRows) : kTileRows;
        // Phase 1: P for 32 key columns starting at col0, kept in sr as fp32
        // bits and packed to bf16 in pk.  MASKED: a tile crossing the causal
        // boundary or holding the last valid key, where some key columns are
        // not eligible.
        auto pchunk = [&](auto masked, uint32_t (&sr)[32], int col0, uint32_t (&pk)[16],
                          const uint32_t (&bh)[BIAS ? 16 : 1]) {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float p0, p1;
            uint64_t t = nl2x2;
            // + bias * log2(e); a hidden key (-inf) gives p = 0
            if constexpr (BIAS) t = ffma2(bf16x2_to_f2(bh[c / 2]), f2_pack(kLog2e, kLog2e), t);
            f2_unpack(ffma2(f2_from(sr[c], sr[c + 1]), c2, t), p0, p1);
            p0 = ex2_approx(p0);
            p1 = ex2_approx(p1);
            if (decltype(masked)::value) {
              if (col0 + c >= lim) p0 = 0.f;
              if (col0 + c + 1 >= lim) p1 = 0.f;
            }
            sr[c] = __float_as_uint(p0);
            sr[c + 1] = __float_as_uint(p1);
            pk[c / 2] = pack_bf16x2(p0, p1);
          }
        };
        // Phase 2: dS = P o (dP - D), its row sum, and dS rounded to bf16
        auto dchunk = [&](const uint32_t (&pr)[32], const uint32_t (&dr)[32], uint32_t (&hk)[16]) {
          uint64_t acc = f2_pack(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float ds0, ds1;
            const uint64_t ds01 = fmul2(f2_from(pr[c], pr[c + 1]), fsub2(f2_from(dr[c], dr[c + 1]), dd2));
            acc = fadd2(acc, ds01);
            f2_unpack(ds01, ds0, ds1);
            hk[c / 2] = pack_bf16x2(ds0, ds1);
          }
          float a0, a1;
          f2_unpack(acc, a0, a1);
          dsum += a0 + a1;
        };
        // After use the warpgroup's slice holds P in S cols [64w, 64w+32) and
        // dS in dP cols [64w, 64w+32); each store lands on columns this
        // thread has already read.  P is published
        // first so that B += P K, and then S of the next key tile, queue
        // behind dP in the tensor pipe.
        const uint32_t tS = tmem + lane_off + L::kColS + 64 * w;
        const uint32_t tD = tmem + lane_off + L::kColDP + 64 * w;
        {
          uint32_t s0[32], s1[32], d0[32], d1[32], pk[16], hk[16];
          tmem_ld32(tS, s0);
          tmem_ld32(tS + 32, s1);
          tmem_ld_wait();
          if (need_mask) pchunk(std::true_type{}, s0, 64 * w, pk, bb0);
          else pchunk(std::false_type{}, s0, 64 * w, pk, bb0);
          tmem_st16(tS, pk);
          if (need_mask) pchunk(std::true_type{}, s1, 64 * w + 32, pk, bb1);
          else pchunk(std::false_type{}, s1, 64 * w + 32, pk, bb1);
          tmem_st16(tS + 16, pk);
          // publish P before taking dP, so that the GEMM reading P (and the
          // next tile's S behind it) queue up while dP is still running
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive_warp(BAR(L::P_READY));
          ok = warp_wait(BAR(L::DP_FULL), sdp_parity, wc, SITE_Q_EW_DP, unit);
          if (!ok) break;
          tc_fence_after();
          tmem_ld32(tD, d0);
          tmem_ld32(tD + 32, d1);
          tmem_ld_wait();
          dchunk(s0, d0, hk);
          tmem_st16(tD, hk);
          dchunk(s1, d1, hk);
          tmem_st16(tD + 16, hk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(BAR(L::DS_FULL));
      }
      if (!ok) break;
      // combine the two warpgroups' halves of delta_i (slots alternate by unit)
      float* slot = xch + (an & 1) * 256;
      slot[w * 128 + r] = dsum;
      mbar_arrive_warp(BAR(L::XCH));
      ok = warp_wait(BAR(L::XCH), an & 1, wc, SITE_Q_EW_XCH, unit);
      if (!ok) break;
      const float dlt = slot[r] + slot[128 + r];
      ok = warp_wait(BAR(L::ACC_FULL), an & 1, wc, SITE_Q_EW_ACC, unit);
      if (!ok) break;
      ++an;
      tc_fence_after();
      if (w == 0 && valid) delta[ridx] = has ? dd + dlt : 0.f;
      // warpgroup w writes dQ columns [w d/2, (w+1) d/2)
      const float mul = has ? scale : 0.f;
#pragma unroll 1
      for (int c = w * (D / 64); c < (w + 1) * (D / 64); ++c) {
        uint32_t v[32], bv[32];
        tmem_ld32(tmem + lane_off + L::kColDQ + 32 * c, v);
        tmem_ld32(tmem + lane_off + L::kColB + 32 * c, bv);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float4 o4;
            o4.x = (__uint_as_float(v[4 * e + 0]) - dlt * __uint_as_float(bv[4 * e + 0])) * mul;
            o4.y = (__uint_as_float(v[4 * e + 1]) - dlt * __uint_as_float(bv[4 * e + 1])) * mul;
            o4.z = (__uint_as_float(v[4 * e + 2]) - dlt * __uint_as_float(bv[4 * e + 2])) * mul;
            o4.w = (__uint_as_float(v[4 * e + 3]) - dlt * __uint_as_float(bv[4 * e + 3])) * mul;
            *reinterpret_cast<float4*>(dst + 32 * c + 4 * e) = o4;
          }
        }
      }
    }
  } else {
   regs_decrease<kQOtherRegs>();
   if (warp == 8) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_keep = l2_policy_evict_last();
      const uint64_t pol_once = l2_policy_evict_first();
      uint32_t qn = 0, kvpos = 0;
      SchedIter it = sched_begin(sp);
      int head, i;
      bool ok = true;
      while (ok && sched_next(it, sp, blockIdx.x, head, i)) {
        const int nk = query_tile_keys(head_len(geom, head), i, CAUSAL);
        if (nk == 0) continue;
        const int unit = head * sp.units_per_head + i;
        ok = wait_bounded(BAR(L::Q_EMPTY), (qn & 1) ^ 1, wc, SITE_Q_LOAD_Q, unit);
        if (!ok) break;
        ++qn;
        mbar_arrive_expect_tx(BAR(L::Q_FULL), 2 * L::kTileBytes);
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb) {
          tma_load_3d_hint(sbase + L::kQOff + kb * 16384, &tm_q, BAR(L::Q_FULL), kb * 64, i * kTileRows, head,
                           pol_once);
          tma_load_3d_hint(sbase + L::kDoOff + kb * 16384, &tm_do, BAR(L::Q_FULL), kb * 64, i * kTileRows, head,
                           pol_once);
        }
        for (int jt = 0; jt < nk; ++jt) {
          const uint32_t s = kvpos % S, use = kvpos / S;
          ok = wait_bounded(BAR(L::KV_EMPTY + s), (use & 1) ^ 1, wc, SITE_Q_LOAD_KV, unit);
          if (!ok) break;
          if (blockIdx.x == 0 && static_cast<int>(qn) - 1 == stall_unit && jt == 0) {
            // testing hook: leave this (K, V) stage unloaded (see dK/dV)
            ++kvpos;
            continue;
          }
          mbar_arrive_expect_tx(BAR(L::KV_FULL + s), 2 * L::kTileBytes);
          const uint32_t ka = sbase + L::kKvOff + s * 2 * L::kTileBytes;
#pragma unroll
          for (int kb = 0; kb < D / 64; ++kb) {
            tma_load_3d_hint(ka + kb * 16384, &tm_k, BAR(L::KV_FULL + s), kb * 64, jt * kTileRows, head, pol_keep);
            tma_load_3d_hint(ka + L::kTileBytes + kb * 16384, &tm_v, BAR(L::KV_FULL + s), kb * 64, jt * kTileRows,
                             head, pol_keep);
          }
          ++kvpos;
        }
      }
      if (!ok) {
        if (qn > 0) drain_wait(BAR(L::Q_FULL), (qn - 1) & 1, limit_ns);
        for (uint32_t s = 0; s < static_cast<uint32_t>(S); ++s) {
          if (kvpos > s) {
            const uint32_t last = kvpos - 1 - ((kvpos - 1 - s) % S);
            drain_wait(BAR(L::KV_FULL + s), (last / S) & 1, limit_ns);
          }
        }
      }
    }
  } else if (warp >= 10) {
    // ---------------------------- row term D'_i = sum_c dO_ic O_ic, one unit ahead
    // Warps 10 and 11 take 64 rows each, 16 rows per step with all their
    // loads in flight (O streams from HBM); within a row, lane l takes
    // columns [CW l, CW l + CW) of O (fp32 or bf16) and dO, then a warp sum.
    constexpr int CW = D / 32;
    constexpr int kRowsPerStep = 16;
    float* dds = reinterpret_cast<float*>(smem + L::kDdOff);
    const int lw = warp - 10;
    uint32_t ddn = 0;
    SchedIter it = sched_begin(sp);
    int head, i;
    bool ok = true;
    while (ok && sched_next(it, sp, blockIdx.x, head, i)) {
      const HeadLen hl = head_len(geom, head);
      if (query_tile_keys(hl, i, CAUSAL) == 0) continue;  // the elementwise warps skip it too
      const int unit = head * sp.units_per_head + i;
      ok = warp_wait(BAR(L::DD_EMPTY + (ddn & 1)), ((ddn >> 1) & 1) ^ 1, wc, SITE_Q_DD_EMPTY, unit);
      if (!ok) break;
      float* slot = dds + (ddn & 1) * 128;
#pragma unroll 1
      for (int r0 = 64 * lw; r0 < 64 * lw + 64; r0 += kRowsPerStep) {
        float ov[kRowsPerStep][CW];
        uint32_t dh[kRowsPerStep][CW / 2];
#pragma unroll
        for (int u = 0; u < kRowsPerStep; ++u) {
          const int row = i * kTileRows + r0 + u;
          const bool in = row < hl.lq;
          const size_t base = (static_cast<size_t>(head) * geom.nq + (in ? row : 0)) * D + CW * lane;
          if (o_bf16) {
            const uint16_t* op = static_cast<const uint16_t*>(o) + base;
            if constexpr (CW == 4) {
              const uint2 h = in ? __ldg(reinterpret_cast<const uint2*>(op)) : make_uint2(0u, 0u);
              ov[u][0] = bf16_bits_to_float(h.x & 0xFFFFu); ov[u][1] = bf16_bits_to_float(h.x >> 16);
              ov[u][2] = bf16_bits_to_float(h.y & 0xFFFFu); ov[u][3] = bf16_bits_to_float(h.y >> 16);
            } else {
              const uint32_t h = in ? __ldg(reinterpret_cast<const unsigned int*>(op)) : 0u;
              ov[u][0] = bf16_bits_to_float(h & 0xFFFFu); ov[u][1] = bf16_bits_to_float(h >> 16);
            }
          } else {
            const float* op = static_cast<const float*>(o) + base;
            if constexpr (CW == 4) {
              const float4 f = in ? __ldg(reinterpret_cast<const float4*>(op)) : make_float4(0.f, 0.f, 0.f, 0.f);
              ov[u][0] = f.x; ov[u][1] = f.y; ov[u][2] = f.z; ov[u][3] = f.w;
            } else {
              const float2 f = in ? __ldg(reinterpret_cast<const float2*>(op)) : make_float2(0.f, 0.f);
              ov[u][0] = f.x; ov[u][1] = f.y;
            }
          }
          if constexpr (CW == 4) {
            const uint2 h = in ? __ldg(reinterpret_cast<const uint2*>(dout + base)) : make_uint2(0u, 0u);
            dh[u][0] = h.x;
            dh[u][1] = h.y;
          } else {
            dh[u][0] = in ? __ldg(reinterpret_cast<const unsigned int*>(dout + base)) : 0u;
          }
        }
        float part[kRowsPerStep];
#pragma unroll
        for (int u = 0; u < kRowsPerStep; ++u) {
          part[u] = 0.f;
#pragma unroll
          for (int c = 0; c < CW / 2; ++c) {
            part[u] = fmaf(ov[u][2 * c], bf16_bits_to_float(dh[u][c] & 0xFFFFu), part[u]);
            part[u] = fmaf(ov[u][2 * c + 1], bf16_bits_to_float(dh[u][c] >> 16), part[u]);
          }
        }
        // sum over the lanes, 16 rows at once: after the butterfly every lane
        // holds all 16 totals, and lane l < 16 stores row r0 + l
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
          for (int u = 0; u < kRowsPerStep; ++u) part[u] += __shfl_xor_sync(0xffffffffu, part[u], off);
        }
        float mine = part[0];
#pragma unroll
        for (int u = 1; u < kRowsPerStep; ++u) mine = ((lane & 15) == u) ? part[u] : mine;
        if (lane < kRowsPerStep) slot[r0 + lane] = mine;
      }
      mbar_arrive_warp(BAR(L::DD_FULL + (ddn & 1)));
      ++ddn;
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_acc = idesc_bf16_f32(128, D, false, true);
      // Descriptors built once (see the dK/dV kernel): Q and dO K-major for
      // S and dP; the K/V stages K-major for S and dP, K MN-major for dQ and B.
      constexpr uint32_t kTileUnits = L::kTileBytes >> 4;
      const SDesc qdesc = sdesc_sw128(sbase + L::kQOff, 16, 1024);
      const SDesc dodesc = sdesc_sw128(sbase + L::kDoOff, 16, 1024);
      const SDesc kv_k0 = sdesc_sw128(sbase + L::kKvOff, 16, 1024);
      const SDesc kv_mn0 = sdesc_sw128(sbase + L::kKvOff, kTileRows * 128, 1024);
      auto kv_k = [&](uint32_t pos) { return kv_k0 + (pos % S) * (2 * kTileUnits); };
      auto kv_mn = [&](uint32_t pos) { return kv_mn0 + (pos % S) * (2 * kTileUnits); };
      uint32_t qn = 0, kvpos = 0, dn = 0;
      SchedIter it = sched_begin(sp);
      int head, i;
      bool ok = true;
      while (ok && sched_next(it, sp, blockIdx.x, head, i)) {
        const int nk = query_tile_keys(head_len(geom, head), i, CAUSAL);
        if (nk == 0) continue;
        const int unit = head * sp.units_per_head + i;
        ok = wait_bounded(BAR(L::Q_FULL), qn & 1, wc, SITE_Q_MMA_Q, unit);
        if (!ok) break;
        ++qn;
        // S = Q K^T and dP = dO V^T of one key tile: M = 128 queries,
        // N = 128 keys, K = d
        auto issue_s = [&](SDesc kd) {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
            umma_ss(tmem + L::kColS, qdesc + off, kd + off, id_s, ks > 0 ? 1u : 0u);
          }
          umma_commit(BAR(L::S_FULL));
        };
        auto issue_dp = [&](SDesc vd) {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
            umma_ss(tmem + L::kColDP, dodesc + off, vd + off, id_s, ks > 0 ? 1u : 0u);
          }
          umma_commit(BAR(L::DP_FULL));
        };
        ok = wait_bounded(BAR(L::KV_FULL + kvpos % S), (kvpos / S) & 1, wc, SITE_Q_MMA_KV, unit);
        if (!ok) break;
        tc_fence_after();
        issue_s(kv_k(kvpos));
        issue_dp(kv_k(kvpos) + kTileUnits);
        // Per key tile jt: B += P K once P is stored; then S of tile jt+1,
        // which overwrites P(jt) only after B(jt) has read it (the tensor
        // pipe runs in issue order); then dQ += dS K (dS in the dP columns);
        // then dP of tile jt+1, behind dQ(jt).  M = 128 queries, N = d,
        // K = 128 keys, K tile MN-major; the warpgroup w's P sits in S
        // columns [64 w, 64 w + 32), its dS in dP columns [64 w, 64 w + 32).
        for (int jt = 0; jt < nk; ++jt) {
          const uint32_t s = kvpos % S;
          const SDesc kmn = kv_mn(kvpos);
          ok = wait_bounded(BAR(L::P_READY), dn & 1, wc, SITE_Q_MMA_P, unit);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {  // B += P K, for the delta correction
            const uint32_t acol = 64 * (ks >> 2) + 8 * (ks & 3);
            umma_ts(tmem + L::kColB, tmem + L::kColS + acol, kmn + static_cast<uint32_t>((ks * 2048) >> 4), id_acc,
                    (jt > 0 || ks > 0) ? 1u : 0u);
          }
          const bool more = jt + 1 < nk;
          if (more) {
            ok = wait_bounded(BAR(L::KV_FULL + (kvpos + 1) % S), ((kvpos + 1) / S) & 1, wc, SITE_Q_MMA_KV, unit);
            if (!ok) break;
            tc_fence_after();
            issue_s(kv_k(kvpos + 1));
          }
          ok = wait_bounded(BAR(L::DS_FULL), dn & 1, wc, SITE_Q_MMA_DS, unit);
          if (!ok) break;
          ++dn;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t acol = 64 * (ks >> 2) + 8 * (ks & 3);
            umma_ts(tmem + L::kColDQ, tmem + L::kColDP + acol, kmn + static_cast<uint32_t>((ks * 2048) >> 4), id_acc,
                    (jt > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(BAR(L::KV_EMPTY + s));
          ++kvpos;
          if (more) issue_dp(kv_k(kvpos) + kTileUnits);
        }
        if (!ok) break;
        umma_commit(BAR(L::ACC_FULL));
        umma_commit(BAR(L::Q_EMPTY));
      }
      umma_commit(BAR(L::DRAIN));
      drain_wait(BAR(L::DRAIN), 0, limit_ns);
    }
  }

  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool BIAS>
cudaError_t launch_stage_t(const BwdArgs& a, int stage, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (stage == 0) {
    // dQ first: it forms D' = rowsum(dO o O) and turns it into the exact row term
    using L = QLayout<D>;
    auto kern = dq_kernel<D, CAUSAL, BIAS>;
    static std::atomic<unsigned long long> ready{0};
    e = setup_kernel_once(kern, L::kSmemBytes, kQLaunchRegs, ready);
    if (e != cudaSuccess) return e;
    kern<<<a.grid_q, kQThreads, L::kSmemBytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.lse, a.o, a.dout,
                                                         a.o_bf16, a.delta, a.dq, a.geom, a.scale, a.scale_log2,
                                                         a.sched_q, a.status, a.wait_limit_ns, a.stall_unit,
                                                         a.bias);
  } else if (stage == 1) {
    using L = KvLayout<D, false>;
    auto kern = dkdv_kernel<D, CAUSAL, BIAS, false>;
    static std::atomic<unsigned long long> ready{0};
    e = setup_kernel_once(kern, L::kSmemBytes, kKvLaunchRegs, ready);
    if (e != cudaSuccess) return e;
    kern<<<a.grid_kv, kKvThreads, L::kSmemBytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.lse, a.delta, a.dk,
                                                           a.dv, nullptr, a.geom, a.scale, a.scale_log2, a.sched_kv,
                                                           a.status, a.wait_limit_ns, a.stall_unit, a.bias);
  } else {
    // single pass: dK, dV and the dQ shares, after the row-term pass
    using L = KvLayout<D, true>;
    auto kern = dkdv_kernel<D, CAUSAL, BIAS, true>;
    static std::atomic<unsigned long long> ready{0};
    e = setup_kernel_once(kern, L::kSmemBytes, kKvLaunchRegs, ready);
    if (e != cudaSuccess) return e;
    kern<<<a.grid_kv, kKvThreads, L::kSmemBytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.lse, a.delta, a.dk,
                                                           a.dv, a.dq, a.geom, a.scale, a.scale_log2, a.sched_kv,
                                                           a.status, a.wait_limit_ns, a.stall_unit, a.bias);
  }
  return cudaGetLastError();
}

template <int D, bool CAUSAL>
cudaError_t launch_stage_c(const BwdArgs& a, int stage, cudaStream_t stream) {
  return a.bias.p ? launch_stage_t<D, CAUSAL, true>(a, stage, stream)
                  : launch_stage_t<D, CAUSAL, false>(a, stage, stream);
}

}  // namespace

cudaError_t launch_bwd_stage(const BwdArgs& a, int stage, cudaStream_t stream) {
  if (stage == 2) return launch_bwd_rowterm(a, stream);
  if (a.d == 64)
    return a.causal ? launch_stage_c<64, true>(a, stage, stream) : launch_stage_c<64, false>(a, stage, stream);
  return a.causal ? launch_stage_c<128, true>(a, stage, stream) : launch_stage_c<128, false>(a, stage, stream);
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  for (int stage = 0; stage < 2; ++stage) {
    const cudaError_t e = launch_bwd_stage(a, stage, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_bwd_single_pass(const BwdArgs& a, cudaStream_t stream) {
  for (int stage = 2; stage < 4; ++stage) {
    const cudaError_t e = launch_bwd_stage(a, stage, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace fa
