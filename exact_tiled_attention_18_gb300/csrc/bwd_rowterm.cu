// Row-term pass of the single-pass backward.
//
// The backward pass needs, for every query row, the row term
//   D_i = sum_j P_ij dP_ij,   P_ij = exp(s_ij - LSE_i),   dP_ij = dO_i . v_j
// before it can form dS_ij = P_ij (dP_ij - D_i) ("FlashAttention Interview
// Questions: IO Complexity, Tiling, and Numerical Stability", section "Why
// can recomputation help training?": the backward rebuilds P from the saved
// log-sum-exp).  D_i also equals rowsum(dO o O), but the forward's O carries
// the rounding of P to bf16 before its P V product, and on rows with large
// queries that rounding moves rowsum(dO o O) by about 1e-2, enough to push dK
// past the gradient tolerance.  This kernel therefore forms D exactly as
// defined, from the recomputed fp32 probabilities: per 128-row query tile it
// sweeps the key tiles with two tcgen05 products, S = Q K^T and dP = dO V^T,
// and each elementwise thread (one query row, 64 key columns) accumulates
// P dP in fp32.  Nothing returns to tensor memory, so S and dP are double
// buffered there and the tensor pipe runs one key tile ahead of the
// elementwise warps.  The kernel also zeroes dQ, which the dK/dV/dQ kernel
// that follows accumulates into.
//
// Warps: 0-7 elementwise (two warpgroups, key columns [64 w, 64 w + 64) of
// each tile), 8 TMA, 9 MMA, 10-11 idle.  Every wait is bounded.
#include <cuda_runtime.h>
#include <math_constants.h>

#include <type_traits>

#include "geom.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

enum RowSite : int {
  SITE_R_LOAD_Q = 51,
  SITE_R_LOAD_KV = 52,
  SITE_R_MMA_Q = 53,
  SITE_R_MMA_KV = 54,
  SITE_R_MMA_SFREE = 55,
  SITE_R_MMA_DFREE = 56,
  SITE_R_EW_S = 57,
  SITE_R_EW_DP = 58,
  SITE_R_EW_XCH = 59,
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

__device__ __forceinline__ uint64_t f2_from(uint32_t a, uint32_t b) {
  return f2_pack(__uint_as_float(a), __uint_as_float(b));
}

__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t u) {
  return f2_pack(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// Additive mask of one query for 64 consecutive keys k0.. as bf16 pairs (keys
// k0..k0+31 in b0, the next 32 in b1); 0 past key nk or without a row.  vec:
// the row starts on a 16-byte boundary, so the 16-byte loads are aligned.
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

template <int D>
struct RowLayout {
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kStages = (D == 128) ? 2 : 4;  // (K, V) ring
  static constexpr int kQOff = 0;
  static constexpr int kDoOff = kTileBytes;
  static constexpr int kKvOff = 2 * kTileBytes;  // stage s: K at +0, V at +kTileBytes
  static constexpr int kXchOff = kKvOff + kStages * 2 * kTileBytes;  // [2 units][2 warpgroups][128] fp32
  static constexpr int kBarOff = kXchOff + 2 * 2 * 128 * 4;
  static constexpr int Q_FULL = 0;
  static constexpr int Q_EMPTY = 1;
  static constexpr int KV_FULL = 2;
  static constexpr int KV_EMPTY = KV_FULL + kStages;
  static constexpr int S_FULL = KV_EMPTY + kStages;  // 2 buffers: S computed
  static constexpr int DP_FULL = S_FULL + 2;         // 2 buffers: dP computed
  static constexpr int S_FREE = DP_FULL + 2;         // 2 buffers: S read out (one arrive per elementwise warp)
  static constexpr int DP_FREE = S_FREE + 2;         // 2 buffers: dP read out
  static constexpr int XCH = DP_FREE + 2;
  static constexpr int DRAIN = XCH + 1;
  static constexpr int kNumBars = DRAIN + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  // tensor memory: buffer b holds S in [256 b, 256 b + 128) and dP in
  // [256 b + 128, 256 b + 256)
  static constexpr uint32_t kColS = 0, kColDP = 128, kBufCols = 256;
};

constexpr int kRowThreads = 384;

template <int D, bool CAUSAL, bool BIAS>
__global__ void __launch_bounds__(kRowThreads, 1)
    rowterm_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const float* __restrict__ lse, float* __restrict__ delta, float* __restrict__ dq,
                   const SeqGeom geom, const float scale_log2, const SchedParams sp, int* status,
                   const unsigned long long limit_ns, const int stall_unit, const BiasRef bias) {
  using L = RowLayout<D>;
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars + 8 * (L::S_FULL + b), 1);
      mbar_init(bars + 8 * (L::DP_FULL + b), 1);
      mbar_init(bars + 8 * (L::S_FREE + b), 8);
      mbar_init(bars + 8 * (L::DP_FREE + b), 8);
    }
    mbar_init(bars + 8 * L::XCH, 8);
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
    // ------------------------------------------- P dP row sums (thread = query row)
    const int w = warp >> 2;  // key columns [64 w, 64 w + 64)
    const int r = ((warp & 3) << 5) + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    float* xch = reinterpret_cast<float*>(smem + L::kXchOff);
    uint32_t tn = 0, un = 0;  // key tiles consumed, units finished
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
      // dQ starts at zero: the dK/dV/dQ kernel adds every key tile's share
      if (valid) {
        float* dst = dq + ridx * D;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int c = w * (D / 2); c < (w + 1) * (D / 2); c += 4) *reinterpret_cast<float4*>(dst + c) = z;
      }
      if (nk == 0) {
        // padding rows, or rows that see no key: row term 0
        if (valid && w == 0) delta[ridx] = 0.f;
        continue;
      }
      const float lv = row < hl.lq ? lse[ridx] : -CUDART_INF_F;
      const bool has = lv > -CUDART_INF_F;  // a valid row with at least one key
      // P = exp2(s * scale * log2 e - LSE * log2 e); +inf for rows without a key gives P = 0
      const uint64_t nl2x2 = f2_pack(has ? -lv * kLog2e : -CUDART_INF_F, has ? -lv * kLog2e : -CUDART_INF_F);
      const uint64_t c2 = f2_pack(scale_log2, scale_log2);
      uint64_t acc = f2_pack(0.f, 0.f);
      const uint16_t* brow = nullptr;
      bool bvec = false;
      if constexpr (BIAS) {
        const int bidx = head / geom.heads_per_batch;
        if (row < hl.lq) {
          brow = bias.p + bidx * bias.sb + (head - bidx * geom.heads_per_batch) * bias.sh + row * bias.sq;
          bvec = (reinterpret_cast<uintptr_t>(brow) & 15) == 0;
        }
      }
      for (int jt = 0; jt < nk; ++jt, ++tn) {
        uint32_t bb0[BIAS ? 16 : 1], bb1[BIAS ? 16 : 1];
        if constexpr (BIAS) {
          load_bias_row(brow, bvec, jt * kTileRows + 64 * w, geom.nk, bb0, bb1);
          const int knext = (jt + 1) * kTileRows + 64 * w;
          if (brow && jt + 1 < nk && knext + 64 <= geom.nk) prefetch_l2(brow + knext);
        }
        const uint32_t b = tn & 1, par = (tn >> 1) & 1;
        const uint32_t colS = tmem + lane_off + b * L::kBufCols + L::kColS + 64 * w;
        const uint32_t colD = tmem + lane_off + b * L::kBufCols + L::kColDP + 64 * w;
        ok = warp_wait(BAR(L::S_FULL + b), par, wc, SITE_R_EW_S, unit);
        if (!ok) break;
        tc_fence_after();
        uint32_t s0[32], s1[32];
        tmem_ld32(colS, s0);
        tmem_ld32(colS + 32, s1);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive_warp(BAR(L::S_FREE + b));
        const bool diag = CAUSAL && tile_crosses_diagonal(hl, i, jt);
        const bool tail = (jt == hl.nkt - 1) && ((hl.lk & (kTileRows - 1)) != 0);
        const bool need_mask = diag || tail;
        // eligible key columns of this tile for this row
        const int lim = need_mask ? ((CAUSAL ? min(row + hl.off + 1, hl.lk) : hl.lk) - jt * kTileRows) : kTileRows;
        // P for 32 key columns from col0, in place (fp32 bits)
        auto pchunk = [&](auto masked, uint32_t (&sr)[32], int col0, const uint32_t (&bh)[BIAS ? 16 : 1]) {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float p0, p1;
            uint64_t t = nl2x2;
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
          }
        };
        if (need_mask) {
          pchunk(std::true_type{}, s0, 64 * w, bb0);
          pchunk(std::true_type{}, s1, 64 * w + 32, bb1);
        } else {
          pchunk(std::false_type{}, s0, 64 * w, bb0);
          pchunk(std::false_type{}, s1, 64 * w + 32, bb1);
        }
        ok = warp_wait(BAR(L::DP_FULL + b), par, wc, SITE_R_EW_DP, unit);
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t d0[32], d1[32];
          tmem_ld32(colD, d0);
          tmem_ld32(colD + 32, d1);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive_warp(BAR(L::DP_FREE + b));
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            acc = ffma2(f2_from(s0[c], s0[c + 1]), f2_from(d0[c], d0[c + 1]), acc);
            acc = ffma2(f2_from(s1[c], s1[c + 1]), f2_from(d1[c], d1[c + 1]), acc);
          }
        }
      }
      if (!ok) break;
      // the two warpgroups' halves of D_i (slots alternate by unit)
      float a0, a1;
      f2_unpack(acc, a0, a1);
      float* slot = xch + (un & 1) * 256;
      slot[w * 128 + r] = a0 + a1;
      mbar_arrive_warp(BAR(L::XCH));
      ok = warp_wait(BAR(L::XCH), un & 1, wc, SITE_R_EW_XCH, unit);
      if (!ok) break;
      ++un;
      if (w == 0 && valid) delta[ridx] = has ? slot[r] + slot[128 + r] : 0.f;
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
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
        ok = wait_bounded(BAR(L::Q_EMPTY), (qn & 1) ^ 1, wc, SITE_R_LOAD_Q, unit);
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
          ok = wait_bounded(BAR(L::KV_EMPTY + s), (use & 1) ^ 1, wc, SITE_R_LOAD_KV, unit);
          if (!ok) break;
          if (blockIdx.x == 0 && static_cast<int>(qn) - 1 == stall_unit && jt == 0) {
            // testing hook: leave this (K, V) stage unloaded so that the
            // waits on it run out and the kernel reports a timeout
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
  } else if (warp == 9) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kTileUnits = L::kTileBytes >> 4;
      const SDesc qdesc = sdesc_sw128(sbase + L::kQOff, 16, 1024);
      const SDesc dodesc = sdesc_sw128(sbase + L::kDoOff, 16, 1024);
      const SDesc kv0 = sdesc_sw128(sbase + L::kKvOff, 16, 1024);
      uint32_t qn = 0, kvpos = 0, tn = 0;
      SchedIter it = sched_begin(sp);
      int head, i;
      bool ok = true;
      while (ok && sched_next(it, sp, blockIdx.x, head, i)) {
        const int nk = query_tile_keys(head_len(geom, head), i, CAUSAL);
        if (nk == 0) continue;
        const int unit = head * sp.units_per_head + i;
        ok = wait_bounded(BAR(L::Q_FULL), qn & 1, wc, SITE_R_MMA_Q, unit);
        if (!ok) break;
        ++qn;
        // per key tile: S = Q K^T and dP = dO V^T (M = 128 queries, N = 128
        // keys, K = d) into tensor-memory buffer tn & 1, once the elementwise
        // warps have read that buffer's previous contents out
        for (int jt = 0; jt < nk; ++jt, ++tn, ++kvpos) {
          const uint32_t s = kvpos % S;
          const uint32_t b = tn & 1, use = tn >> 1;
          const SDesc kd = kv0 + static_cast<uint32_t>(s) * (2 * kTileUnits);
          const SDesc vd = kd + kTileUnits;
          ok = wait_bounded(BAR(L::KV_FULL + s), (kvpos / S) & 1, wc, SITE_R_MMA_KV, unit);
          if (!ok) break;
          ok = wait_bounded(BAR(L::S_FREE + b), (use & 1) ^ 1, wc, SITE_R_MMA_SFREE, unit);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tS = tmem + b * L::kBufCols + L::kColS;
          const uint32_t tD = tmem + b * L::kBufCols + L::kColDP;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
            umma_ss(tS, qdesc + off, kd + off, id_s, ks > 0 ? 1u : 0u);
          }
          umma_commit(BAR(L::S_FULL + b));
          ok = wait_bounded(BAR(L::DP_FREE + b), (use & 1) ^ 1, wc, SITE_R_MMA_DFREE, unit);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
            umma_ss(tD, dodesc + off, vd + off, id_s, ks > 0 ? 1u : 0u);
          }
          umma_commit(BAR(L::DP_FULL + b));
          umma_commit(BAR(L::KV_EMPTY + s));
        }
        if (!ok) break;
        umma_commit(BAR(L::Q_EMPTY));
      }
      umma_commit(BAR(L::DRAIN));
      drain_wait(BAR(L::DRAIN), 0, limit_ns);
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
cudaError_t launch_rowterm_t(const BwdArgs& a, cudaStream_t stream) {
  using L = RowLayout<D>;
  auto kern = rowterm_kernel<D, CAUSAL, BIAS>;
  static std::atomic<unsigned long long> ready{0};
  cudaError_t e = setup_kernel_once(kern, L::kSmemBytes, 0, ready);
  if (e != cudaSuccess) return e;
  kern<<<a.grid_q, kRowThreads, L::kSmemBytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.lse, a.delta, a.dq,
                                                         a.geom, a.scale_log2, a.sched_q, a.status, a.wait_limit_ns,
                                                         a.stall_unit, a.bias);
  return cudaGetLastError();
}

template <int D, bool CAUSAL>
cudaError_t launch_rowterm_c(const BwdArgs& a, cudaStream_t stream) {
  return a.bias.p ? launch_rowterm_t<D, CAUSAL, true>(a, stream) : launch_rowterm_t<D, CAUSAL, false>(a, stream);
}

}  // namespace

cudaError_t launch_bwd_rowterm(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 64)
    return a.causal ? launch_rowterm_c<64, true>(a, stream) : launch_rowterm_c<64, false>(a, stream);
  return a.causal ? launch_rowterm_c<128, true>(a, stream) : launch_rowterm_c<128, false>(a, stream);
}

}  // namespace fa
