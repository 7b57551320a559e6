// FP8 forward kernel: the forward of fwd.cu with E4M3 operands.
//
// Same method (tiles of Q, K, V on chip, online softmax with a lazy
// reference maximum; "FlashAttention Interview Questions", sections "How does
// tiling reduce IO?" and "How can softmax be computed across tiles?") and the
// same roles, ring and scheduler as the bf16 forward, square sequences only
// (Nq = Nk = N), d = 128.  What changes with the 8-bit inputs
// ("FlashAttention 1, 2 & 3", section on FlashAttention-3: FP8 on the tensor
// cores):
//   * Q and K come as E4M3 [B*H][N][128]; V comes transposed, E4M3
//     [B*H][128][N], so that both products read K-major operands.  A tile of
//     128 rows is 16 KB (one 128-byte swizzle row per matrix row).
//   * S = Q K^T and O += P V are kind::f8f6f4 tcgen05 products with fp32
//     accumulation in tensor memory, K = 32 per instruction: four
//     instructions per 128 x 128 x 128 product where bf16 needs eight.
//   * The softmax rounds P to E4M3 (nearest even, saturating; P <= 2^8 under
//     the lazy reference) and writes it into a swizzled shared-memory tile, the
//     A operand of O += P V; l sums the unrounded fp32 P.  Tensor memory holds
//     S_A, S_B, O_A, O_B (512 columns).
// Every pipeline wait is bounded, as in the bf16 kernel.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "geom.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// 12 warps as in the bf16 forward: softmax warpgroups A and B, TMA (warp 8),
// MMA (warp 9), two idle warps; 168 registers at launch, 192 for the
// softmax warpgroups and 120 for the third (2*128*192 + 128*120 = 384*168).
constexpr int kF8Threads = 384;
constexpr int kF8LaunchRegs = 168;
constexpr int kF8SoftmaxRegs = 192;
constexpr int kF8OtherRegs = 120;
static_assert(2 * 128 * kF8SoftmaxRegs + 128 * kF8OtherRegs <= kF8Threads * kF8LaunchRegs,
              "register split exceeds the launch allocation");
constexpr float kF8Tau = 8.0f;  // lazy-rescale threshold, log2 units
constexpr float kF8Ln2 = 0.69314718055994530942f;

enum F8Site : int {
  SITE_F8_LOAD_Q = 41,
  SITE_F8_LOAD_KV = 42,
  SITE_F8_MMA_Q = 43,
  SITE_F8_MMA_KV = 44,
  SITE_F8_MMA_P = 45,
  SITE_F8_SOFTMAX_S = 46,
  SITE_F8_SOFTMAX_O = 47,
};

struct F8Layout {
  static constexpr int D = 128;
  static constexpr int kTileBytes = kTileRows * D;  // 128 rows of 128 one-byte elements
  static constexpr int kSlots = 8;                  // K / V^T ring slots
  static constexpr int kQOff = 0;                   // Q_A, Q_B
  static constexpr int kPOff = 2 * kTileBytes;      // P_A, P_B (written by the softmax warps)
  static constexpr int kRingOff = 4 * kTileBytes;
  static constexpr int kBarOff = kRingOff + kSlots * kTileBytes;
  static constexpr int Q_FULL = 0;
  static constexpr int Q_EMPTY = 1;
  static constexpr int KV_FULL = 2;
  static constexpr int KV_EMPTY = KV_FULL + kSlots;
  static constexpr int S_FULL = KV_EMPTY + kSlots;
  static constexpr int P_FULL = S_FULL + 2;
  static constexpr int O_FULL = P_FULL + 2;
  static constexpr int DRAIN = O_FULL + 2;
  static constexpr int kNumBars = DRAIN + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kColO = 256;
  static_assert(kSmemBytes <= 232448, "FP8 forward layout exceeds 227 KB of shared memory");
};

__device__ __forceinline__ bool f8_warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& w, int site, int unit) {
  const bool ok = wait_bounded(bar, parity, w, site, unit);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void f8_drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

__device__ __forceinline__ float f8_fmax3(float a, float b, float c) { return fmaxf(fmaxf(a, b), c); }

template <bool CAUSAL>
__global__ void __launch_bounds__(kF8Threads, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_vt, float* __restrict__ o, float* __restrict__ lse,
                   const int n, const float scale_log2, const SchedParams sp, int* status,
                   const unsigned long long limit_ns, const int stall_unit) {
  using L = F8Layout;
  constexpr int D = L::D;
  constexpr int S = L::kSlots;
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
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars + 8 * (L::S_FULL + t), 1);
      mbar_init(bars + 8 * (L::P_FULL + t), 4);  // one arrive per softmax warp
      mbar_init(bars + 8 * (L::O_FULL + t), 1);
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
    prefetch_tensormap(&tm_vt);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, status, limit_ns};
  const int nkt = (n + kTileRows - 1) / kTileRows;
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };

  if (warp < 8) {
    // ------------------------------------------------------------ softmax
    regs_increase<kF8SoftmaxRegs>();
    const int t = warp >> 2;
    const int r = ((warp & 3) << 5) + lane;  // row inside the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(t * 128);
    const uint32_t tO = tmem + lane_off + L::kColO + static_cast<uint32_t>(t * D);
    // this row of the P tile: 8-row groups of 1024 bytes, 128 bytes a row,
    // 16-byte chunks placed at (chunk ^ row % 8), the 128-byte swizzle that
    // the K-major operand descriptor expects
    const uint32_t prow = sbase + L::kPOff + t * L::kTileBytes + (r >> 3) * 1024 + (r & 7) * 128;
    const uint32_t pxor = static_cast<uint32_t>(r & 7);
    uint32_t sn = 0, on = 0;
    SchedIter it = sched_begin(sp);
    int head, pair;
    bool ok = true;
    while (ok && sched_next(it, sp, blockIdx.x, head, pair)) {
      const int qtile = 2 * pair + t;
      const int nt = CAUSAL ? min(qtile + 1, nkt) : nkt;
      const int row = qtile * kTileRows + r;
      const int unit = head * sp.units_per_head + pair;
      float m_ref = 0.f, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        ok = f8_warp_wait(BAR(L::S_FULL + t), sn & 1, wc, SITE_F8_SOFTMAX_S, unit);
        if (!ok) break;
        ++sn;
        tc_fence_after();
        float s[128];
        {
          uint32_t sr[128];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sr + 32 * c));
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        }
        // keys past N, or (causal) past the row's own position
        const bool diag = CAUSAL && (j == qtile);
        const bool tail = (j == nkt - 1) && ((n & (kTileRows - 1)) != 0);
        if (diag || tail) {
          const int lim = (CAUSAL ? min(row + 1, n) : n) - j * kTileRows;
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -CUDART_INF_F;
        }
        float t1[43];
#pragma unroll
        for (int c = 0; c < 42; ++c) t1[c] = f8_fmax3(s[3 * c], s[3 * c + 1], s[3 * c + 2]);
        t1[42] = fmaxf(s[126], s[127]);
        float t2[15];
#pragma unroll
        for (int c = 0; c < 14; ++c) t2[c] = f8_fmax3(t1[3 * c], t1[3 * c + 1], t1[3 * c + 2]);
        t2[14] = t1[42];
        float t3[5];
#pragma unroll
        for (int c = 0; c < 5; ++c) t3[c] = f8_fmax3(t2[3 * c], t2[3 * c + 1], t2[3 * c + 2]);
        const float mt = fmaxf(f8_fmax3(t3[0], t3[1], t3[2]), fmaxf(t3[3], t3[4])) * scale_log2;
        if (j == 0) {
          // the first key tile holds a key of every row (key 0)
          m_ref = (mt == -CUDART_INF_F) ? 0.f : mt;
        } else {
          const bool need = mt > m_ref + kF8Tau;
          if (__any_sync(0xffffffffu, need)) {
            // PV of the previous tile is complete (its commit preceded S(j)'s)
            const float m_new = fmaxf(m_ref, mt);
            const float alpha = ex2_approx(m_ref - m_new);
            m_ref = m_new;
            l *= alpha;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t v[32];
              tmem_ld32(tO + 32 * c, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
              tmem_st32(tO + 32 * c, v);
            }
            tmem_st_wait();
          }
        }
        // P = 2^(s*c - m_ref): fp32 into l, E4M3 into the shared P tile,
        // 32 keys (two 16-byte chunks) at a time
        const uint64_t c2 = f2_pack(scale_log2, scale_log2);
        const uint64_t n2 = f2_pack(-m_ref, -m_ref);
        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float x0, x1, x2, x3;
            f2_unpack(ffma2(f2_pack(s[32 * c + 4 * i], s[32 * c + 4 * i + 1]), c2, n2), x0, x1);
            f2_unpack(ffma2(f2_pack(s[32 * c + 4 * i + 2], s[32 * c + 4 * i + 3]), c2, n2), x2, x3);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            acc0 = fadd2(acc0, f2_pack(p0, p1));
            acc1 = fadd2(acc1, f2_pack(p2, p3));
            w8[i] = pack_e4m3x4(p0, p1, p2, p3);
          }
          st_shared_v4(prow + (((2 * c) ^ pxor) << 4), w8[0], w8[1], w8[2], w8[3]);
          st_shared_v4(prow + (((2 * c + 1) ^ pxor) << 4), w8[4], w8[5], w8[6], w8[7]);
        }
        float a0, a1, a2, a3;
        f2_unpack(acc0, a0, a1);
        f2_unpack(acc1, a2, a3);
        l += (a0 + a1) + (a2 + a3);
        fence_proxy_async_smem();  // P is read by the tensor core (async proxy)
        tc_fence_before();
        mbar_arrive_warp(BAR(L::P_FULL + t));
      }
      if (!ok) break;
      // epilogue: O = accumulator / l, LSE = ln(sum exp(scaled scores))
      ok = f8_warp_wait(BAR(L::O_FULL + t), on & 1, wc, SITE_F8_SOFTMAX_O, unit);
      if (!ok) break;
      ++on;
      tc_fence_after();
      const bool valid = row < n;
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      float* orow = o + (static_cast<size_t>(head) * n + row) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tO + 32 * c, v);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4 w4;
            w4.x = __uint_as_float(v[4 * i + 0]) * inv;
            w4.y = __uint_as_float(v[4 * i + 1]) * inv;
            w4.z = __uint_as_float(v[4 * i + 2]) * inv;
            w4.w = __uint_as_float(v[4 * i + 3]) * inv;
            *reinterpret_cast<float4*>(orow + 32 * c + 4 * i) = w4;
          }
        }
      }
      if (valid) lse[static_cast<size_t>(head) * n + row] = l > 0.f ? (m_ref + log2f(l)) * kF8Ln2 : -CUDART_INF_F;
    }
  } else {
   regs_decrease<kF8OtherRegs>();
   if (warp == 8) {
    // -------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_kv = l2_policy_evict_last();
      const uint64_t pol_q = l2_policy_evict_first();
      uint32_t qn = 0, kvpos = 0;
      SchedIter it = sched_begin(sp);
      int head, pair;
      bool ok = true;
      while (ok && sched_next(it, sp, blockIdx.x, head, pair)) {
        const int nmax = CAUSAL ? min(2 * pair + 2, nkt) : nkt;
        const int unit = head * sp.units_per_head + pair;
        ok = wait_bounded(BAR(L::Q_EMPTY), (qn & 1) ^ 1, wc, SITE_F8_LOAD_Q, unit);
        if (!ok) break;
        ++qn;
        mbar_arrive_expect_tx(BAR(L::Q_FULL), 2 * L::kTileBytes);
#pragma unroll
        for (int t = 0; t < 2; ++t)
          tma_load_3d_hint(sbase + L::kQOff + t * L::kTileBytes, &tm_q, BAR(L::Q_FULL), 0,
                           (2 * pair + t) * kTileRows, head, pol_q);
        for (int j = 0; j < nmax && ok; ++j) {
#pragma unroll 1
          for (int w = 0; w < 2; ++w) {
            const uint32_t slot = kvpos % S, use = kvpos / S;
            ok = wait_bounded(BAR(L::KV_EMPTY + slot), (use & 1) ^ 1, wc, SITE_F8_LOAD_KV, unit);
            if (!ok) break;
            if (blockIdx.x == 0 && static_cast<int>(qn) - 1 == stall_unit && j == 0 && w == 0) {
              // testing hook: leave this K tile unloaded so the waits on it
              // run out and the kernel reports a timeout instead of hanging
              ++kvpos;
              continue;
            }
            mbar_arrive_expect_tx(BAR(L::KV_FULL + slot), L::kTileBytes);
            // K tile j: rows are keys, d inner; V^T tile j: rows are the d
            // dimensions, keys inner (the key coordinate j*128 bytes)
            if (w == 0)
              tma_load_3d_hint(sbase + L::kRingOff + slot * L::kTileBytes, &tm_k, BAR(L::KV_FULL + slot), 0,
                               j * kTileRows, head, pol_kv);
            else
              tma_load_3d_hint(sbase + L::kRingOff + slot * L::kTileBytes, &tm_vt, BAR(L::KV_FULL + slot),
                               j * kTileRows, 0, head, pol_kv);
            ++kvpos;
          }
        }
      }
      if (!ok) {
        // let every copy already issued land before the CTA exits
        if (qn > 0) f8_drain_wait(BAR(L::Q_FULL), (qn - 1) & 1, limit_ns);
        for (uint32_t s = 0; s < static_cast<uint32_t>(S); ++s) {
          if (kvpos > s) {
            const uint32_t last = kvpos - 1 - ((kvpos - 1 - s) % S);
            f8_drain_wait(BAR(L::KV_FULL + s), (last / S) & 1, limit_ns);
          }
        }
      }
    }
   } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_mma = idesc_e4m3_f32(128, 128);  // both products: M = N = 128
      // K-major 128-byte-swizzled tiles; a K step of 32 one-byte elements
      // moves the start-address field by 32 bytes (2 units)
      const SDesc qdesc0 = sdesc_sw128(sbase + L::kQOff, 16, 1024);
      const SDesc pdesc0 = sdesc_sw128(sbase + L::kPOff, 16, 1024);
      const SDesc rdesc0 = sdesc_sw128(sbase + L::kRingOff, 16, 1024);
      constexpr uint32_t kTileUnits = L::kTileBytes >> 4;
      // S_t = Q_t K^T : M = 128 queries, N = 128 keys, K = d
      auto issue_s = [&](int t, uint32_t slot) {
        const SDesc qd = qdesc0 + static_cast<uint32_t>(t) * kTileUnits;
        const SDesc kd = rdesc0 + slot * kTileUnits;
#pragma unroll
        for (int ks = 0; ks < D / 32; ++ks)
          umma_ss_f8(tmem + static_cast<uint32_t>(t * 128), qd + 2 * ks, kd + 2 * ks, id_mma, ks > 0 ? 1u : 0u);
      };
      // O_t += P_t V : M = 128 queries, N = d, K = 128 keys; B is the V^T tile
      auto issue_pv = [&](int t, uint32_t slot, bool acc) {
        const SDesc pd = pdesc0 + static_cast<uint32_t>(t) * kTileUnits;
        const SDesc vd = rdesc0 + slot * kTileUnits;
#pragma unroll
        for (int ks = 0; ks < kTileRows / 32; ++ks)
          umma_ss_f8(tmem + L::kColO + static_cast<uint32_t>(t * D), pd + 2 * ks, vd + 2 * ks, id_mma,
                     (acc || ks > 0) ? 1u : 0u);
      };
      uint32_t qn = 0, kvbase = 0, pn0 = 0, pn1 = 0;
      SchedIter it = sched_begin(sp);
      int head, pair;
      bool ok = true;
      while (ok && sched_next(it, sp, blockIdx.x, head, pair)) {
        const int na = CAUSAL ? min(2 * pair + 1, nkt) : nkt;
        const int nb = CAUSAL ? min(2 * pair + 2, nkt) : nkt;
        const int unit = head * sp.units_per_head + pair;
        ok = wait_bounded(BAR(L::Q_FULL), qn & 1, wc, SITE_F8_MMA_Q, unit);
        if (!ok) break;
        ++qn;
        ok = wait_bounded(BAR(L::KV_FULL + kvbase % S), (kvbase / S) & 1, wc, SITE_F8_MMA_KV, unit);
        if (!ok) break;
        tc_fence_after();
        issue_s(0, kvbase % S);
        umma_commit(BAR(L::S_FULL + 0));
        issue_s(1, kvbase % S);
        umma_commit(BAR(L::S_FULL + 1));
        for (int j = 0; j < nb; ++j) {
          const uint32_t kpos = kvbase + 2 * j, vpos = kpos + 1, knext = kpos + 2;
          const bool has_a = j < na, next_a = j + 1 < na, next_b = j + 1 < nb;
          umma_commit(BAR(L::KV_EMPTY + kpos % S));  // K_j is free once S(j) of both tiles completes
          if (!next_b) umma_commit(BAR(L::Q_EMPTY));   // the unit's last S has been issued
          ok = wait_bounded(BAR(L::KV_FULL + vpos % S), (vpos / S) & 1, wc, SITE_F8_MMA_KV, unit);
          if (!ok) break;
          if (has_a) {
            ok = wait_bounded(BAR(L::P_FULL + 0), pn0 & 1, wc, SITE_F8_MMA_P, unit);
            if (!ok) break;
            ++pn0;
            tc_fence_after();
            issue_pv(0, vpos % S, j > 0);
            if (!next_a) umma_commit(BAR(L::O_FULL + 0));
            if (next_a) {
              ok = wait_bounded(BAR(L::KV_FULL + knext % S), (knext / S) & 1, wc, SITE_F8_MMA_KV, unit);
              if (!ok) break;
              tc_fence_after();
              issue_s(0, knext % S);
              umma_commit(BAR(L::S_FULL + 0));
            }
          }
          ok = wait_bounded(BAR(L::P_FULL + 1), pn1 & 1, wc, SITE_F8_MMA_P, unit);
          if (!ok) break;
          ++pn1;
          tc_fence_after();
          issue_pv(1, vpos % S, j > 0);
          if (!next_b) umma_commit(BAR(L::O_FULL + 1));
          umma_commit(BAR(L::KV_EMPTY + vpos % S));  // V_j is free once PV(j) of both tiles completes
          if (next_b) {
            if (!(has_a && next_a)) {  // otherwise tile A's S(j+1) already waited for K_{j+1}
              ok = wait_bounded(BAR(L::KV_FULL + knext % S), (knext / S) & 1, wc, SITE_F8_MMA_KV, unit);
              if (!ok) break;
              tc_fence_after();
            }
            issue_s(1, knext % S);
            umma_commit(BAR(L::S_FULL + 1));
          }
        }
        kvbase += 2 * nb;
      }
      // every MMA this thread issued completes before tensor memory is freed
      umma_commit(BAR(L::DRAIN));
      f8_drain_wait(BAR(L::DRAIN), 0, limit_ns);
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

template <bool CAUSAL>
cudaError_t launch_fp8_t(const FwdArgs& a, cudaStream_t stream) {
  using L = F8Layout;
  auto kern = fwd_fp8_kernel<CAUSAL>;
  static std::atomic<unsigned long long> ready{0};
  const cudaError_t e = setup_kernel_once(kern, L::kSmemBytes, kF8LaunchRegs, ready);
  if (e != cudaSuccess) return e;
  kern<<<a.sched.grid, kF8Threads, L::kSmemBytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, static_cast<float*>(a.o), a.lse,
                                                            a.geom.nq, a.scale_log2, a.sched, a.status,
                                                            a.wait_limit_ns, a.stall_unit);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp8(const FwdArgs& a, cudaStream_t stream) {
  return a.causal ? launch_fp8_t<true>(a, stream) : launch_fp8_t<false>(a, stream);
}

}  // namespace fa
