// Forward kernel: exact attention, tile by tile, with an online softmax.
//
// Method (FlashAttention pages): Q, K and V are split into tiles that fit
// on chip; each query tile sweeps the key/value tiles, keeping per row a
// running maximum m, a running sum l of shifted exponentials and an
// unnormalised accumulator, so the N x N score matrix never reaches HBM
// ("FlashAttention Interview Questions: IO Complexity, Tiling, and Numerical
// Stability", sections "How does tiling reduce IO?" and "How can softmax be
// computed across tiles?"; "FlashAttention 1, 2 & 3", section 2 "Tiling &
// Online Softmax" and "Kernel Fusion").  The update
//   scale = exp(m - m_new); l = scale*l + sum exp(s - m_new);
//   a = scale*a + sum exp(s - m_new) v;  output = a / l
// is carried out in base 2 with a lazy reference: the reference maximum is
// only moved (and l and the accumulator rescaled together) when a row's
// maximum grows by more than 2^8, which keeps every exponent <= 8 and is
// exact because numerator and denominator share the same reference.
//
// GB300 mapping.  One persistent CTA per SM.  A CTA takes two 128-row query
// tiles (A and B) of one head at a time and streams the head's K/V tiles
// through a ring of shared-memory slots filled by TMA.  Roles:
//   warps 0-3  softmax for tile A   (thread = one query row = one TMEM lane)
//   warps 4-7  softmax for tile B
//   warp  8    TMA producer (one thread)
//   warp  9    tcgen05 MMA issuer (one thread); owns the TMEM allocation
//   warps 10-11 idle (complete the third warpgroup for the register split)
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128) S_A, [128,256) S_B, [256,256+d) O_A, [256+d,256+2d) O_B.
//   P (bf16, two per column) overwrites the first 64 columns of its S region
//   and is the A operand of O += P V, read straight from TMEM.
// While softmax A works on S_A(j), the tensor core runs PV_B(j-1) and
// S_B(j); the two tiles ping-pong so MMA and exponentials overlap.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "geom.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// 12 warps: two softmax warpgroups, then TMA (warp 8), MMA (warp 9) and two
// idle warps that only complete the third warpgroup.  Launched at 168
// registers a thread (384 x 168 = 64512); the softmax warpgroups then take 192
// (no spills) and the third warpgroup keeps 120, enough for the MMA thread:
// 2*128*192 + 128*120 = 64512.
constexpr int kFwdThreads = 384;
constexpr int kFwdLaunchRegs = 168;
constexpr int kFwdSoftmaxRegs = 192;
constexpr int kFwdOtherRegs = 120;
static_assert(2 * 128 * kFwdSoftmaxRegs + 128 * kFwdOtherRegs <= kFwdThreads * kFwdLaunchRegs,
              "register split exceeds the launch allocation");
constexpr float kTau = 8.0f;  // lazy-rescale threshold, log2 units
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.4426950408889634f;

enum FwdSite : int {
  SITE_LOAD_Q = 1,
  SITE_LOAD_KV = 2,
  SITE_MMA_Q = 3,
  SITE_MMA_KV = 4,
  SITE_MMA_P = 5,
  SITE_SOFTMAX_S = 6,
  SITE_SOFTMAX_O = 7,
};

template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = kTileRows * D * 2;  // one bf16 tile of Q, K or V
  static constexpr int kSlots = (D == 128) ? 4 : 8;     // K/V ring slots
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = 2 * kTileBytes;
  static constexpr int kBarOff = kRingOff + kSlots * kTileBytes;
  // barrier indices
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
};

// Valid lengths and key-tile counts of one work unit (a head and its query
// tiles 2*pair and 2*pair+1); a count of 0 means the tile has nothing to
// compute (all padding, or no eligible key).  VARLEN = false is the square
// call (Nq = Nk, no per-sequence lengths): offset 0, no padding rows, and tile
// 2*pair never has more key tiles than 2*pair+1 nor none at all, facts the
// compiler folds into the loops below.
//
// SPLIT (split keys): a scheduler unit is (pair, split); the unit covers key
// tiles [k0, k0 + chunk) of its pair only, na and nb count the tiles of that
// range each query tile needs (either may be 0), and the results are partial
// (combined afterwards by log-sum-exp).
struct UnitGeom {
  int lq, lk, off, nkt, na, nb;
  int pair, split, k0;  // SPLIT only: query-tile pair, key split and its first key tile
};

template <bool VARLEN, bool SPLIT>
__device__ __forceinline__ UnitGeom unit_geom(const SeqGeom& g, int head, int unit_idx, bool causal, int splits,
                                              int chunk) {
  UnitGeom u;
  int pair = unit_idx;
  if constexpr (SPLIT) {
    pair = unit_idx / splits;
    u.pair = pair;
    u.split = unit_idx - pair * splits;
  }
  if constexpr (!VARLEN) {
    u.lq = u.lk = g.nq;
    u.off = 0;
    u.nkt = (g.nq + kTileRows - 1) / kTileRows;
    u.na = causal ? min(2 * pair + 1, u.nkt) : u.nkt;
    u.nb = causal ? min(2 * pair + 2, u.nkt) : u.nkt;
  } else {
    const HeadLen h = head_len(g, head);
    u.lq = h.lq;
    u.lk = h.lk;
    u.off = h.off;
    u.nkt = h.nkt;
    u.na = query_tile_keys(h, 2 * pair, causal);
    u.nb = query_tile_keys(h, 2 * pair + 1, causal);
  }
  if constexpr (SPLIT) {
    u.k0 = u.split * chunk;
    u.na = max(0, min(u.na - u.k0, chunk));
    u.nb = max(0, min(u.nb - u.k0, chunk));
  }
  return u;
}

// Wait with every lane of the warp and agree on the outcome, so that the
// warp-collective tcgen05 instructions after it are reached by all lanes or
// by none.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& w, int site, int unit) {
  const bool ok = wait_bounded(bar, parity, w, site, unit);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag: used only to let copies and MMAs
// already in flight land before the CTA releases its resources.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

template <int D, bool CAUSAL, bool VARLEN, bool BIAS, bool SPLIT>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, void* __restrict__ o, float* __restrict__ lse,
               const int o_bf16, const SeqGeom geom, const float scale_log2, const SchedParams sp,
               int* status, const unsigned long long limit_ns, const int stall_unit,
               const uint16_t* __restrict__ bias, const long long bias_sb, const long long bias_sh,
               const long long bias_sq, float* __restrict__ part, const int splits, const int chunk) {
  using L = FwdLayout<D>;
  // a unit may have no key tile for one of its query tiles, or none at all
  constexpr bool GEN = VARLEN || SPLIT;
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
    prefetch_tensormap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, status, limit_ns};
  const int nq = geom.nq;
  // bf16 output is served by the general (VARLEN) instantiation only, so the
  // square fp32 kernel carries no output-type branch
  const bool obf16 = VARLEN && o_bf16;
  auto BAR = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };

  if (warp < 8) {
    // ------------------------------------------------------------ softmax
    regs_increase<kFwdSoftmaxRegs>();
    const int t = warp >> 2;
    const int r = ((warp & 3) << 5) + lane;  // row inside the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(t * 128);
    const uint32_t tO = tmem + lane_off + L::kColO + static_cast<uint32_t>(t * D);
    uint32_t sn = 0, on = 0;
    SchedIter it = sched_begin(sp);
    int head, pair;
    bool ok = true;
    while (ok && sched_next(it, sp, blockIdx.x, head, pair)) {
      const UnitGeom u = unit_geom<VARLEN, SPLIT>(geom, head, pair, CAUSAL, splits, chunk);
      const int nt = t ? u.nb : u.na;
      const int qtile = 2 * (SPLIT ? u.pair : pair) + t;
      const int row = qtile * kTileRows + r;
      const int unit = head * sp.units_per_head + pair;
      // l: running sum of the weights as computed (fp32), for the LSE.  O is
      // divided by l + dl, where dl sums, over the key tiles, how much the
      // bf16 rounding (applied to every weight before the P V product)
      // changed that tile's largest weight.  The reference maximum lags the
      // row maximum by up to 2^kTau, so a dominant weight is rarely exactly 1;
      // without dl its rounding would scale a row dominated by one key by up
      // to 2^-9 (O error near 1e-2 for |v| ~ 5); with it that row returns
      // the key's value row, and the other weights' rounding stays relative.
      float m_ref = 0.f, l = 0.f, dl = 0.f;
      // additive mask: this row's bias (bf16, keys contiguous), none for
      // padding rows (fully masked anyway)
      const uint16_t* brow = nullptr;
      bool bvec = false;  // row start 16-byte aligned: whole tiles in 16-byte loads
      if constexpr (BIAS) {
        const int bidx = head / geom.heads_per_batch;
        if (row < u.lq) {
          brow = bias + bidx * bias_sb + (head - bidx * geom.heads_per_batch) * bias_sh +
                 static_cast<long long>(row) * bias_sq;
          bvec = (reinterpret_cast<uintptr_t>(brow) & 15) == 0;
        }
      }
      if (SPLIT && nt == 0) {
        // no key tile of this split for this query tile: an empty partial
        if (row < nq) {
          const size_t pr = (static_cast<size_t>(head) * splits + u.split) * nq + row;
          float4* prow = reinterpret_cast<float4*>(part + pr * D);
#pragma unroll 1
          for (int c = 0; c < D / 4; ++c) prow[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          part[static_cast<size_t>(sp.heads) * splits * nq * D + pr] = -CUDART_INF_F;
        }
        continue;
      }
      if (VARLEN && nt == 0) {
        // no key for any row of this tile (or all padding): O = 0, LSE = -inf
        if (row < nq) {
          // D fp32 or D bf16 zeros: 4 D or 2 D bytes, in 16-byte stores
          uint4* orow = reinterpret_cast<uint4*>(static_cast<uint8_t*>(o) +
                                                 (static_cast<size_t>(head) * nq + row) * D * (obf16 ? 2 : 4));
#pragma unroll 1
          for (int c = 0; c < (obf16 ? D / 8 : D / 4); ++c) orow[c] = make_uint4(0u, 0u, 0u, 0u);
          lse[static_cast<size_t>(head) * nq + row] = -CUDART_INF_F;
        }
        continue;
      }
      for (int j = 0; j < nt; ++j) {
        const int jk = SPLIT ? u.k0 + j : j;  // key tile index (j counts the unit's tiles)
        // bias of this row's 128 keys of tile jk, fetched while S(j) is computed
        uint4 bq[BIAS ? 16 : 1];
        if constexpr (BIAS) {
          const int col0 = jk * kTileRows;
          if (bvec && col0 + kTileRows <= geom.nk) {
#pragma unroll
            for (int i = 0; i < 16; ++i) bq[i] = __ldg(reinterpret_cast<const uint4*>(brow + col0) + i);
            // the row's next 256 bytes towards L2, a tile ahead of their use
            if (j + 1 < nt && col0 + 2 * kTileRows <= geom.nk) {
              prefetch_l2(brow + col0 + kTileRows);
              prefetch_l2(brow + col0 + kTileRows + 64);
            }
          } else {
            // a row that is not 16-byte aligned, the tile past the end of
            // the bias rows, or a padding row: element loads; keys from Nk on
            // are masked, their bias is never used
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int c0 = col0 + 8 * i + 2 * e;
                const uint32_t lo = (brow && c0 < geom.nk) ? brow[c0] : 0u;
                const uint32_t hi = (brow && c0 + 1 < geom.nk) ? brow[c0 + 1] : 0u;
                w[e] = lo | (hi << 16);
              }
              bq[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
        ok = warp_wait(BAR(L::S_FULL + t), sn & 1, wc, SITE_SOFTMAX_S, unit);
        if (!ok) break;
        ++sn;
        tc_fence_after();
        float s[128];
        if constexpr (BIAS) {
          // t = s * scale * log2(e) + bias * log2(e): the max and the
          // exponentials below work on t directly (log2 units); S is read a
          // chunk at a time so that the bias registers free up as it goes
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t sr[32];
            tmem_ld32(tS + 32 * c, sr);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 b4 = bq[4 * c + i];
              const uint32_t bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int col = 32 * c + 8 * i + 2 * e;
                s[col] = fmaf(__uint_as_float(sr[8 * i + 2 * e]), scale_log2,
                              __uint_as_float(bw[e] << 16) * kLog2e);
                s[col + 1] = fmaf(__uint_as_float(sr[8 * i + 2 * e + 1]), scale_log2,
                                  __uint_as_float(bw[e] & 0xFFFF0000u) * kLog2e);
              }
            }
          }
        } else {
          uint32_t sr[128];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sr + 32 * c));
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        }
        // keys past the valid length, or (causal) past the row's last key; a
        // padding row masks every key, so that it never takes part in the
        // warp's rescale vote and its values cannot change valid rows' rounding
        const bool diag = CAUSAL && (jk * kTileRows + kTileRows - 1 > qtile * kTileRows + u.off);
        const bool tail = (jk == u.nkt - 1) && ((u.lk & (kTileRows - 1)) != 0);
        const bool padq = VARLEN && qtile * kTileRows + kTileRows > u.lq;
        if (diag || tail || padq) {
          const int lim = row < u.lq ? (CAUSAL ? min(row + u.off + 1, u.lk) : u.lk) - jk * kTileRows : 0;
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -CUDART_INF_F;
        }
        // row maximum as a log-depth tree of 3-input max
        float t1[43];
#pragma unroll
        for (int c = 0; c < 42; ++c) t1[c] = fmax3(s[3 * c], s[3 * c + 1], s[3 * c + 2]);
        t1[42] = fmaxf(s[126], s[127]);
        float t2[15];
#pragma unroll
        for (int c = 0; c < 14; ++c) t2[c] = fmax3(t1[3 * c], t1[3 * c + 1], t1[3 * c + 2]);
        t2[14] = t1[42];
        float t3[5];
#pragma unroll
        for (int c = 0; c < 5; ++c) t3[c] = fmax3(t2[3 * c], t2[3 * c + 1], t2[3 * c + 2]);
        const float mt = fmaxf(fmax3(t3[0], t3[1], t3[2]), fmaxf(t3[3], t3[4])) * (BIAS ? 1.f : scale_log2);
        if (j == 0) {
          // without a bias the first key tile holds a key of every row that
          // has one; with a bias it may hide them all, so the reference stays
          // -inf until a finite maximum appears
          m_ref = (mt == -CUDART_INF_F && !BIAS) ? 0.f : mt;
        } else {
          const bool need = mt > m_ref + kTau;
          if (__any_sync(0xffffffffu, need)) {
            // move the reference and rescale l and the accumulator together;
            // PV of the previous tile is complete (its commit preceded S(j)'s)
            const float m_new = fmaxf(m_ref, mt);
            const float alpha = (BIAS && m_new == -CUDART_INF_F) ? 1.f : ex2_approx(m_ref - m_new);
            m_ref = m_new;
            l *= alpha;
            dl *= alpha;
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
        // P = 2^(s*c - m_ref) in bf16 over the first 64 S columns; two lanes
        // of the scale-subtract and of the running sum per instruction
        const float cexp = BIAS ? 1.f : scale_log2;
        const float m_use = (BIAS && m_ref == -CUDART_INF_F) ? 0.f : m_ref;  // every t is -inf then
        const uint64_t c2 = f2_pack(cexp, cexp);
        const uint64_t n2 = f2_pack(-m_use, -m_use);
        {
          // this tile's largest weight (as computed below up to the rounding
          // of the scaled maximum, an ulp of it) and its change by rounding
          const float pmax = ex2_approx(mt - m_use);
          dl += __uint_as_float(pack_bf16x2(pmax, 0.f) << 16) - pmax;
        }
        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            float x0, x1, x2, x3;
            f2_unpack(ffma2(f2_pack(s[32 * c + 2 * i], s[32 * c + 2 * i + 1]), c2, n2), x0, x1);
            f2_unpack(ffma2(f2_pack(s[32 * c + 2 * i + 2], s[32 * c + 2 * i + 3]), c2, n2), x2, x3);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            acc0 = fadd2(acc0, f2_pack(p0, p1));
            acc1 = fadd2(acc1, f2_pack(p2, p3));
            pk[i] = pack_bf16x2(p0, p1);
            pk[i + 1] = pack_bf16x2(p2, p3);
          }
          tmem_st16(tS + 16 * c, pk);
        }
        float a0, a1, a2, a3;
        f2_unpack(acc0, a0, a1);
        f2_unpack(acc1, a2, a3);
        l += (a0 + a1) + (a2 + a3);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(BAR(L::P_FULL + t));
      }
      if (!ok) break;
      // epilogue: O = accumulator / l, LSE = ln(sum exp(scaled scores))
      ok = warp_wait(BAR(L::O_FULL + t), on & 1, wc, SITE_SOFTMAX_O, unit);
      if (!ok) break;
      ++on;
      tc_fence_after();
      // rows past the valid length are padding and rows without an eligible
      // key have l = 0: both get O = 0, LSE = -inf (selected, so that what a
      // padding row accumulated never reaches the output)
      const bool live = l > 0.f && (!VARLEN || row < u.lq);
      const float inv = live ? 1.0f / (l + dl) : 0.f;
      const bool valid = row < nq;
      if constexpr (SPLIT) {
        // this split's normalised output and log2-sum-exp, for the combine
        const size_t pr = (static_cast<size_t>(head) * splits + u.split) * nq + row;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tO + 32 * c, v);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float4 w;
              w.x = __uint_as_float(v[4 * i + 0]) * inv;
              w.y = __uint_as_float(v[4 * i + 1]) * inv;
              w.z = __uint_as_float(v[4 * i + 2]) * inv;
              w.w = __uint_as_float(v[4 * i + 3]) * inv;
              *reinterpret_cast<float4*>(part + pr * D + 32 * c + 4 * i) = w;
            }
          }
        }
        if (valid)
          part[static_cast<size_t>(sp.heads) * splits * nq * D + pr] = live ? m_ref + log2f(l) : -CUDART_INF_F;
        continue;
      }
      float* orow = static_cast<float*>(o) + (static_cast<size_t>(head) * nq + row) * D;
      uint16_t* orow_h = static_cast<uint16_t*>(o) + (static_cast<size_t>(head) * nq + row) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tO + 32 * c, v);
        tmem_ld_wait();
        if (VARLEN && !live) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (valid && obf16) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 h;
            h.x = pack_bf16x2(__uint_as_float(v[8 * i + 0]) * inv, __uint_as_float(v[8 * i + 1]) * inv);
            h.y = pack_bf16x2(__uint_as_float(v[8 * i + 2]) * inv, __uint_as_float(v[8 * i + 3]) * inv);
            h.z = pack_bf16x2(__uint_as_float(v[8 * i + 4]) * inv, __uint_as_float(v[8 * i + 5]) * inv);
            h.w = pack_bf16x2(__uint_as_float(v[8 * i + 6]) * inv, __uint_as_float(v[8 * i + 7]) * inv);
            *reinterpret_cast<uint4*>(orow_h + 32 * c + 8 * i) = h;
          }
        } else if (valid) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4 w;
            w.x = __uint_as_float(v[4 * i + 0]) * inv;
            w.y = __uint_as_float(v[4 * i + 1]) * inv;
            w.z = __uint_as_float(v[4 * i + 2]) * inv;
            w.w = __uint_as_float(v[4 * i + 3]) * inv;
            *reinterpret_cast<float4*>(orow + 32 * c + 4 * i) = w;
          }
        }
      }
      if (valid)
        lse[static_cast<size_t>(head) * nq + row] =
            live ? (m_ref + log2f(l)) * kLn2 : -CUDART_INF_F;
    }
  } else {
   regs_decrease<kFwdOtherRegs>();
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
        const UnitGeom u = unit_geom<VARLEN, SPLIT>(geom, head, pair, CAUSAL, splits, chunk);
        const int nmax = GEN ? max(u.na, u.nb) : u.nb;
        if (GEN && nmax == 0) continue;  // nothing to compute for this unit
        const int unit = head * sp.units_per_head + pair;
        ok = wait_bounded(BAR(L::Q_EMPTY), (qn & 1) ^ 1, wc, SITE_LOAD_Q, unit);
        if (!ok) break;
        ++qn;
        mbar_arrive_expect_tx(BAR(L::Q_FULL), 2 * L::kTileBytes);
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int kb = 0; kb < D / 64; ++kb)
            tma_load_3d_hint(sbase + L::kQOff + t * L::kTileBytes + kb * 16384, &tm_q, BAR(L::Q_FULL), kb * 64,
                             (2 * (SPLIT ? u.pair : pair) + t) * kTileRows, head, pol_q);
        for (int j = 0; j < nmax && ok; ++j) {
#pragma unroll 1
          for (int w = 0; w < 2; ++w) {
            const uint32_t slot = kvpos % S, use = kvpos / S;
            ok = wait_bounded(BAR(L::KV_EMPTY + slot), (use & 1) ^ 1, wc, SITE_LOAD_KV, unit);
            if (!ok) break;
            if (blockIdx.x == 0 && static_cast<int>(qn) - 1 == stall_unit && j == 0 && w == 0) {
              // testing hook: leave this K tile unloaded so the waits on it
              // run out and the kernel reports a timeout instead of hanging
              ++kvpos;
              continue;
            }
            mbar_arrive_expect_tx(BAR(L::KV_FULL + slot), L::kTileBytes);
            const CUtensorMap* tm = (w == 0) ? &tm_k : &tm_v;
#pragma unroll
            for (int kb = 0; kb < D / 64; ++kb)
              tma_load_3d_hint(sbase + L::kRingOff + slot * L::kTileBytes + kb * 16384, tm,
                               BAR(L::KV_FULL + slot), kb * 64, ((SPLIT ? u.k0 : 0) + j) * kTileRows, head, pol_kv);
            ++kvpos;
          }
        }
      }
      if (!ok) {
        // let every copy already issued land before the CTA exits
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
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_pv = idesc_bf16_f32(128, D, false, true);
      auto slot_addr = [&](uint32_t pos) -> uint32_t { return pos % S; };  // ring slot index
      // Descriptors built once: Q tiles for the whole kernel, K (K-major) and
      // V (MN-major) per ring slot.  The K step only moves the start-address
      // field (bits 0-13, 16-byte units), a plain add on the low word.
      const SDesc qdesc0 = sdesc_sw128(sbase + L::kQOff, 16, 1024);
      const SDesc kdesc0 = sdesc_sw128(sbase + L::kRingOff, 16, 1024);
      const SDesc vdesc0 = sdesc_sw128(sbase + L::kRingOff, kTileRows * 128, 1024);
      constexpr uint32_t kTileUnits = L::kTileBytes >> 4;  // one tile in the address field's 16-byte units
      // S_t = Q_t K^T : M=128 query rows, N=128 keys, K=d (both K-major)
      auto issue_s = [&](int t, uint32_t slot) {
        const SDesc qd = qdesc0 + static_cast<uint32_t>(t) * kTileUnits;
        const SDesc kd = kdesc0 + slot * kTileUnits;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
          umma_ss(tmem + static_cast<uint32_t>(t * 128), qd + off, kd + off, id_s, ks > 0 ? 1u : 0u);
        }
      };
      // O_t += P_t V : M=128, N=d, K=128 keys; P from TMEM, V MN-major
      auto issue_pv = [&](int t, uint32_t slot, bool acc) {
        const SDesc vd = vdesc0 + slot * kTileUnits;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          umma_ts(tmem + L::kColO + static_cast<uint32_t>(t * D), tmem + static_cast<uint32_t>(t * 128 + ks * 8),
                  vd + static_cast<uint32_t>((ks * 2048) >> 4), id_pv, (acc || ks > 0) ? 1u : 0u);
        }
      };
      uint32_t qn = 0, kvbase = 0, pn0 = 0, pn1 = 0;
      SchedIter it = sched_begin(sp);
      int head, pair;
      bool ok = true;
      while (ok && sched_next(it, sp, blockIdx.x, head, pair)) {
        const UnitGeom u = unit_geom<VARLEN, SPLIT>(geom, head, pair, CAUSAL, splits, chunk);
        const int na = u.na, nb = u.nb, nmax = GEN ? max(na, nb) : nb;
        if (GEN && nmax == 0) continue;  // nothing to compute for this unit
        const int unit = head * sp.units_per_head + pair;
        ok = wait_bounded(BAR(L::Q_FULL), qn & 1, wc, SITE_MMA_Q, unit);
        if (!ok) break;
        ++qn;
        ok = wait_bounded(BAR(L::KV_FULL + kvbase % S), (kvbase / S) & 1, wc, SITE_MMA_KV, unit);
        if (!ok) break;
        tc_fence_after();
        if (!GEN || na > 0) {
          issue_s(0, slot_addr(kvbase));
          umma_commit(BAR(L::S_FULL + 0));
        }
        if (!GEN || nb > 0) {
          issue_s(1, slot_addr(kvbase));
          umma_commit(BAR(L::S_FULL + 1));
        }
        for (int j = 0; j < nmax; ++j) {
          const uint32_t kpos = kvbase + 2 * j, vpos = kpos + 1, knext = kpos + 2;
          const bool has_a = j < na, next_a = j + 1 < na, has_b = !GEN || j < nb, next_b = j + 1 < nb;
          umma_commit(BAR(L::KV_EMPTY + kpos % S));  // K_j is free once S(j) of both tiles completes
          if (!next_b && (!GEN || !next_a)) umma_commit(BAR(L::Q_EMPTY));  // the unit's last S has been issued
          ok = wait_bounded(BAR(L::KV_FULL + vpos % S), (vpos / S) & 1, wc, SITE_MMA_KV, unit);
          if (!ok) break;
          if (has_a) {
            ok = wait_bounded(BAR(L::P_FULL + 0), pn0 & 1, wc, SITE_MMA_P, unit);
            if (!ok) break;
            ++pn0;
            tc_fence_after();
            issue_pv(0, slot_addr(vpos), j > 0);
            if (!next_a) umma_commit(BAR(L::O_FULL + 0));
            if (next_a) {
              ok = wait_bounded(BAR(L::KV_FULL + knext % S), (knext / S) & 1, wc, SITE_MMA_KV, unit);
              if (!ok) break;
              tc_fence_after();
              issue_s(0, slot_addr(knext));
              umma_commit(BAR(L::S_FULL + 0));
            }
          }
          if (has_b) {
            ok = wait_bounded(BAR(L::P_FULL + 1), pn1 & 1, wc, SITE_MMA_P, unit);
            if (!ok) break;
            ++pn1;
            tc_fence_after();
            issue_pv(1, slot_addr(vpos), j > 0);
            if (!next_b) umma_commit(BAR(L::O_FULL + 1));
          }
          umma_commit(BAR(L::KV_EMPTY + vpos % S));  // V_j is free once PV(j) of both tiles completes
          if (next_b) {
            if (!(has_a && next_a)) {  // otherwise tile A's S(j+1) already waited for K_{j+1}
              ok = wait_bounded(BAR(L::KV_FULL + knext % S), (knext / S) & 1, wc, SITE_MMA_KV, unit);
              if (!ok) break;
              tc_fence_after();
            }
            issue_s(1, slot_addr(knext));
            umma_commit(BAR(L::S_FULL + 1));
          }
        }
        kvbase += 2 * nmax;
      }
      // every MMA this thread issued completes before tensor memory is freed
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

template <int D, bool CAUSAL, bool VARLEN, bool BIAS = false, bool SPLIT = false>
cudaError_t launch_fwd_v(const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D>;
  auto kern = fwd_kernel<D, CAUSAL, VARLEN, BIAS, SPLIT>;
  static std::atomic<unsigned long long> ready{0};
  cudaError_t e = setup_kernel_once(kern, L::kSmemBytes, kFwdLaunchRegs, ready);
  if (e != cudaSuccess) return e;
  kern<<<a.sched.grid, kFwdThreads, L::kSmemBytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.o, a.lse, a.o_bf16, a.geom,
                                                             a.scale_log2, a.sched, a.status, a.wait_limit_ns,
                                                             a.stall_unit, a.bias, a.bias_sb, a.bias_sh,
                                                             a.bias_sq, a.part, a.splits, a.chunk);
  e = cudaGetLastError();
  if (e != cudaSuccess || !SPLIT) return e;
  // merge the key splits of every query row by their log-sum-exp
  return launch_split_combine(a.part, static_cast<float*>(a.o), a.lse, a.sched.heads * a.geom.nq, a.geom.nq,
                              a.splits, D, stream);
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
  if (a.splits > 1) return launch_fwd_v<D, CAUSAL, false, false, true>(a, stream);
  if (a.bias) return launch_fwd_v<D, CAUSAL, true, true>(a, stream);
  const bool square = !a.geom.seqlens_q && !a.geom.seqlens_k && a.geom.nq == a.geom.nk && !a.o_bf16;
  return square ? launch_fwd_v<D, CAUSAL, false>(a, stream) : launch_fwd_v<D, CAUSAL, true>(a, stream);
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return a.causal ? launch_fwd_t<64, true>(a, stream) : launch_fwd_t<64, false>(a, stream);
  return a.causal ? launch_fwd_t<128, true>(a, stream) : launch_fwd_t<128, false>(a, stream);
}

}  // namespace fa
