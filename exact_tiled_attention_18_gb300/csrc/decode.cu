// Decode-shaped forward: a few query rows per head against a long K/V.
//
// Single-token decoding reads the whole key/value history once per step
// while the query side is one row (or a handful), so the work is about one
// FLOP per byte of K/V: bound by HBM, not by the tensor cores ("FlashAttention
// Interview Questions: IO Complexity, Tiling, and Numerical Stability", last
// section: prefill and single-token decoding differ in query shape and data
// reuse).  The kernel therefore streams K/V tiles through shared memory with
// TMA and does the arithmetic on the CUDA cores, and it splits each head's
// keys over many CTAs so that the whole GPU pulls on HBM.
//
//   decode_kernel   one CTA per (head, key split): a TMA producer warp fills
//                   a ring of 64-key K/V stages; four consumer warps each own
//                   16 keys of every stage and keep their own running maximum,
//                   sum and output accumulator (the online softmax of the
//                   same page, section "How can softmax be computed across
//                   tiles?"), merged across warps at the end.
//   decode_combine  merges the splits of a row by their log-sum-exp:
//                   O = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M).
//
// Every pipeline wait is bounded, as in the other kernels.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "geom.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kDecStageKeys = 64;
constexpr int kDecConsumerWarps = 4;
constexpr int kDecThreads = 32 * (kDecConsumerWarps + 1);
constexpr float kDecTau = 8.f;  // lazy rescale threshold (log2 units), as in the prefill kernel
constexpr float kDecLn2 = 0.6931471805599453f;

enum DecSite : int { SITE_DEC_EMPTY = 35, SITE_DEC_FULL = 36 };

// Resident CTAs per SM: two, except with 8 query rows, whose registers need
// the whole file; that case runs one CTA per SM with twice the ring, so the
// bytes in flight per SM stay the same.
template <int NQ>
constexpr int dec_ctas_per_sm() { return NQ > 4 ? 1 : 2; }

template <int D, int NQ>
struct DecLayout {
  static constexpr int kBox = 64 * 64 * 2;       // 64 columns x 64 keys bf16: 128-byte rows, swizzled
  static constexpr int kHalf = (D / 64) * kBox;  // K (or V) of one stage
  static constexpr int kStage = 2 * kHalf;
  static constexpr int kStages = ((D == 128) ? 3 : 6) * (2 / dec_ctas_per_sm<NQ>());
  static constexpr int kBarOff = kStages * kStage;  // FULL[s] then EMPTY[s]
  static constexpr int kMiscOff = kBarOff + 2 * kStages * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  // after the sweep the ring holds the warps' partial results
  static_assert(kDecConsumerWarps * 8 * (D + 2) * 4 <= kBarOff, "combine area exceeds the ring");
};

// Byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled box
// (the chunk index is XORed with the row index modulo 8).
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// bf16 pair (element 2e in the low half) -> fp32 pair
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t u) {
  return f2_pack(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kDecConsumerWarps)); }

template <int D, int NQ>
__global__ void __launch_bounds__(kDecThreads, dec_ctas_per_sm<NQ>())
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const uint16_t* __restrict__ q, float* __restrict__ o, float* __restrict__ lse,
                  float* __restrict__ part, const SeqGeom geom, const float scale_log2, const int causal,
                  const int splits, const int chunk, int* status, const unsigned long long limit_ns,
                  const int stall_unit) {
  using L = DecLayout<D, NQ>;
  constexpr int S = L::kStages;
  constexpr int G = D / 16;        // lanes per key in the score phase, 16 columns each
  constexpr int KP = 32 / G;       // keys per pass
  constexpr int PASSES = 16 / KP;  // passes over a warp's 16 keys of a stage
  constexpr int CW = D / 32;       // output columns per lane
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kBarOff;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int head = blockIdx.x / splits;
  const int split = blockIdx.x - head * splits;
  const HeadLen h = head_len(geom, head);
  // the last valid query sees every valid key, so the split covers keys
  // [k0, k1) of the sequence (nothing when the sequence has no query)
  const int k0 = split * chunk;
  const int k1 = min(k0 + chunk, h.lq > 0 ? h.lk : 0);
  const int nst = k1 > k0 ? (k1 - k0 + kDecStageKeys - 1) / kDecStageKeys : 0;
  const int unit = static_cast<int>(blockIdx.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bars + 8 * s, 1);
      mbar_init(bars + 8 * (S + s), kDecConsumerWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const WaitCtl wc{abort_flag, status, limit_ns};

  if (warp == kDecConsumerWarps) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && nst > 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      int issued = 0;
      bool ok = true;
      for (; issued < nst; ++issued) {
        const int s = issued % S;
        ok = wait_bounded(bars + 8 * (S + s), ((issued / S) & 1) ^ 1, wc, SITE_DEC_EMPTY, unit);
        if (!ok) break;
        if (unit == stall_unit && issued == 0) continue;  // testing hook: leave this stage unloaded
        const uint32_t full = bars + 8 * s;
        mbar_arrive_expect_tx(full, L::kStage);
        const uint32_t st = sbase + s * L::kStage;
        const int key = k0 + issued * kDecStageKeys;
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          tma_load_3d(st + b * L::kBox, &tm_k, full, 64 * b, key, head);
          tma_load_3d(st + L::kHalf + b * L::kBox, &tm_v, full, 64 * b, key, head);
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA can exit
        for (int s = 0; s < S; ++s) {
          if (issued > s) {
            const int last = issued - 1 - ((issued - 1 - s) % S);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bars + 8 * s, (last / S) & 1)) {
              if (globaltimer_ns() - t0 > limit_ns) break;
            }
          }
        }
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int g = lane / G;     // score phase: key g of each pass
  const int part_ = lane % G;  // columns [16 part_, 16 part_ + 16)
  const int kblk = (16 * part_) / 64;
  const int kc0 = ((16 * part_) % 64) / 8;
  uint32_t qp[NQ][8];
  int kend[NQ];
#pragma unroll
  for (int r = 0; r < NQ; ++r) {
    if (r < geom.nq) {
      const uint4* src =
          reinterpret_cast<const uint4*>(q + (static_cast<size_t>(head) * geom.nq + r) * D + 16 * part_);
      const uint4 a = __ldg(src), b = __ldg(src + 1);
      qp[r][0] = a.x; qp[r][1] = a.y; qp[r][2] = a.z; qp[r][3] = a.w;
      qp[r][4] = b.x; qp[r][5] = b.y; qp[r][6] = b.z; qp[r][7] = b.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) qp[r][e] = 0u;
    }
    kend[r] = r < h.lq ? (causal ? min(r + h.off + 1, h.lk) : h.lk) : 0;
  }
  float m_ref[NQ], l[NQ], acc[NQ][CW];
#pragma unroll
  for (int r = 0; r < NQ; ++r) {
    m_ref[r] = -CUDART_INF_F;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < CW; ++c) acc[r][c] = 0.f;
  }
  const float cl2 = scale_log2;
  bool ok = true;
  for (int i = 0; i < nst; ++i) {
    const int s = i % S;
    ok = __all_sync(0xffffffffu, wait_bounded(bars + 8 * s, (i / S) & 1, wc, SITE_DEC_FULL, unit));
    if (!ok) break;
    const uint8_t* kb = smem + s * L::kStage;
    const uint8_t* vb = kb + L::kHalf;
    const int kbase = k0 + i * kDecStageKeys + 16 * warp;
    // scores of this warp's 16 keys: key (pass, g) in every lane of group g
    float sc[PASSES][NQ];
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      const int R = 16 * warp + ps * KP + g;
      const uint8_t* rowp = kb + kblk * L::kBox;
      const uint4 ka = *reinterpret_cast<const uint4*>(rowp + sw128(R, kc0));
      const uint4 kc = *reinterpret_cast<const uint4*>(rowp + sw128(R, kc0 + 1));
      const uint32_t kw[8] = {ka.x, ka.y, ka.z, ka.w, kc.x, kc.y, kc.z, kc.w};
      const int j = kbase + ps * KP + g;
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        uint64_t a2 = f2_pack(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 8; ++e) a2 = ffma2(bf2_to_f2(qp[r][e]), bf2_to_f2(kw[e]), a2);
        float a0, a1;
        f2_unpack(a2, a0, a1);
        float a = a0 + a1;
#pragma unroll
        for (int off = 1; off < G; off <<= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
        sc[ps][r] = (j < kend[r]) ? a : -CUDART_INF_F;
      }
    }
    // online softmax per query row, shared by the whole warp
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      float mx = sc[0][r];
#pragma unroll
      for (int ps = 1; ps < PASSES; ++ps) mx = fmaxf(mx, sc[ps][r]);
#pragma unroll
      for (int off = G; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mt = mx * cl2;
      if (mt > m_ref[r] + kDecTau) {  // warp-uniform
        const float alpha = ex2_approx(m_ref[r] - mt);  // 0 on the first eligible key
        m_ref[r] = mt;
        l[r] *= alpha;
#pragma unroll
        for (int c = 0; c < CW; ++c) acc[r][c] *= alpha;
      }
      const float mu = (m_ref[r] == -CUDART_INF_F) ? 0.f : m_ref[r];
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) {
        const float p = ex2_approx(fmaf(sc[ps][r], cl2, -mu));
        sc[ps][r] = p;
        l[r] += p;  // the same p in every lane of the group
      }
    }
    // O += P V over the warp's 16 keys; lane owns columns [CW lane, CW lane + CW)
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const int R = 16 * warp + kk;
      float vf[CW];
      if constexpr (D == 128) {
        const uint2 v2 =
            *reinterpret_cast<const uint2*>(vb + (lane >> 4) * L::kBox + sw128(R, (lane & 15) >> 1) + ((lane & 1) << 3));
        f2_unpack(bf2_to_f2(v2.x), vf[0], vf[1]);
        f2_unpack(bf2_to_f2(v2.y), vf[2], vf[3]);
      } else {
        const uint32_t v1 = *reinterpret_cast<const uint32_t*>(vb + sw128(R, lane >> 2) + ((lane & 3) << 2));
        f2_unpack(bf2_to_f2(v1), vf[0], vf[1]);
      }
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        const float p = __shfl_sync(0xffffffffu, sc[kk / KP][r], (kk % KP) * G);
#pragma unroll
        for (int c = 0; c < CW; ++c) acc[r][c] = fmaf(p, vf[c], acc[r][c]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (S + s));
  }
  // each lane of a group holds the group's partial sum; add the groups
#pragma unroll
  for (int r = 0; r < NQ; ++r) {
#pragma unroll
    for (int off = G; off < 32; off <<= 1) l[r] += __shfl_xor_sync(0xffffffffu, l[r], off);
  }

  // ------------------------------------------- merge the four warps' results
  consumer_sync();  // every stage consumed: the ring is free
  float* cm = reinterpret_cast<float*>(smem);        // [warp][NQ] reference maximum (log2 units)
  float* cs = cm + kDecConsumerWarps * NQ;           // [warp][NQ] sum
  float* co = cs + kDecConsumerWarps * NQ;           // [warp][NQ][D] accumulator
  const bool aborted = *abort_flag != 0;
  if (!aborted) {
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      if (lane == 0) {
        cm[warp * NQ + r] = m_ref[r];
        cs[warp * NQ + r] = l[r];
      }
#pragma unroll
      for (int c = 0; c < CW; ++c) co[(warp * NQ + r) * D + CW * lane + c] = acc[r][c];
    }
  }
  consumer_sync();
  if (aborted) return;
  const size_t pbase = static_cast<size_t>(head) * splits + split;
  float* part_lse = part + static_cast<size_t>(gridDim.x) * geom.nq * D;  // after every split's O
  for (int item = threadIdx.x; item < NQ * (D / 4); item += 32 * kDecConsumerWarps) {
    const int r = item / (D / 4);
    const int c4 = item - r * (D / 4);
    if (r >= geom.nq) break;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kDecConsumerWarps; ++w) M = fmaxf(M, cm[w * NQ + r]);
    float sum = 0.f;
    float4 ov = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kDecConsumerWarps; ++w) {
        const float f = ex2_approx(cm[w * NQ + r] - M);  // a warp that saw no key has m = -inf: f = 0
        const float4 x = *reinterpret_cast<const float4*>(co + (w * NQ + r) * D + 4 * c4);
        sum = fmaf(f, cs[w * NQ + r], sum);
        ov.x = fmaf(f, x.x, ov.x);
        ov.y = fmaf(f, x.y, ov.y);
        ov.z = fmaf(f, x.z, ov.z);
        ov.w = fmaf(f, x.w, ov.w);
      }
    }
    const bool live = sum > 0.f;
    const float inv = live ? 1.0f / sum : 0.f;
    const float4 res = live ? make_float4(ov.x * inv, ov.y * inv, ov.z * inv, ov.w * inv)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    const float lse2 = live ? M + log2f(sum) : -CUDART_INF_F;
    if (splits == 1) {
      *reinterpret_cast<float4*>(o + (static_cast<size_t>(head) * geom.nq + r) * D + 4 * c4) = res;
      if (c4 == 0) lse[static_cast<size_t>(head) * geom.nq + r] = live ? lse2 * kDecLn2 : -CUDART_INF_F;
    } else {
      *reinterpret_cast<float4*>(part + (pbase * geom.nq + r) * D + 4 * c4) = res;
      if (c4 == 0) part_lse[pbase * geom.nq + r] = lse2;
    }
  }
}

// One warp per (head, query row): merge the splits' normalised outputs by
// their log-sum-exp (log2 units in the workspace).
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const float* __restrict__ part, float* __restrict__ o,
                                                             float* __restrict__ lse, const int rows,
                                                             const int nq, const int splits) {
  constexpr int CW = D / 32;
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // head * nq + r
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;  // uniform across the warp
  const int head = row / nq;
  const int r = row - head * nq;
  const float* part_lse = part + static_cast<size_t>(rows) * splits * D;
  auto lse_of = [&](int s) { return part_lse[(static_cast<size_t>(head) * splits + s) * nq + r]; };
  float M = -CUDART_INF_F;
  for (int s = lane; s < splits; s += 32) M = fmaxf(M, lse_of(s));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float* orow = o + static_cast<size_t>(row) * D + CW * lane;
  if (M == -CUDART_INF_F) {
#pragma unroll
    for (int c = 0; c < CW; ++c) orow[c] = 0.f;
    if (lane == 0) lse[row] = -CUDART_INF_F;
    return;
  }
  float sum = 0.f;
  for (int s = lane; s < splits; s += 32) sum += exp2f(lse_of(s) - M);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  float acc[CW];
#pragma unroll
  for (int c = 0; c < CW; ++c) acc[c] = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float f = exp2f(lse_of(s) - M);
    if (f == 0.f) continue;  // same value in every lane
    const float* src = part + ((static_cast<size_t>(head) * splits + s) * nq + r) * D + CW * lane;
#pragma unroll
    for (int c = 0; c < CW; ++c) acc[c] = fmaf(f, __ldg(src + c), acc[c]);
  }
  const float inv = 1.0f / sum;
#pragma unroll
  for (int c = 0; c < CW; ++c) orow[c] = acc[c] * inv;
  if (lane == 0) lse[row] = (M + log2f(sum)) * kDecLn2;
}

template <int D, int NQ>
cudaError_t launch_decode_t(const DecArgs& a, cudaStream_t stream) {
  using L = DecLayout<D, NQ>;
  auto kern = decode_kernel<D, NQ>;
  static std::atomic<unsigned long long> ready{0};
  cudaError_t e = setup_kernel_once(kern, L::kSmemBytes, 0, ready);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(a.heads) * a.splits;
  kern<<<static_cast<unsigned>(grid), kDecThreads, L::kSmemBytes, stream>>>(
      a.tm_k, a.tm_v, a.q, a.o, a.lse, a.part, a.geom, a.scale_log2, a.causal, a.splits, a.chunk, a.status,
      a.wait_limit_ns, a.stall_unit);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  const int rows = a.heads * a.geom.nq;
  decode_combine_kernel<D><<<(rows + 7) / 8, 256, 0, stream>>>(a.part, a.o, a.lse, rows, a.geom.nq, a.splits);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecArgs& a, cudaStream_t stream) {
  const int nq = a.geom.nq;
  if (nq <= 1) return launch_decode_t<D, 1>(a, stream);
  if (nq <= 2) return launch_decode_t<D, 2>(a, stream);
  if (nq <= 4) return launch_decode_t<D, 4>(a, stream);
  return launch_decode_t<D, 8>(a, stream);
}

}  // namespace

cudaError_t launch_split_combine(const float* part, float* o, float* lse, int rows, int nq, int splits, int d,
                                 cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
  if (d == 64)
    decode_combine_kernel<64><<<grid, 256, 0, stream>>>(part, o, lse, rows, nq, splits);
  else
    decode_combine_kernel<128><<<grid, 256, 0, stream>>>(part, o, lse, rows, nq, splits);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecArgs& a, cudaStream_t stream) {
  return a.d == 64 ? launch_decode_d<64>(a, stream) : launch_decode_d<128>(a, stream);
}

}  // namespace fa
