// C ABI of the library: argument checks, TMA descriptors, launches and the
// device status word.  The operation each entry point computes is stated in
// include/fa.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "internal.h"

// Device status word written by the kernels when a bounded wait gives up:
// [0] code, [1] wait site, [2] block, [3] work unit.  First failure wins.
__device__ int g_fa_status[4];

namespace {

constexpr long long kDefaultL2Budget = 32LL << 20;  // K+V bytes of one L2 head group
constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
int g_last_failure[4];

fa_status device_info(DeviceInfo& out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FA_ERR_LAUNCH;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return FA_ERR_LAUNCH;
    d.status = static_cast<int*>(p);
    d.ready = true;
  }
  out = d;
  return FA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Encoded tensor maps, cached by everything that goes into them (base
// address, element type, extents, box), so that repeated calls on the same
// tensors skip the driver's encoder.  A map depends on nothing else: reusing
// one for a buffer freed and allocated again at the same address with the
// same shape is still exact.  64 entries, replaced round robin.
struct MapKey {
  const void* base;
  int elem_bytes, heads, rows, inner, box_inner, box_rows;
  bool operator==(const MapKey& o) const {
    return base == o.base && elem_bytes == o.elem_bytes && heads == o.heads && rows == o.rows && inner == o.inner &&
           box_inner == o.box_inner && box_rows == o.box_rows;
  }
};

constexpr int kMapCacheSize = 64;
std::mutex g_map_mu;
MapKey g_map_keys[kMapCacheSize];
CUtensorMap g_maps[kMapCacheSize];
int g_map_count = 0, g_map_next = 0;

// 3-D map over [heads][rows][inner] elements of `elem_bytes` (2: bf16, 1:
// E4M3 bytes), box = box_inner x box_rows x 1 with the 128-byte swizzle (the
// layout the MMA descriptors expect).  Rows past `rows` read as zeros.
bool encode_map(CUtensorMap* m, const MapKey& key) {
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < g_map_count; ++i) {
      if (g_map_keys[i] == key) {
        *m = g_maps[i];
        return true;
      }
    }
  }
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t eb = static_cast<cuuint64_t>(key.elem_bytes);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(key.inner), static_cast<cuuint64_t>(key.rows),
                        static_cast<cuuint64_t>(key.heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(key.inner) * eb,
                           static_cast<cuuint64_t>(key.rows) * key.inner * eb};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(key.box_inner), static_cast<cuuint32_t>(key.box_rows), 1};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = fn(m, key.elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                  const_cast<void*>(key.base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  int slot;
  if (g_map_count < kMapCacheSize) {
    slot = g_map_count++;
  } else {
    slot = g_map_next;
    g_map_next = (g_map_next + 1) % kMapCacheSize;
  }
  g_map_keys[slot] = key;
  g_maps[slot] = *m;
  return true;
}

// bf16 [heads][n][d], boxes of 64 columns x box_rows rows.
bool encode_bf16_map(CUtensorMap* m, const void* base, int heads, int n, int d, int box_rows = fa::kTileRows) {
  return encode_map(m, MapKey{base, 2, heads, n, d, 64, box_rows});
}

// one-byte elements [heads][rows][inner], 128 x 128 boxes (one 128-byte row
// of the box per matrix row).
bool encode_u8_map(CUtensorMap* m, const void* base, int heads, int rows, int inner) {
  return encode_map(m, MapKey{base, 1, heads, rows, inner, 128, fa::kTileRows});
}

unsigned long long wait_limit_ns() {
  static unsigned long long v = []() -> unsigned long long {
    const char* s = std::getenv("FA_WAIT_LIMIT_MS");
    long long ms = s ? std::atoll(s) : 0;
    if (ms <= 0) ms = 4000;
    return static_cast<unsigned long long>(ms) * 1000000ULL;
  }();
  return v;
}

// Testing only: a unit index n >= 0 makes CTA 0 of the next launches skip one
// tile load of the n-th work unit it processes (the decode kernel: CTA n
// skips its first stage), so that a pipeline wait runs out and the timeout
// path can be exercised without faulting anything.  -1 (the default) means
// never.  Its first value comes from FA_TEST_STALL_UNIT, read once per
// process; fa_test_set_stall changes it.
std::atomic<int>& stall_unit_cell() {
  static std::atomic<int> cell([]() {
    const char* s = std::getenv("FA_TEST_STALL_UNIT");
    return (s && *s) ? std::atoi(s) : -1;
  }());
  return cell;
}

int test_stall_unit() { return stall_unit_cell().load(std::memory_order_relaxed); }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

fa_status check_sizes(int B, int H, int N, int d, int causal) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * N >= (1LL << 31)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  return FA_OK;
}

// n: rows the units tile (query rows for the forward and dQ, keys for dK/dV);
// n_stream: rows every unit of a head streams through (sizes the L2 groups).
fa::SchedParams make_sched(int heads, int n, int d, int causal, int grid_cap, long long budget,
                           int unit_rows = fa::kUnitRows, int cost_grows = 1, int n_stream = 0) {
  fa::SchedParams sp;
  sp.heads = heads;
  sp.units_per_head = (n + unit_rows - 1) / unit_rows;
  sp.cost_grows = cost_grows;
  sp.group_heads =
      fa::sched_group_heads(heads, n_stream > 0 ? n_stream : n, d, budget > 0 ? budget : kDefaultL2Budget);
  const long long units = static_cast<long long>(heads) * sp.units_per_head;
  sp.grid = static_cast<int>(units < grid_cap ? units : grid_cap);
  sp.causal = causal;
  return sp;
}

// Strides in elements; a query stride of 0 broadcasts one row of key
// biases over the queries, otherwise rows hold Nk keys.
fa_status check_bias(const void* bias, long long sb, long long sh, long long sq, int Nk) {
  if (!bias) return FA_ERR_INVALID_ARG;
  if (sb < 0 || sh < 0 || sq < 0 || (sq != 0 && sq < Nk)) return FA_ERR_INVALID_ARG;
  if (!aligned(bias, 2)) return FA_ERR_MISALIGNED;
  return FA_OK;
}

fa_status fwd_common(const void* q, const void* k, const void* v, void* o, int o_dtype, float* lse,
                     const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale,
                     int causal, fa_stream_t stream, const void* bias = nullptr, long long bias_sb = 0,
                     long long bias_sh = 0, long long bias_sq = 0) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (bias) {
    const fa_status bs = check_bias(bias, bias_sb, bias_sh, bias_sq, Nk);
    if (bs != FA_OK) return bs;
  }
  if (o_dtype != FA_DTYPE_F32 && o_dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, H, Nq, d, causal);
  if (st != FA_OK) return st;
  st = check_sizes(B, H, Nk, d, causal);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      (seqlens_q && !aligned(seqlens_q, 4)) || (seqlens_k && !aligned(seqlens_k, 4)))
    return FA_ERR_MISALIGNED;
  DeviceInfo di;
  if (device_info(di) != FA_OK) return FA_ERR_LAUNCH;
  const int heads = B * H;
  fa::FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  if (!encode_bf16_map(&a.tm_q, q, heads, Nq, d) || !encode_bf16_map(&a.tm_k, k, heads, Nk, d) ||
      !encode_bf16_map(&a.tm_v, v, heads, Nk, d))
    return FA_ERR_LAUNCH;
  a.o = o;
  a.o_bf16 = o_dtype == FA_DTYPE_BF16;
  a.lse = lse;
  a.geom.nq = Nq;
  a.geom.nk = Nk;
  a.geom.seqlens_q = seqlens_q;
  a.geom.seqlens_k = seqlens_k;
  a.geom.heads_per_batch = H;
  a.d = d;
  a.causal = causal;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.sched = make_sched(heads, Nq, d, causal, di.sms, 0, fa::kUnitRows, 1, Nk);
  a.status = di.status;
  a.wait_limit_ns = wait_limit_ns();
  a.stall_unit = test_stall_unit();
  a.bias = static_cast<const uint16_t*>(bias);
  a.bias_sb = bias_sb;
  a.bias_sh = bias_sh;
  a.bias_sq = bias_sq;
  return fa::launch_fwd(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// Key splits of the split-key forward: at most kMaxKeySplits, at least two
// key tiles each, and only as many as it takes to fill the SMs once.
constexpr int kMaxKeySplits = 16;

int key_split_cap(int N) {
  const int nkt = (N + fa::kTileRows - 1) / fa::kTileRows;
  const int cap = nkt / 2;
  return cap < 1 ? 1 : (cap > kMaxKeySplits ? kMaxKeySplits : cap);
}

void key_splits(int heads, int N, int sms, int& splits, int& chunk) {
  const int nkt = (N + fa::kTileRows - 1) / fa::kTileRows;
  const long long units = static_cast<long long>(heads) * ((N + fa::kUnitRows - 1) / fa::kUnitRows);
  long long s = units >= sms ? 1 : (sms + units - 1) / units;
  const int cap = key_split_cap(N);
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  chunk = static_cast<int>((nkt + s - 1) / s);
  splits = (nkt + chunk - 1) / chunk;
}

// Checks the arguments of a backward call (the workspace only for alignment;
// it may be null) and fills every field of `a` but the row-term buffer.  q, dO, o, lse, dq: [B*H][Nq] rows; k, v, dk, dv:
// [B*H][Nk] rows.
// need_o = false (the single-pass backward, which forms D without O): o is
// ignored and may be null.
fa_status bwd_prepare(fa::BwdArgs& a, const void* q, const void* k, const void* v, const void* o, int o_dtype,
                      const float* lse, const void* dO, float* dq, float* dk, float* dv, const float* workspace,
                      const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale,
                      int causal, bool need_o = true) {
  if (!need_o) {
    o = q;  // never read
    o_dtype = FA_DTYPE_F32;
  }
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (o_dtype != FA_DTYPE_F32 && o_dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, H, Nq, d, causal);
  if (st != FA_OK) return st;
  st = check_sizes(B, H, Nk, d, causal);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) ||
      (workspace && !aligned(workspace, 4)) || (seqlens_q && !aligned(seqlens_q, 4)) ||
      (seqlens_k && !aligned(seqlens_k, 4)))
    return FA_ERR_MISALIGNED;
  DeviceInfo di;
  if (device_info(di) != FA_OK) return FA_ERR_LAUNCH;
  const int heads = B * H;
  std::memset(&a, 0, sizeof(a));
  if (!encode_bf16_map(&a.tm_q, q, heads, Nq, d) || !encode_bf16_map(&a.tm_k, k, heads, Nk, d) ||
      !encode_bf16_map(&a.tm_v, v, heads, Nk, d) || !encode_bf16_map(&a.tm_do, dO, heads, Nq, d))
    return FA_ERR_LAUNCH;
  a.o = o;
  a.o_bf16 = o_dtype == FA_DTYPE_BF16;
  a.lse = lse;
  a.dout = static_cast<const uint16_t*>(dO);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.heads = heads;
  a.geom.nq = Nq;
  a.geom.nk = Nk;
  a.geom.seqlens_q = seqlens_q;
  a.geom.seqlens_k = seqlens_k;
  a.geom.heads_per_batch = H;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  // dK/dV: one unit per 128-key tile, heaviest at the start of the sequence,
  // streaming the head's queries; dQ: one unit per 128-query tile, heaviest
  // at the end, streaming the head's keys.
  a.sched_kv = make_sched(heads, Nk, d, causal, di.sms, 0, fa::kTileRows, 0, Nq);
  a.sched_q = make_sched(heads, Nq, d, causal, di.sms, 0, fa::kTileRows, 1, Nk);
  a.grid_kv = a.sched_kv.grid;
  a.grid_q = a.sched_q.grid;
  a.status = di.status;
  a.wait_limit_ns = wait_limit_ns();
  a.stall_unit = test_stall_unit();
  return FA_OK;
}

// Key splits of the decode kernel.  Each split is at least kDecodeMinChunk
// keys; the count aims at a few waves of two resident CTAs per SM over all
// heads, and is capped so that the workspace bound below holds.
constexpr int kDecodeMinChunk = 512;
constexpr int kDecodeMaxSplits = 256;

int decode_max_splits(int Nk) {
  const int s = (Nk + kDecodeMinChunk - 1) / kDecodeMinChunk;
  return s < 1 ? 1 : (s > kDecodeMaxSplits ? kDecodeMaxSplits : s);
}

void decode_splits(int heads, int Nk, int sms, int& splits, int& chunk) {
  const long long target = 4LL * 2 * sms;  // four waves of two CTAs per SM
  long long s = (target + heads - 1) / heads;
  const int cap = decode_max_splits(Nk);
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  chunk = static_cast<int>(((Nk + s - 1) / s + 63) / 64 * 64);
  splits = (Nk + chunk - 1) / chunk;
}

// Both backward kernels on prepared arguments; without a workspace the row
// term lives in a stream-ordered allocation freed behind the kernels.
fa_status bwd_launch(fa::BwdArgs& a, float* workspace, int B, int H, int Nq, fa_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* delta = workspace;
  if (!delta) {
    if (cudaMallocAsync(reinterpret_cast<void**>(&delta), fa_bwd_workspace_bytes(B, H, Nq), s) != cudaSuccess)
      return FA_ERR_LAUNCH;
  }
  a.delta = delta;
  cudaError_t e = fa::launch_bwd(a, s);
  if (!workspace) {
    cudaError_t e2 = cudaFreeAsync(delta, s);
    if (e == cudaSuccess) e = e2;
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}


}  // namespace

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, float* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, fa_stream_t stream) {
  return fwd_common(q, k, v, o, FA_DTYPE_F32, lse, nullptr, nullptr, B, H, N, N, d, scale, causal, stream);
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, float* o, float* lse, const int* seqlens_q,
                        const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                        fa_stream_t stream) {
  return fwd_common(q, k, v, o, FA_DTYPE_F32, lse, seqlens_q, seqlens_k, B, H, Nq, Nk, d, scale, causal, stream);
}

fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, int o_dtype, float* lse,
                    const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale,
                    int causal, fa_stream_t stream) {
  return fwd_common(q, k, v, o, o_dtype, lse, seqlens_q, seqlens_k, B, H, Nq, Nk, d, scale, causal, stream);
}

fa_status fa_fwd_bias(const void* q, const void* k, const void* v, void* o, int o_dtype, float* lse,
                      const void* bias, long long bias_stride_b, long long bias_stride_h, long long bias_stride_q,
                      const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale,
                      int causal, fa_stream_t stream) {
  if (!bias) return FA_ERR_INVALID_ARG;  // fwd_common treats null as no mask
  return fwd_common(q, k, v, o, o_dtype, lse, seqlens_q, seqlens_k, B, H, Nq, Nk, d, scale, causal, stream, bias,
                    bias_stride_b, bias_stride_h, bias_stride_q);
}

size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  if (static_cast<long long>(B) * H * N >= (1LL << 31)) return 0;
  return static_cast<size_t>(B) * H * key_split_cap(N) * N * (d + 1) * sizeof(float);
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, float* o, float* lse, float* workspace, int B,
                         int H, int N, int d, float scale, int causal, fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, H, N, d, causal);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      (workspace && !aligned(workspace, 16)))
    return FA_ERR_MISALIGNED;
  DeviceInfo di;
  if (device_info(di) != FA_OK) return FA_ERR_LAUNCH;
  const int heads = B * H;
  int splits = 1, chunk = 1;
  key_splits(heads, N, di.sms, splits, chunk);
  if (splits == 1) return fwd_common(q, k, v, o, FA_DTYPE_F32, lse, nullptr, nullptr, B, H, N, N, d, scale, causal,
                                     stream);
  fa::FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  if (!encode_bf16_map(&a.tm_q, q, heads, N, d) || !encode_bf16_map(&a.tm_k, k, heads, N, d) ||
      !encode_bf16_map(&a.tm_v, v, heads, N, d))
    return FA_ERR_LAUNCH;
  a.o = o;
  a.lse = lse;
  a.geom.nq = N;
  a.geom.nk = N;
  a.geom.heads_per_batch = H;
  a.d = d;
  a.causal = causal;
  a.scale_log2 = scale * 1.4426950408889634f;
  // units: (head, query pair, key split), heaviest pairs first under the
  // causal mask; splits of one pair are consecutive units
  a.sched = make_sched(heads, N, d, causal, di.sms, 0, fa::kUnitRows, 1, N);
  a.sched.units_per_head *= splits;
  const long long units = static_cast<long long>(heads) * a.sched.units_per_head;
  a.sched.grid = static_cast<int>(units < di.sms ? units : di.sms);
  a.splits = splits;
  a.chunk = chunk;
  a.status = di.status;
  a.wait_limit_ns = wait_limit_ns();
  a.stall_unit = test_stall_unit();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* part = workspace;
  if (!part) {
    if (cudaMallocAsync(reinterpret_cast<void**>(&part), fa_fwd_splitkv_workspace_bytes(B, H, N, d), s) !=
        cudaSuccess)
      return FA_ERR_LAUNCH;
  }
  a.part = part;
  cudaError_t e = fa::launch_fwd(a, s);
  if (!workspace) {
    cudaError_t e2 = cudaFreeAsync(part, s);
    if (e == cudaSuccess) e = e2;
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

size_t fa_fwd_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
  if (B < 1 || H < 1 || Nq < 1 || Nq > FA_DECODE_MAX_Q || Nk < 1 || (d != 64 && d != 128)) return 0;
  if (static_cast<long long>(B) * H * Nk >= (1LL << 31)) return 0;
  return static_cast<size_t>(B) * H * decode_max_splits(Nk) * Nq * (d + 1) * sizeof(float);
}

fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, float* o, float* lse, int B, int H, int N,
                     int d, float scale, int causal, fa_stream_t stream) {
  if (!q8 || !k8 || !vt8 || !o || !lse) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, H, N, d, causal);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED_D;
  if (N % 16 != 0) return FA_ERR_INVALID_ARG;  // rows of v^T: whole 16-byte groups
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(vt8, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_MISALIGNED;
  DeviceInfo di;
  if (device_info(di) != FA_OK) return FA_ERR_LAUNCH;
  const int heads = B * H;
  fa::FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  if (!encode_u8_map(&a.tm_q, q8, heads, N, d) || !encode_u8_map(&a.tm_k, k8, heads, N, d) ||
      !encode_u8_map(&a.tm_v, vt8, heads, d, N))
    return FA_ERR_LAUNCH;
  a.o = o;
  a.lse = lse;
  a.geom.nq = N;
  a.geom.nk = N;
  a.geom.heads_per_batch = H;
  a.d = d;
  a.causal = causal;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.sched = make_sched(heads, N, d, causal, di.sms, 0, fa::kUnitRows, 1, N);
  a.status = di.status;
  a.wait_limit_ns = wait_limit_ns();
  a.stall_unit = test_stall_unit();
  return fa::launch_fwd_fp8(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

fa_status fa_fwd_decode(const void* q, const void* k, const void* v, float* o, float* lse, const int* seqlens_q,
                        const int* seqlens_k, float* workspace, int B, int H, int Nq, int Nk, int d, float scale,
                        int causal, fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, H, Nk, d, causal);
  if (st != FA_OK) return st;
  if (Nq < 1 || Nq > FA_DECODE_MAX_Q) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      (workspace && !aligned(workspace, 16)) || (seqlens_q && !aligned(seqlens_q, 4)) ||
      (seqlens_k && !aligned(seqlens_k, 4)))
    return FA_ERR_MISALIGNED;
  DeviceInfo di;
  if (device_info(di) != FA_OK) return FA_ERR_LAUNCH;
  const int heads = B * H;
  fa::DecArgs a;
  std::memset(&a, 0, sizeof(a));
  if (!encode_bf16_map(&a.tm_k, k, heads, Nk, d, 64) || !encode_bf16_map(&a.tm_v, v, heads, Nk, d, 64))
    return FA_ERR_LAUNCH;
  a.q = static_cast<const uint16_t*>(q);
  a.o = o;
  a.lse = lse;
  a.geom.nq = Nq;
  a.geom.nk = Nk;
  a.geom.seqlens_q = seqlens_q;
  a.geom.seqlens_k = seqlens_k;
  a.geom.heads_per_batch = H;
  a.heads = heads;
  a.d = d;
  a.causal = causal;
  a.scale_log2 = scale * 1.4426950408889634f;
  decode_splits(heads, Nk, di.sms, a.splits, a.chunk);
  a.status = di.status;
  a.wait_limit_ns = wait_limit_ns();
  a.stall_unit = test_stall_unit();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* part = workspace;
  if (a.splits > 1 && !part) {
    if (cudaMallocAsync(reinterpret_cast<void**>(&part), fa_fwd_decode_workspace_bytes(B, H, Nq, Nk, d), s) !=
        cudaSuccess)
      return FA_ERR_LAUNCH;
  }
  a.part = part;
  cudaError_t e = fa::launch_decode(a, s);
  if (part && !workspace) {
    cudaError_t e2 = cudaFreeAsync(part, s);
    if (e == cudaSuccess) e = e2;
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  if (static_cast<long long>(B) * H * N >= (1LL << 31)) return 0;
  return static_cast<size_t>(B) * H * N * sizeof(float);
}

fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, int o_dtype, const float* lse,
                    const void* dO, float* dq, float* dk, float* dv, float* workspace, const int* seqlens_q,
                    const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                    fa_stream_t stream) {
  fa::BwdArgs a;
  fa_status st = bwd_prepare(a, q, k, v, o, o_dtype, lse, dO, dq, dk, dv, workspace, seqlens_q, seqlens_k, B, H, Nq,
                             Nk, d, scale, causal);
  if (st != FA_OK) return st;
  return bwd_launch(a, workspace, B, H, Nq, stream);
}

fa_status fa_bwd_bias(const void* q, const void* k, const void* v, const void* o, int o_dtype, const float* lse,
                      const void* dO, const void* bias, long long bias_stride_b, long long bias_stride_h,
                      long long bias_stride_q, float* dq, float* dk, float* dv, float* workspace,
                      const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale,
                      int causal, fa_stream_t stream) {
  fa_status st = check_bias(bias, bias_stride_b, bias_stride_h, bias_stride_q, Nk);
  if (st != FA_OK) return st;
  fa::BwdArgs a;
  st = bwd_prepare(a, q, k, v, o, o_dtype, lse, dO, dq, dk, dv, workspace, seqlens_q, seqlens_k, B, H, Nq, Nk, d,
                   scale, causal);
  if (st != FA_OK) return st;
  a.bias = fa::BiasRef{static_cast<const uint16_t*>(bias), bias_stride_b, bias_stride_h, bias_stride_q};
  return bwd_launch(a, workspace, B, H, Nq, stream);
}

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const float* o, const float* lse,
                        const void* dO, float* dq, float* dk, float* dv, float* workspace, const int* seqlens_q,
                        const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                        fa_stream_t stream) {
  return fa_bwd_ex(q, k, v, o, FA_DTYPE_F32, lse, dO, dq, dk, dv, workspace, seqlens_q, seqlens_k, B, H, Nq, Nk, d,
                   scale, causal, stream);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const float* o, const float* lse, const void* dO,
                 float* dq, float* dk, float* dv, float* workspace, int B, int H, int N, int d, float scale,
                 int causal, fa_stream_t stream) {
  return fa_bwd_ex(q, k, v, o, FA_DTYPE_F32, lse, dO, dq, dk, dv, workspace, nullptr, nullptr, B, H, N, N, d, scale,
                   causal, stream);
}

// Scratch of fa_bwd_noalloc: the backward row term D for up to
// FA_NOALLOC_MAX_ROWS rows, resident on every device that loads the library.
// Host code must not hand this name to a kernel (on the host it is only a
// stand-in for the symbol); the device address comes from
// cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) float g_fa_noalloc_delta[FA_NOALLOC_MAX_ROWS];

static std::mutex g_noalloc_mu;
static float* g_noalloc_ptr[kMaxDevices];

fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const float* o, const float* lse,
                         const void* dO, float* dq, float* dk, float* dv, int B, int H, int N, int d, float scale,
                         int causal, fa_stream_t stream) {
  // the scratch bound first, before any descriptor is built
  if (B < 1 || H < 1 || N < 1 || static_cast<long long>(B) * H * N > FA_NOALLOC_MAX_ROWS) return FA_ERR_INVALID_ARG;
  fa::BwdArgs a;
  fa_status st =
      bwd_prepare(a, q, k, v, o, FA_DTYPE_F32, lse, dO, dq, dk, dv, nullptr, nullptr, nullptr, B, H, N, N, d, scale,
                  causal);
  if (st != FA_OK) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_LAUNCH;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_fa_noalloc_delta) != cudaSuccess || !p) return FA_ERR_LAUNCH;
      g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    a.delta = g_noalloc_ptr[dev];  // every row is written by the dQ kernel before dK/dV reads it
  }
  return fa::launch_bwd(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

fa_status fa_bwd_single_pass(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                             const void* bias, long long bias_stride_b, long long bias_stride_h,
                             long long bias_stride_q, float* dq, float* dk, float* dv, float* workspace,
                             const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq, int Nk, int d,
                             float scale, int causal, fa_stream_t stream) {
  if (bias) {
    const fa_status bs = check_bias(bias, bias_stride_b, bias_stride_h, bias_stride_q, Nk);
    if (bs != FA_OK) return bs;
  }
  fa::BwdArgs a;
  fa_status st = bwd_prepare(a, q, k, v, nullptr, FA_DTYPE_F32, lse, dO, dq, dk, dv, workspace, seqlens_q, seqlens_k,
                             B, H, Nq, Nk, d, scale, causal, false);
  if (st != FA_OK) return st;
  if (bias) a.bias = fa::BiasRef{static_cast<const uint16_t*>(bias), bias_stride_b, bias_stride_h, bias_stride_q};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* delta = workspace;
  if (!delta) {
    if (cudaMallocAsync(reinterpret_cast<void**>(&delta), fa_bwd_workspace_bytes(B, H, Nq), s) != cudaSuccess)
      return FA_ERR_LAUNCH;
  }
  a.delta = delta;
  cudaError_t e = fa::launch_bwd_single_pass(a, s);
  if (!workspace) {
    cudaError_t e2 = cudaFreeAsync(delta, s);
    if (e == cudaSuccess) e = e2;
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

fa_status fa_bwd_stage(int stage, const void* q, const void* k, const void* v, const float* o, const float* lse,
                       const void* dO, float* dq, float* dk, float* dv, float* workspace, int B, int H, int N, int d,
                       float scale, int causal, fa_stream_t stream) {
  if (stage < 0 || stage > 3 || !workspace) return FA_ERR_INVALID_ARG;
  fa::BwdArgs a;
  fa_status st =
      bwd_prepare(a, q, k, v, o, FA_DTYPE_F32, lse, dO, dq, dk, dv, workspace, nullptr, nullptr, B, H, N, N, d, scale,
                  causal, stage < 2);
  if (st != FA_OK) return st;
  a.delta = workspace;
  return fa::launch_bwd_stage(a, stage, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                              : FA_ERR_LAUNCH;
}

fa_status fa_sync_status(fa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_DEVICE_FAULT;
  int h[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(h, g_fa_status, sizeof(h)) != cudaSuccess) return FA_ERR_DEVICE_FAULT;
  if (h[0] != 0) {
    {
      std::lock_guard<std::mutex> lock(g_mu);
      std::memcpy(g_last_failure, h, sizeof(h));
    }
    const int zero[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_fa_status, zero, sizeof(zero)) != cudaSuccess) return FA_ERR_DEVICE_FAULT;
    return h[0] == FA_ERR_TIMEOUT ? FA_ERR_TIMEOUT : FA_ERR_DEVICE_FAULT;
  }
  return FA_OK;
}

fa_status fa_test_set_stall(int unit) {
  if (unit < -1) return FA_ERR_INVALID_ARG;
  stall_unit_cell().store(unit, std::memory_order_relaxed);
  return FA_OK;
}

fa_status fa_last_failure(int out[4]) {
  if (!out) return FA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  std::memcpy(out, g_last_failure, sizeof(g_last_failure));
  return FA_OK;
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK: success";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null pointer or size/flag out of range";
    case FA_ERR_UNSUPPORTED_D: return "FA_ERR_UNSUPPORTED_D: head dimension must be 64 or 128";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED: tensor pointer breaks the 16-byte (4-byte) alignment rule";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: the CUDA runtime refused a launch or an allocation";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel pipeline wait ran past its limit";
    case FA_ERR_DEVICE_FAULT: return "FA_ERR_DEVICE_FAULT: the stream reported a CUDA error";
  }
  return "unknown fa_status";
}

long long fa_sched_enumerate(int heads, int N, int d, int causal, int grid, long long l2_budget_bytes,
                             int* out_cta, int* out_head, int* out_pair, long long capacity) {
  if (heads < 1 || N < 1 || grid < 1 || (d != 64 && d != 128) || (causal != 0 && causal != 1)) return -1;
  if (static_cast<long long>(heads) * N >= (1LL << 31)) return -1;
  fa::SchedParams sp = make_sched(heads, N, d, causal, grid, l2_budget_bytes);
  long long w = 0;
  for (int c = 0; c < sp.grid; ++c) {
    fa::SchedIter it = fa::sched_begin(sp);
    int head, pair;
    while (fa::sched_next(it, sp, c, head, pair)) {
      if (w < capacity && out_cta && out_head && out_pair) {
        out_cta[w] = c;
        out_head[w] = head;
        out_pair[w] = pair;
      }
      ++w;
    }
  }
  return w;
}

}  // extern "C"
