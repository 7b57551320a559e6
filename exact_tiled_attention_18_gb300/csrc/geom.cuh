// Sequence geometry shared by the forward and backward kernels.
//
// A batch is padded to Nq query rows and Nk key rows per head; sequence b of
// the batch uses only its first lq = seqlens_q[b] queries and lk =
// seqlens_k[b] keys (all rows when no lengths are given).  Under the causal
// mask query i sees key j iff j <= i + (lk - lq): the last query is aligned
// with the last key, which for lq == lk is j <= i, and lets one decoding query
// see every key ("FlashAttention Interview Questions: IO Complexity, Tiling,
// and Numerical Stability", section "Does subtracting the maximum solve every
// numerical issue?": unequal lengths, padding and packed sequences need an
// explicit alignment).
#pragma once

#include "internal.h"

namespace fa {

struct HeadLen {
  int lq, lk, off, nkt;  // valid queries, valid keys, causal offset lk - lq, key tiles
};

__device__ __forceinline__ HeadLen head_len(const SeqGeom& g, int head) {
  HeadLen h;
  const int b = head / g.heads_per_batch;
  h.lq = g.seqlens_q ? min(max(__ldg(g.seqlens_q + b), 0), g.nq) : g.nq;
  h.lk = g.seqlens_k ? min(max(__ldg(g.seqlens_k + b), 0), g.nk) : g.nk;
  h.off = h.lk - h.lq;
  h.nkt = (h.lk + kTileRows - 1) / kTileRows;
  return h;
}

// Key tiles query tile `qtile` needs: 0 if its rows are all padding or see no
// key, otherwise the tiles up to the one holding its last row's last key.
__device__ __forceinline__ int query_tile_keys(const HeadLen& h, int qtile, bool causal) {
  const int first = qtile * kTileRows;
  if (first >= h.lq) return 0;
  if (!causal) return h.nkt;
  const int kmax = min(h.lq, first + kTileRows) - 1 + h.off;
  return kmax < 0 ? 0 : min(h.nkt, kmax / kTileRows + 1);
}

// Query tiles [i0, i1) that see some key of key tile `ktile` (empty when the
// tile is padding or no query reaches it).
__device__ __forceinline__ void key_tile_queries(const HeadLen& h, int ktile, bool causal, int& i0, int& i1) {
  i1 = (h.lq + kTileRows - 1) / kTileRows;
  i0 = 0;
  if (ktile * kTileRows >= h.lk) {
    i0 = i1;
    return;
  }
  if (causal) {
    const int row = ktile * kTileRows - h.off;  // first query that sees the tile's first key
    i0 = row <= 0 ? 0 : row / kTileRows;
    if (i0 > i1) i0 = i1;
  }
}

// Whether some (query, key) pair of tiles (qtile, ktile) is masked by the
// causal rule, i.e. the tile's last key lies past its first query's last key.
__device__ __forceinline__ bool tile_crosses_diagonal(const HeadLen& h, int qtile, int ktile) {
  return ktile * kTileRows + kTileRows - 1 > qtile * kTileRows + h.off;
}

}  // namespace fa
