// Persistent tile scheduler shared by the kernels and by host-side tests.
//
// Work unit: one head (b, h) and one block index p along the sequence (for
// the forward pass a pair of 128-row query tiles, rows [256 p, 256 p + 256);
// for the backward kernels a single 128-row tile).  Under the causal mask
// query tile t sweeps key tiles 0..t, so a forward unit costs about 4p + 3
// tile products and the cost of a unit grows or shrinks with p: the work is
// parallel over heads and over the query sequence, the partitioning the
// FlashAttention-2 discussion on the FlashAttention Interview Questions page
// ("What changed in FlashAttention-2 ...") credits for the speedup.
//
// Order: heads are taken in groups small enough that a group's K and V stay
// resident in L2 while every CTA sweeps them; inside a group units are
// ordered heaviest first (longest-processing-time first).  Units are dealt to
// the G persistent CTAs in rounds that alternate direction ("snake"), so the
// heaviest unit of one round pairs with the lightest of the next.  The partial
// last round of a group always runs forward, and the starting CTA rotates by
// that round's size from group to group, so the leftovers spread evenly.
//
// Every role of a CTA runs the same iterator and sees the same sequence.
#pragma once

#if defined(__CUDACC__)
#define FA_HD __host__ __device__ __forceinline__
#else
#define FA_HD inline
#endif

namespace fa {

constexpr int kTileRows = 128;               // query rows (and keys) per tile
constexpr int kUnitRows = 2 * kTileRows;      // query rows per work unit

struct SchedParams {
  int heads;           // B * H
  int units_per_head;  // ceil(N / 256)
  int group_heads;     // heads per L2 group
  int grid;            // persistent CTAs
  int causal;
  int cost_grows;      // causal only: 1 if a unit's cost grows with its index p
};

struct SchedIter {
  int g;        // current group
  int k;        // next round inside the group
  int rot;      // CTA rotation of the current group
  int hs;       // heads in the current group
  int gsize;    // units in the current group
  int full;     // complete rounds in the current group
  int rounds;   // rounds including a partial one
};

FA_HD void sched_setup_group(SchedIter& it, const SchedParams& p) {
  int left = p.heads - it.g * p.group_heads;
  it.hs = left < p.group_heads ? left : p.group_heads;
  it.gsize = it.hs * p.units_per_head;
  it.full = it.gsize / p.grid;
  it.rounds = it.full + ((it.gsize % p.grid) ? 1 : 0);
  it.k = 0;
}

FA_HD SchedIter sched_begin(const SchedParams& p) {
  SchedIter it;
  it.g = 0;
  it.rot = 0;
  sched_setup_group(it, p);
  return it;
}

// Next unit of CTA `cta`; returns false when the CTA has no work left.
FA_HD bool sched_next(SchedIter& it, const SchedParams& p, int cta, int& head, int& pair) {
  const int num_groups = (p.heads + p.group_heads - 1) / p.group_heads;
  while (it.g < num_groups) {
    while (it.k < it.rounds) {
      const int kk = it.k++;
      int c = cta - it.rot;
      if (c < 0) c += p.grid;
      const bool forward = ((it.full - kk) & 1) == 0;
      const int pos = forward ? c : (p.grid - 1 - c);
      const int r = kk * p.grid + pos;
      if (r < it.gsize) {
        const int level = r / it.hs;
        head = it.g * p.group_heads + (r - level * it.hs);
        pair = (p.causal && p.cost_grows) ? (p.units_per_head - 1 - level) : level;
        return true;
      }
    }
    it.rot = (it.rot + it.gsize % p.grid) % p.grid;
    ++it.g;
    if (it.g < num_groups) sched_setup_group(it, p);
  }
  return false;
}

// Heads per group: as many as keep the group's K and V (bf16) within
// `l2_budget_bytes`, at least one.
FA_HD int sched_group_heads(int heads, int n, int d, long long l2_budget_bytes) {
  long long per_head = 2LL * n * d * 2;
  long long g = per_head > 0 ? l2_budget_bytes / per_head : heads;
  if (g < 1) g = 1;
  if (g > heads) g = heads;
  return static_cast<int>(g);
}

}  // namespace fa
