// Banded schedule of the gradient's leftover tiles (host and device).
//
// After `waves` full waves of whole pair tiles, `ntail` < G pair tiles are
// left for G pairs.  Each of them is a time line of L = B * tblocks K-blocks
// (the samples' 64-token blocks one after another), and the work is cut into
// segments (tile, [t0, t1)) so that every pair gets about ntail * L / G
// K-blocks and, more to the point, so that the pairs that run at the same
// moment read the same (sample, K-block) of different tiles: their A and G
// slabs are then shared in L2 instead of each pair streaming its own from
// HBM, which halved the speed of the tail when every pair sat at its own
// offset.
//
// The cut follows Euclid's algorithm on (n pairs, m tiles) over a time range
// [t0, t1) shared by all m tiles:
//   n >= m ("band" level): q = n / m bands of the range; pair p0 + r m + j
//     takes tile m0 + j over band r, and leaves.  The bands either cover the
//     whole range (a "cover" level, bands of equal length; the n - q m
//     remaining pairs get nothing more) or are cut at t0 + r m l / n, the
//     fair share of each pair ("exact"), and the n mod m remaining pairs go
//     on with the rest of the range on all m tiles.
//   n < m ("take" level): pair p0 + j takes tile m0 + j over the whole range;
//     the pairs go on with the m - n tiles left.
// Every band level runs its pairs in lockstep on one offset, and the levels
// a pair passes through are few (kTailMaxSegs), which bounds the partial
// tiles a pair holds.  Which band levels cover (bit l of `cover` for level
// l) is chosen on the host: exact levels give the best balance, a cover
// level stops the recursion.
//
// Slots: the contribution of pair p0 + x at a level is numbered base + x,
// base counting the pairs of the earlier levels (q m for a band level, n for
// a take level), so no two contributions share a slot and the numbers stay
// below kTailMaxSegs * G.
#pragma once
#include <stdint.h>

namespace dpclip {

constexpr int kTailMaxLevels = 16;
constexpr int kTailMaxSegs = 3;   // segments (partial tiles) per pair at most

struct TailWalk {
  int p0, n, m0, m, q, base, level;
  long long t0, t1;
  bool cover, done;

  __host__ __device__ __forceinline__ void load(uint32_t mask) {
    done = !(level < kTailMaxLevels && n > 0 && m > 0 && t1 > t0);
    q = n >= m ? n / m : 0;
    cover = ((mask >> level) & 1u) != 0;
  }
  __host__ __device__ __forceinline__ void start(int G, int ntail, long long L, uint32_t mask) {
    p0 = 0;
    n = G;
    m0 = 0;
    m = ntail;
    base = 0;
    level = 0;
    t0 = 0;
    t1 = L;
    load(mask);
  }
  __host__ __device__ __forceinline__ bool band() const { return n >= m; }
  // boundary r (0..q) of the bands of a band level
  __host__ __device__ __forceinline__ long long edge(int r) const {
    const long long l = t1 - t0;
    return cover ? t0 + l * r / q : t0 + l * r * m / n;
  }
  __host__ __device__ __forceinline__ void advance(uint32_t mask) {
    if (band()) {
      base += q * m;
      if (cover) {
        done = true;
        return;
      }
      t0 = edge(q);
      p0 += q * m;
      n -= q * m;
    } else {
      base += n;
      m0 += n;
      m -= n;
    }
    ++level;
    load(mask);
  }
};

struct TailSeg {
  int tile;           // tail tile (0 .. ntail-1)
  long long t0, t1;   // K-block range of the time line
  int slot;
};

// Pair c at the walk's current level: -1 if the pair has left (or never had
// a part), 0 if it waits for a later level, 1 with its segment in s.
__host__ __device__ __forceinline__ int tail_seg_of(const TailWalk& w, int c, TailSeg& s) {
  const int x = c - w.p0;
  if (x < 0 || x >= w.n) return -1;
  if (w.band()) {
    if (x >= w.q * w.m) return 0;
    const int r = x / w.m;
    s.tile = w.m0 + x % w.m;
    s.t0 = w.edge(r);
    s.t1 = w.edge(r + 1);
  } else {
    s.tile = w.m0 + x;
    s.t0 = w.t0;
    s.t1 = w.t1;
  }
  s.slot = w.base + x;
  return 1;
}

// Pair c's non-empty segments, shortest first (a stable order), into
// out[0 .. kTailMaxSegs); returns how many there are (the host keeps the
// count within kTailMaxSegs).  Running the short ones first puts a pair's
// longest segment, usually the one that ends a tile, just before its waves,
// whose long items then cover the last CTA's combination of the tile.
// Pairs that reach the same level have the same history, so they keep
// running that level's segments side by side.
__host__ __device__ __forceinline__ int tail_pair_segs(int G, int ntail, long long L,
                                                       uint32_t mask, int c, TailSeg* out) {
  int ns = 0;
  if (ntail <= 0) return 0;
  TailWalk w;
  w.start(G, ntail, L, mask);
  for (; !w.done && ns < kTailMaxSegs; w.advance(mask)) {
    TailSeg sg;
    const int r = tail_seg_of(w, c, sg);
    if (r < 0) break;
    if (r == 0 || sg.t1 <= sg.t0) continue;
    int j = ns++;
    for (; j > 0 && out[j - 1].t1 - out[j - 1].t0 > sg.t1 - sg.t0; --j) out[j] = out[j - 1];
    out[j] = sg;
  }
  return ns;
}

// Calls f(slot) for every non-empty contribution to tail tile tt, in the
// order of the walk (a fixed order: the combination is deterministic).
template <class F>
__host__ __device__ __forceinline__ void tail_tile_slots(int G, int ntail, long long L,
                                                         uint32_t mask, int tt, F&& f) {
  TailWalk w;
  w.start(G, ntail, L, mask);
  for (; !w.done; w.advance(mask)) {
    const int j = tt - w.m0;
    if (j < 0 || j >= w.m) break;
    if (w.band()) {
      for (int r = 0; r < w.q; ++r)
        if (w.edge(r + 1) > w.edge(r)) f(w.base + r * w.m + j);
    } else if (j < w.n) {
      f(w.base + j);
      break;
    }
  }
}

}  // namespace dpclip
