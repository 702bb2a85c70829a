// Tile schedules of the persistent CTA-pair grouped matmul.
//
// Tiles are numbered group by group (column tile fastest); group j owns
// tiles [T[j], T[j+1]).  Two ways to hand them to the ncl clusters of the grid:
//
//   * strided: cluster c takes tiles c, c + ncl, c + 2 ncl, ...  Clusters that
//     work at the same time work on neighbouring tiles, which share operands
//     in L2.  Every tile of the forward and dX contractions costs the same,
//     so this is as balanced as whole tiles allow.
//   * by group (weight gradient): a dW tile of group j contracts over the
//     group's own rows, kb(j) blocks of 64, so tiles of different groups cost
//     differently and the strided order can leave one cluster with twice the
//     average.  Instead group j gets a run of n_j clusters of its own, each
//     taking at most floor(L / kb(j)) of its tiles, with L the smallest load
//     for which the runs fit in the grid.  A cluster then touches one group
//     only, so this is used when the operands of all groups fit in L2.
//
// The functions are plain integer arithmetic, compiled for host and device
// alike, so the schedules can be checked on the host.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {

// Largest j in [0, E) with P[j] <= v (P has E + 1 non-decreasing entries, P[E] > v).
template <typename Int>
MOE_HD int prefix_find(const Int* P, int E, int64_t v) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (P[mid] <= v) lo = mid; else hi = mid;
  }
  return lo;
}

// a / b for a < 2^22, b >= 1.  On the device a float quotient, exact after
// one correction step (its error is below one there), since integer division
// is a long dependent sequence and the schedule search does many.
MOE_HD uint32_t udiv_small(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
  uint32_t q = static_cast<uint32_t>(__fdividef(static_cast<float>(a), static_cast<float>(b)));
  if (q * b > a) --q;
  else if ((q + 1) * b <= a) ++q;
  return q;
#else
  return a / b;
#endif
}

// Clusters that a group of `tiles` tiles of kb blocks each needs when no
// cluster may take more than L blocks: 0 without tiles; ncl + 1 (infeasible)
// when one tile is deeper than L.  The callers keep tiles + L below 2^22.
MOE_HD uint32_t group_clusters(uint32_t tiles, uint32_t kb, uint32_t L, uint32_t ncl) {
  if (tiles == 0 || kb == 0) return 0;
  const uint32_t per = udiv_small(L, kb);
  if (per == 0) return ncl + 1;
  return udiv_small(tiles + per - 1, per);
}

struct TileRef {
  int g;      // group
  int local;  // tile within the group
};

// Walk of one cluster's tiles.  Strided: t runs over the global tile index.
// By group: the cluster's group g, its first tile i0 and the run length n.
struct TileWalk {
  int64_t t;
  int g, i, n;
};

MOE_HD void walk_strided_init(TileWalk& w, int c) { w.t = c; w.g = -1; w.i = 0; w.n = 0; }

MOE_HD bool walk_strided_next(TileWalk& w, const int32_t* T, int E, int ncl, TileRef& r) {
  if (w.t >= T[E]) return false;
  r.g = prefix_find(T, E, w.t);
  r.local = static_cast<int>(w.t - T[r.g]);
  w.t += ncl;
  return true;
}

// C: prefix over the groups of their cluster runs (C[E] = clusters in use).
MOE_HD void walk_group_init(TileWalk& w, int c, const int32_t* C, int E) {
  w.t = 0;
  if (c >= C[E]) { w.g = -1; w.i = 0; w.n = 0; return; }
  w.g = prefix_find(C, E, c);
  w.n = C[w.g + 1] - C[w.g];
  w.i = c - C[w.g];
}

MOE_HD bool walk_group_next(TileWalk& w, const int32_t* T, TileRef& r) {
  if (w.g < 0 || w.i >= T[w.g + 1] - T[w.g]) return false;
  r.g = w.g;
  r.local = w.i;
  w.i += w.n;
  return true;
}

}  // namespace moe
