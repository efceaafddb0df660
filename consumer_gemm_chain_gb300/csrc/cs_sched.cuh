// Dependency-ordered dispatch order of a chain's tile units, as a closed form
// that host and device code share: entry i of a schedule is computed on its
// own, so a schedule can be written by one thread per entry.
//
// Row tiles form groups of group_m.  The fused order takes steps t = 0, 1, ...;
// at step t, stage s lists every unit of group t - s*lag (column-tile-major
// inside the group, or row-major; a split stage after the first may instead
// list K-split 0 of every tile of the group, then K-split 1, ...), so every
// producer unit a consumer waits on is listed at an earlier step or earlier in
// the same step, and an in-order dispatcher cannot deadlock.  A stage alone
// lists its groups in turn.
//
// A causal stage split into key-range pieces (kv[s] > 0: the attention units
// of tile row m cover key groups 0..m, in pieces of kv[s] groups) lists
// n_tiles[s] * ceil((m + 1) / kv[s]) units in row m, row by row, each row's
// units by column tile and then piece.
#pragma once
#include <cstdint>

namespace cs {

struct SchedGeo {
  int stages = 2;
  int m_tiles = 1;    // tile rows
  int group_m = 1;    // tile rows per group
  int lag = 1;        // groups between consecutive stages
  int row_major = 0;  // units of a group row by row instead of column by column
  int ks_major = 0;   // stages after the first: units of a group by K-split, then column, then row
  int n_tiles[3] = {0, 0, 0};
  int splits[3] = {1, 1, 1};
  int kv[3] = {0, 0, 0};  // key groups per piece of a causal stage (0: none)
};

__host__ __device__ inline uint32_t sched_enc(int s, int m, int n, int ks) {
  return (static_cast<uint32_t>(s) << 30) | (static_cast<uint32_t>(ks) << 26) | (static_cast<uint32_t>(m) << 14) |
         static_cast<uint32_t>(n);
}

__host__ __device__ inline int sched_groups(const SchedGeo& g) { return (g.m_tiles + g.group_m - 1) / g.group_m; }

// tile rows in groups [0, k), k clamped to [0, groups]
__host__ __device__ inline long long sched_rows_before(const SchedGeo& g, int k) {
  if (k <= 0) return 0;
  const long long r = static_cast<long long>(k) * g.group_m;
  return r < g.m_tiles ? r : g.m_tiles;
}

// tile rows of group k (0 outside the valid groups)
__host__ __device__ inline long long sched_rows_of(const SchedGeo& g, int k) {
  if (k < 0 || k >= sched_groups(g)) return 0;
  return sched_rows_before(g, k + 1) - sched_rows_before(g, k);
}

__host__ __device__ inline long long sched_units_per_row(const SchedGeo& g, int s) {
  return static_cast<long long>(g.n_tiles[s]) * g.splits[s];
}

// Units of stage s per column tile in tile row m: its K-splits, or its pieces.
__host__ __device__ inline int sched_pieces(const SchedGeo& g, int s, int m) {
  return g.kv[s] > 0 ? (m + g.kv[s]) / g.kv[s] : g.splits[s];
}

// Units of stage s in tile rows [0, r): with pieces, sum over k = 1..r of
// ceil(k / kv) = kv * a * (a + 1) / 2 + b * (a + 1) for r = a * kv + b.
__host__ __device__ inline long long sched_units_rows(const SchedGeo& g, int s, long long r) {
  if (g.kv[s] <= 0) return sched_units_per_row(g, s) * r;
  const long long a = r / g.kv[s], b = r % g.kv[s];
  return static_cast<long long>(g.n_tiles[s]) * (g.kv[s] * a * (a + 1) / 2 + b * (a + 1));
}

// Entries of the fused order before step t.
__host__ __device__ inline long long sched_fused_before(const SchedGeo& g, int t) {
  long long o = 0;
  for (int s = 0; s < g.stages; ++s) o += sched_units_rows(g, s, sched_rows_before(g, t - s * g.lag));
  return o;
}

__host__ __device__ inline int sched_fused_steps(const SchedGeo& g) { return sched_groups(g) + (g.stages - 1) * g.lag; }

__host__ __device__ inline long long sched_fused_count(const SchedGeo& g) {
  return sched_fused_before(g, sched_fused_steps(g));
}

__host__ __device__ inline long long sched_stage_count(const SchedGeo& g, int s) {
  return sched_units_rows(g, s, g.m_tiles);
}

// Entry j of stage s's units in the group of tile rows [m0, m0 + rows).
__host__ __device__ inline uint32_t sched_in_group(const SchedGeo& g, int s, int m0, int rows, long long j) {
  const int sp = g.splits[s];
  int m, n, ks;
  if (g.kv[s] > 0) {
    // row by row; in a row, column tile then piece
    m = m0;
    long long c = static_cast<long long>(g.n_tiles[s]) * sched_pieces(g, s, m);
    while (j >= c && m + 1 < m0 + rows) {
      j -= c;
      ++m;
      c = static_cast<long long>(g.n_tiles[s]) * sched_pieces(g, s, m);
    }
    const int np = sched_pieces(g, s, m);
    n = static_cast<int>(j / np);
    ks = static_cast<int>(j % np);
  } else if (g.row_major) {
    const long long per_row = sched_units_per_row(g, s);
    m = m0 + static_cast<int>(j / per_row);
    const long long r = j % per_row;
    n = static_cast<int>(r / sp);
    ks = static_cast<int>(r % sp);
  } else if (g.ks_major && s > 0 && sp > 1) {
    // K range first: a consumer's K range waits only on the producer column
    // tiles of that range, which a producer stage in several waves finishes first
    const long long per_ks = static_cast<long long>(rows) * g.n_tiles[s];
    ks = static_cast<int>(j / per_ks);
    const long long r = j % per_ks;
    n = static_cast<int>(r / rows);
    m = m0 + static_cast<int>(r % rows);
  } else {
    const long long per_col = static_cast<long long>(rows) * sp;
    n = static_cast<int>(j / per_col);
    const long long r = j % per_col;
    m = m0 + static_cast<int>(r / sp);
    ks = static_cast<int>(r % sp);
  }
  return sched_enc(s, m, n, ks);
}

// Entry i (0 <= i < sched_fused_count) of the fused order.
__host__ __device__ inline uint32_t sched_fused_entry(const SchedGeo& g, long long i) {
  // the step holding entry i: the last t with sched_fused_before(t) <= i
  int lo = 0, hi = sched_fused_steps(g) - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (sched_fused_before(g, mid) <= i)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int t = lo;
  long long j = i - sched_fused_before(g, t);
  for (int s = 0; s < g.stages; ++s) {
    const int k = t - s * g.lag;
    const long long rows = sched_rows_of(g, k);
    const long long c = sched_units_rows(g, s, sched_rows_before(g, k + 1)) - sched_units_rows(g, s, sched_rows_before(g, k));
    if (j < c) return sched_in_group(g, s, static_cast<int>(sched_rows_before(g, k)), static_cast<int>(rows), j);
    j -= c;
  }
  return 0xFFFFFFFFu;  // i out of range
}

// Entry i (0 <= i < sched_stage_count) of stage s run alone.
__host__ __device__ inline uint32_t sched_stage_entry(const SchedGeo& g, int s, long long i) {
  int k;
  if (g.kv[s] > 0) {
    // the group holding entry i: the last k with sched_units_rows(rows before k) <= i
    int lo = 0, hi = sched_groups(g) - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (sched_units_rows(g, s, sched_rows_before(g, mid)) <= i)
        lo = mid;
      else
        hi = mid - 1;
    }
    k = lo;
  } else {
    const long long per_group = static_cast<long long>(g.group_m) * sched_units_per_row(g, s);
    k = static_cast<int>(i / per_group);
    if (k >= sched_groups(g)) k = sched_groups(g) - 1;
  }
  const long long base = sched_units_rows(g, s, sched_rows_before(g, k));
  return sched_in_group(g, s, static_cast<int>(sched_rows_before(g, k)), static_cast<int>(sched_rows_of(g, k)),
                        i - base);
}

}  // namespace cs
