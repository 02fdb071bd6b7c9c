// schedule.h -- persistent tile scheduler: task index -> output tile.
//
// Persistent CTAs ("TIRx GEMM on Blackwell", V6): a fixed grid of clusters,
// cluster c takes tasks c, c + C, c + 2C, ... until the tiles run out, so the
// per-CTA setup (barriers, TMEM allocation) is paid once.
//
// Grouped raster ("Choosing schedules and instructions for a backend",
// section 3, the G = 16 order): the M tiles are split into groups of `group`
// consecutive tiles; tasks walk the groups in order and, inside a group, walk
// the N tiles with the group's M tiles innermost.  Tasks that run at the same
// time then touch few distinct B column panels (reused through L2) and a
// bounded band of A rows.  Unlike the tutorial's order, the last group may be
// shorter than `group`, so any M works; every tile is visited exactly once.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define GB300_HD __host__ __device__ __forceinline__
#else
#define GB300_HD inline
#endif

namespace gb300 {

struct TileGrid {
    int32_t m_tiles;  // ceil(M / block_m)
    int32_t n_tiles;  // ceil(N / block_n)
    int32_t group;    // M tiles per raster group (>= 1)
};

GB300_HD int64_t tile_count(const TileGrid& g) {
    return static_cast<int64_t>(g.m_tiles) * g.n_tiles;
}

// Task -> (m tile, n tile).  Requires 0 <= task < tile_count(g).
GB300_HD void tile_of_task(const TileGrid& g, int64_t task, int32_t& mt, int32_t& nt) {
    const int64_t per_group = static_cast<int64_t>(g.group) * g.n_tiles;
    const int64_t grp = task / per_group;
    const int64_t first_m = grp * g.group;
    const int64_t rows_in_group =
        (g.m_tiles - first_m) < g.group ? (g.m_tiles - first_m) : g.group;
    const int64_t r = task - grp * per_group;
    nt = static_cast<int32_t>(r / rows_in_group);
    mt = static_cast<int32_t>(first_m + r % rows_in_group);
}

}  // namespace gb300
