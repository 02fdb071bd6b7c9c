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

// Largest tile count the scheduler handles: its index arithmetic is 32-bit (a
// 64-bit division is a long software routine on the GPU, and the producer's
// first TMA issue waits on this map).  Far beyond any output that fits in memory.
constexpr int64_t kMaxTiles = int64_t(1) << 31;

// Task -> (m tile, n tile).  Requires 0 <= task < tile_count(g) < kMaxTiles.
GB300_HD void tile_of_task(const TileGrid& g, int64_t task, int32_t& mt, int32_t& nt) {
    const uint32_t t = static_cast<uint32_t>(task);
    const uint32_t group = static_cast<uint32_t>(g.group);
    const uint32_t per_group = group * static_cast<uint32_t>(g.n_tiles);  // <= tile count
    const uint32_t grp = t / per_group;
    const uint32_t first_m = grp * group;
    const uint32_t left = static_cast<uint32_t>(g.m_tiles) - first_m;
    const uint32_t rows_in_group = left < group ? left : group;
    const uint32_t r = t - grp * per_group;
    const uint32_t q = r / rows_in_group;
    nt = static_cast<int32_t>(q);
    mt = static_cast<int32_t>(first_m + (r - q * rows_in_group));
}

}  // namespace gb300
