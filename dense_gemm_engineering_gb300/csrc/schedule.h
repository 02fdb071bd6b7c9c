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
// bounded band of A rows, which stays in L2 while the group walks all of N:
// A is read from DRAM about once and B once per group.  Unlike the tutorial's
// order, the last group may be shorter than `group`, so any M works; every
// tile is visited exactly once.
//
// The same walk with the roles of M and N exchanged (order = kOrderN: groups
// of `group` N tiles, the M tiles walked inside a group with the group's N
// tiles innermost) keeps a band of B columns in L2 instead and reads A once
// per group: the better choice when B's band is the one that fits (the
// tutorial's memory report: the operand whose reuse window exceeds L2 is the
// one that must stream).
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define GB300_HD __host__ __device__ __forceinline__
#else
#define GB300_HD inline
#endif

namespace gb300 {

enum : int32_t { kOrderM = 0, kOrderN = 1 };

struct TileGrid {
    int32_t m_tiles;  // ceil(M / block_m)
    int32_t n_tiles;  // ceil(N / block_n)
    int32_t group;    // tiles per raster group along the grouped dimension (>= 1)
    int32_t order;    // kOrderM: groups of M tiles; kOrderN: groups of N tiles
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
    const bool by_n = (g.order == kOrderN);
    const uint32_t grouped = static_cast<uint32_t>(by_n ? g.n_tiles : g.m_tiles);
    const uint32_t other = static_cast<uint32_t>(by_n ? g.m_tiles : g.n_tiles);
    const uint32_t t = static_cast<uint32_t>(task);
    const uint32_t group = static_cast<uint32_t>(g.group);
    const uint32_t per_group = group * other;  // <= tile count
    const uint32_t grp = t / per_group;
    const uint32_t first = grp * group;
    const uint32_t left = grouped - first;
    const uint32_t in_group = left < group ? left : group;
    const uint32_t r = t - grp * per_group;
    const uint32_t q = r / in_group;                       // position along the other dimension
    const uint32_t g_idx = first + (r - q * in_group);     // position along the grouped one
    mt = static_cast<int32_t>(by_n ? q : g_idx);
    nt = static_cast<int32_t>(by_n ? g_idx : q);
}

}  // namespace gb300
