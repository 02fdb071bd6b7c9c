// gemm_kernel.cuh -- the sm_103a dense GEMM kernel (tcgen05 + TMA + TMEM).
//
// One persistent, warp-specialised kernel computes D = A.B^T (B stored N x K,
// K-major) or D = A.B (B stored K x N, MN-major) with FP16/BF16 operands, an
// FP32 accumulator in Tensor Memory and a 16-bit output; with F8 set it takes
// FP8 (E4M3 / E5M2) A and B, K-major, and writes round(alpha * A.B^T); with MX
// also set every 32 K elements of each row of A and B carry a UE8M0 scale
// (block-scaled FP8, "TIRx: A Unified Tile Primitive ML Compiler", kernel
// performance), which the tensor core applies (kind::mxf8f6f4.block_scale):
// each stage then also carries the k-block's scales, which the MMA issuer
// copies into TMEM (tcgen05.cp) before its four MMAs.
//
// Structure, and the passages it follows:
//   * Operands move GMEM -> SMEM by TMA into a ring of STAGES slots, 128-byte
//     swizzled ("TIRx GEMM on Blackwell", V4 and V5; TileFoundry tutorial,
//     section 5: SW128 TMA ring).  Stage s of the ring carries k-blocks
//     s, s + STAGES, ...; the ring position and its phase bit run on across
//     tiles (TileFoundry tutorial, section 6: the ring slot is a function of
//     the running k-block count, not of the tile).
//   * Four kinds of mbarrier hand buffers between the roles ("TIRx GEMM on
//     Blackwell", V7): full[s] (operands landed, TMA -> MMA), empty[s] (slot
//     free, MMA -> TMA), acc_full[b] (accumulator b ready, MMA -> epilogue),
//     acc_empty[b] (accumulator b drained, epilogue -> MMA).  A waiter on a
//     "free" barrier starts on the opposite parity, so the first pass through
//     the ring does not block; every reuse flips the phase bit (V2, V7).
//   * Warp 0: TMA producer.  Warp 1: allocates TMEM and, in the cluster's
//     leader CTA, issues tcgen05.mma.  Both loops run on the whole warp and
//     one elected lane issues each copy / MMA / commit.  Warps 2-5: epilogue
//     warpgroup (V7's writeback warpgroup).
//   * Persistent CTAs walk the tile list of schedule.h (V6; TileFoundry
//     sections 2-3).
//   * CG == 2: a cluster of two CTAs computes a 256-row tile with
//     tcgen05.mma.cta_group::2; CTA r holds rows 128r..128r+127 of the tile in
//     its own TMEM, loads its own 128 rows of A and its own half of B's tile
//     columns, and the leader's MMA reads both CTAs' shared memory (V8).
//   * The accumulator is double-buffered in TMEM (2 x BN columns), so the
//     epilogue of tile i overlaps the mainloop of tile i+1 ("write back without
//     blocking the next tile", Take away 1).
//   * Epilogue: tcgen05.ld -> FP32 registers -> cvt.rn to 16 bit -> 128-byte
//     swizzled SMEM staging (two buffers per warp, one with MX, outside the
//     load ring) ->
//     TMA store, which clips rows/columns outside D (TileFoundry section 5).
//     D is never cleared: every tile is written exactly once (section 6).
//
// Every barrier wait is bounded (kWaitLimitNs, or a shorter limit a self-test
// passes in GemmArgs).  A wait that runs out records the reason in the device
// status word and raises the abort flag of its CTA and of the other CTA of the
// pair, which every role polls; all roles leave their loops, and each warp
// that sees the flag waits 1 ms (for copies, MMAs and arrivals already in
// flight to land) before it joins the final cluster barrier; the CTA still
// frees TMEM, so the context survives.
#pragma once

#include <cstdint>

#include "ptx.cuh"
#include "schedule.h"

namespace gb300 {

// Device status word (read by gemm_device_status()).
static __device__ uint32_t g_gemm_status;

constexpr int kBlockK = 64;         // 64 x 16 bit = one 128-byte swizzle row
constexpr int kBlockK8 = 128;       // 128 x 8 bit: the same 128-byte row for FP8 inputs
constexpr int kNumThreads = 192;    // 6 warps: producer, MMA, 4 epilogue
constexpr int kEpilogueWarps = 4;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
// Pause between an epilogue warp's 64-column chunk stores (see the epilogue).
constexpr uint32_t kStorePaceNs = 1000;
constexpr int kStorePaceMinKBlocks = 32;

// L2 eviction priorities of the operand loads and the output stores
// (GemmArgs::l2_hints; bit 0 only marks an explicit choice).
enum : uint32_t { kHintALast = 2u, kHintBFirst = 4u, kHintDFirst = 8u };

// Status word layout: bits 0..7 = reason, bits 8..15 = role.
enum : uint32_t { kReasonTimeout = 1u, kReasonCounter = 2u };
enum : uint32_t {
    kRoleProducer = 1u,
    kRoleMma = 2u,
    kRoleEpilogue = 3u,
    kRoleDrain = 4u,
    kRoleSelfTest = 5u
};

template <int CG_, int BN_, int STAGES_, bool B_MN_, bool BF16_, int CONS_ = 1, int F8_ = 0,
          bool MX_ = false, int KS_ = 1>
struct KernelConfig {
    static constexpr int CG = CG_;            // CTAs per MMA (tcgen05 cta_group)
    // K-ranges of one tile computed by the CTAs of a cluster (1-CTA tiles
    // only): CTA k of the cluster multiplies the k-th of KS K-ranges into its
    // own TMEM and owns BN / KS of the tile's columns; the CTAs exchange the
    // FP32 partials of each other's columns through their idle operand rings
    // over distributed shared memory, and each sums and stores its own.
    static constexpr int KS = KS_;
    static constexpr int CLUSTER = CG * KS;   // CTAs per cluster
    // MMA consumers per CTA: 1, or 2 ("TIRx GEMM on Blackwell", V9: two MMAs on
    // different A rows share each staged B tile; each CTA holds 256 A rows).
    static constexpr int CONS = CONS_;
    static constexpr int A_ROWS = 128 * CONS;  // A rows each CTA loads per tile
    static constexpr int BM = A_ROWS * CG;     // tile rows
    static constexpr int BN = BN_;            // tile columns (MMA N)
    static constexpr int STAGES = STAGES_;    // SMEM ring depth
    static constexpr bool B_MN = B_MN_;       // B stored K x N (D = A.B)
    static constexpr bool BF16 = BF16_;       // output type (and input type unless F8)
    // Input type: 0 = the 16-bit output type; 1 = FP8 E4M3, 2 = FP8 E5M2 (OCP
    // 8-bit floating point), multiplied on tcgen05.mma kind::f8f6f4.
    static constexpr int F8 = F8_;
    static constexpr int BK = F8 ? kBlockK8 : kBlockK;  // K elements per ring stage
    static constexpr int ELEM_BYTES = F8 ? 1 : 2;
    static constexpr int MMA_K = F8 ? 32 : 16;         // K per MMA: 32 bytes either way
    static constexpr int B_ROWS = BN / CG;    // tile columns whose B this CTA loads
    // Block-scaled FP8 (MX): one UE8M0 scale per 32 K elements of every row of A
    // and of B, multiplied on tcgen05.mma kind::mxf8f6f4.block_scale.  Shared
    // memory per stage adds the A scales of this CTA's 128 rows (one 512-byte
    // atom) and the tile's B scales (one 4 KiB block, already laid out for the
    // TMEM copy), both loaded by TMA with the operands.
    static constexpr bool MX = MX_;
    static constexpr uint32_t SFA_BYTES = MX ? 512u : 0u;
    static constexpr uint32_t SFB_BYTES = MX ? 4096u : 0u;

    static constexpr uint32_t A_BYTES = uint32_t(A_ROWS) * BK * ELEM_BYTES;  // 16 KiB per consumer
    static constexpr uint32_t B_BYTES = uint32_t(B_ROWS) * BK * ELEM_BYTES;
    static constexpr uint32_t STAGE_TX = uint32_t(CG) * (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES);
    // Two accumulators of BN FP32 columns at a power-of-two stride (the TMEM
    // allocation is a power of two of at least 32 columns).
    static constexpr uint32_t ACC_STRIDE = BN <= 128 ? 128u : 256u;
    // Accumulator slots: with one consumer, two slots (the epilogue of tile i
    // overlaps the MMAs of tile i+1); with two consumers their two
    // accumulators fill TMEM, so one slot.
    static constexpr uint32_t NUM_ACC = CONS == 1 ? 2u : 1u;
    static constexpr uint32_t SLOT_COLS = uint32_t(CONS) * ACC_STRIDE;
    static constexpr uint32_t TMEM_COLS = NUM_ACC * SLOT_COLS;
    // Epilogue chunks: BN / 64 full 64-column chunks, plus one 32-column chunk
    // when BN is an odd multiple of 32.
    static constexpr int FULL_CHUNKS = BN / 64;
    static constexpr bool HALF_CHUNK = (BN % 64) != 0;
    static constexpr uint32_t EPI_BUF_BYTES = 32u * 128u;              // 32 rows x 64 cols
    // Staging buffers per epilogue warp: two (a chunk's store may still be
    // reading one while the next is written), or one for MX, whose scales take
    // the shared memory of the second (each chunk store then waits for the
    // previous one's reads; the stores of a tile are paced 1 us apart anyway).
    static constexpr uint32_t EPI_BUFS = MX ? 1u : 2u;
    static constexpr uint32_t MN_ATOM_BYTES = 64u * 128u;              // MN-major: 64 K x 64 N
    // K-blocks per ring barrier.  The MMA warp pays a fixed cost per pass
    // (~200 cycles for the barrier wait, vote and fence, ~50 for the commit)
    // on top of ~70 cycles per MMA issued; a 1-CTA tile of at most 128
    // columns has only 256 tensor cycles per k-block to hide it in, so its
    // stages go in pairs: one full and one empty barrier per pair, one wait
    // and one commit per two k-blocks.  2-CTA and wider tiles are tensor-bound
    // with one k-block per pass.
    static constexpr int G = (CG == 1 && CONS == 1 && !MX && BN <= 128) ? 2 : 1;
    static constexpr int GROUPS = STAGES / G;  // ring barrier pairs (full, empty)

    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    // (the epilogue staging is 128-byte swizzled: 1 KiB aligned)
    static constexpr uint32_t OFF_EPI = (OFF_SFB + STAGES * SFB_BYTES + 1023u) & ~1023u;
    static constexpr uint32_t OFF_BAR = OFF_EPI + kEpilogueWarps * EPI_BUFS * EPI_BUF_BYTES;
    // full[GROUPS], empty[GROUPS], acc_full[2], acc_empty[2], one per epilogue
    // warp; with KS > 1 also go[4] (every other CTA's ring may receive) and
    // done[4] (every other CTA's piece has arrived), one per lane quarter
    static constexpr uint32_t NUM_BARS = 2u * GROUPS + 4u + kEpilogueWarps + (KS > 1 ? 8u : 0u);
    // Split-tail fix-up: in a cluster's last unit the ring is idle, and each
    // epilogue warp may use RING_BYTES / 4 of it for partial pieces of 8 KiB
    // (32 rows x 64 FP32 columns).
    static constexpr uint32_t RING_BYTES = STAGES * (A_BYTES + B_BYTES);
    static constexpr uint32_t PIECE_BYTES = 32u * 64u * 4u;
    static constexpr uint32_t PIECES_PER_WARP = (RING_BYTES / kEpilogueWarps) / PIECE_BYTES;
    static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8u;
    static constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4u;
    static constexpr uint32_t SMEM_USED = OFF_ABORT + 4u;
    static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024u;  // slack to align the base

    // tcgen05 instruction descriptor (one layout for kind::f16 and
    // kind::f8f6f4): D = F32 (bits 4-5 = 1), the A / B type at bits 7-9 /
    // 10-12 (kind::f16: F16 = 0, BF16 = 1; kind::f8f6f4: E4M3 = 0, E5M2 = 1),
    // A K-major (bit 15 = 0), B major at bit 16, N >> 3 at bits 17-22, M >> 4
    // at bits 24-28.  MMA shape (the same whatever the number of consumers):
    // M = 128 rows per CTA of the group, N = BN.
    static constexpr int MMA_M = 128 * CG;
    static constexpr uint32_t AB_TYPE = F8 ? uint32_t(F8 - 1) : (BF16 ? 1u : 0u);
    static constexpr uint32_t IDESC = (1u << 4) | (AB_TYPE << 7) | (AB_TYPE << 10) |
                                      ((B_MN ? 1u : 0u) << 16) | (uint32_t(BN >> 3) << 17) |
                                      (uint32_t(MMA_M >> 4) << 24);
    // Block-scaled (kind::mxf8f6f4) descriptor: no D-type field (D is F32);
    // bits 4-5 and 29-30 carry the B and A scale ids (the byte of each 32-bit
    // TMEM scale cell: the 32-element K group within the k-block), added per
    // MMA; bit 23 = 1 selects UE8M0 scales.
    static constexpr uint32_t IDESC_MX = (AB_TYPE << 7) | (AB_TYPE << 10) | (uint32_t(BN >> 3) << 17) |
                                         (1u << 23) | (uint32_t(MMA_M >> 4) << 24);
    // MX scale factors in TMEM: two buffers, each in the 32 columns after one
    // accumulator's 224: buffer b holds the A scales at column 256 b + 224 (4
    // columns) and the B scales at 256 b + 240 (8 columns); every scale address
    // is a multiple of 16 columns.
    static constexpr uint32_t SF_COL = 224u;
    static_assert(F8 == 0 || F8 == 1 || F8 == 2, "FP8 input: none, E4M3 or E5M2");
    static_assert(!(F8 && B_MN), "FP8 operands are K-major (A.Bt only)");
    static_assert(BK * ELEM_BYTES == 128 && MMA_K * ELEM_BYTES == 32,
                  "a stage row is one 128-byte swizzle row; an MMA consumes 32 bytes of it");
    static_assert(MMA_M == 128 || MMA_M == 256, "tcgen05 kind::f16 M is 128 (1 CTA) or 256 (2 CTAs)");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "tcgen05 kind::f16 N is a multiple of 16, <= 256");
    static_assert(((IDESC >> 24) & 0x1Fu) == uint32_t(MMA_M >> 4) && ((IDESC >> 17) & 0x3Fu) == uint32_t(BN >> 3),
                  "instruction descriptor fields in range");

    static_assert(CG == 1 || CG == 2, "cta_group is 1 or 2");
    static_assert(BN == 32 || BN == 64 || (BN % 32 == 0 && BN >= 128 && BN <= 256),
                  "tile N is 32, 64 or a multiple of 32 in [128, 256]");
    static_assert(BN >= 128 || (CG == 1 && CONS == 1 && !MX), "32- and 64-wide tiles: 1 CTA, 1 consumer");
    static_assert((BN / CG) % 16 == 0, "each CTA's share of B is whole 16-row SW128 groups");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation is a power of two");
    static_assert(CONS == 1 || CONS == 2, "one or two MMA consumers");
    static_assert(STAGES % G == 0 && GROUPS >= 2, "whole groups of stages, at least two");
    static_assert(CONS * (FULL_CHUNKS + (HALF_CHUNK ? 1 : 0)) * EPI_BUF_BYTES <=
                      PIECES_PER_WARP * PIECE_BYTES,
                  "the last unit's epilogue chunks fit in each warp's share of the ring");
    static_assert(!B_MN || (B_ROWS % 64) == 0, "MN-major B is loaded in 64-column atoms");
    static_assert(SMEM_BYTES <= 232448, "exceeds 227 KiB of shared memory per CTA");
    // In-cluster K split: each other CTA's piece of a lane quarter (32 rows x
    // BN / KS FP32 columns) lands in a slice of its own in the owner's shared
    // memory.  The first RECV_STG_SLOTS of a quarter's KS - 1 pieces go into the
    // epilogue staging buffers of that quarter's warp (idle until the epilogue,
    // which then stages its own output in the ring, at OFF_KS_OUT), so they
    // need no hand-shake; the rest go into the operand ring, once its owner
    // has said that its MMAs are done.
    static constexpr uint32_t RECV_SLICE_BYTES = 32u * uint32_t(BN / KS) * 4u;
    static constexpr uint32_t RECV_STG_SLOTS = (KS > 1) ? (EPI_BUFS * EPI_BUF_BYTES) / RECV_SLICE_BYTES : 0u;
    static constexpr uint32_t RECV_RING_SLOTS =
        (uint32_t(KS - 1) > RECV_STG_SLOTS) ? uint32_t(KS - 1) - RECV_STG_SLOTS : 0u;
    static constexpr uint32_t OFF_KS_OUT = OFF_A + ((RECV_RING_SLOTS * 4u * RECV_SLICE_BYTES + 1023u) & ~1023u);
    // ... and the pieces a CTA sends are staged in its own ring first, each
    // slot's piece leaving as one bulk copy
    static constexpr uint32_t OFF_KS_SEND = OFF_KS_OUT + uint32_t(kEpilogueWarps) * 2u * EPI_BUF_BYTES;
    static_assert(KS == 1 || KS == 2 || KS == 4, "1, 2 or 4 K-ranges per cluster");
    static_assert(KS == 1 || (CG == 1 && CONS == 1 && !MX), "in-cluster K split: 1-CTA, 1-consumer tiles");
    static_assert(KS == 1 || OFF_KS_SEND + uint32_t(KS - 1) * 4u * RECV_SLICE_BYTES <= OFF_A + RING_BYTES,
                  "the pieces the ring receives, the output staging and the sent pieces fit in the ring");
    static_assert(KS == 1 || (BN / KS) % 32 == 0, "each CTA owns whole 32-column units");
    // the epilogue stores 32-column boxes (the last chunk of a 224-wide tile,
    // or a CTA's share of a 128-wide tile split 4 ways)
    static constexpr bool D32 = HALF_CHUNK || (KS > 1 && BN / KS == 32);
    static_assert(!MX || (F8 && BN == 224 && CONS == 1 && !B_MN && ACC_STRIDE == 256 &&
                          NUM_ACC == 2 && BK == 128),
                  "MX: FP8 A.Bt, 224-wide tiles (224 accumulator + 32 scale columns per buffer)");
    static_assert((A_BYTES % 1024) == 0 && (B_BYTES % 1024) == 0, "SW128 atoms are 1 KiB");
    static_assert((OFF_EPI % 1024) == 0 && (OFF_SFA % 512) == 0 && (OFF_SFB % 512) == 0,
                  "swizzled staging 1 KiB aligned; scale buffers aligned for TMA and tcgen05.cp");
};

struct GemmArgs {
    int32_t M, N, K;
    int32_t k_blocks;   // ceil(K / BK)
    float alpha;        // FP8 inputs: D = alpha * (A . Bt) (unused for 16-bit inputs)
    TileGrid grid;
    // Work units.  Units [0, whole_units) are whole tiles (unit u = tile u).
    // The remaining tiles ("tail" tiles, the last partial round of the
    // persistent schedule) are each split into `split` K-ranges, one unit per
    // range, so that clusters that would idle in that round share the work.
    int64_t whole_units;
    int32_t split;      // K-ranges per tail tile; 1 = no split
    uint32_t epoch;     // tag of this launch for the tail counters
    float* partials;    // split > 1: FP32 partial of each (tail tile, range, CTA, warp quarter)
    unsigned long long* counters;  // split > 1: one per (tail tile, CTA, warp quarter)
    uint64_t wait_limit_ns;        // limit of every barrier wait (kWaitLimitNs unless a self-test)
    uint32_t l2_hints;             // kHint* bits: L2 eviction priorities (0 = none)
    // Diagnostic (null normally): CTA 0 writes its SM clock counter and the
    // global nanosecond timer at its start ([0], [1]) and end ([2], [3]).
    unsigned long long* clock_probe;
};

struct WorkUnit {
    int64_t tile;    // task index of the tile in the scheduler order
    int32_t kb0;     // first k-block
    int32_t kb1;     // one past the last k-block
    int32_t range;   // K-range index of a tail tile, -1 for a whole tile
    int64_t tail;    // index of the tail tile, -1 for a whole tile
};

__host__ __device__ __forceinline__ int64_t unit_count(const GemmArgs& a) {
    return a.whole_units + (tile_count(a.grid) - a.whole_units) * a.split;
}

__host__ __device__ __forceinline__ WorkUnit unit_of(const GemmArgs& a, int64_t u) {
    WorkUnit w;
    if (u < a.whole_units) {
        w.tile = u;
        w.kb0 = 0;
        w.kb1 = a.k_blocks;
        w.range = -1;
        w.tail = -1;
    } else {
        // 32-bit arithmetic (unit counts are below 2^31; see kMaxTiles)
        const uint32_t v = uint32_t(u - a.whole_units), split = uint32_t(a.split);
        const uint32_t tail = v / split;
        w.tail = tail;
        w.range = int32_t(v - tail * split);
        w.tile = a.whole_units + tail;
        w.kb0 = int32_t((uint32_t(w.range) * uint32_t(a.k_blocks)) / split);
        w.kb1 = int32_t((uint32_t(w.range + 1) * uint32_t(a.k_blocks)) / split);
    }
    return w;
}

// The k-blocks of unit w that CTA `krank` of a cluster computes: all of them,
// or with an in-cluster K split (KS > 1) the krank-th of KS ranges.
template <int KS>
__device__ __forceinline__ void kb_range(const WorkUnit& w, uint32_t krank, int& kb0, int& kb1) {
    if constexpr (KS == 1) {
        kb0 = w.kb0;
        kb1 = w.kb1;
    } else {
        const int n = w.kb1 - w.kb0;
        kb0 = w.kb0 + int(krank) * n / KS;
        kb1 = w.kb0 + int(krank + 1u) * n / KS;
    }
}

// tcgen05 shared-memory matrix descriptor for a 128-byte-swizzled operand:
// start address >> 4 (bits 0-13), leading-dimension byte offset >> 4 (16-29),
// stride-dimension byte offset >> 4 (32-45), the fixed version value 1 at bits
// 46-48, base offset 0 (atoms are 1 KiB aligned), swizzle mode 2 = 128 B at
// bits 61-63.
//   K-major (A, and B of A.B^T): rows of 128 B = 64 K elements; SBO = 1 KiB
//     between groups of 8 rows; LBO unused (one MMA reads 32 B of K, inside
//     the swizzle row).  The k-th K=16 slice starts 32 B further.
//   MN-major (B of A.B): rows of 128 B = 64 N elements, one row per k; SBO =
//     1 KiB between groups of 8 k rows; LBO = 8 KiB between 64-column atoms.
//     The k-th K=16 slice starts 16 rows = 2 KiB further.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = uint64_t((addr & 0x3FFFFu) >> 4);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}

// tcgen05 shared-memory descriptor without swizzling (the scale-factor
// copies): core matrices of 8 rows x 16 B stored contiguously; LBO = byte
// distance between the two 16-byte halves of a 32-byte row, SBO = byte
// distance between groups of 8 rows.
__device__ __forceinline__ uint64_t noswizzle_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = uint64_t((addr & 0x3FFFFu) >> 4);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;
    return d;
}

// A CTA's abort state in a cluster of N CTAs: its flag (in its shared memory,
// polled by every role; `flag_addr` is its shared::cta address, the same
// offset in every CTA of the cluster), this CTA's rank in the cluster, and the
// limit of every wait.  N is a template parameter so that the waits inlined
// into the hot loops carry no loop over ranks for 1- and 2-CTA clusters.
template <int N>
struct AbortCtl {
    volatile uint32_t* flag;
    uint32_t flag_addr;
    uint32_t my_rank;
    uint64_t limit_ns;
};

// Record the reason and raise the flag in every CTA of the cluster: a role of
// another CTA may be the one that would wait for this CTA's work, and every
// warp that sees the flag settles before it leaves (see the teardown).
template <int N>
__device__ __forceinline__ void raise_abort(const AbortCtl<N>& ac, uint32_t role) {
    *ac.flag = 1u;
    if constexpr (N == 2) {
        ptx::st_cluster_u32(ptx::map_to_rank(ac.flag_addr, ac.my_rank ^ 1u), 1u);
    } else if constexpr (N > 2) {
#pragma unroll
        for (uint32_t r = 0; r < uint32_t(N); ++r)
            if (r != ac.my_rank) ptx::st_cluster_u32(ptx::map_to_rank(ac.flag_addr, r), 1u);
    }
    atomicCAS(&g_gemm_status, 0u, kReasonTimeout | (role << 8));
}

// Wait for phase `parity` of `bar`, giving up after ac.limit_ns or when a role
// of this CTA or of another CTA of its cluster has aborted.  Returns false on
// give-up.  (Kept inline: a wait's slow path is common in the hot loops, and
// moving it out of line measured 4-6 % slower on the 2-CTA plans.)
template <int N>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const AbortCtl<N>& ac,
                                             uint32_t role) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 7u) == 0u) {
            if (*ac.flag) return false;
            if (ptx::global_timer_ns() - t0 > ac.limit_ns) {
                raise_abort(ac, role);
                return false;
            }
        }
    }
}

// wait_bounded for a whole converged warp: every lane waits (and acquires), and
// all lanes return the same result.
template <int N>
__device__ __forceinline__ bool wait_bounded_warp(uint32_t bar, uint32_t parity, const AbortCtl<N>& ac,
                                                  uint32_t role) {
    const bool ok = wait_bounded(bar, parity, ac, role);
    return __all_sync(0xffffffffu, ok);
}

// After an abort: give in-flight asynchronous copies, MMAs and their barrier
// arrivals (which complete in microseconds) time to land before shared memory
// and TMEM are released.
__device__ __forceinline__ void settle_after_abort() {
    const uint64_t t0 = ptx::global_timer_ns();
    while (ptx::global_timer_ns() - t0 < 1000000ull) __nanosleep(10000);
}

// For a converged warp at the end of its role: if this CTA's abort flag is
// up, settle (the whole warp takes one decision, read by lane 0).
template <int N>
__device__ __forceinline__ void settle_if_aborted(const AbortCtl<N>& ac) {
    const uint32_t up = __shfl_sync(0xffffffffu, *ac.flag, 0);
    if (up) settle_after_abort();
    __syncwarp();
}

// Count one finished K-range of a tail tile.  The counter word holds
// (epoch << 32 | count); a word tagged with another launch's epoch counts as
// zero, and the range that finishes last resets the word to zero, so the
// workspace never needs clearing between launches (nor between replays of a
// captured launch, which repeat its epoch).  Returns the
// number of ranges counted before this one (split - 1 means "this was the
// last").  No thread ever waits for another here.
__device__ __forceinline__ uint32_t count_range_done(unsigned long long* word, uint32_t epoch) {
    unsigned long long old = atomicAdd(word, 0ull);
    for (int i = 0; i < (1 << 20); ++i) {
        const uint32_t cnt = (uint32_t(old >> 32) == epoch) ? uint32_t(old) : 0u;
        const unsigned long long want = (static_cast<unsigned long long>(epoch) << 32) | (cnt + 1u);
        const unsigned long long seen = atomicCAS(word, old, want);
        if (seen == old) return cnt;
        old = seen;
    }
    atomicCAS(&g_gemm_status, 0u, kReasonCounter);
    return 0xFFFFFFFFu;
}

template <class C>
__global__ void __launch_bounds__(kNumThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_d, const GemmArgs args,
                        const __grid_constant__ CUtensorMap tmap_sa,
                        const __grid_constant__ CUtensorMap tmap_sb,
                        const __grid_constant__ CUtensorMap tmap_d32) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (args.clock_probe && blockIdx.x == 0 && threadIdx.x == 0) {
        args.clock_probe[0] = clock64();
        args.clock_probe[1] = ptx::global_timer_ns();
    }
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    const uint32_t warp = __shfl_sync(0xffffffffu, threadIdx.x / 32u, 0);
    const uint32_t lane = threadIdx.x % 32u;
    const uint32_t crank = (C::CLUSTER > 1) ? ptx::cluster_ctarank() : 0u;
    const uint32_t rank = crank % uint32_t(C::CG);   // CTA within its MMA pair
    const uint32_t krank = crank / uint32_t(C::CG);  // K-range of the tile (KS > 1)
    const bool leader = (rank == 0u);
    const int64_t cluster_id = blockIdx.x / C::CLUSTER;
    const int64_t num_clusters = gridDim.x / C::CLUSTER;
    const int64_t units = unit_count(args);

    // Ring barriers, one pair per group of C::G stages (g = stage / C::G).
    auto full_bar = [&](uint32_t g) { return base + C::OFF_BAR + 8u * g; };
    auto empty_bar = [&](uint32_t g) { return base + C::OFF_BAR + 8u * (C::GROUPS + g); };
    auto acc_full_bar = [&](uint32_t b) { return base + C::OFF_BAR + 8u * (2u * C::GROUPS + b); };
    auto acc_empty_bar = [&](uint32_t b) {
        return base + C::OFF_BAR + 8u * (2u * C::GROUPS + 2u + b);
    };
    auto epi_bar = [&](uint32_t e) { return base + C::OFF_BAR + 8u * (2u * C::GROUPS + 4u + e); };
    auto go_bar = [&](uint32_t q) {
        return base + C::OFF_BAR + 8u * (2u * C::GROUPS + 4u + kEpilogueWarps + q);
    };
    auto done_bar = [&](uint32_t q) {
        return base + C::OFF_BAR + 8u * (2u * C::GROUPS + 8u + kEpilogueWarps + q);
    };
    volatile uint32_t* const abort_flag =
        reinterpret_cast<volatile uint32_t*>(base_ptr + C::OFF_ABORT);
    const AbortCtl<C::CLUSTER> ac{abort_flag, base + C::OFF_ABORT, crank,
                      args.wait_limit_ns};

    // ---- one-time setup -------------------------------------------------
    if (warp == 0 && lane == 0) {
        for (uint32_t g = 0; g < uint32_t(C::GROUPS); ++g) {
            ptx::mbar_init(full_bar(g), 1);   // the leader's expect_tx arrival
            ptx::mbar_init(empty_bar(g), 1);  // the pair's one tcgen05.commit
        }
        for (uint32_t b = 0; b < 2; ++b) {
            ptx::mbar_init(acc_full_bar(b), 1);                                  // one commit
            ptx::mbar_init(acc_empty_bar(b), uint32_t(C::CG * kEpilogueWarps));  // all epilogue warps
        }
        for (uint32_t e = 0; e < uint32_t(kEpilogueWarps); ++e) ptx::mbar_init(epi_bar(e), 1);
        if constexpr (C::KS > 1) {
            for (uint32_t q = 0; q < 4u; ++q) {
                ptx::mbar_init(go_bar(q), uint32_t(C::KS - 1));  // each other CTA's warp q
                ptx::mbar_init(done_bar(q), 1);  // warp q's expect_tx; the pieces complete its bytes
            }
        }
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(&tmap_a);
        ptx::prefetch_tensormap(&tmap_b);
        ptx::prefetch_tensormap(&tmap_d);
        if constexpr (C::D32) ptx::prefetch_tensormap(&tmap_d32);
        if constexpr (C::MX) {
            ptx::prefetch_tensormap(&tmap_sa);
            ptx::prefetch_tensormap(&tmap_sb);
        }
    }
    if (warp == 0) __syncwarp();  // lane 0's barrier set-up, for the whole producer warp
    if (warp == 1) {
        ptx::tmem_alloc<C::CG>(base + C::OFF_TMEM_SLOT, C::TMEM_COLS);
        ptx::tmem_relinquish<C::CG>();
    }
    // Prologue barrier, split in two: every thread arrives once this CTA's
    // barriers are initialised and its TMEM is allocated, and waits before it
    // uses either.  The producer of a CTA whose loads complete on its own
    // barriers (a CTA alone, or the leader of a pair) needs neither TMEM nor
    // the other CTA, so it does not wait: its first loads leave while TMEM is
    // allocated and the pair meets.  (With a pair it completes its wait at the
    // end of its role: a thread waits once for each cluster barrier phase
    // before it arrives on the next.)
    const bool early_producer = (warp == 0) && (C::CLUSTER == 1 || leader);
    ptx::tc_fence_before();
    if constexpr (C::CLUSTER > 1) {
        ptx::cluster_arrive();
        if (!early_producer) ptx::cluster_wait();
    } else {
        if (early_producer) ptx::named_bar_arrive(1, kNumThreads);
        else ptx::named_bar_sync(1, kNumThreads);
    }
    ptx::tc_fence_after();
    // (the producer never touches TMEM)
    const uint32_t tmem_base =
        (warp == 0) ? 0u : *reinterpret_cast<volatile uint32_t*>(base_ptr + C::OFF_TMEM_SLOT);

    // The producer and the MMA issuer are warp roles whose loops run on the whole
    // warp, with one elected lane issuing each TMA copy, MMA and commit ("TIRx: A
    // Unified Tile Primitive ML Compiler", Figure 3: elect_sync() picks the issuing
    // thread; "TIRx GEMM on Blackwell": one elected thread submits a tcgen05 MMA).
    // Every value the loop computes is then warp-uniform.  With the loop confined
    // to one lane instead, the issuer needed ~535 cycles per k-block (4 MMAs, a
    // barrier wait and a commit): more than the 512 tensor cycles of a 256-wide
    // k-block.
    if (warp == 0) {
        // ---- TMA producer ---------------------------------------------------
        // Optional L2 eviction priorities: A evict_last keeps the band of A
        // rows that a raster group reuses; B evict_first lets the streamed
        // operand leave L2 first.
        const bool hinted = (args.l2_hints & (kHintALast | kHintBFirst)) != 0u;
        uint64_t pol_a = 0, pol_b = 0;
        if (hinted) {
            pol_a = (args.l2_hints & kHintALast) ? ptx::l2_policy_evict_last() : ptx::l2_policy_evict_normal();
            pol_b = (args.l2_hints & kHintBFirst) ? ptx::l2_policy_evict_first() : ptx::l2_policy_evict_normal();
        }
        // One operand box into this CTA's shared memory; with CG == 2 the
        // completion goes to the leader's full barrier.
        auto load = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x, int32_t y,
                        uint64_t pol) {
            if constexpr (C::CG == 1) {
                if (hinted) ptx::tma_load_2d_hint(dst, map, bar, x, y, pol);
                else ptx::tma_load_2d(dst, map, bar, x, y);
            } else {
                if (hinted) ptx::tma_load_2d_pair_hint(dst, map, bar, x, y, pol);
                else ptx::tma_load_2d_pair(dst, map, bar, x, y);
            }
        };
        uint32_t g = 0, ph = 0;  // ring group and its phase
        bool ok = true;
        for (int64_t u = cluster_id; u < units && ok; u += num_clusters) {
            const WorkUnit w = unit_of(args, u);
            int32_t mt, nt;
            tile_of_task(args.grid, w.tile, mt, nt);
            const int32_t a_row = mt * C::BM + int32_t(rank) * C::A_ROWS;
            const int32_t b_row = nt * C::BN + int32_t(rank) * C::B_ROWS;
            int kr0, kr1;
            kb_range<C::KS>(w, krank, kr0, kr1);
            // Group by group: k-blocks kb .. kb + n - 1 into the group's stages
            // (n < G only for the last group of a unit with an odd count).
            for (int kb = kr0; kb < kr1; kb += C::G) {
                // (a compile-time 1 with one k-block per group: the 2-CTA loops
                // have no cycles to spare)
                const int n = (C::G == 1) ? 1 : ((kr1 - kb < C::G) ? kr1 - kb : C::G);
                if (!wait_bounded_warp(empty_bar(g), ph ^ 1u, ac, kRoleProducer)) {
                    ok = false;
                    break;
                }
                if (ptx::elect_one_sync()) {
                    if (leader) ptx::mbar_arrive_expect_tx(full_bar(g), C::G == 1 ? C::STAGE_TX : uint32_t(n) * C::STAGE_TX);
                    // the leader's barrier (a shared::cluster address) for a pair
                    const uint32_t fb = (C::CG == 1) ? full_bar(g) : ptx::map_to_rank(full_bar(g), 0u);
#pragma unroll
                    for (int j = 0; j < C::G; ++j) {
                        if (j >= n) break;
                        const uint32_t s = g * uint32_t(C::G) + uint32_t(j);
                        const uint32_t a_dst = base + C::OFF_A + s * C::A_BYTES;
                        const uint32_t b_dst = base + C::OFF_B + s * C::B_BYTES;
                        const int32_t k0 = (kb + j) * C::BK;
                        load(a_dst, &tmap_a, fb, k0, a_row, pol_a);
                        if constexpr (!C::B_MN) {
                            load(b_dst, &tmap_b, fb, k0, b_row, pol_b);
                        } else {
#pragma unroll
                            for (int c = 0; c < C::B_ROWS / 64; ++c)
                                load(b_dst + c * C::MN_ATOM_BYTES, &tmap_b, fb, b_row + 64 * c, k0, pol_b);
                        }
                        if constexpr (C::MX) {
                            // The scales of k-block kb, into this CTA's shared memory,
                            // completing with the operands: the A atom of this CTA's 128
                            // rows (128 rows x 4 groups) and the tile's B block (the
                            // image of its TMEM copy; both CTAs of a pair load it).
                            const uint32_t sfa_dst = base + C::OFF_SFA + s * C::SFA_BYTES;
                            const uint32_t sfb_dst = base + C::OFF_SFB + s * C::SFB_BYTES;
                            const int32_t sfb_block = nt * args.k_blocks + kb + j;
                            if constexpr (C::CG == 1) {
                                ptx::tma_load_2d(sfa_dst, &tmap_sa, fb, (kb + j) * 128, a_row / 128);
                                ptx::tma_load_2d(sfb_dst, &tmap_sb, fb, 0, sfb_block * 4);
                            } else {
                                ptx::tma_load_2d_pair(sfa_dst, &tmap_sa, fb, (kb + j) * 128, a_row / 128);
                                ptx::tma_load_2d_pair(sfb_dst, &tmap_sb, fb, 0, sfb_block * 4);
                            }
                        }
                    }
                }
                __syncwarp();
                if (++g == uint32_t(C::GROUPS)) { g = 0; ph ^= 1u; }
            }
        }
        if (ok) {
            // Drain: every group must have been released by the MMA, so no
            // tcgen05.commit arrives on this CTA's barriers after it exits.
            for (int i = 0; i < C::GROUPS; ++i) {
                if (!wait_bounded_warp(empty_bar(g), ph ^ 1u, ac, kRoleDrain)) {
                    ok = false;
                    break;
                }
                if (++g == uint32_t(C::GROUPS)) { g = 0; ph ^= 1u; }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer (leader CTA) ------------------------------------------
        if constexpr (C::CONS == 2) {
          if (leader) {
            // Two consumers ("TIRx GEMM on Blackwell", V9): their accumulators
            // fill TMEM, so the next tile's MMAs can only start once the
            // epilogue has drained them.  Each consumer has its own full and
            // empty accumulator barrier (acc_full[h], acc_empty[h]), and the
            // tile is issued so that the drains overlap MMAs: consumer 0 runs
            // alone over the tile's first k-blocks (up to one ring), keeping
            // their stages, while consumer 1 is still being drained; consumer 1
            // catches up on those stages; the middle issues both consumers per
            // k-block as one B tile serves both; and the last k-blocks (up to
            // one ring) go to consumer 0 first, so that its accumulator is
            // complete and drained while consumer 1 finishes them.
            uint32_t s = 0, ph = 0, aph = 0;
            bool ok = true;
            auto issue = [&](uint32_t st, int h, bool first_kb) {
                const uint32_t a_addr = base + C::OFF_A + st * C::A_BYTES + 16384u * uint32_t(h);
                const uint32_t b_addr = base + C::OFF_B + st * C::B_BYTES;
#pragma unroll
                for (int k = 0; k < C::BK / C::MMA_K; ++k) {
                    const uint64_t bd = C::B_MN ? sw128_desc(b_addr + 2048u * k, C::MN_ATOM_BYTES, 1024u)
                                                : sw128_desc(b_addr + 32u * k, 16u, 1024u);
                    const uint64_t ad = sw128_desc(a_addr + 32u * k, 16u, 1024u);
                    ptx::mma_f16<C::CG>(tmem_base + uint32_t(h) * C::ACC_STRIDE, ad, bd, C::IDESC,
                                        uint32_t(!first_kb || k != 0));
                }
            };
            for (int64_t u = cluster_id; u < units && ok; u += num_clusters) {
                const WorkUnit w = unit_of(args, u);
                const int nkb = w.kb1 - w.kb0;
                const int lead = nkb < C::STAGES ? nkb : C::STAGES;
                const int tail = (nkb - lead < C::STAGES) ? nkb - lead : C::STAGES;
                const uint32_t s0 = s;
                if (!wait_bounded_warp(acc_empty_bar(0), aph ^ 1u, ac, kRoleMma)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                for (int i = 0; i < lead; ++i) {  // consumer 0 alone; stages kept
                    if (!wait_bounded_warp(full_bar(s), ph, ac, kRoleMma)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (ptx::elect_one_sync()) issue(s, 0, i == 0);
                    __syncwarp();
                    if (++s == uint32_t(C::STAGES)) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if (tail == 0) {  // consumer 0 is complete
                    if (ptx::elect_one_sync()) ptx::mma_commit<C::CG>(acc_full_bar(0), uint16_t(0x3u));
                    __syncwarp();
                }
                if (!wait_bounded_warp(acc_empty_bar(1), aph ^ 1u, ac, kRoleMma)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                for (int i = 0; i < lead; ++i) {  // consumer 1 catches up, stages released
                    const uint32_t st = (s0 + uint32_t(i)) % uint32_t(C::STAGES);
                    if (ptx::elect_one_sync()) {
                        issue(st, 1, i == 0);
                        ptx::mma_commit<C::CG>(empty_bar(st), uint16_t(0x3u));
                    }
                    __syncwarp();
                }
                for (int i = lead; i < nkb - tail; ++i) {  // both consumers share each B tile
                    if (!wait_bounded_warp(full_bar(s), ph, ac, kRoleMma)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (ptx::elect_one_sync()) {
                        issue(s, 0, false);
                        issue(s, 1, false);
                        ptx::mma_commit<C::CG>(empty_bar(s), uint16_t(0x3u));
                    }
                    __syncwarp();
                    if (++s == uint32_t(C::STAGES)) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if (tail > 0) {
                    const uint32_t s1 = s;
                    for (int i = 0; i < tail; ++i) {  // consumer 0 finishes first; stages kept
                        if (!wait_bounded_warp(full_bar(s), ph, ac, kRoleMma)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        if (ptx::elect_one_sync()) issue(s, 0, false);
                        __syncwarp();
                        if (++s == uint32_t(C::STAGES)) { s = 0; ph ^= 1u; }
                    }
                    if (!ok) break;
                    if (ptx::elect_one_sync()) ptx::mma_commit<C::CG>(acc_full_bar(0), uint16_t(0x3u));
                    __syncwarp();
                    for (int i = 0; i < tail; ++i) {  // consumer 1 on the same stages, released
                        const uint32_t st = (s1 + uint32_t(i)) % uint32_t(C::STAGES);
                        if (ptx::elect_one_sync()) {
                            issue(st, 1, false);
                            ptx::mma_commit<C::CG>(empty_bar(st), uint16_t(0x3u));
                        }
                        __syncwarp();
                    }
                }
                if (ptx::elect_one_sync())
                    ptx::mma_commit<C::CG>(acc_full_bar(1), uint16_t(0x3u));  // consumer 1 is complete
                __syncwarp();
                aph ^= 1u;
            }
            // No drain: the epilogue hands back every accumulator but those of
            // the cluster's last unit, and this loop waited for each hand-back.
          }
        } else if (leader) {
            uint32_t g = 0, ph = 0, ab = 0, aph = 0;  // ring group and its phase
            uint32_t sfbuf = 0;  // MX: TMEM scale buffer of the next k-block
            bool ok = true;
            for (int64_t u = cluster_id; u < units && ok; u += num_clusters) {
                const WorkUnit w = unit_of(args, u);
                if (!wait_bounded_warp(acc_empty_bar(ab), aph ^ 1u, ac, kRoleMma)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + ab * C::SLOT_COLS;
                // One k-block's MMAs from stage st (with MX, after its scale
                // copies into TMEM buffer sfb).
                auto issue_kblock = [&](uint32_t st, uint32_t sfb, bool first) {
                    const uint32_t a_addr = base + C::OFF_A + st * C::A_BYTES;
                    const uint32_t b_addr = base + C::OFF_B + st * C::B_BYTES;
                    const uint32_t sf_t = tmem_base + (sfb << 8) + C::SF_COL;
                    if constexpr (C::MX) {
                        // This k-block's scales into TMEM (each CTA of the pair
                        // from its own shared memory), ordered before the MMAs
                        // below, which read them.
                        ptx::tmem_cp_32x128b_warpx4<C::CG>(
                            sf_t, noswizzle_desc(base + C::OFF_SFA + st * C::SFA_BYTES, 128u, 128u));
                        ptx::tmem_cp_128x256b<C::CG>(
                            sf_t + 16u, noswizzle_desc(base + C::OFF_SFB + st * C::SFB_BYTES, 128u, 256u));
                    }
#pragma unroll
                    for (int k = 0; k < C::BK / C::MMA_K; ++k) {
                        const uint64_t bd = C::B_MN ? sw128_desc(b_addr + 2048u * k, C::MN_ATOM_BYTES, 1024u)
                                                    : sw128_desc(b_addr + 32u * k, 16u, 1024u);
                        const uint64_t ad = sw128_desc(a_addr + 32u * k, 16u, 1024u);
                        const uint32_t acc = uint32_t(!first || k != 0);
                        if constexpr (C::MX)
                            ptx::mma_mxf8f6f4<C::CG>(d_tmem, ad, bd,
                                                     C::IDESC_MX | (uint32_t(k) << 4) | (uint32_t(k) << 29),
                                                     sf_t, sf_t + 16u, acc);
                        else if constexpr (C::F8)
                            ptx::mma_f8f6f4<C::CG>(d_tmem, ad, bd, C::IDESC, acc);
                        else
                            ptx::mma_f16<C::CG>(d_tmem, ad, bd, C::IDESC, acc);
                    }
                };
                // One group of C::G k-blocks per pass: one wait, the group's
                // MMAs, one commit that frees the group's stages (in every CTA
                // that received data for them) once those MMAs finish.  With
                // one k-block per pass a 2-CTA 224-wide k-block takes ~448-508
                // cycles, at or near its 448 tensor cycles, and pairing its
                // stages measured no faster; a 1-CTA 128-wide k-block (256
                // tensor cycles) took ~515.
                int kr0, kr1;
                kb_range<C::KS>(w, krank, kr0, kr1);
                for (int kb = kr0; kb < kr1; kb += C::G) {
                    const int n = (C::G == 1) ? 1 : ((kr1 - kb < C::G) ? kr1 - kb : C::G);
                    if (!wait_bounded_warp(full_bar(g), ph, ac, kRoleMma)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (ptx::elect_one_sync()) {
#pragma unroll
                        for (int j = 0; j < C::G; ++j)
                            if (j < n)
                                issue_kblock(g * uint32_t(C::G) + uint32_t(j), sfbuf ^ uint32_t(j & 1),
                                             kb + j == kr0);
                        ptx::mma_commit<C::CG>(empty_bar(g), uint16_t(0x3u));
                    }
                    __syncwarp();
                    sfbuf ^= uint32_t(n & 1);
                    if (++g == uint32_t(C::GROUPS)) { g = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if (ptx::elect_one_sync())
                    ptx::mma_commit<C::CG>(acc_full_bar(ab), uint16_t(0x3u));  // accumulator ready
                __syncwarp();
                if (++ab == C::NUM_ACC) { ab = 0; aph ^= 1u; }
            }
            if (ok) {
                // Drain: every accumulator slot released by every epilogue warp of
                // the cluster (the peer's arrivals target this CTA's barriers),
                // except the slot of the cluster's last unit, which the epilogue
                // keeps (its release would be the last arrival of the launch).
                for (uint32_t i = 0; i + 1 < C::NUM_ACC; ++i) {
                    if (!wait_bounded_warp(acc_empty_bar(ab), aph ^ 1u, ac, kRoleDrain)) {
                        ok = false;
                        break;
                    }
                    if (++ab == C::NUM_ACC) { ab = 0; aph ^= 1u; }
                }
            }
        }
        __syncwarp();
    } else {
        // ---- epilogue warps 2..5 ----------------------------------------------
        const uint32_t quarter = warp & 3u;  // this warp may read TMEM lanes 32q..32q+31
        const uint32_t buf0 = base + C::OFF_EPI + (warp - 2u) * C::EPI_BUFS * C::EPI_BUF_BYTES;
        const uint32_t my_epi_bar = epi_bar(warp - 2u);
        const uint32_t my_ring = base + C::OFF_A + (warp - 2u) * C::PIECES_PER_WARP * C::PIECE_BYTES;
        uint32_t ab = 0, aph = 0, chunk = 0, eph = 0;
        uint32_t gph = 0, dph = 0;  // in-cluster K split: go / done phases

        // Hand accumulator `b` back to the MMA issuer (all TMEM reads done).
        auto release_acc = [&](uint32_t b) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (C::CG == 2)
                    ptx::mbar_arrive_cluster(ptx::map_to_rank(acc_empty_bar(b), 0u));
                else
                    ptx::mbar_arrive(acc_empty_bar(b));
            }
        };
        // W = 64 (or 32, the last chunk of a 224-wide tile) FP32 values of this
        // lane's row -> 16-bit -> swizzled staging -> TMA store of the warp's
        // 32 x W box at (col, row0), which clips rows and columns outside D.
        // Staging alternates between the warp's buffers, or (in a cluster's last
        // unit, when the ring is idle) takes a fresh 4 KiB slice of the ring per
        // chunk, which never waits for an earlier store.
        // FP8 inputs: D = alpha * (A . Bt), applied to the FP32 sum before the
        // one rounding to 16 bits.
        const float alpha = args.alpha;
        const bool hint_d = (args.l2_hints & kHintDFirst) != 0u;
        const uint64_t pol_d = hint_d ? ptx::l2_policy_evict_first() : 0ull;
        auto scaled = [&](float x) -> float {
            if constexpr (C::F8) return x * alpha; else return x;
        };
        // The whole-tile epilogue's steps, 32 columns at a time (see there):
        // pick the staging buffer of the next chunk (waiting until the store
        // EPI_BUFS chunks ago has read it, unless the ring slice is used) ...
        auto stage_buffer = [&](int32_t ring_slot) -> uint32_t {
            uint32_t b;
            if (ring_slot >= 0) {
                b = my_ring + uint32_t(ring_slot) * C::EPI_BUF_BYTES;
            } else {
                b = buf0 + (chunk % C::EPI_BUFS) * C::EPI_BUF_BYTES;
                if (lane == 0) ptx::bulk_wait_group_read<int(C::EPI_BUFS) - 1>();
            }
            __syncwarp();
            return b;
        };
        // ... convert 32 FP32 values of this lane's row and store them as half
        // `half` of its row in the staging tile (W = 64: 128-byte rows, 128-byte
        // swizzle; W = 32: 64-byte rows, 64-byte swizzle, half 0 only) ...
        auto stage_half = [&](const uint32_t (&v)[32], uint32_t b, int W, int half) {
            const uint32_t row_addr = b + lane * uint32_t(2 * W);
            const uint32_t sw = (W == 64) ? (lane & 7u) : ((lane >> 1) & 3u);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                auto f = [&](int i) { return scaled(__uint_as_float(v[8 * q + i])); };
                const uint32_t p0 = ptx::pack2<C::BF16>(f(0), f(1));
                const uint32_t p1 = ptx::pack2<C::BF16>(f(2), f(3));
                const uint32_t p2 = ptx::pack2<C::BF16>(f(4), f(5));
                const uint32_t p3 = ptx::pack2<C::BF16>(f(6), f(7));
                ptx::st_shared_v4(row_addr + ((uint32_t(4 * half + q) ^ sw) << 4), p0, p1, p2, p3);
            }
        };
        // ... and send the staged 32 x W box to D.
        auto issue_store = [&](uint32_t b, int32_t col, int32_t row0, int W) {
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (row0 < args.M && col < args.N) {
                    const CUtensorMap* map = (W == 64) ? &tmap_d : &tmap_d32;
                    if (hint_d) ptx::tma_store_2d_hint(map, b, col, row0, pol_d);
                    else ptx::tma_store_2d(map, b, col, row0);
                }
                ptx::bulk_commit_group();  // one group per chunk, even if empty
            }
            ++chunk;
        };
        auto store_chunk = [&](const auto& bits, int32_t col, int32_t row0, int32_t ring_slot = -1) {
            constexpr int W = int(sizeof(bits) / sizeof(bits[0]));
            static_assert(W == 64 || W == 32, "a chunk is 64 or 32 columns");
            uint32_t buf;
            if (ring_slot >= 0) {
                buf = my_ring + uint32_t(ring_slot) * C::EPI_BUF_BYTES;
            } else {
                buf = buf0 + (chunk % C::EPI_BUFS) * C::EPI_BUF_BYTES;
                // the store EPI_BUFS chunks ago read `buf`
                if (lane == 0) ptx::bulk_wait_group_read<int(C::EPI_BUFS) - 1>();
            }
            __syncwarp();
            // Row `lane` of the 32 x W staging tile.  W = 64: 128-byte rows,
            // 128-byte swizzle (16-byte chunk c of row r at chunk position
            // c ^ (r % 8)).  W = 32: 64-byte rows, 64-byte swizzle (chunk c of
            // row r at c ^ ((r / 2) % 4)).  Either way the 8 lanes of each
            // quarter-warp phase of a 16-byte store cover all 32 banks.
            const uint32_t row_addr = buf + lane * uint32_t(2 * W);
            const uint32_t sw = (W == 64) ? (lane & 7u) : ((lane >> 1) & 3u);
#pragma unroll
            for (int c = 0; c < W / 8; ++c) {
                auto f = [&](int i) { return scaled(__uint_as_float(bits[8 * c + i])); };
                const uint32_t p0 = ptx::pack2<C::BF16>(f(0), f(1));
                const uint32_t p1 = ptx::pack2<C::BF16>(f(2), f(3));
                const uint32_t p2 = ptx::pack2<C::BF16>(f(4), f(5));
                const uint32_t p3 = ptx::pack2<C::BF16>(f(6), f(7));
                ptx::st_shared_v4(row_addr + ((uint32_t(c) ^ sw) << 4), p0, p1, p2, p3);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (row0 < args.M && col < args.N) {
                    const CUtensorMap* map = (W == 64) ? &tmap_d : &tmap_d32;
                    if (hint_d) ptx::tma_store_2d_hint(map, buf, col, row0, pol_d);
                    else ptx::tma_store_2d(map, buf, col, row0);
                }
                ptx::bulk_commit_group();  // one group per chunk, even if empty
            }
            ++chunk;
        };
        auto load_acc = [&](uint32_t taddr, float (&v)[64]) {
            uint32_t lo[32], hi[32];
            ptx::tmem_ld_32x32b_x32(taddr, lo);
            ptx::tmem_ld_32x32b_x32(taddr + 32u, hi);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                v[i] = __uint_as_float(lo[i]);
                v[32 + i] = __uint_as_float(hi[i]);
            }
        };

        for (int64_t u = cluster_id; u < units; u += num_clusters) {
            const WorkUnit w = unit_of(args, u);
            int32_t mt, nt;
            tile_of_task(args.grid, w.tile, mt, nt);
            uint32_t ok = 1u;
            if (lane == 0) ok = wait_bounded(acc_full_bar(ab), aph, ac, kRoleEpilogue);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            while (!ptx::mbar_try_wait(acc_full_bar(ab), aph)) {
            }  // completed already: gives every lane its own acquire
            ptx::tc_fence_after();

            const int32_t row0 = mt * C::BM + int32_t(rank) * C::A_ROWS + int32_t(quarter) * 32;
            const int32_t col0 = nt * C::BN;
            const uint32_t taddr = tmem_base + ((quarter * 32u) << 16) + ab * C::SLOT_COLS;

            // In the cluster's last unit the accumulator is not handed back: no
            // MMA will write it again, the MMA warp's drain does not wait for it,
            // and the teardown barrier orders these TMEM reads before the
            // dealloc.  (The hand-back is a cluster-scope release arrive that
            // costs the last tile's epilogue ~1.3 k cycles on the critical path.)
            const bool last_unit = (u + num_clusters >= units);
            auto release = [&](uint32_t b) {
                if (!last_unit) release_acc(b);
            };
            // Store pacing: the epilogue's TMA stores share the SM's TMA engine with
            // the operand loads, whose latency the ring only just covers; four
            // warps storing a tile at once delay the loads behind them (measured
            // ~700 cycles of MMA per 4096-deep tile).  Spreading each warp's chunk
            // stores 1 us apart leaves the loads room.  The pauses also delay the
            // accumulator hand-back, so they are used only where the next tile's
            // MMAs (>= 32 k-blocks) outlast them and a second accumulator exists.
            const bool pace = (C::NUM_ACC == 2) && !last_unit && w.kb1 - w.kb0 >= kStorePaceMinKBlocks;
            if (w.range < 0) {
                if constexpr (C::KS > 1) {
                    // In-cluster K split, summed as a reduce-scatter: CTA k owns
                    // columns [k W, (k+1) W) of the tile (W = BN / KS).  It writes
                    // its FP32 partial of each other CTA's columns for these 32 rows
                    // into that CTA's shared memory over distributed shared memory
                    // and arrives on that CTA's done[quarter]; then it adds the
                    // others' partials of its own columns to its own in CTA order
                    // (the same sum, term for term, whichever CTA owns the columns)
                    // and stores them.  The piece from the CTA s places after the
                    // owner (mod KS) fills the owner's slot s - 1: the first slots
                    // are its epilogue staging buffers, free from the start (one
                    // unit per cluster); a slot in its operand ring is free only
                    // once its own MMAs are done, which it announces on every other
                    // CTA's go[quarter] -- the pieces that need no announcement are
                    // written first.
                    constexpr int W = C::BN / C::KS;
                    constexpr int UW = W / 32;             // 32-column units it owns
                    constexpr int T = (C::KS - 1) * UW;    // units it sends
                    constexpr int T_STG = int(C::RECV_STG_SLOTS < uint32_t(C::KS - 1) ? C::RECV_STG_SLOTS
                                                                                   : uint32_t(C::KS - 1)) * UW;
                    constexpr bool NEED_GO = C::RECV_RING_SLOTS > 0;
                    // the address, in any CTA, of the slot `slot` of this quarter
                    auto recv_slot = [&](uint32_t slot) -> uint32_t {
                        return slot < C::RECV_STG_SLOTS
                                   ? buf0 + slot * C::RECV_SLICE_BYTES
                                   : base + C::OFF_A + ((slot - C::RECV_STG_SLOTS) * 4u + quarter) * C::RECV_SLICE_BYTES;
                    };
                    // the CTA that receives this CTA's piece in slot s
                    auto send_dst = [&](int t) -> uint32_t {
                        return (krank + uint32_t(C::KS - 1 - t / UW)) % uint32_t(C::KS);
                    };
                    if (lane == 0) {
                        // the KS - 1 pieces this warp will receive, as bytes on its done barrier
                        // (they may already have begun to land: the count may go below zero)
                        ptx::mbar_arrive_expect_tx(done_bar(quarter), uint32_t(C::KS - 1) * C::RECV_SLICE_BYTES);
                        if constexpr (NEED_GO)
                            for (uint32_t r = 0; r < uint32_t(C::KS); ++r)
                                if (r != krank) ptx::mbar_arrive_cluster(ptx::map_to_rank(go_bar(quarter), r));
                    }
                    // this warp's staged copy of the piece for slot s
                    auto send_slice = [&](uint32_t slot) -> uint32_t {
                        return base + C::OFF_KS_SEND + (slot * 4u + quarter) * C::RECV_SLICE_BYTES;
                    };
                    bool okg = true;
                    {
                        uint32_t ra[32], rb[32];
                        ptx::tmem_ld_32x32b_x32(taddr + send_dst(0) * W, ra);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int t = 0; t < T; ++t) {
                            uint32_t(&cur)[32] = (t % 2 == 0) ? ra : rb;
                            uint32_t(&nxt)[32] = (t % 2 == 0) ? rb : ra;
                            if (t + 1 < T)
                                ptx::tmem_ld_32x32b_x32(taddr + send_dst(t + 1) * W + 32u * uint32_t((t + 1) % UW),
                                                        nxt);
                            const uint32_t sl = send_slice(uint32_t(t / UW));
#pragma unroll
                            for (int g = 0; g < 8; ++g)
                                ptx::st_shared_v4(sl + ((uint32_t(t % UW) * 8u + uint32_t(g)) * 32u + lane) * 16u,
                                                  cur[4 * g], cur[4 * g + 1], cur[4 * g + 2], cur[4 * g + 3]);
                            if (t % UW == UW - 1) {  // the slot's piece is staged: send it
                                if (NEED_GO && t / UW == T_STG / UW) {  // the ring slots: wait for their owners
                                    uint32_t okw = 1u;
                                    if (lane == 0) okw = wait_bounded(go_bar(quarter), gph, ac, kRoleEpilogue);
                                    okw = __shfl_sync(0xffffffffu, okw, 0);
                                    if (!okw) {
                                        okg = false;
                                        if (t + 1 < T) ptx::tmem_wait_ld();
                                        break;
                                    }
                                    gph ^= 1u;
                                }
                                ptx::fence_proxy_async_smem();  // the staged piece, for the copy engine
                                __syncwarp();
                                if (lane == 0) {
                                    const uint32_t dst = send_dst(t);
                                    ptx::bulk_copy_s2cluster(ptx::map_to_rank(recv_slot(uint32_t(t / UW)), dst),
                                                             sl, C::RECV_SLICE_BYTES,
                                                             ptx::map_to_rank(done_bar(quarter), dst));
                                }
                            }
                            if (t + 1 < T) ptx::tmem_wait_ld();
                        }
                    }
                    if (!okg) break;
                    // this CTA's own columns: its partial from TMEM (the first
                    // load in flight while the others' pieces arrive)
                    const uint32_t town = taddr + krank * uint32_t(W);
                    uint32_t ra[32], rb[32];
                    ptx::tmem_ld_32x32b_x32(town, ra);
                    uint32_t okd = 1u;
                    if (lane == 0) okd = wait_bounded(done_bar(quarter), dph, ac, kRoleEpilogue);
                    okd = __shfl_sync(0xffffffffu, okd, 0);
                    ptx::tmem_wait_ld();
                    if (!okd) break;
                    while (!ptx::mbar_try_wait(done_bar(quarter), dph)) {
                    }  // completed already: every lane's own acquire
                    dph ^= 1u;
                    // output staging: the ring past its receiving slots, a fresh
                    // 4 KiB buffer per chunk (at most two per warp)
                    const uint32_t out0 = base + C::OFF_KS_OUT + (warp - 2u) * 2u * C::EPI_BUF_BYTES;
                    uint32_t buf = 0;
#pragma unroll
                    for (int v = 0; v < UW; ++v) {
                        uint32_t(&cur)[32] = (v % 2 == 0) ? ra : rb;
                        uint32_t(&nxt)[32] = (v % 2 == 0) ? rb : ra;
                        if (v + 1 < UW) ptx::tmem_ld_32x32b_x32(town + 32u * uint32_t(v + 1), nxt);
                        else release(ab);  // every TMEM read of this accumulator is done
                        // sum = p_0 + p_1 + ... in CTA order (p_krank from TMEM)
                        float acc[32];
#pragma unroll 1
                        for (uint32_t r = 0; r < uint32_t(C::KS); ++r) {
                            if (r == krank) {
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    const float x = __uint_as_float(cur[i]);
                                    acc[i] = (r == 0) ? x : acc[i] + x;
                                }
                                continue;
                            }
                            // CTA r's piece: r sits (r - krank) mod KS places after this CTA
                            const uint32_t sl = recv_slot((r + uint32_t(C::KS) - krank) % uint32_t(C::KS) - 1u);
#pragma unroll
                            for (int g = 0; g < 8; ++g) {
                                float x[4];
                                ptx::ld_shared_v4(sl + ((uint32_t(v) * 8u + uint32_t(g)) * 32u + lane) * 16u,
                                                  x[0], x[1], x[2], x[3]);
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    acc[4 * g + i] = (r == 0) ? x[i] : acc[4 * g + i] + x[i];
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 32; ++i) cur[i] = __float_as_uint(acc[i]);
                        const bool first_half = (v % 2 == 0);
                        if (first_half) buf = out0 + uint32_t(v / 2) * C::EPI_BUF_BYTES;
                        stage_half(cur, buf, W == 32 ? 32 : 64, first_half ? 0 : 1);
                        if (!first_half || W == 32)
                            issue_store(buf, col0 + int32_t(krank) * W + 64 * (v / 2), row0, W == 32 ? 32 : 64);
                        if (v + 1 < UW) ptx::tmem_wait_ld();
                    }
                } else {
                    // Whole tile: TMEM -> D, consumer by consumer (consumer h holds
                    // the CTA's A rows 128h..128h+127), 32 columns at a time: the
                    // TMEM load of the next 32 columns is in flight while the
                    // current ones are converted and staged, and each 64-column
                    // chunk (or the last 32 columns of a 224-wide tile) leaves as
                    // one TMA store once both of its halves are staged.
                    bool h_aborted = false;
#pragma unroll 1
                    for (int h = 0; h < C::CONS; ++h) {
                        if constexpr (C::CONS == 2) {
                            if (h == 1) {
                                // consumer 1's accumulator completes after consumer 0's
                                uint32_t ok1 = 1u;
                                if (lane == 0) ok1 = wait_bounded(acc_full_bar(1), aph, ac, kRoleEpilogue);
                                ok1 = __shfl_sync(0xffffffffu, ok1, 0);
                                if (!ok1) {
                                    h_aborted = true;
                                    break;
                                }
                                while (!ptx::mbar_try_wait(acc_full_bar(1), aph)) {
                                }  // completed already: every lane's own acquire
                                ptx::tc_fence_after();
                            }
                        }
                        const uint32_t th = taddr + uint32_t(h) * C::ACC_STRIDE;
                        const int32_t rh = row0 + 128 * h;
                        const bool last_h = (h == C::CONS - 1);
                        constexpr int U = C::BN / 32;  // 32-column units
                        constexpr int CHUNKS = C::FULL_CHUNKS + (C::HALF_CHUNK ? 1 : 0);
                        uint32_t ra[32], rb[32];
                        uint32_t buf = 0;
                        ptx::tmem_ld_32x32b_x32(th, ra);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            uint32_t(&cur)[32] = (u % 2 == 0) ? ra : rb;
                            uint32_t(&nxt)[32] = (u % 2 == 0) ? rb : ra;
                            if (u + 1 < U) {
                                ptx::tmem_ld_32x32b_x32(th + 32u * uint32_t(u + 1), nxt);
                            } else {
                                // every TMEM read of this accumulator is done; two
                                // consumers go back each on its own barrier
                                if (C::CONS == 2) release(uint32_t(h));
                                else if (last_h) release(ab);
                            }
                            const int c = u / 2;
                            const bool first_half = (u % 2 == 0);
                            const bool narrow = C::HALF_CHUNK && (c == C::FULL_CHUNKS);  // 32 columns
                            if (first_half) {
                                if (pace && c > 0) __nanosleep(kStorePaceNs);
                                // In the cluster's last unit the ring is idle once every
                                // MMA is done: with two consumers, only when consumer 1
                                // is drained (consumer 0's drain overlaps its last MMAs).
                                const bool ring_idle = last_unit && (C::CONS == 1 || h == C::CONS - 1);
                                buf = stage_buffer(ring_idle ? h * CHUNKS + c : -1);
                            }
                            stage_half(cur, buf, narrow ? 32 : 64, first_half ? 0 : 1);
                            if (!first_half || narrow) issue_store(buf, col0 + 64 * c, rh, narrow ? 32 : 64);
                            if (u + 1 < U) ptx::tmem_wait_ld();
                        }
                    }
                    if (h_aborted) break;
                }
            } else if constexpr (C::KS == 1) {  // (no tail split with an in-cluster split)
                // K-range of a tail tile.  Pass 1: write this range's FP32 partial
                // for the warp's 32 rows to its workspace slot, laid out so that
                // consecutive lanes touch consecutive 16-byte words.
                const int64_t slot_stride = 32 * C::BN / 4;  // float4 per slot
                const int64_t quad = (int64_t(w.tail) * C::CG + rank) * 4 + quarter;
                float4* const slots = reinterpret_cast<float4*>(args.partials);
                float4* const mine = slots + (quad * args.split + w.range) * slot_stride;
#pragma unroll 1
                for (int j = 0; j < C::BN / 64; ++j) {
                    float v[64];
                    load_acc(taddr + 64u * j, v);
#pragma unroll
                    for (int g = 0; g < 16; ++g)
                        mine[(j * 16 + g) * 32 + lane] =
                            make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
                }
                __threadfence();
                __syncwarp();
                uint32_t before = 0;
                if (lane == 0) before = count_range_done(args.counters + quad, args.epoch);
                before = __shfl_sync(0xffffffffu, before, 0);
                // The last range resets the word: every range has counted, so
                // nothing else touches it in this launch, and a later launch
                // that carries the same epoch (a CUDA graph replaying this one)
                // starts from zero.
                if (before == uint32_t(args.split - 1) && lane == 0) atomicExch(args.counters + quad, 0ull);
                if (before != uint32_t(args.split - 1)) {
                    release(ab);  // another range finishes this block of D
                } else if (u + num_clusters >= units &&
                           uint32_t(args.split - 1) <= C::PIECES_PER_WARP) {
                    // Pass 2 (the last range to finish, in this cluster's last
                    // unit, so the ring is idle): bulk-copy the other ranges'
                    // pieces of each 64-column chunk into this warp's share of
                    // the ring, then D = sum of all ranges in range order (this
                    // range's own piece read from TMEM).
                    __threadfence();
                    const uint32_t others = uint32_t(args.split - 1);
                    const int per_batch_max = int(C::PIECES_PER_WARP / others);
                    const int per_batch = per_batch_max < C::BN / 64 ? per_batch_max : C::BN / 64;
                    const float4* const first = slots + quad * args.split * slot_stride;
                    for (int j0 = 0; j0 < C::BN / 64; j0 += per_batch) {
                        const int j1 = (j0 + per_batch < C::BN / 64) ? j0 + per_batch : C::BN / 64;
                        uint32_t ok2 = 1u;
                        if (lane == 0) {
                            ptx::fence_proxy_async_global();
                            ptx::mbar_arrive_expect_tx(my_epi_bar,
                                                       uint32_t(j1 - j0) * others * C::PIECE_BYTES);
                            uint32_t piece = 0;
                            for (int j = j0; j < j1; ++j)
                                for (int r = 0; r < args.split; ++r) {
                                    if (r == w.range) continue;
                                    ptx::bulk_load_g2s(my_ring + piece * C::PIECE_BYTES,
                                                       first + r * slot_stride + j * 16 * 32,
                                                       C::PIECE_BYTES, my_epi_bar);
                                    ++piece;
                                }
                            ok2 = wait_bounded(my_epi_bar, eph, ac, kRoleEpilogue);
                        }
                        ok2 = __shfl_sync(0xffffffffu, ok2, 0);
                        if (ok2) {
                            while (!ptx::mbar_try_wait(my_epi_bar, eph)) {
                            }
                        }
                        eph ^= 1u;
                        uint32_t piece0 = 0;  // pieces of chunk j start at piece0
                        for (int j = j0; j < j1; ++j, piece0 += others) {
                            float acc[64];
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                uint32_t own[32];  // this range's piece, from TMEM
                                ptx::tmem_ld_32x32b_x32(taddr + 64u * j + 32u * h, own);
                                ptx::tmem_wait_ld();
                                uint32_t piece = piece0;
                                for (int r = 0; r < args.split; ++r) {
                                    if (r == w.range) {
#pragma unroll
                                        for (int i = 0; i < 32; ++i) {
                                            const float x = __uint_as_float(own[i]);
                                            acc[32 * h + i] = (r == 0) ? x : acc[32 * h + i] + x;
                                        }
                                        continue;
                                    }
                                    const uint32_t pb = my_ring + piece * C::PIECE_BYTES;
                                    ++piece;
#pragma unroll
                                    for (int g = 8 * h; g < 8 * h + 8; ++g) {
                                        float x, y, z, t;
                                        ptx::ld_shared_v4(pb + (uint32_t(g) * 32u + lane) * 16u, x, y, z, t);
                                        acc[4 * g] = (r == 0) ? x : acc[4 * g] + x;
                                        acc[4 * g + 1] = (r == 0) ? y : acc[4 * g + 1] + y;
                                        acc[4 * g + 2] = (r == 0) ? z : acc[4 * g + 2] + z;
                                        acc[4 * g + 3] = (r == 0) ? t : acc[4 * g + 3] + t;
                                    }
                                }
                            }
                            if (j == C::BN / 64 - 1) release(ab);
                            store_chunk(reinterpret_cast<const uint32_t(&)[64]>(acc), col0 + 64 * j, row0);
                        }
                    }
                } else {
                    // Pass 2 without the ring (a unit that is not this cluster's
                    // last, or a very deep split): read the other ranges'
                    // partials straight from L2.
                    __threadfence();
                    const float4* const first = slots + quad * args.split * slot_stride;
#pragma unroll 1
                    for (int j = 0; j < C::BN / 64; ++j) {
                        float acc[64];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t own[32];
                            ptx::tmem_ld_32x32b_x32(taddr + 64u * j + 32u * h, own);
                            ptx::tmem_wait_ld();
#pragma unroll 1
                            for (int r = 0; r < args.split; ++r) {
                                if (r == w.range) {
#pragma unroll
                                    for (int i = 0; i < 32; ++i) {
                                        const float x = __uint_as_float(own[i]);
                                        acc[32 * h + i] = (r == 0) ? x : acc[32 * h + i] + x;
                                    }
                                    continue;
                                }
                                const float4* src = first + r * slot_stride;
#pragma unroll
                                for (int g = 8 * h; g < 8 * h + 8; ++g) {
                                    const float4 q = __ldcg(src + (j * 16 + g) * 32 + lane);
                                    acc[4 * g] = (r == 0) ? q.x : acc[4 * g] + q.x;
                                    acc[4 * g + 1] = (r == 0) ? q.y : acc[4 * g + 1] + q.y;
                                    acc[4 * g + 2] = (r == 0) ? q.z : acc[4 * g + 2] + q.z;
                                    acc[4 * g + 3] = (r == 0) ? q.w : acc[4 * g + 3] + q.w;
                                }
                            }
                        }
                        if (j == C::BN / 64 - 1) release(ab);
                        store_chunk(reinterpret_cast<const uint32_t(&)[64]>(acc), col0 + 64 * j, row0);
                    }
                }
            }
            if (++ab == C::NUM_ACC) { ab = 0; aph ^= 1u; }
        }
        // Done with TMEM and with the cluster's shared state: arrive on the
        // final cluster barrier now, so that its latency and the skew between
        // the cluster's CTAs overlap the drain of this warp's bulk stores.
        settle_if_aborted(ac);
        ptx::tc_fence_before();
        if constexpr (C::CLUSTER > 1) ptx::cluster_arrive();
        if (lane == 0) ptx::bulk_wait_all();
        __syncwarp();
    }

    // ---- teardown ---------------------------------------------------------
    // Every CTA of the cluster stays until all are done (the peer reads this
    // CTA's shared memory and arrives on its barriers); TMEM is freed after
    // every warp's last TMEM read.  Without an abort every copy, MMA and
    // arrival aimed at a CTA has been waited for by one of its roles before
    // that role gets here.  After an abort (the flag is raised in both CTAs of
    // the pair), each warp that sees the flag settles before it arrives: an
    // operation still in flight was issued either before its issuer arrived
    // (and an issuer that saw the flag settled after it) or before the abort
    // (and the warp that raised it settles after it), and the barrier cannot
    // complete before those warps arrive.
    if (warp < 2) settle_if_aborted(ac);  // the epilogue warps settled already
    if constexpr (C::CLUSTER > 1) {
        if (early_producer) ptx::cluster_wait();  // the prologue phase, long complete
        if (warp < 2) {  // the epilogue warps arrived already
            ptx::tc_fence_before();
            ptx::cluster_arrive();
        }
        ptx::cluster_wait();
    } else {
        ptx::tc_fence_before();
        __syncthreads();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<C::CG>(tmem_base, C::TMEM_COLS);
    }
    if (args.clock_probe && blockIdx.x == 0 && threadIdx.x == 0) {
        args.clock_probe[2] = clock64();
        args.clock_probe[3] = ptx::global_timer_ns();
    }
}

// Failure-path self-test: one thread waits, through wait_bounded, on a
// barrier that nothing arrives on; the wait must give up after `limit_ns` and
// record (kReasonTimeout | kRoleSelfTest << 8) in the status word.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0u;
        ptx::mbar_init(ptx::smem_addr(&bar), 1);
        ptx::fence_mbar_init();
        const AbortCtl<1> ac{&abort_flag, 0u, 0u, limit_ns};
        wait_bounded(ptx::smem_addr(&bar), 0u, ac, kRoleSelfTest);
    }
}

// Block scales (MX) from row-major bytes (rows x groups, row stride ld,
// groups = ceil(K / 32)) to the tiled layout the GEMM loads: ceil(rows / 128)
// x kchunks atoms of 512 bytes (kchunks = ceil(K / 128)), atom (rb, kc) at byte
// (rb * kchunks + kc) * 512; inside it the scale of row rb * 128 + r, group
// kc * 4 + g sits at byte (r % 32) * 16 + (r / 32) * 4 + g.  Rows and groups
// past the ends get 127 (a scale of 1).  One thread per 32-bit word (the four
// groups of one row in one atom): word w of an atom is row (w % 4) * 32 + w / 4.
__global__ void mx_pack_scales_kernel(const uint8_t* __restrict__ src, int64_t rows,
                                      int64_t groups, int64_t ld, int64_t kchunks,
                                      uint32_t* __restrict__ dst, int64_t words) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < words;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t atom = i / 128;
        const int64_t w = i % 128;
        const int64_t row = (atom / kchunks) * 128 + (w % 4) * 32 + w / 4;
        const int64_t g0 = (atom % kchunks) * 4;
        uint32_t v = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint32_t b = (row < rows && g0 + g < groups) ? src[row * ld + g0 + g] : 127u;
            v |= b << (8 * g);
        }
        dst[i] = v;
    }
}

// B scales (MX) from row-major bytes (rows x groups, row stride ld) to the
// blocks the GEMM loads: block (t, kc) of 4096 bytes at (t * kchunks + kc) *
// 4096 holds, for the 224 columns of tile t and K groups 4 kc .. 4 kc + 3, the
// image of the tile's 128 x 256-bit TMEM copy: byte (r / 8) * 256 + (r % 8) *
// 16 + (c / 4) * 128 + (c % 4) * 4 + g is the scale of column 224 t + 32 c +
// r % 32 (c < 7), group 4 kc + g; every lane quarter r / 32 holds the same
// rows.  Past the matrix, and for c = 7, 127 (a scale of 1).  One thread per
// 32-bit word.
__global__ void mx_pack_scales_b_kernel(const uint8_t* __restrict__ src, int64_t rows,
                                        int64_t groups, int64_t ld, int64_t kchunks,
                                        uint32_t* __restrict__ dst, int64_t words) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < words;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t block = i / 1024;
        const uint32_t o = uint32_t(i % 1024) * 4u;  // byte offset in the block
        const uint32_t r = (o / 256u) * 8u + (o % 128u) / 16u;
        const uint32_t c = ((o % 256u) / 128u) * 4u + (o % 16u) / 4u;
        const int64_t col = (block / kchunks) * 224 + 32 * int64_t(c) + (r % 32u);
        const int64_t g0 = (block % kchunks) * 4;
        uint32_t v = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const bool inside = c < 7u && col < rows && g0 + g < groups;
            v |= (inside ? uint32_t(src[col * ld + g0 + g]) : 127u) << (8 * g);
        }
        dst[i] = v;
    }
}

// D = 0 for K == 0 (the empty sum).  One thread per 16-bit element.
__global__ void zero_fill_kernel(uint16_t* __restrict__ d, int64_t M, int64_t N, int64_t ldd) {
    const int64_t total = M * N;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        d[(i / N) * ldd + (i % N)] = 0;
    }
}

}  // namespace gb300
