// gemm_api.cu -- the C ABI of include/gemm.h: validation, TMA tensor maps,
// plan selection and the launch of the sm_103a kernel.
//
// The host builds three TMA tensor maps per call (A, B, D), picks the tile
// configuration and sizes a persistent grid of as many co-resident clusters as
// the device holds (capped by the tile count), then launches once on the
// caller's stream with the cluster dimension as a launch attribute.  This is
// the only host -> device step of a call.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <mutex>
#include <utility>

#include "gemm.h"
#include "gemm_kernel.cuh"
#include "workspace.h"

namespace gb300 {
namespace {

constexpr int kMaxDevices = 64;

// ---- driver entry point for tensor-map encoding ----------------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major 2-D tensor of 16-bit elements: `inner` contiguous elements per row,
// `outer` rows, row stride `ld` elements; boxes of box_inner x box_outer,
// 128-byte swizzle (64-byte for boxes of 64-byte rows), zero fill outside the
// tensor.
// `fmt`: GEMM_F16 / GEMM_BF16 (2-byte elements) or GEMM_E4M3 / GEMM_E5M2
// (1-byte elements, moved as raw bytes).
bool encode_2d(CUtensorMap* map, const void* ptr, int fmt, uint64_t inner, uint64_t outer,
               uint64_t ld, uint32_t box_inner, uint32_t box_outer) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const bool byte = (fmt == GEMM_E4M3 || fmt == GEMM_E5M2);
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {ld * (byte ? 1u : 2u)};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = byte ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : fmt == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint32_t row_bytes = box_inner * (byte ? 1u : 2u);
    const CUtensorMapSwizzle sw = row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    return enc(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Block scales (MX) of a rows x K FP8 operand, in the tiled layout of
// include/gemm.h: ceil(rows / 128) x ceil(K / 128) atoms of 512 bytes, atom
// (rb, kc) at byte (rb * ceil(K / 128) + kc) * 512.  Seen as a 2-D tensor of
// 32-bit words: ceil(K / 128) * 128 words per 128-row block, one block per row;
// boxes of one atom (128 words) x box_atoms consecutive row blocks, no
// swizzle, zero fill past the last block.
bool encode_scales(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t K, uint32_t box_atoms) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const uint64_t kc = (K + 127) / 128, rb = (rows + 127) / 128;
    const cuuint64_t dims[2] = {kc * 128, rb};
    const cuuint64_t strides[1] = {kc * 512};
    const cuuint32_t box[2] = {128, box_atoms};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Block scales (MX) of B, pre-laid-out for 224-column tiles (include/gemm.h):
// ceil(N / 224) * ceil(K / 128) blocks of 4096 bytes, seen as a 2-D tensor of
// 32-bit words with rows of 1 KiB; a box is one block (256 words x 4 rows).
bool encode_scales_b(CUtensorMap* map, const void* ptr, uint64_t N, uint64_t K) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const uint64_t blocks = ((N + 223) / 224) * ((K + 127) / 128);
    const cuuint64_t dims[2] = {256, blocks * 4};
    const cuuint64_t strides[1] = {1024};
    const cuuint32_t box[2] = {256, 4};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---- per-device facts, cached -------------------------------------------------

struct DeviceInfo {
    bool valid = false;
    bool supported = false;
    int sm_count = 0;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];

int current_device(DeviceInfo* out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& di = g_dev[dev];
    if (!di.valid) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        di.supported = (major == 10 && minor == 3);
        di.sm_count = sms;
        di.valid = true;
    }
    *out = di;
    return di.supported ? GEMM_OK : GEMM_ERR_DEVICE;
}

// ---- kernel variants -----------------------------------------------------------

// Opt a variant in to its dynamic shared memory size on the current device
// (once per device; every launch and occupancy query goes through here).
template <class C>
cudaError_t ensure_smem_attribute() {
    static std::atomic<uint64_t> done{0};  // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (bit && (done.load() & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(gemm_tcgen05_kernel<C>),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e == cudaSuccess && bit) done.fetch_or(bit);
    return e;
}

// `msa` / `msb`: the scale maps of a block-scaled (MX) variant; other
// variants ignore them (any valid map may be passed).
template <class C>
void launch_variant(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md,
                    const GemmArgs& args, const CUtensorMap& msa, const CUtensorMap& msb,
                    const CUtensorMap& md32, int clusters, cudaStream_t stream, cudaError_t* err) {
    if ((*err = ensure_smem_attribute<C>()) != cudaSuccess) return;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(clusters * C::CLUSTER), 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = C::CLUSTER > 1 ? 1 : 0;  // a lone CTA is launched as a plain grid
    *err = cudaLaunchKernelEx(&cfg, gemm_tcgen05_kernel<C>, ma, mb, md, args, msa, msb, md32);
}

// Co-resident clusters for a variant on the current device (queried once).
template <class C>
int query_max_clusters(int dev, int sm_count) {
    const void* fn = reinterpret_cast<const void*>(gemm_tcgen05_kernel<C>);
    if (ensure_smem_attribute<C>() != cudaSuccess) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(C::CLUSTER * (sm_count / C::CLUSTER)), 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) return -1;
    (void)dev;
    return n;
}

// Stage counts: as many 128-byte-swizzled K slices as fit next to the
// 32 KiB epilogue staging in 227 KiB.
constexpr int stages_for(int cg, int bn, int cons) {
    // (1-CTA tiles of at most 128 columns pair their stages: an even count)
    return ((227 * 1024 - 32768 - 1024 - 512) / (128 * cons * 64 * 2 + (bn / cg) * 64 * 2)) &
           ((cg == 1 && cons == 1 && bn <= 128) ? ~1 : ~0);
}
template <int CG, int BN, int CONS = 1>
struct Stages {
    // As many stages (16 KiB of A per consumer plus this CTA's share of B) as
    // fit in 227 KiB next to the 32 KiB epilogue staging and the barriers: 6
    // for 2-CTA 256-wide tiles (32 KiB / stage), 4 for 1-CTA 256-wide or for
    // two consumers (48 KiB).
    static constexpr int value = stages_for(CG, BN, CONS);
};

template <int CG, int BN, bool B_MN, bool BF16, int CONS = 1, int F8 = 0, int KS = 1>
using Cfg = KernelConfig<CG, BN, Stages<CG, BN, CONS>::value, B_MN, BF16, CONS, F8, false, KS>;

// Block-scaled FP8 (MX) stages: a stage also holds 512 B of A scales and the
// tile's 4 KiB block of B scales, and the epilogue stages through one 4 KiB
// buffer per warp; 6 stages of 2-CTA 224-wide tiles.
constexpr int stages_for_mx(int cg, int bn) {
    return (227 * 1024 - 16384 - 1024 - 512) / (128 * 128 + (bn / cg) * 128 + 512 + 4096);
}
template <int CG, int BN, bool BF16, int F8>
using CfgMX = KernelConfig<CG, BN, stages_for_mx(CG, BN), false, BF16, 1, F8, true>;

struct Plan {
    int cg, bm, bn, stages;
    int cons;  // MMA consumers per CTA
    int ks;    // K-ranges per tile inside a cluster (1 = none)
    int clusters;
    int64_t tiles;
    int group;            // tiles per raster group
    int order;            // kOrderM / kOrderN
    uint32_t hints;       // kHint* bits
    int64_t k_blocks;
    // Split of the last, partial round of tiles along K (1 = none).
    int64_t whole_units;  // tiles computed whole
    int split;            // K-ranges per remaining ("tail") tile
    size_t ws_counter_bytes, ws_partial_bytes;  // workspace the split needs
};

constexpr int kMaxSplit = 16;  // explicit tail_split limit

// Workspace layout for a split tail: one 8-byte counter per (tail tile, CTA,
// epilogue warp), then (256-byte aligned) one FP32 partial of 32 x block_n per
// (tail tile, CTA, epilogue warp, K-range).
void size_split(Plan* p) {
    const int64_t tail = p->tiles - p->whole_units;
    const int64_t quads = tail * p->cg * kEpilogueWarps;
    p->ws_counter_bytes = size_t(quads) * 8u;
    p->ws_partial_bytes = (p->split > 1) ? size_t(quads) * p->split * 32u * p->bn * 4u : 0u;
    if (p->split <= 1) p->ws_counter_bytes = 0;
}

size_t workspace_bytes_needed(const Plan& p) {
    if (p.split <= 1) return 0;
    return ((p.ws_counter_bytes + 255u) & ~size_t(255)) + p.ws_partial_bytes;
}

// Decide how the last round of the persistent schedule is handled.  With C
// clusters and T tiles there are ceil(T / C) rounds; the last one holds
// tail = T mod C tiles.
//  * Balanced grid (default): run the same number of rounds on the fewest
//    clusters, C' = ceil(T / rounds), so every cluster gets the same tile
//    count and no cluster idles in a partial round.  The clusters left out
//    draw no power, which lets the busy ones clock higher (the clock is set by
//    the power limit: measured ~3 % at 4096^3, 256 tiles on 64 instead of 76
//    clusters).
//  * Split tail (tail_split = s >= 2, with a workspace): keep all C clusters
//    and split each tail tile into s K-ranges whose FP32 partials are summed
//    by the range that finishes last.  Measured: the fix-up (partial write,
//    counter, partial read) costs about what the shorter round saves, so it
//    is not automatic.
//  * Split K of a single round (with a workspace; tail_split 0 = automatic,
//    s >= 2 = s ranges, 1 = never): when all T tiles fit in one round with
//    clusters to spare, every tile is split into s K-ranges, s <= C / T, so
//    the otherwise idle clusters share the K loop.  The fix-up is serial
//    latency (partial writes, a device-scope fence, the counter, the last
//    range reading the others' partials): measured ~4 us plus ~2 us per extra
//    range, so the automatic split keeps at least kMinRangeKBlocks k-blocks
//    per range.  Measured: 512 x 512 x 16384 58.1 -> 30.8 us (4 ranges),
//    1024 x 1024 x 8192 34.1 -> 28.8 us (2); 256 x 4096 x 4096 (2 ranges of
//    32) and 256 x 256 x 1024 (ranges of 8 or less) only got slower.
constexpr int64_t kMinRangeKBlocks = 64;

void plan_split(Plan* p, int requested, bool have_workspace, int max_clusters) {
    p->whole_units = p->tiles;
    p->split = 1;
    const bool splittable = have_workspace && (p->bn % 64) == 0 && p->cons == 1;
    if (splittable && p->tiles > 0 && p->tiles < max_clusters && requested != 1) {
        int64_t s = requested >= 2 ? requested : p->k_blocks / kMinRangeKBlocks;
        if (s > kMaxSplit) s = kMaxSplit;
        if (s > max_clusters / p->tiles) s = max_clusters / p->tiles;
        if (s > p->k_blocks) s = p->k_blocks;
        if (s >= 2) {
            p->split = int(s);
            p->whole_units = 0;
            p->clusters = int(p->tiles * s);
            size_split(p);
            return;
        }
    }
    const int64_t tail = p->clusters > 0 ? p->tiles % p->clusters : 0;
    if (have_workspace && tail > 0 && requested >= 2 && (p->bn % 64) == 0 && p->cons == 1) {
        int64_t s = requested;
        if (s > kMaxSplit) s = kMaxSplit;
        if (s > p->k_blocks) s = p->k_blocks;
        if (s >= 2) {
            p->split = int(s);
            p->whole_units = p->tiles - tail;
        }
    }
    if (p->split == 1 && p->clusters > 0 && p->tiles > 0) {
        const int64_t rounds = (p->tiles + p->clusters - 1) / p->clusters;
        p->clusters = int((p->tiles + rounds - 1) / rounds);
    }
    size_split(p);
}

std::atomic<uint32_t> g_epoch{0};

template <class C>
int run_with(const Plan& p, const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
             int64_t lda, int64_t ldb, int64_t ldd, int in_fmt, int out_dtype, float alpha,
             void* workspace, cudaStream_t stream, const void* SA, const void* SB,
             uint64_t wait_limit_ns, unsigned long long* clock_probe) {
    // An in-cluster K split reuses the operand ring of each CTA for the
    // partials once its own MMAs are done: exactly one tile per cluster.
    if (C::KS > 1 && (p.split != 1 || p.tiles != int64_t(p.clusters))) return GEMM_ERR_OPTION;
    CUtensorMap ma, mb, md;
    if (!encode_2d(&ma, A, in_fmt, uint64_t(K), uint64_t(M), uint64_t(lda), C::BK, C::A_ROWS))
        return GEMM_ERR_CUDA;
    if constexpr (!C::B_MN) {
        if (!encode_2d(&mb, B, in_fmt, uint64_t(K), uint64_t(N), uint64_t(ldb), C::BK, C::B_ROWS))
            return GEMM_ERR_CUDA;
    } else {
        if (!encode_2d(&mb, B, in_fmt, uint64_t(N), uint64_t(K), uint64_t(ldb), 64, C::BK))
            return GEMM_ERR_CUDA;
    }
    if (!encode_2d(&md, D, out_dtype, uint64_t(N), uint64_t(M), uint64_t(ldd), 64, 32))
        return GEMM_ERR_CUDA;
    // The last 32 columns of a tile whose width is an odd multiple of 32 (224),
    // and a CTA's 32 columns of a 128-wide tile split 4 ways inside its
    // cluster: 32 x 32 boxes.  Other variants never use the map.
    CUtensorMap md32 = md;
    if constexpr (C::D32) {
        if (!encode_2d(&md32, D, out_dtype, uint64_t(N), uint64_t(M), uint64_t(ldd), 32, 32))
            return GEMM_ERR_CUDA;
    }
    GemmArgs args;
    args.alpha = alpha;
    args.M = int32_t(M);
    args.N = int32_t(N);
    args.K = int32_t(K);
    args.k_blocks = int32_t((K + C::BK - 1) / C::BK);
    args.grid.m_tiles = int32_t((M + C::BM - 1) / C::BM);
    args.grid.n_tiles = int32_t((N + C::BN - 1) / C::BN);
    args.grid.group = p.group;
    args.grid.order = p.order;
    args.l2_hints = p.hints;
    args.whole_units = p.whole_units;
    args.split = p.split;
    args.epoch = g_epoch.fetch_add(1u) + 1u;
    args.counters = nullptr;
    args.partials = nullptr;
    args.wait_limit_ns = wait_limit_ns;
    args.clock_probe = clock_probe;
    if (p.split > 1) {
        char* ws = static_cast<char*>(workspace);
        args.counters = reinterpret_cast<unsigned long long*>(ws);
        args.partials = reinterpret_cast<float*>(ws + ((p.ws_counter_bytes + 255u) & ~size_t(255)));
    }
    // Block-scale maps: one A atom (this CTA's 128 rows) and the tile's B block
    // per k-block.
    CUtensorMap msa = ma, msb = ma;
    if constexpr (C::MX) {
        if (!encode_scales(&msa, SA, uint64_t(M), uint64_t(K), 1) ||
            !encode_scales_b(&msb, SB, uint64_t(N), uint64_t(K)))
            return GEMM_ERR_CUDA;
    } else {
        (void)SA;
        (void)SB;
    }
    cudaError_t err;
    launch_variant<C>(ma, mb, md, args, msa, msb, md32, p.clusters, stream, &err);
    return err == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// Dispatch on (cta_group, block_n, layout, dtype, FP8 input) to one template
// instance.  `bf16` is the output type (and the input type when f8 == 0).
template <template <class> class Fn, class... Ts>
int dispatch(int cg, int bn, bool b_mn, bool bf16, int cons, int f8, int ks, Ts&&... ts) {
    if (ks != 1) {
        // In-cluster K split: 16-bit, 1-CTA tiles, 128 wide (2 or 4 ranges)
        // or 64 / 256 wide (2 ranges).
        if (f8 != 0 || cons != 1 || cg != 1) return GEMM_ERR_OPTION;
#define GB300_CASEKS(BN_, KS_, MN_, BF_)                                                 \
    if (bn == BN_ && ks == KS_ && b_mn == MN_ && bf16 == BF_)                            \
        return Fn<Cfg<1, BN_, MN_, BF_, 1, 0, KS_>>::call(std::forward<Ts>(ts)...);
#define GB300_CASESKS(BN_, KS_) \
    GB300_CASEKS(BN_, KS_, false, false) GB300_CASEKS(BN_, KS_, false, true) \
    GB300_CASEKS(BN_, KS_, true, false) GB300_CASEKS(BN_, KS_, true, true)
        GB300_CASESKS(128, 2)
        GB300_CASESKS(128, 4)
        GB300_CASESKS(256, 2)
        GB300_CASESKS(64, 2)
#undef GB300_CASESKS
#undef GB300_CASEKS
        return GEMM_ERR_OPTION;
    }
    if (f8 != 0) {
        // FP8 inputs: K-major B, one consumer; 2-CTA 256 / 224-wide and 1-CTA
        // 256-wide tiles.
        if (b_mn || cons != 1) return GEMM_ERR_OPTION;
#define GB300_CASE8(CG_, BN_, F8_, BF_)                                                  \
    if (cg == CG_ && bn == BN_ && f8 == F8_ && bf16 == BF_)                              \
        return Fn<Cfg<CG_, BN_, false, BF_, 1, F8_>>::call(std::forward<Ts>(ts)...);
#define GB300_CASES8(CG_, BN_) \
    GB300_CASE8(CG_, BN_, 1, false) GB300_CASE8(CG_, BN_, 1, true) \
    GB300_CASE8(CG_, BN_, 2, false) GB300_CASE8(CG_, BN_, 2, true)
        GB300_CASES8(2, 256)
        GB300_CASES8(2, 224)
        GB300_CASES8(1, 256)
#undef GB300_CASES8
#undef GB300_CASE8
        return GEMM_ERR_OPTION;
    }
#define GB300_CASE(CG_, BN_, MN_, BF_)                                                   \
    if (cons == 1 && cg == CG_ && bn == BN_ && b_mn == MN_ && bf16 == BF_)               \
        return Fn<Cfg<CG_, BN_, MN_, BF_>>::call(std::forward<Ts>(ts)...);
#define GB300_CASE2(MN_, BF_)                                                            \
    if (cons == 2 && cg == 2 && bn == 256 && b_mn == MN_ && bf16 == BF_)                 \
        return Fn<Cfg<2, 256, MN_, BF_, 2>>::call(std::forward<Ts>(ts)...);
#define GB300_CASES(CG_, BN_) \
    GB300_CASE(CG_, BN_, false, false) GB300_CASE(CG_, BN_, false, true) \
    GB300_CASE(CG_, BN_, true, false) GB300_CASE(CG_, BN_, true, true)
#define GB300_KMAJOR_CASES(CG_, BN_) \
    GB300_CASE(CG_, BN_, false, false) GB300_CASE(CG_, BN_, false, true)
    GB300_CASES(2, 256)
    GB300_CASES(1, 256)
    GB300_CASES(2, 128)
    GB300_CASES(1, 128)
    GB300_CASES(1, 64)
    GB300_KMAJOR_CASES(1, 32)
    GB300_KMAJOR_CASES(2, 224)
    GB300_KMAJOR_CASES(2, 192)
    GB300_KMAJOR_CASES(1, 224)
    GB300_KMAJOR_CASES(1, 192)
    GB300_CASE2(false, false)
    GB300_CASE2(false, true)
    GB300_CASE2(true, false)
    GB300_CASE2(true, true)
#undef GB300_CASE2
#undef GB300_KMAJOR_CASES
#undef GB300_CASES
#undef GB300_CASE
    return GEMM_ERR_OPTION;
}

// Block-scaled FP8 (MX) variants: 2-CTA 224-wide tiles, E4M3 / E5M2 inputs,
// FP16 / BF16 output.
template <template <class> class Fn, class... Ts>
int dispatch_mx(int cg, int bn, bool bf16, int f8, Ts&&... ts) {
#define GB300_CASEMX(F8_, BF_)                                                           \
    if (cg == 2 && bn == 224 && f8 == F8_ && bf16 == BF_)                                \
        return Fn<CfgMX<2, 224, BF_, F8_>>::call(std::forward<Ts>(ts)...);
    GB300_CASEMX(1, false)
    GB300_CASEMX(1, true)
    GB300_CASEMX(2, false)
    GB300_CASEMX(2, true)
#undef GB300_CASEMX
    return GEMM_ERR_OPTION;
}

template <class C>
struct QueryFn {
    static int call(int dev, int sms, int* out) {
        static int cache[kMaxDevices] = {0};
        std::lock_guard<std::mutex> lock(g_mutex);
        if (cache[dev] == 0) {
            const int n = query_max_clusters<C>(dev, sms);
            if (n <= 0) return GEMM_ERR_CUDA;
            cache[dev] = n;
        }
        *out = cache[dev];
        return GEMM_OK;
    }
};

template <class C>
struct RunFn {
    static int call(const Plan& p, const void* A, const void* B, void* D, int64_t M, int64_t N,
                    int64_t K, int64_t lda, int64_t ldb, int64_t ldd, int in_fmt, int out_dtype,
                    float alpha, void* workspace, cudaStream_t stream, const void* SA,
                    const void* SB, uint64_t wait_limit_ns, unsigned long long* clock_probe) {
        return run_with<C>(p, A, B, D, M, N, K, lda, ldb, ldd, in_fmt, out_dtype, alpha, workspace,
                           stream, SA, SB, wait_limit_ns, clock_probe);
    }
};

bool is_fp8(int fmt) { return fmt == GEMM_E4M3 || fmt == GEMM_E5M2; }
int f8_code(int fmt) { return fmt == GEMM_E4M3 ? 1 : fmt == GEMM_E5M2 ? 2 : 0; }

// `dtype` is the input format: GEMM_F16 / GEMM_BF16, or (where FP8 inputs are
// accepted) GEMM_E4M3 / GEMM_E5M2, which take the K-major A.Bt layout only.
int check_sizes(int64_t M, int64_t N, int64_t K, int dtype, int b_layout) {
    if (dtype != GEMM_F16 && dtype != GEMM_BF16 && !is_fp8(dtype)) return GEMM_ERR_DTYPE;
    if (is_fp8(dtype) && b_layout != 0) return GEMM_ERR_OPTION;
    if (b_layout != 0 && b_layout != 1) return GEMM_ERR_OPTION;
    if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return GEMM_ERR_SHAPE;
    return GEMM_OK;
}

int check_options(const gemm_options_t* o) {
    if (!o) return GEMM_OK;
    if (o->cta_group != 0 && o->cta_group != 1 && o->cta_group != 2) return GEMM_ERR_OPTION;
    if (o->block_n != 0 && o->block_n != 32 && o->block_n != 64 && o->block_n != 128 &&
        o->block_n != 192 && o->block_n != 224 && o->block_n != 256)
        return GEMM_ERR_OPTION;
    if (o->raster_group < 0 || o->max_clusters < 0) return GEMM_ERR_OPTION;
    if (o->tail_split < 0 || o->tail_split > kMaxSplit) return GEMM_ERR_OPTION;
    if (o->consumers < 0 || o->consumers > 2) return GEMM_ERR_OPTION;
    // multicast: kept in the struct for layout stability; 0 or 1 (no multicast) only.
    if (o->multicast < 0 || o->multicast > 1) return GEMM_ERR_OPTION;
    if (o->raster_order < 0 || o->raster_order > 2) return GEMM_ERR_OPTION;
    // l2_hints: 0 = automatic, else an odd value (bit 0 marks the explicit choice)
    if (o->l2_hints < 0 || o->l2_hints > 15 || (o->l2_hints != 0 && !(o->l2_hints & 1)))
        return GEMM_ERR_OPTION;
    if (o->cluster_ksplit != 0 && o->cluster_ksplit != 1 && o->cluster_ksplit != 2 &&
        o->cluster_ksplit != 4)
        return GEMM_ERR_OPTION;
    return GEMM_OK;
}

int max_clusters_for(int cg, int bn, int b_layout, int dtype, int dev, int sm_count, int ks = 1) {
    int n = 0;
    if (dispatch<QueryFn>(cg, bn, b_layout == 1, dtype == GEMM_BF16, 1, f8_code(dtype), ks, dev,
                          sm_count, &n) != GEMM_OK)
        return 0;
    return n;
}

// Tile width N for the automatic plan.  Every round of the persistent schedule
// costs one tile time, and a tile's time grows with its width divided by the
// MMA efficiency of that width (narrower tiles move more operand bytes per
// FLOP).  Pick the width with the least rounds x width / efficiency; ties go
// to the wider tile.  4096^3 on 76 clusters: 256-wide tiles take 4 rounds of
// 256, 224-wide tiles 4 rounds of 224 (all 304 tiles busy), and the 224-wide
// plan runs ~7 % faster; at 8192^3 the two tie and 256 wins.
int choose_block_n(int64_t M, int64_t N, int bm, int b_layout, int cg, int dtype, int dev,
                   int sm_count) {
    struct Cand {
        int bn;
        double eff;
    };
    // Relative tensor efficiency of a round of narrower tiles (more epilogue and
    // operand traffic per MMA), measured on 4096^3 .. 8192^3 GEMMs.
    static const Cand kCands[] = {{256, 1.0}, {224, 0.975}, {192, 0.9}};
    if (M <= 0 || N <= 0) return 256;
    int best = 256;
    double best_cost = 0;
    for (const Cand& c : kCands) {
        if (b_layout == 1 && (c.bn % 128) != 0) continue;
        const int C = max_clusters_for(cg, c.bn, b_layout, dtype, dev, sm_count);
        if (C <= 0) continue;
        const int64_t tiles = ((M + bm - 1) / bm) * ((N + c.bn - 1) / c.bn);
        const int64_t rounds = (tiles + C - 1) / C;
        const double cost = double(rounds) * c.bn / c.eff;
        if (best_cost == 0 || cost < best_cost * (1 - 1e-9)) {
            best = c.bn;
            best_cost = cost;
        }
    }
    return best;
}

// L2 bytes a raster group's resident band may take: the band must stay in L2
// while the group walks the other dimension, next to the streamed operand's
// panels and the output tiles in flight.  Measured on 8192 x 17408 x 5120
// BF16 A.B (256 x 256 tiles): bands of 21 and 31 MB (8, 12 M tiles) stay
// resident (DRAM reads within 1.3x of the model below), a 42 MB band (16)
// mostly does, an 84 MB band (32) does not (2.1 GB read instead of 0.26 GB).
constexpr double kBandBudgetBytes = 48.0 * (1 << 20);
constexpr int kGroups[] = {16, 12, 8, 4, 2, 1};

// Raster order and group from the reuse-window argument ("Choosing schedules
// and instructions for a backend", section 2, memory report: the operand whose
// reuse window exceeds L2 is re-read; section 3: grouping M tiles keeps a band
// of A resident while B streams).  With M groups of G tiles, A is read once
// and B once per group: A + B * ceil(m_tiles / G) bytes, if A's band (G x
// block_m rows x K) fits the budget; with N groups the roles swap.  Take the
// order and the largest group with the least predicted traffic (ties: M
// groups, larger groups).  Operands that fit in L2 together are read once
// whatever the order: then the tutorial's G = 16 M groups.  Options override
// any part of the choice; L2 hints are never automatic (measured: they move
// DRAM bytes, not time, and an evict_last band could outlive the call).
void plan_raster(Plan* p, int64_t M, int64_t N, int64_t K, int esize, const gemm_options_t* o) {
    const int64_t m_tiles = (M + p->bm - 1) / p->bm;
    const int64_t n_tiles = (N + p->bn - 1) / p->bn;
    const double a_bytes = double(M) * K * esize, b_bytes = double(N) * K * esize;
    int order = kOrderM, group = 16;
    if (a_bytes + b_bytes > kBandBudgetBytes) {
        double best = 0;
        for (int ord = kOrderM; ord <= kOrderN; ++ord) {
            if (o && o->raster_order && o->raster_order - 1 != ord) continue;
            const int64_t along = ord == kOrderM ? m_tiles : n_tiles;
            const double band_per_tile = double(ord == kOrderM ? p->bm : p->bn) * K * esize;
            const double kept = ord == kOrderM ? a_bytes : b_bytes;
            const double streamed = ord == kOrderM ? b_bytes : a_bytes;
            for (int g : kGroups) {
                if (o && o->raster_group && o->raster_group != g) continue;
                if (g > 1 && g * band_per_tile > kBandBudgetBytes) continue;
                const int64_t gg = g < along ? g : (along > 0 ? along : 1);
                const double traffic = kept + streamed * double((along + gg - 1) / gg);
                if (best == 0 || traffic < best * (1 - 1e-9)) {
                    best = traffic;
                    order = ord;
                    group = g;
                }
            }
        }
    }
    p->order = (o && o->raster_order) ? o->raster_order - 1 : order;
    p->group = (o && o->raster_group) ? o->raster_group : group;
    p->hints = (o && o->l2_hints) ? uint32_t(o->l2_hints) : 0u;
    const int64_t along = p->order == kOrderN ? n_tiles : m_tiles;
    if (p->group > along) p->group = int(along > 0 ? along : 1);
}

// Small problems: when the chosen tiles fit in one round of the persistent
// grid, the time is one tile's latency, which shrinks with the tile's width
// (each SM computes 128 rows x BN whether the tile is one CTA's or a pair's).
// Take the narrowest tile (128 wide, one or two CTAs) that still fits in one
// round, if it is narrower than the choice so far.  Measured on 256 x 256 x
// 1024: 11 us with four 1-CTA 128 x 128 tiles against 12.7 us with two
// 256 x 192 tiles and 14.5 us with one 256 x 256 tile.  Large problems (more
// than one round) keep the wide tiles, which move fewer bytes per FLOP.
void spread_small(int64_t M, int64_t N, int b_layout, int dtype, int dev, int sm_count, bool cg_free,
                  Plan* p) {
    const int C = max_clusters_for(p->cg, p->bn, b_layout, dtype, dev, sm_count);
    if (C <= 0 || M <= 0 || N <= 0) return;
    const int64_t tiles = ((M + p->bm - 1) / p->bm) * ((N + p->bn - 1) / p->bn);
    if (tiles > C || p->bn <= 128) return;  // more than one round: keep the wide tiles
    // 128-wide tiles of one or two CTAs: the one with the most tiles that still
    // fits in one round (ties keep the current CTA count).
    int best_cg = 0;
    int64_t best_t = 0;
    const int cgs[2] = {p->cg, 3 - p->cg};
    for (int cg : cgs) {
        if (!cg_free && cg != p->cg) continue;
        const int Cn = max_clusters_for(cg, 128, b_layout, dtype, dev, sm_count);
        const int64_t t = ((M + 128 * cg - 1) / (128 * cg)) * ((N + 127) / 128);
        if (Cn > 0 && t <= Cn && t >= tiles && t > best_t) {
            best_cg = cg;
            best_t = t;
        }
    }
    if (best_cg) {
        p->cg = best_cg;
        p->bm = 128 * best_cg;
        p->bn = 128;
    }
}

// In-cluster K split (cluster_ksplit: 0 = automatic, 1 = never, 2 / 4 =
// ranges): a problem whose 1-CTA tiles all fit in one round of KS-CTA clusters
// has each tile computed by a cluster of KS CTAs, one K-range each; each CTA
// owns BN / KS of the tile's columns and the partials are exchanged over
// distributed shared memory (no workspace).  The exchange and the cluster
// launch cost a few microseconds (measured: ~3 us with 2 ranges, ~4 us with
// 4), so the automatic choice is the most ranges (4 for 128-wide tiles, 2
// for 256-wide) that keep at least kMinClusterRangeKBlocks k-blocks per
// range, and none when the workspace split (plan_split) would run more
// ranges per tile or when K has fewer than kNarrowMaxKBlocks k-blocks.
constexpr int64_t kMinClusterRangeKBlocks = 16;
// Below kNarrowMaxKBlocks k-blocks (and from kNarrowMinKBlocks) a single-round
// problem takes narrow tiles instead (plan_narrow), which measured faster than
// splitting K in the cluster there (1024 x 1024 x 2048: 14.8 us on 64-wide
// tiles, 16.8 us with 2 ranges per 128-wide tile).
constexpr int64_t kNarrowMinKBlocks = 8;
constexpr int64_t kNarrowMaxKBlocks = 64;

void plan_cluster_split(int b_layout, int dtype, int dev, int sm_count, const gemm_options_t* o,
                        bool have_workspace, int max_clusters, Plan* p) {
    p->ks = 1;
    const int req = o ? o->cluster_ksplit : 0;
    if (req == 1 || is_fp8(dtype) || p->cons != 1 || p->cg != 1) return;
    if (p->bn != 128 && p->bn != 256) return;
    // ranges per tile of the automatic workspace split, for comparison
    int64_t ws_ranges = 1;
    if (req == 0 && have_workspace && (o ? o->tail_split : 0) != 1 && p->tiles > 0 &&
        p->tiles < max_clusters) {
        ws_ranges = p->k_blocks / kMinRangeKBlocks;
        if (ws_ranges > kMaxSplit) ws_ranges = kMaxSplit;
        if (ws_ranges > max_clusters / p->tiles) ws_ranges = max_clusters / p->tiles;
    }
    const int cands[2] = {4, 2};
    for (int ks : cands) {
        if (req >= 2 && ks != req) continue;
        if (ks == 4 && p->bn != 128) continue;
        if (req == 0 && (p->k_blocks < ks * kMinClusterRangeKBlocks || ws_ranges > ks ||
                         p->k_blocks < kNarrowMaxKBlocks))
            continue;
        if (p->k_blocks < ks) continue;
        int C = max_clusters_for(1, p->bn, b_layout, dtype, dev, sm_count, ks);
        if (o && o->max_clusters && o->max_clusters < C) C = o->max_clusters;
        if (C <= 0 || p->tiles > C) continue;
        p->ks = ks;
        p->clusters = int(p->tiles);
        return;
    }
}

// Narrow tiles for shallow single-round problems: a 1-CTA tile's k-block costs
// the MMA warp ~400 cycles of issue whatever its width up to 128 columns
// (paired stages), and a 128-wide one is bound at ~515 cycles by the 32 KiB
// each SM must take in per k-block, so a problem whose 128-wide tiles fit one
// round with SMs to spare finishes sooner on 32- (B N x K only) or 64-wide
// tiles if those still fit one round.  Measured (L2 flushed): 256 x 256 x 1024
// 12.5 -> 10.5 us on 32-wide tiles, 1024 x 1024 x 2048 16.8 -> 14.8 us on
// 64-wide.  Only below kNarrowMaxKBlocks k-blocks: deeper problems gain more
// from splitting K (in the cluster or over the workspace), which needs 64- or
// 128-wide tiles.

void plan_narrow(int64_t M, int64_t N, int b_layout, int dtype, int dev, int sm_count, Plan* p) {
    if (is_fp8(dtype) || p->cg != 1 || p->cons != 1 || p->bn != 128 || p->ks != 1) return;
    if (p->k_blocks < kNarrowMinKBlocks || p->k_blocks >= kNarrowMaxKBlocks) return;
    const int C128 = max_clusters_for(1, 128, b_layout, dtype, dev, sm_count);
    if (C128 <= 0 || p->tiles > C128) return;  // 128-wide tiles take more than one round
    const int cands[2] = {32, 64};
    for (int bn : cands) {
        if (bn == 32 && b_layout != 0) continue;
        const int C = max_clusters_for(1, bn, b_layout, dtype, dev, sm_count);
        const int64_t tiles = ((M + 127) / 128) * ((N + bn - 1) / bn);
        if (C <= 0 || tiles > C) continue;
        p->bn = bn;
        p->tiles = tiles;
        p->clusters = int(tiles);
        p->stages = stages_for(1, bn, 1);
        return;
    }
}

// Choose the tile shape and grid.  Needs the current device (for its SM count
// and cluster occupancy).
int make_plan(int64_t M, int64_t N, int64_t K, int dtype, int b_layout, const gemm_options_t* o,
              bool have_workspace, Plan* p, bool mx = false) {
    DeviceInfo di;
    int st = current_device(&di);
    if (st != GEMM_OK) return st;
    int dev = 0;
    cudaGetDevice(&dev);
    if (mx) {
        // Block-scaled FP8: 2-CTA clusters, 224-wide tiles, whole tiles only.
        if (!is_fp8(dtype) || b_layout != 0) return GEMM_ERR_DTYPE;
        if (o && ((o->cta_group && o->cta_group != 2) || (o->block_n && o->block_n != 224) ||
                  o->consumers > 1 || o->tail_split > 1))
            return GEMM_ERR_OPTION;
        p->cg = 2;
        p->cons = 1;
        p->ks = 1;
        p->bm = 256;
        p->bn = 224;
        const int64_t m_tiles = (M + p->bm - 1) / p->bm;
        p->tiles = m_tiles * ((N + p->bn - 1) / p->bn);
        if (p->tiles >= kMaxTiles) return GEMM_ERR_SHAPE;
        plan_raster(p, M, N, K, 1, o);
        int max_clusters = 0;
        st = dispatch_mx<QueryFn>(p->cg, p->bn, false, f8_code(dtype), dev, di.sm_count, &max_clusters);
        if (st != GEMM_OK) return st;
        if (o && o->max_clusters && o->max_clusters < max_clusters) max_clusters = o->max_clusters;
        p->clusters = int(p->tiles < max_clusters ? p->tiles : max_clusters);
        p->stages = stages_for_mx(p->cg, p->bn);
        p->k_blocks = (K + kBlockK8 - 1) / kBlockK8;
        plan_split(p, 0, false, max_clusters);
        return GEMM_OK;
    }
    p->cg = (o && o->cta_group) ? o->cta_group : (M <= 128 ? 1 : 2);
    p->cons = (o && o->consumers) ? o->consumers : 1;
    if (is_fp8(dtype) && p->cons != 1) return GEMM_ERR_OPTION;
    p->bm = 128 * p->cg * p->cons;
    if (p->cons == 2) {
        // Two consumers: 2-CTA clusters, 256-wide tiles only.
        if (p->cg != 2 || (o && o->block_n && o->block_n != 256)) return GEMM_ERR_OPTION;
        p->bn = 256;
    } else if (o && o->block_n) {
        p->bn = o->block_n;
        // 32- and 64-wide tiles are 1-CTA tiles (an explicit cta_group 2 is an
        // error; an automatic one becomes 1).
        if (p->bn < 128) {
            if (o->cta_group == 2) return GEMM_ERR_OPTION;
            p->cg = 1;
            p->bm = 128;
        }
        // An MN-major B tile is loaded in 64-column atoms: 64- (1-CTA), 128-
        // and 256-wide tiles only.
        if (b_layout == 1 && (p->bn % 128) != 0 && p->bn != 64) return GEMM_ERR_OPTION;
    } else {
        p->bn = choose_block_n(M, N, p->bm, b_layout, p->cg, dtype, dev, di.sm_count);
        const bool cg_free = !(o && o->cta_group);
        if (p->cons == 1 && !is_fp8(dtype)) spread_small(M, N, b_layout, dtype, dev, di.sm_count, cg_free, p);
    }
    const int64_t m_tiles = (M + p->bm - 1) / p->bm;
    const int64_t n_tiles = (N + p->bn - 1) / p->bn;
    p->tiles = m_tiles * n_tiles;
    if (p->tiles >= kMaxTiles) return GEMM_ERR_SHAPE;
    plan_raster(p, M, N, K, is_fp8(dtype) ? 1 : 2, o);
    int max_clusters = 0;
    st = dispatch<QueryFn>(p->cg, p->bn, b_layout == 1, dtype == GEMM_BF16, p->cons, f8_code(dtype),
                           1, dev, di.sm_count, &max_clusters);
    if (st != GEMM_OK) return st;
    if (o && o->max_clusters && o->max_clusters < max_clusters) max_clusters = o->max_clusters;
    p->clusters = int(p->tiles < max_clusters ? p->tiles : max_clusters);
    p->stages = stages_for(p->cg, p->bn, p->cons);
    const int bk = is_fp8(dtype) ? kBlockK8 : kBlockK;
    p->k_blocks = (K + bk - 1) / bk;
    plan_cluster_split(b_layout, dtype, dev, di.sm_count, o, have_workspace, max_clusters, p);
    if (!(o && o->block_n)) {
        const int bn0 = p->bn;
        plan_narrow(M, N, b_layout, dtype, dev, di.sm_count, p);
        if (p->bn != bn0) {
            plan_raster(p, M, N, K, 2, o);
            max_clusters = max_clusters_for(1, p->bn, b_layout, dtype, dev, di.sm_count);
            if (o && o->max_clusters && o->max_clusters < max_clusters) max_clusters = o->max_clusters;
            if (p->clusters > max_clusters) p->clusters = max_clusters;
        }
    }
    if (p->ks > 1) {
        // one cluster per tile; no workspace split on top
        p->whole_units = p->tiles;
        p->split = 1;
        size_split(p);
        return GEMM_OK;
    }
    plan_split(p, o ? o->tail_split : 0, have_workspace, max_clusters);
    return GEMM_OK;
}

bool overlaps(const void* a, int64_t rows_a, int64_t cols_a, int64_t ld_a, int esize_a,
              const void* b, int64_t rows_b, int64_t cols_b, int64_t ld_b, int esize_b) {
    if (rows_a == 0 || cols_a == 0 || rows_b == 0 || cols_b == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a);
    const uintptr_t a1 = a0 + uintptr_t(((rows_a - 1) * ld_a + cols_a) * esize_a);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(b);
    const uintptr_t b1 = b0 + uintptr_t(((rows_b - 1) * ld_b + cols_b) * esize_b);
    return a0 < b1 && b0 < a1;
}

}  // namespace
}  // namespace gb300

using namespace gb300;

namespace gb300 {
namespace {

// Shared body of the 16-bit and FP8 entry points.  in_fmt: GEMM_F16 /
// GEMM_BF16 (then out_dtype == in_fmt) or GEMM_E4M3 / GEMM_E5M2 (A.Bt only).
// Bytes of the block scales (MX) of A (rows = M) and of B.
int64_t mx_scale_bytes(int64_t rows, int64_t K) {
    return ((rows + 127) / 128) * ((K + 127) / 128) * 512;
}
int64_t mx_scale_b_bytes(int64_t N, int64_t K) {
    return ((N + 223) / 224) * ((K + 127) / 128) * 4096;
}

int run_impl(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K, int64_t lda,
             int64_t ldb, int64_t ldd, int in_fmt, int out_dtype, float alpha, int b_layout,
             const gemm_options_t* opts, void* workspace, size_t workspace_bytes,
             cudaStream_t stream, const void* SA = nullptr, const void* SB = nullptr,
             bool mx = false, uint64_t wait_limit_ns = kWaitLimitNs,
             unsigned long long* clock_probe = nullptr) {
    int st = check_sizes(M, N, K, in_fmt, b_layout);
    if (st != GEMM_OK) return st;
    if (out_dtype != GEMM_F16 && out_dtype != GEMM_BF16) return GEMM_ERR_DTYPE;
    if ((st = check_options(opts)) != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    const int esize = is_fp8(in_fmt) ? 1 : 2;
    const int64_t b_rows = b_layout == 0 ? N : K;
    const int64_t b_cols = b_layout == 0 ? K : N;
    if (!D || (K > 0 && (!A || !B))) return GEMM_ERR_NULL;
    if (ldd < N || ldd <= 0) return GEMM_ERR_SHAPE;
    if (K > 0 && (lda < K || ldb < b_cols || lda <= 0 || ldb <= 0)) return GEMM_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(D) & 15u) || (ldd & 7)) return GEMM_ERR_ALIGN;
    // TMA: 16-byte aligned bases and row strides that are multiples of 16 bytes.
    const int64_t ld_mask = (16 / esize) - 1;
    if (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) ||
                  (lda & ld_mask) || (ldb & ld_mask)))
        return GEMM_ERR_ALIGN;
    if (K > 0 && (overlaps(D, M, N, ldd, 2, A, M, K, lda, esize) ||
                  overlaps(D, M, N, ldd, 2, B, b_rows, b_cols, ldb, esize)))
        return GEMM_ERR_ALIAS;
    if (mx && K > 0) {
        if (!SA || !SB) return GEMM_ERR_NULL;
        if ((reinterpret_cast<uintptr_t>(SA) & 15u) || (reinterpret_cast<uintptr_t>(SB) & 15u))
            return GEMM_ERR_ALIGN;
        const int64_t sa = mx_scale_bytes(M, K), sb = mx_scale_b_bytes(N, K);
        if (overlaps(D, M, N, ldd, 2, SA, 1, sa, sa, 1) || overlaps(D, M, N, ldd, 2, SB, 1, sb, sb, 1))
            return GEMM_ERR_ALIAS;
        if (sb / 1024 > INT32_MAX) return GEMM_ERR_SHAPE;  // TMA row coordinates are 32-bit
    }

    if (K == 0) {
        DeviceInfo di;
        if ((st = current_device(&di)) != GEMM_OK) return st;
        const int64_t total = M * N;
        int64_t blocks = (total + 255) / 256;
        if (blocks > 4L * di.sm_count * 8) blocks = 4L * di.sm_count * 8;
        zero_fill_kernel<<<unsigned(blocks), 256, 0, stream>>>(static_cast<uint16_t*>(D), M, N, ldd);
        return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }

    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return GEMM_ERR_WORKSPACE;
    Plan p;
    if ((st = make_plan(M, N, K, in_fmt, b_layout, opts, workspace != nullptr, &p, mx)) != GEMM_OK)
        return st;
    if (workspace_bytes < workspace_bytes_needed(p)) return GEMM_ERR_WORKSPACE;
    if (mx)
        return dispatch_mx<RunFn>(p.cg, p.bn, out_dtype == GEMM_BF16, f8_code(in_fmt), p, A, B, D, M,
                                  N, K, lda, ldb, ldd, in_fmt, out_dtype, alpha, workspace, stream,
                                  SA, SB, wait_limit_ns, clock_probe);
    return dispatch<RunFn>(p.cg, p.bn, b_layout == 1, out_dtype == GEMM_BF16, p.cons, f8_code(in_fmt), p.ks, p, A, B, D, M, N, K, lda, ldb, ldd, in_fmt, out_dtype,
                           alpha, workspace, stream, static_cast<const void*>(nullptr),
                           static_cast<const void*>(nullptr), wait_limit_ns, clock_probe);
}

}  // namespace
}  // namespace gb300

extern "C" int gemm_run_workspace(const void* A, const void* B, void* D, int64_t M, int64_t N,
                                  int64_t K, int64_t lda, int64_t ldb, int64_t ldd, int dtype,
                                  int b_layout, const gemm_options_t* opts, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
    if (is_fp8(dtype)) return GEMM_ERR_DTYPE;  // FP8 inputs: gemm_fp8_run_workspace
    return run_impl(A, B, D, M, N, K, lda, ldb, ldd, dtype, dtype, 1.0f, b_layout, opts, workspace,
                    workspace_bytes, stream);
}

extern "C" int gemm_fp8_run_workspace(const void* A, const void* B, void* D, int64_t M, int64_t N,
                                      int64_t K, int64_t lda, int64_t ldb, int64_t ldd,
                                      int in_format, int out_dtype, float alpha,
                                      const gemm_options_t* opts, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream) {
    if (!is_fp8(in_format)) return GEMM_ERR_DTYPE;
    return run_impl(A, B, D, M, N, K, lda, ldb, ldd, in_format, out_dtype, alpha, 0, opts,
                    workspace, workspace_bytes, stream);
}

extern "C" int gemm_fp8_run(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t ldb, int64_t ldd, int in_format, int out_dtype,
                            float alpha, const gemm_options_t* opts, cudaStream_t stream) {
    return gemm_fp8_run_workspace(A, B, D, M, N, K, lda, ldb, ldd, in_format, out_dtype, alpha,
                                  opts, nullptr, 0, stream);
}

extern "C" int gemm_fp8_abt(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t ldb, int64_t ldd, int in_format, int out_dtype,
                            float alpha, cudaStream_t stream) {
    return gemm_fp8_run(A, B, D, M, N, K, lda, ldb, ldd, in_format, out_dtype, alpha, nullptr,
                        stream);
}

extern "C" int gemm_mx_run(const void* A, const void* B, const void* SA, const void* SB, void* D,
                           int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldd,
                           int in_format, int out_dtype, float alpha, const gemm_options_t* opts,
                           cudaStream_t stream) {
    if (!is_fp8(in_format)) return GEMM_ERR_DTYPE;
    return run_impl(A, B, D, M, N, K, lda, ldb, ldd, in_format, out_dtype, alpha, 0, opts, nullptr,
                    0, stream, SA, SB, true);
}

extern "C" int gemm_mx_abt(const void* A, const void* B, const void* SA, const void* SB, void* D,
                           int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldd,
                           int in_format, int out_dtype, float alpha, cudaStream_t stream) {
    return gemm_mx_run(A, B, SA, SB, D, M, N, K, lda, ldb, ldd, in_format, out_dtype, alpha, nullptr,
                       stream);
}

extern "C" int gemm_mx_scales_size(int64_t rows, int64_t K, size_t* bytes) {
    if (!bytes) return GEMM_ERR_NULL;
    if (rows < 0 || K < 0 || rows > INT32_MAX || K > INT32_MAX) return GEMM_ERR_SHAPE;
    *bytes = size_t(mx_scale_bytes(rows, K));
    return GEMM_OK;
}

namespace gb300 {
namespace {

// Shared checks and launch of the two scale-packing kernels.
int pack_scales(const void* src, int64_t rows, int64_t K, int64_t ld, void* dst, bool for_b,
                cudaStream_t stream) {
    if (rows < 0 || K < 0 || rows > INT32_MAX || K > INT32_MAX) return GEMM_ERR_SHAPE;
    const int64_t groups = (K + 31) / 32;
    const int64_t bytes = for_b ? mx_scale_b_bytes(rows, K) : mx_scale_bytes(rows, K);
    if (bytes == 0) return GEMM_OK;
    if (!src || !dst) return GEMM_ERR_NULL;
    if (ld < groups || ld <= 0) return GEMM_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(dst) & 15u) return GEMM_ERR_ALIGN;
    if (overlaps(dst, 1, bytes, bytes, 1, src, rows, groups, ld, 1)) return GEMM_ERR_ALIAS;
    DeviceInfo di;
    const int st = current_device(&di);
    if (st != GEMM_OK) return st;
    const int64_t words = bytes / 4;
    int64_t blocks = (words + 255) / 256;
    if (blocks > 8L * di.sm_count) blocks = 8L * di.sm_count;
    if (for_b)
        mx_pack_scales_b_kernel<<<unsigned(blocks), 256, 0, stream>>>(
            static_cast<const uint8_t*>(src), rows, groups, ld, (K + 127) / 128,
            static_cast<uint32_t*>(dst), words);
    else
        mx_pack_scales_kernel<<<unsigned(blocks), 256, 0, stream>>>(
            static_cast<const uint8_t*>(src), rows, groups, ld, (K + 127) / 128,
            static_cast<uint32_t*>(dst), words);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace
}  // namespace gb300

extern "C" int gemm_mx_pack_scales(const void* src, int64_t rows, int64_t K, int64_t ld, void* dst,
                                   cudaStream_t stream) {
    return pack_scales(src, rows, K, ld, dst, false, stream);
}

extern "C" int gemm_mx_pack_scales_b(const void* src, int64_t N, int64_t K, int64_t ld, void* dst,
                                     cudaStream_t stream) {
    return pack_scales(src, N, K, ld, dst, true, stream);
}

extern "C" int gemm_mx_scales_b_size(int64_t N, int64_t K, size_t* bytes) {
    if (!bytes) return GEMM_ERR_NULL;
    if (N < 0 || K < 0 || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_SHAPE;
    *bytes = size_t(mx_scale_b_bytes(N, K));
    return GEMM_OK;
}

extern "C" int gemm_mx_plan(int64_t M, int64_t N, int64_t K, int in_format, const gemm_options_t* opts,
                            int* cta_group, int* block_m, int* block_n, int* stages,
                            int* num_clusters, int64_t* num_tiles, int* raster_group,
                            int* raster_order) {
    if (!is_fp8(in_format)) return GEMM_ERR_DTYPE;
    int st = check_sizes(M, N, K, in_format, 0);
    if (st != GEMM_OK) return st;
    if ((st = check_options(opts)) != GEMM_OK) return st;
    Plan p;
    if ((st = make_plan(M, N, K, in_format, 0, opts, false, &p, true)) != GEMM_OK) return st;
    if (cta_group) *cta_group = p.cg;
    if (block_m) *block_m = p.bm;
    if (block_n) *block_n = p.bn;
    if (stages) *stages = p.stages;
    if (num_clusters) *num_clusters = p.clusters;
    if (num_tiles) *num_tiles = p.tiles;
    if (raster_group) *raster_group = p.group;
    if (raster_order) *raster_order = p.order + 1;
    return GEMM_OK;
}

extern "C" int gemm_run(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldd, int dtype, int b_layout,
                        const gemm_options_t* opts, cudaStream_t stream) {
    return gemm_run_workspace(A, B, D, M, N, K, lda, ldb, ldd, dtype, b_layout, opts, nullptr, 0,
                              stream);
}

extern "C" int gemm_workspace_size(int64_t M, int64_t N, int64_t K, int dtype, int b_layout,
                                   const gemm_options_t* opts, size_t* bytes) {
    int st = check_sizes(M, N, K, dtype, b_layout);
    if (st != GEMM_OK) return st;
    if ((st = check_options(opts)) != GEMM_OK) return st;
    if (!bytes) return GEMM_ERR_NULL;
    *bytes = 0;
    if (M == 0 || N == 0 || K == 0) return GEMM_OK;
    Plan p;
    if ((st = make_plan(M, N, K, dtype, b_layout, opts, true, &p)) != GEMM_OK) return st;
    *bytes = workspace_bytes_needed(p);
    return GEMM_OK;
}

int gb300::split_workspace_layout(int64_t M, int64_t N, int64_t K, int dtype, int b_layout,
                                  const gemm_options_t* opts, size_t* counter_bytes,
                                  size_t* total_bytes) {
    int st = check_sizes(M, N, K, dtype, b_layout);
    if (st != GEMM_OK) return st;
    if ((st = check_options(opts)) != GEMM_OK) return st;
    if (!counter_bytes || !total_bytes) return GEMM_ERR_NULL;
    *counter_bytes = *total_bytes = 0;
    if (M == 0 || N == 0 || K == 0) return GEMM_OK;
    Plan p;
    if ((st = make_plan(M, N, K, dtype, b_layout, opts, true, &p)) != GEMM_OK) return st;
    *total_bytes = workspace_bytes_needed(p);
    *counter_bytes = p.split > 1 ? p.ws_counter_bytes : 0;
    return GEMM_OK;
}

extern "C" int gemm_abt(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldd, int dtype, cudaStream_t stream) {
    return gemm_run(A, B, D, M, N, K, lda, ldb, ldd, dtype, 0, nullptr, stream);
}

extern "C" int gemm_ab(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldd, int dtype, cudaStream_t stream) {
    return gemm_run(A, B, D, M, N, K, lda, ldb, ldd, dtype, 1, nullptr, stream);
}

extern "C" int gemm_plan(int64_t M, int64_t N, int64_t K, int dtype, int b_layout,
                         const gemm_options_t* opts, int* cta_group, int* block_m, int* block_n,
                         int* stages, int* num_clusters, int64_t* num_tiles, int* tail_split,
                         int* raster_group, int* raster_order, int* l2_hints, int* cluster_ksplit) {
    int st = check_sizes(M, N, K, dtype, b_layout);
    if (st != GEMM_OK) return st;
    if ((st = check_options(opts)) != GEMM_OK) return st;
    Plan p;
    if ((st = make_plan(M, N, K, dtype, b_layout, opts, true, &p)) != GEMM_OK) return st;
    if (cta_group) *cta_group = p.cg;
    if (block_m) *block_m = p.bm;
    if (block_n) *block_n = p.bn;
    if (stages) *stages = p.stages;
    if (num_clusters) *num_clusters = p.clusters;
    if (num_tiles) *num_tiles = p.tiles;
    if (tail_split) *tail_split = p.split;
    if (raster_group) *raster_group = p.group;
    if (raster_order) *raster_order = p.order + 1;
    if (l2_hints) *l2_hints = int(p.hints | 1u);
    if (cluster_ksplit) *cluster_ksplit = p.ks;
    return GEMM_OK;
}

extern "C" int gemm_tile_origin(int64_t M, int64_t N, int block_m, int block_n, int group,
                                int raster_order, int64_t task, int64_t* m0, int64_t* n0) {
    if (M <= 0 || N <= 0 || block_m <= 0 || block_n <= 0 || group <= 0 || M > INT32_MAX ||
        N > INT32_MAX)
        return GEMM_ERR_SHAPE;
    if (raster_order != 1 && raster_order != 2) return GEMM_ERR_OPTION;
    TileGrid g;
    g.m_tiles = int32_t((M + block_m - 1) / block_m);
    g.n_tiles = int32_t((N + block_n - 1) / block_n);
    g.group = group;
    g.order = raster_order - 1;
    if (tile_count(g) >= kMaxTiles || task < 0 || task >= tile_count(g)) return GEMM_ERR_SHAPE;
    int32_t mt, nt;
    tile_of_task(g, task, mt, nt);
    if (m0) *m0 = int64_t(mt) * block_m;
    if (n0) *n0 = int64_t(nt) * block_n;
    return GEMM_OK;
}

extern "C" int gemm_device_status(uint32_t* status, int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof v) != cudaSuccess) return GEMM_ERR_CUDA;
    if (clear) {
        const uint32_t zero = 0;
        if (cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof zero) != cudaSuccess) return GEMM_ERR_CUDA;
    }
    if (status) *status = v;
    return GEMM_OK;
}

extern "C" int gemm_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
    DeviceInfo di;
    const int st = current_device(&di);
    if (st != GEMM_OK) return st;
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

extern "C" int gemm_selftest_gemm_timeout(const void* A, const void* B, void* D, int64_t M,
                                          int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                          int64_t ldd, int dtype, int b_layout,
                                          const gemm_options_t* opts, uint64_t wait_limit_ns,
                                          cudaStream_t stream) {
    if (is_fp8(dtype)) return GEMM_ERR_DTYPE;
    return run_impl(A, B, D, M, N, K, lda, ldb, ldd, dtype, dtype, 1.0f, b_layout, opts, nullptr, 0,
                    stream, nullptr, nullptr, false, wait_limit_ns);
}

extern "C" int gemm_run_clock_probe(const void* A, const void* B, void* D, int64_t M, int64_t N,
                                    int64_t K, int64_t lda, int64_t ldb, int64_t ldd, int dtype,
                                    int b_layout, const gemm_options_t* opts,
                                    unsigned long long* probe, cudaStream_t stream) {
    if (is_fp8(dtype)) return GEMM_ERR_DTYPE;
    if (!probe) return GEMM_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(probe) & 7u) return GEMM_ERR_ALIGN;
    return run_impl(A, B, D, M, N, K, lda, ldb, ldd, dtype, dtype, 1.0f, b_layout, opts, nullptr, 0,
                    stream, nullptr, nullptr, false, kWaitLimitNs, probe);
}

extern "C" const char* gemm_status_string(int status) {
    switch (status) {
        case GEMM_OK: return "ok";
        case GEMM_ERR_NULL: return "null pointer";
        case GEMM_ERR_DTYPE: return "unsupported dtype (GEMM_F16 or GEMM_BF16)";
        case GEMM_ERR_SHAPE: return "invalid size or leading dimension";
        case GEMM_ERR_ALIGN: return "pointer not 16-byte aligned or leading dimension not a multiple of 8";
        case GEMM_ERR_ALIAS: return "output overlaps an input";
        case GEMM_ERR_CUDA: return "CUDA call failed";
        case GEMM_ERR_DEVICE: return "current device is not an sm_103 GPU";
        case GEMM_ERR_OPTION: return "unsupported option";
        case GEMM_ERR_TIMEOUT: return "a kernel wait timed out";
        case GEMM_ERR_WORKSPACE: return "workspace smaller than gemm_workspace_size() or not 256-byte aligned";
        default: return "unknown status";
    }
}
