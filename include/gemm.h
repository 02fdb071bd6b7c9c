/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library (libgb300gemm.so).
 *
 * The operation ("TIRx GEMM on Blackwell", section "The short version"):
 *
 *     D = A . B^T      A: M x K, B: N x K, D: M x N            (gemm_abt)
 *     D = A . B        A: M x K, B: K x N, D: M x N            (gemm_ab)
 *
 * The A.B form is the program of "Choosing schedules and instructions for a
 * backend" (TileFoundry tutorial), section 1: gemm(a: (M, K), b: (K, N)).
 *
 * A, B and D share one 16-bit storage type (FP16 or BF16).  Products are
 * accumulated in FP32 in Blackwell Tensor Memory and each output is rounded
 * once (round to nearest even) to the 16-bit type.  The order of the FP32
 * additions is unspecified: it depends on the tiling, not on the values.
 *
 * Layout.  Every matrix is row-major with a leading dimension (row stride)
 * given in ELEMENTS: element (i, j) of A is A[i * lda + j].  Requirements,
 * which come from the Tensor Memory Accelerator that moves every tile:
 *   - A, B and D are device pointers, 16-byte aligned;
 *   - lda, ldb and ldd are multiples of 8 elements (16 bytes);
 *   - lda >= K, ldb >= K (gemm_abt) or ldb >= N (gemm_ab), ldd >= N;
 *   - M, N and K are at most 2^31 - 1.
 * Violations return an error code; nothing is launched.  There is no slower
 * fallback path.
 *
 * Ownership.  The caller allocates and owns A, B, D (and the optional
 * workspace of gemm_run_workspace).  The library allocates no device memory
 * on any call: tile descriptors travel as kernel parameters.
 * D is written and never read, so it need not be initialised.  D must not
 * overlap A or B (GEMM_ERR_ALIAS).
 *
 * Stream semantics.  Work is enqueued on `stream` (0 = the legacy default
 * stream) and the call returns without synchronising; results are visible to
 * later work on the same stream.  The current CUDA device must be the device
 * that holds the buffers.
 *
 * Degenerate sizes.  M == 0 or N == 0: nothing to do, returns GEMM_OK.
 * K == 0: D is filled with zeros (the empty sum), as torch.mm does.
 *
 * Errors.  Every entry point returns GEMM_OK (0) or a negative status;
 * gemm_status_string() gives its text.  A launch error is GEMM_ERR_CUDA.
 * Errors that occur while the kernel runs are reported asynchronously through
 * gemm_device_status() (see below).
 */
#ifndef GB300_GEMM_H
#define GB300_GEMM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  GEMM_F16 / GEMM_BF16 are the 16-bit input and output types
 * of gemm_abt / gemm_ab / gemm_run.  GEMM_E4M3 / GEMM_E5M2 are the 8-bit input
 * formats of the gemm_fp8_* entry points (OCP 8-bit floating point: E4M3 =
 * 1 sign, 4 exponent bits with bias 7, 3 fraction bits, no infinities, NaN =
 * S.1111.111; E5M2 = 1 sign, 5 exponent bits with bias 15, 2 fraction bits,
 * IEEE-style inf/NaN); gemm_plan and gemm_workspace_size accept them as
 * `dtype` to describe an FP8 call. */
typedef enum { GEMM_F16 = 0, GEMM_BF16 = 1, GEMM_E4M3 = 2, GEMM_E5M2 = 3 } gemm_dtype_t;

enum {
    GEMM_OK = 0,
    GEMM_ERR_NULL = -1,    /* a null pointer with a non-empty extent           */
    GEMM_ERR_DTYPE = -2,   /* an element type the entry point does not take     */
    GEMM_ERR_SHAPE = -3,   /* negative or too-large size, or ld < row length   */
    GEMM_ERR_ALIGN = -4,   /* pointer not 16-B aligned or ld*elem not 16-B multiple */
    GEMM_ERR_ALIAS = -5,   /* D overlaps A or B                                 */
    GEMM_ERR_CUDA = -6,    /* a CUDA runtime or driver call failed              */
    GEMM_ERR_DEVICE = -7,  /* the current device is not an sm_103 GPU           */
    GEMM_ERR_OPTION = -8,  /* an unsupported gemm_options_t value               */
    GEMM_ERR_TIMEOUT = -9, /* a kernel wait gave up (see gemm_device_status)    */
    GEMM_ERR_WORKSPACE = -10 /* workspace too small or not 256-byte aligned     */
};

/* D[M x N] = A[M x K] . B[N x K]^T, all row-major (ld in elements). */
int gemm_abt(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
             int64_t lda, int64_t ldb, int64_t ldd, int dtype, cudaStream_t stream);

/* D[M x N] = A[M x K] . B[K x N], all row-major (ld in elements). */
int gemm_ab(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
            int64_t lda, int64_t ldb, int64_t ldd, int dtype, cudaStream_t stream);

/* Text for a status code; never NULL, static storage. */
const char* gemm_status_string(int status);

/*
 * Tuning and test controls.  gemm_abt/gemm_ab are gemm_run with opts = NULL.
 * An all-zero gemm_options_t means "automatic" for every field.
 *   cta_group     0 = automatic, 1 = one CTA per 128-row tile (tcgen05
 *                 cta_group::1), 2 = a 2-CTA cluster per 256-row tile
 *                 (cta_group::2, the two CTAs' tensor cores act as one).
 *   block_n       0 = automatic, else the N extent of a tile: 32 or 64
 *                 (1-CTA tiles: cta_group 2 with them is GEMM_ERR_OPTION;
 *                 32 with B N x K only), 128, 192 or 224 (B N x K only) or
 *                 256.  Narrow tiles spread a small problem over more SMs:
 *                 the automatic plan takes them (32 wide, else 64) for
 *                 16-bit problems of 8 to 63 64-wide K blocks whose 128-wide
 *                 1-CTA tiles fit in one round and that still do.
 *   raster_group  0 = automatic, else the number of tiles per raster group
 *                 of the persistent scheduler, counted along the grouped
 *                 dimension (see raster_order).
 *   raster_order  0 = automatic.  1 = groups of raster_group M tiles: tiles
 *                 are visited group by group, and inside a group the N tiles
 *                 in order with the group's M tiles innermost, so tiles that
 *                 run at the same time share B's column panel and the band
 *                 of A rows stays in L2 while the group walks N ("Choosing
 *                 schedules and instructions for a backend", section 3).
 *                 2 = the same with M and N exchanged: groups of N tiles, a
 *                 band of B columns stays in L2 while the group walks M.
 *   max_clusters  0 = as many co-resident clusters as fit, else an upper bound
 *                 on the persistent grid (in clusters).
 *   tail_split    0 = automatic: a balanced grid (the persistent schedule's
 *                 rounds spread over the fewest clusters that keep the same
 *                 round count, so no cluster idles in a partial last round);
 *                 with a workspace (gemm_run_workspace), a problem whose
 *                 tiles all fit in one round with clusters to spare also
 *                 splits every tile's K loop into s ranges over the idle
 *                 clusters (s <= clusters / tiles, at least 64 k-blocks per
 *                 range: the partials' fix-up costs a few microseconds).  1 = never split.  s in [2, 16], only with a
 *                 workspace: split each tile of the last, partial round (of
 *                 a single-round problem: every tile) into s K-ranges
 *                 (capped by the number of k-blocks and, for a single
 *                 round, by clusters / tiles).
 *   consumers     0 or 1 = one MMA accumulator per CTA and tile, two TMEM
 *                 accumulator slots so the epilogue of one tile overlaps the
 *                 next tile's MMAs.  2 = two accumulators per CTA that share
 *                 each staged B tile ("TIRx GEMM on Blackwell", V9): each CTA
 *                 holds 256 rows of A, a tile is 512 x 256 (cta_group 2 and
 *                 block_n 256 only), operand traffic per FLOP drops by a
 *                 quarter, and the two accumulators fill TMEM, so a tile's
 *                 epilogue no longer overlaps the next tile's MMAs.
 *   multicast     must be 0 or 1 (GEMM_ERR_OPTION otherwise): a cluster is
 *                 always the CTAs of one tile, and every CTA loads its own
 *                 operand tiles (no load is multicast to other CTAs).
 *   l2_hints      0 = automatic.  Otherwise an odd value (bit 0 marks the
 *                 choice as explicit; an even non-zero value is
 *                 GEMM_ERR_OPTION) whose other bits set L2 eviction
 *                 priorities: 2 = A's loads evict_last, 4 = B's loads
 *                 evict_first, 8 = D's stores evict_first (1 = no hints).
 *   cluster_ksplit  0 = automatic, 1 = never, 2 or 4 = that many K-ranges per
 *                 tile inside a cluster: a problem whose 1-CTA tiles (128
 *                 wide; 256 wide with 2 ranges) all fit in one round of such
 *                 clusters has each tile computed by a cluster of that many
 *                 CTAs, one K-range each; each CTA owns an equal share of the
 *                 tile's columns, receives the others' FP32 partials of them
 *                 through distributed shared memory and stores their sum,
 *                 taken in CTA order (no workspace).  Automatic: when K has
 *                 at least 64 of its 64-wide blocks, the most ranges that
 *                 keep at least 16 blocks per range, unless the workspace
 *                 split (tail_split) would run more ranges per tile.  16-bit
 *                 inputs only.
 */
typedef struct {
    int cta_group;
    int block_n;
    int raster_group;
    int max_clusters;
    int tail_split;
    int consumers;
    int multicast;
    int raster_order;
    int l2_hints;
    int cluster_ksplit;
} gemm_options_t;

/* b_layout: 0 = B is N x K (D = A.B^T), 1 = B is K x N (D = A.B). */
int gemm_run(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
             int64_t lda, int64_t ldb, int64_t ldd, int dtype, int b_layout,
             const gemm_options_t* opts, cudaStream_t stream);

/*
 * The same GEMM with a caller-owned device workspace, which lets the kernel
 * split the K loop of tiles that would leave clusters idle.  A problem whose
 * T tiles fit in one round of C co-resident clusters with clusters to spare
 * is split automatically: each tile into s <= C / T K-ranges.  The last,
 * partial round of a longer schedule is split on request
 * (gemm_options_t.tail_split = s >= 2): its T mod C tiles are each split into
 * s K-ranges so the clusters that would idle share the work.  Each range writes an FP32
 * partial to the workspace; the range that finishes last (found with an
 * atomic counter, nobody waits) adds the partials in range order and writes D.
 * Results are deterministic for a given plan.
 *
 * workspace        device memory, 256-byte aligned, at least
 *                  gemm_workspace_size() bytes (0 means no split will happen
 *                  for these sizes).  Zero it once before its first use;
 *                  afterwards it may be reused by any number of calls, because
 *                  every launch tags its counters with a fresh launch number.
 *                  A launch replayed from a CUDA graph repeats its number, so
 *                  after a launch that ended with a non-zero
 *                  gemm_device_status() (a wait that gave up may leave its
 *                  counters half-counted) zero the workspace again before the
 *                  graph is replayed.
 *                  Calls that share a workspace must not run concurrently
 *                  (different streams): they would race on it.
 * workspace = NULL runs the plain persistent schedule (as gemm_run).
 * Returns GEMM_ERR_WORKSPACE if the workspace is too small or misaligned.
 */
int gemm_run_workspace(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldd, int dtype, int b_layout,
                       const gemm_options_t* opts, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/*
 * FP8 GEMM: D[M x N] = alpha * A[M x K] . B[N x K]^T, A and B FP8 (in_format
 * GEMM_E4M3 or GEMM_E5M2, both operands in the same format), D 16-bit
 * (out_dtype GEMM_F16 or GEMM_BF16), all row-major with ld in elements.
 *
 * The operation is the FP8 GEMM of "TIRx: A Unified Tile Primitive ML
 * Compiler" (kernel performance: FP8 matrix multiplication with scale
 * factors that adjust the values' range), here with ONE scale for the whole
 * product (alpha, e.g. scale_A * scale_B of per-tensor scaling); the operands
 * are K-major as "Choosing schedules and instructions for a backend"
 * requires of fp8e4m3 (instruction table).  Products accumulate in FP32 in
 * tensor memory (tcgen05.mma kind::f8f6f4); alpha multiplies the FP32 sum,
 * which is then rounded once (nearest even) to out_dtype.
 *
 * Arguments and errors as gemm_run, except: A and B are byte arrays, so lda
 * and ldb must be multiples of 16 (TMA row strides are 16-byte multiples;
 * GEMM_ERR_ALIGN otherwise); ldd a multiple of 8.  Options: cta_group,
 * block_n (0, 256, or 224 with 2-CTA tiles), raster_group, max_clusters and
 * tail_split as for gemm_run; consumers and multicast must be 0 or 1
 * (GEMM_ERR_OPTION otherwise).  A 16-bit in_format gives GEMM_ERR_DTYPE.
 * K = 0 writes zeros; M = 0 or N = 0 does nothing.  No library allocation;
 * gemm_fp8_run_workspace takes a workspace exactly as gemm_run_workspace.
 */
int gemm_fp8_abt(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                 int64_t lda, int64_t ldb, int64_t ldd, int in_format, int out_dtype,
                 float alpha, cudaStream_t stream);
int gemm_fp8_run(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                 int64_t lda, int64_t ldb, int64_t ldd, int in_format, int out_dtype,
                 float alpha, const gemm_options_t* opts, cudaStream_t stream);
int gemm_fp8_run_workspace(const void* A, const void* B, void* D, int64_t M, int64_t N,
                           int64_t K, int64_t lda, int64_t ldb, int64_t ldd, int in_format,
                           int out_dtype, float alpha, const gemm_options_t* opts,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Block-scaled FP8 GEMM (MX):
 *
 *   D[i,j] = alpha * sum_k (A[i,k] * 2^(sa[i][k/32] - 127)) * (B[j,k] * 2^(sb[j][k/32] - 127))
 *
 * A (M x K) and B (N x K) FP8 (in_format GEMM_E4M3 or GEMM_E5M2), row-major
 * with ld in elements as for gemm_fp8_run; D 16-bit (out_dtype GEMM_F16 or
 * GEMM_BF16).  "TIRx: A Unified Tile Primitive ML Compiler" (kernel
 * performance) names FP8 block-scaled matrix multiplication, in which groups
 * of input values share scale factors; the page fixes neither the group nor
 * the scale encoding, and this library takes the OCP Microscaling (MX)
 * reading that the tcgen05.mma kind::mxf8f6f4 instruction implements: every
 * run of 32 consecutive K elements of a row of A and of a row of B shares one
 * scale byte in the UE8M0 encoding (value 2^(x - 127); x = 255 is NaN).
 * Products and scales are applied in the tensor core, the sum accumulates in
 * FP32 in tensor memory, alpha multiplies it, and the result is rounded once
 * (nearest even) to out_dtype.
 *
 * Scale layouts.  SA and SB are device buffers, 16-byte aligned, owned by the
 * caller, not overlapping D; padding bytes (rows or columns past the matrix,
 * K groups past ceil(K / 32)) must not be 255.
 *   SA, the scales of A: gemm_mx_scales_size(M, K) bytes, ceil(M / 128) x
 *   ceil(K / 128) atoms of 512 bytes, atom (rb, kc) at byte offset
 *   (rb * ceil(K / 128) + kc) * 512; inside an atom the scale of row
 *   rb * 128 + r and K group kc * 4 + g (elements 32 (kc * 4 + g) .. +31) is
 *   the byte at (r % 32) * 16 + (r / 32) * 4 + g.  gemm_mx_pack_scales()
 *   writes it from row-major scales.
 *   SB, the scales of B, pre-laid-out for this library's 224-column tiles:
 *   gemm_mx_scales_b_size(N, K) bytes, ceil(N / 224) x ceil(K / 128) blocks
 *   of 4096 bytes, block (t, kc) at byte offset (t * ceil(K / 128) + kc) *
 *   4096; inside a block the scale of column 224 t + 32 c + l (c < 7,
 *   l < 32) and K group kc * 4 + g is the byte at (r / 8) * 256 + (r % 8) * 16
 *   + (c / 4) * 128 + (c % 4) * 4 + g for each r in {l, l + 32, l + 64,
 *   l + 96} (four copies; c = 7 is padding).  This is the image of the tile's
 *   scales that the tensor core copies into tensor memory, so the kernel loads
 *   it in one piece.  gemm_mx_pack_scales_b() writes it from row-major scales.
 *
 * Options: cta_group 0 or 2, block_n 0 or 224, raster_group and
 * max_clusters as for gemm_run; consumers, multicast and tail_split 0 or 1
 * (GEMM_ERR_OPTION otherwise).  Errors as gemm_fp8_run, plus GEMM_ERR_NULL
 * for a null SA or SB and GEMM_ERR_ALIGN for a misaligned one (when K > 0).
 * K = 0 writes zeros; M = 0 or N = 0 does nothing.  No library allocation.
 */
int gemm_mx_abt(const void* A, const void* B, const void* SA, const void* SB, void* D,
                int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldd,
                int in_format, int out_dtype, float alpha, cudaStream_t stream);
int gemm_mx_run(const void* A, const void* B, const void* SA, const void* SB, void* D,
                int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldd,
                int in_format, int out_dtype, float alpha, const gemm_options_t* opts,
                cudaStream_t stream);

/* Bytes of SA for a rows x K operand: ceil(rows / 128) * ceil(K / 128) * 512
 * (written to *bytes). */
int gemm_mx_scales_size(int64_t rows, int64_t K, size_t* bytes);

/* Bytes of SB for an N x K operand: ceil(N / 224) * ceil(K / 128) * 4096. */
int gemm_mx_scales_b_size(int64_t N, int64_t K, size_t* bytes);

/*
 * Tiled scales (the layout above) from row-major ones: src is a device buffer
 * of rows x ceil(K / 32) scale bytes with row stride ld bytes (ld >=
 * ceil(K / 32)); dst (gemm_mx_scales_size(rows, K) bytes, 16-byte aligned,
 * not overlapping src) receives the tiled layout, padding bytes set to 127.
 * One kernel on `stream`, asynchronous.  Errors: GEMM_ERR_SHAPE, _NULL,
 * _ALIGN, _ALIAS, _DEVICE, _CUDA.
 */
int gemm_mx_pack_scales(const void* src, int64_t rows, int64_t K, int64_t ld, void* dst,
                        cudaStream_t stream);

/* SB (the layout above) from row-major scales: as gemm_mx_pack_scales, with
 * rows = N and dst of gemm_mx_scales_b_size(N, K) bytes. */
int gemm_mx_pack_scales_b(const void* src, int64_t N, int64_t K, int64_t ld, void* dst,
                          cudaStream_t stream);

/* The plan gemm_mx_run would use (outputs as gemm_plan; may be NULL). */
int gemm_mx_plan(int64_t M, int64_t N, int64_t K, int in_format, const gemm_options_t* opts,
                 int* cta_group, int* block_m, int* block_n, int* stages, int* num_clusters,
                 int64_t* num_tiles, int* raster_group, int* raster_order);

/*
 * Bytes of workspace gemm_run_workspace needs for these sizes and options on
 * the current device (written to *bytes; 0 = the call would not split).  At
 * most (co-resident clusters) x 256 KiB plus a few KiB of counters.
 */
int gemm_workspace_size(int64_t M, int64_t N, int64_t K, int dtype, int b_layout,
                        const gemm_options_t* opts, size_t* bytes);

/*
 * gemm_run_workspace for callers that cannot allocate device memory: a plugin
 * inside a host framework whose memory manager owns all device memory and
 * must account for every byte; a latency-critical loop, where cudaMalloc or
 * cudaFree can synchronise the device and stall every stream; a process whose
 * device-memory budget is fixed at start-up.  The pages describe no
 * counterpart: it is an addition of this library.
 *
 * The split tail's workspace is a fixed 20 MiB scratch array compiled into
 * the library (a file-scope __device__ array); every GPU that loads the
 * library holds one until the process exits.  The caller passes A, B and D
 * as for gemm_run; no memory is allocated and no allocating routine is
 * called.  A plan that needs more than 20 MiB (a tail_split s with
 * (T mod C) x s larger than the cluster count C) returns GEMM_ERR_WORKSPACE;
 * s <= C / (T mod C), and every automatic split, always fits on a 152-SM
 * GB300.
 *
 * The first call on each device looks up the scratch's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  All calls on a device share the one scratch
 * array, which keeps the last call's contents: a call whose plan splits
 * clears the split tail's counter words first (cudaMemsetAsync on `stream`),
 * and calls that overlap on the GPU (different streams) race on the array
 * and must be serialised by the caller.
 */
int gemm_run_no_alloc(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldd, int dtype, int b_layout,
                      const gemm_options_t* opts, cudaStream_t stream);

/*
 * Plan of a call, without launching: the tile shape, grid, stage count, tail
 * split, raster group and order (1 = M groups, 2 = N groups, as the
 * options), L2 hints (an explicit, odd l2_hints value) and in-cluster K
 * ranges per tile (1 = none) that
 * gemm_run_workspace (with a large enough workspace) would use for these
 * sizes on the current device.  Any out pointer may be NULL.  Returns the
 * same argument errors as gemm_run (pointers are not checked).
 */
int gemm_plan(int64_t M, int64_t N, int64_t K, int dtype, int b_layout,
              const gemm_options_t* opts, int* cta_group, int* block_m, int* block_n,
              int* stages, int* num_clusters, int64_t* num_tiles, int* tail_split,
              int* raster_group, int* raster_order, int* l2_hints, int* cluster_ksplit);

/*
 * The persistent scheduler's task -> tile map (the same function the kernel
 * runs), for host-side checks.  Tiles of block_m x block_n cover the M x N
 * output; `group` tiles along M (raster_order 1) or along N (raster_order 2)
 * form a raster group.  Writes the tile's first row and column.  Returns
 * GEMM_ERR_SHAPE if task is outside [0, tiles) or if there are 2^31 tiles or
 * more (the scheduler's index arithmetic is 32-bit; gemm_run rejects such
 * sizes with the same error), GEMM_ERR_OPTION for another raster_order.
 */
int gemm_tile_origin(int64_t M, int64_t N, int block_m, int block_n, int group,
                     int raster_order, int64_t task, int64_t* m0, int64_t* n0);

/*
 * Device-side error word of the current device.  Every wait inside the kernel
 * is bounded (about 2 s); a wait that runs out makes the kernel record the
 * reason here, end all of its loops, release Tensor Memory and return, so the
 * CUDA context stays usable.  The word is bits 0-7 = reason (1 = timeout),
 * bits 8-15 = role that gave up (1 producer, 2 MMA issuer, 3 epilogue,
 * 4 end-of-kernel drain, 5 self-test); reason 2 = a split-tail counter could
 * not be updated.  Synchronises the device, then writes the word
 * to *status (0 = no error since the last clear) and clears it if `clear`.
 * Returns GEMM_OK or GEMM_ERR_CUDA.
 */
int gemm_device_status(uint32_t* status, int clear);

/*
 * Self-test of that failure path.  Launches one thread that waits, through
 * the same bounded wait the GEMM kernel uses, on an mbarrier that nothing
 * ever arrives on, with a limit of `limit_ns` nanoseconds.  The wait runs
 * out and records 0x501 (reason 1 = timeout, role 5 = self-test) in the
 * device status word; the context stays usable.  Touches no user memory.
 * Returns GEMM_OK once launched, GEMM_ERR_DEVICE or GEMM_ERR_CUDA otherwise.
 */
int gemm_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

/*
 * Self-test of the GEMM kernel's own abort path: gemm_run(A, B, D, ...) with
 * every barrier wait of the kernel limited to `wait_limit_ns` nanoseconds
 * instead of about 2 s.  With a limit far below the time the first operands
 * take to arrive (e.g. 100 ns), a wait gives up: the kernel records
 * reason 1 (timeout) and the role that gave up in the device status word,
 * raises the abort flag in both CTAs of every pair that sees it, leaves all
 * loops, waits 1 ms for work already in flight, frees Tensor Memory and
 * returns; the CUDA context stays usable and later calls run normally.  D's
 * contents are unspecified afterwards (tiles may be partly written).
 * Arguments and errors as gemm_run (16-bit types only).
 */
int gemm_selftest_gemm_timeout(const void* A, const void* B, void* D, int64_t M, int64_t N,
                               int64_t K, int64_t lda, int64_t ldb, int64_t ldd, int dtype,
                               int b_layout, const gemm_options_t* opts, uint64_t wait_limit_ns,
                               cudaStream_t stream);

/*
 * Diagnostic: gemm_run(A, B, D, ...) whose first CTA also records, in
 * `probe` (a device buffer of four 8-byte words, 8-byte aligned), the SM's
 * clock counter (%clock64) and the global nanosecond timer (%globaltimer) at
 * its start (probe[0], probe[1]) and at its end (probe[2], probe[3]).
 * (probe[2] - probe[0]) / (probe[3] - probe[1]) is the SM clock, in GHz,
 * that the kernel ran at, which a driver query sampled from the host may not
 * show.  Nothing else differs from gemm_run; 16-bit types only.  Errors as
 * gemm_run, plus GEMM_ERR_NULL / GEMM_ERR_ALIGN for the probe buffer.  The
 * operation has no counterpart on the pages: it is a measurement aid.
 */
int gemm_run_clock_probe(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                         int64_t lda, int64_t ldb, int64_t ldd, int dtype, int b_layout,
                         const gemm_options_t* opts, unsigned long long* probe,
                         cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_H */
