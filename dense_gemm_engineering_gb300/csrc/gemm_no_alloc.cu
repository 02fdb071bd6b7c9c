// gemm_no_alloc.cu -- gemm_run_no_alloc(): the GEMM for callers that cannot
// allocate device memory.
//
// Some callers must not call cudaMalloc (or any allocator) at the point where
// they run a GEMM: code recorded into a CUDA graph or run under a strict
// memory budget, plugins inside a host framework that owns every allocation,
// real-time loops where an allocation can block or fail.  gemm_run_workspace
// needs a caller-owned workspace for its split tail; this entry point instead
// uses a fixed scratch array compiled into the library, so the caller passes
// only A, B and D.
//
// The scratch is a file-scope device array of kNoAllocScratchBytes (20 MiB).
// Every GPU that loads the library holds its own copy until the process exits.
// 20 MiB covers any split that gives each cluster at most one K-range on a
// 152-SM GB300 (76 two-CTA clusters: at most one 256 KiB FP32 partial per
// cluster, plus counters); plans that need more (a deeper tail_split) are
// rejected with GEMM_ERR_WORKSPACE.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gemm.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(20) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol: its address must be obtained with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Once per device, with that device current: look up the scratch's device
// address and zero it (the split tail's counters must not start out looking
// like those of a live launch).  Runs inside the first call on each device.
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || !p) return GEMM_ERR_CUDA;
        if (cudaMemset(p, 0, kNoAllocScratchBytes) != cudaSuccess) return GEMM_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GEMM_OK;
}

}  // namespace

extern "C" int gemm_run_no_alloc(const void* A, const void* B, void* D, int64_t M, int64_t N,
                                 int64_t K, int64_t lda, int64_t ldb, int64_t ldd, int dtype,
                                 int b_layout, const gemm_options_t* opts, cudaStream_t stream) {
    // Size and option errors first; then the plan's scratch need.
    size_t need = 0;
    int st = gemm_workspace_size(M, N, K, dtype, b_layout, opts, &need);
    if (st != GEMM_OK) return st;
    if (need > kNoAllocScratchBytes) return GEMM_ERR_WORKSPACE;
    void* scratch = nullptr;
    if ((st = scratch_for_current_device(&scratch)) != GEMM_OK) return st;
    return gemm_run_workspace(A, B, D, M, N, K, lda, ldb, ldd, dtype, b_layout, opts, scratch,
                              kNoAllocScratchBytes, stream);
}
