// gemm_no_alloc.cu -- gemm_run_no_alloc(): the GEMM for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc (or any allocator) where they run a
// GEMM: a plugin inside a host framework whose memory manager owns the whole
// device memory and must account for every byte (a raw allocation there can
// fail, or push the framework's own pool out of memory); a latency-critical
// loop, where cudaMalloc / cudaFree can synchronise the device and stall
// every stream; a process whose device-memory budget is fixed and fully
// partitioned at start-up.  gemm_run_workspace needs a caller-owned workspace
// for its split tail; this entry point uses a fixed scratch array compiled
// into the library instead, so the caller passes only A, B and D.
//
// The scratch is a file-scope device array of kNoAllocScratchBytes (20 MiB);
// every GPU that loads the library holds its own copy until the process
// exits.  20 MiB covers any split that gives each cluster at most one K-range
// on a 152-SM GB300 (76 two-CTA clusters: at most one 256 KiB FP32 partial per
// cluster, plus counters); plans that need more (a deeper tail_split) are
// rejected with GEMM_ERR_WORKSPACE.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gemm.h"
#include "workspace.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(20) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol, not a device address: the address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Set-up, inside the first call on each device (that device is current then):
// look up the scratch's device address.  No memory is allocated or written.
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || !p) return GEMM_ERR_CUDA;
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
    size_t counters = 0, need = 0;
    int st = gb300::split_workspace_layout(M, N, K, dtype, b_layout, opts, &counters, &need);
    if (st != GEMM_OK) return st;
    if (need > kNoAllocScratchBytes) return GEMM_ERR_WORKSPACE;
    void* scratch = nullptr;
    if ((st = scratch_for_current_device(&scratch)) != GEMM_OK) return st;
    // The scratch keeps whatever the previous call left.  The split tail's
    // counter words must start at zero (the FP32 partials behind them are
    // written before they are read), so clear them on the caller's stream,
    // ahead of this call's kernel.
    if (counters > 0 && cudaMemsetAsync(scratch, 0, counters, stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
    return gemm_run_workspace(A, B, D, M, N, K, lda, ldb, ldd, dtype, b_layout, opts, scratch,
                              kNoAllocScratchBytes, stream);
}
