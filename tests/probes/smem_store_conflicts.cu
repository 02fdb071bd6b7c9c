// smem_store_conflicts.cu -- shared-memory bank-conflict probe for the GEMM
// epilogue's staging stores.
//
// The epilogue writes each 32 x 64 block of 16-bit outputs into a 128-byte
// swizzled staging tile: lane r stores the 16-byte chunk c of its row at chunk
// position c ^ (r % 8), so the eight lanes of each quarter-warp phase of a
// st.shared.v4 cover all 32 banks.  probe<false> runs exactly that pattern
// (four warps, two 4 KiB buffers each, as the epilogue) and nothing else;
// probe<true> runs it while one thread streams 16 KiB bulk copies
// (cp.async.bulk, global -> shared) into another part of the same SM's shared
// memory, as the operand ring's TMA loads do during the GEMM.  Profiled with
//   l1tex__data_bank_conflicts_pipe_lsu_mem_shared_op_st.sum,
//   l1tex__data_pipe_lsu_wavefronts_mem_shared_op_st.sum,
//   smsp__inst_executed_op_shared_st.sum
// it separates conflicts of the address pattern (probe<false>: the minimum of
// four wavefronts per 512-byte store) from contention with asynchronous writes
// (probe<true>).  Every wait is bounded and every address stays inside the
// 200 KiB of dynamic shared memory the launch requests.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void st4(uint32_t a, uint32_t x) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(x + 1), "r"(x + 2), "r"(x + 3) : "memory");
}

// warps 1..4 store; warp 0 (kernel 2 only) streams bulk copies into [32 KB, 96 KB)
template <bool COPIES>
__global__ void probe(int iters, const uint8_t* src, unsigned* sink) {
    extern __shared__ __align__(1024) uint8_t sm[];
    const uint32_t base = saddr(sm);
    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == 0) {
        if (COPIES && lane == 0) {
            uint32_t ph = 0;
            for (int i = 0; i < iters / 4; ++i) {
                const uint32_t dst = base + 32768u + uint32_t(i % 4) * 16384u;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(&bar)), "r"(16384u) : "memory");
                asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                             ::"r"(dst), "l"(src + size_t(i % 64) * 16384u), "r"(16384u), "r"(saddr(&bar)) : "memory");
                uint32_t done = 0;
                for (long spin = 0; spin < 20000000L && !done; ++spin) {
                    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                                 : "=r"(done) : "r"(saddr(&bar)), "r"(ph) : "memory");
                }
                if (!done) { sink[gridDim.x + blockIdx.x] = 0xdead; break; }
                ph ^= 1u;
            }
        }
        return;
    }
    const uint32_t buf = base + (warp - 1) * 8192u;  // two 4 KB staging buffers per warp, as the epilogue
    uint32_t v = threadIdx.x;
    for (int it = 0; it < iters; ++it) {
        const uint32_t b = buf + uint32_t(it & 1) * 4096u + lane * 128u;
#pragma unroll
        for (int c = 0; c < 8; ++c) st4(b + ((uint32_t(c) ^ (lane & 7u)) << 4), v + c);
        __syncwarp();
        ++v;
    }
    if (lane == 0) atomicAdd(&sink[blockIdx.x], v);
}

int main() {
    uint8_t* src; unsigned* sink;
    cudaMalloc(&src, 64 * 16384); cudaMemset(src, 1, 64 * 16384);
    cudaMalloc(&sink, 2 * 152 * sizeof(unsigned)); cudaMemset(sink, 0, 2 * 152 * sizeof(unsigned));
    const int smem = 200 * 1024;  // one block per SM
    cudaFuncSetAttribute(probe<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(probe<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    probe<false><<<152, 160, smem>>>(4000, src, sink);
    probe<true><<<152, 160, smem>>>(4000, src, sink);
    cudaError_t e = cudaDeviceSynchronize();
    unsigned h[2 * 152];
    cudaMemcpy(h, sink, sizeof h, cudaMemcpyDeviceToHost);
    int bad = 0;
    for (int i = 152; i < 304; ++i) bad += (h[i] == 0xdead);
    printf("status %s, copy waits that ran out: %d\n", cudaGetErrorString(e), bad);
    return e == cudaSuccess ? 0 : 1;
}
