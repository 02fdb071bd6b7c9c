// cluster_exchange.cu -- throughput of an exchange of FP32 pieces between the
// CTAs of a cluster, the step with which the GEMM's in-cluster K split sums its
// K-ranges.
//
// KS CTAs per cluster (2 or 4; 152 CTAs in all), four warps each, as the
// epilogue's lane quarters.  In every repetition warp q of each CTA sends one
// piece of BYTES = 32 rows x W FP32 columns to each other CTA of its cluster,
// the receiver waits until all KS - 1 pieces of its quarter are in and reads
// them, and the cluster synchronises.  Modes:
//   0  st.shared::cluster.v4 stores from registers, fence.acq_rel.cluster,
//      an arrival on the receiver's barrier
//   1  one cp.async.bulk shared::cta -> shared::cluster copy per piece,
//      completing as transaction bytes on the receiver's barrier
//   2  local st.shared.v4 of the same bytes (no exchange: the baseline of a
//      repetition's fixed costs)
//   3  st.global to a per-CTA slot, a fence and a cluster barrier, then
//      ld.global.cg by the receiver (an exchange through L2)
// It prints the mean time per repetition (clock64 and %globaltimer) and the
// bytes sent per CTA per cycle.  Every barrier wait is bounded (its give-ups
// are counted and printed); every address stays inside the dynamic shared
// memory each launch requests and the global buffer main() allocates.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint32_t mapa(uint32_t a, uint32_t r) {
    uint32_t o; asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(o) : "r"(a), "r"(r)); return o;
}
__device__ __forceinline__ uint32_t ctarank() { uint32_t r; asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r)); return r; }
__device__ __forceinline__ void cl_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint64_t gtime() { uint64_t t; asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)); return t; }
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t ph) {
    for (long i = 0; i < 4000000L; ++i) {
        uint32_t d;
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(d) : "r"(bar), "r"(ph) : "memory");
        if (d) return true;
    }
    return false;
}

template <int KS, int MODE, int W>
__global__ void __cluster_dims__(KS, 1, 1) probe(int reps, float* gbuf, unsigned* err, unsigned long long* out) {
    extern __shared__ __align__(1024) uint8_t sm[];
    constexpr uint32_t BYTES = 32u * W * 4u;                 // one piece
    constexpr uint32_t RECV = (KS - 1) * 4u * BYTES;         // receive area
    const uint32_t base = saddr(sm);
    const uint32_t src_area = base + RECV;                    // local copy of the pieces to send
    __shared__ __align__(8) uint64_t bars[4];
    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t me = ctarank();
    if (threadIdx.x == 0) {
        for (int q = 0; q < 4; ++q) {
            const uint32_t cnt = (MODE == 0) ? uint32_t(KS - 1) : 1u;
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&bars[q])), "r"(cnt) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // fill the local send area
    for (uint32_t i = threadIdx.x; i < (KS - 1) * 4u * BYTES / 16u; i += blockDim.x)
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(src_area + i * 16u), "r"(i) : "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    cl_sync();
    const uint32_t bar = saddr(&bars[warp]);
    uint32_t ph = 0;
    float acc = 0.f;
    const unsigned long long c0 = clock64();
    const uint64_t t0 = gtime();
    for (int rep = 0; rep < reps; ++rep) {
        if (MODE == 1 && lane == 0)
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(uint32_t(KS - 1) * BYTES) : "memory");
        for (uint32_t k = 1; k < uint32_t(KS); ++k) {
            const uint32_t dst = (me + k) % KS;
            const uint32_t slot = me - (me > dst ? 1u : 0u);
            const uint32_t roff = (slot * 4u + warp) * BYTES;
            if (MODE == 0) {
                const uint32_t r = mapa(base + roff, dst);
#pragma unroll 4
                for (uint32_t i = 0; i < BYTES / 512u; ++i)
                    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(r + (i * 32u + lane) * 16u),
                                 "r"(i), "r"(lane), "r"(rep), "r"(k) : "memory");
            } else if (MODE == 1) {
                if (lane == 0) {
                    const uint32_t r = mapa(base + roff, dst);
                    const uint32_t rb = mapa(bar, dst);
                    const uint32_t s = src_area + ((k - 1) * 4u + warp) * BYTES;
                    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                                 ::"r"(r), "r"(s), "r"(BYTES), "r"(rb) : "memory");
                }
            } else if (MODE == 2) {
#pragma unroll 4
                for (uint32_t i = 0; i < BYTES / 512u; ++i)
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + roff + (i * 32u + lane) * 16u),
                                 "r"(i), "r"(lane), "r"(rep), "r"(k) : "memory");
            } else {
                float4* g = reinterpret_cast<float4*>(gbuf) +
                            ((size_t(blockIdx.x / KS) * KS + dst) * (KS - 1) * 4 + slot * 4 + warp) * (BYTES / 16);
#pragma unroll 4
                for (uint32_t i = 0; i < BYTES / 512u; ++i)
                    g[i * 32u + lane] = make_float4(float(i), float(lane), float(rep), float(k));
            }
        }
        if (MODE == 0) {
            asm volatile("fence.acq_rel.cluster;" ::: "memory");
            __syncwarp();
            if (lane == 0)
                for (uint32_t k = 1; k < uint32_t(KS); ++k)
                    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(mapa(bar, (me + k) % KS)) : "memory");
        }
        if (MODE == 0 || MODE == 1) {
            uint32_t ok = 1;
            if (lane == 0) ok = wait_bar(bar, ph);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok && lane == 0) atomicAdd(err, 1u);
            if (ok) wait_bar(bar, ph);  // complete already: every lane's acquire
            ph ^= 1u;
        }
        if (MODE == 3) {
            __threadfence();
            cl_sync();
        }
        // read what was received
        for (uint32_t s = 0; s + 1 < uint32_t(KS); ++s) {
            if (MODE == 3) {
                const float4* g = reinterpret_cast<const float4*>(gbuf) +
                                  ((size_t(blockIdx.x / KS) * KS + me) * (KS - 1) * 4 + s * 4 + warp) * (BYTES / 16);
#pragma unroll 4
                for (uint32_t i = 0; i < BYTES / 512u; ++i) {
                    const float4 v = __ldcg(g + i * 32u + lane);
                    acc += v.x + v.w;
                }
            } else {
#pragma unroll 4
                for (uint32_t i = 0; i < BYTES / 512u; ++i) {
                    float x, y, z, w;
                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x), "=f"(y), "=f"(z), "=f"(w)
                                 : "r"(base + (s * 4u + warp) * BYTES + (i * 32u + lane) * 16u) : "memory");
                    acc += x + w;
                }
            }
        }
        __syncthreads();
        cl_sync();
    }
    const unsigned long long c1 = clock64();
    const uint64_t t1 = gtime();
    if (threadIdx.x == 0) {
        out[blockIdx.x * 2] = c1 - c0;
        out[blockIdx.x * 2 + 1] = t1 - t0;
    }
    if (acc == 12345.f) atomicAdd(err, 1000u);
}

template <int KS, int MODE, int W>
bool run(float* gbuf, unsigned* err, unsigned long long* out, unsigned long long* hout) {
    constexpr int smem = 2 * (KS - 1) * 4 * 32 * W * 4 + 1024;
    cudaFuncSetAttribute(probe<KS, MODE, W>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    const int reps = 200;
    for (int trial = 0; trial < 2; ++trial) {
        probe<KS, MODE, W><<<152, 128, smem>>>(reps, gbuf, err, out);
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) { printf("KS%d mode %d W%d: %s\n", KS, MODE, W, cudaGetErrorString(e)); return false; }
    }
    cudaMemcpy(hout, out, 152 * 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    double cyc = 0, ns = 0;
    for (int b = 0; b < 152; ++b) { cyc += hout[2 * b]; ns += hout[2 * b + 1]; }
    cyc /= 152.0 * reps; ns /= 152.0 * reps;
    const double sent = double(KS - 1) * 4 * 32 * W * 4;  // bytes sent (= received) per CTA per rep
    printf("KS%d mode %d W%3d: %8.0f cycles %8.0f ns per exchange; %6.1f KB sent per CTA: %6.1f B/clk, %6.1f GB/s per SM\n",
           KS, MODE, W, cyc, ns, sent / 1024, sent / cyc, sent / ns);
    return true;
}

int main() {
    float* gbuf; unsigned* err; unsigned long long *out, hout[304];
    cudaMalloc(&gbuf, size_t(152) * 4 * 3 * 4 * 32 * 128 * 4);
    cudaMalloc(&err, 4); cudaMemset(err, 0, 4);
    cudaMalloc(&out, 304 * 8);
    bool ok = run<2, 0, 64>(gbuf, err, out, hout) && run<2, 1, 64>(gbuf, err, out, hout) &&
              run<2, 2, 64>(gbuf, err, out, hout) && run<2, 3, 64>(gbuf, err, out, hout) &&
              run<4, 0, 32>(gbuf, err, out, hout) && run<4, 1, 32>(gbuf, err, out, hout) &&
              run<4, 2, 32>(gbuf, err, out, hout) && run<4, 3, 32>(gbuf, err, out, hout) &&
              run<2, 0, 128>(gbuf, err, out, hout) && run<2, 1, 128>(gbuf, err, out, hout) &&
              run<2, 3, 128>(gbuf, err, out, hout);
    unsigned herr = 0;
    cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
    printf("waits that ran out / sink: %u\n", herr);
    return (ok && herr == 0) ? 0 : 1;
}
