// Throughput of the MUFU base-2 exponential (ex2.approx.ftz.f32) on this device, per SM and
// clock: the denominator of the scan's roofline. Every thread runs 32 independent chains
// x <- ex2(x) (nothing else in the loop but the loop counter), 16 CTAs of 128 threads per
// SM. Each CTA records its SM (%smid) and the SM's clock (clock64) before and after its loop;
// an SM's span runs from its first CTA's start to its last CTA's end, so the rate is per SM
// cycle, whatever the clock the GPU runs at and however many CTAs were resident at once. Not part of the scan library: a measurement
// used by the benchmark (`bench.py --measure-ex2`).
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ float ex2_probe(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(128) ex2_chains(int iters, float seed, float *sink, long long *stamps) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = seed * (float)(threadIdx.x + i) * 1e-6f - 0.5f;
    __syncthreads();
    const long long c0 = clock64();
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = ex2_probe(v[i]);
    }
    __syncthreads();
    const long long c1 = clock64();
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) s += v[i];
    if (s == 1234.5f) sink[0] = s;   // keeps the chains alive; never true for these inputs
    if (threadIdx.x == 0) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        stamps[3 * blockIdx.x] = smid;
        stamps[3 * blockIdx.x + 1] = c0;
        stamps[3 * blockIdx.x + 2] = c1;
    }
}

}  // namespace

extern "C" {
#pragma GCC visibility push(default)

// Measures ex2 per SM per clock on the current device. Returns 0 on success with *per_clk_sm
// set; otherwise the cudaError_t of the failing call. Allocates and frees its own buffers.
int ssm_probe_ex2_rate(int iters, double *per_clk_sm, double *elapsed_ms) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    const int per_sm = 16, blocks = sms * per_sm;
    float *sink = nullptr;
    long long *cyc = nullptr;
    if ((e = cudaMalloc(&sink, sizeof(float))) != cudaSuccess) return (int)e;
    if ((e = cudaMalloc(&cyc, sizeof(long long) * 3 * blocks)) != cudaSuccess) {
        cudaFree(sink);
        return (int)e;
    }
    cudaEvent_t a = nullptr, b = nullptr;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    ex2_chains<<<blocks, 128>>>(16, 1.0f, sink, cyc);   // warm-up
    cudaEventRecord(a);
    ex2_chains<<<blocks, 128>>>(iters, 1.0f, sink, cyc);
    cudaEventRecord(b);
    e = cudaEventSynchronize(b);
    if (e == cudaSuccess) e = cudaGetLastError();
    float ms = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
    long long *hc = new long long[3 * blocks];
    if (e == cudaSuccess) e = cudaMemcpy(hc, cyc, sizeof(long long) * 3 * blocks, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) {
        // per SM: CTAs run there and the span from the first start to the last end (clock64 is
        // the SM's own counter); the rate is the median over the SMs
        const int nsm_max = 1024;
        long long lo[nsm_max], hi[nsm_max];
        int cnt[nsm_max];
        for (int i = 0; i < nsm_max; ++i) { lo[i] = 0x7fffffffffffffffLL; hi[i] = 0; cnt[i] = 0; }
        for (int i = 0; i < blocks; ++i) {
            const int sm = (int)hc[3 * i];
            if (sm < 0 || sm >= nsm_max) continue;
            lo[sm] = hc[3 * i + 1] < lo[sm] ? hc[3 * i + 1] : lo[sm];
            hi[sm] = hc[3 * i + 2] > hi[sm] ? hc[3 * i + 2] : hi[sm];
            ++cnt[sm];
        }
        double rates[nsm_max];
        int nr = 0;
        for (int i = 0; i < nsm_max; ++i)
            if (cnt[i] > 0 && hi[i] > lo[i]) rates[nr++] = (double)cnt[i] * 128.0 * 32.0 * (double)iters / (double)(hi[i] - lo[i]);
        for (int i = 1; i < nr; ++i)   // insertion sort, nr <= a few hundred
            for (int j = i; j > 0 && rates[j] < rates[j - 1]; --j) { const double t = rates[j]; rates[j] = rates[j - 1]; rates[j - 1] = t; }
        *per_clk_sm = nr > 0 ? rates[nr / 2] : 0.0;
        *elapsed_ms = ms;
    }
    delete[] hc;
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    cudaFree(sink);
    cudaFree(cyc);
    return (int)e;
}

#pragma GCC visibility pop
}  // extern "C"
