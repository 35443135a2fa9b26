// Sustained per-SM issue rates of the arithmetic the scan is built from,
// measured in SM clock cycles (clock64) so that the result does not depend
// on the clock the GPU runs at.  This is measurement support for the
// roofline the scan is judged against; the selective scan itself has no use
// for it.
//
// Each kernel runs `iters` iterations of a fully unrolled body on CHAINS
// independent dependency chains per thread.  Thread 0 of every CTA reads
// clock64 after a CTA barrier before and after the loop; the host divides
// the CTA's operation count by its cycle count.  One CTA per SM (the host
// launches exactly as many CTAs as SMs, each too large for two to share an
// SM: over 114 KB of dynamic shared memory), with 1 to 8 warps per SM
// sub-partition.
//
// Kinds (operations counted per lane):
//   0 ex2.approx.ftz.f32            x = ex2(x)                       1 MUFU
//   1 lg2.approx.ftz.f32            x = lg2(x)                       1 MUFU
//   2 tanh.approx.f32               x = tanh(x)                      1 MUFU
//   3 fma.rn.f32x2                  h = a*h + b on pairs             2 fp32 lane-ops
//   4 fma.rn.f32                    h = a*h + b                      1 fp32 lane-op
//   5 the scan's state update on a pair of state entries:
//       arg = Delta'*A (f32x2), Abar = ex2 x2, bx = du*B (f32x2),
//       h = Abar*h + bx (f32x2), acc = C*h + acc (f32x2)
//     counted as 2 state updates (2 ex2 + 8 fp32 lane-ops)
// Values drift to 0, 1 or infinity in some chains; these instructions take
// the same time whatever the value.

#include "mamba_scan.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

namespace {

__device__ __forceinline__ float p_ex2(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float p_lg2(float x) {
    float y;
    asm volatile("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float p_tanh(float x) {
    float y;
    asm volatile("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr int kBody = 16;   // unrolled operations per chain per iteration

template <int KIND, int CHAINS>
__global__ void pipe_probe_kernel(int iters, float seed, float* sink, long long* cycles) {
    const int tid = threadIdx.x;
    float x[CHAINS];
    float2 h[CHAINS], aa[CHAINS], bb[CHAINS], acc[CHAINS];
#pragma unroll
    for (int c = 0; c < CHAINS; ++c) {
        x[c] = seed * (float)(tid + 1) + 0.01f * (float)c;
        h[c] = make_float2(x[c], 0.5f * x[c]);
        aa[c] = make_float2(-0.25f - 0.01f * c, -0.5f - 0.01f * c);
        bb[c] = make_float2(0.125f * x[c], 0.25f);
        acc[c] = make_float2(0.0f, 0.0f);
    }
    float dt = seed;
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < kBody; ++k) {
#pragma unroll
            for (int c = 0; c < CHAINS; ++c) {
                if constexpr (KIND == 0) x[c] = p_ex2(x[c]);
                if constexpr (KIND == 1) x[c] = p_lg2(x[c]);
                if constexpr (KIND == 2) x[c] = p_tanh(x[c]);
                if constexpr (KIND == 3) h[c] = __ffma2_rn(aa[c], h[c], bb[c]);
                if constexpr (KIND == 4) x[c] = fmaf(aa[c].x, x[c], bb[c].x);
                if constexpr (KIND == 5) {
                    const float2 arg = __fmul2_rn(make_float2(dt, dt), aa[c]);
                    const float2 ab = make_float2(p_ex2(arg.x), p_ex2(arg.y));
                    const float2 bx = __fmul2_rn(make_float2(x[c], x[c]), bb[c]);
                    h[c] = __ffma2_rn(ab, h[c], bx);
                    acc[c] = __ffma2_rn(bb[c], h[c], acc[c]);
                }
            }
            if constexpr (KIND == 5) dt = dt * 0.999f;   // a new step: Delta changes
        }
    }
    __syncthreads();
    const long long t1 = clock64();
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < CHAINS; ++c) s += x[c] + h[c].x + h[c].y + acc[c].x + acc[c].y;
    if (s == 1.2345f) sink[blockIdx.x * blockDim.x + tid] = s;   // keeps the chains live
    if (tid == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int KIND, int CHAINS>
cudaError_t launch(int grid, int threads, int smem, int iters, float* sink, long long* cyc,
                   cudaStream_t st) {
    auto k = pipe_probe_kernel<KIND, CHAINS>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k<<<grid, threads, smem, st>>>(iters, 0.37f, sink, cyc);
    return cudaGetLastError();
}

template <int CHAINS>
cudaError_t launch_kind(int kind, int grid, int threads, int smem, int iters, float* sink,
                        long long* cyc, cudaStream_t st) {
    switch (kind) {
        case 0: return launch<0, CHAINS>(grid, threads, smem, iters, sink, cyc, st);
        case 1: return launch<1, CHAINS>(grid, threads, smem, iters, sink, cyc, st);
        case 2: return launch<2, CHAINS>(grid, threads, smem, iters, sink, cyc, st);
        case 3: return launch<3, CHAINS>(grid, threads, smem, iters, sink, cyc, st);
        case 4: return launch<4, CHAINS>(grid, threads, smem, iters, sink, cyc, st);
        case 5: return launch<5, CHAINS>(grid, threads, smem, iters, sink, cyc, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

extern "C" int mamba_probe_pipe_rate(int kind, int warps_per_subpartition, int chains,
                                     int64_t iters, double* ops_per_clk_sm,
                                     double* cycles_median, cudaStream_t stream) {
    if (kind < 0 || kind > 5 || iters < 1 || iters > (1 << 24) || !ops_per_clk_sm)
        return MAMBA_ERR_SHAPE;
    if (warps_per_subpartition < 1 || warps_per_subpartition > 8) return MAMBA_ERR_SHAPE;
    if (chains != 1 && chains != 2 && chains != 4 && chains != 8 && chains != 16)
        return MAMBA_ERR_SHAPE;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms < 1)
        return MAMBA_ERR_CUDA;
    const int threads = 4 * 32 * warps_per_subpartition;
    const int smem = 120 * 1024;   // one CTA per SM
    float* sink = nullptr;
    long long* cyc = nullptr;
    if (cudaMalloc(&sink, (size_t)sms * threads * sizeof(float)) != cudaSuccess)
        return MAMBA_ERR_ALLOC;
    if (cudaMalloc(&cyc, (size_t)sms * sizeof(long long)) != cudaSuccess) {
        cudaFree(sink);
        return MAMBA_ERR_ALLOC;
    }
    cudaError_t e;
    if (chains == 1) e = launch_kind<1>(kind, sms, threads, smem, (int)iters, sink, cyc, stream);
    else if (chains == 2) e = launch_kind<2>(kind, sms, threads, smem, (int)iters, sink, cyc, stream);
    else if (chains == 4) e = launch_kind<4>(kind, sms, threads, smem, (int)iters, sink, cyc, stream);
    else if (chains == 8) e = launch_kind<8>(kind, sms, threads, smem, (int)iters, sink, cyc, stream);
    else e = launch_kind<16>(kind, sms, threads, smem, (int)iters, sink, cyc, stream);
    std::vector<long long> h(sms, 0);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess)
        e = cudaMemcpy(h.data(), cyc, sizeof(long long) * sms, cudaMemcpyDeviceToHost);
    cudaFree(sink);
    cudaFree(cyc);
    if (e != cudaSuccess) return MAMBA_ERR_CUDA;
    std::sort(h.begin(), h.end());
    const double med = (double)h[sms / 2];
    // lane operations per CTA: threads * chains * iters * kBody, with the
    // scan mix counted as 2 state updates per chain step and f32x2 FMA as 2
    double per = (double)threads * chains * (double)iters * kBody;
    if (kind == 3 || kind == 5) per *= 2.0;
    *ops_per_clk_sm = per / med;
    if (cycles_median) *cycles_median = med;
    return MAMBA_OK;
}
