// Causal depthwise convolution with SiLU, the short convolution in front of
// the scan in the Mamba block (page "Mamba: linear-time sequence modeling
// with selective state spaces", "What they did", Architecture bullet: the
// block merges the H3 block and a gated MLP):
//
//   xp(t)      = x[b,d,t] for t >= 0, else the carried state (or zero)
//   out[b,d,t] = silu( bias[d] + sum_{k<W} w[d,k] * xp(t - (W-1) + k) )
//
// Both kernels move each input and output once: the work is a handful of
// multiply/adds per element, so they are bound by HBM bandwidth.  The
// sequence kernel gives each thread kConvRun consecutive outputs of one row
// (one CTA per row); neighbouring threads take neighbouring runs, so a
// warp's 16-byte loads and stores are contiguous, and the W-1 inputs a run
// needs from the previous run come from the neighbouring lane.  The
// generation step is one thread per row, shifting the row's W-1 state
// inputs in place.

#include "scan_common.cuh"

#include <algorithm>

namespace mamba {
namespace {

constexpr int kConvRun = 16;         // outputs per thread: 32 bytes of bf16, 64 of fp32
constexpr int kConvThreads = 128;   // one 2048-step row of 16-element runs per CTA
constexpr int kMaxConvWidth = 8;

// kConvRun consecutive elements as 16-byte accesses (8 bf16 or 4 fp32 each)
template <typename T>
__device__ __forceinline__ void load_run(const T* p, float (&v)[kConvRun]) {
    constexpr int kPer = 16 / (int)sizeof(T);
    uint4 r[kConvRun / kPer];
#pragma unroll
    for (int k = 0; k < kConvRun / kPer; ++k) r[k] = reinterpret_cast<const uint4*>(p)[k];
#pragma unroll
    for (int k = 0; k < kConvRun / kPer; ++k) IO<T>::unpack(r[k], v + k * kPer);
}
template <typename T>
__device__ __forceinline__ void store_run(T* p, const float (&v)[kConvRun]) {
    constexpr int kPer = 16 / (int)sizeof(T);
#pragma unroll
    for (int k = 0; k < kConvRun / kPer; ++k)
        reinterpret_cast<uint4*>(p)[k] = IO<T>::pack(v + k * kPer);
}

template <bool ACC>
__device__ __forceinline__ float conv_act(float a, bool silu) {
    return silu ? silu_f<ACC>(a) : a;
}

// One CTA per (batch, channel) row; thread j of the CTA takes runs j,
// j + kConvThreads, ... of the row.  The W-1 inputs before a run are the last
// inputs of the previous run, held by the neighbouring lane: a shuffle, not
// a load, except for lane 0 of each warp.  vec: every row of x and out
// starts 16-byte aligned (runs are then aligned).
template <typename T, int W, bool SILU>
__global__ void __launch_bounds__(kConvThreads)
conv1d_kernel(const T* __restrict__ x, const float* __restrict__ w, const float* __restrict__ bias,
              const T* __restrict__ state, T* __restrict__ out, T* __restrict__ state_out,
              long long dim, long long L, int vec) {
    constexpr bool ACC = IO<T>::kAccurate;
    constexpr int S = W - 1;
    static_assert(S <= kConvRun, "the inputs before a run come from one neighbouring run");
    const long long row = blockIdx.x;
    const long long d = row % dim;
    const int lane = threadIdx.x & 31;
    // extents for the index checks of debug builds (one CTA per row)
    const long long rows = gridDim.x, nx = rows * L, ns = rows * S;
    (void)nx; (void)ns;
    float wk[W];
#pragma unroll
    for (int k = 0; k < W; ++k) wk[k] = MAMBA_LD(w, d * W + k, dim * W);
    const float b0 = bias ? MAMBA_LD(bias, d, dim) : 0.0f;
    const long long runs = (L + kConvRun - 1) / kConvRun;
    // the input at position s of the padded row (s < 0: the carried state)
    auto xp = [&](long long s) -> float {
        return s >= 0 ? IO<T>::to_f(MAMBA_LD(x, row * L + s, nx))
                      : (state ? IO<T>::to_f(MAMBA_LD(state, row * S + S + s, ns)) : 0.0f);
    };
    for (long long r0 = 0; r0 < runs; r0 += kConvThreads) {   // uniform over the CTA
        const long long c = r0 + threadIdx.x;
        const bool act = c < runs;
        const long long t0 = c * kConvRun;
        const bool full = t0 + kConvRun <= L;
        float v[kConvRun + S];
        if (act && vec && full) {
            float r[kConvRun];
#pragma unroll
            for (int j = 0; j < kConvRun; ++j) r[j] = 0.0f;
            if (MAMBA_IN(row * L + t0, nx) && MAMBA_IN(row * L + t0 + kConvRun - 1, nx))
                load_run<T>(x + row * L + t0, r);
#pragma unroll
            for (int j = 0; j < kConvRun; ++j) v[S + j] = r[j];
        } else {
#pragma unroll
            for (int j = 0; j < kConvRun; ++j)
                v[S + j] = (act && t0 + j < L) ? IO<T>::to_f(MAMBA_LD(x, row * L + t0 + j, nx)) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < S; ++j) {
            const float up = __shfl_up_sync(0xffffffffu, v[kConvRun + j], 1);
            v[j] = lane == 0 ? (act ? xp(t0 - S + j) : 0.0f) : up;
        }
        if (!act) continue;
        float o[kConvRun];
#pragma unroll
        for (int j = 0; j < kConvRun; ++j) {
            float acc = b0;
#pragma unroll
            for (int k = 0; k < W; ++k) acc = fmaf(wk[k], v[j + k], acc);
            o[j] = conv_act<ACC>(acc, SILU);
        }
        if (vec && full) {
            if (MAMBA_IN(row * L + t0, nx) && MAMBA_IN(row * L + t0 + kConvRun - 1, nx))
                store_run<T>(out + row * L + t0, o);
        } else {
#pragma unroll
            for (int j = 0; j < kConvRun; ++j)
                if (t0 + j < L) MAMBA_ST(out, row * L + t0 + j, nx, IO<T>::from_f(o[j]));
        }
        // the run holding t = L-1 writes the state after the last input
        if (state_out && c == runs - 1) {
#pragma unroll
            for (int j = 0; j < S; ++j) {
                const long long s = L - S + j;
                MAMBA_ST(state_out, row * S + j, ns,
                         s >= 0 ? MAMBA_LD(x, row * L + s, nx)
                                : (state ? MAMBA_LD(state, row * S + S + s, ns)
                                         : IO<T>::from_f(0.0f)));
            }
        }
    }
}

template <typename T, int W, bool SILU>
__global__ void __launch_bounds__(kConvThreads)
conv1d_update_kernel(T* __restrict__ state, const T* __restrict__ x, const float* __restrict__ w,
                     const float* __restrict__ bias, T* __restrict__ out, long long rows,
                     long long dim) {
    constexpr bool ACC = IO<T>::kAccurate;
    constexpr int S = W - 1;
    const long long row = (long long)blockIdx.x * kConvThreads + threadIdx.x;
    if (row >= rows) return;
    const long long d = row % dim;
    const long long ns = rows * S;   // extent of the state (debug index checks)
    (void)ns;
    float v[W];
#pragma unroll
    for (int j = 0; j < S; ++j) v[j] = IO<T>::to_f(MAMBA_LD(state, row * S + j, ns));
    const T xv = MAMBA_LD(x, row, rows);
    v[S] = IO<T>::to_f(xv);
    float acc = bias ? MAMBA_LD(bias, d, dim) : 0.0f;
#pragma unroll
    for (int k = 0; k < W; ++k) acc = fmaf(MAMBA_LD(w, d * W + k, dim * W), v[k], acc);
    MAMBA_ST(out, row, rows, IO<T>::from_f(conv_act<ACC>(acc, SILU)));
#pragma unroll
    for (int j = 0; j + 1 < S; ++j)
        MAMBA_ST(state, row * S + j, ns, MAMBA_LD(state, row * S + j + 1, ns));
    if constexpr (S > 0) MAMBA_ST(state, row * S + S - 1, ns, xv);
}

template <typename T, int W>
cudaError_t launch_conv(bool silu, const T* x, const float* w, const float* bias, const T* state,
                        T* out, T* state_out, long long rows, long long dim, long long L, int vec,
                        cudaStream_t st) {
    const unsigned grid = (unsigned)rows;
    if (silu)
        conv1d_kernel<T, W, true><<<grid, kConvThreads, 0, st>>>(x, w, bias, state, out,
                                                                 state_out, dim, L, vec);
    else
        conv1d_kernel<T, W, false><<<grid, kConvThreads, 0, st>>>(x, w, bias, state, out,
                                                                  state_out, dim, L, vec);
    return cudaGetLastError();
}

template <typename T, int W>
cudaError_t launch_conv_update(bool silu, T* state, const T* x, const float* w, const float* bias,
                               T* out, long long rows, long long dim, cudaStream_t st) {
    const unsigned grid = (unsigned)((rows + kConvThreads - 1) / kConvThreads);
    if (silu)
        conv1d_update_kernel<T, W, true><<<grid, kConvThreads, 0, st>>>(state, x, w, bias, out,
                                                                        rows, dim);
    else
        conv1d_update_kernel<T, W, false><<<grid, kConvThreads, 0, st>>>(state, x, w, bias, out,
                                                                         rows, dim);
    return cudaGetLastError();
}

#define MAMBA_CONV_WIDTHS(X) X(1) X(2) X(3) X(4) X(5) X(6) X(7) X(8)

template <typename T>
cudaError_t dispatch_conv(int width, bool silu, const void* x, const float* w, const float* bias,
                          const void* state, void* out, void* state_out, long long rows,
                          long long dim, long long L, int vec, cudaStream_t st) {
#define X(W_)                                                                              \
    if (width == W_)                                                                       \
        return launch_conv<T, W_>(silu, static_cast<const T*>(x), w, bias,                 \
                                  static_cast<const T*>(state), static_cast<T*>(out),      \
                                  static_cast<T*>(state_out), rows, dim, L, vec, st);
    MAMBA_CONV_WIDTHS(X)
#undef X
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t dispatch_conv_update(int width, bool silu, void* state, const void* x, const float* w,
                                 const float* bias, void* out, long long rows, long long dim,
                                 cudaStream_t st) {
#define X(W_)                                                                              \
    if (width == W_)                                                                       \
        return launch_conv_update<T, W_>(silu, static_cast<T*>(state),                     \
                                         static_cast<const T*>(x), w, bias,                \
                                         static_cast<T*>(out), rows, dim, st);
    MAMBA_CONV_WIDTHS(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace

int conv_take_debug_word() { return take_debug_word(); }

}  // namespace mamba

using namespace mamba;

extern "C" {

int mamba_conv1d_fwd(int64_t batch, int64_t dim, int64_t seqlen, int width, mamba_dtype_t io_dtype,
                     const void* x, const float* weight, const float* bias,
                     const void* conv_state, int silu, void* out, void* final_conv_state,
                     cudaStream_t stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (batch < 1 || dim < 1 || seqlen < 0 || width < 1 || width > kMaxConvWidth)
        return MAMBA_ERR_SHAPE;
    if ((double)batch * dim >= 2147483647.0 || dim > (1ll << 40) || seqlen > (1ll << 40) ||
        (double)batch * dim * (double)(seqlen > 0 ? seqlen : 1) > 4.0e18)
        return MAMBA_ERR_SHAPE;
    if (!weight || (seqlen > 0 && (!x || !out))) return MAMBA_ERR_NULL;
    const int es = esize(io_dtype);
    const long long rows = batch * dim;
    const size_t xb = (size_t)(rows * seqlen) * es, sb = (size_t)(rows * (width - 1)) * es;
    for (const void* q : {x, conv_state, (const void*)out, (const void*)final_conv_state})
        if (q && !aligned(q, es)) return MAMBA_ERR_ALIGN;
    for (const void* q : {(const void*)weight, (const void*)bias})
        if (q && !aligned(q, 4)) return MAMBA_ERR_ALIGN;
    {
        const void* ins[] = {x, weight, bias, conv_state};
        const size_t insz[] = {xb, (size_t)dim * width * 4, (size_t)dim * 4, sb};
        for (int i = 0; i < 4; ++i) {
            if (overlaps(out, xb, ins[i], insz[i])) return MAMBA_ERR_ALIAS;
            if (overlaps(final_conv_state, sb, ins[i], insz[i])) return MAMBA_ERR_ALIAS;
        }
        if (overlaps(out, xb, final_conv_state, sb)) return MAMBA_ERR_ALIAS;
    }
    if (seqlen == 0) {
        if (final_conv_state && sb > 0) {
            const cudaError_t r =
                conv_state ? cudaMemcpyAsync(final_conv_state, conv_state, sb,
                                             cudaMemcpyDeviceToDevice, stream)
                           : cudaMemsetAsync(final_conv_state, 0, sb, stream);
            if (r != cudaSuccess) return MAMBA_ERR_CUDA;
        }
        return MAMBA_OK;
    }
    const int vec = ((seqlen * es) % 16 == 0) && aligned(x, 16) && aligned(out, 16);
    cudaError_t e;
    {
        ProfScope prof(kKindConv, stream);
        e = io_dtype == MAMBA_BF16
                ? dispatch_conv<__nv_bfloat16>(width, silu != 0, x, weight, bias,
                                               width > 1 ? conv_state : nullptr, out,
                                               width > 1 ? final_conv_state : nullptr, rows, dim,
                                               seqlen, vec, stream)
                : dispatch_conv<float>(width, silu != 0, x, weight, bias,
                                       width > 1 ? conv_state : nullptr, out,
                                       width > 1 ? final_conv_state : nullptr, rows, dim, seqlen,
                                       vec, stream);
    }
    return e == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

int mamba_conv1d_update(int64_t batch, int64_t dim, int width, mamba_dtype_t io_dtype, void* conv_state,
                        const void* x, const float* weight, const float* bias, int silu, void* out,
                        cudaStream_t stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (batch < 1 || dim < 1 || width < 1 || width > kMaxConvWidth) return MAMBA_ERR_SHAPE;
    if ((double)batch * dim > 1.0e15) return MAMBA_ERR_SHAPE;
    if (!x || !weight || !out || (width > 1 && !conv_state)) return MAMBA_ERR_NULL;
    const int es = esize(io_dtype);
    const long long rows = batch * dim;
    const size_t vb = (size_t)rows * es, sb = (size_t)(rows * (width - 1)) * es;
    for (const void* q : {(const void*)conv_state, x, (const void*)out})
        if (q && !aligned(q, es)) return MAMBA_ERR_ALIGN;
    for (const void* q : {(const void*)weight, (const void*)bias})
        if (q && !aligned(q, 4)) return MAMBA_ERR_ALIGN;
    {
        const void* ins[] = {x, weight, bias};
        const size_t insz[] = {vb, (size_t)dim * width * 4, (size_t)dim * 4};
        for (int i = 0; i < 3; ++i) {
            if (overlaps(out, vb, ins[i], insz[i])) return MAMBA_ERR_ALIAS;
            if (overlaps(conv_state, sb, ins[i], insz[i])) return MAMBA_ERR_ALIAS;
        }
        if (overlaps(out, vb, conv_state, sb)) return MAMBA_ERR_ALIAS;
    }
    cudaError_t e;
    {
        ProfScope prof(kKindConv, stream);
        e = io_dtype == MAMBA_BF16
                ? dispatch_conv_update<__nv_bfloat16>(width, silu != 0, conv_state, x, weight,
                                                      bias, out, rows, dim, stream)
                : dispatch_conv_update<float>(width, silu != 0, conv_state, x, weight, bias, out,
                                              rows, dim, stream);
    }
    return e == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

}  // extern "C"
