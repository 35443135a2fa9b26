// Shared by the forward (mamba_scan.cu) and backward (mamba_scan_bwd.cu)
// translation units of libmamba_scan.so: element conversions, the hardware
// ex2/lg2/tanh paths, softplus and silu, argument checks, and the host-side
// services the forward file defines once (B/C packing, the scratch pool, the
// SM count, per-launch timing).
#pragma once

#include "mamba_scan.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <type_traits>

namespace mamba {

constexpr int kMaxN = 16;   // largest dstate
// Steps between the state checkpoints the backward pass recomputes from
// (its reverse tile); the forward kernel's checkpoint mode writes them.
constexpr int kBwdTile = 12;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

template <typename T> struct IO;
template <> struct IO<float> {
    static constexpr bool kAccurate = true;
    __device__ static void unpack(const uint4& r, float* v) {
        v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
        v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
    }
    __device__ static uint4 pack(const float* v) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                          __float_as_uint(v[2]), __float_as_uint(v[3]));
    }
    __device__ static float to_f(float x) { return x; }
    __device__ static float from_f(float x) { return x; }
};
template <> struct IO<__nv_bfloat16> {
    static constexpr bool kAccurate = false;
    __device__ static void unpack(const uint4& r, float* v) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static uint4 pack(const float* v) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&p);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Softplus in log2 units on the hardware ex2/lg2 path: log2(1 + 2^t), i.e.
// softplus(s) / ln 2 for t = s / ln 2, accurate in relative terms for every
// t.  It is evaluated as max(t, 0) + log2(1 + x) with x = 2^-|t| in (0, 1],
// so 2^t never overflows and, for very negative t (a step that keeps the
// state), the result is x / ln 2 to full relative precision instead of the
// rounded 1 + x.  log2(1 + x) = (x - x^2/2 + x^3/3 - ...) / ln 2; for
// x < 2^-7 the first two terms are taken (relative error below x^2/3 <
// 2e-5), otherwise lg2.approx(1 + x) (absolute error about 2^-22 against a
// result of at least 0.011, relative error below 2.2e-5).
__device__ __forceinline__ float softplus_log2_fast(float t) {
    const float x = ex2_approx(-fabsf(t));
    const float series = x * fmaf(x, -0.5f * kLog2e, kLog2e);
    const float full = lg2_approx(1.0f + x);
    return fmaxf(t, 0.0f) + (x < 0.0078125f ? series : full);
}

// softplus(s) = log(1 + e^s); for s > 20 it equals s to within e^-20.
template <bool ACC>
__device__ __forceinline__ float softplus_f(float s) {
    if (ACC) return s > 20.0f ? s : log1pf(expf(s));
    return softplus_log2_fast(s * kLog2e) * kLn2;
}

// silu(z) = z * sigmoid(z).  Accurate path: z / (1 + e^-z).  Fast path:
// sigmoid(z) = (1 + tanh(z/2)) / 2, so silu(z) = h + h * tanh(h) with h = z/2,
// one hardware tanh (max relative error about 2^-11).
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
template <bool ACC>
__device__ __forceinline__ float silu_f(float z) {
    if (ACC) return z / (1.0f + expf(-z));
    const float h = 0.5f * z;
    return fmaf(h, tanh_approx(h), h);
}

// ---------------------------------------------------------------------------
// debug builds: index checks on global accesses
// ---------------------------------------------------------------------------
//
// Built with -DMAMBA_DEBUG, every global access of the scan, generation-step
// and convolution kernels checks its element index against the extent of
// its buffer.  A failed check records kDebugBoundsFlag | source line in the
// translation unit's debug word (the first failure wins) and the access is
// skipped: a load reads 0, a store writes nothing.  Nothing traps, so the
// context stays usable; the host reads and clears the words through
// mamba_device_status.  In release builds the checks compile to nothing.

constexpr int kDebugBoundsFlag = 0x40000000;

// One debug word per translation unit (file-scope static).
static __device__ int g_debug_word;

__device__ __forceinline__ bool debug_in_bounds(long long i, long long n, int line) {
    if (i >= 0 && i < n) return true;
    atomicCAS(&g_debug_word, 0, kDebugBoundsFlag | line);
    return false;
}

// Reads and clears this translation unit's debug word (host side).
static inline int take_debug_word() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_debug_word, sizeof(int)) != cudaSuccess) return -1;
    if (v) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_debug_word, &zero, sizeof(int)) != cudaSuccess) return -1;
    }
    return v;
}

#ifdef MAMBA_DEBUG
#define MAMBA_IN(i, n) ::mamba::debug_in_bounds((long long)(i), (long long)(n), __LINE__)
#else
#define MAMBA_IN(i, n) true
#endif
// element i of p (extent n), or a zero value when the check fails
#define MAMBA_LD(p, i, n) \
    (MAMBA_IN((i), (n)) ? (p)[(i)] : std::remove_cv_t<std::remove_reference_t<decltype((p)[0])>>{})
// store v at element i of p (extent n) when the check passes
#define MAMBA_ST(p, i, n, v)                  \
    do {                                      \
        if (MAMBA_IN((i), (n))) (p)[(i)] = (v); \
    } while (0)

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

inline int esize(int dt) { return dt == MAMBA_BF16 ? 2 : 4; }
// dstate padded to the state sizes the kernels are built for: 4, 8 or 16
inline int padded_state(int64_t dstate) { return dstate <= 4 ? 4 : (dstate <= 8 ? 8 : 16); }
// state checkpoints of a sequence: one before every kBwdTile steps
inline int64_t checkpoint_tiles(int64_t seqlen) { return (seqlen + kBwdTile - 1) / kBwdTile; }

// The debug words of the convolution's and the backward pass's translation
// units (mamba_conv.cu, mamba_scan_bwd.cu).
int conv_take_debug_word();
int bwd_take_debug_word();

inline bool aligned(const void* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Kinds of launch timed by mamba_profile_begin/end.
enum LaunchKind {
    kKindScan = 0, kKindSummary = 1, kKindCarry = 2, kKindStep = 3, kKindPack = 4,
    kKindBwdCheckpoint = 5, kKindBwd = 6, kKindBwdReduce = 7, kKindConv = 8,
    kKindBwdSummary = 9, kKinds = 10
};

// While timing is on, brackets the launches of its scope with CUDA events
// on `s` (defined in mamba_scan.cu).
struct ProfScope {
    cudaEvent_t stop = nullptr;
    cudaStream_t st;
    ProfScope(int kind, cudaStream_t s);
    ~ProfScope();
};

int sm_count(int dev);
// The library's stream-ordered pool of the device (MAMBA_OK or an error).
int get_pool(int dev, cudaMemPool_t* out);
// The forward scan in its checkpoint mode (mamba_scan.cu): the Euler scan
// from initial_state (or zero) with no outputs, writing the state before
// every step that is a multiple of kBwdTile into ckpt[(((b * ck_tiles + k) *
// np / 4 + n / 4) * dim + d) * 4 + n % 4] (np = dstate padded to 4, 8 or
// 16; ck_tiles = ceil(seqlen / kBwdTile)).  Scratch from the stream-ordered
// pool.  Returns a status.
int scan_checkpoints(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int io_dtype,
                     const void* u, const void* delta, const float* dt_bias, const float* A,
                     const void* B, const void* C, int softplus, const float* initial_state,
                     float* ckpt, int ck_tiles, cudaStream_t stream);
// B and C (batch, N, L) in io_dtype -> fp32 rows of NP/2 float4 (s*B pair,
// C pair) per (batch, step), entries n >= N zero.
cudaError_t launch_pack_bc(int io_dtype, const void* B, const void* C, float4* out,
                           long long batch, long long L, int N, int NP, float scale,
                           cudaStream_t stream);

}  // namespace mamba
