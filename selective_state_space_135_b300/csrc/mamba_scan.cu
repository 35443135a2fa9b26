// Selective scan (S6) forward and single-token state update for B300 (sm_103a).
//
// Operation (page "Mamba: linear-time sequence modeling with selective state
// spaces", section "What they did", S6 bullet and sub-bullets; the decode step
// is the generation mode of page "Mamba: Linear-Time Sequence Modeling with
// Selective State Spaces", section "Architecture"):
//
//   Delta = softplus(delta + dt_bias)          (or delta + dt_bias)
//   h[n]  = exp(Delta*A[d,n]) * h[n] + Delta*B[b,n,t]*u[b,d,t]
//   y     = (sum_n C[b,n,t]*h[n] + D_skip[d]*u[b,d,t]) * silu(z[b,d,t])
//
// Design (one GPU, no tensor cores: the work is an elementwise recurrence):
//   * A CTA (4 warps) owns a tile of channels of one batch entry and walks
//     time.  Each thread keeps NT state entries of one channel in registers;
//     with dstate > 8 two lanes share a channel (8 entries each) and split the
//     per-step scalar work (Delta, Delta*u, skip term, gate) between them.
//   * Inputs stream through a shared-memory ring filled by tensor-map bulk
//     copies (cp.async.bulk.tensor, completion on an mbarrier): one
//     [channels x 64 bytes of time] box per tensor per tile, 64-byte
//     swizzled so every thread's 16-byte row reads are bank-conflict free.
//     Output tiles leave the same way (double-buffered, bulk-group stores).
//     Shapes whose rows are not 16-byte multiples run the same kernels with
//     plain, bounds-checked element loads and stores into the same layout.
//   * B and C (shared by all channels of a batch entry) are widened once per
//     tile into an fp32 [t][n] table read with broadcast 128-bit loads.
//   * The expanded (b, d, t, n) tensor is never materialised: Abar and the
//     input term live only in registers; the state leaves the SM only at the
//     end of a work unit.
//   * Work units are whole-sequence channel tiles; when the tiles cannot fill
//     the SMs (few channels, very long sequences) every tile is cut into time
//     chunks: a summary pass computes each chunk's (prod Abar, end state from
//     zero), a carry pass composes them in order, and the main pass restarts
//     every chunk from its exact carried-in state.
//   * fp32 I/O uses the library expf/log1pf; bf16 I/O uses the hardware
//     ex2/lg2 approximations (relative error ~2^-22), far inside the bf16
//     output rounding.  State and accumulation are fp32 in both.
//   * Packed fp32x2 multiply/FMA (sm_100+) halves the instruction count of
//     the state update; exp2 runs on the MUFU pipe alongside.

#include "mamba_scan.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <vector>

namespace mamba {

// ---------------------------------------------------------------------------
// device-side helpers
// ---------------------------------------------------------------------------

__device__ int g_error_word;  // nonzero once a bounded device wait gave up

constexpr int kThreads = 128;        // threads per CTA (4 warps)
constexpr int kMaxStages = 4;
constexpr int kMaxN = 16;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per wait

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

// softplus(s) = log(1 + e^s); for s > 20 it equals s to within e^-20.
template <bool ACC>
__device__ __forceinline__ float softplus_f(float s) {
    float r;
    if (ACC) {
        r = log1pf(expf(s));
    } else {
        r = lg2_approx(1.0f + ex2_approx(s * kLog2e)) * kLn2;
    }
    return s > 20.0f ? s : r;
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z)
template <bool ACC>
__device__ __forceinline__ float silu_f(float z) {
    if (ACC) return z / (1.0f + expf(-z));
    return __fdividef(z, 1.0f + ex2_approx(-z * kLog2e));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, P1;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait: true when the phase completed, false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (unsigned it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && global_ns() - t0 > kWaitLimitNs) return false;
    }
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// scan kernels
// ---------------------------------------------------------------------------

// Tensor-map copies (cp.async.bulk.tensor): one instruction moves a whole
// [channels x time] box between global and shared memory.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

struct ScanArgs {
    CUtensorMap m_u, m_dl, m_z, m_y, m_B, m_C;   // valid when use_tma
    const void* u;
    const void* delta;
    const void* z;
    const void* B;
    const void* C;
    const float* dt_bias;
    const float* A;
    const float* D_skip;
    void* y;
    float* final_state;
    float* ws_P;  // chunk decay products  [(k * tail_rows + wrow) * N + n]
    float* ws_h;  // chunk end states, then carried-in states (same layout)
    long long dim;
    long long seqlen;
    long long chunk_len;  // multiple of the time tile
    int batch;
    int dstate;
    int use_tma;
    int stages;
    int groups_per_batch;  // ceil(dim / CH)
    int n_groups;          // batch * groups_per_batch
    int n_full;            // groups [0, n_full) run the whole sequence
    int nchunks;           // time chunks of each remaining ("tail") group
    int tail_rows;         // (n_groups - n_full) * CH
};

// Work unit of one CTA.
struct Unit {
    int b, d0;          // batch entry, first channel of the tile
    int tail;           // -1 for whole-sequence units, else tail group index
    int k;              // chunk index within the tail group (0 for whole units)
    long long t0, t1;   // time range [t0, t1)
};

// Units are numbered: [0, n_full) whole-sequence groups, then every chunk of
// every tail group.  The summary pass numbers only the chunks that feed the
// carry (all but the last of each tail group).
template <int CH, bool STATE_ONLY>
__device__ __forceinline__ Unit decode_unit(const ScanArgs& a, int idx) {
    Unit w;
    int g;
    if (STATE_ONLY) {
        const int per = a.nchunks - 1;
        g = a.n_full + idx / per;
        w.k = idx % per;
    } else if (idx < a.n_full) {
        g = idx;
        w.k = 0;
    } else {
        const int j = idx - a.n_full;
        g = a.n_full + j / a.nchunks;
        w.k = j % a.nchunks;
    }
    w.b = g / a.groups_per_batch;
    w.d0 = (g % a.groups_per_batch) * CH;
    if (g < a.n_full) {
        w.tail = -1;
        w.t0 = 0;
        w.t1 = a.seqlen;
    } else {
        w.tail = g - a.n_full;
        w.t0 = (long long)w.k * a.chunk_len;
        w.t1 = min(a.seqlen, w.t0 + a.chunk_len);
    }
    return w;
}

// Shared-memory layout, byte offsets from a 1024-aligned base.  A channel's
// time tile is one 64-byte row; rows of the u/delta/z/y tiles are stored
// with the 64-byte swizzle of the tensor-map copies: the 16-byte chunk j of
// row r sits at r*64 + ((j ^ ((r >> 1) & 3)) << 4), which makes the
// per-thread 16-byte row reads and writes bank-conflict free.
//   [0, 1024)           stage mbarriers
//   stage s             u | delta | z tiles (CH x 64 B each) | B raw | C raw (16 x 64 B each)
//   BC table            TT x {B, C} x 16 fp32
//   y tiles             2 x CH x 64 B
template <int CH>
struct Layout {
    static constexpr int kTile = CH * 64;
    static constexpr int kBoff = 3 * kTile;
    static constexpr int kCoff = kBoff + kMaxN * 64;
    static constexpr int kStage = (kCoff + kMaxN * 64 + 1023) / 1024 * 1024;
    __host__ __device__ static constexpr int stage(int s) { return 1024 + s * kStage; }
    __host__ __device__ static constexpr int bct(int stages) { return 1024 + stages * kStage; }
    __host__ __device__ static constexpr int ybuf(int stages, int tt) {
        return (bct(stages) + tt * 2 * kMaxN * 4 + 1023) / 1024 * 1024;
    }
    __host__ __device__ static constexpr int bytes(int stages, int tt) {
        return ybuf(stages, tt) + 2 * kTile + 1024;   // + slack to align the base
    }
};

__device__ __forceinline__ int swz(int row, int chunk) {
    return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
}

// One time step of NT state entries (NT/2 packed pairs) of one channel:
//   h <- exp(Delta*A) * h + (Delta*u) * B ;  returns sum_n C*h over the NT entries.
template <int NT, bool ACC, bool STATE_ONLY>
__device__ __forceinline__ float ssm_step(float2 (&h2)[NT / 2], const float2 (&a2)[NT / 2],
                                          float dt, float du, const float* brow,
                                          const float* crow) {
    const float2 dt2 = make_float2(dt, dt);
    const float2 du2 = make_float2(du, du);
    float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
    if constexpr (NT == 2) {
        const float2 b2 = *reinterpret_cast<const float2*>(brow);
        float2 dA;
        if constexpr (ACC) {
            dA = make_float2(expf(dt * a2[0].x), expf(dt * a2[0].y));
        } else {
            const float2 arg = __fmul2_rn(dt2, a2[0]);
            dA = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
        }
        h2[0] = __ffma2_rn(dA, h2[0], __fmul2_rn(du2, b2));
        if constexpr (!STATE_ONLY) acc0 = __fmul2_rn(*reinterpret_cast<const float2*>(crow), h2[0]);
    } else {
#pragma unroll
        for (int q = 0; q < NT / 4; ++q) {
            const float4 b4 = *reinterpret_cast<const float4*>(brow + 4 * q);
            float4 c4;
            if constexpr (!STATE_ONLY) c4 = *reinterpret_cast<const float4*>(crow + 4 * q);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = 2 * q + j;
                const float2 bp = j ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
                float2 dA;
                if constexpr (ACC) {
                    dA = make_float2(expf(dt * a2[i].x), expf(dt * a2[i].y));
                } else {
                    const float2 arg = __fmul2_rn(dt2, a2[i]);
                    dA = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
                }
                h2[i] = __ffma2_rn(dA, h2[i], __fmul2_rn(du2, bp));
                if constexpr (!STATE_ONLY) {
                    const float2 cp = j ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
                    if (j) acc1 = __ffma2_rn(cp, h2[i], acc1);
                    else acc0 = __ffma2_rn(cp, h2[i], acc0);
                }
            }
        }
    }
    return (acc0.x + acc1.x) + (acc0.y + acc1.y);
}

// The scan over one work unit (CH channels x a time range).  STATE_ONLY is
// the chunk-summary pass: no C, z or y; it returns (exp(A*sum Delta), h_end).
template <typename T, int NT, int S, bool STATE_ONLY, bool SOFTPLUS, bool HAS_Z>
__global__ void __launch_bounds__(kThreads)
scan_kernel(const __grid_constant__ ScanArgs a) {
    constexpr int CH = kThreads / S;             // channels per CTA
    constexpr int G = 16 / sizeof(T);            // time steps per 16-byte chunk
    constexpr int TT = 64 / sizeof(T);           // time steps per tile
    constexpr int NP = NT * S;                   // padded state size
    constexpr bool ACC = IO<T>::kAccurate;
    constexpr int kNPair = NT / 2;
    constexpr unsigned kFull = 0xffffffffu;
    constexpr bool has_z = !STATE_ONLY && HAS_Z;
    static_assert(NT % 2 == 0 && NP <= kMaxN && (S == 1 || S == 2), "bad state split");
    using Lay = Layout<CH>;

    // Offset the __shared__ array itself (not a pointer rebuilt from an
    // integer) so that every access below stays a shared-memory access.
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int tid = threadIdx.x;
    const int c = tid / S;       // channel within the tile
    const int p = tid % S;       // which NT-slice of the state
    const Unit w = decode_unit<CH, STATE_ONLY>(a, blockIdx.x);
    const long long dim = a.dim, L_ = a.seqlen;
    const int N = a.dstate;
    const int d = w.d0 + c;
    const bool chan_ok = d < dim;
    const int rows_valid = (int)min((long long)CH, dim - w.d0);
    const long long row = (long long)w.b * dim + d;
    const int stages = a.stages;
    const bool tma = a.use_tma != 0;
    const int ntiles = (int)((w.t1 - w.t0 + TT - 1) / TT);
    const int wrow = (w.tail >= 0) ? w.tail * CH + c : 0;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    float* bct = reinterpret_cast<float*>(smem + Lay::bct(stages));
    unsigned char* ybuf = smem + Lay::ybuf(stages, TT);

    // ---- per-thread constants and initial state ----
    float2 h2[kNPair], a2[kNPair];
#pragma unroll
    for (int i = 0; i < kNPair; ++i) {
        float av[2], hv[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int n = p * NT + 2 * i + j;
            const bool ok = chan_ok && n < N;
            const float an = ok ? a.A[(long long)d * N + n] : 0.0f;
            av[j] = ACC ? an : an * kLog2e;
            float h0 = 0.0f;
            if (ok && w.tail >= 0 && w.k > 0 && !STATE_ONLY)
                h0 = a.ws_h[((long long)(w.k - 1) * a.tail_rows + wrow) * N + n];
            hv[j] = h0;
        }
        a2[i] = make_float2(av[0], av[1]);
        h2[i] = make_float2(hv[0], hv[1]);
    }
    const float bias = (chan_ok && a.dt_bias) ? a.dt_bias[d] : 0.0f;
    const float dsk = (chan_ok && a.D_skip) ? a.D_skip[d] : 0.0f;
    float dsum = 0.0f;  // sum of Delta over the unit (summary pass)

    const int ntens = has_z ? 3 : 2;
    const int nbc = STATE_ONLY ? 1 : 2;

    // thread 0: tensor-map copies of tile `it` into stage `s`
    auto issue_tile = [&](int it, int s) {
        const int tt0 = (int)(w.t0 + (long long)it * TT);
        const uint32_t bar = smem_u32(&bars[s]);
        unsigned char* st = smem + Lay::stage(s);
        mbar_arrive_expect_tx(bar, (uint32_t)(ntens * Lay::kTile + nbc * N * 64));
        tma_load_3d(smem_u32(st), &a.m_u, tt0, w.d0, w.b, bar);
        tma_load_3d(smem_u32(st + Lay::kTile), &a.m_dl, tt0, w.d0, w.b, bar);
        if constexpr (has_z) tma_load_3d(smem_u32(st + 2 * Lay::kTile), &a.m_z, tt0, w.d0, w.b, bar);
        tma_load_3d(smem_u32(st + Lay::kBoff), &a.m_B, tt0, 0, w.b, bar);
        if (!STATE_ONLY) tma_load_3d(smem_u32(st + Lay::kCoff), &a.m_C, tt0, 0, w.b, bar);
    };

    // all threads: element-wise, bounds-checked fill of stage 0 (any shape)
    auto plain_tile = [&](int it) {
        const long long tt0 = w.t0 + (long long)it * TT;
        const int nv = (int)min((long long)TT, w.t1 - tt0);
        unsigned char* st = smem + Lay::stage(0);
        for (int e = tid; e < ntens * CH * TT; e += kThreads) {
            const int tsr = e / (CH * TT), rem = e % (CH * TT);
            const int cc = rem / TT, t = rem % TT;
            const T* src = static_cast<const T*>(tsr == 0 ? a.u : (tsr == 1 ? a.delta : a.z));
            T v = IO<T>::from_f(0.0f);
            if (cc < rows_valid && t < nv) v = src[((long long)w.b * dim + w.d0 + cc) * L_ + tt0 + t];
            const int byte = t * (int)sizeof(T);
            *reinterpret_cast<T*>(st + tsr * Lay::kTile + swz(cc, byte >> 4) + (byte & 15)) = v;
        }
        for (int e = tid; e < nbc * N * TT; e += kThreads) {
            const int which = e / (N * TT), rem = e % (N * TT);
            const int n = rem / TT, t = rem % TT;
            const T* src = static_cast<const T*>(which ? a.C : a.B);
            T v = IO<T>::from_f(0.0f);
            if (t < nv) v = src[((long long)w.b * N + n) * L_ + tt0 + t];
            reinterpret_cast<T*>(st + (which ? Lay::kCoff : Lay::kBoff) + n * 64)[t] = v;
        }
    };

    if (tma) {
        if (tid == 0) {
            for (int s = 0; s < stages; ++s) mbar_init(smem_u32(&bars[s]), 1);
            fence_mbar_init();
            prefetch_map(&a.m_u);
            prefetch_map(&a.m_dl);
            prefetch_map(&a.m_B);
            if constexpr (has_z) prefetch_map(&a.m_z);
            if (!STATE_ONLY) {
                prefetch_map(&a.m_C);
                prefetch_map(&a.m_y);
            }
        }
        __syncthreads();
        if (tid == 0)
            for (int s = 0; s < stages && s < ntiles; ++s) issue_tile(s, s);
    }

    int issued = tma ? min(stages, ntiles) : 0;
    bool aborted = false;

    for (int it = 0; it < ntiles; ++it) {
        const int s = tma ? it % stages : 0;
        const long long tt0 = w.t0 + (long long)it * TT;
        const int nv = (int)min((long long)TT, w.t1 - tt0);
        unsigned char* st = smem + Lay::stage(s);

        bool timed_out = false;
        if (tma) {
            timed_out = !mbar_wait_bounded(smem_u32(&bars[s]), (uint32_t)((it / stages) & 1));
            if (!STATE_ONLY && tid == 0) bulk_wait_read_1();   // y tile (it & 1) free again
        } else {
            plain_tile(it);
            __syncthreads();
        }

        // widen B and C of this tile into the fp32 [t][{B,C}][n] table
        for (int e = tid; e < TT * 2 * NP; e += kThreads) {
            const int t = e / (2 * NP), which = (e / NP) & 1, n = e % NP;
            float v = 0.0f;
            if (n < N && t < nv && (which == 0 || !STATE_ONLY))
                v = IO<T>::to_f(reinterpret_cast<const T*>(
                    st + (which ? Lay::kCoff : Lay::kBoff) + n * 64)[t]);
            bct[(t * 2 + which) * kMaxN + n] = v;
        }
        if (__syncthreads_or(timed_out)) {   // (A)
            aborted = true;
            break;
        }

        const unsigned char* ut = st;
        const unsigned char* dlt = st + Lay::kTile;
        const unsigned char* zt = st + 2 * Lay::kTile;
        unsigned char* yt = ybuf + (it & 1) * Lay::kTile;

        auto body = [&](auto masked) {
            constexpr bool MASK = decltype(masked)::value;
#pragma unroll 1
            for (int grp = 0; grp < TT / G; ++grp) {
                const int off = swz(c, grp);
                float uv[G], dv[G], zv[G];
                IO<T>::unpack(*reinterpret_cast<const uint4*>(ut + off), uv);
                IO<T>::unpack(*reinterpret_cast<const uint4*>(dlt + off), dv);
                if constexpr (has_z) IO<T>::unpack(*reinterpret_cast<const uint4*>(zt + off), zv);
                float dtv[G], duv[G];
                if constexpr (S == 1) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float sarg = dv[g] + bias;
                        float dt = SOFTPLUS ? softplus_f<ACC>(sarg) : sarg;
                        if (MASK && grp * G + g >= nv) dt = 0.0f;
                        dtv[g] = dt;
                        duv[g] = dt * uv[g];
                        if (STATE_ONLY) dsum += dt;
                    }
                } else {
                    // the two lanes of a channel each evaluate Delta for every
                    // other step and swap results
#pragma unroll
                    for (int k = 0; k < G / 2; ++k) {
                        const float sarg = (p ? dv[2 * k + 1] : dv[2 * k]) + bias;
                        const float um = p ? uv[2 * k + 1] : uv[2 * k];
                        float dtm = SOFTPLUS ? softplus_f<ACC>(sarg) : sarg;
                        if (MASK && grp * G + 2 * k + p >= nv) dtm = 0.0f;
                        const float dum = dtm * um;
                        const float dto = __shfl_xor_sync(kFull, dtm, 1);
                        const float duo = __shfl_xor_sync(kFull, dum, 1);
                        dtv[2 * k] = p ? dto : dtm;
                        dtv[2 * k + 1] = p ? dtm : dto;
                        duv[2 * k] = p ? duo : dum;
                        duv[2 * k + 1] = p ? dum : duo;
                        if (STATE_ONLY) dsum += dtm + dto;
                    }
                }
                float yv[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float* brow = bct + ((grp * G + g) * 2) * kMaxN + p * NT;
                    yv[g] = ssm_step<NT, ACC, STATE_ONLY>(h2, a2, dtv[g], duv[g], brow,
                                                         brow + kMaxN);
                }
                if constexpr (!STATE_ONLY) {
                    if constexpr (S == 1) {
                        float ov[G];
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            float o = yv[g] + dsk * uv[g];
                            if constexpr (has_z) o *= silu_f<ACC>(zv[g]);
                            ov[g] = o;
                        }
                        *reinterpret_cast<uint4*>(yt + off) = IO<T>::pack(ov);
                    } else {
                        // each lane finishes every other step: add the partner's
                        // partial sum, skip term and gate, store one element
                        T* yrow = reinterpret_cast<T*>(yt + off);
#pragma unroll
                        for (int k = 0; k < G / 2; ++k) {
                            const float send = p ? yv[2 * k] : yv[2 * k + 1];
                            const float recv = __shfl_xor_sync(kFull, send, 1);
                            const float mine = (p ? yv[2 * k + 1] : yv[2 * k]) + recv;
                            const float um = p ? uv[2 * k + 1] : uv[2 * k];
                            float o = mine + dsk * um;
                            if constexpr (has_z) o *= silu_f<ACC>(p ? zv[2 * k + 1] : zv[2 * k]);
                            yrow[2 * k + p] = IO<T>::from_f(o);
                        }
                    }
                }
            }
        };
        if (nv == TT) body(std::false_type{});
        else body(std::true_type{});

        if (!STATE_ONLY && tma) fence_proxy_async_smem();
        __syncthreads();   // (B): stage s consumed, y tile complete

        if (!STATE_ONLY) {
            if (tma) {
                if (tid == 0) {
                    tma_store_3d(&a.m_y, smem_u32(yt), (int)tt0, w.d0, w.b);
                    bulk_commit();
                }
            } else {
                for (int e = tid; e < CH * TT; e += kThreads) {
                    const int cc = e / TT, t = e % TT;
                    if (cc < rows_valid && t < nv) {
                        const int byte = t * (int)sizeof(T);
                        static_cast<T*>(a.y)[((long long)w.b * dim + w.d0 + cc) * L_ + tt0 + t] =
                            *reinterpret_cast<const T*>(yt + swz(cc, byte >> 4) + (byte & 15));
                    }
                }
            }
        }
        if (tma && tid == 0 && issued < ntiles) {
            issue_tile(issued, issued % stages);
            ++issued;
        }
    }

    if (tma) {
        if (aborted && tid == 0) {
            atomicExch(&g_error_word, 1);
            // let copies still in flight land before the CTA's memory is released
            for (int it = 0; it < issued; ++it)
                (void)mbar_wait_bounded(smem_u32(&bars[it % stages]), (uint32_t)((it / stages) & 1));
        }
        if (!STATE_ONLY && tid == 0) bulk_wait_all();
        __syncthreads();
        if (aborted) return;
    }

    // ---- results that leave the SM: final state or chunk summary ----
    if (!chan_ok) return;
#pragma unroll
    for (int i = 0; i < kNPair; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int n = p * NT + 2 * i + j;
            if (n >= N) continue;
            const float hv = j ? h2[i].y : h2[i].x;
            if (STATE_ONLY) {
                const long long idx = ((long long)w.k * a.tail_rows + wrow) * N + n;
                const float an = j ? a2[i].y : a2[i].x;
                a.ws_P[idx] = ACC ? expf(an * dsum) : ex2_approx(an * dsum);
                a.ws_h[idx] = hv;
            } else if (a.final_state && w.t1 == L_) {
                a.final_state[row * N + n] = hv;
            }
        }
    }
}

// Compose chunk summaries in time order: h_{k+1} = P_k * h_k + hend_k from
// h_0 = 0.  Overwrites hend_k with h_{k+1}, the state entering chunk k+1.
__global__ void carry_kernel(float* __restrict__ ws_P, float* __restrict__ ws_h,
                             long long entries, int nchunks) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= entries) return;
    float h = 0.0f;
    for (int k = 0; k + 1 < nchunks; ++k) {
        const long long idx = (long long)k * entries + i;
        h = ws_P[idx] * h + ws_h[idx];
        ws_h[idx] = h;
    }
}

// ---------------------------------------------------------------------------
// decode: one step on a (batch, dim, N) state, in place
// ---------------------------------------------------------------------------

struct StepArgs {
    float* state;
    const void* x;
    const void* delta;
    const void* z;
    const void* B;
    const void* C;
    const float* dt_bias;
    const float* A;
    const float* D_skip;
    void* y;
    long long rows;
    long long dim;
    int dstate;
    int vec_state;  // state rows 16-byte aligned and N % 4 == 0
};

// Four lanes per (b, d) row; lane q owns state entries [4q, 4q + 4).
template <typename T>
__global__ void __launch_bounds__(kThreads)
state_update_kernel(const StepArgs a) {
    constexpr bool ACC = IO<T>::kAccurate;
    const long long gid = (long long)blockIdx.x * kThreads + threadIdx.x;
    const long long row = gid >> 2;
    const int q = (int)(gid & 3);
    const bool ok = row < a.rows;
    const int N = a.dstate;
    float acc = 0.0f, xv = 0.0f, zv = 0.0f, dsk = 0.0f;
    if (ok) {
        const long long b = row / a.dim, d = row % a.dim;
        xv = IO<T>::to_f(static_cast<const T*>(a.x)[row]);
        const float s = IO<T>::to_f(static_cast<const T*>(a.delta)[row]) +
                        (a.dt_bias ? a.dt_bias[d] : 0.0f);
        const float dt = softplus_f<ACC>(s);
        const float du = dt * xv;
        if (a.z) zv = IO<T>::to_f(static_cast<const T*>(a.z)[row]);
        dsk = a.D_skip ? a.D_skip[d] : 0.0f;
        const T* Bb = static_cast<const T*>(a.B) + b * N;
        const T* Cb = static_cast<const T*>(a.C) + b * N;
        const float* Ad = a.A + d * N;
        float* h = a.state + row * N;
        const int n0 = 4 * q;
        if (a.vec_state && n0 < N) {
            float4 hv = *reinterpret_cast<const float4*>(h + n0);
            float hs[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + j;
                const float dA = ACC ? expf(dt * Ad[n]) : ex2_approx(dt * (Ad[n] * kLog2e));
                hs[j] = fmaf(dA, hs[j], du * IO<T>::to_f(Bb[n]));
                acc = fmaf(IO<T>::to_f(Cb[n]), hs[j], acc);
            }
            *reinterpret_cast<float4*>(h + n0) = make_float4(hs[0], hs[1], hs[2], hs[3]);
        } else {
            for (int n = n0; n < n0 + 4 && n < N; ++n) {
                const float dA = ACC ? expf(dt * Ad[n]) : ex2_approx(dt * (Ad[n] * kLog2e));
                const float hn = fmaf(dA, h[n], du * IO<T>::to_f(Bb[n]));
                h[n] = hn;
                acc = fmaf(IO<T>::to_f(Cb[n]), hn, acc);
            }
        }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    if (ok && q == 0) {
        float o = acc + dsk * xv;
        if (a.z) o *= silu_f<ACC>(zv);
        static_cast<T*>(a.y)[row] = IO<T>::from_f(o);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

struct Tuning {
    int split = 0;   // lanes per channel (0 = automatic)
    int stages = 0;  // ring depth (0 = automatic)
    int chunks = 0;  // time chunks for every group (0 = automatic)
};
Tuning g_tuning;
std::mutex g_mu;
std::vector<cudaMemPool_t> g_pools;

// Optional per-launch timing: while enabled, every kernel launch is bracketed
// by two CUDA events recorded on its own stream.
enum LaunchKind { kKindScan = 0, kKindSummary = 1, kKindCarry = 2, kKindStep = 3, kKinds = 4 };
struct ProfRec {
    int kind;
    cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_recs;

struct ProfScope {
    cudaEvent_t stop = nullptr;
    cudaStream_t st;
    ProfScope(int kind, cudaStream_t s) : st(s) {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        if (!g_prof_on) return;
        ProfRec r;
        r.kind = kind;
        if (cudaEventCreate(&r.start) != cudaSuccess) return;
        if (cudaEventCreate(&r.stop) != cudaSuccess) {
            cudaEventDestroy(r.start);
            return;
        }
        cudaEventRecord(r.start, st);
        stop = r.stop;
        g_prof_recs.push_back(r);
    }
    ~ProfScope() {
        if (stop) cudaEventRecord(stop, st);
    }
};

int esize(int dt) { return dt == MAMBA_BF16 ? 2 : 4; }

bool aligned(const void* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int get_pool(int dev, cudaMemPool_t* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)g_pools.size() <= dev) g_pools.resize(dev + 1, nullptr);
    if (!g_pools[dev]) {
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return MAMBA_ERR_ALLOC;
        uint64_t keep = UINT64_MAX;  // keep freed blocks cached in the pool
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        g_pools[dev] = pool;
    }
    *out = g_pools[dev];
    return MAMBA_OK;
}

int sm_count(int dev) {
    static std::vector<int> cache;
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (!cache[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = v > 0 ? v : 148;
    }
    return cache[dev];
}

template <typename T, int NT, int S, bool STATE_ONLY, bool SP, bool HZ>
cudaError_t launch_scan(const ScanArgs& a, int grid, int smem, cudaStream_t st) {
    auto k = scan_kernel<T, NT, S, STATE_ONLY, SP, HZ>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    ProfScope prof(STATE_ONLY ? kKindSummary : kKindScan, st);
    k<<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

// (NT, S) variants: S = 1 for dstate <= 8 (NT = 2, 4, 8) and on request for
// dstate <= 16 (NT = 16); S = 2 (NT = 8) is the default for 8 < dstate <= 16.
#define MAMBA_VARIANTS(X) X(2, 1) X(4, 1) X(8, 1) X(16, 1) X(8, 2)

template <typename T, bool STATE_ONLY>
cudaError_t dispatch_scan(int nt, int s, bool sp, bool hz, const ScanArgs& a, int grid, int smem,
                          cudaStream_t st) {
#define X(NT_, S_)                                                                          \
    if (nt == NT_ && s == S_) {                                                              \
        if (STATE_ONLY)                                                                      \
            return sp ? launch_scan<T, NT_, S_, STATE_ONLY, true, false>(a, grid, smem, st)  \
                      : launch_scan<T, NT_, S_, STATE_ONLY, false, false>(a, grid, smem, st); \
        if (sp)                                                                              \
            return hz ? launch_scan<T, NT_, S_, STATE_ONLY, true, true>(a, grid, smem, st)   \
                      : launch_scan<T, NT_, S_, STATE_ONLY, true, false>(a, grid, smem, st); \
        return hz ? launch_scan<T, NT_, S_, STATE_ONLY, false, true>(a, grid, smem, st)      \
                  : launch_scan<T, NT_, S_, STATE_ONLY, false, false>(a, grid, smem, st);    \
    }
    MAMBA_VARIANTS(X)
#undef X
    return cudaErrorInvalidValue;
}

struct Plan {
    int nt, s, ch, stages, tt;
    int groups_per_batch, n_groups, n_full, nchunks;
    long long chunk_len;
    int smem;
};

int smem_bytes(int ch, int stages, int tt) {
    return ch == 128 ? Layout<128>::bytes(stages, tt) : Layout<64>::bytes(stages, tt);
}

// Work decomposition.  Channel tiles scan the whole sequence when there are
// at least as many tiles as SMs: the kernel is bound by instruction issue
// and latency within each CTA, so extra co-resident CTAs on some SMs cost
// little, while time chunks would add a summary pass (about 3/4 of a main
// pass).  With fewer tiles than SMs (few channels, very long sequences)
// every tile is cut into K time chunks so that about two pieces land on
// each SM.
Plan make_plan(int dev, int dt, long long batch, long long dim, int N, long long L, bool tma) {
    Tuning tn;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        tn = g_tuning;
    }
    Plan p;
    int s = 1, nt;
    if (N <= 2) nt = 2;
    else if (N <= 4) nt = 4;
    else if (N <= 8) nt = 8;
    else {
        s = (tn.split == 1) ? 1 : 2;
        nt = 16 / s;
    }
    p.nt = nt;
    p.s = s;
    p.ch = kThreads / s;
    p.tt = 64 / esize(dt);
    p.stages = tma ? (tn.stages > 0 ? std::min(tn.stages, kMaxStages) : 2) : 1;
    p.smem = smem_bytes(p.ch, p.stages, p.tt);
    p.groups_per_batch = (int)((dim + p.ch - 1) / p.ch);
    p.n_groups = (int)(batch * p.groups_per_batch);
    const int sms = sm_count(dev);
    const long long tiles = (L + p.tt - 1) / p.tt;
    const long long min_chunk_tiles = 8;
    int K = 1;
    if (tn.chunks > 0) {
        K = tn.chunks;
    } else if (p.n_groups < sms && tiles >= 2 * min_chunk_tiles) {
        K = (2 * sms + p.n_groups - 1) / p.n_groups;
        K = (int)std::min<long long>(K, tiles / min_chunk_tiles);
    }
    if (K <= 1) {
        p.n_full = p.n_groups;
        p.nchunks = 1;
        p.chunk_len = L;
    } else {
        const long long per = (tiles + K - 1) / K;
        p.chunk_len = per * p.tt;
        p.nchunks = (int)((L + p.chunk_len - 1) / p.chunk_len);
        p.n_full = p.nchunks > 1 ? 0 : p.n_groups;
    }
    return p;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 3-D map over a (d2, d1, d0) row-major tensor, box {b0, b1, 1}.
bool encode_map(CUtensorMap* m, const void* ptr, int dt, long long d0, long long d1, long long d2,
                int b0, int b1, bool swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const int es = esize(dt);
    cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)(d0 * es), (cuuint64_t)(d0 * d1 * es)};
    cuuint32_t box[3] = {(cuuint32_t)b0, (cuuint32_t)b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, dt == MAMBA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                           3, const_cast<void*>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace mamba

using namespace mamba;

extern "C" {

int mamba_version(void) { return 200; }

const char* mamba_status_string(int status) {
    switch (status) {
        case MAMBA_OK: return "ok";
        case MAMBA_ERR_NULL: return "a required pointer is NULL";
        case MAMBA_ERR_SHAPE: return "a size is out of range (1 <= dstate <= 16, sizes >= 1)";
        case MAMBA_ERR_ALIGN: return "a pointer is not aligned to its element type";
        case MAMBA_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
        case MAMBA_ERR_TIMEOUT: return "a device-side wait ran out of time";
        case MAMBA_ERR_ALLOC: return "scratch memory could not be obtained";
        case MAMBA_ERR_DTYPE: return "unsupported io dtype";
        case MAMBA_ERR_ALIAS: return "an output overlaps an input";
        default: return "unknown status";
    }
}

int mamba_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MAMBA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return MAMBA_ERR_CUDA;
    if (v) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int)) != cudaSuccess)
            return MAMBA_ERR_CUDA;
        return MAMBA_ERR_TIMEOUT;
    }
    return MAMBA_OK;
}

int mamba_profile_begin(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto& r : g_prof_recs) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    g_prof_recs.clear();
    g_prof_on = true;
    return MAMBA_OK;
}

int mamba_profile_end(double* total_ms, int64_t* launches, int nkinds) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_on = false;
    int rc = MAMBA_OK;
    for (int k = 0; k < nkinds; ++k) {
        if (total_ms) total_ms[k] = 0.0;
        if (launches) launches[k] = 0;
    }
    for (auto& r : g_prof_recs) {
        float ms = 0.0f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess ||
            cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
            rc = MAMBA_ERR_CUDA;
        if (r.kind < nkinds) {
            if (total_ms) total_ms[r.kind] += ms;
            if (launches) launches[r.kind] += 1;
        }
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    g_prof_recs.clear();
    return rc;
}

int mamba_scan_set_tuning(int split, int stages, int chunks) {
    if (split < 0 || split > 2 || stages < 0 || stages > kMaxStages || chunks < 0)
        return MAMBA_ERR_SHAPE;
    std::lock_guard<std::mutex> lk(g_mu);
    g_tuning.split = split;
    g_tuning.stages = stages;
    g_tuning.chunks = chunks;
    return MAMBA_OK;
}

int mamba_scan_fwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int io_dtype,
                   const void* u, const void* delta, const float* dt_bias, const float* A,
                   const void* B, const void* C, const float* D_skip, const void* z,
                   int softplus, void* y, float* final_state, cudaStream_t stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (batch < 1 || dim < 1 || dstate < 1 || dstate > kMaxN || seqlen < 0) return MAMBA_ERR_SHAPE;
    if (batch > INT32_MAX / 2 || dim > (1ll << 40) || seqlen > (1ll << 40) ||
        (double)batch * dim * (double)(seqlen > 0 ? seqlen : 1) > 4.0e18)
        return MAMBA_ERR_SHAPE;
    if (!A || (seqlen > 0 && (!u || !delta || !B || !C || !y))) return MAMBA_ERR_NULL;
    const int es = esize(io_dtype);
    const size_t big = (size_t)(batch * dim * seqlen) * es;
    const size_t bcb = (size_t)(batch * dstate * seqlen) * es;
    const size_t fsb = (size_t)(batch * dim * dstate) * 4;
    for (const void* q : {u, delta, z, B, C, (const void*)y})
        if (q && !aligned(q, es)) return MAMBA_ERR_ALIGN;
    for (const void* q : {(const void*)dt_bias, (const void*)A, (const void*)D_skip,
                          (const void*)final_state})
        if (q && !aligned(q, 4)) return MAMBA_ERR_ALIGN;
    {
        const void* ins[] = {u, delta, z, B, C, dt_bias, A, D_skip};
        const size_t insz[] = {big, big, big, bcb, bcb, (size_t)dim * 4,
                               (size_t)(dim * dstate) * 4, (size_t)dim * 4};
        for (int i = 0; i < 8; ++i) {
            if (overlaps(y, big, ins[i], insz[i])) return MAMBA_ERR_ALIAS;
            if (overlaps(final_state, fsb, ins[i], insz[i])) return MAMBA_ERR_ALIAS;
        }
        if (overlaps(y, big, final_state, fsb)) return MAMBA_ERR_ALIAS;
    }
    if (seqlen == 0) {
        if (final_state && cudaMemsetAsync(final_state, 0, fsb, stream) != cudaSuccess)
            return MAMBA_ERR_CUDA;
        return MAMBA_OK;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MAMBA_ERR_CUDA;
    // tensor-map path: 16-byte aligned bases and rows, coordinates within int32
    bool tma = ((seqlen * es) % 16) == 0 && seqlen < (1ll << 31) && dim < (1ll << 31) &&
               (double)dim * seqlen * es < 1.0e12;
    for (const void* q : {u, delta, z, B, C, (const void*)y})
        if (q && !aligned(q, 16)) tma = false;

    Plan pl = make_plan(dev, io_dtype, batch, dim, (int)dstate, seqlen, tma);

    ScanArgs a;
    std::memset(&a, 0, sizeof(a));
    if (tma) {
        const int ch = pl.ch, tt = pl.tt;
        tma = encode_map(&a.m_u, u, io_dtype, seqlen, dim, batch, tt, ch, true) &&
              encode_map(&a.m_dl, delta, io_dtype, seqlen, dim, batch, tt, ch, true) &&
              (!z || encode_map(&a.m_z, z, io_dtype, seqlen, dim, batch, tt, ch, true)) &&
              encode_map(&a.m_y, y, io_dtype, seqlen, dim, batch, tt, ch, true) &&
              encode_map(&a.m_B, B, io_dtype, seqlen, dstate, batch, tt, (int)dstate, false) &&
              encode_map(&a.m_C, C, io_dtype, seqlen, dstate, batch, tt, (int)dstate, false);
        if (!tma) pl = make_plan(dev, io_dtype, batch, dim, (int)dstate, seqlen, false);
    }
    a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C;
    a.dt_bias = dt_bias; a.A = A; a.D_skip = D_skip; a.y = y; a.final_state = final_state;
    a.dim = dim; a.seqlen = seqlen; a.chunk_len = pl.chunk_len;
    a.batch = (int)batch; a.dstate = (int)dstate;
    a.use_tma = tma ? 1 : 0; a.stages = pl.stages;
    a.groups_per_batch = pl.groups_per_batch; a.n_groups = pl.n_groups;
    a.n_full = pl.n_full; a.nchunks = pl.nchunks;
    a.tail_rows = (pl.n_groups - pl.n_full) * pl.ch;

    const bool chunked = pl.n_full < pl.n_groups && pl.nchunks > 1;
    void* ws = nullptr;
    if (chunked) {
        const size_t entries = (size_t)a.tail_rows * dstate;
        const size_t bytes = 2 * entries * (size_t)(pl.nchunks - 1) * sizeof(float);
        cudaMemPool_t pool = nullptr;
        int rc = get_pool(dev, &pool);
        if (rc != MAMBA_OK) return rc;
        if (cudaMallocFromPoolAsync(&ws, bytes, pool, stream) != cudaSuccess) {
            cudaGetLastError();
            return MAMBA_ERR_ALLOC;
        }
        a.ws_P = static_cast<float*>(ws);
        a.ws_h = a.ws_P + entries * (pl.nchunks - 1);
    }

    cudaError_t e = cudaSuccess;
    if (chunked) {
        const int grid1 = (pl.n_groups - pl.n_full) * (pl.nchunks - 1);
        e = io_dtype == MAMBA_BF16
                ? dispatch_scan<__nv_bfloat16, true>(pl.nt, pl.s, softplus, false, a, grid1,
                                                     pl.smem, stream)
                : dispatch_scan<float, true>(pl.nt, pl.s, softplus, false, a, grid1, pl.smem,
                                             stream);
        if (e == cudaSuccess) {
            const long long entries = (long long)a.tail_rows * dstate;
            {
                ProfScope prof(kKindCarry, stream);
                carry_kernel<<<(unsigned)((entries + 255) / 256), 256, 0, stream>>>(
                    a.ws_P, a.ws_h, entries, pl.nchunks);
            }
            e = cudaGetLastError();
        }
    }
    if (e == cudaSuccess) {
        const int grid = pl.n_full + (chunked ? (pl.n_groups - pl.n_full) * pl.nchunks : 0);
        e = io_dtype == MAMBA_BF16
                ? dispatch_scan<__nv_bfloat16, false>(pl.nt, pl.s, softplus, z != nullptr, a,
                                                      grid, pl.smem, stream)
                : dispatch_scan<float, false>(pl.nt, pl.s, softplus, z != nullptr, a, grid,
                                              pl.smem, stream);
    }
    if (ws) cudaFreeAsync(ws, stream);
    return e == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

int mamba_state_update(int64_t batch, int64_t dim, int64_t dstate, int io_dtype, float* state,
                       const void* x, const void* delta, const float* dt_bias, const float* A,
                       const void* B, const void* C, const float* D_skip, const void* z, void* y,
                       cudaStream_t stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (batch < 1 || dim < 1 || dstate < 1 || dstate > kMaxN) return MAMBA_ERR_SHAPE;
    if ((double)batch * dim > 1.0e15) return MAMBA_ERR_SHAPE;
    if (!state || !x || !delta || !A || !B || !C || !y) return MAMBA_ERR_NULL;
    const int es = esize(io_dtype);
    for (const void* q : {x, delta, z, B, C, (const void*)y})
        if (q && !aligned(q, es)) return MAMBA_ERR_ALIGN;
    for (const void* q : {(const void*)state, (const void*)dt_bias, (const void*)A,
                          (const void*)D_skip})
        if (q && !aligned(q, 4)) return MAMBA_ERR_ALIGN;
    const long long rows = batch * dim;
    const size_t sb = (size_t)rows * dstate * 4, vb = (size_t)rows * es,
                 bb = (size_t)batch * dstate * es;
    {
        const void* ins[] = {x, delta, z, B, C, dt_bias, A, D_skip};
        const size_t insz[] = {vb, vb, vb, bb, bb, (size_t)dim * 4, (size_t)(dim * dstate) * 4,
                               (size_t)dim * 4};
        for (int i = 0; i < 8; ++i) {
            if (overlaps(state, sb, ins[i], insz[i])) return MAMBA_ERR_ALIAS;
            if (overlaps(y, vb, ins[i], insz[i])) return MAMBA_ERR_ALIAS;
        }
        if (overlaps(state, sb, y, vb)) return MAMBA_ERR_ALIAS;
    }
    StepArgs a;
    a.state = state; a.x = x; a.delta = delta; a.z = z; a.B = B; a.C = C;
    a.dt_bias = dt_bias; a.A = A; a.D_skip = D_skip; a.y = y;
    a.rows = rows; a.dim = dim; a.dstate = (int)dstate;
    a.vec_state = (dstate % 4 == 0) && aligned(state, 16);
    const long long threads = rows * 4;
    const unsigned grid = (unsigned)((threads + kThreads - 1) / kThreads);
    {
        ProfScope prof(kKindStep, stream);
        if (io_dtype == MAMBA_BF16)
            state_update_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(a);
        else
            state_update_kernel<float><<<grid, kThreads, 0, stream>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

}  // extern "C"
