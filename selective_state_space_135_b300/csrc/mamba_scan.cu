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
// Design (one GPU, no tensor cores: the work is an elementwise recurrence
// whose cost is one exp and four fp32 multiply/adds per state entry and step):
//   * A CTA is four warps (one per SM sub-partition).  SPLIT warps share a
//     block of 32 channels, one lane per channel, each warp holding 1/SPLIT
//     of the padded state in registers: for dstate > 8, SPLIT = 2 (8 entries
//     a lane, 64 channels per CTA) when the channel tiles give every SM at
//     least two, else SPLIT = 4 (4 entries a lane, 32 channels per CTA);
//     SPLIT = 2 for dstate <= 8.  Every B/C load of a warp is therefore a
//     single-address broadcast, and each SM sub-partition runs two or more
//     warps (one warp alone cannot issue packed FMAs back to back).  The CTA
//     walks time in tiles of one 32-byte row per channel (16 bf16 or 8 fp32
//     steps).
//   * u, delta, z and y tiles move by tensor-map bulk copies
//     (cp.async.bulk.tensor, completion on an mbarrier ring), 32-byte
//     swizzled so that the per-lane row accesses are bank-conflict free.
//   * B and C (shared by all channels of a batch entry) are packed once per
//     call by a small kernel into fp32 rows of (B pair, C pair) per step and
//     staged by the same bulk copies.
//   * Per tile each slice computes Delta and Delta*u for 1/SPLIT of the
//     steps, two steps at a time with packed fp32x2 arithmetic, and writes
//     them to shared memory as the duplicated operand pairs the step's
//     packed multiplies take; every slice runs the recurrence over the
//     tile; and each slice finishes 1/SPLIT of the outputs (all partial sums
//     C.h in slice order, skip term, gate), again two steps at a time: no
//     per-token work is done twice.
//   * The expanded (b, d, t, n) tensor is never materialised: Abar and the
//     input term live only in registers; the state leaves the SM only at the
//     end of a work unit.
//   * Work units are channel tiles over the whole sequence; tiles that do
//     not fill a whole wave, and all tiles when there are fewer than SMs,
//     are cut into time chunks: a summary pass computes each chunk's
//     (prod Abar, end state from zero), a carry pass composes them in order,
//     and the main pass restarts every chunk from its exact carried-in state.
//   * bf16 I/O keeps Delta in log2 units (Delta' = Delta / ln 2, B scaled by
//     ln 2 when packed) so that Abar = ex2(Delta' * A) needs one multiply and
//     one hardware ex2; fp32 I/O uses the library expf/log1pf.  State and
//     accumulation are fp32 in both.  Packed fp32x2 multiply/FMA (sm_100+)
//     halves the instruction count of the state update.

#include "scan_common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <vector>

namespace mamba {

// ---------------------------------------------------------------------------
// device-side helpers
// ---------------------------------------------------------------------------

__device__ int g_error_word;  // nonzero once a bounded device wait gave up

constexpr int kThreads = 128;        // threads per CTA of the state-update kernel
constexpr int kMaxStages = 4;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per wait

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
// Non-blocking test of phase completion (mbarrier.test_wait): unlike
// try_wait it never suspends the thread, so a phase that has already
// completed is seen at once.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
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
// The global timer is read only after 4096 unsuccessful polls: reading it is
// slow, and a wait that ends within a few microseconds never needs it.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    for (int i = 0; i < 4096; ++i)
        if (mbar_test_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (unsigned it = 0;; ++it) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && global_ns() - t0 > limit_ns) return false;
    }
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Tensor-map copies (cp.async.bulk.tensor): one instruction moves a whole
// box between global and shared memory.
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

// ---------------------------------------------------------------------------
// scan kernels
// ---------------------------------------------------------------------------

constexpr int kScanWarps = 4;   // warps per CTA, one per SM sub-partition
// Five resident CTAs per SM is all the shared memory allows (about 45 KB
// each); saying so lets ptxas spend up to 102 registers a thread on running
// the exponentials of the coming steps further ahead.  Measured on B300: the
// Mamba-130M layer scan 187 -> 163 us, the Mamba-2.8B layer 234 -> 218 us.
#ifndef MAMBA_SCAN_MIN_BLOCKS
#define MAMBA_SCAN_MIN_BLOCKS 5
#endif
constexpr int kScanMinBlocks = MAMBA_SCAN_MIN_BLOCKS;
// SPLIT warps share a block of 32 channels, each holding 1/SPLIT of the
// state; a CTA therefore covers 32 * kScanWarps / SPLIT channels.
template <int SPLIT>
constexpr int channels_per_cta() { return 32 * kScanWarps / SPLIT; }

// One 16-byte chunk of a row <-> fp32 values (8 for bf16, 4 for fp32).
template <typename T> struct Chunk;
// One 16-byte chunk of a row <-> fp32 pairs of consecutive steps (4 pairs
// for bf16, 2 for fp32), the operands of packed fp32x2 arithmetic.
template <> struct Chunk<float> {
    static constexpr int G = 4;
    __device__ static void load(const unsigned char* p, float2* v) {
        const float4 r = *reinterpret_cast<const float4*>(p);
        v[0] = make_float2(r.x, r.y);
        v[1] = make_float2(r.z, r.w);
    }
    __device__ static void store(unsigned char* p, const float2* v) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
    }
};
template <> struct Chunk<__nv_bfloat16> {
    static constexpr int G = 8;
    __device__ static void load(const unsigned char* p, float2* v) {
        const uint4 r = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    }
    __device__ static void store(unsigned char* p, const float2* v) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 q = __floats2bfloat162_rn(v[i].x, v[i].y);
            w[i] = *reinterpret_cast<uint32_t*>(&q);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// Softplus of two steps in log2 units: element by element the arithmetic
// of softplus_log2_fast (each half of a packed operation rounds as the
// scalar one), with the multiplies and adds packed in pairs.
__device__ __forceinline__ float2 softplus2_log2(float2 t) {
    const float2 x = make_float2(ex2_approx(-fabsf(t.x)), ex2_approx(-fabsf(t.y)));
    const float2 series =
        __fmul2_rn(x, __ffma2_rn(x, make_float2(-0.5f * kLog2e, -0.5f * kLog2e),
                                 make_float2(kLog2e, kLog2e)));
    const float2 xp1 = __fadd2_rn(x, make_float2(1.0f, 1.0f));
    const float2 full = make_float2(lg2_approx(xp1.x), lg2_approx(xp1.y));
    const float2 r = make_float2(x.x < 0.0078125f ? series.x : full.x,
                                 x.y < 0.0078125f ? series.y : full.y);
    return __fadd2_rn(make_float2(fmaxf(t.x, 0.0f), fmaxf(t.y, 0.0f)), r);
}

// silu of two values (silu_f, packed): accurate z / (1 + e^-z), or on the
// fast path h + h * tanh(h) with h = z / 2.
template <bool ACC>
__device__ __forceinline__ float2 silu2(float2 z) {
    if (ACC) return make_float2(silu_f<true>(z.x), silu_f<true>(z.y));
    const float2 h = __fmul2_rn(z, make_float2(0.5f, 0.5f));
    return __ffma2_rn(h, make_float2(tanh_approx(h.x), tanh_approx(h.y)), h);
}

// Packs B and C of every step into one fp32 row of 2*NP values, in the order
// the scan reads them: for each pair j of state entries the float4
// (s*B[2j], s*B[2j+1], C[2j], C[2j+1]); entries n >= N are zero.  s is ln 2
// when the scan keeps Delta in log2 units, else 1.  One thread per
// (batch, step, pair); consecutive threads read consecutive steps.
template <typename T>
__global__ void pack_bc_kernel(const T* __restrict__ B, const T* __restrict__ C,
                               float4* __restrict__ out, long long batch, long long L, int N,
                               int NP, float scale) {
    const int half = NP / 2;
    const long long total = batch * L * half;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long bj = i / L, t = i - bj * L;   // bj = b * half + j
        const long long b = bj / half;
        const int j = (int)(bj - b * half);
        const int n0 = 2 * j, n1 = 2 * j + 1;
        const long long nbc = batch * N * L;   // extent of B and C
        (void)nbc;
        const long long i0 = b * N * L + (long long)n0 * L + t, i1 = i0 + L;
        float4 v;
        v.x = n0 < N ? scale * IO<T>::to_f(MAMBA_LD(B, i0, nbc)) : 0.0f;
        v.y = n1 < N ? scale * IO<T>::to_f(MAMBA_LD(B, i1, nbc)) : 0.0f;
        v.z = n0 < N ? IO<T>::to_f(MAMBA_LD(C, i0, nbc)) : 0.0f;
        v.w = n1 < N ? IO<T>::to_f(MAMBA_LD(C, i1, nbc)) : 0.0f;
        MAMBA_ST(out, (b * L + t) * half + j, total, v);
    }
}

struct ScanArgs {
    CUtensorMap m_u, m_dl, m_z, m_y, m_bc;   // valid when use_tma
    const void* u;
    const void* delta;
    const void* z;
    const float4* bc;  // packed B/C rows [batch][seqlen][NP / 2]
    const float* dt_bias;
    const float* A;
    const float* D_skip;
    void* y;
    float* final_state;
    float* ws_P;  // chunk decay products  [(k * tail_rows + wrow) * N + n]
    float* ws_h;  // chunk end states, then carried-in states (same layout)
    const float* h0;       // initial state (batch, dim, N), or null for zero
    const int* seqlens;    // per batch entry: steps in use, or null for all
    float* ckpt;           // checkpoint modes: [batch][ck_tiles][NP / 4][dim][4], the
                           // state before every step that is a multiple of kBwdTile
    int ck_tiles;
    long long dim;
    long long seqlen;
    long long chunk_len;  // multiple of the time tile
    int batch;
    int dstate;
    int use_tma;
    int stages;
    int ch;                // channels per CTA
    int groups_per_batch;  // ceil(dim / ch)
    int n_groups;          // batch * groups_per_batch
    int n_full;            // groups [0, n_full) run the whole sequence
    int nchunks;           // time chunks of each remaining ("tail") group
    int tail_rows;         // (n_groups - n_full) * ch
    int unit_offset;       // first unit of this launch (main pass)
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
template <bool STATE_ONLY>
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
    w.d0 = (g % a.groups_per_batch) * a.ch;
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
// per-lane 16-byte row accesses of a warp bank-conflict free.
//   [0, 1024)       stage mbarriers
//   stage s         u | delta | z tiles (CH x 64 B each) | packed B/C (TT x 2*NP fp32)
//   y tile          CH x 64 B
//   du              (Delta, Delta*u) of every (step, channel) of a tile, as
//                   float4 (Delta_t, Delta_t+1, du_t, du_t+1) per pair of steps
//   part            sum_n C*h of each slice of the state for the steps other
//                   slices finish, [SPLIT][TT - TT/SPLIT][CH] fp32
template <typename T, int NT, int SPLIT>
struct ScanLayout {
    static constexpr int CH = channels_per_cta<SPLIT>();
    static constexpr int NP = SPLIT * NT;             // padded state size
    static constexpr int kTT = 64 / (int)sizeof(T);   // steps per tile
    static constexpr int kG = 16 / (int)sizeof(T);    // steps per 16-byte chunk
    static constexpr int kRows = CH * 64;
    static constexpr int kBCBytes = kTT * 2 * NP * 4;
    static constexpr int kBC = (kBCBytes + 1023) / 1024 * 1024;
    static constexpr int kStage = 3 * kRows + kBC;
    static constexpr int kDU = kTT * CH * 8;
    static constexpr int kPart = SPLIT * (kTT - kTT / SPLIT) * CH * 4;
    __host__ __device__ static constexpr int stage(int s) { return 1024 + s * kStage; }
    __host__ __device__ static constexpr int ybuf(int stages) { return stage(stages); }
    __host__ __device__ static constexpr int du(int stages) { return ybuf(stages) + kRows; }
    __host__ __device__ static constexpr int part(int stages) { return du(stages) + kDU; }
    __host__ __device__ static constexpr int bytes(int stages) {
        return part(stages) + kPart + 1024;   // + slack to align the base
    }
};

__device__ __forceinline__ int swz(int row, int chunk) {
    return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
}

// Abar = exp(Delta * A) of one step for the NT state entries (NT/2 pairs).
// Fast path: dt is Delta / ln 2, so Abar = ex2(dt * A).
template <int NT, bool ACC>
__device__ __forceinline__ void abar_step(float2 (&ab)[NT / 2], const float2 (&a2)[NT / 2],
                                          float dt) {
    const float2 dt2 = make_float2(dt, dt);
#pragma unroll
    for (int i = 0; i < NT / 2; ++i) {
        if constexpr (ACC) {
            ab[i] = make_float2(expf(dt * a2[i].x), expf(dt * a2[i].y));
        } else {
            const float2 arg = __fmul2_rn(dt2, a2[i]);
            ab[i] = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
        }
    }
}

// Per-lane constants of the zero-order-hold input term (see zoh_term).
template <int NT>
struct ZohK {
    float2 ia[NT / 2];   // fast path: 1 / (ln2 * A), 0 where A == 0
    float2 e[NT / 2];    // fast path: 1 where A == 0 (Euler limit), else 0
};

// Input term of one state pair.  Euler (the default): (Delta*u) * B, with
// du = Delta*u.  Zero-order hold, the textbook exact discretisation of
// h' = A h + B x over a step Delta with x held constant (the pages print
// only Abar = exp(Delta*A); with this input term the gated-RNN identity of
// Theorem 1, page "Mamba: linear-time sequence modeling with selective state
// spaces", "Main results", holds exactly): for diagonal A the input weight
// is (exp(Delta*A) - 1) / A per state entry, which tends to Delta as A -> 0;
// here du = u and dt is Delta (log2 units on the fast path, where B carries
// the factor ln 2).  The fast path forms the weight from the step's Abar:
// Abar * ia - ia, plus dt where A == 0.
template <int NT, bool ACC, bool ZOH>
__device__ __forceinline__ float2 input_term(int i, const float2& ab, const float2& a2,
                                             const ZohK<NT>& zk, float dt, float du,
                                             const float4& bc) {
    const float2 b2 = make_float2(bc.x, bc.y);
    if constexpr (!ZOH) {
        return __fmul2_rn(make_float2(du, du), b2);
    } else if constexpr (ACC) {
        const float w0 = a2.x != 0.0f ? expm1f(dt * a2.x) / a2.x : dt;
        const float w1 = a2.y != 0.0f ? expm1f(dt * a2.y) / a2.y : dt;
        return make_float2(w0 * du * b2.x, w1 * du * b2.y);
    } else {
        float2 w = __ffma2_rn(ab, zk.ia[i], make_float2(-zk.ia[i].x, -zk.ia[i].y));
        w = __ffma2_rn(zk.e[i], make_float2(dt, dt), w);
        return __fmul2_rn(w, __fmul2_rn(make_float2(du, du), b2));
    }
}

// One time step of the NT state entries of one channel given Abar:
//   h <- Abar * h + (input term) ;  returns sum_n C*h.
// bc holds the step's NT/2 float4 (B pair, C pair), the same for every lane
// of the warp (on the fast path B carries the factor ln 2 that turns the
// log2-unit Delta back into natural units).  All input terms are formed
// before the state updates; sum_n C*h is one packed multiply-add chain.
template <int NT, bool ACC, bool ZOH, bool STATE_ONLY>
__device__ __forceinline__ float state_step(float2 (&h2)[NT / 2], const float2 (&ab)[NT / 2],
                                            const float2 (&a2)[NT / 2], const ZohK<NT>& zk,
                                            float dt, float du, const float4 (&bc)[NT / 2]) {
    float2 bx[NT / 2];
#pragma unroll
    for (int i = 0; i < NT / 2; ++i) bx[i] = input_term<NT, ACC, ZOH>(i, ab[i], a2[i], zk, dt, du, bc[i]);
#pragma unroll
    for (int i = 0; i < NT / 2; ++i) h2[i] = __ffma2_rn(ab[i], h2[i], bx[i]);
    if constexpr (STATE_ONLY) {
        return 0.0f;
    } else {
        float2 acc = __fmul2_rn(make_float2(bc[0].z, bc[0].w), h2[0]);
#pragma unroll
        for (int i = 1; i < NT / 2; ++i) acc = __ffma2_rn(make_float2(bc[i].z, bc[i].w), h2[i], acc);
        return acc.x + acc.y;
    }
}

// One time step of the state (as state_step) fused with Abar of the next
// step (as abar_step), pair by pair, so that the ex2 work of step t+1 sits
// between the multiply/adds of step t in the instruction stream instead of
// stalling the warp in one burst.
template <int NT, bool ACC, bool ZOH, bool STATE_ONLY>
__device__ __forceinline__ float fused_step(float2 (&h2)[NT / 2], const float2 (&ab)[NT / 2],
                                            float2 (&an)[NT / 2], const float2 (&a2)[NT / 2],
                                            const ZohK<NT>& zk, float dt_next, float dt,
                                            float du, const float4 (&bc)[NT / 2]) {
    const float2 dt2 = make_float2(dt_next, dt_next);
    const float2 du2 = make_float2(du, du);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < NT / 2; ++i) {
        if constexpr (ACC) {
            an[i] = make_float2(expf(dt_next * a2[i].x), expf(dt_next * a2[i].y));
        } else {
            const float2 arg = __fmul2_rn(dt2, a2[i]);
            an[i] = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
        }
        float2 bx;
        if constexpr (!ZOH) bx = __fmul2_rn(du2, make_float2(bc[i].x, bc[i].y));
        else bx = input_term<NT, ACC, ZOH>(i, ab[i], a2[i], zk, dt, du, bc[i]);
        h2[i] = __ffma2_rn(ab[i], h2[i], bx);
        if constexpr (!STATE_ONLY) {
            const float2 cp = make_float2(bc[i].z, bc[i].w);
            acc = i == 0 ? __fmul2_rn(cp, h2[i]) : __ffma2_rn(cp, h2[i], acc);
        }
    }
    return STATE_ONLY ? 0.0f : acc.x + acc.y;
}

template <int NT>
__device__ __forceinline__ void load_bc(float4 (&bc)[NT / 2], const float4* row) {
#pragma unroll
    for (int i = 0; i < NT / 2; ++i) bc[i] = row[i];
}

// The scan over one work unit (CH channels x a time range).  With
// CW = kScanWarps / SPLIT channel blocks per CTA, warp w holds channels
// [32*(w % CW), 32*(w % CW) + 32) of the tile, one lane per channel, and
// state entries [NT*(w / CW), NT*(w / CW) + NT) of each: the SPLIT warps of
// a channel block split the state, so every B/C load of a warp is a
// single-address broadcast.  Per tile:
//   (1) each slice computes Delta and Delta*u for 1/SPLIT of the steps into
//       shared memory (no per-token work is done twice);
//   (2) every slice runs the recurrence over all steps of the tile and
//       stores its partial sums sum_n C*h;
//   (3) each slice finishes 1/SPLIT of the outputs: all partial sums (in a
//       fixed order), skip term and gate.
// STATE_ONLY is the chunk-summary pass: no C, z or y; it returns
// (exp(A*sum Delta), h_end).  MODE: kModePlain (Euler, zero initial state,
// every entry uses all steps), kModeExt (Euler with an initial state and
// per-entry lengths) or kModeExtZoh (the same with the zero-order-hold input
// term).  The plain mode is compiled without the extensions: their per-tile
// bookkeeping costs about 2% on B300.
// kModeCkpt: the Euler scan from an initial state with no outputs, writing
// state checkpoints for the backward pass; kModeTrain: the same scan with
// its outputs and the checkpoints (a training forward).
enum { kModePlain = 0, kModeExt = 1, kModeExtZoh = 2, kModeCkpt = 3, kModeTrain = 4 };
template <typename T, int NT, int SPLIT, bool STATE_ONLY, bool SOFTPLUS, bool HAS_Z, int MODE>
__global__ void __launch_bounds__(32 * kScanWarps, kScanMinBlocks)
scan_kernel(const __grid_constant__ ScanArgs a) {
    using Lay = ScanLayout<T, NT, SPLIT>;
    using CK = Chunk<T>;
    constexpr int NP = Lay::NP, CH = Lay::CH, CW = kScanWarps / SPLIT;
    constexpr int TT = Lay::kTT, G = Lay::kG, HT = TT / SPLIT, QC = HT / G;
    constexpr int kNThr = 32 * kScanWarps;
    constexpr bool ACC = IO<T>::kAccurate;
    constexpr int kNPair = NT / 2;
    constexpr bool CKPT = MODE == kModeCkpt;
    constexpr bool OUT = !STATE_ONLY && !CKPT;   // y (and the partial sums it needs)
    constexpr bool CKW = (CKPT || MODE == kModeTrain) && !STATE_ONLY;   // writes checkpoints
    constexpr bool has_z = OUT && HAS_Z;
    constexpr bool EXT = MODE != kModePlain;
    constexpr bool ZOH = MODE == kModeExtZoh;
    static_assert(NT % 2 == 0 && NP <= kMaxN, "bad state size");
    static_assert(TT <= 32, "the checkpoint schedule of a tile is a 32-bit mask");
    static_assert(CK::G == G && QC * G == HT && QC >= 1, "a slice's steps are whole 16-byte chunks");

    // Offset the __shared__ array itself (not a pointer rebuilt from an
    // integer) so that every access below stays a shared-memory access.
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hh = warp / CW;                 // which slice of the state
    const int c = (warp % CW) * 32 + lane;    // channel within the tile
    const Unit w = decode_unit<STATE_ONLY>(a, (int)blockIdx.x + (STATE_ONLY ? 0 : a.unit_offset));
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
    // extents for the index checks of debug builds
    const long long big_extent = (long long)a.batch * dim * L_;
    const long long ws_extent = (long long)(a.nchunks - 1) * a.tail_rows * N;
    (void)big_extent;
    (void)ws_extent;
    // steps in use for this batch entry: past them Delta is 0 (the state is
    // kept) and y is 0
    long long t_end = w.t1;   // end of the live steps of this unit
    if constexpr (EXT) {
        if (a.seqlens) t_end = min(t_end, max(0LL, (long long)MAMBA_LD(a.seqlens, w.b, a.batch)));
    }

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    unsigned char* yt = smem + Lay::ybuf(stages);
    float4* du_s = reinterpret_cast<float4*>(smem + Lay::du(stages));      // [TT/2][CH]
    // [SPLIT][TT - HT][CH]: slice q's partial of step t sits at row
    // (t < q*HT ? t : t - HT), skipping the steps slice q finishes itself
    float* part_s = reinterpret_cast<float*>(smem + Lay::part(stages));

    // ---- per-thread constants and initial state ----
    // A unit that starts at t = 0 starts from the caller's initial state
    // (zero without one); a later chunk of the main pass from the carried
    // state; a later chunk of the summary pass from zero.
    float2 h2[kNPair], a2[kNPair];
    ZohK<NT> zk;
    (void)zk;
#pragma unroll
    for (int i = 0; i < kNPair; ++i) {
        float av[2], hv[2], iv[2], ev[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int n = hh * NT + 2 * i + j;
            const bool ok = chan_ok && n < N;
            av[j] = ok ? MAMBA_LD(a.A, (long long)d * N + n, dim * N) : 0.0f;
            float h0 = 0.0f;
            if (ok) {
                if (w.tail >= 0 && w.k > 0) {
                    if (!STATE_ONLY)
                        h0 = MAMBA_LD(a.ws_h, ((long long)(w.k - 1) * a.tail_rows + wrow) * N + n,
                                      ws_extent);
                } else if (EXT && a.h0) {
                    h0 = MAMBA_LD(a.h0, row * N + n, (long long)a.batch * dim * N);
                }
            }
            hv[j] = h0;
            iv[j] = av[j] != 0.0f ? 1.0f / (kLn2 * av[j]) : 0.0f;
            ev[j] = av[j] != 0.0f ? 0.0f : 1.0f;
        }
        a2[i] = make_float2(av[0], av[1]);
        h2[i] = make_float2(hv[0], hv[1]);
        zk.ia[i] = make_float2(iv[0], iv[1]);
        zk.e[i] = make_float2(ev[0], ev[1]);
    }
    const float bias0 = (chan_ok && a.dt_bias) ? MAMBA_LD(a.dt_bias, d, dim) : 0.0f;
    const float bias = ACC ? bias0 : bias0 * kLog2e;
    const float2 bias2 = make_float2(bias, bias);
    const float dsk = (chan_ok && a.D_skip) ? MAMBA_LD(a.D_skip, d, dim) : 0.0f;
    const float2 dsk2 = make_float2(dsk, dsk);
    float dsum = 0.0f;  // sum of Delta over the unit (summary pass)

    const int ntens = has_z ? 3 : 2;

    // thread 0: tensor-map copies of tile `it` into stage `s`
    auto issue_tile = [&](int it, int s) {
        const int tt0 = (int)(w.t0 + (long long)it * TT);
        // box origins inside the tensors (the copies themselves clip)
        (void)(MAMBA_IN(tt0, L_) && MAMBA_IN(w.d0, dim) && MAMBA_IN(w.b, a.batch));
        const uint32_t bar = smem_u32(&bars[s]);
        unsigned char* st = smem + Lay::stage(s);
        mbar_arrive_expect_tx(bar, (uint32_t)(ntens * Lay::kRows + Lay::kBCBytes));
        tma_load_3d(smem_u32(st), &a.m_u, tt0, w.d0, w.b, bar);
        tma_load_3d(smem_u32(st + Lay::kRows), &a.m_dl, tt0, w.d0, w.b, bar);
        if constexpr (has_z)
            tma_load_3d(smem_u32(st + 2 * Lay::kRows), &a.m_z, tt0, w.d0, w.b, bar);
        tma_load_3d(smem_u32(st + 3 * Lay::kRows), &a.m_bc, 0, tt0, w.b, bar);
    };

    // all threads: element-wise, bounds-checked fill of stage `sidx` (any shape)
    auto plain_tile = [&](int it, int sidx) {
        const long long tt0 = w.t0 + (long long)it * TT;
        const int nv = (int)min((long long)TT, L_ - tt0);
        unsigned char* st = smem + Lay::stage(sidx);
        for (int e = tid; e < ntens * CH * TT; e += kNThr) {
            const int tsr = e / (CH * TT), rem = e % (CH * TT);
            const int cc = rem / TT, t = rem % TT;
            const T* src = static_cast<const T*>(tsr == 0 ? a.u : (tsr == 1 ? a.delta : a.z));
            T v = IO<T>::from_f(0.0f);
            if (cc < rows_valid && t < nv)
                v = MAMBA_LD(src, ((long long)w.b * dim + w.d0 + cc) * L_ + tt0 + t, big_extent);
            const int byte = t * (int)sizeof(T);
            *reinterpret_cast<T*>(st + tsr * Lay::kRows + swz(cc, byte >> 4) + (byte & 15)) = v;
        }
        float4* bcs = reinterpret_cast<float4*>(st + 3 * Lay::kRows);
        for (int e = tid; e < TT * (NP / 2); e += kNThr) {
            const int t = e / (NP / 2), j = e % (NP / 2);
            bcs[e] = t < nv ? MAMBA_LD(a.bc, ((long long)w.b * L_ + tt0 + t) * (NP / 2) + j,
                                       (long long)a.batch * L_ * (NP / 2))
                            : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
    };

    if (tma) {
        if (tid == 0) {
            for (int s = 0; s < stages; ++s) mbar_init(smem_u32(&bars[s]), 1);
            fence_mbar_init();
            prefetch_map(&a.m_u);
            prefetch_map(&a.m_dl);
            prefetch_map(&a.m_bc);
            if constexpr (has_z) prefetch_map(&a.m_z);
            if (OUT) prefetch_map(&a.m_y);
        }
        __syncthreads();
        if (tid == 0)
            for (int s = 0; s < stages && s < ntiles; ++s) issue_tile(s, s);
    }

    int issued = tma ? min(stages, ntiles) : 0;
    bool aborted = false;

    // Wait for the data of tile `it_` in stage `st_`.  Only lane 0 of each
    // warp polls the mbarrier (polling by every thread of the SM is slow);
    // __syncwarp then orders the other lanes after it.  The plain path fills
    // the stage cooperatively instead.  Returns true when the wait ran out.
    auto acquire = [&](int it_, int st_, uint32_t par_) -> bool {
        if (tma) {
            int to = 0;
            if (lane == 0) to = mbar_wait_bounded(smem_u32(&bars[st_]), par_) ? 0 : 1;
            __syncwarp();
            return __shfl_sync(0xffffffffu, to, 0) != 0;
        }
        plain_tile(it_, st_);
        __syncthreads();
        return false;
    };

    // Delta (log2 units on the fast path) of two steps from the raw delta values
    auto delta2_of = [&](float2 dv) -> float2 {
        if constexpr (ACC) {
            const float2 sarg = __fadd2_rn(dv, bias2);
            if (!SOFTPLUS) return sarg;
            return make_float2(sarg.x > 20.0f ? sarg.x : log1pf(expf(sarg.x)),
                               sarg.y > 20.0f ? sarg.y : log1pf(expf(sarg.y)));
        } else {
            // s * log2(e); softplus in log2 units: log2(1 + 2^tl)
            const float2 tl = __ffma2_rn(dv, make_float2(kLog2e, kLog2e), bias2);
            return SOFTPLUS ? softplus2_log2(tl) : tl;
        }
    };

    // (1) Delta and Delta*u (Euler) or u (zero-order hold) of this slice's
    //     steps [hh*HT, hh*HT + HT) of a tile into du_s, two steps at a time
    //     with packed arithmetic: independent chains, back to back
    auto phase1 = [&](const unsigned char* st_, int nv_) {
#pragma unroll
        for (int q = 0; q < QC; ++q) {
            const int ck = hh * QC + q;
            const int off = swz(c, ck);
            float2 uv[G / 2], dv[G / 2];
            CK::load(st_ + Lay::kRows + off, dv);
            CK::load(st_ + off, uv);
#pragma unroll
            for (int j = 0; j < G / 2; ++j) {
                float2 v = delta2_of(dv[j]);
                float2 du = ZOH ? uv[j] : __fmul2_rn(v, uv[j]);
                const int t = ck * G + 2 * j;
                if (nv_ < TT) {   // past the live steps the state is kept (uniform branch)
                    if (t >= nv_) v.x = du.x = 0.0f;
                    if (t + 1 >= nv_) v.y = du.y = 0.0f;
                }
                du_s[(t / 2) * CH + c] = make_float4(v.x, v.y, du.x, du.y);
            }
        }
    };

    // checkpoint modes: this warp's NT entries of the state before step
    // `step` (a multiple of kBwdTile) into the quad-major layout
    // ckpt[(((b * ck_tiles + step / kBwdTile) * NP / 4 + n / 4) * dim + d) * 4 + n % 4]
    // (entries in quads of four, adjacent channels adjacent: a warp's store
    // of a quad is 512 contiguous bytes).  The unit writes its checkpoints in
    // step order: ck_at is the element index of the next one's first entry,
    // advanced by NP * dim per write.  A unit from step 0 writes checkpoint 0
    // (the initial state) first; a unit from t0 > 0 writes those after its
    // steps, from t0 / kBwdTile + 1 on (the one at t0 itself, if any, is the
    // end state of the unit before it).
    long long ck_at = 0;
    if constexpr (CKW) {
        const long long k0 = w.t0 == 0 ? 0 : w.t0 / kBwdTile + 1;
        const int n_first = hh * NT;
        ck_at = ((((long long)w.b * a.ck_tiles + k0) * (NP / 4) + n_first / 4) * dim + d) * 4 +
                n_first % 4;
    }
    auto write_ckpt = [&](long long step) {
        if (chan_ok && step < L_) {
            const long long ext = (long long)a.batch * dim * a.ck_tiles * NP;
            (void)ext;
            if constexpr (NT >= 4) {   // whole quads: one 16-byte store each
#pragma unroll
                for (int qd = 0; qd < NT / 4; ++qd) {
                    const long long at = ck_at + (long long)qd * dim * 4;
                    if (MAMBA_IN(at, ext) && MAMBA_IN(at + 3, ext))
                        *reinterpret_cast<float4*>(a.ckpt + at) =
                            make_float4(h2[2 * qd].x, h2[2 * qd].y, h2[2 * qd + 1].x,
                                        h2[2 * qd + 1].y);
                }
            } else {   // one pair, half a quad
                if (MAMBA_IN(ck_at, ext) && MAMBA_IN(ck_at + 1, ext))
                    *reinterpret_cast<float2*>(a.ckpt + ck_at) = h2[0];
            }
        }
        ck_at += (long long)NP * dim;
    };
    (void)write_ckpt;
    (void)ck_at;
    if constexpr (CKW) {
        if (w.t0 == 0) write_ckpt(0);   // the initial state
    }

    int stage = 0;          // stage of tile `it`
    uint32_t parity = 0;    // mbarrier phase parity of tile `it`
    if (ntiles > 0) {
        const bool to = acquire(0, 0, 0);
        phase1(smem + Lay::stage(0), (int)max(-1LL, min((long long)TT, t_end - w.t0)));
        aborted = __syncthreads_or(to);
    }

    for (int it = 0; it < ntiles && !aborted; ++it) {
        const long long tt0 = w.t0 + (long long)it * TT;
        // bit t: tt0 + t + 1 is a multiple of kBwdTile (a checkpoint after step t)
        uint32_t ckmask = 0;
        if constexpr (CKW) {
            for (int t1 = kBwdTile - (int)(tt0 % kBwdTile); t1 <= TT; t1 += kBwdTile)
                ckmask |= 1u << (t1 - 1);
        }
        (void)ckmask;
        const int nv = (int)min((long long)TT, w.t1 - tt0);   // steps of this unit in the tile
        // with per-entry lengths, the steps of the tile past them get y = 0
        // (without, steps past the sequence are not stored at all)
        const int ylim =
            (EXT && a.seqlens && t_end - tt0 < TT) ? (int)max(0LL, t_end - tt0) : TT;
        const unsigned char* st = smem + Lay::stage(stage);
        const unsigned char* ut = st;
        const unsigned char* zt = st + 2 * Lay::kRows;
        const float4* bct = reinterpret_cast<const float4*>(st + 3 * Lay::kRows) + hh * kNPair;

        // (2) the recurrence over the tile for this half of the state, as a
        //     three-deep pipeline: at step t the (Delta, Delta*u) of step t+2
        //     and the B/C row of step t+1 are loaded, Abar of step t+1 is
        //     formed, and step t updates the state
        float own[HT];   // partial sums of the steps this slice finishes
        (void)own;
        {
            // where this slice's partial of step t goes: registers for its own
            // steps, row t (steps before them) or row t - HT (steps after)
            float* pseg[SPLIT];
            bool mine[SPLIT];
#pragma unroll
            for (int k = 0; k < SPLIT; ++k) {
                mine[k] = k == hh;
                pseg[k] = part_s + (hh * (TT - HT) - (k < hh ? 0 : HT)) * CH + c;
            }
            (void)pseg;
            (void)mine;
            // (Delta, Delta*u) of the pairs of steps in a ring of three
            // (pair t/2 in slot (t/2) % 3, loaded two pairs ahead), Abar and
            // the B/C row of the current and the next step in rings of two:
            // every index is a compile-time constant of the unrolled loop, so
            // nothing is copied from one step to the next
            float4 qa[3];
            float2 abuf[2][kNPair];
            float4 bbuf[2][kNPair];
            qa[0] = du_s[c];
            qa[1] = du_s[CH + c];
            qa[2] = qa[1];
            abar_step<NT, ACC>(abuf[0], a2, qa[0].x);
            load_bc<NT>(bbuf[0], bct);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                const int cur = t & 1, nxt = cur ^ 1;
                const float4& q = qa[(t / 2) % 3];
                const float dt = (t & 1) ? q.y : q.x;
                const float du = (t & 1) ? q.w : q.z;
                const float dtn = (t & 1) ? qa[(t / 2 + 1) % 3].x : q.y;   // Delta of step t+1
                if (!(t & 1) && t + 4 < TT) qa[(t / 2 + 2) % 3] = du_s[(t / 2 + 2) * CH + c];
                float pt;
                if (t + 1 < TT) {
                    load_bc<NT>(bbuf[nxt], bct + (t + 1) * (NP / 2));
                    pt = fused_step<NT, ACC, ZOH, !OUT>(h2, abuf[cur], abuf[nxt], a2, zk, dtn,
                                                        dt, du, bbuf[cur]);
                } else {
                    pt = state_step<NT, ACC, ZOH, !OUT>(h2, abuf[cur], a2, zk, dt, du, bbuf[cur]);
                }
                if constexpr (STATE_ONLY) {
                    dsum += dt;
                } else if constexpr (OUT) {
                    if (mine[t / HT])
                        own[t % HT] = pt;
                    else
                        pseg[t / HT][t * CH] = pt;
                }
                if constexpr (CKW) {
                    // after step t the state is the one before step tt0 + t + 1
                    if (ckmask & (1u << t)) write_ckpt(tt0 + t + 1);
                }
            }
        }
        if (OUT && tma && tid == 0) bulk_wait_read_0();   // y tile free again
        __syncthreads();   // partial sums complete; every read of du_s done

        // next tile's data, then (3) the outputs of this tile together with
        // (1) for the next tile: independent work, issued side by side
        const bool has_next = it + 1 < ntiles;
        const int next_stage = stage + 1 == stages ? 0 : stage + 1;
        const uint32_t next_parity = stage + 1 == stages ? parity ^ 1u : parity;
        bool to = false;
        if (has_next) {
            to = acquire(it + 1, next_stage, next_parity);
            const long long tn0 = tt0 + TT;
            phase1(smem + Lay::stage(next_stage), (int)max(-1LL, min((long long)TT, t_end - tn0)));
        }
        if constexpr (OUT) {
            // the other slices' partials of this slice's steps t = hh*HT + i:
            // slice r = (hh + k) % SPLIT keeps them at row t (r > hh) or t - HT
            const float* pk[SPLIT > 1 ? SPLIT - 1 : 1];
#pragma unroll
            for (int k = 1; k < SPLIT; ++k) {
                const int r = (hh + k) % SPLIT;
                pk[k - 1] = part_s + (r * (TT - HT) + hh * HT - (r > hh ? 0 : HT)) * CH + c;
            }
#pragma unroll
            for (int q = 0; q < QC; ++q) {
                const int ck = hh * QC + q;
                const int off = swz(c, ck);
                float2 uv[G / 2], zv[G / 2], ov[G / 2];
                (void)zv;
                CK::load(ut + off, uv);
                if constexpr (has_z) CK::load(zt + off, zv);
#pragma unroll
                for (int j = 0; j < G / 2; ++j) {
                    // two steps: own partials, then the other slices' in a
                    // fixed rotation
                    const int i = q * G + 2 * j;
                    float2 o = make_float2(own[i], own[i + 1]);
#pragma unroll
                    for (int k = 1; k < SPLIT; ++k)
                        o = __fadd2_rn(o, make_float2(pk[k - 1][i * CH], pk[k - 1][(i + 1) * CH]));
                    o = __ffma2_rn(dsk2, uv[j], o);
                    if constexpr (has_z) o = __fmul2_rn(o, silu2<ACC>(zv[j]));
                    if (EXT && ylim < TT) {   // uniform over the CTA
                        if (i + hh * HT >= ylim) o.x = 0.0f;
                        if (i + 1 + hh * HT >= ylim) o.y = 0.0f;
                    }
                    ov[j] = o;
                }
                CK::store(yt + off, ov);
            }
            if (tma) fence_proxy_async_smem();
        }
        // stage consumed, y tile complete, next tile's du_s ready
        aborted = __syncthreads_or(to);

        if (OUT) {
            if (tma) {
                if (tid == 0) {
                    tma_store_3d(&a.m_y, smem_u32(yt), (int)tt0, w.d0, w.b);
                    bulk_commit();
                }
            } else {
                for (int e = tid; e < CH * TT; e += kNThr) {
                    const int cc = e / TT, t = e % TT;
                    if (cc < rows_valid && t < nv) {
                        const int byte = t * (int)sizeof(T);
                        MAMBA_ST(static_cast<T*>(a.y),
                                 ((long long)w.b * dim + w.d0 + cc) * L_ + tt0 + t, big_extent,
                                 *reinterpret_cast<const T*>(yt + swz(cc, byte >> 4) + (byte & 15)));
                    }
                }
            }
        }
        if (tma && tid == 0 && issued < ntiles && !aborted) {
            issue_tile(issued, stage);
            ++issued;
        }
        stage = next_stage;
        parity = next_parity;
    }

    if (tma) {
        if (aborted && tid == 0) {
            atomicExch(&g_error_word, 1);
            // let copies still in flight land before the CTA's memory is
            // released; only the last `stages` tiles issued can be in flight
            // (every older one was consumed), and waiting on the parity of an
            // older phase of the same barrier would not return until the bound
            for (int it = max(0, issued - stages); it < issued; ++it)
                (void)mbar_wait_bounded(smem_u32(&bars[it % stages]), (uint32_t)((it / stages) & 1));
        }
        if (OUT && tid == 0) bulk_wait_all();
        __syncthreads();
        if (aborted) return;
    }

    // ---- results that leave the SM: final state or chunk summary ----
    // (the summary also covers the tile's channels past `dim`, whose state
    // stays zero, so that the carry pass reads only written entries)
    if (!chan_ok && !STATE_ONLY) return;
#pragma unroll
    for (int i = 0; i < kNPair; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int n = hh * NT + 2 * i + j;
            if (n >= N) continue;
            const float hv = j ? h2[i].y : h2[i].x;
            if (STATE_ONLY) {
                const long long idx = ((long long)w.k * a.tail_rows + wrow) * N + n;
                const float an = j ? a2[i].y : a2[i].x;
                MAMBA_ST(a.ws_P, idx, ws_extent, ACC ? expf(an * dsum) : ex2_approx(an * dsum));
                MAMBA_ST(a.ws_h, idx, ws_extent, hv);
            } else if (OUT && a.final_state && w.t1 == L_) {
                MAMBA_ST(a.final_state, row * N + n, (long long)a.batch * dim * N, hv);
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
        const long long ext = (long long)(nchunks - 1) * entries;
        (void)ext;
        h = MAMBA_LD(ws_P, idx, ext) * h + MAMBA_LD(ws_h, idx, ext);
        MAMBA_ST(ws_h, idx, ext, h);
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

// Zero-order-hold input weight of one state entry (as the scan's
// input_term): (Abar - 1) / A, Delta where A == 0.  dt is Delta in natural
// units and dA the step's Abar.  The generation step is bound by memory, so
// the division costs nothing here.
template <bool ACC>
__device__ __forceinline__ float zoh_weight(float dA, float dt, float A) {
    if (A == 0.0f) return dt;
    return (ACC ? expm1f(dt * A) : dA - 1.0f) / A;
}

// Four lanes per (b, d) row; lane q owns state entries [4q, 4q + 4).
// SP: softplus on Delta; ZOH: zero-order-hold input term (compile-time, so
// that the common step carries no per-entry branch).
template <typename T, bool SP, bool ZOH>
__global__ void __launch_bounds__(kThreads)
state_update_kernel(const StepArgs a) {
    constexpr bool ACC = IO<T>::kAccurate;
    const long long gid = (long long)blockIdx.x * kThreads + threadIdx.x;
    const long long row = gid >> 2;
    const int q = (int)(gid & 3);
    const bool ok = row < a.rows;
    const int N = a.dstate;
    float acc = 0.0f, xv = 0.0f, zv = 0.0f, dsk = 0.0f;
    // extents for the index checks of debug builds
    const long long nrow = a.rows, nbn = a.rows / a.dim * N, ndn = a.dim * N, nst = a.rows * N;
    (void)nrow; (void)nbn; (void)ndn; (void)nst;
    if (ok) {
        const long long b = row / a.dim, d = row % a.dim;
        const T* xp = static_cast<const T*>(a.x);
        const T* dp = static_cast<const T*>(a.delta);
        const T* zp = static_cast<const T*>(a.z);
        const T* Bp = static_cast<const T*>(a.B);
        const T* Cp = static_cast<const T*>(a.C);
        xv = IO<T>::to_f(MAMBA_LD(xp, row, nrow));
        const float s = IO<T>::to_f(MAMBA_LD(dp, row, nrow)) +
                        (a.dt_bias ? MAMBA_LD(a.dt_bias, d, a.dim) : 0.0f);
        const float dt = SP ? softplus_f<ACC>(s) : s;
        const float du = dt * xv;
        if (a.z) zv = IO<T>::to_f(MAMBA_LD(zp, row, nrow));
        dsk = a.D_skip ? MAMBA_LD(a.D_skip, d, a.dim) : 0.0f;
        const int n0 = 4 * q;
        if (a.vec_state && n0 < N) {
            float4 hv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            const long long hi = row * N + n0;
            if (MAMBA_IN(hi, nst) && MAMBA_IN(hi + 3, nst))
                hv = *reinterpret_cast<const float4*>(a.state + hi);
            float hs[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + j;
                const float An = MAMBA_LD(a.A, d * N + n, ndn);
                const float dA = ACC ? expf(dt * An) : ex2_approx(dt * (An * kLog2e));
                const float bin = ZOH ? zoh_weight<ACC>(dA, dt, An) * xv : du;
                hs[j] = fmaf(dA, hs[j], bin * IO<T>::to_f(MAMBA_LD(Bp, b * N + n, nbn)));
                acc = fmaf(IO<T>::to_f(MAMBA_LD(Cp, b * N + n, nbn)), hs[j], acc);
            }
            if (MAMBA_IN(hi, nst) && MAMBA_IN(hi + 3, nst))
                *reinterpret_cast<float4*>(a.state + hi) = make_float4(hs[0], hs[1], hs[2], hs[3]);
        } else {
            for (int n = n0; n < n0 + 4 && n < N; ++n) {
                const float An = MAMBA_LD(a.A, d * N + n, ndn);
                const float dA = ACC ? expf(dt * An) : ex2_approx(dt * (An * kLog2e));
                const float bin = ZOH ? zoh_weight<ACC>(dA, dt, An) * xv : du;
                const float hn = fmaf(dA, MAMBA_LD(a.state, row * N + n, nst),
                                      bin * IO<T>::to_f(MAMBA_LD(Bp, b * N + n, nbn)));
                MAMBA_ST(a.state, row * N + n, nst, hn);
                acc = fmaf(IO<T>::to_f(MAMBA_LD(Cp, b * N + n, nbn)), hn, acc);
            }
        }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    if (ok && q == 0) {
        float o = acc + dsk * xv;
        if (a.z) o *= silu_f<ACC>(zv);
        MAMBA_ST(static_cast<T*>(a.y), row, nrow, IO<T>::from_f(o));
    }
}

// Vectorised generation step for dstate == 16.  Two lanes per (b, d) row,
// lane q holding state entries [8q, 8q + 8) as two float4.  A block covers
// 32 channels x 8 batch entries, two rows per thread (batch entries bi and
// bi + 4 of the block): every load of both rows is issued before either is
// computed, so each thread keeps 64 bytes of state in flight.  The rows of
// one batch entry are contiguous in memory (coalesced state access) and a
// thread reads its channel's A row once for both.  B and C of a row's half
// are one 16-byte (bf16) or two 16-byte (fp32) loads.  Fast path as in the
// scan: Delta is kept in log2 units and Abar = ex2(Delta' * A).
constexpr int kStepDims = 32, kStepBatches = 4, kStepRows = 2;   // block = 32 x 4 x 2 lanes
template <typename T, bool SP, bool ZOH>
__global__ void __launch_bounds__(2 * kStepDims * kStepBatches, 3)
state_update16_kernel(const StepArgs a) {
    constexpr bool ACC = IO<T>::kAccurate;
    constexpr int N = 16, H = 8, R = kStepRows;
    const int tid = threadIdx.x;
    const int q = tid & 1;
    const int di = (tid >> 1) % kStepDims, bi = (tid >> 1) / kStepDims;
    const long long d = (long long)blockIdx.x * kStepDims + di;
    const long long batch = a.rows / a.dim;
    // extents for the index checks of debug builds
    const long long nrow = a.rows, nbn = batch * N, ndn = a.dim * N, nst = a.rows * N;
    (void)nrow; (void)nbn; (void)ndn; (void)nst;
    const bool dok = d < a.dim && MAMBA_IN(d * N + H * q, ndn) && MAMBA_IN(d * N + H * q + H - 1, ndn);
    float Av[H];
    float bias = 0.0f, dsk = 0.0f;
    if (dok) {
        const float4* Ad = reinterpret_cast<const float4*>(a.A + d * N + H * q);
        const float4 a0 = Ad[0], a1 = Ad[1];
        Av[0] = a0.x; Av[1] = a0.y; Av[2] = a0.z; Av[3] = a0.w;
        Av[4] = a1.x; Av[5] = a1.y; Av[6] = a1.z; Av[7] = a1.w;
        bias = a.dt_bias ? MAMBA_LD(a.dt_bias, d, a.dim) : 0.0f;
        dsk = a.D_skip ? MAMBA_LD(a.D_skip, d, a.dim) : 0.0f;
    }
    // (1) every load of both rows
    bool ok[R];
    long long brow[R];
    // B and C stay packed (bf16: one uint4 per half row) until the update
    constexpr int kBC = sizeof(T) == 2 ? 1 : 2;
    float xv[R], dv[R], zv[R], hs[R][H];
    uint4 Braw[R][kBC], Craw[R][kBC];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const long long b = ((long long)blockIdx.y * R + r) * kStepBatches + bi;
        brow[r] = b;
        const long long row = b * a.dim + d;
        ok[r] = dok && b < batch && MAMBA_IN(b * N + H * q, nbn) && MAMBA_IN(b * N + H * q + H - 1, nbn) &&
                MAMBA_IN(row * N + H * q, nst) && MAMBA_IN(row * N + H * q + H - 1, nst);
        xv[r] = dv[r] = zv[r] = 0.0f;
        if (ok[r]) {
            xv[r] = IO<T>::to_f(MAMBA_LD(static_cast<const T*>(a.x), row, nrow));
            dv[r] = IO<T>::to_f(MAMBA_LD(static_cast<const T*>(a.delta), row, nrow));
            if (a.z) zv[r] = IO<T>::to_f(MAMBA_LD(static_cast<const T*>(a.z), row, nrow));
            const T* Bb = static_cast<const T*>(a.B) + b * N + H * q;
            const T* Cb = static_cast<const T*>(a.C) + b * N + H * q;
#pragma unroll
            for (int k = 0; k < kBC; ++k) {
                Braw[r][k] = reinterpret_cast<const uint4*>(Bb)[k];
                Craw[r][k] = reinterpret_cast<const uint4*>(Cb)[k];
            }
            const float4* hp = reinterpret_cast<const float4*>(a.state + row * N + H * q);
            const float4 h0 = hp[0], h1 = hp[1];
            hs[r][0] = h0.x; hs[r][1] = h0.y; hs[r][2] = h0.z; hs[r][3] = h0.w;
            hs[r][4] = h1.x; hs[r][5] = h1.y; hs[r][6] = h1.z; hs[r][7] = h1.w;
        }
    }
    // (2) the update of both rows, the state stored in place, y
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float acc = 0.0f;
        if (ok[r]) {
            // Delta (log2 units on the fast path), Delta (natural units), Delta*u
            float dt, dtn;
            if constexpr (ACC) {
                const float sarg = dv[r] + bias;
                dt = SP ? softplus_f<true>(sarg) : sarg;
                dtn = dt;
            } else {
                const float tl = fmaf(dv[r], kLog2e, bias * kLog2e);
                dt = SP ? softplus_log2_fast(tl) : tl;
                dtn = dt * kLn2;
            }
            const float du = dtn * xv[r];
            float Bv[H], Cv[H];
#pragma unroll
            for (int k = 0; k < kBC; ++k) {
                IO<T>::unpack(Braw[r][k], Bv + (H / kBC) * k);
                IO<T>::unpack(Craw[r][k], Cv + (H / kBC) * k);
            }
            float acc1 = 0.0f;
#pragma unroll
            for (int k = 0; k < H; ++k) {
                const float dA = ACC ? expf(dt * Av[k]) : ex2_approx(dt * Av[k]);
                const float bin = ZOH ? zoh_weight<ACC>(dA, dtn, Av[k]) * xv[r] : du;
                hs[r][k] = fmaf(dA, hs[r][k], bin * Bv[k]);
                if (k & 1) acc1 = fmaf(Cv[k], hs[r][k], acc1);
                else acc = fmaf(Cv[k], hs[r][k], acc);
            }
            acc += acc1;
            float4* hp = reinterpret_cast<float4*>(a.state + (brow[r] * a.dim + d) * N + H * q);
            hp[0] = make_float4(hs[r][0], hs[r][1], hs[r][2], hs[r][3]);
            hp[1] = make_float4(hs[r][4], hs[r][5], hs[r][6], hs[r][7]);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if (ok[r] && q == 0) {
            float o = acc + dsk * xv[r];
            if (a.z) o *= silu_f<ACC>(zv[r]);
            MAMBA_ST(static_cast<T*>(a.y), brow[r] * a.dim + d, nrow, IO<T>::from_f(o));
        }
    }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that no
// copy and no thread ever completes, with a short limit, then records the
// timeout in the device error word exactly as the scan does, and returns.
// Self-test of the index checks of debug builds: one thread checks an index
// one past the end of an extent, the check records it in the debug word and
// no memory is accessed at all.  In release builds the check is compiled
// out and the kernel does nothing.
__global__ void bounds_selftest_kernel(long long extent) {
    if (threadIdx.x == 0) (void)MAMBA_IN(extent, extent);
}

__global__ void wait_timeout_selftest_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(smem_u32(&bar), 0, limit_ns)) atomicExch(&g_error_word, 1);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

struct Tuning {
    int tail = 0;    // 0 automatic, 1 whole units only, 2 chunk the tail, 3 ... on a side stream
    int stages = 0;  // ring depth (0 = automatic)
    int chunks = 0;  // time chunks for every group (0 = automatic)
    int layout = 0;  // 0 automatic, 1 lane-per-channel kernel, 2 split-state kernel
};

Tuning g_tuning;
std::mutex g_mu;
// source line of the last failed index check seen by mamba_device_status
std::atomic<int> g_debug_last_line{0};

Tuning get_tuning() {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_tuning;
}
std::vector<cudaMemPool_t> g_pools;

// Optional per-launch timing: while enabled, every kernel launch is bracketed
// by two CUDA events recorded on its own stream.
struct ProfRec {
    int kind;
    cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_recs;

ProfScope::ProfScope(int kind, cudaStream_t s) : st(s) {
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
ProfScope::~ProfScope() {
    if (stop) cudaEventRecord(stop, st);
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

// Library-owned side stream and fork/join events of one device, created on
// first use.  The launch sequence that uses them holds g_side_mu.
struct Side {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::vector<Side> g_side;
std::mutex g_side_mu;

int get_side(int dev, Side* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)g_side.size() <= dev) g_side.resize(dev + 1);
    Side& sd = g_side[dev];
    if (!sd.stream) {
        if (cudaStreamCreateWithFlags(&sd.stream, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            sd = Side();
            return MAMBA_ERR_CUDA;
        }
    }
    *out = sd;
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

cudaError_t launch_pack_bc(int io_dtype, const void* B, const void* C, float4* out,
                           long long batch, long long L, int N, int NP, float scale,
                           cudaStream_t stream) {
    int dev = 0;
    cudaGetDevice(&dev);
    const long long items = batch * L * (NP / 2);
    const int blocks = (int)std::max<long long>(
        1, std::min<long long>((items + 255) / 256, 16LL * sm_count(dev)));
    ProfScope prof(kKindPack, stream);
    if (io_dtype == MAMBA_BF16)
        pack_bc_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(B), static_cast<const __nv_bfloat16*>(C), out,
            batch, L, N, NP, scale);
    else
        pack_bc_kernel<float><<<blocks, 256, 0, stream>>>(
            static_cast<const float*>(B), static_cast<const float*>(C), out, batch, L, N, NP,
            scale);
    return cudaGetLastError();
}

template <typename T, int NT, int SPLIT, bool STATE_ONLY, bool SP, bool HZ, int MODE>
cudaError_t launch_scan(const ScanArgs& a, int grid, int smem, cudaStream_t st) {
    auto k = scan_kernel<T, NT, SPLIT, STATE_ONLY, SP, HZ, MODE>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    ProfScope prof(STATE_ONLY ? kKindSummary : kKindScan, st);
    k<<<grid, 32 * kScanWarps, smem, st>>>(a);
    return cudaGetLastError();
}

// (state entries per lane NT, warps sharing a channel block SPLIT): padded
// state NT * SPLIT of 4 -> (2, 2), 8 -> (4, 2), 16 -> (8, 2) or (4, 4).
#define MAMBA_VARIANTS(X) X(2, 2) X(4, 2) X(8, 2) X(4, 4)

// The summary pass reads no z, so it has no HAS_Z instances.
template <typename T, bool STATE_ONLY, int NT, int S, int MODE>
cudaError_t dispatch_flags(bool sp, bool hz, const ScanArgs& a, int grid, int smem,
                           cudaStream_t st) {
    if constexpr (MODE == kModeCkpt && !STATE_ONLY) {   // no outputs: no gate
        return sp ? launch_scan<T, NT, S, false, true, false, MODE>(a, grid, smem, st)
                  : launch_scan<T, NT, S, false, false, false, MODE>(a, grid, smem, st);
    } else if constexpr (STATE_ONLY) {
        return sp ? launch_scan<T, NT, S, true, true, false, MODE>(a, grid, smem, st)
                  : launch_scan<T, NT, S, true, false, false, MODE>(a, grid, smem, st);
    } else {
        if (sp)
            return hz ? launch_scan<T, NT, S, false, true, true, MODE>(a, grid, smem, st)
                      : launch_scan<T, NT, S, false, true, false, MODE>(a, grid, smem, st);
        return hz ? launch_scan<T, NT, S, false, false, true, MODE>(a, grid, smem, st)
                  : launch_scan<T, NT, S, false, false, false, MODE>(a, grid, smem, st);
    }
}

template <typename T, bool STATE_ONLY, int NT, int S>
cudaError_t dispatch_mode(int mode, bool sp, bool hz, const ScanArgs& a, int grid, int smem,
                          cudaStream_t st) {
    if (mode == kModeExtZoh)
        return dispatch_flags<T, STATE_ONLY, NT, S, kModeExtZoh>(sp, hz, a, grid, smem, st);
    if (mode == kModeCkpt || mode == kModeTrain) {   // summary pass: the extended mode's
        if constexpr (STATE_ONLY)
            return dispatch_flags<T, STATE_ONLY, NT, S, kModeExt>(sp, hz, a, grid, smem, st);
        else if (mode == kModeCkpt)
            return dispatch_flags<T, STATE_ONLY, NT, S, kModeCkpt>(sp, hz, a, grid, smem, st);
        else
            return dispatch_flags<T, STATE_ONLY, NT, S, kModeTrain>(sp, hz, a, grid, smem, st);
    }
    if (mode == kModeExt)
        return dispatch_flags<T, STATE_ONLY, NT, S, kModeExt>(sp, hz, a, grid, smem, st);
    return dispatch_flags<T, STATE_ONLY, NT, S, kModePlain>(sp, hz, a, grid, smem, st);
}

template <typename T, bool STATE_ONLY>
cudaError_t dispatch_scan(int nt, int split, bool sp, bool hz, int mode, const ScanArgs& a,
                          int grid, int smem, cudaStream_t st) {
#define X(NT_, S_) \
    if (nt == NT_ && split == S_) return dispatch_mode<T, STATE_ONLY, NT_, S_>(mode, sp, hz, a, grid, smem, st);
    MAMBA_VARIANTS(X)
#undef X
    return cudaErrorInvalidValue;
}

struct Plan {
    bool concurrent;   // chunked tail on a side stream beside the whole-sequence units
    int nt, split, ch, np, stages, tt;
    int groups_per_batch, n_groups, n_full, nchunks;
    long long chunk_len;
    int smem;
};

template <typename T>
int smem_bytes_t(int nt, int split, int stages) {
    if (split == 4) return ScanLayout<T, 4, 4>::bytes(stages);
    if (nt == 2) return ScanLayout<T, 2, 2>::bytes(stages);
    if (nt == 4) return ScanLayout<T, 4, 2>::bytes(stages);
    return ScanLayout<T, 8, 2>::bytes(stages);
}
int smem_bytes(int dt, int nt, int split, int stages) {
    return dt == MAMBA_BF16 ? smem_bytes_t<__nv_bfloat16>(nt, split, stages)
                            : smem_bytes_t<float>(nt, split, stages);
}

int smem_per_sm(int dev) {
    static std::vector<int> cache;
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (!cache[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cache[dev] = v > 0 ? v : 228 * 1024;
    }
    return cache[dev];
}

// Work decomposition.  A unit is a tile of `ch` channels of one batch entry
// (one CTA, one warp per SM sub-partition) over a time range.  The kernel is
// bound by the ex2 and fp32 issue rates of each sub-partition, so the aim is
// an equal number of units per SM:
//   * whole waves of channel tiles (one per SM) scan the whole sequence;
//   * the tiles left over ("tail", fewer than one per SM) are cut into K
//     time chunks, K*tail <= #SM, whose passes run on a side stream beside
//     the whole waves, so that each SM takes at most one extra chunk;
//   * with fewer tiles than SMs, every tile is cut into K chunks that fill
//     the resident CTA slots of all SMs once; for very long sequences into
//     up to kChunkWaves times as many, as long as a chunk keeps at least
//     kMinWaveChunk steps.  One exact wave leaves the SMs that hold one unit
//     fewer idle at the end, but each chunk costs a summary and a carry
//     step.  Measured on B300: the 262144-step scan 3.15 ms with one wave,
//     2.97 ms with four; 16384-, 8192- and 2048-step scans 5-8% slower with
//     four waves than with one.
// A chunk that does not start at t = 0 gets its carried-in state from a
// summary pass (state only, about 3/4 of the work of a main pass) and a
// carry pass.  Tuning: tail = 1 keeps whole-sequence units only, tail = 2
// chunks the tail on the caller's stream, tail = 3 on the side stream;
// chunks > 0 cuts every tile into that many chunks.  side_ok is false for
// the no-allocation entry point, which uses the caller's stream only.
Plan make_plan(int dev, int dt, long long batch, long long dim, int N, long long L, bool tma,
               bool side_ok, const Tuning& tn) {
    Plan p;
    p.concurrent = false;
    const int sms = sm_count(dev);
    // Padded state 4, 8 or 16, split over two warps (each lane holds 2 or 4
    // entries; a CTA covers 64 channels) or, for dstate > 8, over four
    // warps (4 entries per lane, 32 channels per CTA).  Measured on B300 for
    // dstate 16, four slices of 4 beat two of 8 on both Mamba layer
    // workloads: twice the warps per SM sub-partition hide the latency of
    // the recurrence, and the two-way split reads about as much shared memory
    // per state update as the four-way one saves in instructions.  layout 1
    // forces the two-way split of 8 entries a lane.
    p.np = N <= 4 ? 4 : (N <= 8 ? 8 : 16);
    const bool split4 = N > 8 && tn.layout != 1;
    p.split = split4 ? 4 : 2;
    p.nt = p.np / p.split;
    p.ch = 32 * kScanWarps / p.split;
    p.tt = 64 / esize(dt);
    // at least two stages: the next tile is filled while this one finishes
    int stages = tma ? (tn.stages > 1 ? std::min(tn.stages, kMaxStages) : 2) : 2;
    int per_sm = smem_per_sm(dev) / (smem_bytes(dt, p.nt, p.split, stages) + 1024);
    per_sm = std::max(1, std::min(per_sm, kScanMinBlocks));
    p.stages = stages;
    p.smem = smem_bytes(dt, p.nt, p.split, stages);
    p.groups_per_batch = (int)((dim + p.ch - 1) / p.ch);
    p.n_groups = (int)(batch * p.groups_per_batch);
    const long long tiles = (L + p.tt - 1) / p.tt;
    const long long min_chunk_tiles = 4;
    const long long max_k = std::max<long long>(1, tiles / min_chunk_tiles);
    int n_chunked = 0, K = 1;
    if (tn.chunks > 0) {
        n_chunked = p.n_groups;
        K = tn.chunks;
    } else if (p.n_groups >= sms) {
        // The leftover tiles are cut into time chunks whose summary, carry
        // and main passes run on a side stream beside the whole-sequence
        // units (measured on B300: 278 -> 239 us for the Mamba-2.8B layer).
        // Run serially on one stream, the summary pass costs more than the
        // imbalance it removes, so without the side stream (the
        // no-allocation entry point) the tail scans whole sequences.
        const int tail = p.n_groups % sms;
        // automatic: chunk the tail only when it is at most a third of a
        // wave; a larger tail costs more in summary work than it saves
        const int mode = tn.tail != 0 ? tn.tail : (side_ok && 3 * tail <= sms ? 3 : 1);
        if (tail > 0 && (mode == 2 || mode == 3)) {
            n_chunked = tail;
            K = (int)std::max<long long>(2, std::min<long long>(sms / tail, max_k));
            p.concurrent = mode == 3 && side_ok;
        }
    } else if (tn.tail != 1) {
        constexpr long long kChunkWaves = 4, kMinWaveChunk = 4096;
        const long long one_wave = (long long)sms * per_sm / p.n_groups;
        const long long more = std::min<long long>(kChunkWaves * one_wave, L / kMinWaveChunk);
        const int k = (int)std::min<long long>(std::max(one_wave, more), max_k);
        if (k >= 2) {
            n_chunked = p.n_groups;
            K = k;
        }
    }
    if (n_chunked == 0 || K <= 1) {
        p.concurrent = false;
        p.n_full = p.n_groups;
        p.nchunks = 1;
        p.chunk_len = L;
    } else {
        const long long per = (tiles + K - 1) / K;
        p.chunk_len = per * p.tt;
        p.nchunks = (int)((L + p.chunk_len - 1) / p.chunk_len);
        p.n_full = p.nchunks > 1 ? p.n_groups - n_chunked : p.n_groups;
        p.concurrent = p.concurrent && p.n_full > 0 && p.nchunks > 1;
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

// 3-D map over a (d2, d1, d0) row-major tensor of `es`-byte elements, box
// {b0, b1, 1}, with the 32- or 64-byte swizzle (swizzle = 32 or 64) or none (0).
bool encode_map(CUtensorMap* m, const void* ptr, int es, bool is_bf16, long long d0,
                long long d1, long long d2, int b0, int b1, int swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)(d0 * es), (cuuint64_t)(d0 * d1 * es)};
    cuuint32_t box[3] = {(cuuint32_t)b0, (cuuint32_t)b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                           3, const_cast<void*>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                         : (swizzle == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                          : CU_TENSOR_MAP_SWIZZLE_NONE),
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// fixed scratch of the no-allocation entry point
// ---------------------------------------------------------------------------

// Scratch of mamba_scan_fwd_noalloc: a fixed array in the module's global
// memory, so that call never allocates.  Every GPU that loads the library
// holds it until the process exits.  In host code the name is only a
// stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress (noalloc_scratch below).
static __device__ __align__(256) unsigned char g_noalloc_scratch[MAMBA_NOALLOC_SCRATCH_BYTES];

// Device address of the fixed scratch for the calling thread's current
// device and context.  It is looked up on every call (a host-side lookup
// that allocates nothing), so it is never stale: not after cudaDeviceReset,
// nor when a caller switches contexts.
int noalloc_scratch(void** out) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return MAMBA_ERR_CUDA;
    }
    *out = ptr;
    return MAMBA_OK;
}

// Bytes of packed B/C rows per (batch entry, step): 2 * padded state * fp32.
long long packed_row_bytes(int64_t dstate) {
    return 2LL * padded_state(dstate) * (long long)sizeof(float);
}

}  // namespace mamba

using namespace mamba;

// Launch the generation-step kernel (vectorised dstate-16 or generic) with
// its (softplus, ZOH) instance.
#define MAMBA_STEP_LAUNCH(KERNEL)                                                        \
    if (sp) {                                                                            \
        if (zoh) KERNEL<T, true, true><<<grid, threads, 0, st>>>(a);                     \
        else KERNEL<T, true, false><<<grid, threads, 0, st>>>(a);                        \
    } else {                                                                             \
        if (zoh) KERNEL<T, false, true><<<grid, threads, 0, st>>>(a);                    \
        else KERNEL<T, false, false><<<grid, threads, 0, st>>>(a);                       \
    }
template <typename T>
void launch_step16(bool sp, bool zoh, dim3 grid, int threads, const StepArgs& a, cudaStream_t st) {
    MAMBA_STEP_LAUNCH(state_update16_kernel)
}
template <typename T>
void launch_step_generic(bool sp, bool zoh, dim3 grid, int threads, const StepArgs& a,
                         cudaStream_t st) {
    MAMBA_STEP_LAUNCH(state_update_kernel)
}
#undef MAMBA_STEP_LAUNCH

extern "C" {

int mamba_version(void) { return 300; }

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
        case MAMBA_ERR_TOO_BIG:
            return "the call needs more scratch than the fixed MAMBA_NOALLOC_SCRATCH_BYTES";
        case MAMBA_ERR_FLAGS: return "a flags argument has an unknown bit";
        case MAMBA_ERR_BOUNDS:
            return "a debug build's index check failed (the access was skipped)";
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
    }
    // the index checks of debug builds (always zero in release builds)
    const int dbg_scan = take_debug_word(), dbg_conv = conv_take_debug_word(),
              dbg_bwd = bwd_take_debug_word();
    if (dbg_scan < 0 || dbg_conv < 0 || dbg_bwd < 0) return MAMBA_ERR_CUDA;
    const int dbg = dbg_scan ? dbg_scan : (dbg_conv ? dbg_conv : dbg_bwd);
    if (dbg) g_debug_last_line.store(dbg & ~kDebugBoundsFlag);
    if (v) return MAMBA_ERR_TIMEOUT;
    if (dbg) return MAMBA_ERR_BOUNDS;
    return MAMBA_OK;
}

int mamba_debug_build(int* last_failed_line) {
    if (last_failed_line) *last_failed_line = g_debug_last_line.load();
#ifdef MAMBA_DEBUG
    return 1;
#else
    return 0;
#endif
}

int mamba_selftest_bounds(cudaStream_t stream) {
    bounds_selftest_kernel<<<1, 32, 0, stream>>>(1000);
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
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

int mamba_selftest_wait_timeout(int64_t limit_us, cudaStream_t stream) {
    if (limit_us < 1 || limit_us > 2000000) return MAMBA_ERR_SHAPE;
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>((unsigned long long)limit_us * 1000ull);
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

int mamba_scan_set_tuning(int tail, int stages, int chunks, int layout) {
    if (tail < 0 || tail > 3 || stages < 0 || stages > kMaxStages || chunks < 0 || layout < 0 ||
        layout > 2)
        return MAMBA_ERR_SHAPE;
    std::lock_guard<std::mutex> lk(g_mu);
    g_tuning.tail = tail;
    g_tuning.stages = stages;
    g_tuning.chunks = chunks;
    g_tuning.layout = layout;
    return MAMBA_OK;
}

// Shared body of mamba_scan_fwd (scratch from the stream-ordered pool),
// mamba_scan_fwd_noalloc (the fixed scratch array, no allocation) and
// mamba_scan_fwd_ex (either, plus initial state, lengths and ZOH).
static int scan_fwd_common(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                           int io_dtype, const void* u, const void* delta,
                           const float* dt_bias, const float* A, const void* B, const void* C,
                           const float* D_skip, const void* z, int softplus, bool zoh,
                           const float* h0, const int32_t* seqlens, void* y,
                           float* final_state, cudaStream_t stream, bool no_alloc,
                           float* ckpt = nullptr, int ck_tiles = 0) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (batch < 1 || dim < 1 || dstate < 1 || dstate > kMaxN || seqlen < 0) return MAMBA_ERR_SHAPE;
    if (batch > INT32_MAX / 2 || dim > (1ll << 40) || seqlen > (1ll << 40) ||
        (double)batch * dim * (double)(seqlen > 0 ? seqlen : 1) > 4.0e18)
        return MAMBA_ERR_SHAPE;
    if (!A || (seqlen > 0 && (!u || !delta || !B || !C || (!y && !ckpt)))) return MAMBA_ERR_NULL;
    const int es = esize(io_dtype);
    const size_t big = (size_t)(batch * dim * seqlen) * es;
    const size_t bcb = (size_t)(batch * dstate * seqlen) * es;
    const size_t fsb = (size_t)(batch * dim * dstate) * 4;
    for (const void* q : {u, delta, z, B, C, (const void*)y})
        if (q && !aligned(q, es)) return MAMBA_ERR_ALIGN;
    for (const void* q : {(const void*)dt_bias, (const void*)A, (const void*)D_skip,
                          (const void*)final_state, (const void*)h0, (const void*)seqlens})
        if (q && !aligned(q, 4)) return MAMBA_ERR_ALIGN;
    {
        const void* ins[] = {u, delta, z, B, C, dt_bias, A, D_skip, h0, seqlens};
        const size_t insz[] = {big, big, big, bcb, bcb, (size_t)dim * 4,
                               (size_t)(dim * dstate) * 4, (size_t)dim * 4, fsb,
                               (size_t)batch * 4};
        for (int i = 0; i < 10; ++i) {
            if (overlaps(y, big, ins[i], insz[i])) return MAMBA_ERR_ALIAS;
            if (overlaps(final_state, fsb, ins[i], insz[i])) return MAMBA_ERR_ALIAS;
        }
        if (overlaps(y, big, final_state, fsb)) return MAMBA_ERR_ALIAS;
        if (ckpt) {
            const size_t ckb = (size_t)(batch * dim) * ck_tiles * padded_state(dstate) * 4;
            for (int i = 0; i < 10; ++i)
                if (overlaps(ckpt, ckb, ins[i], insz[i])) return MAMBA_ERR_ALIAS;
            if (overlaps(ckpt, ckb, y, big) || overlaps(ckpt, ckb, final_state, fsb))
                return MAMBA_ERR_ALIAS;
        }
    }
    if (seqlen == 0) {
        if (final_state) {
            const cudaError_t r =
                h0 ? cudaMemcpyAsync(final_state, h0, fsb, cudaMemcpyDeviceToDevice, stream)
                   : cudaMemsetAsync(final_state, 0, fsb, stream);
            if (r != cudaSuccess) return MAMBA_ERR_CUDA;
        }
        return MAMBA_OK;
    }

    // the packed B/C rows alone must fit the fixed scratch (checked before
    // any CUDA call; the chunk summaries are checked once the plan is known)
    if (no_alloc && (double)batch * (double)seqlen * (double)packed_row_bytes(dstate) >
                        (double)MAMBA_NOALLOC_SCRATCH_BYTES)
        return MAMBA_ERR_TOO_BIG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MAMBA_ERR_CUDA;
    // tensor-map path: 16-byte aligned bases and rows, coordinates within int32
    bool tma = ((seqlen * es) % 16) == 0 && seqlen < (1ll << 31) && dim < (1ll << 31) &&
               (double)dim * seqlen * es < 1.0e12;
    for (const void* q : {u, delta, z, (const void*)y})
        if (q && !aligned(q, 16)) tma = false;

    // The tuning is read once for the whole call.  The tensor maps of u,
    // delta, z and y are encoded before anything is sized from the plan:
    // if one cannot be encoded, the call is planned again without tensor
    // maps, before any scratch is sized or allocated.
    const Tuning tn = get_tuning();
    Plan pl = make_plan(dev, io_dtype, batch, dim, (int)dstate, seqlen, tma, !no_alloc, tn);
    ScanArgs a;
    std::memset(&a, 0, sizeof(a));
    if (tma) {
        const bool bf = io_dtype == MAMBA_BF16;
        const int tt = pl.tt;
        const int sw = 64;   // the tile's row bytes: one 64-byte row per channel
        tma = encode_map(&a.m_u, u, es, bf, seqlen, dim, batch, tt, pl.ch, sw) &&
              encode_map(&a.m_dl, delta, es, bf, seqlen, dim, batch, tt, pl.ch, sw) &&
              (!z || encode_map(&a.m_z, z, es, bf, seqlen, dim, batch, tt, pl.ch, sw)) &&
              (!y || encode_map(&a.m_y, y, es, bf, seqlen, dim, batch, tt, pl.ch, sw));
        if (!tma) pl = make_plan(dev, io_dtype, batch, dim, (int)dstate, seqlen, false, !no_alloc, tn);
    }
    const bool chunked = pl.n_full < pl.n_groups && pl.nchunks > 1;
    const bool acc = io_dtype == MAMBA_F32;

    // scratch: packed B/C rows, then the chunk summaries
    const size_t bc_bytes = (size_t)batch * (size_t)seqlen * (size_t)pl.np * 2 * sizeof(float);
    const size_t tail_rows = (size_t)(pl.n_groups - pl.n_full) * pl.ch;
    const size_t entries = tail_rows * (size_t)dstate;
    const size_t ws_bytes = chunked ? 2 * entries * (size_t)(pl.nchunks - 1) * sizeof(float) : 0;
    void* scratch = nullptr;
    if (no_alloc) {
        if (bc_bytes + ws_bytes > (size_t)MAMBA_NOALLOC_SCRATCH_BYTES) return MAMBA_ERR_TOO_BIG;
        const int rc = noalloc_scratch(&scratch);
        if (rc != MAMBA_OK) return rc;
    } else {
        cudaMemPool_t pool = nullptr;
        const int rc = get_pool(dev, &pool);
        if (rc != MAMBA_OK) return rc;
        if (cudaMallocFromPoolAsync(&scratch, bc_bytes + ws_bytes, pool, stream) != cudaSuccess) {
            cudaGetLastError();
            return MAMBA_ERR_ALLOC;
        }
    }

    a.bc = static_cast<const float4*>(scratch);
    if (chunked) {
        a.ws_P = reinterpret_cast<float*>(static_cast<char*>(scratch) + bc_bytes);
        a.ws_h = a.ws_P + entries * (pl.nchunks - 1);
    }
    // the packed table's map needs the scratch address (16-byte aligned from
    // either source); the plan is fixed by now, so a failure is an error
    if (tma && !encode_map(&a.m_bc, scratch, 4, false, 2 * pl.np, seqlen, batch, 2 * pl.np,
                           pl.tt, 0)) {
        if (!no_alloc) cudaFreeAsync(scratch, stream);
        return MAMBA_ERR_CUDA;
    }
    a.u = u; a.delta = delta; a.z = z;
    a.dt_bias = dt_bias; a.A = A; a.D_skip = D_skip; a.y = y; a.final_state = final_state;
    a.h0 = h0; a.seqlens = seqlens;
    a.ckpt = ckpt; a.ck_tiles = ck_tiles;
    a.dim = dim; a.seqlen = seqlen; a.chunk_len = pl.chunk_len;
    a.batch = (int)batch; a.dstate = (int)dstate;
    a.use_tma = tma ? 1 : 0; a.stages = pl.stages;
    a.ch = pl.ch;
    a.groups_per_batch = pl.groups_per_batch; a.n_groups = pl.n_groups;
    a.n_full = pl.n_full; a.nchunks = pl.nchunks;
    a.tail_rows = (int)tail_rows;

    cudaError_t e;
    e = launch_pack_bc(io_dtype, B, C, static_cast<float4*>(scratch), batch, seqlen,
                       (int)dstate, pl.np, acc ? 1.0f : kLn2, stream);
    const bool bf = io_dtype == MAMBA_BF16;
    const bool hz = z != nullptr;
    const int mode = ckpt ? (y ? kModeTrain : kModeCkpt)
                          : (zoh ? kModeExtZoh : ((h0 || seqlens) ? kModeExt : kModePlain));
    auto summary_and_carry = [&](cudaStream_t st) -> cudaError_t {
        const int grid1 = (pl.n_groups - pl.n_full) * (pl.nchunks - 1);
        cudaError_t r =
            bf ? dispatch_scan<__nv_bfloat16, true>(pl.nt, pl.split, softplus, false, mode, a,
                                                    grid1, pl.smem, st)
               : dispatch_scan<float, true>(pl.nt, pl.split, softplus, false, mode, a, grid1,
                                            pl.smem, st);
        if (r != cudaSuccess) return r;
        const long long n_ent = (long long)entries;
        {
            ProfScope prof(kKindCarry, st);
            carry_kernel<<<(unsigned)((n_ent + 255) / 256), 256, 0, st>>>(a.ws_P, a.ws_h, n_ent,
                                                                          pl.nchunks);
        }
        return cudaGetLastError();
    };
    auto main_pass = [&](int first, int count, cudaStream_t st) -> cudaError_t {
        ScanArgs m = a;
        m.unit_offset = first;
        return bf ? dispatch_scan<__nv_bfloat16, false>(pl.nt, pl.split, softplus, hz, mode, m,
                                                        count, pl.smem, st)
                  : dispatch_scan<float, false>(pl.nt, pl.split, softplus, hz, mode, m, count,
                                                pl.smem, st);
    };
    const int n_chunk_units = chunked ? (pl.n_groups - pl.n_full) * pl.nchunks : 0;
    if (e == cudaSuccess && pl.concurrent && chunked && !no_alloc) {
        // whole-sequence units on the caller's stream; the chunked tail
        // (summary, carry, its main pass) on the side stream beside them
        Side sd;
        int rc2 = get_side(dev, &sd);
        if (rc2 != MAMBA_OK) {
            cudaFreeAsync(scratch, stream);
            return rc2;
        }
        std::lock_guard<std::mutex> lk(g_side_mu);
        if (cudaEventRecord(sd.fork, stream) != cudaSuccess ||
            cudaStreamWaitEvent(sd.stream, sd.fork, 0) != cudaSuccess)
            e = cudaErrorUnknown;
        if (e == cudaSuccess) e = main_pass(0, pl.n_full, stream);
        if (e == cudaSuccess) e = summary_and_carry(sd.stream);
        if (e == cudaSuccess) e = main_pass(pl.n_full, n_chunk_units, sd.stream);
        if (cudaEventRecord(sd.join, sd.stream) != cudaSuccess ||
            cudaStreamWaitEvent(stream, sd.join, 0) != cudaSuccess)
            e = cudaErrorUnknown;
    } else {
        if (e == cudaSuccess && chunked) e = summary_and_carry(stream);
        if (e == cudaSuccess) e = main_pass(0, pl.n_full + n_chunk_units, stream);
    }
    if (!no_alloc) cudaFreeAsync(scratch, stream);
    return e == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

int mamba_scan_fwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, mamba_dtype_t io_dtype,
                   const void* u, const void* delta, const float* dt_bias, const float* A,
                   const void* B, const void* C, const float* D_skip, const void* z,
                   int softplus, void* y, float* final_state, cudaStream_t stream) {
    return scan_fwd_common(batch, dim, dstate, seqlen, io_dtype, u, delta, dt_bias, A, B, C,
                           D_skip, z, softplus, false, nullptr, nullptr, y, final_state, stream,
                           false);
}

int mamba_scan_fwd_noalloc(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                           mamba_dtype_t io_dtype, const void* u, const void* delta,
                           const float* dt_bias, const float* A, const void* B, const void* C,
                           const float* D_skip, const void* z, int softplus, void* y,
                           float* final_state, cudaStream_t stream) {
    return scan_fwd_common(batch, dim, dstate, seqlen, io_dtype, u, delta, dt_bias, A, B, C,
                           D_skip, z, softplus, false, nullptr, nullptr, y, final_state, stream,
                           true);
}

int64_t mamba_scan_checkpoint_bytes(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen) {
    if (batch < 1 || dim < 1 || dstate < 1 || dstate > kMaxN || seqlen < 0) return -1;
    if ((double)batch * dim * (double)checkpoint_tiles(seqlen) * padded_state(dstate) * 4.0 > 4.0e18)
        return -1;
    return batch * dim * checkpoint_tiles(seqlen) * padded_state(dstate) * (int64_t)sizeof(float);
}

int mamba_scan_fwd_train(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                         mamba_dtype_t io_dtype, const void* u, const void* delta,
                         const float* dt_bias, const float* A, const void* B, const void* C,
                         const float* D_skip, const void* z, int flags,
                         const float* initial_state, void* y, float* final_state,
                         float* checkpoints, cudaStream_t stream) {
    if (flags & ~MAMBA_FLAG_SOFTPLUS) return MAMBA_ERR_FLAGS;
    if (seqlen > 0 && (!y || !checkpoints)) return MAMBA_ERR_NULL;
    if (checkpoints && !aligned(checkpoints, 16)) return MAMBA_ERR_ALIGN;
    if (seqlen < 0 || checkpoint_tiles(seqlen) > INT32_MAX) return MAMBA_ERR_SHAPE;
    return scan_fwd_common(batch, dim, dstate, seqlen, io_dtype, u, delta, dt_bias, A, B, C,
                           D_skip, z, (flags & MAMBA_FLAG_SOFTPLUS) ? 1 : 0, false, initial_state,
                           nullptr, y, final_state, stream, false, seqlen > 0 ? checkpoints : nullptr,
                           (int)checkpoint_tiles(seqlen));
}

int mamba_scan_fwd_ex(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, mamba_dtype_t io_dtype,
                      const void* u, const void* delta, const float* dt_bias, const float* A,
                      const void* B, const void* C, const float* D_skip, const void* z,
                      int flags, const float* initial_state, const int32_t* seqlens, void* y,
                      float* final_state, cudaStream_t stream) {
    if (flags & ~(MAMBA_FLAG_SOFTPLUS | MAMBA_FLAG_ZOH | MAMBA_FLAG_NOALLOC))
        return MAMBA_ERR_FLAGS;
    return scan_fwd_common(batch, dim, dstate, seqlen, io_dtype, u, delta, dt_bias, A, B, C,
                           D_skip, z, (flags & MAMBA_FLAG_SOFTPLUS) ? 1 : 0,
                           (flags & MAMBA_FLAG_ZOH) != 0, initial_state, seqlens, y,
                           final_state, stream, (flags & MAMBA_FLAG_NOALLOC) != 0);
}


static int state_update_common(int64_t batch, int64_t dim, int64_t dstate, int io_dtype,
                               float* state, const void* x, const void* delta,
                               const float* dt_bias, const float* A, const void* B,
                               const void* C, const float* D_skip, const void* z, int flags,
                               void* y, cudaStream_t stream) {
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
    const bool sp = (flags & MAMBA_FLAG_SOFTPLUS) != 0, zoh = (flags & MAMBA_FLAG_ZOH) != 0;
    // dstate 16 with 16-byte aligned rows: the vectorised two-lane kernel
    const bool vec16 = dstate == 16 && aligned(state, 16) && aligned(A, 16) && aligned(B, 16) &&
                       aligned(C, 16) && batch <= 65535LL * kStepBatches * kStepRows;
    if (vec16) {
        const dim3 grid((unsigned)((dim + kStepDims - 1) / kStepDims),
                        (unsigned)((batch + kStepBatches * kStepRows - 1) / (kStepBatches * kStepRows)));
        ProfScope prof(kKindStep, stream);
        if (io_dtype == MAMBA_BF16)
            launch_step16<__nv_bfloat16>(sp, zoh, grid, 2 * kStepDims * kStepBatches, a, stream);
        else
            launch_step16<float>(sp, zoh, grid, 2 * kStepDims * kStepBatches, a, stream);
        return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
    }
    const long long threads = rows * 4;
    const unsigned grid = (unsigned)((threads + kThreads - 1) / kThreads);
    {
        ProfScope prof(kKindStep, stream);
        if (io_dtype == MAMBA_BF16)
            launch_step_generic<__nv_bfloat16>(sp, zoh, dim3(grid), kThreads, a, stream);
        else
            launch_step_generic<float>(sp, zoh, dim3(grid), kThreads, a, stream);
    }
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

int mamba_state_update(int64_t batch, int64_t dim, int64_t dstate, mamba_dtype_t io_dtype, float* state,
                       const void* x, const void* delta, const float* dt_bias, const float* A,
                       const void* B, const void* C, const float* D_skip, const void* z, void* y,
                       cudaStream_t stream) {
    return state_update_common(batch, dim, dstate, io_dtype, state, x, delta, dt_bias, A, B, C,
                               D_skip, z, MAMBA_FLAG_SOFTPLUS, y, stream);
}

int mamba_state_update_ex(int64_t batch, int64_t dim, int64_t dstate, mamba_dtype_t io_dtype,
                          float* state, const void* x, const void* delta, const float* dt_bias,
                          const float* A, const void* B, const void* C, const float* D_skip,
                          const void* z, int flags, void* y, cudaStream_t stream) {
    if (flags & ~(MAMBA_FLAG_SOFTPLUS | MAMBA_FLAG_ZOH)) return MAMBA_ERR_FLAGS;
    return state_update_common(batch, dim, dstate, io_dtype, state, x, delta, dt_bias, A, B, C,
                               D_skip, z, flags, y, stream);
}

}  // extern "C"

namespace mamba {
int scan_checkpoints(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int io_dtype,
                     const void* u, const void* delta, const float* dt_bias, const float* A,
                     const void* B, const void* C, int softplus, const float* initial_state,
                     float* ckpt, int ck_tiles, cudaStream_t stream) {
    if (!ckpt || ck_tiles != (int)checkpoint_tiles(seqlen)) return MAMBA_ERR_SHAPE;
    return scan_fwd_common(batch, dim, dstate, seqlen, io_dtype, u, delta, dt_bias, A, B, C,
                           nullptr, nullptr, softplus, false, initial_state, nullptr, nullptr,
                           nullptr, stream, false, ckpt, ck_tiles);
}
}  // namespace mamba
