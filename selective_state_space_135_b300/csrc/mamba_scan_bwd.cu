// Backward pass of the selective scan (Euler input term) for B300 (sm_103a).
//
// The fused forward keeps the expanded state on chip and the backward pass
// recomputes it instead of reading it back (page "Mamba: linear-time
// sequence modeling with selective state spaces", "What they did").  Here:
//
//   1. checkpoint pass: the forward scan kernel in its checkpoint mode (no
//      outputs) runs the recurrence and stores the state before every tile
//      of kBwdTile steps (B x D x ceil(L / kBwdTile) x N fp32);
//   2. reverse pass: one two-warp CTA per 32 channels, each warp holding half
//      of the entries.  Per tile, last to first, the tile's inputs are staged
//      in shared memory, each warp recomputes its entries' states from the
//      checkpoint into shared memory, then walks the tile backwards carrying
//      dh = dJ/dh (the warps add their partial sums over entries -- C.h, du,
//      dDelta -- through shared memory):
//        g_t   = dy_t * silu(z_t)             dz_t = dy_t * pre_t * silu'(z_t)
//        dh   += g_t C_t                       dC_t += g_t h_t,  dB_t += dh Delta_t u_t
//        du_t  = g_t D + sum_n dh Delta_t B_t  dDelta_t = sum_n dh (A Abar h_{t-1} + B_t u_t)
//        dA   += dh Delta_t Abar h_{t-1}       dh   *= Abar_t
//      with ddelta = dDelta * sigmoid(s) under softplus.  B and C are shared
//      by all channels of a batch entry, so dB and dC are sums over d: the
//      warp sums its 32 channels with a transposing butterfly of shuffles
//      (one shuffle per value), parks the sums of step t in its own pairs of
//      the tile's B/C row t once read, and the CTA writes the tile's rows of
//      partials (one per 32 channels) as whole 16-byte stores;
//   3. reduction passes add the partials in a fixed order (deterministic
//      results, no atomics): dB, dC over channel groups, dA, D_skip and
//      dt_bias gradients over the batch (and the time chunks).
//
// With few units of 32 channels the reverse pass runs in time chunks, each
// chunk a CTA of its own, after a summary and a carry pass that give every
// chunk the gradient entering it from the later ones (see
// bwd_summary_kernel).

#include "scan_common.cuh"

#include <algorithm>
#include <cstring>

namespace mamba {
namespace {

// kBwdTile (scan_common.cuh, 12) steps between checkpoints = the reverse tile
// (42 KB of shared memory per two-warp CTA at dstate 16: five per SM)
constexpr int kReduceThreads = 256;

struct BwdArgs {
    const void* u;
    const void* delta;
    const void* z;
    const void* dy;
    const float4* bc;   // packed rows (B pair, C pair), natural units: [batch][L][NP / 2]
    const float* dt_bias;
    const float* A;
    const float* D_skip;
    const float* h0;      // initial state or null
    const float* dfinal;  // dJ / d final state or null
    float* ckpt;          // [batch][ntiles][NP / 4][dim][4]: state before each tile
    void* du;
    void* ddelta;
    void* dz;
    float* pB;            // [group][batch][L][NP]: dB summed over the group's 32 channels
    float* pC;
    float* pA;            // [chunk][row][NP]
    float* pD;            // [chunk][row]
    float* pbias;         // [chunk][row]
    float* dh0;           // [row][N] or null
    // time chunks of the reverse pass (nchunks = 1: whole sequences)
    float* dloc;          // [chunk][row][NP]: dJ/dh entering the chunk from its own steps
    float* sdt;           // [chunk][row]: sum of Delta over the chunk
    float* dcarry;        // [chunk][row][NP]: dJ/dh at the chunk's end, or null (nchunks = 1)
    long long dim, L;
    int batch, N, groups, ntiles;
    int nchunks, chunk_tiles;   // tiles [c * chunk_tiles, (c + 1) * chunk_tiles) per chunk
    int vec8;   // every (batch, d) row of u, delta, z, dy, du, ddelta, dz is 8-byte aligned
};

// One lane's kBwdTile consecutive elements of its row, starting at a tile
// boundary: 8-byte accesses for a full tile of an aligned row (the tile
// start is 8-byte aligned: kBwdTile elements are 24 or 48 bytes), scalar
// accesses otherwise.
// (row_at, ext: the row's element offset in its tensor and the tensor's
// extent, for the index checks of debug builds)
template <typename T>
__device__ __forceinline__ void load_tile_row(const T* row, long long t0, int nv, bool vec,
                                              bool on, float (&v)[kBwdTile], long long row_at,
                                              long long ext) {
    (void)row_at;
    (void)ext;
    if (on && vec && nv == kBwdTile &&
        (!MAMBA_IN(row_at + t0, ext) || !MAMBA_IN(row_at + t0 + kBwdTile - 1, ext))) {
#pragma unroll
        for (int i = 0; i < kBwdTile; ++i) v[i] = 0.0f;
    } else if (on && vec && nv == kBwdTile) {
        const uint2* p = reinterpret_cast<const uint2*>(row + t0);
        constexpr int kPer = 8 / (int)sizeof(T);
#pragma unroll
        for (int k = 0; k < kBwdTile / kPer; ++k) {
            const uint2 r = p[k];
            if constexpr (sizeof(T) == 2) {
                v[4 * k] = __uint_as_float(r.x << 16);
                v[4 * k + 1] = __uint_as_float(r.x & 0xffff0000u);
                v[4 * k + 2] = __uint_as_float(r.y << 16);
                v[4 * k + 3] = __uint_as_float(r.y & 0xffff0000u);
            } else {
                v[2 * k] = __uint_as_float(r.x);
                v[2 * k + 1] = __uint_as_float(r.y);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < kBwdTile; ++i)
            v[i] = (on && i < nv && MAMBA_IN(row_at + t0 + i, ext)) ? IO<T>::to_f(row[t0 + i]) : 0.0f;
    }
}
template <typename T>
__device__ __forceinline__ void store_tile_row(T* row, long long t0, int nv, bool vec,
                                               const float (&v)[kBwdTile], long long row_at,
                                               long long ext) {
    (void)row_at;
    (void)ext;
    if (vec && nv == kBwdTile &&
        (!MAMBA_IN(row_at + t0, ext) || !MAMBA_IN(row_at + t0 + kBwdTile - 1, ext))) {
        return;
    } else if (vec && nv == kBwdTile) {
        uint2* p = reinterpret_cast<uint2*>(row + t0);
        constexpr int kPer = 8 / (int)sizeof(T);
#pragma unroll
        for (int k = 0; k < kBwdTile / kPer; ++k) {
            uint2 r;
            if constexpr (sizeof(T) == 2) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(v[4 * k], v[4 * k + 1]);
                __nv_bfloat162 hi = __floats2bfloat162_rn(v[4 * k + 2], v[4 * k + 3]);
                r.x = *reinterpret_cast<uint32_t*>(&lo);
                r.y = *reinterpret_cast<uint32_t*>(&hi);
            } else {
                r.x = __float_as_uint(v[2 * k]);
                r.y = __float_as_uint(v[2 * k + 1]);
            }
            p[k] = r;
        }
    } else {
#pragma unroll
        for (int i = 0; i < kBwdTile; ++i)
            if (i < nv && MAMBA_IN(row_at + t0 + i, ext)) row[t0 + i] = IO<T>::from_f(v[i]);
    }
}

// Delta (natural units) and, with softplus, its derivative sigmoid(s).
template <bool ACC, bool SP>
__device__ __forceinline__ float delta_nat(float s) {
    if constexpr (!SP) return s;
    else return softplus_f<ACC>(s);
}
template <bool ACC>
__device__ __forceinline__ float sigmoid_f(float s) {
    if constexpr (ACC) return 1.0f / (1.0f + expf(-s));
    else return __fdividef(1.0f, 1.0f + ex2_approx(-s * kLog2e));
}
// Abar = exp(Delta * A) of a pair of entries.  dtl2 holds Delta / ln 2 (as
// Delta * log2(e)) in both halves, formed once per step, so the fast path
// needs one packed multiply and two ex2 per pair.
template <bool ACC>
__device__ __forceinline__ float2 abar2_of(float dt, const float2& dtl2, const float2& a) {
    if constexpr (ACC) return make_float2(expf(dt * a.x), expf(dt * a.y));
    const float2 arg = __fmul2_rn(dtl2, a);
    return make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
}

// Warp unit of both passes: 32 consecutive channels of one batch entry.
struct WarpUnit {
    int b, grp, lane;
    long long d, row;
    bool ok;
};
__device__ __forceinline__ WarpUnit warp_unit(const BwdArgs& a, long long w) {
    WarpUnit u;
    u.lane = threadIdx.x & 31;
    u.b = (int)(w / a.groups);
    u.grp = (int)(w % a.groups);
    u.d = (long long)u.grp * 32 + u.lane;
    u.ok = u.d < a.dim;
    u.row = (long long)u.b * a.dim + (u.ok ? u.d : 0);
    return u;
}

// The state entries of a unit are split over bwd_split<NP>() warps in the
// reverse pass (their recurrences are independent); warp w of a unit holds
// entries [w * NPW, (w + 1) * NPW).  (Four warps of four entries at dstate
// 16 measured slower on B300: the per-step work outside the entries' own
// arithmetic is paid per warp, and the larger CTAs fit fewer to an SM.)
template <int NP>
__host__ __device__ constexpr int bwd_split() {
    return 2;
}

// Sum v over the 32 lanes of the warp, NV values at once.  At each of the
// first log2(NV) levels a lane keeps half of its values and sends the other
// half to its partner (lane ^ m), so every value costs one shuffle in all;
// then the last partial sums are added over the remaining lanes.  On return
// every lane holds the full sum of the entry bwd_lane_entry<NV>(lane).
//
// So that a lane need not choose, level by level, which half it keeps, its
// entries sit in its registers in a lane-dependent order: slot s of lane l
// holds entry s ^ bwd_slot_xor<NV>(l), the entry bits of every level but the
// last.  At each of those levels the kept half is then slots [0, half) on
// every lane; only the last level (entries 2k and 2k + 1, which stay
// together as a packed pair) selects.
template <int NV>
__host__ __device__ constexpr int bwd_levels() {
    return NV == 16 ? 4 : (NV == 8 ? 3 : (NV == 4 ? 2 : 1));
}
template <int NV>
__device__ __forceinline__ int bwd_lane_entry(int lane) {
    constexpr int LV = bwd_levels<NV>();
    int n = 0;
#pragma unroll
    for (int lev = 0; lev < LV; ++lev) n += ((lane >> (4 - lev)) & 1) * (NV >> (lev + 1));
    return n;
}
template <int NV>
__device__ __forceinline__ int bwd_slot_xor(int lane) {
    return bwd_lane_entry<NV>(lane) & ~1;
}
template <int NV>
__device__ __forceinline__ float warp_sum_lanes(float (&v)[NV]) {
    constexpr int LV = bwd_levels<NV>();
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int lev = 0; lev < LV - 1; ++lev) {
        const int m = 16 >> lev;
        const int half = NV >> (lev + 1);
#pragma unroll
        for (int i = 0; i < NV / 2; ++i)
            if (i < half) v[i] += __shfl_xor_sync(0xffffffffu, v[i + half], m);
    }
    // last level: slots 0 and 1 hold entries e and e + 1 (e even)
    const int m = 16 >> (LV - 1);
    const bool upper = (lane & m) != 0;
    float s = (upper ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, upper ? v[0] : v[1], m);
#pragma unroll
    for (int mm = m >> 1; mm >= 1; mm >>= 1) s += __shfl_xor_sync(0xffffffffu, s, mm);
    return s;
}

// Shared memory of one CTA (bwd_split<NP>() warps, one unit), per tile:
//   hist  [warp][kBwdTile][NPW / 2][32] float2  the warp's states h_t (after
//                                     step t), in the lane's register order
//   srow  [kBwdTile][2][32] float2    per step and lane: (u, Delta) and
//                                     (g = dy silu(z), sigmoid(s))
//   szf   [kBwdTile][32]              per step and lane: dy silu'(z)
//   party [warp][kBwdTile][32]        the warp's partial sum of C.h
//   partd [warp][kBwdTile][32] float2 the warp's partial sums of du, dDelta
//   sbc   [kBwdTile][NP / 2] float4   the tile's packed B/C rows; in the
//                                     reverse walk each warp overwrites its
//                                     own pairs of row t, once read, with
//                                     the step's dB and dC sums (same layout)
template <int NP>
__host__ __device__ constexpr int bwd_smem_floats() {
    return kBwdTile * NP * 32 + 5 * kBwdTile * 32 + bwd_split<NP>() * 3 * kBwdTile * 32 +
           kBwdTile * (NP / 2) * 4;
}

// Registers are allocated per warp on one SM sub-partition (16384 each):
// at most 168 per thread leave room for three warps per sub-partition, so
// five of these two-warp CTAs (the shared-memory limit) fit on an SM; at 190
// only four did, and 640 CTAs took two waves on 148 SMs.  Asking for six
// CTAs per SM caps ptxas at 168.
template <typename T, int NP, bool SP, bool HZ>
__global__ void __launch_bounds__(32 * bwd_split<NP>(), 6)
bwd_kernel(const BwdArgs a) {
    constexpr bool ACC = IO<T>::kAccurate;
    constexpr int SPL = bwd_split<NP>();
    constexpr int NPW = NP / SPL;
    constexpr int NPP = NPW / 2;
    extern __shared__ __align__(16) float bwd_smem[];
    const int warp = threadIdx.x >> 5;
    float2* hist2 = reinterpret_cast<float2*>(bwd_smem + warp * (kBwdTile * NPW * 32));
    float2* srow = reinterpret_cast<float2*>(bwd_smem + kBwdTile * NP * 32);
    float* szf = reinterpret_cast<float*>(srow + kBwdTile * 2 * 32);
    float* party = szf + kBwdTile * 32;
    float2* partd = reinterpret_cast<float2*>(party + SPL * kBwdTile * 32);
    float4* sbc = reinterpret_cast<float4*>(partd + SPL * kBwdTile * 32);
    const WarpUnit q = warp_unit(a, blockIdx.x);
    const int cidx = blockIdx.y;   // time chunk (0 with whole sequences)
    const int k_lo = cidx * a.chunk_tiles;
    const int k_hi = min(a.ntiles, k_lo + a.chunk_tiles) - 1;
    const int lane = q.lane, N = a.N, n0 = warp * NPW;
    const long long L = a.L;
    // extents for the index checks of debug builds
    const long long rows = (long long)a.batch * a.dim;   // (b, d) rows
    const long long big = rows * L;                      // u, delta, z, dy and their gradients
    const long long pext = (long long)a.groups * a.batch * L * NP;
    const long long ckext = (long long)a.batch * a.ntiles * NP * a.dim;
    (void)rows;
    (void)big;
    (void)pext;
    (void)ckext;

    // this warp's entries in pairs: A, dJ/dh, the dA partial sums, and the
    // state at the start of the current tile (from its checkpoint).  Register
    // pair j of this lane holds the entry pair j ^ pj (see warp_sum_lanes).
    const int pj = bwd_slot_xor<NPW>(lane) >> 1;
    float2 A2[NPP], dh2[NPP], dA2[NPP], hs2[NPP];
#pragma unroll
    for (int j = 0; j < NPP; ++j) {
        float av[2], dv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = n0 + 2 * (j ^ pj) + e;
            const bool on = q.ok && n < N;
            av[e] = on ? MAMBA_LD(a.A, q.d * N + n, a.dim * N) : 0.0f;
            if (a.dcarry)   // the gradient entering this chunk from the later ones
                dv[e] = on ? MAMBA_LD(a.dcarry, ((long long)cidx * rows + q.row) * NP + n,
                                      (long long)a.nchunks * rows * NP)
                           : 0.0f;
            else
                dv[e] = (on && a.dfinal) ? MAMBA_LD(a.dfinal, q.row * N + n, rows * N) : 0.0f;
        }
        A2[j] = make_float2(av[0], av[1]);
        dh2[j] = make_float2(dv[0], dv[1]);
        dA2[j] = make_float2(0.0f, 0.0f);
    }
    const float bias = (q.ok && a.dt_bias) ? MAMBA_LD(a.dt_bias, q.d, a.dim) : 0.0f;
    const float dsk = (q.ok && a.D_skip) ? MAMBA_LD(a.D_skip, q.d, a.dim) : 0.0f;
    float dD = 0.0f, dbias = 0.0f;
    const T* ur = static_cast<const T*>(a.u) + q.row * L;
    const T* dl = static_cast<const T*>(a.delta) + q.row * L;
    const T* zr = HZ ? static_cast<const T*>(a.z) + q.row * L : nullptr;
    const T* dyr = static_cast<const T*>(a.dy) + q.row * L;
    T* dur = static_cast<T*>(a.du) + q.row * L;
    T* ddr = static_cast<T*>(a.ddelta) + q.row * L;
    T* dzr = HZ ? static_cast<T*>(a.dz) + q.row * L : nullptr;
    // checkpoints (quad-major: entry n of tile kk at ((kk * NP / 4 + n / 4) *
    // dim + d) * 4 + n % 4 from the batch entry's base): this lane's register
    // pair j (entries n = n0 + 2 (j ^ pj) and n + 1) of tile kk is at
    // ck + kk * NP * dim + (n / 4) * dim * 4 + n % 4
    const float* ck = a.ckpt + (long long)q.b * a.ntiles * NP * a.dim + q.d * 4;
    // after the butterfly this lane holds the sums of entry n0 + le; the first
    // lane of each group that shares an entry stores them into the B/C row
    const int le = bwd_lane_entry<NPW>(lane);
    const bool writer = (lane & ((16 >> bwd_levels<NPW>()) * 2 - 1)) == 0;
    float* sum_at = reinterpret_cast<float*>(sbc + n0 / 2 + (le >> 1)) + (le & 1);
    float* pBg = a.pB + ((long long)q.grp * a.batch + q.b) * L * NP;
    float* pCg = a.pC + ((long long)q.grp * a.batch + q.b) * L * NP;
    const bool vec = a.vec8 != 0;

    // Tile k - 1's global loads are issued before tile k's work: per warp two
    // input rows (warp 0: u, delta; warp 1: dy, z), each thread's share of
    // the B/C rows, and the warp's checkpoint, held in registers.
    constexpr int kRowsPerThread = (kBwdTile * (NP / 2) + 32 * SPL - 1) / (32 * SPL);
    float r1[kBwdTile], r2[kBwdTile];
    float4 bcr[kRowsPerThread];
    float2 ckr[NPP];
    auto fetch = [&](int kk) {
        const long long t0 = (long long)kk * kBwdTile;
        const int nv = (int)min((long long)kBwdTile, L - t0);
        if (warp == 0) {
            load_tile_row<T>(ur, t0, nv, vec, q.ok, r1, q.row * L, big);
            load_tile_row<T>(dl, t0, nv, vec, q.ok, r2, q.row * L, big);
        } else if (warp == 1) {
            load_tile_row<T>(dyr, t0, nv, vec, q.ok, r1, q.row * L, big);
            if constexpr (HZ) load_tile_row<T>(zr, t0, nv, vec, q.ok, r2, q.row * L, big);
        }
#pragma unroll
        for (int r = 0; r < kRowsPerThread; ++r) {
            const int e = r * 32 * SPL + threadIdx.x;
            const int i = e / (NP / 2);
            bcr[r] = (e < kBwdTile * (NP / 2) && i < nv)
                         ? MAMBA_LD(a.bc, (q.b * L + t0 + i) * (NP / 2) + (e % (NP / 2)),
                                    (long long)a.batch * L * (NP / 2))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < NPP; ++j) {
            const int n = n0 + 2 * (j ^ pj);
            const long long at = ((long long)kk * NP + (n & ~3)) * a.dim + (n & 3);
            const long long at_all = (long long)q.b * a.ntiles * NP * a.dim + q.d * 4 + at;
            (void)at_all;
            ckr[j] = (q.ok && MAMBA_IN(at_all, ckext) && MAMBA_IN(at_all + 1, ckext))
                         ? *reinterpret_cast<const float2*>(ck + at)
                         : make_float2(0.f, 0.f);
        }
    };
    if (k_hi >= k_lo) fetch(k_hi);

    for (int k = k_hi; k >= k_lo; --k) {
        const long long t0 = (long long)k * kBwdTile;
        const int nv = (int)min((long long)kBwdTile, L - t0);
        // (a) the tile's per-step inputs, B/C rows and checkpoint from the
        //     registers into shared memory, then the next loads.  Steps
        //     i >= nv of a last, short tile get u = 0, Delta = 0 and zero
        //     B/C rows: they leave the state as it is.
        if (warp == 0) {
#pragma unroll
            for (int i = 0; i < kBwdTile; ++i) {
                const float sarg = r2[i] + bias;
                srow[(2 * i) * 32 + lane] =
                    make_float2(r1[i], (q.ok && i < nv) ? delta_nat<ACC, SP>(sarg) : 0.0f);
                reinterpret_cast<float*>(srow + (2 * i + 1) * 32 + lane)[1] =
                    SP ? sigmoid_f<ACC>(sarg) : 1.0f;
            }
        } else if (warp == 1) {
#pragma unroll
            for (int i = 0; i < kBwdTile; ++i) {
                float* sr = reinterpret_cast<float*>(srow + (2 * i + 1) * 32 + lane);
                if constexpr (HZ) {   // the gate's factors do not depend on the state
                    const float zv = r2[i], sz = sigmoid_f<ACC>(zv);
                    sr[0] = r1[i] * zv * sz;
                    szf[i * 32 + lane] = r1[i] * sz * fmaf(zv, 1.0f - sz, 1.0f);
                } else {
                    sr[0] = r1[i];
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRowsPerThread; ++r) {
            const int e = r * 32 * SPL + threadIdx.x;
            if (e < kBwdTile * (NP / 2)) sbc[e] = bcr[r];
        }
#pragma unroll
        for (int j = 0; j < NPP; ++j) hs2[j] = ckr[j];
        if (k > k_lo) fetch(k - 1);
        __syncthreads();
        // (b) recompute this warp's states and its part of C.h (+ D u), two
        //     entries at a time with packed arithmetic
        {
            float2 h2[NPP];
#pragma unroll
            for (int j = 0; j < NPP; ++j) h2[j] = hs2[j];
#pragma unroll
            for (int i = 0; i < kBwdTile; ++i) {
                const float2 ud = srow[(2 * i) * 32 + lane];
                const float uv = ud.x, dt = ud.y;
                const float2 dtl2 = make_float2(dt * kLog2e, dt * kLog2e);
                const float2 du2 = make_float2(dt * uv, dt * uv);
                const float4* brow = sbc + i * (NP / 2) + n0 / 2;
                float2 acc2 = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < NPP; ++j) {
                    const float4 p = brow[j ^ pj];
                    const float2 ab = abar2_of<ACC>(dt, dtl2, A2[j]);
                    h2[j] = __ffma2_rn(ab, h2[j], __fmul2_rn(du2, make_float2(p.x, p.y)));
                    acc2 = __ffma2_rn(make_float2(p.z, p.w), h2[j], acc2);
                    hist2[(i * NPP + j) * 32 + lane] = h2[j];
                }
                party[(warp * kBwdTile + i) * 32 + lane] =
                    (warp == 0 ? dsk * uv : 0.0f) + (acc2.x + acc2.y);
            }
        }
        __syncwarp();
        // (c) backwards through the tile for this warp's entries, two entries
        //     at a time; h_t of step i is h_{t-1} of step i + 1, so each state
        //     is read once.  (Kept rolled: the unrolled tile's code overflows
        //     the instruction cache; measured on B300 6% slower.)
        float2 hn2[NPP];
#pragma unroll
        for (int j = 0; j < NPP; ++j)
            hn2[j] = nv > 0 ? hist2[((nv - 1) * NPP + j) * 32 + lane] : make_float2(0.0f, 0.0f);
        // Software-pipelined by one step: the step's (u, Delta, g) and Abar
        // are loaded and formed in the iteration before, so that the
        // shared-load and ex2 latency at the head of a step overlaps the
        // previous step's arithmetic and butterflies.
        float uvn = 0.0f, dtn = 0.0f, gn = 0.0f;
        float2 abn[NPP];
        auto head = [&](int i) {
            const float2 ud = srow[(2 * i) * 32 + lane];
            uvn = ud.x;
            dtn = ud.y;
            gn = srow[(2 * i + 1) * 32 + lane].x;
            const float2 dtl2 = make_float2(dtn * kLog2e, dtn * kLog2e);
#pragma unroll
            for (int j = 0; j < NPP; ++j) abn[j] = abar2_of<ACC>(dtn, dtl2, A2[j]);
        };
        head(nv > 0 ? nv - 1 : 0);
        // One step of the walk; the last one (i = 0) is peeled off so that
        // the loop's steps read h_{t-1} from the history without a select
        // (at i = 0 it is the checkpoint, hs2) and prefetch without a clamp.
        auto step = [&](int i, auto last) {
            constexpr bool LAST = decltype(last)::value;
            const float uv = uvn, dt = dtn, g = gn;
            float2 ab2[NPP];
#pragma unroll
            for (int j = 0; j < NPP; ++j) ab2[j] = abn[j];
            if constexpr (!LAST) head(i - 1);
            const float2 g2 = make_float2(g, g), dt2 = make_float2(dt, dt), uv2 = make_float2(uv, uv);
            float2 dus2 = make_float2(0.0f, 0.0f), dds2 = make_float2(0.0f, 0.0f);
            float pb[NPW], pc[NPW];
            const float2* hprev = hist2 + ((LAST ? 0 : i - 1) * NPP) * 32 + lane;
            const float4* brow = sbc + i * (NP / 2) + n0 / 2;
#pragma unroll
            for (int j = 0; j < NPP; ++j) {
                const float4 p = brow[j ^ pj];
                const float2 B2 = make_float2(p.x, p.y), C2 = make_float2(p.z, p.w);
                const float2 ht = hn2[j];
                const float2 hp = LAST ? hs2[j] : hprev[j * 32];
                hn2[j] = hp;
                const float2 ab = ab2[j];
                dh2[j] = __ffma2_rn(g2, C2, dh2[j]);
                const float2 pcv = __fmul2_rn(g2, ht);
                const float2 dhd = __fmul2_rn(dh2[j], dt2);
                const float2 pbv = __fmul2_rn(dhd, uv2);
                pc[2 * j] = pcv.x; pc[2 * j + 1] = pcv.y;
                pb[2 * j] = pbv.x; pb[2 * j + 1] = pbv.y;
                dus2 = __ffma2_rn(dhd, B2, dus2);
                const float2 tin = __ffma2_rn(__fmul2_rn(A2[j], ab), hp, __fmul2_rn(B2, uv2));
                dds2 = __ffma2_rn(dh2[j], tin, dds2);
                dA2[j] = __ffma2_rn(__fmul2_rn(dhd, ab), hp, dA2[j]);
                dh2[j] = __fmul2_rn(dh2[j], ab);
            }
            partd[(warp * kBwdTile + i) * 32 + lane] =
                make_float2((warp == 0 ? g * dsk : 0.0f) + (dus2.x + dus2.y), dds2.x + dds2.y);
            const float sb = warp_sum_lanes<NPW>(pb);
            const float sc = warp_sum_lanes<NPW>(pc);
            __syncwarp();   // every lane has read its pairs of row i
            if (writer) {
                sum_at[i * NP * 2] = sb;
                sum_at[i * NP * 2 + 2] = sc;
            }
        };
#pragma unroll 1
        for (int i = nv - 1; i >= 1; --i) step(i, std::false_type{});
        if (nv > 0) step(0, std::true_type{});
        __syncthreads();
        // (d) the tile's outputs, one lane per row: warp 0 du and ddelta,
        //     warp 1 dz; partial sums added in warp order.  The dB and dC
        //     sums of the tile go out as whole rows of 4 entries.
        if (warp == 0) {
            float o[kBwdTile], od[kBwdTile];
#pragma unroll
            for (int i = 0; i < kBwdTile; ++i) {
                float su = 0.0f, sd = 0.0f;
#pragma unroll
                for (int w = 0; w < SPL; ++w) {
                    const float2 pd = partd[(w * kBwdTile + i) * 32 + lane];
                    su += pd.x;
                    sd += pd.y;
                }
                const float2 ud = srow[(2 * i) * 32 + lane], gs = srow[(2 * i + 1) * 32 + lane];
                o[i] = su;
                od[i] = sd * gs.y;
                if (i < nv) {
                    dbias += od[i];
                    dD = fmaf(gs.x, ud.x, dD);
                }
            }
            if (q.ok) {
                store_tile_row<T>(dur, t0, nv, vec, o, q.row * L, big);
                store_tile_row<T>(ddr, t0, nv, vec, od, q.row * L, big);
            }
        } else if (HZ && warp == 1) {
            float o[kBwdTile];
#pragma unroll
            for (int i = 0; i < kBwdTile; ++i) {
                float sy = 0.0f;
#pragma unroll
                for (int w = 0; w < SPL; ++w) sy += party[(w * kBwdTile + i) * 32 + lane];
                o[i] = szf[i * 32 + lane] * sy;   // dz = dy (C.h + D u) silu'(z)
            }
            if (q.ok) store_tile_row<T>(dzr, t0, nv, vec, o, q.row * L, big);
        }
        {
            constexpr int kQuads = NP / 4;   // 4-entry quads per step
            for (int e = threadIdx.x; e < nv * kQuads; e += 32 * SPL) {
                const int i = e / kQuads, c = e % kQuads;
                const float4 f0 = sbc[i * (NP / 2) + 2 * c];
                const float4 f1 = sbc[i * (NP / 2) + 2 * c + 1];
                const long long off = (t0 + i) * NP + 4 * c;
                const long long at = ((long long)q.grp * a.batch + q.b) * L * NP + off;
                (void)at;
                if (MAMBA_IN(at, pext) && MAMBA_IN(at + 3, pext)) {
                    *reinterpret_cast<float4*>(pBg + off) = make_float4(f0.x, f0.y, f1.x, f1.y);
                    *reinterpret_cast<float4*>(pCg + off) = make_float4(f0.z, f0.w, f1.z, f1.w);
                }
            }
        }
        __syncthreads();   // shared memory is rewritten by the next tile
    }
    if (q.ok) {
#pragma unroll
        for (int j = 0; j < NPP; ++j) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int n = n0 + 2 * (j ^ pj) + e;
                MAMBA_ST(a.pA, ((long long)cidx * rows + q.row) * NP + n,
                         (long long)a.nchunks * rows * NP, e ? dA2[j].y : dA2[j].x);
                if (a.dh0 && n < N && cidx == 0)
                    MAMBA_ST(a.dh0, q.row * N + n, rows * N, e ? dh2[j].y : dh2[j].x);
            }
        }
        if (warp == 0) {
            MAMBA_ST(a.pD, (long long)cidx * rows + q.row, (long long)a.nchunks * rows, dD);
            MAMBA_ST(a.pbias, (long long)cidx * rows + q.row, (long long)a.nchunks * rows, dbias);
        }
    }
}

// dB[b][n][t] and dC[b][n][t] = sums over channel groups of the partials
// (blockIdx.y: 0 for dB, 1 for dC).  A block takes kReduceThreads / S
// consecutive partial elements; each of its S parts of threads adds the
// groups [groups * s / S, groups * (s + 1) / S) in group order, and the part
// sums are added in part order: a fixed order, so the result is
// deterministic.  S = 4 when there are many groups (the 2.8B layer's 160),
// else 1.
template <int S>
__global__ void __launch_bounds__(kReduceThreads)
bwd_reduce_bc_kernel(const float* __restrict__ pB, const float* __restrict__ pC,
                     float* __restrict__ dB, float* __restrict__ dC, int groups, int batch,
                     long long L, int N, int NP) {
    constexpr int kOuts = kReduceThreads / S;
    __shared__ float part_sum[S][kOuts];
    const float* part = blockIdx.y ? pC : pB;
    float* out = blockIdx.y ? dC : dB;
    const long long total = (long long)batch * L * NP;
    const int q = threadIdx.x / kOuts, o = threadIdx.x % kOuts;
    const int g0 = (int)((long long)groups * q / S), g1 = (int)((long long)groups * (q + 1) / S);
    for (long long base = (long long)blockIdx.x * kOuts; base < total;
         base += (long long)gridDim.x * kOuts) {
        const long long i = base + o;
        float s = 0.0f;
        if (i < total) {
#pragma unroll 8
            for (int g = g0; g < g1; ++g) s += MAMBA_LD(part, g * total + i, groups * total);
        }
        if constexpr (S > 1) {
            part_sum[q][o] = s;
            __syncthreads();
            if (q == 0) {
#pragma unroll
                for (int k = 1; k < S; ++k) s += part_sum[k][o];
            }
            __syncthreads();
        }
        if (q == 0 && i < total) {
            const int n = (int)(i % NP);
            if (n < N) {
                const long long bt = i / NP;   // b * L + t
                const long long b = bt / L, t = bt - b * L;
                MAMBA_ST(out, (b * N + n) * L + t, (long long)batch * N * L, s);
            }
        }
    }
}

// dA[d][n] = sum_b pA, dD[d] = sum_b pD, ddt_bias[d] = sum_b pbias, in batch order.
__global__ void __launch_bounds__(kReduceThreads)
bwd_reduce_params_kernel(const float* __restrict__ pA, const float* __restrict__ pD,
                         const float* __restrict__ pbias, float* __restrict__ dA,
                         float* __restrict__ dD, float* __restrict__ dbias, int batch,
                         long long dim, int N, int NP) {
    const long long total = dim * NP;
    for (long long i = (long long)blockIdx.x * kReduceThreads + threadIdx.x; i < total;
         i += (long long)gridDim.x * kReduceThreads) {
        const long long d = i / NP;
        const int n = (int)(i % NP);
        if (n < N) {
            float s = 0.0f;
            for (int b = 0; b < batch; ++b)
                s += MAMBA_LD(pA, ((long long)b * dim + d) * NP + n, batch * dim * NP);
            MAMBA_ST(dA, d * N + n, dim * N, s);
        }
        if (n == 0) {
            float sd = 0.0f, sb = 0.0f;
            for (int b = 0; b < batch; ++b) {
                sd += MAMBA_LD(pD, (long long)b * dim + d, batch * dim);
                sb += MAMBA_LD(pbias, (long long)b * dim + d, batch * dim);
            }
            if (dD) MAMBA_ST(dD, d, dim, sd);
            if (dbias) MAMBA_ST(dbias, d, dim, sb);
        }
    }
}

// Time chunks of the reverse pass.  When the units of 32 channels are too
// few to fill the GPU, every unit's tiles are cut into chunks that run as
// separate CTAs.  A chunk's reverse walk needs dJ/dh at its end, which its
// later chunks send back; the recurrence of dh is linear, so, with
// dloc_c = what chunk c's own steps send into the state before it (walking
// them last to first from dh = 0: dh += g_t C_t, then dh *= Abar_t) and
// P_c = exp(A * (sum of Delta over chunk c)), the gradient at the end of
// chunk c - 1 is dloc_c + P_c * (the gradient at the end of chunk c), from
// d_final_state at the end of the last chunk.

// dloc_c and the chunk's sum of Delta, for chunks 1 .. nchunks - 1: one lane
// per channel; the NP entries split over NP / 4 warps of four entries each;
// grid (units, nchunks - 1).  Per 12-step tile, last to first, as in the
// reverse pass: the tile's Delta and g = dy silu(z) (warp 0, then shared)
// and its packed B/C rows are staged in shared memory, with the next tile's
// global loads issued before the walk.
template <int NP>
__host__ __device__ constexpr int bwd_summary_warps() {
    return NP >= 8 ? NP / 4 : 1;
}
template <typename T, int NP, bool SP, bool HZ>
__global__ void __launch_bounds__(32 * bwd_summary_warps<NP>())
bwd_summary_kernel(const BwdArgs a) {
    constexpr bool ACC = IO<T>::kAccurate;
    constexpr int SW = bwd_summary_warps<NP>();
    constexpr int NW = NP / SW;   // entries per warp: 4
    constexpr int kRowsPerThread = (kBwdTile * (NP / 2) + 32 * SW - 1) / (32 * SW);
    __shared__ float2 sdg[kBwdTile][32];           // (Delta, g) per step and lane
    __shared__ float4 sbc[kBwdTile * (NP / 2)];    // the tile's packed B/C rows
    const int warp = threadIdx.x >> 5;
    const WarpUnit q = warp_unit(a, blockIdx.x);
    const int lane = q.lane;
    const int cidx = blockIdx.y + 1;
    const int N = a.N, n0 = warp * NW;
    const long long L = a.L;
    const long long rows = (long long)a.batch * a.dim, big = rows * L;
    (void)big;
    float Av[NW], dh[NW];
#pragma unroll
    for (int j = 0; j < NW; ++j) {
        const int n = n0 + j;
        Av[j] = (q.ok && n < N) ? MAMBA_LD(a.A, q.d * N + n, a.dim * N) : 0.0f;
        dh[j] = 0.0f;
    }
    const float bias = (q.ok && a.dt_bias) ? MAMBA_LD(a.dt_bias, q.d, a.dim) : 0.0f;
    const T* dl = static_cast<const T*>(a.delta) + q.row * L;
    const T* dyr = static_cast<const T*>(a.dy) + q.row * L;
    const T* zr = HZ ? static_cast<const T*>(a.z) + q.row * L : nullptr;
    const bool vec = a.vec8 != 0;
    const int k_lo = cidx * a.chunk_tiles;
    const int k_hi = min(a.ntiles, k_lo + a.chunk_tiles) - 1;
    float rd[kBwdTile], ry[kBwdTile], rz[kBwdTile];
    float4 bcr[kRowsPerThread];
    auto fetch = [&](int kk) {
        const long long t0 = (long long)kk * kBwdTile;
        const int nv = (int)min((long long)kBwdTile, L - t0);
        if (warp == 0) {
            load_tile_row<T>(dl, t0, nv, vec, q.ok, rd, q.row * L, big);
            load_tile_row<T>(dyr, t0, nv, vec, q.ok, ry, q.row * L, big);
            if constexpr (HZ) load_tile_row<T>(zr, t0, nv, vec, q.ok, rz, q.row * L, big);
        }
#pragma unroll
        for (int r = 0; r < kRowsPerThread; ++r) {
            const int e = r * 32 * SW + threadIdx.x;
            const int i = e / (NP / 2);
            bcr[r] = (e < kBwdTile * (NP / 2) && i < nv)
                         ? MAMBA_LD(a.bc, (q.b * L + t0 + i) * (NP / 2) + (e % (NP / 2)),
                                    (long long)a.batch * L * (NP / 2))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    float sdt = 0.0f;
    if (k_hi >= k_lo) fetch(k_hi);
    for (int k = k_hi; k >= k_lo; --k) {
        const long long t0 = (long long)k * kBwdTile;
        const int nv = (int)min((long long)kBwdTile, L - t0);
        if (warp == 0) {
#pragma unroll
            for (int i = 0; i < kBwdTile; ++i) {
                const float dt = (q.ok && i < nv) ? delta_nat<ACC, SP>(rd[i] + bias) : 0.0f;
                float g = ry[i];
                if constexpr (HZ) g = g * rz[i] * sigmoid_f<ACC>(rz[i]);
                sdt += dt;
                sdg[i][lane] = make_float2(dt, g);
            }
        }
#pragma unroll
        for (int r = 0; r < kRowsPerThread; ++r) {
            const int e = r * 32 * SW + threadIdx.x;
            if (e < kBwdTile * (NP / 2)) sbc[e] = bcr[r];
        }
        if (k > k_lo) fetch(k - 1);
        __syncthreads();
#pragma unroll
        for (int i = kBwdTile - 1; i >= 0; --i) {
            if (i >= nv) continue;
            const float2 dg = sdg[i][lane];
            const float dtl = dg.x * kLog2e;
#pragma unroll
            for (int j = 0; j < NW / 2; ++j) {
                const float4 p = sbc[i * (NP / 2) + n0 / 2 + j];
                dh[2 * j] = fmaf(dg.y, p.z, dh[2 * j]);
                dh[2 * j + 1] = fmaf(dg.y, p.w, dh[2 * j + 1]);
            }
#pragma unroll
            for (int j = 0; j < NW; ++j)
                dh[j] *= ACC ? expf(dg.x * Av[j]) : ex2_approx(dtl * Av[j]);
        }
        __syncthreads();   // shared memory is rewritten by the next tile
    }
    if (q.ok) {
        const long long at = (long long)cidx * rows + q.row;
#pragma unroll
        for (int j = 0; j < NW; ++j)
            MAMBA_ST(a.dloc, at * NP + n0 + j, (long long)a.nchunks * rows * NP, dh[j]);
        if (warp == 0) MAMBA_ST(a.sdt, at, (long long)a.nchunks * rows, sdt);
    }
}

// dJ/dh at the end of every chunk, last chunk first; one thread per (row, n).
__global__ void __launch_bounds__(kReduceThreads)
bwd_chunk_carry_kernel(const BwdArgs a, int NP) {
    const long long rows = (long long)a.batch * a.dim;
    const long long i = (long long)blockIdx.x * kReduceThreads + threadIdx.x;
    if (i >= rows * NP) return;
    const long long row = i / NP, d = row % a.dim;
    const int n = (int)(i % NP);
    const bool on = n < a.N;
    const long long ext = (long long)a.nchunks * rows * NP;
    (void)ext;
    float carry = (on && a.dfinal) ? MAMBA_LD(a.dfinal, row * a.N + n, rows * a.N) : 0.0f;
    const float An = on ? MAMBA_LD(a.A, d * a.N + n, a.dim * a.N) : 0.0f;
    for (int c = a.nchunks - 1; c >= 0; --c) {
        const long long at = ((long long)c * rows + row) * NP + n;
        MAMBA_ST(a.dcarry, at, ext, carry);
        if (c > 0) {
            const float P = expf(An * MAMBA_LD(a.sdt, (long long)c * rows + row,
                                               (long long)a.nchunks * rows));
            carry = fmaf(P, carry, MAMBA_LD(a.dloc, at, ext));
        }
    }
}

template <typename T, int NP, bool SP>
cudaError_t launch_bwd(const BwdArgs& a, bool hz, cudaStream_t st) {
    const long long units = (long long)a.batch * a.groups;
    cudaError_t e;
    const int smem = bwd_smem_floats<NP>() * (int)sizeof(float);
    auto k = hz ? bwd_kernel<T, NP, SP, true> : bwd_kernel<T, NP, SP, false>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (a.nchunks > 1) {
        ProfScope prof(kKindBwdSummary, st);
        auto ks = hz ? bwd_summary_kernel<T, NP, SP, true> : bwd_summary_kernel<T, NP, SP, false>;
        ks<<<dim3((unsigned)units, (unsigned)(a.nchunks - 1)), 32 * bwd_summary_warps<NP>(), 0,
             st>>>(a);
        const long long n = (long long)a.batch * a.dim * NP;
        bwd_chunk_carry_kernel<<<(unsigned)((n + kReduceThreads - 1) / kReduceThreads),
                                 kReduceThreads, 0, st>>>(a, NP);
    }
    {
        ProfScope prof(kKindBwd, st);
        k<<<dim3((unsigned)units, (unsigned)a.nchunks), 32 * bwd_split<NP>(), smem, st>>>(a);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_bwd(int np, bool sp, bool hz, const BwdArgs& a, cudaStream_t st) {
#define X(NP_)                                                                     \
    if (np == NP_) return sp ? launch_bwd<T, NP_, true>(a, hz, st) : launch_bwd<T, NP_, false>(a, hz, st);
    X(4) X(8) X(16)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace

// The debug word of this translation unit (the index checks of debug builds).
int bwd_take_debug_word() { return take_debug_word(); }

}  // namespace mamba

using namespace mamba;

namespace {

// Both backward entry points.  ckpt_in: the checkpoints of a training
// forward (then the checkpoint pass is skipped), or null.
int bwd_common(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int io_dtype,
               const void* u, const void* delta, const float* dt_bias, const float* A,
               const void* B, const void* C, const float* D_skip, const void* z, int flags,
               const float* initial_state, const float* ckpt_in, const void* dy,
               const float* d_final_state, void* du, void* ddelta, float* dA, float* dB,
               float* dC, float* dD_skip, void* dz, float* ddt_bias, float* d_initial_state,
               cudaStream_t stream) {
    if (flags & ~MAMBA_FLAG_SOFTPLUS) return MAMBA_ERR_FLAGS;
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (batch < 1 || dim < 1 || dstate < 1 || dstate > kMaxN || seqlen < 0) return MAMBA_ERR_SHAPE;
    if (batch > INT32_MAX / 2 || dim > (1ll << 40) || seqlen > (1ll << 40) ||
        (double)batch * dim * (double)(seqlen > 0 ? seqlen : 1) > 4.0e18)
        return MAMBA_ERR_SHAPE;
    if (!A || !dA) return MAMBA_ERR_NULL;
    if (seqlen > 0 && (!u || !delta || !B || !C || !dy || !du || !ddelta || !dB || !dC))
        return MAMBA_ERR_NULL;
    if (z && seqlen > 0 && !dz) return MAMBA_ERR_NULL;
    if (seqlen > 0 && checkpoint_tiles(seqlen) > INT32_MAX) return MAMBA_ERR_SHAPE;
    const int es = esize(io_dtype);
    const size_t big = (size_t)(batch * dim * seqlen) * es;
    const size_t bcb = (size_t)(batch * dstate * seqlen) * es;
    const size_t bcf = (size_t)(batch * dstate * seqlen) * 4;
    const size_t stb = (size_t)(batch * dim * dstate) * 4;
    const size_t ab = (size_t)(dim * dstate) * 4, vb = (size_t)dim * 4;
    for (const void* q : {u, delta, z, dy, B, C, (const void*)du, (const void*)ddelta,
                          (const void*)dz})
        if (q && !aligned(q, es)) return MAMBA_ERR_ALIGN;
    for (const void* q : {(const void*)dt_bias, (const void*)A, (const void*)D_skip,
                          (const void*)initial_state, (const void*)d_final_state, (const void*)dA,
                          (const void*)dB, (const void*)dC, (const void*)dD_skip,
                          (const void*)ddt_bias, (const void*)d_initial_state})
        if (q && !aligned(q, 4)) return MAMBA_ERR_ALIGN;
    if (ckpt_in && !aligned(ckpt_in, 16)) return MAMBA_ERR_ALIGN;
    {
        const size_t ckb = (size_t)(batch * dim) * checkpoint_tiles(seqlen) * padded_state(dstate) * 4;
        const void* ins[] = {u, delta, z, dy, B, C, dt_bias, A, D_skip, initial_state,
                             d_final_state, ckpt_in};
        const size_t insz[] = {big, big, big, big, bcb, bcb, vb, ab, vb, stb, stb, ckb};
        void* outs[] = {du, ddelta, dz, dA, dB, dC, dD_skip, ddt_bias, d_initial_state};
        const size_t outsz[] = {big, big, big, ab, bcf, bcf, vb, vb, stb};
        for (int o = 0; o < 9; ++o) {
            for (int i = 0; i < 12; ++i)
                if (overlaps(outs[o], outsz[o], ins[i], insz[i])) return MAMBA_ERR_ALIAS;
            for (int p = o + 1; p < 9; ++p)
                if (overlaps(outs[o], outsz[o], outs[p], outsz[p])) return MAMBA_ERR_ALIAS;
        }
    }
    const bool sp = (flags & MAMBA_FLAG_SOFTPLUS) != 0;
    if (seqlen == 0) {
        // no steps: only the initial state reaches the final state
        cudaError_t e = cudaMemsetAsync(dA, 0, ab, stream);
        if (e == cudaSuccess && dD_skip) e = cudaMemsetAsync(dD_skip, 0, vb, stream);
        if (e == cudaSuccess && ddt_bias) e = cudaMemsetAsync(ddt_bias, 0, vb, stream);
        if (e == cudaSuccess && d_initial_state)
            e = d_final_state ? cudaMemcpyAsync(d_initial_state, d_final_state, stb,
                                                cudaMemcpyDeviceToDevice, stream)
                              : cudaMemsetAsync(d_initial_state, 0, stb, stream);
        return e == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MAMBA_ERR_CUDA;
    const int np = padded_state(dstate);
    const int groups = (int)((dim + 31) / 32);
    const int ntiles = (int)checkpoint_tiles(seqlen);
    // time chunks when the units of 32 channels fill at most a quarter of
    // the reverse pass's CTA slots (five per SM): as many as fill them, of at
    // least four tiles each.  (Measured on B300: b1 d1536 n16, 48 units,
    // L = 262144: 118.6 -> 25.1 ms; b2 d5120, 320 units, L = 8192, in two
    // chunks: 4.85 -> 5.52 ms, the summary pass costing more than the
    // doubled occupancy gains.)
    const long long units = batch * groups;
    const long long slots = 5LL * sm_count(dev);
    int nchunks = 1, chunk_tiles = ntiles;
    if (units * 4 <= slots && ntiles >= 16) {
        const long long want = std::min<long long>(slots / units, ntiles / 4);
        if (want >= 4) {
            chunk_tiles = (int)((ntiles + want - 1) / want);
            nchunks = (ntiles + chunk_tiles - 1) / chunk_tiles;
        }
    }
    const size_t rows = (size_t)(batch * dim);
    const size_t sz_bc = (size_t)batch * seqlen * (np / 2) * sizeof(float4);
    const size_t sz_ck = ckpt_in ? 0 : rows * ntiles * np * sizeof(float);
    const size_t sz_p = (size_t)groups * batch * seqlen * np * sizeof(float);
    const size_t sz_a = (size_t)nchunks * rows * np * sizeof(float);
    const size_t sz_r = (size_t)nchunks * rows * sizeof(float);
    const size_t sz_c = nchunks > 1 ? sz_a : 0;   // dloc and dcarry, each
    const size_t sz_s = nchunks > 1 ? sz_r : 0;   // sdt
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t total = up(sz_bc) + up(sz_ck) + 2 * up(sz_p) + up(sz_a) + 2 * up(sz_r) +
                         2 * up(sz_c) + up(sz_s);
    cudaMemPool_t pool = nullptr;
    int rc = get_pool(dev, &pool);
    if (rc != MAMBA_OK) return rc;
    void* scratch = nullptr;
    if (cudaMallocFromPoolAsync(&scratch, total, pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return MAMBA_ERR_ALLOC;
    }
    char* p = static_cast<char*>(scratch);
    BwdArgs a;
    std::memset(&a, 0, sizeof(a));
    a.bc = reinterpret_cast<const float4*>(p); p += up(sz_bc);
    a.ckpt = ckpt_in ? const_cast<float*>(ckpt_in) : reinterpret_cast<float*>(p);
    p += up(sz_ck);
    a.pB = reinterpret_cast<float*>(p); p += up(sz_p);
    a.pC = reinterpret_cast<float*>(p); p += up(sz_p);
    a.pA = reinterpret_cast<float*>(p); p += up(sz_a);
    a.pD = reinterpret_cast<float*>(p); p += up(sz_r);
    a.pbias = reinterpret_cast<float*>(p); p += up(sz_r);
    if (nchunks > 1) {
        a.dloc = reinterpret_cast<float*>(p); p += up(sz_c);
        a.dcarry = reinterpret_cast<float*>(p); p += up(sz_c);
        a.sdt = reinterpret_cast<float*>(p);
    }
    a.nchunks = nchunks;
    a.chunk_tiles = chunk_tiles;
    a.u = u; a.delta = delta; a.z = z; a.dy = dy;
    a.dt_bias = dt_bias; a.A = A; a.D_skip = D_skip;
    a.h0 = initial_state; a.dfinal = d_final_state;
    a.du = du; a.ddelta = ddelta; a.dz = dz; a.dh0 = d_initial_state;
    a.dim = dim; a.L = seqlen; a.batch = (int)batch; a.N = (int)dstate;
    a.groups = groups; a.ntiles = ntiles;
    a.vec8 = ((seqlen * es) % 8) == 0;
    for (const void* q : {u, delta, z, dy, (const void*)du, (const void*)ddelta, (const void*)dz})
        if (q && !aligned(q, 8)) a.vec8 = 0;

    // checkpoints (unless given): the forward kernel's checkpoint mode (its
    // own B/C table and plan, from the same pool on the same stream)
    if (!ckpt_in) {
        ProfScope prof(kKindBwdCheckpoint, stream);
        rc = scan_checkpoints(batch, dim, dstate, seqlen, io_dtype, u, delta, dt_bias, A, B, C,
                              sp ? 1 : 0, initial_state, a.ckpt, ntiles, stream);
    }
    if (rc != MAMBA_OK) {
        cudaFreeAsync(scratch, stream);
        return rc;
    }
    cudaError_t e = launch_pack_bc(io_dtype, B, C, const_cast<float4*>(a.bc), batch, seqlen,
                                   (int)dstate, np, 1.0f, stream);
    if (e == cudaSuccess)
        e = io_dtype == MAMBA_BF16 ? dispatch_bwd<__nv_bfloat16>(np, sp, z != nullptr, a, stream)
                                   : dispatch_bwd<float>(np, sp, z != nullptr, a, stream);
    if (e == cudaSuccess) {
        ProfScope prof(kKindBwdReduce, stream);
        const int cap = 16 * sm_count(dev);
        const long long nbc = (long long)batch * seqlen * np;
        const int outs = groups >= 96 ? kReduceThreads / 4 : kReduceThreads;
        const int g1 = (int)std::max<long long>(1, std::min<long long>((nbc + outs - 1) / outs, cap));
        if (groups >= 96)
            bwd_reduce_bc_kernel<4><<<dim3(g1, 2), kReduceThreads, 0, stream>>>(
                a.pB, a.pC, dB, dC, groups, (int)batch, seqlen, (int)dstate, np);
        else
            bwd_reduce_bc_kernel<1><<<dim3(g1, 2), kReduceThreads, 0, stream>>>(
                a.pB, a.pC, dB, dC, groups, (int)batch, seqlen, (int)dstate, np);
        const long long npar = dim * np;
        const int g2 = (int)std::max<long long>(1, std::min<long long>((npar + kReduceThreads - 1) / kReduceThreads, cap));
        // partials of every (chunk, batch entry), added in that order
        bwd_reduce_params_kernel<<<g2, kReduceThreads, 0, stream>>>(
            a.pA, a.pD, a.pbias, dA, dD_skip, ddt_bias, (int)(batch * nchunks), dim, (int)dstate,
            np);
        e = cudaGetLastError();
    }
    cudaFreeAsync(scratch, stream);
    return e == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

}  // namespace

extern "C" {

int mamba_scan_bwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, mamba_dtype_t io_dtype,
                   const void* u, const void* delta, const float* dt_bias, const float* A,
                   const void* B, const void* C, const float* D_skip, const void* z, int flags,
                   const float* initial_state, const void* dy, const float* d_final_state,
                   void* du, void* ddelta, float* dA, float* dB, float* dC, float* dD_skip,
                   void* dz, float* ddt_bias, float* d_initial_state, cudaStream_t stream) {
    return bwd_common(batch, dim, dstate, seqlen, io_dtype, u, delta, dt_bias, A, B, C, D_skip,
                      z, flags, initial_state, nullptr, dy, d_final_state, du, ddelta, dA, dB,
                      dC, dD_skip, dz, ddt_bias, d_initial_state, stream);
}

int mamba_scan_bwd_ckpt(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                        mamba_dtype_t io_dtype, const void* u, const void* delta,
                        const float* dt_bias, const float* A, const void* B, const void* C,
                        const float* D_skip, const void* z, int flags, const float* checkpoints,
                        const void* dy, const float* d_final_state, void* du, void* ddelta,
                        float* dA, float* dB, float* dC, float* dD_skip, void* dz,
                        float* ddt_bias, float* d_initial_state, cudaStream_t stream) {
    if (seqlen > 0 && !checkpoints) return MAMBA_ERR_NULL;
    return bwd_common(batch, dim, dstate, seqlen, io_dtype, u, delta, dt_bias, A, B, C, D_skip,
                      z, flags, nullptr, checkpoints, dy, d_final_state, du, ddelta, dA, dB,
                      dC, dD_skip, dz, ddt_bias, d_initial_state, stream);
}

}  // extern "C"
