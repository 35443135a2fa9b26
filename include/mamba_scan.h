/*
 * mamba_scan.h - C ABI of the B300 (sm_103a) selective-scan library.
 *
 * The operation is the selective state space layer "S6" of Mamba
 * (page "Mamba: linear-time sequence modeling with selective state spaces",
 * section "What they did", S6 bullet): Delta, B and C depend on the input,
 * Delta = softplus(parameter + Linear(x)), A is input-independent and enters
 * through Abar = exp(Delta*A), and the time-varying model is evaluated as a
 * recurrent scan over a D x N state per sequence (same page, "the recurrent
 * state is D x N numbers per layer").  Per (b, d) row and time step t:
 *
 *     s        = delta[b,d,t] + dt_bias[d]
 *     Delta    = softplus(s)   (or s when the softplus flag is 0)
 *     h[n]     = exp(Delta*A[d,n]) * h[n] + Delta * B[b,n,t] * u[b,d,t]
 *     y[b,d,t] = (sum_n C[b,n,t]*h[n] + D_skip[d]*u[b,d,t]) * silu(z[b,d,t])
 *
 * The input term is the Euler step Delta*B*u; the skip term and the silu
 * gate are the Mamba block's (page "Mamba: linear-time sequence modeling
 * with selective state spaces", "Architecture": the block merges H3 with a
 * gated MLP).  mamba_state_update is the generation mode: one step of the
 * same recurrence on a caller-held state (page "Mamba: Linear-Time Sequence
 * Modeling with Selective State Spaces", "Architecture": producing a token
 * needs only one update of the state).
 *
 * Entry points
 *   mamba_scan_fwd          the scan from a zero state (the hot path)
 *   mamba_scan_fwd_ex       the scan from an initial state, with per-entry
 *                           lengths, zero-order hold and the no-allocation
 *                           scratch as options
 *   mamba_scan_fwd_noalloc  mamba_scan_fwd with fixed scratch, no allocation
 *   mamba_state_update(_ex) one generation step on a caller-held state
 *   mamba_scan_bwd          gradients of every scan input (state recomputed)
 *   mamba_scan_fwd_train    the forward of a training step: outputs plus the
 *                           state checkpoints mamba_scan_bwd_ckpt reads
 *   mamba_scan_bwd_ckpt     mamba_scan_bwd from those checkpoints
 *   mamba_conv1d_fwd        the causal convolution in front of the scan
 *   mamba_conv1d_update     its generation step
 *   plus status strings, the device error word and its self-test, tuning
 *   and per-launch timing.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers on the current CUDA device and
 *     are dense row-major with the shapes given below.  The caller owns
 *     every buffer; the library never frees or retains caller memory.
 *   - io_dtype selects the storage type of u, delta, z, y, x, B and C:
 *     MAMBA_F32 (float) or MAMBA_BF16 (bfloat16).  A, dt_bias, D_skip and
 *     the state are always fp32; all arithmetic is fp32.  y is rounded to
 *     the storage type with round-to-nearest-even.
 *   - Nullable pointers: dt_bias (taken as 0), D_skip (taken as 0), z (no
 *     gate), final_state (not written).
 *   - Work is enqueued on `stream` and is asynchronous; a return of MAMBA_OK
 *     means the launch was accepted.  Results are ready when the stream is.
 *   - Argument errors are detected on the host before anything is launched
 *     and nothing is written in that case.  Launch failures are reported as
 *     MAMBA_ERR_CUDA.  A device-side wait that exceeds its time bound (1 s)
 *     sets a per-device error word instead of hanging; mamba_device_status
 *     reads and clears it.
 *   - Outputs must not overlap inputs.  Concurrent calls on different
 *     streams are safe; each call's scratch memory is stream-ordered.
 *   - Limits: 1 <= dstate <= 16; batch, dim >= 1; seqlen >= 0 (0 is a
 *     no-op that zeroes final_state).
 *   - Rows whose length in bytes is a multiple of 16 (seqlen % 8 == 0 for
 *     bf16, % 4 == 0 for fp32) with 16-byte aligned base pointers are
 *     streamed with tensor-map bulk copies; any other shape runs through the
 *     same kernels with element-wise, bounds-checked loads and stores.
 */
#ifndef MAMBA_SCAN_H
#define MAMBA_SCAN_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MAMBA_F32 = 0,
    MAMBA_BF16 = 1
} mamba_dtype_t;

typedef enum {
    MAMBA_OK = 0,
    MAMBA_ERR_NULL = -1,     /* a required pointer is NULL */
    MAMBA_ERR_SHAPE = -2,    /* a size is out of range */
    MAMBA_ERR_ALIGN = -3,    /* a pointer is not aligned to its element type */
    MAMBA_ERR_CUDA = -4,     /* a CUDA runtime call or kernel launch failed */
    MAMBA_ERR_TIMEOUT = -5,  /* a device-side wait ran out (mamba_device_status) */
    MAMBA_ERR_ALLOC = -6,    /* scratch memory could not be obtained */
    MAMBA_ERR_DTYPE = -7,    /* io_dtype is not one of mamba_dtype_t */
    MAMBA_ERR_ALIAS = -8,    /* an output overlaps an input */
    MAMBA_ERR_TOO_BIG = -9,  /* needs more than MAMBA_NOALLOC_SCRATCH_BYTES of scratch */
    MAMBA_ERR_FLAGS = -10,   /* a flags argument has a bit the call does not know */
    MAMBA_ERR_BOUNDS = -11   /* a debug build's index check failed (mamba_device_status) */
} mamba_status_t;

/* Bits of the `flags` argument of the extended entry points. */
#define MAMBA_FLAG_SOFTPLUS 1  /* Delta = softplus(delta + dt_bias), else delta + dt_bias */
#define MAMBA_FLAG_ZOH 2       /* zero-order-hold input term, else Euler (Delta * B * u) */
#define MAMBA_FLAG_NOALLOC 4   /* scan: fixed scratch, no allocation (as mamba_scan_fwd_noalloc) */

/* Size of the fixed scratch array used by mamba_scan_fwd_noalloc (16 MiB). */
#define MAMBA_NOALLOC_SCRATCH_BYTES (16ll << 20)

/*
 * Selective scan over a whole sequence, starting from a zero state.
 *
 *   u, delta, z : (batch, dim, seqlen)    io_dtype     z nullable
 *   B, C        : (batch, dstate, seqlen) io_dtype     shared by all d
 *   A           : (dim, dstate)           fp32         input-independent
 *   dt_bias     : (dim)                   fp32         nullable
 *   D_skip      : (dim)                   fp32         nullable
 *   softplus    : nonzero -> Delta = softplus(delta + dt_bias)
 *   y           : (batch, dim, seqlen)    io_dtype     written
 *   final_state : (batch, dim, dstate)    fp32         nullable; h after the last step
 *
 * Every call first packs B and C into an fp32 per-step table (batch *
 * seqlen * 32 floats at most) that the scan kernel streams.  When the
 * channels alone cannot fill the GPU, the sequence is also split into time
 * chunks that run in parallel; a carry pass composes their (decay, state)
 * pairs.  The table and the carry buffers are scratch memory obtained
 * stream-ordered from a library-owned pool on `stream` and returned to it
 * on the same stream.
 */
int mamba_scan_fwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                   mamba_dtype_t io_dtype,
                   const void *u, const void *delta, const float *dt_bias,
                   const float *A, const void *B, const void *C,
                   const float *D_skip, const void *z, int softplus,
                   void *y, float *final_state, cudaStream_t stream);

/*
 * mamba_scan_fwd without any memory allocation.  The paper has no
 * counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc or a stream-ordered allocator, for example code running under a
 * runtime that owns all device memory in a fixed arena, or a latency-critical
 * path where an allocation may block, synchronise or fail under
 * fragmentation.  Arguments, layouts, results and error codes are those of
 * mamba_scan_fwd.
 *
 * Its scratch (the packed B/C table and, for time-chunked plans, the chunk
 * summaries) lives in one fixed array of MAMBA_NOALLOC_SCRATCH_BYTES bytes
 * in the library's device memory, held by every GPU that loads the library
 * until the process exits.  A call whose scratch would exceed it returns
 * MAMBA_ERR_TOO_BIG and launches nothing; the packed table alone needs
 * batch * seqlen * 128 bytes when dstate > 8 (64 bytes for dstate <= 8,
 * 32 for dstate <= 4), so batch * seqlen up to 131072 fits at dstate 16
 * when no time chunks are needed.
 *
 * Every call looks up the array's device address (cudaGetSymbolAddress,
 * which allocates nothing) for the calling thread's current device and
 * context, so the address is never stale.  The first call on a device may
 * load the library's device code; make it before any stream capture.  All
 * calls share the one array: calls whose
 * work overlaps on the GPU (different streams, or different host threads)
 * race on it and must be serialised by the caller.  Every byte a call reads
 * from the array is written earlier in the same call, so nothing needs
 * clearing between calls.
 */
int mamba_scan_fwd_noalloc(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                           mamba_dtype_t io_dtype,
                           const void *u, const void *delta, const float *dt_bias,
                           const float *A, const void *B, const void *C,
                           const float *D_skip, const void *z, int softplus,
                           void *y, float *final_state, cudaStream_t stream);

/*
 * mamba_scan_fwd with an initial state, per-entry lengths and a choice of
 * discretisation: the scan side of chunked prefill (a long sequence handed
 * over in pieces, each starting from the previous piece's final_state) and
 * of a padded batch of sequences with different lengths.  Arguments as in
 * mamba_scan_fwd, plus:
 *
 *   flags         : MAMBA_FLAG_* bits; other bits -> MAMBA_ERR_FLAGS
 *   initial_state : (batch, dim, dstate) fp32, nullable (zero state); h
 *                   before the first step.  Must not overlap y or
 *                   final_state (MAMBA_ERR_ALIAS): ping-pong two buffers to
 *                   chain pieces.
 *   seqlens       : (batch) int32 on the device, nullable (all entries use
 *                   seqlen steps).  Entry b uses steps [0, seqlens[b]);
 *                   values are clamped to [0, seqlen].  For t >= seqlens[b]
 *                   the state is kept, y[b, :, t] is written as 0, and
 *                   final_state[b] is h after step seqlens[b] - 1 (the
 *                   initial state when seqlens[b] == 0).
 *
 * Discretisation.  Euler (the default, as mamba_scan_fwd): h <- Abar h +
 * Delta B u.  MAMBA_FLAG_ZOH: h <- Abar h + ((Abar - 1) / A) B u per state
 * entry (zero-order hold of the continuous system; the weight tends to
 * Delta where A == 0, and that entry takes Delta).  With N = 1, A = -1,
 * B = 1 it makes the scan exactly the gated RNN of Theorem 1 (paper "Mamba:
 * linear-time sequence modeling with selective state spaces", "Main
 * results").  Abar = exp(Delta A) in both.
 *
 * With MAMBA_FLAG_NOALLOC the call takes its scratch from the fixed array
 * of mamba_scan_fwd_noalloc, with the same limits and the same rule on
 * overlapping calls; otherwise from the stream-ordered pool.  When seqlen
 * is 0, final_state (if given) receives initial_state (or zeros).
 */
int mamba_scan_fwd_ex(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                      mamba_dtype_t io_dtype,
                      const void *u, const void *delta, const float *dt_bias,
                      const float *A, const void *B, const void *C,
                      const float *D_skip, const void *z, int flags,
                      const float *initial_state, const int32_t *seqlens,
                      void *y, float *final_state, cudaStream_t stream);

/*
 * One generation step, updating `state` in place:
 *
 *   state       : (batch, dim, dstate)    fp32         read and written
 *   x, delta, z : (batch, dim)            io_dtype     z nullable
 *   B, C        : (batch, dstate)         io_dtype
 *   A           : (dim, dstate)           fp32
 *   dt_bias     : (dim)                   fp32         nullable
 *   D_skip      : (dim)                   fp32         nullable
 *   y           : (batch, dim)            io_dtype     written
 *
 * Delta = softplus(delta + dt_bias) always (the generation step has no flag).
 * `state` must not overlap y or any input.  Allocates nothing.
 */
int mamba_state_update(int64_t batch, int64_t dim, int64_t dstate, mamba_dtype_t io_dtype,
                       float *state, const void *x, const void *delta,
                       const float *dt_bias, const float *A,
                       const void *B, const void *C, const float *D_skip,
                       const void *z, void *y, cudaStream_t stream);

/*
 * mamba_state_update with flags: MAMBA_FLAG_SOFTPLUS (Delta = softplus(delta
 * + dt_bias), else delta + dt_bias) and MAMBA_FLAG_ZOH (the input term of
 * mamba_scan_fwd_ex's zero-order hold).  Any other bit, MAMBA_FLAG_NOALLOC
 * included, returns MAMBA_ERR_FLAGS (the step allocates nothing anyway).
 * With flags = MAMBA_FLAG_SOFTPLUS it is mamba_state_update.  The step that
 * follows a mamba_scan_fwd_ex prefill takes the same SOFTPLUS and ZOH bits.
 */
int mamba_state_update_ex(int64_t batch, int64_t dim, int64_t dstate, mamba_dtype_t io_dtype,
                          float *state, const void *x, const void *delta,
                          const float *dt_bias, const float *A,
                          const void *B, const void *C, const float *D_skip,
                          const void *z, int flags, void *y, cudaStream_t stream);

/*
 * Backward pass of the scan (Euler input term): gradients of a loss J with
 * respect to every input, given dy = dJ/dy and optionally dJ/d final_state.
 * The states are recomputed, not stored by the forward call (paper "Mamba:
 * linear-time sequence modeling with selective state spaces", "What they
 * did": the fused scan recomputes the expanded state in the backward pass):
 * a checkpoint pass keeps the state every 12 steps in scratch memory, and a
 * reverse pass recomputes each 12-step tile from its checkpoint.  With few
 * units of 32 channels (batch * ceil(dim / 32) at most a quarter of five per
 * SM) the reverse pass is cut into time chunks: a summary pass gives each
 * chunk's own contribution to dJ/dh and its decay, a carry pass composes
 * them from the last chunk back, and every chunk then runs as its own CTA.
 *
 *   inputs as in mamba_scan_fwd_ex (u, delta, dt_bias, A, B, C, D_skip, z,
 *   initial_state), plus
 *   flags          : MAMBA_FLAG_SOFTPLUS only (other bits -> MAMBA_ERR_FLAGS)
 *   dy             : (batch, dim, seqlen)    io_dtype
 *   d_final_state  : (batch, dim, dstate)    fp32   nullable (taken as 0)
 * outputs (written, never accumulated into):
 *   du, ddelta     : (batch, dim, seqlen)    io_dtype
 *   dz             : (batch, dim, seqlen)    io_dtype  required when z is given
 *   dA             : (dim, dstate)           fp32
 *   dB, dC         : (batch, dstate, seqlen) fp32   (sums over the channels)
 *   dD_skip        : (dim)                   fp32   nullable
 *   ddt_bias       : (dim)                   fp32   nullable
 *   d_initial_state: (batch, dim, dstate)    fp32   nullable
 *
 * ddelta is dJ/d(delta) (through the softplus when the flag is set), and
 * ddt_bias its sum over batch and time.  Sums over channels, batch and time
 * are formed from per-warp partials added in a fixed order, so results are
 * deterministic.  Scratch (about batch * dim * seqlen * dstate / 3 bytes of
 * checkpoints plus 2 * batch * dstate * seqlen * ceil(dim / 32) * 4 bytes of
 * partials, padded dstate) comes from the stream-ordered pool.  Outputs must
 * not overlap inputs or each other.
 */
int mamba_scan_bwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                   mamba_dtype_t io_dtype,
                   const void *u, const void *delta, const float *dt_bias,
                   const float *A, const void *B, const void *C,
                   const float *D_skip, const void *z, int flags,
                   const float *initial_state, const void *dy,
                   const float *d_final_state,
                   void *du, void *ddelta, float *dA, float *dB, float *dC,
                   float *dD_skip, void *dz, float *ddt_bias,
                   float *d_initial_state, cudaStream_t stream);

/*
 * A training step's pair: the forward keeps the state checkpoints that
 * mamba_scan_bwd would otherwise recompute in its first pass, and the
 * backward starts from them (the recomputation of each 12-step tile inside
 * the reverse pass is unchanged; page "Mamba: linear-time sequence modeling
 * with selective state spaces", "What they did").
 *
 * mamba_scan_checkpoint_bytes: the size of the checkpoint buffer,
 *   batch * dim * ceil(seqlen / 12) * P * 4 bytes with P = dstate padded to
 *   4, 8 or 16 (fp32 states, [batch][ceil(seqlen / 12)][P / 4][dim][4]:
 *   entry n of channel d at ((k * P / 4 + n / 4) * dim + d) * 4 + n % 4 within
 *   a batch entry); -1 for an invalid shape.  (For batch 4, dim 5120, dstate 16, seqlen 2048: 224 MB,
 *   2.7 times one bf16 (batch, dim, seqlen) tensor.)
 *
 * mamba_scan_fwd_train: y and final_state exactly as mamba_scan_fwd_ex with
 *   the same inputs and initial_state (Euler; flags: MAMBA_FLAG_SOFTPLUS
 *   only, other bits -> MAMBA_ERR_FLAGS; no per-entry lengths), and writes
 *   checkpoints (16-byte aligned, caller-owned, required when seqlen > 0):
 *   the state before step 12k for every k < ceil(seqlen / 12), the initial
 *   state (or zero) at k = 0.  Scratch as mamba_scan_fwd.  checkpoints must
 *   not overlap any input or output (MAMBA_ERR_ALIAS).
 *
 * mamba_scan_bwd_ckpt: mamba_scan_bwd with the checkpoint pass replaced by
 *   `checkpoints` from mamba_scan_fwd_train on the same inputs (the initial
 *   state is in them, so there is no initial_state argument).  Results are
 *   bit for bit those of mamba_scan_bwd.  Checkpoints from other inputs give
 *   the gradients of a different forward; nothing checks this.  Scratch:
 *   the partials of mamba_scan_bwd, no checkpoints.
 */
int64_t mamba_scan_checkpoint_bytes(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen);
int mamba_scan_fwd_train(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                         mamba_dtype_t io_dtype,
                         const void *u, const void *delta, const float *dt_bias,
                         const float *A, const void *B, const void *C,
                         const float *D_skip, const void *z, int flags,
                         const float *initial_state, void *y, float *final_state,
                         float *checkpoints, cudaStream_t stream);
int mamba_scan_bwd_ckpt(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                        mamba_dtype_t io_dtype,
                        const void *u, const void *delta, const float *dt_bias,
                        const float *A, const void *B, const void *C,
                        const float *D_skip, const void *z, int flags,
                        const float *checkpoints, const void *dy,
                        const float *d_final_state,
                        void *du, void *ddelta, float *dA, float *dB, float *dC,
                        float *dD_skip, void *dz, float *ddt_bias,
                        float *d_initial_state, cudaStream_t stream);

/*
 * Causal depthwise convolution with optional SiLU: the short convolution in
 * front of the scan in the Mamba block (paper "Mamba: linear-time sequence
 * modeling with selective state spaces", "What they did": the block merges
 * the H3 block and a gated MLP; the pages print no formula, so this is the
 * plain reading, one width-W filter per channel):
 *
 *   xp(t)      = x[b,d,t] for t >= 0, conv_state[b,d,W-1+t] for t < 0 (zero without one)
 *   out[b,d,t] = act(bias[d] + sum_{k<W} weight[d,k] * xp(t - (W-1) + k)),  act = silu or identity
 *
 *   x, out           : (batch, dim, seqlen)   io_dtype
 *   weight           : (dim, width)           fp32      1 <= width <= 8
 *   bias             : (dim)                  fp32      nullable
 *   conv_state       : (batch, dim, width-1)  io_dtype  nullable: the W-1 inputs before t = 0, oldest first
 *   final_conv_state : (batch, dim, width-1)  io_dtype  nullable: the W-1 inputs up to t = seqlen-1
 *
 * final_conv_state must not overlap conv_state (MAMBA_ERR_ALIAS): ping-pong
 * two buffers to chain pieces of a sequence.  Allocates nothing.
 */
int mamba_conv1d_fwd(int64_t batch, int64_t dim, int64_t seqlen, int width, mamba_dtype_t io_dtype,
                     const void *x, const float *weight, const float *bias,
                     const void *conv_state, int silu, void *out, void *final_conv_state,
                     cudaStream_t stream);

/*
 * One generation step of the convolution: out[b,d] from x[b,d] and the
 * row's W-1 previous inputs in conv_state (batch, dim, width-1), which is
 * then shifted by one and gets x[b,d] as its newest entry, in place.
 * Arguments as in mamba_conv1d_fwd (x, out: (batch, dim)).
 */
int mamba_conv1d_update(int64_t batch, int64_t dim, int width, mamba_dtype_t io_dtype, void *conv_state,
                        const void *x, const float *weight, const float *bias, int silu,
                        void *out, cudaStream_t stream);

/* Static, human-readable name of a mamba_status_t value. */
const char *mamba_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * words.  Returns MAMBA_OK, MAMBA_ERR_TIMEOUT (a bounded device wait gave up;
 * the affected outputs are incomplete), MAMBA_ERR_BOUNDS (debug builds only:
 * an index check failed and its access was skipped) or MAMBA_ERR_CUDA.
 */
int mamba_device_status(cudaStream_t stream);

/*
 * Debug builds.  The library built with -DMAMBA_DEBUG (libmamba_scan_debug.so
 * beside libmamba_scan.so; the Python binding loads it when the environment
 * has MAMBA_SCAN_LIBRARY=debug) checks the element index of every global
 * load and store of the scan, generation-step, B/C packing, carry and
 * convolution kernels against the extent of its buffer, and of every
 * tensor-map copy's box origin.  A failed check skips the access (a load
 * reads 0), records the source line and makes the next mamba_device_status
 * return MAMBA_ERR_BOUNDS; nothing traps.  In a release build the checks
 * compile to nothing.
 *
 * mamba_debug_build returns 1 in a debug build, 0 otherwise, and writes the
 * source line of the last failed check that mamba_device_status reported
 * (0 if none) to *last_failed_line when that is not NULL.
 * mamba_selftest_bounds launches one thread that checks an index one past
 * the end of an extent without accessing any memory: in a debug build the
 * next mamba_device_status returns MAMBA_ERR_BOUNDS, in a release build it
 * returns MAMBA_OK.
 */
int mamba_debug_build(int *last_failed_line);
int mamba_selftest_bounds(cudaStream_t stream);

/*
 * Self-test of the failure path of the bounded device waits.  Launches one
 * thread that waits on an mbarrier nothing ever completes, for limit_us
 * microseconds (1 .. 2,000,000), then records the timeout in the device error
 * word and returns, as the scan kernels do when a copy never lands.  A later
 * mamba_device_status(stream) returns MAMBA_ERR_TIMEOUT and clears the word.
 * Nothing hangs and the context stays usable.  Returns MAMBA_ERR_SHAPE for
 * a limit out of range.
 */
int mamba_selftest_wait_timeout(int64_t limit_us, cudaStream_t stream);

/* Library version as major*100 + minor. */
int mamba_version(void);

/*
 * Tuning override for experiments, process-wide, affecting later calls of
 * mamba_scan_fwd: tail = how channel tiles that do not fill a whole wave of
 * SMs are scheduled (0 automatic, 1 whole-sequence units only, 2 cut into
 * time chunks, 3 cut into time chunks whose passes run on a library-owned
 * side stream beside the whole-sequence units; mamba_scan_fwd_noalloc
 * treats 3 as 2), stages = depth of the shared-memory input ring (1..4),
 * chunks = fixed number of time chunks for every channel tile, layout =
 * how the state of a channel is split for dstate 9..16 (1 over two warps,
 * 8 entries a lane and 64 channels per CTA; 2 over four warps, 4 entries a
 * lane and 32 channels per CTA, the automatic choice).  0 restores the
 * automatic choice for that knob.  Results do not depend on these settings beyond fp32 rounding
 * order.  Returns MAMBA_ERR_SHAPE for values out of range.
 */
int mamba_scan_set_tuning(int tail, int stages, int chunks, int layout);

/*
 * Measurement support, not part of the scan: the sustained per-SM rate of
 * one kind of arithmetic, in lane operations per SM clock cycle, measured
 * with the SM cycle counter (independent of the clock frequency).  One CTA
 * per SM with warps_per_subpartition (1 to 8) warps on each of the four SM
 * sub-partitions, `chains` (1, 2, 4, 8 or 16) independent dependency
 * chains per thread, `iters` (1 .. 2^24) iterations of 16 operations per
 * chain.  kind: 0 ex2.approx, 1 lg2.approx, 2 tanh.approx, 3 packed f32x2
 * FMA (2 lane operations each), 4 fp32 FMA, 5 the scan's state update of a
 * pair of entries (2 ex2 and 4 packed multiply/FMAs, counted as 2 state
 * updates).  Writes the rate and the median CTA cycle count;
 * allocates (cudaMalloc) a small buffer per call and synchronises `stream`.
 * Returns MAMBA_ERR_SHAPE for arguments out of range.
 */
int mamba_probe_pipe_rate(int kind, int warps_per_subpartition, int chains, int64_t iters,
                          double *ops_per_clk_sm, double *cycles_median, cudaStream_t stream);

/*
 * Per-launch timing (process-wide).  After mamba_profile_begin, every kernel
 * the library launches is bracketed by two CUDA events on its stream.
 * mamba_profile_end stops recording, waits for those events and writes, for
 * each kernel kind k < nkinds, the summed device time in milliseconds
 * (total_ms[k]) and the number of launches (launches[k]).  Kinds:
 * 0 = scan, 1 = chunk summary, 2 = chunk carry, 3 = state update,
 * 4 = B/C packing (one per scan or backward call), 5 = backward checkpoint
 * pass, 6 = backward reverse pass, 7 = backward reductions (one timing for
 * the three reduction launches of a call), 8 = causal convolution, 9 =
 * backward time-chunk summaries and their carry (one timing per call).
 * Either output may be NULL.  Not meant for use during stream capture.
 */
int mamba_profile_begin(void);
int mamba_profile_end(double *total_ms, int64_t *launches, int nkinds);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_SCAN_H */
