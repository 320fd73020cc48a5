/*
 * mamba2_ssd.h -- C ABI of the deterministic Mamba2 SSD (state-space
 * duality) chunked scan for GB300 (sm_103a).
 *
 * The operation.  "Deterministic bwd kernel for mamba2" (Mamba PR #827)
 * makes the backward of the mamba2 SSD chunked scan reproducible by taking
 * the atomics out of it (section "Atomic add non-determinism") and by fixing
 * the order of every prefix sum (section "Autotuner / kernel-shape
 * non-determinism"); its per-kernel breakdown table names the steps
 * (chunk_cumsum, chunk_state_bwd_dx/_db/_ddAcs, chunk_scan_bwd_dC/_dx).  The
 * recurrence, per batch row b and head h (group g = h / (nheads/ngroups)):
 *
 *     state_t = exp(dt_t * A_h) * state_{t-1} + dt_t * x_t B_t^T   (P x N)
 *     y_t     = state_t C_t + D_h * x_t
 *
 * with state_{t-1} replaced by the initial state (or zero) where a sequence
 * starts.  mamba2_ssd_fwd computes y and the state entering every chunk;
 * mamba2_ssd_bwd computes dx, ddt, dA, dB, dC, dD (and dinit) of
 * L = sum(y * dout).
 *
 * Determinism.  Every output element has exactly one writer; partial sums
 * that several CTAs produce are parked in per-unit slots and folded in one
 * fixed order (the slot pattern of "[PyTorch] Ask cuDNN for a deterministic
 * dprob when determinism is requested", TransformerEngine PR #3407, and of
 * the split-slice reduction in xtuner PR #2235).  No atomics are used unless
 * variant SSD_VARIANT_ATOMIC is requested, which exists only to measure the
 * cost of determinism.  Results are bitwise identical across runs and across
 * every `config` index that mamba2_ssd_num_configs reports.
 *
 * Memory.  The library allocates no device memory: the caller passes every
 * input, output and workspace buffer.  All pointers below are DEVICE
 * pointers unless stated, must be 16-byte aligned and point to densely packed
 * row-major (C-contiguous) arrays of the stated shapes.  Nothing is
 * synchronised inside fwd/bwd (one documented exception: seq_idx validation
 * in fwd); work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 * default stream) and the call returns.  Buffers must stay alive until that
 * work has completed.
 *
 * Errors.  Every argument is checked on the host before anything is
 * launched; a failed check returns its status and launches nothing.  No
 * exception crosses the ABI.  SSD_ERR_CUDA reports a launch failure.
 *
 * Shapes: b = batch, T = seqlen, H = nheads, P = headdim, G = ngroups,
 * N = dstate, Q = chunk_size, nc = ceil(T / Q), nseq = number of sequences.
 */
#ifndef MAMBA2_SSD_H_
#define MAMBA2_SSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1,   /* bad shape, null pointer, misalignment, bad saved struct */
  SSD_ERR_UNSUPPORTED = 2,   /* valid but not supported (e.g. a sequence start inside a chunk) */
  SSD_ERR_WORKSPACE = 3,     /* workspace smaller than the *_workspace_size query */
  SSD_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  SSD_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out (see mamba2_ssd_bwd_check, _fwd_check) */
  SSD_ERR_HANDLE = 6         /* saved struct not produced by mamba2_ssd_fwd or dims mismatch */
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/* Backward variants.  DETERMINISTIC (the product) and ORDERED give the same
 * bits; ORDERED replaces the general path's per-head dB/dC slots by an
 * ordered-semaphore fold (the CTA of head k of a group adds its tile after
 * the CTA of head k-1 has published; the ordered accumulation of
 * "FlashAttention 2 deterministic backward"), general path only.  ATOMIC
 * exists only to measure the cost of determinism. */
typedef enum { SSD_VARIANT_DETERMINISTIC = 0, SSD_VARIANT_ATOMIC = 1, SSD_VARIANT_ORDERED = 2 } ssd_variant;

/* Valid dims (every call checks them; the size queries return 0, the counts
 * -1 or 0, the others SSD_ERR_INVALID_ARG): every size and nseq at least 1
 * (an empty problem is rejected, not treated as a no-op), nheads a multiple
 * of ngroups, chunk_size at most 1024, batch * nc * nheads below 2^31, with
 * SSD_DIMS_SEQ_IDX seqlen and nseq below 2^31, dtype an ssd_dtype, and no
 * flag bits but the SSD_DIMS_* ones (SSD_DIMS_SEQ_ANY_START only together
 * with SSD_DIMS_SEQ_IDX). */
typedef struct {
  int64_t batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size;
  int64_t nseq;       /* rows of init_states / dinit: number of sequences (= batch without seq_idx) */
  int32_t dtype;      /* ssd_dtype of x, B, C, y and dout; dt, A, D, init and all gradients are fp32 */
  int32_t flags;      /* SSD_DIMS_* bits; all others must be 0 */
} ssd_dims;

/* ssd_dims.flags: seq_idx will be passed (packed variable-length batch). */
#define SSD_DIMS_SEQ_IDX 1
/* ssd_dims.flags (with SSD_DIMS_SEQ_IDX): sequences may start anywhere, not
 * only at multiples of chunk_size.  A sequence that starts inside a chunk
 * begins from its own initial state (or zero) exactly as the recurrence
 * says; decay terms never cross a sequence start.  The fused kernels reset
 * states at chunk starts only, so these dims run them on a padded copy of the
 * problem (mamba2_ssd_padded_chunks) when they are bf16 with batch 1,
 * headdim 64, nseq - 1 <= ceil(seqlen / 128), a chunk that is a multiple of
 * 128, and either dstate 128 ("fused-padded") or one group, an even head
 * count and dstate 256 ("fused-split-padded"); seqlen need not be a multiple
 * of the chunk there.  Every other such shape runs the general CUDA-core
 * kernels. */
#define SSD_DIMS_SEQ_ANY_START 2

/* What the backward needs from the forward.  Filled by mamba2_ssd_fwd; it
 * borrows the caller's buffers (inputs and `states`), which must stay alive
 * and unmodified until the backward has run.  Plain data: copy it freely. */
typedef struct {
  ssd_dims dims;
  const void *x;              /* (b,T,H,P) dtype */
  const float *dt;            /* (b,T,H) fp32, the step after any activation */
  const float *A;             /* (H) fp32, A < 0 expected */
  const void *B, *C;          /* (b,T,G,N) dtype; head h uses group h / (H/G) */
  const float *D;             /* (H) fp32 skip weight */
  const int32_t *seq_idx;     /* (b,T) int32 or NULL */
  const float *init_states;   /* (nseq,H,P,N) fp32 or NULL */
  const float *states;        /* (b,nc,H,P,N) states entering each chunk (packed on the fused shapes;
                                 see mamba2_ssd_fwd and mamba2_ssd_states_unpack) */
  const float *aux;           /* dstate-256 fused shapes: the packed states of both state halves, inside
                                 the forward's workspace; "fused-chunk128" shapes: the packed states of
                                 every 128 tokens, inside the forward's workspace; "-padded" shapes: the
                                 forward's workspace itself
                                 (the padded problem); either must then stay alive and unmodified until
                                 the backward has run; NULL otherwise */
  uint32_t magic;
  uint32_t flags;
} ssd_saved;

/* Human-readable name of a status code (static string, never NULL). */
const char *mamba2_ssd_status_string(int status);

/* Number of chunks nc = ceil(seqlen / chunk_size), or -1 for invalid dims. */
int64_t mamba2_ssd_num_chunks(const ssd_dims *dims);

/* Workspace bytes the forward needs (0 if dims are invalid). */
size_t mamba2_ssd_fwd_workspace_size(const ssd_dims *dims);

/* Workspace bytes the backward needs for launch configuration `config`
 * (0 <= config < mamba2_ssd_num_configs) and `variant` (0 if invalid). */
size_t mamba2_ssd_bwd_workspace_size(const ssd_dims *dims, int config, int variant);

/* Number of selectable launch configurations for these dims (>= 1, or 0 if
 * the dims are invalid).  All configurations give bitwise-identical
 * results; they differ in launch shape and scheduling only.  bf16 problems
 * with headdim 64, seqlen a multiple of the chunk, and either chunk 128 and
 * dstate 128 ("fused/...") or one group, an even number of heads, chunk 128
 * or 256 and dstate 256
 * ("fused-split/...": the recurrence never mixes state dimensions, so the
 * fused kernels run once per 128-wide state half, in 128-token chunks, and
 * the halves' contributions are summed in a fixed order) run the fused
 * tensor-core forward and backward (with SSD_DIMS_SEQ_ANY_START set, the
 * "-padded" forms of both, see there).  bf16, headdim 64, dstate 128 and a
 * chunk that is a larger multiple of 128 (256, as in Mamba2's defaults), with
 * seqlen a multiple of 128 ("fused-chunk128/..."), run the same fused kernels
 * in 128-token chunks: y, every gradient and the state entering each chunk
 * are those of the recurrence whatever the chunk length.  Every other shape
 * runs the general CUDA-core forward and backward. */
int mamba2_ssd_num_configs(const ssd_dims *dims);

/* Name of the backward algorithm a configuration selects (static string). */
const char *mamba2_ssd_config_name(const ssd_dims *dims, int config);

/* Number of kernel launches one mamba2_ssd_bwd call enqueues (this
 * library's kernels; stream-ordered memsets are not counted). */
int mamba2_ssd_bwd_num_launches(const ssd_dims *dims, int config, int variant);

/* Name of the k-th kernel launch of mamba2_ssd_bwd (static string;
 * "invalid" when k is out of range). */
const char *mamba2_ssd_bwd_launch_name(const ssd_dims *dims, int config, int variant, int k);

/* Forward.  Inputs x, dt, A, B, C, D as in ssd_saved; seq_idx (b,T) int32
 * (nullable, and given exactly when dims->flags has SSD_DIMS_SEQ_IDX;
 * requires batch == 1, seqlen and nseq below 2^31, non-decreasing ids in
 * [0,nseq) -- else SSD_ERR_INVALID_ARG -- and, unless dims->flags has
 * SSD_DIMS_SEQ_ANY_START, every change of id at a multiple of chunk_size --
 * else SSD_ERR_UNSUPPORTED; checked with one synchronous device-to-host copy
 * of seq_idx, the only synchronisation in this library);
 * init_states (nseq,H,P,N) fp32 (nullable: zero initial states).
 * Outputs: y (b,T,H,P) in dtype; states: b*nc*H*P*N fp32-sized elements
 * holding the state entering each chunk (init/zero at a sequence start), the
 * (P,N) fp32 tile of (b,c,h) at element offset ((b*nc+c)*H+h)*P*N.  On the
 * shapes that run the fused backward (mamba2_ssd_config_name "fused/...")
 * each tile is stored packed instead, in the same 32 KB: the bf16 pair
 * hi = round(S), lo = round(S - hi) as two [N][P] tiles in the 128-byte
 * swizzled tensor-core operand layout (row n at n*128 bytes, its 16-byte
 * chunk j at position j ^ (n % 8)), hi first -- the operand the fused
 * backward copies straight into shared memory.  mamba2_ssd_states_unpack
 * gives the fp32 (b,nc,H,P,N) view of either form.  On the "fused-split",
 * "fused-chunk128" and "-padded" shapes `states` holds the fp32 states
 * themselves and the packed ones (and, padded, the padded copies of x, dt, B,
 * C and seq_idx)
 * stay in the workspace, which must then live, unmodified, until the backward
 * (ssd_saved.aux).  *saved_out (host struct) filled for the backward.
 * workspace: >= fwd_workspace_size bytes. */
ssd_status mamba2_ssd_fwd(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                          const void *B, const void *C, const float *D, const int32_t *seq_idx,
                          const float *init_states, void *y, float *states, void *workspace,
                          size_t workspace_bytes, void *stream, ssd_saved *saved_out);

/* The padded form that runs packed batches whose sequences start inside a
 * chunk on the fused kernels ("fused-padded/..." and "fused-split-padded/..."
 * configurations; see SSD_DIMS_SEQ_ANY_START): the token stream is cut at
 * every sequence start and every multiple of 128 tokens, and piece k becomes
 * chunk k of a padded problem in 128-token chunks, its tokens first, then
 * tokens with dt = 0 and x = B = C = dout = 0, which leave the state and
 * every gradient of the real tokens unchanged.  The padded problem has
 * ceil(seqlen / 128) + nseq - 1 chunks (trailing ones all padding, inside the
 * last sequence); this returns that count, or 0 for dims that do not run the
 * padded form. */
int64_t mamba2_ssd_padded_chunks(const ssd_dims *dims);

/* The piece table of the padded form for a HOST copy of seq_idx (seqlen
 * int32), written to host `table` (3 * padded_chunks + num_chunks int32):
 * start[k], len[k] (0..128) and id[k] of every padded chunk k -- its first
 * token, its count of real tokens and its sequence id -- then, for every
 * chunk c of the caller's chunking, the padded chunk that begins with token
 * c * chunk_size.  Host code only (the forward builds the same table from its
 * own copy of seq_idx).  SSD_ERR_INVALID_ARG for dims that do not run the
 * padded form, null pointers, or ids that are negative, >= nseq or
 * decreasing. */
ssd_status mamba2_ssd_padded_piece_table(const ssd_dims *dims, const int32_t *seq_idx, int32_t *table);

/* Status of the last forward that used this workspace: reads one word
 * written by the device (synchronises `stream`).  SSD_ERR_TIMEOUT when a
 * bounded device-side wait of the tensor-core forward ran out (its outputs
 * are then invalid), SSD_OK otherwise (always for the general forward, which
 * has no device-side waits); SSD_ERR_INVALID_ARG for invalid dims or a null
 * workspace. */
ssd_status mamba2_ssd_fwd_check(const ssd_dims *dims, const void *workspace, void *stream);

/* fp32 (b,nc,H,P,N) copy of the saved chunk states (hi + lo of the packed
 * form on the fused shapes, the states themselves otherwise) into `out`
 * (device, 16-byte aligned), enqueued on `stream`. */
ssd_status mamba2_ssd_states_unpack(const ssd_saved *saved, float *out, void *stream);

/* Backward of L = sum(y * dout).  dout (b,T,H,P) in dtype.  Outputs, all
 * fp32 and fully overwritten: dx (b,T,H,P), ddt (b,T,H), dA (H), dB, dC
 * (b,T,G,N), dD (H), dinit (nseq,H,P,N; may be NULL; must be NULL when the
 * forward had no init_states).  workspace: >= bwd_workspace_size(config,
 * variant) bytes.  variant: SSD_VARIANT_DETERMINISTIC (the product),
 * SSD_VARIANT_ORDERED (general path only, else SSD_ERR_UNSUPPORTED; same
 * bits; dstate <= 512) or SSD_VARIANT_ATOMIC (same kernels with atomic
 * accumulation; for measuring the cost of determinism only, results not
 * reproducible). */
ssd_status mamba2_ssd_bwd(const ssd_saved *saved, const void *dout, float *dx, float *ddt, float *dA,
                          float *dB, float *dC, float *dD, float *dinit, void *workspace,
                          size_t workspace_bytes, int config, int variant, void *stream);

/* Status of the last backward that used this workspace: reads one word
 * written by the device (synchronises `stream`).  SSD_ERR_TIMEOUT when a
 * bounded device-side wait ran out (the fused backward's chain, or the
 * ORDERED variant's semaphore), SSD_ERR_UNSUPPORTED
 * when the fused kernel found its dynamic shared memory not 1 KB aligned and
 * did no work (outputs invalid in both cases), SSD_OK otherwise. */
ssd_status mamba2_ssd_bwd_check(const ssd_dims *dims, int config, const void *workspace, void *stream);

/* Fault-injection diagnostic of the fused backward (fused shapes only): the
 * units of chunk `silent_chunk` never publish their state gradient, and
 * every wait for it gives up after `spin_limit` polls, so the consumer of
 * that chunk times out.  Nothing hangs or faults; the call returns SSD_OK
 * and mamba2_ssd_bwd_check then reports SSD_ERR_TIMEOUT.  Same arguments as
 * mamba2_ssd_bwd otherwise (config and variant 0). */
ssd_status mamba2_ssd_bwd_fault_test(const ssd_saved *saved, const void *dout, float *dx, float *ddt, float *dA,
                                     float *dB, float *dC, float *dD, float *dinit, void *workspace,
                                     size_t workspace_bytes, int64_t silent_chunk, uint32_t spin_limit,
                                     void *stream);

/* mamba2_ssd_bwd with a per-launch timing trace, for profiling: `events`
 * holds num_events caller-created cudaEvent_t handles; events[2k] and
 * events[2k+1] are recorded on `stream` immediately before and after launch
 * k (k < num_launches; extra events are left alone, missing ones skipped).
 * The computation and its result are exactly those of mamba2_ssd_bwd. */
ssd_status mamba2_ssd_bwd_traced(const ssd_saved *saved, const void *dout, float *dx, float *ddt, float *dA,
                                 float *dB, float *dC, float *dD, float *dinit, void *workspace,
                                 size_t workspace_bytes, int config, int variant, void *stream,
                                 void *const *events, int num_events);

/* Diagnostic: one 128 x N x K bf16 product on the tensor cores through the
 * same shared-memory descriptors, TMEM accumulator and (optionally) TMA
 * loads that the fused backward uses.  A and B are device bf16 arrays in
 * storage order: A is [M][K] (a_mn = 0, K-major) or [K][M] (a_mn = 1,
 * MN-major); B is [N][K] (b_mn = 0) or [K][N] (b_mn = 1).  D (device fp32,
 * [M][N]) receives A*B.  M must be 128, N 64 or 128, K 64 or 128.  Enqueued
 * on `stream`; a NaN in D[0] reports a bounded wait that ran out. */
ssd_status mamba2_ssd_selftest_umma(const void *A, const void *B, float *D, int M, int N, int K, int a_mn,
                                    int b_mn, int use_tma, void *stream);

/* Backward for callers that cannot allocate device memory (no counterpart in
 * the pages this library follows; it only changes where the scratch lives).
 * Callers that run inside a fixed, pre-sized memory arena, or inside a host
 * that forbids allocation after start-up, cannot hand mamba2_ssd_bwd a
 * workspace.  This entry point takes the same saved struct, dout and outputs
 * as mamba2_ssd_bwd (deterministic variant) but uses a fixed array of
 * mamba2_ssd_static_scratch_bytes() bytes in device global memory, built
 * into the library, as its workspace; it calls no allocating routine.
 * - Shapes whose workspace (mamba2_ssd_bwd_workspace_size) exceeds that size
 *   are rejected with SSD_ERR_WORKSPACE before anything is launched.
 * - The first call on a device (with that device current) looks the array's
 *   address up once; make that first call before any stream capture.
 * - Every call on a device shares the one array: calls whose work may
 *   overlap on the GPU (unordered streams) race and must not be made.
 * - Every GPU that loads the library holds the array until the process exits.
 * Results are bitwise identical to mamba2_ssd_bwd with the same config. */
size_t mamba2_ssd_static_scratch_bytes(void);
ssd_status mamba2_ssd_bwd_static_scratch(const ssd_saved *saved, const void *dout, float *dx, float *ddt,
                                         float *dA, float *dB, float *dC, float *dD, float *dinit, int config,
                                         void *stream);

/* Status of the last mamba2_ssd_bwd_static_scratch call on the current
 * device: the counterpart of mamba2_ssd_bwd_check for callers that never see
 * the workspace (the device status word sits at the start of the static
 * array).  Same results and synchronisation as mamba2_ssd_bwd_check: reads
 * one word after synchronising `stream`; SSD_ERR_TIMEOUT or
 * SSD_ERR_UNSUPPORTED mean the gradients of that call are invalid.  dims and
 * config must be those of the call being checked.  The cached address of the
 * array is only valid in the device context it was looked up in: after
 * cudaDeviceReset neither static-scratch entry point may be called again. */
ssd_status mamba2_ssd_static_scratch_check(const ssd_dims *dims, int config, void *stream);

/* ---- Steps either side of the scan ------------------------------------
 * The step-size preprocessing that Mamba2 folds into its chunk_cumsum (whose
 * backward "Deterministic bwd kernel for mamba2" lists as chunk_cumsum_bwd)
 * and the z-gate on the scan's output.  Elementwise; all pointers are device
 * pointers, 16-byte aligned, densely packed; enqueued on `stream`; nothing is
 * synchronised.  A count of 0 launches nothing and returns SSD_OK. */

/* dt[r,h] = clamp(sp(dt_raw[r,h] + dt_bias[h]), dt_min, dt_max) for r < rows
 * (rows = batch * seqlen, layout (rows, nheads) fp32), sp(v) = log(1 + e^v)
 * when use_softplus != 0, else sp(v) = v.  dt_bias (nheads) may be NULL
 * (zero).  dt_min <= dt_max, neither NaN (pass 0 and INFINITY, or -INFINITY
 * and INFINITY, for no clamp); rows < 2^36. */
ssd_status mamba2_ssd_dt_fwd(int64_t rows, int64_t nheads, const float *dt_raw, const float *dt_bias,
                             int use_softplus, float dt_min, float dt_max, float *dt, void *stream);

/* Workspace bytes of mamba2_ssd_dt_bwd (0 for invalid sizes). */
size_t mamba2_ssd_dt_bwd_workspace_size(int64_t rows, int64_t nheads);

/* Backward of mamba2_ssd_dt_fwd given ddt = dL/d dt (rows, nheads) fp32:
 * ddt_raw = ddt * sp'(v) where dt_min <= sp(v) <= dt_max, else 0
 * (v = dt_raw + dt_bias, sp' the logistic function or 1); ddt_bias[h] (may
 * be NULL) = sum over rows of ddt_raw[., h], computed over 32 fixed slabs of
 * rows folded in ascending order, so bitwise reproducible.  workspace (only
 * needed with ddt_bias) >= mamba2_ssd_dt_bwd_workspace_size bytes. */
ssd_status mamba2_ssd_dt_bwd(int64_t rows, int64_t nheads, const float *dt_raw, const float *dt_bias,
                             int use_softplus, float dt_min, float dt_max, const float *ddt, float *ddt_raw,
                             float *ddt_bias, void *workspace, size_t workspace_bytes, void *stream);

/* out = y * silu(z), silu(z) = z / (1 + e^-z); y, z, out: n elements of
 * `dtype` (ssd_dtype; fp32 arithmetic, out rounded once). */
ssd_status mamba2_ssd_gate_fwd(int64_t n, int32_t dtype, const void *y, const void *z, void *out, void *stream);

/* Backward of the gate given dout (n elements of `dtype`): dy = dout *
 * silu(z) in `dtype` (ready as the scan's dout), dz = dout * y * silu'(z) in
 * fp32, silu'(z) = s (1 + z (1 - s)), s = 1 / (1 + e^-z). */
ssd_status mamba2_ssd_gate_bwd(int64_t n, int32_t dtype, const void *y, const void *z, const void *dout, void *dy,
                               float *dz, void *stream);

/* ---- Causal depthwise conv1d before the scan ---------------------------
 * "Deterministic bwd kernel for mamba2" (Mamba PR #827), section "Atomic add
 * non-determinism", names the atomics of causal-conv1d next to the SSD
 * backward's.  Per batch row b, token t, channel c (x, y, dy laid out
 * (batch, seqlen, channels), densely packed):
 *     pre[b,t,c] = bias[c] + sum_{k<width} weight[c,k] x[b, t-width+1+k, c]
 *     y = pre (activation 0) or silu(pre) = pre / (1 + e^-pre) (activation 1)
 * where a tap before the row start reads zero and, when seq_idx (batch,
 * seqlen) int32 is given (batch 1, non-decreasing ids), a tap in another
 * sequence than t reads zero.  Sizes: channels a multiple of 4, width 1..4,
 * batch * ceil(seqlen / 128) <= 65535.  weight (channels, width) and bias
 * (channels, may be NULL) fp32; x, y, dy in `dtype` (ssd_dtype); dx, dweight,
 * dbias fp32.  All pointers device, 16-byte aligned.  config in
 * [0, mamba2_ssd_conv1d_num_configs()) picks the block size only: every
 * config gives the same bits.  Enqueued on `stream`; a bad size, pointer or
 * config returns SSD_ERR_INVALID_ARG and launches nothing. */
int mamba2_ssd_conv1d_num_configs(void);
ssd_status mamba2_ssd_conv1d_fwd(int64_t batch, int64_t seqlen, int64_t channels, int32_t width, int32_t dtype,
                                 int32_t activation, const void *x, const float *weight, const float *bias,
                                 const int32_t *seq_idx, void *y, int config, void *stream);

/* Workspace bytes of the deterministic conv1d backward (0 for bad sizes):
 * one slot of (width + 1) x channels partial sums per 128-token tile. */
size_t mamba2_ssd_conv1d_bwd_workspace_size(int64_t batch, int64_t seqlen, int64_t channels, int32_t width);

/* Backward of L = sum(y * dy): dx (batch, seqlen, channels), dweight
 * (channels, width), dbias (channels; may be NULL), all fully overwritten.
 * dweight and dbias sum over every token: each 128-token tile's partial sums
 * (in token order) go to its own slot of the workspace and are folded in
 * ascending tile order -- bitwise reproducible for every run and config.
 * variant SSD_VARIANT_ATOMIC adds the partial sums with atomics instead (no
 * workspace needed; results not reproducible; for measuring the cost of
 * determinism only). */
ssd_status mamba2_ssd_conv1d_bwd(int64_t batch, int64_t seqlen, int64_t channels, int32_t width, int32_t dtype,
                                 int32_t activation, const void *x, const float *weight, const float *bias,
                                 const int32_t *seq_idx, const void *dy, float *dx, float *dweight, float *dbias,
                                 void *workspace, size_t workspace_bytes, int config, int variant, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA2_SSD_H_ */
