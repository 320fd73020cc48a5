// ssd_simt.cu -- general CUDA-core path of the Mamba2 SSD forward and
// backward (any shape, fp32 or bf16 inputs, sequence starts anywhere).
//
// Each kernel is one step of the chunked algorithm whose backward "Deterministic
// bwd kernel for mamba2" (Mamba PR #827) breaks down per kernel:
// chunk_cumsum, chunk_state, state passing, chunk_scan and their backward
// counterparts.  Every output element is produced by exactly one thread that
// sums its terms sequentially in a fixed order, so the result does not depend
// on the block size (the launch configuration) or on scheduling.  Per-head
// contributions to the group-shared dB/dC, and per-chunk contributions to dA
// and dD, are parked in slots and folded in ascending slot order by the
// reduction kernels at the end (unless the atomic variant is requested).
// The ordered variant folds dB/dC without slots instead: the CTA of head k
// adds its tile into dB/dC only after the CTA of head k-1 of the same group
// has published its own (a semaphore per tile, as in the ordered dQ
// accumulation of "FlashAttention 2 deterministic backward"), so each
// element is summed over heads in the same ascending order as the slot fold
// and the bits are identical.
//
// Notation per (batch b, chunk c, head h): local token i in [0, Lc), Lc the
// chunk's length; Acs_i the in-chunk inclusive prefix sum of dt*A (hi+lo);
// E = Acs_{Lc-1}; g = dout.  States are (P, N), n fastest.
//
// Packed variable-length batches (seq_idx, batch row 0 only) may start a
// sequence inside a chunk.  A token then sees the state entering the chunk
// only if its sequence entered the chunk from the previous one (or starts at
// the chunk's first token, where that state is the initial one); a sequence
// that starts at local position f >= 1 begins from its own initial state (or
// zero), decayed from just before f, i.e. by exp(Acs_i - Acs_{f-1}).  Decay
// terms between tokens of different sequences are zero, and only the
// sequence holding the chunk's last token reaches the chunk-end state.  With
// chunk-aligned starts every mask below is a no-op.
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {

namespace {

constexpr int kPassThreads = 256;

__host__ __device__ inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// first[s] = first token of sequence s (batch row 0); one writer per entry
// (the token where the id changes); entries of ids with no token keep the
// -1 of the preceding memset.
__global__ void seq_first_kernel(int64_t T, const int32_t *__restrict__ seq_idx, int32_t *__restrict__ first) {
  const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= T) return;
  if (t == 0 || seq_idx[t] != seq_idx[t - 1]) first[seq_idx[t]] = int32_t(t);
}

// Local position at which the sequence holding token t started inside the
// chunk beginning at t0, or 0 when it entered the chunk from the previous one
// or starts at t0 (it then sees the state entering the chunk).
__device__ __forceinline__ int64_t local_start(const int32_t *seq_idx, const int32_t *first, int64_t bi,
                                               int64_t T, int64_t t, int64_t t0) {
  if (seq_idx == nullptr) return 0;
  const int64_t f = int64_t(first[seq_idx[bi * T + t]]) - t0;
  return f > 0 ? f : 0;
}

// ---------------------------------------------------------------- cumsum --
// Acs (b,H,nc,Q) as hi + lo: left-to-right compensated (two-sum) prefix sum
// of a_i = dt_i * A_h, one thread per (b, c, h), entries past the chunk end
// padded with the last value.  One fixed order for every launch shape.
__global__ void cumsum_fwd_kernel(Shape s, const float *__restrict__ dt, const float *__restrict__ A,
                                  float *__restrict__ acs_hi, float *__restrict__ acs_lo) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= s.b * s.nc * s.H) return;
  const int64_t h = idx % s.H, c = (idx / s.H) % s.nc, bi = idx / (s.H * s.nc);
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
  const float Ah = A[h];
  float hi = 0.f, lo = 0.f;
  float *oh = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  float *ol = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  for (int64_t i = 0; i < s.Q; ++i) {
    if (i < Lc) {
      const float a = __fmul_rn(dt[(bi * s.T + t0 + i) * s.H + h], Ah);
      const float sum = __fadd_rn(hi, a);
      const float bb = __fsub_rn(sum, hi);
      const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(sum, bb)), __fsub_rn(a, bb));
      hi = sum;
      lo = __fadd_rn(lo, err);
    }
    oh[i] = hi;
    ol[i] = lo;
  }
}

// ------------------------------------------------------ chunk_state (fwd) --
// S[b,c,h,p,n] = sum_i exp(E - Acs_i) dt_i x_i[p] B_i[n] over the tokens of
// the sequence holding the chunk's last token (i >= fe); one thread per (p,n).
template <class TIn>
__global__ void chunk_state_fwd_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ Bm,
                                       const float *__restrict__ dt, const float *__restrict__ acs_hi,
                                       const float *__restrict__ acs_lo, const int32_t *__restrict__ seq_idx,
                                       const int32_t *__restrict__ first, float *__restrict__ S) {
  extern __shared__ float w[];
  const int64_t unit = blockIdx.x;  // (b, c, h)
  const int64_t h = unit % s.H, c = (unit / s.H) % s.nc, bi = unit / (s.H * s.nc);
  const int64_t g = h / s.hpg, t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
  const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  for (int64_t i = threadIdx.x; i < Lc; i += blockDim.x)
    w[i] = i < fe ? 0.f
                  : __fmul_rn(expf(acs_diff(ah[Lc - 1], al[Lc - 1], ah[i], al[i])), dt[(bi * s.T + t0 + i) * s.H + h]);
  __syncthreads();
  const int64_t e = int64_t(blockIdx.y) * blockDim.x + threadIdx.x;
  if (e >= s.P * s.N) return;
  const int64_t p = e / s.N, n = e % s.N;
  float acc = 0.f;
  for (int64_t i = 0; i < Lc; ++i) {
    const int64_t t = t0 + i;
    acc = fmaf(w[i] * ld(x + ((bi * s.T + t) * s.H + h) * s.P + p), ld(Bm + ((bi * s.T + t) * s.G + g) * s.N + n), acc);
  }
  S[(((bi * s.nc + c) * s.H + h) * s.P + p) * s.N + n] = acc;
}

// ------------------------------------------------ state passing (fwd) --
// states[b,c] = state entering chunk c: init/zero where chunk c starts a
// sequence, else (carried part) + S[b,c-1], the carried part being
// exp(E_{c-1}) states[b,c-1], or exp(E_{c-1} - Acs_{fe-1}) init[seq] when the
// sequence holding chunk c-1's last token started inside it at fe >= 1.
// One thread per (b,h,e).
__global__ void state_passing_fwd_kernel(Shape s, const float *__restrict__ S, const float *__restrict__ acs_hi,
                                         const float *__restrict__ acs_lo, const int32_t *__restrict__ seq_idx,
                                         const int32_t *__restrict__ first, const float *__restrict__ init,
                                         float *__restrict__ states) {
  const int64_t PN = s.P * s.N;
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= s.b * s.H * PN) return;
  const int64_t e = idx % PN, h = (idx / PN) % s.H, bi = idx / (PN * s.H);
  float run = 0.f;
  for (int64_t c = 0; c < s.nc; ++c) {
    const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
    if (is_seq_start(seq_idx, bi, s.T, t0))
      run = init ? init[(seq_of(seq_idx, bi, s.T, t0) * s.H + h) * PN + e] : 0.f;
    const int64_t o = ((bi * s.nc + c) * s.H + h) * PN + e;
    states[o] = run;
    const int64_t q0 = ((bi * s.H + h) * s.nc + c) * s.Q, q = q0 + (s.Q - 1);
    const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
    if (fe == 0) {
      run = fmaf(expf(__fadd_rn(acs_hi[q], acs_lo[q])), run, S[o]);
    } else {
      const float in = init ? init[(seq_of(seq_idx, bi, s.T, t0 + Lc - 1) * s.H + h) * PN + e] : 0.f;
      run = fmaf(expf(acs_diff(acs_hi[q], acs_lo[q], acs_hi[q0 + fe - 1], acs_lo[q0 + fe - 1])), in, S[o]);
    }
  }
}

// -------------------------------------------------------------- C . B^T --
// CB[b,c,g,i,j] = C_i . B_j for j <= i < Lc, else 0.  One thread per (i,j).
template <class TIn>
__global__ void cb_kernel(Shape s, const TIn *__restrict__ Bm, const TIn *__restrict__ Cm, float *__restrict__ CB) {
  const int64_t unit = blockIdx.x;  // (b, c, g)
  const int64_t g = unit % s.G, c = (unit / s.G) % s.nc, bi = unit / (s.G * s.nc);
  const int64_t e = int64_t(blockIdx.y) * blockDim.x + threadIdx.x;
  if (e >= s.Q * s.Q) return;
  const int64_t i = e / s.Q, j = e % s.Q;
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
  float acc = 0.f;
  if (j <= i && i < Lc) {
    const TIn *ci = Cm + ((bi * s.T + t0 + i) * s.G + g) * s.N;
    const TIn *bj = Bm + ((bi * s.T + t0 + j) * s.G + g) * s.N;
    for (int64_t n = 0; n < s.N; ++n) acc = fmaf(ld(ci + n), ld(bj + n), acc);
  }
  CB[((bi * s.nc + c) * s.G + g) * s.Q * s.Q + e] = acc;
}

// ------------------------------------------------------- chunk_scan (fwd) --
// y_i[p] = sum_{f<=j<=i} CB[i,j] exp(Acs_i - Acs_j) dt_j x_j[p]
//        + din_i sum_n Hin[p,n] C_i[n] + D x_i[p], f = local_start(i): Hin = states
// and din_i = exp(Acs_i) when f = 0, else Hin = init[seq] (or 0) and
// din_i = exp(Acs_i - Acs_{f-1}).  One thread per (b,t,h,p).
template <class TIn>
__global__ void chunk_scan_fwd_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ Cm,
                                      const float *__restrict__ dt, const float *__restrict__ D,
                                      const float *__restrict__ CB, const float *__restrict__ acs_hi,
                                      const float *__restrict__ acs_lo, const float *__restrict__ states,
                                      const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first,
                                      const float *__restrict__ init, TIn *__restrict__ y) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= s.b * s.T * s.H * s.P) return;
  const int64_t p = idx % s.P, h = (idx / s.P) % s.H, t = (idx / (s.P * s.H)) % s.T, bi = idx / (s.P * s.H * s.T);
  const int64_t c = t / s.Q, i = t % s.Q, t0 = c * s.Q, g = h / s.hpg;
  const int64_t f = local_start(seq_idx, first, bi, s.T, t, t0);
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *cb = CB + (((bi * s.nc + c) * s.G + g) * s.Q + i) * s.Q;
  float acc = 0.f;
  for (int64_t j = f; j <= i; ++j) {
    const float wgt = cb[j] * expf(acs_diff(ah[i], al[i], ah[j], al[j])) * dt[(bi * s.T + t0 + j) * s.H + h];
    acc = fmaf(wgt, ld(x + ((bi * s.T + t0 + j) * s.H + h) * s.P + p), acc);
  }
  const float *hs = f == 0 ? states + (((bi * s.nc + c) * s.H + h) * s.P + p) * s.N
                           : (init ? init + ((seq_of(seq_idx, bi, s.T, t) * s.H + h) * s.P + p) * s.N : nullptr);
  const TIn *ci = Cm + ((bi * s.T + t) * s.G + g) * s.N;
  float inter = 0.f;
  if (hs)
    for (int64_t n = 0; n < s.N; ++n) inter = fmaf(hs[n], ld(ci + n), inter);
  const float din = expf(f == 0 ? __fadd_rn(ah[i], al[i]) : acs_diff(ah[i], al[i], ah[f - 1], al[f - 1]));
  const float xv = ld(x + idx);
  const float out = fmaf(din, inter, acc) + D[h] * xv;
  st(y + idx, out);
}

// ============================================================ backward ====

// Per (b,c,h,i,j) with local_start(i) <= j <= i < Lc (same sequence):
// L = exp(Acs_i - Acs_j), Gx = g_i . x_j, M = CB[i,j] L, W = L Gx dt_j,
// MG = M Gx; zero elsewhere.
template <class TIn>
__global__ void mwg_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ dout,
                           const float *__restrict__ dt, const float *__restrict__ CB,
                           const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
                           const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first,
                           float *__restrict__ Mm, float *__restrict__ Wm, float *__restrict__ MGm) {
  const int64_t unit = blockIdx.x;  // (b, c, h)
  const int64_t h = unit % s.H, c = (unit / s.H) % s.nc, bi = unit / (s.H * s.nc);
  const int64_t e = int64_t(blockIdx.y) * blockDim.x + threadIdx.x;
  if (e >= s.Q * s.Q) return;
  const int64_t i = e / s.Q, j = e % s.Q;
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0), g = h / s.hpg;
  float M = 0.f, W = 0.f, MG = 0.f;
  if (j <= i && i < Lc && j >= local_start(seq_idx, first, bi, s.T, t0 + i, t0)) {
    const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
    const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
    const float L = expf(acs_diff(ah[i], al[i], ah[j], al[j]));
    const TIn *gi = dout + ((bi * s.T + t0 + i) * s.H + h) * s.P;
    const TIn *xj = x + ((bi * s.T + t0 + j) * s.H + h) * s.P;
    float gx = 0.f;
    for (int64_t p = 0; p < s.P; ++p) gx = fmaf(ld(gi + p), ld(xj + p), gx);
    const float cbv = CB[(((bi * s.nc + c) * s.G + g) * s.Q + i) * s.Q + j];
    M = cbv * L;
    W = L * gx * dt[(bi * s.T + t0 + j) * s.H + h];
    MG = M * gx;
  }
  const int64_t o = unit * s.Q * s.Q + e;
  Mm[o] = M;
  Wm[o] = W;
  MGm[o] = MG;
}

// dHscan[b,c,h,p,n] = sum_i exp(Acs_i) g_i[p] C_i[n] over the tokens that see
// the state entering the chunk (local_start(i) == 0); one thread per (p,n).
template <class TIn>
__global__ void dhscan_kernel(Shape s, const TIn *__restrict__ dout, const TIn *__restrict__ Cm,
                              const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
                              const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first,
                              float *__restrict__ dH) {
  extern __shared__ float ea[];
  const int64_t unit = blockIdx.x;  // (b, c, h)
  const int64_t h = unit % s.H, c = (unit / s.H) % s.nc, bi = unit / (s.H * s.nc);
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0), g = h / s.hpg;
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  for (int64_t i = threadIdx.x; i < Lc; i += blockDim.x)
    ea[i] = local_start(seq_idx, first, bi, s.T, t0 + i, t0) == 0 ? expf(__fadd_rn(ah[i], al[i])) : 0.f;
  __syncthreads();
  const int64_t e = int64_t(blockIdx.y) * blockDim.x + threadIdx.x;
  if (e >= s.P * s.N) return;
  const int64_t p = e / s.N, n = e % s.N;
  float acc = 0.f;
  for (int64_t i = 0; i < Lc; ++i) {
    const int64_t t = t0 + i;
    acc = fmaf(ea[i] * ld(dout + ((bi * s.T + t) * s.H + h) * s.P + p), ld(Cm + ((bi * s.T + t) * s.G + g) * s.N + n), acc);
  }
  dH[(((bi * s.nc + c) * s.H + h) * s.P + p) * s.N + n] = acc;
}

// Fixed-shape block sum: each warp folds by xor-shuffle, then warp sums are
// added in warp order by thread 0.  Same tree for every call.
__device__ float block_sum(float v, float *red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float tot = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < int(blockDim.x >> 5); ++w) tot += red[w];
  return tot;  // valid in thread 0
}

// Reverse state passing, one CTA per (b,h), in place on buf:
//   in:  buf[c] = dHscan_c;  out: buf[c] = dS_c = gradient reaching the end
//   state of chunk c (dH_{c+1}, or 0 where chunk c+1 starts a sequence);
//   dH_c = dHscan_c + exp(E_c) dS_c when the sequence holding the chunk's
//   last token entered the chunk (fe = 0), else dH_c = dHscan_c;
//   dEpass[b,h,c] = exp(E_c) <states_c, dS_c> (fe = 0), or
//   exp(E_c - Acs_{fe-1}) <init[seq], dS_c> (fe >= 1: the carried part of the
//   chunk-end state then starts from that sequence's initial state);
//   dinit[seq] += dH_c where chunk c starts a sequence at its first token.
__global__ void state_passing_bwd_kernel(Shape s, float *__restrict__ buf, float *__restrict__ carry,
                                         const float *__restrict__ states, const float *__restrict__ acs_hi,
                                         const float *__restrict__ acs_lo, const int32_t *__restrict__ seq_idx,
                                         const int32_t *__restrict__ first, const float *__restrict__ init,
                                         float *__restrict__ dEpass, float *__restrict__ dinit) {
  __shared__ float red[32];
  const int64_t h = blockIdx.x % s.H, bi = blockIdx.x / s.H;
  const int64_t PN = s.P * s.N;
  float *cr = carry + (bi * s.H + h) * PN;
  for (int64_t c = s.nc - 1; c >= 0; --c) {
    const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
    const bool nxt_start = (c + 1 >= s.nc) || is_seq_start(seq_idx, bi, s.T, (c + 1) * s.Q);
    const bool here_start = is_seq_start(seq_idx, bi, s.T, t0);
    const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
    const int64_t q0 = ((bi * s.H + h) * s.nc + c) * s.Q, q = q0 + (s.Q - 1);
    const float eE = expf(__fadd_rn(acs_hi[q], acs_lo[q]));
    const float eIn = fe == 0 ? eE : expf(acs_diff(acs_hi[q], acs_lo[q], acs_hi[q0 + fe - 1], acs_lo[q0 + fe - 1]));
    const float eCarry = fe == 0 ? eE : 0.f;
    float *bc = buf + ((bi * s.nc + c) * s.H + h) * PN;
    const float *hin = fe == 0 ? states + ((bi * s.nc + c) * s.H + h) * PN
                               : (init ? init + (seq_of(seq_idx, bi, s.T, t0 + Lc - 1) * s.H + h) * PN : nullptr);
    float *di = (here_start && dinit) ? dinit + (seq_of(seq_idx, bi, s.T, t0) * s.H + h) * PN : nullptr;
    float part = 0.f;
    for (int64_t e = threadIdx.x; e < PN; e += blockDim.x) {
      const float cur = nxt_start ? 0.f : cr[e];
      const float dh = bc[e];
      bc[e] = cur;
      if (hin) part = fmaf(hin[e], cur, part);
      const float dHc = fmaf(eCarry, cur, dh);
      cr[e] = dHc;
      if (di) di[e] += dHc;
    }
    const float tot = block_sum(part, red);
    if (threadIdx.x == 0) dEpass[(bi * s.H + h) * s.nc + c] = eIn * tot;
  }
}

// Gradient of the initial state of a sequence that starts inside a chunk, at
// local position f >= 1 of chunk c (one thread per (seq, h, p, n)):
//   dinit[seq] = sum_{i of seq in chunk c} exp(Acs_i - Acs_{f-1}) g_i C_i^T
//              + exp(E_c - Acs_{f-1}) dS_c   when seq holds the chunk's last token.
// Sequences that start at a chunk's first token get theirs from the reverse
// state passing; ids with no token keep the zeros of the preceding memset.
template <class TIn>
__global__ void dinit_mid_kernel(Shape s, const TIn *__restrict__ dout, const TIn *__restrict__ Cm,
                                 const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
                                 const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first,
                                 const float *__restrict__ dS, float *__restrict__ dinit) {
  const int64_t PN = s.P * s.N;
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (dinit == nullptr || idx >= s.nseq * s.H * PN) return;
  const int64_t e = idx % PN, h = (idx / PN) % s.H, sq = idx / (PN * s.H);
  const int64_t p = e / s.N, n = e % s.N, g = h / s.hpg;
  const int64_t ts = first[sq];
  if (ts < 0 || ts % s.Q == 0) return;
  const int64_t c = ts / s.Q, t0 = c * s.Q, Lc = min(s.Q, s.T - t0), f = ts - t0;
  const float *ah = acs_hi + (h * s.nc + c) * s.Q;   // batch row 0
  const float *al = acs_lo + (h * s.nc + c) * s.Q;
  float acc = 0.f;
  for (int64_t i = f; i < Lc && seq_idx[t0 + i] == sq; ++i) {
    const float w = expf(acs_diff(ah[i], al[i], ah[f - 1], al[f - 1]));
    acc = fmaf(w * ld(dout + ((t0 + i) * s.H + h) * s.P + p), ld(Cm + ((t0 + i) * s.G + g) * s.N + n), acc);
  }
  if (seq_idx[t0 + Lc - 1] == sq)
    acc = fmaf(expf(acs_diff(ah[Lc - 1], al[Lc - 1], ah[f - 1], al[f - 1])), dS[(c * s.H + h) * PN + e], acc);
  dinit[idx] = acc;
}

// dx_i[p] = dt_i sum_{j>=i} M[j,i] g_j[p] + w_i sum_n B_i[n] dS[p,n] + D g_i[p],
// w_i = exp(E - Acs_i) dt_i for the tokens of the sequence holding the
// chunk's last token (i >= fe), else 0.  One thread per (b,t,h,p).
template <class TIn>
__global__ void dx_kernel(Shape s, const TIn *__restrict__ dout, const TIn *__restrict__ Bm,
                          const float *__restrict__ dt, const float *__restrict__ D, const float *__restrict__ Mm,
                          const float *__restrict__ dS, const float *__restrict__ acs_hi,
                          const float *__restrict__ acs_lo, const int32_t *__restrict__ seq_idx,
                          const int32_t *__restrict__ first, float *__restrict__ dx) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= s.b * s.T * s.H * s.P) return;
  const int64_t p = idx % s.P, h = (idx / s.P) % s.H, t = (idx / (s.P * s.H)) % s.T, bi = idx / (s.P * s.H * s.T);
  const int64_t c = t / s.Q, i = t % s.Q, t0 = c * s.Q, Lc = min(s.Q, s.T - t0), g = h / s.hpg;
  const int64_t unit = (bi * s.nc + c) * s.H + h;
  const float *M = Mm + unit * s.Q * s.Q;
  float d1 = 0.f;
  for (int64_t j = i; j < Lc; ++j) d1 = fmaf(M[j * s.Q + i], ld(dout + ((bi * s.T + t0 + j) * s.H + h) * s.P + p), d1);
  const float *ds = dS + (unit * s.P + p) * s.N;
  const TIn *bi_ = Bm + ((bi * s.T + t) * s.G + g) * s.N;
  float y = 0.f;
  for (int64_t n = 0; n < s.N; ++n) y = fmaf(ld(bi_ + n), ds[n], y);
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float dti = dt[(bi * s.T + t) * s.H + h];
  const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
  const float wi = i < fe ? 0.f : expf(acs_diff(ah[Lc - 1], al[Lc - 1], ah[i], al[i])) * dti;
  dx[idx] = fmaf(dti, d1, fmaf(wi, y, D[h] * ld(dout + idx)));
}

// Per-head dB / dC rows, one thread per (b,t,h,n):
//   dC_h[i,n] = sum_{j<=i} W[i,j] B_j[n] + din_i sum_p Hin[p,n] g_i[p]
//   dB_h[i,n] = sum_{j>=i} W[j,i] C_j[n] + w_i sum_p dS[p,n] x_i[p]
// (din_i, Hin as in chunk_scan_fwd; w_i as in dx_kernel).  Deterministic
// variant: written to per-head slots (b,T,H,N); atomic variant: added into
// dB/dC (b,T,G,N) with atomics.
template <class TIn, bool kAtomic>
__global__ void dbdc_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ dout,
                            const TIn *__restrict__ Bm, const TIn *__restrict__ Cm, const float *__restrict__ dt,
                            const float *__restrict__ Wm, const float *__restrict__ states,
                            const float *__restrict__ dS, const float *__restrict__ acs_hi,
                            const float *__restrict__ acs_lo, const int32_t *__restrict__ seq_idx,
                            const int32_t *__restrict__ first, const float *__restrict__ init,
                            float *__restrict__ dBo, float *__restrict__ dCo) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= s.b * s.T * s.H * s.N) return;
  const int64_t n = idx % s.N, h = (idx / s.N) % s.H, t = (idx / (s.N * s.H)) % s.T, bi = idx / (s.N * s.H * s.T);
  const int64_t c = t / s.Q, i = t % s.Q, t0 = c * s.Q, Lc = min(s.Q, s.T - t0), g = h / s.hpg;
  const int64_t unit = (bi * s.nc + c) * s.H + h;
  const float *W = Wm + unit * s.Q * s.Q;
  float dc = 0.f, db = 0.f;
  for (int64_t j = 0; j <= i; ++j) dc = fmaf(W[i * s.Q + j], ld(Bm + ((bi * s.T + t0 + j) * s.G + g) * s.N + n), dc);
  for (int64_t j = i; j < Lc; ++j) db = fmaf(W[j * s.Q + i], ld(Cm + ((bi * s.T + t0 + j) * s.G + g) * s.N + n), db);
  const int64_t f = local_start(seq_idx, first, bi, s.T, t, t0);
  const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
  const float *hs = f == 0 ? states + unit * s.P * s.N + n
                           : (init ? init + (seq_of(seq_idx, bi, s.T, t) * s.H + h) * s.P * s.N + n : nullptr);
  const float *ds = dS + unit * s.P * s.N + n;
  const TIn *gi = dout + ((bi * s.T + t) * s.H + h) * s.P;
  const TIn *xi = x + ((bi * s.T + t) * s.H + h) * s.P;
  float hg = 0.f, sx = 0.f;
  for (int64_t p = 0; p < s.P; ++p) {
    if (hs) hg = fmaf(hs[p * s.N], ld(gi + p), hg);
    sx = fmaf(ds[p * s.N], ld(xi + p), sx);
  }
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float wi = i < fe ? 0.f : expf(acs_diff(ah[Lc - 1], al[Lc - 1], ah[i], al[i])) * dt[(bi * s.T + t) * s.H + h];
  const float din = expf(f == 0 ? __fadd_rn(ah[i], al[i]) : acs_diff(ah[i], al[i], ah[f - 1], al[f - 1]));
  dc = fmaf(din, hg, dc);
  db = fmaf(wi, sx, db);
  if (kAtomic) {
    const int64_t o = ((bi * s.T + t) * s.G + g) * s.N + n;
    atomicAdd(dBo + o, db);
    atomicAdd(dCo + o, dc);
  } else {
    dBo[idx] = db;
    dCo[idx] = dc;
  }
}

constexpr int kOrdTile = 32;   // tokens per tile of the ordered dB/dC fold

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(int *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Ordered dB/dC fold.  Work unit = (b, c, g, token tile tt, head k of the
// group), k fastest, handed out in that order by an atomic ticket, so a CTA
// only ever waits for units with smaller tickets, which are already running.
// The CTA computes its tile's per-head dB/dC rows exactly as dbdc_kernel does
// (same terms, same order) into shared memory, waits until the tile's
// semaphore reads k (a bounded spin: past spin_limit polls it sets status
// bit 1 and skips its add), then stores (k = 0) or adds its rows into dB/dC,
// and releases the semaphore to k + 1.
template <class TIn>
__global__ void dbdc_ordered_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ dout,
                                    const TIn *__restrict__ Bm, const TIn *__restrict__ Cm,
                                    const float *__restrict__ dt, const float *__restrict__ Wm,
                                    const float *__restrict__ states, const float *__restrict__ dS,
                                    const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
                                    const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first,
                                    const float *__restrict__ init, int *__restrict__ status, int *__restrict__ sem,
                                    uint32_t spin_limit, float *__restrict__ dBo, float *__restrict__ dCo) {
  extern __shared__ float tile[];   // [2][kOrdTile][N]: dB rows then dC rows
  __shared__ int s_unit, s_go;
  if (threadIdx.x == 0) s_unit = atomicAdd(status + 1, 1);
  __syncthreads();
  const int64_t ntt = cdiv(s.Q, kOrdTile);
  const int64_t unit = s_unit;
  const int64_t k = unit % s.hpg, tileid = unit / s.hpg;
  const int64_t tt = tileid % ntt, g = (tileid / ntt) % s.G, c = (tileid / (ntt * s.G)) % s.nc;
  const int64_t bi = tileid / (ntt * s.G * s.nc);
  const int64_t h = g * s.hpg + k, t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
  const int64_t i0 = tt * kOrdTile, i1 = min(Lc, i0 + kOrdTile);
  const int64_t hunit = (bi * s.nc + c) * s.H + h;
  const float *W = Wm + hunit * s.Q * s.Q;
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
  for (int64_t e = threadIdx.x; e < (i1 - i0) * s.N; e += blockDim.x) {
    const int64_t i = i0 + e / s.N, n = e % s.N, t = t0 + i;
    float dc = 0.f, db = 0.f;
    for (int64_t j = 0; j <= i; ++j) dc = fmaf(W[i * s.Q + j], ld(Bm + ((bi * s.T + t0 + j) * s.G + g) * s.N + n), dc);
    for (int64_t j = i; j < Lc; ++j) db = fmaf(W[j * s.Q + i], ld(Cm + ((bi * s.T + t0 + j) * s.G + g) * s.N + n), db);
    const int64_t f = local_start(seq_idx, first, bi, s.T, t, t0);
    const float *hs = f == 0 ? states + hunit * s.P * s.N + n
                             : (init ? init + (seq_of(seq_idx, bi, s.T, t) * s.H + h) * s.P * s.N + n : nullptr);
    const float *ds = dS + hunit * s.P * s.N + n;
    const TIn *gi = dout + ((bi * s.T + t) * s.H + h) * s.P;
    const TIn *xi = x + ((bi * s.T + t) * s.H + h) * s.P;
    float hg = 0.f, sx = 0.f;
    for (int64_t p = 0; p < s.P; ++p) {
      if (hs) hg = fmaf(hs[p * s.N], ld(gi + p), hg);
      sx = fmaf(ds[p * s.N], ld(xi + p), sx);
    }
    const float wi = i < fe ? 0.f : expf(acs_diff(ah[Lc - 1], al[Lc - 1], ah[i], al[i])) * dt[(bi * s.T + t) * s.H + h];
    const float din = expf(f == 0 ? __fadd_rn(ah[i], al[i]) : acs_diff(ah[i], al[i], ah[f - 1], al[f - 1]));
    tile[e] = fmaf(wi, sx, db);
    tile[kOrdTile * s.N + e] = fmaf(din, hg, dc);
  }
  __syncthreads();
  int *sm_flag = sem + tileid;
  if (threadIdx.x == 0) {
    int go = 1;
    if (k > 0) {
      uint32_t it = 0;
      while (ld_acquire_gpu(sm_flag) != int(k)) {
        if (++it > spin_limit) {   // predecessor never published: report, skip the add
          atomicOr(status, 1);
          go = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    s_go = go;
  }
  __syncthreads();
  if (!s_go) return;
  for (int64_t e = threadIdx.x; e < (i1 - i0) * s.N; e += blockDim.x) {
    const int64_t i = i0 + e / s.N, n = e % s.N;
    const int64_t o = ((bi * s.T + t0 + i) * s.G + g) * s.N + n;
    const float db = tile[e], dc = tile[kOrdTile * s.N + e];
    dBo[o] = (k == 0 ? 0.f : dBo[o]) + db;   // 0 + s0 + s1 + ..., as the slot fold adds
    dCo[o] = (k == 0 ? 0.f : dCo[o]) + dc;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) st_release_gpu(sm_flag, int(k) + 1);
}

// Per token (b,c,h,i): the dt-weight part of ddt and the gradient reaching
// Acs_i, before the reverse cumsum:
//   ddt_part = sum_{j>=i} MG[j,i] + exp(E - Acs_i) sx_i
//   dAcs_i   = sum_{j<i} MG[i,j] dt_j - dt_i sum_{j>i} MG[j,i]
//            + v_i - u_i,   v_i = din_i g_i . (Hin C_i),   u_i = w_i sx_i
// with sx_i = x_i . (dS B_i) (din_i, Hin as in chunk_scan_fwd; w_i and the
// exp(E - Acs_i) factor zero before fe).  Also gx_i = g_i . x_i for dD, and
// vin_i = v_i for tokens of a sequence that started inside the chunk (their
// decay exp(Acs_i - Acs_{f-1}) also depends on Acs_{f-1}), else 0.
template <class TIn>
__global__ void ddt_dacs_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ dout,
                                const TIn *__restrict__ Bm, const TIn *__restrict__ Cm,
                                const float *__restrict__ dt, const float *__restrict__ MGm,
                                const float *__restrict__ states, const float *__restrict__ dS,
                                const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
                                const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first,
                                const float *__restrict__ init, float *__restrict__ ddt_part,
                                float *__restrict__ dAcs, float *__restrict__ u_buf, float *__restrict__ gx_buf,
                                float *__restrict__ vin_buf) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= s.b * s.H * s.nc * s.Q) return;
  const int64_t i = idx % s.Q, c = (idx / s.Q) % s.nc, h = (idx / (s.Q * s.nc)) % s.H, bi = idx / (s.Q * s.nc * s.H);
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0), g = h / s.hpg, t = t0 + i;
  if (i >= Lc) {
    dAcs[idx] = 0.f;
    u_buf[idx] = 0.f;
    gx_buf[idx] = 0.f;
    vin_buf[idx] = 0.f;
    return;
  }
  const int64_t unit = (bi * s.nc + c) * s.H + h;
  const float *MG = MGm + unit * s.Q * s.Q;
  const float *dtc = dt + (bi * s.T + t0) * s.H + h;  // dtc[j * H]
  float col = 0.f, row = 0.f;
  const float diag = MG[i * s.Q + i];
  for (int64_t j = i + 1; j < Lc; ++j) col += MG[j * s.Q + i];
  for (int64_t j = 0; j < i; ++j) row = fmaf(MG[i * s.Q + j], dtc[j * s.H], row);
  const float dti = dtc[i * s.H];
  const int64_t f = local_start(seq_idx, first, bi, s.T, t, t0);
  const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
  const float *hs = f == 0 ? states + unit * s.P * s.N
                           : (init ? init + (seq_of(seq_idx, bi, s.T, t) * s.H + h) * s.P * s.N : nullptr);
  const float *ds = dS + unit * s.P * s.N;
  const TIn *ci = Cm + ((bi * s.T + t) * s.G + g) * s.N;
  const TIn *b_i = Bm + ((bi * s.T + t) * s.G + g) * s.N;
  const TIn *gi = dout + ((bi * s.T + t) * s.H + h) * s.P;
  const TIn *xi = x + ((bi * s.T + t) * s.H + h) * s.P;
  float inter = 0.f, sx = 0.f, gx = 0.f;
  for (int64_t p = 0; p < s.P; ++p) {
    float hc = 0.f, dsb = 0.f;
    for (int64_t n = 0; n < s.N; ++n) {
      if (hs) hc = fmaf(hs[p * s.N + n], ld(ci + n), hc);
      dsb = fmaf(ds[p * s.N + n], ld(b_i + n), dsb);
    }
    const float gp = ld(gi + p), xp = ld(xi + p);
    inter = fmaf(gp, hc, inter);
    sx = fmaf(xp, dsb, sx);
    gx = fmaf(gp, xp, gx);
  }
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float eEi = i < fe ? 0.f : expf(acs_diff(ah[Lc - 1], al[Lc - 1], ah[i], al[i]));
  const float din = expf(f == 0 ? __fadd_rn(ah[i], al[i]) : acs_diff(ah[i], al[i], ah[f - 1], al[f - 1]));
  const float u = eEi * dti * sx;
  const float v = din * inter;
  ddt_part[(bi * s.T + t) * s.H + h] = (col + diag) + eEi * sx;
  dAcs[idx] = row - dti * col + v - u;
  u_buf[idx] = u;
  gx_buf[idx] = gx;
  vin_buf[idx] = f == 0 ? 0.f : v;
}

// Reverse in-chunk cumsum, one thread per (b,c,h), sequential in one fixed
// order: dAcs_{Lc-1} += sum_i u_i + dEpass; da_i = sum_{k>=i} dAcs_k;
// ddt_i = ddt_part_i + A da_i; per-chunk partials dA = sum_i dt_i da_i and
// dD = sum_i gx_i (slot (b,c,h)), or atomics in the atomic variant.  Where a
// sequence starts inside the chunk at f >= 1, the decays measured from
// Acs_{f-1} give dAcs_{f-1} -= sum of that sequence's vin (plus dEpass when
// it holds the chunk's last token).
template <bool kAtomic>
__global__ void cumsum_bwd_kernel(Shape s, const float *__restrict__ dt, const float *__restrict__ A,
                                  const float *__restrict__ dAcs, const float *__restrict__ u_buf,
                                  const float *__restrict__ gx_buf, const float *__restrict__ vin_buf,
                                  const float *__restrict__ dEpass, const int32_t *__restrict__ seq_idx,
                                  const int32_t *__restrict__ first, const float *__restrict__ ddt_part,
                                  float *__restrict__ ddt, float *__restrict__ dA_part, float *__restrict__ dD_part) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= s.b * s.nc * s.H) return;
  const int64_t h = idx % s.H, c = (idx / s.H) % s.nc, bi = idx / (s.H * s.nc);
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
  const int64_t base = ((bi * s.H + h) * s.nc + c) * s.Q;
  float su = 0.f, sg = 0.f;
  for (int64_t i = 0; i < Lc; ++i) {
    su += u_buf[base + i];
    sg += gx_buf[base + i];
  }
  const float Ah = A[h];
  const float dEp = dEpass[(bi * s.H + h) * s.nc + c];
  const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
  float da = su + dEp;
  float pend = fe > 0 ? dEp : 0.f;  // owed by Acs_{f-1} of the sequence being walked
  float dAp = 0.f;
  for (int64_t i = Lc - 1; i >= 0; --i) {
    float d = dAcs[base + i];
    if (seq_idx && i + 1 < Lc && seq_idx[bi * s.T + t0 + i] != seq_idx[bi * s.T + t0 + i + 1]) {
      d -= pend;  // token i + 1 starts a sequence inside the chunk
      pend = 0.f;
    }
    da += d;
    pend += vin_buf[base + i];
    const int64_t o = (bi * s.T + t0 + i) * s.H + h;
    ddt[o] = fmaf(Ah, da, ddt_part[o]);
    dAp = fmaf(dt[o], da, dAp);
  }
  if (kAtomic) {
    atomicAdd(dA_part + h, dAp);
    atomicAdd(dD_part + h, sg);
  } else {
    dA_part[idx] = dAp;
    dD_part[idx] = sg;
  }
}

// dB[b,t,g,n] = sum over the group's heads, ascending, of the per-head slots.
__global__ void reduce_heads_kernel(Shape s, const float *__restrict__ slot_b, const float *__restrict__ slot_c,
                                    float *__restrict__ dB, float *__restrict__ dC) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= s.b * s.T * s.G * s.N) return;
  const int64_t n = idx % s.N, g = (idx / s.N) % s.G, bt = idx / (s.N * s.G);
  float sb = 0.f, sc = 0.f;
  for (int64_t k = 0; k < s.hpg; ++k) {
    const int64_t o = (bt * s.H + g * s.hpg + k) * s.N + n;
    sb += slot_b[o];
    sc += slot_c[o];
  }
  dB[idx] = sb;
  dC[idx] = sc;
}

// dA[h], dD[h] = sum over (b, c) ascending of the per-chunk partials.
__global__ void reduce_heads_scalars_kernel(Shape s, const float *__restrict__ dA_part,
                                            const float *__restrict__ dD_part, float *__restrict__ dA,
                                            float *__restrict__ dD) {
  const int64_t h = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (h >= s.H) return;
  float a = 0.f, d = 0.f;
  for (int64_t bc = 0; bc < s.b * s.nc; ++bc) {
    a += dA_part[bc * s.H + h];
    d += dD_part[bc * s.H + h];
  }
  dA[h] = a;
  dD[h] = d;
}

struct BwdWs {
  int *status;   // [0] error bits (bit 1: an ordered-fold wait gave up), [1] ticket; first in the workspace
  float *acs_hi, *acs_lo, *CB, *Mm, *Wm, *MGm, *buf, *carry, *dEpass, *dAcs, *u, *gx, *vin, *ddt_part, *dA_part,
      *dD_part, *slot_b, *slot_c;
  int32_t *first;
  int *sem;
};

int64_t ordered_tiles(const Shape &s) { return s.b * s.nc * s.G * cdiv(s.Q, kOrdTile); }

BwdWs carve_bwd(Carver &cv, const Shape &s, int variant) {
  const bool atomic = variant == 1, ordered = variant == 2;
  BwdWs w;
  w.status = cv.take<int>(2);
  const int64_t acs = s.b * s.H * s.nc * s.Q, qq = s.b * s.nc * s.H * s.Q * s.Q;
  w.acs_hi = cv.take<float>(acs);
  w.acs_lo = cv.take<float>(acs);
  w.CB = cv.take<float>(s.b * s.nc * s.G * s.Q * s.Q);
  w.Mm = cv.take<float>(qq);
  w.Wm = cv.take<float>(qq);
  w.MGm = cv.take<float>(qq);
  w.buf = cv.take<float>(s.b * s.nc * s.H * s.P * s.N);
  w.carry = cv.take<float>(s.b * s.H * s.P * s.N);
  w.dEpass = cv.take<float>(s.b * s.H * s.nc);
  w.dAcs = cv.take<float>(acs);
  w.u = cv.take<float>(acs);
  w.gx = cv.take<float>(acs);
  w.vin = cv.take<float>(acs);
  w.ddt_part = cv.take<float>(s.b * s.T * s.H);
  w.dA_part = cv.take<float>(s.b * s.nc * s.H);
  w.dD_part = cv.take<float>(s.b * s.nc * s.H);
  w.slot_b = (atomic || ordered) ? nullptr : cv.take<float>(s.b * s.T * s.H * s.N);
  w.slot_c = (atomic || ordered) ? nullptr : cv.take<float>(s.b * s.T * s.H * s.N);
  w.first = cv.take<int32_t>(s.nseq);
  w.sem = ordered ? cv.take<int>(ordered_tiles(s)) : nullptr;
  return w;
}

struct FwdWs {
  float *acs_hi, *acs_lo, *CB, *S;
  int32_t *first;
};

FwdWs carve_fwd(Carver &cv, const Shape &s) {
  FwdWs w;
  const int64_t acs = s.b * s.H * s.nc * s.Q;
  w.acs_hi = cv.take<float>(acs);
  w.acs_lo = cv.take<float>(acs);
  w.CB = cv.take<float>(s.b * s.nc * s.G * s.Q * s.Q);
  w.S = cv.take<float>(s.b * s.nc * s.H * s.P * s.N);
  w.first = cv.take<int32_t>(s.nseq);
  return w;
}

// Table of sequence first tokens (only with seq_idx; batch row 0).
cudaError_t build_first(const Shape &s, const int32_t *seq_idx, int32_t *first, int bs, cudaStream_t st) {
  const cudaError_t err = cudaMemsetAsync(first, 0xff, size_t(s.nseq) * sizeof(int32_t), st);
  if (err != cudaSuccess) return err;
  seq_first_kernel<<<unsigned(cdiv(s.T, bs)), bs, 0, st>>>(s.T, seq_idx, first);
  return cudaSuccess;
}

inline unsigned grid1(int64_t n, int bs) { return unsigned(cdiv(n, bs)); }

template <class TIn>
cudaError_t fwd_impl(const Shape &s, const Args &a, void *ws, int bs, cudaStream_t st) {
  Carver cv(ws);
  FwdWs w = carve_fwd(cv, s);
  const TIn *x = static_cast<const TIn *>(a.x), *Bm = static_cast<const TIn *>(a.B), *Cm = static_cast<const TIn *>(a.C);
  const int32_t *first = a.seq_idx ? w.first : nullptr;
  if (a.seq_idx) {
    const cudaError_t err = build_first(s, a.seq_idx, w.first, bs, st);
    if (err != cudaSuccess) return err;
  }
  cumsum_fwd_kernel<<<grid1(s.b * s.nc * s.H, bs), bs, 0, st>>>(s, a.dt, a.A, w.acs_hi, w.acs_lo);
  chunk_state_fwd_kernel<TIn><<<dim3(unsigned(s.b * s.nc * s.H), grid1(s.P * s.N, bs)), bs, s.Q * sizeof(float), st>>>(
      s, x, Bm, a.dt, w.acs_hi, w.acs_lo, a.seq_idx, first, w.S);
  state_passing_fwd_kernel<<<grid1(s.b * s.H * s.P * s.N, bs), bs, 0, st>>>(s, w.S, w.acs_hi, w.acs_lo, a.seq_idx,
                                                                            first, a.init, a.states_out);
  cb_kernel<TIn><<<dim3(unsigned(s.b * s.nc * s.G), grid1(s.Q * s.Q, bs)), bs, 0, st>>>(s, Bm, Cm, w.CB);
  chunk_scan_fwd_kernel<TIn><<<grid1(s.b * s.T * s.H * s.P, bs), bs, 0, st>>>(
      s, x, Cm, a.dt, a.D, w.CB, w.acs_hi, w.acs_lo, a.states_out, a.seq_idx, first, a.init,
      static_cast<TIn *>(a.y));
  return cudaGetLastError();
}

template <class TIn>
cudaError_t bwd_impl(const Shape &s, const Args &a, void *ws, int bs, int variant, uint32_t spin_limit, cudaStream_t st,
                     Trace &tr) {
  const bool atomic = variant == 1, ordered = variant == 2;
  Carver cv(ws);
  BwdWs w = carve_bwd(cv, s, variant);
  const TIn *x = static_cast<const TIn *>(a.x), *Bm = static_cast<const TIn *>(a.B), *Cm = static_cast<const TIn *>(a.C);
  const TIn *g = static_cast<const TIn *>(a.dout);
  const int64_t PN = s.P * s.N;
  cudaError_t err;
  if (a.dinit) {
    err = cudaMemsetAsync(a.dinit, 0, size_t(s.nseq * s.H * PN) * sizeof(float), st);
    if (err != cudaSuccess) return err;
  }
  err = cudaMemsetAsync(w.carry, 0, size_t(s.b * s.H * PN) * sizeof(float), st);
  if (err != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(w.status, 0, 2 * sizeof(int), st)) != cudaSuccess) return err;
  if (ordered && (err = cudaMemsetAsync(w.sem, 0, size_t(ordered_tiles(s)) * sizeof(int), st)) != cudaSuccess)
    return err;
  if (atomic) {
    const size_t nbg = size_t(s.b * s.T * s.G * s.N) * sizeof(float);
    if ((err = cudaMemsetAsync(a.dB, 0, nbg, st)) != cudaSuccess) return err;
    if ((err = cudaMemsetAsync(a.dC, 0, nbg, st)) != cudaSuccess) return err;
    if ((err = cudaMemsetAsync(a.dA, 0, size_t(s.H) * sizeof(float), st)) != cudaSuccess) return err;
    if ((err = cudaMemsetAsync(a.dD, 0, size_t(s.H) * sizeof(float), st)) != cudaSuccess) return err;
  }
  const unsigned nbch = unsigned(s.b * s.nc * s.H);
  const int32_t *first = a.seq_idx ? w.first : nullptr;
  if (a.seq_idx) {
    tr.mark(st);
    if ((err = build_first(s, a.seq_idx, w.first, bs, st)) != cudaSuccess) return err;
    tr.mark(st);
  }
  tr.mark(st);
  cumsum_fwd_kernel<<<grid1(s.b * s.nc * s.H, bs), bs, 0, st>>>(s, a.dt, a.A, w.acs_hi, w.acs_lo);
  tr.mark(st);
  tr.mark(st);
  cb_kernel<TIn><<<dim3(unsigned(s.b * s.nc * s.G), grid1(s.Q * s.Q, bs)), bs, 0, st>>>(s, Bm, Cm, w.CB);
  tr.mark(st);
  tr.mark(st);
  mwg_kernel<TIn><<<dim3(nbch, grid1(s.Q * s.Q, bs)), bs, 0, st>>>(s, x, g, a.dt, w.CB, w.acs_hi, w.acs_lo,
                                                                    a.seq_idx, first, w.Mm, w.Wm, w.MGm);
  tr.mark(st);
  tr.mark(st);
  dhscan_kernel<TIn><<<dim3(nbch, grid1(PN, bs)), bs, s.Q * sizeof(float), st>>>(s, g, Cm, w.acs_hi, w.acs_lo,
                                                                                 a.seq_idx, first, w.buf);
  tr.mark(st);
  tr.mark(st);
  // fixed block: this kernel folds per-thread partial dot products, so its
  // shape must not follow the launch configuration
  state_passing_bwd_kernel<<<unsigned(s.b * s.H), kPassThreads, 0, st>>>(
      s, w.buf, w.carry, a.states_in, w.acs_hi, w.acs_lo, a.seq_idx, first, a.init, w.dEpass, a.dinit);
  tr.mark(st);
  if (a.seq_idx) {
    tr.mark(st);
    dinit_mid_kernel<TIn><<<grid1(s.nseq * s.H * PN, bs), bs, 0, st>>>(s, g, Cm, w.acs_hi, w.acs_lo, a.seq_idx,
                                                                       first, w.buf, a.dinit);
    tr.mark(st);
  }
  tr.mark(st);
  dx_kernel<TIn><<<grid1(s.b * s.T * s.H * s.P, bs), bs, 0, st>>>(s, g, Bm, a.dt, a.D, w.Mm, w.buf, w.acs_hi,
                                                                  w.acs_lo, a.seq_idx, first, a.dx);
  tr.mark(st);
  if (atomic) {
    tr.mark(st);
    dbdc_kernel<TIn, true><<<grid1(s.b * s.T * s.H * s.N, bs), bs, 0, st>>>(
        s, x, g, Bm, Cm, a.dt, w.Wm, a.states_in, w.buf, w.acs_hi, w.acs_lo, a.seq_idx, first, a.init, a.dB, a.dC);
    tr.mark(st);
  } else if (ordered) {
    tr.mark(st);
    const int64_t units = ordered_tiles(s) * s.hpg;
    const size_t shm = size_t(2 * kOrdTile * s.N) * sizeof(float);
    if (shm > 48 * 1024 &&
        (err = cudaFuncSetAttribute(dbdc_ordered_kernel<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    int(shm))) != cudaSuccess)
      return err;
    dbdc_ordered_kernel<TIn><<<unsigned(units), bs, shm, st>>>(
        s, x, g, Bm, Cm, a.dt, w.Wm, a.states_in, w.buf, w.acs_hi, w.acs_lo, a.seq_idx, first, a.init, w.status,
        w.sem, spin_limit, a.dB, a.dC);
    tr.mark(st);
  } else {
    tr.mark(st);
    dbdc_kernel<TIn, false><<<grid1(s.b * s.T * s.H * s.N, bs), bs, 0, st>>>(
        s, x, g, Bm, Cm, a.dt, w.Wm, a.states_in, w.buf, w.acs_hi, w.acs_lo, a.seq_idx, first, a.init, w.slot_b,
        w.slot_c);
    tr.mark(st);
  }
  tr.mark(st);
  ddt_dacs_kernel<TIn><<<grid1(s.b * s.H * s.nc * s.Q, bs), bs, 0, st>>>(
      s, x, g, Bm, Cm, a.dt, w.MGm, a.states_in, w.buf, w.acs_hi, w.acs_lo, a.seq_idx, first, a.init, w.ddt_part,
      w.dAcs, w.u, w.gx, w.vin);
  tr.mark(st);
  if (atomic) {
    tr.mark(st);
    cumsum_bwd_kernel<true><<<grid1(s.b * s.nc * s.H, bs), bs, 0, st>>>(
        s, a.dt, a.A, w.dAcs, w.u, w.gx, w.vin, w.dEpass, a.seq_idx, first, w.ddt_part, a.ddt, a.dA, a.dD);
    tr.mark(st);
  } else {
    tr.mark(st);
    cumsum_bwd_kernel<false><<<grid1(s.b * s.nc * s.H, bs), bs, 0, st>>>(
        s, a.dt, a.A, w.dAcs, w.u, w.gx, w.vin, w.dEpass, a.seq_idx, first, w.ddt_part, a.ddt, w.dA_part, w.dD_part);
    tr.mark(st);
    if (!ordered) {
      tr.mark(st);
      reduce_heads_kernel<<<grid1(s.b * s.T * s.G * s.N, bs), bs, 0, st>>>(s, w.slot_b, w.slot_c, a.dB, a.dC);
      tr.mark(st);
    }
    tr.mark(st);
    reduce_heads_scalars_kernel<<<grid1(s.H, bs), bs, 0, st>>>(s, w.dA_part, w.dD_part, a.dA, a.dD);
    tr.mark(st);
  }
  return cudaGetLastError();
}

}  // namespace

size_t simt_fwd_workspace(const Shape &s) {
  Carver cv(nullptr);
  carve_fwd(cv, s);
  return cv.bytes();
}

size_t simt_bwd_workspace(const Shape &s, int variant) {
  Carver cv(nullptr);
  carve_bwd(cv, s, variant);
  return cv.bytes();
}

int simt_bwd_launches(const Shape &, int variant, bool seq) {
  return (variant == 1 ? 9 : (variant == 2 ? 10 : 11)) + (seq ? 2 : 0);
}

const char *simt_bwd_launch_name(int variant, bool seq, int k) {
  static const char *det[] = {"cumsum_fwd", "cb", "mwg", "dhscan", "state_passing_bwd", "dx", "dbdc",
                              "ddt_dacs", "cumsum_bwd", "reduce_heads", "reduce_heads_scalars"};
  static const char *atm[] = {"cumsum_fwd", "cb", "mwg", "dhscan", "state_passing_bwd", "dx", "dbdc_atomic",
                              "ddt_dacs", "cumsum_bwd_atomic"};
  static const char *ord[] = {"cumsum_fwd", "cb", "mwg", "dhscan", "state_passing_bwd", "dx", "dbdc_ordered",
                              "ddt_dacs", "cumsum_bwd", "reduce_heads_scalars"};
  const int n = variant == 1 ? 9 : (variant == 2 ? 10 : 11);
  if (k < 0 || k >= n + (seq ? 2 : 0)) return "invalid";
  if (seq) {
    // seq_first runs first, dinit_mid right after the reverse state passing
    if (k == 0) return "seq_first";
    if (k == 6) return "dinit_mid";
    k = k < 6 ? k - 1 : k - 2;
  }
  return variant == 1 ? atm[k] : (variant == 2 ? ord[k] : det[k]);
}

cudaError_t simt_fwd(const Shape &s, bool bf16, const Args &a, void *ws, int block, cudaStream_t st) {
  return bf16 ? fwd_impl<__nv_bfloat16>(s, a, ws, block, st) : fwd_impl<float>(s, a, ws, block, st);
}

cudaError_t simt_bwd(const Shape &s, bool bf16, const Args &a, void *ws, int block, int variant, uint32_t spin_limit,
                     cudaStream_t st, Trace &tr) {
  return bf16 ? bwd_impl<__nv_bfloat16>(s, a, ws, block, variant, spin_limit, st, tr)
              : bwd_impl<float>(s, a, ws, block, variant, spin_limit, st, tr);
}

}  // namespace ssd
