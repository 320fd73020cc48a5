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

// ------------------------------------------------------------ tile products --
// The per-chunk products below are computed by CTAs of 256 threads, each
// producing a tile of (16 RA) x 64 outputs D[r][q] = sum_k A(r, k) B(q, k) with
// the operands staged through shared memory in k blocks of 16.  Every output
// element is still one sequential fmaf chain over its k index, ascending, one
// term per k (terms outside a product's range are exact zeros), so its bits
// depend neither on the tiling nor on the launch configuration.  Thread
// (ty, tx) = (tid / 16, tid % 16) holds rows RA ty + a and columns 4 tx + b,
// read from shared memory as vectors.
constexpr int kTileThreads = 256, kTK = 16, kTC = 64;

template <int RA>
struct TileBuf {
  float a[kTK][16 * RA + 4];
  float b[kTK][kTC + 4];
};

template <int RA>
struct RowVec;
template <>
struct RowVec<4> {
  using T = float4;
};
template <>
struct RowVec<2> {
  using T = float2;
};

// fa(r, k) = A(r, k), fb(q, k) = B(q, k) (0 outside their ranges);
// kAKFast / kBKFast: consecutive k adjacent in memory (else consecutive r, q),
// which picks the thread order of the loads so that they coalesce.  Only k in
// [kb, K) is visited: a causal product whose terms outside that window are
// exact zeros for every row of the tile passes the window, which drops only
// zero terms at the start or the end of each ascending chain (an accumulator
// that starts at +0 stays +0 across them, and x + 0 = x), so the bits are those
// of the full range.
template <int RA, bool kAKFast, bool kBKFast, class FA, class FB>
__device__ __forceinline__ void tile_mm(int64_t K, const FA &fa, const FB &fb, TileBuf<RA> &sb,
                                        float (&acc)[RA][4], int64_t kb = 0) {
  constexpr int R = 16 * RA;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
#pragma unroll
  for (int a = 0; a < RA; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
  // the next k block is read from global memory into registers while the
  // current one is multiplied out of shared memory
  constexpr int NA = R * kTK / kTileThreads, NB = kTC * kTK / kTileThreads;
  float ra[NA], rb[NB];
  auto fetch = [&](int64_t k0) {
#pragma unroll
    for (int u = 0; u < NA; ++u) {
      const int e = u * kTileThreads + tid;
      const int r = kAKFast ? e / kTK : e % R, kk = kAKFast ? e % kTK : e / R;
      ra[u] = (k0 + kk < K) ? fa(r, k0 + kk) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int e = u * kTileThreads + tid;
      const int q = kBKFast ? e / kTK : e % kTC, kk = kBKFast ? e % kTK : e / kTC;
      rb[u] = (k0 + kk < K) ? fb(q, k0 + kk) : 0.f;
    }
  };
  if (K > kb) fetch(kb);
  for (int64_t k0 = kb; k0 < K; k0 += kTK) {
#pragma unroll
    for (int u = 0; u < NA; ++u) {
      const int e = u * kTileThreads + tid;
      const int r = kAKFast ? e / kTK : e % R, kk = kAKFast ? e % kTK : e / R;
      sb.a[kk][r] = ra[u];
    }
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int e = u * kTileThreads + tid;
      const int q = kBKFast ? e / kTK : e % kTC, kk = kBKFast ? e % kTK : e / kTC;
      sb.b[kk][q] = rb[u];
    }
    __syncthreads();
    if (k0 + kTK < K) fetch(k0 + kTK);
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      const typename RowVec<RA>::T avv = *reinterpret_cast<const typename RowVec<RA>::T *>(&sb.a[kk][RA * ty]);
      const float4 bvv = *reinterpret_cast<const float4 *>(&sb.b[kk][4 * tx]);
      const float *av = reinterpret_cast<const float *>(&avv);
      const float bv[4] = {bvv.x, bvv.y, bvv.z, bvv.w};
#pragma unroll
      for (int a = 0; a < RA; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(av[a], bv[b], acc[a][b]);
    }
    __syncthreads();
  }
}

// row and column of this thread's output (a, b) within the tile
template <int RA>
__device__ __forceinline__ int tile_row(int a) { return RA * int(threadIdx.x >> 4) + a; }
__device__ __forceinline__ int tile_col(int b) { return 4 * int(threadIdx.x & 15) + b; }

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
// the sequence holding the chunk's last token (i >= fe), i ascending; a CTA
// per (b, c, h) and 64 x 64 tile of (p, n).
template <class TIn>
__global__ void __launch_bounds__(kTileThreads)
    chunk_state_fwd_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ Bm, const float *__restrict__ dt,
                           const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
                           const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first,
                           float *__restrict__ S) {
  extern __shared__ float w[];
  __shared__ TileBuf<4> sb;
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
  const int64_t ntn = cdiv(s.N, kTC);
  const int64_t p0 = (blockIdx.y / ntn) * 64, n0 = (blockIdx.y % ntn) * kTC;
  const TIn *xc = x + ((bi * s.T + t0) * s.H + h) * s.P;   // token i: xc + i * H P
  const TIn *bc = Bm + ((bi * s.T + t0) * s.G + g) * s.N;  // token i: bc + i * G N
  const int64_t HP = s.H * s.P, GN = s.G * s.N;
  float acc[4][4];
  tile_mm<4, false, false>(
      Lc, [&](int r, int64_t i) { const int64_t p = p0 + r; return p < s.P ? w[i] * ld(xc + i * HP + p) : 0.f; },
      [&](int q, int64_t i) { const int64_t n = n0 + q; return n < s.N ? ld(bc + i * GN + n) : 0.f; }, sb, acc);
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t p = p0 + tile_row<4>(a), n = n0 + tile_col(b);
      if (p < s.P && n < s.N) S[(unit * s.P + p) * s.N + n] = acc[a][b];
    }
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
// CB[b,c,g,i,j] = C_i . B_j for j <= i < Lc, else 0; a CTA per (b, c, g) and
// 64 x 64 tile of (i, j) (tiles above the diagonal are zeros).
template <class TIn>
__global__ void __launch_bounds__(kTileThreads)
    cb_kernel(Shape s, const TIn *__restrict__ Bm, const TIn *__restrict__ Cm, float *__restrict__ CB) {
  __shared__ TileBuf<4> sb;
  const int64_t unit = blockIdx.x;  // (b, c, g)
  const int64_t g = unit % s.G, c = (unit / s.G) % s.nc, bi = unit / (s.G * s.nc);
  const int64_t nt = cdiv(s.Q, 64);
  const int64_t i0 = (blockIdx.y / nt) * 64, j0 = (blockIdx.y % nt) * 64;
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0), GN = s.G * s.N;
  const TIn *cc = Cm + ((bi * s.T + t0) * s.G + g) * s.N;
  const TIn *bc = Bm + ((bi * s.T + t0) * s.G + g) * s.N;
  float acc[4][4] = {};
  if (j0 <= i0 && i0 < Lc)   // the tile reaches the lower triangle (same for the whole CTA)
    tile_mm<4, true, true>(
        s.N, [&](int r, int64_t n) { const int64_t i = i0 + r; return i < Lc ? ld(cc + i * GN + n) : 0.f; },
        [&](int q, int64_t n) { const int64_t j = j0 + q; return j < Lc ? ld(bc + j * GN + n) : 0.f; }, sb, acc);
  float *o = CB + unit * s.Q * s.Q;
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t i = i0 + tile_row<4>(a), j = j0 + tile_col(b);
      if (i < s.Q && j < s.Q) o[i * s.Q + j] = (j <= i && i < Lc) ? acc[a][b] : 0.f;
    }
}

// ------------------------------------------------------- chunk_scan (fwd) --
// y_i[p] = sum_{f<=j<=i} CB[i,j] exp(Acs_i - Acs_j) dt_j x_j[p]
//        + din_i sum_n Hin[p,n] C_i[n] + D x_i[p], f = local_start(i): Hin = states
// and din_i = exp(Acs_i) when f = 0, else Hin = init[seq] (or 0) and
// din_i = exp(Acs_i - Acs_{f-1}).  A CTA per (b, c, h) and 64 x 64 tile of (i, p).
template <class TIn>
__global__ void __launch_bounds__(kTileThreads, 3)
    chunk_scan_fwd_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ Cm, const float *__restrict__ dt,
                          const float *__restrict__ D, const float *__restrict__ CB, const float *__restrict__ acs_hi,
                          const float *__restrict__ acs_lo, const float *__restrict__ states,
                          const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first,
                          const float *__restrict__ init, TIn *__restrict__ y) {
  __shared__ TileBuf<4> sb;
  __shared__ int fr[64];   // local sequence start of each row of the tile
  const int64_t unit = blockIdx.x;  // (b, c, h)
  const int64_t h = unit % s.H, c = (unit / s.H) % s.nc, bi = unit / (s.H * s.nc);
  const int64_t g = h / s.hpg, t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
  const int64_t ntp = cdiv(s.P, kTC);
  const int64_t i0 = (blockIdx.y / ntp) * 64, p0 = (blockIdx.y % ntp) * kTC;
  if (i0 >= Lc) return;   // (the whole CTA)
  for (int r = threadIdx.x; r < 64; r += blockDim.x)
    fr[r] = i0 + r < Lc ? int(local_start(seq_idx, first, bi, s.T, t0 + i0 + r, t0)) : 0;
  __syncthreads();
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *cb = CB + ((bi * s.nc + c) * s.G + g) * s.Q * s.Q;
  const float *dtc = dt + (bi * s.T + t0) * s.H + h;      // token j: dtc[j * H]
  const TIn *xc = x + ((bi * s.T + t0) * s.H + h) * s.P;  // token j: xc + j * H P
  const TIn *cc = Cm + ((bi * s.T + t0) * s.G + g) * s.N; // token i: cc + i * G N
  const int64_t HP = s.H * s.P, GN = s.G * s.N;
  float acc[4][4], inter[4][4];
  tile_mm<4, true, false>(
      min(Lc, i0 + 64),   // (j <= i: the tile's rows see no token after its last row)
      [&](int r, int64_t j) {
        const int64_t i = i0 + r;
        if (i >= Lc || j > i || j < fr[r]) return 0.f;
        return cb[i * s.Q + j] * expf(acs_diff(ah[i], al[i], ah[j], al[j])) * dtc[j * s.H];
      },
      [&](int q, int64_t j) { const int64_t p = p0 + q; return p < s.P ? ld(xc + j * HP + p) : 0.f; }, sb, acc);
  const float *hst = states + unit * s.P * s.N;
  tile_mm<4, true, true>(
      s.N, [&](int r, int64_t n) { const int64_t i = i0 + r; return i < Lc ? ld(cc + i * GN + n) : 0.f; },
      [&](int q, int64_t n) { const int64_t p = p0 + q; return p < s.P ? hst[p * s.N + n] : 0.f; }, sb, inter);
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t i = i0 + tile_row<4>(a), p = p0 + tile_col(b);
      if (i >= Lc || p >= s.P) continue;
      const int64_t t = t0 + i, f = fr[tile_row<4>(a)];
      float in = inter[a][b];
      if (f > 0) {   // a sequence that started inside the chunk: its own initial state
        in = 0.f;
        if (init) {
          const float *hs = init + ((seq_of(seq_idx, bi, s.T, t) * s.H + h) * s.P + p) * s.N;
          const TIn *ci = cc + i * GN;
          for (int64_t n = 0; n < s.N; ++n) in = fmaf(hs[n], ld(ci + n), in);
        }
      }
      const float din = expf(f == 0 ? __fadd_rn(ah[i], al[i]) : acs_diff(ah[i], al[i], ah[f - 1], al[f - 1]));
      const int64_t idx = ((bi * s.T + t) * s.H + h) * s.P + p;
      const float xv = ld(x + idx);
      st(y + idx, fmaf(din, in, acc[a][b]) + D[h] * xv);
    }
}

// ============================================================ backward ====

// Per (b,c,h,i,j) with local_start(i) <= j <= i < Lc (same sequence):
// L = exp(Acs_i - Acs_j), Gx = g_i . x_j, M = CB[i,j] L, W = L Gx dt_j,
// MG = M Gx; zero elsewhere.  A CTA per (b, c, h) and 64 x 64 tile of (i, j).
// MG is only needed through its sums, so it is not stored: each tile leaves,
// per row i, its part of sum_{j<i} MG[i,j] dt_j (rowp[unit][tile column][i]),
// per column j its part of sum_{i>j} MG[i,j] (colp[unit][tile row][j]), and
// MG[i,i] (dg[unit][i]), each summed in one fixed order (the thread's four
// elements, then a fixed shuffle tree over the tile's row or a fixed loop
// over its column).
template <class TIn>
__global__ void __launch_bounds__(kTileThreads)
    mwg_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ dout, const float *__restrict__ dt,
               const float *__restrict__ CB, const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
               const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first, float *__restrict__ Mm,
               float *__restrict__ Wm, float *__restrict__ rowp, float *__restrict__ colp, float *__restrict__ dg) {
  __shared__ TileBuf<4> sb;
  __shared__ int fr[64];
  __shared__ float cpart[16][kTC];   // column partials of each thread row
  const int64_t unit = blockIdx.x;  // (b, c, h)
  const int64_t h = unit % s.H, c = (unit / s.H) % s.nc, bi = unit / (s.H * s.nc);
  const int64_t nt = cdiv(s.Q, 64);
  const int64_t i0 = (blockIdx.y / nt) * 64, j0 = (blockIdx.y % nt) * 64;
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0), g = h / s.hpg, HP = s.H * s.P;
  for (int r = threadIdx.x; r < 64; r += blockDim.x)
    fr[r] = i0 + r < Lc ? int(local_start(seq_idx, first, bi, s.T, t0 + i0 + r, t0)) : 0;
  __syncthreads();
  const TIn *gc = dout + ((bi * s.T + t0) * s.H + h) * s.P;
  const TIn *xc = x + ((bi * s.T + t0) * s.H + h) * s.P;
  const bool live = j0 <= i0 && i0 < Lc;   // (the whole CTA)
  float acc[4][4] = {};
  if (live)
    tile_mm<4, true, true>(
        s.P, [&](int r, int64_t p) { const int64_t i = i0 + r; return i < Lc ? ld(gc + i * HP + p) : 0.f; },
        [&](int q, int64_t p) { const int64_t j = j0 + q; return j < Lc ? ld(xc + j * HP + p) : 0.f; }, sb, acc);
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *cb = CB + ((bi * s.nc + c) * s.G + g) * s.Q * s.Q;
  float rp[4] = {0.f, 0.f, 0.f, 0.f}, cp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t i = i0 + tile_row<4>(a), j = j0 + tile_col(b);
      if (i >= s.Q || j >= s.Q) continue;
      float M = 0.f, W = 0.f, MG = 0.f, dtj = 0.f;
      if (live && j <= i && i < Lc && j >= fr[tile_row<4>(a)]) {
        const float L = expf(acs_diff(ah[i], al[i], ah[j], al[j]));
        const float gx = acc[a][b];
        dtj = dt[(bi * s.T + t0 + j) * s.H + h];
        M = cb[i * s.Q + j] * L;
        W = L * gx * dtj;
        MG = M * gx;
      }
      const int64_t o = unit * s.Q * s.Q + i * s.Q + j;
      Mm[o] = M;
      Wm[o] = W;
      if (j < i) rp[a] += MG * dtj;
      if (i > j) cp[b] += MG;
      if (i == j) dg[unit * s.Q + i] = MG;
    }
  // row parts: the 16 threads of a tile row (lanes 16 ty .. 16 ty + 15 of one warp)
  const int64_t nt2 = cdiv(s.Q, 64), it = blockIdx.y / nt2, jt = blockIdx.y % nt2;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    float v = rp[a];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int64_t i = i0 + tile_row<4>(a);
    if ((threadIdx.x & 15) == 0 && i < s.Q) rowp[(unit * nt2 + jt) * s.Q + i] = v;
  }
#pragma unroll
  for (int b = 0; b < 4; ++b) cpart[threadIdx.x >> 4][tile_col(b)] = cp[b];
  __syncthreads();
  if (threadIdx.x < kTC && j0 + threadIdx.x < s.Q) {
    float v = 0.f;
    for (int r = 0; r < 16; ++r) v += cpart[r][threadIdx.x];
    colp[(unit * nt2 + it) * s.Q + j0 + threadIdx.x] = v;
  }
}

// dHscan[b,c,h,p,n] = sum_i exp(Acs_i) g_i[p] C_i[n] over the tokens that see
// the state entering the chunk (local_start(i) == 0), i ascending; a CTA per
// (b, c, h) and 64 x 64 tile of (p, n).
template <class TIn>
__global__ void __launch_bounds__(kTileThreads)
    dhscan_kernel(Shape s, const TIn *__restrict__ dout, const TIn *__restrict__ Cm, const float *__restrict__ acs_hi,
                  const float *__restrict__ acs_lo, const int32_t *__restrict__ seq_idx,
                  const int32_t *__restrict__ first, float *__restrict__ dH) {
  extern __shared__ float ea[];
  __shared__ TileBuf<4> sb;
  const int64_t unit = blockIdx.x;  // (b, c, h)
  const int64_t h = unit % s.H, c = (unit / s.H) % s.nc, bi = unit / (s.H * s.nc);
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0), g = h / s.hpg;
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  for (int64_t i = threadIdx.x; i < Lc; i += blockDim.x)
    ea[i] = local_start(seq_idx, first, bi, s.T, t0 + i, t0) == 0 ? expf(__fadd_rn(ah[i], al[i])) : 0.f;
  __syncthreads();
  const int64_t ntn = cdiv(s.N, kTC);
  const int64_t p0 = (blockIdx.y / ntn) * 64, n0 = (blockIdx.y % ntn) * kTC;
  const TIn *gc = dout + ((bi * s.T + t0) * s.H + h) * s.P;
  const TIn *cc = Cm + ((bi * s.T + t0) * s.G + g) * s.N;
  const int64_t HP = s.H * s.P, GN = s.G * s.N;
  float acc[4][4];
  tile_mm<4, false, false>(
      Lc, [&](int r, int64_t i) { const int64_t p = p0 + r; return p < s.P ? ea[i] * ld(gc + i * HP + p) : 0.f; },
      [&](int q, int64_t i) { const int64_t n = n0 + q; return n < s.N ? ld(cc + i * GN + n) : 0.f; }, sb, acc);
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t p = p0 + tile_row<4>(a), n = n0 + tile_col(b);
      if (p < s.P && n < s.N) dH[(unit * s.P + p) * s.N + n] = acc[a][b];
    }
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

// Reverse state passing, in place on buf:
//   in:  buf[c] = dHscan_c;  out: buf[c] = dS_c = gradient reaching the end
//   state of chunk c (dH_{c+1}, or 0 where chunk c+1 starts a sequence);
//   dH_c = dHscan_c + exp(E_c) dS_c when the sequence holding the chunk's
//   last token entered the chunk (fe = 0), else dH_c = dHscan_c;
//   dEpass[b,h,c] = exp(E_c) <states_c, dS_c> (fe = 0), or
//   exp(E_c - Acs_{fe-1}) <init[seq], dS_c> (fe >= 1: the carried part of the
//   chunk-end state then starts from that sequence's initial state);
//   dinit[seq] += dH_c where chunk c starts a sequence at its first token.
// The recurrence is elementwise in (p, n): a CTA per (b, h) and slice of
// kPassSlice state elements walks the chunks in reverse with the running dH
// of its elements in registers; dEpass is left as one partial per slice
// (dEpart[b,h,c,slice], the slice's block sum times the decay factor), which
// the cumsum backward adds in slice order.
constexpr int kPassSlice = 4 * kPassThreads;

__global__ void __launch_bounds__(kPassThreads)
    state_passing_bwd_kernel(Shape s, float *__restrict__ buf, const float *__restrict__ states,
                             const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
                             const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first,
                             const float *__restrict__ init, float *__restrict__ dEpart, float *__restrict__ dinit) {
  __shared__ float red[32];
  const int64_t h = blockIdx.x % s.H, bi = blockIdx.x / s.H;
  const int64_t PN = s.P * s.N, nsl = cdiv(PN, kPassSlice), sl = blockIdx.y;
  const int64_t e0 = sl * kPassSlice + threadIdx.x;
  float cr[4] = {0.f, 0.f, 0.f, 0.f};   // dH of the chunk after, per owned element
  // Chunk c's dHscan and carried-in state (the state entering the chunk, or the
  // initial state of the sequence holding its last token) for the owned elements.
  auto hin_of = [&](int64_t c) -> const float * {
    const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
    const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
    return fe == 0 ? states + ((bi * s.nc + c) * s.H + h) * PN
                   : (init ? init + (seq_of(seq_idx, bi, s.T, t0 + Lc - 1) * s.H + h) * PN : nullptr);
  };
  auto load = [&](int64_t c, float (&dh)[4], float (&hv)[4]) {
    const float *bc = buf + ((bi * s.nc + c) * s.H + h) * PN;
    const float *hin = hin_of(c);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t e = e0 + k * kPassThreads;
      dh[k] = e < PN ? bc[e] : 0.f;
      hv[k] = (hin && e < PN) ? hin[e] : 0.f;
    }
  };
  float dh_n[4], hv_n[4];   // the next chunk down, loaded one step ahead
  load(s.nc - 1, dh_n, hv_n);
  for (int64_t c = s.nc - 1; c >= 0; --c) {
    float dh[4], hv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      dh[k] = dh_n[k];
      hv[k] = hv_n[k];
    }
    if (c > 0) load(c - 1, dh_n, hv_n);
    const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
    const bool nxt_start = (c + 1 >= s.nc) || is_seq_start(seq_idx, bi, s.T, (c + 1) * s.Q);
    const bool here_start = is_seq_start(seq_idx, bi, s.T, t0);
    const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
    const int64_t q0 = ((bi * s.H + h) * s.nc + c) * s.Q, q = q0 + (s.Q - 1);
    const float eE = expf(__fadd_rn(acs_hi[q], acs_lo[q]));
    const float eIn = fe == 0 ? eE : expf(acs_diff(acs_hi[q], acs_lo[q], acs_hi[q0 + fe - 1], acs_lo[q0 + fe - 1]));
    const float eCarry = fe == 0 ? eE : 0.f;
    const bool has_hin = hin_of(c) != nullptr;
    float *bc = buf + ((bi * s.nc + c) * s.H + h) * PN;
    float *di = (here_start && dinit) ? dinit + (seq_of(seq_idx, bi, s.T, t0) * s.H + h) * PN : nullptr;
    float part = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t e = e0 + k * kPassThreads;
      if (e >= PN) continue;
      const float cur = nxt_start ? 0.f : cr[k];
      bc[e] = cur;
      if (has_hin) part = fmaf(hv[k], cur, part);
      const float dHc = fmaf(eCarry, cur, dh[k]);
      cr[k] = dHc;
      if (di) di[e] += dHc;
    }
    const float tot = block_sum(part, red);
    if (threadIdx.x == 0) dEpart[((bi * s.H + h) * s.nc + c) * nsl + sl] = eIn * tot;
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
// chunk's last token (i >= fe), else 0.  A CTA per (b, c, h) and 64 x 64 tile
// of (i, p).
template <class TIn>
__global__ void __launch_bounds__(kTileThreads, 3)
    dx_kernel(Shape s, const TIn *__restrict__ dout, const TIn *__restrict__ x, const TIn *__restrict__ Bm,
              const float *__restrict__ dt, const float *__restrict__ D, const float *__restrict__ Mm,
              const float *__restrict__ dS, const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
              const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first, float *__restrict__ dx,
              float *__restrict__ sx_part) {
  __shared__ TileBuf<4> sb;
  const int64_t unit = blockIdx.x;  // (b, c, h)
  const int64_t h = unit % s.H, c = (unit / s.H) % s.nc, bi = unit / (s.H * s.nc);
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0), g = h / s.hpg;
  const int64_t ntp = cdiv(s.P, kTC);
  const int64_t i0 = (blockIdx.y / ntp) * 64, p0 = (blockIdx.y % ntp) * kTC;
  if (i0 >= Lc) return;   // (the whole CTA)
  const float *M = Mm + unit * s.Q * s.Q;
  const TIn *gc = dout + ((bi * s.T + t0) * s.H + h) * s.P;
  const TIn *bc = Bm + ((bi * s.T + t0) * s.G + g) * s.N;
  const float *ds = dS + unit * s.P * s.N;
  const int64_t HP = s.H * s.P, GN = s.G * s.N;
  float d1[4][4], yv[4][4];
  tile_mm<4, false, false>(
      Lc, [&](int r, int64_t j) { const int64_t i = i0 + r; return i < Lc ? M[j * s.Q + i] : 0.f; },
      [&](int q, int64_t j) { const int64_t p = p0 + q; return p < s.P ? ld(gc + j * HP + p) : 0.f; }, sb, d1,
      i0);   // (M[j][i] = 0 for j < i: no row of the tile takes a token before its first row)
  tile_mm<4, true, true>(
      s.N, [&](int r, int64_t n) { const int64_t i = i0 + r; return i < Lc ? ld(bc + i * GN + n) : 0.f; },
      [&](int q, int64_t n) { const int64_t p = p0 + q; return p < s.P ? ds[p * s.N + n] : 0.f; }, sb, yv);
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int64_t i = i0 + tile_row<4>(a);
    if (i >= Lc) continue;
    const int64_t t = t0 + i;
    const float dti = dt[(bi * s.T + t) * s.H + h];
    const float wi = i < fe ? 0.f : expf(acs_diff(ah[Lc - 1], al[Lc - 1], ah[i], al[i])) * dti;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t p = p0 + tile_col(b);
      if (p >= s.P) continue;
      const int64_t idx = ((bi * s.T + t) * s.H + h) * s.P + p;
      dx[idx] = fmaf(dti, d1[a][b], fmaf(wi, yv[a][b], D[h] * ld(dout + idx)));
    }
  }
  // x . Y over this tile's head-dim columns, per token (the decay gradient's u
  // term and ddt's state term take it): the thread's four columns in order,
  // then a fixed xor tree over the 16 threads of the tile row; one partial per
  // (token, column tile), summed in tile order by ddt_dacs_kernel
  const int64_t ntp2 = cdiv(s.P, kTC);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int64_t i = i0 + tile_row<4>(a);
    float v = 0.f;
    if (i < Lc) {
      const TIn *xi = x + ((bi * s.T + t0 + i) * s.H + h) * s.P;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int64_t p = p0 + tile_col(b);
        if (p < s.P) v = fmaf(ld(xi + p), yv[a][b], v);
      }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 15) == 0 && i < s.Q) sx_part[(unit * ntp2 + p0 / kTC) * s.Q + i] = v;
  }
}

// Per-head dB / dC rows of tokens i0 .. i0 + 16 RA - 1 of chunk c, state
// columns n0 .. n0 + 63 (shared by the slot and the ordered fold, so both
// produce the same bits):
//   dC_h[i,n] = sum_{j<=i} W[i,j] B_j[n] + din_i sum_p Hin[p,n] g_i[p]   (kDB false)
//   dB_h[i,n] = sum_{j>=i} W[j,i] C_j[n] + w_i sum_p dS[p,n] x_i[p]      (kDB true)
// (din_i, Hin as in chunk_scan_fwd; w_i as in dx_kernel; fr[r]: local start
// of row i0 + r).
template <bool kDB, int RA, class TIn>
__device__ __forceinline__ void dbdc_tile(const Shape &s, const TIn *__restrict__ x, const TIn *__restrict__ dout,
                                          const TIn *__restrict__ Bm, const TIn *__restrict__ Cm,
                                          const float *__restrict__ dt, const float *__restrict__ Wm,
                                          const float *__restrict__ states, const float *__restrict__ dS,
                                          const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
                                          const int32_t *__restrict__ seq_idx, const float *__restrict__ init,
                                          int64_t bi, int64_t c, int64_t h, int64_t i0, int64_t n0, const int *fr,
                                          int64_t fe, TileBuf<RA> &sb, float (&res)[RA][4]) {
  const int64_t g = h / s.hpg, t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
  const int64_t unit = (bi * s.nc + c) * s.H + h;
  const int64_t HP = s.H * s.P, GN = s.G * s.N;
  const float *W = Wm + unit * s.Q * s.Q;
  const float *ah = acs_hi + ((bi * s.H + h) * s.nc + c) * s.Q;
  const float *al = acs_lo + ((bi * s.H + h) * s.nc + c) * s.Q;
  float t1[RA][4];
  auto row_ok = [&](int r) { return i0 + r < Lc; };
  if (!kDB) {
    const TIn *bc = Bm + ((bi * s.T + t0) * s.G + g) * s.N;
    const TIn *gc = dout + ((bi * s.T + t0) * s.H + h) * s.P;
    const float *hst = states + unit * s.P * s.N;
    tile_mm<RA, true, false>(
        min(Lc, i0 + 16 * RA),   // (W[i][j] = 0 for j > i)
        [&](int r, int64_t j) { return row_ok(r) ? W[(i0 + r) * s.Q + j] : 0.f; },
        [&](int q, int64_t j) { const int64_t n = n0 + q; return n < s.N ? ld(bc + j * GN + n) : 0.f; }, sb, res);
    tile_mm<RA, true, false>(
        s.P, [&](int r, int64_t p) { return row_ok(r) ? ld(gc + (i0 + r) * HP + p) : 0.f; },
        [&](int q, int64_t p) { const int64_t n = n0 + q; return n < s.N ? hst[p * s.N + n] : 0.f; }, sb, t1);
#pragma unroll
    for (int a = 0; a < RA; ++a) {
      const int64_t i = i0 + tile_row<RA>(a);
      if (i >= Lc) continue;
      const int64_t f = fr[tile_row<RA>(a)];
      const float din = expf(f == 0 ? __fadd_rn(ah[i], al[i]) : acs_diff(ah[i], al[i], ah[f - 1], al[f - 1]));
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int64_t n = n0 + tile_col(b);
        if (n >= s.N) continue;
        float hg = t1[a][b];
        if (f > 0) {   // a sequence that started inside the chunk: its own initial state
          hg = 0.f;
          if (init) {
            const float *hs = init + (seq_of(seq_idx, bi, s.T, t0 + i) * s.H + h) * s.P * s.N + n;
            const TIn *gi = gc + i * HP;
            for (int64_t p = 0; p < s.P; ++p) hg = fmaf(hs[p * s.N], ld(gi + p), hg);
          }
        }
        res[a][b] = fmaf(din, hg, res[a][b]);
      }
    }
  } else {
    const TIn *cc = Cm + ((bi * s.T + t0) * s.G + g) * s.N;
    const TIn *xc = x + ((bi * s.T + t0) * s.H + h) * s.P;
    const float *ds = dS + unit * s.P * s.N;
    tile_mm<RA, false, false>(
        Lc, [&](int r, int64_t j) { return row_ok(r) ? W[j * s.Q + i0 + r] : 0.f; },
        [&](int q, int64_t j) { const int64_t n = n0 + q; return n < s.N ? ld(cc + j * GN + n) : 0.f; }, sb, res,
        i0);   // (W[j][i] = 0 for j < i)
    tile_mm<RA, true, false>(
        s.P, [&](int r, int64_t p) { return row_ok(r) ? ld(xc + (i0 + r) * HP + p) : 0.f; },
        [&](int q, int64_t p) { const int64_t n = n0 + q; return n < s.N ? ds[p * s.N + n] : 0.f; }, sb, t1);
#pragma unroll
    for (int a = 0; a < RA; ++a) {
      const int64_t i = i0 + tile_row<RA>(a);
      if (i >= Lc) continue;
      const float wi =
          i < fe ? 0.f : expf(acs_diff(ah[Lc - 1], al[Lc - 1], ah[i], al[i])) * dt[(bi * s.T + t0 + i) * s.H + h];
#pragma unroll
      for (int b = 0; b < 4; ++b) res[a][b] = fmaf(wi, t1[a][b], res[a][b]);
    }
  }
}

// Deterministic variant: per-head slots (b,T,H,N); atomic variant: added into
// dB/dC (b,T,G,N) with atomics.  A CTA per (b, c, h), 64 x 64 tile of (i, n)
// and output (blockIdx.z: 0 dC, 1 dB).
template <class TIn, bool kAtomic>
__global__ void __launch_bounds__(kTileThreads, 3)
    dbdc_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ dout, const TIn *__restrict__ Bm,
                const TIn *__restrict__ Cm, const float *__restrict__ dt, const float *__restrict__ Wm,
                const float *__restrict__ states, const float *__restrict__ dS, const float *__restrict__ acs_hi,
                const float *__restrict__ acs_lo, const int32_t *__restrict__ seq_idx,
                const int32_t *__restrict__ first, const float *__restrict__ init, float *__restrict__ dBo,
                float *__restrict__ dCo) {
  __shared__ TileBuf<4> sb;
  __shared__ int fr[64];
  const int64_t unit = blockIdx.x;  // (b, c, h)
  const int64_t h = unit % s.H, c = (unit / s.H) % s.nc, bi = unit / (s.H * s.nc);
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0), g = h / s.hpg;
  const int64_t ntn = cdiv(s.N, kTC);
  const int64_t i0 = (blockIdx.y / ntn) * 64, n0 = (blockIdx.y % ntn) * kTC;
  if (i0 >= Lc) return;   // (the whole CTA)
  for (int r = threadIdx.x; r < 64; r += blockDim.x)
    fr[r] = i0 + r < Lc ? int(local_start(seq_idx, first, bi, s.T, t0 + i0 + r, t0)) : 0;
  __syncthreads();
  const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
  const bool is_db = blockIdx.z != 0;
  float res[4][4];
  if (is_db)
    dbdc_tile<true, 4, TIn>(s, x, dout, Bm, Cm, dt, Wm, states, dS, acs_hi, acs_lo, seq_idx, init, bi, c, h, i0, n0,
                            fr, fe, sb, res);
  else
    dbdc_tile<false, 4, TIn>(s, x, dout, Bm, Cm, dt, Wm, states, dS, acs_hi, acs_lo, seq_idx, init, bi, c, h, i0, n0,
                             fr, fe, sb, res);
  float *out = is_db ? dBo : dCo;
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t i = i0 + tile_row<4>(a), n = n0 + tile_col(b);
      if (i >= Lc || n >= s.N) continue;
      const int64_t t = t0 + i;
      if (kAtomic)
        atomicAdd(out + ((bi * s.T + t) * s.G + g) * s.N + n, res[a][b]);
      else
        out[((bi * s.T + t) * s.H + h) * s.N + n] = res[a][b];
    }
}

// Tokens per tile of the ordered dB/dC fold: 64 (the slot path's tile, four
// rows a thread) where the tile's rows of dB and dC (2 x 64 x dstate fp32) fit
// three CTAs an SM, else 32.  The tile shape does not change any output's bits.
inline int ord_tile(const Shape &s) { return s.N <= 128 ? 64 : 32; }

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
// The CTA computes its tile's per-head dB/dC rows with dbdc_tile (the same
// terms in the same order as the slot fold) into shared memory, waits until
// the tile's semaphore reads k (a bounded spin: past spin_limit polls it sets
// status bit 1 and skips its add), then stores (k = 0) or adds its rows into
// dB/dC, and releases the semaphore to k + 1.
template <class TIn, int OT>
__global__ void __launch_bounds__(kTileThreads, 2)
    dbdc_ordered_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ dout, const TIn *__restrict__ Bm,
                        const TIn *__restrict__ Cm, const float *__restrict__ dt, const float *__restrict__ Wm,
                        const float *__restrict__ states, const float *__restrict__ dS,
                        const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
                        const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first,
                        const float *__restrict__ init, int *__restrict__ status, int *__restrict__ sem,
                        uint32_t spin_limit, float *__restrict__ dBo, float *__restrict__ dCo) {
  extern __shared__ float tile[];   // [2][OT][N]: dB rows then dC rows
  __shared__ TileBuf<OT / 16> sb;
  __shared__ int fr[OT];
  __shared__ int s_unit, s_go;
  if (threadIdx.x == 0) s_unit = atomicAdd(status + 1, 1);
  __syncthreads();
  const int64_t ntt = cdiv(s.Q, OT);
  const int64_t unit = s_unit;
  // tickets head-major over the tiles: a head's predecessor on the same tile drew its ticket one
  // sweep of the tiles earlier, so it has usually released the tile by the time this CTA waits
  const int64_t ntiles = s.b * s.nc * s.G * ntt;
  const int64_t k = unit / ntiles, tileid = unit % ntiles;
  const int64_t tt = tileid % ntt, g = (tileid / ntt) % s.G, c = (tileid / (ntt * s.G)) % s.nc;
  const int64_t bi = tileid / (ntt * s.G * s.nc);
  const int64_t h = g * s.hpg + k, t0 = c * s.Q, Lc = min(s.Q, s.T - t0);
  const int64_t i0 = tt * OT, i1 = min(Lc, i0 + OT);
  for (int r = threadIdx.x; r < OT; r += blockDim.x)
    fr[r] = i0 + r < Lc ? int(local_start(seq_idx, first, bi, s.T, t0 + i0 + r, t0)) : 0;
  __syncthreads();
  const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
  if (i0 < Lc) {   // (the whole CTA)
    for (int64_t n0 = 0; n0 < s.N; n0 += kTC) {
      float dcv[OT / 16][4], dbv[OT / 16][4];
      dbdc_tile<false, OT / 16, TIn>(s, x, dout, Bm, Cm, dt, Wm, states, dS, acs_hi, acs_lo, seq_idx, init, bi,
                                           c, h, i0, n0, fr, fe, sb, dcv);
      dbdc_tile<true, OT / 16, TIn>(s, x, dout, Bm, Cm, dt, Wm, states, dS, acs_hi, acs_lo, seq_idx, init, bi,
                                          c, h, i0, n0, fr, fe, sb, dbv);
#pragma unroll
      for (int a = 0; a < OT / 16; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int64_t r = tile_row<OT / 16>(a), n = n0 + tile_col(b);
          if (n >= s.N) continue;
          tile[r * s.N + n] = dbv[a][b];
          tile[OT * s.N + r * s.N + n] = dcv[a][b];
        }
    }
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
    const float db = tile[e], dc = tile[OT * s.N + e];
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
// decay exp(Acs_i - Acs_{f-1}) also depends on Acs_{f-1}), else 0.  The MG
// sums come from mwg_kernel's tile parts (tiles in ascending order).  A CTA
// per (b, c, h) and 64 tokens: the products C Hin^T and B dS^T of its tokens
// come out of tile products (64 state columns p at a time); four threads per
// token each sum a quarter of every p tile, p ascending, and the quarters are
// added in a fixed tree.
template <class TIn>
__global__ void __launch_bounds__(kTileThreads, 3)
    ddt_dacs_kernel(Shape s, const TIn *__restrict__ x, const TIn *__restrict__ dout, const TIn *__restrict__ Bm,
                    const TIn *__restrict__ Cm, const float *__restrict__ dt, const float *__restrict__ rowp,
                    const float *__restrict__ colp, const float *__restrict__ dg, const float *__restrict__ states,
                    const float *__restrict__ dS, const float *__restrict__ acs_hi, const float *__restrict__ acs_lo,
                    const int32_t *__restrict__ seq_idx, const int32_t *__restrict__ first,
                    const float *__restrict__ init, const float *__restrict__ sx_part, float *__restrict__ ddt_part,
                    float *__restrict__ dAcs, float *__restrict__ u_buf, float *__restrict__ gx_buf,
                    float *__restrict__ vin_buf) {
  __shared__ TileBuf<4> sb;
  __shared__ float chs[64][kTC + 1];
  const int64_t unit = blockIdx.x;  // (b, c, h)
  const int64_t h = unit % s.H, c = (unit / s.H) % s.nc, bi = unit / (s.H * s.nc);
  const int64_t t0 = c * s.Q, Lc = min(s.Q, s.T - t0), g = h / s.hpg;
  const int64_t i0 = int64_t(blockIdx.y) * 64;
  const int64_t GN = s.G * s.N;
  const TIn *cc = Cm + ((bi * s.T + t0) * s.G + g) * s.N;
  const float *hst = states + unit * s.P * s.N;
  // this thread's token and quarter of the state columns
  const int r = threadIdx.x >> 2, part = threadIdx.x & 3;
  const int64_t i = i0 + r, t = t0 + i;
  const bool mine = i < Lc;
  const int64_t f = mine ? local_start(seq_idx, first, bi, s.T, t, t0) : 0;
  const float *hsi = nullptr;   // initial state of a sequence that started inside the chunk
  if (mine && f > 0 && init) hsi = init + (seq_of(seq_idx, bi, s.T, t) * s.H + h) * s.P * s.N;
  const TIn *gi = dout + ((bi * s.T + t) * s.H + h) * s.P;
  const TIn *xi = x + ((bi * s.T + t) * s.H + h) * s.P;
  const TIn *ci = cc + i * GN;
  float inter = 0.f, sx = 0.f, gx = 0.f;
  if (i0 < Lc) {   // (the whole CTA)
    for (int64_t p0 = 0; p0 < s.P; p0 += kTC) {
      float acc[4][4];
      tile_mm<4, true, true>(
          s.N, [&](int rr, int64_t n) { const int64_t ii = i0 + rr; return ii < Lc ? ld(cc + ii * GN + n) : 0.f; },
          [&](int q, int64_t n) { const int64_t p = p0 + q; return p < s.P ? hst[p * s.N + n] : 0.f; }, sb, acc);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) chs[tile_row<4>(a)][tile_col(b)] = acc[a][b];
      __syncthreads();
      if (mine) {
        const int64_t pe = min(int64_t(kTC), s.P - p0);
        for (int64_t pp = 16 * part; pp < min(pe, int64_t(16 * part + 16)); ++pp) {
          const int64_t p = p0 + pp;
          float hc = chs[r][pp];
          if (f > 0) {   // a sequence that started inside the chunk: its own initial state
            hc = 0.f;
            if (hsi)
              for (int64_t n = 0; n < s.N; ++n) hc = fmaf(hsi[p * s.N + n], ld(ci + n), hc);
          }
          const float gp = ld(gi + p), xp = ld(xi + p);
          inter = fmaf(gp, hc, inter);
          gx = fmaf(gp, xp, gx);
        }
      }
      __syncthreads();
    }
  }
  // the four quarters of each token (lanes 4 r .. 4 r + 3 of one warp), fixed tree
  inter += __shfl_xor_sync(0xffffffffu, inter, 1);
  gx += __shfl_xor_sync(0xffffffffu, gx, 1);
  inter += __shfl_xor_sync(0xffffffffu, inter, 2);
  gx += __shfl_xor_sync(0xffffffffu, gx, 2);
  if (part != 0 || i >= s.Q) return;
  const int64_t idx = ((bi * s.H + h) * s.nc + c) * s.Q + i;
  if (i >= Lc) {
    dAcs[idx] = 0.f;
    u_buf[idx] = 0.f;
    gx_buf[idx] = 0.f;
    vin_buf[idx] = 0.f;
    return;
  }
  const int64_t nt = cdiv(s.Q, 64);
  float col = 0.f, row = 0.f;
  for (int64_t k = 0; k < nt; ++k) {
    row += rowp[(unit * nt + k) * s.Q + i];
    col += colp[(unit * nt + k) * s.Q + i];
  }
  const float diag = dg[unit * s.Q + i];
  // x . Y: the per-column-tile partials of dx_kernel, in tile order
  const int64_t ntp = cdiv(s.P, kTC);
  for (int64_t k = 0; k < ntp; ++k) sx += sx_part[(unit * ntp + k) * s.Q + i];
  const float *dtc = dt + (bi * s.T + t0) * s.H + h;  // dtc[j * H]
  const float dti = dtc[i * s.H];
  const int64_t fe = local_start(seq_idx, first, bi, s.T, t0 + Lc - 1, t0);
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
  const int64_t nsl = cdiv(s.P * s.N, kPassSlice);
  float dEp = 0.f;   // the slices' parts of exp(E) <Hin, dS>, in slice order
  for (int64_t k = 0; k < nsl; ++k) dEp += dEpass[((bi * s.H + h) * s.nc + c) * nsl + k];
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
  dA[h] = column_sum(dA_part + h, s.b * s.nc, s.H, 0.f);
  dD[h] = column_sum(dD_part + h, s.b * s.nc, s.H, 0.f);
}

struct BwdWs {
  int *status;   // [0] error bits (bit 1: an ordered-fold wait gave up), [1] ticket; first in the workspace
  float *acs_hi, *acs_lo, *CB, *Mm, *Wm, *rowp, *colp, *dg, *sx_part, *buf, *dEpass, *dAcs, *u, *gx, *vin, *ddt_part, *dA_part,
      *dD_part, *slot_b, *slot_c;
  int32_t *first;
  int *sem;
};

int64_t ordered_tiles(const Shape &s) { return s.b * s.nc * s.G * cdiv(s.Q, ord_tile(s)); }

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
  const int64_t parts = s.b * s.nc * s.H * cdiv(s.Q, 64) * s.Q;   // MG sums, per 64-wide tile
  w.rowp = cv.take<float>(parts);
  w.colp = cv.take<float>(parts);
  w.dg = cv.take<float>(s.b * s.nc * s.H * s.Q);
  w.sx_part = cv.take<float>(s.b * s.nc * s.H * cdiv(s.P, kTC) * s.Q);
  w.buf = cv.take<float>(s.b * s.nc * s.H * s.P * s.N);
  w.dEpass = cv.take<float>(s.b * s.H * s.nc * cdiv(s.P * s.N, kPassSlice));
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
  const unsigned nbch = unsigned(s.b * s.nc * s.H);
  const unsigned tiles_pn = unsigned(cdiv(s.P, 64) * cdiv(s.N, kTC)), tiles_qq = unsigned(cdiv(s.Q, 64) * cdiv(s.Q, 64));
  const unsigned tiles_qp = unsigned(cdiv(s.Q, 64) * cdiv(s.P, kTC));
  chunk_state_fwd_kernel<TIn><<<dim3(nbch, tiles_pn), kTileThreads, s.Q * sizeof(float), st>>>(
      s, x, Bm, a.dt, w.acs_hi, w.acs_lo, a.seq_idx, first, w.S);
  state_passing_fwd_kernel<<<grid1(s.b * s.H * s.P * s.N, bs), bs, 0, st>>>(s, w.S, w.acs_hi, w.acs_lo, a.seq_idx,
                                                                            first, a.init, a.states_out);
  cb_kernel<TIn><<<dim3(unsigned(s.b * s.nc * s.G), tiles_qq), kTileThreads, 0, st>>>(s, Bm, Cm, w.CB);
  chunk_scan_fwd_kernel<TIn><<<dim3(nbch, tiles_qp), kTileThreads, 0, st>>>(
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
  const unsigned tiles_pn = unsigned(cdiv(s.P, 64) * cdiv(s.N, kTC)), tiles_qq = unsigned(cdiv(s.Q, 64) * cdiv(s.Q, 64));
  const unsigned tiles_qp = unsigned(cdiv(s.Q, 64) * cdiv(s.P, kTC)), tiles_qn = unsigned(cdiv(s.Q, 64) * cdiv(s.N, kTC));
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
  cb_kernel<TIn><<<dim3(unsigned(s.b * s.nc * s.G), tiles_qq), kTileThreads, 0, st>>>(s, Bm, Cm, w.CB);
  tr.mark(st);
  tr.mark(st);
  mwg_kernel<TIn><<<dim3(nbch, tiles_qq), kTileThreads, 0, st>>>(s, x, g, a.dt, w.CB, w.acs_hi, w.acs_lo, a.seq_idx,
                                                                  first, w.Mm, w.Wm, w.rowp, w.colp, w.dg);
  tr.mark(st);
  tr.mark(st);
  dhscan_kernel<TIn><<<dim3(nbch, tiles_pn), kTileThreads, s.Q * sizeof(float), st>>>(s, g, Cm, w.acs_hi, w.acs_lo,
                                                                                      a.seq_idx, first, w.buf);
  tr.mark(st);
  tr.mark(st);
  // fixed block: this kernel folds per-thread partial dot products, so its
  // shape must not follow the launch configuration
  state_passing_bwd_kernel<<<dim3(unsigned(s.b * s.H), unsigned(cdiv(PN, kPassSlice))), kPassThreads, 0, st>>>(
      s, w.buf, a.states_in, w.acs_hi, w.acs_lo, a.seq_idx, first, a.init, w.dEpass, a.dinit);
  tr.mark(st);
  if (a.seq_idx) {
    tr.mark(st);
    dinit_mid_kernel<TIn><<<grid1(s.nseq * s.H * PN, bs), bs, 0, st>>>(s, g, Cm, w.acs_hi, w.acs_lo, a.seq_idx,
                                                                       first, w.buf, a.dinit);
    tr.mark(st);
  }
  tr.mark(st);
  dx_kernel<TIn><<<dim3(nbch, tiles_qp), kTileThreads, 0, st>>>(s, g, x, Bm, a.dt, a.D, w.Mm, w.buf, w.acs_hi,
                                                                w.acs_lo, a.seq_idx, first, a.dx, w.sx_part);
  tr.mark(st);
  if (atomic) {
    tr.mark(st);
    dbdc_kernel<TIn, true><<<dim3(nbch, tiles_qn, 2), kTileThreads, 0, st>>>(
        s, x, g, Bm, Cm, a.dt, w.Wm, a.states_in, w.buf, w.acs_hi, w.acs_lo, a.seq_idx, first, a.init, a.dB, a.dC);
    tr.mark(st);
  } else if (ordered) {
    tr.mark(st);
    const int64_t units = ordered_tiles(s) * s.hpg;
    const int ot = ord_tile(s);
    const size_t shm = size_t(2 * ot * s.N) * sizeof(float);
    // (the kernel's static tile buffers come on top of this)
    auto kern = ot == 64 ? dbdc_ordered_kernel<TIn, 64> : dbdc_ordered_kernel<TIn, 32>;
    if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(shm))) != cudaSuccess)
      return err;
    kern<<<unsigned(units), kTileThreads, shm, st>>>(s, x, g, Bm, Cm, a.dt, w.Wm, a.states_in, w.buf, w.acs_hi,
                                                     w.acs_lo, a.seq_idx, first, a.init, w.status, w.sem,
                                                     spin_limit, a.dB, a.dC);
    tr.mark(st);
  } else {
    tr.mark(st);
    dbdc_kernel<TIn, false><<<dim3(nbch, tiles_qn, 2), kTileThreads, 0, st>>>(
        s, x, g, Bm, Cm, a.dt, w.Wm, a.states_in, w.buf, w.acs_hi, w.acs_lo, a.seq_idx, first, a.init, w.slot_b,
        w.slot_c);
    tr.mark(st);
  }
  tr.mark(st);
  ddt_dacs_kernel<TIn><<<dim3(nbch, unsigned(cdiv(s.Q, 64))), kTileThreads, 0, st>>>(
      s, x, g, Bm, Cm, a.dt, w.rowp, w.colp, w.dg, a.states_in, w.buf, w.acs_hi, w.acs_lo, a.seq_idx, first, a.init,
      w.sx_part, w.ddt_part, w.dAcs, w.u, w.gx, w.vin);
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
