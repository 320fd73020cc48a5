// ssd_padded.cu -- packed batches whose sequences start inside a chunk, run
// on the tensor-core forward and backward.
//
// The recurrence h_t = exp(dt_t A) h_{t-1} + dt_t B_t x_t^T, y_t = C_t h_t +
// D x_t ("Mamba2 / state space duality": the SSM recurrence; the state resets
// to the sequence's initial state, or zero, at each sequence start) leaves
// the state unchanged across a token with dt = 0 and x = B = C = 0: the decay
// is exp(0) = 1, the input term is 0, and its y is 0.  With dout = 0 there as
// well, such a token adds nothing to any gradient of the real tokens (its
// dt factor makes its share of dA exactly 0).  So the token stream is cut at
// every sequence start and every 128-token boundary; each piece (at most 128
// tokens of one sequence) becomes one 128-token chunk of a padded problem,
// its tokens first and padding tokens after.  In the padded problem every
// sequence starts on a chunk start -- the form the fused kernels handle --
// and it has the same y, the same gradients at the real tokens, and the same
// state entering every chunk of the caller's chunking (those chunk starts are
// multiples of 128, so each begins a piece).
//
// The number of pieces is at most ceil(T / 128) + nseq - 1 (one per 128-token
// chunk plus one per sequence start inside one); the padded problem always
// has that many chunks, so every size follows from the dims alone.  Unused
// trailing chunks hold padding only and carry the last sequence's id.
//
// Forward workspace (kept until the backward, which reads the padded inputs
// and the packed states from it): the piece table, the padded seq_idx, x,
// dt, B, C and y, the packed states (dstate 128) and the inner forward's
// workspace.  Backward workspace: the inner backward's workspace first (its
// status word at offset 0, where the status check reads it), then the padded
// dout and the padded gradients, scattered back to the caller's rows.
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "ssd_internal.h"
#include "tile_io.cuh"

namespace ssd {
namespace {

constexpr int kRows = 128;   // tokens per padded chunk
constexpr int kP = 64, kN = 128;

struct PadTables {
  const int32_t *start, *len, *id;   // per padded chunk: first caller token, real tokens, sequence id
};

struct PadFwdWs {
  int32_t *start, *len, *id, *map;   // piece table (npc each) and caller chunk -> padded chunk (nc)
  int32_t *seq;                      // padded seq_idx (Tp)
  __nv_bfloat16 *x, *B, *C, *y;      // padded token rows
  float *dt;
  float *packed;                     // dstate 128: packed states (npc, H) tiles; else null
  void *inner;                       // the inner forward's workspace
};

PadFwdWs carve_pad_fwd(Carver &cv, const Shape &s, bool split) {
  const Shape p = padded_shape(s);
  PadFwdWs w;
  int32_t *tab = cv.take<int32_t>(3 * p.nc);   // start | len | id, uploaded as one block
  w.start = tab;
  w.len = tab ? tab + p.nc : nullptr;
  w.id = tab ? tab + 2 * p.nc : nullptr;
  w.map = cv.take<int32_t>(s.nc);
  w.seq = cv.take<int32_t>(p.T);
  w.x = cv.take<__nv_bfloat16>(p.T * s.H * s.P);
  w.y = cv.take<__nv_bfloat16>(p.T * s.H * s.P);
  w.B = cv.take<__nv_bfloat16>(p.T * s.G * s.N);
  w.C = cv.take<__nv_bfloat16>(p.T * s.G * s.N);
  w.dt = cv.take<float>(p.T * s.H);
  w.packed = split ? nullptr : cv.take<float>(p.nc * s.H * s.P * s.N);
  const size_t inner = split ? fused_fwd_split_workspace(p) : fused_fwd_workspace(p);
  w.inner = cv.take<char>(int64_t(inner));
  return w;
}

struct PadBwdWs {
  void *inner;                       // the inner backward's workspace (offset 0)
  __nv_bfloat16 *dout;
  float *dx, *ddt, *dB, *dC;
};

PadBwdWs carve_pad_bwd(Carver &cv, const Shape &s, bool split, int ring_depth) {
  const Shape p = padded_shape(s);
  PadBwdWs w;
  const size_t inner = split ? fused_bwd_split_workspace(p, ring_depth) : fused_bwd_workspace(p, ring_depth);
  w.inner = cv.take<char>(int64_t(inner));
  w.dout = cv.take<__nv_bfloat16>(p.T * s.H * s.P);
  w.dx = cv.take<float>(p.T * s.H * s.P);
  w.ddt = cv.take<float>(p.T * s.H);
  w.dB = cv.take<float>(p.T * s.G * s.N);
  w.dC = cv.take<float>(p.T * s.G * s.N);
  return w;
}

// ---------------------------------------------------------------------------
// Row moves between the caller's token rows and the padded ones.  One set is
// one token-major tensor (rows of `bytes`, a multiple of 4); a CTA moves
// `rows` consecutive rows of one padded chunk (rows * bytes about 64 KB), its
// 256 threads split into groups of `lanes` (a power of two) per row.
struct RowSet {
  const void *src;
  void *dst;
  int64_t bytes;
  int rows, lanes;
};
constexpr int kMaxSets = 4;
struct RowSets {
  RowSet set[kMaxSets];
  int count;
};

RowSet row_set(const void *src, void *dst, int64_t bytes) {
  RowSet r;
  r.src = src;
  r.dst = dst;
  r.bytes = bytes;
  int rows = 1;
  while (rows < kRows && int64_t(rows) * 2 * bytes <= 65536) rows *= 2;
  r.rows = rows;
  const int64_t vecs = bytes % 16 == 0 ? bytes / 16 : bytes / 4;
  int lanes = 1;
  while (lanes < 256 && lanes < vecs) lanes *= 2;
  r.lanes = lanes;
  return r;
}

template <class V, bool kGather>
__device__ __forceinline__ void move_rows(const RowSet &rs, const PadTables &t, int64_t k, int r0) {
  const int64_t nv = rs.bytes / int64_t(sizeof(V));
  const int lane = threadIdx.x & (rs.lanes - 1), ro = threadIdx.x / rs.lanes, rp = blockDim.x / rs.lanes;
  const int len = t.len[k];
  const int64_t first = t.start[k];
  const V *src = static_cast<const V *>(rs.src);
  V *dst = static_cast<V *>(rs.dst);
  for (int r = r0 + ro; r < r0 + rs.rows; r += rp) {
    const int64_t padded = k * kRows + r, caller = first + r;
    if (kGather) {
      V *d = dst + padded * nv;
      if (r < len) {
        const V *sp = src + caller * nv;
        for (int64_t i = lane; i < nv; i += rs.lanes) d[i] = __ldg(sp + i);
      } else {
        for (int64_t i = lane; i < nv; i += rs.lanes) d[i] = V{};
      }
    } else if (r < len) {
      const V *sp = src + padded * nv;
      V *d = dst + caller * nv;
      for (int64_t i = lane; i < nv; i += rs.lanes) d[i] = __ldg(sp + i);
    }
  }
}

// Gather (caller rows -> padded rows, padding rows zero) or scatter (padded
// rows -> caller rows, padding rows dropped).  blockIdx.y picks the set; with
// `seq` set, the CTAs of the extra y index write the padded seq_idx.
template <bool kGather>
__global__ void __launch_bounds__(256) pad_rows_kernel(RowSets sets, PadTables t, int64_t npc, int32_t *seq) {
  if (int(blockIdx.y) == sets.count) {   // padded seq_idx: every token of chunk k carries its piece's id
    const int64_t k = blockIdx.x;
    if (k < npc && threadIdx.x < kRows) seq[k * kRows + threadIdx.x] = t.id[k];
    return;
  }
  const RowSet rs = sets.set[blockIdx.y];
  const int per_chunk = kRows / rs.rows;
  if (int64_t(blockIdx.x) >= npc * per_chunk) return;
  const int64_t k = blockIdx.x / per_chunk;
  const int r0 = int(blockIdx.x % per_chunk) * rs.rows;
  if (rs.bytes % 16 == 0)
    move_rows<uint4, kGather>(rs, t, k, r0);
  else
    move_rows<uint32_t, kGather>(rs, t, k, r0);
}

template <bool kGather>
cudaError_t launch_rows(const RowSets &sets, const PadTables &t, int64_t npc, int32_t *seq, cudaStream_t st) {
  int64_t ctas = seq ? npc : 0;
  for (int i = 0; i < sets.count; ++i) {
    const int64_t c = npc * (kRows / sets.set[i].rows);
    if (c > ctas) ctas = c;
  }
  const dim3 grid(unsigned(ctas), unsigned(sets.count + (seq ? 1 : 0)));
  pad_rows_kernel<kGather><<<grid, 256, 0, st>>>(sets, t, npc, seq);
  return cudaGetLastError();
}

// fp32 (nc, H, P, halves * 128) states entering each caller chunk from the
// packed state tiles of the padded problem ([half][npc][H] tiles of P x 128:
// bf16 hi then lo, each [128][64] in the 128-byte swizzled operand layout);
// one CTA per (caller chunk, head, half).
__global__ void __launch_bounds__(256) pad_states_view_kernel(int64_t H, int halves, int64_t npc,
                                                               const int32_t *__restrict__ map,
                                                               const float *__restrict__ packed,
                                                               float *__restrict__ out) {
  __shared__ float t[64][129];
  const int64_t tile = blockIdx.x;
  const int j = int(tile % halves);
  const int64_t h = (tile / halves) % H, c = tile / halves / H;
  const uint8_t *in = reinterpret_cast<const uint8_t *>(packed + ((j * npc + map[c]) * H + h) * (kP * kN));
  const int64_t pitch = int64_t(halves) * kN;
  unpack_state_tile(in, out + (c * H + h) * kP * pitch + j * kN, pitch, t);
}

PadTables tables_of(const PadFwdWs &f) { return PadTables{f.start, f.len, f.id}; }

}  // namespace

int64_t padded_chunks(const Shape &s) { return (s.T + kRows - 1) / kRows + s.nseq - 1; }

Shape padded_shape(const Shape &s) {
  Shape p = s;
  p.b = 1;
  p.Q = kRows;
  p.nc = padded_chunks(s);
  p.T = p.nc * kRows;
  return p;
}

bool build_piece_table(const Shape &s, const int32_t *seq, std::vector<int32_t> &tab) {
  const int64_t npc = padded_chunks(s);
  tab.assign(size_t(3 * npc + s.nc), 0);
  int32_t *start = tab.data(), *len = start + npc, *id = len + npc, *map = id + npc;
  int64_t k = 0;
  for (int64_t t = 0; t < s.T; ++t) {
    if (t % kRows == 0 || seq[t] != seq[t - 1]) {   // a new piece
      if (k >= npc) return false;                   // more sequence starts than nseq allows
      start[k] = int32_t(t);
      id[k] = seq[t];
      if (t % s.Q == 0) map[t / s.Q] = int32_t(k);
      ++k;
    }
    ++len[k - 1];
  }
  for (; k < npc; ++k) {   // trailing chunks: padding only, inside the last sequence
    start[k] = int32_t(s.T);
    id[k] = seq[s.T - 1];
  }
  return true;
}

size_t padded_fwd_workspace(const Shape &s, bool split) {
  Carver cv(nullptr);
  carve_pad_fwd(cv, s, split);
  return cv.bytes();
}

int *padded_fwd_status(const Shape &s, bool split, void *ws) {
  Carver cv(ws);
  void *inner = carve_pad_fwd(cv, s, split).inner;
  const Shape p = padded_shape(s);
  return split ? fused_fwd_split_status(p, inner) : fused_fwd_status(p, inner);
}

size_t padded_bwd_workspace(const Shape &s, bool split, int ring_depth) {
  Carver cv(nullptr);
  carve_pad_bwd(cv, s, split, ring_depth);
  return cv.bytes();
}

cudaError_t padded_fwd(const Shape &s, bool split, const Args &a, const int32_t *host_seq, void *ws,
                       cudaStream_t st) {
  const Shape p = padded_shape(s);
  Carver cv(ws);
  const PadFwdWs f = carve_pad_fwd(cv, s, split);
  std::vector<int32_t> tab;
  if (!build_piece_table(s, host_seq, tab)) return cudaErrorInvalidValue;
  // (pageable source: the call returns once the table is staged, so `tab` may go)
  cudaError_t err = cudaMemcpyAsync(f.start, tab.data(), size_t(3 * p.nc) * sizeof(int32_t),
                                    cudaMemcpyHostToDevice, st);
  if (err == cudaSuccess)
    err = cudaMemcpyAsync(f.map, tab.data() + 3 * p.nc, size_t(s.nc) * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (err != cudaSuccess) return err;
  const PadTables t = tables_of(f);
  RowSets in{};
  in.set[0] = row_set(a.x, f.x, s.H * s.P * 2);
  in.set[1] = row_set(a.dt, f.dt, s.H * 4);
  in.set[2] = row_set(a.B, f.B, s.G * s.N * 2);
  in.set[3] = row_set(a.C, f.C, s.G * s.N * 2);
  in.count = 4;
  if ((err = launch_rows<true>(in, t, p.nc, f.seq, st)) != cudaSuccess) return err;
  Args ai{};
  ai.x = f.x; ai.B = f.B; ai.C = f.C; ai.dt = f.dt; ai.A = a.A; ai.D = a.D;
  ai.init = a.init; ai.seq_idx = f.seq; ai.y = f.y;
  ai.states_out = f.packed;   // null on the split form: its packed states stay in its own workspace
  if ((err = split ? fused_fwd_split(p, ai, f.inner, st) : fused_fwd(p, ai, f.inner, st)) != cudaSuccess) return err;
  RowSets out{};
  out.set[0] = row_set(f.y, a.y, s.H * s.P * 2);
  out.count = 1;
  if ((err = launch_rows<false>(out, t, p.nc, nullptr, st)) != cudaSuccess) return err;
  const int halves = int(s.N / kN);
  const float *packed = split ? fused_split_aux(p, f.inner) : f.packed;
  pad_states_view_kernel<<<unsigned(s.nc * s.H * halves), 256, 0, st>>>(s.H, halves, p.nc, f.map, packed,
                                                                          a.states_out);
  return cudaGetLastError();
}

cudaError_t padded_bwd(const Shape &s, bool split, const Args &a, const void *fwd_ws, void *ws,
                       const FusedOptions &opt, cudaStream_t st, Trace &tr) {
  const Shape p = padded_shape(s);
  Carver fc(const_cast<void *>(fwd_ws));
  const PadFwdWs f = carve_pad_fwd(fc, s, split);
  Carver cv(ws);
  const PadBwdWs w = carve_pad_bwd(cv, s, split, opt.ring_depth);
  const PadTables t = tables_of(f);
  RowSets in{};
  in.set[0] = row_set(a.dout, w.dout, s.H * s.P * 2);
  in.count = 1;
  tr.mark(st);
  cudaError_t err = launch_rows<true>(in, t, p.nc, nullptr, st);
  tr.mark(st);
  if (err != cudaSuccess) return err;
  Args ai{};
  ai.x = f.x; ai.B = f.B; ai.C = f.C; ai.dout = w.dout; ai.dt = f.dt; ai.A = a.A; ai.D = a.D; ai.init = a.init;
  ai.states_in = split ? fused_split_aux(p, f.inner) : f.packed;
  ai.seq_idx = f.seq;
  ai.dx = w.dx; ai.ddt = w.ddt; ai.dB = w.dB; ai.dC = w.dC;
  ai.dA = a.dA; ai.dD = a.dD; ai.dinit = a.dinit;   // not per token: written in place
  if ((err = split ? fused_bwd_split(p, ai, w.inner, opt, st, tr) : fused_bwd(p, ai, w.inner, opt, st, tr)) !=
      cudaSuccess)
    return err;
  RowSets out{};
  out.set[0] = row_set(w.dx, a.dx, s.H * s.P * 4);
  out.set[1] = row_set(w.ddt, a.ddt, s.H * 4);
  out.set[2] = row_set(w.dB, a.dB, s.G * s.N * 4);
  out.set[3] = row_set(w.dC, a.dC, s.G * s.N * 4);
  out.count = 4;
  tr.mark(st);
  err = launch_rows<false>(out, t, p.nc, nullptr, st);
  tr.mark(st);
  return err;
}

}  // namespace ssd
