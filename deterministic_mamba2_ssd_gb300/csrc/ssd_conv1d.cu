// ssd_conv1d.cu -- causal depthwise conv1d before the scan, forward and a
// deterministic backward.
//
// "Deterministic bwd kernel for mamba2" (Mamba PR #827), section "Atomic add
// non-determinism", names causal-conv1d's atomics, next to the SSD
// backward's, as a source of run-to-run differences.  Per batch row b,
// token t and channel c (x laid out (batch, seqlen, channels)):
//
//     pre[t,c] = bias[c] + sum_{k<K} w[c,k] x[t-K+1+k, c],   y = act(pre)
//
// with taps before the row start, or (packed batch) in another sequence than
// t, reading zero; act is the identity or silu.  Its backward:
//
//     dpre = dy act'(pre),  dx[s] = sum_k w[k] dpre[s+K-1-k],
//     dw[c,k] = sum_t dpre[t,c] x[t-K+1+k, c],  dbias[c] = sum_t dpre[t,c].
//
// dw and dbias sum over every token of every batch row: this is where the
// atomics were.  Here each thread owns a fixed tile of kTile consecutive
// tokens of one batch row and 4 consecutive channels, sums its tile's terms in
// token order and parks the partial sums in the tile's slot; a second kernel
// folds the slots in ascending tile order.  The tiles are fixed by the shape
// alone, so the bits are the same for every launch configuration (block
// size).  Everything else has one writer per element.
#include <cuda_bf16.h>

#include "mamba2_ssd.h"
#include "ssd_common.cuh"

namespace ssd {

namespace {

constexpr int kTile = 128;   // tokens per thread (and per dw/dbias slot)
constexpr int kVec = 4;      // channels per thread

__device__ __forceinline__ void load4(const float *p, float (&v)[4]) {
  const float4 u = __ldg(reinterpret_cast<const float4 *>(p));
  v[0] = u.x, v[1] = u.y, v[2] = u.z, v[3] = u.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&v)[4]) {
  const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
  v[0] = a.x, v[1] = a.y, v[2] = b.x, v[3] = b.y;
}
__device__ __forceinline__ void store4(float *p, const float (&v)[4]) {
  *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16 *p, const float (&v)[4]) {
  uint2 u;
  *reinterpret_cast<__nv_bfloat162 *>(&u.x) = __floats2bfloat162_rn(v[0], v[1]);
  *reinterpret_cast<__nv_bfloat162 *>(&u.y) = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2 *>(p) = u;
}

// Each thread streams the rows it will read next into its own slots of a
// shared-memory ring with asynchronous copies, kDepth tokens ahead: the loads
// are in flight without holding registers.  Slot (d, a) of thread i is the
// 16-byte word at ((d * 2 + a) * blockDim.x + i) * 16 (a = 0: x, 1: dy).
constexpr int kDepth = 8;
static_assert((kDepth & (kDepth - 1)) == 0, "ring depth: a power of two");

__device__ __forceinline__ uint32_t ring_slot(uint32_t base, int d, int a) {
  return base + uint32_t(((d * 2 + a) * int(blockDim.x) + int(threadIdx.x)) * 16);
}
// Copy the 4 channels of one token (8 bytes of bf16 or 16 of fp32) into a ring
// slot, or zeros when `valid` is false (nothing is read then).
template <class TIn>
__device__ __forceinline__ void stream_row(uint32_t dst, const TIn *src, bool valid) {
  if (sizeof(TIn) == 2)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(valid ? 8 : 0) : "memory");
  else
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void stream_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// the oldest of the kDepth groups in flight has landed
__device__ __forceinline__ void stream_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(kDepth - 1) : "memory"); }

__device__ __forceinline__ void read_slot(uint32_t a, const float *, float (&v)[4]) {
  float4 u;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(u.x), "=f"(u.y), "=f"(u.z), "=f"(u.w) : "r"(a));
  v[0] = u.x, v[1] = u.y, v[2] = u.z, v[3] = u.w;
}
__device__ __forceinline__ void read_slot(uint32_t a, const __nv_bfloat16 *, float (&v)[4]) {
  uint32_t lo, hi;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(lo), "=r"(hi) : "r"(a));
  const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&lo));
  const float2 q = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi));
  v[0] = p.x, v[1] = p.y, v[2] = q.x, v[3] = q.y;
}

// logistic function, no overflow for either sign of v (the fast exponential
// and the fast division, whose argument 1 + e lies in [1, 2]; relative error
// a few 1e-7)
__device__ __forceinline__ float sigmoid(float v) {
  const float e = __expf(-fabsf(v));
  const float r = __fdividef(1.f, 1.f + e);
  return v >= 0.f ? r : e * r;
}

struct ConvShape {
  int64_t b, T, C;
  int tiles_per_row;
  int silu;
};

// Token t of batch row bi starts a sequence (row start, or a new id).
__device__ __forceinline__ bool starts_seq(const int32_t *seq_idx, int64_t bi, int64_t T, int64_t t) {
  return t == 0 || (seq_idx != nullptr && __ldg(seq_idx + bi * T + t) != __ldg(seq_idx + bi * T + t - 1));
}

template <class TIn, int K>
__global__ void conv_fwd_kernel(ConvShape s, const TIn *__restrict__ x, const float *__restrict__ w,
                                const float *__restrict__ bias, const int32_t *__restrict__ seq_idx,
                                TIn *__restrict__ y) {
  const int64_t cv = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (cv * kVec >= s.C) return;
  const int64_t c0 = cv * kVec;
  const int64_t bi = blockIdx.y / s.tiles_per_row;
  const int64_t t0 = int64_t(blockIdx.y % s.tiles_per_row) * kTile, t1 = min(s.T, t0 + kTile);
  float wv[K][kVec], bv[kVec];
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    bv[i] = bias ? __ldg(bias + c0 + i) : 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) wv[k][i] = __ldg(w + (c0 + i) * K + k);
  }
  float win[K][kVec];   // x of tokens t-K+1 .. t (win[K-1] = token t)
#pragma unroll
  for (int k = 0; k < K; ++k)
#pragma unroll
    for (int i = 0; i < kVec; ++i) win[k][i] = 0.f;
  extern __shared__ __align__(16) uint8_t ring_raw[];
  const uint32_t ring = uint32_t(__cvta_generic_to_shared(ring_raw));
  const int64_t u0 = t0 - (K - 1);
  const TIn *row = x + (bi * s.T + u0) * s.C + c0;   // token u0 (read only where it exists)
  auto issue = [&](int64_t u, int d, const TIn *p) {
    const bool ok = u >= 0 && u < t1;
    stream_row(ring_slot(ring, d, 0), ok ? p : x, ok);
    stream_commit();
  };
  for (int j = 0; j < kDepth; ++j) issue(u0 + j, j, row + j * s.C);
  int d = 0;   // ring slot of token t
  for (int64_t t = u0; t < t1; ++t, d = (d + 1) & (kDepth - 1), row += s.C) {
#pragma unroll
    for (int k = 0; k + 1 < K; ++k)
#pragma unroll
      for (int i = 0; i < kVec; ++i) win[k][i] = win[k + 1][i];
    stream_wait();
    read_slot(ring_slot(ring, d, 0), x, win[K - 1]);   // zeros before the row start
    issue(t + kDepth, d, row + kDepth * s.C);          // the slot just read takes the token kDepth ahead
    if (t < 0) continue;
    if (starts_seq(seq_idx, bi, s.T, t)) {   // earlier taps belong to another sequence
#pragma unroll
      for (int k = 0; k + 1 < K; ++k)
#pragma unroll
        for (int i = 0; i < kVec; ++i) win[k][i] = 0.f;
    }
    if (t < t0) continue;
    float out[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      float acc = bv[i];
#pragma unroll
      for (int k = 0; k < K; ++k) acc = fmaf(wv[k][i], win[k][i], acc);
      out[i] = s.silu ? acc * sigmoid(acc) : acc;
    }
    store4(y + (row - x) , out);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Backward of one (tile, 4 channels): dpre of the tile's tokens and of the
// K-1 tokens after it (for dx at the tile's end), dx of the tile's tokens,
// and the tile's partial sums of dw and dbias in token order -- into slot
// `tile` (part[(tile * (K + 1) + k) * C + c], k = K for dbias) or, in the
// atomic variant, added straight into dw and dbias.  The token loop is
// unrolled by four: token u lives in window slot u % 4 of xw (x) and dz
// (dpre), so the windows need no shifting and every slot index is a
// compile-time constant (the walk starts at a multiple of 4, four tokens
// before the tile).  Tokens past the row end take part as zeros, so dx of the
// tile's last tokens comes out of the same loop.  kSeq: seq_idx is given (a
// sequence may start at any token); without it the only start is the row's
// first token, whose earlier taps read zeros anyway.
template <class TIn, int K, bool kAtomic, bool kSeq>
__global__ void conv_bwd_kernel(ConvShape s, const TIn *__restrict__ x, const float *__restrict__ w,
                                 const float *__restrict__ bias, const int32_t *__restrict__ seq_idx,
                                 const TIn *__restrict__ dy, float *__restrict__ dx, float *__restrict__ part,
                                 float *__restrict__ dw, float *__restrict__ dbias) {
  const int64_t cv = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (cv * kVec >= s.C) return;
  const int64_t c0 = cv * kVec;
  const int64_t tile = blockIdx.y;
  const int64_t bi = tile / s.tiles_per_row;
  const int64_t t0 = int64_t(tile % s.tiles_per_row) * kTile, t1 = min(s.T, t0 + kTile);
  float wv[K][kVec], bv[kVec];
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    bv[i] = bias ? __ldg(bias + c0 + i) : 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) wv[k][i] = __ldg(w + (c0 + i) * K + k);
  }
  float xw[4][kVec], dz[4][kVec];   // slot u % 4: x and dpre of token u
  bool sst[4] = {false, false, false, false};   // slot u % 4: token u starts a sequence (kSeq)
  float dwp[K][kVec], dbp[kVec];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < kVec; ++i) xw[j][i] = dz[j][i] = 0.f;
#pragma unroll
  for (int k = 0; k < K; ++k)
#pragma unroll
    for (int i = 0; i < kVec; ++i) dwp[k][i] = 0.f;
#pragma unroll
  for (int i = 0; i < kVec; ++i) dbp[i] = 0.f;
  extern __shared__ __align__(16) uint8_t ring_raw[];
  const uint32_t ring = uint32_t(__cvta_generic_to_shared(ring_raw));
  const int64_t ub = t0 - 4, u1 = t1 + (K - 1), ue = ub + ((u1 - ub + 3) / 4) * 4;
  const int64_t off0 = (bi * s.T + ub) * s.C + c0;   // element offset of token ub (read only where it exists)
  auto issue = [&](int64_t u, int d, int64_t off) {
    const bool okx = u >= 0 && u < s.T && u < u1, okg = okx && u >= t0;
    stream_row(ring_slot(ring, d, 0), okx ? x + off : x, okx);
    stream_row(ring_slot(ring, d, 1), okg ? dy + off : dy, okg);
    stream_commit();
  };
  for (int j = 0; j < kDepth; ++j) issue(ub + j, j, off0 + j * s.C);
  int dslot = 0;   // ring slot of token u
  int64_t off = off0;
  for (int64_t ug = ub; ug < ue; ug += 4) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // token u = ug + j, window slot j
      const int64_t u = ug + j;
      float g[kVec];
      stream_wait();
      read_slot(ring_slot(ring, dslot, 0), x, xw[j]);   // zeros outside the row
      read_slot(ring_slot(ring, dslot, 1), dy, g);      // zeros before the tile and outside the row
      issue(u + kDepth, dslot, off + kDepth * s.C);
      dslot = (dslot + 1) & (kDepth - 1);
      off += s.C;
      if (kSeq) {
        sst[j] = u >= 0 && u < s.T && starts_seq(seq_idx, bi, s.T, u);
        if (sst[j]) {   // earlier taps belong to another sequence
#pragma unroll
          for (int k = 1; k < 4; ++k)
#pragma unroll
            for (int i = 0; i < kVec; ++i) xw[(j - k) & 3][i] = 0.f;
        }
      }
      // dpre of token u (zero before the tile and outside the row: dy is zero there)
#pragma unroll
      for (int i = 0; i < kVec; ++i) {
        float acc = bv[i];
#pragma unroll
        for (int k = 0; k < K; ++k) acc = fmaf(wv[k][i], xw[(j - (K - 1) + k) & 3][i], acc);
        if (s.silu) {
          const float sg = sigmoid(acc);
          dz[j][i] = g[i] * (sg * fmaf(acc, 1.f - sg, 1.f));
        } else {
          dz[j][i] = g[i];
        }
      }
      if (u >= t0 && u < t1) {   // the tile's own tokens: partial sums of dw and dbias, in token order
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
#pragma unroll
          for (int k = 0; k < K; ++k) dwp[k][i] = fmaf(dz[j][i], xw[(j - (K - 1) + k) & 3][i], dwp[k][i]);
          dbp[i] += dz[j][i];
        }
      }
      // dx of token sx = u-K+1 (complete now): sum_m w[K-1-m] dz[sx+m] over taps that stay in sx's sequence
      const int64_t sx = u - (K - 1);
      if (sx >= t0 && sx < t1) {
        float o[kVec];
#pragma unroll
        for (int i = 0; i < kVec; ++i) o[i] = 0.f;
        bool live = true;
#pragma unroll
        for (int m = 0; m < K; ++m) {   // token sx + m sits in slot (j - (K-1) + m) % 4
          const int sl = (j - (K - 1) + m) & 3;
          if (kSeq && m > 0 && sst[sl]) live = false;
          if (live) {
#pragma unroll
            for (int i = 0; i < kVec; ++i) o[i] = fmaf(wv[K - 1 - m][i], dz[sl][i], o[i]);
          }
        }
        store4(dx + off - K * s.C, o);   // token sx (off has moved on to token u + 1)
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (kAtomic) {
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
#pragma unroll
      for (int k = 0; k < K; ++k) atomicAdd(dw + (c0 + i) * K + k, dwp[k][i]);
      if (dbias) atomicAdd(dbias + c0 + i, dbp[i]);
    }
  } else {
    float *p = part + tile * (K + 1) * s.C + c0;
#pragma unroll
    for (int k = 0; k < K; ++k) store4(p + k * s.C, dwp[k]);
    store4(p + K * s.C, dbp);
  }
}

// dw[c,k] (k < K) and dbias[c] (k = K): the tiles' partial sums in ascending
// tile order; one thread per (k, c).
__global__ void conv_fold_kernel(int64_t C, int K, int64_t tiles, const float *__restrict__ part,
                                 float *__restrict__ dw, float *__restrict__ dbias) {
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= (K + 1) * C) return;
  const int64_t k = idx / C, c = idx % C;
  float acc = 0.f;
  for (int64_t t = 0; t < tiles; ++t) acc += __ldcs(part + (t * (K + 1) + k) * C + c);
  if (k < K)
    dw[c * K + k] = acc;
  else if (dbias)
    dbias[c] = acc;
}

constexpr int kConvBlocks[] = {128, 256};
// dynamic shared memory of a block: each thread's kDepth x {x, dy} 16-byte slots
size_t ring_bytes(int block) { return size_t(kDepth) * 2 * 16 * size_t(block); }
constexpr int kNumConvConfigs = 2;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validity of the sizes; fills the kernel shape.
bool conv_shape(int64_t batch, int64_t seqlen, int64_t channels, int32_t width, int32_t dtype, int32_t activation,
                const int32_t *seq_idx, ConvShape *s) {
  if (batch <= 0 || seqlen <= 0 || channels <= 0 || channels % kVec != 0) return false;
  if (width < 1 || width > 4) return false;
  if (dtype != SSD_F32 && dtype != SSD_BF16) return false;
  if (activation != 0 && activation != 1) return false;
  if (seq_idx && batch != 1) return false;
  const int64_t tpr = (seqlen + kTile - 1) / kTile;
  if (batch * tpr > 65535 || (channels / kVec + 127) / 128 > (int64_t(1) << 31) - 1) return false;
  s->b = batch;
  s->T = seqlen;
  s->C = channels;
  s->tiles_per_row = int(tpr);
  s->silu = activation;
  return true;
}

// Launch with the block's ring of shared memory (above the 48 KB default for 256 threads).
template <class Kern, class... Args>
cudaError_t launch_ring(Kern kernel, dim3 grid, int block, cudaStream_t st, Args... args) {
  const size_t smem = ring_bytes(block);
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (err != cudaSuccess) return err;
  kernel<<<grid, block, smem, st>>>(args...);
  return cudaGetLastError();
}

template <class TIn>
cudaError_t launch_fwd(const ConvShape &s, int K, dim3 grid, int block, const void *x, const float *w,
                       const float *bias, const int32_t *seq_idx, void *y, cudaStream_t st) {
  const TIn *xx = static_cast<const TIn *>(x);
  TIn *yy = static_cast<TIn *>(y);
  switch (K) {
    case 1: return launch_ring(conv_fwd_kernel<TIn, 1>, grid, block, st, s, xx, w, bias, seq_idx, yy);
    case 2: return launch_ring(conv_fwd_kernel<TIn, 2>, grid, block, st, s, xx, w, bias, seq_idx, yy);
    case 3: return launch_ring(conv_fwd_kernel<TIn, 3>, grid, block, st, s, xx, w, bias, seq_idx, yy);
    default: return launch_ring(conv_fwd_kernel<TIn, 4>, grid, block, st, s, xx, w, bias, seq_idx, yy);
  }
}

template <class TIn, bool kAtomic>
cudaError_t launch_bwd(const ConvShape &s, int K, dim3 grid, int block, const void *x, const float *w,
                       const float *bias, const int32_t *seq_idx, const void *dy, float *dx, float *part, float *dw,
                       float *dbias, cudaStream_t st) {
  const TIn *xx = static_cast<const TIn *>(x), *gg = static_cast<const TIn *>(dy);
#define SSD_CONV_BWD(KK, SEQ) \
  launch_ring(conv_bwd_kernel<TIn, KK, kAtomic, SEQ>, grid, block, st, s, xx, w, bias, seq_idx, gg, dx, part, dw, dbias)
  if (seq_idx) {
    switch (K) {
      case 1: return SSD_CONV_BWD(1, true);
      case 2: return SSD_CONV_BWD(2, true);
      case 3: return SSD_CONV_BWD(3, true);
      default: return SSD_CONV_BWD(4, true);
    }
  }
  switch (K) {
    case 1: return SSD_CONV_BWD(1, false);
    case 2: return SSD_CONV_BWD(2, false);
    case 3: return SSD_CONV_BWD(3, false);
    default: return SSD_CONV_BWD(4, false);
  }
#undef SSD_CONV_BWD
}

}  // namespace

}  // namespace ssd

extern "C" {

int mamba2_ssd_conv1d_num_configs(void) { return ssd::kNumConvConfigs; }

size_t mamba2_ssd_conv1d_bwd_workspace_size(int64_t batch, int64_t seqlen, int64_t channels, int32_t width) {
  ssd::ConvShape s;
  if (!ssd::conv_shape(batch, seqlen, channels, width, SSD_F32, 0, nullptr, &s)) return 0;
  return size_t(batch * s.tiles_per_row) * size_t(width + 1) * size_t(channels) * sizeof(float);
}

ssd_status mamba2_ssd_conv1d_fwd(int64_t batch, int64_t seqlen, int64_t channels, int32_t width, int32_t dtype,
                                 int32_t activation, const void *x, const float *weight, const float *bias,
                                 const int32_t *seq_idx, void *y, int config, void *stream) {
  ssd::ConvShape s;
  if (!ssd::conv_shape(batch, seqlen, channels, width, dtype, activation, seq_idx, &s)) return SSD_ERR_INVALID_ARG;
  if (config < 0 || config >= ssd::kNumConvConfigs) return SSD_ERR_INVALID_ARG;
  const void *req[] = {x, weight, y};
  for (const void *p : req)
    if (!p || !ssd::aligned16(p)) return SSD_ERR_INVALID_ARG;
  if ((bias && !ssd::aligned16(bias)) || (seq_idx && !ssd::aligned16(seq_idx))) return SSD_ERR_INVALID_ARG;
  const int block = ssd::kConvBlocks[config];
  const dim3 grid(unsigned((channels / ssd::kVec + block - 1) / block), unsigned(batch * s.tiles_per_row));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t err = dtype == SSD_BF16
                              ? ssd::launch_fwd<__nv_bfloat16>(s, width, grid, block, x, weight, bias, seq_idx, y, st)
                              : ssd::launch_fwd<float>(s, width, grid, block, x, weight, bias, seq_idx, y, st);
  return err == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status mamba2_ssd_conv1d_bwd(int64_t batch, int64_t seqlen, int64_t channels, int32_t width, int32_t dtype,
                                 int32_t activation, const void *x, const float *weight, const float *bias,
                                 const int32_t *seq_idx, const void *dy, float *dx, float *dweight, float *dbias,
                                 void *workspace, size_t workspace_bytes, int config, int variant, void *stream) {
  ssd::ConvShape s;
  if (!ssd::conv_shape(batch, seqlen, channels, width, dtype, activation, seq_idx, &s)) return SSD_ERR_INVALID_ARG;
  if (config < 0 || config >= ssd::kNumConvConfigs) return SSD_ERR_INVALID_ARG;
  if (variant != SSD_VARIANT_DETERMINISTIC && variant != SSD_VARIANT_ATOMIC) return SSD_ERR_INVALID_ARG;
  const void *req[] = {x, weight, dy, dx, dweight};
  for (const void *p : req)
    if (!p || !ssd::aligned16(p)) return SSD_ERR_INVALID_ARG;
  if ((bias && !ssd::aligned16(bias)) || (seq_idx && !ssd::aligned16(seq_idx)) || (dbias && !ssd::aligned16(dbias)))
    return SSD_ERR_INVALID_ARG;
  const bool atomic = variant == SSD_VARIANT_ATOMIC;
  if (!atomic) {
    if (workspace_bytes < mamba2_ssd_conv1d_bwd_workspace_size(batch, seqlen, channels, width))
      return SSD_ERR_WORKSPACE;
    if (!workspace || !ssd::aligned16(workspace)) return SSD_ERR_INVALID_ARG;
  }
  const int block = ssd::kConvBlocks[config];
  const dim3 grid(unsigned((channels / ssd::kVec + block - 1) / block), unsigned(batch * s.tiles_per_row));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float *part = static_cast<float *>(workspace);
  cudaError_t err;
  if (atomic) {
    if ((err = cudaMemsetAsync(dweight, 0, size_t(channels * width) * sizeof(float), st)) != cudaSuccess)
      return SSD_ERR_CUDA;
    if (dbias && (err = cudaMemsetAsync(dbias, 0, size_t(channels) * sizeof(float), st)) != cudaSuccess)
      return SSD_ERR_CUDA;
    err = dtype == SSD_BF16 ? ssd::launch_bwd<__nv_bfloat16, true>(s, width, grid, block, x, weight, bias, seq_idx, dy,
                                                                    dx, part, dweight, dbias, st)
                            : ssd::launch_bwd<float, true>(s, width, grid, block, x, weight, bias, seq_idx, dy, dx,
                                                           part, dweight, dbias, st);
    return err == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
  }
  err = dtype == SSD_BF16 ? ssd::launch_bwd<__nv_bfloat16, false>(s, width, grid, block, x, weight, bias, seq_idx, dy,
                                                                   dx, part, dweight, dbias, st)
                          : ssd::launch_bwd<float, false>(s, width, grid, block, x, weight, bias, seq_idx, dy, dx, part,
                                                          dweight, dbias, st);
  if (err != cudaSuccess) return SSD_ERR_CUDA;
  const int64_t outs = int64_t(width + 1) * channels;
  ssd::conv_fold_kernel<<<unsigned((outs + 255) / 256), 256, 0, st>>>(channels, width, batch * s.tiles_per_row, part,
                                                                     dweight, dbias);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
