// ssd_adjacent.cu -- the two steps either side of the SSD scan, with their
// backward passes: the step-size preprocessing that Mamba2 folds into its
// chunk_cumsum (the step "Deterministic bwd kernel for mamba2", Mamba PR #827,
// lists as chunk_cumsum_bwd in its per-kernel breakdown) and the z-gate on the
// scan's output.
//
//   dt  = clamp(sp(dt_raw + dt_bias), dt_min, dt_max),  sp = softplus or identity
//   out = y * silu(z),  silu(z) = z * sigmoid(z)
//
// Both are elementwise and bandwidth-bound: grid-stride loops over 16-byte
// vectors, one CTA wave sized from the SM count.  The one reduction (the
// gradient of dt_bias, a sum over all rows per head) is deterministic: the
// rows are cut into a fixed number of slabs, each summed in a fixed order,
// and a second kernel folds the slabs in ascending order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mamba2_ssd.h"

namespace {

constexpr int kThreads = 256;
constexpr int kSlabs = 32;       // fixed row slabs of the dt_bias reduction
constexpr int kSlabWarps = 32;   // warps per CTA of the dt backward
constexpr int kRowBatch = 4;     // rows whose loads a thread issues together

inline int num_sms() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0)
      sms = 152;
  }
  return sms;
}

inline unsigned grid_for(int64_t work_items) {
  const int64_t want = (work_items + kThreads - 1) / kThreads;
  const int64_t cap = int64_t(num_sms()) * 8;
  return unsigned(want < 1 ? 1 : (want < cap ? want : cap));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// log(1 + e^v) in fp32: beyond 20 the correction e^-v is below half an ulp of v.
__device__ __forceinline__ float softplus_f(float v) { return v > 20.f ? v : log1pf(expf(v)); }

// 1 / (1 + e^-v) without overflow of the exponential on either side:
// e = e^-|v| <= 1, r = 1 / (1 + e) (correctly rounded reciprocal); the value
// is r for v >= 0 and e r for v < 0.
__device__ __forceinline__ float sigmoid_f(float v) {
  const float e = expf(-fabsf(v));
  const float r = __frcp_rn(1.f + e);
  return v >= 0.f ? r : e * r;
}

struct DtParams {
  int softplus;
  int clamps;   // 0 when no value can leave [lo, hi] (e.g. softplus with lo <= 0, hi = inf)
  float lo, hi;
};

__device__ __forceinline__ float dt_value(float v, const DtParams &q) {
  const float s = q.softplus ? softplus_f(v) : v;
  return fminf(fmaxf(s, q.lo), q.hi);
}

// d dt / d v: the softplus slope where the clamp passes (lo <= s <= hi), else 0.
template <bool kClamp>
__device__ __forceinline__ float dt_slope(float v, const DtParams &q) {
  if (kClamp) {
    const float s = q.softplus ? softplus_f(v) : v;
    if (!(s >= q.lo && s <= q.hi)) return 0.f;
  }
  return q.softplus ? sigmoid_f(v) : 1.f;
}

DtParams dt_params(int use_softplus, float lo, float hi) {
  DtParams q;
  q.softplus = use_softplus != 0;
  q.lo = lo;
  q.hi = hi;
  // softplus is positive (or an underflowed +0), so a lower bound <= 0 never binds
  const bool lo_binds = q.softplus ? lo > 0.f : lo > -INFINITY;
  q.clamps = lo_binds || hi < INFINITY;
  return q;
}

__global__ void dt_fwd_kernel(int64_t total, int64_t H, const float *__restrict__ raw,
                              const float *__restrict__ bias, DtParams q, float *__restrict__ dt) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  if ((H & 3) == 0) {  // four consecutive heads of one row per vector
    const int64_t nv = total >> 2;
    for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < nv; v += stride) {
      float4 r = reinterpret_cast<const float4 *>(raw)[v];
      const int64_t h = (v << 2) % H;
      if (bias) {
        r.x += bias[h];
        r.y += bias[h + 1];
        r.z += bias[h + 2];
        r.w += bias[h + 3];
      }
      reinterpret_cast<float4 *>(dt)[v] = make_float4(dt_value(r.x, q), dt_value(r.y, q), dt_value(r.z, q),
                                                      dt_value(r.w, q));
    }
  } else {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride)
      dt[i] = dt_value(raw[i] + (bias ? bias[i % H] : 0.f), q);
  }
}

// Rows are cut into kSlabs fixed slabs; CTA (head block of 32, slab), lane =
// head, warp w takes the slab's rows w, w + 32, ... in ascending order and
// writes ddt_raw; the CTA then adds its 32 warp sums in warp order into the
// slab's partial.  The cut depends on rows only, so the sum is reproducible.
template <bool kClamp>
__global__ void __launch_bounds__(32 * kSlabWarps) dt_bwd_kernel(int64_t rows, int64_t H, const float *__restrict__ raw,
                              const float *__restrict__ bias, DtParams q, const float *__restrict__ ddt,
                              float *__restrict__ ddt_raw, float *__restrict__ partial) {
  __shared__ float red[kSlabWarps][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t hblocks = (H + 31) / 32;
  const int64_t hb = blockIdx.x % hblocks, slab = blockIdx.x / hblocks;
  const int64_t h = hb * 32 + lane;
  const int64_t per = (rows + kSlabs - 1) / kSlabs;
  const int64_t r0 = slab * per, r1 = min(rows, r0 + per);
  float acc = 0.f;
  if (h < H) {
    const float b = bias ? bias[h] : 0.f;
    for (int64_t rb = r0 + warp; rb < r1; rb += int64_t(kSlabWarps) * kRowBatch) {
      float v[kRowBatch], g[kRowBatch];
#pragma unroll
      for (int k = 0; k < kRowBatch; ++k) {   // all loads of the batch first
        const int64_t r = rb + int64_t(k) * kSlabWarps;
        v[k] = r < r1 ? raw[r * H + h] : 0.f;
        g[k] = r < r1 ? ddt[r * H + h] : 0.f;
      }
#pragma unroll
      for (int k = 0; k < kRowBatch; ++k) {   // then rows in ascending order
        const int64_t r = rb + int64_t(k) * kSlabWarps;
        if (r < r1) {
          const float d = g[k] * dt_slope<kClamp>(v[k] + b, q);
          ddt_raw[r * H + h] = d;
          acc += d;
        }
      }
    }
  }
  if (partial == nullptr) return;
  red[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && h < H) {
    float tot = 0.f;
    for (int k = 0; k < kSlabWarps; ++k) tot += red[k][lane];
    partial[slab * H + h] = tot;
  }
}

// ddt_bias[h] = sum of the kSlabs slab partials in ascending order.
__global__ void dt_bias_fold_kernel(int64_t H, const float *__restrict__ partial, float *__restrict__ ddt_bias) {
  const int64_t h = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (h >= H) return;
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < kSlabs; ++k) acc += partial[k * H + h];
  ddt_bias[h] = acc;
}

__device__ __forceinline__ float silu_f(float z) { return z * sigmoid_f(z); }

// silu(z) = z s and its slope s (1 + z (1 - s)), s = sigmoid(z), from one s.
__device__ __forceinline__ void silu_and_slope(float z, float &silu, float &slope) {
  const float s = sigmoid_f(z);
  silu = z * s;
  slope = s * fmaf(z, 1.f - s, 1.f);
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, int64_t v, float (&o)[8]) {
  const uint4 u = reinterpret_cast<const uint4 *>(p)[v];
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    o[2 * k] = __uint_as_float(w[k] << 16);
    o[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}

__device__ __forceinline__ void store8(__nv_bfloat16 *p, int64_t v, const float (&o)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(o[2 * k], o[2 * k + 1]);
    w[k] = *reinterpret_cast<const uint32_t *>(&b);
  }
  reinterpret_cast<uint4 *>(p)[v] = make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float ld1(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float ld1(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ void st1(__nv_bfloat16 *p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }
__device__ __forceinline__ void st1(float *p, int64_t i, float v) { p[i] = v; }

template <class T>
__global__ void gate_fwd_kernel(int64_t n, const T *__restrict__ y, const T *__restrict__ z, T *__restrict__ out) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t t0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  int64_t done = 0;
  if constexpr (sizeof(T) == 2) {
    const int64_t nv = n >> 3;
    for (int64_t v = t0; v < nv; v += stride) {
      float a[8], b[8];
      load8(y, v, a);
      load8(z, v, b);
#pragma unroll
      for (int k = 0; k < 8; ++k) a[k] *= silu_f(b[k]);
      store8(out, v, a);
    }
    done = nv << 3;
  } else {
    const int64_t nv = n >> 2;
    for (int64_t v = t0; v < nv; v += stride) {
      const float4 a = reinterpret_cast<const float4 *>(y)[v];
      const float4 b = reinterpret_cast<const float4 *>(z)[v];
      reinterpret_cast<float4 *>(out)[v] =
          make_float4(a.x * silu_f(b.x), a.y * silu_f(b.y), a.z * silu_f(b.z), a.w * silu_f(b.w));
    }
    done = nv << 2;
  }
  for (int64_t i = done + t0; i < n; i += stride) st1(out, i, ld1(y, i) * silu_f(ld1(z, i)));
}

template <class T>
__global__ void gate_bwd_kernel(int64_t n, const T *__restrict__ y, const T *__restrict__ z,
                                const T *__restrict__ g, T *__restrict__ dy, float *__restrict__ dz) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t t0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  int64_t done = 0;
  if constexpr (sizeof(T) == 2) {
    const int64_t nv = n >> 3;
    for (int64_t v = t0; v < nv; v += stride) {
      float a[8], b[8], c[8], d[8];
      load8(y, v, a);
      load8(z, v, b);
      load8(g, v, c);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float si, sl;
        silu_and_slope(b[k], si, sl);
        d[k] = c[k] * a[k] * sl;
        c[k] *= si;
      }
      store8(dy, v, c);
      float4 *o = reinterpret_cast<float4 *>(dz) + 2 * v;
      o[0] = make_float4(d[0], d[1], d[2], d[3]);
      o[1] = make_float4(d[4], d[5], d[6], d[7]);
    }
    done = nv << 3;
  } else {
    const int64_t nv = n >> 2;
    for (int64_t v = t0; v < nv; v += stride) {
      const float4 a = reinterpret_cast<const float4 *>(y)[v];
      const float4 b = reinterpret_cast<const float4 *>(z)[v];
      const float4 c = reinterpret_cast<const float4 *>(g)[v];
      float si[4], sl[4];
      silu_and_slope(b.x, si[0], sl[0]);
      silu_and_slope(b.y, si[1], sl[1]);
      silu_and_slope(b.z, si[2], sl[2]);
      silu_and_slope(b.w, si[3], sl[3]);
      reinterpret_cast<float4 *>(dy)[v] = make_float4(c.x * si[0], c.y * si[1], c.z * si[2], c.w * si[3]);
      reinterpret_cast<float4 *>(dz)[v] =
          make_float4(c.x * a.x * sl[0], c.y * a.y * sl[1], c.z * a.z * sl[2], c.w * a.w * sl[3]);
    }
    done = nv << 2;
  }
  for (int64_t i = done + t0; i < n; i += stride) {
    const float a = ld1(y, i), b = ld1(z, i), c = ld1(g, i);
    float si, sl;
    silu_and_slope(b, si, sl);
    st1(dy, i, c * si);
    dz[i] = c * a * sl;
  }
}

bool dt_args_ok(int64_t rows, int64_t H, float lo, float hi) {
  // rows < 2^36 keeps the tile grid of the backward below 2^31 CTAs
  if (rows < 0 || H <= 0 || rows >= (int64_t(1) << 36) || rows > (int64_t(1) << 40) / H) return false;
  return !(isnan(lo) || isnan(hi) || lo > hi);
}


}  // namespace

extern "C" {

ssd_status mamba2_ssd_dt_fwd(int64_t rows, int64_t nheads, const float *dt_raw, const float *dt_bias,
                             int use_softplus, float dt_min, float dt_max, float *dt, void *stream) {
  if (!dt_args_ok(rows, nheads, dt_min, dt_max)) return SSD_ERR_INVALID_ARG;
  if (rows == 0) return SSD_OK;
  if (!dt_raw || !dt || !aligned16(dt_raw) || !aligned16(dt) || (dt_bias && !aligned16(dt_bias)))
    return SSD_ERR_INVALID_ARG;
  const int64_t total = rows * nheads;
  const DtParams q = dt_params(use_softplus, dt_min, dt_max);
  dt_fwd_kernel<<<grid_for((nheads & 3) == 0 ? total / 4 : total), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      total, nheads, dt_raw, dt_bias, q, dt);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

size_t mamba2_ssd_dt_bwd_workspace_size(int64_t rows, int64_t nheads) {
  if (!dt_args_ok(rows, nheads, 0.f, 0.f)) return 0;
  return size_t(kSlabs) * size_t(nheads) * sizeof(float);
}

ssd_status mamba2_ssd_dt_bwd(int64_t rows, int64_t nheads, const float *dt_raw, const float *dt_bias,
                             int use_softplus, float dt_min, float dt_max, const float *ddt, float *ddt_raw,
                             float *ddt_bias, void *workspace, size_t workspace_bytes, void *stream) {
  if (!dt_args_ok(rows, nheads, dt_min, dt_max)) return SSD_ERR_INVALID_ARG;
  if (ddt_bias && !aligned16(ddt_bias)) return SSD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows == 0) {
    if (ddt_bias && cudaMemsetAsync(ddt_bias, 0, size_t(nheads) * sizeof(float), st) != cudaSuccess)
      return SSD_ERR_CUDA;
    return SSD_OK;
  }
  const void *req[] = {dt_raw, ddt, ddt_raw};
  for (const void *p : req)
    if (!p || !aligned16(p)) return SSD_ERR_INVALID_ARG;
  if (dt_bias && !aligned16(dt_bias)) return SSD_ERR_INVALID_ARG;
  if (ddt_bias) {
    if (workspace_bytes < mamba2_ssd_dt_bwd_workspace_size(rows, nheads)) return SSD_ERR_WORKSPACE;
    if (!workspace || !aligned16(workspace)) return SSD_ERR_INVALID_ARG;
  }
  const DtParams q = dt_params(use_softplus, dt_min, dt_max);
  float *partial = ddt_bias ? static_cast<float *>(workspace) : nullptr;
  const int64_t hblocks = (nheads + 31) / 32;
  if (q.clamps)
    dt_bwd_kernel<true><<<unsigned(hblocks * kSlabs), 32 * kSlabWarps, 0, st>>>(rows, nheads, dt_raw, dt_bias, q, ddt,
                                                                             ddt_raw, partial);
  else
    dt_bwd_kernel<false><<<unsigned(hblocks * kSlabs), 32 * kSlabWarps, 0, st>>>(rows, nheads, dt_raw, dt_bias, q,
                                                                              ddt, ddt_raw, partial);
  if (ddt_bias)
    dt_bias_fold_kernel<<<unsigned((nheads + kThreads - 1) / kThreads), kThreads, 0, st>>>(nheads, partial, ddt_bias);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status mamba2_ssd_gate_fwd(int64_t n, int32_t dtype, const void *y, const void *z, void *out, void *stream) {
  if (n < 0 || (dtype != SSD_F32 && dtype != SSD_BF16)) return SSD_ERR_INVALID_ARG;
  if (n == 0) return SSD_OK;
  const void *req[] = {y, z, out};
  for (const void *p : req)
    if (!p || !aligned16(p)) return SSD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == SSD_BF16)
    gate_fwd_kernel<__nv_bfloat16><<<grid_for(n / 8 + 1), kThreads, 0, st>>>(
        n, static_cast<const __nv_bfloat16 *>(y), static_cast<const __nv_bfloat16 *>(z),
        static_cast<__nv_bfloat16 *>(out));
  else
    gate_fwd_kernel<float><<<grid_for(n / 4 + 1), kThreads, 0, st>>>(n, static_cast<const float *>(y),
                                                                    static_cast<const float *>(z),
                                                                    static_cast<float *>(out));
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status mamba2_ssd_gate_bwd(int64_t n, int32_t dtype, const void *y, const void *z, const void *dout, void *dy,
                               float *dz, void *stream) {
  if (n < 0 || (dtype != SSD_F32 && dtype != SSD_BF16)) return SSD_ERR_INVALID_ARG;
  if (n == 0) return SSD_OK;
  const void *req[] = {y, z, dout, dy, dz};
  for (const void *p : req)
    if (!p || !aligned16(p)) return SSD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == SSD_BF16)
    gate_bwd_kernel<__nv_bfloat16><<<grid_for(n / 8 + 1), kThreads, 0, st>>>(
        n, static_cast<const __nv_bfloat16 *>(y), static_cast<const __nv_bfloat16 *>(z),
        static_cast<const __nv_bfloat16 *>(dout), static_cast<__nv_bfloat16 *>(dy), dz);
  else
    gate_bwd_kernel<float><<<grid_for(n / 4 + 1), kThreads, 0, st>>>(
        n, static_cast<const float *>(y), static_cast<const float *>(z), static_cast<const float *>(dout),
        static_cast<float *>(dy), dz);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
