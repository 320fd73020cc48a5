// ssd_common.cuh -- shapes, workspace carving and small device helpers
// shared by the kernels of the Mamba2 SSD library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

// Problem shape as the kernels see it (all int64 to keep index math safe).
struct Shape {
  int64_t b, T, H, P, G, N, Q, nc, hpg, nseq;
};

// Raw pointers of one forward or backward call.
struct Args {
  const void *x, *B, *C, *dout;
  const float *dt, *A, *D, *init, *states_in;
  const int32_t *seq_idx;
  void *y;
  float *states_out;
  float *dx, *ddt, *dA, *dB, *dC, *dD, *dinit;
};

// Optional per-launch event trace: when `events` is set, marks 2k and 2k+1
// are recorded on the stream right before and after launch k.
struct Trace {
  cudaEvent_t *events = nullptr;
  int count = 0;
  int next = 0;
  void mark(cudaStream_t st) {
    if (events && next < count) cudaEventRecord(events[next], st);
    ++next;
  }
};

// Bump allocator over the caller's workspace; every piece 256-byte aligned.
struct Carver {
  char *base;
  size_t off = 0;
  explicit Carver(void *p) : base(static_cast<char *>(p)) {}
  template <class T>
  T *take(int64_t count) {
    off = (off + 255) & ~size_t(255);
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off += size_t(count) * sizeof(T);
    return p;
  }
  size_t bytes() const { return (off + 255) & ~size_t(255); }
};

__device__ __forceinline__ float ld(const float *p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float *p, float v) { *p = v; }
__device__ __forceinline__ void st(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// In-chunk cumulative decay is carried as an unevaluated sum hi + lo (a
// compensated prefix sum).  The decay between two tokens of a chunk is then
// exp(diff) with diff accurate to a few ulp of the difference itself rather
// than of the (possibly large) cumulative values.
__device__ __forceinline__ float acs_diff(float hi_t, float lo_t, float hi_s, float lo_s) {
  return __fadd_rn(__fsub_rn(hi_t, hi_s), __fsub_rn(lo_t, lo_s));
}

__device__ __forceinline__ bool is_seq_start(const int32_t *seq_idx, int64_t bi, int64_t T, int64_t t) {
  if (t == 0) return true;
  if (seq_idx == nullptr) return false;
  return seq_idx[bi * T + t] != seq_idx[bi * T + t - 1];
}

__device__ __forceinline__ int64_t seq_of(const int32_t *seq_idx, int64_t bi, int64_t T, int64_t t) {
  return seq_idx ? int64_t(seq_idx[bi * T + t]) : bi;
}

// p[0] + p[stride] + ... + p[(n-1) stride], added one term at a time in
// ascending order onto acc.  The loads of each batch of 32 terms are issued
// before any of their adds, so the sum waits on one memory latency per batch
// rather than one per term; the order of the adds, and so the bits, are those
// of the plain loop.
__device__ __forceinline__ float column_sum(const float *__restrict__ p, int64_t n, int64_t stride, float acc) {
  constexpr int kBatch = 32;
  int64_t k = 0;
  for (; k + kBatch <= n; k += kBatch) {
    float v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) v[j] = __ldcg(p + (k + j) * stride);
#pragma unroll
    for (int j = 0; j < kBatch; ++j) acc += v[j];
  }
  for (; k < n; ++k) acc += __ldcg(p + k * stride);
  return acc;
}

}  // namespace ssd
