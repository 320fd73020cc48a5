// ssd_fused_fwd.cu -- tensor-core forward of the Mamba2 SSD for the shape
// family of the fused backward (bf16 inputs, chunk 128, dstate 128, headdim
// 64, sequence starts at chunk boundaries).
//
// The forward is the chunked scan whose backward "Deterministic bwd kernel
// for mamba2" (Mamba PR #827) breaks down per kernel; its three steps here:
//   1. chunk states   S_c = sum_t exp(E - Acs_t) dt_t x_t B_t^T      (tcgen05)
//   2. state passing  H_{c+1} = exp(E_c) H_c + S_c, reset to the initial
//                     state (or zero) where a sequence starts          (CUDA cores)
//   3. chunk scan     y_t = sum_{s<=t} (C_t.B_s) exp(Acs_t - Acs_s) dt_s x_s
//                           + exp(Acs_t) H_c C_t + D x_t               (tcgen05)
// with Acs the in-chunk cumulative sum of dt*A and E its value at the chunk's
// last token.  Step 2 writes each state entering a chunk straight into the
// packed operand form the fused backward copies into shared memory: the bf16
// pair hi = round(H), lo = round(H - hi), two [n][p] tiles in the 128-byte
// swizzled layout.
//
// Operand precision: B, C, x are the bf16 inputs themselves; every computed
// operand (w o x, the intra-chunk matrix, the states) enters the tensor cores
// as a bf16 hi + lo pair, so products keep about 16 significant bits before
// the fp32 accumulation.  The prefix sums use one fixed shuffle tree per
// chunk (the same for every launch).
#include <cstring>

#include "ssd_common.cuh"
#include "ssd_internal.h"
#include "tile_io.cuh"
#include "tmap.h"
#include "umma.cuh"

namespace ssd {

namespace {

constexpr int kQ = 128, kN = 128, kP = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitCycles = 2000000000LL;  // about one second

// Bounded mbarrier wait (records error bit 2 and gives up after about a
// second instead of hanging; results are then invalid).
__device__ __forceinline__ void fwait(uint64_t *b, uint32_t parity, int *err) {
  if (umma::mbar_try_wait(b, parity)) return;
  const long long t0 = clock64();
  while (!umma::mbar_try_wait_sleep(b, parity, 20000u)) {
    if (clock64() - t0 > kWaitCycles) {
      if (err) atomicOr(err, 2);
      return;
    }
  }
}

// 1 KB-aligned start of the dynamic shared memory (the swizzled tiles need it;
// every launch reserves 1 KB of slack for this).
__device__ __forceinline__ uint8_t *align1k(uint8_t *p) {
  const uint32_t a = umma::smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

// K-major / MN-major shared-memory descriptors of K step kk (as in the backward)
__device__ __forceinline__ uint64_t kdesc(uint32_t base, uint32_t panel_bytes, int kk) {
  return umma::smem_desc_sw128(base, 16, 1024) + uint64_t((uint32_t(kk / 64) * panel_bytes + uint32_t(kk % 64) * 2) >> 4);
}
__device__ __forceinline__ uint64_t mdesc(uint32_t base, uint32_t panel_bytes, int kk) {
  return umma::smem_desc_sw128(base, panel_bytes, 1024) + uint64_t((uint32_t(kk) * 128) >> 4);
}

// Inclusive prefix sum of v over the 128 tokens of a chunk held by the
// threads [g0, g0 + 128) (thread g0 + t holds token t): shuffle tree inside
// each warp, then the warp totals of the lower warps added in warp order.
// wtot: 4 floats of shared memory owned by this group; `sync` is a barrier
// over every thread that calls this.
template <class Sync>
__device__ __forceinline__ float chunk_scan128(float v, float *wtot, int t, Sync sync) {
  const int lane = t & 31, w = t >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) wtot[w] = v;
  sync();
  float pre = 0.f;
  for (int k = 0; k < w; ++k) pre += wtot[k];
  return v + pre;
}

struct FwdParams {
  Shape s;
  const float *dt, *A, *D, *init;
  const int32_t *seq_idx;
  float *ST;        // (b, nc, H, N, P) fp32: chunk states, transposed, n-major
  float *decay;     // (b, nc, H): exp(E) of each chunk
  float *states;    // (b, nc, H) packed 32 KB tiles: the state entering each chunk
  __nv_bfloat16 *y;
  float *y_acc;     // fp32 partial y (state halves of a 256-wide state, see fused_fwd_split)
  int y_mode;       // 0: y in bf16; 1: partial y to y_acc; 2: y = y_acc + this partial, in bf16
  int slices;       // head slices per (chunk, group) unit of the state and scan kernels
  int *err;
};

// =============================================== 1. chunk states (tcgen05) ==
// One CTA of 128 threads per (batch row, chunk, group, head slice); thread t owns token t
// (and TMEM lane t = state row n for the result).  Per head: w = exp(E - Acs)
// dt, w o x as a bf16 hi/lo pair in shared memory, S^T = B^T (w o x) on the
// tensor cores (M = n, N = p, K = t) into one of two TMEM buffers, and the
// previous head's S^T stored while this head's product runs.
constexpr uint32_t K1_B = 0;         // B chunk [t][n] bf16, 2 panels
constexpr uint32_t K1_X = 32768;     // x [t][p] bf16, 2 stages of 16 KB
constexpr uint32_t K1_WH = 65536;    // (w o x) hi [t][p]
constexpr uint32_t K1_WL = 81920;    // (w o x) lo
constexpr uint32_t K1_STG = 98304;    // per warp: 32 rows x 16 floats, the store staging of S^T
constexpr uint32_t K1_SMALL = 106496;
struct K1Small {
  float wtot[2][4];
  uint64_t bfull, xfull[2], mma;
  uint32_t tmem;
};
constexpr uint32_t K1_SMEM = K1_SMALL + 256 + 1024;

__global__ void __launch_bounds__(128) fwd_state_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_x,
                                                        const __grid_constant__ CUtensorMap tm_b) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *const base = align1k(smem_raw);
  K1Small *sm = reinterpret_cast<K1Small *>(base + K1_SMALL);
  const Shape &s = p.s;
  const int t = threadIdx.x, warp = t >> 5;
  // unit: (batch row, chunk, group, head slice); a slice's heads run in order
  const int unit = blockIdx.x, ns = p.slices;
  const int64_t gn = s.G * ns;
  const int gsl = int(unit % gn), g = gsl / ns;
  const int c = int((unit / gn) % s.nc), bi = int(unit / (gn * s.nc));
  const int row0 = bi * int(s.T) + c * kQ;
  const int nh = int(s.hpg) / ns;                 // heads of this unit
  const int hb = g * int(s.hpg) + (gsl % ns) * nh;   // its first head

  if (warp == 0) {
    umma::tmem_alloc(&sm->tmem, 128);
    umma::tmem_relinquish();
  }
  if (t == 0) {
    umma::mbar_init(&sm->bfull, 1);
    umma::mbar_init(&sm->xfull[0], 1);
    umma::mbar_init(&sm->xfull[1], 1);
    umma::mbar_init(&sm->mma, 1);
    umma::fence_mbar_init();
    umma::mbar_expect_tx(&sm->bfull, 32768);
    for (int j = 0; j < 2; ++j)
      umma::tma_load_2d(base + K1_B + j * 16384, &tm_b, g * kN + j * 64, row0, &sm->bfull);
    for (int k = 0; k < 2 && k < nh; ++k) {
      umma::mbar_expect_tx(&sm->xfull[k], 16384);
      umma::tma_load_2d(base + K1_X + k * 16384, &tm_x, (hb + k) * kP, row0, &sm->xfull[k]);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = sm->tmem;
  const uint32_t lane_off = uint32_t(32 * warp) << 16;
  const uint32_t aB = umma::smem_u32(base + K1_B), aWh = umma::smem_u32(base + K1_WH),
                 aWl = umma::smem_u32(base + K1_WL);
  constexpr uint32_t id_mm64 = umma::idesc_bf16_f32(128, 64, 1, 1);

  // S^T of head k from TMEM buffer k & 1 to ST (row n = t: 64 contiguous
  // floats), 16 columns at a time through this warp's staging rows, so that
  // each store instruction writes 8 rows x 64 contiguous bytes
  uint8_t *const stg = base + K1_STG + warp * 2048;
  const int lane = t & 31;
  auto store_state = [&](int k) {
    const int64_t h = int64_t(hb) + k;
    float *o = p.ST + (((int64_t(bi) * s.nc + c) * s.H + h) * kN + 32 * warp) * kP;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float v[16];
      umma::tmem_ld16(tmem + lane_off + 64 * (k & 1) + 16 * j, v);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *stage_slot(stg, lane, i) = make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                                               __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = 8 * i + (lane >> 2), ch = lane & 3;
        __stcg(reinterpret_cast<uint4 *>(o + int64_t(row) * kP + 16 * j + 4 * ch), *stage_slot(stg, row, ch));
      }
      __syncwarp();
    }
  };

  float dt_next = __ldg(p.dt + int64_t(row0 + t) * s.H + hb);
  for (int k = 0; k < nh; ++k) {
    const int64_t h = int64_t(hb) + k;
    const float dtv = dt_next;
    if (k + 1 < nh) dt_next = __ldg(p.dt + int64_t(row0 + t) * s.H + h + 1);
    const float Ah = __ldg(p.A + h) * kLog2e;
    float *wt = sm->wtot[k & 1];
    const float cum = chunk_scan128(dtv, wt, t, [] { __syncthreads(); });
    const float cumE = ((wt[0] + wt[1]) + wt[2]) + wt[3];   // the same bits as token 127's cum
    const float w = umma::ex2_approx((cumE - cum) * Ah) * dtv;   // exp(E - Acs_t) dt_t
    if (t == 0) __stcg(p.decay + (int64_t(bi) * s.nc + c) * s.H + h, umma::ex2_approx(cumE * Ah));
    fwait(&sm->xfull[k & 1], uint32_t((k >> 1) & 1), p.err);
    if (k >= 1) {
      fwait(&sm->mma, uint32_t((k - 1) & 1), p.err);   // the product of head k-1 has read w o x
      umma::fence_after_sync();
    }
    {
      const uint8_t *xs = base + K1_X + (k & 1) * 16384;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        float v[8];
        ld8_bf16(xs, t, 8 * c8, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] *= w;
        st8_bf16_hilo(base + K1_WH, base + K1_WL, t, 8 * c8, v);
      }
    }
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    if (t == 0) {
      if (k + 2 < nh) {   // x of head k has been read: stage k & 1 takes head k + 2
        umma::mbar_expect_tx(&sm->xfull[k & 1], 16384);
        umma::tma_load_2d(base + K1_X + (k & 1) * 16384, &tm_x, int(h + 2) * kP, row0, &sm->xfull[k & 1]);
      }
      if (k == 0) fwait(&sm->bfull, 0, p.err);
      umma::fence_after_sync();
      for (int part = 0; part < 2; ++part)
        for (int kk = 0; kk < kQ; kk += 16)
          umma::mma_bf16(tmem + 64 * (k & 1), mdesc(aB, 16384, kk), mdesc(part ? aWl : aWh, 16384, kk), id_mm64,
                         (part > 0) || (kk > 0));
      umma::mma_commit(&sm->mma);
    }
    __syncwarp();
    if (k >= 1) store_state(k - 1);   // its product completed before this head's w o x was written
    umma::fence_before_sync();
  }
  fwait(&sm->mma, uint32_t((nh - 1) & 1), p.err);
  umma::fence_after_sync();
  store_state(nh - 1);
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, 128);
  }
}

// ============================================ 2. state passing (CUDA cores) ==
// Thread per (batch row, head, state row n, 8 consecutive p); serial over
// chunks: the state entering chunk c (the initial state or zero where chunk c
// starts a sequence) is written in packed form, then carried:
// H <- exp(E_c) H + S_c.
__global__ void __launch_bounds__(256) fwd_pass_kernel(const FwdParams p) {
  const Shape &s = p.s;
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= s.b * s.H * kN * 8) return;
  const int oct = int(idx & 7), n = int((idx >> 3) % kN);
  const int64_t h = (idx >> 3) / kN % s.H, bi = (idx >> 3) / (kN * s.H);
  const int p0 = 8 * oct;
  float carry[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) carry[i] = 0.f;
  const float *st = p.ST + ((bi * s.nc * s.H + h) * kN + n) * kP + p0;   // chunk 0
  float4 s0 = __ldcs(reinterpret_cast<const float4 *>(st)), s1 = __ldcs(reinterpret_cast<const float4 *>(st + 4));
  for (int64_t c = 0; c < s.nc; ++c) {
    const int64_t t0 = c * kQ;
    if (is_seq_start(p.seq_idx, bi, s.T, t0)) {
      const float *in = p.init ? p.init + ((seq_of(p.seq_idx, bi, s.T, t0) * s.H + h) * kP + p0) * kN + n : nullptr;
#pragma unroll
      for (int i = 0; i < 8; ++i) carry[i] = in ? __ldg(in + i * kN) : 0.f;
    }
    uint8_t *tile = reinterpret_cast<uint8_t *>(p.states + ((bi * s.nc + c) * s.H + h) * (kP * kN));
    st8_bf16_hilo(tile, tile + 16384, n, p0, carry);
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    if (c + 1 < s.nc) {   // next chunk's S in flight while this one is folded in
      const float *nx = st + (c + 1) * s.H * kN * kP;
      s0 = __ldcs(reinterpret_cast<const float4 *>(nx));
      s1 = __ldcs(reinterpret_cast<const float4 *>(nx + 4));
    }
    const float e = __ldg(p.decay + (bi * s.nc + c) * s.H + h);
#pragma unroll
    for (int i = 0; i < 8; ++i) carry[i] = fmaf(e, carry[i], sv[i]);
  }
}

// ================================================= 3. chunk scan (tcgen05) ==
// One CTA of 256 threads per (batch row, chunk, group, head slice).  Warp w handles TMEM
// lane quadrant q = w % 4 (tokens 32q..32q+31) and half w / 4 of the columns.
// Per head: the intra-chunk matrix M'[t,s] = (C_t.B_s) exp(Acs_t - Acs_s) dt_s
// for s <= t (plus D on the diagonal, which folds the skip term into the
// product) as a bf16 hi/lo pair; Y = M' x and C H (saved state, packed pair)
// on the tensor cores; y = Y + exp(Acs_t) (C H)_t, stored while the next
// head's products run.  TMEM: C B^T (columns 0-127), then two head buffers of
// 128 columns (Y at +0, C H at +64).
constexpr uint32_t K3_B = 0, K3_C = 32768;   // [t][n] bf16, 2 panels each
constexpr uint32_t K3_X = 65536;             // x [t][p], 2 stages of 16 KB
constexpr uint32_t K3_H = 98304;             // packed states, 2 stages of 32 KB (hi | lo)
constexpr uint32_t K3_MH = 163840;           // M' hi [t][s], 2 panels
constexpr uint32_t K3_ML = 196608;           // M' lo
constexpr uint32_t K3_SMALL = 229376;
struct K3Small {
  float a2[kQ];      // Acs in log2 units, current head
  float dtv[kQ];     // step sizes, current head
  float ecd[kQ];     // column factors exp(Acs_ref - Acs_s) dt_s, ref = s | 15, current head
  float wtot[2][2][4];
  uint64_t bcfull, cbdone, xfull[2], hfull[2], mma;
  uint32_t tmem;
};
constexpr uint32_t K3_SMEM = K3_SMALL + 2048 + 1024;
static_assert(sizeof(K3Small) <= 2048, "small region");
static_assert(K3_SMEM <= 232448, "shared memory budget");

__global__ void __launch_bounds__(256, 1) fwd_scan_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_x,
                                                          const __grid_constant__ CUtensorMap tm_b,
                                                          const __grid_constant__ CUtensorMap tm_c) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *const base = align1k(smem_raw);
  K3Small *sm = reinterpret_cast<K3Small *>(base + K3_SMALL);
  const Shape &s = p.s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = warp & 3, half = warp >> 2;
  const int r = 32 * q + lane;   // token row of this thread
  // unit: (batch row, chunk, group, head slice); a slice's heads run in order
  const int unit = blockIdx.x, ns = p.slices;
  const int64_t gn = s.G * ns;
  const int gsl = int(unit % gn), g = gsl / ns;
  const int c = int((unit / gn) % s.nc), bi = int(unit / (gn * s.nc));
  const int row0 = bi * int(s.T) + c * kQ;
  const int nh = int(s.hpg) / ns;                 // heads of this unit
  const int hb = g * int(s.hpg) + (gsl % ns) * nh;   // its first head
  const float *states = p.states + ((int64_t(bi) * s.nc + c) * s.H + int64_t(hb)) * (kP * kN);

  if (warp == 0) {
    umma::tmem_alloc(&sm->tmem, 512);
    umma::tmem_relinquish();
  }
  if (tid == 0) {
    umma::mbar_init(&sm->bcfull, 1);
    umma::mbar_init(&sm->cbdone, 1);
    for (int j = 0; j < 2; ++j) {
      umma::mbar_init(&sm->xfull[j], 1);
      umma::mbar_init(&sm->hfull[j], 1);
    }
    umma::mbar_init(&sm->mma, 1);
    umma::fence_mbar_init();
    umma::mbar_expect_tx(&sm->bcfull, 65536);
    for (int j = 0; j < 2; ++j) {
      umma::tma_load_2d(base + K3_B + j * 16384, &tm_b, g * kN + j * 64, row0, &sm->bcfull);
      umma::tma_load_2d(base + K3_C + j * 16384, &tm_c, g * kN + j * 64, row0, &sm->bcfull);
    }
    for (int k = 0; k < 2 && k < nh; ++k) {
      umma::mbar_expect_tx(&sm->xfull[k], 16384);
      umma::tma_load_2d(base + K3_X + k * 16384, &tm_x, (hb + k) * kP, row0, &sm->xfull[k]);
      umma::mbar_expect_tx(&sm->hfull[k], kP * kN * 4);
      umma::bulk_load(base + K3_H + k * 32768, states + int64_t(k) * kP * kN, kP * kN * 4, &sm->hfull[k]);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = sm->tmem;
  const uint32_t lane_off = uint32_t(32 * q) << 16;
  const uint32_t aB = umma::smem_u32(base + K3_B), aC = umma::smem_u32(base + K3_C);
  const uint32_t aMh = umma::smem_u32(base + K3_MH), aMl = umma::smem_u32(base + K3_ML);
  constexpr uint32_t id_kk128 = umma::idesc_bf16_f32(128, 128, 0, 0);
  constexpr uint32_t id_km64 = umma::idesc_bf16_f32(128, 64, 0, 1);
  if (tid == 0) {
    fwait(&sm->bcfull, 0, p.err);
    umma::fence_after_sync();
    for (int kk = 0; kk < kN; kk += 16) umma::mma_bf16(tmem, kdesc(aC, 16384, kk), kdesc(aB, 16384, kk), id_kk128, kk > 0);
    umma::mma_commit(&sm->cbdone);
  }
  __syncwarp();
  if (lane == 0) fwait(&sm->cbdone, 0, p.err);
  __syncwarp();
  umma::fence_after_sync();

  // y of head k from TMEM buffer k & 1: this thread's row, 32 columns.  The
  // rows go to and from global memory through this warp's 2 KB of staging in
  // the x stage (bf16 y) and the H stage (the fp32 partials of the split form)
  // of head k, both free once head k's products are done, so that each global
  // access instruction moves 8 rows x 64 contiguous bytes.
  auto store_y = [&](int k, float eacs) {
    const int64_t h = int64_t(hb) + k;
    const uint32_t buf = 128 + 128 * uint32_t(k & 1);
    uint8_t *const stg = base + K3_X + (k & 1) * 16384 + warp * 2048;
    uint8_t *const stg32 = base + K3_H + (k & 1) * 32768 + warp * 2048;
    float *const accw = p.y_acc ? p.y_acc + (int64_t(row0 + 32 * q) * s.H + h) * kP + 32 * half : nullptr;
    const int64_t pitch = s.H * kP;   // elements between consecutive token rows
    const int srow = lane >> 2, sch = lane & 3;   // the row (of each 8) and chunk this lane moves
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float yv[16], ch[16];
      umma::tmem_ld16(tmem + lane_off + buf + 32 * half + 16 * j, yv);
      umma::tmem_ld16(tmem + lane_off + buf + 64 + 32 * half + 16 * j, ch);
#pragma unroll
      for (int i = 0; i < 16; ++i) yv[i] = fmaf(eacs, ch[i], yv[i]);
      if (p.y_mode == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *stage_slot(stg32, lane, i) = make_uint4(__float_as_uint(yv[4 * i]), __float_as_uint(yv[4 * i + 1]),
                                                   __float_as_uint(yv[4 * i + 2]), __float_as_uint(yv[4 * i + 3]));
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i)
          __stcg(reinterpret_cast<uint4 *>(accw + (8 * i + srow) * pitch + 16 * j + 4 * sch),
                 *stage_slot(stg32, 8 * i + srow, sch));
        __syncwarp();
        continue;
      }
      if (p.y_mode == 2) {   // the other state half's partial first, then this one
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *stage_slot(stg32, 8 * i + srow, sch) =
              __ldcs(reinterpret_cast<const uint4 *>(accw + (8 * i + srow) * pitch + 16 * j + 4 * sch));
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 a = *stage_slot(stg32, lane, i);
          yv[4 * i] = __uint_as_float(a.x) + yv[4 * i];
          yv[4 * i + 1] = __uint_as_float(a.y) + yv[4 * i + 1];
          yv[4 * i + 2] = __uint_as_float(a.z) + yv[4 * i + 2];
          yv[4 * i + 3] = __uint_as_float(a.w) + yv[4 * i + 3];
        }
        __syncwarp();
      }
      uint4 u[2];
      __nv_bfloat162 *yb = reinterpret_cast<__nv_bfloat162 *>(u);
#pragma unroll
      for (int i = 0; i < 8; ++i) yb[i] = __floats2bfloat162_rn(yv[2 * i], yv[2 * i + 1]);
      *stage_slot(stg, lane, 2 * j) = u[0];
      *stage_slot(stg, lane, 2 * j + 1) = u[1];
    }
    if (p.y_mode != 1) {
      __syncwarp();
      __nv_bfloat16 *const yw = p.y + (int64_t(row0 + 32 * q) * s.H + h) * kP + 32 * half;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4 *>(yw + (8 * i + srow) * pitch + 8 * sch) = *stage_slot(stg, 8 * i + srow, sch);
    }
    // both stages are next written by the copies of head k + 2's x and H (async proxy)
    umma::fence_proxy_async_smem();
  };

  float eacs_prev = 0.f;
  const int grp = tid >> 7, t = tid & 127;   // two groups of 128 threads run the same scan
  float dt_next = __ldg(p.dt + int64_t(row0 + t) * s.H + hb);
  for (int k = 0; k < nh; ++k) {
    const int64_t h = int64_t(hb) + k;
    const float dtv = dt_next;
    if (k + 1 < nh) dt_next = __ldg(p.dt + int64_t(row0 + t) * s.H + h + 1);
    const float Ah = __ldg(p.A + h) * kLog2e, Dh = __ldg(p.D + h);
    // ---- step sizes: cumulative decay (both groups compute identical bits)
    const float cum = chunk_scan128(dtv, sm->wtot[k & 1][grp], t, [] { __syncthreads(); });
    const float a2t = cum * Ah;
    // a2 of the last token of this token's 16-token block (the same warp)
    const float a2ref = __shfl_sync(0xffffffffu, a2t, (t & 31) | 15);
    if (grp == 0) {
      sm->a2[t] = a2t;
      sm->dtv[t] = dtv;
      sm->ecd[t] = umma::ex2_approx(a2ref - a2t) * dtv;
    }
    if (k >= 1 && lane == 0) fwait(&sm->mma, uint32_t((k - 1) & 1), p.err);   // head k-1 products done
    __syncwarp();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const float a2r = sm->a2[r];
    const float eacs = umma::ex2_approx(a2r);

    // ---- M' of this head: blocks of 16 columns j = half, half + 2, ... (balanced within a quadrant)
#pragma unroll
    for (int jb = 0; jb < 4; ++jb) {
      const int s0 = 16 * (2 * jb + half);
      uint8_t *ph = base + K3_MH + (s0 >> 6) * 16384, *pl = base + K3_ML + (s0 >> 6) * 16384;
      const int cc = s0 & 63;
      if (s0 > 32 * q + 31) {   // strictly above the diagonal for the whole quadrant
        const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        st8_bf16_hilo(ph, pl, r, cc, z);
        st8_bf16_hilo(ph, pl, r, cc + 8, z);
        continue;
      }
      float cb[16];
      umma::tmem_ld16(tmem + lane_off + s0, cb);
      if (s0 + 16 <= 32 * q) {
        // every column of the block precedes every row of the quadrant: the decay
        // exp(Acs_r - Acs_s) as the row factor exp(Acs_r - Acs_ref) (ref = the block's
        // last column) times the column factor, both at most one, so one exp per row
        const float er = umma::ex2_approx(a2r - sm->a2[s0 + 15]);
#pragma unroll
        for (int e8 = 0; e8 < 2; ++e8) {
          const float4 c0 = *reinterpret_cast<const float4 *>(&sm->ecd[s0 + 8 * e8]);
          const float4 c1 = *reinterpret_cast<const float4 *>(&sm->ecd[s0 + 8 * e8 + 4]);
          const float ec[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = cb[8 * e8 + i] * er * ec[i];
          st8_bf16_hilo(ph, pl, r, cc + 8 * e8, v);
        }
        continue;
      }
#pragma unroll
      for (int e8 = 0; e8 < 2; ++e8) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int sc = s0 + 8 * e8 + i;
          const float m = (sc <= r) ? cb[8 * e8 + i] * umma::ex2_approx(a2r - sm->a2[sc]) * sm->dtv[sc] : 0.f;
          v[i] = (sc == r) ? m + Dh : m;
        }
        st8_bf16_hilo(ph, pl, r, cc + 8 * e8, v);
      }
    }
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      // products of head k: C H and Y = M' x into buffer k & 1
      const uint32_t buf = 128 + 128 * uint32_t(k & 1);
      const uint32_t aH = umma::smem_u32(base + K3_H + (k & 1) * 32768);
      const uint32_t aX = umma::smem_u32(base + K3_X + (k & 1) * 16384);
      fwait(&sm->hfull[k & 1], uint32_t((k >> 1) & 1), p.err);
      fwait(&sm->xfull[k & 1], uint32_t((k >> 1) & 1), p.err);
      umma::fence_after_sync();
      for (int part = 0; part < 2; ++part)
        for (int kk = 0; kk < kN; kk += 16)
          umma::mma_bf16(tmem + buf + 64, kdesc(aC, 16384, kk), mdesc(aH + part * 16384, 16384, kk), id_km64,
                         (part > 0) || (kk > 0));
      for (int part = 0; part < 2; ++part)
        for (int kk = 0; kk < kQ; kk += 16)
          umma::mma_bf16(tmem + buf, kdesc(part ? aMl : aMh, 16384, kk), mdesc(aX, 16384, kk), id_km64,
                         (part > 0) || (kk > 0));
      umma::mma_commit(&sm->mma);
    }
    __syncwarp();
    // ---- y of the previous head while this head's products run
    if (k >= 1) store_y(k - 1, eacs_prev);
    eacs_prev = eacs;
    umma::fence_before_sync();
    __syncthreads();
    if (tid == 0 && k >= 1 && k + 1 < nh) {
      // head k-1's products are done (waited above): its x and H stages take head k + 1
      const int st = (k + 1) & 1;
      umma::mbar_expect_tx(&sm->xfull[st], 16384);
      umma::tma_load_2d(base + K3_X + st * 16384, &tm_x, int(h + 1) * kP, row0, &sm->xfull[st]);
      umma::mbar_expect_tx(&sm->hfull[st], kP * kN * 4);
      umma::bulk_load(base + K3_H + st * 32768, states + int64_t(k + 1) * kP * kN, kP * kN * 4, &sm->hfull[st]);
      if (k + 2 < nh) {
        umma::tma_prefetch_2d(&tm_x, int(h + 2) * kP, row0);
        umma::prefetch_l2(states + int64_t(k + 2) * kP * kN, kP * kN * 4);
      }
    }
  }
  if (lane == 0) fwait(&sm->mma, uint32_t((nh - 1) & 1), p.err);
  __syncwarp();
  umma::fence_after_sync();
  store_y(nh - 1, eacs_prev);
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, 512);
  }
}

struct FwdWs {
  int *status;
  float *ST, *decay;
};

FwdWs carve_fwd_fused(Carver &cv, const Shape &s) {
  FwdWs w;
  w.status = cv.take<int>(64);
  w.ST = cv.take<float>(s.b * s.nc * s.H * kN * kP);
  w.decay = cv.take<float>(s.b * s.nc * s.H);
  return w;
}

// Head slices per (chunk, group) unit: the power of two (at least 16 heads a
// slice) that minimises the heads run by the busiest SM of the scan kernel
// (one unit per SM at a time), the smallest on a tie.  The forward's heads are
// independent, so slicing changes which CTA runs a head and nothing else.
int fwd_slices(const Shape &s, int64_t units) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess || sms <= 0)
    return 1;
  int best = 1;
  int64_t best_load = (units + sms - 1) / sms * s.hpg;
  for (int ns = 2; s.hpg % ns == 0 && s.hpg / ns >= 16 && units * ns <= (int64_t(1) << 30); ns *= 2) {
    const int64_t load = (units * ns + sms - 1) / sms * (s.hpg / ns);
    if (load < best_load) {
      best = ns;
      best_load = load;
    }
  }
  return best;
}

}  // namespace

size_t fused_fwd_workspace(const Shape &s) {
  Carver cv(nullptr);
  carve_fwd_fused(cv, s);
  return cv.bytes();
}

int *fused_fwd_status(const Shape &s, void *ws) {
  Carver cv(ws);
  return carve_fwd_fused(cv, s).status;
}

cudaError_t fused_fwd(const Shape &s, const Args &a, void *ws, cudaStream_t st) {
  Carver cv(ws);
  FwdWs w = carve_fwd_fused(cv, s);
  CUtensorMap tm_x, tm_b, tm_c;
  const uint64_t rows = uint64_t(s.b * s.T);
  if (!make_tmap_2d(&tm_x, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, uint64_t(s.H * kP), uint64_t(s.H * kP), 64,
                    128, true) ||
      !make_tmap_2d(&tm_b, a.B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, uint64_t(s.G * kN), uint64_t(s.G * kN), 64,
                    128, true) ||
      !make_tmap_2d(&tm_c, a.C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, uint64_t(s.G * kN), uint64_t(s.G * kN), 64,
                    128, true))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaMemsetAsync(w.status, 0, 64 * sizeof(int), st);
  if (err != cudaSuccess) return err;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.s = s;
  p.dt = a.dt;
  p.A = a.A;
  p.D = a.D;
  p.init = a.init;
  p.seq_idx = a.seq_idx;
  p.ST = w.ST;
  p.decay = w.decay;
  p.states = a.states_out;
  p.y = static_cast<__nv_bfloat16 *>(a.y);
  p.err = w.status;
  if ((err = cudaFuncSetAttribute(fwd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, K1_SMEM)) !=
          cudaSuccess ||
      (err = cudaFuncSetAttribute(fwd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, K3_SMEM)) !=
          cudaSuccess)
    return err;
  p.slices = fwd_slices(s, s.b * s.nc * s.G);
  const unsigned units = unsigned(s.b * s.nc * s.G * p.slices);
  fwd_state_kernel<<<units, 128, K1_SMEM, st>>>(p, tm_x, tm_b);
  fwd_pass_kernel<<<unsigned((s.b * s.H * kN * 8 + 255) / 256), 256, 0, st>>>(p);
  fwd_scan_kernel<<<units, 256, K3_SMEM, st>>>(p, tm_x, tm_b, tm_c);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// dstate 128, chunk length a larger multiple of 128: the kernels above in
// 128-token chunks.  The chunked form is exact for any chunk length (the
// state entering a chunk and every per-token result are those of the
// token-by-token recurrence), so only the saved states differ: one per 128
// tokens here, packed, kept in the workspace (`aux`) for the backward, and
// the caller's buffer gets the fp32 (b, nc, H, P, N) states entering each of
// its chunks (every ratio-th of them).
namespace {

struct Chunk128Ws {
  float *aux;    // packed states (b, T / 128, H) tiles of P x 128
  void *inner;   // the 128-token forward's workspace (its status word first)
};

Chunk128Ws carve_chunk128(Carver &cv, const Shape &s) {
  const Shape h = fused_chunk128_shape(s);
  Chunk128Ws w;
  w.aux = cv.take<float>(h.b * h.nc * h.H * kP * kN);
  w.inner = cv.take<char>(int64_t(fused_fwd_workspace(h)));
  return w;
}

// fp32 state entering caller chunk c (the packed tile of 128-token chunk
// c * ratio); one CTA per (b, caller chunk, head)
__global__ void __launch_bounds__(256) chunk_states_view_kernel(Shape s, int ratio, const float *__restrict__ aux,
                                                                float *__restrict__ out) {
  __shared__ float t[64][129];
  const int64_t tile = blockIdx.x;   // (b * nc + c) * H + h
  const int64_t h = tile % s.H, c = tile / s.H % s.nc, bi = tile / (s.H * s.nc);
  const int64_t nch = s.T / kQ;
  const uint8_t *in = reinterpret_cast<const uint8_t *>(aux + ((bi * nch + c * ratio) * s.H + h) * (kP * kN));
  unpack_state_tile(in, out + tile * (kP * kN), kN, t);
}

}  // namespace

Shape fused_chunk128_shape(const Shape &s) {
  Shape h = s;
  h.Q = kQ;
  h.nc = s.T / kQ;
  return h;
}

bool fused_chunk128_supported(const Shape &s, bool bf16) {
  return s.Q > kQ && s.Q % kQ == 0 && s.T % kQ == 0 && fused_bwd_supported(fused_chunk128_shape(s), bf16);
}

size_t fused_fwd_chunk128_workspace(const Shape &s) {
  Carver cv(nullptr);
  carve_chunk128(cv, s);
  return cv.bytes();
}

float *fused_chunk128_aux(const Shape &s, void *ws) {
  Carver cv(ws);
  return carve_chunk128(cv, s).aux;
}

int *fused_fwd_chunk128_status(const Shape &s, void *ws) {
  Carver cv(ws);
  return fused_fwd_status(fused_chunk128_shape(s), carve_chunk128(cv, s).inner);
}

cudaError_t fused_fwd_chunk128(const Shape &s, const Args &a, void *ws, cudaStream_t st) {
  Carver cv(ws);
  const Chunk128Ws w = carve_chunk128(cv, s);
  Args ai = a;
  ai.states_out = w.aux;
  cudaError_t err = fused_fwd(fused_chunk128_shape(s), ai, w.inner, st);
  if (err != cudaSuccess || !a.states_out) return err;
  chunk_states_view_kernel<<<unsigned(s.b * s.nc * s.H), 256, 0, st>>>(s, int(s.Q / kQ), w.aux, a.states_out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// dstate 256 (one group), chunk 128 or 256: the recurrence never mixes state
// dimensions, so the scan is the sum of two scans over the state halves
// n < 128 and n >= 128 (B, C split the same way), with D counted once.  Each
// half runs the kernels above as a dstate-128 problem in 128-token chunks (the
// chunked form is exact for any chunk length); the halves' y are added in
// fp32 before the single rounding to bf16.  The saved states of both halves
// (packed, every 128 tokens) live in the forward workspace (`aux`), and the
// caller's state buffer receives the fp32 (b, nc, H, P, 256) states entering
// each chunk of the caller's chunk length.
namespace {

Shape half_shape(const Shape &s) {
  Shape h = s;
  h.N = kN;
  h.Q = kQ;
  h.nc = s.T / kQ;
  return h;
}

struct SplitFwdWs {
  float *aux;   // packed states of both halves: [half][b][nc'][H] tiles of P x 128
  FwdWs k;      // status, ST, decay of one half at a time
  float *y_acc, *init_half, *zeros;
};

SplitFwdWs carve_fwd_split(Carver &cv, const Shape &s) {
  const Shape h = half_shape(s);
  SplitFwdWs w;
  w.aux = cv.take<float>(2 * h.b * h.nc * h.H * kP * kN);
  w.k = carve_fwd_fused(cv, h);
  w.y_acc = cv.take<float>(s.b * s.T * s.H * kP);
  w.init_half = cv.take<float>(s.nseq * s.H * kP * kN);
  w.zeros = cv.take<float>(s.H);
  return w;
}

// init (nseq, H, P, 256) -> its half j as (nseq, H, P, 128)
__global__ void init_half_kernel(int64_t rows, int j, const float *__restrict__ init, float *__restrict__ out) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;   // one float4 of the half
  if (i >= rows * (kN / 4)) return;
  const int64_t row = i / (kN / 4), q = i % (kN / 4);
  reinterpret_cast<float4 *>(out)[i] = __ldg(reinterpret_cast<const float4 *>(init + row * 2 * kN + j * kN) + q);
}

// fp32 (b, nc, H, P, 256) states entering each caller chunk (ratio = caller
// chunk / 128) from the packed halves; one CTA per (b, caller chunk, head, half)
__global__ void __launch_bounds__(256) states_view_kernel(Shape s, int ratio, const float *__restrict__ aux,
                                                           float *__restrict__ out) {
  __shared__ float t[64][129];
  const int64_t tile = blockIdx.x;   // ((b * nc + c) * H + h) * 2 + j
  const int j = int(tile & 1);
  const int64_t h = (tile >> 1) % s.H, c = (tile >> 1) / s.H % s.nc, bi = (tile >> 1) / (s.H * s.nc);
  const int64_t nch = s.T / kQ;
  const uint8_t *in = reinterpret_cast<const uint8_t *>(
      aux + (((int64_t(j) * s.b + bi) * nch + c * ratio) * s.H + h) * (kP * kN));
  unpack_state_tile(in, out + (((bi * s.nc + c) * s.H + h) * kP) * (2 * kN) + j * kN, 2 * kN, t);
}

}  // namespace

bool fused_split_supported(const Shape &s, bool bf16) {
  // (the backward splits each group's heads into two or four slices: an even head count)
  return bf16 && s.N == 2 * kN && s.G == 1 && s.H % 2 == 0 && s.P == kP && (s.Q == kQ || s.Q == 2 * kQ) &&
         s.T % s.Q == 0 &&
         s.b * (s.T / kQ) <= (int64_t(1) << 30) && s.b * s.T <= (int64_t(1) << 30);
}

size_t fused_fwd_split_workspace(const Shape &s) {
  Carver cv(nullptr);
  carve_fwd_split(cv, s);
  return cv.bytes();
}

float *fused_split_aux(const Shape &s, void *ws) {
  Carver cv(ws);
  return carve_fwd_split(cv, s).aux;
}

int *fused_fwd_split_status(const Shape &s, void *ws) {
  Carver cv(ws);
  return carve_fwd_split(cv, s).k.status;
}

cudaError_t fused_fwd_split(const Shape &s, const Args &a, void *ws, cudaStream_t st) {
  const Shape h = half_shape(s);
  Carver cv(ws);
  SplitFwdWs w = carve_fwd_split(cv, s);
  const uint64_t rows = uint64_t(s.b * s.T);
  CUtensorMap tm_x, tm_b[2], tm_c[2];
  if (!make_tmap_2d(&tm_x, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, uint64_t(s.H * kP), uint64_t(s.H * kP), 64,
                    128, true))
    return cudaErrorInvalidValue;
  for (int j = 0; j < 2; ++j) {
    // the half j of each token's 256 state values: 128 columns at offset 128 j, row pitch 256
    const __nv_bfloat16 *Bj = static_cast<const __nv_bfloat16 *>(a.B) + j * kN;
    const __nv_bfloat16 *Cj = static_cast<const __nv_bfloat16 *>(a.C) + j * kN;
    if (!make_tmap_2d(&tm_b[j], Bj, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, kN, 2 * kN, 64, 128, true) ||
        !make_tmap_2d(&tm_c[j], Cj, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, kN, 2 * kN, 64, 128, true))
      return cudaErrorInvalidValue;
  }
  cudaError_t err;
  if ((err = cudaMemsetAsync(w.k.status, 0, 64 * sizeof(int), st)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(w.zeros, 0, size_t(s.H) * sizeof(float), st)) != cudaSuccess) return err;
  if ((err = cudaFuncSetAttribute(fwd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, K1_SMEM)) !=
          cudaSuccess ||
      (err = cudaFuncSetAttribute(fwd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, K3_SMEM)) !=
          cudaSuccess)
    return err;
  const int64_t tiles = h.b * h.nc * h.H * kP * kN;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.s = h;
  p.slices = fwd_slices(h, h.b * h.nc);
  const unsigned units = unsigned(h.b * h.nc * p.slices);
  p.dt = a.dt;
  p.A = a.A;
  p.seq_idx = a.seq_idx;
  p.ST = w.k.ST;
  p.decay = w.k.decay;
  p.y = static_cast<__nv_bfloat16 *>(a.y);
  p.y_acc = w.y_acc;
  p.err = w.k.status;
  // chunk states and state passing, one half at a time
  for (int j = 0; j < 2; ++j) {
    if (a.init) {
      const int64_t rws = s.nseq * s.H * kP;
      init_half_kernel<<<unsigned((rws * (kN / 4) + 255) / 256), 256, 0, st>>>(rws, j, a.init, w.init_half);
    }
    p.init = a.init ? w.init_half : nullptr;
    p.states = w.aux + j * tiles;
    fwd_state_kernel<<<units, 128, K1_SMEM, st>>>(p, tm_x, tm_b[j]);
    fwd_pass_kernel<<<unsigned((h.b * h.H * kN * 8 + 255) / 256), 256, 0, st>>>(p);
  }
  if (a.states_out)   // (a caller that reads the packed states itself passes none)
    states_view_kernel<<<unsigned(s.b * s.nc * s.H * 2), 256, 0, st>>>(s, int(s.Q / kQ), w.aux, a.states_out);
  // y: half 0 (with D) into fp32, then half 1 (no D) added and rounded once
  for (int j = 0; j < 2; ++j) {
    p.states = w.aux + j * tiles;
    p.D = j == 0 ? a.D : w.zeros;
    p.y_mode = j == 0 ? 1 : 2;
    fwd_scan_kernel<<<units, 256, K3_SMEM, st>>>(p, tm_x, tm_b[j], tm_c[j]);
  }
  return cudaGetLastError();
}

}  // namespace ssd
