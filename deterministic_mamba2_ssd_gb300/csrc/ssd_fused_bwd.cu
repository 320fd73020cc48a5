// ssd_fused_bwd.cu -- fused tensor-core backward of the Mamba2 SSD for the
// shape family chunk 128, dstate 128, headdim 64, bf16 inputs.
//
// One CTA owns one (batch row b, chunk c, group g) unit and walks the
// group's heads in ascending order.  For each head it computes, on the
// tcgen05 tensor cores with TMEM accumulators, every product of the chunked
// backward that "Deterministic bwd kernel for mamba2" (Mamba PR #827) splits
// into chunk_scan_bwd_dC/_dx, chunk_state_bwd_dx/_db/_ddAcs and the
// combined dx kernel; the cumsum backward and the reverse state recurrence
// run in its CUDA-core epilogue.  Determinism comes from ownership instead
// of atomics:
//   * dB and dC of the unit's (chunk, group) are accumulated over the heads
//     inside the CTA (TMEM accumulators, head order fixed), so no cross-CTA
//     fold of them exists at all;
//   * every dx/ddt element has exactly one writer;
//   * the reverse state recurrence dH_c = dHscan_c + exp(E_c) dH_{c+1} is
//     chained between chunk CTAs: the unit of chunk c waits for the unit of
//     chunk c+1 to publish dH_{c+1} (an L2-resident ring plus a flag), so
//     each dH_c has one formula whatever the schedule;
//   * per-(chunk, head) partials of dA and dD are folded in ascending chunk
//     order by a second small kernel.
// Units are handed out in descending chunk order through an atomic ticket,
// so a unit only ever waits for a unit that is already running: no deadlock
// whatever the number of resident CTAs.
//
// Roles (576 threads): warps 0-15 epilogue (thread = one row of a 128-row
// tile and one quarter of its columns; the TMEM lane quadrant of a warp is
// its index mod 4; the intra-chunk phase instead gives each warp 16 x 16
// blocks of the causal triangle, two threads a row, over rows paired so that
// every quadrant holds the same share of it), warp 16 TMA producer, warp 17
// TMEM owner and MMA issuer.  Operand precision: bf16 operands, fp32 accumulation;
// the one product whose rounding dominates the error (dx_intra = M^T g with
// M = CB o L) runs in fp16 with exact power-of-two scaling of both operands,
// and the head-summed intra-chunk matrix for dB/dC, G~, the saved state H and
// the chained state gradient dS (in Y = B dS^T and in dB's state term) are
// split into bf16 hi + lo pairs (a single bf16 dS left dA, a sum of
// cancelling terms, at relL2 4.6e-3 on a four-head problem, and dB at 2.3e-3
// without decay, where dS accumulates over every chunk; with the pair 4.9e-4
// and 1.6e-3).
#include <cuda_fp16.h>

#include <cstring>
#include <mutex>

#include "ssd_common.cuh"
#include "ssd_internal.h"
#include "tile_io.cuh"
#include "tmap.h"
#include "umma.cuh"

namespace ssd {

namespace {

constexpr int kQ = 128, kN = 128, kP = 64;
constexpr int kEpiWarps = 16;                // 4 TMEM lane quadrants x 4 column quarters
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kTmaWarp = kEpiWarps, kMmaWarp = kEpiWarps + 1;
constexpr int kThreads = kEpiThreads + 64;

// shared memory map (offsets from the 1024-byte aligned base)
constexpr uint32_t OFF_B = 0;          // B chunk  [t][n] bf16, 2 panels x 16 KB
constexpr uint32_t OFF_C = 32768;      // C chunk  [t][n] bf16, 2 panels
constexpr uint32_t OFF_XG = 65536;     // x [t][p] 16 KB, g 16 KB (bf16 from TMA, then scaled fp16 in place)
constexpr uint32_t OFF_STG = 98304;    // fp32 [p][n] 32 KB: dS, the chained state gradient (bulk copy)
constexpr uint32_t OFF_HD = 131072;    // H hi | H lo: [n][p] bf16, 16 KB each (bulk copy of the packed
                                       // saved state); later dS hi | lo [n][p]
constexpr uint32_t OFF_GW = 163840;    // exp(Acs) o g hi | lo: [t][p] bf16; later w o x (hi half) + scratch (lo half)
constexpr uint32_t OFF_M16 = 196608;   // scaled M: [t][s] fp16, 2 panels x 16 KB
constexpr uint32_t OFF_SMALL = 229376;
constexpr uint32_t SMALL_BYTES = 3072;
constexpr uint32_t SMEM_BYTES = OFF_SMALL + SMALL_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
// scratch that lives in the idle lo half of GW between the dC/dHscan products and the next head
constexpr uint32_t OFF_XBUF = OFF_GW + 16384;
// at the end of a unit the head-summed matrix W (hi, lo) reuses the x/g stages
constexpr uint32_t OFF_WHI = OFF_XG, OFF_WLO = OFF_STG;

// TMEM columns
// RA holds, in turn: C B^T (unit start), g x^T, then dHscan^T (cols 64-127,
// the half of g x^T the epilogue reads first) and C H (0-63), then Y (64-127)
// and D1 (0-63).  WS accumulates W.
constexpr uint32_t T_DB = 0, T_DC = 128, T_RA = 256, T_WS = 384;
constexpr uint32_t T_DH = T_RA + 64, T_CH = T_RA, T_Y = T_RA + 64, T_D1 = T_RA;

// Row order of the token tiles that the intra-chunk phase reads through TMEM
// lanes: C, g, G~, the fp16 M and W are held with the 16-token group q in
// rows (lanes) 32q..32q+15 and the group 7-q in rows 32q+16..32q+31, so that
// the causal triangle of g x^T and C B^T spreads evenly over the four lane
// quadrants, i.e. over the four SM sub-partitions (the quadrant holding tokens
// 96-127 in natural order had 8 of the 20 column blocks).  x, B, w o x, H and
// dS stay in natural order; every product pairs rows of one order along its
// K dimension, so C B^T, g x^T, C H and dC come out with permuted lanes and
// Y, D1, dHscan^T and dB with natural ones.
__device__ __forceinline__ int tok_of_row(int l) {   // token held in row (lane) l
  return ((l & 16) ? 7 - (l >> 5) : (l >> 5)) * 16 + (l & 15);
}
__host__ __device__ constexpr int row_of_tok(int t) {   // row (lane) holding token t
  return ((t >> 4) < 4 ? 32 * (t >> 4) : 32 * (7 - (t >> 4)) + 16) + (t & 15);
}

enum Bar {
  B_BC, B_CB, E_CBREAD, B_XG, E_XG, B_H, B_DSL, E_X16, B_GX1, B_GX2, E_GX1, B_DHS, B_CH, E_M16, E_CHR, E_RING, E_DS0, E_DS1, B_G4, B_DBD, E_RA, E_WSUM, B_FIN,
  NBARS
};

struct Small {
  float a2[kQ];    // in-chunk cumulative decay of the current head, log2 units: A log2(e) cumsum(dt)
  float dtv[kQ];   // step sizes of the current head
  float dtu[kQ];   // column decay factors of E1 (per 16-column block)
  float cdt[kQ];   // cumulative step sizes of the head about to run (E5 reads them)
  float red[64];
  uint64_t bars[NBARS];
  uint32_t tmem_base;
  int unit;
  int has_next;          // the chunk after this one belongs to the same sequence
  float *dst0;           // where head g*hpg's dH goes: ring slot or initial-state gradient (or null)
  int64_t dst_stride;    // elements between consecutive heads' dH tiles
  float ad[2];           // A and D of the head about to start
  volatile int abort;  // set when a bounded wait ran out: later waits give up at once
};
static_assert(sizeof(Small) <= SMALL_BYTES, "small region");

// exchange scratch between the two column halves of a row, and the
// per-quadrant partial column sums (strict lower part of M o Gx)
struct XBuf {
  float v[5][4][kQ];     // per column quarter: row sum of M o Gx o dt, x.D1, inter, g.x, x.Y
};
static_assert(sizeof(XBuf) <= 16384, "scratch");

struct Params {
  Shape s;
  const __nv_bfloat16 *x, *dout;
  const float *dt, *A, *D, *states;
  const int32_t *seq_idx;
  float *dx, *ddt, *dB, *dC, *dinit;
  float *ring;
  int ring_depth;
  int *flags, *ticket, *err;
  float *dA_part, *dD_part;
  float *dA, *dD;         // atomic variant: accumulated directly
  uint32_t spin_limit;
  int atomic;
  int64_t silent_chunk;   // fault injection: this chunk's units never publish (-1: none)
};

// ------------------------------------------------------------- helpers --
__device__ __forceinline__ void ep_sync() { umma::named_bar(1, kEpiThreads); }
__device__ __forceinline__ void scan_sync() { umma::named_bar(2, 128); }  // warps 8-11 (column quarter 2)


__device__ __forceinline__ void st_row16_bf16(uint8_t *panel, int r, int c0, const float (&v)[16]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
    const int chunk = ((c0 >> 3) + j) ^ (r & 7);
    *reinterpret_cast<uint4 *>(panel + r * 128 + chunk * 16) = u;
  }
}

__device__ __forceinline__ void f16x8_to_f32(uint4 u, float *f) {
  const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __half22float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}


__device__ __forceinline__ void st_row8_f16(uint8_t *panel, int r, int c0, const float (&v)[8]) {
  uint4 u;
  __half2 *h = reinterpret_cast<__half2 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
  const int chunk = (c0 >> 3) ^ (r & 7);
  *reinterpret_cast<uint4 *>(panel + r * 128 + chunk * 16) = u;
}

__device__ __forceinline__ void ld8_f16(const uint8_t *panel, int r, int c0, float (&v)[8]) {
  f16x8_to_f32(*reinterpret_cast<const uint4 *>(panel + r * 128 + (((c0 >> 3) ^ (r & 7)) << 4)), v);
}
__device__ __forceinline__ void st8_bf16(uint8_t *panel, int r, int c0, const float (&v)[8]) {
  uint4 u;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4 *>(panel + r * 128 + (((c0 >> 3) ^ (r & 7)) << 4)) = u;
}

// exponent k with max * 2^k in [2^14, 2^15) (0 for max == 0 or not finite);
// read from the float's exponent field (max is normal: the fp16 path only
// sees bf16 data and products of it)
__device__ __forceinline__ int fp16_scale_exp(float mx) {
  if (!(mx > 0.f) || !(mx < 3.0e38f)) return 0;
  const int e = int((__float_as_uint(mx) >> 23) & 0xffu) - 126;   // mx in [2^(e-1), 2^e)
  const int k = 15 - e;
  return max(-120, min(120, k));
}
// 2^k for |k| <= 126, exact (callers keep k within +-120)
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float(uint32_t(127 + k) << 23); }

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

constexpr long long kWaitCycles = 2000000000LL;  // about one second

// Bounded mbarrier wait: gives up after kWaitCycles (or at once once any
// wait of this CTA gave up), recording error bit 2.  The kernel then runs to
// its end with invalid results instead of hanging.
__device__ __forceinline__ void wait_bar_impl(uint64_t *b, uint32_t parity, int *err, volatile int *abort) {
  if (*abort) return;
  if (umma::mbar_try_wait(b, parity)) return;
  const long long t0 = clock64();
  // sleep in the barrier (woken when the phase completes) rather than spin
  while (!umma::mbar_try_wait_sleep(b, parity, 20000u)) {
    if (*abort) return;
    if (clock64() - t0 > kWaitCycles) {
      *abort = 1;
      atomicOr(err, 2);
      return;
    }
  }
}
// single-lane roles (TMA, MMA issuer)
#define wait_bar(b, parity, err) wait_bar_impl((b), (parity), (err), &sm->abort)
// full epilogue warps: lane 0 waits, the warp reconverges before any
// warp-collective TMEM access
#define ewait(b, parity, err)                                  \
  do {                                                         \
    if (lane == 0) wait_bar_impl((b), (parity), (err), &sm->abort); \
    __syncwarp();                                              \
  } while (0)

// Maxima of two values over all epilogue threads in one round.
__device__ __forceinline__ void ep_max2(float &a, float &b, Small *sm) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  const int warp = threadIdx.x >> 5;
  // red[0 .. 2 kEpiWarps) is free here: every earlier reader passed a barrier since
  if ((threadIdx.x & 31) == 0) {
    sm->red[warp] = a;
    sm->red[kEpiWarps + warp] = b;
  }
  ep_sync();
  a = 0.f;
  b = 0.f;
#pragma unroll
  for (int w = 0; w < kEpiWarps; ++w) {
    a = fmaxf(a, sm->red[w]);
    b = fmaxf(b, sm->red[kEpiWarps + w]);
  }
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ============================================================== kernel ===
// kDxAdd: add dx into the existing dx (the state halves of a 256-wide state:
// two adds onto zero per element) instead of storing it.  kSliceShift: the
// heads of a group are split into 2^kSliceShift slices, one unit each (unit
// group g covers heads [g * hpg, (g + 1) * hpg) and reads the B, C columns of
// group g >> kSliceShift; its dB, dC are that slice's partial sums).
template <bool kDxAdd, int kSliceShift>
__global__ void __launch_bounds__(kThreads, 1)
    fused_bwd_kernel(const Params p, const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_g,
                     const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_c,
                     const __grid_constant__ CUtensorMap tm_dx) {
  // The 128-byte swizzled tiles need a 1 KB aligned base, which is where the
  // dynamic shared memory of this kernel starts (no static shared memory).
  // Checked rather than assumed: a misaligned base reports and exits.  With a
  // fixed base every shared-memory address is a constant offset, so no base
  // pointer has to stay in a register.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *const sm_base = smem_raw;
  if (umma::smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, 4);
    return;
  }
  Small *sm = reinterpret_cast<Small *>(sm_base + OFF_SMALL);
  uint64_t *bars = sm->bars;
  const Shape &s = p.s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == kMmaWarp) {
    umma::tmem_alloc(&sm->tmem_base, 512);
    umma::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < NBARS; ++i) umma::mbar_init(&bars[i], (i == E_CHR || i == E_GX1 || i == E_RING || i == E_DS0 || i == E_DS1) ? kEpiWarps : 1);  // per-warp arrivals
    umma::fence_mbar_init();
    sm->unit = atomicAdd(p.ticket, 1);
    sm->abort = 0;
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = sm->tmem_base;

  // unit from the ticket: chunks in descending order, then batch row, then group
  // (32-bit: the supported shapes keep units and token rows below 2^30; every
  // index that can grow past that is formed with the 64-bit shape fields)
  const int unit = sm->unit;
  const int per_row = int(s.b * s.G);
  const int c = int(s.nc) - 1 - unit / per_row;
  const int bi = (unit % per_row) / int(s.G);
  const int g = unit % int(s.G);
  const int t0 = c * kQ;
  const int row0 = bi * int(s.T) + t0;  // first global token row of the chunk
  const int hpg = int(s.hpg);

  if (warp == kTmaWarp) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      umma::tma_prefetch_desc(&tm_x);
      umma::tma_prefetch_desc(&tm_g);
      umma::tma_prefetch_desc(&tm_b);
      umma::tma_prefetch_desc(&tm_c);
      umma::mbar_expect_tx(&bars[B_BC], 65536);
      for (int j = 0; j < 2; ++j) {
        umma::tma_load_2d(sm_base + OFF_B + j * 16384, &tm_b, int((g >> kSliceShift) * kN + j * 64), int(row0),
                          &bars[B_BC]);
        // C in the paired row order: one 16-row box per token group
        for (int tg = 0; tg < 8; ++tg)
          umma::tma_load_2d(sm_base + OFF_C + j * 16384 + row_of_tok(16 * tg) * 128, &tm_c,
                            int((g >> kSliceShift) * kN + j * 64), int(row0 + 16 * tg), &bars[B_BC]);
      }
      const bool has_next = (c + 1 < s.nc) && !is_seq_start(p.seq_idx, bi, s.T, t0 + kQ);
      // this thread also publishes each head's state gradient to the chunk before
      const bool publish = !is_seq_start(p.seq_idx, bi, s.T, t0) && c != p.silent_chunk;
      const float *states = p.states + (bi * s.nc + c) * s.H * kP * kN;
      int n_h = 0, n_xg = 0, n_ds = 0;   // copies issued per barrier (drained before exit)
      for (int k = 0; k < hpg; ++k) {
        const int64_t h = g * hpg + k;
        const uint32_t par = uint32_t(k & 1);
        if (k > 0) {
          // every epilogue warp stored its part of head k-1's dH (warp barrier + arrive), and
          // the staging buffer is free again
          wait_bar(&bars[E_RING], uint32_t((k - 1) & 1), p.err);
          if (sm->abort) break;
          if (publish) st_release_gpu(p.flags + ((bi * s.nc + c) * s.H + h - 1), 1);
          // the products that read head k-1's dS from the H tiles (Y, dB) are done
          wait_bar(&bars[B_DBD], uint32_t((k - 1) & 1), p.err);
          if (sm->abort) break;
        }
        // the state tile entering the chunk, saved by the forward as the bf16 hi | lo pair of
        // [n][p] tiles in the 128-byte swizzled operand layout: one copy straight into place
        umma::mbar_expect_tx(&bars[B_H], kP * kN * 4);
        umma::bulk_load(sm_base + OFF_HD, states + h * kP * kN, kP * kN * 4, &bars[B_H]);
        ++n_h;
        if (k + 1 < hpg) umma::prefetch_l2(states + (h + 1) * kP * kN, kP * kN * 4);
        // x and g of this head once the previous head's are consumed
        if (k > 0) {
          wait_bar(&bars[E_XG], par ^ 1u, p.err);
          if (sm->abort) break;
        }
        umma::mbar_expect_tx(&bars[B_XG], 32768);
        umma::tma_load_2d(sm_base + OFF_XG, &tm_x, int(h * kP), int(row0), &bars[B_XG]);
        for (int tg = 0; tg < 8; ++tg)   // g in the paired row order
          umma::tma_load_2d(sm_base + OFF_XG + 16384 + row_of_tok(16 * tg) * 128, &tm_g, int(h * kP),
                            int(row0 + 16 * tg), &bars[B_XG]);
        ++n_xg;
        if (k + 1 < hpg) {
          umma::tma_prefetch_2d(&tm_x, int((h + 1) * kP), int(row0));
          for (int tg = 0; tg < 8; ++tg) umma::tma_prefetch_2d(&tm_g, int((h + 1) * kP), int(row0 + 16 * tg));
        }
        if (has_next) {
          // dS = dH of the chunk after, once its unit has published it (the staging
          // buffer was freed by the E_RING wait above)
          const int *flag = p.flags + ((bi * s.nc + c + 1) * s.H + h);
          uint32_t it = 0;
          while (!sm->abort && ld_acquire_gpu(flag) == 0) {
            if (++it > p.spin_limit) {
              atomicOr(p.err, 1);
              sm->abort = 1;   // every later wait of this CTA gives up at once
              break;
            }
            __nanosleep(64);
          }
          if (sm->abort) break;
          umma::fence_proxy_async_global();   // the bulk copy reads what the acquire made visible
          umma::mbar_expect_tx(&bars[B_DSL], kP * kN * 4);
          umma::bulk_load(sm_base + OFF_STG, p.ring + ((((c + 1) % p.ring_depth) * s.b + bi) * s.H + h) * (kP * kN),
                          kP * kN * 4, &bars[B_DSL]);
          ++n_ds;
        }
      }
      if (!sm->abort) {
        wait_bar(&bars[E_RING], uint32_t((hpg - 1) & 1), p.err);
        if (!sm->abort && publish) st_release_gpu(p.flags + ((bi * s.nc + c) * s.H + g * hpg + hpg - 1), 1);
      }
      // every issued copy has landed before the CTA may exit (bounded; after a
      // give-up nobody else waited for them)
      auto drain = [&](uint64_t *b, int n) {
        if (n == 0) return;
        const long long w0 = clock64();
        while (!umma::mbar_try_wait(b, uint32_t((n - 1) & 1)) && clock64() - w0 < kWaitCycles) {
        }
      };
      drain(&bars[B_H], n_h);
      drain(&bars[B_XG], n_xg);
      drain(&bars[B_DSL], n_ds);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      const uint32_t aB = umma::smem_u32(sm_base + OFF_B), aC = umma::smem_u32(sm_base + OFF_C);
      const uint32_t aHh = umma::smem_u32(sm_base + OFF_HD), aHl = aHh + 16384;
      const uint32_t aGh = umma::smem_u32(sm_base + OFF_GW), aGl = aGh + 16384;
      const uint32_t aM16 = umma::smem_u32(sm_base + OFF_M16);
      constexpr uint32_t id_kk128 = umma::idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t id_km64 = umma::idesc_bf16_f32(128, 64, 0, 1);
      constexpr uint32_t id_mm64 = umma::idesc_bf16_f32(128, 64, 1, 1);
      constexpr uint32_t id_km128 = umma::idesc_bf16_f32(128, 128, 0, 1);
      constexpr uint32_t id_mm128 = umma::idesc_bf16_f32(128, 128, 1, 1);
      // fp16 A/B (formats 0): D1 MN-major/MN-major N = 64
      constexpr uint32_t id_kk64 = umma::idesc_bf16_f32(128, 64, 0, 0);
      constexpr uint32_t id_f16_mm64 = (1u << 4) | (1u << 15) | (1u << 16) | ((64u >> 3) << 17) | ((128u >> 4) << 24);
      // Descriptors of a K step kk: the start-address field (address >> 4, 14 bits) of the
      // operand's base descriptor plus the step's byte offset >> 4.  Every operand lies below
      // 256 KB, so the field never wraps and the base descriptor is loop-invariant.
      auto kdesc = [](uint32_t base, uint32_t panel_bytes, int kk) {  // K-major operand, K step kk
        return umma::smem_desc_sw128(base, 16, 1024) +
               uint64_t((uint32_t(kk / 64) * panel_bytes + uint32_t(kk % 64) * 2) >> 4);
      };
      auto mdesc = [](uint32_t base, uint32_t panel_bytes, int kk) {  // MN-major operand, K step kk
        return umma::smem_desc_sw128(base, panel_bytes, 1024) + uint64_t((uint32_t(kk) * 128) >> 4);
      };
      wait_bar(&bars[B_BC], 0, p.err);
      umma::fence_after_sync();
      // CB = C B^T  (M = t, N = s, K = n)
      for (int kk = 0; kk < kN; kk += 16)
        umma::mma_bf16(tmem + T_RA, kdesc(aC, 16384, kk), kdesc(aB, 16384, kk), id_kk128, kk > 0);
      umma::mma_commit(&bars[B_CB]);
      wait_bar(&bars[E_CBREAD], 0, p.err);
      for (int k = 0; k < hpg; ++k) {
        const int st = k & 1;
        const uint32_t par = uint32_t(k & 1);
        const uint32_t aX = umma::smem_u32(sm_base + OFF_XG), aG = aX + 16384;
        if (k > 0) wait_bar(&bars[E_RA], par ^ 1u, p.err);
        wait_bar(&bars[B_XG], par, p.err);   // x, g landed (bf16)
        umma::fence_after_sync();
        // Gx = g x^T (M = t, N = s, K = p), bf16 operands, in two column halves,
        // the right one (s >= 64: only the later tokens' rows) first, so that the
        // epilogue can hand it back early
        for (int kk = 0; kk < kP; kk += 16)
          umma::mma_bf16(tmem + T_RA + 64, kdesc(aG, 16384, kk), kdesc(aX + 8192, 16384, kk), id_kk64, kk > 0);
        umma::mma_commit(&bars[B_GX1]);
        for (int kk = 0; kk < kP; kk += 16)
          umma::mma_bf16(tmem + T_RA, kdesc(aG, 16384, kk), kdesc(aX, 16384, kk), id_kk64, kk > 0);
        umma::mma_commit(&bars[B_GX2]);
        wait_bar(&bars[E_X16], par, p.err);  // G~ in smem
        wait_bar(&bars[B_H], par, p.err);    // H (hi, lo) landed
        umma::fence_after_sync();
        // dC += G~ H^T  (M = t, N = n, K = p): hi*hi + hi*lo + lo*hi; runs while the epilogue reads g x^T
        for (int part = 0; part < 3; ++part) {
          const uint32_t aA = part == 2 ? aGl : aGh, aBb = part == 1 ? aHl : aHh;
          for (int kk = 0; kk < kP; kk += 16)
            umma::mma_bf16(tmem + T_DC, kdesc(aA, 16384, kk), kdesc(aBb, 16384, kk), id_kk128,
                           (k > 0) || (part > 0) || (kk > 0));
        }
        wait_bar(&bars[E_GX1], par, p.err);  // right half of g x^T read: dHscan^T goes there
        umma::fence_after_sync();
        // dHscan^T = C^T (G~_hi + G~_lo)  (M = n, N = p, K = t)
        for (int part = 0; part < 2; ++part)
          for (int kk = 0; kk < kQ; kk += 16)
            umma::mma_bf16(tmem + T_DH, mdesc(aC, 16384, kk), mdesc(part ? aGl : aGh, 16384, kk), id_mm64,
                           (part > 0) || (kk > 0));
        umma::mma_commit(&bars[B_DHS]);
        wait_bar(&bars[E_M16], par, p.err);  // left half read too; M16 in smem
        umma::fence_after_sync();
        // CH = C (H_hi + H_lo)  (M = t, N = p, K = n)
        for (int part = 0; part < 2; ++part)
          for (int kk = 0; kk < kN; kk += 16)
            umma::mma_bf16(tmem + T_CH, kdesc(aC, 16384, kk), mdesc(part ? aHl : aHh, 16384, kk), id_km64,
                           (part > 0) || (kk > 0));
        umma::mma_commit(&bars[B_CH]);
        wait_bar(&bars[E_DS0 + st], uint32_t((k >> 1) & 1), p.err);  // dHscan read; dS and w o x in smem
        umma::fence_after_sync();
        // Y = B (dS_hi + dS_lo)^T  (M = t, N = p, K = n); dS stored [n][p]
        for (int part = 0; part < 2; ++part)
          for (int kk = 0; kk < kN; kk += 16)
            umma::mma_bf16(tmem + T_Y, kdesc(aB, 16384, kk), mdesc(part ? aHl : aHh, 16384, kk), id_km64,
                           (part > 0) || (kk > 0));
        wait_bar(&bars[E_CHR], par, p.err);  // CH read and g in fp16: D1 into CH's columns
        umma::fence_after_sync();
        // D1 = M^T g  (fp16 scaled operands; M = s, N = p, K = t)
        for (int kk = 0; kk < kQ; kk += 16)
          umma::mma_bf16(tmem + T_D1, mdesc(aM16, 16384, kk), mdesc(aG, 16384, kk), id_f16_mm64, kk > 0);
        umma::mma_commit(&bars[B_G4]);
        // dB += (w o x) (dS_hi + dS_lo)  (M = t, N = n, K = p): read only at the unit's end, so
        // issued after the products the epilogue waits for (its own barrier frees the H tiles)
        for (int part = 0; part < 2; ++part)
          for (int kk = 0; kk < kP; kk += 16)
            umma::mma_bf16(tmem + T_DB, kdesc(aGh, 16384, kk), kdesc(part ? aHl : aHh, 16384, kk), id_kk128,
                           (k > 0) || (part > 0) || (kk > 0));
        umma::mma_commit(&bars[B_DBD]);
      }
      wait_bar(&bars[E_WSUM], 0, p.err);
      umma::fence_after_sync();
      const uint32_t aWh = umma::smem_u32(sm_base + OFF_WHI), aWl = umma::smem_u32(sm_base + OFF_WLO);
      for (int part = 0; part < 2; ++part) {
        const uint32_t aW = part ? aWl : aWh;
        // dC += W B  (M = t, N = n, K = s)
        for (int kk = 0; kk < kQ; kk += 16)
          umma::mma_bf16(tmem + T_DC, kdesc(aW, 16384, kk), mdesc(aB, 16384, kk), id_km128, 1);
        // dB += W^T C  (M = s, N = n, K = t)
        for (int kk = 0; kk < kQ; kk += 16)
          umma::mma_bf16(tmem + T_DB, mdesc(aW, 16384, kk), mdesc(aC, 16384, kk), id_mm128, 1);
      }
      umma::mma_commit(&bars[B_FIN]);
    }
  } else if (warp < kEpiWarps) {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3, cq = warp >> 2;            // TMEM lane quadrant, column quarter
    const int r = 32 * q + lane;                       // row (token / state index) of this thread
    const uint32_t lane_off = uint32_t(32 * q) << 16;  // TMEM lane field of this warp's quadrant
    const float *dtg = p.dt + row0 * s.H;
    XBuf *xb = reinterpret_cast<XBuf *>(sm_base + OFF_XBUF);
    constexpr float kLog2e = 1.4426950408889634f;

    // The intra-chunk phase E1 works on blocks of 16 tokens x 16 columns of
    // the causal triangle: in quadrant q, those of token group 7-q (column
    // blocks 0..7-q) and of group q (0..q), nine per quadrant.  Warp cq takes
    // R: block 4+cq of group 7-q (the right half, read first) if cq < 4-q;
    // L: block cq of group 7-q; A: block (cq+q) mod 4 of group q if that is
    // at most q.  Two threads share a row (lanes of the 16-lane TMEM form):
    // threads 0-15 take its columns 0-7 of the block, threads 16-31 8-15.
    const bool hasR = cq < 4 - q;
    const int blkA = (cq + q) & 3;
    const bool hasA = blkA <= q;
    const int j16 = lane & 15, hsel = lane >> 4;
    const uint32_t lanesA = uint32_t(32 * q) << 16, lanesB = uint32_t(32 * q + 16) << 16;
    const int tokA = 16 * q + j16, tokB = 16 * (7 - q) + j16;   // this thread's tokens in groups q, 7-q
    // C B^T of those blocks into registers, pre-scaled by the power of two
    // that brings M = CB o L into the fp16 range
    float cbR[8], cbL[8], cbA[8];
    ewait(&bars[B_CB], 0, p.err);
    umma::fence_after_sync();
    float cbmax = 0.f;
    umma::tmem_ld8_h16(tmem + lanesB + T_RA + 16 * cq, cbL);
    if (hasR) umma::tmem_ld8_h16(tmem + lanesB + T_RA + 16 * (4 + cq), cbR);
    if (hasA) umma::tmem_ld8_h16(tmem + lanesA + T_RA + 16 * blkA, cbA);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (!hasR) cbR[i] = 0.f;
      if (!hasA) cbA[i] = 0.f;
      cbmax = fmaxf(cbmax, fmaxf(fabsf(cbL[i]), fmaxf(fabsf(cbR[i]), fabsf(cbA[i]))));
    }
    {
      float z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j) umma::tmem_st16(tmem + lane_off + T_WS + 64 * j + 16 * cq, z);
      umma::tmem_wait_st();
    }
    umma::fence_before_sync();
    {
      float dummy = 0.f;
      ep_max2(cbmax, dummy, sm);
    }
    if (tid == 0) umma::mbar_arrive(&bars[E_CBREAD]);
    const int kM = fp16_scale_exp(cbmax);
    const float sM = exp2i(kM), sMinv = exp2i(-kM);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      cbR[i] *= sM;
      cbL[i] *= sM;
      cbA[i] *= sM;
    }

    if (tid == 0) {
      sm->has_next = (c + 1 < s.nc) && !is_seq_start(p.seq_idx, bi, s.T, t0 + kQ);
      const int64_t h0 = g * hpg;
      if (is_seq_start(p.seq_idx, bi, s.T, t0)) {
        sm->dst0 = p.dinit ? p.dinit + ((seq_of(p.seq_idx, bi, s.T, t0) * s.H + h0) * kP) * kN : nullptr;
      } else {
        sm->dst0 = p.ring + (((c % p.ring_depth) * s.b + bi) * s.H + h0) * (kP * kN);
      }
      sm->dst_stride = kP * kN;
      sm->ad[0] = __ldcg(p.A + g * hpg);
      sm->ad[1] = __ldcg(p.D + g * hpg);
    }
    ep_sync();
    const int n = r;  // for [p][n] tiles (states, state gradients): this thread's state index
    const int tr = tok_of_row(r);   // token of row r of the paired tiles (g, G~, C B^T, C H, dC lanes)

    // (scalar loads and stores below bypass L1: its few KB beside the shared
    // memory carve-out are left to the register spill slots)
    // Step-size scan of a head (fixed tree: warp shuffles, then the four row
    // quadrants in order), run by the column-quarter-2 warps one head ahead:
    // Acs in log2 units into a2, dt into dtv, the cumulative step into cdt,
    // the chunk's total into red[36 + head parity].
    auto scan_head = [&](int kk, float dtr_in, float Ak) {
      float cum = dtr_in;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, cum, o);
        if (lane >= o) cum += v;
      }
      if (lane == 31) sm->red[32 + q] = cum;
      scan_sync();
      float pre = 0.f;
      for (int w = 0; w < q; ++w) pre += sm->red[32 + w];
      cum += pre;
      sm->a2[r] = cum * (Ak * kLog2e);
      sm->dtv[r] = dtr_in;
      sm->cdt[r] = cum;
      if (r == kQ - 1) sm->red[36 + (kk & 1)] = cum;
    };
    float dt_next = (cq == 2) ? __ldcg(dtg + int64_t(r) * s.H + g * hpg) : 0.f;  // step size of the first head
    if (cq == 2) scan_head(0, dt_next, sm->ad[0]);
    for (int k = 0; k < hpg; ++k) {
      const int st = k & 1;
      const uint32_t par = uint32_t(k & 1);
      const int h = g * hpg + k;
      uint8_t *sX = sm_base + OFF_XG;
      uint8_t *sG = sX + 16384;
      const float Ah = sm->ad[0], Dh = sm->ad[1];

      // ---- P0 (the step-size scan of this head ran at the end of the previous one)
      ewait(&bars[B_XG], par, p.err);
      ewait(&bars[B_H], par, p.err);
      ep_sync();
      // per-row values are re-read from shared memory in each phase that uses
      // them rather than kept in registers across phases (fewer spills)
      const float eacs = umma::ex2_approx(sm->a2[tr]);   // exp(Acs) of token tr (row r of g, G~)
      // Column factors of the decay below the diagonal blocks: within each
      // 16-column block, exp(Acs_ref - Acs_s) with ref the block's last
      // column, so that exp(Acs_r - Acs_s) = exp(Acs_r - Acs_ref) exp(Acs_ref - Acs_s)
      // with both factors at most one (kept in dtu until E3 reuses it).
      if (cq == 0) sm->dtu[r] = umma::ex2_approx(sm->a2[r | 15] - sm->a2[r]);

      // G~ = exp(Acs) o g as a bf16 hi + lo pair; max |g| for the fp16 scaling of g; g . x
      // (row r of g and G~ holds token tr; x is in natural order)
      float gmax = 0.f, gx = 0.f;
#pragma unroll
      for (int c8 = 0; c8 < 2; ++c8) {
        const int c0 = 16 * cq + 8 * c8;
        float gv[8], xv[8], t[8];
        ld8_bf16(sG, r, c0, gv);
        ld8_bf16(sX, tr, c0, xv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          t[i] = eacs * gv[i];
          gmax = fmaxf(gmax, fabsf(gv[i]));
          gx = fmaf(gv[i], xv[i], gx);
        }
        st8_bf16_hilo(sm_base + OFF_GW, sm_base + OFF_GW + 16384, r, c0, t);
      }
      // per-warp maxima of |g|; read after the barrier that ends E1
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
      if (lane == 0) sm->red[warp] = gmax;
      umma::fence_proxy_async_smem();
      if (tid == 128) umma::tma_store_wait_read();  // dx staging (the M16 buffer) has been read out
      ep_sync();
      if (tid == 0) umma::mbar_arrive(&bars[E_X16]);

      // ---- E1: intra-chunk matrices from g x^T (TMEM, bf16 products) and C B^T (registers).
      // The decay gradient needs the row and the column sums of M o Gx o dt;
      // both are taken from the same fp16-rounded M that the dx product
      // uses (the column sums come out of that product in E4), so their
      // difference keeps its cancellation exact up to fp32 accumulation.
      // The right column half of g x^T comes first (block R); every warp then
      // hands it back so that dHscan^T can be computed there while the left
      // half (blocks L and A) is processed.
      float rowpA = 0.f, rowpB = 0.f;   // sum_s M16_ts Gx_ts dt_s over this thread's columns, times sM
      const float a2A = sm->a2[tokA], a2B = sm->a2[tokB];
      // one 16 x 16 block: token group 7-q (grp 1) or q (grp 0), column block cb
      auto e1_block = [&](int grp, int cb, const float(&cbv)[8], float &rowp) {
        const int t = grp ? tokB : tokA;
        const float a2t = grp ? a2B : a2A;
        const uint32_t lanes = grp ? lanesB : lanesA;
        const int s0 = 16 * cb + 8 * hsel;             // first of this thread's 8 columns
        const bool diag = cb == (grp ? 7 - q : q);     // the block holds the group's diagonal (warp-uniform)
        const float er = diag ? 0.f : umma::ex2_approx(a2t - sm->a2[16 * cb + 15]);
        float gxv[8], ws[8];
        uint32_t m16[4];
        umma::tmem_ld8x2_h16(tmem + lanes + T_RA + 16 * cb, tmem + lanes + T_WS + 16 * cb, gxv, ws);
#pragma unroll
        for (int e4 = 0; e4 < 2; ++e4) {
          const int cb4 = s0 + 4 * e4;   // first of these 4 columns
          const float4 duv = *reinterpret_cast<const float4 *>(&sm->dtv[cb4]);
          const float dus[4] = {duv.x, duv.y, duv.z, duv.w};
          float Lv[4];
          if (diag) {
            const float4 a2v = *reinterpret_cast<const float4 *>(&sm->a2[cb4]);
            const float a2s[4] = {a2v.x, a2v.y, a2v.z, a2v.w};
#pragma unroll
            for (int e1 = 0; e1 < 4; ++e1) Lv[e1] = (cb4 + e1 <= t) ? umma::ex2_approx(a2t - a2s[e1]) : 0.f;
          } else {
            const float4 ecv = *reinterpret_cast<const float4 *>(&sm->dtu[cb4]);
            Lv[0] = er * ecv.x;
            Lv[1] = er * ecv.y;
            Lv[2] = er * ecv.z;
            Lv[3] = er * ecv.w;
          }
          float mv[4], gd[4];
#pragma unroll
          for (int e1 = 0; e1 < 4; ++e1) {
            const int e = 4 * e4 + e1;
            gd[e1] = gxv[e] * dus[e1];       // Gx dt (true units)
            ws[e] = fmaf(Lv[e1], gd[e1], ws[e]);
            mv[e1] = cbv[e] * Lv[e1];
          }
          const __half2 h01 = __floats2half2_rn(mv[0], mv[1]), h23 = __floats2half2_rn(mv[2], mv[3]);
          const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
          rowp = fmaf(f01.x, gd[0], rowp);
          rowp = fmaf(f01.y, gd[1], rowp);
          rowp = fmaf(f23.x, gd[2], rowp);
          rowp = fmaf(f23.y, gd[3], rowp);
          m16[2 * e4] = *reinterpret_cast<const uint32_t *>(&h01);
          m16[2 * e4 + 1] = *reinterpret_cast<const uint32_t *>(&h23);
        }
        umma::tmem_st8_h16(tmem + lanes + T_WS + 16 * cb, ws);
        const int row = 32 * q + 16 * grp + j16;   // row of the M16 tile (paired order)
        *reinterpret_cast<uint4 *>(sm_base + OFF_M16 + (s0 >> 6) * 16384 + row * 128 +
                                   ((((s0 & 63) >> 3) ^ (row & 7)) << 4)) = make_uint4(m16[0], m16[1], m16[2], m16[3]);
      };
      ewait(&bars[B_GX1], par, p.err);   // right half of g x^T
      umma::fence_after_sync();
      if (hasR) e1_block(1, 4 + cq, cbR, rowpB);
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&bars[E_GX1]);
      ewait(&bars[B_GX2], par, p.err);  // left half
      umma::fence_after_sync();
      e1_block(1, cq, cbL, rowpB);
      if (hasA) e1_block(0, blkA, cbA, rowpA);
      // zeros in the blocks of M16 above the diagonal (group q: blocks q+1..7,
      // group 7-q: 8-q..7; seven per quadrant, spread over its warps)
      for (int z = cq; z < 7; z += 4) {
        const int grp = z < 7 - q ? 0 : 1;
        const int cb = grp ? 8 - q + (z - (7 - q)) : q + 1 + z;
        const int s0 = 16 * cb + 8 * hsel;
        const int row = 32 * q + 16 * grp + j16;
        *reinterpret_cast<uint4 *>(sm_base + OFF_M16 + (s0 >> 6) * 16384 + row * 128 +
                                   ((((s0 & 63) >> 3) ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
      }
      // a row's two column halves summed in a fixed order (left half first): threads 0-15
      // hold the total of token tokA, threads 16-31 that of tokB
      float rowp_tok;
      {
        const float oA = __shfl_xor_sync(0xffffffffu, rowpA, 16), oB = __shfl_xor_sync(0xffffffffu, rowpB, 16);
        rowp_tok = hsel ? oB + rowpB : rowpA + oA;
      }
      umma::tmem_wait_st();
      umma::fence_before_sync();
      umma::fence_proxy_async_smem();
      ep_sync();
      if (tid == 0) umma::mbar_arrive(&bars[E_M16]);

      // ---- E3: chain step (dH to the chunk before), then E2: carried-in state term
      ewait(&bars[B_DHS], par, p.err);   // dHscan^T in TMEM; dC and dHscan have read G~ (GW)
      umma::fence_after_sync();
      const float a2E3 = sm->a2[kQ - 1], dtr = sm->dtv[r];
      const float wr3 = umma::ex2_approx(a2E3 - sm->a2[r]) * dtr;   // w = exp(E - Acs_r) dt_r
      const float eE = umma::ex2_approx(a2E3);                        // exp(E)
      // GW is idle from here to the next head: exchange scratch (lo half) and w o x (hi half)
      xb->v[0][cq][hsel ? tokB : tokA] = rowp_tok;
      xb->v[3][cq][tr] = gx;
      {
#pragma unroll
        for (int c8 = 0; c8 < 2; ++c8) {
          float xv[8];
          ld8_bf16(sX, r, 16 * cq + 8 * c8, xv);
#pragma unroll
          for (int i = 0; i < 8; ++i) xv[i] *= wr3;
          st8_bf16(sm_base + OFF_GW, r, 16 * cq + 8 * c8, xv);
        }
      }
      const bool has_next = sm->has_next != 0;
      if (has_next) {
        ewait(&bars[B_DSL], par, p.err);   // dS in the staging buffer
        // The ring slot has been copied for the last time: its L2 lines are
        // dropped rather than written back to DRAM (the slot is next written
        // after this chunk's flag is published, which these threads precede).
        if (tid < kP * kN / 32 && !sm->abort)
          umma::discard_l2_line(p.ring + ((((c + 1) % p.ring_depth) * s.b + bi) * s.H + h) * (kP * kN) + 32 * tid);
      }
      float hdot = 0.f;
      float ds[16];   // this thread's dS values (state index n, 16 p values)
      {
        const float *src = reinterpret_cast<const float *>(sm_base + OFF_STG);
        float *dst = sm->dst0 ? sm->dst0 + k * sm->dst_stride : nullptr;
        if (has_next) {
#pragma unroll
          for (int i = 0; i < 16; ++i) ds[i] = src[(16 * cq + i) * kN + n];
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) ds[i] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int p0 = 16 * cq + 8 * u;
          float hh[8], hl[8], dh[8];
          // H = hi + lo (row n of the [n][p] tiles), read before dS overwrites the hi tile
          ld8_bf16(sm_base + OFF_HD, n, p0, hh);
          ld8_bf16(sm_base + OFF_HD + 16384, n, p0, hl);
          umma::tmem_ld8(tmem + lane_off + T_DH + p0, dh);  // lane = n, columns p
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            hdot = fmaf(hh[i] + hl[i], ds[8 * u + i], hdot);
            if (dst) __stcg(dst + (p0 + i) * kN + n, fmaf(eE, ds[8 * u + i], dh[i]));
          }
        }
      }
      // Per-warp hand-off of the chain step: the producer thread waits for
      // every warp before it releases the chunk's flag (the warp barrier
      // orders all lanes' ring stores before lane 0's arrival).
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&bars[E_RING]);
      // per-warp partials of <H, dS>, folded in fixed order in E5
      hdot = warp_sum(hdot);
      if (lane == 0) sm->red[40 + warp] = hdot;
      // atomic variant: every warp adds its own share of dA as soon as it has
      // it (exp(E) <H, dS> times the chunk's total step), in whatever order
      // the warps and CTAs get there
      if (p.atomic && lane == 0) atomicAdd(p.dA + h, eE * hdot * sm->red[36 + (k & 1)]);

      ewait(&bars[B_CH], par, p.err);   // C H done: both H tiles may now give way to dS
      umma::fence_after_sync();
      {
        float d8[8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
#pragma unroll
          for (int i = 0; i < 8; ++i) d8[i] = ds[8 * u + i];
          st8_bf16_hilo(sm_base + OFF_HD, sm_base + OFF_HD + 16384, n, 16 * cq + 8 * u, d8);  // [n][p] hi | lo
        }
      }
      umma::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&bars[E_DS0 + st]);   // Y and dB may start
      // g -> fp16 scaled by an exact power of two, in place (the dx product
      // pairs it with the fp16 M); g x^T has been computed from the bf16 g
      float gmw[kEpiWarps];
#pragma unroll
      for (int w = 0; w < kEpiWarps; ++w) gmw[w] = sm->red[w];
#pragma unroll
      for (int st2 = kEpiWarps / 2; st2 > 0; st2 >>= 1)
#pragma unroll
        for (int w = 0; w < st2; ++w) gmw[w] = fmaxf(gmw[w], gmw[w + st2]);
      const float gm = gmw[0];
      const int kg = fp16_scale_exp(gm);
      float inter_part = 0.f;
      {
        const float sg = exp2i(kg);
        float ch0[8], ch1[8], gv[8];
        umma::tmem_ld8x2(tmem + lane_off + T_CH + 16 * cq, tmem + lane_off + T_CH + 16 * cq + 8, ch0, ch1);
        ld8_bf16(sG, r, 16 * cq, gv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          inter_part = fmaf(gv[i], ch0[i], inter_part);
          gv[i] *= sg;
        }
        st_row8_f16(sG, r, 16 * cq, gv);
        ld8_bf16(sG, r, 16 * cq + 8, gv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          inter_part = fmaf(gv[i], ch1[i], inter_part);
          gv[i] *= sg;
        }
        st_row8_f16(sG, r, 16 * cq + 8, gv);
      }
      xb->v[2][cq][tr] = inter_part;   // (C H lane r and g row r: token tr)
      umma::fence_proxy_async_smem();   // g16 is read by the dx product issued after E_CHR
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) umma::mbar_arrive(&bars[E_CHR]);

      // ---- E4: dx and the row dot product x . Y
      if (cq == 2 && k + 1 < hpg) dt_next = __ldcg(dtg + int64_t(r) * s.H + h + 1);  // next head's step size
      float a_next = 0.f, d_next = 0.f;
      if (tid == 0 && k + 1 < hpg) {
        a_next = __ldcg(p.A + h + 1);
        d_next = __ldcg(p.D + h + 1);
      }
      ewait(&bars[B_G4], par, p.err);
      umma::fence_after_sync();
      const float unscale = exp2i(-kM) * exp2i(-kg);
      float sxy = 0.f, xd1 = 0.f;   // x . Y and x . D1 (raw units) of this row
      {
        // dx rows staged in the (now idle) M16 buffer, 128-byte swizzled fp32, then TMA-stored
        uint8_t *stage = sm_base + OFF_M16 + (cq >> 1) * 16384;
        const float dg = Dh * exp2i(-kg);
#pragma unroll
        for (int c8 = 0; c8 < 2; ++c8) {
          float d1[8], y[8], xv[8], gv[8];
          umma::tmem_ld8x2(tmem + lane_off + T_D1 + 16 * cq + 8 * c8, tmem + lane_off + T_Y + 16 * cq + 8 * c8, d1, y);
          ld8_bf16(sX, r, 16 * cq + 8 * c8, xv);
          ld8_f16(sG, row_of_tok(r), 16 * cq + 8 * c8, gv);   // g of token r (paired order)
#pragma unroll
          for (int i4 = 0; i4 < 2; ++i4) {
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = 4 * i4 + e;
              sxy = fmaf(xv[i], y[i], sxy);
              xd1 = fmaf(xv[i], d1[i], xd1);
              o[e] = fmaf(dtr, d1[i] * unscale, fmaf(wr3, y[i], dg * gv[i]));
            }
            const int chunk = (4 * (cq & 1) + 2 * c8 + i4) ^ (r & 7);
            *reinterpret_cast<float4 *>(stage + r * 128 + chunk * 16) = make_float4(o[0], o[1], o[2], o[3]);
          }
        }
      }
      umma::fence_before_sync();
      umma::fence_proxy_async_smem();
      xb->v[4][cq][r] = sxy;
      xb->v[1][cq][r] = xd1;
      if (tid == 0 && k + 1 < hpg) {   // every thread read this head's A, D at the top of the head
        sm->ad[0] = a_next;
        sm->ad[1] = d_next;
      }
      ep_sync();
      // a thread of the upper column half issues the hand-offs: warps 0-3 go straight on to E5
      if (tid == 128) {
        umma::mbar_arrive(&bars[E_RA]);
        umma::mbar_arrive(&bars[E_XG]);
        if (kDxAdd) {
          umma::tma_reduce_add_2d(&tm_dx, sm_base + OFF_M16, int(h * kP), int(row0));
          umma::tma_reduce_add_2d(&tm_dx, sm_base + OFF_M16 + 16384, int(h * kP + 32), int(row0));
        } else {
          umma::tma_store_2d(&tm_dx, sm_base + OFF_M16, int(h * kP), int(row0));
          umma::tma_store_2d(&tm_dx, sm_base + OFF_M16 + 16384, int(h * kP + 32), int(row0));
        }
        umma::tma_store_commit();
      }

      // ---- E5: decay gradient, reverse cumsum, ddt, dA/dD partials
      // Every column quarter forms the same per-row values (from shared
      // memory); quarter 0 runs the suffix scan while quarter 1 runs the row
      // sums, in parallel, then quarter 0 finishes the rows.
      {
        const float a2r5 = sm->a2[r], a2E5 = sm->a2[kQ - 1], dt5 = sm->dtv[r];
        const float eEA5 = umma::ex2_approx(a2E5 - a2r5), wr5 = eEA5 * dt5;
        const float raw = exp2i(-kM) * exp2i(-kg);   // x . D1 in true units
        // inclusive row and column sums of M o Gx o dt: the diagonal cancels in their difference
        auto qsum = [&](int i) {   // the four column quarters, fixed order
          return (xb->v[i][0][r] + xb->v[i][1][r]) + (xb->v[i][2][r] + xb->v[i][3][r]);
        };
        const float rowp5 = qsum(0) * sMinv;
        const float dintra = qsum(1) * raw;   // sum_t M_tr Gx_tr (x . D1)
        const float inter = umma::ex2_approx(a2r5) * qsum(2);
        const float gx5 = qsum(3);
        const float sxy5 = qsum(4);
        const float cumdt5 = sm->cdt[r];
        const float colp = dt5 * dintra;
        const float u = wr5 * sxy5;
        const float dacs = rowp5 - colp + inter - u;
        float sfx = dacs;
        if (cq == 0) {
          // suffix sum over rows: fixed tree in the warp, fixed order across warps
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_down_sync(0xffffffffu, sfx, o);
            if (lane + o < 32) sfx += v;
          }
          if (lane == 0) sm->red[q] = sfx;
        } else if (cq == 1) {
          // warp totals of u, g.x and dacs * cumdt
          const float wu = warp_sum(u), wg = warp_sum(gx5), wc = warp_sum(dacs * cumdt5);
          if (lane == 0) {
            sm->red[4 + q] = wu;
            sm->red[8 + q] = wg;
            sm->red[12 + q] = wc;
            if (p.atomic) {   // this warp's share of dA and dD, added straight away
              atomicAdd(p.dA + h, fmaf(wu, sm->red[36 + (k & 1)], wc));
              atomicAdd(p.dD + h, wg);
            }
          }
        }
        ep_sync();
        // every E5 read of a2, dtv and cdt is done: the next head's scan may overwrite them
        if (cq == 2 && k + 1 < hpg) scan_head(k + 1, dt_next, sm->ad[0]);
        if (cq == 0) {
          float off = 0.f;
          for (int w = 3; w > q; --w) off += sm->red[w];
          const float su = ((sm->red[4] + sm->red[5]) + sm->red[6]) + sm->red[7];
          // <H, dS> from the 16 per-warp partials: a fixed shuffle tree within each
          // 16-lane half (every lane ends with the same total)
          float hsum = sm->red[40 + (lane & (kEpiWarps - 1))];
#pragma unroll
          for (int o = kEpiWarps / 2; o > 0; o >>= 1) hsum += __shfl_xor_sync(0xffffffffu, hsum, o);
          const float K = su + umma::ex2_approx(a2E5) * hsum;   // + dEpass = exp(E) <H, dS>
          const float da = (sfx + off) + K;
          __stcg(p.ddt + (row0 + r) * s.H + h, fmaf(Ah, da, dintra + eEA5 * sxy5));
          if (tid == 0 && !p.atomic) {
            const float sg = ((sm->red[8] + sm->red[9]) + sm->red[10]) + sm->red[11];
            const float sc = ((sm->red[12] + sm->red[13]) + sm->red[14]) + sm->red[15];
            const float dap = fmaf(K, sm->red[36 + (k & 1)], sc);
            __stcg(p.dA_part + (bi * s.nc + c) * s.H + h, dap);
            __stcg(p.dD_part + (bi * s.nc + c) * s.H + h, sg);
          }
        }
      }
      // No barrier here: only quarter-0 warps go on using this head's shared
      // values, and everything the next head overwrites is read before E5's
      // barrier above (or, for the step-size total, kept per head parity).
    }
    ep_sync();

    // ---- unit end: head-summed W (hi + lo) for the intra-chunk dB/dC products
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float w[16], hi[16], lo[16];
      umma::tmem_ld16(tmem + lane_off + T_WS + 64 * j + 16 * cq, w);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        hi[i] = __bfloat162float(__float2bfloat16_rn(w[i]));
        lo[i] = w[i] - hi[i];
      }
      st_row16_bf16(sm_base + OFF_WHI + j * 16384, r, 16 * cq, hi);
      st_row16_bf16(sm_base + OFF_WLO + j * 16384, r, 16 * cq, lo);
    }
    umma::fence_before_sync();
    umma::fence_proxy_async_smem();
    ep_sync();
    if (tid == 0) umma::mbar_arrive(&bars[E_WSUM]);
    ewait(&bars[B_FIN], 0, p.err);
    umma::fence_after_sync();
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int n0 = 32 * cq + 16 * j;
      float v[16];
      umma::tmem_ld16(tmem + lane_off + T_DB + n0, v);
      float *o = p.dB + ((row0 + r) * s.G + g) * kN + n0;
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4)
        __stcg(reinterpret_cast<float4 *>(o + 4 * i4), make_float4(v[4 * i4], v[4 * i4 + 1], v[4 * i4 + 2], v[4 * i4 + 3]));
      umma::tmem_ld16(tmem + lane_off + T_DC + n0, v);   // dC lanes: paired order
      o = p.dC + ((row0 + tr) * s.G + g) * kN + n0;
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4)
        __stcg(reinterpret_cast<float4 *>(o + 4 * i4), make_float4(v[4 * i4], v[4 * i4 + 1], v[4 * i4 + 2], v[4 * i4 + 3]));
    }
    umma::fence_before_sync();
    if (tid == 128) umma::tma_store_wait_all();
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    // after a give-up, let the tensor cores drain (bounded) before freeing TMEM
    if (sm->abort && lane == 0) {
      const long long t0 = clock64();
      while (!umma::mbar_try_wait(&bars[B_FIN], 0) && clock64() - t0 < kWaitCycles) {
      }
    }
    __syncwarp();
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, 512);
  }
}

// fp32 [p][n] view (hi + lo) of packed saved states, for inspection.
__global__ void __launch_bounds__(256) unpack_states_kernel(const float *__restrict__ packed, float *__restrict__ out) {
  const uint8_t *in = reinterpret_cast<const uint8_t *>(packed + int64_t(blockIdx.x) * kP * kN);
  float *o = out + int64_t(blockIdx.x) * kP * kN;
  for (int i = threadIdx.x; i < kN * (kP / 8); i += blockDim.x) {
    const int n = i >> 3, c0 = 8 * (i & 7);
    float hi[8], lo[8];
    ld8_bf16(in, n, c0, hi);
    ld8_bf16(in + 16384, n, c0, lo);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[(c0 + e) * kN + n] = hi[e] + lo[e];
  }
}

// dA[h], dD[h]: per-(batch, chunk) partials summed in ascending order.
__global__ void fold_scalars_kernel(Shape s, const float *__restrict__ dA_part, const float *__restrict__ dD_part,
                                    float *__restrict__ dA, float *__restrict__ dD) {
  const int64_t h = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (h >= s.H) return;
  dA[h] = column_sum(dA_part + h, s.b * s.nc, s.H, 0.f);
  dD[h] = column_sum(dD_part + h, s.b * s.nc, s.H, 0.f);
}

struct FusedWs {
  int *status;   // [0] error bits, [1] ticket
  int *flags;
  float *ring, *dA_part, *dD_part;
};

FusedWs carve_fused(Carver &cv, const Shape &s, int ring_depth) {
  FusedWs w;
  w.status = cv.take<int>(64);
  w.flags = cv.take<int>(s.b * s.nc * s.H);
  w.dA_part = cv.take<float>(s.b * s.nc * s.H);
  w.dD_part = cv.take<float>(s.b * s.nc * s.H);
  w.ring = cv.take<float>(int64_t(ring_depth) * s.b * s.H * kP * kN);
  return w;
}

}  // namespace

cudaError_t fused_unpack_states(const Shape &s, const float *packed, float *out, cudaStream_t st) {
  unpack_states_kernel<<<unsigned(s.b * s.nc * s.H), 256, 0, st>>>(packed, out);
  return cudaGetLastError();
}

bool fused_bwd_supported(const Shape &s, bool bf16) {
  // (dstate 256 with one group runs this kernel once per state half: fused_bwd_split)
  return bf16 && s.Q == kQ && s.N == kN && s.P == kP && s.T % kQ == 0 && s.hpg >= 1 &&
         s.b * s.nc * s.G <= (int64_t(1) << 30) && s.b * s.T <= (int64_t(1) << 30);
}

size_t fused_bwd_workspace(const Shape &s, int ring_depth) {
  Carver cv(nullptr);
  carve_fused(cv, s, ring_depth);
  return cv.bytes();
}

namespace {

// One launch of the fused kernel.  `bc_pitch`: elements per token row of B and C
// (the kernel reads columns [g * 128, g * 128 + 128) from `a.B`, `a.C`); `pass`
// picks the ticket counter (status[1 + pass]) so that consecutive launches on
// one workspace do not share one.
cudaError_t launch_pass(const Shape &s, const Args &a, const FusedWs &w, const FusedOptions &opt, int64_t bc_pitch,
                        int pass, int slice_shift, cudaStream_t st, Trace &tr) {
  // (slice_shift > 0: the sliced instantiation, adding its dx into dx; the unit groups of `s` are
  // then head slices, 2^slice_shift per group)
  const bool dx_add = slice_shift > 0;
  CUtensorMap tm_x, tm_g, tm_b, tm_c, tm_dx;
  const uint64_t rows = uint64_t(s.b * s.T);
  if (!make_tmap_2d(&tm_x, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, uint64_t(s.H * kP), uint64_t(s.H * kP), 64,
                    128, true) ||
      // g and C are copied in 16-token boxes (the paired row order of the kernel)
      !make_tmap_2d(&tm_g, a.dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, uint64_t(s.H * kP), uint64_t(s.H * kP),
                    64, 16, true) ||
      !make_tmap_2d(&tm_b, a.B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, uint64_t((s.G >> slice_shift) * kN),
                    uint64_t(bc_pitch), 64, 128, true) ||
      !make_tmap_2d(&tm_c, a.C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, uint64_t((s.G >> slice_shift) * kN),
                    uint64_t(bc_pitch), 64, 16, true) ||
      !make_tmap_2d(&tm_dx, a.dx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, rows, uint64_t(s.H * kP), uint64_t(s.H * kP), 32,
                    128, true))
    return cudaErrorInvalidValue;
  cudaError_t err;
  if ((err = cudaMemsetAsync(w.flags, 0, size_t(s.b * s.nc * s.H) * sizeof(int), st)) != cudaSuccess) return err;
  if ((err = cudaFuncSetAttribute(fused_bwd_kernel<false, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  SMEM_BYTES)) != cudaSuccess ||
      (err = cudaFuncSetAttribute(fused_bwd_kernel<true, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  SMEM_BYTES)) != cudaSuccess ||
      (err = cudaFuncSetAttribute(fused_bwd_kernel<true, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  SMEM_BYTES)) != cudaSuccess)
    return err;
  Params p;
  memset(&p, 0, sizeof(p));
  p.s = s;
  p.x = static_cast<const __nv_bfloat16 *>(a.x);
  p.dout = static_cast<const __nv_bfloat16 *>(a.dout);
  p.dt = a.dt;
  p.A = a.A;
  p.D = a.D;
  p.states = a.states_in;
  p.seq_idx = a.seq_idx;
  p.dx = a.dx;
  p.ddt = a.ddt;
  p.dB = a.dB;
  p.dC = a.dC;
  p.dinit = a.dinit;
  p.ring = w.ring;
  p.ring_depth = opt.ring_depth;
  p.flags = w.flags;
  p.err = w.status;
  p.ticket = w.status + 1 + pass;
  p.dA_part = w.dA_part;
  p.dD_part = w.dD_part;
  p.dA = a.dA;
  p.dD = a.dD;
  p.spin_limit = opt.spin_limit;
  p.atomic = opt.atomic ? 1 : 0;
  p.silent_chunk = opt.silent_chunk;
  const unsigned units = unsigned(s.b * s.nc * s.G);
  tr.mark(st);
  if (slice_shift == 2)
    fused_bwd_kernel<true, 2><<<units, kThreads, SMEM_BYTES, st>>>(p, tm_x, tm_g, tm_b, tm_c, tm_dx);
  else if (slice_shift == 1)
    fused_bwd_kernel<true, 1><<<units, kThreads, SMEM_BYTES, st>>>(p, tm_x, tm_g, tm_b, tm_c, tm_dx);
  else
    fused_bwd_kernel<false, 0><<<units, kThreads, SMEM_BYTES, st>>>(p, tm_x, tm_g, tm_b, tm_c, tm_dx);
  tr.mark(st);
  return cudaGetLastError();
}

// ---- dstate 256, one group: two state halves (see fused_fwd_split) --------
struct SplitBwdWs {
  FusedWs w, w1;                   // one per state half (the halves run concurrently)
  float *dD_scratch, *zeros;
  float *ddt1;                     // the second half's ddt
  float *dBh[2], *dCh[2], *dinit_h[2];
};

Shape split_half(const Shape &s) {
  Shape h = s;
  h.N = kN;
  h.Q = kQ;
  h.nc = s.T / kQ;
  return h;
}

// The half as the kernel sees it: the group's heads in 2^split_shift slices
// (four when the head count allows, else two), one unit each per chunk and
// half.  Shorter units pack the SMs more evenly, and more of them are
// independent: a unit waits only for the unit of the same slice in the chunk
// after, so more slices mean more, shorter chains of waiting units running
// side by side.  dB and dC are then per-slice partial sums.
int split_shift(const Shape &s) { return s.hpg % 4 == 0 ? 2 : 1; }
Shape split_units(const Shape &s) {
  Shape h = split_half(s);
  h.G = s.G << split_shift(s);
  h.hpg = s.hpg >> split_shift(s);
  return h;
}

SplitBwdWs carve_split(Carver &cv, const Shape &s, int ring_depth) {
  const Shape h = split_half(s);
  SplitBwdWs w;
  w.w = carve_fused(cv, h, ring_depth);
  w.w1 = carve_fused(cv, h, ring_depth);
  w.dD_scratch = cv.take<float>(h.H);
  w.zeros = cv.take<float>(h.H);
  w.ddt1 = cv.take<float>(s.b * s.T * s.H);
  const int64_t ns = int64_t(1) << split_shift(s);
  for (int j = 0; j < 2; ++j) {   // dB, dC: (b, T, slice, 128) partial sums of each half
    w.dBh[j] = cv.take<float>(s.b * s.T * ns * kN);
    w.dCh[j] = cv.take<float>(s.b * s.T * ns * kN);
    w.dinit_h[j] = cv.take<float>(s.nseq * s.H * kP * kN);
  }
  return w;
}

// ddt += ddt of the second half; dB, dC assembled from their halves (each the
// sum of its ns head slices in ascending slice order) and dinit from its
// halves (grid-stride over float4 groups of each array in turn)
__global__ void split_fold_kernel(int64_t n_ddt4, int64_t rows, int64_t init_rows, int ns, float *__restrict__ ddt,
                                  const float *__restrict__ ddt1, float *__restrict__ dB, float *__restrict__ dC,
                                  const float *__restrict__ dB0, const float *__restrict__ dB1,
                                  const float *__restrict__ dC0, const float *__restrict__ dC1,
                                  float *__restrict__ dinit, const float *__restrict__ di0,
                                  const float *__restrict__ di1) {
  const int64_t q = kN / 4;   // float4 groups in a 128-wide half row
  const int64_t n_bc = rows * 2 * q, n_in = init_rows * 2 * q;
  const int64_t total = n_ddt4 + 2 * n_bc + n_in;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    int64_t k = i;
    if (k < n_ddt4) {
      float4 a = reinterpret_cast<float4 *>(ddt)[k];
      const float4 b = __ldcs(reinterpret_cast<const float4 *>(ddt1) + k);
      a.x += b.x, a.y += b.y, a.z += b.z, a.w += b.w;
      reinterpret_cast<float4 *>(ddt)[k] = a;
      continue;
    }
    k -= n_ddt4;
    // output float4 k of a 256-wide row array: row k / (2q), half j, group within the half
    const float *src0, *src1;
    float *out;
    if (k < n_bc) {
      src0 = dB0, src1 = dB1, out = dB;
    } else if (k < 2 * n_bc) {
      k -= n_bc;
      src0 = dC0, src1 = dC1, out = dC;
    } else {
      k -= 2 * n_bc;
      src0 = di0, src1 = di1, out = dinit;
    }
    const int64_t row = k / (2 * q), rem = k % (2 * q), j = rem / q, g4 = rem % q;
    const float4 *src = reinterpret_cast<const float4 *>(j ? src1 : src0);
    if (out == dinit) {
      reinterpret_cast<float4 *>(out)[k] = __ldcs(src + row * q + g4);
    } else {   // head slices in ascending order
      float4 a = __ldcs(src + (row * ns) * q + g4);
      for (int sl = 1; sl < ns; ++sl) {
        const float4 b = __ldcs(src + (row * ns + sl) * q + g4);
        a.x += b.x, a.y += b.y, a.z += b.z, a.w += b.w;
      }
      reinterpret_cast<float4 *>(out)[k] = a;
    }
  }
}

// dA[h]: both halves' per-(batch, chunk) partials, half 0 then half 1, each in
// ascending chunk order; dD[h] from half 0 (its g . x terms do not depend on
// the state half).
__global__ void split_scalars_kernel(Shape h, const float *__restrict__ a0, const float *__restrict__ a1,
                                     const float *__restrict__ d0, float *__restrict__ dA, float *__restrict__ dD) {
  const int64_t hd = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (hd >= h.H) return;
  const int64_t n = h.b * h.nc;
  dA[hd] = column_sum(a1 + hd, n, h.H, column_sum(a0 + hd, n, h.H, 0.f));
  dD[hd] = column_sum(d0 + hd, n, h.H, 0.f);
}

}  // namespace

cudaError_t fused_bwd(const Shape &s, const Args &a, void *ws, const FusedOptions &opt, cudaStream_t st,
                      Trace &tr) {
  Carver cv(ws);
  FusedWs w = carve_fused(cv, s, opt.ring_depth);
  cudaError_t err = cudaMemsetAsync(w.status, 0, 64 * sizeof(int), st);
  if (err != cudaSuccess) return err;
  if (a.dinit && (err = cudaMemsetAsync(a.dinit, 0, size_t(s.nseq * s.H * kP * kN) * sizeof(float), st)) !=
                     cudaSuccess)
    return err;
  if (opt.atomic) {
    if ((err = cudaMemsetAsync(a.dA, 0, size_t(s.H) * sizeof(float), st)) != cudaSuccess) return err;
    if ((err = cudaMemsetAsync(a.dD, 0, size_t(s.H) * sizeof(float), st)) != cudaSuccess) return err;
  }
  if ((err = launch_pass(s, a, w, opt, s.G * kN, 0, 0, st, tr)) != cudaSuccess) return err;
  if (!opt.atomic) {
    tr.mark(st);
    fold_scalars_kernel<<<unsigned((s.H + 127) / 128), 128, 0, st>>>(s, w.dA_part, w.dD_part, a.dA, a.dD);
    tr.mark(st);
  }
  return cudaGetLastError();
}

size_t fused_bwd_split_workspace(const Shape &s, int ring_depth) {
  Carver cv(nullptr);
  carve_split(cv, s, ring_depth);
  return cv.bytes();
}

// A second stream per device on which the second state half runs next to the
// first (created once, kept for the life of the process).
cudaError_t side_stream(cudaStream_t *out) {
  static std::mutex mu;
  static cudaStream_t streams[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!streams[dev]) {
    const cudaError_t err = cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking);
    if (err != cudaSuccess) return err;
  }
  *out = streams[dev];
  return cudaSuccess;
}

cudaError_t fused_bwd_split(const Shape &s, const Args &a, void *ws, const FusedOptions &opt, cudaStream_t st,
                            Trace &tr) {
  const Shape h = split_half(s), hu = split_units(s);
  Carver cv(ws);
  SplitBwdWs w = carve_split(cv, s, opt.ring_depth);
  cudaError_t err;
  cudaStream_t side;
  if ((err = side_stream(&side)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(w.w.status, 0, 64 * sizeof(int), st)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(w.w1.status, 0, 64 * sizeof(int), st)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(w.zeros, 0, size_t(s.H) * sizeof(float), st)) != cudaSuccess) return err;
  // both halves add their dx into zeros: with two addends onto zero the sum is
  // the same bits in either order (0 + a = a exactly, and a + b = b + a)
  if ((err = cudaMemsetAsync(a.dx, 0, size_t(s.b * s.T * s.H * kP) * sizeof(float), st)) != cudaSuccess) return err;
  for (int j = 0; j < 2 && a.dinit; ++j)
    if ((err = cudaMemsetAsync(w.dinit_h[j], 0, size_t(s.nseq * s.H * kP * kN) * sizeof(float), st)) != cudaSuccess)
      return err;
  if (opt.atomic) {
    if ((err = cudaMemsetAsync(a.dA, 0, size_t(s.H) * sizeof(float), st)) != cudaSuccess) return err;
    if ((err = cudaMemsetAsync(a.dD, 0, size_t(s.H) * sizeof(float), st)) != cudaSuccess) return err;
  }
  // fork: the second half runs on the side stream once everything above is done
  cudaEvent_t fork, join;
  if ((err = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming)) != cudaSuccess) return err;
  if ((err = cudaEventCreateWithFlags(&join, cudaEventDisableTiming)) != cudaSuccess) {
    cudaEventDestroy(fork);
    return err;
  }
  err = cudaEventRecord(fork, st);
  if (err == cudaSuccess) err = cudaStreamWaitEvent(side, fork, 0);
  const int64_t tiles = h.b * h.nc * h.H * kP * kN;
  for (int j = 0; j < 2 && err == cudaSuccess; ++j) {
    Args aj = a;
    aj.B = static_cast<const __nv_bfloat16 *>(a.B) + j * kN;
    aj.C = static_cast<const __nv_bfloat16 *>(a.C) + j * kN;
    aj.states_in = a.states_in + j * tiles;
    aj.dB = w.dBh[j];
    aj.dC = w.dCh[j];
    aj.dinit = a.dinit ? w.dinit_h[j] : nullptr;
    if (j == 1) {
      aj.D = w.zeros;          // the skip term D x belongs to one half only
      aj.ddt = w.ddt1;
      aj.dD = w.dD_scratch;    // (atomic variant) g . x is counted by half 0
    }
    FusedWs wj = j ? w.w1 : w.w;
    wj.status = w.w.status;    // one status word (ticket status[1 + j] per half) for the check
    err = launch_pass(hu, aj, wj, opt, 2 * kN, j, split_shift(s), j ? side : st, tr);
  }
  if (err == cudaSuccess) err = cudaEventRecord(join, side);
  if (err == cudaSuccess) err = cudaStreamWaitEvent(st, join, 0);   // join before the fold
  cudaEventDestroy(fork);
  cudaEventDestroy(join);
  if (err != cudaSuccess) return err;
  const int64_t n_ddt4 = s.b * s.T * s.H / 4;
  const int64_t rows = s.b * s.T, init_rows = a.dinit ? s.nseq * s.H * kP : 0;
  tr.mark(st);
  split_fold_kernel<<<unsigned(8 * 152), 256, 0, st>>>(n_ddt4, rows, init_rows, 1 << split_shift(s), a.ddt, w.ddt1, a.dB, a.dC, w.dBh[0],
                                                       w.dBh[1], w.dCh[0], w.dCh[1], a.dinit, w.dinit_h[0],
                                                       w.dinit_h[1]);
  tr.mark(st);
  if (!opt.atomic) {
    tr.mark(st);
    split_scalars_kernel<<<unsigned((s.H + 127) / 128), 128, 0, st>>>(h, w.w.dA_part, w.w1.dA_part, w.w.dD_part,
                                                                       a.dA, a.dD);
    tr.mark(st);
  }
  return cudaGetLastError();
}

}  // namespace ssd
