// ssd_api.cu -- the C ABI: argument checks, launch-configuration table,
// workspace sizing and dispatch to the kernel families.  Nothing here
// allocates device memory or synchronises (except the documented seq_idx
// check in the forward).
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "mamba2_ssd.h"
#include "ssd_internal.h"

namespace {

constexpr uint32_t kSavedMagic = 0x53534432u;  // "SSD2"

bool dims_ok(const ssd_dims *d) {
  if (!d) return false;
  if (d->batch <= 0 || d->seqlen <= 0 || d->nheads <= 0 || d->headdim <= 0 || d->ngroups <= 0 || d->dstate <= 0 ||
      d->chunk_size <= 0 || d->nseq <= 0)
    return false;
  if (d->nheads % d->ngroups != 0) return false;
  if (d->dtype != SSD_F32 && d->dtype != SSD_BF16) return false;
  if ((d->flags & ~(SSD_DIMS_SEQ_IDX | SSD_DIMS_SEQ_ANY_START)) != 0) return false;
  if ((d->flags & SSD_DIMS_SEQ_ANY_START) && !(d->flags & SSD_DIMS_SEQ_IDX)) return false;
  // with seq_idx the kernels keep token positions and sequence ids in int32
  if ((d->flags & SSD_DIMS_SEQ_IDX) && (d->seqlen > INT32_MAX || d->nseq > INT32_MAX)) return false;
  if (d->chunk_size > 1024) return false;
  const int64_t nc = (d->seqlen + d->chunk_size - 1) / d->chunk_size;
  if (d->batch * nc * d->nheads > (int64_t(1) << 31) - 1) return false;
  return true;
}

ssd::Shape shape_of(const ssd_dims *d) {
  ssd::Shape s;
  s.b = d->batch;
  s.T = d->seqlen;
  s.H = d->nheads;
  s.P = d->headdim;
  s.G = d->ngroups;
  s.N = d->dstate;
  s.Q = d->chunk_size;
  s.nc = (d->seqlen + d->chunk_size - 1) / d->chunk_size;
  s.hpg = d->nheads / d->ngroups;
  s.nseq = d->nseq;
  return s;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch configurations.  General path: block sizes only (each output
// element is computed by one thread in one fixed order).  Fused path: depth
// of the state-gradient ring (scheduling slack only; the arithmetic and its
// order are the same).  Within a shape every configuration gives the same
// bits; the two paths are never both selectable for one shape.
constexpr int kSimtBlocks[] = {256, 128};
constexpr int kNumSimt = 2;
constexpr int kFusedRings[] = {4, 2};
constexpr int kNumFused = 2;

// Which backward a shape runs.  The fused kernels reset the state at chunk
// starts only; dstate 256 with one group runs them once per state half;
// dstate 128 with a longer chunk (a multiple of 128) runs them in 128-token
// chunks.
// Sequence starts inside a chunk run them on a padded copy of the problem
// (every piece of a sequence inside one 128-token chunk padded to a chunk of
// its own) when the padding at most doubles the chunk count, and take the
// general path otherwise.
enum Kind { kSimt = 0, kFused = 1, kSplit = 2, kFusedPad = 3, kSplitPad = 4, kChunk128 = 5 };
Kind kind_of(const ssd_dims *d) {
  const ssd::Shape s = shape_of(d);
  const bool bf16 = d->dtype == SSD_BF16;
  if (d->flags & SSD_DIMS_SEQ_ANY_START) {
    if (d->batch != 1 || !bf16 || s.nseq - 1 > (s.T + 127) / 128) return kSimt;
    const ssd::Shape p = ssd::padded_shape(s);
    // (the padded problem is in 128-token chunks whatever the caller's chunk, a multiple of 128)
    if (s.Q % 128 == 0 && ssd::fused_bwd_supported(p, bf16)) return kFusedPad;
    if (s.Q % 128 == 0 && ssd::fused_split_supported(p, bf16)) return kSplitPad;
    return kSimt;
  }
  if (ssd::fused_bwd_supported(s, bf16)) return kFused;
  if (ssd::fused_split_supported(s, bf16)) return kSplit;
  if (ssd::fused_chunk128_supported(s, bf16)) return kChunk128;
  return kSimt;
}
bool use_fused(const ssd_dims *d) { return kind_of(d) != kSimt; }
bool is_split(Kind k) { return k == kSplit || k == kSplitPad; }
bool is_padded(Kind k) { return k == kFusedPad || k == kSplitPad; }

bool has_seq(const ssd_dims *d) { return (d->flags & SSD_DIMS_SEQ_IDX) != 0; }

// Which variants a shape supports: the fused path folds dB/dC over heads
// inside one CTA, so the ordered-semaphore fold exists for the general path
// only (and needs its tile of 2 x 32 x dstate fp32 in shared memory and a
// unit count that fits a 1-D grid).
bool variant_ok(const ssd_dims *d, int variant) {
  if (variant == SSD_VARIANT_DETERMINISTIC || variant == SSD_VARIANT_ATOMIC) return true;
  if (variant != SSD_VARIANT_ORDERED || use_fused(d)) return false;
  const int64_t nc = (d->seqlen + d->chunk_size - 1) / d->chunk_size;
  const int64_t units = d->batch * nc * d->nheads * ((d->chunk_size + 31) / 32);
  return d->dstate <= 512 && units < (int64_t(1) << 31);
}

constexpr uint32_t kOrderedSpinLimit = 1u << 24;   // polls before an ordered-fold wait gives up

ssd::FusedOptions fused_options(const ssd_dims *d, int config, int variant) {
  ssd::FusedOptions o;
  // with sequence starts the chain can be cut, so every (128-token) chunk gets its own slot
  o.ring_depth = (d->flags & SSD_DIMS_SEQ_IDX) ? int((d->seqlen + 127) / 128) : kFusedRings[config];
  if (is_padded(kind_of(d))) o.ring_depth = int(ssd::padded_chunks(shape_of(d)));
  o.atomic = variant == SSD_VARIANT_ATOMIC;
  return o;
}

}  // namespace

extern "C" {

const char *mamba2_ssd_status_string(int status) {
  switch (status) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_ARG: return "invalid argument";
    case SSD_ERR_UNSUPPORTED: return "unsupported configuration";
    case SSD_ERR_WORKSPACE: return "workspace too small";
    case SSD_ERR_CUDA: return "CUDA error";
    case SSD_ERR_TIMEOUT: return "device-side wait timed out";
    case SSD_ERR_HANDLE: return "invalid saved struct";
    default: return "unknown status";
  }
}

int64_t mamba2_ssd_num_chunks(const ssd_dims *dims) {
  if (!dims_ok(dims)) return -1;
  return (dims->seqlen + dims->chunk_size - 1) / dims->chunk_size;
}

size_t mamba2_ssd_fwd_workspace_size(const ssd_dims *dims) {
  if (!dims_ok(dims)) return 0;
  switch (kind_of(dims)) {
    case kFused: return ssd::fused_fwd_workspace(shape_of(dims));
    case kChunk128: return ssd::fused_fwd_chunk128_workspace(shape_of(dims));
    case kSplit: return ssd::fused_fwd_split_workspace(shape_of(dims));
    case kFusedPad: return ssd::padded_fwd_workspace(shape_of(dims), false);
    case kSplitPad: return ssd::padded_fwd_workspace(shape_of(dims), true);
    default: return ssd::simt_fwd_workspace(shape_of(dims));
  }
}

int mamba2_ssd_num_configs(const ssd_dims *dims) {
  if (!dims_ok(dims)) return 0;
  return use_fused(dims) ? kNumFused : kNumSimt;
}

const char *mamba2_ssd_config_name(const ssd_dims *dims, int config) {
  if (!dims_ok(dims) || config < 0 || config >= mamba2_ssd_num_configs(dims)) return "invalid";
  switch (kind_of(dims)) {
    case kSplit: return config == 0 ? "fused-split/ring4" : "fused-split/ring2";
    case kFused: return config == 0 ? "fused/ring4" : "fused/ring2";
    case kChunk128: return config == 0 ? "fused-chunk128/ring4" : "fused-chunk128/ring2";
    // (with seq_idx every chunk has its own ring slot, so both configurations run the same launches)
    case kSplitPad: return config == 0 ? "fused-split-padded/0" : "fused-split-padded/1";
    case kFusedPad: return config == 0 ? "fused-padded/0" : "fused-padded/1";
    default: break;
  }
  return config == 0 ? "simt/block256" : "simt/block128";
}

size_t mamba2_ssd_bwd_workspace_size(const ssd_dims *dims, int config, int variant) {
  if (!dims_ok(dims) || config < 0 || config >= mamba2_ssd_num_configs(dims)) return 0;
  if (!variant_ok(dims, variant)) return 0;
  const int ring = fused_options(dims, config, variant).ring_depth;
  switch (kind_of(dims)) {
    case kSplit: return ssd::fused_bwd_split_workspace(shape_of(dims), ring);
    case kFused: return ssd::fused_bwd_workspace(shape_of(dims), ring);
    case kChunk128: return ssd::fused_bwd_workspace(ssd::fused_chunk128_shape(shape_of(dims)), ring);
    case kFusedPad: return ssd::padded_bwd_workspace(shape_of(dims), false, ring);
    case kSplitPad: return ssd::padded_bwd_workspace(shape_of(dims), true, ring);
    default: break;
  }
  return ssd::simt_bwd_workspace(shape_of(dims), variant);
}

int mamba2_ssd_bwd_num_launches(const ssd_dims *dims, int config, int variant) {
  if (!dims_ok(dims) || config < 0 || config >= mamba2_ssd_num_configs(dims)) return 0;
  if (!variant_ok(dims, variant)) return 0;
  const Kind kind = kind_of(dims);
  if (kind != kSimt) {
    const int core = is_split(kind) ? (variant == SSD_VARIANT_ATOMIC ? 3 : 4) : (variant == SSD_VARIANT_ATOMIC ? 1 : 2);
    return core + (is_padded(kind) ? 2 : 0);   // (padded: the dout gather before, the gradient scatter after)
  }
  return ssd::simt_bwd_launches(shape_of(dims), variant, has_seq(dims));
}

const char *mamba2_ssd_bwd_launch_name(const ssd_dims *dims, int config, int variant, int k) {
  if (!dims_ok(dims) || config < 0 || config >= mamba2_ssd_num_configs(dims)) return "invalid";
  if (!variant_ok(dims, variant)) return "invalid";
  const Kind kind = kind_of(dims);
  if (kind != kSimt) {
    const int n = mamba2_ssd_bwd_num_launches(dims, config, variant);
    if (k < 0 || k >= n) return "invalid";
    if (is_padded(kind)) {   // the gather and the scatter around the launches of the unpadded form
      if (k == 0) return "pad_gather";
      if (k == n - 1) return "pad_scatter";
      --k;
    }
    if (is_split(kind)) {   // one fused launch per state half, then the fold
      static const char *det[] = {"fused_bwd", "fused_bwd", "split_fold", "split_scalars"};
      static const char *atm[] = {"fused_bwd_atomic", "fused_bwd_atomic", "split_fold"};
      return variant == SSD_VARIANT_ATOMIC ? atm[k] : det[k];
    }
    if (variant == SSD_VARIANT_ATOMIC) return "fused_bwd_atomic";
    return k == 0 ? "fused_bwd" : "fold_scalars";
  }
  return ssd::simt_bwd_launch_name(variant, has_seq(dims), k);
}

ssd_status mamba2_ssd_bwd_check(const ssd_dims *dims, int config, const void *workspace, void *stream) {
  if (!dims_ok(dims) || config < 0 || config >= mamba2_ssd_num_configs(dims) || !workspace)
    return SSD_ERR_INVALID_ARG;
  // both paths keep their status word at the start of the workspace
  int word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return SSD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
  if (word & 4) return SSD_ERR_UNSUPPORTED;   // the fused kernel found its shared memory misaligned
  return word ? SSD_ERR_TIMEOUT : SSD_OK;
}

ssd_status mamba2_ssd_fwd_check(const ssd_dims *dims, const void *workspace, void *stream) {
  if (!dims_ok(dims) || !workspace) return SSD_ERR_INVALID_ARG;
  const ssd::Shape s = shape_of(dims);
  void *ws = const_cast<void *>(workspace);
  const int *status = nullptr;
  switch (kind_of(dims)) {
    case kFused: status = ssd::fused_fwd_status(s, ws); break;
    case kChunk128: status = ssd::fused_fwd_chunk128_status(s, ws); break;
    case kSplit: status = ssd::fused_fwd_split_status(s, ws); break;
    case kFusedPad: status = ssd::padded_fwd_status(s, false, ws); break;
    case kSplitPad: status = ssd::padded_fwd_status(s, true, ws); break;
    default: return SSD_OK;   // the general forward has no device-side waits
  }
  int word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return SSD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
  return word ? SSD_ERR_TIMEOUT : SSD_OK;
}

ssd_status mamba2_ssd_fwd(const ssd_dims *dims, const void *x, const float *dt, const float *A, const void *B,
                          const void *C, const float *D, const int32_t *seq_idx, const float *init_states, void *y,
                          float *states, void *workspace, size_t workspace_bytes, void *stream,
                          ssd_saved *saved_out) {
  if (!dims_ok(dims) || !saved_out) return SSD_ERR_INVALID_ARG;
  const void *req[] = {x, dt, A, B, C, D, y, states};
  for (const void *p : req)
    if (!p || !aligned16(p)) return SSD_ERR_INVALID_ARG;
  if ((seq_idx && !aligned16(seq_idx)) || (init_states && !aligned16(init_states))) return SSD_ERR_INVALID_ARG;
  if (!seq_idx && dims->nseq != dims->batch) return SSD_ERR_INVALID_ARG;
  if ((seq_idx != nullptr) != ((dims->flags & SSD_DIMS_SEQ_IDX) != 0)) return SSD_ERR_INVALID_ARG;
  const ssd::Shape s = shape_of(dims);
  if (workspace_bytes < mamba2_ssd_fwd_workspace_size(dims)) return SSD_ERR_WORKSPACE;
  if (!workspace || !aligned16(workspace)) return SSD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<int32_t> host_seq;
  if (seq_idx) {
    // Ids must be valid and non-decreasing; without SSD_DIMS_SEQ_ANY_START
    // every sequence start must also fall on a chunk start (the fused
    // backward resets the state there only).  One synchronous copy, documented.
    if (dims->batch != 1) return SSD_ERR_UNSUPPORTED;
    std::vector<int32_t> &h = host_seq;
    h.resize(size_t(s.T));
    if (cudaMemcpyAsync(h.data(), seq_idx, size_t(s.T) * sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return SSD_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
    for (int64_t t = 0; t < s.T; ++t) {
      if (h[t] < 0 || h[t] >= dims->nseq) return SSD_ERR_INVALID_ARG;
      if (t > 0 && h[t] < h[t - 1]) return SSD_ERR_INVALID_ARG;
      if (t > 0 && h[t] != h[t - 1] && t % s.Q != 0 && !(dims->flags & SSD_DIMS_SEQ_ANY_START))
        return SSD_ERR_UNSUPPORTED;
    }
  }
  ssd::Args a{};
  a.x = x; a.B = B; a.C = C; a.dt = dt; a.A = A; a.D = D;
  a.init = init_states; a.seq_idx = seq_idx; a.y = y; a.states_out = states;
  // The fused shape family runs the tensor-core forward, which writes each saved state as the
  // packed bf16 hi | lo operand pair the fused backward takes; dstate 256 runs it per state half
  // (packed states of both halves kept in the workspace), dstate 128 with a longer chunk in
  // 128-token chunks (packed states kept in the workspace); every other shape the general one.
  // Sequence starts inside a chunk run the fused kernels on a padded copy kept in the workspace.
  const Kind kind = kind_of(dims);
  cudaError_t err;
  switch (kind) {
    case kFused: err = ssd::fused_fwd(s, a, workspace, st); break;
    case kChunk128: err = ssd::fused_fwd_chunk128(s, a, workspace, st); break;
    case kSplit: err = ssd::fused_fwd_split(s, a, workspace, st); break;
    case kFusedPad:
    case kSplitPad: err = ssd::padded_fwd(s, kind == kSplitPad, a, host_seq.data(), workspace, st); break;
    default: err = ssd::simt_fwd(s, dims->dtype == SSD_BF16, a, workspace, kSimtBlocks[0], st);
  }
  if (err != cudaSuccess) return SSD_ERR_CUDA;
  saved_out->aux = kind == kSplit      ? ssd::fused_split_aux(s, workspace)
                   : kind == kChunk128 ? ssd::fused_chunk128_aux(s, workspace)
                   : is_padded(kind)   ? static_cast<const float *>(workspace)
                                       : nullptr;
  saved_out->dims = *dims;
  saved_out->x = x; saved_out->dt = dt; saved_out->A = A; saved_out->B = B; saved_out->C = C; saved_out->D = D;
  saved_out->seq_idx = seq_idx; saved_out->init_states = init_states; saved_out->states = states;
  saved_out->magic = kSavedMagic;
  saved_out->flags = 0;
  return SSD_OK;
}

int64_t mamba2_ssd_padded_chunks(const ssd_dims *dims) {
  if (!dims_ok(dims) || !is_padded(kind_of(dims))) return 0;
  return ssd::padded_chunks(shape_of(dims));
}

ssd_status mamba2_ssd_padded_piece_table(const ssd_dims *dims, const int32_t *seq_idx, int32_t *table) {
  if (!dims_ok(dims) || !is_padded(kind_of(dims)) || !seq_idx || !table) return SSD_ERR_INVALID_ARG;
  const ssd::Shape s = shape_of(dims);
  for (int64_t t = 0; t < s.T; ++t)
    if (seq_idx[t] < 0 || seq_idx[t] >= s.nseq || (t > 0 && seq_idx[t] < seq_idx[t - 1])) return SSD_ERR_INVALID_ARG;
  std::vector<int32_t> tab;
  if (!ssd::build_piece_table(s, seq_idx, tab)) return SSD_ERR_INVALID_ARG;
  std::copy(tab.begin(), tab.end(), table);
  return SSD_OK;
}

ssd_status mamba2_ssd_states_unpack(const ssd_saved *saved, float *out, void *stream) {
  if (!saved || saved->magic != kSavedMagic || !dims_ok(&saved->dims)) return SSD_ERR_HANDLE;
  if (!saved->states || !out || !aligned16(out)) return SSD_ERR_INVALID_ARG;
  const ssd::Shape s = shape_of(&saved->dims);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (kind_of(&saved->dims) == kFused)
    return ssd::fused_unpack_states(s, saved->states, out, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
  const size_t bytes = size_t(s.b * s.nc * s.H * s.P * s.N) * sizeof(float);
  return cudaMemcpyAsync(out, saved->states, bytes, cudaMemcpyDeviceToDevice, st) == cudaSuccess ? SSD_OK
                                                                                                 : SSD_ERR_CUDA;
}

ssd_status mamba2_ssd_bwd_traced(const ssd_saved *saved, const void *dout, float *dx, float *ddt, float *dA,
                                 float *dB, float *dC, float *dD, float *dinit, void *workspace,
                                 size_t workspace_bytes, int config, int variant, void *stream,
                                 void *const *events, int num_events) {
  if (!saved || saved->magic != kSavedMagic || !dims_ok(&saved->dims)) return SSD_ERR_HANDLE;
  const ssd_dims *dims = &saved->dims;
  const void *req[] = {saved->x, saved->dt, saved->A, saved->B, saved->C, saved->D, saved->states,
                       dout, dx, ddt, dA, dB, dC, dD};
  for (const void *p : req)
    if (!p || !aligned16(p)) return SSD_ERR_INVALID_ARG;
  if (dinit && (!aligned16(dinit) || !saved->init_states)) return SSD_ERR_INVALID_ARG;
  if (variant != SSD_VARIANT_DETERMINISTIC && variant != SSD_VARIANT_ATOMIC && variant != SSD_VARIANT_ORDERED)
    return SSD_ERR_INVALID_ARG;
  if (config < 0 || config >= mamba2_ssd_num_configs(dims)) return SSD_ERR_INVALID_ARG;
  if (!variant_ok(dims, variant)) return SSD_ERR_UNSUPPORTED;
  const ssd::Shape s = shape_of(dims);
  if (workspace_bytes < mamba2_ssd_bwd_workspace_size(dims, config, variant)) return SSD_ERR_WORKSPACE;
  if (!workspace || !aligned16(workspace)) return SSD_ERR_INVALID_ARG;
  ssd::Args a{};
  a.x = saved->x; a.B = saved->B; a.C = saved->C; a.dout = dout;
  a.dt = saved->dt; a.A = saved->A; a.D = saved->D; a.init = saved->init_states; a.states_in = saved->states;
  a.seq_idx = saved->seq_idx;
  a.dx = dx; a.ddt = ddt; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.dinit = dinit;
  if (num_events < 0 || (num_events > 0 && !events)) return SSD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ssd::Trace tr;
  tr.events = reinterpret_cast<cudaEvent_t *>(const_cast<void **>(events));
  tr.count = num_events;
  cudaError_t err;
  const Kind kind = kind_of(dims);
  if (is_padded(kind) || kind == kSplit || kind == kChunk128) {
    if (!saved->aux) return SSD_ERR_HANDLE;   // the packed states live in the forward's workspace
  }
  if (is_padded(kind)) {
    err = ssd::padded_bwd(s, kind == kSplitPad, a, saved->aux, workspace, fused_options(dims, config, variant), st, tr);
  } else if (kind == kSplit) {
    a.states_in = saved->aux;
    err = ssd::fused_bwd_split(s, a, workspace, fused_options(dims, config, variant), st, tr);
  } else if (kind == kChunk128) {
    a.states_in = saved->aux;
    err = ssd::fused_bwd(ssd::fused_chunk128_shape(s), a, workspace, fused_options(dims, config, variant), st, tr);
  } else if (kind == kFused)
    err = ssd::fused_bwd(s, a, workspace, fused_options(dims, config, variant), st, tr);
  else
    err = ssd::simt_bwd(s, dims->dtype == SSD_BF16, a, workspace, kSimtBlocks[config], variant, kOrderedSpinLimit, st,
                        tr);
  return err == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status mamba2_ssd_bwd_fault_test(const ssd_saved *saved, const void *dout, float *dx, float *ddt, float *dA,
                                     float *dB, float *dC, float *dD, float *dinit, void *workspace,
                                     size_t workspace_bytes, int64_t silent_chunk, uint32_t spin_limit,
                                     void *stream) {
  if (!saved || saved->magic != kSavedMagic || !dims_ok(&saved->dims)) return SSD_ERR_HANDLE;
  const ssd_dims *dims = &saved->dims;
  if (kind_of(dims) != kFused) return SSD_ERR_UNSUPPORTED;
  const void *req[] = {saved->x, saved->dt, saved->A, saved->B, saved->C, saved->D, saved->states,
                       dout, dx, ddt, dA, dB, dC, dD};
  for (const void *p : req)
    if (!p || !aligned16(p)) return SSD_ERR_INVALID_ARG;
  if (workspace_bytes < mamba2_ssd_bwd_workspace_size(dims, 0, 0)) return SSD_ERR_WORKSPACE;
  if (!workspace || !aligned16(workspace) || spin_limit == 0) return SSD_ERR_INVALID_ARG;
  ssd::Args a{};
  a.x = saved->x; a.B = saved->B; a.C = saved->C; a.dout = dout;
  a.dt = saved->dt; a.A = saved->A; a.D = saved->D; a.init = saved->init_states; a.states_in = saved->states;
  a.seq_idx = saved->seq_idx;
  a.dx = dx; a.ddt = ddt; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.dinit = dinit;
  ssd::FusedOptions o = fused_options(dims, 0, 0);
  o.silent_chunk = silent_chunk;
  o.spin_limit = spin_limit;
  ssd::Trace tr;
  return ssd::fused_bwd(shape_of(dims), a, workspace, o, static_cast<cudaStream_t>(stream), tr) == cudaSuccess
             ? SSD_OK
             : SSD_ERR_CUDA;
}

ssd_status mamba2_ssd_bwd(const ssd_saved *saved, const void *dout, float *dx, float *ddt, float *dA, float *dB,
                          float *dC, float *dD, float *dinit, void *workspace, size_t workspace_bytes, int config,
                          int variant, void *stream) {
  return mamba2_ssd_bwd_traced(saved, dout, dx, ddt, dA, dB, dC, dD, dinit, workspace, workspace_bytes, config,
                               variant, stream, nullptr, 0);
}

}  // extern "C"
