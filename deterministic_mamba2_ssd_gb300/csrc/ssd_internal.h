// ssd_internal.h -- entry points of the kernel families, called by the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include <vector>

#include "ssd_common.cuh"

namespace ssd {

// General CUDA-core path (any shape; fp32 or bf16 inputs).
size_t simt_fwd_workspace(const Shape &s);
// variant: 0 per-head slots folded in order, 1 atomics, 2 ordered semaphore fold
size_t simt_bwd_workspace(const Shape &s, int variant);
int simt_bwd_launches(const Shape &s, int variant, bool seq);
const char *simt_bwd_launch_name(int variant, bool seq, int k);
cudaError_t simt_fwd(const Shape &s, bool bf16, const Args &a, void *ws, int block, cudaStream_t st);
cudaError_t simt_bwd(const Shape &s, bool bf16, const Args &a, void *ws, int block, int variant, uint32_t spin_limit,
                     cudaStream_t st, Trace &tr);

// Fused tensor-core backward (bf16, chunk 128, dstate 128, headdim 64).
struct FusedOptions {
  int ring_depth = 4;              // chunk slots of the state-gradient ring
  uint32_t spin_limit = 1u << 22;  // polls before a chain wait gives up (error bit 1)
  bool atomic = false;             // dA/dD by atomics instead of ordered partials
  int64_t silent_chunk = -1;       // fault injection: units of this chunk never publish
};
bool fused_bwd_supported(const Shape &s, bool bf16);
// Saved states of the fused family are the bf16 hi | lo operand tiles the
// fused backward copies straight into shared memory (32 KB per (P, N) tile,
// written by fused_fwd); this gives the fp32 view of them (hi + lo).
cudaError_t fused_unpack_states(const Shape &s, const float *packed, float *out, cudaStream_t st);
size_t fused_bwd_workspace(const Shape &s, int ring_depth);
// Tensor-core forward of the same family: y, and the states entering each
// chunk written directly in the packed form above.
size_t fused_fwd_workspace(const Shape &s);
cudaError_t fused_fwd(const Shape &s, const Args &a, void *ws, cudaStream_t st);
// Device status word of the tensor-core forward in its workspace (error bits of
// its bounded waits), for the plain, split and padded forms.
int *fused_fwd_status(const Shape &s, void *ws);
int *fused_fwd_split_status(const Shape &s, void *ws);
int *padded_fwd_status(const Shape &s, bool split, void *ws);

// dstate 256 with one group (chunk 128 or 256): the same kernels run once per
// state half (n < 128, n >= 128) as dstate-128 problems in 128-token chunks,
// their contributions summed in a fixed order.  The forward keeps the packed
// states of both halves in its workspace (fused_split_aux); the caller's state
// buffer gets the fp32 states entering each chunk.
bool fused_split_supported(const Shape &s, bool bf16);
size_t fused_fwd_split_workspace(const Shape &s);
float *fused_split_aux(const Shape &s, void *ws);
cudaError_t fused_fwd_split(const Shape &s, const Args &a, void *ws, cudaStream_t st);
size_t fused_bwd_split_workspace(const Shape &s, int ring_depth);
cudaError_t fused_bwd_split(const Shape &s, const Args &a, void *ws, const FusedOptions &opt, cudaStream_t st,
                            Trace &tr);
cudaError_t fused_bwd(const Shape &s, const Args &a, void *ws, const FusedOptions &opt, cudaStream_t st, Trace &tr);

// dstate 128 with a chunk length that is a larger multiple of 128 (the 256 of
// Mamba2's defaults, for one): y, the gradients and the state entering each
// chunk do not depend on the chunk length, so the kernels above run the
// problem in 128-token chunks (fused_chunk128_shape).  The forward keeps their
// packed states (one per 128 tokens) in its workspace (fused_chunk128_aux),
// which the backward reads; the caller's state buffer gets the fp32 states
// entering each of the caller's chunks.
bool fused_chunk128_supported(const Shape &s, bool bf16);
Shape fused_chunk128_shape(const Shape &s);
size_t fused_fwd_chunk128_workspace(const Shape &s);
float *fused_chunk128_aux(const Shape &s, void *ws);
int *fused_fwd_chunk128_status(const Shape &s, void *ws);
cudaError_t fused_fwd_chunk128(const Shape &s, const Args &a, void *ws, cudaStream_t st);

// Packed batches (batch 1, seq_idx) whose sequences may start inside a chunk:
// the token stream is cut at every sequence start and every 128 tokens, each
// piece padded to a 128-token chunk with tokens that leave the state and all
// real gradients unchanged, and the fused kernels above run the padded
// problem (`split`: the dstate-256 form).  The forward keeps the padded inputs
// and packed states in its workspace for the backward; the caller's state
// buffer gets the fp32 states entering each of its chunks.
int64_t padded_chunks(const Shape &s);   // ceil(T / 128) + nseq - 1
Shape padded_shape(const Shape &s);      // batch 1, padded_chunks chunks of 128 tokens
// Piece table from the host copy of seq_idx: start[npc] | len[npc] | id[npc] |
// map[nc] (caller chunk -> padded chunk); false if the ids change more often
// than nseq allows.
bool build_piece_table(const Shape &s, const int32_t *seq, std::vector<int32_t> &tab);
size_t padded_fwd_workspace(const Shape &s, bool split);
size_t padded_bwd_workspace(const Shape &s, bool split, int ring_depth);
cudaError_t padded_fwd(const Shape &s, bool split, const Args &a, const int32_t *host_seq, void *ws, cudaStream_t st);
cudaError_t padded_bwd(const Shape &s, bool split, const Args &a, const void *fwd_ws, void *ws,
                       const FusedOptions &opt, cudaStream_t st, Trace &tr);

}  // namespace ssd
