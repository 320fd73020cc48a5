// ssd_internal.h -- entry points of the kernel families, called by the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "ssd_common.cuh"

namespace ssd {

// General CUDA-core path (any shape; fp32 or bf16 inputs).
size_t simt_fwd_workspace(const Shape &s);
size_t simt_bwd_workspace(const Shape &s, bool atomic);
int simt_bwd_launches(const Shape &s, bool atomic);
const char *simt_bwd_launch_name(bool atomic, int k);
cudaError_t simt_fwd(const Shape &s, bool bf16, const Args &a, void *ws, int block, cudaStream_t st);
cudaError_t simt_bwd(const Shape &s, bool bf16, const Args &a, void *ws, int block, bool atomic, cudaStream_t st,
                     Trace &tr);

}  // namespace ssd
