// Internal launch table shared by the kernel translation units and the C ABI.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace rs {

using LaunchFn = cudaError_t (*)(const KArgs &, cudaStream_t);

// nullptr when the (d_v, d_k, checkpoint dtype) combination is not built in.
LaunchFn find_mamba2(int d_v, int d_k, int ckpt_dtype);
LaunchFn find_gdn(int d_v, int d_k, int ckpt_dtype);
LaunchFn find_conventional(int variant, int d_v, int d_k, int ckpt_dtype);

// Raise a kernel's dynamic shared-memory limit (once per device and kernel)
// when a launch needs more than the 48 KiB default.
cudaError_t ensure_smem(const void *kernel, size_t bytes);

}  // namespace rs
