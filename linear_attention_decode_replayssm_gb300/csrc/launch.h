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

// Launch shape of a persistent bulk-copy pipeline: CTAs, stages per CTA and
// dynamic shared memory, chosen from the device's shared-memory limits
// (two CTAs per SM when two stages each still fit, else one CTA per SM) and
// the kernel's occupancy.
struct PipePlan {
  unsigned grid;
  int nstage;
  size_t smem;
};
using HeadFn = uint32_t (*)(int nstage);
cudaError_t plan_pipe(const void *kernel, int threads, size_t stage_bytes, HeadFn head, int max_stages, int units,
                      PipePlan *out);

// Raise a kernel's dynamic shared-memory limit (once per device and kernel)
// when a launch needs more than the 48 KiB default.
cudaError_t ensure_smem(const void *kernel, size_t bytes);

}  // namespace rs
