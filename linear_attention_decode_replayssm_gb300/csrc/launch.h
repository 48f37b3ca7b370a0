// Internal launch table shared by the kernel translation units and the C ABI.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace rs {

using LaunchFn = cudaError_t (*)(const KArgs &, cudaStream_t);

// nullptr when the (d_v, d_k, checkpoint dtype) combination is not built in.
LaunchFn find_mamba2(int d_v, int d_k, int ckpt_dtype, int in_dtype);
LaunchFn find_gdn(int d_v, int d_k, int ckpt_dtype, int ring_dtype, int in_dtype);
LaunchFn find_conventional(int variant, int d_v, int d_k, int ckpt_dtype);

// Launch shape of a persistent bulk-copy pipeline: CTAs, stages per CTA and
// dynamic shared memory, chosen from the device's shared-memory limits
// (`ctas_per_sm` CTAs per SM when two stages each still fit, else fewer) and
// the kernel's occupancy.
struct PipePlan {
  unsigned grid;
  int nstage;
  size_t smem;
};
using HeadFn = uint32_t (*)(int nstage);
cudaError_t plan_pipe(const void *kernel, int threads, size_t stage_bytes, HeadFn head, int max_stages,
                      int ctas_per_sm, int units, PipePlan *out);

// Launch shape of a kernel with a checkpoint-slot ring (nsc slots of
// `ck_bytes`) and a record-slot ring (nsr slots of `rec_bytes`): two CTAs
// per SM with 2 checkpoint and 4 record slots when that fits, else smaller or
// single-CTA shapes (see plan_rings).
struct RingPlan {
  unsigned grid;
  int nsr, nsc;
  size_t smem;
};
using RingHeadFn = uint32_t (*)(int nsr, int nsc);
cudaError_t plan_rings(const void *kernel, int threads, size_t ck_bytes, size_t rec_bytes, RingHeadFn head,
                       int units, RingPlan *out);

// Raise a kernel's dynamic shared-memory limit (once per device and kernel)
// when a launch needs more than the 48 KiB default.
cudaError_t ensure_smem(const void *kernel, size_t bytes);

}  // namespace rs
