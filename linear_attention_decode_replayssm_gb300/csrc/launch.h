// Internal launch table shared by the kernel translation units and the C ABI.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"
#include "replayssm.h"

namespace rs {

using LaunchFn = cudaError_t (*)(const KArgs &, cudaStream_t);

// nullptr when the (d_v, d_k, checkpoint dtype) combination is not built in.
// lp_dtype: read-copy type of a two-precision checkpoint, or -1 for none;
// grouped: keys and queries shared by groups of heads
LaunchFn find_mamba2(int d_v, int d_k, int ckpt_dtype, int in_dtype, int lp_dtype, bool grouped);
LaunchFn find_gdn(int d_v, int d_k, int ckpt_dtype, int ring_dtype, int in_dtype);
LaunchFn find_conventional(int variant, int d_v, int d_k, int ckpt_dtype);

// State materialisation; `gdn` selects log-gate weights (exp of suffix sums)
// over decay products.
using MatLaunchFn = cudaError_t (*)(const rs_materialize_args &, int gdn, cudaStream_t);
MatLaunchFn find_materialize(int d_v, int d_k, int ckpt_dtype);
// the pipelined materialisation (materialize_pipe.cu) for 64 x 128 Mamba-2
// and 128 x 128 GDN heads, or nullptr where it is not built
MatLaunchFn find_mat_pipe(int gdn, int d_v, int d_k, int ckpt_dtype, int ring_dtype);

// Speculative verification (Mamba-2) and the device-side commit.
using SpecLaunchFn = cudaError_t (*)(const rs_spec_args &, cudaStream_t);
SpecLaunchFn find_spec(int d_v, int d_k, int ckpt_dtype, int in_dtype);
// the tensor-core verification (spec_tc.cu), or nullptr where it is not built
SpecLaunchFn find_spec_tc(int d_v, int d_k, int ckpt_dtype, int in_dtype);
cudaError_t launch_spec_commit(const int32_t *committed, const uint8_t *is_flush, const int32_t *accepted, int B,
                               int L, int T, int32_t *committed_out, uint8_t *is_flush_out, int32_t *dev_err,
                               cudaStream_t s);

// Launch shape of a kernel with a checkpoint-slot ring (nsc slots of
// `ck_bytes`) and a record-slot ring (nsr slots of `rec_bytes`): two CTAs
// per SM with 2 checkpoint and 4 record slots when that fits, else smaller or
// single-CTA shapes (see plan_rings).
struct RingPlan {
  unsigned grid;
  int nsr, nsc;
  size_t smem;
};
// `shapes` ({CTAs per SM, checkpoint slots, record slots}, best first)
// replaces the default list when given.
using RingHeadFn = uint32_t (*)(int nsr, int nsc);
cudaError_t plan_rings(const void *kernel, int threads, size_t ck_bytes, size_t rec_bytes, RingHeadFn head,
                       int units, RingPlan *out, const int (*shapes)[3] = nullptr, int n_shapes = 0);

// The read copy of a two-precision checkpoint cast from its recurrence copy
// (materialize.cu): n_rows rows of d_k fp32 values.
cudaError_t launch_seed_read_copy(const float *ckpt, int64_t n_rows, int d_k, int lp_dtype, void *ckpt_lp, float *scale,
                                  cudaStream_t s);

// Raise a kernel's dynamic shared-memory limit (once per device and kernel)
// when a launch needs more than the 48 KiB default.
cudaError_t ensure_smem(const void *kernel, size_t bytes);

}  // namespace rs
