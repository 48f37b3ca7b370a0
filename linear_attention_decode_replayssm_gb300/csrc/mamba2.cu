// ReplaySSM Mamba-2 cached decode step: the launch table.  The kernels are in
// mamba2.cuh; their instantiations are spread over three translation units
// (this one: one checkpoint copy, bf16 inputs; mamba2_variants.cu: read
// copies and group-shared keys; mamba2_f32in.cu: fp32 inputs) so that they
// compile in parallel.
#include "mamba2.cuh"

namespace rs {

LaunchFn find_mamba2_read_copy(int d_v, int d_k, int lp_dtype, int in_dtype);  // mamba2_variants.cu
LaunchFn find_mamba2_grouped(int d_v, int d_k, int ckpt_dtype, int in_dtype);  // mamba2_variants.cu
LaunchFn find_mamba2_f32_inputs(int d_v, int d_k, int ckpt_dtype);             // mamba2_f32in.cu

// launch_mamba2<d_v, d_k, checkpoint type, input type, consumer warps per
// group, groups, read-copy type, chunks per lane and row, fine window bounds,
// window warp>; the 64 x 128 fp32 and fp16 layers run with the window warp
static LaunchFn find_mamba2_bf16_inputs(int d_v, int d_k, int ckpt_dtype) {
  using RT = __nv_bfloat16;
  if (ckpt_dtype == kF32) {
    if (d_v == 16 && d_k == 32) return launch_mamba2<16, 32, float, RT, 4, 1>;
    if (d_v == 64 && d_k == 128) return launch_mamba2<64, 128, float, RT, 4, 2, float, 2, true, true>;
    if (d_v == 128 && d_k == 128) return launch_mamba2<128, 128, float, RT, 8, 1>;
  } else if (ckpt_dtype == kF16) {
    if (d_v == 16 && d_k == 32) return launch_mamba2<16, 32, __half, RT, 2, 1>;
    if (d_v == 64 && d_k == 128) return launch_mamba2<64, 128, __half, RT, 4, 2, __half, 1, true, true>;
    if (d_v == 128 && d_k == 128) return launch_mamba2<128, 128, __half, RT, 8, 1>;
  }
  return nullptr;
}

LaunchFn find_mamba2(int d_v, int d_k, int ckpt_dtype, int in_dtype, int lp_dtype, bool grouped) {
  if (grouped) return lp_dtype >= 0 ? nullptr : find_mamba2_grouped(d_v, d_k, ckpt_dtype, in_dtype);
  if (lp_dtype >= 0) return ckpt_dtype == kF32 ? find_mamba2_read_copy(d_v, d_k, lp_dtype, in_dtype) : nullptr;
  return in_dtype == kF32 ? find_mamba2_f32_inputs(d_v, d_k, ckpt_dtype) : find_mamba2_bf16_inputs(d_v, d_k, ckpt_dtype);
}

}  // namespace rs
