// Launch table of the Mamba-2 decode with fp32 inputs and records (one
// checkpoint copy); kernels in mamba2.cuh.
#include "mamba2.cuh"

namespace rs {

LaunchFn find_mamba2_f32_inputs(int d_v, int d_k, int ckpt_dtype) {
  using RT = float;
  if (ckpt_dtype == kF32) {
    if (d_v == 16 && d_k == 32) return launch_mamba2<16, 32, float, RT, 4, 1>;
    if (d_v == 64 && d_k == 128) return launch_mamba2<64, 128, float, RT, 4, 2, float, 2>;
    if (d_v == 128 && d_k == 128) return launch_mamba2<128, 128, float, RT, 8, 1>;
  } else if (ckpt_dtype == kF16) {
    if (d_v == 16 && d_k == 32) return launch_mamba2<16, 32, __half, RT, 2, 1>;
    if (d_v == 64 && d_k == 128) return launch_mamba2<64, 128, __half, RT, 4, 2>;
    if (d_v == 128 && d_k == 128) return launch_mamba2<128, 128, __half, RT, 8, 1>;
  }
  return nullptr;
}

}  // namespace rs
