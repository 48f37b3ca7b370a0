// Launch table of the Mamba-2 decode with a two-precision checkpoint (read
// copy) or group-shared keys; kernels in mamba2.cuh.
#include "mamba2.cuh"

namespace rs {

// template arguments as in mamba2.cu; the 64 x 128 layer's read-copy and
// grouped-key kernels run with the window warp
template <typename RT>
static LaunchFn read_copy_t(int d_v, int d_k, int lp_dtype) {
  if (lp_dtype == kF16) {
    if (d_v == 16 && d_k == 32) return launch_mamba2<16, 32, float, RT, 4, 1, __half>;
    if (d_v == 64 && d_k == 128) return launch_mamba2<64, 128, float, RT, 4, 2, __half, 4, false, true>;
    if (d_v == 128 && d_k == 128) return launch_mamba2<128, 128, float, RT, 8, 1, __half>;
  } else if (lp_dtype == kBF16) {
    if (d_v == 16 && d_k == 32) return launch_mamba2<16, 32, float, RT, 4, 1, __nv_bfloat16>;
    if (d_v == 64 && d_k == 128) return launch_mamba2<64, 128, float, RT, 4, 2, __nv_bfloat16, 4, false, true>;
    if (d_v == 128 && d_k == 128) return launch_mamba2<128, 128, float, RT, 8, 1, __nv_bfloat16>;
  } else if (lp_dtype == kF8) {
    // E4M3 with a power-of-two scale per state row
    if (d_v == 64 && d_k == 128) return launch_mamba2<64, 128, float, RT, 4, 2, __nv_fp8_e4m3, 4, false, true>;
  }
  return nullptr;
}

template <typename RT>
static LaunchFn grouped_t(int d_v, int d_k, int ckpt_dtype) {
  if (ckpt_dtype == kF32) {
    if (d_v == 16 && d_k == 32) return launch_mamba2_grp<16, 32, float, RT, 4, 1>;
    if (d_v == 64 && d_k == 128) return launch_mamba2_grp<64, 128, float, RT, 4, 2, 1, true>;
  } else if (ckpt_dtype == kF16) {
    if (d_v == 64 && d_k == 128) return launch_mamba2_grp<64, 128, __half, RT, 8, 1>;
  }
  return nullptr;
}

// the fp32 checkpoint's read copy (lp_dtype fp16, bf16 or E4M3)
LaunchFn find_mamba2_read_copy(int d_v, int d_k, int lp_dtype, int in_dtype) {
  return in_dtype == kF32 ? read_copy_t<float>(d_v, d_k, lp_dtype) : read_copy_t<__nv_bfloat16>(d_v, d_k, lp_dtype);
}

LaunchFn find_mamba2_grouped(int d_v, int d_k, int ckpt_dtype, int in_dtype) {
  return in_dtype == kF32 ? grouped_t<float>(d_v, d_k, ckpt_dtype) : grouped_t<__nv_bfloat16>(d_v, d_k, ckpt_dtype);
}

}  // namespace rs
