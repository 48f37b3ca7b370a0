// Conventional load-update-store decode step (the baseline ReplaySSM is measured against).
//
// Sources:
//   [Ghana] S. Ghana, "ReplaySSM: an SSM decoder that writes its state once
//           every 16 tokens", §Why a fixed-size state is not cheap to decode
//           (Mamba-2: S_t = alpha_t S_{t-1} + v_t k_t^T, o_t = S_t q_t; every
//           step loads the state, updates it and stores it back) and §The
//           delta-rule wrinkle (S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T)
//           + beta_t v_t k_t^T, written as alpha_t S_{t-1} + u_t k_t^T with
//           u_t = beta_t (v_t - alpha_t S_{t-1} k_t)).
//
// Same tiling and streaming loads as the ReplaySSM kernels, so the two differ
// only in the bytes they move: this one reads and writes the whole state on
// every step.
#include "common.cuh"
#include "launch.h"

namespace rs {

// A unit is RB = DV / NSPLIT state rows of one (row, head): the rows of the
// update are independent once the row dots are known, so a 128 x 128 fp32
// head is two 32 KiB units, the same shape as a 64 x 128 Mamba-2 head.
template <int DV, int DK, typename TC, int NT, bool DELTA, int NSPLIT>
__device__ __forceinline__ void conventional_step(const KArgs &a) {
  using V = CkVec<TC>;
  constexpr int RB = DV / NSPLIT;
  constexpr int E = V::E;
  constexpr int G = DK / E;
  constexpr int RPP = NT / G;
  constexpr int VPT = RB / RPP;
  static_assert(G <= 32 && 32 % G == 0, "a state row must fit in one warp");
  static_assert(NT % G == 0 && RB % RPP == 0 && VPT >= 1 && VPT <= G, "bad tiling");

  __shared__ float sK[DK], sQ[DK], sV[RB], sU[RB], sC[RB];

  const int tid = threadIdx.x, lane = tid & 31;
  const int b = blockIdx.x / (a.H * NSPLIT);
  const int rem = blockIdx.x - b * (a.H * NSPLIT);
  const int h = rem / NSPLIT, row_off = (rem - h * NSPLIT) * RB;
  float *orow = a.out + (size_t)b * a.so + (size_t)h * DV + row_off;
  const int slot = __ldg(a.slot_idx + b);
  if (slot < 0) {
    for (int i = tid; i < RB; i += NT) orow[i] = 0.f;
    return;
  }
  if (slot >= a.num_slots) {
    if (tid == 0) report(a.dev_err, 1);
    for (int i = tid; i < RB; i += NT) orow[i] = 0.f;
    return;
  }
  const size_t unit = (size_t)slot * a.H + h;
  TC *st = static_cast<TC *>(a.ckpt) + unit * (size_t)(DV * DK) + (size_t)row_off * DK;
  const int row0 = tid / G, cv = tid - (tid / G) * G;

  uint4 raw[VPT];
#pragma unroll
  for (int r = 0; r < VPT; ++r) raw[r] = ld_stream(st + (size_t)(row0 + r * RPP) * DK + cv * E);

  for (int idx = tid; idx < DK / 8; idx += NT) {
    float f[8], g[8];
    load8(a.k, (size_t)b * a.sk + (size_t)h * DK + idx * 8, a.in_dtype, f);
    load8(a.q, (size_t)b * a.sq + (size_t)h * DK + idx * 8, a.in_dtype, g);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sK[idx * 8 + e] = f[e];
      sQ[idx * 8 + e] = g[e];
    }
  }
  for (int idx = tid; idx < RB / 8; idx += NT) {
    float f[8];
    load8(a.v, (size_t)b * a.sv + (size_t)h * DV + row_off + idx * 8, a.in_dtype, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) sV[idx * 8 + e] = f[e];
  }
  const float a_in = __ldg(a.alpha + (size_t)b * a.H + h);
  const float alpha = DELTA ? expf(a_in) : a_in;
  __syncthreads();

  float kv[E], qv[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    kv[e] = sK[cv * E + e];
    qv[e] = sQ[cv * E + e];
  }
  // rows are widened as they are used (the packed rows stay in registers):
  // fewer registers, more CTAs and bytes in flight per SM
  if (DELTA) {
    // u = beta (v - alpha S k): needs the full row dot S k first
    float part[VPT];
#pragma unroll
    for (int r = 0; r < VPT; ++r) {
      float fr[E];
      V::unpack(raw[r], fr);
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) s = fmaf(fr[e], kv[e], s);
      part[r] = s;
    }
    group_reduce<VPT, G>(part, lane);
    if (group_reduce_writer<VPT, G>(lane)) sC[row0 + group_reduce_index<VPT, G>(lane) * RPP] = part[0];
    __syncthreads();
    const float beta = __ldg(a.beta + (size_t)b * a.H + h);
    for (int i = tid; i < RB; i += NT) sU[i] = beta * (sV[i] - alpha * sC[i]);
    __syncthreads();
  }

  const float *upd = DELTA ? sU : sV;
  float part[VPT];
#pragma unroll
  for (int r = 0; r < VPT; ++r) {
    const float vv = upd[row0 + r * RPP];
    float fr[E];
    V::unpack(raw[r], fr);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      fr[e] = fmaf(alpha, fr[e], vv * kv[e]);
      s = fmaf(fr[e], qv[e], s);
    }
    part[r] = s;
    st_vec(st + (size_t)(row0 + r * RPP) * DK + cv * E, V::pack(fr));
  }
  group_reduce<VPT, G>(part, lane);
  if (group_reduce_writer<VPT, G>(lane)) sC[row0 + group_reduce_index<VPT, G>(lane) * RPP] = part[0];
  __syncthreads();
  for (int i = tid; i < RB; i += NT) orow[i] = sC[i];
}

template <int DV, int DK, typename TC, int NT, bool DELTA, int NSPLIT>
__global__ void __launch_bounds__(NT) conventional_kernel(const KArgs a) {
  conventional_step<DV, DK, TC, NT, DELTA, NSPLIT>(a);
}

// the same step with registers bounded so that MINB CTAs fit on an SM
template <int DV, int DK, typename TC, int NT, bool DELTA, int NSPLIT, int MINB>
__global__ void __launch_bounds__(NT, MINB) conventional_kernel_bounded(const KArgs a) {
  conventional_step<DV, DK, TC, NT, DELTA, NSPLIT>(a);
}

template <int DV, int DK, typename TC, int NT, bool DELTA, int NSPLIT = 1, int MINB = 0>
static cudaError_t launch_conv(const KArgs &a, cudaStream_t s) {
  const unsigned grid = (unsigned)((size_t)a.B * a.H * NSPLIT);
  if constexpr (MINB > 0)
    conventional_kernel_bounded<DV, DK, TC, NT, DELTA, NSPLIT, MINB><<<grid, NT, 0, s>>>(a);
  else
    conventional_kernel<DV, DK, TC, NT, DELTA, NSPLIT><<<grid, NT, 0, s>>>(a);
  return cudaGetLastError();
}

template <bool DELTA>
static LaunchFn find_conv_t(int d_v, int d_k, int ckpt_dtype) {
  if (ckpt_dtype == kF32) {
    if (d_v == 16 && d_k == 32) return launch_conv<16, 32, float, 128, DELTA>;
    if (d_v == 64 && d_k == 128) return launch_conv<64, 128, float, 256, DELTA>;
    if (d_v == 128 && d_k == 128) return launch_conv<128, 128, float, 256, DELTA, 2>;
  } else if (ckpt_dtype == kF16) {
    if (d_v == 16 && d_k == 32) return launch_conv<16, 32, __half, 64, DELTA>;
    // eight 16 KiB CTAs per SM keep enough bytes in flight (Mamba-2: 207 ->
    // 172 us at batch 256 with the rows widened as used); the delta rule
    // would spill at that bound
    if (d_v == 64 && d_k == 128) return launch_conv<64, 128, __half, 128, DELTA, 1, DELTA ? 0 : 8>;
    if (d_v == 128 && d_k == 128) return launch_conv<128, 128, __half, 256, DELTA>;
  }
  return nullptr;
}

LaunchFn find_conventional(int variant, int d_v, int d_k, int ckpt_dtype) {
  return variant == 1 ? find_conv_t<true>(d_v, d_k, ckpt_dtype) : find_conv_t<false>(d_v, d_k, ckpt_dtype);
}

}  // namespace rs
