// Materialisation of the exact recurrent state from a checkpoint and the
// records its ring holds, for prefix caching.
//
// Sources:
//   [Ghana] S. Ghana, "ReplaySSM: an SSM decoder that writes its state once
//           every 16 tokens", §What actually shipped (a cached prefix needs
//           the exact state at a cache-block boundary; between flushes only
//           the checkpoint and the ring exist, so a separate kernel builds
//           the state) and §The identity (the state after h records is
//           gamma_h S_ckpt + sum_j gamma_{j+1:h} v_j k_j^T).
//   [PR48792] vLLM pull request 48792, §Core concept (Gated DeltaNet: the same
//           unroll over cached corrected values d_j with gate weights
//           exp(sum_{l>j} g_l)).
//
// Work per (row, head): read the checkpoint and the held records once, write
// the state once.  One CTA per (row, head, row block), the checkpoint streamed
// into registers as in the conventional kernel; the held records are staged in
// shared memory 16 at a time, values pre-scaled by their window weight.
#include "common.cuh"
#include "launch.h"

namespace rs {

template <int DV, int DK, typename TC, int NT, int NSPLIT>
__global__ void __launch_bounds__(NT) materialize_kernel(const rs_materialize_args a, int gdn) {
  using V = CkVec<TC>;
  constexpr int RB = DV / NSPLIT;
  constexpr int E = V::E;
  constexpr int G = DK / E;
  constexpr int RPP = NT / G;
  constexpr int VPT = RB / RPP;
  constexpr int CH = 16;  // records staged per pass
  static_assert(G <= 32 && 32 % G == 0, "a state row must fit in one warp");
  static_assert(NT % G == 0 && RB % RPP == 0 && VPT >= 1, "bad tiling");
  static_assert(RB % 8 == 0 && DK % 8 == 0 && RS_MAX_L <= 64, "bad staging");

  __shared__ __align__(16) float sK[CH][DK];
  __shared__ float sV[CH][RB];
  __shared__ float sW[64];
  __shared__ float sGam;

  const int tid = threadIdx.x, lane = tid & 31;
  const int b = blockIdx.x / (a.H * NSPLIT);
  const int rem = blockIdx.x - b * (a.H * NSPLIT);
  const int h = rem / NSPLIT, row_off = (rem - h * NSPLIT) * RB;
  const int slot = __ldg(a.slot_idx + b), dst = __ldg(a.dst_idx + b);
  if (slot < 0 || dst < 0) return;
  const int p = __ldg(a.held + b);
  const int bad = (slot >= a.num_slots ? RS_DERR_SLOT : 0) | (dst >= a.num_dst ? RS_DERR_DST : 0) |
                  (p < 0 || p >= a.L ? RS_DERR_WRITE_POS : 0);
  if (bad) {
    if (tid == 0) report(a.dev_err, bad);
    return;
  }

  const size_t unit = (size_t)slot * a.H + h;
  const TC *src = static_cast<const TC *>(a.ckpt) + unit * (size_t)(DV * DK) + (size_t)row_off * DK;
  TC *out = static_cast<TC *>(a.dst) + ((size_t)dst * a.H + h) * (size_t)(DV * DK) + (size_t)row_off * DK;
  const int row0 = tid / G, cv = tid - (tid / G) * G;

  uint4 raw[VPT];
#pragma unroll
  for (int r = 0; r < VPT; ++r) raw[r] = ld_stream(src + (size_t)(row0 + r * RPP) * DK + cv * E);

  if (tid < 32) {
    // window weights: w_j = decay of the records after j, gamma = decay of all
    // p records; Mamba-2 multiplies decays, GDN sums log-gates then exponentiates
    const float ident = gdn ? 0.f : 1.f;
    const float *ra = a.ring_a + unit * a.L;
    float x0 = lane < p ? __ldg(ra + lane) : ident;
    float x1 = lane + 32 < p ? __ldg(ra + lane + 32) : ident;
    if (gdn)
      suffix_scan64(x0, x1, lane, [](float x, float y) { return x + y; });
    else
      suffix_scan64(x0, x1, lane, [](float x, float y) { return x * y; });
    const float n0 = __shfl_down_sync(0xffffffffu, x0, 1);
    const float n1 = __shfl_down_sync(0xffffffffu, x1, 1);
    const float hi0 = __shfl_sync(0xffffffffu, x1, 0);
    float w0 = lane == 31 ? hi0 : n0, w1 = lane == 31 ? ident : n1;
    if (gdn) {
      w0 = expf(w0);
      w1 = expf(w1);
    }
    sW[lane] = w0;
    sW[lane + 32] = w1;
    if (lane == 0) sGam = gdn ? expf(x0) : x0;
  }
  __syncthreads();

  float f[VPT][E];
  const float gam = sGam;
#pragma unroll
  for (int r = 0; r < VPT; ++r) {
    V::unpack(raw[r], f[r]);
#pragma unroll
    for (int e = 0; e < E; ++e) f[r][e] *= gam;
  }

  const size_t rec0 = unit * a.L;
  for (int j0 = 0; j0 < p; j0 += CH) {
    const int cnt = min(CH, p - j0);
    for (int idx = tid; idx < cnt * (DK / 8); idx += NT) {
      const int jj = idx / (DK / 8), c8 = idx - jj * (DK / 8);
      float t[8];
      load8(a.ring_k, (rec0 + j0 + jj) * DK + c8 * 8, a.ring_dtype, t);
#pragma unroll
      for (int e = 0; e < 8; ++e) sK[jj][c8 * 8 + e] = t[e];
    }
    for (int idx = tid; idx < cnt * (RB / 8); idx += NT) {
      const int jj = idx / (RB / 8), c8 = idx - jj * (RB / 8);
      float t[8];
      load8(a.ring_v, (rec0 + j0 + jj) * DV + row_off + c8 * 8, a.ring_dtype, t);
      const float w = sW[j0 + jj];
#pragma unroll
      for (int e = 0; e < 8; ++e) sV[jj][c8 * 8 + e] = w * t[e];
    }
    __syncthreads();
    for (int jj = 0; jj < cnt; ++jj) {
      float kv[E];
#pragma unroll
      for (int e = 0; e < E; ++e) kv[e] = sK[jj][cv * E + e];
#pragma unroll
      for (int r = 0; r < VPT; ++r) {
        const float vv = sV[jj][row0 + r * RPP];
#pragma unroll
        for (int e = 0; e < E; ++e) f[r][e] = fmaf(vv, kv[e], f[r][e]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int r = 0; r < VPT; ++r) st_vec(out + (size_t)(row0 + r * RPP) * DK + cv * E, V::pack(f[r]));
}

// The read copy of a two-precision checkpoint from its recurrence copy: one
// warp per state row; E4M3 rows on their power-of-two scale.
__global__ void __launch_bounds__(256) seed_read_copy_kernel(const float *ckpt, int64_t n_rows, int d_k, int lp_dtype,
                                                             void *ckpt_lp, float *scale) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  const float *src = ckpt + row * d_k;
  const int nq = d_k / 4;  // 4-column groups
  if (lp_dtype == kF8) {
    float amax = 0.f;
    for (int c = lane; c < nq; c += 32) {
      const float4 x = reinterpret_cast<const float4 *>(src)[c];
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const int e = e4m3_row_exponent(amax);
    uint32_t *dst = reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(ckpt_lp) + row * d_k);
    for (int c = lane; c < nq; c += 32) {
      const float4 x = reinterpret_cast<const float4 *>(src)[c];
      dst[c] = e4m3_pack4(x.x, x.y, x.z, x.w, e);
    }
    if (lane == 0) scale[row] = ldexpf(1.f, e);
  } else {
    uint2 *dst = reinterpret_cast<uint2 *>(static_cast<unsigned char *>(ckpt_lp) + row * d_k * 2);
    for (int c = lane; c < nq; c += 32) {
      const float4 x = reinterpret_cast<const float4 *>(src)[c];
      const float f[4] = {x.x, x.y, x.z, x.w};
      dst[c] = lp_dtype == kF16 ? LpVec<__half>::pack(f) : LpVec<__nv_bfloat16>::pack(f);
    }
  }
}

cudaError_t launch_seed_read_copy(const float *ckpt, int64_t n_rows, int d_k, int lp_dtype, void *ckpt_lp, float *scale,
                                  cudaStream_t s) {
  seed_read_copy_kernel<<<(unsigned)((n_rows + 7) / 8), 256, 0, s>>>(ckpt, n_rows, d_k, lp_dtype, ckpt_lp, scale);
  return cudaGetLastError();
}

template <int DV, int DK, typename TC, int NT, int NSPLIT = 1>
static cudaError_t launch_mat(const rs_materialize_args &a, int gdn, cudaStream_t s) {
  materialize_kernel<DV, DK, TC, NT, NSPLIT><<<(unsigned)((size_t)a.B * a.H * NSPLIT), NT, 0, s>>>(a, gdn);
  return cudaGetLastError();
}

MatLaunchFn find_materialize(int d_v, int d_k, int ckpt_dtype) {
  if (ckpt_dtype == kF32) {
    if (d_v == 16 && d_k == 32) return launch_mat<16, 32, float, 128>;
    if (d_v == 64 && d_k == 128) return launch_mat<64, 128, float, 256>;
    if (d_v == 128 && d_k == 128) return launch_mat<128, 128, float, 256, 2>;
  } else if (ckpt_dtype == kF16) {
    if (d_v == 16 && d_k == 32) return launch_mat<16, 32, __half, 64>;
    if (d_v == 64 && d_k == 128) return launch_mat<64, 128, __half, 256>;
    if (d_v == 128 && d_k == 128) return launch_mat<128, 128, __half, 256>;
  }
  return nullptr;
}

}  // namespace rs
