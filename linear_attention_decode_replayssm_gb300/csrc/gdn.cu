// ReplaySSM Gated DeltaNet cached decode step: non-flush and flush rows in one launch.
//
// Sources:
//   [Ghana] S. Ghana, "ReplaySSM: an SSM decoder that writes its state once
//           every 16 tokens", §The delta-rule wrinkle: S_t = alpha_t S_{t-1}
//           + u_t k_t^T with u_t = beta_t (v_t - alpha_t S_{t-1} k_t); cache u.
//   [PR48792] vLLM PR 48792, "[Kernel] ReplaySSM: cache SSM inputs for faster
//           Gated DeltaNet standard decode": §Core concept (the ring holds the
//           key k, the corrected value d and the scalar gate g), §Paged cache
//           layout (fp16 d and k caches, fp32 g), and the review comment that
//           S_{t-1} q_t and S_{t-1} k_t both expand over the checkpoint and the
//           ring, so the output needs no rebuilt state.
//
// One CTA per (row b, head h).  With p ring records (d_j, k_j, g_j), j < p:
//   G_j = exp(sum_{l=j+1..p-1} g_l),  Gamma = exp(sum_{l<p} g_l),
//   a = S_{t-1} k_t = Gamma (S_ckpt k_t) + sum_j G_j (k_j . k_t) d_j,
//   c = S_{t-1} q_t = Gamma (S_ckpt q_t) + sum_j G_j (k_j . q_t) d_j,
//   alpha_t = exp(g_t),  d_t = beta_t (v_t - alpha_t a),
//   non-flush: o = alpha_t c + (k_t . q_t) d_t; append (d_t, k_t, g_t) with d
//              and k rounded to the ring type;
//   flush:     S_new = alpha_t (Gamma S_ckpt + sum_j G_j d_j k_j^T) + d_t k_t^T
//              with the unrounded d_t, o = S_new q_t, S_new stored.
// One streaming pass over the checkpoint yields S_ckpt k_t and S_ckpt q_t
// together: both partial-dot sets go through one transposed group reduction.
#include "common.cuh"
#include "launch.h"

namespace rs {

template <int DV, int DK, typename TC, int NT, int MINB>
__global__ void __launch_bounds__(NT, MINB) gdn_replay_kernel(const KArgs a) {
  using V = CkVec<TC>;
  constexpr int E = V::E;
  constexpr int G = DK / E;
  constexpr int RPP = NT / G;
  constexpr int VPT = DV / RPP;
  constexpr int NW = NT / 32;
  static_assert(G <= 32 && 32 % G == 0, "a state row must fit in one warp");
  static_assert(NT % G == 0 && DV % RPP == 0 && VPT >= 1 && 2 * VPT <= G, "bad tiling");
  static_assert(DK % 8 == 0 && DV % 8 == 0, "head dims must be multiples of 8");

  const int L = a.L;
  extern __shared__ float smem[];
  float *sQ = smem;            // [DK] q_t
  float *sK = sQ + DK;         // [L][DK] keys: records 0..p-1, current k_t at p
  float *sD = sK + L * DK;     // [L][DV] corrected values; d_t at p (flush)
  float *sVt = sD + L * DV;    // [DV] v_t
  float *sG = sVt + DV;        // [L] log-gates of records
  float *sW = sG + L;          // [L] G_j
  float *sDk = sW + L;         // [L] k_j . k_t
  float *sDq = sDk + L;        // [L] k_j . q_t
  float *sAk = sDq + L;        // [DV] S_ckpt k_t
  float *sAq = sAk + DV;       // [DV] S_ckpt q_t
  float *sC = sAq + DV;        // [DV] flush output
  float *sScal = sC + DV;      // [0] Gamma, [1] k_t . q_t

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.H;
  const int h = blockIdx.x - b * a.H;
  float *orow = a.out + (size_t)b * a.so + (size_t)h * DV;

  const int slot = __ldg(a.slot_idx + b);
  if (slot < 0) {
    for (int i = tid; i < DV; i += NT) orow[i] = 0.f;
    return;
  }
  const int p = __ldg(a.write_pos + b);
  const bool flush = __ldg(a.is_flush + b) != 0;
  if (slot >= a.num_slots || p < 0 || p >= L) {
    if (tid == 0) report(a.dev_err, slot >= a.num_slots ? 1 : 2);
    for (int i = tid; i < DV; i += NT) orow[i] = 0.f;
    return;
  }
  const size_t unit = (size_t)slot * a.H + h;
  TC *ck = static_cast<TC *>(a.ckpt) + unit * (size_t)(DV * DK);
  const int row0 = tid / G, cv = tid - (tid / G) * G;

  uint4 raw[VPT];
#pragma unroll
  for (int r = 0; r < VPT; ++r) raw[r] = ld_stream(ck + (size_t)(row0 + r * RPP) * DK + cv * E);

  // stage the ring records and the current token; append k_t and g_t now
  const size_t ring_rec = unit * (size_t)L;
  const int n = p + 1;
  for (int idx = tid; idx < n * (DK / 8); idx += NT) {
    const int j = idx / (DK / 8), c = (idx - j * (DK / 8)) * 8;
    float f[8];
    if (j < p) {
      load8(a.ring_k, (ring_rec + j) * DK + c, a.ring_dtype, f);
    } else {
      load8(a.k, (size_t)b * a.sk + (size_t)h * DK + c, a.in_dtype, f);
      if (!flush) store8(a.ring_k, (ring_rec + p) * DK + c, a.ring_dtype, f);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sK[j * DK + c + e] = f[e];
  }
  for (int idx = tid; idx < p * (DV / 8); idx += NT) {
    const int j = idx / (DV / 8), c = (idx - j * (DV / 8)) * 8;
    float f[8];
    load8(a.ring_v, (ring_rec + j) * DV + c, a.ring_dtype, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) sD[j * DV + c + e] = f[e];
  }
  for (int idx = tid; idx < DV / 8; idx += NT) {
    float f[8];
    load8(a.v, (size_t)b * a.sv + (size_t)h * DV + idx * 8, a.in_dtype, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) sVt[idx * 8 + e] = f[e];
  }
  for (int idx = tid; idx < DK / 8; idx += NT) {
    float f[8];
    load8(a.q, (size_t)b * a.sq + (size_t)h * DK + idx * 8, a.in_dtype, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) sQ[idx * 8 + e] = f[e];
  }
  for (int j = tid; j < p; j += NT) sG[j] = __ldg(a.ring_a + ring_rec + j);
  const float g_t = __ldg(a.alpha + (size_t)b * a.H + h);
  const float beta_t = __ldg(a.beta + (size_t)b * a.H + h);
  if (!flush && tid == 0) a.ring_a[ring_rec + p] = g_t;
  __syncthreads();

  // decay weights over the p held records (warp 0); dot products (all warps)
  if (warp == 0) {
    float x0 = lane < p ? sG[lane] : 0.f;
    float x1 = lane + 32 < p ? sG[lane + 32] : 0.f;
    suffix_scan64(x0, x1, lane, [](float u, float w) { return u + w; });
    const float n0 = __shfl_down_sync(0xffffffffu, x0, 1);
    const float n1 = __shfl_down_sync(0xffffffffu, x1, 1);
    const float hi0 = __shfl_sync(0xffffffffu, x1, 0);
    const float e0 = lane == 31 ? hi0 : n0;
    const float e1 = lane == 31 ? 0.f : n1;
    if (lane < p) sW[lane] = expf(e0);
    if (lane + 32 < p) sW[lane + 32] = expf(e1);
    if (lane == 0) sScal[0] = expf(x0);
  }
  for (int j = warp; j <= p; j += NW) {  // j == p gives k_t . q_t
    float sk = 0.f, sq = 0.f;
    for (int c = lane; c < DK; c += 32) {
      const float kj = sK[j * DK + c];
      sk = fmaf(kj, sK[p * DK + c], sk);
      sq = fmaf(kj, sQ[c], sq);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      sk += __shfl_xor_sync(0xffffffffu, sk, off);
      sq += __shfl_xor_sync(0xffffffffu, sq, off);
    }
    if (lane == 0) {
      if (j < p) {
        sDk[j] = sk;
        sDq[j] = sq;
      } else {
        sScal[1] = sq;
      }
    }
  }

  // S_ckpt k_t and S_ckpt q_t from the registers: 2 * VPT partials per lane
  float part[2 * VPT];
  {
    float kt[E], qt[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      kt[e] = sK[p * DK + cv * E + e];
      qt[e] = sQ[cv * E + e];
    }
#pragma unroll
    for (int r = 0; r < VPT; ++r) {
      float f[E];
      V::unpack(raw[r], f);
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        s0 = fmaf(f[e], kt[e], s0);
        s1 = fmaf(f[e], qt[e], s1);
      }
      part[r] = s0;
      part[VPT + r] = s1;
    }
  }
  group_reduce<2 * VPT, G>(part, lane);
  if (group_reduce_writer<2 * VPT, G>(lane)) {
    const int vi = group_reduce_index<2 * VPT, G>(lane);
    if (vi < VPT)
      sAk[row0 + vi * RPP] = part[0];
    else
      sAq[row0 + (vi - VPT) * RPP] = part[0];
  }
  __syncthreads();

  // per value row: rebuild S_{t-1} k_t and S_{t-1} q_t, then d_t
  const float alpha_t = expf(g_t);
  const float Gam = sScal[0];
  for (int i = tid; i < DV; i += NT) {
    float ak = Gam * sAk[i], aq = Gam * sAq[i];
    for (int j = 0; j < p; ++j) {
      const float dj = sW[j] * sD[j * DV + i];
      ak = fmaf(sDk[j], dj, ak);
      aq = fmaf(sDq[j], dj, aq);
    }
    const float d_t = beta_t * (sVt[i] - alpha_t * ak);
    if (!flush) {
      orow[i] = fmaf(alpha_t, aq, d_t * sScal[1]);
      store1(a.ring_v, (ring_rec + p) * DV + i, a.ring_dtype, d_t);
    } else {
      sD[p * DV + i] = d_t;
    }
  }
  if (!flush) return;
  __syncthreads();

  // flush: S_new = alpha_t (Gamma S_ckpt + sum_j G_j d_j k_j^T) + d_t k_t^T
  {
    float f[VPT][E];
    const float scale0 = alpha_t * Gam;
#pragma unroll
    for (int r = 0; r < VPT; ++r) {
      V::unpack(raw[r], f[r]);
#pragma unroll
      for (int e = 0; e < E; ++e) f[r][e] *= scale0;
    }
    for (int j = 0; j <= p; ++j) {
      float kk[E];
#pragma unroll
      for (int e = 0; e < E; ++e) kk[e] = sK[j * DK + cv * E + e];
      const float wj = j < p ? alpha_t * sW[j] : 1.f;
#pragma unroll
      for (int r = 0; r < VPT; ++r) {
        const float dd = wj * sD[j * DV + row0 + r * RPP];
#pragma unroll
        for (int e = 0; e < E; ++e) f[r][e] = fmaf(dd, kk[e], f[r][e]);
      }
    }
    float qv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) qv[e] = sQ[cv * E + e];
    float po[VPT];
#pragma unroll
    for (int r = 0; r < VPT; ++r) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) s = fmaf(f[r][e], qv[e], s);
      po[r] = s;
      st_vec(ck + (size_t)(row0 + r * RPP) * DK + cv * E, V::pack(f[r]));
    }
    group_reduce<VPT, G>(po, lane);
    if (group_reduce_writer<VPT, G>(lane)) sC[row0 + group_reduce_index<VPT, G>(lane) * RPP] = po[0];
  }
  __syncthreads();
  for (int i = tid; i < DV; i += NT) orow[i] = sC[i];
}

template <int DV, int DK>
static size_t gdn_smem(int L) {
  return sizeof(float) * (size_t)(DK + L * (DK + DV) + DV + 4 * L + 3 * DV + 4);
}

template <int DV, int DK, typename TC, int NT, int MINB = 1>
static cudaError_t launch_gdn(const KArgs &a, cudaStream_t s) {
  auto kern = gdn_replay_kernel<DV, DK, TC, NT, MINB>;
  const size_t smem = gdn_smem<DV, DK>(a.L);
  cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)((size_t)a.B * a.H), NT, smem, s>>>(a);
  return cudaGetLastError();
}

LaunchFn find_gdn(int d_v, int d_k, int ckpt_dtype) {
  if (ckpt_dtype == kF32) {
    if (d_v == 16 && d_k == 32) return launch_gdn<16, 32, float, 128>;
    if (d_v == 64 && d_k == 128) return launch_gdn<64, 128, float, 256>;
    if (d_v == 128 && d_k == 128) return launch_gdn<128, 128, float, 512, 2>;
  } else if (ckpt_dtype == kF16) {
    if (d_v == 16 && d_k == 32) return launch_gdn<16, 32, __half, 64>;
    if (d_v == 64 && d_k == 128) return launch_gdn<64, 128, __half, 256>;
    if (d_v == 128 && d_k == 128) return launch_gdn<128, 128, __half, 256>;
  }
  return nullptr;
}

}  // namespace rs
