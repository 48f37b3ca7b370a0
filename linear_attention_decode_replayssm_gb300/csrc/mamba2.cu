// ReplaySSM Mamba-2 cached decode step: non-flush and flush rows in one launch.
//
// Sources:
//   [Ghana] S. Ghana, "ReplaySSM: an SSM decoder that writes its state once
//           every 16 tokens", §The identity and §Output without a state.
//   [PR48792] vLLM PR 48792, "[Kernel] ReplaySSM: cache SSM inputs for faster
//           Gated DeltaNet standard decode", §CUDA graphs and continuous
//           batching (the flush flag is per-row runtime data).
//
// One CTA per (row b, head h).  With p = write_pos[b] ring records held and the
// current token as record p (0-based), w_j = prod_{l=j+1..p} alpha_l and
// gamma = prod_{l=0..p} alpha_l:
//   non-flush: o = gamma * (S_ckpt q) + sum_{j<=p} w_j (k_j . q) v_j, and the
//              record (alpha, v, k) is copied into ring slot p;
//   flush:     S_new = gamma * S_ckpt + sum_{j<=p} w_j v_j k_j^T, o = S_new q
//              from the fp32 registers, S_new stored (cast) over S_ckpt.
// The checkpoint is the only large operand: it streams from HBM once per step
// with 128-bit loads issued before anything else, while the <= L records are
// staged in shared memory as fp32.  Dot products are warp reductions; the
// decay weights are a warp suffix scan.  No tensor cores: the step is a
// bandwidth-bound GEMV (about 0.6 FLOP per byte).
#include "common.cuh"
#include "launch.h"

namespace rs {

template <int DV, int DK, typename TC, int NT, int MINB>
__global__ void __launch_bounds__(NT, MINB) mamba2_replay_kernel(const KArgs a) {
  using V = CkVec<TC>;
  constexpr int E = V::E;
  constexpr int G = DK / E;    // lanes per state row
  constexpr int RPP = NT / G;  // rows covered by one pass of the CTA
  constexpr int VPT = DV / RPP;
  constexpr int NW = NT / 32;
  static_assert(G <= 32 && 32 % G == 0, "a state row must fit in one warp");
  static_assert(NT % G == 0 && DV % RPP == 0 && VPT >= 1 && VPT <= G, "bad tiling");
  static_assert(DK % 8 == 0 && DV % 8 == 0, "head dims must be multiples of 8");

  const int L = a.L;
  extern __shared__ float smem[];
  float *sQ = smem;             // [DK]
  float *sK = sQ + DK;          // [L][DK] keys of records 0..p (p = current)
  float *sV = sK + L * DK;      // [L][DV] values
  float *sA = sV + L * DV;      // [L] decays
  float *sW = sA + L;           // [L] window weights w_j
  float *sS = sW + L;           // [L] k_j . q
  float *sC = sS + L;           // [DV] row results
  float *sGam = sC + DV;        // [1] gamma

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.H;
  const int h = blockIdx.x - b * a.H;
  float *orow = a.out + (size_t)b * a.so + (size_t)h * DV;

  const int slot = __ldg(a.slot_idx + b);
  if (slot < 0) {  // padded row
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

  // 1) the checkpoint: every load in flight before any other work
  uint4 raw[VPT];
#pragma unroll
  for (int r = 0; r < VPT; ++r) raw[r] = ld_stream(ck + (size_t)(row0 + r * RPP) * DK + cv * E);

  // 2) stage records 0..p-1 from the ring and the current token as record p;
  //    a non-flush row also appends the current record at ring slot p
  const int n = p + 1;
  const size_t ring_rec = unit * (size_t)L;
  for (int idx = tid; idx < n * (DK / 8); idx += NT) {
    const int j = idx / (DK / 8), c = (idx - j * (DK / 8)) * 8;
    float f[8];
    if (j < p) {
      load8(a.ring_k, (ring_rec + j) * DK + c, a.ring_dtype, f);
    } else {
      const size_t off = (size_t)b * a.sk + (size_t)h * DK + c;
      load8(a.k, off, a.in_dtype, f);
      if (!flush) copy8(a.ring_k, (ring_rec + p) * DK + c, a.k, off, a.in_dtype);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sK[j * DK + c + e] = f[e];
  }
  for (int idx = tid; idx < n * (DV / 8); idx += NT) {
    const int j = idx / (DV / 8), c = (idx - j * (DV / 8)) * 8;
    float f[8];
    if (j < p) {
      load8(a.ring_v, (ring_rec + j) * DV + c, a.ring_dtype, f);
    } else {
      const size_t off = (size_t)b * a.sv + (size_t)h * DV + c;
      load8(a.v, off, a.in_dtype, f);
      if (!flush) copy8(a.ring_v, (ring_rec + p) * DV + c, a.v, off, a.in_dtype);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sV[j * DV + c + e] = f[e];
  }
  for (int idx = tid; idx < DK / 8; idx += NT) {
    float f[8];
    load8(a.q, (size_t)b * a.sq + (size_t)h * DK + idx * 8, a.in_dtype, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) sQ[idx * 8 + e] = f[e];
  }
  for (int j = tid; j < n; j += NT) {
    float al;
    if (j < p) {
      al = __ldg(a.ring_a + ring_rec + j);
    } else {
      al = __ldg(a.alpha + (size_t)b * a.H + h);
      if (!flush) a.ring_a[ring_rec + p] = al;
    }
    sA[j] = al;
  }
  __syncthreads();

  // 3) window weights (warp 0) and, for non-flush rows, k_j . q (all warps)
  if (warp == 0) {
    float x0 = lane <= p ? sA[lane] : 1.f;
    float x1 = lane + 32 <= p ? sA[lane + 32] : 1.f;
    suffix_scan64(x0, x1, lane, [](float u, float w) { return u * w; });
    // exclusive suffix product: w_j = incl[j + 1]
    const float n0 = __shfl_down_sync(0xffffffffu, x0, 1);
    const float n1 = __shfl_down_sync(0xffffffffu, x1, 1);
    const float hi0 = __shfl_sync(0xffffffffu, x1, 0);
    const float w0 = lane == 31 ? hi0 : n0;
    const float w1 = lane == 31 ? 1.f : n1;
    if (lane <= p) sW[lane] = w0;
    if (lane + 32 <= p) sW[lane + 32] = w1;
    if (lane == 0) sGam[0] = x0;
  }
  if (!flush) {
    for (int j = warp; j <= p; j += NW) {
      float s = 0.f;
#pragma unroll
      for (int c = lane; c < DK; c += 32) s += sK[j * DK + c] * sQ[c];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (lane == 0) sS[j] = s;
    }
  }
  __syncthreads();

  float qv[E];
#pragma unroll
  for (int e = 0; e < E; ++e) qv[e] = sQ[cv * E + e];

  float part[VPT];
  if (!flush) {
    // 4a) checkpoint GEMV: partial row dots, reduced across the G lanes of a row
#pragma unroll
    for (int r = 0; r < VPT; ++r) {
      float f[E];
      V::unpack(raw[r], f);
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) s = fmaf(f[e], qv[e], s);
      part[r] = s;
    }
  } else {
    // 4b) flush: fold the window into the state in registers
    const float gam = sGam[0];
    float f[VPT][E];
#pragma unroll
    for (int r = 0; r < VPT; ++r) {
      V::unpack(raw[r], f[r]);
#pragma unroll
      for (int e = 0; e < E; ++e) f[r][e] *= gam;
    }
    for (int j = 0; j <= p; ++j) {
      float kk[E];
#pragma unroll
      for (int e = 0; e < E; ++e) kk[e] = sK[j * DK + cv * E + e];
      const float wj = sW[j];
#pragma unroll
      for (int r = 0; r < VPT; ++r) {
        const float vv = wj * sV[j * DV + row0 + r * RPP];
#pragma unroll
        for (int e = 0; e < E; ++e) f[r][e] = fmaf(vv, kk[e], f[r][e]);
      }
    }
#pragma unroll
    for (int r = 0; r < VPT; ++r) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) s = fmaf(f[r][e], qv[e], s);
      part[r] = s;
      st_vec(ck + (size_t)(row0 + r * RPP) * DK + cv * E, V::pack(f[r]));
    }
  }
  group_reduce<VPT, G>(part, lane);
  if (group_reduce_writer<VPT, G>(lane)) sC[row0 + group_reduce_index<VPT, G>(lane) * RPP] = part[0];
  __syncthreads();

  // 5) output row
  if (!flush) {
    const float gam = sGam[0];
    for (int i = tid; i < DV; i += NT) {
      float acc = gam * sC[i];
      for (int j = 0; j <= p; ++j) acc = fmaf(sW[j] * sS[j], sV[j * DV + i], acc);
      orow[i] = acc;
    }
  } else {
    for (int i = tid; i < DV; i += NT) orow[i] = sC[i];
  }
}

template <int DV, int DK>
static size_t mamba2_smem(int L) {
  return sizeof(float) * (size_t)(DK + L * (DK + DV) + 3 * L + DV + 4);
}

template <int DV, int DK, typename TC, int NT, int MINB = 1>
static cudaError_t launch_mamba2(const KArgs &a, cudaStream_t s) {
  auto kern = mamba2_replay_kernel<DV, DK, TC, NT, MINB>;
  const size_t smem = mamba2_smem<DV, DK>(a.L);
  cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)((size_t)a.B * a.H), NT, smem, s>>>(a);
  return cudaGetLastError();
}

LaunchFn find_mamba2(int d_v, int d_k, int ckpt_dtype) {
  if (ckpt_dtype == kF32) {
    if (d_v == 16 && d_k == 32) return launch_mamba2<16, 32, float, 128>;
    if (d_v == 64 && d_k == 128) return launch_mamba2<64, 128, float, 256>;
    if (d_v == 128 && d_k == 128) return launch_mamba2<128, 128, float, 512>;
  } else if (ckpt_dtype == kF16) {
    if (d_v == 16 && d_k == 32) return launch_mamba2<16, 32, __half, 64>;
    if (d_v == 64 && d_k == 128) return launch_mamba2<64, 128, __half, 256>;
    if (d_v == 128 && d_k == 128) return launch_mamba2<128, 128, __half, 256>;
  }
  return nullptr;
}

}  // namespace rs
