// ReplaySSM speculative verification for Mamba-2, and the on-device commit.
//
// Sources:
//   [Ghana] S. Ghana, "ReplaySSM: an SSM decoder that writes its state once
//           every 16 tokens", §Speculative decoding: rollback becomes a
//           pointer (T drafts appended behind the h committed records, all T
//           outputs without a state, commit by advancing the pointer, flush
//           of the committed records when h + T > L, decided on the device).
//   [NV]    NVIDIA technical blog, "ReplaySSM: Rethinking State Storage for
//           Faster Hybrid Model Decoding", §Benefit 2 (output-only
//           evaluation: the checkpoint is read once for all T queries, the
//           rest is products over cached keys, cached values and the draft
//           queries, with D the cumulative decays of the draft positions and
//           W a causally masked matrix of decays).
//
// One CTA per (row, head).  With nb committed records ahead of the drafts
// (nb = h, or 0 on a flush step, whose committed records are first folded
// into the checkpoint) and the records r_0 .. r_{nb+T-1} (committed, then
// drafts), draft i's output is
//   o_i = D_i (S q_i) + sum_{j <= nb+i} W_{j,i} (k_j . q_i) v_j,
//   D_i = prod_{l <= nb+i} alpha_l,  W_{j,i} = prod_{j < l <= nb+i} alpha_l,
// with S the checkpoint (non-flush) or the unrounded folded state (flush).
// The drafts' records go to ring slots nb .. nb+T-1.
#include "common.cuh"
#include "launch.h"

namespace rs {

struct SpecLayout {
  uint32_t k, v, q, a, w, d, wf, s, c, bytes;
};

// records: up to L committed + T drafts, in the ring type
__host__ __device__ inline SpecLayout spec_layout(int DV, int DK, int res, int L, int T) {
  SpecLayout o;
  uint32_t x = 0;
  const int R = L + T;
  o.k = x;  x = align128(x + R * DK * res);
  o.v = x;  x = align128(x + R * DV * res);
  o.q = x;  x = align128(x + T * DK * 4);
  o.a = x;  x = align128(x + R * 4);
  o.w = x;  x = align128(x + T * 64 * 4);   // W_{j,i}, [i][j]
  o.d = x;  x = align128(x + T * 4);        // D_i
  o.wf = x; x = align128(x + 65 * 4);       // fold weights and gamma
  o.s = x;  x = align128(x + R * T * 4);    // W_{j,i} (k_j . q_i), [j][i]
  o.c = x;  x = align128(x + T * DV * 4);   // S q_i
  o.bytes = x;
  return o;
}

template <int DV, int DK, typename TC, typename RT, int NT>
__global__ void __launch_bounds__(NT) spec_verify_kernel(const rs_spec_args a) {
  using V = CkVec<TC>;
  constexpr int E = V::E;
  constexpr int G = DK / E;
  constexpr int RPP = NT / G;
  constexpr int VPT = DV / RPP;
  constexpr int NW = NT / 32;
  constexpr int RES = (int)sizeof(RT);
  constexpr int RDT = Rec<RT>::kDtype;
  static_assert(G <= 32 && 32 % G == 0 && NT % G == 0 && DV % RPP == 0 && VPT >= 1, "bad tiling");
  static_assert(DK % 128 == 0 || DK <= 128, "key chunks");

  extern __shared__ __align__(128) unsigned char smem[];
  const int T = a.T, L = a.L;
  const SpecLayout lay = spec_layout(DV, DK, RES, L, T);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.H, h = blockIdx.x - (blockIdx.x / a.H) * a.H;
  const int slot = __ldg(a.slot_idx + b);
  float *out0 = a.out + ((size_t)b * T * a.H + h) * DV;  // draft i at + i * H * DV
  const size_t ostride = (size_t)a.H * DV;
  if (slot < 0) {
    for (int x = tid; x < T * DV; x += NT) out0[(x / DV) * ostride + x % DV] = 0.f;
    return;
  }
  const int hc = __ldg(a.committed + b);
  const bool flush = __ldg(a.is_flush + b) != 0;
  const int bad = (slot >= a.num_slots ? RS_DERR_SLOT : 0) |
                  ((hc < 0 || hc > L || (!flush && hc + T > L)) ? RS_DERR_WRITE_POS : 0);
  if (bad) {
    if (tid == 0) report(a.dev_err, bad);
    for (int x = tid; x < T * DV; x += NT) out0[(x / DV) * ostride + x % DV] = 0.f;
    return;
  }
  const size_t unit = (size_t)slot * a.H + h;
  TC *ck = static_cast<TC *>(a.ckpt) + unit * (size_t)(DV * DK);
  const int row0 = tid / G, cv = tid - (tid / G) * G;

  uint4 raw[VPT];
#pragma unroll
  for (int r = 0; r < VPT; ++r) raw[r] = ld_stream(ck + (size_t)(row0 + r * RPP) * DK + cv * E);

  // stage the records: hc committed ones from the ring, then the T drafts
  unsigned char *sk = smem + lay.k, *sv = smem + lay.v;
  float *sq = reinterpret_cast<float *>(smem + lay.q), *sa = reinterpret_cast<float *>(smem + lay.a);
  float *sW = reinterpret_cast<float *>(smem + lay.w), *sD = reinterpret_cast<float *>(smem + lay.d);
  float *sWf = reinterpret_cast<float *>(smem + lay.wf), *sS = reinterpret_cast<float *>(smem + lay.s);
  float *sC = reinterpret_cast<float *>(smem + lay.c);
  {
    constexpr int KC = DK * RES / 16, VC = DV * RES / 16;
    const uint4 *rk = reinterpret_cast<const uint4 *>(static_cast<const unsigned char *>(a.ring_k) + unit * L * DK * RES);
    const uint4 *rv = reinterpret_cast<const uint4 *>(static_cast<const unsigned char *>(a.ring_v) + unit * L * DV * RES);
    for (int x = tid; x < hc * KC; x += NT) reinterpret_cast<uint4 *>(sk)[x] = __ldg(rk + x);
    for (int x = tid; x < hc * VC; x += NT) reinterpret_cast<uint4 *>(sv)[x] = __ldg(rv + x);
    for (int x = tid; x < T * KC; x += NT) {
      const int i = x / KC, c = x - i * KC;
      const unsigned char *src = static_cast<const unsigned char *>(a.k) + (((size_t)b * T + i) * a.H + h) * DK * RES;
      reinterpret_cast<uint4 *>(sk + (size_t)(hc + i) * DK * RES)[c] = __ldg(reinterpret_cast<const uint4 *>(src) + c);
    }
    for (int x = tid; x < T * VC; x += NT) {
      const int i = x / VC, c = x - i * VC;
      const unsigned char *src = static_cast<const unsigned char *>(a.v) + (((size_t)b * T + i) * a.H + h) * DV * RES;
      reinterpret_cast<uint4 *>(sv + (size_t)(hc + i) * DV * RES)[c] = __ldg(reinterpret_cast<const uint4 *>(src) + c);
    }
    for (int x = tid; x < T * (DK / 8); x += NT) {
      const int i = x / (DK / 8), c = x - i * (DK / 8);
      float f[8];
      load8(a.q, (((size_t)b * T + i) * a.H + h) * DK + c * 8, a.in_dtype, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sq[i * DK + c * 8 + e] = f[e];
    }
    for (int x = tid; x < hc; x += NT) sa[x] = __ldg(a.ring_a + unit * L + x);
    for (int x = tid; x < T; x += NT) sa[hc + x] = __ldg(a.alpha + ((size_t)b * T + x) * a.H + h);
  }
  __syncthreads();

  // window weights.  Records of the outputs start at r0 (the drafts only on a
  // flush step); draft i's window is r0 .. r0+nb+i.
  const int nb = flush ? 0 : hc, r0 = flush ? hc : 0;
  for (int i = warp; i < T; i += NW) {
    const int n = nb + i + 1;  // entries of draft i's window (<= 64)
    float x0 = lane < n ? sa[r0 + lane] : 1.f;
    float x1 = lane + 32 < n ? sa[r0 + lane + 32] : 1.f;
    suffix_scan64(x0, x1, lane, [](float x, float y) { return x * y; });
    const float n0 = __shfl_down_sync(0xffffffffu, x0, 1);
    const float n1 = __shfl_down_sync(0xffffffffu, x1, 1);
    const float hi0 = __shfl_sync(0xffffffffu, x1, 0);
    sW[i * 64 + lane] = lane == 31 ? hi0 : n0;       // W_{j,i} = product of the decays after j
    sW[i * 64 + lane + 32] = lane == 31 ? 1.f : n1;
    if (lane == 0) sD[i] = x0;
  }
  if (flush && warp == NW - 1) {
    // fold weights of the hc committed records and their total decay
    float x0 = lane < hc ? sa[lane] : 1.f;
    float x1 = lane + 32 < hc ? sa[lane + 32] : 1.f;
    suffix_scan64(x0, x1, lane, [](float x, float y) { return x * y; });
    const float n0 = __shfl_down_sync(0xffffffffu, x0, 1);
    const float n1 = __shfl_down_sync(0xffffffffu, x1, 1);
    const float hi0 = __shfl_sync(0xffffffffu, x1, 0);
    sWf[lane] = lane == 31 ? hi0 : n0;
    sWf[lane + 32] = lane == 31 ? 1.f : n1;
    if (lane == 0) sWf[64] = x0;
  }
  // s_{j,i} = k_j . q_i over the records of the outputs: a warp takes a
  // record, a lane four key columns per 128
  for (int j = warp; j < nb + T; j += NW) {
    constexpr int KPL = DK >= 128 ? DK / 128 : 1;  // 4-column chunks per lane
    float part[16];
    float kk[4 * KPL];
#pragma unroll
    for (int c = 0; c < KPL; ++c) {
      if (lane * 4 + c * 128 < DK) {
        float t4[4];
        lds_cols<4>(sk, (r0 + j) * DK + lane * 4 + c * 128, RDT, t4);
        kk[4 * c] = t4[0]; kk[4 * c + 1] = t4[1]; kk[4 * c + 2] = t4[2]; kk[4 * c + 3] = t4[3];
      } else {
        kk[4 * c] = kk[4 * c + 1] = kk[4 * c + 2] = kk[4 * c + 3] = 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = 0.f;
      if (i < T) {
#pragma unroll
        for (int c = 0; c < KPL; ++c) {
          const int col = lane * 4 + c * 128;
          if (col < DK) {
            const float4 q4 = *reinterpret_cast<const float4 *>(sq + i * DK + col);
            acc = fmaf(kk[4 * c], q4.x, fmaf(kk[4 * c + 1], q4.y, fmaf(kk[4 * c + 2], q4.z, fmaf(kk[4 * c + 3], q4.w, acc))));
          }
        }
      }
      part[i] = acc;
    }
    group_reduce<16, 32>(part, lane);
    if (group_reduce_writer<16, 32>(lane)) {
      const int i = group_reduce_index<16, 32>(lane);
      if (i < T) sS[j * T + i] = part[0];
    }
  }
  __syncthreads();
  // coefficients W_{j,i} s_{j,i}, causally masked
  for (int x = tid; x < (nb + T) * T; x += NT) {
    const int j = x / T, i = x - j * T;
    sS[x] = j <= nb + i ? sW[i * 64 + j] * sS[x] : 0.f;
  }

  // the state the outputs run from: the checkpoint, or on a flush the fold
  // gamma S_ckpt + sum_j w_j v_j k_j^T of the committed records, stored
  float f[VPT][E];
#pragma unroll
  for (int r = 0; r < VPT; ++r) V::unpack(raw[r], f[r]);
  if (flush) {
    const float gam = sWf[64];
#pragma unroll
    for (int r = 0; r < VPT; ++r)
#pragma unroll
      for (int e = 0; e < E; ++e) f[r][e] *= gam;
    for (int j = 0; j < hc; ++j) {
      float kk[E];
      lds_cols<E>(sk, j * DK + cv * E, RDT, kk);
      const float wj = sWf[j];
#pragma unroll
      for (int r = 0; r < VPT; ++r) {
        const float vv = wj * lds_elem(sv, j * DV + row0 + r * RPP, RDT);
#pragma unroll
        for (int e = 0; e < E; ++e) f[r][e] = fmaf(vv, kk[e], f[r][e]);
      }
    }
#pragma unroll
    for (int r = 0; r < VPT; ++r) st_vec(ck + (size_t)(row0 + r * RPP) * DK + cv * E, V::pack(f[r]));
  }
  // c_i = S q_i for every draft
  for (int i = 0; i < T; ++i) {
    float qv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) qv[e] = sq[i * DK + cv * E + e];
    float part[VPT];
#pragma unroll
    for (int r = 0; r < VPT; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc = fmaf(f[r][e], qv[e], acc);
      part[r] = acc;
    }
    group_reduce<VPT, G>(part, lane);
    if (group_reduce_writer<VPT, G>(lane)) sC[i * DV + row0 + group_reduce_index<VPT, G>(lane) * RPP] = part[0];
  }
  __syncthreads();

  // o_i = D_i c_i + sum_j W_{j,i} s_{j,i} v_j
  for (int x = tid; x < T * DV; x += NT) {
    const int i = x / DV, r = x - i * DV;
    float acc = sD[i] * sC[x];
    for (int j = 0; j <= nb + i; ++j) acc = fmaf(sS[j * T + i], lds_elem(sv, (r0 + j) * DV + r, RDT), acc);
    out0[i * ostride + r] = acc;
  }
  // the drafts' records go to ring slots nb .. nb+T-1
  {
    constexpr int KC = DK * RES / 16, VC = DV * RES / 16;
    uint4 *rk = reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.ring_k) + (unit * L + nb) * DK * RES);
    uint4 *rv = reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.ring_v) + (unit * L + nb) * DV * RES);
    const uint4 *dk = reinterpret_cast<const uint4 *>(sk + (size_t)hc * DK * RES);
    const uint4 *dv = reinterpret_cast<const uint4 *>(sv + (size_t)hc * DV * RES);
    for (int x = tid; x < T * KC; x += NT) rk[x] = dk[x];
    for (int x = tid; x < T * VC; x += NT) rv[x] = dv[x];
    for (int x = tid; x < T; x += NT) a.ring_a[unit * L + nb + x] = sa[hc + x];
  }
}

// next step's committed count and flag, from the accepted counts
__global__ void spec_commit_kernel(const int32_t *committed, const uint8_t *is_flush, const int32_t *accepted,
                                   int B, int L, int T, int32_t *committed_out, uint8_t *is_flush_out,
                                   int32_t *dev_err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int h = committed[b];
  const bool fl = is_flush[b] != 0;
  const int acc = accepted[b];
  int h2 = fl ? 0 : h;
  if (acc >= 1 && acc <= T) {
    h2 += acc;
  } else {
    report(dev_err, RS_DERR_ACCEPTED);  // nothing of this step is committed
  }
  committed_out[b] = h2;
  is_flush_out[b] = (uint8_t)(h2 + T > L);
}

template <int DV, int DK, typename TC, typename RT, int NT>
static cudaError_t launch_spec(const rs_spec_args &a, cudaStream_t s) {
  auto kern = spec_verify_kernel<DV, DK, TC, RT, NT>;
  const size_t smem = spec_layout(DV, DK, (int)sizeof(RT), a.L, a.T).bytes;
  cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)((size_t)a.B * a.H), NT, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename RT>
static SpecLaunchFn find_spec_t(int d_v, int d_k, int ckpt_dtype) {
  if (ckpt_dtype == kF32) {
    if (d_v == 16 && d_k == 32) return launch_spec<16, 32, float, RT, 128>;
    if (d_v == 64 && d_k == 128) return launch_spec<64, 128, float, RT, 256>;
    if (d_v == 128 && d_k == 128) return launch_spec<128, 128, float, RT, 256>;
  } else if (ckpt_dtype == kF16) {
    if (d_v == 16 && d_k == 32) return launch_spec<16, 32, __half, RT, 64>;
    if (d_v == 64 && d_k == 128) return launch_spec<64, 128, __half, RT, 256>;
    if (d_v == 128 && d_k == 128) return launch_spec<128, 128, __half, RT, 256>;
  }
  return nullptr;
}

SpecLaunchFn find_spec(int d_v, int d_k, int ckpt_dtype, int in_dtype) {
  return in_dtype == kF32 ? find_spec_t<float>(d_v, d_k, ckpt_dtype)
                          : find_spec_t<__nv_bfloat16>(d_v, d_k, ckpt_dtype);
}

cudaError_t launch_spec_commit(const int32_t *committed, const uint8_t *is_flush, const int32_t *accepted, int B,
                               int L, int T, int32_t *committed_out, uint8_t *is_flush_out, int32_t *dev_err,
                               cudaStream_t s) {
  spec_commit_kernel<<<(unsigned)((B + 255) / 256), 256, 0, s>>>(committed, is_flush, accepted, B, L, T,
                                                                 committed_out, is_flush_out, dev_err);
  return cudaGetLastError();
}

}  // namespace rs
