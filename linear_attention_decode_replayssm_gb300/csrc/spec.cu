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
// A work unit is one (row, head).  With nb committed records ahead of the drafts
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

// Record slot of a unit: up to L committed + T draft records in the ring
// type, the T queries, the decays, per-unit metadata and scratch.
struct SpecRec {
  uint32_t k, v, q, qf, a, meta, w, d, wf, s, c, bytes;
};

__host__ __device__ inline SpecRec spec_rec(int DV, int DK, int res, int L, int T) {
  SpecRec o;
  uint32_t x = 0;
  const int R = L + T;
  o.k = x;    x = align128(x + R * DK * res);
  o.v = x;    x = align128(x + R * DV * res);
  o.q = x;    x = align128(x + T * DK * res);
  o.qf = x;   x = align128(x + T * DK * 4);   // the queries in fp32
  o.a = x;    x = align128(x + R * 4);
  o.meta = x; x = align128(x + 16);
  o.w = x;    x = align128(x + T * 64 * 4);   // W_{j,i}, [i][j]
  o.d = x;    x = align128(x + T * 4);        // D_i
  o.wf = x;   x = align128(x + 65 * 4);       // fold weights and gamma
  o.s = x;    x = align128(x + R * T * 4);    // W_{j,i} (k_j . q_i), [j][i]
  o.c = x;    x = align128(x + T * DV * 4);   // S q_i
  o.bytes = x;
  return o;
}

// barriers full/rec_empty[nsr], ck_empty[nsc] and the abort flag
__host__ __device__ inline uint32_t spec_head(int nsr, int nsc) { return align128(8 * (2 * nsr + nsc) + 16); }

// Persistent and warp-specialised like the decode kernel: a producer warp
// streams each unit's checkpoint (one bulk copy) and its records, queries
// and decays (per-lane cp.async) into slot rings; NCW consumer warps compute
// the unit's T outputs from them.  TMAX >= T bounds the drafts at compile
// time (the dot loops unroll over it); a consumer lane holds CPR 16-byte
// checkpoint chunks per state row (chunks cv, cv + G, ...), so the per-query
// row reductions run over G = DK / (E CPR) lanes.
template <int DV, int DK, typename TC, typename RT, int NCW, int TMAX, int CPR>
__global__ void __launch_bounds__(NCW * 32 + 32, 2) spec_verify_kernel(const rs_spec_args a, int nsr, int nsc) {
  using V = CkVec<TC>;
  constexpr int E = V::E;
  constexpr int NCH = DK / E;
  constexpr int G = NCH / CPR;
  constexpr int NC = NCW * 32;
  constexpr int RPP = NC / G;
  constexpr int VPT = DV / RPP;
  constexpr int RES = (int)sizeof(RT);
  constexpr int RDT = Rec<RT>::kDtype;
  constexpr uint32_t CKB = DV * DK * (uint32_t)sizeof(TC);
  constexpr int KC = DK * RES / 16, VC = DV * RES / 16;  // 16-byte chunks per k / v record
  static_assert(G <= 32 && 32 % G == 0 && NC % G == 0 && DV % RPP == 0 && VPT >= 1 && VPT <= G && NCH % CPR == 0,
                "bad tiling");
  static_assert(TMAX >= 1 && TMAX <= 16 && (TMAX & (TMAX - 1)) == 0, "TMAX: a power of two up to 16");
  static_assert(DK * RES % 16 == 0 && DV * RES % 16 == 0, "records must be whole 16-byte chunks");

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *rec_empty = full + nsr;
  uint64_t *ck_empty = rec_empty + nsr;
  int *s_abort = reinterpret_cast<int *>(ck_empty + nsc);
  const int T = a.T, L = a.L;
  const SpecRec lay = spec_rec(DV, DK, RES, L, T);
  unsigned char *ck_slots = smem + spec_head(nsr, nsc);
  unsigned char *rec_slots = ck_slots + (size_t)nsc * CKB;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_units = a.B * a.H;
  const int stride = gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < nsr; ++s) {
      mbar_init(&full[s], 33);
      mbar_init(&rec_empty[s], NC);
    }
    for (int c = 0; c < nsc; ++c) mbar_init(&ck_empty[c], NC);
    *s_abort = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == NCW) {
    // ----------------------------------------------------------------- producer
    const uint64_t pol_stream = policy_evict_first();
    int it = 0, ps = 0, pc = 0;
    uint32_t phs = 0, phc = 0;
    for (int u = blockIdx.x; u < n_units; u += stride) {
      const int b = u / a.H, h = u - (u / a.H) * a.H;
      if (it >= nsr || it >= nsc) {
        int w = 1;
        if (lane == 0) {
          if (it >= nsr) w = mbar_wait(&rec_empty[ps], phs ^ 1u) ? 1 : 0;
          if (w && it >= nsc) w = mbar_wait(&ck_empty[pc], phc ^ 1u) ? 1 : 0;
        }
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w || *(volatile int *)s_abort) {
          if (lane == 0) *(volatile int *)s_abort = 1;
          break;
        }
      }
      __syncwarp();
      const int slot = __ldg(a.slot_idx + b);
      const int hc = __ldg(a.committed + b);
      const int fl = __ldg(a.is_flush + b) != 0;
      const int status = slot < 0 ? kStatusPad
                         : slot >= a.num_slots ? kStatusBadSlot
                         : (hc < 0 || hc > L || (!fl && hc + T > L)) ? kStatusBadPos
                         : kStatusOk;
      unsigned char *st = rec_slots + (size_t)ps * lay.bytes;
      int *meta = reinterpret_cast<int *>(st + lay.meta);
      if (status == kStatusOk) {
        const size_t unit = (size_t)slot * a.H + h;
        if (lane == 0) {
          meta[0] = slot; meta[1] = hc; meta[2] = fl; meta[3] = status;
          mbar_expect_tx(&full[ps], CKB);
          bulk_load(ck_slots + (size_t)pc * CKB, static_cast<const TC *>(a.ckpt) + unit * (DV * DK), CKB, &full[ps],
                    pol_stream);
        }
        const unsigned char *rk = static_cast<const unsigned char *>(a.ring_k) + unit * L * DK * RES;
        const unsigned char *rv = static_cast<const unsigned char *>(a.ring_v) + unit * L * DV * RES;
        // draft i of row b, head h sits at ((b * T + i) * H + h) in the [B, T, H, d] inputs
        const size_t d0 = (size_t)b * T * a.H + h, dstep = (size_t)a.H;
        const unsigned char *kin = static_cast<const unsigned char *>(a.k);
        const unsigned char *vin = static_cast<const unsigned char *>(a.v);
        const unsigned char *qin = static_cast<const unsigned char *>(a.q);
        for (int cc = lane; cc < (hc + T) * KC; cc += 32) {
          const int j = cc / KC, x = cc - j * KC;
          const unsigned char *src = j < hc ? rk + (size_t)cc * 16 : kin + ((d0 + (j - hc) * dstep) * DK * RES + x * 16);
          cp_async16(st + lay.k + cc * 16, src);
        }
        for (int cc = lane; cc < (hc + T) * VC; cc += 32) {
          const int j = cc / VC, x = cc - j * VC;
          const unsigned char *src = j < hc ? rv + (size_t)cc * 16 : vin + ((d0 + (j - hc) * dstep) * DV * RES + x * 16);
          cp_async16(st + lay.v + cc * 16, src);
        }
        for (int cc = lane; cc < T * KC; cc += 32) {
          const int i = cc / KC, x = cc - i * KC;
          cp_async16(st + lay.q + cc * 16, qin + ((d0 + i * dstep) * DK * RES + x * 16));
        }
        float *sa = reinterpret_cast<float *>(st + lay.a);
        for (int j = lane; j < hc + T; j += 32)
          cp_async4(sa + j, j < hc ? a.ring_a + unit * L + j : a.alpha + (d0 + (j - hc) * dstep));
      } else if (lane == 0) {
        meta[0] = slot; meta[1] = hc; meta[2] = fl; meta[3] = status;
      }
      if (lane == 0) mbar_arrive(&full[ps]);
      cp_async_arrive(&full[ps]);
      ++it;
      if (++ps == nsr) {
        ps = 0;
        phs ^= 1u;
      }
      if (++pc == nsc) {
        pc = 0;
        phc ^= 1u;
      }
    }
    if (lane == 0) {
      for (int k = it > nsr ? it - nsr : 0; k < it; ++k) mbar_wait(&full[k % nsr], (uint32_t)(k / nsr) & 1u);
    }
    __syncwarp();
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int row0 = tid / G, cv = tid - (tid / G) * G;
  auto csync = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory"); };
  int s = 0, c = 0;
  uint32_t ph = 0;
  for (int u = blockIdx.x; u < n_units; u += stride) {
    const int b = u / a.H, h = u - (u / a.H) * a.H;
    if (lane == 0 && !mbar_wait(&full[s], ph)) *(volatile int *)s_abort = 1;
    csync();
    if (*(volatile int *)s_abort) break;
    const unsigned char *st = rec_slots + (size_t)s * lay.bytes;
    const int4 m = *reinterpret_cast<const int4 *>(st + lay.meta);
    const int slot = m.x, hc = m.y, flush = m.z, status = m.w;
    float *out0 = a.out + ((size_t)b * T * a.H + h) * DV;  // draft i at + i * H * DV
    const size_t ostride = (size_t)a.H * DV;
    if (status != kStatusOk) {
      for (int x = tid; x < T * DV; x += NC) out0[(x / DV) * ostride + x % DV] = 0.f;
      if (tid == 0 && status != kStatusPad) report(a.dev_err, status == kStatusBadSlot ? RS_DERR_SLOT : RS_DERR_WRITE_POS);
    } else {
      const size_t unit = (size_t)slot * a.H + h;
      uint4 raw[VPT][CPR];
      const uint4 *ck4 = reinterpret_cast<const uint4 *>(ck_slots + (size_t)c * CKB);
#pragma unroll
      for (int r = 0; r < VPT; ++r)
#pragma unroll
        for (int i = 0; i < CPR; ++i) raw[r][i] = ck4[(row0 + r * RPP) * NCH + cv + G * i];
      mbar_arrive(&ck_empty[c]);

      const unsigned char *sk = st + lay.k, *sv = st + lay.v, *sq = st + lay.q;
      float *qf = reinterpret_cast<float *>(const_cast<unsigned char *>(st) + lay.qf);
      // the queries once in fp32, for the dots and the checkpoint products
      for (int x = tid; x < T * DK / 4; x += NC) {
        float q4[4];
        lds_cols<4>(sq, x * 4, RDT, q4);
        *reinterpret_cast<float4 *>(qf + x * 4) = make_float4(q4[0], q4[1], q4[2], q4[3]);
      }
      csync();
      const float *sa = reinterpret_cast<const float *>(st + lay.a);
      float *sW = reinterpret_cast<float *>(const_cast<unsigned char *>(st) + lay.w);
      float *sD = reinterpret_cast<float *>(const_cast<unsigned char *>(st) + lay.d);
      float *sWf = reinterpret_cast<float *>(const_cast<unsigned char *>(st) + lay.wf);
      float *sS = reinterpret_cast<float *>(const_cast<unsigned char *>(st) + lay.s);
      float *sC = reinterpret_cast<float *>(const_cast<unsigned char *>(st) + lay.c);
      // records of the outputs start at r0 (the drafts only, on a flush);
      // draft i's window is r0 .. r0+nb+i
      const int nb = flush ? 0 : hc, r0 = flush ? hc : 0;
      for (int i = warp; i < T; i += NCW) {
        const int n = nb + i + 1;
        float x0 = lane < n ? sa[r0 + lane] : 1.f;
        float x1 = lane + 32 < n ? sa[r0 + lane + 32] : 1.f;
        suffix_scan64(x0, x1, lane, [](float x, float y) { return x * y; });
        const float n0 = __shfl_down_sync(0xffffffffu, x0, 1);
        const float n1 = __shfl_down_sync(0xffffffffu, x1, 1);
        const float hi0 = __shfl_sync(0xffffffffu, x1, 0);
        sW[i * 64 + lane] = lane == 31 ? hi0 : n0;
        sW[i * 64 + lane + 32] = lane == 31 ? 1.f : n1;
        if (lane == 0) sD[i] = x0;
      }
      if (flush && warp == NCW - 1) {
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
      // s_{j,i} = k_j . q_i: a warp takes a record; a lane holds four key
      // columns per 128 and the drafts' queries at them
      constexpr int KPL = DK >= 128 ? DK / 128 : 1;
      float qr[TMAX][KPL][4];
#pragma unroll
      for (int i = 0; i < TMAX; ++i)
#pragma unroll
        for (int cq = 0; cq < KPL; ++cq) {
          const int col = lane * 4 + cq * 128;
          if (i < T && col < DK) {
            const float4 q4 = *reinterpret_cast<const float4 *>(qf + i * DK + col);
            qr[i][cq][0] = q4.x; qr[i][cq][1] = q4.y; qr[i][cq][2] = q4.z; qr[i][cq][3] = q4.w;
          } else {
            qr[i][cq][0] = qr[i][cq][1] = qr[i][cq][2] = qr[i][cq][3] = 0.f;
          }
        }
      for (int j = warp; j < nb + T; j += NCW) {
        float kk[KPL][4];
#pragma unroll
        for (int cq = 0; cq < KPL; ++cq) {
          if (lane * 4 + cq * 128 < DK) {
            lds_cols<4>(sk, (r0 + j) * DK + lane * 4 + cq * 128, RDT, kk[cq]);
          } else {
            kk[cq][0] = kk[cq][1] = kk[cq][2] = kk[cq][3] = 0.f;
          }
        }
        float part[TMAX];
#pragma unroll
        for (int i = 0; i < TMAX; ++i) {
          float acc = 0.f;
#pragma unroll
          for (int cq = 0; cq < KPL; ++cq)
            acc = fmaf(kk[cq][0], qr[i][cq][0], fmaf(kk[cq][1], qr[i][cq][1],
                       fmaf(kk[cq][2], qr[i][cq][2], fmaf(kk[cq][3], qr[i][cq][3], acc))));
          part[i] = acc;
        }
        group_reduce<TMAX, 32>(part, lane);
        if (group_reduce_writer<TMAX, 32>(lane)) {
          const int i = group_reduce_index<TMAX, 32>(lane);
          if (i < T) sS[j * T + i] = part[0];
        }
      }
      csync();
      for (int x = tid; x < (nb + T) * T; x += NC) {
        const int j = x / T, i = x - j * T;
        sS[x] = j <= nb + i ? sW[i * 64 + j] * sS[x] : 0.f;
      }
      // the state the outputs run from: the checkpoint, or on a flush the
      // fold of the committed records into it, stored
      float f[VPT][CPR][E];
#pragma unroll
      for (int r = 0; r < VPT; ++r)
#pragma unroll
        for (int ci = 0; ci < CPR; ++ci) V::unpack(raw[r][ci], f[r][ci]);
      if (flush) {
        const float gam = sWf[64];
#pragma unroll
        for (int r = 0; r < VPT; ++r)
#pragma unroll
          for (int ci = 0; ci < CPR; ++ci)
#pragma unroll
            for (int e = 0; e < E; ++e) f[r][ci][e] *= gam;
        for (int j = 0; j < hc; ++j) {
          float kk[CPR][E];
#pragma unroll
          for (int ci = 0; ci < CPR; ++ci) lds_cols<E>(sk, j * DK + (cv + G * ci) * E, RDT, kk[ci]);
          const float wj = sWf[j];
#pragma unroll
          for (int r = 0; r < VPT; ++r) {
            const float vv = wj * lds_elem(sv, j * DV + row0 + r * RPP, RDT);
#pragma unroll
            for (int ci = 0; ci < CPR; ++ci)
#pragma unroll
              for (int e = 0; e < E; ++e) f[r][ci][e] = fmaf(vv, kk[ci][e], f[r][ci][e]);
          }
        }
        TC *ckg = static_cast<TC *>(a.ckpt) + unit * (DV * DK);
#pragma unroll
        for (int r = 0; r < VPT; ++r)
#pragma unroll
          for (int ci = 0; ci < CPR; ++ci)
            st_vec(ckg + (size_t)(row0 + r * RPP) * DK + (cv + G * ci) * E, V::pack(f[r][ci]));
      }
      // c_i = S q_i for every draft
      for (int i = 0; i < T; ++i) {
        float part[VPT];
#pragma unroll
        for (int r = 0; r < VPT; ++r) part[r] = 0.f;
#pragma unroll
        for (int ci = 0; ci < CPR; ++ci) {
          float qv[E];
#pragma unroll
          for (int e4 = 0; e4 < E; e4 += 4) {
            const float4 q4 = *reinterpret_cast<const float4 *>(qf + i * DK + (cv + G * ci) * E + e4);
            qv[e4] = q4.x; qv[e4 + 1] = q4.y; qv[e4 + 2] = q4.z; qv[e4 + 3] = q4.w;
          }
#pragma unroll
          for (int r = 0; r < VPT; ++r)
#pragma unroll
            for (int e = 0; e < E; ++e) part[r] = fmaf(f[r][ci][e], qv[e], part[r]);
        }
        group_reduce<VPT, G>(part, lane);
        if (group_reduce_writer<VPT, G>(lane)) sC[i * DV + row0 + group_reduce_index<VPT, G>(lane) * RPP] = part[0];
      }
      csync();
      // o_i = D_i c_i + sum_j W_{j,i} s_{j,i} v_j
      for (int x = tid; x < T * DV; x += NC) {
        const int i = x / DV, r = x - i * DV;
        float acc = sD[i] * sC[x];
        for (int j = 0; j <= nb + i; ++j) acc = fmaf(sS[j * T + i], lds_elem(sv, (r0 + j) * DV + r, RDT), acc);
        out0[i * ostride + r] = acc;
      }
      // the drafts' records go to ring slots nb .. nb+T-1
      uint4 *rkg = reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.ring_k) + (unit * L + nb) * DK * RES);
      uint4 *rvg = reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.ring_v) + (unit * L + nb) * DV * RES);
      const uint4 *dk4 = reinterpret_cast<const uint4 *>(sk + (size_t)hc * DK * RES);
      const uint4 *dv4 = reinterpret_cast<const uint4 *>(sv + (size_t)hc * DV * RES);
      for (int x = tid; x < T * KC; x += NC) rkg[x] = dk4[x];
      for (int x = tid; x < T * VC; x += NC) rvg[x] = dv4[x];
      for (int x = tid; x < T; x += NC) a.ring_a[unit * L + nb + x] = sa[hc + x];
    }
    if (status != kStatusOk) mbar_arrive(&ck_empty[c]);
    mbar_arrive(&rec_empty[s]);
    if (++s == nsr) {
      s = 0;
      ph ^= 1u;
    }
    if (++c == nsc) c = 0;
  }
  if (tid == 0 && *(volatile int *)s_abort) report(a.dev_err, kDerrTimeout);
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

template <int DV, int DK, typename TC, typename RT, int NCW, int TMAX, int CPR>
static cudaError_t launch_spec_t(const rs_spec_args &a, cudaStream_t s) {
  auto kern = spec_verify_kernel<DV, DK, TC, RT, NCW, TMAX, CPR>;
  constexpr int threads = NCW * 32 + 32;
  const size_t ckb = (size_t)DV * DK * sizeof(TC);
  const size_t rb = spec_rec(DV, DK, (int)sizeof(RT), a.L, a.T).bytes;
  RingPlan plan;
  cudaError_t e = plan_rings(reinterpret_cast<const void *>(kern), threads, ckb, rb, spec_head, a.B * a.H, &plan);
  if (e != cudaSuccess) return e;
  kern<<<plan.grid, threads, plan.smem, s>>>(a, plan.nsr, plan.nsc);
  return cudaGetLastError();
}

// the drafts bound the dot loops at compile time: T rounds up to a power of two
template <int DV, int DK, typename TC, typename RT, int NCW, int CPR = 1>
static cudaError_t launch_spec(const rs_spec_args &a, cudaStream_t s) {
  if (a.T <= 1) return launch_spec_t<DV, DK, TC, RT, NCW, 1, CPR>(a, s);
  if (a.T <= 2) return launch_spec_t<DV, DK, TC, RT, NCW, 2, CPR>(a, s);
  if (a.T <= 4) return launch_spec_t<DV, DK, TC, RT, NCW, 4, CPR>(a, s);
  if (a.T <= 8) return launch_spec_t<DV, DK, TC, RT, NCW, 8, CPR>(a, s);
  return launch_spec_t<DV, DK, TC, RT, NCW, 16, CPR>(a, s);
}

template <typename RT>
static SpecLaunchFn find_spec_t(int d_v, int d_k, int ckpt_dtype) {
  if (ckpt_dtype == kF32) {
    if (d_v == 16 && d_k == 32) return launch_spec<16, 32, float, RT, 4>;
    if (d_v == 64 && d_k == 128) return launch_spec<64, 128, float, RT, 8, 4>;
    if (d_v == 128 && d_k == 128) return launch_spec<128, 128, float, RT, 8, 2>;
  } else if (ckpt_dtype == kF16) {
    if (d_v == 16 && d_k == 32) return launch_spec<16, 32, __half, RT, 2>;
    if (d_v == 64 && d_k == 128) return launch_spec<64, 128, __half, RT, 8>;
    if (d_v == 128 && d_k == 128) return launch_spec<128, 128, __half, RT, 8>;
  }
  return nullptr;
}

SpecLaunchFn find_spec(int d_v, int d_k, int ckpt_dtype, int in_dtype) {
  if (SpecLaunchFn f = find_spec_tc(d_v, d_k, ckpt_dtype, in_dtype)) return f;
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
