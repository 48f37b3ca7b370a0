// ReplaySSM speculative verification for Mamba-2 on the tensor cores (64 x 128
// heads, bf16 records and drafts, fp32 or fp16 checkpoint).
//
// Sources:
//   [Ghana] S. Ghana, "ReplaySSM: an SSM decoder that writes its state once
//           every 16 tokens", §Speculative decoding (T drafts behind the h
//           committed records, all T outputs without a state, flush of the
//           committed records when h + T > L).
//   [NV]    NVIDIA technical blog, "ReplaySSM: Rethinking State Storage for
//           Faster Hybrid Model Decoding", §Benefit 2 (the checkpoint is read
//           once for all T queries; the rest are products over cached keys
//           and values with a causally masked matrix of decays).
//
// It computes the verification of spec.cu: with nb records ahead of the
// drafts (nb = h, or 0 on a flush step after the h committed records are
// folded into the checkpoint) and the window's records r_0 .. r_{nb+T-1},
//   o_i = D_i (S q_i) + sum_{j <= nb+i} W_{j,i} (k_j . q_i) v_j,
// as four small matrix products per unit, each on the tensor cores:
//   the dots    Sd = K Q          (records x 128) by (128 x T), bf16, exact
//                                 operands, fp32 accumulate;
//   the state   C = S Q           (64 x 128) by (128 x T), each fp32 state
//                                 element split into two bf16 terms (hi + lo
//                                 keep ~16 mantissa bits: relative error at
//                                 most 2^-17), the bf16 queries exact;
//   the window  Y = V^T (W o Sd)  (64 x records) by (records x T), the bf16
//                                 values exact, the weighted dots split;
//   the fold    S_new = gamma S + sum_{j<h} w_j v_j k_j^T on a flush, m16n8k16
//                                 bf16 over 16 records a tile, the weighted
//                                 values split into two bf16 terms (relative
//                                 error at most 2^-17), the bf16 keys exact.
// o = D o C + Y is then formed in registers: C and Y share the accumulator
// layout (a warp's 16 state rows, lane 4g+t holding rows g and g+8 of drafts
// 2t and 2t+1).  The state sits in accumulator layout too, each lane holding
// four consecutive columns of every 16-column block, and a 16-column block is
// one k16 tile of S Q and of K Q with its columns taken in the order
// (4t, 4t+1 | 4t+2, 4t+3) <-> k (2t, 2t+1 | 2t+8, 2t+9): one 8-byte load of
// the queries serves both products.
//
// Shared-memory layout: the producer permutes the 16-byte chunks of each key
// and query record (chunk ^ 2 (j mod 4)) and of each value record (chunk ^
// (j mod 8)), so that the fragment loads of eight records at one column fall
// in distinct banks.
//
// Persistent and warp-specialised: a producer warp streams each unit's
// checkpoint (one bulk copy) and its records, drafts and decays (per-lane
// cp.async) into slot rings; groups of four consumer warps take alternate
// units.  Within a group, per unit: warp 1 computes the causal decays W and D
// (warp 2 the fold weights on a flush) while the dots run on warp 0 (and on
// the others for windows longer than 16 records), one named barrier, then
// each warp forms its 16 state rows of all T outputs.  Every wait is
// bounded.
#include "common.cuh"
#include "launch.h"

namespace rs {

namespace {

// Record slot of a unit: up to L committed + T draft records, the T queries,
// the decays, metadata, the causal decays W [record][draft], D, the fold
// weights and the dots [record][draft].
struct SpecTcRec {
  uint32_t k, v, q, a, meta, w, d, wf, s, bytes;
  int sp;  // row stride (floats) of W and the dots
};

__host__ __device__ inline SpecTcRec spec_tc_rec(int DV, int DK, int L, int T) {
  SpecTcRec o;
  uint32_t x = 0;
  const int R = L + T;
  const int R16 = (R + 15) / 16 * 16;
  o.sp = T <= 8 ? 12 : 20;  // bank-spread strides for the window's B fragments
  o.k = x;    x = align128(x + R * DK * 2);
  o.v = x;    x = align128(x + R * DV * 2);
  o.q = x;    x = align128(x + T * DK * 2);
  o.a = x;    x = align128(x + R * 4);
  o.meta = x; x = align128(x + 20);              // slot, h, flush, status, unit
  o.w = x;    x = align128(x + R16 * o.sp * 4);   // W_{j,i}, [j][i]
  o.d = x;    x = align128(x + T * 4);            // D_i
  o.wf = x;   x = align128(x + 65 * 4);           // fold weights and gamma
  o.s = x;    x = align128(x + R16 * o.sp * 4);   // k_j . q_i, [j][i]
  o.bytes = x;
  return o;
}

// barriers full/rec_empty[nsr], ck_empty[nsc] and the abort flag
__host__ __device__ inline uint32_t spec_tc_head(int nsr, int nsc) { return align128(8 * (2 * nsr + nsc) + 16); }

// Element position of column col of key or query record j in its permuted
// record (16-byte chunks of 8 bf16: chunk ^ 2 (j mod 4)).
__device__ __forceinline__ int kq_pos(int j, int col) { return ((col >> 3) ^ ((j & 3) << 1)) * 8 + (col & 7); }
// Element position of row r of value record j (chunk ^ (j mod 8)).
__device__ __forceinline__ int v_pos(int j, int r) { return ((r >> 3) ^ (j & 7)) * 8 + (r & 7); }

__device__ __forceinline__ float bf16_at(const unsigned char *base, int elem) {
  return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(base)[elem]) << 16);
}

__device__ __forceinline__ uint32_t pack_bf16(uint16_t lo, uint16_t hi) {
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

}  // namespace

template <int DV, int DK, typename TC, int NGRP, int TMAX>
__global__ void __launch_bounds__(NGRP * (DV / 16) * 32 + 32, 2)
    spec_verify_tc_kernel(const rs_spec_args a, int nsr, int nsc) {
  constexpr int RES = 2;                     // bf16 records, drafts and queries
  constexpr int NCW = DV / 16;               // consumer warps per group: 16 state rows each
  constexpr int NC = NCW * 32;
  constexpr int NB = DK / 16;                // 16-column blocks (k16 tiles)
  constexpr int NT = (TMAX + 7) / 8;         // n8 tiles of drafts
  constexpr int PROD = NGRP * NCW;
  constexpr uint32_t CKB = DV * DK * (uint32_t)sizeof(TC);
  constexpr int KC = DK * RES / 16, VC = DV * RES / 16;  // 16-byte chunks per key / value record
  static_assert(DV == 64 && DK == 128, "tiles of 16 rows and 16 columns; 8-chunk records");
  static_assert(TMAX >= 1 && TMAX <= 16 && (TMAX & (TMAX - 1)) == 0, "TMAX: a power of two up to 16");

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *rec_empty = full + nsr;
  uint64_t *ck_empty = rec_empty + nsr;
  int *s_abort = reinterpret_cast<int *>(ck_empty + nsc);
  const int T = a.T, L = a.L;
  const SpecTcRec lay = spec_tc_rec(DV, DK, L, T);
  const int SP = lay.sp;
  unsigned char *ck_slots = smem + spec_tc_head(nsr, nsc);
  unsigned char *rec_slots = ck_slots + (size_t)nsc * CKB;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_units = a.B * a.H;
  const int stride = gridDim.x;
  auto fail = [&]() {
    if (lane == 0) {
      *(volatile int *)s_abort = 1;
      report(a.dev_err, kDerrTimeout);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < nsr; ++s) {
      mbar_init(&full[s], 33);
      mbar_init(&rec_empty[s], NC);  // the consuming group
    }
    for (int c = 0; c < nsc; ++c) mbar_init(&ck_empty[c], NC);
    for (int s = 0; s < nsr; ++s) reinterpret_cast<int *>(rec_slots + (size_t)s * lay.bytes + lay.meta)[4] = -1;
    *s_abort = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == PROD) {
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
          fail();
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
          meta[0] = slot; meta[1] = hc; meta[2] = fl; meta[3] = status; meta[4] = u;
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
          cp_async16(st + lay.k + (j * DK + kq_pos(j, 8 * x)) * RES, src);
        }
        for (int cc = lane; cc < (hc + T) * VC; cc += 32) {
          const int j = cc / VC, x = cc - j * VC;
          const unsigned char *src = j < hc ? rv + (size_t)cc * 16 : vin + ((d0 + (j - hc) * dstep) * DV * RES + x * 16);
          cp_async16(st + lay.v + (j * DV + v_pos(j, 8 * x)) * RES, src);
        }
        for (int cc = lane; cc < T * KC; cc += 32) {
          const int i = cc / KC, x = cc - i * KC;
          cp_async16(st + lay.q + (i * DK + kq_pos(i, 8 * x)) * RES, qin + ((d0 + i * dstep) * DK * RES + x * 16));
        }
        float *sa = reinterpret_cast<float *>(st + lay.a);
        for (int j = lane; j < hc + T; j += 32)
          cp_async4(sa + j, j < hc ? a.ring_a + unit * L + j : a.alpha + (d0 + (j - hc) * dstep));
      } else if (lane == 0) {
        meta[0] = slot; meta[1] = hc; meta[2] = fl; meta[3] = status; meta[4] = u;
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
  const int grp = warp / NCW, lw = warp - grp * NCW, ctid = tid - grp * NC;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int rA = 16 * lw + g8, rB = rA + 8;
  auto gsync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(NC) : "memory"); };
  int s = grp % nsr, c = grp % nsc;
  uint32_t ph = (uint32_t)(grp / nsr) & 1u;
  for (int it = grp;; it += NGRP) {
    if (it != grp) {
      // a plan may have fewer slots than groups: wrap as often as needed
      s += NGRP;
      while (s >= nsr) {
        s -= nsr;
        ph ^= 1u;
      }
      c += NGRP;
      while (c >= nsc) c -= nsc;
    }
    const int u = blockIdx.x + it * stride;
    if (u >= n_units) break;
    const int b = u / a.H, h = u - (u / a.H) * a.H;
    const bool w = mbar_wait_unit(&full[s], ph,
                                  reinterpret_cast<const int *>(rec_slots + (size_t)s * lay.bytes + lay.meta) + 4, u);
    // every warp of the group leaves together: one warp's timeout stops all
    // of them at the barrier below
    if (!__all_sync(0xffffffffu, w)) fail();
    gsync();
    if (*(volatile int *)s_abort) break;
    unsigned char *st = rec_slots + (size_t)s * lay.bytes;
    const int4 m = *reinterpret_cast<const int4 *>(st + lay.meta);
    const int slot = m.x, hc = m.y, flush = m.z, status = m.w;
    float *out0 = a.out + ((size_t)b * T * a.H + h) * DV;  // draft i at + i * H * DV
    const size_t ostride = (size_t)a.H * DV;
    if (status != kStatusOk) {
      for (int x = lane; x < T * 16; x += 32) out0[(x >> 4) * ostride + 16 * lw + (x & 15)] = 0.f;
      if (ctid == 0 && status != kStatusPad) report(a.dev_err, status == kStatusBadSlot ? RS_DERR_SLOT : RS_DERR_WRITE_POS);
      mbar_arrive(&ck_empty[c]);
      mbar_arrive(&rec_empty[s]);
      continue;
    }
    const size_t unit = (size_t)slot * a.H + h;
    const unsigned char *sk = st + lay.k, *sv = st + lay.v, *sq = st + lay.q;
    const float *sa = reinterpret_cast<const float *>(st + lay.a);
    float *sWt = reinterpret_cast<float *>(st + lay.w), *sD = reinterpret_cast<float *>(st + lay.d);
    float *sWf = reinterpret_cast<float *>(st + lay.wf), *sS = reinterpret_cast<float *>(st + lay.s);
    // the window's records start at r0 (the drafts only, on a flush): draft
    // i's window is r0 .. r0+nb+i, R = nb + T records in all
    const int nb = flush ? 0 : hc, r0 = flush ? hc : 0, R = nb + T;
    const unsigned char *ck_slot = ck_slots + (size_t)c * CKB;
    auto ld4 = [&](int r, int col) -> float4 {
      if constexpr (sizeof(TC) == 4) {
        return *reinterpret_cast<const float4 *>(ck_slot + ((size_t)r * DK + col) * 4);
      } else {
        float f[4];
        LpVec<__half>::unpack(*reinterpret_cast<const uint2 *>(ck_slot + ((size_t)r * DK + col) * 2), f);
        return make_float4(f[0], f[1], f[2], f[3]);
      }
    };
    // B fragments of the queries for k16 tile bk (columns in the tile order
    // above), n8 tile n: draft 8n + g8
    auto qfrag = [&](int bk, int n) -> uint2 {
      const int qi = 8 * n + g8;
      if (qi >= T) return make_uint2(0u, 0u);
      return *reinterpret_cast<const uint2 *>(sq + ((size_t)qi * DK + kq_pos(qi, 16 * bk + 4 * t4)) * RES);
    };

    // ---- phase A: decays (warp 1), fold weights (warp 2), dots (warp 0
    // first, the others for longer windows) ----
    if (lw == 1) {
      // W_{j,0} and D_0 from one suffix scan over the first draft's window;
      // each later draft multiplies in its own decay
      float x0 = lane <= nb ? sa[r0 + lane] : 1.f;
      float x1 = lane + 32 <= nb ? sa[r0 + lane + 32] : 1.f;
      suffix_scan64(x0, x1, lane, [](float x, float y) { return x * y; });
      const float n0 = __shfl_down_sync(0xffffffffu, x0, 1);
      const float n1 = __shfl_down_sync(0xffffffffu, x1, 1);
      const float hi0 = __shfl_sync(0xffffffffu, x1, 0);
      float wa = lane == 31 ? hi0 : n0, wb = lane == 31 ? 1.f : n1;
      float dcum = __shfl_sync(0xffffffffu, x0, 0);
      for (int i = 0; i < T; ++i) {
        if (i > 0) {
          const int jn = nb + i;
          const float al = sa[r0 + jn];
          wa = lane < jn ? wa * al : (lane == jn ? 1.f : wa);
          wb = lane + 32 < jn ? wb * al : (lane + 32 == jn ? 1.f : wb);
          dcum *= al;
        }
        // causal mask: records after the draft's own weigh 0
        if (lane < R) sWt[lane * SP + i] = lane <= nb + i ? wa : 0.f;
        if (lane + 32 < R) sWt[(lane + 32) * SP + i] = lane + 32 <= nb + i ? wb : 0.f;
        if (lane == 0) sD[i] = dcum;
      }
      // records of the last 16-tile past R weigh 0 for every draft
      for (int x = R + lane; x < (R + 15) / 16 * 16; x += 32)
        for (int i = 0; i < T; ++i) sWt[x * SP + i] = 0.f;
    } else if (lw == 2 && flush) {
      // fold weights of the committed records, and their gamma
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
    // Sd = K Q over the window's records, 16 records per tile, tiles shared
    // by the group's warps (warp 0 first: with a window of at most 16
    // records the decays and the fold weights run beside it); records past
    // R read as 0
    for (int rt = (NCW - lw) % NCW; rt * 16 < R; rt += NCW) {
      const int ja = rt * 16 + g8, jb = ja + 8;  // window records of rows g8, g8 + 8
      float dacc[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) dacc[n][0] = dacc[n][1] = dacc[n][2] = dacc[n][3] = 0.f;
#pragma unroll
      for (int bk = 0; bk < NB; ++bk) {
        const int col = 16 * bk + 4 * t4;
        uint2 ka = make_uint2(0u, 0u), kb = make_uint2(0u, 0u);
        if (ja < R) ka = *reinterpret_cast<const uint2 *>(sk + ((size_t)(r0 + ja) * DK + kq_pos(r0 + ja, col)) * RES);
        if (jb < R) kb = *reinterpret_cast<const uint2 *>(sk + ((size_t)(r0 + jb) * DK + kq_pos(r0 + jb, col)) * RES);
        const uint32_t af[4] = {ka.x, kb.x, ka.y, kb.y};
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const uint2 bq = qfrag(bk, n);
          mma_bf16(dacc[n], af, bq.x, bq.y);
        }
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int i0 = 8 * n + 2 * t4;
        // rows past R hold zeros (their keys read as 0)
        *reinterpret_cast<float2 *>(sS + (size_t)ja * SP + i0) = make_float2(dacc[n][0], dacc[n][1]);
        *reinterpret_cast<float2 *>(sS + (size_t)jb * SP + i0) = make_float2(dacc[n][2], dacc[n][3]);
      }
    }

    gsync();  // decays, fold weights and dots are in the slot

    // ---- phase B: this warp's 16 state rows of all T outputs ----
    // The state streams from the slot one 16-column block at a time: on a
    // flush the block is folded, S_new = gamma S + sum_{j<h} w_j v_j k_j^T
    // (unrounded), and stored; then C += S_block Q_block with each state
    // element split into two bf16 terms.
    const float gam = flush ? sWf[64] : 1.f;
    TC *ckg = static_cast<TC *>(a.ckpt) + unit * (DV * DK);
    // the fold's A operands for the 16 committed records from j0, records
    // j0 + 2t + {0, 1} and j0 + 2t + 8 + {0, 1} of an m16n8k16 tile (weighted
    // values of rows rA and rB, each split into two bf16 terms: relative error
    // at most 2^-17, as for S Q); past h they weigh 0 and read record 0
    auto fold_a = [&](int j0, uint32_t (&ah)[4], uint32_t (&al)[4], int (&rj)[4]) {
      float w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = j0 + 2 * t4 + (e & 1) + 8 * (e >> 1);
        rj[e] = j < hc ? j : 0;
        w[e] = j < hc ? sWf[j] : 0.f;
      }
      auto wv = [&](int e, int r) { return w[e] * bf16_at(sv, rj[e] * DV + v_pos(rj[e], r)); };
      split_bf16x2(wv(0, rA), wv(1, rA), ah[0], al[0]);
      split_bf16x2(wv(0, rB), wv(1, rB), ah[1], al[1]);
      split_bf16x2(wv(2, rA), wv(3, rA), ah[2], al[2]);
      split_bf16x2(wv(2, rB), wv(3, rB), ah[3], al[3]);
    };
    // the first 16 committed records' operands are formed once for all
    // column blocks (a window of L <= 16 fits); later ones per block
    uint32_t fh[4], fl[4];
    int frj[4];
    if (flush) fold_a(0, fh, fl, frj);
    float cacc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) cacc[n][0] = cacc[n][1] = cacc[n][2] = cacc[n][3] = 0.f;
#pragma unroll 1
    for (int bk = 0; bk < NB; ++bk) {
      float4 pa = ld4(rA, 16 * bk + 4 * t4), pb = ld4(rB, 16 * bk + 4 * t4);
      if (flush) {
        pa.x *= gam; pa.y *= gam; pa.z *= gam; pa.w *= gam;
        pb.x *= gam; pb.y *= gam; pb.z *= gam; pb.w *= gam;
        const uint16_t *sk16 = reinterpret_cast<const uint16_t *>(sk);
        for (int j0 = 0; j0 < hc; j0 += 16) {
          uint32_t ah[4], al[4];
          int rj[4];
          if (j0 == 0) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              ah[e] = fh[e];
              al[e] = fl[e];
              rj[e] = frj[e];
            }
          } else {
            fold_a(j0, ah, al, rj);
          }
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int col = 16 * bk + 4 * (g8 >> 1) + (g8 & 1) + 2 * hf;  // column of tile index n = g8
            float d[4] = {hf ? pa.z : pa.x, hf ? pa.w : pa.y, hf ? pb.z : pb.x, hf ? pb.w : pb.y};
            // the bf16 keys of the tile's records at this column, exact
            const uint32_t b0 = pack_bf16(sk16[rj[0] * DK + kq_pos(rj[0], col)], sk16[rj[1] * DK + kq_pos(rj[1], col)]);
            const uint32_t b1 = pack_bf16(sk16[rj[2] * DK + kq_pos(rj[2], col)], sk16[rj[3] * DK + kq_pos(rj[3], col)]);
            mma_bf16(d, ah, b0, b1);
            mma_bf16(d, al, b0, b1);
            if (hf) {
              pa.z = d[0]; pa.w = d[1]; pb.z = d[2]; pb.w = d[3];
            } else {
              pa.x = d[0]; pa.y = d[1]; pb.x = d[2]; pb.y = d[3];
            }
          }
        }
        const size_t offA = (size_t)rA * DK + 16 * bk + 4 * t4, offB = (size_t)rB * DK + 16 * bk + 4 * t4;
        const float fa[4] = {pa.x, pa.y, pa.z, pa.w};
        const float fb[4] = {pb.x, pb.y, pb.z, pb.w};
        if constexpr (sizeof(TC) == 4) {
          st_vec(ckg + offA, CkVec<float>::pack(fa));
          st_vec(ckg + offB, CkVec<float>::pack(fb));
        } else {
          st_vec2(ckg + offA, LpVec<__half>::pack(fa));
          st_vec2(ckg + offB, LpVec<__half>::pack(fb));
        }
      }
      uint32_t hi[4], lo[4];
      split_bf16x2(pa.x, pa.y, hi[0], lo[0]);
      split_bf16x2(pb.x, pb.y, hi[1], lo[1]);
      split_bf16x2(pa.z, pa.w, hi[2], lo[2]);
      split_bf16x2(pb.z, pb.w, hi[3], lo[3]);
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const uint2 bq = qfrag(bk, n);
        mma_bf16(cacc[n], hi, bq.x, bq.y);
        mma_bf16(cacc[n], lo, bq.x, bq.y);
      }
    }
    mbar_arrive(&ck_empty[c]);
    // Y = V^T (W o Sd): k16 tiles over the window's records (natural order),
    // the bf16 values exact, the weighted dots split into two bf16 terms
    float yacc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) yacc[n][0] = yacc[n][1] = yacc[n][2] = yacc[n][3] = 0.f;
    const uint16_t *sv16 = reinterpret_cast<const uint16_t *>(sv);
    for (int j0 = 0; j0 < R; j0 += 16) {
      uint16_t vv[2][4];  // [row rA / rB][records j0 + 2t4, +1, +8, +9]
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = j0 + 2 * t4 + (e & 1) + 8 * (e >> 1);
        const int jr = r0 + j;
        vv[0][e] = j < R ? sv16[jr * DV + v_pos(jr, rA)] : (uint16_t)0;
        vv[1][e] = j < R ? sv16[jr * DV + v_pos(jr, rB)] : (uint16_t)0;
      }
      const uint32_t af[4] = {pack_bf16(vv[0][0], vv[0][1]), pack_bf16(vv[1][0], vv[1][1]),
                              pack_bf16(vv[0][2], vv[0][3]), pack_bf16(vv[1][2], vv[1][3])};
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int i = 8 * n + g8;  // the draft of this lane's B column
        float sw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = j0 + 2 * t4 + (e & 1) + 8 * (e >> 1);
          sw[e] = i < T ? sWt[j * SP + i] * sS[j * SP + i] : 0.f;
        }
        uint32_t bh0, bl0, bh1, bl1;
        split_bf16x2(sw[0], sw[1], bh0, bl0);
        split_bf16x2(sw[2], sw[3], bh1, bl1);
        mma_bf16(yacc[n], af, bh0, bh1);
        mma_bf16(yacc[n], af, bl0, bl1);
      }
    }
    // o_i = D_i (S q_i) + Y, rows rA and rB, drafts 8n + 2t4 and 8n + 2t4 + 1
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = 8 * n + 2 * t4 + e;
        if (i < T) {
          const float di = sD[i];
          out0[i * ostride + rA] = fmaf(di, cacc[n][e], yacc[n][e]);
          out0[i * ostride + rB] = fmaf(di, cacc[n][2 + e], yacc[n][2 + e]);
        }
      }
    }
    // the drafts' records (slot records hc .. hc+T-1) go to ring slots nb .. nb+T-1
    uint4 *rkg = reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.ring_k) + (unit * L + nb) * DK * RES);
    uint4 *rvg = reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.ring_v) + (unit * L + nb) * DV * RES);
    for (int x = ctid; x < T * KC; x += NC) {
      const int i = x / KC, ch = x - i * KC, j = hc + i;
      rkg[x] = *reinterpret_cast<const uint4 *>(sk + (j * DK + kq_pos(j, 8 * ch)) * RES);
    }
    for (int x = ctid; x < T * VC; x += NC) {
      const int i = x / VC, ch = x - i * VC, j = hc + i;
      rvg[x] = *reinterpret_cast<const uint4 *>(sv + (j * DV + v_pos(j, 8 * ch)) * RES);
    }
    if (ctid < T) a.ring_a[unit * L + nb + ctid] = sa[hc + ctid];
    mbar_arrive(&rec_empty[s]);
  }
  if (tid == 0 && *(volatile int *)s_abort) report(a.dev_err, kDerrTimeout);
}

template <int DV, int DK, typename TC, int TMAX>
static cudaError_t launch_spec_tc_t(const rs_spec_args &a, cudaStream_t s) {
  constexpr int NGRP = 2;
  auto kern = spec_verify_tc_kernel<DV, DK, TC, NGRP, TMAX>;
  constexpr int threads = NGRP * (DV / 16) * 32 + 32;
  const size_t ckb = (size_t)DV * DK * sizeof(TC);
  const size_t rb = spec_tc_rec(DV, DK, a.L, a.T).bytes;
  RingPlan plan;
  cudaError_t e = plan_rings(reinterpret_cast<const void *>(kern), threads, ckb, rb, spec_tc_head, a.B * a.H, &plan);
  if (e != cudaSuccess) return e;
  kern<<<plan.grid, threads, plan.smem, s>>>(a, plan.nsr, plan.nsc);
  return cudaGetLastError();
}

template <int DV, int DK, typename TC>
static cudaError_t launch_spec_tc(const rs_spec_args &a, cudaStream_t s) {
  if (a.T <= 1) return launch_spec_tc_t<DV, DK, TC, 1>(a, s);
  if (a.T <= 2) return launch_spec_tc_t<DV, DK, TC, 2>(a, s);
  if (a.T <= 4) return launch_spec_tc_t<DV, DK, TC, 4>(a, s);
  if (a.T <= 8) return launch_spec_tc_t<DV, DK, TC, 8>(a, s);
  return launch_spec_tc_t<DV, DK, TC, 16>(a, s);
}

// the 64 x 128 heads with bf16 records and drafts; nullptr for the others
SpecLaunchFn find_spec_tc(int d_v, int d_k, int ckpt_dtype, int in_dtype) {
  if (in_dtype != kBF16 || d_v != 64 || d_k != 128) return nullptr;
  if (ckpt_dtype == kF32) return launch_spec_tc<64, 128, float>;
  if (ckpt_dtype == kF16) return launch_spec_tc<64, 128, __half>;
  return nullptr;
}

}  // namespace rs
