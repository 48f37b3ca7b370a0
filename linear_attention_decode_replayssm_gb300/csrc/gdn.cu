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
// With p ring records (d_j, k_j, g_j), j < p, of one (row b, head h):
//   G_j = exp(sum_{l=j+1..p-1} g_l),  Gamma = exp(sum_{l<p} g_l),
//   a = S_{t-1} k_t = Gamma (S_ckpt k_t) + sum_j G_j (k_j . k_t) d_j,
//   c = S_{t-1} q_t = Gamma (S_ckpt q_t) + sum_j G_j (k_j . q_t) d_j,
//   alpha_t = exp(g_t),  d_t = beta_t (v_t - alpha_t a),
//   non-flush: o = alpha_t c + (k_t . q_t) d_t; append (d_t, k_t, g_t) with d
//              and k rounded to the ring type;
//   flush:     S_new = alpha_t (Gamma S_ckpt + sum_j G_j d_j k_j^T) + d_t k_t^T
//              with the unrounded d_t, o = S_new q_t, S_new stored.
// Every row of the state is independent given the dot products, so a work
// unit is a block of RB state rows of one head (a 128 x 128 fp32 head is two
// 32 KiB units); both halves compute the (cheap) key dot products.
//
// Same pipeline as the Mamba-2 kernel: persistent, two CTAs per SM, one
// producer warp (the unit's checkpoint rows as one bulk copy into a
// checkpoint slot, the ring records, this token's inputs and the gates as
// per-lane cp.async into a record slot).  A window warp takes each record
// slot as it lands and computes everything that does not touch the
// checkpoint: the gate weights G_j and Gamma, the key dots k_j . k_t and
// k_j . q_t (eight records per reduction) and the window terms
// sum_j G_j (k_j . k_t) d_j and sum_j G_j (k_j . q_t) d_j of every state row;
// it signals the consumers on a second barrier.
// Two groups of four consumer warps take alternate units.  On a non-flush
// unit a group forms S_ckpt k_t and S_ckpt q_t in one pass over the slot
// (freeing it after the pass) with one transposed group reduction; the lanes
// that finish a row add the window terms and form d_t and the output.  On a
// flush each warp takes 16 whole rows in tensor-core accumulator layout and
// folds the window on the tensor cores.  A state row never leaves its warp,
// so the consumer warps never wait for each other.  All waits are bounded
// and report RS_DERR_TIMEOUT instead of hanging.
#include "common.cuh"
#include "launch.h"
#include "replayssm.h"

namespace rs {

// Byte offsets of one record slot.
struct GdnRec {
  uint32_t k, kt, q, d, vt, a, meta, scr, bytes;
};

__host__ __device__ inline GdnRec gdn_rec(int RB, int DK, int res, int ies, int L) {
  GdnRec s;
  uint32_t o = 0;
  s.k = o;    o = align128(o + L * DK * res);    // key records 0..p-1 (ring type)
  s.kt = o;   o = align128(o + DK * ies);        // this token's key (input type)
  s.q = o;    o = align128(o + DK * ies);
  s.d = o;    o = align128(o + L * RB * res);    // corrected values of this unit's rows
  s.vt = o;   o = align128(o + RB * ies);
  s.a = o;    o = align128(o + (L + 4) * 4);     // g_0..g_{p-1}; [L] = g_t, [L+1] = beta_t
  s.meta = o; o = align128(o + 20);  // slot, p, flush, status, unit
  s.scr = o;  o = align128(o + (3 * L + 3 * RB + 4) * 4);  // G_j, weighted key dots, row window terms, d_t, scalars
  s.bytes = o;
  return s;
}

// barriers: full, ready and empty per record slot, empty per checkpoint slot
__host__ __device__ inline uint32_t gdn_head(int nsr, int nsc) { return align128(8 * (3 * nsr + nsc) + 16); }

// LMAX bounds the buffer length at compile time (L <= LMAX).
// CPR: 16-byte checkpoint chunks a consumer lane holds per state row (chunks
// cv, cv + G, ...), so the row reductions run over G = DK / (E CPR) lanes.
// NGRP consumer groups of NCW warps take alternate units (a flush unit's
// fold in one group overlaps the other group's units); MINB CTAs per SM.
template <int DV, int DK, typename TC, typename RT, typename IT, int NCW, int NSPLIT, int LMAX, int CPR, int NGRP,
          int MINB>
__global__ void __launch_bounds__(NGRP * NCW * 32 + 64, MINB) gdn_replay_kernel(const KArgs a, int nsr, int nsc) {
  using V = CkVec<TC>;
  constexpr int RB = DV / NSPLIT;    // state rows per unit
  constexpr int E = V::E;
  constexpr int NCH = DK / E;        // 16-byte chunks per state row
  constexpr int G = NCH / CPR;       // lanes per state row
  constexpr int NC = NCW * 32;       // consumer threads per group
  constexpr int RPP = NC / G;        // state rows per pass
  constexpr int VPT = RB / RPP;      // state rows per consumer thread
  constexpr int WIN = NGRP * NCW;    // warp index of the window warp
  constexpr int PROD = WIN + 1;      // warp index of the producer
  constexpr int RPL = (RB + 31) / 32;  // state rows per window-warp lane
  constexpr uint32_t CKB = RB * DK * (uint32_t)sizeof(TC);
  static_assert(G <= 32 && 32 % G == 0 && NCH % CPR == 0, "a state row must fit in one warp");
  static_assert(NC % G == 0 && RB % RPP == 0 && VPT >= 1 && 2 * VPT <= G, "bad tiling");
  static_assert(DK % 8 == 0 && RB % 8 == 0 && DK <= 128 && RB <= 32 * RPL, "bad head dims");
  // flush on the tensor cores: 64-row units of an fp32 or fp16 checkpoint,
  // each warp of the group one 16-row tile (of half the columns with eight
  // warps, of all of them with four)
  constexpr bool MMAF = (sizeof(TC) == 4 || sizeof(TC) == 2) && RB == 64 && DK % 32 == 0 && (DK & (DK - 1)) == 0 &&
                        (NCW == 8 || NCW == 4);

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *ready = full + nsr;
  uint64_t *rec_empty = ready + nsr;
  uint64_t *ck_empty = rec_empty + nsr;
  int *s_abort = reinterpret_cast<int *>(ck_empty + nsc);
  const int L = a.L;
  constexpr int rdt = Rec<RT>::kDtype, idt = Rec<IT>::kDtype;  // ring and input element types
  constexpr int res = (int)sizeof(RT), ies = (int)sizeof(IT);
  const GdnRec lay = gdn_rec(RB, DK, res, ies, L);
  unsigned char *ck_slots = smem + gdn_head(nsr, nsc);
  unsigned char *rec_slots = ck_slots + (size_t)nsc * CKB;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per_row = a.H * NSPLIT;
  const int n_units = a.B * per_row;
  const int stride = gridDim.x;
  // a wait that ran out: flag every warp to stop and report it once per warp
  auto fail = [&]() {
    if (lane == 0) {
      *(volatile int *)s_abort = 1;
      report(a.dev_err, kDerrTimeout);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < nsr; ++s) {
      mbar_init(&full[s], 33);
      mbar_init(&ready[s], 32);           // the window warp's lanes
      mbar_init(&rec_empty[s], NC + 32);  // the consuming group's threads and the window warp
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
    int it = 0;
    auto fetch = [&](int ub, int &sl, int &wp, int &fl) {
      const int u = ub + lane * stride;
      if (u < n_units) {
        const int b = u / per_row;
        sl = __ldg(a.slot_idx + b);
        wp = __ldg(a.write_pos + b);
        fl = __ldg(a.is_flush + b);
      } else {
        sl = -1; wp = 0; fl = 0;
      }
    };
    int c_sl, c_wp, c_fl;
    fetch(blockIdx.x, c_sl, c_wp, c_fl);
    bool ok = true;
    for (int ub = blockIdx.x; ok && ub < n_units; ub += 32 * stride) {
      int n_sl, n_wp, n_fl;
      fetch(ub + 32 * stride, n_sl, n_wp, n_fl);
      for (int j = 0; j < 32; ++j) {
        const int u = ub + j * stride;
        if (u >= n_units) break;
        const int slot = __shfl_sync(0xffffffffu, c_sl, j);
        const int p = __shfl_sync(0xffffffffu, c_wp, j);
        const int fl = __shfl_sync(0xffffffffu, c_fl, j);
        const int s = it % nsr, c = it % nsc;
        if (it >= nsr || it >= nsc) {
          int w = 1;
          if (lane == 0) {
            if (it >= nsr) w = mbar_wait(&rec_empty[s], ((uint32_t)(it / nsr) & 1u) ^ 1u) ? 1 : 0;
            if (w && it >= nsc) w = mbar_wait(&ck_empty[c], ((uint32_t)(it / nsc) & 1u) ^ 1u) ? 1 : 0;
          }
          w = __shfl_sync(0xffffffffu, w, 0);
          if (!w || *(volatile int *)s_abort) {
            fail();
            ok = false;
            break;
          }
        }
        __syncwarp();
        const int b = u / per_row;
        const int rem = u - b * per_row;
        const int h = rem / NSPLIT, row_off = (rem - h * NSPLIT) * RB;
        const int status = slot < 0 ? kStatusPad
                           : slot >= a.num_slots ? kStatusBadSlot
                           : (p < 0 || p >= L) ? kStatusBadPos
                           : kStatusOk;
        unsigned char *st = rec_slots + (size_t)s * lay.bytes;
        int *meta = reinterpret_cast<int *>(st + lay.meta);
        if (status == kStatusOk) {
          const size_t unit = (size_t)slot * a.H + h;
          if (lane == 0) {
            meta[0] = slot; meta[1] = p; meta[2] = fl; meta[3] = status; meta[4] = u;
            mbar_expect_tx(&full[s], CKB);
            bulk_load(ck_slots + (size_t)c * CKB,
                      static_cast<const TC *>(a.ckpt) + unit * (DV * DK) + (size_t)row_off * DK, CKB, &full[s],
                      pol_stream);
          }
          constexpr int KC = DK * res / 16, DC = RB * res / 16, ITC = DK * ies / 16, VTC = RB * ies / 16;
          const unsigned char *rk = static_cast<const unsigned char *>(a.ring_k) + unit * L * DK * res;
          const unsigned char *rd = static_cast<const unsigned char *>(a.ring_v);
#pragma unroll
          for (int i = 0; i < (LMAX * KC + 31) / 32; ++i) {
            const int cc = lane + 32 * i;
            if (cc < p * KC) cp_async16(st + lay.k + cc * 16, rk + cc * 16);
          }
#pragma unroll
          for (int i = 0; i < (LMAX * DC + 31) / 32; ++i) {
            const int cc = lane + 32 * i;
            if (cc < p * DC) {
              const int jj = cc / DC;
              cp_async16(st + lay.d + cc * 16,
                         rd + ((unit * L + jj) * DV + row_off) * res + (size_t)(cc - jj * DC) * 16);
            }
          }
          const unsigned char *kin =
              static_cast<const unsigned char *>(a.k) + ((size_t)b * a.sk + (size_t)h * DK) * ies;
          const unsigned char *qin =
              static_cast<const unsigned char *>(a.q) + ((size_t)b * a.sq + (size_t)h * DK) * ies;
          const unsigned char *vin =
              static_cast<const unsigned char *>(a.v) + ((size_t)b * a.sv + (size_t)h * DV + row_off) * ies;
          for (int cc = lane; cc < ITC; cc += 32) {
            cp_async16(st + lay.kt + cc * 16, kin + cc * 16);
            cp_async16(st + lay.q + cc * 16, qin + cc * 16);
          }
          for (int cc = lane; cc < VTC; cc += 32) cp_async16(st + lay.vt + cc * 16, vin + cc * 16);
          float *sa = reinterpret_cast<float *>(st + lay.a);
#pragma unroll
          for (int i = 0; i < (LMAX + 31) / 32; ++i) {
            const int jj = lane + 32 * i;
            if (jj < p) cp_async4(sa + jj, a.ring_a + unit * L + jj);
          }
          if (lane == 30) cp_async4(sa + L, a.alpha + (size_t)b * a.H + h);
          if (lane == 31) cp_async4(sa + L + 1, a.beta + (size_t)b * a.H + h);
        } else if (lane == 0) {
          meta[0] = slot; meta[1] = p; meta[2] = fl; meta[3] = status; meta[4] = u;
        }
        if (lane == 0) mbar_arrive(&full[s]);
        cp_async_arrive(&full[s]);
        ++it;
      }
      c_sl = n_sl; c_wp = n_wp; c_fl = n_fl;
    }
    if (lane == 0) {
      for (int k = it > nsr ? it - nsr : 0; k < it; ++k) mbar_wait(&full[k % nsr], (uint32_t)(k / nsr) & 1u);
    }
    __syncwarp();
    return;
  }


  if (warp == WIN) {
    // --------------------------------------------------------------- window
    int s = 0;
    uint32_t ph = 0;
    for (int it = 0;; ++it) {
      if (it && ++s == nsr) {
        s = 0;
        ph ^= 1u;
      }
      const int u = blockIdx.x + it * stride;
      if (u >= n_units) break;
      const bool w = mbar_wait(&full[s], ph);
      if (!__all_sync(0xffffffffu, w) || *(volatile int *)s_abort) {
        fail();
        break;
      }
      unsigned char *st = rec_slots + (size_t)s * lay.bytes;
      const int *meta = reinterpret_cast<const int *>(st + lay.meta);
      const int p = meta[1], status = meta[3];
      const float *sa = reinterpret_cast<const float *>(st + lay.a);
      float *scr = reinterpret_cast<float *>(st + lay.scr);
      float *sW = scr, *sDk = scr + L, *sDq = scr + 2 * L;
      float *sCk = scr + 3 * L, *sCq = sCk + RB, *sScal = sCq + 2 * RB;
      const unsigned char *sk = st + lay.k, *skt = st + lay.kt, *sq = st + lay.q, *sd = st + lay.d;
      if (status == kStatusOk) {
        // gate weights: G_j = exp(sum of the gates after record j), Gamma =
        // exp(sum of all); lane j keeps G_j (and G_{j+32}) for the dots below
        float x0 = lane < p ? sa[lane] : 0.f;
        float x1 = lane + 32 < p ? sa[lane + 32] : 0.f;
        suffix_scan64(x0, x1, lane, [](float x, float y) { return x + y; });
        const float n0 = __shfl_down_sync(0xffffffffu, x0, 1);
        const float n1 = __shfl_down_sync(0xffffffffu, x1, 1);
        const float hi0 = __shfl_sync(0xffffffffu, x1, 0);
        const float gw0 = expf(lane == 31 ? hi0 : n0);
        float gw1 = 0.f;
        if constexpr (LMAX > 32) gw1 = expf(lane == 31 ? 0.f : n1);
        if (lane < p) sW[lane] = gw0;
        if (LMAX > 32 && lane + 32 < p) sW[lane + 32] = gw1;
        if (lane == 0) {
          sScal[0] = expf(x0);
          sScal[2] = expf(sa[L]);  // alpha_t
        }
        // k_j . k_t and k_j . q_t, eight records per transposed reduction;
        // record p is this token's key (its q-dot is k_t . q_t)
        float kt4[4], q4[4];
        const int col = lane * 4;
        if (col < DK) {
          lds_cols<4>(skt, col, idt, kt4);
          lds_cols<4>(sq, col, idt, q4);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) kt4[e] = q4[e] = 0.f;
        }
#pragma unroll 1
        for (int j0 = 0; j0 <= p; j0 += 8) {
          float part[16];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const int j = j0 + r;
            float kk[4] = {0.f, 0.f, 0.f, 0.f};
            if (col < DK) {
              if (j < p) {
                lds_cols<4>(sk, j * DK + col, rdt, kk);
              } else if (j == p) {
#pragma unroll
                for (int e = 0; e < 4; ++e) kk[e] = kt4[e];
              }
            }
            // both dots of the record share its key: one packed FMA per element
            float2 dkq = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 4; ++e) dkq = ffma2(make_float2(kk[e], kk[e]), make_float2(kt4[e], q4[e]), dkq);
            part[r] = dkq.x;
            part[8 + r] = dkq.y;
          }
          group_reduce<16, 32>(part, lane);
          const int vi = group_reduce_index<16, 32>(lane);
          const int j = j0 + (vi & 7);
          float gj = __shfl_sync(0xffffffffu, gw0, j & 31);
          if constexpr (LMAX > 32) {
            const float g1 = __shfl_sync(0xffffffffu, gw1, j & 31);
            if (j >= 32) gj = g1;
          }
          if (group_reduce_writer<16, 32>(lane)) {
            if (j < p) {
              if (vi < 8)
                sDk[j] = gj * part[0];
              else
                sDq[j] = gj * part[0];
            } else if (j == p && vi >= 8) {
              sScal[1] = part[0];  // k_t . q_t
            }
          }
        }
        __syncwarp();
        // window terms of S_{t-1} k_t and S_{t-1} q_t for this lane's rows
        if (lane * RPL < RB) {
          float cK[RPL], cQ[RPL];
#pragma unroll
          for (int e = 0; e < RPL; ++e) cK[e] = cQ[e] = 0.f;
#pragma unroll 4
          for (int j = 0; j < p; ++j) {
            const float wk = sDk[j], wq = sDq[j];
#pragma unroll
            for (int e = 0; e < RPL; ++e) {
              const float dd = lds_elem(sd, j * RB + lane * RPL + e, rdt);
              cK[e] = fmaf(wk, dd, cK[e]);
              cQ[e] = fmaf(wq, dd, cQ[e]);
            }
          }
#pragma unroll
          for (int e = 0; e < RPL; ++e) {
            sCk[lane * RPL + e] = cK[e];
            sCq[lane * RPL + e] = cQ[e];
          }
        }
        __syncwarp();
      }
      mbar_arrive(&ready[s]);
      mbar_arrive(&rec_empty[s]);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  // group g takes the CTA's units g, g + NGRP, ...; the lanes of a state row
  // are in one warp, so the warps run independently of each other
  const int grp = warp / NCW, lw = warp - grp * NCW, ctid = tid - grp * NC;
  const int row0 = ctid / G, cv = ctid - (ctid / G) * G;
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
    // the checkpoint and records have landed; the window warp's terms are
    // awaited only after the checkpoint pass, so its latency does not hold
    // the checkpoint slot
    const bool w = mbar_wait_unit(&full[s], ph,
                                  reinterpret_cast<const int *>(rec_slots + (size_t)s * lay.bytes + lay.meta) + 4, u);
    if (!__all_sync(0xffffffffu, w) || *(volatile int *)s_abort) {
      fail();
      break;
    }

    unsigned char *st = rec_slots + (size_t)s * lay.bytes;
    const int *meta = reinterpret_cast<const int *>(st + lay.meta);
    const int slot = meta[0], p = meta[1], flush = meta[2], status = meta[3];
    const int b = u / per_row;
    const int rem = u - b * per_row;
    const int h = rem / NSPLIT, half = rem - h * NSPLIT, row_off = half * RB;
    float *orow = a.out + (size_t)b * a.so + (size_t)h * DV + row_off;
    if (status != kStatusOk) {
      for (int i = ctid; i < RB; i += NC) orow[i] = 0.f;
      if (ctid == 0 && status != kStatusPad) report(a.dev_err, status == kStatusBadSlot ? 1 : 2);
      mbar_arrive(&ck_empty[c]);
      mbar_arrive(&rec_empty[s]);  // the window warp arrives on it too before the slot is reused
      continue;
    }
    if constexpr (MMAF) {
      if (flush) {
        // Flush on the tensor cores.  Warp lw holds state rows rA = 16 (lw % 4)
        // + g and rB = rA + 8 of the unit, columns (DK / CW) (lw / 4) + 16 bk +
        // 4t .. + 3 in accumulator layout (CW = NCW / 4 warps share a row).  S_ckpt k_t and S_ckpt q_t of its rows
        // come from the whole rows in the slot; then d_t, the output by the
        // expansion o = alpha_t (Gamma S_ckpt q_t + window term) + d_t (k_t .
        // q_t) (the unrounded S_new applied to q_t), and the fold S_new =
        // alpha_t Gamma S_ckpt + sum_{j<p} alpha_t G_j d_j k_j^T + d_t k_t^T
        // as a rank-(p+1) m16n8k8 tf32 product: each weighted value split into
        // two tf32 terms (the current d_t unrounded), 16-bit keys exact, fp32
        // keys split too.
        constexpr int CW = NCW / 4;        // warps per row
        constexpr int NBH = DK / 16 / CW;  // 16-column blocks a warp holds
        const int g8 = lane >> 2, t4 = lane & 3;
        const int rA = 16 * (lw & 3) + g8, rB = rA + 8, cb = (DK / CW) * (lw >> 2);
        const unsigned char *ck_slot = ck_slots + (size_t)c * CKB;
        const unsigned char *skt = st + lay.kt, *sq = st + lay.q, *sk = st + lay.k, *sd = st + lay.d;
        auto ld4 = [&](int r, int col) -> float4 {
          if constexpr (sizeof(TC) == 4) {
            return *reinterpret_cast<const float4 *>(ck_slot + ((size_t)r * DK + col) * 4);
          } else {
            float f[4];
            LpVec<__half>::unpack(*reinterpret_cast<const uint2 *>(ck_slot + ((size_t)r * DK + col) * 2), f);
            return make_float4(f[0], f[1], f[2], f[3]);
          }
        };
        auto dot4 = [](const float4 &x, const float (&y)[4], float acc) {
          return fmaf(x.x, y[0], fmaf(x.y, y[1], fmaf(x.z, y[2], fmaf(x.w, y[3], acc))));
        };
        float4 xa[NBH], xb[NBH];
        float kA = 0.f, kB = 0.f, qA = 0.f, qB = 0.f;
#pragma unroll
        for (int bk = 0; bk < DK / 16; ++bk) {
          const int col = (cb + 16 * bk + 4 * t4) & (DK - 1);  // own columns first, then the rest
          const float4 ya = ld4(rA, col), yb = ld4(rB, col);
          float k4[4], q4[4];
          lds_cols<4>(skt, col, idt, k4);
          lds_cols<4>(sq, col, idt, q4);
          kA = dot4(ya, k4, kA); kB = dot4(yb, k4, kB);
          qA = dot4(ya, q4, qA); qB = dot4(yb, q4, qB);
          if (bk < NBH) {
            xa[bk] = ya;
            xb[bk] = yb;
          }
        }
        mbar_arrive(&ck_empty[c]);
        kA += __shfl_xor_sync(0xffffffffu, kA, 1); kA += __shfl_xor_sync(0xffffffffu, kA, 2);
        kB += __shfl_xor_sync(0xffffffffu, kB, 1); kB += __shfl_xor_sync(0xffffffffu, kB, 2);
        qA += __shfl_xor_sync(0xffffffffu, qA, 1); qA += __shfl_xor_sync(0xffffffffu, qA, 2);
        qB += __shfl_xor_sync(0xffffffffu, qB, 1); qB += __shfl_xor_sync(0xffffffffu, qB, 2);
        {
          const bool wr = mbar_wait(&ready[s], ph);
          if (!__all_sync(0xffffffffu, wr) || *(volatile int *)s_abort) {
            fail();
            break;
          }
        }
        const float *sa = reinterpret_cast<const float *>(st + lay.a);
        const float *scr = reinterpret_cast<const float *>(st + lay.scr);
        const float *sW = scr, *sCk = scr + 3 * L, *sCq = sCk + RB, *sScal = sCk + 3 * RB;
        const float gam = sScal[0], kq = sScal[1], alpha_t = sScal[2], beta_t = sa[L + 1];
        // d_t of rows rA and rB: beta_t (v_t - alpha_t S_{t-1} k_t)
        const float dA = beta_t * (lds_elem(st + lay.vt, rA, idt) - alpha_t * fmaf(gam, kA, sCk[rA]));
        const float dB = beta_t * (lds_elem(st + lay.vt, rB, idt) - alpha_t * fmaf(gam, kB, sCk[rB]));
        if (lw < 4 && t4 == 0) {
          orow[rA] = fmaf(alpha_t, fmaf(gam, qA, sCq[rA]), dA * kq);
          orow[rB] = fmaf(alpha_t, fmaf(gam, qB, sCq[rB]), dB * kq);
        }
        const float sc = alpha_t * gam;
#pragma unroll
        for (int bk = 0; bk < NBH; ++bk) {
          xa[bk].x *= sc; xa[bk].y *= sc; xa[bk].z *= sc; xa[bk].w *= sc;
          xb[bk].x *= sc; xb[bk].y *= sc; xb[bk].z *= sc; xb[bk].w *= sc;
        }
        for (int j0 = 0; j0 <= p; j0 += 8) {
          // records j0 + t and j0 + t + 4: ring records below p (weight
          // alpha_t G_j), this token at p (weight 1), none past p (weight 0,
          // its key read from k_t so nothing stale enters)
          const int ja = j0 + t4, jb = ja + 4;
          auto val = [&](int j, int r, float d_cur) -> float {
            if (j < p) return alpha_t * sW[j] * lds_elem(sd, j * RB + r, rdt);
            return j == p ? d_cur : 0.f;
          };
          uint32_t ah[4], al[4];
          split_tf32(val(ja, rA, dA), ah[0], al[0]);
          split_tf32(val(ja, rB, dB), ah[1], al[1]);
          split_tf32(val(jb, rA, dA), ah[2], al[2]);
          split_tf32(val(jb, rB, dB), ah[3], al[3]);
          auto key = [&](int j, int col) -> float {
            return j < p ? lds_elem(sk, j * DK + col, rdt) : lds_elem(skt, col, idt);
          };
#pragma unroll
          for (int bk = 0; bk < NBH; ++bk) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int col = cb + 16 * bk + 4 * (g8 >> 1) + (g8 & 1) + 2 * hf;  // column of tile index n = g
              float d[4] = {hf ? xa[bk].z : xa[bk].x, hf ? xa[bk].w : xa[bk].y, hf ? xb[bk].z : xb[bk].x,
                            hf ? xb[bk].w : xb[bk].y};
              if constexpr (sizeof(RT) == 2 && sizeof(IT) == 2) {
                const uint32_t bb[2] = {__float_as_uint(key(ja, col)), __float_as_uint(key(jb, col))};
                mma_tf32(d, ah, bb);
                mma_tf32(d, al, bb);
              } else {
                uint32_t bh[2], bl[2];
                split_tf32(key(ja, col), bh[0], bl[0]);
                split_tf32(key(jb, col), bh[1], bl[1]);
                mma_tf32(d, ah, bh);
                mma_tf32(d, al, bh);
                mma_tf32(d, ah, bl);
              }
              if (hf) {
                xa[bk].z = d[0]; xa[bk].w = d[1]; xb[bk].z = d[2]; xb[bk].w = d[3];
              } else {
                xa[bk].x = d[0]; xa[bk].y = d[1]; xb[bk].x = d[2]; xb[bk].y = d[3];
              }
            }
          }
        }
        TC *ckg = static_cast<TC *>(a.ckpt) + ((size_t)slot * a.H + h) * (DV * DK) + (size_t)row_off * DK;
#pragma unroll
        for (int bk = 0; bk < NBH; ++bk) {
          const size_t offA = (size_t)rA * DK + cb + 16 * bk + 4 * t4, offB = (size_t)rB * DK + cb + 16 * bk + 4 * t4;
          const float fa[4] = {xa[bk].x, xa[bk].y, xa[bk].z, xa[bk].w};
          const float fb[4] = {xb[bk].x, xb[bk].y, xb[bk].z, xb[bk].w};
          if constexpr (sizeof(TC) == 4) {
            st_vec(ckg + offA, V::pack(fa));
            st_vec(ckg + offB, V::pack(fb));
          } else {
            st_vec2(ckg + offA, LpVec<__half>::pack(fa));
            st_vec2(ckg + offB, LpVec<__half>::pack(fb));
          }
        }
        mbar_arrive(&rec_empty[s]);
        continue;
      }
    }
    // the checkpoint rows of this thread: held in registers for the fold of
    // a CUDA-core flush; with the tensor-core flush (a branch of its own)
    // they are read row by row as the products need them
    constexpr int VH = MMAF ? 1 : VPT;
    uint4 raw[VH][CPR];
    const uint4 *ck = reinterpret_cast<const uint4 *>(ck_slots + (size_t)c * CKB);
    if constexpr (!MMAF) {
#pragma unroll
      for (int r = 0; r < VPT; ++r)
#pragma unroll
        for (int i = 0; i < CPR; ++i) raw[r][i] = ck[(row0 + r * RPP) * NCH + cv + G * i];
      mbar_arrive(&ck_empty[c]);
    }

    const size_t unit = (size_t)slot * a.H + h;
    const float *sa = reinterpret_cast<const float *>(st + lay.a);
    float *scr = reinterpret_cast<float *>(st + lay.scr);
    const float *sW = scr, *sCk = scr + 3 * L, *sCq = sCk + RB;
    float *sDt = scr + 3 * L + 2 * RB;
    const float *sScal = sDt + RB;
    const unsigned char *sk = st + lay.k, *skt = st + lay.kt, *sq = st + lay.q, *sd = st + lay.d;

    // S_ckpt k_t and S_ckpt q_t for this thread's rows
    float ktc[CPR][E], qc[CPR][E];
#pragma unroll
    for (int i = 0; i < CPR; ++i) {
      lds_cols<E>(skt, (cv + G * i) * E, idt, ktc[i]);
      lds_cols<E>(sq, (cv + G * i) * E, idt, qc[i]);
    }
    float part[2 * VPT];
#pragma unroll
    for (int r = 0; r < VPT; ++r) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int i = 0; i < CPR; ++i) {
        float f[E];
        V::unpack(MMAF ? ck[(row0 + r * RPP) * NCH + cv + G * i] : raw[MMAF ? 0 : r][i], f);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          s0 = fmaf(f[e], ktc[i][e], s0);
          s1 = fmaf(f[e], qc[i][e], s1);
        }
      }
      part[r] = s0;
      part[VPT + r] = s1;
    }
    if constexpr (MMAF) mbar_arrive(&ck_empty[c]);
    group_reduce<2 * VPT, G>(part, lane);
    {
      const bool wr = mbar_wait(&ready[s], ph);
      if (!__all_sync(0xffffffffu, wr) || *(volatile int *)s_abort) {
        fail();
        break;
      }
    }
    // the lane holding row r's S_ckpt k_t and the one holding its S_ckpt q_t
    // differ in lane bit G/2
    const float gam = sScal[0], kq = sScal[1], alpha_t = sScal[2], beta_t = sa[L + 1];
    const int vi = group_reduce_index<2 * VPT, G>(lane);
    const bool isK = vi < VPT;
    const int rrow = row0 + (isK ? vi : vi - VPT) * RPP;
    const float A = fmaf(gam, part[0], isK ? sCk[rrow] : sCq[rrow]);  // S_{t-1} k_t or S_{t-1} q_t
    const float d_t = isK ? beta_t * (lds_elem(st + lay.vt, rrow, idt) - alpha_t * A) : 0.f;
    const float d_pair = __shfl_xor_sync(0xffffffffu, d_t, G / 2);
    const bool wr = group_reduce_writer<2 * VPT, G>(lane);
    if (!flush) {
      if (wr) {
        if (isK)
          store1(a.ring_v, (unit * L + p) * DV + row_off + rrow, rdt, d_t);
        else
          orow[rrow] = fmaf(alpha_t, A, d_pair * kq);
      }
      if (lw == NCW - 1 && half == 0) {
        // append this token's key (rounded to the ring type) and gate, once per head
        for (int cc = lane; cc < DK / 8; cc += 32) {
          float f[8];
          lds_cols<8>(skt, cc * 8, idt, f);
          store8(a.ring_k, (unit * L + p) * DK + cc * 8, rdt, f);
        }
        if (lane == 0) a.ring_a[unit * L + p] = sa[L];
      }
    } else {
      if (wr && isK) sDt[rrow] = d_t;
      __syncwarp();
      TC *ckg = static_cast<TC *>(a.ckpt) + unit * (DV * DK) + (size_t)row_off * DK;
      const float scale0 = alpha_t * gam;
      float f[VPT][CPR][E];
#pragma unroll
      for (int r = 0; r < VPT; ++r)
#pragma unroll
        for (int i = 0; i < CPR; ++i) {
          V::unpack(raw[r][i], f[r][i]);
#pragma unroll
          for (int e = 0; e < E; ++e) f[r][i][e] *= scale0;
        }
#pragma unroll 4
      for (int j = 0; j < p; ++j) {
        float kk[CPR][E];
#pragma unroll
        for (int i = 0; i < CPR; ++i) lds_cols<E>(sk, j * DK + (cv + G * i) * E, rdt, kk[i]);
        const float wj = alpha_t * sW[j];
#pragma unroll
        for (int r = 0; r < VPT; ++r) {
          const float dd = wj * lds_elem(sd, j * RB + row0 + r * RPP, rdt);
#pragma unroll
          for (int i = 0; i < CPR; ++i)
#pragma unroll
            for (int e = 0; e < E; ++e) f[r][i][e] = fmaf(dd, kk[i][e], f[r][i][e]);
        }
      }
      float po[VPT];
#pragma unroll
      for (int r = 0; r < VPT; ++r) {
        const float dd = sDt[row0 + r * RPP];
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < CPR; ++i) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            f[r][i][e] = fmaf(dd, ktc[i][e], f[r][i][e]);
            acc = fmaf(f[r][i][e], qc[i][e], acc);
          }
          st_vec(ckg + (size_t)(row0 + r * RPP) * DK + (cv + G * i) * E, V::pack(f[r][i]));
        }
        po[r] = acc;
      }
      group_reduce<VPT, G>(po, lane);
      if (group_reduce_writer<VPT, G>(lane)) orow[row0 + group_reduce_index<VPT, G>(lane) * RPP] = po[0];
    }
    mbar_arrive(&rec_empty[s]);
  }
}

template <int DV, int DK, typename TC, typename RT, typename IT, int NCW, int NSPLIT, int LMAX, int CPR, int NGRP,
          int MINB>
static cudaError_t launch_gdn_l(const KArgs &a, cudaStream_t s) {
  auto kern = gdn_replay_kernel<DV, DK, TC, RT, IT, NCW, NSPLIT, LMAX, CPR, NGRP, MINB>;
  constexpr int threads = NGRP * NCW * 32 + 64;
  const size_t ckb = (size_t)(DV / NSPLIT) * DK * sizeof(TC);
  const size_t rb = gdn_rec(DV / NSPLIT, DK, (int)sizeof(RT), (int)sizeof(IT), a.L).bytes;
  // one CTA per SM: a checkpoint slot per group, two record slots per group
  static const int one_cta[][3] = {{1, NGRP, 2 * NGRP}, {1, 2, 4}, {1, 2, 3}, {1, 1, 2}};
  RingPlan plan;
  cudaError_t e = plan_rings(reinterpret_cast<const void *>(kern), threads, ckb, rb, gdn_head, a.B * a.H * NSPLIT,
                             &plan, MINB == 1 ? one_cta : nullptr, 4);
  if (e != cudaSuccess) return e;
  kern<<<plan.grid, threads, plan.smem, s>>>(a, plan.nsr, plan.nsc);
  return cudaGetLastError();
}

// the common short windows get a kernel unrolled for L <= 16
template <int DV, int DK, typename TC, typename RT, typename IT, int NCW, int NSPLIT, int CPR = 1, int NGRP = 1,
          int MINB = 2>
static cudaError_t launch_gdn(const KArgs &a, cudaStream_t s) {
  return a.L <= 16 ? launch_gdn_l<DV, DK, TC, RT, IT, NCW, NSPLIT, 16, CPR, NGRP, MINB>(a, s)
                   : launch_gdn_l<DV, DK, TC, RT, IT, NCW, NSPLIT, RS_MAX_L, CPR, NGRP, MINB>(a, s);
}

template <typename TC, typename RT, typename IT>
static LaunchFn find_gdn_t(int d_v, int d_k) {
  constexpr bool f32 = sizeof(TC) == 4;
  if (d_v == 16 && d_k == 32) return launch_gdn<16, 32, TC, RT, IT, f32 ? 4 : 2, 1>;
  // 64-row units: two groups of four warps per CTA (measured 100.6 us against
  // 105.7 for one group of eight at batch 256, 32 heads of 128 x 128)
  if (d_v == 64 && d_k == 128) return launch_gdn<64, 128, TC, RT, IT, 4, 1, f32 ? 2 : 1, 2>;
  if (d_v == 128 && d_k == 128) return launch_gdn<128, 128, TC, RT, IT, 4, 2, f32 ? 2 : 1, 2>;
  return nullptr;
}

template <typename TC>
static LaunchFn find_gdn_c(int d_v, int d_k, int ring_dtype, int in_dtype) {
  if (ring_dtype == kF16)
    return in_dtype == kF32 ? find_gdn_t<TC, __half, float>(d_v, d_k) : find_gdn_t<TC, __half, __nv_bfloat16>(d_v, d_k);
  if (ring_dtype == kF32)
    return in_dtype == kF32 ? find_gdn_t<TC, float, float>(d_v, d_k) : find_gdn_t<TC, float, __nv_bfloat16>(d_v, d_k);
  return nullptr;
}

LaunchFn find_gdn(int d_v, int d_k, int ckpt_dtype, int ring_dtype, int in_dtype) {
  if (ckpt_dtype == kF32) return find_gdn_c<float>(d_v, d_k, ring_dtype, in_dtype);
  if (ckpt_dtype == kF16) return find_gdn_c<__half>(d_v, d_k, ring_dtype, in_dtype);
  return nullptr;
}

}  // namespace rs
