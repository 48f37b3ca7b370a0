// ReplaySSM Mamba-2 cached decode step: non-flush and flush rows in one launch.
//
// Sources:
//   [Ghana] S. Ghana, "ReplaySSM: an SSM decoder that writes its state once
//           every 16 tokens", §The identity and §Output without a state.
//   [PR48792] vLLM PR 48792, "[Kernel] ReplaySSM: cache SSM inputs for faster
//           Gated DeltaNet standard decode", §CUDA graphs and continuous
//           batching (the flush flag is per-row runtime data).
//
// A work unit is one (row b, head h).  With p = write_pos[b] ring records held
// and the current token as record p (0-based), w_j = prod_{l=j+1..p} alpha_l
// and gamma = prod_{l=0..p} alpha_l:
//   non-flush: o = gamma * (S_ckpt q) + sum_{j<=p} w_j (k_j . q) v_j, and the
//              record (alpha, v, k) is copied into ring slot p;
//   flush:     S_new = gamma * S_ckpt + sum_{j<=p} w_j v_j k_j^T, o = S_new q
//              from the fp32 registers, S_new stored (cast) over S_ckpt.
//
// Persistent, warp-specialised kernel, two CTAs per SM.  A producer warp
// streams each unit's checkpoint into a checkpoint slot with one 1-D bulk
// copy (cp.async.bulk, completion counted on an mbarrier) and its ring
// records, this token's k, v, q and the decays into a record slot with
// per-lane cp.async.  It prefetches the per-row slot, cursor and flag 32
// units ahead, so no dependent global load sits on the streaming path.  A
// read-copy kernel splits each checkpoint slot in two: a non-flush row's
// half-size read copy fills one half-slot, a flush row's fp32 rows two.
// Consumer groups (two groups of four warps for the 64 x 128 fp32 layer)
// take alternate units: a group waits for its unit, takes its share of the
// checkpoint into registers (freeing that slot for the next load at once),
// computes from the record slot and releases it.  The step is bound by
// instruction issue as much as by bandwidth, so the per-warp fixed costs of a
// unit are paid by four warps rather than eight; with the window warp (WW)
// the window's weights, key dots and per-row sums move off the consumers
// entirely, and the consumer warps run without a named barrier.  The units a
// CTA owns are strided across the batch, so the ~1/L flush rows (which also
// write their state) spread evenly over the CTAs.  Every wait is bounded: on
// a timeout the kernel reports RS_DERR_TIMEOUT, drains its own copies and
// returns.
// The per-step products stay on the CUDA cores (a bandwidth-bound GEMV, about
// 0.6 FLOP/byte); the flush fold of an fp32 or fp16 checkpoint, a rank-(p+1) update of
// the whole state held in registers, runs on the tensor cores.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "replayssm.h"

namespace rs {


// Shared memory holds two rings: checkpoint slots (the 32 KiB-class state
// block of a unit, released as soon as the consumers hold it in registers)
// and record slots (ring records, query, decays, per-unit metadata and
// scratch, released when the unit is done).  Small record slots are cheap, so
// there are more of them, and the checkpoint slots turn over at the speed of
// the memory system rather than of the arithmetic.
struct M2Rec {
  uint32_t k, v, q, a, meta, scr, scl, bytes;
};

// scl_bytes: row scales of an E4M3 read copy (0 for other kernels)
__host__ __device__ inline M2Rec m2_rec(int DV, int DK, int rec_es, int L, int scl_bytes = 0) {
  M2Rec s;
  uint32_t o = 0;
  s.k = o;    o = align128(o + L * DK * rec_es);   // records 0..p, current token at p
  s.v = o;    o = align128(o + L * DV * rec_es);
  s.q = o;    o = align128(o + DK * rec_es);
  s.a = o;    o = align128(o + L * 4);             // decays of records 0..p
  s.meta = o; o = align128(o + 36);                // slot, p, flush, status, read-copy parts, unit
  s.scr = o;  o = align128(o + (2 * L + 2 * DV + 4) * 4);  // w_j, k_j.q, row dots, gamma, window term
  s.scl = o;  o = align128(o + scl_bytes);
  s.bytes = o;
  return s;
}

// barriers full/rec_empty[nsr], ck_empty[NP nsc] (a read-copy kernel splits
// each checkpoint slot into NP parts: two for a 16-bit read copy, four for
// E4M3) and the abort flag
template <int NP>
__host__ __device__ inline uint32_t m2_head(int nsr, int nsc) { return align128(8 * (2 * nsr + NP * nsc) + 16); }
// with a window warp: one more barrier per record slot (window terms ready)
template <int NP>
__host__ __device__ inline uint32_t m2_head_ww(int nsr, int nsc) { return align128(8 * (3 * nsr + NP * nsc) + 16); }


// LMAX bounds the buffer length at compile time (L <= LMAX): loops over a
// window's records unroll to a fixed count with predicated bodies.
// TL is the read-copy type of a two-precision checkpoint (TL == TC: one copy):
// fp16 or bf16, or E4M3 (__nv_fp8_e4m3) with a power-of-two scale per state
// row in a.lp_scale.
// GRP: group-shared keys and queries (k, q [B, G, d_k], ring_k [slots, G, L,
// d_k]); the window's k_j . q_t were computed once per group by
// mamba2_group_kq_kernel into a.kq, and non-flush units read those instead of
// key records.
// CPR: 16-byte checkpoint chunks a consumer lane holds per state row; its
// chunks are cv, cv + G, cv + 2G, ... so that a warp's loads of one chunk
// index cover whole 128-byte lines of the row.
// WW: a window warp computes, for each record slot as it lands, everything
// that does not touch the checkpoint -- the weights w_j and gamma, the dots
// k_j . q and the window term sum_j w_j (k_j . q) v_j of every state row --
// and signals the consumers on a second barrier.  The consumer warps then
// need no named barrier: a state row never leaves its warp.
template <int DV, int DK, typename TC, typename TL, typename RT, int NCW, int NGRP, int LMAX, bool GRP, int CPR,
          bool WW>
__global__ void __launch_bounds__(NGRP * NCW * 32 + (WW ? 64 : 32), 2)
    mamba2_replay_kernel(const KArgs a, int nsr, int nsc) {
  using V = CkVec<TC>;
  constexpr bool TWO = !std::is_same<TC, TL>::value;
  constexpr bool F8 = std::is_same<TL, __nv_fp8_e4m3>::value;
  constexpr int E = V::E;
  constexpr int NCH = DK / E;        // 16-byte chunks per state row
  constexpr int G = NCH / CPR;       // lanes per state row
  constexpr int NC = NCW * 32;       // consumer threads per group
  constexpr int RPP = NC / G;        // state rows per pass of a group
  constexpr int VPT = DV / RPP;      // state rows per consumer thread
  constexpr int RDT = Rec<RT>::kDtype;
  constexpr int RES = (int)sizeof(RT);
  constexpr int WINW = NGRP * NCW;   // warp index of the window warp (WW)
  constexpr int PROD = NGRP * NCW + (WW ? 1 : 0);  // warp index of the producer
  constexpr uint32_t CKB = DV * DK * (uint32_t)sizeof(TC);
  constexpr uint32_t CKB_LP = DV * DK * (uint32_t)sizeof(TL);
  // a read-copy kernel's checkpoint slot holds NPART read copies, or one
  // flush row's fp32 rows in NPART row blocks
  constexpr int NPART = TWO ? (int)(CKB / CKB_LP) : 1;
  constexpr int NPH = NPART > 2 ? NPART : 2;  // ck_empty barriers per slot in the head
  static_assert(NPART <= 4, "at most four parts per checkpoint slot");
  static_assert(!TWO || (E == 4 && (sizeof(TL) == 2 || F8)), "read copy: 16-bit or E4M3 under an fp32 checkpoint");
  // flush fold on the tensor cores: fp32 or fp16 checkpoint, one warp per 16
  // state rows
  constexpr bool MMAF = (std::is_same<TC, float>::value || std::is_same<TC, __half>::value) && DV == 16 * NCW &&
                        DK % 16 == 0;
  static_assert(G <= 32 && 32 % G == 0 && NCH % CPR == 0, "a state row must fit in one warp");
  static_assert(NC % G == 0 && DV % RPP == 0 && VPT >= 1 && VPT <= G, "bad tiling");
  static_assert(DK % 8 == 0 && DV % 8 == 0, "head dims must be multiples of 8");
  static_assert(!F8 || (MMAF && WW), "an E4M3 read copy runs with the window warp and the tensor-core fold");

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // per record slot: all bytes of a unit landed
  uint64_t *rec_empty = full + nsr;                     // per record slot: the unit is done
  uint64_t *ck_empty = rec_empty + nsr;                 // per checkpoint slot: consumers hold it in registers
  uint64_t *ready = ck_empty + NPH * nsc;               // per record slot: window terms written (WW)
  int *s_abort = reinterpret_cast<int *>(ready + (WW ? nsr : 0));
  const int L = a.L;
  const M2Rec lay = m2_rec(DV, DK, RES, L, F8 ? DV * 4 : 0);
  unsigned char *ck_slots = smem + (WW ? m2_head_ww<NPH>(nsr, nsc) : m2_head<NPH>(nsr, nsc));
  unsigned char *rec_slots = ck_slots + (size_t)nsc * CKB;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_units = a.B * a.H;
  const int stride = gridDim.x;
  // a wait that ran out: flag every warp to stop and report it
  auto fail = [&]() {
    if (lane == 0) {
      *(volatile int *)s_abort = 1;
      report(a.dev_err, kDerrTimeout);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < nsr; ++s) {
      mbar_init(&full[s], 33);       // 32 producer-lane cp.async arrivals + lane 0 (+ bulk bytes)
      mbar_init(&rec_empty[s], NC + (WW ? 32 : 0));  // every thread of the consuming group (+ window warp)
      if (WW) mbar_init(&ready[s], 32);
    }
    for (int c = 0; c < NPART * nsc; ++c) mbar_init(&ck_empty[c], NC);
    for (int s = 0; s < nsr; ++s) reinterpret_cast<int *>(rec_slots + (size_t)s * lay.bytes + lay.meta)[8] = -1;
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
        const int b = u / a.H;
        sl = __ldg(a.slot_idx + b);
        wp = __ldg(a.write_pos + b);
        fl = __ldg(a.is_flush + b);
      } else {
        sl = -1; wp = 0; fl = 0;
      }
    };
    int c_sl, c_wp, c_fl;
    int ps = 0, pc = 0;         // record and checkpoint slot of unit `it`
    uint32_t phs = 0, phc = 0;  // parity of it / nsr and it / nsc
    // read-copy kernels: a ring of NPART nsc parts (CKB_LP bytes each); a
    // non-flush row's read copy takes one, a flush row's fp32 rows take
    // NPART (row blocks of DV / NPART rows, in order); per part: used yet,
    // and the parity of its use count
    const int nhs = NPART * nsc;
    int hc = 0;
    uint32_t hused = 0, hpar = 0;
    fetch(blockIdx.x, c_sl, c_wp, c_fl);
    bool ok = true;
    for (int ub = blockIdx.x; ok && ub < n_units; ub += 32 * stride) {
      int n_sl, n_wp, n_fl;
      fetch(ub + 32 * stride, n_sl, n_wp, n_fl);  // next batch, in flight meanwhile
      for (int j = 0; j < 32; ++j) {
        const int u = ub + j * stride;
        if (u >= n_units) break;
        const int slot = __shfl_sync(0xffffffffu, c_sl, j);
        const int p = __shfl_sync(0xffffffffu, c_wp, j);
        const int fl = __shfl_sync(0xffffffffu, c_fl, j);
        const int s = ps, c = pc;
        int hp[4] = {-1, -1, -1, -1};  // parts of this unit (read-copy kernels)
        if constexpr (TWO) {
          if (slot >= 0 && slot < a.num_slots && p >= 0 && p < L) {
#pragma unroll
            for (int k = 0; k < NPART; ++k) {
              if (k == 0 || fl) {
                hp[k] = hc;
                hc = hc + 1 == nhs ? 0 : hc + 1;
              }
            }
          }
        }
        if (it >= nsr || (TWO ? hp[0] >= 0 : it >= nsc)) {
          int w = 1;
          if (lane == 0) {
            if (it >= nsr) w = mbar_wait(&rec_empty[s], phs ^ 1u) ? 1 : 0;
            if constexpr (TWO) {
#pragma unroll
              for (int k = 0; k < NPART; ++k) {
                const int h = hp[k];
                if (w && h >= 0 && ((hused >> h) & 1u)) w = mbar_wait(&ck_empty[h], ((hpar >> h) & 1u) ^ 1u) ? 1 : 0;
              }
            } else {
              if (w && it >= nsc) w = mbar_wait(&ck_empty[c], phc ^ 1u) ? 1 : 0;
            }
          }
          w = __shfl_sync(0xffffffffu, w, 0);
          if (!w || *(volatile int *)s_abort) {
            fail();
            ok = false;
            break;
          }
        }
        __syncwarp();
        if constexpr (TWO) {
#pragma unroll
          for (int k = 0; k < NPART; ++k) {
            if (hp[k] >= 0) {
              hused |= 1u << hp[k];
              hpar ^= 1u << hp[k];
            }
          }
        }
        const int b = u / a.H, h = u - (u / a.H) * a.H;
        const int status = slot < 0 ? kStatusPad
                           : slot >= a.num_slots ? kStatusBadSlot
                           : (p < 0 || p >= L) ? kStatusBadPos
                           : kStatusOk;
        unsigned char *st = rec_slots + (size_t)s * lay.bytes;
        int *meta = reinterpret_cast<int *>(st + lay.meta);
        if (status == kStatusOk) {
          // The checkpoint, the only large operand, is one bulk copy from lane
          // 0.  The small pieces -- ring records, this token's k, v, q and the
          // decays -- go as 16- and 4-byte cp.async over the 32 lanes: a bulk
          // copy carries a fixed cost of ~0.2 us that five small copies per
          // unit would pay five times.
          const size_t unit = (size_t)slot * a.H + h;
          if (lane == 0) {
            meta[0] = slot; meta[1] = p; meta[2] = fl; meta[3] = status;
            meta[4] = hp[0]; meta[5] = hp[1]; meta[6] = hp[2]; meta[7] = hp[3];
            meta[8] = u;
            const TC *ck32 = static_cast<const TC *>(a.ckpt) + unit * (DV * DK);
            if constexpr (TWO) {
              if (!fl) {
                // a two-precision non-flush row reads only the read copy
                mbar_expect_tx(&full[s], CKB_LP);
                bulk_load(ck_slots + (size_t)hp[0] * CKB_LP,
                          static_cast<const unsigned char *>(a.ckpt_lp) + unit * (size_t)CKB_LP, CKB_LP, &full[s],
                          pol_stream);
              } else {
                static_assert(CKB == NPART * CKB_LP, "an fp32 checkpoint fills NPART parts");
                mbar_expect_tx(&full[s], CKB);
#pragma unroll
                for (int k = 0; k < NPART; ++k)
                  bulk_load(ck_slots + (size_t)hp[k] * CKB_LP, ck32 + k * (DV / NPART) * DK, CKB_LP, &full[s],
                            pol_stream);
              }
            } else {
              mbar_expect_tx(&full[s], CKB);
              bulk_load(ck_slots + (size_t)c * CKB, ck32, CKB, &full[s], pol_stream);
            }
          }
          constexpr uint32_t kb = DK * RES, vb = DV * RES;
          constexpr int KC = kb / 16, VC = vb / 16;  // 16-byte chunks per k / v record
          // key and query of the unit: its own (per-head layout) or its group's
          const int kh = GRP ? h / (a.H / a.n_groups) : h;
          const size_t kunit = GRP ? (size_t)slot * a.n_groups + kh : unit;
          const unsigned char *rk = static_cast<const unsigned char *>(a.ring_k) + kunit * L * kb;
          const unsigned char *rv = static_cast<const unsigned char *>(a.ring_v) + unit * L * vb;
          const unsigned char *kin =
              static_cast<const unsigned char *>(a.k) + ((size_t)b * a.sk + (size_t)kh * DK) * RES;
          const unsigned char *vin =
              static_cast<const unsigned char *>(a.v) + ((size_t)b * a.sv + (size_t)h * DV) * RES;
          const unsigned char *qin =
              static_cast<const unsigned char *>(a.q) + ((size_t)b * a.sq + (size_t)kh * DK) * RES;
          if constexpr (!GRP && LMAX >= 32) {
            // Long windows: the ring records, this token's k, v and q, the
            // decays and an E4M3 copy's row scales as bulk copies, one piece
            // per lane (measured faster than 16-byte cp.async pieces at
            // L = 32, slower at L <= 16).  Decays past the last whole 16
            // bytes of the ring row (at most three) and this token's decay
            // go by cp.async.
            float *sa = reinterpret_cast<float *>(st + lay.a);
            const uint32_t rkb = (uint32_t)p * kb, rvb = (uint32_t)p * vb;
            const bool a16 = (L & 3) == 0 && (reinterpret_cast<uintptr_t>(a.ring_a) & 15) == 0;
            const int na = a16 ? (p & ~3) : 0;  // decays by bulk copy
            const bool scl = F8 && !fl;
            if (lane == 0) mbar_expect_tx(&full[s], rkb + rvb + 2 * kb + vb + na * 4 + (scl ? DV * 4 : 0));
            __syncwarp();
            if (lane == 1 && p > 0) bulk_load(st + lay.k, rk, rkb, &full[s], pol_stream);
            if (lane == 2) bulk_load(st + lay.k + rkb, kin, kb, &full[s], pol_stream);
            if (lane == 3 && p > 0) bulk_load(st + lay.v, rv, rvb, &full[s], pol_stream);
            if (lane == 4) bulk_load(st + lay.v + rvb, vin, vb, &full[s], pol_stream);
            if (lane == 5) bulk_load(st + lay.q, qin, kb, &full[s], pol_stream);
            if (lane == 6 && na > 0) bulk_load(sa, a.ring_a + unit * L, na * 4, &full[s], pol_stream);
            if (scl && lane == 7) bulk_load(st + lay.scl, a.lp_scale + unit * DV, DV * 4, &full[s], pol_stream);
            for (int jj = na + lane; jj < p; jj += 32) cp_async4(sa + jj, a.ring_a + unit * L + jj);
            if (lane == 31) cp_async4(sa + p, a.alpha + (size_t)b * a.H + h);
          } else {
            if (!GRP || fl) {
#pragma unroll
              for (int i = 0; i < (LMAX * KC + 31) / 32; ++i) {
                const int cc = lane + 32 * i;
                if (cc < (p + 1) * KC)
                  cp_async16(st + lay.k + cc * 16, (cc < p * KC ? rk + cc * 16 : kin + (cc - p * KC) * 16));
              }
            } else {
              // the group's k_j . q_t of the window, into the dots scratch of the slot
              float *ss = reinterpret_cast<float *>(st + lay.scr) + L;
              const float *kq = a.kq + ((size_t)b * a.n_groups + kh) * L;
#pragma unroll
              for (int i = 0; i < (LMAX + 31) / 32; ++i) {
                const int jj = lane + 32 * i;
                if (jj <= p) cp_async4(ss + jj, kq + jj);
              }
            }
#pragma unroll
            for (int i = 0; i < (LMAX * VC + 31) / 32; ++i) {
              const int cc = lane + 32 * i;
              if (cc < (p + 1) * VC)
                cp_async16(st + lay.v + cc * 16, (cc < p * VC ? rv + cc * 16 : vin + (cc - p * VC) * 16));
            }
            for (int cc = lane; cc < KC; cc += 32) cp_async16(st + lay.q + cc * 16, qin + cc * 16);
            float *sa = reinterpret_cast<float *>(st + lay.a);
#pragma unroll
            for (int i = 0; i < (LMAX + 31) / 32; ++i) {
              const int jj = lane + 32 * i;
              if (jj < p) cp_async4(sa + jj, a.ring_a + unit * L + jj);
            }
            if (lane == 31) cp_async4(sa + p, a.alpha + (size_t)b * a.H + h);
            if constexpr (F8) {
              // a non-flush row's read copy comes with its row scales
              if (!fl && lane < DV / 4) cp_async16(st + lay.scl + lane * 16, a.lp_scale + unit * DV + lane * 4);
            }
          }
        } else if (lane == 0) {
          meta[0] = slot; meta[1] = p; meta[2] = fl; meta[3] = status;
          meta[4] = -1; meta[5] = -1; meta[6] = -1; meta[7] = -1;
          meta[8] = u;
        }
        if (lane == 0) mbar_arrive(&full[s]);  // releases the meta words
        cp_async_arrive(&full[s]);
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
      c_sl = n_sl; c_wp = n_wp; c_fl = n_fl;
    }
    // drain: every copy this warp issued has landed before the CTA may exit
    if (lane == 0) {
      for (int k = it > nsr ? it - nsr : 0; k < it; ++k) mbar_wait(&full[k % nsr], (uint32_t)(k / nsr) & 1u);
    }
    __syncwarp();
    return;
  }

  if constexpr (WW) {
    if (warp == WINW) {
      // --------------------------------------------------------------- window
      // every unit of the CTA in order: weights w_j and gamma; on non-flush
      // units also c_j = w_j (k_j . q) and the window term y = sum_j c_j v_j
      constexpr int RPL = (DV + 31) / 32;  // state rows per lane of the window term
      int s = 0;
      uint32_t ph = 0;
      for (int it = 0;; ++it) {
        if (it && ++s == nsr) {
          s = 0;
          ph ^= 1u;
        }
        if (blockIdx.x + it * stride >= n_units) break;
        const bool w = mbar_wait(&full[s], ph);
        if (!__all_sync(0xffffffffu, w) || *(volatile int *)s_abort) {
          fail();
          break;
        }
        const unsigned char *st = rec_slots + (size_t)s * lay.bytes;
        const int4 m = *reinterpret_cast<const int4 *>(st + lay.meta);
        const int p = m.y, flush = m.z, status = m.w;
        if (status == kStatusOk) {
          const float *sa = reinterpret_cast<const float *>(st + lay.a);
          float *scr = reinterpret_cast<float *>(const_cast<unsigned char *>(st) + lay.scr);
          float *sW = scr, *sS = scr + L, *sGam = scr + 2 * L + DV, *sY = sGam + 4;
          const unsigned char *sk = st + lay.k, *sv = st + lay.v;
          // w_j = product of the decays after record j, gamma = product of all
          float x0 = lane <= p ? sa[lane] : 1.f;
          float x1 = lane + 32 <= p ? sa[lane + 32] : 1.f;
          suffix_scan64(x0, x1, lane, [](float x, float y) { return x * y; });
          const float n0 = __shfl_down_sync(0xffffffffu, x0, 1);
          const float n1 = __shfl_down_sync(0xffffffffu, x1, 1);
          const float hi0 = __shfl_sync(0xffffffffu, x1, 0);
          const float wv0 = lane == 31 ? hi0 : n0;
          const float wv1 = lane == 31 ? 1.f : n1;
          if (lane <= p) sW[lane] = wv0;
          if (LMAX > 32 && lane + 32 <= p) sW[lane + 32] = wv1;
          if (lane == 0) sGam[0] = x0;
          if (!flush) {
            if constexpr (GRP) {
              // the group's dots are in sS already
              if (lane <= p) sS[lane] *= wv0;
              if (LMAX > 32 && lane + 32 <= p) sS[lane + 32] *= wv1;
            } else {
              // k_j . q for j <= p, eight records per transposed reduction
              float q4[4];
              const int col = lane * 4;
              static_assert(DK <= 128, "one 4-column chunk of q per lane");
              if (col < DK) {
                lds_cols<4>(st + lay.q, col, RDT, q4);
              } else {
                q4[0] = q4[1] = q4[2] = q4[3] = 0.f;
              }
              uint2 qw = make_uint2(0u, 0u);  // the chunk as bf16 pairs
              if (RDT == kBF16 && col < DK) qw = *reinterpret_cast<const uint2 *>(st + lay.q + (size_t)col * 2);
#pragma unroll 1
              for (int j0 = 0; j0 <= p; j0 += 8) {
                float part[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                  const int j = j0 + r;
                  float acc = 0.f;
                  if (j <= p && col < DK) {
                    if constexpr (RDT == kBF16) {
                      // bf16 keys and query on the mixed-precision FMA, no widening
                      const uint2 kw = *reinterpret_cast<const uint2 *>(sk + ((size_t)j * DK + col) * 2);
                      acc = fma_bf16x2_acc(kw.x, qw.x, fma_bf16x2_acc(kw.y, qw.y, 0.f));
                    } else {
                      float kk[4];
                      lds_cols<4>(sk, j * DK + col, RDT, kk);
                      acc = fmaf(kk[0], q4[0], fmaf(kk[1], q4[1], fmaf(kk[2], q4[2], kk[3] * q4[3])));
                    }
                  }
                  part[r] = acc;
                }
                group_reduce<8, 32>(part, lane);
                const int j = j0 + group_reduce_index<8, 32>(lane);
                float wj = __shfl_sync(0xffffffffu, wv0, j & 31);
                if constexpr (LMAX > 32) {
                  const float w1 = __shfl_sync(0xffffffffu, wv1, j & 31);
                  if (j >= 32) wj = w1;
                }
                if (group_reduce_writer<8, 32>(lane) && j <= p) sS[j] = wj * part[0];
              }
            }
            __syncwarp();
            // y = sum_{j <= p} c_j v_j for this lane's state rows
            if (lane * RPL < DV) {
              if constexpr (RPL == 2 && RDT == kBF16) {
                // the lane's two rows as one bf16 pair, both sums in one
                // packed fp32 FMA
                float2 y = make_float2(0.f, 0.f);
#pragma unroll 4
                for (int j = 0; j <= p; ++j) {
                  const float cj = sS[j];
                  const uint32_t w = reinterpret_cast<const uint32_t *>(sv)[(j * DV) / 2 + lane];
                  y = ffma2(make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)),
                            make_float2(cj, cj), y);
                }
                sY[2 * lane] = y.x;
                sY[2 * lane + 1] = y.y;
              } else {
                float y[RPL];
#pragma unroll
                for (int e = 0; e < RPL; ++e) y[e] = 0.f;
#pragma unroll 4
                for (int j = 0; j <= p; ++j) {
                  const float cj = sS[j];
#pragma unroll
                  for (int e = 0; e < RPL; ++e) y[e] = fmaf(cj, lds_elem(sv, j * DV + lane * RPL + e, RDT), y[e]);
                }
#pragma unroll
                for (int e = 0; e < RPL; ++e) sY[lane * RPL + e] = y[e];
              }
            }
          }
          __syncwarp();
        }
        mbar_arrive(&ready[s]);
        mbar_arrive(&rec_empty[s]);
      }
      return;
    }
  }

  // ------------------------------------------------------------------ consumers
  // group g takes the CTA's units g, g + NGRP, ...; each group has its own
  // named barrier, so the groups run independently of each other
  const int grp = warp / NCW;
  const int lw = warp - grp * NCW;  // warp within the group
  const int ctid = tid - grp * NC;  // 0 .. NC-1
  const int row0 = ctid / G, cv = ctid - (ctid / G) * G;
  auto gsync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(NC) : "memory"); };
  // row and head of the unit, stepped instead of divided
  const int ustep = NGRP * stride;
  const int step_b = ustep / a.H, step_h = ustep - (ustep / a.H) * a.H;
  int b = (int)(blockIdx.x + grp * stride) / a.H;
  int h = (int)(blockIdx.x + grp * stride) - b * a.H;
  // slot indices and the full-barrier phase, stepped instead of divided
  int s = grp % nsr, c = grp % nsc;
  uint32_t ph = (uint32_t)(grp / nsr) & 1u;
  for (int it = grp; ; it += NGRP, h += step_h, b += step_b) {
    if (h >= a.H) {
      h -= a.H;
      ++b;
    }
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
    const int *slot_unit = reinterpret_cast<const int *>(rec_slots + (size_t)s * lay.bytes + lay.meta) + 8;
    if constexpr (WW) {
      // every warp waits for itself: no named barrier in this mode
      const bool w = mbar_wait_unit(&full[s], ph, slot_unit, u);
      if (!__all_sync(0xffffffffu, w) || *(volatile int *)s_abort) {
        fail();
        break;
      }
    } else {
      if (lane == 0 && !mbar_wait_unit(&full[s], ph, slot_unit, u)) *(volatile int *)s_abort = 1;
      gsync();
      if (*(volatile int *)s_abort) break;
    }

    const unsigned char *st = rec_slots + (size_t)s * lay.bytes;
    const int4 m = *reinterpret_cast<const int4 *>(st + lay.meta);
    const int slot = m.x, p = m.y, flush = m.z, status = m.w;
    float *orow = a.out + (size_t)b * a.so + (size_t)h * DV;
    if (status != kStatusOk) {
      for (int i = ctid; i < DV; i += NC) orow[i] = 0.f;
      if (ctid == 0 && status != kStatusPad) report(a.dev_err, status == kStatusBadSlot ? 1 : 2);
      if (!TWO) mbar_arrive(&ck_empty[c]);  // a read-copy kernel gave the unit no part
      mbar_arrive(&rec_empty[s]);
      continue;
    }
    const size_t unit = (size_t)slot * a.H + h;
    const float *sa = reinterpret_cast<const float *>(st + lay.a);
    float *scr = reinterpret_cast<float *>(const_cast<unsigned char *>(st) + lay.scr);
    float *sW = scr, *sS = scr + L, *sC = scr + 2 * L, *sGam = scr + 2 * L + DV, *sY = sGam + 4;
    const unsigned char *sk = st + lay.k, *sv = st + lay.v;
    // the unit's checkpoint slot; a read-copy kernel names its parts in the
    // metadata: the read copy in one, or a flush row's fp32 row blocks of
    // DV / NPART rows in NPART
    int hs[4] = {c, -1, -1, -1};
    if constexpr (TWO) {
      const int4 hm = *reinterpret_cast<const int4 *>(st + lay.meta + 16);
      hs[0] = hm.x; hs[1] = hm.y; hs[2] = hm.z; hs[3] = hm.w;
    }
    const unsigned char *ck_slot = ck_slots + (size_t)hs[0] * (TWO ? CKB_LP : CKB);
    // fp32 state row r of a flush row
    auto ck_row = [&](int r) -> const unsigned char * {
      if constexpr (TWO) {
        constexpr int RB = DV / NPART;  // rows per part
        const int k = r / RB;
        const int hk = k == 0 ? hs[0] : k == 1 ? hs[1] : k == 2 ? hs[2] : hs[3];
        return ck_slots + (size_t)hk * CKB_LP + (size_t)(r - k * RB) * DK * sizeof(TC);
      } else {
        return ck_slot + (size_t)r * DK * sizeof(TC);
      }
    };
    auto release_ck = [&]() {
      mbar_arrive(&ck_empty[hs[0]]);
      if constexpr (TWO) {
#pragma unroll
        for (int k = 1; k < NPART; ++k)
          if (hs[k] >= 0) mbar_arrive(&ck_empty[hs[k]]);
      }
    };

    // window weights w_j (suffix products of the decays) and gamma
    auto weights = [&]() {
      if (!WW && lw == 0) {
        float x0 = lane <= p ? sa[lane] : 1.f;
        float x1 = lane + 32 <= p ? sa[lane + 32] : 1.f;
        suffix_scan64(x0, x1, lane, [](float x, float y) { return x * y; });
        const float n0 = __shfl_down_sync(0xffffffffu, x0, 1);
        const float n1 = __shfl_down_sync(0xffffffffu, x1, 1);
        const float hi0 = __shfl_sync(0xffffffffu, x1, 0);
        if (lane <= p) sW[lane] = lane == 31 ? hi0 : n0;
        if (lane + 32 <= p) sW[lane + 32] = lane == 31 ? 1.f : n1;
        if (lane == 0) sGam[0] = x0;
      }
    };
    // WW: the window warp's weights and terms of this unit are in the slot
    auto window_ready = [&]() {
      const bool w = mbar_wait(&ready[s], ph);
      return __all_sync(0xffffffffu, w) && !*(volatile int *)s_abort;
    };

    float part[VPT];
    if (!flush) {
      if constexpr (F8) {
        // E4M3 read copy: a lane holds 16 codes (16 columns) of each of its
        // rows, G8 lanes a row; the row's power-of-two scale is applied to
        // the finished row dot
        constexpr int G8 = DK / 16;       // lanes per state row
        constexpr int RPP8 = NC / G8;     // rows per pass of the group
        constexpr int VPT8 = DV / RPP8;   // rows per lane
        static_assert(G8 <= 32 && 32 % G8 == 0 && DV % RPP8 == 0 && VPT8 >= 1 && VPT8 <= G8, "E4M3 tiling");
        const int r8 = ctid / G8, c8 = ctid - (ctid / G8) * G8;
        uint4 raw8[VPT8];
#pragma unroll
        for (int r = 0; r < VPT8; ++r) raw8[r] = reinterpret_cast<const uint4 *>(ck_slot)[(r8 + r * RPP8) * G8 + c8];
        release_ck();
        float q16[16];
        lds_cols<16>(st + lay.q, 16 * c8, RDT, q16);
        float p8[VPT8];
        static_assert(VPT8 % 2 == 0, "two rows per packed FMA");
#pragma unroll
        for (int r = 0; r < VPT8; r += 2) {
          // rows r and r + 1 in one packed FMA per column (each row's order
          // of accumulation: columns 3, 2, 1, 0 of every 4)
          const uint32_t wa[4] = {raw8[r].x, raw8[r].y, raw8[r].z, raw8[r].w};
          const uint32_t wb[4] = {raw8[r + 1].x, raw8[r + 1].y, raw8[r + 1].z, raw8[r + 1].w};
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            const float2 loa = e4m3x2_to_f2(wa[wi]), hia = e4m3x2_to_f2(wa[wi] >> 16);
            const float2 lob = e4m3x2_to_f2(wb[wi]), hib = e4m3x2_to_f2(wb[wi] >> 16);
            const float *qq = q16 + 4 * wi;
            acc = ffma2(make_float2(hia.y, hib.y), make_float2(qq[3], qq[3]), acc);
            acc = ffma2(make_float2(hia.x, hib.x), make_float2(qq[2], qq[2]), acc);
            acc = ffma2(make_float2(loa.y, lob.y), make_float2(qq[1], qq[1]), acc);
            acc = ffma2(make_float2(loa.x, lob.x), make_float2(qq[0], qq[0]), acc);
          }
          p8[r] = acc.x;
          p8[r + 1] = acc.y;
        }
        group_reduce<VPT8, G8>(p8, lane);
        if (!window_ready()) {
          fail();
          break;
        }
        if (group_reduce_writer<VPT8, G8>(lane)) {
          const int row = r8 + group_reduce_index<VPT8, G8>(lane) * RPP8;
          const float *scl = reinterpret_cast<const float *>(st + lay.scl);
          orow[row] = fmaf(sGam[0] * scl[row], p8[0], sY[row]);
        }
      } else {
        // take this thread's share of the checkpoint (the read copy of a
        // two-precision checkpoint) into registers and hand the slot straight
        // back to the producer
        using Raw = typename std::conditional<TWO, uint2, uint4>::type;
        Raw raw[VPT][CPR];
#pragma unroll
        for (int r = 0; r < VPT; ++r)
#pragma unroll
          for (int i = 0; i < CPR; ++i)
            raw[r][i] = reinterpret_cast<const Raw *>(ck_slot)[(row0 + r * RPP) * NCH + cv + G * i];
        release_ck();
        weights();
        float qv[CPR][E];
#pragma unroll
        for (int i = 0; i < CPR; ++i) lds_cols<E>(st + lay.q, (cv + G * i) * E, RDT, qv[i]);
        // s_j = k_j . q: a warp takes records four at a time; each lane holds
        // its 4-column chunk of q and accumulates four partial dots, and one
        // transposed reduction finishes the chunk (group-shared keys: the
        // producer brought the group's dots instead)
        if constexpr (!GRP && !WW) {
          constexpr int QPL = (DK + 127) / 128;  // 4-column chunks of q per lane
          float qq[QPL][4];
#pragma unroll
          for (int i = 0; i < QPL; ++i) {
            if (lane * 4 + i * 128 < DK) {
              lds_cols<4>(st + lay.q, lane * 4 + i * 128, RDT, qq[i]);
            } else {
              qq[i][0] = qq[i][1] = qq[i][2] = qq[i][3] = 0.f;
            }
          }
#pragma unroll
          for (int ci = 0; ci < (LMAX / 4 + NCW - 1) / NCW; ++ci) {
            const int ch = lw + ci * NCW;
            if (ch * 4 > p) break;
            float part4[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int j = ch * 4 + r;
              float acc = 0.f;
              if (j <= p) {
#pragma unroll
                for (int i = 0; i < QPL; ++i) {
                  const int cc = lane * 4 + i * 128;
                  if (cc < DK) {
                    float kk[4];
                    lds_cols<4>(sk, j * DK + cc, RDT, kk);
                    acc = fmaf(kk[0], qq[i][0], fmaf(kk[1], qq[i][1], fmaf(kk[2], qq[i][2], fmaf(kk[3], qq[i][3], acc))));
                  }
                }
              }
              part4[r] = acc;
            }
            group_reduce<4, 32>(part4, lane);
            if (group_reduce_writer<4, 32>(lane)) {
              const int j = ch * 4 + group_reduce_index<4, 32>(lane);
              if (j <= p) sS[j] = part4[0];
            }
          }
        }
        // checkpoint GEMV partials from the stage (two rows per packed FMA
        // when a thread holds an even number of rows)
        auto unpack_raw = [&](int r, int i, float (&f)[E]) {
          if constexpr (TWO) {
            LpVec<TL>::unpack(raw[r][i], f);
          } else {
            V::unpack(raw[r][i], f);
          }
        };
        if constexpr (VPT % 2 == 0) {
#pragma unroll
          for (int r = 0; r < VPT; r += 2) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < CPR; ++i) {
              float f0[E], f1[E];
              unpack_raw(r, i, f0);
              unpack_raw(r + 1, i, f1);
#pragma unroll
              for (int e = 0; e < E; ++e) acc = ffma2(make_float2(f0[e], f1[e]), make_float2(qv[i][e], qv[i][e]), acc);
            }
            part[r] = acc.x;
            part[r + 1] = acc.y;
          }
        } else {
#pragma unroll
          for (int r = 0; r < VPT; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < CPR; ++i) {
              float f[E];
              unpack_raw(r, i, f);
#pragma unroll
              for (int e = 0; e < E; ++e) acc = fmaf(f[e], qv[i][e], acc);
            }
            part[r] = acc;
          }
        }
        group_reduce<VPT, G>(part, lane);
        if constexpr (WW) {
          // o = gamma c + the window warp's sum_j w_j s_j v_j, by the lane that
          // finished the row
          if (!window_ready()) {
            fail();
            break;
          }
          if (group_reduce_writer<VPT, G>(lane)) {
            const int row = row0 + group_reduce_index<VPT, G>(lane) * RPP;
            orow[row] = fmaf(sGam[0], part[0], sY[row]);
          }
        } else {
          if (group_reduce_writer<VPT, G>(lane)) sC[row0 + group_reduce_index<VPT, G>(lane) * RPP] = part[0];
          gsync();
        }

        // o = gamma c + sum_j w_j s_j v_j, by one warp: a lane covers 8 output
        // rows (one 16-byte load of a v record) for every OG-th record, then
        // lanes sharing rows add up; the other warps append the record
        if (!WW && lw == 0) {
          constexpr int RG = DV / 8;   // 8-row groups
          constexpr int OG = 32 / RG;  // record groups
          static_assert(DV % 8 == 0 && 32 % RG == 0 && OG >= 1, "bad output layout");
          const int rg = lane % RG, og = lane / RG;
          float acc[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
          for (int i = 0; i < (LMAX + OG - 1) / OG; ++i) {
            const int j = og + i * OG;
            if (j <= p) {
              const float cj = sW[j] * sS[j];
              float vv[8];
              lds_cols<8>(sv, j * DV + rg * 8, RDT, vv);
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[e] = fmaf(cj, vv[e], acc[e]);
            }
          }
#pragma unroll
          for (int off = RG; off < 32; off <<= 1) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
          }
          if (og == 0) {
            const float gam = sGam[0];
#pragma unroll
            for (int e = 0; e < 8; ++e) orow[rg * 8 + e] = fmaf(gam, sC[rg * 8 + e], acc[e]);
          }
        }
      }
      // append the current record (k, v verbatim, alpha) at ring slot p; a
      // group-shared key was appended by the group's dot kernel
      constexpr int KCH = GRP ? 0 : DK * RES / 16, VCH = DV * RES / 16;
      constexpr int APP0 = (NCW > 1 && !WW) ? 32 : 0;  // warp 0 is busy with the output
      for (int c = ctid - APP0; c >= 0 && c < KCH + VCH; c += NC - APP0) {
        if (c < KCH) {
          const uint4 x = reinterpret_cast<const uint4 *>(sk + (size_t)p * DK * RES)[c];
          reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.ring_k) + (unit * L + p) * DK * RES)[c] = x;
        } else {
          const uint4 x = reinterpret_cast<const uint4 *>(sv + (size_t)p * DV * RES)[c - KCH];
          reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.ring_v) + (unit * L + p) * DV * RES)[c - KCH] = x;
        }
      }
      if (ctid == NC - 1) a.ring_a[unit * L + p] = sa[p];
    } else if constexpr (MMAF) {
      // Flush on the tensor cores.  Warp lw holds state rows rA = 16 lw + g
      // and rB = rA + 8 in accumulator layout: four consecutive columns per
      // 16-column block (columns 4t, 4t+1 form one 8-column tile, 4t+2, 4t+3
      // the other).  The window folds in as a rank-(p+1) product, m16n8k8
      // tf32 with each weighted value split into two tf32 terms (the 16-bit
      // keys are exact), so S_new keeps fp32 accuracy.
      constexpr int NB = DK / 16;
      const int g8 = lane >> 2, t4 = lane & 3;
      const int rA = 16 * lw + g8, rB = rA + 8;
      float4 xa[NB], xb[NB];
      // four consecutive checkpoint elements of a state row, widened to fp32
      auto ld4 = [&](int r, int col) -> float4 {
        if constexpr (sizeof(TC) == 4) {
          return *reinterpret_cast<const float4 *>(ck_row(r) + col * 4);
        } else {
          float f[4];
          LpVec<__half>::unpack(*reinterpret_cast<const uint2 *>(ck_row(r) + col * 2), f);
          return make_float4(f[0], f[1], f[2], f[3]);
        }
      };
#pragma unroll
      for (int bk = 0; bk < NB; ++bk) {
        xa[bk] = ld4(rA, 16 * bk + 4 * t4);
        xb[bk] = ld4(rB, 16 * bk + 4 * t4);
      }
      release_ck();
      if constexpr (WW) {
        if (!window_ready()) {
          fail();
          break;
        }
      } else {
        weights();
        gsync();  // weights ready
      }
      const float gam = sGam[0];
#pragma unroll
      for (int bk = 0; bk < NB; ++bk) {
        xa[bk].x *= gam; xa[bk].y *= gam; xa[bk].z *= gam; xa[bk].w *= gam;
        xb[bk].x *= gam; xb[bk].y *= gam; xb[bk].z *= gam; xb[bk].w *= gam;
      }
      for (int j0 = 0; j0 <= p; j0 += 8) {
        // records j0 + t and j0 + t + 4 of the window; past p they weigh 0
        // (and read record 0, so no stale ring slot enters the product)
        const int ja = j0 + t4, jb = ja + 4;
        const int ra = ja <= p ? ja : 0, rb = jb <= p ? jb : 0;
        const float wa = ja <= p ? sW[ja] : 0.f, wb = jb <= p ? sW[jb] : 0.f;
        uint32_t ah[4], al[4];
        split_tf32(wa * lds_elem(sv, ra * DV + rA, RDT), ah[0], al[0]);
        split_tf32(wa * lds_elem(sv, ra * DV + rB, RDT), ah[1], al[1]);
        split_tf32(wb * lds_elem(sv, rb * DV + rA, RDT), ah[2], al[2]);
        split_tf32(wb * lds_elem(sv, rb * DV + rB, RDT), ah[3], al[3]);
#pragma unroll
        for (int bk = 0; bk < NB; ++bk) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int col = 16 * bk + 4 * (g8 >> 1) + (g8 & 1) + 2 * hf;  // column of tile index n = g
            float d[4] = {hf ? xa[bk].z : xa[bk].x, hf ? xa[bk].w : xa[bk].y, hf ? xb[bk].z : xb[bk].x,
                          hf ? xb[bk].w : xb[bk].y};
            if constexpr (sizeof(RT) == 2) {
              const uint32_t bb[2] = {__float_as_uint(lds_elem(sk, ra * DK + col, RDT)),
                                      __float_as_uint(lds_elem(sk, rb * DK + col, RDT))};
              mma_tf32(d, ah, bb);
              mma_tf32(d, al, bb);
            } else {
              uint32_t bh[2], bl[2];
              split_tf32(lds_elem(sk, ra * DK + col, RDT), bh[0], bl[0]);
              split_tf32(lds_elem(sk, rb * DK + col, RDT), bh[1], bl[1]);
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
      // store S_new (and its read copy), and o = S_new q from the same registers
      TC *ckg = static_cast<TC *>(a.ckpt) + unit * (DV * DK);
      float oA = 0.f, oB = 0.f;
      // an E4M3 read copy: the power-of-two scale of rows rA and rB from
      // their maxima (the four lanes t4 of a row group hold all its columns)
      int eA = 0, eB = 0;
      if constexpr (F8) {
        float mA = 0.f, mB = 0.f;
#pragma unroll
        for (int bk = 0; bk < NB; ++bk) {
          mA = fmaxf(mA, fmaxf(fmaxf(fabsf(xa[bk].x), fabsf(xa[bk].y)), fmaxf(fabsf(xa[bk].z), fabsf(xa[bk].w))));
          mB = fmaxf(mB, fmaxf(fmaxf(fabsf(xb[bk].x), fabsf(xb[bk].y)), fmaxf(fabsf(xb[bk].z), fabsf(xb[bk].w))));
        }
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 1));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 1));
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 2));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 2));
        eA = e4m3_row_exponent(mA);
        eB = e4m3_row_exponent(mB);
        if (t4 == 0) {
          a.lp_scale[unit * DV + rA] = ldexpf(1.f, eA);
          a.lp_scale[unit * DV + rB] = ldexpf(1.f, eB);
        }
      }
#pragma unroll
      for (int bk = 0; bk < NB; ++bk) {
        const size_t offA = (size_t)rA * DK + 16 * bk + 4 * t4, offB = (size_t)rB * DK + 16 * bk + 4 * t4;
        const float fa[4] = {xa[bk].x, xa[bk].y, xa[bk].z, xa[bk].w};
        const float fb[4] = {xb[bk].x, xb[bk].y, xb[bk].z, xb[bk].w};
        if constexpr (sizeof(TC) == 4) {
          st_vec(ckg + offA, V::pack(fa));
          st_vec(ckg + offB, V::pack(fb));
        } else {
          st_vec2(ckg + offA, LpVec<__half>::pack(fa));
          st_vec2(ckg + offB, LpVec<__half>::pack(fb));
        }
        if constexpr (F8) {
          unsigned char *lpg = static_cast<unsigned char *>(a.ckpt_lp) + unit * (DV * DK);
          *reinterpret_cast<uint32_t *>(lpg + offA) = e4m3_pack4(fa[0], fa[1], fa[2], fa[3], eA);
          *reinterpret_cast<uint32_t *>(lpg + offB) = e4m3_pack4(fb[0], fb[1], fb[2], fb[3], eB);
        } else if constexpr (TWO) {
          TL *lpg = static_cast<TL *>(a.ckpt_lp) + unit * (DV * DK);
          st_vec2(lpg + offA, LpVec<TL>::pack(fa));
          st_vec2(lpg + offB, LpVec<TL>::pack(fb));
        }
        float q4[4];
        lds_cols<4>(st + lay.q, 16 * bk + 4 * t4, RDT, q4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          oA = fmaf(fa[e], q4[e], oA);
          oB = fmaf(fb[e], q4[e], oB);
        }
      }
      oA += __shfl_xor_sync(0xffffffffu, oA, 1);
      oB += __shfl_xor_sync(0xffffffffu, oB, 1);
      oA += __shfl_xor_sync(0xffffffffu, oA, 2);
      oB += __shfl_xor_sync(0xffffffffu, oB, 2);
      if constexpr (WW) {
        if (t4 == 0) {
          orow[rA] = oA;
          orow[rB] = oB;
        }
      } else {
        if (t4 == 0) {
          sC[rA] = oA;
          sC[rB] = oB;
        }
        gsync();
        for (int i = ctid; i < DV; i += NC) orow[i] = sC[i];
      }
    } else {
      uint4 raw[VPT][CPR];
#pragma unroll
      for (int r = 0; r < VPT; ++r)
#pragma unroll
        for (int i = 0; i < CPR; ++i)
          raw[r][i] = reinterpret_cast<const uint4 *>(ck_row(row0 + r * RPP))[cv + G * i];
      release_ck();
      weights();
      float qv[CPR][E];
#pragma unroll
      for (int i = 0; i < CPR; ++i) lds_cols<E>(st + lay.q, (cv + G * i) * E, RDT, qv[i]);
      if constexpr (WW) {
        if (!window_ready()) {
          fail();
          break;
        }
      } else {
        gsync();  // weights ready
      }
      const float gam = sGam[0];
      TC *ckg = static_cast<TC *>(a.ckpt) + unit * (DV * DK);
      float f[VPT][CPR][E];
#pragma unroll
      for (int r = 0; r < VPT; ++r)
#pragma unroll
        for (int i = 0; i < CPR; ++i) {
          V::unpack(raw[r][i], f[r][i]);
#pragma unroll
          for (int e = 0; e < E; ++e) f[r][i][e] *= gam;
        }
#pragma unroll 4
      for (int j = 0; j <= p; ++j) {
        float kk[CPR][E];
#pragma unroll
        for (int i = 0; i < CPR; ++i) lds_cols<E>(sk, j * DK + (cv + G * i) * E, RDT, kk[i]);
        const float wj = sW[j];
#pragma unroll
        for (int r = 0; r < VPT; ++r) {
          const float vv = wj * lds_elem(sv, j * DV + row0 + r * RPP, RDT);
#pragma unroll
          for (int i = 0; i < CPR; ++i)
#pragma unroll
            for (int e = 0; e < E; ++e) f[r][i][e] = fmaf(vv, kk[i][e], f[r][i][e]);
        }
      }
#pragma unroll
      for (int r = 0; r < VPT; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < CPR; ++i) {
#pragma unroll
          for (int e = 0; e < E; ++e) acc = fmaf(f[r][i][e], qv[i][e], acc);
          const size_t off = (size_t)(row0 + r * RPP) * DK + (cv + G * i) * E;
          st_vec(ckg + off, V::pack(f[r][i]));
          if constexpr (TWO) {
            // the read copy: an independent rounding of the same fp32 matrix
            TL *lpg = static_cast<TL *>(a.ckpt_lp) + unit * (DV * DK);
            float g4[4] = {f[r][i][0], f[r][i][1], f[r][i][2], f[r][i][3]};
            st_vec2(lpg + off, LpVec<TL>::pack(g4));
          }
        }
        part[r] = acc;
      }
      group_reduce<VPT, G>(part, lane);
      if constexpr (WW) {
        if (group_reduce_writer<VPT, G>(lane)) orow[row0 + group_reduce_index<VPT, G>(lane) * RPP] = part[0];
      } else {
        if (group_reduce_writer<VPT, G>(lane)) sC[row0 + group_reduce_index<VPT, G>(lane) * RPP] = part[0];
        gsync();
        for (int i = ctid; i < DV; i += NC) orow[i] = sC[i];
      }
    }
    mbar_arrive(&rec_empty[s]);
  }
  if (tid == 0 && *(volatile int *)s_abort) report(a.dev_err, kDerrTimeout);
}

// Group-shared keys ([Ghana] §Output without a state: the released kernel
// reads precomputed k_j . q from a small kernel that runs once per group):
// one warp per (row, group) computes s_j = k_j . q_t for the window's records
// j < p and the current key (j = p) into a.kq[b, g, :], and on a non-flush
// row appends the current key to the group's ring at slot p.  Rows whose
// slot or cursor is out of range are left to the decode kernel to report.
template <int DK, typename RT>
__global__ void __launch_bounds__(256) mamba2_group_kq_kernel(const KArgs a) {
  constexpr int RES = (int)sizeof(RT);
  constexpr int RDT = Rec<RT>::kDtype;
  constexpr int KPL = (DK + 127) / 128;  // 4-column chunks per lane
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (pair >= a.B * a.n_groups) return;
  const int b = pair / a.n_groups, g = pair - (pair / a.n_groups) * a.n_groups;
  const int slot = __ldg(a.slot_idx + b), p = __ldg(a.write_pos + b), L = a.L;
  if (slot < 0 || slot >= a.num_slots || p < 0 || p >= L) return;
  const bool flush = __ldg(a.is_flush + b) != 0;
  const size_t kunit = (size_t)slot * a.n_groups + g;
  const unsigned char *rk = static_cast<const unsigned char *>(a.ring_k) + kunit * L * DK * RES;
  const unsigned char *kin = static_cast<const unsigned char *>(a.k) + ((size_t)b * a.sk + (size_t)g * DK) * RES;
  const unsigned char *qin = static_cast<const unsigned char *>(a.q) + ((size_t)b * a.sq + (size_t)g * DK) * RES;
  float qq[KPL][4];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int col = lane * 4 + i * 128;
    if (col < DK) {
      lds_cols<4>(qin, col, RDT, qq[i]);
    } else {
      qq[i][0] = qq[i][1] = qq[i][2] = qq[i][3] = 0.f;
    }
  }
  float *kq = a.kq + (size_t)pair * L;
  for (int j0 = 0; j0 <= p; j0 += 4) {
    float part[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = j0 + r;
      float acc = 0.f;
      if (j <= p) {
        const unsigned char *rec = j < p ? rk + (size_t)j * DK * RES : kin;
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
          const int col = lane * 4 + i * 128;
          if (col < DK) {
            float kk[4];
            lds_cols<4>(rec, col, RDT, kk);
            acc = fmaf(kk[0], qq[i][0], fmaf(kk[1], qq[i][1], fmaf(kk[2], qq[i][2], fmaf(kk[3], qq[i][3], acc))));
          }
        }
      }
      part[r] = acc;
    }
    group_reduce<4, 32>(part, lane);
    if (group_reduce_writer<4, 32>(lane)) {
      const int j = j0 + group_reduce_index<4, 32>(lane);
      if (j <= p) kq[j] = part[0];
    }
  }
  if (!flush) {
    constexpr int KC = DK * RES / 16;
    for (int c = lane; c < KC; c += 32)
      reinterpret_cast<uint4 *>(const_cast<unsigned char *>(rk) + (size_t)p * DK * RES)[c] =
          reinterpret_cast<const uint4 *>(kin)[c];
  }
}

template <int DV, int DK, typename TC, typename TL, typename RT, int NCW, int NGRP, int LMAX, bool GRP = false,
          int CPR = 1, bool WW = false>
static cudaError_t launch_mamba2_l(const KArgs &a, cudaStream_t s) {
  if (GRP) {
    mamba2_group_kq_kernel<DK, RT><<<(unsigned)(((size_t)a.B * a.n_groups + 7) / 8), 256, 0, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  auto kern = mamba2_replay_kernel<DV, DK, TC, TL, RT, NCW, NGRP, LMAX, GRP, CPR, WW>;
  constexpr int threads = NGRP * NCW * 32 + (WW ? 64 : 32);
  const size_t ckb = (size_t)DV * DK * sizeof(TC);
  constexpr bool F8 = std::is_same<TL, __nv_fp8_e4m3>::value;
  constexpr int NPH = !std::is_same<TC, TL>::value && sizeof(TC) / sizeof(TL) > 2 ? (int)(sizeof(TC) / sizeof(TL)) : 2;
  const size_t rb = m2_rec(DV, DK, (int)sizeof(RT), a.L, F8 ? DV * 4 : 0).bytes;
  RingPlan plan;
  cudaError_t e = plan_rings(reinterpret_cast<const void *>(kern), threads, ckb, rb,
                             WW ? m2_head_ww<NPH> : m2_head<NPH>, a.B * a.H, &plan);
  if (e != cudaSuccess) return e;
  kern<<<plan.grid, threads, plan.smem, s>>>(a, plan.nsr, plan.nsc);
  return cudaGetLastError();
}

// the common short windows get a kernel unrolled for L <= 16
// FINE: the window bound is the next of 8, 16, 32 or 64 above L (fewer
// predicated-off iterations for short and long windows), else 16 or 64
template <int DV, int DK, typename TC, typename RT, int NCW, int NGRP, typename TL = TC, int CPR = 1, bool FINE = false,
          bool WW = false>
static cudaError_t launch_mamba2(const KArgs &a, cudaStream_t s) {
  if (FINE && a.L <= 8) return launch_mamba2_l<DV, DK, TC, TL, RT, NCW, NGRP, 8, false, CPR, WW>(a, s);
  if (a.L <= 16) return launch_mamba2_l<DV, DK, TC, TL, RT, NCW, NGRP, 16, false, CPR, WW>(a, s);
  if (FINE && a.L <= 32) return launch_mamba2_l<DV, DK, TC, TL, RT, NCW, NGRP, 32, false, CPR, WW>(a, s);
  return launch_mamba2_l<DV, DK, TC, TL, RT, NCW, NGRP, RS_MAX_L, false, CPR, WW>(a, s);
}

// group-shared keys: the group dot kernel, then the decode
template <int DV, int DK, typename TC, typename RT, int NCW, int NGRP, int CPR = 1, bool WW = false>
static cudaError_t launch_mamba2_grp(const KArgs &a, cudaStream_t s) {
  return a.L <= 16 ? launch_mamba2_l<DV, DK, TC, TC, RT, NCW, NGRP, 16, true, CPR, WW>(a, s)
                   : launch_mamba2_l<DV, DK, TC, TC, RT, NCW, NGRP, RS_MAX_L, true, CPR, WW>(a, s);
}

}  // namespace rs
