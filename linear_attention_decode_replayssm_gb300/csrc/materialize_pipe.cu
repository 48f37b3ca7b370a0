// State materialisation on the decode's pipeline, for 64 x 128 Mamba-2 heads
// and 128 x 128 GDN heads (two 64-row units per head).
//
// Sources:
//   [Ghana] S. Ghana, "ReplaySSM: an SSM decoder that writes its state once
//           every 16 tokens", §What actually shipped (a cached prefix needs
//           the exact state at a block boundary; a separate kernel builds it
//           from the checkpoint and the ring) and §The identity (the state
//           after h records is gamma_h S_ckpt + sum_j gamma_{j+1:h} v_j k_j^T).
//   [PR48792] vLLM pull request 48792, §Core concept (Gated DeltaNet: the same
//           unroll over cached corrected values d_j with gate weights
//           exp(sum_{l>j} g_l)).
//
// It computes what materialize.cu computes, dst[dst_idx[b]] = the unroll of
// the checkpoint and the held records, rounded once, with the memory shape
// of a decode flush: a producer warp streams each unit's checkpoint rows
// (one bulk copy) and its held records and decays (per-lane cp.async) into
// slot rings; groups of four consumer warps take the units in turn, each
// warp 16 state rows in the accumulator layout of an m16n8k8 tile.  A warp
// scans the decays itself (products for Mamba-2, sums of log-gates then exp
// for GDN), folds the records on the tensor cores (each weighted value split
// into two tf32 terms, the keys split too when they are fp32) and stores its
// rows.  The checkpoint and the ring are only read.  Every wait is bounded.
#include "common.cuh"
#include "launch.h"

namespace rs {

namespace {

// Record slot of a unit: the held records (keys, values of the unit's rows),
// their decays, metadata and per-warp window weights.
struct MatRec {
  uint32_t k, v, a, meta, w, bytes;
};

__host__ __device__ inline MatRec mat_rec(int RB, int DK, int res, int L, int nwarps) {
  MatRec o;
  uint32_t x = 0;
  o.k = x;    x = align128(x + L * DK * res);
  o.v = x;    x = align128(x + L * RB * res);
  o.a = x;    x = align128(x + L * 4);
  o.meta = x; x = align128(x + 24);               // slot, held, dst, status, unit
  o.w = x;    x = align128(x + nwarps * 65 * 4);  // per consumer warp of a group: w_j, gamma
  o.bytes = x;
  return o;
}

// unit status above the error bits of a row the call skips
constexpr int kStatusErr = 1 << 8;

// barriers full/rec_empty[nsr], ck_empty[nsc] and the abort flag
__host__ __device__ inline uint32_t mat_head(int nsr, int nsc) { return align128(8 * (2 * nsr + nsc) + 16); }

}  // namespace

// RB state rows per unit (NSPLIT units per head), TC checkpoint type, RT ring
// type, GDNW: log-gate weights (exp of suffix sums) instead of decay products,
// NGRP consumer groups of four warps
template <int DV, int DK, int NSPLIT, typename TC, typename RT, bool GDNW, int NGRP>
// One CTA per SM: the state held in accumulator layout and the split
// operands fit in 112 registers without spilling (two CTAs of two groups
// would allow 96 -- 18 warps, five on one scheduler -- and measured slower);
// three groups and the producer are 13 warps, at most four a scheduler.
__global__ void __maxnreg__(112) mat_pipe_kernel(const rs_materialize_args a, int nsr, int nsc) {
  constexpr int RB = DV / NSPLIT;
  constexpr int NCW = RB / 16;  // consumer warps per group: 16 rows each
  constexpr int NC = NCW * 32;
  constexpr int PROD = NGRP * NCW;
  constexpr int NB = DK / 16;
  constexpr int RES = (int)sizeof(RT);
  constexpr int RDT = Rec<RT>::kDtype;
  constexpr uint32_t CKB = RB * DK * (uint32_t)sizeof(TC);
  constexpr int KC = DK * RES / 16, VC = RB * RES / 16;  // 16-byte chunks per key / value record
  static_assert(NCW == 4 && DK % 16 == 0 && RB * RES % 16 == 0 && DK * RES % 16 == 0, "64-row units");

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *rec_empty = full + nsr;
  uint64_t *ck_empty = rec_empty + nsr;
  int *s_abort = reinterpret_cast<int *>(ck_empty + nsc);
  const int L = a.L;
  const MatRec lay = mat_rec(RB, DK, RES, L, NCW);
  unsigned char *ck_slots = smem + mat_head(nsr, nsc);
  unsigned char *rec_slots = ck_slots + (size_t)nsc * CKB;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per_row = a.H * NSPLIT;
  const int n_units = a.B * per_row;
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
      mbar_init(&rec_empty[s], NC);
      reinterpret_cast<int *>(rec_slots + (size_t)s * lay.bytes + lay.meta)[4] = -1;
    }
    for (int c = 0; c < nsc; ++c) mbar_init(&ck_empty[c], NC);
    *s_abort = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == PROD) {
    // ----------------------------------------------------------------- producer
    const uint64_t pol_stream = policy_evict_first();
    // slot, held count and destination of the rows 32 units ahead, one unit per lane
    auto fetch = [&](int ub, int &sl, int &hd, int &ds) {
      const int u = ub + lane * stride;
      if (u < n_units) {
        const int b = u / per_row;
        sl = __ldg(a.slot_idx + b);
        hd = __ldg(a.held + b);
        ds = __ldg(a.dst_idx + b);
      } else {
        sl = -1; hd = 0; ds = -1;
      }
    };
    int it = 0, ps = 0, pc = 0;
    uint32_t phs = 0, phc = 0;
    int c_sl, c_hd, c_ds;
    fetch(blockIdx.x, c_sl, c_hd, c_ds);
    bool ok = true;
    for (int ub = blockIdx.x; ok && ub < n_units; ub += 32 * stride) {
      int n_sl, n_hd, n_ds;
      fetch(ub + 32 * stride, n_sl, n_hd, n_ds);
      for (int j = 0; j < 32; ++j) {
        const int u = ub + j * stride;
        if (u >= n_units) break;
        const int slot = __shfl_sync(0xffffffffu, c_sl, j);
        const int p = __shfl_sync(0xffffffffu, c_hd, j);
        const int dst = __shfl_sync(0xffffffffu, c_ds, j);
        if (it >= nsr || it >= nsc) {
          int w = 1;
          if (lane == 0) {
            if (it >= nsr) w = mbar_wait(&rec_empty[ps], phs ^ 1u) ? 1 : 0;
            if (w && it >= nsc) w = mbar_wait(&ck_empty[pc], phc ^ 1u) ? 1 : 0;
          }
          w = __shfl_sync(0xffffffffu, w, 0);
          if (!w || *(volatile int *)s_abort) {
            fail();
            ok = false;
            break;
          }
        }
        __syncwarp();
        const int rem = u - (u / per_row) * per_row;
        const int h = rem / NSPLIT, row_off = (rem - h * NSPLIT) * RB;
        // skipped row, or the error bits of a bad one above kStatusErr
        const int bad = (slot >= a.num_slots ? RS_DERR_SLOT : 0) | (dst >= a.num_dst ? RS_DERR_DST : 0) |
                        (p < 0 || p >= L ? RS_DERR_WRITE_POS : 0);
        const int status = (slot < 0 || dst < 0) ? kStatusPad : bad ? kStatusErr | bad : kStatusOk;
        unsigned char *st = rec_slots + (size_t)ps * lay.bytes;
        int *meta = reinterpret_cast<int *>(st + lay.meta);
        if (status == kStatusOk) {
          const size_t unit = (size_t)slot * a.H + h;
          if (lane == 0) {
            meta[0] = slot; meta[1] = p; meta[2] = dst; meta[3] = status; meta[4] = u;
            mbar_expect_tx(&full[ps], CKB);
            bulk_load(ck_slots + (size_t)pc * CKB,
                      static_cast<const TC *>(a.ckpt) + unit * (DV * DK) + (size_t)row_off * DK, CKB, &full[ps],
                      pol_stream);
          }
          const unsigned char *rk = static_cast<const unsigned char *>(a.ring_k) + unit * L * DK * RES;
          const unsigned char *rv = static_cast<const unsigned char *>(a.ring_v) + (unit * L * DV + row_off) * RES;
          for (int cc = lane; cc < p * KC; cc += 32) cp_async16(st + lay.k + cc * 16, rk + (size_t)cc * 16);
          for (int cc = lane; cc < p * VC; cc += 32) {
            const int jr = cc / VC, x = cc - jr * VC;  // record jr, its x-th chunk of the unit's rows
            cp_async16(st + lay.v + cc * 16, rv + ((size_t)jr * DV * RES + x * 16));
          }
          float *sa = reinterpret_cast<float *>(st + lay.a);
          for (int jj = lane; jj < p; jj += 32) cp_async4(sa + jj, a.ring_a + unit * L + jj);
        } else if (lane == 0) {
          meta[0] = slot; meta[1] = p; meta[2] = dst; meta[3] = status; meta[4] = u;
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
      c_sl = n_sl; c_hd = n_hd; c_ds = n_ds;
    }
    if (lane == 0) {
      for (int k = it > nsr ? it - nsr : 0; k < it; ++k) mbar_wait(&full[k % nsr], (uint32_t)(k / nsr) & 1u);
    }
    __syncwarp();
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int grp = warp / NCW, lw = warp - grp * NCW;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int rA = 16 * lw + g8, rB = rA + 8;
  int s = grp % nsr, c = grp % nsc;
  uint32_t ph = (uint32_t)(grp / nsr) & 1u;
  for (int it = grp;; it += NGRP) {
    if (it != grp) {
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
    unsigned char *st = rec_slots + (size_t)s * lay.bytes;
    const bool w = mbar_wait_unit(&full[s], ph, reinterpret_cast<const int *>(st + lay.meta) + 4, u);
    if (!__all_sync(0xffffffffu, w) || *(volatile int *)s_abort) {
      fail();
      break;
    }
    const int4 m = *reinterpret_cast<const int4 *>(st + lay.meta);
    const int slot = m.x, p = m.y, dst = m.z, status = m.w;
    if (status != kStatusOk) {
      if (lw == 0 && lane == 0 && status != kStatusPad) report(a.dev_err, status & ~kStatusErr);
      mbar_arrive(&ck_empty[c]);
      mbar_arrive(&rec_empty[s]);
      continue;
    }
    const int rem = u - (u / per_row) * per_row;
    const int h = rem / NSPLIT, row_off = (rem - h * NSPLIT) * RB;
    const unsigned char *sk = st + lay.k, *sv = st + lay.v;
    const float *sa = reinterpret_cast<const float *>(st + lay.a);
    // this warp's window weights: w_j = decay of the records after j, gamma =
    // decay of all p (Mamba-2: products; GDN: exp of sums of log-gates)
    float *sw = reinterpret_cast<float *>(st + lay.w) + lw * 65;
    {
      const float ident = GDNW ? 0.f : 1.f;
      float x0 = lane < p ? sa[lane] : ident;
      float x1 = lane + 32 < p ? sa[lane + 32] : ident;
      if constexpr (GDNW)
        suffix_scan64(x0, x1, lane, [](float x, float y) { return x + y; });
      else
        suffix_scan64(x0, x1, lane, [](float x, float y) { return x * y; });
      const float n0 = __shfl_down_sync(0xffffffffu, x0, 1);
      const float n1 = __shfl_down_sync(0xffffffffu, x1, 1);
      const float hi0 = __shfl_sync(0xffffffffu, x1, 0);
      float w0 = lane == 31 ? hi0 : n0, w1 = lane == 31 ? ident : n1;
      if constexpr (GDNW) {
        w0 = expf(w0);
        w1 = expf(w1);
        x0 = expf(x0);
      }
      sw[lane] = w0;
      sw[lane + 32] = w1;
      if (lane == 0) sw[64] = x0;
      __syncwarp();
    }
    // the warp's 16 rows in accumulator layout: rows rA and rB, four
    // consecutive columns 16 bk + 4 t4 .. + 3 of every 16-column block
    const unsigned char *ck_slot = ck_slots + (size_t)c * CKB;
    float4 xa[NB], xb[NB];
#pragma unroll
    for (int bk = 0; bk < NB; ++bk) {
      if constexpr (sizeof(TC) == 4) {
        xa[bk] = *reinterpret_cast<const float4 *>(ck_slot + ((size_t)rA * DK + 16 * bk + 4 * t4) * 4);
        xb[bk] = *reinterpret_cast<const float4 *>(ck_slot + ((size_t)rB * DK + 16 * bk + 4 * t4) * 4);
      } else {
        float f[4];
        LpVec<__half>::unpack(*reinterpret_cast<const uint2 *>(ck_slot + ((size_t)rA * DK + 16 * bk + 4 * t4) * 2), f);
        xa[bk] = make_float4(f[0], f[1], f[2], f[3]);
        LpVec<__half>::unpack(*reinterpret_cast<const uint2 *>(ck_slot + ((size_t)rB * DK + 16 * bk + 4 * t4) * 2), f);
        xb[bk] = make_float4(f[0], f[1], f[2], f[3]);
      }
    }
    mbar_arrive(&ck_empty[c]);
    const float gam = sw[64];
#pragma unroll
    for (int bk = 0; bk < NB; ++bk) {
      xa[bk].x *= gam; xa[bk].y *= gam; xa[bk].z *= gam; xa[bk].w *= gam;
      xb[bk].x *= gam; xb[bk].y *= gam; xb[bk].z *= gam; xb[bk].w *= gam;
    }
    // + sum_{j<p} w_j v_j k_j^T as m16n8k8 tf32 products over eight records
    for (int j0 = 0; j0 < p; j0 += 8) {
      // records j0 + t and j0 + t + 4; past p they weigh 0 (and read record 0)
      const int ja = j0 + t4, jb = ja + 4;
      const int ra = ja < p ? ja : 0, rb = jb < p ? jb : 0;
      const float wa = ja < p ? sw[ja] : 0.f, wb = jb < p ? sw[jb] : 0.f;
      uint32_t ah[4], al[4];
      split_tf32(wa * lds_elem(sv, ra * RB + rA, RDT), ah[0], al[0]);
      split_tf32(wa * lds_elem(sv, ra * RB + rB, RDT), ah[1], al[1]);
      split_tf32(wb * lds_elem(sv, rb * RB + rA, RDT), ah[2], al[2]);
      split_tf32(wb * lds_elem(sv, rb * RB + rB, RDT), ah[3], al[3]);
#pragma unroll
      for (int bk = 0; bk < NB; ++bk) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int col = 16 * bk + 4 * (g8 >> 1) + (g8 & 1) + 2 * hf;  // column of tile index n = g8
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
    // the state, rounded once to the checkpoint type, into the destination
    TC *outp = static_cast<TC *>(a.dst) + ((size_t)dst * a.H + h) * (DV * DK) + (size_t)row_off * DK;
#pragma unroll
    for (int bk = 0; bk < NB; ++bk) {
      const size_t offA = (size_t)rA * DK + 16 * bk + 4 * t4, offB = (size_t)rB * DK + 16 * bk + 4 * t4;
      const float fa[4] = {xa[bk].x, xa[bk].y, xa[bk].z, xa[bk].w};
      const float fb[4] = {xb[bk].x, xb[bk].y, xb[bk].z, xb[bk].w};
      if constexpr (sizeof(TC) == 4) {
        st_vec(outp + offA, CkVec<float>::pack(fa));
        st_vec(outp + offB, CkVec<float>::pack(fb));
      } else {
        st_vec2(outp + offA, LpVec<__half>::pack(fa));
        st_vec2(outp + offB, LpVec<__half>::pack(fb));
      }
    }
    (void)slot;
    mbar_arrive(&rec_empty[s]);
  }
  if (tid == 0 && *(volatile int *)s_abort) report(a.dev_err, kDerrTimeout);
}

template <int DV, int DK, int NSPLIT, typename TC, typename RT, bool GDNW, int NGRP = 3>
static cudaError_t launch_mat_pipe(const rs_materialize_args &a, int gdn, cudaStream_t s) {
  (void)gdn;
  auto kern = mat_pipe_kernel<DV, DK, NSPLIT, TC, RT, GDNW, NGRP>;
  constexpr int RB = DV / NSPLIT;
  constexpr int threads = NGRP * 4 * 32 + 32;
  const size_t ckb = (size_t)RB * DK * sizeof(TC);
  const size_t rb = mat_rec(RB, DK, (int)sizeof(RT), a.L, 4).bytes;
  // three checkpoint slots for the three groups: measured faster than both
  // two and four (batch 256, 128 heads of 64 x 128: 346 us against 357 and
  // 363)
  static const int shapes[][3] = {{1, 3, 6}, {1, 2, 4}, {1, 2, 3}, {1, 1, 2}};
  RingPlan plan;
  cudaError_t e = plan_rings(reinterpret_cast<const void *>(kern), threads, ckb, rb, mat_head, a.B * a.H * NSPLIT,
                             &plan, shapes, 4);
  if (e != cudaSuccess) return e;
  kern<<<plan.grid, threads, plan.smem, s>>>(a, plan.nsr, plan.nsc);
  return cudaGetLastError();
}

template <typename TC>
static MatLaunchFn find_mat_pipe_c(int gdn, int d_v, int d_k, int ring_dtype) {
  if (!gdn && d_v == 64 && d_k == 128) {
    if (ring_dtype == kBF16) return launch_mat_pipe<64, 128, 1, TC, __nv_bfloat16, false>;
    if (ring_dtype == kF32) return launch_mat_pipe<64, 128, 1, TC, float, false>;
  }
  if (gdn && d_v == 128 && d_k == 128) {
    if (ring_dtype == kF16) return launch_mat_pipe<128, 128, 2, TC, __half, true>;
    if (ring_dtype == kF32) return launch_mat_pipe<128, 128, 2, TC, float, true>;
  }
  return nullptr;
}

MatLaunchFn find_mat_pipe(int gdn, int d_v, int d_k, int ckpt_dtype, int ring_dtype) {
  if (ckpt_dtype == kF32) return find_mat_pipe_c<float>(gdn, d_v, d_k, ring_dtype);
  if (ckpt_dtype == kF16) return find_mat_pipe_c<__half>(gdn, d_v, d_k, ring_dtype);
  return nullptr;
}

}  // namespace rs
