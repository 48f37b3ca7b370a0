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
// Persistent, warp-specialised kernel.  One producer warp streams each unit's
// checkpoint, ring records and inputs into a ring of shared-memory stages with
// 1-D bulk copies (cp.async.bulk, completion counted on an mbarrier); the
// decays come in with 4-byte cp.async.  The per-row slot, cursor and flag are
// prefetched 32 units ahead by the producer's lanes, so no dependent global
// load sits on the streaming path.  Eight consumer warps wait on a stage,
// compute from shared memory and release it.  The units a CTA owns are
// strided across the batch, so the ~1/L flush rows (which also write their
// state) spread evenly over the CTAs.  Every wait is bounded: on a timeout
// the kernel reports RS_DERR_TIMEOUT, drains its own copies and returns.
// No tensor cores: the step is a bandwidth-bound GEMV (about 0.6 FLOP/byte).
#include "common.cuh"
#include "launch.h"

namespace rs {

namespace {

constexpr int kStatusOk = 0, kStatusPad = 1, kStatusBadSlot = 2, kStatusBadPos = 3;

__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst_smem)), "l"(src) : "memory");
}

// arrive on the barrier once this thread's earlier cp.async copies have landed
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void bulk_load_plain(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst_smem)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

}  // namespace

// Byte offsets of one pipeline stage (host and device agree on this layout).
struct M2Stage {
  uint32_t ck, k, v, q, a, meta, scr, bytes;
};

__host__ __device__ inline uint32_t align128(uint32_t x) { return (x + 127u) & ~127u; }

__host__ __device__ inline M2Stage m2_stage(int DV, int DK, int ck_es, int rec_es, int L) {
  M2Stage s;
  uint32_t o = 0;
  s.ck = o;   o = align128(o + DV * DK * ck_es);
  s.k = o;    o = align128(o + L * DK * rec_es);   // records 0..p, current token at p
  s.v = o;    o = align128(o + L * DV * rec_es);
  s.q = o;    o = align128(o + DK * rec_es);
  s.a = o;    o = align128(o + L * 4);             // decays of records 0..p
  s.meta = o; o = align128(o + 16);                // slot, p, flush, status
  s.scr = o;  o = align128(o + (2 * L + DV + 4) * 4);  // w_j, k_j.q, row dots, gamma
  s.bytes = o;
  return s;
}

// barriers (full[ns], empty[ns]) and the abort flag precede the stages
__host__ __device__ inline uint32_t m2_head(int nstage) { return align128(16 * nstage + 16); }

template <int DV, int DK, typename TC, int NCW>
__global__ void __launch_bounds__(NCW * 32 + 32) mamba2_replay_kernel(const KArgs a, int nstage) {
  using V = CkVec<TC>;
  constexpr int E = V::E;
  constexpr int G = DK / E;          // lanes per state row
  constexpr int NC = NCW * 32;       // consumer threads
  constexpr int RPP = NC / G;        // state rows per pass of the consumers
  constexpr int VPT = DV / RPP;      // state rows per consumer thread
  static_assert(G <= 32 && 32 % G == 0, "a state row must fit in one warp");
  static_assert(NC % G == 0 && DV % RPP == 0 && VPT >= 1 && VPT <= G, "bad tiling");
  static_assert(DK % 8 == 0 && DV % 8 == 0, "head dims must be multiples of 8");

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + nstage;
  int *s_abort = reinterpret_cast<int *>(smem + 16 * nstage);
  const int L = a.L;
  const int rdt = a.in_dtype;  // records are the inputs verbatim
  const int res = rdt == kF32 ? 4 : 2;
  const M2Stage lay = m2_stage(DV, DK, (int)sizeof(TC), res, L);
  unsigned char *stages = smem + m2_head(nstage);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_units = a.B * a.H;
  const int stride = gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(&full[s], 33);   // 32 producer-lane cp.async arrivals + 1 expect_tx
      mbar_init(&empty[s], NC);  // every consumer thread
    }
    *s_abort = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == NCW) {
    // ---------------------------------------------------------------- producer
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
        const int s = it % nstage;
        const uint32_t par = (uint32_t)(it / nstage) & 1u;
        if (it >= nstage) {
          int w = 1;
          if (lane == 0) w = mbar_wait(&empty[s], par ^ 1u) ? 1 : 0;
          w = __shfl_sync(0xffffffffu, w, 0);
          if (!w || *(volatile int *)s_abort) {
            if (lane == 0) *(volatile int *)s_abort = 1;
            ok = false;
            break;
          }
        }
        __syncwarp();
        unsigned char *st = stages + (size_t)s * lay.bytes;
        const int b = u / a.H, h = u - (u / a.H) * a.H;
        const int status = slot < 0 ? kStatusPad
                           : slot >= a.num_slots ? kStatusBadSlot
                           : (p < 0 || p >= L) ? kStatusBadPos
                           : kStatusOk;
        if (status == kStatusOk) {
          const size_t unit = (size_t)slot * a.H + h;
          float *sa = reinterpret_cast<float *>(st + lay.a);
          for (int jj = lane; jj < p; jj += 32) cp_async4(sa + jj, a.ring_a + unit * L + jj);
          if (lane == 0) cp_async4(sa + p, a.alpha + (size_t)b * a.H + h);
          if (lane == 0) {
            int *meta = reinterpret_cast<int *>(st + lay.meta);
            meta[0] = slot; meta[1] = p; meta[2] = fl; meta[3] = status;
            const uint32_t ckb = DV * DK * (uint32_t)sizeof(TC);
            const uint32_t kb = DK * res, vb = DV * res;
            mbar_arrive_expect_tx(&full[s], ckb + (uint32_t)(p + 1) * (kb + vb) + kb);
            bulk_load(st + lay.ck, static_cast<const TC *>(a.ckpt) + unit * (DV * DK), ckb, &full[s], pol_stream);
            if (p > 0) {
              bulk_load_plain(st + lay.k, static_cast<const unsigned char *>(a.ring_k) + unit * L * kb,
                              (uint32_t)p * kb, &full[s]);
              bulk_load_plain(st + lay.v, static_cast<const unsigned char *>(a.ring_v) + unit * L * vb,
                              (uint32_t)p * vb, &full[s]);
            }
            const unsigned char *kin = static_cast<const unsigned char *>(a.k);
            const unsigned char *vin = static_cast<const unsigned char *>(a.v);
            const unsigned char *qin = static_cast<const unsigned char *>(a.q);
            bulk_load_plain(st + lay.k + p * kb, kin + ((size_t)b * a.sk + (size_t)h * DK) * res, kb, &full[s]);
            bulk_load_plain(st + lay.v + p * vb, vin + ((size_t)b * a.sv + (size_t)h * DV) * res, vb, &full[s]);
            bulk_load_plain(st + lay.q, qin + ((size_t)b * a.sq + (size_t)h * DK) * res, kb, &full[s]);
          }
        } else if (lane == 0) {
          int *meta = reinterpret_cast<int *>(st + lay.meta);
          meta[0] = slot; meta[1] = p; meta[2] = fl; meta[3] = status;
          mbar_arrive(&full[s]);
        }
        cp_async_arrive(&full[s]);
        ++it;
      }
      c_sl = n_sl; c_wp = n_wp; c_fl = n_fl;
    }
    // drain: every copy this warp issued has landed before the CTA may exit
    if (lane == 0) {
      for (int k = it > nstage ? it - nstage : 0; k < it; ++k) mbar_wait(&full[k % nstage], (uint32_t)(k / nstage) & 1u);
    }
    __syncwarp();
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int ctid = tid;  // 0 .. NC-1
  const int row0 = ctid / G, cv = ctid - (ctid / G) * G;
  int it = 0;
  for (int u = blockIdx.x; u < n_units; u += stride, ++it) {
    const int s = it % nstage;
    const uint32_t par = (uint32_t)(it / nstage) & 1u;
    if (lane == 0 && !mbar_wait(&full[s], par)) *(volatile int *)s_abort = 1;
    consumer_sync<NC>();
    if (*(volatile int *)s_abort) break;

    const unsigned char *st = stages + (size_t)s * lay.bytes;
    const int *meta = reinterpret_cast<const int *>(st + lay.meta);
    const int slot = meta[0], p = meta[1], flush = meta[2], status = meta[3];
    const int b = u / a.H, h = u - (u / a.H) * a.H;
    float *orow = a.out + (size_t)b * a.so + (size_t)h * DV;
    if (status != kStatusOk) {
      for (int i = ctid; i < DV; i += NC) orow[i] = 0.f;
      if (ctid == 0 && status != kStatusPad) report(a.dev_err, status == kStatusBadSlot ? 1 : 2);
      mbar_arrive(&empty[s]);
      continue;
    }
    const size_t unit = (size_t)slot * a.H + h;
    const float *sa = reinterpret_cast<const float *>(st + lay.a);
    float *scr = reinterpret_cast<float *>(const_cast<unsigned char *>(st) + lay.scr);
    float *sW = scr, *sS = scr + L, *sC = scr + 2 * L, *sGam = scr + 2 * L + DV;
    const unsigned char *sk = st + lay.k, *sv = st + lay.v;
    const uint4 *ck = reinterpret_cast<const uint4 *>(st + lay.ck);

    // window weights w_j (suffix products of the decays) and gamma
    if (warp == 0) {
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
    float qv[E];
    lds_cols<E>(st + lay.q, cv * E, rdt, qv);

    float part[VPT];
    if (!flush) {
      // k_j . q for every record of the window
      for (int j = warp; j <= p; j += NCW) {
        float acc = 0.f;
        for (int c = lane * 4; c < DK; c += 128) {
          float kk[4], qq[4];
          lds_cols<4>(sk, j * DK + c, rdt, kk);
          lds_cols<4>(st + lay.q, c, rdt, qq);
          acc += kk[0] * qq[0] + kk[1] * qq[1] + kk[2] * qq[2] + kk[3] * qq[3];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) sS[j] = acc;
      }
      // checkpoint GEMV partials from the stage
#pragma unroll
      for (int r = 0; r < VPT; ++r) {
        float f[E];
        V::unpack(ck[(row0 + r * RPP) * G + cv], f);
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc = fmaf(f[e], qv[e], acc);
        part[r] = acc;
      }
      group_reduce<VPT, G>(part, lane);
      if (group_reduce_writer<VPT, G>(lane)) sC[row0 + group_reduce_index<VPT, G>(lane) * RPP] = part[0];
      consumer_sync<NC>();

      const float gam = sGam[0];
      for (int i = ctid; i < DV; i += NC) {
        float acc = gam * sC[i];
        for (int j = 0; j <= p; ++j) acc = fmaf(sW[j] * sS[j], lds_elem(sv, j * DV + i, rdt), acc);
        orow[i] = acc;
      }
      // append the current record (k, v verbatim, alpha) at ring slot p
      constexpr int KCH = DK / 8, VCH = DV / 8;  // 16-byte chunks at bf16; doubled at fp32
      const int kch = KCH * (res / 2), vch = VCH * (res / 2);
      for (int c = ctid; c < kch + vch; c += NC) {
        if (c < kch) {
          const uint4 x = reinterpret_cast<const uint4 *>(sk + (size_t)p * DK * res)[c];
          reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.ring_k) + (unit * L + p) * DK * res)[c] = x;
        } else {
          const uint4 x = reinterpret_cast<const uint4 *>(sv + (size_t)p * DV * res)[c - kch];
          reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.ring_v) + (unit * L + p) * DV * res)[c - kch] = x;
        }
      }
      if (ctid == 0) a.ring_a[unit * L + p] = sa[p];
    } else {
      consumer_sync<NC>();  // weights ready
      const float gam = sGam[0];
      TC *ckg = static_cast<TC *>(a.ckpt) + unit * (DV * DK);
      float f[VPT][E];
#pragma unroll
      for (int r = 0; r < VPT; ++r) {
        V::unpack(ck[(row0 + r * RPP) * G + cv], f[r]);
#pragma unroll
        for (int e = 0; e < E; ++e) f[r][e] *= gam;
      }
      for (int j = 0; j <= p; ++j) {
        float kk[E];
        lds_cols<E>(sk, j * DK + cv * E, rdt, kk);
        const float wj = sW[j];
#pragma unroll
        for (int r = 0; r < VPT; ++r) {
          const float vv = wj * lds_elem(sv, j * DV + row0 + r * RPP, rdt);
#pragma unroll
          for (int e = 0; e < E; ++e) f[r][e] = fmaf(vv, kk[e], f[r][e]);
        }
      }
#pragma unroll
      for (int r = 0; r < VPT; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc = fmaf(f[r][e], qv[e], acc);
        part[r] = acc;
        st_vec(ckg + (size_t)(row0 + r * RPP) * DK + cv * E, V::pack(f[r]));
      }
      group_reduce<VPT, G>(part, lane);
      if (group_reduce_writer<VPT, G>(lane)) sC[row0 + group_reduce_index<VPT, G>(lane) * RPP] = part[0];
      consumer_sync<NC>();
      for (int i = ctid; i < DV; i += NC) orow[i] = sC[i];
    }
    mbar_arrive(&empty[s]);
  }
  if (ctid == 0 && *(volatile int *)s_abort) report(a.dev_err, kDerrTimeout);
}

template <int DV, int DK, typename TC, int NCW>
static cudaError_t launch_mamba2(const KArgs &a, cudaStream_t s) {
  auto kern = mamba2_replay_kernel<DV, DK, TC, NCW>;
  const int res = a.in_dtype == kF32 ? 4 : 2;
  const M2Stage lay = m2_stage(DV, DK, (int)sizeof(TC), res, a.L);
  PipePlan plan;
  cudaError_t e = plan_pipe(reinterpret_cast<const void *>(kern), NCW * 32 + 32, lay.bytes, m2_head, 4,
                            a.B * a.H, &plan);
  if (e != cudaSuccess) return e;
  kern<<<plan.grid, NCW * 32 + 32, plan.smem, s>>>(a, plan.nstage);
  return cudaGetLastError();
}

LaunchFn find_mamba2(int d_v, int d_k, int ckpt_dtype) {
  if (ckpt_dtype == kF32) {
    if (d_v == 16 && d_k == 32) return launch_mamba2<16, 32, float, 4>;
    if (d_v == 64 && d_k == 128) return launch_mamba2<64, 128, float, 8>;
    if (d_v == 128 && d_k == 128) return launch_mamba2<128, 128, float, 8>;
  } else if (ckpt_dtype == kF16) {
    if (d_v == 16 && d_k == 32) return launch_mamba2<16, 32, __half, 2>;
    if (d_v == 64 && d_k == 128) return launch_mamba2<64, 128, __half, 8>;
    if (d_v == 128 && d_k == 128) return launch_mamba2<128, 128, __half, 8>;
  }
  return nullptr;
}

}  // namespace rs
