// C ABI of libreplayssm.so: argument validation, the host step plan and
// dispatch to the kernels.  Declarations and their documentation are in
// include/replayssm.h.
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <utility>

#include "replayssm.h"
#include "launch.h"

#include <algorithm>

namespace rs {

cudaError_t ensure_smem(const void *kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  static std::mutex mu;
  static std::set<std::pair<int, const void *>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({dev, kernel})) return cudaSuccess;
  // allow the largest opt-in size once, so later, larger L need no new call
  int max_optin = 0;
  e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if ((size_t)max_optin < bytes) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin);
  if (e == cudaSuccess) done.insert({dev, kernel});
  return e;
}

namespace {

struct DevInfo {
  int sms = 0, smem_sm = 0, smem_block = 0;
};

cudaError_t dev_info(int dev, DevInfo *out) {
  static std::mutex mu;
  static std::map<int, DevInfo> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  DevInfo d;
  cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.smem_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cache[dev] = d;
  *out = d;
  return cudaSuccess;
}

}  // namespace

cudaError_t plan_rings(const void *kernel, int threads, size_t ck_bytes, size_t rec_bytes, RingHeadFn head,
                       int units, RingPlan *out, const int (*shapes)[3], int n_shapes) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void *, size_t, size_t>, RingPlan> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_tuple(dev, kernel, ck_bytes, rec_bytes);
  RingPlan plan{};
  bool hit = false;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      plan = it->second;
      hit = true;
    }
  }
  if (!hit) {
    DevInfo d;
    e = dev_info(dev, &d);
    if (e != cudaSuccess) return e;
    auto need = [&](int nsr, int nsc) { return (size_t)head(nsr, nsc) + nsc * ck_bytes + nsr * rec_bytes; };
    // preferred shapes, best first: two CTAs per SM each with two
    // checkpoint slots (two producers per SM keep bulk-copy issue off the
    // critical path), then one CTA per SM with fewer or more slots
    // (a shape whose CTAs per SM the kernel's registers and threads do not
    // allow is skipped: it would run fewer CTAs with the smaller rings)
    static const int defaults[][3] = {{2, 2, 4}, {2, 2, 3}, {2, 2, 2}, {1, 4, 8}, {1, 3, 6}, {1, 2, 4}, {1, 2, 3}, {1, 1, 2}};
    if (!shapes) {
      shapes = defaults;
      n_shapes = (int)(sizeof(defaults) / sizeof(defaults[0]));
    }
    int fit_regs = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit_regs, kernel, threads, 0);
    if (e != cudaSuccess) return e;
    int ctas = 0;
    for (int k = 0; k < n_shapes; ++k) {
      const int *sh = shapes[k];
      if (sh[0] > fit_regs) continue;
      const size_t budget = (size_t)std::min<long>(d.smem_sm / sh[0] - 1024, d.smem_block);
      if (need(sh[2], sh[1]) <= budget) {
        ctas = sh[0];
        plan.nsc = sh[1];
        plan.nsr = sh[2];
        break;
      }
    }
    if (!ctas) return cudaErrorInvalidValue;
    plan.smem = need(plan.nsr, plan.nsc);
    e = ensure_smem(kernel, plan.smem);
    if (e != cudaSuccess) return e;
    int fit = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, kernel, threads, plan.smem);
    if (e != cudaSuccess) return e;
    if (fit < 1) return cudaErrorInvalidConfiguration;
    plan.grid = (unsigned)(d.sms * std::min(ctas, fit));
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = plan;
  }
  plan.grid = std::min<unsigned>(plan.grid, (unsigned)units);
  *out = plan;
  return cudaSuccess;
}

}  // namespace rs

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

size_t esize(int dt) { return dt == RS_F32 ? 4 : 2; }

bool shape_supported(int d_v, int d_k) {
  return (d_v == 16 && d_k == 32) || (d_v == 64 && d_k == 128) || (d_v == 128 && d_k == 128);
}

// Validation shared by every decode entry point.  `replay` adds the ring and
// cursor arguments; `gdn` adds beta and the GDN ring rule.
int validate(const rs_step_args *a, bool replay, bool gdn) {
  if (!a) return RS_EINVAL;
  if (a->reserved != 0) return RS_EINVAL;
  if (a->B < 0 || a->H < 1 || a->num_slots < 1 || a->d_v < 1 || a->d_k < 1) return RS_EINVAL;
  if (replay && (a->L < 2 || a->L > RS_MAX_L)) return RS_EINVAL;
  if (a->ckpt_dtype != RS_F32 && a->ckpt_dtype != RS_F16) return RS_EUNSUPPORTED;
  if (a->in_dtype != RS_F32 && a->in_dtype != RS_BF16) return RS_EUNSUPPORTED;
  if (!shape_supported(a->d_v, a->d_k)) return RS_EUNSUPPORTED;
  if (replay) {
    if (gdn) {
      if (a->ring_dtype != RS_F16 && a->ring_dtype != RS_F32) return RS_EUNSUPPORTED;
    } else if (a->ring_dtype != a->in_dtype) {
      return RS_EUNSUPPORTED;  // Mamba-2 records are the inputs verbatim
    }
  }
  if (a->B == 0) return RS_OK;
  if (!a->slot_idx || !a->v || !a->k || !a->q || !a->alpha || !a->ckpt || !a->out) return RS_EINVAL;
  if (gdn && !a->beta) return RS_EINVAL;
  if (replay && (!a->write_pos || !a->is_flush || !a->ring_v || !a->ring_k || !a->ring_a)) return RS_EINVAL;
  const int64_t H = a->H;
  if (a->n_groups < 0 || a->reserved3 != 0) return RS_EINVAL;
  const int64_t KH = a->n_groups > 0 ? a->n_groups : H;  // key / query vectors per row
  if (a->stride_v_row < H * a->d_v || a->stride_k_row < KH * a->d_k || a->stride_q_row < KH * a->d_k ||
      a->stride_out_row < H * a->d_v)
    return RS_EINVAL;
  const size_t ie = esize(a->in_dtype);
  if (!aligned16(a->ckpt) || !aligned16(a->v) || !aligned16(a->k) || !aligned16(a->q)) return RS_EALIGN;
  if ((a->stride_v_row * ie) % 16 || (a->stride_k_row * ie) % 16 || (a->stride_q_row * ie) % 16) return RS_EALIGN;
  if (!aligned4(a->out) || !aligned4(a->alpha) || !aligned4(a->slot_idx)) return RS_EALIGN;
  if (gdn && !aligned4(a->beta)) return RS_EALIGN;
  if (replay) {
    if (!aligned16(a->ring_v) || !aligned16(a->ring_k) || !aligned4(a->ring_a) || !aligned4(a->write_pos))
      return RS_EALIGN;
  }
  if ((int64_t)a->B * a->H > 0x7fffffffLL) return RS_EINVAL;
  if (a->reserved2 != 0) return RS_EINVAL;
  if (a->n_groups > 0) {
    // group-shared keys: Mamba-2 replay only, with its scratch
    if (!replay || gdn || a->ckpt_lp) return RS_EUNSUPPORTED;
    if (a->H % a->n_groups != 0) return RS_EINVAL;
    if (!a->kq_scratch) return RS_EINVAL;
    if (!aligned4(a->kq_scratch)) return RS_EALIGN;
  }
  if (a->ckpt_lp) {
    // two-precision checkpoint: Mamba-2 replay, fp32 recurrence copy, 16-bit
    // or E4M3 (row-scaled) read copy
    if (!replay || gdn) return RS_EUNSUPPORTED;
    if (a->ckpt_dtype != RS_F32 || (a->lp_dtype != RS_F16 && a->lp_dtype != RS_BF16 && a->lp_dtype != RS_F8E4M3))
      return RS_EUNSUPPORTED;
    if (!aligned16(a->ckpt_lp)) return RS_EALIGN;
    if ((a->lp_dtype == RS_F8E4M3) != (a->ckpt_lp_scale != nullptr)) return RS_EINVAL;  // scales with E4M3 only
    if (a->ckpt_lp_scale && !aligned16(a->ckpt_lp_scale)) return RS_EALIGN;
  } else if (a->ckpt_lp_scale) {
    return RS_EINVAL;
  }
  return RS_OK;
}

rs::KArgs to_kargs(const rs_step_args *a) {
  rs::KArgs k;
  k.B = a->B;
  k.H = a->H;
  k.L = a->L;
  k.num_slots = a->num_slots;
  k.in_dtype = a->in_dtype;
  k.ring_dtype = a->ring_dtype;
  k.slot_idx = a->slot_idx;
  k.write_pos = a->write_pos;
  k.is_flush = a->is_flush;
  k.v = a->v;
  k.k = a->k;
  k.q = a->q;
  k.alpha = a->alpha;
  k.beta = a->beta;
  k.ckpt = a->ckpt;
  k.ring_v = a->ring_v;
  k.ring_k = a->ring_k;
  k.ring_a = a->ring_a;
  k.ckpt_lp = a->ckpt_lp;
  k.lp_scale = a->ckpt_lp_scale;
  k.n_groups = a->n_groups;
  k.kq = a->kq_scratch;
  k.out = a->out;
  k.sv = a->stride_v_row;
  k.sk = a->stride_k_row;
  k.sq = a->stride_q_row;
  k.so = a->stride_out_row;
  k.dev_err = a->dev_err;
  return k;
}

int run(rs::LaunchFn fn, const rs_step_args *a, rs_stream_t stream) {
  if (!fn) return RS_EUNSUPPORTED;
  const cudaError_t e = fn(to_kargs(a), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RS_OK : RS_ECUDA;
}

}  // namespace

extern "C" {

int replayssm_abi_version(void) { return RS_ABI_VERSION; }

int replayssm_supported(int variant, int d_v, int d_k, int ckpt_dtype) {
  if (variant != RS_MAMBA2 && variant != RS_GDN) return 0;
  if (variant == RS_MAMBA2) return rs::find_mamba2(d_v, d_k, ckpt_dtype, RS_BF16, -1, false) != nullptr;
  return rs::find_gdn(d_v, d_k, ckpt_dtype, RS_F16, RS_BF16) != nullptr;
}

int replayssm_plan_step(const int64_t *decode_step, const uint8_t *force_flush, int32_t B, int32_t L,
                        int32_t *write_pos, uint8_t *is_flush) {
  if (B < 0 || L < 1 || L > RS_MAX_L) return RS_EINVAL;
  if (B == 0) return RS_OK;
  if (!decode_step || !write_pos || !is_flush) return RS_EINVAL;
  for (int32_t b = 0; b < B; ++b)
    if (decode_step[b] < 0) return RS_EINVAL;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t wp = (int32_t)(decode_step[b] % L);
    write_pos[b] = wp;
    is_flush[b] = (uint8_t)((wp == L - 1) || (force_flush && force_flush[b]));
  }
  return RS_OK;
}

int replayssm_plan_align(const int64_t *position, const int64_t *start, int32_t block, int32_t B, int32_t L,
                         int32_t *write_pos, uint8_t *is_flush) {
  if (B < 0 || L < 1 || L > RS_MAX_L || block < 0) return RS_EINVAL;
  if (B == 0) return RS_OK;
  if (!position || !start || !write_pos || !is_flush) return RS_EINVAL;
  for (int32_t b = 0; b < B; ++b)
    if (start[b] < 0 || position[b] < start[b]) return RS_EINVAL;
  for (int32_t b = 0; b < B; ++b) {
    int64_t anchor = start[b];
    bool completes = false;
    if (block > 0) {
      anchor = std::max<int64_t>(anchor, position[b] / block * block);
      completes = (position[b] + 1) % block == 0;
    }
    const int32_t wp = (int32_t)((position[b] - anchor) % L);
    write_pos[b] = wp;
    is_flush[b] = (uint8_t)(wp == L - 1 || completes);
  }
  return RS_OK;
}

int replayssm_materialize(const rs_materialize_args *a, int variant, rs_stream_t stream) {
  if (!a || (variant != RS_MAMBA2 && variant != RS_GDN)) return RS_EINVAL;
  if (a->reserved != 0) return RS_EINVAL;
  if (a->B < 0 || a->H < 1 || a->num_slots < 1 || a->num_dst < 1 || a->d_v < 1 || a->d_k < 1) return RS_EINVAL;
  if (a->L < 2 || a->L > RS_MAX_L) return RS_EINVAL;
  if (a->ckpt_dtype != RS_F32 && a->ckpt_dtype != RS_F16) return RS_EUNSUPPORTED;
  if (a->ring_dtype != RS_F32 && a->ring_dtype != RS_F16 && a->ring_dtype != RS_BF16) return RS_EUNSUPPORTED;
  rs::MatLaunchFn fn = rs::find_mat_pipe(variant == RS_GDN, a->d_v, a->d_k, a->ckpt_dtype, a->ring_dtype);
  if (!fn) fn = rs::find_materialize(a->d_v, a->d_k, a->ckpt_dtype);
  if (!fn) return RS_EUNSUPPORTED;
  if (a->B == 0) return RS_OK;
  if (!a->slot_idx || !a->held || !a->dst_idx || !a->ckpt || !a->ring_v || !a->ring_k || !a->ring_a || !a->dst)
    return RS_EINVAL;
  if (!aligned16(a->ckpt) || !aligned16(a->dst) || !aligned16(a->ring_v) || !aligned16(a->ring_k)) return RS_EALIGN;
  if (!aligned4(a->ring_a) || !aligned4(a->slot_idx) || !aligned4(a->held) || !aligned4(a->dst_idx))
    return RS_EALIGN;
  if ((int64_t)a->B * a->H * 2 > 0x7fffffffLL) return RS_EINVAL;
  const cudaError_t e = fn(*a, variant == RS_GDN, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RS_OK : RS_ECUDA;
}

int replayssm_spec_verify_mamba2(const rs_spec_args *a, rs_stream_t stream) {
  if (!a || a->reserved != 0) return RS_EINVAL;
  if (a->B < 0 || a->H < 1 || a->num_slots < 1 || a->d_v < 1 || a->d_k < 1) return RS_EINVAL;
  if (a->L < 1 || a->L > RS_MAX_L || a->T < 1 || a->T > 16 || a->T > a->L) return RS_EINVAL;
  if (a->ckpt_dtype != RS_F32 && a->ckpt_dtype != RS_F16) return RS_EUNSUPPORTED;
  if (a->in_dtype != RS_F32 && a->in_dtype != RS_BF16) return RS_EUNSUPPORTED;
  const rs::SpecLaunchFn fn = rs::find_spec(a->d_v, a->d_k, a->ckpt_dtype, a->in_dtype);
  if (!fn) return RS_EUNSUPPORTED;
  if (a->B == 0) return RS_OK;
  if (!a->slot_idx || !a->committed || !a->is_flush || !a->v || !a->k || !a->q || !a->alpha || !a->ckpt ||
      !a->ring_v || !a->ring_k || !a->ring_a || !a->out)
    return RS_EINVAL;
  if (!aligned16(a->ckpt) || !aligned16(a->ring_v) || !aligned16(a->ring_k) || !aligned16(a->v) ||
      !aligned16(a->k) || !aligned16(a->q))
    return RS_EALIGN;
  if (!aligned4(a->ring_a) || !aligned4(a->alpha) || !aligned4(a->out) || !aligned4(a->slot_idx) ||
      !aligned4(a->committed))
    return RS_EALIGN;
  if ((int64_t)a->B * a->H > 0x7fffffffLL) return RS_EINVAL;
  const cudaError_t e = fn(*a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RS_OK : RS_ECUDA;
}

int replayssm_plan_spec(const int32_t *committed, int32_t B, int32_t L, int32_t T, uint8_t *is_flush) {
  if (B < 0 || L < 1 || L > RS_MAX_L || T < 1 || T > 16 || T > L) return RS_EINVAL;
  if (B == 0) return RS_OK;
  if (!committed || !is_flush) return RS_EINVAL;
  for (int32_t b = 0; b < B; ++b)
    if (committed[b] < 0 || committed[b] > L) return RS_EINVAL;
  for (int32_t b = 0; b < B; ++b) is_flush[b] = (uint8_t)(committed[b] + T > L);
  return RS_OK;
}

int replayssm_spec_commit(const int32_t *committed, const uint8_t *is_flush, const int32_t *accepted, int32_t B,
                          int32_t L, int32_t T, int32_t *committed_out, uint8_t *is_flush_out, int32_t *dev_err,
                          rs_stream_t stream) {
  if (B < 0 || L < 1 || L > RS_MAX_L || T < 1 || T > 16 || T > L) return RS_EINVAL;
  if (B == 0) return RS_OK;
  if (!committed || !is_flush || !accepted || !committed_out || !is_flush_out) return RS_EINVAL;
  if (!aligned4(committed) || !aligned4(accepted) || !aligned4(committed_out)) return RS_EALIGN;
  const cudaError_t e = rs::launch_spec_commit(committed, is_flush, accepted, B, L, T, committed_out,
                                               is_flush_out, dev_err, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RS_OK : RS_ECUDA;
}

int replayssm_seed_read_copy(const float *ckpt, int64_t n_rows, int32_t d_k, int32_t lp_dtype, void *ckpt_lp,
                             float *scale, rs_stream_t stream) {
  if (n_rows < 0 || d_k < 8 || d_k > 1024 || d_k % 8) return RS_EINVAL;
  if (lp_dtype != RS_F16 && lp_dtype != RS_BF16 && lp_dtype != RS_F8E4M3) return RS_EINVAL;
  if (n_rows == 0) return RS_OK;
  if (!ckpt || !ckpt_lp || (lp_dtype == RS_F8E4M3 && !scale)) return RS_EINVAL;
  if (!aligned16(ckpt) || !aligned16(ckpt_lp) || (scale && !aligned4(scale))) return RS_EALIGN;
  if (n_rows > 0x7fffffffLL * 8) return RS_EINVAL;
  const cudaError_t e = rs::launch_seed_read_copy(ckpt, n_rows, d_k, lp_dtype, ckpt_lp, scale,
                                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RS_OK : RS_ECUDA;
}

int replayssm_decode_mamba2(const rs_step_args *args, rs_stream_t stream) {
  const int st = validate(args, /*replay=*/true, /*gdn=*/false);
  if (st != RS_OK || args->B == 0) return st;
  const int lp = args->ckpt_lp ? args->lp_dtype : -1;
  return run(rs::find_mamba2(args->d_v, args->d_k, args->ckpt_dtype, args->in_dtype, lp, args->n_groups > 0), args,
             stream);
}

int replayssm_decode_gdn(const rs_step_args *args, rs_stream_t stream) {
  const int st = validate(args, /*replay=*/true, /*gdn=*/true);
  if (st != RS_OK || args->B == 0) return st;
  return run(rs::find_gdn(args->d_v, args->d_k, args->ckpt_dtype, args->ring_dtype, args->in_dtype), args, stream);
}

int conventional_decode(const rs_step_args *args, int variant, rs_stream_t stream) {
  if (variant != RS_MAMBA2 && variant != RS_GDN) return RS_EINVAL;
  const int st = validate(args, /*replay=*/false, /*gdn=*/variant == RS_GDN);
  if (st != RS_OK || args->B == 0) return st;
  return run(rs::find_conventional(variant, args->d_v, args->d_k, args->ckpt_dtype), args, stream);
}

const char *replayssm_status_string(int status) {
  switch (status) {
    case RS_OK: return "RS_OK";
    case RS_EINVAL: return "RS_EINVAL: invalid argument";
    case RS_EUNSUPPORTED: return "RS_EUNSUPPORTED: shape or dtype not built into the library";
    case RS_EALIGN: return "RS_EALIGN: pointer or row stride not aligned";
    case RS_ECUDA: return "RS_ECUDA: CUDA launch error";
    default: return "unknown rs_status";
  }
}

}  // extern "C"
