// replayssm_decode_mamba2_noalloc: the Mamba-2 decode with group-shared keys
// for callers that hold no scratch buffer.  The group dots k_j . q_t go to a
// library-owned device array instead of caller memory; nothing is allocated
// at call time.  Declaration and documentation: include/replayssm.h.
#include <cuda_runtime.h>

#include <mutex>

#include "replayssm.h"

namespace {

constexpr long long kScratchFloats = RS_NOALLOC_KQ_FLOATS;

// one copy per device, created with the module
static __device__ __align__(256) float g_kq_scratch[kScratchFloats];

// device address of the scratch on the current device, looked up once per device
cudaError_t scratch_address(float **out) {
  static std::mutex mu;
  static float *addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_kq_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<float *>(p);
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int replayssm_decode_mamba2_noalloc(const rs_step_args *args, rs_stream_t stream) {
  if (!args) return RS_EINVAL;
  if (args->n_groups <= 0) return replayssm_decode_mamba2(args, stream);  // no scratch needed
  if (args->kq_scratch) return RS_EINVAL;                                 // the library provides it
  if (args->B < 0 || args->L < 1) return RS_EINVAL;
  if ((long long)args->B * args->n_groups * args->L > kScratchFloats) return RS_EINVAL;
  if (args->B == 0) return replayssm_decode_mamba2(args, stream);
  float *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return RS_ECUDA;
  rs_step_args a = *args;
  a.kq_scratch = scratch;
  return replayssm_decode_mamba2(&a, stream);
}
