// replayssm_decode_mamba2_noalloc: the group-shared-key Mamba-2 decode for
// callers that cannot allocate device memory.  The group dots k_j . q_t go to
// a fixed-size device array that the library itself holds, so the call
// allocates and frees nothing.  Declaration and documentation:
// include/replayssm.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "replayssm.h"

namespace {

constexpr long long kScratchFloats = RS_NOALLOC_KQ_FLOATS;

// One copy on every device that loads the library's module, until exit.  In
// host code this name is a host-side stand-in, not a device address: kernels
// get the address from scratch_address().
static __device__ __align__(256) float g_kq_scratch[kScratchFloats];

// Identity of the current context (driver API, reached through the runtime
// so that the library does not link libcuda): a reset device gets a new
// context, in which the module, and the array, may sit at another address.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

bool current_context_id(unsigned long long *id) {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch on the current device.  Looked up with
// cudaGetSymbolAddress once per device and context, with that device current;
// later calls reuse it.
cudaError_t scratch_address(float **out) {
  struct Entry {
    float *addr;
    unsigned long long ctx;
    bool ctx_known;
  };
  static std::mutex mu;
  static Entry cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  unsigned long long ctx = 0;
  const bool known = current_context_id(&ctx);
  std::lock_guard<std::mutex> lock(mu);
  Entry &c = cache[dev];
  if (c.addr && c.ctx_known == known && (!known || c.ctx == ctx)) {
    *out = c.addr;
    return cudaSuccess;
  }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_kq_scratch);
  if (e != cudaSuccess) return e;
  // the lookup made the device's primary context current if it was not yet
  c.ctx_known = current_context_id(&c.ctx);
  c.addr = static_cast<float *>(p);
  *out = c.addr;
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
