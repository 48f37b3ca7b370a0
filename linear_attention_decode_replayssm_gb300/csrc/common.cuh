// Device helpers shared by the ReplaySSM kernels (sm_103a).
//
// Memory layout conventions (all row-major, last dimension contiguous):
//   checkpoint / state  [num_slots, H, d_v, d_k]  fp32 or fp16
//   ring_v              [num_slots, H, L, d_v]
//   ring_k              [num_slots, H, L, d_k]
//   ring_a              [num_slots, H, L]          fp32
// A CTA owns one (row, head) unit.  Its threads tile the d_v x d_k block in
// 16-byte vectors: G = d_k * sizeof(T) / 16 consecutive lanes cover one state
// row, so every warp-wide load instruction reads whole 512-byte (fp32) or
// 256-byte (fp16) rows, fully coalesced.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rs {

constexpr int kF32 = 0;
constexpr int kF16 = 1;
constexpr int kBF16 = 2;
constexpr int kF8 = 3;  // E4M3, the read copy of a two-precision checkpoint

// Kernel arguments, copied by value into the launch (mirrors rs_step_args).
struct KArgs {
  int B, H, L, num_slots, in_dtype, ring_dtype;
  const int32_t *slot_idx;
  const int32_t *write_pos;
  const uint8_t *is_flush;
  const void *v, *k, *q;
  const float *alpha, *beta;
  void *ckpt, *ring_v, *ring_k;
  void *ckpt_lp;  // read copy of a two-precision checkpoint, or nullptr
  float *lp_scale;  // row scales of an E4M3 read copy [slots, H, d_v], or nullptr
  int n_groups;   // 0: a key per head; > 0: keys and queries shared by groups
  float *kq;      // [B, n_groups, L] scratch for the group dots k_j . q_t
  float *ring_a, *out;
  long long sv, sk, sq, so;  // row strides in elements
  int32_t *dev_err;
};

// ---------------------------------------------------------------------------
// 16-byte checkpoint vectors
// ---------------------------------------------------------------------------
template <typename TC>
struct CkVec;

template <>
struct CkVec<float> {
  static constexpr int E = 4;  // elements per 16-byte vector
  __device__ __forceinline__ static void unpack(const uint4 &r, float (&f)[4]) {
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

template <>
struct CkVec<__half> {
  static constexpr int E = 8;
  __device__ __forceinline__ static float2 h2f(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    return __half22float2(h);
  }
  __device__ __forceinline__ static uint32_t f2h(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
  }
  __device__ __forceinline__ static void unpack(const uint4 &r, float (&f)[8]) {
    float2 a = h2f(r.x), b = h2f(r.y), c = h2f(r.z), d = h2f(r.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
    return make_uint4(f2h(f[0], f[1]), f2h(f[2], f[3]), f2h(f[4], f[5]), f2h(f[6], f[7]));
  }
};

// Streaming read of data used once: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_vec(void *p, const uint4 &v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------
// 8-element staging of inputs and ring records with a runtime element type
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bf16x2_to_f(uint32_t w, float &a, float &b) {
  a = __uint_as_float(w << 16);
  b = __uint_as_float(w & 0xffff0000u);
}

// Load 8 consecutive elements starting at element offset `off` (16-byte
// aligned for 16-bit types, 32-byte aligned for fp32) and widen to fp32.
__device__ __forceinline__ void load8(const void *base, size_t off, int dt, float (&f)[8]) {
  if (dt == kF32) {
    const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + off);
    float4 a = __ldg(p), b = __ldg(p + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else {
    uint4 r = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + off));
    if (dt == kBF16) {
      bf16x2_to_f(r.x, f[0], f[1]);
      bf16x2_to_f(r.y, f[2], f[3]);
      bf16x2_to_f(r.z, f[4], f[5]);
      bf16x2_to_f(r.w, f[6], f[7]);
    } else {
      float tmp[8];
      CkVec<__half>::unpack(r, tmp);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = tmp[i];
    }
  }
}

// Copy 8 elements verbatim (same element type on both sides).
__device__ __forceinline__ void copy8(void *dst, size_t doff, const void *src, size_t soff, int dt) {
  if (dt == kF32) {
    const float4 *s = reinterpret_cast<const float4 *>(static_cast<const float *>(src) + soff);
    float4 *d = reinterpret_cast<float4 *>(static_cast<float *>(dst) + doff);
    d[0] = __ldg(s);
    d[1] = __ldg(s + 1);
  } else {
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(dst) + doff) =
        __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(src) + soff));
  }
}

// Store 8 fp32 values as fp32 or fp16 (round to nearest even).
__device__ __forceinline__ void store8(void *dst, size_t off, int dt, const float (&f)[8]) {
  if (dt == kF32) {
    float4 *d = reinterpret_cast<float4 *>(static_cast<float *>(dst) + off);
    d[0] = make_float4(f[0], f[1], f[2], f[3]);
    d[1] = make_float4(f[4], f[5], f[6], f[7]);
  } else {
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(dst) + off) = CkVec<__half>::pack(f);
  }
}

// Store one fp32 value as fp32 or fp16 (round to nearest even).
__device__ __forceinline__ void store1(void *dst, size_t off, int dt, float x) {
  if (dt == kF32)
    static_cast<float *>(dst)[off] = x;
  else
    static_cast<__half *>(dst)[off] = __float2half_rn(x);
}

// ---------------------------------------------------------------------------
// Transposed group reduction.
// Each lane holds N partial sums; lanes are grouped G at a time (G a power of
// two dividing 32, groups contiguous in the warp).  Every halving stage trades
// half of the values with the partner lane `G/2` away, so after log2(N)
// stages each lane holds one fully combined value instead of N; the remaining
// G/N lanes finish with a plain butterfly.  Costs N-1 + log2(G/N) shuffles
// instead of N*log2(G).  Requires N <= G.
// ---------------------------------------------------------------------------
template <int N, int G>
__device__ __forceinline__ void group_reduce(float *v, int lane) {
  static_assert(N <= G, "group_reduce needs N <= G");
  if constexpr (N > 1) {
    constexpr int off = G / 2;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const float send = upper ? v[i] : v[i + N / 2];
      const float keep = upper ? v[i + N / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
    group_reduce<N / 2, off>(v, lane);
  } else {
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
  }
}

// Which of the N original values a lane holds after group_reduce<N, G>.
template <int N, int G>
__device__ __forceinline__ int group_reduce_index(int lane) {
  if constexpr (N > 1) {
    constexpr int off = G / 2;
    return ((lane & off) ? N / 2 : 0) + group_reduce_index<N / 2, off>(lane);
  } else {
    return 0;
  }
}

// Lanes that hold a distinct result after group_reduce<N, G> (one per value).
template <int N, int G>
__device__ __forceinline__ bool group_reduce_writer(int lane) {
  constexpr int rem = G / N;  // lanes sharing one result
  return (lane & (rem - 1)) == 0;
}

// Warp-wide inclusive suffix scan over 64 entries held two per lane
// (entry `lane` in x0, entry `lane + 32` in x1), combining with op.
template <typename Op>
__device__ __forceinline__ void suffix_scan64(float &x0, float &x1, int lane, Op op) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y0 = __shfl_down_sync(0xffffffffu, x0, off);
    const float y1 = __shfl_down_sync(0xffffffffu, x1, off);
    if (lane + off < 32) {
      x0 = op(x0, y0);
      x1 = op(x1, y1);
    }
  }
  x0 = op(x0, __shfl_sync(0xffffffffu, x1, 0));
}

__device__ __forceinline__ void report(int32_t *dev_err, int bit) {
  if (dev_err) atomicOr(dev_err, bit);
}

// ---------------------------------------------------------------------------
// 8-byte vectors of four 16-bit elements: the read copy of a two-precision
// checkpoint, in the element positions of a 16-byte fp32 vector
// ---------------------------------------------------------------------------
template <typename TL>
struct LpVec;

template <>
struct LpVec<__half> {
  __device__ __forceinline__ static void unpack(const uint2 &r, float (&f)[4]) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  }
  __device__ __forceinline__ static uint2 pack(const float (&f)[4]) {
    const __half2 a = __floats2half2_rn(f[0], f[1]), b = __floats2half2_rn(f[2], f[3]);
    return make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
  }
};

template <>
struct LpVec<__nv_bfloat16> {
  __device__ __forceinline__ static void unpack(const uint2 &r, float (&f)[4]) {
    bf16x2_to_f(r.x, f[0], f[1]);
    bf16x2_to_f(r.y, f[2], f[3]);
  }
  __device__ __forceinline__ static uint2 pack(const float (&f)[4]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]), b = __floats2bfloat162_rn(f[2], f[3]);
    return make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
  }
};

// m16n8k8 tf32 tensor-core product with fp32 accumulate (D += A B); fragment
// layouts as in the PTX ISA: lane = 4 g + t holds A[g][t], A[g+8][t],
// A[g][t+4], A[g+8][t+4]; B[t][g], B[t+4][g]; D[g][2t], D[g][2t+1],
// D[g+8][2t], D[g+8][2t+1]
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// x = hi + lo with hi and lo tf32 (round to nearest): two tf32 products carry
// about 21 mantissa bits of an fp32 operand
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
  const float r = x - __uint_as_float(hi);
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(r));
}

// acc + lo(a) lo(b) + hi(a) hi(b), in that order: bf16 pairs multiplied on
// the mixed-precision FMA (16-bit operands, fp32 addend and result, one
// rounding), the same value as widening both to fp32 and using fmaf
__device__ __forceinline__ float fma_bf16x2_acc(uint32_t a, uint32_t b, float acc) {
  asm("{\n .reg .b16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1;\n mov.b32 {b0, b1}, %2;\n"
      " fma.rn.f32.bf16 %0, a0, b0, %0;\n fma.rn.f32.bf16 %0, a1, b1, %0;\n}"
      : "+f"(acc) : "r"(a), "r"(b));
  return acc;
}

// a * b + c elementwise on fp32 pairs, one packed FMA (each component
// rounded once, as fmaf)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ void st_vec2(void *p, const uint2 &v) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

}  // namespace rs

// ---------------------------------------------------------------------------
// Bulk-copy (TMA) pipeline primitives: mbarriers in shared memory, 1-D
// cp.async.bulk global -> shared with transaction-count completion, and waits
// bounded by the global timer so a lost arrival ends in an error code instead
// of a hung GPU.
// ---------------------------------------------------------------------------
namespace rs {

constexpr int kDerrTimeout = 4;                       // RS_DERR_TIMEOUT
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// make barrier initialisation visible to the async (bulk copy) proxy
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// raise the barrier's expected transaction bytes without arriving
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the barrier phase with the given parity; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// Wait for the fill of a record slot with unit u: the phase of its full
// barrier with parity `parity`.  When consumer groups take alternate units
// and the slot count is not a multiple of the group count, a group can come
// to a slot while the slot's previous fill (another group's unit) has not
// landed yet; a parity wait then returns at once, on the phase before.  The
// producer writes the unit index into the slot (*slot_unit) only after that
// previous unit was released, before it completes the new phase, so a slot
// that does not show u yet means the wait returned early: wait until it
// does, then wait for the phase again.  false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_unit(uint64_t *bar, uint32_t parity, const int *slot_unit, int u) {
  if (!mbar_wait(bar, parity)) return false;
  if (*(const volatile int *)slot_unit == u) return true;
  const unsigned long long t0 = global_ns();
  while (*(const volatile int *)slot_unit != u) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return mbar_wait(bar, parity);
}

// 1-D bulk copy global -> shared, completing `bytes` on the barrier's
// transaction count.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// element type tag of ring records and inputs, as a compile-time dtype
template <typename T>
struct Rec;
template <>
struct Rec<float> {
  static constexpr int kDtype = kF32;
};
template <>
struct Rec<__nv_bfloat16> {
  static constexpr int kDtype = kBF16;
};
template <>
struct Rec<__half> {
  static constexpr int kDtype = kF16;
};

// per-unit status the producer hands to the consumers
constexpr int kStatusOk = 0, kStatusPad = 1, kStatusBadSlot = 2, kStatusBadPos = 3;

__host__ __device__ inline uint32_t align128(uint32_t x) { return (x + 127u) & ~127u; }

// 16- and 4-byte asynchronous global -> shared copies (per thread)
__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst_smem)), "l"(src) : "memory");
}

// arrive on the barrier once this thread's earlier cp.async copies have landed
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// barrier among the consumer warps only (the producer warp does not take part)
template <int NTHREADS>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NTHREADS) : "memory");
}

// widen E consecutive 16-bit or fp32 elements from shared memory
template <int E>
__device__ __forceinline__ void lds_cols(const unsigned char *base, int elem, int dt, float (&f)[E]) {
  if (dt == kF32) {
    const float4 *p = reinterpret_cast<const float4 *>(base + (size_t)elem * 4);
#pragma unroll
    for (int i = 0; i < E / 4; ++i) {
      const float4 x = p[i];
      f[4 * i] = x.x; f[4 * i + 1] = x.y; f[4 * i + 2] = x.z; f[4 * i + 3] = x.w;
    }
  } else {
    const uint32_t *p = reinterpret_cast<const uint32_t *>(base + (size_t)elem * 2);
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
      const uint32_t w = p[i];
      if (dt == kBF16) {
        bf16x2_to_f(w, f[2 * i], f[2 * i + 1]);
      } else {
        const float2 x = CkVec<__half>::h2f(w);
        f[2 * i] = x.x; f[2 * i + 1] = x.y;
      }
    }
  }
}

__device__ __forceinline__ float lds_elem(const unsigned char *base, int elem, int dt) {
  if (dt == kF32) return reinterpret_cast<const float *>(base)[elem];
  const uint16_t h = reinterpret_cast<const uint16_t *>(base)[elem];
  if (dt == kBF16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
  return __half2float(__ushort_as_half(h));
}

}  // namespace rs

namespace rs {

// m16n8k16 bf16 tensor-core product with fp32 accumulate (D += A B); lane
// 4 g + t holds A rows g and g+8 at columns 2t, 2t+1 (a0, a1) and 2t+8,
// 2t+9 (a2, a3), each register two bf16 with the lower column in its low
// half; B rows 2t, 2t+1 (b0) and 2t+8, 2t+9 (b1) of column g; D as for
// mma_tf32
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (x0, x1) = hi + lo with hi and lo pairs of bf16 (round to nearest even,
// x0 in the low halves): two bf16 products carry about 16 mantissa bits of
// an fp32 operand, a relative error of at most 2^-17
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

}  // namespace rs

namespace rs {

// ---------------------------------------------------------------------------
// E4M3 read copy: each state row on a power-of-two scale 2^e, e the smallest
// integer with max |row| <= 448 * 2^e; codes rounded to nearest even with
// saturation, column c of a row at byte c
// ---------------------------------------------------------------------------
__device__ __forceinline__ int e4m3_row_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int k;
  const float m = frexpf(amax, &k);  // amax = m 2^k, 0.5 <= m < 1; 448 = 0.875 2^9
  return m <= 0.875f ? k - 9 : k - 8;
}

// four consecutive columns times 2^-e as E4M3 codes, the first in the low byte
__device__ __forceinline__ uint32_t e4m3_pack4(float a, float b, float c, float d, int e) {
  const __nv_fp8x2_storage_t lo =
      __nv_cvt_float2_to_fp8x2(make_float2(ldexpf(a, -e), ldexpf(b, -e)), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi =
      __nv_cvt_float2_to_fp8x2(make_float2(ldexpf(c, -e), ldexpf(d, -e)), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// two E4M3 codes (the low byte first) widened to fp32
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t w16) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w16 & 0xffffu), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

}  // namespace rs
