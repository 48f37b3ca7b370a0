/*
 * replayssm.h -- C ABI of libreplayssm.so, the GB300 (sm_103a) ReplaySSM
 * cached SSM decode step.
 *
 * Sources, cited below by short name:
 *   [Ghana]   S. Ghana, "ReplaySSM: an SSM decoder that writes its state once
 *             every 16 tokens".
 *   [PR48792] vLLM pull request 48792, "[Kernel] ReplaySSM: cache SSM inputs
 *             for faster Gated DeltaNet standard decode".
 *   [NV]      NVIDIA technical blog, "ReplaySSM: Rethinking State Storage for
 *             Faster Hybrid Model Decoding".
 *
 * What a decode step computes (per batch row b and head h, p = write_pos[b]
 * records already in the row's ring, the current token being record p + 1):
 *
 *   Mamba-2 non-flush ([Ghana] §Output without a state):
 *     o = gamma_{p+1} S_ckpt q + sum_{j=1..p+1} gamma_{j+1:p+1} v_j (k_j . q),
 *     then the record (alpha, v, k) is appended at ring slot p.
 *   Two-precision checkpoint ([Ghana] §The precision argument, derived):
 *     non-flush rows read a low-precision copy of the checkpoint, flushes
 *     read the full-precision one and refresh both (rs_step_args.ckpt_lp).
 *   Mamba-2 flush ([Ghana] §The identity):
 *     S_new = gamma_{p+1} S_ckpt + sum_j gamma_{j+1:p+1} v_j k_j^T,
 *     o = S_new q (unrounded), S_ckpt <- S_new cast to the checkpoint type;
 *     no record is appended and the ring is logically empty afterwards.
 *   Gated DeltaNet ([Ghana] §The delta-rule wrinkle; [PR48792] §Core concept
 *   and the review comment on S_{t-1} q and S_{t-1} k): the ring holds the
 *   corrected value d, the key k and the log-gate g; with
 *     G_j = exp(sum_{l=j+1..p} g_l), Gamma = exp(sum_{l<=p} g_l),
 *     S_{t-1} x = Gamma S_ckpt x + sum_{j<=p} G_j (k_j . x) d_j  (x = k_t, q_t),
 *     alpha_t = exp(g_t), d_t = beta_t (v_t - alpha_t S_{t-1} k_t),
 *     o = alpha_t S_{t-1} q_t + d_t (k_t . q_t);
 *   non-flush appends (d_t, k_t, g_t) rounded to the ring type; flush stores
 *   S_new = alpha_t S_{t-1} + d_t k_t^T (from the unrounded d_t) and outputs
 *   S_new q_t.
 *   Conventional baseline ([Ghana] §Why a fixed-size state is not cheap to
 *   decode): load the state, S <- alpha S + v k^T (delta rule for GDN),
 *   o = S q, store the state, every step.
 *
 * Memory and ownership: every pointer in rs_step_args is a DEVICE pointer
 * owned by the caller (PyTorch allocates and frees everything).  The library
 * never allocates, frees or synchronises, and never reads device memory on
 * the host, so a call is asynchronous on `stream`, and the decode,
 * verification, commit and materialisation calls can be captured in a CUDA
 * graph ([PR48792] §CUDA graphs and continuous batching).  (The no-alloc
 * decode variant below has its own set-up rule.)  Checkpoint and
 * rings are updated in place.  Two rows of one call must not name the same
 * slot (their updates would race).
 *
 * Errors: arguments are validated on the host before anything is launched; an
 * invalid call returns a negative rs_status and launches nothing.  A failed
 * launch returns RS_ECUDA.  Values only the device sees (slot_idx, write_pos)
 * are range-checked in the kernel: a row with an out-of-range slot or cursor
 * is skipped (its output row is zero-filled, no state is touched) and the
 * matching RS_DERR_* bit is OR-ed into *dev_err when dev_err is not NULL.  The
 * kernels never trap.
 */
#ifndef REPLAYSSM_H_
#define REPLAYSSM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *rs_stream_t;

#define RS_ABI_VERSION 4
#define RS_MAX_L 64 /* largest supported buffer length */

typedef enum {
  RS_OK = 0,
  RS_EINVAL = -1,       /* a null pointer, a bad size or an inconsistent argument */
  RS_EUNSUPPORTED = -2, /* shape / dtype combination not built into the library */
  RS_EALIGN = -3,       /* a pointer or row stride breaks the 16-byte rule below */
  RS_ECUDA = -4         /* the CUDA runtime reported an error at launch */
} rs_status;

typedef enum {
  RS_F32 = 0,
  RS_F16 = 1,
  RS_BF16 = 2,
  RS_F8E4M3 = 3 /* read copy of a two-precision checkpoint only (see ckpt_lp) */
} rs_dtype;

typedef enum { RS_MAMBA2 = 0, RS_GDN = 1 } rs_variant;

/* Bits the kernels OR into *dev_err. */
typedef enum {
  RS_DERR_SLOT = 1,      /* slot_idx[b] >= num_slots */
  RS_DERR_WRITE_POS = 2, /* write_pos[b] outside [0, L) */
  RS_DERR_TIMEOUT = 4,   /* a pipeline wait gave up after 2 s: outputs of the
                            call are incomplete (never expected; reported
                            instead of hanging the GPU) */
  RS_DERR_DST = 8,       /* dst_idx[b] >= num_dst (replayssm_materialize) */
  RS_DERR_ACCEPTED = 16  /* accepted[b] outside [1, T] (replayssm_spec_commit) */
} rs_dev_error;

/*
 * One decode step of a batch over a paged state pool ([PR48792] §Paged cache
 * layout: checkpoint and ring caches live in the per-request state block;
 * the block table becomes slot_idx here).
 *
 * Layouts (row-major, last dimension contiguous):
 *   ckpt    [num_slots, H, d_v, d_k]  ckpt_dtype (RS_F32 or RS_F16)
 *   ring_v  [num_slots, H, L, d_v]    ring_dtype: Mamba-2 v records (must equal
 *                                     in_dtype: records are the inputs verbatim);
 *                                     GDN corrected values d (RS_F16 or RS_F32)
 *   ring_k  [num_slots, H, L, d_k]    ring_dtype: key records
 *   ring_a  [num_slots, H, L]         fp32: Mamba-2 decay alpha / GDN log-gate g
 *   v       [B, .. H, d_v]            in_dtype (RS_BF16 or RS_F32); row b starts
 *   k, q    [B, .. H, d_k]            at b * stride_*_row elements, heads packed
 *   alpha   [B, H]                    fp32, packed: Mamba-2 decay in (0,1), or
 *                                     GDN log-gate g (alpha_t = exp(g) )
 *   beta    [B, H]                    fp32, packed; GDN only (NULL for Mamba-2)
 *   out     [B, .. H, d_v]            fp32 output
 *   slot_idx  [B] int32: slot of row b; a negative value marks a padded row,
 *             which touches no state and gets a zero output row.
 *   write_pos [B] int32 in [0, L): records already held by the row's ring.
 *   is_flush  [B] uint8: nonzero = fold the ring and write the checkpoint.
 * Alignment: ckpt, ring_v, ring_k, v, k, q must be 16-byte aligned, and each
 * row stride times the element size a multiple of 16 bytes.
 * Cursor and flag come from replayssm_plan_step (host) each step.
 */
typedef struct rs_step_args {
  int32_t B;          /* rows in the batch (0 = nothing to do) */
  int32_t H;          /* heads per row */
  int32_t d_v, d_k;   /* head dimensions (see replayssm_supported) */
  int32_t L;          /* buffer length, 2 <= L <= RS_MAX_L */
  int32_t num_slots;  /* slots in the paged pools */
  int32_t ckpt_dtype; /* rs_dtype */
  int32_t in_dtype;   /* rs_dtype of v, k, q */
  int32_t ring_dtype; /* rs_dtype of ring_v, ring_k */
  int32_t reserved;   /* must be 0 */
  const int32_t *slot_idx;
  const int32_t *write_pos;
  const uint8_t *is_flush;
  const void *v;
  const void *k;
  const void *q;
  const float *alpha;
  const float *beta;
  void *ckpt;
  void *ring_v;
  void *ring_k;
  float *ring_a;
  float *out;
  int64_t stride_v_row, stride_k_row, stride_q_row, stride_out_row; /* elements */
  int32_t *dev_err; /* optional device int32, see rs_dev_error */
  /* Two-precision checkpoint (Mamba-2 only; NULL = one checkpoint copy):
   * ckpt_lp [num_slots, H, d_v, d_k] of lp_dtype (RS_F16, RS_BF16 or
   * RS_F8E4M3) is the read copy, ckpt (RS_F32) the recurrence copy.  A
   * non-flush row reads only ckpt_lp; a flush row reads ckpt, and casts
   * S_new into both copies, each rounded once (RN-even) from the same fp32
   * matrix.  An RS_F8E4M3 copy (64 x 128 heads) holds each state row on a
   * power-of-two scale: element (s, h, i, j) is its E4M3 code times
   * ckpt_lp_scale[s, h, i], the smallest power of two 2^e with
   * max_j |S[i][j]| <= 448 * 2^e.  The caller seeds ckpt_lp (and the scales)
   * from the same state as ckpt when a request starts
   * (replayssm_seed_read_copy). */
  void *ckpt_lp;
  int32_t lp_dtype;
  int32_t reserved2; /* must be 0 */
  /* Group-shared keys (Mamba-2 only; 0 = a key per head): with n_groups = G
   * dividing H, k and q are [B, .. G, d_k] (head h reads group h / (H / G)),
   * ring_k is [num_slots, G, L, d_k], and kq_scratch is caller-owned device
   * memory of B * G * L floats that the call uses for the group dots
   * k_j . q_t ([Ghana] §Output without a state: computed once per group by
   * a small kernel ahead of the decode).  Not combinable with ckpt_lp. */
  int32_t n_groups;
  int32_t reserved3; /* must be 0 */
  float *kq_scratch;
  /* RS_F8E4M3 read copy: fp32 row scales [num_slots, H, d_v], 16-byte
   * aligned; NULL for any other read copy */
  float *ckpt_lp_scale;
} rs_step_args;

/* RS_ABI_VERSION of the loaded library. */
int replayssm_abi_version(void);

/* 1 if (variant, d_v, d_k, ckpt_dtype) is built into the library, else 0. */
int replayssm_supported(int variant, int d_v, int d_k, int ckpt_dtype);

/*
 * Host-side step plan ([PR48792] §CUDA graphs and continuous batching):
 *   write_pos[b] = decode_step[b] mod L,
 *   is_flush[b]  = (write_pos[b] == L - 1) or force_flush[b] != 0.
 * decode_step [B] >= 0 (tokens the row has decoded), force_flush [B] or NULL;
 * outputs write_pos [B], is_flush [B].  All HOST memory.  After a forced flush
 * the caller re-anchors decode_step so the next cursor is 0 (align mode).
 * Returns RS_OK, or RS_EINVAL (null pointer, B < 0, L outside [1, RS_MAX_L],
 * negative decode_step: outputs untouched).
 */
int replayssm_plan_step(const int64_t *decode_step, const uint8_t *force_flush,
                        int32_t B, int32_t L, int32_t *write_pos, uint8_t *is_flush);

/*
 * Align (prefix-caching) mode step plan ([PR48792] §What this PR adds, the
 * prefix-caching bullet, and §Tests; [Ghana] §What actually shipped).  A
 * cached prefix needs the exact state at every cache-block boundary, and the
 * checkpoint is exact only right after a flush, so the step that completes a
 * block of `block` tokens is forced to flush and the ring is re-anchored at
 * each block start:
 *   anchor[b]    = max(start[b], floor(position[b] / block) * block),
 *   write_pos[b] = (position[b] - anchor[b]) mod L,
 *   is_flush[b]  = (write_pos[b] == L - 1) or ((position[b] + 1) mod block == 0).
 * position [B]: absolute position of the token decoded this step (tokens
 * before it); start [B]: position of the row's first decoded token (the
 * prefill left an exact checkpoint covering the tokens before it).  block = 0
 * turns align mode off: the plain plan of decode_step = position - start.
 * Any L works with any block (L need not divide the block).  All HOST memory.
 * Returns RS_OK, or RS_EINVAL (null pointer, B < 0, L outside [1, RS_MAX_L],
 * block < 0, start < 0 or position < start: outputs untouched).
 */
int replayssm_plan_align(const int64_t *position, const int64_t *start, int32_t block, int32_t B,
                         int32_t L, int32_t *write_pos, uint8_t *is_flush);

/*
 * State materialisation for prefix caching ([Ghana] §What actually shipped:
 * between flushes only the checkpoint and the ring exist, so a separate
 * kernel builds the exact state; §The identity for the unroll).  For each row
 * b with p = held[b] records in its ring, writes
 *   Mamba-2: S = gamma S_ckpt + sum_{j<p} w_j v_j k_j^T,
 *            w_j = product of the decays of records j+1..p-1, gamma = all p;
 *   GDN:     the same with d_j for v_j, w_j = exp(sum of g after j),
 *            gamma = exp(sum of all p log-gates),
 * rounded once (RN-even) to ckpt_dtype, into dst[dst_idx[b]].  The
 * checkpoint and the ring are only read.  held[b] is the cursor the row's
 * next decode step would get (write_pos + 1 after a non-flush step, 0 after
 * a flush).
 *
 * Layouts: ckpt [num_slots, H, d_v, d_k] and dst [num_dst, H, d_v, d_k], both
 * ckpt_dtype (RS_F32 or RS_F16); ring_v [num_slots, H, L, d_v], ring_k
 * [num_slots, H, L, d_k] ring_dtype (RS_F32, RS_F16 or RS_BF16); ring_a
 * [num_slots, H, L] fp32; slot_idx, held, dst_idx [B] int32.  All DEVICE
 * pointers owned by the caller; ckpt, dst, ring_v, ring_k 16-byte aligned.
 * A row with slot_idx or dst_idx negative is skipped.  dst may be ckpt itself
 * when every row's dst_idx equals its slot_idx (an in-place fold: the caller
 * then restarts the row's cursor at 0); otherwise dst must not overlap the
 * checkpoints or rings the call reads, and two rows must not name the same
 * dst slot.  Out-of-range slot_idx, dst_idx or held skip the row and set
 * RS_DERR_SLOT, RS_DERR_DST or RS_DERR_WRITE_POS in *dev_err (when not NULL).
 * variant is RS_MAMBA2 or RS_GDN.  Asynchronous on stream; graph-capturable.
 */
typedef struct rs_materialize_args {
  int32_t B, H, d_v, d_k, L;
  int32_t num_slots;  /* slots in the checkpoint and ring pools */
  int32_t num_dst;    /* slots in the destination pool */
  int32_t ckpt_dtype; /* rs_dtype of ckpt and dst */
  int32_t ring_dtype; /* rs_dtype of ring_v and ring_k */
  int32_t reserved;   /* must be 0 */
  const int32_t *slot_idx;
  const int32_t *held;
  const int32_t *dst_idx;
  const void *ckpt;
  const void *ring_v;
  const void *ring_k;
  const float *ring_a;
  void *dst;
  int32_t *dev_err; /* optional device int32, see rs_dev_error */
} rs_materialize_args;

int replayssm_materialize(const rs_materialize_args *args, int variant, rs_stream_t stream);

/*
 * Speculative verification, Mamba-2 ([Ghana] §Speculative decoding: rollback
 * becomes a pointer; [NV] §Benefit 2, output-only evaluation).  Each row
 * holds h = committed[b] records in its ring (0 <= h <= L) and verifies T
 * draft tokens (1 <= T <= 16, T <= L):
 *   non-flush (h + T <= L): the drafts' records go to ring slots h..h+T-1
 *     and draft i's output is the state after the h committed records and
 *     drafts 0..i, applied to q_i, evaluated without forming that state;
 *   flush (is_flush[b], set when h + T > L): the h committed records are
 *     folded into the checkpoint first (stored, cast to ckpt_dtype), then the
 *     drafts go to ring slots 0..T-1 and their outputs run from the unrounded
 *     folded state.
 * Nothing is committed here: after sampling, replayssm_spec_commit advances
 * the committed count by the accepted drafts; rejected records are simply
 * overwritten later (rollback is a pointer move).
 *
 * Layouts: ckpt [num_slots, H, d_v, d_k] ckpt_dtype (RS_F32 | RS_F16);
 * ring_v [num_slots, H, L, d_v], ring_k [num_slots, H, L, d_k] in in_dtype
 * (records are the inputs verbatim), ring_a [num_slots, H, L] fp32;
 * v [B, T, H, d_v], k, q [B, T, H, d_k] in_dtype (RS_BF16 | RS_F32), packed;
 * alpha [B, T, H] fp32; out [B, T, H, d_v] fp32; slot_idx, committed [B]
 * int32; is_flush [B] uint8.  DEVICE pointers owned by the caller; ckpt,
 * rings, v, k, q 16-byte aligned.  A padded row (slot_idx < 0) gets zero
 * outputs.  An out-of-range slot or committed count (h > L, or h + T > L
 * without is_flush) skips the row (zero outputs) and sets RS_DERR_SLOT /
 * RS_DERR_WRITE_POS in *dev_err.  Asynchronous on stream; graph-capturable.
 */
typedef struct rs_spec_args {
  int32_t B, H, d_v, d_k, L, T;
  int32_t num_slots;
  int32_t ckpt_dtype, in_dtype;
  int32_t reserved; /* must be 0 */
  const int32_t *slot_idx;
  const int32_t *committed;
  const uint8_t *is_flush;
  const void *v;
  const void *k;
  const void *q;
  const float *alpha;
  void *ckpt;
  void *ring_v;
  void *ring_k;
  float *ring_a;
  float *out;
  int32_t *dev_err;
} rs_spec_args;

int replayssm_spec_verify_mamba2(const rs_spec_args *args, rs_stream_t stream);

/*
 * Host plan of a verification step ([Ghana] §Speculative decoding: the flush
 * rule depends only on h and T): is_flush[b] = committed[b] + T > L.  HOST
 * memory.  RS_EINVAL for a null pointer, B < 0, L outside [1, RS_MAX_L], T
 * outside [1, min(L, 16)] or committed[b] outside [0, L] (outputs untouched).
 */
int replayssm_plan_spec(const int32_t *committed, int32_t B, int32_t L, int32_t T, uint8_t *is_flush);

/*
 * Pointer commit after sampling, on the device so it can sit in the same
 * CUDA graph as the verification: with a = accepted[b] in [1, T],
 *   committed_out[b] = (is_flush[b] ? 0 : committed[b]) + a,
 *   is_flush_out[b]  = committed_out[b] + T > L   (the next step's flag).
 * DEVICE pointers; the outputs may alias the inputs.  An accepted count
 * outside [1, T] commits nothing for that row and sets RS_DERR_ACCEPTED.
 */
int replayssm_spec_commit(const int32_t *committed, const uint8_t *is_flush, const int32_t *accepted,
                          int32_t B, int32_t L, int32_t T, int32_t *committed_out, uint8_t *is_flush_out,
                          int32_t *dev_err, rs_stream_t stream);

/*
 * Seed the read copy of a two-precision checkpoint from its recurrence copy
 * ([Ghana] §The precision argument: both copies are roundings of one fp32
 * matrix), e.g. when a request starts: n_rows rows of d_k fp32 values at
 * ckpt (a whole pool is num_slots * H * d_v rows; one slot's heads are H *
 * d_v rows starting at slot * H * d_v) are each rounded once, to nearest
 * even, to lp_dtype in ckpt_lp.  For RS_F8E4M3 each row is first scaled by
 * 2^-e, e the smallest integer with max |row| <= 448 * 2^e (0 for a row of
 * zeros), the E4M3 cast saturates, and 2^e goes to scale[row]; scale is
 * unused (may be NULL) for RS_F16 and RS_BF16.  DEVICE pointers owned by the
 * caller; ckpt and ckpt_lp 16-byte aligned, scale 4-byte aligned; d_k a
 * multiple of 8, at most 1024.  Returns RS_EINVAL for a bad size, a null
 * pointer or another dtype, RS_EALIGN, or RS_ECUDA.  Asynchronous on stream.
 */
int replayssm_seed_read_copy(const float *ckpt, int64_t n_rows, int32_t d_k, int32_t lp_dtype, void *ckpt_lp,
                             float *scale, rs_stream_t stream);

/* ReplaySSM Mamba-2 cached decode step, non-flush and flush rows in one
 * launch (beta unused). */
int replayssm_decode_mamba2(const rs_step_args *args, rs_stream_t stream);

/* Capacity, in floats, of the library-owned group-dot scratch that
 * replayssm_decode_mamba2_noalloc uses: B * n_groups * L must not exceed it
 * (4 MiB; with 8 groups and L = 16 that is up to 8192 rows). */
#define RS_NOALLOC_KQ_FLOATS (1 << 20)

/*
 * replayssm_decode_mamba2 for callers that cannot allocate device memory.
 * The pages have no counterpart: this entry point exists for the callers of
 * this library, not for the method.  The group-shared-key decode needs
 * B * n_groups * L floats of scratch for the group dots k_j . q_t.  Some
 * callers cannot provide it: a plugin inside a serving engine that owns all
 * device memory through its own pool and offers plugins no way to allocate,
 * or a decode loop that must never call cudaMalloc, which can synchronise
 * the device and stall every other stream.  Here the scratch is a
 * fixed-size device array inside the library (RS_NOALLOC_KQ_FLOATS floats,
 * 4 MiB, created when the library's module loads on a device and held by
 * every device that loads it until the process exits); the caller still
 * passes all inputs and outputs, and the call allocates and frees nothing.
 *
 * Set-up: the first call on a device (and the first call after the device's
 * context was reset) looks up the array's device address on the current
 * device, with cudaGetSymbolAddress.  Make that first call before any stream
 * capture begins.  Later calls reuse the address.
 *
 * Sharing: every call uses the same array, which keeps what the last call
 * wrote.  Nothing in it needs clearing: each entry a call reads was written
 * earlier in that same call.  Calls whose kernels overlap on the GPU (on
 * different streams, or in graphs replayed side by side) race on the array
 * and give wrong results: order them.
 *
 * kq_scratch must be NULL.  With n_groups == 0 no scratch is needed and this
 * is replayssm_decode_mamba2.  Returns RS_EINVAL when kq_scratch is set or
 * B * n_groups * L > RS_NOALLOC_KQ_FLOATS (nothing launched), RS_ECUDA when
 * the address lookup fails, otherwise what replayssm_decode_mamba2 returns.
 */
int replayssm_decode_mamba2_noalloc(const rs_step_args *args, rs_stream_t stream);

/* ReplaySSM Gated DeltaNet cached decode step (alpha = log-gate g, beta used). */
int replayssm_decode_gdn(const rs_step_args *args, rs_stream_t stream);

/* Conventional load-update-store step on the same state tensor (ckpt is the
 * state; ring_*, write_pos and is_flush are ignored and may be NULL).
 * variant is RS_MAMBA2 or RS_GDN. */
int conventional_decode(const rs_step_args *args, int variant, rs_stream_t stream);

/* Static string naming an rs_status value. */
const char *replayssm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* REPLAYSSM_H_ */
