"""Thin ctypes binding of libreplayssm.so (same entry-point names as the C ABI).

Argument marshalling only: tensors are checked for device, dtype and layout,
their ``data_ptr()`` and strides go into an ``rs_step_args`` struct, and the
call runs on the current torch CUDA stream (or the one given).  Every step of
the computation runs in the library's CUDA kernels; there is no CPU fallback,
and loading fails loudly when the library has not been built.

C declarations and their documentation: include/replayssm.h.
"""

import ctypes
import os

import numpy as np

from . import build as _build

RS_OK, RS_EINVAL, RS_EUNSUPPORTED, RS_EALIGN, RS_ECUDA = 0, -1, -2, -3, -4
RS_F32, RS_F16, RS_BF16, RS_F8E4M3 = 0, 1, 2, 3
RS_MAMBA2, RS_GDN = 0, 1
RS_DERR_SLOT, RS_DERR_WRITE_POS, RS_DERR_TIMEOUT, RS_DERR_DST, RS_DERR_ACCEPTED = 1, 2, 4, 8, 16
RS_ABI_VERSION = 4
RS_MAX_L = 64
RS_NOALLOC_KQ_FLOATS = 1 << 20

# every symbol include/replayssm.h declares
EXPORTS = (
    "replayssm_abi_version",
    "replayssm_supported",
    "replayssm_plan_step",
    "replayssm_plan_align",
    "replayssm_materialize",
    "replayssm_spec_verify_mamba2",
    "replayssm_plan_spec",
    "replayssm_spec_commit",
    "replayssm_seed_read_copy",
    "replayssm_decode_mamba2",
    "replayssm_decode_mamba2_noalloc",
    "replayssm_decode_gdn",
    "conventional_decode",
    "replayssm_status_string",
)


class StepArgs(ctypes.Structure):
    """Mirror of ``rs_step_args``."""

    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("d_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
        ("L", ctypes.c_int32), ("num_slots", ctypes.c_int32), ("ckpt_dtype", ctypes.c_int32),
        ("in_dtype", ctypes.c_int32), ("ring_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("slot_idx", ctypes.c_void_p), ("write_pos", ctypes.c_void_p), ("is_flush", ctypes.c_void_p),
        ("v", ctypes.c_void_p), ("k", ctypes.c_void_p), ("q", ctypes.c_void_p),
        ("alpha", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("ckpt", ctypes.c_void_p), ("ring_v", ctypes.c_void_p), ("ring_k", ctypes.c_void_p),
        ("ring_a", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("stride_v_row", ctypes.c_int64), ("stride_k_row", ctypes.c_int64),
        ("stride_q_row", ctypes.c_int64), ("stride_out_row", ctypes.c_int64),
        ("dev_err", ctypes.c_void_p),
        ("ckpt_lp", ctypes.c_void_p), ("lp_dtype", ctypes.c_int32), ("reserved2", ctypes.c_int32),
        ("n_groups", ctypes.c_int32), ("reserved3", ctypes.c_int32), ("kq_scratch", ctypes.c_void_p),
        ("ckpt_lp_scale", ctypes.c_void_p),
    ]


class MaterializeArgs(ctypes.Structure):
    """Mirror of ``rs_materialize_args``."""

    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("d_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
        ("L", ctypes.c_int32), ("num_slots", ctypes.c_int32), ("num_dst", ctypes.c_int32),
        ("ckpt_dtype", ctypes.c_int32), ("ring_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("slot_idx", ctypes.c_void_p), ("held", ctypes.c_void_p), ("dst_idx", ctypes.c_void_p),
        ("ckpt", ctypes.c_void_p), ("ring_v", ctypes.c_void_p), ("ring_k", ctypes.c_void_p),
        ("ring_a", ctypes.c_void_p), ("dst", ctypes.c_void_p), ("dev_err", ctypes.c_void_p),
    ]


class SpecArgs(ctypes.Structure):
    """Mirror of ``rs_spec_args``."""

    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("d_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
        ("L", ctypes.c_int32), ("T", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("ckpt_dtype", ctypes.c_int32), ("in_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("slot_idx", ctypes.c_void_p), ("committed", ctypes.c_void_p), ("is_flush", ctypes.c_void_p),
        ("v", ctypes.c_void_p), ("k", ctypes.c_void_p), ("q", ctypes.c_void_p), ("alpha", ctypes.c_void_p),
        ("ckpt", ctypes.c_void_p), ("ring_v", ctypes.c_void_p), ("ring_k", ctypes.c_void_p),
        ("ring_a", ctypes.c_void_p), ("out", ctypes.c_void_p), ("dev_err", ctypes.c_void_p),
    ]


_LIB = None


def load():
    """Load the library (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (linear_attention_decode_replayssm_gb300.build.build())")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.replayssm_abi_version.restype = ctypes.c_int
    lib.replayssm_abi_version.argtypes = []
    lib.replayssm_supported.restype = ctypes.c_int
    lib.replayssm_supported.argtypes = [ctypes.c_int] * 4
    lib.replayssm_plan_step.restype = ctypes.c_int
    lib.replayssm_plan_step.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_void_p, ctypes.c_void_p]
    lib.replayssm_plan_align.restype = ctypes.c_int
    lib.replayssm_plan_align.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    lib.replayssm_materialize.restype = ctypes.c_int
    lib.replayssm_materialize.argtypes = [P(MaterializeArgs), ctypes.c_int, ctypes.c_void_p]
    lib.replayssm_spec_verify_mamba2.restype = ctypes.c_int
    lib.replayssm_spec_verify_mamba2.argtypes = [P(SpecArgs), ctypes.c_void_p]
    lib.replayssm_plan_spec.restype = ctypes.c_int
    lib.replayssm_plan_spec.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_void_p]
    lib.replayssm_spec_commit.restype = ctypes.c_int
    lib.replayssm_spec_commit.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int32] * 3 + [ctypes.c_void_p] * 4
    for name in ("replayssm_decode_mamba2", "replayssm_decode_mamba2_noalloc", "replayssm_decode_gdn"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [P(StepArgs), ctypes.c_void_p]
    lib.conventional_decode.restype = ctypes.c_int
    lib.conventional_decode.argtypes = [P(StepArgs), ctypes.c_int, ctypes.c_void_p]
    lib.replayssm_seed_read_copy.restype = ctypes.c_int
    lib.replayssm_seed_read_copy.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.replayssm_status_string.restype = ctypes.c_char_p
    lib.replayssm_status_string.argtypes = [ctypes.c_int]
    got = lib.replayssm_abi_version()
    if got != RS_ABI_VERSION:
        raise RuntimeError(f"libreplayssm ABI version {got}, binding expects {RS_ABI_VERSION}")
    _LIB = lib
    return lib


def status_string(status):
    return load().replayssm_status_string(int(status)).decode()


def _check(status, what):
    if status != RS_OK:
        raise RuntimeError(f"{what}: {status_string(status)}")
    return status


def replayssm_abi_version():
    return load().replayssm_abi_version()


def replayssm_supported(variant, d_v, d_k, ckpt_dtype):
    return bool(load().replayssm_supported(int(variant), int(d_v), int(d_k), int(ckpt_dtype)))


# --------------------------------------------------------------------------
# host step plan
# --------------------------------------------------------------------------
def replayssm_plan_step(decode_step, L, force_flush=None, write_pos=None, is_flush=None):
    """Per-row cursor and flush flag on the host (NumPy arrays; optional
    preallocated outputs, e.g. pinned-memory views)."""
    ds = np.ascontiguousarray(decode_step, dtype=np.int64)
    B = ds.shape[0]
    if write_pos is None:
        write_pos = np.empty(B, dtype=np.int32)
    if is_flush is None:
        is_flush = np.empty(B, dtype=np.uint8)
    ff = None
    if force_flush is not None:
        ff = np.ascontiguousarray(force_flush, dtype=np.uint8)
        if ff.shape != (B,):
            raise ValueError("force_flush must have shape [B]")
    if write_pos.dtype != np.int32 or is_flush.dtype != np.uint8 or not (
            write_pos.flags.c_contiguous and is_flush.flags.c_contiguous):
        raise ValueError("write_pos must be contiguous int32 and is_flush contiguous uint8")
    _check(load().replayssm_plan_step(ds.ctypes.data, None if ff is None else ff.ctypes.data, B, int(L),
                                      write_pos.ctypes.data, is_flush.ctypes.data), "replayssm_plan_step")
    return write_pos, is_flush


def replayssm_plan_align(position, start, L, block, write_pos=None, is_flush=None):
    """Align (prefix-caching) mode cursor and flag on the host: forced flush
    on the token that completes a cache block of ``block`` tokens, ring
    re-anchored at each block start (block 0 = off)."""
    pos = np.ascontiguousarray(position, dtype=np.int64)
    st = np.ascontiguousarray(start, dtype=np.int64)
    B = pos.shape[0]
    if st.shape != (B,):
        raise ValueError("start must have shape [B]")
    if write_pos is None:
        write_pos = np.empty(B, dtype=np.int32)
    if is_flush is None:
        is_flush = np.empty(B, dtype=np.uint8)
    if write_pos.dtype != np.int32 or is_flush.dtype != np.uint8 or not (
            write_pos.flags.c_contiguous and is_flush.flags.c_contiguous):
        raise ValueError("write_pos must be contiguous int32 and is_flush contiguous uint8")
    _check(load().replayssm_plan_align(pos.ctypes.data, st.ctypes.data, int(block), B, int(L),
                                       write_pos.ctypes.data, is_flush.ctypes.data), "replayssm_plan_align")
    return write_pos, is_flush


# --------------------------------------------------------------------------
# decode steps
# --------------------------------------------------------------------------
def _torch():
    import torch

    return torch


def _dtype_code(t):
    torch = _torch()
    m = {torch.float32: RS_F32, torch.float16: RS_F16, torch.bfloat16: RS_BF16, torch.float8_e4m3fn: RS_F8E4M3}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def _need(t, name, dtype=None, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t


def _rows(t, name, H, d):
    """[B, H, d] with packed heads and a free row stride; returns row stride."""
    if t.shape[1:] != (H, d) or t.stride(2) != 1 or t.stride(1) != d:
        raise ValueError(f"{name} must be [B, {H}, {d}] with packed heads (got {tuple(t.shape)}, strides {t.stride()})")
    return t.stride(0)


def _fill(args, *, variant, ckpt, slot_idx, v, k, q, alpha, out, beta=None, ring_v=None, ring_k=None,
          ring_a=None, write_pos=None, is_flush=None, dev_err=None, ckpt_lp=None, kq_scratch=None,
          library_scratch=False, ckpt_lp_scale=None):
    torch = _torch()
    _need(ckpt, "ckpt", ndim=4)
    if not ckpt.is_contiguous():
        raise ValueError("ckpt must be contiguous [num_slots, H, d_v, d_k]")
    S, H, d_v, d_k = ckpt.shape
    _need(slot_idx, "slot_idx", torch.int32, 1)
    B = slot_idx.shape[0]
    for name, t in (("v", v), ("k", k), ("q", q)):
        _need(t, name, ndim=3)
        if t.shape[0] != B:
            raise ValueError(f"{name} has {t.shape[0]} rows, slot_idx has {B}")
    if not (v.dtype == k.dtype == q.dtype):
        raise TypeError("v, k, q must share one dtype")
    _need(alpha, "alpha", torch.float32, 2)
    _need(out, "out", torch.float32, 3)
    if alpha.shape != (B, H) or not alpha.is_contiguous():
        raise ValueError("alpha must be contiguous [B, H]")
    if out.shape[0] != B:
        raise ValueError("out must have B rows")
    args.B, args.H, args.d_v, args.d_k, args.num_slots = B, H, d_v, d_k, S
    args.ckpt_dtype, args.in_dtype = _dtype_code(ckpt), _dtype_code(v)
    args.reserved = 0
    args.slot_idx, args.ckpt = slot_idx.data_ptr(), ckpt.data_ptr()
    args.v, args.k, args.q = v.data_ptr(), k.data_ptr(), q.data_ptr()
    args.alpha, args.out = alpha.data_ptr(), out.data_ptr()
    # group-shared keys and queries: k, q [B, G, d_k] with G dividing H
    KH = k.shape[1]
    G = 0 if KH == H else KH
    if G and (H % G or q.shape[1] != G):
        raise ValueError(f"k and q must have H = {H} heads or a number of groups dividing it")
    args.stride_v_row = _rows(v, "v", H, d_v)
    args.stride_k_row = _rows(k, "k", KH, d_k)
    args.stride_q_row = _rows(q, "q", KH, d_k)
    args.n_groups, args.reserved3 = G, 0
    if G and library_scratch:
        args.kq_scratch = None
    elif G:
        _need(kq_scratch, "kq_scratch", torch.float32)
        if kq_scratch.numel() < B * G * ring_a.shape[2] or not kq_scratch.is_contiguous():
            raise ValueError("kq_scratch must be a contiguous float32 buffer of at least B * G * L elements")
        args.kq_scratch = kq_scratch.data_ptr()
    else:
        args.kq_scratch = None
    args.stride_out_row = _rows(out, "out", H, d_v)
    if variant == RS_GDN:
        _need(beta, "beta", torch.float32, 2)
        if beta.shape != (B, H) or not beta.is_contiguous():
            raise ValueError("beta must be contiguous [B, H]")
        args.beta = beta.data_ptr()
    else:
        args.beta = None
    if ring_v is not None:
        for name, t, shp in (("ring_v", ring_v, (S, H, None, d_v)), ("ring_k", ring_k, (S, k.shape[1], None, d_k)),
                             ("ring_a", ring_a, (S, H, None))):
            _need(t, name)
            if not t.is_contiguous() or t.dim() != len(shp) or any(
                    want is not None and got != want for got, want in zip(t.shape, shp)):
                raise ValueError(f"{name} must be contiguous with shape {shp} (None = L)")
        L = ring_a.shape[2]
        if ring_v.shape[2] != L or ring_k.shape[2] != L:
            raise ValueError("ring_v, ring_k and ring_a disagree on L")
        if ring_v.dtype != ring_k.dtype or ring_a.dtype != torch.float32:
            raise TypeError("ring_v and ring_k share a dtype; ring_a is float32")
        _need(write_pos, "write_pos", torch.int32, 1)
        _need(is_flush, "is_flush", torch.uint8, 1)
        if write_pos.shape[0] != B or is_flush.shape[0] != B:
            raise ValueError("write_pos and is_flush must have B entries")
        args.L = L
        args.ring_dtype = _dtype_code(ring_v)
        args.ring_v, args.ring_k, args.ring_a = ring_v.data_ptr(), ring_k.data_ptr(), ring_a.data_ptr()
        args.write_pos, args.is_flush = write_pos.data_ptr(), is_flush.data_ptr()
    else:
        args.L, args.ring_dtype = 0, args.in_dtype
        args.ring_v = args.ring_k = args.ring_a = args.write_pos = args.is_flush = None
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32)
        args.dev_err = dev_err.data_ptr()
    else:
        args.dev_err = None
    args.reserved2 = 0
    if ckpt_lp is not None:
        _need(ckpt_lp, "ckpt_lp", ndim=4)
        if not ckpt_lp.is_contiguous() or ckpt_lp.shape != ckpt.shape:
            raise ValueError("ckpt_lp must be contiguous with the shape of ckpt")
        args.ckpt_lp, args.lp_dtype = ckpt_lp.data_ptr(), _dtype_code(ckpt_lp)
    else:
        args.ckpt_lp, args.lp_dtype = None, 0
    if ckpt_lp_scale is not None:
        _need(ckpt_lp_scale, "ckpt_lp_scale", torch.float32)
        if not ckpt_lp_scale.is_contiguous() or ckpt_lp_scale.shape != ckpt.shape[:3]:
            raise ValueError("ckpt_lp_scale must be contiguous float32 [num_slots, H, d_v]")
        args.ckpt_lp_scale = ckpt_lp_scale.data_ptr()
    else:
        args.ckpt_lp_scale = None
    return args


def _stream(stream):
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def replayssm_decode_mamba2(*, ckpt, ring_v, ring_k, ring_a, slot_idx, write_pos, is_flush, v, k, q, alpha,
                            out, dev_err=None, stream=None, ckpt_lp=None, kq_scratch=None, ckpt_lp_scale=None):
    """One ReplaySSM Mamba-2 decode step in place on ckpt and the rings; o in
    ``out``.  ``ckpt_lp`` (fp16, bf16 or float8_e4m3fn, shape of ckpt) makes
    ckpt the recurrence copy of a two-precision checkpoint and ckpt_lp its
    read copy; an E4M3 copy takes its row scales in ``ckpt_lp_scale``
    (float32 [slots, H, d_v]).  k and q of shape [B, G, d_k] (G < H groups)
    select group-shared keys, with ring_k [slots, G, L, d_k] and a float32
    ``kq_scratch`` of B * G * L."""
    args = _fill(StepArgs(), variant=RS_MAMBA2, ckpt=ckpt, slot_idx=slot_idx, v=v, k=k, q=q, alpha=alpha,
                 out=out, ring_v=ring_v, ring_k=ring_k, ring_a=ring_a, write_pos=write_pos,
                 is_flush=is_flush, dev_err=dev_err, ckpt_lp=ckpt_lp, kq_scratch=kq_scratch,
                 ckpt_lp_scale=ckpt_lp_scale)
    return _check(load().replayssm_decode_mamba2(ctypes.byref(args), _stream(stream)), "replayssm_decode_mamba2")


def replayssm_seed_read_copy(*, ckpt, ckpt_lp, scale=None, stream=None):
    """Cast the recurrence copy ``ckpt`` (float32, last dim d_k) into its read
    copy ``ckpt_lp`` (same shape; fp16, bf16 or float8_e4m3fn, the last with
    its row scales in ``scale``, float32 of shape ckpt.shape[:-1])."""
    torch = _torch()
    _need(ckpt, "ckpt", torch.float32)
    _need(ckpt_lp, "ckpt_lp")
    if not ckpt.is_contiguous() or not ckpt_lp.is_contiguous() or ckpt_lp.shape != ckpt.shape:
        raise ValueError("ckpt and ckpt_lp must be contiguous with one shape")
    d_k = ckpt.shape[-1]
    n_rows = ckpt.numel() // d_k
    lp = _dtype_code(ckpt_lp)
    sp = None
    if lp == RS_F8E4M3:
        _need(scale, "scale", torch.float32)
        if not scale.is_contiguous() or scale.shape != ckpt.shape[:-1]:
            raise ValueError("scale must be contiguous float32 of shape ckpt.shape[:-1]")
        sp = scale.data_ptr()
    return _check(load().replayssm_seed_read_copy(ckpt.data_ptr(), n_rows, d_k, lp, ckpt_lp.data_ptr(), sp,
                                                  _stream(stream)), "replayssm_seed_read_copy")


def replayssm_decode_mamba2_noalloc(*, ckpt, ring_v, ring_k, ring_a, slot_idx, write_pos, is_flush, v, k, q,
                                    alpha, out, dev_err=None, stream=None):
    """As ``replayssm_decode_mamba2``, for callers that cannot allocate device
    memory: group-shared keys use a fixed-size device array held by the
    library (B * G * L <= RS_NOALLOC_KQ_FLOATS) instead of caller scratch.
    The first call on a device looks up that array's address, so make it
    before any stream capture; calls that overlap on the GPU race on it."""
    args = _fill(StepArgs(), variant=RS_MAMBA2, ckpt=ckpt, slot_idx=slot_idx, v=v, k=k, q=q, alpha=alpha,
                 out=out, ring_v=ring_v, ring_k=ring_k, ring_a=ring_a, write_pos=write_pos,
                 is_flush=is_flush, dev_err=dev_err, library_scratch=True)
    return _check(load().replayssm_decode_mamba2_noalloc(ctypes.byref(args), _stream(stream)),
                  "replayssm_decode_mamba2_noalloc")


def replayssm_decode_gdn(*, ckpt, ring_v, ring_k, ring_a, slot_idx, write_pos, is_flush, v, k, q, alpha, beta,
                         out, dev_err=None, stream=None):
    """One ReplaySSM Gated DeltaNet decode step (alpha holds the log-gate g)."""
    args = _fill(StepArgs(), variant=RS_GDN, ckpt=ckpt, slot_idx=slot_idx, v=v, k=k, q=q, alpha=alpha,
                 beta=beta, out=out, ring_v=ring_v, ring_k=ring_k, ring_a=ring_a, write_pos=write_pos,
                 is_flush=is_flush, dev_err=dev_err)
    return _check(load().replayssm_decode_gdn(ctypes.byref(args), _stream(stream)), "replayssm_decode_gdn")


def conventional_decode(*, variant, state, slot_idx, v, k, q, alpha, out, beta=None, dev_err=None, stream=None):
    """One conventional load-update-store step on ``state`` [num_slots, H, d_v, d_k]."""
    args = _fill(StepArgs(), variant=variant, ckpt=state, slot_idx=slot_idx, v=v, k=k, q=q, alpha=alpha,
                 beta=beta, out=out, dev_err=dev_err)
    return _check(load().conventional_decode(ctypes.byref(args), int(variant), _stream(stream)),
                  "conventional_decode")


def replayssm_materialize(*, variant, ckpt, ring_v, ring_k, ring_a, slot_idx, held, dst, dst_idx, dev_err=None,
                          stream=None):
    """Exact state of each row (checkpoint unrolled with its ``held`` ring
    records) written to ``dst[dst_idx[b]]``; checkpoint and ring only read."""
    torch = _torch()
    _need(ckpt, "ckpt", ndim=4)
    _need(dst, "dst", ckpt.dtype, 4)
    if not ckpt.is_contiguous() or not dst.is_contiguous() or dst.shape[1:] != ckpt.shape[1:]:
        raise ValueError("ckpt and dst must be contiguous [slots, H, d_v, d_k] of one shape and dtype")
    S, H, d_v, d_k = ckpt.shape
    for name, t, shp in (("ring_v", ring_v, (S, H, None, d_v)), ("ring_k", ring_k, (S, H, None, d_k)),
                         ("ring_a", ring_a, (S, H, None))):
        _need(t, name)
        if not t.is_contiguous() or t.dim() != len(shp) or any(
                want is not None and got != want for got, want in zip(t.shape, shp)):
            raise ValueError(f"{name} must be contiguous with shape {shp} (None = L)")
    L = ring_a.shape[2]
    if ring_v.shape[2] != L or ring_k.shape[2] != L or ring_v.dtype != ring_k.dtype:
        raise ValueError("ring_v, ring_k and ring_a disagree on L or dtype")
    _need(ring_a, "ring_a", torch.float32)
    for name, t in (("slot_idx", slot_idx), ("held", held), ("dst_idx", dst_idx)):
        _need(t, name, torch.int32, 1)
    B = slot_idx.shape[0]
    if held.shape[0] != B or dst_idx.shape[0] != B:
        raise ValueError("slot_idx, held and dst_idx must have B entries")
    a = MaterializeArgs()
    a.B, a.H, a.d_v, a.d_k, a.L, a.num_slots, a.num_dst = B, H, d_v, d_k, L, S, dst.shape[0]
    a.ckpt_dtype, a.ring_dtype, a.reserved = _dtype_code(ckpt), _dtype_code(ring_v), 0
    a.slot_idx, a.held, a.dst_idx = slot_idx.data_ptr(), held.data_ptr(), dst_idx.data_ptr()
    a.ckpt, a.ring_v, a.ring_k, a.ring_a = ckpt.data_ptr(), ring_v.data_ptr(), ring_k.data_ptr(), ring_a.data_ptr()
    a.dst = dst.data_ptr()
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32)
        a.dev_err = dev_err.data_ptr()
    else:
        a.dev_err = None
    return _check(load().replayssm_materialize(ctypes.byref(a), int(variant), _stream(stream)),
                  "replayssm_materialize")


def replayssm_plan_spec(committed, L, T, is_flush=None):
    """Host flag of a verification step: committed + T > L (NumPy arrays)."""
    h = np.ascontiguousarray(committed, dtype=np.int32)
    B = h.shape[0]
    if is_flush is None:
        is_flush = np.empty(B, dtype=np.uint8)
    if is_flush.dtype != np.uint8 or not is_flush.flags.c_contiguous:
        raise ValueError("is_flush must be contiguous uint8")
    _check(load().replayssm_plan_spec(h.ctypes.data, B, int(L), int(T), is_flush.ctypes.data), "replayssm_plan_spec")
    return is_flush


def replayssm_spec_verify_mamba2(*, ckpt, ring_v, ring_k, ring_a, slot_idx, committed, is_flush, v, k, q, alpha,
                                 out, dev_err=None, stream=None):
    """Verify T draft tokens per row (v [B, T, H, d_v], k, q [B, T, H, d_k],
    alpha [B, T, H]); outputs in ``out`` [B, T, H, d_v].  Commits nothing."""
    torch = _torch()
    _need(ckpt, "ckpt", ndim=4)
    if not ckpt.is_contiguous():
        raise ValueError("ckpt must be contiguous [num_slots, H, d_v, d_k]")
    S, H, d_v, d_k = ckpt.shape
    _need(slot_idx, "slot_idx", torch.int32, 1)
    B = slot_idx.shape[0]
    _need(alpha, "alpha", torch.float32, 3)
    T = alpha.shape[1]
    for name, t, d in (("v", v, d_v), ("k", k, d_k), ("q", q, d_k)):
        _need(t, name, ndim=4)
        if t.shape != (B, T, H, d) or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [B, T, H, {d}]")
    if not (v.dtype == k.dtype == q.dtype):
        raise TypeError("v, k, q must share one dtype")
    if alpha.shape != (B, T, H) or not alpha.is_contiguous():
        raise ValueError("alpha must be contiguous [B, T, H]")
    _need(out, "out", torch.float32, 4)
    if out.shape != (B, T, H, d_v) or not out.is_contiguous():
        raise ValueError("out must be contiguous [B, T, H, d_v]")
    for name, t, shp in (("ring_v", ring_v, (S, H, None, d_v)), ("ring_k", ring_k, (S, H, None, d_k)),
                         ("ring_a", ring_a, (S, H, None))):
        _need(t, name)
        if not t.is_contiguous() or t.dim() != len(shp) or any(
                want is not None and got != want for got, want in zip(t.shape, shp)):
            raise ValueError(f"{name} must be contiguous with shape {shp} (None = L)")
    if ring_v.dtype != v.dtype or ring_k.dtype != v.dtype:
        raise TypeError("Mamba-2 rings hold the inputs verbatim: ring dtype must equal the input dtype")
    _need(committed, "committed", torch.int32, 1)
    _need(is_flush, "is_flush", torch.uint8, 1)
    a = SpecArgs()
    a.B, a.H, a.d_v, a.d_k, a.L, a.T, a.num_slots = B, H, d_v, d_k, ring_a.shape[2], T, S
    a.ckpt_dtype, a.in_dtype, a.reserved = _dtype_code(ckpt), _dtype_code(v), 0
    a.slot_idx, a.committed, a.is_flush = slot_idx.data_ptr(), committed.data_ptr(), is_flush.data_ptr()
    a.v, a.k, a.q, a.alpha = v.data_ptr(), k.data_ptr(), q.data_ptr(), alpha.data_ptr()
    a.ckpt, a.ring_v, a.ring_k, a.ring_a = ckpt.data_ptr(), ring_v.data_ptr(), ring_k.data_ptr(), ring_a.data_ptr()
    a.out = out.data_ptr()
    a.dev_err = dev_err.data_ptr() if dev_err is not None else None
    return _check(load().replayssm_spec_verify_mamba2(ctypes.byref(a), _stream(stream)),
                  "replayssm_spec_verify_mamba2")


def replayssm_spec_commit(*, committed, is_flush, accepted, L, T, committed_out=None, is_flush_out=None,
                          dev_err=None, stream=None):
    """Device-side pointer commit; in place unless outputs are given."""
    torch = _torch()
    _need(committed, "committed", torch.int32, 1)
    _need(is_flush, "is_flush", torch.uint8, 1)
    _need(accepted, "accepted", torch.int32, 1)
    committed_out = committed if committed_out is None else committed_out
    is_flush_out = is_flush if is_flush_out is None else is_flush_out
    B = committed.shape[0]
    return _check(load().replayssm_spec_commit(committed.data_ptr(), is_flush.data_ptr(), accepted.data_ptr(), B,
                                               int(L), int(T), committed_out.data_ptr(), is_flush_out.data_ptr(),
                                               None if dev_err is None else dev_err.data_ptr(), _stream(stream)),
                  "replayssm_spec_commit")


class PreparedStep:
    """One decode entry point with its arguments marshalled once.

    For a serving loop whose buffers stay at the same addresses from step to
    step: the tensors are checked and their addresses written into an
    ``rs_step_args`` struct once, and each ``launch`` is then a single call
    of the C entry point.  The call reads the tensors' contents when it runs
    on the stream, so they may change between launches; the tensors
    themselves must stay alive (this object keeps references to them).
    """

    def __init__(self, name, args, tensors):
        self.name, self._args, self._tensors = name, args, tensors
        self._fn = getattr(load(), name)

    def launch(self, stream=None):
        return _check(self._fn(ctypes.byref(self._args), _stream(stream)), self.name)


def prepare_decode(name, **kw):
    """A ``PreparedStep`` of ``replayssm_decode_mamba2`` or
    ``replayssm_decode_gdn``, with the keyword arguments of that function
    (``stream`` is given to ``launch`` instead)."""
    variants = {"replayssm_decode_mamba2": RS_MAMBA2, "replayssm_decode_gdn": RS_GDN}
    if name not in variants:
        raise ValueError(f"no prepared form of {name}")
    return PreparedStep(name, _fill(StepArgs(), variant=variants[name], **kw), dict(kw))


def raw_call(name, args, *extra):
    """Call an entry point with a prepared StepArgs and return the status
    (no exception).  Used to exercise the C-side validation."""
    fn = getattr(load(), name)
    return fn(ctypes.byref(args), *extra)
