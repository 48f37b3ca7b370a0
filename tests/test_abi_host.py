"""Host-side checks of the C ABI that need no GPU.

The library is built here with nvcc (cross-compiling for sm_103a) and loaded;
these tests make no CUDA compute call: the plan is host code, and every decode
call below is rejected by host-side validation before anything is launched.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    with open(os.path.join(ROOT, "include", "replayssm.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|const char \*)\s*(\w+)\(", text, flags=re.M)))


def test_header_and_binding_agree(lib):
    assert sorted(lib.EXPORTS) == _declared_functions()


def test_every_declared_symbol_is_exported(lib):
    so = lib.load()
    for name in _declared_functions():
        assert hasattr(so, name), name
    assert lib.replayssm_abi_version() == lib.RS_ABI_VERSION


def test_supported_set(lib):
    for variant in (lib.RS_MAMBA2, lib.RS_GDN):
        for dv, dk in ((16, 32), (64, 128), (128, 128)):
            for dt in (lib.RS_F32, lib.RS_F16):
                assert lib.replayssm_supported(variant, dv, dk, dt)
    assert not lib.replayssm_supported(lib.RS_MAMBA2, 64, 96, lib.RS_F32)
    assert not lib.replayssm_supported(lib.RS_MAMBA2, 64, 128, lib.RS_BF16)
    assert not lib.replayssm_supported(7, 64, 128, lib.RS_F32)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4):
        assert lib.status_string(code).startswith("RS_")
    assert "unknown" in lib.status_string(99)


# --------------------------------------------------------------------------
# the host step plan, bit-exact against the oracle's closed form
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L", [2, 4, 8, 16, 32, 64])
def test_plan_step_matches_oracle(lib, L):
    r = np.random.default_rng(L)
    ds = r.integers(0, 10 ** 6, size=1000).astype(np.int64)
    ds[:L] = np.arange(L)
    ff = (r.random(1000) < 0.05).astype(np.uint8)
    for force in (None, ff):
        wp, fl = lib.replayssm_plan_step(ds, L, force)
        wp_o, fl_o = oracle.plan_step(ds, L, force)
        np.testing.assert_array_equal(wp, wp_o)
        np.testing.assert_array_equal(fl, fl_o)
        assert wp.dtype == np.int32 and fl.dtype == np.uint8


def test_plan_step_through_a_window_walk(lib):
    # continuous decoding of one row: cursor walks 0..L-1 and flushes once per window
    L = 16
    wp_sim, fl_sim = oracle.simulate_cursors(100, L, start_step=5)
    wp, fl = lib.replayssm_plan_step(5 + np.arange(100), L)
    np.testing.assert_array_equal(wp, wp_sim)
    np.testing.assert_array_equal(fl, fl_sim)


def test_plan_step_rejects_bad_input(lib):
    so = lib.load()
    ds = np.array([0, -1, 3], dtype=np.int64)
    wp = np.full(3, 77, dtype=np.int32)
    fl = np.full(3, 9, dtype=np.uint8)
    assert so.replayssm_plan_step(ds.ctypes.data, None, 3, 16, wp.ctypes.data, fl.ctypes.data) == lib.RS_EINVAL
    np.testing.assert_array_equal(wp, 77)  # outputs untouched on error
    ds = np.zeros(3, dtype=np.int64)
    assert so.replayssm_plan_step(ds.ctypes.data, None, 3, 0, wp.ctypes.data, fl.ctypes.data) == lib.RS_EINVAL
    assert so.replayssm_plan_step(ds.ctypes.data, None, 3, 65, wp.ctypes.data, fl.ctypes.data) == lib.RS_EINVAL
    assert so.replayssm_plan_step(None, None, 3, 16, wp.ctypes.data, fl.ctypes.data) == lib.RS_EINVAL
    assert so.replayssm_plan_step(None, None, 0, 16, None, None) == lib.RS_OK


# --------------------------------------------------------------------------
# argument validation: every case fails before any launch
# --------------------------------------------------------------------------
def _args(lib, **kw):
    a = lib.StepArgs()
    base = dict(B=4, H=2, d_v=64, d_k=128, L=16, num_slots=8, ckpt_dtype=lib.RS_F32, in_dtype=lib.RS_BF16,
                ring_dtype=lib.RS_BF16, reserved=0, slot_idx=0x1000, write_pos=0x2000, is_flush=0x3000,
                v=0x4000, k=0x5000, q=0x6000, alpha=0x7000, beta=0x8000, ckpt=0x9000, ring_v=0xA000,
                ring_k=0xB000, ring_a=0xC000, out=0xD000, stride_v_row=2 * 64, stride_k_row=2 * 128,
                stride_q_row=2 * 128, stride_out_row=2 * 64, dev_err=None)
    base.update(kw)
    for k_, v_ in base.items():
        setattr(a, k_, v_)
    return a


@pytest.mark.parametrize("change, want", [
    (dict(L=1), "RS_EINVAL"),
    (dict(L=65), "RS_EINVAL"),
    (dict(H=0), "RS_EINVAL"),
    (dict(B=-1), "RS_EINVAL"),
    (dict(num_slots=0), "RS_EINVAL"),
    (dict(reserved=1), "RS_EINVAL"),
    (dict(d_k=96), "RS_EUNSUPPORTED"),
    (dict(ckpt_dtype=2), "RS_EUNSUPPORTED"),
    (dict(in_dtype=1, ring_dtype=1), "RS_EUNSUPPORTED"),
    (dict(ring_dtype=0), "RS_EUNSUPPORTED"),          # Mamba-2 ring must equal the input type
    (dict(slot_idx=None), "RS_EINVAL"),
    (dict(ring_a=None), "RS_EINVAL"),
    (dict(write_pos=None), "RS_EINVAL"),
    (dict(stride_k_row=100), "RS_EINVAL"),             # shorter than a row
    (dict(stride_v_row=2 * 64 + 4), "RS_EALIGN"),      # 8-byte multiple only
    (dict(ckpt=0x9008), "RS_EALIGN"),
    (dict(v=0x4002), "RS_EALIGN"),
    (dict(ring_k=0xB004), "RS_EALIGN"),
    (dict(out=0xD002), "RS_EALIGN"),
])
def test_mamba2_validation(lib, change, want):
    st = lib.raw_call("replayssm_decode_mamba2", _args(lib, **change), None)
    assert st == getattr(lib, want), lib.status_string(st)


def test_gdn_and_conventional_validation(lib):
    # GDN needs beta and an fp16/fp32 ring
    assert lib.raw_call("replayssm_decode_gdn", _args(lib, beta=None, ring_dtype=lib.RS_F16), None) == lib.RS_EINVAL
    assert lib.raw_call("replayssm_decode_gdn", _args(lib, ring_dtype=lib.RS_BF16), None) == lib.RS_EUNSUPPORTED
    # conventional ignores rings and cursors but checks the variant
    a = _args(lib, ring_v=None, ring_k=None, ring_a=None, write_pos=None, is_flush=None, L=0, out=0xD001)
    assert lib.raw_call("conventional_decode", a, 0, None) == lib.RS_EALIGN
    assert lib.raw_call("conventional_decode", a, 5, None) == lib.RS_EINVAL
    assert lib.raw_call("conventional_decode", _args(lib, beta=None, L=0, out=0xD001), 1, None) == lib.RS_EINVAL


def test_empty_batch_is_a_no_op(lib):
    # B = 0 with every pointer null: accepted without touching the device
    a = _args(lib, B=0, slot_idx=None, write_pos=None, is_flush=None, v=None, k=None, q=None, alpha=None,
              beta=None, ckpt=None, ring_v=None, ring_k=None, ring_a=None, out=None)
    assert lib.raw_call("replayssm_decode_mamba2", a, None) == lib.RS_OK
    assert lib.raw_call("replayssm_decode_gdn", _args(lib, B=0, ring_dtype=lib.RS_F16), None) == lib.RS_OK
    assert lib.raw_call("conventional_decode", a, 0, None) == lib.RS_OK


def test_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    z = torch.zeros(1, 2, 64)
    with pytest.raises(ValueError, match="CUDA"):
        lib.replayssm_decode_mamba2(ckpt=torch.zeros(1, 2, 64, 128), ring_v=z, ring_k=z, ring_a=z,
                                    slot_idx=torch.zeros(1, dtype=torch.int32), write_pos=z, is_flush=z,
                                    v=z, k=z, q=z, alpha=z, out=z)


# --------------------------------------------------------------------------
# align-mode plan and materialisation (host side)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L, block", [(16, 0), (16, 40), (16, 64), (8, 5), (4, 1), (64, 100)])
def test_plan_align_matches_oracle(lib, L, block):
    r = np.random.default_rng(L * 1000 + block)
    start = r.integers(0, 300, 500)
    pos = start + r.integers(0, 400, 500)
    wp, fl = lib.replayssm_plan_align(pos, start, L, block)
    wp_o, fl_o = oracle.plan_align(pos, start, L, block)
    np.testing.assert_array_equal(wp, wp_o)
    np.testing.assert_array_equal(fl, fl_o)


def test_plan_align_rejects_bad_input(lib):
    so = lib.load()
    pos = np.array([5, 6, 7], dtype=np.int64)
    st = np.array([0, 7, 0], dtype=np.int64)  # row 1 starts after its position
    wp = np.full(3, -9, dtype=np.int32)
    fl = np.full(3, 9, dtype=np.uint8)
    assert so.replayssm_plan_align(pos.ctypes.data, st.ctypes.data, 8, 3, 16, wp.ctypes.data, fl.ctypes.data) \
        == lib.RS_EINVAL
    assert np.all(wp == -9) and np.all(fl == 9)  # outputs untouched
    st[1] = 0
    assert so.replayssm_plan_align(pos.ctypes.data, st.ctypes.data, -1, 3, 16, wp.ctypes.data, fl.ctypes.data) \
        == lib.RS_EINVAL
    assert so.replayssm_plan_align(pos.ctypes.data, st.ctypes.data, 8, 3, 65, wp.ctypes.data, fl.ctypes.data) \
        == lib.RS_EINVAL
    assert so.replayssm_plan_align(None, st.ctypes.data, 8, 3, 16, wp.ctypes.data, fl.ctypes.data) == lib.RS_EINVAL
    assert so.replayssm_plan_align(None, None, 8, 0, 16, None, None) == lib.RS_OK


def _mat_args(lib, **kw):
    a = lib.MaterializeArgs()
    base = dict(B=4, H=2, d_v=64, d_k=128, L=16, num_slots=8, num_dst=8, ckpt_dtype=lib.RS_F32,
                ring_dtype=lib.RS_BF16, reserved=0, slot_idx=0x1000, held=0x2000, dst_idx=0x3000,
                ckpt=0x9000, ring_v=0xA000, ring_k=0xB000, ring_a=0xC000, dst=0xD000, dev_err=None)
    base.update(kw)
    for k_, v_ in base.items():
        setattr(a, k_, v_)
    return a


@pytest.mark.parametrize("change, variant, want", [
    (dict(), 7, "RS_EINVAL"),
    (dict(L=1), 0, "RS_EINVAL"),
    (dict(num_dst=0), 0, "RS_EINVAL"),
    (dict(reserved=3), 1, "RS_EINVAL"),
    (dict(ckpt_dtype=2), 0, "RS_EUNSUPPORTED"),
    (dict(ring_dtype=5), 0, "RS_EUNSUPPORTED"),
    (dict(d_v=32), 0, "RS_EUNSUPPORTED"),
    (dict(held=None), 0, "RS_EINVAL"),
    (dict(dst=None), 1, "RS_EINVAL"),
    (dict(dst=0xD008), 0, "RS_EALIGN"),
    (dict(ring_v=0xA004), 1, "RS_EALIGN"),
    (dict(dst_idx=0x3002), 0, "RS_EALIGN"),
])
def test_materialize_validation(lib, change, variant, want):
    st = lib.raw_call("replayssm_materialize", _mat_args(lib, **change), variant, None)
    assert st == getattr(lib, want), lib.status_string(st)


def test_materialize_empty_batch_is_a_no_op(lib):
    a = _mat_args(lib, B=0, slot_idx=None, held=None, dst_idx=None, ckpt=None, ring_v=None, ring_k=None,
                  ring_a=None, dst=None)
    assert lib.raw_call("replayssm_materialize", a, 0, None) == lib.RS_OK


@pytest.mark.parametrize("change, entry, want", [
    (dict(ckpt_lp=0xE000, lp_dtype=1), "replayssm_decode_gdn", "RS_EUNSUPPORTED"),      # Mamba-2 only
    (dict(ckpt_lp=0xE000, lp_dtype=1, ckpt_dtype=1), "replayssm_decode_mamba2", "RS_EUNSUPPORTED"),
    (dict(ckpt_lp=0xE000, lp_dtype=0), "replayssm_decode_mamba2", "RS_EUNSUPPORTED"),  # 16-bit read copy
    (dict(ckpt_lp=0xE008, lp_dtype=2), "replayssm_decode_mamba2", "RS_EALIGN"),
    (dict(reserved2=1), "replayssm_decode_mamba2", "RS_EINVAL"),
])
def test_two_precision_validation(lib, change, entry, want):
    kw = dict(change)
    if entry == "replayssm_decode_gdn":
        kw["ring_dtype"] = lib.RS_F16
    st = lib.raw_call(entry, _args(lib, **kw), None)
    assert st == getattr(lib, want), lib.status_string(st)
    a = _args(lib, ckpt_lp=0xE000, lp_dtype=1, ring_v=None, ring_k=None, ring_a=None, write_pos=None,
              is_flush=None, L=0)
    assert lib.raw_call("conventional_decode", a, 0, None) == lib.RS_EUNSUPPORTED


# --------------------------------------------------------------------------
# speculative verification (host side)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L, T", [(16, 4), (16, 8), (8, 8), (64, 16), (4, 1)])
def test_plan_spec_matches_oracle(lib, L, T):
    h = np.random.default_rng(L + T).integers(0, L + 1, 300).astype(np.int32)
    np.testing.assert_array_equal(lib.replayssm_plan_spec(h, L, T), oracle.spec.spec_plan(h, L, T))


def test_plan_spec_rejects_bad_input(lib):
    so = lib.load()
    h = np.array([0, 17], dtype=np.int32)
    fl = np.full(2, 9, dtype=np.uint8)
    assert so.replayssm_plan_spec(h.ctypes.data, 2, 16, 4, fl.ctypes.data) == lib.RS_EINVAL  # h > L
    assert np.all(fl == 9)
    h[1] = 3
    assert so.replayssm_plan_spec(h.ctypes.data, 2, 16, 17, fl.ctypes.data) == lib.RS_EINVAL  # T > 16
    assert so.replayssm_plan_spec(h.ctypes.data, 2, 4, 5, fl.ctypes.data) == lib.RS_EINVAL   # T > L
    assert so.replayssm_plan_spec(h.ctypes.data, 2, 16, 4, fl.ctypes.data) == lib.RS_OK
    assert list(fl) == [0, 0]
    assert so.replayssm_spec_commit(None, None, None, 0, 16, 4, None, None, None, None) == lib.RS_OK
    assert so.replayssm_spec_commit(None, None, None, 3, 16, 4, None, None, None, None) == lib.RS_EINVAL


def _spec_args(lib, **kw):
    a = lib.SpecArgs()
    base = dict(B=4, H=2, d_v=64, d_k=128, L=16, T=4, num_slots=8, ckpt_dtype=lib.RS_F32, in_dtype=lib.RS_BF16,
                reserved=0, slot_idx=0x1000, committed=0x2000, is_flush=0x3000, v=0x4000, k=0x5000, q=0x6000,
                alpha=0x7000, ckpt=0x9000, ring_v=0xA000, ring_k=0xB000, ring_a=0xC000, out=0xD000, dev_err=None)
    base.update(kw)
    for k_, v_ in base.items():
        setattr(a, k_, v_)
    return a


@pytest.mark.parametrize("change, want", [
    (dict(T=0), "RS_EINVAL"),
    (dict(T=17, L=32), "RS_EINVAL"),
    (dict(T=5, L=4), "RS_EINVAL"),
    (dict(reserved=2), "RS_EINVAL"),
    (dict(ckpt_dtype=2), "RS_EUNSUPPORTED"),
    (dict(d_v=32), "RS_EUNSUPPORTED"),
    (dict(committed=None), "RS_EINVAL"),
    (dict(q=0x6008), "RS_EALIGN"),
    (dict(committed=0x2002), "RS_EALIGN"),
])
def test_spec_verify_validation(lib, change, want):
    st = lib.raw_call("replayssm_spec_verify_mamba2", _spec_args(lib, **change), None)
    assert st == getattr(lib, want), lib.status_string(st)


@pytest.mark.parametrize("change, entry, want", [
    (dict(n_groups=3, H=4, kq_scratch=0xF000), "replayssm_decode_mamba2", "RS_EINVAL"),     # must divide H
    (dict(n_groups=2, H=4, kq_scratch=None), "replayssm_decode_mamba2", "RS_EINVAL"),       # scratch needed
    (dict(n_groups=2, H=4, kq_scratch=0xF002), "replayssm_decode_mamba2", "RS_EALIGN"),
    (dict(n_groups=2, H=4, kq_scratch=0xF000, ckpt_lp=0xE000, lp_dtype=1), "replayssm_decode_mamba2",
     "RS_EUNSUPPORTED"),
    (dict(n_groups=2, H=4, kq_scratch=0xF000, ring_dtype=1), "replayssm_decode_gdn", "RS_EUNSUPPORTED"),
    (dict(n_groups=-1), "replayssm_decode_mamba2", "RS_EINVAL"),
    (dict(reserved3=1), "replayssm_decode_mamba2", "RS_EINVAL"),
    (dict(n_groups=2, H=4, kq_scratch=0xF000, stride_k_row=128), "replayssm_decode_mamba2", "RS_EINVAL"),
])
def test_grouped_key_validation(lib, change, entry, want):
    kw = dict(stride_v_row=4 * 64, stride_k_row=4 * 128, stride_q_row=4 * 128, stride_out_row=4 * 64)
    kw.update(change)
    st = lib.raw_call(entry, _args(lib, **kw), None)
    assert st == getattr(lib, want), lib.status_string(st)
    # with 2 groups of 2 heads the key rows may be as short as G * d_k
    ok = _args(lib, H=4, n_groups=2, kq_scratch=0xF000, stride_v_row=4 * 64, stride_k_row=2 * 128,
               stride_q_row=2 * 128, stride_out_row=4 * 64)
    assert lib.raw_call("conventional_decode", ok, 0, None) == lib.RS_EUNSUPPORTED
