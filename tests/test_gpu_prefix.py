"""Prefix caching on the GPU against the oracle: align-mode decode (forced
flush on the token that completes a cache block, ring re-anchored at each
block start) and state materialisation (checkpoint unrolled with the held
records, written to a separate pool or folded in place).

Gates as in test_gpu_parity: fp32 checkpoints against the exact recurrence
at max relative error 1e-4 (GDN with an fp32 ring, so the comparison is with
the exact delta rule); fp16 destinations against the oracle's unroll rounded
once to fp16, 2e-3 (one fp16 rounding of values that differ in the last fp32
bits can land one ulp apart: 2^-11 relative).  Cursors and flags bit-exact;
materialisation must leave the checkpoint and the rings bit-identical.
"""

import numpy as np
import pytest

import oracle
from linear_attention_decode_replayssm_gb300 import synth
from tests._harness import GpuRun, OracleRun, dev, tdt
from tests._util import rel_err

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_F16_DST = 2e-3


@pytest.fixture(scope="module")
def cuda(lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def _workload(variant, B, H, steps, seed, **kw):
    if variant == "mamba2":
        return synth.make_workload("mamba2_bs256", B=B, H=H, steps=steps, seed=seed, **kw)
    return synth.make_workload("gdn_bs256", B=B, H=H, steps=steps, seed=seed, ring_dtype="f32", **kw)


def _same_bits(a, b):
    import torch

    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def _materialize(lib, g, w, held, dst, dst_idx, dev_err=None):
    import torch

    lib.replayssm_materialize(variant=lib.RS_GDN if w.variant == "gdn" else lib.RS_MAMBA2, ckpt=g.ckpt,
                              ring_v=g.ring_v, ring_k=g.ring_k, ring_a=g.ring_a, slot_idx=g.slot_idx,
                              held=torch.as_tensor(np.asarray(held, dtype=np.int32), device="cuda"),
                              dst=dst, dst_idx=torch.as_tensor(np.asarray(dst_idx, dtype=np.int32), device="cuda"),
                              dev_err=g.dev_err if dev_err is None else dev_err)


@pytest.mark.parametrize("variant", ["mamba2", "gdn"])
@pytest.mark.parametrize("L, block", [(16, 40), (8, 12), (16, 64)])
def test_align_mode_decode_and_materialize(cuda, variant, L, block):
    """Rows start decoding at random positions with empty rings; every step's
    plan comes from the align-mode host plan.  Outputs track the exact
    recurrence; at every block end the checkpoint itself is the exact state;
    every 5 steps all rows are materialised into a separate pool (rows in a
    shuffled order) and match the exact state, with checkpoint and rings
    untouched."""
    import torch

    lib = cuda
    B, H, steps = 10, 4, 3 * max(block, L) + 9
    w = _workload(variant, B, H, steps, seed=L + block, L=L, cursor0=np.zeros(B, dtype=np.int64),
                  pad_rows=1, num_slots=13, permute_slots=True)
    r = np.random.default_rng(block)
    start = r.integers(0, 3 * block, B)
    g, o = GpuRun(lib, w), OracleRun(w, replay=False)
    live = w.slot_idx >= 0
    dst = torch.full((B + 3, H, w.d_v, w.d_k), 7.0, device="cuda", dtype=tdt(w.ckpt_dtype))
    worst_o = worst_b = worst_m = 0.0
    n_boundary = n_mat = 0
    for t in range(steps):
        pos = start + t
        wp, fl = lib.replayssm_plan_align(pos, start, L, block)
        wp_o, fl_o = oracle.plan_align(pos, start, L, block)
        np.testing.assert_array_equal(wp, wp_o)
        np.testing.assert_array_equal(fl, fl_o)
        x = w.inputs(t)
        out, _, _ = g.step(x, None, plan=(wp, fl))
        _, o_e = o.step(x, wp, fl)
        worst_o = max(worst_o, rel_err(out[live], o_e[live]))
        done = live & ((pos + 1) % block == 0)
        if done.any():
            assert np.all(fl[done] == 1)
            n_boundary += int(done.sum())
            slots = w.slot_idx[done]
            ck = g.ckpt[torch.as_tensor(slots, device="cuda")].double().cpu().numpy()
            worst_b = max(worst_b, rel_err(ck, o.ex.S[slots], nd=2))
        if t % 5 == 4:
            held = np.where(fl != 0, 0, wp + 1)
            dst_idx = r.permutation(B + 3)[:B]
            dst.fill_(7.0)
            snap = [x_.clone() for x_ in (g.ckpt, g.ring_v, g.ring_k, g.ring_a)]
            _materialize(lib, g, w, held, dst, dst_idx)
            for a_, b_ in zip(snap, (g.ckpt, g.ring_v, g.ring_k, g.ring_a)):
                assert _same_bits(a_, b_)
            got = dst[torch.as_tensor(dst_idx[live], device="cuda")].double().cpu().numpy()
            worst_m = max(worst_m, rel_err(got, o.ex.S[w.slot_idx[live]], nd=2))
            n_mat += 1
            # the padded row and the unused destination slots hold the fill
            untouched = np.setdiff1d(np.arange(B + 3), dst_idx[live])
            assert bool((dst[torch.as_tensor(untouched, device="cuda")] == 7.0).all())
    assert n_boundary >= 2 * (B - 1) and n_mat >= 5
    assert int(g.dev_err.item()) == 0
    assert worst_o <= TOL_F32 and worst_b <= TOL_F32 and worst_m <= TOL_F32, (worst_o, worst_b, worst_m)


@pytest.mark.parametrize("variant", ["mamba2", "gdn"])
def test_materialize_in_place_then_continue(cuda, variant):
    """Fold the held records into the checkpoint in place (dst = ckpt,
    dst_idx = slot_idx), restart each row's cursor at 0, and keep decoding:
    outputs and flushed checkpoints still match the exact recurrence."""
    import torch

    lib = cuda
    B, H, L, steps = 8, 4, 16, 70
    w = _workload(variant, B, H, steps, seed=3)
    g, o = GpuRun(lib, w), OracleRun(w, replay=False)
    ds = w.decode_step0.copy()
    worst = 0.0
    for t in range(steps):
        if t in (9, 37):
            held = (ds % L).astype(np.int32)
            _materialize(lib, g, w, held, g.ckpt, w.slot_idx)
            got = g.ckpt[torch.as_tensor(w.slot_idx, device="cuda")].double().cpu().numpy()
            worst = max(worst, rel_err(got, o.ex.S[w.slot_idx], nd=2))
            ds = np.zeros(B, dtype=np.int64)  # re-anchored: the ring is logically empty
        x = w.inputs(t)
        out, wp, fl = g.step(x, ds)
        _, o_e = o.step(x, wp, fl)
        worst = max(worst, rel_err(out, o_e))
        ds += 1
    assert int(g.dev_err.item()) == 0
    assert worst <= TOL_F32, worst


@pytest.mark.parametrize("variant, ring", [("mamba2", "bf16"), ("gdn", "f16")])
def test_materialize_fp16_checkpoint(cuda, variant, ring):
    """fp16 checkpoint pool and destination: the unroll rounded once to fp16."""
    import torch

    lib = cuda
    B, H = 12, 4
    w = synth.make_workload("mamba2_bs256" if variant == "mamba2" else "gdn_bs256", B=B, H=H, steps=1, seed=5,
                            ckpt_dtype="f16", ring_dtype=ring)
    g = GpuRun(lib, w)
    held = (w.decode_step0 % w.L).astype(np.int32)
    dst = torch.zeros(B, H, w.d_v, w.d_k, device="cuda", dtype=torch.float16)
    _materialize(lib, g, w, held, dst, np.arange(B))
    rs = oracle.ReplayState(w.variant, w.ckpt0.astype(np.float64), w.ring_v0.astype(np.float64),
                            w.ring_k0.astype(np.float64), w.ring_a0.astype(np.float64))
    want = oracle.materialize(rs, w.slot_idx, held, "f16")
    assert int(g.dev_err.item()) == 0
    assert rel_err(dst.double().cpu().numpy(), want, nd=2) <= TOL_F16_DST


@pytest.mark.parametrize("variant, ring, ckpt", [("mamba2", "bf16", "f32"), ("mamba2", "f32", "f32"),
                                                  ("mamba2", "bf16", "f16"), ("gdn", "f16", "f32"),
                                                  ("gdn", "f32", "f32"), ("gdn", "f16", "f16")])
def test_materialize_many_units(cuda, variant, ring, ckpt):
    """More units than the launch has CTAs (each CTA takes several, its two
    consumer groups alternating over the slot rings, a unit count that is
    not a multiple of the groups or the grid), every held count from 0 to
    L - 1, padded rows and a permuted destination: every element against
    the oracle."""
    import torch

    lib = cuda
    B, H = 97, 8
    name = "mamba2_bs256" if variant == "mamba2" else "gdn_bs256"
    kw = dict(in_dtype=ring) if variant == "mamba2" else {}  # Mamba-2 records are its inputs verbatim
    held = (np.arange(B) % synth.SPECS[name]["L"]).astype(np.int32)
    w = synth.make_workload(name, B=B, H=H, steps=1, seed=31, ckpt_dtype=ckpt, ring_dtype=ring, cursor0=held, **kw)
    g = GpuRun(lib, w)
    dst_idx = np.random.default_rng(6).permutation(B + 5)[:B].astype(np.int32)
    dst_idx[[3, 50]] = -1  # skipped rows
    dst = torch.full((B + 5, H, w.d_v, w.d_k), 5.0, device="cuda", dtype=tdt(ckpt))
    before = [x.clone() for x in (g.ckpt, g.ring_v, g.ring_k, g.ring_a)]
    _materialize(lib, g, w, held, dst, dst_idx)
    assert int(g.dev_err.item()) == 0
    for a_, b_ in zip(before, (g.ckpt, g.ring_v, g.ring_k, g.ring_a)):
        assert _same_bits(a_, b_)
    rs = oracle.ReplayState(w.variant, w.ckpt0.astype(np.float64), w.ring_v0.astype(np.float64),
                            w.ring_k0.astype(np.float64), w.ring_a0.astype(np.float64))
    want = oracle.materialize(rs, w.slot_idx, held, ckpt)
    rows = np.flatnonzero(dst_idx >= 0)
    got = dst[torch.as_tensor(dst_idx[rows].astype(np.int64), device="cuda")].double().cpu().numpy()
    assert rel_err(got, want[rows], nd=2) <= (TOL_F16_DST if ckpt == "f16" else TOL_F32)
    untouched = np.setdiff1d(np.arange(B + 5), dst_idx[rows])
    assert bool((dst[torch.as_tensor(untouched, device="cuda")] == 5.0).all())


def test_materialize_range_checks(cuda):
    """Out-of-range slot, destination or held count: the row is skipped, the
    matching bit is set, and nothing is written."""
    import torch

    lib = cuda
    B, H = 4, 2
    w = _workload("mamba2", B, H, 1, seed=8)
    g = GpuRun(lib, w)
    dst = torch.full((B, H, w.d_v, w.d_k), 3.0, device="cuda")
    for held, dst_idx, slot, bit in (([0, 1, 16, 2], [0, 1, 2, 3], None, lib.RS_DERR_WRITE_POS),
                                     ([0, 1, 2, 3], [0, 1, 9, 3], None, lib.RS_DERR_DST),
                                     ([0, 1, 2, 3], [0, 1, 2, 3], [0, 1, 40, 3], lib.RS_DERR_SLOT)):
        if slot is not None:
            g.slot_idx.copy_(torch.as_tensor(np.array(slot, dtype=np.int32)))
        err = torch.zeros(1, device="cuda", dtype=torch.int32)
        dst.fill_(3.0)
        _materialize(lib, g, w, held, dst, dst_idx, dev_err=err)
        assert int(err.item()) == bit
        assert bool((dst[2] == 3.0).all())      # the bad row (index 2) wrote nothing
        assert not bool((dst[0] == 3.0).all())  # the good rows did
        g.slot_idx.copy_(torch.as_tensor(w.slot_idx))


def test_materialize_full_size_sampled(cuda):
    """Batch 256 x 128 heads of 64 x 128, fp32, L 16, staggered cursors (the
    decode bench's layer): every row materialised at once, 4 heads of every
    row checked against the oracle."""
    import torch

    lib = cuda
    B, H, dv, dk, L = 256, 128, 64, 128, 16
    heads = np.array([0, 33, 90, 127])
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    ckpt = synth.device_draw((B, H, dv, dk), "scaled", gen, d_k=dk)
    ring_v = synth.device_draw((B, H, L, dv), "scaled", gen, d_k=dk).to(torch.bfloat16)
    ring_k = synth.device_draw((B, H, L, dk), "scaled", gen, d_k=dk).to(torch.bfloat16)
    ring_a = synth.device_draw((B, H, L), "sigmoid3", gen)
    held = np.random.default_rng(4).integers(0, L, B).astype(np.int32)
    held[:2] = (0, L - 1)
    dst = torch.empty_like(ckpt)
    slot_idx = torch.arange(B, device="cuda", dtype=torch.int32)
    dst_idx = torch.flip(slot_idx, (0,)).contiguous()
    err = torch.zeros(1, device="cuda", dtype=torch.int32)
    lib.replayssm_materialize(variant=lib.RS_MAMBA2, ckpt=ckpt, ring_v=ring_v, ring_k=ring_k, ring_a=ring_a,
                              slot_idx=slot_idx, held=torch.as_tensor(held, device="cuda"), dst=dst,
                              dst_idx=dst_idx, dev_err=err)
    hs = torch.as_tensor(heads, device="cuda")
    sub = lambda x: x[:, hs].double().cpu().numpy()
    rs = oracle.ReplayState("mamba2", sub(ckpt), sub(ring_v), sub(ring_k), sub(ring_a))
    want = oracle.materialize(rs, np.arange(B), held)
    got = dst.flip(0)[:, hs].double().cpu().numpy()
    assert int(err.item()) == 0
    assert rel_err(got, want, nd=2) <= TOL_F32
