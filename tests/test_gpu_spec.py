"""Speculative verification (Mamba-2) on the GPU against the oracle.

Each step verifies T drafts per row through the C ABI, draws how many drafts
the row accepts, and commits them with the device-side commit kernel; the
next step's flags come from that kernel, as they would inside one captured
graph.  The exact result is the recurrence over the committed tokens followed
by the drafts (rejected drafts leave no trace), kept here in float64.

Gates: outputs and flushed fp32 checkpoints at max relative error 1e-4
against that exact result (the rings hold the inputs verbatim, so only fp32
arithmetic order differs); committed counts and flags bit-exact against the
oracle's commit rule; the ring records written bit-exact against the inputs.
"""

import numpy as np
import pytest

import oracle
from oracle import spec
from linear_attention_decode_replayssm_gb300 import synth
from tests._harness import dev, tdt
from tests._util import rel_err

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def cuda(lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def _drafts(w, t, T):
    """Seeded draft inputs of step t: v [B,T,H,d_v], k, q [B,T,H,d_k] (bf16
    values), alpha [B,T,H] fp32, with the workload's laws."""
    r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 90_000 + t])))
    B, H, sk = w.B, w.H, np.sqrt(np.float32(w.d_k))
    v = r.standard_normal((B, T, H, w.d_v), dtype=np.float32) / sk
    k = r.standard_normal((B, T, H, w.d_k), dtype=np.float32) / sk
    q = r.standard_normal((B, T, H, w.d_k), dtype=np.float32) / sk
    a = (1.0 / (1.0 + np.exp(-r.normal(w.alpha_mu, w.alpha_sd, (B, T, H))))).astype(np.float32)
    q_ = lambda x: synth.quantize(x, w.in_dtype)
    return q_(v), q_(k), q_(q), a


def _run(lib, w, T, steps, heads=None, seed=0):
    import torch

    L, B = w.L, w.B
    hs = np.arange(w.H) if heads is None else np.asarray(heads)
    hs_t = torch.as_tensor(hs, device="cuda")
    ckpt = dev(w.ckpt0, tdt(w.ckpt_dtype))
    ring_v, ring_k = dev(w.ring_v0, tdt(w.ring_dtype)), dev(w.ring_k0, tdt(w.ring_dtype))
    ring_a = dev(w.ring_a0, torch.float32)
    slot_idx = dev(w.slot_idx, torch.int32)
    out = torch.empty(B, T, w.H, w.d_v, device="cuda")
    dev_err = torch.zeros(1, device="cuda", dtype=torch.int32)
    live = w.slot_idx >= 0
    # committed counts start at the records the workload placed in each ring
    h = (w.decode_step0 % L).astype(np.int32)
    fl = lib.replayssm_plan_spec(h, L, T)
    np.testing.assert_array_equal(fl, spec.spec_plan(h, L, T))
    h_d, fl_d = dev(h, torch.int32), dev(fl, torch.uint8)
    # exact committed state per slot (sampled heads), float64
    rs0 = oracle.ReplayState("mamba2", w.ckpt0[:, hs].astype(np.float64), w.ring_v0[:, hs].astype(np.float64),
                             w.ring_k0[:, hs].astype(np.float64), w.ring_a0[:, hs].astype(np.float64))
    exact = oracle.ExactState.from_replay(rs0, w.held_records()).S
    r = np.random.default_rng(seed)
    worst_o = worst_c = 0.0
    n_flush = 0
    for t in range(steps):
        v, k, q, a = _drafts(w, t, T)
        td = tdt(w.in_dtype)
        lib.replayssm_spec_verify_mamba2(ckpt=ckpt, ring_v=ring_v, ring_k=ring_k, ring_a=ring_a, slot_idx=slot_idx,
                                         committed=h_d, is_flush=fl_d, v=dev(v, td), k=dev(k, td), q=dev(q, td),
                                         alpha=dev(a, torch.float32), out=out, dev_err=dev_err)
        o_g = out[:, :, hs_t].double().cpu().numpy()
        acc = r.integers(1, T + 1, B).astype(np.int32)
        for b in np.nonzero(live)[0]:
            s = w.slot_idx[b]
            if fl[b]:
                n_flush += 1
                ck = ckpt[s][hs_t].double().cpu().numpy()
                worst_c = max(worst_c, rel_err(ck, exact[s], nd=2))
            # the drafts' records sit at slots nb .. nb+T-1
            nb = 0 if fl[b] else h[b]
            got_k = ring_k[s][hs_t][:, nb:nb + T].float().cpu().numpy()
            np.testing.assert_array_equal(got_k, np.moveaxis(k[b][:, hs], 0, 1))
            S = exact[s].copy()
            for i in range(T):
                S, o_i = oracle.mamba2_step(S, a[b, i, hs], v[b, i, hs], k[b, i, hs], q[b, i, hs])
                worst_o = max(worst_o, rel_err(o_g[b, i], o_i))
                if i + 1 == acc[b]:
                    exact[s] = S.copy()
        assert np.all(o_g[~live] == 0)
        # commit on the device; the next flags come from the kernel
        lib.replayssm_spec_commit(committed=h_d, is_flush=fl_d, accepted=dev(acc, torch.int32), L=L, T=T,
                                  dev_err=dev_err)
        h, fl = spec.spec_commit(h, fl, acc, L, T)
        np.testing.assert_array_equal(h_d.cpu().numpy(), h)
        np.testing.assert_array_equal(fl_d.cpu().numpy(), fl)
    return int(dev_err.item()), worst_o, worst_c, n_flush


@pytest.mark.parametrize("T", [1, 4, 8])
def test_spec_verify_small(cuda, T):
    w = synth.make_workload("mamba2_bs256", B=6, H=3, steps=1, seed=30 + T, pad_rows=1, num_slots=9,
                            permute_slots=True)
    err, worst_o, worst_c, n_flush = _run(cuda, w, T, 40, seed=T)
    assert err == 0 and n_flush > 0
    assert worst_o <= TOL and worst_c <= TOL, (worst_o, worst_c)


@pytest.mark.parametrize("L, T", [(4, 4), (32, 16), (64, 8)])
def test_spec_verify_window_lengths(cuda, L, T):
    w = synth.make_workload("mamba2_bs256", B=4, H=2, steps=1, seed=L + T, L=L)
    err, worst_o, worst_c, n_flush = _run(cuda, w, T, max(24, 3 * L // T), seed=L)
    assert err == 0 and n_flush > 0
    assert worst_o <= TOL and worst_c <= TOL, (worst_o, worst_c)


def test_spec_verify_bs256_full_size_sampled(cuda):
    """Batch 256, 128 heads of 64 x 128, fp32, L 16, T 4: two heads of every
    row followed by the exact recurrence for 20 steps."""
    w = synth.make_workload("mamba2_bs256", steps=1, seed=4)
    err, worst_o, worst_c, n_flush = _run(cuda, w, 4, 20, heads=[7, 99], seed=4)
    assert err == 0 and n_flush > 100
    assert worst_o <= TOL and worst_c <= TOL, (worst_o, worst_c)


def test_spec_range_checks(cuda):
    """A committed count past the window without a flush, or an accepted count
    outside [1, T], is reported and never written past the ring."""
    import torch

    lib = cuda
    w = synth.make_workload("mamba2_bs256", B=3, H=2, steps=1, seed=6)
    T, L = 4, w.L
    ckpt = dev(w.ckpt0, torch.float32)
    ring_v, ring_k = dev(w.ring_v0, torch.bfloat16), dev(w.ring_k0, torch.bfloat16)
    ring_a = dev(w.ring_a0, torch.float32)
    snap = [x.clone() for x in (ckpt, ring_v, ring_k, ring_a)]
    v, k, q, a = _drafts(w, 0, T)
    out = torch.full((3, T, 2, 64), 5.0, device="cuda")
    err = torch.zeros(1, device="cuda", dtype=torch.int32)
    lib.replayssm_spec_verify_mamba2(ckpt=ckpt, ring_v=ring_v, ring_k=ring_k, ring_a=ring_a,
                                     slot_idx=dev(np.array([0, 1, 2]), torch.int32),
                                     committed=dev(np.array([L - 1, L + 1, L - T]), torch.int32),
                                     is_flush=dev(np.array([0, 1, 0]), torch.uint8),
                                     v=dev(v, torch.bfloat16), k=dev(k, torch.bfloat16), q=dev(q, torch.bfloat16),
                                     alpha=dev(a, torch.float32), out=out, dev_err=err)
    assert int(err.item()) == lib.RS_DERR_WRITE_POS
    assert bool((out[:2] == 0).all())             # rows 0 and 1 skipped
    for s in (0, 1):                              # and their state untouched
        for x, y in zip(snap, (ckpt, ring_v, ring_k, ring_a)):
            assert torch.equal(x[s].view(torch.uint8), y[s].view(torch.uint8))
    h_d = dev(np.array([3, 5, 0]), torch.int32)
    fl_d = dev(np.array([0, 1, 0]), torch.uint8)
    err.zero_()
    lib.replayssm_spec_commit(committed=h_d, is_flush=fl_d, accepted=dev(np.array([2, 0, 9]), torch.int32), L=L,
                              T=T, dev_err=err)
    assert int(err.item()) == lib.RS_DERR_ACCEPTED
    assert h_d.cpu().tolist() == [5, 0, 0]


def test_spec_verify_fp16_checkpoint(cuda):
    """fp16 checkpoint, T = 4: against the oracle's verification with the same
    storage rounding (the folded checkpoint rounded to fp16 at each flush),
    max relative error 2e-3 (one fp16 rounding of the checkpoint, where the
    fp32 and float64 folds may round a midpoint apart), and against the exact
    recurrence 2e-2 (the fp16 checkpoint gate)."""
    import torch

    lib = cuda
    T, steps = 4, 40
    w = synth.make_workload("mamba2_bs256", B=6, H=3, steps=1, seed=61, ckpt_dtype="f16")
    L, B, td = w.L, w.B, tdt(w.in_dtype)
    ckpt = dev(w.ckpt0, torch.float16)
    ring_v, ring_k = dev(w.ring_v0, td), dev(w.ring_k0, td)
    ring_a = dev(w.ring_a0, torch.float32)
    slot_idx = dev(w.slot_idx, torch.int32)
    out = torch.empty(B, T, w.H, w.d_v, device="cuda")
    err = torch.zeros(1, device="cuda", dtype=torch.int32)
    h = (w.decode_step0 % L).astype(np.int32)
    fl = spec.spec_plan(h, L, T)
    h_d, fl_d = dev(h, torch.int32), dev(fl, torch.uint8)
    rs = oracle.ReplayState("mamba2", w.ckpt0.astype(np.float64), w.ring_v0.astype(np.float64),
                            w.ring_k0.astype(np.float64), w.ring_a0.astype(np.float64), ckpt_dtype="f16")
    exact = oracle.ExactState.from_replay(rs, w.held_records()).S
    r = np.random.default_rng(61)
    worst_emu = worst_exact = 0.0
    for t in range(steps):
        v, k, q, a = _drafts(w, t, T)
        lib.replayssm_spec_verify_mamba2(ckpt=ckpt, ring_v=ring_v, ring_k=ring_k, ring_a=ring_a, slot_idx=slot_idx,
                                         committed=h_d, is_flush=fl_d, v=dev(v, td), k=dev(k, td), q=dev(q, td),
                                         alpha=dev(a, torch.float32), out=out, dev_err=err)
        o_g = out.double().cpu().numpy()
        o_emu = spec.spec_verify_step(rs, w.slot_idx, h, fl, v, k, q, a)
        worst_emu = max(worst_emu, rel_err(o_g, o_emu))
        acc = r.integers(1, T + 1, B).astype(np.int32)
        for b in range(B):
            S = exact[w.slot_idx[b]].copy()
            for i in range(T):
                S, o_i = oracle.mamba2_step(S, a[b, i], v[b, i], k[b, i], q[b, i])
                worst_exact = max(worst_exact, rel_err(o_g[b, i], o_i))
                if i + 1 == acc[b]:
                    exact[w.slot_idx[b]] = S.copy()
        lib.replayssm_spec_commit(committed=h_d, is_flush=fl_d, accepted=dev(acc, torch.int32), L=L, T=T,
                                  dev_err=err)
        h, fl = spec.spec_commit(h, fl, acc, L, T)
    assert int(err.item()) == 0
    assert worst_emu <= 2e-3 and worst_exact <= 2e-2, (worst_emu, worst_exact)
