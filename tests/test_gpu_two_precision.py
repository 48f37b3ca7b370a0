"""Two-precision Mamba-2 checkpoint on the GPU against the oracle.

The recurrence copy is fp32, the read copy fp16 or bf16.  What the pages fix
("ReplaySSM: an SSM decoder that writes its state once every 16 tokens",
§The precision argument, derived), and what is gated here:

  * flush rows start from the recurrence copy, so every flushed fp32
    checkpoint matches the exact recurrence at max relative error 1e-4, as
    with one copy;
  * the read copy written at a flush is one round-to-nearest-even of the new
    state: every element lies within half a unit in the last place (of the
    read type) of the exact state, plus 2e-6 for the fp32 arithmetic, and at
    least 99.9 % of the elements equal the oracle's own rounding exactly (the
    rest sit on a rounding midpoint, where fp32 and fp64 may round apart);
  * a non-flush output errs by gamma_h eps_m q_t only: against the exact
    recurrence, each output element is within gamma_h * sum_j (ulp_ij / 2)
    |q_j| of the exact value (the rounding bound of the last flushed state,
    computed by the oracle from the exact state), plus 1e-4 for the fp32
    arithmetic; and the error must be visible (the read copy is really read).
  * cursors and flags bit-exact.
"""

import numpy as np
import pytest

import oracle
from linear_attention_decode_replayssm_gb300 import synth
from tests._harness import GpuRun, OracleRun, dev, tdt
from tests._util import rel_err

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
ARITH = 2e-6          # fp32 arithmetic of the fold, relative to the head's scale
MIN_EXACT = 0.999


@pytest.fixture(scope="module")
def cuda(lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def _half_ulp(x, lp):
    """Half the spacing of ``lp`` numbers in the binade of each |x| (E4M3: on
    the row's power-of-two scale, rows along the last axis)."""
    if lp == "e4m3":
        e = oracle.row_scale_exponent(x)[..., None].astype(np.float64)
        xs = np.abs(x) * 2.0 ** -e
        step = np.where(xs < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(xs, 2.0 ** -6))) - 3))
        return 0.5 * step * 2.0 ** e
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    mant, emin = {"f16": (10, -14), "bf16": (7, -126)}[lp]
    return 0.5 * 2.0 ** (np.maximum(e, emin) - mant)


def _scale(S):
    """max(|x|, rms of the head's matrix), per element."""
    rms = np.sqrt(np.mean(S * S, axis=(-2, -1), keepdims=True))
    return np.maximum(np.abs(S), rms)


def _run(lib, w, lp, steps, heads=None):
    import torch

    g = GpuRun(lib, w, lp_dtype=lp)
    o = OracleRun(w, heads=heads, replay=False, exact=True)
    hs = o.heads
    hs_t = torch.as_tensor(hs, device="cuda")
    live = w.slot_idx >= 0
    slots = w.slot_idx[live]
    # exact state at the last flush (at the start: the checkpoint itself), and
    # the decay applied since (per head)
    S_m = w.ckpt0[:, hs].astype(np.float64)
    held = w.held_records()
    gam = np.ones((w.num_slots, len(hs)))
    for s in slots:
        gam[s] = np.prod(w.ring_a0[s][hs][:, : held[s]].astype(np.float64), axis=1)
    worst_ck = worst_excess = seen = 0.0
    n_lp = n_lp_exact = 0
    for t in range(steps):
        x = w.inputs(t)
        out, wp, fl = g.step(x, w.decode_step(t))
        np.testing.assert_array_equal((wp, fl), oracle.plan_step(w.decode_step(t), w.L))
        sub = o.sub(x)
        _, o_e = o.step(x, wp, fl)
        q = sub["q"].astype(np.float64)
        a = sub["alpha"].astype(np.float64)
        o_g = out[:, hs]
        for b in np.nonzero(live)[0]:
            s = w.slot_idx[b]
            gam[s] *= a[b]
            if fl[b]:
                continue
            # the pages' bound: gamma_h * |eps_m| |q|, eps_m <= half an ulp of the flushed state
            bound = gam[s][:, None] * np.einsum("hij,hj->hi", _half_ulp(S_m[s], lp), np.abs(q[b]))
            scale = np.maximum(np.abs(o_e[b]), np.sqrt(np.mean(o_e[b] ** 2, axis=-1, keepdims=True)))
            err = np.abs(o_g[b] - o_e[b])
            worst_excess = max(worst_excess, float(np.max((err - bound) / scale)))
            seen = max(seen, float(np.max(err / scale)))
        fl_rows = np.nonzero(live & (fl != 0))[0]
        if len(fl_rows):
            fs = w.slot_idx[fl_rows]
            fs_t = torch.as_tensor(fs, device="cuda")
            hp = g.ckpt[fs_t][:, hs_t].double().cpu().numpy()
            lpv = g.read_copy(fs, hs)
            S_new = o.ex.S[fs]
            worst_ck = max(worst_ck, rel_err(hp, S_new, nd=2))
            lim = _half_ulp(S_new, lp) + ARITH * _scale(S_new)
            assert np.all(np.abs(lpv - S_new) <= lim), "read copy is not a rounding of the new state"
            n_lp += lpv.size
            n_lp_exact += int(np.sum(lpv == oracle.round_read_copy(S_new, lp)))
            for s in fs:
                S_m[s] = o.ex.S[s].copy()
                gam[s] = 1.0
    return g, dict(ck=worst_ck, excess=worst_excess, seen=seen, lp_exact=n_lp_exact / max(n_lp, 1), n_lp=n_lp)


@pytest.mark.parametrize("lp", ["f16", "bf16", "e4m3"])
def test_two_precision_small(cuda, lp):
    """Padded rows, permuted slots, staggered cursors, 48 steps (3 windows)."""
    w = synth.make_workload("mamba2_bs256", B=7, H=3, steps=48, seed=21, pad_rows=1, num_slots=11,
                            permute_slots=True)
    g, r = _run(cuda, w, lp, 48)
    assert int(g.dev_err.item()) == 0
    assert r["n_lp"] > 0 and r["lp_exact"] >= MIN_EXACT, r
    assert r["ck"] <= TOL_F32, r
    assert r["excess"] <= TOL_F32, r
    assert r["seen"] > 3 * TOL_F32, r  # the read copy's rounding shows in the outputs


@pytest.mark.parametrize("lp", ["bf16", "e4m3"])
@pytest.mark.parametrize("L", [4, 32])
def test_two_precision_buffer_lengths(cuda, L, lp):
    w = synth.make_workload("mamba2_bs256", B=5, H=2, steps=2 * L + 3, seed=L, L=L)
    g, r = _run(cuda, w, lp, 2 * L + 3)
    assert int(g.dev_err.item()) == 0
    assert r["lp_exact"] >= MIN_EXACT and r["ck"] <= TOL_F32 and r["excess"] <= TOL_F32, r


@pytest.mark.parametrize("lp", ["f16", "e4m3"])
def test_two_precision_bs256_full_size_sampled(cuda, lp):
    """The bench's layer (batch 256, 128 heads of 64 x 128, L 16, fp16 or
    E4M3 read copy) for 32 steps in its launch configuration, two heads of
    every row followed by the oracle."""
    w = synth.make_workload("mamba2_bs256", steps=32, seed=2)
    g, r = _run(cuda, w, lp, 32, heads=[5, 100])
    assert int(g.dev_err.item()) == 0
    assert r["lp_exact"] >= MIN_EXACT and r["ck"] <= TOL_F32 and r["excess"] <= TOL_F32, r


@pytest.mark.parametrize("lp", ["f16", "bf16", "e4m3"])
def test_seed_read_copy_is_the_oracle_rounding(cuda, lp):
    """replayssm_seed_read_copy rounds each element of the fp32 recurrence
    copy once: bit for bit the oracle's rounding (E4M3: with the same
    power-of-two row scales)."""
    import torch

    w = synth.make_workload("mamba2_bs256", B=6, H=4, steps=1, seed=8)
    ck = w.ckpt0.copy()
    ck[0, 0, 3] = 0.0                      # a row of zeros
    ck[1, 1, 5] *= 1e-6                    # a tiny row
    ck[2, 2, 7] = 448.0 * 2.0 ** -5        # a maximum on a binade edge
    g = GpuRun(cuda, w, ckpt0=ck, lp_dtype=lp)
    torch.cuda.synchronize()
    got = g.read_copy(np.arange(w.num_slots), np.arange(w.H))
    want = oracle.round_read_copy(ck.astype(np.float64), lp)
    np.testing.assert_array_equal(got, want)
    if lp == "e4m3":
        e = oracle.row_scale_exponent(ck.astype(np.float64))
        np.testing.assert_array_equal(g.ckpt_lp_scale.double().cpu().numpy(), 2.0 ** e)
