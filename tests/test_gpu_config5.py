"""Multi-layer Mamba-2 decode with continuous batching, GPU against the oracle.

Each layer is an independent state pool (there are no weights, so no data
flows between layers); one churn schedule drives all layers: every 8 steps,
at a random offset per row, a row's request may finish and a new request takes
its slot at decode step 0 with a fresh checkpoint, leaving the slot's ring as
it was.  Cursors and flags come from the host plan each step.

Gates as in test_gpu_parity: fp32 checkpoint, max relative error 1e-4 against
the exact recurrence, for outputs and for every flushed checkpoint.
"""

import numpy as np
import pytest

import oracle
from linear_attention_decode_replayssm_gb300 import synth
from tests._harness import GpuRun, OracleRun, dev, tdt
from tests._util import rel_err

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def cuda(lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def _fresh(w, layer, t, rows):
    """Fresh checkpoints for requests joining at step t (stand-in for prefill)."""
    r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 5000 + layer, t])))
    x = r.standard_normal((len(rows), w.H, w.d_v, w.d_k), dtype=np.float32) / np.sqrt(np.float32(w.d_k))
    return synth.quantize(x, w.ckpt_dtype)


def test_layers_with_churn_reduced(cuda):
    import torch

    lib = cuda
    n_layers, steps = 3, 96
    ds0 = np.random.default_rng(3).integers(0, 16, 12)
    ws = [synth.make_workload("mamba2_bs256", B=12, H=4, steps=steps, seed=40 + l, cursor0=ds0)
          for l in range(n_layers)]
    sched = synth.ChurnSchedule(12, 16, steps, period=8, p_churn=0.3, seed=9, decode_step0=ds0)
    gs = [GpuRun(lib, w) for w in ws]
    os_ = [OracleRun(w, replay=False) for w in ws]
    worst_o = worst_c = 0.0
    joins = 0
    for t in range(steps):
        ds = sched.decode_step(t)
        rows = sched.joins(t)
        joins += len(rows)
        for l, (w, g, o) in enumerate(zip(ws, gs, os_)):
            if len(rows):
                fresh = _fresh(w, l, t, rows)
                for i, b in enumerate(rows):
                    s = int(w.slot_idx[b])
                    g.ckpt[s].copy_(dev(fresh[i], tdt(w.ckpt_dtype)))
                    o.ex.reset_slot(s, fresh[i].astype(np.float64))
            x = w.inputs(t)
            out, wp, fl = g.step(x, ds)
            wp_o, fl_o = oracle.plan_step(ds, w.L)
            np.testing.assert_array_equal(wp, wp_o)
            np.testing.assert_array_equal(fl, fl_o)
            _, o_e = o.step(x, wp, fl)
            worst_o = max(worst_o, rel_err(out, o_e))
            if fl.any():
                slots = w.slot_idx[fl != 0]
                ck = g.ckpt[torch.as_tensor(slots, device="cuda")].double().cpu().numpy()
                worst_c = max(worst_c, rel_err(ck, o.ex.S[slots], nd=2))
    assert joins > 10
    assert int(sum(g.dev_err.item() for g in gs)) == 0
    assert worst_o <= TOL and worst_c <= TOL, (worst_o, worst_c)


def test_forty_layers_with_churn_full_size(cuda):
    """40 layers, batch 256, 128 heads of 64 x 128, fp32 checkpoints, L = 16,
    512 steps with churn.  Inputs are drawn on the device with a seeded
    generator; the oracle follows 4 heads of every row in 3 of the layers."""
    import torch

    lib = cuda
    B, H, dv, dk, L, steps, n_layers = 256, 128, 64, 128, 16, 512, 40
    check_layers, heads = (0, 19, 39), np.array([0, 41, 86, 127])
    hs_t = torch.as_tensor(heads, device="cuda")
    r0 = np.random.default_rng(11)
    ds0 = r0.integers(0, L, B)
    sched = synth.ChurnSchedule(B, L, steps, period=8, p_churn=0.25, seed=12, decode_step0=ds0)
    gen = torch.Generator(device="cuda")
    slot_idx = torch.arange(B, device="cuda", dtype=torch.int32)
    layers = []
    for l in range(n_layers):
        gen.manual_seed(1000 + l)
        ckpt = synth.device_draw((B, H, dv, dk), "scaled", gen, d_k=dk)
        ring_v = synth.device_draw((B, H, L, dv), "scaled", gen, d_k=dk).to(torch.bfloat16)
        ring_k = synth.device_draw((B, H, L, dk), "scaled", gen, d_k=dk).to(torch.bfloat16)
        ring_a = synth.device_draw((B, H, L), "sigmoid3", gen)
        layers.append(dict(ckpt=ckpt, ring_v=ring_v, ring_k=ring_k, ring_a=ring_a))
    # oracle: exact state of the sampled heads, rebuilt from checkpoint + held records
    ex = {}
    for l in check_layers:
        lay = layers[l]
        rs = oracle.ReplayState("mamba2", lay["ckpt"][:, hs_t].double().cpu().numpy(),
                                lay["ring_v"][:, hs_t].double().cpu().numpy(),
                                lay["ring_k"][:, hs_t].double().cpu().numpy(),
                                lay["ring_a"][:, hs_t].double().cpu().numpy())
        ex[l] = oracle.ExactState.from_replay(rs, ds0 % L)
    out = torch.empty(B, H, dv, device="cuda")
    wp_d = torch.empty(B, device="cuda", dtype=torch.int32)
    fl_d = torch.empty(B, device="cuda", dtype=torch.uint8)
    dev_err = torch.zeros(1, device="cuda", dtype=torch.int32)
    worst_o = worst_c = 0.0
    for t in range(steps):
        ds = sched.decode_step(t)
        wp, fl = lib.replayssm_plan_step(ds, L)
        np.testing.assert_array_equal((wp, fl), oracle.plan_step(ds, L))
        wp_d.copy_(torch.from_numpy(wp))
        fl_d.copy_(torch.from_numpy(fl))
        rows = sched.joins(t)
        for l in range(n_layers):
            lay = layers[l]
            gen.manual_seed(10_000_000 + 1000 * t + l)
            if len(rows):
                rows_t = torch.as_tensor(rows, device="cuda")
                fresh = synth.device_draw((len(rows), H, dv, dk), "scaled", gen, d_k=dk)
                lay["ckpt"][rows_t] = fresh
                if l in ex:
                    f64 = fresh[:, hs_t].double().cpu().numpy()
                    for i, b in enumerate(rows):
                        ex[l].reset_slot(int(b), f64[i])
            v = synth.device_draw((B, H, dv), "scaled", gen, d_k=dk).to(torch.bfloat16)
            k = synth.device_draw((B, H, dk), "scaled", gen, d_k=dk).to(torch.bfloat16)
            q = synth.device_draw((B, H, dk), "scaled", gen, d_k=dk).to(torch.bfloat16)
            alpha = synth.device_draw((B, H), "sigmoid3", gen)
            lib.replayssm_decode_mamba2(ckpt=lay["ckpt"], ring_v=lay["ring_v"], ring_k=lay["ring_k"],
                                        ring_a=lay["ring_a"], slot_idx=slot_idx, write_pos=wp_d, is_flush=fl_d,
                                        v=v, k=k, q=q, alpha=alpha, out=out, dev_err=dev_err)
            if l in ex:
                sub = lambda x: x[:, hs_t].double().cpu().numpy()
                o_e = oracle.exact_step(ex[l], np.arange(B), sub(v), sub(k), sub(q), sub(alpha))
                worst_o = max(worst_o, rel_err(out[:, hs_t].double().cpu().numpy(), o_e))
                if fl.any():
                    rs_ = np.nonzero(fl)[0]
                    ck = lay["ckpt"][torch.as_tensor(rs_, device="cuda")][:, hs_t].double().cpu().numpy()
                    worst_c = max(worst_c, rel_err(ck, ex[l].S[rs_], nd=2))
    assert int(dev_err.item()) == 0
    assert sched.join.sum() > 1000
    assert worst_o <= TOL and worst_c <= TOL, (worst_o, worst_c)
