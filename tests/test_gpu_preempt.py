"""Preemption and load-back of a row in the middle of a window.

Among the faults the shipped method met in the field the pages list ring
cursors that were not reset after a cache load-back, checkpoints left
unflushed, and pending updates lost when a request was retracted to the host
("ReplaySSM: an SSM decoder that writes its state once every 16 tokens",
§What actually shipped); their test plan re-anchors the ring when a request
resumes after preemption ("[Kernel] ReplaySSM: cache SSM inputs for faster
Gated DeltaNet standard decode", §Tests).  A row is preempted while its ring
holds p > 0 records and resumes later in a different slot, by one of two
routes, both through the C ABI:

  copy         its checkpoint and ring go to host memory and come back into
               the new slot; the row keeps its decode-step counter, so its
               cursor continues in the middle of the window;
  materialise  the held records are folded into the state once
               (replayssm_materialize into a staging pool), only that state
               goes to host memory and comes back as the new slot's
               checkpoint, and the row's cursor restarts at 0.  The new
               slot's ring is poisoned with NaN, so a cursor that was not
               reset would show in the outputs.

Meanwhile a new request takes the preempted row's old slot (fresh
checkpoint, decode step 0) and overwrites its ring and, at its first flush,
its checkpoint.  The oracle keeps the exact state per request, not per slot.

Gates: outputs and every flushed checkpoint at max relative error 1e-4
against the exact recurrence of each request (fp32 checkpoints; GDN with fp32
rings); cursors and flags bit-exact against the oracle's plan.
"""

import numpy as np
import pytest

import oracle
from linear_attention_decode_replayssm_gb300 import synth
from tests._harness import GpuRun, dev, tdt
from tests._util import rel_err

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def cuda(lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


@pytest.mark.parametrize("route", ["copy", "materialise"])
@pytest.mark.parametrize("variant", ["mamba2", "gdn"])
def test_preempt_and_resume_in_another_slot(cuda, variant, route):
    import torch

    lib = cuda
    B, H, L, steps = 6, 4, 16, 60
    n_slots = B + 3
    name = "mamba2_bs256" if variant == "mamba2" else "gdn_bs256"
    kw = dict(ring_dtype="f32") if variant == "gdn" else {}
    w = synth.make_workload(name, B=B, H=H, L=L, steps=steps, num_slots=n_slots, seed=71 + len(route), **kw)
    g = GpuRun(lib, w)
    fresh = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 555])))
    # batch positions B-2 and B-1 start empty; preempted requests resume there
    phys = w.slot_idx.copy()
    phys[B - 2:] = -1
    ds = w.decode_step0.copy()
    ds[B - 2:] = 0
    # exact state per request id; requests 0..B-3 start in slots 0..B-3
    rs0 = oracle.ReplayState(variant, w.ckpt0.astype(np.float64), w.ring_v0.astype(np.float64),
                             w.ring_k0.astype(np.float64), w.ring_a0.astype(np.float64))
    held0 = w.held_records()
    S = np.zeros((n_slots + 8, H, w.d_v, w.d_k))
    S[:n_slots] = oracle.ExactState.from_replay(rs0, held0).S
    ex = oracle.ExactState(variant, S)
    rid = phys.copy()  # request served by each batch position (-1: none)
    next_rid = n_slots
    free_slots = [n_slots - 2, n_slots - 1]  # slots no row uses yet
    saved = None
    events = {8: "preempt", 17: "resume", 29: "preempt", 41: "resume"}
    worst_o = worst_c = 0.0
    n_flush = n_resumed = 0
    for t in range(steps):
        ev = events.get(t)
        if ev == "preempt":
            # the live row holding the most records (p > 0), between two steps
            live = np.nonzero(phys >= 0)[0]
            b = int(live[np.argmax(ds[live] % L)])
            p = int(ds[b] % L)
            assert p > 0
            old = int(phys[b])
            if route == "copy":
                host = {n: getattr(g, n)[old].cpu() for n in ("ckpt", "ring_v", "ring_k", "ring_a")}
            else:
                staging = torch.full((1, H, w.d_v, w.d_k), np.nan, device="cuda", dtype=tdt(w.ckpt_dtype))
                lib.replayssm_materialize(variant=lib.RS_GDN if variant == "gdn" else lib.RS_MAMBA2,
                                          ckpt=g.ckpt, ring_v=g.ring_v, ring_k=g.ring_k, ring_a=g.ring_a,
                                          slot_idx=dev(np.array([old]), torch.int32),
                                          held=dev(np.array([p]), torch.int32), dst=staging,
                                          dst_idx=dev(np.array([0]), torch.int32), dev_err=g.dev_err)
                host = {"ckpt": staging[0].cpu()}
            saved = dict(rid=int(rid[b]), ds=int(ds[b]), p=p, host=host)
            # a new request takes the old slot at decode step 0
            ck = w.fresh_checkpoint(fresh, 1)[0]
            g.ckpt[old] = dev(ck, tdt(w.ckpt_dtype))
            ex.reset_slot(next_rid, ck)
            rid[b], ds[b] = next_rid, 0
            next_rid += 1
        elif ev == "resume":
            new = free_slots.pop(0)
            for n, x in saved["host"].items():
                getattr(g, n)[new].copy_(x.to("cuda"))
            if route == "materialise":
                for n in ("ring_v", "ring_k", "ring_a"):
                    getattr(g, n)[new].fill_(np.nan)  # stale ring: must never be read
            b = int(np.nonzero(phys < 0)[0][-1])
            phys[b], rid[b] = new, saved["rid"]
            ds[b] = saved["ds"] if route == "copy" else 0
            resumed_row, saved = b, None
        g.slot_idx.copy_(dev(phys, torch.int32))
        x = w.inputs(t)
        step_ds = np.where(phys >= 0, ds, 0)
        out, wp, fl = g.step(x, step_ds)
        np.testing.assert_array_equal((wp, fl), oracle.plan_step(step_ds, L))
        if ev == "resume":
            n_resumed += 1
            want = (ds[resumed_row] % L) if route == "copy" else 0
            assert wp[resumed_row] == want
            if route == "copy":
                assert want > 0  # continues mid-window
        o_e = oracle.exact_step(ex, rid, x["v"], x["k"], x["q"], x["alpha"], x.get("beta"))
        live = phys >= 0
        assert np.all(np.isfinite(out)), f"non-finite output at step {t}"
        assert np.all(out[~live] == 0)
        worst_o = max(worst_o, rel_err(out[live], o_e[live]))
        rows = np.nonzero(live & (fl != 0))[0]
        if len(rows):
            n_flush += len(rows)
            ck = g.ckpt[torch.as_tensor(phys[rows], device="cuda")].double().cpu().numpy()
            worst_c = max(worst_c, rel_err(ck, ex.S[rid[rows]], nd=2))
        ds = np.where(live, ds + 1, ds)
    assert n_resumed == 2 and n_flush > 0
    assert int(g.dev_err.item()) == 0
    assert worst_o <= TOL and worst_c <= TOL, (worst_o, worst_c)
