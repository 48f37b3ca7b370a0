"""Group-shared keys (Mamba-2) on the GPU against the oracle.

Keys and queries are [B, G, d_k], one per group of H / G value heads, and the
key ring is kept once per group; the group dot kernel computes k_j . q_t once
per (row, group) and the decode reads those dots.  The oracle runs the
per-head recurrence on the keys expanded to heads (``heads_from_groups``),
which is what the grouped layout computes.

Gates as in test_gpu_parity: outputs and flushed fp32 checkpoints at max
relative error 1e-4 against the exact recurrence; the group key ring
(appended once per group on non-flush rows) bit-exact; cursors bit-exact.
"""

import numpy as np
import pytest

import oracle
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


def _to_heads(x, H, axis):
    """Group axis ``axis`` of x expanded to H heads."""
    return np.moveaxis(oracle.heads_from_groups(np.moveaxis(x, axis, -2), H), -2, axis)


def _group_keys(w, G, t):
    """Seeded group keys and queries of step t, [B, G, d_k] (bf16 values)."""
    r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 70_000 + t])))
    sk = np.sqrt(np.float32(w.d_k))
    k = r.standard_normal((w.B, G, w.d_k), dtype=np.float32) / sk
    q = r.standard_normal((w.B, G, w.d_k), dtype=np.float32) / sk
    return synth.quantize(k, w.in_dtype), synth.quantize(q, w.in_dtype)


def _run(lib, w, G, steps, heads=None):
    import torch

    B, H, L, S = w.B, w.H, w.L, w.num_slots
    hs = np.arange(H) if heads is None else np.asarray(heads)
    hs_t = torch.as_tensor(hs, device="cuda")
    # the group key ring: p held records per slot, the rest NaN
    r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 69_999])))
    ring_kg = np.full((S, G, L, w.d_k), np.nan, dtype=np.float32)
    held = w.held_records()
    for s in range(S):
        if held[s]:
            x = r.standard_normal((G, held[s], w.d_k), dtype=np.float32) / np.sqrt(np.float32(w.d_k))
            ring_kg[s, :, : held[s]] = synth.quantize(x, w.ring_dtype)
    td = tdt(w.in_dtype)
    ckpt = dev(w.ckpt0, tdt(w.ckpt_dtype))
    ring_v, ring_k = dev(w.ring_v0, td), dev(ring_kg, td)
    ring_a = dev(w.ring_a0, torch.float32)
    slot_idx = dev(w.slot_idx, torch.int32)
    out = torch.empty(B, H, w.d_v, device="cuda")
    wp_d = torch.empty(B, device="cuda", dtype=torch.int32)
    fl_d = torch.empty(B, device="cuda", dtype=torch.uint8)
    kq = torch.full((B * G * L,), np.nan, device="cuda")
    dev_err = torch.zeros(1, device="cuda", dtype=torch.int32)
    rk_heads = np.stack([_to_heads(ring_kg[s], H, 0)[hs] for s in range(S)])  # slot by slot: no [S, H] copy
    rs = oracle.ReplayState("mamba2", w.ckpt0[:, hs].astype(np.float64), w.ring_v0[:, hs].astype(np.float64),
                            rk_heads.astype(np.float64), w.ring_a0[:, hs].astype(np.float64))
    ex = oracle.ExactState.from_replay(rs, held)
    live = w.slot_idx >= 0
    worst_o = worst_c = 0.0
    n_flush = 0
    for t in range(steps):
        ds = w.decode_step(t)
        wp, fl = lib.replayssm_plan_step(ds, L)
        wp_d.copy_(torch.from_numpy(wp))
        fl_d.copy_(torch.from_numpy(fl))
        x = w.inputs(t)
        kg, qg = _group_keys(w, G, t)
        lib.replayssm_decode_mamba2(ckpt=ckpt, ring_v=ring_v, ring_k=ring_k, ring_a=ring_a, slot_idx=slot_idx,
                                    write_pos=wp_d, is_flush=fl_d, v=dev(x["v"], td), k=dev(kg, td), q=dev(qg, td),
                                    alpha=dev(x["alpha"], torch.float32), out=out, dev_err=dev_err, kq_scratch=kq)
        kh, qh = _to_heads(kg, H, 1)[:, hs], _to_heads(qg, H, 1)[:, hs]
        o_e = oracle.exact_step(ex, w.slot_idx, x["v"][:, hs], kh, qh, x["alpha"][:, hs])
        o_g = out[:, hs_t].double().cpu().numpy()
        worst_o = max(worst_o, rel_err(o_g[live], o_e[live]))
        assert np.all(o_g[~live] == 0)
        rows = np.nonzero(live & (fl != 0))[0]
        if len(rows):
            n_flush += len(rows)
            sl = torch.as_tensor(w.slot_idx[rows], device="cuda")
            worst_c = max(worst_c, rel_err(ckpt[sl][:, hs_t].double().cpu().numpy(), ex.S[w.slot_idx[rows]], nd=2))
        # non-flush rows appended their group's key once, at slot write_pos
        for b in np.nonzero(live & (fl == 0))[0][:8]:
            got = ring_k[int(w.slot_idx[b]), :, int(wp[b])].float().cpu().numpy()
            np.testing.assert_array_equal(got, kg[b])
    return int(dev_err.item()), worst_o, worst_c, n_flush


@pytest.mark.parametrize("G", [1, 2, 4])
def test_grouped_small(cuda, G):
    w = synth.make_workload("mamba2_bs256", B=7, H=8, steps=40, seed=50 + G, pad_rows=1, num_slots=10,
                            permute_slots=True)
    err, worst_o, worst_c, n_flush = _run(cuda, w, G, 40)
    assert err == 0 and n_flush > 0
    assert worst_o <= TOL and worst_c <= TOL, (worst_o, worst_c)


def test_grouped_buffer_length_32(cuda):
    w = synth.make_workload("mamba2_bs256", B=5, H=4, steps=70, seed=9, L=32)
    err, worst_o, worst_c, n_flush = _run(cuda, w, 2, 70)
    assert err == 0 and n_flush > 0
    assert worst_o <= TOL and worst_c <= TOL, (worst_o, worst_c)


def test_grouped_bs256_full_size_sampled(cuda):
    """Batch 256, 128 heads of 64 x 128 in 8 groups of 16 (the layer's own
    key layout), fp32, L 16, 32 steps; three heads of every row checked."""
    w = synth.make_workload("mamba2_bs256", steps=32, seed=12)
    err, worst_o, worst_c, n_flush = _run(cuda, w, 8, 32, heads=[0, 47, 127])
    assert err == 0 and n_flush >= 256
    assert worst_o <= TOL and worst_c <= TOL, (worst_o, worst_c)
