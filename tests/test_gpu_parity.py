"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerances (max relative error, per element against max(|ref|, rms of the
head's vector or matrix)):
  * fp32 checkpoint, Mamba-2: 1e-4 against the exact recurrence (the ring holds
    the inputs verbatim, so only fp32 arithmetic order differs).
  * fp16 checkpoint: 2e-2 against the exact recurrence, and 2e-3 against the
    storage-emulating oracle (same roundings as the method).
  * Gated DeltaNet with an fp32 ring: 1e-4 against the exact recurrence (the
    arithmetic of the GDN kernel at fp32 accuracy).
  * Gated DeltaNet with fp16 d/k rings, against the storage-emulating oracle:
    the corrected value d_t is computed (fp32 on the GPU, fp64 in the oracle)
    and then rounded to fp16, so where d_t lies near an fp16 rounding midpoint
    the two sides store codes one ulp apart, and later outputs of the window
    inherit that difference: up to ~|k_c| * ulp(d) / rms, about 5e-4 relative
    on a checkpoint element.  The gate is the pages' own fp32 tolerance (the
    vLLM PR's tests: output rtol = atol = 1e-4, state rtol 1e-3 / atol 2e-3),
    plus a max relative error of 2e-3 derived from one fp16 ulp.
  * Cursors, flags, Mamba-2 ring records, GDN key and gate records: bit-exact.
    GDN corrected values (fp16, rounded on both sides from slightly different
    fp32/fp64 values): within one fp16 rounding, 1e-3.
"""

import numpy as np
import pytest

import oracle
from linear_attention_decode_replayssm_gb300 import synth
from tests._harness import GpuRun, OracleRun, dev, tdt
from tests._util import rel_err

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_F16 = 2e-2
TOL_F16_EMU = 2e-3
TOL_D_RING = 1e-3
TOL_F16_RING = 2e-3            # derived bound for GDN with fp16 d/k rings
PR_OUT = (1e-4, 1e-4)          # (rtol, atol) on outputs
PR_STATE = (1e-3, 2e-3)        # (rtol, atol) on the checkpoint


@pytest.fixture(scope="module")
def cuda(lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def run_parity(lib, w, steps, heads=None, replay=True, exact=True, conventional=False,
               exact_state_dtype="f64", check_rings=True):
    """Step GPU and oracle together; return the worst errors seen."""
    import torch

    g = GpuRun(lib, w, conventional=conventional)
    o = OracleRun(w, heads, replay=replay and not conventional, exact=exact or conventional,
                  exact_state_dtype=exact_state_dtype)
    hs = o.heads
    hs_t = torch.as_tensor(hs, device="cuda")
    res = dict(o_exact=0.0, o_replay=0.0, ck_exact=0.0, ck_replay=0.0, flush_rows=0, pr_out=0.0, pr_state=0.0)
    for t in range(steps):
        x = w.inputs(t)
        ds = w.decode_step(t)
        o_gpu, wp, fl = g.step(x, ds)
        wp_o, fl_o = oracle.plan_step(ds, w.L)
        np.testing.assert_array_equal(wp, wp_o)
        np.testing.assert_array_equal(fl, fl_o)
        assert np.all(np.isfinite(o_gpu)), f"non-finite output at step {t}"
        o_r, o_e = o.step(x, wp, fl)
        og = o_gpu[:, hs]
        pad = w.slot_idx < 0
        assert np.all(og[pad] == 0)
        if o_e is not None:
            res["o_exact"] = max(res["o_exact"], rel_err(og, o_e))
        if o_r is not None:
            res["o_replay"] = max(res["o_replay"], rel_err(og, o_r))
            res["pr_out"] = max(res["pr_out"], _allclose_excess(og, o_r, *PR_OUT))
        flushed = (fl != 0) & ~pad
        if conventional:
            flushed = ~pad
        if flushed.any() and (t % 4 == 0 or steps <= 64 or not conventional):
            slots = w.slot_idx[flushed]
            ck = g.ckpt[torch.as_tensor(slots, device="cuda")][:, hs_t].double().cpu().numpy()
            res["flush_rows"] += int(flushed.sum())
            if o.ex is not None:
                res["ck_exact"] = max(res["ck_exact"], rel_err(ck, o.ex.S[slots], nd=2))
            if o.rs is not None:
                res["ck_replay"] = max(res["ck_replay"], rel_err(ck, o.rs.ckpt[slots], nd=2))
                res["pr_state"] = max(res["pr_state"], _allclose_excess(ck, o.rs.ckpt[slots], *PR_STATE))
    assert int(g.dev_err.item()) == 0
    if check_rings and not conventional and o.rs is not None:
        res["ring"] = compare_rings(g, o, w, steps)
    return res


def same_bits(a, b):
    """Bitwise tensor equality (NaN-poisoned stale ring slots compare equal)."""
    import torch

    ints = {4: torch.int32, 2: torch.int16, 1: torch.uint8}
    return torch.equal(a.view(ints[a.element_size()]), b.view(ints[b.element_size()]))


def _allclose_excess(x, y, rtol, atol):
    """max(|x - y| - rtol |y|) / atol: <= 1 exactly when allclose(x, y, rtol, atol)."""
    return float(np.max(np.abs(x - y) - rtol * np.abs(y)) / atol) if np.size(y) else 0.0


def assert_gdn_f16_ring(r):
    assert r["pr_out"] <= 1.0 and r["pr_state"] <= 1.0, r
    assert r["o_replay"] <= TOL_F16_RING and r["ck_replay"] <= TOL_F16_RING, r


def compare_rings(g, o, w, steps):
    """Records each live slot holds after ``steps``: Mamba-2 and GDN keys and
    gates bit-exact; GDN corrected values within one fp16 rounding."""
    import torch

    hs = torch.as_tensor(o.heads, device="cuda")
    held = w.decode_step(steps) % w.L
    worst_d = 0.0
    for b in range(w.B):
        s = int(w.slot_idx[b])
        p = int(held[b])
        if s < 0 or p == 0:
            continue
        rv = g.ring_v[s][hs, :p].double().cpu().numpy()
        rk = g.ring_k[s][hs, :p].double().cpu().numpy()
        ra = g.ring_a[s][hs, :p].double().cpu().numpy()
        np.testing.assert_array_equal(rk, o.rs.ring_k[s, :, :p])
        np.testing.assert_array_equal(ra, o.rs.ring_a[s, :, :p])
        if w.variant == "mamba2":
            np.testing.assert_array_equal(rv, o.rs.ring_v[s, :, :p])
        else:
            worst_d = max(worst_d, rel_err(rv, o.rs.ring_v[s, :, :p]))
    assert worst_d <= TOL_D_RING, worst_d
    return worst_d


# --------------------------------------------------------------------------
# Mamba-2
# --------------------------------------------------------------------------
def test_tiny_mamba2_fp32(cuda):
    # batch 2, 2 heads, 16 x 32, L = 4, 64 steps from a zero checkpoint, fp32 state and inputs
    w = synth.make_workload("tiny")
    r = run_parity(cuda, w, w.steps)
    assert r["flush_rows"] == 2 * 16
    assert r["o_exact"] <= TOL_F32, r
    assert r["ck_exact"] <= TOL_F32, r
    assert r["o_replay"] <= TOL_F32, r


def test_tiny_mamba2_fp16_checkpoint(cuda):
    w = synth.make_workload("tiny", ckpt_dtype="f16", stagger=True, zero_ckpt=False)
    r = run_parity(cuda, w, w.steps)
    assert r["o_exact"] <= TOL_F16, r
    assert r["o_replay"] <= TOL_F16_EMU, r
    assert r["ck_replay"] <= TOL_F16_EMU, r


@pytest.mark.parametrize("ckpt_dtype", ["f32", "f16"])
def test_mamba2_paged_padded_ragged(cuda, ckpt_dtype):
    # production head shape; permuted slots in a larger pool, padded rows, L = 5
    w = synth.make_workload("mamba2_bs256", B=7, H=3, L=5, steps=23, num_slots=16, permute_slots=True,
                            pad_rows=2, ckpt_dtype=ckpt_dtype, seed=3)
    r = run_parity(cuda, w, w.steps)
    tol = TOL_F32 if ckpt_dtype == "f32" else TOL_F16
    assert r["o_exact"] <= tol, r
    assert r["ck_exact"] <= tol, r
    assert r["flush_rows"] > 0


@pytest.mark.parametrize("L", [2, 8, 32, 64])
@pytest.mark.parametrize("ckpt_dtype", ["f32", "f16"])
def test_mamba2_buffer_lengths(cuda, L, ckpt_dtype):
    w = synth.make_workload("mamba2_bs256", B=4, H=2, L=L, steps=2 * L + 3, ckpt_dtype=ckpt_dtype, seed=L)
    r = run_parity(cuda, w, w.steps)
    if ckpt_dtype == "f32":
        assert r["o_exact"] <= TOL_F32 and r["ck_exact"] <= TOL_F32, r
    else:
        assert r["o_exact"] <= TOL_F16 and r["o_replay"] <= TOL_F16_EMU, r


def test_mamba2_head_dim_128(cuda):
    w = synth.make_workload("mamba2_bs256", B=5, H=2, d_v=128, d_k=128, steps=40, seed=5)
    r = run_parity(cuda, w, w.steps)
    assert r["o_exact"] <= TOL_F32 and r["ck_exact"] <= TOL_F32, r


def test_mamba2_bs256_full_size_sampled(cuda):
    # batch 256, 128 heads of 64 x 128, fp32 checkpoint, bf16 inputs, L = 16,
    # staggered cursors, 256 steps -- the launch the benchmark times; the
    # oracle follows three heads of every row
    w = synth.make_workload("mamba2_bs256")
    r = run_parity(cuda, w, w.steps, heads=[0, 77, 127], replay=False, check_rings=False)
    assert r["o_exact"] <= TOL_F32, r
    assert r["ck_exact"] <= TOL_F32, r
    assert r["flush_rows"] == 256 * 16


# --------------------------------------------------------------------------
# Gated DeltaNet
# --------------------------------------------------------------------------
def test_tiny_gdn(cuda):
    w = synth.make_workload("tiny", variant="gdn", ring_dtype="f16", alpha_mu=3.0, alpha_sd=1.0)
    r = run_parity(cuda, w, w.steps)
    assert_gdn_f16_ring(r)


def test_gdn_fp32_ring_matches_exact(cuda):
    w = synth.make_workload("gdn_bs256", B=4, H=2, steps=40, ring_dtype="f32", seed=7)
    r = run_parity(cuda, w, w.steps)
    assert r["o_exact"] <= TOL_F32 and r["ck_exact"] <= TOL_F32, r


@pytest.mark.parametrize("ckpt_dtype", ["f32", "f16"])
def test_gdn_paged_padded(cuda, ckpt_dtype):
    w = synth.make_workload("gdn_bs256", B=6, H=3, steps=40, num_slots=9, permute_slots=True, pad_rows=1,
                            ckpt_dtype=ckpt_dtype, seed=11)
    r = run_parity(cuda, w, w.steps)
    if ckpt_dtype == "f32":
        assert_gdn_f16_ring(r)
    else:
        assert r["o_exact"] <= TOL_F16 and r["o_replay"] <= TOL_F16_EMU, r


@pytest.mark.parametrize("L", [4, 32])
def test_gdn_buffer_lengths(cuda, L):
    w = synth.make_workload("gdn_bs256", B=3, H=2, L=L, steps=2 * L + 1, seed=L)
    r = run_parity(cuda, w, w.steps)
    assert_gdn_f16_ring(r)
    w32 = synth.make_workload("gdn_bs256", B=3, H=2, L=L, steps=2 * L + 1, seed=L, ring_dtype="f32")
    r32 = run_parity(cuda, w32, w32.steps)
    assert r32["o_exact"] <= TOL_F32 and r32["ck_exact"] <= TOL_F32, r32


@pytest.mark.parametrize("d_v, in_dtype, ckpt_dtype", [(64, "bf16", "f32"), (128, "f32", "f32"), (64, "f32", "f16")])
def test_gdn_other_shapes_and_inputs(cuda, d_v, in_dtype, ckpt_dtype):
    # 64 x 128 heads (one unit per head) and fp32 inputs, with fp32 rings so
    # that the comparison with the exact recurrence is tight
    w = synth.make_workload("gdn_bs256", B=5, H=3, d_v=d_v, steps=40, in_dtype=in_dtype, ring_dtype="f32",
                            ckpt_dtype=ckpt_dtype, pad_rows=1, seed=d_v + len(in_dtype))
    r = run_parity(cuda, w, w.steps)
    if ckpt_dtype == "f32":
        assert r["o_exact"] <= TOL_F32 and r["ck_exact"] <= TOL_F32, r
    else:
        assert r["o_exact"] <= TOL_F16 and r["o_replay"] <= TOL_F16_EMU, r


def test_gdn_bs256_full_size_sampled(cuda):
    # batch 256, 32 value heads of 128 x 128, fp32 checkpoint, fp16 d/k rings,
    # fp32 g ring, L = 16 staggered, 256 steps; the oracle follows two heads
    w = synth.make_workload("gdn_bs256")
    r = run_parity(cuda, w, w.steps, heads=[0, 31], exact=False)
    assert_gdn_f16_ring(r)
    assert r["flush_rows"] == 256 * 16


# --------------------------------------------------------------------------
# conventional baseline
# --------------------------------------------------------------------------
@pytest.mark.parametrize("variant", ["mamba2", "gdn"])
@pytest.mark.parametrize("ckpt_dtype", ["f32", "f16"])
def test_conventional(cuda, variant, ckpt_dtype):
    name = "mamba2_bs256" if variant == "mamba2" else "gdn_bs256"
    w = synth.make_workload(name, B=5, H=3, steps=30, ckpt_dtype=ckpt_dtype, num_slots=8, permute_slots=True,
                            pad_rows=1, stagger=False, seed=13)
    # the oracle rounds the state to its storage type after every step, as the
    # kernel does; with an fp16 state the two sides' roundings diverge on
    # near-midpoint elements and compound step by step, so that case takes the
    # fp16-state tolerance
    r = run_parity(cuda, w, w.steps, conventional=True, exact_state_dtype=ckpt_dtype)
    tol = TOL_F32 if ckpt_dtype == "f32" else TOL_F16
    assert r["o_exact"] <= tol and r["ck_exact"] <= tol, r


def test_conventional_tiny(cuda):
    w = synth.make_workload("tiny")
    r = run_parity(cuda, w, w.steps, conventional=True, exact_state_dtype="f32")
    assert r["o_exact"] <= TOL_F32, r


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------
def test_device_range_checks(cuda):
    import torch

    lib = cuda
    w = synth.make_workload("mamba2_bs256", B=4, H=2, steps=1, seed=17)
    g = GpuRun(lib, w)
    bad_slot = w.slot_idx.copy()
    bad_slot[1] = w.num_slots + 3
    g.slot_idx.copy_(dev(bad_slot, torch.int32))
    ds = w.decode_step(0).copy()
    out, _, _ = g.step(w.inputs(0), ds)
    assert int(g.dev_err.item()) & lib.RS_DERR_SLOT
    assert np.all(out[1] == 0)
    # a cursor outside [0, L): written straight to the device buffer
    g.dev_err.zero_()
    g.slot_idx.copy_(dev(w.slot_idx, torch.int32))
    wp, fl = lib.replayssm_plan_step(ds, w.L)
    wp[2] = w.L + 5
    g.wp.copy_(dev(wp, torch.int32))
    g.fl.copy_(dev(fl, torch.uint8))
    t = g.tensors(w.inputs(0))
    ck0 = g.ckpt.clone()
    ra0 = g.ring_a.clone()
    lib.replayssm_decode_mamba2(ckpt=g.ckpt, ring_v=g.ring_v, ring_k=g.ring_k, ring_a=g.ring_a,
                                slot_idx=g.slot_idx, write_pos=g.wp, is_flush=g.fl, v=t["v"], k=t["k"],
                                q=t["q"], alpha=t["alpha"], out=g.out, dev_err=g.dev_err)
    assert int(g.dev_err.item()) == lib.RS_DERR_WRITE_POS
    assert torch.all(g.out[2] == 0)
    s2 = int(w.slot_idx[2])
    assert same_bits(g.ckpt[s2], ck0[s2]) and same_bits(g.ring_a[s2], ra0[s2])


def test_strided_rows_match_packed(cuda):
    import torch

    lib = cuda
    w = synth.make_workload("mamba2_bs256", B=6, H=4, steps=20, seed=19)
    a, b = GpuRun(lib, w), GpuRun(lib, w)
    for t in range(w.steps):
        x = w.inputs(t)
        oa, _, _ = a.step(x, w.decode_step(t))
        tb = b.tensors(x)
        padded = {}
        for n in ("v", "k", "q"):
            big = torch.zeros(w.B, tb[n].shape[1] * tb[n].shape[2] + 24, dtype=tb[n].dtype, device="cuda")
            view = big[:, : tb[n].shape[1] * tb[n].shape[2]].view(w.B, tb[n].shape[1], tb[n].shape[2])
            view.copy_(tb[n])
            padded[n] = view
        big_o = torch.full((w.B, w.H * w.d_v + 8), 7.0, device="cuda")
        out_view = big_o[:, : w.H * w.d_v].view(w.B, w.H, w.d_v)
        ob, _, _ = b.step(x, w.decode_step(t), out=out_view, **padded)
        np.testing.assert_array_equal(oa, ob)
        assert torch.all(big_o[:, w.H * w.d_v:] == 7.0)


def test_cuda_graph_replay_matches_eager(cuda):
    import torch

    lib = cuda
    w = synth.make_workload("mamba2_bs256", B=16, H=8, steps=16, seed=23)
    eager, graphed = GpuRun(lib, w), GpuRun(lib, w)
    GpuRun(lib, w).step(w.inputs(0), w.decode_step(0))  # load the kernel before capturing
    xs = [graphed.tensors(w.inputs(t)) for t in range(w.steps)]
    plans = [lib.replayssm_plan_step(w.decode_step(t), w.L) for t in range(w.steps)]
    wps = torch.stack([dev(p[0], torch.int32) for p in plans])
    fls = torch.stack([dev(p[1], torch.uint8) for p in plans])
    outs = torch.empty(w.steps, w.B, w.H, w.d_v, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for t in range(w.steps):
                lib.replayssm_decode_mamba2(ckpt=graphed.ckpt, ring_v=graphed.ring_v, ring_k=graphed.ring_k,
                                            ring_a=graphed.ring_a, slot_idx=graphed.slot_idx, write_pos=wps[t],
                                            is_flush=fls[t], v=xs[t]["v"], k=xs[t]["k"], q=xs[t]["q"],
                                            alpha=xs[t]["alpha"], out=outs[t])
    # capture records without running; the state is still the starting one
    graph.replay()
    torch.cuda.synchronize()
    for t in range(w.steps):
        o_e, _, _ = eager.step(w.inputs(t), w.decode_step(t))
        np.testing.assert_array_equal(outs[t].double().cpu().numpy(), o_e)
    for name in ("ckpt", "ring_v", "ring_k", "ring_a"):
        assert same_bits(getattr(eager, name), getattr(graphed, name)), name
