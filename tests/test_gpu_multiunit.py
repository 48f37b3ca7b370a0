"""Every kernel of the launch tables against the oracle with several units per CTA.

The decode, verification and read-copy kernels are persistent: a CTA takes
the units (row, head[, half]) strided across the batch, two consumer groups
take alternate units, and the checkpoint and record slots of the CTA's
shared-memory rings are reused unit after unit, flipping their barrier
phases.  A launch with fewer units than CTAs runs none of that, so every
case here has at least four units per CTA: the grid is at most two CTAs per
SM, and each case asserts units >= 8 x SMs before it runs.  The oracle
follows two or three heads of every row, which keeps its CPU cost small while
every CTA still computes its full share.

Coverage follows the pages' test plan ("[Kernel] ReplaySSM: cache SSM inputs
for faster Gated DeltaNet standard decode", §Tests: small and production
geometries, a buffer-length sweep, a per-row write-position sweep -- here
staggered cursors -- and every state precision the kernels take):

  * Mamba-2, one checkpoint copy: 64 x 128 fp32 and fp16 at L 8 / 16 / 32 /
    64 (the compile-time window bounds 8, 16, 32 and 64), 128 x 128 and
    16 x 32 heads, bf16 and fp32 inputs; batch 512 at L 16 in fp32 and fp16;
    an odd head count;
  * the two-precision checkpoint with fp16 and bf16 read copies, both input
    types and every head shape, and the E4M3 read copy (64 x 128 heads) at
    L 16 / 32 / 64;
  * group-shared keys with fp32 and fp16 checkpoints;
  * Gated DeltaNet with fp32 and fp16 checkpoints, fp16 and fp32 rings, L 4 /
    16 / 32, and the batch-256 layer with fp32 rings against the exact
    recurrence;
  * speculative verification at T 1, 2, 8 and 16 with L 16, 32 and 64, and an
    fp16 checkpoint.

Gates are those of the other GPU parity tests: max relative error 1e-4
against the exact recurrence for fp32 checkpoints (Mamba-2, GDN with fp32
rings, verification); 2e-2 against exact and 2e-3 against the
storage-emulating oracle for fp16 checkpoints; the pages' allclose plus 2e-3
for GDN's fp16 d/k rings; ring records and cursors bit-exact.
"""

import numpy as np
import pytest

from linear_attention_decode_replayssm_gb300 import synth
from tests import test_gpu_grouped as grouped
from tests import test_gpu_parity as par
from tests import test_gpu_spec as spec
from tests import test_gpu_two_precision as twop

pytestmark = pytest.mark.gpu

UNITS_PER_CTA = 4
CTAS_PER_SM = 2  # the most any launch plan puts on one SM


@pytest.fixture(scope="module")
def cuda(lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return lib


def assert_many_units(B, H, per_head=1):
    """The launch runs at least UNITS_PER_CTA units on every CTA."""
    import torch

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = B * H * per_head
    assert units >= UNITS_PER_CTA * CTAS_PER_SM * sms, (units, sms)


def _mamba2_gates(r, ckpt_dtype):
    if ckpt_dtype == "f32":
        assert r["o_exact"] <= par.TOL_F32 and r["ck_exact"] <= par.TOL_F32, r
    else:
        assert r["o_exact"] <= par.TOL_F16 and r["ck_exact"] <= par.TOL_F16, r
        assert r["o_replay"] <= par.TOL_F16_EMU and r["ck_replay"] <= par.TOL_F16_EMU, r
    assert r["flush_rows"] > 0, r


# --------------------------------------------------------------------------
# Mamba-2, one checkpoint copy
# --------------------------------------------------------------------------
@pytest.mark.parametrize("ckpt_dtype", ["f32", "f16"])
@pytest.mark.parametrize("L", [8, 16, 32, 64])
def test_mamba2_64x128_window_bounds(cuda, L, ckpt_dtype):
    # 80 rows x 32 heads = 2560 units; staggered cursors, padded rows and
    # permuted slots; every row flushes at least once
    B, H = 80, 32
    assert_many_units(B, H)
    w = synth.make_workload("mamba2_bs256", B=B, H=H, L=L, steps=L + 6, num_slots=88, permute_slots=True,
                            pad_rows=3, ckpt_dtype=ckpt_dtype, seed=400 + L)
    r = par.run_parity(cuda, w, w.steps, heads=[0, 17, 31])
    _mamba2_gates(r, ckpt_dtype)


@pytest.mark.parametrize("L", [8, 16])
def test_mamba2_fp16_odd_heads(cuda, L):
    # an odd head count (48 x 27 = 1296 units): no unit arithmetic may assume
    # heads come in pairs
    B, H = 48, 27
    assert_many_units(B, H)
    w = synth.make_workload("mamba2_bs256", B=B, H=H, L=L, steps=L + 6, pad_rows=2, ckpt_dtype="f16",
                            seed=470 + L)
    r = par.run_parity(cuda, w, w.steps, heads=[0, 13, 26])
    _mamba2_gates(r, "f16")


@pytest.mark.parametrize("ckpt_dtype", ["f32", "f16"])
@pytest.mark.parametrize("L", [16, 40])
def test_mamba2_128x128(cuda, L, ckpt_dtype):
    B, H = 40, 32
    assert_many_units(B, H)
    w = synth.make_workload("mamba2_bs256", B=B, H=H, d_v=128, d_k=128, L=L, steps=L + 4, pad_rows=2,
                            ckpt_dtype=ckpt_dtype, seed=410 + L)
    r = par.run_parity(cuda, w, w.steps, heads=[3, 30])
    _mamba2_gates(r, ckpt_dtype)


@pytest.mark.parametrize("in_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("ckpt_dtype", ["f32", "f16"])
@pytest.mark.parametrize("L", [16, 64])
def test_mamba2_16x32(cuda, L, ckpt_dtype, in_dtype):
    B, H = 24, 64
    assert_many_units(B, H)
    w = synth.make_workload("mamba2_bs256", B=B, H=H, d_v=16, d_k=32, L=L, steps=L + 4, pad_rows=1,
                            ckpt_dtype=ckpt_dtype, in_dtype=in_dtype, ring_dtype=in_dtype, seed=420 + L)
    r = par.run_parity(cuda, w, w.steps, heads=[0, 63])
    _mamba2_gates(r, ckpt_dtype)


@pytest.mark.parametrize("ckpt_dtype", ["f32", "f16"])
@pytest.mark.parametrize("d_v, L", [(64, 16), (64, 40), (128, 16)])
def test_mamba2_fp32_inputs(cuda, d_v, L, ckpt_dtype):
    B, H = 40, 32
    assert_many_units(B, H)
    w = synth.make_workload("mamba2_bs256", B=B, H=H, d_v=d_v, L=L, steps=L + 4, pad_rows=2, in_dtype="f32",
                            ring_dtype="f32", ckpt_dtype=ckpt_dtype, seed=430 + d_v + L)
    r = par.run_parity(cuda, w, w.steps, heads=[1, 29])
    _mamba2_gates(r, ckpt_dtype)


@pytest.mark.parametrize("ckpt_dtype", ["f32", "f16"])
def test_mamba2_bs512(cuda, ckpt_dtype):
    # batch 512 of the 128-head layer at L 16 (65 536 units): the largest batch
    # of the sweep; two heads of every row followed by the oracle
    w = synth.make_workload("mamba2_bs256", B=512, steps=20, ckpt_dtype=ckpt_dtype, seed=440)
    assert_many_units(w.B, w.H)
    r = par.run_parity(cuda, w, w.steps, heads=[9, 120])
    _mamba2_gates(r, ckpt_dtype)
    assert r["flush_rows"] >= 512


# --------------------------------------------------------------------------
# two-precision checkpoint
# --------------------------------------------------------------------------
@pytest.mark.parametrize("lp, d_v, d_k, H, L, in_dtype", [
    (lp, *shape) for lp in ("f16", "bf16") for shape in
    ((64, 128, 32, 16, "bf16"), (64, 128, 32, 32, "bf16"), (64, 128, 32, 16, "f32"), (128, 128, 32, 16, "bf16"),
     (16, 32, 64, 16, "bf16"))] + [
    ("e4m3", 64, 128, 32, 16, "bf16"), ("e4m3", 64, 128, 32, 32, "bf16"), ("e4m3", 64, 128, 32, 64, "bf16"),
    ("e4m3", 64, 128, 32, 16, "f32")])
def test_two_precision(cuda, lp, d_v, d_k, H, L, in_dtype):
    B = 40
    assert_many_units(B, H)
    w = synth.make_workload("mamba2_bs256", B=B, H=H, d_v=d_v, d_k=d_k, L=L, steps=L + 6, pad_rows=2,
                            in_dtype=in_dtype, ring_dtype=in_dtype, seed=450 + d_v + L)
    g, r = twop._run(cuda, w, lp, w.steps, heads=[2, H - 1])
    assert int(g.dev_err.item()) == 0
    assert r["n_lp"] > 0 and r["lp_exact"] >= twop.MIN_EXACT, r
    assert r["ck"] <= twop.TOL_F32 and r["excess"] <= twop.TOL_F32, r
    assert r["seen"] > 3 * twop.TOL_F32, r


# --------------------------------------------------------------------------
# group-shared keys
# --------------------------------------------------------------------------
@pytest.mark.parametrize("ckpt_dtype, L, d_v, d_k, H, G, in_dtype", [
    ("f32", 16, 64, 128, 32, 4, "bf16"),
    ("f32", 32, 64, 128, 32, 2, "bf16"),
    ("f16", 16, 64, 128, 32, 4, "bf16"),
    ("f16", 32, 64, 128, 32, 8, "bf16"),
    ("f32", 16, 64, 128, 32, 4, "f32"),
    ("f32", 16, 16, 32, 64, 8, "bf16"),
])
def test_grouped(cuda, ckpt_dtype, L, d_v, d_k, H, G, in_dtype):
    B = 40
    assert_many_units(B, H)
    w = synth.make_workload("mamba2_bs256", B=B, H=H, d_v=d_v, d_k=d_k, L=L, steps=L + 6, pad_rows=2,
                            num_slots=44, permute_slots=True, ckpt_dtype=ckpt_dtype, in_dtype=in_dtype,
                            ring_dtype=in_dtype, seed=470 + L + G)
    err, worst_o, worst_c, n_flush = grouped._run(cuda, w, G, w.steps, heads=[0, H // 2 + 1, H - 1])
    tol = par.TOL_F32 if ckpt_dtype == "f32" else par.TOL_F16
    assert err == 0 and n_flush > 0
    assert worst_o <= tol and worst_c <= tol, (worst_o, worst_c)


# --------------------------------------------------------------------------
# Gated DeltaNet
# --------------------------------------------------------------------------
@pytest.mark.parametrize("ckpt_dtype", ["f32", "f16"])
@pytest.mark.parametrize("L", [4, 16, 32])
def test_gdn_fp16_rings(cuda, L, ckpt_dtype):
    # 128 x 128 heads: an fp32 checkpoint is two units per head, fp16 one
    B, H = 40, 32
    assert_many_units(B, H)
    w = synth.make_workload("gdn_bs256", B=B, H=H, L=L, steps=L + 6, pad_rows=2, num_slots=45,
                            permute_slots=True, ckpt_dtype=ckpt_dtype, seed=490 + L)
    if ckpt_dtype == "f32":
        r = par.run_parity(cuda, w, w.steps, heads=[0, 31], exact=False)
        par.assert_gdn_f16_ring(r)
    else:
        r = par.run_parity(cuda, w, w.steps, heads=[0, 31])
        assert r["o_exact"] <= par.TOL_F16 and r["o_replay"] <= par.TOL_F16_EMU, r
    assert r["flush_rows"] > 0


@pytest.mark.parametrize("ckpt_dtype, d_v, in_dtype, L", [("f32", 128, "bf16", 32), ("f16", 128, "bf16", 16),
                                                         ("f32", 64, "bf16", 16), ("f32", 128, "f32", 16),
                                                         ("f16", 64, "f32", 32)])
def test_gdn_fp32_rings(cuda, ckpt_dtype, d_v, in_dtype, L):
    B, H = 40, 32
    assert_many_units(B, H)
    w = synth.make_workload("gdn_bs256", B=B, H=H, d_v=d_v, L=L, steps=L + 6, pad_rows=1, ring_dtype="f32",
                            in_dtype=in_dtype, ckpt_dtype=ckpt_dtype, seed=500 + d_v + L)
    r = par.run_parity(cuda, w, w.steps, heads=[4, 27])
    if ckpt_dtype == "f32":
        assert r["o_exact"] <= par.TOL_F32 and r["ck_exact"] <= par.TOL_F32, r
    else:
        assert r["o_exact"] <= par.TOL_F16 and r["o_replay"] <= par.TOL_F16_EMU, r
    assert r["flush_rows"] > 0


def test_gdn_bs256_fp32_rings_exact(cuda):
    # the batch-256 GDN layer (16 384 units) with fp32 d/k rings, so that its
    # arithmetic is held to the exact recurrence at 1e-4
    w = synth.make_workload("gdn_bs256", steps=40, ring_dtype="f32", seed=510)
    assert_many_units(w.B, w.H)
    r = par.run_parity(cuda, w, w.steps, heads=[0, 31])
    assert r["o_exact"] <= par.TOL_F32 and r["ck_exact"] <= par.TOL_F32, r
    assert r["flush_rows"] >= 256 * 2


# --------------------------------------------------------------------------
# speculative verification
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L, T", [(16, 1), (16, 2), (16, 8), (32, 8), (32, 16), (64, 16)])
def test_spec_verify(cuda, L, T):
    B, H = 40, 32
    assert_many_units(B, H)
    w = synth.make_workload("mamba2_bs256", B=B, H=H, L=L, steps=1, pad_rows=2, num_slots=48,
                            permute_slots=True, seed=520 + L + T)
    err, worst_o, worst_c, n_flush = spec._run(cuda, w, T, max(12, 2 * L // T + 4), heads=[5, 30], seed=L + T)
    assert err == 0 and n_flush > 0
    assert worst_o <= spec.TOL and worst_c <= spec.TOL, (worst_o, worst_c)


@pytest.mark.parametrize("T", [4, 8])
def test_spec_verify_fp16_checkpoint(cuda, T):
    # against the exact recurrence at the fp16-checkpoint gate
    B, H = 40, 32
    assert_many_units(B, H)
    w = synth.make_workload("mamba2_bs256", B=B, H=H, steps=1, pad_rows=1, ckpt_dtype="f16", seed=540 + T)
    err, worst_o, worst_c, n_flush = spec._run(cuda, w, T, 12, heads=[0, 31], seed=T)
    assert err == 0 and n_flush > 0
    assert worst_o <= par.TOL_F16 and worst_c <= par.TOL_F16, (worst_o, worst_c)


@pytest.mark.parametrize("d_v, d_k, H, in_dtype, T", [(128, 128, 32, "bf16", 4), (64, 128, 32, "f32", 8),
                                                     (16, 32, 64, "bf16", 4), (128, 128, 32, "bf16", 16)])
def test_spec_verify_other_shapes(cuda, d_v, d_k, H, in_dtype, T):
    # the CUDA-core verification kernel: 128 x 128 and 16 x 32 heads, fp32 drafts
    B = 40
    assert_many_units(B, H)
    w = synth.make_workload("mamba2_bs256", B=B, H=H, d_v=d_v, d_k=d_k, L=16, steps=1, pad_rows=1,
                            in_dtype=in_dtype, ring_dtype=in_dtype, seed=560 + d_v + T)
    err, worst_o, worst_c, n_flush = spec._run(cuda, w, T, 12, heads=[1, H - 2], seed=T)
    assert err == 0 and n_flush > 0
    assert worst_o <= spec.TOL and worst_c <= spec.TOL, (worst_o, worst_c)
