"""replayssm_decode_mamba2_noalloc: the group-shared-key decode for callers
that cannot allocate device memory (a plugin of a serving engine that owns all
device memory through its own pool, or a decode loop that must not call
cudaMalloc because it can synchronise the device).  The group dots go to a
fixed-size device array held by the library instead of caller scratch.

Host checks (no GPU): the call refuses a caller scratch and batches whose
dots would not fit the library's array, before touching the device.  GPU
check: on forty calls in a row, each call's outputs, and the checkpoints at
the end, are bit-identical to those of replayssm_decode_mamba2 given caller
scratch on the same inputs, and match the exact recurrence at max relative
error 1e-4.  This file is collected last, so a run that stops at its first
failure has run every other test before it.
"""

import numpy as np
import pytest

import oracle
from linear_attention_decode_replayssm_gb300 import synth
from tests._harness import dev, tdt
from tests._util import rel_err


def _args(lib, **kw):
    a = lib.StepArgs()
    base = dict(B=4, H=4, d_v=64, d_k=128, L=16, num_slots=8, ckpt_dtype=lib.RS_F32, in_dtype=lib.RS_BF16,
                ring_dtype=lib.RS_BF16, reserved=0, slot_idx=0x1000, write_pos=0x2000, is_flush=0x3000,
                v=0x4000, k=0x5000, q=0x6000, alpha=0x7000, beta=None, ckpt=0x9000, ring_v=0xA000,
                ring_k=0xB000, ring_a=0xC000, out=0xD000, stride_v_row=4 * 64, stride_k_row=2 * 128,
                stride_q_row=2 * 128, stride_out_row=4 * 64, dev_err=None, n_groups=2, kq_scratch=None)
    base.update(kw)
    for k_, v_ in base.items():
        setattr(a, k_, v_)
    return a


def test_noalloc_refuses_caller_scratch_and_oversize(lib):
    assert lib.raw_call("replayssm_decode_mamba2_noalloc", _args(lib, kq_scratch=0xF000), None) == lib.RS_EINVAL
    too_many = lib.RS_NOALLOC_KQ_FLOATS // (2 * 16) + 1  # rows whose group dots would not fit
    big = _args(lib, B=too_many)
    assert lib.raw_call("replayssm_decode_mamba2_noalloc", big, None) == lib.RS_EINVAL
    assert lib.raw_call("replayssm_decode_mamba2_noalloc", _args(lib, B=0), None) == lib.RS_OK
    # without groups it is the plain entry point (same validation)
    assert lib.raw_call("replayssm_decode_mamba2_noalloc", _args(lib, n_groups=0, L=1), None) == lib.RS_EINVAL


@pytest.mark.gpu
def test_noalloc_matches_caller_scratch_and_oracle(lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B, H, G, steps = 9, 8, 2, 40
    w = synth.make_workload("mamba2_bs256", B=B, H=H, steps=steps, seed=77, pad_rows=1)
    L, td = w.L, tdt(w.in_dtype)
    r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 1])))
    held = w.held_records()
    ring_kg = np.full((w.num_slots, G, L, w.d_k), np.nan, dtype=np.float32)
    for s in range(w.num_slots):
        if held[s]:
            x = r.standard_normal((G, held[s], w.d_k), dtype=np.float32) / np.sqrt(np.float32(w.d_k))
            ring_kg[s, :, : held[s]] = synth.quantize(x, w.ring_dtype)
    sides = []
    for _ in range(2):
        sides.append(dict(ckpt=dev(w.ckpt0, torch.float32), ring_v=dev(w.ring_v0, td), ring_k=dev(ring_kg, td),
                          ring_a=dev(w.ring_a0, torch.float32), out=torch.empty(B, H, w.d_v, device="cuda")))
    slot_idx = dev(w.slot_idx, torch.int32)
    kq = torch.empty(B * G * L, device="cuda")
    err = torch.zeros(1, device="cuda", dtype=torch.int32)
    to_heads = lambda x: np.moveaxis(oracle.heads_from_groups(np.moveaxis(x, 1, -2), H), -2, 1)
    rs = oracle.ReplayState("mamba2", w.ckpt0.astype(np.float64), w.ring_v0.astype(np.float64),
                            np.stack([to_heads(ring_kg[s][None])[0] for s in range(w.num_slots)]).astype(np.float64),
                            w.ring_a0.astype(np.float64))
    ex = oracle.ExactState.from_replay(rs, held)
    live = w.slot_idx >= 0
    worst = 0.0
    for t in range(steps):
        wp, fl = lib.replayssm_plan_step(w.decode_step(t), L)
        wp_d, fl_d = dev(wp, torch.int32), dev(fl, torch.uint8)
        x = w.inputs(t)
        kg = synth.quantize(r.standard_normal((B, G, w.d_k), dtype=np.float32) / np.sqrt(np.float32(w.d_k)), "bf16")
        qg = synth.quantize(r.standard_normal((B, G, w.d_k), dtype=np.float32) / np.sqrt(np.float32(w.d_k)), "bf16")
        common = dict(slot_idx=slot_idx, write_pos=wp_d, is_flush=fl_d, v=dev(x["v"], td), k=dev(kg, td),
                      q=dev(qg, td), alpha=dev(x["alpha"], torch.float32), dev_err=err)
        a, b = sides
        lib.replayssm_decode_mamba2(ckpt=a["ckpt"], ring_v=a["ring_v"], ring_k=a["ring_k"], ring_a=a["ring_a"],
                                    out=a["out"], kq_scratch=kq, **common)
        lib.replayssm_decode_mamba2_noalloc(ckpt=b["ckpt"], ring_v=b["ring_v"], ring_k=b["ring_k"],
                                            ring_a=b["ring_a"], out=b["out"], **common)
        assert torch.equal(a["out"].view(torch.int32), b["out"].view(torch.int32))
        o_e = oracle.exact_step(ex, w.slot_idx, x["v"], to_heads(kg), to_heads(qg), x["alpha"])
        worst = max(worst, rel_err(b["out"].double().cpu().numpy()[live], o_e[live]))
    assert torch.equal(sides[0]["ckpt"].view(torch.int32), sides[1]["ckpt"].view(torch.int32))
    assert int(err.item()) == 0
    assert worst <= 1e-4, worst
