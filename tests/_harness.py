"""Drivers that run one workload on the GPU (through the C ABI) and in the oracle.

Both sides take the same seeded inputs from ``synth``; nothing computed on
the GPU ever feeds the oracle.
"""

import numpy as np

import oracle

TORCH_DTYPES = {}


def tdt(name):
    import torch

    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}[name]


def dev(a, dtype, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


class GpuRun:
    """ReplaySSM (or conventional) state on the GPU, stepped through the C ABI."""

    def __init__(self, lib, w, conventional=False, ckpt0=None, lp_dtype=None):
        import torch

        self.lib, self.w, self.conventional = lib, w, conventional
        self.ckpt = dev(w.ckpt0 if ckpt0 is None else ckpt0, tdt(w.ckpt_dtype))
        # two-precision checkpoint: the read copy starts as the library's cast
        # of the checkpoint (RN-even; E4M3 on a power-of-two scale per row)
        self.ckpt_lp = self.ckpt_lp_scale = None
        if lp_dtype is not None:
            self.ckpt_lp = torch.empty(self.ckpt.shape, device="cuda", dtype=tdt(lp_dtype))
            if lp_dtype == "e4m3":
                self.ckpt_lp_scale = torch.empty(self.ckpt.shape[:3], device="cuda", dtype=torch.float32)
            lib.replayssm_seed_read_copy(ckpt=self.ckpt, ckpt_lp=self.ckpt_lp, scale=self.ckpt_lp_scale)
        self.ring_v = dev(w.ring_v0, tdt(w.ring_dtype))
        self.ring_k = dev(w.ring_k0, tdt(w.ring_dtype))
        self.ring_a = dev(w.ring_a0, torch.float32)
        self.slot_idx = dev(w.slot_idx, torch.int32)
        self.out = torch.empty(w.B, w.H, w.d_v, device="cuda", dtype=torch.float32)
        self.wp = torch.empty(w.B, device="cuda", dtype=torch.int32)
        self.fl = torch.empty(w.B, device="cuda", dtype=torch.uint8)
        self.dev_err = torch.zeros(1, device="cuda", dtype=torch.int32)

    def read_copy(self, slots, heads):
        """The read copy of the given slots and heads as float64 values (an
        E4M3 copy's codes times its row scales)."""
        import torch

        sl = torch.as_tensor(np.asarray(slots), device="cuda")
        hs = torch.as_tensor(np.asarray(heads), device="cuda")
        x = self.ckpt_lp[sl][:, hs].double()
        if self.ckpt_lp_scale is not None:
            x = x * self.ckpt_lp_scale[sl][:, hs].double()[..., None]
        return x.cpu().numpy()

    def tensors(self, x):
        import torch

        w = self.w
        t = {n: dev(x[n], tdt(w.in_dtype)) for n in ("v", "k", "q")}
        t["alpha"] = dev(x["alpha"], torch.float32)
        t["beta"] = dev(x["beta"], torch.float32) if "beta" in x else None
        return t

    def step(self, x, decode_step, out=None, plan=None, **override):
        """One step; returns (o on host as float64, write_pos, is_flush).
        ``plan`` = (write_pos, is_flush) from another host plan (align mode)
        replaces the plan of ``decode_step``."""
        w, lib = self.w, self.lib
        wp, fl = lib.replayssm_plan_step(decode_step, w.L) if plan is None else plan
        self.wp.copy_(dev(wp, self.wp.dtype))
        self.fl.copy_(dev(fl, self.fl.dtype))
        t = self.tensors(x)
        t.update(override)
        out = self.out if out is None else out
        if self.conventional:
            lib.conventional_decode(variant=lib.RS_GDN if w.variant == "gdn" else lib.RS_MAMBA2,
                                    state=self.ckpt, slot_idx=self.slot_idx, v=t["v"], k=t["k"], q=t["q"],
                                    alpha=t["alpha"], beta=t["beta"], out=out, dev_err=self.dev_err)
        elif w.variant == "mamba2":
            lib.replayssm_decode_mamba2(ckpt=self.ckpt, ring_v=self.ring_v, ring_k=self.ring_k,
                                        ring_a=self.ring_a, slot_idx=self.slot_idx, write_pos=self.wp,
                                        is_flush=self.fl, v=t["v"], k=t["k"], q=t["q"], alpha=t["alpha"],
                                        out=out, dev_err=self.dev_err, ckpt_lp=self.ckpt_lp,
                                        ckpt_lp_scale=self.ckpt_lp_scale)
        else:
            lib.replayssm_decode_gdn(ckpt=self.ckpt, ring_v=self.ring_v, ring_k=self.ring_k, ring_a=self.ring_a,
                                     slot_idx=self.slot_idx, write_pos=self.wp, is_flush=self.fl, v=t["v"],
                                     k=t["k"], q=t["q"], alpha=t["alpha"], beta=t["beta"], out=out,
                                     dev_err=self.dev_err)
        return out.double().cpu().numpy(), wp, fl


class OracleRun:
    """The oracle on the same workload, optionally on a subset of heads."""

    def __init__(self, w, heads=None, replay=True, exact=True, exact_state_dtype="f64", ckpt0=None,
                 lp_dtype=None):
        self.w = w
        self.heads = np.arange(w.H) if heads is None else np.asarray(heads)
        hs = self.heads
        c0 = w.ckpt0 if ckpt0 is None else ckpt0
        rs = oracle.ReplayState(w.variant, c0[:, hs].astype(np.float64), w.ring_v0[:, hs].astype(np.float64),
                                w.ring_k0[:, hs].astype(np.float64), w.ring_a0[:, hs].astype(np.float64),
                                ckpt_dtype=w.ckpt_dtype, ring_dtype=w.ring_dtype, a_dtype="f32")
        if lp_dtype is not None:
            rs.with_read_copy(lp_dtype)
        self.rs = rs if replay else None
        self.ex = oracle.ExactState.from_replay(rs, w.held_records(), exact_state_dtype) if exact else None

    def sub(self, x):
        hs = self.heads
        return {n: np.asarray(a)[:, hs] for n, a in x.items()}

    def step(self, x, write_pos, is_flush):
        x = self.sub(x)
        args = (x["v"], x["k"], x["q"], x["alpha"], x.get("beta"))
        o_r = oracle.replay_step(self.rs, self.w.slot_idx, write_pos, is_flush, *args) if self.rs else None
        o_e = oracle.exact_step(self.ex, self.w.slot_idx, *args) if self.ex else None
        return o_r, o_e
