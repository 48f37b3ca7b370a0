"""Seeded synthetic workloads for the ReplaySSM decode step.

This module only draws numbers: it holds none of the decode step's arithmetic,
so both the CUDA path and the CPU oracle can take their inputs from it.
Arrays come back as NumPy float32 (or int) arrays whose values are exactly
representable in the storage type they are tagged with, so converting them to
a bf16 / fp16 tensor, or to float64 for the oracle, is exact.

The pages evaluate on real models and datasets that are not available here;
these generators stand in for them at the pages' layer shapes:

* Mamba-2 layer of Nemotron-3-Super: 128 heads, d_v = 64, d_k = 128, fp32
  state (4 MiB per row), buffer length L = 16 ("ReplaySSM: an SSM decoder that
  writes its state once every 16 tokens", §Why a fixed-size state is not cheap
  to decode).
* Gated DeltaNet layer: 32 value heads of 128 x 128, fp16 d/k caches and an
  fp32 g cache ("[Kernel] ReplaySSM: cache SSM inputs for faster Gated DeltaNet
  standard decode", §Paged cache layout).

Distributions (the pages are silent; these are the stated recipe):
  Mamba-2  v, k, q ~ N(0, 1) / sqrt(d_k); alpha = sigmoid(N(mu, sd)).
  GDN      q, k ~ N(0, 1), L2-normalised in fp32; v ~ N(0, 1) / sqrt(d_k);
           beta = sigmoid(N(0, 1)); g = log(sigmoid(N(3, 1))).
  Starting checkpoint ~ N(0, 1) / sqrt(d_k) in its storage type (or zero), and
  a row whose cursor starts at p holds p earlier records drawn from the same
  input laws (for GDN the stored corrected value d ~ N(0, 1) / sqrt(d_k)).
  Ring slots a row does not hold are filled with NaN, so that reading a stale
  record anywhere shows up in the outputs.
"""

from dataclasses import dataclass, field

import numpy as np

# storage type tags shared with the binding
DTYPES = ("f32", "f16", "bf16")


def _rng(seed, *stream):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def quantize(x, dtype):
    """Round float32/float64 values to ``dtype`` (round to nearest even) and
    return them as float32.  Input quantisation of synthetic data only."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f32":
        return x.copy()
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float32)
    if dtype == "bf16":
        import torch

        return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float32).numpy()
    raise ValueError(dtype)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-np.asarray(x, dtype=np.float64)))


def _l2norm(x):
    x = np.asarray(x, dtype=np.float32)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))


SPECS = {
    # tiny Mamba-2 case the oracle runs in well under a second
    "tiny": dict(variant="mamba2", B=2, H=2, d_v=16, d_k=32, L=4, steps=64,
                 ckpt_dtype="f32", in_dtype="f32", ring_dtype="f32",
                 alpha_mu=2.0, alpha_sd=0.5, stagger=False, zero_ckpt=True),
    # one Mamba-2 layer at Nemotron-3-Super shapes, batch 256, staggered cursors
    "mamba2_bs256": dict(variant="mamba2", B=256, H=128, d_v=64, d_k=128, L=16, steps=256,
                         ckpt_dtype="f32", in_dtype="bf16", ring_dtype="bf16",
                         alpha_mu=3.0, alpha_sd=1.0, stagger=True, zero_ckpt=False),
    # one Gated DeltaNet layer, batch 256, 32 value heads of 128 x 128
    "gdn_bs256": dict(variant="gdn", B=256, H=32, d_v=128, d_k=128, L=16, steps=256,
                      ckpt_dtype="f32", in_dtype="bf16", ring_dtype="f16",
                      alpha_mu=3.0, alpha_sd=1.0, stagger=True, zero_ckpt=False),
}


@dataclass
class Workload:
    variant: str
    B: int
    H: int
    d_v: int
    d_k: int
    L: int
    steps: int
    ckpt_dtype: str
    in_dtype: str
    ring_dtype: str
    alpha_mu: float
    alpha_sd: float
    stagger: bool
    zero_ckpt: bool
    seed: int = 0
    num_slots: int = 0
    pad_rows: int = 0          # rows (chosen at random) whose slot is -1
    permute_slots: bool = False
    cursor0: np.ndarray = None  # optional starting decode steps [B] (else drawn)
    # filled by build()
    slot_idx: np.ndarray = field(default=None, repr=False)
    decode_step0: np.ndarray = field(default=None, repr=False)
    ckpt0: np.ndarray = field(default=None, repr=False)
    ring_v0: np.ndarray = field(default=None, repr=False)
    ring_k0: np.ndarray = field(default=None, repr=False)
    ring_a0: np.ndarray = field(default=None, repr=False)

    # -- starting state ---------------------------------------------------
    def build(self):
        if self.num_slots <= 0:
            self.num_slots = self.B
        if self.num_slots < self.B:
            raise ValueError("num_slots must be >= B")
        r = _rng(self.seed, 0)
        S, H, L = self.num_slots, self.H, self.L
        slots = r.permutation(S)[: self.B] if self.permute_slots else np.arange(self.B)
        slots = slots.astype(np.int32)
        if self.pad_rows:
            slots[r.choice(self.B, self.pad_rows, replace=False)] = -1
        self.slot_idx = slots
        if self.cursor0 is not None:
            self.decode_step0 = np.asarray(self.cursor0, dtype=np.int64).copy()
        elif self.stagger:
            self.decode_step0 = r.integers(0, self.L, size=self.B).astype(np.int64)
        else:
            self.decode_step0 = np.zeros(self.B, dtype=np.int64)
        if self.zero_ckpt:
            self.ckpt0 = np.zeros((S, H, self.d_v, self.d_k), dtype=np.float32)
        else:
            self.ckpt0 = self.fresh_checkpoint(r, S)
        nan = np.float32(np.nan)
        self.ring_v0 = np.full((S, H, L, self.d_v), nan, dtype=np.float32)
        self.ring_k0 = np.full((S, H, L, self.d_k), nan, dtype=np.float32)
        self.ring_a0 = np.full((S, H, L), nan, dtype=np.float32)
        for b in range(self.B):
            s = slots[b]
            p = int(self.decode_step0[b] % L)
            if s < 0 or p == 0:
                continue
            rec = self._records(r, p)
            self.ring_v0[s, :, :p] = rec["v"]
            self.ring_k0[s, :, :p] = rec["k"]
            self.ring_a0[s, :, :p] = rec["a"]
        return self

    def fresh_checkpoint(self, r, n):
        x = r.standard_normal((n, self.H, self.d_v, self.d_k), dtype=np.float32)
        return quantize(x / np.sqrt(np.float32(self.d_k)), self.ckpt_dtype)

    def _records(self, r, p):
        """p earlier ring records per head, [H, p, d] (already in ring type)."""
        H = self.H
        if self.variant == "mamba2":
            v = r.standard_normal((H, p, self.d_v), dtype=np.float32) / np.sqrt(np.float32(self.d_k))
            k = r.standard_normal((H, p, self.d_k), dtype=np.float32) / np.sqrt(np.float32(self.d_k))
            a = _sigmoid(r.normal(self.alpha_mu, self.alpha_sd, size=(H, p))).astype(np.float32)
        else:
            v = r.standard_normal((H, p, self.d_v), dtype=np.float32) / np.sqrt(np.float32(self.d_k))
            k = _l2norm(r.standard_normal((H, p, self.d_k), dtype=np.float32))
            a = np.log(_sigmoid(r.normal(self.alpha_mu, self.alpha_sd, size=(H, p)))).astype(np.float32)
        return dict(v=quantize(v, self.ring_dtype), k=quantize(k, self.ring_dtype), a=a)

    # -- per-step inputs ----------------------------------------------------
    def inputs(self, t):
        """Inputs of decode step ``t`` (independent stream per step).

        Returns dict with v [B,H,d_v], k, q [B,H,d_k] (values of ``in_dtype``),
        alpha [B,H] float32 (decay for Mamba-2, log-gate g for GDN) and, for
        GDN, beta [B,H] float32.
        """
        r = _rng(self.seed, 1000 + t)
        B, H = self.B, self.H
        sk = np.sqrt(np.float32(self.d_k))
        if self.variant == "mamba2":
            v = r.standard_normal((B, H, self.d_v), dtype=np.float32) / sk
            k = r.standard_normal((B, H, self.d_k), dtype=np.float32) / sk
            q = r.standard_normal((B, H, self.d_k), dtype=np.float32) / sk
            a = _sigmoid(r.normal(self.alpha_mu, self.alpha_sd, size=(B, H))).astype(np.float32)
            out = dict(alpha=a)
        else:
            q = _l2norm(r.standard_normal((B, H, self.d_k), dtype=np.float32))
            k = _l2norm(r.standard_normal((B, H, self.d_k), dtype=np.float32))
            v = r.standard_normal((B, H, self.d_v), dtype=np.float32) / sk
            beta = _sigmoid(r.standard_normal((B, H))).astype(np.float32)
            g = np.log(_sigmoid(r.normal(self.alpha_mu, self.alpha_sd, size=(B, H)))).astype(np.float32)
            out = dict(alpha=g, beta=beta)
        out.update(v=quantize(v, self.in_dtype), k=quantize(k, self.in_dtype), q=quantize(q, self.in_dtype))
        return out

    def decode_step(self, t):
        """Per-row decode step counter at step t (no churn)."""
        return self.decode_step0 + t

    def held_records(self):
        """Records each slot holds at the start: decode_step0 mod L (0 for
        slots no row uses)."""
        held = np.zeros(self.num_slots, dtype=np.int64)
        for b in range(self.B):
            if self.slot_idx[b] >= 0:
                held[self.slot_idx[b]] = self.decode_step0[b] % self.L
        return held


def make_workload(name, seed=0, **overrides):
    """A built ``Workload`` from a named spec with optional field overrides."""
    spec = dict(SPECS[name])
    spec.update(overrides)
    return Workload(seed=seed, **spec).build()


# ---------------------------------------------------------------------------
# continuous batching: rows leave and new requests take their slots
# ---------------------------------------------------------------------------
class ChurnSchedule:
    """Per-row decode-step counters under continuous batching.

    Every ``period`` steps each row, at its own random offset, finishes with
    probability ``p_churn``; a new request takes the same batch position and
    slot at decode step 0 with a fresh checkpoint (stand-in for its prefill
    state).  The slot's ring is left as it was: the cursor restarts at 0, so
    no stale record is ever read ("[Kernel] ReplaySSM: cache SSM inputs for
    faster Gated DeltaNet standard decode", §CUDA graphs and continuous
    batching: recycled blocks need no zero-init).
    """

    def __init__(self, B, L, steps, period=8, p_churn=0.25, seed=0, decode_step0=None):
        r = _rng(seed, 7)
        self.B, self.L, self.steps = B, L, steps
        self.offset = r.integers(0, period, size=B)
        churn = np.zeros((steps, B), dtype=bool)
        for t in range(1, steps):
            due = (t % period) == self.offset
            churn[t] = due & (r.random(B) < p_churn)
        self.join = churn  # [steps, B]: a new request starts at this step
        ds = np.empty((steps, B), dtype=np.int64)
        cur = np.zeros(B, dtype=np.int64) if decode_step0 is None else np.asarray(decode_step0, dtype=np.int64).copy()
        for t in range(steps):
            cur = np.where(churn[t], 0, cur)
            ds[t] = cur
            cur = cur + 1
        self.decode_steps = ds  # [steps, B]

    def decode_step(self, t):
        return self.decode_steps[t]

    def joins(self, t):
        return np.nonzero(self.join[t])[0]


# ---------------------------------------------------------------------------
# the same laws drawn on a CUDA device (for GiB-sized workloads)
# ---------------------------------------------------------------------------
def device_draw(shape, law, generator, device="cuda", d_k=None):
    """Draw a float32 tensor on the device from one of the input laws:
    'scaled' N(0,1)/sqrt(d_k), 'unit' N(0,1) L2-normalised over the last axis,
    'sigmoid3' sigmoid(N(3,1)), 'logsigmoid3' log(sigmoid(N(3,1))),
    'sigmoid0' sigmoid(N(0,1))."""
    import torch

    x = torch.randn(*shape, generator=generator, device=device, dtype=torch.float32)
    if law == "scaled":
        return x / float(np.sqrt(d_k))
    if law == "unit":
        return x / x.norm(dim=-1, keepdim=True)
    if law == "sigmoid3":
        return torch.sigmoid(x + 3.0)
    if law == "logsigmoid3":
        return torch.log(torch.sigmoid(x + 3.0))
    if law == "sigmoid0":
        return torch.sigmoid(x)
    raise ValueError(law)
