"""Batched decode steps over paged per-slot state (oracle; test infrastructure only).

Two references for one decode step of a batch of rows, each row owning one
slot of a paged pool ([PR48792] §Design notes / Paged cache layout: the
checkpoint and the ring caches live in the per-request paged state block,
indexed by the block table; null-padded slots are allowed, §Tests):

``exact_step``   the conventional recurrence on a float64 state per slot, with
                 no storage rounding (``state_dtype="f64"``), or with the state
                 rounded to its storage type after every step, which is what a
                 conventional load-update-store kernel with that state type
                 does (``state_dtype="f32"`` / ``"f16"``).

``replay_step``  the method's own bookkeeping: a checkpoint plus a ring of the
                 records since it, float64 arithmetic, and the storage
                 roundings the method performs at the points it stores data
                 (checkpoint cast at a flush; ring records cast on append).
                 Each row rebuilds its previous state from the checkpoint and
                 the ring ([Ghana] §The identity), takes the conventional step
                 from it, and then either appends the new record (non-flush) or
                 stores the new state as the checkpoint (flush) ([Ghana]
                 §The identity: "When the buffer holds L records, a flush step
                 folds them into the checkpoint, writes the checkpoint once,
                 and empties the buffer"; [PR48792] §Core concept).  This is
                 the state-reconstruction route; the output-only route gives
                 the same numbers up to rounding order ([Ghana] §Output without
                 a state; [PR48792] review comment on S_{t-1} q_t and
                 S_{t-1} k_t).

Two-precision checkpoint ([Ghana] §The precision argument, derived): a
Mamba-2 ``ReplayState`` may carry a low-precision read copy ``ckpt_lp``.
Non-flush steps start from the read copy; a flush starts from the recurrence
copy ``ckpt`` and casts its unrounded result into both copies.  (Gated
DeltaNet is left out: there the pages' flush recomputes the corrected values
from raw cached v, a ring this layout does not keep.)

Readings taken where the pages leave a step open:
  * The current token is record h = p + 1 of its window, where p = write_pos
    is the number of records already in the ring.  A flush folds those p
    records plus the current token and writes no ring record; the next step
    sees an empty ring (write_pos 0).
  * The flush output is S_new q_t from the unrounded new state; the stored
    checkpoint is a separate rounding of the same matrix ([Ghana] §The
    precision argument, derived: both copies are cast "from the same unrounded
    matrix").
  * Delta rule: the current step uses its own unrounded corrected value d_t
    (for its output and for a flush fold); the ring stores d_t and k_t rounded
    to the ring type, and later steps read the rounded values ([PR48792]
    §Paged cache layout: fp16 d and k caches, fp32 g cache).
  * A padded row (slot < 0) touches no state and outputs zeros.

Parity: pinned.  With every storage type float64, ``replay_step`` equals
``exact_step`` to 1e-12 over multi-window runs with staggered cursors, padded
rows and recycled slots (``tests/test_oracle_pins.py``); ``exact_step`` is
pinned through ``mamba2_step`` / ``gdn_step``.
"""

from dataclasses import dataclass

import numpy as np

from .recurrence import (
    gdn_corrected_value,
    gdn_step,
    gdn_unroll,
    mamba2_step,
    unroll,
)
from .storage import round_read_copy, round_to

VARIANTS = ("mamba2", "gdn")


@dataclass
class ExactState:
    """Conventional state per slot: S [num_slots, H, d_v, d_k] as float64."""

    variant: str
    S: np.ndarray
    state_dtype: str = "f64"

    @classmethod
    def from_replay(cls, rs, held, state_dtype="f64"):
        """Exact state equal to a ReplayState whose slot s holds ``held[s]``
        ring records: the unroll of the checkpoint and those records."""
        S = np.empty_like(rs.ckpt)
        for s in range(rs.ckpt.shape[0]):
            p = int(held[s])
            rebuild = unroll if rs.variant == "mamba2" else gdn_unroll
            S[s] = rebuild(rs.ckpt[s], rs.ring_a[s, :, :p], rs.ring_v[s, :, :p], rs.ring_k[s, :, :p])
        return cls(rs.variant, S, state_dtype)

    def reset_slot(self, s, S0):
        self.S[s] = np.asarray(S0, dtype=np.float64)


@dataclass
class ReplayState:
    """Checkpoint and ring per slot, values held as float64.

    ckpt   [num_slots, H, d_v, d_k]   checkpoint, values of ``ckpt_dtype``
    ring_v [num_slots, H, L, d_v]     v records (Mamba-2) / corrected d (GDN)
    ring_k [num_slots, H, L, d_k]     key records
    ring_a [num_slots, H, L]          alpha (Mamba-2) / log-gate g (GDN), fp32
    """

    variant: str
    ckpt: np.ndarray
    ring_v: np.ndarray
    ring_k: np.ndarray
    ring_a: np.ndarray
    ckpt_dtype: str = "f64"
    ring_dtype: str = "f64"
    a_dtype: str = "f32"
    # two-precision checkpoint (Mamba-2): a low-precision read copy
    ckpt_lp: np.ndarray = None
    lp_dtype: str = None

    @property
    def L(self):
        return self.ring_a.shape[2]

    def with_read_copy(self, lp_dtype):
        """Add the low-precision read copy of the two-precision checkpoint
        ([Ghana] §The precision argument, derived): the copy is cast from the
        same values as the recurrence copy (here: the starting checkpoint).
        ``lp_dtype`` fp16 or bf16, or e4m3 on a power-of-two scale per state
        row (``storage.round_read_copy``)."""
        if self.variant != "mamba2":
            raise NotImplementedError("two-precision checkpoint: Mamba-2 only")
        self.lp_dtype = lp_dtype
        self.ckpt_lp = round_read_copy(self.ckpt, lp_dtype)
        return self

    def reset_slot(self, s, ckpt0):
        """A new request takes slot s: fresh checkpoint, ring left as it was
        ([PR48792] §CUDA graphs and continuous batching: the cursor is derived
        from decode_step mod L, so recycled blocks need no zero-init)."""
        self.ckpt[s] = np.asarray(ckpt0, dtype=np.float64)
        if self.ckpt_lp is not None:
            self.ckpt_lp[s] = round_read_copy(ckpt0, self.lp_dtype)


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def exact_step(st, slot_idx, v, k, q, alpha, beta=None):
    """One conventional decode step of a batch, in place on ``st.S``.

    v [B, H, d_v]; k, q [B, H, d_k]; alpha [B, H] is the decay (Mamba-2) or
    the log-gate g (GDN); beta [B, H] for GDN.  Returns o [B, H, d_v].
    """
    v, k, q, alpha, beta = map(_f64, (v, k, q, alpha, beta))
    B, H = alpha.shape
    o = np.zeros((B, H, st.S.shape[2]))
    for b in range(B):
        s = int(slot_idx[b])
        if s < 0:
            continue
        if st.variant == "mamba2":
            S_new, o[b] = mamba2_step(st.S[s], alpha[b], v[b], k[b], q[b])
        else:
            S_new, o[b] = gdn_step(st.S[s], alpha[b], beta[b], v[b], k[b], q[b])
        st.S[s] = round_to(S_new, st.state_dtype)
    return o


def replay_step(st, slot_idx, write_pos, is_flush, v, k, q, alpha, beta=None):
    """One ReplaySSM decode step of a batch, in place on ``st``.

    Arguments as ``exact_step`` plus the per-row cursor ``write_pos`` [B] and
    flag ``is_flush`` [B] (``oracle.plan.plan_step``).  Returns o [B, H, d_v].
    """
    v, k, q, alpha, beta = map(_f64, (v, k, q, alpha, beta))
    B, H = alpha.shape
    o = np.zeros((B, H, st.ring_v.shape[3]))
    for b in range(B):
        s = int(slot_idx[b])
        if s < 0:
            continue
        p = int(write_pos[b])
        if not 0 <= p < st.L:
            raise ValueError(f"row {b}: write_pos {p} outside [0, {st.L})")
        recs = (st.ring_a[s, :, :p], st.ring_v[s, :, :p], st.ring_k[s, :, :p])
        if st.variant == "mamba2":
            # two-precision checkpoint: a non-flush step only reads, so it
            # starts from the read copy; a flush starts from the recurrence copy
            base = st.ckpt[s] if (st.ckpt_lp is None or is_flush[b]) else st.ckpt_lp[s]
            S_prev = unroll(base, *recs)
            S_t, o[b] = mamba2_step(S_prev, alpha[b], v[b], k[b], q[b])
            new_v = v[b]
        else:
            S_prev = gdn_unroll(st.ckpt[s], *recs)
            new_v = gdn_corrected_value(S_prev, alpha[b], beta[b], v[b], k[b])
            S_t, o[b] = gdn_step(S_prev, alpha[b], beta[b], v[b], k[b], q[b])
        if is_flush[b]:
            st.ckpt[s] = round_to(S_t, st.ckpt_dtype)
            if st.ckpt_lp is not None:  # both copies cast from the same unrounded matrix
                st.ckpt_lp[s] = round_read_copy(S_t, st.lp_dtype)
        else:
            st.ring_v[s, :, p] = round_to(new_v, st.ring_dtype)
            st.ring_k[s, :, p] = round_to(k[b], st.ring_dtype)
            st.ring_a[s, :, p] = round_to(alpha[b], st.a_dtype)
    return o


def materialize(rs, slot_idx, held, dst_dtype="f64"):
    """Exact state of each row from its checkpoint and held records, without
    touching either: what a prefix cache stores for a block boundary that did
    not fall on a flush ([Ghana] §What actually shipped: a cached prefix needs
    the exact state at a block boundary, and FlashInfer added a separate
    materialisation kernel for it).

    slot_idx [B] source slot (negative: row skipped, result left zero);
    held [B] records the slot's ring holds (the cursor its next step would
    get).  The state is the window unroll ([Ghana] §The identity; delta rule:
    the (d, k, g) unroll) rounded once to ``dst_dtype``.
    Returns S [B, H, d_v, d_k] float64.

    Parity: pinned through ``unroll`` / ``gdn_unroll`` (identity tests) and by
    ``tests/test_oracle_pins.py`` against the state ``exact_step`` reaches.
    """
    B = len(slot_idx)
    _, H, d_v, d_k = rs.ckpt.shape
    out = np.zeros((B, H, d_v, d_k))
    rebuild = unroll if rs.variant == "mamba2" else gdn_unroll
    for b in range(B):
        s, p = int(slot_idx[b]), int(held[b])
        if s < 0:
            continue
        out[b] = round_to(rebuild(rs.ckpt[s], rs.ring_a[s, :, :p], rs.ring_v[s, :, :p], rs.ring_k[s, :, :p]),
                          dst_dtype)
    return out


def heads_from_groups(x, n_heads):
    """Expand group-shared keys or queries to one per value head.

    Mamba-2 layers share the key (B) and query (C) projections across groups
    of value heads: with G groups, head h uses group h // (n_heads / G)
    ([Ghana] §Output without a state: "a small kernel computes them once per
    group"; §The identity prices the record of the shipped layout, x and dt
    per head and B per group).  x [..., G, d] -> [..., n_heads, d].  With the
    keys expanded, the group layout computes exactly what the per-head
    recurrence computes.

    Parity: pinned by a hand case in ``tests/test_oracle_pins.py``.
    """
    x = np.asarray(x)
    G = x.shape[-2]
    if n_heads % G:
        raise ValueError("the number of heads must be a multiple of the number of groups")
    return np.repeat(x, n_heads // G, axis=-2)
