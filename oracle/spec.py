"""Speculative verification with pointer commit, Mamba-2 (oracle; test
infrastructure only).

[Ghana] §Speculative decoding: rollback becomes a pointer.  A verification
step appends the records of all T draft tokens behind the h committed records
of the row's ring, computes the T outputs without forming a state for any
draft, and, once the sampler knows how many drafts a it accepts, commits them
by advancing the committed count by a.  Rejected records lie past the count
and are overwritten later.  A flush folds only the committed records, so it
can run in the same step, before acceptance is known; it is due when
h + T > L, because otherwise the next step's T records could run past the
window.  The decision depends only on h and T, so the commit can compute the
next step's flag on the device.

Readings taken where the pages leave a step open:
  * On a flush step the committed records are folded into the checkpoint
    first; the drafts are then written at the start of the emptied ring, and
    their outputs run from the unrounded new state.  With this placement a
    non-flush step writes slots h .. h+T-1 <= L-1 and a flush step slots
    0 .. T-1, so L slots suffice (the pages size the ring L + T).
  * The verifier commits 1 <= a <= T tokens per step (a fully rejected step
    still commits one token).
  * Draft i's output is the state after the committed records and drafts
    0 .. i, applied to q_i: the conventional recurrence over that prefix.

Parity: pinned (``tests/test_oracle_spec.py``): outputs equal the exact
recurrence over committed prefix + drafts, whatever was rejected before; the
committed state after any accept pattern equals the exact recurrence over
the accepted tokens only; the flag rule never lets a write pass slot L - 1.
"""

import numpy as np

from .recurrence import mamba2_step, unroll
from .storage import round_to


def spec_plan(committed, L, T):
    """Flush flag of a verification step: h + T > L (closed form)."""
    committed = np.asarray(committed, dtype=np.int64)
    if np.any(committed < 0) or np.any(committed > L) or not 1 <= T <= L:
        raise ValueError("need 0 <= committed <= L and 1 <= T <= L")
    return (committed + T > L).astype(np.uint8)


def spec_commit(committed, is_flush, accepted, L, T):
    """Committed count and flush flag of the next step after ``accepted``
    drafts were taken: h' = (0 if the step flushed else h) + a."""
    committed = np.asarray(committed, dtype=np.int64)
    accepted = np.asarray(accepted, dtype=np.int64)
    if np.any(accepted < 1) or np.any(accepted > T):
        raise ValueError("need 1 <= accepted <= T")
    h_new = np.where(np.asarray(is_flush) != 0, 0, committed) + accepted
    return h_new.astype(np.int32), spec_plan(h_new, L, T)


def spec_verify_step(rs, slot_idx, committed, is_flush, v, k, q, alpha):
    """One verification step of a batch, in place on ``rs`` (a Mamba-2
    ``ReplayState`` whose ring holds L slots).

    committed [B]: h, records committed in the row's ring; is_flush [B];
    v [B, T, H, d_v], k, q [B, T, H, d_k], alpha [B, T, H]: the drafts.
    Returns o [B, T, H, d_v].
    """
    if rs.variant != "mamba2":
        raise NotImplementedError("speculative verification: Mamba-2 only")
    v, k, q, alpha = (np.asarray(x, dtype=np.float64) for x in (v, k, q, alpha))
    B, T, H = alpha.shape
    L = rs.L
    o = np.zeros((B, T, H, rs.ring_v.shape[3]))
    for b in range(B):
        s = int(slot_idx[b])
        if s < 0:
            continue
        h = int(committed[b])
        recs = (rs.ring_a[s, :, :h], rs.ring_v[s, :, :h], rs.ring_k[s, :, :h])
        if is_flush[b]:
            S = unroll(rs.ckpt[s], *recs)          # fold the committed records
            rs.ckpt[s] = round_to(S, rs.ckpt_dtype)
            base = 0
        else:
            if h + T > L:
                raise ValueError(f"row {b}: {h} committed + {T} drafts overrun the window")
            S = unroll(rs.ckpt[s], *recs)
            base = h
        for i in range(T):
            S, o[b, i] = mamba2_step(S, alpha[b, i], v[b, i], k[b, i], q[b, i])
            rs.ring_v[s, :, base + i] = round_to(v[b, i], rs.ring_dtype)
            rs.ring_k[s, :, base + i] = round_to(k[b, i], rs.ring_dtype)
            rs.ring_a[s, :, base + i] = round_to(alpha[b, i], rs.a_dtype)
    return o
