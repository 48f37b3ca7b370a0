"""Pins of the speculative-verification oracle (``oracle/spec.py``).

The exact result of verifying T drafts is fixed by the recurrence itself:
draft i's output is the conventional state after the committed tokens and
drafts 0..i, applied to q_i; after the sampler accepts a drafts the row's
state is the recurrence over the committed tokens plus those a drafts only
([Ghana] §Speculative decoding: rollback becomes a pointer).  The tests run
the oracle against that definition, kept here as an independent float64
recurrence, over many steps with random accept counts.
"""

import numpy as np
import pytest

import oracle
from oracle import spec
from tests._util import rel_err


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _run(L, T, steps=60, B=4, H=2, dv=6, dk=10, seed=0, bad=None):
    r = _rng(seed)
    S0 = r.standard_normal((B, H, dv, dk)) * 0.3
    nan = lambda *sh: np.full(sh, np.nan)
    rs = oracle.ReplayState("mamba2", S0.copy(), nan(B, H, L, dv), nan(B, H, L, dk), nan(B, H, L), a_dtype="f64")
    exact = S0.copy()            # the recurrence over the committed tokens
    slots = np.arange(B)
    h = np.zeros(B, dtype=np.int64)
    fl = spec.spec_plan(h, L, T)
    worst_o = worst_c = 0.0
    n_flush = 0
    for t in range(steps):
        v = r.standard_normal((B, T, H, dv)) * 0.3
        k = r.standard_normal((B, T, H, dk)) * 0.3
        q = r.standard_normal((B, T, H, dk)) * 0.3
        a = r.uniform(0.6, 1.0, (B, T, H))
        o = (bad or spec.spec_verify_step)(rs, slots, h, fl, v, k, q, a)
        acc = r.integers(1, T + 1, B)
        for b in range(B):
            if fl[b]:
                n_flush += 1
                worst_c = max(worst_c, rel_err(rs.ckpt[b], exact[b], nd=2))
            S = exact[b].copy()
            for i in range(T):
                S, o_i = oracle.mamba2_step(S, a[b, i], v[b, i], k[b, i], q[b, i])
                worst_o = max(worst_o, rel_err(o[b, i], o_i))
                if i + 1 == acc[b]:
                    exact[b] = S.copy()   # commit the accepted prefix only
        h, fl = spec.spec_commit(h, fl, acc, L, T)
    return worst_o, worst_c, n_flush


@pytest.mark.parametrize("L, T", [(4, 1), (8, 3), (16, 4), (16, 8), (5, 5)])
def test_verify_equals_recurrence_over_committed_prefix(L, T):
    worst_o, worst_c, n_flush = _run(L, T, seed=L * 10 + T)
    assert n_flush > 0
    assert worst_o < 1e-12 and worst_c < 1e-12


def test_plan_and_commit_rule_by_brute_force():
    """Walk every (h, T, a) and check the closed forms against the ring
    occupancy: a non-flush step writes slots h..h+T-1 and must stay inside
    the L-slot window; a flush step folds h records and writes 0..T-1."""
    for L in range(1, 17):
        for T in range(1, L + 1):
            for h in range(0, L + 1):
                fl = int(spec.spec_plan([h], L, T)[0])
                assert fl == (h + T > L)
                last = (T - 1) if fl else (h + T - 1)
                assert last <= L - 1
                for a in range(1, T + 1):
                    h2, fl2 = spec.spec_commit([h], [fl], [a], L, T)
                    assert h2[0] == (a if fl else h + a)
                    assert 0 <= h2[0] <= L and fl2[0] == (h2[0] + T > L)


def test_commit_walk_by_hand():
    # L = 4, T = 2: accept 2, 2 -> the third step flushes (4 + 2 > 4)
    h, fl = np.array([0]), spec.spec_plan([0], 4, 2)
    seen = []
    for a in (2, 2, 1, 2, 1):
        seen.append((int(h[0]), int(fl[0])))
        h, fl = spec.spec_commit(h, fl, [a], 4, 2)
    assert seen == [(0, 0), (2, 0), (4, 1), (1, 0), (3, 1)]
    with pytest.raises(ValueError):
        spec.spec_commit([0], [0], [0], 4, 2)
    with pytest.raises(ValueError):
        spec.spec_plan([5], 4, 2)


def test_flush_folding_drafts_is_caught():
    """Planted mistake: a flush that also folds this step's drafts into the
    checkpoint (so rejected drafts survive) must fail the pin."""
    good = spec.spec_verify_step

    def bad(rs, slot_idx, committed, is_flush, v, k, q, alpha):
        o = good(rs, slot_idx, committed, is_flush, v, k, q, alpha)
        for b, s in enumerate(slot_idx):
            if is_flush[b]:
                T = alpha.shape[1]
                rs.ckpt[s] = oracle.unroll(rs.ckpt[s], np.moveaxis(alpha[b], 0, 1), np.moveaxis(v[b], 0, 1),
                                           np.moveaxis(k[b], 0, 1))
        return o

    worst_o, worst_c, _ = _run(8, 3, seed=3, bad=bad)
    assert worst_o > 1e-6 or worst_c > 1e-6
