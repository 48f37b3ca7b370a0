"""Pins for the CPU oracle: it is checked here against things other than itself.

Each test fixes part of the oracle to a closed form, an invariant, a brute-force
evaluation on tiny inputs, a library routine, or a number printed on the pages
(``tests/golden``).  The pins are chosen so that a dropped term, a wrong sign,
an off-by-one in the window indexing or a transposed operand fails at least one
of them; ``test_oracle_mutations.py`` plants such mistakes and checks that.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import traffic
from tests._util import rel_err

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# cursor and flush flag
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L", [2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("start", [0, 1, 7, 15, 100])
def test_plan_matches_ring_simulation(L, start):
    n = 5 * L + 3
    wp_sim, fl_sim = oracle.simulate_cursors(n, L, start_step=start)
    wp, fl = oracle.plan_step(start + np.arange(n), L)
    assert wp.dtype == np.int32 and fl.dtype == np.uint8
    np.testing.assert_array_equal(wp, wp_sim)
    np.testing.assert_array_equal(fl, fl_sim)


def test_plan_forced_flush_and_errors():
    wp, fl = oracle.plan_step([0, 3, 5, 15], 16, force_flush=[0, 1, 0, 0])
    np.testing.assert_array_equal(wp, [0, 3, 5, 15])
    np.testing.assert_array_equal(fl, [0, 1, 0, 1])
    with pytest.raises(ValueError):
        oracle.plan_step([-1], 16)
    # one flush per window of L tokens, exactly
    wp, fl = oracle.plan_step(np.arange(1600), 16)
    assert fl.sum() == 100


@pytest.mark.parametrize("L", [2, 4, 16])
@pytest.mark.parametrize("block", [0, 1, 3, 6, 16, 40, 64])
@pytest.mark.parametrize("start", [0, 5, 39, 41, 130])
def test_plan_align_matches_ring_simulation(L, block, start):
    n = 4 * max(L, block) + 7
    wp_sim, fl_sim = oracle.simulate_align(start, n, L, block)
    pos = start + np.arange(n)
    wp, fl = oracle.plan_align(pos, np.full(n, start), L, block)
    assert wp.dtype == np.int32 and fl.dtype == np.uint8
    np.testing.assert_array_equal(wp, wp_sim)
    np.testing.assert_array_equal(fl, fl_sim)
    if block:
        # every block-completing token flushes, and the next token starts an empty ring
        done = (pos + 1) % block == 0
        assert np.all(fl[done] == 1)
        assert np.all(wp[1:][done[:-1]] == 0)


def test_plan_align_small_case_by_hand():
    # L = 4, blocks of 6 tokens, decoding from position 0: the second window
    # of each block is cut short by the forced flush on the block's last token
    wp, fl = oracle.plan_align(np.arange(12), np.zeros(12), 4, 6)
    np.testing.assert_array_equal(wp, [0, 1, 2, 3, 0, 1, 0, 1, 2, 3, 0, 1])
    np.testing.assert_array_equal(fl, [0, 0, 0, 1, 0, 1, 0, 0, 0, 1, 0, 1])
    # decode starting inside a block (position 9 of blocks of 8): anchored at 9
    wp, fl = oracle.plan_align(9 + np.arange(9), np.full(9, 9), 4, 8)
    np.testing.assert_array_equal(wp, [0, 1, 2, 3, 0, 1, 2, 0, 1])
    np.testing.assert_array_equal(fl, [0, 0, 0, 1, 0, 0, 1, 0, 0])


def test_plan_align_reduces_to_plain_plan():
    pos = np.arange(0, 500)
    # align off: the plain plan of the decoded-token count
    np.testing.assert_array_equal(oracle.plan_align(pos + 7, np.full(500, 7), 16, 0),
                                  oracle.plan_step(pos, 16))
    # blocks a multiple of L, decode from a block start: forced flushes coincide
    np.testing.assert_array_equal(oracle.plan_align(pos, np.zeros(500), 16, 64), oracle.plan_step(pos, 16))
    with pytest.raises(ValueError):
        oracle.plan_align([3], [4], 16, 8)


# --------------------------------------------------------------------------
# storage roundings
# --------------------------------------------------------------------------
def test_round_f16_ties_to_even():
    r = oracle.round_to
    assert r(1.0 + 2.0 ** -11, "f16") == 1.0                      # tie -> even
    assert r(1.0 + 3 * 2.0 ** -11, "f16") == 1.0 + 2.0 ** -9      # tie -> even
    assert r(1.0 + 2.0 ** -11 + 2.0 ** -40, "f16") == 1.0 + 2.0 ** -10
    assert r(65520.0, "f16") == np.inf                             # rounds past max
    assert r(2.0 ** -24, "f16") == 2.0 ** -24                      # smallest subnormal
    assert r(2.0 ** -26, "f16") == 0.0


def test_round_bf16_ties_and_library():
    r = oracle.round_to
    assert r(1.0 + 2.0 ** -8, "bf16") == 1.0
    assert r(1.0 + 3 * 2.0 ** -8, "bf16") == 1.0 + 2.0 ** -6
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -30, "bf16") == 1.0 + 2.0 ** -7
    assert r(-3.0, "bf16") == -3.0
    assert r(3.5e38, "bf16") == np.inf
    # against torch's fp32 -> bf16 conversion (round to nearest even) on fp32 values
    torch = pytest.importorskip("torch")
    x = _rng(1).standard_normal(20000).astype(np.float32) * np.float32(3.0) ** _rng(2).integers(-30, 30, 20000)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(r(x.astype(np.float64), "bf16"), ref)


def test_round_e4m3_ties_saturation_and_library():
    r = oracle.round_to
    assert r(1.0 + 2.0 ** -4, "e4m3") == 1.0                      # tie -> even
    assert r(1.0 + 3 * 2.0 ** -4, "e4m3") == 1.25                 # tie -> even
    assert r(1.0 + 2.0 ** -4 + 2.0 ** -30, "e4m3") == 1.125
    assert r(0.3, "e4m3") == 0.3125
    assert r(2.0 ** -9, "e4m3") == 2.0 ** -9                      # smallest subnormal
    assert r(2.0 ** -10, "e4m3") == 0.0                           # half of it: tie -> 0
    assert r(3 * 2.0 ** -10, "e4m3") == 2.0 ** -8                 # tie between 1 and 2 steps -> even
    assert r(2.0 ** -6 + 2.0 ** -10, "e4m3") == 2.0 ** -6         # smallest normal, below half a step
    assert r(448.0, "e4m3") == 448.0 and r(464.0, "e4m3") == 448.0  # largest finite; tie -> even
    assert r(1e6, "e4m3") == 448.0 and r(-1e6, "e4m3") == -448.0  # saturation
    assert np.isnan(r(np.nan, "e4m3"))
    # against torch's float32 -> float8_e4m3fn conversion (nearest even) on
    # values inside the finite range, normal and subnormal
    torch = pytest.importorskip("torch")
    rng = _rng(9)
    x = np.concatenate([rng.standard_normal(20000) * 30.0, rng.standard_normal(20000) * 0.01]).astype(np.float32)
    x = x[np.abs(x) <= 440.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(r(x.astype(np.float64), "e4m3"), ref)


def test_e4m3_read_copy_row_scales():
    """The E4M3 read copy scales each state row by a power of two so that its
    largest element lands in (224, 448], then rounds once on that grid."""
    e = oracle.row_scale_exponent
    assert list(e(np.array([[1.0, -0.5], [448.0, 1.0], [-449.0, 0.0], [0.0, 0.0], [0.875, 0.1]]))) == [-8, 0, 1, 0, -9]
    rng = _rng(4)
    x = rng.standard_normal((50, 128)) * np.exp(rng.uniform(-12, 6, (50, 1)))
    y = oracle.round_rows_scaled(x)
    ex = e(x)[:, None]
    amax = np.max(np.abs(x), axis=1, keepdims=True)
    assert np.all(amax * 2.0 ** -ex > 224.0) and np.all(amax * 2.0 ** -ex <= 448.0)
    # one rounding on the row's grid: within half a step of E4M3 at x / 2^e
    xs = np.abs(x) * 2.0 ** -ex
    step = np.where(xs < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(xs, 2.0 ** -6))) - 3))
    assert np.all(np.abs(y - x) <= 0.5 * step * 2.0 ** ex * (1 + 1e-12))
    # power-of-two scaling of a row commutes with the copy; a zero row stays zero
    np.testing.assert_array_equal(oracle.round_rows_scaled(x * 2.0 ** 7), y * 2.0 ** 7)
    assert np.all(oracle.round_rows_scaled(np.zeros((2, 8))) == 0)
    assert oracle.round_read_copy(x, "e4m3") is not None
    np.testing.assert_array_equal(oracle.round_read_copy(x, "f16"), oracle.round_to(x, "f16"))


def test_round_f32_matches_cast():
    x = _rng(3).standard_normal(1000)
    np.testing.assert_array_equal(oracle.round_to(x, "f32"), x.astype(np.float32).astype(np.float64))


# --------------------------------------------------------------------------
# conventional Mamba-2 recurrence: closed forms
# --------------------------------------------------------------------------
def _run_mamba2(S0, alphas, V, K, Q):
    S = S0.copy()
    outs = []
    for t in range(len(alphas)):
        S, o = oracle.mamba2_step(S, alphas[t], V[t], K[t], Q[t])
        outs.append(o)
    return S, np.array(outs)


def test_mamba2_no_decay_is_causal_linear_attention():
    # alpha = 1 and a zero state: o_t = sum_{j<=t} v_j (k_j . q_t) = tril(Q K^T) V
    r = _rng(4)
    T, dv, dk = 12, 5, 7
    V, K, Q = r.standard_normal((T, dv)), r.standard_normal((T, dk)), r.standard_normal((T, dk))
    _, O = _run_mamba2(np.zeros((dv, dk)), np.ones(T), V, K, Q)
    np.testing.assert_allclose(O, np.tril(Q @ K.T) @ V, rtol=1e-13, atol=1e-13)


def test_mamba2_decay_is_masked_attention_form():
    # zero state, decays a_t: o = (M * Q K^T) V with M[t, j] = exp(c_t - c_j), j <= t,
    # c = cumsum(log a) (the decayed, causally masked attention form)
    r = _rng(5)
    T, dv, dk = 20, 6, 9
    V, K, Q = r.standard_normal((T, dv)), r.standard_normal((T, dk)), r.standard_normal((T, dk))
    a = r.uniform(0.3, 0.99, T)
    c = np.cumsum(np.log(a))
    M = np.tril(np.exp(c[:, None] - c[None, :]))
    _, O = _run_mamba2(np.zeros((dv, dk)), a, V, K, Q)
    np.testing.assert_allclose(O, (M * (Q @ K.T)) @ V, rtol=1e-12, atol=1e-13)


def test_mamba2_initial_state_term():
    # from S0 with a zero stream of inputs: o_t = (prod_{l<=t} a_l) S0 q_t
    r = _rng(6)
    T, dv, dk = 9, 4, 6
    S0 = r.standard_normal((dv, dk))
    a = r.uniform(0.5, 1.0, T)
    Q = r.standard_normal((T, dk))
    _, O = _run_mamba2(S0, a, np.zeros((T, dv)), np.zeros((T, dk)), Q)
    np.testing.assert_allclose(O, np.cumprod(a)[:, None] * (Q @ S0.T), rtol=1e-13)


def test_mamba2_zero_decay_forgets_everything():
    r = _rng(7)
    S0 = r.standard_normal((3, 5))
    v, k, q = r.standard_normal(3), r.standard_normal(5), r.standard_normal(5)
    S, o = oracle.mamba2_step(S0, 0.0, v, k, q)
    np.testing.assert_allclose(o, v * (k @ q), rtol=1e-14)
    np.testing.assert_allclose(S, np.outer(v, k), rtol=1e-14)


def test_mamba2_brute_force_tiny():
    # element-by-element sums with Python loops, no array algebra
    r = _rng(8)
    T, dv, dk = 5, 2, 3
    S0 = r.standard_normal((dv, dk))
    a = r.uniform(0.2, 1.0, T)
    V, K, Q = r.standard_normal((T, dv)), r.standard_normal((T, dk)), r.standard_normal((T, dk))
    S = S0.copy()
    for t in range(T):
        S, o = oracle.mamba2_step(S, a[t], V[t], K[t], Q[t])
        for i in range(dv):
            for c in range(dk):
                decay0 = 1.0
                for l in range(t + 1):
                    decay0 *= a[l]
                want = decay0 * S0[i][c]
                for j in range(t + 1):
                    w = 1.0
                    for l in range(j + 1, t + 1):
                        w *= a[l]
                    want += w * V[j][i] * K[j][c]
                assert abs(S[i, c] - want) <= 1e-12 * max(1.0, abs(want))
        for i in range(dv):
            want_o = sum(S[i, c] * Q[t][c] for c in range(dk))
            assert abs(o[i] - want_o) <= 1e-12 * max(1.0, abs(want_o))


# --------------------------------------------------------------------------
# the window identity and the output-only formula
# --------------------------------------------------------------------------
@pytest.mark.parametrize("h", [0, 1, 2, 5, 16])
def test_unroll_equals_stepped_state(h):
    r = _rng(10 + h)
    H, dv, dk = 3, 8, 16
    S0 = r.standard_normal((H, dv, dk))
    a = r.uniform(0.1, 1.0, (H, h))
    V, K, Q = r.standard_normal((H, h, dv)), r.standard_normal((H, h, dk)), r.standard_normal((H, dk))
    S = S0.copy()
    for j in range(h):
        S, _ = oracle.mamba2_step(S, a[:, j], V[:, j], K[:, j], Q)
    U = oracle.unroll(S0, a, V, K)
    assert rel_err(U, S, nd=2) < 1e-12


@pytest.mark.parametrize("h", [1, 2, 7, 16])
def test_window_output_equals_state_output(h):
    r = _rng(30 + h)
    H, dv, dk = 2, 8, 16
    S0 = r.standard_normal((H, dv, dk))
    a = r.uniform(0.1, 1.0, (H, h))
    V, K, Q = r.standard_normal((H, h, dv)), r.standard_normal((H, h, dk)), r.standard_normal((H, dk))
    S = S0.copy()
    for j in range(h):
        S, o = oracle.mamba2_step(S, a[:, j], V[:, j], K[:, j], Q)
    assert rel_err(oracle.window_output(S0, a, V, K, Q), o) < 1e-12


def test_window_decays_small_case():
    w, gamma = oracle.window_decays(np.array([0.5, 0.25, 2.0]))
    np.testing.assert_allclose(w, [0.5, 2.0, 1.0])
    assert gamma == 0.25


# --------------------------------------------------------------------------
# delta rule
# --------------------------------------------------------------------------
def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def test_gdn_key_direction_closed_form():
    # unit k: S_t k = alpha (1 - beta) S_{t-1} k + beta v
    r = _rng(40)
    dv, dk = 6, 10
    for _ in range(5):
        S = r.standard_normal((dv, dk))
        k, q, v = _unit(r.standard_normal(dk)), r.standard_normal(dk), r.standard_normal(dv)
        g, beta = np.log(r.uniform(0.3, 1.0)), r.uniform(0, 1)
        S1, o = oracle.gdn_step(S, g, beta, v, k, q)
        a = math.exp(g)
        np.testing.assert_allclose(S1 @ k, a * (1 - beta) * (S @ k) + beta * v, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(o, S1 @ q, rtol=1e-13)


def test_gdn_orthogonal_complement_only_decays():
    r = _rng(41)
    dv, dk = 5, 9
    S = r.standard_normal((dv, dk))
    k, v, q = _unit(r.standard_normal(dk)), r.standard_normal(dv), r.standard_normal(dk)
    x = r.standard_normal(dk)
    x -= (x @ k) * k
    g, beta = np.log(0.7), 0.6
    S1, _ = oracle.gdn_step(S, g, beta, v, k, q)
    np.testing.assert_allclose(S1 @ x, 0.7 * (S @ x), rtol=1e-12, atol=1e-13)


def test_gdn_special_cases():
    r = _rng(42)
    dv, dk = 4, 8
    S = r.standard_normal((dv, dk))
    k, v, q = _unit(r.standard_normal(dk)), r.standard_normal(dv), r.standard_normal(dk)
    S1, _ = oracle.gdn_step(S, np.log(0.8), 0.0, v, k, q)          # beta = 0: pure decay
    np.testing.assert_allclose(S1, 0.8 * S, rtol=1e-14)
    S2, _ = oracle.gdn_step(S, 0.0, 1.0, v, k, q)                   # overwrite
    np.testing.assert_allclose(S2 @ k, v, rtol=1e-12, atol=1e-13)


def test_gdn_orthonormal_keys_replay():
    # alpha = 1, orthonormal keys used once each: S_t k_j = (1 - beta_j) S_0 k_j + beta_j v_j
    r = _rng(43)
    dv, dk, T = 5, 12, 7
    Kmat, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    K = Kmat[:, :T].T
    V = r.standard_normal((T, dv))
    beta = r.uniform(0, 1, T)
    S0 = r.standard_normal((dv, dk))
    S = S0.copy()
    for t in range(T):
        S, _ = oracle.gdn_step(S, 0.0, beta[t], V[t], K[t], np.zeros(dk))
    for j in range(T):
        np.testing.assert_allclose(S @ K[j], (1 - beta[j]) * (S0 @ K[j]) + beta[j] * V[j], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("h", [0, 1, 3, 16])
def test_gdn_unroll_with_corrected_values(h):
    # caching d_j and replaying reproduces the delta-rule state
    r = _rng(50 + h)
    H, dv, dk = 2, 6, 8
    S0 = r.standard_normal((H, dv, dk)) * 0.3
    g = np.log(r.uniform(0.5, 1.0, (H, h)))
    beta = r.uniform(0, 1, (H, h))
    V = r.standard_normal((H, h, dv))
    K = _unit(r.standard_normal((H, h, dk)))
    S = S0.copy()
    D = np.zeros((H, h, dv))
    for j in range(h):
        D[:, j] = oracle.gdn_corrected_value(S, g[:, j], beta[:, j], V[:, j], K[:, j])
        S, _ = oracle.gdn_step(S, g[:, j], beta[:, j], V[:, j], K[:, j], np.zeros((H, dk)))
    assert rel_err(oracle.gdn_unroll(S0, g, D, K), S, nd=2) < 1e-12


# --------------------------------------------------------------------------
# batched references: the method's bookkeeping equals the recurrence
# --------------------------------------------------------------------------
def _run_pair(variant, B=5, H=3, dv=8, dk=16, L=4, steps=23, num_slots=8, seed=0, churn=False):
    """Replay (all storage float64) against exact over staggered, paged, padded rows."""
    r = _rng(seed)
    slots = r.permutation(num_slots)[:B].astype(np.int32)
    slots[1] = -1  # a padded row
    step0 = r.integers(0, L, B)
    ckpt = r.standard_normal((num_slots, H, dv, dk)) * 0.2
    ring_v = np.full((num_slots, H, L, dv), np.nan)
    ring_k = np.full((num_slots, H, L, dk), np.nan)
    ring_a = np.full((num_slots, H, L), np.nan)
    for b in range(B):
        s, p = slots[b], step0[b] % L
        if s >= 0 and p:
            ring_v[s, :, :p] = r.standard_normal((H, p, dv)) * 0.2
            ring_k[s, :, :p] = _unit(r.standard_normal((H, p, dk))) if variant == "gdn" else r.standard_normal((H, p, dk))
            ring_a[s, :, :p] = r.uniform(0.5, 1.0, (H, p)) if variant == "mamba2" else np.log(r.uniform(0.5, 1.0, (H, p)))
    rs = oracle.ReplayState(variant, ckpt, ring_v, ring_k, ring_a, "f64", "f64", "f64")
    held = np.zeros(num_slots, dtype=int)
    for b in range(B):
        if slots[b] >= 0:
            held[slots[b]] = step0[b] % L
    ex = oracle.ExactState.from_replay(rs, held)
    dstep = step0.copy()
    worst = 0.0
    for t in range(steps):
        if churn and t % 6 == 5:
            # one live row leaves; a new request reuses its slot from decode step 0
            b = 0
            fresh = r.standard_normal((H, dv, dk)) * 0.2
            rs.reset_slot(slots[b], fresh)
            ex.reset_slot(slots[b], fresh)
            dstep[b] = 0
        wp, fl = oracle.plan_step(dstep, L)
        v = r.standard_normal((B, H, dv))
        k = r.standard_normal((B, H, dk))
        q = r.standard_normal((B, H, dk))
        if variant == "mamba2":
            a, beta = r.uniform(0.5, 1.0, (B, H)), None
        else:
            k = _unit(k)
            a, beta = np.log(r.uniform(0.5, 1.0, (B, H))), r.uniform(0, 1, (B, H))
        o_r = oracle.replay_step(rs, slots, wp, fl, v, k, q, a, beta)
        o_e = oracle.exact_step(ex, slots, v, k, q, a, beta)
        assert np.all(o_r[1] == 0) and np.all(o_e[1] == 0)
        worst = max(worst, rel_err(o_r, o_e))
        dstep += 1
    # checkpoint + held records rebuild the exact state at the end
    held_now = np.zeros(num_slots, dtype=int)
    for b in range(B):
        if slots[b] >= 0:
            held_now[slots[b]] = dstep[b] % L
    rebuilt = oracle.ExactState.from_replay(rs, held_now)
    live = slots[slots >= 0]
    return worst, rel_err(rebuilt.S[live], ex.S[live], nd=2)


@pytest.mark.parametrize("variant", ["mamba2", "gdn"])
@pytest.mark.parametrize("churn", [False, True])
def test_replay_equals_exact_float64(variant, churn):
    worst_o, worst_S = _run_pair(variant, churn=churn, seed=1 if churn else 0)
    assert worst_o < 1e-11
    assert worst_S < 1e-11


def test_replay_storage_rounding_is_small_and_nonzero():
    # with an fp32 checkpoint and f32 records the outputs move by about fp32 rounding
    r = _rng(60)
    H, dv, dk, L, B = 2, 8, 16, 4, 2
    ckpt = r.standard_normal((B, H, dv, dk)).astype(np.float32).astype(np.float64)
    mk = lambda: oracle.ReplayState("mamba2", ckpt.copy(), np.zeros((B, H, L, dv)), np.zeros((B, H, L, dk)),
                                   np.zeros((B, H, L)), "f64", "f64", "f64")
    a64, a16 = mk(), mk()
    a16.ckpt_dtype = "f16"
    slots = np.arange(B, dtype=np.int32)
    worst = 0.0
    for t in range(12):
        wp, fl = oracle.plan_step(np.full(B, t), L)
        args = (r.standard_normal((B, H, dv)), r.standard_normal((B, H, dk)), r.standard_normal((B, H, dk)),
                r.uniform(0.8, 1.0, (B, H)))
        o64 = oracle.replay_step(a64, slots, wp, fl, *args)
        o16 = oracle.replay_step(a16, slots, wp, fl, *args)
        worst = max(worst, rel_err(o16, o64))
    assert 1e-6 < worst < 2e-2


# --------------------------------------------------------------------------
# traffic model against the numbers the pages print
# --------------------------------------------------------------------------
def _golden():
    with open(os.path.join(GOLDEN, "traffic_model.json")) as f:
        return {e["name"]: e for e in json.load(f)["entries"]}


def _model_values():
    dv, dk, H, L = 64, 128, 128, 16
    M_S = traffic.state_bytes(dv, dk)
    r = traffic.record_bytes(dv, dk)
    layer_state = H * M_S
    grouped = traffic.grouped_record_bytes(H, dv, 8, dk)
    kv_token = 2 * 128 * 2 * 1  # fp8 K and V, 2 KV heads of 128: 0.5 KiB
    return {
        "layer_state_MiB": layer_state / traffic.MiB,
        "model_state_MiB_40_layers": 40 * layer_state / traffic.MiB,
        "batch256_state_GiB": 256 * 40 * layer_state / traffic.GiB,
        "kv_equivalent_tokens": traffic.kv_equivalent_tokens(layer_state, kv_token),
        "crossover_tokens": traffic.crossover_tokens(40, 2 * layer_state, 8, kv_token),
        "arithmetic_intensity": traffic.arithmetic_intensity(dv, dk),
        "traffic_ratio_L16": traffic.traffic_ratio(L, M_S, r),
        "grouped_record_bytes": grouped,
        "grouped_MiB_per_token": traffic.replay_bytes_per_token(L, layer_state, grouped) / traffic.MiB,
        "conventional_MiB_per_token": traffic.conventional_bytes_per_token(layer_state) / traffic.MiB,
        "grouped_ratio": traffic.replay_bytes_per_token(L, layer_state, grouped)
        / traffic.conventional_bytes_per_token(layer_state),
        "state_over_record": M_S / r,
        "optimal_window_standard": traffic.optimal_window(M_S / r, T=1, a_bar=1.0),
    }


def test_traffic_model_reproduces_printed_numbers():
    gold = _golden()
    vals = _model_values()
    assert set(gold) == set(vals)
    for name, e in gold.items():
        assert abs(vals[name] - e["value"]) <= e["tol"] + 1e-12, (name, vals[name], e["value"])


def test_traffic_state_term_limit():
    # the state term alone tends to one half as the window grows; L = 1 is no saving
    assert traffic.state_term_ratio(1) == 1.0
    assert abs(traffic.state_term_ratio(10 ** 6) - 0.5) < 1e-6
    M_S, r = traffic.state_bytes(64, 128), traffic.record_bytes(64, 128)
    assert traffic.replay_window_bytes(1, M_S, r) == traffic.conventional_window_bytes(1, M_S)
    # brute force: count per-step reads and writes of a window
    for L in (2, 8, 16, 32):
        total = 0
        for i in range(1, L + 1):
            total += M_S + (i - 1) * r          # read the state and the records before it
            total += M_S if i == L else r        # flush writes the state, others append
        assert total == traffic.replay_window_bytes(L, M_S, r)


@pytest.mark.parametrize("variant", ["mamba2", "gdn"])
def test_align_mode_checkpoint_is_exact_at_block_ends(variant):
    """Align mode: the forced flush leaves the exact state in the checkpoint at
    every block boundary, and materialising checkpoint + held records gives
    the exact state after every step."""
    r = _rng(7)
    B, H, dv, dk, L, block, steps = 4, 2, 8, 16, 4, 6, 40
    slots = np.array([2, 0, 3, 1], dtype=np.int32)
    start = np.array([0, 3, 5, 11])
    ckpt = r.standard_normal((4, H, dv, dk)) * 0.2
    nan = lambda *sh: np.full(sh, np.nan)
    rs = oracle.ReplayState(variant, ckpt, nan(4, H, L, dv), nan(4, H, L, dk), nan(4, H, L), "f64", "f64", "f64")
    ex = oracle.ExactState(variant, ckpt.copy())
    boundary_checks = 0
    for t in range(steps):
        pos = start + t
        wp, fl = oracle.plan_align(pos, start, L, block)
        v = r.standard_normal((B, H, dv))
        k = r.standard_normal((B, H, dk))
        q = r.standard_normal((B, H, dk))
        if variant == "mamba2":
            a, beta = r.uniform(0.5, 1.0, (B, H)), None
        else:
            k = _unit(k)
            a, beta = np.log(r.uniform(0.5, 1.0, (B, H))), r.uniform(0, 1, (B, H))
        oracle.replay_step(rs, slots, wp, fl, v, k, q, a, beta)
        oracle.exact_step(ex, slots, v, k, q, a, beta)
        held = np.where(fl != 0, 0, wp + 1)
        S = oracle.materialize(rs, slots, held)
        assert rel_err(S, ex.S[slots], nd=2) < 1e-11
        done = (pos + 1) % block == 0
        if done.any():
            boundary_checks += int(done.sum())
            assert rel_err(rs.ckpt[slots[done]], ex.S[slots[done]], nd=2) < 1e-11
    assert boundary_checks >= 4 * (steps // block) - 4
    # held = 0 returns the checkpoint itself; a padded row stays zero
    S = oracle.materialize(rs, np.array([1, -1]), np.array([0, 2]))
    np.testing.assert_array_equal(S[0], rs.ckpt[1])
    assert np.all(S[1] == 0)


# --------------------------------------------------------------------------
# two-precision checkpoint (Mamba-2): read copy for non-flush steps
# --------------------------------------------------------------------------
def _two_precision_run(lp_dtype, steps, alpha_lo, alpha_hi, L=4, H=2, dv=8, dk=16, seed=11, single=None):
    """One row, recurrence copy in float64 and a read copy in ``lp_dtype``
    (or, with ``single``, one checkpoint rounded to ``single`` at every flush).
    Returns per-step outputs of the method and of the exact recurrence, the
    flags, and the predicted read error of the pages' derivation."""
    r = _rng(seed)
    ckpt = r.standard_normal((1, H, dv, dk)) * 0.3
    nan = lambda *sh: np.full(sh, np.nan)
    rs = oracle.ReplayState("mamba2", ckpt.copy(), nan(1, H, L, dv), nan(1, H, L, dk), nan(1, H, L),
                            ckpt_dtype=single or "f64", a_dtype="f64")
    if single is None:
        rs.with_read_copy(lp_dtype)
    ex = oracle.ExactState("mamba2", ckpt.copy())
    S_m = ckpt[0].copy()           # exact state at the last flush
    gam = np.ones(H)               # decay since then
    outs, exact, flags, predicted = [], [], [], []
    for t in range(steps):
        wp, fl = oracle.plan_step([t], L)
        v = r.standard_normal((1, H, dv)) * 0.3
        k = r.standard_normal((1, H, dk)) * 0.3
        q = r.standard_normal((1, H, dk)) * 0.3
        a = r.uniform(alpha_lo, alpha_hi, (1, H))
        o_r = oracle.replay_step(rs, [0], wp, fl, v, k, q, a)
        o_e = oracle.exact_step(ex, [0], v, k, q, a)
        gam = gam * a[0]
        if single is None:
            eps = oracle.round_read_copy(S_m, lp_dtype) - S_m
            predicted.append(gam[:, None] * np.einsum("hij,hj->hi", eps, q[0]))
        if fl[0]:
            S_m = ex.S[0].copy()
            gam = np.ones(H)
        outs.append(o_r[0])
        exact.append(o_e[0])
        flags.append(int(fl[0]))
    return np.array(outs), np.array(exact), np.array(flags), np.array(predicted) if predicted else None


def test_two_precision_with_exact_read_copy_is_exact():
    outs, exact, _, _ = _two_precision_run("f64", 40, 0.5, 1.0)
    assert rel_err(outs, exact) < 1e-12


@pytest.mark.parametrize("lp", ["f16", "bf16", "e4m3"])
def test_two_precision_read_error_is_one_rounding(lp):
    """The pages' derivation: a non-flush step h records after the last flush
    errs by exactly gamma_h * eps_m * q, eps_m the read copy's rounding of the
    flushed state; a flush step is exact (it starts from the recurrence copy)."""
    outs, exact, flags, pred = _two_precision_run(lp, 48, 0.8, 1.0)
    err = outs - exact
    nf = flags == 0
    assert np.abs(err[nf]).max() > 0                      # the read copy does err
    np.testing.assert_allclose(err[nf], pred[nf], rtol=0, atol=1e-12 * np.abs(exact).max())
    assert np.abs(err[~nf]).max() < 1e-12 * np.abs(exact).max()


def test_two_precision_error_does_not_accumulate():
    """Long-memory head: with separate copies the error stays at one rounding
    of the latest checkpoint; one fp16 checkpoint rounded at every flush keeps
    accumulating ([Ghana] §The precision argument, derived)."""
    n, lo, hi = 2000, 0.9995, 0.99999
    o2, e2, _, _ = _two_precision_run("f16", n, lo, hi, seed=5)
    o1, e1, _, _ = _two_precision_run(None, n, lo, hi, seed=5, single="f16")
    early, late = slice(8, 40), slice(n - 32, n)
    two_early, two_late = rel_err(o2[early], e2[early]), rel_err(o2[late], e2[late])
    one_early, one_late = rel_err(o1[early], e1[early]), rel_err(o1[late], e1[late])
    assert two_late < 2.0 * two_early
    assert one_late > 2.5 * one_early
    assert two_late < one_late / 3.0


def test_heads_from_groups_by_hand():
    # 4 heads in 2 groups: heads 0, 1 read group 0; heads 2, 3 read group 1
    x = np.array([[[1.0, 2.0], [3.0, 4.0]]])          # [B=1, G=2, d=2]
    y = oracle.heads_from_groups(x, 4)
    np.testing.assert_array_equal(y, [[[1, 2], [1, 2], [3, 4], [3, 4]]])
    assert oracle.heads_from_groups(x, 2).shape == (1, 2, 2)
    with pytest.raises(ValueError):
        oracle.heads_from_groups(x, 3)
    # the grouped record prices to the printed 18 944 bytes at 128 heads, 8 groups
    assert oracle.traffic.grouped_record_bytes(128, 64, 8, 128) == 18944
