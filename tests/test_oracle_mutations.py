"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

Every mutation below is a bug someone could plausibly write: an off-by-one in
the window decays, a dropped decay factor, a flipped sign in the delta rule, a
missing gate in the corrected value, a wrong flush slot, an append at the wrong
ring slot.  Each must make at least one pin of ``test_oracle_pins`` fail.
"""

import numpy as np
import pytest

import oracle
import oracle.plan
import oracle.recurrence
import oracle.replay
from tests import test_oracle_pins as pins


def _plant(monkeypatch, name, fn):
    for mod in (oracle, oracle.recurrence, oracle.replay, oracle.plan):
        if hasattr(mod, name):
            monkeypatch.setattr(mod, name, fn)


def _fails(fn, *args, **kw):
    try:
        fn(*args, **kw)
    except (AssertionError, ValueError):
        return True
    return False


def test_decay_off_by_one_is_caught(monkeypatch):
    def bad(alphas):
        alphas = np.asarray(alphas, dtype=np.float64)
        w = np.empty_like(alphas)
        for j in range(alphas.shape[-1]):
            w[..., j] = np.prod(alphas[..., j:], axis=-1)  # includes its own decay
        return w, np.prod(alphas, axis=-1)

    _plant(monkeypatch, "window_decays", bad)
    assert _fails(pins.test_unroll_equals_stepped_state, 5)
    assert _fails(pins.test_window_output_equals_state_output, 7)


def test_dropped_checkpoint_decay_is_caught(monkeypatch):
    good = oracle.recurrence.window_decays

    def bad(alphas):
        w, _ = good(alphas)
        return w, np.prod(np.asarray(alphas)[..., :-1], axis=-1)  # forgets alpha_t

    _plant(monkeypatch, "window_decays", bad)
    assert _fails(pins.test_unroll_equals_stepped_state, 2)


def test_transposed_outer_product_is_caught(monkeypatch):
    def bad(S, alpha, v, k, q):
        alpha = np.asarray(alpha, dtype=np.float64)
        S_new = alpha[..., None, None] * S + k[..., :, None] * v[..., None, :]
        return S_new, np.einsum("...ij,...j->...i", S_new, q)

    _plant(monkeypatch, "mamba2_step", bad)
    assert _fails(pins.test_mamba2_no_decay_is_causal_linear_attention)


def test_delta_rule_sign_is_caught(monkeypatch):
    def bad(S, g, beta, v, k, q):
        alpha = np.exp(g)
        proj = np.eye(k.shape[-1]) + np.asarray(beta)[..., None, None] * k[..., :, None] * k[..., None, :]
        S_new = alpha[..., None, None] * (S @ proj) + np.asarray(beta)[..., None, None] * v[..., :, None] * k[..., None, :]
        return S_new, np.einsum("...ij,...j->...i", S_new, q)

    _plant(monkeypatch, "gdn_step", bad)
    assert _fails(pins.test_gdn_key_direction_closed_form)


def test_corrected_value_missing_gate_is_caught(monkeypatch):
    def bad(S_prev, g, beta, v, k):
        return np.asarray(beta)[..., None] * (v - np.einsum("...ij,...j->...i", S_prev, k))

    _plant(monkeypatch, "gdn_corrected_value", bad)
    assert _fails(pins.test_gdn_unroll_with_corrected_values, 3)


def test_flush_on_wrong_slot_is_caught(monkeypatch):
    def bad(decode_step, L, force_flush=None):
        wp = np.mod(np.asarray(decode_step, dtype=np.int64), L).astype(np.int32)
        return wp, (wp == 0).astype(np.uint8)

    monkeypatch.setattr(oracle, "plan_step", bad)
    assert _fails(pins.test_plan_matches_ring_simulation, 16, 0)
    assert _fails(pins.test_replay_equals_exact_float64, "mamba2", False)


def test_append_at_wrong_slot_is_caught(monkeypatch):
    good = oracle.replay.replay_step

    def bad(st, slot_idx, write_pos, is_flush, *args):
        shifted = np.minimum(np.asarray(write_pos) + 1, st.L - 1)
        return good(st, slot_idx, np.where(np.asarray(is_flush) != 0, write_pos, shifted), is_flush, *args)

    monkeypatch.setattr(oracle, "replay_step", bad)
    assert _fails(pins.test_replay_equals_exact_float64, "mamba2", False)
    assert _fails(pins.test_replay_equals_exact_float64, "gdn", False)


@pytest.mark.parametrize("variant", ["mamba2", "gdn"])
def test_flush_that_skips_current_token_is_caught(monkeypatch, variant):
    def bad(st, slot_idx, write_pos, is_flush, v, k, q, alpha, beta=None):
        # flush stores the previous state instead of the new one
        o = np.zeros((len(slot_idx), st.ckpt.shape[1], st.ckpt.shape[2]))
        for b, s in enumerate(slot_idx):
            if s < 0:
                continue
            p = int(write_pos[b])
            recs = (st.ring_a[s, :, :p], st.ring_v[s, :, :p], st.ring_k[s, :, :p])
            rebuild = oracle.unroll if st.variant == "mamba2" else oracle.gdn_unroll
            S_prev = rebuild(st.ckpt[s], *recs)
            if st.variant == "mamba2":
                _, o[b] = oracle.mamba2_step(S_prev, alpha[b], v[b], k[b], q[b])
                new_v = v[b]
            else:
                new_v = oracle.gdn_corrected_value(S_prev, alpha[b], beta[b], v[b], k[b])
                _, o[b] = oracle.gdn_step(S_prev, alpha[b], beta[b], v[b], k[b], q[b])
            if is_flush[b]:
                st.ckpt[s] = S_prev
            else:
                st.ring_v[s, :, p], st.ring_k[s, :, p], st.ring_a[s, :, p] = new_v, k[b], alpha[b]
        return o

    monkeypatch.setattr(oracle, "replay_step", bad)
    assert _fails(pins.test_replay_equals_exact_float64, variant, False)


def test_align_anchor_at_block_start_only_is_caught(monkeypatch):
    """Forgetting the decode-start anchor (cursor counted from the block start
    even when decoding began inside the block) must fail a pin."""
    def bad(position, start, L, block):
        position = np.asarray(position, dtype=np.int64)
        if block == 0:
            return oracle.plan.plan_step(position - np.asarray(start), L)
        wp = np.mod(position - (position // block) * block, L).astype(np.int32)
        return wp, ((wp == L - 1) | (np.mod(position + 1, block) == 0)).astype(np.uint8)

    monkeypatch.setattr(oracle, "plan_align", bad)
    assert _fails(pins.test_plan_align_matches_ring_simulation, 4, 40, 5)
    assert _fails(pins.test_plan_align_small_case_by_hand)


def test_align_without_forced_flush_is_caught(monkeypatch):
    def bad(position, start, L, block):
        return oracle.plan.plan_step(np.asarray(position, dtype=np.int64) - np.asarray(start), L)

    monkeypatch.setattr(oracle, "plan_align", bad)
    assert _fails(pins.test_plan_align_matches_ring_simulation, 16, 40, 0)
    assert _fails(pins.test_align_mode_checkpoint_is_exact_at_block_ends, "mamba2")


def test_materialize_dropping_last_record_is_caught(monkeypatch):
    good = oracle.replay.materialize

    def bad(rs, slot_idx, held, dst_dtype="f64"):
        return good(rs, slot_idx, np.maximum(np.asarray(held) - 1, 0), dst_dtype)

    monkeypatch.setattr(oracle, "materialize", bad)
    assert _fails(pins.test_align_mode_checkpoint_is_exact_at_block_ends, "gdn")


def test_two_precision_flush_from_read_copy_is_caught(monkeypatch):
    """A flush that starts from the low-precision read copy (so its rounding
    enters the recurrence) must fail a pin."""
    good = oracle.replay.replay_step

    def bad(st, slot_idx, write_pos, is_flush, *args):
        if st.ckpt_lp is not None:
            hp = st.ckpt.copy()
            st.ckpt[...] = st.ckpt_lp
            o = good(st, slot_idx, write_pos, is_flush, *args)
            keep = np.asarray(is_flush) == 0
            for b, s in enumerate(slot_idx):
                if keep[b]:
                    st.ckpt[s] = hp[s]
            return o
        return good(st, slot_idx, write_pos, is_flush, *args)

    monkeypatch.setattr(oracle, "replay_step", bad)
    assert _fails(pins.test_two_precision_read_error_is_one_rounding, "f16")


def test_two_precision_reading_the_recurrence_copy_is_caught(monkeypatch):
    """Non-flush steps that read the recurrence copy instead of the read copy
    (so no read error at all) must fail a pin."""
    good = oracle.replay.replay_step

    def bad(st, slot_idx, write_pos, is_flush, *args):
        lp = st.ckpt_lp
        st.ckpt_lp = None
        try:
            o = good(st, slot_idx, write_pos, is_flush, *args)
        finally:
            st.ckpt_lp = lp
        if lp is not None:
            for b, s in enumerate(slot_idx):
                if is_flush[b]:
                    lp[s] = oracle.round_to(st.ckpt[s], st.lp_dtype)
        return o

    monkeypatch.setattr(oracle, "replay_step", bad)
    assert _fails(pins.test_two_precision_read_error_is_one_rounding, "bf16")


def test_e4m3_row_scale_off_by_one_is_caught(monkeypatch):
    import oracle.storage

    good = oracle.storage.row_scale_exponent

    def bad(x):
        return good(x) - 1  # one binade too fine: the row maximum saturates

    monkeypatch.setattr(oracle.storage, "row_scale_exponent", bad)
    monkeypatch.setattr(oracle, "row_scale_exponent", bad)
    assert _fails(pins.test_e4m3_read_copy_row_scales)


def test_e4m3_rounding_toward_zero_is_caught(monkeypatch):
    import oracle.storage

    def bad(x):
        x = np.asarray(x, dtype=np.float64)
        m, e = np.frexp(x)
        return np.clip(np.ldexp(np.trunc(m * 16.0) / 16.0, e), -448.0, 448.0)  # truncates instead of rounding

    monkeypatch.setattr(oracle.storage, "_round_e4m3", bad)
    assert _fails(pins.test_round_e4m3_ties_saturation_and_library)
