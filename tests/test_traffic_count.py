"""The product's byte accounting for the roofline against the pages' traffic
model (the oracle's, pinned to the printed numbers) and hand counts."""

import numpy as np

from linear_attention_decode_replayssm_gb300 import traffic
from oracle import traffic as model


def _window(variant, H, d_v, d_k, L, ckpt, inp, ring, replay=True):
    """Sum of step_bytes over one window of L steps with the batch spread
    evenly over the L cursors (every row sees every cursor once)."""
    B = 2 * L
    slot = np.arange(B, dtype=np.int32)
    ds0 = np.arange(B) % L
    tot = 0
    for t in range(L):
        wp = ((ds0 + t) % L).astype(np.int32)
        fl = (wp == L - 1).astype(np.uint8)
        tot += traffic.step_bytes(variant=variant, H=H, d_v=d_v, d_k=d_k, ckpt_dtype=ckpt, in_dtype=inp,
                                  ring_dtype=ring, slot_idx=slot, write_pos=wp, is_flush=fl, replay=replay)
    return B, tot


def test_mamba2_window_matches_the_model():
    H, d_v, d_k, L = 128, 64, 128, 16
    B, tot = _window("mamba2", H, d_v, d_k, L, "f32", "bf16", "bf16")
    M_S, r = model.state_bytes(d_v, d_k), model.record_bytes(d_v, d_k)
    io = (d_v + 2 * d_k) * 2 + 4 + 4 * d_v  # v, k, q bf16, alpha, fp32 output
    per_head_window = model.replay_window_bytes(L, M_S, r)
    assert per_head_window == 17 * 32768 + 120 * 388 + 15 * 388
    assert tot == B * H * (per_head_window + L * io) + L * B * 9
    B2, conv = _window("mamba2", H, d_v, d_k, L, "f32", "bf16", "bf16", replay=False)
    assert conv == B2 * H * (model.conventional_window_bytes(L, M_S) + L * io) + L * B2 * 4
    # state and record terms alone reproduce the model's ratio
    assert abs((tot - B * H * L * io - L * B * 9) / (conv - B * H * L * io - L * B * 4)
               - model.traffic_ratio(L, M_S, r)) < 1e-12


def test_batch_256_step_sizes():
    # a step of the bench's Mamba-2 layer: 256 rows spread over the 16 cursors
    H, L = 128, 16
    B, tot = _window("mamba2", H, 64, 128, L, "f32", "bf16", "bf16")
    per_step_256 = tot / L * (256 / B)
    assert abs(per_step_256 / 2 ** 20 - 1218.4) < 0.05
    _, conv = _window("mamba2", H, 64, 128, L, "f32", "bf16", "bf16", replay=False)
    assert abs(conv / L * (256 / B) / 2 ** 20 - 2076.1) < 0.05


def test_gdn_records_and_padding():
    # GDN: fp16 d/k records (2 * 128 + 2 * 128 + 4 bytes), beta in the inputs;
    # a padded row moves its slot index and a zero output row only
    H, d_v, d_k, L = 32, 128, 128, 16
    slot = np.array([0, -1], dtype=np.int32)
    wp = np.array([3, 5], dtype=np.int32)
    fl = np.zeros(2, dtype=np.uint8)
    got = traffic.step_bytes(variant="gdn", H=H, d_v=d_v, d_k=d_k, ckpt_dtype="f32", in_dtype="bf16",
                             ring_dtype="f16", slot_idx=slot, write_pos=wp, is_flush=fl)
    rec = 2 * 128 + 2 * 128 + 4
    io = 3 * 128 * 2 + 4 + 4 + 4 * 128
    want = H * (128 * 128 * 4 + io + 3 * rec + rec) + 9 + (4 + H * 4 * 128)
    assert got == want


def test_materialize_bytes_by_hand():
    H, d_v, d_k = 2, 64, 128
    got = traffic.materialize_bytes(H=H, d_v=d_v, d_k=d_k, ckpt_dtype="f32", ring_dtype="bf16",
                                    slot_idx=[0, 1, -1, 3], held=[0, 5, 9, 15], dst_idx=[2, 3, 0, -1])
    # rows 0 and 1 are materialised; rows 2 and 3 are skipped
    rec = 2 * (64 + 128) + 4
    want = 2 * (H * 2 * 32768 + 12) + (0 + 5) * H * rec + 2 * 8
    assert got == want


def test_two_precision_window_by_hand():
    """fp32 recurrence copy + fp16 read copy: per head and window, L-1 reads
    of the read copy, one read of the recurrence copy, one write of each."""
    H, d_v, d_k, L = 4, 64, 128, 16
    B = 2 * L
    slot = np.arange(B, dtype=np.int32)
    ds0 = np.arange(B) % L
    tot = 0
    for t in range(L):
        wp = ((ds0 + t) % L).astype(np.int32)
        fl = (wp == L - 1).astype(np.uint8)
        tot += traffic.step_bytes(variant="mamba2", H=H, d_v=d_v, d_k=d_k, ckpt_dtype="f32", in_dtype="bf16",
                                  ring_dtype="bf16", slot_idx=slot, write_pos=wp, is_flush=fl, lp_dtype="f16")
    hp, lp = 64 * 128 * 4, 64 * 128 * 2
    r = model.record_bytes(d_v, d_k)
    io = (d_v + 2 * d_k) * 2 + 4 + 4 * d_v
    per_head_window = (L - 1) * lp + hp + hp + lp + (L * (L - 1) // 2) * r + (L - 1) * r
    assert tot == B * H * (per_head_window + L * io) + L * B * 9


def test_grouped_records_match_the_printed_record():
    """Group-shared keys: a step's record traffic is the 18 944-byte layer
    record the pages price ([Ghana] §The identity) per held record and row."""
    H, d_v, d_k, G = 128, 64, 128, 8
    kw = dict(variant="mamba2", H=H, d_v=d_v, d_k=d_k, ckpt_dtype="f32", in_dtype="bf16", ring_dtype="bf16",
              slot_idx=np.array([0]), is_flush=np.array([0]), n_groups=G)
    one = traffic.step_bytes(write_pos=np.array([1]), **kw)
    zero = traffic.step_bytes(write_pos=np.array([0]), **kw)
    assert one - zero == model.grouped_record_bytes(H, d_v, G, d_k) == 18944


def test_spec_bytes_by_hand():
    """Speculative verification: per live row and head the checkpoint once,
    the committed records, T drafts in (v, k, q bf16 + decay), T fp32
    outputs and T records out; a flush row also writes the checkpoint."""
    H, d_v, d_k, T = 2, 64, 128, 4
    got = traffic.spec_bytes(H=H, d_v=d_v, d_k=d_k, T=T, ckpt_dtype="f32", in_dtype="bf16",
                             slot_idx=[0, 1, -1], committed=[3, 14, 5], is_flush=[0, 1, 0])
    state, rec = 64 * 128 * 4, 2 * (64 + 128) + 4
    draft_in, out = 2 * (64 + 2 * 128) + 4, 4 * 64
    per_row = H * (state + T * (draft_in + out + rec)) + 9
    want = 2 * per_row + (3 + 14) * H * rec + 1 * H * state + (4 + T * H * 4 * d_v)
    assert got == want
