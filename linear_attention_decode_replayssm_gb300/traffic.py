"""Algorithmic bytes of one decode-step launch (for the roofline figure).

The count is what the step must move at minimum, per row of the batch:
  every live row, every head:  the inputs v, k, q (+ alpha, + beta for GDN),
                               the fp32 output row, and the state read once;
  ReplaySSM:                   plus the p ring records the row holds, and then
                               either one appended record (non-flush) or the
                               state written once (flush);
  conventional:                plus the state written back every step;
  per row:                     slot index, cursor and flag (9 bytes);
  padded rows:                 the slot index and a zero output row.
A ring record is (d_v + d_k) ring elements plus the 4-byte decay/gate, the
per-head record of "ReplaySSM: an SSM decoder that writes its state once every
16 tokens", §The identity (2 d_v + 2 d_k + 4 bytes with 16-bit records).
"""

import numpy as np

ESIZE = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}


def step_bytes(*, variant, H, d_v, d_k, ckpt_dtype, in_dtype, ring_dtype, slot_idx, write_pos=None,
               is_flush=None, replay=True, lp_dtype=None, n_groups=0):
    """Bytes one launch moves for the given per-row cursors (NumPy arrays [B]).

    With a two-precision checkpoint (``lp_dtype``), a non-flush row reads the
    read copy instead of the checkpoint (with its row scales for E4M3), and a
    flush row reads the checkpoint and writes both copies.  With group-shared keys (``n_groups`` > 0) a row's
    keys, queries and key records are counted once per group: a record is
    H (d_v + 1 decay) values plus G d_k keys (the group dots exchanged through
    the small scratch between the two kernels are not counted)."""
    slot_idx = np.asarray(slot_idx)
    live = slot_idx >= 0
    n_live = int(live.sum())
    n_pad = int((~live).sum())
    state = d_v * d_k * ESIZE[ckpt_dtype]
    ie, re = ESIZE[in_dtype], ESIZE[ring_dtype]
    meta = 4 + (5 if replay else 0)
    if n_groups:
        io_row = H * (d_v * ie + 4 + 4 * d_v) + n_groups * 2 * d_k * ie
        rec_row = H * (d_v * re + 4) + n_groups * d_k * re
    else:
        io_row = H * ((d_v + 2 * d_k) * ie + 4 + (4 if variant == "gdn" else 0) + 4 * d_v)
        rec_row = H * ((d_v + d_k) * re + 4)
    if not replay:
        return n_live * (H * 2 * state + io_row + meta) + n_pad * (4 + H * 4 * d_v)
    total = n_live * (io_row + meta) + n_pad * (4 + H * 4 * d_v)
    p = np.asarray(write_pos, dtype=np.int64)[live]
    fl = np.asarray(is_flush)[live] != 0
    n_fl, n_nf = int(fl.sum()), int((~fl).sum())
    # an E4M3 read copy carries a 4-byte scale per state row
    lp_copy = 0 if lp_dtype is None else d_v * d_k * ESIZE[lp_dtype] + (4 * d_v if lp_dtype == "e4m3" else 0)
    read_nf = state if lp_dtype is None else lp_copy
    write_fl = state if lp_dtype is None else state + lp_copy
    total += int(p.sum()) * rec_row
    total += n_fl * H * (state + write_fl) + n_nf * (H * read_nf + rec_row)
    return total


def step_flops(*, variant, H, d_v, d_k, slot_idx, write_pos=None, is_flush=None, replay=True):
    """Floating-point operations of one launch (multiply-add = 2), for context."""
    live = np.asarray(slot_idx) >= 0
    mn = d_v * d_k
    if not replay:
        per = (5 if variant == "mamba2" else 7) * mn
        return int(live.sum()) * H * per
    p = np.asarray(write_pos, dtype=np.int64)[live]
    fl = np.asarray(is_flush)[live] != 0
    dots = 2 if variant == "gdn" else 1
    nonflush = dots * 2 * mn + (p + 1) * (2 * d_k * dots + 2 * d_v * dots)
    flush = 2 * mn + (p + 1) * 2 * mn + 2 * mn + (2 * mn if variant == "gdn" else 0)
    return int(H * np.where(fl, flush, nonflush).sum())


def materialize_bytes(*, H, d_v, d_k, ckpt_dtype, ring_dtype, slot_idx, held, dst_idx=None):
    """Bytes one materialisation launch moves: per materialised row and head,
    the checkpoint read once, the ``held`` ring records read once and the state
    written once; per row, the slot, count and destination index (12 bytes).
    Rows skipped (negative slot or destination) move their two indices only."""
    slot_idx = np.asarray(slot_idx)
    live = slot_idx >= 0
    if dst_idx is not None:
        live &= np.asarray(dst_idx) >= 0
    state = d_v * d_k * ESIZE[ckpt_dtype]
    rec = (d_v + d_k) * ESIZE[ring_dtype] + 4
    p = np.asarray(held, dtype=np.int64)[live]
    n_live = int(live.sum())
    return n_live * (H * 2 * state + 12) + int(p.sum()) * H * rec + int((~live).sum()) * 8


def spec_bytes(*, H, d_v, d_k, T, ckpt_dtype, in_dtype, slot_idx, committed, is_flush):
    """Bytes one speculative-verification launch (Mamba-2) moves: per live row
    and head, the checkpoint read once, the committed records read (on a
    flush they are folded, and the checkpoint written), the T drafts' inputs
    read, their T outputs and T records written; per row the slot, count and
    flag (9 bytes).  Padded rows move their slot index and zero outputs."""
    slot_idx = np.asarray(slot_idx)
    live = slot_idx >= 0
    state = d_v * d_k * ESIZE[ckpt_dtype]
    rec = (d_v + d_k) * ESIZE[in_dtype] + 4
    draft_in = (d_v + 2 * d_k) * ESIZE[in_dtype] + 4
    h = np.asarray(committed, dtype=np.int64)[live]
    fl = np.asarray(is_flush)[live] != 0
    n_live = int(live.sum())
    per_row = H * (state + T * (draft_in + 4 * d_v + rec)) + 9
    total = n_live * per_row + int(h.sum()) * H * rec + int(fl.sum()) * H * state
    return total + int((~live).sum()) * (4 + T * H * 4 * d_v)
