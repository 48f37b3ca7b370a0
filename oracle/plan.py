"""Per-row ring cursor and flush flag (oracle; test infrastructure only).

[PR48792] §Design notes / CUDA graphs and continuous batching: whether a row
flushes is per-row runtime data.  The write position is the row's decode step
modulo the buffer length L, computed on the host every step; a row flushes at
its last buffer slot (write_pos == L - 1), and additionally on any step the
caller forces (the align prefix-caching mode forces the block-completing step).

Parity: pinned.  ``plan_step`` is the closed form; ``simulate_cursors`` is an
independent step-by-step simulation of a ring cursor (advance by one record per
non-flush step, reset to zero after a flush) that the tests compare it with.
"""

import numpy as np


def plan_step(decode_step, L, force_flush=None):
    """Closed-form cursor and flag for one decode step of a batch.

    decode_step : int array [B], number of tokens the row has decoded so far
                  (>= 0; the current token is token ``decode_step``).
    L           : buffer length (records per window).
    force_flush : optional bool/uint8 array [B]; a nonzero entry forces a flush.

    Returns (write_pos int32 [B], is_flush uint8 [B]).
    """
    decode_step = np.asarray(decode_step, dtype=np.int64)
    if np.any(decode_step < 0):
        raise ValueError("decode_step must be >= 0")
    if L < 1:
        raise ValueError("L must be >= 1")
    write_pos = np.mod(decode_step, L).astype(np.int32)
    is_flush = write_pos == (L - 1)
    if force_flush is not None:
        is_flush = is_flush | (np.asarray(force_flush) != 0)
    return write_pos, is_flush.astype(np.uint8)


def simulate_cursors(n_steps, L, start_step=0):
    """Walk one row's ring for ``n_steps`` tokens, record by record.

    The ring starts empty at ``start_step`` tokens into a window that began at a
    flush (so ``start_step mod L`` records are already held).  Each token either
    appends a record (cursor + 1) or, when the ring already holds L - 1 records
    and this token would be the L-th, folds everything into the checkpoint
    (flush) and empties the ring.  Returns (write_pos[n], is_flush[n]) as the
    cursor seen by each token, for comparison with ``plan_step``.
    """
    held = start_step % L
    wps, flags = [], []
    for _ in range(n_steps):
        wps.append(held)
        if held + 1 == L:  # this token completes the window of L records
            flags.append(1)
            held = 0
        else:
            flags.append(0)
            held += 1
    return np.array(wps, dtype=np.int32), np.array(flags, dtype=np.uint8)
