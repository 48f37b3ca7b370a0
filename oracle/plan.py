"""Per-row ring cursor and flush flag (oracle; test infrastructure only).

[PR48792] §Design notes / CUDA graphs and continuous batching: whether a row
flushes is per-row runtime data.  The write position is the row's decode step
modulo the buffer length L, computed on the host every step; a row flushes at
its last buffer slot (write_pos == L - 1), and additionally on any step the
caller forces (the align prefix-caching mode forces the block-completing step).

Align mode ([PR48792] §What this PR adds, the prefix-caching bullet, and
§Tests; [Ghana] §What actually shipped): prefix caching needs the exact state
at every cache-block boundary, and a checkpoint is exact only right after a
flush.  So the step that completes a block of ``block`` tokens is forced to
flush, and the ring is re-anchored at each block start.  ``plan_align`` is the
closed form of that cursor: the anchor of a token is the later of the row's
decode start and the start of its cache block, and the cursor counts the
tokens since the anchor modulo L.  (Reading: the decode start is an anchor
because the prefill leaves an exact state there; the pages do not spell out a
decode start that falls inside a block.)

Parity: pinned.  ``plan_step`` and ``plan_align`` are closed forms;
``simulate_cursors`` and ``simulate_align`` are independent step-by-step
simulations of a ring cursor (advance by one record per non-flush step, reset
to zero after a flush; in align mode also flush on the token that completes a
block) that the tests compare them with.
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


def plan_align(position, start, L, block):
    """Closed-form cursor and flag in align (prefix-caching) mode.

    position : int array [B], absolute position of the token decoded this step
               (the number of tokens before it in the sequence).
    start    : int array [B], position of the row's first decoded token (the
               prefill left an exact checkpoint covering tokens < start).
    L        : buffer length.
    block    : cache block size in tokens; 0 turns align mode off, which gives
               ``plan_step(position - start, L)``.

    Returns (write_pos int32 [B], is_flush uint8 [B]).
    """
    position = np.asarray(position, dtype=np.int64)
    start = np.asarray(start, dtype=np.int64)
    if np.any(start < 0) or np.any(position < start):
        raise ValueError("need 0 <= start <= position")
    if L < 1 or block < 0:
        raise ValueError("need L >= 1 and block >= 0")
    if block == 0:
        return plan_step(position - start, L)
    anchor = np.maximum(start, (position // block) * block)
    write_pos = np.mod(position - anchor, L).astype(np.int32)
    completes = np.mod(position + 1, block) == 0
    return write_pos, ((write_pos == L - 1) | completes).astype(np.uint8)


def simulate_align(start, n_steps, L, block):
    """Walk one row that starts decoding at ``start`` with an empty ring, token
    by token, in align mode: each token sees the number of records held; it
    flushes (and empties the ring) when it would be the L-th record of the
    window or when it is the last token of a cache block, and otherwise
    appends.  Returns (write_pos[n], is_flush[n])."""
    held = 0
    wps, flags = [], []
    for t in range(n_steps):
        pos = start + t
        wps.append(held)
        if held + 1 == L or (block and (pos + 1) % block == 0):
            flags.append(1)
            held = 0
        else:
            flags.append(0)
            held += 1
    return np.array(wps, dtype=np.int32), np.array(flags, dtype=np.uint8)
