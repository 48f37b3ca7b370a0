"""The multi-rank path on CPU: gloo, world size 2 (no GPU).

Each rank owns a block of rows (``shard.rows_of_rank``) and steps only those
rows with the oracle; gathering the per-rank outputs must reproduce a
single-process run, because the decode step has no exchange between rows.
The bench's timing reduction (max over ranks) is exercised with gloo too.
"""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from linear_attention_decode_replayssm_gb300.shard import rows_of_rank  # noqa: E402

B, STEPS = 10, 12


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_rows(rows, steps=STEPS):
    """Oracle ReplaySSM run of the given global rows of a fixed workload."""
    import oracle
    from linear_attention_decode_replayssm_gb300 import synth

    w = synth.make_workload("mamba2_bs256", B=B, H=3, L=4, steps=steps, seed=21)
    rs = oracle.ReplayState("mamba2", w.ckpt0.astype(np.float64), w.ring_v0.astype(np.float64),
                            w.ring_k0.astype(np.float64), w.ring_a0.astype(np.float64), "f32", "bf16")
    sl = w.slot_idx[rows]
    outs = []
    for t in range(steps):
        x = w.inputs(t)
        wp, fl = oracle.plan_step(w.decode_step(t)[rows], w.L)
        outs.append(oracle.replay_step(rs, sl, wp, fl, x["v"][rows], x["k"][rows], x["q"][rows], x["alpha"][rows]))
    return np.stack(outs)  # [steps, rows, H, d_v]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lo, hi = rows_of_rank(B, rank, world)
    mine = torch.from_numpy(_run_rows(np.arange(lo, hi)))
    sizes = [rows_of_rank(B, r, world) for r in range(world)]
    bufs = [torch.empty(STEPS, hi_ - lo_, *mine.shape[2:], dtype=mine.dtype) for lo_, hi_ in sizes]
    dist.all_gather(bufs, mine)
    t = torch.tensor([float(rank + 1)])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)  # bench: max over ranks of the timed region
    if rank == 0:
        q.put((torch.cat(bufs, dim=1).numpy(), float(t.item())))
    dist.barrier()
    dist.destroy_process_group()


def test_row_blocks_partition_the_batch():
    for gb in (0, 1, 7, 256, 1000):
        for world in (1, 2, 3, 8):
            spans = [rows_of_rank(gb, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == gb
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [h - l for l, h in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        rows_of_rank(8, 2, 2)


def test_two_gloo_ranks_match_one_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered, tmax = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    full = _run_rows(np.arange(B))
    np.testing.assert_array_equal(gathered, full)
    assert tmax == 2.0
