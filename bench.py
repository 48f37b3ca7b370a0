#!/usr/bin/env python3
"""Benchmark of the ReplaySSM cached decode step on GB300; prints one JSON line.

Workload (default): one Mamba-2 layer at Nemotron-3-Super shapes -- batch 256,
128 heads, d_v = 64, d_k = 128, fp32 checkpoint (4 MiB per row), bf16 v/k/q,
fp32 alpha = sigmoid(N(3, 1)), L = 16, staggered per-row cursors so about 16
rows flush on every step.  A step is one decode step of the layer: the host
plan (cursor and flush flag per row) and one launch of the cached-decode
kernel over the batch; the timed region replays K such steps as one CUDA
graph, with every input already in HBM.  The checkpoint and rings (1.2 GiB)
exceed the 129 MB L2, so every step streams its state from HBM.

Reported beside it, on the same inputs: the conventional load-update-store
kernel, the Gated DeltaNet layer (32 value heads of 128 x 128, fp16 d/k
rings) and its conventional kernel, an end-to-end figure through the C ABI
with pinned host buffers, and the CPU oracle timed on the host cores.

``--impl reference`` times the CPU oracle instead (the reference arm).
Under torchrun every rank runs its own batch of 256 rows on its own GPU (rows
are independent: weak scaling, no collective on the data path).
"""

import argparse
import datetime as _dt
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ReplaySSM decode tokens/s per layer at bs256; achieved HBM GB/s vs roofline"
UNIT = "tokens/s/layer"
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    "mamba2_bs256": dict(variant="mamba2", B=256, H=128, d_v=64, d_k=128, L=16, ckpt="f32", inp="bf16",
                         ring="bf16",
                         desc="Mamba-2 layer, Nemotron-3-Super shapes: batch 256, 128 heads, d_v 64, d_k 128, "
                              "fp32 checkpoint, bf16 v/k/q, fp32 alpha=sigmoid(N(3,1)), L 16, staggered cursors"),
    "mamba2_bs256_lp16": dict(variant="mamba2", B=256, H=128, d_v=64, d_k=128, L=16, ckpt="f32", inp="bf16",
                              ring="bf16", lp="f16",
                              desc="Mamba-2 layer as mamba2_bs256 with a two-precision checkpoint: fp32 "
                                   "recurrence copy, fp16 read copy for non-flush rows"),
    "mamba2_bs256_lp8": dict(variant="mamba2", B=256, H=128, d_v=64, d_k=128, L=16, ckpt="f32", inp="bf16",
                             ring="bf16", lp="e4m3",
                             desc="Mamba-2 layer as mamba2_bs256 with a two-precision checkpoint: fp32 "
                                  "recurrence copy, E4M3 read copy (a power-of-two scale per state row) for "
                                  "non-flush rows"),
    "mamba2_bs256_g8": dict(variant="mamba2", B=256, H=128, d_v=64, d_k=128, L=16, ckpt="f32", inp="bf16",
                            ring="bf16", groups=8,
                            desc="Mamba-2 layer as mamba2_bs256 with the model's own key layout: keys and queries "
                                 "shared by 8 groups of 16 heads, key ring per group, group dots k_j.q computed "
                                 "once per group"),
    "mamba2_bs256_L8": dict(variant="mamba2", B=256, H=128, d_v=64, d_k=128, L=8, ckpt="f32", inp="bf16",
                            ring="bf16", desc="Mamba-2 layer as mamba2_bs256 with buffer length L 8"),
    "mamba2_bs256_L32": dict(variant="mamba2", B=256, H=128, d_v=64, d_k=128, L=32, ckpt="f32", inp="bf16",
                             ring="bf16", desc="Mamba-2 layer as mamba2_bs256 with buffer length L 32"),
    "mamba2_bs512": dict(variant="mamba2", B=512, H=128, d_v=64, d_k=128, L=16, ckpt="f32", inp="bf16",
                         ring="bf16", desc="Mamba-2 layer as mamba2_bs256 at batch 512"),
    "mamba2_bs256_f16": dict(variant="mamba2", B=256, H=128, d_v=64, d_k=128, L=16, ckpt="f16", inp="bf16",
                             ring="bf16", desc="Mamba-2 layer as mamba2_bs256 with an fp16 checkpoint (2 MiB per row)"),
    "gdn_bs256": dict(variant="gdn", B=256, H=32, d_v=128, d_k=128, L=16, ckpt="f32", inp="bf16", ring="f16",
                      desc="Gated DeltaNet layer: batch 256, 32 value heads of 128 x 128, fp32 checkpoint, "
                           "fp16 d/k rings, fp32 g ring, L 16, staggered cursors"),
}
N_INPUT_SETS = 16  # distinct per-step input sets cycled through the timed steps


# ---------------------------------------------------------------------------
# CPU oracle timing (runs in spawned workers, before any CUDA call)
# ---------------------------------------------------------------------------
def _oracle_worker(job):
    """Time oracle.exact_step on one row of ``heads`` heads for warmup + steps."""
    variant, heads, d_v, d_k, warmup, steps, seed = job
    import numpy as np

    import oracle

    r = np.random.default_rng(seed)
    S = r.standard_normal((1, heads, d_v, d_k)) / math.sqrt(d_k)
    st = oracle.ExactState(variant, S)
    slots = np.zeros(1, dtype=np.int32)
    n_sets = 16  # input sets cycled through the steps
    v = r.standard_normal((n_sets, 1, heads, d_v)) / math.sqrt(d_k)
    k = r.standard_normal((n_sets, 1, heads, d_k)) / math.sqrt(d_k)
    q = r.standard_normal((n_sets, 1, heads, d_k)) / math.sqrt(d_k)
    a = 1.0 / (1.0 + np.exp(-r.normal(3.0, 1.0, (n_sets, 1, heads))))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((n_sets, 1, heads)))) if variant == "gdn" else [None] * n_sets
    if variant == "gdn":
        a = np.log(a)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    for t in range(warmup):
        i = t % n_sets
        oracle.exact_step(st, slots, v[i], k[i], q[i], a[i], beta[i])
    t0 = time.perf_counter()
    for t in range(steps):
        i = t % n_sets
        oracle.exact_step(st, slots, v[i], k[i], q[i], a[i], beta[i])
    return time.perf_counter() - t0


def oracle_throughput(spec, budget_s, warmup=1, steps=None):
    """Tokens/s/layer of the CPU oracle on the host cores.

    Every core runs one row of the layer in a spawned process (BLAS limited to
    one thread per process); the sample is sized to about ``budget_s`` of work.
    Returns (tokens_per_s, cores, sample description).
    """
    import multiprocessing as mp

    cores = os.cpu_count() or 1
    H = spec["H"]
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(cores) as pool:
            # calibrate: one step of one row of all heads
            t1 = pool.map(_oracle_worker, [(spec["variant"], H, spec["d_v"], spec["d_k"], 1, 1, 99)])[0]
            heads = H
            if steps is None:
                steps = max(1, min(4096, int(budget_s / max(t1, 1e-6))))
            else:
                # fixed step count: shrink the per-step sample to fit the budget
                heads = max(1, min(H, int(H * budget_s / max(t1 * (steps + warmup), 1e-9))))
            jobs = [(spec["variant"], heads, spec["d_v"], spec["d_k"], warmup, steps, 1000 + i) for i in range(cores)]
            t0 = time.perf_counter()
            elapsed = pool.map(_oracle_worker, jobs)
            wall = time.perf_counter() - t0
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    t_max = max(elapsed)
    tokens = cores * steps * heads / H  # rows x steps, scaled to all heads
    sample = (f"{cores} processes x 1 row x {heads}/{H} heads x {steps} steps of the {spec['variant']} layer "
              f"(float64 NumPy, exact conventional recurrence), {t_max:.1f} s; wall {wall:.1f} s")
    return tokens / t_max, cores, sample


def _oracle_batch_worker(job):
    """Time the oracle's conventional step called on a whole block of rows:
    ``rows`` rows x ``heads`` heads in one call per step (the oracle's
    functions broadcast over leading axes), float64."""
    variant, rows, heads, d_v, d_k, warmup, steps, seed = job
    import numpy as np

    import oracle

    r = np.random.default_rng(seed)
    S = r.standard_normal((rows, heads, d_v, d_k)) / math.sqrt(d_k)
    n_sets = 4
    sets = []
    for _ in range(n_sets):
        v = r.standard_normal((rows, heads, d_v)) / math.sqrt(d_k)
        k = r.standard_normal((rows, heads, d_k)) / math.sqrt(d_k)
        q = r.standard_normal((rows, heads, d_k)) / math.sqrt(d_k)
        a = 1.0 / (1.0 + np.exp(-r.normal(3.0, 1.0, (rows, heads))))
        if variant == "gdn":
            k /= np.linalg.norm(k, axis=-1, keepdims=True)
            q /= np.linalg.norm(q, axis=-1, keepdims=True)
            beta = 1.0 / (1.0 + np.exp(-r.standard_normal((rows, heads))))
            sets.append((np.log(a), beta, v, k, q))
        else:
            sets.append((a, v, k, q))
    step = oracle.gdn_step if variant == "gdn" else oracle.mamba2_step
    for t in range(warmup):
        S, _ = step(S, *sets[t % n_sets])
    t0 = time.perf_counter()
    for t in range(steps):
        S, _ = step(S, *sets[t % n_sets])
    return time.perf_counter() - t0


def oracle_batched_throughput(spec, budget_s, warmup=1, steps=16):
    """Tokens/s/layer of the CPU oracle batched over (rows, heads) on the host
    cores: every core runs its block of the batch's rows through the oracle's
    step in one call per step, for ``steps`` steps (one window of 16 by
    default); the rows per core shrink (then the heads) so that the sample
    fits about ``budget_s``.  Returns (tokens_per_s, cores, sample)."""
    import multiprocessing as mp

    cores = os.cpu_count() or 1
    B, H = spec["B"], spec["H"]
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(cores) as pool:
            t1 = pool.map(_oracle_batch_worker, [(spec["variant"], 1, H, spec["d_v"], spec["d_k"], 1, 2, 99)])[0] / 2
            rows = -(-B // cores)
            heads = H
            fit = budget_s / max(t1 * (steps + warmup), 1e-9)  # rows of all heads that fit the budget
            if fit < rows:
                rows = max(1, int(fit))
                if fit < 1:
                    heads = max(1, int(H * fit))
            jobs = [(spec["variant"], rows, heads, spec["d_v"], spec["d_k"], warmup, steps, 2000 + i)
                    for i in range(cores)]
            t0 = time.perf_counter()
            elapsed = pool.map(_oracle_batch_worker, jobs)
            wall = time.perf_counter() - t0
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    t_max = max(elapsed)
    tokens = cores * rows * steps * heads / H
    sample = (f"{cores} processes x {rows} rows x {heads}/{H} heads x {steps} steps of the {spec['variant']} layer, "
              f"the oracle's conventional step called once per step on each process's whole block (float64 "
              f"NumPy, batched over rows and heads), {t_max:.1f} s; wall {wall:.1f} s")
    return tokens / t_max, cores, sample


# ---------------------------------------------------------------------------
# clocks sampled during the timed regions
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.windows = []
        try:
            import torch

            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = str(device_index)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)
        except (OSError, ValueError):
            self.proc = None

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        time.sleep(0.2)
        self.proc.terminate()
        out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[4:8]))
            except ValueError:
                continue
        inside = [r for r in rows if any(a <= r[0] <= b for a, b in self.windows)]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        use = inside or rows
        reasons = sorted({n for r in use for n, v in zip(names, r[4]) if v.lower().startswith("active")})
        return {
            "sm_mhz": statistics.median(r[1] for r in use) if use else None,
            "sm_max_mhz": max(r[2] for r in use) if use else None,
            "reasons": reasons,
            "samples_in_timed_regions": len(inside),
            "power_w_max": max((float(r[3]) for r in use if r[3].replace(".", "", 1).isdigit()), default=None),
        }


# ---------------------------------------------------------------------------
# GPU side
# ---------------------------------------------------------------------------
def _peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


def _kernel_traffic(kernel, workload):
    """ncu DRAM bytes per launch for ``kernel`` if its sources are unchanged
    since the counters were taken (profiles/ncu_traffic.json), else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
    except (OSError, ValueError, KeyError):
        return None
    if rec.get("workload") != workload or rec.get("source_sha256") != source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


KERNEL_SOURCES = {"mamba2_replay": ["mamba2.cuh", "mamba2.cu"], "gdn_replay": ["gdn.cu"],
                  "conventional": ["conventional.cu"]}


def code_digest(texts):
    """SHA-256 of CUDA sources with comments and blank space removed, so that
    an edit to comments alone does not count as a kernel change."""
    import re

    h = hashlib.sha256()
    for t in texts:
        t = re.sub(r"/\*.*?\*/", "", t, flags=re.S)
        t = re.sub(r"//[^\n]*", "", t)
        h.update("\n".join(line.strip() for line in t.splitlines() if line.strip()).encode())
    return h.hexdigest()


def source_hash(kernel):
    texts = []
    for name in KERNEL_SOURCES[kernel] + ["common.cuh"]:
        with open(os.path.join(ROOT, "linear_attention_decode_replayssm_gb300", "csrc", name)) as f:
            texts.append(f.read())
    return code_digest(texts)


class Layer:
    """Device state, inputs and per-step plans for one synthetic layer."""

    def __init__(self, lib, spec, device, seed, n_steps, plans=None, with_state=True):
        import numpy as np
        import torch

        self.lib, self.spec, self.device = lib, spec, device
        B, H, dv, dk, L = (spec[k] for k in ("B", "H", "d_v", "d_k", "L"))
        td = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        gdn = spec["variant"] == "gdn"

        def randn(*shape):
            return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)

        def unit(x):
            return x / x.norm(dim=-1, keepdim=True)

        def decay(*shape):
            a = torch.sigmoid(3.0 + randn(*shape))
            return torch.log(a) if gdn else a

        sk = math.sqrt(dk)
        self.ckpt = (randn(B, H, dv, dk) / sk).to(td[spec["ckpt"]])
        self.state = self.ckpt.clone() if with_state else None  # for the conventional kernel
        self.ckpt_lp = self.ckpt_lp_scale = None  # two-precision read copy, cast by the library
        if spec.get("lp"):
            self.ckpt_lp = torch.empty(self.ckpt.shape, device=device, dtype=td[spec["lp"]])
            if spec["lp"] == "e4m3":
                self.ckpt_lp_scale = torch.empty(self.ckpt.shape[:3], device=device)
            lib.replayssm_seed_read_copy(ckpt=self.ckpt, ckpt_lp=self.ckpt_lp, scale=self.ckpt_lp_scale)
        self.ring_v = (randn(B, H, L, dv) / sk).to(td[spec["ring"]])
        G = spec.get("groups", 0)
        KH = G or H  # key / query vectors per row
        self.ring_k = (unit(randn(B, KH, L, dk)) if gdn else randn(B, KH, L, dk) / sk).to(td[spec["ring"]])
        self.kq = torch.empty(B * G * L, device=device) if G else None
        self.ring_a = decay(B, H, L)
        self.slot_idx = torch.arange(B, device=device, dtype=torch.int32)
        self.out = torch.empty(B, H, dv, device=device)
        self.inputs = []
        for _ in range(N_INPUT_SETS):
            x = dict(v=(randn(B, H, dv) / sk).to(td[spec["inp"]]))
            if gdn:
                x.update(k=unit(randn(B, H, dk)).to(td[spec["inp"]]), q=unit(randn(B, H, dk)).to(td[spec["inp"]]),
                         alpha=decay(B, H), beta=torch.sigmoid(randn(B, H)))
            else:
                x.update(k=(randn(B, KH, dk) / sk).to(td[spec["inp"]]), q=(randn(B, KH, dk) / sk).to(td[spec["inp"]]),
                         alpha=decay(B, H), beta=None)
            if G:  # the conventional kernel takes a key per head
                x.update(k_h=x["k"].repeat_interleave(H // G, dim=1), q_h=x["q"].repeat_interleave(H // G, dim=1))
            self.inputs.append(x)
        rng = np.random.default_rng(seed)
        self.decode_step0 = rng.integers(0, L, size=B).astype(np.int64)
        if plans is None:
            wps, fls = [], []
            for t in range(n_steps):
                wp, fl = lib.replayssm_plan_step(self.decode_step0 + t, L)
                wps.append(wp)
                fls.append(fl)
            plans = (np.stack(wps), np.stack(fls))
        self.wp_host, self.fl_host = plans
        self.wp = torch.from_numpy(self.wp_host).to(device)
        self.fl = torch.from_numpy(self.fl_host).to(device)
        self.variant_code = lib.RS_GDN if gdn else lib.RS_MAMBA2

    def replay_step(self, t, stream=None, x=None, wp=None, fl=None, out=None):
        x = self.inputs[t % N_INPUT_SETS] if x is None else x
        kw = dict(ckpt=self.ckpt, ring_v=self.ring_v, ring_k=self.ring_k, ring_a=self.ring_a,
                  slot_idx=self.slot_idx, write_pos=self.wp[t] if wp is None else wp,
                  is_flush=self.fl[t] if fl is None else fl, v=x["v"], k=x["k"], q=x["q"], alpha=x["alpha"],
                  out=self.out if out is None else out, stream=stream)
        if self.spec["variant"] == "gdn":
            self.lib.replayssm_decode_gdn(beta=x["beta"], **kw)
        else:
            self.lib.replayssm_decode_mamba2(ckpt_lp=self.ckpt_lp, ckpt_lp_scale=self.ckpt_lp_scale, kq_scratch=self.kq,
                                             **kw)

    def conventional_step(self, t, stream=None):
        x = self.inputs[t % N_INPUT_SETS]
        self.lib.conventional_decode(variant=self.variant_code, state=self.state, slot_idx=self.slot_idx, v=x["v"],
                                     k=x.get("k_h", x["k"]), q=x.get("q_h", x["q"]), alpha=x["alpha"],
                                     beta=x["beta"], out=self.out, stream=stream)

    def bytes_per_step(self, t0, t1, replay=True):
        from linear_attention_decode_replayssm_gb300 import traffic

        s = self.spec
        slot = self.slot_idx.cpu().numpy()
        tot = 0
        for t in range(t0, t1):
            tot += traffic.step_bytes(variant=s["variant"], H=s["H"], d_v=s["d_v"], d_k=s["d_k"],
                                      ckpt_dtype=s["ckpt"], in_dtype=s["inp"], ring_dtype=s["ring"],
                                      slot_idx=slot, write_pos=self.wp_host[t], is_flush=self.fl_host[t],
                                      replay=replay, lp_dtype=s.get("lp") if replay else None,
                                      n_groups=s.get("groups", 0) if replay else 0)
        return tot / (t1 - t0)


def _timed_graph(torch, fn, t0, t1, stream, eager, dist, sampler):
    """Run steps t0..t1-1 (captured as one CUDA graph unless ``eager``) in a
    timed region on ``stream``; returns the max over ranks of the elapsed ms."""
    graph = None
    if not eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for t in range(t0, t1):
                    fn(t, stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    w0 = time.time()
    with torch.cuda.stream(stream):  # graph.replay() launches on the current stream
        start.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for t in range(t0, t1):
                fn(t, stream)
        end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    w1 = time.time()
    if dist is not None:
        dist.barrier()
    if sampler is not None:
        sampler.mark(w0, w1)
    ms = start.elapsed_time(end)
    if dist is not None:
        tt = torch.tensor([ms], device=torch.cuda.current_device())
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    del graph
    return ms


def measure_layer(lib, torch, spec, device, args, dist, sampler, seed):
    """Device-timed ReplaySSM and conventional steps of one layer."""
    K, W = args.steps, args.warmup
    layer = Layer(lib, spec, device, seed, W + K)
    stream = torch.cuda.Stream(device=device)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for t in range(W):
            layer.replay_step(t, stream)
    ms = _timed_graph(torch, layer.replay_step, W, W + K, stream, args.eager, dist, sampler)
    res = dict(ms_per_step=ms / K, bytes_per_step=layer.bytes_per_step(W, W + K))
    with torch.cuda.stream(stream):
        for t in range(W):
            layer.conventional_step(t, stream)
    cms = _timed_graph(torch, layer.conventional_step, W, W + K, stream, args.eager, dist, sampler)
    res.update(conv_ms_per_step=cms / K, conv_bytes_per_step=layer.bytes_per_step(W, W + 1, replay=False))
    return layer, res


def measure_e2e(lib, torch, layer, steps, dist):
    """Tokens/s through the public API with host buffers.

    Each step: the host plan (cursor and flag per row) is written into the
    step's pinned staging buffer, which also holds the step's inputs (v, k,
    q, decays and, for GDN, beta, packed at 256-byte offsets); one H2D copy
    moves the buffer; the decode is launched through the C ABI with its
    arguments marshalled once per device buffer (``prepare_decode``); one D2H
    copy brings the output back and the host reads it.  Uploads, decodes and
    downloads run on three streams with three device buffers, and the host
    issues step t+2 before it waits for step t's output, so the next uploads
    and the last download overlap a decode and the host's own work never sits
    between two decodes."""
    dev = layer.device
    s = layer.spec
    B, H, dv, dk, L = (s[k] for k in ("B", "H", "d_v", "d_k", "L"))
    gdn = s["variant"] == "gdn"
    x0 = layer.inputs[0]
    KH = x0["k"].shape[1]
    fields = [("v", x0["v"].dtype, (B, H, dv)), ("k", x0["k"].dtype, (B, KH, dk)), ("q", x0["q"].dtype, (B, KH, dk)),
              ("alpha", torch.float32, (B, H))]
    if gdn:
        fields.append(("beta", torch.float32, (B, H)))
    fields += [("wp", torch.int32, (B,)), ("fl", torch.uint8, (B,))]
    offs, off = {}, 0
    for name, dt, shp in fields:
        offs[name] = off
        off += (math.prod(shp) * torch.empty((), dtype=dt).element_size() + 255) // 256 * 256
    nbytes = off

    def views(buf):
        out = {}
        for name, dt, shp in fields:
            n = math.prod(shp) * torch.empty((), dtype=dt).element_size()
            out[name] = buf[offs[name]:offs[name] + n].view(dt).view(shp)
        return out

    host_buf, host = [], []
    for x in layer.inputs:
        hb = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        hv = views(hb)
        for name in ("v", "k", "q", "alpha", "beta"):
            if name in hv:
                hv[name].copy_(x[name])
        host_buf.append(hb)
        host.append((hv["wp"].numpy(), hv["fl"].numpy()))
    NBUF = 3  # steps in flight
    assert N_INPUT_SETS > NBUF  # a staging buffer is rewritten only after its upload is done
    dev_buf = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(NBUF)]
    outs = [torch.empty_like(layer.out) for _ in range(NBUF)]
    o_h = [torch.empty(layer.out.shape, dtype=torch.float32).pin_memory() for _ in range(NBUF)]
    calls = []
    for i in range(NBUF):
        dv_ = views(dev_buf[i])
        kw = dict(ckpt=layer.ckpt, ring_v=layer.ring_v, ring_k=layer.ring_k, ring_a=layer.ring_a,
                  slot_idx=layer.slot_idx, write_pos=dv_["wp"], is_flush=dv_["fl"], v=dv_["v"], k=dv_["k"],
                  q=dv_["q"], alpha=dv_["alpha"], out=outs[i])
        if gdn:
            calls.append(lib.prepare_decode("replayssm_decode_gdn", beta=dv_["beta"], **kw))
        else:
            calls.append(lib.prepare_decode("replayssm_decode_mamba2", ckpt_lp=layer.ckpt_lp,
                                            ckpt_lp_scale=layer.ckpt_lp_scale, kq_scratch=layer.kq, **kw))
    d2h = o_h[0].numel() * 4
    up_s, comp, down_s = (torch.cuda.Stream(device=dev) for _ in range(3))
    up = [torch.cuda.Event() for _ in range(NBUF)]     # a device buffer holds this step's inputs
    used = [torch.cuda.Event() for _ in range(NBUF)]   # the decode that read a device buffer is done
    back = [torch.cuda.Event() for _ in range(NBUF)]   # an output buffer has reached host memory
    ds = layer.decode_step0.copy()

    def launch(t):
        i, hs = t % NBUF, t % N_INPUT_SETS
        wp, fl = host[hs]
        lib.replayssm_plan_step(ds + t, L, write_pos=wp, is_flush=fl)
        up_s.wait_event(used[i])
        with torch.cuda.stream(up_s):
            dev_buf[i].copy_(host_buf[hs], non_blocking=True)
        up[i].record(up_s)
        comp.wait_event(up[i])
        comp.wait_event(back[i])
        calls[i].launch(comp)
        used[i].record(comp)
        down_s.wait_event(used[i])
        with torch.cuda.stream(down_s):
            o_h[i].copy_(outs[i], non_blocking=True)
        back[i].record(down_s)

    def read(t):
        back[t % NBUF].synchronize()  # the host holds this step's output
        return float(o_h[t % NBUF][0, 0, 0])

    def run(n):
        for t in range(min(NBUF - 1, n)):
            launch(t)
        for t in range(n):
            if t + NBUF - 1 < n:
                launch(t + NBUF - 1)
            read(t)

    run(3)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    run(steps)
    el = time.perf_counter() - t0
    if dist is not None:
        tt = torch.tensor([el], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        el = float(tt.item())
    return el, nbytes, d2h


def measure_materialize(lib, torch, layer, args, sampler, launches=32):
    """Prefix-cache materialisation of every row of the layer (checkpoint
    unrolled with the records its ring holds, written to a separate pool),
    device-timed over a CUDA graph of ``launches`` calls."""
    import numpy as np

    from linear_attention_decode_replayssm_gb300 import traffic

    s = layer.spec
    held_np = layer.wp_host[0].astype(np.int32)
    held = torch.from_numpy(held_np).to(layer.device)
    dst = torch.empty_like(layer.ckpt)
    dst_idx = layer.slot_idx.flip(0).contiguous()
    stream = torch.cuda.Stream(device=layer.device)
    stream.wait_stream(torch.cuda.current_stream())

    def one(t, st):
        lib.replayssm_materialize(variant=layer.variant_code, ckpt=layer.ckpt, ring_v=layer.ring_v,
                                  ring_k=layer.ring_k, ring_a=layer.ring_a, slot_idx=layer.slot_idx, held=held,
                                  dst=dst, dst_idx=dst_idx, stream=st)

    with torch.cuda.stream(stream):
        for t in range(3):
            one(t, stream)
    ms = _timed_graph(torch, one, 0, launches, stream, args.eager, None, sampler)
    nbytes = traffic.materialize_bytes(H=s["H"], d_v=s["d_v"], d_k=s["d_k"], ckpt_dtype=s["ckpt"],
                                       ring_dtype=s["ring"], slot_idx=layer.slot_idx.cpu().numpy(), held=held_np)
    del dst
    return dict(ms_per_launch=ms / launches, bytes_per_launch=nbytes, launches=launches)


def measure_spec(lib, torch, layer, args, sampler, T, n_sets=4):
    """Speculative verification of T drafts per row on the layer, with the
    device-side commit of a seeded random number of accepted drafts (1..T),
    both inside one CUDA graph of ``steps`` steps."""
    import numpy as np

    from linear_attention_decode_replayssm_gb300 import traffic

    s, dev = layer.spec, layer.device
    steps = min(256, max(16, args.steps))
    B, H, dv, dk, L = (s[k] for k in ("B", "H", "d_v", "d_k", "L"))
    td = {"f32": torch.float32, "bf16": torch.bfloat16}[s["inp"]]
    g = torch.Generator(device=dev)
    g.manual_seed(31 + T)
    sk = math.sqrt(dk)
    sets = []
    for _ in range(n_sets):
        rn = lambda *sh: torch.randn(*sh, generator=g, device=dev)
        sets.append(dict(v=(rn(B, T, H, dv) / sk).to(td), k=(rn(B, T, H, dk) / sk).to(td),
                         q=(rn(B, T, H, dk) / sk).to(td), alpha=torch.sigmoid(3.0 + rn(B, T, H))))
    rng = np.random.default_rng(T)
    acc = rng.integers(1, T + 1, (steps + 3, B)).astype(np.int32)
    h0 = (layer.decode_step0 % L).astype(np.int32)
    # host walk of the commit rule, for the byte count of each step
    hs, fls, h = [], [], h0.copy()
    fl = lib.replayssm_plan_spec(h, L, T)
    for t in range(steps + 3):
        hs.append(h.copy())
        fls.append(fl.copy())
        h = (np.where(fl != 0, 0, h) + acc[t]).astype(np.int32)
        fl = lib.replayssm_plan_spec(h, L, T)
    acc_d = torch.from_numpy(acc).to(dev)
    h_d = torch.from_numpy(h0).to(dev)
    fl_d = torch.from_numpy(fls[0]).to(dev)
    out = torch.empty(B, T, H, dv, device=dev)
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())

    def one(t, st):
        x = sets[t % n_sets]
        lib.replayssm_spec_verify_mamba2(ckpt=layer.ckpt, ring_v=layer.ring_v, ring_k=layer.ring_k,
                                         ring_a=layer.ring_a, slot_idx=layer.slot_idx, committed=h_d, is_flush=fl_d,
                                         v=x["v"], k=x["k"], q=x["q"], alpha=x["alpha"], out=out, stream=st)
        lib.replayssm_spec_commit(committed=h_d, is_flush=fl_d, accepted=acc_d[t], L=L, T=T, stream=st)

    with torch.cuda.stream(stream):
        for t in range(3):
            one(t, stream)
    ms = _timed_graph(torch, one, 3, steps + 3, stream, args.eager, None, sampler)
    slot = layer.slot_idx.cpu().numpy()
    nbytes = sum(traffic.spec_bytes(H=H, d_v=dv, d_k=dk, T=T, ckpt_dtype=s["ckpt"], in_dtype=s["inp"],
                                    slot_idx=slot, committed=hs[t], is_flush=fls[t]) for t in range(3, steps + 3))
    del sets
    return dict(ms_per_step=ms / steps, bytes_per_step=nbytes / steps, T=T, steps=steps,
                mean_accepted=float(acc[3:].mean()), flush_frac=float(np.mean([f.mean() for f in fls[3:]])))


def measure_layers40(lib, torch, args, device, sampler):
    """40 independent Mamba-2 layer pools at batch 256 under continuous
    batching (rows leave and new requests join at random offsets every 8
    steps; a joining row restarts at decode step 0), one CUDA graph of 40
    launches per decode step."""
    import numpy as np

    from linear_attention_decode_replayssm_gb300 import synth

    spec = WORKLOADS["mamba2_bs256"]
    B, L, n_layers, K = spec["B"], spec["L"], 40, args.layers40_steps
    W = 4
    ds0 = np.random.default_rng(5).integers(0, L, B)
    sched = synth.ChurnSchedule(B, L, W + K, period=8, p_churn=0.25, seed=6, decode_step0=ds0)
    wps, fls = [], []
    for t in range(W + K):
        wp, fl = lib.replayssm_plan_step(sched.decode_step(t), L)
        wps.append(wp)
        fls.append(fl)
    plans = (np.stack(wps), np.stack(fls))
    layers = [Layer(lib, spec, device, 200 + l, W + K, plans=plans, with_state=False) for l in range(n_layers)]
    for l in range(1, n_layers):  # one set of 16 input batches serves every layer
        layers[l].inputs = layers[0].inputs
        layers[l].wp, layers[l].fl = layers[0].wp, layers[0].fl
    stream = torch.cuda.Stream(device=device)
    stream.wait_stream(torch.cuda.current_stream())

    def step(t, st):
        for l in range(n_layers):
            layers[l].replay_step(t, st, x=layers[l].inputs[(t + l) % N_INPUT_SETS])

    with torch.cuda.stream(stream):
        for t in range(W):
            step(t, stream)
    ms = _timed_graph(torch, step, W, W + K, stream, args.eager, None, sampler)
    bytes_step = layers[0].bytes_per_step(W, W + K) * n_layers
    joins = int(sched.join[W:].sum())
    del layers
    torch.cuda.empty_cache()
    return dict(ms_per_step=ms / K, bytes_per_step=bytes_step, joins=joins, steps=K, layers=n_layers)


def run_sweep(args):
    """Batch x buffer length x checkpoint dtype, ReplaySSM next to the
    conventional kernel on the same inputs; small batches rotate several state
    pools so that every step reads its state from HBM (cold L2)."""
    import numpy as np
    import torch

    from linear_attention_decode_replayssm_gb300 import _lib, build, traffic

    build.build()
    _lib.load()
    device = torch.device("cuda", 0)
    peak, _ = _peak()
    base = WORKLOADS["mamba2_bs256"]
    sampler = ClockSampler(0)
    out = []
    for ck in ("f32", "f16"):
        for L in (8, 16, 32):
            for B in (1, 8, 32, 128, 256, 512):
                spec = dict(base, B=B, L=L, ckpt=ck)
                state_bytes = B * spec["H"] * spec["d_v"] * spec["d_k"] * (4 if ck == "f32" else 2)
                n_pools = max(1, int(np.ceil(3 * 129e6 / state_bytes)))
                K = 96 if B >= 128 else 256
                K = (K // n_pools + 1) * n_pools if n_pools > 1 else K
                pools = [Layer(_lib, spec, device, 300 + i, 8 + K) for i in range(n_pools)]
                stream = torch.cuda.Stream(device=device)
                stream.wait_stream(torch.cuda.current_stream())
                rep = lambda t, st: pools[t % n_pools].replay_step(t, st)
                con = lambda t, st: pools[t % n_pools].conventional_step(t, st)
                with torch.cuda.stream(stream):
                    for t in range(8):
                        rep(t, stream)
                        con(t, stream)
                ms_r = _timed_graph(torch, rep, 8, 8 + K, stream, False, None, sampler) / K
                ms_c = _timed_graph(torch, con, 8, 8 + K, stream, False, None, sampler) / K
                by_r = np.mean([p.bytes_per_step(8, 8 + K) for p in pools[:1]])
                by_c = pools[0].bytes_per_step(8, 9, replay=False)
                row = dict(ckpt=ck, L=L, B=B, pools=n_pools, replay_us=ms_r * 1e3, conventional_us=ms_c * 1e3,
                           speedup=ms_c / ms_r, replay_frac=by_r / (ms_r / 1e3) / 1e9 / peak,
                           conventional_frac=by_c / (ms_c / 1e3) / 1e9 / peak,
                           replay_tok_s=B / (ms_r / 1e3), modelled_ratio=by_r / by_c)
                out.append(row)
                print(json.dumps(row), flush=True)
                del pools
                torch.cuda.empty_cache()
    print(json.dumps({"clocks": sampler.finish()}), flush=True)
    return out


def run_native(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    spec = WORKLOADS[args.workload]

    # CPU baseline first: spawned oracle workers start before any CUDA call
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        val, cores, sample = oracle_batched_throughput(spec, args.cpu_seconds)
        cpu = {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
        pval, pcores, psample = oracle_throughput(spec, args.cpu_seconds / 2)
        cpu["per_row"] = {"value": pval, "unit": UNIT, "cores": pcores, "sample": psample}

    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist_mod.init_process_group("nccl")
        dist = dist_mod
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    from linear_attention_decode_replayssm_gb300 import _lib, build

    if rank == 0:
        build.build()
    if dist is not None:
        dist.barrier()
    _lib.load()

    sampler = ClockSampler(local) if rank == 0 else None
    layer, main = measure_layer(_lib, torch, spec, device, args, dist, sampler, seed=rank)
    extra = {}
    if not args.no_extras:
        others = [n for n in WORKLOADS if n != args.workload]
        del layer
        torch.cuda.empty_cache()
        for i, other in enumerate(others):
            _, o = measure_layer(_lib, torch, WORKLOADS[other], device, args, dist, sampler, seed=100 + i + rank)
            extra[other] = o
            torch.cuda.empty_cache()
        layer = Layer(_lib, spec, device, rank, args.warmup + args.e2e_steps + 4)
    mat, specs = None, []
    if not args.no_extras:
        mat = measure_materialize(_lib, torch, layer, args, sampler, launches=min(32, max(4, args.steps)))
        torch.cuda.empty_cache()
        if spec["variant"] == "mamba2" and not spec.get("lp"):
            for T in (4, 8):
                specs.append(measure_spec(_lib, torch, layer, args, sampler, T))
                torch.cuda.empty_cache()
            layer = Layer(_lib, spec, device, rank, args.warmup + args.e2e_steps + 4)
    layers40 = None
    if not args.no_extras and args.layers40_steps > 0:
        del layer
        torch.cuda.empty_cache()
        layers40 = measure_layers40(_lib, torch, args, device, sampler)
        layer = Layer(_lib, spec, device, rank, args.warmup + args.e2e_steps + 4)
    clocks = sampler.finish() if sampler is not None else None

    e2e_el, h2d, d2h = measure_e2e(_lib, torch, layer, args.e2e_steps, dist)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    K, B = args.steps, spec["B"]
    peak, peak_kind = _peak()
    ms = main["ms_per_step"]
    value = world * B / (ms / 1e3)
    achieved = main["bytes_per_step"] / (ms / 1e3) / 1e9
    conv_ms = main["conv_ms_per_step"]
    conv_gbs = main["conv_bytes_per_step"] / (conv_ms / 1e3) / 1e9
    kernel = "gdn_replay" if spec["variant"] == "gdn" else "mamba2_replay"
    traffic = _kernel_traffic(kernel, args.workload)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; no model weights or datasets)",
        "config": {
            "workload": spec["desc"],
            "global_batch": world * B,
            "layers": 1,
            "l2": "inputs larger than L2: 1.2 GiB of checkpoint and rings streamed every step (L2 is 129 MB)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "timing": "CUDA graph of K steps, CUDA events on the launching stream",
        },
        "hbm_gbs": achieved,
        "roofline": {
            "bound": "hbm",
            "kernel": kernel,
            "achieved": achieved,
            "peak": peak,
            "peak_kind": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "algorithmic_bytes_per_launch": main["bytes_per_step"],
        },
        "conventional": {
            "ms_per_step": conv_ms,
            "value": world * B / (conv_ms / 1e3),
            "hbm_gbs": conv_gbs,
            "frac": conv_gbs / peak,
            "algorithmic_bytes_per_launch": main["conv_bytes_per_step"],
        },
        "speedup_vs_conventional": conv_ms / ms,
        "modelled_traffic_ratio": main["bytes_per_step"] / main["conv_bytes_per_step"],
        "cpu_baseline": cpu,
        "e2e": {
            "value": world * B * args.e2e_steps / e2e_el,
            "unit": UNIT,
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "steps": args.e2e_steps,
            "how": "C ABI with pinned host buffers: per step the host plan into the step's staging buffer, one H2D "
                   "of that buffer (v/k/q/alpha and the plan), the decode (arguments marshalled once per device "
                   "buffer), one D2H of o and a host read of it; uploads, decodes and downloads on three streams, "
                   "so step t+1's upload and step t-1's download overlap step t's decode",
        },
        "gpu_launches": K,
        "clocks": clocks,
    }
    for name, o in extra.items():
        s = WORKLOADS[name]
        line[name] = {
            "workload": s["desc"],
            "ms_per_step": o["ms_per_step"],
            "value": world * s["B"] / (o["ms_per_step"] / 1e3),
            "hbm_gbs": o["bytes_per_step"] / (o["ms_per_step"] / 1e3) / 1e9,
            "frac": o["bytes_per_step"] / (o["ms_per_step"] / 1e3) / 1e9 / peak,
            "conventional_ms_per_step": o["conv_ms_per_step"],
            "conventional_hbm_gbs": o["conv_bytes_per_step"] / (o["conv_ms_per_step"] / 1e3) / 1e9,
            "speedup_vs_conventional": o["conv_ms_per_step"] / o["ms_per_step"],
            "modelled_traffic_ratio": o["bytes_per_step"] / o["conv_bytes_per_step"],
        }
    if mat is not None:
        gbs = mat["bytes_per_launch"] / (mat["ms_per_launch"] / 1e3) / 1e9
        line["materialize"] = {
            "workload": "prefix-cache state materialisation of every row of the main workload's layer "
                        "(checkpoint + held records read, state written to a separate pool)",
            "ms_per_launch": mat["ms_per_launch"],
            "rows_per_s": world * B / (mat["ms_per_launch"] / 1e3),
            "hbm_gbs": gbs,
            "frac": gbs / peak,
            "algorithmic_bytes_per_launch": mat["bytes_per_launch"],
            "launches": mat["launches"],
        }
    for sp in specs:
        gbs = sp["bytes_per_step"] / (sp["ms_per_step"] / 1e3) / 1e9
        line[f"spec_verify_T{sp['T']}"] = {
            "workload": f"speculative verification of {sp['T']} drafts per row on the main workload's layer, "
                        f"device-side commit of a random 1..{sp['T']} accepted drafts, one graph of "
                        f"{sp['steps']} steps",
            "ms_per_step": sp["ms_per_step"],
            "vs_standard_step": sp["ms_per_step"] / ms,
            "committed_tokens_per_s": world * B * sp["mean_accepted"] / (sp["ms_per_step"] / 1e3),
            "mean_accepted": sp["mean_accepted"],
            "flush_frac": sp["flush_frac"],
            "hbm_gbs": gbs,
            "frac": gbs / peak,
            "algorithmic_bytes_per_step": sp["bytes_per_step"],
        }
    if layers40 is not None:
        ms40 = layers40["ms_per_step"]
        line["layers40_churn"] = {
            "workload": "40 independent Mamba-2 layer pools (Nemotron-3-Super shapes), batch 256, fp32 checkpoints, "
                        "L 16, continuous batching: rows leave and new requests join every 8 steps at random offsets",
            "ms_per_step": ms40,
            "ms_per_layer_step": ms40 / layers40["layers"],
            "tokens_per_s": world * B / (ms40 / 1e3),
            "tokens_per_s_per_layer": world * B * layers40["layers"] / (ms40 / 1e3),
            "hbm_gbs": layers40["bytes_per_step"] / (ms40 / 1e3) / 1e9,
            "frac": layers40["bytes_per_step"] / (ms40 / 1e3) / 1e9 / peak,
            "steps": layers40["steps"],
            "joins": layers40["joins"],
        }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args):
    """The reference arm: the CPU oracle, timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    spec = WORKLOADS[args.workload]
    val, cores, sample = oracle_batched_throughput(spec, args.ref_seconds, warmup=args.warmup, steps=args.steps)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": val,
        "unit": UNIT,
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": spec["B"] / val * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": spec["desc"], "global_batch": spec["B"], "layers": 1,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": val, "unit": UNIT, "kind": "oracle", "cores": cores, "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="mamba2_bs256")
    ap.add_argument("--eager", action="store_true", help="launch steps one by one instead of a CUDA graph")
    ap.add_argument("--no-extras", action="store_true", help="skip the second layer type")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle timing")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0)
    ap.add_argument("--e2e-steps", type=int, default=256)
    ap.add_argument("--layers40-steps", type=int, default=64, help="steps of the 40-layer churn loop (0: skip)")
    ap.add_argument("--sweep", action="store_true", help="batch x L x checkpoint dtype sweep (JSON lines)")
    args = ap.parse_args()
    if args.sweep:
        run_sweep(args)
        return
    if args.warmup < 3 and args.impl == "native" and not args.eager:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
