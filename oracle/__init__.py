"""CPU oracle for the ReplaySSM cached SSM decode step.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plain, float64 statement
of what the decode step computes.  It exists to check the CUDA path, never to
stand in for it: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference legs of ``bench.py`` may import it.  The product library
(``linear_attention_decode_replayssm_gb300``) never imports, links or calls
anything here, and nothing here imports the product library: the two share no
code.  Inputs reach both sides from the seeded generators in
``linear_attention_decode_replayssm_gb300.synth``, which hold none of the
method's arithmetic; the oracle only ever receives plain NumPy arrays.

Sources, cited below by short name:

  [Ghana]   S. Ghana, "ReplaySSM: an SSM decoder that writes its state once
            every 16 tokens" (analysis of the method).
  [PR48792] vLLM pull request 48792, "[Kernel] ReplaySSM: cache SSM inputs for
            faster Gated DeltaNet standard decode" (design notes, tests and a
            review comment).
  [NV]      NVIDIA technical blog, "ReplaySSM: Rethinking State Storage for
            Faster Hybrid Model Decoding".

Modules
  plan        per-row write cursor and flush flag, plain and align
              (prefix-caching) mode                          (closed form)
  recurrence  conventional Mamba-2 and delta-rule steps, the window unroll and
              the output-only window formula                 (definitions)
  replay      the method's ckpt + ring bookkeeping, with the storage roundings
              it performs, in float64 arithmetic             (algorithm steps)
  spec        speculative verification with pointer commit (Mamba-2)
                                                             (algorithm steps)
  storage     round-to-nearest-even casts to fp32 / fp16 / bf16 / e4m3, and
              the read copy's e4m3 rounding on a power-of-two row scale
  traffic     the byte and FLOP model the pages price the method with

Every function states the passage it follows.  Parity status of each function
is recorded in its docstring: all are pinned by ``tests/test_oracle_*.py``
against closed forms, invariants, brute force or numbers printed on the pages.
"""

from .plan import plan_step, simulate_cursors, plan_align, simulate_align
from .recurrence import (
    mamba2_step,
    gdn_step,
    gdn_corrected_value,
    window_decays,
    unroll,
    gdn_unroll,
    window_output,
)
from .replay import (
    ExactState,
    ReplayState,
    exact_step,
    replay_step,
    materialize,
    heads_from_groups,
)
from .storage import round_to, round_read_copy, round_rows_scaled, row_scale_exponent, STORAGE_DTYPES
from . import spec, traffic

__all__ = [
    "plan_step",
    "simulate_cursors",
    "plan_align",
    "simulate_align",
    "mamba2_step",
    "gdn_step",
    "gdn_corrected_value",
    "window_decays",
    "unroll",
    "gdn_unroll",
    "window_output",
    "ExactState",
    "ReplayState",
    "exact_step",
    "replay_step",
    "materialize",
    "heads_from_groups",
    "round_to",
    "round_read_copy",
    "round_rows_scaled",
    "row_scale_exponent",
    "STORAGE_DTYPES",
    "spec",
    "traffic",
]
