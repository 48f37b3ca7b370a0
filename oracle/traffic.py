"""The byte and FLOP model the pages price the method with (oracle; test only).

Pure arithmetic, pinned against the numbers the pages print
(``tests/golden/traffic_model.json``).  The product's own byte accounting for
the roofline (``linear_attention_decode_replayssm_gb300.traffic``) is written
separately and tested against this model.

All byte counts are per head unless a function says otherwise.
"""

import math

MiB = 1 << 20
GiB = 1 << 30


def state_bytes(d_v, d_k, elem_bytes=4):
    """One head's state, d_v x d_k elements ([Ghana] §Why a fixed-size state
    is not cheap to decode: 128 heads x 64 x 128 x 4 B is 4 MiB per layer)."""
    return d_v * d_k * elem_bytes


def record_bytes(d_v, d_k, elem_bytes=2, decay_bytes=4):
    """One head's ring record (alpha_j, v_j, k_j) in 16-bit v/k plus a 4-byte
    decay: 2 d_v + 2 d_k + 4 bytes ([Ghana] §The identity, pricing from the
    paper's appendix)."""
    return elem_bytes * (d_v + d_k) + decay_bytes


def conventional_window_bytes(L, M_S):
    """Conventional decoding reads and writes the state every step: 2 L M_S
    over a window of L tokens ([Ghana] §The identity)."""
    return 2 * L * M_S


def replay_window_bytes(L, M_S, r):
    """ReplaySSM over a window of L tokens: the state is read on every step and
    written once, (L + 1) M_S; step i reads the i - 1 records before it, so the
    window reads L (L - 1) / 2 records and writes L - 1 ([Ghana] §The identity)."""
    return (L + 1) * M_S + (L * (L - 1) // 2 + (L - 1)) * r


def state_term_ratio(L):
    """(L + 1) / 2L: the state term alone ([Ghana] §The identity)."""
    return (L + 1) / (2 * L)


def traffic_ratio(L, M_S, r):
    """ReplaySSM bytes over conventional bytes for one window."""
    return replay_window_bytes(L, M_S, r) / conventional_window_bytes(L, M_S)


def grouped_record_bytes(n_heads, d_v, n_groups, d_k, elem_bytes=2, dt_bytes=4):
    """Per-layer record when the key is stored once per group: each value head
    keeps x (d_v 16-bit values) and a 4-byte dt, each group keeps one d_k-wide
    B ([Ghana] §The identity, the released kernel's buffer layout)."""
    return n_heads * (elem_bytes * d_v + dt_bytes) + n_groups * elem_bytes * d_k


def replay_bytes_per_token(L, layer_state_bytes, layer_record_bytes):
    """Per-layer bytes per decoded token, averaged over a window."""
    return replay_window_bytes(L, layer_state_bytes, layer_record_bytes) / L


def conventional_bytes_per_token(layer_state_bytes):
    return 2 * layer_state_bytes


def optimal_window(state_over_record, T=1, a_bar=1.0):
    """L* = sqrt(2 a_bar (M_S / r - T)) ([Ghana] §Why 16), with T tokens
    verified per step and a_bar accepted on average (standard decoding: 1, 1)."""
    return math.sqrt(2.0 * a_bar * (state_over_record - T))


def step_flops(d_v, d_k):
    """About 5 d_v d_k FLOPs per head-step ([Ghana] §Why a fixed-size state is
    not cheap to decode: decay, rank-1 update and output read)."""
    return 5 * d_v * d_k


def arithmetic_intensity(d_v, d_k, elem_bytes=4):
    """FLOPs per byte of the conventional step: 5 d_v d_k over 2 x 4 d_v d_k."""
    return step_flops(d_v, d_k) / (2 * state_bytes(d_v, d_k, elem_bytes))


def kv_equivalent_tokens(layer_state_bytes, kv_bytes_per_token):
    """How many tokens of KV cache one layer's SSM state is worth."""
    return layer_state_bytes / kv_bytes_per_token


def crossover_tokens(n_ssm_layers, ssm_bytes_per_step, n_attn_layers, kv_bytes_per_token):
    """Context length N at which attention reads as many bytes per step as the
    SSM layers read and write: n_ssm * step_bytes = n_attn * N * kv_bytes
    ([Ghana] §Why a fixed-size state is not cheap to decode)."""
    return n_ssm_layers * ssm_bytes_per_step / (n_attn_layers * kv_bytes_per_token)
