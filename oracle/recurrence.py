"""Conventional recurrences, the window unroll and the output-only formula.

Oracle; test infrastructure only.  Plain float64 NumPy, one head or a stack of
heads at a time (leading axes broadcast).  Shapes: state S [..., d_v, d_k],
values v [..., d_v], keys and queries k, q [..., d_k], scalars [...].

Parity: pinned.  ``mamba2_step`` and ``gdn_step`` by closed forms (causal
linear attention, its decayed masked form, the delta-rule overwrite and
projection properties, orthonormal-key replay); ``unroll`` and ``gdn_unroll``
by the step-by-step recurrence they must equal; ``window_output`` by the
reconstructed state.  See ``tests/test_oracle_pins.py``.
"""

import numpy as np


def _outer(a, b):
    return a[..., :, None] * b[..., None, :]


def _matvec(S, x):
    return np.einsum("...ij,...j->...i", S, x)


def mamba2_step(S, alpha, v, k, q):
    """One conventional Mamba-2 decode step.

    [Ghana] §Why a fixed-size state is not cheap to decode: per head the state
    is a d_v x d_k matrix updated once per token,
        S_t = alpha_t * S_{t-1} + v_t k_t^T,   o_t = S_t q_t,
    with alpha_t in (0, 1) a data-dependent decay (Mamba-2 names x, B, C for
    v, k, q).  Returns (S_t, o_t).
    """
    alpha = np.asarray(alpha, dtype=np.float64)
    S_new = alpha[..., None, None] * S + _outer(v, k)
    return S_new, _matvec(S_new, q)


def gdn_step(S, g, beta, v, k, q):
    """One conventional Gated DeltaNet (delta-rule) decode step.

    [Ghana] §The delta-rule wrinkle:
        S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
    and o_t = S_t q_t.  The gate is cached as the scalar g = log(alpha)
    ([PR48792] §Core concept: "the scalar gate g"; §Paged cache layout: g_cache
    is fp32), so alpha_t = exp(g_t).  Written with the explicit projector
    (I - beta k k^T), as the page prints it.  Returns (S_t, o_t).
    """
    g = np.asarray(g, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    alpha = np.exp(g)
    d_k = k.shape[-1]
    proj = np.eye(d_k) - beta[..., None, None] * _outer(k, k)
    S_new = alpha[..., None, None] * (S @ proj) + beta[..., None, None] * _outer(v, k)
    return S_new, _matvec(S_new, q)


def gdn_corrected_value(S_prev, g, beta, v, k):
    """The corrected value the delta-rule variant caches in its ring.

    [Ghana] §The delta-rule wrinkle: expanding the product gives
    S_t = alpha_t S_{t-1} + u_t k_t^T with u_t = beta_t (v_t - alpha_t S_{t-1} k_t);
    [PR48792] §Core concept calls the cached vector "the corrected value d".
    """
    g = np.asarray(g, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    return beta[..., None] * (v - np.exp(g)[..., None] * _matvec(S_prev, k))


def window_decays(alphas):
    """Decay weights of a window of h records.

    [Ghana] §The identity: gamma_{i:j} = prod_{l=i..j} alpha_l and
    gamma_h = gamma_{1:h}.  Record j (1-based) of an h-record window is weighted
    by gamma_{j+1:h}, the decay accumulated after it (an empty product, 1, for
    the newest record).  ``alphas`` is [..., h] with record 1 first.
    Returns (weights [..., h], gamma_h [...]).
    """
    alphas = np.asarray(alphas, dtype=np.float64)
    h = alphas.shape[-1]
    weights = np.empty_like(alphas)
    for j in range(h):  # 0-based j holds record j+1; weight = prod of later alphas
        weights[..., j] = np.prod(alphas[..., j + 1:], axis=-1)
    gamma_h = np.prod(alphas, axis=-1)
    return weights, gamma_h


def unroll(S_ckpt, alphas, vs, ks):
    """State after h records, rebuilt from a checkpoint and the records.

    [Ghana] §The identity (also [NV] §How ReplaySSM represents the state):
        S = gamma_h S_ckpt + sum_{j=1..h} gamma_{j+1:h} v_j k_j^T.
    ``alphas`` [..., h], ``vs`` [..., h, d_v], ``ks`` [..., h, d_k]; h may be 0.
    """
    weights, gamma_h = window_decays(alphas)
    S = gamma_h[..., None, None] * S_ckpt
    for j in range(np.asarray(alphas).shape[-1]):
        S = S + weights[..., j, None, None] * _outer(vs[..., j, :], ks[..., j, :])
    return S


def gdn_unroll(S_ckpt, gs, ds, ks):
    """Delta-rule state rebuilt from a checkpoint and cached (d, k, g) records.

    [Ghana] §The delta-rule wrinkle: with the corrected value cached, the
    delta-rule step has the same outer-product form as Mamba-2, so the window
    unrolls identically with alpha_j = exp(g_j) and v_j replaced by d_j
    ([PR48792] §Core concept: the ring holds k, d and the scalar gate g).
    """
    return unroll(S_ckpt, np.exp(np.asarray(gs, dtype=np.float64)), ds, ks)


def window_output(S_ckpt, alphas, vs, ks, q):
    """Output of the newest record without forming a state.

    [Ghana] §Output without a state (also [NV] §Benefit 2):
        o_t = gamma_h S_ckpt q_t + sum_{j=1..h} gamma_{j+1:h} v_j (k_j^T q_t),
    where the window's h records include the current token as record h.
    """
    weights, gamma_h = window_decays(alphas)
    o = gamma_h[..., None] * _matvec(S_ckpt, q)
    for j in range(np.asarray(alphas).shape[-1]):
        s_j = np.sum(ks[..., j, :] * q, axis=-1)
        o = o + (weights[..., j] * s_j)[..., None] * vs[..., j, :]
    return o
