"""Independent brute force for one (request, head) of the KDA RecoverSSM
verify, written in matrix form with NumPy / SciPy library routines.

It shares nothing with the C oracle: the short convolution is
``numpy.convolve``; softplus is ``numpy.logaddexp``; the sigmoid is
``scipy.special.expit``; norms are ``numpy.linalg.norm``; and each
delta-rule step is the product form
    S_t = S_{t-1} diag(e^{g_t}) (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T,
which equals the pages' update S' = S diag(e^g); S = S' + beta (v - S' k^) k^T
("vLLM/vllm/models/kimi_k3/nvidia/ops/recoverssm.py", ``_kda_recurrent_step``)
only if the decay acts on the key axis, the correction uses the decayed state
and the signs are right.  The closed-form fold of accepted records
("_commit_kda_state_kernel") is written as a sum of rank-1 terms.
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit

import oracle


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def conv_silu(hist: np.ndarray, x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """hist [W-1, C], x [n, C] (values), w [C, W] -> bf16-rounded SiLU(conv) [n, C].
    Causal: the last tap multiplies the newest input."""
    seq = np.concatenate([hist, x], axis=0)
    n = x.shape[0]
    C = x.shape[1]
    y = np.empty((n, C))
    for c in range(C):
        # np.convolve flips its second operand; 'valid' keeps windows fully inside seq
        y[:, c] = np.convolve(seq[:, c], w[c, ::-1], mode="valid")[:n]
    s = y * expit(y)
    return np.vectorize(lambda v: bf16_values(np.array([oracle.bf16_round(v)], np.uint16))[0])(s)


def gate(raw_g, dt_bias, A, lower_bound):
    u = raw_g + dt_bias
    if lower_bound is not None:
        return lower_bound * expit(A * u)
    sp = np.where(u > 20.0, u, np.logaddexp(0.0, u))
    return -A * sp


def window(S0, q, k, v, raw_g, raw_beta, dt_bias, A_log, lower_bound):
    """S0 [V,K]; q,k [n,K]; v [n,V]; raw_g [n,K]; raw_beta [n].
    Returns (o [n,V], c [n,V], states [n,V,K])."""
    n, K = k.shape
    A = np.exp(A_log)
    S = S0.copy()
    outs, cs, states = [], [], []
    I = np.eye(K)
    for t in range(n):
        kh = k[t] / np.sqrt(np.linalg.norm(k[t]) ** 2 + 1e-6)
        qh = q[t] / np.sqrt(np.linalg.norm(q[t]) ** 2 + 1e-6) / np.sqrt(K)
        Dg = np.diag(np.exp(gate(raw_g[t], dt_bias, A, lower_bound)))
        beta = expit(raw_beta[t])
        c = beta * (v[t] - S @ Dg @ kh)
        S = S @ Dg @ (I - beta * np.outer(kh, kh)) + beta * np.outer(v[t], kh)
        outs.append(S @ qh)
        cs.append(c)
        states.append(S.copy())
    return np.array(outs), np.array(cs), np.array(states)


def fold(S0, c, k, raw_g, dt_bias, A_log, lower_bound):
    """Closed form of m accepted steps: S0 diag(prod_t e^{g_t}) +
    sum_t c_t (k^_t * prod_{u>t} e^{g_u})^T.  c [m,V]; k, raw_g [m,K]."""
    m, K = k.shape
    A = np.exp(A_log)
    eg = np.array([np.exp(gate(raw_g[t], dt_bias, A, lower_bound)) for t in range(m)])
    kh = k / np.sqrt((k ** 2).sum(axis=1, keepdims=True) + 1e-6)
    out = S0 * np.prod(eg, axis=0)[None, :]
    for t in range(m):
        after = np.prod(eg[t + 1:], axis=0) if t + 1 < m else np.ones(K)
        out = out + np.outer(c[t], kh[t] * after)
    return out
