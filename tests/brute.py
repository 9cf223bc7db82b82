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


def conv_silu_exact(hist: np.ndarray, x: np.ndarray, w: np.ndarray):
    """hist [W-1, C], x [n, C] (values), w [C, W] -> (SiLU(conv) in double [n, C],
    sum_j |w_j x_j| [n, C]).  Causal: the last tap multiplies the newest input."""
    seq = np.concatenate([hist, x], axis=0)
    n = x.shape[0]
    C = x.shape[1]
    y = np.empty((n, C))
    mag = np.empty((n, C))
    for c in range(C):
        # np.convolve flips its second operand; 'valid' keeps windows fully inside seq
        y[:, c] = np.convolve(seq[:, c], w[c, ::-1], mode="valid")[:n]
        mag[:, c] = np.convolve(np.abs(seq[:, c]), np.abs(w[c, ::-1]), mode="valid")[:n]
    return y * expit(y), mag, y


def bf16_rne(v: np.ndarray) -> np.ndarray:
    """bf16 codes of double values, nearest even (the oracle's straight rounding)."""
    v = np.asarray(v, np.float64)
    return np.array([oracle.bf16_round(float(e)) for e in v.ravel()], np.uint16).reshape(v.shape)


def assert_codes_round_exact(codes: np.ndarray, s: np.ndarray, mag: np.ndarray, y: np.ndarray,
                             max_frac: float = 2e-3):
    """bf16 codes of an fp32 evaluation of s = SiLU(y), y = sum_j w_j x_j, are
    the correct rounding of the exact s except near a rounding boundary: a
    differing code must be the rounding of some value within the fp32
    evaluation's error of s.  That error is a few fp32 ulp of s plus
    |SiLU'(y)| times the summation error 2^-22 sum_j |w_j x_j|."""
    codes = np.asarray(codes, np.uint16).ravel()
    s = np.asarray(s, np.float64).ravel()
    exact = bf16_rne(s)
    bad = np.nonzero(codes != exact)[0]
    assert len(bad) <= max(1, max_frac * codes.size), f"{len(bad)} of {codes.size} codes differ"
    if len(bad) == 0:
        return
    yb = np.asarray(y, np.float64).ravel()[bad]
    sig = expit(yb)
    dsilu = np.abs(sig * (1 + yb * (1 - sig)))
    slack = (np.abs(s[bad]) * 2.0 ** -20 + dsilu * np.asarray(mag, np.float64).ravel()[bad] * 2.0 ** -22
             + 2.0 ** -130)
    got = bf16_values(codes[bad])
    lo = bf16_values(bf16_rne(s[bad] - slack))
    hi = bf16_values(bf16_rne(s[bad] + slack))
    ok = (got >= lo) & (got <= hi)
    assert np.all(ok), (f"codes {codes[bad][~ok][:4]} for exact values {s[bad][~ok][:4]} "
                        "are not the rounding of any value within the fp32 error")


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
