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



def bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def conv_silu_exact(hist: np.ndarray, x: np.ndarray, w: np.ndarray):
    """hist [W-1, C], x [n, C] (values), w [C, W] -> (SiLU(conv) in double [n, C],
    sum_j |w_j x_j| [n, C], the conv y [n, C]).  Causal: the last tap
    multiplies the newest input."""
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
    """bf16 codes of double values, nearest even, from the value itself: the
    quantum of a bf16 at |v| is 2^(e-8) for |v| in [2^(e-1), 2^e), at least
    the subnormal quantum 2^-133, and numpy's rint rounds half to even."""
    v = np.asarray(v, np.float64)
    _, e = np.frexp(np.abs(v))
    q = np.ldexp(1.0, np.maximum(e - 8, -133))
    r = np.rint(np.abs(v) / q) * q                     # exact: at most 8 significant bits
    bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return np.where(np.signbit(v), bits | 0x8000, bits).astype(np.uint16)


def bf16_midpoint_distance(v: np.ndarray) -> np.ndarray:
    """|v - m| / |v| for the bf16 rounding boundary m nearest to v."""
    v = np.asarray(v, np.float64)
    _, e = np.frexp(np.abs(v))
    q = np.ldexp(1.0, np.maximum(e - 8, -133))
    m = (np.floor(np.abs(v) / q) + 0.5) * q
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(v != 0, np.abs(np.abs(v) - m) / np.abs(v), np.inf)


def silu_codes_exact(y, digits: int = 60) -> np.ndarray:
    """bf16 codes of SiLU(y) = y / (1 + e^-y), correctly rounded, evaluated in
    ``digits`` decimal digits (mpmath) beyond what separates SiLU(y) from y
    (about 0.43 y digits for large positive y, so that a y lying exactly on a
    bf16 midpoint is resolved to the side SiLU(y) lies on), and rounded to
    nearest against the bf16 grid at that magnitude.  y: [n] doubles taken
    as exact, or [n, W] terms whose exact sum is y."""
    import mpmath
    y = np.asarray(y, np.float64)
    terms = y.reshape(y.shape[0], -1) if y.ndim == 2 else y.reshape(-1, 1)
    out = np.empty(terms.shape[0], np.uint16)
    for i in range(terms.shape[0]):
        extra = int(max(0.0, float(terms[i].sum())) * 0.4343) + 5
        with mpmath.workdps(digits + extra):
            half = mpmath.mpf(1) / 2
            yy = mpmath.fsum(mpmath.mpf(float(t)) for t in terms[i])
            s = yy / (1 + mpmath.exp(-yy))
            if s == 0:
                out[i] = 0x8000 if np.signbit(terms[i].sum()) else 0
                continue
            a = abs(s)
            _, e = mpmath.frexp(a)                           # a = f 2^e, f in [1/2, 1)
            q = mpmath.ldexp(1, max(int(e) - 8, -133))
            k = int(mpmath.floor(a / q))
            rem = a / q - k
            # never exactly 1/2 (SiLU(y) is transcendental for y != 0) unless
            # the precision fell short of separating SiLU(y) from y
            assert rem != half, f"y = {float(yy)!r}: SiLU not resolved from a bf16 midpoint"
            if rem > half:
                k += 1
            val = float(k * q)                               # at most 8 significant bits: exact
            bits = int(np.array([val], np.float32).view(np.uint32)[0] >> 16)
            out[i] = bits | (0x8000 if s < 0 else 0)
    return out


def assert_codes_exact(codes: np.ndarray, y: np.ndarray, rel_doubt: float = 2.0 ** -40):
    """bf16 codes of SiLU(y) must be its correct rounding.  Where the double
    value lies farther than ``rel_doubt`` (relative) from a rounding boundary,
    numpy's double evaluation decides; the closer ones are decided in 60 digits."""
    codes = np.asarray(codes, np.uint16).ravel()
    y = np.asarray(y, np.float64).ravel()
    s = y * expit(y)
    want = bf16_rne(s)
    close = np.flatnonzero(bf16_midpoint_distance(s) <= rel_doubt)
    if close.size:
        want[close] = silu_codes_exact(y[close])
    bad = np.flatnonzero(codes != want)
    assert bad.size == 0, (f"{bad.size} of {codes.size} codes are not the correct rounding: "
                           f"y {y[bad][:4]}, got {codes[bad][:4]}, want {want[bad][:4]}")


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
