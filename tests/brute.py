"""Brute-force token-by-token Mamba-2 recurrence in float64 (test-only).

This is the plain state-space recurrence, run one token at a time:
    S <- exp(A dt') S + dt' x (outer) B,      y = S C + D x
It shares nothing with the oracle's checkpoint-plus-replay closed form; the
two must agree (up to the oracle's fp32 cumulative sums and dt').
"""
import numpy as np


def softplus64(v):
    v = np.asarray(v, np.float64)
    return np.where(v > 20.0, v, np.log1p(np.exp(np.minimum(v, 20.0))))


def bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def recurrence(S0, live, new, A, D):
    """S0 [64][128] float64.  live: list of (x[64], B[128], dt') already
    accepted (no outputs).  new: list of (x[64], B[128], dt', C[128]).
    Returns (ys [T][64], state after live tokens, state after all tokens)."""
    S = np.array(S0, np.float64, copy=True)
    for x, B, dtp in live:
        S = np.exp(A * dtp) * S + dtp * np.outer(x, B)
    S_live = S.copy()
    ys = []
    for x, B, dtp, C in new:
        S = np.exp(A * dtp) * S + dtp * np.outer(x, B)
        ys.append(S @ C + D * x)
    return np.array(ys), S_live, S
