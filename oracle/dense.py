"""Matrix-form brute force of the Gated Residual read/write, fp64 numpy (tiny sizes only).

Test infrastructure only. A second formulation of the same definition as gr_oracle.c, used to
cross-check it: the whole branch stack is flattened with an explicit vec (branch-major), the
projections are full matrix products over all tokens at once, and unvec is a reshape.
Source: "【论文解读】 Qwen3.8 Flash Next", §二.4, eq rms, eq gate, eq use_gate, eq s, eq write.
"""
from __future__ import annotations

import numpy as np


def _vec(M: np.ndarray) -> np.ndarray:
    """[n, nb, D] -> [n, nb*D], branch-major (branch i occupies entries i*D .. i*D+D-1)."""
    n, nb, D = M.shape
    out = np.empty((n, nb * D))
    for i in range(nb):
        out[:, i * D:(i + 1) * D] = M[:, i, :]
    return out


def _unvec(v: np.ndarray, nb: int) -> np.ndarray:
    n, K = v.shape
    D = K // nb
    return np.stack([v[:, i * D:(i + 1) * D] for i in range(nb)], axis=1)


def _logistic(a: np.ndarray) -> np.ndarray:
    out = np.empty_like(a)
    pos = a >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-a[pos]))
    e = np.exp(a[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def read(R, gamma, w_down, w_up, w_write, eps=1e-6):
    R = np.asarray(R, dtype=np.float64)
    n, nb, D = R.shape
    rms = np.sqrt(np.mean(R * R, axis=2, keepdims=True) + eps)          # [n, nb, 1]
    Rhat = R / rms * np.asarray(gamma, dtype=np.float64)[None]           # eq rms
    v = _vec(Rhat)                                                       # [n, nb*D]
    Wd = np.asarray(w_down, dtype=np.float64)
    Wu = np.asarray(w_up, dtype=np.float64)
    Ww = np.asarray(w_write, dtype=np.float64)
    z = (v @ Wd.T) / nb                                                  # [n, r]
    h = z * _logistic(z)                                                 # SiLU
    G = _unvec(_logistic(h @ Wu.T), nb)                                  # eq gate
    x = (G * Rhat).sum(axis=1) / nb                                      # eq use_gate
    s = 2.0 * _logistic((v @ Ww.T) / nb)                                 # eq s
    return x, s


def write(R, y, s):
    R = np.asarray(R, dtype=np.float64)
    return R + np.asarray(s, dtype=np.float64)[:, :, None] * np.asarray(y, np.float64)[:, None]
