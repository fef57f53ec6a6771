"""Gated multi-scale retention layer, float64 -- TEST INFRASTRUCTURE ONLY.

MSR(X) = (swish(X W_G) (.) Y) W_O with Y = GroupNorm_h(head_1, ..., head_H)
and head_h = Retention(X, gamma_h), Q = (X W_Q) (.) Theta,
K = (X W_K) (.) conj(Theta), V = X W_V
(m0nads.wordpress.com "A dubious successor to Transformer", section "Last
piece: Gated Multi-Scale Retention"; m.sdkjxy.cn RetNet walkthrough,
"Gated Multi-Scale Retention").  swish(x) = x * sigmoid(x).  The projections
are numpy float64 matmuls (a library primitive); retention is the oracle's
chunkwise form, whose equality with the parallel form the CPU tests pin.

Parity unpinned beyond that: the pages print no worked MSR example, so the
layer is checked for self-consistency only (the matmul steps against direct
loops on small shapes, the retention step through the pinned forms).
"""
from __future__ import annotations

import numpy as np

from . import Problem, chunkwise


def swish(x):
    return x / (1.0 + np.exp(-x))


def msr_layer(X, WQ, WK, WV, WG, WO, *, H, dk, dv, gamma, chunk,
              theta_base=10000.0, norm_flags=0, gn_eps=1e-6, pos0=0, threads=0):
    """X [B, N, d]; W_Q, W_K [d, H dk]; W_V, W_G [d, H dv]; W_O [H dv, d]."""
    X = np.asarray(X, dtype=np.float64)
    B, N, _ = X.shape
    Q = X @ np.asarray(WQ, dtype=np.float64)
    K = X @ np.asarray(WK, dtype=np.float64)
    V = X @ np.asarray(WV, dtype=np.float64)
    G = X @ np.asarray(WG, dtype=np.float64)
    q = Q.reshape(B, N, H, dk).transpose(0, 2, 1, 3)
    k = K.reshape(B, N, H, dk).transpose(0, 2, 1, 3)
    v = V.reshape(B, N, H, dv).transpose(0, 2, 1, 3)
    p = Problem(B, H, N, dk, dv, gamma, theta_base=theta_base, pos0=pos0,
                rotate=True, norm_flags=norm_flags, gn_eps=gn_eps, threads=threads)
    o, _, _ = chunkwise(p, chunk, q, k, v)
    Y = o.transpose(0, 2, 1, 3).reshape(B, N, H * dv)
    return (swish(G) * Y) @ np.asarray(WO, dtype=np.float64)
