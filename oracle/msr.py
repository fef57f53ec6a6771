"""Gated multi-scale retention layer and the RetNet block, float64 -- TEST
INFRASTRUCTURE ONLY.

MSR(X) = (swish(X W_G) (.) Y) W_O with Y = GroupNorm_h(head_1, ..., head_H)
and head_h = Retention(X, gamma_h), Q = (X W_Q) (.) Theta,
K = (X W_K) (.) conj(Theta), V = X W_V
(m0nads.wordpress.com "A dubious successor to Transformer", section "Last
piece: Gated Multi-Scale Retention"; m.sdkjxy.cn RetNet walkthrough,
"Gated Multi-Scale Retention").  swish(x) = x * sigmoid(x).  The projections
are numpy float64 matmuls (a library primitive); retention is the oracle's
chunkwise form, whose equality with the parallel form the CPU tests pin.

Pinned by a two-token example worked by hand from the definitions above
(tests/golden/msr_two_tokens_hand.txt: projections, gate and output
projection around the hand-worked retention example), with six planted
mistakes that it catches, and by direct loops on a small shape.
"""
from __future__ import annotations

import numpy as np

from . import Problem, chunkwise


def swish(x):
    return x / (1.0 + np.exp(-x))


def msr_layer(X, WQ, WK, WV, WG, WO, *, H, dk, dv, gamma, chunk,
              theta_base=10000.0, norm_flags=0, gn_eps=1e-6, pos0=0, threads=0,
              S_in=None, z_in=None, return_state=False):
    """X [B, N, d]; W_Q, W_K [d, H dk]; W_V, W_G [d, H dv]; W_O [H dv, d].
    S_in [B, H, dk, dv] / z_in [B, H, dk]: the retention state entering the
    call (None = zeros); with return_state the result is (out, S_out, z_out)."""
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
    o, S_out, z_out = chunkwise(p, chunk, q, k, v, S_in=S_in, z_in=z_in)
    Y = o.transpose(0, 2, 1, 3).reshape(B, N, H * dv)
    out = (swish(G) * Y) @ np.asarray(WO, dtype=np.float64)
    return (out, S_out, z_out) if return_state else out


def layernorm(x, w, b, eps):
    """LayerNorm over the last axis: (x - mean) / sqrt(var + eps) * w + b, with
    the biased variance (the mean of squared deviations)."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(w, np.float64) + np.asarray(b, np.float64)


def gelu(x):
    """x * Phi(x), Phi the standard normal distribution function, written with
    the error function: Phi(x) = (1 + erf(x / sqrt(2))) / 2."""
    from scipy.special import erf
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def retnet_block(X, ln1_w, ln1_b, WQ, WK, WV, WG, WO, ln2_w, ln2_b, W1, W2, *, H, dk, dv,
                 gamma, chunk, ln_eps=1e-5, theta_base=10000.0, norm_flags=0, gn_eps=1e-6,
                 pos0=0, threads=0, S_in=None, z_in=None, return_state=False):
    """One RetNet block (m0nads.wordpress.com "A dubious successor to
    Transformer", section "Overall architecture": MSR and FFN, each after a
    LayerNorm and each with a skip connection):
        Y = MSR(LN(X)) + X,   X' = FFN(LN(Y)) + Y,   FFN(x) = gelu(x W1) W2.
    The pages name the FFN but not its activation; GELU is the reading taken."""
    X = np.asarray(X, dtype=np.float64)
    M, S_out, z_out = msr_layer(layernorm(X, ln1_w, ln1_b, ln_eps), WQ, WK, WV, WG, WO, H=H,
                                dk=dk, dv=dv, gamma=gamma, chunk=chunk, theta_base=theta_base,
                                norm_flags=norm_flags, gn_eps=gn_eps, pos0=pos0,
                                threads=threads, S_in=S_in, z_in=z_in, return_state=True)
    Y = M + X
    F = gelu(layernorm(Y, ln2_w, ln2_b, ln_eps) @ np.asarray(W1, np.float64))
    out = F @ np.asarray(W2, np.float64) + Y
    return (out, S_out, z_out) if return_state else out


BLOCK_WEIGHTS = ("ln1_w", "ln1_b", "WQ", "WK", "WV", "WG", "WO", "ln2_w", "ln2_b", "W1", "W2")


def retnet_stack(X, layers, *, states=None, pos0=0, **kw):
    """A stack of RetNet blocks over the tokens of X [B, N, d] (m0nads.wordpress.com,
    "Overall architecture": L stacked blocks).  `layers` is a list of dicts
    with the keys of BLOCK_WEIGHTS; `states` a list of (S, z) per layer
    (None = zeros).  Returns (out, new states).  Called with N = 1 it is one
    decode step of the whole stack; the recurrent state of every layer is
    carried in `states`."""
    out = np.asarray(X, dtype=np.float64)
    new = []
    for li, W in enumerate(layers):
        S_in, z_in = (None, None) if states is None else states[li]
        out, S, z = retnet_block(out, *(W[n] for n in BLOCK_WEIGHTS), pos0=pos0, S_in=S_in,
                                 z_in=z_in, return_state=True, **kw)
        new.append((S, z))
    return out, new
