"""Pins of the multi-layer oracle (oracle.msr.retnet_stack) for decode with
per-layer states: the recurrent and chunkwise representations are one
function (hwhale.com/article/285883), so a stack of blocks run token by token
with each layer's (S, z) carried must equal the stack run over the whole
sequence at once, and a prefill followed by decode steps must equal both.
Rotation positions and the decay-row normalisation follow the absolute
position pos0 + n in every call."""
import numpy as np

from oracle.msr import BLOCK_WEIGHTS, retnet_stack

KW = dict(H=2, dk=4, dv=6, gamma=[0.9, 0.7], chunk=4, ln_eps=1e-5, norm_flags=7, gn_eps=1e-6)


def layers(seed, n_layers, d=8, dff=12, std=0.3):
    g = np.random.default_rng(seed)
    shapes = dict(WQ=(d, 8), WK=(d, 8), WV=(d, 12), WG=(d, 12), WO=(12, d), W1=(d, dff),
                  W2=(dff, d))
    out = []
    for _ in range(n_layers):
        W = {n: g.standard_normal(s) * std for n, s in shapes.items()}
        for n in ("ln1", "ln2"):
            W[n + "_w"] = 1 + 0.1 * g.standard_normal(d)
            W[n + "_b"] = 0.1 * g.standard_normal(d)
        assert set(W) == set(BLOCK_WEIGHTS)
        out.append(W)
    return out


def test_token_by_token_equals_whole_sequence():
    B, N, d = 2, 11, 8
    L = layers(5, 3)
    X = np.random.default_rng(6).standard_normal((B, N, d))
    full, st_full = retnet_stack(X, L, **KW)
    states, outs = None, []
    for t in range(N):
        o, states = retnet_stack(X[:, t:t + 1], L, states=states, pos0=t, **KW)
        outs.append(o)
    assert np.max(np.abs(np.concatenate(outs, axis=1) - full)) < 1e-10
    for (S1, z1), (S2, z2) in zip(states, st_full):
        assert np.max(np.abs(S1 - S2)) < 1e-10 and np.max(np.abs(z1 - z2)) < 1e-10


def test_prefill_then_decode_equals_whole_sequence():
    B, N, P, d = 1, 13, 9, 8
    L = layers(7, 2)
    X = np.random.default_rng(8).standard_normal((B, N, d))
    full, _ = retnet_stack(X, L, **KW)
    pre, states = retnet_stack(X[:, :P], L, **KW)
    outs = [pre]
    for t in range(P, N):
        o, states = retnet_stack(X[:, t:t + 1], L, states=states, pos0=t, **KW)
        outs.append(o)
    assert np.max(np.abs(np.concatenate(outs, axis=1) - full)) < 1e-10


def test_empty_stack_is_identity():
    X = np.random.default_rng(9).standard_normal((1, 3, 8))
    out, states = retnet_stack(X, [], **KW)
    assert np.array_equal(out, X) and states == []
