"""Pins of the RetNet-block oracle (oracle.msr: layernorm, gelu,
retnet_block) against what the mathematics fixes:

  * LayerNorm: every output row (with unit gain, zero bias) has mean 0 and
    mean square var / (var + eps); it ignores a constant added to a row; the
    gain and bias act per feature;
  * GELU = x Phi(x): gelu(x) - gelu(-x) = x (Phi(x) + Phi(-x) = 1),
    gelu(0) = 0, gelu(1) = Phi(1) = 0.8413447460685429 (standard normal
    table), gelu(-8) ~ 0, gelu(8) ~ 8;
  * the block with W_O = 0 and W2 = 0 is the identity (both skip
    connections alone); with W2 = 0 it is X + MSR(LN(X)), the pinned-by-parts
    MSR oracle; with W_O = 0 it is X + FFN(LN(X)) computed by direct loops.

  * a one-token block worked by hand from the definitions
    (tests/golden/block_one_token_hand.txt), which four planted mistakes in
    the block's composition fail (FFN on LN(X) instead of LN(Y), GELU after
    W2, no second skip connection, the skips swapped for the LayerNorm
    inputs).
"""
import math
import os

import numpy as np
import pytest

from oracle.msr import gelu, layernorm, msr_layer, retnet_block


def test_layernorm_moments_and_shift_invariance():
    g = np.random.default_rng(1)
    x = g.standard_normal((3, 5, 16)) * 3.0 + 2.0
    eps = 1e-5
    y = layernorm(x, np.ones(16), np.zeros(16), eps)
    var = x.var(axis=-1)
    assert np.max(np.abs(y.mean(axis=-1))) < 1e-14
    assert np.max(np.abs((y ** 2).mean(axis=-1) - var / (var + eps))) < 1e-13
    assert np.max(np.abs(layernorm(x + 7.5, np.ones(16), np.zeros(16), eps) - y)) < 1e-12
    w, b = g.standard_normal(16), g.standard_normal(16)
    assert np.max(np.abs(layernorm(x, w, b, eps) - (y * w + b))) < 1e-14


def test_layernorm_hand_example():
    # Row (1, 2, 3, 6): mean 3, deviations (-2, -1, 0, 3), variance 14/4 = 3.5.
    y = layernorm(np.array([[1.0, 2.0, 3.0, 6.0]]), np.ones(4), np.zeros(4), 0.0)
    assert np.max(np.abs(y - np.array([-2.0, -1.0, 0.0, 3.0]) / math.sqrt(3.5))) < 1e-15


def test_gelu_values_and_symmetry():
    x = np.linspace(-6, 6, 97)
    assert np.max(np.abs(gelu(x) - gelu(-x) - x)) < 1e-14
    assert gelu(np.array([0.0]))[0] == 0.0
    assert abs(gelu(np.array([1.0]))[0] - 0.8413447460685429) < 1e-15
    assert abs(gelu(np.array([-8.0]))[0]) < 1e-13
    assert abs(gelu(np.array([8.0]))[0] - 8.0) < 1e-13


def _weights(seed, d, H, dk, dv, dff, std=0.3):
    g = np.random.default_rng(seed)
    W = dict(WQ=g.standard_normal((d, H * dk)) * std, WK=g.standard_normal((d, H * dk)) * std,
             WV=g.standard_normal((d, H * dv)) * std, WG=g.standard_normal((d, H * dv)) * std,
             WO=g.standard_normal((H * dv, d)) * std, W1=g.standard_normal((d, dff)) * std,
             W2=g.standard_normal((dff, d)) * std)
    ln = dict(ln1_w=1 + 0.1 * g.standard_normal(d), ln1_b=0.1 * g.standard_normal(d),
              ln2_w=1 + 0.1 * g.standard_normal(d), ln2_b=0.1 * g.standard_normal(d))
    return W, ln


def _block(X, W, ln, **kw):
    return retnet_block(X, ln["ln1_w"], ln["ln1_b"], W["WQ"], W["WK"], W["WV"], W["WG"],
                        W["WO"], ln["ln2_w"], ln["ln2_b"], W["W1"], W["W2"], **kw)


KW = dict(H=2, dk=4, dv=6, gamma=[0.9, 0.6], chunk=3, ln_eps=1e-5, norm_flags=7, gn_eps=1e-6)


def test_block_reduces_to_its_parts():
    B, N, d, dff = 2, 7, 8, 16
    W, ln = _weights(3, d, 2, 4, 6, dff)
    X = np.random.default_rng(4).standard_normal((B, N, d))
    Z = dict(W, WO=np.zeros_like(W["WO"]), W2=np.zeros_like(W["W2"]))
    assert np.array_equal(_block(X, Z, ln, **KW), X)
    M = dict(W, W2=np.zeros_like(W["W2"]))
    msr = msr_layer(layernorm(X, ln["ln1_w"], ln["ln1_b"], 1e-5), W["WQ"], W["WK"], W["WV"],
                    W["WG"], W["WO"], H=2, dk=4, dv=6, gamma=[0.9, 0.6], chunk=3, norm_flags=7,
                    gn_eps=1e-6)
    assert np.max(np.abs(_block(X, M, ln, **KW) - (X + msr))) < 1e-12
    F = dict(W, WO=np.zeros_like(W["WO"]))
    ref = np.empty_like(X)
    for b in range(B):
        for n in range(N):
            row = X[b, n]
            mu = sum(row) / d
            var = sum((r - mu) ** 2 for r in row) / d
            xn = [(row[i] - mu) / math.sqrt(var + 1e-5) * ln["ln2_w"][i] + ln["ln2_b"][i]
                  for i in range(d)]
            h = [sum(xn[i] * W["W1"][i, j] for i in range(d)) for j in range(dff)]
            h = [t * 0.5 * (1 + math.erf(t / math.sqrt(2))) for t in h]
            for o in range(d):
                ref[b, n, o] = row[o] + sum(h[j] * W["W2"][j, o] for j in range(dff))
    assert np.max(np.abs(_block(X, F, ln, **KW) - ref)) < 1e-12


GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ONE = np.eye(2)


def _hand_block_expect():
    env = {"math": math}
    out = {}
    for line in open(os.path.join(GOLDEN, "block_one_token_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kind, name, expr = [c.strip() for c in line.split("|")]
        val = eval(expr, env)
        if kind == "let":
            env[name] = val
        else:
            out[int(name)] = val
    return np.array([out[0], out[1]])


def _hand_block_pins(block):
    X = np.array([[[1.0, -1.0]]])
    u1, z1 = np.ones(2), np.zeros(2)
    got = block(X, u1, z1, ONE, ONE, ONE, ONE, ONE, u1, z1, ONE, np.array([[1.0, 2.0], [0.0, 1.0]]),
                H=1, dk=2, dv=2, gamma=[0.5], chunk=1, ln_eps=1e-5, norm_flags=0, gn_eps=-1.0)
    assert np.max(np.abs(got[0, 0] - _hand_block_expect())) < 1e-14


def test_block_hand_example():
    _hand_block_pins(retnet_block)


def _block_mutant(kind):
    def block(X, ln1_w, ln1_b, WQ, WK, WV, WG, WO, ln2_w, ln2_b, W1, W2, *, H, dk, dv, gamma,
              chunk, ln_eps, norm_flags, gn_eps):
        M = msr_layer(layernorm(X, ln1_w, ln1_b, ln_eps), WQ, WK, WV, WG, WO, H=H, dk=dk, dv=dv,
                      gamma=gamma, chunk=chunk, norm_flags=norm_flags, gn_eps=gn_eps)
        Y = M + X
        src = X if kind == "FFN on LN(X)" else Y
        if kind == "GELU after W2":
            F = gelu(layernorm(src, ln2_w, ln2_b, ln_eps) @ W1 @ W2)
        else:
            F = gelu(layernorm(src, ln2_w, ln2_b, ln_eps) @ W1) @ W2
        if kind == "no second skip":
            return F
        if kind == "skips swapped":
            return F + X
        return F + Y
    return block


@pytest.mark.parametrize("kind", ["FFN on LN(X)", "GELU after W2", "no second skip",
                                  "skips swapped"])
def test_block_mutants_are_caught(kind):
    with pytest.raises(AssertionError):
        _hand_block_pins(_block_mutant(kind))


def test_block_mutant_harness_is_faithful():
    _hand_block_pins(_block_mutant("none"))
