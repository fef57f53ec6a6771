"""Pins of the oracle's gradients (oracle.recurrent_bwd) against what the
mathematics fixes, independently of the gradient code itself:

  * five-point finite differences of the FORWARD oracle: the loss
    L = <dO, o> + <dS_out, S_out> is a polynomial of degree three along any
    line through (q, k, v, S_in), and the five-point stencil differentiates
    polynomials up to degree four exactly, so the directional derivative
    must match <grad, direction> to rounding;
  * Euler's theorem for homogeneous functions: o is linear in q, and
    (o, S_out) is linear in (v, S_in) and in (k, S_in) jointly, so
    <dq, q> = <dO, o> and <dk, k> + <dS_in, S_in> = <dv, v> + <dS_in, S_in> = L;
  * textbook special cases: gamma = 1 without rotation is causal linear
    attention (dQ = tril(dO V^T) K, dK = tril(dO V^T)^T Q,
    dV = tril(Q K^T)^T dO); gamma = 0 keeps only each token's own term;
  * a two-token example worked by hand (tests/golden/).

The forward they differentiate is the recurrent form of
hwhale.com/article/285883 (S_n = gamma S_{n-1} + K_n^T V_n, O_n = Q_n S_n)
with the xPos/RoPE rotation and the first two normalisations, which the
forward pins in test_oracle_pins.py tie to the page.  A last test plants
mistakes in copies of the gradient code and checks that a pin catches each.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import NORM_DROW, NORM_SCALE, Problem

TWO_NORMS = NORM_SCALE | NORM_DROW


def rnd(g, *shape):
    return g.standard_normal(shape)


def case(seed=0, B=1, H=2, N=9, dk=6, dv=5, gam=(0.9, 0.6), rotate=True, pos0=3,
         flags=TWO_NORMS, with_S=True, with_dS=True):
    g = np.random.default_rng(seed)
    p = Problem(B, H, N, dk, dv, list(gam), rotate=rotate, pos0=pos0, norm_flags=flags,
                gn_eps=-1.0)
    x = dict(q=rnd(g, B, H, N, dk), k=rnd(g, B, H, N, dk), v=rnd(g, B, H, N, dv),
             S=rnd(g, B, H, dk, dv) if with_S else np.zeros((B, H, dk, dv)))
    up = dict(dO=rnd(g, B, H, N, dv), dS=rnd(g, B, H, dk, dv) if with_dS else None)
    return p, x, up


def loss(p, x, up):
    o, S_out, _ = oracle.recurrent(p, x["q"], x["k"], x["v"], S_in=x["S"])
    L = float(np.sum(up["dO"] * o))
    if up["dS"] is not None:
        L += float(np.sum(up["dS"] * S_out))
    return L


def grads(p, x, up):
    dq, dk, dv, dS = oracle.recurrent_bwd(p, x["q"], x["k"], x["v"], up["dO"],
                                          S_in=x["S"], dS_out=up["dS"])
    return dict(q=dq, k=dk, v=dv, S=dS)


def five_point(f, h):
    return (8.0 * (f(h) - f(-h)) - (f(2 * h) - f(-2 * h))) / (12.0 * h)


@pytest.mark.parametrize("which", ["q", "k", "v", "S", "all"])
@pytest.mark.parametrize("rotate,flags", [(True, TWO_NORMS), (False, 0), (True, NORM_SCALE)])
def test_gradient_matches_finite_differences(which, rotate, flags):
    p, x, up = case(seed=11, rotate=rotate, flags=flags)
    gr = grads(p, x, up)
    dirs = {n: np.random.default_rng(100 + i).standard_normal(x[n].shape)
            for i, n in enumerate(x)}
    use = list(x) if which == "all" else [which]

    def f(h):
        return loss(p, {n: x[n] + (h * dirs[n] if n in use else 0.0) for n in x}, up)

    fd = five_point(f, 0.5)
    an = sum(float(np.sum(gr[n] * dirs[n])) for n in use)
    assert abs(fd - an) <= 1e-9 * max(1.0, abs(an)), (which, fd, an)


@pytest.mark.parametrize("with_S,with_dS", [(True, True), (False, True), (True, False)])
def test_euler_identities(with_S, with_dS):
    p, x, up = case(seed=21, N=17, dk=8, dv=7, gam=(0.97, 1.0), pos0=40,
                    with_S=with_S, with_dS=with_dS)
    gr = grads(p, x, up)
    o, S_out, _ = oracle.recurrent(p, x["q"], x["k"], x["v"], S_in=x["S"])
    Lo = float(np.sum(up["dO"] * o))
    L = Lo + (float(np.sum(up["dS"] * S_out)) if up["dS"] is not None else 0.0)
    sS = float(np.sum(gr["S"] * x["S"]))
    tol = 1e-11 * max(1.0, abs(L))
    assert abs(float(np.sum(gr["q"] * x["q"])) - Lo) <= tol
    assert abs(float(np.sum(gr["k"] * x["k"])) + sS - L) <= tol
    assert abs(float(np.sum(gr["v"] * x["v"])) + sS - L) <= tol


def test_gamma_one_is_causal_linear_attention_backward():
    p, x, up = case(seed=31, B=1, H=1, N=12, dk=5, dv=4, gam=(1.0,), rotate=False,
                    pos0=0, flags=0, with_S=False, with_dS=False)
    gr = grads(p, x, up)
    Q, K, V, dO = x["q"][0, 0], x["k"][0, 0], x["v"][0, 0], up["dO"][0, 0]
    M = np.tril(np.ones((12, 12)))
    P = M * (dO @ V.T)
    assert np.max(np.abs(gr["q"][0, 0] - P @ K)) < 1e-12
    assert np.max(np.abs(gr["k"][0, 0] - P.T @ Q)) < 1e-12
    assert np.max(np.abs(gr["v"][0, 0] - (M * (Q @ K.T)).T @ dO)) < 1e-12
    # With no upstream state gradient the entry-state gradient is sum_n q_n^T dO_n.
    assert np.max(np.abs(gr["S"][0, 0] - Q.T @ dO)) < 1e-12


def test_gamma_zero_keeps_each_tokens_own_term():
    p, x, up = case(seed=41, B=2, H=1, N=6, dk=4, dv=3, gam=(0.0,), rotate=False,
                    pos0=0, flags=0)
    gr = grads(p, x, up)
    q, k, v, dO, dS = x["q"], x["k"], x["v"], up["dO"], up["dS"]
    w = np.sum(dO * v, axis=-1, keepdims=True)        # dO_n . v_n
    s = np.sum(q * k, axis=-1, keepdims=True)         # q_n . k_n
    dq, dk, dv = w * k, w * q, s * dO
    # The last token also feeds the final state S_out = k_{N-1}^T v_{N-1}.
    dk[:, :, -1] += np.einsum("bhae,bhe->bha", dS, v[:, :, -1])
    dv[:, :, -1] += np.einsum("bha,bhae->bhe", k[:, :, -1], dS)
    for a, b in [(gr["q"], dq), (gr["k"], dk), (gr["v"], dv)]:
        assert np.max(np.abs(a - b)) < 1e-12
    assert np.max(np.abs(gr["S"])) == 0.0


def test_rejects_what_it_does_not_cover():
    p, x, up = case()
    p.norm_flags = oracle.NORM_RSUM
    with pytest.raises(ValueError):
        grads(p, x, up)
    p.norm_flags, p.gn_eps = 0, 1e-6
    with pytest.raises(ValueError):
        grads(p, x, up)


# Planted mistakes in the gradient code: (description, text, replacement).
MUTANTS = [
    ("reverse carry not decayed",
     "for (size_t i = 0; i < G.size(); ++i) G[i] *= g;",
     "for (size_t i = 0; i < G.size(); ++i) G[i] *= 1.0;"),
    ("forward sweep without decay",
     "S[(size_t)a * dV + e] = g * S[(size_t)a * dV + e] + kn[a] * vn[e];",
     "S[(size_t)a * dV + e] = S[(size_t)a * dV + e] + kn[a] * vn[e];"),
    ("back-rotation sign", "y[2 * j + 1] = b * cs - a * sn;", "y[2 * j + 1] = b * cs + a * sn;"),
    ("dq without the row factor", "dqr[(size_t)n * dK + a] = sn * dot(",
     "dqr[(size_t)n * dK + a] = dot("),
    ("dv from a shifted column", "acc += kn[a] * G[(size_t)a * dV + e];",
     "acc += kn[a] * G[(size_t)a * dV + (e + 1) % dV];"),
    ("entry-state gradient one decay short",
     "dS_in[so + i] = G[i];", "dS_in[so + i] = G[i] / (g > 0.0 ? g : 1.0);"),
    ("q gradient added to G after use",
     "G[(size_t)a * dV + e] += sn * qn[a] * don[e];",
     "G[(size_t)a * dV + e] += 0.0 * sn * qn[a] * don[e];"),
]

PINS = [
    lambda: test_hand_derived_two_token_gradients(),
    lambda: test_gradient_matches_finite_differences("all", True, TWO_NORMS),
    lambda: test_gradient_matches_finite_differences("S", True, TWO_NORMS),
    lambda: test_euler_identities(True, True),
    test_gamma_one_is_causal_linear_attention_backward,
    test_gamma_zero_keeps_each_tokens_own_term,
]


@pytest.mark.parametrize("desc,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_gradient_mistakes_are_caught(desc, find, repl):
    here = os.path.dirname(oracle.__file__)
    src = open(os.path.join(here, "retention_oracle.cpp")).read()
    assert src.count(find) == 1, desc
    tmp = tempfile.mkdtemp(prefix="orc_bwd_mut_")
    try:
        shutil.copy(os.path.join(here, "retention_oracle.h"), tmp)
        with open(os.path.join(tmp, "m.cpp"), "w") as f:
            f.write(src.replace(find, repl, 1))
        so = os.path.join(tmp, "libm.so")
        subprocess.run(["g++", "-O1", "-fPIC", "-shared", "-std=c++17", "-o", so,
                        os.path.join(tmp, "m.cpp")], check=True, capture_output=True)
        caught = False
        with oracle.use_library(so):
            for pin in PINS:
                try:
                    pin()
                except AssertionError:
                    caught = True
                    break
        assert caught, f"planted mistake not caught: {desc}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def test_hand_derived_two_token_gradients():
    """tests/golden/backward_two_tokens_hand.txt: a two-token example worked
    by hand (derivation in the file)."""
    path = os.path.join(os.path.dirname(__file__), "golden", "backward_two_tokens_hand.txt")
    want = {}
    for line in open(path):
        if line.startswith("#") or "|" not in line:
            continue
        name, vals = (s.strip() for s in line.split("|"))
        want[name] = np.array([float(x) for x in vals.split()])
    p = Problem(1, 1, 2, 2, 1, 0.5, rotate=False, norm_flags=0, gn_eps=-1.0)
    q = np.array([[1.0, 0.0], [0.0, 1.0]])[None, None]
    k = np.array([[1.0, 1.0], [2.0, 0.0]])[None, None]
    v = np.array([[3.0], [-1.0]])[None, None]
    dO = np.array([[1.0], [2.0]])[None, None]
    dq, dk, dv, dS = oracle.recurrent_bwd(p, q, k, v, dO)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv), ("dS_in", dS)):
        assert np.max(np.abs(got.ravel() - want[name])) < 1e-15, name
