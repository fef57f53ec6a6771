"""Pins of the float64 oracle against what the pages and mathematics fix.

Each pin checks the oracle against something other than itself:
  * algebraic identities the pages state: the parallel, recurrent and
    chunkwise representations are one function (hwhale.com/article/285883,
    parallel / recurrent / chunkwise equations);
  * the diagonalised closed form with complex arithmetic (same page, closed
    form O_n = sum_m gamma^(n-m) (Q_n e^{in theta})(K_m e^{im theta})^dagger V_m);
  * GroupNorm's invariance to row scalings (same page, the claim that the
    three normalisations do not change the GroupNorm output);
  * textbook special cases: gamma=1 without rotation is causal linear
    attention; gamma=0 keeps only the diagonal; N=1;
  * hand-derived fixtures under tests/golden/;
  * the geometric-series closed form of the decay row sum.
A final test plants mistakes in copies of the oracle source and checks that
some pin catches each one.
"""
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import NORM_ALL, Problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def relerr(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def small_inputs(B=2, H=2, N=13, dk=6, dv=5, seed=0):
    return rnd(seed, B, H, N, dk), rnd(seed + 1, B, H, N, dk), rnd(seed + 2, B, H, N, dv)


@pytest.mark.parametrize("flags", [0, 1, 2, 4, NORM_ALL])
@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("pos0", [0, 5])
@pytest.mark.parametrize("gn_eps", [-1.0, 1e-6])
def test_three_forms_agree(flags, rotate, pos0, gn_eps):
    q, k, v = small_inputs()
    p = Problem(2, 2, 13, 6, 5, [0.9, 0.6], theta_base=10000.0, pos0=pos0,
                rotate=rotate, norm_flags=flags, gn_eps=gn_eps)
    o_par = oracle.parallel(p, q, k, v)
    o_rec, S_rec, z_rec = oracle.recurrent(p, q, k, v)
    assert relerr(o_rec, o_par) < 1e-12
    for chunk in (1, 3, 4, 13, 16):
        o_ch, S_ch, z_ch = oracle.chunkwise(p, chunk, q, k, v)
        assert relerr(o_ch, o_par) < 1e-12, chunk
        assert relerr(S_ch, S_rec) < 1e-12, chunk
        assert relerr(z_ch, z_rec) < 1e-12, chunk


def test_state_is_decayed_outer_product_sum():
    """S_N = sum_m gamma^(N-1-m) K'_m^T V_m (the recurrence unrolled, with
    zero initial state) and z_N = sum_m gamma^(N-1-m) K'_m."""
    q, k, v = small_inputs(B=1, H=1, N=9, dk=4, dv=3)
    g = 0.7
    p = Problem(1, 1, 9, 4, 3, g, rotate=True, gn_eps=-1.0)
    _, S, z = oracle.chunkwise(p, 4, q, k, v)
    kr = oracle.rotate(p, k, 4)[0, 0]
    w = g ** (8 - np.arange(9))
    S_ref = np.einsum("m,ma,me->ae", w, kr, v[0, 0])
    assert relerr(S[0, 0], S_ref) < 1e-13
    assert relerr(z[0, 0], w @ kr) < 1e-13


def test_state_passing_splits_the_sequence():
    """Running [0,a) then [a,N) with the carried state and pos0 = a equals one
    run over [0,N) (outputs and final state)."""
    q, k, v = small_inputs(B=1, H=2, N=20, dk=4, dv=6, seed=3)
    kw = dict(theta_base=100.0, rotate=True, norm_flags=NORM_ALL, gn_eps=1e-6)
    full = Problem(1, 2, 20, 4, 6, [0.95, 0.5], **kw)
    o, S, z = oracle.chunkwise(full, 8, q, k, v)
    a = 7
    p1 = Problem(1, 2, a, 4, 6, [0.95, 0.5], **kw)
    p2 = Problem(1, 2, 20 - a, 4, 6, [0.95, 0.5], pos0=a, **kw)
    o1, S1, z1 = oracle.chunkwise(p1, 8, q[:, :, :a], k[:, :, :a], v[:, :, :a])
    o2, S2, z2 = oracle.recurrent(p2, q[:, :, a:], k[:, :, a:], v[:, :, a:], S1, z1)
    assert relerr(np.concatenate([o1, o2], axis=2), o) < 1e-12
    assert relerr(S2, S) < 1e-12 and relerr(z2, z) < 1e-12


@pytest.mark.parametrize("flags", [0, NORM_ALL])
def test_real_rotation_matches_complex_closed_form(flags):
    q, k, v = small_inputs(B=1, H=2, N=11, dk=8, dv=4, seed=7)
    p = Problem(1, 2, 11, 8, 4, [0.8, 1.0], theta_base=10.0, pos0=3,
                rotate=True, norm_flags=flags, gn_eps=-1.0)
    assert relerr(oracle.parallel(p, q, k, v), oracle.closed_form(p, q, k, v)) < 1e-12


def test_rotation_preserves_norm_and_relative_phase():
    """|Theta x| = |x| pairwise, and <Theta_t q, Theta_m k> depends on t-m only."""
    x = rnd(11, 1, 1, 6, 8)
    p = Problem(1, 1, 6, 8, 1, 0.5, theta_base=10000.0, pos0=2)
    xr = oracle.rotate(p, x, 8)
    assert np.allclose(np.hypot(xr[..., 0::2], xr[..., 1::2]),
                       np.hypot(x[..., 0::2], x[..., 1::2]), atol=1e-14)
    qv, kv = rnd(12, 8), rnd(13, 8)
    xs = np.stack([qv, kv, qv, kv])[None, None]          # positions 2,3,4,5
    r = oracle.rotate(Problem(1, 1, 4, 8, 1, 0.5, pos0=2), xs, 8)[0, 0]
    assert abs(r[0] @ r[1] - r[2] @ r[3]) < 1e-12        # both have t-m = -1


def test_rotation_frequencies_hand():
    """theta_j = base^(-2j/dk), pair (x_2j, x_2j+1) turned by t theta_j.
    dk=4, base=100: theta_0 = 1, theta_1 = 100^(-1/2) = 0.1; at t=10 the unit
    vectors (1,0) of both pairs turn by 10 rad and 1 rad."""
    x = np.array([1.0, 0.0, 1.0, 0.0])[None, None, None]
    p = Problem(1, 1, 1, 4, 1, 0.5, theta_base=100.0, pos0=10)
    y = oracle.rotate(p, x, 4)[0, 0, 0]
    exp = [math.cos(10.0), math.sin(10.0), math.cos(1.0), math.sin(1.0)]
    assert np.max(np.abs(y - exp)) < 1e-14
    # (0,1) turns to (-sin, cos): the counter-clockwise direction of e^{+i t theta}
    y = oracle.rotate(p, np.array([0.0, 1.0, 0.0, 1.0])[None, None, None], 4)[0, 0, 0]
    exp = [-math.sin(10.0), math.cos(10.0), -math.sin(1.0), math.cos(1.0)]
    assert np.max(np.abs(y - exp)) < 1e-14


def test_gamma_one_no_rotation_is_causal_linear_attention():
    q, k, v = small_inputs(B=1, H=1, N=10, dk=6, dv=4, seed=21)
    p = Problem(1, 1, 10, 6, 4, 1.0, rotate=False, gn_eps=-1.0)
    kv = np.cumsum(np.einsum("na,ne->nae", k[0, 0], v[0, 0]), axis=0)
    ref = np.einsum("na,nae->ne", q[0, 0], kv)
    for f in (oracle.parallel, oracle.closed_form):
        assert relerr(f(p, q, k, v)[0, 0], ref) < 1e-12
    assert relerr(oracle.recurrent(p, q, k, v)[0][0, 0], ref) < 1e-12
    assert relerr(oracle.chunkwise(p, 3, q, k, v)[0][0, 0], ref) < 1e-12


def test_gamma_zero_keeps_only_the_diagonal():
    """D = I: o_t = (Theta_t q_t . Theta_t k_t) v_t = (q_t . k_t) v_t, because
    equal rotations preserve the dot product."""
    q, k, v = small_inputs(B=1, H=1, N=7, dk=6, dv=3, seed=31)
    p = Problem(1, 1, 7, 6, 3, 0.0, rotate=True, pos0=4, gn_eps=-1.0)
    ref = np.einsum("na,na->n", q[0, 0], k[0, 0])[:, None] * v[0, 0]
    assert relerr(oracle.parallel(p, q, k, v)[0, 0], ref) < 1e-12
    assert relerr(oracle.recurrent(p, q, k, v)[0][0, 0], ref) < 1e-12
    assert relerr(oracle.chunkwise(p, 4, q, k, v)[0][0, 0], ref) < 1e-12


def test_single_token_is_groupnorm_of_signed_v():
    q, k, v = small_inputs(B=1, H=1, N=1, dk=4, dv=6, seed=41)
    p = Problem(1, 1, 1, 4, 6, 0.9, rotate=True, pos0=0, gn_eps=0.0, norm_flags=NORM_ALL)
    s = np.sign(q[0, 0, 0] @ k[0, 0, 0])
    x = v[0, 0, 0]
    ref = s * (x - x.mean()) / x.std()
    assert np.max(np.abs(oracle.parallel(p, q, k, v)[0, 0, 0] - ref)) < 1e-12


def test_groupnorm_removes_positive_row_scalings():
    """The three normalisations only rescale each row by a positive constant,
    so with eps=0 GroupNorm's output is the same with and without them; with
    eps=1e-6 the difference is bounded by eps / var."""
    q, k, v = small_inputs(B=1, H=2, N=12, dk=4, dv=8, seed=51)
    outs = {}
    for eps in (0.0, 1e-6):
        for flags in (0, NORM_ALL):
            p = Problem(1, 2, 12, 4, 8, [0.9, 0.99], rotate=True, norm_flags=flags,
                        gn_eps=eps)
            outs[(eps, flags)] = oracle.parallel(p, q, k, v)
    assert np.max(np.abs(outs[(0.0, 0)] - outs[(0.0, NORM_ALL)])) < 1e-10
    raw = oracle.parallel(Problem(1, 2, 12, 4, 8, [0.9, 0.99], rotate=True,
                                  norm_flags=NORM_ALL, gn_eps=-1.0), q, k, v)
    bound = 1e-6 / raw.var(axis=-1).min()
    assert np.max(np.abs(outs[(1e-6, 0)] - outs[(1e-6, NORM_ALL)])) < 2 * bound + 1e-12
    y = oracle.groupnorm(raw, 0.0)
    assert np.max(np.abs(oracle.groupnorm(3.7 * raw, 0.0) - y)) < 1e-12


@pytest.mark.parametrize("g", [0.0, 0.3, 0.9, 0.96875, 1.0 - 2.0 ** -20, 1.0])
def test_decay_row_sum_is_geometric_series(g):
    for n in (1, 2, 7, 64, 1000):
        # (1 - g^n)/(1 - g), evaluated without cancellation for g near 1
        if g == 1.0:
            closed = n
        elif g == 0.0:
            closed = 1.0
        else:
            closed = -math.expm1(n * math.log1p(-(1.0 - g))) / (1.0 - g)
        assert abs(oracle.decay_row_sum(g, n) - closed) <= 1e-12 * closed
    # and equals the literal row sum of the D matrix for pos0 = 0
    n = 9
    assert abs(oracle.decay_row_sum(g, n) - sum(g ** (n - i) for i in range(1, n + 1))) < 1e-12


def _golden_rows(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append([c.strip() for c in line.split("|")])
    return rows


def test_hand_derived_two_token_example():
    q = np.array([[1.0, 0.0], [0.0, 1.0]])[None, None]
    k = np.array([[1.0, 0.0], [1.0, 1.0]])[None, None]
    v = np.array([[2.0], [3.0]])[None, None]
    rows = _golden_rows("retention_dk2_hand.txt")
    assert len(rows) == 3
    for name, flags, pos0, expect in rows:
        exp = np.array([eval(e, {"math": math}) for e in expect.split(";")])
        p = Problem(1, 1, 2, 2, 1, 0.5, theta_base=10000.0, pos0=int(pos0),
                    rotate=True, norm_flags=int(flags), gn_eps=-1.0)
        for f in (oracle.parallel, oracle.closed_form):
            assert np.max(np.abs(f(p, q, k, v)[0, 0, :, 0] - exp)) < 1e-14, name
        assert np.max(np.abs(oracle.recurrent(p, q, k, v)[0][0, 0, :, 0] - exp)) < 1e-14
        assert np.max(np.abs(oracle.chunkwise(p, 1, q, k, v)[0][0, 0, :, 0] - exp)) < 1e-14
    # third normalisation active: o_0 = v_0 exactly
    p = Problem(1, 1, 1, 2, 1, 0.5, rotate=True, norm_flags=NORM_ALL, gn_eps=-1.0)
    o = oracle.parallel(p, np.array([[[[2.0, 0.0]]]]), np.array([[[[2.0, 0.0]]]]),
                        np.array([[[[2.0]]]]))
    assert abs(o[0, 0, 0, 0] - 2.0) < 1e-14


def test_hand_derived_negative_row_sum():
    """The third normalisation divides by |sum R| when the row sum is below
    -1 (tests/golden/retention_negative_rowsum_hand.txt)."""
    q = np.array([[1.0, 0.0], [-3.0, 0.0]])[None, None]
    k = np.array([[1.0, 0.0], [1.0, 0.0]])[None, None]
    v = np.array([[2.0], [3.0]])[None, None]
    rows = _golden_rows("retention_negative_rowsum_hand.txt")
    assert len(rows) == 3
    for name, flags, expect in rows:
        exp = np.array([eval(e, {"math": math}) for e in expect.split(";")])
        p = Problem(1, 1, 2, 2, 1, 0.5, theta_base=10000.0, rotate=True,
                    norm_flags=int(flags), gn_eps=-1.0)
        for f in (oracle.parallel, oracle.closed_form):
            assert np.max(np.abs(f(p, q, k, v)[0, 0, :, 0] - exp)) < 1e-14, name
        assert np.max(np.abs(oracle.recurrent(p, q, k, v)[0][0, 0, :, 0] - exp)) < 1e-14, name
        for chunk in (1, 2):
            got = oracle.chunkwise(p, chunk, q, k, v)[0][0, 0, :, 0]
            assert np.max(np.abs(got - exp)) < 1e-14, (name, chunk)


_MSR_HAND = dict(
    X=np.array([[[1.0, 0.0], [0.0, 1.0]]]),
    WQ=np.array([[1.0, 0.0], [0.0, 1.0]]),
    WK=np.array([[1.0, 0.0], [1.0, 1.0]]),
    WV=np.array([[2.0, 1.0], [3.0, -1.0]]),
    WG=np.array([[1.0, 2.0], [-1.0, 0.0]]),
    WO=np.array([[1.0, -2.0], [3.0, 1.0]]),
)


def _msr_hand_pins(layer):
    """The gated MSR layer on the two-token example worked by hand in
    tests/golden/msr_two_tokens_hand.txt (GroupNorm off, no normalisations)."""
    rows = _golden_rows("msr_two_tokens_hand.txt")
    assert len(rows) == 2
    m = _MSR_HAND
    out = layer(m["X"], m["WQ"], m["WK"], m["WV"], m["WG"], m["WO"], H=1, dk=2, dv=2,
                gamma=[0.5], chunk=1, norm_flags=0, gn_eps=-1.0)
    for tok, expect in rows:
        exp = np.array([eval(e, {"math": math}) for e in expect.split(";")])
        assert np.max(np.abs(out[0, int(tok)] - exp)) < 1e-14, tok


def test_msr_layer_hand_example():
    from oracle.msr import msr_layer
    _msr_hand_pins(msr_layer)


def _msr_mutant(kind):
    """The MSR layer with one plausible mistake planted (a copy of the
    oracle's steps, changed in one place)."""
    from oracle import msr as M

    def layer(X, WQ, WK, WV, WG, WO, *, H, dk, dv, gamma, chunk, norm_flags, gn_eps):
        B, N, _ = X.shape
        Q, K, V, G = X @ WQ, X @ WK, X @ WV, X @ WG
        if kind == "projections transposed":
            Q, K = X @ WQ.T, X @ WK.T
        if kind == "gate reads V":
            G = V
        q = Q.reshape(B, N, H, dk).transpose(0, 2, 1, 3)
        k = K.reshape(B, N, H, dk).transpose(0, 2, 1, 3)
        v = V.reshape(B, N, H, dv).transpose(0, 2, 1, 3)
        if kind == "queries and keys swapped":
            q, k = k, q
        p = Problem(B, H, N, dk, dv, gamma, rotate=True, norm_flags=norm_flags, gn_eps=gn_eps)
        o, _, _ = oracle.chunkwise(p, chunk, q, k, v)
        Y = o.transpose(0, 2, 1, 3).reshape(B, N, H * dv)
        gate = M.swish(G)
        if kind == "sigmoid gate":
            gate = 1.0 / (1.0 + np.exp(-G))
        if kind == "gate after the output projection":
            return (Y @ WO) * gate
        if kind == "output projection transposed":
            return (gate * Y) @ WO.T
        return (gate * Y) @ WO
    return layer


MSR_MUTANTS = ["projections transposed", "gate reads V", "queries and keys swapped",
               "sigmoid gate", "gate after the output projection", "output projection transposed"]


@pytest.mark.parametrize("kind", MSR_MUTANTS)
def test_msr_mutants_are_caught(kind):
    with pytest.raises(AssertionError):
        _msr_hand_pins(_msr_mutant(kind))


def test_msr_mutant_harness_is_faithful():
    """With no mistake planted the copy passes the same pins."""
    _msr_hand_pins(_msr_mutant("none"))


def test_hand_derived_groupnorm():
    for eps, xs, expect in _golden_rows("groupnorm_hand.txt"):
        x = np.array([float(t) for t in xs.split()])
        exp = np.array([eval(e, {"math": math}) for e in expect.split(";")])
        assert np.max(np.abs(oracle.groupnorm(x[None], float(eps))[0] - exp)) < 1e-15


# Planted mistakes: (description, text to find, replacement).  Each mutant of
# the oracle source must fail at least one pin above.
MUTANTS = [
    ("xi uses gamma^i", "std::pow(g, i + 1)", "std::pow(g, i)"),
    ("zeta off by one", "std::pow(g, L - 1 - j)", "std::pow(g, L - j)"),
    ("rotation sign", "y[2 * j + 1] = a * sn + b * cs;", "y[2 * j + 1] = -a * sn + b * cs;"),
    ("unbiased GroupNorm variance", "var /= dv;", "var /= (dv - 1);"),
    ("decay row sum without sqrt", "s *= 1.0 / std::sqrt(cn);", "s *= 1.0 / cn;"),
    ("output before state update",
     "          S[(size_t)a * dv + e] = g * S[(size_t)a * dv + e] + kr[a] * vt[e];",
     "          S[(size_t)a * dv + e] = g * S[(size_t)a * dv + e];"),
    ("intra-chunk decay dropped", "dk) * std::pow(g, i - j);", "dk) * std::pow(g, 0);"),
    ("parallel decay exponent", "std::pow(g, n - m) : 0.0", "std::pow(g, n - m + 1) : 0.0"),
    ("theta exponent", "std::pow(base, -2.0 * j / static_cast<double>(d))",
     "std::pow(base, -1.0 * j / static_cast<double>(d))"),
    ("third normalisation without the absolute value", "std::fabs(rowsum)", "rowsum"),
]

PINS = [
    lambda: test_three_forms_agree(NORM_ALL, True, 5, 1e-6),
    lambda: test_three_forms_agree(0, False, 0, -1.0),
    test_state_is_decayed_outer_product_sum,
    lambda: test_real_rotation_matches_complex_closed_form(0),
    test_gamma_one_no_rotation_is_causal_linear_attention,
    test_gamma_zero_keeps_only_the_diagonal,
    test_hand_derived_two_token_example,
    test_hand_derived_negative_row_sum,
    test_hand_derived_groupnorm,
    lambda: test_decay_row_sum_is_geometric_series(0.9),
    test_rotation_preserves_norm_and_relative_phase,
    test_rotation_frequencies_hand,
]


def _caught(lib_path):
    with oracle.use_library(lib_path):
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                return True
    return False


@pytest.mark.parametrize("desc,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistakes_are_caught(desc, find, repl):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "retention_oracle.cpp")).read()
    assert find in src, desc
    tmp = tempfile.mkdtemp(prefix="orc_mut_")
    try:
        shutil.copy(os.path.join(os.path.dirname(oracle.__file__), "retention_oracle.h"), tmp)
        with open(os.path.join(tmp, "m.cpp"), "w") as f:
            f.write(src.replace(find, repl, 1))
        so = os.path.join(tmp, "libm.so")
        subprocess.run(["g++", "-O1", "-fPIC", "-shared", "-std=c++17", "-o", so,
                        os.path.join(tmp, "m.cpp")], check=True, capture_output=True)
        assert _caught(so), f"planted mistake not caught: {desc}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def test_msr_layer_matches_direct_loops():
    """Self-consistency of the MSR oracle on a tiny shape: projections by
    explicit loops, retention by the (pinned) parallel form per head, swish
    gate and output projection by loops.  Parity of the layer is otherwise
    unpinned: the pages print no worked MSR example."""
    from oracle.msr import msr_layer
    B, N, d, H, dk, dv = 1, 5, 4, 2, 2, 3
    g = np.random.default_rng(5)
    X = g.standard_normal((B, N, d))
    WQ, WK = g.standard_normal((d, H * dk)), g.standard_normal((d, H * dk))
    WV, WG = g.standard_normal((d, H * dv)), g.standard_normal((d, H * dv))
    WO = g.standard_normal((H * dv, d))
    gam = [0.9, 0.5]
    out = msr_layer(X, WQ, WK, WV, WG, WO, H=H, dk=dk, dv=dv, gamma=gam, chunk=2,
                    norm_flags=NORM_ALL, gn_eps=1e-6)

    def proj(W):
        return np.array([[[sum(X[b, n, i] * W[i, j] for i in range(d))
                           for j in range(W.shape[1])] for n in range(N)] for b in range(B)])
    Q, K, V, G = proj(WQ), proj(WK), proj(WV), proj(WG)
    Y = np.zeros((B, N, H * dv))
    for h in range(H):
        p = Problem(B, 1, N, dk, dv, gam[h], rotate=True, norm_flags=NORM_ALL, gn_eps=1e-6)
        o = oracle.parallel(p, Q[:, None, :, h * dk:(h + 1) * dk],
                            K[:, None, :, h * dk:(h + 1) * dk], V[:, None, :, h * dv:(h + 1) * dv])
        Y[:, :, h * dv:(h + 1) * dv] = o[:, 0]
    gate = np.array([[[G[b, n, j] / (1.0 + math.exp(-G[b, n, j])) for j in range(H * dv)]
                      for n in range(N)] for b in range(B)])
    Z = gate * Y
    ref = np.array([[[sum(Z[b, n, j] * WO[j, i] for j in range(H * dv)) for i in range(d)]
                     for n in range(N)] for b in range(B)])
    assert relerr(out, ref) < 1e-12


# ------------------------------------------------------------------ swish
# The gate's swish(x) = x sigmoid(x) (m0nads.wordpress.com "A dubious
# successor to Transformer", section "Last piece: Gated Multi-Scale
# Retention"; sigmoid with unit slope), pinned by what the mathematics fixes
# rather than by a second copy of its formula:
#   swish(0) = 0;  swish(x) - swish(-x) = x  (since sigmoid(x) + sigmoid(-x) = 1);
#   swish(x)/x -> 1 as x -> +inf and swish(x) -> 0 as x -> -inf;
#   swish(1) = 1/(1 + e^-1) = 0.7310585786300049 (the logistic function at 1,
#   printed to 16 digits from its series value).
SWISH_AT_1 = 0.7310585786300049


def _swish_pins(sw):
    assert sw(np.array([0.0]))[0] == 0.0
    x = np.linspace(-30.0, 30.0, 241)
    assert np.max(np.abs(sw(x) - sw(-x) - x)) < 1e-12
    assert abs(sw(np.array([1.0]))[0] - SWISH_AT_1) < 1e-15
    big = np.array([40.0, 60.0])
    assert np.max(np.abs(sw(big) / big - 1.0)) < 1e-15
    assert np.max(np.abs(sw(-big))) < 1e-15


def test_swish_pins():
    from oracle.msr import swish
    _swish_pins(swish)


SWISH_MUTANTS = [
    ("sigmoid of -x", lambda x: x / (1.0 + np.exp(x))),
    ("slope 2", lambda x: x / (1.0 + np.exp(-2.0 * x))),
    ("tanh gate", lambda x: x * np.tanh(x)),
    ("sigmoid without x", lambda x: 1.0 / (1.0 + np.exp(-x))),
    ("x times (1 + sigmoid)", lambda x: x + x / (1.0 + np.exp(-x))),
]


@pytest.mark.parametrize("desc,sw", SWISH_MUTANTS, ids=[m[0] for m in SWISH_MUTANTS])
def test_swish_mutants_are_caught(desc, sw):
    with np.errstate(over="ignore"):
        with pytest.raises(AssertionError):
            _swish_pins(sw)
