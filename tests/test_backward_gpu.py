"""GPU parity of the backward (retention_chunkwise_bwd) against the oracle's
gradients (oracle.recurrent_bwd, pinned by finite differences of the forward
oracle in test_oracle_backward_pins.py), on the same seeded inputs.

Tolerances:
  * fp32 inputs and gradients: max |gpu - ref| / max |ref| <= 1e-4
    (normwise relative; fp32 accumulation over at most a few hundred terms);
  * bf16 inputs: the gradients are rounded to bf16 once (at most 2^-9 of each
    element, so of the largest), over fp32 arithmetic:
    max |gpu - ref| / max |ref| <= 1e-2;
  * the fp32 entry-state gradient: 1e-4 normwise relative on the CUDA-core
    path; 1e-2 where bf16 inputs take the tensor-core path (d_k 128 or 256,
    d_v a multiple of 128, gamma^64 >= 2^-16), whose runs of the forward
    kernel round the reversed-time operands (k', q', dO) to bf16 and fp16 as
    the forward rounds its own: the forward's final state carries the same
    1e-2 bound.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrent_sequence_gb300 import synth
from tests.helpers import check_f32, host, seeded

pytestmark = pytest.mark.gpu

TOL_BF16_GRAD_REL = 1e-2
TOL_TC_STATE_REL = 1e-2


def takes_tensor_cores(dtype, dk, dv, gam):
    """The shapes the library's backward runs on the tensor cores."""
    g = np.atleast_1d(np.asarray(gam, np.float64))
    return (dtype == "bf16" and dk in (128, 256) and dv % 128 == 0 and dv <= 1024
            and bool(np.all(g > 0)) and bool(np.all(np.log(np.maximum(g, 1e-300)) * 64
                                                    >= -16 * np.log(2) * 0.999)))


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from linear_recurrent_sequence_gb300 import retention
    oracle.build()
    return retention


def check_rel(got, ref, tol, what):
    err = np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30)
    assert err <= tol, f"{what}: normwise rel err {err:.3e} > {tol}"
    return err


def run_case(R, seed, B, H, N, dk, dv, dtype, gam, *, flags=oracle.NORM_SCALE | oracle.NORM_DROW,
             rotate=True, pos0=0, with_S=True, with_dS=True, bnhd=False, heads=None,
             do_dtype=None):
    """Seeded inputs, the CUDA backward and the oracle's gradients; compares
    all heads or only `heads` (each head is an independent problem)."""
    shp_k, shp_v = (B, H, N, dk), (B, H, N, dv)
    if bnhd:  # [B, N, H, d] storage seen as [B, H, N, d] views
        def mk(name, shp, dt, std=1.0):
            t, x64 = seeded(seed, name, (shp[0], shp[2], shp[1], shp[3]), dt, std)
            return t.permute(0, 2, 1, 3), x64.transpose(0, 2, 1, 3)
    else:
        def mk(name, shp, dt, std=1.0):
            return seeded(seed, name, shp, dt, std)
    q, q64 = mk("q", shp_k, dtype)
    k, k64 = mk("k", shp_k, dtype)
    v, v64 = mk("v", shp_v, dtype)
    dO, dO64 = mk("dO", shp_v, do_dtype or dtype)
    S_in = dS_out = None
    S64 = dS64 = None
    if with_S:
        S_in, S64 = seeded(seed, "S", (B, H, dk, dv), "f32")
    if with_dS:
        dS_out, dS64 = seeded(seed, "dS", (B, H, dk, dv), "f32")
    dS_in = torch.full((B, H, dk, dv), float("nan"), device="cuda")
    dq, dk_, dv_, _ = R.chunkwise_bwd(q, k, v, dO, gam, norm_flags=flags, pos0=pos0,
                                      rotate=rotate, S_in=S_in, dS_out=dS_out, dS_in=dS_in)
    torch.cuda.synchronize()
    got = dict(q=host(dq), k=host(dk_), v=host(dv_), S=host(dS_in))
    hs = list(range(H)) if heads is None else heads
    gam = np.broadcast_to(np.asarray(gam, dtype=np.float64), (H,))
    tc = takes_tensor_cores(dtype, dk, dv, gam)
    for h in hs:
        p = oracle.Problem(B, 1, N, dk, dv, gam[h], rotate=rotate, pos0=pos0,
                           norm_flags=flags, gn_eps=-1.0)
        sl = slice(h, h + 1)
        ref = oracle.recurrent_bwd(
            p, q64[:, sl], k64[:, sl], v64[:, sl], dO64[:, sl],
            S_in=None if S64 is None else S64[:, sl],
            dS_out=None if dS64 is None else dS64[:, sl])
        for name, r in zip("qkvS", ref):
            g = got[name][:, sl]
            if name == "S" and tc:
                check_rel(g, r, TOL_TC_STATE_REL, f"dS head {h}")
            elif name == "S" or dtype == "f32":
                check_f32(g, r, f"d{name} head {h}")
            else:
                check_rel(g, r, TOL_BF16_GRAD_REL, f"d{name} head {h}")
    return got


def test_fp32_ragged_tail_three_gammas(R):
    # N = 77: several 16- and 32-token steps and a ragged tail; gamma 0 and 1
    # are the degenerate decays.
    run_case(R, 2001, 2, 3, 77, 32, 48, "f32", [0.9, 0.0, 1.0], pos0=5)


def test_bf16_strided_views_no_norms(R):
    run_case(R, 2002, 1, 4, 200, 64, 128, "bf16", synth.head_gammas(4), flags=0,
             with_S=False, with_dS=False, bnhd=True)


def test_bf16_bench_head_dims(R):
    run_case(R, 2003, 1, 2, 300, 256, 512, "bf16", [0.96875, 0.999], pos0=100)


def test_bf16_tensor_core_three_value_pieces_strided(R):
    # d_v = 384 splits into three 128-wide pieces for dq and dk; [B, N, H, d]
    # storage; N = 200 ends in a ragged chunk; both states present.
    run_case(R, 2009, 2, 2, 200, 128, 384, "bf16", [0.9, 0.999], pos0=7, bnhd=True)


def test_bf16_tensor_core_fp32_output_gradient(R):
    # dO in fp32 (the gradient of an fp32 output): converted once to bf16.
    run_case(R, 2013, 1, 2, 130, 256, 512, "bf16", [0.9, 0.995], pos0=3, do_dtype="f32")


def test_bf16_tensor_core_shorter_than_a_chunk(R):
    run_case(R, 2010, 1, 3, 37, 256, 256, "bf16", [0.96875, 0.99, 0.999], with_S=False)
    run_case(R, 2011, 1, 1, 1, 128, 128, "bf16", [0.95], with_dS=False, flags=0)


def test_fp32_widest_values(R):
    run_case(R, 2004, 1, 1, 40, 16, 1024, "f32", [0.95])


def test_fp32_ragged_slices_single_token(R):
    # d_k = 6 and d_v = 5 fill part of one CTA slice; N = 1.
    run_case(R, 2005, 2, 2, 1, 6, 5, "f32", [0.5, 0.8], rotate=True, pos0=9)
    run_case(R, 2006, 1, 2, 33, 6, 5, "f32", [0.5, 0.8], rotate=False)


def test_no_tokens_passes_the_state_gradient(R):
    B, H, dk, dv = 1, 2, 8, 8
    e = torch.empty(B, H, 0, dk, device="cuda")
    ev = torch.empty(B, H, 0, dv, device="cuda")
    dS_out = torch.randn(B, H, dk, dv, device="cuda")
    dS_in = torch.zeros(B, H, dk, dv, device="cuda")
    R.chunkwise_bwd(e, e, ev, ev, [0.9, 0.5], dS_out=dS_out, dS_in=dS_in)
    torch.cuda.synchronize()
    assert torch.equal(dS_in, dS_out)
    R.chunkwise_bwd(e, e, ev, ev, [0.9, 0.5], dS_in=dS_in)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dS_in).item() == 0


def test_state_gradient_in_place(R):
    B, H, N, dk, dv = 1, 2, 50, 16, 32
    q, _ = seeded(2007, "q", (B, H, N, dk), "f32")
    k, _ = seeded(2007, "k", (B, H, N, dk), "f32")
    v, _ = seeded(2007, "v", (B, H, N, dv), "f32")
    dO, _ = seeded(2007, "dO", (B, H, N, dv), "f32")
    dS, _ = seeded(2007, "dS", (B, H, dk, dv), "f32")
    out = torch.empty_like(dS)
    ref = R.chunkwise_bwd(q, k, v, dO, [0.9, 0.7], dS_out=dS, dS_in=out)
    same = dS.clone()
    got = R.chunkwise_bwd(q, k, v, dO, [0.9, 0.7], dS_out=same, dS_in=same)
    torch.cuda.synchronize()
    for a, b in zip(ref[:3], got[:3]):
        assert torch.equal(a, b)
    assert torch.equal(out, same)


def test_state_gradient_in_place_tensor_cores(R):
    B, H, N, dk, dv = 1, 2, 150, 128, 256
    q, _ = seeded(2012, "q", (B, H, N, dk), "bf16")
    k, _ = seeded(2012, "k", (B, H, N, dk), "bf16")
    v, _ = seeded(2012, "v", (B, H, N, dv), "bf16")
    dO, _ = seeded(2012, "dO", (B, H, N, dv), "bf16")
    dS, _ = seeded(2012, "dS", (B, H, dk, dv), "f32")
    out = torch.empty_like(dS)
    ref = R.chunkwise_bwd(q, k, v, dO, [0.9, 0.97], dS_out=dS, dS_in=out)
    same = dS.clone()
    got = R.chunkwise_bwd(q, k, v, dO, [0.9, 0.97], dS_out=same, dS_in=same)
    torch.cuda.synchronize()
    for a, b in zip(ref[:3], got[:3]):
        assert torch.equal(a, b)
    assert torch.equal(out, same)


def test_third_normalisation_is_refused(R):
    x = torch.zeros(1, 1, 4, 4, device="cuda")
    with pytest.raises(R.RetentionError) as ei:
        R.chunkwise_bwd(x, x, x, x, [0.9], norm_flags=R.NORM_RSUM)
    assert ei.value.status == 2


def test_bench_size_sampled_heads_and_euler_identity(R):
    """B=1, H=16, N=8192, d_k=256, d_v=512 (the benchmark's forward shape):
    heads 0 and 15 against the oracle; then, for every head, Euler's identity
    <dq, q> = <dO, o> (o is linear in q) with dO = o, o from the library's
    own forward without GroupNorm, so that the right side is |o|^2."""
    B, H, N, dk, dv = 1, 16, 8192, 256, 512
    gam = synth.head_gammas(H)
    run_case(R, 2008, B, H, N, dk, dv, "bf16", gam, flags=0, with_S=False,
             with_dS=False, heads=[0, 15])
    q, q64 = seeded(2008, "q", (B, H, N, dk), "bf16")
    k, _ = seeded(2008, "k", (B, H, N, dk), "bf16")
    v, _ = seeded(2008, "v", (B, H, N, dv), "bf16")
    o = R.chunkwise_fwd(q, k, v, gam, gn_eps=None, out_dtype=torch.float32)
    dq, _, _, _ = R.chunkwise_bwd(q, k, v, o, gam)
    torch.cuda.synchronize()
    lhs = np.einsum("bhnd,bhnd->h", host(dq), q64)
    o64 = host(o)
    rhs = np.einsum("bhnd,bhnd->h", o64, o64)
    assert np.max(np.abs(lhs - rhs) / rhs) < 1e-2, (lhs, rhs)
