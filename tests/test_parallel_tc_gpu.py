"""GPU parity of the parallel form on the tensor cores (parallel_tc_kernel,
taken by retention_parallel_fwd for bf16 inputs with d_k a multiple of 64 up
to 256, d_v a multiple of 128 up to 1024 and gamma^64 >= 2^-16) against the
float64 oracle, on seeded inputs.

Tolerance: the bf16 bound of the other tensor-core paths (check_bf16: 2e-2
max abs beyond bf16 storage, 1e-2 RMS, after GroupNorm to unit variance).
The kernel rounds the rotated q, k to fp16 (as the chunkwise path does) and
the decayed scores to bf16 (the operand type of V): 2^-9 relative per score,
whose effect on an output row is about 2^-9 / sqrt(3) of its scale for
independent roundings.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrent_sequence_gb300 import synth
from tests.helpers import check_bf16, host, seeded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from linear_recurrent_sequence_gb300 import retention
    oracle.build()
    return retention


def ran_tensor_cores(R):
    torch.cuda.synchronize()
    return "parallel_tc" in R.kernel_times()


def run_parallel(R, q, k, v, gam, **kw):
    R.lib.retention_kernel_timer_reset()
    o = R.parallel_fwd(q, k, v, gam, **kw)
    assert ran_tensor_cores(R), "the parallel form did not take the tensor-core kernel"
    return o


def test_training_shape_sampled_heads(R):
    """B=4, H=8, N=2048, d_k=128, d_v=256 (the chunkwise training shape),
    all normalisations and GroupNorm; every head of batch 0 and 3 against
    the oracle's chunkwise form (the same function as the parallel form, up
    to rounding, and much faster in float64)."""
    B, H, N, dk, dv = 4, 8, 2048, 128, 256
    q, q64 = seeded(3101, "q", (B, H, N, dk), "bf16")
    k, k64 = seeded(3101, "k", (B, H, N, dk), "bf16")
    v, v64 = seeded(3101, "v", (B, H, N, dv), "bf16")
    gam = synth.head_gammas(H)
    o = run_parallel(R, q, k, v, gam, norm_flags=R.NORM_ALL)
    got = host(o)
    for b in (0, 3):
        p = oracle.Problem(1, H, N, dk, dv, gam, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
        ref, _, _ = oracle.chunkwise(p, 256, q64[b:b + 1], k64[b:b + 1], v64[b:b + 1])
        check_bf16(got[b:b + 1], ref, f"parallel tensor cores, batch {b}")


def test_ragged_strided_three_value_slices(R):
    """N = 333 (a ragged 128-query block and a ragged 64-key block), pos0 > 0,
    [B, N, H, d] strided views, d_k = 256, d_v = 384 (three 128-wide CTAs per
    head), fp32 output."""
    B, H, N, dk, dv = 2, 3, 333, 256, 384
    qb, q64 = seeded(3102, "q", (B, N, H, dk), "bf16")
    kb, k64 = seeded(3102, "k", (B, N, H, dk), "bf16")
    vb, v64 = seeded(3102, "v", (B, N, H, dv), "bf16")
    q, k, v = (t.permute(0, 2, 1, 3) for t in (qb, kb, vb))
    gam = [0.9, 0.97, 1.0]
    o = run_parallel(R, q, k, v, gam, pos0=5, norm_flags=R.NORM_ALL, out_dtype=torch.float32)
    p = oracle.Problem(B, H, N, dk, dv, gam, pos0=5, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    ref = oracle.parallel(p, q64.transpose(0, 2, 1, 3), k64.transpose(0, 2, 1, 3),
                          v64.transpose(0, 2, 1, 3))
    check_bf16(host(o), ref, "parallel tensor cores, ragged strided")


@pytest.mark.parametrize("N", [1, 37, 64, 129])
def test_short_sequences(R, N):
    B, H, dk, dv = 1, 2, 64, 128
    q, q64 = seeded(3103 + N, "q", (B, H, N, dk), "bf16")
    k, k64 = seeded(3103 + N, "k", (B, H, N, dk), "bf16")
    v, v64 = seeded(3103 + N, "v", (B, H, N, dv), "bf16")
    gam = [0.95, 0.999]
    o = run_parallel(R, q, k, v, gam, norm_flags=R.NORM_ALL, out_dtype=torch.float32)
    p = oracle.Problem(B, H, N, dk, dv, gam, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    check_bf16(host(o), oracle.parallel(p, q64, k64, v64), f"parallel tensor cores, N={N}")


def test_dk_192(R):
    """d_k = 192 (a multiple of 64 that is not a power of two), ragged N,
    all normalisations."""
    B, H, N, dk, dv = 1, 2, 300, 192, 256
    q, q64 = seeded(3110, "q", (B, H, N, dk), "bf16")
    k, k64 = seeded(3110, "k", (B, H, N, dk), "bf16")
    v, v64 = seeded(3110, "v", (B, H, N, dv), "bf16")
    gam = [0.95, 0.999]
    o = run_parallel(R, q, k, v, gam, norm_flags=R.NORM_ALL, out_dtype=torch.float32)
    p = oracle.Problem(B, H, N, dk, dv, gam, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    check_bf16(host(o), oracle.parallel(p, q64, k64, v64), "parallel tensor cores, d_k=192")


def test_negative_row_sums_without_groupnorm(R):
    """k = -q: most rows' sums of R fall below -1, so the third
    normalisation divides by |sum R| (hwhale.com/article/285883, R_nm /
    max(|sum_i R_ni|, 1)); GroupNorm off, so the row factor reaches the
    output.  Checked relative to the output's largest value."""
    B, H, N, dk, dv = 1, 2, 200, 128, 128
    q, q64 = seeded(6162, "q", (B, H, N, dk), "bf16")
    v, v64 = seeded(6162, "v", (B, H, N, dv), "bf16")
    k, k64 = -q, -q64
    gam = [0.9, 0.97]
    o = run_parallel(R, q, k, v, gam, norm_flags=R.NORM_ALL, gn_eps=None,
                     out_dtype=torch.float32)
    p = oracle.Problem(B, H, N, dk, dv, gam, norm_flags=oracle.NORM_ALL, gn_eps=-1.0)
    ref = oracle.parallel(p, q64, k64, v64)
    err = np.max(np.abs(host(o) - ref)) / np.max(np.abs(ref))
    assert err <= 1e-2, err


def test_input_scale_extremes(R):
    """q scaled by 2^40 and k by 2^-60: the block exponents keep every
    operand finite; without normalisations or GroupNorm the output is the
    raw (Q K^T (.) D) V, 2^-20 times that of the unscaled inputs."""
    B, H, N, dk, dv = 1, 1, 150, 128, 128
    q, q64 = seeded(3104, "q", (B, H, N, dk), "bf16")
    k, k64 = seeded(3104, "k", (B, H, N, dk), "bf16")
    v, v64 = seeded(3104, "v", (B, H, N, dv), "bf16")
    qs, ks = q * 2.0 ** 40, k * 2.0 ** -60
    o = run_parallel(R, qs, ks, v, [0.97], gn_eps=None, out_dtype=torch.float32)
    p = oracle.Problem(B, H, N, dk, dv, [0.97], gn_eps=-1.0)
    ref = oracle.parallel(p, q64 * 2.0 ** 40, k64 * 2.0 ** -60, v64)
    err = np.max(np.abs(host(o) - ref)) / np.max(np.abs(ref))
    assert err <= 1e-2, err


def test_agrees_with_chunkwise_tensor_cores(R):
    """The parallel and chunkwise forms are one function: on the same bf16
    inputs their tensor-core results agree to the same bound."""
    B, H, N, dk, dv = 1, 4, 1000, 256, 512
    q, _ = seeded(3105, "q", (B, H, N, dk), "bf16")
    k, _ = seeded(3105, "k", (B, H, N, dk), "bf16")
    v, _ = seeded(3105, "v", (B, H, N, dv), "bf16")
    gam = synth.head_gammas(H)
    o_par = run_parallel(R, q, k, v, gam, norm_flags=R.NORM_ALL, out_dtype=torch.float32)
    o_chk = R.chunkwise_fwd(q, k, v, gam, norm_flags=R.NORM_ALL, out_dtype=torch.float32)
    check_bf16(host(o_par), host(o_chk), "parallel vs chunkwise")
