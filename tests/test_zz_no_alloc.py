"""The allocation-free chunkwise entry point, for callers that cannot call
cudaMalloc (for example a plugin that its host runtime gives only input and
output buffers).  Its output must match the ordinary entry point's, which
uses a caller workspace, on two calls in a row: the second call reuses the
library's scratch array with the first call's leftovers still in it.  The
second call is also checked against the float64 oracle, so the test does
not rest on the CUDA path alone.

This file is collected last on purpose."""
import ctypes

import pytest
import torch

import oracle
from tests.helpers import check_bf16, check_f32, host, seeded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from linear_recurrent_sequence_gb300 import retention
    return retention


def _case(seed, dtype, B, H, N, dk, dv):
    q, q64 = seeded(seed, "q", (B, H, N, dk), dtype)
    k, k64 = seeded(seed, "k", (B, H, N, dk), dtype)
    v, v64 = seeded(seed, "v", (B, H, N, dv), dtype)
    return (q, k, v), (q64, k64, v64)


def test_noalloc_matches_workspace_entry_point_twice(R):
    # call 1: fp32, plain equations, zero initial state
    (q, k, v), _ = _case(11, "f32", 1, 2, 96, 32, 32)
    ref = R.chunkwise_fwd(q, k, v, [0.9, 0.97], chunk=16)
    got = R.chunkwise_fwd_noalloc(q, k, v, [0.9, 0.97], chunk=16)
    torch.cuda.synchronize()
    check_f32(host(got), host(ref), "no-alloc call 1")
    # call 2: bf16, all normalisations, carried state in and out
    (q, k, v), (q64, k64, v64) = _case(12, "bf16", 2, 4, 200, 64, 128)
    gam = [0.96875, 0.984375, 0.9921875, 0.99609375]
    S0 = torch.randn(2, 4, 64, 128, device="cuda")
    z0 = torch.randn(2, 4, 64, device="cuda")
    S_ref, z_ref = torch.empty_like(S0), torch.empty_like(z0)
    S_got, z_got = torch.empty_like(S0), torch.empty_like(z0)
    ref = R.chunkwise_fwd(q, k, v, gam, chunk=64, norm_flags=R.NORM_ALL, pos0=300, S_in=S0,
                          z_in=z0, S_out=S_ref, z_out=z_ref)
    got = R.chunkwise_fwd_noalloc(q, k, v, gam, chunk=64, norm_flags=R.NORM_ALL, pos0=300,
                                  S_in=S0, z_in=z0, S_out=S_got, z_out=z_got)
    torch.cuda.synchronize()
    check_bf16(host(got), host(ref), "no-alloc call 2")
    check_f32(host(S_got), host(S_ref), "no-alloc state")
    check_f32(host(z_got), host(z_ref), "no-alloc z")
    oracle.build()
    p = oracle.Problem(2, 4, 200, 64, 128, gam, pos0=300, norm_flags=oracle.NORM_ALL,
                       gn_eps=1e-6)
    o64, S64, z64 = oracle.chunkwise(p, 64, q64, k64, v64, host(S0), host(z0))
    check_bf16(host(got), o64, "no-alloc call 2 against the oracle")
    assert (host(S_got) - S64).__abs__().max() / abs(S64).max() < 1e-2
    assert (host(z_got) - z64).__abs__().max() / abs(z64).max() < 1e-2


def test_noalloc_rejects_problems_beyond_its_scratch(R):
    q = torch.empty(4, 8, 2048, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.empty(4, 8, 2048, 256, dtype=torch.bfloat16, device="cuda")
    d, g = R.make_desc(q, q, v, v, [0.9] * 8)
    assert R.workspace_size(d) > (32 << 20)
    rc = R.lib.retention_chunkwise_fwd_noalloc(ctypes.byref(d), R._ptr(q), R._ptr(q), R._ptr(v),
                                               None, None, None, None, R._ptr(v), None)
    assert rc == 2  # RET_EUNSUPPORTED, nothing launched
