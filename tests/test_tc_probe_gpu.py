"""Tensor-core building blocks on the GPU: one tcgen05 MMA chain per case
with the shared-memory layouts the retention kernels use, against a float64
product of the same bf16 values.  Also pins the TMEM lane layout of an
M=64 accumulator (row r in lane 32*(r//16) + r%16)."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

SW_ROW = 128  # bytes per swizzled row


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from linear_recurrent_sequence_gb300 import retention
    return retention


def run_probe(R, a_mode, b_mode, M, N, K, a_strides=(0, 0), b_strides=(0, 0), seed=0):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = A.double() @ B.double().T
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.zeros(128, N, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = R.lib.retention_tc_probe(a_mode, b_mode, M, N, K, a_strides[0], a_strides[1],
                                  b_strides[0], b_strides[1], ctypes.c_void_p(Ad.data_ptr()),
                                  ctypes.c_void_p(Bd.data_ptr()), ctypes.c_void_p(D.data_ptr()),
                                  ctypes.c_void_p(st.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 0
    return D.double().cpu().numpy(), ref.numpy()


def m64_lane(r):
    return 32 * (r // 16) + r % 16


def close(got, ref):
    return np.max(np.abs(got - ref)) <= 1e-3 * max(1.0, np.max(np.abs(ref)))


@pytest.mark.parametrize("N,K", [(128, 128), (256, 64), (64, 128)])
def test_kmajor_both(R, N, K):
    D, ref = run_probe(R, 0, 0, 128, N, K)
    assert close(D, ref)


@pytest.mark.parametrize("K", [64, 128])
def test_mn_major_a(R, K):
    # MN-major: LBO = stride between 64-wide MN blocks, SBO = stride between
    # groups of 8 K rows.
    D, ref = run_probe(R, 1, 0, 128, 128, K, a_strides=(K * SW_ROW, 8 * SW_ROW))
    assert close(D, ref)


@pytest.mark.parametrize("N", [128, 256])
def test_mn_major_b(R, N):
    D, ref = run_probe(R, 0, 1, 128, N, 64, b_strides=(64 * SW_ROW, 8 * SW_ROW))
    assert close(D, ref)


def test_mn_major_both(R):
    D, ref = run_probe(R, 1, 1, 128, 256, 64, a_strides=(64 * SW_ROW, 8 * SW_ROW),
                       b_strides=(64 * SW_ROW, 8 * SW_ROW))
    assert close(D, ref)


def test_a_from_tmem(R):
    D, ref = run_probe(R, 2, 0, 128, 64, 128)
    assert close(D, ref)
    D, ref = run_probe(R, 2, 1, 128, 256, 64, b_strides=(64 * SW_ROW, 8 * SW_ROW))
    assert close(D, ref)


def test_m64_accumulator_lanes(R):
    D, ref = run_probe(R, 0, 0, 64, 64, 128)
    lanes = [m64_lane(r) for r in range(64)]
    assert close(D[lanes], ref)


@pytest.mark.parametrize("n", [0, 1, 5, 15])
def test_accumulator_scale_operand(R, n):
    """tcgen05.mma's scale-input-d operand: D' = A B^T + D 2^-n, checked with
    D = A B^T from a first chain, so D' = A B^T (1 + 2^-n)."""
    g = torch.Generator().manual_seed(40 + n)
    A = torch.randn(128, 64, generator=g).to(torch.bfloat16)
    B = torch.randn(128, 64, generator=g).to(torch.bfloat16)
    ref = (A.double() @ B.double().T).numpy() * (1.0 + 2.0 ** -n)
    D = torch.zeros(128, 128, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Ad, Bd = A.cuda(), B.cuda()
    rc = R.lib.retention_tc_probe_scale_d(n, ctypes.c_void_p(Ad.data_ptr()),
                                          ctypes.c_void_p(Bd.data_ptr()),
                                          ctypes.c_void_p(D.data_ptr()),
                                          ctypes.c_void_p(st.data_ptr()),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 0
    assert close(D.double().cpu().numpy(), ref)


@pytest.mark.parametrize("N,K", [(128, 64), (256, 128)])
def test_cta_pair_mma(R, N, K):
    """tcgen05.mma with .cta_group::2: the two CTAs of a cluster compute a
    256-row product, each holding its 128 rows of A and half of B's columns
    and receiving its rows of D in its own TMEM; their allocations return the
    same TMEM address."""
    g = torch.Generator().manual_seed(50 + N + K)
    A = torch.randn(256, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = (A.double() @ B.double().T).numpy()
    D = torch.full((256, N), float("nan"), dtype=torch.float32, device="cuda")
    tb = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Ad, Bd = A.cuda(), B.cuda()
    rc = R.lib.retention_tc_probe_pair(N, K, ctypes.c_void_p(Ad.data_ptr()),
                                       ctypes.c_void_p(Bd.data_ptr()),
                                       ctypes.c_void_p(D.data_ptr()),
                                       ctypes.c_void_p(tb.data_ptr()),
                                       ctypes.c_void_p(st.data_ptr()),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 0
    t = tb.cpu().tolist()
    assert t[0] == t[1], t
    assert close(D.double().cpu().numpy(), ref)
