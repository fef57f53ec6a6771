"""The MSR layer's projection GEMM (C = A B, bf16 in/out, fp32 accumulate)
against a float32 product of the same bf16 values: tensor-core shapes and a
ragged shape served by the CUDA-core kernel."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from linear_recurrent_sequence_gb300 import retention
    return retention


@pytest.mark.parametrize("M,N,K,tc", [(128, 256, 64, True), (384, 512, 192, True),
                                      (2048, 2048, 2048, True), (100, 200, 50, False),
                                      (32, 512, 4096, True), (300, 256, 192, True),
                                      (20, 256, 4096, True), (128, 256, 4096, True),
                                      (64, 1024, 2048, True), (1000, 768, 320, True),
                                      (4096, 4096, 1024, True)])
def test_gemm_matches_fp32_product(R, M, N, K, tc):
    """Tensor-core shapes (including M not a multiple of the 128-row tile,
    whose last tile is partly outside A and C, and few-row shapes that the
    tensor cores run split over K with fp32 partials added by a reduce) and a
    CUDA-core shape."""
    g = torch.Generator(device="cuda").manual_seed(M + N + K)
    A = torch.randn(M, K, device="cuda", generator=g).bfloat16()
    B = (torch.randn(K, N, device="cuda", generator=g) * 0.05).bfloat16()
    R.lib.retention_kernel_timer_reset()
    C = R.gemm_bf16(A, B)
    torch.cuda.synchronize()
    ref = A.float() @ B.float()
    err = (C.float() - ref).abs()
    # bf16 output rounding (2^-9 relative) plus fp32 summation-order effects
    assert float((err - ref.abs() * 2.0 ** -8).max()) <= 1e-3 * float(ref.abs().max())
    names = R.kernel_times()
    assert ("gemm_tc" in names) == tc and ("gemm_simt" in names) == (not tc), names


def test_msr_layer_all_tensor_core_shapes(R):
    """MSR layer whose projections all run on the tensor-core GEMM."""
    import numpy as np

    import oracle
    from linear_recurrent_sequence_gb300 import synth
    from oracle.msr import msr_layer
    from tests.helpers import check_bf16, host, seeded
    B, N, dm, H, dk, dv = 1, 256, 256, 2, 128, 128
    X, X64 = seeded(88, "x", (B, N, dm), "bf16")
    W = {}
    for name, shp in (("wq", (dm, H * dk)), ("wk", (dm, H * dk)), ("wv", (dm, H * dv)),
                      ("wg", (dm, H * dv)), ("wo", (H * dv, dm))):
        W[name] = seeded(88, name, shp, "bf16", std=0.05)
    gam = synth.head_gammas(H)
    R.lib.retention_kernel_timer_reset()
    Y = R.msr_layer_fwd(X, W["wq"][0], W["wk"][0], W["wv"][0], W["wg"][0], W["wo"][0], H=H,
                        d_k=dk, d_v=dv, gamma=gam, chunk=64, norm_flags=R.NORM_ALL)
    torch.cuda.synchronize()
    names = R.kernel_times()
    assert "gemm_tc" in names and "gemm_simt" not in names, names
    ref = msr_layer(X64, W["wq"][1], W["wk"][1], W["wv"][1], W["wg"][1], W["wo"][1], H=H,
                    dk=dk, dv=dv, gamma=gam, chunk=64, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    check_bf16(host(Y), ref, "msr all-TC")


@pytest.mark.parametrize("M,N,K", [
    (1, 8, 3),          # one row, the narrowest N, K below one unroll group
    (3, 2056, 1000),    # N not a multiple of the 2048-column CTA block
    (9, 4096, 777),     # K not a multiple of 8 nor of the slice length
    (16, 24, 4099),     # the largest row count, tiny N, odd K
    (16, 6144, 2048),   # a decode-shaped projection
])
def test_skinny_gemm_matches_float64_product(R, M, N, K):
    """The weight-streaming kernel for few rows (split-K fp32 partials added
    in a fixed order) against a float64 product of the same bf16 values."""
    g = torch.Generator(device="cuda").manual_seed(7 * M + N + K)
    A = torch.randn(M, K, device="cuda", generator=g).bfloat16()
    B = (torch.randn(K, N, device="cuda", generator=g) * 0.05).bfloat16()
    R.lib.retention_kernel_timer_reset()
    C = R.gemm_bf16(A, B)
    torch.cuda.synchronize()
    names = R.kernel_times()
    assert "gemm_skinny" in names and "skinny_reduce" in names, names
    ref = A.double().cpu() @ B.double().cpu()
    err = (C.double().cpu() - ref).abs()
    # bf16 output rounding (2^-9 relative) plus fp32 accumulation over K terms
    assert float((err - ref.abs() * 2.0 ** -8).max()) <= 1e-4 * float(ref.abs().max())
    # deterministic: the partials are added in slice order
    C2 = R.gemm_bf16(A, B)
    assert torch.equal(C, C2)
