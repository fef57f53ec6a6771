"""The tensor-core paths inside CUDA graphs: each call captured once and
replayed on new inputs (copied into the captured buffers) gives exactly the
result of the same call made directly.  The kernels are deterministic (no
atomics; fixed summation orders), so the comparison is bitwise."""
import pytest
import torch

from linear_recurrent_sequence_gb300 import synth
from tests.helpers import seeded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from linear_recurrent_sequence_gb300 import retention
    return retention


def capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_chunkwise_segments_in_a_graph(R):
    """N = 2048 at H = 4 runs as concurrent sequence segments (the state pass
    feeds the later ones): prologue, state pass and chunk kernel in one graph."""
    B, H, N, dk, dv = 1, 4, 2048, 256, 512
    gam = synth.head_gammas(H)
    q = torch.empty(B, H, N, dk, dtype=torch.bfloat16, device="cuda")
    k, v = torch.empty_like(q), torch.empty(B, H, N, dv, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(v)
    S = torch.empty(B, H, dk, dv, device="cuda")
    d, _ = R.make_desc(q, k, v, o, gam, norm_flags=R.NORM_ALL)
    ws = R.new_workspace(R.workspace_size(d), q.device)

    def fn():
        R.chunkwise_fwd(q, k, v, gam, norm_flags=R.NORM_ALL, out=o, S_out=S, workspace=ws)

    for seed in (501, 502):
        q.copy_(seeded(seed, "q", (B, H, N, dk), "bf16")[0])
        k.copy_(seeded(seed, "k", (B, H, N, dk), "bf16")[0])
        v.copy_(seeded(seed, "v", (B, H, N, dv), "bf16")[0])
        if seed == 501:
            g = capture(fn)
        fn()
        torch.cuda.synchronize()
        o_ref, S_ref = o.clone(), S.clone()
        o.zero_()
        S.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(S, S_ref), seed


def test_decode_steps_in_a_graph(R):
    B, H, dk, dv, T = 2, 4, 256, 512, 16
    gam = synth.head_gammas(H)
    q, _ = seeded(503, "q", (B, H, T, dk), "bf16")
    k, _ = seeded(503, "k", (B, H, T, dk), "bf16")
    v, _ = seeded(503, "v", (B, H, T, dv), "bf16")
    S0 = seeded(503, "S", (B, H, dk, dv), "f32")[0] * 0.01
    S = S0.clone()
    o = torch.empty(B, H, T, dv, dtype=torch.bfloat16, device="cuda")
    ws = R.new_workspace(256, q.device)

    def fn():
        for t in range(T):
            R.recurrent_step(q[:, :, t], k[:, :, t], v[:, :, t], S, gam, pos=100 + t,
                             out=o[:, :, t:t + 1], workspace=ws)

    S.copy_(S0)
    fn()
    torch.cuda.synchronize()
    o_ref, S_ref = o.clone(), S.clone()
    S.copy_(S0)
    g = capture(fn)
    S.copy_(S0)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(S, S_ref)


def test_backward_and_parallel_in_graphs(R):
    B, H, N, dk, dv = 1, 2, 600, 256, 512
    gam = [0.97, 0.999]
    q, _ = seeded(504, "q", (B, H, N, dk), "bf16")
    k, _ = seeded(504, "k", (B, H, N, dk), "bf16")
    v, _ = seeded(504, "v", (B, H, N, dv), "bf16")
    dO, _ = seeded(504, "dO", (B, H, N, dv), "bf16")
    dq, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    d, _ = R.make_desc(q, k, v, dO, gam, gn_eps=None)
    wsb = R.new_workspace(R.backward_workspace_size(d), q.device)

    def bwd():
        R.chunkwise_bwd(q, k, v, dO, gam, dq=dq, dk=dk_, dv=dv_, workspace=wsb)

    bwd()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (dq, dk_, dv_)]
    g = capture(bwd)
    for t in (dq, dk_, dv_):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip((dq, dk_, dv_), ref):
        assert torch.equal(a, b)

    o = torch.empty_like(v)
    dp, _ = R.make_desc(q, k, v, o, gam, norm_flags=R.NORM_ALL)
    wsp = R.new_workspace(R.workspace_size(dp), q.device)

    def par():
        R.parallel_fwd(q, k, v, gam, norm_flags=R.NORM_ALL, out=o, workspace=wsp)

    par()
    torch.cuda.synchronize()
    o_ref = o.clone()
    g = capture(par)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)
