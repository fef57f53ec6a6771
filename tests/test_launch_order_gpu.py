"""Launch order with programmatic dependent launch: kernels may be placed
while the kernel before them still runs, and must not touch data that an
earlier kernel writes or reads before their own wait.  Each test runs a
chain of calls with nothing but stream order between them, where every call
reads what the call before it wrote, and compares it bitwise with the same
chain synchronised after every call (every kernel is deterministic)."""
import numpy as np
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


def test_chunkwise_calls_consume_the_previous_output(R):
    """Four chunkwise calls, each taking the previous call's output as its
    queries and values (d_k = d_v), N = 2048 so the path runs its prologue,
    state pass and two sequence segments."""
    B, H, N, d = 1, 4, 2048, 128
    gam = synth.head_gammas(H)
    q0, _ = seeded(601, "q", (B, H, N, d), "bf16")
    k, _ = seeded(601, "k", (B, H, N, d), "bf16")
    v0, _ = seeded(601, "v", (B, H, N, d), "bf16")

    def chain(sync):
        q, v, outs = q0, v0, []
        for _ in range(4):
            o = R.chunkwise_fwd(q, k, v, gam, norm_flags=R.NORM_ALL)
            if sync:
                torch.cuda.synchronize()
            outs.append(o)
            q, v = o, o
        torch.cuda.synchronize()
        return [o.clone() for o in outs]

    ref = chain(True)
    for _ in range(3):
        got = chain(False)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


@pytest.mark.parametrize("B", [2, 20])
def test_decode_stack_sees_weights_written_just_before(R, B):
    """The decode stack's GEMMs copy weight rows before their wait; the call's
    first kernel starts only once earlier work is complete.  A weight is
    rewritten on the stream right before each call (no synchronisation), and
    every call must see the new values.  B = 2 runs the weight-streaming
    GEMM, B = 20 the tensor-core GEMM split over K."""
    dm, H, dk, dv, dff, L = 512, 4, 64, 128, 1024, 2
    gam = synth.head_gammas(H)
    shapes = dict(WQ=(dm, H * dk), WK=(dm, H * dk), WV=(dm, H * dv), WG=(dm, H * dv),
                  WO=(H * dv, dm), W1=(dm, dff), W2=(dff, dm))
    layers = []
    for li in range(L):
        W = {k: seeded(700 + li, k.lower(), shp, "bf16", std=0.05)[0] for k, shp in shapes.items()}
        for k in ("ln1_w", "ln2_w"):
            W[k] = torch.ones(dm, device="cuda")
        for k in ("ln1_b", "ln2_b"):
            W[k] = torch.zeros(dm, device="cuda")
        layers.append(W)
    base = {k: [W[k].clone() for W in layers] for k in shapes}
    X0, _ = seeded(702, "x", (B, dm), "bf16")
    d, _g = R.stack_desc(B, dm, H, dk, dv, dff, L, gam, pos=10)
    ws = R.new_workspace(int(R.lib.retnet_decode_workspace_size(d)), X0.device)

    def run(sync):
        for k in shapes:
            for W, w0 in zip(layers, base[k]):
                W[k].copy_(w0)
        X = X0.clone()
        S = [torch.zeros(B, H, dk, dv, device="cuda") for _ in range(L)]
        outs = []
        for t in range(4):
            # a different weight of each layer changes just before each step
            key = ("WQ", "WV", "W1", "W2")[t]
            for W in layers:
                W[key].mul_(-1.5)
            if sync:
                torch.cuda.synchronize()
            R.retnet_decode_step(X, layers, S, H=H, d_k=dk, d_v=dv, gamma=gam, pos=10 + t,
                                 workspace=ws)
            if sync:
                torch.cuda.synchronize()
            outs.append(X.clone())
        torch.cuda.synchronize()
        return outs

    ref = run(True)
    assert all(np.isfinite(o.float().cpu().numpy()).all() for o in ref)
    for _ in range(3):
        got = run(False)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
