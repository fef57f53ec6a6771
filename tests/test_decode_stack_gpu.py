"""GPU parity of the multi-layer decode step (retnet_decode_step) against the
oracle's stack of blocks run one token at a time with each layer's state
carried (oracle.msr.retnet_stack, pinned equal to the whole-sequence run in
test_oracle_decode_pins.py).

Tolerance: normwise max |gpu - ref| / max |ref| <= 3e-2 and RMS(gpu - ref) /
RMS(ref) <= 2e-2 over every step's output.  A float64 run with bf16
roundings at the GPU path's points (LayerNorm outputs, projections,
retention output, gate, W_O output, skip sums, FFN hidden, output) stays
within 1e-2 max and 8.5e-3 RMS of the oracle on these inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrent_sequence_gb300 import synth
from tests.helpers import host

pytestmark = pytest.mark.gpu

TOL_MAX_REL, TOL_RMS_REL = 3e-2, 2e-2
KEYS = (("wq", "WQ"), ("wk", "WK"), ("wv", "WV"), ("wg", "WG"), ("wo", "WO"), ("w1", "W1"),
        ("w2", "W2"))


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from linear_recurrent_sequence_gb300 import retention
    oracle.build()
    return retention


def stack_inputs(seed, n, dm, H, dk, dv, dff, std):
    """Per layer: (device dict, float64 dict) of the weights and LayerNorm
    parameters, seeds seed * 16 + layer."""
    dev, ref = [], []
    for layer in range(n):
        s = seed * 16 + layer
        D, W = {}, {}
        shapes = dict(WQ=(dm, H * dk), WK=(dm, H * dk), WV=(dm, H * dv), WG=(dm, H * dv),
                      WO=(H * dv, dm), W1=(dm, dff), W2=(dff, dm))
        for name, key in KEYS:
            bits, W[key] = synth.tensor(s, name, shapes[key], "bf16", std)
            D[key] = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
        _, z = synth.tensor(s, "ln", (4, dm), "f32", 0.1)
        ln = (z + np.array([1.0, 0.0, 1.0, 0.0])[:, None]).astype(np.float32)
        for i, key in enumerate(("ln1_w", "ln1_b", "ln2_w", "ln2_b")):
            D[key] = torch.from_numpy(ln[i].copy()).cuda()
            W[key] = ln[i].astype(np.float64)
        dev.append(D)
        ref.append(W)
    return dev, ref


def run_decode(R, seed, B, dm, H, dk, dv, dff, n, std, T, flags):
    from oracle.msr import retnet_stack
    gam = synth.head_gammas(H)
    dev, ref = stack_inputs(seed, n, dm, H, dk, dv, dff, std)
    bits, Xs = synth.tensor(seed, "x", (T, B, dm), "bf16", 1.0)
    Xd = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    S = [torch.zeros(B, H, dk, dv, device="cuda") for _ in range(n)]
    z = [torch.zeros(B, H, dk, device="cuda") for _ in range(n)]
    st = None
    worst = [0.0, 0.0]
    for t in range(T):
        X = Xd[t].clone()
        R.retnet_decode_step(X, dev, S, z, H=H, d_k=dk, d_v=dv, gamma=gam, pos=t,
                             norm_flags=flags)
        torch.cuda.synchronize()
        out, st = retnet_stack(Xs[t][:, None], ref, states=st, pos0=t, H=H, dk=dk, dv=dv,
                               gamma=gam, chunk=64, ln_eps=1e-5, norm_flags=flags, gn_eps=1e-6)
        d = host(X) - out[:, 0]
        worst[0] = max(worst[0], np.max(np.abs(d)) / np.max(np.abs(out)))
        worst[1] = max(worst[1], np.sqrt(np.mean(d ** 2) / np.mean(out ** 2)))
    assert worst[0] <= TOL_MAX_REL and worst[1] <= TOL_RMS_REL, worst
    for layer in range(n):  # the carried states against the oracle's
        rel = np.max(np.abs(host(S[layer]) - st[layer][0])) / np.max(np.abs(st[layer][0]))
        assert rel < 3e-2, (layer, rel)


def test_decode_small_stack_all_normalisations(R):
    """B=3 (the weight-streaming GEMM), two layers, six steps from zero states."""
    run_decode(R, 91, 3, 64, 2, 32, 64, 96, 2, 0.1, 6, oracle.NORM_ALL)


def test_decode_msr_shape_stack(R):
    """B=2, d_model=2048, H=8, d_k=256, d_v=512, d_ffn=4096, two layers, three steps."""
    run_decode(R, 91, 2, 2048, 8, 256, 512, 4096, 2, 0.02, 3, oracle.NORM_ALL)


def test_decode_batch_past_the_skinny_gemm(R):
    """B=20 rows: the projections take the general GEMM."""
    run_decode(R, 92, 20, 64, 2, 32, 64, 96, 1, 0.1, 3, 0)


def test_decode_batch_tensor_core_split(R):
    """B=20 rows with projection widths that the tensor-core GEMM takes
    (multiples of 256): the four input projections run as one job split over
    K into fp32 partials, added by the reduce with its epilogues.  One layer:
    with these weights a second layer makes batch row 14 ill-conditioned
    (its second-layer retention output is near zero before GroupNorm), and
    the weight-streaming path, which the other tests pin, shows the same
    0.19 deviation there, so it says nothing about this GEMM."""
    R.lib.retention_kernel_timer_reset()
    run_decode(R, 93, 20, 256, 2, 128, 128, 512, 1, 0.05, 3, oracle.NORM_ALL)
    torch.cuda.synchronize()
    names = R.kernel_times()
    assert "gemm_tc" in names and "skinny_reduce" in names and "gemm_skinny" not in names, names
