"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle
on the same seeded inputs, for every workload shape and the edge cases.

Workloads (seed = 1000 + index):
  1. fp32, B=1 H=1 N=64 d_k=d_v=32, gamma=0.9, chunk 16: parallel, recurrent
     and chunkwise forms.
  2. bf16, B=4 H=8 N=2048 d_k=128 d_v=256, gamma_h = 1-2^(-5-h), chunk 64,
     all three normalisations, GroupNorm.
  3. bf16, B=1 H=16 N=8192 d_k=256 d_v=512, chunks 64/128/256 (heads
     0, 5, 10, 15 compared in full).
  4. decode: H=16 d_k=256 d_v=512, state from a 1024-token chunkwise prefill,
     then one-token steps.
  5. MSR layer: B=2 N=4096 d=2048 H=8 d_k=256 d_v=512, chunk 128.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrent_sequence_gb300 import synth
from tests.helpers import check_bf16, check_f32, host, operand_sensitivity, seeded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from linear_recurrent_sequence_gb300 import retention
    oracle.build()
    return retention


def inputs(seed, B, H, N, dk, dv, dtype):
    q, q64 = seeded(seed, "q", (B, H, N, dk), dtype)
    k, k64 = seeded(seed, "k", (B, H, N, dk), dtype)
    v, v64 = seeded(seed, "v", (B, H, N, dv), dtype)
    return (q, k, v), (q64, k64, v64)


# ------------------------------------------------------------------ config 1
@pytest.mark.parametrize("flags", [0, oracle.NORM_ALL])
def test_config1_fp32_three_forms(R, flags):
    B, H, N, dk, dv, C = 1, 1, 64, 32, 32, 16
    (q, k, v), (q64, k64, v64) = inputs(1001, B, H, N, dk, dv, "f32")
    p = oracle.Problem(B, H, N, dk, dv, 0.9, norm_flags=flags, gn_eps=1e-6)
    ref = oracle.parallel(p, q64, k64, v64)
    o_par = R.parallel_fwd(q, k, v, [0.9], norm_flags=flags)
    check_f32(host(o_par), ref, "parallel")
    o_ch = R.chunkwise_fwd(q, k, v, [0.9], chunk=C, norm_flags=flags)
    check_f32(host(o_ch), ref, "chunkwise")
    S = torch.zeros(B, H, dk, dv, device="cuda")
    z = torch.zeros(B, H, dk, device="cuda")
    outs = [R.recurrent_step(q[:, :, t], k[:, :, t], v[:, :, t], S, [0.9], z=z, pos=t,
                             norm_flags=flags) for t in range(N)]
    check_f32(host(torch.cat(outs, dim=2)), ref, "recurrent")
    _, S_ref, _ = oracle.recurrent(p, q64, k64, v64)
    check_f32(host(S), S_ref, "state")


# ------------------------------------------------------------------ config 2
def test_config2_training_shape(R):
    B, H, N, dk, dv, C = 4, 8, 2048, 128, 256, 64
    (q, k, v), (q64, k64, v64) = inputs(1002, B, H, N, dk, dv, "bf16")
    gam = synth.head_gammas(H)
    S_out = torch.empty(B, H, dk, dv, device="cuda")
    o = R.chunkwise_fwd(q, k, v, gam, chunk=C, norm_flags=R.NORM_ALL, S_out=S_out)
    p = oracle.Problem(B, H, N, dk, dv, gam, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    ref, S_ref, _ = oracle.chunkwise(p, C, q64, k64, v64)
    check_bf16(host(o), ref, "config2 output")
    rel = np.max(np.abs(host(S_out) - S_ref)) / np.max(np.abs(S_ref))
    assert rel < 1e-2, rel


# ------------------------------------------------------------------ config 3
HEADS3 = [0, 5, 10, 15]


@pytest.fixture(scope="module")
def config3(R):
    B, H, N, dk, dv = 1, 16, 8192, 256, 512
    (q, k, v), (q64, k64, v64) = inputs(1003, B, H, N, dk, dv, "bf16")
    gam = synth.head_gammas(H)
    sel = HEADS3
    p = oracle.Problem(B, len(sel), N, dk, dv, gam[sel], norm_flags=oracle.NORM_ALL,
                       gn_eps=1e-6)
    ref, S_ref, _ = oracle.chunkwise(p, 256, q64[:, sel], k64[:, sel], v64[:, sel])
    return (q, k, v), gam, ref, S_ref


@pytest.mark.parametrize("C,odt", [(64, torch.bfloat16), (128, torch.bfloat16),
                                   (256, torch.bfloat16), (64, torch.float32)])
def test_config3_long_sequence(R, config3, C, odt):
    """bf16 output (the bench's form) and fp32 output, which shows the
    arithmetic error with no storage rounding on top."""
    (q, k, v), gam, ref, S_ref = config3
    S_out = torch.empty(1, 16, 256, 512, device="cuda")
    o = R.chunkwise_fwd(q, k, v, gam, chunk=C, norm_flags=R.NORM_ALL, S_out=S_out,
                        out_dtype=odt)
    check_bf16(host(o[:, HEADS3]), ref, f"config3 C={C} {odt}")
    rel = np.max(np.abs(host(S_out[:, HEADS3]) - S_ref)) / np.max(np.abs(S_ref))
    assert rel < 1e-2, rel


# ------------------------------------------------------------------ config 4
# Prefill of 1024 tokens by the chunkwise form, then 2048 one-token decode
# steps, as the workload states.  The inputs are drawn on the host with
# torch's seeded CPU generator (1.6e9 values at B=32: the splitmix generator
# of synth is too slow for that size) and rounded to bf16; the device and the
# oracle get the same bits.
DEC_H, DEC_DK, DEC_DV, DEC_P, DEC_T = 16, 256, 512, 1024, 2048


def _host_bf16(seed, shape):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).bfloat16()


def _decode_run(R, q, k, v, gam, keep=None, odt=torch.bfloat16):
    """Prefill then every decode step on the device; returns (prefill
    output, decode outputs [B, H, T, dv] or only the (b, h) pairs in keep,
    final S)."""
    B = q.shape[0]
    P, T = DEC_P, DEC_T
    S = torch.empty(B, DEC_H, DEC_DK, DEC_DV, device="cuda")
    o_pre = R.chunkwise_fwd(q[:, :, :P], k[:, :, :P], v[:, :, :P], gam, chunk=64, S_out=S,
                            out_dtype=odt)
    if keep is None:
        out = torch.empty(B, DEC_H, T, DEC_DV, dtype=odt, device="cuda")
    else:
        out = torch.empty(len(keep), T, DEC_DV, dtype=torch.bfloat16, device="cuda")
        o_t = torch.empty(B, DEC_H, 1, DEC_DV, dtype=torch.bfloat16, device="cuda")
        bi = torch.tensor([b for b, _ in keep], device="cuda")
        hi = torch.tensor([h for _, h in keep], device="cuda")
    ws = R.new_workspace(256, "cuda")
    for t in range(T):
        pos = P + t
        if keep is None:
            R.recurrent_step(q[:, :, pos], k[:, :, pos], v[:, :, pos], S, gam, pos=pos,
                             out=out[:, :, t:t + 1], workspace=ws)
        else:
            R.recurrent_step(q[:, :, pos], k[:, :, pos], v[:, :, pos], S, gam, pos=pos,
                             out=o_t, workspace=ws)
            out[:, t] = o_t[bi, hi, 0]
    torch.cuda.synchronize()
    assert R.poll_status(ws) == 0
    return o_pre, out, S


@pytest.mark.parametrize("B,odt", [(1, torch.bfloat16), (32, torch.bfloat16),
                                   (1, torch.float32)])
def test_config4_decode_2048_steps(R, B, odt):
    """Every (batch, head) pair, every one of the 2048 steps and the final
    fp32 state against the oracle's chunkwise form over all 3072 tokens
    (equal to the recurrent form by the oracle's pins), so that any drift of
    the fp32 state over the steps shows.  bf16 outputs, and fp32 outputs
    (the arithmetic error with no storage rounding on top)."""
    N = DEC_P + DEC_T
    gam = synth.head_gammas(DEC_H)
    qh = _host_bf16(40401 + B, (B, DEC_H, N, DEC_DK))
    kh = _host_bf16(40402 + B, (B, DEC_H, N, DEC_DK))
    vh = _host_bf16(40403 + B, (B, DEC_H, N, DEC_DV))
    o_pre, out, S = _decode_run(R, qh.cuda(), kh.cuda(), vh.cuda(), gam, odt=odt)
    o_pre, out, S = host(o_pre), host(out), host(S)
    p = oracle.Problem(1, DEC_H, N, DEC_DK, DEC_DV, gam, gn_eps=1e-6)
    pp = oracle.Problem(1, DEC_H, DEC_P, DEC_DK, DEC_DV, gam, gn_eps=1e-6)
    for b in range(B):
        ref, S_ref, _ = oracle.chunkwise(p, 64, qh[b:b + 1].double().numpy(),
                                         kh[b:b + 1].double().numpy(),
                                         vh[b:b + 1].double().numpy())
        # The prefill runs on the tensor cores (fp16 operands): rows whose
        # exact result is itself sensitive to rounding q and k at fp16
        # precision get that sensitivity added to their bound.
        v64 = vh[b:b + 1, :, :DEC_P].double().numpy()
        spread = operand_sensitivity(
            lambda q_, k_: oracle.chunkwise(pp, 64, q_, k_, v64)[0],
            qh[b:b + 1, :, :DEC_P].double().numpy(), kh[b:b + 1, :, :DEC_P].double().numpy())
        check_bf16(o_pre[b:b + 1], ref[:, :, :DEC_P], f"prefill b={b}", spread=spread)
        check_bf16(out[b:b + 1], ref[:, :, DEC_P:], f"decode steps b={b}")
        rel = np.max(np.abs(S[b:b + 1] - S_ref)) / np.max(np.abs(S_ref))
        assert rel < 1e-2, (b, rel)


def test_config4_decode_full_batch_sampled(R):
    """Decode at the largest bench batch (B=128, H=16: the 8-rows-a-thread
    form of the decode kernel) after the full 1024-token prefill, all 2048
    steps.  Three (batch, head) pairs carry seeded inputs and are compared
    with the oracle at every step and in the final state; the other pairs
    are device random numbers that only fill the launch (pairs are
    independent)."""
    B, N = 128, DEC_P + DEC_T
    g = torch.Generator(device="cuda").manual_seed(4040)
    q = torch.randn(B, DEC_H, N, DEC_DK, device="cuda", generator=g).bfloat16()
    k = torch.randn(B, DEC_H, N, DEC_DK, device="cuda", generator=g).bfloat16()
    v = torch.randn(B, DEC_H, N, DEC_DV, device="cuda", generator=g).bfloat16()
    samples = [(0, 0), (63, 7), (127, 15)]
    ref_in = {}
    for i, (b, h) in enumerate(samples):
        qs = _host_bf16(41000 + 3 * i, (N, DEC_DK))
        ks = _host_bf16(41001 + 3 * i, (N, DEC_DK))
        vs = _host_bf16(41002 + 3 * i, (N, DEC_DV))
        q[b, h], k[b, h], v[b, h] = qs.cuda(), ks.cuda(), vs.cuda()
        ref_in[(b, h)] = (qs, ks, vs)
    gam = synth.head_gammas(DEC_H)
    o_pre, out, S = _decode_run(R, q, k, v, gam, keep=samples)
    for i, ((b, h), (qs, ks, vs)) in enumerate(ref_in.items()):
        p = oracle.Problem(1, 1, N, DEC_DK, DEC_DV, [gam[h]], gn_eps=1e-6)
        ref, S_ref, _ = oracle.chunkwise(p, 64, qs.double().numpy()[None, None],
                                         ks.double().numpy()[None, None],
                                         vs.double().numpy()[None, None])
        check_bf16(host(o_pre[b:b + 1, h:h + 1]), ref[:, :, :DEC_P], f"prefill ({b},{h})")
        check_bf16(host(out[i])[None, None], ref[:, :, DEC_P:], f"decode B=128 ({b},{h})")
        rel = np.max(np.abs(host(S[b, h]) - S_ref[0, 0])) / np.max(np.abs(S_ref))
        assert rel < 1e-2, ((b, h), rel)


@pytest.mark.parametrize("dk,dv,flags,gn,odt", [
    (256, 1024, 0, 1e-6, torch.bfloat16),             # 8 CTAs, two column slices a thread
    (64, 20, oracle.NORM_ALL, 1e-6, torch.float32),   # one CTA: two row blocks, 20 columns
    (96, 96, oracle.NORM_ALL, None, torch.float32),   # 8 CTAs of 12 rows, no GroupNorm
    (2, 4, 0, 1e-6, torch.float32),                   # smallest shape
    (256, 512, oracle.NORM_ALL, 1e-6, torch.float32),  # decode head shape, with z
])
def test_decode_shapes(R, dk, dv, flags, gn, odt):
    """Decode steps from a random fp32 (S, z) at absolute positions 5000..,
    on shapes that take each path of the decode kernel (cluster sizes 1 and
    8, several row blocks or column slices per thread, GroupNorm off)."""
    B, H, T, pos = 2, 3, 4, 5000
    (q, k, v), (q64, k64, v64) = inputs(4242 + dk + dv, B, H, T, dk, dv, "bf16")
    gam = [0.9, 0.99, 1.0]
    _decode_steps_vs_oracle(R, B, H, T, pos, dk, dv, flags, gn, odt, gam, q, k, v, q64, k64, v64)


def test_decode_many_heads_with_z(R):
    """B*H*8 CTAs above the SM count take the 8-rows-a-thread form of the
    decode kernel; all three normalisations and z on, fp32 output."""
    B, H, T, pos, dk, dv = 3, 16, 3, 777, 256, 512
    (q, k, v), (q64, k64, v64) = inputs(4747, B, H, T, dk, dv, "bf16")
    gam = synth.head_gammas(H)
    _decode_steps_vs_oracle(R, B, H, T, pos, dk, dv, oracle.NORM_ALL, 1e-6, torch.float32, gam,
                            q, k, v, q64, k64, v64)


def _decode_steps_vs_oracle(R, B, H, T, pos, dk, dv, flags, gn, odt, gam, q, k, v, q64, k64, v64):
    S, S64 = seeded(4343, "S", (B, H, dk, dv), "f32")
    z, z64 = seeded(4343, "z", (B, H, dk), "f32")
    outs = [R.recurrent_step(q[:, :, t], k[:, :, t], v[:, :, t], S, gam, z=z, pos=pos + t,
                             norm_flags=flags, gn_eps=gn, out_dtype=odt) for t in range(T)]
    p = oracle.Problem(B, H, T, dk, dv, gam, pos0=pos, norm_flags=flags, gn_eps=gn)
    ref, S_ref, z_ref = oracle.recurrent(p, q64, k64, v64, S_in=S64, z_in=z64)
    got = host(torch.cat(outs, dim=2))
    if odt == torch.bfloat16:
        check_bf16(got, ref, "decode out")
    else:
        check_f32(got, ref, "decode out")
    check_f32(host(S), S_ref, "decode S")
    if flags & oracle.NORM_RSUM:
        check_f32(host(z), z_ref, "decode z")


# ------------------------------------------------------------------ config 5
def test_config5_msr_layer(R):
    from oracle.msr import msr_layer
    B, N, dm, H, dk, dv, C = 2, 4096, 2048, 8, 256, 512, 128
    X, X64 = seeded(1005, "x", (B, N, dm), "bf16")
    W = {}
    for name, shp in (("wq", (dm, H * dk)), ("wk", (dm, H * dk)), ("wv", (dm, H * dv)),
                      ("wg", (dm, H * dv)), ("wo", (H * dv, dm))):
        W[name] = seeded(1005, name, shp, "bf16", std=0.02)
    gam = synth.head_gammas(H)
    Y = R.msr_layer_fwd(X, W["wq"][0], W["wk"][0], W["wv"][0], W["wg"][0], W["wo"][0], H=H,
                        d_k=dk, d_v=dv, gamma=gam, chunk=C, norm_flags=R.NORM_ALL)
    ref = msr_layer(X64, W["wq"][1], W["wk"][1], W["wv"][1], W["wg"][1], W["wo"][1], H=H,
                    dk=dk, dv=dv, gamma=gam, chunk=C, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    check_bf16(host(Y), ref, "msr layer")


# ------------------------------------------------------------------ edges
def test_ragged_tail_gamma_extremes_and_strides(R):
    """N not a multiple of the chunk, gamma 0 and 1 among the heads, pos0 > 0,
    [B,N,H,d] strided views, fp32 output from bf16 input."""
    B, H, N, dk, dv = 2, 3, 203, 64, 96
    qb, q64 = seeded(77, "q", (B, N, H, dk), "bf16")
    kb, k64 = seeded(77, "k", (B, N, H, dk), "bf16")
    vb, v64 = seeded(77, "v", (B, N, H, dv), "bf16")
    q, k, v = (t.permute(0, 2, 1, 3) for t in (qb, kb, vb))
    gam = [0.0, 0.97, 1.0]
    p = oracle.Problem(B, H, N, dk, dv, gam, pos0=11, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    ref = oracle.parallel(p, q64.transpose(0, 2, 1, 3), k64.transpose(0, 2, 1, 3),
                          v64.transpose(0, 2, 1, 3))
    out = torch.empty(B, N, H, dv, device="cuda").permute(0, 2, 1, 3)
    for C in (16, 64, 128):
        R.chunkwise_fwd(q, k, v, gam, chunk=C, pos0=11, norm_flags=R.NORM_ALL, out=out)
        check_bf16(host(out), ref, f"ragged C={C}")
    o = R.parallel_fwd(q, k, v, gam, pos0=11, norm_flags=R.NORM_ALL, out_dtype=torch.float32)
    check_bf16(host(o), ref, "parallel strided")


def test_state_passing_and_aliasing(R):
    """Two chunkwise calls with the carried (S, z), S_out aliasing S_in, equal
    one call over the whole sequence; N = 0 passes the state through."""
    B, H, N, dk, dv = 1, 2, 300, 32, 64
    (q, k, v), (q64, k64, v64) = inputs(91, B, H, N, dk, dv, "f32")
    gam = [0.9, 0.999]
    p = oracle.Problem(B, H, N, dk, dv, gam, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    ref, S_ref, z_ref = oracle.chunkwise(p, 64, q64, k64, v64)
    S = torch.zeros(B, H, dk, dv, device="cuda")
    z = torch.zeros(B, H, dk, device="cuda")
    a = 137
    o1 = R.chunkwise_fwd(q[:, :, :a], k[:, :, :a], v[:, :, :a], gam, chunk=32,
                         norm_flags=R.NORM_ALL, S_in=S, z_in=z, S_out=S, z_out=z)
    o2 = R.chunkwise_fwd(q[:, :, a:], k[:, :, a:], v[:, :, a:], gam, chunk=64, pos0=a,
                         norm_flags=R.NORM_ALL, S_in=S, z_in=z, S_out=S, z_out=z)
    check_f32(host(torch.cat([o1, o2], dim=2)), ref, "split")
    check_f32(host(S), S_ref, "S")
    check_f32(host(z), z_ref, "z")
    S2, z2 = torch.empty_like(S), torch.empty_like(z)
    R.chunkwise_fwd(q[:, :, :0], k[:, :, :0], v[:, :, :0], gam, S_in=S, z_in=z, S_out=S2,
                    z_out=z2, pos0=N)
    assert torch.equal(S2, S) and torch.equal(z2, z)


def test_checkpoint_through_host_is_bitwise(R):
    """The resumable state of the method is (S, z, position).  Prefill, copy
    (S, z) to the host, wipe and restore them, then continue with a second
    chunkwise call and decode steps: bitwise equal to the same calls without
    the round trip (every reduction has a fixed order)."""
    B, H, N, dk, dv, P = 1, 4, 640, 256, 512, 384
    (q, k, v), _ = inputs(515, B, H, N, dk, dv, "bf16")
    gam = synth.head_gammas(H)

    def run(via_host):
        S = torch.empty(B, H, dk, dv, device="cuda")
        z = torch.empty(B, H, dk, device="cuda")
        o1 = R.chunkwise_fwd(q[:, :, :P], k[:, :, :P], v[:, :, :P], gam, chunk=64,
                             norm_flags=R.NORM_ALL, S_out=S, z_out=z)
        if via_host:
            S_h, z_h = S.cpu(), z.cpu()
            S.fill_(float("nan"))
            z.fill_(float("nan"))
            S.copy_(S_h)
            z.copy_(z_h)
        o2 = R.chunkwise_fwd(q[:, :, P:N - 2], k[:, :, P:N - 2], v[:, :, P:N - 2], gam,
                             chunk=64, pos0=P, norm_flags=R.NORM_ALL, S_in=S, z_in=z,
                             S_out=S, z_out=z)
        o3 = [R.recurrent_step(q[:, :, t], k[:, :, t], v[:, :, t], S, gam, z=z, pos=t,
                               norm_flags=R.NORM_ALL) for t in (N - 2, N - 1)]
        return torch.cat([o1, o2] + o3, dim=2), S, z

    a, Sa, za = run(False)
    b, Sb, zb = run(True)
    assert torch.equal(a, b) and torch.equal(Sa, Sb) and torch.equal(za, zb)


def test_single_token_and_no_groupnorm(R):
    B, H, N, dk, dv = 2, 2, 1, 16, 8
    (q, k, v), (q64, k64, v64) = inputs(5, B, H, N, dk, dv, "f32")
    p = oracle.Problem(B, H, N, dk, dv, [0.5, 0.8], gn_eps=-1.0)
    ref = oracle.parallel(p, q64, k64, v64)
    o = R.chunkwise_fwd(q, k, v, [0.5, 0.8], gn_eps=None)
    check_f32(host(o), ref, "N=1 raw")


@pytest.mark.parametrize("dtype,dk,dv,chunk", [("bf16", 128, 128, 64), ("f32", 32, 48, 16)])
def test_negative_row_sums_without_groupnorm(R, dtype, dk, dv, chunk):
    """Keys are the negated queries, so each row's own term q_n . k_n =
    -|q_n|^2 dominates and most row sums of R fall below -1: the third
    normalisation must divide by |sum R| (hwhale.com/article/285883, R_nm /
    max(|sum_i R_ni|, 1)).  GroupNorm is off, so r(n) reaches the output
    (with GroupNorm on, r only rescales a row).  bf16 takes the tensor-core
    kernel (N ragged against its 64-token chunk), fp32 the CUDA-core forms."""
    B, H, N = 1, 2, 200
    q, q64 = seeded(6161, "q", (B, H, N, dk), dtype)
    v, v64 = seeded(6161, "v", (B, H, N, dv), dtype)
    k, k64 = -q, -q64
    gam = [0.9, 0.97]
    p = oracle.Problem(B, H, N, dk, dv, gam, norm_flags=oracle.NORM_ALL, gn_eps=-1.0)
    ref = oracle.parallel(p, q64, k64, v64)
    # coverage: the row sums (first two normalisations applied; v = 1)
    p1 = oracle.Problem(B, H, N, dk, 1, gam, norm_flags=oracle.NORM_SCALE | oracle.NORM_DROW,
                        gn_eps=-1.0)
    rowsum = oracle.parallel(p1, q64, k64, np.ones((B, H, N, 1)))[..., 0]
    assert (rowsum < -1.0).mean() > 0.5
    R.lib.retention_kernel_timer_reset()
    o = R.chunkwise_fwd(q, k, v, gam, chunk=chunk, norm_flags=R.NORM_ALL, gn_eps=None,
                        out_dtype=torch.float32)
    torch.cuda.synchronize()
    if dtype == "bf16":
        assert "chunk_tc" in R.kernel_times()
        check_bf16(host(o), ref, "row sums < -1, tensor cores")
    else:
        check_f32(host(o), ref, "row sums < -1, chunkwise")
        o = R.parallel_fwd(q, k, v, gam, norm_flags=R.NORM_ALL, gn_eps=None,
                           out_dtype=torch.float32)
        check_f32(host(o), ref, "row sums < -1, parallel")
        S = torch.zeros(B, H, dk, dv, device="cuda")
        z = torch.zeros(B, H, dk, device="cuda")
        outs = [R.recurrent_step(q[:, :, t], k[:, :, t], v[:, :, t], S, gam, z=z, pos=t,
                                 norm_flags=R.NORM_ALL, gn_eps=None, out_dtype=torch.float32)
                for t in range(N)]
        check_f32(host(torch.cat(outs, dim=2)), ref, "row sums < -1, recurrent")


def test_rotate_entry_point(R):
    x, x64 = seeded(3, "q", (1, 2, 50, 64), "f32")
    got = R.rotate(x, pos0=4000, theta_base=10000.0)
    p = oracle.Problem(1, 2, 50, 64, 1, [0.9, 0.9], pos0=4000)
    ref = oracle.rotate(p, x64, 64)
    assert np.max(np.abs(host(got) - ref)) < 5e-6


def test_workspace_status_is_clean(R):
    ws = R.new_workspace(1 << 20, "cuda")
    assert R.poll_status(ws) == 0


def test_zero_report_budget_surfaces_a_timeout(R):
    """With no tries for the prologue's reporting wait, every TMA wait there
    records RET_ETIMEOUT; the bounded data wait behind it keeps the output
    valid, retention_poll_status reports and clears the word, and the next
    call runs clean (the context stays usable)."""
    B, H, N, dk, dv = 1, 2, 256, 64, 128
    (q, k, v), (q64, k64, v64) = inputs(31, B, H, N, dk, dv, "bf16")
    gam = synth.head_gammas(H)
    o = torch.empty(B, H, N, dv, device="cuda", dtype=torch.bfloat16)
    d, _g = R.make_desc(q, k, v, o, gam, chunk=64, norm_flags=R.NORM_ALL)
    ws = R.new_workspace(R.workspace_size(d), "cuda")
    R.lib.retention_set_report_wait_budget(0)
    try:
        R.chunkwise_fwd(q, k, v, gam, chunk=64, norm_flags=R.NORM_ALL, out=o, workspace=ws)
        st = R.poll_status(ws)
    finally:
        R.lib.retention_set_report_wait_budget(1 << 24)
    assert R.STATUS[st] == "RET_ETIMEOUT", st
    p = oracle.Problem(B, H, N, dk, dv, gam, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    ref, _, _ = oracle.chunkwise(p, 64, q64, k64, v64)
    check_bf16(host(o), ref, "output under a reported timeout")
    o2 = R.chunkwise_fwd(q, k, v, gam, chunk=64, norm_flags=R.NORM_ALL, workspace=ws)
    assert R.poll_status(ws) == 0
    assert torch.equal(o2, o)


# ------------------------------------------------------------------ tensor-core chunk kernel
@pytest.mark.parametrize("B,H,N,dk,dv", [
    (1, 2, 64, 64, 128),      # one chunk, cluster of 1
    (2, 3, 333, 128, 256),    # ragged tail, cluster of 2
    (1, 2, 200, 192, 384),    # d_k not a power of two, cluster of 3
    (1, 1, 130, 256, 1024),   # cluster of 8
])
@pytest.mark.parametrize("flags", [0, oracle.NORM_ALL])
def test_tc_chunk_shapes(R, B, H, N, dk, dv, flags):
    (q, k, v), (q64, k64, v64) = inputs(2000 + dk + dv, B, H, N, dk, dv, "bf16")
    gam = [0.85, 0.96875, 0.999, 1.0][:H] if H <= 4 else synth.head_gammas(H)
    S = torch.empty(B, H, dk, dv, device="cuda")
    z = torch.empty(B, H, dk, device="cuda")
    o = R.chunkwise_fwd(q, k, v, gam, chunk=64, norm_flags=flags, S_out=S, z_out=z, pos0=5)
    p = oracle.Problem(B, H, N, dk, dv, gam, pos0=5, norm_flags=flags, gn_eps=1e-6)
    ref, S_ref, z_ref = oracle.chunkwise(p, 64, q64, k64, v64)
    check_bf16(host(o), ref, f"tc {B}x{H}x{N} dk{dk} dv{dv}")
    assert np.max(np.abs(host(S) - S_ref)) / np.max(np.abs(S_ref)) < 1e-2
    assert np.max(np.abs(host(z) - z_ref)) / np.max(np.abs(z_ref)) < 1e-2


@pytest.mark.parametrize("N", [1, 63, 65])
def test_tc_chunk_path_at_chunk_edges(R, N):
    """The tensor-core chunk path at the shortest sequences (one token; one
    token short of and one past a 64-token chunk), all normalisations, a
    carried (S, z) in and out."""
    B, H, dk, dv = 1, 2, 128, 256
    (q, k, v), (q64, k64, v64) = inputs(2700 + N, B, H, N, dk, dv, "bf16")
    gam = [0.96875, 0.999]
    S0, S064 = seeded(2750, "S", (B, H, dk, dv), "f32")
    z0, z064 = seeded(2750, "z", (B, H, dk), "f32")
    S = torch.empty_like(S0)
    z = torch.empty_like(z0)
    R.lib.retention_kernel_timer_reset()
    o = R.chunkwise_fwd(q, k, v, gam, chunk=64, norm_flags=R.NORM_ALL, pos0=40, S_in=S0, z_in=z0,
                        S_out=S, z_out=z)
    torch.cuda.synchronize()
    assert "chunk_tc" in R.kernel_times()
    p = oracle.Problem(B, H, N, dk, dv, gam, pos0=40, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    ref, S_ref, z_ref = oracle.chunkwise(p, 64, q64, k64, v64, S064, z064)
    check_bf16(host(o), ref, f"tc chunk path N={N}")
    assert np.max(np.abs(host(S) - S_ref)) / np.max(np.abs(S_ref)) < 1e-2
    assert np.max(np.abs(host(z) - z_ref)) / np.max(np.abs(z_ref)) < 1e-2


def test_max_heads_every_path(R):
    """RET_MAX_HEADS (256) heads, so the last heads' constants (gamma and
    its logarithm, the decay sums) reach every kernel: the chunkwise
    tensor-core path over 130 tokens, one decode step that continues from
    its state, and the parallel form of the same 130 tokens, each against
    the oracle's chunkwise run over all 131 tokens."""
    B, H, N, dk, dv = 1, 256, 130, 64, 128
    (q, k, v), (q64, k64, v64) = inputs(2600, B, H, N + 1, dk, dv, "bf16")
    gam = synth.head_gammas(H)
    S = torch.empty(B, H, dk, dv, device="cuda")
    z = torch.empty(B, H, dk, device="cuda")
    o = R.chunkwise_fwd(q[:, :, :N], k[:, :, :N], v[:, :, :N], gam, chunk=64,
                        norm_flags=R.NORM_ALL, S_out=S, z_out=z)
    o_last = R.recurrent_step(q[:, :, N], k[:, :, N], v[:, :, N], S, gam, z=z, pos=N,
                              norm_flags=R.NORM_ALL)
    o_par = R.parallel_fwd(q[:, :, :N], k[:, :, :N], v[:, :, :N], gam, norm_flags=R.NORM_ALL)
    p = oracle.Problem(B, H, N + 1, dk, dv, gam, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    ref, _, _ = oracle.chunkwise(p, 64, q64, k64, v64)
    check_bf16(host(o), ref[:, :, :N], "256 heads, chunkwise")
    check_bf16(host(o_last).reshape(B, H, 1, dv), ref[:, :, N:], "256 heads, decode step")
    check_bf16(host(o_par), ref[:, :, :N], "256 heads, parallel form")


def test_tc_chunk_state_in_strided_fp32_out(R):
    """Carried (S, z) in, [B,N,H,d] strided q/k/v/o, fp32 output, two calls
    that split the sequence (state passed through aliasing S_out = S_in)."""
    B, H, N, dk, dv = 2, 2, 300, 128, 256
    qb, q64 = seeded(31, "q", (B, N, H, dk), "bf16")
    kb, k64 = seeded(31, "k", (B, N, H, dk), "bf16")
    vb, v64 = seeded(31, "v", (B, N, H, dv), "bf16")
    q, k, v = (t.permute(0, 2, 1, 3) for t in (qb, kb, vb))
    gam = [0.97, 0.995]
    S0 = torch.randn(B, H, dk, dv, device="cuda")
    z0 = torch.randn(B, H, dk, device="cuda")
    p = oracle.Problem(B, H, N, dk, dv, gam, pos0=40, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    ref, S_ref, _ = oracle.chunkwise(p, 64, q64.transpose(0, 2, 1, 3), k64.transpose(0, 2, 1, 3),
                                     v64.transpose(0, 2, 1, 3), S0.double().cpu().numpy(),
                                     z0.double().cpu().numpy())
    out = torch.empty(B, N, H, dv, device="cuda", dtype=torch.float32).permute(0, 2, 1, 3)
    S, z = S0.clone(), z0.clone()
    a = 128
    R.chunkwise_fwd(q[:, :, :a], k[:, :, :a], v[:, :, :a], gam, chunk=64, pos0=40,
                    norm_flags=R.NORM_ALL, S_in=S, z_in=z, S_out=S, z_out=z, out=out[:, :, :a])
    R.chunkwise_fwd(q[:, :, a:], k[:, :, a:], v[:, :, a:], gam, chunk=64, pos0=40 + a,
                    norm_flags=R.NORM_ALL, S_in=S, z_in=z, S_out=S, z_out=z, out=out[:, :, a:])
    check_bf16(host(out), ref, "tc strided split")
    assert np.max(np.abs(host(S) - S_ref)) / np.max(np.abs(S_ref)) < 1e-2


def test_tc_msr_layer_chunk64(R):
    """The gated MSR layer with chunk 64: tensor-core chunk kernel, gate in
    the W_G GEMM's epilogue."""
    from oracle.msr import msr_layer
    B, N, dm, H, dk, dv = 1, 256, 256, 2, 64, 128
    X, X64 = seeded(77, "x", (B, N, dm), "bf16")
    W = {}
    for name, shp in (("wq", (dm, H * dk)), ("wk", (dm, H * dk)), ("wv", (dm, H * dv)),
                      ("wg", (dm, H * dv)), ("wo", (H * dv, dm))):
        W[name] = seeded(77, name, shp, "bf16", std=0.05)
    gam = synth.head_gammas(H)
    Y = R.msr_layer_fwd(X, W["wq"][0], W["wk"][0], W["wv"][0], W["wg"][0], W["wo"][0], H=H,
                        d_k=dk, d_v=dv, gamma=gam, chunk=64, norm_flags=R.NORM_ALL)
    ref = msr_layer(X64, W["wq"][1], W["wk"][1], W["wv"][1], W["wg"][1], W["wo"][1], H=H,
                    dk=dk, dv=dv, gamma=gam, chunk=64, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    check_bf16(host(Y), ref, "msr chunk 64")


def test_msr_layer_ragged_tokens_gate_pass(R):
    """B*N not a multiple of the GEMM tile: CUDA-core projections and the
    gate as its own pass (swish_gate_kernel).

    Tolerance rule for ill-conditioned tokens: the layer is also evaluated in
    float64 with its intermediates rounded to bf16 where the GPU path stores
    them (the projections Q, K, V, G, the retention output, the gated
    product, the output).  Tokens on which that rounded run moves by more
    than the tolerance from the unrounded one are ill-conditioned (with
    these inputs the first token's retention output is tiny, and GroupNorm
    with eps 1e-6 turns the rounding of q and k into an O(1) change); they
    are compared with the rounded run, every other token with the unrounded
    oracle, both at the stated bf16 tolerance."""
    from oracle.msr import msr_layer, swish
    from tests.helpers import bf16_round, split_ill_conditioned
    B, N, dm, H, dk, dv = 1, 100, 64, 2, 32, 64
    X, X64 = seeded(66, "x", (B, N, dm), "bf16")
    W = {}
    for name, shp in (("wq", (dm, H * dk)), ("wk", (dm, H * dk)), ("wv", (dm, H * dv)),
                      ("wg", (dm, H * dv)), ("wo", (H * dv, dm))):
        W[name] = seeded(66, name, shp, "bf16", std=0.1)
    gam = synth.head_gammas(H)
    R.lib.retention_kernel_timer_reset()
    Y = R.msr_layer_fwd(X, W["wq"][0], W["wk"][0], W["wv"][0], W["wg"][0], W["wo"][0], H=H,
                        d_k=dk, d_v=dv, gamma=gam, chunk=16, norm_flags=R.NORM_ALL)
    torch.cuda.synchronize()
    names = R.kernel_times()
    assert "swish_gate" in names and "gemm_simt" in names, names
    ref = msr_layer(X64, W["wq"][1], W["wk"][1], W["wv"][1], W["wg"][1], W["wo"][1], H=H,
                    dk=dk, dv=dv, gamma=gam, chunk=16, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    # the same layer with bf16 rounding at the GPU path's storage points
    Q, K, V, G = (bf16_round(X64 @ W[n][1]) for n in ("wq", "wk", "wv", "wg"))
    heads = lambda A, d: A.reshape(B, N, H, d).transpose(0, 2, 1, 3)
    p = oracle.Problem(B, H, N, dk, dv, gam, rotate=True, norm_flags=oracle.NORM_ALL,
                       gn_eps=1e-6)
    o, _, _ = oracle.chunkwise(p, 16, heads(Q, dk), heads(K, dk), heads(V, dv))
    Yr = bf16_round(o.transpose(0, 2, 1, 3).reshape(B, N, H * dv))
    ref_r = bf16_round(bf16_round(swish(G) * Yr) @ W["wo"][1])
    ill = split_ill_conditioned(ref, ref_r)
    assert ill.sum() <= 2, ill.sum()          # the rule singles out a few tokens at most
    got = host(Y)
    check_bf16(got[:, ~ill], ref[:, ~ill], "msr ragged tokens (well-conditioned)")
    if ill.any():
        check_bf16(got[:, ill], ref_r[:, ill], "msr ragged tokens (ill-conditioned)")


def test_small_gamma_takes_the_cuda_core_kernel(R):
    """gamma^64 < 2^-16 (here 0.6) is outside the tensor-core kernel's fp16
    range; the CUDA-core kernel serves it and matches the oracle."""
    (q, k, v), (q64, k64, v64) = inputs(9, 1, 2, 130, 64, 128, "bf16")
    R.lib.retention_kernel_timer_reset()
    o = R.chunkwise_fwd(q, k, v, [0.6, 0.97], chunk=64, norm_flags=R.NORM_ALL)
    torch.cuda.synchronize()
    assert "chunk_simt" in R.kernel_times()
    p = oracle.Problem(1, 2, 130, 64, 128, [0.6, 0.97], norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    check_bf16(host(o), oracle.chunkwise(p, 64, q64, k64, v64)[0], "gamma 0.6")


def test_tc_kernel_is_used(R):
    """The tensor-core kernel (not the CUDA-core fallback) serves bf16,
    chunk 64, d_v % 128 == 0."""
    (q, k, v), _ = inputs(5, 1, 2, 256, 128, 256, "bf16")
    R.lib.retention_kernel_timer_reset()
    R.chunkwise_fwd(q, k, v, [0.9, 0.99], chunk=64)
    torch.cuda.synchronize()
    names = R.kernel_times()
    assert "chunk_tc" in names and "chunk_simt" not in names, names


@pytest.mark.parametrize("scale", [2.0 ** -10, 2.0 ** 10])
def test_tc_chunk_extreme_magnitudes(R, scale):
    """The fp16 operands carry power-of-two block scales: inputs 2^+-10 times
    larger or smaller (exact in bf16) must still match the oracle."""
    B, H, N, dk, dv = 1, 2, 256, 128, 256
    (q, k, v), (q64, k64, v64) = inputs(61, B, H, N, dk, dv, "bf16")
    q, k, v = q * scale, k * scale, v * scale
    gam = [0.9, 0.999]
    o = R.chunkwise_fwd(q, k, v, gam, chunk=64, gn_eps=0.0)
    p = oracle.Problem(B, H, N, dk, dv, gam, gn_eps=0.0)
    ref, _, _ = oracle.chunkwise(p, 64, q64 * scale, k64 * scale, v64 * scale)
    check_bf16(host(o), ref, f"scale {scale}")


@pytest.mark.parametrize("B,H,N,dk,dv", [
    (1, 2, 64 * 40 + 17, 128, 128),  # 7 segments of 6 chunks, one piece each, ragged tail
    (1, 1, 64 * 16, 64, 256),        # 4 segments, two pieces per segment
    (2, 2, 64 * 9 + 1, 256, 512),    # 2 segments, one-chunk pieces, 1-token last chunk
])
@pytest.mark.parametrize("inplace", [False, True])
def test_tc_sequence_segments(R, B, H, N, dk, dv, inplace):
    """Few heads on a long sequence: the chunk kernel runs the sequence as
    several segments whose entry states come from the state kernel's pieces.
    Carried (S, z) in and out, in place or not, all three normalisations."""
    (q, k, v), (q64, k64, v64) = inputs(3000 + N, B, H, N, dk, dv, "bf16")
    gam = [0.9, 0.99][:H]
    S0 = torch.randn(B, H, dk, dv, device="cuda")
    z0 = torch.randn(B, H, dk, device="cuda")
    p = oracle.Problem(B, H, N, dk, dv, gam, pos0=3, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    ref, S_ref, z_ref = oracle.chunkwise(p, 64, q64, k64, v64, S0.double().cpu().numpy(),
                                         z0.double().cpu().numpy())
    if inplace:
        S, z = S0.clone(), z0.clone()
        S_in, z_in, S_out, z_out = S, z, S, z
    else:
        S_in, z_in = S0, z0
        S_out = torch.full_like(S0, float("nan"))
        z_out = torch.full_like(z0, float("nan"))
    R.lib.retention_kernel_timer_reset()
    o = R.chunkwise_fwd(q, k, v, gam, chunk=64, pos0=3, norm_flags=R.NORM_ALL, S_in=S_in,
                        z_in=z_in, S_out=S_out, z_out=z_out)
    torch.cuda.synchronize()
    assert "state_pass" in R.kernel_times()
    check_bf16(host(o), ref, f"segments {B}x{H}x{N}")
    assert np.max(np.abs(host(S_out) - S_ref)) / np.max(np.abs(S_ref)) < 1e-2
    assert np.max(np.abs(host(z_out) - z_ref)) / np.max(np.abs(z_ref)) < 1e-2
    if not inplace:
        assert torch.equal(S_in, S0) and torch.equal(z_in, z0)
