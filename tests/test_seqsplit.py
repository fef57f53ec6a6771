"""Sequence split of one chunkwise call across ranks (seqsplit.py).

CPU: the host logic (segment bounds, the decayed exclusive scan, absolute
positions, the all-gathers) with gloo ranks, world sizes 2 and 3 (one rank
with an empty segment), the three local steps done by the float64 oracle;
the joined outputs and the final state must equal the oracle's single call
over the whole sequence.

GPU: the same steps through the C ABI (retention_chunkwise_state,
retention_state_combine, retention_chunkwise_fwd) for several segments in
one process, against the oracle and against one call over the whole
sequence.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from linear_recurrent_sequence_gb300 import seqsplit, synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The three local steps by the float64 oracle (test infrastructure)."""

    def __init__(self, chunk, gn_eps):
        self.chunk, self.gn_eps = chunk, gn_eps

    def _problem(self, B, H, N, dk, dv, gamma, pos0, flags=0, gn_eps=-1.0):
        return oracle.Problem(B, H, N, dk, dv, list(gamma), pos0=pos0, rotate=True,
                              norm_flags=flags, gn_eps=gn_eps)

    def state(self, k, v, gamma, *, pos0, with_z):
        B, H, N, dk = k.shape
        dv = v.shape[3]
        if N == 0:
            return torch.zeros(B, H, dk, dv, dtype=torch.float64), \
                torch.zeros(B, H, dk, dtype=torch.float64)
        p = self._problem(B, H, N, dk, dv, gamma, pos0)
        _, S, z = oracle.chunkwise(p, self.chunk, np.zeros((B, H, N, dk)), k.numpy(), v.numpy())
        return torch.from_numpy(S), torch.from_numpy(z)

    def combine(self, parts, tokens, gamma, like_S, like_z):
        g = np.asarray(gamma, np.float64)
        S = np.zeros(tuple(like_S.shape))
        z = np.zeros(tuple(like_z.shape)) if like_z is not None else None
        for (Sp, zp), t in zip(parts, tokens):
            w = g ** t
            if Sp is not None:
                S += w[None, :, None, None] * Sp.numpy()
            if z is not None and zp is not None:
                z += w[None, :, None] * zp.numpy()
        return torch.from_numpy(S), (torch.from_numpy(z) if z is not None else None)

    def forward(self, q, k, v, gamma, *, S_in, z_in, pos0, norm_flags=0):
        B, H, N, dk = q.shape
        dv = v.shape[3]
        if N == 0:
            return torch.zeros(B, H, 0, dv, dtype=torch.float64)
        p = self._problem(B, H, N, dk, dv, gamma, pos0, norm_flags, self.gn_eps)
        o, _, _ = oracle.chunkwise(p, self.chunk, q.numpy(), k.numpy(), v.numpy(),
                                   S_in.numpy(), None if z_in is None else z_in.numpy())
        return torch.from_numpy(o)


def _inputs(B, H, N, dk, dv, seed):
    g = np.random.default_rng(seed)
    return [torch.from_numpy(g.standard_normal(s)) for s in
            ((B, H, N, dk), (B, H, N, dk), (B, H, N, dv), (B, H, dk, dv), (B, H, dk))]


def _rank(rank, world, port, counts, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        oracle.build()
        B, H, dk, dv = 1, 2, 4, 6
        q, k, v, S0, z0 = _inputs(B, H, sum(counts), dk, dv, 5)
        a = sum(counts[:rank])
        b = a + counts[rank]
        o, (S, z) = seqsplit.split_chunkwise_fwd(
            q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], [0.9, 0.995], pos0=7, S_in=S0, z_in=z0,
            norm_flags=oracle.NORM_ALL, ops=OracleOps(4, 1e-6), return_state=True)
        out[rank] = (o.numpy(), S.numpy(), z.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("counts", [[9, 14], [6, 0, 11]])
def test_gloo_ranks_join_to_the_single_call(counts):
    world = len(counts)
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, counts, out), nprocs=world, join=True)
        res = dict(out)
    oracle.build()
    B, H, dk, dv = 1, 2, 4, 6
    N = sum(counts)
    q, k, v, S0, z0 = _inputs(B, H, N, dk, dv, 5)
    p = oracle.Problem(B, H, N, dk, dv, [0.9, 0.995], pos0=7, rotate=True,
                       norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    ref, S_ref, z_ref = oracle.chunkwise(p, 4, q.numpy(), k.numpy(), v.numpy(), S0.numpy(),
                                         z0.numpy())
    got = np.concatenate([res[r][0] for r in range(world)], axis=2)
    assert np.max(np.abs(got - ref)) < 1e-11
    for r in range(world):
        assert np.max(np.abs(res[r][1] - S_ref)) < 1e-11 * np.max(np.abs(S_ref))
        assert np.max(np.abs(res[r][2] - z_ref)) < 1e-11 * np.max(np.abs(z_ref))


def test_scan_terms():
    """The decays of the exclusive scan: segment q's state reaches segment
    p after the tokens between them; the initial state after s_p tokens."""
    bounds = seqsplit.segment_bounds([5, 0, 7, 3])
    assert bounds == [(0, 5), (5, 5), (5, 12), (12, 15)]
    assert seqsplit.entry_terms(0, bounds, True) == [(-1, 0)]
    assert seqsplit.entry_terms(3, bounds, False) == [(0, 7), (1, 7), (2, 0)]
    assert seqsplit.final_terms(bounds, True) == [(-1, 15), (0, 10), (1, 10), (2, 3), (3, 0)]


# ------------------------------------------------------------------ GPU
@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from linear_recurrent_sequence_gb300 import retention
    oracle.build()
    return retention


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,B,H,N,dk,dv", [
    ("bf16", 1, 3, 64 * 37 + 5, 128, 256),  # tensor-core state pass, ragged last chunk
    ("f32", 2, 2, 150, 32, 48),             # CUDA-core state pass
])
def test_state_pass_matches_oracle(R, dtype, B, H, N, dk, dv):
    from tests.helpers import host, seeded
    q, q64 = seeded(808, "q", (B, H, N, dk), dtype)
    k, k64 = seeded(808, "k", (B, H, N, dk), dtype)
    v, v64 = seeded(808, "v", (B, H, N, dv), dtype)
    gam = [0.9, 0.99, 1.0][:H]
    S0, S064 = seeded(808, "S", (B, H, dk, dv), "f32")
    z0, z064 = seeded(808, "z", (B, H, dk), "f32")
    p = oracle.Problem(B, H, N, dk, dv, gam, pos0=9, gn_eps=1e-6)
    _, S_ref, z_ref = oracle.chunkwise(p, 64, q64, k64, v64, S064, z064)
    R.lib.retention_kernel_timer_reset()
    S, z = R.chunkwise_state(k, v, gam, pos0=9, S_in=S0, z_in=z0)
    torch.cuda.synchronize()
    names = R.kernel_times()
    assert ("state_pass" in names) == (dtype == "bf16"), names
    rel = 1e-2 if dtype == "bf16" else 1e-5
    assert np.max(np.abs(host(S) - S_ref)) / np.max(np.abs(S_ref)) < rel
    assert np.max(np.abs(host(z) - z_ref)) / np.max(np.abs(z_ref)) < rel
    # in place, and without z
    S1 = S0.clone()
    R.chunkwise_state(k, v, gam, pos0=9, S_in=S1, S_out=S1, with_z=False)
    assert np.max(np.abs(host(S1) - S_ref)) / np.max(np.abs(S_ref)) < rel


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,dk,dv,cuts", [("bf16", 128, 256, [0, 700, 1500, 2213]),
                                              ("f32", 32, 48, [0, 40, 40, 130])])
def test_segments_through_the_abi(R, dtype, dk, dv, cuts):
    """Emulates the ranks one after another in one process: each segment's
    state from zero, the decayed scan by retention_state_combine, each
    segment's forward from its entry state; joined, they equal the oracle
    and one call over the whole sequence."""
    from tests.helpers import check_bf16, check_f32, host, seeded
    B, H, N = 1, 2, cuts[-1]
    q, q64 = seeded(909, "q", (B, H, N, dk), dtype)
    k, k64 = seeded(909, "k", (B, H, N, dk), dtype)
    v, v64 = seeded(909, "v", (B, H, N, dv), dtype)
    gam = synth.head_gammas(H)
    S0 = torch.randn(B, H, dk, dv, device="cuda")
    z0 = torch.randn(B, H, dk, device="cuda")
    flags = R.NORM_ALL
    counts = [cuts[i + 1] - cuts[i] for i in range(len(cuts) - 1)]
    bounds = seqsplit.segment_bounds(counts)
    dS = [R.chunkwise_state(k[:, :, a:b], v[:, :, a:b], gam, pos0=3 + a) for a, b in bounds]
    outs = []
    for r, (a, b) in enumerate(bounds):
        terms = seqsplit.entry_terms(r, bounds, True)
        parts = [(S0, z0) if s < 0 else dS[s] for s, _ in terms]
        S_e, z_e = R.state_combine(parts, [t for _, t in terms], gam,
                                   S_out=torch.empty_like(S0), z_out=torch.empty_like(z0))
        outs.append(R.chunkwise_fwd(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], gam, pos0=3 + a,
                                    norm_flags=flags, S_in=S_e, z_in=z_e,
                                    out_dtype=torch.float32))
    got = host(torch.cat(outs, dim=2))
    p = oracle.Problem(B, H, N, dk, dv, gam, pos0=3, norm_flags=oracle.NORM_ALL, gn_eps=1e-6)
    ref, S_ref, _ = oracle.chunkwise(p, 64, q64, k64, v64, host(S0), host(z0))
    whole = host(R.chunkwise_fwd(q, k, v, gam, pos0=3, norm_flags=flags, S_in=S0, z_in=z0,
                                 out_dtype=torch.float32))
    if dtype == "bf16":
        check_bf16(got, ref, "segments vs oracle")
        check_bf16(got, whole, "segments vs one call")
    else:
        check_f32(got, ref, "segments vs oracle")
        check_f32(got, whole, "segments vs one call")
    terms = seqsplit.final_terms(bounds, True)
    parts = [(S0, z0) if s < 0 else dS[s] for s, _ in terms]
    S_f, _ = R.state_combine(parts, [t for _, t in terms], gam, S_out=torch.empty_like(S0))
    assert np.max(np.abs(host(S_f) - S_ref)) / np.max(np.abs(S_ref)) < 1e-2


@pytest.mark.gpu
def test_state_pass_magnitude_jumps(R):
    """The state kernel keeps its accumulator in units set by the data: a
    run of all-zero values, then values 2^-20 smaller, then 2^20 larger (the
    last jump needs more than the MMA's own 2^-15 accumulator scale, so the
    kernel rescales on the CUDA cores) must still give the oracle's state."""
    from tests.helpers import host, seeded
    B, H, N, dk, dv = 1, 2, 64 * 40, 128, 128
    q, q64 = seeded(717, "q", (B, H, N, dk), "bf16")
    k, k64 = seeded(717, "k", (B, H, N, dk), "bf16")
    v, v64 = seeded(717, "v", (B, H, N, dv), "bf16")
    scale = np.ones(N)
    scale[:640] = 0.0
    scale[640:1280] = 2.0 ** -20
    scale[1280:] = 2.0 ** 20
    v = v * torch.from_numpy(scale).float().cuda()[None, None, :, None].bfloat16()
    v64 = v64 * scale[None, None, :, None]
    gam = [0.96875, 0.999]
    p = oracle.Problem(B, H, N, dk, dv, gam, gn_eps=1e-6)
    _, S_ref, z_ref = oracle.chunkwise(p, 64, q64, k64, v64)
    R.lib.retention_kernel_timer_reset()
    S, z = R.chunkwise_state(k, v, gam)
    torch.cuda.synchronize()
    assert "state_pass" in R.kernel_times()
    got = host(S)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - S_ref)) / np.max(np.abs(S_ref)) < 1e-2
