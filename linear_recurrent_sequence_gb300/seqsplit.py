"""One chunkwise retention call with its sequence split across ranks.

Each rank (one process per GPU) holds one contiguous segment of the
sequence, the ranks' segments in rank order, every (batch, head) on every
rank.  The chunkwise form carries the recurrent state from chunk to chunk
(hwhale.com/article/285883, chunkwise form: parallel within chunks,
recurrent across them); split across ranks, that carry becomes one exchange:

  1. every rank computes the state its segment produces from a zero state,
     dS_p (and dz_p), without outputs (retention_chunkwise_state);
  2. the ranks all-gather those states and their segment lengths n_p;
  3. rank p joins them into the state that enters its segment, a decayed
     exclusive scan (the recurrence is linear):
        S_in,p = gamma^(s_p) S_in + sum_{q<p} gamma^(s_p - e_q) dS_q,
     s_p / e_q the first / one-past-last token of a segment counted from the
     start of the sequence (retention_state_combine);
  4. every rank runs the ordinary chunkwise forward on its segment from
     S_in,p, z_in,p at its absolute position, so the third normalisation's
     row sums and GroupNorm see exactly the single-device values.

The exchange is one all-gather of B*H*d_k*(d_v+1) floats per rank.  Step 1
re-reads the segment's keys and values once, which keeps step 4 free of any
fix-up of outputs.  The arithmetic of every step runs in the library's CUDA
kernels; this module only orders the calls and the exchange.  `ops` lets a
test drive the same host logic with other implementations of the three
local steps.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


class CudaOps:
    """The three local steps through the library's C ABI."""

    def __init__(self):
        from . import retention
        self.R = retention

    def state(self, k, v, gamma, *, pos0, with_z):
        return self.R.chunkwise_state(k, v, gamma, pos0=pos0, with_z=with_z)

    def combine(self, parts, tokens, gamma, like_S, like_z):
        S = torch.empty_like(like_S)
        z = torch.empty_like(like_z) if like_z is not None else None
        return self.R.state_combine(parts, tokens, gamma, S_out=S, z_out=z)

    def forward(self, q, k, v, gamma, *, S_in, z_in, pos0, **kw):
        return self.R.chunkwise_fwd(q, k, v, gamma, S_in=S_in, z_in=z_in, pos0=pos0, **kw)


def segment_bounds(counts):
    """(start, end) token offsets of each rank's segment."""
    bounds, s = [], 0
    for n in counts:
        bounds.append((s, s + n))
        s += n
    return bounds


def entry_terms(rank, bounds, has_init):
    """The parts of the state entering `rank`'s segment, as (source, decay
    tokens): source -1 is the caller's initial state, q >= 0 rank q's
    segment state."""
    start = bounds[rank][0]
    terms = [(-1, start)] if has_init else []
    terms += [(q, start - bounds[q][1]) for q in range(rank)]
    return terms


def final_terms(bounds, has_init):
    """The parts of the state after the whole sequence."""
    total = bounds[-1][1] if bounds else 0
    terms = [(-1, total)] if has_init else []
    terms += [(q, total - bounds[q][1]) for q in range(len(bounds))]
    return terms


def split_chunkwise_fwd(q, k, v, gamma, *, pos0=0, S_in=None, z_in=None, norm_flags=0,
                        group=None, ops=None, return_state=False, **kw):
    """Chunkwise retention over a sequence split across the ranks of `group`.

    q, k [B,H,n_p,d_k] and v [B,H,n_p,d_v] are this rank's segment (n_p may
    differ between ranks, and may be 0); pos0 is the absolute position of the
    sequence's first token; S_in, z_in the state entering the sequence
    (None: zero), the same on every rank.  Returns this rank's outputs, and
    with return_state also the (S, z) after the whole sequence (every rank
    gets it)."""
    ops = ops or CudaOps()
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    B, H, n, dk = q.shape
    dv = v.shape[3]
    need_z = bool(norm_flags & 4) or z_in is not None or return_state
    # segment lengths (on the host: they only set decays and positions)
    mine = torch.tensor([n], dtype=torch.int64)
    counts = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(counts, mine, group=group)
    bounds = segment_bounds([int(c.item()) for c in counts])
    start = bounds[rank][0]
    # 1. this segment's own state, from zero
    dS, dz = ops.state(k, v, gamma, pos0=pos0 + start, with_z=need_z)
    # 2. every segment's state on every rank
    S_all = [torch.empty_like(dS) for _ in range(world)]
    dist.all_gather(S_all, dS.contiguous(), group=group)
    z_all = None
    if need_z:
        z_all = [torch.empty_like(dz) for _ in range(world)]
        dist.all_gather(z_all, dz.contiguous(), group=group)

    def gather(terms):
        parts, tokens = [], []
        for src, t in terms:
            if src < 0:
                parts.append((S_in, z_in if need_z else None))
            else:
                parts.append((S_all[src], z_all[src] if need_z else None))
            tokens.append(t)
        return parts, tokens

    # 3. the state entering this segment
    has_init = S_in is not None or z_in is not None
    parts, tokens = gather(entry_terms(rank, bounds, has_init))
    S_e, z_e = ops.combine(parts, tokens, gamma, dS, dz if need_z else None)
    # 4. this segment's outputs from its entry state
    o = ops.forward(q, k, v, gamma, S_in=S_e, z_in=z_e, pos0=pos0 + start,
                    norm_flags=norm_flags, **kw)
    if not return_state:
        return o
    parts, tokens = gather(final_terms(bounds, has_init))
    S_f, z_f = ops.combine(parts, tokens, gamma, dS, dz if need_z else None)
    return o, (S_f, z_f)
