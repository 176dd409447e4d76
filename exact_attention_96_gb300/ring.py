"""Ring attention over sequence shards, forward and backward, emulated on one GPU ("Flash
Attention 原理与实践" §5.2: the key/value sequence is split across workers, shards pass around
a ring, each worker runs FlashAttention of its own queries against the shard it currently
holds, and the partial results are merged with log-sum-exp).

On a ring of `world` workers, at hop t worker r holds the key/value shard that started on
worker (r - t) mod world.  With a causal mask worker r needs only shards s <= r, the shard
s == r with the causal mask of the diagonal block.  Here every worker runs in turn on the same
GPU, so "passing a shard" is indexing; each hop calls fa_fwd_partial and each worker's hops are
merged by fa_merge_partials.  The backward pass runs one fa_bwd_accumulate per (worker, shard)
pair into fp32 per-shard accumulators and rounds the sums once (fa_convert_f32_to_bf16).
"""

from __future__ import annotations

import math

import torch

from . import abi


def ring_hops(rank: int, world: int, causal: bool):
    """The shards worker `rank` processes, in ring order: [(hop, shard, diagonal)]."""
    out = []
    for t in range(world):
        s = (rank - t) % world
        if causal and s > rank:
            continue
        out.append((t, s, s == rank))
    return out


def ring_attention_forward(q, k, v, world: int, causal: bool = False, scale: float | None = None):
    """O, LSE of attention over [B, H, N, d] inputs, computed as `world` ring workers would,
    each owning N / world consecutive positions.  N must be a multiple of `world`."""
    B, H, N, d = q.shape
    if N % world:
        raise ValueError("sequence length must be a multiple of the ring size")
    ns = N // world
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    shard = lambda t, i: t[:, :, i * ns:(i + 1) * ns].contiguous()  # noqa: E731
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rows = B * H * ns
    for r in range(world):
        q_r = shard(q, r)
        hops = ring_hops(r, world, causal)
        o_parts = torch.empty((len(hops), rows, d), dtype=torch.float32, device=q.device)
        lse_parts = torch.empty((len(hops), rows), dtype=torch.float32, device=q.device)
        for slot, (_, s, diag) in enumerate(hops):
            k_s, v_s = shard(k, s), shard(v, s)
            abi.check("fa_fwd_partial", abi.fa_fwd_partial(
                q_r.data_ptr(), k_s.data_ptr(), v_s.data_ptr(), o_parts[slot].data_ptr(),
                lse_parts[slot].data_ptr(), B, H, ns, ns, d, scale, causal and diag, stream))
        o_r = torch.empty_like(q_r)
        lse_r = torch.empty((B, H, ns), dtype=torch.float32, device=q.device)
        abi.check("fa_merge_partials", abi.fa_merge_partials(
            o_parts.data_ptr(), lse_parts.data_ptr(), len(hops), rows, d, o_r.data_ptr(),
            lse_r.data_ptr(), stream))
        o[:, :, r * ns:(r + 1) * ns] = o_r
        lse[:, :, r * ns:(r + 1) * ns] = lse_r
    return o, lse


def ring_attention_backward(q, k, v, o, do, lse, world: int, causal: bool = False,
                            scale: float | None = None):
    """dQ, dK, dV of ring attention.  With the global LSE (from the forward) every
    probability is fixed, so the contribution of query shard r and key/value shard s is
    exactly the backward pass of that block pair (O_r, dO_r and LSE_r of the whole problem;
    the diagonal pair causal, later shards skipped).  Worker r accumulates dQ_r over the shards
    it sees; dK_s, dV_s collect the contributions of every worker that saw shard s (on a real
    ring they travel back with the shard).  fa_bwd_accumulate adds each block pair's
    contribution in fp32 into per-shard accumulators, and fa_convert_f32_to_bf16 rounds each
    sum once at the end."""
    from . import attention as fa  # local import: attention imports nothing from here

    B, H, N, d = q.shape
    if N % world:
        raise ValueError("sequence length must be a multiple of the ring size")
    ns = N // world
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    shard = lambda t, i: t[:, :, i * ns:(i + 1) * ns].contiguous()  # noqa: E731
    # fp32 accumulators, shard-major: acc[g, s] is gradient g (dQ, dK, dV) of shard s
    acc = torch.zeros((3, world, B, H, ns, d), dtype=torch.float32, device=q.device)
    ws = torch.empty(fa.workspace_bytes(B, H, ns, d), dtype=torch.uint8, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    k_sh = [shard(k, s) for s in range(world)]
    v_sh = [shard(v, s) for s in range(world)]
    for r in range(world):
        q_r, o_r, do_r, lse_r = shard(q, r), shard(o, r), shard(do, r), shard(lse, r)
        for _, s, diag in ring_hops(r, world, causal):
            abi.check("fa_bwd_accumulate", abi.fa_bwd_accumulate(
                q_r.data_ptr(), k_sh[s].data_ptr(), v_sh[s].data_ptr(), o_r.data_ptr(), do_r.data_ptr(),
                lse_r.data_ptr(), acc[0, r].data_ptr(), acc[1, s].data_ptr(), acc[2, s].data_ptr(),
                B, H, ns, d, scale, causal and diag, ws.data_ptr(), ws.numel(), stream))
    out = torch.empty(acc.shape, dtype=q.dtype, device=q.device)
    abi.check("fa_convert_f32_to_bf16", abi.fa_convert_f32_to_bf16(acc.data_ptr(), out.data_ptr(),
                                                                   acc.numel(), stream))
    # shard-major [world, B, H, ns, d] -> [B, H, N, d] (a copy, no arithmetic)
    dq, dk, dv = (out[g].permute(1, 2, 0, 3, 4).reshape(B, H, N, d) for g in range(3))
    return dq, dk, dv
