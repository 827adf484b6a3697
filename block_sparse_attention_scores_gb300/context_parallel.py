"""Head-wise context parallelism for one MSA layer over torch.distributed ranks.

dothoosh.com "how Flash-MSA cuts million-token training cost", "Current
limits and future scaling": very long sequences are spread over devices by a
head-wise all-gather (or a ring). Here each rank holds a contiguous shard of
T / W tokens of every tensor (the sequence-parallel layout of the layers
around attention). For the MSA layer the ranks exchange that layout for a
group-parallel one:

1. all-to-all: Q, dO (query heads), K, V (KV heads), q_idx (index queries)
   go from "T / W tokens, all groups" to "all T tokens, G / W groups"; the
   shared index key k_idx is all-gathered (every group scores against it);
2. each rank runs the whole MSA hot path on its group slice (index top-k,
   block map, sparse forward, fused backward) with no further exchange: the
   selection, the attention, KV heads and the KL are per group;
3. dk_idx, the only term summed over groups, is reduce-scattered over T;
4. all-to-all back: O, LSE, dQ, dK, dV, dq_idx, KL and block_idx return to
   the sequence-sharded layout.

Requirements: G % W == 0 and T % W == 0 (each shard a whole number of
tokens; the per-rank T stays the full T, so the kernels' own T % 128 rule
applies unchanged). ``compute`` is the per-rank hot path: ``cuda_compute``
(the library's entry points on the rank's current GPU) in production,
``cuda_compute_dense`` for the indexer warmup's full attention (itinai.ru
"How to solve the memory problem with MiniMax Sparse Attention", "Training
sparse attention"; no selection, so no block_idx); any function of the same
signature for checking the exchange on CPU ranks.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist

# (T axis, head/group axis) of every per-token tensor of the layer
AXES = {
    "Q": (1, 2), "dO": (1, 2), "O": (1, 2), "dQ": (1, 2), "LSE": (1, 2),
    "K": (1, 2), "V": (1, 2), "dK": (1, 2), "dV": (1, 2),
    "q_idx": (1, 2), "dq_idx": (1, 2),
    "block_idx": (2, 1), "KL": (2, 1),
}
INPUTS = ("Q", "K", "V", "dO", "q_idx", "k_idx")
OUTPUTS = ("block_idx", "O", "LSE", "dQ", "dK", "dV", "dq_idx", "dk_idx", "KL")


@dataclass(frozen=True)
class LayerShape:
    """Shape of the whole layer (all ranks): the C ABI's msa_shape fields."""

    B: int
    T: int
    Hq: int
    G: int
    d: int = 128
    d_idx: int = 64
    Bk: int = 128
    k: int = 16


def group_range(G: int, world: int, rank: int) -> tuple[int, int]:
    """The GQA groups [g0, g1) that rank `rank` owns (contiguous, G / world each)."""
    if G % world:
        raise ValueError(f"G={G} groups do not split over {world} ranks")
    n = G // world
    return rank * n, (rank + 1) * n


def local_shape(s: LayerShape, world: int) -> LayerShape:
    """Per-rank problem: all T tokens, G / world groups and their query heads."""
    if s.G % world or s.T % world:
        raise ValueError(f"G={s.G} and T={s.T} must be multiples of world={world}")
    return LayerShape(s.B, s.T, s.Hq // world, s.G // world, s.d, s.d_idx, s.Bk, s.k)


def _bytes(x: torch.Tensor) -> torch.Tensor:
    """The tensor's storage as uint8 (last dim times the item size)."""
    return x.contiguous().view(torch.uint8)


def seq_to_heads(x: torch.Tensor, t_axis: int, h_axis: int, world: int, group=None) -> torch.Tensor:
    """All-to-all from [.., T/W (t_axis), H (h_axis), ..] to [.., T, H/W, ..]."""
    xm = x.movedim((t_axis, h_axis), (1, 2))
    B, Tl, H = xm.shape[:3]
    rest = tuple(xm.shape[3:])
    send = xm.reshape(B, Tl, world, H // world, *rest).movedim(2, 0).contiguous()  # [W, B, Tl, H/W, ..]
    recv = torch.empty_like(send)
    dist.all_to_all_single(_bytes(recv), _bytes(send), group=group)  # recv[s] = rank s's tokens of my heads
    out = recv.movedim(0, 1).reshape(B, world * Tl, H // world, *rest)
    return out.movedim((1, 2), (t_axis, h_axis)).contiguous()


def heads_to_seq(y: torch.Tensor, t_axis: int, h_axis: int, world: int, group=None) -> torch.Tensor:
    """All-to-all from [.., T (t_axis), H/W (h_axis), ..] back to [.., T/W, H, ..]."""
    ym = y.movedim((t_axis, h_axis), (1, 2))
    B, T, Hl = ym.shape[:3]
    rest = tuple(ym.shape[3:])
    send = ym.reshape(B, world, T // world, Hl, *rest).movedim(1, 0).contiguous()  # send[s] = my heads of shard s
    recv = torch.empty_like(send)
    dist.all_to_all_single(_bytes(recv), _bytes(send), group=group)  # recv[r] = rank r's heads of my shard
    out = recv.movedim(0, 2).reshape(B, T // world, world * Hl, *rest)
    return out.movedim((1, 2), (t_axis, h_axis)).contiguous()


def gather_seq(x: torch.Tensor, world: int, group=None) -> torch.Tensor:
    """All-gather of a [B, T/W, ..] tensor into [B, T, ..] (rank order = token order)."""
    xb = _bytes(x)
    parts = [torch.empty_like(xb) for _ in range(world)]
    dist.all_gather(parts, xb, group=group)
    return torch.cat([p.view(x.dtype) for p in parts], dim=1)


def reduce_scatter_seq(x: torch.Tensor, world: int, group=None) -> torch.Tensor:
    """Sum over ranks of a [B, T, ..] tensor, each rank keeping its [B, T/W, ..] shard."""
    B, T = x.shape[:2]
    send = x.reshape(B, world, T // world, *x.shape[2:]).movedim(1, 0).contiguous()  # [W, B, T/W, ..]
    out = torch.empty_like(send[0])
    dist.reduce_scatter_tensor(out, send.reshape(world * B, *send.shape[2:]), group=group)
    return out


def cp_step(s: LayerShape, shards: dict, compute, kl_weight: float = 1.0, group=None) -> dict:
    """One MSA layer step (index top-k, sparse forward, fused backward) on
    sequence-sharded tensors.

    shards: this rank's T / W tokens of Q, K, V, dO [B, T/W, heads, d],
    q_idx [B, T/W, G, d_idx] and k_idx [B, T/W, d_idx]. compute(local_shape,
    tensors, kl_weight) runs the hot path on one group slice and returns the
    outputs in the C ABI's layouts (dk_idx summed over that slice's groups).
    Returns this rank's T / W tokens of every output.
    """
    world = dist.get_world_size(group)
    loc = local_shape(s, world)
    t = {n: seq_to_heads(shards[n], *AXES[n], world, group) for n in ("Q", "K", "V", "dO", "q_idx")}
    t["k_idx"] = gather_seq(shards["k_idx"], world, group)
    out = compute(loc, t, kl_weight)
    # the outputs the compute gives (full attention has no block_idx)
    res = {n: heads_to_seq(out[n], *AXES[n], world, group) for n in OUTPUTS if n != "dk_idx" and n in out}
    res["dk_idx"] = reduce_scatter_seq(out["dk_idx"], world, group)
    return res


def cuda_compute(s: LayerShape, t: dict, kl_weight: float = 1.0) -> dict:
    """The hot path on the current GPU through the library's entry points:
    msa_index_topk -> msa_block_map -> msa_sparse_fwd_mapped -> msa_bwd_mapped."""
    import block_sparse_attention_scores_gb300 as msa

    shape = msa.Shape(B=s.B, T=s.T, Hq=s.Hq, G=s.G, d=s.d, d_idx=s.d_idx, Bk=s.Bk, k=s.k)
    dev = t["Q"].device
    ws = msa.alloc_workspace(shape, msa.MSA_WS_BWD, dev)
    st = torch.cuda.current_stream(dev)
    bi = torch.empty((s.B, s.G, s.T, s.k), dtype=torch.int32, device=dev)
    O = torch.empty_like(t["Q"])
    LSE = torch.empty((s.B, s.T, s.Hq), dtype=torch.float32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(dQ=torch.empty(t["Q"].shape, **f32), dK=torch.empty(t["K"].shape, **f32),
             dV=torch.empty(t["V"].shape, **f32), dq_idx=torch.empty(t["q_idx"].shape, **f32),
             dk_idx=torch.empty(t["k_idx"].shape, **f32), KL=torch.empty((s.B, s.G, s.T), **f32))
    msa.msa_index_topk(shape, t["q_idx"], t["k_idx"], bi, ws, st)
    msa.msa_block_map(shape, bi, ws, st)
    msa.msa_sparse_fwd_mapped(shape, t["Q"], t["K"], t["V"], bi, O, LSE, ws, st)
    msa.msa_bwd_mapped(shape, t["Q"], t["K"], t["V"], O, t["dO"], LSE, t["q_idx"], t["k_idx"], bi, kl_weight,
                       g["dQ"], g["dK"], g["dV"], g["dq_idx"], g["dk_idx"], g["KL"], ws, st)
    msa.msa_check_device_status(ws, st)
    return dict(block_idx=bi, O=O, LSE=LSE, **g)


def cuda_compute_dense(s: LayerShape, t: dict, kl_weight: float = 1.0) -> dict:
    """Full attention (the indexer warmup) on the current GPU: msa_dense_fwd ->
    msa_dense_bwd over every visible token of the rank's groups (4 or 8 heads
    per group). The outputs are those of cuda_compute without block_idx."""
    import block_sparse_attention_scores_gb300 as msa

    shape = msa.Shape(B=s.B, T=s.T, Hq=s.Hq, G=s.G, d=s.d, d_idx=s.d_idx, Bk=s.Bk, k=1)
    dev = t["Q"].device
    ws = msa.alloc_workspace(shape, msa.MSA_WS_DENSE, dev)
    st = torch.cuda.current_stream(dev)
    O = torch.empty_like(t["Q"])
    LSE = torch.empty((s.B, s.T, s.Hq), dtype=torch.float32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(dQ=torch.empty(t["Q"].shape, **f32), dK=torch.empty(t["K"].shape, **f32),
             dV=torch.empty(t["V"].shape, **f32), dq_idx=torch.empty(t["q_idx"].shape, **f32),
             dk_idx=torch.empty(t["k_idx"].shape, **f32), KL=torch.empty((s.B, s.G, s.T), **f32))
    msa.msa_dense_fwd(shape, t["Q"], t["K"], t["V"], O, LSE, ws, st)
    msa.msa_dense_bwd(shape, t["Q"], t["K"], t["V"], O, t["dO"], LSE, t["q_idx"], t["k_idx"], kl_weight,
                      g["dQ"], g["dK"], g["dV"], g["dq_idx"], g["dk_idx"], g["KL"], ws, st)
    msa.msa_check_device_status(ws, st)
    return dict(O=O, LSE=LSE, **g)
