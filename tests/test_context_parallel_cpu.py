"""Head-wise context parallelism over two gloo ranks on the CPU.

dothoosh.com "how Flash-MSA cuts million-token training cost", "Current
limits and future scaling" (head-wise all-gather context parallelism). Each
rank holds half of the tokens of every input; the exchange moves them to a
per-group-slice layout, each rank runs its slice through the fp64 oracle
(standing in for the GPU hot path, which has the same per-group contract),
dk_idx is reduce-scattered and the outputs return to the token-sharded
layout. Reassembled, every output must equal the single-rank oracle on the
whole layer: bit for bit where a group's arithmetic is untouched by the
split, and to fp64 rounding for dk_idx, whose sum over groups is regrouped.
The same holds for the indexer warmup's full attention (the oracle with no
block list, every visible token), which returns no block_idx.
"""
import os
import socket

import numpy as np
import pytest

import synth

W = synth.T1024.with_(T=512, Hq=8, G=4, k=3, name="cp_b1_t512_hq8_g4_k3")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_compute(loc, t, kl_weight):
    """The hot path on one group slice, by the fp64 oracle (bf16 bit patterns in)."""
    import torch

    import oracle

    a = {n: t[n].numpy().view(np.uint16) for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")}
    s = oracle.shape(loc.B, loc.T, loc.Hq, loc.G, loc.d, loc.d_idx, loc.Bk, loc.k, kl_weight=kl_weight)
    bi, _, _ = oracle.full_topk(s, a["q_idx"], a["k_idx"])
    O, LSE = oracle.full_fwd(s, a["Q"], a["K"], a["V"], bi)
    g = oracle.full_bwd(s, a["Q"], a["K"], a["V"], a["dO"], a["q_idx"], a["k_idx"], bi)
    out = {n: torch.from_numpy(np.ascontiguousarray(v)) for n, v in g.items()}
    out.update(block_idx=torch.from_numpy(np.ascontiguousarray(bi)), O=torch.from_numpy(O), LSE=torch.from_numpy(LSE))
    return out


def _oracle_compute_dense(loc, t, kl_weight):
    """Full attention on one group slice by the fp64 oracle (no block list)."""
    import torch

    import oracle

    a = {n: t[n].numpy().view(np.uint16) for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")}
    s = oracle.shape(loc.B, loc.T, loc.Hq, loc.G, loc.d, loc.d_idx, loc.Bk, loc.k, kl_weight=kl_weight)
    O, LSE = oracle.full_fwd(s, a["Q"], a["K"], a["V"], None)
    g = oracle.full_bwd(s, a["Q"], a["K"], a["V"], a["dO"], a["q_idx"], a["k_idx"], None)
    out = {n: torch.from_numpy(np.ascontiguousarray(v)) for n, v in g.items()}
    out.update(O=torch.from_numpy(O), LSE=torch.from_numpy(LSE))
    return out


def _rank(rank, world, port, q, mode):
    import torch
    import torch.distributed as dist

    from block_sparse_attention_scores_gb300 import context_parallel as cp

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = synth.make_inputs(W)
        tl = W.T // world
        shards = {n: torch.from_numpy(np.ascontiguousarray(inp[n][:, rank * tl:(rank + 1) * tl]).view(np.int16))
                  for n in cp.INPUTS}
        # the exchange helpers are inverses of each other
        x = torch.arange(W.B * tl * W.Hq * 3, dtype=torch.float64).reshape(W.B, tl, W.Hq, 3) + 1e6 * rank
        back = cp.heads_to_seq(cp.seq_to_heads(x, 1, 2, world), 1, 2, world)
        assert torch.equal(back, x)
        s = cp.LayerShape(B=W.B, T=W.T, Hq=W.Hq, G=W.G, d=W.d, d_idx=W.d_idx, Bk=W.Bk, k=W.k)
        compute = _oracle_compute if mode == "sparse" else _oracle_compute_dense
        res = cp.cp_step(s, shards, compute, kl_weight=0.5)
        q.put((rank, {n: v.numpy() for n, v in res.items()}))
    except Exception as e:  # reported to the parent, which fails the test at once
        q.put((rank, f"{type(e).__name__}: {e}"))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["sparse", "dense"])
def test_context_parallel_two_ranks_equal_single_rank(mode):
    import torch.multiprocessing as mp

    import oracle
    from block_sparse_attention_scores_gb300 import context_parallel as cp

    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q, mode)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=300) for _ in range(world))
    for r in range(world):
        assert not isinstance(got[r], str), f"rank {r}: {got[r]}"
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # reassemble the token shards
    names = [n for n in cp.OUTPUTS if mode == "sparse" or n != "block_idx"]
    assert sorted(got[0]) == sorted(names)
    full = {}
    for n in names:
        t_axis = 1 if n in ("dk_idx",) else cp.AXES[n][0]
        full[n] = np.concatenate([got[r][n] for r in range(world)], axis=t_axis)

    inp = synth.make_inputs(W)
    s = oracle.shape_of(W, kl_weight=0.5)
    bi = oracle.full_topk(s, inp["q_idx"], inp["k_idx"])[0] if mode == "sparse" else None
    O, LSE = oracle.full_fwd(s, inp["Q"], inp["K"], inp["V"], bi)
    ref = oracle.full_bwd(s, *[inp[n] for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")], bi)
    ref.update(block_idx=bi, O=O, LSE=LSE)
    for n in names:
        assert full[n].shape == np.asarray(ref[n]).shape, n
        if n == "dk_idx":
            np.testing.assert_allclose(full[n], ref[n], rtol=1e-12, atol=1e-14)
        else:
            np.testing.assert_array_equal(full[n], ref[n], err_msg=n)
    assert np.abs(ref["dk_idx"]).max() > 1e-3  # the reduced term is not trivially zero


def test_group_split_rules():
    from block_sparse_attention_scores_gb300 import context_parallel as cp

    assert cp.group_range(8, 4, 3) == (6, 8)
    s = cp.LayerShape(B=1, T=1024, Hq=32, G=8)
    assert cp.local_shape(s, 2) == cp.LayerShape(B=1, T=1024, Hq=16, G=4)
    with pytest.raises(ValueError):
        cp.group_range(6, 4, 0)
    with pytest.raises(ValueError):
        cp.local_shape(cp.LayerShape(B=1, T=1000, Hq=8, G=4), 3)
