"""Parity of msa_index_topk (CUDA) with the fp64 oracle: bit-exact block ids
except at near-ties (oracle k-th/(k+1)-th pooled-score gap < 1e-4)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import compare_block_idx, to_dev, valid_selection

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__

    __graft_entry__.build_library()
    import block_sparse_attention_scores_gb300 as m

    return m


def _run(msa, w):
    import torch

    inp = synth.make_inputs(w, ("q_idx", "k_idx"))
    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    ws = msa.alloc_workspace(s, msa.MSA_WS_TOPK)
    bi = msa.index_topk(s, to_dev(inp["q_idx"]), to_dev(inp["k_idx"]), workspace=ws)
    msa.msa_check_device_status(ws)
    torch.cuda.synchronize()
    return inp, bi.cpu().numpy()


@pytest.mark.parametrize("cfg", [
    synth.T1024,                                           # T=1024, G=2, k=4 (fewer blocks than k early on)
    synth.T1024.with_(T=128, name="single_block"),         # only the own block exists
    synth.T1024.with_(T=384, k=1, name="k1"),              # own block only
    synth.T1024.with_(T=640, k=8, name="k_gt_blocks"),     # k > number of blocks: all visible kept
    synth.T1024.with_(B=2, T=768, G=3, Hq=3, k=5, name="b2_g3_hg1"),
    synth.T1024.with_(T=2048, G=1, Hq=8, k=20, name="k20"),
    synth.T1024.with_(T=1536, G=2, Hq=16, k=33, name="k33"),
])
def test_index_topk_matches_oracle_full(msa, cfg):
    inp, got = _run(msa, cfg)
    valid_selection(got, cfg.T, cfg.Bk)
    want, gap, _ = oracle.full_topk(oracle.shape_of(cfg), inp["q_idx"], inp["k_idx"])
    n, ties, bad, bad_tie = compare_block_idx(got, want, gap)
    print(f"{cfg.name}: rows={n} near_ties={ties} mismatches(outside ties)={bad} mismatches(in ties)={bad_tie}")
    assert bad == 0


def test_index_topk_t8192_full(msa):
    w = synth.T8192
    inp, got = _run(msa, w)
    valid_selection(got, w.T, w.Bk)
    want, gap, _ = oracle.full_topk(oracle.shape_of(w), inp["q_idx"], inp["k_idx"])
    n, ties, bad, bad_tie = compare_block_idx(got, want, gap)
    print(f"{w.name}: rows={n} near_ties={ties} mismatches(outside ties)={bad} mismatches(in ties)={bad_tie}")
    assert bad == 0


@pytest.mark.parametrize("cfg", [
    synth.T1024.with_(T=4096, G=2, Hq=2, k=5, name="ties_k5"),
    synth.T1024.with_(T=4096, G=2, Hq=16, k=16, name="ties_k16"),
    synth.T1024.with_(T=8192, G=1, Hq=8, k=33, name="ties_k33"),
    synth.T1024.with_(T=12288, G=1, Hq=8, k=64, name="ties_k64"),
], ids=["k5", "k16", "k33", "k64"])
def test_index_topk_exact_ties(msa, cfg):
    """Pooled scores that tie exactly (tied_index_inputs): every row must match the
    oracle bit for bit, ties included: equal scores go to the lower block id."""
    import torch

    q_idx, k_idx = synth.tied_index_inputs(cfg)
    s = msa.Shape(B=cfg.B, T=cfg.T, Hq=cfg.Hq, G=cfg.G, k=cfg.k)
    ws = msa.alloc_workspace(s, msa.MSA_WS_TOPK)
    got = msa.index_topk(s, to_dev(q_idx), to_dev(k_idx), workspace=ws)
    msa.msa_check_device_status(ws)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    want, gap, _ = oracle.full_topk(oracle.shape_of(cfg), q_idx, k_idx)
    bad = int((got != want).any(axis=-1).sum())
    print(f"{cfg.name}: rows={got.shape[1] * got.shape[2]} tied at the boundary={(gap == 0).sum()} mismatches={bad}")
    assert bad == 0


def _sampled_rows(w, n_per_group, seed):
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(w.B):
        for g in range(w.G):
            t = np.concatenate([
                np.arange(0, 3), np.arange(w.T - 3, w.T),                      # first and last positions
                rng.integers(0, w.T, n_per_group),                             # random positions
                ((rng.integers(1, w.n_blocks, 8) * w.Bk)[:, None] + np.array([-1, 0])).ravel(),  # block edges
            ])
            rows.append((b * w.G + g) * w.T + np.unique(t))
    return np.concatenate(rows)


@pytest.mark.parametrize("w,n_per_group,seed", [(synth.B4_T8192, 96, 2), (synth.T131072, 64, 3),
                                               (synth.T1048576, 24, 4)], ids=["b4_t8192", "t131072", "t1048576"])
def test_index_topk_large_workloads_sampled(msa, w, n_per_group, seed):
    inp, got = _run(msa, w)
    rows = _sampled_rows(w, n_per_group, seed=seed)
    b = rows // (w.G * w.T)
    g = (rows // w.T) % w.G
    t = rows % w.T
    sub = got[b, g, t]
    valid_selection(got[:, :, : min(w.T, 4096)], min(w.T, 4096), w.Bk)
    want, gap, _ = oracle.index_topk(oracle.shape_of(w), inp["q_idx"], inp["k_idx"], rows=rows)
    n, ties, bad, bad_tie = compare_block_idx(sub, want, gap)
    print(f"{w.name}: sampled rows={n} near_ties={ties} mismatches(outside ties)={bad} (in ties)={bad_tie}")
    assert bad == 0
