"""Parity of msa_index_topk_fp8 (CUDA) with the oracle's FP8 index top-k:
bit-exact block ids except at near-ties (oracle k-th/(k+1)-th pooled-score
gap < 1e-4), given the same E4M3 quantization (per-row q scales, per-block k
scales, ties to even, saturation). The overlap with the bf16 selection is
printed: quantization may reorder blocks whose pooled scores are close.
"""
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
    ws = msa.alloc_workspace(s, msa.MSA_WS_TOPK_FP8)
    bi = torch.empty((w.B, w.G, w.T, w.k), dtype=torch.int32, device="cuda")
    msa.msa_index_topk_fp8(s, to_dev(inp["q_idx"]), to_dev(inp["k_idx"]), bi, ws)
    msa.msa_check_device_status(ws)
    torch.cuda.synchronize()
    return inp, bi.cpu().numpy()


@pytest.mark.parametrize("cfg", [
    synth.T1024,
    synth.T1024.with_(T=128, name="single_block"),
    synth.T1024.with_(B=2, T=768, G=3, Hq=3, k=5, name="b2_g3_hg1"),
    synth.T1024.with_(T=1536, G=2, Hq=16, k=33, name="k33"),
    synth.T8192,
], ids=["cfg0", "single_block", "b2_g3_hg1", "k33", "cfg1"])
def test_index_topk_fp8_matches_oracle(msa, cfg):
    inp, got = _run(msa, cfg)
    valid_selection(got, cfg.T, cfg.Bk)
    s = oracle.shape_of(cfg)
    want, gap, _ = oracle.index_topk_fp8(s, inp["q_idx"], inp["k_idx"])
    want = want.reshape(got.shape)
    n, ties, bad, bad_tie = compare_block_idx(got, want, gap)
    bf16, _, _ = oracle.index_topk(s, inp["q_idx"], inp["k_idx"])
    bf16 = bf16.reshape(got.shape)
    sel = got >= 0
    overlap = np.mean([len(set(a[a >= 0]) & set(b_[b_ >= 0])) / max(1, (a >= 0).sum())
                       for a, b_ in zip(got.reshape(-1, cfg.k), bf16.reshape(-1, cfg.k))])
    print(f"{cfg.name}: rows={n} near_ties={ties} mismatches(outside ties)={bad} (in ties)={bad_tie} "
          f"overlap with the bf16 selection={overlap:.4f} selected={int(sel.sum())}")
    assert bad == 0


def test_fp8_workspace_kind(msa):
    w = synth.T1024
    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    need = msa.msa_workspace_size(s, msa.MSA_WS_TOPK_FP8)
    assert need >= w.B * w.T * (w.G + 1) * w.d_idx + w.B * w.n_blocks * 4


@pytest.mark.parametrize("cfg", [
    synth.T1024.with_(T=4096, G=2, Hq=16, k=16, name="ties_k16"),
    synth.T1024.with_(T=8192, G=1, Hq=8, k=33, name="ties_k33"),
], ids=["k16", "k33"])
def test_index_topk_fp8_exact_ties(msa, cfg):
    """tied_index_inputs through the FP8 path: the keys of every block share one
    set of E4M3 codes and the block scales differ by powers of two, so equal
    levels tie exactly; every row must match the oracle's FP8 selection."""
    import torch

    q_idx, k_idx = synth.tied_index_inputs(cfg)
    s = msa.Shape(B=cfg.B, T=cfg.T, Hq=cfg.Hq, G=cfg.G, k=cfg.k)
    ws = msa.alloc_workspace(s, msa.MSA_WS_TOPK_FP8)
    got = torch.empty((cfg.B, cfg.G, cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    msa.msa_index_topk_fp8(s, to_dev(q_idx), to_dev(k_idx), got, ws)
    msa.msa_check_device_status(ws)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    want, gap, _ = oracle.index_topk_fp8(oracle.shape_of(cfg), q_idx, k_idx)
    want = want.reshape(got.shape)
    bad = int((got != want).any(axis=-1).sum())
    print(f"{cfg.name}: rows={want.shape[0] * want.shape[2]} tied at the boundary={(gap == 0).sum()} mismatches={bad}")
    assert bad == 0


@pytest.mark.parametrize("w,n_per_group,seed", [(synth.T131072, 64, 103), (synth.T1048576, 24, 104)],
                         ids=["t131072", "t1048576"])
def test_index_topk_fp8_large_workloads_sampled(msa, w, n_per_group, seed):
    """The full-size workloads (T = 131072 and T = 2^20), in the launch
    configuration the bench times: sampled rows (first and last positions,
    block edges, random positions) against the oracle's FP8 selection."""
    inp, got = _run(msa, w)
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(w.B):
        for g in range(w.G):
            t = np.concatenate([np.arange(0, 3), np.arange(w.T - 3, w.T), rng.integers(0, w.T, n_per_group),
                                ((rng.integers(1, w.n_blocks, 8) * w.Bk)[:, None] + np.array([-1, 0])).ravel()])
            rows.append((b * w.G + g) * w.T + np.unique(t))
    rows = np.concatenate(rows)
    b, g, t = rows // (w.G * w.T), (rows // w.T) % w.G, rows % w.T
    valid_selection(got[:, :, : min(w.T, 4096)], min(w.T, 4096), w.Bk)
    want, gap, _ = oracle.index_topk_fp8(oracle.shape_of(w), inp["q_idx"], inp["k_idx"], rows=rows)
    n, ties, bad, bad_tie = compare_block_idx(got[b, g, t], want, gap)
    print(f"{w.name}: sampled rows={n} near_ties={ties} mismatches(outside ties)={bad} (in ties)={bad_tie}")
    assert bad == 0
