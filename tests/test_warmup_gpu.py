"""Indexer warmup (full attention while the indexer learns): msa_warmup_block_idx
writes the full causal selection, and msa_sparse_fwd / msa_bwd given it compute
dense causal attention and the dense-teacher KL over every visible token.

Parity with the fp64 oracle on the same selection, at the bar of the sparse path:
max |err| <= 2e-2 and cosine >= 0.999 for O, LSE and the fp32 gradients, and
the selection itself bit-exact against its closed form.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close, assert_kl_sum, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__

    __graft_entry__.build_library()
    import block_sparse_attention_scores_gb300 as m

    return m


def _closed_form(w):
    t = np.arange(w.T)
    sel = np.where(np.arange(w.k)[None, :] <= (t // w.Bk)[:, None], np.arange(w.k)[None, :], -1).astype(np.int32)
    return np.broadcast_to(sel, (w.B, w.G, w.T, w.k))


def _warm(w):
    return w.with_(k=w.T // w.Bk, name=w.name + "_warmup")


def _run(msa, w, inp):
    import torch

    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    ws = msa.alloc_workspace(s, msa.MSA_WS_BWD)
    d = {n: to_dev(inp[n]) for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")}
    bi = msa.warmup_block_idx(s)
    O, LSE = msa.sparse_fwd(s, d["Q"], d["K"], d["V"], bi, workspace=ws)
    out = msa.bwd(s, d["Q"], d["K"], d["V"], O, d["dO"], LSE, d["q_idx"], d["k_idx"], bi, workspace=ws)
    msa.msa_check_device_status(ws)
    torch.cuda.synchronize()
    out["O"], out["LSE"], out["block_idx"] = O, LSE, bi
    return out


@pytest.mark.parametrize("w", [
    synth.T1024.with_(T=128, k=1, name="one_block"),
    synth.T1024.with_(T=1024, k=8, name="t1024_k8"),
    synth.T1024.with_(T=1024, k=11, name="t1024_k11_padded"),
    synth.T8192.with_(B=2, k=64, name="t8192_k64"),
    synth.T8192.with_(T=16384, k=128, name="t16384_k128"),
], ids=lambda w: w.name)
def test_warmup_selection_is_every_visible_block(msa, w):
    import torch

    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    bi = msa.warmup_block_idx(s)
    torch.cuda.synchronize()
    assert np.array_equal(bi.cpu().numpy(), _closed_form(w))


SMALL = [
    _warm(synth.T1024),                                                  # T=1024, hg=4, k=8
    _warm(synth.T1024.with_(B=2, T=768, Hq=3, G=3, name="b2_hg1")),     # k=6
    _warm(synth.T1024.with_(T=1024, Hq=16, G=2, name="hg8")),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_warmup_step_matches_oracle_full(msa, w):
    inp = synth.make_inputs(w)
    s = oracle.shape_of(w)
    bi = np.ascontiguousarray(_closed_form(w))
    O_ref, LSE_ref = oracle.sparse_fwd(s, inp["Q"], inp["K"], inp["V"], bi)
    ref = oracle.full_bwd(s, *[inp[n] for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")], bi)
    got = _run(msa, w, inp)
    msg = []
    msg.append(("O",) + assert_close("O", to_f64(got["O"]).reshape(O_ref.shape), O_ref))
    msg.append(("LSE",) + assert_close("LSE", to_f64(got["LSE"]).reshape(LSE_ref.shape), LSE_ref))
    for name in ("dQ", "dK", "dV", "dq_idx", "dk_idx", "KL"):
        msg.append((name,) + assert_close(name, to_f64(got[name]), ref[name]))
    assert_kl_sum(to_f64(got["KL"]), ref["KL"])
    print(w.name + ": " + "  ".join(f"{n} err={e:.1e} cos={c:.6f}" for n, e, c in msg))


def _sampled_parity(msa, w, bi, label, seed, blocks):
    """Sampled query rows (O, LSE, dQ, dq_idx, KL) and KV blocks `blocks`
    ((b, c) pairs: dK, dV, dk_idx) of one forward + backward on selection `bi`
    against the oracle. The oracle's cost for a block grows with the number of
    queries that selected it."""
    import torch

    inp = synth.make_inputs(w)
    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    ws = msa.alloc_workspace(s, msa.MSA_WS_BWD)
    d = {n: to_dev(inp[n]) for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")}
    bit = to_dev(np.ascontiguousarray(bi, dtype=np.int32), "int32")
    O, LSE = msa.sparse_fwd(s, d["Q"], d["K"], d["V"], bit, workspace=ws)
    got = msa.bwd(s, d["Q"], d["K"], d["V"], O, d["dO"], LSE, d["q_idx"], d["k_idx"], bit, workspace=ws)
    msa.msa_check_device_status(ws)
    torch.cuda.synchronize()
    got["O"], got["LSE"] = O, LSE
    os_ = oracle.shape_of(w)
    rng = np.random.default_rng(seed)
    n_rows = 96
    b = rng.integers(0, w.B, n_rows)
    g = rng.integers(0, w.G, n_rows)
    t = np.concatenate([np.array([0, 127, 128, w.T - 1]), rng.integers(0, w.T, n_rows - 4)])
    hg = w.Hq // w.G
    res = []
    heads = g * hg + rng.integers(0, hg, n_rows)
    O_ref, LSE_ref = oracle.sparse_fwd(os_, inp["Q"], inp["K"], inp["V"], bi, rows=(b * w.T + t) * w.Hq + heads)
    res.append(("O",) + assert_close("O", to_f64(got["O"])[b, t, heads], O_ref))
    res.append(("LSE",) + assert_close("LSE", to_f64(got["LSE"])[b, t, heads], LSE_ref))
    names = ("Q", "K", "V", "dO", "q_idx", "k_idx")
    dQ, dqi, KL = oracle.bwd_rows(os_, *[inp[n] for n in names], bi, rows=(b * w.G + g) * w.T + t)
    gdQ = to_f64(got["dQ"])[b, t].reshape(n_rows, w.G, hg, w.d)[np.arange(n_rows), g]
    res.append(("dQ",) + assert_close("dQ", gdQ, dQ))
    res.append(("dq_idx",) + assert_close("dq_idx", to_f64(got["dq_idx"])[b, t, g], dqi))
    res.append(("KL",) + assert_close("KL", to_f64(got["KL"])[b, g, t], KL))
    assert_kl_sum(to_f64(got["KL"])[b, g, t], KL)
    bb = np.array([x[0] for x in blocks])
    cc = np.array([x[1] for x in blocks])
    dK, dV, dki = oracle.bwd_blocks(os_, *[inp[n] for n in names], bi, blocks=bb * w.n_blocks + cc)
    gK, gV, gki = to_f64(got["dK"]), to_f64(got["dV"]), to_f64(got["dk_idx"])
    for i, (b0, c0) in enumerate(blocks):
        sl = slice(c0 * w.Bk, (c0 + 1) * w.Bk)
        res.append(("dK",) + assert_close("dK", gK[b0, sl].transpose(1, 0, 2), dK[i]))
        res.append(("dV",) + assert_close("dV", gV[b0, sl].transpose(1, 0, 2), dV[i]))
        res.append(("dk_idx",) + assert_close("dk_idx", gki[b0, sl], dki[i]))
    print(label + ": " + "  ".join(f"{n} err={e:.1e} cos={c:.6f}" for n, e, c in res))


@pytest.mark.parametrize("w,blocks", [
    # T=8192, all 64 blocks; block 0 is selected by every query of its batch
    (_warm(synth.T8192.with_(B=2)), [(0, 0), (1, 31), (1, 63)]),
    # T=16384, all 128 blocks; the last block keeps the oracle's per-block work small
    (_warm(synth.T8192.with_(T=16384, name="t16384")), [(0, 127)]),
], ids=["t8192_k64", "t16384_k128"])
def test_warmup_step_sampled(msa, w, blocks):
    """Dense causal attention and the dense-teacher KL at the largest sizes the
    warmup covers (Hq = 32, G = 8): sampled rows and blocks."""
    _sampled_parity(msa, w, np.ascontiguousarray(_closed_form(w)), "warmup " + w.name, seed=5, blocks=blocks)


def test_wide_sparse_selection_sampled(msa):
    """A random selection of 96 blocks per row (between 64 and 128 slots) at
    T = 16384: the forward and backward merges' wide path."""
    w = synth.T8192.with_(T=16384, G=2, Hq=8, k=96, name="k96")
    _sampled_parity(msa, w, synth.synthetic_block_idx(w), "sparse k96", seed=7, blocks=[(0, 124), (0, 127)])
