"""Full attention at any T (msa_dense_fwd / msa_dense_bwd): the indexer
warmup's dense causal attention and dense-teacher KL without a block list.

Parity with the fp64 oracle's full-attention form (no block_idx: every
visible token), at the bar of the sparse path (max |err| <= 2e-2, cosine >=
0.999): every element at small T, including logits large enough that the
running row maximum moves by more than the forward's rescale headroom; sampled
rows and KV blocks whose queries span several of the backward's 4096-query
segments; sampled rows and one (block, group) at T = 131072. And, on the GPU,
the dense calls against msa_sparse_fwd / msa_bwd given msa_warmup_block_idx's
selection (every visible block), element by element at T = 8192 and 16384.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close, assert_kl_sum, to_dev, to_f64

pytestmark = pytest.mark.gpu
NAMES = ("Q", "K", "V", "dO", "q_idx", "k_idx")


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__

    __graft_entry__.build_library()
    import block_sparse_attention_scores_gb300 as m

    return m


def _shape(msa, w, scale=0.0):
    return msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=1, scale=scale)


def _run_dense(msa, w, inp, scale=0.0, kl_weight=1.0):
    import torch

    s = _shape(msa, w, scale)
    ws = msa.alloc_workspace(s, msa.MSA_WS_DENSE)
    d = {n: to_dev(inp[n]) for n in NAMES}
    O, LSE = msa.dense_fwd(s, d["Q"], d["K"], d["V"], workspace=ws)
    out = msa.dense_bwd(s, d["Q"], d["K"], d["V"], O, d["dO"], LSE, d["q_idx"], d["k_idx"], kl_weight=kl_weight,
                        workspace=ws)
    msa.msa_check_device_status(ws)
    torch.cuda.synchronize()
    out["O"], out["LSE"] = O, LSE
    return out


SMALL = [
    (synth.T1024.with_(T=128, name="one_block"), 0.0),
    (synth.T1024.with_(name="t1024_hg4"), 0.0),
    (synth.T1024.with_(B=2, T=768, Hq=16, G=2, name="b2_t768_hg8"), 0.0),
    # scale 1: logits about 16x the default, so the running maximum of a row moves by more than 2^8
    (synth.T1024.with_(T=1024, Hq=4, G=1, name="t1024_large_logits"), 1.0),
]


@pytest.mark.parametrize("w,scale", SMALL, ids=[w.name for w, _ in SMALL])
def test_dense_matches_oracle_full(msa, w, scale):
    inp = synth.make_inputs(w)
    s = oracle.shape_of(w, scale=scale or None, kl_weight=0.5)
    O_ref, LSE_ref = oracle.full_fwd(s, inp["Q"], inp["K"], inp["V"], None)
    ref = oracle.full_bwd(s, *[inp[n] for n in NAMES], None)
    got = _run_dense(msa, w, inp, scale=scale, kl_weight=0.5)
    msg = [("O",) + assert_close("O", to_f64(got["O"]), O_ref),
           ("LSE",) + assert_close("LSE", to_f64(got["LSE"]), LSE_ref)]
    for name in ("dQ", "dK", "dV", "dq_idx", "dk_idx", "KL"):
        # P and dS enter the MMAs as bf16 (relative rounding 2^-9): the absolute error of a gradient grows
        # with its magnitude, which large logits raise to tens (dQ up to 45, dK 70 at scale 1)
        bound = 2e-2 * max(1.0, float(np.abs(ref[name]).max()))
        msg.append((name,) + assert_close(name, to_f64(got[name]), ref[name], max_abs=bound))
    assert_kl_sum(to_f64(got["KL"]), ref["KL"])
    print(w.name + ": " + "  ".join(f"{n} err={e:.1e} cos={c:.6f}" for n, e, c in msg))


@pytest.mark.parametrize("w", [
    synth.T8192.with_(B=2, name="b2_t8192"),
    synth.T8192.with_(T=16384, name="t16384"),
], ids=lambda w: w.name)
def test_dense_equals_sparse_path_on_full_selection(msa, w):
    """Two independent GPU paths to the same full attention: query-outer dense
    forward + segmented dense backward, and the KV-outer sparse kernels with
    per-slot partials on the all-blocks selection (4 segments at T = 16384)."""
    import torch

    inp = synth.make_inputs(w)
    got = _run_dense(msa, w, inp, kl_weight=0.8)
    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.T // w.Bk)
    ws = msa.alloc_workspace(s, msa.MSA_WS_BWD)
    d = {n: to_dev(inp[n]) for n in NAMES}
    bi = msa.warmup_block_idx(s)
    O, LSE = msa.sparse_fwd(s, d["Q"], d["K"], d["V"], bi, workspace=ws)
    ref = msa.bwd(s, d["Q"], d["K"], d["V"], O, d["dO"], LSE, d["q_idx"], d["k_idx"], bi, kl_weight=0.8, workspace=ws)
    msa.msa_check_device_status(ws)
    torch.cuda.synchronize()
    ref["O"], ref["LSE"] = O, LSE
    msg = []
    for name in ("O", "LSE", "dQ", "dK", "dV", "dq_idx", "dk_idx", "KL"):
        msg.append((name,) + assert_close(name, to_f64(got[name]), to_f64(ref[name])))
    print(w.name + ": " + "  ".join(f"{n} err={e:.1e} cos={c:.6f}" for n, e, c in msg))


def _pick(t, *idx):
    """t[idx] gathered on the device (the full tensors are GBs at T = 131072), as float64 numpy."""
    import torch

    return to_f64(t[tuple(torch.as_tensor(np.asarray(i), device=t.device) for i in idx)])


def _sampled(msa, w, rows_n, blocks, seed, group=None):
    """Sampled query rows (O, LSE, dQ, dq_idx, KL) and KV blocks ((b, c) pairs:
    dK, dV, and dk_idx unless `group` restricts the block sums to one group) of
    one dense forward + backward against the oracle's full-attention form."""
    inp = synth.make_inputs(w)
    got = _run_dense(msa, w, inp)
    s = oracle.shape_of(w)
    rng = np.random.default_rng(seed)
    b = rng.integers(0, w.B, rows_n)
    g = rng.integers(0, w.G, rows_n)
    t = np.concatenate([np.array([0, 127, 128, 4095, 4096, w.T - 1]), rng.integers(0, w.T, rows_n - 6)]) % w.T
    heads = g * w.hg + rng.integers(0, w.hg, rows_n)
    res = []
    O_ref, LSE_ref = oracle.sparse_fwd(s, inp["Q"], inp["K"], inp["V"], None, rows=(b * w.T + t) * w.Hq + heads)
    res.append(("O",) + assert_close("O", _pick(got["O"], b, t, heads), O_ref))
    res.append(("LSE",) + assert_close("LSE", _pick(got["LSE"], b, t, heads), LSE_ref))
    dQ, dqi, KL = oracle.bwd_rows(s, *[inp[n] for n in NAMES], None, rows=(b * w.G + g) * w.T + t)
    gdQ = _pick(got["dQ"], b, t).reshape(rows_n, w.G, w.hg, w.d)[np.arange(rows_n), g]
    res.append(("dQ",) + assert_close("dQ", gdQ, dQ))
    res.append(("dq_idx",) + assert_close("dq_idx", _pick(got["dq_idx"], b, t, g), dqi))
    res.append(("KL",) + assert_close("KL", _pick(got["KL"], b, g, t), KL))
    assert_kl_sum(_pick(got["KL"], b, g, t), KL)
    bb = np.array([x[0] for x in blocks])
    cc = np.array([x[1] for x in blocks])
    dK, dV, dki = oracle.bwd_blocks(s, *[inp[n] for n in NAMES], None, blocks=bb * w.n_blocks + cc, group=group)
    for i, (b0, c0) in enumerate(blocks):
        sl = slice(c0 * w.Bk, (c0 + 1) * w.Bk)
        gsel = slice(None) if group is None else slice(group, group + 1)
        gK = to_f64(got["dK"][b0, sl]).transpose(1, 0, 2)[gsel]
        gV = to_f64(got["dV"][b0, sl]).transpose(1, 0, 2)[gsel]
        res.append(("dK",) + assert_close("dK", gK, dK[i][gsel]))
        res.append(("dV",) + assert_close("dV", gV, dV[i][gsel]))
        if group is None:
            res.append(("dk_idx",) + assert_close("dk_idx", to_f64(got["dk_idx"][b0, sl]), dki[i]))
    print(w.name + ": " + "  ".join(f"{n} err={e:.1e} cos={c:.6f}" for n, e, c in res))


@pytest.mark.parametrize("w,blocks", [
    # 4608 queries: segments [0, 4096) and [4096, 4608); block 30's queries lie in both, block 24's too
    (synth.T1024.with_(B=2, T=4608, name="b2_t4608_hg4"), [(0, 30), (1, 24), (1, 35)]),
    (synth.T1024.with_(T=4608, Hq=16, G=2, name="t4608_hg8"), [(0, 31), (0, 33)]),
], ids=["b2_t4608_hg4", "t4608_hg8"])
def test_dense_sampled_across_segments(msa, w, blocks):
    _sampled(msa, w, 64, blocks, seed=11)


def test_dense_full_size_sampled(msa):
    """T = 131072, Hq = 32, G = 8 (the headline layer): sampled rows, and the
    last KV block's dK, dV for one group (every group's queries of one block
    would cost the oracle a minute)."""
    w = synth.T131072
    _sampled(msa, w, 40, [(0, w.n_blocks - 1)], seed=13, group=3)
