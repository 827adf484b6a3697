"""Parity of msa_sparse_fwd (CUDA) with the fp64 oracle, given identical block_idx.

Tolerance (bf16 inputs, fp32 accumulation): max |err| <= 2e-2 and cosine >= 0.999
for O and LSE. Small shapes compare every element; the large workloads compare
sampled query rows, with a random (structurally valid) block selection.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__

    __graft_entry__.build_library()
    import block_sparse_attention_scores_gb300 as m

    return m


def _gpu_fwd(msa, w, inp, bi):
    import torch

    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    ws = msa.alloc_workspace(s, msa.MSA_WS_FWD)
    O, LSE = msa.sparse_fwd(s, to_dev(inp["Q"]), to_dev(inp["K"]), to_dev(inp["V"]),
                            to_dev(np.ascontiguousarray(bi, dtype=np.int32), "int32"), workspace=ws)
    msa.msa_check_device_status(ws)
    torch.cuda.synchronize()
    return O, LSE


SMALL = [
    synth.T1024,
    synth.T1024.with_(T=128, name="single_block"),
    synth.T1024.with_(T=512, k=1, name="k1_own_block_only"),
    synth.T1024.with_(T=640, k=8, name="k_gt_blocks_dense_causal"),
    synth.T1024.with_(B=2, T=768, Hq=3, G=3, k=3, name="b2_hg1"),
    synth.T1024.with_(T=1024, Hq=4, G=2, k=5, name="hg2"),
    synth.T1024.with_(T=1024, Hq=16, G=2, k=6, name="hg8"),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_sparse_fwd_matches_oracle_full(msa, w):
    inp = synth.make_inputs(w)
    s = oracle.shape_of(w)
    bi, _, _ = oracle.full_topk(s, inp["q_idx"], inp["k_idx"])
    O_ref, L_ref = oracle.full_fwd(s, inp["Q"], inp["K"], inp["V"], bi)
    O, LSE = _gpu_fwd(msa, w, inp, bi)
    e1 = assert_close("O", to_f64(O), O_ref)
    e2 = assert_close("LSE", to_f64(LSE), L_ref)
    print(f"{w.name}: O err={e1[0]:.2e} cos={e1[1]:.6f}  LSE err={e2[0]:.2e}")


def test_sparse_fwd_t8192_full(msa):
    w = synth.T8192
    inp = synth.make_inputs(w)
    s = oracle.shape_of(w)
    bi, _, _ = oracle.full_topk(s, inp["q_idx"], inp["k_idx"])
    O, LSE = _gpu_fwd(msa, w, inp, bi)
    O_ref, L_ref = oracle.full_fwd(s, inp["Q"], inp["K"], inp["V"], bi)
    e1 = assert_close("O", to_f64(O), O_ref)
    e2 = assert_close("LSE", to_f64(LSE), L_ref)
    print(f"{w.name}: O err={e1[0]:.2e} cos={e1[1]:.6f}  LSE err={e2[0]:.2e}")


def _sample_rows(w, n, seed):
    rng = np.random.default_rng(seed)
    b = rng.integers(0, w.B, n)
    t = np.concatenate([np.arange(4), np.arange(w.T - 4, w.T), rng.integers(0, w.T, n - 8)])
    h = rng.integers(0, w.Hq, n)
    return (b * w.T + t) * w.Hq + h


@pytest.mark.parametrize("w,n,seed", [(synth.B4_T8192, 512, 2), (synth.T131072, 512, 3), (synth.T1048576, 256, 4)],
                         ids=["b4_t8192", "t131072", "t1048576"])
def test_sparse_fwd_large_workloads_sampled(msa, w, n, seed):
    inp = synth.make_inputs(w, ("Q", "K", "V"))
    bi = synth.synthetic_block_idx(w)
    O, LSE = _gpu_fwd(msa, w, inp, bi)
    rows = _sample_rows(w, n, seed)
    O_ref, L_ref = oracle.sparse_fwd(oracle.shape_of(w), inp["Q"], inp["K"], inp["V"], bi, rows=rows)
    Og = to_f64(O.view(-1, w.d)[rows.tolist()])
    Lg = to_f64(LSE.view(-1)[rows.tolist()])
    e1 = assert_close("O", Og, O_ref)
    e2 = assert_close("LSE", Lg, L_ref)
    print(f"{w.name}: sampled rows={rows.size} O err={e1[0]:.2e} cos={e1[1]:.6f} LSE err={e2[0]:.2e}")


def test_sparse_fwd_rejects_bad_block_idx(msa):
    """A row without its own block is reported through the device error word."""
    import torch

    w = synth.T1024.with_(T=256, k=2)
    inp = synth.make_inputs(w, ("Q", "K", "V"))
    bi = synth.synthetic_block_idx(w)
    bi[0, 0, 200] = [0, -1]  # own block (1) missing
    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    ws = msa.alloc_workspace(s, msa.MSA_WS_FWD)
    msa.sparse_fwd(s, to_dev(inp["Q"]), to_dev(inp["K"]), to_dev(inp["V"]), to_dev(bi, "int32"), workspace=ws)
    with pytest.raises(msa.MsaError) as e:
        msa.msa_check_device_status(ws)
    assert e.value.status == msa.MSA_ERR_DEVICE
    msa.msa_check_device_status(ws)  # the word was cleared
    torch.cuda.synchronize()
