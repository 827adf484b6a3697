"""Repeatability of the CUDA path: two runs on the same inputs give the same bits.

The block map is built without atomics on global counters (every list comes
out sorted by query), and every sum over tiles, slots, groups or key quarters
runs in a fixed order (a KL partial per slot and key quarter, added in order by
the merge), so block_idx, O, LSE, dQ, dK, dV, dq_idx, dk_idx and KL must be
bit-identical between runs, for both backward kernels (128-row tiles for 4
heads per group, 64-row tiles for 2).
"""
import numpy as np
import pytest

import synth
from helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__

    __graft_entry__.build_library()
    import block_sparse_attention_scores_gb300 as m

    return m


def _run(msa, w, inp):
    import torch

    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    ws = msa.alloc_workspace(s, msa.MSA_WS_BWD)
    d = {n: to_dev(inp[n]) for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")}
    bi = msa.index_topk(s, d["q_idx"], d["k_idx"], workspace=ws)
    O, LSE = msa.sparse_fwd(s, d["Q"], d["K"], d["V"], bi, workspace=ws)
    out = msa.bwd(s, d["Q"], d["K"], d["V"], O, d["dO"], LSE, d["q_idx"], d["k_idx"], bi, workspace=ws)
    msa.msa_check_device_status(ws)
    torch.cuda.synchronize()
    res = {"block_idx": bi, "O": O, "LSE": LSE}
    res.update(out)
    # bf16 has no numpy type: compare its bit patterns
    return {k: (v.view(torch.int16) if v.dtype == torch.bfloat16 else v).cpu().numpy() for k, v in res.items()}


@pytest.mark.parametrize("w", [synth.T1024, synth.T1024.with_(T=4096, Hq=16, G=4, k=8, name="t4096_hg4"),
                               synth.T1024.with_(T=2048, Hq=4, G=2, k=8, name="t2048_hg2")],
                         ids=["cfg0", "t4096_hg4", "t2048_hg2"])
def test_two_runs_give_identical_bits(msa, w):
    inp = synth.make_inputs(w)
    a = _run(msa, w, inp)
    b = _run(msa, w, inp)
    assert set(a) == set(b)
    for name in a:
        assert np.array_equal(a[name].view(np.uint8), b[name].view(np.uint8)), name
