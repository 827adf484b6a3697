"""IndexShare: msa_block_map once, then msa_sparse_fwd_mapped / msa_bwd_mapped.

The mapped calls run on a map built once from block_idx (lists padded to whole
forward tiles, work items for both kernels) and must give the same bits as
msa_sparse_fwd / msa_bwd, which build their own map (KL to within fp32
rounding: it sums key quarters with shared-memory atomics). Two layers with
different Q, K, V, dO but one shared selection reuse the same map.
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


def _host(t):
    import torch

    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).cpu().numpy()


def _outputs(msa, s, w, d, bi, ws, mapped):
    import torch

    f32 = dict(dtype=torch.float32, device="cuda")
    O = torch.empty_like(d["Q"])
    LSE = torch.empty((w.B, w.T, w.Hq), **f32)
    g = {n: torch.empty(d[src].shape, **f32) for n, src in
         (("dQ", "Q"), ("dK", "K"), ("dV", "V"), ("dq_idx", "q_idx"), ("dk_idx", "k_idx"))}
    KL = torch.empty((w.B, w.G, w.T), **f32)
    fwd = msa.msa_sparse_fwd_mapped if mapped else msa.msa_sparse_fwd
    bwd = msa.msa_bwd_mapped if mapped else msa.msa_bwd
    fwd(s, d["Q"], d["K"], d["V"], bi, O, LSE, ws)
    bwd(s, d["Q"], d["K"], d["V"], O, d["dO"], LSE, d["q_idx"], d["k_idx"], bi, 1.0, g["dQ"], g["dK"], g["dV"],
        g["dq_idx"], g["dk_idx"], KL, ws)
    msa.msa_check_device_status(ws)
    torch.cuda.synchronize()
    out = {"O": O, "LSE": LSE, "KL": KL}
    out.update(g)
    return {k: _host(v) for k, v in out.items()}


@pytest.mark.parametrize("w", [synth.T1024, synth.T1024.with_(T=4096, Hq=16, G=4, k=8, name="t4096_hg4"),
                               synth.T1024.with_(B=2, T=768, Hq=3, G=3, k=3, name="b2_hg1")],
                         ids=["cfg0", "t4096_hg4", "b2_hg1"])
def test_mapped_calls_match_unmapped(msa, w):
    inp = synth.make_inputs(w)
    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    d = {n: to_dev(inp[n]) for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")}
    ws_ref = msa.alloc_workspace(s, msa.MSA_WS_BWD)
    bi = msa.index_topk(s, d["q_idx"], d["k_idx"], workspace=ws_ref)
    ref = _outputs(msa, s, w, d, bi, ws_ref, mapped=False)

    ws = msa.alloc_workspace(s, msa.MSA_WS_BWD)
    msa.msa_block_map(s, bi, ws)
    # a second layer: new activations, the same selection and map
    inp2 = synth.make_inputs(w.with_(seed=w.seed + 1000))
    d2 = {n: to_dev(inp2[n]) for n in ("Q", "K", "V", "dO")}
    d2.update({"q_idx": d["q_idx"], "k_idx": d["k_idx"]})
    for layer, dd in enumerate((d, d2, d)):
        got = _outputs(msa, s, w, dd, bi, ws, mapped=True)
        want = ref if layer != 1 else _outputs(msa, s, w, d2, bi, ws_ref, mapped=False)
        for name in want:
            if name == "KL":
                np.testing.assert_allclose(got[name], want[name], rtol=1e-5, atol=1e-7)
            else:
                assert np.array_equal(got[name].view(np.uint8), want[name].view(np.uint8)), (layer, name)


def test_mapped_calls_need_a_backward_workspace(msa):
    import torch

    w = synth.T1024
    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    small = msa.alloc_workspace(s, msa.MSA_WS_FWD)
    bi = torch.zeros((w.B, w.G, w.T, w.k), dtype=torch.int32, device="cuda")
    with pytest.raises(msa.MsaError) as e:
        msa.msa_block_map(s, bi, small)
    assert e.value.status == msa.MSA_ERR_WORKSPACE
