"""The per-rank hot path of head-wise context parallelism on one GPU.

Every rank of block_sparse_attention_scores_gb300.context_parallel runs the
library on its own slice of G / W groups (all T tokens, the full k_idx). Here
the W = 2 slices of one layer run one after the other on one GPU through
``cuda_compute``, with no collective, and are compared with a single call on
the whole layer: selection, forward outputs and per-group gradients must be
bit-identical (a group's work does not depend on the other groups), KL equal
to fp32 rounding (it sums with shared-memory atomics), and dk_idx, the term
the ranks reduce, equal to fp32 rounding once the two slices' sums are added.
"""
import numpy as np
import pytest
import torch

import synth
from helpers import to_dev

pytestmark = pytest.mark.gpu


def test_group_slices_equal_whole_layer():
    import __graft_entry__

    __graft_entry__.build_library()
    from block_sparse_attention_scores_gb300 import context_parallel as cp

    w = synth.T8192.with_(T=2048, name="cp_b1_t2048_hq32_g8_k16")
    inp = synth.make_inputs(w)
    d = {n: to_dev(inp[n]) for n in cp.INPUTS}
    s = cp.LayerShape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    full = cp.cuda_compute(s, d)
    world = 2
    loc = cp.local_shape(s, world)
    hg = w.Hq // w.G
    parts = []
    for r in range(world):
        g0, g1 = cp.group_range(w.G, world, r)
        t = dict(Q=d["Q"][:, :, g0 * hg:g1 * hg].contiguous(), dO=d["dO"][:, :, g0 * hg:g1 * hg].contiguous(),
                 K=d["K"][:, :, g0:g1].contiguous(), V=d["V"][:, :, g0:g1].contiguous(),
                 q_idx=d["q_idx"][:, :, g0:g1].contiguous(), k_idx=d["k_idx"])
        parts.append(cp.cuda_compute(loc, t))
    torch.cuda.synchronize()
    for n in ("block_idx", "O", "LSE", "dQ", "dK", "dV", "dq_idx", "KL"):
        t_axis, h_axis = cp.AXES[n]
        got = torch.cat([p[n] for p in parts], dim=h_axis)
        if n == "KL":
            torch.testing.assert_close(got, full[n], rtol=1e-5, atol=1e-6)
        else:
            assert torch.equal(got, full[n]), n
    dki = parts[0]["dk_idx"] + parts[1]["dk_idx"]
    torch.testing.assert_close(dki, full["dk_idx"], rtol=1e-4, atol=1e-5)
    assert float(full["dk_idx"].abs().max()) > 1e-3


def test_full_attention_group_slices_equal_whole_layer():
    """The same for the indexer warmup's full attention (cuda_compute_dense):
    the forward is deterministic and per group, so O and LSE are bit-identical;
    the backward adds its sums with atomics, so the gradients and KL match the
    whole-layer call to fp32 rounding, dk_idx once the slices' sums are added."""
    import __graft_entry__

    __graft_entry__.build_library()
    from block_sparse_attention_scores_gb300 import context_parallel as cp

    w = synth.T8192.with_(T=2048, name="cp_dense_b1_t2048_hq32_g8")
    inp = synth.make_inputs(w)
    d = {n: to_dev(inp[n]) for n in cp.INPUTS}
    s = cp.LayerShape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=1)
    full = cp.cuda_compute_dense(s, d)
    world = 2
    loc = cp.local_shape(s, world)
    hg = w.Hq // w.G
    parts = []
    for r in range(world):
        g0, g1 = cp.group_range(w.G, world, r)
        t = dict(Q=d["Q"][:, :, g0 * hg:g1 * hg].contiguous(), dO=d["dO"][:, :, g0 * hg:g1 * hg].contiguous(),
                 K=d["K"][:, :, g0:g1].contiguous(), V=d["V"][:, :, g0:g1].contiguous(),
                 q_idx=d["q_idx"][:, :, g0:g1].contiguous(), k_idx=d["k_idx"])
        parts.append(cp.cuda_compute_dense(loc, t))
    torch.cuda.synchronize()
    assert "block_idx" not in full
    for n in ("O", "LSE", "dQ", "dK", "dV", "dq_idx", "KL"):
        t_axis, h_axis = cp.AXES[n]
        got = torch.cat([p[n] for p in parts], dim=h_axis)
        if n in ("O", "LSE"):
            assert torch.equal(got, full[n]), n
        else:
            torch.testing.assert_close(got, full[n], rtol=1e-4, atol=1e-5)
    dki = parts[0]["dk_idx"] + parts[1]["dk_idx"]
    torch.testing.assert_close(dki, full["dk_idx"], rtol=1e-4, atol=1e-5)
    assert float(full["dk_idx"].abs().max()) > 1e-3
