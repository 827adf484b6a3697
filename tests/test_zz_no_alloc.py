"""msa_index_topk_noalloc: the index top-k for callers that cannot allocate
device memory (a plugin whose host owns all device memory, or a path where
cudaMalloc's implicit synchronisation is not acceptable). Its scratch lives in
a static device array inside the library. Called through the C ABI directly,
twice in a row, its block indices must equal those of msa_index_topk (the
workspace-taking entry point) exactly, as block indices are compared
everywhere in these tests. Collected last so that a failing run has already
run every other test."""
import ctypes

import numpy as np
import pytest

import synth
from helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [synth.T1024.with_(T=2048, name="t2048"),
                               synth.T1024.with_(B=2, T=1536, G=3, Hq=6, k=6, name="b2_g3_k6")],
                         ids=lambda w: w.name)
def test_noalloc_topk_matches_workspace_topk_twice(w):
    import torch

    import __graft_entry__

    __graft_entry__.build_library()
    import block_sparse_attention_scores_gb300 as msa

    lib = ctypes.CDLL(msa.LIB_PATH)
    lib.msa_index_topk_noalloc.argtypes = [ctypes.POINTER(msa.MsaShape), ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    lib.msa_index_topk_noalloc.restype = ctypes.c_int
    lib.msa_last_error.restype = ctypes.c_char_p

    inp = synth.make_inputs(w, ("q_idx", "k_idx"))
    qi, ki = to_dev(inp["q_idx"]), to_dev(inp["k_idx"])
    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    ref = msa.index_topk(s, qi, ki)  # the workspace-taking entry point
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    cs = s.c()
    for call in range(2):
        out = torch.full((w.B, w.G, w.T, w.k), -7, dtype=torch.int32, device="cuda")
        st = lib.msa_index_topk_noalloc(ctypes.byref(cs), qi.data_ptr(), ki.data_ptr(), out.data_ptr(), 1, stream)
        assert st == msa.MSA_OK, lib.msa_last_error().decode()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), ref.cpu().numpy(), err_msg=f"call {call}")


def test_noalloc_rejects_bad_arguments_before_any_work():
    import __graft_entry__

    __graft_entry__.build_library()
    import block_sparse_attention_scores_gb300 as msa

    lib = ctypes.CDLL(msa.LIB_PATH)
    lib.msa_index_topk_noalloc.argtypes = [ctypes.POINTER(msa.MsaShape), ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    lib.msa_index_topk_noalloc.restype = ctypes.c_int
    cs = msa.Shape(B=1, T=1024, Hq=8, G=2, k=4).c()
    assert lib.msa_index_topk_noalloc(ctypes.byref(cs), None, None, None, 1, None) == msa.MSA_ERR_INVALID_ARG
    bad = msa.Shape(B=1, T=1000, Hq=8, G=2, k=4).c()
    assert lib.msa_index_topk_noalloc(ctypes.byref(bad), 4096, 4096, 4096, 1, None) == msa.MSA_ERR_UNSUPPORTED
