"""msa_set_timing_events: caller-owned CUDA events recorded by the library around
one stage's main kernel measure that kernel alone (inside the whole call)."""
import numpy as np
import pytest

import synth
from helpers import to_dev

pytestmark = pytest.mark.gpu


def test_kernel_events_bracket_only_the_main_kernel():
    import torch

    import __graft_entry__

    __graft_entry__.build_library()
    import block_sparse_attention_scores_gb300 as msa

    w = synth.T1024.with_(T=4096, k=8)
    inp = synth.make_inputs(w)
    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, k=w.k)
    d = {n: to_dev(inp[n]) for n in inp}
    ws = msa.alloc_workspace(s, msa.MSA_WS_BWD)
    bi = msa.index_topk(s, d["q_idx"], d["k_idx"], workspace=ws)
    O, LSE = msa.sparse_fwd(s, d["Q"], d["K"], d["V"], bi, workspace=ws)
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in ev:
        e.record(stream)
    torch.cuda.synchronize()
    msa.msa_set_timing_events(msa.MSA_TIME_BWD, ev[1], ev[2])
    try:
        ev[0].record(stream)
        out = msa.bwd(s, d["Q"], d["K"], d["V"], O, d["dO"], LSE, d["q_idx"], d["k_idx"], bi, workspace=ws)
        ev[3].record(stream)
    finally:
        msa.msa_set_timing_events(msa.MSA_TIME_BWD, None, None)
    torch.cuda.synchronize()
    msa.msa_check_device_status(ws)
    whole = ev[0].elapsed_time(ev[3])
    kernel = ev[1].elapsed_time(ev[2])
    before, after = ev[0].elapsed_time(ev[1]), ev[2].elapsed_time(ev[3])
    print(f"msa_bwd {whole:.3f} ms, bwd_kernel {kernel:.3f} ms")
    assert 0 < kernel < whole and before > 0 and after > 0  # pre-passes before it, merges after it
    assert np.isfinite(out["dQ"].cpu().numpy()).all()
