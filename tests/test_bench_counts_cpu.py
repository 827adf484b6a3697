"""The bench's counted work (selected pairs and FLOPs) against the table the
five workloads were specified with, and against a direct count on a
selection generated for a small shape."""
import pytest

import bench
import synth

# per workload: selected, causally visible (query, key) pairs per (b, g); forward (index + main) and
# forward+backward FLOPs, to the table's precision
COUNTS = [
    (synth.T1024, 360_960, 1.61e9, 5.59e9),
    (synth.T8192, 14_290_944, 2.69e11, 8.98e11),
    (synth.B4_T8192, 14_290_944, 1.07e12, 3.59e12),
    (synth.T131072, 258_146_304, 1.30e13, 2.44e13),
    (synth.T1048576, 2_078_932_992, 2.99e14, 3.44e14),
]


@pytest.mark.parametrize("w,n_sel,fwd,fwd_bwd", COUNTS, ids=[c[0].name for c in COUNTS])
def test_selected_pairs_and_flops(w, n_sel, fwd, fwd_bwd):
    assert bench.n_selected(w) == n_sel
    f = bench.counted_flops(w)
    assert f["index"] + f["fwd"] == pytest.approx(fwd, rel=6e-3)
    assert f["total"] == pytest.approx(fwd_bwd, rel=6e-3)


def test_selected_pairs_equal_a_direct_count():
    w = synth.T1024.with_(T=2048, k=5)
    bi = synth.synthetic_block_idx(w)
    direct = 0
    for row_t in range(w.T):
        for c in bi[0, 0, row_t]:
            if c >= 0:
                direct += min(w.Bk, row_t - c * w.Bk + 1)
    assert direct == bench.n_selected(w)


def test_algorithmic_bytes_are_the_entry_points_tensor_sizes():
    """Each stage's algorithmic bytes = its inputs read once + its outputs
    written once, counted here from arrays of the C ABI's shapes and dtypes."""
    import numpy as np

    import bench

    for w in (synth.T1024, synth.T8192.with_(B=2, T=1024)):
        B, T, Hq, G, d, E, k = w.B, w.T, w.Hq, w.G, w.d, w.d_idx, w.k
        bf, f32, i32 = np.uint16, np.float32, np.int32
        t = dict(Q=((B, T, Hq, d), bf), K=((B, T, G, d), bf), V=((B, T, G, d), bf), O=((B, T, Hq, d), bf),
                 dO=((B, T, Hq, d), bf), q_idx=((B, T, G, E), bf), k_idx=((B, T, E), bf),
                 block_idx=((B, G, T, k), i32), LSE=((B, T, Hq), f32), dQ=((B, T, Hq, d), f32),
                 dK=((B, T, G, d), f32), dV=((B, T, G, d), f32), dq_idx=((B, T, G, E), f32),
                 dk_idx=((B, T, E), f32), KL=((B, G, T), f32))
        nb = {n: np.zeros(sh, dt).nbytes for n, (sh, dt) in t.items()}
        want = dict(
            index=nb["q_idx"] + nb["k_idx"] + nb["block_idx"],
            fwd=nb["Q"] + nb["K"] + nb["V"] + nb["block_idx"] + nb["O"] + nb["LSE"],
            bwd=sum(nb[n] for n in ("Q", "K", "V", "O", "dO", "LSE", "q_idx", "k_idx", "block_idx", "dQ", "dK",
                                    "dV", "dq_idx", "dk_idx", "KL")))
        got = bench.algorithmic_bytes(w)
        for n in want:
            assert got[n] == want[n], n
        assert got["total"] == sum(want.values())
