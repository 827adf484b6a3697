"""The bench's counted work (selected pairs and FLOPs) against the workload
table the configurations were specified with, and against a direct count on
a selection generated for a small shape."""
import pytest

import bench
import synth

# selected, causally visible (query, key) pairs per (b, g) for the five workloads
N_SEL = {0: 360_960, 1: 14_290_944, 2: 14_290_944, 3: 258_146_304, 4: 2_078_932_992}
# forward (index + main) and forward+backward FLOPs, to the table's precision
FWD = {0: 1.61e9, 1: 2.69e11, 2: 1.07e12, 3: 1.30e13, 4: 2.99e14}
FWD_BWD = {0: 5.59e9, 1: 8.98e11, 2: 3.59e12, 3: 2.44e13, 4: 3.44e14}


@pytest.mark.parametrize("cfg", range(5))
def test_selected_pairs_and_flops(cfg):
    w = synth.CONFIGS[cfg]
    assert bench.n_selected(w) == N_SEL[cfg]
    f = bench.counted_flops(w)
    assert f["index"] + f["fwd"] == pytest.approx(FWD[cfg], rel=6e-3)
    assert f["total"] == pytest.approx(FWD_BWD[cfg], rel=6e-3)


def test_selected_pairs_equal_a_direct_count():
    w = synth.CONFIGS[0].with_(T=2048, k=5)
    bi = synth.synthetic_block_idx(w)
    direct = 0
    for row_t in range(w.T):
        for c in bi[0, 0, row_t]:
            if c >= 0:
                direct += min(w.Bk, row_t - c * w.Bk + 1)
    assert direct == bench.n_selected(w)


def test_forward_algorithmic_bytes_closed_form():
    import bench

    for w in (synth.CONFIGS[1], synth.CONFIGS[3], synth.CONFIGS[0].with_(T=640, k=8)):
        n, k, hg = w.n_blocks, w.k, w.Hq // w.G
        # queries of block c keep min(k, c + 1) blocks: k(k+1)/2 + (n - k) k pairs per query row of a block when n >= k
        per = k * (k + 1) // 2 + (n - k) * k if n >= k else n * (n + 1) // 2
        pairs = w.Bk * per * w.B * w.G
        assert bench.fwd_algorithmic_bytes(w) == pairs * hg * (2 * w.d * 2 + 4)
