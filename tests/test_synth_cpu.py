"""The seeded input generator both sides of every parity check draw from.

Pinned to things outside itself: SplitMix64's published output sequence,
torch's own fp32 -> bf16 conversion, the normal distribution's symmetry and
moments, and the workload names' stated sizes. The counter-based property
(any element drawn on its own) is what lets the GPU tests and the oracle
sample rows of a 2^20-token workload independently.
"""
import numpy as np
import pytest

import synth


def test_hash_is_splitmix64_sequence():
    # SplitMix64 from state 1234567: its first five outputs, as published with the generator's
    # reference implementation. hash_at(key, i) is output i of a SplitMix64 started at state key.
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
            16408922859458223821]
    got = synth.hash_at(np.uint64(1234567), np.arange(5, dtype=np.uint64))
    assert [int(x) for x in got] == want


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 32, 200_000, dtype=np.uint64).astype(np.uint32)
    # exact ties (low 16 bits 0x8000) with even and odd kept mantissas, and values next to them
    ties = (rng.integers(0, 1 << 16, 2000, dtype=np.uint64).astype(np.uint32) << np.uint32(16)) | np.uint32(0x8000)
    bits = np.concatenate([bits, ties, ties - np.uint32(1), ties + np.uint32(1)])
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(synth.f32_to_bf16_bits(x), want)


def test_bf16_widening_is_exact():
    b = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_bits_to_f32(b)
    finite = np.isfinite(f)
    np.testing.assert_array_equal(synth.f32_to_bf16_bits(f[finite]), b[finite])
    np.testing.assert_array_equal(synth.bf16_bits_to_f64(b[finite]), f[finite].astype(np.float64))


def test_normal_table_is_symmetric_with_unit_moments():
    t = synth.NORMAL_F32.astype(np.float64)
    np.testing.assert_array_equal(t, -t[::-1])       # bin centres u and 1 - u
    assert np.all(np.diff(t) > 0)
    assert abs(t.mean()) < 1e-12
    # the bin-centre quantisation loses only the tails: the variance stays within 1e-3 of 1
    assert abs(t.var() - 1.0) < 1e-3
    # fourth moment of N(0, 1) is 3
    assert abs((t ** 4).mean() - 3.0) < 2e-2


def test_draws_are_counter_based():
    seed, tid = 20260712, synth.TID_Q
    whole = synth.normal_f32(seed, tid, 0, 5000)
    np.testing.assert_array_equal(synth.normal_f32(seed, tid, 1234, 777), whole[1234:2011])
    # the bf16 draws are the rounded fp32 draws of the same stream
    np.testing.assert_array_equal(synth.normal_bf16(seed, tid, (50, 100)).ravel(),
                                  synth.f32_to_bf16_bits(whole))
    # another tensor id or seed gives another stream
    assert not np.array_equal(synth.normal_f32(seed, synth.TID_K, 0, 5000), whole)
    assert not np.array_equal(synth.normal_f32(seed + 1, tid, 0, 5000), whole)


def test_chunked_draws_equal_one_pass():
    n = 4 * (1 << 20) + 12345     # above the threaded path's threshold
    seed, tid = 7, synth.TID_V
    a = synth.normal_f32(seed, tid, 0, n)
    np.testing.assert_array_equal(a[-1000:], synth.normal_f32(seed, tid, n - 1000, 1000))
    np.testing.assert_array_equal(a[(1 << 20) - 3:(1 << 20) + 3], synth.normal_f32(seed, tid, (1 << 20) - 3, 6))


def test_draw_moments():
    x = synth.normal_f32(11, synth.TID_DO, 0, 1 << 20).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.var() - 1.0) < 5e-3


def test_index_keys_carry_a_per_block_mean():
    w = synth.T1024.with_(T=128 * 64, name="k_idx_recipe")
    k = synth.bf16_bits_to_f64(synth.k_idx_bf16(w))[0]            # [T, d_idx]
    m = synth.normal_f32(w.seed, synth.TID_KMEAN, 0, w.n_blocks * w.d_idx).reshape(w.n_blocks, w.d_idx)
    z = synth.normal_f32(w.seed, synth.TID_KIDX, 0, w.T * w.d_idx).reshape(w.T, w.d_idx)
    # summed in fp32 and rounded once
    want = synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(z + np.float32(0.5) * m[np.arange(w.T) // w.Bk]))
    np.testing.assert_array_equal(k, want)
    # the block means of k_idx recover 0.5 m up to the N(0, 1/128) noise of a 128-token mean
    blk = k.reshape(w.n_blocks, w.Bk, w.d_idx).mean(axis=1)
    assert np.corrcoef(blk.ravel(), m.ravel())[0, 1] > 0.7
    assert abs(np.std(blk - 0.5 * m) - 1 / np.sqrt(w.Bk)) < 0.02


@pytest.mark.parametrize("w", [synth.T1024, synth.T8192, synth.B4_T8192, synth.T131072, synth.T1048576],
                         ids=lambda w: w.name)
def test_workload_names_state_their_sizes(w):
    assert w.name == f"msa_b{w.B}_t{w.T}_hq{w.Hq}_g{w.G}_k{w.k}"
    assert (w.d, w.d_idx, w.Bk) == (128, 64, 128)
    assert w.Hq % w.G == 0 and w.T % w.Bk == 0
    assert w.seed == synth.SEED_BASE + list(synth.CONFIGS.values()).index(w)
