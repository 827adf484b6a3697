"""Pins of the oracle's FP8 (E4M3) index inputs, checked against things other than itself.

- Rounding: every finite E4M3 value, decoded here by hand from its 8 bits,
  rounds to itself; midpoints go to the neighbour with the even mantissa;
  and random fp32 values agree with PyTorch's float8_e4m3fn conversion
  inside the finite range (PyTorch is a library routine, not this code).
- Saturation at +-448 (the format has no infinities).
- Quantization: each q_idx row and each k_idx block reaches +-448 at its
  largest magnitude, and values times scales stay within E4M3's relative
  spacing of the inputs.
- Special case: inputs already on the E4M3 grid with a largest magnitude of
  exactly 448 per row and per block quantize to themselves with scale 1, so
  the FP8 selection equals the (separately pinned) bf16 selection.
"""
import numpy as np
import pytest

import oracle
import synth


def _e4m3_table():
    vals = []
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp = (code >> 3) & 0xF
        man = code & 0x7
        if exp == 0xF and man == 0x7:
            continue  # NaN
        if exp == 0:
            v = man / 8.0 * 2.0 ** -6
        else:
            v = (1.0 + man / 8.0) * 2.0 ** (exp - 7)
        vals.append((sign * v, code))
    return vals


def test_every_finite_e4m3_value_rounds_to_itself():
    vals = np.array([v for v, _ in _e4m3_table()])
    assert np.array_equal(oracle.e4m3(vals), vals)
    assert vals.max() == 448.0 and np.sort(np.abs(vals))[2] == 2.0 ** -9


def test_midpoints_round_to_even_mantissa():
    pos = sorted({v for v, c in _e4m3_table() if v >= 0})
    code = {v: c for v, c in _e4m3_table() if v >= 0 and not (v == 0 and c & 0x80)}
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    got = oracle.e4m3(np.array(mids))
    for (a, b), m, r in zip(zip(pos[:-1], pos[1:]), mids, got):
        want = a if code[a] % 2 == 0 else b
        assert r == want, (m, r, want)


def test_saturation():
    x = np.array([448.0, 449.0, 464.0, 500.0, 1e6, -500.0, -1e30])
    assert np.array_equal(oracle.e4m3(x), np.array([448.0, 448.0, 448.0, 448.0, 448.0, -448.0, -448.0]))


def test_rounding_agrees_with_torch_float8():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1, 20000) * 2.0 ** rng.integers(-12, 8, 20000),
                        rng.uniform(-2.0 ** -6, 2.0 ** -6, 5000)]).astype(np.float32)
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3(x.astype(np.float64)), ref)


def test_quantization_reaches_full_range_and_stays_close():
    w = synth.T1024.with_(T=512)
    inp = synth.make_inputs(w, which=("q_idx", "k_idx"))
    s = oracle.shape_of(w)
    q_deq, k_deq, sq, sk = oracle.quantize_fp8(s, inp["q_idx"], inp["k_idx"])
    q = synth.bf16_bits_to_f64(inp["q_idx"])
    k = synth.bf16_bits_to_f64(inp["k_idx"])
    # largest magnitude of each row / block lands on +-448 in E4M3 units
    q8 = q_deq / sq[..., None].astype(np.float64)
    assert np.allclose(np.abs(q8).max(axis=-1), 448.0)
    kb = k.reshape(w.B, w.n_blocks, w.Bk, w.d_idx)
    k8 = k_deq.reshape(kb.shape) / sk[:, :, None, None].astype(np.float64)
    assert np.allclose(np.abs(k8).max(axis=(-1, -2)), 448.0)
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 above the subnormals
    big = np.abs(q8) >= 2.0 ** -6
    assert np.all(np.abs(q_deq - q)[big] <= 2.0 ** -4 * np.abs(q)[big] * 1.001)


def test_fp8_selection_equals_bf16_selection_on_the_e4m3_grid():
    w = synth.T1024.with_(T=768, k=3)
    rng = np.random.default_rng(11)
    grid = np.array(sorted(v for v, _ in _e4m3_table() if 0.25 <= abs(v) <= 448))
    q = rng.choice(grid, size=(w.B, w.T, w.G, w.d_idx))
    k = rng.choice(grid, size=(w.B, w.T, w.d_idx))
    q[..., 0] = 448.0  # every row and every block reaches 448 exactly: scale 1
    k[:, ::w.Bk, 0] = 448.0
    qb, kb = synth.f32_to_bf16_bits(q.astype(np.float32)), synth.f32_to_bf16_bits(k.astype(np.float32))
    s = oracle.shape_of(w)
    q_deq, k_deq, sq, sk = oracle.quantize_fp8(s, qb, kb)
    assert np.all(sq == 1.0) and np.all(sk == 1.0)
    assert np.array_equal(q_deq, q) and np.array_equal(k_deq, k)
    bi8, _, _ = oracle.index_topk_fp8(s, qb, kb)
    bi16, _, _ = oracle.index_topk(s, qb, kb)
    assert np.array_equal(bi8, bi16)


def test_all_zero_row_and_block_quantize_with_scale_one_and_tie_to_lowest_blocks():
    # amax = 0: scale 1 and zero codes; a zero query row scores 0 against every
    # block, so the tie rule alone decides: the own block plus the lowest ids
    w = synth.T1024.with_(T=1024, k=4)
    inp = synth.make_inputs(w, which=("q_idx", "k_idx"))
    q = inp["q_idx"].copy()
    k = inp["k_idx"].copy()
    q[0, 700, 1] = 0  # bf16 +0 bits
    k[0, 256:384] = 0  # key block 2
    s = oracle.shape_of(w)
    q_deq, k_deq, sq, sk = oracle.quantize_fp8(s, q, k)
    assert sq[0, 700, 1] == 1.0 and np.all(q_deq[0, 700, 1] == 0.0)
    assert sk[0, 2] == 1.0 and np.all(k_deq[0, 256:384] == 0.0)
    bi, gap, _ = oracle.index_topk_fp8(s, q, k)
    row = bi.reshape(w.B, w.G, w.T, w.k)[0, 1, 700]
    assert row.tolist() == [0, 1, 2, 700 // w.Bk]
    assert gap.reshape(w.B, w.G, w.T)[0, 1, 700] == 0.0
