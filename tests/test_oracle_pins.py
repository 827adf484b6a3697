"""Pins of the fp64 CPU oracle to things other than itself.

Each check is an independent formulation: hand-worked fixtures, brute force,
the dense-attention special case, the blockwise online-softmax recurrence,
finite differences, and closed-form special cases. A plausible slip in the
oracle (a dropped term, a wrong sign or index, a transposed operand, a wrong
tie rule) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(T=64, Bk=8, Hq=4, G=2, d=8, d_idx=4, k=3, B=2, seed=7):
    return synth.Workload("tiny", B=B, T=T, Hq=Hq, G=G, d=d, d_idx=d_idx, Bk=Bk, k=k, seed=seed)


def _f64(x):
    return synth.bf16_bits_to_f64(x)


# ------------------------------------------------------------------ top-k
def test_topk_handworked_fixture():
    g = json.load(open(os.path.join(GOLDEN, "topk_handworked.json")))
    q = np.array(g["q_idx"], dtype=np.float64)[None, :, None, :]  # [B,T,G,E]
    kk = np.array(g["k_idx"], dtype=np.float64)[None, :, :]  # [B,T,E]
    T, E = q.shape[1], q.shape[3]
    for case in g["cases"]:
        s = oracle.shape(1, T, 1, 1, 2, E, g["Bk"], case["k"], scale=1.0, scale_idx=1.0)
        bi, gap, pool = oracle.index_topk(s, q, kk, want_pool=True)
        assert bi.tolist() == case["block_idx"]
        want_gap = np.array([np.inf if x is None else x for x in case["gap"]])
        np.testing.assert_array_equal(gap, want_gap)
        want_pool = np.array([[-np.inf if x is None else x for x in r] for r in g["pool"]])
        np.testing.assert_array_equal(pool, want_pool)


def _dense_pool_np(w, q_idx, k_idx, scale_idx):
    """Independent pooled scores: full score matrix with numpy, causal -inf, reshape-max."""
    q = _f64(q_idx)  # [B,T,G,E]
    kk = _f64(k_idx)  # [B,T,E]
    S = scale_idx * np.einsum("btge,bje->bgtj", q, kk)
    T, Bk = w.T, w.Bk
    nb = w.n_blocks
    causal = np.arange(T)[None, :] <= np.arange(T)[:, None]
    S = np.where(causal[None, None], S, -np.inf)
    pad = nb * Bk - T
    if pad:
        S = np.concatenate([S, np.full(S.shape[:-1] + (pad,), -np.inf)], axis=-1)
    return S.reshape(S.shape[:-1] + (nb, Bk)).max(axis=-1)  # [B,G,T,nb]


@pytest.mark.parametrize("T,Bk,k", [(64, 8, 3), (60, 8, 4), (48, 8, 1), (40, 8, 6)])
def test_topk_brute_force(T, Bk, k):
    w = _small(T=T, Bk=Bk, k=k)
    inp = synth.make_inputs(w, ("q_idx", "k_idx"))
    s = oracle.shape_of(w)
    bi, gap, pool = oracle.full_topk(s, inp["q_idx"], inp["k_idx"], want_pool=True)
    ref_pool = _dense_pool_np(w, inp["q_idx"], inp["k_idx"], s.scale_idx)
    np.testing.assert_allclose(pool, ref_pool, rtol=0, atol=1e-12)
    for b, g, t in itertools.product(range(w.B), range(w.G), range(T)):
        own = t // Bk
        cands = list(range(own))
        m = min(k - 1, own)
        best = None
        for sub in itertools.combinations(cands, m):
            # rank subsets by their descending score vector, ties to lower ids
            key = sorted((-ref_pool[b, g, t, c], c) for c in sub)
            if best is None or key < best[0]:
                best = (key, sub)
        want = sorted(list(best[1]) + [own])
        want += [-1] * (k - len(want))
        assert bi[b, g, t].tolist() == want, (b, g, t)
        if k >= 2 and own >= k:
            order = sorted(cands, key=lambda c: (-ref_pool[b, g, t, c], c))
            assert gap[b, g, t] == pytest.approx(
                ref_pool[b, g, t, order[k - 2]] - ref_pool[b, g, t, order[k - 1]], abs=1e-12)
        else:
            assert gap[b, g, t] == np.inf


def test_topk_invariants():
    w = _small(T=96, Bk=8, k=5, G=3, Hq=6)
    inp = synth.make_inputs(w, ("q_idx", "k_idx"))
    bi, _, _ = oracle.full_topk(oracle.shape_of(w), inp["q_idx"], inp["k_idx"])
    for b, g, t in itertools.product(range(w.B), range(w.G), range(w.T)):
        row = bi[b, g, t]
        own = t // w.Bk
        valid = row[row >= 0]
        assert own in valid
        assert np.all(np.diff(valid) > 0) and valid.max() == own
        assert (row == -1).sum() == max(0, w.k - own - 1)
        assert np.all(row[: len(valid)] == valid)  # padding at the end


def test_topk_constructed_ties_pick_lowest_block():
    # key blocks 1, 2 and 4 are exact copies: equal pooled scores for every query
    w = _small(T=64, Bk=8, k=3, B=1, G=1, Hq=1)
    inp = synth.make_inputs(w, ("q_idx", "k_idx"))
    kk = _f64(inp["k_idx"]).copy()
    kk[:, 8:16] = kk[:, 32:40] = kk[:, 16:24]
    kk[:, 0:8] = -50.0  # block 0 never wins
    kk[:, 24:32] = -50.0
    q = np.abs(_f64(inp["q_idx"]))
    s = oracle.shape_of(w)
    bi, gap, _ = oracle.index_topk(s, q, kk)
    bi = bi.reshape(w.T, w.k)
    for t in range(40, 64):  # own block >= 5: candidates 0..own-1 include 1, 2, 4
        own = t // 8
        # the two slots go to the tied copies with the lowest indices, 1 and 2
        pools = {c: np.max(q[0, t, 0] @ kk[0, c * 8:(c + 1) * 8].T) for c in range(own)}
        if max(pools.values()) == pools[1]:
            assert bi[t].tolist() == [1, 2, own], t


def _tied_closed_form(w, q_idx, k_idx):
    """Selection for tied_index_inputs by the tie rule alone: every earlier block c
    scores a_c * (q . u) / sqrt(d_idx); order by (score desc, block asc)."""
    q = _f64(q_idx)
    kk = _f64(k_idx)
    u = kk[0, 0] / (kk[0, 0, 0])          # the shared vector (u[0] == 1)
    a = kk[:, ::w.Bk, 0]                  # a_c per (b, block)
    out = np.full((w.B, w.G, w.T, w.k), -1, dtype=np.int32)
    for b in range(w.B):
        for g in range(w.G):
            s0 = q[b, :, g] @ u
            for t in range(w.T):
                own = t // w.Bk
                cand = sorted(range(own), key=lambda c: (-a[b, c] * s0[t], c))[: min(w.k - 1, own)]
                sel = sorted(cand + [own])
                out[b, g, t, : len(sel)] = sel
    return out


@pytest.mark.parametrize("k", [2, 4, 7])
def test_topk_exact_tie_levels_match_tie_rule(k):
    # many exact ties at every rank, including larger values arriving after runs of equal ones
    w = synth.T1024.with_(T=1024, G=2, Hq=2, k=k, name="tied")
    q_idx, k_idx = synth.tied_index_inputs(w)
    bi, gap, _ = oracle.full_topk(oracle.shape_of(w), q_idx, k_idx)
    assert np.array_equal(bi, _tied_closed_form(w, q_idx, k_idx))
    assert (gap[..., 3 * w.Bk:] == 0).mean() > 0.1  # many rows have a tie at the k-boundary


@pytest.mark.parametrize("selection", ["all_blocks", "none"])
def test_warmup_selection_is_dense_causal_attention_with_dense_teacher_kl(selection):
    """Indexer warmup (full attention while the indexer learns): with every
    visible block selected -- listed in block_idx, or with no block_idx at all
    (the oracle's full-attention form) -- the oracle's forward, backward and KL
    equal torch autograd (fp64) of the dense formulation: causal softmax
    attention, and the KL of the index softmax against the detached head mean
    of the attention weights, both over all visible tokens. T = 60 leaves the
    last block partial."""
    torch = pytest.importorskip("torch")
    w = _small(T=60, Bk=8, Hq=4, G=2, d=8, d_idx=4, k=8, B=2)  # k = ceil(T / Bk)
    inp = synth.make_inputs(w)
    s = oracle.shape_of(w, kl_weight=0.7)
    bi, _, _ = oracle.full_topk(s, inp["q_idx"], inp["k_idx"])
    t = np.arange(w.T)
    want_sel = np.where(np.arange(w.k)[None, :] <= (t // w.Bk)[:, None], np.arange(w.k)[None, :], -1)
    assert np.array_equal(bi.reshape(w.B, w.G, w.T, w.k), np.broadcast_to(want_sel, (w.B, w.G, w.T, w.k)))
    if selection == "none":
        bi = None
    names = ("Q", "K", "V", "dO", "q_idx", "k_idx")
    O_ref, LSE_ref = oracle.sparse_fwd(s, inp["Q"], inp["K"], inp["V"], bi)
    ref = oracle.full_bwd(s, *[inp[n] for n in names], bi)

    x = {n: torch.tensor(_f64(inp[n]), requires_grad=n != "dO") for n in names}
    hg = w.Hq // w.G
    mask = torch.tril(torch.ones(w.T, w.T, dtype=torch.bool))
    Kh = x["K"].repeat_interleave(hg, dim=2)
    Vh = x["V"].repeat_interleave(hg, dim=2)
    S = torch.einsum("bthd,bshd->bhts", x["Q"], Kh) / math.sqrt(w.d)
    S = S.masked_fill(~mask, -math.inf)
    P = torch.softmax(S, dim=-1)
    O = torch.einsum("bhts,bshd->bthd", P, Vh)
    LSE = torch.logsumexp(S, dim=-1).permute(0, 2, 1)
    Spx = torch.einsum("btge,bse->bgts", x["q_idx"], x["k_idx"]) / math.sqrt(w.d_idx)
    logp_px = torch.log_softmax(Spx.masked_fill(~mask, -math.inf), dim=-1)
    p_main = P.detach().reshape(w.B, w.G, hg, w.T, w.T).mean(dim=2)
    term = torch.where(mask, p_main * (torch.log(torch.where(mask, p_main, 1.0)) - torch.where(mask, logp_px, 0.0)),
                       0.0)
    KL = term.sum(dim=-1)
    ((O * x["dO"]).sum() + 0.7 * KL.sum()).backward()

    np.testing.assert_allclose(O_ref.reshape(O.shape), O.detach().numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(LSE_ref.reshape(LSE.shape), LSE.detach().numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(ref["KL"].reshape(KL.shape), KL.detach().numpy(), rtol=1e-9, atol=1e-11)
    for name, grad in (("dQ", x["Q"].grad), ("dK", x["K"].grad), ("dV", x["V"].grad),
                       ("dq_idx", x["q_idx"].grad), ("dk_idx", x["k_idx"].grad)):
        np.testing.assert_allclose(ref[name].reshape(grad.shape), grad.numpy(), rtol=1e-8, atol=1e-10, err_msg=name)


# ------------------------------------------------------------------ forward
def test_fwd_handworked_fixture():
    g = json.load(open(os.path.join(GOLDEN, "fwd_handworked.json")))
    Q = np.array(g["Q"], dtype=np.float64)[None, :, None, :]
    K = np.array(g["K"], dtype=np.float64)[None, :, None, :]
    V = np.array(g["V"], dtype=np.float64)[None, :, None, :]
    bi = np.array(g["block_idx"], dtype=np.int32)[None, None]
    s = oracle.shape(1, 4, 1, 1, 2, 2, 2, 1, scale=1.0)
    O, LSE = oracle.full_fwd(s, Q, K, V, bi)
    np.testing.assert_allclose(O[0, :, 0], np.array(g["O"], dtype=float), atol=1e-15)
    ln2 = math.log(2.0)
    want = {"0": 0.0, "ln2": ln2, "2": 2.0, "1+ln2": 1.0 + ln2}
    np.testing.assert_allclose(LSE[0, :, 0], [want[x] for x in g["LSE"]], atol=1e-15)


def _dense_attention_np(Q, K, V, allowed, scale):
    """Textbook masked softmax attention: allowed [B,G,T,T] bool, GQA heads."""
    B, T, Hq, d = Q.shape
    G = K.shape[2]
    hg = Hq // G
    O = np.zeros((B, T, Hq, d))
    L = np.zeros((B, T, Hq))
    for h in range(Hq):
        g = h // hg
        S = scale * np.einsum("btd,bjd->btj", Q[:, :, h], K[:, :, g])
        S = np.where(allowed[:, g], S, -np.inf)
        m = S.max(axis=-1, keepdims=True)
        E = np.exp(S - m)
        Z = E.sum(-1, keepdims=True)
        O[:, :, h] = np.einsum("btj,bjd->btd", E / Z, V[:, :, g])
        L[:, :, h] = (m + np.log(Z))[..., 0]
    return O, L


def test_fwd_equals_dense_causal_when_all_blocks_selected():
    w = _small(T=40, Bk=8, k=6)  # k >= number of blocks (5)
    inp = synth.make_inputs(w, ("Q", "K", "V", "q_idx", "k_idx"))
    s = oracle.shape_of(w)
    bi, _, _ = oracle.full_topk(s, inp["q_idx"], inp["k_idx"])
    O, LSE = oracle.full_fwd(s, inp["Q"], inp["K"], inp["V"], bi)
    causal = np.tril(np.ones((w.T, w.T), bool))
    allowed = np.broadcast_to(causal, (w.B, w.G, w.T, w.T))
    O2, L2 = _dense_attention_np(_f64(inp["Q"]), _f64(inp["K"]), _f64(inp["V"]), allowed, s.scale)
    np.testing.assert_allclose(O, O2, atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, L2, atol=1e-12, rtol=0)


def test_fwd_equals_masked_dense_for_sparse_selection():
    w = _small(T=64, Bk=8, k=3)
    inp = synth.make_inputs(w, ("Q", "K", "V", "q_idx", "k_idx"))
    s = oracle.shape_of(w)
    bi, _, _ = oracle.full_topk(s, inp["q_idx"], inp["k_idx"])
    allowed = np.zeros((w.B, w.G, w.T, w.T), bool)
    for b, g, t in itertools.product(range(w.B), range(w.G), range(w.T)):
        for c in bi[b, g, t]:
            if c >= 0:
                allowed[b, g, t, c * w.Bk:(c + 1) * w.Bk] = True
    allowed &= np.tril(np.ones((w.T, w.T), bool))[None, None]
    O, LSE = oracle.full_fwd(s, inp["Q"], inp["K"], inp["V"], bi)
    O2, L2 = _dense_attention_np(_f64(inp["Q"]), _f64(inp["K"]), _f64(inp["V"]), allowed, s.scale)
    np.testing.assert_allclose(O, O2, atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, L2, atol=1e-12, rtol=0)


def test_fwd_matches_online_softmax_recurrence():
    """The blockwise (m, l, a) merge, block by block, gives the oracle's O and LSE."""
    w = _small(T=64, Bk=8, k=4, B=1)
    inp = synth.make_inputs(w, ("Q", "K", "V", "q_idx", "k_idx"))
    s = oracle.shape_of(w)
    bi, _, _ = oracle.full_topk(s, inp["q_idx"], inp["k_idx"])
    O, LSE = oracle.full_fwd(s, inp["Q"], inp["K"], inp["V"], bi)
    Q, K, V = _f64(inp["Q"]), _f64(inp["K"]), _f64(inp["V"])
    hg = w.Hq // w.G
    for t in range(w.T):
        for h in range(w.Hq):
            g = h // hg
            m, l, a = -np.inf, 0.0, np.zeros(w.d)
            for c in bi[0, g, t]:
                if c < 0:
                    continue
                j = np.arange(c * w.Bk, min((c + 1) * w.Bk, t + 1))
                sb = s.scale * K[0, j, g] @ Q[0, t, h]
                m_new = max(m, sb.max())
                alpha = math.exp(m - m_new) if m > -np.inf else 0.0
                p = np.exp(sb - m_new)
                l = alpha * l + p.sum()
                a = alpha * a + p @ V[0, j, g]
                m = m_new
            np.testing.assert_allclose(O[0, t, h], a / l, atol=1e-12, rtol=0)
            assert LSE[0, t, h] == pytest.approx(m + math.log(l), abs=1e-12)


# ------------------------------------------------------------------ backward
def _fd_setup(seed=3, k=3):
    w = _small(T=32, Bk=8, k=k, B=1, Hq=4, G=2, d=6, d_idx=5, seed=seed)
    inp = synth.make_inputs(w)
    s = oracle.shape_of(w)
    bi, _, _ = oracle.full_topk(s, inp["q_idx"], inp["k_idx"])
    x = {n: _f64(v).copy() for n, v in inp.items()}
    return w, s, bi, x


def _loss_main(s, x, bi):
    O, _ = oracle.full_fwd(s, x["Q"], x["K"], x["V"], bi)
    return float(np.sum(O * x["dO"]))


def _loss_kl(s, x, bi):
    _, _, KL = oracle.bwd_rows(s, x["Q"], x["K"], x["V"], x["dO"], x["q_idx"], x["k_idx"], bi)
    return float(KL.sum())


@pytest.mark.parametrize("name,out", [("Q", "dQ"), ("K", "dK"), ("V", "dV")])
def test_main_backward_finite_differences(name, out):
    w, s, bi, x = _fd_setup()
    g = oracle.full_bwd(s, x["Q"], x["K"], x["V"], x["dO"], x["q_idx"], x["k_idx"], bi)[out]
    rng = np.random.default_rng(11)
    h = 1e-5
    for _ in range(12):
        idx = tuple(rng.integers(0, n) for n in x[name].shape)
        xp = {k: v.copy() for k, v in x.items()}
        xm = {k: v.copy() for k, v in x.items()}
        xp[name][idx] += h
        xm[name][idx] -= h
        fd = (_loss_main(s, xp, bi) - _loss_main(s, xm, bi)) / (2 * h)
        assert g[idx] == pytest.approx(fd, rel=1e-6, abs=1e-9), (name, idx)


@pytest.mark.parametrize("name,out", [("q_idx", "dq_idx"), ("k_idx", "dk_idx")])
def test_kl_gradient_finite_differences(name, out):
    w, s, bi, x = _fd_setup(seed=5)
    g = oracle.full_bwd(s, x["Q"], x["K"], x["V"], x["dO"], x["q_idx"], x["k_idx"], bi)[out]
    rng = np.random.default_rng(12)
    h = 1e-5
    for _ in range(12):
        idx = tuple(rng.integers(0, n) for n in x[name].shape)
        xp = {k: v.copy() for k, v in x.items()}
        xm = {k: v.copy() for k, v in x.items()}
        xp[name][idx] += h
        xm[name][idx] -= h
        fd = (_loss_kl(s, xp, bi) - _loss_kl(s, xm, bi)) / (2 * h)
        assert g[idx] == pytest.approx(fd, rel=1e-6, abs=1e-9), (name, idx)


def test_kl_closed_form_score_gradient():
    """d KL(p_main || softmax(s)) / d s = softmax(s) - p_main, by finite differences."""
    rng = np.random.default_rng(1)
    for n in (1, 2, 7, 40):
        pm = rng.random(n)
        pm[rng.random(n) < 0.2] = 0.0
        if pm.sum() == 0:
            pm[0] = 1.0
        pm /= pm.sum()
        s = rng.normal(size=n)

        def kl(sv):
            lse = np.log(np.sum(np.exp(sv - sv.max()))) + sv.max()
            nz = pm > 0
            return float(np.sum(pm[nz] * (np.log(pm[nz]) - (sv[nz] - lse))))

        p = np.exp(s - s.max())
        p /= p.sum()
        for i in range(n):
            e = np.zeros(n)
            e[i] = 1e-6
            fd = (kl(s + e) - kl(s - e)) / 2e-6
            assert p[i] - pm[i] == pytest.approx(fd, abs=1e-8)


def test_kl_nonnegative_and_detached():
    w, s, bi, x = _fd_setup(seed=9)
    full = oracle.full_bwd(s, x["Q"], x["K"], x["V"], x["dO"], x["q_idx"], x["k_idx"], bi)
    assert np.all(full["KL"] >= -1e-14)
    # index inputs do not reach dQ/dK/dV; dO does not reach dq_idx/dk_idx
    x2 = {k: v.copy() for k, v in x.items()}
    x2["q_idx"] *= 1.7
    x2["k_idx"] += 0.3
    x2["dO"] *= -2.0
    f2 = oracle.full_bwd(s, x2["Q"], x2["K"], x2["V"], x2["dO"], x2["q_idx"], x2["k_idx"], bi)
    np.testing.assert_allclose(f2["dQ"], -2.0 * full["dQ"], atol=1e-12)
    np.testing.assert_allclose(f2["dV"], -2.0 * full["dV"], atol=1e-12)
    s3 = oracle.shape_of(w, kl_weight=0.25)
    f3 = oracle.full_bwd(s3, x["Q"], x["K"], x["V"], x["dO"], x["q_idx"], x["k_idx"], bi)
    np.testing.assert_allclose(f3["dK"], full["dK"], atol=1e-15)
    np.testing.assert_allclose(f3["dq_idx"], 0.25 * full["dq_idx"], atol=1e-15)
    np.testing.assert_allclose(f3["KL"], full["KL"], atol=1e-15)


def test_kl_vanishes_when_index_branch_equals_main_branch():
    """hg = 1, d_idx = d, q_idx = Q, k_idx = K, equal scales: p_px = p_main."""
    w = _small(T=32, Bk=8, k=2, B=1, Hq=2, G=2, d=6, d_idx=6, seed=4)
    inp = synth.make_inputs(w)
    s = oracle.shape_of(w, scale=0.37, scale_idx=0.37)
    q_idx = inp["Q"].reshape(w.B, w.T, w.G, w.d)  # hg = 1: head g is group g
    k_idx = inp["K"][:, :, 0, :]
    K = np.repeat(inp["K"][:, :, :1, :], w.G, axis=2)
    bi, _, _ = oracle.full_topk(s, q_idx, k_idx)
    f = oracle.full_bwd(s, inp["Q"], K, inp["V"], inp["dO"], q_idx, k_idx, bi)
    assert np.max(np.abs(f["KL"])) < 1e-12
    assert np.max(np.abs(f["dq_idx"])) < 1e-12
    assert np.max(np.abs(f["dk_idx"])) < 1e-12


def test_row_and_block_views_agree_with_partial_last_block():
    """The per-block backward of a sample equals the same slice of the full one."""
    w = _small(T=60, Bk=8, k=3)
    inp = synth.make_inputs(w)
    s = oracle.shape_of(w)
    bi, _, _ = oracle.full_topk(s, inp["q_idx"], inp["k_idx"])
    full = oracle.full_bwd(s, *[inp[n] for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")], bi)
    blocks = np.array([1 * w.n_blocks + 7, 0 * w.n_blocks + 2])
    dK, dV, dki = oracle.bwd_blocks(s, *[inp[n] for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")], bi,
                                    blocks=blocks)
    # block 7 of batch 1 is partial: tokens 56..59
    np.testing.assert_allclose(dK[0, :, :4].transpose(1, 0, 2), full["dK"][1, 56:60], atol=1e-15)
    np.testing.assert_allclose(dV[1, :, :].transpose(1, 0, 2), full["dV"][0, 16:24], atol=1e-15)
    np.testing.assert_allclose(dki[1], full["dk_idx"][0, 16:24], atol=1e-15)
    assert np.all(dK[0, :, 4:] == 0)


def test_block_view_group_filter_splits_the_sums():
    """Restricting the per-block backward to one group keeps that group's dK, dV
    rows, zeroes the others, and splits dk_idx into shares summing to the whole
    (with a block list and in the full-attention form)."""
    w = _small(T=64, Bk=8, Hq=6, G=3, k=3)
    inp = synth.make_inputs(w)
    s = oracle.shape_of(w)
    names = ("Q", "K", "V", "dO", "q_idx", "k_idx")
    bi, _, _ = oracle.full_topk(s, inp["q_idx"], inp["k_idx"])
    blocks = np.array([0 * w.n_blocks + 1, 1 * w.n_blocks + 5])
    for sel in (bi, None):
        dK, dV, dki = oracle.bwd_blocks(s, *[inp[n] for n in names], sel, blocks=blocks)
        share = np.zeros_like(dki)
        for g in range(w.G):
            gK, gV, gki = oracle.bwd_blocks(s, *[inp[n] for n in names], sel, blocks=blocks, group=g)
            np.testing.assert_array_equal(gK[:, g], dK[:, g])
            np.testing.assert_array_equal(gV[:, g], dV[:, g])
            assert not np.any(np.delete(gK, g, axis=1)) and not np.any(np.delete(gV, g, axis=1))
            share += gki
        np.testing.assert_allclose(share, dki, rtol=1e-12, atol=1e-15)
        assert np.abs(dki).max() > 1e-6


def test_oracle_is_independent_of_cuda_path():
    here = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for fn in os.listdir(os.path.join(here, "oracle")):
        if fn.endswith((".c", ".py", ".h")):
            src = open(os.path.join(here, "oracle", fn)).read()
            assert "block_sparse_attention_scores_gb300" not in src
            assert "csrc" not in src
    pkg = os.path.join(here, "block_sparse_attention_scores_gb300")
    for root, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(root, fn)).read()
                assert "import oracle" not in src and "from oracle" not in src, fn
                assert "msa_oracle" not in src, fn
