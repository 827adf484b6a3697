"""Shared test helpers: moving seeded inputs to the GPU and comparing results."""
import numpy as np

import synth


def to_dev(x, dtype="bf16"):
    """uint16 bf16 bit patterns (numpy) -> torch CUDA tensor of the same bits."""
    import torch

    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def to_f64(t):
    """torch tensor (bf16/fp32, any device) -> float64 numpy."""
    import torch

    return t.detach().to(torch.float64).cpu().numpy()


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


def assert_close(name, got, want, max_abs=2e-2, min_cos=0.999):
    """The parity bar for bf16 inputs with fp32 accumulation: max |err| <= 2e-2 and cosine >= 0.999."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = float(np.max(np.abs(got - want))) if got.size else 0.0
    cos = cosine(got, want)
    assert err <= max_abs, f"{name}: max abs err {err:.3e} > {max_abs}"
    assert cos >= min_cos, f"{name}: cosine {cos:.6f} < {min_cos}"
    return err, cos


def assert_kl_sum(got, want, rtol=1e-3):
    """Sum of the per-row KL over the compared rows, to a relative error of rtol
    (the per-row bound above is absolute; this one catches a small bias that
    every row shares, e.g. a dropped term or a wrong logarithm base)."""
    sg = float(np.sum(np.asarray(got, np.float64)))
    sw = float(np.sum(np.asarray(want, np.float64)))
    rel = abs(sg - sw) / max(abs(sw), 1e-30)
    assert rel <= rtol, f"sum of KL {sg:.9g} against {sw:.9g}: relative error {rel:.3e} > {rtol}"
    return rel


def compare_block_idx(got, want, gap, tie_eps=1e-4):
    """Bit-exact block ids, except rows whose oracle k-th/(k+1)-th gap < tie_eps.

    Returns (n_rows, n_near_ties, n_mismatch_outside_ties, n_mismatch_in_ties).
    """
    got = np.asarray(got).reshape(-1, got.shape[-1])
    want = np.asarray(want).reshape(-1, want.shape[-1])
    gap = np.asarray(gap).reshape(-1)
    diff = np.any(got != want, axis=1)
    tie = gap < tie_eps
    return int(got.shape[0]), int(tie.sum()), int((diff & ~tie).sum()), int((diff & tie).sum())


def valid_selection(bi, T, Bk):
    """Structural validity of block_idx rows: own block, ascending, unique, -1 padded."""
    B, G, TT, k = bi.shape
    t = np.arange(TT)
    own = t // Bk
    for row_b in range(B):
        for g in range(G):
            rows = bi[row_b, g]
            valid = rows >= 0
            nval = valid.sum(axis=1)
            assert np.all(nval == np.minimum(k, own + 1)), "wrong number of selected blocks"
            # padding at the end
            assert np.all(valid[:, :-1] >= valid[:, 1:]), "padding not at the end"
            last = rows[np.arange(TT), nval - 1]
            assert np.all(last == own), "own block missing"
            vv = np.where(valid, rows, np.iinfo(np.int32).max)
            assert np.all(np.diff(vv, axis=1)[valid[:, 1:]] > 0), "ids not strictly ascending"
