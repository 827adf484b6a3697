"""Seeded synthetic inputs for the MSA training hot path.

Both sides of every parity check draw their inputs from here: the fp64 CPU
oracle (``oracle/``) and the CUDA path (``block_sparse_attention_scores_gb300``).
This module holds none of the method's arithmetic. It only has

* a counter-based generator: SplitMix64's finaliser applied to
  ``key + (i + 1) * 0x9E3779B97F4A7C15``, so any element of any tensor can be
  drawn on its own, in any order, on any machine;
* a fixed 65,536-entry inverse-normal table (``ndtri`` at the bin centres), so
  that a draw is the bf16 rounding of a quantised N(0, 1) value;
* round-to-nearest-even fp32 -> bf16 rounding;
* the workload presets (shapes of the five MSA configurations).

Distributions (the MSA GQA layer workloads):

* ``Q, K, V, dO ~ N(0, 1)`` in bf16;
* ``q_idx[b, t, g, :] ~ N(0, I)`` independently per GQA group;
* ``k_idx[b, t, :] = N(0, I) + m[b, t // Bk, :]`` with a per-KV-block mean
  ``m ~ N(0, 0.5^2 I)``, summed in fp32 and rounded once to bf16.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np

SEED_BASE = 20260712

# tensor ids of the counter-based streams
TID_Q, TID_K, TID_V, TID_DO, TID_QIDX, TID_KIDX, TID_KMEAN, TID_BLOCKIDX, TID_TIES = range(1, 10)

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20


def _mix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser (wrapping uint64 arithmetic), in place on ``x``."""
    x ^= x >> np.uint64(30)
    x *= _M1
    x ^= x >> np.uint64(27)
    x *= _M2
    x ^= x >> np.uint64(31)
    return x


def stream_key(seed: int, tid: int) -> np.uint64:
    """Key of tensor stream ``tid`` under ``seed``."""
    with np.errstate(over="ignore"):
        x = np.array([(seed * 0x100000001B3 + tid * 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF],
                     dtype=np.uint64)
        return _mix64(x)[0]


def hash_at(key: np.uint64, idx: np.ndarray) -> np.ndarray:
    """64-bit hash of the elements ``idx`` (uint64) of the stream ``key``."""
    x = (idx.astype(np.uint64) + np.uint64(1)) * _GOLDEN
    x += np.uint64(key)
    return _mix64(x)


def _normal_table() -> np.ndarray:
    from scipy.special import ndtri

    u = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
    return ndtri(u).astype(np.float32)


NORMAL_F32 = _normal_table()


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16, returned as uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


def _workers() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _chunked(n: int, work) -> None:
    starts = range(0, n, _CHUNK)
    if n > 4 * _CHUNK:
        with ThreadPoolExecutor(_workers()) as ex:
            list(ex.map(work, starts))
    else:
        for lo in starts:
            work(lo)


def normal_f32(seed: int, tid: int, start: int, n: int) -> np.ndarray:
    """Quantised N(0,1) draws of elements ``[start, start + n)`` of a stream, fp32."""
    key = stream_key(seed, tid)
    out = np.empty(n, dtype=np.float32)

    def work(lo: int) -> None:
        hi = min(n, lo + _CHUNK)
        h = hash_at(key, np.arange(start + lo, start + hi, dtype=np.uint64))
        out[lo:hi] = NORMAL_F32[(h >> np.uint64(48)).astype(np.intp)]

    _chunked(n, work)
    return out


def normal_bf16(seed: int, tid: int, shape, start: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0,1) draws, shaped ``shape``."""
    n = int(np.prod(shape))
    key = stream_key(seed, tid)
    out = np.empty(n, dtype=np.uint16)

    def work(lo: int) -> None:
        hi = min(n, lo + _CHUNK)
        h = hash_at(key, np.arange(start + lo, start + hi, dtype=np.uint64))
        out[lo:hi] = f32_to_bf16_bits(NORMAL_F32[(h >> np.uint64(48)).astype(np.intp)])

    _chunked(n, work)
    return out.reshape(shape)


# --------------------------------------------------------------------------- workloads
@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hq: int
    G: int
    d: int = 128
    d_idx: int = 64
    Bk: int = 128
    k: int = 16
    seed: int = SEED_BASE

    @property
    def n_blocks(self) -> int:
        return (self.T + self.Bk - 1) // self.Bk

    @property
    def hg(self) -> int:
        return self.Hq // self.G

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five MSA GQA-layer configurations (index dim 64, head dim 128, 128-token blocks).
CONFIGS = {
    0: Workload("msa_b1_t1024_hq8_g2_k4", B=1, T=1024, Hq=8, G=2, k=4, seed=SEED_BASE + 0),
    1: Workload("msa_b1_t8192_hq32_g8_k16", B=1, T=8192, Hq=32, G=8, seed=SEED_BASE + 1),
    2: Workload("msa_b4_t8192_hq32_g8_k16", B=4, T=8192, Hq=32, G=8, seed=SEED_BASE + 2),
    3: Workload("msa_b1_t131072_hq32_g8_k16", B=1, T=131072, Hq=32, G=8, seed=SEED_BASE + 3),
    4: Workload("msa_b1_t1048576_hq16_g4_k16", B=1, T=1048576, Hq=16, G=4, seed=SEED_BASE + 4),
}
# The same five by their sizes (the id above only fixes each one's seed).
T1024 = CONFIGS[0]      # B=1, T=1024, Hq=8, G=2, k=4
T8192 = CONFIGS[1]      # B=1, T=8192, Hq=32, G=8, k=16
B4_T8192 = CONFIGS[2]   # B=4, T=8192, Hq=32, G=8, k=16
T131072 = CONFIGS[3]    # B=1, T=131072, Hq=32, G=8, k=16
T1048576 = CONFIGS[4]   # B=1, T=1048576, Hq=16, G=4, k=16


def make_inputs(w: Workload, which=("Q", "K", "V", "dO", "q_idx", "k_idx")) -> dict:
    """All requested inputs of a workload as bf16 bit patterns (uint16 numpy arrays).

    Layouts: Q, dO [B,T,Hq,d]; K, V [B,T,G,d]; q_idx [B,T,G,d_idx]; k_idx [B,T,d_idx].
    """
    out = {}
    s = w.seed
    if "Q" in which:
        out["Q"] = normal_bf16(s, TID_Q, (w.B, w.T, w.Hq, w.d))
    if "K" in which:
        out["K"] = normal_bf16(s, TID_K, (w.B, w.T, w.G, w.d))
    if "V" in which:
        out["V"] = normal_bf16(s, TID_V, (w.B, w.T, w.G, w.d))
    if "dO" in which:
        out["dO"] = normal_bf16(s, TID_DO, (w.B, w.T, w.Hq, w.d))
    if "q_idx" in which:
        out["q_idx"] = normal_bf16(s, TID_QIDX, (w.B, w.T, w.G, w.d_idx))
    if "k_idx" in which:
        out["k_idx"] = k_idx_bf16(w)
    return out


def k_idx_bf16(w: Workload) -> np.ndarray:
    """Index keys with a per-KV-block mean offset: bf16(z + 0.5 * m[block])."""
    z = normal_f32(w.seed, TID_KIDX, 0, w.B * w.T * w.d_idx).reshape(w.B, w.T, w.d_idx)
    m = normal_f32(w.seed, TID_KMEAN, 0, w.B * w.n_blocks * w.d_idx).reshape(w.B, w.n_blocks, w.d_idx)
    blk = np.arange(w.T) // w.Bk
    x = z + np.float32(0.5) * m[:, blk, :]
    return f32_to_bf16_bits(x.astype(np.float32)).reshape(w.B, w.T, w.d_idx)


def tied_index_inputs(w: Workload):
    """Index inputs whose pooled block scores tie exactly, with no rounding anywhere.

    q_idx entries are multiples of 1/8 in [-2, 2]. Every key of block c is
    a_c * u, with u one shared vector of multiples of 1/8 in [-1, 1] (one entry
    exactly 1) and a_c drawn from {1, 2, 4}. All products and sums of the index
    scores are then exact in fp32 and fp64, and so are the E4M3 codes of the
    keys (the per-block scale absorbs a_c). Blocks with the same a_c thus have
    bit-identical pooled scores for every query, and distinct levels differ by a
    factor of 2. Returns (q_idx [B,T,G,d_idx], k_idx [B,T,d_idx]) as bf16 bit patterns.
    """
    key = stream_key(w.seed, TID_TIES)
    nq = w.B * w.T * w.G * w.d_idx
    hq = hash_at(key, np.arange(nq, dtype=np.uint64))
    q = ((hq % np.uint64(33)).astype(np.int64) - 16).astype(np.float32) / np.float32(8)
    hu = hash_at(key, np.arange(nq, nq + w.d_idx, dtype=np.uint64))
    u = ((hu % np.uint64(17)).astype(np.int64) - 8).astype(np.float32) / np.float32(8)
    u[0] = 1.0
    nb = w.B * w.n_blocks
    ha = hash_at(key, np.arange(nq + w.d_idx, nq + w.d_idx + nb, dtype=np.uint64))
    a = np.array([1.0, 2.0, 4.0], dtype=np.float32)[(ha % np.uint64(3)).astype(np.intp)].reshape(w.B, w.n_blocks)
    blk = np.arange(w.T) // w.Bk
    k = a[:, blk, None] * u[None, None, :]
    return (f32_to_bf16_bits(q).reshape(w.B, w.T, w.G, w.d_idx),
            f32_to_bf16_bits(k.astype(np.float32)).reshape(w.B, w.T, w.d_idx))


def synthetic_block_idx(w: Workload, seed_offset: int = 0) -> np.ndarray:
    """A structurally valid block selection drawn at random (not by any score).

    For every (b, g, t): the own block t // Bk plus min(k-1, own) distinct
    earlier blocks chosen uniformly (Floyd's sampling), ascending, -1 padded.
    Used to drive the sparse forward/backward on workloads too large for the
    dense fp64 index scores.
    """
    B, G, T, k, Bk = w.B, w.G, w.T, w.k, w.Bk
    rows = B * G * T
    own = (np.arange(rows, dtype=np.int64) % T) // Bk
    out = np.full((rows, k), -1, dtype=np.int32)
    key = stream_key(w.seed + seed_offset, TID_BLOCKIDX)
    few = own < k  # all visible blocks fit
    # rows with few blocks: 0..own
    if few.any():
        r = np.nonzero(few)[0]
        cols = np.arange(k)
        vals = np.where(cols[None, :] <= own[r, None], cols[None, :], -1)
        out[r] = vals.astype(np.int32)
    many = ~few
    if many.any():
        r = np.nonzero(many)[0]
        C = own[r]
        kk = k - 1
        chosen = np.empty((r.size, kk), dtype=np.int64)
        for i in range(kk):
            j = C - kk + i
            h = hash_at(key, r.astype(np.uint64) * np.uint64(max(64, k)) + np.uint64(i))
            cand = (h % (j + 1).astype(np.uint64)).astype(np.int64)
            dup = (chosen[:, :i] == cand[:, None]).any(axis=1) if i else np.zeros(r.size, bool)
            chosen[:, i] = np.where(dup, j, cand)
        chosen.sort(axis=1)
        out[r, :kk] = chosen.astype(np.int32)
        out[r, kk] = C.astype(np.int32)
    return out.reshape(B, G, T, k)
