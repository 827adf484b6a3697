"""Plain fp64 CPU oracle of the MSA training hot path.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package. The
CUDA path never imports it, and it imports nothing from the CUDA path.

The arithmetic lives in ``msa_oracle.c`` (plain C, double precision, OpenMP
over independent rows); this module compiles it with gcc on first use and
marshals numpy arrays. Which page passage each step follows is stated in the
C file's header and at each function.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIB = os.path.join(_HERE, "libmsa_oracle.so")
_lock = threading.Lock()
_lib = None

DT_BF16, DT_F64 = 0, 1


class OShape(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("Hq", ctypes.c_int32), ("G", ctypes.c_int32),
        ("d", ctypes.c_int32), ("d_idx", ctypes.c_int32), ("Bk", ctypes.c_int32), ("k", ctypes.c_int32),
        ("scale", ctypes.c_double), ("scale_idx", ctypes.c_double), ("kl_weight", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, OpenMP). Returns its path."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".{os.getpid()}.tmp"
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
                   "-Wno-unused-parameter", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_index_topk.argtypes = [ctypes.POINTER(OShape), P, P, ctypes.c_int, P, I64, P, P, P]
        lib.oracle_e4m3.argtypes = [ctypes.c_double]
        lib.oracle_e4m3.restype = ctypes.c_double
        lib.oracle_quantize_fp8.argtypes = [ctypes.POINTER(OShape), P, P, P, P, P, P]
        lib.oracle_sparse_fwd.argtypes = [ctypes.POINTER(OShape), P, P, P, ctypes.c_int, P, P, I64, P, P]
        lib.oracle_bwd_rows.argtypes = [ctypes.POINTER(OShape), P, P, P, P, P, P, ctypes.c_int, P, P, I64,
                                        P, P, P]
        lib.oracle_bwd_blocks.argtypes = [ctypes.POINTER(OShape), P, P, P, P, P, P, ctypes.c_int, P, P, I64,
                                          ctypes.c_int, P, P, P]
        for f in (lib.oracle_index_topk, lib.oracle_sparse_fwd, lib.oracle_bwd_rows, lib.oracle_bwd_blocks):
            f.restype = ctypes.c_int
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def shape(B, T, Hq, G, d, d_idx, Bk, k, scale=None, scale_idx=None, kl_weight=1.0) -> OShape:
    """Problem shape; scales default to 1/sqrt(d) and 1/sqrt(d_idx)."""
    return OShape(B, T, Hq, G, d, d_idx, Bk, k,
                  float(scale) if scale else 1.0 / np.sqrt(d),
                  float(scale_idx) if scale_idx else 1.0 / np.sqrt(d_idx),
                  float(kl_weight))


def shape_of(w, **kw) -> OShape:
    return shape(w.B, w.T, w.Hq, w.G, w.d, w.d_idx, w.Bk, w.k, **kw)


def _arr(x):
    """(pointer, dtype flag, keep-alive) for a bf16-bits (uint16) or float64 array."""
    if x is None:
        return None, DT_F64, None
    if x.dtype == np.uint16:
        a = np.ascontiguousarray(x)
        return a.ctypes.data, DT_BF16, a
    a = np.ascontiguousarray(x, dtype=np.float64)
    return a.ctypes.data, DT_F64, a


def _inputs(*xs):
    ptrs, keep, dts = [], [], set()
    for x in xs:
        p, dt, a = _arr(x)
        ptrs.append(p)
        keep.append(a)
        if a is not None:
            dts.add(dt)
    if len(dts) > 1:
        raise TypeError("oracle inputs must all be bf16 bits (uint16) or all float64")
    return ptrs, (dts.pop() if dts else DT_F64), keep


def _rows(rows, total):
    if rows is None:
        return None, total, None
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r.ctypes.data, r.size, r


def index_topk(s: OShape, q_idx, k_idx, rows=None, want_pool=False):
    """Steps 1-3 (index scores, block max-pool, top-k with own block forced).

    rows: ids (b*G + g)*T + t, default all. Returns (block_idx [n,k] int32,
    gap [n] float64, pool [n, n_blocks] or None).
    """
    lib = _load()
    (qp, kp), dt, keep = _inputs(q_idx, k_idx)
    rp, n, rk = _rows(rows, s.B * s.G * s.T)
    nb = (s.T + s.Bk - 1) // s.Bk
    bi = np.empty((n, s.k), dtype=np.int32)
    gap = np.empty(n, dtype=np.float64)
    pool = np.empty((n, nb), dtype=np.float64) if want_pool else None
    lib.oracle_index_topk(ctypes.byref(s), qp, kp, dt, rp, n, bi.ctypes.data, gap.ctypes.data,
                          pool.ctypes.data if pool is not None else None)
    return bi, gap, pool


def e4m3(x):
    """E4M3 (FN) rounding, ties to even, saturating at +-448, of each value of x (float64 array)."""
    lib = _load()
    x = np.asarray(x, dtype=np.float64)
    return np.array([lib.oracle_e4m3(float(v)) for v in x.ravel()], dtype=np.float64).reshape(x.shape)


def quantize_fp8(s: OShape, q_idx, k_idx):
    """FP8 index inputs: (q_deq [B,T,G,E], k_deq [B,T,E] float64 = quantized values times their scales,
    sq [B,T,G] float32, sk [B,n_blocks] float32). q_idx, k_idx are bf16 bit patterns (uint16)."""
    lib = _load()
    q = np.ascontiguousarray(q_idx, dtype=np.uint16)
    k = np.ascontiguousarray(k_idx, dtype=np.uint16)
    nb = (s.T + s.Bk - 1) // s.Bk
    q_deq = np.empty((s.B, s.T, s.G, s.d_idx), dtype=np.float64)
    k_deq = np.empty((s.B, s.T, s.d_idx), dtype=np.float64)
    sq = np.empty((s.B, s.T, s.G), dtype=np.float32)
    sk = np.empty((s.B, nb), dtype=np.float32)
    lib.oracle_quantize_fp8(ctypes.byref(s), q.ctypes.data, k.ctypes.data, q_deq.ctypes.data, k_deq.ctypes.data,
                            sq.ctypes.data, sk.ctypes.data)
    return q_deq, k_deq, sq, sk


def index_topk_fp8(s: OShape, q_idx, k_idx, rows=None, want_pool=False):
    """Steps 1-3 on the FP8 index inputs (quantize_fp8): same returns as index_topk."""
    q_deq, k_deq, _, _ = quantize_fp8(s, q_idx, k_idx)
    return index_topk(s, q_deq, k_deq, rows=rows, want_pool=want_pool)


def _selection(block_idx):
    """block_idx as int32 and its pointer; None (a NULL pointer) selects every
    causally visible token (full attention, as in the indexer warmup)."""
    if block_idx is None:
        return None, None
    bi = np.ascontiguousarray(block_idx, dtype=np.int32)
    return bi, bi.ctypes.data


def sparse_fwd(s: OShape, Q, K, V, block_idx, rows=None):
    """Steps 4-5. rows: ids (b*T + t)*Hq + h, default all. Returns (O [n,d], LSE [n]).

    block_idx None: every visible token (full causal attention)."""
    lib = _load()
    (qp, kp, vp), dt, keep = _inputs(Q, K, V)
    bi, bip = _selection(block_idx)
    rp, n, rk = _rows(rows, s.B * s.T * s.Hq)
    O = np.empty((n, s.d), dtype=np.float64)
    LSE = np.empty(n, dtype=np.float64)
    lib.oracle_sparse_fwd(ctypes.byref(s), qp, kp, vp, dt, bip, rp, n, O.ctypes.data,
                          LSE.ctypes.data)
    return O, LSE


def bwd_rows(s: OShape, Q, K, V, dO, q_idx, k_idx, block_idx, rows=None):
    """Steps 6-7, per query. rows: ids (b*G + g)*T + t, default all.

    Returns (dQ [n, hg, d], dq_idx [n, d_idx], KL [n]).
    """
    lib = _load()
    ptrs, dt, keep = _inputs(Q, K, V, dO, q_idx, k_idx)
    bi, bip = _selection(block_idx)
    rp, n, rk = _rows(rows, s.B * s.G * s.T)
    hg = s.Hq // s.G
    dQ = np.empty((n, hg, s.d), dtype=np.float64)
    dqi = np.empty((n, s.d_idx), dtype=np.float64)
    KL = np.empty(n, dtype=np.float64)
    lib.oracle_bwd_rows(ctypes.byref(s), *ptrs, dt, bip, rp, n, dQ.ctypes.data, dqi.ctypes.data,
                        KL.ctypes.data)
    return dQ, dqi, KL


def bwd_blocks(s: OShape, Q, K, V, dO, q_idx, k_idx, block_idx, blocks=None, group=None):
    """Steps 6-7, per key block. blocks: ids b*n_blocks + c, default all.
    group: only that group's queries (dK, dV of the other groups zero, dk_idx
    that group's share); default every group.

    Returns (dK [n, G, Bk, d], dV [n, G, Bk, d], dk_idx [n, Bk, d_idx]).
    """
    lib = _load()
    ptrs, dt, keep = _inputs(Q, K, V, dO, q_idx, k_idx)
    bi, bip = _selection(block_idx)
    nb = (s.T + s.Bk - 1) // s.Bk
    rp, n, rk = _rows(blocks, s.B * nb)
    dK = np.empty((n, s.G, s.Bk, s.d), dtype=np.float64)
    dV = np.empty((n, s.G, s.Bk, s.d), dtype=np.float64)
    dki = np.empty((n, s.Bk, s.d_idx), dtype=np.float64)
    lib.oracle_bwd_blocks(ctypes.byref(s), *ptrs, dt, bip, rp, n, -1 if group is None else int(group),
                          dK.ctypes.data, dV.ctypes.data, dki.ctypes.data)
    return dK, dV, dki


def full_bwd(s: OShape, Q, K, V, dO, q_idx, k_idx, block_idx):
    """Whole-tensor backward in the CUDA path's layouts (small problems only).

    Returns dict with dQ [B,T,Hq,d], dK/dV [B,T,G,d], dq_idx [B,T,G,d_idx],
    dk_idx [B,T,d_idx], KL [B,G,T].
    """
    B, T, Hq, G, d, E, Bk = s.B, s.T, s.Hq, s.G, s.d, s.d_idx, s.Bk
    hg = Hq // G
    nb = (T + Bk - 1) // Bk
    dQ, dqi, KL = bwd_rows(s, Q, K, V, dO, q_idx, k_idx, block_idx)
    dQ = dQ.reshape(B, G, T, hg, d).transpose(0, 2, 1, 3, 4).reshape(B, T, Hq, d)
    dqi = dqi.reshape(B, G, T, E).transpose(0, 2, 1, 3)
    KL = KL.reshape(B, G, T)
    dKb, dVb, dkib = bwd_blocks(s, Q, K, V, dO, q_idx, k_idx, block_idx)
    Tp = nb * Bk
    dK = dKb.reshape(B, nb, G, Bk, d).transpose(0, 1, 3, 2, 4).reshape(B, Tp, G, d)[:, :T]
    dV = dVb.reshape(B, nb, G, Bk, d).transpose(0, 1, 3, 2, 4).reshape(B, Tp, G, d)[:, :T]
    dki = dkib.reshape(B, Tp, E)[:, :T]
    return dict(dQ=dQ, dK=np.ascontiguousarray(dK), dV=np.ascontiguousarray(dV), dq_idx=np.ascontiguousarray(dqi),
                dk_idx=np.ascontiguousarray(dki), KL=KL)


def full_fwd(s: OShape, Q, K, V, block_idx):
    """Whole-tensor forward: O [B,T,Hq,d], LSE [B,T,Hq]."""
    O, LSE = sparse_fwd(s, Q, K, V, block_idx)
    return O.reshape(s.B, s.T, s.Hq, s.d), LSE.reshape(s.B, s.T, s.Hq)


def full_topk(s: OShape, q_idx, k_idx, want_pool=False):
    """Whole-tensor index top-k: block_idx [B,G,T,k], gap [B,G,T] (and pool)."""
    bi, gap, pool = index_topk(s, q_idx, k_idx, want_pool=want_pool)
    nb = (s.T + s.Bk - 1) // s.Bk
    return (bi.reshape(s.B, s.G, s.T, s.k), gap.reshape(s.B, s.G, s.T),
            pool.reshape(s.B, s.G, s.T, nb) if pool is not None else None)
