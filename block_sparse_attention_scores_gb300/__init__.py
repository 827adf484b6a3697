"""GB300-native MiniMax Sparse Attention (MSA) training hot path.

A thin ctypes binding over ``libmsa_gb300.so`` (C ABI declared in
``include/msa.h``): argument marshalling only. Every step of the path runs in
the library's sm_103a kernels; there is no CPU fallback, and importing the
binding without the compiled library raises.

Entry points (same names as the C ABI):

* ``msa_index_topk(shape, q_idx, k_idx, block_idx, workspace, stream=None)``
* ``msa_sparse_fwd(shape, Q, K, V, block_idx, O, LSE, workspace, stream=None)``
* ``msa_bwd(shape, Q, K, V, O, dO, LSE, q_idx, k_idx, block_idx, kl_weight,
  dQ, dK, dV, dq_idx, dk_idx, KL, workspace, stream=None)``
* ``msa_workspace_size(shape, which)``, ``msa_check_device_status(workspace, stream)``

Tensors are torch CUDA tensors (bf16 / int32 / fp32, contiguous, layouts as
in the header) or raw device addresses (int). ``stream`` is a
``torch.cuda.Stream``, a raw ``cudaStream_t`` (int) or ``None`` for torch's
current stream.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa_gb300.so")

MSA_OK, MSA_ERR_INVALID_ARG, MSA_ERR_UNSUPPORTED, MSA_ERR_WORKSPACE, MSA_ERR_CUDA, MSA_ERR_DEVICE = range(6)
MSA_WS_TOPK, MSA_WS_FWD, MSA_WS_BWD, MSA_WS_TOPK_FP8, MSA_WS_DENSE = 0, 1, 2, 3, 4
MSA_TIME_INDEX_TOPK, MSA_TIME_SPARSE_FWD, MSA_TIME_BWD, MSA_TIME_DENSE_FWD, MSA_TIME_DENSE_BWD = 0, 1, 2, 3, 4

EXPORTED = ("msa_workspace_size", "msa_index_topk", "msa_sparse_fwd", "msa_bwd", "msa_last_error",
            "msa_check_device_status", "msa_selftest_wait_timeout", "msa_kernel_launches", "msa_version",
            "msa_index_topk_noalloc", "msa_index_topk_fp8", "msa_block_map", "msa_sparse_fwd_mapped", "msa_bwd_mapped",
            "msa_warmup_block_idx", "msa_set_timing_events", "msa_dense_fwd", "msa_dense_bwd")


class MsaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"MSA status {status}: {msg}")
        self.status = status


class MsaShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("Hq", ctypes.c_int32), ("G", ctypes.c_int32),
                ("d", ctypes.c_int32), ("d_idx", ctypes.c_int32), ("Bk", ctypes.c_int32), ("k", ctypes.c_int32),
                ("scale", ctypes.c_float), ("scale_idx", ctypes.c_float)]


@dataclass(frozen=True)
class Shape:
    B: int
    T: int
    Hq: int
    G: int
    d: int = 128
    d_idx: int = 64
    Bk: int = 128
    k: int = 16
    scale: float = 0.0
    scale_idx: float = 0.0

    def c(self) -> MsaShape:
        return MsaShape(self.B, self.T, self.Hq, self.G, self.d, self.d_idx, self.Bk, self.k, self.scale,
                        self.scale_idx)


_lib = None


def load_library():
    """Load the compiled library; raises if it is missing (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, S = ctypes.c_void_p, ctypes.POINTER(MsaShape)
    lib.msa_workspace_size.argtypes = [S, ctypes.c_int]
    lib.msa_workspace_size.restype = ctypes.c_size_t
    lib.msa_index_topk.argtypes = [S, P, P, P, P, ctypes.c_size_t, P]
    lib.msa_sparse_fwd.argtypes = [S, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.msa_bwd.argtypes = [S, P, P, P, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.msa_index_topk_fp8.argtypes = lib.msa_index_topk.argtypes
    lib.msa_index_topk_fp8.restype = ctypes.c_int
    lib.msa_sparse_fwd_mapped.argtypes = lib.msa_sparse_fwd.argtypes
    lib.msa_bwd_mapped.argtypes = lib.msa_bwd.argtypes
    lib.msa_block_map.argtypes = [S, P, P, ctypes.c_size_t, P]
    lib.msa_warmup_block_idx.argtypes = [S, P, P]
    lib.msa_set_timing_events.argtypes = [ctypes.c_int32, P, P]
    for f in (lib.msa_index_topk, lib.msa_sparse_fwd, lib.msa_bwd, lib.msa_sparse_fwd_mapped, lib.msa_bwd_mapped,
              lib.msa_block_map, lib.msa_warmup_block_idx, lib.msa_set_timing_events):
        f.restype = ctypes.c_int
    lib.msa_last_error.argtypes = []
    lib.msa_last_error.restype = ctypes.c_char_p
    lib.msa_check_device_status.argtypes = [P, P]
    lib.msa_check_device_status.restype = ctypes.c_int
    lib.msa_version.restype = ctypes.c_int32
    lib.msa_kernel_launches.restype = ctypes.c_int64
    lib.msa_index_topk_noalloc.argtypes = [S, P, P, P, ctypes.c_int32, P]
    lib.msa_index_topk_noalloc.restype = ctypes.c_int
    lib.msa_dense_fwd.argtypes = [S, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.msa_dense_fwd.restype = ctypes.c_int
    lib.msa_dense_bwd.argtypes = [S, P, P, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.msa_dense_bwd.restype = ctypes.c_int
    lib.msa_selftest_wait_timeout.argtypes = [P, ctypes.c_int32, P]
    lib.msa_selftest_wait_timeout.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("tensor arguments must live on the GPU")
    if not x.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return x.data_ptr()


def _nbytes(x) -> int:
    return x.numel() * x.element_size() if not isinstance(x, int) else 0


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _shape(shape) -> MsaShape:
    return shape.c() if isinstance(shape, Shape) else shape


def _check(status: int) -> None:
    if status != MSA_OK:
        raise MsaError(status, load_library().msa_last_error().decode())


def msa_version() -> int:
    return load_library().msa_version()


def msa_kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load_library().msa_kernel_launches())


def msa_workspace_size(shape, which: int) -> int:
    return int(load_library().msa_workspace_size(ctypes.byref(_shape(shape)), which))


def msa_index_topk(shape, q_idx, k_idx, block_idx, workspace, stream=None, workspace_bytes=None) -> None:
    wb = workspace_bytes if workspace_bytes is not None else _nbytes(workspace)
    _check(load_library().msa_index_topk(ctypes.byref(_shape(shape)), _ptr(q_idx), _ptr(k_idx), _ptr(block_idx),
                                         _ptr(workspace), wb, _stream(stream)))


def msa_index_topk_fp8(shape, q_idx, k_idx, block_idx, workspace, stream=None, workspace_bytes=None) -> None:
    """msa_index_topk on E4M3 copies of q_idx and k_idx (workspace sized with MSA_WS_TOPK_FP8)."""
    wb = workspace_bytes if workspace_bytes is not None else _nbytes(workspace)
    _check(load_library().msa_index_topk_fp8(ctypes.byref(_shape(shape)), _ptr(q_idx), _ptr(k_idx),
                                             _ptr(block_idx), _ptr(workspace), wb, _stream(stream)))


def msa_index_topk_noalloc(shape, q_idx, k_idx, block_idx, check: bool = True, stream=None) -> None:
    """msa_index_topk without a workspace (static scratch inside the library)."""
    _check(load_library().msa_index_topk_noalloc(ctypes.byref(_shape(shape)), _ptr(q_idx), _ptr(k_idx),
                                                 _ptr(block_idx), 1 if check else 0, _stream(stream)))


def msa_sparse_fwd(shape, Q, K, V, block_idx, O, LSE, workspace, stream=None, workspace_bytes=None) -> None:
    wb = workspace_bytes if workspace_bytes is not None else _nbytes(workspace)
    _check(load_library().msa_sparse_fwd(ctypes.byref(_shape(shape)), _ptr(Q), _ptr(K), _ptr(V), _ptr(block_idx),
                                         _ptr(O), _ptr(LSE), _ptr(workspace), wb, _stream(stream)))


def msa_block_map(shape, block_idx, workspace, stream=None, workspace_bytes=None) -> None:
    """Build the shared block map of block_idx in a MSA_WS_BWD-sized workspace (IndexShare)."""
    wb = workspace_bytes if workspace_bytes is not None else _nbytes(workspace)
    _check(load_library().msa_block_map(ctypes.byref(_shape(shape)), _ptr(block_idx), _ptr(workspace), wb,
                                        _stream(stream)))


def msa_warmup_block_idx(shape, block_idx, stream=None) -> None:
    """Full causal selection (every visible block) into block_idx [B,G,T,k] for the indexer warmup."""
    _check(load_library().msa_warmup_block_idx(ctypes.byref(_shape(shape)), _ptr(block_idx), _stream(stream)))


def msa_set_timing_events(which: int, start=None, stop=None) -> None:
    """Record two CUDA events (torch.cuda.Event with enable_timing, already
    recorded once so that they exist, or raw handles) around every launch of
    kernel `which`; no events stops the recording."""
    def handle(e):
        if e is None or isinstance(e, int):
            return e
        return e.cuda_event
    _check(load_library().msa_set_timing_events(int(which), handle(start), handle(stop)))


def msa_sparse_fwd_mapped(shape, Q, K, V, block_idx, O, LSE, workspace, stream=None, workspace_bytes=None) -> None:
    wb = workspace_bytes if workspace_bytes is not None else _nbytes(workspace)
    _check(load_library().msa_sparse_fwd_mapped(ctypes.byref(_shape(shape)), _ptr(Q), _ptr(K), _ptr(V),
                                                _ptr(block_idx), _ptr(O), _ptr(LSE), _ptr(workspace), wb,
                                                _stream(stream)))


def msa_bwd(shape, Q, K, V, O, dO, LSE, q_idx, k_idx, block_idx, kl_weight, dQ, dK, dV, dq_idx, dk_idx, KL,
            workspace, stream=None, workspace_bytes=None) -> None:
    wb = workspace_bytes if workspace_bytes is not None else _nbytes(workspace)
    _check(load_library().msa_bwd(ctypes.byref(_shape(shape)), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO),
                                  _ptr(LSE), _ptr(q_idx), _ptr(k_idx), _ptr(block_idx), float(kl_weight), _ptr(dQ),
                                  _ptr(dK), _ptr(dV), _ptr(dq_idx), _ptr(dk_idx), _ptr(KL), _ptr(workspace), wb,
                                  _stream(stream)))


def msa_bwd_mapped(shape, Q, K, V, O, dO, LSE, q_idx, k_idx, block_idx, kl_weight, dQ, dK, dV, dq_idx, dk_idx, KL,
                   workspace, stream=None, workspace_bytes=None) -> None:
    wb = workspace_bytes if workspace_bytes is not None else _nbytes(workspace)
    _check(load_library().msa_bwd_mapped(ctypes.byref(_shape(shape)), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO),
                                         _ptr(LSE), _ptr(q_idx), _ptr(k_idx), _ptr(block_idx), float(kl_weight),
                                         _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(dq_idx), _ptr(dk_idx), _ptr(KL),
                                         _ptr(workspace), wb, _stream(stream)))


def msa_dense_fwd(shape, Q, K, V, O, LSE, workspace, stream=None, workspace_bytes=None) -> None:
    wb = workspace_bytes if workspace_bytes is not None else _nbytes(workspace)
    _check(load_library().msa_dense_fwd(ctypes.byref(_shape(shape)), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                                        _ptr(workspace), wb, _stream(stream)))


def msa_dense_bwd(shape, Q, K, V, O, dO, LSE, q_idx, k_idx, kl_weight, dQ, dK, dV, dq_idx, dk_idx, KL, workspace,
                  stream=None, workspace_bytes=None) -> None:
    wb = workspace_bytes if workspace_bytes is not None else _nbytes(workspace)
    _check(load_library().msa_dense_bwd(ctypes.byref(_shape(shape)), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO),
                                        _ptr(LSE), _ptr(q_idx), _ptr(k_idx), float(kl_weight), _ptr(dQ), _ptr(dK),
                                        _ptr(dV), _ptr(dq_idx), _ptr(dk_idx), _ptr(KL), _ptr(workspace), wb,
                                        _stream(stream)))


def msa_selftest_wait_timeout(workspace, limit_us: int, stream=None) -> None:
    _check(load_library().msa_selftest_wait_timeout(_ptr(workspace), int(limit_us), _stream(stream)))


def msa_check_device_status(workspace, stream=None) -> None:
    _check(load_library().msa_check_device_status(_ptr(workspace), _stream(stream)))


# ----------------------------------------------------------------- allocation helpers (torch plumbing)
def alloc_workspace(shape, which: int = MSA_WS_BWD, device="cuda"):
    import torch

    n = msa_workspace_size(shape, which)
    if n == 0:
        raise MsaError(MSA_ERR_UNSUPPORTED, "shape not supported (see include/msa.h)")
    return torch.empty(n, dtype=torch.uint8, device=device)


def index_topk(shape: Shape, q_idx, k_idx, workspace=None, stream=None):
    """Allocate block_idx [B,G,T,k] int32 and run msa_index_topk."""
    import torch

    ws = workspace if workspace is not None else alloc_workspace(shape, MSA_WS_TOPK, q_idx.device)
    bi = torch.empty((shape.B, shape.G, shape.T, shape.k), dtype=torch.int32, device=q_idx.device)
    msa_index_topk(shape, q_idx, k_idx, bi, ws, stream)
    return bi


def warmup_block_idx(shape: Shape, device="cuda", stream=None):
    """Allocate block_idx [B,G,T,k] int32 and fill it with msa_warmup_block_idx."""
    import torch

    bi = torch.empty((shape.B, shape.G, shape.T, shape.k), dtype=torch.int32, device=device)
    msa_warmup_block_idx(shape, bi, stream)
    return bi


def sparse_fwd(shape: Shape, Q, K, V, block_idx, workspace=None, stream=None):
    """Allocate O [B,T,Hq,d] bf16 and LSE [B,T,Hq] fp32 and run msa_sparse_fwd."""
    import torch

    ws = workspace if workspace is not None else alloc_workspace(shape, MSA_WS_FWD, Q.device)
    O = torch.empty_like(Q)
    LSE = torch.empty((shape.B, shape.T, shape.Hq), dtype=torch.float32, device=Q.device)
    msa_sparse_fwd(shape, Q, K, V, block_idx, O, LSE, ws, stream)
    return O, LSE


def bwd(shape: Shape, Q, K, V, O, dO, LSE, q_idx, k_idx, block_idx, kl_weight=1.0, workspace=None, stream=None):
    """Allocate the fp32 gradients and KL and run msa_bwd. Returns a dict."""
    import torch

    ws = workspace if workspace is not None else alloc_workspace(shape, MSA_WS_BWD, Q.device)
    f32 = dict(dtype=torch.float32, device=Q.device)
    out = dict(dQ=torch.empty(Q.shape, **f32), dK=torch.empty(K.shape, **f32), dV=torch.empty(V.shape, **f32),
               dq_idx=torch.empty(q_idx.shape, **f32), dk_idx=torch.empty(k_idx.shape, **f32),
               KL=torch.empty((shape.B, shape.G, shape.T), **f32))
    msa_bwd(shape, Q, K, V, O, dO, LSE, q_idx, k_idx, block_idx, kl_weight, out["dQ"], out["dK"], out["dV"],
            out["dq_idx"], out["dk_idx"], out["KL"], ws, stream)
    return out


def dense_fwd(shape: Shape, Q, K, V, workspace=None, stream=None):
    """Allocate O and LSE and run msa_dense_fwd (full causal attention)."""
    import torch

    ws = workspace if workspace is not None else alloc_workspace(shape, MSA_WS_DENSE, Q.device)
    O = torch.empty_like(Q)
    LSE = torch.empty((shape.B, shape.T, shape.Hq), dtype=torch.float32, device=Q.device)
    msa_dense_fwd(shape, Q, K, V, O, LSE, ws, stream)
    return O, LSE


def dense_bwd(shape: Shape, Q, K, V, O, dO, LSE, q_idx, k_idx, kl_weight=1.0, workspace=None, stream=None):
    """Allocate the fp32 gradients and KL and run msa_dense_bwd. Returns a dict."""
    import torch

    ws = workspace if workspace is not None else alloc_workspace(shape, MSA_WS_DENSE, Q.device)
    f32 = dict(dtype=torch.float32, device=Q.device)
    out = dict(dQ=torch.empty(Q.shape, **f32), dK=torch.empty(K.shape, **f32), dV=torch.empty(V.shape, **f32),
               dq_idx=torch.empty(q_idx.shape, **f32), dk_idx=torch.empty(k_idx.shape, **f32),
               KL=torch.empty((shape.B, shape.G, shape.T), **f32))
    msa_dense_bwd(shape, Q, K, V, O, dO, LSE, q_idx, k_idx, kl_weight, out["dQ"], out["dK"], out["dV"],
                  out["dq_idx"], out["dk_idx"], out["KL"], ws, stream)
    return out
