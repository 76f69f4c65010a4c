"""Thin Python binding of the TreeWY C ABI (include/treewy.h).

Argument marshalling only: every step of verification and commit runs in the
CUDA library.  There is no CPU fallback; if the library is missing this
module raises instead of computing anything.

Entry points keep the C names: ``treewy_verify``, ``treewy_commit``,
``treewy_storeall_verify``, ``treewy_storeall_commit``, ``treewy_last_error``
and ``treewy_version``.  ``TreewyBatch`` mirrors ``struct treewy_batch``;
``make_batch`` fills one from torch tensors (device memory and streams are
PyTorch's; the library only receives raw pointers).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtreewy.so")

TREEWY_OK = 0
TREEWY_ERR_INVALID_ARG = 1
TREEWY_ERR_UNSUPPORTED = 3
TREEWY_ERR_CUDA = 4

STATUS_BAD_TREE = 1
STATUS_TOO_MANY_NODES = 2
STATUS_BAD_ACCEPTED = 4
STATUS_BAD_SLOT = 8
STATUS_TIMEOUT = 16
STATUS_COMMIT_REFUSED = 32

DTYPE_BF16 = 0
DTYPE_F32 = 1
FLAG_FORCE_GENERIC = 1
FLAG_STATE_BF16 = 2
MAX_NODES = 64


class TreewyError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"treewy error {code}: {message}")
        self.code = code


class TreewyBatch(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("dk", ctypes.c_int32),
        ("dv", ctypes.c_int32),
        ("max_nodes", ctypes.c_int32),
        ("qkv_dtype", ctypes.c_int32),
        ("T", ctypes.c_int64),
        ("num_slots", ctypes.c_int64),
        ("node_offset", ctypes.c_void_p),
        ("parent", ctypes.c_void_p),
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("alpha", ctypes.c_void_p),
        ("beta", ctypes.c_void_p),
        ("state", ctypes.c_void_p),
        ("state_slot", ctypes.c_void_p),
        ("o", ctypes.c_void_p),
        ("U", ctypes.c_void_p),
        ("gamma", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
        ("flags", ctypes.c_uint32),
        ("reserved", ctypes.c_uint32),
    ]


_lib: Optional[ctypes.CDLL] = None

ENTRY_POINTS = ("treewy_verify", "treewy_commit", "treewy_commit_verify", "treewy_storeall_verify",
                "treewy_storeall_commit", "treewy_selftest_wait_timeout", "treewy_last_error",
                "treewy_version")


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libtreewy.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"TreeWY CUDA library not found at {p}; build it with "
            "gdn_speculative_tree_gb300.build.build() (there is no CPU fallback)")
    lib = ctypes.CDLL(p)
    bp = ctypes.POINTER(TreewyBatch)
    vp = ctypes.c_void_p
    lib.treewy_verify.argtypes = [bp, vp]
    lib.treewy_commit.argtypes = [bp, vp, vp]
    lib.treewy_commit_verify.argtypes = [bp, vp, bp, vp]
    lib.treewy_storeall_verify.argtypes = [bp, vp, vp]
    lib.treewy_storeall_commit.argtypes = [bp, vp, vp, vp]
    lib.treewy_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint32, vp]
    for name in ("treewy_verify", "treewy_commit", "treewy_commit_verify", "treewy_storeall_verify",
                 "treewy_storeall_commit", "treewy_selftest_wait_timeout"):
        getattr(lib, name).restype = ctypes.c_int
    lib.treewy_last_error.argtypes = []
    lib.treewy_last_error.restype = ctypes.c_char_p
    lib.treewy_version.argtypes = []
    lib.treewy_version.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def _check(code: int) -> None:
    if code != TREEWY_OK:
        raise TreewyError(code, treewy_last_error())


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def treewy_last_error() -> str:
    return load().treewy_last_error().decode()


def treewy_version() -> str:
    return load().treewy_version().decode()


def treewy_selftest_wait_timeout(status, limit_us: int, stream=None) -> None:
    """Diagnostic of the bounded barrier wait: ``status`` is a device int32
    tensor of 3 words (status[0] gets TREEWY_STATUS_TIMEOUT, status[1:3] the
    wait in nanoseconds, low and high word)."""
    _check(load().treewy_selftest_wait_timeout(_ptr(status), int(limit_us), _stream_handle(stream)))


def treewy_verify(batch: TreewyBatch, stream=None) -> None:
    """Verify every draft node (asynchronous on ``stream``)."""
    _check(load().treewy_verify(ctypes.byref(batch), _stream_handle(stream)))


def treewy_commit(batch: TreewyBatch, accepted, stream=None) -> None:
    """Rebuild the accepted state in place; ``accepted`` int32 [R] on the device."""
    _check(load().treewy_commit(ctypes.byref(batch), _ptr(accepted), _stream_handle(stream)))


def treewy_commit_verify(prev: TreewyBatch, prev_accepted, next_batch: TreewyBatch,
                         stream=None) -> None:
    """Apply the previous round's commit inside this round's verification."""
    _check(load().treewy_commit_verify(ctypes.byref(prev), _ptr(prev_accepted), ctypes.byref(next_batch),
                                       _stream_handle(stream)))


def treewy_storeall_verify(batch: TreewyBatch, snapshots, stream=None) -> None:
    """Snapshot-per-node comparator: writes every node's state to ``snapshots``."""
    _check(load().treewy_storeall_verify(ctypes.byref(batch), _ptr(snapshots), _stream_handle(stream)))


def treewy_storeall_commit(batch: TreewyBatch, snapshots, accepted, stream=None) -> None:
    """Snapshot rollback: copy the accepted node's snapshot into the state pool."""
    _check(load().treewy_storeall_commit(ctypes.byref(batch), _ptr(snapshots), _ptr(accepted),
                                         _stream_handle(stream)))


def make_batch(*, node_offset, parent, q, k, v, alpha, beta, state, state_slot, o, U, status,
               gamma=None, max_nodes: int = MAX_NODES, T: Optional[int] = None,
               flags: int = 0) -> TreewyBatch:
    """Fill a TreewyBatch from torch tensors (shapes as in include/treewy.h).

    The tensors must stay alive while the library uses them; the returned
    structure keeps references to them in ``_keep``.
    """
    import torch
    R = int(node_offset.numel()) - 1
    Tn = int(q.shape[0]) if T is None else int(T)
    H = int(q.shape[1])
    dk = int(q.shape[2])
    dv = int(v.shape[2])
    if q.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif q.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise TypeError(f"q/k/v dtype {q.dtype} is not bf16 or fp32")
    for name, x in (("q", q), ("k", k), ("v", v), ("alpha", alpha), ("beta", beta), ("state", state),
                    ("o", o), ("U", U), ("status", status), ("node_offset", node_offset),
                    ("parent", parent), ("state_slot", state_slot)):
        if x is not None and not x.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if state.dtype == torch.bfloat16:
        flags |= FLAG_STATE_BF16
    elif state.dtype != torch.float32:
        raise TypeError(f"state dtype {state.dtype} is not fp32 or bf16")
    b = TreewyBatch()
    b.R, b.H, b.dk, b.dv = R, H, dk, dv
    b.max_nodes = int(max_nodes)
    b.qkv_dtype = dt
    b.T = Tn
    b.num_slots = int(state.shape[0])
    b.node_offset = _ptr(node_offset)
    b.parent = _ptr(parent)
    b.q, b.k, b.v = _ptr(q), _ptr(k), _ptr(v)
    b.alpha, b.beta = _ptr(alpha), _ptr(beta)
    b.state = _ptr(state)
    b.state_slot = _ptr(state_slot)
    b.o, b.U = _ptr(o), _ptr(U)
    b.gamma = _ptr(gamma)
    b.status = _ptr(status)
    b.flags = int(flags)
    b._keep = (node_offset, parent, q, k, v, alpha, beta, state, state_slot, o, U, gamma, status)
    return b


class TreeVerifier:
    """Convenience holder: one layer's device tensors, outputs and batch struct.

    ``wl`` is a workloads.Workload already on the device.  Outputs o, U,
    gamma and status are allocated once (torch) and reused across calls.
    """

    def __init__(self, wl, flags: int = 0, max_nodes: Optional[int] = None):
        import torch
        dev = wl.q.device
        self.wl = wl
        self.o = torch.empty(wl.T, wl.H, wl.dv, device=dev, dtype=torch.float32)
        self.U = torch.empty_like(self.o)
        self.gamma = torch.empty(wl.T, wl.H, device=dev, dtype=torch.float32)
        self.status = torch.zeros(wl.R, device=dev, dtype=torch.int32)
        self.batch = make_batch(node_offset=wl.node_offset, parent=wl.parent, q=wl.q, k=wl.k,
                                v=wl.v, alpha=wl.alpha, beta=wl.beta, state=wl.state,
                                state_slot=wl.state_slot, o=self.o, U=self.U, status=self.status,
                                gamma=self.gamma, max_nodes=max_nodes or wl.max_nodes, flags=flags)

    def verify(self, stream=None) -> None:
        treewy_verify(self.batch, stream)

    def commit(self, accepted=None, stream=None) -> None:
        treewy_commit(self.batch, self.wl.accepted if accepted is None else accepted, stream)
