"""CPU oracle of the Tensor-Train embedding bag -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
binding) never calls it and shares no code with it.

The arithmetic lives in ``tt_oracle.c`` (plain fp64 C, one naive chained
contraction per lookup, see its header for the definitions and the passages
they follow).  This module only compiles it with gcc and marshals numpy arrays
through ctypes.

Pins (tests/test_oracle_pins.py): a hand-worked example (tests/golden/),
exact reconstruction of a dense table through a TT-SVD, Kronecker rows for
rank-1 cores, a materialised table + torch embedding_bag (sum, mean and
per-sample weights), multilinearity, integer weights against repeated
lookups, exact TT-SVD reconstruction and torch autograd for chains of d cores, the adjoint identity, central differences and torch autograd for the
backward (core and weight gradients), and numpy lexsort/unique for the
grouping.  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tt_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libtt_oracle.so")
_lib = None
_lock = threading.Lock()

TTO_OK, TTO_ERR_ARG, TTO_ERR_INDEX, TTO_ERR_OFFSETS, TTO_ERR_NOMEM = 0, -1, -2, -3, -4


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} returned {code}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile tt_oracle.c into oracle/_build/libtt_oracle.so (gcc, -O2)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.tto_forward.argtypes = [P, P, P, P, P, P, P, I64, P, I64, P, ctypes.c_int]
            lib.tto_forward.restype = ctypes.c_int
            lib.tto_backward.argtypes = [P, P, P, P, P, P, P, P, I64, P, I64, P, P, P,
                                         ctypes.c_int, I64, ctypes.c_int]
            lib.tto_backward.restype = ctypes.c_int
            lib.tto_forward_ex.argtypes = [P, P, P, P, P, P, P, I64, P, I64, P, ctypes.c_int, P,
                                           ctypes.c_int]
            lib.tto_forward_ex.restype = ctypes.c_int
            lib.tto_backward_ex.argtypes = [P, P, P, P, P, P, P, P, I64, P, I64, P, ctypes.c_int,
                                            P, P, P, P, ctypes.c_int, I64, ctypes.c_int]
            lib.tto_backward_ex.restype = ctypes.c_int
            lib.tto_forward_d.argtypes = [ctypes.c_int, P, P, P, P, P, I64, P, I64, P]
            lib.tto_forward_d.restype = ctypes.c_int
            lib.tto_backward_d.argtypes = [ctypes.c_int, P, P, P, P, P, P, I64, P, I64, P]
            lib.tto_backward_d.restype = ctypes.c_int
            lib.tto_sgd.argtypes = [P, P, I64, ctypes.c_double, P]
            lib.tto_sgd.restype = None
            lib.tto_group.argtypes = [P, I64, P, P, P, P, P, P, P, P, P, P]
            lib.tto_group.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _shape_args(m, n, R):
    m_a = np.ascontiguousarray(m, dtype=np.int64)
    n_a = np.ascontiguousarray(n, dtype=np.int32)
    R_a = np.ascontiguousarray(R, dtype=np.int32)
    return m_a, n_a, R_a


def _cores(cores):
    return [np.ascontiguousarray(c, dtype=np.float32) for c in cores]


_MODES = {"sum": 0, "mean": 1}


def _weights(weights, nnz):
    if weights is None:
        return None
    w = np.ascontiguousarray(weights, dtype=np.float32)
    if w.shape != (nnz,):
        raise ValueError(f"weights must have shape ({nnz},)")
    return w


def forward(cores, m, n, R, indices, offsets, threads: int = 1, strict: bool = True,
            weights=None, mode: str = "sum"):
    """fp64 pooled output [B][D] (naive chained contraction per lookup, then the bag's sum;
    ``weights`` scale each lookup's row, ``mode="mean"`` divides by the bag length)."""
    lib = _load()
    G = _cores(cores)
    m_a, n_a, R_a = _shape_args(m, n, R)
    idx = np.ascontiguousarray(indices, dtype=np.int64)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    w = _weights(weights, idx.shape[0])
    B = off.shape[0] - 1
    D = int(n_a.prod())
    out = np.zeros((max(B, 0), D), dtype=np.float64)
    rc = lib.tto_forward_ex(_p(G[0]), _p(G[1]), _p(G[2]), _p(m_a), _p(n_a), _p(R_a), _p(idx),
                            idx.shape[0], _p(off), B, None if w is None else _p(w),
                            _MODES[mode], _p(out), int(threads))
    if rc != TTO_OK and (strict or rc != TTO_ERR_INDEX):
        raise OracleError(rc, "tto_forward_ex")
    return out


def backward(grad_out, cores, m, n, R, indices, offsets, threads: int = 1,
             filter_core: int = 0, filter_value: int = 0, strict: bool = True,
             weights=None, mode: str = "sum", want_dw: bool = False):
    """fp64 core gradients [dG1, dG2, dG3] of <grad_out, out> (fresh zeros, then +=); with
    ``want_dw`` also the gradient of the per-sample weights, fp64 [nnz]."""
    lib = _load()
    G = _cores(cores)
    m_a, n_a, R_a = _shape_args(m, n, R)
    idx = np.ascontiguousarray(indices, dtype=np.int64)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    g = np.ascontiguousarray(grad_out, dtype=np.float32)
    w = _weights(weights, idx.shape[0])
    B = off.shape[0] - 1
    dG = [np.zeros(c.shape, dtype=np.float64) for c in G]
    dW = np.zeros(idx.shape[0], dtype=np.float64) if want_dw else None
    rc = lib.tto_backward_ex(_p(g), _p(G[0]), _p(G[1]), _p(G[2]), _p(m_a), _p(n_a), _p(R_a),
                             _p(idx), idx.shape[0], _p(off), B, None if w is None else _p(w),
                             _MODES[mode], _p(dG[0]), _p(dG[1]), _p(dG[2]),
                             None if dW is None else _p(dW), int(filter_core), int(filter_value),
                             int(threads))
    if rc != TTO_OK and (strict or rc != TTO_ERR_INDEX):
        raise OracleError(rc, "tto_backward_ex")
    return (dG, dW) if want_dw else dG


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def forward_d(cores, m, n, R, indices, offsets, strict: bool = True):
    """fp64 pooled output [B][D] of a chain of d = len(cores) cores (sum pooling)."""
    lib = _load()
    G = [np.ascontiguousarray(c, dtype=np.float32) for c in cores]
    d = len(G)
    m_a = np.ascontiguousarray(m, dtype=np.int64)
    n_a = np.ascontiguousarray(n, dtype=np.int32)
    R_a = np.ascontiguousarray(R, dtype=np.int32)
    idx = np.ascontiguousarray(indices, dtype=np.int64)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    B = off.shape[0] - 1
    out = np.zeros((max(B, 0), int(n_a.prod())), dtype=np.float64)
    gp = _ptr_array(G)
    rc = lib.tto_forward_d(d, gp, _p(m_a), _p(n_a), _p(R_a), _p(idx), idx.shape[0], _p(off), B,
                           _p(out))
    if rc != TTO_OK and (strict or rc != TTO_ERR_INDEX):
        raise OracleError(rc, "tto_forward_d")
    return out


def backward_d(grad_out, cores, m, n, R, indices, offsets, strict: bool = True):
    """fp64 gradients of <grad_out, out> for every core of a d-core chain (fresh zeros, +=)."""
    lib = _load()
    G = [np.ascontiguousarray(c, dtype=np.float32) for c in cores]
    d = len(G)
    m_a = np.ascontiguousarray(m, dtype=np.int64)
    n_a = np.ascontiguousarray(n, dtype=np.int32)
    R_a = np.ascontiguousarray(R, dtype=np.int32)
    idx = np.ascontiguousarray(indices, dtype=np.int64)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    g = np.ascontiguousarray(grad_out, dtype=np.float32)
    B = off.shape[0] - 1
    dG = [np.zeros(c.shape, dtype=np.float64) for c in G]
    rc = lib.tto_backward_d(d, _p(g), _ptr_array(G), _p(m_a), _p(n_a), _p(R_a), _p(idx),
                            idx.shape[0], _p(off), B, _ptr_array(dG))
    if rc != TTO_OK and (strict or rc != TTO_ERR_INDEX):
        raise OracleError(rc, "tto_backward_d")
    return dG


def sgd(core, dcore, lr: float):
    """fp64 G - lr*dG."""
    lib = _load()
    G = np.ascontiguousarray(core, dtype=np.float32)
    dG = np.ascontiguousarray(dcore, dtype=np.float64)
    out = np.empty(G.shape, dtype=np.float64)
    lib.tto_sgd(_p(G), _p(dG), G.size, float(lr), _p(out))
    return out


def group(indices, m):
    """Grouping reference: stable sort by (i2, i1, i3) and unique runs (see tt_oracle.c)."""
    lib = _load()
    idx = np.ascontiguousarray(indices, dtype=np.int64)
    nnz = idx.shape[0]
    m_a = np.ascontiguousarray(m, dtype=np.int64)
    cap = max(nnz, 1)
    perm = np.empty(cap, np.int32)
    row_start = np.empty(cap + 1, np.int32)
    row_index = np.empty(cap, np.int64)
    row_pair = np.empty(cap, np.int32)
    pair_row_start = np.empty(cap + 1, np.int32)
    pair_i1 = np.empty(cap, np.int32)
    pair_i2 = np.empty(cap, np.int32)
    uid = np.empty(cap, np.int32)
    counts = np.zeros(3, np.int64)
    rc = lib.tto_group(_p(idx), nnz, _p(m_a), _p(perm), _p(row_start), _p(row_index),
                       _p(row_pair), _p(pair_row_start), _p(pair_i1), _p(pair_i2), _p(uid),
                       _p(counts))
    if rc not in (TTO_OK, TTO_ERR_INDEX):
        raise OracleError(rc, "tto_group")
    nv, ur, up = (int(v) for v in counts)
    return dict(n_valid=nv, U_r=ur, U_12=up, perm=perm[:nv].copy(),
                row_start=row_start[:ur + 1].copy(), row_index=row_index[:ur].copy(),
                row_pair=row_pair[:ur].copy(), pair_row_start=pair_row_start[:up + 1].copy(),
                pair_i1=pair_i1[:up].copy(), pair_i2=pair_i2[:up].copy(),
                uid=uid[:nnz].copy(), status=rc)
