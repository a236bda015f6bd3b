"""ctypes binding of libtt_emb.so: argument marshalling only.

Every function has the name and the argument order of its C entry point
(include/tt_emb.h).  Array arguments are CUDA torch tensors; the binding
checks dtype, device and contiguity, passes raw pointers and the current
CUDA stream, and turns a negative return code into TTEmbError.  All work runs
in the library's kernels; there is no fallback of any kind, and a missing
library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

TT_EMB_OK = 0
TT_EMB_ERR_ARG = -1
TT_EMB_ERR_WORKSPACE = -2
TT_EMB_ERR_CUDA = -3
TT_EMB_ERR_INDEX = -4
TT_EMB_ERR_OFFSETS = -5
TT_EMB_ERR_TIMEOUT = -6
TT_EMB_ERR_UNSUPPORTED = -7
TT_EMB_ERR_REUSE = -8
_NAMES = {v: k for k, v in list(globals().items()) if k.startswith("TT_EMB_")}
TT_EMB_POOL_SUM = 0
TT_EMB_POOL_MEAN = 1
TT_EMB_CORES_SPLIT = 1
TT_EMB_FORWARD_ONLY = 2
TT_EMB_INDICES_I32 = 4
_POOLING = {"sum": TT_EMB_POOL_SUM, "mean": TT_EMB_POOL_MEAN}

EXPORTED = ("tt_emb_workspace_bytes", "tt_emb_group", "tt_emb_forward", "tt_emb_backward",
            "tt_emb_forward_ex", "tt_emb_backward_ex", "tt_emb_split", "tt_emb_sgd_ex",
            "tt_emb_forward_tables", "tt_emb_forward_tables_ex", "tt_emb_workspace_bytes_d", "tt_emb_forward_d",
            "tt_emb_backward_d", "tt_emb_sgd_d", "tt_emb_step_host",
            "tt_emb_sgd", "tt_emb_get_error", "tt_emb_grouping_view", "tt_emb_profile_start",
            "tt_emb_profile_stop", "tt_emb_profile_read", "tt_emb_forward_static",
            "tt_emb_version")


class TTEmbError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {_NAMES.get(code, code)}")
        self.code = code


class Table(ctypes.Structure):
    """tt_emb_table of include/tt_emb.h."""
    _fields_ = [("cores", ctypes.c_void_p * 3), ("m", ctypes.c_int64 * 3), ("n", ctypes.c_int32 * 3),
                ("R", ctypes.c_int32 * 4), ("indices", ctypes.c_void_p), ("nnz", ctypes.c_int64),
                ("offsets", ctypes.c_void_p), ("num_bags", ctypes.c_int64),
                ("out", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("ws_bytes", ctypes.c_size_t)]


class HostBatch(ctypes.Structure):
    """tt_emb_host_batch of include/tt_emb.h."""
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "h_indices", "h_offsets", "h_grad_out", "h_out", "d_indices", "d_offsets", "d_grad_out",
        "d_out")] + [("nnz", ctypes.c_int64), ("num_bags", ctypes.c_int64)]


class Grouping(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "counts", "perm", "row_start", "row_i3", "row_pair", "pair_row_start", "pair_i1",
        "pair_i2", "uid", "bag_of", "chunk_start", "rowbuf", "chunk_order")]


_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libtt_emb.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "tensor_train_compressed_gb300.build.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(path)
        P, I64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
        L.tt_emb_workspace_bytes.argtypes = [P, P, P, I64, I64, ctypes.POINTER(SZ)]
        L.tt_emb_group.argtypes = [P, P, P, P, I64, P, I64, P, SZ, P]
        L.tt_emb_forward.argtypes = [P, P, P, P, P, I64, P, I64, P, P, SZ, P]
        L.tt_emb_backward.argtypes = [P, P, P, P, P, P, I64, P, I64, P, P, SZ, ctypes.c_int, P]
        L.tt_emb_forward_ex.argtypes = [P, P, P, P, P, I64, P, I64, P, ctypes.c_int, ctypes.c_int,
                                        P, P, SZ, P]
        L.tt_emb_split.argtypes = [P, P, P, P, P, SZ, P]
        L.tt_emb_forward_tables.argtypes = [ctypes.c_int, P, P]
        L.tt_emb_forward_tables_ex.argtypes = [ctypes.c_int, P, ctypes.c_int, P]
        C = ctypes.c_int
        L.tt_emb_workspace_bytes_d.argtypes = [C, P, P, P, I64, I64, ctypes.POINTER(SZ)]
        L.tt_emb_forward_d.argtypes = [C, P, P, P, P, P, I64, P, I64, P, P, SZ, P]
        L.tt_emb_backward_d.argtypes = [C, P, P, P, P, P, P, I64, P, I64, P, P, SZ, C, P]
        L.tt_emb_sgd_d.argtypes = [C, P, P, P, P, P, ctypes.c_float, C, P]
        L.tt_emb_sgd_ex.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_int, P, SZ, P]
        L.tt_emb_backward_ex.argtypes = [P, P, P, P, P, P, I64, P, I64, P, ctypes.c_int, P, P, P,
                                         SZ, ctypes.c_int, P]
        L.tt_emb_sgd.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_int, P]
        L.tt_emb_get_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_int)]
        L.tt_emb_grouping_view.argtypes = [P, P, P, I64, I64, P, ctypes.POINTER(Grouping)]
        L.tt_emb_forward_static.argtypes = [P, P, P, P, P, I64, P, I64, P, P]
        L.tt_emb_profile_start.argtypes = []
        L.tt_emb_profile_stop.argtypes = []
        L.tt_emb_profile_read.argtypes = [ctypes.c_int, ctypes.c_char_p, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_float)]
        for name in EXPORTED:
            getattr(L, name).restype = ctypes.c_int
        L.tt_emb_version.argtypes = []
        _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != TT_EMB_OK:
        raise TTEmbError(rc, what)


def _shape(m, n, R):
    return ((ctypes.c_int64 * 3)(*[int(v) for v in m]), (ctypes.c_int32 * 3)(*[int(v) for v in n]),
            (ctypes.c_int32 * 4)(*[int(v) for v in R]))


def _dev(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _ptrs3(ts, name):
    return (ctypes.c_void_p * 3)(*[_dev(t, torch.float32, f"{name}[{k}]").value
                                   for k, t in enumerate(ts)])


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def tt_emb_workspace_bytes(m, n, R, nnz: int, num_bags: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().tt_emb_workspace_bytes(*_shape(m, n, R), int(nnz), int(num_bags),
                                        ctypes.byref(out)), "tt_emb_workspace_bytes")
    return int(out.value)


def tt_emb_group(m, n, R, indices, offsets, workspace, stream=None):
    _check(lib().tt_emb_group(*_shape(m, n, R), _dev(indices, torch.int64, "indices"),
                              indices.numel(), _dev(offsets, torch.int64, "offsets"),
                              offsets.numel() - 1, _dev(workspace, torch.uint8, "workspace"),
                              workspace.numel(), _stream(stream)), "tt_emb_group")


def tt_emb_forward(cores, m, n, R, indices, offsets, out, workspace, stream=None):
    """Sum pooling; int32 indices go through tt_emb_forward_ex with TT_EMB_INDICES_I32."""
    if isinstance(indices, torch.Tensor) and indices.dtype == torch.int32:
        return tt_emb_forward_ex(cores, m, n, R, indices, offsets, None, "sum", out, workspace,
                                 stream)
    _check(lib().tt_emb_forward(_ptrs3(cores, "cores"), *_shape(m, n, R),
                                _dev(indices, torch.int64, "indices"), indices.numel(),
                                _dev(offsets, torch.int64, "offsets"), offsets.numel() - 1,
                                _dev(out, torch.float32, "out"),
                                _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                _stream(stream)), "tt_emb_forward")


def _bwd_indices(indices, reuse_grouping):
    """A backward that reuses the forward's grouping reads no index, so the forward's int32
    indices may be passed; one that regroups reads int64."""
    if reuse_grouping and isinstance(indices, torch.Tensor) and indices.dtype == torch.int32:
        return _dev(indices, torch.int32, "indices")
    return _dev(indices, torch.int64, "indices")


def tt_emb_backward(grad_out, cores, m, n, R, indices, offsets, core_grads, workspace,
                    reuse_grouping: bool = True, stream=None):
    _check(lib().tt_emb_backward(_dev(grad_out, torch.float32, "grad_out"),
                                 _ptrs3(cores, "cores"), *_shape(m, n, R),
                                 _bwd_indices(indices, reuse_grouping), indices.numel(),
                                 _dev(offsets, torch.int64, "offsets"), offsets.numel() - 1,
                                 _ptrs3(core_grads, "core_grads"),
                                 _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                 int(bool(reuse_grouping)), _stream(stream)), "tt_emb_backward")


def _opt(t, dtype, name):
    return None if t is None else _dev(t, dtype, name)


def _index_flag(t, name: str) -> int:
    """TT_EMB_INDICES_I32 for an int32 index tensor, 0 for int64 (either dtype is accepted
    by the calls that take flags)."""
    if isinstance(t, torch.Tensor) and t.dtype == torch.int32:
        return TT_EMB_INDICES_I32
    if isinstance(t, torch.Tensor) and t.dtype == torch.int64:
        return 0
    raise TypeError(f"{name} must be an int64 or int32 tensor")


def tt_emb_forward_ex(cores, m, n, R, indices, offsets, per_sample_weights, pooling, out,
                      workspace, stream=None, flags: int = 0):
    """pooling: "sum" / "mean" (or the TT_EMB_POOL_* value); per_sample_weights: None or a
    float32 CUDA tensor [nnz] (sum only); flags: 0, TT_EMB_CORES_SPLIT and/or
    TT_EMB_FORWARD_ONLY.  indices: int64 or int32 (TT_EMB_INDICES_I32 is set for int32)."""
    ixf = _index_flag(indices, "indices")
    flags = int(flags) | ixf
    _check(lib().tt_emb_forward_ex(_ptrs3(cores, "cores"), *_shape(m, n, R),
                                   _dev(indices, indices.dtype, "indices"), indices.numel(),
                                   _dev(offsets, torch.int64, "offsets"), offsets.numel() - 1,
                                   _opt(per_sample_weights, torch.float32, "per_sample_weights"),
                                   int(_POOLING.get(pooling, pooling)), int(flags),
                                   _dev(out, torch.float32, "out"),
                                   _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                   _stream(stream)), "tt_emb_forward_ex")


def tt_emb_backward_ex(grad_out, cores, m, n, R, indices, offsets, per_sample_weights, pooling,
                       core_grads, grad_weights, workspace, reuse_grouping: bool = True,
                       stream=None):
    _check(lib().tt_emb_backward_ex(_dev(grad_out, torch.float32, "grad_out"),
                                    _ptrs3(cores, "cores"), *_shape(m, n, R),
                                    _bwd_indices(indices, reuse_grouping), indices.numel(),
                                    _dev(offsets, torch.int64, "offsets"), offsets.numel() - 1,
                                    _opt(per_sample_weights, torch.float32, "per_sample_weights"),
                                    int(_POOLING.get(pooling, pooling)),
                                    _ptrs3(core_grads, "core_grads"),
                                    _opt(grad_weights, torch.float32, "grad_weights"),
                                    _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                    int(bool(reuse_grouping)), _stream(stream)),
           "tt_emb_backward_ex")


def tt_emb_sgd(cores, core_grads, m, n, R, lr: float, zero_grads: bool = False, stream=None):
    _check(lib().tt_emb_sgd(_ptrs3(cores, "cores"), _ptrs3(core_grads, "core_grads"),
                            *_shape(m, n, R), ctypes.c_float(lr), int(bool(zero_grads)),
                            _stream(stream)), "tt_emb_sgd")


def tt_emb_forward_tables(tables, stream=None, flags: int = 0):
    """tables: sequence of dicts with the tt_emb_forward arguments (cores, m, n, R, indices,
    offsets, out, workspace); every table needs its own workspace.  flags != 0 calls
    tt_emb_forward_tables_ex (TT_EMB_CORES_SPLIT: every workspace holds its table's split).
    Index tensors: all int64 or all int32 (TT_EMB_INDICES_I32 is set for int32)."""
    ixf = {_index_flag(t["indices"], f"tables[{k}].indices") for k, t in enumerate(tables)}
    if len(ixf) > 1:
        raise TypeError("the tables' index tensors must share one dtype")
    flags = int(flags) | (ixf.pop() if ixf else 0)
    arr = (Table * len(tables))()
    for k, t in enumerate(tables):
        e = arr[k]
        for j, c in enumerate(t["cores"]):
            e.cores[j] = _dev(c, torch.float32, f"tables[{k}].cores[{j}]").value
        m, n, R = _shape(t["m"], t["n"], t["R"])
        e.m[:], e.n[:], e.R[:] = list(m), list(n), list(R)
        e.indices = _dev(t["indices"], t["indices"].dtype, "indices")
        e.nnz = t["indices"].numel()
        e.offsets = _dev(t["offsets"], torch.int64, "offsets")
        e.num_bags = t["offsets"].numel() - 1
        e.out = _dev(t["out"], torch.float32, "out")
        e.workspace = _dev(t["workspace"], torch.uint8, "workspace")
        e.ws_bytes = t["workspace"].numel()
    if flags:
        _check(lib().tt_emb_forward_tables_ex(len(tables), ctypes.cast(arr, ctypes.c_void_p),
                                              int(flags), _stream(stream)),
               "tt_emb_forward_tables_ex")
    else:
        _check(lib().tt_emb_forward_tables(len(tables), ctypes.cast(arr, ctypes.c_void_p),
                                           _stream(stream)), "tt_emb_forward_tables")


def _shape_d(m, n, R):
    d = len(m)
    if len(n) != d or len(R) != d + 1:
        raise ValueError("a chain of d cores needs d row factors, d output factors, d + 1 ranks")
    return (d, (ctypes.c_int64 * d)(*[int(v) for v in m]), (ctypes.c_int32 * d)(*[int(v) for v in n]),
            (ctypes.c_int32 * (d + 1))(*[int(v) for v in R]))


def _ptrs_d(ts, name):
    return (ctypes.c_void_p * len(ts))(*[_dev(t, torch.float32, f"{name}[{k}]").value
                                         for k, t in enumerate(ts)])


def tt_emb_workspace_bytes_d(m, n, R, nnz: int, num_bags: int) -> int:
    out = ctypes.c_size_t(0)
    d, m_, n_, R_ = _shape_d(m, n, R)
    _check(lib().tt_emb_workspace_bytes_d(d, m_, n_, R_, int(nnz), int(num_bags), ctypes.byref(out)),
           "tt_emb_workspace_bytes_d")
    return int(out.value)


def tt_emb_forward_d(cores, m, n, R, indices, offsets, out, workspace, stream=None):
    d, m_, n_, R_ = _shape_d(m, n, R)
    _check(lib().tt_emb_forward_d(d, _ptrs_d(cores, "cores"), m_, n_, R_,
                                  _dev(indices, torch.int64, "indices"), indices.numel(),
                                  _dev(offsets, torch.int64, "offsets"), offsets.numel() - 1,
                                  _dev(out, torch.float32, "out"),
                                  _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                  _stream(stream)), "tt_emb_forward_d")


def tt_emb_backward_d(grad_out, cores, m, n, R, indices, offsets, core_grads, workspace,
                      reuse_grouping: bool = True, stream=None):
    d, m_, n_, R_ = _shape_d(m, n, R)
    _check(lib().tt_emb_backward_d(d, _dev(grad_out, torch.float32, "grad_out"),
                                   _ptrs_d(cores, "cores"), m_, n_, R_,
                                   _dev(indices, torch.int64, "indices"), indices.numel(),
                                   _dev(offsets, torch.int64, "offsets"), offsets.numel() - 1,
                                   _ptrs_d(core_grads, "core_grads"),
                                   _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                   int(bool(reuse_grouping)), _stream(stream)), "tt_emb_backward_d")


def tt_emb_sgd_d(cores, core_grads, m, n, R, lr: float, zero_grads: bool = False, stream=None):
    d, m_, n_, R_ = _shape_d(m, n, R)
    _check(lib().tt_emb_sgd_d(d, _ptrs_d(cores, "cores"), _ptrs_d(core_grads, "core_grads"), m_, n_,
                              R_, ctypes.c_float(lr), int(bool(zero_grads)), _stream(stream)),
           "tt_emb_sgd_d")


def tt_emb_split(cores, m, n, R, workspace, stream=None):
    _check(lib().tt_emb_split(_ptrs3(cores, "cores"), *_shape(m, n, R),
                              _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                              _stream(stream)), "tt_emb_split")


def tt_emb_sgd_ex(cores, core_grads, m, n, R, lr: float, zero_grads: bool, workspace, stream=None):
    _check(lib().tt_emb_sgd_ex(_ptrs3(cores, "cores"), _ptrs3(core_grads, "core_grads"),
                               *_shape(m, n, R), ctypes.c_float(lr), int(bool(zero_grads)),
                               _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                               _stream(stream)), "tt_emb_sgd_ex")


def _host(t, dtype, name: str):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


_copy_streams = {}


def tt_emb_step_host(cores, core_grads, m, n, R, h_indices, h_offsets, h_grad_out, h_out,
                     d_indices, d_offsets, d_grad_out, d_out, lr: float, workspace, flags: int = 0,
                     stream=None, copy_stream=None):
    """One step from host tensors (pinned for the copies to overlap): h_grad_out None runs a
    forward only, h_out None leaves the output on the device.  Without copy_stream a copy
    stream of this module (one per device) is used.  h_indices and d_indices: both int64 or
    both int32 (TT_EMB_INDICES_I32 is set for int32).  From the second call with the same
    tensors, sizes, lr, flags and streams the library replays a CUDA graph of the step
    (page-locked host tensors and non-default streams only)."""
    if copy_stream is None:
        dev = torch.cuda.current_device()
        if dev not in _copy_streams:
            _copy_streams[dev] = torch.cuda.Stream(device=dev)
        copy_stream = _copy_streams[dev]
    train = h_grad_out is not None
    b = HostBatch()
    ixf = _index_flag(h_indices, "h_indices")
    flags = int(flags) | ixf
    b.h_indices = _host(h_indices, h_indices.dtype, "h_indices")
    b.h_offsets = _host(h_offsets, torch.int64, "h_offsets")
    b.h_grad_out = _host(h_grad_out, torch.float32, "h_grad_out") if train else None
    b.h_out = None if h_out is None else _host(h_out, torch.float32, "h_out")
    b.d_indices = _dev(d_indices, h_indices.dtype, "d_indices")
    b.d_offsets = _dev(d_offsets, torch.int64, "d_offsets")
    b.d_grad_out = _dev(d_grad_out, torch.float32, "d_grad_out") if train else None
    b.d_out = _dev(d_out, torch.float32, "d_out")
    b.nnz = h_indices.numel()
    b.num_bags = h_offsets.numel() - 1
    if d_indices.numel() < b.nnz or d_offsets.numel() < b.num_bags + 1:
        raise ValueError("device staging tensors smaller than the host batch")
    D = int(n[0]) * int(n[1]) * int(n[2])
    for name, t in (("h_grad_out", h_grad_out), ("h_out", h_out), ("d_grad_out", d_grad_out),
                    ("d_out", d_out)):
        if t is not None and (name != "d_grad_out" or train) and t.numel() < b.num_bags * D:
            raise ValueError(f"{name} holds fewer than num_bags * D floats")
    grads = _ptrs3(core_grads, "core_grads") if train else None
    _check(lib().tt_emb_step_host(_ptrs3(cores, "cores"), grads, *_shape(m, n, R),
                                  ctypes.byref(b), ctypes.c_float(lr), int(flags),
                                  _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                  _stream(stream), _stream(copy_stream)), "tt_emb_step_host")


def tt_emb_get_error(workspace, stream=None) -> tuple[int, int]:
    """(return code, raw device status bits); synchronises the stream."""
    st = ctypes.c_int(0)
    rc = lib().tt_emb_get_error(_dev(workspace, torch.uint8, "workspace"), _stream(stream),
                                ctypes.byref(st))
    return int(rc), int(st.value)


def tt_emb_grouping_view(m, n, R, nnz: int, num_bags: int, workspace) -> dict:
    """Device addresses of the grouping arrays inside a workspace."""
    g = Grouping()
    _check(lib().tt_emb_grouping_view(*_shape(m, n, R), int(nnz), int(num_bags),
                                      _dev(workspace, torch.uint8, "workspace"), ctypes.byref(g)),
           "tt_emb_grouping_view")
    return {name: getattr(g, name) for name, _ in Grouping._fields_}


def tt_emb_forward_static(cores, m, n, R, indices, offsets, out, stream=None):
    """Forward without a workspace argument: the library's own fixed-size device array is used
    (for callers that cannot allocate; calls must not overlap on the GPU)."""
    _check(lib().tt_emb_forward_static(_ptrs3(cores, "cores"), *_shape(m, n, R),
                                       _dev(indices, torch.int64, "indices"), indices.numel(),
                                       _dev(offsets, torch.int64, "offsets"), offsets.numel() - 1,
                                       _dev(out, torch.float32, "out"), _stream(stream)),
           "tt_emb_forward_static")


def tt_emb_profile_start():
    _check(lib().tt_emb_profile_start(), "tt_emb_profile_start")


def tt_emb_profile_stop() -> int:
    return int(lib().tt_emb_profile_stop())


def tt_emb_profile_read(i: int) -> tuple[str, float]:
    """(kernel name, device ms) of the i-th recorded launch (synchronises its end event)."""
    buf = ctypes.create_string_buffer(64)
    ms = ctypes.c_float(0.0)
    _check(lib().tt_emb_profile_read(int(i), buf, 64, ctypes.byref(ms)), "tt_emb_profile_read")
    return buf.value.decode(), float(ms.value)


def tt_emb_version() -> int:
    return int(lib().tt_emb_version())
