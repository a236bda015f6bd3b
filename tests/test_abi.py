"""The C-ABI library loads and exports every entry point its header declares (no GPU).

Only host-side argument checks are exercised here: each call below returns
before anything is enqueued on a device.
"""
import ctypes
import glob
import os
import re

import pytest

import tensor_train_compressed_gb300 as tte
from tensor_train_compressed_gb300 import _binding as B
from tensor_train_compressed_gb300 import build as tbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    tbuild.build()
    return tte.lib()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names |= set(re.findall(r"^\s*int\s+(tt_emb_\w+)\s*\(", src, flags=re.M))
    return names


def test_header_symbols_exported(L):
    names = _declared()
    assert {"tt_emb_forward", "tt_emb_backward", "tt_emb_sgd", "tt_emb_workspace_bytes"} <= names
    for n in names:
        assert hasattr(L, n), n
    assert set(B.EXPORTED) >= names


def test_version(L):
    assert tte.tt_emb_version() >= 100


def test_workspace_bytes_and_shape_errors(L):
    b = tte.tt_emb_workspace_bytes((200, 240, 250), (4, 8, 4), (1, 32, 32, 1), 655360, 32768)
    # the unique-row buffer dominates: min(nnz, M) rows of D floats
    assert b >= 655360 * 128 * 4
    small = tte.tt_emb_workspace_bytes((10, 10, 10), (2, 4, 2), (1, 4, 4, 1), 100, 10)
    assert small >= 100 * 16 * 4 and small < b
    with pytest.raises(tte.TTEmbError) as e:
        tte.tt_emb_workspace_bytes((10, 10, 10), (2, 4, 2), (2, 4, 4, 1), 100, 10)
    assert e.value.code == tte.TT_EMB_ERR_ARG
    with pytest.raises(tte.TTEmbError) as e:   # G2 slice beyond shared memory
        tte.tt_emb_workspace_bytes((10, 10, 10), (4, 16, 4), (1, 128, 128, 1), 100, 10)
    assert e.value.code == tte.TT_EMB_ERR_UNSUPPORTED
    with pytest.raises(tte.TTEmbError) as e:   # M beyond 2^32 - 2
        tte.tt_emb_workspace_bytes((70000, 70000, 2), (2, 2, 2), (1, 2, 2, 1), 100, 10)
    assert e.value.code == tte.TT_EMB_ERR_UNSUPPORTED


def _shape(m, n, R):
    return B._shape(m, n, R)


def test_forward_host_side_argument_checks(L):
    """Null, misaligned and undersized arguments are refused before any launch."""
    m, n, R = (10, 10, 10), (2, 4, 2), (1, 4, 4, 1)
    fake = 1 << 20                       # never dereferenced: the checks fail first
    cores = (ctypes.c_void_p * 3)(fake, fake, fake)
    P = ctypes.c_void_p
    need = tte.tt_emb_workspace_bytes(m, n, R, 100, 10)
    rc = L.tt_emb_forward(cores, *_shape(m, n, R), P(fake), 100, P(fake), 10, P(fake), P(fake),
                          need - 1, None)
    assert rc == tte.TT_EMB_ERR_WORKSPACE
    rc = L.tt_emb_forward(cores, *_shape(m, n, R), P(fake), 100, P(fake), 10, P(fake),
                          P(fake + 8), need, None)
    assert rc == tte.TT_EMB_ERR_ARG      # workspace not 256-byte aligned
    rc = L.tt_emb_forward(cores, *_shape(m, n, R), None, 100, P(fake), 10, P(fake), P(fake),
                          need, None)
    assert rc == tte.TT_EMB_ERR_ARG      # null indices
    rc = L.tt_emb_forward(cores, *_shape(m, n, R), P(fake), 100, P(fake), 0, P(fake), P(fake),
                          need, None)
    assert rc == tte.TT_EMB_ERR_ARG      # lookups without bags
    bad = (ctypes.c_void_p * 3)(fake, fake + 4, fake)
    rc = L.tt_emb_forward(bad, *_shape(m, n, R), P(fake), 100, P(fake), 10, P(fake), P(fake),
                          need, None)
    assert rc == tte.TT_EMB_ERR_ARG      # core not 16-byte aligned
    rc = L.tt_emb_backward(P(fake), cores, *_shape(m, n, R), P(fake), 100, P(fake), 10, None,
                           P(fake), need, 1, None)
    assert rc == tte.TT_EMB_ERR_ARG      # null core_grads
    rc = L.tt_emb_sgd(cores, None, *_shape(m, n, R), ctypes.c_float(0.1), 0, None)
    assert rc == tte.TT_EMB_ERR_ARG


def test_pooling_variant_argument_checks(L):
    """Weights go with the sum only; the weight gradient needs weights; unknown rules fail."""
    m, n, R = (10, 10, 10), (2, 4, 2), (1, 4, 4, 1)
    fake = 1 << 20
    cores = (ctypes.c_void_p * 3)(fake, fake, fake)
    P = ctypes.c_void_p
    need = tte.tt_emb_workspace_bytes(m, n, R, 100, 10)
    fwd = lambda psw, pooling, ws=need, flags=0: L.tt_emb_forward_ex(
        cores, *_shape(m, n, R), P(fake), 100, P(fake), 10, psw, pooling, flags, P(fake),
        P(fake), ws, None)
    assert fwd(P(fake), tte.TT_EMB_POOL_MEAN) == tte.TT_EMB_ERR_ARG     # weights with the mean
    assert fwd(None, 7) == tte.TT_EMB_ERR_ARG                           # unknown pooling
    assert fwd(P(fake + 2), tte.TT_EMB_POOL_SUM) == tte.TT_EMB_ERR_ARG  # misaligned weights
    assert fwd(None, tte.TT_EMB_POOL_MEAN, need - 1) == tte.TT_EMB_ERR_WORKSPACE
    assert fwd(None, tte.TT_EMB_POOL_SUM, need, 8) == tte.TT_EMB_ERR_ARG    # unknown flag
    bwd = lambda psw, pooling, gw: L.tt_emb_backward_ex(
        P(fake), cores, *_shape(m, n, R), P(fake), 100, P(fake), 10, psw, pooling, cores, gw,
        P(fake), need - 1, 1, None)
    assert bwd(None, tte.TT_EMB_POOL_SUM, P(fake)) == tte.TT_EMB_ERR_ARG   # no weights
    assert bwd(P(fake), tte.TT_EMB_POOL_MEAN, None) == tte.TT_EMB_ERR_ARG
    assert bwd(P(fake), tte.TT_EMB_POOL_SUM, P(fake + 1)) == tte.TT_EMB_ERR_ARG
    assert bwd(P(fake), tte.TT_EMB_POOL_SUM, P(fake)) == tte.TT_EMB_ERR_WORKSPACE


def test_index_width_argument_checks(L):
    """Indices are int64 (8-byte aligned) or, with TT_EMB_INDICES_I32, int32 (4-byte
    aligned); the flag is known to the three calls that take flags."""
    m, n, R = (10, 10, 10), (2, 4, 2), (1, 4, 4, 1)
    fake = 1 << 20
    cores = (ctypes.c_void_p * 3)(fake, fake, fake)
    P = ctypes.c_void_p
    need = tte.tt_emb_workspace_bytes(m, n, R, 100, 10)
    fwd = lambda idx, flags: L.tt_emb_forward_ex(
        cores, *_shape(m, n, R), P(idx), 100, P(fake), 10, None, tte.TT_EMB_POOL_SUM, flags,
        P(fake), P(fake), need, None)
    assert fwd(fake + 4, 0) == tte.TT_EMB_ERR_ARG                        # int64 at 4 bytes
    assert fwd(fake + 2, tte.TT_EMB_INDICES_I32) == tte.TT_EMB_ERR_ARG   # int32 at 2 bytes
    assert tte.TT_EMB_INDICES_I32 == 4
    from tensor_train_compressed_gb300._binding import Table
    arr = (Table * 1)()
    arr[0].cores[:] = [fake, fake, fake]
    arr[0].m[:], arr[0].n[:], arr[0].R[:] = list(m), list(n), list(R)
    arr[0].indices, arr[0].nnz, arr[0].offsets, arr[0].num_bags = fake + 2, 100, fake, 10
    arr[0].out, arr[0].workspace, arr[0].ws_bytes = fake, fake, need
    ptr = ctypes.cast(arr, P)
    assert L.tt_emb_forward_tables_ex(1, ptr, tte.TT_EMB_INDICES_I32, None) == tte.TT_EMB_ERR_ARG
    assert L.tt_emb_forward_tables_ex(1, ptr, 8, None) == tte.TT_EMB_ERR_ARG   # unknown flag


def test_index_dtype_binding_checks():
    """The binding takes int64 or int32 index tensors and sets the flag from the dtype."""
    import torch
    assert B._index_flag(torch.zeros(3, dtype=torch.int64), "i") == 0
    assert B._index_flag(torch.zeros(3, dtype=torch.int32), "i") == tte.TT_EMB_INDICES_I32
    for bad in (torch.zeros(3, dtype=torch.int16), torch.zeros(3), [0, 1]):
        with pytest.raises(TypeError):
            B._index_flag(bad, "i")


def test_product_path_has_no_oracle_dependency():
    """The package never imports the oracle."""
    pkg = os.path.join(ROOT, "tensor_train_compressed_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h")):
            src = open(path).read()
            assert "import oracle" not in src and "from oracle" not in src, path
            assert "tt_oracle" not in src, path


def test_split_and_fused_sgd_argument_checks(L):
    """The planes' workspace part depends on the shape alone; too small or misaligned
    workspaces are refused before any launch."""
    m, n, R = (200, 240, 250), (4, 8, 4), (1, 32, 32, 1)
    fake = 1 << 20
    cores = (ctypes.c_void_p * 3)(fake, fake, fake)
    P = ctypes.c_void_p
    small = tte.tt_emb_workspace_bytes(m, n, R, 0, 0)
    # any batch's workspace holds the planes
    assert tte.tt_emb_workspace_bytes(m, n, R, 1000, 10) >= small
    assert L.tt_emb_split(cores, *_shape(m, n, R), P(fake), 1024, None) == tte.TT_EMB_ERR_WORKSPACE
    assert L.tt_emb_split(cores, *_shape(m, n, R), P(fake + 16), small, None) == tte.TT_EMB_ERR_ARG
    assert L.tt_emb_sgd_ex(cores, cores, *_shape(m, n, R), ctypes.c_float(0.1), 0, P(fake), 1024,
                           None) == tte.TT_EMB_ERR_WORKSPACE
    assert L.tt_emb_sgd_ex(cores, None, *_shape(m, n, R), ctypes.c_float(0.1), 0, P(fake), small,
                           None) == tte.TT_EMB_ERR_ARG


def test_forward_tables_argument_checks(L):
    """Table counts outside 1..8 and tables that share a workspace are refused before any
    launch."""
    from tensor_train_compressed_gb300._binding import Table
    fake = 1 << 20
    m, n, R = (10, 10, 10), (2, 4, 2), (1, 4, 4, 1)
    need = tte.tt_emb_workspace_bytes(m, n, R, 100, 10)
    arr = (Table * 9)()
    for t in arr:
        t.cores[:] = [fake, fake, fake]
        t.m[:], t.n[:], t.R[:] = list(m), list(n), list(R)
        t.indices, t.nnz, t.offsets, t.num_bags = fake, 100, fake, 10
        t.out, t.workspace, t.ws_bytes = fake, fake, need
    P = ctypes.c_void_p
    ptr = ctypes.cast(arr, P)
    assert L.tt_emb_forward_tables(0, ptr, None) == tte.TT_EMB_ERR_ARG
    assert L.tt_emb_forward_tables(9, ptr, None) == tte.TT_EMB_ERR_ARG
    assert L.tt_emb_forward_tables(2, ptr, None) == tte.TT_EMB_ERR_ARG   # shared workspace
    arr[1].workspace = fake + need + 256
    arr[1].n[1] = 8
    assert L.tt_emb_forward_tables(2, ptr, None) == tte.TT_EMB_ERR_ARG   # other n


def test_chain_workspace_and_shape_checks(L):
    # four cores: the three-core view of (10, 12, 20, 30) x (2, 2, 8, 4) is (120, 20, 30) x (4, 8, 4)
    m, n, R = (10, 12, 20, 30), (2, 2, 8, 4), (1, 16, 32, 32, 1)
    b4 = tte.tt_emb_workspace_bytes_d(m, n, R, 1000, 100)
    b3 = tte.tt_emb_workspace_bytes((120, 20, 30), (4, 8, 4), (1, 32, 32, 1), 1000, 100)
    # the merged core (120 x 4 x 32 floats) and its gradient come on top
    assert b4 >= b3 + 2 * 120 * 4 * 32 * 4
    assert tte.tt_emb_workspace_bytes_d((10, 20, 30), (4, 8, 4), (1, 32, 32, 1), 10, 2) == \
        tte.tt_emb_workspace_bytes((10, 20, 30), (4, 8, 4), (1, 32, 32, 1), 10, 2)
    with pytest.raises(tte.TTEmbError) as e:      # R[0] != 1
        tte.tt_emb_workspace_bytes_d(m, n, (2, 16, 32, 32, 1), 10, 1)
    assert e.value.code == tte.TT_EMB_ERR_ARG
    with pytest.raises(tte.TTEmbError) as e:      # merged core beyond 2^28 floats
        tte.tt_emb_workspace_bytes_d((1000, 1000, 100, 10, 10), (4, 4, 4, 2, 2),
                                     (1, 32, 32, 32, 32, 1), 10, 1)
    assert e.value.code == tte.TT_EMB_ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        tte.tt_emb_workspace_bytes_d(m, n, R[:-1], 10, 1)


def test_step_host_argument_checks(L):
    """The host-buffer step checks every argument of the calls it makes before it
    enqueues its first copy."""
    m, n, R = (10, 10, 10), (2, 4, 2), (1, 4, 4, 1)
    fake = 1 << 20
    cores = (ctypes.c_void_p * 3)(fake, fake, fake)
    P = ctypes.c_void_p
    need = tte.tt_emb_workspace_bytes(m, n, R, 100, 10)

    def batch(**kw):
        b = B.HostBatch()
        for name in ("h_indices", "h_offsets", "h_grad_out", "h_out", "d_indices", "d_offsets",
                     "d_grad_out", "d_out"):
            setattr(b, name, fake)
        b.nnz, b.num_bags = 100, 10
        for k, v in kw.items():
            setattr(b, k, v)
        return b

    def call(b, grads=cores, flags=0, ws=fake, ws_bytes=need):
        return L.tt_emb_step_host(cores, grads, *_shape(m, n, R),
                                  None if b is None else ctypes.byref(b), ctypes.c_float(0.1),
                                  flags, P(ws), ws_bytes, None, None)

    assert call(None) == tte.TT_EMB_ERR_ARG
    assert call(batch(), ws_bytes=need - 1) == tte.TT_EMB_ERR_WORKSPACE
    assert call(batch(), ws=fake + 8) == tte.TT_EMB_ERR_ARG          # workspace alignment
    assert call(batch(), flags=2) == tte.TT_EMB_ERR_ARG              # forward-only with a gradient
    assert call(batch(), flags=8) == tte.TT_EMB_ERR_ARG              # unknown flag
    assert call(batch(d_indices=fake + 4)) == tte.TT_EMB_ERR_ARG     # int64 indices alignment
    assert call(batch(d_indices=fake + 2), flags=tte.TT_EMB_INDICES_I32) == tte.TT_EMB_ERR_ARG
    assert call(batch(), grads=None) == tte.TT_EMB_ERR_ARG           # training needs gradients
    assert call(batch(d_grad_out=None)) == tte.TT_EMB_ERR_ARG
    assert call(batch(d_out=fake + 4)) == tte.TT_EMB_ERR_ARG         # out alignment
    assert call(batch(h_indices=None)) == tte.TT_EMB_ERR_ARG
    assert call(batch(d_offsets=None)) == tte.TT_EMB_ERR_ARG
    assert call(batch(num_bags=0)) == tte.TT_EMB_ERR_ARG             # lookups without bags
    assert call(batch(nnz=-1)) == tte.TT_EMB_ERR_ARG
    bad_shape = (ctypes.c_int32 * 4)(2, 4, 4, 1)
    assert L.tt_emb_step_host(cores, cores, _shape(m, n, R)[0], _shape(m, n, R)[1], bad_shape,
                              ctypes.byref(batch()), ctypes.c_float(0.1), 0, P(fake), need, None,
                              None) == tte.TT_EMB_ERR_ARG


def test_step_host_binding_checks_tensor_kinds(L):
    """The binding refuses host tensors of the wrong type and device staging that is not on
    the GPU before it calls the library."""
    import torch
    m, n, R = (10, 10, 10), (2, 4, 2), (1, 4, 4, 1)
    cores = [torch.zeros(4) for _ in range(3)]
    h_idx, h_off = torch.zeros(5, dtype=torch.int64), torch.tensor([0, 5], dtype=torch.int64)
    h_g, h_out = torch.zeros(1, 16), torch.zeros(1, 16)
    with pytest.raises(TypeError):                 # indices must be int64 or int32
        tte.tt_emb_step_host(cores, cores, m, n, R, h_idx.short(), h_off, h_g, h_out, h_idx, h_off,
                             h_g, h_out, 0.1, torch.zeros(8, dtype=torch.uint8), copy_stream=0)
    with pytest.raises(TypeError):                 # device staging must be CUDA tensors
        tte.tt_emb_step_host(cores, cores, m, n, R, h_idx, h_off, h_g, h_out, h_idx, h_off, h_g,
                             h_out, 0.1, torch.zeros(8, dtype=torch.uint8), copy_stream=0)
