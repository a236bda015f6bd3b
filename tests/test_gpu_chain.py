"""Chains of d > 3 cores through the C ABI (tt_emb_*_d) against the d-core
oracle: forward within 1e-4 * max|ref| over the whole output, every core's
gradient within 1e-3 * max|ref|, with the grouping reused and rebuilt, and the
chain's SGD.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_gb300 as tte
from tensor_train_compressed_gb300.inputs import make_custom

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-4
BWD_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tensor_train_compressed_gb300 import build
    build.build()


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _rel_err(a, ref):
    return float(np.abs(a.astype(np.float64) - ref).max() / max(np.abs(ref).max(), 1e-30))


SHAPES = [
    # four cores whose three-core view (120, 20, 30), n (4, 8, 4), R 32 runs the tensor-core kernels
    ((10, 12, 20, 30), (2, 2, 8, 4), (1, 16, 32, 32, 1)),
    # four cores on the shape-generic kernels
    ((5, 4, 6, 7), (2, 1, 3, 2), (1, 3, 4, 2, 1)),
    # five and six cores
    ((3, 4, 5, 6, 7), (1, 2, 2, 2, 2), (1, 2, 3, 4, 2, 1)),
    ((2, 3, 2, 3, 2, 5), (2, 1, 2, 1, 2, 2), (1, 2, 2, 3, 2, 3, 1)),
]


@pytest.mark.parametrize("reuse", [True, False])
@pytest.mark.parametrize("shape", SHAPES)
def test_chain_forward_backward(shape, reuse):
    m, n, R = shape
    x = make_custom(m, n, R, num_bags=700, max_len=9, seed=81, empty_frac=0.1,
                    dist=("zipf", 1.1, "identity"))
    cores = [_dev(c) for c in x.cores]
    idx, off = _dev(x.indices), _dev(x.offsets)
    ws = torch.empty(tte.tt_emb_workspace_bytes_d(m, n, R, x.nnz, x.num_bags), dtype=torch.uint8,
                     device="cuda")
    out = torch.full((x.num_bags, x.D), float("nan"), device="cuda")
    tte.tt_emb_forward_d(cores, m, n, R, idx, off, out, ws)
    ref = oracle.forward_d(x.cores, m, n, R, x.indices, x.offsets)
    assert _rel_err(out.cpu().numpy(), ref) <= FWD_TOL
    grads = [torch.zeros_like(c) for c in cores]
    tte.tt_emb_backward_d(_dev(x.grad_out), cores, m, n, R, idx, off, grads, ws,
                          reuse_grouping=reuse)
    dref = oracle.backward_d(x.grad_out, x.cores, m, n, R, x.indices, x.offsets)
    for k in range(len(m)):
        assert _rel_err(grads[k].cpu().numpy(), dref[k]) <= BWD_TOL, k
    rc, bits = tte.tt_emb_get_error(ws)
    assert rc == tte.TT_EMB_OK, bits


def test_chain_out_of_range_index_is_reported():
    m, n, R = (5, 4, 6, 7), (2, 1, 3, 2), (1, 3, 4, 2, 1)
    x = make_custom(m, n, R, num_bags=40, max_len=5, seed=84)
    bad = x.indices.copy()
    bad[3] = int(np.prod(m))
    cores = [_dev(c) for c in x.cores]
    ws = torch.empty(tte.tt_emb_workspace_bytes_d(m, n, R, x.nnz, x.num_bags), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((x.num_bags, x.D), device="cuda")
    tte.tt_emb_forward_d(cores, m, n, R, _dev(bad), _dev(x.offsets), out, ws)
    rc, bits = tte.tt_emb_get_error(ws)
    assert rc == tte.TT_EMB_ERR_INDEX and bits & 1
    ref = oracle.forward_d(x.cores, m, n, R, bad, x.offsets, strict=False)
    assert _rel_err(out.cpu().numpy(), ref) <= FWD_TOL


def test_chain_sgd_updates_every_core():
    m, n, R = (3, 4, 5, 6, 7), (1, 2, 2, 2, 2), (1, 2, 3, 4, 2, 1)
    x = make_custom(m, n, R, num_bags=10, max_len=3, seed=82)
    cores = [_dev(c) for c in x.cores]
    rng = np.random.default_rng(83)
    dg = [rng.standard_normal(c.shape).astype(np.float32) for c in x.cores]
    grads = [_dev(g) for g in dg]
    tte.tt_emb_sgd_d(cores, grads, m, n, R, 0.25, zero_grads=True)
    for k in range(len(m)):
        exp = x.cores[k] - np.float32(0.25) * dg[k]
        assert np.allclose(cores[k].cpu().numpy(), exp, rtol=0, atol=1e-6)
        assert not grads[k].any()
