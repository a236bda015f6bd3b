"""Parity of the mean and weighted-sum pooling (forward, core gradients and the
per-sample weight gradient) of the CUDA path, through the C ABI, with the CPU
oracle.

Bars as for the sum: outputs within 1e-4 * max|ref|, core gradients within
1e-3 * max|ref| per core, weight gradients (one dot product of an output
gradient with a row per lookup) within 1e-4 * max|ref|.  Unit weights and
one-lookup bags must leave the sum bit for bit.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_gb300 as tte
from tensor_train_compressed_gb300.inputs import make_custom, make_inputs, make_sample_weights

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-4
BWD_TOL = 1e-3
DW_TOL = 1e-4


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


class _Run:
    """One forward_ex and one backward_ex on the device for inputs x."""

    def __init__(self, x, weights, mode, want_dw=True, reuse=True):
        self.cores = [_dev(c) for c in x.cores]
        self.idx, self.off = _dev(x.indices.astype(np.int64)), _dev(x.offsets.astype(np.int64))
        self.psw = None if weights is None else _dev(weights)
        self.ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                              dtype=torch.uint8, device="cuda")
        out = torch.full((x.num_bags, x.D), float("nan"), device="cuda")
        tte.tt_emb_forward_ex(self.cores, x.m, x.n, x.R, self.idx, self.off, self.psw, mode, out,
                              self.ws)
        self.rc_fwd, self.bits_fwd = tte.tt_emb_get_error(self.ws)
        self.out = out.cpu().numpy()
        grads = [torch.zeros_like(c) for c in self.cores]
        dw = None
        if want_dw and weights is not None:
            dw = torch.full((x.nnz,), float("nan"), device="cuda")
        tte.tt_emb_backward_ex(_dev(x.grad_out), self.cores, x.m, x.n, x.R, self.idx, self.off,
                               self.psw, mode, grads, dw, self.ws, reuse_grouping=reuse)
        self.rc_bwd, self.bits_bwd = tte.tt_emb_get_error(self.ws)
        self.dG = [g.cpu().numpy() for g in grads]
        self.dW = None if dw is None else dw.cpu().numpy()


def _check_against_oracle(x, weights, mode, run, strict=True, threads=8):
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=threads,
                         weights=weights, mode=mode, strict=strict)
    assert _rel_err(run.out, ref) <= FWD_TOL
    res = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets,
                          threads=threads, weights=weights, mode=mode,
                          want_dw=weights is not None, strict=strict)
    dref, dwref = res if weights is not None else (res, None)
    for k in range(3):
        assert _rel_err(run.dG[k], dref[k]) <= BWD_TOL, k
    if dwref is not None:
        assert _rel_err(run.dW, dwref) <= DW_TOL


SHAPES = [((3, 4, 5), (2, 3, 2), (1, 3, 2, 1)),        # generic kernels, D = 12
          ((7, 1, 9), (3, 1, 5), (1, 5, 2, 1)),        # D = 15: scalar pooling and gathers
          ((5, 6, 7), (4, 8, 4), (1, 32, 32, 1)),      # tensor-core kernels, D = 128
          ((13, 11, 17), (4, 4, 4), (1, 16, 16, 1)),   # tiled kernel, D = 64
          ((9, 8, 7), (4, 8, 4), (1, 64, 64, 1))]      # tiled kernel, R = 64


@pytest.mark.parametrize("mode", ["mean", "weighted"])
@pytest.mark.parametrize("shape", SHAPES)
def test_pooling_variants_edge_shapes(shape, mode):
    m, n, R = shape
    x = make_custom(m, n, R, num_bags=1500, max_len=9, seed=77, empty_frac=0.15)
    w = make_sample_weights(x.nnz, 78, -1.0, 2.0) if mode == "weighted" else None
    run = _Run(x, w, "sum" if w is not None else "mean")
    assert run.rc_fwd == tte.TT_EMB_OK and run.rc_bwd == tte.TT_EMB_OK
    assert not run.out[np.diff(x.offsets) == 0].any()
    _check_against_oracle(x, w, "sum" if w is not None else "mean", run)


@pytest.mark.parametrize("mode", ["mean", "weighted"])
def test_pooling_variants_config5_reduced(mode):
    """The training table's shape and index distribution, 3000 bags, all outputs compared."""
    x = make_inputs(5, num_bags=3000)
    w = make_sample_weights(x.nnz, 5) if mode == "weighted" else None
    pm = "sum" if w is not None else "mean"
    run = _Run(x, w, pm)
    assert run.rc_fwd == tte.TT_EMB_OK and run.rc_bwd == tte.TT_EMB_OK
    _check_against_oracle(x, w, pm, run)


def test_weighted_full_size_sampled():
    """Full training table and batch: 300 sampled bags (outputs and weight gradients) and
    four sampled core slices."""
    x = make_inputs(5)
    w = make_sample_weights(x.nnz, 9)
    run = _Run(x, w, "sum")
    assert run.rc_fwd == tte.TT_EMB_OK and run.rc_bwd == tte.TT_EMB_OK
    rng = np.random.default_rng(11)
    bags = np.sort(rng.choice(x.num_bags, size=300, replace=False))
    sel = np.concatenate([np.arange(x.offsets[b], x.offsets[b + 1]) for b in bags])
    off = np.concatenate([[0], np.cumsum(np.diff(x.offsets)[bags])])
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices[sel], off, threads=8, weights=w[sel])
    # tolerance scales: the oracle's own largest values over the sampled bags
    assert np.abs(run.out[bags] - ref).max() <= FWD_TOL * np.abs(ref).max()
    _, dwref = oracle.backward(x.grad_out[bags], x.cores, x.m, x.n, x.R, x.indices[sel], off,
                               threads=8, weights=w[sel], want_dw=True)
    assert np.abs(run.dW[sel] - dwref).max() <= DW_TOL * np.abs(dwref).max()
    r = x.indices
    i1, i2, i3 = r // (x.m[1] * x.m[2]), (r // x.m[2]) % x.m[1], r % x.m[2]
    for core, v in [(1, int(i1[3])), (2, int(i2[9])), (3, int(i3[0])), (3, int(i3[4242]))]:
        dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets,
                               threads=8, weights=w, filter_core=core,
                               filter_value=v)[core - 1][v]
        assert _rel_err(run.dG[core - 1][v], dref) <= BWD_TOL, (core, v)


@pytest.mark.parametrize("mode", ["mean", "weighted"])
def test_pooling_variants_full_size_every_element(mode):
    """The full training table and batch (655,893 lookups): every pooled output, every
    core-gradient element and (weighted) every weight-gradient element against the
    oracle, threaded over the host's cores."""
    x = make_inputs(5)
    w = make_sample_weights(x.nnz, 9) if mode == "weighted" else None
    m = "sum" if mode == "weighted" else "mean"
    run = _Run(x, w, m)
    assert run.rc_fwd == tte.TT_EMB_OK and run.rc_bwd == tte.TT_EMB_OK
    _check_against_oracle(x, w, m, run, threads=max(1, min(16, os.cpu_count() or 1)))


def test_unit_weights_and_single_lookup_bags_leave_the_sum_bitwise():
    x = make_inputs(5, num_bags=2000)
    cores = [_dev(c) for c in x.cores]
    idx, off = _dev(x.indices), _dev(x.offsets)
    ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                     dtype=torch.uint8, device="cuda")
    plain = torch.empty((x.num_bags, x.D), device="cuda")
    tte.tt_emb_forward(cores, x.m, x.n, x.R, idx, off, plain, ws)
    ones = torch.ones(x.nnz, device="cuda")
    wsum = torch.empty_like(plain)
    tte.tt_emb_forward_ex(cores, x.m, x.n, x.R, idx, off, ones, "sum", wsum, ws)
    assert torch.equal(plain, wsum)
    single = _dev(np.arange(x.nnz + 1, dtype=np.int64))
    a = torch.empty((x.nnz, x.D), device="cuda")
    b = torch.empty_like(a)
    tte.tt_emb_forward(cores, x.m, x.n, x.R, idx, single, a, ws)
    tte.tt_emb_forward_ex(cores, x.m, x.n, x.R, idx, single, None, "mean", b, ws)
    assert torch.equal(a, b)


def test_out_of_range_lookups_with_weights_and_mean():
    """Out-of-range lookups contribute nothing, count in a bag's length for the mean, and
    get a zero weight gradient."""
    x = make_custom((5, 6, 7), (4, 8, 4), (1, 32, 32, 1), num_bags=400, max_len=6, seed=15)
    bad = x.indices.copy()
    bad[::13] = 210
    bad[2] = -1
    x.indices = bad
    w = make_sample_weights(x.nnz, 16)
    for weights, mode in [(w, "sum"), (None, "mean")]:
        run = _Run(x, weights, mode)
        assert run.rc_fwd == tte.TT_EMB_ERR_INDEX and run.bits_fwd & 1
        _check_against_oracle(x, weights, mode, run, strict=False)
        if weights is not None:
            assert not run.dW[(bad < 0) | (bad >= 210)].any()


def test_weight_gradient_without_reused_grouping():
    x = make_inputs(5, num_bags=700)
    w = make_sample_weights(x.nnz, 21, -0.5, 1.5)
    run = _Run(x, w, "sum", reuse=False)
    assert run.rc_bwd == tte.TT_EMB_OK
    _check_against_oracle(x, w, "sum", run)


def test_owner_object_mean_and_weights():
    x = make_inputs(5, num_bags=500)
    mean = tte.TTEmbeddingBag(x.cores, x.m, x.n, x.R, mode="mean")
    out = mean.forward(torch.from_numpy(x.indices), torch.from_numpy(x.offsets))
    mean.backward(torch.from_numpy(x.grad_out))
    mean.check()
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8, mode="mean")
    assert _rel_err(out.cpu().numpy(), ref) <= FWD_TOL
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8,
                           mode="mean")
    for k in range(3):
        assert _rel_err(mean.grads[k].cpu().numpy(), dref[k]) <= BWD_TOL
    w = make_sample_weights(x.nnz, 22)
    emb = tte.TTEmbeddingBag(x.cores, x.m, x.n, x.R)
    out = emb.forward(x.indices, x.offsets, per_sample_weights=w)
    dw = torch.empty(x.nnz, device="cuda")
    emb.backward(x.grad_out, grad_weights=dw)
    emb.check()
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8, weights=w)
    assert _rel_err(out.cpu().numpy(), ref) <= FWD_TOL
    dref, dwref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets,
                                  threads=8, weights=w, want_dw=True)
    for k in range(3):
        assert _rel_err(emb.grads[k].cpu().numpy(), dref[k]) <= BWD_TOL
    assert _rel_err(dw.cpu().numpy(), dwref) <= DW_TOL
