"""The per-lookup forward of small forward-only batches (k_fwd_direct): each
row formed on its own from the three cores in FP32, the bag pooled in registers,
no grouping.  A forward-only call takes it when the batch's arithmetic in that
form is at most 2^27 multiply-adds and D <= 256.

Cases: the tiny and the one-lookup-bag workloads at full size, the three pooling
rules, shapes with odd n and R, empty bags, out-of-range indices and bad offsets
(reported as a grouping reports them), a backward that asks to reuse the call's
grouping (refused), the split of the cores the call leaves in the workspace,
and the batch size at which the grouped forward takes over.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_gb300 as tte
from tensor_train_compressed_gb300.inputs import make_custom, make_inputs

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-4
FO = tte.TT_EMB_FORWARD_ONLY


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tensor_train_compressed_gb300 import build
    build.build()


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _ws(x):
    return torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                       dtype=torch.uint8, device="cuda")


def _forward(x, ws, flags=FO, weights=None, mode="sum", cores=None):
    cores = cores if cores is not None else [_dev(c) for c in x.cores]
    out = torch.full((x.num_bags, x.D), float("nan"), device="cuda")
    psw = None if weights is None else _dev(weights.astype(np.float32))
    tte.tt_emb_forward_ex(cores, x.m, x.n, x.R, _dev(x.indices), _dev(x.offsets), psw, mode, out,
                          ws, flags=flags)
    rc, bits = tte.tt_emb_get_error(ws)
    return out.cpu().numpy(), rc, bits


def _method(x, ws):
    return tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, ws)["method"]


def _rel_err(a, ref):
    return float(np.abs(a.astype(np.float64) - ref).max() / max(np.abs(ref).max(), 1e-30))


@pytest.mark.parametrize("cfg", [1, 2])
def test_small_workloads_full_size(cfg):
    x = make_inputs(cfg)
    ws = _ws(x)
    out, rc, bits = _forward(x, ws)
    assert rc == tte.TT_EMB_OK, bits
    assert _method(x, ws) == "direct"
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    assert _rel_err(out, ref) <= FWD_TOL


@pytest.mark.parametrize("mode", ["sum", "weighted", "mean"])
def test_pooling_rules_odd_shape_and_empty_bags(mode):
    # D = 30 (one partial column of lanes), R1 = 7, R2 = 5; a tenth of the bags empty,
    # bags longer than 32 lookups (a second batch of lane-held indices)
    x = make_custom((9, 11, 13), (3, 5, 2), (1, 7, 5, 1), num_bags=400, max_len=45, seed=71,
                    empty_frac=0.1)
    ws = _ws(x)
    w = np.random.default_rng(5).uniform(-2, 2, x.nnz) if mode == "weighted" else None
    m = "mean" if mode == "mean" else "sum"
    out, rc, bits = _forward(x, ws, weights=w, mode=m)
    assert rc == tte.TT_EMB_OK, bits
    assert _method(x, ws) == "direct"
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, weights=w, mode=m)
    assert _rel_err(out, ref) <= FWD_TOL
    assert not out[np.diff(x.offsets) == 0].any()


def test_d_256_and_the_tensor_core_shape():
    # the largest D the kernel takes (8 columns per lane) and the benchmark's n and R
    for m, n, R, seed in [((20, 30, 40), (4, 8, 8), (1, 6, 5, 1), 72),
                          ((200, 240, 250), (4, 8, 4), (1, 32, 32, 1), 73)]:
        x = make_custom(m, n, R, num_bags=60, max_len=20, seed=seed)
        ws = _ws(x)
        out, rc, bits = _forward(x, ws)
        assert rc == tte.TT_EMB_OK, bits
        assert _method(x, ws) == "direct"
        ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets)
        assert _rel_err(out, ref) <= FWD_TOL


def test_out_of_range_indices_and_bad_offsets():
    x = make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=300, max_len=6, seed=5)
    bad = x.indices.copy()
    bad[::11] = 60
    bad[5] = -3
    x.indices = bad
    ws = _ws(x)
    out, rc, bits = _forward(x, ws, mode="mean")
    assert rc == tte.TT_EMB_ERR_INDEX and bits & 1
    ref = oracle.forward(x.cores, x.m, x.n, x.R, bad, x.offsets, strict=False, mode="mean")
    assert _rel_err(out, ref) <= FWD_TOL
    y = make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=50, max_len=4, seed=6)
    off = y.offsets.copy()
    off[10] = off[12] + 1          # not monotone
    y.offsets = off
    _, rc, bits = _forward(y, _ws(y))
    assert rc == tte.TT_EMB_ERR_OFFSETS and bits & 2
    z = make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=50, max_len=4, seed=7)
    z.offsets = z.offsets.copy()
    z.offsets[-1] -= 1             # the last offset is not nnz
    _, rc, bits = _forward(z, _ws(z))
    assert rc == tte.TT_EMB_ERR_OFFSETS and bits & 2


def test_backward_refuses_to_reuse_it():
    x = make_custom((9, 11, 13), (2, 4, 2), (1, 4, 4, 1), num_bags=100, max_len=5, seed=74)
    cores = [_dev(c) for c in x.cores]
    ws = _ws(x)
    _, rc, _ = _forward(x, ws, cores=cores)
    assert rc == tte.TT_EMB_OK and _method(x, ws) == "direct"
    grads = [torch.zeros_like(c) for c in cores]
    tte.tt_emb_backward(_dev(x.grad_out), cores, x.m, x.n, x.R, _dev(x.indices), _dev(x.offsets),
                        grads, ws, reuse_grouping=True)
    rc, bits = tte.tt_emb_get_error(ws)
    assert rc == tte.TT_EMB_ERR_REUSE and bits & 8
    assert not any(g.any() for g in grads)


def test_it_leaves_the_split_for_later_presplit_calls():
    # a small call without TT_EMB_CORES_SPLIT splits the cores; a grouped forward-only
    # call on the same workspace with the flag then reads that split
    small = make_inputs(3, num_bags=40)
    big = make_inputs(3, num_bags=3000)
    ws = _ws(big)
    cores = [_dev(c) for c in big.cores]
    _, rc, _ = _forward(small, ws, cores=cores)
    assert rc == tte.TT_EMB_OK and _method(small, ws) == "direct"
    out, rc, _ = _forward(big, ws, flags=FO | tte.TT_EMB_CORES_SPLIT, cores=cores)
    assert rc == tte.TT_EMB_OK and _method(big, ws) == "bitmap"
    ref, rc, _ = _forward(big, _ws(big), flags=FO, cores=cores)
    assert rc == tte.TT_EMB_OK and np.array_equal(out, ref)


def test_grouped_forward_takes_over_above_the_limit():
    # n = (4, 8, 4), R = 32: 36,864 multiply-adds per lookup, so 3,640 lookups are the
    # most the per-lookup kernel takes
    per = 4 * 8 * 32 * 32 + 128 * 32
    assert (1 << 27) // per == 3640
    for bags, direct in [(180, True), (190, False)]:          # fixed bag length 20
        x = make_inputs(3, num_bags=bags)
        ws = _ws(x)
        out, rc, _ = _forward(x, ws)
        assert rc == tte.TT_EMB_OK and (_method(x, ws) == "direct") == direct
        ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets)
        assert _rel_err(out, ref) <= FWD_TOL
    # the same batch without TT_EMB_FORWARD_ONLY is grouped (a backward may reuse it)
    x = make_inputs(3, num_bags=40)
    ws = _ws(x)
    _, rc, _ = _forward(x, ws, flags=0)
    assert rc == tte.TT_EMB_OK and _method(x, ws) != "direct"
