"""The bf16 split of the cores kept in the workspace across calls: tt_emb_split,
tt_emb_sgd_ex (SGD and split in one pass) and forwards with TT_EMB_CORES_SPLIT,
through the C ABI.

A forward that uses planes made by tt_emb_split or tt_emb_sgd_ex must equal,
bit for bit, a forward that splits the same core values itself (the two
splits round identically); SGD with the split must update the cores exactly
as plain SGD; gradients after a forward on kept planes meet the usual bar.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_gb300 as tte
from tensor_train_compressed_gb300.inputs import make_custom, make_inputs

pytestmark = pytest.mark.gpu

BWD_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tensor_train_compressed_gb300 import build
    build.build()


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _ws(x, nnz=None, bags=None):
    n = tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz if nnz is None else nnz,
                                   x.num_bags if bags is None else bags)
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def _fwd(x, cores, idx, off, ws, flags=0):
    out = torch.full((off.numel() - 1, x.D), float("nan"), device="cuda")
    tte.tt_emb_forward_ex(cores, x.m, x.n, x.R, idx, off, None, "sum", out, ws, flags=flags)
    rc, bits = tte.tt_emb_get_error(ws)
    assert rc == tte.TT_EMB_OK, bits
    return out


def test_kept_planes_survive_other_batches():
    x = make_inputs(5, num_bags=1500)
    y = make_custom(x.m, x.n, x.R, num_bags=900, max_len=17, seed=5)
    cores = [_dev(c) for c in x.cores]
    ws = _ws(x)
    tte.tt_emb_split(cores, x.m, x.n, x.R, ws)
    for z in (x, y, x):                     # groupings of other batches keep the planes
        idx, off = _dev(z.indices), _dev(z.offsets)
        kept = _fwd(x, cores, idx, off, ws, flags=tte.TT_EMB_CORES_SPLIT)
        fresh = _fwd(x, cores, idx, off, _ws(x, z.nnz, z.num_bags))
        assert torch.equal(kept, fresh)


def test_fused_sgd_split_matches_sgd_and_a_fresh_split():
    x = make_inputs(5, num_bags=1200)
    idx, off, g = _dev(x.indices), _dev(x.offsets), _dev(x.grad_out)
    cores = [_dev(c) for c in x.cores]
    grads = [torch.zeros_like(c) for c in cores]
    ws = _ws(x)
    tte.tt_emb_split(cores, x.m, x.n, x.R, ws)
    _fwd(x, cores, idx, off, ws, flags=tte.TT_EMB_CORES_SPLIT)
    tte.tt_emb_backward(g, cores, x.m, x.n, x.R, idx, off, grads, ws, reuse_grouping=True)
    # the gradients of a forward on kept planes
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    for k in range(3):
        got = grads[k].cpu().numpy().astype(np.float64)
        assert np.abs(got - dref[k]).max() <= BWD_TOL * np.abs(dref[k]).max(), k
    # SGD with and without the split: the same core values, gradients reset
    plain = [c.clone() for c in cores]
    plain_grads = [d.clone() for d in grads]
    tte.tt_emb_sgd(plain, plain_grads, x.m, x.n, x.R, 0.01, zero_grads=True)
    tte.tt_emb_sgd_ex(cores, grads, x.m, x.n, x.R, 0.01, True, ws)
    for k in range(3):
        assert torch.equal(cores[k], plain[k])
        assert not grads[k].any()
    # the planes written by the SGD are the split of the updated cores
    kept = _fwd(x, cores, idx, off, ws, flags=tte.TT_EMB_CORES_SPLIT)
    fresh = _fwd(x, cores, idx, off, _ws(x))
    assert torch.equal(kept, fresh)


def test_split_is_a_no_op_without_tensor_core_kernels():
    x = make_custom((13, 11, 17), (4, 4, 4), (1, 16, 16, 1), num_bags=300, max_len=6, seed=3)
    cores = [_dev(c) for c in x.cores]
    ws = _ws(x)
    tte.tt_emb_split(cores, x.m, x.n, x.R, ws)
    idx, off = _dev(x.indices), _dev(x.offsets)
    a = _fwd(x, cores, idx, off, ws, flags=tte.TT_EMB_CORES_SPLIT)
    b = _fwd(x, cores, idx, off, ws)
    assert torch.equal(a, b)
    grads = [torch.zeros_like(c) for c in cores]
    plain = [c.clone() for c in cores]
    tte.tt_emb_sgd_ex(cores, grads, x.m, x.n, x.R, 0.5, False, ws)
    for k in range(3):
        assert torch.equal(cores[k], plain[k])
