"""The backward chunk kernel's batches of rows: a chunk's rows beyond the first
24 (a hot prefix's, or those of a chunk of several prefixes) are staged by the
consumers, with the S rows and row i3 of each later batch loaded while the
batch before it is computed.  Hot prefixes of 25, 47, 48, 49, 72, 73, 100 and
200 unique rows (one more than a batch, batch multiples and their
neighbours, a whole i3 range) and a chunk of four 10-row prefixes of one i2
(40 rows, not hot) put every boundary of that staging under test; every
core-gradient element and every pooled output is compared with the oracle.
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
    return float(np.abs(np.asarray(a, np.float64) - ref).max() / max(np.abs(ref).max(), 1e-30))


def _batch_edge_inputs(seed):
    m = (4, 5, 200)
    x = make_custom(m, (4, 8, 4), (1, 32, 32, 1), num_bags=10, max_len=3, seed=seed)
    rng = np.random.default_rng(seed)
    # (i1, i2, unique rows): hot prefixes around multiples of the 24-row batch
    plan = [(0, 0, 25), (1, 0, 47), (2, 0, 48), (3, 0, 49), (0, 1, 72), (1, 1, 73),
            (2, 1, 100), (3, 2, 200)]
    plan += [(i1, 4, 10) for i1 in range(4)]           # one chunk of four prefixes, 40 rows
    plan += [(i1, 3, 3) for i1 in range(4)]            # small prefixes
    rows = []
    for i1, i2, k in plan:
        i3 = rng.choice(m[2], size=k, replace=False)
        r = (i1 * m[1] + i2) * m[2] + i3
        rows.append(np.repeat(r, rng.integers(1, 4, size=k)))   # 1-3 lookups per row
    idx = np.concatenate(rows).astype(np.int64)
    rng.shuffle(idx)
    nnz = idx.size
    cuts = np.sort(rng.choice(np.arange(1, nnz), size=nnz // 12, replace=False))
    x.indices = idx
    x.offsets = np.concatenate([[0], cuts, [nnz]]).astype(np.int64)
    x.grad_out = rng.standard_normal((x.num_bags, x.D)).astype(np.float32)
    return x


@pytest.mark.parametrize("seed", [91, 92])
def test_backward_later_batches_every_gradient(seed):
    x = _batch_edge_inputs(seed)
    g = oracle.group(x.indices, x.m)
    sizes = np.diff(g["pair_row_start"])
    assert {25, 47, 48, 49, 72, 73, 100, 200} <= set(sizes.tolist())
    cores = [_dev(c) for c in x.cores]
    idx, off = _dev(x.indices), _dev(x.offsets)
    ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((x.num_bags, x.D), device="cuda")
    tte.tt_emb_forward(cores, x.m, x.n, x.R, idx, off, out, ws)
    grads = [torch.zeros_like(c) for c in cores]
    tte.tt_emb_backward(_dev(x.grad_out), cores, x.m, x.n, x.R, idx, off, grads, ws,
                        reuse_grouping=True)
    rc, bits = tte.tt_emb_get_error(ws)
    assert rc == tte.TT_EMB_OK, bits
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    assert _rel_err(out.cpu().numpy(), ref) <= FWD_TOL
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    for k in range(3):
        assert _rel_err(grads[k].cpu().numpy(), dref[k]) <= BWD_TOL, k
