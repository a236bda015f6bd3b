"""tt_emb_forward_tables: several tables in one call, through the C ABI.

Every table's output must equal, bit for bit, what tt_emb_forward writes for
that table alone (the same kernels compute the same rows and sums; only the
order in which chunks are taken differs), and match the oracle on sampled
bags.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_gb300 as tte
from tensor_train_compressed_gb300.inputs import make_custom, make_inputs

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tensor_train_compressed_gb300 import build
    build.build()


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _table(x):
    ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                     dtype=torch.uint8, device="cuda")
    return dict(cores=[_dev(c) for c in x.cores], m=x.m, n=x.n, R=x.R, indices=_dev(x.indices),
                offsets=_dev(x.offsets),
                out=torch.full((x.num_bags, x.D), float("nan"), device="cuda"), workspace=ws)


def _alone(t):
    out = torch.full_like(t["out"], float("nan"))
    ws = torch.empty_like(t["workspace"])
    tte.tt_emb_forward(t["cores"], t["m"], t["n"], t["R"], t["indices"], t["offsets"], out, ws)
    return out


def _check_all(xs, tables):
    for t in tables:
        rc, bits = tte.tt_emb_get_error(t["workspace"])
        assert rc == tte.TT_EMB_OK, bits
    for x, t in zip(xs, tables):
        assert torch.equal(t["out"], _alone(t))


def test_eight_tables_of_the_multi_table_workload():
    xs = [make_inputs(4, table=k, num_bags=1500) for k in range(8)]
    tables = [_table(x) for x in xs]
    tte.tt_emb_forward_tables(tables)
    # the tables dense in their rows (at most 8 bitmap words per lookup) are grouped by
    # the key bitmap of a forward-only call, the others by the radix sort
    for x, t in zip(xs, tables):
        g = tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, t["workspace"])
        dense = (int(np.prod(x.m)) + 31) // 32 <= 8 * x.nnz
        assert g["method"] == ("bitmap" if dense else "coop_sort"), (x.m, g["method"])
    _check_all(xs, tables)
    rng = np.random.default_rng(3)
    for k in (0, 7):
        x = xs[k]
        bags = np.sort(rng.choice(x.num_bags, size=200, replace=False))
        idx = np.concatenate([x.indices[x.offsets[b]:x.offsets[b + 1]] for b in bags])
        off = np.concatenate([[0], np.cumsum(np.diff(x.offsets)[bags])])
        ref = oracle.forward(x.cores, x.m, x.n, x.R, idx, off, threads=8)
        got = tables[k]["out"].cpu().numpy()[bags].astype(np.float64)
        assert np.abs(got - ref).max() <= FWD_TOL * max(np.abs(ref).max(), 1e-30)


def test_tables_with_no_lookups_empty_bags_and_other_factors():
    n, R = (4, 8, 4), (1, 64, 64, 1)
    xs = [make_custom((9, 8, 7), n, R, num_bags=400, max_len=9, seed=1, empty_frac=0.2),
          make_custom((3, 4, 5), n, R, num_bags=50, max_len=0, seed=2),          # no lookups
          make_custom((30, 2, 41), n, R, num_bags=700, max_len=25, seed=3),
          make_custom((1, 1, 1), n, R, num_bags=10, max_len=4, seed=4)]
    tables = [_table(x) for x in xs]
    tte.tt_emb_forward_tables(tables)
    _check_all(xs, tables)
    assert not tables[1]["out"].any()
    for x, t in zip(xs, tables):
        if x.nnz:
            ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
            got = t["out"].cpu().numpy().astype(np.float64)
            assert np.abs(got - ref).max() <= FWD_TOL * max(np.abs(ref).max(), 1e-30)


def test_tensor_core_shape_runs_table_by_table():
    xs = [make_custom((5, 6, 7), (4, 8, 4), (1, 32, 32, 1), num_bags=300, max_len=8, seed=s)
          for s in (5, 6, 7)]
    tables = [_table(x) for x in xs]
    tte.tt_emb_forward_tables(tables)
    _check_all(xs, tables)


def test_shared_workspace_and_mixed_ranks_are_refused():
    a = make_custom((9, 8, 7), (4, 8, 4), (1, 64, 64, 1), num_bags=50, max_len=3, seed=8)
    b = make_custom((9, 8, 7), (4, 8, 4), (1, 32, 32, 1), num_bags=50, max_len=3, seed=9)
    ta, tb = _table(a), _table(a)
    tb["workspace"] = ta["workspace"]
    with pytest.raises(tte.TTEmbError) as e:
        tte.tt_emb_forward_tables([ta, tb])
    assert e.value.code == tte.TT_EMB_ERR_ARG
    with pytest.raises(tte.TTEmbError) as e:
        tte.tt_emb_forward_tables([_table(a), _table(b)])
    assert e.value.code == tte.TT_EMB_ERR_ARG
