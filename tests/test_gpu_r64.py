"""Tables with n = (4, 8, 4) and R1 = R2 = 64: the tensor-core chunk kernel that
works each chunk in two column halves (k_fwd_mma64), alone and over several
tables in one launch, against the oracle.

Cases: chunks with more rows than the kernel stages (rows read from the global
split planes), hot prefixes split into pieces that reuse a checkpointed prefix
partial, the forward-only and pre-split flags (bit-identical outputs), and
the eight-table workload at full size on every output.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_gb300 as tte
from tensor_train_compressed_gb300.inputs import make_custom, make_inputs

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-4
N, R = (4, 8, 4), (1, 64, 64, 1)


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


def _forward(x, ws, flags=0, split=False):
    cores = [_dev(c) for c in x.cores]
    idx, off = _dev(x.indices), _dev(x.offsets)
    out = torch.full((x.num_bags, x.D), float("nan"), device="cuda")
    if split:
        tte.tt_emb_split(cores, x.m, x.n, x.R, ws)
    tte.tt_emb_forward_ex(cores, x.m, x.n, x.R, idx, off, None, "sum", out, ws, flags=flags)
    rc, bits = tte.tt_emb_get_error(ws)
    assert rc == tte.TT_EMB_OK, bits
    return out.cpu().numpy()


def _rel_err(a, ref):
    return float(np.abs(a.astype(np.float64) - ref).max() / max(np.abs(ref).max(), 1e-30))


def test_chunks_with_more_rows_than_are_staged():
    # 32 prefixes of 30 rows each, four prefixes of one i2 per chunk: 120-row chunks,
    # more than the 32 G3 rows a chunk stages
    x = make_custom((8, 4, 30), N, R, num_bags=3000, max_len=12, seed=21)
    ws = _ws(x)
    out = _forward(x, ws)
    g = tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, ws)
    assert np.diff(g["chunk_start"]).max() > 32
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    assert _rel_err(out, ref) <= FWD_TOL
    grp = oracle.group(x.indices, x.m)
    assert g["U_r"] == grp["U_r"] and np.array_equal(g["uid"], grp["uid"])


def test_hot_prefixes_reuse_checkpointed_partials():
    # 6 prefixes of about 15,000 rows each: 32-row pieces, later pieces reuse the
    # first piece's P2 from its L2 slot (the buffer has spare rows for slots).  A
    # piece reuses the slot only if its owner has published it by the time the
    # piece is staged, so the batch gives each CTA many pieces to work
    x = make_custom((3, 2, 5000), N, R, num_bags=12000, max_len=14, seed=22)
    ws = _ws(x)
    out = _forward(x, ws)
    g = tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, ws)
    assert g["U_12"] == 6 and g["ckpt_reused"] > 0
    assert g["ckpt_reused"] <= g["n_chunks"] - 6
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    assert _rel_err(out, ref) <= FWD_TOL
    # a reused partial is the same bf16 planes: the same output with and without reuse,
    # through the key-bitmap grouping of a forward-only call and a pre-made split
    ws2 = _ws(x)
    out2 = _forward(x, ws2, flags=tte.TT_EMB_FORWARD_ONLY | tte.TT_EMB_CORES_SPLIT, split=True)
    assert tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, ws2)["method"] == "bitmap"
    assert np.array_equal(out, out2)


def test_few_rows_per_prefix_and_empty_bags():
    # prefixes of one to three rows (pairs with a single row), many short chunks
    x = make_custom((40, 50, 3), N, R, num_bags=2000, max_len=5, seed=23, empty_frac=0.1)
    ws = _ws(x)
    out = _forward(x, ws)
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    assert _rel_err(out, ref) <= FWD_TOL
    assert not out[np.diff(x.offsets) == 0].any()


def _table(x):
    return dict(cores=[_dev(c) for c in x.cores], m=x.m, n=x.n, R=x.R, indices=_dev(x.indices),
                offsets=_dev(x.offsets),
                out=torch.full((x.num_bags, x.D), float("nan"), device="cuda"), workspace=_ws(x))


def test_tables_with_presplit_cores_are_bit_identical():
    xs = [make_custom(m, N, R, num_bags=600, max_len=20, seed=30 + k)
          for k, m in enumerate([(9, 8, 7), (3, 2, 900), (20, 20, 20)])]
    a = [_table(x) for x in xs]
    tte.tt_emb_forward_tables(a)
    b = [_table(x) for x in xs]
    for x, t in zip(xs, b):
        tte.tt_emb_split(t["cores"], x.m, x.n, x.R, t["workspace"])
    tte.tt_emb_forward_tables(b, flags=tte.TT_EMB_CORES_SPLIT)
    for ta, tb in zip(a, b):
        assert torch.equal(ta["out"], tb["out"])
    with pytest.raises(tte.TTEmbError) as e:
        tte.tt_emb_forward_tables(b, flags=2)
    assert e.value.code == tte.TT_EMB_ERR_ARG


def test_eight_tables_full_size_every_output():
    """All eight config-4 tables at full size in one tt_emb_forward_tables call (the
    bench's launch configuration): every pooled output element of every table against
    the oracle, scaled by the oracle's largest value for that table."""
    xs = [make_inputs(4, table=k) for k in range(8)]
    tables = [_table(x) for x in xs]
    tte.tt_emb_forward_tables(tables)
    reused = 0
    threads = max(1, min(16, os.cpu_count() or 1))
    for x, t in zip(xs, tables):
        rc, bits = tte.tt_emb_get_error(t["workspace"])
        assert rc == tte.TT_EMB_OK, bits
        g = tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, t["workspace"])
        reused += g["ckpt_reused"]
        ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=threads)
        got = t["out"].cpu().numpy().astype(np.float64)
        assert np.abs(got - ref).max() <= FWD_TOL * np.abs(ref).max()
    assert reused > 0
