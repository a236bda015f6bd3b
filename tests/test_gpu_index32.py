"""int32 indices (TT_EMB_INDICES_I32): every grouping the code launches, the
per-lookup forward, the multi-table call, the host-buffer step and the module
class read int32 indices and give what the same calls give on the int64 copy of
those indices, bit for bit (outputs, groupings, status), out-of-range values
(negative ones included) reported the same way.  The int64 calls themselves are
checked against the oracle by the other GPU tests; here each int32 result is
also checked against the oracle at the usual tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_gb300 as tte
from tensor_train_compressed_gb300.inputs import make_custom, make_inputs

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-4
BWD_TOL = 1e-3
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


def _rel_err(a, ref):
    return float(np.abs(np.asarray(a, np.float64) - ref).max() / max(np.abs(ref).max(), 1e-30))


def _forward(x, idx, cores, flags):
    ws = _ws(x)
    out = torch.full((x.num_bags, x.D), float("nan"), device="cuda")
    tte.tt_emb_forward_ex(cores, x.m, x.n, x.R, idx, _dev(x.offsets), None, "sum", out, ws,
                          flags=flags)
    rc, bits = tte.tt_emb_get_error(ws)
    return out, ws, rc, bits


def _same_grouping(x, ws_a, ws_b):
    a = tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, ws_a)
    b = tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, ws_b)
    assert a["method"] == b["method"]
    for k in ("n_valid", "U_r", "U_12", "n_chunks", "status"):
        assert a[k] == b[k], k
    if a["method"] == "direct":
        return a["method"]
    keys = ["uid", "row_i3", "row_pair", "pair_row_start", "pair_i1", "pair_i2", "chunk_start",
            "chunk_order"]
    if a["method"] != "bitmap":
        keys += ["perm", "row_start"]
    for k in keys:
        assert np.array_equal(a[k], b[k]), k
    return a["method"]


@pytest.mark.parametrize("case", ["bitmap", "coop_sort", "multi_sort", "direct"])
def test_forward_int32_equals_int64(case):
    if case == "bitmap":
        x, flags = make_inputs(3), FO
    elif case == "coop_sort":
        x, flags = make_inputs(5, num_bags=3000), 0
    elif case == "multi_sort":
        # more lookups than the register-resident cooperative grouping holds
        x = make_custom((5, 6, 7), (4, 8, 4), (1, 32, 32, 1), num_bags=70000, max_len=40,
                        seed=19)
        flags = 0
    else:
        x, flags = make_inputs(1), FO
    cores = [_dev(c) for c in x.cores]
    assert x.indices.max() < 2 ** 31
    o64, w64, rc64, _ = _forward(x, _dev(x.indices), cores, flags)
    o32, w32, rc32, bits = _forward(x, _dev(x.indices.astype(np.int32)), cores, flags)
    assert rc64 == tte.TT_EMB_OK and rc32 == tte.TT_EMB_OK, bits
    assert _same_grouping(x, w64, w32) == case
    assert torch.equal(o32, o64)
    if case == "coop_sort":                 # the plain entry point takes int32 too
        o = torch.empty_like(o64)
        tte.tt_emb_forward(cores, x.m, x.n, x.R, _dev(x.indices.astype(np.int32)),
                           _dev(x.offsets), o, w32)
        assert torch.equal(o, o64)
    if case in ("direct", "coop_sort"):
        ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
        assert _rel_err(o32.cpu().numpy(), ref) <= FWD_TOL


@pytest.mark.parametrize("flags", [0, FO])
def test_out_of_range_int32_indices(flags):
    # negative values and values >= M in int32: reported, skipped, as in int64
    for x in (make_custom((9, 11, 13), (4, 8, 4), (1, 32, 32, 1), num_bags=2000, max_len=30,
                          seed=81),                                     # grouped
              make_custom((9, 11, 13), (4, 8, 4), (1, 32, 32, 1), num_bags=40, max_len=5,
                          seed=82)):                                    # per-lookup when FO
        bad = x.indices.copy()
        M = int(np.prod(x.m))
        bad[::7] = M + 3
        bad[1::11] = -5
        bad[2] = -(2 ** 31)
        x.indices = bad
        cores = [_dev(c) for c in x.cores]
        o64, w64, rc64, _ = _forward(x, _dev(bad), cores, flags)
        o32, w32, rc32, bits = _forward(x, _dev(bad.astype(np.int32)), cores, flags)
        assert rc64 == tte.TT_EMB_ERR_INDEX and rc32 == tte.TT_EMB_ERR_INDEX and bits & 1
        _same_grouping(x, w64, w32)
        assert torch.equal(o32, o64)
        ref = oracle.forward(x.cores, x.m, x.n, x.R, bad, x.offsets, strict=False)
        assert _rel_err(o32.cpu().numpy(), ref) <= FWD_TOL


def test_forward_tables_int32():
    xs = [make_inputs(4, table=t, num_bags=2000) for t in (0, 5)]
    outs = {}
    for dt in (np.int64, np.int32):
        tables = []
        for x in xs:
            tables.append(dict(cores=[_dev(c) for c in x.cores], m=x.m, n=x.n, R=x.R,
                               indices=_dev(x.indices.astype(dt)), offsets=_dev(x.offsets),
                               out=torch.empty((x.num_bags, x.D), device="cuda"),
                               workspace=_ws(x)))
        tte.tt_emb_forward_tables(tables)
        for t in tables:
            rc, bits = tte.tt_emb_get_error(t["workspace"])
            assert rc == tte.TT_EMB_OK, bits
        outs[dt] = [t["out"] for t in tables]
    for a, b in zip(outs[np.int64], outs[np.int32]):
        assert torch.equal(a, b)
    with pytest.raises(TypeError):          # one index dtype for all tables
        tte.tt_emb_forward_tables([dict(tables[0]), dict(tables[1], indices=tables[1]["indices"].long())])


def test_forward_tables_int32_tiled_shape():
    # n = (4, 4, 4), R = 16: the tables share the tiled FP32 chunk kernel
    xs = [make_custom((30, 40, 50), (4, 4, 4), (1, 16, 16, 1), num_bags=900, max_len=25,
                      seed=83 + t) for t in range(3)]
    outs = {}
    for dt in (np.int64, np.int32):
        tables = [dict(cores=[_dev(c) for c in x.cores], m=x.m, n=x.n, R=x.R,
                       indices=_dev(x.indices.astype(dt)), offsets=_dev(x.offsets),
                       out=torch.empty((x.num_bags, x.D), device="cuda"), workspace=_ws(x))
                  for x in xs]
        tte.tt_emb_forward_tables(tables)
        for t in tables:
            rc, bits = tte.tt_emb_get_error(t["workspace"])
            assert rc == tte.TT_EMB_OK, bits
        outs[dt] = [t["out"] for t in tables]
    for x, a, b in zip(xs, outs[np.int64], outs[np.int32]):
        assert torch.equal(a, b)
        ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets)
        assert _rel_err(b.cpu().numpy(), ref) <= FWD_TOL


def test_step_host_with_int32_indices():
    x = make_inputs(5, num_bags=1500)
    lr = 0.5
    cores0 = [_dev(c) for c in x.cores]
    res = {}
    for dt in (np.int64, np.int32):
        cores = [c.clone() for c in cores0]
        grads = [torch.zeros_like(c) for c in cores]
        ws = _ws(x)
        h_idx = torch.from_numpy(x.indices.astype(dt)).pin_memory()
        h_off = torch.from_numpy(x.offsets).pin_memory()
        h_g = torch.from_numpy(x.grad_out).pin_memory()
        h_out = torch.full((x.num_bags, x.D), float("nan")).pin_memory()
        d_idx = torch.empty(x.nnz, dtype=h_idx.dtype, device="cuda")
        d_off = torch.empty(x.num_bags + 1, dtype=torch.int64, device="cuda")
        d_g = torch.empty((x.num_bags, x.D), device="cuda")
        d_out = torch.empty((x.num_bags, x.D), device="cuda")
        tte.tt_emb_step_host(cores, grads, x.m, x.n, x.R, h_idx, h_off, h_g, h_out, d_idx, d_off,
                             d_g, d_out, lr, ws)
        torch.cuda.synchronize()
        rc, bits = tte.tt_emb_get_error(ws)
        assert rc == tte.TT_EMB_OK, bits
        res[dt] = (h_out.clone(), [c.clone() for c in cores])
    assert torch.equal(res[np.int32][0], res[np.int64][0])
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    for k in range(3):
        dg = (cores0[k].cpu().numpy().astype(np.float64) - res[np.int32][1][k].cpu().numpy()) / lr
        assert _rel_err(dg, dref[k]) <= BWD_TOL, k


def test_module_keeps_int32_indices():
    x = make_inputs(5, num_bags=800)
    a = tte.TTEmbeddingBag(x.cores, x.m, x.n, x.R)
    b = tte.TTEmbeddingBag(x.cores, x.m, x.n, x.R)
    out_a = a.forward(x.indices.astype(np.int32), x.offsets)
    assert a._batch[0].dtype == torch.int32
    out_b = b.forward(x.indices, x.offsets)
    assert torch.equal(out_a, out_b)
    a.backward(x.grad_out)               # reuses the grouping: no index is read
    b.backward(x.grad_out)
    torch.cuda.synchronize()
    a.check()
    for k in range(3):
        # the two gradients differ only in the order of their float atomics
        tol = 1e-4 * b.grads[k].abs().max().item()
        assert (a.grads[k] - b.grads[k]).abs().max().item() <= tol, k
    with pytest.raises(TypeError):       # a backward that regroups reads int64
        tte.tt_emb_backward(_dev(x.grad_out), a.cores, x.m, x.n, x.R, a._batch[0], a._batch[1],
                            a.grads, a.workspace, reuse_grouping=False)
