"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars: the grouping is bit-exact; the fp32 forward is within
1e-4 * max|ref| over the whole output; fp32 core gradients (float atomics)
within 1e-3 * max|ref| per core; SGD within 0.01 * 1e-3 * max|dG_ref| plus
fp32 rounding of the cores.  Full-size configurations are checked on sampled
bags (forward) and on sampled core slices (backward), computed one by one by
the oracle.
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
BWD_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tensor_train_compressed_gb300 import build
    build.build()


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _gpu_forward(x, ws=None, flags=0):
    cores = [_dev(c) for c in x.cores]
    idx, off = _dev(x.indices.astype(np.int64)), _dev(x.offsets.astype(np.int64))
    B = x.num_bags
    need = tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, B)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.full((B, x.D), float("nan"), dtype=torch.float32, device="cuda")
    if flags:
        tte.tt_emb_forward_ex(cores, x.m, x.n, x.R, idx, off, None, "sum", out, ws, flags=flags)
    else:
        tte.tt_emb_forward(cores, x.m, x.n, x.R, idx, off, out, ws)
    rc, bits = tte.tt_emb_get_error(ws)
    return out.cpu().numpy(), rc, bits, dict(cores=cores, idx=idx, off=off, ws=ws)


def _gpu_backward(x, st):
    grads = [torch.zeros_like(c) for c in st["cores"]]
    tte.tt_emb_backward(_dev(x.grad_out), st["cores"], x.m, x.n, x.R, st["idx"], st["off"],
                        grads, st["ws"], reuse_grouping=True)
    rc, bits = tte.tt_emb_get_error(st["ws"])
    assert rc == tte.TT_EMB_OK, bits
    # the backward writes the bag of every lookup into the workspace
    g = tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, st["ws"])
    assert np.array_equal(g["bag_of"], np.repeat(np.arange(x.num_bags), np.diff(x.offsets)))
    return [g.cpu().numpy() for g in grads]


def _rel_err(a, ref):
    return float(np.abs(a.astype(np.float64) - ref).max() / max(np.abs(ref).max(), 1e-30))


def _check_grouping(x, ws, method=None):
    """The grouping in ``ws`` against the oracle's, bit for bit: unique rows, prefixes,
    the unique row of every lookup and (except for a forward-only key-bitmap grouping,
    which has none) the lookups of every row in position order with their CSR offsets;
    chunks valid, each chunk's prefixes sharing one i2, the claim order a permutation of
    the chunks.  ``method`` (if given) must be the one that ran."""
    ref = oracle.group(x.indices, x.m)
    g = tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, ws)
    if method is not None:
        assert g["method"] == method, g["method"]
    assert g["n_valid"] == ref["n_valid"] and g["U_r"] == ref["U_r"] and g["U_12"] == ref["U_12"]
    nv = ref["n_valid"]
    if g["method"] != "bitmap":                  # a forward-only grouping has no lookup lists
        assert np.array_equal(g["row_start"], ref["row_start"])
        assert np.array_equal(g["perm"][:nv], ref["perm"])
    assert np.array_equal(g["row_pair"], ref["row_pair"])
    assert np.array_equal(g["pair_row_start"], ref["pair_row_start"])
    assert np.array_equal(g["pair_i1"], ref["pair_i1"])
    assert np.array_equal(g["pair_i2"], ref["pair_i2"])
    assert np.array_equal(g["uid"], ref["uid"])
    m2, m3 = x.m[1], x.m[2]
    rows = (g["pair_i1"][g["row_pair"]].astype(np.int64) * m2 + g["pair_i2"][g["row_pair"]]) * m3 \
        + g["row_i3"]
    assert np.array_equal(rows, ref["row_index"])
    # chunks partition the unique rows, each chunk's prefixes share one i2
    cs = g["chunk_start"]
    assert cs[0] == 0 and cs[-1] == g["U_r"] and np.all(np.diff(cs) > 0)
    for c in range(g["n_chunks"]):
        p = g["row_pair"][cs[c]:cs[c + 1]]
        assert np.unique(g["pair_i2"][p]).size == 1
    order = g["chunk_order"]
    assert np.array_equal(np.sort(order), np.arange(g["n_chunks"]))
    return g


def _sample_bags(x, bags):
    idx = np.concatenate([x.indices[x.offsets[b]:x.offsets[b + 1]] for b in bags])
    off = np.concatenate([[0], np.cumsum([x.offsets[b + 1] - x.offsets[b] for b in bags])])
    return idx, off


# ------------------------------------------------------------------ grouping + forward


@pytest.mark.parametrize("cfg", [1, 2])
def test_forward_small_configs_full(cfg):
    x = make_inputs(cfg)
    out, rc, _, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    assert _rel_err(out, ref) <= FWD_TOL
    _check_grouping(x, st["ws"])


def test_config1_against_materialised_table():
    x = make_inputs(1)
    out, rc, _, _ = _gpu_forward(x)
    G1, G2, G3 = (c.astype(np.float64) for c in x.cores)
    T = np.einsum("xpa,yaqb,zbr->xyzpqr", G1[:, 0], G2, G3[:, :, :, 0]).reshape(1000, 16)
    ref = np.stack([T[x.indices[x.offsets[b]:x.offsets[b + 1]]].sum(0) for b in range(64)])
    assert _rel_err(out, ref) <= FWD_TOL


@pytest.mark.parametrize("cfg,bags", [(3, 3000), (5, 3000), (4, 3000)])
def test_forward_reduced_configs_full_compare(cfg, bags):
    """Config shapes and index distributions, fewer bags: every output compared."""
    x = make_inputs(cfg, table=3 if cfg == 4 else 0, num_bags=bags)
    out, rc, _, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    assert _rel_err(out, ref) <= FWD_TOL
    _check_grouping(x, st["ws"])


@pytest.mark.parametrize("cfg,table", [(3, 0), (5, 0), (4, 0), (4, 7)])
def test_forward_full_size_sampled(cfg, table):
    x = make_inputs(cfg, table=table)
    out, rc, _, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK
    rng = np.random.default_rng(100 + cfg)
    bags = np.sort(rng.choice(x.num_bags, size=300, replace=False))
    idx, off = _sample_bags(x, bags)
    ref = oracle.forward(x.cores, x.m, x.n, x.R, idx, off, threads=8)
    # the tolerance scale is the oracle's own largest pooled value over the sampled bags
    assert np.abs(out[bags] - ref).max() <= FWD_TOL * np.abs(ref).max()
    assert np.isfinite(out).all()
    # the full-size grouping (the register-resident variant the full batch selects)
    # against the oracle's, element by element
    g = _check_grouping(x, st["ws"])
    assert g["U_r"] == np.unique(x.indices).size and g["n_valid"] == x.nnz
    if cfg in (3, 5):
        # the later pieces of hot prefixes took their P2 from the L2 checkpoint (the
        # sampled bags above include rows made that way: the hot rows are in most bags)
        assert g["method"] == "coop_sort"
        cs = g["chunk_start"]
        pieces = sum(1 for c in range(g["n_chunks"])
                     if g["pair_row_start"][g["row_pair"][cs[c]]] != cs[c])
        assert 0 < g["ckpt_reused"] <= pieces, (g["ckpt_reused"], pieces)


def _oracle_threads():
    return max(1, min(16, os.cpu_count() or 1))


@pytest.mark.parametrize("cfg,table,mapping", [(3, 0, None), (5, 0, None), (4, 7, None),
                                               (3, 0, "permuted")])
def test_forward_full_size_every_output(cfg, table, mapping):
    """The whole batch at full size (32,768 bags; config 4: its largest table, 4e7 rows;
    the 12M-row batch also with its Zipf ranks mapped through a random row permutation)
    in the launch configuration the bench times: every pooled output element against
    the oracle, scaled by the oracle's largest value."""
    x = make_inputs(cfg, table=table, mapping=mapping)
    out, rc, _, _ = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=_oracle_threads())
    assert np.abs(out - ref).max() <= FWD_TOL * np.abs(ref).max()


def test_backward_full_size_every_gradient():
    """The 48M-row training batch at full size: every element of the three core
    gradients against the oracle's, each scaled by the oracle's largest value."""
    x = make_inputs(5, with_grad=True)
    _, rc, _, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK
    dG = _gpu_backward(x, st)
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets,
                           threads=_oracle_threads())
    for k in range(3):
        assert np.abs(dG[k] - dref[k]).max() <= BWD_TOL * np.abs(dref[k]).max(), k


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("items", [4, 8, 12, 16])
def test_bitmap_grouping_every_variant(items):
    """The key-bitmap grouping of a forward-only call keeps ceil(nnz / SMs) lookups per
    CTA in registers, 4, 8, 12 or 16 per thread (512 threads); the batch size picks the
    variant.  Each one runs here on the benchmark table's shape and index distribution
    (dense in the table: at most 8 bitmap words per lookup), is compared with the
    oracle's grouping, and its output equals the sort-grouped forward's bit for bit."""
    G = _sms()
    lo, hi = G * 512 * {4: 0, 8: 4, 12: 8, 16: 12}[items], G * 512 * items
    target = (lo + hi) // 2 if items > 4 else hi - 1000
    x = make_inputs(3, num_bags=target // 20)                # fixed bag length 20
    assert lo < x.nnz <= hi
    out, rc, _, st = _gpu_forward(x, flags=tte.TT_EMB_FORWARD_ONLY)
    assert rc == tte.TT_EMB_OK
    _check_grouping(x, st["ws"], method="bitmap")
    ref_out, rc, _, _ = _gpu_forward(x)                      # the same batch, sort-grouped
    assert rc == tte.TT_EMB_OK and np.array_equal(out, ref_out)
    rng = np.random.default_rng(items)
    bags = np.sort(rng.choice(x.num_bags, size=200, replace=False))
    idx, off = _sample_bags(x, bags)
    ref = oracle.forward(x.cores, x.m, x.n, x.R, idx, off, threads=8)
    assert np.abs(out[bags] - ref).max() <= FWD_TOL * np.abs(ref).max()


@pytest.mark.parametrize("items", [4, 8, 12, 16])
def test_sort_grouping_every_cooperative_variant(items):
    """The one-launch radix-sort grouping (4, 8, 12 or 16 lookups per thread), which
    serves batches sparse in their table: 343M rows = 700^3, so the key bitmap would
    take more than 8 words per lookup.  Its grouping must equal the oracle's in every
    array, the order of each row's lookups included."""
    G = _sms()
    lo, hi = G * 512 * (items - 4), G * 512 * items
    target = (lo + hi) // 2 if items > 4 else hi - 1000
    x = make_custom((700, 700, 700), (4, 8, 4), (1, 32, 32, 1), num_bags=target // 20,
                    max_len=39, seed=800 + items, dist=("zipf", 1.2, "identity"))
    assert lo < x.nnz <= hi and (700 ** 3 + 31) // 32 > 8 * x.nnz
    out, rc, _, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK
    _check_grouping(x, st["ws"], method="coop_sort")
    rng = np.random.default_rng(items)
    bags = np.sort(rng.choice(x.num_bags, size=200, replace=False))
    idx, off = _sample_bags(x, bags)
    ref = oracle.forward(x.cores, x.m, x.n, x.R, idx, off, threads=8)
    assert np.abs(out[bags] - ref).max() <= FWD_TOL * np.abs(ref).max()


@pytest.mark.parametrize("cfg", [3, 5])
def test_forward_only_grouping_full_size(cfg):
    """A forward-only call (TT_EMB_FORWARD_ONLY) groups without the per-row lookup
    lists: its output equals the plain forward's bit for bit, and its grouping (unique
    rows, prefixes, uid, chunks) equals the oracle's."""
    x = make_inputs(cfg)
    ref_out, rc, _, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK
    out = torch.full((x.num_bags, x.D), float("nan"), dtype=torch.float32, device="cuda")
    tte.tt_emb_forward_ex(st["cores"], x.m, x.n, x.R, st["idx"], st["off"], None, "sum", out,
                          st["ws"], flags=tte.TT_EMB_FORWARD_ONLY)
    rc, bits = tte.tt_emb_get_error(st["ws"])
    assert rc == tte.TT_EMB_OK, bits
    assert np.array_equal(out.cpu().numpy(), ref_out)
    _check_grouping(x, st["ws"], method="bitmap")


def test_backward_refuses_a_forward_only_grouping():
    """A backward that reuses the grouping of a forward-only call reports
    TT_EMB_ERR_REUSE and leaves the core gradients untouched; rebuilding the grouping
    (reuse_grouping=False) then gives the right gradients."""
    x = make_inputs(3, num_bags=3000, with_grad=True)     # dense in its table: key bitmap
    cores = [_dev(c) for c in x.cores]
    idx, off = _dev(x.indices), _dev(x.offsets)
    ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((x.num_bags, x.D), dtype=torch.float32, device="cuda")
    tte.tt_emb_forward_ex(cores, x.m, x.n, x.R, idx, off, None, "sum", out, ws,
                          flags=tte.TT_EMB_FORWARD_ONLY)
    assert tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, ws)["method"] == "bitmap"
    grads = [torch.zeros_like(c) for c in cores]
    tte.tt_emb_backward(_dev(x.grad_out), cores, x.m, x.n, x.R, idx, off, grads, ws,
                        reuse_grouping=True)
    rc, bits = tte.tt_emb_get_error(ws)
    assert rc == tte.TT_EMB_ERR_REUSE and bits & 8
    assert not any(g.any() for g in grads)
    tte.tt_emb_backward(_dev(x.grad_out), cores, x.m, x.n, x.R, idx, off, grads, ws,
                        reuse_grouping=False)
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    for k in range(3):
        assert _rel_err(grads[k].cpu().numpy(), dref[k]) <= BWD_TOL, k


def test_large_batch_uses_the_multi_kernel_grouping():
    """1.3M lookups exceed the register-resident cooperative grouping: the multi-kernel
    grouping path must give the same bit-exact grouping and forward."""
    x = make_custom((5, 6, 7), (4, 8, 4), (1, 32, 32, 1), num_bags=70000, max_len=40, seed=19)
    assert x.nnz > _sms() * 512 * 16
    out, rc, _, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK
    _check_grouping(x, st["ws"], method="multi_sort")
    rng = np.random.default_rng(5)
    bags = np.sort(rng.choice(x.num_bags, size=400, replace=False))
    idx, off = _sample_bags(x, bags)
    ref = oracle.forward(x.cores, x.m, x.n, x.R, idx, off, threads=8)
    assert np.abs(out[bags] - ref).max() <= FWD_TOL * np.abs(ref).max()


def test_forward_is_deterministic():
    x = make_inputs(3, num_bags=2000)
    a, _, _, st = _gpu_forward(x)
    b, _, _, _ = _gpu_forward(x, ws=st["ws"])
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ edge cases


@pytest.mark.parametrize("shape", [((3, 4, 5), (2, 3, 2), (1, 3, 2, 1)),
                                   ((7, 1, 9), (3, 1, 5), (1, 5, 2, 1)),
                                   ((1, 1, 1), (1, 1, 1), (1, 1, 1, 1)),
                                   ((5, 6, 7), (4, 8, 4), (1, 32, 32, 1)),
                                   ((13, 11, 17), (4, 4, 4), (1, 16, 16, 1)),
                                   ((9, 8, 7), (4, 8, 4), (1, 64, 64, 1))])
def test_edge_shapes_ragged_and_empty_bags(shape):
    m, n, R = shape
    x = make_custom(m, n, R, num_bags=2500, max_len=7, seed=42, empty_frac=0.15)
    out, rc, _, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK
    ref = oracle.forward(x.cores, m, n, R, x.indices, x.offsets, threads=8)
    assert _rel_err(out, ref) <= FWD_TOL
    assert not out[np.diff(x.offsets) == 0].any()
    _check_grouping(x, st["ws"])
    dG = _gpu_backward(x, st)
    dref = oracle.backward(x.grad_out, x.cores, m, n, R, x.indices, x.offsets, threads=8)
    for k in range(3):
        assert _rel_err(dG[k], dref[k]) <= BWD_TOL, k


def test_no_lookups_and_all_empty_bags():
    x = make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=17, max_len=0, seed=1)
    assert x.nnz == 0
    out, rc, _, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK and not out.any() and out.shape == (17, 12)
    dG = _gpu_backward(x, st)
    assert not any(g.any() for g in dG)


def test_out_of_range_indices_are_reported_and_skipped():
    x = make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=300, max_len=6, seed=5)
    bad = x.indices.copy()
    bad[::11] = 60
    bad[5] = -3
    x.indices = bad
    out, rc, bits, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_ERR_INDEX and bits & 1
    keep = (bad >= 0) & (bad < 60)
    ref = oracle.forward(x.cores, x.m, x.n, x.R, bad, x.offsets, strict=False)
    assert _rel_err(out, ref) <= FWD_TOL
    g = _check_grouping(x, st["ws"])
    assert g["n_valid"] == keep.sum()


def test_bad_offsets_are_reported():
    x = make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=50, max_len=4, seed=6)
    off = x.offsets.copy()
    off[10] = off[12] + 1          # not monotone
    x.offsets = off
    _, rc, bits, _ = _gpu_forward(x)
    assert rc == tte.TT_EMB_ERR_OFFSETS and bits & 2


def test_largest_table_32_bit_keys():
    """The largest table the ABI takes: M = 65535 x 65535 x 1 = 4,294,836,225 rows, just
    under the 2^32 - 2 limit, so the grouping keys use all 32 bits (four radix passes,
    and the out-of-range sentinel is all ones).  Uniform indices plus the extremes
    0, 1, M - 2, M - 1 and rows around 2^31; forward (whole output), grouping and every
    core gradient (whole cores) against the oracle; then one index = M is reported and
    contributes nothing."""
    m, n, R = (65535, 65535, 1), (2, 2, 2), (1, 4, 4, 1)
    M = 65535 * 65535
    x = make_custom(m, n, R, num_bags=3000, max_len=6, seed=61)
    x.indices[:6] = [0, 1, M - 2, M - 1, 2 ** 31 - 1, 2 ** 31]
    x.indices[-3:] = [M - 1, 65535 * 7 + 65534, M - 65535]
    out, rc, bits, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK, bits
    ref = oracle.forward(x.cores, m, n, R, x.indices, x.offsets, threads=8)
    assert _rel_err(out, ref) <= FWD_TOL
    _check_grouping(x, st["ws"], method="coop_sort")
    dG = _gpu_backward(x, st)
    dref = oracle.backward(x.grad_out, x.cores, m, n, R, x.indices, x.offsets, threads=8)
    for k in range(3):
        assert _rel_err(dG[k], dref[k]) <= BWD_TOL, k
    x.indices[100] = M                                       # one past the last row
    out, rc, bits, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_ERR_INDEX and bits & 1
    ref = oracle.forward(x.cores, m, n, R, x.indices, x.offsets, strict=False)
    assert _rel_err(out, ref) <= FWD_TOL
    _check_grouping(x, st["ws"], method="coop_sort")


def test_single_hot_row_and_all_same_prefix():
    """Every lookup on one row (a 40k-lookup run) and one prefix with many rows."""
    m, n, R = (4, 5, 300), (4, 8, 4), (1, 32, 32, 1)
    x = make_custom(m, n, R, num_bags=2000, max_len=40, seed=9)
    x.indices[:] = 7
    x.indices[::3] = np.arange(x.indices[::3].size) % 300 + 600   # prefix (0, 2), all i3
    out, rc, _, st = _gpu_forward(x)
    ref = oracle.forward(x.cores, m, n, R, x.indices, x.offsets, threads=8)
    assert rc == tte.TT_EMB_OK and _rel_err(out, ref) <= FWD_TOL
    _check_grouping(x, st["ws"])
    dG = _gpu_backward(x, st)
    dref = oracle.backward(x.grad_out, x.cores, m, n, R, x.indices, x.offsets, threads=8)
    for k in range(3):
        assert _rel_err(dG[k], dref[k]) <= BWD_TOL, k


# ------------------------------------------------------------------ backward + SGD


def test_backward_config5_reduced_full_compare_and_sgd():
    x = make_inputs(5, num_bags=1500)
    _, rc, _, st = _gpu_forward(x)
    dG = _gpu_backward(x, st)
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    for k in range(3):
        assert _rel_err(dG[k], dref[k]) <= BWD_TOL, k
    grads = [_dev(g) for g in dG]
    tte.tt_emb_sgd(st["cores"], grads, x.m, x.n, x.R, 0.01, zero_grads=True)
    for k in range(3):
        upd = st["cores"][k].cpu().numpy().astype(np.float64)
        ref = oracle.sgd(x.cores[k], dref[k], 0.01)
        tol = 0.01 * BWD_TOL * np.abs(dref[k]).max() + 2e-7 * np.abs(ref).max()
        assert np.abs(upd - ref).max() <= tol, k
        assert not grads[k].any(), k          # reset in the same pass


def test_sgd_ragged_segments_without_reset():
    """Core sizes that are not multiples of 4 exercise the scalar tails of the fused update."""
    m, n, R = (3, 5, 7), (3, 1, 3), (1, 3, 5, 1)
    x = make_custom(m, n, R, num_bags=1, max_len=1, seed=3)
    cores = [_dev(c) for c in x.cores]
    rng = np.random.default_rng(4)
    dG = [rng.standard_normal(c.shape).astype(np.float32) for c in x.cores]
    grads = [_dev(g) for g in dG]
    tte.tt_emb_sgd(cores, grads, m, n, R, 0.25)
    for k in range(3):
        ref = oracle.sgd(x.cores[k], dG[k].astype(np.float64), 0.25)
        assert np.abs(cores[k].cpu().numpy() - ref).max() <= 2e-7 * max(1.0, np.abs(ref).max())
        assert np.array_equal(grads[k].cpu().numpy(), dG[k])


@pytest.mark.parametrize("cfg", [5, 3])
def test_backward_full_size_sampled_slices(cfg):
    x = make_inputs(cfg, with_grad=True)
    _, rc, _, st = _gpu_forward(x)
    dG = _gpu_backward(x, st)
    r = x.indices
    i1, i2, i3 = r // (x.m[1] * x.m[2]), (r // x.m[2]) % x.m[1], r % x.m[2]
    picks = [(1, int(i1[7])), (1, int(np.max(i1))), (2, int(i2[3])), (2, int(i2[1000])),
             (3, int(i3[0])), (3, int(i3[555]))]
    for core, v in picks:
        ref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets,
                              threads=8, filter_core=core, filter_value=v)[core - 1][v]
        got = dG[core - 1][v]
        assert _rel_err(got, ref) <= BWD_TOL, (core, v)
    for k in range(3):
        assert np.isfinite(dG[k]).all()


def test_backward_rebuilds_grouping_when_not_reused():
    x = make_inputs(5, num_bags=800)
    cores = [_dev(c) for c in x.cores]
    idx, off = _dev(x.indices), _dev(x.offsets)
    ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                     dtype=torch.uint8, device="cuda")
    grads = [torch.zeros_like(c) for c in cores]
    tte.tt_emb_backward(_dev(x.grad_out), cores, x.m, x.n, x.R, idx, off, grads, ws,
                        reuse_grouping=False)
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    for k in range(3):
        assert _rel_err(grads[k].cpu().numpy(), dref[k]) <= BWD_TOL


def test_wide_dynamic_range_cores():
    """The contractions run as three-term bf16 split products; cores whose
    slices span six orders of magnitude (log-uniform scale per i_k slice, and a
    tenth of the entries with their sign flipped against their neighbours) must
    still meet the forward and gradient tolerances against the fp64 oracle."""
    x = make_custom((23, 17, 29), (4, 8, 4), (1, 32, 32, 1), num_bags=900, max_len=24,
                    seed=314, dist=("zipf", 1.1, "identity"))
    rng = np.random.default_rng(2718)
    for k, c in enumerate(x.cores):
        scale = 10.0 ** rng.uniform(-3.0, 3.0, size=(c.shape[0],) + (1,) * (c.ndim - 1))
        flip = np.where(rng.random(c.shape) < 0.1, -1.0, 1.0)
        x.cores[k] = (c * scale * flip).astype(np.float32)
    out, rc, bits, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK, bits
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    assert _rel_err(out, ref) <= FWD_TOL
    dG = _gpu_backward(x, st)
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    for k in range(3):
        assert _rel_err(dG[k], dref[k]) <= BWD_TOL, k


def test_reused_grouping_resplits_other_or_regrouped_cores():
    """The backward reuses the forward's bf16 split of the cores only when the
    core addresses match and no grouping ran since; both other cases must split
    again (else the gradients would use another table's cores)."""
    x = make_inputs(5, num_bags=600)
    rng = np.random.default_rng(5)
    other = [rng.normal(0.0, 1.0 / np.sqrt(32), c.shape).astype(np.float32) for c in x.cores]
    _, rc, bits, st = _gpu_forward(x)
    assert rc == tte.TT_EMB_OK, bits
    # (a) a reusing backward on different cores
    cores_b = [_dev(c) for c in other]
    grads = [torch.zeros_like(c) for c in cores_b]
    tte.tt_emb_backward(_dev(x.grad_out), cores_b, x.m, x.n, x.R, st["idx"], st["off"], grads,
                        st["ws"], reuse_grouping=True)
    dref = oracle.backward(x.grad_out, other, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    for k in range(3):
        assert _rel_err(grads[k].cpu().numpy(), dref[k]) <= BWD_TOL, k
    # (b) the forward's cores again, after a grouping-only call on the workspace
    tte.tt_emb_group(x.m, x.n, x.R, st["idx"], st["off"], st["ws"])
    grads = [torch.zeros_like(c) for c in st["cores"]]
    tte.tt_emb_backward(_dev(x.grad_out), st["cores"], x.m, x.n, x.R, st["idx"], st["off"], grads,
                        st["ws"], reuse_grouping=True)
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    for k in range(3):
        assert _rel_err(grads[k].cpu().numpy(), dref[k]) <= BWD_TOL, k


def test_owner_object_host_inputs():
    x = make_inputs(5, num_bags=500)
    emb = tte.TTEmbeddingBag(x.cores, x.m, x.n, x.R)
    out = emb.forward(torch.from_numpy(x.indices).pin_memory(),
                      torch.from_numpy(x.offsets).pin_memory())
    emb.backward(torch.from_numpy(x.grad_out))
    emb.check()
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    assert _rel_err(out.cpu().numpy(), ref) <= FWD_TOL
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    for k in range(3):
        assert _rel_err(emb.grads[k].cpu().numpy(), dref[k]) <= BWD_TOL
