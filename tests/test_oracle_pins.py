"""Pins of the CPU oracle against facts outside the oracle itself (no GPU).

Each test would fail under a plausible mistake in the oracle: a transposed
core index, a swapped mixed-radix digit, a wrong output order, a dropped term
of the chain, a wrong sign or operand in the backward, or a broken run split
in the grouping.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from tensor_train_compressed_gb300.inputs import make_custom, make_inputs, make_sample_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _materialize(cores, m, n):
    """Dense M x D table, contracting G2 with G3 first (a different order from the oracle)."""
    G1, G2, G3 = (np.asarray(c, dtype=np.float64) for c in cores)
    G23 = np.einsum("yaqb,zbr->yzaqr", G2, G3[:, :, :, 0])
    T = np.einsum("xpa,yzaqr->xyzpqr", G1[:, 0, :, :], G23)
    return T.reshape(m[0] * m[1] * m[2], n[0] * n[1] * n[2])


def _embedding_bag(table, indices, offsets, mode="sum", weights=None):
    """torch.nn.functional.embedding_bag, fp64 on CPU."""
    W = torch.from_numpy(np.ascontiguousarray(table, dtype=np.float64))
    idx = torch.from_numpy(np.asarray(indices, dtype=np.int64))
    off = torch.from_numpy(np.asarray(offsets[:-1], dtype=np.int64))
    psw = None if weights is None else torch.from_numpy(np.asarray(weights, dtype=np.float64))
    return torch.nn.functional.embedding_bag(idx, W, off, mode=mode,
                                             per_sample_weights=psw).numpy()


def _tt_svd(W, m, n):
    """Exact (full-rank) TT-SVD of the table W viewed as modes (m_k*n_k), k = 1..3."""
    m1, m2, m3 = m
    n1, n2, n3 = n
    X = W.reshape(m1, m2, m3, n1, n2, n3).transpose(0, 3, 1, 4, 2, 5)
    U, S, Vt = np.linalg.svd(X.reshape(m1 * n1, -1), full_matrices=False)
    R1 = U.shape[1]
    G1 = U.reshape(m1, n1, R1)[:, None, :, :]
    C = (S[:, None] * Vt).reshape(R1 * m2 * n2, m3 * n3)
    U2, S2, V2t = np.linalg.svd(C, full_matrices=False)
    R2 = U2.shape[1]
    G2 = U2.reshape(R1, m2, n2, R2).transpose(1, 0, 2, 3)
    G3 = (S2[:, None] * V2t).reshape(R2, m3, n3).transpose(1, 0, 2)[:, :, :, None]
    return [G1, G2, G3], (1, R1, R2, 1)


def _dyadic_cores(m, n, R, seed):
    rng = np.random.default_rng(seed)
    shapes = [(m[k], R[k], n[k], R[k + 1]) for k in range(3)]
    return [(rng.integers(-4, 5, size=s) / 4.0).astype(np.float32) for s in shapes]


# ---------------------------------------------------------------- forward


def test_golden_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_worked_2x1x2.json")) as f:
        g = json.load(f)
    m, n, R = g["m"], g["n"], g["R"]
    cores = [np.array(g["G1"], np.float32).reshape(m[0], R[0], n[0], R[1]),
             np.array(g["G2"], np.float32).reshape(m[1], R[1], n[1], R[2]),
             np.array(g["G3"], np.float32).reshape(m[2], R[2], n[2], R[3])]
    out = oracle.forward(cores, m, n, R, g["indices"], g["offsets"])
    assert np.array_equal(out, np.array(g["out"], np.float64))
    dG = oracle.backward(np.array(g["grad_out"], np.float32), cores, m, n, R, g["indices"],
                         g["offsets"])
    for k, key in enumerate(("dG1", "dG2", "dG3")):
        assert np.array_equal(dG[k].ravel(), np.array(g[key], np.float64)), key


@pytest.mark.parametrize("m,n", [((3, 4, 5), (2, 3, 2)), ((2, 3, 2), (3, 1, 2)),
                                 ((4, 2, 3), (1, 2, 4))])
def test_tt_svd_reconstructs_dense_table(m, n):
    """Cores from an exact TT-SVD of a known table must give back its rows."""
    rng = np.random.default_rng(7)
    M, D = m[0] * m[1] * m[2], n[0] * n[1] * n[2]
    W = rng.standard_normal((M, D))
    cores, R = _tt_svd(W, m, n)
    cores32 = [c.astype(np.float32) for c in cores]
    idx = np.arange(M, dtype=np.int64)
    off = np.arange(M + 1, dtype=np.int64)
    out = oracle.forward(cores32, m, n, R, idx, off)
    assert np.abs(out - W).max() <= 1e-5 * np.abs(W).max()
    # and the bag sums of the known table
    idx2 = rng.integers(0, M, size=50)
    off2 = np.array([0, 3, 3, 10, 25, 50])
    out2 = oracle.forward(cores32, m, n, R, idx2, off2)
    ref2 = np.stack([W[idx2[off2[b]:off2[b + 1]]].sum(0) for b in range(5)])
    assert np.abs(out2 - ref2).max() <= 1e-5 * np.abs(ref2).max() * 10


def test_rank1_cores_give_kronecker_rows():
    m, n, R = (3, 4, 5), (2, 3, 2), (1, 1, 1, 1)
    x = make_custom(m, n, R, num_bags=1, max_len=1, seed=11)
    M = 60
    idx = np.arange(M)
    off = np.arange(M + 1)
    out = oracle.forward(x.cores, m, n, R, idx, off)
    G1, G2, G3 = (c.astype(np.float64) for c in x.cores)
    for r in range(M):
        i1, i2, i3 = r // 20, (r // 5) % 4, r % 5
        ref = np.kron(np.kron(G1[i1, 0, :, 0], G2[i2, 0, :, 0]), G3[i3, 0, :, 0])
        assert np.allclose(out[r], ref, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("case", ["config1", "ragged"])
def test_materialized_table_and_torch_embedding_bag(case):
    if case == "config1":
        x = make_inputs(1)
    else:
        x = make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=37, max_len=9, seed=3,
                        empty_frac=0.2)
    out = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    ref = _embedding_bag(_materialize(x.cores, x.m, x.n), x.indices, x.offsets)
    assert out.shape == ref.shape
    assert np.abs(out - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("k", [0, 1, 2])
def test_multilinear_in_each_core(k):
    m, n, R = (3, 4, 5), (2, 3, 2), (1, 3, 2, 1)
    A = _dyadic_cores(m, n, R, 1)
    Bc = _dyadic_cores(m, n, R, 2)
    x = make_custom(m, n, R, num_bags=20, max_len=6, seed=5)
    f = lambda cs: oracle.forward(cs, m, n, R, x.indices, x.offsets)
    mix = list(A)
    mix[k] = (3.0 * A[k] - 2.0 * Bc[k]).astype(np.float32)
    other = list(A)
    other[k] = Bc[k]
    # dyadic values: every product and sum is exact in fp64
    assert np.array_equal(f(mix), 3.0 * f(A) - 2.0 * f(other))


def test_single_core_reduces_to_plain_embedding_bag():
    """m2 = m3 = 1, R = 1 and unit G2, G3: the table is G1 itself."""
    m, n, R = (50, 1, 1), (8, 1, 1), (1, 1, 1, 1)
    rng = np.random.default_rng(9)
    G1 = rng.standard_normal((50, 1, 8, 1)).astype(np.float32)
    cores = [G1, np.ones((1, 1, 1, 1), np.float32), np.ones((1, 1, 1, 1), np.float32)]
    idx = rng.integers(0, 50, 200)
    off = np.concatenate([[0], np.sort(rng.integers(0, 200, 30)), [200]])
    out = oracle.forward(cores, m, n, R, idx, off)
    ref = _embedding_bag(G1.reshape(50, 8), idx, off)
    assert np.abs(out - ref).max() <= 1e-12


def test_bag_permutation_duplicates_and_empty_bags():
    x = make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=10, max_len=5, seed=21)
    out = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    order = np.random.default_rng(0).permutation(10)
    bags = [x.indices[x.offsets[b]:x.offsets[b + 1]] for b in order]
    idx2 = np.concatenate(bags)
    off2 = np.concatenate([[0], np.cumsum([len(b) for b in bags])])
    assert np.array_equal(oracle.forward(x.cores, x.m, x.n, x.R, idx2, off2), out[order])
    # a bag holding the same row twice is twice the row; an empty bag is zero
    r = int(x.indices[0])
    one = oracle.forward(x.cores, x.m, x.n, x.R, [r], [0, 1])
    two = oracle.forward(x.cores, x.m, x.n, x.R, [r, r], [0, 0, 2, 2])
    assert np.array_equal(two[1], 2.0 * one[0])
    assert not two[0].any() and not two[2].any()


def test_errors_on_bad_indices_and_offsets():
    x = make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=4, max_len=3, seed=2)
    bad = x.indices.copy()
    bad[0] = 60
    with pytest.raises(oracle.OracleError) as e:
        oracle.forward(x.cores, x.m, x.n, x.R, bad, x.offsets)
    assert e.value.code == oracle.TTO_ERR_INDEX
    off = x.offsets.copy()
    off[1], off[2] = off[2], off[1] - 1
    with pytest.raises(oracle.OracleError) as e:
        oracle.forward(x.cores, x.m, x.n, x.R, x.indices, off)
    assert e.value.code in (oracle.TTO_ERR_OFFSETS,)
    with pytest.raises(oracle.OracleError):
        oracle.forward(x.cores, x.m, x.n, (2, 3, 2, 1), x.indices, x.offsets)


def test_threads_do_not_change_forward():
    x = make_custom((5, 6, 7), (2, 2, 3), (1, 4, 3, 1), num_bags=101, max_len=7, seed=4)
    a = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=1)
    b = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=4)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- backward


def _bwd_case():
    return make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=23, max_len=6, seed=8)


@pytest.mark.parametrize("k", [0, 1, 2])
def test_backward_adjoint_identity(k):
    """<grad_out, out(G with G_k -> dGk)> == <dG_k, dGk> since out is linear in G_k."""
    x = _bwd_case()
    dG = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    delta = np.random.default_rng(30 + k).standard_normal(x.cores[k].shape).astype(np.float32)
    cs = list(x.cores)
    cs[k] = delta
    lhs = float((oracle.forward(cs, x.m, x.n, x.R, x.indices, x.offsets)
                 * x.grad_out.astype(np.float64)).sum())
    rhs = float((dG[k] * delta.astype(np.float64)).sum())
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs))


def test_backward_matches_torch_autograd():
    x = _bwd_case()
    dG = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    G = [torch.tensor(c, dtype=torch.float64, requires_grad=True) for c in x.cores]
    G23 = torch.einsum("yaqb,zbr->yzaqr", G[1], G[2][:, :, :, 0])
    T = torch.einsum("xpa,yzaqr->xyzpqr", G[0][:, 0], G23).reshape(60, 12)
    out = torch.nn.functional.embedding_bag(torch.from_numpy(x.indices), T,
                                            torch.from_numpy(x.offsets[:-1]), mode="sum")
    (out * torch.from_numpy(x.grad_out.astype(np.float64))).sum().backward()
    for k in range(3):
        ref = G[k].grad.numpy()
        assert np.abs(dG[k] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_backward_central_differences():
    """out is affine in every single core entry, so a central difference is exact."""
    m, n, R = (3, 4, 5), (2, 3, 2), (1, 3, 2, 1)
    cores = _dyadic_cores(m, n, R, 12)
    x = make_custom(m, n, R, num_bags=15, max_len=5, seed=13)
    g = (np.random.default_rng(14).integers(-3, 4, size=x.grad_out.shape) / 2.0).astype(
        np.float32)
    dG = oracle.backward(g, cores, m, n, R, x.indices, x.offsets)
    rng = np.random.default_rng(15)
    for k in range(3):
        for _ in range(6):
            pos = tuple(int(rng.integers(0, s)) for s in cores[k].shape)
            up, dn = [c.copy() for c in cores], [c.copy() for c in cores]
            up[k][pos] += 0.25
            dn[k][pos] -= 0.25
            fu = (oracle.forward(up, m, n, R, x.indices, x.offsets) * g).sum()
            fd = (oracle.forward(dn, m, n, R, x.indices, x.offsets) * g).sum()
            assert (fu - fd) / 0.5 == dG[k][pos]


@pytest.mark.parametrize("k", [1, 2, 3])
def test_backward_filter_gives_the_exact_slice(k):
    x = _bwd_case()
    full = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    v = 1
    part = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets,
                           filter_core=k, filter_value=v)
    assert np.allclose(part[k - 1][v], full[k - 1][v], rtol=1e-13, atol=1e-13)


def test_backward_threads():
    x = _bwd_case()
    a = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=1)
    b = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=3)
    for k in range(3):
        assert np.allclose(a[k], b[k], rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("lr", [1.0 / 64, 0.25])
def test_sgd_step_is_the_exact_descent_of_the_loss(lr):
    """L(G) = <g, out(G)> is linear in each core on its own (the row is a product of one
    slice of every core), so L(G_k + delta) = L(G_k) + <dL/dG_k, delta> exactly.  One SGD
    step on core k alone must therefore change L by exactly -lr * ||dL/dG_k||^2, with L
    evaluated by the forward oracle.  Dyadic cores, output gradient and step keep every
    value exact, so a sign, a scale, a dropped lr or a misplaced element fails."""
    m, n, R = (3, 4, 5), (2, 3, 2), (1, 3, 2, 1)
    cores = _dyadic_cores(m, n, R, 21)
    x = make_custom(m, n, R, num_bags=15, max_len=5, seed=22)
    g = (np.random.default_rng(23).integers(-3, 4, size=x.grad_out.shape) / 2.0).astype(
        np.float32)
    dG = oracle.backward(g, cores, m, n, R, x.indices, x.offsets)
    L0 = (oracle.forward(cores, m, n, R, x.indices, x.offsets) * g).sum()
    for k in range(3):
        assert np.abs(dG[k]).max() > 0
        upd = oracle.sgd(cores[k], dG[k], lr)
        assert np.array_equal(upd.astype(np.float32).astype(np.float64), upd)   # exact in fp32
        stepped = [c.copy() for c in cores]
        stepped[k] = upd.astype(np.float32)
        L1 = (oracle.forward(stepped, m, n, R, x.indices, x.offsets) * g).sum()
        assert L1 - L0 == -lr * float((dG[k] ** 2).sum()), k


# ------------------------------------------------- mean and weighted pooling


def _pool_case():
    return make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=41, max_len=9, seed=17,
                       empty_frac=0.15)


@pytest.mark.parametrize("mode", ["mean", "weighted"])
def test_pooling_variants_match_torch_embedding_bag(mode):
    x = _pool_case()
    table = _materialize(x.cores, x.m, x.n)
    if mode == "mean":
        out = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, mode="mean")
        ref = _embedding_bag(table, x.indices, x.offsets, mode="mean")
    else:
        w = make_sample_weights(len(x.indices), 5, -1.0, 2.0)
        out = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, weights=w)
        ref = _embedding_bag(table, x.indices, x.offsets, weights=w)
    assert np.abs(np.diff(x.offsets)).min() == 0          # the case holds empty bags
    assert np.abs(out - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_integer_weights_equal_repeated_lookups():
    """A weight k in {0, 1, 2, 3} gives the bag with that lookup repeated k times
    (dyadic cores: every sum is exact, so the two agree bit for bit)."""
    m, n, R = (3, 4, 5), (2, 3, 2), (1, 3, 2, 1)
    cores = _dyadic_cores(m, n, R, 40)
    x = make_custom(m, n, R, num_bags=25, max_len=6, seed=41)
    k = np.random.default_rng(42).integers(0, 4, size=len(x.indices))
    out = oracle.forward(cores, m, n, R, x.indices, x.offsets, weights=k.astype(np.float32))
    idx2 = np.repeat(x.indices, k)
    lens = [int(k[x.offsets[b]:x.offsets[b + 1]].sum()) for b in range(25)]
    off2 = np.concatenate([[0], np.cumsum(lens)])
    assert np.array_equal(out, oracle.forward(cores, m, n, R, idx2, off2))


def test_unit_weights_and_unit_bags_leave_the_sum():
    x = _pool_case()
    s = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    ones = np.ones(len(x.indices), np.float32)
    assert np.array_equal(oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets,
                                         weights=ones), s)
    single = np.arange(len(x.indices) + 1)
    assert np.array_equal(oracle.forward(x.cores, x.m, x.n, x.R, x.indices, single, mode="mean"),
                          oracle.forward(x.cores, x.m, x.n, x.R, x.indices, single))


@pytest.mark.parametrize("mode", ["mean", "weighted"])
def test_pooling_variants_backward_match_torch_autograd(mode):
    x = _pool_case()
    w = make_sample_weights(len(x.indices), 6, -1.0, 2.0) if mode == "weighted" else None
    if w is None:
        dG = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets,
                             mode="mean")
    else:
        dG, dW = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets,
                                 weights=w, want_dw=True)
    G = [torch.tensor(c, dtype=torch.float64, requires_grad=True) for c in x.cores]
    G23 = torch.einsum("yaqb,zbr->yzaqr", G[1], G[2][:, :, :, 0])
    T = torch.einsum("xpa,yzaqr->xyzpqr", G[0][:, 0], G23).reshape(60, 12)
    psw = None if w is None else torch.tensor(w, dtype=torch.float64, requires_grad=True)
    out = torch.nn.functional.embedding_bag(torch.from_numpy(x.indices), T,
                                            torch.from_numpy(x.offsets[:-1]),
                                            mode="mean" if w is None else "sum",
                                            per_sample_weights=psw)
    (out * torch.from_numpy(x.grad_out.astype(np.float64))).sum().backward()
    for k in range(3):
        ref = G[k].grad.numpy()
        assert np.abs(dG[k] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
    if w is not None:
        ref = psw.grad.numpy()
        assert np.abs(dW - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_weight_gradient_central_differences():
    """out is linear in every weight, so a central difference is exact (dyadic data)."""
    m, n, R = (3, 4, 5), (2, 3, 2), (1, 3, 2, 1)
    cores = _dyadic_cores(m, n, R, 50)
    x = make_custom(m, n, R, num_bags=12, max_len=5, seed=51)
    g = (np.random.default_rng(52).integers(-3, 4, size=x.grad_out.shape) / 2.0).astype(
        np.float32)
    w = (np.random.default_rng(53).integers(-4, 5, size=len(x.indices)) / 4.0).astype(np.float32)
    _, dW = oracle.backward(g, cores, m, n, R, x.indices, x.offsets, weights=w, want_dw=True)
    for l in range(0, len(x.indices), 3):
        up, dn = w.copy(), w.copy()
        up[l] += 0.5
        dn[l] -= 0.5
        fu = (oracle.forward(cores, m, n, R, x.indices, x.offsets, weights=up) * g).sum()
        fd = (oracle.forward(cores, m, n, R, x.indices, x.offsets, weights=dn) * g).sum()
        assert fu - fd == dW[l]


def test_pooling_variant_errors():
    x = _pool_case()
    w = np.ones(len(x.indices), np.float32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets, weights=w, mode="mean")
    assert e.value.code == oracle.TTO_ERR_ARG
    with pytest.raises(oracle.OracleError) as e:
        oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, want_dw=True)
    assert e.value.code == oracle.TTO_ERR_ARG


# ---------------------------------------------------------------- chains of d cores


def _tt_svd_d(W, m, n):
    """Exact (full-rank) TT-SVD of W viewed as modes (m_k*n_k), k = 1..d."""
    d = len(m)
    X = W.reshape(*m, *n)
    X = X.transpose([a for k in range(d) for a in (k, d + k)])     # (m1, n1, m2, n2, ...)
    cores, Rprev, rest = [], 1, X.reshape(m[0] * n[0], -1)
    for k in range(d - 1):
        U, S, Vt = np.linalg.svd(rest.reshape(Rprev * m[k] * n[k], -1), full_matrices=False)
        Rk = U.shape[1]
        cores.append(U.reshape(Rprev, m[k], n[k], Rk).transpose(1, 0, 2, 3))
        rest = S[:, None] * Vt
        Rprev = Rk
    cores.append(rest.reshape(Rprev, m[-1], n[-1], 1).transpose(1, 0, 2, 3))
    return cores, tuple([1] + [c.shape[3] for c in cores])


def _materialize_d(cores, m, n):
    """Dense table, contracting the chain from the last core backwards (the oracle goes
    forwards)."""
    G = [torch.tensor(np.asarray(c, dtype=np.float64)) for c in cores]
    T = G[-1][:, :, :, 0]                       # [m_d][R][n_d]
    for k in range(len(G) - 2, -1, -1):
        T = torch.einsum("xaqb,ybr->xyaqr", G[k], T)
        T = T.reshape(T.shape[0] * T.shape[1], T.shape[2], T.shape[3] * T.shape[4])
    return T[:, 0, :]


@pytest.mark.parametrize("m,n", [((2, 3, 2, 3), (2, 2, 1, 2)), ((3, 2, 2, 2, 2), (1, 2, 2, 1, 2))])
def test_tt_svd_reconstructs_dense_table_d_cores(m, n):
    rng = np.random.default_rng(61)
    M, D = int(np.prod(m)), int(np.prod(n))
    W = rng.standard_normal((M, D))
    cores, R = _tt_svd_d(W, m, n)
    out = oracle.forward_d([c.astype(np.float32) for c in cores], m, n, R, np.arange(M),
                           np.arange(M + 1))
    # the cores are rounded to fp32 on the way in: compare at fp32 resolution
    assert np.abs(out - W).max() <= 1e-5 * np.abs(W).max()


@pytest.mark.parametrize("shape", [((3, 2, 4, 2), (2, 3, 1, 2), (1, 3, 2, 4, 1)),
                                   ((2, 2, 3, 2, 3), (1, 2, 2, 2, 1), (1, 2, 3, 2, 2, 1)),
                                   ((5, 7), (3, 2), (1, 4, 1))])
def test_d_cores_materialized_table_and_torch_autograd(shape):
    m, n, R = shape
    x = make_custom(m, n, R, num_bags=31, max_len=7, seed=63, empty_frac=0.15)
    out = oracle.forward_d(x.cores, m, n, R, x.indices, x.offsets)
    T = _materialize_d(x.cores, m, n).numpy()
    ref = _embedding_bag(T, x.indices, x.offsets)
    assert np.abs(out - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
    dG = oracle.backward_d(x.grad_out, x.cores, m, n, R, x.indices, x.offsets)
    G = [torch.tensor(c, dtype=torch.float64, requires_grad=True) for c in x.cores]
    Tt = G[-1][:, :, :, 0]
    for k in range(len(G) - 2, -1, -1):
        Tt = torch.einsum("xaqb,ybr->xyaqr", G[k], Tt)
        Tt = Tt.reshape(Tt.shape[0] * Tt.shape[1], Tt.shape[2], Tt.shape[3] * Tt.shape[4])
    o = torch.nn.functional.embedding_bag(torch.from_numpy(x.indices), Tt[:, 0, :],
                                          torch.from_numpy(x.offsets[:-1]), mode="sum")
    (o * torch.from_numpy(x.grad_out.astype(np.float64))).sum().backward()
    for k in range(len(G)):
        gr = G[k].grad.numpy()
        assert np.abs(dG[k] - gr).max() <= 1e-12 * max(1.0, np.abs(gr).max()), k


def test_three_cores_of_the_chain_equal_the_three_core_oracle():
    x = _bwd_case()
    a = oracle.forward_d(x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    assert np.array_equal(a, oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets))
    b = oracle.backward_d(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    c = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    for k in range(3):
        assert np.allclose(b[k], c[k], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- grouping


@pytest.mark.parametrize("seed", [0, 1])
def test_grouping_matches_numpy_lexsort(seed):
    m = (7, 5, 6)
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, 210, size=500)
    idx[::7] = idx[0]          # a heavy row
    idx[3] = 210               # out of range: excluded
    g = oracle.group(idx, m)
    assert g["status"] == oracle.TTO_ERR_INDEX
    valid = np.flatnonzero(idx < 210)
    r = idx[valid]
    i1, i2, i3 = r // 30, (r // 6) % 5, r % 6
    key = (i2 * 7 + i1) * 6 + i3
    order = np.lexsort((valid, key))
    assert np.array_equal(g["perm"], valid[order])
    skey = key[order]
    ukey, first = np.unique(skey, return_index=True)
    assert np.array_equal(g["row_start"], np.append(first, len(skey)))
    assert np.array_equal(g["row_index"], r[order][first])
    upair, pfirst, pinv = np.unique(ukey // 6, return_index=True, return_inverse=True)
    assert np.array_equal(g["pair_row_start"], np.append(pfirst, len(ukey)))
    assert np.array_equal(g["row_pair"], pinv)
    assert np.array_equal(g["pair_i2"], upair // 7)
    assert np.array_equal(g["pair_i1"], upair % 7)
    uid = np.full(500, -1)
    uid[valid[order]] = np.searchsorted(ukey, skey)
    assert np.array_equal(g["uid"], uid)


def test_grouping_empty():
    g = oracle.group(np.zeros(0, np.int64), (2, 2, 2))
    assert g["U_r"] == 0 and g["U_12"] == 0 and g["n_valid"] == 0
    assert list(g["row_start"]) == [0] and list(g["pair_row_start"]) == [0]
