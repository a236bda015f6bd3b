"""The seeded input recipe: shapes, determinism, factorisation and distributions."""
import numpy as np

from tensor_train_compressed_gb300.inputs import CONFIGS, factor3, make_inputs


def test_factor3_recipe():
    want = {100_000: (47, 47, 46), 1_000_000: (100, 100, 100), 4_000_000: (159, 159, 159),
            10_000_000: (216, 216, 215), 20_000_000: (272, 272, 271),
            30_000_000: (311, 311, 311), 40_000_000: (342, 342, 342)}
    for N, m in want.items():
        assert factor3(N) == m
        assert m[0] * m[1] * m[2] >= N


def test_config_shapes_and_determinism():
    for cfg in (1, 2):
        a, b = make_inputs(cfg), make_inputs(cfg)
        assert np.array_equal(a.indices, b.indices) and np.array_equal(a.offsets, b.offsets)
        for k in range(3):
            assert np.array_equal(a.cores[k], b.cores[k])
            assert a.cores[k].dtype == np.float32
            assert a.cores[k].shape == (a.m[k], a.R[k], a.n[k], a.R[k + 1])
        assert a.offsets[0] == 0 and a.offsets[-1] == a.nnz
        assert np.all(np.diff(a.offsets) >= 1)
        assert a.indices.min() >= 0 and a.indices.max() < a.N
    x = make_inputs(1)
    assert x.num_bags == 64 and x.D == 16 and np.diff(x.offsets).max() <= 4


def test_zipf_head_and_bag_lengths():
    x = make_inputs(3, num_bags=2048)
    assert np.all(np.diff(x.offsets) == 20)
    # P(rank 1) = 1/H(12e6, 1.2) ~ 0.185
    assert abs((x.indices == 0).mean() - 0.185) < 0.02
    y = make_inputs(5, num_bags=4096)
    L = np.diff(y.offsets)
    assert L.min() >= 10 and L.max() <= 30 and y.grad_out.shape == (4096, 128)
    assert CONFIGS[5]["train"] and y.m == (360, 360, 370)
