"""tt_emb_forward_static: the forward for callers that cannot allocate device memory.

Such callers (an allocator-less runtime that only hands out input and output
buffers, a plugin whose host framework owns every device allocation, code
that must not allocate once in steady state) cannot give tt_emb_forward its
workspace; this entry point uses the library's fixed 16 MiB device array
instead.  The test calls it through the C ABI twice in a row, on different
batches, and checks each output against tt_emb_forward's within the forward
tolerance of the parity tests.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import tensor_train_compressed_gb300 as tte
from tensor_train_compressed_gb300.inputs import make_custom, make_inputs

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-4


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _both(x):
    cores = [_dev(c) for c in x.cores]
    idx, off = _dev(x.indices), _dev(x.offsets)
    ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                     dtype=torch.uint8, device="cuda")
    ref = torch.empty((x.num_bags, x.D), dtype=torch.float32, device="cuda")
    tte.tt_emb_forward(cores, x.m, x.n, x.R, idx, off, ref, ws)
    out = torch.full((x.num_bags, x.D), float("nan"), dtype=torch.float32, device="cuda")
    tte.tt_emb_forward_static(cores, x.m, x.n, x.R, idx, off, out)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ref.cpu().numpy()


def test_static_forward_matches_workspace_forward_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tensor_train_compressed_gb300 import build
    build.build()
    # 15k lookups into a 720,000-row table of the benchmark tables' factor shape (its
    # bf16 split planes fit the array with the rest of the scratch)
    first = make_custom((100, 60, 120), (4, 8, 4), (1, 32, 32, 1), num_bags=1000, max_len=30,
                        seed=71)
    second = make_custom((5, 6, 7), (4, 8, 4), (1, 32, 32, 1), num_bags=700, max_len=9,
                         seed=77, empty_frac=0.1)             # a different shape right after
    for x in (first, second):
        assert tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags) <= 16 << 20
        out, ref = _both(x)
        assert np.isfinite(out).all()
        scale = max(np.abs(ref).max(), 1e-30)
        assert np.abs(out - ref).max() <= FWD_TOL * scale


def test_static_forward_rejects_sizes_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    x = make_inputs(3, num_bags=3000)                         # ~60k lookups, 12M rows: > 16 MiB
    assert tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags) > 16 << 20
    cores = [_dev(c) for c in x.cores]
    out = torch.empty((x.num_bags, x.D), dtype=torch.float32, device="cuda")
    with pytest.raises(tte.TTEmbError) as e:
        tte.tt_emb_forward_static(cores, x.m, x.n, x.R, _dev(x.indices), _dev(x.offsets), out)
    assert e.value.code == tte.TT_EMB_ERR_WORKSPACE
