"""tt_emb_step_host: one step from page-locked host tensors through the C ABI.

The pooled output copied back must equal, bit for bit, the output of the same
forward on device buffers (the forward is deterministic); the updated cores
must be the cores minus lr times gradients that meet the usual bar against the
oracle, with the gradients reset; a forward-only step leaves the cores alone;
steps with the copy stream equal to the compute stream, consecutive steps on
the kept split and a batch with no lookups behave the same way.
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tensor_train_compressed_gb300 import build
    build.build()


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _pinned(x):
    return torch.from_numpy(np.ascontiguousarray(x)).pin_memory()


def _rel_err(a, ref):
    return float(np.abs(np.asarray(a, np.float64) - ref).max() / max(np.abs(ref).max(), 1e-30))


class Staging:
    """Pinned host copies of a batch and the device tensors they are copied to."""

    def __init__(self, x, train=True):
        self.h_idx, self.h_off = _pinned(x.indices), _pinned(x.offsets)
        self.h_g = _pinned(x.grad_out) if train else None
        self.h_out = torch.full((x.num_bags, x.D), float("nan")).pin_memory()
        self.d_idx = torch.empty(x.nnz, dtype=torch.int64, device="cuda")
        self.d_off = torch.empty(x.num_bags + 1, dtype=torch.int64, device="cuda")
        self.d_g = torch.empty((x.num_bags, x.D), device="cuda") if train else None
        self.d_out = torch.empty((x.num_bags, x.D), device="cuda")

    def step(self, x, cores, grads, ws, lr, flags=0, stream=None, copy_stream=None):
        tte.tt_emb_step_host(cores, grads, x.m, x.n, x.R, self.h_idx, self.h_off, self.h_g,
                             self.h_out, self.d_idx, self.d_off, self.d_g, self.d_out, lr, ws,
                             flags=flags, stream=stream, copy_stream=copy_stream)


def _device_forward(x, cores, ws):
    out = torch.empty((x.num_bags, x.D), device="cuda")
    tte.tt_emb_forward(cores, x.m, x.n, x.R, _dev(x.indices), _dev(x.offsets), out, ws)
    return out


@pytest.mark.parametrize("same_stream", [False, True])
def test_training_step_from_host_buffers(same_stream):
    x = make_inputs(5, num_bags=1200)
    lr = 0.5
    cores0 = [_dev(c) for c in x.cores]
    cores = [c.clone() for c in cores0]
    grads = [torch.zeros_like(c) for c in cores]
    ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                     dtype=torch.uint8, device="cuda")
    expect = _device_forward(x, cores0, torch.empty_like(ws)).cpu()
    s = Staging(x)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()              # cores and workspace made on the default stream
    with torch.cuda.stream(stream):
        s.step(x, cores, grads, ws, lr, stream=stream, copy_stream=stream if same_stream else None)
    stream.synchronize()
    rc, bits = tte.tt_emb_get_error(ws, stream)
    assert rc == tte.TT_EMB_OK, bits
    assert torch.equal(s.h_out, expect)
    ref = oracle.forward(x.cores, x.m, x.n, x.R, x.indices, x.offsets)
    assert _rel_err(s.h_out.numpy(), ref) <= FWD_TOL
    dref = oracle.backward(x.grad_out, x.cores, x.m, x.n, x.R, x.indices, x.offsets, threads=8)
    for k in range(3):
        dg = (cores0[k].cpu().numpy().astype(np.float64) - cores[k].cpu().numpy()) / lr
        assert _rel_err(dg, dref[k]) <= BWD_TOL, k
        assert not grads[k].any()


def test_forward_only_step_and_kept_split_across_steps():
    x = make_inputs(5, num_bags=900)
    cores = [_dev(c) for c in x.cores]
    plain = [c.clone() for c in cores]
    grads = [torch.zeros_like(c) for c in cores]
    ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                     dtype=torch.uint8, device="cuda")
    # forward only: the output, no change to the cores
    f = Staging(x, train=False)
    f.step(x, cores, None, ws, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(f.h_out, _device_forward(x, plain, torch.empty_like(ws)).cpu())
    for k in range(3):
        assert torch.equal(cores[k], plain[k])
    # two training steps, the second on the split the first one's SGD left
    t = Staging(x)
    t.step(x, cores, grads, ws, 0.05)
    after_first = [c.clone() for c in cores]
    t.step(x, cores, grads, ws, 0.05, flags=tte.TT_EMB_CORES_SPLIT)
    torch.cuda.synchronize()
    rc, bits = tte.tt_emb_get_error(ws)
    assert rc == tte.TT_EMB_OK, bits
    assert torch.equal(t.h_out, _device_forward(x, after_first, torch.empty_like(ws)).cpu())


def test_step_with_no_lookups():
    x = make_custom((3, 4, 5), (2, 3, 2), (1, 3, 2, 1), num_bags=17, max_len=0, seed=1)
    assert x.nnz == 0
    cores = [_dev(c) for c in x.cores]
    plain = [c.clone() for c in cores]
    grads = [torch.zeros_like(c) for c in cores]
    ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                     dtype=torch.uint8, device="cuda")
    s = Staging(x)
    s.step(x, cores, grads, ws, 0.5)
    torch.cuda.synchronize()
    assert not s.h_out.any()
    for k in range(3):
        assert torch.equal(cores[k], plain[k])


def test_class_train_step_from_host_matches_the_device_calls():
    x = make_inputs(5, num_bags=600)
    a = tte.TTEmbeddingBag(x.cores, x.m, x.n, x.R)
    b = tte.TTEmbeddingBag(x.cores, x.m, x.n, x.R)
    h_out = torch.full((x.num_bags, x.D), float("nan")).pin_memory()
    d_out = a.train_step_host(_pinned(x.indices), _pinned(x.offsets), _pinned(x.grad_out), 0.5,
                              h_out=h_out)
    out_b = b.forward(x.indices, x.offsets)
    b.backward(x.grad_out)
    dg = [g.clone() for g in b.grads]
    b.sgd_step(0.5, zero_grads=True)
    torch.cuda.synchronize()
    a.check()
    assert torch.equal(h_out, out_b.cpu()) and torch.equal(d_out, out_b)
    for k in range(3):
        # the two gradients differ only in the order of their float atomics
        tol = 0.5 * 1e-3 * dg[k].abs().max().item()
        assert (a.cores[k] - b.cores[k]).abs().max().item() <= tol, k
        assert not a.grads[k].any()


@pytest.mark.parametrize("same_stream", [False, True])
def test_repeated_forward_steps_replay_a_graph(same_stream):
    # the second call with the same arguments captures the work into a graph and
    # later ones replay it: every call's output is the device forward's, bit for bit
    # (also with the copy stream equal to the compute stream)
    x = make_inputs(3, num_bags=2000)
    cores = [_dev(c) for c in x.cores]
    ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                     dtype=torch.uint8, device="cuda")
    expect = _device_forward(x, cores, torch.empty_like(ws)).cpu()
    f = Staging(x, train=False)
    stream = torch.cuda.Stream()
    copy_stream = stream if same_stream else torch.cuda.Stream()
    torch.cuda.synchronize()
    for it in range(5):
        f.h_out.fill_(float("nan"))
        f.d_out.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            f.step(x, cores, None, ws, 0.1, flags=tte.TT_EMB_FORWARD_ONLY, stream=stream,
                   copy_stream=copy_stream)
        stream.synchronize()
        rc, bits = tte.tt_emb_get_error(ws, stream)
        assert rc == tte.TT_EMB_OK, (it, bits)
        assert torch.equal(f.h_out, expect), it
        assert torch.equal(f.d_out.cpu(), expect), it


def test_repeated_training_steps_replay_a_graph():
    # five training steps with the same arguments (the last three replayed from
    # a graph) against five steps of the device calls
    x = make_inputs(5, num_bags=1500)
    lr = 1e-3                # repeated steps on one fixed output gradient: kept small
    ws_a = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                       dtype=torch.uint8, device="cuda")
    ws_b = torch.empty_like(ws_a)
    a = [_dev(c) for c in x.cores]
    b = [c.clone() for c in a]
    ga = [torch.zeros_like(c) for c in a]
    gb = [torch.zeros_like(c) for c in b]
    tte.tt_emb_split(a, x.m, x.n, x.R, ws_a)
    tte.tt_emb_split(b, x.m, x.n, x.R, ws_b)
    s = Staging(x)
    stream, copy_stream = torch.cuda.Stream(), torch.cuda.Stream()
    idx, off, g = _dev(x.indices), _dev(x.offsets), _dev(x.grad_out)
    out_b = torch.empty((x.num_bags, x.D), device="cuda")
    torch.cuda.synchronize()
    for it in range(5):
        with torch.cuda.stream(stream):
            s.step(x, a, ga, ws_a, lr, flags=tte.TT_EMB_CORES_SPLIT, stream=stream,
                   copy_stream=copy_stream)
        stream.synchronize()
        tte.tt_emb_forward_ex(b, x.m, x.n, x.R, idx, off, None, "sum", out_b, ws_b,
                              flags=tte.TT_EMB_CORES_SPLIT)
        tte.tt_emb_backward(g, b, x.m, x.n, x.R, idx, off, gb, ws_b, reuse_grouping=True)
        tte.tt_emb_sgd_ex(b, gb, x.m, x.n, x.R, lr, True, ws_b)
        torch.cuda.synchronize()
        for ws in (ws_a, ws_b):
            rc, bits = tte.tt_emb_get_error(ws)
            assert rc == tte.TT_EMB_OK, (it, bits)
        # outputs and cores differ only by the order of the backward's float atomics
        ref = out_b.cpu()
        assert (s.h_out - ref).abs().max().item() <= 1e-5 * ref.abs().max().item(), it
        for k in range(3):
            assert (a[k] - b[k]).abs().max().item() <= 1e-5 * b[k].abs().max().item(), (it, k)
            assert not ga[k].any()


def test_graph_replay_follows_changed_arguments():
    # alternating output buffers and a pageable host output: every call writes
    # where its own arguments say
    x = make_inputs(3, num_bags=800)
    cores = [_dev(c) for c in x.cores]
    ws = torch.empty(tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags),
                     dtype=torch.uint8, device="cuda")
    expect = _device_forward(x, cores, torch.empty_like(ws)).cpu()
    f = Staging(x, train=False)
    outs = [torch.empty((x.num_bags, x.D), device="cuda") for _ in range(2)]
    pageable = torch.empty((x.num_bags, x.D))
    stream, copy_stream = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for it in range(6):
        d_out = outs[it % 2]
        h_out = pageable if it == 4 else f.h_out
        d_out.fill_(float("nan"))
        h_out.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            tte.tt_emb_step_host(cores, None, x.m, x.n, x.R, f.h_idx, f.h_off, None, h_out,
                                 f.d_idx, f.d_off, None, d_out, 0.1, ws,
                                 flags=tte.TT_EMB_FORWARD_ONLY, stream=stream,
                                 copy_stream=copy_stream)
        stream.synchronize()
        assert torch.equal(d_out.cpu(), expect), it
        assert torch.equal(h_out, expect), it
