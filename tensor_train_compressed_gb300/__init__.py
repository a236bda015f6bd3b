"""GB300-native Tensor-Train embedding bag (forward, backward, SGD).

The compute runs in libtt_emb.so (hand-written CUDA for sm_103a behind the C
ABI of include/tt_emb.h).  This package is the thin Python side: the ctypes
binding with the C names (``tt_emb_*``), a small owner object for cores and
workspace, and the seeded input recipe (``inputs``).  PyTorch supplies device
memory and streams only.
"""
from __future__ import annotations

import numpy as np
import torch

from ._binding import (EXPORTED, TTEmbError, library_path, lib, tt_emb_backward,
                       tt_emb_backward_ex, tt_emb_forward, tt_emb_forward_ex, tt_emb_get_error,
                       tt_emb_forward_tables, tt_emb_sgd_ex, tt_emb_split,
                       tt_emb_workspace_bytes_d, tt_emb_forward_d, tt_emb_backward_d, tt_emb_sgd_d, tt_emb_group, tt_emb_grouping_view,
                       tt_emb_forward_static, tt_emb_profile_read, tt_emb_profile_start,
                       tt_emb_profile_stop,
                       tt_emb_sgd, tt_emb_step_host, tt_emb_version, tt_emb_workspace_bytes)
from ._binding import (TT_EMB_ERR_ARG, TT_EMB_ERR_CUDA, TT_EMB_ERR_INDEX, TT_EMB_ERR_OFFSETS,
                       TT_EMB_ERR_TIMEOUT, TT_EMB_ERR_UNSUPPORTED, TT_EMB_ERR_WORKSPACE, TT_EMB_OK,
                       TT_EMB_CORES_SPLIT, TT_EMB_POOL_MEAN, TT_EMB_POOL_SUM,
                       TT_EMB_FORWARD_ONLY, TT_EMB_INDICES_I32, TT_EMB_ERR_REUSE)

__all__ = ["TTEmbeddingBag", "TTEmbError", "tt_emb_forward", "tt_emb_forward_static", "tt_emb_backward", "tt_emb_sgd",
           "tt_emb_forward_ex", "tt_emb_backward_ex", "tt_emb_split", "tt_emb_sgd_ex",
           "tt_emb_forward_tables", "tt_emb_workspace_bytes_d", "tt_emb_forward_d",
           "tt_emb_backward_d", "tt_emb_sgd_d", "tt_emb_step_host",
           "tt_emb_group", "tt_emb_get_error", "tt_emb_grouping_view", "tt_emb_workspace_bytes",
           "tt_emb_version", "tt_emb_profile_start", "tt_emb_profile_stop", "tt_emb_profile_read",
           "read_grouping", "lib", "library_path", "EXPORTED"]


def read_grouping(m, n, R, nnz: int, num_bags: int, workspace: torch.Tensor) -> dict:
    """Copy the grouping held in ``workspace`` to host numpy arrays (inspection/tests)."""
    view = tt_emb_grouping_view(m, n, R, nnz, num_bags, workspace)
    base = workspace.data_ptr()

    def arr(name, count, dtype=torch.int32):
        off = view[name] - base
        esz = torch.tensor([], dtype=dtype).element_size()
        return workspace[off:off + count * esz].view(dtype).cpu().numpy()

    counts = arr("counts", 7)
    nv, ur, up, nc = (int(v) for v in counts[:4])
    D = int(n[0] * n[1] * n[2])
    method = {1: "bitmap", 2: "coop_sort", 3: "multi_sort", 4: "direct"}.get(int(counts[5]), "none")
    return dict(n_valid=nv, U_r=ur, U_12=up, n_chunks=nc, status=int(counts[4]), method=method,
                ckpt_reused=int(counts[6]),
                perm=arr("perm", nnz), row_start=arr("row_start", ur + 1),
                row_i3=arr("row_i3", ur), row_pair=arr("row_pair", ur),
                pair_row_start=arr("pair_row_start", up + 1), pair_i1=arr("pair_i1", up),
                pair_i2=arr("pair_i2", up), uid=arr("uid", nnz), bag_of=arr("bag_of", nnz),
                chunk_start=arr("chunk_start", nc + 1), chunk_order=arr("chunk_order", nc),
                rowbuf=arr("rowbuf", ur * D, torch.float32).reshape(ur, D))


class TTEmbeddingBag:
    """A TT-compressed embedding table resident on one GPU.

    ``cores`` are float32 arrays [m_k][R_{k-1}][n_k][R_k].  ``forward`` takes
    int64 indices and CSR offsets (host or device tensors / numpy arrays; host
    inputs are copied in on the current stream), optionally per-sample weights
    (sum pooling), and returns the pooled float32 [num_bags][D] output on the
    device.  ``mode`` is "sum" or "mean".
    """

    def __init__(self, cores, m, n, R, device="cuda", mode: str = "sum"):
        if mode not in ("sum", "mean"):
            raise ValueError("mode must be 'sum' or 'mean'")
        self.mode = mode
        self.m, self.n, self.R = tuple(int(v) for v in m), tuple(int(v) for v in n), \
            tuple(int(v) for v in R)
        self.D = self.n[0] * self.n[1] * self.n[2]
        self.device = torch.device(device)
        self.cores = [torch.as_tensor(np.ascontiguousarray(c, np.float32) if not
                                      isinstance(c, torch.Tensor) else c)
                      .to(self.device, torch.float32).contiguous() for c in cores]
        self.grads = [torch.zeros_like(c) for c in self.cores]
        self.workspace = torch.empty(0, dtype=torch.uint8, device=self.device)
        self._batch = None
        self._staging = None

    def _ensure_ws(self, nnz, num_bags):
        need = tt_emb_workspace_bytes(self.m, self.n, self.R, nnz, num_bags)
        if self.workspace.numel() < need:
            # the old workspace may still be in use by work enqueued on another stream
            # (a caller's stream, the host step's copy stream); growth is rare, so wait
            # for the device before handing its memory back to torch's allocator
            torch.cuda.synchronize(self.device)
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)

    def _to_dev(self, x, keep_int32=False):
        t = torch.as_tensor(x)
        dtype = torch.int32 if keep_int32 and t.dtype == torch.int32 else torch.int64
        return t.to(self.device, dtype, non_blocking=True).contiguous()

    def forward(self, indices, offsets, per_sample_weights=None, out=None, stream=None):
        # int32 indices stay int32 (TT_EMB_INDICES_I32); offsets are int64
        idx, off = self._to_dev(indices, keep_int32=True), self._to_dev(offsets)
        B = off.numel() - 1
        self._ensure_ws(idx.numel(), B)
        if out is None:
            out = torch.empty((B, self.D), dtype=torch.float32, device=self.device)
        psw = None
        if per_sample_weights is not None:
            psw = torch.as_tensor(per_sample_weights).to(self.device, torch.float32,
                                                         non_blocking=True).contiguous()
        if psw is None and self.mode == "sum" and idx.dtype == torch.int64:
            tt_emb_forward(self.cores, self.m, self.n, self.R, idx, off, out, self.workspace,
                           stream)
        else:
            tt_emb_forward_ex(self.cores, self.m, self.n, self.R, idx, off, psw, self.mode, out,
                              self.workspace, stream)
        self._batch = (idx, off, psw)
        return out

    def backward(self, grad_out, grad_weights=None, stream=None):
        """Accumulate d<grad_out, out>/dG into self.grads, reusing the last forward's grouping.
        With per-sample weights in that forward and ``grad_weights`` (a float32 CUDA tensor
        [nnz]), the weights' gradient is written there too."""
        if self._batch is None:
            raise RuntimeError("backward needs a forward on the same batch first")
        idx, off, psw = self._batch
        g = torch.as_tensor(grad_out).to(self.device, torch.float32, non_blocking=True)
        if psw is None and self.mode == "sum" and grad_weights is None:
            tt_emb_backward(g.contiguous(), self.cores, self.m, self.n, self.R, idx, off,
                            self.grads, self.workspace, reuse_grouping=True, stream=stream)
        else:
            tt_emb_backward_ex(g.contiguous(), self.cores, self.m, self.n, self.R, idx, off, psw,
                               self.mode, self.grads, grad_weights, self.workspace,
                               reuse_grouping=True, stream=stream)
        return self.grads

    def train_step_host(self, h_indices, h_offsets, h_grad_out, lr: float, h_out=None,
                        stream=None):
        """One training step (sum pooling) from host tensors through tt_emb_step_host: the
        batch is copied in on a copy stream while the kernels run, the cores take an SGD
        step and the gradients are reset; the pooled output lands in ``h_out`` (a float32
        host tensor [num_bags][D]) if given, and is returned on the device.  Page-locked
        host tensors (``.pin_memory()``) let the copies overlap the kernels.

        The returned device tensor is a view of this module's staging buffer: it is
        valid until the next ``train_step_host`` call, which overwrites it (clone it to
        keep it)."""
        if self.mode != "sum":
            raise ValueError("train_step_host pools by sum")
        nnz, B = h_indices.numel(), h_offsets.numel() - 1
        self._ensure_ws(nnz, B)
        st = self._staging
        if (st is None or st[0].numel() < nnz or st[0].dtype != h_indices.dtype
                or st[1].numel() < B + 1 or st[2].shape[0] < B):
            if st is not None:
                torch.cuda.synchronize(self.device)     # old staging may still be in use
            st = (torch.empty(max(nnz, 1), dtype=h_indices.dtype, device=self.device),
                  torch.empty(B + 1, dtype=torch.int64, device=self.device),
                  torch.empty((max(B, 1), self.D), dtype=torch.float32, device=self.device),
                  torch.empty((max(B, 1), self.D), dtype=torch.float32, device=self.device))
            self._staging = st
        d_idx, d_off, d_g, d_out = st[0][:nnz], st[1][:B + 1], st[2][:B], st[3][:B]
        tt_emb_step_host(self.cores, self.grads, self.m, self.n, self.R, h_indices, h_offsets,
                         h_grad_out, h_out, d_idx, d_off, d_g, d_out, lr, self.workspace,
                         stream=stream)
        self._batch = None          # the grouping now belongs to this step's batch
        return d_out

    def zero_grad(self):
        for g in self.grads:
            g.zero_()

    def sgd_step(self, lr: float, zero_grads: bool = False, stream=None):
        """G <- G - lr * dG; with zero_grads the gradients are reset in the same pass."""
        tt_emb_sgd(self.cores, self.grads, self.m, self.n, self.R, lr, zero_grads, stream)

    def check(self, stream=None):
        """Raise TTEmbError if a kernel flagged bad input (synchronises)."""
        rc, bits = tt_emb_get_error(self.workspace, stream)
        if rc != TT_EMB_OK:
            raise TTEmbError(rc, f"device status bits {bits}")
