"""sparse_graph_recurrent_gb300 -- a leaky-tanh recurrence over a fixed sparse
directed graph, trained with hand-written CUDA kernels for one GB300 (sm_103a).

Python surface (connectome-kernels page, "Use"):

    graph = SparseGraph(src, dst, num_nodes=N, input_nodes=input_nodes)
    out = sparse_recurrence(edge_values, leak, bias, drives, state0, graph, microsteps=2)
    # out: [T, B, N] node states after each input step; differentiable in
    # edge_values, leak, bias, drives [T, n_in, B] and state0 [B, N]

Everything runs in libck (include/ck.h); this package only marshals arguments.
"""
from __future__ import annotations

import torch

from . import _ck
from ._ck import CKError  # noqa: F401

__all__ = ["SparseGraph", "sparse_recurrence", "CKError", "forward", "backward"]


class SparseGraph:
    """A fixed directed graph src[e] -> dst[e] with designated input nodes.

    Built once on the GPU by ck_graph_create; edge parameters stay in the
    caller's edge order.  With edges_in_host_memory the arrays indexed by edge
    (24 bytes per edge) live in pinned host memory that the kernels read in
    place over the CPU-GPU link, leaving O(N) of the graph on the device;
    results are bitwise the same.  With tiling the graph also holds the
    shared-memory tilings the opt-in tiled kernels need (CK_OPT_TILED).
    """

    def __init__(self, src, dst, num_nodes: int, input_nodes, edges_in_host_memory: bool = False,
                 tiling: bool = False):
        if src.shape != dst.shape or src.dim() != 1:
            raise ValueError("src and dst must be 1-D and of equal length")
        self.device = src.device
        self.num_nodes = int(num_nodes)
        self.num_edges = int(src.numel())
        self.num_inputs = int(input_nodes.numel())
        self.edges_in_host_memory = bool(edges_in_host_memory)
        self.tiling = bool(tiling)
        flags = ((_ck.GRAPH_EDGES_IN_HOST_MEMORY if self.edges_in_host_memory else 0) |
                 (_ck.GRAPH_TILING if self.tiling else 0))
        with torch.cuda.device(self.device):
            self._h = _ck.ck_graph_create(src.contiguous(), dst.contiguous(), self.num_nodes,
                                          input_nodes.contiguous(), flags=flags)
        self._ws = {}

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                _ck.ck_graph_destroy(h)
            except Exception:
                pass
            self._h = None

    @property
    def handle(self):
        return self._h

    def export(self):
        with torch.cuda.device(self.device):
            return _ck.ck_graph_export(self._h, self.device)

    def workspace_size(self, B: int, T: int, microsteps: int):
        return _ck.ck_workspace_size(self._h, B, T, microsteps)

    def scratch(self, B: int, T: int, microsteps: int):
        """A cached scratch buffer for (B, T, microsteps) on this graph's device
        (the last shape asked for is kept).  Calls that may run at the same
        time, on different streams, need buffers of their own: pass scratch=
        to forward / backward."""
        key = (B, T, microsteps)
        buf = self._ws.get(key)
        if buf is None:
            _, nbytes = self.workspace_size(B, T, microsteps)
            buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            self._ws = {key: buf}
        return buf


def forward(graph: SparseGraph, edge_values, leak, bias, drives, state0, microsteps: int,
            scratch=None):
    """Raw forward: returns (out [T,B,N], saved buffer, scratch buffer)."""
    B, N = state0.shape
    T = drives.shape[0]
    saved_b, _ = graph.workspace_size(B, T, microsteps)
    saved = torch.empty(saved_b, dtype=torch.uint8, device=state0.device)
    if scratch is None:
        scratch = graph.scratch(B, T, microsteps)
    out = torch.empty((T, B, N), dtype=torch.float32, device=state0.device)
    _ck.ck_forward(graph.handle, edge_values, leak, bias, drives, state0, microsteps, out,
                   saved, scratch)
    return out, saved, scratch


def backward(graph: SparseGraph, edge_values, leak, B: int, T: int, microsteps: int, saved,
             d_out, scratch=None):
    """Raw backward: returns (d_edge_values, d_leak, d_bias, d_drives, d_state0)."""
    dev = d_out.device
    N, E, n_in = graph.num_nodes, graph.num_edges, graph.num_inputs
    if scratch is None:
        scratch = graph.scratch(B, T, microsteps)
    dw = torch.empty(E, dtype=torch.float32, device=dev)
    dl = torch.empty(N, dtype=torch.float32, device=dev)
    db = torch.empty(N, dtype=torch.float32, device=dev)
    dd = torch.empty((T, n_in, B), dtype=torch.float32, device=dev)
    dh = torch.empty((B, N), dtype=torch.float32, device=dev)
    _ck.ck_backward(graph.handle, edge_values, leak, B, T, microsteps, saved, d_out.contiguous(),
                    dw, dl, db, dd, dh, scratch)
    return dw, dl, db, dd, dh


def forward_checkpointed(graph: SparseGraph, edge_values, leak, bias, drives, state0,
                         microsteps: int):
    """Forward that keeps only the state after every input step: returns
    (out [T,B,N], checkpoints, scratch buffer) for backward_recompute."""
    B, N = state0.shape
    T = drives.shape[0]
    ckpt_b, scratch_b = _ck.ck_workspace_size_recompute(graph.handle, B, T, microsteps)
    ckpt = torch.empty(ckpt_b, dtype=torch.uint8, device=state0.device)
    scratch = torch.empty(scratch_b, dtype=torch.uint8, device=state0.device)
    out = torch.empty((T, B, N), dtype=torch.float32, device=state0.device)
    _ck.ck_forward_checkpointed(graph.handle, edge_values, leak, bias, drives, state0,
                                microsteps, out, ckpt, scratch)
    return out, ckpt, scratch


def backward_recompute(graph: SparseGraph, edge_values, leak, bias, drives, B: int, T: int,
                       microsteps: int, ckpt, d_out, scratch=None):
    """Backward from checkpoints (recomputes each input step's microsteps):
    returns (d_edge_values, d_leak, d_bias, d_drives, d_state0)."""
    dev = d_out.device
    N, E, n_in = graph.num_nodes, graph.num_edges, graph.num_inputs
    if scratch is None:
        _, scratch_b = _ck.ck_workspace_size_recompute(graph.handle, B, T, microsteps)
        scratch = torch.empty(scratch_b, dtype=torch.uint8, device=dev)
    dw = torch.empty(E, dtype=torch.float32, device=dev)
    dl = torch.empty(N, dtype=torch.float32, device=dev)
    db = torch.empty(N, dtype=torch.float32, device=dev)
    dd = torch.empty((T, n_in, B), dtype=torch.float32, device=dev)
    dh = torch.empty((B, N), dtype=torch.float32, device=dev)
    _ck.ck_backward_recompute(graph.handle, edge_values, leak, bias, drives, B, T, microsteps,
                              ckpt, d_out.contiguous(), dw, dl, db, dd, dh, scratch)
    return dw, dl, db, dd, dh


class TrainStep:
    """One training step -- forward, backward of L = sum(out * d_out), and an
    update of edge_values, leak and bias (SGD, or Adam with optimizer="adam") --
    captured once as a CUDA graph and replayed (TrainKernel page: a captured
    step holds the forward, the gradients and the parameter update, with no
    per-operator host launches).  Adam's moments and step count live on the
    device, and each replay advances the count.

    The parameters are updated in place; drives, state0 and d_out are read from
    the tensors given here, so copy new inputs into them before a replay.
    Calling the object replays the step and returns the step's output tensor
    (overwritten by the next replay)."""

    def __init__(self, graph: SparseGraph, edge_values, leak, bias, drives, state0, d_out,
                 microsteps: int, lr: float, optimizer: str = "sgd", betas=(0.9, 0.999),
                 eps: float = 1e-8):
        if optimizer not in ("sgd", "adam"):
            raise ValueError("optimizer is 'sgd' or 'adam'")
        self.graph, self.M = graph, microsteps
        self.optimizer, self.betas, self.eps = optimizer, tuple(betas), eps
        self.w, self.leak, self.bias = edge_values, leak, bias
        self.drives, self.state0, self.d_out = drives, state0, d_out
        dev = state0.device
        B, N = state0.shape
        T = drives.shape[0]
        self.B, self.T = B, T
        saved_b, _ = graph.workspace_size(B, T, microsteps)
        self.saved = torch.empty(saved_b, dtype=torch.uint8, device=dev)
        self.scratch = graph.scratch(B, T, microsteps)
        self.out = torch.empty((T, B, N), dtype=torch.float32, device=dev)
        E, n_in = graph.num_edges, graph.num_inputs
        self.grads = (torch.empty(E, device=dev), torch.empty(N, device=dev),
                      torch.empty(N, device=dev), torch.empty((T, n_in, B), device=dev),
                      torch.empty((B, N), device=dev))
        params = (edge_values, leak, bias)
        self.moments = [(torch.zeros_like(p), torch.zeros_like(p)) for p in params]
        self.step_count = torch.zeros(1, dtype=torch.int64, device=dev)
        # one uncaptured pass with lr = 0 sets the kernels up and leaves the
        # parameters as they are (Adam's moments and count are reset after it)
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            self._step(0.0)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        for m, v in self.moments:
            m.zero_()
            v.zero_()
        self.step_count.zero_()
        torch.cuda.synchronize(dev)
        self.cuda_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.cuda_graph):
            self._step(lr)

    def _step(self, lr: float):
        g, M = self.graph, self.M
        dw, dl, db, dd, dh = self.grads
        _ck.ck_forward(g.handle, self.w, self.leak, self.bias, self.drives, self.state0, M,
                       self.out, self.saved, self.scratch)
        _ck.ck_backward(g.handle, self.w, self.leak, self.B, self.T, M, self.saved, self.d_out,
                        dw, dl, db, dd, dh, self.scratch)
        if self.optimizer == "sgd":
            _ck.ck_sgd_update(self.w, dw, lr)
            _ck.ck_sgd_update(self.leak, dl, lr)
            _ck.ck_sgd_update(self.bias, db, lr)
        else:
            _ck.ck_step_advance(self.step_count)
            b1, b2 = self.betas
            for p, gr, (m, v) in zip((self.w, self.leak, self.bias), (dw, dl, db), self.moments):
                _ck.ck_adam_update(p, gr, m, v, self.step_count, lr, b1, b2, self.eps)

    def __call__(self):
        self.cuda_graph.replay()
        return self.out


class _SparseRecurrence(torch.autograd.Function):
    @staticmethod
    def forward(ctx, edge_values, leak, bias, drives, state0, graph, microsteps, recompute):
        ev = edge_values.detach().contiguous()
        lk = leak.detach().contiguous()
        bs = bias.detach().contiguous()
        dr = drives.detach().contiguous()
        if recompute:
            out, saved, _ = forward_checkpointed(graph, ev, lk, bs, dr,
                                                 state0.detach().contiguous(), microsteps)
            ctx.save_for_backward(ev, lk, bs, dr)
        else:
            out, saved, _ = forward(graph, ev, lk, bs, dr, state0.detach().contiguous(),
                                    microsteps)
            ctx.save_for_backward(ev, lk)
        ctx.graph, ctx.microsteps, ctx.recompute = graph, microsteps, recompute
        ctx.shape = (state0.shape[0], drives.shape[0])
        ctx.saved_buf = saved
        return out

    @staticmethod
    def backward(ctx, d_out):
        B, T = ctx.shape
        if ctx.recompute:
            ev, lk, bs, dr = ctx.saved_tensors
            grads = backward_recompute(ctx.graph, ev, lk, bs, dr, B, T, ctx.microsteps,
                                       ctx.saved_buf, d_out)
        else:
            ev, lk = ctx.saved_tensors
            grads = backward(ctx.graph, ev, lk, B, T, ctx.microsteps, ctx.saved_buf, d_out)
        ctx.saved_buf = None
        return (*grads, None, None, None)


def sparse_recurrence(edge_values, leak, bias, drives, state0, graph: SparseGraph,
                      microsteps: int = 1, recompute: bool = False):
    """out[T, B, N]: node states after each of the T input steps.  With
    recompute=True only the state after every input step is kept for the
    backward, which recomputes the microsteps (about M times less memory, the
    same results)."""
    return _SparseRecurrence.apply(edge_values, leak, bias, drives, state0, graph, microsteps,
                                   recompute)
