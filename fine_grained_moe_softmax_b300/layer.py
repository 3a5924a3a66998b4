"""Device-resident MoE layer: packed weights, workspace and outputs for repeated forward calls.

PyTorch only provides the device memory and the stream here; the forward pass itself is one call
of the C ABI's ``moe_layer_forward``.
"""
from __future__ import annotations

import copy
from typing import Optional

import torch

from . import binding as B


class MoELayer:
    """Holds one layer's weights in the library's packed layout plus a workspace sized for up to
    ``cfg.T`` tokens per call.

    centroids [N', d], w_gate / w_up [K_s + N', I, d], w_down [K_s + N', d, I] (shared experts
    first), logit_bias [N'] fp32 or None; all in the config's dtype (bias fp32). With
    ``backward=True`` the transposed weight copies and the workspace of ``backward`` are set up too.
    """

    def __init__(self, cfg: B.MoEConfig, centroids, w_gate, w_up, w_down, logit_bias=None,
                 device="cuda", stream=None, backward: bool = False):
        self.cfg = copy.copy(cfg)
        self.device = torch.device(device)
        dt = cfg.torch_dtype()
        dev = self.device
        self.centroids = centroids.to(dev, dt).contiguous()
        self.logit_bias = None if logit_bias is None else logit_bias.to(dev, torch.float32).contiguous()
        self.packed = torch.empty(B.moe_packed_weight_bytes(self.cfg), dtype=torch.uint8,
                                  device=dev)
        w_gate = w_gate.to(dev, dt).contiguous()
        w_up = w_up.to(dev, dt).contiguous()
        w_down = w_down.to(dev, dt).contiguous()
        B.moe_pack_weights(self.cfg, w_gate, w_up, w_down, self.packed, stream)
        self.packed_bwd = None
        self.ws_bwd = None
        if backward:
            self.packed_bwd = torch.empty(B.moe_packed_backward_bytes(self.cfg), dtype=torch.uint8,
                                          device=dev)
            B.moe_pack_weights_backward(self.cfg, w_gate, w_up, w_down, self.packed_bwd, stream)
            self.ws_bwd = torch.empty(max(B.moe_backward_workspace_bytes(self.cfg), 256),
                                      dtype=torch.uint8, device=dev)
        if stream is None:
            torch.cuda.current_stream(dev).synchronize()
        else:
            stream.synchronize()
        del w_gate, w_up, w_down
        self.ws = torch.empty(max(B.moe_workspace_bytes(self.cfg), 256), dtype=torch.uint8,
                              device=dev)
        T, K, N = cfg.T, cfg.top_k, cfg.n_routed
        self.h = torch.empty(T, cfg.d, dtype=dt, device=dev)
        self.topk_idx = torch.empty(T, K, dtype=torch.int32, device=dev)
        self.topk_gate = torch.empty(T, K, dtype=torch.float32, device=dev)
        self.counts = torch.empty(N, dtype=torch.int32, device=dev)
        self.f = torch.empty(N, dtype=torch.float32, device=dev)
        self.P = torch.empty(N, dtype=torch.float32, device=dev)
        self.losses = torch.empty(2, dtype=torch.float32, device=dev)

    def cfg_for(self, T: int) -> B.MoEConfig:
        if T > self.cfg.T:
            raise ValueError(f"{T} tokens exceed the {self.cfg.T} this layer was sized for")
        c = copy.copy(self.cfg)
        c.T = T
        return c

    def forward(self, u: torch.Tensor, h: Optional[torch.Tensor] = None, stream=None):
        """Runs the layer on u [T, d]; returns h (written into ``self.h[:T]`` unless given)."""
        T = u.shape[0]
        cfg = self.cfg_for(T)
        out = self.h[:T] if h is None else h
        B.moe_layer_forward(cfg, u, self.centroids, self.logit_bias, self.packed, out,
                            self.topk_idx[:T], self.topk_gate[:T], self.counts, self.f, self.P,
                            self.losses, self.ws, stream)
        return out

    def backward(self, u: torch.Tensor, dh: torch.Tensor, stream=None) -> dict:
        """Gradients of sum_t dh_t . h_t + L_ExpBal + L_DevBal (one moe_layer_backward call):
        du, d_centroids, d_bias, dw_gate, dw_up, dw_down as fp32 device tensors."""
        if self.ws_bwd is None:
            raise RuntimeError("construct the layer with backward=True")
        T = u.shape[0]
        cfg = self.cfg_for(T)
        g = self._grad_buffers(T)
        B.moe_layer_backward(cfg, u, self.centroids, self.logit_bias, self.packed,
                             self.packed_bwd, dh, g["du"], g["d_centroids"], g["d_bias"],
                             g["dw_gate"], g["dw_up"], g["dw_down"], self.ws_bwd, stream)
        return g

    def forward_train(self, u: torch.Tensor, h: Optional[torch.Tensor] = None, stream=None):
        """Forward of a training step (moe_layer_forward_train): returns h like ``forward`` and
        keeps in the backward workspace what ``backward_saved`` needs."""
        if self.ws_bwd is None:
            raise RuntimeError("construct the layer with backward=True")
        T = u.shape[0]
        cfg = self.cfg_for(T)
        out = self.h[:T] if h is None else h
        B.moe_layer_forward_train(cfg, u, self.centroids, self.logit_bias, self.packed, out,
                                  self.topk_idx[:T], self.topk_gate[:T], self.counts, self.f,
                                  self.P, self.losses, self.ws_bwd, stream)
        self._saved_T = T
        return out

    def backward_saved(self, u: torch.Tensor, dh: torch.Tensor, stream=None) -> dict:
        """Gradients like ``backward`` from the state of the last ``forward_train`` on the same u
        (moe_layer_backward_saved), without recomputing the forward."""
        T = u.shape[0]
        if getattr(self, "_saved_T", None) != T:
            raise RuntimeError("backward_saved needs a forward_train on the same batch first")
        g = self._grad_buffers(T)
        B.moe_layer_backward_saved(self.cfg_for(T), u, self.centroids, self.logit_bias,
                                   self.packed_bwd, dh, g["du"], g["d_centroids"], g["d_bias"],
                                   g["dw_gate"], g["dw_up"], g["dw_down"], self.ws_bwd, stream)
        return g

    def _grad_buffers(self, T: int) -> dict:
        c, dev, f32 = self.cfg, self.device, torch.float32
        E = c.n_shared + c.n_routed
        return {"du": torch.empty(T, c.d, dtype=f32, device=dev),
                "d_centroids": torch.empty(c.n_routed, c.d, dtype=f32, device=dev),
                "d_bias": torch.empty(c.n_routed, dtype=f32, device=dev),
                "dw_gate": torch.empty(E, c.inter, c.d, dtype=f32, device=dev),
                "dw_up": torch.empty(E, c.inter, c.d, dtype=f32, device=dev),
                "dw_down": torch.empty(E, c.d, c.inter, dtype=f32, device=dev)}

    def capture(self, u: torch.Tensor):
        """Records one forward on the fixed input buffer ``u`` into a CUDA graph and returns
        (graph, kernels_per_replay). Replaying the graph reruns the same kernels on the current
        contents of ``u``, writing the same output buffers; it removes the host-side launch cost,
        which dominates at decode-sized batches. The call before capture sets up per-device state
        (tensor-map encoder, shared-memory limits) so that capture records kernels only."""
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self.forward(u)
        torch.cuda.current_stream(self.device).wait_stream(side)
        torch.cuda.synchronize(self.device)
        graph = torch.cuda.CUDAGraph()
        n0 = B.moe_launch_count()
        with torch.cuda.graph(graph):
            self.forward(u)
        return graph, B.moe_launch_count() - n0

    def routing(self, T: Optional[int] = None) -> dict:
        """The routing tables of the last ``forward`` on T tokens (default: the layer's T), as
        views into the workspace (moe_layer_routing): offsets, perm_token, perm_slot, psum.
        They are overwritten by the next call."""
        return B.moe_layer_routing(self.cfg_for(self.cfg.T if T is None else T), self.ws)

    def device_status(self, stream=None) -> int:
        return B.moe_device_status(self.ws, stream)

    def global_balance_stats(self, T_local: int, group=None, stream=None, via_host=False):
        """Balance statistics over the tokens of every rank in ``group`` after a ``forward`` on
        T_local tokens: the per-rank selection counts and affinity sums (2N' values, the raw sums
        the forward left in its workspace) are summed across ranks, then moe_balance_stats runs
        with the global token count. Returns (f, P, losses) device tensors. Only needed when the
        token batch is split across GPUs; a single GPU's forward already fills f, P and losses.
        ``via_host`` all-reduces CPU copies (for a gloo group)."""
        counts = self.counts.clone()
        psum = self.routing(T_local)["psum"].clone()
        if via_host:
            c_h, p_h = counts.cpu(), psum.cpu()
            T_total = allreduce_routing_stats(c_h, p_h, T_local, group)
            counts.copy_(c_h)
            psum.copy_(p_h)
        else:
            T_total = allreduce_routing_stats(counts, psum, T_local, group)
        cfg = copy.copy(self.cfg)
        cfg.T = T_total
        f = torch.empty_like(self.f)
        P = torch.empty_like(self.P)
        losses = torch.empty_like(self.losses)
        B.moe_balance_stats(cfg, counts, psum, f, P, losses, stream)
        return f, P, losses


def allreduce_routing_stats(counts: torch.Tensor, psum: torch.Tensor, T_local: int,
                            group=None) -> int:
    """Sums per-expert selection counts (int32) and affinity sums (fp32) over the ranks of
    ``group`` in place and returns the total token count. Works on CPU tensors with gloo and on
    CUDA tensors with NCCL."""
    import torch.distributed as dist
    dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(psum, op=dist.ReduceOp.SUM, group=group)
    t = torch.tensor([int(T_local)], dtype=torch.int64, device=counts.device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return int(t.item())
