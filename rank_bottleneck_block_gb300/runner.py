"""Device-buffer plumbing around the C ABI for one MLP block, one projection
group and one block stack.

torch only allocates device memory and supplies the stream; every computation
is a call into liblowrank.so through the ctypes binding.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import torch

from . import lowrank as L
from .inputs import MlpShape, ProjShape

_U8 = torch.uint8


def _dt(name: str) -> int:
    return L.LR_BF16 if name == "bf16" else L.LR_F32


def _tdt(name: str) -> torch.dtype:
    return torch.bfloat16 if name == "bf16" else torch.float32


def _buf(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=_U8, device=device)


class MlpBlock:
    """One low-rank SwiGLU MLP block resident on the device (weights, saved set, workspaces, grads)."""

    def __init__(self, shape: MlpShape, case: Dict[str, torch.Tensor], mode: int = L.LR_SAVE_CKPT,
                 device="cuda", act: int = L.LR_ACT_SILU):
        self.s, self.mode, self.device, self.act = shape, mode, device, act
        self.dt = _dt(shape.dtype)
        dev = {k: v.to(device) for k, v in case.items()}
        self.t = dev
        T, d, f, r = shape.T, shape.d, shape.f, shape.r
        self.out = torch.empty(T, d, dtype=_tdt(shape.dtype), device=device)
        self.dx = torch.empty_like(self.out)
        self.saved = _buf(L.lr_mlp_saved_bytes(self.dt, mode, T, d, f, r), device)
        self.ws_f = _buf(L.lr_mlp_fwd_workspace_bytes(self.dt, mode, T, d, f, r), device)
        self.ws_b = _buf(L.lr_mlp_bwd_workspace_bytes(self.dt, mode, T, d, f, r), device)
        f32 = dict(dtype=torch.float32, device=device)
        self.dg = torch.empty(d, **f32)
        self.grads = {}
        for k, (ri, co) in {"gate": (r, d), "up": (r, d), "down": (r, f)}.items():
            do = f if k != "down" else d
            self.grads[f"dA_{k}"] = torch.empty(ri, co, **f32)
            self.grads[f"dB_{k}"] = torch.empty(do, r, **f32)

    def pairs(self):
        t = self.t
        return (L.pair(t["A_gate"], t["B_gate"]), L.pair(t["A_up"], t["B_up"]), L.pair(t["A_down"], t["B_down"]))

    def forward(self, x: Optional[torch.Tensor] = None, stream=None, out: Optional[torch.Tensor] = None):
        s = self.s
        x = self.t["x"] if x is None else x
        out = self.out if out is None else out
        L.lr_mlp_fwd(self.dt, self.mode, s.T, s.d, s.f, s.r, s.eps, x, self.t["g"], *self.pairs(), out,
                     self.saved, self.ws_f, stream, act=self.act)
        return out

    def backward(self, dout: Optional[torch.Tensor] = None, x: Optional[torch.Tensor] = None, stream=None,
                 dx: Optional[torch.Tensor] = None):
        s, gr = self.s, self.grads
        x = self.t["x"] if x is None else x
        dout = self.t["G"] if dout is None else dout
        dx = self.dx if dx is None else dx
        L.lr_mlp_bwd(self.dt, self.mode, s.T, s.d, s.f, s.r, s.eps, x, self.t["g"], *self.pairs(), self.saved, dout,
                     dx, self.dg, L.pair_grad(gr["dA_gate"], gr["dB_gate"]),
                     L.pair_grad(gr["dA_up"], gr["dB_up"]), L.pair_grad(gr["dA_down"], gr["dB_down"]), self.ws_b,
                     stream, act=self.act)
        return dx

    def step(self, stream=None):
        self.forward(stream=stream)
        self.backward(stream=stream)


class DenseBlock:
    """The full-rank SwiGLU MLP block of the same d, f, resident on the device: the reference point
    the low-rank block is compared with."""

    def __init__(self, shape: MlpShape, case: Dict[str, torch.Tensor], device="cuda"):
        self.s, self.device = shape, device
        self.dt = _dt(shape.dtype)
        self.t = {k: v.to(device) for k, v in case.items()}
        T, d, f = shape.T, shape.d, shape.f
        self.out = torch.empty(T, d, dtype=_tdt(shape.dtype), device=device)
        self.dx = torch.empty_like(self.out)
        self.saved = _buf(L.lr_dense_saved_bytes(self.dt, T, d, f), device)
        self.ws_f = _buf(L.lr_dense_fwd_workspace_bytes(self.dt, T, d, f), device)
        self.ws_b = _buf(L.lr_dense_bwd_workspace_bytes(self.dt, T, d, f), device)
        f32 = dict(dtype=torch.float32, device=device)
        self.dg = torch.empty(d, **f32)
        self.grads = {"dW_gate": torch.empty(f, d, **f32), "dW_up": torch.empty(f, d, **f32),
                      "dW_down": torch.empty(d, f, **f32)}

    def forward(self, x: Optional[torch.Tensor] = None, stream=None):
        s, t = self.s, self.t
        x = t["x"] if x is None else x
        L.lr_dense_fwd(self.dt, s.T, s.d, s.f, s.eps, x, t["g"], t["W_gate"], t["W_up"], t["W_down"], self.out,
                       self.saved, self.ws_f, stream)
        return self.out

    def backward(self, dout: Optional[torch.Tensor] = None, x: Optional[torch.Tensor] = None, stream=None):
        s, t, gr = self.s, self.t, self.grads
        x = t["x"] if x is None else x
        dout = t["G"] if dout is None else dout
        L.lr_dense_bwd(self.dt, s.T, s.d, s.f, s.eps, x, t["g"], t["W_gate"], t["W_up"], t["W_down"], self.saved,
                       dout, self.dx, self.dg, gr["dW_gate"], gr["dW_up"], gr["dW_down"], self.ws_b, stream)
        return self.dx

    def step(self, stream=None):
        self.forward(stream=stream)
        self.backward(stream=stream)


class HostPipeline:
    """fwd + bwd of an MlpBlock over batches that live in (pinned) host memory.

    Step i copies x_i and dout_i to the device on a copy stream, runs the block on the
    compute stream and copies out_i and dx_i back on a second copy stream; with two device
    buffer sets the copies of steps i+1 and i-1 overlap the compute of step i.
    """

    def __init__(self, blk: MlpBlock):
        self.blk = blk
        s, dev = blk.s, blk.device
        td = _tdt(s.dtype)
        self.x = [torch.empty(s.T, s.d, dtype=td, device=dev) for _ in range(2)]
        self.G = [torch.empty(s.T, s.d, dtype=td, device=dev) for _ in range(2)]
        self.out = [torch.empty(s.T, s.d, dtype=td, device=dev) for _ in range(2)]
        self.dx = [torch.empty(s.T, s.d, dtype=td, device=dev) for _ in range(2)]
        self.h2d = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)
        self.ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the set copied in
        self.ev_done = [torch.cuda.Event() for _ in range(2)]  # compute of the set finished
        self.ev_read = [torch.cuda.Event() for _ in range(2)]  # results of the set copied out

    def bytes_per_step(self):
        e = self.x[0].element_size() * self.x[0].numel()
        return 2 * e, 2 * e  # (host -> device: x, dout), (device -> host: out, dx)

    def run(self, xh: List[torch.Tensor], gh: List[torch.Tensor], outh: torch.Tensor, dxh: torch.Tensor,
            steps: int, stream=None):
        """Runs `steps` steps on batches xh[i % len], gh[i % len]; results land in outh, dxh."""
        blk = self.blk
        comp = stream if stream is not None else torch.cuda.current_stream(blk.device)
        self.h2d.wait_stream(comp)
        self.d2h.wait_stream(comp)
        for i in range(steps):
            b = i % 2
            with torch.cuda.stream(self.h2d):
                if i >= 2:
                    self.h2d.wait_event(self.ev_done[b])  # step i-2 no longer reads this input set
                self.x[b].copy_(xh[i % len(xh)], non_blocking=True)
                self.G[b].copy_(gh[i % len(gh)], non_blocking=True)
                self.ev_in[b].record(self.h2d)
            comp.wait_event(self.ev_in[b])
            if i >= 2:
                comp.wait_event(self.ev_read[b])  # step i-2's results have been copied out of this set
            blk.forward(self.x[b], stream=comp.cuda_stream, out=self.out[b])
            blk.backward(self.G[b], self.x[b], stream=comp.cuda_stream, dx=self.dx[b])
            self.ev_done[b].record(comp)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(self.ev_done[b])
                outh.copy_(self.out[b], non_blocking=True)
                dxh.copy_(self.dx[b], non_blocking=True)
                self.ev_read[b].record(self.d2h)
        comp.wait_stream(self.d2h)
        comp.wait_stream(self.h2d)


class ProjGroup:
    """A group of low-rank pairs sharing one input, optionally behind an RMSNorm."""

    def __init__(self, shape: ProjShape, case: Dict[str, object], device="cuda", act: int = L.LR_ACT_SILU):
        self.s, self.device, self.act = shape, device, act
        self.dt = _dt(shape.dtype)
        s = shape
        self.x = case["x"].to(device)
        self.g = case["g"].to(device) if case["g"] is not None else None
        self.A = [a.to(device) for a in case["A"]]
        self.B = [b.to(device) for b in case["B"]]
        self.G = [gg.to(device) for gg in case["G"]] if "G" in case else None
        td = _tdt(s.dtype)
        self.outs = [torch.empty(s.T, s.d_out, dtype=td, device=device) for _ in range(s.group)]
        self.dx = torch.empty(s.T, s.d_in, dtype=td, device=device)
        norm = self.g is not None
        self.saved = _buf(L.lr_proj_saved_bytes(self.dt, s.T, s.d_in, s.d_out, s.r, s.group, norm), device)
        self.ws_f = _buf(L.lr_proj_fwd_workspace_bytes(self.dt, s.T, s.d_in, s.d_out, s.r, s.group, norm), device)
        self.ws_b = _buf(L.lr_proj_bwd_workspace_bytes(self.dt, s.T, s.d_in, s.d_out, s.r, s.group, norm), device)
        f32 = dict(dtype=torch.float32, device=device)
        self.dg = torch.empty(s.d_in, **f32) if norm else None
        self.dA = [torch.empty(s.r, s.d_in, **f32) for _ in range(s.group)]
        self.dB = [torch.empty(s.d_out, s.r, **f32) for _ in range(s.group)]

    def pairs(self):
        return [L.pair(a, b) for a, b in zip(self.A, self.B)]

    def forward(self, stream=None):
        s = self.s
        L.lr_proj_fwd(self.dt, s.T, s.d_in, s.d_out, s.r, self.pairs(), self.g, s.eps, self.x, self.outs, self.saved,
                      self.ws_f, stream, act=self.act)
        return self.outs

    def backward(self, stream=None):
        s = self.s
        L.lr_proj_bwd(self.dt, s.T, s.d_in, s.d_out, s.r, self.pairs(), self.g, s.eps, self.x, self.saved, self.G,
                      self.dx, self.dg, [L.pair_grad(a, b) for a, b in zip(self.dA, self.dB)], self.ws_b, stream,
                      act=self.act)
        return self.dx

    def step(self, stream=None):
        self.forward(stream)
        self.backward(stream)


class BlockStack:
    """A residual stack of MLP blocks trained with an MSE loss (one call per step)."""

    def __init__(self, shape: MlpShape, case: Dict[str, object], mode: int = L.LR_SAVE_CKPT, device="cuda"):
        self.s, self.mode, self.device = shape, mode, device
        self.dt = _dt(shape.dtype)
        s = shape
        self.x = case["x"].to(device)
        self.target = case["target"].to(device)
        self.blocks: List[Dict[str, torch.Tensor]] = [{k: v.to(device) for k, v in b.items()}
                                                      for b in case["blocks"]]
        n = len(self.blocks)
        self.ws = _buf(L.lr_stack_workspace_bytes(self.dt, mode, n, s.T, s.d, s.f, s.r), device)
        f32 = dict(dtype=torch.float32, device=device)
        self.loss = torch.zeros(1, **f32)
        self.dx = torch.empty(s.T, s.d, dtype=_tdt(s.dtype), device=device)
        self.dgs = [torch.empty(s.d, **f32) for _ in range(n)]
        self.grads = []
        for _ in range(n):
            gr = {}
            for k, (ri, co, do) in {"gate": (s.r, s.d, s.f), "up": (s.r, s.d, s.f), "down": (s.r, s.f, s.d)}.items():
                gr[f"dA_{k}"] = torch.empty(ri, co, **f32)
                gr[f"dB_{k}"] = torch.empty(do, s.r, **f32)
            self.grads.append(gr)

    def step(self, stream=None):
        s = self.s
        pairs, grads = [], []
        for b, gr in zip(self.blocks, self.grads):
            for k in ("gate", "up", "down"):
                pairs.append(L.pair(b[f"A_{k}"], b[f"B_{k}"]))
                grads.append(L.pair_grad(gr[f"dA_{k}"], gr[f"dB_{k}"]))
        L.lr_stack_step(self.dt, self.mode, s.T, s.d, s.f, s.r, s.eps, self.x, self.target,
                        [b["g"] for b in self.blocks], pairs, self.loss, self.dx, self.dgs, grads, self.ws, stream)
        return self.loss


class GraphStep:
    """A step captured once as a CUDA graph and replayed with one launch.

    `fn` enqueues the step on torch's current stream (every runner above does when given no
    stream).  Capture records its launches, programmatic-launch edges included, with their
    arguments: the buffers the step reads and writes must stay where they are, and new inputs
    are copied into them.  Replaying removes the host cost of issuing each launch, which bounds
    steps of a few tens of microseconds.
    """

    def __init__(self, fn, warmup: int = 2):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # first launches (kernel attributes, caches) outside the capture
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()

    def __call__(self) -> None:
        self.graph.replay()


class Attention:
    """Causal multi-head self-attention between the projection groups, resident on the device.

    q, k, v [b*s, H*dh] bf16 (token-major, as the projections write them); forward() writes o
    and keeps the row log-sum-exp; backward() takes dout and writes dq, dk, dv.
    """

    def __init__(self, b: int, s: int, H: int, dh: int, q, k, v, device="cuda", scale: Optional[float] = None):
        self.b, self.s, self.H, self.dh = b, s, H, dh
        self.scale = float(scale if scale is not None else dh ** -0.5)
        self.q, self.k, self.v = (t.to(device=device, dtype=torch.bfloat16).contiguous() for t in (q, k, v))
        self.o = torch.empty_like(self.q)
        self.dq, self.dk, self.dv = (torch.empty_like(self.q) for _ in range(3))
        self.dout = torch.empty_like(self.q)
        self.saved = _buf(L.lr_attn_saved_bytes(b, s, H, dh), device)
        self.ws = _buf(L.lr_attn_workspace_bytes(b, s, H, dh), device)

    def forward(self, stream=None):
        L.lr_attn_fwd(L.LR_BF16, self.b, self.s, self.H, self.dh, self.scale, self.q, self.k, self.v, self.o,
                      self.saved, self.ws, stream)

    def backward(self, dout: Optional[torch.Tensor] = None, stream=None):
        if dout is not None:
            self.dout.copy_(dout)
        L.lr_attn_bwd(L.LR_BF16, self.b, self.s, self.H, self.dh, self.scale, self.q, self.k, self.v, self.o,
                      self.saved, self.dout, self.dq, self.dk, self.dv, self.ws, stream)

    def step(self, stream=None):
        self.forward(stream)
        self.backward(None, stream)


class TransformerBlock:
    """One low-rank transformer block (q/k/v group, causal attention, o-projection with its
    residual, MLP block in checkpoint mode) resident on the device, bf16."""

    def __init__(self, shape, case: Dict[str, torch.Tensor], device="cuda"):
        self.sh = shape
        self.t = {k: v.to(device).contiguous() for k, v in case.items()}
        t = self.t
        self.w = L.lr_block_weights(
            L._p(t["g_attn"]), *(L.pair(t[f"A_{n}"], t[f"B_{n}"]) for n in "qkvo"), L._p(t["g_mlp"]),
            *(L.pair(t[f"A_{n}"], t[f"B_{n}"]) for n in ("gate", "up", "down")))
        self.grads = {}
        for n in ("q", "k", "v", "o", "gate", "up", "down"):
            self.grads[f"dA_{n}"] = torch.empty(t[f"A_{n}"].shape, dtype=torch.float32, device=device)
            self.grads[f"dB_{n}"] = torch.empty(t[f"B_{n}"].shape, dtype=torch.float32, device=device)
        self.dg_attn = torch.empty(shape.d, dtype=torch.float32, device=device)
        self.dg_mlp = torch.empty(shape.d, dtype=torch.float32, device=device)
        gr = self.grads
        self.g = L.lr_block_grads(
            L._p(self.dg_attn), *(L.pair_grad(gr[f"dA_{n}"], gr[f"dB_{n}"]) for n in "qkvo"), L._p(self.dg_mlp),
            *(L.pair_grad(gr[f"dA_{n}"], gr[f"dB_{n}"]) for n in ("gate", "up", "down")))
        dims = (shape.b, shape.s, shape.H, shape.dh, shape.f, shape.ra, shape.rm)
        self.dims = dims
        self.out = torch.empty_like(t["x"])
        self.dx = torch.empty_like(t["x"])
        self.saved = _buf(L.lr_block_saved_bytes(*dims), device)
        self.ws = _buf(L.lr_block_workspace_bytes(*dims), device)

    def forward(self, stream=None):
        L.lr_block_fwd(L.LR_BF16, *self.dims, self.sh.eps, self.t["x"], self.w, self.out, self.saved, self.ws, stream)

    def backward(self, stream=None):
        L.lr_block_bwd(L.LR_BF16, *self.dims, self.sh.eps, self.t["x"], self.w, self.saved, self.t["G"], self.dx,
                       self.g, self.ws, stream)

    def step(self, stream=None):
        self.forward(stream)
        self.backward(stream)
