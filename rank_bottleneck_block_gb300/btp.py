"""Bottleneck-aware tensor parallelism (BTP) for a normed group of low-rank pairs.

BOOST technical summary §2.1: BTP keeps the activations of a block sharded along the
hidden width d across the tensor-parallel ranks; a group of A's that reads the (normed)
block input runs row-parallel, each rank reducing over its own d-shard, and the only
collective is one all-reduce of [T, group*r] partial sums at the bottleneck width instead
of [T, d].  §2.2 Online-RMSNorm: RMSNorm needs the global statistic sum_j x_j^2, so each
rank appends its shard's sums of squares to that payload and the normalisation is applied
after the all-reduce (exact: the gain folds into A and 1/rms is a per-row scale).

One rank's step is three calls: lr_btp_partial (device: folded-A GEMM over the shard, fp32
partials and the shard's sums of squares into one payload), an all-reduce of the payload
(torch.distributed: NCCL between GPUs), and lr_btp_finish (device: 1/rms, u, sigma(u)).
`btp_norm_group` is that protocol with the three steps passed in, which is how its sharding,
payload layout and reduction are exercised with CPU ranks.
"""
from __future__ import annotations

from typing import Callable, List, Sequence, Tuple

import torch

from . import lowrank as L


def shard_bounds(d: int, world: int, rank: int, align: int = 8) -> Tuple[int, int]:
    """Columns [lo, hi) of the d-shard of `rank`: contiguous, multiples of `align` (TMA rows)."""
    if d % align or d // align < world:
        raise ValueError(f"d = {d} does not split into {world} shards of multiples of {align}")
    units = d // align
    base, extra = divmod(units, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo * align, hi * align


def payload_floats(T: int, r: int, group: int) -> int:
    """[acc: T x group*r | ss: T]."""
    return T * group * r + T


def btp_norm_group(partial: Callable[[], torch.Tensor], all_reduce: Callable[[torch.Tensor], None],
                   finish: Callable[[torch.Tensor], object]):
    """One rank's BTP step: its partial payload, the all-reduce (sum) over the TP group, the finish."""
    payload = partial()
    all_reduce(payload)
    return finish(payload)


class BtpNormGroup:
    """One rank's share of a normed group of `group` pairs under BTP, resident on its device.

    A_full: the group's A matrices [r, d] (the rank keeps its d-shard of columns); g_full [d].
    forward(x_shard) returns (u, z, s) for the whole [T, group*r] bottleneck, identical on every
    rank, as lr_proj_fwd computes them unsharded (up to the summation order of the partials).
    """

    def __init__(self, dtype: str, T: int, d: int, r: int, A_full: Sequence[torch.Tensor], g_full: torch.Tensor,
                 rank: int = 0, world: int = 1, device="cuda", process_group=None):
        self.dt = L.LR_BF16 if dtype == "bf16" else L.LR_F32
        self.T, self.d, self.r, self.group = T, d, r, len(A_full)
        self.rank, self.world, self.pg = rank, world, process_group
        self.lo, self.hi = shard_bounds(d, world, rank)
        self.A = [a[:, self.lo:self.hi].contiguous().to(device) for a in A_full]
        self.g = g_full[self.lo:self.hi].contiguous().to(device)
        td = torch.bfloat16 if dtype == "bf16" else torch.float32
        n = self.group * r
        self.payload = torch.empty(payload_floats(T, r, self.group), dtype=torch.float32, device=device)
        ws = L.lr_btp_workspace_bytes(self.dt, self.hi - self.lo, r, self.group)
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=device)
        self.u = torch.empty(T, n, dtype=td, device=device)
        self.z = torch.empty_like(self.u)
        self.s = torch.empty(T, dtype=torch.float32, device=device)

    def pairs(self) -> List[L.lr_pair]:
        return [L.lr_pair(a.data_ptr(), 0) for a in self.A]

    def partial(self, x_shard: torch.Tensor, stream=None) -> torch.Tensor:
        L.lr_btp_partial(self.dt, self.T, self.hi - self.lo, self.r, self.pairs(), self.g, x_shard, self.payload,
                         self.ws, stream)
        return self.payload

    def finish(self, payload: torch.Tensor, eps: float, act: int = L.LR_ACT_SILU, stream=None):
        L.lr_btp_finish(self.dt, act, self.T, self.d, self.r, self.group, payload, eps, self.u, self.z, self.s,
                        stream)
        return self.u, self.z, self.s

    def forward(self, x_shard: torch.Tensor, eps: float = 1e-6, act: int = L.LR_ACT_SILU, stream=None):
        def reduce(p: torch.Tensor) -> None:
            if self.world > 1:
                import torch.distributed as dist

                dist.all_reduce(p, op=dist.ReduceOp.SUM, group=self.pg)

        return btp_norm_group(lambda: self.partial(x_shard, stream), reduce,
                              lambda p: self.finish(p, eps, act, stream))


# ----------------------------------------------------------- payload model
def allreduce_floats_per_token(d: int, f: int, r: int) -> dict:
    """All-reduce payload per token of one transformer layer (attention q, k, v, o pairs and the
    SwiGLU MLP gate, up, down pairs), forward pass.

    Low-rank TP that keeps each pair one shard unit (A column-parallel and B row-parallel over r)
    all-reduces every pair's output: q, k, v, o and down are d wide, gate and up f wide.  BTP
    all-reduces the row-parallel A groups at the bottleneck: q/k/v (3r) and gate/up (2r), each
    with one appended RMS statistic, and the o and down A's (r each).
    """
    vanilla = 5 * d + 2 * f
    btp = (3 * r + 1) + r + (2 * r + 1) + r
    return {"vanilla": vanilla, "btp": btp, "ratio": vanilla / btp}
