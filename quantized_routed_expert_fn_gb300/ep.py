"""Expert-parallel split of the routed MoE step over G ranks, one GPU each.

The experts of a layer are partitioned over the ranks in contiguous blocks;
the router (and so the routing) is replicated on every rank.  Rank r holds
only the records of its own experts: in its `moe_layer` the other experts'
`expert_addr` entries are 0, so the kernel routes them as usual but computes
nothing for them.  The shared expert and the residual add live on rank 0.
Each rank's layer output is then its partial combine, and a sum all-reduce
of the fp32 [nb][H] outputs gives every rank the full layer output, which is
the next layer's input.  This is the one exchange step of the path.

Source: `Gpu::experts_b` (struct Gpu page): the combine is a sum over the
union's experts plus the shared expert, so any partition of the experts
gives partial sums that add up to it.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import moe, synth


def owned_range(n_experts: int, rank: int, world: int) -> tuple[int, int]:
    """Experts [lo, hi) of `rank`: contiguous blocks whose sizes differ by at most one."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside 0..{world - 1}")
    return n_experts * rank // world, n_experts * (rank + 1) // world


def owned_mask(n_experts: int, rank: int, world: int) -> np.ndarray:
    lo, hi = owned_range(n_experts, rank, world)
    m = np.zeros(n_experts, dtype=bool)
    m[lo:hi] = True
    return m


def holds_shared(rank: int) -> bool:
    """The shared expert (and the residual add) live on rank 0 only."""
    return rank == 0


def shard_flags(flags: int, rank: int) -> int:
    """Rank 0 keeps the residual add; every rank keeps the pre-norm (the norm
    of the replicated input is the same on every rank)."""
    return flags if holds_shared(rank) else flags & ~moe.RESIDUAL


def run_layers(n_layers: int, x, layer_step, all_reduce):
    """x_{l+1} = all_reduce(layer_step(l, x_l)) for l = 0 .. n_layers - 1.

    layer_step(l, x) returns this rank's partial output of layer l (a new
    tensor); all_reduce sums it over the ranks in place.  Returns x_n."""
    for l in range(n_layers):
        y = layer_step(l, x)
        all_reduce(y)
        x = y
    return x


class ShardLayers:
    """This rank's device copy of a layer stack: the replicated router, the
    records of its own experts only, the shared expert on rank 0."""

    def __init__(self, layers, rank: int, world: int, device="cuda"):
        self.rank, self.world = rank, world
        self.tensors = []
        arr = (moe.MoeLayer * len(layers))()
        for i, L in enumerate(layers):
            lo, hi = owned_range(L.n_experts, rank, world)
            dev_layer = isinstance(L, synth.DeviceLayer)
            if dev_layer:
                router, recs = L.router, L.records[lo:hi]
            else:
                router = torch.from_numpy(L.router.view(np.int16)).to(device)
                recs = torch.from_numpy(np.ascontiguousarray(L.records[lo:hi])).to(device)
            stride = L.layout.stride
            eaddr = torch.zeros(L.n_experts, dtype=torch.int64, device=router.device)
            if hi > lo:
                eaddr[lo:hi] = torch.arange(hi - lo, dtype=torch.int64, device=router.device) * stride + recs.data_ptr()
            sg = srec = None
            if L.shared_gate is not None and holds_shared(rank):
                if dev_layer:
                    sg, srec = L.shared_gate, L.shared_record
                else:
                    sg = torch.from_numpy(L.shared_gate.view(np.int16)).to(device)
                    srec = torch.from_numpy(L.shared_record).to(device)
            self.tensors += [router, recs, eaddr, sg, srec]
            c = arr[i]
            c.hidden, c.n_experts, c.top_k, c.inter = L.hidden, L.n_experts, L.top_k, L.inter
            c.bits, c.group, c.flags = L.bits, 64, shard_flags(L.flags, rank)
            c.router = router.data_ptr()
            c.shared_gate = None if sg is None else sg.data_ptr()
            c.shared_record = None if srec is None else srec.data_ptr()
            if sg is not None:
                c.sh_gate_up, c.sh_down = moe._q(L.shared_layout.gate_up), moe._q(L.shared_layout.down)
            c.expert_addr = eaddr.data_ptr()
            c.gate_up, c.down = moe._q(L.layout.gate_up), moe._q(L.layout.down)
        self.c = arr
        self.n = len(layers)
        self.src = layers


def forward(shard: ShardLayers, x: torch.Tensor, work: torch.Tensor, status: torch.Tensor, all_reduce,
            slot_tab=None, wmap=None, stream=None) -> torch.Tensor:
    """The stacked layers on this rank: per layer one moe_forward of the
    rank's shard, then the sum all-reduce of its output.  `all_reduce` is
    e.g. `torch.distributed.all_reduce` (a sum by default).  slot_tab /
    wmap ([n_layers][64] / [n_layers][4][64], or None) receive each layer's
    resident slots.  Returns the last layer's output."""

    def step(l, xl):
        out = torch.empty_like(xl)
        moe.forward(shard, xl, out, work, status, None if slot_tab is None else slot_tab[l],
                    None if wmap is None else wmap[l], n_layers=1, stream=stream, layer_offset=l)
        return out

    return run_layers(shard.n, x, step, all_reduce)


def workspace(shard: ShardLayers, nb: int) -> int:
    """Workspace bytes of one layer's moe_forward on this shard."""
    arr = ctypes.cast(ctypes.byref(shard.c, 0), ctypes.POINTER(moe.MoeLayer))
    return int(moe.lib().moe_forward_workspace(arr, 1, nb))
