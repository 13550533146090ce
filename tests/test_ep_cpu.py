"""Expert-parallel split, host logic on gloo CPU ranks (world sizes 2 and 4).

Every rank runs the oracle on its shard of each layer -- the router
replicated, the records of other ranks' experts absent (written here as
all-zero records: code 0, scale 0, bias 0, so their weights and outputs are
0), the shared expert and the residual add on rank 0 -- and the shards'
outputs are summed with a gloo all-reduce before the next layer.  The result
must equal the unsharded oracle over the same stacked layers.
"""
import copy
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as td
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# small stack: hidden 256, 16 experts, top-4, inter 128, shared expert,
# pre-norm + residual, 3 layers, 4 rows
H, E, K, I, NL, NB = 256, 16, 4, 128, 3, 4


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def make_stack():
    from quantized_routed_expert_fn_gb300 import synth
    rng = np.random.default_rng(77)
    layers = [synth.make_layer(rng, H, E, K, I, 4, shared=True, flags=synth.RESIDUAL | synth.PRENORM)
              for _ in range(NL)]
    x = synth.make_x(rng, NB, H)
    return layers, x


def shard_for_oracle(layer, rank, world):
    from quantized_routed_expert_fn_gb300 import ep
    m = ep.owned_mask(layer.n_experts, rank, world)
    L = copy.copy(layer)
    L.records = layer.records.copy()
    L.records[~m] = 0
    if not ep.holds_shared(rank):
        L.shared_gate = L.shared_record = L.shared_layout = None
    L.flags = ep.shard_flags(layer.flags, rank)
    return L


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    td.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from quantized_routed_expert_fn_gb300 import ep
    layers, x = make_stack()
    shards = [oracle.Layer(shard_for_oracle(L, rank, world)) for L in layers]
    ids = []

    def step(l, xl):
        r = oracle.moe_layer(shards[l], xl.numpy())
        ids.append(r["idx"])
        return torch.from_numpy(r["out"])

    y = ep.run_layers(NL, torch.from_numpy(x.astype(np.float64)), step, td.all_reduce)
    out[rank] = (y.numpy(), np.stack(ids))
    td.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_expert_parallel_sum_equals_unsharded_oracle(world):
    import oracle
    layers, x = make_stack()
    ref = oracle.moe_forward([oracle.Layer(L) for L in layers], x)
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    scale = np.abs(ref["out"]).max()
    for r in range(world):
        y, ids = res[r]
        # every rank ends each layer with the same (reduced) activations
        assert np.allclose(y, ref["out"], rtol=0, atol=1e-12 * scale), f"rank {r}"
        # the replicated router routes identically on every rank
        assert np.array_equal(ids, ref["idx"]), f"rank {r} routing"


@pytest.mark.parametrize("n_experts,world", [(16, 2), (16, 4), (512, 8), (10, 4), (3, 4), (128, 3)])
def test_partition_covers_every_expert_once(n_experts, world):
    from quantized_routed_expert_fn_gb300 import ep
    masks = np.stack([ep.owned_mask(n_experts, r, world) for r in range(world)])
    assert (masks.sum(axis=0) == 1).all()
    sizes = masks.sum(axis=1)
    assert sizes.max() - sizes.min() <= 1
    for r in range(world):
        lo, hi = ep.owned_range(n_experts, r, world)
        assert masks[r, lo:hi].all() and masks[r].sum() == hi - lo


def test_shared_expert_and_residual_on_rank_zero_only():
    from quantized_routed_expert_fn_gb300 import ep, synth
    f = synth.RESIDUAL | synth.PRENORM
    assert ep.holds_shared(0) and not any(ep.holds_shared(r) for r in range(1, 8))
    assert ep.shard_flags(f, 0) == f
    assert all(ep.shard_flags(f, r) == synth.PRENORM for r in range(1, 8))
    with pytest.raises(ValueError):
        ep.owned_range(16, 4, 4)


def test_shard_of_one_rank_is_the_masked_sum():
    """One layer, no exchange: rank r's oracle output is exactly the combine
    over its own experts (plus shared and residual on rank 0)."""
    import oracle
    from quantized_routed_expert_fn_gb300 import ep
    layers, x = make_stack()
    L = layers[0]
    full = oracle.moe_layer(oracle.Layer(L), x)
    xn = x / np.sqrt((x.astype(np.float64) ** 2).mean(axis=1, keepdims=True) + 1e-6)
    total = np.zeros_like(full["out"])
    for r in range(4):
        part = oracle.moe_layer(oracle.Layer(shard_for_oracle(L, r, 4)), x)["out"]
        m = ep.owned_mask(E, r, 4)
        want = np.zeros_like(part)
        for b in range(NB):
            for j in range(K):
                e = int(full["idx"][b, j])
                if m[e]:
                    want[b] += full["w"][b, j] * oracle.expert(oracle.Layer(L), e, xn[b])
            if r == 0:
                want[b] += full["gamma"][b] * oracle.shared_expert(oracle.Layer(L), xn[b]) + x[b]
        assert np.allclose(part, want, rtol=0, atol=1e-12 * np.abs(full["out"]).max()), f"rank {r}"
        total += part
    assert np.allclose(total, full["out"], rtol=0, atol=1e-12 * np.abs(full["out"]).max())
