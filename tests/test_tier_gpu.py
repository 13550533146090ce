"""Two-tier records on the GPU: routed records in pinned host memory (read
by the kernel over NVLink-C2C) and device-memory slots managed by the
store's LRU, plus the deadline cut of weak host-memory experts.

Where a record lives changes only the order of the union's slots (device
records first) and so the order of the per-slot sums: a tiered step must
match the untiered step (same inputs, same routing) to fp32 rounding, and
list exactly the untiered union with the device-memory records first.  The
cut is graded against the oracle given the same tiers and threshold.
"""
import numpy as np
import pytest

import oracle
from helpers import GAP, TOL, assert_close_rows, topk_gap
from quantized_routed_expert_fn_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_fn_gb300 import build, moe
    build.build()
    moe.lib()
    return moe


def tiered(m, layers, n_slots, cut_weak=0.0):
    nl, E = len(layers), layers[0].n_experts
    stride = layers[0].layout.stride
    host = torch.empty((nl, E, stride), dtype=torch.uint8).pin_memory()
    for l, L in enumerate(layers):
        host[l] = torch.from_numpy(L.records)
    slots = torch.zeros((max(n_slots, 1), stride), dtype=torch.uint8, device="cuda")
    addr = torch.zeros((nl, E), dtype=torch.int64, device="cuda")
    tier = torch.zeros((nl, E), dtype=torch.uint8, device="cuda")
    t = m.Tier(nl, E, stride, host, n_slots, slots, addr, tier)
    dl = m.DeviceLayers(layers)
    for l in range(nl):
        dl.set_tier(l, addr[l], tier[l], cut_weak)
    torch.cuda.synchronize()
    return t, dl, (host, slots, addr, tier)


def run(m, dl, x, nl, offset=0):
    nb, H = x.shape
    xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    out = torch.empty_like(xt)
    ws = m.alloc_workspace(m.forward_workspace(dl.c, nb, nl))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    slot = torch.zeros((nl, 64), dtype=torch.int64, device="cuda")
    wmap = torch.zeros((nl, 4, 64), dtype=torch.float32, device="cuda")
    m.forward(dl, xt, out, ws, status, slot, wmap, n_layers=nl, layer_offset=offset)
    torch.cuda.synchronize()
    assert status.item() == 0, m.STATUS_NAMES.get(status.item())
    return out.cpu().numpy(), slot.cpu().numpy().view(np.uint64), wmap.cpu().numpy()


def cut_between(w):
    """A cut threshold at the median of the routed weights w, but midway
    between two neighbouring weights at least 1e-4 apart, so that no weight
    sits on it (the kernel's fp32 weights and the oracle's fp64 ones then
    fall on the same side)."""
    v = np.unique(np.asarray(w, dtype=np.float64).ravel())
    i = len(v) // 2
    while i + 1 < len(v) and v[i + 1] - v[i] < 1e-4:
        i += 1
    assert i + 1 < len(v), "no gap in the routed weights"
    return float((v[i] + v[i + 1]) / 2)


def experts_of(slot_row, addr_row, n):
    a2e = {int(a): e for e, a in enumerate(addr_row)}
    return [a2e[int(a)] for a in slot_row[:n]]


def test_tiered_steps_match_untiered_and_promote(m):
    """Three layers, 16 experts each, 10 device slots for 48 records; each
    step runs the layers one by one on the untiered trajectory's inputs.
    The first step reads every routed record from host memory; each update
    promotes what the step read, evicting least recently used records.
    Every layer: the same union (device records first, first-seen order
    within each tier), the untiered output to fp32 rounding (1e-5 x row
    RMS: only the order of the per-slot sums differs) and the oracle's
    within 2e-3 x row RMS."""
    rng = np.random.default_rng(950)
    nl, H, E, k, I, nb = 3, 512, 16, 4, 256, 2
    layers = [synth.make_layer(rng, H, E, k, I, 4, shared=True, flags=synth.RESIDUAL | synth.PRENORM)
              for _ in range(nl)]
    ols = [oracle.Layer(L) for L in layers]
    plain = m.DeviceLayers(layers)
    t, dl, keep = tiered(m, layers, n_slots=10)
    addr, tier = keep[2], keep[3]
    eaddr_plain = [plain.tensors[5 * l + 2].cpu().numpy() for l in range(nl)]
    promoted_total, worst, worst_o = 0, 0.0, 0.0
    for step in range(6):
        x = synth.make_x(np.random.default_rng(960 + step), nb, H)
        tier_before = tier.cpu().numpy()
        addr_before = addr.cpu().numpy().view(np.uint64)
        slot = np.zeros((nl, 64), dtype=np.uint64)
        cur = x
        for l in range(nl):
            ref, rslot, _ = run(m, plain, cur, 1, offset=l)
            got, sl, _ = run(m, dl, cur, 1, offset=l)
            slot[l] = sl[0]
            o = oracle.moe_layer(ols[l], cur.astype(np.float64))
            worst = max(worst, assert_close_rows(got, ref, o["moe"], tol=1e-5, what=f"step {step} layer {l} vs untiered"))
            worst_o = max(worst_o, assert_close_rows(got, o["out"], o["moe"], what=f"step {step} layer {l} vs oracle"))
            U = int(rslot[0, 63])
            assert int(sl[0, 63]) == U
            want = experts_of(rslot[0], eaddr_plain[l], U)
            have = experts_of(sl[0], addr_before[l], U)
            assert sorted(have) == sorted(want), f"step {step} layer {l}: union"
            ndev = int(sl[0, 62])
            assert all(tier_before[l][e] == 0 for e in have[:ndev]) and all(tier_before[l][e] == 1 for e in have[ndev:])
            order = {e: i for i, e in enumerate(want)}
            assert [order[e] for e in have[:ndev]] == sorted(order[e] for e in have[:ndev])
            assert [order[e] for e in have[ndev:]] == sorted(order[e] for e in have[ndev:])
            cur = ref
        if step == 0:
            assert all(int(slot[l, 62]) == 0 for l in range(nl)), "every record starts in host memory"
        promoted_total += t.update(slot)
        torch.cuda.synchronize()
        st = t.stats()
        tier_after = tier.cpu().numpy()
        assert int((tier_after == 0).sum()) == st["resident"] <= 10
        for l in range(nl):
            for e in range(E):
                assert (t.slot(l, e) >= 0) == (tier_after[l, e] == 0)
    assert promoted_total >= 10 and t.stats()["evictions"] > 0
    print(f"[tier] 6 steps: {promoted_total} promotions, {t.stats()['evictions']} evictions; "
          f"max err {worst:.3f} of 1e-5 x RMS against untiered, {worst_o:.4f} of 2e-3 x RMS against the oracle")
    t.close()


def test_cut_of_weak_host_experts_matches_oracle(m):
    """Half the records in host memory, the cut near the median routed weight:
    ids exact, the listed slots = the union minus the oracle's cut (device
    records first), output within 2e-3 x row RMS of the oracle with the
    same tiers and threshold."""
    rng = np.random.default_rng(970)
    H, E, k, I, nb = 1024, 32, 6, 256, 4
    layer = synth.make_layer(rng, H, E, k, I, 4, shared=True, flags=synth.PRENORM)
    tier_np = (np.arange(E) % 2).astype(np.uint8)
    for s in range(50):
        x = synth.make_x(np.random.default_rng(980 + s), nb, H)
        r0 = oracle.route(oracle.Layer(layer), x)
        if all(topk_gap(r0["logits"][b], k) >= GAP for b in range(nb)):
            break
    cut_w = cut_between(r0["w"])
    layer.expert_tier, layer.cut_w = tier_np, cut_w
    ol = oracle.Layer(layer)
    ref = oracle.moe_layer(ol, x)
    cut = oracle.cut(ol, ref["idx"], ref["w"])
    assert cut.any()
    # all records stay in device memory, but the tier table marks half as host
    # memory: the cut is a decision on tiers and weights alone
    dl = m.DeviceLayers([layer])
    eaddr = dl.tensors[2]
    tier = torch.from_numpy(tier_np).cuda()
    dl.set_tier(0, eaddr, tier, cut_w)
    got, slot, wmap = run(m, dl, x, 1)
    kept = [int(e) for e in ref["union"] if not cut[e]]
    dev = [e for e in kept if tier_np[e] == 0]
    hst = [e for e in kept if tier_np[e] == 1]
    assert int(slot[0, 62]) == len(dev) and int(slot[0, 63]) == len(ref["union"])
    listed = experts_of(slot[0], eaddr.cpu().numpy(), len(kept))
    assert listed == dev + hst
    assert int(slot[0, len(kept)]) == 0
    r = assert_close_rows(got, ref["out"], ref["moe"], what="cut")
    print(f"[parity] cut of weak host experts (w = {cut_w:.3f}, {int(cut.sum())} cut): max err = {r:.4f} of the bound")


def test_host_memory_records_read_over_c2c(m):
    """Every routed record in pinned host memory, no slots: the kernel reads
    them all over the link; graded against the oracle."""
    rng = np.random.default_rng(990)
    H, E, k, I, nb = 2048, 64, 8, 512, 3
    layer = synth.make_layer(rng, H, E, k, I, 4, shared=True, flags=synth.RESIDUAL | synth.PRENORM)
    ol = oracle.Layer(layer)
    for s in range(50):
        x = synth.make_x(np.random.default_rng(995 + s), nb, H)
        ref = oracle.moe_layer(ol, x)
        if all(topk_gap(ref["logits"][b], k) >= GAP for b in range(nb)):
            break
    t, dl, keep = tiered(m, [layer], n_slots=0)
    got, slot, _ = run(m, dl, x, 1)
    assert int(slot[0, 62]) == 0 and int(slot[0, 63]) == len(ref["union"])
    r = assert_close_rows(got, ref["out"], ref["moe"], what="host-memory records")
    print(f"[parity] all routed records in host memory: max err = {r:.4f} of the bound")
    t.close()


def test_mixed_widths_in_host_memory_with_cut(m):
    """4-, 3- and 2-bit records, every routed record in pinned host memory
    (read over the link by the mixed-width kernel, each at its own width),
    and the cut near the median routed weight: the listed slots are the union
    minus the oracle's cut, in union order; the output is within 2e-3 x row
    RMS of the oracle with the same widths, tiers and threshold."""
    rng = np.random.default_rng(1010)
    H, E, k, I, nb = 1024, 30, 6, 256, 4
    eb = np.array([4, 3, 2] * (E // 3), dtype=np.uint8)
    np.random.default_rng(1011).shuffle(eb)
    layer = synth.make_mixed_layer(rng, H, E, k, I, eb, shared=True, flags=synth.PRENORM)
    for s_ in range(200):
        x = synth.make_x(np.random.default_rng(1020 + s_), nb, H)
        r0 = oracle.route(oracle.Layer(layer), x)
        if all(topk_gap(r0["logits"][b], k) >= GAP for b in range(nb)) and set(eb[r0["union"]].tolist()) == {2, 3, 4}:
            break
    else:
        pytest.fail("no seed with the top-k gap and every width in the union")
    cut_w = cut_between(r0["w"])
    layer.expert_tier, layer.cut_w = np.ones(E, dtype=np.uint8), cut_w
    ol = oracle.Layer(layer)
    ref = oracle.moe_layer(ol, x)
    cut = oracle.cut(ol, ref["idx"], ref["w"])
    assert cut.any() and not cut[ref["union"]].all()
    t, dl, keep = tiered(m, [layer], n_slots=0, cut_weak=cut_w)
    addr = keep[2]
    got, slot, _ = run(m, dl, x, 1)
    kept = [int(e) for e in ref["union"] if not cut[e]]
    assert int(slot[0, 62]) == 0 and int(slot[0, 63]) == len(ref["union"])
    assert experts_of(slot[0], addr[0].cpu().numpy().view(np.uint64), len(kept)) == kept
    r = assert_close_rows(got, ref["out"], ref["moe"], what="mixed widths in host memory, cut")
    print(f"[parity] mixed 4/3/2-bit records in host memory, {int(cut.sum())} cut (w = {cut_w:.3f}): "
          f"max err = {r:.4f} of the bound")
    t.close()


def test_lookahead_with_host_memory_records_changes_nothing(m):
    """A three-layer stack whose records sit partly in device slots and
    partly in pinned host memory (after one promoting step).  With the
    one-layer lookahead on every layer (predicted device records prefetched
    into L2, host ones left to the kernel's own reads), the outputs, slot
    tables and weight maps are bitwise those of the same call without it."""
    rng = np.random.default_rng(1010)
    nl, H, E, k, I, nb = 3, 512, 16, 4, 256, 2
    flags = synth.RESIDUAL | synth.PRENORM
    layers = [synth.make_layer(rng, H, E, k, I, 4, shared=True, flags=flags) for _ in range(nl)]
    t, dl, keep = tiered(m, layers, n_slots=10)
    _, slot0, _ = run(m, dl, synth.make_x(np.random.default_rng(1011), nb, H), nl)
    t.update(slot0)
    torch.cuda.synchronize()
    x = synth.make_x(np.random.default_rng(1012), nb, H)
    base, bslot, bw = run(m, dl, x, nl)
    la = torch.zeros((nl, nb, k), dtype=torch.int32, device="cuda")
    dl.set_flags(flags | m.LOOKAHEAD)
    for l in range(nl):
        dl.c[l].lookahead_idx = la[l].data_ptr()
    got, gslot, gw = run(m, dl, x, nl)
    assert np.array_equal(got.view(np.uint32), base.view(np.uint32)), "lookahead changed the result"
    assert np.array_equal(gslot, bslot) and np.array_equal(gw.view(np.uint32), bw.view(np.uint32))
    ndev = [int(bslot[l, 62]) for l in range(nl)]
    nun = [int(bslot[l, 63]) for l in range(nl)]
    assert any(0 < d < u for d, u in zip(ndev, nun)), "no union mixes the tiers"
    print(f"[tier + lookahead] device / union records per layer: {list(zip(ndev, nun))}; bitwise equal")
    t.close()
