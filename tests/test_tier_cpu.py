"""The two-tier expert store's policy (LRU over device slots, promotion of
the records a step read from host memory), run policy-only on the CPU: no
device memory and no CUDA call, the slots at stand-in addresses."""
import numpy as np
import pytest

from quantized_routed_expert_fn_gb300 import build

NL, E, STRIDE, SLOTS = 2, 8, 4096, 3
HOST = 1 << 32


@pytest.fixture()
def m():
    build.build()
    from quantized_routed_expert_fn_gb300 import moe
    moe.lib()
    return moe


def host(l, e):
    return HOST + (l * E + e) * STRIDE


def slot_base():
    return HOST + NL * E * STRIDE + 4096


def table(rows):
    """Slot tables listing the given addresses per layer (zero after them)."""
    t = np.zeros((NL, 64), dtype=np.uint64)
    for l, addrs in rows.items():
        t[l, :len(addrs)] = addrs
    return t


def test_starts_in_host_memory(m):
    t = m.Tier(NL, E, STRIDE, HOST, SLOTS)
    a = t.addresses()
    assert all(a[l, e] == host(l, e) for l in range(NL) for e in range(E))
    assert all(t.slot(l, e) == -1 for l in range(NL) for e in range(E))
    assert t.stats()["resident"] == 0


def test_promotes_host_reads_then_evicts_least_recently_used(m):
    t = m.Tier(NL, E, STRIDE, HOST, SLOTS)
    # step 1 reads (0,1), (0,5), (1,2) from host memory: all three fit
    assert t.update(table({0: [host(0, 1), host(0, 5)], 1: [host(1, 2)]})) == 3
    s = {k: t.slot(*k) for k in [(0, 1), (0, 5), (1, 2)]}
    assert sorted(s.values()) == [0, 1, 2]
    a = t.addresses()
    for (l, e), sl in s.items():
        assert a[l, e] == slot_base() + sl * STRIDE
    st = t.stats()
    assert st["resident"] == 3 and st["last_host_reads"] == 3 and st["promotions"] == 3
    # step 2 uses (0,1) from its slot and reads (0,7) from host memory: the
    # least recently used record, (0,5), gives up its slot
    a = t.addresses()
    assert t.update(table({0: [int(a[0, 1]), host(0, 7)]})) == 1
    assert t.slot(0, 5) == -1 and t.slot(0, 7) == s[(0, 5)] and t.slot(0, 1) == s[(0, 1)]
    assert t.addresses()[0, 5] == host(0, 5)
    assert t.stats()["evictions"] == 1
    # step 3 uses all three resident records and reads one more: no slot is free
    a = t.addresses()
    n = t.update(table({0: [int(a[0, 1]), int(a[0, 7]), host(0, 3)], 1: [int(a[1, 2])]}))
    assert n == 0 and t.slot(0, 3) == -1
    assert t.stats()["last_host_reads"] == 1


def test_a_record_listed_twice_counts_once(m):
    t = m.Tier(NL, E, STRIDE, HOST, SLOTS)
    assert t.update(table({0: [host(0, 2), host(0, 2)]})) == 1
    assert t.stats()["last_host_reads"] == 1


def test_no_slots_keeps_everything_in_host_memory(m):
    t = m.Tier(NL, E, STRIDE, HOST, 0)
    assert t.update(table({0: [host(0, 1)], 1: [host(1, 1)]})) == 0
    assert t.slot(0, 1) == -1


def test_rejects_an_address_of_another_layer_or_no_record(m):
    t = m.Tier(NL, E, STRIDE, HOST, SLOTS)
    with pytest.raises(m.MoeError):
        t.update(table({0: [host(1, 3)]}))
    with pytest.raises(m.MoeError):
        t.update(table({1: [HOST - STRIDE]}))
    with pytest.raises(m.MoeError):
        m.Tier(NL, E, 1000, HOST, SLOTS)  # stride not a multiple of 256


def test_lru_matches_a_reference_model(m):
    """Random steps against a plain Python LRU with the same rules."""
    rng = np.random.default_rng(5)
    t = m.Tier(NL, E, STRIDE, HOST, SLOTS)
    resident = []  # keys, least recently used first
    for step in range(60):
        a = t.addresses()
        keys = []
        rows = {}
        for l in range(NL):
            es = rng.choice(E, size=rng.integers(1, 4), replace=False)
            rows[l] = [int(a[l, e]) for e in es]
            keys += [(l, int(e)) for e in es]
        missed = []
        for k in keys:
            if k in resident:
                resident.remove(k)
                resident.append(k)
            else:
                missed.append(k)
        promoted = 0
        for k in missed:
            if len(resident) < SLOTS:
                resident.append(k)
            elif resident[0] not in keys:
                resident.pop(0)
                resident.append(k)
            else:
                break
            promoted += 1
        assert t.update(table(rows)) == promoted
        got = sorted(k for k in [(l, e) for l in range(NL) for e in range(E)] if t.slot(*k) >= 0)
        assert got == sorted(resident), step
