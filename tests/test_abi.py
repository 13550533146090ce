"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

from quantized_routed_expert_fn_gb300 import build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    build.build()
    from quantized_routed_expert_fn_gb300 import moe
    moe.lib()
    return moe


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(m):
    names = declared_functions()
    assert {"moe_route", "moe_forward", "moe_forward_workspace", "moe_last_error"} <= set(names)
    lib = m.lib()
    for n in names:
        assert hasattr(lib, n), n


def _layer(H=512, E=16, k=2, I=256, bits=4, shared=True):
    c = (np.random.default_rng(0))
    L = synth.make_layer(c, H, E, k, I, bits, shared=shared)
    return L


def _struct(m, L, **over):
    arr = (m.MoeLayer * 1)()
    c = arr[0]
    c.hidden, c.n_experts, c.top_k, c.inter, c.bits, c.group, c.flags = L.hidden, L.n_experts, L.top_k, L.inter, L.bits, 64, 0
    c.router, c.expert_addr = 0x10000, 0x20000
    if L.shared_layout is not None:
        c.shared_gate, c.shared_record = 0x30000, 0x40000
        c.sh_gate_up, c.sh_down = m._q(L.shared_layout.gate_up), m._q(L.shared_layout.down)
    c.gate_up, c.down = m._q(L.layout.gate_up), m._q(L.layout.down)
    for k, v in over.items():
        setattr(c, k, v)
    return arr


def test_workspace_size(m):
    L = _layer()
    arr = _struct(m, L)
    n = m.lib().moe_forward_workspace(arr, 1, 4)
    assert n > 0
    assert m.lib().moe_forward_workspace(arr, 1, 5) == 0


@pytest.mark.parametrize("over,code", [
    (dict(hidden=300), -2), (dict(inter=200), -2), (dict(group=32), -2), (dict(bits=5), -2),
    (dict(top_k=0), -2), (dict(flags=0x80), -1), (dict(router=0), -1), (dict(router=0x10008), -3),
    (dict(shared_gate=0), -1), (dict(cut_weak=1.5), -1), (dict(cut_weak=-0.1), -1),
])
def test_forward_rejects_bad_layers(m, over, code):
    L = _layer()
    arr = _struct(m, L, **over)
    r = m.lib().moe_forward(arr, 1, 0x1000, 1, 0x2000, 0x100000, 1 << 30, None, None, None, 0x3000, None)
    assert r == code, m.last_error()
    assert m.last_error()


def test_forward_rejects_bad_calls(m):
    L = _layer(k=16)
    arr = _struct(m, L)
    lib = m.lib()
    # k * nb must stay below the 64-entry slot table
    assert lib.moe_forward(arr, 1, 0x1000, 4, 0x200000, 0x100000, 1 << 30, None, None, None, 0x3000, None) == -2
    L = _layer()
    arr = _struct(m, L)
    assert lib.moe_forward(arr, 1, 0x1000, 0, 0x200000, 0x100000, 1 << 30, None, None, None, 0x3000, None) == -1
    assert lib.moe_forward(arr, 0, 0x1000, 1, 0x200000, 0x100000, 1 << 30, None, None, None, 0x3000, None) == -1
    # out overlapping x
    assert lib.moe_forward(arr, 1, 0x1000, 1, 0x1100, 0x100000, 1 << 30, None, None, None, 0x3000, None) == -1
    # misaligned or small workspace
    assert lib.moe_forward(arr, 1, 0x1000, 1, 0x200000, 0x100010, 1 << 30, None, None, None, 0x3000, None) == -3
    assert lib.moe_forward(arr, 1, 0x1000, 1, 0x200000, 0x100000, 16, None, None, None, 0x3000, None) == -7
    # misaligned record offset
    bad = m.MoeQ(L.layout.gate_up.w + 16, L.layout.gate_up.s, L.layout.gate_up.b, L.layout.gate_up.out,
                 L.layout.gate_up.inp)
    arr = _struct(m, L, gate_up=bad)
    assert lib.moe_forward(arr, 1, 0x1000, 1, 0x200000, 0x100000, 1 << 30, None, None, None, 0x3000, None) == -3


def test_route_requires_outputs(m):
    L = _layer()
    arr = _struct(m, L)
    r = m.lib().moe_route(arr, 0x1000, 1, None, None, 0x2000, 0x3000, 0x4000, 0x100000, 1 << 30, 0x5000, None)
    assert r == -1


@pytest.mark.parametrize("bits,inter,ok", [(4, 256, True), (3, 256, True), (2, 256, True), (2, 192, True),
                                           (3, 192, False), (5, 256, False)])
def test_prefill_workspace_by_width(m, bits, inter, ok):
    """moe_prefill_workspace sizes 4/3/2-bit layers alike and returns 0 for
    layers prefill rejects: a width outside {2, 3, 4}, or 3-bit rows that are
    not whole 16-byte pieces (inter % 128 != 0)."""
    L = _layer(I=inter, bits=bits if bits != 5 else 4)
    arr = _struct(m, L, bits=bits)
    n = m.lib().moe_prefill_workspace(arr, 4096)
    assert (n > 0) == ok, m.last_error()
    if ok:
        ref = m.lib().moe_prefill_workspace(_struct(m, _layer(I=inter)), 4096)
        assert n == ref  # the workspace does not depend on the record width


def test_prefill_rejects_bad_calls(m):
    L = _layer()
    arr = _struct(m, L)
    lib = m.lib()
    assert lib.moe_prefill_workspace(arr, 0) == 0
    assert lib.moe_prefill_workspace(arr, (1 << 20) + 1) == 0
    assert lib.moe_prefill_workspace(_struct(m, L, top_k=33), 16) == 0


def test_prefill_rejects_chunks_past_the_tma_coordinate_range(m):
    """The expert GEMMs reach a row of the grouped operands with a signed
    32-bit tensor-map coordinate: (hidden / 64) * t * (top_k + 1) must stay
    below 2^31, and a larger chunk is refused on the host."""
    H, I, E = 16384, 256, 64
    lay = synth.record_layout(H, I, 4)

    def workspace(k, t):
        arr = (m.MoeLayer * 1)()
        c = arr[0]
        c.hidden, c.n_experts, c.top_k, c.inter, c.bits, c.group, c.flags = H, E, k, I, 4, 64, 0
        c.router, c.expert_addr = 0x10000, 0x20000
        c.gate_up, c.down = m._q(lay.gate_up), m._q(lay.down)
        return m.lib().moe_prefill_workspace(arr, t)

    assert workspace(6, 1 << 20) > 0  # 256 k-panels x 7 x 2^20 rows < 2^31
    assert workspace(7, 1 << 20) == 0  # = 2^31
    assert workspace(7, (1 << 20) - 1) > 0


def _mixed_struct(m, L, n_layers=1):
    arr = (m.MoeLayer * n_layers)()
    for i in range(n_layers):
        arr[i] = _struct(m, L)[0]
        c = arr[i]
        c.expert_bits = 0x50000
        for j, b in enumerate((4, 3, 2)):
            lay = synth.record_layout(L.hidden, L.inter, b)
            c.gate_up_w[j], c.down_w[j] = m._q(lay.gate_up), m._q(lay.down)
    return arr


def _forward(m, arr, n=1):
    return m.lib().moe_forward(arr, n, 0x1000, 1, 0x200000, 0x100000, 1 << 30, None, None, None, 0x3000, None)


def test_mixed_width_layers_host_checks(m):
    """Per-record widths: the per-width offsets are checked like the uniform
    ones, every layer of a call must say the same, and prefill rejects them."""
    L = _layer()
    assert m.lib().moe_forward_workspace(_mixed_struct(m, L), 1, 4) > 0
    arr = _mixed_struct(m, L)
    q = arr[0].down_w[2]
    arr[0].down_w[2] = m.MoeQ(q.w + 16, q.s, q.b, q.out, q.inp)
    assert _forward(m, arr) == -3, m.last_error()
    arr = _mixed_struct(m, L)
    q = arr[0].gate_up_w[1]
    arr[0].gate_up_w[1] = m.MoeQ(q.w, q.s, q.b, q.out, q.inp + 64)
    assert _forward(m, arr) == -2, m.last_error()
    arr = _mixed_struct(m, L, n_layers=2)
    arr[1].expert_bits = None
    assert _forward(m, arr, 2) == -1, m.last_error()
    # the uniform offsets are not consulted when widths are per record
    arr = _mixed_struct(m, L)
    arr[0].bits = 7
    arr[0].gate_up = m.MoeQ(1, 1, 1, 1, 1)
    assert m.lib().moe_forward_workspace(arr, 1, 1) > 0, m.last_error()
    assert m.lib().moe_prefill_workspace(_mixed_struct(m, L), 16) == 0


def test_prefill_rejects_host_memory_records(m):
    """Tiers and the cut are decode features: prefill refuses a layer that uses them."""
    L = _layer()
    assert m.lib().moe_prefill_workspace(_struct(m, L, expert_tier=0x60000), 16) == 0
    assert m.lib().moe_prefill_workspace(_struct(m, L, cut_weak=0.1), 16) == 0
    assert m.lib().moe_prefill_workspace(_struct(m, L), 16) > 0
