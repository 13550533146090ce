"""Python binding of the C ABI in include/moe_api.h (argument marshalling only).

Every step of the path runs in libmoe_gb300.so; this module only turns torch
tensors into pointers, fills the ABI structs and checks return codes.  There
is no fallback: if the library is missing the import of `lib()` raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build
from . import synth

RESIDUAL = 1
PRENORM = 2
LOOKAHEAD = 4
TEST_WITHHOLD = 0x100

OK, EINVAL, ESHAPE, EALIGN, ECUDA, ETIMEOUT, EDEVICE, ENOSPACE = 0, -1, -2, -3, -4, -5, -6, -7
STATUS_NAMES = {0: "MOE_OK", -1: "MOE_EINVAL", -2: "MOE_ESHAPE", -3: "MOE_EALIGN", -4: "MOE_ECUDA",
                -5: "MOE_ETIMEOUT", -6: "MOE_EDEVICE", -7: "MOE_ENOSPACE"}

EXPORTS = ["moe_route", "moe_forward", "moe_forward_traced", "moe_forward_noalloc", "moe_forward_workspace",
           "moe_prefill", "moe_prefill_timed", "moe_prefill_workspace", "moe_prefill_group", "moe_last_error",
           "moe_tier_create", "moe_tier_update", "moe_tier_slot", "moe_tier_get_stats", "moe_tier_addresses",
           "moe_tier_destroy", "moe_tier_last_error"]
PREFILL_KERNELS = 10
PREFILL_KERNEL_NAMES = ["prep", "router_gemm", "topk", "group_count", "group_scan", "group_fill", "gather",
                        "gate_up_gemm", "down_gemm", "output"]
NOALLOC_MAX_WORKSPACE = 4 << 20
TRACE_CTAS, TRACE_PHASES = 1024, 16


class MoeQ(ctypes.Structure):
    _fields_ = [("w", ctypes.c_uint64), ("s", ctypes.c_uint64), ("b", ctypes.c_uint64),
                ("out", ctypes.c_uint32), ("inp", ctypes.c_uint32)]


class MoeLayer(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_uint32), ("n_experts", ctypes.c_uint32), ("top_k", ctypes.c_uint32),
                ("inter", ctypes.c_uint32), ("bits", ctypes.c_uint32), ("group", ctypes.c_uint32),
                ("flags", ctypes.c_uint32),
                ("router", ctypes.c_void_p), ("shared_gate", ctypes.c_void_p), ("shared_record", ctypes.c_void_p),
                ("sh_gate_up", MoeQ), ("sh_down", MoeQ),
                ("expert_addr", ctypes.c_void_p),
                ("gate_up", MoeQ), ("down", MoeQ),
                ("expert_bits", ctypes.c_void_p), ("gate_up_w", MoeQ * 3), ("down_w", MoeQ * 3),
                ("expert_tier", ctypes.c_void_p), ("cut_weak", ctypes.c_float),
                ("lookahead_idx", ctypes.c_void_p)]


class TierStats(ctypes.Structure):
    _fields_ = [("resident", ctypes.c_int), ("last_host_reads", ctypes.c_int), ("last_promoted", ctypes.c_int),
                ("promotions", ctypes.c_longlong), ("evictions", ctypes.c_longlong)]


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None


def lib(path: str | None = None) -> ctypes.CDLL:
    """Load libmoe_gb300.so (built by build.build()); raise if it is absent."""
    global _lib
    if _lib is None:
        path = path or _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with quantized_routed_expert_fn_gb300.build.build()")
        L = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_forward_workspace.restype = sz
        L.moe_forward_workspace.argtypes = [ctypes.POINTER(MoeLayer), i32, i32]
        L.moe_forward.restype = i32
        L.moe_forward.argtypes = [ctypes.POINTER(MoeLayer), i32, vp, i32, vp, vp, sz, vp, vp, vp, vp, vp]
        L.moe_forward_traced.restype = i32
        L.moe_forward_traced.argtypes = [ctypes.POINTER(MoeLayer), i32, vp, i32, vp, vp, sz, vp, vp, vp, vp, vp, vp]
        L.moe_forward_noalloc.restype = i32
        L.moe_forward_noalloc.argtypes = [ctypes.POINTER(MoeLayer), i32, vp, i32, vp, vp, vp, vp, vp, vp]
        L.moe_route.restype = i32
        L.moe_route.argtypes = [ctypes.POINTER(MoeLayer), vp, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp]
        L.moe_prefill_workspace.restype = sz
        L.moe_prefill_workspace.argtypes = [ctypes.POINTER(MoeLayer), i32]
        L.moe_prefill.restype = i32
        L.moe_prefill.argtypes = [ctypes.POINTER(MoeLayer), vp, i32, vp, vp, sz, vp, vp, vp]
        L.moe_prefill_timed.restype = i32
        L.moe_prefill_timed.argtypes = [ctypes.POINTER(MoeLayer), vp, i32, vp, vp, sz, vp, vp, vp, vp]
        L.moe_prefill_group.restype = i32
        L.moe_prefill_group.argtypes = [ctypes.POINTER(MoeLayer), vp, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp]
        L.moe_tier_create.restype = i32
        L.moe_tier_create.argtypes = [i32, i32, sz, vp, vp, i32, vp, vp, vp, ctypes.POINTER(vp)]
        L.moe_tier_update.restype = i32
        L.moe_tier_update.argtypes = [vp, vp, i32, vp]
        L.moe_tier_slot.restype = i32
        L.moe_tier_slot.argtypes = [vp, i32, i32]
        L.moe_tier_get_stats.restype = i32
        L.moe_tier_get_stats.argtypes = [vp, ctypes.POINTER(TierStats)]
        L.moe_tier_addresses.restype = ctypes.POINTER(ctypes.c_uint64)
        L.moe_tier_addresses.argtypes = [vp]
        L.moe_tier_destroy.restype = None
        L.moe_tier_destroy.argtypes = [vp]
        L.moe_tier_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def last_error() -> str:
    return lib().moe_last_error().decode()


def _check(code: int) -> None:
    if code != OK:
        raise MoeError(code, last_error())


def _p(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _q(q) -> MoeQ:
    return MoeQ(q.w, q.s, q.b, q.out, q.inp)


class DeviceLayers:
    """Device copies of synth.Layer weights plus the ABI structs that point at them."""

    def __init__(self, layers, device="cuda"):
        self.tensors = []  # per layer: router, records, expert addresses, shared gate, shared record
        self.keep = []
        arr = (MoeLayer * len(layers))()
        for i, L in enumerate(layers):
            if isinstance(L, synth.DeviceLayer):
                router, recs, sg, srec = L.router, L.records, L.shared_gate, L.shared_record
            else:
                router = torch.from_numpy(L.router.view(np.int16)).to(device)
                recs = torch.from_numpy(L.records).to(device)
                sg = srec = None
                if L.shared_gate is not None:
                    sg = torch.from_numpy(L.shared_gate.view(np.int16)).to(device)
                    srec = torch.from_numpy(L.shared_record).to(device)
            stride = L.layout.stride
            base = recs.data_ptr()
            eaddr = torch.arange(L.n_experts, dtype=torch.int64, device=recs.device) * stride + base
            self.tensors += [router, recs, eaddr, sg, srec]
            c = arr[i]
            c.hidden, c.n_experts, c.top_k, c.inter = L.hidden, L.n_experts, L.top_k, L.inter
            c.bits, c.group, c.flags = L.bits, 64, L.flags
            c.router = router.data_ptr()
            c.shared_gate = _p(sg)
            c.shared_record = _p(srec)
            if L.shared_layout is not None:
                c.sh_gate_up, c.sh_down = _q(L.shared_layout.gate_up), _q(L.shared_layout.down)
            c.expert_addr = eaddr.data_ptr()
            c.gate_up, c.down = _q(L.layout.gate_up), _q(L.layout.down)
            if getattr(L, "expert_bits", None) is not None:
                # mixed widths: a width per routed record, offsets per width
                eb = L.expert_bits
                eb = eb if isinstance(eb, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(eb))
                eb = eb.to(device=recs.device, dtype=torch.uint8)
                self.keep.append(eb)
                c.expert_bits = eb.data_ptr()
                for j, b in enumerate((4, 3, 2)):
                    c.gate_up_w[j], c.down_w[j] = _q(L.layouts[b].gate_up), _q(L.layouts[b].down)
        self.c = arr
        self.n = len(layers)
        self.src = layers

    def set_tier(self, layer: int, expert_addr: torch.Tensor, expert_tier: torch.Tensor | None,
                 cut_weak: float = 0.0) -> None:
        """Point layer `layer` at other record addresses (device or host
        memory) with their tiers (uint8 [E], 1 = host memory), and set its cut."""
        self.keep += [expert_addr, expert_tier]
        c = self.c[layer]
        c.expert_addr = expert_addr.data_ptr()
        c.expert_tier = None if expert_tier is None else expert_tier.data_ptr()
        c.cut_weak = cut_weak

    def set_flags(self, flags: int) -> None:
        for i in range(self.n):
            self.c[i].flags = flags


def forward_workspace(layers: DeviceLayers | ctypes.Array, nb: int, n_layers: int | None = None) -> int:
    arr = layers.c if isinstance(layers, DeviceLayers) else layers
    n = n_layers if n_layers is not None else len(arr)
    return int(lib().moe_forward_workspace(arr, n, nb))


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(nbytes + 256, dtype=torch.uint8, device=device)


def _aligned(ws: torch.Tensor) -> tuple[int, int]:
    p = ws.data_ptr()
    a = (p + 255) // 256 * 256
    return a, ws.numel() - (a - p)


def forward(layers: DeviceLayers, x: torch.Tensor, out: torch.Tensor, work: torch.Tensor, status: torch.Tensor,
            slot_tab=None, wmap=None, topk_idx=None, n_layers: int | None = None, stream=None,
            layer_offset: int = 0) -> None:
    """moe_forward over layers[layer_offset : layer_offset + n_layers]."""
    n = n_layers if n_layers is not None else layers.n - layer_offset
    arr = ctypes.cast(ctypes.byref(layers.c, layer_offset * ctypes.sizeof(MoeLayer)), ctypes.POINTER(MoeLayer))
    wp, wb = _aligned(work)
    _check(lib().moe_forward(arr, n, _p(x), x.shape[0], _p(out), wp, wb, _p(slot_tab), _p(wmap), _p(topk_idx),
                             _p(status), _stream(stream)))


def forward_traced(layers: DeviceLayers, x: torch.Tensor, out: torch.Tensor, work: torch.Tensor,
                   status: torch.Tensor, trace: torch.Tensor, slot_tab=None, wmap=None, topk_idx=None,
                   stream=None) -> None:
    """moe_forward with per-phase timestamps into trace (int64 [n_layers][1024][16])."""
    wp, wb = _aligned(work)
    _check(lib().moe_forward_traced(layers.c, layers.n, _p(x), x.shape[0], _p(out), wp, wb, _p(slot_tab), _p(wmap),
                                    _p(topk_idx), _p(status), _p(trace), _stream(stream)))


def forward_noalloc(layers: DeviceLayers, x: torch.Tensor, out: torch.Tensor, status: torch.Tensor,
                    slot_tab=None, wmap=None, topk_idx=None, stream=None) -> None:
    """moe_forward on the library's fixed scratch (no workspace, no allocation)."""
    _check(lib().moe_forward_noalloc(layers.c, layers.n, _p(x), x.shape[0], _p(out), _p(slot_tab), _p(wmap),
                                     _p(topk_idx), _p(status), _stream(stream)))


def route(layers: DeviceLayers, x: torch.Tensor, topk_idx, topk_w, slot_row, wmap_row, work, status,
          logits=None, layer: int = 0, stream=None) -> None:
    arr = ctypes.cast(ctypes.byref(layers.c, layer * ctypes.sizeof(MoeLayer)), ctypes.POINTER(MoeLayer))
    wp, wb = _aligned(work)
    _check(lib().moe_route(arr, _p(x), x.shape[0], _p(logits), _p(topk_idx), _p(topk_w), _p(slot_row),
                           _p(wmap_row), wp, wb, _p(status), _stream(stream)))


def _layer_ptr(layers: DeviceLayers, layer: int):
    return ctypes.cast(ctypes.byref(layers.c, layer * ctypes.sizeof(MoeLayer)), ctypes.POINTER(MoeLayer))


def prefill_workspace(layers: DeviceLayers, t: int, layer: int = 0) -> int:
    return int(lib().moe_prefill_workspace(_layer_ptr(layers, layer), t))


def prefill(layers: DeviceLayers, x: torch.Tensor, out: torch.Tensor, work: torch.Tensor, status: torch.Tensor,
            topk_idx=None, layer: int = 0, stream=None) -> None:
    """moe_prefill: x float32 [t][H] -> out bf16 bits (int16 tensor) [t][H]."""
    wp, wb = _aligned(work)
    _check(lib().moe_prefill(_layer_ptr(layers, layer), _p(x), x.shape[0], _p(out), wp, wb, _p(topk_idx),
                             _p(status), _stream(stream)))


def prefill_group(layers: DeviceLayers, x: torch.Tensor, topk_idx, topk_w, group_offs, group_rows, group_w,
                  work, status, layer: int = 0, stream=None) -> None:
    """moe_prefill_group: routing and the stable expert grouping of a prefill chunk."""
    wp, wb = _aligned(work)
    _check(lib().moe_prefill_group(_layer_ptr(layers, layer), _p(x), x.shape[0], _p(topk_idx), _p(topk_w),
                                   _p(group_offs), _p(group_rows), _p(group_w), wp, wb, _p(status),
                                   _stream(stream)))


def prefill_timed(layers: DeviceLayers, x: torch.Tensor, out: torch.Tensor, work: torch.Tensor,
                  status: torch.Tensor, events, topk_idx=None, layer: int = 0, stream=None) -> None:
    """moe_prefill recording events[i] (torch.cuda.Event, already recorded once so
    that it exists) before kernel i and events[PREFILL_KERNELS] after the last."""
    assert len(events) == PREFILL_KERNELS + 1
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    wp, wb = _aligned(work)
    _check(lib().moe_prefill_timed(_layer_ptr(layers, layer), _p(x), x.shape[0], _p(out), wp, wb, _p(topk_idx),
                                   _p(status), arr, _stream(stream)))


class Tier:
    """The two-tier expert store (moe_tier_*): records in pinned host memory,
    the most recently used ones cached in device slots.

    host_records: address (int) or pinned uint8 tensor [n_layers][n_experts][stride];
    slots: device uint8 tensor [n_slots][stride] or None; expert_addr /
    expert_tier: device int64 / uint8 tensors [n_layers][n_experts], or None
    for a policy-only store (no CUDA call)."""

    def __init__(self, n_layers, n_experts, stride, host_records, n_slots, slots=None, expert_addr=None,
                 expert_tier=None, stream=None):
        self.n_layers, self.n_experts, self.stride = n_layers, n_experts, stride
        self._keep = [host_records, slots, expert_addr, expert_tier]
        h = host_records if isinstance(host_records, int) else host_records.data_ptr()
        self.dry = expert_addr is None
        t = ctypes.c_void_p()
        code = lib().moe_tier_create(n_layers, n_experts, stride, h, _p(slots), n_slots, _p(expert_addr),
                                     _p(expert_tier), None if self.dry else _stream(stream), ctypes.byref(t))
        if code != OK:
            raise MoeError(code, lib().moe_tier_last_error().decode())
        self.t = t

    def update(self, slot_tab, stream=None) -> int:
        """slot_tab: host uint64 array [n_layers][64] of the step just run."""
        st = np.ascontiguousarray(slot_tab, dtype=np.uint64)
        r = lib().moe_tier_update(self.t, st.ctypes.data, st.shape[0], None if self.dry else _stream(stream))
        if r < 0:
            raise MoeError(r, lib().moe_tier_last_error().decode())
        return r

    def slot(self, layer: int, expert: int) -> int:
        return int(lib().moe_tier_slot(self.t, layer, expert))

    def stats(self) -> dict:
        s = TierStats()
        _check(lib().moe_tier_get_stats(self.t, ctypes.byref(s)))
        return {f: getattr(s, f) for f, _ in TierStats._fields_}

    def addresses(self) -> np.ndarray:
        p = lib().moe_tier_addresses(self.t)
        return np.ctypeslib.as_array(p, shape=(self.n_layers, self.n_experts)).copy()

    def close(self) -> None:
        if self.t:
            lib().moe_tier_destroy(self.t)
            self.t = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
