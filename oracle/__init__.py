"""Python face of the oracle (oracle.c): build it with gcc and call it via ctypes.

Test infrastructure only: the tests, the smoke check and the bench's CPU
baseline use it; the product path never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

RESIDUAL = 1
PRENORM = 2


class OQ(ctypes.Structure):
    _fields_ = [("w", ctypes.c_uint64), ("s", ctypes.c_uint64), ("b", ctypes.c_uint64),
                ("out", ctypes.c_uint32), ("inp", ctypes.c_uint32)]


class OLayer(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("bits", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("router", ctypes.c_void_p), ("shared_gate", ctypes.c_void_p),
                ("shared_record", ctypes.c_void_p), ("sh_gate_up", OQ), ("sh_down", OQ),
                ("experts", ctypes.c_void_p), ("stride", ctypes.c_uint64),
                ("gate_up", OQ), ("down", OQ),
                ("expert_bits", ctypes.c_void_p), ("gate_up_w", OQ * 3), ("down_w", OQ * 3),
                ("expert_tier", ctypes.c_void_p), ("cut_w", ctypes.c_double)]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (OpenMP when the compiler has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:5] + ["-fopenmp"] + base[5:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        d, i32, p = ctypes.c_double, ctypes.c_int, ctypes.c_void_p
        _lib.oracle_bf16.restype = d
        _lib.oracle_bf16.argtypes = [ctypes.c_uint16]
        _lib.oracle_code_at.restype = ctypes.c_uint32
        _lib.oracle_code_at.argtypes = [p, ctypes.c_int64, i32]
        _lib.oracle_dequant.argtypes = [p, ctypes.POINTER(OQ), i32, p]
        _lib.oracle_topk_softmax.argtypes = [p, i32, i32, p, p]
        _lib.oracle_union.restype = i32
        _lib.oracle_union.argtypes = [p, i32, p]
        _lib.oracle_expert.argtypes = [ctypes.POINTER(OLayer), i32, p, p]
        _lib.oracle_shared_expert.argtypes = [ctypes.POINTER(OLayer), p, p]
        _lib.oracle_moe_layer.restype = i32
        _lib.oracle_moe_layer.argtypes = [ctypes.POINTER(OLayer), i32, p, p, p, p, p, p, p, p, p]
        _lib.oracle_route.restype = i32
        _lib.oracle_route.argtypes = [ctypes.POINTER(OLayer), i32, p, p, p, p, p]
        _lib.oracle_moe_forward.argtypes = [ctypes.POINTER(OLayer), i32, i32, p, p, p, p]
        _lib.oracle_prefill_rows.argtypes = [ctypes.POINTER(OLayer), p, p, i32, i32, p, p, p, p]
        _lib.oracle_route_rows.argtypes = [ctypes.POINTER(OLayer), p, i32, p, p, p, p]
        _lib.oracle_group.restype = i32
        _lib.oracle_group.argtypes = [i32, i32, i32, p, p, p, p, p, p]
        _lib.oracle_threads.restype = i32
        _lib.oracle_set_parallel_rows.argtypes = [i32]
        _lib.oracle_cut.restype = i32
        _lib.oracle_cut.argtypes = [ctypes.POINTER(OLayer), i32, p, p, p]
        _lib.oracle_round_bf16.restype = d
        _lib.oracle_round_bf16.argtypes = [d]
        _lib.oracle_expert_mirror.argtypes = [p, ctypes.POINTER(OQ), ctypes.POINTER(OQ), i32, i32, p, d, p, p]
    return _lib


def _ptr(a: np.ndarray | None) -> int | None:
    return None if a is None else a.ctypes.data


def _oq(q) -> OQ:
    return OQ(q.w, q.s, q.b, q.out, q.inp)


class Layer:
    """Oracle view of a synth.Layer (keeps the numpy buffers alive)."""

    def __init__(self, layer):
        self.src = layer
        self._keep = [layer.router, layer.records, layer.shared_gate, layer.shared_record]
        sl = layer.shared_layout
        self.c = OLayer(layer.hidden, layer.n_experts, layer.top_k, layer.inter, layer.bits, layer.flags,
                        _ptr(layer.router), _ptr(layer.shared_gate), _ptr(layer.shared_record),
                        _oq(sl.gate_up) if sl else OQ(), _oq(sl.down) if sl else OQ(),
                        _ptr(layer.records), layer.layout.stride,
                        _oq(layer.layout.gate_up), _oq(layer.layout.down))
        if getattr(layer, "expert_tier", None) is not None:
            # two tiers: host-memory experts below cut_w in every row are cut
            self._keep.append(layer.expert_tier)
            self.c.expert_tier = _ptr(layer.expert_tier)
            self.c.cut_w = float(getattr(layer, "cut_w", 0.0))
        if getattr(layer, "expert_bits", None) is not None:
            # mixed widths: each routed record at its own width, the
            # projections' offsets per width (index 4 - width)
            self._keep.append(layer.expert_bits)
            self.c.expert_bits = _ptr(layer.expert_bits)
            for i, b in enumerate((4, 3, 2)):
                self.c.gate_up_w[i] = _oq(layer.layouts[b].gate_up)
                self.c.down_w[i] = _oq(layer.layouts[b].down)


def code_at(words: np.ndarray, i: int, bits: int) -> int:
    words = np.ascontiguousarray(words, dtype=np.uint32)
    return int(lib().oracle_code_at(_ptr(words), i, bits))


def bf16(bits_value: int) -> float:
    return float(lib().oracle_bf16(bits_value))


def dequant(record: np.ndarray, q, bits: int) -> np.ndarray:
    record = np.ascontiguousarray(record, dtype=np.uint8)
    W = np.empty((q.out, q.inp), dtype=np.float64)
    lib().oracle_dequant(_ptr(record), ctypes.byref(_oq(q)), bits, _ptr(W))
    return W


def topk_softmax(logits: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    idx = np.empty(k, dtype=np.int32)
    w = np.empty(k, dtype=np.float64)
    lib().oracle_topk_softmax(_ptr(logits), logits.shape[0], k, _ptr(idx), _ptr(w))
    return idx, w


def union(ids: np.ndarray) -> np.ndarray:
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    u = np.empty(ids.shape[0], dtype=np.int32)
    n = lib().oracle_union(_ptr(ids), ids.shape[0], _ptr(u))
    return u[:n].copy()


def expert(layer: Layer, e: int, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(layer.src.hidden, dtype=np.float64)
    lib().oracle_expert(ctypes.byref(layer.c), e, _ptr(x), _ptr(y))
    return y


def shared_expert(layer: Layer, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(layer.src.hidden, dtype=np.float64)
    lib().oracle_shared_expert(ctypes.byref(layer.c), _ptr(x), _ptr(y))
    return y


def moe_layer(layer: Layer, x: np.ndarray) -> dict:
    """One layer over nb rows; returns out, moe, logits, idx, w, gamma, union, wmap."""
    src = layer.src
    x = np.ascontiguousarray(x, dtype=np.float64)
    nb = x.shape[0]
    H, E, k = src.hidden, src.n_experts, src.top_k
    r = dict(out=np.empty((nb, H)), moe=np.empty((nb, H)), logits=np.empty((nb, E)),
             idx=np.empty((nb, k), dtype=np.int32), w=np.empty((nb, k)), gamma=np.empty(nb),
             union=np.empty(64, dtype=np.int32), wmap=np.empty((4, 64)))
    U = lib().oracle_moe_layer(ctypes.byref(layer.c), nb, _ptr(x), _ptr(r["out"]), _ptr(r["moe"]),
                               _ptr(r["logits"]), _ptr(r["idx"]), _ptr(r["w"]), _ptr(r["gamma"]),
                               _ptr(r["union"]), _ptr(r["wmap"]))
    r["union"] = r["union"][:U].copy()
    return r


def cut(layer: Layer, idx: np.ndarray, w: np.ndarray) -> np.ndarray:
    """The deadline cut of one call's routing: bool [E], True for each
    host-memory expert below the layer's cut_w in every row."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    out = np.zeros(layer.src.n_experts, dtype=np.uint8)
    lib().oracle_cut(ctypes.byref(layer.c), idx.shape[0], _ptr(idx), _ptr(w), _ptr(out))
    return out.astype(bool)


def route(layer: Layer, x: np.ndarray) -> dict:
    """Routing alone: logits, idx, w, union."""
    src = layer.src
    x = np.ascontiguousarray(x, dtype=np.float64)
    nb = x.shape[0]
    r = dict(logits=np.empty((nb, src.n_experts)), idx=np.empty((nb, src.top_k), dtype=np.int32),
             w=np.empty((nb, src.top_k)), union=np.empty(256, dtype=np.int32))
    U = lib().oracle_route(ctypes.byref(layer.c), nb, _ptr(x), _ptr(r["logits"]), _ptr(r["idx"]), _ptr(r["w"]),
                           _ptr(r["union"]))
    r["union"] = r["union"][:U].copy()
    return r


def moe_forward(layers: list[Layer], x: np.ndarray) -> dict:
    """Stacked layers; returns out [nb][H], inputs [L][nb][H], idx [L][nb][k]."""
    arr = (OLayer * len(layers))(*[l.c for l in layers])
    x = np.ascontiguousarray(x, dtype=np.float64)
    nb, H = x.shape
    k = layers[0].src.top_k
    out = np.empty((nb, H))
    inputs = np.empty((len(layers), nb, H))
    idx = np.empty((len(layers), nb, k), dtype=np.int32)
    lib().oracle_moe_forward(arr, len(layers), nb, _ptr(x), _ptr(out), _ptr(inputs), _ptr(idx))
    return dict(out=out, inputs=inputs, idx=idx)


def prefill_rows(layer: Layer, x: np.ndarray, rows, mirror: bool) -> dict:
    """Listed rows of a prefill chunk: out, idx, w; in mirror mode also
    `allow`, the one-flip allowance of the h rounding (a test tolerance term)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.shape[0]
    H, k = layer.src.hidden, layer.src.top_k
    out = np.empty((n, H))
    idx = np.empty((n, k), dtype=np.int32)
    w = np.empty((n, k))
    allow = np.zeros((n, H)) if mirror else None
    lib().oracle_prefill_rows(ctypes.byref(layer.c), _ptr(x), _ptr(rows), n, int(mirror),
                              _ptr(out), _ptr(idx), _ptr(w), _ptr(allow))
    return dict(out=out, idx=idx, w=w, allow=allow)


def route_rows(layer: Layer, x: np.ndarray) -> dict:
    """Routing of every row of a prefill chunk: logits, idx, w, gamma (None without a shared expert)."""
    src = layer.src
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.shape[0]
    r = dict(logits=np.empty((n, src.n_experts)), idx=np.empty((n, src.top_k), dtype=np.int32),
             w=np.empty((n, src.top_k)), gamma=np.empty(n) if src.shared_gate is not None else None)
    lib().oracle_route_rows(ctypes.byref(layer.c), _ptr(x), n, _ptr(r["logits"]), _ptr(r["idx"]), _ptr(r["w"]),
                            _ptr(r["gamma"]))
    return r


def group(n_experts: int, idx: np.ndarray, w: np.ndarray, gamma: np.ndarray | None) -> dict:
    """Rows grouped by expert (then the shared group): offs [G+1], rows, wts."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    n, k = idx.shape
    G = n_experts + (1 if gamma is not None else 0)
    ent = n * k + (n if gamma is not None else 0)
    offs = np.empty(G + 1, dtype=np.int32)
    rows = np.empty(ent, dtype=np.int32)
    wts = np.empty(ent)
    g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float64)
    lib().oracle_group(n_experts, k, n, _ptr(idx), _ptr(w), _ptr(g), _ptr(offs), _ptr(rows), _ptr(wts))
    return dict(offs=offs, rows=rows, wts=wts)


def round_bf16(v: float) -> float:
    """The oracle's bf16 rounding (nearest, ties to even) of one value."""
    return float(lib().oracle_round_bf16(float(v)))


def expert_mirror(record: np.ndarray, layout, x: np.ndarray, weight: float) -> dict:
    """One expert record on one row in bf16-mirror mode: y and the one-flip
    allowance of the h rounding (a test tolerance term)."""
    record = np.ascontiguousarray(record, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(layout.hidden)
    allow = np.zeros(layout.hidden)
    lib().oracle_expert_mirror(_ptr(record), ctypes.byref(_oq(layout.gate_up)), ctypes.byref(_oq(layout.down)),
                               layout.bits, layout.inter, _ptr(x), float(weight), _ptr(y), _ptr(allow))
    return dict(y=y, allow=allow)


def threads() -> int:
    return int(lib().oracle_threads())


def set_parallel_rows(on: bool) -> None:
    """Spread the decode matvecs' output rows over host threads (timing only;
    every output is computed the same way either way)."""
    lib().oracle_set_parallel_rows(1 if on else 0)
