"""Seeded synthetic inputs for the routed quantized mixture-of-experts step.

This module draws the workloads' random inputs and stores them in the record
format; it holds none of the step's arithmetic (no dequantisation, no dot
products, no routing).  Both the CUDA path's tests and the CPU oracle are fed
from here, so it is the one module the two share.

Record format (the `Q` projection of the gpu.rs source page, `struct Q`: byte
offsets `w`/`s`/`b` of codes, scales and biases inside one buffer, plus `out`
and `inp`):

* codes: uint32 words, row-major `[out][inp*bits/32]`; each row is one
  little-endian bitstream, code `i` in bits `[i*bits, i*bits+bits)`, LSB first
  (8 codes per word at 4 bits, 16 at 2 bits; 3-bit codes straddle words);
* scales and biases: bf16, row-major `[out][inp/64]`, one per 64-code group;
* a routed expert record holds `gate_up` (`out = 2*inter`, rows `0..inter-1`
  the gate, `inter..2*inter-1` the up projection, `inp = hidden`) and then
  `down` (`out = hidden`, `inp = inter`); every tensor starts on a 256-byte
  boundary.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GROUP = 64
ALIGN = 256
SLOT_STRIDE = 64
MAX_NB = 4


def _align(n: int, a: int = ALIGN) -> int:
    return (n + a - 1) // a * a


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Widen bf16 bits to the float32 values they denote."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack integer codes `[rows][n]` (each < 2**bits) into uint32 words, LSB first."""
    codes = np.asarray(codes)
    rows, n = codes.shape
    if (n * bits) % 32:
        raise ValueError("row bit length must be a multiple of 32")
    bitplanes = ((codes[..., None].astype(np.uint32) >> np.arange(bits, dtype=np.uint32)) & 1)
    stream = bitplanes.reshape(rows, n * bits).astype(np.uint8)
    packed = np.packbits(stream, axis=1, bitorder="little")
    return packed.view("<u4").reshape(rows, n * bits // 32).astype(np.uint32)


@dataclasses.dataclass(frozen=True)
class QDesc:
    """Byte offsets of one quantized projection inside its record."""
    w: int
    s: int
    b: int
    out: int
    inp: int


@dataclasses.dataclass(frozen=True)
class RecordLayout:
    bits: int
    hidden: int
    inter: int
    gate_up: QDesc
    down: QDesc
    stride: int


def q_bytes(out: int, inp: int, bits: int) -> tuple[int, int, int]:
    """(code bytes, scale bytes, bias bytes) of one projection."""
    return out * inp * bits // 8, out * (inp // GROUP) * 2, out * (inp // GROUP) * 2


def record_layout(hidden: int, inter: int, bits: int) -> RecordLayout:
    off = 0
    descs = []
    for out, inp in ((2 * inter, hidden), (hidden, inter)):
        cw, cs, cb = q_bytes(out, inp, bits)
        w = off
        off = _align(off + cw)
        s = off
        off = _align(off + cs)
        b = off
        off = _align(off + cb)
        descs.append(QDesc(w, s, b, out, inp))
    return RecordLayout(bits, hidden, inter, descs[0], descs[1], _align(off, 4096))


def _fill_q(rng, rec: np.ndarray, q: QDesc, bits: int, scale_lo: float, scale_hi: float,
            bias_noise: float, codes=None) -> None:
    n_rec = rec.shape[0]
    cw, cs, _ = q_bytes(q.out, q.inp, bits)
    if codes is None:
        # i.i.d. uniform codes packed LSB first form i.i.d. uniform bits, so
        # uniform random words are exactly such a packing.
        words = np.frombuffer(rng.bytes(n_rec * cw), dtype=np.uint32).reshape(n_rec, cw // 4)
    else:
        words = np.stack([pack_codes(c, bits).reshape(-1) for c in codes])
    rec[:, q.w:q.w + cw] = words.view(np.uint8).reshape(n_rec, cw)
    ng = q.out * (q.inp // GROUP)
    scale = rng.uniform(scale_lo, scale_hi, size=(n_rec, ng)).astype(np.float32)
    s_bits = f32_to_bf16_bits(scale)
    s_val = bf16_bits_to_f32(s_bits).reshape(n_rec, ng)
    bias = -float(2 ** (bits - 1)) * s_val
    if bias_noise:
        bias = bias + rng.normal(0.0, bias_noise, size=bias.shape).astype(np.float32)
    b_bits = f32_to_bf16_bits(bias)
    rec[:, q.s:q.s + cs] = s_bits.reshape(n_rec, ng).view(np.uint8)
    rec[:, q.b:q.b + cs] = b_bits.reshape(n_rec, ng).view(np.uint8)


def make_records(rng, n: int, layout: RecordLayout, scale_lo: float, scale_hi: float,
                 bias_noise: float) -> np.ndarray:
    """`n` records `[n][stride]` (uint8) with uniform codes and affine scale/bias."""
    rec = np.zeros((n, layout.stride), dtype=np.uint8)
    for q in (layout.gate_up, layout.down):
        _fill_q(rng, rec, q, layout.bits, scale_lo, scale_hi, bias_noise)
    return rec


def make_uniform_record(layout: RecordLayout, code: int, scale_bits: int, bias_bits: int) -> np.ndarray:
    """One record whose every code, scale and bias take the given values (hand-worked cases)."""
    rec = np.zeros((1, layout.stride), dtype=np.uint8)
    for q in (layout.gate_up, layout.down):
        cw, cs, _ = q_bytes(q.out, q.inp, layout.bits)
        words = pack_codes(np.full((q.out, q.inp), code, dtype=np.uint32), layout.bits)
        rec[0, q.w:q.w + cw] = words.reshape(-1).view(np.uint8)
        ng = q.out * (q.inp // GROUP)
        rec[0, q.s:q.s + cs] = np.full(ng, scale_bits, dtype=np.uint16).view(np.uint8)
        rec[0, q.b:q.b + cs] = np.full(ng, bias_bits, dtype=np.uint16).view(np.uint8)
    return rec


@dataclasses.dataclass
class Layer:
    """Host copy of one MoE layer's weights (all experts resident)."""
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    bits: int
    flags: int
    router: np.ndarray            # uint16 [E][H] bf16 bits
    shared_gate: np.ndarray | None  # uint16 [H] bf16 bits
    shared_record: np.ndarray | None  # uint8 [stride4] (4-bit record)
    shared_layout: RecordLayout | None
    records: np.ndarray           # uint8 [E][stride]
    layout: RecordLayout
    # mixed widths: the code width of each routed record (uint8 [E]) and the
    # record layout of each width; records stay `layout.stride` (the 4-bit
    # stride) apart, a narrower record using the front of its slot
    expert_bits: np.ndarray | None = None
    layouts: dict | None = None


# per-layer flags (same values as the C ABI)
RESIDUAL = 1
PRENORM = 2


def make_layer(rng, hidden: int, n_experts: int, top_k: int, inter: int, bits: int = 4,
               shared: bool = True, flags: int = 0, scale=(0.005, 0.02), bias_noise=1e-3,
               router_std: float = 0.05, gate_std: float = 0.05,
               shared_scale=(0.005, 0.02), shared_bias_noise=1e-3) -> Layer:
    lay = record_layout(hidden, inter, bits)
    router = f32_to_bf16_bits(rng.normal(0.0, router_std, size=(n_experts, hidden)).astype(np.float32))
    records = make_records(rng, n_experts, lay, scale[0], scale[1], bias_noise)
    sg = srec = slay = None
    if shared:
        slay = record_layout(hidden, inter, 4)
        sg = f32_to_bf16_bits(rng.normal(0.0, gate_std, size=hidden).astype(np.float32))
        srec = make_records(rng, 1, slay, shared_scale[0], shared_scale[1], shared_bias_noise)[0]
    return Layer(hidden, n_experts, top_k, inter, bits, flags, router, sg, srec, slay, records, lay)


LOWBIT_SCALE, LOWBIT_BIAS_NOISE = (0.01, 0.04), 0.0


def make_mixed_layer(rng, hidden: int, n_experts: int, top_k: int, inter: int, expert_bits,
                     shared: bool = True, flags: int = 0) -> Layer:
    """A layer whose routed records have per-expert widths (4, 3 or 2 bits):
    4-bit records drawn as in make_layer, 3- and 2-bit ones with the low-bit
    scales (and no bias noise) of the low-bit workloads."""
    expert_bits = np.ascontiguousarray(expert_bits, dtype=np.uint8)
    assert expert_bits.shape == (n_experts,) and set(expert_bits.tolist()) <= {2, 3, 4}
    layouts = {b: record_layout(hidden, inter, b) for b in (4, 3, 2)}
    base = make_layer(rng, hidden, n_experts, top_k, inter, 4, shared=shared, flags=flags)
    recs = np.zeros_like(base.records)
    for e in range(n_experts):
        b = int(expert_bits[e])
        lay = layouts[b]
        if b == 4:
            recs[e] = base.records[e]
        else:
            recs[e, :lay.stride] = make_records(rng, 1, lay, LOWBIT_SCALE[0], LOWBIT_SCALE[1], LOWBIT_BIAS_NOISE)[0]
    base.records = recs
    base.expert_bits = expert_bits
    base.layouts = layouts
    return base


def make_x(rng, nb: int, hidden: int, rho: float = 0.0) -> np.ndarray:
    """Rows `x_b = sqrt(rho)*c + sqrt(1-rho)*z_b`, each marginally N(0,1), float32."""
    z = rng.normal(0.0, 1.0, size=(nb, hidden))
    if rho:
        c = rng.normal(0.0, 1.0, size=(1, hidden))
        z = math.sqrt(rho) * c + math.sqrt(1.0 - rho) * z
    return z.astype(np.float32)


# ---------------------------------------------------------------- workloads
# The five workloads of the step, with the sizes, distributions and seeds
# that parity tests and the bench use.

CONFIGS = {
    # one layer, nb=1, no shared expert
    "c0": dict(hidden=256, n_experts=8, top_k=2, inter=128, bits=4, shared=False, n_layers=1, nb=1),
    # 48 stacked layers with residual add (and unit RMSNorm before each), decode nb=1
    "c1": dict(hidden=2048, n_experts=128, top_k=8, inter=768, bits=4, shared=True, n_layers=48, nb=1,
               flags=RESIDUAL | PRENORM),
    # speculative-verify batch nb=4, union of 20-40 experts
    "c2": dict(hidden=2048, n_experts=512, top_k=10, inter=512, bits=4, shared=True, n_layers=1, nb=4),
    # low-bit records, shape of c2
    "c3b3": dict(hidden=2048, n_experts=512, top_k=10, inter=512, bits=3, shared=True, n_layers=1, nb=4,
                 scale=(0.01, 0.04), bias_noise=0.0),
    "c3b2": dict(hidden=2048, n_experts=512, top_k=10, inter=512, bits=2, shared=True, n_layers=1, nb=4,
                 scale=(0.01, 0.04), bias_noise=0.0),
    # prefill chunk of 4096 tokens
    "c4": dict(hidden=2048, n_experts=512, top_k=10, inter=512, bits=4, shared=True, n_layers=1, nb=4096),
    # the same chunk over 3-bit routed records
    "c4b3": dict(hidden=2048, n_experts=512, top_k=10, inter=512, bits=3, shared=True, n_layers=1, nb=4096,
                 scale=(0.01, 0.04), bias_noise=0.0),
}


def make_config_layers(name: str, seed: int = 0, n_layers: int | None = None, **over) -> list[Layer]:
    cfg = dict(CONFIGS[name])
    cfg.update(over)
    nl = n_layers if n_layers is not None else cfg["n_layers"]
    rng = np.random.default_rng(seed)
    layers = []
    for _ in range(nl):
        layers.append(make_layer(rng, cfg["hidden"], cfg["n_experts"], cfg["top_k"], cfg["inter"],
                                 cfg["bits"], cfg["shared"], cfg.get("flags", 0),
                                 scale=cfg.get("scale", (0.005, 0.02)),
                                 bias_noise=cfg.get("bias_noise", 1e-3)))
    return layers


def zipf_router_bits(rng, n_experts: int, hidden: int, s: float = 1.1, noise_std: float = 0.028) -> np.ndarray:
    """Prefill popularity: channel 0 of x is held at 1 and router column 0 carries
    `-s*ln(rank)` for a seeded permutation of expert ranks, the rest N(0, noise_std);
    top-k then draws experts roughly as Zipf(s) without replacement.  bf16 bits [E][H]."""
    rank = rng.permutation(n_experts) + 1
    r = rng.normal(0.0, noise_std, size=(n_experts, hidden)).astype(np.float32)
    r[:, 0] = (-s * np.log(rank)).astype(np.float32)
    return f32_to_bf16_bits(r)


def zipf_router(rng, layer: Layer, s: float = 1.1, noise_std: float = 0.028) -> None:
    layer.router = zipf_router_bits(rng, layer.n_experts, layer.hidden, s, noise_std)


def make_prefill_x(rng, t: int, hidden: int) -> np.ndarray:
    x = rng.normal(0.0, 1.0, size=(t, hidden)).astype(np.float32)
    x[:, 0] = 1.0
    return x


# ------------------------------------------------------------- device-side draws
# Same distributions as above, drawn with torch directly on the GPU (used where
# the host draw would take minutes, e.g. the 48-layer stack's 16 GB of records).

@dataclasses.dataclass
class DeviceLayer:
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    bits: int
    flags: int
    router: "object"          # torch.int16 [E][H] (bf16 bits)
    shared_gate: "object"     # torch.int16 [H] or None
    shared_record: "object"   # torch.uint8 [stride4] or None
    shared_layout: RecordLayout | None
    records: "object"         # torch.uint8 [E][stride]
    layout: RecordLayout
    expert_bits: "object" = None  # mixed widths: numpy uint8 [E]
    layouts: dict | None = None


def _dev_fill_q(torch, gen, rec, q: QDesc, bits: int, scale_lo: float, scale_hi: float, bias_noise: float):
    n = rec.shape[0]
    cw, cs, _ = q_bytes(q.out, q.inp, bits)
    words = torch.randint(-2**31, 2**31 - 1, (n, cw // 4), dtype=torch.int32, device=rec.device, generator=gen)
    rec[:, q.w:q.w + cw] = words.view(torch.uint8)
    ng = q.out * (q.inp // GROUP)
    s = (torch.rand((n, ng), device=rec.device, generator=gen) * (scale_hi - scale_lo) + scale_lo).to(torch.bfloat16)
    b = -float(2 ** (bits - 1)) * s.float()
    if bias_noise:
        b = b + torch.randn((n, ng), device=rec.device, generator=gen) * bias_noise
    rec[:, q.s:q.s + cs] = s.view(torch.int16).view(torch.uint8)
    rec[:, q.b:q.b + cs] = b.to(torch.bfloat16).view(torch.int16).view(torch.uint8)


def make_device_mixed_layer(name: str, expert_bits, seed: int = 0, device="cuda") -> DeviceLayer:
    """One layer of workload `name` whose routed records have the given
    per-expert widths (4, 3 or 2; records stay the 4-bit stride apart), the
    3- and 2-bit ones drawn with the low-bit scales, on the GPU."""
    import torch
    layer = make_device_layers(name, seed=seed, device=device, n_layers=1)[0]
    eb = np.ascontiguousarray(expert_bits, dtype=np.uint8)
    layouts = {b: record_layout(layer.hidden, layer.inter, b) for b in (4, 3, 2)}
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 77)
    for b in (3, 2):
        idx = torch.from_numpy(np.nonzero(eb == b)[0]).to(device)
        if idx.numel() == 0:
            continue
        sub = torch.zeros((idx.numel(), layer.layout.stride), dtype=torch.uint8, device=device)
        for q in (layouts[b].gate_up, layouts[b].down):
            _dev_fill_q(torch, gen, sub, q, b, LOWBIT_SCALE[0], LOWBIT_SCALE[1], LOWBIT_BIAS_NOISE)
        layer.records[idx] = sub
    layer.expert_bits, layer.layouts = eb, layouts
    return layer


def make_device_layers(name: str, seed: int = 0, device="cuda", n_layers: int | None = None, **over):
    import torch
    cfg = dict(CONFIGS[name])
    cfg.update(over)
    nl = n_layers if n_layers is not None else cfg["n_layers"]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    H, E, k, I, bits = cfg["hidden"], cfg["n_experts"], cfg["top_k"], cfg["inter"], cfg["bits"]
    scale = cfg.get("scale", (0.005, 0.02))
    noise = cfg.get("bias_noise", 1e-3)
    lay = record_layout(H, I, bits)
    out = []
    for _ in range(nl):
        router = (torch.randn((E, H), device=device, generator=gen) * 0.05).to(torch.bfloat16).view(torch.int16)
        recs = torch.zeros((E, lay.stride), dtype=torch.uint8, device=device)
        for q in (lay.gate_up, lay.down):
            _dev_fill_q(torch, gen, recs, q, bits, scale[0], scale[1], noise)
        sg = srec = slay = None
        if cfg["shared"]:
            slay = record_layout(H, I, 4)
            sg = (torch.randn(H, device=device, generator=gen) * 0.05).to(torch.bfloat16).view(torch.int16)
            srec = torch.zeros((1, slay.stride), dtype=torch.uint8, device=device)
            for q in (slay.gate_up, slay.down):
                _dev_fill_q(torch, gen, srec, q, 4, 0.005, 0.02, 1e-3)
            srec = srec[0]
        out.append(DeviceLayer(H, E, k, I, bits, cfg.get("flags", 0), router, sg, srec, slay, recs, lay))
    return out
