"""Throughput of the routed quantized MoE step on GB300.

Workload (default): 48 stacked MoE layers, decode nb=1 -- hidden 2048, 128
experts, top-8, expert width 768, 4-bit g64 records, shared expert of width
768 with a sigmoid gate, unit RMSNorm before each layer and a residual add.
One step = one moe_forward call over all 48 layers (one persistent kernel).
Metric: MoE-layer rows per second = nb * layers / step time; the HBM roofline
fraction of the kernel is reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload c1|c2|c3b3|c3b2|c4|c4b3] [--nb NB]

--workload c4 times the prefill chunk instead (moe_prefill, 10 kernels per
step; the roofline is the tensor-pipe one of its largest GEMM).

Under torchrun each rank runs an independent replica on its own GPU (the path
has no exchange step); value = rows of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    "c1": "48 stacked MoE layers, nb=1 decode: hidden 2048, 128 experts, top-8, inter 768, shared expert "
          "(inter 768, sigmoid gate), 4-bit g64 records, RMSNorm + residual",
    "c2": "one MoE layer, verify batch nb=4: hidden 2048, 512 experts, top-10, inter 512, shared expert, 4-bit g64",
    "c3b3": "one MoE layer, nb=4: hidden 2048, 512 experts, top-10, inter 512, 3-bit routed records",
    "c3b2": "one MoE layer, nb=4: hidden 2048, 512 experts, top-10, inter 512, 2-bit routed records",
    "c4": "prefill chunk of 4096 rows through one MoE layer: hidden 2048, 512 experts, top-10, inter 512, "
          "shared expert, 4-bit g64 records, Zipf(1.1) expert popularity; bf16 tensor-core GEMMs, bf16 out",
    "c4b3": "prefill chunk of 4096 rows through one MoE layer: hidden 2048, 512 experts, top-10, inter 512, "
            "shared expert (4-bit), 3-bit g64 routed records, Zipf(1.1) expert popularity; bf16 tensor-core "
            "GEMMs, bf16 out",
}
METRIC = "MoE-layer rows/sec and achieved HBM GB/s (% of roofline) at nb=1/4 on 1 GB300"


# DRAM traffic per launch of the dominant kernel, from one ncu capture each
# (the decode and prefill capture summaries under profiles/).  Reported only while the
# kernel's sources hash to the value they had when the counters were taken.
NCU_TRAFFIC = {
    "c1": dict(bytes=1209.7e6, sources=["decode.cu", "decode.cuh", "codec.cuh", "common.cuh"],
               sha="52d8d7ec859df41e"),
    "c4": dict(bytes=640.6e6, sources=["prefill.cu", "prefill.cuh", "tc05.cuh", "common.cuh"],
               sha="a30e93d7d5107b13"),
}


def ncu_traffic(workload):
    import hashlib
    t = NCU_TRAFFIC.get(workload)
    if t is None:
        return None
    m = hashlib.sha256()
    for f in t["sources"]:
        with open(os.path.join(ROOT, "quantized_routed_expert_fn_gb300", "csrc", f), "rb") as fh:
            m.update(fh.read())
    return t["bytes"] if m.hexdigest()[:16] == t["sha"] else None


def load_peaks(kind="hbm"):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs" if kind == "hbm" else "bf16_tflops"]), "measured"
    return (6800.0 if kind == "hbm" else 1900.0), "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_over_ranks(values, world: int, device="cpu"):
    """Max of each timing over the ranks: the slowest replica sets the job time."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as td
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_rows_per_s(rows_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank's rows over the (max) step time."""
    return rows_per_rank * world / (ms * 1e-3)


def layer_bytes(L, union_size: int, nb: int, widths=None) -> int:
    """Algorithmic bytes of one layer: router + shared gate + union records +
    shared record + layer input and output.  widths: the code width of each
    record read (mixed-width layers), else union_size records of L's width."""
    b = L.n_experts * L.hidden * 2
    if widths is None:
        b += union_size * record_bytes(L.layout)
    else:
        b += sum(record_bytes(L.layouts[int(w)]) for w in widths)
    if L.shared_layout is not None:
        b += L.hidden * 2 + record_bytes(L.shared_layout)
    b += 2 * nb * L.hidden * 4
    return b


def record_bytes(lay) -> int:
    from quantized_routed_expert_fn_gb300.synth import q_bytes
    tot = 0
    for q in (lay.gate_up, lay.down):
        tot += sum(q_bytes(q.out, q.inp, lay.bits))
    return tot


def l2_bytes(device) -> int:
    import torch
    return int(torch.cuda.get_device_properties(device).L2_cache_size)


def decode_inputs(base, nb: int, n_views: int, seed: int) -> list:
    """n_views inputs [nb][H] whose top-k sets are pairwise disjoint over the
    views and the rows: row b of view i is the normalised sum of the router
    rows of k experts drawn without replacement (plus noise), so those k
    experts lead its logits by a wide margin.  Returns float32 arrays."""
    import torch
    R = base.router.view(torch.bfloat16).float().cpu().numpy().astype(np.float64)
    E, H = R.shape
    k = base.top_k
    rng = np.random.default_rng(seed)
    perm = rng.permutation(E)
    xs = []
    for i in range(n_views):
        S = perm[(i * nb * k) % E:][: nb * k]
        if len(S) < nb * k:  # wrap around the permutation
            S = np.concatenate([S, perm[: nb * k - len(S)]])
        x = R[S.reshape(nb, k)].sum(axis=1) + rng.normal(0.0, 0.05, (nb, H))
        x /= np.sqrt((x * x).mean(axis=1, keepdims=True))
        xs.append(x.astype(np.float32))
    return xs


def view_bytes(dl, slots, nb) -> int:
    """Algorithmic bytes of one call over the layers of dl, from its slot
    tables: the records it listed (cut and absent ones are not read), at
    their widths."""
    tot = 0
    for l, L in enumerate(dl.src):
        row = [int(a) for a in slots[l][:62]]
        listed = row.index(0) if 0 in row else 62
        widths = None
        if getattr(L, "expert_bits", None) is not None:
            base, stride = L.records.data_ptr(), L.layout.stride
            widths = [L.expert_bits[(a - base) // stride] for a in row[:listed]]
        tot += layer_bytes(L, listed, nb, widths)
    return tot


def decode_setup(name, nb, device, seed, n_layers=None, mixed=False):
    """Device layers and inputs of a decode workload.

    The 48-layer stack reads every layer's union once per step (about 1.2 GB,
    several times L2).  A one-layer workload would re-read the same records
    every step, so it rotates views: each view has its own router,
    shared-gate and shared-record copies over a common routed-record pool (a
    second pool once one cannot hold enough disjoint unions), and its own
    input whose union is disjoint from every other view's.  The number of
    views is the smallest that makes one cycle touch at least 4x the L2 size
    queried at run time, so no record, router or shared record is read again
    before at least that many other bytes."""
    import dataclasses
    import torch
    from quantized_routed_expert_fn_gb300 import moe, synth
    cfg = synth.CONFIGS[name]
    E = cfg["n_experts"]

    def mixed_widths(s):
        eb = np.array([4, 3, 2] * (E // 3 + 1), dtype=np.uint8)[:E]
        np.random.default_rng(s).shuffle(eb)
        return eb

    if mixed:
        layers = [synth.make_device_mixed_layer(name, mixed_widths(seed), seed=seed, device=device)]
    else:
        layers = synth.make_device_layers(name, seed=seed, device=device, n_layers=n_layers or None)
    if len(layers) > 1:
        gen = torch.Generator(device="cpu").manual_seed(100 + seed)
        x = torch.randn((nb, cfg["hidden"]), generator=gen, dtype=torch.float32)
        if nb > 1:  # correlated rows
            c = torch.randn((1, cfg["hidden"]), generator=gen)
            x = (0.55 ** 0.5) * c + (0.45 ** 0.5) * x
        return dict(views=[moe.DeviceLayers(layers, device=device)], xs=[x], layers=layers,
                    rotation=None)
    base = layers[0]
    L2 = l2_bytes(device)
    U = nb * base.top_k
    per_view = layer_bytes(base, U, nb)
    n_views = max(2, -(-4 * L2 // per_view))
    per_pool = base.n_experts // U
    pools = [base]
    while len(pools) * per_pool < n_views:
        s2 = seed + 1000 * len(pools)
        pools.append(synth.make_device_mixed_layer(name, mixed_widths(s2), seed=s2, device=device) if mixed
                     else synth.make_device_layers(name, seed=s2, device=device, n_layers=1)[0])
    views, xs = [], []
    for i in range(n_views):
        pool = pools[i // per_pool]
        v = dataclasses.replace(
            pool, router=pool.router.clone(),
            shared_gate=None if pool.shared_gate is None else pool.shared_gate.clone(),
            shared_record=None if pool.shared_record is None else pool.shared_record.clone())
        views.append(v)
    for pi, pool in enumerate(pools):
        n_here = min(per_pool, n_views - pi * per_pool)
        xs += [torch.from_numpy(x) for x in decode_inputs(pool, nb, n_here, seed=11 + seed + pi)]
    return dict(views=[moe.DeviceLayers([v], device=device) for v in views], xs=xs, layers=views, pools=pools,
                rotation=dict(views=n_views, pools=len(pools), l2_bytes=L2))


def time_decode(setup, nb, steps, warmup, rank, world, device, e2e=True):
    """Device-timed and end-to-end moe_forward over the setup's views in turn."""
    import torch
    from quantized_routed_expert_fn_gb300 import moe
    views, xs_host = setup["views"], setup["xs"]
    nv, nl = len(views), views[0].n
    H = xs_host[0].shape[1]
    xs = [x.to(device) for x in xs_host]
    out = torch.empty((nb, H), dtype=torch.float32, device=device)
    ws = moe.alloc_workspace(moe.forward_workspace(views[0], nb), device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    slot = torch.zeros((nl, 64), dtype=torch.int64, device=device)
    wmap = torch.zeros((nl, 4, 64), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    # every view once: its union sizes, record addresses and bytes read
    unions, addrs, bytes_per_view, kept = [], [], [], []
    for i in range(nv):
        moe.forward(views[i], xs[i], out, ws, status, slot, wmap, stream=stream)
        torch.cuda.synchronize()
        if status.item() != 0:
            raise RuntimeError(f"device status {moe.STATUS_NAMES.get(status.item())}")
        st = slot.cpu().numpy().astype(np.int64)
        u = [int(v) for v in st[:, 63].tolist()]
        unions.append(u)
        rows = [[int(a) for a in st[l, :62]] for l in range(nl)]
        listed = [r.index(0) if 0 in r else 62 for r in rows]
        kept.append(sum(listed))
        addrs.append(set(a for l in range(nl) for a in rows[l][: listed[l]]))
        bytes_per_view.append(view_bytes(views[i], st, nb))
    for s in range(max(warmup, 3)):
        moe.forward(views[s % nv], xs[s % nv], out, ws, status, slot, wmap, stream=stream)
    torch.cuda.synchronize()
    bytes_per_step = sum(bytes_per_view[s % nv] for s in range(steps)) / steps

    dist = world > 1
    if dist:
        import torch.distributed as td
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        td.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for s in range(steps):
        moe.forward(views[s % nv], xs[s % nv], out, ws, status, slot, wmap, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    if dist:
        td.barrier()
    ms = ev0.elapsed_time(ev1) / steps
    clocks = sampler.stop() if sampler else None
    if status.item() != 0:
        raise RuntimeError(f"device status {moe.STATUS_NAMES.get(status.item())}")

    e2e_ms = None
    if e2e:
        # end to end through the same call with host buffers: H2D of x, D2H of out
        x_pin = [x.pin_memory() for x in xs_host]
        o_pin = torch.empty((nb, H), dtype=torch.float32).pin_memory()
        xd = torch.empty((nb, H), dtype=torch.float32, device=device)

        def e2e_step(s):
            xd.copy_(x_pin[s % nv], non_blocking=True)
            moe.forward(views[s % nv], xd, out, ws, status, slot, wmap, stream=stream)
            o_pin.copy_(out, non_blocking=True)

        for s in range(3):
            e2e_step(s)
        torch.cuda.synchronize()
        if dist:
            td.barrier()
        t0 = time.perf_counter()
        for s in range(steps):
            e2e_step(s)
        torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / steps
        if dist:
            td.barrier()
        ms, e2e_ms = reduce_over_ranks([ms, e2e_ms], world, device)
    peak, peak_kind = load_peaks()
    achieved = bytes_per_step / (ms * 1e-3) / 1e9
    rot = setup["rotation"]
    if rot is None:
        L2 = l2_bytes(device)
        l2 = (f"inputs larger than L2: each step reads every layer's union once, {bytes_per_step / 1e6:.0f} MB "
              f"= {bytes_per_step / L2:.1f}x the {L2 / 1e6:.0f} MB L2 (queried at run time)")
    else:
        distinct = len(set().union(*addrs)) == sum(len(a) for a in addrs)
        cycle = sum(bytes_per_view)
        l2 = (f"{nv} rotated views (own router, shared gate and shared record copies over "
              f"{rot['pools']} routed-record pool(s)), inputs built for "
              f"{'pairwise-disjoint' if distinct else 'overlapping'} unions: one cycle reads "
              f"{cycle / 1e6:.0f} MB = {cycle / rot['l2_bytes']:.1f}x the {rot['l2_bytes'] / 1e6:.0f} MB L2 "
              f"(queried at run time) before any byte is read again")
    return dict(ms=ms, e2e_ms=e2e_ms, nb=nb, nl=nl, bytes=bytes_per_step, achieved=achieved, peak=peak,
                peak_kind=peak_kind, clocks=clocks, unions=sorted(set(u for uu in unions for u in uu)), l2=l2,
                kept_per_step=sum(kept[s % nv] for s in range(steps)) / steps,
                union_per_step=sum(sum(unions[s % nv]) for s in range(steps)) / steps)


def run_ours(args, rank, world, device):
    import torch
    from quantized_routed_expert_fn_gb300 import build, moe, synth

    build.build()
    moe.lib()
    torch.cuda.set_device(device)
    cfg = synth.CONFIGS[args.workload]
    nb = args.nb or cfg["nb"]
    setup = decode_setup(args.workload, nb, device, seed=1 + rank, n_layers=args.layers or None)
    return time_decode(setup, nb, args.steps, args.warmup, rank, world, device)


def c2c_copy_gbs(device, nbytes=1 << 30, reps=5) -> float:
    """Host -> device copy bandwidth from pinned memory (best of reps): the
    denominator of the host-memory reads' link fraction."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=device)
    best = 0.0
    for _ in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del h, d
    return best


def decode_line(name, nb, r, extra=None):
    line = {"workload": WORKLOADS[name].replace("nb=4", f"nb={nb}"), "ms_per_step": r["ms"],
            "rows_per_s": nb * r["nl"] / (r["ms"] * 1e-3), "union_sizes": r["unions"],
            "roofline": {"bound": "hbm", "achieved": r["achieved"], "peak": r["peak"], "unit": "GB/s",
                         "frac": r["achieved"] / r["peak"], "peak_source": r["peak_kind"],
                         "algorithmic_bytes_per_launch": r["bytes"]},
            "l2": r["l2"], "clocks": r["clocks"]}
    line.update(extra or {})
    return line


def host_tier_extra(device, nb, cut_weak, c2c):
    """The verify batch with every routed record in pinned host memory (a
    two-tier store with no device slots): the kernel reads the union over
    NVLink-C2C.  With cut_weak, host experts below it in every row are cut."""
    import torch
    from quantized_routed_expert_fn_gb300 import moe
    setup = decode_setup("c2", nb, device, seed=1)
    pool = setup["pools"][0]
    E, stride = pool.n_experts, pool.layout.stride
    host = torch.empty((1, E, stride), dtype=torch.uint8).pin_memory()
    host[0].copy_(pool.records)
    addr = torch.zeros((1, E), dtype=torch.int64, device=device)
    tier = torch.zeros((1, E), dtype=torch.uint8, device=device)
    store = moe.Tier(1, E, stride, host, 0, None, addr, tier)
    for v in setup["views"]:
        v.set_tier(0, addr[0], tier[0], cut_weak)
    torch.cuda.synchronize()
    r = time_decode(setup, nb, 200, 5, 0, 1, device, e2e=False)
    rec = record_bytes(pool.layout)
    host_bytes = r["kept_per_step"] * rec
    link = host_bytes / (r["ms"] * 1e-3) / 1e9
    extra = {"host_memory": {"records_read_from_host_per_step": r["kept_per_step"],
                             "union_per_step": r["union_per_step"],
                             "host_bytes_per_step": host_bytes, "achieved_link_gbs": link,
                             "link_copy_gbs": c2c, "link_frac": link / c2c,
                             "link_peak_source": "pinned host-to-device copy measured in this run"}}
    if cut_weak:
        extra["cut_weak"] = cut_weak
    store.close()
    return r, extra


def extras(args, device):
    """The other decode and prefill workloads of the metric, timed on this GPU
    after the headline: verify batches, low-bit records, mixed widths,
    records in host memory (with and without the cut), the lookahead, the
    prefill chunk with 4-bit and with 3-bit routed records."""
    import argparse as _ap
    import torch
    res = {}
    for name, nb in (("c2", 4), ("c2", 1), ("c3b3", 4), ("c3b3", 1), ("c3b2", 4), ("c3b2", 1)):
        setup = decode_setup(name, nb, device, seed=1)
        r = time_decode(setup, nb, args.steps, args.warmup, 0, 1, device, e2e=False)
        res[f"{name}_nb{nb}"] = decode_line(name, nb, r)
        del setup
        torch.cuda.empty_cache()
    # a union mixing 4-, 3- and 2-bit records (a third of the experts each)
    setup = decode_setup("c2", 4, device, seed=1, mixed=True)
    r = time_decode(setup, 4, args.steps, args.warmup, 0, 1, device, e2e=False)
    res["c2mix_nb4"] = decode_line("c2", 4, r, {"record_widths": "4/3/2-bit, a third of the experts each"})
    del setup
    torch.cuda.empty_cache()
    # every routed record in host memory, read over the C2C link
    c2c = c2c_copy_gbs(device)
    for key, cut in (("c2host_nb4", 0.0), ("c2hostcut_nb4", 0.08)):
        r, extra = host_tier_extra(device, 4, cut, c2c)
        res[key] = decode_line("c2", 4, r, extra)
        torch.cuda.empty_cache()
    # the 48-layer stack with the one-layer lookahead on every layer
    setup = decode_setup("c1", 1, device, seed=1)
    dl = setup["views"][0]
    dl.set_flags(dl.src[0].flags | 4)
    r = time_decode(setup, 1, args.steps, args.warmup, 0, 1, device, e2e=False)
    res["c1_lookahead"] = decode_line("c1", 1, r, {"lookahead": "every layer predicts the next and prefetches "
                                                                "its device-memory records into L2"})
    del setup, dl
    torch.cuda.empty_cache()
    # the prefill chunk with 4-bit records, then with 3-bit routed records
    for name in ("c4", "c4b3"):
        a = _ap.Namespace(**vars(args))
        a.workload, a.nb = name, 0
        r = run_prefill(a, 0, 1, device)
        gu = r["flops"]["gate_up_gemm"] / (r["kernel_ms"]["gate_up_gemm"] * 1e-3) / 1e12
        dn = r["flops"]["down_gemm"] / (r["kernel_ms"]["down_gemm"] * 1e-3) / 1e12
        res[name] = {"workload": WORKLOADS[name], "ms_per_step": r["ms"], "rows_per_s": r["t"] / (r["ms"] * 1e-3),
                     "roofline": {"bound": "tensor", "kernel": "gate_up_gemm", "achieved": gu, "peak": r["peak"],
                                  "unit": "TFLOP/s", "frac": gu / r["peak"],
                                  "peak_source": r["peak_kind"] + " bf16 burst",
                                  "algorithmic_flops_per_launch": r["flops"]["gate_up_gemm"]},
                     "down_gemm": {"achieved": dn, "frac": dn / r["peak"]},
                     "kernel_ms": r["kernel_ms"], "clocks": r["clocks"]}
        torch.cuda.empty_cache()
    return res


def run_prefill(args, rank, world, device):
    """One step = one moe_prefill call over the 4096-row chunk (10 kernels)."""
    import torch
    from quantized_routed_expert_fn_gb300 import build, moe, synth

    build.build()
    moe.lib()
    torch.cuda.set_device(device)
    cfg = synth.CONFIGS[args.workload]
    t = args.nb or cfg["nb"]
    H, E, k, I = cfg["hidden"], cfg["n_experts"], cfg["top_k"], cfg["inter"]
    layers = synth.make_device_layers(args.workload, seed=1 + rank, device=device)
    rng = np.random.default_rng(40 + rank)
    layers[0].router = torch.from_numpy(synth.zipf_router_bits(rng, E, H).view(np.int16)).to(device)
    dl = moe.DeviceLayers(layers, device=device)
    x_host = torch.from_numpy(synth.make_prefill_x(rng, t, H))
    x = x_host.to(device)
    out = torch.empty((t, H), dtype=torch.int16, device=device)
    idx = torch.zeros((t, k), dtype=torch.int32, device=device)
    ws = moe.alloc_workspace(moe.prefill_workspace(dl, t), device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    nk = moe.PREFILL_KERNELS

    def new_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
        for e in evs:
            e.record(stream)  # creates the event
        return evs

    for _ in range(max(args.warmup, 3)):
        moe.prefill(dl, x, out, ws, status, idx, stream=stream)
    torch.cuda.synchronize()
    if status.item() != 0:
        raise RuntimeError(f"device status {moe.STATUS_NAMES.get(status.item())}")
    ids = idx.cpu().numpy()
    counts = np.bincount(ids.ravel(), minlength=E)
    used = int((counts > 0).sum())
    ent = t * k + t  # routed entries + the shared expert over every row
    flops = {"router_gemm": 2.0 * E * t * 2 * H, "gate_up_gemm": 2.0 * ent * 2 * I * H,
             "down_gemm": 2.0 * ent * H * I}
    from quantized_routed_expert_fn_gb300.synth import record_layout
    rec, srec = record_bytes(record_layout(H, I, cfg["bits"])), record_bytes(record_layout(H, I, 4))
    bytes_per_step = used * rec + srec + E * H * 2 + H * 2 + t * H * 4 + t * H * 2

    dist = world > 1
    if dist:
        import torch.distributed as td
    sets = [new_events() for _ in range(args.steps)]
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        td.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(args.steps):
        moe.prefill(dl, x, out, ws, status, idx, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    if dist:
        td.barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    # per-kernel device times: the same steps again, an event before each kernel
    # (the events' own gaps stay out of the step time above)
    for i in range(args.steps):
        moe.prefill_timed(dl, x, out, ws, status, sets[i], idx, stream=stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    if status.item() != 0:
        raise RuntimeError(f"device status {moe.STATUS_NAMES.get(status.item())}")
    kernel_ms = {name: sum(s[j].elapsed_time(s[j + 1]) for s in sets) / args.steps
                 for j, name in enumerate(moe.PREFILL_KERNEL_NAMES)}

    x_pin = x_host.pin_memory()
    o_pin = torch.empty((t, H), dtype=torch.int16).pin_memory()

    def e2e_step():
        x.copy_(x_pin, non_blocking=True)
        moe.prefill(dl, x, out, ws, status, idx, stream=stream)
        o_pin.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    if dist:
        td.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    ms, e2e_ms = reduce_over_ranks([ms, e2e_ms], world, device)
    top = max(flops, key=lambda n: kernel_ms[n])
    peak, peak_kind = load_peaks("tensor")
    achieved = flops[top] / (kernel_ms[top] * 1e-3) / 1e12
    return dict(ms=ms, e2e_ms=e2e_ms, rows=t * world, t=t, kernel_ms=kernel_ms, top=top, flops=flops,
                achieved=achieved, peak=peak, peak_kind=peak_kind, clocks=clocks, bytes=bytes_per_step,
                used_experts=used, max_rows=int(counts.max()))


def oracle_prefill_sample(t, budget_s, workload="c4"):
    """Time the oracle's prefill rows (bf16 mirror, as the parity tests use it)
    on host cores over the first rows of the same chunk, drawn on the host."""
    import oracle
    from quantized_routed_expert_fn_gb300 import synth
    rng = np.random.default_rng(40)
    layer = synth.make_config_layers(workload, seed=1000, n_layers=1)[0]
    synth.zipf_router(rng, layer)
    x = synth.make_prefill_x(rng, t, layer.hidden)
    ol = oracle.Layer(layer)
    cores = oracle.threads()
    done, secs, chunk = 0, 0.0, max(cores, 1)
    while secs < budget_s and done < t:
        rows = np.arange(done, min(t, done + chunk))
        t0 = time.perf_counter()
        oracle.prefill_rows(ol, x, rows, mirror=True)
        secs += time.perf_counter() - t0
        done += len(rows)
    return dict(value=done / secs, rows=done, seconds=secs, cores=cores)


def oracle_sample(name, nb, budget_s, parallel=False, n_src=2):
    """Time the oracle (as it stands) on host cores over the first layers of
    the same workload, drawn on the host with the same distributions; layers
    cycle over n_src generated ones (the time of a layer does not depend on
    its values).  parallel: the matvecs' output rows over every host thread."""
    import oracle
    from quantized_routed_expert_fn_gb300 import synth
    cfg = synth.CONFIGS[name]
    rng = np.random.default_rng(5)
    x = synth.make_x(rng, nb, cfg["hidden"])
    src = [oracle.Layer(L) for L in synth.make_config_layers(name, seed=1000, n_layers=min(n_src, cfg["n_layers"]))]
    oracle.set_parallel_rows(parallel)
    layers_done, t_total = 0, 0.0
    try:
        while t_total < budget_s and layers_done < cfg["n_layers"]:
            t0 = time.perf_counter()
            r = oracle.moe_layer(src[layers_done % len(src)], x)
            t_total += time.perf_counter() - t0
            x = r["out"]
            layers_done += 1
    finally:
        oracle.set_parallel_rows(False)
    return dict(value=nb * layers_done / t_total, layers=layers_done, seconds=t_total,
                cores=oracle.threads() if parallel else 1)


def reference_arm(args, config, prefill):
    """The reference arm: the oracle, as it stands, on all host cores.  Each of
    the W + K steps is a bounded sample of the workload -- one layer of nb rows
    (decode) or a fixed block of the chunk's rows (prefill) -- and the line
    reports exactly the K steps it timed."""
    import oracle
    from quantized_routed_expert_fn_gb300 import synth
    cfg = synth.CONFIGS[args.workload]
    nb = args.nb or cfg["nb"]
    cores = oracle.threads()
    config = dict(config, l2="not applicable: the oracle runs on the host")
    if prefill:
        rng = np.random.default_rng(40)
        layer = synth.make_config_layers(args.workload, seed=1000, n_layers=1)[0]
        synth.zipf_router(rng, layer)
        x = synth.make_prefill_x(rng, nb, layer.hidden)
        ol = oracle.Layer(layer)
        per = max(cores, 8)
        rows_of = lambda s: np.arange(s * per, s * per + per) % nb

        def step(s):
            oracle.prefill_rows(ol, x, rows_of(s), mirror=True)
        rows_per_step, what = per, f"{per} rows of the chunk (bf16 mirror)"
    else:
        src = [oracle.Layer(L) for L in synth.make_config_layers(args.workload, seed=1000,
                                                                 n_layers=min(2, cfg["n_layers"]))]
        state = {"x": synth.make_x(np.random.default_rng(5), nb, cfg["hidden"])}
        oracle.set_parallel_rows(True)

        def step(s):
            state["x"] = oracle.moe_layer(src[s % len(src)], state["x"])["out"]
        rows_per_step, what = nb, f"one layer of {nb} row(s), output rows over the host threads"
    for s in range(args.warmup):
        step(s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(args.warmup + s)
    secs = time.perf_counter() - t0
    oracle.set_parallel_rows(False)
    value = rows_per_step * args.steps / secs
    line = {"metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step {what}; {args.steps} steps in {secs:.1f} s"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c1", choices=sorted(WORKLOADS))
    ap.add_argument("--nb", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=0, help="override the stack depth (profiling a smaller case)")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="c1 only: skip the other workloads' figures")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from quantized_routed_expert_fn_gb300 import synth
    cfg = synth.CONFIGS[args.workload]
    nb = args.nb or cfg["nb"]
    config = {"workload": WORKLOADS[args.workload], "nb": nb, "layers": args.layers or cfg["n_layers"],
              "l2": "inputs larger than L2 (each step streams every layer's union records once)"}

    prefill = args.workload in ("c4", "c4b3")
    if prefill:
        config = {"workload": WORKLOADS[args.workload], "t": nb, "layers": 1,
                  "l2": "inputs larger than L2 (about 0.9 GB of expert records per step)"}
    if args.impl == "reference":
        if rank == 0:
            reference_arm(args, config, prefill)
        return

    import torch
    if world > 1:
        import torch.distributed as td
        td.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    device = torch.device(f"cuda:{local}")
    if prefill:
        r = run_prefill(args, rank, world, device)
        if rank == 0:
            cpu = oracle_prefill_sample(nb, budget_s=args.cpu_budget, workload=args.workload)
            H = synth.CONFIGS[args.workload]["hidden"]
            line = {
                "metric": METRIC, "value": job_rows_per_s(r["t"], world, r["ms"]), "unit": "rows/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
                "e2e": {"value": job_rows_per_s(r["t"], world, r["e2e_ms"]), "unit": "rows/s",
                        "h2d_bytes_per_step": nb * H * 4, "d2h_bytes_per_step": nb * H * 2},
                "gpu_launches": args.steps * 10,
                "roofline": {"bound": "tensor", "achieved": r["achieved"], "peak": r["peak"], "unit": "TFLOP/s",
                             "frac": r["achieved"] / r["peak"],
                             "traffic": ncu_traffic(args.workload) if r["top"] == "gate_up_gemm" else None,
                             "kernel": r["top"],
                             "peak_source": r["peak_kind"] + " bf16 burst",
                             "algorithmic_flops_per_launch": r["flops"][r["top"]]},
                "kernel_ms": r["kernel_ms"],
                "gemm_tflops": {n: r["flops"][n] / (r["kernel_ms"][n] * 1e-3) / 1e12 for n in r["flops"]},
                "step_hbm_gbs": r["bytes"] / (r["ms"] * 1e-3) / 1e9,
                "used_experts": r["used_experts"], "max_expert_rows": r["max_rows"],
                "cpu_baseline": {"value": cpu["value"], "unit": "rows/s", "cores": cpu["cores"], "kind": "oracle",
                                 "sample": f"first {cpu['rows']} rows of the chunk (bf16 mirror), "
                                           f"{cpu['seconds']:.1f} s"},
                "clocks": r["clocks"],
            }
            print(json.dumps(line))
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    r = run_ours(args, rank, world, device)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    config["l2"] = r["l2"]
    cpu1 = oracle_sample(args.workload, nb, budget_s=args.cpu_budget, parallel=False)
    cpun = oracle_sample(args.workload, nb, budget_s=args.cpu_budget, parallel=True)
    value = job_rows_per_s(r["nb"] * r["nl"], world, r["ms"])
    e2e_value = job_rows_per_s(r["nb"] * r["nl"], world, r["e2e_ms"])
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config,
        "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": nb * cfg["hidden"] * 4,
                "d2h_bytes_per_step": nb * cfg["hidden"] * 4},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": r["achieved"], "peak": r["peak"], "unit": "GB/s",
                     "frac": r["achieved"] / r["peak"],
                     "traffic": ncu_traffic(args.workload) if args.workload == "c1" and not args.layers else None,
                     "peak_source": r["peak_kind"], "algorithmic_bytes_per_launch": r["bytes"]},
        "cpu_baseline": {"value": cpun["value"], "unit": "rows/s", "cores": cpun["cores"], "kind": "oracle",
                         "sample": f"first {cpun['layers']} layers of the workload, {cpun['seconds']:.1f} s, "
                                   f"output rows over {cpun['cores']} host threads"},
        "cpu_baseline_1core": {"value": cpu1["value"], "unit": "rows/s", "cores": 1, "kind": "oracle",
                               "sample": f"first {cpu1['layers']} layers of the workload, {cpu1['seconds']:.1f} s"},
        "clocks": r["clocks"],
        "union_sizes": r["unions"],
    }
    if args.extras and world == 1 and args.workload == "c1" and not args.layers:
        line["extras"] = extras(args, device)
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
