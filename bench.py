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
    "c1": dict(bytes=1211.6e6, sources=["decode.cu", "decode.cuh", "codec.cuh", "common.cuh"],
               sha="59453414ceb4f5e0"),
    "c4": dict(bytes=640.8e6, sources=["prefill.cu", "prefill.cuh", "tc05.cuh", "common.cuh"],
               sha="c9912dbb7f4bb4a7"),
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


def layer_bytes(L, union_size: int, nb: int) -> int:
    """Algorithmic bytes of one layer: router + shared gate + union records +
    shared record + layer input and output."""
    b = L.n_experts * L.hidden * 2
    b += union_size * record_bytes(L.layout)
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


def run_ours(args, rank, world, device):
    import torch
    from quantized_routed_expert_fn_gb300 import build, moe, synth

    build.build()
    moe.lib()
    torch.cuda.set_device(device)
    name = args.workload
    cfg = synth.CONFIGS[name]
    nb = args.nb or cfg["nb"]
    layers = synth.make_device_layers(name, seed=1 + rank, device=device, n_layers=args.layers or None)
    dl = moe.DeviceLayers(layers, device=device)
    nl = dl.n
    H = cfg["hidden"]
    gen = torch.Generator(device="cpu").manual_seed(100 + rank)
    x_host = torch.randn((nb, H), generator=gen, dtype=torch.float32)
    if nb > 1:  # correlated rows: union of about 30 of 40 possible experts
        c = torch.randn((1, H), generator=gen)
        x_host = (0.55 ** 0.5) * c + (0.45 ** 0.5) * x_host
    x = x_host.to(device)
    out = torch.empty_like(x)
    ws = moe.alloc_workspace(moe.forward_workspace(dl, nb), device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    slot = torch.zeros((nl, 64), dtype=torch.int64, device=device)
    wmap = torch.zeros((nl, 4, 64), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        moe.forward(dl, x, out, ws, status, slot, wmap, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if status.item() != 0:
        raise RuntimeError(f"device status {moe.STATUS_NAMES.get(status.item())}")
    unions = [int(v) for v in slot[:, 63].cpu().tolist()]
    bytes_per_step = sum(layer_bytes(L, u, nb) for L, u in zip(layers, unions))

    dist = world > 1
    if dist:
        import torch.distributed as td
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.3)
    # device-timed region: inputs resident in HBM
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        td.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    if dist:
        td.barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    clocks = sampler.stop() if sampler else None
    if status.item() != 0:
        raise RuntimeError(f"device status {moe.STATUS_NAMES.get(status.item())}")

    # end to end through the same call with host buffers: H2D of x, D2H of out
    x_pin = x_host.pin_memory()
    o_pin = torch.empty((nb, H), dtype=torch.float32).pin_memory()

    def e2e_step():
        x.copy_(x_pin, non_blocking=True)
        moe.forward(dl, x, out, ws, status, slot, wmap, stream=stream)
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
    if dist:
        td.barrier()

    ms, e2e_ms = reduce_over_ranks([ms, e2e_ms], world, device)
    rows = nb * nl * world
    peak, peak_kind = load_peaks()
    achieved = bytes_per_step / (ms * 1e-3) / 1e9
    return dict(ms=ms, e2e_ms=e2e_ms, rows=rows, nb=nb, nl=nl, bytes=bytes_per_step, achieved=achieved,
                peak=peak, peak_kind=peak_kind, clocks=clocks, unions=unions)


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
        moe.prefill_timed(dl, x, out, ws, status, sets[i], idx, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    if dist:
        td.barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
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


def oracle_sample(name, nb, budget_s):
    """Time the oracle (as it stands) on host cores on the first layers of the
    same workload, drawn on the host with the same distributions."""
    import oracle
    from quantized_routed_expert_fn_gb300 import synth
    cfg = synth.CONFIGS[name]
    rng = np.random.default_rng(5)
    x = synth.make_x(rng, nb, cfg["hidden"])
    layers_done, t_total = 0, 0.0
    layer_iter = 0
    while t_total < budget_s and layer_iter < cfg["n_layers"]:
        L = synth.make_config_layers(name, seed=1000 + layer_iter, n_layers=1)[0]
        ol = oracle.Layer(L)
        t0 = time.perf_counter()
        r = oracle.moe_layer(ol, x)
        t_total += time.perf_counter() - t0
        x = r["out"]
        layers_done += 1
        layer_iter += 1
    # the oracle's layer path is serial C: one host core
    return dict(value=nb * layers_done / t_total, layers=layers_done, seconds=t_total, cores=1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c1", choices=sorted(WORKLOADS))
    ap.add_argument("--nb", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--layers", type=int, default=0, help="override the stack depth (profiling a smaller case)")
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
    if args.impl == "reference" and prefill:
        if rank != 0:
            return
        s = oracle_prefill_sample(nb, budget_s=min(args.cpu_budget, 20.0), workload=args.workload)
        line = {"metric": METRIC, "value": s["value"], "unit": "rows/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1000.0 * nb / s["value"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "impl": "reference",
                "cpu_baseline": {"value": s["value"], "unit": "rows/s", "cores": s["cores"], "kind": "oracle",
                                 "sample": f"first {s['rows']} rows of the chunk, {s['seconds']:.1f} s"},
                "e2e": {"value": s["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    if args.impl == "reference":
        if rank != 0:
            return
        s = oracle_sample(args.workload, nb, budget_s=min(args.cpu_budget, 20.0))
        ms = 1000.0 * nb * (args.layers or cfg["n_layers"]) / s["value"]
        line = {"metric": METRIC, "value": s["value"], "unit": "rows/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config, "impl": "reference",
                "cpu_baseline": {"value": s["value"], "unit": "rows/s", "cores": s["cores"], "kind": "oracle",
                                 "sample": f"first {s['layers']} layers of the workload, {s['seconds']:.1f} s"},
                "e2e": {"value": s["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
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
    cpu = oracle_sample(args.workload, nb, budget_s=args.cpu_budget) if world == 1 or rank == 0 else None
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
        "cpu_baseline": {"value": cpu["value"], "unit": "rows/s", "cores": cpu["cores"], "kind": "oracle",
                         "sample": f"first {cpu['layers']} layers of the workload, {cpu['seconds']:.1f} s"},
        "clocks": r["clocks"],
        "union_sizes": sorted(set(r["unions"])),
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
