"""Benchmark of the MoE layer forward (libmoe on one GB300, replicas for N > 1).

Headline workload: the Mixtral-8x7B-shaped MoE layer (H=4096, E=8, top-2 softmax, SwiGLU
I=14336, bf16 weights N(0, 0.02), x ~ N(0, 1) bf16, router fp32 N(0, 0.02)), T = 4096 tokens
per step, all experts VRAM-resident.  One step = one full layer forward (router, gating,
dispatch, gather, grouped SwiGLU, combine) through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--T 4096] [--impl ours|reference]

Prints ONE JSON line (rank 0).  See the design notes for the roofline arithmetic.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

WORKLOADS = {"tiny": wl.TINY, "mixtral": wl.MIXTRAL, "qwen": wl.QWEN, "deepseek": wl.DEEPSEEK,
             "qwen_nvfp4": wl.QWEN_NVFP4}
CANONICAL_E = {name: c.E for name, c in WORKLOADS.items()}   # before any --experts override
WORKLOAD_NAMES = {"tiny": "Tiny", "mixtral": "Mixtral-8x7B-shaped", "qwen": "Qwen1.5-MoE-A2.7B-shaped",
                  "deepseek": "DeepSeek-V3-shaped INT4",
                  "qwen_nvfp4": "Qwen1.5-MoE-A2.7B-shaped NVFP4"}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 7900.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            flat = {}

            def walk(o, pre=""):
                if isinstance(o, dict):
                    for k, v in o.items():
                        walk(v, f"{pre}{k}.")
                elif isinstance(o, (int, float)):
                    flat[pre[:-1]] = float(o)
            walk(d)
            get = lambda *names: next((flat[k] for k in flat for n in names if k.split(".")[-1] == n), None)  # noqa
            hbm, tf, tfs = get("hbm_gbs"), get("bf16_tflops"), get("bf16_tflops_sustained")
            if hbm and tf:
                return {"hbm_gbs": hbm, "bf16_tflops": tf, "bf16_tflops_sustained": tfs or tf,
                        "source": "measured"}
        except Exception:
            pass
    return dict(FALLBACK_PEAKS, source="fallback")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if len(r) > 2 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if len(r) > 5 + i and r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(self.rows)}


def layer_work(cfg, T, n_unique, shared_merged=False):
    """Algorithmic FLOPs and bytes of one layer call and of its two expert GEMM launches (which
    include the shared expert when the library runs it inside the routed launches)."""
    H, I, k, E, Is = cfg.H, cfg.I, cfg.k, cfg.E, cfg.Is
    rows = T * k
    # bytes per weight: bf16; INT4 codes + a bf16 scale per 128; NVFP4 codes + an E4M3 per 16
    bpw = {"bf16": 2.0, "int4_g128": 0.5 + 2.0 / 128, "nvfp4": 0.5 + 1.0 / 16}[cfg.wdtype]
    gu_flops = 2.0 * rows * H * 2 * I
    dn_flops = 2.0 * rows * I * H
    gu_bytes = n_unique * 2 * I * H * bpw + rows * H * 2 + rows * I * 2
    dn_bytes = n_unique * H * I * bpw + rows * I * 2 + rows * H * 2
    flops = gu_flops + dn_flops + 2.0 * T * H * E + 6.0 * T * H * Is
    nbytes = (n_unique * 3 * H * I * bpw + 3 * H * Is * bpw + 4.0 * H * E + 2 * T * H * 2
              + 2 * 2 * rows * H * 2)
    if shared_merged and Is:
        gu_flops += 2.0 * T * H * 2 * Is
        dn_flops += 2.0 * T * Is * H
        gu_bytes += 2 * Is * H * bpw + T * H * 2 + T * Is * 2
        dn_bytes += Is * H * bpw + T * Is * 2 + T * H * 2
    return dict(flops=flops, bytes=nbytes, gu=(gu_flops, gu_bytes), dn=(dn_flops, dn_bytes))


KERNEL_SOURCES = ["expert_dispatch_streaming_gb300/csrc/tc_gemm.cu",
                  "expert_dispatch_streaming_gb300/csrc/common.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def kernel_sources_sha256(files=None):
    h = hashlib.sha256()
    for f in (files or KERNEL_SOURCES):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(workload, T, E, kernel):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu capture of the
    same workload (profiles/traffic.json), or None when there is none or the kernel sources
    changed since it was taken (each entry records the sources' sha256)."""
    if E != CANONICAL_E.get(workload) or not os.path.exists(TRAFFIC_FILE):
        return None
    try:
        entries = json.load(open(TRAFFIC_FILE))["entries"]
    except (ValueError, KeyError):
        return None
    for e in entries:
        if (e.get("workload"), e.get("T"), e.get("kernel")) == (workload, T, kernel):
            # the entry's own source list (default: the expert GEMM's)
            if e.get("kernel_source_sha256") != kernel_sources_sha256(e.get("sources")):
                return None
            return int(e["traffic_bytes_per_launch"])
    return None


def roofline_of(flops, nbytes, seconds, pk, sustained=False):
    tf_peak = pk["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    t_tc = flops / (tf_peak * 1e12)
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    if t_tc >= t_hbm:
        ach = flops / seconds / 1e12
        return {"bound": "tensor", "achieved": round(ach, 2), "peak": tf_peak, "unit": "TFLOP/s",
                "frac": round(ach / tf_peak, 4)}
    ach = nbytes / seconds / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / pk["hbm_gbs"], 4)}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (timing: the job ends when its slowest replica ends)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job throughput of N independent replicas: all ranks' units over the max time."""
    return units_per_rank * world / seconds


def run_ours(args, rank, world, local_rank):
    import torch
    import expert_dispatch_streaming_gb300 as moe
    from expert_dispatch_streaming_gb300 import synthetic as syn

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    moe.set_ffn_kernel(args.ffn_kernel)
    moe.set_pdl(args.pdl)
    cfg = WORKLOADS[args.workload]
    pk = peaks()
    layer = syn.DeviceLayer(cfg, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def measure(T, steps, warmup, with_e2e, layer=layer, cfg=cfg):
        xb = wl.tokens(cfg, T)
        x = syn.to_device_bits(xb, dev)
        out = torch.empty_like(x)
        ws = layer.workspace(T)
        ids = torch.empty((T, cfg.k), dtype=torch.int32, device=dev)
        with torch.cuda.stream(stream):
            layer.forward(x, ws, out, stream=stream, ids_out=ids)
        stream.synchronize()
        n_unique = int(np.unique(ids.cpu().numpy()).size)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_N_PHASE_EVENTS)]
               for _ in range(steps)]
        for row in evs:          # torch creates the CUDA events on first record
            for ev in row:
                ev.record(stream)
        for _ in range(warmup):
            layer.forward(x, ws, out, stream=stream)
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        launches = 0
        merged = False
        fused = False
        with ClockSampler(local_rank) as clk:
            t0.record(stream)
            for i in range(steps):
                _, st = layer.forward(x, ws, out, stream=stream, phase_events=evs[i])
                launches += st.n_launches
                merged = bool(st.shared_merged)
                fused = bool(st.fused_decode)
            t1.record(stream)
            stream.synchronize()
        torch.cuda.synchronize()
        ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
        if world > 1:
            torch.distributed.barrier()
        ph = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(5)]
                       for i in range(steps)])
        res = dict(T=T, ms_per_step=ms / steps, tokens_per_s=job_throughput(T * steps, world, ms / 1e3),
                   n_unique=n_unique, phase_ms=ph.mean(0).tolist(), launches=launches, merged=merged,
                   fused=fused,
                   clocks=clk.summary(), mode="eager")
        if args.graph:
            # the same call captured once in a CUDA graph (a resident-layer call is fully
            # asynchronous, so it captures as is) and replayed: removes host launch gaps
            gevs = [torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_N_PHASE_EVENTS)]
            for ev in gevs:
                ev.record(stream)
            stream.synchronize()
            # the timed graph has no phase events (event nodes between the kernels would cut the
            # programmatic launch edges between them); a second graph with events gives the split
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                layer.forward(x, ws, out, stream=stream)
            gp = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gp, stream=stream):
                layer.forward(x, ws, out, stream=stream, phase_events=gevs)
            for _ in range(warmup):
                g.replay()
                gp.replay()
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            gph = []
            with ClockSampler(local_rank) as gclk:
                t0.record(stream)
                with torch.cuda.stream(stream):
                    for i in range(steps):
                        g.replay()
                t1.record(stream)
                stream.synchronize()
            gms = max_over_ranks(t0.elapsed_time(t1), world, dev)
            # phase split of one replay (events inside the graph are re-recorded per replay)
            with torch.cuda.stream(stream):
                gp.replay()
            stream.synchronize()
            gph = [gevs[j].elapsed_time(gevs[j + 1]) for j in range(5)]
            res["graph"] = dict(ms_per_step=gms / steps,
                                tokens_per_s=T * steps * world / (gms / 1e3), phase_ms=gph,
                                clocks=gclk.summary())
            if gms < ms:
                res.update(ms_per_step=gms / steps, tokens_per_s=T * steps * world / (gms / 1e3),
                           phase_ms=gph, clocks=gclk.summary(), mode="cuda_graph")
            res["eager_ms_per_step"] = ms / steps
            del g, gp
        if with_e2e:
            # End to end through the public call with host buffers: every step copies its
            # input from pinned host memory and its result back.  As a serving loop would run
            # it, the copies of neighbouring steps overlap this step's layer: inputs and outputs
            # are double-buffered on the device, host-to-device copies run on one copy stream
            # and device-to-host copies on another, ordered by events.
            xh = torch.from_numpy(xb.view(np.int16)).pin_memory()
            oh = torch.empty_like(xh).pin_memory()
            xs, outs = [x, torch.empty_like(x)], [out, torch.empty_like(out)]
            hs, ds = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
            ev_in = [torch.cuda.Event() for _ in range(2)]
            ev_used = [torch.cuda.Event() for _ in range(2)]
            ev_out = [torch.cuda.Event() for _ in range(2)]

            def e2e_steps(n):
                for i in range(n):
                    b = i & 1
                    if i >= 2:
                        hs.wait_event(ev_used[b])      # step i - 2's layer read xs[b]
                    with torch.cuda.stream(hs):
                        xs[b].copy_(xh, non_blocking=True)
                        ev_in[b].record(hs)
                    stream.wait_event(ev_in[b])
                    if i >= 2:
                        stream.wait_event(ev_out[b])   # step i - 2's result left outs[b]
                    layer.forward(xs[b], ws, outs[b], stream=stream)
                    ev_used[b].record(stream)
                    ds.wait_event(ev_used[b])
                    with torch.cuda.stream(ds):
                        oh.copy_(outs[b], non_blocking=True)
                        ev_out[b].record(ds)
                stream.wait_event(ev_out[(n - 1) & 1])

            e2e_steps(3)
            torch.cuda.synchronize(dev)
            if world > 1:
                torch.distributed.barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            hs.wait_event(e0)
            e2e_steps(steps)
            e1.record(stream)
            stream.synchronize()
            ems = max_over_ranks(e0.elapsed_time(e1), world, dev)
            res["e2e"] = {"value": round(T * steps * world / (ems / 1e3), 1), "unit": "tokens/s",
                          "h2d_bytes_per_step": int(xh.numel() * 2),
                          "d2h_bytes_per_step": int(oh.numel() * 2),
                          "copies": "overlapped with neighbouring steps (two copy streams)"}
        return res

    names = ["route+dispatch+gather", "shared_expert", "gate_up_gemm", "down_gemm", "combine"]

    def dominant(wname, c, T, r):
        """Roofline of the larger of the two expert-FFN phases (gate/up or down); with the
        fused decode kernel, of that one launch (the whole layer)."""
        w = layer_work(c, T, r["n_unique"], r["merged"])
        if r.get("fused"):
            roof = roofline_of(w["flops"], w["bytes"], sum(r["phase_ms"]) / 1e3, pk)
            roof.update({"kernel": "decode_layer_kernel (whole layer)",
                         "traffic": profiled_traffic(wname, T, c.E, "decode_layer_kernel"),
                         "peak_source": pk["source"], "share_of_step": 1.0})
            return w, roof
        share = np.array(r["phase_ms"]) / max(sum(r["phase_ms"]), 1e-9)
        dom = 2 if share[2] >= share[3] else 3
        roof = roofline_of(*(w["gu"] if dom == 2 else w["dn"]), r["phase_ms"][dom] / 1e3, pk)
        roof.update({"kernel": names[dom],
                     "traffic": profiled_traffic(wname, T, c.E, names[dom]),
                     "peak_source": pk["source"], "share_of_step": round(float(share[dom]), 4)})
        return w, roof

    def entry(wname, c, T, r):
        w, roof = dominant(wname, c, T, r)
        return {"tokens_per_s": round(r["tokens_per_s"], 1),
                "ms_per_step": round(r["ms_per_step"], 4), "mode": r["mode"],
                "eager_ms_per_step": round(r.get("eager_ms_per_step", r["ms_per_step"]), 4),
                "n_unique": r["n_unique"], "phase_ms": [round(v, 4) for v in r["phase_ms"]],
                "layer_roofline": roofline_of(w["flops"], w["bytes"], r["ms_per_step"] / 1e3, pk),
                # (the fused decode kernel has no separate gate/up phase)
                "gate_up_roofline": (roofline_of(*w["gu"], r["phase_ms"][2] / 1e3, pk)
                                     if r["phase_ms"][2] > 0 and not r.get("fused") else None),
                "dominant_roofline": roof}

    head = measure(args.T, args.steps, args.warmup, True)
    sweep = {}
    if args.sweep:
        for T in cfg.Ts:
            if T == args.T:
                continue
            r = measure(T, max(5, min(args.steps, 20)), 3, False)
            sweep[str(T)] = entry(args.workload, cfg, T, r)
    del layer
    torch.cuda.empty_cache()

    # every other workload of the task, each over its batch sizes (weights resident)
    configs = {}
    for wname in (args.configs.split(",") if args.configs else []):
        if wname == args.workload or wname not in WORKLOADS:
            continue
        c = WORKLOADS[wname]
        t0 = time.time()
        lay = syn.DeviceLayer(c, device=dev)
        per_t = {}
        for T in c.Ts:
            r = measure(T, max(5, min(args.steps, 10)), 3, False, layer=lay, cfg=c)
            per_t[str(T)] = entry(wname, c, T, r)
        configs[wname] = {"workload": f"{WORKLOAD_NAMES[wname]} MoE layer forward",
                          "H": c.H, "E": c.E, "k": c.k, "I": c.I, "Is": c.Is,
                          "weights": c.wdtype, "setup_s": round(time.time() - t0, 1),
                          "T": per_t}
        del lay
        torch.cuda.empty_cache()

    w, roof = dominant(args.workload, cfg, args.T, head)
    result = {
        "metric": f"MoE-layer tokens/s ({WORKLOAD_NAMES[args.workload]} layer)",
        "value": round(head["tokens_per_s"], 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(head["ms_per_step"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) tokens)",
        "config": {"workload": f"{WORKLOAD_NAMES[args.workload]} MoE layer forward, T={args.T}",
                   "H": cfg.H, "E": cfg.E, "k": cfg.k, "I": cfg.I, "Is": cfg.Is,
                   "weights": cfg.wdtype, "T": args.T,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "expert weights exceed L2 (126 MB) and are streamed every step"},
        "layer_roofline": roofline_of(w["flops"], w["bytes"], head["ms_per_step"] / 1e3, pk),
        "roofline": roof,
        "phase_ms": {n: round(v, 4) for n, v in zip(names, head["phase_ms"])},
        "launch_mode": head["mode"],
        "eager_ms_per_step": round(head.get("eager_ms_per_step", head["ms_per_step"]), 4),
        "n_unique_experts": head["n_unique"],
        "e2e": head.get("e2e"), "gpu_launches": head["launches"], "clocks": head["clocks"],
        "sweep": sweep,
        "configs": configs,
    }
    return result


def tier_bound_ms(resident_ms, miss_bytes_per_step, link_gbs):
    """Lower bound on one streamed decode step from the two memory tiers it crosses ("The
    Billion-Token Bottleneck", "Tiered Memory": hot experts in HBM, the rest streamed from system
    RAM over the host link): the step's compute with every bundle resident, and its missed
    bytes at the probed host-link rate.  Copies that overlap compute perfectly reach the larger
    of the two."""
    return max(resident_ms, miss_bytes_per_step / (link_gbs * 1e6))


def run_streamed(args, local_rank):
    """Expert-streamed decode: 16 Qwen1.5-MoE-shaped layers, every routed bundle (16.6 GB) in
    pinned host memory, a 4 GiB VRAM slot cache under LRU, 256 decode steps per batch size,
    routing injected from the seeded locality trace.  Also runs the same trace with every
    bundle resident (a cache large enough for all bundles, pre-filled) for the overlap
    fraction."""
    import torch
    import expert_dispatch_streaming_gb300 as moe
    from expert_dispatch_streaming_gb300 import synthetic as syn

    cfg = wl.STREAMED
    dev = torch.device("cuda", local_rank)
    t0 = time.time()
    store, table = syn.host_bundle_table(cfg, cfg.layers)
    nb = store.shape[1]
    layers = [syn.DeviceLayer(cfg, layer=l, cached=True, device=dev) for l in range(cfg.layers)]
    setup_s = time.time() - t0

    def make(cap_bytes, prefetch=0, device_lru=0, copy_kernel=None):
        ck = args.copy_kernel if copy_kernel is None else copy_kernel
        c = moe.moe_expert_cache_config(slot_bytes=nb, capacity_bytes=cap_bytes,
                                        n_layers=cfg.layers, n_experts=cfg.E, bundles=table,
                                        timeout_ms=20000, verify_checksums=1, device=local_rank,
                                        time_copies=1, prefetch_next_layer=prefetch,
                                        device_lru=device_lru, copy_kernel=int(ck))
        return moe.moe_expert_cache_create(c)

    # probe: pinned H2D bandwidth of one bundle-sized copy on this machine (best of 3 rounds)
    d = torch.empty(nb, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)
    probe_gbs = 0.0
    for _ in range(3):
        with torch.cuda.stream(s):
            for i in range(4):
                d.copy_(store[i], non_blocking=True)
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for i in range(32):
                d.copy_(store[i % store.shape[0]], non_blocking=True)
            e1.record(s)
        s.synchronize()
        probe_gbs = max(probe_gbs, 32 * nb / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del d

    stream = torch.cuda.Stream(device=dev)
    out = {"setup_s": round(setup_s, 1), "bundle_bytes": nb,
           "cache_bytes": wl.STREAM_CACHE_BYTES, "slots": wl.STREAM_CACHE_BYTES // nb,
           "probe_h2d_gbs": round(probe_gbs, 1), "steps": args.stream_steps, "T": {}}
    for T in cfg.Ts:
        trace = wl.stream_trace(cfg, T, steps=args.stream_steps)
        ids_dev = torch.from_numpy(trace).to(dev)
        xs = [syn.to_device_bits(wl.stream_tokens(cfg, T, st), dev) for st in range(args.stream_steps)]
        ws = layers[0].workspace(T)
        bufs = [torch.empty_like(xs[0]) for _ in range(4)]

        def stack(x0, ids_of, cache):
            # pre-normalised stack: layer l reads u_l, adds to the residual stream x_l and
            # writes x_{l+1} and u_{l+1} = rmsnorm(x_{l+1}) (u_0 = x_0)
            x = u = x0
            for l in range(cfg.layers):
                y, un = bufs[l & 1], bufs[2 + (l & 1)]
                layers[l].forward(u, ws, out=y, forced_ids=ids_of(l), residual=x, cache=cache,
                                  stream=stream, out_normed=un)
                x, u = y, un

        def run(cache, steps):
            with torch.cuda.stream(stream):
                for st in range(steps):
                    stack(xs[st], lambda l: ids_dev[st, l], cache)

        res = {}
        cache = make(wl.STREAM_CACHE_BYTES)
        try:
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            w0 = time.perf_counter()
            run(cache, args.stream_steps)
            e1.record(stream)
            stream.synchronize()
            wall = time.perf_counter() - w0
            t_stream = e0.elapsed_time(e1) / 1e3
            st_ = moe.moe_expert_cache_stats(cache)
            copy_ms, ncopies = moe.moe_expert_cache_copy_time(cache)
            tr = moe.moe_expert_cache_trace(cache)
        finally:
            moe.moe_expert_cache_destroy(cache)
        warm = [r for r in tr if r[0] >= 16 * cfg.layers]
        res.update(tokens_per_s=round(T * args.stream_steps / t_stream, 1),
                   ms_per_step=round(1e3 * t_stream / args.stream_steps, 3),
                   wall_s=round(wall, 2),
                   hit_rate=round(st_["hits"] / max(1, st_["hits"] + st_["misses"]), 4),
                   hit_rate_after_step16=round(sum(1 - r[3] for r in warm) / max(1, len(warm)), 4),
                   misses=st_["misses"], bytes_h2d=st_["bytes_h2d"],
                   h2d_gbs=round(st_["bytes_h2d"] / max(copy_ms, 1e-9) / 1e6, 1),
                   copy_busy_s=round(copy_ms / 1e3, 4))
        res["h2d_frac_of_probe"] = round(res["h2d_gbs"] / probe_gbs, 4)
        res["miss_copies"] = "fill kernel" if args.copy_kernel else "copy engine"
        # the other copy path on the first quarter of the same trace, for comparison
        alt_steps = max(1, args.stream_steps // 4)
        alt = make(wl.STREAM_CACHE_BYTES, copy_kernel=1 - int(args.copy_kernel))
        try:
            torch.cuda.synchronize()
            e0.record(stream)
            run(alt, alt_steps)
            e1.record(stream)
            stream.synchronize()
            t_alt = e0.elapsed_time(e1) / 1e3
            sa = moe.moe_expert_cache_stats(alt)
            acopy_ms, _ = moe.moe_expert_cache_copy_time(alt)
        finally:
            moe.moe_expert_cache_destroy(alt)
        res["other_copy_path"] = {
            "miss_copies": "copy engine" if args.copy_kernel else "fill kernel",
            "steps": alt_steps, "tokens_per_s": round(T * alt_steps / t_alt, 1),
            "ms_per_step": round(1e3 * t_alt / alt_steps, 3),
            "h2d_gbs": round(sa["bytes_h2d"] / max(acopy_ms, 1e-9) / 1e6, 1)}
        # the same ids with every bundle resident (pre-filled full-size cache)
        full = make(cfg.layers * cfg.E * nb)
        try:
            run(full, min(args.stream_steps, 8))       # fill: every bundle copied once
            stream.synchronize()
            moe.moe_expert_cache_copy_time(full)
            torch.cuda.synchronize()
            e0.record(stream)
            run(full, args.stream_steps)
            e1.record(stream)
            stream.synchronize()
            t_res = e0.elapsed_time(e1) / 1e3
            assert moe.moe_expert_cache_stats(full)["misses"] <= cfg.layers * cfg.E
        finally:
            moe.moe_expert_cache_destroy(full)
        res["resident_ms_per_step"] = round(1e3 * t_res / args.stream_steps, 3)
        bound = tier_bound_ms(1e3 * t_res / args.stream_steps,
                              res["bytes_h2d"] / args.stream_steps, probe_gbs)
        res["tier_bound_ms_per_step"] = round(bound, 3)
        res["frac_of_tier_bound"] = round(bound / res["ms_per_step"], 4)
        t_copy = copy_ms / 1e3
        res["overlap_fraction"] = (round(min(1.0, max(0.0, 1 - (t_stream - t_res) / t_copy)), 4)
                                   if t_copy > 0 else None)
        # lookahead prefetch: each layer call ends by prefetching the next layer's experts,
        # predicted from that layer's previous step (never from the trace's future)
        pc = make(wl.STREAM_CACHE_BYTES, prefetch=1)
        try:
            torch.cuda.synchronize()
            e0.record(stream)
            run(pc, args.stream_steps)
            e1.record(stream)
            stream.synchronize()
            t_pf = e0.elapsed_time(e1) / 1e3
            sp = moe.moe_expert_cache_stats(pc)
            pcopy_ms, _ = moe.moe_expert_cache_copy_time(pc)
        finally:
            moe.moe_expert_cache_destroy(pc)
        res["prefetch"] = {
            "tokens_per_s": round(T * args.stream_steps / t_pf, 1),
            "ms_per_step": round(1e3 * t_pf / args.stream_steps, 3),
            "hit_rate": round(sp["hits"] / max(1, sp["hits"] + sp["misses"]), 4),
            "demand_misses": sp["misses"], "prefetch_fills": sp["prefetch_fills"],
            "prefetch_used": sp["prefetch_used"],
            "prefetch_accuracy": round(sp["prefetch_used"] / max(1, sp["prefetch_fills"]), 4),
            "bytes_h2d": sp["bytes_h2d"],
            "h2d_gbs": round(sp["bytes_h2d"] / max(pcopy_ms, 1e-9) / 1e6, 1),
            "overlap_fraction": (round(min(1.0, max(0.0, 1 - (t_pf - t_res) / (pcopy_ms / 1e3))), 4)
                                 if pcopy_ms > 0 else None)}
        # the LRU on the GPU: no host round trip per layer; one decode step (16 layers, their
        # cache decisions and miss copies) captured once as a CUDA graph and replayed per step
        # with that step's tokens and routing staged into the graph's input buffers
        dc = make(wl.STREAM_CACHE_BYTES, device_lru=1)
        try:
            x_in = torch.empty_like(xs[0])
            ids_in = torch.empty_like(ids_dev[0])

            def dstep():
                stack(x_in, lambda l: ids_in[l], dc)

            with torch.cuda.stream(stream):
                x_in.copy_(xs[0])
                ids_in.copy_(ids_dev[0])
                dstep()                                   # step 0 eagerly
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                dstep()
            torch.cuda.synchronize()
            e0.record(stream)
            with torch.cuda.stream(stream):
                for st in range(1, args.stream_steps):
                    x_in.copy_(xs[st], non_blocking=True)
                    ids_in.copy_(ids_dev[st], non_blocking=True)
                    g.replay()
            e1.record(stream)
            stream.synchronize()
            t_dev = e0.elapsed_time(e1) / 1e3
            sd = moe.moe_expert_cache_stats(dc)
            del g
        finally:
            moe.moe_expert_cache_destroy(dc)
        n_dev = args.stream_steps - 1
        ms_dev = 1e3 * t_dev / n_dev
        res["device_lru_graph"] = {
            "tokens_per_s": round(T * n_dev / t_dev, 1),
            "ms_per_step": round(ms_dev, 3),
            "hit_rate": round(sd["hits"] / max(1, sd["hits"] + sd["misses"]), 4),
            "misses": sd["misses"], "bytes_h2d": sd["bytes_h2d"],
            "steps_timed": n_dev,
            # the same tier bound (same trace, same misses) against this path's step time
            "frac_of_tier_bound": round(bound / ms_dev, 4)}
        # the faster of the two residency paths (host LRU eager, LRU on the GPU in a graph)
        res["best"] = ({"path": "device_lru_graph", "tokens_per_s": res["device_lru_graph"]["tokens_per_s"],
                        "ms_per_step": round(ms_dev, 3), "frac_of_tier_bound": round(bound / ms_dev, 4)}
                       if ms_dev < res["ms_per_step"] else
                       {"path": "host_lru", "tokens_per_s": res["tokens_per_s"],
                        "ms_per_step": res["ms_per_step"], "frac_of_tier_bound": res["frac_of_tier_bound"]})
        out["T"][str(T)] = res
        if T == 8 and args.capacity_sweep:
            # hit rate and throughput against the slot budget (the LRU thrash cliff): from one
            # layer call's working set (NovaLLM's load-before / free-after-compute mode, "3.
            # Optimization #1": VRAM holds one layer's experts) up to every bundle resident
            sweep = {}
            steps = min(args.stream_steps, 64)
            ws_max = max(int(np.unique(trace[s_, l_]).size)
                         for s_ in range(steps) for l_ in range(cfg.layers))
            points = [("layer_working_set", ws_max * nb)]
            points += [(f"{gib}GiB", min(gib << 30, cfg.layers * cfg.E * nb))
                       for gib in (1, 2, 4, 8, 16)]
            for label, cap in points:
                try:
                    c2 = make(cap)
                    try:
                        torch.cuda.synchronize()
                        e0.record(stream)
                        run(c2, steps)
                        e1.record(stream)
                        stream.synchronize()
                        t_c = e0.elapsed_time(e1) / 1e3
                        st2 = moe.moe_expert_cache_stats(c2)
                        moe.moe_expert_cache_copy_time(c2)
                    finally:
                        moe.moe_expert_cache_destroy(c2)
                    sweep[label] = {
                        "slots": cap // nb, "steps": steps,
                        "hit_rate": round(st2["hits"] / max(1, st2["hits"] + st2["misses"]), 4),
                        "tokens_per_s": round(T * steps / t_c, 1)}
                except Exception as exc:          # a point that fails is reported, not fatal
                    sweep[label] = {"slots": cap // nb, "error": str(exc)[:200]}
            out["capacity_sweep_T8"] = sweep
        del xs, ids_dev, ws
    del store
    return out


def oracle_sample(cfg, T_sample, weights_cache):
    """One oracle layer forward on T_sample tokens; returns seconds."""
    from oracle import moe_ref
    xb = wl.tokens(cfg, T_sample, step=7)
    t = time.perf_counter()
    moe_ref.layer_forward(cfg, 0, xb, weights=lambda layer, e, sh=False: weights_cache(e, sh))
    return time.perf_counter() - t


def cpu_baseline(cfg, T_sample=16, reps=1):
    cache = {}

    def getw(e, sh):
        if (e, sh) not in cache:
            cache[(e, sh)] = wl.expert(cfg, 0, e, shared=sh)
        return cache[(e, sh)]
    for e in range(cfg.E):        # pre-generate (generation is not the oracle's work)
        getw(e, False)
    secs = [oracle_sample(cfg, T_sample, getw) for _ in range(reps)]
    s = float(np.median(secs))
    return {"value": round(T_sample / s, 3), "unit": "tokens/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"fp64 NumPy oracle, full layer on {T_sample} tokens of the same workload "
                      f"({s:.1f} s per sample)"}


def streamed_cpu_baseline(T=1, step=1):
    """The oracle on one sampled decode step of the expert-streamed stack: the LRU simulator's
    request for every layer and the oracle's pre-normalised stack of 16 layers (weights of the
    step's experts generated beforehand: generation is not the oracle's work)."""
    from oracle import bf16, moe_ref
    from oracle.lru_sim import LRUSim
    cfg = wl.STREAMED
    trace = wl.stream_trace(cfg, T, steps=step + 1)
    routed = {(l, int(e)): wl.expert(cfg, l, int(e))
              for l in range(cfg.layers) for e in np.unique(trace[step, l])}
    shared = {l: wl.expert(cfg, l, 0, shared=True) for l in range(cfg.layers)}
    getw = lambda layer, e, sh=False: shared[layer] if sh else routed[(layer, e)]  # noqa: E731
    import expert_dispatch_streaming_gb300 as moe
    nb = moe.moe_bundle_bytes(cfg.H, cfg.I, cfg.wdtype)
    t0 = time.perf_counter()
    sim = LRUSim(wl.STREAM_CACHE_BYTES // nb)
    x = bf16.decode(wl.stream_tokens(cfg, T, step))
    u = x
    for l in range(cfg.layers):
        sim.request(l, np.unique(trace[step, l]).tolist())
        r = moe_ref.layer_forward(cfg, l, bf16.to_bits(u), forced_ids=trace[step, l],
                                  weights=getw)
        x = bf16.round_rne(x + r["out"])
        u = moe_ref.rms_normalize(x, wl.STACK_NORM_EPS)
    sec = time.perf_counter() - t0
    return {"value": round(T / sec, 3), "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"one decode step (step {step}, T={T}) of the 16-layer stack: the LRU "
                      f"simulator's 16 requests and the fp64 oracle's layers ({sec:.1f} s)"}


def free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def launch_replicas(n, argv):
    """Runs this script as n ranks on this node (one process per GPU) through
    torch.distributed.run, rendezvous on 127.0.0.1; rank 0 prints the JSON line.  Returns the
    launcher's exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1",
           "--master-port", str(free_port()), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--workload", default="mixtral", choices=list(WORKLOADS))
    ap.add_argument("--experts", type=int, default=None,
                    help="override the routed expert count (smaller profiling cases)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--configs", default="qwen,deepseek,qwen_nvfp4",
                    help="other workloads measured over their batch sizes ('' = none)")
    ap.add_argument("--no-cpu", dest="cpu", action="store_false")
    ap.add_argument("--ffn-kernel", default="auto", choices=["auto", "stream", "tcgen05"])
    ap.add_argument("--pdl", action="store_true",
                    help="launch the layer's kernels with programmatic dependent launch")
    ap.add_argument("--no-streamed", dest="streamed", action="store_false")
    ap.add_argument("--no-graph", dest="graph", action="store_false")
    ap.add_argument("--stream-steps", type=int, default=wl.STREAM_STEPS)
    ap.add_argument("--no-capacity-sweep", dest="capacity_sweep", action="store_false")
    ap.add_argument("--copy-engine", dest="copy_kernel", action="store_false",
                    help="host-LRU miss copies by cudaMemcpyAsync (default: the fill kernel)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.T is None:
        args.T = max(WORKLOADS[args.workload].Ts)
    if args.experts:
        WORKLOADS[args.workload] = WORKLOADS[args.workload].with_(E=args.experts)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # N replicas, one process per GPU, as torchrun would start them
        sys.exit(launch_replicas(args.gpus, sys.argv[1:]))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = WORKLOADS[args.workload]

    if args.impl == "reference":
        # the reference arm is the CPU oracle, on rank 0 only
        if rank != 0:
            return
        cache = {}

        def getw(e, sh):
            if (e, sh) not in cache:
                cache[(e, sh)] = wl.expert(cfg, 0, e, shared=sh)
            return cache[(e, sh)]
        for e in range(cfg.E):
            getw(e, False)
        T_s = 8
        for _ in range(min(args.warmup, 1)):
            oracle_sample(cfg, T_s, getw)
        secs = [oracle_sample(cfg, T_s, getw) for _ in range(args.steps)]
        tot = float(np.sum(secs))
        v = T_s * args.steps / tot
        line = {"metric": f"MoE-layer tokens/s ({WORKLOAD_NAMES[args.workload]} layer)", "value": round(v, 3),
                "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1e3 * tot / args.steps, 2), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "impl": "reference",
                "config": {"workload": f"{WORKLOAD_NAMES[args.workload]} MoE layer forward, T={args.T}",
                           "sample_tokens_per_step": T_s},
                "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "kind": "oracle",
                                 "cores": len(os.sched_getaffinity(0)),
                                 "sample": f"{T_s} tokens of the T={args.T} workload per step"},
                "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if args.streamed and rank == 0:
        # the streamed decode pins every bundle of the stack (16.6 GB) in host memory: it runs
        # on rank 0 only (one replica's figure), not once per rank
        res["streamed_decode"] = run_streamed(args, local_rank)
        if world > 1:
            res["streamed_decode"]["ranks"] = "rank 0 only"
        if args.cpu:
            res["streamed_decode"]["cpu_baseline"] = streamed_cpu_baseline()
    if rank == 0:
        if args.cpu:
            res["cpu_baseline"] = cpu_baseline(cfg)
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
