#!/usr/bin/env python
"""Benchmark: µs per routed-expert MoE layer and weight-byte HBM GB/s on one GB300.

One step = one whole MoE layer on the device: route (expert-major row lists) -> gate/up rows
(+ SwiGLU + E4M3 quantiser) -> down rows -> combine, in one launch of libtfx_moe.so
(tfx_xp_moe_rows; --path separate times the four separate launches instead). Default workload: the DeepSeek-class 1-row decode layer (H 7168, I 2048, 256 experts,
top-8, E4M3 activations, MXFP4 weights), synthetic and seeded. Inputs are resident in HBM
before the timed region; each step uses the next of 4 packed layer copies (different expert
weights), so 4 x 187 MB of distinct weights rotate and no step finds the last one's in L2.

Prints one JSON line (rank 0). ``--impl reference`` times the CPU oracle instead (the only
reference this method has), on a bounded sample per step, scaled to µs per layer.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per MoE layer and weight-byte HBM GB/s vs peak at R=1..16 rows"
UNIT = "us per MoE layer"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def expert_bytes(H, I):
    """Codes + scales of one expert's gate, up and down projections."""
    return 3 * I * (H // 2) + 3 * I * (H // 32)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat each timed region of --steps steps until the repeats total this much device time")
    ap.add_argument("--no-sweep", action="store_true", help="time the named workload only")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode", choices=["tiny", "decode", "shared", "apart", "chunk"])
    ap.add_argument("--rows", type=int, default=None)
    ap.add_argument("--act", choices=["e4m3", "bf16"], default=None,
                    help="override the workload's activation format")
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--experts", type=int, default=None, help="override E (profiling aid: same widths, less memory)")
    ap.add_argument("--eager", action="store_true", help="launch each step from Python instead of graph replay")
    ap.add_argument("--path", choices=["fused", "separate", "chunk"], default=None,
                    help="fused: one launch per layer (tfx_xp_moe_rows); separate: route, gate/up, down, combine "
                         "(rows kernels); chunk: route, gate/up and down on the tensor cores, combine. Default: "
                         "chunk for the chunk workload, else fused")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value, world):
    """The largest of every rank's value (the job's time is its slowest rank's); one rank: the value."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def tensor_peak_fp8():
    """Dense E4M3 x E2M1 (kind::mxf8f6f4) tensor peak: the measured bf16 peak times the nominal
    fp8:bf16 ratio of 2 (4.5 vs 2.25 PFLOP/s dense)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return 2.0 * float(j["bf16_tflops"]), "measured bf16 x 2"
    return 2.0 * FALLBACK_BF16_TFLOPS, "fallback bf16 x 2"


def kernel_hash(files=("tfx_rows.cu", "tfx_rows.cuh", "tfx_common.cuh")):
    h = hashlib.sha256()
    for n in files:
        with open(os.path.join(ROOT, "moe_routed_expert_major_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(name, files=("tfx_rows.cu", "tfx_rows.cuh", "tfx_common.cuh")):
    """dram bytes (read + write) per launch of the timed kernel from the committed ncu summary
    profiles/<name>.md, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "%s.md" % name)
    if not os.path.exists(p):
        return None
    src = None
    traffic = None
    for line in open(p):
        if line.startswith("kernel_source_hash:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if src == kernel_hash(files) else None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [t.strip() for t in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, fl in rows for i, v in enumerate(fl) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------ ours

# Configurations of the metric beside the headline (decode, 1 row): rows on the same 8 experts
# (E4M3), rows routed apart (bf16), and the 4,096-row prompt chunk on the tensor cores.
SWEEP = ([("shared", R, "e4m3", "fused") for R in (2, 3, 4, 5, 8, 16)] +
         [("apart", R, "bf16", "fused") for R in (2, 4, 8, 16)] + [("chunk", 4096, "e4m3", "chunk")])


def layer_bytes(H, I, R, k, n_distinct, e4m3):
    """Algorithmic bytes of one layer: the distinct experts' weights once, the activations in, h
    written and read back, the expert outputs written and read back by the combine, the ids and
    weights, and y (bf16)."""
    P = R * k
    act_b = 1 if e4m3 else 2
    x_b = R * H * act_b + (R * (H // 32) if e4m3 else 0)
    h_b = P * I * act_b + (P * (I // 32) if e4m3 else 0)
    return n_distinct * expert_bytes(H, I) + x_b + 2 * h_b + 2 * P * H * 4 + P * 8 + R * H * 2


def layer_fmas(H, I, R, k):
    """Multiply-adds of the fp32 chains of one layer: one per weight per routed pair (gate, up
    and down: 3 H I)."""
    return R * k * 3 * H * I


def fma_peak(sms, mhz):
    """fp32-chain multiply-adds per second: SMs x 128 fma lanes per clock x the SM clock."""
    return sms * 128 * mhz * 1e6


class Runner:
    """One workload on the device: inputs resident in HBM, the step (one whole layer), CUDA
    graphs of its steps, and the timed repeats."""

    def __init__(self, ctx, workload, R, act, path):
        import numpy as np
        import torch

        import synth
        from moe_routed_expert_major_gb300 import tfx
        self.ctx = ctx
        tfx_ = tfx
        over = {"R": R}
        if act is not None:
            over["kind"] = synth.ACT_E4M3 if act == "e4m3" else synth.ACT_BF16
        if ctx["E_over"] is not None:
            over["E"] = ctx["E_over"]
        cfg = synth.workload(workload, **over)
        self.cfg = cfg
        H, I, E, k, R, kind = cfg["H"], cfg["I"], cfg["E"], cfg["k"], cfg["R"], cfg["kind"]
        dev = ctx["dev"]
        self.d = tfx_.dims(H, I, E, k)
        self.inp = inp = synth.make_inputs(cfg)
        if kind == synth.ACT_E4M3:
            self.x = torch.from_numpy(inp["x"]).to(dev)
            self.xs = torch.from_numpy(inp["sx"]).to(dev)
        else:
            self.x = torch.from_numpy(inp["x"].view(np.int16)).to(dev)
            self.xs = None
        self.ids = torch.from_numpy(inp["ids"]).to(dev)
        self.w = torch.from_numpy(inp["w"]).to(dev)
        self.path = path
        self.chunk = path == "chunk"
        self.fused = path == "fused" and R * k <= 256
        self.buf = tfx_.alloc_layer(R, H, I, E, k, kind, dev, chunk=self.chunk)
        self.n_distinct = len(set(int(e) for e in inp["ids"].ravel()))
        self.wbytes = self.n_distinct * expert_bytes(H, I)
        self.alg_bytes = layer_bytes(H, I, R, k, self.n_distinct, kind == synth.ACT_E4M3)
        self.fmas = layer_fmas(H, I, R, k)
        self.flops = 2.0 * self.fmas    # the same as flops, for the tensor-core path
        self.launches = 1 if self.fused else (5 if self.chunk else 4)
        self.tfx = tfx_

    def step(self, i, ev=None, st=None):
        tfx, d, R, kind, buf = self.tfx, self.d, self.cfg["R"], self.cfg["kind"], self.buf
        pk = self.ctx["packed"][i % len(self.ctx["packed"])]
        x, xs, ids, w = self.x, self.xs, self.ids, self.w
        if self.fused:
            if ev is not None:
                ev[0].record(st)
            tfx.tfx_xp_moe_rows(d, R, kind, pk, x, xs, ids, w, buf["route"], buf["h"], buf["h_scale"], buf["out"],
                                buf["y"], buf["scratch"], buf["status"])
            if ev is not None:
                ev[1].record(st)
            return
        tfx.tfx_xp_route(d, R, ids, buf["route"], buf["status"])
        if ev is not None:
            ev[0].record(st)
        if self.chunk:
            tfx.tfx_xp_upc_chunk(d, R, kind, pk, x, xs, buf["route"], buf["h"], buf["h_scale"], buf["chunk_ws"],
                                 buf["status"])
        else:
            tfx.tfx_xp_upc_rows(d, R, kind, pk, x, xs, buf["route"], buf["h"], buf["h_scale"], buf["status"])
        if ev is not None:
            ev[1].record(st)
        if self.chunk:
            tfx.tfx_xp_down_chunk(d, R, kind, pk, buf["h"], buf["h_scale"], buf["route"], buf["out"], buf["status"])
        else:
            tfx.tfx_xp_down_rows(d, R, kind, pk, buf["h"], buf["h_scale"], buf["route"], buf["out"], buf["status"])
        tfx.tfx_xp_combine(d, R, buf["out"], w, buf["y"])

    def warm(self, W):
        import torch
        for i in range(max(3, W)):
            self.step(i)
        torch.cuda.synchronize()
        st = int(self.buf["status"].item())
        if st != 0:
            raise RuntimeError("device status %d during warm-up (%s)" % (st, self.cfg["name"]))

    def capture(self, n, events=None):
        """A CUDA graph of steps 0..n-1 (cycling over the layer copies), or None."""
        import torch
        if n <= 0:
            return None
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(self.ctx["stream"])
        with torch.cuda.stream(cs):
            with torch.cuda.graph(g, stream=cs):
                for i in range(n):
                    self.step(i, None if events is None else events[i], torch.cuda.current_stream())
        torch.cuda.synchronize()
        return g

    def timed(self, K, min_total_s, world, eager=False, clock_index=0):
        """Exactly K steps per timed region, the region repeated (barrier and synchronisation on
        both sides of each) until the repeats add up to min_total_s of device time; returns the
        median repeat and the clock record of the whole loop."""
        import torch
        G = 8 * len(self.ctx["packed"])
        graph = rem = None
        if not eager:
            try:
                graph = self.capture(min(G, K))
                rem = self.capture(K % min(G, K)) if K > G else None
                for _ in range(2):
                    graph.replay()
                    if rem is not None:
                        rem.replay()
                torch.cuda.synchronize()
            except (TypeError, RuntimeError) as ex:
                sys.stderr.write("graph capture unavailable (%s); timing eager launches\n" % ex)
                graph = rem = None
        full = K // min(G, K) if graph is not None else 0
        stream = self.ctx["stream"]
        clk = Clocks(clock_index)
        clk.start()
        time.sleep(0.25)
        times = []
        total = 0.0
        while (total < 1000.0 * min_total_s or len(times) < 3) and len(times) < 100000:
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize()
            t0.record(stream)
            if graph is not None:
                for _ in range(full):
                    graph.replay()
                if rem is not None:
                    rem.replay()
            else:
                for i in range(K):
                    self.step(i)
            t1.record(stream)
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            ms = t0.elapsed_time(t1)
            times.append(ms)
            total += ms
        clocks = clk.stop()
        med = statistics.median(times)
        return {"ms": med, "repeats": len(times), "clocks": clocks,
                "launch": ("cuda graph replay: %d x a %d-step graph%s" % (full, min(G, K), (
                    " + a %d-step graph" % (K % min(G, K))) if rem is not None else "")) if graph is not None
                else "eager"}

    def kernel_ms(self, K):
        """Average duration of the roofline kernel (the fused launch, or gate/up) by CUDA
        events captured around it in a graph of the same steps, replayed after the timed region."""
        import torch
        G = min(8 * len(self.ctx["packed"]), K)
        kev = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in range(G)]
        try:
            g = self.capture(G, kev)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            return statistics.fmean(a.elapsed_time(b) for a, b in kev), "events around the kernel in a graph replay"
        except (TypeError, RuntimeError):
            kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(G)]
            for i in range(G):
                self.step(i, kev[i], self.ctx["stream"])
            torch.cuda.synchronize()
            return statistics.fmean(a.elapsed_time(b) for a, b in kev), "events around eager launches"


def bound_of(run, us, hbm, sm_mhz, sms):
    """The binding roofline of one measured layer: HBM on its algorithmic bytes, the fp32-chain
    fma rate (rows path), or the tensor cores (chunk path), whichever takes longest."""
    t_hbm = run.alg_bytes / (hbm * 1e9)
    out = {"hbm_us": round(1e6 * t_hbm, 2), "hbm_frac": round(1e6 * t_hbm / us, 4)}
    if run.chunk:
        tpeak, tsrc = tensor_peak_fp8()
        t_t = run.flops / (tpeak * 1e12)
        out.update({"tensor_us": round(1e6 * t_t, 2), "tensor_peak_tflops": tpeak, "tensor_peak_source": tsrc,
                    "tensor_frac": round(1e6 * t_t / us, 4)})
        bound, t = ("tensor", t_t) if t_t > t_hbm else ("hbm", t_hbm)
    else:
        fpk = fma_peak(sms, sm_mhz)
        t_a = run.fmas / fpk
        out.update({"alu_us": round(1e6 * t_a, 2), "alu_frac": round(1e6 * t_a / us, 4),
                    "alu_peak": "%d SMs x 128 fp32 fma/clk x %.0f MHz (median SM clock sampled under load) = %.1f T fma/s"
                                % (sms, sm_mhz, fpk / 1e12)})
        bound, t = ("alu", t_a) if t_a > t_hbm else ("hbm", t_hbm)
    out["bound"] = bound
    out["frac"] = round(1e6 * t / us, 4)
    return out


def run_ours(args):
    import numpy as np
    import torch

    import synth
    from moe_routed_expert_major_gb300 import build as _build
    from moe_routed_expert_major_gb300 import tfx

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = "cuda:%d" % local
    _build.build()
    tfx.load()
    sms = torch.cuda.get_device_properties(local).multi_processor_count

    # packed weight copies, shared by every workload (same widths): each step uses the next one
    E = args.experts if args.experts is not None else synth.WORKLOADS["decode"]["E"]
    H, I = synth.WORKLOADS["decode"]["H"], synth.WORKLOADS["decode"]["I"]
    L = max(1, args.layers)
    d0 = tfx.dims(H, I, E, synth.WORKLOADS["decode"]["k"])
    packed = []
    for l in range(L):
        dw = synth.weights_torch(E, H, I, synth.workload(args.workload)["seed"] + 7919 * l, dev)
        p = torch.empty(tfx.tfx_xp_packed_bytes(d0), dtype=torch.uint8, device=dev)
        tfx.tfx_xp_pack(d0, dw, p)
        packed.append(p)
        del dw
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    ctx = {"dev": dev, "packed": packed, "stream": torch.cuda.current_stream(), "E_over": args.experts}

    path = args.path or ("chunk" if args.workload == "chunk" else "fused")
    main = Runner(ctx, args.workload, args.rows if args.rows is not None else synth.WORKLOADS[args.workload]["R"],
                  args.act, path)
    cfg = main.cfg
    H, I, E, k, R, kind = cfg["H"], cfg["I"], cfg["E"], cfg["k"], cfg["R"], cfg["kind"]
    d = main.d
    K = max(1, args.steps)
    main.warm(args.warmup)

    # ---------------------------------------------------------------- timed region
    tm = main.timed(K, args.min_seconds, world, eager=args.eager, clock_index=local)
    elapsed_ms = max_over_ranks(tm["ms"], world)
    clocks = tm["clocks"]
    status = int(main.buf["status"].item())
    kern_ms, kern_how = main.kernel_ms(K)
    if main.fused and not args.eager:
        # one launch per step: the step time bounds the launch's duration from above, and the
        # event brackets of the replay add their own delay
        kern_ms = min(kern_ms, elapsed_ms / K)

    # per-kernel breakdown of the separate launches (diagnostic, outside the timed region)
    names = ["route", "upc_chunk", "down_chunk", "combine"] if main.chunk else ["route", "upc_rows", "down_rows",
                                                                               "combine"]
    buf, stream = main.buf, ctx["stream"]
    nb = 200
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(nb)]
    for i in range(nb):
        pk = packed[i % L]
        e = evs[i]
        e[0].record(stream)
        tfx.tfx_xp_route(d, R, main.ids, buf["route"], buf["status"])
        e[1].record(stream)
        if main.chunk:
            tfx.tfx_xp_upc_chunk(d, R, kind, pk, main.x, main.xs, buf["route"], buf["h"], buf["h_scale"],
                                 buf["chunk_ws"], buf["status"])
        else:
            tfx.tfx_xp_upc_rows(d, R, kind, pk, main.x, main.xs, buf["route"], buf["h"], buf["h_scale"], buf["status"])
        e[2].record(stream)
        if main.chunk:
            tfx.tfx_xp_down_chunk(d, R, kind, pk, buf["h"], buf["h_scale"], buf["route"], buf["out"], buf["status"])
        else:
            tfx.tfx_xp_down_rows(d, R, kind, pk, buf["h"], buf["h_scale"], buf["route"], buf["out"], buf["status"])
        e[3].record(stream)
        tfx.tfx_xp_combine(d, R, buf["out"], main.w, buf["y"])
        e[4].record(stream)
    torch.cuda.synchronize()
    breakdown = {n: 1000.0 * statistics.median(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(nb))
                 for j, n in enumerate(names)}
    # the device router (top-k from logits) on logits of the same shape, for reference
    lg = torch.randn((R, E), generator=torch.Generator().manual_seed(1), dtype=torch.float32).to(dev)
    rids = torch.empty((R, k), dtype=torch.int32, device=dev)
    rw = torch.empty((R, k), dtype=torch.float32, device=dev)
    rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    for a, b in rev:
        a.record(stream)
        tfx.tfx_xp_router(lg, k, rids, rw)
        b.record(stream)
    torch.cuda.synchronize()
    breakdown["router (logits -> ids, w; not in the step)"] = 1000.0 * statistics.median(a.elapsed_time(b) for a, b in rev)
    if E % 8 == 0 and E >= 16 and k <= 4 * (E // 8):  # group-limited sigmoid routing: 8 groups, 4 kept
        rb = (0.1 * torch.randn(E, generator=torch.Generator().manual_seed(2), dtype=torch.float32)).to(dev)
        for a, b in rev:
            a.record(stream)
            tfx.tfx_xp_router_grouped(lg, k, 8, 4, rids, rw, bias=rb, scale=2.5)
            b.record(stream)
        torch.cuda.synchronize()
        breakdown["grouped router (8 groups, 4 kept; not in the step)"] = 1000.0 * statistics.median(
            a.elapsed_time(b) for a, b in rev)

    # ---------------------------------------------------------------- end to end (host buffers)
    e2e = None
    if not args.no_e2e:
        inp = main.inp
        # the step's inputs travel in one copy: x, its scales, ids and weights packed into one
        # pinned host buffer (256-byte aligned parts) and read on the device through views
        parts = [("x", np.ascontiguousarray(inp["x"] if kind == synth.ACT_E4M3 else inp["x"].view(np.int16))),
                 ("xs", np.ascontiguousarray(inp["sx"]) if kind == synth.ACT_E4M3 else None),
                 ("ids", np.ascontiguousarray(inp["ids"])), ("w", np.ascontiguousarray(inp["w"]))]
        offs, tot = {}, 0
        if main.fused:
            # the host-buffer entry's own block layout: it then moves the four parts in one copy
            lay, tot = tfx.tfx_xp_moe_rows_host_layout(d, R, kind)
            offs = {"x": lay[0], "xs": lay[1], "ids": lay[2], "w": lay[3]}
        else:
            for name, a in parts:
                if a is not None:
                    offs[name] = tot
                    tot = (tot + a.nbytes + 255) // 256 * 256
        hin = torch.zeros(tot, dtype=torch.uint8).pin_memory()
        din = torch.empty(tot, dtype=torch.uint8, device=dev)
        dv, hv = {}, {}
        for name, a in parts:
            if a is None:
                continue
            t = torch.from_numpy(a.reshape(-1).view(np.uint8))
            hin[offs[name]:offs[name] + a.nbytes].copy_(t)
            tdt = {np.dtype(np.uint8): torch.uint8, np.dtype(np.int16): torch.int16, np.dtype(np.int32): torch.int32,
                   np.dtype(np.float32): torch.float32}[a.dtype]
            dv[name] = din[offs[name]:offs[name] + a.nbytes].view(tdt).view(a.shape)
            hv[name] = hin[offs[name]:offs[name] + a.nbytes].view(tdt).view(a.shape)
        dx, dxs, dids, dwt = dv["x"], dv.get("xs"), dv["ids"], dv["w"]
        if main.fused:
            host_ws = torch.zeros(tfx.tfx_xp_moe_rows_host_ws_bytes(d, R, kind), dtype=torch.uint8, device=dev)
        hy = torch.empty(buf["y"].shape, dtype=buf["y"].dtype).pin_memory()
        h2d = tot
        d2h = hy.numel() * hy.element_size()
        Ke = max(K, min(2000, int(0.5e6 / max(1.0, 1000.0 * elapsed_ms / K)))) if not main.chunk else min(K, 20)

        def e2e_step(i):
            pk = packed[i % L]
            if main.fused:
                # one call: the inputs' copy, the layer and the copy of y, queued on the stream
                tfx.tfx_xp_moe_rows_host(d, R, kind, pk, hv["x"], hv.get("xs"), hv["ids"], hv["w"], hy,
                                         buf["status"], host_ws)
                return
            din.copy_(hin, non_blocking=True)
            if main.chunk:
                tfx.tfx_xp_route(d, R, dids, buf["route"], buf["status"])
                tfx.tfx_xp_upc_chunk(d, R, kind, pk, dx, dxs, buf["route"], buf["h"], buf["h_scale"], buf["chunk_ws"],
                                     buf["status"])
                tfx.tfx_xp_down_chunk(d, R, kind, pk, buf["h"], buf["h_scale"], buf["route"], buf["out"],
                                      buf["status"])
                tfx.tfx_xp_combine(d, R, buf["out"], dwt, buf["y"])
            else:
                tfx.tfx_xp_route(d, R, dids, buf["route"], buf["status"])
                tfx.tfx_xp_upc_rows(d, R, kind, pk, dx, dxs, buf["route"], buf["h"], buf["h_scale"], buf["status"])
                tfx.tfx_xp_down_rows(d, R, kind, pk, buf["h"], buf["h_scale"], buf["route"], buf["out"], buf["status"])
                tfx.tfx_xp_combine(d, R, buf["out"], dwt, buf["y"])
            hy.copy_(buf["y"], non_blocking=True)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(Ke):
            e2e_step(i)
        b.record(stream)
        torch.cuda.synchronize()
        e2e = {"value": round(1000.0 * a.elapsed_time(b) / Ke, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": Ke,
               "how": ("the public API's host-buffer entry (tfx_xp_moe_rows_host through the ctypes binding), one "
                       "call from Python each step: the layer reads the step's inputs in place from pinned host "
                       "memory (h2d bytes: those inputs) and its combine stores y into pinned host memory (d2h "
                       "bytes: y), queued on one stream" if main.fused else
                       "the public API (ctypes binding of libtfx_moe.so) launched from Python each step: one pinned "
                       "H2D copy of the step's inputs, the layer, one D2H copy of y, back to back on one stream")}

    # ---------------------------------------------------------------- the rest of the metric
    hbm, hbm_src = peaks()
    sm_mhz = clocks.get("sm_mhz") or 2070.0
    sweep = []
    if not args.no_sweep:
        for wl, Rs, act, pth in SWEEP:
            if (wl, Rs) == (args.workload, R):
                continue
            try:
                run = Runner(ctx, wl, Rs, act, pth)
                run.warm(args.warmup)
                t = run.timed(K, args.min_seconds, world, eager=args.eager, clock_index=local)
                ms = max_over_ranks(t["ms"], world)
                us = 1000.0 * ms / K
                mhz = t["clocks"].get("sm_mhz") or sm_mhz
                ent = {"workload": wl, "rows": Rs, "act": act, "path": "fused one-launch layer" if run.fused else (
                    "route + gate/up chunk + down chunk (tensor cores) + combine" if run.chunk else "four launches"),
                       "distinct_experts": run.n_distinct, "us_per_layer": round(us, 3),
                       "weight_gbs": round(run.wbytes / (us * 1e-6) / 1e9, 1),
                       "weight_gbs_frac_of_peak": round(run.wbytes / (us * 1e-6) / 1e9 / hbm, 4),
                       "algorithmic_bytes": int(run.alg_bytes), "fma_per_layer": int(run.fmas),
                       "steps": K, "repeats": t["repeats"], "launch": t["launch"], "clocks": t["clocks"],
                       "status": int(run.buf["status"].item())}
                ent.update(bound_of(run, us, hbm, mhz, sms))
                sweep.append(ent)
                del run
                torch.cuda.empty_cache()
            except (RuntimeError, torch.cuda.OutOfMemoryError) as ex:
                sweep.append({"workload": wl, "rows": Rs, "act": act, "error": str(ex)[:200]})

    # ---------------------------------------------------------------- CPU oracle baseline
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_full_layer(cfg, main.inp, packed_seed=cfg["seed"], dev=dev, seconds=args.cpu_seconds,
                                      sample_rows=8 if R > 64 else None)

    us_per_layer = 1000.0 * elapsed_ms / K
    kb = bound_of(main, us_per_layer, hbm, sm_mhz, sms)
    if main.fused:
        kern_name = "moe_rows (route+gate/up+down+combine, one launch)"
        kern_alg = main.alg_bytes
    elif main.chunk:
        kern_name = "upc_chunk (activation rows into pair order + gate/up chunk kernel, tcgen05 mxf8f6f4)"
        kern_alg = main.n_distinct * 2 * I * (H // 2 + H // 32)
    else:
        kern_name = "upc_rows"
        kern_alg = main.n_distinct * 2 * I * (H // 2 + H // 32)
    achieved = kern_alg / (kern_ms * 1e-3) / 1e9
    tensor = None
    if main.chunk:
        flops = 2.0 * R * k * 2 * I * H
        tpeak, tsrc = tensor_peak_fp8()
        tensor = {"achieved_tflops": round(flops / (kern_ms * 1e-3) / 1e12, 1), "peak_tflops": tpeak,
                  "peak_source": tsrc, "frac": round(flops / (kern_ms * 1e-3) / 1e12 / tpeak, 4),
                  "flops_per_launch": flops}
    rbound = "hbm" if not main.fused else ("alu" if kb["bound"] == "alu" else "hbm")
    roof = {"kernel": kern_name, "bound": rbound, "achieved": round(achieved, 1), "peak": hbm, "peak_source": hbm_src,
            "unit": "GB/s", "frac": round(achieved / hbm, 4), "algorithmic_bytes_per_launch": int(kern_alg),
            "avg_launch_us": round(1000 * kern_ms, 3), "launch_timing": kern_how,
            "traffic": (profiled_traffic("upc_chunk_%s_%drow" % (args.workload, R), ("tfx_chunk.cu", "tfx_common.cuh"))
                        if main.chunk else profiled_traffic("%s_rows_%s_%drow" % ("fused" if main.fused else "upc",
                                                                                  args.workload, R))),
            "tensor": tensor}
    if rbound == "alu":
        # the fp32 chains' multiply-adds bind: the fraction is of the fma rate, stated beside
        roof.update({"achieved": round(main.fmas / (kern_ms * 1e-3) / 1e12, 3), "unit": "T fma/s",
                     "peak": round(fma_peak(sms, sm_mhz) / 1e12, 3), "peak_source": kb["alu_peak"],
                     "frac": round(main.fmas / (kern_ms * 1e-3) / fma_peak(sms, sm_mhz), 4)})
    line = {
        "metric": METRIC, "value": round(us_per_layer, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / K, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "%s: H %d, I %d, E %d, top-%d, R %d, %s activations, MXFP4 weights" % (
            args.workload, H, I, E, k, R, "E4M3" if kind == synth.ACT_E4M3 else "bf16"),
            "rows": R, "distinct_experts": main.n_distinct, "weight_bytes_per_layer": main.wbytes,
            "layers_rotated": L, "l2": "inputs larger than L2: %d packed layer copies rotate (%.0f MB of distinct "
                                        "weights per rotation vs 129 MB L2)" % (L, L * main.wbytes / 1e6),
            "path": "fused one-launch layer" if main.fused else (
                "route + gate/up chunk + down chunk (tensor cores) + combine" if main.chunk
                else "route + gate/up + down + combine"),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "timing": "exactly %d steps per timed region (%s), the region repeated %d times (barrier and "
                      "synchronisation around each) for %.2f s of device time; value = median repeat / %d"
                      % (K, tm["launch"], tm["repeats"], tm["repeats"] * tm["ms"] / 1000.0, K)},
        "weight_gbs": round(main.wbytes / (us_per_layer * 1e-6) / 1e9, 1),
        "weight_gbs_frac_of_peak": round(main.wbytes / (us_per_layer * 1e-6) / 1e9 / hbm, 4),
        "bound": kb,
        "separate_kernels_us": {n: round(v, 3) for n, v in breakdown.items()},
        "roofline": roof,
        "sweep": sweep,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": main.launches * K, "gpu_launches_per_step": main.launches,
        "timed_repeats": tm["repeats"], "clocks": clocks, "status": status, "launch": tm["launch"],
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def _host_layer(cfg, inp, dev, rows=None):
    import synth
    dw = synth.weights_torch(cfg["E"], cfg["H"], cfg["I"], cfg["seed"], dev)
    ids = inp["ids"] if rows is None else inp["ids"][rows]
    experts = sorted(set(int(e) for e in ids.ravel() if 0 <= int(e) < cfg["E"]))
    lay = dict(H=cfg["H"], I=cfg["I"], E=cfg["E"], k=cfg["k"], kind=cfg["kind"])
    for n, t in dw.items():
        full = {}
        for e in experts:
            full[e] = t[e].cpu().numpy()
        lay[n] = _ExpertDict(full)
    lay.update(inp)
    return lay


class _ExpertDict:
    def __init__(self, d):
        self.d = d

    def __getitem__(self, e):
        return self.d[int(e)]


def cpu_baseline_full_layer(cfg, inp, packed_seed, dev, seconds, sample_rows=None):
    """The oracle (fp32-chain mode, as it stands) on whole layers of the same workload, or, for
    a large layer, on its first `sample_rows` rows, scaled to the layer by the row count."""
    import oracle
    R, k = inp["ids"].shape
    rows = None if sample_rows is None else list(range(min(sample_rows, R)))
    lay = _host_layer(cfg, inp, dev, rows=rows)
    threads = min(os.cpu_count() or 1, R * k if rows is None else len(rows) * k)
    oracle.layer_chain(lay, threads=threads, rows=[0])  # load and warm the library
    n = 0
    t = time.perf_counter()
    while True:
        oracle.layer_chain(lay, threads=threads, rows=rows)
        n += 1
        el = time.perf_counter() - t
        if el >= seconds or n >= 50:
            break
    per = el / n
    if rows is None:
        return {"value": round(1e6 * per, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
                "sample": "%d whole %s layer(s) (route, %d gate/up + SwiGLU + quantiser + down pairs, combine), "
                          "fp32-chain mode, pairs spread over %d host threads" % (n, cfg["name"], R * k, threads)}
    return {"value": round(1e6 * per * R / len(rows), 1), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "rows 0-%d of the %s layer (%d pairs: gate/up + SwiGLU + quantiser + down, combine) %d "
                      "time(s), fp32-chain mode over %d host threads, scaled by %d/%d rows" % (
                          len(rows) - 1, cfg["name"], len(rows) * k, n, threads, R, len(rows))}


# ------------------------------------------------------------------------------- reference

def run_reference(args):
    """The CPU oracle timed on the host cores: each step computes a bounded sample of the
    layer (gate/up for 8 outputs and down for 16 outputs of one (row, slot) pair, rotating
    over the pairs), and the time is scaled to a whole layer by the share of multiply-adds."""
    import numpy as np
    import torch

    import oracle
    import synth

    rank, world, _ = dist_env()
    if rank != 0:
        return
    over = {} if args.rows is None else {"R": args.rows}
    if args.act is not None:
        over["kind"] = synth.ACT_E4M3 if args.act == "e4m3" else synth.ACT_BF16
    cfg = synth.workload(args.workload, **over)
    H, I, k, R, kind = cfg["H"], cfg["I"], cfg["k"], cfg["R"], cfg["kind"]
    inp = synth.make_inputs(cfg)
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    lay = _host_layer(cfg, inp, dev)
    rt = oracle.route(inp["ids"], cfg["E"])
    P = len(rt["pair_row"])
    # unscaled activation values and group scales, decoded by the oracle's own element formats
    e4 = np.array([oracle.e4m3_value(c) for c in range(256)], np.float32)

    def act(r):
        if kind == synth.ACT_E4M3:
            xc = e4[inp["x"][r]]
            xs = np.array([oracle.ue8m0_value(int(s)) for s in inp["sx"][r]], np.float32)
        else:
            xc = oracle.bf16_to_f32(inp["x"][r])
            xs = np.ones(H // 32, np.float32)
        return np.ascontiguousarray(xc), xs

    acts = {r: act(r) for r in set(int(r) for r in rt["pair_row"])}
    hc = np.ones(I, np.float32)
    hsc = np.ones(I // 32, np.float32)
    NG, ND = 8, 16

    def one(i):
        p = i % P
        r, j = int(rt["pair_row"][p]), int(rt["pair_slot"][p])
        e = int(inp["ids"][r, j])
        xc, xs = acts[r]
        for q in range(NG):
            n = (i * NG + q) % I
            oracle.chain_dot(lay["wg"][e][n], lay["sg"][e][n], xc, xs)
            oracle.chain_dot(lay["wu"][e][n], lay["su"][e][n], xc, xs)
        for q in range(ND):
            m = (i * ND + q) % H
            oracle.chain_dot(lay["wd"][e][m], lay["sd"][e][m], hc, hsc)

    for i in range(args.warmup):
        one(i)
    t = time.perf_counter()
    for i in range(args.steps):
        one(i)
    el = time.perf_counter() - t
    frac = (NG * 2 * H + ND * I) / float(P * 3 * H * I)
    us = 1e6 * (el / args.steps) / frac
    line = {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * el / args.steps, 4),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "%s: H %d, I %d, E %d, top-%d, R %d, %s activations, MXFP4 weights" % (
                args.workload, H, I, cfg["E"], k, R, "E4M3" if kind == synth.ACT_E4M3 else "bf16"), "rows": R,
                "step": "a bounded sample of the layer, not a whole layer: gate/up for %d outputs and down for %d "
                        "outputs of one routed pair; ms_per_step is that sample's time and value scales it to "
                        "a whole layer by multiply-adds" % (NG, ND)},
            "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "per step: gate/up for %d outputs and down for %d outputs of one routed pair "
                                       "(fp32-chain mode, one thread), scaled by multiply-adds to a whole layer of "
                                       "%d pairs" % (NG, ND, P)},
            "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
