#!/usr/bin/env python
"""Benchmark of the routed MoE FFN layer over block-quantized experts.

One step = one pass of the whole layer (router, bucketing, grouped gate/up
with fused SwiGLU, grouped down, combine) through each of `--layers` stacked
independent layers (different seeds, so the selected experts' weights stream
from HBM rather than L2), replayed as one CUDA graph. Inputs are seeded
synthetic data; the weights are written on the device by the seeded filler.

Prints one JSON line. The headline workload (``--config``, default the
2048-token mixed-tier prefill chunk, the largest single-GPU configuration) is
timed over exactly ``--steps`` steps. `value` is MoE-layer tokens/s
(token-layers per second, i.e. T / per-layer time, summed over ranks); `e2e`
is the same metric through the public API with pinned host buffers copied in
and out every layer (the copies of one layer overlapping the computation of
its neighbours, on three streams, one step replayed as a CUDA graph); `roofline` is the dominant kernel's algorithmic bytes
per launch over its event-timed duration against the measured HBM copy
bandwidth; `cpu_baseline` is the fp64 oracle on the host cores (all cores,
and single-threaded in `cpu_baseline.single_thread`) on a bounded sample of
the same workload. `per_config` carries the same measurements for the decode
workloads (1-token, 16-row, 6-row mixed-tier), each timed for at least
``--min-seconds``.

--impl reference runs the oracle as the reference arm (there is no runnable
reference implementation: the source pages ship no code).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s; expert-weight HBM GB/s and % of GB300 roofline"
UNIT = "tokens/s"
KERNELS_PER_LAYER = {1: 4,   # GEMV: route, gate/up, down, combine (+ bucketing)
                     2: 6,   # tensor: route, prep, gate/up GEMM, h conversion, down GEMM, combine (+ bucketing)
                     3: 1}   # fused decode: one kernel (its own routing and bucketing)


def launches_per_layer(path: int, pairs: int) -> int:
    """Our kernel launches per layer: the bucketing is one kernel up to 2,048
    (token, slot) pairs and three (histograms, scan, scatter) above."""
    if path == 3:
        return 1
    return KERNELS_PER_LAYER[path] + (1 if pairs <= 2048 else 3)


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="prefill2048", help="tiny|decode1|decode16|mtp6|prefill2048")
    p.add_argument("--per-config", default="decode1,decode16,mtp6",
                   help="comma-separated workloads measured after the headline ('none': skip)")
    p.add_argument("--min-seconds", type=float, default=1.0, help="timed region of each per-config workload")
    p.add_argument("--layers", type=int, default=48)
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--cpu-budget", type=float, default=12.0,
                   help="seconds of oracle work for each cpu_baseline leg (single thread, all cores)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--path", type=int, default=0, help="0 auto, 1 grouped GEMV, 2 tensor cores, 3 fused decode")
    return p.parse_args(argv)


# ----------------------------------------------------------------------------
# oracle worker (host CPU baseline / reference arm); runs in a subprocess
# started before any CUDA work. mode "serial": the per-pair evaluation with
# BLAS on one thread; mode "pool": the expert-by-expert evaluation over a
# spawned process pool of every host core (one BLAS thread per worker).
# ----------------------------------------------------------------------------
def oracle_worker(spec: dict) -> dict:
    import multiprocessing as mp

    import numpy as np
    import synth
    from oracle import ffn as offn
    from oracle import router as orouter

    cfg = synth.CONFIGS[spec["config"]]
    budget = float(spec["budget_s"])
    n_tok = min(cfg.tokens, int(spec.get("tokens_per_sample") or cfg.tokens))
    pool = mp.get_context("spawn").Pool(os.cpu_count() or 1) if spec["mode"] == "pool" else None
    cores = (os.cpu_count() or 1) if pool else 1
    # Untimed: the layer's inputs, routing and the routed experts' bytes (the
    # oracle's input); timed: the oracle's arithmetic (decode + routed FFN).
    t_work, token_layers, layer = 0.0, 0, 0
    steps = []
    n_samples = int(spec.get("samples") or 0)
    while (t_work < budget if not n_samples else layer < n_samples) and layer < 1000:
        L = synth.make_layer(cfg, layer % 48, with_weights=False)
        lazy = synth.LazyExperts(cfg, L.seed, L.fmts)
        # a different window of tokens per layer sample
        t0_tok = (layer * 97) % max(1, cfg.tokens - n_tok + 1)
        toks = list(range(t0_tok, t0_tok + n_tok))
        if pool is None:
            ids, _, _ = orouter.route_topk(L.logits, cfg.k)
            for e in list(np.unique(ids[toks])) + list(range(cfg.n_experts, cfg.n_entries)):
                lazy[int(e)]
            t0 = time.perf_counter()
            offn.moe_ffn(lazy, L.x_bf16, L.logits, cfg.k, tokens=toks, gate_formats=lazy.gate_formats(),
                         n_shared=cfg.n_shared)
        else:
            t0 = time.perf_counter()
            offn.moe_ffn_by_expert(lazy, L.x_bf16, L.logits, cfg.k, tokens=toks,
                                   gate_formats=lazy.gate_formats(), map_fn=pool.map, n_shared=cfg.n_shared)
        dt = time.perf_counter() - t0
        steps.append(dt)
        t_work += dt
        token_layers += len(toks)
        layer += 1
    if pool is not None:
        pool.close()
        pool.join()
    return {"value": token_layers / t_work, "token_layers": token_layers, "seconds": t_work, "layers": layer,
            "tokens_per_layer": n_tok, "cores": cores, "step_seconds": steps}


def run_oracle_subprocess(spec: dict) -> dict:
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = "1"
    env["MOE_BENCH_ORACLE_WORKER"] = json.dumps(spec)
    r = subprocess.run([sys.executable, os.path.abspath(__file__)], env=env, capture_output=True, text=True,
                       timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"oracle worker failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


# tokens per oracle sample, a window of the layer's tokens: each token costs
# about ten expert decodes (plus ~40 MFLOP of fp64 per pair), so one thread
# takes 2 tokens per sample and the pool 48 (whole layers up to 16 rows)
def oracle_sample_tokens(cfg, mode: str) -> int:
    return min(cfg.tokens, 2 if mode == "serial" else 48)


def cpu_baseline(config: str, budget: float) -> dict:
    import synth
    cfg = synth.CONFIGS[config]
    legs = {}
    for mode in ("pool", "serial"):
        n_tok = oracle_sample_tokens(cfg, mode)
        res = run_oracle_subprocess({"config": config, "budget_s": budget, "mode": mode,
                                     "tokens_per_sample": n_tok})
        what = ("expert by expert over a spawned pool, one BLAS thread per process" if mode == "pool"
                else "pair by pair, BLAS limited to 1 thread")
        legs[mode] = {"value": res["value"], "unit": UNIT, "cores": res["cores"], "kind": "oracle",
                      "sample": f"{config}: {res['layers']} layer samples of {res['tokens_per_layer']} token(s) "
                                f"(all their routed experts), {res['seconds']:.1f} s of fp64 oracle arithmetic, "
                                f"{what}"}
    line = dict(legs["pool"])
    line["single_thread"] = legs["serial"]
    return line


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t_start - 0.1 <= r[0] <= self.t_end + 0.1]
        window = "timed"
        if not inside:
            # timed region shorter than the sampling period: nearest samples
            inside = sorted(rows, key=lambda r: abs(r[0] - (self.t_start + self.t_end) / 2))[:3]
            window = "adjacent"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ----------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_traffic(kernel: str, config: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel (same hash of the files it lists); else
    None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(f"{kernel}:{config}")
    if not ent:
        return None
    if ent.get("source_sha256") != source_hash(ent.get("sources", [])):
        return None
    return ent.get("dram_bytes_per_launch")


def source_hash(files) -> str:
    """sha256 (16 hex digits) over the named files of the package's csrc/."""
    h = hashlib.sha256()
    cs = os.path.join(ROOT, "quantized_moe_expert_route_gb300", "csrc")
    for f in sorted(files):
        with open(os.path.join(cs, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def allreduce_max(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------
def run_reference(args, world, rank):
    if rank != 0:
        return None
    import synth
    cfg = synth.CONFIGS[args.config]
    n_tok = cfg.tokens if cfg.tokens <= 16 else 16
    res = run_oracle_subprocess({"config": args.config, "budget_s": 0.0, "mode": "pool",
                                 "tokens_per_sample": n_tok, "samples": args.warmup + args.steps})
    timed = res["step_seconds"][args.warmup:]
    secs = sum(timed)
    v = n_tok * len(timed) / secs
    sample = (f"{args.config}: each step one layer sample of {n_tok} token(s) (all their routed experts), "
              f"{len(timed)} timed steps after {args.warmup} warm-up, {secs:.1f} s of fp64 oracle arithmetic, "
              f"expert by expert over a spawned pool of {res['cores']} processes")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / max(len(timed), 1) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(cfg, getattr(args, "layers", 48))},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": res["cores"], "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


def workload_name(cfg, NL: int) -> str:
    shared = f" + {cfg.n_shared} shared" if cfg.n_shared else ""
    return (f"{cfg.name}: E{cfg.n_experts}{shared} k{cfg.k} H{cfg.hidden} I{cfg.inter} T{cfg.tokens} "
            f"({cfg.tiers} tiers), {NL} stacked layers per step")


def measure_workload(M, name, args, world, rank, local, steps=None, min_seconds=None):
    """Build the workload's stacked layers, time `steps` steps (or as many as
    fill `min_seconds`) of the CUDA graph, then the profiling and end-to-end
    regions; returns the JSON fields of the workload. Frees its device memory."""
    import numpy as np
    import torch

    import synth
    from synth import gpu as sgpu

    dev = torch.device("cuda", local)
    cfg = synth.CONFIGS[name]
    T, E, k, H, I = cfg.tokens, cfg.n_experts, cfg.k, cfg.hidden, cfg.inter
    NL = args.layers

    layers, tables, wss, outs = [], [], [], []
    for l in range(NL):
        DL = sgpu.make_device_layer(cfg, rank * NL + l)
        layers.append(DL)
        tables.append(M.WeightTable(DL.experts, H, I, grid=DL.grid, n_shared=cfg.n_shared))
        wss.append(M.Workspace(tables[-1], T, k, path=args.path))
        outs.append(torch.empty((T, H), dtype=torch.float32, device=dev))
    torch.cuda.synchronize()

    stream = torch.cuda.Stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(NL)]
    opts_plain = M.make_options(n_experts=cfg.n_entries, path=args.path)
    opts_timed = [M.make_options(n_experts=cfg.n_entries, path=args.path, timing_events=ev[l]) for l in range(NL)]

    def step(timed: bool):
        for l in range(NL):
            M.ffn_forward(tables[l], layers[l].x_bf16, layers[l].logits, k, out=outs[l], ws=wss[l],
                          options=opts_timed[l] if timed else opts_plain)

    # eager warm-up (sets kernel attributes before any capture)
    with torch.cuda.stream(stream):
        step(False)
    stream.synchronize()

    graphs = {}
    if not args.no_graph:
        for timed in (False, True):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(timed)
            graphs[timed] = g

    def run(timed: bool):
        with torch.cuda.stream(stream):
            if args.no_graph:
                step(timed)
            else:
                graphs[timed].replay()

    # algorithmic bytes: distinct routed experts per layer, from the GPU's own
    # bucketing output (read back outside the timed region)
    per_layer_expert_bytes, per_layer_gu_bytes, per_layer_dn_bytes, per_layer_pairs = [], [], [], []
    for l in range(NL):
        routing = wss[l].routing()
        active = routing["active"].cpu().numpy()
        offsets = routing["offsets"].cpu().numpy()
        ids = active[1:1 + active[0]]
        gu = sum(2 * I * synth.row_bytes(layers[l].fmts[e][0], H) for e in ids)
        dn = sum(H * synth.row_bytes(layers[l].fmts[e][1], I) for e in ids)
        per_layer_gu_bytes.append(gu)
        per_layer_dn_bytes.append(dn)
        per_layer_expert_bytes.append(gu + dn)
        per_layer_pairs.append(int(offsets[cfg.n_entries]))
    io_bytes = T * H * 2 + T * E * 4 + T * H * 4

    for _ in range(args.warmup):
        run(False)
    torch.cuda.synchronize()
    if steps is None:
        # as many steps as fill min_seconds, from the period of a few
        t0 = time.perf_counter()
        for _ in range(3):
            run(False)
        torch.cuda.synchronize()
        per = (time.perf_counter() - t0) / 3
        steps = max(3, int(min_seconds / max(per, 1e-6)) + 1)

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.3)

    # ---- timed region 1: the headline (no profiling hooks)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    e0.record(stream)
    for _ in range(steps):
        run(False)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    barrier(world)
    elapsed = allreduce_max(e0.elapsed_time(e1) / 1e3, world)

    # ---- timed region 2: event nodes around the mat-mul kernels of every layer
    gu_ms, dn_ms = [], []
    prof_steps = max(1, min(steps, 20))
    for _ in range(prof_steps):
        run(True)
        stream.synchronize()
        for l in range(NL):
            gu_ms.append(ev[l][0].elapsed_time(ev[l][1]))
            dn_ms.append(ev[l][1].elapsed_time(ev[l][2]))
    clk = clocks.stop()

    # ---- e2e: public API with pinned host buffers, copies inside the region
    # all layers' inputs and outputs in contiguous pinned and device buffers,
    # so that a group of consecutive layers moves in one copy each way
    x_pin = torch.from_numpy(np.stack([L.x_host.view(np.int16) for L in layers])).pin_memory()
    lg_pin = torch.from_numpy(np.stack([L.logits_host for L in layers])).pin_memory()
    out_pin = torch.empty((NL, T, H), dtype=torch.float32).pin_memory()
    x_dev = torch.empty((NL, T, H), dtype=torch.int16, device=dev)
    lg_dev = torch.empty((NL, T, E), dtype=torch.float32, device=dev)
    out_dev = torch.empty((NL, T, H), dtype=torch.float32, device=dev)
    n_e2e = max(1, min(args.e2e_steps, steps))
    # layers per copy: about 2 MB a copy (one layer per copy for the prefill
    # chunk, whose copies are bandwidth-bound and overlap the compute; every
    # layer of a 1-token step in one copy, where each copy's fixed cost would
    # otherwise add ~4 us to a 15 us layer)
    group = max(1, min(NL, (2 << 20) // max(T * (H * 2 + E * 4), T * H * 4)))
    groups = [(g0, min(NL, g0 + group)) for g0 in range(0, NL, group)]

    # Three streams, as a serving loop would run them: the inputs of layer l
    # go up on s_in while earlier layers compute on `stream`, and its output
    # comes back on s_out while later layers compute; one step (all layers,
    # all copies) is captured as a CUDA graph, like the headline's, so that
    # the host does not pace the small layers. Replays of the graph on
    # `stream` run one after another, so every buffer is reused in order.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in groups]
    ev_comp = [torch.cuda.Event() for _ in groups]

    def e2e_step():
        root = torch.cuda.Event()
        root.record(stream)
        s_in.wait_event(root)
        s_out.wait_event(root)
        for gi, (g0, g1) in enumerate(groups):
            with torch.cuda.stream(s_in):
                x_dev[g0:g1].copy_(x_pin[g0:g1], non_blocking=True)
                lg_dev[g0:g1].copy_(lg_pin[g0:g1], non_blocking=True)
                ev_in[gi].record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in[gi])
                for l in range(g0, g1):
                    M.ffn_forward(tables[l], x_dev[l], lg_dev[l], k, out=out_dev[l], ws=wss[l], options=opts_plain)
                ev_comp[gi].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[gi])
                out_pin[g0:g1].copy_(out_dev[g0:g1], non_blocking=True)
        done = torch.cuda.Event()
        done.record(s_out)
        stream.wait_event(done)

    with torch.cuda.stream(stream):
        e2e_step()          # eager once
    torch.cuda.synchronize()
    g_e2e = None
    if not args.no_graph:
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e, stream=stream):
            e2e_step()

    def e2e_run():
        with torch.cuda.stream(stream):
            if g_e2e is None:
                e2e_step()
            else:
                g_e2e.replay()

    for _ in range(2):
        e2e_run()
    torch.cuda.synchronize()
    barrier(world)
    h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0.record(stream)
    for _ in range(n_e2e):
        e2e_run()
    h1.record(stream)
    torch.cuda.synchronize()
    e2e_elapsed = allreduce_max(h0.elapsed_time(h1) / 1e3, world)

    # status of every workspace (device-detected input errors) after all runs
    bad = sum(ws.read_status() for ws in wss)

    hbm_peak, peak_kind = measured_peaks()
    token_layers = T * NL * steps * world
    value = token_layers / elapsed
    per_layer_s = elapsed / (steps * NL)
    mean_expert_bytes = float(np.mean(per_layer_expert_bytes))
    layer_bytes = mean_expert_bytes + io_bytes
    gu_avg, dn_avg = statistics.mean(gu_ms) / 1e3, statistics.mean(dn_ms) / 1e3
    # algorithmic bytes per launch: the routed experts' quantized bytes plus the
    # kernel's activation traffic (x in, h out | h in, y out)
    mean_pairs = float(np.mean(per_layer_pairs))
    gu_bytes = float(np.mean(per_layer_gu_bytes)) + T * H * 2 + mean_pairs * I * 4
    dn_bytes = float(np.mean(per_layer_dn_bytes)) + mean_pairs * I * 4 + mean_pairs * H * 4
    path = M.ffn_path(tables[0], T, k, opts_plain)
    if path == M.PATH_TENSOR:
        gu_name, dn_name = "tc_gemm_kernel<gate/up>", "tc_hprep_kernel + tc_gemm_kernel<down>"
    elif M.gemv_kernels(tables[0], T, k) == M.GEMV_STREAMING:
        gu_name, dn_name = "sg_gateup_kernel", "sg_down_kernel"
    else:
        gu_name, dn_name = "gateup_gemv_kernel", "down_gemv_kernel"
    if path == M.PATH_TENSOR:
        # the h conversion runs between the two timing events of the down projection
        dn_bytes += mean_pairs * I * 2
    if path == M.PATH_FUSED:
        # one kernel runs the whole layer: its algorithmic bytes are the layer's,
        # and its average launch duration is the headline region's period (CUDA
        # events around the timed steps; back to back, one launch per layer).
        # The per-launch event nodes of region 2 would serialise the launches
        # and add their own overhead to each.
        kname, kbytes, kdur = "decode_fused_kernel", layer_bytes, per_layer_s
    elif gu_avg >= dn_avg:
        kname, kbytes, kdur = gu_name, gu_bytes, gu_avg
    else:
        kname, kbytes, kdur = dn_name, dn_bytes, dn_avg
    achieved = kbytes / kdur / 1e9
    tensor_pipe = None
    if path == M.PATH_TENSOR:
        # dense fp16 MMA work of the gate/up and down GEMMs (2 flops per MAC,
        # 3 matrices of H x I per routed pair), against the measured bf16
        # peak (fp16 and bf16 share the dense tensor rate)
        flops = 2.0 * mean_pairs * 3 * H * I
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        tf = flops / (gu_avg + dn_avg) / 1e12
        tensor_pipe = {"flops_per_layer": flops, "achieved_tflops": tf, "peak_tflops": pk["bf16_tflops"],
                       "frac": tf / pk["bf16_tflops"], "peak_kind": "measured bf16 dense burst",
                       "window": "gate/up GEMM + h conversion + down GEMM"}
    res = {
        "value": value, "steps": steps, "ms_per_step": elapsed / steps * 1e3,
        "config": {"workload": workload_name(cfg, NL),
                   "tokens": T, "layers_per_step": NL, "graph": not args.no_graph,
                   "l2": f"inputs exceed L2: {NL} distinct layers, {NL * mean_expert_bytes / 1e9:.2f} GB of "
                         f"routed expert weights per step vs {props.L2_cache_size / 1e6:.0f} MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "per_layer_us": per_layer_s * 1e6,
        "expert_weight_gbs": mean_expert_bytes / per_layer_s / 1e9,
        "layer_roofline": {"bound": "hbm", "bytes_per_layer": layer_bytes,
                           "achieved": layer_bytes / per_layer_s / 1e9, "peak": hbm_peak, "unit": "GB/s",
                           "frac": layer_bytes / per_layer_s / 1e9 / hbm_peak, "peak_kind": peak_kind},
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": kernel_traffic(kname, name),
                     "bytes_per_launch": kbytes, "launch_us": kdur * 1e6, "peak_kind": peak_kind,
                     "launch_timing": ("timed-region period per launch" if path == M.PATH_FUSED
                                       else "event nodes around each kernel"),
                     "other_kernel_us": (0.0 if path == M.PATH_FUSED else
                                         (dn_avg if kname == gu_name else gu_avg) * 1e6)},
        "tensor_pipe": tensor_pipe,
        "e2e": {"value": T * NL * n_e2e * world / e2e_elapsed, "unit": UNIT,
                "h2d_bytes_per_step": NL * (T * H * 2 + T * E * 4), "d2h_bytes_per_step": NL * T * H * 4,
                "layers_per_copy": group},
        "gpu_launches": launches_per_layer(path, T * (k + cfg.n_shared)) * NL * steps,
        "path": {M.PATH_FUSED: "fused decode kernel", M.PATH_GEMV: "grouped GEMV kernels",
                 M.PATH_TENSOR: "tensor-core grouped GEMM"}.get(path, str(path)),
        # the arithmetic of the mat-muls: fp16 operands with fp32 accumulation on
        # the tensor cores; int16 activations times the integer codes (int32 sums,
        # fp32 scales) in the fused and streaming kernels; fp32 in the tiled ones
        "dtype": ("f16" if path == M.PATH_TENSOR else
                  "i16" if path == M.PATH_FUSED or M.gemv_kernels(tables[0], T, k) == M.GEMV_STREAMING else "f32"),
        "clocks": clk,
        "device_status_flags": bad,
    }
    del graphs, layers, tables, wss, outs, x_pin, lg_pin, out_pin, x_dev, lg_dev, out_dev
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_ours(args, world, rank, local):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_moe_expert_route_gb300 as M

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    head = measure_workload(M, args.config, args, world, rank, local, steps=args.steps)
    line = {"metric": METRIC, "value": head.pop("value"), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head.pop("ms_per_step"), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head.pop("dtype"),
            "data": "synthetic (seeded SplitMix64 weights written on the device; bf16 N(0,1) activations; "
                    "Zipf-biased fp32 logits)"}
    head.pop("steps")
    line.update(head)
    line["gpu"] = torch.cuda.get_device_properties(dev).name
    others = [c for c in args.per_config.split(",") if c and c != "none" and c != args.config]
    if world == 1 and others:
        per = {}
        for c in others:
            r = measure_workload(M, c, args, world, rank, local, min_seconds=args.min_seconds)
            r["timed_seconds"] = r["ms_per_step"] * r["steps"] / 1e3
            per[c] = r
        line["per_config"] = per
    return line


def main():
    if "MOE_BENCH_ORACLE_WORKER" in os.environ:
        print(json.dumps(oracle_worker(json.loads(os.environ["MOE_BENCH_ORACLE_WORKER"]))))
        return
    args = parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    # CPU baseline first (before any CUDA work in this process), rank 0, N = 1
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.config, args.cpu_budget)
    line = run_ours(args, world, rank, local)
    if rank == 0:
        line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
