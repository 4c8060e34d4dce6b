#!/usr/bin/env python
"""Throughput of the mixed-adapter LoRA linear layer on GB300.

The default workload is the largest single-GPU one: the 8B-class LoRA stack (32 layers x 7
projections -- q/o 4096->4096, k/v 4096->1024, gate/up 4096->14336, down 14336->4096 --
rank 16 on all 7, 100 resident adapter slots, 512 decode tokens with uniform slot ids,
layer outputs chained).  One step = one chained pass: every projection is one
set_batch_segments + lora_forward of the library's C ABI (BGMV shrink + expand, then the
tcgen05 base GEMM that adds the low-rank term in its epilogue), the whole pass replayed
from one CUDA graph.  Each pass streams ~22 GB of weights and slots, far beyond L2.

--config selects a single-layer workload instead (decode BGMV, prefill SGMV, continuous
batch): one step = set_batch_segments + lora_forward on one batch, rotating over
independent layer instances so that consecutive steps never find their data in L2.

Timing: warm-up steps, then exactly --steps steps bracketed by a barrier and a device
synchronize, CUDA events on the launching stream, max over ranks.

Prints one JSON line.  --impl reference times the CPU oracle instead (rank 0 only).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "mixed-adapter LoRA layer tokens/s; SGMV/BGMV HBM GB/s and % of roofline"
UNIT = "tokens/s"

CONFIGS = {
    "decode_bgmv": dict(seed=1002, desc="decode BGMV: T=256 tokens, K=N=4096, r=16, "
                        "128 slots, 10% base-only, bf16 (fp32 accumulate)"),
    "mixed_continuous": dict(seed=1004, desc="continuous batch: 8x448 prefill + 512 decode rows, "
                             "unsorted, Zipf(1.1) over 1000 ids -> 100 slots, K=14336, "
                             "N=4096, r=16, bf16"),
    "prefill_sgmv": dict(seed=1003, desc="prefill SGMV: T=8192 in 32 geometric segments, "
                         "K=4096, N=14336, r in {8,16,32,64} padded to 64, bf16"),
    "stack_8b": dict(seed=1005, desc="8B-class LoRA stack: 32 layers x 7 projections (q/o "
                     "4096->4096, k/v 4096->1024, gate/up 4096->14336, down 14336->4096), rank 16 "
                     "on all 7, 100 resident slots, 512 decode tokens, outputs chained, bf16"),
}


def make_workload(name, seed, device):
    from segmented_rank_gemm_gb300 import workloads
    fn = getattr(workloads, name)
    return fn(seed=seed, device=device)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------------------------
# algorithmic work per step (what the method must move / compute)
# ------------------------------------------------------------------------------------

def algorithmic(wl, delta_mode=None, fp8=False):
    """Bytes and FLOPs per step: x, W, y once; each distinct adapter slice used in the
    batch once at its true rank; ids; the fp32 intermediate of the low-rank term once
    (v [T_a, r] in v mode; delta [T_a, N] in delta mode, batches of <= 512 bf16 rows).
    fp8 (e4m3 base): W one byte an element, and the quantised x (one byte an element)
    written once and read by the GEMM instead of x."""
    T, K, N = wl.T, wl.K, wl.N
    es = 2 if wl.dtype == torch.bfloat16 else 4
    if delta_mode is None:
        delta_mode = wl.dtype == torch.bfloat16 and T <= 512
    ids = wl.token_slot.cpu().numpy()
    used = sorted(set(int(s) for s in ids if s >= 0))
    ranks = {s: int(wl.adapters[s][0].shape[1]) for s in used}
    adapted = ids >= 0
    n_ad = int(adapted.sum())
    a_bytes = sum(K * ranks[s] * es for s in used)
    b_bytes = sum(ranks[s] * N * es for s in used)
    v_bytes = int(sum(ranks[int(s)] for s in ids[adapted])) * 4
    d_bytes = n_ad * N * 4
    base = {"x": T * K * es, "W": K * N * es, "y": T * N * es, "ids": T * 4}
    lora_flops = 2 * sum(ranks[int(s)] * (K + N) for s in ids[adapted])
    if fp8:
        base["W"] = K * N
        base["xq"] = 2 * T * K  # written by the quantiser, read by the GEMM
    if delta_mode:  # low-rank kernel: x, A, B -> delta; GEMM: x, W, delta -> y
        gemm = (T * K if fp8 else base["x"]) + base["W"] + base["y"] + d_bytes + base["ids"]
        lowrank = base["x"] + a_bytes + b_bytes + d_bytes + base["ids"]
    else:  # tile kernel: x, A -> v; GEMM: x, W, v, B -> y
        gemm = (T * K if fp8 else base["x"]) + base["W"] + base["y"] + b_bytes + v_bytes + base["ids"]
        lowrank = base["x"] + a_bytes + v_bytes
    return {
        "step_bytes": sum(base.values()) + a_bytes + b_bytes,
        "gemm_bytes": gemm,
        "lowrank_bytes": lowrank,
        "base_flops": 2 * T * K * N,
        "lora_flops": lora_flops,
        "distinct_slots": len(used),
        "adapted_rows": n_ad,
        "mode": "delta" if delta_mode else "v",
    }


# ------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, out_path=None):
        self.out_path = out_path
        self.proc = None
        self.lines = []
        self.t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t0 = time.time()
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.out_path:
            with open(self.out_path, "w") as f:
                f.write(self.FIELDS + "\n")
                for t, l in self.lines:
                    f.write("%.3f, %s\n" % (t, l))

    def summary(self, t_from, t_to):
        rows = []
        for t, l in self.lines:
            if not (t_from <= t <= t_to):
                continue
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        gpu = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
        idxs = sorted(set(r[0] for r in rows))
        pick = gpu if gpu in idxs else idxs[0]
        if len(idxs) > 1 and gpu not in idxs:  # the busiest GPU is ours
            pick = max(idxs, key=lambda i: max(float(r[3]) for r in rows if r[0] == i))
        rows = [r for r in rows if r[0] == pick]
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted(set(n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"))
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows)}


# ------------------------------------------------------------------------------------
# distributed helpers (one process per GPU; the layer needs no collective)
# ------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    """The slowest rank's value (host timing reduction; no data of the layer moves)."""
    if world == 1:
        return value
    if torch.distributed.get_backend() == "gloo":
        device = "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units processed by all ranks / the slowest rank's time."""
    return units_per_rank * steps * world / max_seconds


# ------------------------------------------------------------------------------------
# our implementation
# ------------------------------------------------------------------------------------

def traffic_from_profile(kernel_src: str, config: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, if it
    was taken on the current kernel source (else None); e4m3-base runs look up
    ``<config>_fp8``."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    entry = rec.get(config)
    if not entry:
        return None
    with open(kernel_src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    if entry.get("kernel_sha256_16") != h:
        return None
    return entry.get("dram_bytes_per_launch")


def _stack_flops_bytes(T, n_layers, S, fp8=False):
    """Algorithmic work of one chained pass: every projection's base FLOPs 2 T K N; bytes
    W once (e4m3: one byte an element), each distinct adapter slice once (rank 16), the
    projection's input and output once."""
    from segmented_rank_gemm_gb300.workloads import STACK_PROJECTIONS
    flops = sum(2 * T * k * n for _, k, n in STACK_PROJECTIONS) * n_layers
    base_bytes = sum(k * n * (1 if fp8 else 2) for _, k, n in STACK_PROJECTIONS) * n_layers
    ad_bytes = sum(16 * (k + n) * 2 for _, k, n in STACK_PROJECTIONS) * n_layers * S
    act_bytes = sum(T * (k + n) * 2 for _, k, n in STACK_PROJECTIONS) * n_layers
    return flops, base_bytes, ad_bytes, act_bytes


def _stack_oracle_layer(seed, S, T):
    """Layer 0 of the stack drawn on the host (same recipe and seed; the host generator's
    values), as fp64 arrays for the oracle: per projection (x [T,K], W [K,N], slot table),
    with x the projection's generator input; and the slot ids."""
    import oracle
    from segmented_rank_gemm_gb300 import workloads
    _, ids = workloads.stack_tokens(seed=seed, T=T, S=S, device="cpu")
    projs = []
    for p in range(len(workloads.STACK_PROJECTIONS)):
        W, adapters = workloads.stack_projection(0, p, seed=seed, S=S, device="cpu")
        x = workloads.stack_input(p, T=T, seed=seed, device="cpu")
        table = oracle.SlotTable(adapters, W.shape[0], W.shape[1])
        projs.append((x.double().numpy(), W.double().numpy(), table))
        del W, adapters
    return oracle, projs, ids.numpy().astype(np.int32)


def _stack_oracle_rows(oracle, projs, ids, rows):
    """The oracle on `rows` through the 7 projections of one layer (seconds)."""
    t0 = time.time()
    for x, W, table in projs:
        oracle.forward_rows(x, W, table, ids, rows=rows)
    return time.time() - t0


def stack_cpu_baseline(seed, S, T, n_layers, seconds):
    """The oracle (plain C fp64, OpenMP over rows) on this host's cores, on a bounded
    sample of the stack: one thread's worth of rows per round through the 7 projections of
    layer 0, repeated for ``seconds``; tokens/s for the whole stack is rows / (n_layers x
    the time per layer)."""
    oracle, projs, ids = _stack_oracle_layer(seed, S, T)
    threads = oracle.num_threads()
    rng = np.random.default_rng(11)
    rows_done, t = 0, 0.0
    while t < seconds:
        rows = np.sort(rng.choice(T, size=min(threads, T), replace=False)).astype(np.int64)
        t += _stack_oracle_rows(oracle, projs, ids, rows)
        rows_done += rows.shape[0]
    return {"value": rows_done / (t * n_layers), "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": "%d rows (%d per round, seeded) through the 7 projections of layer 0 in "
                      "%.1f s, scaled to the %d-layer stack (per-row work is the same in every "
                      "layer)" % (rows_done, min(threads, T), t, n_layers)}


def run_stack(args):
    """The 8B-class stack: one step = one chained pass over its 224 projections (captured
    in one CUDA graph); every pass streams ~22 GB of weights and slots, far beyond L2."""
    from segmented_rank_gemm_gb300.lora import lora_set_trace_events, LORA_OK
    from segmented_rank_gemm_gb300.stack import LoraStack
    from segmented_rank_gemm_gb300.workloads import STACK_PROJECTIONS

    world, rank, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    t_setup = time.time()
    st = LoraStack(seed=CONFIGS["stack_8b"]["seed"] + 104729 * rank, device=dev,
                   fp8_base=args.fp8, n_layers=args.stack_layers)
    stream = torch.cuda.Stream(device=dev)
    g = st.capture(stream)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            g.replay()
    stream.synchronize()
    setup_s = time.time() - t_setup
    sampler = ClockSampler(args.clocks_csv)
    sampler.start()
    t_soak = time.time()
    while time.time() - t_soak < args.soak_seconds:
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    seconds = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    T = st.T
    step_s = seconds / args.steps

    # ---- per-kernel durations: one eager pass on one stream with the trace events of
    # every projection (each GEMM then runs alone; the pass itself is not the timed one) ----
    n_proj = len(STACK_PROJECTIONS)
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_proj)]
           for _ in st.layers]
    for l, row in enumerate(st.layers):
        for p, layer in enumerate(row):
            lora_set_trace_events(layer.handle, evs[l][p])
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(4e6))  # keeps the GPU behind the host while it enqueues
        st.step(stream, concurrent=False)
    torch.cuda.synchronize()
    for row in st.layers:
        for layer in row:
            lora_set_trace_events(layer.handle, None)
    gemm_us = [[evs[l][p][4].elapsed_time(evs[l][p][5]) * 1e3 for p in range(n_proj)]
               for l in range(len(st.layers))]
    bgmv_us = [[evs[l][p][2].elapsed_time(evs[l][p][3]) * 1e3 for p in range(n_proj)]
               for l in range(len(st.layers))]
    t_clock_end = time.time()
    sampler.stop()
    clocks = sampler.summary(t_soak, t_clock_end)

    # ---- end to end: h0 and the ids from pinned host memory, the chained pass through the
    # C ABI (the captured graph of its 448 calls), h back to pinned host memory ----
    e2e = None
    if not args.no_e2e:
        h0_h = st.h0.cpu().pin_memory()
        ids_h = st.ids.cpu().pin_memory()
        out_h = torch.empty(T, st.buf["h"].shape[1], dtype=torch.bfloat16).pin_memory()

        def e2e_step():
            with torch.cuda.stream(stream):
                st.h0.copy_(h0_h, non_blocking=True)
                st.ids.copy_(ids_h, non_blocking=True)
                g.replay()
                out_h.copy_(st.buf["h"], non_blocking=True)

        for _ in range(2):
            e2e_step()
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e_sec = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
        e2e = {"value": aggregate(T, args.steps, world, e_sec), "unit": UNIT,
               "h2d_bytes_per_step": h0_h.numel() * 2 + ids_h.numel() * 4,
               "d2h_bytes_per_step": out_h.numel() * 2,
               "ms_per_step": e_sec * 1e3 / args.steps,
               "path": "pinned h0 and ids H2D, the chained pass (224 x set_batch_segments + "
                       "lora_forward, one CUDA graph), h D2H"}
    for row in st.layers:
        for layer in row:
            assert layer.status(stream) == LORA_OK

    flops, base_bytes, ad_bytes, act_bytes = _stack_flops_bytes(T, st.n_layers, st.S, args.fp8)
    pk = peaks()
    tf_step = flops / step_s / 1e12
    peak = pk["bf16_tflops_sustained"] or pk["bf16_tflops"]
    peak_note = pk["source"] + " sustained bf16"
    if args.fp8:  # e4m3 contractions: the measured bf16 peak x the nominal ratio 4.5 / 2.25
        peak *= 2.0
        peak_note += " x 2 (nominal e4m3 / bf16 ratio)"
    gemm_total_s = sum(sum(r) for r in gemm_us) * 1e-6
    n_gemm = len(st.layers) * n_proj
    gemm_tf = flops / gemm_total_s / 1e12
    per_shape = {}
    for p, (name, k, n) in enumerate(STACK_PROJECTIONS):
        us = statistics.mean(gemm_us[l][p] for l in range(len(st.layers)))
        per_shape[name] = {"K": k, "N": n, "gemm_us": us,
                           "gemm_tflops": 2 * T * k * n / (us * 1e-6) / 1e12,
                           "bgmv_us": statistics.mean(bgmv_us[l][p] for l in range(len(st.layers)))}
    kernel_src = os.path.join(ROOT, "segmented_rank_gemm_gb300", "csrc", "gemm_tc.cu")
    out = {
        "metric": METRIC, "value": aggregate(T, args.steps, world, seconds), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 base, bf16 low-rank" if args.fp8 else "bf16",
        "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": CONFIGS["stack_8b"]["desc"] + (", base in e4m3 (x per row, W "
                                                             "per column)" if args.fp8 else ""),
                   "T": T, "layers": st.n_layers,
                   "projections": n_proj * st.n_layers, "slots": st.S,
                   "graphs": "one graph per chained pass",
                   "parallelism": "replicas x%d" % world,
                   "l2": "inputs larger than L2: each pass streams %.1f GB of weights and "
                         "slots" % ((base_bytes + ad_bytes) / 1e9)},
        "roofline": {"kernel": "gemm_tc_kernel (base GEMM + fused delta add), all %d launches "
                               "of a pass" % n_gemm,
                     "bound": "tensor", "achieved": gemm_tf, "peak": peak, "unit": "TFLOP/s",
                     "frac": gemm_tf / peak,
                     "traffic": traffic_from_profile(kernel_src, "stack_8b" + ("_fp8" if args.fp8 else "")),
                     "peak_source": peak_note,
                     "frac_of_burst_peak": gemm_tf / (pk["bf16_tflops"] * (2 if args.fp8 else 1)),
                     "algorithmic_flops_per_launch": flops / n_gemm,
                     "avg_launch_us": gemm_total_s * 1e6 / n_gemm},
        "step_tensor": {"achieved_tflops": tf_step, "frac_of_peak": tf_step / peak,
                        "algorithmic_flops": flops},
        "step_hbm": {"algorithmic_bytes": base_bytes + ad_bytes + act_bytes,
                     "achieved_gbs": (base_bytes + ad_bytes + act_bytes) / step_s / 1e9},
        "per_projection": per_shape,
        # per projection: BGMV + GEMM (two launches for a split batch), + the e4m3 row
        # quantiser; counted by the layers themselves (no segment builder at 512 rows)
        "gpu_launches": sum(layer.launch_count() for row in st.layers for layer in row) *
                        args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "setup_s": setup_s,
        "wall_s_timed": t_wall1 - t_wall0,
    }
    st.close()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = stack_cpu_baseline(CONFIGS["stack_8b"]["seed"], st.S, T,
                                                 st.n_layers, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


def run_ours(args):
    from segmented_rank_gemm_gb300.lora import LoraLayer, lora_set_trace_events, LORA_OK
    if args.config == "stack_8b":
        return run_stack(args)

    world, rank, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = CONFIGS[args.config]

    # L independent instances; instance 0 is drawn on the host (the oracle baseline uses
    # the same values), the others on the device from their own seeds.
    layers, inputs, wls = [], [], []
    for i in range(args.layers):
        seed = cfg["seed"] + 7919 * i + 104729 * rank
        wl = make_workload(args.config, seed, "cpu" if i == 0 else dev)
        pool_rows = 0
        if args.pooled:  # adapters at their true rank (rounded up to 8) in a row pool
            pool_rows = sum((int(ad[0].shape[1]) + 7) // 8 * 8 for ad in wl.adapters
                            if ad is not None)
        layer = LoraLayer(wl.W.to(dev), wl.S, wl.R, wl.T, fp8_base=args.fp8, pool_rows=pool_rows)
        for s, ad in enumerate(wl.adapters):
            if ad is not None:
                layer.load(s, ad[0].to(dev), ad[1].to(dev), ad[2])
        if i == 0:
            pool_usage = layer.pool_usage()  # after the loads
        x = wl.x.to(dev)
        ids = wl.token_slot.to(dev)
        y = torch.empty(wl.T, wl.N, dtype=wl.dtype, device=dev)
        layers.append(layer)
        inputs.append((x, ids, y))
        if i == 0:
            wl0 = wl
        else:
            del wl
    torch.cuda.synchronize()
    T, K, N = wl0.T, wl0.K, wl0.N
    work = algorithmic(wl0, fp8=args.fp8)

    stream = torch.cuda.Stream(device=dev)

    def step(i):
        layer = layers[i % len(layers)]
        x, ids, y = inputs[i % len(layers)]
        layer.set_batch(ids, stream)
        layer.forward(x, y, stream)

    # warm-up (eager), then capture one graph per instance
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1) * len(layers)):
            step(i)
    stream.synchronize()
    for l in layers:
        assert l.status(stream) == LORA_OK
    # one graph per step and instance, and one graph of a whole rotation (one step on each
    # instance in turn, as the layers of a model's decode step are captured together)
    graphs, rot_graph = [], None
    if not args.no_graph:
        for i in range(len(layers)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(i)
            graphs.append(g)
        rot_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(rot_graph, stream=stream):
            for i in range(len(layers)):
                step(i)
        for i in range(len(layers)):
            graphs[i].replay()
        rot_graph.replay()
        torch.cuda.synchronize()

    def run_steps(n, offset=0):
        """Exactly n steps: whole rotations from the rotation graph, the rest one by one."""
        if graphs:
            with torch.cuda.stream(stream):
                i = 0
                while i < n and (i + offset) % len(graphs) != 0:
                    graphs[(i + offset) % len(graphs)].replay()
                    i += 1
                while n - i >= len(graphs):
                    rot_graph.replay()
                    i += len(graphs)
                while i < n:
                    graphs[(i + offset) % len(graphs)].replay()
                    i += 1
        else:
            with torch.cuda.stream(stream):
                for i in range(n):
                    step(i + offset)

    # clocks: sample through a short soak and the timed region
    sampler = ClockSampler(args.clocks_csv)
    sampler.start()
    t_soak = time.time()
    with torch.cuda.stream(stream):
        for _ in range(3):
            run_steps(args.warmup)
    stream.synchronize()
    while time.time() - t_soak < args.soak_seconds:
        run_steps(max(len(layers), 64))
        stream.synchronize()

    # ---- timed region: exactly args.steps steps ----
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    run_steps(args.steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    seconds = ev0.elapsed_time(ev1) / 1e3
    seconds_max = max_over_ranks(seconds, world, dev)
    value = aggregate(T, args.steps, world, seconds_max)
    ms_per_step = seconds_max * 1e3 / args.steps

    # ---- per-kernel durations: eager steps with the library's trace events ----
    n_prof = min(args.steps, 400)
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_prof)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for c0 in range(0, n_prof, 32):
            # a bounded device-side delay keeps the GPU behind the host while it enqueues
            # the next 32 steps, so no host gap falls between a kernel's trace events
            torch.cuda._sleep(int(4e6))
            for i in range(c0, min(n_prof, c0 + 32)):
                lora_set_trace_events(layers[i % len(layers)].handle, ev_sets[i])
                step(i)
    torch.cuda.synchronize()
    for l in layers:
        lora_set_trace_events(l.handle, None)
    dur = {"builder": [], "shrink": [], "gemm": []}
    for evs in ev_sets:
        dur["builder"].append(evs[0].elapsed_time(evs[1]) * 1e3)
        dur["shrink"].append(evs[2].elapsed_time(evs[3]) * 1e3)
        dur["gemm"].append(evs[4].elapsed_time(evs[5]) * 1e3)
    kern_us = {k: statistics.mean(v) for k, v in dur.items()}
    t_clock_end = time.time()
    sampler.stop()
    clocks = sampler.summary(t_soak, t_clock_end)

    # ---- end to end through the C ABI with host buffers ----
    e2e = None
    if not args.no_e2e:
        x_h = [inp[0].cpu().pin_memory() for inp in inputs]
        ids_h = [inp[1].cpu().pin_memory() for inp in inputs]
        y_h = [torch.empty(T, N, dtype=wl0.dtype).pin_memory() for _ in inputs]
        with torch.cuda.stream(stream):
            for i in range(len(layers)):
                layers[i].forward_host(x_h[i], ids_h[i], y_h[i], stream)
        stream.synchronize()
        n_e2e = args.steps
        # consecutive steps go to several streams (instance j always to stream j % n, so
        # each layer object and its staging stay on one stream), as a serving loop would
        # issue them: steps' host copies overlap other steps' kernels
        n_st = max(1, min(args.e2e_streams, len(layers)))
        streams = (stream,) + tuple(torch.cuda.Stream(device=dev) for _ in range(n_st - 1))
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s_k in streams[1:]:
            s_k.wait_event(e0)
        for i in range(n_e2e):
            j = i % len(layers)
            s_j = streams[j % n_st]
            with torch.cuda.stream(s_j):
                layers[j].forward_host(x_h[j], ids_h[j], y_h[j], s_j)
        for s_k in streams[1:]:
            stream.wait_stream(s_k)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e_sec = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
        es = 2 if wl0.dtype == torch.bfloat16 else 4
        e2e = {"value": aggregate(T, n_e2e, world, e_sec), "unit": UNIT,
               "h2d_bytes_per_step": T * K * es + T * 4, "d2h_bytes_per_step": T * N * es,
               "ms_per_step": e_sec * 1e3 / n_e2e,
               "streams": n_st,
               "path": "lora_forward_host: pinned x/ids H2D, %s, y D2H" % (
                   "BGMV, GEMM" if work["mode"] == "delta" else "builder, SGMV shrink, GEMM")}

    for l in layers:
        assert l.status(stream) == LORA_OK

    pk = peaks()
    gemm_s = kern_us["gemm"] * 1e-6
    achieved = work["gemm_bytes"] / gemm_s / 1e9
    kernel_src = os.path.join(ROOT, "segmented_rank_gemm_gb300", "csrc", "gemm_tc.cu")
    roofline = {"kernel": "gemm_tc_kernel (base GEMM%s + fused expand)"
                          % (", e4m3" if args.fp8 else ""), "bound": "hbm",
                "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"],
                "traffic": traffic_from_profile(kernel_src, args.config + ("_fp8" if args.fp8 else "")),
                "peak_source": pk["source"], "algorithmic_bytes_per_launch": work["gemm_bytes"],
                "avg_launch_us": kern_us["gemm"]}
    if args.config != "decode_bgmv":
        # the GEMM is timed inside a long run of back-to-back steps (after the soak), under
        # the same power cap as the measured sustained cuBLAS loop: that is its peak; the
        # burst fraction is given beside it
        tflops = work["base_flops"] / gemm_s / 1e12
        # e4m3 contractions: the measured bf16 peak x the nominal ratio 4.5 / 2.25
        ratio = 2.0 if args.fp8 else 1.0
        peak = (pk["bf16_tflops_sustained"] or pk["bf16_tflops"]) * ratio
        roofline.update({"bound": "tensor", "achieved": tflops, "peak": peak,
                         "unit": "TFLOP/s", "frac": tflops / peak,
                         "peak_source": pk["source"] + " sustained" +
                                        (" bf16 x 2 (nominal e4m3 / bf16 ratio)" if args.fp8 else ""),
                         "frac_of_burst_peak": tflops / (pk["bf16_tflops"] * ratio),
                         "algorithmic_flops_per_launch": work["base_flops"]})

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 base, bf16 low-rank" if args.fp8 else "bf16")
        if wl0.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded, shapes of the pages' 8B-class workloads)",
        "config": {"workload": cfg["desc"] + (", base in e4m3 (x per row, W per column)"
                                              if args.fp8 else ""),
                   "T": T, "K": K, "N": N, "slots": wl0.S,
                   "slot_rank_width": wl0.R, "distinct_slots": work["distinct_slots"],
                   "adapted_rows": work["adapted_rows"], "parallelism": "replicas x%d" % world,
                   "l2": "rotating %d independent layer instances (~%d MB of weights and slots)%s"
                         % (len(layers), len(layers) * work["step_bytes"] // 10**6,
                            " > 129 MB L2" if len(layers) * work["step_bytes"] > 129 * 10**6
                            else ": fits the 129 MB L2, steps may hit it (not a bench number)"),
                   "graphs": ("one graph per rotation of %d steps (one per instance)" % len(layers))
                             if not args.no_graph else False},
        "roofline": roofline,
        "slot_pool": {"pooled": bool(args.pooled), "rows_used": pool_usage[0],
                      "rows": pool_usage[1], "padded_rows": wl0.S * ((wl0.R + 7) // 8 * 8)},
        "step_hbm": {"algorithmic_bytes": work["step_bytes"],
                     "achieved_gbs": work["step_bytes"] / (ms_per_step * 1e-3) / 1e9,
                     "frac_of_measured": work["step_bytes"] / (ms_per_step * 1e-3) / 1e9 / pk["hbm_gbs"],
                     "frac_of_8tbs_spec": work["step_bytes"] / (ms_per_step * 1e-3) / 8e12},
        "kernels_us": kern_us,
        "lowrank_kernel": {"algorithmic_bytes": work["lowrank_bytes"],
                           "achieved_gbs": work["lowrank_bytes"] / (kern_us["shrink"] * 1e-6) / 1e9,
                           "mode": work["mode"]},
        # decode batches (bf16, <= 512 rows): BGMV + GEMM; larger: builder + shrink + GEMM;
        # + the e4m3 row quantiser, + a split GEMM's second launch (counted by the layer)
        "gpu_launches": layers[0].launch_count() * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "wall_s_timed": t_wall1 - t_wall0,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl0, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out))
    for l in layers:
        l.close()
    if world > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------------------------
# the CPU oracle as a baseline
# ------------------------------------------------------------------------------------

def _oracle_inputs(wl):
    import oracle
    table = oracle.SlotTable(wl.adapters, wl.K, wl.N)
    x = wl.x.double().numpy()
    W = wl.W.double().numpy()
    ids = wl.token_slot.numpy().astype(np.int32)
    return oracle, table, x, W, ids


def cpu_baseline(wl, seconds: float):
    """The oracle as it stands (plain C fp64, OpenMP over rows) on this host's cores:
    whole batches repeated until ``seconds`` have passed."""
    oracle, table, x, W, ids = _oracle_inputs(wl)
    rows = np.arange(wl.T, dtype=np.int64)
    t0 = time.time()
    reps = 0
    while True:
        oracle.forward_rows(x, W, table, ids, rows=rows)
        reps += 1
        if time.time() - t0 >= seconds:
            break
    dt = time.time() - t0
    return {"value": reps * wl.T / dt, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle", "sample": "%d repetitions of the full %d-row batch (%.1f s)"
            % (reps, wl.T, dt)}


def run_reference_stack(args):
    """The oracle on the stack's workload: each step a seeded sample of rows (one per host
    thread) through the 7 projections of layer 0; tokens/s for the whole stack is rows /
    (layers x the time per layer)."""
    seed, S, T, n_layers = CONFIGS["stack_8b"]["seed"], 100, 512, args.stack_layers
    oracle, projs, ids = _stack_oracle_layer(seed, S, T)
    threads = oracle.num_threads()
    n_rows = min(threads, T)
    rng = np.random.default_rng(0)
    samples = [np.sort(rng.choice(T, size=n_rows, replace=False)).astype(np.int64)
               for _ in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        _stack_oracle_rows(oracle, projs, ids, samples[i])
    t = 0.0
    for i in range(args.steps):
        t += _stack_oracle_rows(oracle, projs, ids, samples[args.warmup + i])
    step_s = t * n_layers / args.steps  # one step: the sampled rows through the whole stack
    value = n_rows / (step_s)
    sample = ("%d of %d rows per step (seeded) through the 7 projections of layer 0, scaled "
              "to %d layers, %d steps" % (n_rows, T, n_layers, args.steps))
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": CONFIGS["stack_8b"]["desc"], "T": T, "layers": n_layers,
                   "projections": 7 * n_layers, "slots": S,
                   "parallelism": "host cores, rank 0"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return  # the oracle runs on rank 0's host cores only
    if args.config == "stack_8b":
        return run_reference_stack(args)
    cfg = CONFIGS[args.config]
    wl = make_workload(args.config, cfg["seed"], "cpu")
    oracle, table, x, W, ids = _oracle_inputs(wl)
    threads = oracle.num_threads()
    # size each step's sample so that the whole run stays within ~2 minutes
    t0 = time.time()
    oracle.forward_rows(x, W, table, ids, rows=np.arange(min(threads, wl.T), dtype=np.int64))
    t_row = (time.time() - t0) / min(threads, wl.T)
    budget = 120.0 / max(args.steps + args.warmup, 1)
    n_rows = int(max(1, min(wl.T, budget / max(t_row, 1e-9))))
    rng = np.random.default_rng(0)
    samples = [np.sort(rng.choice(wl.T, size=n_rows, replace=False)).astype(np.int64)
               for _ in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        oracle.forward_rows(x, W, table, ids, rows=samples[i])
    t0 = time.time()
    for i in range(args.steps):
        oracle.forward_rows(x, W, table, ids, rows=samples[args.warmup + i])
    dt = time.time() - t0
    value = n_rows * args.steps / dt
    sample = "%d of %d rows per step (seeded), %d steps" % (n_rows, wl.T, args.steps)
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, shapes of the pages' 8B-class workloads)",
        "config": {"workload": cfg["desc"], "T": wl.T, "K": wl.K, "N": wl.N, "slots": wl.S,
                   "slot_rank_width": wl.R, "parallelism": "host cores, rank 0"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


def run_swap_in(args):
    """Adapter residency on the 8B-class stack (224 projections, rank 16, ~80 MiB per
    adapter): (1) the swap-in of one adapter from the cache's pinned host tier into a GPU
    slot of every projection (one host-to-device copy + one scatter kernel), timed with
    CUDA events on the cache's stream; (2) chained passes over the stack, each naming three
    adapters, first with every adapter resident, then sliding one new adapter into every
    batch by a prefetch issued while the previous pass computes -- the pages' claim that a
    prefetched swap-in hides behind the running batch."""
    from segmented_rank_gemm_gb300.lora import AdapterCache
    from segmented_rank_gemm_gb300.stack import LoraStack
    from segmented_rank_gemm_gb300.workloads import STACK_PROJECTIONS

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    S, H, r = 4, 8, 16
    st = LoraStack(S=S, seed=CONFIGS["stack_8b"]["seed"], device=dev)
    layers = [layer for row in st.layers for layer in row]
    cache = AdapterCache(layers, S, H)
    g = torch.Generator().manual_seed(7)
    shapes = {}
    for _, k, n in STACK_PROJECTIONS:  # one random (A, B) per shape; content is irrelevant
        if (k, n) not in shapes:
            shapes[(k, n)] = ((torch.randn(k, r, generator=g) * 0.02).to(torch.bfloat16),
                              (torch.randn(r, n, generator=g) * 0.02).to(torch.bfloat16))
    A_list = [shapes[(L.K, L.N)][0] for L in layers]
    B_list = [shapes[(L.K, L.N)][1] for L in layers]
    t0 = time.perf_counter()
    for a in range(H):
        cache.add(a, A_list, B_list, 2.0 * r)
    add_ms = (time.perf_counter() - t0) * 1e3 / H
    image = sum((L.max_rank + 7) // 8 * 8 * (L.K + L.N) * 2 for L in layers)
    cs = torch.cuda.ExternalStream(cache.stream, device=dev)

    # (1) swap-in latency: no batch in flight, each prefetch evicts the LRU adapter
    order = [a % H for a in range(S, S + 4 * H)]
    for a in order[:H]:
        cache.prefetch([a])
    cache.sync()
    host_s = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cs)
    for a in order[H:]:
        t = time.perf_counter()
        cache.prefetch([a])
        host_s.append(time.perf_counter() - t)
    e1.record(cs)
    cache.sync()
    n_swaps = len(order) - H
    swap_ms = e0.elapsed_time(e1) / n_swaps

    # (2) passes: resident adapters only, then one prefetched newcomer per batch
    stream = torch.cuda.Stream(device=dev)
    graph = st.capture(stream)
    rng = np.random.default_rng(3)
    T = st.T

    def passes(n, sliding):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for k in range(n + 3):
            if k == 3:
                ev[0].record(stream)
            base = k if sliding else 0
            names = [(base + j) % H for j in range(3)]
            ids = np.asarray(names)[rng.integers(0, 3, size=T)].astype(np.int64)
            slots = cache.map_batch(ids, stream)
            with torch.cuda.stream(stream):
                st.ids.copy_(torch.from_numpy(slots.astype(np.int32)), non_blocking=True)
                graph.replay()
            if sliding:
                cache.prefetch([(base + 3) % H])  # the next batch's newcomer
        ev[1].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / n

    cache.prefetch([0, 1, 2])
    n = max(args.steps, 8)
    resident_ms = passes(n, False)
    before = cache.stats()
    sliding_ms = passes(n, True)
    after = cache.stats()
    cache.close()
    st.close()
    out = {
        "metric": "adapter swap-in, host DRAM -> GPU slots (8B-class rank-16 adapter)",
        "value": swap_ms, "unit": "ms per adapter", "higher_is_better": False, "n_gpus": 1,
        "steps": n_swaps, "dtype": "bf16", "data": "synthetic (random-init adapters)",
        "config": {"workload": "8B-class stack, 32 layers x 7 projections, rank 16, "
                   "%d GPU slots, %d adapters in the pinned host tier" % (S, H),
                   "image_bytes": image, "projections": len(layers)},
        "swap_in": {"ms": swap_ms, "gbs": image / (swap_ms * 1e-3) / 1e9,
                    "host_call_ms_median": statistics.median(host_s) * 1e3,
                    "launches": 2, "add_ms_per_adapter": add_ms},
        "overlap": {"passes": n, "ms_per_pass_resident": resident_ms,
                    "ms_per_pass_one_prefetched_swap_in": sliding_ms,
                    "swap_ins": after["prefetches"] - before["prefetches"],
                    "misses": after["misses"] - before["misses"],
                    "hidden_fraction": max(0.0, 1.0 - max(0.0, sliding_ms - resident_ms)
                                           / swap_ms)},
    }
    print(json.dumps(out))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 40 for the stack, 400 for the single layers)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(CONFIGS), default="stack_8b")
    ap.add_argument("--stack-layers", type=int, default=32,
                    help="layers of the 8B-class stack (32 is the workload; fewer for profiling)")
    ap.add_argument("--layers", type=int, default=8, help="independent instances rotated")
    ap.add_argument("--soak-seconds", type=float, default=1.5)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=4,
                    help="streams the end-to-end steps rotate over (instance j on stream j %% n)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="also write the nvidia-smi clock samples to this CSV file")
    ap.add_argument("--pooled", action="store_true",
                    help="adapters at their true rank in a row pool (lora_layer_create_pooled)")
    ap.add_argument("--fp8", action="store_true",
                    help="the base in e4m3 (lora_layer_create_fp8), for any --config")
    ap.add_argument("--swap-in", action="store_true",
                    help="measure adapter swap-ins through the adapter cache instead")
    args = ap.parse_args(argv)
    if args.steps is None:
        args.steps = 40 if args.config == "stack_8b" else 400
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3  # at least 3 warm-up steps
    if args.swap_in:
        run_swap_in(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
