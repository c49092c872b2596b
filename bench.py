"""Benchmark: routed FP4 MoE expert-FFN decode on one GB300 (or N replicas).

Workload (default `stack_b1`, the metric's configuration): a decode step of a
40-layer MoE stack at batch 1 -- each layer 128 resident experts (H=4096,
I=2880, FP4 E2M1 + ue8m0 per 32; 96 GB for the stack), top-6 routing drawn per
layer, residual + RMSNorm per layer, the whole step one CUDA graph
(moe_stack_forward).  `layer_b1` is one layer with 384 resident experts (7.2
GB), a fresh token per step, consecutive steps sharing no expert (every step
streams its 6 experts, 112.8 MB, from HBM: inputs far larger than L2),
replayed from CUDA graphs of up to 500 calls.

Other workloads (`--workload`): the same layer at batch 64 (uniform routing)
and 512 (Zipf expert popularity) with E4M3 activations, and a 40-layer stack
of 128-expert layers (residual + RMSNorm per layer, one CUDA graph per step)
at batch 1 and 32.

One JSON line on rank 0.  `value` is tokens/s of the layer (or of the whole
stack) summed over ranks (each rank an independent replica: "scaling":
"weak").  `--impl reference` times the CPU oracle instead (on this host's
cores).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    # one MoE layer, decode batch 1 (the per-layer headline)
    "layer_b1": dict(E=384, H=4096, I=2880, k=6, T=1, L=1, act="bf16", dist="uniform", steps=20000),
    # same step (6 experts streamed per token) with 64 resident experts (1.2 GB,
    # still far above L2): the size used for ncu captures
    "layer_b1_e64": dict(E=64, H=4096, I=2880, k=6, T=1, L=1, act="bf16", dist="uniform", steps=20000),
    # the 384-expert layer at decode batch 64 (uniform) and 512 (Zipf 1.1 expert
    # popularity), activations quantized to E4M3 with ue8m0 per 128
    "layer_b64": dict(E=384, H=4096, I=2880, k=6, T=64, L=1, act="e4m3", dist="uniform", steps=1000),
    "layer_b512": dict(E=384, H=4096, I=2880, k=6, T=512, L=1, act="e4m3", dist="zipf", steps=100),
    # expert-major path with 64 resident experts (1.2 GB, above L2) at batch 16: 1-2
    # slots per group as at batch 64; the size used for ncu captures of k_glayer
    "layer_b16_e64": dict(E=64, H=4096, I=2880, k=6, T=16, L=1, act="e4m3", dist="uniform", steps=2000),
    # 40-layer stack of 128-expert layers (96 GB resident), residual + RMSNorm (stack_b1:
    # the default, the metric's configuration),
    # the whole step as one CUDA graph, at batch 1 and 32
    "stack_b1": dict(E=128, H=4096, I=2880, k=6, T=1, L=40, act="bf16", dist="uniform", steps=500),
    "stack_b32": dict(E=128, H=4096, I=2880, k=6, T=32, L=40, act="bf16", dist="uniform", steps=50),
    # expert-sharing batching: pools of 256 sequences from 8 prompt clusters
    # (alike prompts route alike), cut into batches of 32 by the planner
    # (moe_batch_plan on the previous step's routing) or in arrival order; each
    # step runs one batch's next-step routing through the 384-expert layer
    "layer_b32_shared": dict(E=384, H=4096, I=2880, k=6, T=32, L=1, act="e4m3", dist="clustered_planned",
                             steps=1000),
    "layer_b32_arrival": dict(E=384, H=4096, I=2880, k=6, T=32, L=1, act="e4m3", dist="clustered_arrival",
                              steps=1000),
    # a compute-bound shape of the same formats: 8 experts, each chosen by all
    # 2048 tokens (M = 2048 rows per expert), E4M3 activations x E2M1 weights --
    # 1.16 TFLOP a step against 150 MB of weights, far right of the ridge point
    "gemm_e8_b2048": dict(E=8, H=4096, I=2880, k=8, T=2048, L=1, act="e4m3", dist="uniform", steps=20,
                          bound="tensor"),
}
SHARING_POOL, SHARING_CLUSTERS, SHARING_SIG_LAYERS = 256, 8, 8
# host-resident experts: the 384 experts of the layer in page-locked host memory,
# 64 of them cached in HBM; consecutive steps share no expert, so every step
# copies its 6 experts over NVLink-C2C unless a predictor prefetched them
WORKLOADS["layer_b1_host"] = dict(E=384, H=4096, I=2880, k=6, T=1, L=1, act="bf16", dist="uniform", steps=300,
                                  host=True, slots=64, guess=0.0)
WORKLOADS["layer_b1_host_prefetch"] = dict(E=384, H=4096, I=2880, k=6, T=1, L=1, act="bf16", dist="uniform",
                                           steps=300, host=True, slots=64, guess=0.8)
METRIC = "MoE expert-FFN decode tokens/s per layer-stack & HBM GB/s (% of GB300 roofline)"
FALLBACK_HBM_GBS = 6800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# dense tensor rates relative to bf16 (nominal per-GPU figures: bf16 2.25,
# fp8 / kind::mxf8f6f4 4.5, fp4 / kind::mxf4 13.5 PFLOP/s)
FP8_PER_BF16, FP4_PER_BF16 = 2.0, 6.0
FALLBACK_BF16_TFLOPS = 1900.0


def tensor_peak_bf16():
    """Measured dense bf16 TFLOP/s (burst: a kernel timed alone) and its kind."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def expert_bytes(H, I):
    return 3 * H * I // 2 + 3 * H * I // 32


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([s.strip() for s in line.split(",")])

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            if len(r) >= 9:
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def draw_routings(R, E, k, T, seed, dist="uniform", layer=0):
    """R pre-drawn routings of T tokens.  At batch 1 consecutive ones share no
    expert, so every step streams its experts from HBM."""
    import numpy as np

    import synth

    idx = np.zeros((R, T, k), np.int32)
    prev = None
    if dist.startswith("clustered"):
        # batches of T from pools of alike-routing sequences: planned on the
        # previous step's routing (SHARING_SIG_LAYERS layers), measured on the
        # next step's routing of this layer
        import fp4_block_scaled_gb300 as moe

        per_pool = SHARING_POOL // T
        for p in range((R + per_pool - 1) // per_pool):
            r0, _ = synth.routing_clustered(SHARING_POOL, SHARING_SIG_LAYERS, E, k, SHARING_CLUSTERS,
                                            seed=seed * 1000 + p, step=0)
            r1, _ = synth.routing_clustered(SHARING_POOL, SHARING_SIG_LAYERS, E, k, SHARING_CLUSTERS,
                                            seed=seed * 1000 + p, step=1)
            order = (moe.moe_batch_plan(r0, E, T) if dist == "clustered_planned"
                     else np.arange(SHARING_POOL, dtype=np.int32))
            for b in range(per_pool):
                r = p * per_pool + b
                if r < R:
                    idx[r] = r1[order[b * T:(b + 1) * T], layer % SHARING_SIG_LAYERS]
    for r in range(R if not dist.startswith("clustered") else 0):
        st = synth.S_ROUTE + 1000 * (r + 1) + 7 * layer
        if dist == "zipf":
            cur = synth.routing_zipf(T, E, k, s=1.1, seed=seed, stream=st)
        else:
            cur = synth.routing_uniform(T, E, k, seed=seed, stream=st, avoid=prev if T == 1 else None)
        idx[r] = cur
        prev = set(int(v) for v in cur.reshape(-1))
    w = np.stack([synth.routing_weights(T, k, seed=seed, stream=synth.S_LOGIT + 1000 * (r + 1) + 7 * layer)
                  for r in range(R)])
    return idx, w


def source_fingerprint(path):
    """sha256 of a C/CUDA source, and of the in-tree headers it includes
    (recursively), without comments and whitespace: the code the counters
    were taken on (a comment edit does not invalidate them)."""
    import re

    seen, parts = set(), []

    def add(p):
        p = os.path.normpath(p)
        if p in seen or not os.path.exists(p):
            return
        seen.add(p)
        text = open(p, encoding="utf-8").read()
        for inc in re.findall(r'^\s*#\s*include\s+"([^"]+)"', text, flags=re.M):
            add(os.path.join(os.path.dirname(p), inc))
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        parts.append(re.sub(r"\s+", "", text))

    add(path)
    return hashlib.sha256("".join(parts).encode()).hexdigest()


def traffic_record(kernel, workload, act, algorithmic_bytes):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source, on this workload's launch shape and in this
    activation mode (else None):
    the captured bytes, or the captured dram/algorithmic ratio times this
    workload's algorithmic bytes per launch."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(kernel)
    if not rec or workload not in rec.get("workloads", []) or act != rec.get("activations"):
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src):
        return None
    if source_fingerprint(src) != rec.get("source_fingerprint"):
        return None
    if "dram_bytes_per_algorithmic_byte" in rec:
        return rec["dram_bytes_per_algorithmic_byte"] * algorithmic_bytes
    return rec["dram_bytes_per_launch"]


# --------------------------------------------------------------- CPU oracle

def _act_mode(wl):
    import oracle

    return {"e4m3": oracle.ACT_E4M3_UE8M0_128, "e2m1": oracle.ACT_E2M1_UE8M0_32}.get(wl["act"], oracle.ACT_BF16)


def _oracle_token(wl, n, seed):
    """Inputs of the n-th sampled (token, layer) of the workload: the oracle's
    cost is per token and layer, so whole tokens of single layers are the unit
    of every CPU sample (a stack token costs L of them)."""
    import synth

    E, H, I, k, L = wl["E"], wl["H"], wl["I"], wl["k"], wl["L"]
    layer = n % L
    if wl["dist"] == "zipf":
        idx = synth.routing_zipf(1, E, k, s=1.1, seed=seed + 17, stream=synth.S_ROUTE + 7 * n)
    else:
        idx = synth.routing_uniform(1, E, k, seed=seed + 17, stream=synth.S_ROUTE + 7 * n)
    w = synth.routing_weights(1, k, seed=seed + 17, stream=synth.S_LOGIT + 7 * n)
    x = synth.activations_bf16(1, H, seed=seed + 17, n0=H * n)
    codes, scales = [None] * E, [None] * E
    for e in set(int(v) for v in idx.reshape(-1)):
        codes[e], scales[e] = synth.expert_canonical(H, I, e, layer=layer)
    return codes, scales, x, idx, w


def cpu_sample(wl, budget_s=12.0, seed=0):
    """The oracle, as it stands, on whole tokens of single layers of the
    workload until the budget is used (at least one).  Returns (tokens/s of the
    workload, threads, sample)."""
    import oracle

    E, H, I, k, L = wl["E"], wl["H"], wl["I"], wl["k"], wl["L"]
    act = _act_mode(wl)
    threads = min(cores(), k)
    done, spent = 0, 0.0
    while spent < budget_s and done < 64:
        codes, scales, x, idx, w = _oracle_token(wl, done, seed)
        t0 = time.perf_counter()
        oracle.moe_ffn(codes, scales, H, I, x, idx, w, act_mode=act, nthreads=threads)
        spent += time.perf_counter() - t0
        done += 1
    per_layer = done / spent
    what = f"{done} whole tokens of one layer (top-{k} of {E}, H={H}, I={I}, {wl['act']} activations, {wl['dist']} routing)"
    if L > 1:
        what += f", scaled to the {L}-layer stack as 1/{L} of the per-layer rate"
    return per_layer / L, threads, what + f", fp64 oracle, {threads} threads over slots"


def run_reference(args, wl):
    """--impl reference: the CPU oracle on this host's cores, same metric."""
    import numpy as np

    import oracle
    import synth

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    E, H, I, k, L = wl["E"], wl["H"], wl["I"], wl["k"], wl["L"]
    act = _act_mode(wl)
    threads = min(cores(), k)
    per_token_weights = k * 3 * H * I
    # calibrate one token of one layer
    codes, scales, x, idx, w = _oracle_token(wl, 0, 3)
    used = sorted(set(int(v) for v in idx.reshape(-1)))
    t0 = time.perf_counter()
    oracle.moe_ffn(codes, scales, H, I, x, idx, w, act_mode=act, nthreads=threads)
    t_token = time.perf_counter() - t0
    budget = 90.0
    nsteps = args.steps + args.warmup
    if nsteps * t_token <= budget:
        mode, rows = "token", None
        sample = (f"one whole token of one layer per step (top-{k} of {E}, H={H}, I={I}, "
                  f"{wl['act']} activations), {threads} threads")
    else:
        mode = "rows"
        # rows of one gate matrix per step, single thread, sized to the budget
        t_row = t_token * threads / (k * 3 * I)          # seconds per H-long row, one thread
        rows = max(1, min(I, int(budget / nsteps / t_row)))
        threads = 1
        sample = (f"{rows} gate rows (K={H}) of one expert per step, 1 thread, scaled to "
                  f"tokens by weights processed")
    if L > 1:
        sample += f"; a stack token costs {L} layer-tokens, the rate is divided by {L}"
    e0 = used[0]
    xr = synth.bf16_bits_to_f32(x[0]).astype(np.float64)

    def step():
        if mode == "token":
            oracle.moe_ffn(codes, scales, H, I, x, idx, w, act_mode=act, nthreads=threads)
        else:
            oracle.matvec(codes[e0][:rows * H // 2], scales[e0][:rows * H // 32], rows, H, xr)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    if mode == "token":
        value = args.steps / dt / L
    else:
        value = args.steps * rows * H / dt / per_token_weights / L
    ms = dt * 1000.0 / args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "layers": L, "experts": E, "hidden": H, "inter": I,
                   "topk": k, "tokens_per_step": wl["T"], "routing": wl["dist"],
                   "activations": wl["act"], "l2": "cpu run"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- ranks

def max_over_ranks(v, dist, device):
    """The largest v over the ranks: a replicated job takes as long as its
    slowest rank (dist: torch.distributed, or None for one rank)."""
    if dist is None:
        return float(v)
    import torch

    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, tokens_per_step, steps, ms_total):
    """Tokens per second of `world` independent replicas that each ran `steps`
    steps of `tokens_per_step` tokens within ms_total (the slowest rank's time)."""
    return world * tokens_per_step * steps / (ms_total / 1000.0)


# --------------------------------------------------------------- GPU arm

def run_ours(args, wl):
    import numpy as np
    import torch

    import fp4_block_scaled_gb300 as moe
    import synth
    from fp4_block_scaled_gb300.experts import ExpertSet

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    E, H, I, k, T, L = wl["E"], wl["H"], wl["I"], wl["k"], wl["T"], wl["L"]
    act = {"e4m3": moe.MOE_ACT_E4M3_UE8M0_128, "e2m1": moe.MOE_ACT_E2M1_UE8M0_32}.get(wl["act"], moe.MOE_ACT_BF16)
    gmin = {"auto": 0, "slot": T + 1, "group": 1}[args.path]
    cfg = moe.config(E, H, I, k, T, act_mode=act, out_dtype=moe.MOE_OUT_F32, gemm_min_tokens=gmin)
    grouped = T >= (gmin or moe.DEFAULT_GEMM_MIN_TOKENS)
    # the quantized modes' expert-major form (E4M3: kind::mxf8f6f4, E2M1:
    # kind::mxf4, activations as they are): as asked, or the library's choice (auto)
    f8 = (grouped and wl["act"] in ("e4m3", "e2m1")
          and (args.mma == "f8" or (args.mma == "auto" and T * k >= 128 * E)))
    # route, prep, layer, combine | route, prep, gate/up, h quantizer, down, combine | prep, layer
    launches_per_layer = (6 if f8 else 4) if grouped else 2
    kernel = ("k_f8gemm" if f8 else "k_glayer") if grouped else "k_layer"
    h = moe.moe_ffn_create(cfg, local)
    if grouped and wl["act"] in ("e4m3", "e2m1"):
        moe.moe_ffn_set_mma_kind(h, {"auto": moe.MOE_MMA_AUTO, "pieces": moe.MOE_MMA_MXF4_PIECES,
                                     "f8": moe.MOE_MMA_MXF8F6F4}[args.mma])
    nc, ns = synth.expert_sizes(H, I)
    tc = torch.empty(nc, dtype=torch.uint8, device="cuda")
    ts = torch.empty(ns, dtype=torch.uint8, device="cuda")
    sets = []
    for l in range(L):
        es = ExpertSet(h, cfg, device=local)
        for e in range(E):
            synth.device_fill_expert(tc.data_ptr(), ts.data_ptr(), H, I, e, layer=l, seed=0)
            es.load(e, tc, ts)
        sets.append(es)
    torch.cuda.synchronize()
    del tc, ts

    # pre-drawn routings and inputs: R steps (x L layers)
    R = min(500, max(4, 2048 // T)) if L == 1 else 4
    draws = [draw_routings(R, E, k, T, seed=rank, dist=wl["dist"], layer=l) for l in range(L)]
    idx_np = np.stack([d[0] for d in draws], axis=1)          # [R][L][T][k]
    w_np = np.stack([d[1] for d in draws], axis=1)
    x_np = synth.activations_bf16(R * T, H, seed=rank).reshape(R, T, H)
    idx_d = torch.from_numpy(idx_np).cuda()
    w_d = torch.from_numpy(w_np).cuda()
    x_d = torch.from_numpy(x_np.view(np.int16)).cuda()
    stream = torch.cuda.Stream()
    K, W = args.steps, args.warmup
    if L == 1:
        y_d = torch.empty((R, T, H), dtype=torch.float32, device="cuda")

        def fwd(i, s):
            moe.moe_ffn_forward(h, x_d[i], idx_d[i, 0], w_d[i, 0], sets[0].table, y_d[i], T, s)

        def capture(n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    fwd(i % R, torch.cuda.current_stream())
            return g

        chunk = min(K, R)
        g_full = capture(chunk)
        rem = K % chunk
        g_rem = capture(rem) if rem else None

        def timed_steps():
            for _ in range(K // chunk):
                g_full.replay()
            if g_rem is not None:
                g_rem.replay()
    else:
        # the residual: each step starts again from the step's own input
        x0 = x_d.view(torch.bfloat16).float()                  # [R][T][H]
        xs = torch.empty((T, H), dtype=torch.float32, device="cuda")
        tables = [es.table for es in sets]

        def fwd(i, s):
            xs.copy_(x0[i])
            moe.moe_stack_forward(h, xs, tables, idx_d[i], w_d[i], L, T, s)

        chunk = None

        def timed_steps():
            for i in range(K):
                fwd(i % R, stream)

    with torch.cuda.stream(stream):
        for i in range(max(W, R if L > 1 else 0)):       # the stack captures one graph per routing
            fwd(i % R, stream)
    stream.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- timed region: exactly K steps
    barrier()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        timed_steps()
        ev1.record(stream)
    stream.synchronize()
    clocks = sampler.stop()
    barrier()
    ms_total = ev0.elapsed_time(ev1)
    ms_total = max_over_ranks(ms_total, dist, "cuda")
    ms_step = ms_total / K
    value = replica_throughput(world, T, K, ms_total)

    # algorithmic bytes: distinct experts per layer per step x bytes per expert + activations
    def distinct(i, l):
        return len(set(int(v) for v in idx_np[i % R, l].reshape(-1)))

    act_io = T * H * 2 + T * H * 4 + 2 * T * k * 4
    bytes_step = sum(distinct(i, l) for i in range(K) for l in range(L)) / K * expert_bytes(H, I) + L * act_io
    gbs_step = bytes_step / (ms_step / 1000.0) / 1e9

    # ---- dominant kernel (k_layer: both projections) timed with CUDA events on its
    # stream: single-layer forwards (layer 0 of the workload) in profiling mode
    peak, peak_kind = peaks()
    yp = torch.empty((T, H), dtype=torch.float32, device="cuda")
    moe.moe_ffn_profile_enable(h, True)
    nprof = min(K * L, 2000 if T == 1 else 50)
    with torch.cuda.stream(stream):
        for i in range(nprof):
            moe.moe_ffn_forward(h, x_d[i % R], idx_d[i % R, 0], w_d[i % R, 0], sets[0].table, yp, T, stream)
    stream.synchronize()
    ms_ph, n_ph = moe.moe_ffn_profile_read(h)
    moe.moe_ffn_profile_enable(h, False)
    # the layer's MMA kernel time per forward (the kind::mxf8f6f4 path: its two launches)
    ly_ms = ms_ph[moe.MOE_PHASE_GATE_UP] / max(1, n_ph[moe.MOE_PHASE_GATE_UP] // (2 if f8 else 1))
    pr_ms = ms_ph[moe.MOE_PHASE_PREP] / max(1, n_ph[moe.MOE_PHASE_PREP])
    ro_ms = ms_ph[moe.MOE_PHASE_ROUTE] / max(1, n_ph[moe.MOE_PHASE_ROUTE])
    co_ms = ms_ph[moe.MOE_PHASE_DOWN] / max(1, n_ph[moe.MOE_PHASE_DOWN])
    ly_bytes = sum(distinct(i, 0) for i in range(nprof)) / nprof * expert_bytes(H, I) + act_io
    # the same kernel inside a step: on the slot-major path, a CUDA graph of
    # layer-kernel launches back to back (measurement mode: the layer kernel
    # alone, on the pieces of the last full call; each launch overlaps the
    # previous one's tail as programmatic dependent launch lets it, as in a
    # step), the routings cycling as in the timed steps.  The profiling events
    # above separate the launches (no overlap), so they read longer.
    ly_graph_ms = None
    if not grouped:
        nlg = 200 if T == 1 else 20
        with torch.cuda.stream(stream):
            moe.moe_ffn_forward(h, x_d[0], idx_d[0, 0], w_d[0, 0], sets[0].table, yp, T, stream)
        stream.synchronize()
        moe.moe_ffn_profile_layer_only(h, True)
        # launch i: routing (i / L) mod R of layer i mod L (a stack's layers have
        # weights of their own, so no two consecutive launches share an expert)
        lg = [((i // L) % R, i % L) for i in range(nlg)]
        g_l = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_l, stream=stream):
            for r_, l_ in lg:
                moe.moe_ffn_forward(h, x_d[0], idx_d[r_, l_], w_d[r_, l_], sets[l_].table, yp, T, stream)
        moe.moe_ffn_profile_layer_only(h, False)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_l.replay()
            evl0, evl1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            evl0.record(stream)
            for _ in range(5):
                g_l.replay()
            evl1.record(stream)
        stream.synchronize()
        ly_graph_ms = evl0.elapsed_time(evl1) / (5 * nlg)
        del g_l
        lg_bytes = sum(distinct(r_, l_) for r_, l_ in lg) / nlg * expert_bytes(H, I) + act_io
        achieved = lg_bytes / (ly_graph_ms / 1000.0) / 1e9
    else:
        achieved = ly_bytes / (ly_ms / 1000.0) / 1e9
    traffic = traffic_record(kernel, args.workload, wl["act"], ly_bytes)
    tensor = None
    if wl.get("bound") == "tensor":
        # the two projections' MMA flops per forward over the layer kernels' time,
        # against the dense rate of the MMA's kind (E4M3 x E2M1: kind::mxf8f6f4,
        # the fp8 rate; E2M1 x E2M1: kind::mxf4, the fp4 rate), derived from the
        # measured bf16 rate by the nominal ratios
        flops = 2.0 * T * k * 3 * H * I
        bf16, bf16_kind = tensor_peak_bf16()
        tf = flops / (ly_ms / 1000.0) / 1e12
        rate = FP4_PER_BF16 if wl["act"] == "e2m1" else FP8_PER_BF16
        tensor = {"bound": "tensor", "kernel": kernel, "achieved": tf, "peak": bf16 * rate,
                  "peak_kind": f"{bf16_kind} bf16 {bf16:.1f} TFLOP/s x {rate:g} (nominal ratio of the MMA kind)",
                  "unit": "TFLOP/s", "frac": tf / (bf16 * rate),
                  "frac_of_fp4_peak": tf / (bf16 * FP4_PER_BF16),
                  "flops_per_launch": flops, "traffic": None,
                  "timing": f"events around each launch (launches separated): {ly_ms * 1e3:.2f} us per forward"}

    # ---- the router ahead of the path (logits = W x, top-k, softmax): one
    # launch per call up to 8 tokens, two above; timed (a) back to back in a CUDA graph of nrg calls,
    # as a decode step would run it, and (b) alone, events around each call
    Wr = torch.from_numpy(synth.router_weights_bf16(E, H).view(np.int16)).cuda()
    r_idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    r_w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    # distinct router matrices, 256 MB in all (> L2), so that each call reads its weights from HBM
    nrg = max(2, -(-256 * 2 ** 20 // (E * H * 2)))
    gen = torch.Generator(device="cuda").manual_seed(7)
    Wrs = torch.randn((nrg, E, H), generator=gen, device="cuda").to(torch.bfloat16).view(torch.int16)
    with torch.cuda.stream(stream):
        moe.moe_router_topk(h, x_d[0], Wr, T, r_idx, r_w, stream=stream)     # warm-up outside capture
    stream.synchronize()
    def router_graph_us():
        g_r = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_r, stream=stream):
            for i in range(nrg):
                moe.moe_router_topk(h, x_d[i % R], Wrs[i], T, r_idx, r_w, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_r.replay()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(10):
                g_r.replay()
            ev1.record(stream)
        stream.synchronize()
        return ev0.elapsed_time(ev1) * 1e3 / (10 * nrg)

    r_us_graph = router_graph_us()
    # (d) with the handle's layer kernels reading the routing after their
    # dependency wait (moe_ffn_set_routing_wait), the router lets the next
    # launch start at once
    moe.moe_ffn_set_routing_wait(h, 1)
    r_us_graph_rel = router_graph_us()
    moe.moe_ffn_set_routing_wait(h, 0)
    del Wrs
    moe.moe_ffn_profile_enable(h, True)
    nrt = 200
    with torch.cuda.stream(stream):
        for i in range(nrt):
            moe.moe_router_topk(h, x_d[i % R], Wr, T, r_idx, r_w, stream=stream)
    stream.synchronize()
    ms_r, n_r = moe.moe_ffn_profile_read(h)
    moe.moe_ffn_profile_enable(h, False)
    r_us = ms_r[moe.MOE_PHASE_ROUTER] / max(1, n_r[moe.MOE_PHASE_ROUTER]) * 1e3
    r_bytes = E * H * 2 + T * H * 2 + 2 * T * E * 4 + T * k * 8     # W, x, logits out and back, routing
    # (c) inside a decode step: 40 layers of (router -> layer on the router's
    # routing), each layer with router weights of its own, against the same 40
    # layer calls on the pre-drawn routings, both one CUDA graph; the difference
    # per layer is what the router adds to a step (its launch and weight loads
    # overlap the previous layer's kernel as programmatic dependent launch allows)
    r_in_step = r_in_step_rel = None
    if T <= 8:
        nl = 40
        Wl = torch.randn((nl, E, H), generator=gen, device="cuda").to(torch.bfloat16).view(torch.int16)
        ri = torch.empty((nl, T, k), dtype=torch.int32, device="cuda")
        rw = torch.empty((nl, T, k), dtype=torch.float32, device="cuda")
        yl = torch.empty((T, H), dtype=torch.float32, device="cuda")

        def step_graph(mode):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(nl):
                    l_ = i % L
                    if mode == "router":      # the router call, then the layer call on its routing
                        moe.moe_router_topk(h, x_d[i % R], Wl[i], T, ri[i], rw[i], stream=stream)
                        moe.moe_ffn_forward(h, x_d[i % R], ri[i], rw[i], sets[l_].table, yl, T, stream)
                    else:
                        moe.moe_ffn_forward(h, x_d[i % R], idx_d[i % R, l_], w_d[i % R, l_], sets[l_].table, yl,
                                            T, stream)
            return g

        times = []
        for mode in ("none", "router", "router_rel"):
            moe.moe_ffn_set_routing_wait(h, 1 if mode == "router_rel" else 0)
            g = step_graph("router" if mode == "router_rel" else mode)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(10):
                    g.replay()
                e1.record(stream)
            stream.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / (10 * nl))
            del g
        r_in_step = times[1] - times[0]
        r_in_step_rel = times[2] - times[0]
        moe.moe_ffn_set_routing_wait(h, 0)
        del Wl
    router = {"kernels": ("k_router_cluster (one thread-block cluster: logits, then the selection in its first CTA)"
                          if T == 1 and E <= 256 else
                          "k_router_logits (selection in its last CTA per token tile)") if T <= 8
              else "k_router_mma + k_router_select",
              "us": r_us_graph, "us_alone": r_us, "us_in_step": r_in_step,
              "routing_wait": {"us": r_us_graph_rel, "us_in_step": r_in_step_rel},
              "algorithmic_bytes": r_bytes,
              "gbs": r_bytes / (r_us_graph * 1e-6) / 1e9,
              "frac_of_hbm": r_bytes / (r_us_graph * 1e-6) / 1e9 / peak,
              "launches": 1 if T <= 8 else 2, "timing": f"us: per call, {nrg} calls back to back in a CUDA graph, each on its "
                                       "own router matrix (256 MB in all, > L2); us_alone: events around "
                                       "each call, one matrix; us_in_step: per layer, a graph of 40 "
                                       "(moe_router_topk -> moe_ffn_forward on its routing) pairs less a graph "
                                       "of the same 40 layers on pre-drawn routings; routing_wait: the same two "
                                       "with moe_ffn_set_routing_wait(h, 1) (the layer reads the routing after its "
                                       "dependency wait, so the router releases the next launch at once)"}

    # ---- end to end through the public API from host buffers: every step copies
    # its inputs in from pinned host memory and its result back
    ne2e = min(K, 2000 if T * L == 1 else 20)
    xh = torch.from_numpy(x_np.view(np.int16)).pin_memory()
    ih = torch.from_numpy(idx_np).pin_memory()
    wh = torch.from_numpy(w_np).pin_memory()
    yh = torch.empty((T, H), dtype=torch.float32).pin_memory()
    if L == 1:
        # the host addresses of each step's inputs, taken once (tensor views cost microseconds)
        xp = [xh[i].data_ptr() for i in range(R)]
        ip = [ih[i, 0].data_ptr() for i in range(R)]
        wp = [wh[i, 0].data_ptr() for i in range(R)]
        yp, tb0, sp = yh.data_ptr(), sets[0].table, stream.cuda_stream

        def e2e_step(i):
            moe.moe_ffn_forward_host(h, xp[i], ip[i], wp[i], tb0, yp, T, sp)
        h2d = T * H * 2 + 2 * T * k * 4
    else:
        # the residual of each step in host memory (fp32, updated in place by the
        # call), reset from the step's input before every call
        tables = [es.table for es in sets]
        x32 = (x_np.view(np.uint16).astype(np.uint32) << 16).view(np.float32)      # bf16 -> fp32, exact
        xw = torch.empty((T, H), dtype=torch.float32).pin_memory()
        xw_np = xw.numpy()
        ih_np = [np.ascontiguousarray(idx_np[i]) for i in range(R)]
        wh_np = [np.ascontiguousarray(w_np[i]) for i in range(R)]
        xwp, sp = xw.data_ptr(), stream.cuda_stream

        def e2e_step(i):
            np.copyto(xw_np, x32[i])
            moe.moe_stack_forward_host(h, xwp, tables, ih_np[i].ctypes.data, wh_np[i].ctypes.data, L, T, sp)
        h2d = T * H * 4 + 2 * L * T * k * 4
    for i in range(3):
        e2e_step(i % R)
    t0 = time.perf_counter()
    for i in range(ne2e):
        e2e_step(i % R)
    e2e_s = time.perf_counter() - t0
    e2e_value = world * T * ne2e / e2e_s
    status = moe.moe_ffn_status(h, stream)
    assert status == moe.MOE_OK, moe.strerror(status)

    cpu = None
    if rank == 0 and not args.no_cpu:
        v, thr, sample = cpu_sample(wl)
        cpu = {"value": v, "unit": "tokens/s", "cores": thr, "kind": "oracle", "sample": sample}

    if rank == 0:
        resident = L * E * expert_bytes(H, I) / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": {"e4m3": "e4m3xe2m1->f32", "e2m1": "e2m1xe2m1->f32"}.get(wl["act"], "bf16xe2m1->f32"),
            "data": "synthetic",
            "config": {"workload": args.workload, "layers": L, "experts": E, "hidden": H, "inter": I,
                       "topk": k, "tokens_per_step": T, "routing": wl["dist"], "activations": wl["act"],
                       "path": ("expert-major, kind::mxf8f6f4" if f8 else "expert-major (grouped)")
                       if grouped else "slot-major",
                       "parallelism": f"replicas{world}",
                       "l2": f"inputs larger than L2: {resident:.1f} GB resident experts"
                             + (", consecutive steps share no expert" if T == 1 and L == 1 else ""),
                       "graph_chunk": chunk,
                       "distinct_experts_per_layer_step": round(
                           sum(distinct(i, l) for i in range(R) for l in range(L)) / (R * L), 2)},
            "hbm_gbs": gbs_step, "hbm_frac": gbs_step / peak,
            "per_layer": {"us": ms_step / L * 1e3, "tokens_s": value * L} if L > 1 else None,
            "bytes_per_step": bytes_step,
            "phase_us": {"route": ro_ms * 1e3, "prep": pr_ms * 1e3, "layer": ly_ms * 1e3,
                         "combine": co_ms * 1e3},
            "roofline": tensor if tensor is not None else {"bound": "hbm", "kernel": kernel, "achieved": achieved,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "algorithmic_bytes_per_launch": ly_bytes,
                         "timing": ("in a CUDA graph of layer-kernel launches back to back, "
                                    f"{ly_graph_ms * 1e3:.2f} us per launch; with events around each launch "
                                    f"(launches separated) {ly_ms * 1e3:.2f} us")
                         if ly_graph_ms is not None else
                         f"events around each launch (launches separated): {ly_ms * 1e3:.2f} us"},
            "router": router,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": T * H * 4},
            "gpu_launches": launches_per_layer * K * L,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    moe.moe_ffn_destroy(h)
    if dist is not None:
        dist.destroy_process_group()


def run_host_experts(args, wl):
    """One layer whose experts live in page-locked host memory, served by the
    HBM expert cache (moe_expert_cache_*): per step fetch (copies of the misses
    over NVLink-C2C), the layer, and -- with a predictor -- a prefetch of the
    experts guessed for the next step (each of them right with probability
    `guess`, else a random expert)."""
    import numpy as np
    import torch

    import fp4_block_scaled_gb300 as moe
    import synth
    from fp4_block_scaled_gb300.experts import ExpertSet

    if args.gpus != 1 or int(os.environ.get("WORLD_SIZE", "1")) != 1:
        raise SystemExit("the host-resident workloads run on one GPU")
    torch.cuda.set_device(0)
    E, H, I, k, T = wl["E"], wl["H"], wl["I"], wl["k"], wl["T"]
    cfg = moe.config(E, H, I, k, T, out_dtype=moe.MOE_OUT_F32)
    h = moe.moe_ffn_create(cfg, 0)
    stage = ExpertSet(h, cfg, num_experts=1)
    host = torch.empty(E * stage.stride, dtype=torch.uint8, pin_memory=True)
    nc, ns = synth.expert_sizes(H, I)
    tc = torch.empty(nc, dtype=torch.uint8, device="cuda")
    ts = torch.empty(ns, dtype=torch.uint8, device="cuda")
    for e in range(E):
        synth.device_fill_expert(tc.data_ptr(), ts.data_ptr(), H, I, e, layer=0, seed=0)
        stage.load(0, tc, ts)
        host[e * stage.stride:(e + 1) * stage.stride].copy_(stage.blobs)
    torch.cuda.synchronize()
    del tc, ts
    c = moe.moe_expert_cache_create(cfg, 0, [host.data_ptr() + e * stage.stride for e in range(E)], wl["slots"])

    K, W = args.steps, args.warmup
    n = K + W + 1
    idx_np, w_np = draw_routings(n, E, k, T, seed=0)
    rng = np.random.default_rng(1)
    guesses = []
    for i in range(n):
        g = idx_np[i].reshape(-1).copy()
        for j in range(g.size):
            if rng.random() >= wl["guess"]:
                g[j] = rng.integers(0, E)
        guesses.append(g)
    x_np = synth.activations_bf16(n * T, H, seed=0).reshape(n, T, H)
    idx_d = torch.from_numpy(idx_np).cuda()
    w_d = torch.from_numpy(w_np).cuda()
    x_d = torch.from_numpy(x_np.view(np.int16)).cuda()
    y_d = torch.empty((T, H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def step(i):
        tbl = moe.moe_expert_cache_fetch(c, idx_np[i], stream)
        moe.moe_ffn_forward(h, x_d[i], idx_d[i], w_d[i], tbl, y_d, T, stream)
        if wl["guess"] > 0:
            moe.moe_expert_cache_prefetch(c, guesses[i + 1], stream)

    with torch.cuda.stream(stream):
        for i in range(W):
            step(i)
    stream.synchronize()
    h0, m0, b0 = moe.moe_expert_cache_stats(c)
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(W, W + K):
            step(i)
        ev1.record(stream)
    stream.synchronize()
    clocks = sampler.stop()
    ms_total = ev0.elapsed_time(ev1)
    h1, m1, b1 = moe.moe_expert_cache_stats(c)
    status = moe.moe_ffn_status(h, stream)
    assert status == moe.MOE_OK, moe.strerror(status)
    ms_step = ms_total / K
    copied = b1 - b0
    h2d_gbs = copied / (ms_total / 1000.0) / 1e9

    # host -> device copy peak on this machine: one 1 GiB page-locked copy
    big_h = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    big_d = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        big_d.copy_(big_h, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(4):
        big_d.copy_(big_h, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    h2d_peak = 4 * (1 << 30) / (e0.elapsed_time(e1) / 1000.0) / 1e9
    del big_h, big_d

    # end to end from host buffers (inputs in, y out) with the cache
    xh = torch.from_numpy(x_np.view(np.int16)).pin_memory()
    ih = torch.from_numpy(idx_np).pin_memory()
    wh = torch.from_numpy(w_np).pin_memory()
    yh = torch.empty((T, H), dtype=torch.float32).pin_memory()
    ne2e = min(K, 100)
    t0 = time.perf_counter()
    for i in range(ne2e):
        tbl = moe.moe_expert_cache_fetch(c, idx_np[i], stream)
        moe.moe_ffn_forward_host(h, xh[i], ih[i], wh[i], tbl, yh, T, stream)
        if wl["guess"] > 0:
            moe.moe_expert_cache_prefetch(c, guesses[i + 1], stream)
    e2e_value = T * ne2e / (time.perf_counter() - t0)

    cpu = None
    if not args.no_cpu:
        v, thr, sample = cpu_sample(wl)
        cpu = {"value": v, "unit": "tokens/s", "cores": thr, "kind": "oracle", "sample": sample}
    line = {
        "metric": METRIC, "value": T * K / (ms_total / 1000.0), "unit": "tokens/s", "n_gpus": 1, "steps": K,
        "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16xe2m1->f32", "data": "synthetic",
        "config": {"workload": args.workload, "layers": 1, "experts": E, "hidden": H, "inter": I, "topk": k,
                   "tokens_per_step": T, "routing": "uniform, consecutive steps share no expert",
                   "activations": "bf16", "path": "slot-major", "parallelism": "replicas1",
                   "experts_resident": f"page-locked host memory ({E * expert_bytes(H, I) / 1e9:.1f} GB), "
                                       f"{wl['slots']} cached in HBM",
                   "l2": "inputs larger than L2: every step copies its experts in"},
        "host_experts": {"slots": wl["slots"], "prefetch_guess_accuracy": wl["guess"], "hits": h1 - h0,
                         "misses": m1 - m0, "copied_gb": copied / 1e9, "h2d_gbs": h2d_gbs,
                         "h2d_peak_gbs": h2d_peak, "h2d_frac": h2d_gbs / h2d_peak},
        "roofline": {"bound": "h2d", "kernel": "host-to-device expert copies (copy engines)",
                     "achieved": h2d_gbs, "peak": h2d_peak,
                     "peak_kind": "measured in this run: 1 GiB page-locked host-to-device copies",
                     "unit": "GB/s", "frac": h2d_gbs / h2d_peak, "traffic": None},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2 + 2 * T * k * 4,
                "d2h_bytes_per_step": T * H * 4},
        "gpu_launches": 2 * K,
        "clocks": clocks,
    }
    print(json.dumps(line))
    moe.moe_expert_cache_destroy(c)
    moe.moe_ffn_destroy(h)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: per workload)")
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="stack_b1")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle cpu_baseline leg")
    ap.add_argument("--path", choices=["auto", "slot", "group"], default="auto",
                    help="layer path: the library's choice for T, or forced slot-major / expert-major")
    ap.add_argument("--act", choices=["bf16", "e4m3", "e2m1"], default=None,
                    help="activation numerics (default: the workload's)")
    ap.add_argument("--mma", choices=["auto", "pieces", "f8"], default="auto",
                    help="quantized modes' expert-major form: the library's choice (auto), the activations "
                         "as they are (f8: kind::mxf8f6f4 for E4M3, kind::mxf4 for E2M1) or E2M1 pieces")
    args = ap.parse_args()
    wl = dict(WORKLOADS[args.workload])
    if args.act:
        wl["act"] = args.act
    if args.steps is None:
        args.steps = wl["steps"] if args.impl == "ours" else 10
    if args.warmup is None:
        args.warmup = 50 if args.impl == "ours" else 3
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args, wl)
    elif wl.get("host"):
        run_host_experts(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
