#!/usr/bin/env python3
"""Benchmark of the InfLLM v2 sparse-attention hot path on GB300.

Headline: single-token decode at 128K context, batch 4 (32 query / 2 KV heads,
head dim 128, 64-token blocks, top-64 + 1 initial + 2 local blocks) -- the
workload "decode_128k_b4".  One step is one call of infllmv2_decode: block
scoring over the cached semantic kernels, top-k selection, split-KV attention
over the selected blocks and the merge of the splits, for the 4 sequences.
The semantic-kernel cache is resident (pooled once before timing), as the
workload states; Q, K/V and kernels are synthetic (seeded N(0,1) bf16 with
planted blocks).  Inputs are larger than L2: eight replicas of Q, the K/V
caches and the kernel cache sit at distinct addresses and the steps cycle
through them, so no step finds its data in L2 (8 x 34.4 MB touched per cycle
against a 129 MB L2).  The K timed steps run back to back, as a CUDA graph of
eight steps replayed, between two CUDA events on the launching stream; the
single-step latency with L2 flushed before the step is reported beside it.

Also reported: the 32K-context chunked prefill (4096 queries, block 128,
top-16) as "prefill", the per-kernel stage times, the roofline of the
dominant kernel, an end-to-end number through the C ABI with host buffers,
and the fp64 CPU oracle's throughput on a bounded sample.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica (the path
shards by sequence with no exchange); value = all ranks' query tokens over
the slowest rank's time.
"""
from __future__ import annotations

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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse-attn query tok/s at 128K ctx; % of HBM / tensor-core roofline"
UNIT = "query tok/s"
HEADLINE = "decode_128k_b4"
PREFILL = "chunked_prefill_32k"
FLUSH_BYTES = 1 << 30


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--prefill-steps", type=int, default=20)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--replicas", type=int, default=REPLICAS,
                    help="copies of the decode inputs cycled step by step (fewer: a smaller footprint for "
                         "profiler captures; the timed steps then find their inputs in L2)")
    ap.add_argument("--no-decode", action="store_true",
                    help="profiling aid: run only the chunked-prefill part (no headline value)")
    return ap.parse_args()


def max_over_ranks(value: float, world: int, device: str = "cuda") -> float:
    """The largest of the ranks' values (the job's time is its slowest rank's): an all-reduce
    over the default process group on `device` (the GPU under NCCL, "cpu" under gloo)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) of this GPU's clocks and throttle reasons."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        import torch
        self.proc = None
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        props = torch.cuda.get_device_properties(device)
        self.bus = None
        try:
            self.bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
        except AttributeError:
            pass

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.bus:
            cmd.insert(1, f"--id={self.bus}")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names[1:], parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ helpers

def dev_bf16(a):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def source_sha(*names) -> str:
    h = hashlib.sha1()
    for n in names:
        with open(os.path.join(ROOT, "block_sparse_long_infllm_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def ncu_traffic(kernel: str, sha: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was
    taken on the current source (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and parts[0] == kernel and parts[1] == sha:
                return float(parts[2])
    return None


class Flusher:
    def __init__(self):
        import torch
        self.buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def __call__(self):
        self.buf.fill_(1)


# ------------------------------------------------------------------ decode (headline)

REPLICAS = 8  # distinct copies of the workload's tensors, cycled step by step


def setup_decode(name: str, replicas: int = REPLICAS):
    """The workload, pooled once, plus replicas-1 copies of every per-step input
    (Q, K/V caches, kernel cache) at distinct addresses: consecutive steps never
    find their data in L2 (8 x 34.4 MB touched per cycle > 2 x the 129 MB L2)."""
    import torch

    from block_sparse_long_infllm_gb300 import infllmv2, synth
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w)
    p = w.params()
    d = dict(w=w, inp=inp, p=p)
    q = dev_bf16(inp["q"])
    k = dev_bf16(inp["k_cache"])
    v = dev_bf16(inp["v_cache"])
    d["kv_len"] = torch.from_numpy(inp["kv_len"]).cuda()
    M = (w.L - w.kernel_size) // w.kernel_stride + 1
    kern = torch.zeros((w.B, w.Hkv, M, w.d), dtype=torch.bfloat16, device="cuda")
    infllmv2.kernel_pool(k, kern, 0, w.L, p)   # resident kernel cache (not timed)
    d["rep"] = [dict(q=q, k=k, v=v, kern=kern)]
    for _ in range(replicas - 1):
        d["rep"].append(dict(q=q.clone(), k=k.clone(), v=v.clone(), kern=kern.clone()))
    d["o"] = torch.empty_like(q)
    d["lse"] = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device="cuda")
    d["ws"] = torch.empty(infllmv2.workspace_size(infllmv2.ENTRY_DECODE, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, p),
                          dtype=torch.uint8, device="cuda")
    S_cap = infllmv2.selection_capacity(p, w.L_max)
    d["idx"] = torch.empty((w.B, w.Hkv, w.Tq, S_cap), dtype=torch.int32, device="cuda")
    d["counts"] = torch.empty((w.B, w.Hkv, w.Tq), dtype=torch.int32, device="cuda")
    return d


def decode_call(d, r: int = 0, q=None, kv_len=None, selection: bool = False):
    """One decode step: o and lse.  With selection=True the step also writes the block lists
    (idx, counts), which the timed steps do not ask for."""
    from block_sparse_long_infllm_gb300 import infllmv2
    rep = d["rep"][r % len(d["rep"])]
    infllmv2.decode(rep["q"] if q is None else q, rep["k"], rep["v"], rep["kern"],
                    d["kv_len"] if kv_len is None else kv_len, d["o"], d["ws"], d["p"], lse=d["lse"],
                    idx_out=d["idx"] if selection else None, counts_out=d["counts"] if selection else None)


def decode_algorithmic_bytes(d) -> dict:
    """Bytes each stage must move at least: the kernel-cache scan (score) and the
    selected K/V blocks (attend), from the selection the step made."""
    w = d["w"]
    M = (w.L - w.kernel_size) // w.kernel_stride + 1
    kern_bytes = w.B * w.Hkv * M * w.d * 2
    q_bytes = w.B * w.Tq * w.Hq * w.d * 2
    counts = d["counts"].cpu().numpy()
    # selected tokens: whole blocks except a partial last block past kv_len
    idx = d["idx"].cpu().numpy()
    L = int(d["kv_len"][0].item())
    toks = 0
    for b in range(w.B):
        for g in range(w.Hkv):
            for t in range(w.Tq):
                blks = idx[b, g, t, :counts[b, g, t]]
                toks += int(sum(min(w.block_size, L - int(x) * w.block_size) for x in blks))
    kv_bytes = toks * w.d * 2 * 2
    return dict(score=kern_bytes + q_bytes, attend=kv_bytes + q_bytes, topk=0, combine=0,
                total=kern_bytes + kv_bytes + 2 * q_bytes, kernel_cache=kern_bytes, selected_kv=kv_bytes)


def capture_graph(step, n: int):
    """One CUDA graph holding step(0), ..., step(n-1) (the launch path warmed outside capture)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for r in range(n):
            step(r)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for r in range(n):
            step(r)
    torch.cuda.synchronize()
    return g


class StepGraphs:
    """Exactly K steps back to back: a graph of one step per replica (R steps) replayed K // R
    times, then a graph of the first K % R replicas' steps, so the step count is the one asked
    for and every step still runs on the next replica's inputs."""

    def __init__(self, step, R: int, K: int):
        self.full = capture_graph(step, R) if K >= R else None
        self.n_full = K // R
        self.tail = capture_graph(step, K % R) if K % R else None

    def replay(self):
        for _ in range(self.n_full):
            self.full.replay()
        if self.tail is not None:
            self.tail.replay()


def run_decode(args, world, rank):
    import torch

    from block_sparse_long_infllm_gb300 import infllmv2
    d = setup_decode(HEADLINE, replicas=max(1, args.replicas))
    w = d["w"]
    R = len(d["rep"])
    stream = torch.cuda.current_stream()
    for i in range(max(args.warmup, 3)):
        decode_call(d, i)
    torch.cuda.synchronize()
    if infllmv2.sync_status() != 0:
        raise RuntimeError("device error during warm-up")
    # ---- timed region: exactly K steps back to back (graphs of R steps replayed), each step on the
    # next replica so no step finds its inputs in L2
    K = max(1, args.steps)
    graphs = StepGraphs(lambda r: decode_call(d, r), R, K)
    graphs.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_wall = time.perf_counter()
    ev0.record(stream)
    graphs.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    total_ms = ev0.elapsed_time(ev1)
    total_ms = max_over_ranks(total_ms, world)
    status = infllmv2.sync_status()

    # ---- the same K steps launched one call at a time (no graph)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_ng = min(K, 2000)
    torch.cuda.synchronize()
    a.record(stream)
    for i in range(n_ng):
        decode_call(d, i)
    b.record(stream)
    torch.cuda.synchronize()
    nograph_ms = a.elapsed_time(b) / n_ng
    # the same, each step also writing its block lists (an optional output of the call)
    a.record(stream)
    for i in range(n_ng):
        decode_call(d, i, selection=True)
    b.record(stream)
    torch.cuda.synchronize()
    nograph_sel_ms = a.elapsed_time(b) / n_ng

    # ---- stage times: library stage events around each kernel, replicas cycled
    stage_n = min(K, 400)
    infllmv2.profile_enable(True)
    stages: dict[str, list[float]] = {}
    for i in range(stage_n):
        decode_call(d, i)
        for name, ms in infllmv2.profile_read():
            stages.setdefault(name, []).append(ms)
    infllmv2.profile_enable(False)
    stage_ms = {k: statistics.median(v) for k, v in stages.items()}

    # ---- single-step latency with L2 flushed before the step
    flush = Flusher()
    lat = []
    for i in range(50):
        flush()
        a.record(stream)
        decode_call(d, i)
        b.record(stream)
        torch.cuda.synchronize()
        lat.append(a.elapsed_time(b))
    del flush

    decode_call(d, 0, selection=True)  # the selection the steps make, for the algorithmic bytes
    torch.cuda.synchronize()
    alg = decode_algorithmic_bytes(d)
    pk = peaks()
    fused = "fused" in stage_ms
    if fused:
        # one kernel per step (scores, selection, attention, merge): its average launch duration
        # is the timed region's device time over the K launches it holds
        dom = "fused"
        achieved = alg["total"] / (total_ms / K * 1e-3) / 1e9
        alg = dict(alg, fused=alg["total"])
        src = "decode_cluster.cu"
    else:
        dom = max(("score", "attend"), key=lambda s: stage_ms.get(s, 0.0))
        achieved = alg[dom] / (stage_ms[dom] * 1e-3) / 1e9
        src = "select.cu" if dom == "score" else "decode.cu"
    kernel_names = {"score": "score_decode_kernel", "attend": "decode_split_kernel", "fused": "decode_cluster_kernel"}
    sha = source_sha(src, "attn_warp.cuh", "common.cuh", "tma.cuh")
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": ncu_traffic(kernel_names[dom], sha),
                "kernel": kernel_names[dom], "algorithmic_bytes": alg[dom], "peak_source": pk["source"],
                "timing": ("device time of the timed region (CUDA events on the launching stream) / launches; "
                           f"one launch per step; event-bracketed single launch: {stage_ms.get('fused', 0.0) * 1e3:.1f} us"
                           if fused else "median stage time between the library's CUDA events on the launching stream")}
    step_ms = total_ms / K
    step_alg_gbs = alg["total"] / (step_ms * 1e-3) / 1e9

    out = dict(metric=METRIC, value=None, unit=UNIT, n_gpus=world, steps=K, warmup=args.warmup,
               ms_per_step=step_ms, higher_is_better=True, scaling="weak", vs_baseline=None,
               dtype="bf16", data="synthetic (seeded N(0,1) bf16, planted blocks)",
               config={"workload": HEADLINE, "batch": w.B, "kv_len": w.L, "q_heads": w.Hq, "kv_heads": w.Hkv,
                       "head_dim": w.d, "block_size": w.block_size, "kernel": [w.kernel_size, w.kernel_stride],
                       "topk": w.topk, "n_init": w.n_init, "n_local": w.n_local, "dense_len": w.dense_len,
                       "parallelism": f"replicas x{world}",
                       "l2": (f"inputs larger than L2: {R} replicas of Q, K/V and kernel caches cycled step by step "
                              f"({R} x {alg['total'] / 1e6:.1f} MB touched per cycle)" if R * alg["total"] > 2 * 129e6
                              else f"{R} replica(s): the steps find their inputs in L2 (a profiling run, not the "
                                   f"benchmark)"),
                       "launch": (f"exactly {K} steps: a CUDA graph of one step per replica ({R} steps) replayed "
                                  f"{K // R} times, then a graph of the first {K % R}; " +
                                  ("one cluster kernel per step (one thread-block cluster per row, the largest size whose "
                                   "clusters all fit the device: 12 CTAs for 8 rows on a GB300)" if fused else
                                   "kernels chained with programmatic dependent launch")),
                       "kernel_cache": "resident (pooled before timing)",
                       "outputs": "o and lse per step; the block lists are an optional output the timed steps "
                                  "do not ask for (step.no_graph_with_block_lists_ms_per_step times them)"},
               roofline=roofline, clocks=clk, gpu_launches=(1 if fused else 4) * K, device_status=status)
    out["value"] = world * w.B * w.Tq * K / (total_ms * 1e-3)
    out["step"] = {"algorithmic_bytes": alg["total"], "kernel_cache_bytes": alg["kernel_cache"],
                   "selected_kv_bytes": alg["selected_kv"], "achieved_gbs": round(step_alg_gbs, 1),
                   "frac_hbm": round(step_alg_gbs / pk["hbm_gbs"], 4), "frac_8tbs": round(step_alg_gbs / 8000, 4),
                   "wall_s": round(t_wall, 3), "no_graph_ms_per_step": round(nograph_ms, 5),
                   "no_graph_with_block_lists_ms_per_step": round(nograph_sel_ms, 5),
                   "latency_ms_l2_flushed": round(statistics.median(lat), 5),
                   "latency_frac_hbm": round(alg["total"] / (statistics.median(lat) * 1e-3) / 1e9 / pk["hbm_gbs"], 4)}
    out["stages_ms"] = {k: round(v, 5) for k, v in stage_ms.items()}
    out["e2e"] = run_decode_e2e(d, n=min(K, 400))
    return out, d


def run_decode_32k(args) -> dict:
    """Single-token decode at 32K context, batch 1 (workload "decode_32k": 64-token blocks, top-64
    + 1 initial + 2 local blocks): exactly K steps back to back in CUDA graphs, each step on the next
    of 48 replicas (48 x 5.5 MB touched per cycle, over twice the L2), and the single-step latency
    with L2 flushed before the step."""
    import torch
    d = setup_decode("decode_32k", replicas=48)
    w = d["w"]
    R = len(d["rep"])
    K = max(1, min(args.steps, 2000))
    for i in range(max(args.warmup, 3)):
        decode_call(d, i)
    graphs = StepGraphs(lambda r: decode_call(d, r), R, K)
    graphs.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    graphs.replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / K
    flush = Flusher()
    lat = []
    for i in range(30):
        flush()
        a.record(stream)
        decode_call(d, i)
        b.record(stream)
        torch.cuda.synchronize()
        lat.append(a.elapsed_time(b))
    del flush
    decode_call(d, 0, selection=True)
    torch.cuda.synchronize()
    from block_sparse_long_infllm_gb300 import infllmv2
    assert infllmv2.sync_status() == 0
    alg = decode_algorithmic_bytes(d)
    pk = peaks()
    lat_ms = statistics.median(lat)
    gbs = alg["total"] / (ms * 1e-3) / 1e9
    return {"workload": "decode_32k", "batch": w.B, "kv_len": w.L, "ms_per_step": ms, "steps": K,
            "value": w.B * w.Tq / (ms * 1e-3), "unit": UNIT, "algorithmic_bytes": alg["total"],
            "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
            "latency_ms_l2_flushed": round(lat_ms, 5),
            "latency_frac_hbm": round(alg["total"] / (lat_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
            "gpu_launches_per_step": 1}


def run_decode_append(args, d) -> dict:
    """The whole decode step of a serving loop through infllmv2_decode_step: append the new
    token's K and V (and pool the semantic kernel it completes) and decode, in the CUDA graph,
    replicas cycled as in the headline.  The appended token is the cache's last row, which completes a kernel: every step
    pays the pooling (the worst case; a kernel completes every 16 tokens)."""
    import numpy as np
    import torch

    from block_sparse_long_infllm_gb300 import infllmv2, synth
    w = d["w"]
    R = len(d["rep"])
    rng = np.random.default_rng(w.seed + 11)
    news = [(dev_bf16(synth.f32_to_bf16_bits(rng.standard_normal((w.B, w.Hkv, w.d)).astype(np.float32))),
             dev_bf16(synth.f32_to_bf16_bits(rng.standard_normal((w.B, w.Hkv, w.d)).astype(np.float32))))
            for _ in range(R)]

    def step(r):
        rep = d["rep"][r % R]
        kn, vn = news[r % R]
        infllmv2.decode_step(rep["q"], kn, vn, rep["k"], rep["v"], rep["kern"], d["kv_len"], d["o"], d["ws"], d["p"],
                             lse=d["lse"])

    K = max(1, min(args.steps, 2000))
    graphs = StepGraphs(step, R, K)
    graphs.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    graphs.replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / K
    infllmv2.profile_enable(True)
    names = set()
    for r in range(8):
        step(r)
        names.update(nm for nm, _ in infllmv2.profile_read())
    infllmv2.profile_enable(False)
    assert infllmv2.sync_status() == 0
    fused = names == {"fused"}
    return {"ms_per_step": ms, "steps": K, "value": w.B * w.Tq / (ms * 1e-3), "unit": UNIT,
            "gpu_launches_per_step": 1 if fused else 2,
            "note": "CUDA graph of infllmv2_decode_step per step (append of the new token's K/V and the kernel it "
                    "completes, then decode" + (", one cluster kernel" if fused else ", append kernel then decode") +
                    "); each step pools a kernel (worst case)"}


def run_decode_e2e(d, n: int) -> dict:
    """Same step through the public host-buffer call (infllmv2_decode_host): each step copies its
    query and lengths from pinned host memory, decodes, copies o and lse back and waits; wall clock
    per step, replicas cycled."""
    import torch

    from block_sparse_long_infllm_gb300 import infllmv2
    w = d["w"]
    q_host = d["rep"][0]["q"].view(w.B, w.Hq, w.d).cpu().pin_memory()
    kv_host = d["kv_len"].cpu().pin_memory()
    o_host = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16).pin_memory()
    lse_host = torch.empty((w.B, w.Hq), dtype=torch.float32).pin_memory()
    q_dev = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    kv_dev = torch.empty_like(d["kv_len"])
    o_dev = torch.empty_like(q_dev)
    lse_dev = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    # one prepared call per replica (static buffers bound once, as a serving loop would)
    steps = [infllmv2.DecodeHostStep(q_host, kv_host, o_host, q_dev, kv_dev, o_dev, rep["k"], rep["v"], rep["kern"],
                                     d["ws"], d["p"], lse_host=lse_host, lse_dev=lse_dev) for rep in d["rep"]]
    times = []
    for i in range(n + 3):
        t0 = time.perf_counter()
        steps[i % len(steps)]()
        if i >= 3:
            times.append(time.perf_counter() - t0)
    h2d = q_host.numel() * q_host.element_size() + kv_host.numel() * kv_host.element_size()
    d2h = o_host.numel() * o_host.element_size() + lse_host.numel() * lse_host.element_size()
    return {"value": w.B * w.Tq / statistics.mean(times), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * statistics.mean(times),
            "note": "wall clock per step of infllmv2_decode_host through the binding's prepared call: q and the "
                    "lengths come from page-locked host memory and o and lse go back to it (the decode kernel "
                    "reads and writes those mapped host buffers directly, over NVLink-C2C on this Grace host: "
                    "one launch, its error word in page-locked host memory, one wait); replicas cycled; KV and "
                    "kernel caches resident"}


# ------------------------------------------------------------------ prefill (secondary)

def run_prefill(args) -> dict:
    import numpy as np
    import torch

    from block_sparse_long_infllm_gb300 import infllmv2, synth
    w = synth.WORKLOADS[PREFILL]
    inp = synth.make_inputs(w)
    p = w.params()
    q, k, v = dev_bf16(inp["q"]), dev_bf16(inp["k_cache"]), dev_bf16(inp["v_cache"])
    kv_len = torch.from_numpy(inp["kv_len"]).cuda()
    M = (w.L - w.kernel_size) // w.kernel_stride + 1
    kern = torch.zeros((w.B, w.Hkv, M, w.d), dtype=torch.bfloat16, device="cuda")
    infllmv2.kernel_pool(k, kern, 0, w.q_pos0, p)     # kernels of the cached prefix (not timed)
    S_cap = infllmv2.selection_capacity(p, w.L_max)
    idx = torch.empty((w.B, w.Hkv, w.Tq, S_cap), dtype=torch.int32, device="cuda")
    cnt = torch.empty((w.B, w.Hkv, w.Tq), dtype=torch.int32, device="cuda")
    ws = torch.empty(infllmv2.workspace_size(infllmv2.ENTRY_BLOCK_SELECT, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, p),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device="cuda")
    flush = Flusher()
    stream = torch.cuda.current_stream()

    def step(record=None):
        infllmv2.kernel_pool(k, kern, w.q_pos0, w.L, p)
        if record is not None:
            record.append(infllmv2.profile_read())
        infllmv2.block_select(q, kern, kv_len, idx, cnt, ws, p, w.L_max)
        if record is not None:
            record.append(infllmv2.profile_read())
        infllmv2.sparse_attn_fwd(q, k, v, idx, cnt, kv_len, o, p, lse=lse)
        if record is not None:
            record.append(infllmv2.profile_read())

    for _ in range(3):
        flush()
        step()
    torch.cuda.synchronize()
    K = args.prefill_steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    infllmv2.profile_enable(True)
    stages: dict[str, list[float]] = {}
    for _ in range(max(3, K // 2)):
        flush()
        rec = []
        step(rec)
        for part in rec:
            for name, t in part:
                stages.setdefault(name, []).append(t)
    infllmv2.profile_enable(False)
    stage_ms = {kk: statistics.median(vv) for kk, vv in stages.items()}

    # algorithmic FLOPs: 4 d per attended (query, head, key) and 2 d per scored (query, head, kernel)
    counts = cnt.cpu().numpy()
    sel = idx.cpu().numpy()
    attended = 0
    scored = 0
    for t in range(w.Tq):
        pos = w.L - w.Tq + t
        vis_kernels = (pos + 1 - w.kernel_size) // w.kernel_stride + 1
        scored += vis_kernels * w.Hq
        for g in range(w.Hkv):
            blks = sel[0, g, t, :counts[0, g, t]].astype(np.int64)
            keys = np.minimum(pos + 1 - blks * w.block_size, w.block_size).clip(min=0).sum()
            attended += int(keys) * (w.Hq // w.Hkv)
    fl_attn = 4.0 * w.d * attended
    fl_score = 2.0 * w.d * scored
    pk = peaks()
    att_tf = fl_attn / (stage_ms["attend"] * 1e-3) / 1e12
    step_tf = (fl_attn + fl_score) / (ms * 1e-3) / 1e12
    backward = run_prefill_backward(args, w, p, q, k, v, o, lse, idx, cnt, kv_len, flush, 10.0 * w.d * attended, pk)
    return {"workload": PREFILL, "value": w.Tq / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "steps": K,
            "stages_ms": {kk: round(vv, 4) for kk, vv in stage_ms.items()},
            "algorithmic_gflop": {"attention": fl_attn / 1e9, "score": fl_score / 1e9},
            "keys_per_query": attended / (w.Tq * w.Hq),
            "roofline": {"bound": "tensor", "kernel": "prefill_tc_kernel", "achieved": round(att_tf, 2),
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(att_tf / pk["bf16_tflops"], 4),
                         "traffic": ncu_traffic("prefill_tc_kernel",
                                                source_sha("prefill_tc.cu", "umma.cuh", "common.cuh", "tma.cuh", "tc_extra.cuh"))},
            "step_tflops": round(step_tf, 2), "step_frac": round(step_tf / pk["bf16_tflops"], 4),
            "gpu_launches": 4 * K, "backward": backward}


def run_prefill_backward(args, w, p, q, k, v, o, lse, idx, cnt, kv_len, flush, flops: float, pk: dict) -> dict:
    """dQ, dK, dV of the chunk's attention through its selection (the trainable sparse attention's
    backward), timed like the forward: L2 flushed before every call, CUDA events on the stream.
    Algorithmic FLOPs: 10 d per attended (query head, key) -- S and dP recomputed, dV, dK, dQ."""
    import numpy as np
    import torch

    from block_sparse_long_infllm_gb300 import infllmv2, synth
    rng = np.random.default_rng(w.seed + 7)
    dout = dev_bf16(synth.f32_to_bf16_bits(rng.standard_normal(tuple(q.shape)).astype(np.float32)))
    dq = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    dk = torch.empty(k.shape, dtype=torch.float32, device="cuda")
    dv = torch.empty(v.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(infllmv2.workspace_size(infllmv2.ENTRY_SPARSE_ATTN_BWD, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max,
                                             p), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        infllmv2.sparse_attn_bwd(q, k, v, o, lse, dout, idx, cnt, kv_len, dq, dk, dv, ws, p)

    for _ in range(3):
        flush()
        call()
    torch.cuda.synchronize()
    K = args.prefill_steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    infllmv2.profile_enable(True)
    stages: dict[str, list[float]] = {}
    for _ in range(max(3, K // 2)):
        flush()
        call()
        for name, t in infllmv2.profile_read():
            stages.setdefault(name, []).append(t)
    infllmv2.profile_enable(False)
    stage_ms = {kk: statistics.median(vv) for kk, vv in stages.items()}
    assert infllmv2.sync_status() == 0
    grad_tf = flops / (stage_ms["bwd_grad"] * 1e-3) / 1e12
    return {"ms_per_call": ms, "calls": K, "stages_ms": {kk: round(vv, 4) for kk, vv in stage_ms.items()},
            "algorithmic_gflop": flops / 1e9, "call_tflops": round(flops / (ms * 1e-3) / 1e12, 2),
            "roofline": {"bound": "tensor", "kernel": "bwd_tc_kernel", "achieved": round(grad_tf, 2),
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(grad_tf / pk["bf16_tflops"], 4),
                         "traffic": ncu_traffic("bwd_tc_kernel",
                                                source_sha("bwd_tc.cu", "umma.cuh", "common.cuh", "tma.cuh"))},
            "gpu_launches_per_call": 6, "memsets_per_call": 4}


# ------------------------------------------------------------------ variable-length batched prefill (secondary)

VARLEN_LENS = [512, 1024, 2048, 4096, 256, 1536, 768, 3072]          # chunk lengths of 8 sequences
VARLEN_KV = [8192, 16384, 32768, 24576, 12000, 20000, 30000, 28000]  # their cache lengths after the chunk


def run_varlen_prefill(args) -> dict:
    """One prefill step of 8 sequences with different chunk lengths, packed into one launch per
    kernel: the chunks' kernels, selection, attention (parameters of the 32K chunked-prefill
    workload; seeded N(0,1) bf16 inputs).  L2 flushed before each step."""
    import numpy as np
    import torch

    from block_sparse_long_infllm_gb300 import infllmv2, synth
    w = synth.WORKLOADS[PREFILL]
    p = w.params()
    B, Hq, Hkv, d, L_max = len(VARLEN_LENS), w.Hq, w.Hkv, w.d, max(VARLEN_KV)
    cu = np.concatenate([[0], np.cumsum(VARLEN_LENS)]).astype(np.int32)
    total = int(cu[-1])
    rng = np.random.default_rng(2024)
    q = dev_bf16(synth.f32_to_bf16_bits(rng.standard_normal((total, Hq, d), dtype=np.float32)))
    k = dev_bf16(synth.f32_to_bf16_bits(rng.standard_normal((B, Hkv, L_max, d), dtype=np.float32)))
    v = dev_bf16(synth.f32_to_bf16_bits(rng.standard_normal((B, Hkv, L_max, d), dtype=np.float32)))
    kv = torch.tensor(VARLEN_KV, dtype=torch.int32, device="cuda")
    cu_d = torch.from_numpy(cu).cuda()
    M = (L_max - w.kernel_size) // w.kernel_stride + 1
    kern = torch.zeros((B, Hkv, M, d), dtype=torch.bfloat16, device="cuda")
    infllmv2.kernel_pool(k, kern, 0, L_max, p)   # the cached prefixes' kernels (not timed)
    S_cap = infllmv2.selection_capacity(p, L_max)
    idx = torch.empty((Hkv, total, S_cap), dtype=torch.int32, device="cuda")
    cnt = torch.empty((Hkv, total), dtype=torch.int32, device="cuda")
    ws = torch.empty(infllmv2.workspace_size(infllmv2.ENTRY_BLOCK_SELECT, 1, total, Hq, Hkv, d, L_max, p),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((Hq, total), dtype=torch.float32, device="cuda")
    Tq_max = max(VARLEN_LENS)
    flush = Flusher()
    stream = torch.cuda.current_stream()

    def step(record=None):
        infllmv2.kernel_pool_varlen(k, kern, kv, cu_d, Tq_max, p)
        if record is not None:
            record.append(infllmv2.profile_read())
        infllmv2.block_select_varlen(q, kern, kv, cu_d, Tq_max, idx, cnt, ws, p, L_max)
        if record is not None:
            record.append(infllmv2.profile_read())
        infllmv2.sparse_attn_fwd_varlen(q, k, v, idx, cnt, kv, cu_d, Tq_max, o, p, lse=lse)
        if record is not None:
            record.append(infllmv2.profile_read())

    for _ in range(3):
        flush()
        step()
    torch.cuda.synchronize()
    K = args.prefill_steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    infllmv2.profile_enable(True)
    stages: dict[str, list[float]] = {}
    for _ in range(max(3, K // 2)):
        flush()
        rec = []
        step(rec)
        for part in rec:
            for nm, t in part:
                stages.setdefault(nm, []).append(t)
    infllmv2.profile_enable(False)
    assert infllmv2.sync_status() == 0
    counts, sel = cnt.cpu().numpy(), idx.cpu().numpy()
    attended = 0
    G = Hq // Hkv
    for b in range(B):
        for t in range(VARLEN_LENS[b]):
            pos = VARLEN_KV[b] - VARLEN_LENS[b] + t
            for g in range(Hkv):
                blks = sel[g, cu[b] + t, :counts[g, cu[b] + t]].astype(np.int64)
                attended += int(np.minimum(pos + 1 - blks * w.block_size, w.block_size).clip(min=0).sum()) * G
    stage_ms = {kk: statistics.median(vv) for kk, vv in stages.items()}
    att_tf = 4.0 * d * attended / (stage_ms["attend"] * 1e-3) / 1e12
    pk = peaks()
    return {"sequences": B, "chunk_lengths": VARLEN_LENS, "kv_lengths": VARLEN_KV, "query_tokens": total,
            "ms_per_step": ms, "steps": K, "value": total / (ms * 1e-3), "unit": UNIT,
            "stages_ms": {kk: round(vv, 4) for kk, vv in stage_ms.items()},
            "attention_tflops": round(att_tf, 2), "attention_frac": round(att_tf / pk["bf16_tflops"], 4),
            "gpu_launches_per_step": 4}


# ------------------------------------------------------------------ tree verification (secondary)

def run_tree(args, name: str, **scale) -> dict:
    """Verification of a draft tree (one call scores, selects and attends for every draft),
    timed with the L2 flushed before each call.  Algorithmic bytes: the kernel cache once per
    (sequence, KV head), K and V of the union of the drafts' selected blocks once, the drafts'
    own K and V."""
    import numpy as np
    import torch

    from block_sparse_long_infllm_gb300 import infllmv2, synth
    w = synth.WORKLOADS[name].scaled(**scale) if scale else synth.WORKLOADS[name]
    inp = synth.make_inputs(w)
    p = w.params()
    q, k, v = dev_bf16(inp["q"]), dev_bf16(inp["k_cache"]), dev_bf16(inp["v_cache"])
    dk, dvv = dev_bf16(inp["draft_k"]), dev_bf16(inp["draft_v"])
    mask = torch.from_numpy(np.ascontiguousarray(inp["tree_mask"]).view(np.int64)).cuda()
    kv_len = torch.from_numpy(inp["kv_len"]).cuda()
    M = (w.L - w.kernel_size) // w.kernel_stride + 1
    kern = torch.zeros((w.B, w.Hkv, M, w.d), dtype=torch.bfloat16, device="cuda")
    infllmv2.kernel_pool(k, kern, 0, w.L, p)
    S_cap = infllmv2.selection_capacity(p, w.L_max)
    idx = torch.empty((w.B, w.Hkv, w.Tq, S_cap), dtype=torch.int32, device="cuda")
    cnt = torch.empty((w.B, w.Hkv, w.Tq), dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    ws = torch.empty(infllmv2.workspace_size(infllmv2.ENTRY_DECODE, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, p),
                     dtype=torch.uint8, device="cuda")
    flush = Flusher()
    stream = torch.cuda.current_stream()

    def call():
        infllmv2.decode(q, k, v, kern, kv_len, o, ws, p, draft_k=dk, draft_v=dvv, tree_mask=mask,
                        idx_out=idx, counts_out=cnt)

    for _ in range(3):
        flush()
        call()
    torch.cuda.synchronize()
    K = args.prefill_steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    infllmv2.profile_enable(True)
    stages: dict[str, list[float]] = {}
    for _ in range(max(3, K // 2)):
        flush()
        call()
        for nm, t in infllmv2.profile_read():
            stages.setdefault(nm, []).append(t)
    infllmv2.profile_enable(False)
    assert infllmv2.sync_status() == 0
    counts, sel = cnt.cpu().numpy(), idx.cpu().numpy()
    kv_tok = 0
    for b in range(w.B):
        for g in range(w.Hkv):
            union = set()
            for t in range(w.Tq):
                union.update(sel[b, g, t, :counts[b, g, t]].tolist())
            L = int(inp["kv_len"][b])
            kv_tok += sum(min(w.block_size, L - x * w.block_size) for x in union)
    alg = (w.B * w.Hkv * M * w.d * 2 + kv_tok * w.d * 4 + 2 * w.B * w.Hkv * w.Tq * w.d * 2
           + 2 * w.B * w.Tq * w.Hq * w.d * 2)
    gbs = alg / (ms * 1e-3) / 1e9
    pk = peaks()
    return {"workload": name if not scale else f"{name} scaled {scale}", "batch": w.B, "drafts": w.Tq,
            "ms_per_call": ms, "calls": K, "drafts_per_s": w.B * w.Tq / (ms * 1e-3),
            "stages_ms": {kk: round(statistics.median(vv), 4) for kk, vv in stages.items()},
            "algorithmic_bytes": alg, "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4)}


# ------------------------------------------------------------------ oracle (CPU) baseline

def oracle_rows(inp, w, kern, rows):
    """The oracle's decode step restricted to the listed (b, g) rows and heads."""
    import numpy as np

    import oracle
    p = w.params()
    for (b, g, heads) in rows:
        G = w.Hq // w.Hkv
        hsel = list(range(g * G, g * G + heads))
        q = np.ascontiguousarray(inp["q"][b:b + 1][:, :, hsel])
        kern_bg = np.ascontiguousarray(kern[b:b + 1, g:g + 1])
        kv = inp["kv_len"][b:b + 1]
        S = oracle.block_scores(q, kern_bg, kv, 1, p)
        idx, cnt, _, _ = oracle.select(S, kv, 1, p)
        oracle.attention(q, np.ascontiguousarray(inp["k_cache"][b:b + 1, g:g + 1]),
                         np.ascontiguousarray(inp["v_cache"][b:b + 1, g:g + 1]), kv, idx, cnt, p)


def oracle_setup():
    import oracle
    from block_sparse_long_infllm_gb300 import synth
    w = synth.WORKLOADS[HEADLINE]
    inp = synth.make_inputs(w)
    M = oracle.n_kernels(w.L, w.kernel_size, w.kernel_stride)
    kern, _ = oracle.kernel_pool(inp["k_cache"], inp["kv_len"], w.kernel_size, w.kernel_stride, M)
    return w, inp, kern


def cpu_baseline(seconds: float = 12.0, prepared=None) -> dict:
    """The oracle (as it stands) on whole decode rows of the headline workload,
    for about `seconds` of host time."""
    import oracle
    w, inp, kern = prepared or oracle_setup()
    G = w.Hq // w.Hkv
    n = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or n == 0:
        b, g = divmod(n % (w.B * w.Hkv), w.Hkv)
        oracle_rows(inp, w, kern, [(b, g, G)])
        n += 1
    el = time.perf_counter() - t0
    queries = n * G / w.Hq
    return {"value": queries / el, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} decode rows (sequence, KV head: 16 heads = 1/2 query token each) of {HEADLINE}, "
                      f"{el:.1f} s; kernel cache precomputed as in the workload"}


def secondary_cpu_baselines(out: dict, seconds: float = 3.0) -> None:
    """The oracle, as it stands, beside each secondary leg, on bounded samples (about `seconds` of
    host time each): chunked-prefill queries (scores, selection, attention), their gradients (one
    query at a time, with the selection of the query's own row), and one tree row's drafts."""
    import numpy as np

    import oracle
    from block_sparse_long_infllm_gb300 import synth
    cores = oracle.num_threads()
    if "prefill" in out:
        w = synth.WORKLOADS[PREFILL]
        inp = synth.make_inputs(w)
        p = w.params()
        M = oracle.n_kernels(w.L, w.kernel_size, w.kernel_stride)
        kern, _ = oracle.kernel_pool(inp["k_cache"], inp["kv_len"], w.kernel_size, w.kernel_stride, M)
        rng = np.random.default_rng(3)
        n, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < seconds or n == 0:
            t_list = np.sort(rng.choice(w.Tq, 8, replace=False)).astype(np.int32)
            oracle.run(inp, w, t_list=t_list, kern=kern)
            n += 8
        el = time.perf_counter() - t0
        out["prefill"]["cpu_baseline"] = {"value": n / el, "unit": UNIT, "cores": cores, "kind": "oracle",
                                          "sample": f"{n} random queries of {PREFILL} (all 32 heads), {el:.1f} s; "
                                                    "kernel cache precomputed"}
        if "backward" in out["prefill"]:
            dout = synth.f32_to_bf16_bits(rng.standard_normal((1, 1, w.Hq, w.d)).astype(np.float32))
            q64 = synth.bf16_bits_to_f32(inp["q"]).astype(np.float64)
            k64 = synth.bf16_bits_to_f32(inp["k_cache"]).astype(np.float64)
            v64 = synth.bf16_bits_to_f32(inp["v_cache"]).astype(np.float64)
            do64 = synth.bf16_bits_to_f32(dout).astype(np.float64)
            n, t0 = 0, time.perf_counter()
            while time.perf_counter() - t0 < seconds or n == 0:
                t = int(rng.integers(w.Tq))
                pos = w.L - w.Tq + t
                S = oracle.block_scores(inp["q"][:, t:t + 1], kern, np.array([pos + 1], dtype=np.int32), w.Hkv, p)
                idx, cnt, _, _ = oracle.select(S, np.array([pos + 1], dtype=np.int32), 1, p)
                oracle.attention_bwd(q64[:, t:t + 1], k64, v64, np.array([pos + 1], dtype=np.int32), idx, cnt, p, do64)
                n += 1
            el = time.perf_counter() - t0
            out["prefill"]["backward"]["cpu_baseline"] = {
                "value": n / el, "unit": "query gradients/s", "cores": cores, "kind": "oracle",
                "sample": f"{n} random queries of {PREFILL}: selection, then dq and the query's dk, dv "
                          f"contributions (fp64, all 32 heads), {el:.1f} s"}
    if out.get("tree_verify"):
        w = synth.WORKLOADS["tree_verify_64k"]
        inp = synth.make_inputs(w)
        M = oracle.n_kernels(w.L, w.kernel_size, w.kernel_stride)
        kern, _ = oracle.kernel_pool(inp["k_cache"], inp["kv_len"], w.kernel_size, w.kernel_stride, M)
        n, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < seconds or n == 0:
            oracle.run(inp, w, kern=kern)
            n += w.Tq
        el = time.perf_counter() - t0
        out["tree_verify"][0]["cpu_baseline"] = {
            "value": n / el, "unit": "drafts/s", "cores": cores, "kind": "oracle",
            "sample": f"{n // w.Tq} whole verifications of tree_verify_64k ({w.Tq} drafts), {el:.1f} s; "
                      "kernel cache precomputed"}


def run_reference(args, world, rank):
    """The fp64 oracle as the reference arm: each step is one decode row of the
    headline workload with as many of its 16 heads as keep the run within a few minutes."""
    if rank != 0:
        return None
    import oracle
    prepared = oracle_setup()
    w, inp, kern = prepared
    G = w.Hq // w.Hkv
    t0 = time.perf_counter()
    oracle_rows(inp, w, kern, [(0, 0, G)])
    t_row = time.perf_counter() - t0
    heads = G
    budget = 150.0
    while heads > 1 and (args.steps + args.warmup) * t_row * heads / G > budget:
        heads //= 2
    for i in range(args.warmup):
        b, g = divmod(i % (w.B * w.Hkv), w.Hkv)
        oracle_rows(inp, w, kern, [(b, g, heads)])
    t0 = time.perf_counter()
    for i in range(args.steps):
        b, g = divmod(i % (w.B * w.Hkv), w.Hkv)
        oracle_rows(inp, w, kern, [(b, g, heads)])
    el = time.perf_counter() - t0
    value = args.steps * heads / w.Hq / el
    cfg = {"workload": HEADLINE, "batch": w.B, "kv_len": w.L, "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.d,
           "block_size": w.block_size, "topk": w.topk}
    sample = f"each step: one decode row (sequence, KV head) of {HEADLINE} with {heads} of its {G} query heads"
    return dict(impl="reference", metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=1e3 * el / args.steps, higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="f64", data="synthetic (seeded N(0,1) bf16, planted blocks)", config=cfg,
                cpu_baseline={"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                              "sample": sample},
                e2e={"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0})


# ------------------------------------------------------------------ main

def main():
    args = parse_args()
    world, rank, local = dist_info()
    if args.impl == "reference":
        out = run_reference(args, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    import torch

    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.no_decode:
        out = {"metric": METRIC, "profiling_only": True}
    else:
        out, dec = run_decode(args, world, rank)
        out["decode_step_with_append"] = run_decode_append(args, dec)
        out["decode_32k"] = run_decode_32k(args)
    if not args.no_prefill:
        out["prefill"] = run_prefill(args)
        out["varlen_prefill"] = run_varlen_prefill(args)
        out["tree_verify"] = [run_tree(args, "tree_verify_64k"),
                              run_tree(args, "tree_verify_64k", B=4, Tq=64, seed=1104)]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline()
        secondary_cpu_baselines(out)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
