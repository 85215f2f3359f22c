#!/usr/bin/env python3
"""Benchmark of the Ulysses sequence<->head relayout on GB300.

One step = the whole hot path on the video-DiT workload (P=4 logical shards,
B=1, S=32760 = 21x30x52 tokens, H=40, D=128, bf16): one grouped scatter of Q, K
and V into the cached final-layout targets, with RMSNorm + interleaved RoPE at
global positions fused on Q/K and V read as a strided view of a fused
projection, then the head->sequence gather of a synthetic attention output.

Metric: relayout GB/s = algorithmic payload bytes (every element read once and
written once: 3 x 2 x 335.5 MB for the scatter, 2 x 335.5 MB for the gather)
per second, plus tokens/s.  Timing: CUDA events on the launching stream around
K steps after W warm-up steps, synchronised on both sides, max over ranks.
Inputs rotate over two sets of ~2 GB each, so every step reads from HBM (the
inputs are larger than the 129 MB L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (the reference arm) on a bounded
token-sample of the same workload.  N>1 (torchrun) runs independent replicas,
one per GPU ("replicas only": all P shards of the relayout live in one GPU's
memory, so the path has no cross-GPU exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "relayout GB/s (read+write) and % of GB300 HBM peak; fused Q/K/V tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = dict(name="video_dit_p4_s32760", P=4, B=1, S=32760, H=40, D=128, eps=1e-6, theta=10000.0)
PROFILE = os.path.join(ROOT, "profiles", "fused_scatter_video_dit_p4_s32760.txt")
# the fused scatter's kernel: its template and instantiation, the shared device helpers and the parameter block
KERNEL_SOURCES = [os.path.join(ROOT, "ulysses_sequence_attention_tf_gb300", "csrc", f)
                  for f in ("block_kernel.cuh", "block_kernels.cu", "device_common.cuh", "relayout.h")]
E2E_REPEATS = 9  # interleaved repeats of the e2e steps and of the copies alone
FUSED_KERNEL = "block_kernel<bf16, D=128 (8 lanes/row), V copied + Q/K fused, interleaved> (one launch per step)"


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=12)
    ap.add_argument("--sets", type=int, default=2, help="rotating input sets (each ~2 GB)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-projection", action="store_true", help="skip the fused QKV projection measurement")
    ap.add_argument("--no-noalloc", action="store_true", help="skip the allocation-free scatter measurement")
    ap.add_argument("--no-qk-only", action="store_true", help="skip the Q/K-only fused scatter measurement")
    ap.add_argument("--cpu-tokens", type=int, default=4096, help="tokens per shard in the CPU-baseline sample")
    return ap.parse_args()


def step_bytes(w, S=None):
    """Algorithmic bytes of one step: (scatter payload, scatter extra, gather payload)."""
    S = w["S"] if S is None else S
    tensor = w["B"] * S * w["H"] * w["D"] * 2  # one of Q/K/V over all shards, bf16
    scatter_payload = 3 * 2 * tensor  # Q, K, V each read once and written once
    scatter_extra = S * w["D"] * 4 + 2 * w["D"] * 2  # fp32 (cos, sin) rows + two RMSNorm weights
    gather_payload = 2 * tensor
    return scatter_payload, scatter_extra, gather_payload


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, torch copy)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


def kernel_source_hash():
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the fused scatter from the committed ncu summary,
    or None if the summary is missing or the kernel changed since it was taken."""
    try:
        fields = {}
        with open(PROFILE) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("kernel_source_sha256_16", "").split()[:1] != [kernel_source_hash()]:
            return None
        return int(float(fields["dram_bytes_per_full_launch"].split()[0]))
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons, n = [], [], set(), 0
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            n += 1
            for name, val in zip(self.NAMES, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


def gpu_id_for_smi(torch, dev):
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if uuid:
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:  # noqa: BLE001
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    return vis.split(",")[dev] if vis else str(dev)


# ------------------------------------------------------------------ CPU oracle leg
def oracle_step(w, Sl, seed=0):
    """One step of the workload on the CPU oracle with S_local = Sl tokens per
    shard; returns seconds."""
    import torch

    import oracle
    from ulysses_sequence_attention_tf_gb300 import synth
    P, B, H, D = w["P"], w["B"], w["H"], w["D"]
    d = synth.qkv_shards(P, B, Sl, H, D, torch.bfloat16, seed=seed, layout="v_strided")
    wq, wk = synth.norm_weights(D, torch.bfloat16, seed=0)
    attn = synth.attn_outputs(P, B, P * Sl, H // P, D, torch.bfloat16, seed=seed)
    oracle.load()
    t0 = time.perf_counter()
    table = oracle.rope_table(w["theta"], P * Sl, D)
    oracle.scatter(d["v"], P)
    oracle.scatter_norm_rope(d["q"], P, wq, w["eps"], table)
    oracle.scatter_norm_rope(d["k"], P, wk, w["eps"], table)
    oracle.gather(attn, P)
    return time.perf_counter() - t0


def cpu_cores_used():
    return 1  # the oracle is single-threaded C


def run_reference(args):
    """Reference arm: the CPU oracle, as it stands, on a bounded token-sample per step."""
    w = WORKLOAD
    # calibrate: seconds per token per shard, then size each step's sample so the
    # whole --warmup + --steps run stays within about two and a half minutes
    cal = oracle_step(w, 4) / 4
    budget = 150.0 / max(1, args.steps + args.warmup)
    Sl = max(1, min(w["S"] // w["P"], int(budget / cal)))
    for i in range(args.warmup):
        oracle_step(w, Sl, seed=i)
    times = [oracle_step(w, Sl, seed=100 + i) for i in range(args.steps)]
    t = sum(times) / len(times)
    sp, _, gp = step_bytes(w, S=w["P"] * Sl)
    value = (sp + gp) / t / 1e9
    sample = (f"S_local={Sl} tokens per shard (of {w['S'] // w['P']}), every other size as the workload; "
              f"one oracle step = fused Q/K scatter, V scatter, cos/sin table, output gather")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w["name"], "P": w["P"], "B": w["B"], "S": w["S"], "H": w["H"], "D": w["D"],
                   "parallelism": "replicas", "l2": "CPU oracle; no GPU"},
        "tokens_per_s": w["P"] * Sl * w["B"] / t,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores_used(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
def measure_projection(torch, binding, synth, w, stream, dev, wq, wk, iters=10):
    """The fused QKV projection (tcgen05 GEMM with the RMSNorm/RoPE/scatter
    epilogue) on the workload's shape: hidden = H*D, weight [3*H*D, hidden]."""
    P, B, S, H, D = w["P"], w["B"], w["S"], w["H"], w["D"]
    Sl, Hl, hidden = S // P, H // P, H * D
    xs, wqkv = synth.projection_inputs(P, B, Sl, hidden, H, D, torch.bfloat16, seed=11, device=dev)
    outs = {k: [torch.empty((B, S, Hl, D), dtype=torch.bfloat16, device=dev) for _ in range(P)] for k in "qkv"}

    def call():
        binding.project_qkv_into(xs, wqkv, H, outs["q"], outs["k"], outs["v"], norm_rope=True, q_weight=wq,
                                 k_weight=wk, eps=w["eps"], theta=w["theta"], stream=stream)

    for _ in range(3):
        call()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / iters
    flops = 2.0 * B * S * 3 * H * D * hidden
    tflops = flops / (ms / 1e3) / 1e12
    peak, peak_sus, src = measured_tensor_peak()
    return {"kernel": "qkv_gemm_pair_kernel<fused, interleaved> (tcgen05 cta_group::2, persistent CTA pairs, "
                      "256x256 tiles)",
            "shape": f"M={B * S} (P={P} shards), N={3 * H * D}, K={hidden}, bf16", "ms": ms,
            "TFLOP/s": tflops, "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak,
                                             "unit": "TFLOP/s", "frac": tflops / peak,
                                             "frac_of_sustained": tflops / peak_sus, "peak_source": src},
            "iters": iters}


def measure_noalloc(torch, binding, w, sets, wq, wk, stream, dev, rounds=5, calls=10):
    """The allocation-free scatter (its cos/sin table in the library's fixed
    scratch) against scatter_qkv_into on the same caller-owned targets: rounds of
    `calls` calls each, the two interleaved, CUDA events on the stream; inputs
    rotate over the input sets (larger than L2)."""
    P, B, S, H, D = w["P"], w["B"], w["S"], w["H"], w["D"]
    outs = [[torch.empty((B, S, H // P, D), dtype=torch.bfloat16, device=dev) for _ in range(P)] for _ in "qkv"]
    kw = dict(norm_rope=True, q_weight=wq, k_weight=wk, eps=w["eps"], theta=w["theta"], stream=stream)
    fns = {"noalloc": binding.scatter_qkv_noalloc, "into": binding.scatter_qkv_into}

    def run(name, n):
        for j in range(n):
            g = sets[j % len(sets)]
            fns[name](g["q"], g["k"], g["v"], *outs, **kw)

    for name in fns:
        run(name, 3)
    torch.cuda.synchronize(dev)
    ms = {name: [] for name in fns}
    for _ in range(rounds):
        for name in fns:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run(name, calls)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms[name].append(e0.elapsed_time(e1) / calls)
    med = {name: statistics.median(v) for name, v in ms.items()}
    sp, sx, _ = step_bytes(w)
    return {"ms_per_call": med["noalloc"], "GB/s": (sp + sx) / (med["noalloc"] / 1e3) / 1e9,
            "into_ms_per_call": med["into"], "ratio_to_into": med["noalloc"] / med["into"],
            "repeats_ms": ms,
            "note": "tf_ulysses_scatter_qkv_noalloc, fused Q/K/V scatter into caller-owned targets, table in the "
                    "fixed scratch (built by the first call, reused after); medians of interleaved rounds"}


def measure_qk_only(torch, binding, w, sets, wq, wk, stream, dev, peak, rounds=5, calls=10):
    """The fused scatter of Q and K alone (V moved by another path) at the same
    shape, interleaved and half-split RoPE: rounds of `calls` calls into
    caller-owned targets, CUDA events on the stream, inputs rotating over the
    input sets (each launch reads 671 MB, more than L2)."""
    P, B, S, H, D = w["P"], w["B"], w["S"], w["H"], w["D"]
    outs = [[torch.empty((B, S, H // P, D), dtype=torch.bfloat16, device=dev) for _ in range(P)] for _ in "qk"]
    sp, sx, _ = step_bytes(w)
    nbytes = sp * 2 // 3 + sx  # Q and K read and written, the table and the weights
    res = {}
    for name, rope in (("interleaved", "interleaved"), ("half_split", "neox")):
        kw = dict(norm_rope=True, q_weight=wq, k_weight=wk, eps=w["eps"], theta=w["theta"], rope=rope, stream=stream)

        def run(n):
            for j in range(n):
                g = sets[j % len(sets)]
                binding.scatter_qkv_into(g["q"], g["k"], None, outs[0], outs[1], None, **kw)

        run(3)
        torch.cuda.synchronize(dev)
        ms = []
        for _ in range(rounds):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run(calls)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms.append(e0.elapsed_time(e1) / calls)
        med = statistics.median(ms)
        gbs = nbytes / (med / 1e3) / 1e9
        res[name] = {"ms_per_call": med, "GB/s": gbs, "frac": gbs / peak, "repeats_ms": ms}
    res["bytes"] = nbytes
    res["note"] = ("tf_ulysses_scatter_qkv_into with Q and K only, RMSNorm + RoPE, into caller-owned targets; "
                   "back-to-back calls, medians of rounds")
    return res


def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured (MEASURED_PEAKS.json, cuBLAS bf16)"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, "fallback (1.9 PF burst / 1.7 PF sustained, earlier GB300 measurement)"


def max_over_ranks(torch, dist, ms, dev):
    """The slowest rank's time: replicas finish when the last one does."""
    t = torch.tensor([float(ms)], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(world, payload_bytes_per_step, steps, max_ms):
    """Whole-job GB/s of N replicas: every rank moves the per-step payload each
    step, and the job takes the slowest rank's time."""
    return world * payload_bytes_per_step * steps / (max_ms / 1e3) / 1e9


def run_e2e(args, torch, binding, src, wq, wk, w, stream, dev, world, step_payload):
    """The same step through the public API with the inputs in pinned host memory
    and the results read back, every step: host->device copies of Q/K/V and the
    attention output, the fused scatter and the gather, device->host copies of
    every target and output.  Two buffer sets (two cache tags) let step k's
    upload, step k-1's calls and step k-2's download run on three streams at once;
    events order each buffer's reuse."""
    import torch.distributed as dist
    nbuf = 2
    H, D = w["H"], w["D"]
    # Q/K contiguous; V uploaded as the fused projection buffer [B, Sl, 3*H*D] it is a
    # view of, and passed as that strided view: the same call as the device-timed steps
    h_in = {key: [x.contiguous().cpu().pin_memory() for x in src[key]] for key in ("q", "k", "attn")}
    h_in["vbuf"] = [b.cpu().pin_memory() for b in src["backing"]]
    d_in = [{key: [torch.empty_like(x, device=dev) for x in h_in[key]] for key in h_in} for _ in range(nbuf)]
    d_v = [[b[..., 2 * H * D:].unflatten(-1, (H, D)) for b in d_in[i]["vbuf"]] for i in range(nbuf)]
    assert d_v[0][0].stride() == src["v"][0].stride()
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_cmp = stream
    results = []

    def calls(i):
        tq, tk, tv, _ = binding.scatter_qkv(f"bench_e2e{i}", d_in[i]["q"], d_in[i]["k"], d_v[i],
                                            norm_rope=True, q_weight=wq, k_weight=wk, eps=w["eps"],
                                            theta=w["theta"], stream=s_cmp)
        o, _ = binding.gather_out(f"bench_e2e{i}", d_in[i]["attn"], stream=s_cmp)
        return tq + tk + tv + o

    for i in range(nbuf):
        results.append(calls(i))
    h_out = [[torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in results[0]] for _ in range(nbuf)]
    h2d = sum(x.numel() * x.element_size() for key in h_in for x in h_in[key])
    d2h = sum(x.numel() * x.element_size() for x in h_out[0])
    loaded = [torch.cuda.Event() for _ in range(nbuf)]
    computed = [torch.cuda.Event() for _ in range(nbuf)]
    drained = [torch.cuda.Event() for _ in range(nbuf)]
    for i in range(nbuf):
        computed[i].record(s_cmp)
        drained[i].record(s_d2h)

    def e2e_step(k):
        i = k % nbuf
        s_h2d.wait_event(computed[i])  # the calls of step k - nbuf have read d_in[i]
        with torch.cuda.stream(s_h2d):
            for key in h_in:
                for dx, hx in zip(d_in[i][key], h_in[key]):
                    dx.copy_(hx, non_blocking=True)
        loaded[i].record(s_h2d)
        s_cmp.wait_event(loaded[i])
        s_cmp.wait_event(drained[i])  # step k - nbuf's results are on the host
        res = calls(i)
        computed[i].record(s_cmp)
        s_d2h.wait_event(computed[i])
        with torch.cuda.stream(s_d2h):
            for hx, dx in zip(h_out[i], res):
                hx.copy_(dx, non_blocking=True)
        drained[i].record(s_d2h)

    for k in range(nbuf):  # warm the pipeline
        e2e_step(k)
    torch.cuda.synchronize(dev)

    def time_e2e():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_h2d)  # the first operation of the timed steps
        for k in range(args.e2e_steps):
            e2e_step(k)
        e1.record(s_d2h)  # after the last download, which follows every other operation
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    def time_copies():
        """The host link's ceiling for the same traffic: each step's uploads and
        downloads alone (same pinned buffers, both directions at once, no kernels)."""
        torch.cuda.synchronize(dev)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(s_h2d)
        s_d2h.wait_event(c0)
        for k in range(args.e2e_steps):
            i = k % nbuf
            with torch.cuda.stream(s_h2d):
                for key in h_in:
                    for dx, hx in zip(d_in[i][key], h_in[key]):
                        dx.copy_(hx, non_blocking=True)
            with torch.cuda.stream(s_d2h):
                for hx, dx in zip(h_out[i], results[i]):
                    hx.copy_(dx, non_blocking=True)
        s_h2d.wait_stream(s_d2h)
        c1.record(s_h2d)
        torch.cuda.synchronize(dev)
        return c0.elapsed_time(c1)

    # nine interleaved repeats of each (the host link is shared with the rest of
    # the machine, and a window can catch other traffic: three of five repeats at
    # half speed once): the e2e median, and the copies' best as the link's
    # ceiling -- their median has come out both above and below the e2e time on
    # different boxes (2.0x once), so it bounds nothing
    e2e_runs, copy_runs = [], []
    for _ in range(E2E_REPEATS):
        e2e_runs.append(time_e2e())
        copy_runs.append(time_copies())
    e2e_ms, copy_ms = statistics.median(e2e_runs), min(copy_runs)
    if world > 1:
        e2e_ms = max_over_ranks(torch, dist, e2e_ms, dev)
        copy_ms = max_over_ranks(torch, dist, copy_ms, dev)
    return {"value": aggregate_gbs(world, step_payload, args.e2e_steps, e2e_ms), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.e2e_steps,
            "steps": args.e2e_steps, "repeats_gbs": [aggregate_gbs(world, step_payload, args.e2e_steps, m)
                                                    for m in e2e_runs],
            "host_link": {"copies_only_ms_per_step": copy_ms / args.e2e_steps,
                          "copies_only_repeats_ms_per_step": [m / args.e2e_steps for m in copy_runs],
                          "gbs_per_direction": max(h2d, d2h) / (copy_ms / args.e2e_steps / 1e3) / 1e9,
                          "e2e_frac_of_copies_only": copy_ms / e2e_ms},
            "note": "pinned host Q/K/attention inputs and V's fused projection buffer [B, Sl, 3*H*D] copied "
                    "in (V passed as its strided view, as in the device-timed steps), all targets and outputs "
                    "copied out, every step; upload, calls and download of consecutive steps overlap on "
                    "three streams (two buffer sets); median of nine repeats of the timed steps, interleaved "
                    "with nine repeats of host_link: the same copies without the calls (best repeat)"}


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    import torch
    import torch.distributed as dist

    from ulysses_sequence_attention_tf_gb300 import binding, build, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    build.build()
    binding.lib()
    binding.use_torch_allocator(True)

    w = WORKLOAD
    P, B, S, H, D = w["P"], w["B"], w["S"], w["H"], w["D"]
    Sl, Hl = S // P, H // P
    dtype = torch.bfloat16
    nsets = max(1, args.sets)
    sets = []
    for s in range(nsets):
        g = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=1000 * rank + s, layout="v_strided", device=dev)
        g["attn"] = synth.attn_outputs(P, B, S, Hl, D, dtype, seed=1000 * rank + s, device=dev)
        sets.append(g)
    wq, wk = synth.norm_weights(D, dtype, seed=0, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(g):
        binding.scatter_qkv("bench_qkv", g["q"], g["k"], g["v"], norm_rope=True, q_weight=wq, k_weight=wk,
                            eps=w["eps"], theta=w["theta"], stream=stream)
        binding.gather_out("bench_out", g["attn"], stream=stream)

    for i in range(args.warmup):
        step(sets[i % nsets])
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for_smi(torch, local_rank))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    # the timed steps, back to back: each launch may start while the one before it
    # drains (the library launches its kernels for programmatic dependent launch)
    n_launch0 = binding.launch_count()
    start.record(stream)
    for k in range(K):
        step(sets[k % nsets])
    end.record(stream)
    torch.cuda.synchronize(dev)
    launches = binding.launch_count() - n_launch0
    total_ms = start.elapsed_time(end)
    # each kernel's duration: K more steps with an event before, between and after
    # the two calls (events between launches keep them from overlapping)
    for k in range(K):
        g = sets[k % nsets]
        ev[k][0].record(stream)
        binding.scatter_qkv("bench_qkv", g["q"], g["k"], g["v"], norm_rope=True, q_weight=wq, k_weight=wk,
                            eps=w["eps"], theta=w["theta"], stream=stream)
        ev[k][1].record(stream)
        binding.gather_out("bench_out", g["attn"], stream=stream)
        ev[k][2].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    scat_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    gath_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)]
    if world > 1:
        total_ms = max_over_ranks(torch, dist, total_ms, dev)
        dist.barrier()

    sp, sx, gp = step_bytes(w)
    ms_per_step = total_ms / K
    value = aggregate_gbs(world, sp + gp, K, total_ms)
    scat_avg = sum(scat_ms) / K
    gath_avg = sum(gath_ms) / K
    peak, peak_src = measured_peak()
    achieved = (sp + sx) / (scat_avg / 1e3) / 1e9

    # ---------------- end to end through the public API with host buffers
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, torch, binding, sets[0], wq, wk, w, stream, dev, world, sp + gp)

    noalloc = None if args.no_noalloc else measure_noalloc(torch, binding, w, sets, wq, wk, stream, dev)
    qk_only = None if args.no_qk_only else measure_qk_only(torch, binding, w, sets, wq, wk, stream, dev, peak)

    projection = None
    if not args.no_projection:
        projection = measure_projection(torch, binding, synth, w, stream, dev, wq, wk)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        Sl_cpu = min(args.cpu_tokens, Sl)
        t_cpu = oracle_step(w, Sl_cpu, seed=7)
        sp_c, _, gp_c = step_bytes(w, S=P * Sl_cpu)
        cpu = {"value": (sp_c + gp_c) / t_cpu / 1e9, "unit": "GB/s", "cores": cpu_cores_used(), "kind": "oracle",
               "sample": f"one step at S_local={Sl_cpu} tokens per shard (of {Sl}), other sizes as the workload: "
                         f"fused Q/K scatter, V scatter, cos/sin table, output gather; {t_cpu:.2f} s",
               "host_cpu_count": os.cpu_count()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w["name"], "P": P, "B": B, "S": S, "H": H, "D": D,
                       "step": "fused Q/K/V scatter (RMSNorm+RoPE on Q/K, V strided view of a fused "
                               "projection) into cached targets + head->sequence output gather",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": f"inputs larger than L2: {nsets} rotating input set(s) of ~2 GB",
                       "timing": "value: K steps back to back between two events; kernels: K further steps "
                                 "with an event before, between and after the two calls"},
            "tokens_per_s": world * B * S * K / (total_ms / 1e3),
            "pct_of_hbm_measured": 100.0 * value / world / peak,
            "pct_of_hbm_nominal_8000": 100.0 * value / world / NOMINAL_HBM_GBS,
            "kernels": {
                "scatter_fused": {"ms": scat_avg, "GB/s": achieved, "bytes": sp + sx,
                                  "kcycles_at_median_sm_clock": scat_avg * (clocks["sm_mhz"] or 0)},
                "gather": {"ms": gath_avg, "GB/s": gp / (gath_avg / 1e3) / 1e9, "bytes": gp,
                           "kcycles_at_median_sm_clock": gath_avg * (clocks["sm_mhz"] or 0)},
            },
            "tolerance": {"relayout": "bit-exact", "fused_qk": "max-abs 1e-2 (bf16) / 2e-3 (fp16); an element "
                          "above that must differ by exactly 1 ulp (checked by the -m gpu tests)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": profiled_traffic(), "peak_source": peak_src,
                         "kernel": FUSED_KERNEL},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "noalloc_fused": noalloc,
            "qk_only_fused": qk_only,
            "qkv_projection": projection,
            "clocks": clocks,
            "gpu_launches": launches,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
