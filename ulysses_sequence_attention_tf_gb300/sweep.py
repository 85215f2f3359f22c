"""Configuration and size sweep of the relayout kernels, with comparison baselines.

    python -m ulysses_sequence_attention_tf_gb300.sweep [--iters 20] [--warmup 3] [--only C5] [--no-baselines]

Configurations (seeded synthetic inputs from ``synth``):
  C1  P=2, B=1, S=256, H=8, D=64, fp16: Q/K/V scatter and the output gather (latency-bound; no gate)
  C2  P=4, B=1, S=4096, H=24, D=128, bf16: Q/K/V views of a fused projection, RMSNorm + RoPE
  C3  P=4, B=1, S=32760, H=40, D=128, bf16: the video-DiT step (fused scatter, gather)
  C4  P in {2,4,6,8} x {fp16, bf16} x D in {64,128}, H=48, B=2, S=6001 padded to a multiple
      of P: Q/K/V scatter and the output gather (one tensor, as the attention output)
  C5  bf16, P in {2,4,8}, D=128, H=32, B=1, one tensor, 64 KiB .. 2 GiB per direction
      (S = 8, 32, .., 131072 and 262144): scatter and gather
  F   the fused scatter across shapes: P in {2,4,8} x D in {64,128} x {bf16, fp16},
      H=48, B=1, S=32760 padded to a multiple of P, V a view into a fused projection,
      RMSNorm + interleaved RoPE on Q/K
  FQK the same shapes with Q and K only (V moved by another path)

Every point prints one JSON line:
  * GB/s over algorithmic bytes (each payload element read once and written once;
    the fused points add the cos/sin rows and the RMSNorm weights);
  * the median and best over ``--iters`` CUDA-event-timed replays (after
    ``--warmup``) of a CUDA graph holding the call, so that the GPU's time is
    measured rather than the host's per-call work: without a flush, after an L2
    flush by writing 256 MiB, and after one by reading 256 MiB; and the eager
    calls' median after the write flush.  The write flush leaves L2 full of
    dirty lines, so the timed launch also pays for writing back up to the L2's
    size of the flush's data; the read flush leaves clean lines, so the launch
    starts from a cold L2 and owes nothing.  The gate uses the read flush;
  * the fraction of the measured HBM copy peak, and for messages of 64 MiB or more
    whether the read-flushed median clears 0.8 of it (and the write-flushed one);
  * the same measurement of one contiguous copy of the same bytes by the
    library's bulk-copy kernel (the ceiling at that size, launch, fill and drain
    included).
For the pure relayouts it also prints the same movement (medians after either
flush, and whether the call could be captured in a graph) done by:
  * ``torch_copy``: a strided ``copy_`` per (shard, head group) and tensor;
  * ``torch_permute``: ``stack`` of the shards, then ``permute(...).contiguous()``;
  * ``memcpy2d``: ``cudaMemcpy2DAsync`` per (shard, head group, batch) and tensor.
"""
from __future__ import annotations

import argparse
import ctypes
import ctypes.util
import json
import os
import statistics
import subprocess

import torch

from . import binding, build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GATE_BYTES = 64 << 20
GATE_FRAC = 0.8
FLUSH_BYTES = 256 << 20


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def _cudart():
    """The CUDA runtime, for the cudaMemcpy2DAsync baseline (None if not found)."""
    cands = [ctypes.util.find_library("cudart"), "/usr/local/cuda/lib64/libcudart.so", "libcudart.so.13",
             "libcudart.so.12"]
    for c in cands:
        if not c:
            continue
        try:
            lib = ctypes.CDLL(c)
            lib.cudaMemcpy2DAsync.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t,
                                              ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
            lib.cudaMemcpy2DAsync.restype = ctypes.c_int
            return lib
        except (OSError, AttributeError):
            continue
    return None


class Timer:
    def __init__(self, iters, warmup, flush_buf):
        self.iters, self.warmup, self.flush_buf = iters, warmup, flush_buf
        self.flush_sink = torch.empty((), dtype=torch.int64, device=flush_buf.device)

    def flush(self, mode):
        """Evict L2 before a timed launch.  "write": write a 256 MiB buffer (L2 is then
        full of dirty lines, whose write-back the timed launch pays for); "read": read
        it (L2 is left holding clean lines, so the launch starts cold and owes nothing)."""
        if mode == "write":
            self.flush_buf.zero_()
        elif mode == "read":
            torch.sum(self.flush_buf.view(torch.int64), dim=0, out=self.flush_sink)

    def run(self, fn, flush):
        for _ in range(self.warmup):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(self.iters)]
        for a, b in ev:
            self.flush(flush)
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        ms = sorted(a.elapsed_time(b) for a, b in ev)
        return statistics.median(ms), ms[0]

    def graph(self, fn):
        """fn captured once in a CUDA graph: replays time the GPU work alone."""
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g


def _gbs(nbytes, ms):
    return nbytes / (ms / 1e3) / 1e9


def _stats(timer, fn, nbytes, peak):
    """GPU time from CUDA-graph replays of fn (without and with an L2 flush before
    each), and the eager calls' time for reference (which includes the host's
    per-call work when that is longer than the GPU's)."""
    try:
        g = timer.graph(fn)
        replay, timing = g.replay, "graph"
    except Exception:  # a call that cannot be captured is timed eagerly, and says so
        torch.cuda.synchronize()
        g, replay, timing = None, fn, "eager"
    med, best = timer.run(replay, flush=None)
    fmed, fbest = timer.run(replay, flush="write")
    rmed, rbest = timer.run(replay, flush="read")
    emed, _ = timer.run(fn, flush="write")
    del g
    return {"gbs_median": _gbs(nbytes, med), "gbs_best": _gbs(nbytes, best),
            "gbs_median_flushed": _gbs(nbytes, fmed), "gbs_best_flushed": _gbs(nbytes, fbest),
            "frac_median_flushed": _gbs(nbytes, fmed) / peak, "ms_median": med, "ms_median_flushed": fmed,
            "gbs_median_read_flushed": _gbs(nbytes, rmed), "gbs_best_read_flushed": _gbs(nbytes, rbest),
            "frac_median_read_flushed": _gbs(nbytes, rmed) / peak,
            "eager_gbs_median_flushed": _gbs(nbytes, emed), "timing": timing}


# ---------------------------------------------------------------- baselines
def _pieces(P, B, Sl, Hl, D, esize, direction):
    """(shard r, group g, batch b) -> (src offset, src pitch, dst offset, dst pitch) in bytes for a
    contiguous [B, Sl, H, D] shard and a contiguous [B, S, Hl, D] group buffer."""
    H, S = Hl * P, Sl * P
    for r in range(P):
        for g in range(P):
            for b in range(B):
                shard = ((b * Sl) * H + g * Hl) * D * esize
                group = ((b * S + r * Sl) * Hl) * D * esize
                if direction == "scatter":
                    yield r, g, shard, H * D * esize, group, Hl * D * esize
                else:
                    yield r, g, group, Hl * D * esize, shard, H * D * esize


def baselines(timer, tensors_src, tensors_dst, P, B, Sl, Hl, D, direction, nbytes, peak, cudart):
    """The same relayout by torch and by cudaMemcpy2DAsync; sources and destinations are lists
    (one per tensor) of P contiguous buffers, shards [B, Sl, H, D] or groups [B, S, Hl, D]."""
    out = {}

    def torch_copy():
        for src, dst in zip(tensors_src, tensors_dst):
            for r in range(P):
                for g in range(P):
                    if direction == "scatter":
                        dst[g][:, r * Sl:(r + 1) * Sl].copy_(src[r][:, :, g * Hl:(g + 1) * Hl])
                    else:
                        dst[r][:, :, g * Hl:(g + 1) * Hl].copy_(src[g][:, r * Sl:(r + 1) * Sl])

    def torch_permute():
        for src in tensors_src:
            if direction == "scatter":  # [r, B, Sl, g, Hl, D] -> [g, B, r, Sl, Hl, D]
                torch.stack(src).view(P, B, Sl, P, Hl, D).permute(3, 1, 0, 2, 4, 5).contiguous()
            else:  # [g, B, r, Sl, Hl, D] -> [r, B, Sl, g, Hl, D]
                torch.stack(src).view(P, B, P, Sl, Hl, D).permute(2, 1, 3, 0, 4, 5).contiguous()

    def keep(st):
        return {"read_flushed": st["gbs_median_read_flushed"], "write_flushed": st["gbs_median_flushed"],
                "timing": st["timing"]}

    out["torch_copy"] = keep(_stats(timer, torch_copy, nbytes, peak))
    out["torch_permute"] = keep(_stats(timer, torch_permute, nbytes, peak))
    if cudart is not None:
        esize = tensors_src[0][0].element_size()
        plan = list(_pieces(P, B, Sl, Hl, D, esize, direction))
        width = Hl * D * esize

        def memcpy2d():
            stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            for src, dst in zip(tensors_src, tensors_dst):
                for r, g, so, sp, do, dp in plan:
                    s_buf, d_buf = (src[r], dst[g]) if direction == "scatter" else (src[g], dst[r])
                    rc = cudart.cudaMemcpy2DAsync(ctypes.c_void_p(d_buf.data_ptr() + do), dp,
                                                  ctypes.c_void_p(s_buf.data_ptr() + so), sp, width, Sl, 3, stream)
                    if rc != 0:
                        raise RuntimeError(f"cudaMemcpy2DAsync returned {rc}")

        out["memcpy2d"] = keep(_stats(timer, memcpy2d, nbytes, peak))
    else:
        out["memcpy2d"] = None
    return out


def same_size_copy(timer, nbytes, peak):
    """One contiguous copy of the same bytes (nbytes / 2 each way) by the library's
    bulk-copy kernel (the exchange with P = 1): the same engine with nothing to
    relayout, so launch, fill and drain at this size are included."""
    half = (nbytes // 2) // 16 * 16
    a = torch.empty((1, half), dtype=torch.uint8, device="cuda")
    b = torch.empty_like(a)
    st = _stats(timer, lambda: binding.exchange_chunks([a], [b]), 2 * half, peak)
    del a, b
    return st["gbs_median_flushed"], st["gbs_median_read_flushed"]


# ---------------------------------------------------------------- points
def emit(rec):
    print(json.dumps(rec), flush=True)


def point_relayout(name, timer, peak, cudart, P, B, S, H, D, dtype, ntensors, direction, with_baselines,
                   seed=0):
    Sl, Hl = S // P, H // P
    dev = torch.device("cuda")
    esize = torch.empty((), dtype=dtype).element_size()
    nbytes = 2 * ntensors * B * S * H * D * esize
    if direction == "scatter":
        g = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=seed, device=dev, with_k=ntensors > 1,
                             with_v=ntensors > 2)
        srcs = [g[k] for k in ("q", "k", "v")[:ntensors]]
        args = srcs + [None] * (3 - ntensors)

        def ours():
            binding.scatter_qkv(f"sweep_{name}", *args)
    else:
        srcs = [synth.attn_outputs(P, B, S, Hl, D, dtype, seed=seed + t, device=dev) for t in range(ntensors)]
        tags = [f"sweep_{name}_{t}" for t in range(ntensors)]

        def ours():
            for tag, a in zip(tags, srcs):
                binding.gather_out(tag, a)
    rec = {"sweep": name, "direction": direction, "P": P, "B": B, "S": S, "H": H, "D": D,
           "dtype": str(dtype).replace("torch.", ""), "tensors": ntensors, "bytes": nbytes,
           "bytes_per_direction": nbytes // 2}
    rec.update(_stats(timer, ours, nbytes, peak))
    rec["contiguous_copy_gbs_median_flushed"], rec["contiguous_copy_gbs_median_read_flushed"] = \
        same_size_copy(timer, nbytes, peak)
    gated = nbytes // 2 >= GATE_BYTES
    rec["gate"] = f">= {GATE_FRAC} of peak (read-flushed median)" if gated else None
    rec["pass"] = (rec["frac_median_read_flushed"] >= GATE_FRAC) if gated else None
    rec["pass_write_flushed"] = (rec["frac_median_flushed"] >= GATE_FRAC) if gated else None
    if with_baselines:
        if direction == "scatter":
            dsts = [[torch.empty((B, S, Hl, D), dtype=dtype, device=dev) for _ in range(P)] for _ in srcs]
        else:
            dsts = [[torch.empty((B, Sl, H, D), dtype=dtype, device=dev) for _ in range(P)] for _ in srcs]
        rec["baselines_gbs_median"] = baselines(timer, srcs, dsts, P, B, Sl, Hl, D, direction, nbytes, peak,
                                                        cudart)
        del dsts
    emit(rec)
    del srcs
    binding.cache_clear()
    torch.cuda.empty_cache()
    return rec


def point_fused(name, timer, peak, P, B, S, H, D, dtype, layout, seed=0, with_v=True):
    Sl, Hl = S // P, H // P
    dev = torch.device("cuda")
    g = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=seed, device=dev, layout=layout, with_v=with_v)
    wq, wk = synth.norm_weights(D, dtype, seed=seed, device=dev)
    esize = torch.empty((), dtype=dtype).element_size()
    tensors = 3 if with_v else 2
    nbytes = 2 * tensors * B * S * H * D * esize + S * D * 4 + 2 * D * esize

    def ours():
        binding.scatter_qkv(f"sweep_{name}", g["q"], g["k"], g["v"], norm_rope=True, q_weight=wq, k_weight=wk)
    rec = {"sweep": name, "direction": "scatter_norm_rope", "P": P, "B": B, "S": S, "H": H, "D": D,
           "dtype": str(dtype).replace("torch.", ""), "tensors": tensors, "layout": layout, "bytes": nbytes,
           "bytes_per_direction": nbytes // 2}
    rec.update(_stats(timer, ours, nbytes, peak))
    rec["contiguous_copy_gbs_median_flushed"], rec["contiguous_copy_gbs_median_read_flushed"] = \
        same_size_copy(timer, nbytes, peak)
    gated = nbytes // 2 >= GATE_BYTES
    rec["gate"] = f">= {GATE_FRAC} of peak (read-flushed median)" if gated else None
    rec["pass"] = (rec["frac_median_read_flushed"] >= GATE_FRAC) if gated else None
    rec["pass_write_flushed"] = (rec["frac_median_flushed"] >= GATE_FRAC) if gated else None
    emit(rec)
    del g
    binding.cache_clear()
    torch.cuda.empty_cache()
    return rec


def sm_clock():
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm", "--format=csv,noheader,nounits",
                              f"--id={torch.cuda.current_device()}"], capture_output=True, text=True, timeout=10)
        return out.stdout.strip()
    except (OSError, subprocess.SubprocessError):
        return None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--only", default=None, help="comma-separated subset of C1..C5, F, FQK")
    ap.add_argument("--no-baselines", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3 or args.iters < 20:
        raise SystemExit("--warmup >= 3 and --iters >= 20")
    if not torch.cuda.is_available():
        raise SystemExit("the sweep needs a CUDA device")
    build.build()
    binding.lib()
    binding.use_torch_allocator(True)
    peak, peak_src = measured_peak()
    timer = Timer(args.iters, args.warmup, torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda"))
    cudart = None if args.no_baselines else _cudart()
    only = set(args.only.split(",")) if args.only else {"C1", "C2", "C3", "C4", "C5", "F", "FQK"}
    base = not args.no_baselines
    recs = []
    bf16, fp16 = torch.bfloat16, torch.float16
    if "C1" in only:
        for d in ("scatter", "gather"):
            recs.append(point_relayout("C1", timer, peak, cudart, 2, 1, 256, 8, 64, fp16, 3 if d == "scatter" else 1,
                                       d, base))
    if "C2" in only:
        recs.append(point_fused("C2", timer, peak, 4, 1, 4096, 24, 128, bf16, "fused"))
        recs.append(point_relayout("C2", timer, peak, cudart, 4, 1, 4096, 24, 128, bf16, 3, "scatter", base))
    if "C3" in only:
        recs.append(point_fused("C3", timer, peak, 4, 1, 32760, 40, 128, bf16, "v_strided"))
        recs.append(point_relayout("C3", timer, peak, cudart, 4, 1, 32760, 40, 128, bf16, 1, "gather", base))
    if "C4" in only:
        for P in (2, 4, 6, 8):
            for dt in (fp16, bf16):
                for D in (64, 128):
                    for d in ("scatter", "gather"):
                        recs.append(point_relayout("C4", timer, peak, cudart, P, 2, synth.padded_seq(6001, P), 48, D,
                                                   dt, 3 if d == "scatter" else 1, d, base))
    if "C5" in only:
        for P in (2, 4, 8):
            for S in (8, 32, 128, 512, 2048, 8192, 32768, 131072, 262144):
                for d in ("scatter", "gather"):
                    recs.append(point_relayout("C5", timer, peak, cudart, P, 1, S, 32, 128, bf16, 1, d,
                                               base and S >= 2048))
    if "F" in only:
        for P in (2, 4, 8):
            for D in (64, 128):
                for dt in (bf16, fp16):
                    recs.append(point_fused("F", timer, peak, P, 1, synth.padded_seq(32760, P), 48, D, dt, "v_strided"))
    if "FQK" in only:
        for P in (2, 4, 8):
            for D in (64, 128):
                for dt in (bf16, fp16):
                    recs.append(point_fused("FQK", timer, peak, P, 1, synth.padded_seq(32760, P), 48, D, dt,
                                            "v_strided", with_v=False))
    gated = [r for r in recs if r["pass"] is not None]
    emit({"summary": {"points": len(recs), "gated_points": len(gated), "gated_pass": sum(r["pass"] for r in gated),
                      "gated_pass_write_flushed": sum(r["pass_write_flushed"] for r in gated),
                      "min_frac_gated": min((r["frac_median_read_flushed"] for r in gated), default=None),
                      "peak_gbs": peak, "peak_source": peak_src, "sm_clock_mhz_now_max": sm_clock(),
                      "iters": args.iters, "warmup": args.warmup}})


if __name__ == "__main__":
    main()
