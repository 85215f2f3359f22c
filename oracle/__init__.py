"""CPU oracle for the Ulysses sequence<->head relayout and the fused Q/K RMSNorm + RoPE.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the product library never imports it and
shares no code with it.  The arithmetic lives in ``tf_oracle.c`` (plain C,
compiled with gcc, no FMA contraction); this module only compiles it on demand
and marshals torch CPU tensors (``data_ptr`` + element strides) into it.

Definitions and their sources are documented in ``tf_oracle.c``:
  * scatter  T_g[b, r*Sl + t, h, d] = S_r[b, t, g*Hl + h, d]
    (TeleFuser docs "Communication Architecture", Ulysses section)
  * gather   O_r[b, t, g*Hl + h, d] = A_g[b, r*Sl + t, h, d]   (same section)
  * RMSNorm + interleaved RoPE on Q/K rows (flashinfer PR #6332, "Assumptions"),
    and the half-split pairing (i, i + D/2) as a variant
  * the fused receive layout (flashinfer PR #6332, "Description", "Layouts")
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tf_oracle.c")
_LIB = os.path.join(_HERE, "libtf_oracle.so")
_CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
_lock = threading.Lock()
_lib = None

FMT = {torch.float16: 0, torch.bfloat16: 1}


def build(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc), if missing or stale."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, src, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the oracle library and declare its symbols."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.tfo_decode16.argtypes = [i32, ctypes.c_uint16]
        lib.tfo_decode16.restype = ctypes.c_double
        lib.tfo_encode16.argtypes = [i32, ctypes.c_double]
        lib.tfo_encode16.restype = ctypes.c_uint16
        lib.tfo_scatter.argtypes = [i32] * 6 + [vp, i64, i64, i64, vp]
        lib.tfo_scatter.restype = None
        lib.tfo_gather.argtypes = [i32] * 6 + [vp, i64, i64, i64, vp]
        lib.tfo_gather.restype = None
        lib.tfo_rope_table.argtypes = [ctypes.c_double, i32, i32, vp]
        lib.tfo_rope_table.restype = None
        lib.tfo_rmsnorm_rope_row.argtypes = [i32, i32, vp, vp, ctypes.c_float, vp, vp]
        lib.tfo_rmsnorm_rope_row.restype = None
        lib.tfo_rmsnorm_rope_neox_row.argtypes = [i32, i32, vp, vp, ctypes.c_float, vp, vp]
        lib.tfo_rmsnorm_rope_neox_row.restype = None
        lib.tfo_scatter_norm_rope.argtypes = [i32] * 6 + [vp, i64, i64, i64, vp, ctypes.c_float, vp, vp, i32]
        lib.tfo_scatter_norm_rope.restype = None
        lib.tfo_project_row.argtypes = [i32, i32, vp, vp, i64, i32, i32, vp]
        lib.tfo_project_row.restype = None
        lib.tfo_project.argtypes = [i32, i32, i32, i32, vp, i64, vp, i64, vp]
        lib.tfo_project.restype = None
        if path is None:
            _lib = lib
        return lib


def _ptrs(ts):
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    return arr


def _check_cpu(ts):
    for t in ts:
        if t.device.type != "cpu":
            raise ValueError("the oracle takes CPU tensors")
        if t.stride(-1) != 1:
            raise ValueError("the oracle needs unit stride along D")


def scatter(srcs, P: int, lib=None):
    """Sequence->head scatter of P source shards ``[B, Sl, H, D]`` (any strides with
    unit d stride, same strides for every shard) into P new contiguous targets
    ``[B, P*Sl, H/P, D]``.  Bit copy; any element type."""
    lib = lib or load()
    _check_cpu(srcs)
    B, Sl, H, D = srcs[0].shape
    sb, st, sh, _ = srcs[0].stride()
    Hl = H // P
    dsts = [torch.empty((B, P * Sl, Hl, D), dtype=srcs[0].dtype) for _ in range(P)]
    lib.tfo_scatter(P, B, Sl, H, D, srcs[0].element_size(), _ptrs(srcs), sb, st, sh, _ptrs(dsts))
    return dsts


def gather(srcs, P: int, lib=None):
    """Head->sequence gather of P head-group buffers ``[B, P*Sl, Hl, D]`` into P new
    contiguous outputs ``[B, Sl, P*Hl, D]``.  Bit copy; any element type."""
    lib = lib or load()
    _check_cpu(srcs)
    B, S, Hl, D = srcs[0].shape
    ab, at, ah, _ = srcs[0].stride()
    Sl, H = S // P, Hl * P
    dsts = [torch.empty((B, Sl, H, D), dtype=srcs[0].dtype) for _ in range(P)]
    lib.tfo_gather(P, B, Sl, H, D, srcs[0].element_size(), _ptrs(srcs), ab, at, ah, _ptrs(dsts))
    return dsts


def rope_table(theta: float, S: int, D: int, lib=None) -> torch.Tensor:
    """fp32 ``[S, D/2, 2]`` table of (cos, sin) of p * theta^(-2i/D)."""
    lib = lib or load()
    out = torch.empty((S, D // 2, 2), dtype=torch.float32)
    lib.tfo_rope_table(float(theta), S, D, out.data_ptr())
    return out


ROPE_STYLES = ("interleaved", "neox")


def rmsnorm_rope_row(x: torch.Tensor, w: torch.Tensor, eps: float, cs_row: torch.Tensor, lib=None,
                     style: str = "interleaved"):
    """RMSNorm + weight + RoPE of one head row ``x[D]`` with table row ``cs_row[D/2, 2]``:
    pairs (2i, 2i+1) for ``style="interleaved"``, (i, i + D/2) for ``style="neox"``."""
    if style not in ROPE_STYLES:
        raise ValueError(f"unknown RoPE style {style!r}")
    lib = lib or load()
    x, w, cs_row = x.contiguous(), w.contiguous(), cs_row.contiguous()
    _check_cpu([x, w, cs_row])
    out = torch.empty_like(x)
    fn = lib.tfo_rmsnorm_rope_neox_row if style == "neox" else lib.tfo_rmsnorm_rope_row
    fn(FMT[x.dtype], x.numel(), x.data_ptr(), w.data_ptr(), eps, cs_row.data_ptr(), out.data_ptr())
    return out


def scatter_norm_rope(srcs, P: int, w: torch.Tensor, eps: float, table: torch.Tensor, lib=None,
                      style: str = "interleaved"):
    """Scatter of one Q or K tensor with RMSNorm + RoPE (``style`` as in
    ``rmsnorm_rope_row``) at global positions p = r*Sl + t."""
    if style not in ROPE_STYLES:
        raise ValueError(f"unknown RoPE style {style!r}")
    lib = lib or load()
    w, table = w.contiguous(), table.contiguous()
    _check_cpu(list(srcs) + [w, table])
    B, Sl, H, D = srcs[0].shape
    sb, st, sh, _ = srcs[0].stride()
    if table.shape[0] < P * Sl or table.shape[1] * 2 != D:
        raise ValueError("table too small for the positions")
    Hl = H // P
    dsts = [torch.empty((B, P * Sl, Hl, D), dtype=srcs[0].dtype) for _ in range(P)]
    lib.tfo_scatter_norm_rope(FMT[srcs[0].dtype], P, B, Sl, H, D, _ptrs(srcs), sb, st, sh,
                              w.data_ptr(), eps, table.data_ptr(), _ptrs(dsts), int(style == "neox"))
    return dsts


def fused_payload(tq, tk, tv):
    """The fused receive layout of one scatter: per head group g the payload
    ``[B, S, Hl, 3*D]`` whose head row is the Q row, then the K row, then the V
    row of the separate targets (flashinfer PR #6332, "Description", layout
    "fused"; its 2-D form ``[B*S, 3*Hl*D]`` is the same memory)."""
    return [torch.cat([q, k, v], dim=-1) for q, k, v in zip(tq, tk, tv)]


def exchange_chunks(srcs, P: int):
    """All-to-all over destination-major payloads (flashinfer UlyssesCommunicator
    PCIe PR description, "Transforms", ``exchange_chunks``: each rank's payload
    already holds one chunk per destination, in destination order, and the
    exchange interleaves nothing): out_g = concat over r of chunk g of src_r.
    srcs: P byte tensors [P, chunk]; returns P new [P, chunk] tensors."""
    _check_cpu(srcs)
    out = []
    for g in range(P):
        out.append(torch.stack([srcs[r][g].clone() for r in range(P)]))
    return out


def scatter_heads_chunk(srcs, P: int, h0: int, h1: int, full_targets):
    """Head-chunk scatter: the targets ``full_targets`` (P tensors [B, P*Sl, Hl, D],
    copied) with heads [h0, h1) of every head group replaced by the plain
    scatter's values there; every other element keeps its previous value."""
    full = scatter(srcs, P)
    out = [t.clone() for t in full_targets]
    for g in range(P):
        out[g][:, :, h0:h1] = full[g][:, :, h0:h1]
    return out


def project(x: torch.Tensor, w: torch.Tensor, lib=None) -> torch.Tensor:
    """QKV projection of the rows of ``x`` [M, K] by the nn.Linear weight ``w``
    [N, K]: out[m, n] = round16(sum_k x[m, k] * w[n, k]) (exact sum, one rounding)."""
    lib = lib or load()
    w = w.contiguous()
    if x.stride(-1) != 1:
        x = x.contiguous()
    _check_cpu([x, w])
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K or K > 8192:
        raise ValueError("x [M, K] and w [N, K] with K <= 8192")
    out = torch.empty((M, N), dtype=x.dtype)
    lib.tfo_project(FMT[x.dtype], M, N, K, x.data_ptr(), x.stride(0), w.data_ptr(), w.stride(0), out.data_ptr())
    return out


def project_row_range(x_row: torch.Tensor, w: torch.Tensor, n0: int, n1: int, lib=None) -> torch.Tensor:
    """Features [n0, n1) of the projection of one hidden vector ``x_row`` [K]."""
    lib = lib or load()
    x_row, w = x_row.contiguous(), w.contiguous()
    _check_cpu([x_row, w])
    out = torch.empty((n1 - n0,), dtype=x_row.dtype)
    lib.tfo_project_row(FMT[x_row.dtype], x_row.numel(), x_row.data_ptr(), w.data_ptr(), w.stride(0), n0, n1,
                        out.data_ptr())
    return out


def project_qkv(x_shards, w: torch.Tensor, H: int, D: int, lib=None):
    """Q, K, V shards [B, Sl, H, D] of the projection of hidden-state shards
    ``x_shards`` [B, Sl, hidden] by ``w`` [3*H*D, hidden] (Q, K, V feature blocks
    in that order, head h at features [h*D, (h+1)*D) of each block)."""
    out = {"q": [], "k": [], "v": []}
    for x in x_shards:
        B, Sl, K = x.shape
        y = project(x.reshape(B * Sl, K), w, lib=lib).view(B, Sl, 3, H, D)
        for i, key in enumerate("qkv"):
            out[key].append(y[:, :, i].contiguous())
    return out


def decode16(dtype, bits: int) -> float:
    return load().tfo_decode16(FMT[dtype], bits & 0xFFFF)


def encode16(dtype, x: float) -> int:
    return load().tfo_encode16(FMT[dtype], float(x))
