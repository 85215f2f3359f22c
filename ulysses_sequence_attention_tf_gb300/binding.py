"""Thin ctypes binding of ``libtf_ulysses.so`` (the C ABI in include/tf_ulysses.h).

Argument marshalling only: torch supplies device memory, streams and the
tensors' data pointers/strides; every step of the relayout runs in the
library's CUDA kernels.  There is no fallback: if the library is missing or a
call fails, a ``TfUlyssesError`` is raised.

Names follow the C ABI: ``scatter_qkv`` / ``scatter_qkv_into`` / ``gather_out``
/ ``rope_table`` / ``cache_clear`` ...
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# the in-tree build, or another build of the same library named by TF_ULYSSES_LIBRARY
LIB_PATH = os.environ.get("TF_ULYSSES_LIBRARY") or os.path.join(_PKG, "libtf_ulysses.so")

TF_OK, TF_ERR_INVALID, TF_ERR_DIVISIBILITY, TF_ERR_ALIGNMENT = 0, 1, 2, 3
TF_ERR_UNSUPPORTED, TF_ERR_OOM, TF_ERR_CUDA, TF_ERR_BUSY = 4, 5, 6, 7
STATUS_NAMES = {0: "TF_OK", 1: "TF_ERR_INVALID", 2: "TF_ERR_DIVISIBILITY", 3: "TF_ERR_ALIGNMENT",
                4: "TF_ERR_UNSUPPORTED", 5: "TF_ERR_OOM", 6: "TF_ERR_CUDA", 7: "TF_ERR_BUSY"}
TF_MODE_SCATTER, TF_MODE_SCATTER_NORM_ROPE, TF_MODE_GATHER = 0, 1, 2
TF_MODE_FLAG_FUSED_LAYOUT, TF_MODE_FLAG_ROPE_NEOX = 0x100, 0x200
MAX_SHARDS = 8
CACHE_CAPACITY = 12

_DTYPE_CODE = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2, torch.int32: 2,
               torch.uint8: 3, torch.int8: 3}
for _name in ("float8_e4m3fn", "float8_e5m2"):
    if hasattr(torch, _name):
        _DTYPE_CODE[getattr(torch, _name)] = 3


class TfUlyssesError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Strides(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("t", ctypes.c_int64), ("h", ctypes.c_int64)]


class NormRope(ctypes.Structure):
    _fields_ = [("q_weight", ctypes.c_void_p), ("k_weight", ctypes.c_void_p), ("eps", ctypes.c_float),
                ("theta", ctypes.c_float), ("cos_sin", ctypes.c_void_p)]


class Targets(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p * MAX_SHARDS), ("k", ctypes.c_void_p * MAX_SHARDS),
                ("v", ctypes.c_void_p * MAX_SHARDS), ("done", ctypes.c_void_p)]


ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p)

_lock = threading.Lock()
_lib = None


def _declare(lib):
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    PP = ctypes.POINTER(ctypes.c_void_p)
    lib.tf_ulysses_scatter_qkv.argtypes = [ctypes.c_char_p, PP, PP, PP, ctypes.POINTER(Strides),
                                           i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(NormRope),
                                           vp, ctypes.POINTER(Targets)]
    lib.tf_ulysses_scatter_qkv_into.argtypes = [PP, PP, PP, ctypes.POINTER(Strides), i32, i32, i32, i32, i32,
                                                i32, i32, ctypes.POINTER(NormRope), PP, PP, PP, vp]
    lib.tf_ulysses_scatter_qkv_noalloc.argtypes = lib.tf_ulysses_scatter_qkv_into.argtypes
    lib.tf_ulysses_scatter_qkv_heads_into.argtypes = [PP, PP, PP, ctypes.POINTER(Strides), i32, i32, i32, i32, i32,
                                                      i32, i32, ctypes.POINTER(NormRope), i32, i32, PP, PP, PP, vp]
    lib.tf_ulysses_exchange_chunks.argtypes = [PP, PP, i32, ctypes.c_size_t, vp]
    lib.tf_ulysses_project_qkv_into.argtypes = [PP, i64, vp, i64, i32, i32, i32, i32, i32, i32, i32, i32,
                                                ctypes.POINTER(NormRope), PP, PP, PP, vp]
    lib.tf_ulysses_gather_out.argtypes = [ctypes.c_char_p, PP, ctypes.POINTER(Strides), i32, i32, i32, i32, i32,
                                          i32, PP, ctypes.POINTER(Strides), vp, ctypes.POINTER(Targets)]
    lib.tf_ulysses_rope_table.argtypes = [ctypes.c_float, i32, i32, vp, ctypes.POINTER(ctypes.c_void_p)]
    for name in ("tf_ulysses_scatter_qkv_heads_into", "tf_ulysses_exchange_chunks", "tf_ulysses_project_qkv_into",
                 "tf_ulysses_scatter_qkv", "tf_ulysses_scatter_qkv_into", "tf_ulysses_scatter_qkv_noalloc",
                 "tf_ulysses_gather_out",
                 "tf_ulysses_rope_table", "tf_ulysses_cache_clear"):
        getattr(lib, name).restype = i32
    lib.tf_ulysses_cache_clear.argtypes = []
    lib.tf_ulysses_cache_entries.argtypes = []
    lib.tf_ulysses_cache_entries.restype = i32
    lib.tf_ulysses_set_allocator.argtypes = [ALLOC_FN, FREE_FN, vp]
    lib.tf_ulysses_set_allocator.restype = None
    lib.tf_ulysses_device_status.argtypes = [i32, ctypes.POINTER(ctypes.c_uint)]
    lib.tf_ulysses_device_status.restype = i32
    lib.tf_ulysses_last_error.argtypes = []
    lib.tf_ulysses_last_error.restype = ctypes.c_char_p
    lib.tf_ulysses_launch_count.argtypes = []
    lib.tf_ulysses_launch_count.restype = ctypes.c_uint64
    lib.tf_ulysses_selftest_wait.argtypes = [ctypes.c_ulonglong, vp]
    lib.tf_ulysses_selftest_wait.restype = i32
    lib.tf_ulysses_set_slots.argtypes = [ctypes.c_char_p, i32]
    lib.tf_ulysses_set_slots.restype = i32
    lib.tf_ulysses_alloc_count.argtypes = []
    lib.tf_ulysses_alloc_count.restype = ctypes.c_uint64
    lib.tf_ulysses_abi_version.argtypes = []
    lib.tf_ulysses_abi_version.restype = i32
    return lib


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise TfUlyssesError(TF_ERR_INVALID, f"{LIB_PATH} is not built (run __graft_entry__.build())")
                _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def _check(status: int):
    if status != TF_OK:
        raise TfUlyssesError(status, lib().tf_ulysses_last_error().decode(errors="replace"))


# ---------------------------------------------------------------- marshalling
def _ptr_array(ts):
    if ts is None:
        return None
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _strides_of(ts, ndim_names="[B, tokens, heads, D]"):
    s = ts[0].stride()
    if ts[0].dim() != 4:
        raise ValueError(f"expected 4-d views {ndim_names}")
    if ts[0].shape[-1] > 1 and s[3] != 1:
        raise ValueError("the D dimension must have stride 1")
    for t in ts[1:]:
        if t.stride() != s or t.shape != ts[0].shape or t.dtype != ts[0].dtype:
            raise ValueError("all shards of a tensor must share shape, dtype and strides")
    return Strides(s[0], s[1], s[2])


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class _DeviceBuffer:
    """Zero-copy view of library-owned device memory for torch.as_tensor."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 2, "strides": None}


# Flat tensors over library-owned memory, by (address, elements, dtype, device).
# Cached targets come back at the same addresses call after call, so their views
# are cut from a cached flat tensor instead of being built from the array
# interface each time; a view owns no memory, so an entry whose memory was freed
# and reused still views exactly that address range.
_WRAP_CACHE = {}
_WRAP_CACHE_MAX = 4096


def _wrap(ptr, shape, dtype, device):
    if not ptr or 0 in shape:
        return torch.empty(shape, dtype=dtype, device=device)
    numel = 1
    for n in shape:
        numel *= n
    key = (ptr, numel, dtype, device)
    flat = _WRAP_CACHE.get(key)
    if flat is None:
        esize = torch.empty((), dtype=dtype).element_size()
        typestr = {1: "|u1", 2: "<i2", 4: "<i4", 8: "<i8"}[esize]
        with torch.cuda.device(device):
            flat = torch.as_tensor(_DeviceBuffer(ptr, (numel,), typestr), device=device).view(dtype)
        if len(_WRAP_CACHE) >= _WRAP_CACHE_MAX:
            _WRAP_CACHE.clear()
        _WRAP_CACHE[key] = flat
    return flat.view(shape)


def _dtype_code(dtype):
    if dtype not in _DTYPE_CODE:
        raise ValueError(f"unsupported dtype {dtype}")
    return _DTYPE_CODE[dtype]


def _norm_rope(q_weight, k_weight, eps, theta, cos_sin):
    nr = NormRope()
    nr.q_weight = q_weight.data_ptr() if q_weight is not None else None
    nr.k_weight = k_weight.data_ptr() if k_weight is not None else None
    nr.eps = float(eps)
    nr.theta = float(theta)
    nr.cos_sin = cos_sin.data_ptr() if cos_sin is not None else None
    return nr


def _scatter_args(q, k, v):
    P = len(q)
    if not 1 <= P <= MAX_SHARDS:
        raise ValueError(f"P={P} outside [1, {MAX_SHARDS}]")
    B, Sl, H, D = q[0].shape
    strides = (Strides * 3)()
    for i, ts in enumerate((q, k, v)):
        if ts is None:
            continue
        if len(ts) != P or ts[0].shape != q[0].shape or ts[0].dtype != q[0].dtype:
            raise ValueError("q, k and v must have P shards of the same shape and dtype")
        strides[i] = _strides_of(ts)
    return P, B, Sl, H, D, strides


def _mode(norm_rope, rope, layout):
    if rope not in ("interleaved", "neox"):
        raise ValueError(f"rope must be 'interleaved' or 'neox', not {rope!r}")
    if layout not in ("bshd", "fused"):
        raise ValueError(f"layout must be 'bshd' or 'fused', not {layout!r}")
    mode = TF_MODE_SCATTER_NORM_ROPE if norm_rope else TF_MODE_SCATTER
    if rope == "neox":
        mode |= TF_MODE_FLAG_ROPE_NEOX  # the library rejects it without norm_rope
    if layout == "fused":
        mode |= TF_MODE_FLAG_FUSED_LAYOUT
    return mode


def _check_targets(outs, layout):
    for o in outs:
        if o is not None and any(not t.is_contiguous() for t in o):
            raise ValueError("targets must be contiguous " +
                             ("[B, S, H/P, 3*D] payloads" if layout == "fused" else "[B, S, H/P, D]"))


# ---------------------------------------------------------------- public API
def scatter_qkv(tag, q, k=None, v=None, *, norm_rope=False, q_weight=None, k_weight=None, eps=1e-6,
                theta=10000.0, cos_sin=None, rope="interleaved", layout="bshd", stream=None):
    """Sequence->head scatter of P shards ``[B, S_local, H, D]`` of Q (and K, V)
    into cached final-layout targets, in one launch.

    Returns ``(q_targets, k_targets, v_targets, done_event_handle)``: lists of P
    ``[B, P*S_local, H/P, D]`` tensors viewing library-owned memory (valid until the
    next call with the same key, eviction or ``cache_clear``), ``None`` for absent
    tensors.  With ``norm_rope=True``, Q and K get RMSNorm (eps, q_weight/k_weight)
    and RoPE at global positions (theta, or an fp32 ``cos_sin`` table
    ``[>= S, D/2, 2]``), pairs (2i, 2i+1) for ``rope="interleaved"`` or (i, i + D/2)
    for ``rope="neox"``; V is copied bit for bit.  ``layout="fused"`` (q, k, v
    all required) writes one ``[B, S, H/P, 3*D]`` payload per head group and returns
    Q, K and V as views into it (``fused_payloads`` recovers the payloads).
    """
    P, B, Sl, H, D, strides = _scatter_args(q, k, v)
    mode = _mode(norm_rope, rope, layout)
    nr = _norm_rope(q_weight, k_weight, eps, theta, cos_sin) if norm_rope else None
    out = Targets()
    _check(lib().tf_ulysses_scatter_qkv(
        tag.encode() if isinstance(tag, str) else tag, _ptr_array(q), _ptr_array(k), _ptr_array(v), strides,
        P, B, Sl, H, D, _dtype_code(q[0].dtype), mode, ctypes.byref(nr) if nr is not None else None,
        _stream_handle(stream), ctypes.byref(out)))
    S, Hl = P * Sl, H // P
    dev = q[0].device
    if layout == "fused":
        pay = [_wrap(out.q[g], (B, S, Hl, 3 * D), q[0].dtype, dev) for g in range(P)]
        return ([t[..., :D] for t in pay], [t[..., D:2 * D] for t in pay], [t[..., 2 * D:] for t in pay],
                out.done)
    res = []
    for arr, ts in ((out.q, q), (out.k, k), (out.v, v)):
        res.append(None if ts is None else [_wrap(arr[g], (B, S, Hl, D), q[0].dtype, dev) for g in range(P)])
    return res[0], res[1], res[2], out.done


def fused_payloads(q_targets):
    """The ``[B, S, H/P, 3*D]`` payloads behind the Q views returned by
    ``scatter_qkv(..., layout="fused")``."""
    res = []
    for t in q_targets:
        B, S, Hl, D = t.shape
        if t.stride() != (S * Hl * 3 * D, Hl * 3 * D, 3 * D, 1):
            raise ValueError("not a Q view of a fused-layout payload")
        res.append(t.as_strided((B, S, Hl, 3 * D), (S * Hl * 3 * D, Hl * 3 * D, 3 * D, 1)))
    return res


def scatter_qkv_into(q, k, v, q_out, k_out=None, v_out=None, *, norm_rope=False, q_weight=None, k_weight=None,
                     eps=1e-6, theta=10000.0, cos_sin=None, rope="interleaved", layout="bshd", stream=None):
    """Same scatter into caller-owned contiguous targets ``[B, P*S_local, H/P, D]``;
    with ``layout="fused"``, ``q_out`` holds the P payloads ``[B, P*S_local, H/P, 3*D]``
    and ``k_out``, ``v_out`` stay None."""
    P, B, Sl, H, D, strides = _scatter_args(q, k, v)
    _check_targets((q_out, k_out, v_out), layout)
    mode = _mode(norm_rope, rope, layout)
    nr = _norm_rope(q_weight, k_weight, eps, theta, cos_sin) if norm_rope else None
    _check(lib().tf_ulysses_scatter_qkv_into(
        _ptr_array(q), _ptr_array(k), _ptr_array(v), strides, P, B, Sl, H, D, _dtype_code(q[0].dtype), mode,
        ctypes.byref(nr) if nr is not None else None, _ptr_array(q_out), _ptr_array(k_out), _ptr_array(v_out),
        _stream_handle(stream)))
    return q_out, k_out, v_out


def scatter_qkv_noalloc(q, k, v, q_out, k_out=None, v_out=None, *, norm_rope=False, q_weight=None, k_weight=None,
                        eps=1e-6, theta=10000.0, cos_sin=None, rope="interleaved", layout="bshd", stream=None):
    """``scatter_qkv_into`` for callers that cannot allocate device memory: the
    library allocates nothing; a needed cos/sin table lives in the library's
    fixed 16 MiB device scratch (P*S_local*D <= 4 Mi floats), rebuilt only when
    it does not already hold this (theta, rows, D).  A rebuild whose work
    overlaps on the GPU with another call's scatter races with it."""
    P, B, Sl, H, D, strides = _scatter_args(q, k, v)
    _check_targets((q_out, k_out, v_out), layout)
    mode = _mode(norm_rope, rope, layout)
    nr = _norm_rope(q_weight, k_weight, eps, theta, cos_sin) if norm_rope else None
    _check(lib().tf_ulysses_scatter_qkv_noalloc(
        _ptr_array(q), _ptr_array(k), _ptr_array(v), strides, P, B, Sl, H, D, _dtype_code(q[0].dtype), mode,
        ctypes.byref(nr) if nr is not None else None, _ptr_array(q_out), _ptr_array(k_out), _ptr_array(v_out),
        _stream_handle(stream)))
    return q_out, k_out, v_out


def scatter_qkv_heads_into(q, k, v, q_out, k_out=None, v_out=None, *, h0, h1, norm_rope=False, q_weight=None,
                           k_weight=None, eps=1e-6, theta=10000.0, cos_sin=None, rope="interleaved", layout="bshd",
                           stream=None):
    """``scatter_qkv_into`` restricted to heads [h0, h1) of every head band: those
    heads of the caller's targets are written, every other element is kept."""
    P, B, Sl, H, D, strides = _scatter_args(q, k, v)
    _check_targets((q_out, k_out, v_out), layout)
    mode = _mode(norm_rope, rope, layout)
    nr = _norm_rope(q_weight, k_weight, eps, theta, cos_sin) if norm_rope else None
    _check(lib().tf_ulysses_scatter_qkv_heads_into(
        _ptr_array(q), _ptr_array(k), _ptr_array(v), strides, P, B, Sl, H, D, _dtype_code(q[0].dtype), mode,
        ctypes.byref(nr) if nr is not None else None, int(h0), int(h1), _ptr_array(q_out), _ptr_array(k_out),
        _ptr_array(v_out), _stream_handle(stream)))
    return q_out, k_out, v_out


def project_qkv_into(x, w_qkv, H, q_out, k_out=None, v_out=None, *, norm_rope=False, q_weight=None, k_weight=None,
                     eps=1e-6, theta=10000.0, cos_sin=None, rope="interleaved", layout="bshd", stream=None):
    """QKV projection fused with the scatter: ``x`` is P shards ``[B, S_local,
    hidden]`` (bf16, unit stride along hidden, rows of one shard equally spaced),
    ``w_qkv`` the ``[3*H*D, hidden]`` weight (nn.Linear layout, D = 128).  Q, K, V
    head rows land in the targets as ``scatter_qkv_into`` writes them, after the
    RMSNorm + RoPE on Q/K when ``norm_rope``."""
    P = len(x)
    B, Sl, hidden = x[0].shape
    for t in x:
        if t.shape != x[0].shape or t.stride() != x[0].stride() or t.dtype != x[0].dtype:
            raise ValueError("all x shards must share shape, strides and dtype")
    if x[0].stride(2) != 1 or (B > 1 and x[0].stride(0) != Sl * x[0].stride(1)):
        raise ValueError("x rows must be equally spaced with unit stride along hidden")
    if w_qkv.stride(1) != 1:
        raise ValueError("w_qkv needs unit stride along hidden")
    D = w_qkv.shape[0] // (3 * H)
    _check_targets((q_out, k_out, v_out), layout)
    mode = _mode(norm_rope, rope, layout)
    nr = _norm_rope(q_weight, k_weight, eps, theta, cos_sin) if norm_rope else None
    _check(lib().tf_ulysses_project_qkv_into(
        _ptr_array(x), x[0].stride(1) if Sl > 1 or B > 1 else hidden, ctypes.c_void_p(w_qkv.data_ptr()),
        w_qkv.stride(0), P, B, Sl, hidden, H, D, _dtype_code(x[0].dtype), mode,
        ctypes.byref(nr) if nr is not None else None, _ptr_array(q_out), _ptr_array(k_out), _ptr_array(v_out),
        _stream_handle(stream)))
    return q_out, k_out, v_out


def exchange_chunks(src, dst=None, *, stream=None):
    """All-to-all over destination-major payloads: P tensors ``src[r]`` of P equal
    chunks (chunk g goes to rank g) -> ``dst[g]`` holding chunk g of every rank in
    rank order.  Tensors must be contiguous with P*chunk bytes, chunk a multiple
    of 16 bytes; ``dst`` defaults to new tensors shaped like ``src``."""
    P = len(src)
    if any(not t.is_contiguous() or t.shape != src[0].shape or t.dtype != src[0].dtype for t in src):
        raise ValueError("src must be P contiguous tensors of one shape and dtype")
    nbytes = src[0].numel() * src[0].element_size()
    if nbytes % P:
        raise ValueError("a payload must split into P equal chunks")
    if dst is None:
        dst = [torch.empty_like(t) for t in src]
    if any(not t.is_contiguous() or t.numel() * t.element_size() != nbytes for t in dst):
        raise ValueError("dst must be P contiguous tensors of the payload size")
    _check(lib().tf_ulysses_exchange_chunks(_ptr_array(src), _ptr_array(dst), P, nbytes // P, _stream_handle(stream)))
    return dst


def gather_out(tag, attn, out=None, *, stream=None):
    """Head->sequence gather of P head-group outputs ``[B, S, H/P, D]`` into P shard
    outputs ``[B, S/P, H, D]`` -- cached library buffers, or ``out`` (P caller tensors,
    any strides with unit D stride).  Returns ``(outputs, done_event_handle)``."""
    P = len(attn)
    B, S, Hl, D = attn[0].shape
    if S % P:
        raise ValueError(f"S={S} is not divisible by P={P}")
    Sl, H = S // P, Hl * P
    a_str = _strides_of(attn)
    o_str = _strides_of(out) if out is not None else None
    res = Targets()
    _check(lib().tf_ulysses_gather_out(
        tag.encode() if isinstance(tag, str) else tag, _ptr_array(attn), ctypes.byref(a_str), P, B, Sl, H, D,
        _dtype_code(attn[0].dtype), _ptr_array(out), ctypes.byref(o_str) if o_str is not None else None,
        _stream_handle(stream), ctypes.byref(res)))
    if out is not None:
        return list(out), res.done
    return [_wrap(res.q[r], (B, Sl, H, D), attn[0].dtype, attn[0].device) for r in range(P)], res.done


def rope_table(theta, S, D, *, stream=None, device=None):
    """The library's resident fp32 cos/sin table ``[S, D/2, 2]`` (a view)."""
    ptr = ctypes.c_void_p()
    _check(lib().tf_ulysses_rope_table(float(theta), int(S), int(D), _stream_handle(stream), ctypes.byref(ptr)))
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    return _wrap(ptr.value, (S, D // 2, 2), torch.float32, dev)


def cache_clear():
    _check(lib().tf_ulysses_cache_clear())


def device_status(clear: bool = False) -> int:
    """The staged kernels' device status word (0 = every in-kernel wait completed)."""
    v = ctypes.c_uint()
    _check(lib().tf_ulysses_device_status(1 if clear else 0, ctypes.byref(v)))
    return int(v.value)


def selftest_wait(cycles: int, *, stream=None):
    """Launch the bounded-wait self-test (a wait nothing satisfies, given up after
    ``cycles`` clock cycles); ``device_status()`` then has bit 1 set."""
    _check(lib().tf_ulysses_selftest_wait(int(cycles), _stream_handle(stream)))


def set_slots(tag, num_slots: int):
    """Rotating target sets for cache entries of ``tag`` created from now on."""
    _check(lib().tf_ulysses_set_slots(tag.encode() if isinstance(tag, str) else tag, int(num_slots)))


def alloc_count() -> int:
    """Device allocations the library has made in this process."""
    return int(lib().tf_ulysses_alloc_count())


def cache_entries() -> int:
    return lib().tf_ulysses_cache_entries()


def launch_count() -> int:
    return int(lib().tf_ulysses_launch_count())


def abi_version() -> int:
    return lib().tf_ulysses_abi_version()


# torch-backed allocator: cached targets and tables come from torch's caching allocator
_alloc_refs = None


def _torch_alloc(nbytes, stream, ctx):
    try:
        return torch.cuda.caching_allocator_alloc(int(nbytes), stream=int(stream or 0))
    except Exception:  # noqa: BLE001 -- the library reports TF_ERR_OOM
        return None


def _torch_free(ptr, nbytes, stream, ctx):
    torch.cuda.caching_allocator_delete(ptr)


def use_torch_allocator(enable: bool = True):
    """Route the library's device allocations through torch's caching allocator
    (default: cudaMallocAsync on the calling stream)."""
    global _alloc_refs
    if enable:
        _alloc_refs = (ALLOC_FN(_torch_alloc), FREE_FN(_torch_free))
        lib().tf_ulysses_set_allocator(_alloc_refs[0], _alloc_refs[1], None)
    else:
        lib().tf_ulysses_set_allocator(ALLOC_FN(), FREE_FN(), None)
        _alloc_refs = None
