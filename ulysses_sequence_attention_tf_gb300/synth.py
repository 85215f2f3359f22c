"""Seeded synthetic inputs shaped like the pages' Ulysses workloads.

This module draws random numbers and lays them out; it holds none of the
relayout, normalisation or rotation arithmetic.  Both the CUDA path and the CPU
oracle consume what it produces (the oracle after a device->host copy), so the
two sides always see the same bits.

Recipes (all values N(0, 1) unless stated, drawn in fp32 then rounded to the
16-bit I/O type; one ``torch.Generator`` per call, seeded, draws in a fixed order
q shards 0..P-1, then k, then v):

* ``contiguous``: each shard's Q/K/V is its own ``[B, S_local, H, D]`` buffer.
* ``fused``: each shard holds one fused projection ``[B, S_local, 3*H*D]`` and
  Q/K/V are views at column offsets 0, H*D, 2*H*D (row stride 3*H*D), the layout
  of a fused QKV projection output.
* ``v_strided``: Q/K contiguous, V a view into a fused ``[B, S_local, 3*H*D]``
  buffer at offset 2*H*D (the strided V that is handed over before Q/K
  normalisation in the TeleFuser MiniMax H3 path).
* RMSNorm weights: N(1, 0.1), shape ``[D]``, in the I/O type.
"""
from __future__ import annotations

import torch

# Named workloads (sizes of the pages' shapes; see the design notes for sources).
WORKLOADS = {
    # P=2, S=256, H=8, D=64 fp16, contiguous, pure scatter then gather.
    "tiny_p2": dict(P=2, B=1, S=256, H=8, D=64, dtype=torch.float16, layout="contiguous", norm_rope=False),
    # FLUX-like front end: P=4, S=4096, H=24, D=128 bf16, fused projection views, norm+RoPE.
    "flux_p4_s4096": dict(P=4, B=1, S=4096, H=24, D=128, dtype=torch.bfloat16, layout="fused", norm_rope=True),
    # Video-DiT: 21x30x52 = 32760 tokens, P=4, H=40, D=128 bf16, V strided, norm+RoPE.
    "video_dit_p4_s32760": dict(P=4, B=1, S=32760, H=40, D=128, dtype=torch.bfloat16, layout="v_strided",
                                norm_rope=True),
}


def padded_seq(S: int, P: int) -> int:
    """Smallest multiple of P that is >= S (sequence padding before sharding)."""
    return ((S + P - 1) // P) * P


def _normal(shape, dtype, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def make_generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def qkv_shards(P, B, S_local, H, D, dtype, *, seed=0, device="cpu", layout="contiguous",
               with_k=True, with_v=True, pad_from=None):
    """P shards of Q/K/V, each ``[B, S_local, H, D]``.

    ``pad_from``: if given (< S_local*P), global token rows at index >= pad_from are
    zero padding (the last shards' tails), as produced by padding a sequence of
    ``pad_from`` tokens up to a multiple of P.
    Returns dict(q=[..], k=[..] or None, v=[..] or None, backing=[..]).
    """
    gen = make_generator(seed, device)
    HD = H * D
    q, k, v, backing = [], [], [], []
    if layout == "contiguous":
        q = [_normal((B, S_local, H, D), dtype, gen, device) for _ in range(P)]
        k = [_normal((B, S_local, H, D), dtype, gen, device) for _ in range(P)] if with_k else None
        v = [_normal((B, S_local, H, D), dtype, gen, device) for _ in range(P)] if with_v else None
        backing = []
    elif layout == "fused":
        for _ in range(P):
            buf = _normal((B, S_local, 3 * HD), dtype, gen, device)
            backing.append(buf)
            q.append(buf[..., 0:HD].unflatten(-1, (H, D)))
            k.append(buf[..., HD:2 * HD].unflatten(-1, (H, D)))
            v.append(buf[..., 2 * HD:3 * HD].unflatten(-1, (H, D)))
        if not with_k:
            k = None
        if not with_v:
            v = None
    elif layout == "v_strided":
        q = [_normal((B, S_local, H, D), dtype, gen, device) for _ in range(P)]
        k = [_normal((B, S_local, H, D), dtype, gen, device) for _ in range(P)] if with_k else None
        if with_v:
            v = []
            for _ in range(P):
                buf = _normal((B, S_local, 3 * HD), dtype, gen, device)
                backing.append(buf)
                v.append(buf[..., 2 * HD:3 * HD].unflatten(-1, (H, D)))
        else:
            v = None
    else:
        raise ValueError(f"unknown layout {layout!r}")
    if pad_from is not None:
        for lst in (q, k, v):
            if lst is None:
                continue
            for r, x in enumerate(lst):
                lo = max(0, pad_from - r * S_local)
                if lo < S_local:
                    x[:, lo:].zero_()
    return dict(q=q, k=k, v=v, backing=backing)


def projection_inputs(P, B, S_local, hidden, H, D, dtype, *, seed=0, device="cpu", x_pad=0, w_pad=0,
                      dist="normal"):
    """Hidden-state shards ``x[r]`` [B, S_local, hidden] and the QKV weight ``w``
    [3*H*D, hidden] in the I/O type.  dist="normal": x ~ N(0, 1), w ~ N(0, 1/hidden)
    (projected values ~N(0, 1)).  dist="dyadic": x = i/8 and w = j/16 for uniform
    integers |i| <= 8, |j| <= 16, so every product is a multiple of 2^-7 of
    magnitude <= 1 and every partial sum of up to 2^16 of them is exact in fp32.
    ``x_pad`` / ``w_pad`` extra elements per row make the rows of x / w strided
    views (row stride hidden + pad)."""
    gen = make_generator(seed + 104729, device)

    def draw(shape, scale):
        if dist == "dyadic":
            return torch.randint(-scale, scale + 1, shape, generator=gen, device=device).to(torch.float32) / scale
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)

    xs = []
    for _ in range(P):
        xs.append(draw((B, S_local, hidden + x_pad), 8).to(dtype)[..., :hidden])
    wb = draw((3 * H * D, hidden + w_pad), 16)
    if dist != "dyadic":
        wb = wb * hidden ** -0.5
    w = wb.to(dtype)[:, :hidden]
    return xs, w


def norm_weights(D, dtype, *, seed=0, device="cpu"):
    """(w_q, w_k), each ``[D]`` ~ N(1, 0.1) in the I/O type."""
    gen = make_generator(seed + 7919, device)
    wq = (1.0 + 0.1 * torch.randn((D,), generator=gen, device=device, dtype=torch.float32)).to(dtype)
    wk = (1.0 + 0.1 * torch.randn((D,), generator=gen, device=device, dtype=torch.float32)).to(dtype)
    return wq, wk


def attn_outputs(P, B, S, Hl, D, dtype, *, seed=0, device="cpu"):
    """P head-group attention outputs ``[B, S, Hl, D]`` ~ N(0, 1)."""
    gen = make_generator(seed + 104729, device)
    return [_normal((B, S, Hl, D), dtype, gen, device) for _ in range(P)]


def unique_id_shards(P, B, S_local, H, D, *, device="cpu"):
    """P int16 shards whose elements are all distinct (a running counter), for
    exactly-once checks; requires P*B*S_local*H*D <= 65536."""
    n = B * S_local * H * D
    if P * n > 65536:
        raise ValueError("too many elements for distinct 16-bit ids")
    ids = torch.arange(P * n, dtype=torch.int32, device=device) - 32768
    return [ids[r * n:(r + 1) * n].to(torch.int16).view(B, S_local, H, D).clone() for r in range(P)]


# Head rows with extreme or non-finite values, for the fused path's edge cases.
# bf16 reaches 3.4e38, so squares overflow fp32 from |x| = 2^64 on; fp16 tops out
# at 65504 (no overflow), so its cases are the non-finite and the tiny ones.
EDGE_KINDS = {
    torch.bfloat16: ("const_2^63", "const_2^64", "const_2^100", "normal_2^60", "normal_2^62", "spike_2^64",
                     "spike_2^100", "inf", "-inf", "nan", "subnormal", "zero", "tiny"),
    torch.float16: ("max", "inf", "-inf", "nan", "subnormal", "zero", "tiny"),
}


def edge_row(kind, D, dtype, gen):
    """One head row [D] of the edge kind ``kind`` (CPU): constant rows, N(0, 1)
    rows scaled by a power of two, a single large element in an N(0, 1) row, one
    +-inf or NaN element in an N(0, 1) row, random subnormals, zeros, or N(0, 1)
    scaled to 2^-70 (bf16) / 2^-20 (fp16)."""
    base = torch.randn((D,), generator=gen)
    at = int(torch.randint(D, (1,), generator=gen))
    name, _, arg = kind.partition("_")
    if name == "const":
        return torch.full((D,), 2.0 ** int(arg[2:]), dtype=dtype)
    if name == "normal":
        return (base * 2.0 ** int(arg[2:])).to(dtype)
    if name in ("spike", "inf", "-inf", "nan"):
        row = base.to(dtype)
        row[at] = {"spike": 2.0 ** int(arg[2:] or 0), "inf": float("inf"), "-inf": float("-inf"),
                   "nan": float("nan")}[name]
        return row
    if name == "max":
        return torch.full((D,), torch.finfo(dtype).max, dtype=dtype) * torch.sign(base).to(dtype)
    if name == "subnormal":
        frac_bits = 7 if dtype == torch.bfloat16 else 10
        mag = torch.randint(1, 1 << frac_bits, (D,), generator=gen, dtype=torch.int32)
        sign = torch.randint(0, 2, (D,), generator=gen, dtype=torch.int32) << 15
        return (sign | mag).to(torch.int16).view(dtype)
    if name == "zero":
        return torch.zeros((D,), dtype=dtype)
    if name == "tiny":
        return (base * 2.0 ** (-70 if dtype == torch.bfloat16 else -20)).to(dtype)
    raise ValueError(f"unknown edge kind {kind!r}")


def plant_edge_rows(shards, *, seed=0, every=7):
    """Overwrite head rows of P shard tensors [B, S_local, H, D] (CPU, in place)
    with edge rows: every ``every``-th row in shard-major order cycles through the
    kinds of the element type, and shard 0's first token gets one kind on all its
    heads.  Returns the number of rows planted."""
    dtype = shards[0].dtype
    kinds = EDGE_KINDS[dtype]
    gen = make_generator(seed + 1299709, "cpu")
    B, Sl, H, D = shards[0].shape
    n = 0
    for r, x in enumerate(shards):
        for b in range(B):
            for t in range(Sl):
                for h in range(H):
                    i = ((r * B + b) * Sl + t) * H + h
                    if i % every == 0 or (r == 0 and b == 0 and t == 0):
                        kind = kinds[(i // every + (0 if t else h)) % len(kinds)]
                        x[b, t, h] = edge_row(kind, D, dtype, gen)
                        n += 1
    return n


def move(d, device):
    """Copy a ``qkv_shards`` result to ``device`` keeping every view's strides
    (views into a fused projection stay views into the copied projection)."""
    backing = [b.to(device) for b in d["backing"]]
    ptrs = [b.data_ptr() for b in d["backing"]]
    out = {"backing": backing}
    for key in ("q", "k", "v"):
        if d[key] is None:
            out[key] = None
            continue
        res = []
        for x in d[key]:
            base = x._base
            if base is None or base.data_ptr() not in ptrs:
                res.append(x.to(device))
                continue
            i = ptrs.index(base.data_ptr())
            off = x.storage_offset() - base.storage_offset()
            res.append(backing[i].as_strided(x.shape, x.stride(), backing[i].storage_offset() + off))
        out[key] = res
    return out
