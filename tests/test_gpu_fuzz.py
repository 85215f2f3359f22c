"""Seeded random parity cases over the plan space, through the C ABI.

Each case draws P, B, S_local, heads per group, D, the element type, the source
strides (contiguous, views of a fused projection, padded rows), the mode (plain
or RMSNorm + RoPE, interleaved or half-split), the target layout (separate or
fused payload) and, sometimes, a head chunk, and compares the library's targets
with the oracle: relayout bit for bit, fused rows with parity_util's rule.  The
cases reach every kernel the host chooses between (block, staged bulk-copy,
register) and the 32- and 16-byte vector paths.
"""
import random

import pytest
import torch

import oracle
from parity_util import assert_fused_ok, bits_equal

pytestmark = pytest.mark.gpu

EPS = 1e-6
N_CASES = 150


@pytest.fixture(scope="module")
def tf():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ulysses_sequence_attention_tf_gb300 import binding, build
    build.build()
    binding.lib()
    binding.use_torch_allocator(True)
    yield binding
    torch.cuda.synchronize()
    binding.cache_clear()


def _draw(rng):
    fused = rng.random() < 0.5
    if fused:
        dtype = rng.choice([torch.bfloat16, torch.float16])
        D = rng.choice([32, 64, 128, 256])
    else:
        dtype = rng.choice([torch.bfloat16, torch.float16, torch.float32, torch.uint8])
        esize = torch.empty((), dtype=dtype).element_size()
        D = rng.choice([d for d in (8, 16, 24, 32, 48, 64, 96, 128, 256) if (d * esize) % 16 == 0])
    P = rng.randint(1, 8)
    Hl = rng.randint(1, 5)
    return dict(P=P, B=rng.randint(1, 3), Sl=rng.randint(1, 40), H=P * Hl, D=D, dtype=dtype, fused=fused,
                neox=fused and rng.random() < 0.4, layout=rng.choice(["contiguous", "fused", "padded"]),
                fused_layout=rng.random() < 0.3, chunk=rng.random() < 0.3, theta=rng.choice([500.0, 10000.0]))


def _sources(c, gen):
    """Q, K, V shard views [B, Sl, H, D] with the case's strides (CPU)."""
    P, B, Sl, H, D, dtype = c["P"], c["B"], c["Sl"], c["H"], c["D"], c["dtype"]
    esize = torch.empty((), dtype=dtype).element_size()
    pad = 16 // esize  # a row padding that keeps 16-byte strides

    def block(shape):
        if dtype == torch.uint8:
            return torch.randint(0, 256, shape, generator=gen, dtype=torch.uint8)
        return torch.randn(shape, generator=gen).to(dtype)

    out = {"q": [], "k": [], "v": []}
    for _ in range(P):
        if c["layout"] == "fused":
            buf = block((B, Sl, 3 * H * D))
            for i, key in enumerate("qkv"):
                out[key].append(buf[..., i * H * D:(i + 1) * H * D].unflatten(-1, (H, D)))
        elif c["layout"] == "padded":  # heads and tokens both padded
            for key in "qkv":
                buf = block((B, Sl, H, D + pad))
                out[key].append(buf[..., :D])
        else:
            for key in "qkv":
                out[key].append(block((B, Sl, H, D)))
    return out


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_case_vs_oracle(tf, case):
    rng = random.Random(1000 + case)
    c = _draw(rng)
    gen = torch.Generator().manual_seed(2000 + case)
    src = _sources(c, gen)
    P, B, Sl, H, D, dtype = c["P"], c["B"], c["Sl"], c["H"], c["D"], c["dtype"]
    Hl, S = H // P, P * Sl
    g = {k: [t.to("cuda") if t.is_contiguous() else
             torch.as_strided(torch.empty(t.untyped_storage().nbytes() // t.element_size(), dtype=dtype,
                                          device="cuda"), t.shape, t.stride()).copy_(t) for t in src[k]]
         for k in "qkv"}
    kw = {}
    wq = wk = None
    if c["fused"]:
        wq = (1.0 + 0.1 * torch.randn(D, generator=gen)).to(dtype)
        wk = (1.0 + 0.1 * torch.randn(D, generator=gen)).to(dtype)
        kw = dict(norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=c["theta"],
                  rope="neox" if c["neox"] else "interleaved")
    layout = "fused" if c["fused_layout"] else "bshd"
    fill = -3 if dtype != torch.uint8 else 7
    if c["fused_layout"]:
        outs = ([torch.full((B, S, Hl, 3 * D), fill, dtype=dtype, device="cuda") for _ in range(P)], None, None)
    else:
        outs = tuple([torch.full((B, S, Hl, D), fill, dtype=dtype, device="cuda") for _ in range(P)] for _ in "qkv")
    h0, h1 = 0, Hl
    if c["chunk"] and Hl > 1:
        h0 = rng.randint(0, Hl - 1)
        h1 = rng.randint(h0 + 1, Hl)
        tf.scatter_qkv_heads_into(g["q"], g["k"], g["v"], *outs, h0=h0, h1=h1, layout=layout, **kw)
    else:
        tf.scatter_qkv_into(g["q"], g["k"], g["v"], *outs, layout=layout, **kw)
    torch.cuda.synchronize()
    table = oracle.rope_table(c["theta"], S, D) if c["fused"] else None
    for x, key in enumerate("qkv"):
        if c["fused"] and key != "v":
            want = oracle.scatter_norm_rope(src[key], P, wq if key == "q" else wk, EPS, table,
                                            style="neox" if c["neox"] else "interleaved")
        else:
            want = oracle.scatter(src[key], P)
        for gi in range(P):
            got_full = outs[0][gi][..., x * D:(x + 1) * D] if c["fused_layout"] else outs[x][gi]
            got_full = got_full.cpu()
            got, exp = got_full[:, :, h0:h1], want[gi][:, :, h0:h1]
            if c["fused"] and key != "v":
                assert_fused_ok(got.contiguous(), exp.contiguous())
            else:
                assert bits_equal(got, exp), (c, key, gi)
            # heads outside the chunk keep the fill value
            outside = torch.cat([got_full[:, :, :h0], got_full[:, :, h1:]], dim=2)
            if outside.numel():
                assert bool((outside == fill).all()), (c, key, gi)


N_GATHER = 60


def _draw_gather(rng):
    dtype = rng.choice([torch.bfloat16, torch.float16, torch.bfloat16, torch.float32, torch.uint8])
    esize = torch.empty((), dtype=dtype).element_size()
    sizes = [d for d in (8, 16, 24, 32, 48, 64, 96, 128, 256) if (d * esize) % 16 == 0]
    D = rng.choice(sizes) if rng.random() < 0.4 else rng.choice([d for d in sizes if d * esize >= 256] or sizes)
    P = rng.randint(1, 8)
    Hl = rng.randint(1, 12)
    Sl = rng.choice([1, 7, 33, 64, 129, rng.randint(1, 200)])
    if rng.random() < 0.3:  # head bands of 1-2 KiB over many tokens: bulk copies with stores dealt to lanes
        rb = rng.choice([r for r in (256, 512) if r // esize in sizes] or [D * esize])
        D = rb // esize
        Hl = rng.randint(1024 // rb + 1, max(1024 // rb + 1, 2048 // rb))
        Sl = rng.randint(16, 200)
    return dict(P=P, B=rng.randint(1, 3), Sl=Sl, Hl=Hl, D=D, dtype=dtype, src=rng.choice(["contiguous", "padded"]),
                out=rng.choice(["cached", "own", "padded"]))


@pytest.mark.parametrize("case", range(N_GATHER))
def test_random_gather_vs_oracle(tf, case):
    """Head->sequence gather over random shapes, element types and strides: the
    host picks the register or the bulk-copy kernel by the size of the shards'
    head bands, and the bulk-copy kernel deals its stores out to the warp's lanes
    for units of many runs; every choice must give the oracle's bits."""
    rng = random.Random(3000 + case)
    c = _draw_gather(rng)
    P, B, Sl, Hl, D, dtype = c["P"], c["B"], c["Sl"], c["Hl"], c["D"], c["dtype"]
    S, H = P * Sl, P * Hl
    esize = torch.empty((), dtype=dtype).element_size()
    pad = 16 // esize
    gen = torch.Generator().manual_seed(4000 + case)

    def block(shape):
        if dtype == torch.uint8:
            return torch.randint(0, 256, shape, generator=gen, dtype=torch.uint8)
        return torch.randn(shape, generator=gen).to(dtype)

    if c["src"] == "padded":  # head rows padded: a strided view
        attn = [block((B, S, Hl, D + pad))[..., :D] for _ in range(P)]
    else:
        attn = [block((B, S, Hl, D)) for _ in range(P)]
    g_attn = []
    for t in attn:
        base = torch.empty(t.untyped_storage().nbytes() // t.element_size(), dtype=dtype, device="cuda")
        g_attn.append(torch.as_strided(base, t.shape, t.stride()).copy_(t))
    want = oracle.gather(attn, P)
    fill = 5 if dtype == torch.uint8 else -2
    if c["out"] == "cached":
        outs, _ = tf.gather_out(f"fuzz_gather_{case}", g_attn)
    else:
        width = H * D + (pad if c["out"] == "padded" else 0)  # padded token rows
        slabs = [torch.full((B, Sl, width), fill, dtype=dtype, device="cuda") for _ in range(P)]
        outs = [s[..., :H * D].unflatten(-1, (H, D)) for s in slabs]
        tf.gather_out(f"fuzz_gather_{case}", g_attn, outs)
    torch.cuda.synchronize()
    for r in range(P):
        assert bits_equal(outs[r].cpu(), want[r]), (c, r)
        if c["out"] == "padded":
            assert bool((slabs[r][..., H * D:] == fill).all()), (c, r)
