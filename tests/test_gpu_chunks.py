"""Parity of the head-chunk scatter and of the chunk exchange with the CPU oracle,
through the C ABI.

Head chunk: heads [h0, h1) of every band into the final-layout targets, every
other target element kept (flashinfer PR #6332 commit message, "Speedup",
baselines B2/B3 with `scatter_qkv_head_chunk`).  Chunk exchange: the all-to-all
over destination-major payloads (flashinfer UlyssesCommunicator PCIe PR
description, "Transforms", `exchange_chunks`).  Both are bit copies (the fused
rows of a head chunk use the tolerance of parity_util).
"""
import pytest
import torch

import oracle
from parity_util import assert_fused_ok, bits_equal
from ulysses_sequence_attention_tf_gb300 import synth

pytestmark = pytest.mark.gpu

EPS = 1e-6
THETA = 10000.0
SENTINEL = -3.0


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


def _targets(P, B, S, Hl, D, dtype, width=1):
    return [torch.full((B, S, Hl, width * D), SENTINEL, dtype=dtype, device="cuda") for _ in range(P)]


# ------------------------------------------------------------------ head chunks
@pytest.mark.parametrize("D,dtype", [(128, torch.bfloat16), (64, torch.float16), (36, torch.float32)])
def test_head_chunks_partition_equals_whole_scatter(tf, D, dtype):
    P, B, Sl, H = 4, 2, 33, 24
    Hl, S = H // P, P * Sl
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=D, layout="fused")
    g = synth.move(d, "cuda")
    outs = {k: _targets(P, B, S, Hl, D, dtype) for k in "qkv"}
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for i, (h0, h1) in enumerate(((0, 1), (1, 4), (4, Hl))):  # chunks on alternating streams
        tf.scatter_qkv_heads_into(g["q"], g["k"], g["v"], outs["q"], outs["k"], outs["v"], h0=h0, h1=h1,
                                  stream=streams[i % 2])
    torch.cuda.synchronize()
    for key in "qkv":
        want = oracle.scatter(d[key], P)
        for i in range(P):
            assert bits_equal(outs[key][i].cpu(), want[i]), (key, i)


def test_single_head_chunk_leaves_other_heads(tf):
    P, B, Sl, H, D = 2, 1, 40, 8, 128
    Hl, S = H // P, P * Sl
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=3)
    g = synth.move(d, "cuda")
    outs = {k: _targets(P, B, S, Hl, D, dtype) for k in "qkv"}
    tf.scatter_qkv_heads_into(g["q"], g["k"], g["v"], outs["q"], outs["k"], outs["v"], h0=1, h1=3)
    for key in "qkv":
        before = [torch.full((B, S, Hl, D), SENTINEL, dtype=dtype) for _ in range(P)]
        want = oracle.scatter_heads_chunk(d[key], P, 1, 3, before)
        for i in range(P):
            assert bits_equal(outs[key][i].cpu(), want[i]), (key, i)


@pytest.mark.parametrize("rope", ["interleaved", "neox"])
def test_fused_head_chunks(tf, rope):
    P, B, Sl, H, D = 4, 1, 50, 16, 128
    Hl, S = H // P, P * Sl
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=9, layout="v_strided")
    wq, wk = synth.norm_weights(D, dtype, seed=9)
    g = synth.move(d, "cuda")
    outs = {k: _targets(P, B, S, Hl, D, dtype) for k in "qkv"}
    for h0, h1 in ((0, 3), (3, Hl)):
        tf.scatter_qkv_heads_into(g["q"], g["k"], g["v"], outs["q"], outs["k"], outs["v"], h0=h0, h1=h1,
                                  norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA,
                                  rope=rope)
    table = oracle.rope_table(THETA, S, D)
    for key, w in (("q", wq), ("k", wk)):
        want = oracle.scatter_norm_rope(d[key], P, w, EPS, table, style=rope)
        for i in range(P):
            assert_fused_ok(outs[key][i], want[i])
    want_v = oracle.scatter(d["v"], P)
    for i in range(P):
        assert bits_equal(outs["v"][i].cpu(), want_v[i])


@pytest.mark.parametrize("rope", ["interleaved", "neox"])
def test_fused_head_chunks_qk_only(tf, rope):
    """Q and K alone (V moved by another path) in head chunks: the Q/K-only launch
    (its (cos, sin) ring and paired rows) reading head bands Hg heads apart."""
    P, B, Sl, H, D = 4, 2, 70, 24, 128
    Hl, S = H // P, P * Sl
    dtype = torch.float16 if rope == "neox" else torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=19, layout="v_strided", with_v=False)
    wq, wk = synth.norm_weights(D, dtype, seed=19)
    g = synth.move(d, "cuda")
    outs = {k: _targets(P, B, S, Hl, D, dtype) for k in "qk"}
    for h0, h1 in ((0, 2), (2, 5), (5, Hl)):
        tf.scatter_qkv_heads_into(g["q"], g["k"], None, outs["q"], outs["k"], None, h0=h0, h1=h1,
                                  norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA,
                                  rope=rope)
    table = oracle.rope_table(THETA, S, D)
    for key, w in (("q", wq), ("k", wk)):
        want = oracle.scatter_norm_rope(d[key], P, w, EPS, table, style=rope)
        for i in range(P):
            assert_fused_ok(outs[key][i], want[i])


def test_head_chunks_into_fused_layout(tf):
    P, B, Sl, H, D = 2, 2, 21, 8, 64
    Hl, S = H // P, P * Sl
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=12, layout="fused")
    g = synth.move(d, "cuda")
    pay = _targets(P, B, S, Hl, D, dtype, width=3)
    for h0, h1 in ((0, 2), (2, Hl)):
        tf.scatter_qkv_heads_into(g["q"], g["k"], g["v"], pay, h0=h0, h1=h1, layout="fused")
    want = oracle.fused_payload(*[oracle.scatter(d[k], P) for k in "qkv"])
    for i in range(P):
        assert bits_equal(pay[i].cpu(), want[i])


def test_video_dit_head_chunks_equal_whole_launch(tf):
    """Full video-DiT size, fused mode: two head chunks into caller targets give
    the same bits as the whole cached scatter (itself checked against the oracle
    in test_gpu_parity), and sampled rows match the oracle."""
    P, B, S, H, D = 4, 1, 32760, 40, 128
    Sl, Hl = S // P, H // P
    dtype = torch.bfloat16
    wq, wk = synth.norm_weights(D, dtype, seed=21, device="cuda")
    g = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=21, layout="v_strided", device="cuda")
    kw = dict(norm_rope=True, q_weight=wq, k_weight=wk, eps=EPS, theta=THETA)
    tq, tk, tv, _ = tf.scatter_qkv("vd_whole", g["q"], g["k"], g["v"], **kw)
    outs = {k: [torch.empty((B, S, Hl, D), dtype=dtype, device="cuda") for _ in range(P)] for k in "qkv"}
    for h0, h1 in ((0, 5), (5, Hl)):
        tf.scatter_qkv_heads_into(g["q"], g["k"], g["v"], outs["q"], outs["k"], outs["v"], h0=h0, h1=h1, **kw)
    for key, whole in (("q", tq), ("k", tk), ("v", tv)):
        for i in range(P):
            assert bits_equal(outs[key][i], whole[i]), (key, i)
    table = oracle.rope_table(THETA, S, D)
    gen = torch.Generator().manual_seed(22)
    got, want = [], []
    for _ in range(100):
        gi, p, h = (int(torch.randint(n, (1,), generator=gen)) for n in (P, S, Hl))
        r, t = divmod(p, Sl)
        want.append(oracle.rmsnorm_rope_row(g["q"][r][0, t, gi * Hl + h].cpu(), wq.cpu(), EPS, table[p]))
        got.append(outs["q"][gi][0, p, h].cpu())
    assert_fused_ok(torch.stack(got), torch.stack(want))


# ------------------------------------------------------------------ chunk exchange
@pytest.mark.parametrize("P", [1, 2, 3, 8])
@pytest.mark.parametrize("chunk", [16, 48, 4096, 100000, 65552])
def test_exchange_chunks_vs_oracle(tf, P, chunk):
    gen = torch.Generator().manual_seed(P * 1000 + chunk)
    src = [torch.randint(0, 256, (P, chunk), generator=gen, dtype=torch.uint8) for _ in range(P)]
    dst = tf.exchange_chunks([s.cuda() for s in src])
    want = oracle.exchange_chunks(src, P)
    for g in range(P):
        assert bits_equal(dst[g].cpu(), want[g]), g


def test_exchange_chunks_large_and_typed(tf):
    """P=8 payloads of 8 x 8 MiB (bf16 elements): against the same exchange
    written as tensor indexing on the GPU."""
    P, chunk_elems = 8, 4 << 20
    gen = torch.Generator(device="cuda").manual_seed(5)
    src = [torch.randn((P, chunk_elems), generator=gen, device="cuda").to(torch.bfloat16) for _ in range(P)]
    dst = tf.exchange_chunks(src)
    for g in range(P):
        want = torch.stack([src[r][g] for r in range(P)])
        assert bits_equal(dst[g], want), g


def test_device_status_clean(tf):
    torch.cuda.synchronize()
    assert tf.device_status(clear=False) == 0
