"""Whole outputs at full size against the oracle, element by element.

The benchmark's workload -- the video-DiT shape (P=4, S=32760 = 21x30x52, H=40,
D=128, bf16, V a strided view of a fused projection), fused RMSNorm + RoPE on
Q/K into the cached targets, then the output gather -- in the launch
configuration the benchmark times (one V+Q+K launch of the block kernel walking
its units one at a time), and one point of the fused portfolio per head size
(P=8, S=32760, H=48, bf16) are compared with the oracle on every element: Q/K
under the fused rule (parity_util.assert_fused_ok), V and the gather bit for
bit.  The projection at the video-DiT shape is compared on two whole row tiles
over every feature (all column tiles, Q/K/V), one of them the ragged last tile
of 126 rows, on dyadic inputs, where the sums are exact in any order.

The oracle runs on threads (its C code releases the interpreter lock and keeps
no global state): each (head group g, shard r) block of the fused scatter is one
oracle call with P = 1 on shard r's head band g and the table from position
r*S_local on, which are the same rows the P-shard call computes (the scatter
moves each row as a whole; the fused row depends only on the row and its
position).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import pytest
import torch

import oracle
from parity_util import assert_fused_ok, bits_equal
from ulysses_sequence_attention_tf_gb300 import synth

pytestmark = pytest.mark.gpu

EPS = 1e-6
THETA = 10000.0


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


@pytest.fixture(scope="module")
def pool():
    with ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        yield ex


def fused_oracle(pool, srcs, P, w, table, style="interleaved"):
    """oracle.scatter_norm_rope of P shards, block by block on the pool's threads."""
    B, Sl, H, D = srcs[0].shape
    Hl = H // P
    out = [torch.empty((B, P * Sl, Hl, D), dtype=srcs[0].dtype) for _ in range(P)]

    def block(g, r):
        band = srcs[r][:, :, g * Hl:(g + 1) * Hl]
        res = oracle.scatter_norm_rope([band], 1, w, EPS, table[r * Sl:(r + 1) * Sl], style=style)[0]
        out[g][:, r * Sl:(r + 1) * Sl] = res

    list(pool.map(lambda gr: block(*gr), [(g, r) for g in range(P) for r in range(P)]))
    return out


def _check_fused(got, want):
    flips = 0
    for g in range(len(want)):
        st = assert_fused_ok(got[g], want[g])
        flips += st["n_bit_diff"]
    return flips


def test_video_dit_whole_step_vs_oracle(tf, pool):
    P, B, S, H, D = 4, 1, 32760, 40, 128
    Sl, Hl = S // P, H // P
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=71, layout="v_strided")
    attn = synth.attn_outputs(P, B, S, Hl, D, dtype, seed=71)
    wq, wk = synth.norm_weights(D, dtype, seed=71)
    g = synth.move(d, "cuda")
    assert g["v"][0].stride() == (Sl * 3 * H * D, 3 * H * D, D, 1)
    tq, tk, tv, _ = tf.scatter_qkv("full_size_video_dit", g["q"], g["k"], g["v"], norm_rope=True,
                                   q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA)
    back, _ = tf.gather_out("full_size_video_dit_out", [a.cuda() for a in attn])
    torch.cuda.synchronize()
    got = {"q": [t.cpu() for t in tq], "k": [t.cpu() for t in tk], "v": [t.cpu() for t in tv],
           "o": [t.cpu() for t in back]}
    del g, tq, tk, tv, back
    table = oracle.rope_table(THETA, S, D)
    flips = _check_fused(got["q"], fused_oracle(pool, d["q"], P, wq, table))
    flips += _check_fused(got["k"], fused_oracle(pool, d["k"], P, wk, table))
    want_v = oracle.scatter(d["v"], P)
    for i in range(P):
        assert bits_equal(got["v"][i], want_v[i]), i
    want_o = oracle.gather(attn, P)
    for r in range(P):
        assert bits_equal(got["o"][r], want_o[r]), r
    print(f"video DiT whole step: {2 * P * B * S * Hl * D} fused elements, {flips} one-ulp flips")
    assert tf.device_status(clear=False) == 0


def test_back_to_back_launches_keep_stream_order(tf):
    """Relayout kernels are launched to overlap the kernel before them in the
    stream, and wait for it before touching memory.  A chain where each launch
    reads what the previous one wrote -- V scattered at full size, the targets
    gathered straight back, the result scattered again, all enqueued without a
    synchronisation -- must give back V and its scatter bit for bit."""
    P, B, S, H, D = 4, 1, 32760, 40, 128
    Sl = S // P
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=74, layout="v_strided", device="cuda")
    v = d["v"]
    for _ in range(3):
        tv, _, _, _ = tf.scatter_qkv("b2b_scatter", v)
        back, _ = tf.gather_out("b2b_gather", tv)
        tv2, _, _, _ = tf.scatter_qkv("b2b_rescatter", back)
        torch.cuda.synchronize()
        for r in range(P):
            assert bits_equal(back[r], v[r].contiguous()), r
        for g in range(P):
            assert bits_equal(tv2[g], tv[g]), g


@pytest.mark.parametrize("rope", ["interleaved", "neox"])
def test_video_dit_qk_only_whole_output_vs_oracle(tf, pool, rope):
    """The Q/K-only launch (V moved by another path) at the video-DiT shape, both
    RoPE styles: the (cos, sin) ring and the paired Q/K rows over ~26 rounds of
    units, every element against the oracle."""
    P, B, S, H, D = 4, 1, 32760, 40, 128
    Sl, Hl = S // P, H // P
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=91, layout="v_strided", with_v=False)
    wq, wk = synth.norm_weights(D, dtype, seed=91)
    g = synth.move(d, "cuda")
    outs = [[torch.empty((B, S, Hl, D), dtype=dtype, device="cuda") for _ in range(P)] for _ in "qk"]
    tf.scatter_qkv_into(g["q"], g["k"], None, outs[0], outs[1], None, norm_rope=True, q_weight=wq.cuda(),
                        k_weight=wk.cuda(), eps=EPS, theta=THETA, rope=rope)
    torch.cuda.synchronize()
    got = [[t.cpu() for t in o] for o in outs]
    del g, outs
    table = oracle.rope_table(THETA, S, D)
    flips = _check_fused(got[0], fused_oracle(pool, d["q"], P, wq, table, style=rope))
    flips += _check_fused(got[1], fused_oracle(pool, d["k"], P, wk, table, style=rope))
    assert flips <= 8, flips


@pytest.mark.parametrize("D", [64, 128])
def test_fused_portfolio_p8_whole_output_vs_oracle(tf, pool, D):
    P, B, S, H = 8, 1, 32760, 48
    Sl, Hl = S // P, H // P
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=72 + D, layout="v_strided")
    wq, wk = synth.norm_weights(D, dtype, seed=72 + D)
    g = synth.move(d, "cuda")
    outs = [[torch.empty((B, S, Hl, D), dtype=dtype, device="cuda") for _ in range(P)] for _ in "qkv"]
    tf.scatter_qkv_into(g["q"], g["k"], g["v"], *outs, norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(),
                        eps=EPS, theta=THETA)
    torch.cuda.synchronize()
    got = [[t.cpu() for t in o] for o in outs]
    del g, outs
    table = oracle.rope_table(THETA, S, D)
    _check_fused(got[0], fused_oracle(pool, d["q"], P, wq, table))
    _check_fused(got[1], fused_oracle(pool, d["k"], P, wk, table))
    want_v = oracle.scatter(d["v"], P)
    for i in range(P):
        assert bits_equal(got[2][i], want_v[i]), i


def test_projection_video_dit_whole_row_tiles_vs_oracle(tf, pool):
    """Two whole row tiles over every feature (all heads of Q, K and V): shard 0's
    first tile (128 rows) and the last shard's ragged last tile (126 rows), on
    dyadic inputs -- bit-exact up to the fused rule's isolated flips."""
    P, B, Sl, H, D = 4, 1, 8190, 40, 128
    hidden, S, Hl, HD = H * D, P * Sl, H // P, H * D
    dtype = torch.bfloat16
    assert Sl % 128 == 126  # the last row tile of every shard is ragged
    xs, w = synth.projection_inputs(P, B, Sl, hidden, H, D, dtype, seed=73, dist="dyadic")
    wq, wk = synth.norm_weights(D, dtype, seed=73)
    outs = {k: [torch.empty((B, S, Hl, D), dtype=dtype, device="cuda") for _ in range(P)] for k in "qkv"}
    tf.project_qkv_into([x.cuda() for x in xs], w.cuda(), H, outs["q"], outs["k"], outs["v"], norm_rope=True,
                        q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA)
    torch.cuda.synchronize()
    table = oracle.rope_table(THETA, S, D)
    chunk = 960  # features per oracle call (16 calls per tile)
    for r, t0, t1 in ((0, 0, 128), (P - 1, Sl - 126, Sl)):
        n = t1 - t0
        x_rows = xs[r][0, t0:t1].contiguous()
        proj = torch.empty((n, 3 * HD), dtype=dtype)

        def project(c):
            proj[:, c:c + chunk] = oracle.project(x_rows, w[c:c + chunk].contiguous())

        list(pool.map(project, range(0, 3 * HD, chunk)))
        proj = proj.view(1, n, 3, H, D)
        pos = r * Sl + t0
        for sec, key, wn in ((0, "q", wq), (1, "k", wk), (2, "v", None)):
            rows = proj[:, :, sec].contiguous()
            if wn is not None:
                want = oracle.scatter_norm_rope([rows], 1, wn, EPS, table[pos:pos + n])[0]
            else:
                want = rows
            got = torch.cat([outs[key][g][:, pos:pos + n].cpu() for g in range(P)], dim=2)
            if wn is not None:
                assert_fused_ok(got, want)
            else:
                assert bits_equal(got, want), (r, key)
    assert tf.device_status(clear=False) == 0
