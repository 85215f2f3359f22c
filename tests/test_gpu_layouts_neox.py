"""Parity of the fused receive layout and of half-split (NeoX) RoPE with the CPU
oracle, through the C ABI.

Fused receive layout (flashinfer PR #6332 commit message, "Description",
"Layouts"): one [B, S, Hl, 3*D] payload per head group whose head row is the
Q row, the K row, then the V row.  Half-split RoPE pairs element i with
i + D/2 (the GPT-NeoX pairing; the pages name only the interleaved form).
Relayout is bit-exact; the fused rows use the tolerance of parity_util.
"""
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


def _oracle_targets(d, P, norm_rope, wq, wk, table, style):
    out = {}
    for key in ("q", "k", "v"):
        if d[key] is None:
            out[key] = None
        elif norm_rope and key != "v":
            out[key] = oracle.scatter_norm_rope(d[key], P, wq if key == "q" else wk, EPS, table, style=style)
        else:
            out[key] = oracle.scatter(d[key], P)
    return out


# ------------------------------------------------------------------ half-split RoPE, separate targets
@pytest.mark.parametrize("with_k,with_v", [(True, True), (False, True), (True, False)])
@pytest.mark.parametrize("D", [32, 64, 128, 256])
def test_neox_slot_patterns_and_head_dims(tf, with_k, with_v, D):
    P, B, Sl, H = 2, 2, 29, 6
    dtype = torch.bfloat16 if D in (32, 128) else torch.float16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=60 + D, layout="fused", with_k=with_k, with_v=with_v)
    wq, wk = synth.norm_weights(D, dtype, seed=60 + D)
    g = synth.move(d, "cuda")
    tq, tk, tv, _ = tf.scatter_qkv(f"neox{D}{with_k}{with_v}", g["q"], g["k"], g["v"], norm_rope=True,
                                   q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA, rope="neox")
    want = _oracle_targets(d, P, True, wq, wk, oracle.rope_table(THETA, P * Sl, D), "neox")
    for key, tg in (("q", tq), ("k", tk), ("v", tv)):
        if want[key] is None:
            assert tg is None
            continue
        for i in range(P):
            if key == "v":
                assert bits_equal(tg[i].cpu(), want[key][i])
            else:
                assert_fused_ok(tg[i], want[key][i])


def test_neox_differs_from_interleaved(tf):
    """The two pairings give different rows (so the flag reaches the kernel)."""
    P, B, Sl, H, D = 2, 1, 16, 4, 128
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=5, device="cuda")
    wq, wk = synth.norm_weights(D, dtype, seed=5, device="cuda")
    a, _, _, _ = tf.scatter_qkv("style_i", d["q"], norm_rope=True, q_weight=wq, k_weight=wk)
    b, _, _, _ = tf.scatter_qkv("style_n", d["q"], norm_rope=True, q_weight=wq, k_weight=wk, rope="neox")
    # position 0 has no rotation: identical there, different elsewhere
    assert bits_equal(a[0][:, :1], b[0][:, :1])
    assert not bits_equal(a[0][:, 1:], b[0][:, 1:])


def test_neox_16_byte_vectors_and_caller_table(tf):
    """Sources only 16-byte aligned take the register kernel; a caller table."""
    P, B, Sl, H, D = 2, 1, 40, 4, 64
    dtype = torch.float16
    gen = torch.Generator().manual_seed(91)
    HD = H * D
    bufs = [torch.randn(B, Sl, 3 * HD + 8, generator=gen).to(dtype) for _ in range(P)]
    views = lambda bs, o: [b[..., 8 + o * HD:8 + (o + 1) * HD].unflatten(-1, (H, D)) for b in bs]
    gb = [b.cuda() for b in bufs]
    wq, wk = synth.norm_weights(D, dtype, seed=91)
    table = oracle.rope_table(500.0, P * Sl, D)
    assert views(gb, 0)[0].data_ptr() % 32 == 16
    tq, tk, tv, _ = tf.scatter_qkv("neox16", views(gb, 0), views(gb, 1), views(gb, 2), norm_rope=True,
                                   q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, cos_sin=table.cuda(),
                                   rope="neox")
    for o, tg, w in ((0, tq, wq), (1, tk, wk)):
        want = oracle.scatter_norm_rope(views(bufs, o), P, w, EPS, table, style="neox")
        for i in range(P):
            assert_fused_ok(tg[i], want[i])
    want_v = oracle.scatter(views(bufs, 2), P)
    for i in range(P):
        assert bits_equal(tv[i].cpu(), want_v[i])


# ------------------------------------------------------------------ fused receive layout
@pytest.mark.parametrize("norm_rope,style", [(False, "interleaved"), (True, "interleaved"), (True, "neox")])
@pytest.mark.parametrize("D", [64, 128])
def test_fused_layout_cached(tf, norm_rope, style, D):
    P, B, Sl, H = 4, 2, 37, 8
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=70 + D, layout="fused")
    wq, wk = synth.norm_weights(D, dtype, seed=70 + D)
    g = synth.move(d, "cuda")
    kw = dict(norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA, rope=style) \
        if norm_rope else {}
    tq, tk, tv, _ = tf.scatter_qkv(f"fl{D}{norm_rope}{style}", g["q"], g["k"], g["v"], layout="fused", **kw)
    pay = tf.fused_payloads(tq)
    want = _oracle_targets(d, P, norm_rope, wq, wk, oracle.rope_table(THETA, P * Sl, D), style)
    want_pay = oracle.fused_payload(want["q"], want["k"], want["v"])
    for i in range(P):
        assert pay[i].shape == (B, P * Sl, H // P, 3 * D) and pay[i].is_contiguous()
        assert tk[i].data_ptr() == pay[i].data_ptr() + D * 2 and tv[i].data_ptr() == pay[i].data_ptr() + 4 * D
        if norm_rope:
            assert bits_equal(tv[i].cpu(), want["v"][i])
            assert_fused_ok(tq[i].contiguous(), want["q"][i])
            assert_fused_ok(tk[i].contiguous(), want["k"][i])
        else:
            assert bits_equal(pay[i].cpu(), want_pay[i])


def test_fused_layout_into_noalloc_and_key(tf):
    P, B, Sl, H, D = 2, 1, 50, 4, 128
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=81, layout="v_strided")
    wq, wk = synth.norm_weights(D, dtype, seed=81)
    g = synth.move(d, "cuda")
    want = _oracle_targets(d, P, True, wq, wk, oracle.rope_table(THETA, P * Sl, D), "interleaved")
    guard = 64
    for fn in (tf.scatter_qkv_into, tf.scatter_qkv_noalloc):
        slab = [torch.full((B * P * Sl * (H // P) * 3 * D + 2 * guard,), -7.0, dtype=dtype, device="cuda")
                for _ in range(P)]
        pay = [s[guard:-guard].view(B, P * Sl, H // P, 3 * D) for s in slab]
        fn(g["q"], g["k"], g["v"], pay, norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS,
           theta=THETA, layout="fused")
        for i in range(P):
            assert torch.all(slab[i][:guard] == -7.0) and torch.all(slab[i][-guard:] == -7.0)
            assert_fused_ok(pay[i][..., :D].contiguous(), want["q"][i])
            assert_fused_ok(pay[i][..., D:2 * D].contiguous(), want["k"][i])
            assert bits_equal(pay[i][..., 2 * D:].cpu(), want["v"][i])
        with pytest.raises(tf.TfUlyssesError):  # the payloads go in q_out only
            fn(g["q"], g["k"], g["v"], pay, pay, layout="fused")
    with pytest.raises(tf.TfUlyssesError):  # the fused layout needs all of q, k, v
        tf.scatter_qkv("fl_missing", g["q"], g["k"], None, layout="fused")
    torch.cuda.synchronize()
    tf.cache_clear()
    a, _, _, _ = tf.scatter_qkv("fl_key", g["q"], g["k"], g["v"])
    b, _, _, _ = tf.scatter_qkv("fl_key", g["q"], g["k"], g["v"], layout="fused")
    assert tf.cache_entries() == 2  # the layout is part of the key
    assert a[0].data_ptr() != b[0].data_ptr()


@pytest.mark.parametrize("dtype,D", [(torch.float32, 36), (torch.float16, 8), (torch.uint8, 48)])
def test_fused_layout_plain_odd_rows(tf, dtype, D):
    """Rows that are not 64..512 bytes (staged kernel with per-row stores) or only
    16-byte multiples: still bit-exact."""
    P, B, Sl, H = 3, 2, 11, 6
    if dtype == torch.uint8:
        gen = torch.Generator().manual_seed(D)
        src = {k: [torch.randint(0, 256, (B, Sl, H, D), generator=gen, dtype=torch.uint8) for _ in range(P)]
               for k in ("q", "k", "v")}
    else:
        d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=D)
        src = {k: d[k] for k in ("q", "k", "v")}
    tq, tk, tv, _ = tf.scatter_qkv(f"flodd{D}", *[[t.cuda() for t in src[k]] for k in ("q", "k", "v")],
                                   layout="fused")
    want = oracle.fused_payload(*[oracle.scatter(src[k], P) for k in ("q", "k", "v")])
    pay = tf.fused_payloads(tq)
    for i in range(P):
        assert bits_equal(pay[i].cpu(), want[i])


def test_video_dit_fused_layout_neox_sampled(tf):
    """Full video-DiT size (P=4, S=32760, H=40, D=128, bf16, V strided) into the
    fused layout with half-split RoPE: V whole against the all-gather
    formulation, Q/K on sampled rows against the oracle row by row."""
    P, B, S, H, D = 4, 1, 32760, 40, 128
    Sl, Hl = S // P, H // P
    dtype = torch.bfloat16
    wq, wk = synth.norm_weights(D, dtype, seed=11)
    g = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=11, layout="v_strided", device="cuda")
    tq, tk, tv, _ = tf.scatter_qkv("vd_fl_neox", g["q"], g["k"], g["v"], norm_rope=True, q_weight=wq.cuda(),
                                   k_weight=wk.cuda(), eps=EPS, theta=THETA, rope="neox", layout="fused")
    full_v = torch.cat([x.contiguous() for x in g["v"]], dim=1)
    for i in range(P):
        assert bits_equal(tv[i], full_v[:, :, i * Hl:(i + 1) * Hl])
    table = oracle.rope_table(THETA, S, D)
    gen = torch.Generator().manual_seed(12)
    for key, tg, w in (("q", tq, wq), ("k", tk, wk)):
        got, want = [], []
        for _ in range(200):
            gi, p, h = (int(torch.randint(n, (1,), generator=gen)) for n in (P, S, Hl))
            r, t = divmod(p, Sl)
            want.append(oracle.rmsnorm_rope_row(g[key][r][0, t, gi * Hl + h].cpu(), w, EPS, table[p], style="neox"))
            got.append(tg[gi][0, p, h].cpu())
        assert_fused_ok(torch.stack(got), torch.stack(want))


def test_device_status_clean(tf):
    torch.cuda.synchronize()
    assert tf.device_status(clear=False) == 0
