"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Pure relayout must be bit-exact; the fused Q/K RMSNorm + RoPE must be within
max-abs 1e-2 (bf16) / 2e-3 (fp16), any element above that differing by exactly
one ulp, and is expected to be bit-exact apart from isolated flips.

Workloads (seeded, synthetic): the P=2 fp16 round trip, the P=4 S=4096 H=24
fused-projection case with norm+RoPE, the P=4 S=32760 H=40 video-DiT case with
a strided V over repeated steps into cached targets, the P in {2,4,6,8}
portfolio with S=6001 padded to a multiple of P, and the bf16 bandwidth sweep
up to 2 GiB per direction.  At full size the oracle checks sampled rows one by
one and the whole output is checked against the all-gather formulation
(concatenate shards in rank order, slice head bands) on the GPU.
"""
import pytest
import torch

import oracle
from parity_util import assert_fused_ok, bits_equal, ulp_diff
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


def cuda(ts):
    return None if ts is None else [t.cuda() for t in ts]


def cpu(ts):
    return None if ts is None else [t.cpu() for t in ts]


def to_device_like(d):
    return synth.move(d, "cuda")


def allgather_scatter(srcs, P):
    full = torch.cat([s.contiguous() for s in srcs], dim=1)
    Hl = full.shape[2] // P
    return [full[:, :, g * Hl:(g + 1) * Hl].contiguous() for g in range(P)]


def allgather_gather(attn, P):
    full = torch.cat([a.contiguous() for a in attn], dim=2)
    Sl = full.shape[1] // P
    return [full[:, r * Sl:(r + 1) * Sl].contiguous() for r in range(P)]


# ------------------------------------------------------------------ config: P=2 fp16 round trip
def test_tiny_p2_scatter_then_gather_bit_exact(tf):
    P, B, S, H, D = 2, 1, 256, 8, 64
    d = synth.qkv_shards(P, B, S // P, H, D, torch.float16, seed=0)
    g = to_device_like(d)
    tq, tk, tv, _ = tf.scatter_qkv("tiny_p2", g["q"], g["k"], g["v"])
    for key, tg in (("q", tq), ("k", tk), ("v", tv)):
        want = oracle.scatter(d[key], P)
        for i in range(P):
            assert bits_equal(tg[i].cpu(), want[i]), (key, i)
        back, _ = tf.gather_out("tiny_p2_" + key, tg)
        want_back = oracle.gather(want, P)
        for r in range(P):
            assert bits_equal(back[r].cpu(), want_back[r]), (key, r)
            assert bits_equal(back[r].cpu(), d[key][r]), (key, r)


# ------------------------------------------------------------------ fused: FLUX-like P=4 S=4096 H=24
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_flux_fused_projection_norm_rope(tf, dtype):
    P, B, S, H, D = 4, 1, 4096, 24, 128
    d = synth.qkv_shards(P, B, S // P, H, D, dtype, seed=1, layout="fused")
    wq, wk = synth.norm_weights(D, dtype, seed=1)
    g = to_device_like(d)
    assert g["v"][0].stride() == (S // P * 3 * H * D, 3 * H * D, D, 1)
    tq, tk, tv, _ = tf.scatter_qkv("flux", g["q"], g["k"], g["v"], norm_rope=True,
                                   q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA)
    table = oracle.rope_table(THETA, S, D)
    for key, tg, w in (("q", tq, wq), ("k", tk, wk)):
        want = oracle.scatter_norm_rope(d[key], P, w, EPS, table)
        for i in range(P):
            assert_fused_ok(tg[i], want[i])
    want_v = oracle.scatter(d["v"], P)
    for i in range(P):
        assert bits_equal(tv[i].cpu(), want_v[i])


# Q/K only (V moved by another path): P=4, S=8192, H=24 -- 1024 units of 192 rows,
# about 3.4 per CTA, so every CTA streams its loads (and its lanes' (cos, sin)
# ring) from one unit into the next; six rows per lane group and unit cross
# token boundaries (Hl = 6).
@pytest.mark.parametrize("dtype,rope", [(torch.bfloat16, "interleaved"), (torch.float16, "interleaved"),
                                        (torch.bfloat16, "neox"), (torch.float16, "neox")])
def test_qk_only_several_units_per_cta(tf, dtype, rope):
    P, B, S, H, D = 4, 1, 8192, 24, 128
    d = synth.qkv_shards(P, B, S // P, H, D, dtype, seed=5, layout="fused", with_v=False)
    wq, wk = synth.norm_weights(D, dtype, seed=5)
    g = to_device_like(d)
    tq, tk, tv, _ = tf.scatter_qkv(f"qk_units_{rope}", g["q"], g["k"], None, norm_rope=True, q_weight=wq.cuda(),
                                   k_weight=wk.cuda(), eps=EPS, theta=THETA, rope=rope)
    assert tv is None
    table = oracle.rope_table(THETA, S, D)
    for key, tg, w in (("q", tq, wq), ("k", tk, wk)):
        want = oracle.scatter_norm_rope(d[key], P, w, EPS, table, style=rope)
        for i in range(P):
            assert_fused_ok(tg[i], want[i])


def test_rope_table_matches_oracle(tf):
    for S, D in ((4096, 128), (777, 64), (32760, 128)):
        lib_tab = tf.rope_table(THETA, S, D).cpu()
        ora = oracle.rope_table(THETA, S, D)
        diff = (lib_tab.view(torch.int32) - ora.view(torch.int32)).abs()
        # cos/sin in double on both sides, then one fp32 rounding: equal unless the
        # double results straddle an fp32 rounding point
        assert int(diff.max()) <= 1, (S, D)
        assert int((diff > 0).sum()) <= max(4, ora.numel() // 100000), (S, D, int((diff > 0).sum()))


def test_caller_table_gives_same_result(tf):
    P, B, S, H, D = 2, 2, 96, 8, 64
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, S // P, H, D, dtype, seed=5, layout="fused")
    wq, wk = synth.norm_weights(D, dtype, seed=5)
    g = to_device_like(d)
    table = oracle.rope_table(THETA, S, D)
    tq, tk, _, _ = tf.scatter_qkv("own_table", g["q"], g["k"], None, norm_rope=True, q_weight=wq.cuda(),
                                  k_weight=wk.cuda(), eps=EPS, cos_sin=table.cuda())
    for key, tg, w in (("q", tq, wq), ("k", tk, wk)):
        want = oracle.scatter_norm_rope(d[key], P, w, EPS, table)
        for i in range(P):
            assert_fused_ok(tg[i], want[i])


# ------------------------------------------------------------------ video-DiT P=4 S=32760 H=40, cached steps
def _sample_rows(P, B, Sl, Hl, n, seed):
    gen = torch.Generator().manual_seed(seed)
    S = P * Sl
    rows = [(0, 0, 0, 0), (P - 1, B - 1, S - 1, Hl - 1), (P - 1, 0, Sl, 0), (0, B - 1, Sl - 1, Hl - 1)]
    for _ in range(n):
        rows.append((int(torch.randint(P, (1,), generator=gen)), int(torch.randint(B, (1,), generator=gen)),
                     int(torch.randint(S, (1,), generator=gen)), int(torch.randint(Hl, (1,), generator=gen))))
    return rows


def test_video_dit_steps_cached_targets(tf):
    P, B, S, H, D = 4, 1, 32760, 40, 128
    Sl, Hl = S // P, H // P
    dtype = torch.bfloat16
    wq, wk = synth.norm_weights(D, dtype, seed=0)
    wq_g, wk_g = wq.cuda(), wk.cuda()
    table = oracle.rope_table(THETA, S, D)
    ptrs = None
    for step in range(3):
        g = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=step, layout="v_strided", device="cuda")
        tq, tk, tv, _ = tf.scatter_qkv("video_dit", g["q"], g["k"], g["v"], norm_rope=True,
                                       q_weight=wq_g, k_weight=wk_g, eps=EPS, theta=THETA)
        now = [t.data_ptr() for t in tq + tk + tv]
        if ptrs is not None:
            assert now == ptrs, "cache hit must reuse the same targets"
        ptrs = now
        # V: the whole output against the all-gather formulation
        for i, want in enumerate(allgather_scatter(g["v"], P)):
            assert bits_equal(tv[i], want)
        # Q/K: sampled rows against the oracle, one row at a time
        for key, tg, w in (("q", tq, wq), ("k", tk, wk)):
            got_rows, want_rows = [], []
            for (gi, b, p, h) in _sample_rows(P, B, Sl, Hl, 300, seed=step):
                r, t = divmod(p, Sl)
                src_row = g[key][r][b, t, gi * Hl + h].cpu()
                want_rows.append(oracle.rmsnorm_rope_row(src_row, w, EPS, table[p]))
                got_rows.append(tg[gi][b, p, h].cpu())
            assert_fused_ok(torch.stack(got_rows), torch.stack(want_rows))
    # output gather of a synthetic attention output, whole output vs the all-gather formulation
    attn = synth.attn_outputs(P, B, S, Hl, D, dtype, seed=3, device="cuda")
    outs, _ = tf.gather_out("video_dit_out", attn)
    for r, want in enumerate(allgather_gather(attn, P)):
        assert bits_equal(outs[r], want)
    # and sampled tokens against the oracle on the CPU (all heads of the token)
    for t in (0, 1, Sl // 2, Sl - 1):
        sub = [a[:, [r * Sl + t for r in range(P)]].cpu() for a in attn]  # token t of every shard
        want = oracle.gather(sub, P)
        for r in range(P):
            assert bits_equal(outs[r][:, t:t + 1].cpu(), want[r])


# ------------------------------------------------------------------ portfolio P in {2,4,6,8}, S=6001 padded
@pytest.mark.parametrize("P", [2, 4, 6, 8])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
def test_portfolio_full_size(tf, P, dtype, D):
    B, H, S0 = 2, 48, 6001
    S = synth.padded_seq(S0, P)
    Sl = S // P
    g = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=P * 10 + D, device="cuda", pad_from=S0)
    tq, tk, tv, _ = tf.scatter_qkv(f"pf{P}", g["q"], g["k"], g["v"])
    for key, tg in (("q", tq), ("k", tk), ("v", tv)):
        for i, want in enumerate(allgather_scatter(g[key], P)):
            assert bits_equal(tg[i], want), (key, i)
    back, _ = tf.gather_out(f"pf{P}", tq)
    full_in = torch.cat(g["q"], dim=1)[:, :S0]
    full_out = torch.cat(back, dim=1)[:, :S0]  # trim the padding after the gather
    assert bits_equal(full_out, full_in)


@pytest.mark.parametrize("P", [2, 4, 6, 8])
def test_portfolio_small_vs_oracle(tf, P):
    B, H, S0, D = 2, 48, 601, 64
    for dtype in (torch.float16, torch.bfloat16):
        S = synth.padded_seq(S0, P)
        d = synth.qkv_shards(P, B, S // P, H, D, dtype, seed=P, pad_from=S0)
        g = to_device_like(d)
        tq, tk, tv, _ = tf.scatter_qkv("pf_small", g["q"], g["k"], g["v"])
        for key, tg in (("q", tq), ("k", tk), ("v", tv)):
            want = oracle.scatter(d[key], P)
            for i in range(P):
                assert bits_equal(tg[i].cpu(), want[i]), (P, dtype, key, i)
        attn = synth.attn_outputs(P, B, S, H // P, D, dtype, seed=P)
        outs, _ = tf.gather_out("pf_small", cuda(attn))
        want = oracle.gather(attn, P)
        for r in range(P):
            assert bits_equal(outs[r].cpu(), want[r]), (P, dtype, r)


@pytest.mark.parametrize("P", [2, 4, 6, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_portfolio_fused_vs_oracle(tf, P, D):
    """The portfolio shapes through the fused scatter (RMSNorm + RoPE on Q/K,
    V copied), fp16 and bf16, S=601 padded to a multiple of P, B=2."""
    B, H, S0 = 2, 48, 601
    for dtype in (torch.float16, torch.bfloat16):
        S = synth.padded_seq(S0, P)
        d = synth.qkv_shards(P, B, S // P, H, D, dtype, seed=100 + P * D, layout="fused", pad_from=S0)
        wq, wk = synth.norm_weights(D, dtype, seed=P)
        g = to_device_like(d)
        tq, tk, tv, _ = tf.scatter_qkv(f"pf_fused{D}", g["q"], g["k"], g["v"], norm_rope=True, q_weight=wq.cuda(),
                                       k_weight=wk.cuda(), eps=EPS, theta=THETA)
        table = oracle.rope_table(THETA, S, D)
        for key, tg, w in (("q", tq, wq), ("k", tk, wk)):
            want = oracle.scatter_norm_rope(d[key], P, w, EPS, table)
            for i in range(P):
                assert_fused_ok(tg[i], want[i])
        want_v = oracle.scatter(d["v"], P)
        for i in range(P):
            assert bits_equal(tv[i].cpu(), want_v[i]), (P, D, dtype, i)


# ------------------------------------------------------------------ bandwidth sweep, bf16, single tensor
@pytest.mark.parametrize("P", [2, 4, 8])
def test_sweep_single_tensor(tf, P):
    H, D = 32, 128
    for S in (8, 32, 128, 512, 2048, 8192, 32768, 131072, 262144):
        q = synth.qkv_shards(P, 1, S // P, H, D, torch.bfloat16, seed=S, device="cuda", with_k=False,
                             with_v=False)["q"]
        tq, tk, tv, _ = tf.scatter_qkv("sweep", q)
        assert tk is None and tv is None
        for i, want in enumerate(allgather_scatter(q, P)):
            assert bits_equal(tq[i], want), (P, S, i)
        back, _ = tf.gather_out("sweep", tq)
        for r in range(P):
            assert bits_equal(back[r], q[r]), (P, S, r)
        del q, tq, back
        tf.cache_clear()


# ------------------------------------------------------------------ edge cases
def test_empty_problems_launch_nothing(tf):
    for B, Sl in ((0, 4), (2, 0)):
        q = [torch.empty((B, Sl, 4, 64), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        n0 = tf.launch_count()
        tq, _, _, ev = tf.scatter_qkv("empty", q)
        assert tf.launch_count() == n0
        assert all(t.numel() == 0 for t in tq) and ev
        outs, _ = tf.gather_out("empty", [torch.empty((B, 2 * Sl, 2, 64), dtype=torch.bfloat16, device="cuda")] * 2)
        assert all(o.numel() == 0 for o in outs)


def test_one_launch_per_call(tf):
    g = synth.qkv_shards(4, 1, 64, 8, 64, torch.bfloat16, seed=2, device="cuda", layout="fused")
    wq, wk = synth.norm_weights(64, torch.bfloat16, device="cuda")
    tf.rope_table(THETA, 256, 64)  # build the table first
    n0 = tf.launch_count()
    tf.scatter_qkv("one", g["q"], g["k"], g["v"], norm_rope=True, q_weight=wq, k_weight=wk)
    assert tf.launch_count() == n0 + 1
    tq, _, _, _ = tf.scatter_qkv("one_plain", g["q"], g["k"], g["v"])
    tf.gather_out("one", tq)
    assert tf.launch_count() == n0 + 3


@pytest.mark.parametrize("P,H", [(1, 4), (3, 3), (8, 8), (5, 10)])
def test_shapes_identity_and_single_head_groups(tf, P, H):
    d = synth.qkv_shards(P, 2, 7, H, 32, torch.float16, seed=H)
    g = to_device_like(d)
    tq, _, _, _ = tf.scatter_qkv("shapes", g["q"])
    want = oracle.scatter(d["q"], P)
    for i in range(P):
        assert bits_equal(tq[i].cpu(), want[i])
    if P == 1:
        assert bits_equal(tq[0].cpu(), d["q"][0])


@pytest.mark.parametrize("dtype,D", [(torch.float32, 4), (torch.float32, 36), (torch.uint8, 16),
                                     (torch.uint8, 48), (torch.bfloat16, 8), (torch.float16, 24)])
def test_element_types_and_odd_head_dims(tf, dtype, D):
    P, B, Sl, H = 3, 2, 37, 6
    base = synth.qkv_shards(P, B, Sl, H, D, torch.float32, seed=D, layout="fused")
    conv = (lambda x: ((x * 40).to(torch.int32) % 256).to(torch.uint8)) if dtype == torch.uint8 else (lambda x: x.to(dtype))
    d = {k: [conv(x) for x in base[k]] for k in ("q", "k", "v")}
    tq, tk, tv, _ = tf.scatter_qkv("dtypes", cuda(d["q"]), cuda(d["k"]), cuda(d["v"]))
    for key, tg in (("q", tq), ("k", tk), ("v", tv)):
        want = oracle.scatter(d[key], P)
        for i in range(P):
            assert bits_equal(tg[i].cpu(), want[i]), (dtype, D, key, i)
    back, _ = tf.gather_out("dtypes", tq)
    for r in range(P):
        assert bits_equal(back[r].cpu(), d["q"][r])


def test_exactly_once_unique_ids(tf):
    P, B, Sl, H, D = 4, 2, 16, 8, 32
    ids = synth.unique_id_shards(P, B, Sl, H, D)
    q = [x.view(torch.float16).cuda() for x in ids]
    tq, _, _, _ = tf.scatter_qkv("ids", q)
    got = torch.cat([t.cpu().view(torch.int16).flatten() for t in tq]).sort().values
    want = torch.cat([x.flatten() for x in ids]).sort().values
    assert torch.equal(got, want)


def test_strided_gather_destination_and_guard_bands(tf):
    P, B, Sl, H, D = 4, 2, 33, 8, 64
    dtype = torch.bfloat16
    attn = synth.attn_outputs(P, B, P * Sl, H // P, D, dtype, seed=9)
    # destinations: [B, Sl, H, D] views into a wider buffer; the rest must stay untouched
    canvases = [torch.full((B, Sl, H + 3, D + 8), 7.0, dtype=dtype, device="cuda") for _ in range(P)]
    dst = [c[:, :, 1:H + 1, 8:D + 8] for c in canvases]
    before = [c.clone() for c in canvases]
    outs, _ = tf.gather_out("strided_dst", cuda(attn), out=dst)
    want = oracle.gather(attn, P)
    for r in range(P):
        assert bits_equal(outs[r].cpu(), want[r])
        mask = torch.ones_like(canvases[r], dtype=torch.bool)
        mask[:, :, 1:H + 1, 8:D + 8] = False
        assert torch.equal(canvases[r][mask], before[r][mask]), "wrote outside the destination view"


def test_scatter_into_guard_bands_and_no_write_on_error(tf):
    P, B, Sl, H, D = 2, 1, 50, 4, 64
    dtype = torch.float16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=4)
    n = B * P * Sl * (H // P) * D
    slab = torch.full((P, n + 256), 3.0, dtype=dtype, device="cuda")
    outs = [slab[i, 128:128 + n].view(B, P * Sl, H // P, D) for i in range(P)]
    tf.scatter_qkv_into(cuda(d["q"]), None, None, outs)
    want = oracle.scatter(d["q"], P)
    for i in range(P):
        assert bits_equal(outs[i].cpu(), want[i])
        assert torch.all(slab[i, :128] == 3.0) and torch.all(slab[i, 128 + n:] == 3.0)
    # a rejected call writes nothing
    fresh = torch.full_like(slab, 5.0)
    bad = [fresh[i, 128 + 4:128 + 4 + n].view(B, P * Sl, H // P, D) for i in range(P)]  # 8-byte offset
    with pytest.raises(tf.TfUlyssesError) as ei:
        tf.scatter_qkv_into(cuda(d["q"]), None, None, bad)
    assert ei.value.status == tf.TF_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert torch.all(fresh == 5.0)


def test_cache_capacity_and_lru(tf):
    tf.cache_clear()
    q = synth.qkv_shards(2, 1, 8, 4, 64, torch.bfloat16, seed=1, device="cuda")["q"]
    first, _, _, _ = tf.scatter_qkv("lru0", q)
    for i in range(1, 13):
        tf.scatter_qkv(f"lru{i}", q)
    assert tf.cache_entries() == 12
    again, _, _, _ = tf.scatter_qkv("lru12", q)  # hit
    assert tf.cache_entries() == 12
    torch.cuda.synchronize()
    fresh, _, _, _ = tf.scatter_qkv("lru0", q)  # lru0 was evicted by lru12: a new entry
    assert tf.cache_entries() == 12
    for i, want in enumerate(allgather_scatter(q, 2)):
        assert bits_equal(fresh[i], want) and bits_equal(again[i], want)
    tf.cache_clear()
    assert tf.cache_entries() == 0


def test_other_stream_and_default_allocator(tf):
    tf.use_torch_allocator(False)  # cudaMallocAsync / cudaFreeAsync
    try:
        s = torch.cuda.Stream()
        g = synth.qkv_shards(4, 2, 100, 8, 128, torch.bfloat16, seed=8, device="cuda", layout="fused")
        wq, wk = synth.norm_weights(128, torch.bfloat16, device="cuda", seed=8)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            tq, tk, tv, _ = tf.scatter_qkv("stream", g["q"], g["k"], g["v"], norm_rope=True, q_weight=wq,
                                           k_weight=wk, stream=s)
        s.synchronize()
        table = oracle.rope_table(THETA, 400, 128)
        want = oracle.scatter_norm_rope(cpu(g["q"]), 4, wq.cpu(), EPS, table)
        for i in range(4):
            assert_fused_ok(tq[i], want[i])
        tf.cache_clear()
    finally:
        tf.use_torch_allocator(True)


def test_padding_rows_normalise_to_zero(tf):
    P, B, S0, H, D = 4, 1, 1001, 8, 128
    S = synth.padded_seq(S0, P)
    d = synth.qkv_shards(P, B, S // P, H, D, torch.bfloat16, seed=6, pad_from=S0)
    wq, wk = synth.norm_weights(D, torch.bfloat16, seed=6)
    tq, _, _, _ = tf.scatter_qkv("pad", cuda(d["q"]), norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda())
    for i in range(P):
        assert torch.all(tq[i][:, S0:].float() == 0)
    want = oracle.scatter_norm_rope(d["q"], P, wq, EPS, oracle.rope_table(THETA, S, D))
    for i in range(P):
        assert_fused_ok(tq[i], want[i])
    assert int(ulp_diff(tq[0].cpu(), want[0]).max()) <= 1


# ------------------------------------------------------------------ fused: slot patterns, head dims, unit tails
@pytest.mark.parametrize("with_k,with_v", [(True, True), (True, False), (False, True), (False, False)])
@pytest.mark.parametrize("D", [32, 64, 128, 256])
def test_fused_slot_patterns_and_head_dims(tf, with_k, with_v, D):
    """Q alone, Q+K, Q+V, Q+K+V, for every supported D; 3 * 37 * Hl rows per block
    do not fill whole units of token blocks, and B=2 covers the batch stride."""
    P, B, Sl, H = 3, 2, 37, 6
    dtype = torch.bfloat16 if D != 64 else torch.float16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=40 + D, layout="fused", with_k=with_k, with_v=with_v)
    wq, wk = synth.norm_weights(D, dtype, seed=D)
    g = to_device_like(d)
    tq, tk, tv, _ = tf.scatter_qkv(f"slots{D}{with_k}{with_v}", g["q"], g["k"], g["v"], norm_rope=True,
                                   q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA)
    assert (tk is None) == (not with_k) and (tv is None) == (not with_v)
    table = oracle.rope_table(THETA, P * Sl, D)
    fused = [("q", tq, wq)] + ([("k", tk, wk)] if with_k else [])
    for key, tg, w in fused:
        want = oracle.scatter_norm_rope(d[key], P, w, EPS, table)
        for i in range(P):
            assert_fused_ok(tg[i], want[i])
    if with_v:
        want_v = oracle.scatter(d["v"], P)
        for i in range(P):
            assert bits_equal(tv[i].cpu(), want_v[i])


def test_fused_16_byte_aligned_sources(tf):
    """Sources only 16-byte aligned (an 8-element offset into the projection):
    the fused scatter falls back to 16-byte vectors with the same results."""
    P, B, Sl, H, D = 2, 1, 300, 4, 128
    dtype = torch.bfloat16
    gen = torch.Generator().manual_seed(77)
    HD = H * D
    bufs = [torch.randn(B, Sl, 3 * HD + 8, generator=gen).to(dtype) for _ in range(P)]
    q = [b[..., 8:8 + HD].unflatten(-1, (H, D)) for b in bufs]
    k = [b[..., 8 + HD:8 + 2 * HD].unflatten(-1, (H, D)) for b in bufs]
    v = [b[..., 8 + 2 * HD:8 + 3 * HD].unflatten(-1, (H, D)) for b in bufs]
    wq, wk = synth.norm_weights(D, dtype, seed=77)
    gb = [b.cuda() for b in bufs]
    gq = [b[..., 8:8 + HD].unflatten(-1, (H, D)) for b in gb]
    gk = [b[..., 8 + HD:8 + 2 * HD].unflatten(-1, (H, D)) for b in gb]
    gv = [b[..., 8 + 2 * HD:8 + 3 * HD].unflatten(-1, (H, D)) for b in gb]
    assert gq[0].data_ptr() % 32 == 16
    tq, tk, tv, _ = tf.scatter_qkv("align16", gq, gk, gv, norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(),
                                   eps=EPS, theta=THETA)
    table = oracle.rope_table(THETA, P * Sl, D)
    for src, tg, w in ((q, tq, wq), (k, tk, wk)):
        want = oracle.scatter_norm_rope(src, P, w, EPS, table)
        for i in range(P):
            assert_fused_ok(tg[i], want[i])
    want_v = oracle.scatter(v, P)
    for i in range(P):
        assert bits_equal(tv[i].cpu(), want_v[i])


def test_device_status_clean_after_all_launches(tf):
    """No bounded in-kernel wait gave up during any launch of this process so far,
    and (checked builds) no block-kernel access fell outside its planned buffer."""
    torch.cuda.synchronize()
    assert tf.device_status(clear=False) == 0
