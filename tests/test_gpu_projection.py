"""Parity of the fused QKV projection (tcgen05 GEMM + RMSNorm/RoPE + scatter
epilogue) with the CPU oracle, through the C ABI.

The oracle projects with the exact sum rounded once to bf16; the tensor cores
sum in fp32 in their own order.  Two kinds of input:
  * dyadic (x = i/8, w = j/16): every product and partial sum is exact in fp32,
    so any summation order gives the exact sum and the whole path -- projection,
    RMSNorm, RoPE, scatter -- must match the oracle bit for bit (the fused rows
    up to the isolated flips of parity_util.assert_fused_ok);
  * N(0, 1): a value can land on the other side of a bf16 rounding boundary
    (flashinfer PR #6332 commit message, "Assumptions / Tolerance"), checked with
    the pages' atol = rtol = 1e-2 and the one-ulp classification.
"""
import pytest
import torch

import oracle
from parity_util import assert_fused_ok, assert_projected_ok, bits_equal
from ulysses_sequence_attention_tf_gb300 import synth

pytestmark = pytest.mark.gpu

EPS = 1e-6
THETA = 10000.0
D = 128
DT = torch.bfloat16


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


def _targets(P, B, S, Hl, width=1, fill=-5.0):
    return [torch.full((B, S, Hl, width * D), fill, dtype=DT, device="cuda") for _ in range(P)]


def _oracle(xs, w, P, H, norm_rope, wq, wk, style, S):
    proj = oracle.project_qkv(xs, w, H, D)
    out = {}
    table = oracle.rope_table(THETA, S, D) if norm_rope else None
    for key in "qkv":
        if norm_rope and key != "v":
            out[key] = oracle.scatter_norm_rope(proj[key], P, wq if key == "q" else wk, EPS, table, style=style)
        else:
            out[key] = oracle.scatter(proj[key], P)
    return out


def _check(got, want, exact, fused_row):
    if exact and fused_row:
        assert_fused_ok(got, want)
    elif exact:
        assert bits_equal(got.cpu(), want)
    else:
        assert_projected_ok(got, want, min_identical=0.9 if fused_row else 0.98)


@pytest.mark.parametrize("dist", ["dyadic", "normal"])
@pytest.mark.parametrize("norm_rope,style", [(False, "interleaved"), (True, "interleaved"), (True, "neox")])
@pytest.mark.parametrize("P,B,Sl,hidden,H", [(2, 1, 200, 256, 4), (4, 2, 70, 192, 8), (1, 1, 128, 64, 2)])
def test_projection_vs_oracle(tf, dist, norm_rope, style, P, B, Sl, hidden, H):
    S, Hl = P * Sl, H // P
    xs, w = synth.projection_inputs(P, B, Sl, hidden, H, D, DT, seed=P * 100 + hidden, dist=dist)
    wq, wk = synth.norm_weights(D, DT, seed=hidden)
    outs = {k: _targets(P, B, S, Hl) for k in "qkv"}
    kw = dict(norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA, rope=style) \
        if norm_rope else {}
    tf.project_qkv_into([x.cuda() for x in xs], w.cuda(), H, outs["q"], outs["k"], outs["v"], **kw)
    torch.cuda.synchronize()
    want = _oracle(xs, w, P, H, norm_rope, wq, wk, style, S)
    for key in "qkv":
        for g in range(P):
            _check(outs[key][g], want[key][g], dist == "dyadic", norm_rope and key != "v")


def test_projection_strided_inputs_fused_layout_and_guards(tf):
    P, B, Sl, hidden, H = 2, 1, 150, 128, 4
    S, Hl = P * Sl, H // P
    xs, w = synth.projection_inputs(P, B, Sl, hidden, H, D, DT, seed=7, x_pad=8, w_pad=64, dist="dyadic")
    assert xs[0].stride(1) == hidden + 8 and w.stride(0) == hidden + 64
    wq, wk = synth.norm_weights(D, DT, seed=7)
    guard = 256
    slabs = [torch.full((B * S * Hl * 3 * D + 2 * guard,), -9.0, dtype=DT, device="cuda") for _ in range(P)]
    pay = [s[guard:-guard].view(B, S, Hl, 3 * D) for s in slabs]
    gx = [torch.as_strided(torch.empty(B * Sl * (hidden + 8), dtype=DT, device="cuda"), x.shape, x.stride())
          .copy_(x) for x in xs]  # device copies with the same row strides
    gw = torch.as_strided(torch.empty(w.shape[0] * (hidden + 64), dtype=DT, device="cuda"), w.shape,
                          w.stride()).copy_(w)
    tf.project_qkv_into(gx, gw, H, pay, norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS,
                        theta=THETA, layout="fused")
    torch.cuda.synchronize()
    want = _oracle(xs, w, P, H, True, wq, wk, "interleaved", S)
    for g in range(P):
        assert torch.all(slabs[g][:guard] == -9.0) and torch.all(slabs[g][-guard:] == -9.0)
        assert_fused_ok(pay[g][..., :D].contiguous(), want["q"][g])
        assert_fused_ok(pay[g][..., D:2 * D].contiguous(), want["k"][g])
        assert bits_equal(pay[g][..., 2 * D:].cpu(), want["v"][g])


def test_projection_rejects_unsupported(tf):
    xs, w = synth.projection_inputs(2, 1, 8, 100, 4, D, DT, seed=1)  # hidden not a multiple of 64
    outs = {k: _targets(2, 1, 16, 2) for k in "qkv"}
    with pytest.raises(tf.TfUlyssesError) as e:
        tf.project_qkv_into([x.cuda() for x in xs], w.cuda(), 4, outs["q"], outs["k"], outs["v"])
    assert e.value.status == tf.TF_ERR_UNSUPPORTED
    assert torch.all(outs["q"][0] == -5.0)


@pytest.mark.parametrize("dist", ["dyadic", "normal"])
def test_projection_video_dit_sampled(tf, dist):
    """Video-DiT shape (P=4, S=32760, H=40, hidden=5120, bf16), fused Q/K:
    sampled rows of every tensor against the oracle, row by row."""
    P, B, Sl, H = 4, 1, 8190, 40
    hidden, S, Hl = H * D, P * Sl, H // P
    xs, w = synth.projection_inputs(P, B, Sl, hidden, H, D, DT, seed=3, device="cuda", dist=dist)
    wq, wk = synth.norm_weights(D, DT, seed=3, device="cuda")
    outs = {k: [torch.empty((B, S, Hl, D), dtype=DT, device="cuda") for _ in range(P)] for k in "qkv"}
    tf.project_qkv_into(xs, w, H, outs["q"], outs["k"], outs["v"], norm_rope=True, q_weight=wq, k_weight=wk,
                        eps=EPS, theta=THETA)
    torch.cuda.synchronize()
    w_cpu, wq_c, wk_c = w.cpu(), wq.cpu(), wk.cpu()
    table = oracle.rope_table(THETA, S, D)
    gen = torch.Generator().manual_seed(5)
    HD = H * D
    for key, sec in (("q", 0), ("k", 1), ("v", 2)):
        got, want = [], []
        for i in range(24):
            g, p, hh = (int(torch.randint(n, (1,), generator=gen)) for n in (P, S, Hl))
            if i == 0:
                p = S - 1
            r, t = divmod(p, Sl)
            h = g * Hl + hh
            n0 = sec * HD + h * D
            row = oracle.project_row_range(xs[r][0, t].cpu(), w_cpu, n0, n0 + D)
            if key != "v":
                row = oracle.rmsnorm_rope_row(row, wq_c if key == "q" else wk_c, EPS, table[p])
            want.append(row)
            got.append(outs[key][g][0, p, hh].cpu())
        got, want = torch.stack(got), torch.stack(want)
        if dist == "dyadic":
            _check(got, want, True, key != "v")
        else:
            assert_projected_ok(got, want, min_identical=0.8 if key != "v" else 0.95)


def test_device_status_clean(tf):
    torch.cuda.synchronize()
    assert tf.device_status(clear=False) == 0
