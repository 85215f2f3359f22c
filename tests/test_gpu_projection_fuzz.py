"""Seeded random cases of the fused QKV projection, through the C ABI.

Each case draws P, B, S_local, H (even, a multiple of P), hidden (a multiple of
64), the mode (plain, RMSNorm + interleaved RoPE, RMSNorm + half-split RoPE),
the target layout (separate Q/K/V or one fused payload per head group) and
padded row strides of x and the weight.  Inputs are dyadic (x = i/8, w = j/16),
so every sum is exact in fp32 and the whole path must match the oracle bit for
bit (fused rows up to the isolated flips of parity_util.assert_fused_ok).  The
shapes reach odd numbers of 128-row tiles (a CTA pair whose second CTA has no
rows), ragged last tiles, a single row, and raster passes that end part way.
"""
import random

import pytest
import torch

import oracle
from parity_util import assert_fused_ok, bits_equal
from ulysses_sequence_attention_tf_gb300 import synth

pytestmark = pytest.mark.gpu

EPS = 1e-6
D = 128
DT = torch.bfloat16
N_CASES = 40
MAX_MACS = 6e7  # oracle cost bound per case (about a second)


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
    while True:
        P = rng.randint(1, 8)
        Hl = rng.randint(1, 3)
        if (P * Hl) % 2:
            Hl += 1
        Sl = rng.choice([1, 7, 127, 128, 129, 200, 256, 300, rng.randint(1, 400)])
        c = dict(P=P, H=P * Hl, B=rng.randint(1, 2), Sl=Sl, hidden=64 * rng.randint(1, 8),
                 mode=rng.choice(["plain", "interleaved", "neox"]),
                 layout=rng.choice(["bshd", "fused"]), x_pad=rng.choice([0, 8]), w_pad=rng.choice([0, 64]),
                 theta=rng.choice([500.0, 10000.0]))
        macs = c["P"] * c["B"] * c["Sl"] * 3 * c["H"] * D * c["hidden"]
        if macs <= MAX_MACS:
            return c


def _device_copy(t):
    """A device tensor with the same shape and strides as the host view t."""
    base = torch.empty(t.untyped_storage().nbytes() // t.element_size(), dtype=t.dtype, device="cuda")
    return torch.as_strided(base, t.shape, t.stride(), t.storage_offset()).copy_(t)


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_projection_vs_oracle(tf, case):
    rng = random.Random(5000 + case)
    c = _draw(rng)
    P, B, Sl, H, hidden = c["P"], c["B"], c["Sl"], c["H"], c["hidden"]
    S, Hl = P * Sl, H // P
    xs, w = synth.projection_inputs(P, B, Sl, hidden, H, D, DT, seed=6000 + case, x_pad=c["x_pad"],
                                    w_pad=c["w_pad"], dist="dyadic")
    wq, wk = synth.norm_weights(D, DT, seed=case)
    fused = c["mode"] != "plain"
    style = "neox" if c["mode"] == "neox" else "interleaved"
    kw = dict(norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=c["theta"], rope=style) \
        if fused else {}
    gx, gw = [_device_copy(x) for x in xs], _device_copy(w)
    fill = -7.0
    if c["layout"] == "fused":
        pay = [torch.full((B, S, Hl, 3 * D), fill, dtype=DT, device="cuda") for _ in range(P)]
        tf.project_qkv_into(gx, gw, H, pay, layout="fused", **kw)
        got = {key: [p[..., i * D:(i + 1) * D] for p in pay] for i, key in enumerate("qkv")}
    else:
        got = {key: [torch.full((B, S, Hl, D), fill, dtype=DT, device="cuda") for _ in range(P)] for key in "qkv"}
        tf.project_qkv_into(gx, gw, H, got["q"], got["k"], got["v"], **kw)
    torch.cuda.synchronize()
    assert tf.device_status(clear=False) == 0
    proj = oracle.project_qkv(xs, w, H, D)
    table = oracle.rope_table(c["theta"], S, D) if fused else None
    for key in "qkv":
        if fused and key != "v":
            want = oracle.scatter_norm_rope(proj[key], P, wq if key == "q" else wk, EPS, table, style=style)
        else:
            want = oracle.scatter(proj[key], P)
        for g in range(P):
            out = got[key][g].cpu().contiguous()
            if fused and key != "v":
                assert_fused_ok(out, want[g])
            else:
                assert bits_equal(out, want[g]), (c, key, g)
