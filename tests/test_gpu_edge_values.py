"""The fused RMSNorm + RoPE on rows with extreme and non-finite values, against
the oracle, through the C ABI.

bf16 holds values up to 3.4e38, so a head row can hold elements whose squares
(from |x| = 2^64) or whose sum of squares overflow fp32 while the row's mean
still fits; the fp32 RMSNorm of flashinfer PR #6332 ("Assumptions / Operator
math") then needs the exact mean, and where the mean itself leaves the fp32
range it is +inf and the row normalises to zeros.  Infinite and NaN inputs
follow IEEE arithmetic at every step: a NaN turns its whole row NaN, an
infinite element (no NaN) gives zeros except NaN at the element and its
rotation partner.  Rows of subnormals, zeros and tiny values have means far
below eps.

Planted among N(0, 1) rows (synth.plant_edge_rows): constant rows at 2^63,
2^64 and 2^100, N(0, 1) rows scaled by 2^60 and 2^62, single elements of 2^64
and 2^100, +-inf, NaN, subnormals, zeros, tiny rows (bf16); fp16 max, +-inf,
NaN, subnormals, zeros, tiny rows (fp16).  Paths: the block kernel (32-byte
aligned sources; V+Q+K and Q/K only; interleaved and half-split; D = 32 ... 256)
and the register kernel (16-byte aligned sources), and the projection's
epilogue with projected values that overflow fp32 squares.
"""
import pytest
import torch

import oracle
from parity_util import assert_fused_ok_nonfinite, bits_equal
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


def _device_copy(t):
    """A device copy of a CPU view that keeps its strides (and 16-byte alignment)."""
    if t.is_contiguous():
        return t.cuda()
    store = torch.empty(t.untyped_storage().nbytes() // t.element_size(), dtype=t.dtype, device="cuda")
    return torch.as_strided(store, t.shape, t.stride(), t.storage_offset()).copy_(t)


def _sources(P, B, Sl, H, D, dtype, layout, gen):
    """Q, K, V shards [B, Sl, H, D] on the CPU: 'v_strided' (Q/K contiguous, V a
    view of a fused projection: 32-byte aligned rows), or 'pad16' (every head row
    16 bytes apart from the next row's start modulo 32: the register kernel)."""
    out = {"q": [], "k": [], "v": []}
    for _ in range(P):
        if layout == "v_strided":
            for key in "qk":
                out[key].append(torch.randn((B, Sl, H, D), generator=gen).to(dtype))
            buf = torch.randn((B, Sl, 3 * H * D), generator=gen).to(dtype)
            out["v"].append(buf[..., 2 * H * D:].unflatten(-1, (H, D)))
        else:
            for key in "qkv":
                buf = torch.randn((B, Sl, H, D + 8), generator=gen).to(dtype)  # rows 2*D + 16 bytes apart
                out[key].append(buf[..., :D])
    return out


CASES = [
    # P, B, Sl, H, D, dtype, layout, with_v, rope
    (4, 1, 96, 16, 128, torch.bfloat16, "v_strided", True, "interleaved"),
    (4, 1, 96, 16, 128, torch.bfloat16, "v_strided", True, "neox"),
    (4, 1, 96, 16, 128, torch.bfloat16, "v_strided", False, "interleaved"),
    (4, 1, 96, 16, 128, torch.bfloat16, "v_strided", False, "neox"),
    (2, 2, 70, 8, 64, torch.bfloat16, "v_strided", True, "interleaved"),
    (2, 1, 40, 4, 256, torch.bfloat16, "v_strided", True, "neox"),
    (3, 1, 50, 6, 32, torch.bfloat16, "v_strided", True, "interleaved"),
    (4, 1, 96, 16, 128, torch.float16, "v_strided", True, "interleaved"),
    (4, 1, 96, 16, 128, torch.float16, "v_strided", False, "neox"),
    (4, 1, 96, 16, 128, torch.bfloat16, "pad16", True, "interleaved"),
    (4, 1, 96, 16, 128, torch.bfloat16, "pad16", True, "neox"),
    (2, 1, 64, 4, 256, torch.bfloat16, "pad16", True, "interleaved"),
    (4, 1, 96, 16, 64, torch.float16, "pad16", True, "neox"),
    # Q/K only at every lane count and with 16-byte-aligned rows (the (cos, sin)
    # ring and the paired rows, then the recompute pass)
    (2, 2, 70, 8, 64, torch.float16, "v_strided", False, "interleaved"),
    (3, 1, 50, 6, 32, torch.bfloat16, "v_strided", False, "neox"),
    (4, 1, 96, 16, 128, torch.bfloat16, "pad16", False, "interleaved"),
    (2, 1, 64, 4, 256, torch.float16, "pad16", False, "neox"),
]


@pytest.mark.parametrize("P,B,Sl,H,D,dtype,layout,with_v,rope", CASES)
def test_edge_rows_vs_oracle(tf, P, B, Sl, H, D, dtype, layout, with_v, rope):
    gen = torch.Generator().manual_seed(P * 1000 + Sl + D)
    src = _sources(P, B, Sl, H, D, dtype, layout, gen)
    planted = sum(synth.plant_edge_rows(src[key], seed=i, every=5 + i) for i, key in enumerate("qk"))
    assert planted > 0
    S, Hl = P * Sl, H // P
    g = {key: [_device_copy(t) for t in src[key]] for key in "qkv"}
    wq, wk = synth.norm_weights(D, dtype, seed=D)
    outs = [[torch.full((B, S, Hl, D), 7.0, dtype=dtype, device="cuda") for _ in range(P)] for _ in "qkv"]
    tf.scatter_qkv_into(g["q"], g["k"], g["v"] if with_v else None, outs[0], outs[1], outs[2] if with_v else None,
                        norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA, rope=rope)
    torch.cuda.synchronize()
    table = oracle.rope_table(THETA, S, D)
    n_nan = n_zero_rows = 0
    for x, (key, w) in enumerate((("q", wq), ("k", wk))):
        want = oracle.scatter_norm_rope(src[key], P, w, EPS, table, style=rope)
        for gi in range(P):
            assert_fused_ok_nonfinite(outs[x][gi], want[gi])
            n_nan += int(torch.isnan(want[gi].float()).sum())
            n_zero_rows += int((want[gi].float() == 0).all(-1).sum())
    assert n_nan > 0 and n_zero_rows > 0  # the non-finite and the overflowing rows were there
    if with_v:
        want_v = oracle.scatter(src["v"], P)
        for gi in range(P):
            assert bits_equal(outs[2][gi].cpu(), want_v[gi])
    assert tf.device_status(clear=False) == 0


def test_projection_edge_rows_vs_oracle(tf):
    """Projected head rows that hold a value of 2^64 (the square overflows fp32,
    the mean fits: the epilogue's rescaled path), rows whose mean overflows (2^80:
    zeros), an element that overflows the projection itself (2^140 -> inf) and a
    NaN hidden state, among dyadic rows whose sums are exact in any order."""
    P, B, Sl, hidden, H, D = 2, 1, 256, 128, 4, 128
    dtype = torch.bfloat16
    S, Hl, HD = P * Sl, H // P, H * D
    xs, w = synth.projection_inputs(P, B, Sl, hidden, H, D, dtype, seed=17, dist="dyadic")
    xs = [x.clone() for x in xs]
    w = w.clone()
    for x in xs:
        x[..., 0] = 0  # column 0 carries only the planted products below
    w[:, 0] = 0
    f_spike = 0 * HD + 1 * D + 5  # Q, head 1, element 5
    f_big = 1 * HD + 2 * D  # K, head 2, all elements
    f_inf = 1 * HD + 0 * D + 9  # K, head 0, element 9
    w[f_spike, 0] = 2.0 ** 32
    w[f_big:f_big + D, 0] = 2.0 ** 20
    w[f_inf, 0] = 2.0 ** 40
    xs[0][0, 3, 0] = 2.0 ** 32  # -> 2^64 at f_spike
    xs[1][0, 100, 0] = 2.0 ** 60  # -> 2^80 over K head 2: the mean overflows
    xs[0][0, 250, 0] = 2.0 ** 100  # -> 2^140: the projection itself overflows to inf
    xs[1][0, 7, 0] = float("nan")  # a NaN hidden state: its whole token row is NaN
    for r, t in ((0, 3), (1, 100), (0, 250)):  # several rows of one tile take the rescaled path
        xs[r][0, t + 1, 0] = xs[r][0, t, 0]
    wq, wk = synth.norm_weights(D, dtype, seed=17)
    outs = {k: [torch.full((B, S, Hl, D), -5.0, dtype=dtype, device="cuda") for _ in range(P)] for k in "qkv"}
    tf.project_qkv_into([x.cuda() for x in xs], w.cuda(), H, outs["q"], outs["k"], outs["v"], norm_rope=True,
                        q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA)
    torch.cuda.synchronize()
    proj = oracle.project_qkv(xs, w, H, D)
    assert float(proj["q"][0][0, 3, 1, 5]) == 2.0 ** 64 and float(proj["k"][1][0, 100, 2, 0]) == 2.0 ** 80
    assert torch.isinf(proj["k"][0][0, 250, 0, 9].float())
    table = oracle.rope_table(THETA, S, D)
    for key, wn in (("q", wq), ("k", wk)):
        want = oracle.scatter_norm_rope(proj[key], P, wn, EPS, table)
        for g in range(P):
            assert_fused_ok_nonfinite(outs[key][g], want[g])
    want_v = oracle.scatter(proj["v"], P)
    for g in range(P):
        got, ref = outs["v"][g].cpu(), want_v[g]
        nan = torch.isnan(ref.float())
        assert torch.equal(torch.isnan(got.float()), nan)
        assert bits_equal(got[~nan], ref[~nan])
    # the planted rows came out as the reading says: the 2^64 row normalised (finite,
    # nonzero), the 2^80 row zeros, the inf row NaN at its pair, the NaN token NaN
    q_spike = outs["q"][0][0, 3, 1].float().cpu()  # head 1 is local head 1 of group 0
    assert torch.isfinite(q_spike).all() and q_spike.abs().max() > 1.0
    assert torch.all(outs["k"][1][0, Sl + 100, 0].float() == 0)  # K head 2: group 1, local head 0
    k_inf = outs["k"][0][0, 250, 0].float().cpu()  # K head 0: group 0, local head 0
    assert int(torch.isnan(k_inf).sum()) == 2 and torch.all(k_inf[~torch.isnan(k_inf)] == 0)
    assert torch.isnan(outs["v"][0][0, Sl + 7].float()).all()
    assert tf.device_status(clear=False) == 0
