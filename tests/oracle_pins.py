"""Pins of the CPU oracle to things other than itself.

Each ``check_*`` takes a loaded oracle library (``oracle.load(path)``) and raises
AssertionError when the oracle disagrees with what the pages, the mathematics or
an independent library routine fix.  ``test_oracle_pins.py`` runs them on the
oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle with a
planted mistake and expects at least one to fail.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle
from ulysses_sequence_attention_tf_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def ordered16(bits: torch.Tensor) -> torch.Tensor:
    """Map 16-bit float patterns to integers whose difference counts ulps."""
    b = bits.to(torch.int32) & 0xFFFF
    mag = b & 0x7FFF
    return torch.where(b >= 0x8000, -mag, mag)


def ulp_diff(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    return (ordered16(a.view(torch.int16)) - ordered16(b.view(torch.int16))).abs()


# ----------------------------------------------------------------------------
# 16-bit codecs vs the library conversions (torch for bfloat16, numpy for binary16)
# ----------------------------------------------------------------------------

def check_codec_decode(lib):
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref_bf = bits.view(torch.bfloat16).double().numpy()
    ref_h = bits.numpy().view(np.float16).astype(np.float64)
    for fmt, ref in ((1, ref_bf), (0, ref_h)):
        step = 7 if fmt == 1 else 5  # a spread of patterns over every exponent
        for i in list(range(0, 65536, step)) + [0x0000, 0x8000, 0x0001, 0x7F7F, 0x7F80, 0xFF80, 0x7BFF, 0x7C00, 0x03FF]:
            got = lib.tfo_decode16(fmt, i)
            want = ref[i]
            assert (math.isnan(got) and math.isnan(want)) or got == want, (fmt, hex(i), got, want)


def _fp32_probe_values(n=60000, seed=3):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    # exact ties for bf16 (low 16 bits 0x8000) and for fp16 (13 low bits at the half point)
    ties_bf = (rng.integers(0, 2**16, size=4000, dtype=np.uint64).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    mant = rng.integers(0, 2**10, size=4000, dtype=np.uint64).astype(np.uint32)
    exps = rng.integers(100, 143, size=4000, dtype=np.uint64).astype(np.uint32)  # around fp16 range
    ties_h = ((exps << 23) | (mant << 13) | (1 << 12)).view(np.float32)
    normal = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    tiny = (rng.standard_normal(4000) * 1e-6).astype(np.float32)  # fp16 subnormal range
    big = np.array([65504.0, 65519.99, 65520.0, 65536.0, 3.3895314e38, 3.4e38, -65520.0, 0.0, -0.0,
                    5.96e-8, 2.98e-8, 2.99e-8, 1e-40, -1e-45], dtype=np.float32)
    allv = np.concatenate([vals, ties_bf[np.isfinite(ties_bf)], ties_h, normal, tiny, big])
    return allv.astype(np.float32)


def check_codec_encode(lib):
    vals = _fp32_probe_values()
    want_bf = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    with np.errstate(over="ignore"):  # overflow to infinity is part of what is checked
        want_h = vals.astype(np.float16).view(np.uint16)
    for i, x in enumerate(vals.tolist()):
        gb = lib.tfo_encode16(1, x)
        assert gb == want_bf[i], ("bf16", x, hex(gb), hex(want_bf[i]))
        gh = lib.tfo_encode16(0, x)
        assert gh == want_h[i], ("fp16", x, hex(gh), hex(want_h[i]))


# ----------------------------------------------------------------------------
# Relayout
# ----------------------------------------------------------------------------

def check_relayout_golden(lib):
    with open(os.path.join(GOLDEN, "relayout_handworked.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        P = case["P"]
        srcs = [torch.tensor(s, dtype=torch.int32).unsqueeze(0) for s in case["sources"]]
        tgts = [torch.tensor(s, dtype=torch.int32).unsqueeze(0) for s in case["targets"]]
        got = oracle.scatter(srcs, P, lib=lib)
        for g in range(P):
            assert torch.equal(got[g], tgts[g]), (case, g, got[g])
        back = oracle.gather(tgts, P, lib=lib)
        for r in range(P):
            assert torch.equal(back[r], srcs[r]), (case, r)


def _allgather_scatter_reference(srcs, P):
    """The all-gather formulation: concatenate the shards along the sequence in
    rank order, then take head band g (library routines only)."""
    full = torch.cat([s.contiguous() for s in srcs], dim=1)
    Hl = full.shape[2] // P
    return [full[:, :, g * Hl:(g + 1) * Hl, :].contiguous() for g in range(P)]


def _allgather_gather_reference(attn, P):
    """Inverse: concatenate the head groups along heads, then take shard r's tokens."""
    full = torch.cat([a.contiguous() for a in attn], dim=2)
    Sl = full.shape[1] // P
    return [full[:, r * Sl:(r + 1) * Sl].contiguous() for r in range(P)]


RELAYOUT_SHAPES = [
    # P, B, Sl, H, D, layout, dtype
    (1, 1, 3, 2, 4, "contiguous", torch.int16),
    (2, 1, 5, 4, 8, "contiguous", torch.bfloat16),
    (3, 2, 3, 6, 2, "fused", torch.float16),
    (4, 2, 1, 8, 3, "v_strided", torch.bfloat16),
    (2, 3, 4, 6, 1, "fused", torch.float32),
    (5, 1, 2, 10, 5, "contiguous", torch.int8),
    (4, 1, 6, 4, 16, "v_strided", torch.float64),
]


def _shards(P, B, Sl, H, D, layout, dtype, seed):
    if dtype in (torch.int8, torch.int16):
        d = synth.qkv_shards(P, B, Sl, H, D, torch.float32, seed=seed, layout=layout)
        cast = lambda x: (x * 50).to(dtype)  # noqa: E731  (views keep their strides below)
        out = {}
        for key in ("q", "k", "v"):
            out[key] = [cast(x) for x in d[key]]
        return out
    return synth.qkv_shards(P, B, Sl, H, D, dtype, seed=seed, layout=layout)


def check_relayout_allgather(lib):
    for i, (P, B, Sl, H, D, layout, dtype) in enumerate(RELAYOUT_SHAPES):
        d = _shards(P, B, Sl, H, D, layout, dtype, seed=11 + i)
        for key in ("q", "v"):
            srcs = d[key]
            got = oracle.scatter(srcs, P, lib=lib)
            want = _allgather_scatter_reference(srcs, P)
            for g in range(P):
                assert torch.equal(got[g].view(torch.uint8), want[g].view(torch.uint8)), (P, B, Sl, H, D, layout, key, g)
            back = oracle.gather(got, P, lib=lib)
            want_back = _allgather_gather_reference(got, P)
            for r in range(P):
                assert torch.equal(back[r].view(torch.uint8), want_back[r].view(torch.uint8)), ("gather", P, key, r)


def check_relayout_invariants(lib):
    # exactly once: distinct ids land once each; gather(scatter(x)) == x; P = 1 is the identity layout
    for P, B, Sl, H, D in [(2, 1, 4, 4, 2), (3, 2, 2, 6, 4), (4, 1, 3, 8, 2), (1, 2, 5, 3, 4), (8, 1, 2, 8, 8)]:
        srcs = synth.unique_id_shards(P, B, Sl, H, D)
        tg = oracle.scatter(srcs, P, lib=lib)
        src_ids = torch.cat([s.flatten() for s in srcs]).sort().values
        tgt_ids = torch.cat([t.flatten() for t in tg]).sort().values
        assert torch.equal(src_ids, tgt_ids), "an element was lost or duplicated"
        back = oracle.gather(tg, P, lib=lib)
        for r in range(P):
            assert torch.equal(back[r], srcs[r]), ("round trip", P, r)
        if P == 1:
            assert torch.equal(tg[0], srcs[0]), "P = 1 must be the identity layout"


# ----------------------------------------------------------------------------
# RMSNorm + RoPE
# ----------------------------------------------------------------------------

def _table_row(lib, theta, S, D, p):
    return oracle.rope_table(theta, S, D, lib=lib)[p]


def check_rope_table_textbook(lib):
    with open(os.path.join(GOLDEN, "rope_textbook.json")) as f:
        gold = json.load(f)
    c1, s1 = np.float32(gold["cos_1"]), np.float32(gold["sin_1"])
    for case in gold["cases"]:
        tab = oracle.rope_table(case["theta"], case["p"] + 1, case["D"], lib=lib)
        c, s = tab[case["p"], case["i"]].tolist()
        assert np.float32(c) == c1 and np.float32(s) == s1, (case, c, s)
    # position 0 is the identity rotation
    tab = oracle.rope_table(10000.0, 3, 128, lib=lib)
    assert torch.all(tab[0, :, 0] == 1.0) and torch.all(tab[0, :, 1] == 0.0)
    # pair 0 rotates by exactly p radians; every entry lies on the unit circle
    tab = oracle.rope_table(10000.0, 4096, 64, lib=lib).double()
    r2 = tab[..., 0] ** 2 + tab[..., 1] ** 2
    assert torch.all((r2 - 1).abs() < 4e-7)
    # angle addition: rot((p+q) f) = rot(p f) rot(q f) for a frequency f of the table
    p, q = 1234, 987
    cp, sp = tab[p, :, 0], tab[p, :, 1]
    cq, sq = tab[q, :, 0], tab[q, :, 1]
    assert torch.all((cp * cq - sp * sq - tab[p + q, :, 0]).abs() < 2e-6)
    assert torch.all((sp * cq + cp * sq - tab[p + q, :, 1]).abs() < 2e-6)


def _rms_norm_torch(x: torch.Tensor, w: torch.Tensor, eps: float):
    """Library reference of the normalise step: fp32 rms_norm, cast, then 16-bit weight scale."""
    y = torch.nn.functional.rms_norm(x.float(), (x.shape[-1],), eps=eps).to(x.dtype)
    return y * w  # 16-bit x 16-bit product, rounded to the 16-bit type


def check_rmsnorm_vs_torch(lib):
    eps = 1e-6
    for dtype in (torch.bfloat16, torch.float16):
        for D in (64, 128):
            gen = synth.make_generator(5, "cpu")
            x = torch.randn((400, D), generator=gen).to(dtype)
            x[0] = 0  # zero row: 0 * 1/sqrt(eps) = 0
            x[1] = 3.0  # constant row
            x[2] *= 1e-3  # tiny row, where eps matters
            # rows whose squares are fp32 subnormals or vanish, and subnormal inputs:
            # the mean is negligible next to eps, so y = x / sqrt(eps) rounded
            x[3] = (torch.randn((D,), generator=gen) * 2.0 ** -70).to(dtype)
            frac_bits = 7 if dtype == torch.bfloat16 else 10
            mag = torch.randint(0, 1 << frac_bits, (D,), generator=gen, dtype=torch.int32)
            sign = torch.randint(0, 2, (D,), generator=gen, dtype=torch.int32) << 15
            x[4] = (sign | mag).to(torch.int16).view(dtype)  # exponent field 0: zeros and subnormals
            wq, _ = synth.norm_weights(D, dtype, seed=9)
            ones = torch.ones(D, dtype=dtype)
            ident = oracle.rope_table(10000.0, 1, D, lib=lib)[0]  # p = 0: no rotation
            for w in (ones, wq):
                want = _rms_norm_torch(x, w, eps)
                got = torch.stack([oracle.rmsnorm_rope_row(x[i], w, eps, ident, lib=lib) for i in range(x.shape[0])])
                ud = ulp_diff(got, want)
                # torch's fp32 reduction order may flip an isolated value by one ulp
                assert int(ud.max()) <= 1, (dtype, D, int(ud.max()))
                assert int((ud > 0).sum()) <= max(2, x.numel() // 2000), (dtype, D, int((ud > 0).sum()))


def check_rmsnorm_closed_forms(lib):
    eps = 1e-6
    D = 64
    ident = oracle.rope_table(10000.0, 1, D, lib=lib)[0]
    for dtype in (torch.bfloat16, torch.float16):
        ones = torch.ones(D, dtype=dtype)
        for c in (3.0, -0.5, 1e-3, 2e-4):
            x = torch.full((D,), c, dtype=dtype)
            cx = float(x[0])
            # mean(x^2) = c^2 exactly; y = c / sqrt(c^2 + eps), one rounding to the 16-bit type
            exact = cx / math.sqrt(cx * cx + eps)
            got = oracle.rmsnorm_rope_row(x, ones, eps, ident, lib=lib)
            want = torch.tensor([exact], dtype=torch.float64).to(dtype)
            assert int(ulp_diff(got, want.expand(D)).max()) <= 1, (dtype, c, got[0], exact)
        # weight 1, no rotation: the output has rms 1 up to 16-bit rounding
        gen = synth.make_generator(21, "cpu")
        x = torch.randn((D,), generator=gen).to(dtype)
        got = oracle.rmsnorm_rope_row(x, ones, eps, ident, lib=lib).double()
        assert abs(float(got.pow(2).mean().sqrt()) - 1.0) < 2 ** -7


def check_rmsnorm_large_magnitudes(lib):
    """Rows whose squares overflow fp32 (bf16 reaches 3.4e38; any |x| >= 2^64 has
    a square beyond fp32).  The fused path's RMSNorm is fp32 (flashinfer PR #6332,
    "Assumptions / Operator math"); its mean of squares is the exact mean rounded
    once to fp32.  Fixed by the mathematics, independently of that code:
      * RMSNorm is invariant under x -> 2^k x while the mean stays in fp32's normal
        range and far above eps (the scaling is exact at every step), so rows of
        rms ~2^6 scaled by up to 2^57 -- single squares up to ~2^130 -- give the
        same bits as the unscaled row, whose values torch's rms_norm pins;
      * a row (c, 0, ..., 0) normalises to sqrt(D) at element 0 whatever c, while
        c^2/D fits fp32;
      * once the mean itself exceeds fp32 it is +inf, 1/sqrt(inf) = 0 and the row
        is all zeros -- what torch's fp32 rms_norm returns for such rows too."""
    eps, D = 1e-6, 128
    dtype = torch.bfloat16
    tab = oracle.rope_table(10000.0, 40, D, lib=lib)
    wq, _ = synth.norm_weights(D, dtype, seed=31)
    gen = synth.make_generator(44, "cpu")
    for trial in range(6):
        x = (torch.randn((D,), generator=gen) * 64.0).to(dtype)
        for p in (0, 7, 39):
            for style in oracle.ROPE_STYLES:
                base = oracle.rmsnorm_rope_row(x, wq, eps, tab[p], lib=lib, style=style)
                for k in (1, 20, 40, 56, 57):
                    xs = x * (2.0 ** k)  # exact: a power of two, no bf16 overflow (|x| < 2^66)
                    assert torch.equal((xs.float() / 2.0 ** k).to(dtype).view(torch.int16), x.view(torch.int16))
                    got = oracle.rmsnorm_rope_row(xs, wq, eps, tab[p], lib=lib, style=style)
                    assert torch.equal(got.view(torch.int16), base.view(torch.int16)), (trial, p, style, k)
    ones = torch.ones(D, dtype=dtype)
    ident = tab[0]
    spike_ref = None
    for e in (10, 40, 64, 67):  # c^2 / D = 2^(2e - 7) <= 2^127
        x = torch.zeros(D, dtype=dtype)
        x[0] = 2.0 ** e
        got = oracle.rmsnorm_rope_row(x, ones, eps, ident, lib=lib)
        assert torch.all(got[1:].float() == 0), e
        assert abs(float(got[0]) - math.sqrt(D)) <= math.sqrt(D) * 2 ** -8, (e, float(got[0]))
        spike_ref = got if spike_ref is None else spike_ref
        assert torch.equal(got.view(torch.int16), spike_ref.view(torch.int16)), e
    # the largest constant whose square fits fp32: mean = c^2, y = c / sqrt(c^2) = 1
    c = float(torch.tensor(2.0 ** 63 * 255 / 128, dtype=dtype))
    x = torch.full((D,), c, dtype=dtype)
    got = oracle.rmsnorm_rope_row(x, ones, eps, ident, lib=lib)
    assert torch.all(got.float() == 1.0), got[:4]
    # means beyond fp32: zeros, as torch's fp32 rms_norm gives
    bf16_max = torch.tensor(0x7F7F, dtype=torch.int16).view(torch.bfloat16).item()
    rows = [torch.full((D,), v, dtype=dtype) for v in (2.0 ** 64, -(2.0 ** 70), 2.0 ** 100, bf16_max)]
    spike = torch.zeros(D, dtype=dtype)
    spike[5] = 2.0 ** 68  # c^2 / D = 2^129
    rows.append(spike)
    for x in rows:
        for w in (ones, wq):
            got = oracle.rmsnorm_rope_row(x, w, eps, ident, lib=lib)
            assert torch.all(got.float() == 0), (float(x.abs().max()), got[:4])
            want = _rms_norm_torch(x.unsqueeze(0), w, eps)[0]
            assert torch.all(want.float() == 0)
            for style in oracle.ROPE_STYLES:
                rot = oracle.rmsnorm_rope_row(x, w, eps, tab[9], lib=lib, style=style)
                assert torch.all(rot.float() == 0), style


def check_rmsnorm_non_finite_rows(lib):
    """The reading for infinite and NaN inputs, which the pages do not address,
    taken from IEEE fp32 arithmetic at each step of the fp32 RMSNorm: a NaN makes
    the mean NaN, so the whole row is NaN; an infinite element (no NaN) makes the
    mean +inf and 1/sqrt(+inf) = 0, so every finite element normalises to zero
    and the infinite one to inf * 0 = NaN, which the rotation then also gives to
    its partner (the pair's other element)."""
    eps, D, p = 1e-6, 64, 5
    tab = oracle.rope_table(10000.0, 8, D, lib=lib)
    gen = synth.make_generator(45, "cpu")
    for dtype in (torch.bfloat16, torch.float16):
        w, _ = synth.norm_weights(D, dtype, seed=32)
        for i in (0, 1, 17, 40, 63):
            base = torch.randn((D,), generator=gen).to(dtype)
            x = base.clone()
            x[i] = float("nan")
            for style in oracle.ROPE_STYLES:
                got = oracle.rmsnorm_rope_row(x, w, eps, tab[p], lib=lib, style=style)
                assert torch.all(torch.isnan(got.float())), (dtype, i, style)
            for inf in (float("inf"), float("-inf")):
                x = base.clone()
                x[i] = inf
                for style in oracle.ROPE_STYLES:
                    partner = i ^ 1 if style == "interleaved" else (i + D // 2) % D
                    got = oracle.rmsnorm_rope_row(x, w, eps, tab[p], lib=lib, style=style).float()
                    nan = torch.isnan(got)
                    assert bool(nan[i]) and bool(nan[partner]) and int(nan.sum()) == 2, (dtype, i, style)
                    rest = torch.ones(D, dtype=torch.bool)
                    rest[[i, partner]] = False
                    assert torch.all(got[rest] == 0), (dtype, i, style)
                x[(i + 3) % D] = float("nan")
                got = oracle.rmsnorm_rope_row(x, w, eps, tab[p], lib=lib).float()
                assert torch.all(torch.isnan(got)), (dtype, i)


def _rotate_complex(z: torch.Tensor, angles: torch.Tensor) -> torch.Tensor:
    """Interleaved RoPE as multiplication of (z[2i] + j z[2i+1]) by exp(j angle_i), complex128."""
    zc = torch.view_as_complex(z.double().reshape(-1, 2).contiguous())
    out = zc * torch.polar(torch.ones_like(angles), angles)
    return torch.view_as_real(out).reshape(-1)


def check_rope_vs_complex(lib):
    eps = 1e-6
    theta = 10000.0
    for dtype in (torch.bfloat16, torch.float16):
        for D in (64, 128):
            S = 300
            tab = oracle.rope_table(theta, S, D, lib=lib)
            ident = tab[0]
            gen = synth.make_generator(33, "cpu")
            wq, _ = synth.norm_weights(D, dtype, seed=2)
            worst = 0
            for p in (1, 2, 17, 123, 299):
                x = torch.randn((D,), generator=gen).to(dtype)
                z = oracle.rmsnorm_rope_row(x, wq, eps, ident, lib=lib)  # normalised + scaled, unrotated
                got = oracle.rmsnorm_rope_row(x, wq, eps, tab[p], lib=lib)
                angles = torch.tensor([p * theta ** (-2.0 * i / D) for i in range(D // 2)], dtype=torch.float64)
                want = _rotate_complex(z, angles)
                err = (got.double() - want).abs()
                # one rounding of the output plus the fp32 table rounding
                bound = want.abs() * 2.0 ** (-7 if dtype == torch.bfloat16 else -10) + 2e-6 * z.double().abs().max()
                assert torch.all(err <= bound + 1e-12), (dtype, D, p, float((err - bound).max()))
                worst = max(worst, int((err > 0).sum()))
                # rotation keeps each pair's length
                n_in = z.double().reshape(-1, 2).pow(2).sum(-1).sqrt()
                n_out = got.double().reshape(-1, 2).pow(2).sum(-1).sqrt()
                rel = 2.0 ** (-6 if dtype == torch.bfloat16 else -9)
                assert torch.all((n_in - n_out).abs() <= rel * n_in + 1e-6), (dtype, D, p)


def check_fused_scatter_composition(lib):
    """The fused scatter equals the plain scatter followed by the row operation at
    target row index p (global position), so the two oracle entry points agree."""
    P, B, Sl, H, D = 3, 2, 5, 6, 64
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=4, layout="fused")
    wq, _ = synth.norm_weights(D, dtype, seed=4)
    tab = oracle.rope_table(10000.0, P * Sl, D, lib=lib)
    fused = oracle.scatter_norm_rope(d["q"], P, wq, 1e-6, tab, lib=lib)
    plain = oracle.scatter(d["q"], P, lib=lib)
    for g in range(P):
        for b in range(B):
            for p in range(P * Sl):
                for h in range(H // P):
                    row = oracle.rmsnorm_rope_row(plain[g][b, p, h], wq, 1e-6, tab[p], lib=lib)
                    assert torch.equal(row.view(torch.int16), fused[g][b, p, h].view(torch.int16)), (g, b, p, h)


# ----------------------------------------------------------------------------
# Half-split (NeoX) RoPE and the fused receive layout
# ----------------------------------------------------------------------------

def _neox_to_interleaved(v: torch.Tensor) -> torch.Tensor:
    """Reorder a head row so that half-split pair (i, i + D/2) sits at (2i, 2i+1)."""
    h = v.shape[-1] // 2
    return torch.stack([v[..., :h], v[..., h:]], dim=-1).reshape(v.shape).contiguous()


def _interleaved_to_neox(v: torch.Tensor) -> torch.Tensor:
    h = v.shape[-1] // 2
    pairs = v.reshape(*v.shape[:-1], h, 2)
    return torch.cat([pairs[..., 0], pairs[..., 1]], dim=-1).contiguous()


def check_neox_vs_interleaved_reordering(lib):
    """The half-split rotation of a row equals the interleaved rotation of the row
    reordered so pair (i, i + D/2) sits at (2i, 2i+1), reordered back: RMSNorm does
    not depend on the order (the double sum of squares of 16-bit values is exact
    here) and both forms rotate pair i by table entry i."""
    eps = 1e-6
    for dtype in (torch.bfloat16, torch.float16):
        for D in (32, 64, 128, 256):
            tab = oracle.rope_table(10000.0, 64, D, lib=lib)
            w, _ = synth.norm_weights(D, dtype, seed=D + 1)
            gen = synth.make_generator(D + 2, "cpu")
            for p in (0, 1, 5, 63):
                x = torch.randn((D,), generator=gen).to(dtype)
                got = oracle.rmsnorm_rope_row(x, w, eps, tab[p], lib=lib, style="neox")
                inter = oracle.rmsnorm_rope_row(_neox_to_interleaved(x), _neox_to_interleaved(w), eps, tab[p],
                                                lib=lib)
                want = _interleaved_to_neox(inter)
                assert torch.equal(got.view(torch.int16), want.view(torch.int16)), (dtype, D, p)


def check_neox_rotate_half_textbook(lib):
    """Half-split RoPE in its textbook form, z * [cos, cos] + rotate_half(z) * [sin, sin]
    with rotate_half(z) = [-z2, z1], evaluated in numpy float32 (one rounding per
    product and per sum, as the step-by-step fp32 definition) and cast to 16 bits
    by torch, from the oracle's own unrotated row (table row p = 0)."""
    eps = 1e-6
    for dtype in (torch.bfloat16, torch.float16):
        for D in (64, 128):
            tab = oracle.rope_table(10000.0, 40, D, lib=lib)
            _, w = synth.norm_weights(D, dtype, seed=3 * D)
            gen = synth.make_generator(3 * D + 1, "cpu")
            for p in (1, 7, 39):
                x = torch.randn((D,), generator=gen).to(dtype)
                z = oracle.rmsnorm_rope_row(x, w, eps, tab[0], lib=lib, style="neox").float().numpy()
                c = tab[p][:, 0].numpy().astype(np.float32)
                s_ = tab[p][:, 1].numpy().astype(np.float32)
                cos2 = np.concatenate([c, c])
                sin2 = np.concatenate([s_, s_])
                h = D // 2
                rot = np.concatenate([-z[h:], z[:h]]).astype(np.float32)
                want32 = (z * cos2).astype(np.float32) + (rot * sin2).astype(np.float32)
                want = torch.from_numpy(want32.astype(np.float32)).to(dtype)
                got = oracle.rmsnorm_rope_row(x, w, eps, tab[p], lib=lib, style="neox")
                assert torch.equal(got.view(torch.int16), want.view(torch.int16)), (dtype, D, p)


def check_fused_scatter_neox_composition(lib):
    """The half-split fused scatter equals the plain scatter followed by the
    half-split row operation at the global position."""
    P, B, Sl, H, D = 2, 1, 4, 4, 32
    dtype = torch.float16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=8)
    _, wk = synth.norm_weights(D, dtype, seed=8)
    tab = oracle.rope_table(500.0, P * Sl, D, lib=lib)
    fused = oracle.scatter_norm_rope(d["k"], P, wk, 1e-6, tab, lib=lib, style="neox")
    plain = oracle.scatter(d["k"], P, lib=lib)
    for g in range(P):
        for p in range(P * Sl):
            for h in range(H // P):
                row = oracle.rmsnorm_rope_row(plain[g][0, p, h], wk, 1e-6, tab[p], lib=lib, style="neox")
                assert torch.equal(row.view(torch.int16), fused[g][0, p, h].view(torch.int16)), (g, p, h)


def check_fused_payload_brute_force(lib):
    """Fused receive layout by index enumeration on distinct ids:
    payload_g[b, r*Sl + t, h, x*D + d] = S^x_r[b, t, g*Hl + h, d] for x = Q, K, V."""
    P, B, Sl, H, D = 2, 2, 3, 4, 8
    srcs = synth.unique_id_shards(3 * P, B, Sl, H, D)
    q, k, v = srcs[0:P], srcs[P:2 * P], srcs[2 * P:3 * P]
    pay = oracle.fused_payload(oracle.scatter(q, P, lib=lib), oracle.scatter(k, P, lib=lib),
                               oracle.scatter(v, P, lib=lib))
    Hl = H // P
    seen = 0
    for g in range(P):
        assert tuple(pay[g].shape) == (B, P * Sl, Hl, 3 * D)
        for b in range(B):
            for r in range(P):
                for t in range(Sl):
                    for h in range(Hl):
                        for x, src in enumerate((q, k, v)):
                            for dd in range(D):
                                assert int(pay[g][b, r * Sl + t, h, x * D + dd]) == int(src[r][b, t, g * Hl + h, dd])
                                seen += 1
    assert seen == 3 * P * B * Sl * H * D


def check_head_chunks_compose_to_the_scatter(lib):
    """Head-chunk scatters of a partition of [0, Hl) into one set of targets equal
    the whole scatter, and a single chunk leaves the other heads untouched."""
    P, B, Sl, H, D = 2, 2, 3, 8, 8
    srcs = synth.unique_id_shards(P, B, Sl, H, D)
    whole = oracle.scatter(srcs, P, lib=lib)
    Hl = H // P
    fill = [torch.full_like(t, -1) for t in whole]
    acc = fill
    for h0, h1 in ((0, 1), (1, 3), (3, Hl)):
        acc = oracle.scatter_heads_chunk(srcs, P, h0, h1, acc)
    for g in range(P):
        assert torch.equal(acc[g], whole[g]), g
    one = oracle.scatter_heads_chunk(srcs, P, 1, 3, fill)
    for g in range(P):
        assert torch.equal(one[g][:, :, 1:3], whole[g][:, :, 1:3])
        assert bool((one[g][:, :, :1] == -1).all()) and bool((one[g][:, :, 3:] == -1).all())


def check_exchange_chunks_is_the_scatter_of_single_head_bands(lib):
    """The chunk exchange equals the Ulysses scatter with one head per band and the
    chunk as the head row (sequence length 1): the same all-to-all."""
    P = 3
    gen = torch.Generator().manual_seed(5)
    payloads = [torch.randint(0, 256, (P, 32), generator=gen, dtype=torch.uint8) for _ in range(P)]
    ex = oracle.exchange_chunks(payloads, P)
    as_shards = [x.view(1, 1, P, 32) for x in payloads]  # [B=1, Sl=1, H=P, D=32]
    sc = oracle.scatter(as_shards, P, lib=lib)  # [1, P, 1, 32] per group
    for g in range(P):
        assert torch.equal(ex[g], sc[g].view(P, 32)), g


# ----------------------------------------------------------------------------
# QKV projection
# ----------------------------------------------------------------------------

def check_projection_vs_fp64_matmul(lib):
    """The projection equals a float64 library matmul of the same 16-bit values
    rounded once to the 16-bit type (torch's round-to-nearest-even cast)."""
    for dtype in (torch.bfloat16, torch.float16):
        gen = synth.make_generator(31, "cpu")
        for M, N, K in ((7, 40, 64), (33, 96, 320)):
            x = torch.randn((M, K), generator=gen).to(dtype)
            w = (torch.randn((N, K), generator=gen) / K ** 0.5).to(dtype)
            got = oracle.project(x, w, lib=lib)
            want = (x.double() @ w.double().T).to(dtype)
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), (dtype, M, N, K)
            # a column range of one row agrees with the whole projection
            part = oracle.project_row_range(x[M // 2], w, 5, 29, lib=lib)
            assert torch.equal(part.view(torch.int16), got[M // 2, 5:29].view(torch.int16))


def check_projection_closed_forms(lib):
    """Identity and permutation weights reproduce / permute the input exactly,
    and a weight row of twos doubles the row sum (a power-of-two scale)."""
    K = 48
    x = (torch.arange(6 * K, dtype=torch.float32).view(6, K) / 7.0 - 17.0).to(torch.bfloat16)
    eye = torch.eye(K).to(torch.bfloat16)
    assert torch.equal(oracle.project(x, eye, lib=lib).view(torch.int16), x.view(torch.int16))
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(3))
    got = oracle.project(x, eye[perm], lib=lib)
    assert torch.equal(got.view(torch.int16), x[:, perm].view(torch.int16))
    xs = torch.tensor([[1.0, 2.0, -0.5, 0.25]], dtype=torch.bfloat16)
    twos = torch.full((1, 4), 2.0, dtype=torch.bfloat16)
    assert float(oracle.project(xs, twos, lib=lib)[0, 0]) == 5.5


def check_project_qkv_blocks(lib):
    """Q, K, V come from feature blocks [0, HD), [HD, 2HD), [2HD, 3HD) of the
    weight, head h from features [h*D, (h+1)*D) of its block."""
    B, Sl, H, D, K = 2, 3, 2, 4, 8
    gen = torch.Generator().manual_seed(4)
    x = [torch.randn((B, Sl, K), generator=gen).to(torch.bfloat16)]
    w = torch.randn((3 * H * D, K), generator=gen).to(torch.bfloat16)
    out = oracle.project_qkv(x, w, H, D, lib=lib)
    full = oracle.project(x[0].reshape(B * Sl, K), w, lib=lib)
    for i, key in enumerate("qkv"):
        for h in range(H):
            want = full[:, i * H * D + h * D:i * H * D + (h + 1) * D].reshape(B, Sl, D)
            assert torch.equal(out[key][0][:, :, h].view(torch.int16), want.view(torch.int16)), (key, h)


ALL_CHECKS = [
    check_codec_decode,
    check_codec_encode,
    check_relayout_golden,
    check_relayout_allgather,
    check_relayout_invariants,
    check_rope_table_textbook,
    check_rmsnorm_vs_torch,
    check_rmsnorm_closed_forms,
    check_rmsnorm_large_magnitudes,
    check_rmsnorm_non_finite_rows,
    check_rope_vs_complex,
    check_fused_scatter_composition,
    check_neox_vs_interleaved_reordering,
    check_neox_rotate_half_textbook,
    check_fused_scatter_neox_composition,
    check_fused_payload_brute_force,
    check_head_chunks_compose_to_the_scatter,
    check_exchange_chunks_is_the_scatter_of_single_head_bands,
    check_projection_vs_fp64_matmul,
    check_projection_closed_forms,
    check_project_qkv_blocks,
]
