"""Comparison helpers for the GPU parity tests (no method arithmetic here)."""
from __future__ import annotations

import torch

# Tolerance of the fused RMSNorm + RoPE path: max-abs 1e-2 for bf16 and 2e-3 for
# fp16; an element above it passes only if it differs from the oracle by exactly
# one unit in the last place of the output type (an isolated rounding flip, the
# classification of flashinfer PR #6332, "Assumptions / Tolerance").
FUSED_ATOL = {torch.bfloat16: 1e-2, torch.float16: 2e-3}


def ordered16(bits: torch.Tensor) -> torch.Tensor:
    b = bits.to(torch.int32) & 0xFFFF
    mag = b & 0x7FFF
    return torch.where(b >= 0x8000, -mag, mag)


def ulp_diff(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    return (ordered16(a.view(torch.int16)) - ordered16(b.view(torch.int16))).abs()


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    if a.shape != b.shape:
        return False
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def fused_compare(got: torch.Tensor, want: torch.Tensor) -> dict:
    """Classify the differences of a fused (normalised + rotated) output."""
    got, want = got.cpu(), want.cpu()
    assert got.shape == want.shape and got.dtype == want.dtype
    tol = FUSED_ATOL[got.dtype]
    diff = (got.float() - want.float()).abs()
    ulp = ulp_diff(got, want)
    over = diff > tol
    return dict(
        n=got.numel(),
        n_bit_diff=int((ulp > 0).sum()),
        max_abs=float(diff.max()) if got.numel() else 0.0,
        max_ulp=int(ulp.max()) if got.numel() else 0,
        n_over_tol=int(over.sum()),
        tol=tol,
        ok=bool((ulp[over] == 1).all()),
    )


def assert_projected_ok(got, want, min_identical=0.9):
    """Outputs of the projection path on N(0, 1) data (the tensor cores sum in fp32
    in their own order; the oracle rounds the exact sum once): flashinfer PR #6332
    ("Assumptions / Tolerance") checks against a step-by-step reference with
    atol = rtol = 1e-2, single-ulp differences classified apart.  Every element
    within atol + rtol*|want| or one ulp, and most elements bit-identical."""
    got, want = got.cpu(), want.cpu()
    diff = (got.float() - want.float()).abs()
    ulp = ulp_diff(got, want)
    ok = (diff <= 1e-2 + 1e-2 * want.float().abs()) | (ulp <= 1)
    assert bool(ok.all()), (float(diff.max()), int((~ok).sum()))
    same = float((ulp == 0).float().mean()) if got.numel() else 1.0
    assert same >= min_identical, same
    return same


def assert_fused_ok(got, want, max_flip_fraction=1e-5):
    st = fused_compare(got, want)
    assert st["ok"], st
    assert st["n_bit_diff"] <= max(2, int(st["n"] * max_flip_fraction)), st
    return st


def assert_fused_ok_nonfinite(got, want, max_flip_fraction=1e-5):
    """assert_fused_ok for outputs that may hold NaN: every NaN of the oracle must
    be a NaN in ``got`` and nothing else may be (a NaN's bits are not compared);
    the other elements follow assert_fused_ok."""
    got, want = got.cpu(), want.cpu()
    gn, wn = torch.isnan(got.float()), torch.isnan(want.float())
    assert torch.equal(gn, wn), ("NaN positions differ", int((gn & ~wn).sum()), int((wn & ~gn).sum()))
    keep = ~wn
    return assert_fused_ok(got[keep], want[keep], max_flip_fraction)
