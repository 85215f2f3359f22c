"""The comparison baselines of the configuration sweep move exactly the bytes of
the relayout they stand beside (CPU, no GPU): the cudaMemcpy2DAsync plan
(sweep._pieces, simulated byte by byte), the per-(shard, group) strided copies
and the stack + permute form, each against the oracle's scatter and gather."""
import numpy as np
import pytest
import torch

import oracle
from ulysses_sequence_attention_tf_gb300 import sweep

SHAPES = [(2, 1, 3, 2, 8), (4, 2, 5, 3, 16), (3, 2, 2, 1, 8), (8, 1, 2, 2, 8)]


def _apply_plan(plan, srcs, dsts, Sl, width, direction):
    for r, g, so, sp, do, dp in plan:
        s_buf, d_buf = (srcs[r], dsts[g]) if direction == "scatter" else (srcs[g], dsts[r])
        sb = s_buf.numpy().view(np.uint8).reshape(-1)
        db = d_buf.numpy().view(np.uint8).reshape(-1)
        for row in range(Sl):
            assert so + row * sp + width <= sb.size and do + row * dp + width <= db.size
            db[do + row * dp:do + row * dp + width] = sb[so + row * sp:so + row * sp + width]


@pytest.mark.parametrize("P,B,Sl,Hl,D", SHAPES)
def test_scatter_baselines_match_oracle(P, B, Sl, Hl, D):
    H, S = P * Hl, P * Sl
    gen = torch.Generator().manual_seed(P * 100 + D)
    src = [torch.randint(-30000, 30000, (B, Sl, H, D), generator=gen, dtype=torch.int16) for _ in range(P)]
    want = oracle.scatter(src, P)
    dst = [torch.zeros((B, S, Hl, D), dtype=torch.int16) for _ in range(P)]
    _apply_plan(sweep._pieces(P, B, Sl, Hl, D, 2, "scatter"), src, dst, Sl, Hl * D * 2, "scatter")
    assert all(torch.equal(dst[g], want[g]) for g in range(P))
    dst2 = [torch.zeros((B, S, Hl, D), dtype=torch.int16) for _ in range(P)]
    for r in range(P):
        for g in range(P):
            dst2[g][:, r * Sl:(r + 1) * Sl].copy_(src[r][:, :, g * Hl:(g + 1) * Hl])
    assert all(torch.equal(dst2[g], want[g]) for g in range(P))
    perm = torch.stack(src).view(P, B, Sl, P, Hl, D).permute(3, 1, 0, 2, 4, 5).contiguous()
    assert all(torch.equal(perm[g].reshape(B, S, Hl, D), want[g]) for g in range(P))


@pytest.mark.parametrize("P,B,Sl,Hl,D", SHAPES)
def test_gather_baselines_match_oracle(P, B, Sl, Hl, D):
    H, S = P * Hl, P * Sl
    gen = torch.Generator().manual_seed(P * 100 + D + 1)
    attn = [torch.randint(-30000, 30000, (B, S, Hl, D), generator=gen, dtype=torch.int16) for _ in range(P)]
    want = oracle.gather(attn, P)
    out = [torch.zeros((B, Sl, H, D), dtype=torch.int16) for _ in range(P)]
    _apply_plan(sweep._pieces(P, B, Sl, Hl, D, 2, "gather"), attn, out, Sl, Hl * D * 2, "gather")
    assert all(torch.equal(out[r], want[r]) for r in range(P))
    out2 = [torch.zeros((B, Sl, H, D), dtype=torch.int16) for _ in range(P)]
    for r in range(P):
        for g in range(P):
            out2[r][:, :, g * Hl:(g + 1) * Hl].copy_(attn[g][:, r * Sl:(r + 1) * Sl])
    assert all(torch.equal(out2[r], want[r]) for r in range(P))
    perm = torch.stack(attn).view(P, B, P, Sl, Hl, D).permute(2, 1, 3, 0, 4, 5).contiguous()
    assert all(torch.equal(perm[r].reshape(B, Sl, H, D), want[r]) for r in range(P))
