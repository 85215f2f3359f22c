"""The allocation-free scatter entry point (tf_ulysses_scatter_qkv_noalloc).

It serves callers that cannot allocate device memory: code working inside a
device-memory budget reserved up front, where another allocator already owns
the free memory, and latency-bound loops that cannot take the device
synchronisation of cudaMalloc/cudaFree.  Its cos/sin table lives in a fixed
device array of the library instead of an allocation, and stays there for the
next call of the same (theta, rows, D).

Checked here through the C ABI, call after call: the first call on its shape
builds the table in the fixed array; the next one with new data reuses it; a
call of another shape and RoPE base rebuilds it; a shorter sequence with the
first base reuses the longer table built before it.  A table built on one
stream is waited for by a reuse on another.  Every call's targets equal
those of the existing caller-owned-target entry point bit for bit (both read
the same table bits through the same kernels) and the oracle's under the fused
rule; no allocation callback fires and the library's allocation count does not
move; a size beyond the fixed capacity is rejected.  This file is collected
last so that a run stopping at its first failure has already run every other
test.
"""
import pytest
import torch

import oracle
from parity_util import assert_fused_ok, bits_equal
from ulysses_sequence_attention_tf_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tf():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ulysses_sequence_attention_tf_gb300 import binding, build
    build.build()
    binding.lib()
    binding.use_torch_allocator(True)
    return binding


def _targets(P, B, S, Hl, D, dtype, fill):
    return [torch.full((B, S, Hl, D), fill, dtype=dtype, device="cuda") for _ in range(P)]


class _CountingAllocator:
    """Allocation callbacks that count calls and refuse to allocate."""

    def __init__(self, tf):
        self.calls = 0
        self.fns = (tf.ALLOC_FN(self._alloc), tf.FREE_FN(self._free))

    def _alloc(self, nbytes, stream, ctx):
        self.calls += 1
        return None

    def _free(self, ptr, nbytes, stream, ctx):
        self.calls += 1


CALLS = [
    # P, B, S, H, D, dtype, theta, layout, what the fixed table does
    (4, 1, 4096, 24, 128, torch.bfloat16, 10000.0, "fused", "built"),
    (4, 1, 4096, 24, 128, torch.bfloat16, 10000.0, "v_strided", "reused"),
    (2, 2, 998, 16, 64, torch.float16, 500000.0, "v_strided", "rebuilt"),
    (2, 1, 2048, 8, 128, torch.bfloat16, 10000.0, "contiguous", "rebuilt"),
    (4, 1, 1024, 8, 128, torch.bfloat16, 10000.0, "contiguous", "reused (a longer table)"),
]


def test_noalloc_matches_existing_entry_point_call_after_call(tf):
    counter = _CountingAllocator(tf)
    for i, (P, B, S, H, D, dtype, theta, layout, _) in enumerate(CALLS):
        Sl, Hl = S // P, H // P
        d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=40 + i, layout=layout)
        g = synth.move(d, "cuda")
        wq, wk = synth.norm_weights(D, dtype, seed=40 + i)
        kw = dict(norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=1e-6, theta=theta)
        ref = [_targets(P, B, S, Hl, D, dtype, 0.0) for _ in range(3)]
        tf.scatter_qkv_into(g["q"], g["k"], g["v"], *ref, **kw)
        out = [_targets(P, B, S, Hl, D, dtype, 9.0) for _ in range(3)]
        torch.cuda.synchronize()
        allocs = tf.alloc_count()
        tf.lib().tf_ulysses_set_allocator(counter.fns[0], counter.fns[1], None)
        try:
            tf.scatter_qkv_noalloc(g["q"], g["k"], g["v"], *out, **kw)
            torch.cuda.synchronize()
        finally:
            tf.use_torch_allocator(True)
        assert counter.calls == 0, "the allocation-free entry point called the allocator"
        assert tf.alloc_count() == allocs, "the allocation-free entry point allocated"
        table = oracle.rope_table(theta, S, D)
        for x, key in enumerate("qkv"):
            want = (oracle.scatter_norm_rope(d[key], P, wq if key == "q" else wk, 1e-6, table) if key != "v"
                    else oracle.scatter(d[key], P))
            for gi in range(P):
                assert bits_equal(out[x][gi], ref[x][gi]), (i, key, gi)
                if key == "v":
                    assert bits_equal(out[x][gi].cpu(), want[gi]), (i, gi)
                else:
                    assert_fused_ok(out[x][gi], want[gi])


@pytest.mark.parametrize("rope", ["interleaved", "neox"])
def test_noalloc_qk_only(tf, rope):
    """Q and K alone through the allocation-free entry point (the Q/K-only launch
    with its (cos, sin) ring): bit for bit what scatter_qkv_into gives, no
    allocation."""
    P, B, S, H, D, dtype = 4, 1, 2048, 16, 128, torch.bfloat16
    Sl, Hl = S // P, H // P
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=77, layout="v_strided", with_v=False)
    g = synth.move(d, "cuda")
    wq, wk = synth.norm_weights(D, dtype, seed=77)
    kw = dict(norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=1e-6, theta=10000.0, rope=rope)
    ref = [_targets(P, B, S, Hl, D, dtype, 0.0) for _ in range(2)]
    tf.scatter_qkv_into(g["q"], g["k"], None, ref[0], ref[1], None, **kw)
    out = [_targets(P, B, S, Hl, D, dtype, 9.0) for _ in range(2)]
    torch.cuda.synchronize()
    allocs = tf.alloc_count()
    counter = _CountingAllocator(tf)
    tf.lib().tf_ulysses_set_allocator(counter.fns[0], counter.fns[1], None)
    try:
        tf.scatter_qkv_noalloc(g["q"], g["k"], None, out[0], out[1], None, **kw)
        torch.cuda.synchronize()
    finally:
        tf.use_torch_allocator(True)
    assert counter.calls == 0 and tf.alloc_count() == allocs
    for x in range(2):
        for gi in range(P):
            assert bits_equal(out[x][gi], ref[x][gi]), (rope, x, gi)


def test_noalloc_rejects_sizes_beyond_the_fixed_scratch(tf):
    P, B, Sl, H, D = 2, 1, 16385, 4, 128  # P * S_local * D = 4,194,560 > 4 Mi floats
    dtype = torch.bfloat16
    g = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=1, device="cuda", with_k=False, with_v=False)
    wq, wk = synth.norm_weights(D, dtype, device="cuda")
    out = _targets(P, B, P * Sl, H // P, D, dtype, 5.0)
    with pytest.raises(tf.TfUlyssesError) as ei:
        tf.scatter_qkv_noalloc(g["q"], None, None, out, norm_rope=True, q_weight=wq, k_weight=wk)
    assert ei.value.status == tf.TF_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert all(torch.all(o == 5.0) for o in out), "a rejected call wrote its targets"
    # with a caller table no scratch is needed, so the same size is accepted
    table = torch.zeros((P * Sl, D // 2, 2), dtype=torch.float32, device="cuda")
    table[..., 0] = 1.0
    tf.scatter_qkv_noalloc(g["q"], None, None, out, norm_rope=True, q_weight=wq, k_weight=wk, cos_sin=table)
    ref = _targets(P, B, P * Sl, H // P, D, dtype, 0.0)
    tf.scatter_qkv_into(g["q"], None, None, ref, norm_rope=True, q_weight=wq, k_weight=wk, cos_sin=table)
    for gi in range(P):
        assert bits_equal(out[gi], ref[gi])


def test_noalloc_reuse_on_another_stream_waits_for_the_build(tf):
    """A call that rebuilds the fixed table on one stream, then a call of the same
    (theta, rows, D) on a second stream with no synchronisation between them: the
    second waits on the end of the build (the event recorded after it), so both
    give the targets of scatter_qkv_into bit for bit."""
    P, B, S, H, D = 4, 1, 8192, 16, 128
    Sl, Hl = S // P, H // P
    dtype = torch.bfloat16
    theta = 31337.0  # a base no other call of this file uses: the first call rebuilds
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=60, layout="v_strided", device="cuda")
    wq, wk = synth.norm_weights(D, dtype, seed=60, device="cuda")
    kw = dict(norm_rope=True, q_weight=wq, k_weight=wk, eps=1e-6, theta=theta)
    ref = [_targets(P, B, S, Hl, D, dtype, 0.0) for _ in range(3)]
    tf.scatter_qkv_into(d["q"], d["k"], d["v"], *ref, **kw)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = [[_targets(P, B, S, Hl, D, dtype, 9.0) for _ in range(3)] for _ in range(2)]
    torch.cuda.synchronize()
    tf.scatter_qkv_noalloc(d["q"], d["k"], d["v"], *outs[0], stream=s1, **kw)
    tf.scatter_qkv_noalloc(d["q"], d["k"], d["v"], *outs[1], stream=s2, **kw)
    torch.cuda.synchronize()
    for o in outs:
        for x in range(3):
            for gi in range(P):
                assert bits_equal(o[x][gi], ref[x][gi]), (x, gi)
