"""CUDA-graph capture protocol and rotating target slots, through the C ABI
(flashinfer PR #6332 commit message, "Description", "CUDA graphs": a prepared
call allocates nothing, a size first seen inside a capture raises instead of
allocating, replays interleave with eager calls, outputs stay valid until their
slot is reused num_slots calls later).

Every captured call is checked after replays with fresh inputs against the
oracle (relayout bit-exact, fused rows within the tolerance of parity_util).
"""
import pytest
import torch

import oracle
from parity_util import assert_fused_ok, bits_equal
from ulysses_sequence_attention_tf_gb300 import synth

pytestmark = pytest.mark.gpu

EPS = 1e-6
THETA = 10000.0
P, B, Sl, H, D = 4, 1, 96, 8, 128
S, Hl = P * Sl, H // P
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


def _inputs(seed):
    d = synth.qkv_shards(P, B, Sl, H, D, DT, seed=seed)
    d["attn"] = synth.attn_outputs(P, B, S, Hl, D, DT, seed=seed)
    return d


def _static_inputs(seed):
    d = _inputs(seed)
    return {k: [t.cuda() for t in d[k]] for k in ("q", "k", "v", "attn")}


def _refill(static, seed):
    """Copy fresh host inputs into the captured input buffers; returns the host copy."""
    d = _inputs(seed)
    for k in ("q", "k", "v", "attn"):
        for dst, src in zip(static[k], d[k]):
            dst.copy_(src)
    return d


def _check_scatter(tq, tk, tv, d, wq, wk):
    table = oracle.rope_table(THETA, S, D)
    for key, tg, w in (("q", tq, wq), ("k", tk, wk)):
        want = oracle.scatter_norm_rope(d[key], P, w, EPS, table)
        for i in range(P):
            assert_fused_ok(tg[i], want[i])
    want_v = oracle.scatter(d["v"], P)
    for i in range(P):
        assert bits_equal(tv[i].cpu(), want_v[i])


def test_capture_replay_with_fresh_inputs_allocates_nothing(tf):
    wq, wk = synth.norm_weights(D, DT, seed=1)
    kw = dict(norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS, theta=THETA)
    x = _static_inputs(0)
    tf.scatter_qkv("cap_a", x["q"], x["k"], x["v"], **kw)  # prepare: entry + table
    tf.gather_out("cap_a_out", x["attn"])
    torch.cuda.synchronize()
    n_alloc, n_entries = tf.alloc_count(), tf.cache_entries()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        tq, tk, tv, done = tf.scatter_qkv("cap_a", x["q"], x["k"], x["v"], **kw)
        outs, _ = tf.gather_out("cap_a_out", x["attn"])
    assert tf.alloc_count() == n_alloc and tf.cache_entries() == n_entries
    assert done
    for seed in (11, 12, 13):
        d = _refill(x, seed)
        graph.replay()
        torch.cuda.synchronize()
        _check_scatter(tq, tk, tv, d, wq, wk)
        want = oracle.gather(d["attn"], P)
        for r in range(P):
            assert bits_equal(outs[r].cpu(), want[r])
    assert tf.alloc_count() == n_alloc


def test_first_use_inside_capture_raises_and_allocates_nothing(tf):
    x = _static_inputs(1)
    torch.cuda.synchronize()
    n_alloc, n_entries = tf.alloc_count(), tf.cache_entries()
    graph = torch.cuda.CUDAGraph()
    with pytest.raises(tf.TfUlyssesError) as err:
        with torch.cuda.graph(graph):
            tf.scatter_qkv("never_prepared", x["q"], x["k"], x["v"])
    assert err.value.status == tf.TF_ERR_UNSUPPORTED
    # a table first needed inside a capture is refused the same way
    wq, wk = synth.norm_weights(D, DT, seed=2, device="cuda")
    tf.scatter_qkv("prepared_plain", x["q"], x["k"], x["v"])  # entry exists, mode differs below
    torch.cuda.synchronize()
    n_alloc, n_entries = tf.alloc_count(), tf.cache_entries()
    outs = [[torch.empty((B, S, Hl, D), dtype=DT, device="cuda") for _ in range(P)] for _ in range(3)]
    torch.cuda.synchronize()
    graph2 = torch.cuda.CUDAGraph()
    with pytest.raises(tf.TfUlyssesError) as err2:
        with torch.cuda.graph(graph2):
            tf.scatter_qkv_into(x["q"], x["k"], x["v"], *outs, norm_rope=True, q_weight=wq, k_weight=wk,
                                theta=1234.5)
    assert err2.value.status == tf.TF_ERR_UNSUPPORTED
    assert tf.alloc_count() == n_alloc and tf.cache_entries() == n_entries
    # the library is still usable eagerly afterwards
    tq, _, _, _ = tf.scatter_qkv("prepared_plain", x["q"], x["k"], x["v"])
    torch.cuda.synchronize()
    want = oracle.scatter([t.cpu() for t in x["q"]], P)
    assert bits_equal(tq[0].cpu(), want[0])


def test_rotating_slots_keep_earlier_targets(tf):
    tf.set_slots("rot3", 3)
    seen, data = [], []
    for step in range(4):
        d = _inputs(20 + step)
        tq, tk, tv, _ = tf.scatter_qkv("rot3", [t.cuda() for t in d["q"]], [t.cuda() for t in d["k"]],
                                       [t.cuda() for t in d["v"]])
        seen.append((tq, tk, tv))
        data.append(d)
        torch.cuda.synchronize()
        # the targets of the previous num_slots - 1 calls are untouched
        for back in range(min(step + 1, 3)):
            tq_b, _, tv_b = seen[step - back]
            d_b = data[step - back]
            assert bits_equal(tq_b[1].cpu(), oracle.scatter(d_b["q"], P)[1]), (step, back)
            assert bits_equal(tv_b[2].cpu(), oracle.scatter(d_b["v"], P)[2]), (step, back)
    ptrs = [s[0][0].data_ptr() for s in seen]
    assert len(set(ptrs[:3])) == 3 and ptrs[3] == ptrs[0]
    with pytest.raises(tf.TfUlyssesError):
        tf.set_slots("rot3", 9)


def test_two_slots_captured_in_one_graph(tf):
    tf.set_slots("rot2", 2)
    x, y = _static_inputs(30), _static_inputs(31)
    tf.scatter_qkv("rot2", x["q"], x["k"], x["v"])  # prepare (writes slot 0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ax = tf.scatter_qkv("rot2", x["q"], x["k"], x["v"])  # slot 1
        ay = tf.scatter_qkv("rot2", y["q"], y["k"], y["v"])  # slot 0
    assert ax[0][0].data_ptr() != ay[0][0].data_ptr()
    for seed in (40, 41):
        dx, dy = _refill(x, seed), _refill(y, seed + 100)
        graph.replay()
        torch.cuda.synchronize()
        for a, d in ((ax, dx), (ay, dy)):
            for key, tg in zip("qkv", a[:3]):
                want = oracle.scatter(d[key], P)
                for i in range(P):
                    assert bits_equal(tg[i].cpu(), want[i]), (seed, key, i)


def test_replays_interleave_with_eager_calls(tf):
    x, z = _static_inputs(50), _static_inputs(51)
    dz = {k: [t.cpu() for t in z[k]] for k in z}
    tf.scatter_qkv("mix", x["q"], x["k"], x["v"])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        tq, _, _, _ = tf.scatter_qkv("mix", x["q"], x["k"], x["v"])
    for seed in (52, 53):
        d = _refill(x, seed)
        graph.replay()
        torch.cuda.synchronize()
        assert bits_equal(tq[3].cpu(), oracle.scatter(d["q"], P)[3])
        eq, _, _, _ = tf.scatter_qkv("mix", z["q"], z["k"], z["v"])  # same key, same slot, eager
        torch.cuda.synchronize()
        assert eq[3].data_ptr() == tq[3].data_ptr()
        assert bits_equal(eq[3].cpu(), oracle.scatter(dz["q"], P)[3])


def test_capture_head_chunks_and_exchange(tf):
    x = _static_inputs(60)
    outs = [torch.empty((B, S, Hl, D), dtype=DT, device="cuda") for _ in range(P)]
    pay = [torch.empty((P, 4096), dtype=torch.uint8, device="cuda") for _ in range(P)]
    got = [torch.empty_like(t) for t in pay]
    torch.cuda.synchronize()
    n_alloc = tf.alloc_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        tf.scatter_qkv_heads_into(x["q"], None, None, outs, h0=0, h1=1)
        tf.scatter_qkv_heads_into(x["q"], None, None, outs, h0=1, h1=Hl)
        tf.exchange_chunks(pay, got)
    assert tf.alloc_count() == n_alloc
    gen = torch.Generator().manual_seed(61)
    host_pay = [torch.randint(0, 256, (P, 4096), generator=gen, dtype=torch.uint8) for _ in range(P)]
    for dst, src in zip(pay, host_pay):
        dst.copy_(src)
    d = _refill(x, 62)
    graph.replay()
    torch.cuda.synchronize()
    want = oracle.scatter(d["q"], P)
    want_x = oracle.exchange_chunks(host_pay, P)
    for i in range(P):
        assert bits_equal(outs[i].cpu(), want[i])
        assert bits_equal(got[i].cpu(), want_x[i])


def test_device_status_clean(tf):
    torch.cuda.synchronize()
    assert tf.device_status(clear=False) == 0


def test_bounded_wait_gives_up_and_reports(tf):
    """Failure detection without a fault: a wait on an mbarrier that nothing
    arrives on gives up after its budget, the status word reports it, and the
    context keeps working."""
    torch.cuda.synchronize()
    assert tf.device_status(clear=True) == 0
    tf.selftest_wait(2_000_000)  # ~1 ms at 2 GHz
    torch.cuda.synchronize()
    assert tf.device_status(clear=True) == 2  # bit 1: the projection kernel's bounded waits
    assert tf.device_status(clear=False) == 0
    x = _static_inputs(70)
    tq, _, _, _ = tf.scatter_qkv("after_selftest", x["q"], x["k"], x["v"])
    torch.cuda.synchronize()
    assert bits_equal(tq[1].cpu(), oracle.scatter([t.cpu() for t in x["q"]], P)[1])
    with pytest.raises(tf.TfUlyssesError):
        tf.selftest_wait(0)
