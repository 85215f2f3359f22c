"""Host fault injection without a GPU fault.

* An allocator callback that runs out: the library's device memory comes from
  the caller's allocator (tf_ulysses_set_allocator).  A callback that returns
  NULL must turn into TF_ERR_OOM before any launch: no kernel runs, caller-owned
  targets keep their bytes, no cache entry appears for the failed key, and every
  allocation the library did get is handed back through the same callback.  Once
  allocations succeed again the same calls give the oracle's results.
* A cache entry evicted while its launch is still waiting behind other work on
  its stream (a sleep kernel): with the default allocator the evicting call
  returns at once and its stream waits for the entry's completion before the
  targets are freed; with a caller allocator, release() runs only after the
  entry's launch has completed (the host waits).
"""
import time

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
    binding.use_torch_allocator(True)


class BudgetAllocator:
    """torch-backed device allocations until `budget` runs out, then NULL."""

    def __init__(self, binding, budget):
        self.budget = budget
        self.allocs = 0
        self.frees = 0
        self.refs = (binding.ALLOC_FN(self._alloc), binding.FREE_FN(self._free))  # kept alive here

    def _alloc(self, nbytes, stream, ctx):
        if self.budget <= 0:
            return None
        self.budget -= 1
        self.allocs += 1
        return torch.cuda.caching_allocator_alloc(int(nbytes), stream=int(stream or 0))

    def _free(self, ptr, nbytes, stream, ctx):
        self.frees += 1
        torch.cuda.caching_allocator_delete(ptr)


def test_allocation_failure_reports_oom_and_launches_nothing(tf):
    P, B, S, H, D = 4, 1, 512, 8, 128
    Sl, Hl = S // P, H // P
    dtype = torch.bfloat16
    d = synth.qkv_shards(P, B, Sl, H, D, dtype, seed=3, layout="v_strided")
    wq, wk = synth.norm_weights(D, dtype, seed=3)
    g = synth.move(d, "cuda")
    kw = dict(norm_rope=True, q_weight=wq.cuda(), k_weight=wk.cuda(), eps=EPS)
    tf.cache_clear()
    ba = BudgetAllocator(tf, budget=0)
    tf.lib().tf_ulysses_set_allocator(ba.refs[0], ba.refs[1], None)
    try:
        launches, entries = tf.launch_count(), tf.cache_entries()

        # 1. the cached targets cannot be allocated
        with pytest.raises(tf.TfUlyssesError) as ex:
            tf.scatter_qkv("oom_targets", g["q"], g["k"], g["v"], theta=THETA, **kw)
        assert ex.value.status == tf.TF_ERR_OOM, ex.value
        assert tf.launch_count() == launches and tf.cache_entries() == entries

        # 2. caller-owned targets (nothing to allocate for them), a new RoPE table
        #    that cannot be allocated: nothing is written
        outs = [[torch.full((B, S, Hl, D), 7.0, dtype=dtype, device="cuda") for _ in range(P)] for _ in "qkv"]
        with pytest.raises(tf.TfUlyssesError) as ex:
            tf.scatter_qkv_into(g["q"], g["k"], g["v"], *outs, theta=THETA + 1.0, **kw)
        assert ex.value.status == tf.TF_ERR_OOM, ex.value
        torch.cuda.synchronize()
        assert tf.launch_count() == launches
        assert all(bool((t == 7.0).all()) for o in outs for t in o)

        # 3. the targets are allocated, the table is not: the call fails before its launch
        ba.budget = 1
        with pytest.raises(tf.TfUlyssesError) as ex:
            tf.scatter_qkv("oom_table", g["q"], g["k"], g["v"], theta=THETA + 2.0, **kw)
        assert ex.value.status == tf.TF_ERR_OOM, ex.value
        assert tf.launch_count() == launches
        assert ba.allocs == 1

        # 4. allocations succeed again: the same calls give the oracle's results
        ba.budget = 100
        tq, tk, tv, _ = tf.scatter_qkv("oom_targets", g["q"], g["k"], g["v"], theta=THETA, **kw)
        tf.scatter_qkv_into(g["q"], g["k"], g["v"], *outs, theta=THETA + 1.0, **kw)
        torch.cuda.synchronize()
        assert tf.launch_count() > launches
        for theta, (oq, ok, ov) in ((THETA, (tq, tk, tv)), (THETA + 1.0, outs)):
            table = oracle.rope_table(theta, S, D)
            for key, tg, w in (("q", oq, wq), ("k", ok, wk)):
                want = oracle.scatter_norm_rope(d[key], P, w, EPS, table)
                for i in range(P):
                    assert_fused_ok(tg[i], want[i])
            want_v = oracle.scatter(d["v"], P)
            for i in range(P):
                assert bits_equal(ov[i].cpu(), want_v[i])

        # every allocation the library got goes back through the same callback
        tf.cache_clear()
        assert ba.frees == ba.allocs
    finally:
        torch.cuda.synchronize()
        tf.cache_clear()
        tf.use_torch_allocator(True)


def _plain_inputs(P=2, B=1, Sl=64, H=4, D=64, seed=11):
    return synth.move(synth.qkv_shards(P, B, Sl, H, D, torch.bfloat16, seed=seed, layout="contiguous",
                                       with_k=False, with_v=False), "cuda")["q"]


SLEEP_CYCLES = 200_000_000  # about 0.1 s of one spinning thread block


def _fill_and_evict(tf, q, busy_stream, other_stream, mark, before=None):
    """`busy` enters the cache behind a sleep on busy_stream; twelve new keys on
    other_stream then evict it (capacity 12, `busy` least recently used; the
    twelfth key evicts).  `before`, if given, is recorded on other_stream
    between the eleventh and the twelfth key.  Returns the host time of the
    twelve calls."""
    with torch.cuda.stream(busy_stream):
        torch.cuda._sleep(SLEEP_CYCLES)
    mark.record(busy_stream)  # completes when the sleep ends, before busy's launch
    tf.scatter_qkv("busy", q, stream=busy_stream)
    assert not mark.query()  # the sleep is still running: busy's launch is pending
    t0 = time.perf_counter()
    for i in range(11):
        tf.scatter_qkv(f"evictor{i}", q, stream=other_stream)
    if before is not None:
        before.record(other_stream)
    assert tf.cache_entries() == 12
    tf.scatter_qkv("evictor11", q, stream=other_stream)
    return time.perf_counter() - t0


def test_evicting_a_busy_entry_default_allocator_orders_the_free_on_the_stream(tf):
    """The evicting calls return without waiting for busy's launch, and the
    evicting stream's work ends after it.  (Whether the evicting stream ran
    ahead before the eviction is not checked: two streams may share one
    hardware queue, and then the second waits behind the sleep anyway.)"""
    tf.cache_clear()
    tf.use_torch_allocator(False)  # cudaMallocAsync / cudaFreeAsync
    try:
        q = _plain_inputs()
        a, b = torch.cuda.Stream(), torch.cuda.Stream()
        mark = torch.cuda.Event(enable_timing=True)
        host_s = _fill_and_evict(tf, q, a, b, mark)
        b_end = torch.cuda.Event(enable_timing=True)
        b_end.record(b)
        assert not mark.query(), "the evicting calls waited on the host"
        assert host_s < 0.05, host_s
        torch.cuda.synchronize()
        assert tf.cache_entries() == 12
        # b's work ends after busy's completion (its targets are freed in b's order after it)
        assert mark.elapsed_time(b_end) >= 0.0
        want = oracle.scatter(cpu_list(q), len(q))
        tq, _, _, _ = tf.scatter_qkv("evictor11", q, stream=b)
        torch.cuda.synchronize()
        for i in range(len(q)):
            assert bits_equal(tq[i].cpu(), want[i])
    finally:
        torch.cuda.synchronize()
        tf.cache_clear()
        tf.use_torch_allocator(True)


def test_evicting_a_busy_entry_caller_allocator_releases_after_completion(tf):
    tf.cache_clear()
    mark = torch.cuda.Event()
    seen = []

    class Recording(BudgetAllocator):
        def _free(self, ptr, nbytes, stream, ctx):
            seen.append(mark.query())  # busy's launch, behind `mark`, is complete only if mark is
            super()._free(ptr, nbytes, stream, ctx)

    ra = Recording(tf, budget=1000)
    tf.lib().tf_ulysses_set_allocator(ra.refs[0], ra.refs[1], None)
    try:
        q = _plain_inputs(seed=12)
        a, b = torch.cuda.Stream(), torch.cuda.Stream()
        _fill_and_evict(tf, q, a, b, mark)
        assert seen == [True], seen  # exactly one eviction, released after busy's launch completed
        torch.cuda.synchronize()
        tf.cache_clear()
        assert ra.frees == ra.allocs
    finally:
        torch.cuda.synchronize()
        tf.cache_clear()
        tf.use_torch_allocator(True)


def cpu_list(ts):
    return [t.cpu() for t in ts]
