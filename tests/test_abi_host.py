"""Host-only checks of the C ABI: the library builds for sm_103a, loads, exports
every entry point include/tf_ulysses.h declares, and rejects bad arguments with
the documented status before touching CUDA (so these run without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tf_ulysses.h")


@pytest.fixture(scope="module")
def tf():
    from ulysses_sequence_attention_tf_gb300 import binding, build
    build.build()
    return binding


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"TF_API\s+[\w\s\*]+?\b(tf_ulysses_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("tf_ulysses_scatter_qkv", "tf_ulysses_gather_out", "tf_ulysses_cache_clear",
                 "tf_ulysses_last_error", "tf_ulysses_set_allocator"):
        assert must in names


def test_library_exports_every_declared_symbol(tf):
    lib = tf.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", tf.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT (tf_ulysses_\w+)", out.stdout))
    assert exported == set(declared_functions()), exported ^ set(declared_functions())
    assert tf.abi_version() == 1


FAKE = 0x10000  # 16-byte aligned; never dereferenced: validation fails first


def _scatter(tf, P=2, B=1, Sl=4, H=4, D=64, dtype=1, mode=0, q=True, k=True, v=True, strides=None, nr=None,
             tag=b"t", ptr=FAKE):
    lib = tf.lib()
    arr = (ctypes.c_void_p * max(P, 1))(*([ptr] * max(P, 1)))
    st = (tf.Strides * 3)()
    for i in range(3):
        st[i] = strides[i] if strides else tf.Strides(Sl * H * D, H * D, D)
    out = tf.Targets()
    return lib.tf_ulysses_scatter_qkv(tag, arr if q else None, arr if k else None, arr if v else None, st,
                                      P, B, Sl, H, D, dtype, mode, ctypes.byref(nr) if nr else None, None,
                                      ctypes.byref(out))


@pytest.mark.parametrize("kw,status", [
    (dict(P=0), 1), (dict(P=9), 1), (dict(B=-1), 1), (dict(H=0), 1),
    (dict(H=6, P=4), 2),                                  # heads not divisible by shards
    (dict(D=4), 3),                                       # a 8-byte head row is not a 16-byte vector
    (dict(dtype=7), 1),                                   # unknown dtype
    (dict(q=False), 1),                                   # q is required
    (dict(ptr=FAKE + 8), 3),                              # misaligned source
    (dict(ptr=0), 1),                                     # NULL source
    (dict(mode=2), 1),                                    # gather is not a scatter mode
    (dict(mode=1), 1),                                    # fused without parameters
    (dict(mode=1, dtype=2), 4),                           # fused fp32
    (dict(mode=1, D=96), 4),                              # fused D outside {32,64,128,256}
    (dict(tag=b"x" * 64), 1),                             # tag too long
    (dict(mode=3), 1),                                    # unknown base mode
    (dict(mode=0x400), 1),                                # unknown flag
    (dict(mode=0x200), 1),                                # half-split RoPE without the fused mode
    (dict(mode=0x100, v=False), 1),                       # fused layout without v
    (dict(mode=0x100, k=False), 1),                       # fused layout without k
    (dict(mode=0x102), 1),                                # fused layout on the gather mode
])
def test_scatter_rejects_before_any_cuda_call(tf, kw, status):
    assert _scatter(tf, **kw) == status
    assert tf.lib().tf_ulysses_last_error()


def test_bad_strides_rejected(tf):
    bad_t = [tf.Strides(1000, 8 * 64 + 4, 64)] * 3   # token stride not a multiple of 16 bytes
    assert _scatter(tf, strides=bad_t) == 3
    neg = [tf.Strides(1000, -512, 64)] * 3
    assert _scatter(tf, strides=neg) == 4


def test_fused_parameter_checks(tf):
    nr = tf.NormRope(FAKE + 4, FAKE, 1e-6, 10000.0, None)  # misaligned weight
    assert _scatter(tf, mode=1, nr=nr) == 3
    nr = tf.NormRope(FAKE, FAKE, float("nan"), 10000.0, None)
    assert _scatter(tf, mode=1, nr=nr) == 1
    nr = tf.NormRope(FAKE, FAKE, 1e-6, -1.0, None)  # no table and no valid theta
    assert _scatter(tf, mode=1, nr=nr) == 1
    nr = tf.NormRope(FAKE, FAKE, 1e-6, 10000.0, FAKE + 4)  # misaligned table
    assert _scatter(tf, mode=1, nr=nr) == 3


def test_fused_layout_targets_checked_before_any_cuda_call(tf):
    lib = tf.lib()
    P, B, Sl, H, D = 2, 1, 4, 4, 64
    arr = (ctypes.c_void_p * P)(*([FAKE] * P))
    st = (tf.Strides * 3)(*([tf.Strides(Sl * H * D, H * D, D)] * 3))
    into = lib.tf_ulysses_scatter_qkv_into
    # the payloads go in q_out; k_out / v_out must be NULL
    assert into(arr, arr, arr, st, P, B, Sl, H, D, 1, 0x100, None, None, None, None, None) == 1
    assert into(arr, arr, arr, st, P, B, Sl, H, D, 1, 0x100, None, arr, arr, None, None) == 1
    bad = (ctypes.c_void_p * P)(FAKE, FAKE + 8)
    assert into(arr, arr, arr, st, P, B, Sl, H, D, 1, 0x100, None, bad, None, None, None) == 3
    assert lib.tf_ulysses_scatter_qkv_noalloc(arr, arr, arr, st, P, B, Sl, H, D, 1, 0x100, None, arr, None, arr,
                                              None) == 1


def test_head_chunk_and_exchange_checked_before_any_cuda_call(tf):
    lib = tf.lib()
    P, B, Sl, H, D = 2, 1, 4, 8, 64
    arr = (ctypes.c_void_p * P)(*([FAKE] * P))
    st = (tf.Strides * 3)(*([tf.Strides(Sl * H * D, H * D, D)] * 3))
    heads = lib.tf_ulysses_scatter_qkv_heads_into
    for h0, h1 in ((-1, 2), (2, 2), (3, 1), (0, 5)):  # Hl = 4
        assert heads(arr, arr, arr, st, P, B, Sl, H, D, 1, 0, None, h0, h1, arr, arr, arr, None) == 1, (h0, h1)
    bad = (ctypes.c_void_p * P)(FAKE, FAKE + 8)
    assert heads(arr, arr, arr, st, P, B, Sl, H, D, 1, 0, None, 0, 2, bad, arr, arr, None) == 3
    ex = lib.tf_ulysses_exchange_chunks
    assert ex(arr, arr, 0, 64, None) == 1
    assert ex(None, arr, P, 64, None) == 1
    assert ex(arr, arr, P, 40, None) == 3    # chunk not a multiple of 16 bytes
    assert ex(bad, arr, P, 64, None) == 3    # misaligned payload


def test_slot_configuration_checked(tf):
    lib = tf.lib()
    assert lib.tf_ulysses_set_slots(b"rot", 0) == 1
    assert lib.tf_ulysses_set_slots(b"rot", 9) == 1
    assert lib.tf_ulysses_set_slots(b"x" * 64, 2) == 1
    assert lib.tf_ulysses_set_slots(b"rot", 2) == 0  # configuration only: no CUDA call
    assert lib.tf_ulysses_alloc_count() == 0
    assert lib.tf_ulysses_selftest_wait(0, None) == 1
    assert lib.tf_ulysses_selftest_wait(2_000_000_000, None) == 1


def test_gather_rejects_before_any_cuda_call(tf):
    lib = tf.lib()
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    out = tf.Targets()
    assert lib.tf_ulysses_gather_out(b"g", arr, None, 2, 1, 4, 5, 64, 1, None, None, None, ctypes.byref(out)) == 2
    assert lib.tf_ulysses_gather_out(b"g", None, None, 2, 1, 4, 4, 64, 1, None, None, None, ctypes.byref(out)) == 1
    bad = (ctypes.c_void_p * 2)(FAKE, FAKE + 2)
    assert lib.tf_ulysses_gather_out(b"g", arr, None, 2, 1, 4, 4, 64, 1, bad, None, None, ctypes.byref(out)) == 3
    assert lib.tf_ulysses_rope_table(10000.0, 16, 3, None, ctypes.byref(ctypes.c_void_p())) == 4
    assert lib.tf_ulysses_cache_entries() == 0


def test_fastdiv_exhaustive_on_host(tmp_path):
    """The invariant-divisor division used for index math is exact (checked in
    host code compiled from the same header)."""
    src = tmp_path / "fd.cpp"
    src.write_text(r'''
#include <cstdio>
#include <cstdint>
#include "relayout.h"
int main() {
  uint64_t bad = 0, x = 88172645463325252ull;
  auto rnd = [&]() { x ^= x << 13; x ^= x >> 7; x ^= x << 17; return uint32_t(x); };
  uint32_t edges[] = {0u, 1u, 2u, 3u, 0x7fffffffu, 0x80000000u, 0xfffffffeu, 0xffffffffu};
  for (uint32_t d = 1; d < 3000; ++d) {
    tfu::FastDiv f = tfu::make_fastdiv(d);
    for (uint32_t e : edges) bad += tfu::fastdiv(e, f) != e / d;
    for (int i = 0; i < 2000; ++i) { uint32_t n = rnd(); bad += tfu::fastdiv(n, f) != n / d; }
    for (uint32_t k = 1; k < 64; ++k) { uint32_t n = d * k; bad += tfu::fastdiv(n, f) != k;
                                        bad += tfu::fastdiv(n - 1, f) != k - 1; }
  }
  for (int j = 0; j < 20000; ++j) {
    uint32_t d = rnd() | 1u; tfu::FastDiv f = tfu::make_fastdiv(d);
    for (int i = 0; i < 50; ++i) { uint32_t n = rnd(); bad += tfu::fastdiv(n, f) != n / d; }
  }
  std::printf("%llu\n", (unsigned long long)bad);
  return bad != 0;
}
''')
    exe = tmp_path / "fd"
    csrc = os.path.join(ROOT, "ulysses_sequence_attention_tf_gb300", "csrc")
    subprocess.run(["g++", "-O2", "-std=c++17", f"-I{csrc}", "-I/usr/local/cuda/include", str(src), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "0", r.stdout
