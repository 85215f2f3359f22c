"""Host check of the projection kernel's tile order (csrc/gemm.h, the same
function the kernel runs): for many shapes, pass widths and cluster sizes,
every (shard, row tile, column tile) is computed by exactly one CTA, and the
only extra tiles (clusters of 2 with an odd number of row tiles) lie past the
last row tile, where nothing is stored."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "ulysses_sequence_attention_tf_gb300", "csrc")

HARNESS = r'''
#include <cstdio>
#include <cstdint>
#include <vector>
#include "gemm.h"
using namespace tfu;
static uint64_t s = 0x2545F4914F6CDD1Dull;
static uint32_t rnd(uint32_t n) { s ^= s << 13; s ^= s >> 7; s ^= s << 17; return uint32_t(s % n); }
template <int C>
long check(uint32_t P, uint32_t mt, uint32_t nt, uint32_t G) {
    long bad = 0;
    std::vector<int> seen(size_t(P) * mt * nt, 0);
    const uint32_t units = (P * mt + C - 1) / C * nt;
    for (uint32_t t = 0; t < units; ++t)
        for (uint32_t rank = 0; rank < uint32_t(C); ++rank) {
            GemmTile tl = gemm_tile<C>(P, mt, nt, G, t, rank);
            if (tl.n_tile >= nt) { ++bad; continue; }
            if (tl.m_tile == mt) { bad += tl.r != 0; continue; }  // a filler past the rows
            if (tl.r >= P || tl.m_tile > mt) { ++bad; continue; }
            ++seen[(size_t(tl.r) * mt + tl.m_tile) * nt + tl.n_tile];
        }
    for (int v : seen) bad += v != 1;
    return bad;
}
int main() {
    long bad = 0, cases = 0;
    for (int it = 0; it < 3000; ++it) {
        const uint32_t P = 1 + rnd(8), mt = 1 + rnd(40), nt = 1 + rnd(70), G = 1 + rnd(nt);
        bad += check<1>(P, mt, nt, G) + check<2>(P, mt, nt, G);
        cases += 2;
    }
    bad += check<1>(4, 64, 60, 18) + check<2>(4, 64, 60, 18) + check<2>(1, 1, 1, 1) + check<2>(3, 1, 5, 2);
    std::printf("%ld %ld\n", bad, cases);
    return bad != 0;
}
'''


def test_projection_tiles_cover_every_output_tile_once(tmp_path):
    src = tmp_path / "plan.cpp"
    src.write_text(HARNESS)
    exe = tmp_path / "plan"
    subprocess.run(["g++", "-O2", "-std=c++17", f"-I{CSRC}", "-I/usr/local/cuda/include", str(src), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    bad, cases = r.stdout.split()
    assert r.returncode == 0 and bad == "0", r.stdout
    assert int(cases) >= 6000
