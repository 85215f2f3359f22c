"""Host check of the staged kernel's work decomposition (csrc/tma_plan.h), the
same code the kernel runs: for many shapes and strides and both stage rings,
every unit fits one shared-memory stage, the planner's stage choice follows its
rule, its bulk-copy runs tile the unit's rows exactly and in
order, every run is really contiguous under the strides, stays inside the
plane, and has 16-byte aligned offsets and sizes; and the same runs dealt out
to the lanes of a warp (for_each_run_lane) are, over all lanes, exactly those
runs, and no lane but the first gets a run of a side whose full units have
fewer runs than the split threshold (unit_split_runs)."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "ulysses_sequence_attention_tf_gb300", "csrc")

HARNESS = r'''
#include <cstdio>
#include <cstdint>
#include <algorithm>
#include <utility>
#include <vector>
#include "tma_plan.h"
using namespace tfu;
static uint64_t x = 0x9E3779B97F4A7C15ull;
static uint32_t rnd(uint32_t n) { x ^= x << 13; x ^= x >> 7; x ^= x << 17; return uint32_t(x % n); }
int main() {
  long bad = 0, cases = 0, lane_checks = 0;
  for (int it = 0; it < 4000; ++it) {
    const uint32_t Sl = 1 + rnd(300), Hl = rnd(4) == 0 ? 1 : 1 + rnd(70);
    const uint32_t rb = 16 * (1 + rnd(40));            // D * esize, a multiple of 16
    // source-like strides: packed heads or spread heads, token stride >= band
    const bool packed = rnd(3) != 0;
    const int64_t sh = packed ? rb : int64_t(rb) + 16 * (1 + rnd(8));
    const int64_t band = int64_t(Hl - 1) * sh + rb;
    const int64_t st = rnd(3) == 0 && packed ? int64_t(Hl) * rb : band + 16 * rnd(64);
    const uint32_t stage = (it & 1) ? kStageBytes : kStageBytesSmall;  // both rings
    const uint32_t rpu = tma_rows_per_unit(Hl, rb, stage);
    const uint32_t rows = Sl * Hl;
    if (rb > stage) { if (rpu != 0) ++bad; continue; }
    if (rpu == 0 || uint64_t(rpu) * rb > stage) { ++bad; continue; }
    if (uint64_t(Hl) * rb <= stage && rpu % Hl != 0) { ++bad; continue; }  // whole tokens
    // the stage choice: the small ring only for bands under 3 KiB on launches over 288 MiB
    const uint32_t big = staged_stage_bytes(uint64_t(Hl) * rb, rb, uint64_t(320) << 20);
    if (big != ((uint64_t(Hl) * rb >= 3072 || rb > kStageBytesSmall) ? kStageBytes : kStageBytesSmall)) ++bad;
    if (staged_stage_bytes(uint64_t(Hl) * rb, rb, uint64_t(288) << 20) != kStageBytes) ++bad;
    const int64_t extent = int64_t(Sl - 1) * st + band;
    for (uint32_t R0 = 0; R0 < rows; R0 += rpu) {
      const uint32_t R1 = R0 + rpu < rows ? R0 + rpu : rows;
      uint32_t next = 0;
      for_each_run(R0, R1, Hl, st, sh, rb, [&](uint32_t i, uint32_t n, int64_t off) {
        ++cases;
        if (i != next || n == 0 || i + n > R1 - R0) ++bad;
        if (off % 16 != 0 || (uint64_t(n) * rb) % 16 != 0) ++bad;
        for (uint32_t k = 0; k < n; ++k) {  // each row of the run where the strides put it
          const uint32_t R = R0 + i + k, t = R / Hl, h = R % Hl;
          if (off + int64_t(k) * rb != int64_t(t) * st + int64_t(h) * sh) ++bad;
        }
        if (off < 0 || off + int64_t(n) * rb > extent) ++bad;
        next = i + n;
      });
      if (next != R1 - R0) ++bad;
      // the same runs dealt out to lanes: their union is exactly for_each_run's runs
      std::vector<std::pair<uint32_t, std::pair<uint32_t, int64_t>>> want, got;
      for_each_run(R0, R1, Hl, st, sh, rb, [&](uint32_t i, uint32_t n, int64_t off) { want.push_back({i, {n, off}}); });
      for (uint32_t lanes : {32u, 7u, 1u})
        for (uint32_t min_split : {1u, 17u, 1000u}) {
          got.clear();
          for (uint32_t lane = 0; lane < lanes; ++lane)
            for_each_run_lane(R0, R1, Hl, st, sh, rb, lane, lanes, min_split,
                              [&](uint32_t i, uint32_t n, int64_t off) { got.push_back({i, {n, off}}); });
          std::sort(got.begin(), got.end());
          if (got != want) ++bad;
          ++lane_checks;
          // a side whose full units give fewer runs than min_split stays on worker 0
          if (unit_split_runs(rpu, Hl, st, sh, rb) < min_split)
            for (uint32_t lane = 1; lane < lanes; ++lane)
              for_each_run_lane(R0, R1, Hl, st, sh, rb, lane, lanes, min_split,
                                [&](uint32_t, uint32_t, int64_t) { ++bad; });
        }
    }
  }
  // a row larger than a stage is refused
  if (tma_rows_per_unit(4, kStageBytes + 16) != 0) ++bad;
  if (tma_rows_per_unit(4, kStageBytesSmall + 16, kStageBytesSmall) != 0) ++bad;
  std::printf("%ld %ld %ld\n", bad, cases, lane_checks);
  return bad != 0;
}
'''


def test_staged_plan_runs_tile_units_exactly(tmp_path):
    src = tmp_path / "plan.cpp"
    src.write_text(HARNESS)
    exe = tmp_path / "plan"
    subprocess.run(["g++", "-O2", "-std=c++17", f"-I{CSRC}", str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    bad, cases, lane_checks = r.stdout.split()
    assert r.returncode == 0 and bad == "0", r.stdout
    assert int(cases) > 10000 and int(lane_checks) > 10000
