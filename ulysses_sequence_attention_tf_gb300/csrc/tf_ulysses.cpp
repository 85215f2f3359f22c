// tf_ulysses.cpp -- host side of the C ABI declared in include/tf_ulysses.h:
// argument validation (all of it before any CUDA call), the tagged target cache,
// the resident RoPE tables, the allocator hook and the launches.
//
// Sources: TeleFuser PR #27 "Add CUDA IPC Ulysses overlap and lossless LingBot
// streaming", "Changes Made" (final-layout targets; a bounded cache of at most 12 target
// sets, keyed on the tag, the shape, the dtype, a mode and the device; one
// grouped completion for tagged Q/K/V) and "Additional Notes" (no protocol switch once a grouped transfer
// started -- here: nothing is launched unless every check passed); TeleFuser PR
// #22 (RoPE tables kept resident); TeleFuser docs "Communication Architecture",
// "Cross-Worker Tensor Channel" (slot reuse ordered by an event, no device-wide
// synchronisation) for how cache reuse and eviction are ordered.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "gemm.h"
#include "noalloc.h"
#include "relayout.h"
#include "tf_ulysses.h"
#include "tma_plan.h"

namespace {

// A named NVTX range around each C-ABI call, so that a profiler's timeline shows
// which library call issued which launches (header-only NVTX; a few nanoseconds
// when no profiler is attached).
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};

using tfu::RelayoutParams;

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_allocs{0};  // device allocations made (cache entries, tables)
std::mutex g_mu;  // guards the cache, the tables and the allocator
// The relayout launchers fill per-kernel launch facts (occupancy, the shared-memory
// opt-in) into function-local statics on first use; calls that launch without
// g_mu serialise on this one, which is never held while taking g_mu.
std::mutex g_launch_mu;

tf_status fail(tf_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

tf_status cuda_fail(cudaError_t e, const char* what) {
    return fail(TF_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ---------------------------------------------------------------- stream capture
// CUDA-graph capture protocol (flashinfer PR #6332 commit message, "Description",
// "CUDA graphs": a prepared call allocates nothing; a size first seen inside a
// capture fails rather than allocate; captured calls interleave with eager
// ones).  Inside a capture the library allocates and frees nothing, records its
// events as external event nodes (so every replay records them) and waits on
// events recorded outside the capture as external waits.
tf_status capture_state(cudaStream_t s, bool* capturing) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    *capturing = st != cudaStreamCaptureStatusNone;
    return TF_OK;
}

cudaError_t record_event(cudaEvent_t ev, cudaStream_t s, bool capturing) {
    return capturing ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal) : cudaEventRecord(ev, s);
}

cudaError_t wait_event(cudaStream_t s, cudaEvent_t ev, bool capturing) {
    return cudaStreamWaitEvent(s, ev, capturing ? cudaEventWaitExternal : 0);
}

// ---------------------------------------------------------------- allocator
struct Allocator {
    tf_alloc_fn alloc = nullptr;
    tf_free_fn release = nullptr;
    void* ctx = nullptr;
};
Allocator g_alloc;

void* dev_alloc(const Allocator& a, size_t bytes, cudaStream_t s) {
    if (bytes == 0) return nullptr;
    g_allocs.fetch_add(1);
    if (a.alloc) return a.alloc(bytes, s, a.ctx);
    void* p = nullptr;
    if (cudaMallocAsync(&p, bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return p;
}

// Release memory whose last use is `last_use` (an event recorded after it).
void dev_release(const Allocator& a, void* ptr, size_t bytes, cudaEvent_t last_use, cudaStream_t s) {
    if (!ptr) return;
    if (a.release) {
        if (last_use) cudaEventSynchronize(last_use);
        a.release(ptr, bytes, s, a.ctx);
    } else {
        if (last_use) cudaStreamWaitEvent(s, last_use, 0);
        cudaFreeAsync(ptr, s);
    }
}

// ---------------------------------------------------------------- validation
int elem_size(tf_dtype d) {
    switch (d) {
        case TF_FP16: return 2;
        case TF_BF16: return 2;
        case TF_FP32: return 4;
        case TF_BYTE: return 1;
    }
    return 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Shape {
    int P, B, Sl, H, D, Hl, esize;
    tf_dtype dtype;
    int Hg;  // heads between consecutive head groups on the head-major side (Hl unless a head chunk)
};

tf_status check_shape(int P, int B, int Sl, int H, int D, tf_dtype dtype, Shape* sh) {
    if (P < 1 || P > TF_ULYSSES_MAX_SHARDS) return fail(TF_ERR_INVALID, "P=%d outside [1, %d]", P, TF_ULYSSES_MAX_SHARDS);
    if (B < 0 || Sl < 0) return fail(TF_ERR_INVALID, "B=%d, S_local=%d must be >= 0", B, Sl);
    if (H < 1 || D < 1) return fail(TF_ERR_INVALID, "H=%d, D=%d must be >= 1", H, D);
    const int e = elem_size(dtype);
    if (e == 0) return fail(TF_ERR_INVALID, "unknown dtype %d", int(dtype));
    if (H % P != 0) return fail(TF_ERR_DIVISIBILITY, "H=%d is not divisible by P=%d", H, P);
    if ((int64_t(D) * e) % 16 != 0)
        return fail(TF_ERR_ALIGNMENT, "a head row (D=%d x %d B) must be a multiple of 16 bytes", D, e);
    if (int64_t(P) * Sl > INT32_MAX) return fail(TF_ERR_UNSUPPORTED, "P*S_local too large");
    *sh = Shape{P, B, Sl, H, D, H / P, e, dtype, H / P};
    return TF_OK;
}

tf_status check_ptrs(const char* what, const void* const* a, int P) {
    for (int i = 0; i < P; ++i) {
        if (!a[i]) return fail(TF_ERR_INVALID, "%s[%d] is NULL", what, i);
        if (!aligned16(a[i])) return fail(TF_ERR_ALIGNMENT, "%s[%d] is not 16-byte aligned", what, i);
    }
    return TF_OK;
}

// strides of a [nb, nt, nh, D] view; a stride of an extent-1 dimension is never used
tf_status check_strides(const char* what, const tf_strides& s, int esize, int64_t nb, int64_t nt, int64_t nh) {
    const int64_t v[3] = {s.b, s.t, s.h};
    const int64_t n[3] = {nb, nt, nh};
    const char* name[3] = {"b", "t", "h"};
    for (int i = 0; i < 3; ++i) {
        if (n[i] <= 1) continue;
        if (v[i] < 0) return fail(TF_ERR_UNSUPPORTED, "%s stride %s=%lld is negative", what, name[i], (long long)v[i]);
        if ((v[i] * esize) % 16 != 0)
            return fail(TF_ERR_ALIGNMENT, "%s stride %s=%lld elements is not a multiple of 16 bytes", what, name[i],
                        (long long)v[i]);
    }
    return TF_OK;
}

// 32-byte vectors when every address the kernel forms is 32-byte aligned
// (bases, strides of dimensions longer than 1, weights, the head row), else 16.
uint32_t pick_vec_bytes(const RelayoutParams& p, const Shape& sh, int64_t src_tokens, int64_t dst_tokens) {
    auto ok = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 31u) == 0; };
    auto ok_stride = [](int64_t st, int64_t extent) { return extent <= 1 || st % 32 == 0; };
    if ((int64_t(sh.D) * sh.esize) % 32 != 0) return 16;
    for (uint32_t x = 0; x < p.nx; ++x) {
        for (int i = 0; i < sh.P; ++i)
            if (!ok(p.src[x][i]) || !ok(p.dst[x][i])) return 16;
        if (!ok_stride(p.s_b[x], sh.B) || !ok_stride(p.s_t[x], src_tokens) || !ok_stride(p.s_h[x], sh.H) ||
            !ok_stride(p.d_b[x], sh.B) || !ok_stride(p.d_t[x], dst_tokens) || !ok_stride(p.d_h[x], sh.H))
            return 16;
        if (((p.fused_mask >> x) & 1u) && !ok(p.weight[x])) return 16;
    }
    return 32;
}

// Sizes of the unit grid for vectors of p.vec_bytes; everything indexed in 32
// bits must fit.
tf_status plan_units(RelayoutParams& p, const Shape& sh) {
    p.P = uint32_t(sh.P);
    p.B = uint32_t(sh.B);
    p.Sl = uint32_t(sh.Sl);
    p.Hl = uint32_t(sh.Hl);
    p.Hg = uint32_t(sh.Hg);
    if (p.vec_bytes != 16 && p.vec_bytes != 32) p.vec_bytes = 16;
    p.vpr = uint32_t(int64_t(sh.D) * sh.esize / p.vec_bytes);
    const uint64_t nv = uint64_t(sh.Sl) * uint64_t(sh.Hl) * p.vpr;
    if (nv > (uint64_t(1) << 31)) return fail(TF_ERR_UNSUPPORTED, "one shard/head-group block exceeds 2^31 vectors");
    p.nv = uint32_t(nv);
    const uint64_t cv = uint64_t(tfu::chunk_vecs(int(p.vec_bytes)));
    const uint64_t planes = uint64_t(sh.B) * sh.P * p.nx * sh.P;
    const uint64_t chunks = (nv + cv - 1) / cv;
    if (planes * chunks >= (uint64_t(1) << 31)) return fail(TF_ERR_UNSUPPORTED, "problem exceeds 2^31 work units");
    p.n_planes = uint32_t(planes);
    p.n_chunks = uint32_t(chunks);
    p.n_units = uint32_t(planes * chunks);
    p.div_vpr = tfu::make_fastdiv(p.vpr);
    p.div_hl = tfu::make_fastdiv(p.Hl);
    p.div_planes = tfu::make_fastdiv(p.n_planes ? p.n_planes : 1);
    return TF_OK;
}

#ifndef TFU_SMALL_BAND
// Token head bands (Hl * D * esize bytes) up to this size take the register paths
// for pure relayouts: the block kernel for copy scatters, the register kernel for
// gathers (measured on GB300: 768-byte bands gather at 0.77-0.78 of the copy peak
// by registers against 0.58 by bulk copies, and scatter at 0.85-0.86 against 0.73).
#define TFU_SMALL_BAND 1024
#endif
constexpr uint64_t kSmallBandBytes = TFU_SMALL_BAND;
#ifndef TFU_BLOCK_COPY_BAND
// Copy scatters of head rows of 256 bytes or more take the block kernel up to this
// band as well (GB300, fractions of the copy peak after a read flush: 72 MB
// FLUX-like scatter, 1.5 KiB bands, 0.90 against 0.83 by bulk copies; 2 KiB bands
// 0.97-0.98 against 0.94-0.96; the video-DiT copy scatter, 2.5 KiB, 6276 against
// 6050 GB/s back to back).  Bands of 3 KiB or more stay on the bulk-copy kernel.
#define TFU_BLOCK_COPY_BAND 2560
#endif
constexpr uint64_t kBlockCopyBandBytes = TFU_BLOCK_COPY_BAND;
#ifndef TFU_BLOCK_PASSES
#define TFU_BLOCK_PASSES 0  // pipeline passes per row group and unit of the block kernel; 0: by slot count
#endif

// Plan and launch one relayout:
//  * scatters with D * esize in {64, 128, 256, 512} bytes: every fused scatter
//    (32-byte vectors, or two 16-byte halves per lane when the rows are only
//    16-byte aligned), and with 32-byte vectors the copies into the fused
//    receive layout and the copies whose token head band is at most 1 KiB -- or
//    2.5 KiB for head rows of 256 bytes or more: the block kernel, all slots of a
//    token block in one pass;
//  * other pure relayouts whose head row fits a stage, except gathers of small
//    bands or 128-byte rows: the shared-memory-staged (bulk-copy) kernel;
//  * the rest: the register kernel with 32- or 16-byte vectors.
tf_status launch_planned(RelayoutParams& p, const Shape& sh, tfu::Dir dir, tfu::Fused fused, int64_t src_tokens,
                         int64_t dst_tokens, cudaStream_t stream) {
    const uint32_t rb = uint32_t(int64_t(sh.D) * sh.esize);
    const uint64_t rows = uint64_t(sh.Sl) * uint64_t(sh.Hl);
    if (rows >= (uint64_t(1) << 31)) return fail(TF_ERR_UNSUPPORTED, "one shard/head-group block exceeds 2^31 rows");
    p.P = uint32_t(sh.P);
    p.B = uint32_t(sh.B);
    p.Sl = uint32_t(sh.Sl);
    p.Hl = uint32_t(sh.Hl);
    p.Hg = uint32_t(sh.Hg);
    p.row_bytes = rb;
    p.plane_rows = uint32_t(rows);
    p.div_hl = tfu::make_fastdiv(p.Hl);
#if TFU_CHECKED
    {
        // the last byte a kernel may touch in each slot's buffers: token rows
        // [0, tokens), heads [0, span) of the head-major side (bands Hg apart) or
        // [0, Hl) of the token-major side, batch rows [0, B)
        const int64_t span_heads = int64_t(sh.P - 1) * sh.Hg + sh.Hl;
        const bool scatter = dir == tfu::Dir::kScatter;
        for (uint32_t x = 0; x < p.nx; ++x)
            for (int i = 0; i < sh.P; ++i) {
                const int64_t src_heads = scatter ? span_heads : sh.Hl;
                const int64_t dst_heads = scatter ? sh.Hl : span_heads;
                p.src_end[x][i] = p.src[x][i] ? p.src[x][i] + (sh.B - 1) * p.s_b[x] + (src_tokens - 1) * p.s_t[x] +
                                                    (src_heads - 1) * p.s_h[x] + rb
                                              : nullptr;
                p.dst_end[x][i] = p.dst[x][i] ? p.dst[x][i] + (sh.B - 1) * p.d_b[x] + (dst_tokens - 1) * p.d_t[x] +
                                                    (dst_heads - 1) * p.d_h[x] + rb
                                              : nullptr;
            }
        p.table_end = p.table ? p.table + dst_tokens * int64_t(sh.D) : nullptr;
    }
#endif
    // row-unit grids (block and staged kernels): `blocks` row ranges of rpu rows
    auto plan_rows = [&](uint64_t blocks, uint32_t rpu) -> tf_status {
        const uint64_t chunks = (rows + rpu - 1) / rpu;
        if (blocks * chunks >= (uint64_t(1) << 31)) return fail(TF_ERR_UNSUPPORTED, "problem exceeds 2^31 work units");
        p.rpu = rpu;
        p.n_planes = uint32_t(blocks);
        p.n_chunks = uint32_t(chunks);
        p.n_units = uint32_t(blocks * chunks);
        p.div_planes = tfu::make_fastdiv(p.n_planes ? p.n_planes : 1);
        return TF_OK;
    };
    tf_status s;
    cudaError_t e;
    bool dst_rows_packed = true;  // scatter target rows adjacent (else the fused receive layout)
    bool dst_shared = true;       // every slot's targets have the same strides (the block kernel's assumption)
    for (uint32_t x = 0; x < p.nx; ++x) {
        dst_rows_packed = dst_rows_packed && p.d_h[x] == int64_t(rb);
        dst_shared = dst_shared && p.d_t[x] == p.d_t[0] && p.d_h[x] == p.d_h[0];
    }
    // a token's head band: the contiguous piece of the strided side (the scatter's
    // source, the gather's destination); the bulk-copy engine moves pieces of a KiB
    // or less, and gathers of 128-byte rows, slower than the register paths
    const bool small_band = uint64_t(sh.Hl) * rb <= kSmallBandBytes;
    // copy scatters of 256- or 512-byte head rows in bands up to 2.5 KiB also move
    // faster through the registers than through the bulk-copy engine
    const bool mid_band = rb >= 256 && uint64_t(sh.Hl) * rb <= kBlockCopyBandBytes;
    const bool block_ok = dir == tfu::Dir::kScatter && dst_shared && (rb == 64 || rb == 128 || rb == 256 || rb == 512) &&
                          (fused != tfu::Fused::kNone || !dst_rows_packed || small_band || mid_band);
    const bool staged_ok = fused == tfu::Fused::kNone && !(dir == tfu::Dir::kGather && (small_band || rb <= 128));
    const uint32_t vec = pick_vec_bytes(p, sh, src_tokens, dst_tokens);
    // staged units: the stage ring by head band and launch size (tma_plan.h)
    const uint64_t band = uint64_t(sh.Hl) * rb;
    const uint64_t bytes_per_direction = uint64_t(sh.B) * sh.P * p.nx * sh.P * rows * rb;
    const uint32_t rpu = tfu::tma_rows_per_unit(uint32_t(sh.Hl), rb,
                                                tfu::staged_stage_bytes(band, rb, bytes_per_direction));
    if (block_ok && (vec == 32 || fused != tfu::Fused::kNone)) {
        p.vec_bytes = vec;  // 16: the fused rows are moved as two 16-byte halves per lane
        p.vpr = rb / 32;
        // a unit gives every row group of the CTA whole pipeline passes (kThreads / vpr
        // groups, depth rows each): one pass when three slots share the rows, else two
        const uint32_t depth = fused == tfu::Fused::kNone ? tfu::kCopyBlockDepth
                               : (p.fused_mask & 1u)       ? tfu::kQkBlockDepth
                                                           : tfu::kBlockDepth;
        const uint32_t passes = TFU_BLOCK_PASSES > 0 ? TFU_BLOCK_PASSES : (p.nx >= 3 ? 1u : 2u);
        const uint32_t unit_rows = uint32_t(tfu::kThreads) / p.vpr * depth * passes;
        if ((s = plan_rows(uint64_t(sh.B) * sh.P * sh.P, unit_rows)) != TF_OK) return s;
        std::lock_guard<std::mutex> launch_lock(g_launch_mu);
        e = tfu::launch_blocks(p, fused, stream);
    } else if (staged_ok && rpu > 0) {
        if ((s = plan_rows(uint64_t(sh.B) * sh.P * p.nx * sh.P, rpu)) != TF_OK) return s;
        std::lock_guard<std::mutex> launch_lock(g_launch_mu);
        e = tfu::launch_relayout_staged(p, dir, fused, stream);
    } else {
        if (fused != tfu::Fused::kNone) return fail(TF_ERR_UNSUPPORTED, "this fused scatter has no kernel");
        p.vec_bytes = vec;
        if ((s = plan_units(p, sh)) != TF_OK) return s;
        std::lock_guard<std::mutex> launch_lock(g_launch_mu);
        e = tfu::launch_relayout(p, dir, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "launching the relayout kernel");
    g_launches.fetch_add(1);
    return TF_OK;
}

// ---------------------------------------------------------------- RoPE tables
constexpr int kMaxTables = 4;
struct Table {
    float theta = 0;
    int S = 0, D = 0, device = -1;
    float* ptr = nullptr;
    size_t bytes = 0;
    Allocator alloc;
    cudaEvent_t last_use = nullptr;  // recorded after the build and after every launch that reads it
    uint64_t stamp = 0;
};
std::vector<Table> g_tables;
uint64_t g_clock = 0;

// Caller holds g_mu.  Returns a table with >= S rows for (theta, D) on `device`,
// ordered on `stream` after its build.
tf_status get_table(float theta, int S, int D, int device, cudaStream_t stream, bool capturing, Table** out) {
    for (auto& t : g_tables) {
        if (t.device == device && t.D == D && t.S >= S && std::memcmp(&t.theta, &theta, sizeof theta) == 0) {
            t.stamp = ++g_clock;
            cudaError_t e = wait_event(stream, t.last_use, capturing);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(table)");
            *out = &t;
            return TF_OK;
        }
    }
    if (capturing)
        return fail(TF_ERR_UNSUPPORTED,
                    "the RoPE table for (theta, S=%d, D=%d) is first needed inside a stream capture: make one eager "
                    "call (or tf_ulysses_rope_table) before capturing; nothing is allocated during a capture", S, D);
    if (int(g_tables.size()) >= kMaxTables) {  // evict the least recently used table
        size_t lru = 0;
        for (size_t i = 1; i < g_tables.size(); ++i)
            if (g_tables[i].stamp < g_tables[lru].stamp) lru = i;
        Table& t = g_tables[lru];
        dev_release(t.alloc, t.ptr, t.bytes, t.last_use, stream);
        cudaEventDestroy(t.last_use);
        g_tables.erase(g_tables.begin() + lru);
    }
    Table t;
    t.theta = theta;
    t.S = S;
    t.D = D;
    t.device = device;
    t.bytes = size_t(S) * size_t(D) * sizeof(float);
    t.alloc = g_alloc;
    t.ptr = static_cast<float*>(dev_alloc(t.alloc, t.bytes, stream));
    if (t.bytes && !t.ptr) return fail(TF_ERR_OOM, "allocating a %zu-byte RoPE table failed", t.bytes);
    cudaError_t e = cudaEventCreateWithFlags(&t.last_use, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        dev_release(t.alloc, t.ptr, t.bytes, nullptr, stream);
        return cuda_fail(e, "cudaEventCreate");
    }
    // frequencies of the interleaved pairs, theta^(-2i/D), in double on the host
    std::vector<double> inv_freq(size_t(D / 2));
    for (int i = 0; i < D / 2; ++i) inv_freq[size_t(i)] = std::pow(double(theta), -2.0 * i / D);
    e = tfu::launch_rope_table(t.ptr, inv_freq.data(), S, D, stream);
    if (e == cudaSuccess && S > 0) g_launches.fetch_add(1);
    if (e == cudaSuccess) e = cudaEventRecord(t.last_use, stream);
    if (e != cudaSuccess) {
        dev_release(t.alloc, t.ptr, t.bytes, nullptr, stream);
        cudaEventDestroy(t.last_use);
        return cuda_fail(e, "building the RoPE table");
    }
    t.stamp = ++g_clock;
    g_tables.push_back(t);
    *out = &g_tables.back();
    return TF_OK;
}

// ---------------------------------------------------------------- target cache
struct Entry {
    std::string tag;
    int mode = 0, present = 0, P = 0, B = 0, Sl = 0, H = 0, D = 0, dtype = 0, device = -1;
    void* slab = nullptr;
    size_t bytes = 0;
    Allocator alloc;
    void* buf[3][TF_ULYSSES_MAX_SHARDS] = {};  // slot 0's buffers
    size_t slot_bytes = 0;                     // slot s's buffers are slot 0's + s * slot_bytes
    int slots = 1, next_slot = 0;              // rotating target sets; the next call writes next_slot
    cudaEvent_t done = nullptr;
    cudaStream_t last_stream = nullptr;  // null: unknown (e.g. last written by a graph replay)
    uint64_t stamp = 0;
};
std::vector<Entry> g_entries;

// Rotating target sets per tag (tf_ulysses_set_slots), read when an entry is created.
std::vector<std::pair<std::string, int>> g_tag_slots;

int slots_of(const std::string& tag) {
    for (auto& ts : g_tag_slots)
        if (ts.first == tag) return ts.second;
    return 1;
}

// The buffer of tensor x, group/shard i, in the slot a call uses.
void* slot_buffer(const Entry& e, int slot, int x, int i) {
    uint8_t* base = static_cast<uint8_t*>(e.buf[x][i]);
    return base ? base + size_t(slot) * e.slot_bytes : nullptr;
}

void reclaim_entry(Entry& e, cudaStream_t stream) {
    dev_release(e.alloc, e.slab, e.bytes, e.done, stream);
    if (e.done) cudaEventDestroy(e.done);
    e.slab = nullptr;
    e.done = nullptr;
}

size_t round_up(size_t n, size_t a) { return (n + a - 1) / a * a; }

// Caller holds g_mu.  buffer_bytes: size of one target; counts[x]: buffers of tensor x.
tf_status get_entry(const std::string& tag, int mode, int present, const Shape& sh, int device, size_t buffer_bytes,
                    const int counts[3], cudaStream_t stream, bool capturing, Entry** out) {
    for (auto& e : g_entries) {
        if (e.tag == tag && e.mode == mode && e.present == present && e.P == sh.P && e.B == sh.B && e.Sl == sh.Sl &&
            e.H == sh.H && e.D == sh.D && e.dtype == int(sh.dtype) && e.device == device) {
            if (e.last_stream != stream) {  // order the rewrite after the previous one
                cudaError_t err = wait_event(stream, e.done, capturing);
                if (err != cudaSuccess) return cuda_fail(err, "cudaStreamWaitEvent(entry)");
            }
            e.stamp = ++g_clock;
            *out = &e;
            return TF_OK;
        }
    }
    if (capturing)
        return fail(TF_ERR_UNSUPPORTED,
                    "cache key (tag \"%s\", this shape, dtype and mode) first seen inside a stream capture: make one "
                    "eager call with it before capturing; nothing is allocated during a capture", tag.c_str());
    if (int(g_entries.size()) >= TF_ULYSSES_CACHE_CAPACITY) {
        size_t lru = 0;
        for (size_t i = 1; i < g_entries.size(); ++i)
            if (g_entries[i].stamp < g_entries[lru].stamp) lru = i;
        reclaim_entry(g_entries[lru], stream);
        g_entries.erase(g_entries.begin() + lru);
    }
    Entry e;
    e.tag = tag;
    e.mode = mode;
    e.present = present;
    e.P = sh.P;
    e.B = sh.B;
    e.Sl = sh.Sl;
    e.H = sh.H;
    e.D = sh.D;
    e.dtype = int(sh.dtype);
    e.device = device;
    e.alloc = g_alloc;
    e.slots = slots_of(tag);
    const size_t stride = round_up(buffer_bytes, 256);
    e.slot_bytes = stride * size_t(counts[0] + counts[1] + counts[2]);
    e.bytes = e.slot_bytes * size_t(e.slots);
    e.slab = dev_alloc(e.alloc, e.bytes, stream);
    if (e.bytes && !e.slab) return fail(TF_ERR_OOM, "allocating %zu bytes of targets failed", e.bytes);
    size_t off = 0;
    for (int x = 0; x < 3; ++x)
        for (int i = 0; i < counts[x]; ++i, off += stride)
            e.buf[x][i] = buffer_bytes ? static_cast<uint8_t*>(e.slab) + off : nullptr;
    cudaError_t err = cudaEventCreateWithFlags(&e.done, cudaEventDisableTiming);
    if (err != cudaSuccess) {
        dev_release(e.alloc, e.slab, e.bytes, nullptr, stream);
        return cuda_fail(err, "cudaEventCreate");
    }
    e.last_stream = stream;
    e.stamp = ++g_clock;
    g_entries.push_back(e);
    *out = &g_entries.back();
    return TF_OK;
}

// ---------------------------------------------------------------- scatter core
struct ScatterPlan {
    Shape sh;
    RelayoutParams p{};
    tfu::Fused fused = tfu::Fused::kNone;
    int slot_of[3] = {-1, -1, -1};  // tensor (q=0, k=1, v=2) -> slot
    int present = 0;                // bit per tensor
    bool empty = false;
    bool fused_layout = false;       // one [B, S, Hl, 3*D] payload per head group
    int64_t row_off[3] = {0, 0, 0};  // byte offset of tensor x's row inside a payload row
};

constexpr int kModeBase = 0xff;
constexpr int kModeFlags = TF_MODE_FLAG_FUSED_LAYOUT | TF_MODE_FLAG_ROPE_NEOX;

tf_status plan_scatter(const void* const* q, const void* const* k, const void* const* v, const tf_strides* strides,
                       int P, int B, int Sl, int H, int D, tf_dtype dtype, tf_mode mode, const tf_norm_rope* nr,
                       ScatterPlan* plan) {
    ScatterPlan& pl = *plan;
    tf_status s = check_shape(P, B, Sl, H, D, dtype, &pl.sh);
    if (s != TF_OK) return s;
    const int base = int(mode) & kModeBase, flags = int(mode) & ~kModeBase;
    if (base != TF_MODE_SCATTER && base != TF_MODE_SCATTER_NORM_ROPE)
        return fail(TF_ERR_INVALID, "mode %d is not a scatter mode", int(mode));
    if (flags & ~kModeFlags) return fail(TF_ERR_INVALID, "unknown mode flags 0x%x", unsigned(flags & ~kModeFlags));
    const bool neox = (flags & TF_MODE_FLAG_ROPE_NEOX) != 0;
    if (neox && base != TF_MODE_SCATTER_NORM_ROPE)
        return fail(TF_ERR_INVALID, "TF_MODE_FLAG_ROPE_NEOX needs TF_MODE_SCATTER_NORM_ROPE");
    pl.fused_layout = (flags & TF_MODE_FLAG_FUSED_LAYOUT) != 0;
    if (pl.fused_layout && (!k || !v)) return fail(TF_ERR_INVALID, "the fused layout needs q, k and v");
    if (!q) return fail(TF_ERR_INVALID, "q is NULL");
    if (!strides) return fail(TF_ERR_INVALID, "strides is NULL");
    const void* const* src[3] = {q, k, v};
    const char* names[3] = {"q", "k", "v"};
    for (int x = 0; x < 3; ++x) {
        if (!src[x]) continue;
        pl.present |= 1 << x;
        if (B > 0 && Sl > 0 && (s = check_ptrs(names[x], src[x], P)) != TF_OK) return s;
        if ((s = check_strides(names[x], strides[x], pl.sh.esize, B, Sl, H)) != TF_OK) return s;
    }
    if (base == TF_MODE_SCATTER_NORM_ROPE) {
        if (dtype != TF_FP16 && dtype != TF_BF16)
            return fail(TF_ERR_UNSUPPORTED, "the fused mode needs fp16 or bf16 (dtype %d)", int(dtype));
        if (D != 32 && D != 64 && D != 128 && D != 256)
            return fail(TF_ERR_UNSUPPORTED, "the fused mode is built for D in {32, 64, 128, 256}, not %d", D);
        if (!nr) return fail(TF_ERR_INVALID, "the fused mode needs norm/rope parameters");
        if (!nr->q_weight || !aligned16(nr->q_weight)) return fail(TF_ERR_ALIGNMENT, "q_weight NULL or misaligned");
        if (k && (!nr->k_weight || !aligned16(nr->k_weight)))
            return fail(TF_ERR_ALIGNMENT, "k_weight NULL or misaligned");
        if (!std::isfinite(nr->eps) || nr->eps < 0) return fail(TF_ERR_INVALID, "eps must be finite and >= 0");
        if (nr->cos_sin) {
            if (!aligned16(nr->cos_sin)) return fail(TF_ERR_ALIGNMENT, "cos_sin is not 16-byte aligned");
        } else if (!std::isfinite(nr->theta) || nr->theta <= 0) {
            return fail(TF_ERR_INVALID, "theta must be finite and > 0");
        }
        pl.fused = dtype == TF_BF16 ? tfu::Fused::kBF16 : tfu::Fused::kFP16;
    }
    // slots in launch order: V first, then Q, then K
    RelayoutParams& p = pl.p;
    const int order[3] = {2, 0, 1};
    uint32_t nx = 0;
    for (int j = 0; j < 3; ++j) {
        const int x = order[j];
        if (!src[x]) continue;
        const int slot = int(nx++);
        pl.slot_of[x] = slot;
        for (int r = 0; r < P; ++r) p.src[slot][r] = static_cast<const uint8_t*>(src[x][r]);
        p.s_b[slot] = strides[x].b * pl.sh.esize;
        p.s_t[slot] = strides[x].t * pl.sh.esize;
        p.s_h[slot] = strides[x].h * pl.sh.esize;
        // targets: contiguous [B, S, Hl, D], or [B, S, Hl, 3*D] payloads holding Q, K, V rows
        const int64_t rowb = int64_t(D) * pl.sh.esize;
        const int64_t pitch = pl.fused_layout ? 3 * rowb : rowb;
        pl.row_off[x] = pl.fused_layout ? int64_t(x) * rowb : 0;
        p.d_h[slot] = pitch;
        p.d_t[slot] = pitch * pl.sh.Hl;
        p.d_b[slot] = pitch * pl.sh.Hl * int64_t(P) * Sl;
        if (base == TF_MODE_SCATTER_NORM_ROPE && x != 2) {
            p.fused_mask |= 1u << slot;
            p.weight[slot] = x == 0 ? nr->q_weight : nr->k_weight;
        }
    }
    p.nx = nx;
    p.rope_neox = neox ? 1u : 0u;
    p.eps = nr ? nr->eps : 0.f;
    p.table = nr ? nr->cos_sin : nullptr;
    p.vec_bytes = 16;  // size limits checked for the larger vector count; re-planned at launch
    if ((s = plan_units(p, pl.sh)) != TF_OK) return s;
    pl.empty = B == 0 || Sl == 0;
    return TF_OK;
}

// Destinations of the _into / _noalloc entry points: one array per present
// tensor, or with the fused layout the P payloads in q_out (k_out, v_out NULL).
tf_status set_caller_targets(ScatterPlan& pl, void* const* q_out, void* const* k_out, void* const* v_out) {
    const int P = pl.sh.P;
    tf_status s;
    if (pl.fused_layout) {
        if (!q_out) return fail(TF_ERR_INVALID, "q_out (the payloads) is NULL");
        if (k_out || v_out) return fail(TF_ERR_INVALID, "the fused layout takes its payloads in q_out only");
        if (!pl.empty && (s = check_ptrs("q_out", q_out, P)) != TF_OK) return s;
        for (int x = 0; x < 3; ++x)
            for (int g = 0; g < P; ++g)
                pl.p.dst[pl.slot_of[x]][g] = static_cast<uint8_t*>(q_out[g]) + (q_out[g] ? pl.row_off[x] : 0);
        return TF_OK;
    }
    void* const* dsts[3] = {q_out, k_out, v_out};
    const char* names[3] = {"q_out", "k_out", "v_out"};
    for (int x = 0; x < 3; ++x) {
        if (!(pl.present & (1 << x))) continue;
        if (!dsts[x]) return fail(TF_ERR_INVALID, "%s is NULL for a present source", names[x]);
        if (!pl.empty && (s = check_ptrs(names[x], dsts[x], P)) != TF_OK) return s;
        for (int g = 0; g < P; ++g) pl.p.dst[pl.slot_of[x]][g] = static_cast<uint8_t*>(dsts[x][g]);
    }
    return TF_OK;
}

// Caller holds g_mu when the plan needs a library table.
tf_status launch_scatter(ScatterPlan& pl, const tf_norm_rope* nr, int device, cudaStream_t stream, bool capturing,
                         Table** used) {
    *used = nullptr;
    if (pl.empty) return TF_OK;
    if (pl.fused != tfu::Fused::kNone && !nr->cos_sin) {
        Table* t = nullptr;
        tf_status s = get_table(nr->theta, pl.sh.P * pl.sh.Sl, pl.sh.D, device, stream, capturing, &t);
        if (s != TF_OK) return s;
        pl.p.table = t->ptr;
        *used = t;
    }
    tf_status s = launch_planned(pl.p, pl.sh, tfu::Dir::kScatter, pl.fused, pl.sh.Sl, int64_t(pl.sh.P) * pl.sh.Sl,
                                 stream);
    if (s != TF_OK) return s;
    if (*used) record_event((*used)->last_use, stream, capturing);
    return TF_OK;
}

tf_status current_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    return TF_OK;
}

tf_status check_tag(const char* tag, std::string* out) {
    if (!tag) tag = "";
    const size_t n = strnlen(tag, 64);
    if (n > 63) return fail(TF_ERR_INVALID, "tag longer than 63 bytes");
    out->assign(tag, n);
    return TF_OK;
}

}  // namespace

extern "C" {

TF_API tf_status tf_ulysses_scatter_qkv(const char* tag, const void* const* q, const void* const* k,
                                        const void* const* v, const tf_strides* strides, int P, int B, int S_local,
                                        int H, int D, tf_dtype dtype, tf_mode mode, const tf_norm_rope* nr,
                                        void* stream, tf_targets* out) {
    CallRange call_range("tf_ulysses_scatter_qkv");
    std::string key;
    tf_status s = check_tag(tag, &key);
    if (s != TF_OK) return s;
    if (!out) return fail(TF_ERR_INVALID, "out is NULL");
    ScatterPlan pl;
    if ((s = plan_scatter(q, k, v, strides, P, B, S_local, H, D, dtype, mode, nr, &pl)) != TF_OK) return s;
    int device = 0;
    if ((s = current_device(&device)) != TF_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool cap = false;
    if ((s = capture_state(st, &cap)) != TF_OK) return s;

    std::lock_guard<std::mutex> lock(g_mu);
    size_t target_bytes = size_t(B) * size_t(P) * size_t(S_local) * size_t(pl.sh.Hl) * size_t(D) * pl.sh.esize;
    int counts[3] = {0, 0, 0};
    for (int x = 0; x < 3; ++x)
        if (pl.present & (1 << x)) counts[x] = P;
    if (pl.fused_layout) {  // P payloads holding all three tensors
        target_bytes *= 3;
        counts[1] = counts[2] = 0;
    }
    Entry* e = nullptr;
    if ((s = get_entry(key, int(mode), pl.present, pl.sh, device, target_bytes, counts, st, cap, &e)) != TF_OK)
        return s;
    const int slot_now = e->next_slot;
    void* bufs[3][TF_ULYSSES_MAX_SHARDS] = {};
    for (int x = 0; x < 3; ++x)
        for (int g = 0; g < P; ++g) {
            uint8_t* base = static_cast<uint8_t*>(slot_buffer(*e, slot_now, pl.fused_layout ? 0 : x, g));
            bufs[x][g] = base ? base + pl.row_off[x] : nullptr;
        }
    for (int x = 0; x < 3; ++x) {
        const int slot = pl.slot_of[x];
        if (slot < 0) continue;
        for (int g = 0; g < P; ++g) pl.p.dst[slot][g] = static_cast<uint8_t*>(bufs[x][g]);
    }
    Table* used = nullptr;
    if ((s = launch_scatter(pl, nr, device, st, cap, &used)) != TF_OK) return s;
    cudaError_t err = record_event(e->done, st, cap);
    if (err != cudaSuccess) return cuda_fail(err, "cudaEventRecord");
    e->last_stream = cap ? nullptr : st;  // a replay may run on any stream
    e->next_slot = (slot_now + 1) % e->slots;
    std::memset(out, 0, sizeof *out);
    for (int g = 0; g < P; ++g) {
        out->q[g] = bufs[0][g];
        out->k[g] = bufs[1][g];
        out->v[g] = bufs[2][g];
    }
    out->done = e->done;
    return TF_OK;
}

TF_API tf_status tf_ulysses_scatter_qkv_into(const void* const* q, const void* const* k, const void* const* v,
                                             const tf_strides* strides, int P, int B, int S_local, int H, int D,
                                             tf_dtype dtype, tf_mode mode, const tf_norm_rope* nr,
                                             void* const* q_out, void* const* k_out, void* const* v_out,
                                             void* stream) {
    CallRange call_range("tf_ulysses_scatter_qkv_into");
    ScatterPlan pl;
    tf_status s = plan_scatter(q, k, v, strides, P, B, S_local, H, D, dtype, mode, nr, &pl);
    if (s != TF_OK) return s;
    if ((s = set_caller_targets(pl, q_out, k_out, v_out)) != TF_OK) return s;
    int device = 0;
    if ((s = current_device(&device)) != TF_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool cap = false;
    if ((s = capture_state(st, &cap)) != TF_OK) return s;
    Table* used = nullptr;
    if (pl.fused != tfu::Fused::kNone && !nr->cos_sin) {  // the resident table lives under the lock
        std::lock_guard<std::mutex> lock(g_mu);
        return launch_scatter(pl, nr, device, st, cap, &used);
    }
    return launch_scatter(pl, nr, device, st, cap, &used);
}

// Allocation-free scatter: the library-built cos/sin table lives in the fixed
// scratch of noalloc.cu, rebuilt in stream order only when it does not already
// hold the table of this (theta, rows, D).
TF_API tf_status tf_ulysses_scatter_qkv_noalloc(const void* const* q, const void* const* k, const void* const* v,
                                                const tf_strides* strides, int P, int B, int S_local, int H, int D,
                                                tf_dtype dtype, tf_mode mode, const tf_norm_rope* nr,
                                                void* const* q_out, void* const* k_out, void* const* v_out,
                                                void* stream) {
    CallRange call_range("tf_ulysses_scatter_qkv_noalloc");
    ScatterPlan pl;
    tf_status s = plan_scatter(q, k, v, strides, P, B, S_local, H, D, dtype, mode, nr, &pl);
    if (s != TF_OK) return s;
    if ((s = set_caller_targets(pl, q_out, k_out, v_out)) != TF_OK) return s;
    const bool own_table = pl.fused != tfu::Fused::kNone && !nr->cos_sin;
    const uint64_t table_floats = uint64_t(P) * uint64_t(S_local) * uint64_t(D);
    if (own_table && table_floats > tfu::kNoAllocTableFloats)
        return fail(TF_ERR_UNSUPPORTED,
                    "P*S_local*D = %llu exceeds the fixed cos/sin scratch of %llu floats of the allocation-free entry "
                    "point",
                    (unsigned long long)table_floats, (unsigned long long)tfu::kNoAllocTableFloats);
    int device = 0;
    if ((s = current_device(&device)) != TF_OK) return s;
    if (pl.empty) return TF_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (own_table) {
        bool cap = false;
        if ((s = capture_state(st, &cap)) != TF_OK) return s;
        float* table = nullptr;
        bool built = false;
        cudaError_t e = tfu::noalloc_table(nr->theta, P * S_local, D, st, cap, &table, &built);
        if (e != cudaSuccess) return cuda_fail(e, "preparing the cos/sin table in the fixed scratch");
        if (built) g_launches.fetch_add(1);
        pl.p.table = table;
    }
    return launch_planned(pl.p, pl.sh, tfu::Dir::kScatter, pl.fused, pl.sh.Sl, int64_t(P) * S_local, st);
}

// Head-chunk scatter into caller-owned targets: heads [h0, h1) of every band.
TF_API tf_status tf_ulysses_scatter_qkv_heads_into(const void* const* q, const void* const* k, const void* const* v,
                                                   const tf_strides* strides, int P, int B, int S_local, int H,
                                                   int D, tf_dtype dtype, tf_mode mode, const tf_norm_rope* nr,
                                                   int h0, int h1, void* const* q_out, void* const* k_out,
                                                   void* const* v_out, void* stream) {
    CallRange call_range("tf_ulysses_scatter_qkv_heads_into");
    ScatterPlan pl;
    tf_status s = plan_scatter(q, k, v, strides, P, B, S_local, H, D, dtype, mode, nr, &pl);
    if (s != TF_OK) return s;
    if (h0 < 0 || h1 <= h0 || h1 > pl.sh.Hl)
        return fail(TF_ERR_INVALID, "head chunk [%d, %d) is not a non-empty range within [0, %d)", h0, h1, pl.sh.Hl);
    if ((s = set_caller_targets(pl, q_out, k_out, v_out)) != TF_OK) return s;
    // the chunk: sources start h0 heads into every band, targets h0 heads into every token;
    // bands stay Hl heads apart (Hg), a plane has (h1 - h0) heads per token
    RelayoutParams& p = pl.p;
    for (uint32_t x = 0; x < p.nx; ++x)
        for (int i = 0; i < P; ++i) {
            if (p.src[x][i]) p.src[x][i] += int64_t(h0) * p.s_h[x];
            if (p.dst[x][i]) p.dst[x][i] += int64_t(h0) * p.d_h[x];
        }
    pl.sh.Hg = pl.sh.Hl;
    pl.sh.Hl = h1 - h0;
    int device = 0;
    if ((s = current_device(&device)) != TF_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool cap = false;
    if ((s = capture_state(st, &cap)) != TF_OK) return s;
    Table* used = nullptr;
    if (pl.fused != tfu::Fused::kNone && !nr->cos_sin) {
        std::lock_guard<std::mutex> lock(g_mu);
        return launch_scatter(pl, nr, device, st, cap, &used);
    }
    return launch_scatter(pl, nr, device, st, cap, &used);
}

// All-to-all over destination-major payloads: out_g[r] = in_r[g], chunks of
// chunk_bytes.  As a scatter: B = 1, one head per band (H = P), a chunk is
// S_local rows of `row` bytes, sources read with token stride `row` and head
// stride chunk_bytes.
TF_API tf_status tf_ulysses_exchange_chunks(const void* const* src, void* const* dst, int P, size_t chunk_bytes,
                                            void* stream) {
    CallRange call_range("tf_ulysses_exchange_chunks");
    if (P < 1 || P > TF_ULYSSES_MAX_SHARDS) return fail(TF_ERR_INVALID, "P=%d outside [1, %d]", P, TF_ULYSSES_MAX_SHARDS);
    if (!src || !dst) return fail(TF_ERR_INVALID, "src or dst is NULL");
    if (chunk_bytes % 16 != 0) return fail(TF_ERR_ALIGNMENT, "chunk_bytes=%zu is not a multiple of 16", chunk_bytes);
    tf_status s;
    if (chunk_bytes > 0) {
        if ((s = check_ptrs("src", src, P)) != TF_OK) return s;
        if ((s = check_ptrs("dst", dst, P)) != TF_OK) return s;
    }
    // row: the whole chunk when it fits a stage, else the largest power of two <= a
    // stage that divides it (consecutive rows of a chunk are contiguous on both sides)
    size_t row = chunk_bytes <= tfu::kStageBytes && chunk_bytes > 0 ? chunk_bytes : size_t(tfu::kStageBytes);
    while (row > 16 && chunk_bytes % row != 0) row /= 2;
    const uint64_t rows = chunk_bytes / row;
    if (rows > uint64_t(INT32_MAX)) return fail(TF_ERR_UNSUPPORTED, "chunk_bytes too large");
    Shape sh;
    if ((s = check_shape(P, 1, int(rows), P, int(row), TF_BYTE, &sh)) != TF_OK) return s;
    RelayoutParams p{};
    p.nx = 1;
    for (int i = 0; i < P; ++i) {
        p.src[0][i] = static_cast<const uint8_t*>(src[i]);
        p.dst[0][i] = static_cast<uint8_t*>(dst[i]);
    }
    p.s_b[0] = int64_t(P) * int64_t(chunk_bytes);
    p.s_t[0] = int64_t(row);
    p.s_h[0] = int64_t(chunk_bytes);
    p.d_b[0] = int64_t(P) * int64_t(chunk_bytes);
    p.d_t[0] = int64_t(row);
    p.d_h[0] = int64_t(row);
    p.vec_bytes = 16;
    if ((s = plan_units(p, sh)) != TF_OK) return s;
    int device = 0;
    if ((s = current_device(&device)) != TF_OK) return s;
    if (rows == 0) return TF_OK;
    return launch_planned(p, sh, tfu::Dir::kScatter, tfu::Fused::kNone, int64_t(rows), int64_t(P) * int64_t(rows),
                          static_cast<cudaStream_t>(stream));
}

// Fused QKV projection: the tcgen05 GEMM whose epilogue applies the Q/K
// RMSNorm + RoPE and stores every head row into its head-group target.
#ifndef TFU_GEMM_PASS_MB
// Weight bytes per raster pass of the projection, kept in L2 while the rows stream
// past: small enough that the pass's weight columns and the row slabs in flight
// share L2 (32 MB: 1880-1900 TFLOP/s on the video-DiT projection; 48 MB 1700-1800,
// 96 MB 1670-1700, 16 MB 1710-1750).
#define TFU_GEMM_PASS_MB 32
#endif

TF_API tf_status tf_ulysses_project_qkv_into(const void* const* x, int64_t x_row_stride, const void* w_qkv,
                                             int64_t w_row_stride, int P, int B, int S_local, int hidden, int H,
                                             int D, tf_dtype dtype, tf_mode mode, const tf_norm_rope* nr,
                                             void* const* q_out, void* const* k_out, void* const* v_out,
                                             void* stream) {
    CallRange call_range("tf_ulysses_project_qkv_into");
    Shape sh;
    tf_status s = check_shape(P, B, S_local, H, D, dtype, &sh);
    if (s != TF_OK) return s;
    if (dtype != TF_BF16) return fail(TF_ERR_UNSUPPORTED, "the projection is built for bf16 (dtype %d)", int(dtype));
    if (D != tfu::kGemmHeadDim) return fail(TF_ERR_UNSUPPORTED, "the projection is built for D = 128, not %d", D);
    if (H % 2 != 0) return fail(TF_ERR_UNSUPPORTED, "the projection needs an even H (two heads per tile), not %d", H);
    if (hidden <= 0 || hidden % tfu::kGemmBK != 0)
        return fail(TF_ERR_UNSUPPORTED, "hidden=%d must be a positive multiple of %d", hidden, tfu::kGemmBK);
    const int base = int(mode) & kModeBase, flags = int(mode) & ~kModeBase;
    if (base != TF_MODE_SCATTER && base != TF_MODE_SCATTER_NORM_ROPE)
        return fail(TF_ERR_INVALID, "mode %d is not a scatter mode", int(mode));
    if (flags & ~kModeFlags) return fail(TF_ERR_INVALID, "unknown mode flags 0x%x", unsigned(flags & ~kModeFlags));
    const bool fused = base == TF_MODE_SCATTER_NORM_ROPE, neox = (flags & TF_MODE_FLAG_ROPE_NEOX) != 0;
    const bool fused_layout = (flags & TF_MODE_FLAG_FUSED_LAYOUT) != 0;
    if (neox && !fused) return fail(TF_ERR_INVALID, "TF_MODE_FLAG_ROPE_NEOX needs TF_MODE_SCATTER_NORM_ROPE");
    const bool empty = B == 0 || S_local == 0;
    if (!x || !w_qkv) return fail(TF_ERR_INVALID, "x or w_qkv is NULL");
    if (!empty && (s = check_ptrs("x", x, P)) != TF_OK) return s;
    if (!aligned16(w_qkv)) return fail(TF_ERR_ALIGNMENT, "w_qkv is not 16-byte aligned");
    if (x_row_stride < hidden || (x_row_stride * 2) % 16 != 0)
        return fail(TF_ERR_ALIGNMENT, "x_row_stride=%lld must be >= hidden and a multiple of 8 elements",
                    (long long)x_row_stride);
    if (w_row_stride < hidden || (w_row_stride * 2) % 16 != 0)
        return fail(TF_ERR_ALIGNMENT, "w_row_stride=%lld must be >= hidden and a multiple of 8 elements",
                    (long long)w_row_stride);
    if (fused) {
        if (!nr) return fail(TF_ERR_INVALID, "the fused mode needs norm/rope parameters");
        if (!nr->q_weight || !aligned16(nr->q_weight) || !nr->k_weight || !aligned16(nr->k_weight))
            return fail(TF_ERR_ALIGNMENT, "q_weight/k_weight NULL or misaligned");
        if (!std::isfinite(nr->eps) || nr->eps < 0) return fail(TF_ERR_INVALID, "eps must be finite and >= 0");
        if (nr->cos_sin) {
            if (!aligned16(nr->cos_sin)) return fail(TF_ERR_ALIGNMENT, "cos_sin is not 16-byte aligned");
        } else if (!std::isfinite(nr->theta) || nr->theta <= 0) {
            return fail(TF_ERR_INVALID, "theta must be finite and > 0");
        }
    }
    // targets: as tf_ulysses_scatter_qkv_into (all three tensors are produced)
    const int64_t rowb = int64_t(D) * 2, pitch = fused_layout ? 3 * rowb : rowb;
    void* const* outs[3] = {q_out, k_out, v_out};
    const char* names[3] = {"q_out", "k_out", "v_out"};
    tfu::GemmParams p{};
    if (fused_layout) {
        if (!q_out) return fail(TF_ERR_INVALID, "q_out (the payloads) is NULL");
        if (k_out || v_out) return fail(TF_ERR_INVALID, "the fused layout takes its payloads in q_out only");
        if (!empty && (s = check_ptrs("q_out", q_out, P)) != TF_OK) return s;
        for (int xi = 0; xi < 3; ++xi)
            for (int g = 0; g < P; ++g)
                p.dst[xi][g] = static_cast<uint8_t*>(q_out[g]) + (q_out[g] ? int64_t(xi) * rowb : 0);
    } else {
        for (int xi = 0; xi < 3; ++xi) {
            if (!outs[xi]) return fail(TF_ERR_INVALID, "%s is NULL (the projection writes Q, K and V)", names[xi]);
            if (!empty && (s = check_ptrs(names[xi], outs[xi], P)) != TF_OK) return s;
            for (int g = 0; g < P; ++g) p.dst[xi][g] = static_cast<uint8_t*>(outs[xi][g]);
        }
    }
    const uint64_t rows = uint64_t(B) * uint64_t(S_local);
    const uint64_t m_tiles = (rows + tfu::kGemmBM - 1) / tfu::kGemmBM;
    const uint64_t n_tiles = uint64_t(3) * H * D / tfu::kGemmBN;
    if (rows >= (uint64_t(1) << 31) || uint64_t(P) * m_tiles * n_tiles >= (uint64_t(1) << 31))
        return fail(TF_ERR_UNSUPPORTED, "problem exceeds 2^31 tiles or rows");
    int device = 0;
    if ((s = current_device(&device)) != TF_OK) return s;
    if (empty) return TF_OK;
    for (int r = 0; r < P; ++r)
        if (!tfu::encode_tensor_map_2d(&p.tmap_x[r], x[r], uint64_t(hidden), rows, uint64_t(x_row_stride) * 2,
                                       tfu::kGemmBM))
            return fail(TF_ERR_UNSUPPORTED, "the driver refused the tensor map of x[%d]", r);
    if (!tfu::encode_tensor_map_2d(&p.tmap_w, w_qkv, uint64_t(hidden), n_tiles * tfu::kGemmBN,
                                   uint64_t(w_row_stride) * 2, tfu::kGemmBN) ||
        !tfu::encode_tensor_map_2d(&p.tmap_w_part, w_qkv, uint64_t(hidden), n_tiles * tfu::kGemmBN,
                                   uint64_t(w_row_stride) * 2, tfu::kGemmBN / 2))
        return fail(TF_ERR_UNSUPPORTED, "the driver refused the tensor map of w_qkv");
    p.d_h = pitch;
    p.d_t = pitch * sh.Hl;
    p.d_b = pitch * sh.Hl * int64_t(P) * S_local;
    p.eps = fused ? nr->eps : 0.f;
    p.weight[0] = fused ? nr->q_weight : nullptr;
    p.weight[1] = fused ? nr->k_weight : nullptr;
    p.P = uint32_t(P);
    p.B = uint32_t(B);
    p.Sl = uint32_t(S_local);
    p.H = uint32_t(H);
    p.Hl = uint32_t(sh.Hl);
    p.K = uint32_t(hidden);
    p.rows = uint32_t(rows);
    p.m_tiles = uint32_t(m_tiles);
    p.n_tiles = uint32_t(n_tiles);
    // a pass over all row tiles reads n_group column tiles of the weight (L2-resident)
    const uint64_t wbytes_tile = uint64_t(tfu::kGemmBN) * uint64_t(hidden) * 2;
    uint64_t G = (uint64_t(TFU_GEMM_PASS_MB) << 20) / wbytes_tile;
    p.n_group = uint32_t(G < 1 ? 1 : (G > n_tiles ? n_tiles : G));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool cap = false;
    if ((s = capture_state(st, &cap)) != TF_OK) return s;
    std::lock_guard<std::mutex> lock(g_mu);
    Table* used = nullptr;
    if (fused) {
        if (nr->cos_sin) {
            p.table = nr->cos_sin;
        } else {
            if ((s = get_table(nr->theta, P * S_local, D, device, st, cap, &used)) != TF_OK) return s;
            p.table = used->ptr;
        }
    }
    cudaError_t e = tfu::launch_qkv_gemm(p, fused, neox, st);
    if (e != cudaSuccess) return cuda_fail(e, "launching the projection kernel");
    g_launches.fetch_add(1);
    if (used) record_event(used->last_use, st, cap);
    return TF_OK;
}

TF_API tf_status tf_ulysses_gather_out(const char* tag, const void* const* attn, const tf_strides* attn_strides,
                                       int P, int B, int S_local, int H, int D, tf_dtype dtype, void* const* dst,
                                       const tf_strides* dst_strides, void* stream, tf_targets* out) {
    CallRange call_range("tf_ulysses_gather_out");
    std::string key;
    tf_status s = check_tag(tag, &key);
    if (s != TF_OK) return s;
    if (!out) return fail(TF_ERR_INVALID, "out is NULL");
    Shape sh;
    if ((s = check_shape(P, B, S_local, H, D, dtype, &sh)) != TF_OK) return s;
    if (!attn) return fail(TF_ERR_INVALID, "attn is NULL");
    const bool empty = B == 0 || S_local == 0;  // nothing is dereferenced then
    if (!empty && (s = check_ptrs("attn", attn, P)) != TF_OK) return s;
    const int64_t S = int64_t(P) * S_local;
    const tf_strides a_def{S * sh.Hl * D, int64_t(sh.Hl) * D, D};
    const tf_strides o_def{int64_t(S_local) * H * D, int64_t(H) * D, D};
    const tf_strides as = attn_strides ? *attn_strides : a_def;
    const tf_strides os = dst_strides ? *dst_strides : o_def;
    if ((s = check_strides("attn", as, sh.esize, B, S, sh.Hl)) != TF_OK) return s;
    if (dst) {
        if (!empty && (s = check_ptrs("dst", dst, P)) != TF_OK) return s;
        if ((s = check_strides("dst", os, sh.esize, B, S_local, H)) != TF_OK) return s;
    }
    RelayoutParams p{};
    p.nx = 1;
    for (int g = 0; g < P; ++g) p.src[0][g] = static_cast<const uint8_t*>(attn[g]);
    p.s_b[0] = as.b * sh.esize;
    p.s_t[0] = as.t * sh.esize;
    p.s_h[0] = as.h * sh.esize;
    p.d_b[0] = os.b * sh.esize;
    p.d_t[0] = os.t * sh.esize;
    p.d_h[0] = os.h * sh.esize;
    p.vec_bytes = 16;
    if ((s = plan_units(p, sh)) != TF_OK) return s;
    int device = 0;
    if ((s = current_device(&device)) != TF_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool cap = false;
    if ((s = capture_state(st, &cap)) != TF_OK) return s;

    std::lock_guard<std::mutex> lock(g_mu);
    const size_t out_bytes = size_t(B) * size_t(S_local) * size_t(H) * size_t(D) * sh.esize;
    int counts[3] = {dst ? 0 : P, 0, 0};
    Entry* e = nullptr;
    const int present = dst ? 0 : 1;  // caller-owned outputs and cached outputs are different keys
    if ((s = get_entry(key, int(TF_MODE_GATHER), present, sh, device, dst ? 0 : out_bytes, counts, st, cap, &e)) !=
        TF_OK)
        return s;
    const int slot_now = e->next_slot;
    for (int r = 0; r < P; ++r) p.dst[0][r] = static_cast<uint8_t*>(dst ? dst[r] : slot_buffer(*e, slot_now, 0, r));
    if (!empty) {
        if ((s = launch_planned(p, sh, tfu::Dir::kGather, tfu::Fused::kNone, S, S_local, st)) != TF_OK) return s;
    }
    cudaError_t err = record_event(e->done, st, cap);
    if (err != cudaSuccess) return cuda_fail(err, "cudaEventRecord");
    e->last_stream = cap ? nullptr : st;
    e->next_slot = (slot_now + 1) % e->slots;
    std::memset(out, 0, sizeof *out);
    for (int r = 0; r < P; ++r) out->q[r] = p.dst[0][r];
    if (empty)
        for (int r = 0; r < P; ++r) out->q[r] = dst ? dst[r] : nullptr;
    out->done = e->done;
    return TF_OK;
}

TF_API tf_status tf_ulysses_rope_table(float theta, int S, int D, void* stream, const float** table) {
    CallRange call_range("tf_ulysses_rope_table");
    if (!table) return fail(TF_ERR_INVALID, "table is NULL");
    if (S < 0) return fail(TF_ERR_INVALID, "S must be >= 0");
    if (D < 2 || D > 256 || D % 2) return fail(TF_ERR_UNSUPPORTED, "D must be even and in [2, 256]");
    if (!std::isfinite(theta) || theta <= 0) return fail(TF_ERR_INVALID, "theta must be finite and > 0");
    int device = 0;
    tf_status s = current_device(&device);
    if (s != TF_OK) return s;
    bool cap = false;
    if ((s = capture_state(static_cast<cudaStream_t>(stream), &cap)) != TF_OK) return s;
    std::lock_guard<std::mutex> lock(g_mu);
    Table* t = nullptr;
    if ((s = get_table(theta, S, D, device, static_cast<cudaStream_t>(stream), cap, &t)) != TF_OK) return s;
    *table = t->ptr;
    return TF_OK;
}

TF_API tf_status tf_ulysses_cache_clear(void) {
    CallRange call_range("tf_ulysses_cache_clear");
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_entries.empty() && g_tables.empty()) return TF_OK;
    for (auto& e : g_entries) {
        if (e.done) cudaEventSynchronize(e.done);
        reclaim_entry(e, nullptr);
    }
    g_entries.clear();
    for (auto& t : g_tables) {
        dev_release(t.alloc, t.ptr, t.bytes, t.last_use, nullptr);
        if (t.last_use) cudaEventDestroy(t.last_use);
    }
    g_tables.clear();
    cudaError_t e = cudaStreamSynchronize(nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return TF_OK;
}

TF_API tf_status tf_ulysses_set_slots(const char* tag, int num_slots) {
    std::string key;
    tf_status s = check_tag(tag, &key);
    if (s != TF_OK) return s;
    if (num_slots < 1 || num_slots > TF_ULYSSES_MAX_SLOTS)
        return fail(TF_ERR_INVALID, "num_slots=%d outside [1, %d]", num_slots, TF_ULYSSES_MAX_SLOTS);
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto& ts : g_tag_slots)
        if (ts.first == key) {
            ts.second = num_slots;
            return TF_OK;
        }
    g_tag_slots.emplace_back(key, num_slots);
    return TF_OK;
}

TF_API uint64_t tf_ulysses_alloc_count(void) { return g_allocs.load(); }

TF_API int tf_ulysses_cache_entries(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    return int(g_entries.size());
}

TF_API void tf_ulysses_set_allocator(tf_alloc_fn alloc, tf_free_fn release, void* ctx) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (alloc && release) {
        g_alloc = Allocator{alloc, release, ctx};
    } else {
        g_alloc = Allocator{};
    }
}

TF_API tf_status tf_ulysses_device_status(int clear, unsigned* status) {
    if (!status) return fail(TF_ERR_INVALID, "status is NULL");
    unsigned staged = 0, gemm = 0, block = 0, block16 = 0;
    cudaError_t e = tfu::read_staged_status(&staged, clear != 0);
    if (e == cudaSuccess) e = tfu::read_gemm_status(&gemm, clear != 0);
    if (e == cudaSuccess) e = tfu::read_block_status(&block, clear != 0);
    if (e == cudaSuccess) e = tfu::read_block_status_v16(&block16, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status words");
    *status = (staged ? 1u : 0u) | (gemm ? 2u : 0u) | ((block | block16) ? 4u : 0u);
    return TF_OK;
}

TF_API tf_status tf_ulysses_selftest_wait(unsigned long long cycles, void* stream) {
    if (cycles == 0 || cycles > 1000000000ull)
        return fail(TF_ERR_INVALID, "cycles=%llu outside [1, 1e9]", (unsigned long long)cycles);
    cudaError_t e = tfu::launch_wait_selftest((long long)cycles, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "launching the bounded-wait self-test");
    g_launches.fetch_add(1);
    return TF_OK;
}

TF_API const char* tf_ulysses_last_error(void) { return g_last_error.c_str(); }

TF_API uint64_t tf_ulysses_launch_count(void) { return g_launches.load(); }

TF_API int tf_ulysses_abi_version(void) { return TF_ULYSSES_ABI_VERSION; }

}  // extern "C"
