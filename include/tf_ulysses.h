/*
 * tf_ulysses.h -- C ABI of the GB300 (sm_103a) Ulysses sequence<->head relayout.
 *
 * Ulysses sequence parallelism (TeleFuser docs, "Communication Architecture",
 * section "Sequence Parallel Communication / Ulysses") converts sequence shards
 * with all heads, [B, S_local, H, D], into head groups with the full sequence,
 * [B, S, H/P, D], with an all-to-all, and converts the attention output back with
 * the inverse all-to-all.  This library performs both relayouts for P logical
 * shards that all live in one GPU's memory: P source buffers in, P target buffers
 * out, one kernel launch per call, no peers and no collectives.
 *
 * Notation: P shards (1..8), B batch, S_local tokens per shard, S = P * S_local,
 * H heads, Hl = H / P heads per group, D head dim.  Shard r holds global tokens
 * [r*S_local, (r+1)*S_local); head group g holds heads [g*Hl, (g+1)*Hl).
 *
 *   scatter:  T_g[b, r*S_local + t, h, d] = S_r[b, t, g*Hl + h, d]
 *   gather:   O_r[b, t, g*Hl + h, d]       = A_g[b, r*S_local + t, h, d]
 *
 * Shards are concatenated in rank order (same page, "Shared Collective
 * Primitives / Equal-shape gather"); every group receives its head band of all
 * tokens (flashinfer PR #6332 commit message, "Assumptions / Exchange algorithm").
 *
 * Conventions common to every entry point:
 *  - Pointers named "device" are CUDA device (or managed) addresses of the
 *    current device.  Streams and events are passed as void* and are
 *    cudaStream_t / cudaEvent_t handles (NULL stream = legacy default stream).
 *  - Element strides are in elements, not bytes; the D dimension always has
 *    stride 1.  Every base address must be 16-byte aligned and every stride
 *    times the element size must be a multiple of 16 bytes (the kernels move
 *    16-byte vectors); otherwise TF_ERR_ALIGNMENT.
 *  - Every argument is validated before any CUDA call or launch (the pages:
 *    constraints are validated before communicating, and a started group never
 *    falls back midway -- the Ulysses section above and TeleFuser PR #27,
 *    "Additional Notes").  A non-TF_OK status therefore means nothing was written;
 *    tf_ulysses_last_error() gives a one-line reason (thread-local).
 *  - An empty problem (B == 0 or S_local == 0) is valid: nothing is launched, data
 *    pointers may then be NULL, and the completion event is still recorded.
 *  - The work is enqueued on `stream` and is asynchronous: a TF_OK return means
 *    the launch was enqueued, not that it finished.
 *  - All entry points are thread-safe; the target cache is process-wide and
 *    guarded by a mutex.
 *
 * CUDA graphs (flashinfer PR #6332 commit message, "Description", "CUDA graphs":
 * a prepared call allocates nothing; a size first seen inside a capture fails
 * rather than allocate; replays interleave with eager calls).  Every entry
 * point except tf_ulysses_scatter_qkv_noalloc (below; no claim is made for it)
 * may be called while `stream` is being captured (cudaStreamBeginCapture,
 * torch.cuda.graph).  Inside a capture the library allocates and frees nothing:
 * a call whose cache entry or RoPE table does not exist yet returns
 * TF_ERR_UNSUPPORTED before enqueuing anything -- make one eager call with the
 * same key (or tf_ulysses_rope_table) first.  Events are recorded as external
 * event nodes, so every replay records `done`; waits on events recorded outside
 * the capture become external waits.  A captured call writes the targets (the
 * rotating slot, see tf_ulysses_set_slots) current at capture time, and every
 * replay rewrites those; ordering replays against eager calls that read or
 * write the same targets is the caller's, as for two eager calls on different
 * streams.
 *
 * Kernel launches (every relayout kernel; not the projection): each launch may
 * start while the kernel before it in the stream drains (programmatic dependent
 * launch) and waits, before it touches memory, until that kernel has completed
 * and its writes are visible, so the results are those of plain stream order.
 */
#ifndef TF_ULYSSES_H
#define TF_ULYSSES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define TF_API __declspec(dllexport)
#else
#define TF_API __attribute__((visibility("default")))
#endif

#define TF_ULYSSES_ABI_VERSION 1
#define TF_ULYSSES_MAX_SHARDS 8      /* largest P */
#define TF_ULYSSES_CACHE_CAPACITY 12 /* cached target sets (the cache bound of TeleFuser PR #27, "Changes Made") */
#define TF_ULYSSES_MAX_SLOTS 8       /* rotating target sets per cache entry (tf_ulysses_set_slots) */

typedef enum tf_status {
    TF_OK = 0,
    TF_ERR_INVALID = 1,      /* bad pointer, size, dtype or mode */
    TF_ERR_DIVISIBILITY = 2, /* H % P != 0 */
    TF_ERR_ALIGNMENT = 3,    /* address or stride not a multiple of 16 bytes */
    TF_ERR_UNSUPPORTED = 4,  /* valid but not built: e.g. fused mode with D not in {32,64,128,256} */
    TF_ERR_OOM = 5,          /* the allocator returned NULL */
    TF_ERR_CUDA = 6,         /* a CUDA runtime call failed (message has the CUDA error) */
    TF_ERR_BUSY = 7          /* reserved: a cache entry could not be reclaimed in stream order */
} tf_status;

typedef enum tf_dtype {
    TF_FP16 = 0, /* IEEE binary16 */
    TF_BF16 = 1, /* bfloat16 */
    TF_FP32 = 2, /* 4-byte elements (pure relayout only) */
    TF_BYTE = 3  /* any 1-byte element, e.g. fp8 or int8 (pure relayout only) */
} tf_dtype;

/*
 * The mode of a call: one base mode, plus for the scatter entry points any of
 * the flags below OR-ed in (cast the result to tf_mode).  The whole value is
 * part of the cache key.
 *
 * TF_MODE_FLAG_FUSED_LAYOUT -- the fused receive layout (flashinfer PR #6332
 *   commit message, "Description", "Layouts": one [B, S_global, H_local, 3*D]
 *   payload, in 2-D form [B*S_global, 3*H_local*D]): head group g's targets are
 *   ONE contiguous payload [B, S, Hl, 3*D] whose head row holds the Q row, then
 *   the K row, then the V row.  q, k and v must all be present.  Cached calls
 *   return out->q[g] = the payload, out->k[g] = payload + D elements,
 *   out->v[g] = payload + 2*D elements (each a [B, S, Hl, D] view with element
 *   strides (S*Hl*3*D, Hl*3*D, 3*D, 1)); the _into/_noalloc entry points take
 *   the P payloads in q_out and require k_out == v_out == NULL.
 * TF_MODE_FLAG_ROPE_NEOX -- with TF_MODE_SCATTER_NORM_ROPE only: half-split RoPE
 *   (the GPT-NeoX pairing, not on the pages, which name the interleaved form):
 *   element i pairs with element i + D/2, both rotated by table entry i:
 *     o[i]       = round16(z[i] * cos(p, i) - z[i + D/2] * sin(p, i))
 *     o[i + D/2] = round16(z[i] * sin(p, i) + z[i + D/2] * cos(p, i))
 *   The table and every other step are those of tf_norm_rope.
 */
typedef enum tf_mode {
    TF_MODE_SCATTER = 0,                 /* bit-exact relayout of Q, K and V */
    TF_MODE_SCATTER_NORM_ROPE = 1,       /* V relayout; Q and K RMSNorm + RoPE, then relayout */
    TF_MODE_GATHER = 2,                  /* head->sequence relayout (tf_ulysses_gather_out) */
    TF_MODE_FLAG_FUSED_LAYOUT = 0x100,   /* scatter: one [B, S, Hl, 3*D] payload per head group */
    TF_MODE_FLAG_ROPE_NEOX = 0x200       /* fused scatter: half-split RoPE pairs (i, i + D/2) */
} tf_mode;

/* Element strides of a [B, tokens, heads, D] view (D stride is 1). */
typedef struct tf_strides {
    int64_t b, t, h;
} tf_strides;

/*
 * Parameters of the fused per-head RMSNorm and interleaved RoPE on Q and K
 * (flashinfer PR #6332 commit message, "Assumptions / Operator math" and
 * "Tests"): for each head row x[0..D) of Q (resp. K) at global token p = r*S_local + t,
 *   ms = mean(x^2) in fp32;  inv = 1 / sqrt(ms + eps) in fp32;
 *   y  = round16(x * inv);    z = round16(y * w)          (w: q_weight or k_weight)
 *   o[2i]   = round16(z[2i] * cos(p, i) - z[2i+1] * sin(p, i))
 *   o[2i+1] = round16(z[2i] * sin(p, i) + z[2i+1] * cos(p, i))
 * round16 = round to nearest even in the I/O dtype.  cos/sin come from an fp32
 * table; the library builds (once, then keeps resident) the table of
 * cos/sin(p * theta^(-2i/D)) evaluated in double when cos_sin is NULL.
 */
typedef struct tf_norm_rope {
    const void *q_weight;  /* device, [D] in the I/O dtype, 16-byte aligned */
    const void *k_weight;  /* device, [D] in the I/O dtype, 16-byte aligned */
    float eps;             /* finite, >= 0 (the pages use 1e-6) */
    float theta;           /* RoPE base (> 0), used when cos_sin is NULL */
    const float *cos_sin;  /* device fp32 [>= P*S_local][D/2][2] = (cos, sin) pairs, 16-byte
                              aligned, read-only; or NULL for the library-built resident table */
} tf_norm_rope;

/*
 * Targets returned by the cached entry points.  scatter: q[g], k[g], v[g] are head
 * group g's [B, S, Hl, D] contiguous buffers (NULL for an absent tensor or an
 * empty problem).  gather: q[r] is shard r's [B, S_local, H, D] output, k and v
 * unused.  `done` is the cudaEvent_t recorded on `stream` after the launch; it
 * is owned by the cache entry.  Buffers and event belong to the library's target
 * cache and stay valid until the next call with the same key rewrites them, the
 * entry is evicted (least recently used, when a 13th key arrives), or
 * tf_ulysses_cache_clear().
 */
typedef struct tf_targets {
    void *q[TF_ULYSSES_MAX_SHARDS];
    void *k[TF_ULYSSES_MAX_SHARDS];
    void *v[TF_ULYSSES_MAX_SHARDS];
    void *done;
} tf_targets;

/*
 * tf_ulysses_scatter_qkv -- sequence->head scatter of Q, K and V in one grouped
 * launch into cached final-layout targets (TeleFuser PR #27, "Changes Made":
 * direct writes into final-layout targets; a bounded cache of at most 12 target
 * sets keyed on the tag, the shape, the dtype and a mode; one grouped completion
 * for tagged Q/K/V).
 *
 *  tag        NUL-terminated cache tag (<= 63 bytes); NULL means "".  The cache key is
 *             (tag, mode, tensors present, P, B, S_local, H, D, dtype, device).
 *  q, k, v    host arrays of P device pointers; shard r's view [B, S_local, H, D].
 *             q is required; k and/or v may be NULL (then absent from the launch).
 *             Sources are read-only, owned by the caller, and must stay valid
 *             until the work on `stream` completes.
 *  strides    host array of 3 tf_strides: for q, k, v in that order (an absent
 *             tensor's entry is ignored).  All P shards of a tensor share strides;
 *             V may be a view into a fused projection (row stride 3*H*D).
 *  P, B, S_local, H, D, dtype   as in the notation above.  H % P == 0 is required.
 *  mode       TF_MODE_SCATTER or TF_MODE_SCATTER_NORM_ROPE (then nr is required,
 *             dtype is FP16 or BF16 and D is one of 32, 64, 128, 256), optionally
 *             with TF_MODE_FLAG_FUSED_LAYOUT and (fused mode only)
 *             TF_MODE_FLAG_ROPE_NEOX; other bits give TF_ERR_INVALID.
 *  nr         fused parameters, or NULL for TF_MODE_SCATTER.
 *  stream     cudaStream_t the launch (and any first-use allocation) is ordered on.
 *  out        receives the target pointers and the completion event.
 * Errors: see tf_status; nothing is written on error.  On TF_ERR_OOM nothing is
 * launched, but the least recently used entry may already have been evicted to
 * make room for the new one.  On a cache hit the targets are rewritten in place: readers of
 * the previous contents on other streams must be ordered before this call.
 */
TF_API tf_status tf_ulysses_scatter_qkv(const char *tag,
                                        const void *const *q, const void *const *k, const void *const *v,
                                        const tf_strides *strides,
                                        int P, int B, int S_local, int H, int D,
                                        tf_dtype dtype, tf_mode mode, const tf_norm_rope *nr,
                                        void *stream, tf_targets *out);

/*
 * tf_ulysses_scatter_qkv_into -- the same scatter into caller-owned targets
 * (flashinfer PR #6332, "Description": `out=` copies into caller-owned tensors).
 *  q_out, k_out, v_out  host arrays of P device pointers to contiguous [B, S, Hl, D]
 *             targets, one array per present source tensor (NULL where the source
 *             is NULL); with TF_MODE_FLAG_FUSED_LAYOUT, q_out holds the P
 *             contiguous [B, S, Hl, 3*D] payloads and k_out, v_out are NULL.
 *             Targets must not overlap the sources.
 * No cache entry and no event are involved.  The library allocates nothing when
 * mode is TF_MODE_SCATTER or nr->cos_sin is non-NULL; otherwise the first call for
 * a (theta, S, D) builds the resident RoPE table.
 */
TF_API tf_status tf_ulysses_scatter_qkv_into(const void *const *q, const void *const *k, const void *const *v,
                                             const tf_strides *strides,
                                             int P, int B, int S_local, int H, int D,
                                             tf_dtype dtype, tf_mode mode, const tf_norm_rope *nr,
                                             void *const *q_out, void *const *k_out, void *const *v_out,
                                             void *stream);

/*
 * tf_ulysses_scatter_qkv_noalloc -- the scatter of tf_ulysses_scatter_qkv_into for
 * callers that cannot allocate device memory: code running under a device-memory
 * budget reserved up front (another allocator already owns the GPU's free
 * memory, so a cudaMalloc may fail or break that accounting), and latency-bound
 * loops where the implicit device synchronisation of cudaMalloc/cudaFree is not
 * acceptable.  None of the cited pages describes a counterpart; this is an
 * interface of this library only.
 *
 * Arguments, layouts and errors are those of tf_ulysses_scatter_qkv_into; the
 * caller passes the inputs and the targets.  When mode is
 * TF_MODE_SCATTER_NORM_ROPE and nr->cos_sin is NULL, the cos/sin table comes
 * from a fixed 16 MiB device array that is part of the library (file-scope,
 * held by every GPU that loads the library until exit), so P * S_local * D must
 * not exceed 4,194,304 (4 Mi floats); larger sizes return TF_ERR_UNSUPPORTED
 * before any launch.  The array keeps the last table built into it: a call
 * whose (theta, P * S_local rows, D) it already holds (or a longer table of the
 * same theta and D) uses it as it is, after the end of that build in stream
 * order; any other call rebuilds it on `stream` first.  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library routine is called.
 * The first call on a device sets the device up with that device current: it
 * looks up the array's device address (cudaGetSymbolAddress) and creates the
 * event that marks the end of each build; make that first call before any
 * stream capture.  The address is kept for the life of the process, so a
 * device must not be reset (cudaDeviceReset) while the library is loaded.  All
 * calls share the one array: a rebuild whose work overlaps on the GPU with
 * another call's scatter (e.g. calls of different theta, rows or D on two
 * streams without ordering) races with it.
 */
TF_API tf_status tf_ulysses_scatter_qkv_noalloc(const void *const *q, const void *const *k, const void *const *v,
                                                const tf_strides *strides,
                                                int P, int B, int S_local, int H, int D,
                                                tf_dtype dtype, tf_mode mode, const tf_norm_rope *nr,
                                                void *const *q_out, void *const *k_out, void *const *v_out,
                                                void *stream);

/*
 * tf_ulysses_scatter_qkv_heads_into -- the scatter of tf_ulysses_scatter_qkv_into
 * restricted to a head chunk: heads [h0, h1) of every head band, written to the
 * same heads of the caller's final-layout targets; every other target element
 * is left as it was.  Chunks of a partition of [0, Hl), issued one after
 * another (or on several streams), produce the whole scatter, so attention on
 * the first chunk can start while later chunks still move (flashinfer PR #6332
 * commit message, "Speedup": baselines B2/B3 exchange Q/K/V per head chunk with
 * `scatter_qkv_head_chunk`).
 *  h0, h1     0 <= h0 < h1 <= Hl = H / P; otherwise TF_ERR_INVALID.
 * Every other argument, layout flag and error is that of _into; targets keep
 * their full shape ([B, S, Hl, D], or [B, S, Hl, 3*D] payloads).
 */
TF_API tf_status tf_ulysses_scatter_qkv_heads_into(const void *const *q, const void *const *k, const void *const *v,
                                                   const tf_strides *strides,
                                                   int P, int B, int S_local, int H, int D,
                                                   tf_dtype dtype, tf_mode mode, const tf_norm_rope *nr,
                                                   int h0, int h1,
                                                   void *const *q_out, void *const *k_out, void *const *v_out,
                                                   void *stream);

/*
 * tf_ulysses_exchange_chunks -- the all-to-all over destination-major payloads
 * (flashinfer UlyssesCommunicator PCIe PR description, "Transforms":
 * `exchange_chunks` takes [1, 1, world_size, chunk] to the same shape, over a
 * payload a preceding pack already laid out destination-major, and interleaves
 * nothing): for P logical ranks,
 *     dst[g][r*chunk_bytes + i] = src[r][g*chunk_bytes + i]
 *  src, dst      host arrays of P device pointers, each to P*chunk_bytes bytes,
 *                16-byte aligned; dst must not overlap src.
 *  chunk_bytes   a multiple of 16 (otherwise TF_ERR_ALIGNMENT); 0 = nothing to do.
 * Bit copy of any element type, one launch on `stream`, no allocation.
 */
TF_API tf_status tf_ulysses_exchange_chunks(const void *const *src, void *const *dst, int P, size_t chunk_bytes,
                                            void *stream);

/*
 * tf_ulysses_project_qkv_into -- the QKV projection in front of the exchange,
 * fused with it (flashinfer PR #6332 commit message, "Description": the BF16
 * QKV projection, per-head RMSNorm of Q and K, interleaved RoPE and the head
 * exchange in one call, every head band stored straight from the GEMM
 * epilogue).  For shard r, token row m = b*S_local + t and feature n:
 *     Y[m, n] = round_bf16( sum_k x_r[m, k] * w_qkv[n, k] )   (fp32 accumulation
 *                                                             on the tensor cores)
 * Features [0, HD), [HD, 2HD), [2HD, 3HD) (HD = H*D) are Q, K and V, head h at
 * features [h*D, (h+1)*D) of its block; each head row is written to head group
 * h / Hl of the targets exactly as tf_ulysses_scatter_qkv_into writes a shard's
 * head row, after the RMSNorm + RoPE of tf_norm_rope for Q and K when mode is
 * TF_MODE_SCATTER_NORM_ROPE.  The projection output is rounded to bf16 before
 * the normalisation, as a separate bf16 projection would (the pages' order
 * projection -> QK-norm -> RoPE, BF16 operands and outputs).
 *  x            host array of P device pointers; shard r's hidden states, rows
 *               m = b*S_local + t of `hidden` bf16 elements, x_row_stride elements
 *               apart (>= hidden, a multiple of 8).
 *  w_qkv        device [3*H*D][hidden] bf16 weight (the nn.Linear layout: row n
 *               is output feature n), rows w_row_stride elements apart.
 *  dtype        TF_BF16;  D = 128;  H even (two heads per output tile);
 *               hidden a multiple of 64.  Otherwise TF_ERR_UNSUPPORTED.
 *  mode, nr, q_out, k_out, v_out   as tf_ulysses_scatter_qkv_into (every target
 *               array is required: the projection produces Q, K and V).
 * One kernel launch on `stream` (plus the resident table's first build).
 */
TF_API tf_status tf_ulysses_project_qkv_into(const void *const *x, int64_t x_row_stride, const void *w_qkv,
                                             int64_t w_row_stride, int P, int B, int S_local, int hidden, int H,
                                             int D, tf_dtype dtype, tf_mode mode, const tf_norm_rope *nr,
                                             void *const *q_out, void *const *k_out, void *const *v_out,
                                             void *stream);

/*
 * tf_ulysses_gather_out -- head->sequence gather of the attention output (the
 * inverse all-to-all of the Ulysses section; TeleFuser PR #27 keeps it for the
 * output path).
 *  tag        as for scatter; the key's mode is TF_MODE_GATHER.
 *  attn       host array of P device pointers; head group g's view [B, S, Hl, D],
 *             S = P * S_local, read through attn_strides (NULL = contiguous).
 *  dst        host array of P device pointers to shard outputs [B, S_local, H, D]
 *             read through dst_strides (NULL = contiguous), or NULL: the outputs
 *             are then cached library buffers returned in out->q[r].
 *  out        receives out->q[r] (dst[r] or the cached buffer) and out->done.
 */
TF_API tf_status tf_ulysses_gather_out(const char *tag, const void *const *attn, const tf_strides *attn_strides,
                                       int P, int B, int S_local, int H, int D, tf_dtype dtype,
                                       void *const *dst, const tf_strides *dst_strides,
                                       void *stream, tf_targets *out);

/*
 * tf_ulysses_rope_table -- the resident fp32 cos/sin table [S][D/2][2] for
 * (theta, S, D) on the current device, built on `stream` on first use and kept
 * (up to 4 tables; least recently used evicted).  *table receives its device
 * address, valid until eviction or tf_ulysses_cache_clear().  D even, 2..256.
 */
TF_API tf_status tf_ulysses_rope_table(float theta, int S, int D, void *stream, const float **table);

/* Waits for every cached entry's completion event, then frees all cached
 * targets and tables.  Call it only once consumers of the targets are done. */
TF_API tf_status tf_ulysses_cache_clear(void);

/* Number of live cached target sets (0..TF_ULYSSES_CACHE_CAPACITY). */
TF_API int tf_ulysses_cache_entries(void);

/*
 * Allocator used for cached targets and tables (device memory).  alloc(bytes,
 * stream, ctx) returns a device pointer or NULL; release(ptr, bytes, stream, ctx)
 * frees it.  Passing NULL functions restores the default, cudaMallocAsync /
 * cudaFreeAsync on the calling stream.  Entries remember the allocator that made
 * them.  With a custom allocator, an evicted entry's event is synchronised on the
 * host before release() is called.
 */
typedef void *(*tf_alloc_fn)(size_t bytes, void *stream, void *ctx);
typedef void (*tf_free_fn)(void *ptr, size_t bytes, void *stream, void *ctx);
TF_API void tf_ulysses_set_allocator(tf_alloc_fn alloc, tf_free_fn release, void *ctx);

/*
 * Device status of the current device's kernels that wait in-kernel: 0 when
 * every wait completed; bit 0 is set when a bounded wait of the staged
 * (bulk-copy) kernel gave up, bit 1 when one of the projection kernel did --
 * that kernel then stopped early and its outputs are incomplete.  Bit 2 exists
 * in checked builds of the library (compiled with TFU_CHECKED=1) only: a block
 * kernel access fell outside the buffer the plan allows and was skipped.
 * Synchronises with the device.  clear != 0 resets the words after reading them.
 */
TF_API tf_status tf_ulysses_device_status(int clear, unsigned *status);

/*
 * tf_ulysses_set_slots -- rotating target sets for a tag (flashinfer PR #6332
 * commit message, "Description": outputs are views of the current receive slot
 * and stay valid until the slot is reused num_slots calls later).  Cache entries
 * created for `tag` after this call hold num_slots target sets (1..8, default 1)
 * and successive calls with the same key write them in turn: the targets a call
 * returns stay untouched for the next num_slots - 1 calls of that key.  Entries
 * that already exist keep their slot count (tf_ulysses_cache_clear drops them).
 * At most num_slots calls of one key may be captured into one graph without an
 * eager call between (later captured calls would rewrite earlier ones' slots).
 * Errors: TF_ERR_INVALID for a bad tag or num_slots.
 */
TF_API tf_status tf_ulysses_set_slots(const char *tag, int num_slots);

/* Number of device allocations (cache entries and RoPE tables) this library has
 * made in this process: unchanged across calls that hit the cache. */
TF_API uint64_t tf_ulysses_alloc_count(void);

/*
 * tf_ulysses_selftest_wait -- failure-detection self-test of the in-kernel
 * bounded waits: one thread waits, on `stream`, for a phase of an mbarrier that
 * nothing ever arrives on, with a budget of `cycles` SM clock cycles (1..1e9).
 * The wait gives up, the kernel returns, and tf_ulysses_device_status then
 * reports bit 1 (clear it with clear != 0).  Nothing faults or hangs; the
 * context stays usable.  Errors: TF_ERR_INVALID for cycles out of range.
 */
TF_API tf_status tf_ulysses_selftest_wait(unsigned long long cycles, void *stream);

/* One-line reason for the calling thread's last non-TF_OK status ("" if none). */
TF_API const char *tf_ulysses_last_error(void);

/* Number of CUDA kernels this library has launched in this process. */
TF_API uint64_t tf_ulysses_launch_count(void);

/* TF_ULYSSES_ABI_VERSION of the built library. */
TF_API int tf_ulysses_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TF_ULYSSES_H */
