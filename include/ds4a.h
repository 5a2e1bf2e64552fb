/*
 * ds4a.h — C ABI of the GB300 (sm_103a) three-tier compressed-attention step
 * of the DeepSeek V4 Flash engine described for DwarfStar (ds4).
 *
 * The step, per query token and layer (a "unit"):
 *   1. indexer score  — score every compressed KV row with the light indexer
 *                       (64 heads x 128 dims);
 *   2. top-k select   — keep the 512 highest-scoring rows;
 *   3. sparse attention — 64 query heads (head dim 512, one shared KV head)
 *                       attend over those rows plus the 128-row raw window,
 *                       in one joint softmax.
 * Sources: "Redis 作者が DeepSeek V4 専用の推論エンジンを C で書いた ―
 * DwarfStar(ds4.c) のアーキテクチャを読む【第1回/全8回】" (Qiita), §2
 * (DS4_SHAPE_FLASH), §3 (three-tier attention), §3-1 (raw sliding-window KV,
 * rows rounded through f16), §3-2 (compressed rows, ratio 4 with an indexer),
 * §3-3 (indexer keys, one per compressed row; top-k rows go to attention);
 * "antirez/ds4 深度阅读笔记", 固定模型形状 (fixed shapes).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named as device buffers are CUDA device pointers owned by the
 *    caller; the library never frees, keeps or allocates memory.  Scratch
 *    memory, where an op needs it, is a caller-provided workspace `ws` of at
 *    least ds4a_workspace_bytes(...) bytes (NULL/0 when that returns 0).
 *  - bf16 and fp16 tensors are passed as uint16_t storage words.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every op only enqueues kernels on it and returns; nothing
 *    synchronises except ds4a_get_device_status().
 *  - The shapes of the pages are fixed at compile time: 64 attention heads x
 *    512, 64 indexer heads x 128, raw window 128.  top_k is a runtime value in
 *    [1, DS4A_MAX_TOP_K] (512 on Flash, 1024 on Pro).
 *  - Arguments are validated on the host before anything is launched; a
 *    failure returns a negative status and launches nothing.  A CUDA launch
 *    error returns DS4A_ECUDA.  Conditions only the device can see (a row
 *    index out of range, an internal wait that gave up) set bits in a
 *    per-process device status word, read by ds4a_get_device_status().
 *  - Thread-safety: entry points keep no per-call host state (host globals:
 *    the test hook ds4a_debug_inject_error and the per-device set-up below)
 *    and may be called concurrently on different streams.
 *  - Per-device set-up: the first call on a device looks up, with that device
 *    current, its SM count and the device addresses of the library's own
 *    device globals (the status word; the scratch of 2'), and keeps them for
 *    the life of the process.  Make that first call before any stream
 *    capture, and do not use the library on a device after cudaDeviceReset()
 *    on it in the same process (the kept addresses would be stale).
 */
#ifndef DS4A_H
#define DS4A_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int ds4a_status;

#define DS4A_OK 0
#define DS4A_EINVAL (-1)        /* bad pointer, size, alignment or value      */
#define DS4A_EUNSUPPORTED (-2)  /* no device of compute capability 10.3       */
#define DS4A_ECUDA (-3)         /* a CUDA runtime call or launch failed        */
#define DS4A_EWORKSPACE (-4)    /* ws missing or smaller than required         */
#define DS4A_EDEVICE (-5)       /* device status word has bits set             */

/* Fixed shapes ("DwarfStar(ds4.c) のアーキテクチャを読む" §2 DS4_SHAPE_FLASH). */
#define DS4A_N_HEAD 64          /* attention query heads (n_head)              */
#define DS4A_HEAD_DIM 512       /* row width = head dim (n_head_kv = 1)        */
#define DS4A_N_INDEXER_HEAD 64  /* n_indexer_head                              */
#define DS4A_INDEXER_DIM 128    /* n_indexer_head_dim                          */
#define DS4A_N_SWA 128          /* raw sliding window (n_swa)                  */
#define DS4A_MAX_TOP_K 2048

/* Bits of the device status word. */
#define DS4A_DEV_TIMEOUT 1u     /* a bounded device-side wait gave up          */
#define DS4A_DEV_BOUNDS 2u      /* a row index or count was out of range; the
                                   offending row was masked out               */

/* Ops for ds4a_workspace_bytes. */
#define DS4A_OP_INDEXER_SCORE 0
#define DS4A_OP_TOPK_SELECT 1
#define DS4A_OP_SPARSE_ATTN_DECODE 2
#define DS4A_OP_SPARSE_ATTN_PREFILL 3
#define DS4A_OP_DENSE_ATTN_DECODE 4
#define DS4A_OP_INDEXER_TOPK 5
/* OR-ed into an attention op: the workspace of the 128-head (Pro shape) call. */
#define DS4A_OP_FLAG_128_HEADS 0x100

/* Human-readable text of a status code (static storage). */
const char *ds4a_strerror(ds4a_status status);

/* Library version, (major << 16) | minor. */
int ds4a_version(void);

/*
 * Workspace bytes an op needs for the given sizes (0: pass ws = NULL).
 * U = units, Q = queries per unit (prefill: T with U = 1), N_cap = row
 * capacity per unit.  Returns (size_t)-1 for out-of-range sizes.
 */
size_t ds4a_workspace_bytes(int op, int U, int Q, int N_cap, int top_k);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  *flags (if not NULL) receives the DS4A_DEV_* bits.  Returns DS4A_OK
 * when no bit was set, DS4A_EDEVICE when some were, DS4A_ECUDA on a CUDA error.
 *
 * There is one status word per device and process: the kernels of every
 * stream, thread and caller on the device set bits in the same word, and a
 * read returns and clears all of them, including bits raised by another
 * caller's ops (or by ops still running on other streams).  Callers sharing
 * a device should agree on one reader.
 */
ds4a_status ds4a_get_device_status(void *stream, unsigned *flags);

/*
 * Test hook: the next call of any compute entry point returns `code` without
 * launching (0 disarms).  For exercising callers' error paths on the host.
 */
void ds4a_debug_inject_error(ds4a_status code);

/*
 * Test hook for the device-side failure path: launches one thread that waits
 * on an mbarrier nothing completes, gives up after limit_us microseconds
 * (1 .. 100,000, else DS4A_EINVAL) and sets DS4A_DEV_TIMEOUT in the device
 * status word, as a compute kernel's bounded wait does when a producer never
 * arrives.  Nothing faults and the context stays usable; the next
 * ds4a_get_device_status() returns DS4A_EDEVICE with that flag and clears it.
 */
ds4a_status ds4a_debug_wait_timeout(unsigned limit_us, void *stream);

/*
 * 1. Indexer score ("DwarfStar(ds4.c) のアーキテクチャを読む" §3-3: the
 *    indexer's light query system scores each compressed row through its
 *    128-d key; the pages print no formula, this library specifies it):
 *
 *      scores[u,q,r] = sum_h w[u,q,h] * max(0, sum_d iq[u,q,h,d] * ik[u,r,d])
 *
 *    bf16 inputs, fp32 accumulation on the tensor cores, fp32 result.
 *
 *    iq      bf16 [U][Q][64][128], contiguous (device).
 *    w       fp32 [U][Q][64], contiguous (device).
 *    ik      bf16 [U][N_cap][128]; unit u starts at ik + u*ik_unit_stride
 *            elements (device).  ik and ik_unit_stride*2 bytes must be
 *            16-byte aligned (the keys are streamed by TMA).
 *    n_rows  int32 [U]: rows 0..n_rows[u]-1 of unit u exist, 0 <= n_rows[u]
 *            <= N_cap (device).  A count outside [0, N_cap] sets
 *            DS4A_DEV_BOUNDS and is clamped into it.
 *    q_pos, row_pos   NULL for decode.  For a causal prefill chunk: q_pos
 *            int32 [U][Q] query positions and row_pos int32 [U][N_cap] (unit
 *            stride N_cap) row positions; row r is visible to query q only
 *            if row_pos[u,r] <= q_pos[u,q].  Both NULL or both set.
 *    scores  fp32 [U][Q][N_cap] (device), written for r < n_rows[u];
 *            -inf marks a row the query may not see.  Entries r >= n_rows[u]
 *            are left untouched.
 *    Sizes: U >= 1, Q >= 1, N_cap >= 1, U*Q*N_cap < 2^40.
 */
ds4a_status ds4a_indexer_score(const uint16_t *iq, const float *w, const uint16_t *ik,
                               int64_t ik_unit_stride, const int32_t *n_rows,
                               const int32_t *q_pos, const int32_t *row_pos,
                               float *scores, int U, int Q, int N_cap, void *stream);

/*
 * 2. Top-k select (§3-3: only the n_indexer_top_k highest-scoring compressed
 *    rows reach the main attention).  For each (u,q): among rows r <
 *    n_rows[u] whose score is neither -inf nor NaN, select the top_k highest
 *    scores; equal scores prefer the lower row index.  -0.0 and +0.0 compare
 *    equal.
 *
 *    scores  fp32 [U][Q][N_cap] (device), as written by ds4a_indexer_score.
 *    n_rows  int32 [U] (device).  Read as soon as the kernels start, before
 *            they wait for the previous kernel on the stream: it must not be
 *            written by a kernel that lets its dependents launch early
 *            (programmatic dependent launch) right before this call.  Work
 *            without that feature, copies, and every call of this library
 *            are fine.
 *    idx     int32 [U][Q][top_k] (device): the selected row indices in
 *            ascending order, then -1 padding.
 *    count   int32 [U][Q] (device): number selected = min(top_k, visible).
 *    ws      workspace of ds4a_workspace_bytes(DS4A_OP_TOPK_SELECT, U, Q,
 *            N_cap, top_k) bytes, 256-byte aligned (device); NULL when that
 *            is 0.  Only batches of up to 76 (u,q) rows longer than 524,288
 *            scores use one (each row is then cut over several CTAs);
 *            it is at most about 5 MB whatever the sizes.
 */
ds4a_status ds4a_topk_select(const float *scores, const int32_t *n_rows, int U, int Q,
                             int N_cap, int top_k, int32_t *idx, int32_t *count,
                             void *ws, size_t ws_bytes, void *stream);

/*
 * 1+2. Indexer score and top-k select fused: the result of ds4a_indexer_score
 *    followed by ds4a_topk_select (the same idx and count, bit for bit),
 *    without materialising the scores.  While the indexer scans, each query
 *    keeps a histogram of its score keys and a threshold: a histogram bin edge
 *    with at least top_k keys at or above it among the rows counted so far
 *    (shared across the CTAs that scan one query's rows).  Only rows whose
 *    key reaches the threshold are written out, as (key, row) candidates;
 *    the threshold never passes the final k-th key, so every row of the
 *    top k, ties included, is among them, and an exact select over the
 *    candidates finishes the job.  Scores of random rows leave a few percent
 *    of the rows as candidates: instead of 8 bytes per row of score traffic,
 *    8 bytes per candidate.
 *
 *    Arguments as in 1 and 2 (no scores array).  N_cap <= 2^20 (else
 *    DS4A_EUNSUPPORTED: use 1 then 2).  ws: ds4a_workspace_bytes(
 *    DS4A_OP_INDEXER_TOPK, U, Q, N_cap, top_k) bytes (8 per row per query:
 *    the candidate lists), 256-byte aligned (device).
 */
ds4a_status ds4a_indexer_topk(const uint16_t *iq, const float *w, const uint16_t *ik,
                              int64_t ik_unit_stride, const int32_t *n_rows,
                              const int32_t *q_pos, const int32_t *row_pos, int U, int Q,
                              int N_cap, int top_k, int32_t *idx, int32_t *count,
                              void *ws, size_t ws_bytes, void *stream);

/* Capacity of the scratch array behind ds4a_topk_select_noalloc (bytes). */
#define DS4A_TOPK_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * 2'. Top-k select with no workspace argument, for callers that cannot
 *    allocate device memory.  The pages have no counterpart: this is a service
 *    of the library, not a step of the method.
 *
 *    Some callers cannot call cudaMalloc or hand over a buffer: a plugin
 *    running inside a serving engine that has reserved the device's memory for
 *    its own pool, or a runtime with a fixed memory plan decided before it
 *    starts.  This entry point computes exactly what ds4a_topk_select computes
 *    (same kernels, same results), with its scratch in a fixed array of
 *    DS4A_TOPK_NOALLOC_SCRATCH_BYTES (8 MiB) in the library's device memory;
 *    every GPU that loads the library holds that array until the process exits.
 *
 *    Limits and rules:
 *    - the request must fit: ds4a_workspace_bytes(DS4A_OP_TOPK_SELECT, U, Q,
 *      N_cap, top_k) <= DS4A_TOPK_NOALLOC_SCRATCH_BYTES, else DS4A_EWORKSPACE
 *      and nothing is launched.  Every request fits today: only up to 76
 *      rows of more than 524,288 scores use scratch, at most about 5 MB;
 *    - the first call on a device looks up the array's device address (one
 *      cudaGetSymbolAddress with that device current) and keeps it for the
 *      process: make that first call before any stream capture, and do not
 *      call it after cudaDeviceReset() on that device;
 *    - all calls on a device share the one array, and it keeps what the last
 *      call left (each call writes every scratch word it reads): calls whose
 *      kernels overlap on the GPU (other streams, other threads) race and give
 *      wrong results; serialise them on one stream;
 *    - it calls no cudaMalloc, cudaFree or allocating routine.
 *    Arguments as for ds4a_topk_select.
 */
ds4a_status ds4a_topk_select_noalloc(const float *scores, const int32_t *n_rows, int U, int Q,
                                     int N_cap, int top_k, int32_t *idx, int32_t *count,
                                     void *stream);

/*
 * 3a. Sparse attention, decode (one query per unit; §3 three tiers: the raw
 *    window plus the indexer-selected compressed rows, one KV head whose
 *    512-d rows serve as key and value).  Per unit u and head h, over the
 *    joint row set X = {rows[u, idx[u,j]] : j < count[u]} U {raw[u, s] : s <
 *    n_raw[u]}:
 *
 *      l_j = scale * q[u,h,:] . x_j ;  a = softmax(l) ;  out[u,h,:] = sum_j a_j x_j
 *      lse[u,h] = log sum_j exp(l_j)            (natural log)
 *
 *    fp32 softmax and accumulation on the tensor cores.  Compressed rows
 *    multiply in bf16; raw rows (kept rounded to f16, §3-1) multiply in fp16
 *    with q rounded to fp16 and the probabilities in fp16.  An empty row set
 *    gives out = 0, lse = -inf.
 *
 *    q       bf16 [U][64][512] (device).
 *    rows    bf16 [U][N_cap][512]; unit u at rows + u*rows_unit_stride (device).
 *    idx     int32 [U][top_k], count int32 [U] (device), as from
 *            ds4a_topk_select with Q = 1.  An index outside [0, N_cap) or a
 *            count outside [0, top_k] sets DS4A_DEV_BOUNDS and is masked.
 *    raw     fp16 [U][128][512] raw-window ring; unit u at raw +
 *            u*raw_unit_stride; slots 0..n_raw[u]-1 valid, in any order
 *            (softmax does not depend on row order) (device).
 *    n_raw   int32 [U], 0..128 (device).
 *    out     fp32 [U][64][512] (device).   lse   fp32 [U][64] or NULL (device).
 *    ws      workspace of ds4a_workspace_bytes(DS4A_OP_SPARSE_ATTN_DECODE, U, 1,
 *            N_cap, top_k) bytes: the work is cut into equal per-SM shares of
 *            64-row tiles, and a unit cut by a share boundary is computed in
 *            pieces whose partials (at most two per SM, 131,584 bytes each)
 *            are combined afterwards.  0 only when everything fits one share.
 *    q, rows, raw and out must be 16-byte aligned; with U > 1 the unit strides must
 *    be whole rows (multiples of 512 elements), at least N_cap resp. 128 rows
 *    (each buffer is addressed as one array of 512-element rows).
 */
ds4a_status ds4a_sparse_attn_decode(const uint16_t *q, const uint16_t *rows,
                                    int64_t rows_unit_stride, int N_cap,
                                    const int32_t *idx, const int32_t *count, int top_k,
                                    const uint16_t *raw, int64_t raw_unit_stride,
                                    const int32_t *n_raw, float scale, float *out, float *lse,
                                    int U, void *ws, size_t ws_bytes, void *stream);

/*
 * 3c. Dense attention of the ratio-128 layers (§3-2: the 128:1 layers keep so
 *    few compressed rows that they attend to all of them; they have no
 *    indexer).  Per unit u and head h, over the joint row set
 *    X = {rows[u, r] : r < n_rows[u]} U {raw[u, s] : s < n_raw[u]}, the same
 *    arithmetic as 3a (it is 3a with the row list 0 .. n_rows[u]-1).
 *
 *    q       bf16 [U][64][512] (device).
 *    rows    bf16 [U][N_cap][512]; unit u at rows + u*rows_unit_stride (device).
 *    n_rows  int32 [U] (device): compressed rows of unit u; a value outside
 *            [0, N_cap] sets DS4A_DEV_BOUNDS and is clamped.
 *    raw, n_raw, out, lse, strides and alignment as in 3a.
 *    ws      workspace of ds4a_workspace_bytes(DS4A_OP_DENSE_ATTN_DECODE, U, 1,
 *            N_cap, 0) bytes.
 */
ds4a_status ds4a_dense_attn_decode(const uint16_t *q, const uint16_t *rows,
                                   int64_t rows_unit_stride, int N_cap, const int32_t *n_rows,
                                   const uint16_t *raw, int64_t raw_unit_stride,
                                   const int32_t *n_raw, float scale, float *out, float *lse,
                                   int U, void *ws, size_t ws_bytes, void *stream);

/*
 * 3b. Sparse attention, one prefill chunk of T queries of one sequence (the
 *    engine prefills in 2,048-token chunks).  Query t (position q_pos[t])
 *    attends over its own selected compressed rows {rows[idx[t,j]] : j <
 *    count[t]} and the raw rows at positions q_pos[t]-127 .. q_pos[t] (the
 *    128 tokens ending at the query, its own row included) that the raw
 *    buffer holds.  Same arithmetic as 3a.
 *
 *    q       bf16 [T][64][512] (device).    q_pos  int32 [T] (device).
 *    rows    bf16 [N_cap][512] (device).
 *    idx     int32 [T][top_k], count int32 [T] (device), from the causal
 *            scores (so every selected row is at or before its query).
 *    raw     fp16 [n_raw_rows][512] (device): row i holds position raw_pos0 + i.
 *    out     fp32 [T][64][512]; lse fp32 [T][64] or NULL (device).
 *    ws      workspace of ds4a_workspace_bytes(DS4A_OP_SPARSE_ATTN_PREFILL, 1, T,
 *            N_cap, top_k) bytes.
 */
ds4a_status ds4a_sparse_attn_prefill(const uint16_t *q, const int32_t *q_pos,
                                     const uint16_t *rows, int N_cap,
                                     const int32_t *idx, const int32_t *count, int top_k,
                                     const uint16_t *raw, int32_t raw_pos0, int n_raw_rows,
                                     float scale, float *out, float *lse, int T,
                                     void *ws, size_t ws_bytes, void *stream);

/*
 * 3d. The attention calls for the Pro shape's 128 query heads (§2: the Pro
 *    variant has 128 heads and an indexer top_k of 1,024; its other attention
 *    shapes are those of Flash: one KV head of 512-d rows, a 128-row raw
 *    window).  n_head is 64 or 128 (another value returns DS4A_EUNSUPPORTED);
 *    q is [..][n_head][512], out [..][n_head][512] and lse [..][n_head]; every
 *    other argument is that of the call without the suffix, and the result of
 *    each head is what that call computes for it.  The workspace is
 *    ds4a_workspace_bytes(op | DS4A_OP_FLAG_128_HEADS, ...) for 128 heads.
 */
ds4a_status ds4a_sparse_attn_decode_heads(int n_head, const uint16_t *q, const uint16_t *rows,
                                          int64_t rows_unit_stride, int N_cap,
                                          const int32_t *idx, const int32_t *count, int top_k,
                                          const uint16_t *raw, int64_t raw_unit_stride,
                                          const int32_t *n_raw, float scale, float *out,
                                          float *lse, int U, void *ws, size_t ws_bytes,
                                          void *stream);
ds4a_status ds4a_sparse_attn_prefill_heads(int n_head, const uint16_t *q, const int32_t *q_pos,
                                           const uint16_t *rows, int N_cap, const int32_t *idx,
                                           const int32_t *count, int top_k, const uint16_t *raw,
                                           int32_t raw_pos0, int n_raw_rows, float scale,
                                           float *out, float *lse, int T, void *ws,
                                           size_t ws_bytes, void *stream);
ds4a_status ds4a_dense_attn_decode_heads(int n_head, const uint16_t *q, const uint16_t *rows,
                                         int64_t rows_unit_stride, int N_cap,
                                         const int32_t *n_rows, const uint16_t *raw,
                                         int64_t raw_unit_stride, const int32_t *n_raw,
                                         float scale, float *out, float *lse, int U, void *ws,
                                         size_t ws_bytes, void *stream);

/*
 * 4a. Raw-window push (§3-1: the raw tier keeps the K/V rows of the last 128
 *    tokens at high precision, each rounded through f16).  For each unit u,
 *    the row kv[u] of the token at position pos[u] is rounded to f16 (round
 *    to nearest even; overflow gives +-inf) and written to ring slot
 *    pos[u] % 128, and n_raw[u] = min(pos[u] + 1, 128).  Pushing positions
 *    0, 1, 2, ... leaves the ring holding the last min(P, 128) rows, the same
 *    rows as the pages' oldest-first window (which slides its rows down one
 *    slot when full), in rotated order; 3a attends to the valid slots in any
 *    order.
 *
 *    kv      fp32 [U][512] (device).
 *    raw     fp16 [U][128][512] ring; unit u at raw + u*raw_unit_stride (device).
 *    pos     int32 [U] (device): position of each unit's new row; a negative
 *            position sets DS4A_DEV_BOUNDS and writes nothing for that unit.
 *    n_raw   int32 [U] (device, written).
 *    kv and raw must be 16-byte aligned; with U > 1, raw_unit_stride is a
 *    multiple of 512 elements and at least 128 rows.
 */
ds4a_status ds4a_kv_push_raw(const float *kv, uint16_t *raw, int64_t raw_unit_stride,
                             const int32_t *pos, int32_t *n_raw, int U, void *stream);

/*
 * 4b. Compressor pooling (§3-2: the compressor folds a frontier of `ratio`
 *    token rows, 4 in the ratio-4 layers and 128 in the ratio-128 layers,
 *    into one compressed row by a softmax of learned scores).  For each unit
 *    u and column j, over the frontier rows r < ratio:
 *
 *      m = max_r score[u,r,j]
 *      out[u,j] = sum_r e^(score[u,r,j] - m) kv[u,r,j] / sum_r e^(score[u,r,j] - m)
 *
 *    and out[u,j] = 0 when no score of the column is finite.  fp32 throughout.
 *    The projections that produce kv and score, the positional bias added to
 *    the scores and the normalisation and RoPE after pooling need trained
 *    weights and are not part of this library; the FP8 round trip is 4c.
 *
 *    kv, score  fp32 [U][ratio][width] (device).    out  fp32 [U][width] (device).
 *    ratio >= 1; width a positive multiple of 4; pointers 16-byte aligned.
 */
ds4a_status ds4a_compressor_pool(const float *kv, const float *score, int ratio, int width,
                                 float *out, int U, void *stream);

/*
 * 4c. FP8 row store (§3-2: after pooling, the new compressed row is
 *    normalised, its tail rotated, and put through an FP8 quantisation round
 *    trip before it is stored).  The pages name neither the FP8 format nor
 *    its scaling; this library reads the round trip as E4M3 codes (1 sign, 4
 *    exponent bits with bias 7, 3 fraction bits; no infinities; largest
 *    finite 448) with one power-of-two scale per row, and stores exactly that
 *    pair, so the stored values are the round trip's values.  Per row r of
 *    512 fp32 values x:
 *
 *      amax        = max_d |x[r,d]|            (NaN elements do not count)
 *      e           = the smallest integer with amax <= 448 * 2^e, kept in
 *                    [-126, 127]; e = 0 when amax is 0 or infinite
 *      row_scale[r]= 2^e
 *      rows8[r,d]  = E4M3 of x[r,d] / 2^e, rounded to nearest (ties to
 *                    even), saturating at +-448; NaN stays NaN (code 0x7F)
 *
 *    The stored value of element (r,d) is e4m3(rows8[r,d]) * row_scale[r].
 *    The normalisation and RoPE before it need trained weights and are not
 *    part of this library.
 *
 *    x          fp32 [n_rows][512] (device), 16-byte aligned.
 *    rows8      uint8 [n_rows][512] (device, written), 16-byte aligned.
 *    row_scale  fp32 [n_rows] (device, written), 4-byte aligned.
 *    n_rows >= 0 (0: nothing is launched).
 */
ds4a_status ds4a_rows_to_fp8(const float *x, int64_t n_rows, uint8_t *rows8, float *row_scale,
                             void *stream);

/*
 * 3e. Sparse attention over the FP8 row store (4c): 3a and 3b with the
 *    compressed rows given as E4M3 codes and per-row scales instead of bf16.
 *    Element d of compressed row i is e4m3(rows8[i][d]) * row_scale[i]; the
 *    kernel expands each gathered row to exactly these values in bf16 (exact
 *    down to 2^-133) and multiplies as 3a does.  64 query heads.
 *
 *    The FP8 store is a storage format, not a speed-up: a row takes 516 bytes
 *    of HBM instead of 1,024 (twice the context in the same memory) and a
 *    gather moves half the bytes, but these calls are slower than 3a / 3b over
 *    bf16 rows, because the expansion of the codes sits on each row tile's
 *    critical path while the gather is latency-bound.
 *
 *    rows8      uint8 [U][N_cap][512] E4M3 codes; unit u at rows8 +
 *               u*rows_unit_stride (elements = bytes), 16-byte aligned (device).
 *    row_scale  fp32 powers of two, one per row, indexed like the rows: unit
 *               u's row r at row_scale[u*rows_unit_stride/512 + r] (device).
 *    Everything else, including the workspace (DS4A_OP_SPARSE_ATTN_DECODE /
 *    _PREFILL) and the bounds reporting, is as in 3a / 3b.
 */
ds4a_status ds4a_sparse_attn_decode_fp8(const uint16_t *q, const uint8_t *rows8,
                                        const float *row_scale, int64_t rows_unit_stride,
                                        int N_cap, const int32_t *idx, const int32_t *count,
                                        int top_k, const uint16_t *raw, int64_t raw_unit_stride,
                                        const int32_t *n_raw, float scale, float *out, float *lse,
                                        int U, void *ws, size_t ws_bytes, void *stream);
ds4a_status ds4a_sparse_attn_prefill_fp8(const uint16_t *q, const int32_t *q_pos,
                                         const uint8_t *rows8, const float *row_scale, int N_cap,
                                         const int32_t *idx, const int32_t *count, int top_k,
                                         const uint16_t *raw, int32_t raw_pos0, int n_raw_rows,
                                         float scale, float *out, float *lse, int T,
                                         void *ws, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DS4A_H */
