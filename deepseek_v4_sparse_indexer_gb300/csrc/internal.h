// Internal launcher interface between the C ABI (ds4a_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ds4a {

constexpr int kNHead = 64;       // attention heads
constexpr int kHeadDim = 512;    // row width
constexpr int kNIdxHead = 64;    // indexer heads
constexpr int kIdxDim = 128;     // indexer width
constexpr int kNSwa = 128;       // raw window
constexpr int kMaxTopK = 2048;

// ---- indexer score -------------------------------------------------------
struct IndexerArgs {
    CUtensorMap tm_ik;          // 3-D (128, N_cap, U) bf16, box (64, 128, 1), 128B swizzle
    CUtensorMap tm_iq;          // 2-D (128, U*Q*64) bf16, box (64, 64*G), 128B swizzle
    const float *w;             // [U*Q][64]
    const int32_t *n_rows;      // [U]
    const int32_t *q_pos;       // [U*Q] or null
    const int32_t *row_pos;     // [U*N_cap] or null
    float *scores;              // [U*Q][N_cap] (not written when fused)
    // Fused selection (scores not materialised): per (u,q) row R = u*Q + q,
    // candidates (order-preserving key, row) whose key reached the row's
    // running threshold, their count, the visible-row count and the threshold
    // key (all zeroed before the launch).
    int fused;
    uint2 *cand;                // [U*Q][N_cap]
    uint32_t *cand_n, *vis_n, *tau;   // [U*Q] each
    uint32_t *status;
    int U, Q, N_cap;
    int top_k;                  // fused: the k the threshold is kept for
    int G;                      // queries per UMMA (1 or 4)
    int n_groups;               // ceil(Q / G)
    int nt_cap;                 // 128-row tiles per (unit, group): ceil(N_cap / 128)
    long long total_tiles;      // U * n_groups * nt_cap, split evenly over the CTAs
    int grid;
};
cudaError_t launch_indexer_score(const IndexerArgs &a, cudaStream_t s);
cudaError_t launch_clear_counters(uint32_t *c, long long n, int num_sms, cudaStream_t s);
int indexer_group_size(int Q);                       // G for a given Q
void indexer_plan(IndexerArgs &a, int num_sms);      // fills n_groups .. grid

// ---- top-k ---------------------------------------------------------------
// Exact top-k over the fused indexer's candidate lists (see IndexerArgs).
struct TopkCandArgs {
    uint2 *cand;                // read; rows of tied keys may be compacted in place
    const uint32_t *cand_n, *vis_n;
    int R, N_cap, top_k;
    int32_t *idx, *count;
};
cudaError_t launch_topk_cand(const TopkCandArgs &a, cudaStream_t s);
// Workspace of the fused score + select for R rows: candidates [R][N_cap]
// (key, row), then cand_n, vis_n and tau [R] u32 each.
inline size_t indexer_topk_ws_bytes(long long R, int N_cap) {
    return static_cast<size_t>(R) * N_cap * 8 + static_cast<size_t>(R) * 12;
}
constexpr int kTopkCandMaxRows = 1 << 20;   // N_cap limit of the candidate path (its row bitmap)
// Very long rows (more than kTopkSplitMinRow scores) in batches of up to
// kTopkSplitMaxCtas / 2 rows: each row is cut over at least two CTAs (at most
// kTopkSplitMaxCtas in all, one wave on GB300's 152 SMs), each with a
// candidate slot of at most kTopkSplitSlot entries in the workspace, then one
// CTA per row selects.  Shorter rows need no workspace (a cluster of CTAs per
// row for a few rows, one CTA per row otherwise).
constexpr int kTopkSplitMaxCtas = 152;
constexpr int kTopkSplitSlot = 4096;
constexpr int kTopkSplitMinRow = 1 << 19;
struct TopkArgs {
    const float *scores;
    const int32_t *n_rows;
    int U, Q, N_cap, top_k;
    int32_t *idx;
    int32_t *count;
    void *ws;
    uint32_t *status;
};
size_t topk_ws_bytes(long long R, int N_cap);   // 0: no workspace
cudaError_t launch_topk(const TopkArgs &a, int num_sms, cudaStream_t s);

// ---- sparse attention ----------------------------------------------------
struct AttnArgs {
    CUtensorMap tm_q;            // 2-D (512, units*64) bf16, box (64, 64), 128B swizzle
    CUtensorMap tm_rows;         // 2-D (512, all rows) bf16, box (64, 64): whole contiguous row tiles
    CUtensorMap tm_raw;          // 2-D (512, all raw rows) fp16, box (64, 64)
    int tma_rows, tma_raw;       // the maps above are valid
    long long rows_per_unit;     // row offset between units' compressed rows (0 in prefill)
    long long raw_per_unit;      // decode: row offset between units' raw rings
    const uint16_t *q;           // [units][64][512] bf16
    const uint16_t *rows;        // bf16 rows base
    const uint8_t *rows8;        // FP8 row store (E4M3 codes [row][512]) or null: then rows is unused
    const float *row_scale;      // FP8 row store: power-of-two scale per row (same row index)
    long long rows_unit_stride;  // elements (0 in prefill: one shared row store)
    int N_cap;
    const int32_t *idx;          // [units][top_k]
    const int32_t *count;        // [units]
    int top_k;
    const uint16_t *raw;         // fp16
    long long raw_unit_stride;   // decode: per-unit ring stride (elements)
    const int32_t *n_raw;        // decode: [units]; null in prefill
    const int32_t *q_pos;        // prefill: [units]; null in decode
    int raw_pos0, n_raw_rows;    // prefill raw buffer
    float scale;
    float *out;                  // [units][64][512]
    float *lse;                  // [units][64] or null
    int units;                   // 64-head sub-units: row-side units x hsplit
    int hsplit;                  // 1 (64 heads) or 2 (128 heads: two sub-units per row-side unit)
    void *ws;
    uint32_t *status;
};
size_t attn_ws_bytes(int units, int top_k);
cudaError_t launch_debug_wait(uint32_t *status, unsigned long long limit_ns, cudaStream_t s);
cudaError_t launch_sparse_attn(const AttnArgs &a, int num_sms, cudaStream_t s);

// ---- cache producer --------------------------------------------------------
cudaError_t launch_kv_push_raw(const float *kv, uint16_t *raw, long long raw_unit_stride, const int32_t *pos,
                               int32_t *n_raw, int U, uint32_t *status, cudaStream_t s);
cudaError_t launch_compressor_pool(const float *kv, const float *score, int ratio, int width, float *out, int U,
                                   cudaStream_t s);
cudaError_t launch_rows_to_fp8(const float *x, long long n_rows, uint8_t *codes, float *row_scale, cudaStream_t s);

// ---- shared host helpers of the C ABI -------------------------------------
// Optional NVTX range around each C-ABI op (one range per call, named after
// the entry point), for timelines in Nsight Systems.  On only when the
// environment variable DS4A_NVTX is "1" when the process first calls an op;
// otherwise each call costs one test of a cached flag.
bool nvtx_enabled();
void nvtx_push(const char *name);
void nvtx_pop();
struct NvtxRange {
    bool on;
    explicit NvtxRange(const char *name) : on(nvtx_enabled()) {
        if (on) nvtx_push(name);
    }
    ~NvtxRange() {
        if (on) nvtx_pop();
    }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
// Status word address and SM count of the current device (set up on first use).
int current_device_info(uint32_t **status, int *sms);
// Returns (and disarms) the error code armed by ds4a_debug_inject_error, or 0.
int take_injected_error();
// 2-D tiled tensor map over a row-major [rows][cols] 16-bit matrix (row pitch
// cols*2 bytes) with the 128-byte swizzle.  False if the driver rejects it.
bool encode_2d_sw128(CUtensorMap *m, bool f16, const void *base, unsigned long long cols, unsigned long long rows,
                     unsigned box_cols, unsigned box_rows);

}  // namespace ds4a
