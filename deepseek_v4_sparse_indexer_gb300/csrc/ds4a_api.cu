// C ABI of the ds4a library: argument validation, TMA descriptor encoding and
// kernel launches.  Every function validates on the host before launching and
// returns a ds4a_status; nothing here synchronises except
// ds4a_get_device_status().
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/ds4a.h"
#include "internal.h"

using namespace ds4a;

namespace {

// Per-process device status word: kernels OR DS4A_DEV_* bits into it.
__device__ uint32_t g_device_status;

std::atomic<int> g_inject{0};

struct DevInfo {
    bool init = false;
    int sms = 0;
    uint32_t *status = nullptr;
};
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Looks up (once per device) the SM count and the status word's address on
// the current device.  Only compute capability 10.3 (GB300) runs this code.
ds4a_status current_device(DevInfo **out) {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return DS4A_ECUDA;
    if (d < 0 || d >= kMaxDevices) return DS4A_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo &di = g_dev[d];
    if (!di.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess)
            return DS4A_ECUDA;
        if (major != 10 || minor != 3) return DS4A_EUNSUPPORTED;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return DS4A_ECUDA;
        di.status = static_cast<uint32_t *>(p);
        di.sms = sms;
        di.init = true;
    }
    *out = &di;
    return DS4A_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// bf16 tensor map with 128-byte swizzle and a 64-element inner box.
bool encode_bf16(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides_bytes,
                 const cuuint32_t *box) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint32_t es[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides_bytes, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

ds4a_status take_injected() {
    const int c = g_inject.exchange(0);
    return c;
}

}  // namespace

namespace ds4a {
bool nvtx_enabled() {
    static const bool on = [] {
        const char *v = std::getenv("DS4A_NVTX");
        return v != nullptr && std::strcmp(v, "1") == 0;
    }();
    return on;
}
void nvtx_push(const char *name) { nvtxRangePushA(name); }
void nvtx_pop() { nvtxRangePop(); }
int current_device_info(uint32_t **status, int *sms) {
    DevInfo *di = nullptr;
    const ds4a_status st = current_device(&di);
    if (st) return st;
    *status = di->status;
    *sms = di->sms;
    return DS4A_OK;
}
int take_injected_error() { return take_injected(); }
bool encode_2d_sw128(CUtensorMap *m, bool f16, const void *base, unsigned long long cols, unsigned long long rows,
                     unsigned box_cols, unsigned box_rows) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return f(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace ds4a

extern "C" {

const char *ds4a_strerror(ds4a_status s) {
    switch (s) {
    case DS4A_OK: return "ok";
    case DS4A_EINVAL: return "invalid argument (null pointer, size, alignment or value out of range)";
    case DS4A_EUNSUPPORTED: return "unsupported device (needs compute capability 10.3, sm_103a)";
    case DS4A_ECUDA: return "CUDA runtime error or kernel launch failure";
    case DS4A_EWORKSPACE: return "workspace missing, misaligned or too small";
    case DS4A_EDEVICE: return "device status word has error bits set";
    default: return "unknown ds4a status";
    }
}

int ds4a_version(void) { return (1 << 16) | 0; }

size_t ds4a_workspace_bytes(int op, int U, int Q, int N_cap, int top_k) {
    if (U < 1 || Q < 1 || N_cap < 1) return static_cast<size_t>(-1);
    // 128 heads run as two 64-head sub-units per unit (the attention ops only)
    const int h = (op & DS4A_OP_FLAG_128_HEADS) ? 2 : 1;
    op &= ~DS4A_OP_FLAG_128_HEADS;
    if (h == 2 && op != DS4A_OP_SPARSE_ATTN_DECODE && op != DS4A_OP_SPARSE_ATTN_PREFILL &&
        op != DS4A_OP_DENSE_ATTN_DECODE)
        return static_cast<size_t>(-1);
    if (static_cast<long long>(U) * h > 0x7fffffffLL) return static_cast<size_t>(-1);
    U *= h;
    switch (op) {
    case DS4A_OP_INDEXER_SCORE: return 0;
    case DS4A_OP_TOPK_SELECT:
        if (top_k < 1 || top_k > DS4A_MAX_TOP_K) return static_cast<size_t>(-1);
        return topk_ws_bytes(static_cast<long long>(U) * Q, N_cap);
    case DS4A_OP_SPARSE_ATTN_DECODE:
        if (top_k < 1 || top_k > DS4A_MAX_TOP_K) return static_cast<size_t>(-1);
        return attn_ws_bytes(U, top_k);
    case DS4A_OP_DENSE_ATTN_DECODE: return attn_ws_bytes(U, N_cap);
    case DS4A_OP_INDEXER_TOPK:
        if (top_k < 1 || top_k > DS4A_MAX_TOP_K) return static_cast<size_t>(-1);
        return indexer_topk_ws_bytes(static_cast<long long>(U) * Q, N_cap);
    case DS4A_OP_SPARSE_ATTN_PREFILL: {
        if (top_k < 1 || top_k > DS4A_MAX_TOP_K) return static_cast<size_t>(-1);
        const long long units = static_cast<long long>(U) * Q;
        if (units > 0x7fffffffLL) return static_cast<size_t>(-1);
        return attn_ws_bytes(static_cast<int>(units), top_k);
    }
    default: return static_cast<size_t>(-1);
    }
}

ds4a_status ds4a_get_device_status(void *stream, unsigned *flags) {
    DevInfo *di = nullptr;
    ds4a_status st = current_device(&di);
    if (st) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DS4A_ECUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, di->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DS4A_ECUDA;
    if (v && cudaMemset(di->status, 0, sizeof(v)) != cudaSuccess) return DS4A_ECUDA;
    if (flags) *flags = v;
    return v ? DS4A_EDEVICE : DS4A_OK;
}

void ds4a_debug_inject_error(ds4a_status code) { g_inject.store(code); }

ds4a_status ds4a_debug_wait_timeout(unsigned limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 100000) return DS4A_EINVAL;
    DevInfo *di = nullptr;
    if (ds4a_status st = current_device(&di)) return st;
    return ds4a::launch_debug_wait(di->status, 1000ull * limit_us, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DS4A_OK
               : DS4A_ECUDA;
}

}  // extern "C"

namespace {
// Checks and fills everything of an indexer launch but the outputs.
ds4a_status indexer_setup(IndexerArgs &a, DevInfo **dio, const uint16_t *iq, const float *w, const uint16_t *ik,
                          int64_t ik_unit_stride, const int32_t *n_rows, const int32_t *q_pos,
                          const int32_t *row_pos, int U, int Q, int N_cap) {
    if (!iq || !w || !ik || !n_rows) return DS4A_EINVAL;
    if ((q_pos == nullptr) != (row_pos == nullptr)) return DS4A_EINVAL;
    if (U < 1 || Q < 1 || N_cap < 1) return DS4A_EINVAL;
    if (static_cast<long long>(U) * Q > (1LL << 24)) return DS4A_EINVAL;           // TMA row coordinate
    if (static_cast<long long>(U) * Q * N_cap >= (1LL << 40)) return DS4A_EINVAL;
    if (!aligned(iq, 16) || !aligned(ik, 16) || !aligned(w, 4)) return DS4A_EINVAL;
    if (U > 1 && (ik_unit_stride < static_cast<int64_t>(N_cap) * kIdxDim || (ik_unit_stride & 7) != 0))
        return DS4A_EINVAL;
    DevInfo *di = nullptr;
    if (ds4a_status st = current_device(&di)) return st;
    *dio = di;
    a.w = w;
    a.n_rows = n_rows;
    a.q_pos = q_pos;
    a.row_pos = row_pos;
    a.status = di->status;
    a.U = U;
    a.Q = Q;
    a.N_cap = N_cap;
    indexer_plan(a, di->sms);
    const int64_t unit_stride = U > 1 ? ik_unit_stride : static_cast<int64_t>(N_cap) * kIdxDim;
    {
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(kIdxDim), static_cast<cuuint64_t>(N_cap),
                              static_cast<cuuint64_t>(U)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(kIdxDim) * 2, static_cast<cuuint64_t>(unit_stride) * 2};
        cuuint32_t box[3] = {64, 128, 1};
        if (!encode_bf16(&a.tm_ik, ik, 3, dims, strides, box)) return DS4A_EINVAL;
    }
    {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(kIdxDim),
                              static_cast<cuuint64_t>(U) * static_cast<cuuint64_t>(Q) * kNIdxHead};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(kIdxDim) * 2};
        cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kNIdxHead * a.G)};
        if (!encode_bf16(&a.tm_iq, iq, 2, dims, strides, box)) return DS4A_EINVAL;
    }
    return DS4A_OK;
}
}  // namespace

extern "C" {

ds4a_status ds4a_indexer_score(const uint16_t *iq, const float *w, const uint16_t *ik, int64_t ik_unit_stride,
                               const int32_t *n_rows, const int32_t *q_pos, const int32_t *row_pos, float *scores,
                               int U, int Q, int N_cap, void *stream) {
    const NvtxRange nvtx_range("ds4a_indexer_score");
    if (ds4a_status inj = take_injected()) return inj;
    if (!scores || !aligned(scores, 4)) return DS4A_EINVAL;
    IndexerArgs a{};
    DevInfo *di = nullptr;
    if (ds4a_status st = indexer_setup(a, &di, iq, w, ik, ik_unit_stride, n_rows, q_pos, row_pos, U, Q, N_cap))
        return st;
    a.scores = scores;
    if (a.total_tiles == 0) return DS4A_OK;
    return launch_indexer_score(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DS4A_OK : DS4A_ECUDA;
}

ds4a_status ds4a_indexer_topk(const uint16_t *iq, const float *w, const uint16_t *ik, int64_t ik_unit_stride,
                              const int32_t *n_rows, const int32_t *q_pos, const int32_t *row_pos, int U, int Q,
                              int N_cap, int top_k, int32_t *idx, int32_t *count, void *ws, size_t ws_bytes,
                              void *stream) {
    const NvtxRange nvtx_range("ds4a_indexer_topk");
    if (ds4a_status inj = take_injected()) return inj;
    if (!idx || !count || top_k < 1 || top_k > DS4A_MAX_TOP_K) return DS4A_EINVAL;
    if (N_cap > kTopkCandMaxRows) return DS4A_EUNSUPPORTED;
    IndexerArgs a{};
    DevInfo *di = nullptr;
    if (ds4a_status st = indexer_setup(a, &di, iq, w, ik, ik_unit_stride, n_rows, q_pos, row_pos, U, Q, N_cap))
        return st;
    const long long R = static_cast<long long>(U) * Q;
    const size_t need = indexer_topk_ws_bytes(R, N_cap);
    if (!ws || ws_bytes < need || !aligned(ws, 256)) return DS4A_EWORKSPACE;
    uint8_t *p = static_cast<uint8_t *>(ws);
    a.fused = 1;
    a.top_k = top_k;
    a.cand = reinterpret_cast<uint2 *>(p);
    uint32_t *counters = reinterpret_cast<uint32_t *>(p + static_cast<size_t>(R) * N_cap * 8);
    a.cand_n = counters;
    a.vis_n = counters + R;
    a.tau = counters + 2 * R;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_clear_counters(counters, 3 * R, di->sms, s) != cudaSuccess) return DS4A_ECUDA;
    if (a.total_tiles > 0 && launch_indexer_score(a, s) != cudaSuccess) return DS4A_ECUDA;
    TopkCandArgs t{a.cand, a.cand_n, a.vis_n, static_cast<int>(R), N_cap, top_k, idx, count};
    return launch_topk_cand(t, s) == cudaSuccess ? DS4A_OK : DS4A_ECUDA;
}

ds4a_status ds4a_topk_select(const float *scores, const int32_t *n_rows, int U, int Q, int N_cap, int top_k,
                             int32_t *idx, int32_t *count, void *ws, size_t ws_bytes, void *stream) {
    const NvtxRange nvtx_range("ds4a_topk_select");
    if (ds4a_status inj = take_injected()) return inj;
    if (!scores || !n_rows || !idx || !count) return DS4A_EINVAL;
    if (U < 1 || Q < 1 || N_cap < 1 || top_k < 1 || top_k > DS4A_MAX_TOP_K) return DS4A_EINVAL;
    if (static_cast<long long>(U) * Q > (1LL << 24)) return DS4A_EINVAL;
    if (!aligned(scores, 4)) return DS4A_EINVAL;
    const size_t need = topk_ws_bytes(static_cast<long long>(U) * Q, N_cap);
    if (need && (!ws || ws_bytes < need || !aligned(ws, 256))) return DS4A_EWORKSPACE;
    DevInfo *di = nullptr;
    if (ds4a_status st = current_device(&di)) return st;
    TopkArgs a{scores, n_rows, U, Q, N_cap, top_k, idx, count, ws, di->status};
    return launch_topk(a, di->sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DS4A_OK : DS4A_ECUDA;
}

namespace {
ds4a_status check_attn_common(const uint16_t *q, const uint16_t *rows, int N_cap, const int32_t *idx,
                              const int32_t *count, int top_k, float *out) {
    if (!q || !rows || !idx || !count || !out) return DS4A_EINVAL;
    if (N_cap < 1 || top_k < 1 || top_k > DS4A_MAX_TOP_K) return DS4A_EINVAL;
    if (!aligned(q, 16) || !aligned(rows, 16) || !aligned(out, 16)) return DS4A_EINVAL;
    return DS4A_OK;
}
}  // namespace

namespace {
// Decode attention over an explicit row list (idx, count, top_k) or, with
// idx == nullptr, over rows 0 .. count[u]-1 (count = n_rows, top_k = N_cap).
// rows8 != nullptr: the compressed rows are the FP8 store (rows8, row_scale)
// and rows is not read.
ds4a_status attn_decode(int hsplit, const uint16_t *q, const uint16_t *rows, int64_t rows_unit_stride, int N_cap,
                        const int32_t *idx, const int32_t *count, int top_k, const uint16_t *raw,
                        int64_t raw_unit_stride, const int32_t *n_raw, float scale, float *out, float *lse, int U,
                        void *ws, size_t ws_bytes, void *stream, const uint8_t *rows8 = nullptr,
                        const float *row_scale = nullptr) {
    if (!raw || !n_raw || U < 1) return DS4A_EINVAL;
    if (static_cast<long long>(U) * hsplit * kNHead >= (1LL << 31)) return DS4A_EINVAL;
    if (!aligned(raw, 16)) return DS4A_EINVAL;
    if (U > 1 && (rows_unit_stride < static_cast<int64_t>(N_cap) * kHeadDim || rows_unit_stride % kHeadDim ||
                  raw_unit_stride < static_cast<int64_t>(kNSwa) * kHeadDim || raw_unit_stride % kHeadDim))
        return DS4A_EINVAL;
    const long long rows_per_unit = U > 1 ? rows_unit_stride / kHeadDim : N_cap;
    const long long raw_per_unit = U > 1 ? raw_unit_stride / kHeadDim : kNSwa;
    const long long total_rows = (static_cast<long long>(U) - 1) * rows_per_unit + N_cap;
    const long long total_raw = (static_cast<long long>(U) - 1) * raw_per_unit + kNSwa;
    if (total_rows >= (1LL << 31) || total_raw >= (1LL << 31) || static_cast<long long>(U) * kNHead >= (1LL << 31))
        return DS4A_EINVAL;
    if (!(scale == scale)) return DS4A_EINVAL;
    const size_t need = attn_ws_bytes(U * hsplit, top_k);
    if (need && (!ws || ws_bytes < need || !aligned(ws, 256))) return DS4A_EWORKSPACE;
    DevInfo *di = nullptr;
    if (ds4a_status st = current_device(&di)) return st;
    AttnArgs a{};
    a.q = q;
    a.rows = rows;
    a.rows_unit_stride = rows_unit_stride;
    a.N_cap = N_cap;
    a.idx = idx;
    a.count = count;
    a.top_k = top_k;
    a.raw = raw;
    a.raw_unit_stride = raw_unit_stride;
    a.n_raw = n_raw;
    a.q_pos = nullptr;
    a.scale = scale;
    a.out = out;
    a.lse = lse;
    a.units = U * hsplit;
    a.hsplit = hsplit;
    a.ws = ws;
    a.status = di->status;
    a.rows_per_unit = rows_per_unit;
    a.raw_per_unit = raw_per_unit;
    a.rows8 = rows8;
    a.row_scale = row_scale;
    if (!encode_2d_sw128(&a.tm_q, false, q, kHeadDim, static_cast<unsigned long long>(U) * hsplit * kNHead, 64, 64))
        return DS4A_EINVAL;
    a.tma_rows = !rows8 &&
                 encode_2d_sw128(&a.tm_rows, false, rows, kHeadDim, static_cast<unsigned long long>(total_rows), 64, 64);
    a.tma_raw = encode_2d_sw128(&a.tm_raw, true, raw, kHeadDim, static_cast<unsigned long long>(total_raw), 64, 64);
    return launch_sparse_attn(a, di->sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DS4A_OK : DS4A_ECUDA;
}
}  // namespace

ds4a_status ds4a_sparse_attn_decode_heads(int n_head, const uint16_t *q, const uint16_t *rows,
                                          int64_t rows_unit_stride, int N_cap, const int32_t *idx,
                                          const int32_t *count, int top_k, const uint16_t *raw,
                                          int64_t raw_unit_stride, const int32_t *n_raw, float scale, float *out,
                                          float *lse, int U, void *ws, size_t ws_bytes, void *stream) {
    const NvtxRange nvtx_range("ds4a_sparse_attn_decode_heads");
    if (ds4a_status inj = take_injected()) return inj;
    if (n_head != 64 && n_head != 128) return DS4A_EUNSUPPORTED;
    if (ds4a_status st = check_attn_common(q, rows, N_cap, idx, count, top_k, out)) return st;
    return attn_decode(n_head / kNHead, q, rows, rows_unit_stride, N_cap, idx, count, top_k, raw, raw_unit_stride,
                       n_raw, scale, out, lse, U, ws, ws_bytes, stream);
}

ds4a_status ds4a_sparse_attn_decode(const uint16_t *q, const uint16_t *rows, int64_t rows_unit_stride, int N_cap,
                                    const int32_t *idx, const int32_t *count, int top_k, const uint16_t *raw,
                                    int64_t raw_unit_stride, const int32_t *n_raw, float scale, float *out,
                                    float *lse, int U, void *ws, size_t ws_bytes, void *stream) {
    return ds4a_sparse_attn_decode_heads(64, q, rows, rows_unit_stride, N_cap, idx, count, top_k, raw,
                                         raw_unit_stride, n_raw, scale, out, lse, U, ws, ws_bytes, stream);
}

ds4a_status ds4a_sparse_attn_decode_fp8(const uint16_t *q, const uint8_t *rows8, const float *row_scale,
                                        int64_t rows_unit_stride, int N_cap, const int32_t *idx,
                                        const int32_t *count, int top_k, const uint16_t *raw,
                                        int64_t raw_unit_stride, const int32_t *n_raw, float scale, float *out,
                                        float *lse, int U, void *ws, size_t ws_bytes, void *stream) {
    const NvtxRange nvtx_range("ds4a_sparse_attn_decode_fp8");
    if (ds4a_status inj = take_injected()) return inj;
    const uint16_t *as16 = reinterpret_cast<const uint16_t *>(rows8);   // only its pointer checks are used
    if (ds4a_status st = check_attn_common(q, as16, N_cap, idx, count, top_k, out)) return st;
    if (!row_scale || !aligned(row_scale, 4)) return DS4A_EINVAL;
    return attn_decode(1, q, as16, rows_unit_stride, N_cap, idx, count, top_k, raw, raw_unit_stride, n_raw, scale,
                       out, lse, U, ws, ws_bytes, stream, rows8, row_scale);
}

ds4a_status ds4a_dense_attn_decode_heads(int n_head, const uint16_t *q, const uint16_t *rows,
                                         int64_t rows_unit_stride, int N_cap, const int32_t *n_rows,
                                         const uint16_t *raw, int64_t raw_unit_stride, const int32_t *n_raw,
                                         float scale, float *out, float *lse, int U, void *ws, size_t ws_bytes,
                                         void *stream) {
    const NvtxRange nvtx_range("ds4a_dense_attn_decode_heads");
    if (ds4a_status inj = take_injected()) return inj;
    if (n_head != 64 && n_head != 128) return DS4A_EUNSUPPORTED;
    if (!q || !rows || !n_rows || !out || N_cap < 1) return DS4A_EINVAL;
    if (!aligned(q, 16) || !aligned(rows, 16) || !aligned(out, 16)) return DS4A_EINVAL;
    return attn_decode(n_head / kNHead, q, rows, rows_unit_stride, N_cap, nullptr, n_rows, N_cap, raw,
                       raw_unit_stride, n_raw, scale, out, lse, U, ws, ws_bytes, stream);
}

ds4a_status ds4a_dense_attn_decode(const uint16_t *q, const uint16_t *rows, int64_t rows_unit_stride, int N_cap,
                                   const int32_t *n_rows, const uint16_t *raw, int64_t raw_unit_stride,
                                   const int32_t *n_raw, float scale, float *out, float *lse, int U, void *ws,
                                   size_t ws_bytes, void *stream) {
    return ds4a_dense_attn_decode_heads(64, q, rows, rows_unit_stride, N_cap, n_rows, raw, raw_unit_stride, n_raw,
                                        scale, out, lse, U, ws, ws_bytes, stream);
}

namespace {
ds4a_status attn_prefill(int hsplit, const uint16_t *q, const int32_t *q_pos, const uint16_t *rows, int N_cap,
                         const int32_t *idx, const int32_t *count, int top_k, const uint16_t *raw, int32_t raw_pos0,
                         int n_raw_rows, float scale, float *out, float *lse, int T, void *ws, size_t ws_bytes,
                         void *stream, const uint8_t *rows8, const float *row_scale) {
    const int n_head = hsplit * kNHead;
    if (!q_pos || T < 1 || n_raw_rows < 0) return DS4A_EINVAL;
    if (n_raw_rows > 0 && (!raw || !aligned(raw, 16))) return DS4A_EINVAL;
    if (!(scale == scale)) return DS4A_EINVAL;
    if (static_cast<long long>(T) * n_head >= (1LL << 31)) return DS4A_EINVAL;
    const size_t need = attn_ws_bytes(T * hsplit, top_k);
    if (need && (!ws || ws_bytes < need || !aligned(ws, 256))) return DS4A_EWORKSPACE;
    DevInfo *di = nullptr;
    if (ds4a_status st = current_device(&di)) return st;
    AttnArgs a{};
    a.q = q;
    a.rows = rows;
    a.rows_unit_stride = 0;
    a.N_cap = N_cap;
    a.idx = idx;
    a.count = count;
    a.top_k = top_k;
    a.raw = n_raw_rows > 0 ? raw : q;    // never read when the buffer is empty
    a.raw_unit_stride = 0;
    a.n_raw = nullptr;
    a.q_pos = q_pos;
    a.raw_pos0 = raw_pos0;
    a.n_raw_rows = n_raw_rows;
    a.scale = scale;
    a.out = out;
    a.lse = lse;
    a.units = T * hsplit;
    a.hsplit = hsplit;
    a.ws = ws;
    a.status = di->status;
    a.rows_per_unit = 0;
    a.raw_per_unit = 0;
    a.rows8 = rows8;
    a.row_scale = row_scale;
    if (!encode_2d_sw128(&a.tm_q, false, q, kHeadDim, static_cast<unsigned long long>(T) * n_head, 64, 64))
        return DS4A_EINVAL;
    a.tma_rows = !rows8 &&
                 encode_2d_sw128(&a.tm_rows, false, rows, kHeadDim, static_cast<unsigned long long>(N_cap), 64, 64);
    a.tma_raw = n_raw_rows > 0 &&
                encode_2d_sw128(&a.tm_raw, true, raw, kHeadDim, static_cast<unsigned long long>(n_raw_rows), 64, 64);
    return launch_sparse_attn(a, di->sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DS4A_OK : DS4A_ECUDA;
}
}  // namespace

ds4a_status ds4a_sparse_attn_prefill_heads(int n_head, const uint16_t *q, const int32_t *q_pos,
                                           const uint16_t *rows, int N_cap, const int32_t *idx,
                                           const int32_t *count, int top_k, const uint16_t *raw, int32_t raw_pos0,
                                           int n_raw_rows, float scale, float *out, float *lse, int T, void *ws,
                                           size_t ws_bytes, void *stream) {
    const NvtxRange nvtx_range("ds4a_sparse_attn_prefill_heads");
    if (ds4a_status inj = take_injected()) return inj;
    if (n_head != 64 && n_head != 128) return DS4A_EUNSUPPORTED;
    if (ds4a_status st = check_attn_common(q, rows, N_cap, idx, count, top_k, out)) return st;
    return attn_prefill(n_head / kNHead, q, q_pos, rows, N_cap, idx, count, top_k, raw, raw_pos0, n_raw_rows, scale,
                        out, lse, T, ws, ws_bytes, stream, nullptr, nullptr);
}

ds4a_status ds4a_sparse_attn_prefill_fp8(const uint16_t *q, const int32_t *q_pos, const uint8_t *rows8,
                                         const float *row_scale, int N_cap, const int32_t *idx,
                                         const int32_t *count, int top_k, const uint16_t *raw, int32_t raw_pos0,
                                         int n_raw_rows, float scale, float *out, float *lse, int T, void *ws,
                                         size_t ws_bytes, void *stream) {
    const NvtxRange nvtx_range("ds4a_sparse_attn_prefill_fp8");
    if (ds4a_status inj = take_injected()) return inj;
    const uint16_t *as16 = reinterpret_cast<const uint16_t *>(rows8);   // only its pointer checks are used
    if (ds4a_status st = check_attn_common(q, as16, N_cap, idx, count, top_k, out)) return st;
    if (!row_scale || !aligned(row_scale, 4)) return DS4A_EINVAL;
    return attn_prefill(1, q, q_pos, as16, N_cap, idx, count, top_k, raw, raw_pos0, n_raw_rows, scale, out, lse, T,
                        ws, ws_bytes, stream, rows8, row_scale);
}

ds4a_status ds4a_sparse_attn_prefill(const uint16_t *q, const int32_t *q_pos, const uint16_t *rows, int N_cap,
                                     const int32_t *idx, const int32_t *count, int top_k, const uint16_t *raw,
                                     int32_t raw_pos0, int n_raw_rows, float scale, float *out, float *lse, int T,
                                     void *ws, size_t ws_bytes, void *stream) {
    return ds4a_sparse_attn_prefill_heads(64, q, q_pos, rows, N_cap, idx, count, top_k, raw, raw_pos0, n_raw_rows,
                                          scale, out, lse, T, ws, ws_bytes, stream);
}

ds4a_status ds4a_rows_to_fp8(const float *x, int64_t n_rows, uint8_t *rows8, float *row_scale, void *stream) {
    const NvtxRange nvtx_range("ds4a_rows_to_fp8");
    if (ds4a_status inj = take_injected()) return inj;
    if (n_rows < 0 || (n_rows > 0 && (!x || !rows8 || !row_scale))) return DS4A_EINVAL;
    if (n_rows == 0) return DS4A_OK;
    if (!aligned(x, 16) || !aligned(rows8, 16) || !aligned(row_scale, 4)) return DS4A_EINVAL;
    if (n_rows >= (1LL << 40) / kHeadDim) return DS4A_EINVAL;
    DevInfo *di = nullptr;
    if (ds4a_status st = current_device(&di)) return st;
    return launch_rows_to_fp8(x, n_rows, rows8, row_scale, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DS4A_OK
               : DS4A_ECUDA;
}

ds4a_status ds4a_kv_push_raw(const float *kv, uint16_t *raw, int64_t raw_unit_stride, const int32_t *pos,
                             int32_t *n_raw, int U, void *stream) {
    const NvtxRange nvtx_range("ds4a_kv_push_raw");
    if (ds4a_status inj = take_injected()) return inj;
    if (!kv || !raw || !pos || !n_raw || U < 1) return DS4A_EINVAL;
    if (!aligned(kv, 16) || !aligned(raw, 16)) return DS4A_EINVAL;
    if (U > 1 && (raw_unit_stride < static_cast<int64_t>(kNSwa) * kHeadDim || raw_unit_stride % kHeadDim))
        return DS4A_EINVAL;
    DevInfo *di = nullptr;
    if (ds4a_status st = current_device(&di)) return st;
    return launch_kv_push_raw(kv, raw, U > 1 ? raw_unit_stride : 0, pos, n_raw, U, di->status,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DS4A_OK
               : DS4A_ECUDA;
}

ds4a_status ds4a_compressor_pool(const float *kv, const float *score, int ratio, int width, float *out, int U,
                                 void *stream) {
    const NvtxRange nvtx_range("ds4a_compressor_pool");
    if (ds4a_status inj = take_injected()) return inj;
    if (!kv || !score || !out || U < 1 || ratio < 1 || width < 4 || width % 4) return DS4A_EINVAL;
    if (!aligned(kv, 16) || !aligned(score, 16) || !aligned(out, 16)) return DS4A_EINVAL;
    if (static_cast<long long>(U) * ratio * width >= (1LL << 40)) return DS4A_EINVAL;
    DevInfo *di = nullptr;
    if (ds4a_status st = current_device(&di)) return st;
    return launch_compressor_pool(kv, score, ratio, width, out, U, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DS4A_OK
               : DS4A_ECUDA;
}

}  // extern "C"
