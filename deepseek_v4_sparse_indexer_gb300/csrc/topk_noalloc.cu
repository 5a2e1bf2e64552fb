// ds4a_topk_select_noalloc: the top-k selection for callers that cannot
// allocate device memory (a plugin inside a serving engine that owns the
// device's memory pool, a runtime with a fixed memory plan).  It runs the same
// kernels as ds4a_topk_select; only the scratch comes from a fixed array in
// this file instead of a caller-provided workspace.
#include <mutex>

#include "../../include/ds4a.h"
#include "internal.h"

using namespace ds4a;

namespace {

// The scratch every call on a device shares.  In host code the name below is
// a host-side stand-in, never a device address: the device address comes from
// cudaGetSymbolAddress (scratch_address()).
static __device__ __align__(256) uint8_t g_topk_scratch[DS4A_TOPK_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Set-up, once per device, with that device current.
ds4a_status scratch_address(void **out) {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return DS4A_ECUDA;
    if (d < 0 || d >= kMaxDevices) return DS4A_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[d]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || p == nullptr) return DS4A_ECUDA;
        g_scratch_addr[d] = p;
    }
    *out = g_scratch_addr[d];
    return DS4A_OK;
}

}  // namespace

extern "C" ds4a_status ds4a_topk_select_noalloc(const float *scores, const int32_t *n_rows, int U, int Q, int N_cap,
                                                int top_k, int32_t *idx, int32_t *count, void *stream) {
    const NvtxRange nvtx_range("ds4a_topk_select_noalloc");
    if (const int inj = take_injected_error()) return inj;
    if (!scores || !n_rows || !idx || !count) return DS4A_EINVAL;
    if (U < 1 || Q < 1 || N_cap < 1 || top_k < 1 || top_k > DS4A_MAX_TOP_K) return DS4A_EINVAL;
    if (static_cast<long long>(U) * Q > (1LL << 24)) return DS4A_EINVAL;
    if ((reinterpret_cast<uintptr_t>(scores) & 3) != 0) return DS4A_EINVAL;
    // Only few very long rows use scratch (at most about 5 MB, whatever the
    // sizes); the check guards the fixed array should that ever change.
    const size_t need = topk_ws_bytes(static_cast<long long>(U) * Q, N_cap);
    if (need > DS4A_TOPK_NOALLOC_SCRATCH_BYTES) return DS4A_EWORKSPACE;   // nothing launched
    uint32_t *status = nullptr;
    int sms = 0;
    if (const int st = current_device_info(&status, &sms)) return st;
    void *ws = nullptr;
    if (const ds4a_status st = scratch_address(&ws)) return st;
    // The kernels write every scratch word they later read: nothing needs clearing.
    TopkArgs a{scores, n_rows, U, Q, N_cap, top_k, idx, count, ws, status};
    return launch_topk(a, sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DS4A_OK : DS4A_ECUDA;
}
