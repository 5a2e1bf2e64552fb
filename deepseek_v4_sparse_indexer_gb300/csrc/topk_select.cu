// Top-k row selection per (unit, query) ("DwarfStar(ds4.c) のアーキテクチャを
// 読む" §3-3: only the n_indexer_top_k best-scoring compressed rows reach the
// main attention).
//
// Radix select on the order-preserving 32-bit key of each fp32 score, MSB
// first, in three kernels so that a few very long rows (long-context decode)
// and many shorter rows (decode batches, prefill chunks) both spread over the
// whole GPU without any inter-CTA waiting (stream order is the only sync):
//
//   1. hist    (chunks x rows CTAs): 4096-bin histogram of key bits 31..20 in
//               shared memory, added into a per-row global histogram.
//   2. filter  (chunks x rows CTAs): every CTA finds the row's threshold bin
//               b1 (the bin where the count from the top reaches k), then
//               appends rows with a higher bin to the row's "sure" list and
//               rows in bin b1 to its candidate list (warp-aggregated atomics).
//   3. final   (one CTA per row): resolves the exact k-th key inside the
//               candidate list (digits 19..8 and 7..0), applies the tie rule
//               (lower row index first), sorts the chosen indices ascending and
//               writes them with -1 padding.  If the candidate list overflowed
//               (pathological ties) it falls back to exact passes over the
//               row's scores with an order-preserving compaction.
//
// Scores read: twice per row (hist + filter), 8 bytes per row in total.
#include "common.cuh"
#include "internal.h"

namespace ds4a {
namespace {

constexpr int kBins = kTopkBins;
constexpr int kCandCap = kTopkCandCap;
constexpr int kHistThreads = 256;
constexpr int kFinalThreads = 512;

// Workspace layout for R rows:
//   hist  [R][4096] u32 | meta [R][4] u32 (n_sure, n_cand, b1+1, n_visible)
//   | sure [R][top_k] i32 | cand [R][kCandCap] (key u32, idx i32)
struct TopkWs {
    uint32_t *hist, *meta;
    int32_t *sure;
    uint2 *cand;
};
__host__ __device__ inline TopkWs topk_ws(void *base, long long R, int top_k) {
    TopkWs w;
    uint8_t *p = static_cast<uint8_t *>(base);
    w.hist = reinterpret_cast<uint32_t *>(p);
    p += R * kBins * 4;
    w.meta = reinterpret_cast<uint32_t *>(p);
    p += R * 16;
    w.sure = reinterpret_cast<int32_t *>(p);
    p += ((R * top_k * 4 + 15) / 16) * 16;
    w.cand = reinterpret_cast<uint2 *>(p);
    return w;
}

DS4A_DEV int row_len(const int32_t *n_rows, int u, int N_cap) {
    int n = n_rows[u];
    return n < 0 ? 0 : (n > N_cap ? N_cap : n);
}

// ---------------------------------------------------------------- 1. histogram
__global__ void __launch_bounds__(kHistThreads) topk_hist_kernel(const float *__restrict__ scores,
                                                                 const int32_t *__restrict__ n_rows, int Q,
                                                                 int N_cap, int chunk, int n_chunks, TopkWs ws,
                                                                 uint32_t *status) {
    __shared__ uint32_t h[kBins];
    const long long row = blockIdx.x / n_chunks;
    const int cidx = static_cast<int>(blockIdx.x - row * n_chunks);
    const int u = static_cast<int>(row / Q);
    const int n = row_len(n_rows, u, N_cap);
    if (cidx == 0 && threadIdx.x == 0 && (n_rows[u] < 0 || n_rows[u] > N_cap))
        report(status, DS4A_DEV_BOUNDS);
    const int start = cidx * chunk;
    const int end = min(start + chunk, n);
    if (start >= end) return;
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const float *s = scores + row * N_cap;
    if ((N_cap & 3) == 0) {
        const int vend = start + ((end - start) & ~3);
        for (int i = start + 4 * threadIdx.x; i < vend; i += 4 * blockDim.x) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(s + i));
            if (score_visible(v.x)) atomicAdd(&h[float_key(v.x) >> 20], 1u);
            if (score_visible(v.y)) atomicAdd(&h[float_key(v.y) >> 20], 1u);
            if (score_visible(v.z)) atomicAdd(&h[float_key(v.z) >> 20], 1u);
            if (score_visible(v.w)) atomicAdd(&h[float_key(v.w) >> 20], 1u);
        }
        for (int i = vend + threadIdx.x; i < end; i += blockDim.x) {
            const float f = s[i];
            if (score_visible(f)) atomicAdd(&h[float_key(f) >> 20], 1u);
        }
    } else {
        for (int i = start + threadIdx.x; i < end; i += blockDim.x) {
            const float f = s[i];
            if (score_visible(f)) atomicAdd(&h[float_key(f) >> 20], 1u);
        }
    }
    __syncthreads();
    uint32_t *gh = ws.hist + row * kBins;
    for (int i = threadIdx.x; i < kBins; i += blockDim.x)
        if (h[i]) atomicAdd(&gh[i], h[i]);
}

// Block-wide: finds the largest bin b with sum_{b' >= b} hist[b'] >= k.
// Returns b (-1 when the total is below k), the count strictly above b in
// *above and the total in *total.  `hist` is in shared memory, nbins a
// multiple of NT = blockDim.x.  Every thread gets the same result.
template <int NT>
DS4A_DEV int find_threshold_bin(const uint32_t *hist, int nbins, uint32_t k, uint32_t *above, uint32_t *total,
                                uint32_t *scratch /* NT + 4 u32 in smem */) {
    const int per = nbins / NT;
    const int t = threadIdx.x;
    uint32_t mine = 0;
    for (int i = 0; i < per; ++i) mine += hist[t * per + i];
    scratch[t] = mine;
    __syncthreads();
    if (t == 0) {
        // Serial walk from the top over the NT partial sums, then inside the
        // partial where the running count reaches k.
        uint32_t run = 0;
        int hit = -1;
        uint32_t hit_above = 0;
        for (int j = NT - 1; j >= 0; --j) {
            const uint32_t v = scratch[j];
            if (hit < 0 && run + v >= k) {
                hit = j;
                hit_above = run;
            }
            run += v;
        }
        int b = -1;
        uint32_t ab = run;
        if (hit >= 0) {
            uint32_t r2 = hit_above;
            for (b = hit * per + per - 1; b > hit * per; --b) {
                if (r2 + hist[b] >= k) break;
                r2 += hist[b];
            }
            ab = r2;
        }
        scratch[NT] = static_cast<uint32_t>(b);
        scratch[NT + 1] = ab;
        scratch[NT + 2] = run;
    }
    __syncthreads();
    const int b = static_cast<int>(scratch[NT]);
    *above = scratch[NT + 1];
    *total = scratch[NT + 2];
    __syncthreads();
    return b;
}

// Warp-aggregated append: returns the slot for this lane (valid if pred).
DS4A_DEV uint32_t warp_append(uint32_t *counter, bool pred) {
    const uint32_t mask = __ballot_sync(0xffffffffu, pred);
    if (!mask) return 0;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(mask) - 1;
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(counter, static_cast<uint32_t>(__popc(mask)));
    base = __shfl_sync(0xffffffffu, base, leader);
    return base + __popc(mask & ((1u << lane) - 1u));
}

// ---------------------------------------------------------------- 2. filter
__global__ void __launch_bounds__(kHistThreads) topk_filter_kernel(const float *__restrict__ scores,
                                                                   const int32_t *__restrict__ n_rows, int Q,
                                                                   int N_cap, int top_k, int chunk, int n_chunks,
                                                                   TopkWs ws) {
    __shared__ uint32_t h[kBins];
    __shared__ uint32_t scratch[kHistThreads + 4];
    const long long row = blockIdx.x / n_chunks;
    const int cidx = static_cast<int>(blockIdx.x - row * n_chunks);
    const int u = static_cast<int>(row / Q);
    const int n = row_len(n_rows, u, N_cap);
    const int start = cidx * chunk;
    const int end = min(start + chunk, n);
    if (start >= end && cidx != 0) return;
    const uint32_t *gh = ws.hist + row * kBins;
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = gh[i];
    __syncthreads();
    uint32_t above, total;
    int b1 = find_threshold_bin<kHistThreads>(h, kBins, static_cast<uint32_t>(top_k), &above, &total, scratch);
    if (total <= static_cast<uint32_t>(top_k)) b1 = -1;     // everything visible is selected
    uint32_t *meta = ws.meta + row * 4;
    if (cidx == 0 && threadIdx.x == 0) {
        meta[2] = static_cast<uint32_t>(b1 + 1);
        meta[3] = total;
    }
    if (start >= end) return;
    const float *s = scores + row * N_cap;
    int32_t *sure = ws.sure + row * top_k;
    uint2 *cand = ws.cand + row * kCandCap;
    // Whole warps iterate together so the ballots see every lane.
    const int span = end - start;
    const int iters = (span + blockDim.x - 1) / blockDim.x;
    for (int it = 0; it < iters; ++it) {
        const int i = start + it * blockDim.x + threadIdx.x;
        bool vis = false;
        uint32_t key = 0;
        if (i < end) {
            const float f = s[i];
            vis = score_visible(f);
            key = float_key(f);
        }
        const int d = static_cast<int>(key >> 20);
        const bool is_sure = vis && d > b1;
        const bool is_cand = vis && b1 >= 0 && d == b1;
        const uint32_t ps = warp_append(&meta[0], is_sure);
        if (is_sure && ps < static_cast<uint32_t>(top_k)) sure[ps] = i;
        const uint32_t pc = warp_append(&meta[1], is_cand);
        if (is_cand && pc < static_cast<uint32_t>(kCandCap)) cand[pc] = make_uint2(key, static_cast<uint32_t>(i));
    }
}

// ---------------------------------------------------------------- 3. final
DS4A_DEV void block_bitonic_sort_asc(int32_t *a, int n_pow2) {
    for (int k = 2; k <= n_pow2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n_pow2; i += blockDim.x) {
                const int p = i ^ j;
                if (p > i) {
                    const int32_t x = a[i], y = a[p];
                    const bool up = (i & k) == 0;
                    if ((x > y) == up) {
                        a[i] = y;
                        a[p] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Block-wide exclusive prefix count of `pred` over the block's threads.
// Returns this thread's rank; *total receives the block total.
DS4A_DEV uint32_t block_rank(bool pred, uint32_t *warp_sums /* 32 u32 smem */, uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t m = __ballot_sync(0xffffffffu, pred);
    if (lane == 0) warp_sums[warp] = __popc(m);
    __syncthreads();
    uint32_t before = 0, tot = 0;
    for (int w = 0; w < nwarps; ++w) {
        const uint32_t v = warp_sums[w];
        if (w < warp) before += v;
        tot += v;
    }
    __syncthreads();
    *total = tot;
    return before + __popc(m & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(kFinalThreads) topk_final_kernel(const float *__restrict__ scores,
                                                                   const int32_t *__restrict__ n_rows, int Q,
                                                                   int N_cap, int top_k, TopkWs ws,
                                                                   int32_t *__restrict__ idx_out,
                                                                   int32_t *__restrict__ count_out) {
    __shared__ uint32_t h[kBins];
    __shared__ uint32_t scratch[kFinalThreads + 4];
    __shared__ int32_t sel[kMaxTopK];
    __shared__ uint32_t n_sel;
    __shared__ uint32_t warp_sums[32];
    const long long row = blockIdx.x;
    const int u = static_cast<int>(row / Q);
    const int n = row_len(n_rows, u, N_cap);
    const uint32_t *meta = ws.meta + row * 4;
    const uint32_t n_sure = meta[0];
    const uint32_t n_cand = meta[1];
    const int b1 = static_cast<int>(meta[2]) - 1;
    const uint32_t total = meta[3];
    const uint32_t k = static_cast<uint32_t>(top_k);
    const uint32_t m = total < k ? total : k;          // number selected
    int32_t *out = idx_out + row * top_k;
    const int32_t *sure = ws.sure + row * top_k;
    const uint2 *cand = ws.cand + row * kCandCap;
    const float *s = scores + row * N_cap;

    if (threadIdx.x == 0) n_sel = 0;
    __syncthreads();

    if (b1 < 0) {
        // Everything visible is selected (total <= k): the sure list holds it.
        for (uint32_t i = threadIdx.x; i < n_sure && i < k; i += blockDim.x) sel[i] = sure[i];
        if (threadIdx.x == 0) n_sel = n_sure < k ? n_sure : k;
        __syncthreads();
    } else if (n_cand <= static_cast<uint32_t>(kCandCap)) {
        const uint32_t need = k - n_sure;     // taken from bin b1 (1 <= need <= n_cand)
        // Digit 2: key bits 19..8 among candidates.
        for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
        __syncthreads();
        for (uint32_t i = threadIdx.x; i < n_cand; i += blockDim.x) atomicAdd(&h[(cand[i].x >> 8) & 0xFFFu], 1u);
        __syncthreads();
        uint32_t gt2, tot2;
        int b2 = find_threshold_bin<kFinalThreads>(h, kBins, need, &gt2, &tot2, scratch);
        if (b2 < 0) { b2 = 0; gt2 = 0; }      // cannot happen: need <= n_cand
        // Digit 3: key bits 7..0 among candidates in bin b2.
        for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
        __syncthreads();
        for (uint32_t i = threadIdx.x; i < n_cand; i += blockDim.x) {
            const uint32_t key = cand[i].x;
            if (static_cast<int>((key >> 8) & 0xFFFu) == b2) atomicAdd(&h[key & 0xFFu], 1u);
        }
        __syncthreads();
        uint32_t gt3, tot3;
        int b3 = find_threshold_bin<kFinalThreads>(h, kBins, need - gt2, &gt3, &tot3, scratch);
        if (b3 < 0) { b3 = 0; gt3 = 0; }
        const uint32_t T = (static_cast<uint32_t>(b1) << 20) | (static_cast<uint32_t>(b2) << 8) |
                           static_cast<uint32_t>(b3);
        const uint32_t need_eq = need - gt2 - gt3;    // equal-to-T keys to take, lowest rows first
        const uint32_t n_eq = h[b3];
        // Sure rows.
        for (uint32_t i = threadIdx.x; i < n_sure; i += blockDim.x) sel[i] = sure[i];
        // Candidates above T, and the need_eq lowest-index ones equal to T.
        for (uint32_t i = threadIdx.x; i < n_cand; i += blockDim.x) {
            const uint2 c = cand[i];
            bool take = c.x > T;
            if (c.x == T) {
                if (n_eq == need_eq) {
                    take = true;
                } else {
                    uint32_t lower = 0;
                    for (uint32_t j = 0; j < n_cand; ++j) {
                        const uint2 o = cand[j];
                        lower += (o.x == T && static_cast<int>(o.y) < static_cast<int>(c.y)) ? 1u : 0u;
                    }
                    take = lower < need_eq;
                }
            }
            if (take) {
                const uint32_t p = atomicAdd(&n_sel, 1u);
                if (n_sure + p < k) sel[n_sure + p] = static_cast<int32_t>(c.y);
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) n_sel = n_sure + n_sel < k ? n_sure + n_sel : k;
        __syncthreads();
    } else {
        // Candidate list overflowed: exact passes over the row's scores.
        const uint32_t need = k - n_sure;
        for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const float f = s[i];
            if (!score_visible(f)) continue;
            const uint32_t key = float_key(f);
            if (static_cast<int>(key >> 20) == b1) atomicAdd(&h[(key >> 8) & 0xFFFu], 1u);
        }
        __syncthreads();
        uint32_t gt2, tot2;
        int b2 = find_threshold_bin<kFinalThreads>(h, kBins, need, &gt2, &tot2, scratch);
        if (b2 < 0) { b2 = 0; gt2 = 0; }
        for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
        __syncthreads();
        const uint32_t pre12 = (static_cast<uint32_t>(b1) << 12) | static_cast<uint32_t>(b2);
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const float f = s[i];
            if (!score_visible(f)) continue;
            const uint32_t key = float_key(f);
            if ((key >> 8) == pre12) atomicAdd(&h[key & 0xFFu], 1u);
        }
        __syncthreads();
        uint32_t gt3, tot3;
        int b3 = find_threshold_bin<kFinalThreads>(h, kBins, need - gt2, &gt3, &tot3, scratch);
        if (b3 < 0) { b3 = 0; gt3 = 0; }
        const uint32_t T = (pre12 << 8) | static_cast<uint32_t>(b3);
        const uint32_t need_eq = need - gt2 - gt3;
        // Order-preserving compaction over the row: output is ascending.
        uint32_t written = 0, eq_seen = 0;
        for (int base = 0; base < n; base += blockDim.x) {
            const int i = base + threadIdx.x;
            bool vis = false;
            uint32_t key = 0;
            if (i < n) {
                const float f = s[i];
                vis = score_visible(f);
                key = float_key(f);
            }
            const bool is_eq = vis && key == T;
            uint32_t eq_tot;
            const uint32_t eq_rank = eq_seen + block_rank(is_eq, warp_sums, &eq_tot);
            const bool take = vis && (key > T || (is_eq && eq_rank < need_eq));
            uint32_t tk_tot;
            const uint32_t pos = written + block_rank(take, warp_sums, &tk_tot);
            if (take && pos < k) out[pos] = i;
            written += tk_tot;
            eq_seen += eq_tot;
        }
        for (uint32_t i = m + threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
        if (threadIdx.x == 0) count_out[row] = static_cast<int32_t>(m);
        return;
    }

    // Sort the chosen indices ascending and write them with -1 padding.
    const uint32_t ns = n_sel;
    int p2 = 1;
    while (p2 < static_cast<int>(ns)) p2 <<= 1;
    for (int i = static_cast<int>(ns) + threadIdx.x; i < p2; i += blockDim.x) sel[i] = 0x7fffffff;
    __syncthreads();
    block_bitonic_sort_asc(sel, p2);
    for (uint32_t i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < ns ? sel[i] : -1;
    if (threadIdx.x == 0) count_out[row] = static_cast<int32_t>(ns);
}

}  // namespace

size_t topk_ws_bytes(long long R, int top_k) {
    size_t b = static_cast<size_t>(R) * kBins * 4 + static_cast<size_t>(R) * 16;
    b += ((static_cast<size_t>(R) * top_k * 4 + 15) / 16) * 16;
    b += static_cast<size_t>(R) * kCandCap * 8;
    return b;
}

cudaError_t launch_topk(const TopkArgs &a, int num_sms, cudaStream_t s) {
    const long long R = static_cast<long long>(a.U) * a.Q;
    TopkWs ws = topk_ws(a.ws, R, a.top_k);
    // Zero the histograms and counters (contiguous at the front).
    cudaError_t e = cudaMemsetAsync(a.ws, 0, static_cast<size_t>(R) * (kBins * 4 + 16), s);
    if (e != cudaSuccess) return e;
    // Chunk length: enough CTAs to cover the GPU twice, 2K..32K scores per CTA.
    long long target = 2LL * num_sms;
    long long per = (R * static_cast<long long>(a.N_cap) + target - 1) / target;
    int chunk = 2048;
    while (chunk < 32768 && chunk < per) chunk <<= 1;
    const int n_chunks = (a.N_cap + chunk - 1) / chunk;
    const long long blocks = R * n_chunks;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>(blocks);
    topk_hist_kernel<<<grid, kHistThreads, 0, s>>>(a.scores, a.n_rows, a.Q, a.N_cap, chunk, n_chunks, ws,
                                                   a.status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    topk_filter_kernel<<<grid, kHistThreads, 0, s>>>(a.scores, a.n_rows, a.Q, a.N_cap, a.top_k, chunk, n_chunks,
                                                     ws);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    topk_final_kernel<<<dim3(static_cast<unsigned>(R), 1), kFinalThreads, 0, s>>>(a.scores, a.n_rows, a.Q, a.N_cap,
                                                                                  a.top_k, ws, a.idx, a.count);
    return cudaGetLastError();
}

}  // namespace ds4a
