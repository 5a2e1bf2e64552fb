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
//               rows in bin b1 to its candidate list (staged in shared queues).
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
    pdl_launch_dependents();
    pdl_wait();
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
        auto add = [&](float f) {
            if (score_visible(f)) atomicAdd(&h[float_key(f) >> 20], 1u);
        };
        // Four 16-byte loads in flight per thread before any is consumed.
        constexpr int B = 4;
        const int stride = 4 * blockDim.x;
        int i = start + 4 * threadIdx.x;
        for (; i + (B - 1) * stride < vend; i += B * stride) {
            float4 v[B];
#pragma unroll
            for (int j = 0; j < B; ++j) v[j] = __ldg(reinterpret_cast<const float4 *>(s + i + j * stride));
#pragma unroll
            for (int j = 0; j < B; ++j) {
                add(v[j].x);
                add(v[j].y);
                add(v[j].z);
                add(v[j].w);
            }
        }
        for (; i < vend; i += stride) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(s + i));
            add(v.x);
            add(v.y);
            add(v.z);
            add(v.w);
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
// multiple of NT = blockDim.x, NT a multiple of 32 and at most 1024.  Every
// thread gets the same result.
//   1. every thread sums nbins/NT consecutive bins;
//   2. warp 0: each lane sums NT/32 consecutive partials, an inclusive suffix
//      scan over the lanes finds the lane whose range crosses k, and that lane
//      walks its partials, then the bins of the crossing partial.
template <int NT>
DS4A_DEV int find_threshold_bin(const uint32_t *hist, int nbins, uint32_t k, uint32_t *above, uint32_t *total,
                                uint32_t *scratch /* NT + 4 u32 in smem */) {
    static_assert(NT % 32 == 0 && NT <= 1024, "block size");
    constexpr int PPL = NT / 32;               // partials per lane
    const int per = nbins / NT;
    const int t = threadIdx.x;
    uint32_t mine = 0;
    for (int i = 0; i < per; ++i) mine += hist[t * per + i];
    scratch[t] = mine;
    __syncthreads();
    if (t < 32) {
        uint32_t lane_sum = 0;
#pragma unroll
        for (int i = 0; i < PPL; ++i) lane_sum += scratch[t * PPL + i];
        // Inclusive suffix sum over lanes: suf = sum of lane_sum for lanes >= t.
        uint32_t suf = lane_sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t v = __shfl_down_sync(0xffffffffu, suf, off);
            if (t + off < 32) suf += v;
        }
        const uint32_t tot = __shfl_sync(0xffffffffu, suf, 0);
        // The crossing lane: the highest lane whose suffix reaches k.
        const uint32_t hit_mask = __ballot_sync(0xffffffffu, suf >= k);
        if (t == 0) {
            scratch[NT + 2] = tot;
            if (hit_mask == 0) {
                scratch[NT] = static_cast<uint32_t>(-1);
                scratch[NT + 1] = tot;
            }
        }
        if (hit_mask != 0) {
            const int L = 31 - __clz(hit_mask);
            if (t == L) {
                uint32_t run = suf - lane_sum;     // count above this lane's range
                int p = t * PPL + PPL - 1;
                for (; p > t * PPL; --p) {
                    if (run + scratch[p] >= k) break;
                    run += scratch[p];
                }
                int b = p * per + per - 1;
                for (; b > p * per; --b) {
                    if (run + hist[b] >= k) break;
                    run += hist[b];
                }
                scratch[NT] = static_cast<uint32_t>(b);
                scratch[NT + 1] = run;
            }
        }
    }
    __syncthreads();
    const int b = static_cast<int>(scratch[NT]);
    *above = scratch[NT + 1];
    *total = scratch[NT + 2];
    __syncthreads();
    return b;
}

// ---------------------------------------------------------------- 2. filter
// Qualifying rows (bin >= b1, about 2 % of a random row) are staged in shared
// queues with one shared atomic each, then appended to the row's global lists
// with one global atomic per list per CTA.  A full candidate queue spills
// straight to the global list.
constexpr int kQueueCap = 2048;

__global__ void __launch_bounds__(kHistThreads) topk_filter_kernel(const float *__restrict__ scores,
                                                                   const int32_t *__restrict__ n_rows, int Q,
                                                                   int N_cap, int top_k, int chunk, int n_chunks,
                                                                   TopkWs ws) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ uint32_t h[kBins];
    __shared__ uint32_t scratch[kHistThreads + 4];
    __shared__ int32_t q_sure[kMaxTopK];
    __shared__ uint2 q_cand[kQueueCap];
    __shared__ uint32_t n_qs, n_qc, base_s, base_c;
    const long long row = blockIdx.x / n_chunks;
    const int cidx = static_cast<int>(blockIdx.x - row * n_chunks);
    const int u = static_cast<int>(row / Q);
    const int n = row_len(n_rows, u, N_cap);
    const int start = cidx * chunk;
    const int end = min(start + chunk, n);
    if (start >= end && cidx != 0) return;
    const uint32_t *gh = ws.hist + row * kBins;
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = gh[i];
    if (threadIdx.x == 0) n_qs = n_qc = 0;
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
    const uint32_t key_lo = b1 < 0 ? 0u : (static_cast<uint32_t>(b1) << 20);
    auto consider = [&](int i, float f) {
        if (!score_visible(f)) return;
        const uint32_t key = float_key(f);
        if (key < key_lo) return;
        if (static_cast<int>(key >> 20) > b1) {
            const uint32_t p = atomicAdd(&n_qs, 1u);
            if (p < static_cast<uint32_t>(top_k)) q_sure[p] = i;      // never more than k in total
        } else {
            const uint32_t p = atomicAdd(&n_qc, 1u);
            if (p < static_cast<uint32_t>(kQueueCap)) {
                q_cand[p] = make_uint2(key, static_cast<uint32_t>(i));
            } else {
                const uint32_t g = atomicAdd(&meta[1], 1u);
                if (g < static_cast<uint32_t>(kCandCap)) cand[g] = make_uint2(key, static_cast<uint32_t>(i));
            }
        }
    };
    if ((N_cap & 3) == 0) {
        const int vend = start + ((end - start) & ~3);
        constexpr int B = 4;
        const int stride = 4 * blockDim.x;
        int i = start + 4 * threadIdx.x;
        for (; i + (B - 1) * stride < vend; i += B * stride) {
            float4 v[B];
#pragma unroll
            for (int j = 0; j < B; ++j) v[j] = __ldg(reinterpret_cast<const float4 *>(s + i + j * stride));
#pragma unroll
            for (int j = 0; j < B; ++j) {
                const int b = i + j * stride;
                consider(b, v[j].x);
                consider(b + 1, v[j].y);
                consider(b + 2, v[j].z);
                consider(b + 3, v[j].w);
            }
        }
        for (; i < vend; i += stride) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(s + i));
            consider(i, v.x);
            consider(i + 1, v.y);
            consider(i + 2, v.z);
            consider(i + 3, v.w);
        }
        for (int i = vend + threadIdx.x; i < end; i += blockDim.x) consider(i, s[i]);
    } else {
        for (int i = start + threadIdx.x; i < end; i += blockDim.x) consider(i, s[i]);
    }
    __syncthreads();
    const uint32_t ns = min(n_qs, static_cast<uint32_t>(top_k));
    const uint32_t nc = min(n_qc, static_cast<uint32_t>(kQueueCap));
    if (threadIdx.x == 0) {
        base_s = ns ? atomicAdd(&meta[0], ns) : 0u;
        base_c = nc ? atomicAdd(&meta[1], nc) : 0u;
    }
    __syncthreads();
    for (uint32_t j = threadIdx.x; j < ns; j += blockDim.x)
        if (base_s + j < static_cast<uint32_t>(top_k)) sure[base_s + j] = q_sure[j];
    for (uint32_t j = threadIdx.x; j < nc; j += blockDim.x)
        if (base_c + j < static_cast<uint32_t>(kCandCap)) cand[base_c + j] = q_cand[j];
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
    pdl_launch_dependents();
    pdl_wait();
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


// ---------------------------------------------------------------- one CTA per row
// For batches with at least as many rows as SMs (decode batches, prefill
// chunks): each CTA selects one row's top-k alone and reads the row's scores
// once from HBM in the common case.
//   1. A sample of kSample scores (64 whole 128-byte lines spread evenly over
//      the row, so that the sample costs whole lines, not scattered sectors) sets
//      a threshold key T0: the r-th largest visible sample key with
//      r = 3k*kSample/n, resolved to 24 bits (two 4096-bin digits over the
//      sample), so that about 3k rows of the row lie at or above it.
//   2. One pass over the row counts the visible scores and appends every row
//      with key >= T0 to a shared candidate list (warp-aggregated appends).
//   3. If at least k candidates arrived and none was dropped, the exact k-th
//      key T and the tie count come from three radix digits over the
//      candidates; otherwise (a sample that missed, heavy ties) the same
//      digits come from passes over the row itself, which the pass above left
//      in L2.  Rows with at most k visible scores take all of them.
//   4. Output: the chosen candidates in ascending row order (a bitmap of the
//      row and a prefix sum of its popcounts; a bitonic sort for rows longer
//      than 131,072), -1 padded; the fallback compacts the row in order.

// Two shapes: 512 threads, 8,192 candidates, two CTAs per SM (any k, any
// length); and for k <= kRowSmallMaxK and rows up to kRowSmallMaxN (the
// reach of the row bitmap), 256 threads, 4,096 candidates and a 1,024-entry
// sort buffer, four CTAs per SM: a row's phases are latency-bound, so twice
// the rows in flight beat twice the threads per row (2,048 x 16,896: 140 vs
// 169 us; 2,048 x 66,048: 224 vs 250 us; 1,376 x 65,536: 165 vs 177 us).
constexpr int kSample = 2048;
constexpr int kSampleOver = 3;     // expected candidates / k
constexpr int kRowSmallMaxK = 640;
constexpr int kRowSmallMaxN = kBins * 32;   // 131,072
template <int NT, int CAP, int SEL>
struct RowShape {
    static constexpr int kSmem = CAP * 8 + kBins * 4 + SEL * 4;   // candidates, histogram, chosen
};

template <int NT, int CAP, int SEL>
__global__ void __launch_bounds__(NT, NT == 512 ? 2 : 4) topk_row_kernel(const float *__restrict__ scores,
                                                                  const int32_t *__restrict__ n_rows, int Q,
                                                                  int N_cap, int top_k,
                                                                  int32_t *__restrict__ idx_out,
                                                                  int32_t *__restrict__ count_out, uint32_t *status) {
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(16) uint8_t row_smem[];
    uint2 *cand = reinterpret_cast<uint2 *>(row_smem);                               // [CAP]
    uint32_t *h = reinterpret_cast<uint32_t *>(row_smem + CAP * 8);           // [kBins]
    int32_t *sel = reinterpret_cast<int32_t *>(row_smem + CAP * 8 + kBins * 4);   // [SEL]
    __shared__ uint32_t scratch[NT + 4];
    __shared__ uint32_t n_cand, n_sel;
    __shared__ uint32_t warp_sums[32];
    const long long row = blockIdx.x;
    const int u = static_cast<int>(row / Q);
    const int n = row_len(n_rows, u, N_cap);
    if (threadIdx.x == 0 && row % Q == 0 && (n_rows[u] < 0 || n_rows[u] > N_cap)) report(status, DS4A_DEV_BOUNDS);
    const float *s = scores + row * N_cap;
    const uint32_t k = static_cast<uint32_t>(top_k);
    int32_t *out = idx_out + row * top_k;
    const int lane = threadIdx.x & 31;

    auto clear_hist = [&]() {
        for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
        __syncthreads();
    };
    constexpr int B = 4;
    const int ngroups = (n + 3) / 4;
    const bool vec4 = (N_cap & 3) == 0;
    auto load = [&](float4 (&v)[B], int g0) {
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int g = g0 + j * NT + static_cast<int>(threadIdx.x);
            v[j] = g < ngroups ? __ldg(reinterpret_cast<const float4 *>(s) + g) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    float4 cur[B], nxt[B];
    if (vec4) load(cur, 0);                              // in flight during the threshold estimate
    // ---- 1. threshold estimate
    uint32_t T0 = 0;
    if (n > CAP) {
        uint32_t skey[kSample / NT];
        bool svis[kSample / NT];
        clear_hist();
#pragma unroll
        for (int j = 0; j < kSample / NT; ++j) {
            // sample sj: score (sj & 31) of one of 64 whole 128-byte lines spread
            // evenly over the row (a warp loads one line: no scattered sectors)
            const int sj = static_cast<int>(threadIdx.x) + j * NT;
            const int line = static_cast<int>((static_cast<long long>(sj >> 5) * (n / 32 - 1)) / (kSample / 32 - 1));
            const int i = line * 32 + (sj & 31);
            const float f = __ldg(s + i);
            svis[j] = score_visible(f);
            skey[j] = float_key(f);
            hist_add_warp(h, skey[j] >> 20, svis[j]);
        }
        __syncthreads();
        const long long r_want = (static_cast<long long>(kSampleOver) * k * kSample + n - 1) / n;
        const uint32_t rank = static_cast<uint32_t>(r_want < kSample ? r_want : kSample);
        uint32_t above, total;
        const int sb1 = find_threshold_bin<NT>(h, kBins, rank, &above, &total, scratch);
        if (sb1 >= 0) {
            clear_hist();
#pragma unroll
            for (int j = 0; j < kSample / NT; ++j)
                hist_add_warp(h, (skey[j] >> 8) & 0xFFFu, svis[j] && static_cast<int>(skey[j] >> 20) == sb1);
            __syncthreads();
            uint32_t above2, total2;
            int sb2 = find_threshold_bin<NT>(h, kBins, rank - above, &above2, &total2, scratch);
            if (sb2 < 0) sb2 = 0;
            T0 = (static_cast<uint32_t>(sb1) << 20) | (static_cast<uint32_t>(sb2) << 8);
        }
    }
    // ---- 2. one pass: visible count and candidates (key >= T0)
    if (threadIdx.x == 0) n_cand = 0;
    __syncthreads();
    uint32_t my_vis = 0;
    // Appends the lanes' rows with key >= T0 (warp-aggregated); all lanes call it.
    auto append = [&](int i, uint32_t key, bool take) {
        const uint32_t bal = __ballot_sync(0xffffffffu, take);
        if (bal) {
            uint32_t base = 0;
            if (lane == 0) base = atomicAdd(&n_cand, static_cast<uint32_t>(__popc(bal)));
            base = __shfl_sync(0xffffffffu, base, 0);
            const uint32_t p = base + __popc(bal & ((1u << lane) - 1u));
            if (take && p < static_cast<uint32_t>(CAP)) cand[p] = make_uint2(key, static_cast<uint32_t>(i));
        }
    };
    if (vec4) {
        // Whole float4 groups, B per thread in flight plus the next B prefetched;
        // every thread runs the same iterations (the ballots are warp-wide).
        for (int g0 = 0; g0 < ngroups; g0 += B * NT) {
            if (g0 + B * NT < ngroups) load(nxt, g0 + B * NT);
#pragma unroll
            for (int j = 0; j < B; ++j) {
                const int i = 4 * (g0 + j * NT + static_cast<int>(threadIdx.x));
                const float f[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
                uint32_t key[4];
                bool take[4];
                bool any = false;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const bool vis = i + c < n && score_visible(f[c]);
                    key[c] = float_key(f[c]);
                    my_vis += vis ? 1u : 0u;
                    take[c] = vis && key[c] >= T0;
                    any |= take[c];
                }
                if (__any_sync(0xffffffffu, any)) {
                    // one shared atomic per warp and float4
                    uint32_t bal[4], tot = 0;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        bal[c] = __ballot_sync(0xffffffffu, take[c]);
                        tot += __popc(bal[c]);
                    }
                    uint32_t pos = 0;
                    if (lane == 0) pos = atomicAdd(&n_cand, tot);
                    pos = __shfl_sync(0xffffffffu, pos, 0);
                    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t p = pos + __popc(bal[c] & lt);
                        if (take[c] && p < static_cast<uint32_t>(CAP)) cand[p] = make_uint2(key[c], static_cast<uint32_t>(i + c));
                        pos += __popc(bal[c]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < B; ++j) cur[j] = nxt[j];
        }
    } else {
        for (int b = 0; b < n; b += NT) {
            const int i = b + static_cast<int>(threadIdx.x);
            const float f = i < n ? s[i] : 0.f;
            const bool vis = i < n && score_visible(f);
            const uint32_t key = float_key(f);
            my_vis += vis ? 1u : 0u;
            append(i, key, vis && key >= T0);
        }
    }
    uint32_t total;
    {
        // block sum of my_vis
        uint32_t v = my_vis;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) warp_sums[threadIdx.x >> 5] = v;
        __syncthreads();
        total = 0;
        for (int w = 0; w < NT / 32; ++w) total += warp_sums[w];
        __syncthreads();
    }
    const uint32_t nc = n_cand;
    const uint32_t m = total < k ? total : k;           // number selected

    // ---- 3. the exact k-th key T and how many keys equal to T to take
    uint32_t T = 0, need_eq = 0;
    const bool all_visible = total <= k;
    const bool from_cand = all_visible ? nc == total : (nc >= k && nc <= static_cast<uint32_t>(CAP));
    if (!all_visible) {
        // digit d: bits [lo, lo + w) of keys whose higher bits equal prefix
        uint32_t need = k;
        uint32_t prefix = 0;
        const int shifts[3] = {20, 8, 0};
        const uint32_t masks[3] = {0xFFFu, 0xFFFu, 0xFFu};
        for (int d = 0; d < 3; ++d) {
            clear_hist();
            const int sh = shifts[d];
            const int hs = d == 0 ? 32 : shifts[d - 1];        // bits above this digit: key >> hs == prefix
            if (from_cand) {
                for (uint32_t i0 = 0; i0 < nc; i0 += blockDim.x) {   // block-uniform trip count
                    const uint32_t i = i0 + threadIdx.x;
                    const uint32_t key = i < nc ? cand[i].x : 0u;
                    hist_add_warp(h, (key >> sh) & masks[d], i < nc && (hs == 32 || (key >> hs) == prefix));
                }
            } else {
                for (int i = threadIdx.x; i < n; i += blockDim.x) {
                    const float f = s[i];
                    if (!score_visible(f)) continue;
                    const uint32_t key = float_key(f);
                    if (hs == 32 || (key >> hs) == prefix) atomicAdd(&h[(key >> sh) & masks[d]], 1u);
                }
            }
            __syncthreads();
            uint32_t gt, tot;
            int b = find_threshold_bin<NT>(h, kBins, need, &gt, &tot, scratch);
            if (b < 0) { b = 0; gt = 0; }     // cannot happen: need <= count of keys with this prefix
            prefix = (d == 0 ? 0u : prefix << (d == 1 ? 12 : 8)) | static_cast<uint32_t>(b);
            need -= gt;
        }
        T = prefix;                                     // bits 31..20 | 19..8 | 7..0
        need_eq = need;                                 // keys equal to T to take, lowest rows first
    }
    if (from_cand) {
        // ---- 4a. the chosen candidates in ascending row order: a bitmap of
        // the row (in the histogram's space) and a block prefix sum of its
        // popcounts; rows longer than the bitmap take a bitonic sort instead.
        const bool use_bitmap = n <= kBins * 32;
        if (threadIdx.x == 0) n_sel = 0;
        uint32_t n_eq = 0;
        if (!all_visible) {
            for (uint32_t i = threadIdx.x; i < nc; i += blockDim.x) n_eq += cand[i].x == T ? 1u : 0u;
            uint32_t v = n_eq;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) warp_sums[threadIdx.x >> 5] = v;
            __syncthreads();
            n_eq = 0;
            for (int w = 0; w < NT / 32; ++w) n_eq += warp_sums[w];
        }
        if (use_bitmap)
            for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0;
        __syncthreads();
        for (uint32_t i0 = 0; i0 < nc; i0 += blockDim.x) {            // block-uniform trip count
            const uint32_t i = i0 + threadIdx.x;
            bool take = false;
            uint2 c = make_uint2(0u, 0u);
            if (i < nc) {
                c = cand[i];
                take = all_visible || c.x > T;
                if (!all_visible && c.x == T) {
                    if (n_eq == need_eq) {
                        take = true;
                    } else {
                        uint32_t lower = 0;
                        for (uint32_t j = 0; j < nc; ++j) {
                            const uint2 o = cand[j];
                            lower += (o.x == T && static_cast<int>(o.y) < static_cast<int>(c.y)) ? 1u : 0u;
                        }
                        take = lower < need_eq;
                    }
                }
            }
            if (use_bitmap) {
                if (take) atomicOr(&h[c.y >> 5], 1u << (c.y & 31));
            } else {
                const uint32_t bal = __ballot_sync(0xffffffffu, take);
                uint32_t base = 0;
                if (lane == 0 && bal) base = atomicAdd(&n_sel, static_cast<uint32_t>(__popc(bal)));
                base = __shfl_sync(0xffffffffu, base, 0);
                const uint32_t p = base + __popc(bal & ((1u << lane) - 1u));
                if (take && p < k) sel[p] = static_cast<int32_t>(c.y);
            }
        }
        __syncthreads();
        if (use_bitmap) {
            // thread t owns words 8t..8t+7 (rows 256t..256t+255)
            constexpr int kWords = kBins / NT;
            uint32_t wv[kWords], cnt = 0;
#pragma unroll
            for (int j = 0; j < kWords; ++j) {
                wv[j] = h[threadIdx.x * kWords + j];
                cnt += __popc(wv[j]);
            }
            // block exclusive prefix sum of cnt
            uint32_t incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            if (lane == 31) warp_sums[threadIdx.x >> 5] = incl;
            __syncthreads();
            uint32_t before = 0, ns = 0;
            for (int w = 0; w < NT / 32; ++w) {
                const uint32_t v = warp_sums[w];
                if (w < static_cast<int>(threadIdx.x >> 5)) before += v;
                ns += v;
            }
            uint32_t pos = before + incl - cnt;
#pragma unroll
            for (int j = 0; j < kWords; ++j) {
                uint32_t bits = wv[j];
                while (bits) {
                    const int b = __ffs(bits) - 1;
                    bits &= bits - 1;
                    if (pos < k) out[pos] = static_cast<int32_t>((threadIdx.x * kWords + j) * 32 + b);
                    ++pos;
                }
            }
            ns = ns < k ? ns : k;
            for (uint32_t i = ns + threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
            if (threadIdx.x == 0) count_out[row] = static_cast<int32_t>(ns);
            return;
        }
        const uint32_t ns = n_sel < k ? n_sel : k;
        int p2 = 1;
        while (p2 < static_cast<int>(ns)) p2 <<= 1;
        for (int i = static_cast<int>(ns) + threadIdx.x; i < p2; i += blockDim.x) sel[i] = 0x7fffffff;
        __syncthreads();
        block_bitonic_sort_asc(sel, p2);
        for (uint32_t i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < ns ? sel[i] : -1;
        if (threadIdx.x == 0) count_out[row] = static_cast<int32_t>(ns);
        return;
    }
    // ---- 4b. order-preserving compaction over the row: ascending output
    uint32_t written = 0, eq_seen = 0;
    for (int base = 0; base < n; base += blockDim.x) {
        const int i = base + static_cast<int>(threadIdx.x);
        bool vis = false;
        uint32_t key = 0;
        if (i < n) {
            const float f = s[i];
            vis = score_visible(f);
            key = float_key(f);
        }
        bool take;
        if (all_visible) {
            take = vis;
        } else {
            const bool is_eq = vis && key == T;
            uint32_t eq_tot;
            const uint32_t eq_rank = eq_seen + block_rank(is_eq, warp_sums, &eq_tot);
            take = vis && (key > T || (is_eq && eq_rank < need_eq));
            eq_seen += eq_tot;
        }
        uint32_t tk_tot;
        const uint32_t pos = written + block_rank(take, warp_sums, &tk_tot);
        if (take && pos < k) out[pos] = i;
        written += tk_tot;
        if (written >= m) break;                        // block-uniform
    }
    for (uint32_t i = m + threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
    if (threadIdx.x == 0) count_out[row] = static_cast<int32_t>(m);
}


// ---------------------------------------------------------------- candidates
// Exact top-k of one (u,q) row from the fused indexer's candidate list
// (order-preserving key, row): every row whose key is at or above the row's
// k-th key is in the list (the indexer's threshold never passed it), so the
// selection over the list is the selection over the row.  One CTA per row:
//   1. the k-th key T by radix select over the list (digits 31..20, 19..8,
//      7..0), and need_eq = how many keys equal to T the selection takes;
//   2. a row bitmap: the need_eq lowest rows with key T (a prefix count over
//      the bitmap of tied rows), then every row with key > T;
//   3. the set rows in ascending order (prefix count again), -1 padding.
// The list is cached in shared memory when it fits, else read from global.
constexpr int kCandThreads = 512;
// 6,144 cached candidates (48 KB) let three CTAs share an SM (72 KB each at
// 65,536-row rows; 8,192 allowed two): the decode select runs in fewer waves
// (1,376 rows: 84.5 vs 91 us), and the few lists longer than the cache are
// read from global memory.
constexpr int kCandCache = 6144;

// Block-wide exclusive prefix count of set bits over words [0, nw) of bm,
// thread t owning the contiguous words [t*wpt, (t+1)*wpt).  Returns the
// number of set bits before this thread's words; *total gets the block total.
DS4A_DEV uint32_t bitmap_prefix(const uint32_t *bm, int nw, int wpt, uint32_t *warp_sums, uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t cnt = 0;
    for (int j = 0; j < wpt; ++j) {
        const int w = threadIdx.x * wpt + j;
        if (w < nw) cnt += __popc(bm[w]);
    }
    uint32_t incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    uint32_t before = 0, tot = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
        const uint32_t v = warp_sums[w];
        if (w < warp) before += v;
        tot += v;
    }
    __syncthreads();
    *total = tot;
    return before + incl - cnt;
}

__global__ void __launch_bounds__(kCandThreads) topk_cand_kernel(const __grid_constant__ TopkCandArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(16) uint8_t cand_smem[];
    uint2 *cache = reinterpret_cast<uint2 *>(cand_smem);                          // [kCandCache]
    uint32_t *h = reinterpret_cast<uint32_t *>(cand_smem + kCandCache * 8);       // [kBins]
    uint32_t *bm = h + kBins;                                                      // [ceil(N_cap / 32)]
    __shared__ uint32_t scratch[kCandThreads + 4];
    __shared__ uint32_t warp_sums[32];
    const long long row = blockIdx.x;
    const uint32_t k = static_cast<uint32_t>(a.top_k);
    uint32_t nc = a.cand_n[row];
    if (nc > static_cast<uint32_t>(a.N_cap)) nc = static_cast<uint32_t>(a.N_cap);
    const uint32_t total = a.vis_n[row];
    const uint2 *gc = a.cand + row * a.N_cap;
    const bool cached = nc <= static_cast<uint32_t>(kCandCache);
    if (cached)
        for (uint32_t i = threadIdx.x; i < nc; i += blockDim.x) cache[i] = gc[i];
    const uint2 *c = cached ? cache : gc;
    const int nw = (a.N_cap + 31) / 32;
    const int wpt = (nw + kCandThreads - 1) / kCandThreads;
    for (int i = threadIdx.x; i < nw; i += blockDim.x) bm[i] = 0u;
    __syncthreads();
    if (total <= k) {
        // every visible row is listed (the threshold never rose): take all
        for (uint32_t i = threadIdx.x; i < nc; i += blockDim.x) atomicOr(&bm[c[i].y >> 5], 1u << (c[i].y & 31));
    } else {
        // ---- 1. the k-th key
        uint32_t need = k, prefix = 0;
        const int shifts[3] = {20, 8, 0};
        const uint32_t masks[3] = {0xFFFu, 0xFFFu, 0xFFu};
        for (int d = 0; d < 3; ++d) {
            for (int i = threadIdx.x; i < kBins; i += blockDim.x) h[i] = 0u;
            __syncthreads();
            const int sh = shifts[d];
            const int hs = d == 0 ? 32 : shifts[d - 1];
            for (uint32_t i0 = 0; i0 < nc; i0 += blockDim.x) {        // block-uniform trip count
                const uint32_t i = i0 + threadIdx.x;
                const uint32_t key = i < nc ? c[i].x : 0u;
                hist_add_warp(h, (key >> sh) & masks[d], i < nc && (hs == 32 || (key >> hs) == prefix));
            }
            __syncthreads();
            uint32_t gt, tot;
            int b = find_threshold_bin<kCandThreads>(h, kBins, need, &gt, &tot, scratch);
            if (b < 0) { b = 0; gt = 0; }      // cannot happen: need <= listed keys with this prefix
            prefix = (d == 0 ? 0u : prefix << (d == 1 ? 12 : 8)) | static_cast<uint32_t>(b);
            need -= gt;
        }
        const uint32_t T = prefix;
        // ---- 2. ties at T: the need lowest rows
        for (uint32_t i = threadIdx.x; i < nc; i += blockDim.x)
            if (c[i].x == T) atomicOr(&bm[c[i].y >> 5], 1u << (c[i].y & 31));
        __syncthreads();
        uint32_t ttot;
        uint32_t pos = bitmap_prefix(bm, nw, wpt, warp_sums, &ttot);
        for (int j = 0; j < wpt; ++j) {
            const int w = threadIdx.x * wpt + j;
            if (w >= nw) break;
            uint32_t bits = bm[w], keep = 0;
            while (bits) {
                const uint32_t low = bits & (0u - bits);
                if (pos < need) keep |= low;
                ++pos;
                bits ^= low;
            }
            bm[w] = keep;
        }
        __syncthreads();
        for (uint32_t i = threadIdx.x; i < nc; i += blockDim.x)
            if (c[i].x > T) atomicOr(&bm[c[i].y >> 5], 1u << (c[i].y & 31));
    }
    __syncthreads();
    // ---- 3. ascending output
    uint32_t ns;
    uint32_t pos = bitmap_prefix(bm, nw, wpt, warp_sums, &ns);
    int32_t *out = a.idx + row * a.top_k;
    for (int j = 0; j < wpt; ++j) {
        const int w = threadIdx.x * wpt + j;
        if (w >= nw) break;
        uint32_t bits = bm[w];
        while (bits) {
            const int b = __ffs(bits) - 1;
            bits &= bits - 1;
            if (pos < k) out[pos] = w * 32 + b;
            ++pos;
        }
    }
    ns = ns < k ? ns : k;
    for (uint32_t i = ns + threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
    if (threadIdx.x == 0) a.count[row] = static_cast<int32_t>(ns);
}

}  // namespace

size_t topk_ws_bytes(long long R, int top_k) {
    size_t b = static_cast<size_t>(R) * kBins * 4 + static_cast<size_t>(R) * 16;
    b += ((static_cast<size_t>(R) * top_k * 4 + 15) / 16) * 16;
    b += static_cast<size_t>(R) * kCandCap * 8;
    return b;
}

constexpr int kRowKernelMaxShortRow = 32768;   // rows up to this length take the one-CTA-per-row kernel

cudaError_t launch_topk(const TopkArgs &a, int num_sms, cudaStream_t s) {
    const long long R = static_cast<long long>(a.U) * a.Q;
    if (R >= num_sms || a.N_cap <= kRowKernelMaxShortRow) {
        // Enough rows to fill the GPU, or rows short enough for one CTA each
        // (a single launch beats three on small batches): one CTA per row, no
        // workspace.
        if (R > 0x7fffffffLL) return cudaErrorInvalidValue;
        auto go = [&](auto kern, int nt, int smem) -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            return launch_k(kern, dim3(static_cast<unsigned>(R)), dim3(nt), smem, s, a.scores, a.n_rows, a.Q, a.N_cap,
                            a.top_k, a.idx, a.count, a.status);
        };
        if (a.top_k <= kRowSmallMaxK && a.N_cap <= kRowSmallMaxN)
            return go(topk_row_kernel<256, 4096, 1024>, 256, RowShape<256, 4096, 1024>::kSmem);
        return go(topk_row_kernel<512, 8192, kMaxTopK>, 512, RowShape<512, 8192, kMaxTopK>::kSmem);
    }
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
    e = launch_k(topk_hist_kernel, dim3(grid), dim3(kHistThreads), 0, s, a.scores, a.n_rows, a.Q, a.N_cap, chunk, n_chunks,
                 ws, a.status);
    if (e != cudaSuccess) return e;
    e = launch_k(topk_filter_kernel, dim3(grid), dim3(kHistThreads), 0, s, a.scores, a.n_rows, a.Q, a.N_cap, a.top_k, chunk,
                 n_chunks, ws);
    if (e != cudaSuccess) return e;
    return launch_k(topk_final_kernel, dim3(static_cast<unsigned>(R), 1), dim3(kFinalThreads), 0, s, a.scores, a.n_rows,
                    a.Q, a.N_cap, a.top_k, ws, a.idx, a.count);
}

}  // namespace ds4a

namespace ds4a {
cudaError_t launch_topk_cand(const TopkCandArgs &a, cudaStream_t s) {
    if (a.R <= 0) return cudaSuccess;
    const size_t smem = static_cast<size_t>(kCandCache) * 8 + kBins * 4 + static_cast<size_t>((a.N_cap + 31) / 32) * 4;
    cudaError_t e = cudaFuncSetAttribute(topk_cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_k(topk_cand_kernel, dim3(a.R), dim3(kCandThreads), smem, s, a);
}
}  // namespace ds4a
