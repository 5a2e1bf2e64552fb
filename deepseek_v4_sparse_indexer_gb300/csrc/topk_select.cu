// Top-k row selection per (unit, query) ("DwarfStar(ds4.c) のアーキテクチャを
// 読む" §3-3: only the n_indexer_top_k best-scoring compressed rows reach the
// main attention).
//
// Every path compares scores through an order-preserving 32-bit key
// (float_key: a > b as floats, -0 == +0, implies key(a) > key(b)).  A
// selection is the rows whose key is above the k-th largest key T, then the
// lowest-index rows whose key equals T until k rows are taken; they are
// written in ascending row order, then -1 padding.
//
// The row is first cut down to a short candidate list: a sample of the row's
// scores gives a threshold T0 near the key of rank 3k (2k for the smallest
// row shape), and every visible row with key >= T0 becomes a candidate.  The
// list decides the selection exactly when it holds at least k rows (then
// T >= T0, and every row at or above T is listed) or, when the row has at most
// k visible scores, all of them.  Over the list, T comes from a count of the
// candidates in 32 buckets of their key range (ballots, no atomics) and a rank
// (or an 8-bit-per-round narrowing) of the keys in the bucket where the count
// from the top reaches k; the chosen rows go out through a bitmap of the row,
// a count of smaller rows, or a bitonic sort.  Otherwise (a sample that missed,
// heavy ties) T is found over the whole row by 8-bit radix digits in 256-bin
// shared-memory histograms, which is exact whatever the scores.
//
// Four launch shapes:
//   topk_cluster_kernel     up to 16 rows of 4,097 .. 524,288 scores (long-
//                           context and small decode batches): a cluster of
//                           eight CTAs per row (sixteen for up to 4 rows), the
//                           selection agreed through distributed shared memory
//                           (up to 8 rows: each CTA's chunk comes in by bulk
//                           copies);
//   topk_split_kernel +     up to 76 rows of more than 524,288 scores: C CTAs
//   topk_split_final_kernel per row each filter a chunk of the row against the
//                           same T0 into a candidate slot of their own in the
//                           workspace; then one CTA per row selects;
//   topk_row_kernel         one CTA per row: everything else (decode batches,
//                           prefill chunks, short rows);
//   topk_cand_kernel        the candidate lists of the fused indexer scan.
#include "common.cuh"
#include "internal.h"

namespace ds4a {
namespace {

constexpr int kDigitBins = 256;        // 8-bit radix digits: four per key
constexpr int kSampleRow = 2048;       // scores sampled for the threshold T0: one CTA per row
constexpr int kSampleSplit = 4096;     // and split rows (longer, heavier tails)
constexpr int kSampleOver = 3;         // expected candidates / k
constexpr int kSplitThreads = 256;
constexpr int kSplitFinalThreads = 512;
constexpr int kSplitCache = 8192;      // candidates a split row's final CTA holds in shared memory

DS4A_DEV int clamp_rows(int n, int N_cap) { return n < 0 ? 0 : (n > N_cap ? N_cap : n); }
DS4A_DEV int row_len(const int32_t *n_rows, int u, int N_cap) { return clamp_rows(n_rows[u], N_cap); }

// Shared scratch of the block-wide selection helpers.
struct __align__(16) SelSmem {
    uint32_t h[2][kDigitBins];         // digit histograms (alternating)
    uint32_t bc[4];                    // broadcast words
    uint32_t cnt[4];                   // block counters
    uint32_t mm[4];                    // smallest and largest candidate key (2 used: uni 16-byte aligned)
    uint32_t warp_sums[32];
    uint32_t uni[128];                 // the warps' largest sample keys (threshold estimate)
};
static_assert(offsetof(SelSmem, uni) % 16 == 0, "uni is read as uint4");
constexpr int kFastList = 1024;        // keys of the crossing bucket the one-warp search takes

// Clears what select_from_list expects cleared (counters, key range).  A
// __syncthreads must follow before any thread uses them (the key-range fold
// included).
DS4A_DEV void sel_reset(SelSmem &S) {
    if (threadIdx.x == 0) {
        S.cnt[0] = S.cnt[1] = S.cnt[2] = S.cnt[3] = 0u;
        S.mm[0] = 0xffffffffu;
        S.mm[1] = 0u;
    }
}
// Folds every lane's (smallest, largest) key into S.mm (all 32 lanes call it;
// lanes with no key pass 0xffffffff, 0).
DS4A_DEV void warp_fold_minmax(uint32_t kmn, uint32_t kmx, SelSmem &S) {
    kmn = __reduce_min_sync(0xffffffffu, kmn);
    kmx = __reduce_max_sync(0xffffffffu, kmx);
    if ((threadIdx.x & 31) == 0) {
        if (kmn != 0xffffffffu) atomicMin(&S.mm[0], kmn);
        if (kmx != 0u) atomicMax(&S.mm[1], kmx);
    }
}

// Warp-aggregated append of `val` to dst[*counter ...] for the lanes with
// pred (entries past cap are dropped; the counter still counts them).  All 32
// lanes call it.
template <typename T>
DS4A_DEV void warp_append(T *dst, uint32_t *counter, uint32_t cap, bool pred, T val) {
    const uint32_t bal = __ballot_sync(0xffffffffu, pred);
    if (bal == 0) return;
    const int lane = threadIdx.x & 31;
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(counter, static_cast<uint32_t>(__popc(bal)));
    base = __shfl_sync(0xffffffffu, base, 0);
    const uint32_t p = base + __popc(bal & ((1u << lane) - 1u));
    if (pred && p < cap) dst[p] = val;
}

// Warp-wide (all 32 lanes): in the 256-bin histogram h, the largest bin b with
// sum_{b' >= b} h[b'] >= k, and the count strictly above b in *above.  b = -1
// when the total is below k (then *above = the total).  Lane l holds bins
// 8l .. 8l+7; one suffix scan over the lanes finds the crossing lane, which
// walks its eight bins from the top in registers.
DS4A_DEV int warp_find_bin(const uint32_t *h, uint32_t k, uint32_t *above) {
    const int lane = threadIdx.x & 31;
    const uint4 v0 = reinterpret_cast<const uint4 *>(h)[2 * lane];
    const uint4 v1 = reinterpret_cast<const uint4 *>(h)[2 * lane + 1];
    const uint32_t c[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += c[j];
    uint32_t suf = s;                                   // sum over lanes >= this one
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, suf, off);
        if (lane + off < 32) suf += v;
    }
    const uint32_t hit = __ballot_sync(0xffffffffu, suf >= k);
    if (hit == 0) {
        *above = __shfl_sync(0xffffffffu, suf, 0);
        return -1;
    }
    const int L = 31 - __clz(hit);
    uint32_t run = suf - s;                             // count above this lane's bins
    int b = 0;
    uint32_t ab = 0;
    if (lane == L) {
        b = 8 * L;
        ab = run + c[1] + c[2] + c[3] + c[4] + c[5] + c[6] + c[7];
#pragma unroll
        for (int j = 7; j >= 1; --j) {
            if (run + c[j] >= k) {
                b = 8 * L + j;
                ab = run;
                break;
            }
            run += c[j];
        }
    }
    *above = __shfl_sync(0xffffffffu, ab, L);
    return __shfl_sync(0xffffffffu, b, L);
}

// Block-wide k-th largest key among the valid keys get(i) (i < n), by four
// 8-bit digits.  Needs at least k valid keys.  Returns T and, in *need_eq,
// how many keys equal to T a selection of k takes.  get(i, valid, key) is
// called for i < n; every thread calls this function.
template <int NT, class Get>
DS4A_DEV uint32_t block_kth_key(Get get, uint32_t n, uint32_t k, SelSmem &S, uint32_t *need_eq) {
    static_assert(NT >= 64 && NT % 32 == 0, "block size");
    for (int i = threadIdx.x; i < kDigitBins; i += NT) S.h[0][i] = 0u;
    __syncthreads();
    uint32_t prefix = 0, need = k;
#pragma unroll 1
    for (int d = 0; d < 4; ++d) {
        const int sh = 24 - 8 * d;
        uint32_t *h = S.h[d & 1];
        for (uint32_t i0 = 0; i0 < n; i0 += NT) {                  // block-uniform trip count
            const uint32_t i = i0 + threadIdx.x;
            bool v = false;
            uint32_t key = 0;
            if (i < n) get(i, v, key);
            const bool take = v && (d == 0 || (key >> (sh + 8)) == prefix);
            hist_add_warp(h, (key >> sh) & 0xFFu, take);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            uint32_t above;
            const int b = warp_find_bin(h, need, &above);
            if (threadIdx.x == 0) {
                S.bc[0] = static_cast<uint32_t>(b < 0 ? 0 : b);     // b < 0 cannot happen: >= k valid keys
                S.bc[1] = b < 0 ? 0u : above;
            }
        } else if (d < 3) {
            for (int i = threadIdx.x - 32; i < kDigitBins; i += NT - 32) S.h[(d + 1) & 1][i] = 0u;
        }
        __syncthreads();
        prefix = (prefix << 8) | S.bc[0];
        need -= S.bc[1];
    }
    *need_eq = need;
    return prefix;
}

// One warp (all 32 lanes): the need-th largest key among the keys of list[0 ..
// L) that lie in [lo, lo + 2^cs) (at least `need` of them do), by narrowing the
// range 8 bits per round with a warp-private 256-bin histogram (S.h[1]).
// Lane 0 leaves the key in S.bc[2] and how many keys equal to it the `need`
// largest take in S.bc[3].
DS4A_DEV void warp_narrow(const uint32_t *list, uint32_t L, uint32_t lo, int cs, uint32_t need, SelSmem &S) {
    const int lane = threadIdx.x & 31;
    uint32_t *h = S.h[1];
    while (cs > 0) {
        const int s2 = cs > 8 ? cs - 8 : 0;
        for (int i = lane; i < kDigitBins; i += 32) h[i] = 0u;
        __syncwarp();
        for (uint32_t i = lane; i < L; i += 32) {
            const uint32_t d = list[i] - lo;
            if (d < (1u << cs)) atomicAdd(&h[d >> s2], 1u);
        }
        __syncwarp();
        uint32_t above;
        const int b = warp_find_bin(h, need, &above);           // >= 0: the range holds >= need keys
        need -= b < 0 ? 0u : above;
        lo += static_cast<uint32_t>(b < 0 ? 0 : b) << s2;
        cs = s2;
        __syncwarp();
    }
    if (lane == 0) {
        S.bc[2] = lo;
        S.bc[3] = need;
    }
}

// Block-wide k-th largest key among the list keys c[0 .. nc) (nc >= k >= 1),
// all in [kmin, kmax], by buckets fitted to that range: 32 buckets of
// (key - kmin) >> s, s the least shift that leaves at most 32, counted by
// ballots (no atomics), find the bucket holding the k-th key; its keys are
// copied to `list` and one warp narrows the bucket by 8 bits per round (a
// warp-private histogram) until it is one key wide.  Returns false (the
// caller then takes block_kth_key) when the bucket holds more than kFastList
// keys.  Expects S.cnt[2] cleared (sel_reset).
template <int NT>
DS4A_DEV bool fast_kth(const uint2 *c, uint32_t nc, uint32_t k, uint32_t kmin, uint32_t kmax, uint32_t *list,
                       SelSmem &S, uint32_t *T_out, uint32_t *need_eq_out) {
    constexpr int kWarps = NT / 32;
    static_assert(kWarps <= 16, "warp counts live in the two digit histograms");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t range = kmax - kmin;
    const int s = range > 31u ? 27 - __clz(range) : 0;      // (range >> s) < 32
    // 32 buckets counted without atomics: per 32 keys, five ballots of the
    // bucket bits; lane b keeps the count of bucket b.
    uint32_t mine = 0;
    for (uint32_t i0 = warp * 32; i0 < nc; i0 += NT) {        // warp-uniform trip count
        const uint32_t i = i0 + lane;
        const bool v = i < nc;
        const uint32_t b = v ? (c[i].x - kmin) >> s : 0u;
        uint32_t match = __ballot_sync(0xffffffffu, v);
#pragma unroll
        for (int bit = 0; bit < 5; ++bit) {
            const uint32_t m = __ballot_sync(0xffffffffu, (b >> bit) & 1u);
            match &= ((lane >> bit) & 1) ? m : ~m;
        }
        mine += __popc(match);
    }
    uint32_t *wc = &S.h[0][0];                               // [kWarps][32] per-warp bucket counts
    wc[warp * 32 + lane] = mine;
    __syncthreads();
    if (warp == 0) {
        uint32_t cnt = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) cnt += wc[w * 32 + lane];
        uint32_t suf = cnt;                                  // keys in buckets >= lane
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t t = __shfl_down_sync(0xffffffffu, suf, off);
            if (lane + off < 32) suf += t;
        }
        const uint32_t hit = __ballot_sync(0xffffffffu, suf >= k);
        const int L = hit ? 31 - __clz(hit) : 0;             // hit != 0: nc >= k
        const uint32_t above = __shfl_sync(0xffffffffu, suf - cnt, L);
        if (lane == 0) {
            S.bc[0] = static_cast<uint32_t>(L);
            S.bc[1] = above;
        }
    }
    __syncthreads();
    const uint32_t b0 = S.bc[0];
    uint32_t need = k - S.bc[1];
    uint32_t lo = kmin + (b0 << s);
    if (s == 0) {                                            // one key per bucket
        *T_out = lo;
        *need_eq_out = need;
        return true;
    }
    for (uint32_t i0 = 0; i0 < nc; i0 += NT) {                  // block-uniform trip count
        const uint32_t i = i0 + threadIdx.x;
        const uint32_t key = i < nc ? c[i].x : 0u;
        warp_append<uint32_t>(list, &S.cnt[2], kFastList, i < nc && ((key - kmin) >> s) == b0, key);
    }
    __syncthreads();
    const uint32_t L = S.cnt[2];
    if (L > static_cast<uint32_t>(kFastList)) return false;     // block-uniform
    if (L <= static_cast<uint32_t>(NT < 256 ? NT : 256)) {
        // Few keys: thread i ranks key i against the whole bucket (16-byte
        // loads every lane of a warp shares); the key with fewer than `need`
        // larger keys and at least `need` at or above it is T.
        if (threadIdx.x < L) {
            const uint32_t v = list[threadIdx.x];
            const uint4 *l4 = reinterpret_cast<const uint4 *>(list);
            uint32_t gt = 0, ge = 0;
            for (uint32_t j = 0; j < L / 4; ++j) {
                const uint4 o = l4[j];
                gt += (o.x > v) + (o.y > v) + (o.z > v) + (o.w > v);
                ge += (o.x >= v) + (o.y >= v) + (o.z >= v) + (o.w >= v);
            }
            for (uint32_t j = L & ~3u; j < L; ++j) {
                gt += list[j] > v;
                ge += list[j] >= v;
            }
            if (gt < need && ge >= need) {                       // every such thread holds the same key
                S.bc[2] = v;
                S.bc[3] = need - gt;
            }
        }
        __syncthreads();
        *T_out = S.bc[2];
        *need_eq_out = S.bc[3];
        return true;
    }
    if (threadIdx.x < 32) warp_narrow(list, L, lo, s, need, S);
    __syncthreads();
    *T_out = S.bc[2];
    *need_eq_out = S.bc[3];
    return true;
}

// Block-wide ascending sort of a[0 .. n_pow2) (n_pow2 a power of two).
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

// Writes the rows sel[0 .. m) (distinct, each < n_bound) in ascending order
// to out[0 .. k) with -1 padding, and the count.  Rows below 131,072 with the
// bitmap room below: the bitmap.  Otherwise up to 512 rows: each row's rank
// by counting (sel 16-byte aligned).  Otherwise, when a bitmap of n_bound
// bits fits bm (bm_words words of shared memory): the rows' bits are set,
// the popcounts of each 32-word chunk summed and scanned, and every lane then
// writes the set bits of one word at the place the chunk and lane prefixes
// give (no sort; a handful of barriers).  Otherwise, up to 1,024 rows: a bitonic sort held in
// registers (E = p2 / threads elements per thread, each warp owning whole
// 32-element chunks), whose exchanges with partners less than 32 apart are
// warp shuffles and the others go through shared memory (sel and tmp
// alternating, one barrier per such stage).  Larger sets sort in sel in
// place.  sel must have room for the next power of two >= max(m, 32) when m
// > 1,024; tmp: shared int32 [1,024].
DS4A_DEV void write_sorted(int32_t *sel, int32_t *tmp, uint32_t *bm, int bm_words, int n_bound, uint32_t m,
                           uint32_t k, int32_t *out, int32_t *count_out) {
    const int nt = blockDim.x;
    const int words = (n_bound + 31) / 32, chunks = (words + 31) / 32;
    const bool bitmap = m > 1 && chunks * 32 <= bm_words && chunks <= 1024;
    if (m > 1 && m <= 512 && !(bitmap && chunks <= 128)) {
        // Each row goes to its rank: the count of smaller rows, from 16-byte
        // loads of sel that every lane of a warp shares (no barrier, no sort).
        const int4 *s4 = reinterpret_cast<const int4 *>(sel);
        const int m4 = static_cast<int>(m) >> 2;
        for (uint32_t i = threadIdx.x; i < m; i += nt) {
            const int32_t e = sel[i];
            int r = 0;
            for (int j = 0; j < m4; ++j) {
                const int4 v = s4[j];
                r += (v.x < e) + (v.y < e) + (v.z < e) + (v.w < e);
            }
            for (int j = 4 * m4; j < static_cast<int>(m); ++j) r += sel[j] < e;
            out[r] = e;
        }
        for (uint32_t i = m + threadIdx.x; i < k; i += nt) out[i] = -1;
        if (threadIdx.x == 0) *count_out = static_cast<int32_t>(m);
        return;
    }
    if (bitmap) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = nt >> 5;
        for (int i = threadIdx.x; i < chunks * 32; i += nt) bm[i] = 0u;
        __syncthreads();
        for (uint32_t i = threadIdx.x; i < m; i += nt) {
            const int32_t r = sel[i];
            if (r >= 0 && r < chunks * 1024) atomicOr(&bm[r >> 5], 1u << (r & 31));   // (always in range)
        }
        __syncthreads();
        for (int ch = warp; ch < chunks; ch += nw) {
            const uint32_t c = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(__popc(bm[ch * 32 + lane])));
            if (lane == 0) tmp[ch] = static_cast<int32_t>(c);
        }
        __syncthreads();
        if (warp == 0) {                                     // exclusive scan of the chunk counts
            const int per = (chunks + 31) / 32;
            int32_t run = 0;
            for (int j = 0; j < per; ++j) {
                const int ch = lane * per + j;
                run += ch < chunks ? tmp[ch] : 0;
            }
            int32_t incl = run;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int32_t t = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += t;
            }
            int32_t base = incl - run;
            for (int j = 0; j < per; ++j) {
                const int ch = lane * per + j;
                if (ch < chunks) {
                    const int32_t v = tmp[ch];
                    tmp[ch] = base;
                    base += v;
                }
            }
        }
        __syncthreads();
        for (int ch = warp; ch < chunks; ch += nw) {
            uint32_t w = bm[ch * 32 + lane];
            const int32_t c = __popc(w);
            int32_t incl = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int32_t t = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += t;
            }
            int32_t pos = tmp[ch] + incl - c;
            const int32_t row0 = (ch * 32 + lane) * 32;
            while (w) {
                const int b = __ffs(w) - 1;
                w &= w - 1;
                if (pos < static_cast<int32_t>(k)) out[pos] = row0 + b;
                ++pos;
            }
        }
        for (uint32_t i = m + threadIdx.x; i < k; i += nt) out[i] = -1;
        if (threadIdx.x == 0) *count_out = static_cast<int32_t>(m);
        return;
    }
    int p2 = 32;
    while (p2 < static_cast<int>(m)) p2 <<= 1;
    if (p2 > 1024) {
        for (int i = static_cast<int>(m) + threadIdx.x; i < p2; i += nt) sel[i] = 0x7fffffff;
        __syncthreads();
        block_bitonic_sort_asc(sel, p2);
        for (uint32_t i = threadIdx.x; i < k; i += nt) out[i] = i < m ? sel[i] : -1;
    } else {
        constexpr int kMaxE = 4;       // p2 / threads: 1,024 / 256, or 512 / 128 (the 128-thread shape has k <= 512)
        const int E = p2 > nt ? p2 / nt : 1;
        const bool active = static_cast<int>(threadIdx.x) < p2;  // warp-uniform (p2 >= 32)
        int32_t x[kMaxE];
#pragma unroll
        for (int e = 0; e < kMaxE; ++e) {
            const int i = threadIdx.x + e * nt;
            x[e] = (e < E && active && i < static_cast<int>(m)) ? sel[i] : 0x7fffffff;
        }
        int cur = 0;
        __syncthreads();                                         // every read of sel done
        for (int k2 = 2; k2 <= p2; k2 <<= 1) {
            for (int j = k2 >> 1; j > 0; j >>= 1) {
                if (j >= 32) {
                    int32_t *d = cur ? tmp : sel;
                    cur ^= 1;
#pragma unroll
                    for (int e = 0; e < kMaxE; ++e)
                        if (e < E && active) d[threadIdx.x + e * nt] = x[e];
                    __syncthreads();
#pragma unroll
                    for (int e = 0; e < kMaxE; ++e) {
                        if (e < E && active) {
                            const int i = threadIdx.x + e * nt;
                            const int32_t y = d[i ^ j];
                            x[e] = (((i & j) == 0) == ((i & k2) == 0)) ? min(x[e], y) : max(x[e], y);
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < kMaxE; ++e) {
                        if (e < E) {                             // uniform
                            const int i = threadIdx.x + e * nt;
                            const int32_t y = __shfl_xor_sync(0xffffffffu, x[e], j);
                            x[e] = (((i & j) == 0) == ((i & k2) == 0)) ? min(x[e], y) : max(x[e], y);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int e = 0; e < kMaxE; ++e) {
            const int i = threadIdx.x + e * nt;
            if (e < E && active && i < static_cast<int>(m)) out[i] = x[e];
        }
        for (uint32_t i = m + threadIdx.x; i < k; i += nt) out[i] = -1;
    }
    if (threadIdx.x == 0) *count_out = static_cast<int32_t>(m);
}

// The selection from a candidate list c[0 .. nc) of (key, row) that decides
// it: total = visible rows of the row; when total <= k the list holds all of
// them, otherwise at least k and every row whose key is at or above the k-th.
// Expects sel_reset(S) and a barrier since, and S.mm = the list's smallest and
// largest key.  sel: shared int32 with room for the next power of two >= k
// (and >= 32); list: shared u32 [kFastList].  Tied rows beyond kFastList are
// resolved by an in-place compaction of their rows into c (read-write here).
// bm / bm_words: shared memory free once the list has been read (the list's
// own cache, when it is one) for the output bitmap; n_bound: rows are < it.
template <int NT>
DS4A_DEV void select_from_list(uint2 *c, uint32_t nc, uint32_t total, uint32_t k, int32_t *sel, uint32_t *list,
                               SelSmem &S, uint32_t *bm, int bm_words, int n_bound, int32_t *out,
                               int32_t *count_out) {
    if (total <= k) {
        for (uint32_t i = threadIdx.x; i < nc; i += NT) sel[i] = static_cast<int32_t>(c[i].y);
        __syncthreads();
        write_sorted(sel, reinterpret_cast<int32_t *>(list), bm, bm_words, n_bound, nc < k ? nc : k, k, out,
                     count_out);
        return;
    }
    uint32_t T, need_eq;
    if (!fast_kth<NT>(c, nc, k, S.mm[0], S.mm[1], list, S, &T, &need_eq))
        T = block_kth_key<NT>([&](uint32_t i, bool &v, uint32_t &key) { v = true; key = c[i].x; }, nc, k, S,
                              &need_eq);
    // rows above T into sel, rows equal to T into the tie list
    int32_t *tie = reinterpret_cast<int32_t *>(list);
    for (uint32_t i0 = 0; i0 < nc; i0 += NT) {
        const uint32_t i = i0 + threadIdx.x;
        const uint2 e = i < nc ? c[i] : make_uint2(0u, 0u);
        warp_append<int32_t>(sel, &S.cnt[0], k, i < nc && e.x > T, static_cast<int32_t>(e.y));
        warp_append<int32_t>(tie, &S.cnt[1], kFastList, i < nc && e.x == T, static_cast<int32_t>(e.y));
    }
    __syncthreads();
    const uint32_t n_gt = S.cnt[0], n_eq = S.cnt[1];     // n_gt = k - need_eq
    if (n_eq == need_eq) {
        for (uint32_t i = threadIdx.x; i < n_eq; i += NT) sel[n_gt + i] = tie[i];
    } else if (n_eq <= static_cast<uint32_t>(kFastList)) {
        // More rows tie at T than the selection takes: the lowest rows win.
        int p2 = 1;
        while (p2 < static_cast<int>(n_eq)) p2 <<= 1;
        for (int i = static_cast<int>(n_eq) + threadIdx.x; i < p2; i += NT) tie[i] = 0x7fffffff;
        __syncthreads();
        block_bitonic_sort_asc(tie, p2);
        for (uint32_t i = threadIdx.x; i < need_eq; i += NT) sel[n_gt + i] = tie[i];
    } else {
        // Very many ties: compact the tied rows in place (round r writes below
        // the entries round r+1 reads), sort them and take the first need_eq.
        int32_t *tc = reinterpret_cast<int32_t *>(c);
        uint32_t w = 0;
        for (uint32_t i0 = 0; i0 < nc; i0 += NT) {
            const uint32_t i = i0 + threadIdx.x;
            const uint2 e = i < nc ? c[i] : make_uint2(0u, 0u);
            const bool is_eq = i < nc && e.x == T;
            uint32_t tot;
            const uint32_t r = block_rank(is_eq, S.warp_sums, &tot);      // synchronises: reads done
            if (is_eq) tc[w + r] = static_cast<int32_t>(e.y);
            w += tot;
            __syncthreads();
        }
        int p2 = 1;
        while (p2 < static_cast<int>(w)) p2 <<= 1;
        for (int i = static_cast<int>(w) + threadIdx.x; i < p2; i += NT) tc[i] = 0x7fffffff;
        __syncthreads();
        block_bitonic_sort_asc(tc, p2);
        for (uint32_t i = threadIdx.x; i < need_eq; i += NT) sel[n_gt + i] = tc[i];
    }
    __syncthreads();
    write_sorted(sel, tie, bm, bm_words, n_bound, k, k, out, count_out);
}

// Exact selection over the whole row s[0 .. n) (global memory), whatever the
// scores: the visible count, the k-th key by four digit passes over the row,
// then an order-preserving compaction of the chosen rows (ascending output).
template <int NT>
DS4A_DEV void select_exact_row(const float *__restrict__ s, int n, uint32_t k, SelSmem &S, int32_t *out,
                               int32_t *count_out) {
    uint32_t my_vis = 0;
    for (int i = threadIdx.x; i < n; i += NT) my_vis += score_visible(s[i]) ? 1u : 0u;
    uint32_t total;
    {
        uint32_t v = my_vis;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if ((threadIdx.x & 31) == 0) S.warp_sums[threadIdx.x >> 5] = v;
        __syncthreads();
        total = 0;
        for (int w = 0; w < NT / 32; ++w) total += S.warp_sums[w];
        __syncthreads();
    }
    const uint32_t m = total < k ? total : k;
    uint32_t T = 0, need_eq = 0;
    const bool all = total <= k;
    if (!all)
        T = block_kth_key<NT>(
            [&](uint32_t i, bool &v, uint32_t &key) {
                const float f = s[i];
                v = score_visible(f);
                key = float_key(f);
            },
            static_cast<uint32_t>(n), k, S, &need_eq);
    uint32_t written = 0, eq_seen = 0;
    for (int base = 0; base < n && written < m; base += NT) {     // block-uniform
        const int i = base + static_cast<int>(threadIdx.x);
        bool vis = false;
        uint32_t key = 0;
        if (i < n) {
            const float f = s[i];
            vis = score_visible(f);
            key = float_key(f);
        }
        bool take = vis;
        if (!all) {
            const bool is_eq = vis && key == T;
            uint32_t eq_tot;
            const uint32_t eq_rank = eq_seen + block_rank(is_eq, S.warp_sums, &eq_tot);
            take = vis && (key > T || (is_eq && eq_rank < need_eq));
            eq_seen += eq_tot;
        }
        uint32_t tk_tot;
        const uint32_t pos = written + block_rank(take, S.warp_sums, &tk_tot);
        if (take && pos < k) out[pos] = i;
        written += tk_tot;
    }
    for (uint32_t i = m + threadIdx.x; i < k; i += NT) out[i] = -1;
    if (threadIdx.x == 0) *count_out = static_cast<int32_t>(m);
}

// Threshold estimate for a row of n > all_below >= 4,096 scores: a key T0 with
// about (or a little more than) kOver * k of the row's visible keys at or
// above it, from up to kSample scores (whole 128-byte lines spread evenly over the row, so
// that the sample costs whole lines, not scattered sectors).  Each
// warp's share of the sample is spread over the whole row; a warp pulls out
// its rw largest visible keys by rw rounds of a warp-wide max (rw = ceil(r /
// warps) + 2 for the wanted sample rank r), and T0 is the r-th largest key of
// the union of the warps' lists (when the union does not fit, the smallest of
// the warps' last keys), so at least r sample keys lie at or above it.  0
// (every visible row) when n <= all_below or the sample has fewer than r
// visible keys.
template <int NT, int kSample, int kOver = kSampleOver>
DS4A_DEV uint32_t sample_threshold(const float *__restrict__ s, int n, uint32_t k, int all_below, SelSmem &S) {
    if (n <= all_below) return 0u;
    constexpr int kPer = kSample / NT;
    constexpr int kWarps = NT / 32;
    // Shorter rows take a smaller sample (at least NT and 1,024 scores): the
    // wanted sample rank stays near 64 instead of growing with kSample / n.
    int samples = kSample;
    while (samples > NT && samples > 1024 &&
           static_cast<long long>(kOver) * k * (samples / 2) >= 64LL * n)
        samples >>= 1;
    const int per = samples / NT, lines = samples / 32;
    const int lsh = 31 - __clz(lines);                        // lines is a power of two
    uint32_t key[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        key[j] = 0u;                                          // visible keys are >= 0x00800000
        if (j < per) {
            // line li of the sample: row line li * (n / 32) / lines (n / 32 >= lines:
            // distinct lines, the last one inside the row)
            const int sj = static_cast<int>(threadIdx.x) + j * NT;
            const int line = static_cast<int>((static_cast<long long>(sj >> 5) * (n >> 5)) >> lsh);
            const float f = __ldg(s + line * 32 + (sj & 31));
            key[j] = score_visible(f) ? float_key(f) : 0u;
        }
    }
    const long long r_want = (static_cast<long long>(kOver) * k * samples + n - 1) / n;
    const int r = static_cast<int>(r_want < samples ? r_want : samples);
    // rw = the wanted rank's share per warp and two more, so that the union of
    // the warps' lists most likely holds the sample's r largest keys; when the
    // union would not fit (short rows, large r), each warp takes its share
    // and T0 is the smallest of the warps' last keys (a looser threshold).
    constexpr int kUni = 128 / kWarps;
    const int share = (r + kWarps - 1) / kWarps;
    const bool use_union = share + 2 <= kUni;
    const int rw = min(use_union ? share + 2 : share, kPer * 32);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t t = 0;
    for (int round = 0; round < rw; ++round) {
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) m = max(m, key[j]);
        t = __reduce_max_sync(0xffffffffu, m);
        if (use_union && lane == 0) S.uni[warp * kUni + round] = t;
        if (t == 0u) break;                                   // warp-uniform
        const uint32_t holders = __ballot_sync(0xffffffffu, m == t);
        if (lane == __ffs(holders) - 1) {
            bool done = false;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const bool hit = !done && key[j] == t;
                key[j] = hit ? 0u : key[j];
                done |= hit;
            }
        }
    }
    if (use_union && lane == 0)
        for (int round = rw; round < kUni; ++round) S.uni[warp * kUni + round] = 0u;   // past a warp's visible keys
    if (lane == 0) S.warp_sums[warp] = t;
    if (threadIdx.x == 0) S.bc[3] = 0u;
    __syncthreads();
    uint32_t T0;
    if (use_union) {
        // the r-th largest of the union's 128 keys: thread i < 128 counts the
        // keys above and at key i (16-byte loads that every lane of a warp
        // shares); the key with fewer than r above it and at least r at or
        // above it is T0 (0 when the sample has fewer than r visible keys)
        static_assert(NT >= 128 && sizeof(S.uni) == 512, "one thread per union entry");
        if (threadIdx.x < 128) {
            const uint32_t v = S.uni[threadIdx.x];
            const uint4 *u4 = reinterpret_cast<const uint4 *>(S.uni);
            uint32_t gt = 0, ge = 0;
#pragma unroll 8
            for (int j = 0; j < 32; ++j) {
                const uint4 o = u4[j];
                gt += (o.x > v) + (o.y > v) + (o.z > v) + (o.w > v);
                ge += (o.x >= v) + (o.y >= v) + (o.z >= v) + (o.w >= v);
            }
            if (gt < static_cast<uint32_t>(r) && ge >= static_cast<uint32_t>(r)) S.bc[3] = v;   // all such threads agree
        }
        __syncthreads();
        T0 = S.bc[3];
    } else {
        T0 = 0xffffffffu;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) T0 = min(T0, S.warp_sums[w]);
    }
    __syncthreads();                                         // S reusable after this
    return T0;
}

// ---------------------------------------------------------------- one CTA per row
// 1. T0 from the sample (0 when the row fits the candidate list whole);
// 2. one pass over the row (float4 loads, the next batch in flight, one ballot
//    per float4, one shared atomic per warp and float4) counts the visible
//    scores and appends every row with key >= T0 to the shared candidate list;
// 3. the selection from the list when it decides it, else from the row.
// Three shapes: 512 threads and 8,192 candidates (any k), two CTAs per SM; for
// k <= kRowSmallMaxK 256 threads, 4,096 candidates, four CTAs per SM; and for
// k <= kRowTinyMaxK in batches of at least four rows per SM, 128 threads, 2,048
// candidates (the threshold aimed at 2k), eight CTAs per SM.  A row's phases
// are latency-bound: more rows in flight beat more threads per row.
constexpr int kRowSmallMaxK = 640;
constexpr int kRowTinyMaxK = 512;
template <int NT, int CAP, int SEL>
struct RowShape {
    static constexpr int kSmem = CAP * 8 + SEL * 4 + kFastList * 4 + static_cast<int>(sizeof(SelSmem));
};

template <int NT, int CAP, int SEL>
__global__ void __launch_bounds__(NT, 1024 / NT) topk_row_kernel(const float *__restrict__ scores,
                                                                  const int32_t *__restrict__ n_rows, int Q,
                                                                  int N_cap, int top_k,
                                                                  int32_t *__restrict__ idx_out,
                                                                  int32_t *__restrict__ count_out, uint32_t *status) {
    pdl_launch_dependents();
    const long long row = blockIdx.x;
    const int u = static_cast<int>(row / Q);
    const int n_given = n_rows[u];                      // no kernel of this library writes n_rows
    const int n = clamp_rows(n_given, N_cap);
    pdl_wait();
    extern __shared__ __align__(16) uint8_t row_smem[];
    uint2 *cand = reinterpret_cast<uint2 *>(row_smem);                          // [CAP]
    int32_t *sel = reinterpret_cast<int32_t *>(row_smem + CAP * 8);             // [SEL]
    uint32_t *list = reinterpret_cast<uint32_t *>(row_smem + CAP * 8 + SEL * 4);   // [kFastList]
    SelSmem &S = *reinterpret_cast<SelSmem *>(row_smem + CAP * 8 + SEL * 4 + kFastList * 4);
    if (threadIdx.x == 0 && row % Q == 0 && n != n_given) report(status, DS4A_DEV_BOUNDS);
    const float *s = scores + row * N_cap;
    const uint32_t k = static_cast<uint32_t>(top_k);
    int32_t *out = idx_out + row * top_k;
    const int lane = threadIdx.x & 31;

    constexpr int B = 4;
    const int ngroups = (n + 3) / 4;
    const bool vec4 = (N_cap & 3) == 0 && (reinterpret_cast<uintptr_t>(scores) & 15) == 0;
    auto load = [&](float4 (&v)[B], int g0) {
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int g = g0 + j * NT + static_cast<int>(threadIdx.x);
            v[j] = g < ngroups ? __ldg(reinterpret_cast<const float4 *>(s) + g) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    float4 cur[B], nxt[B];
    if (vec4) load(cur, 0);                              // in flight during the threshold estimate
    // 2,048 candidates (128 threads) aim at 2k, the larger lists at 3k
    const uint32_t T0 = sample_threshold<NT, kSampleRow, CAP <= 2048 ? 2 : kSampleOver>(s, n, k, CAP, S);
    sel_reset(S);
    __syncthreads();
    uint32_t my_vis = 0, kmn = 0xffffffffu, kmx = 0u;      // visible count, candidates' key range
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
                    kmn = take[c] ? min(kmn, key[c]) : kmn;
                    kmx = take[c] ? max(kmx, key[c]) : kmx;
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
                    if (lane == 0) pos = atomicAdd(&S.cnt[3], tot);
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
            const bool take = vis && key >= T0;
            kmn = take ? min(kmn, key) : kmn;
            kmx = take ? max(kmx, key) : kmx;
            warp_append<uint2>(cand, &S.cnt[3], CAP, take, make_uint2(key, static_cast<uint32_t>(i)));
        }
    }
    warp_fold_minmax(kmn, kmx, S);
    uint32_t total;
    {
        uint32_t v = my_vis;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) S.warp_sums[threadIdx.x >> 5] = v;
        __syncthreads();
        total = 0;
        for (int w = 0; w < NT / 32; ++w) total += S.warp_sums[w];
    }
    const uint32_t nc = S.cnt[3];
    __syncthreads();
    const bool decides = total <= k ? nc == total : (nc >= k && nc <= static_cast<uint32_t>(CAP));
    if (decides)
        select_from_list<NT>(cand, nc, total, k, sel, list, S, reinterpret_cast<uint32_t *>(cand), 2 * CAP, n, out,
                             count_out + row);
    else
        select_exact_row<NT>(s, n, k, S, out, count_out + row);
}

// ---------------------------------------------------------------- few long rows
// Rows are cut into C chunks; CTA (row, c) filters chunk c against the row's
// T0 (every CTA of the row derives the same T0 from the same sample) into its
// own slot of `slot` candidates, and writes its candidate and visible counts
// (slot + 1 = the slot overflowed).  Nothing is accumulated across CTAs, so
// the workspace needs no clearing.  The final kernel (one CTA per row) joins
// the row's slots and selects.
struct SplitArgs {
    const float *scores;
    const int32_t *n_rows;
    int Q, N_cap, top_k;
    int C, chunk, slot;
    uint2 *cand;              // [R][C][slot]
    uint32_t *cnt, *vis;      // [R][C]
    int32_t *idx, *count;
    uint32_t *status;
};

__global__ void __launch_bounds__(kSplitThreads) topk_split_kernel(const __grid_constant__ SplitArgs a) {
    pdl_launch_dependents();
    const long long row = blockIdx.x / a.C;
    const int c = static_cast<int>(blockIdx.x - row * a.C);
    const int u = static_cast<int>(row / a.Q);
    const int n_given = a.n_rows[u];                    // no kernel of this library writes n_rows
    const int n = clamp_rows(n_given, a.N_cap);
    pdl_wait();
    __shared__ SelSmem S;
    __shared__ uint2 queue[kTopkSplitSlot];
    if (c == 0 && threadIdx.x == 0 && row % a.Q == 0 && n != n_given)
        report(a.status, DS4A_DEV_BOUNDS);
    const float *s = a.scores + row * a.N_cap;
    const uint32_t k = static_cast<uint32_t>(a.top_k);
    const int start = c * a.chunk;
    const int end = min(start + a.chunk, n);
    // chunk is a multiple of 4: float4 groups stay inside
    const bool vec4 = (a.N_cap & 3) == 0 && (reinterpret_cast<uintptr_t>(a.scores) & 15) == 0;
    // The first batch of the chunk's loads goes out before the sample's.
    constexpr int B = 8;
    const int g_beg = start / 4, g_end = (end + 3) / 4;
    float4 v[B];
    auto load = [&](int g0) {
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int g = g0 + j * kSplitThreads + static_cast<int>(threadIdx.x);
            v[j] = g < g_end ? __ldg(reinterpret_cast<const float4 *>(s) + g) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    if (vec4 && start < end) load(g_beg);
    const uint32_t T0 = sample_threshold<kSplitThreads, kSampleSplit>(s, n, k, kSplitCache, S);
    if (threadIdx.x == 0) S.cnt[3] = 0u;
    __syncthreads();
    uint32_t my_vis = 0;
    const uint32_t cap = static_cast<uint32_t>(a.slot);
    if (vec4) {
        for (int g0 = g_beg; g0 < g_end; g0 += B * kSplitThreads) {    // block-uniform
            if (g0 != g_beg) load(g0);
#pragma unroll
            for (int j = 0; j < B; ++j) {
                const int i = 4 * (g0 + j * kSplitThreads + static_cast<int>(threadIdx.x));
                const float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                uint32_t key[4], bal[4], tot = 0;
                bool take[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const bool vis = i + q < end && score_visible(f[q]);
                    key[q] = float_key(f[q]);
                    my_vis += vis ? 1u : 0u;
                    take[q] = vis && key[q] >= T0;
                    bal[q] = __ballot_sync(0xffffffffu, take[q]);
                    tot += __popc(bal[q]);
                }
                if (tot) {                                    // warp-uniform: one shared atomic per float4
                    const int lane = threadIdx.x & 31;
                    uint32_t pos = 0;
                    if (lane == 0) pos = atomicAdd(&S.cnt[3], tot);
                    pos = __shfl_sync(0xffffffffu, pos, 0);
                    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t p = pos + __popc(bal[q] & lt);
                        if (take[q] && p < cap) queue[p] = make_uint2(key[q], static_cast<uint32_t>(i + q));
                        pos += __popc(bal[q]);
                    }
                }
            }
        }
    } else {
        for (int b = start; b < end; b += kSplitThreads) {              // block-uniform
            const int i = b + static_cast<int>(threadIdx.x);
            const float f = i < end ? s[i] : 0.f;
            const bool vis = i < end && score_visible(f);
            const uint32_t key = float_key(f);
            my_vis += vis ? 1u : 0u;
            warp_append<uint2>(queue, &S.cnt[3], cap, vis && key >= T0, make_uint2(key, static_cast<uint32_t>(i)));
        }
    }
    {
        uint32_t t = my_vis;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        if ((threadIdx.x & 31) == 0) S.warp_sums[threadIdx.x >> 5] = t;
    }
    __syncthreads();
    const uint32_t nq = S.cnt[3];
    const uint32_t nw = nq < cap ? nq : cap;
    uint2 *dst = a.cand + (row * a.C + c) * static_cast<long long>(a.slot);
    for (uint32_t i = threadIdx.x; i < nw; i += kSplitThreads) dst[i] = queue[i];
    if (threadIdx.x == 0) {
        uint32_t tot = 0;
        for (int w = 0; w < kSplitThreads / 32; ++w) tot += S.warp_sums[w];
        a.cnt[row * a.C + c] = nq > cap ? cap + 1 : nq;
        a.vis[row * a.C + c] = tot;
    }
}

__global__ void __launch_bounds__(kSplitFinalThreads) topk_split_final_kernel(const __grid_constant__ SplitArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(16) uint8_t split_smem[];
    uint2 *cache = reinterpret_cast<uint2 *>(split_smem);                                // [kSplitCache]
    int32_t *sel = reinterpret_cast<int32_t *>(split_smem + kSplitCache * 8);            // [kMaxTopK]
    uint32_t *list = reinterpret_cast<uint32_t *>(split_smem + kSplitCache * 8 + kMaxTopK * 4);   // [kFastList]
    SelSmem &S = *reinterpret_cast<SelSmem *>(split_smem + kSplitCache * 8 + kMaxTopK * 4 + kFastList * 4);
    __shared__ uint32_t base[kTopkSplitMaxCtas + 1];
    sel_reset(S);
    const long long row = blockIdx.x;
    const int u = static_cast<int>(row / a.Q);
    const int n = row_len(a.n_rows, u, a.N_cap);
    const uint32_t k = static_cast<uint32_t>(a.top_k);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // Exclusive prefix of the C slot counts (C <= kTopkSplitMaxCtas <= 8 warps x 32).
    uint32_t my_c = 0, my_v = 0;
    if (static_cast<int>(threadIdx.x) < a.C) {
        my_c = a.cnt[row * a.C + threadIdx.x];
        my_v = a.vis[row * a.C + threadIdx.x];
    }
    const bool overflow = __syncthreads_or(my_c > static_cast<uint32_t>(a.slot));
    uint32_t incl = my_c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    uint32_t vsum = my_v;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) vsum += __shfl_xor_sync(0xffffffffu, vsum, off);
    if (lane == 31) S.warp_sums[warp] = incl;
    __syncthreads();
    uint32_t before = 0, nc = 0;
    for (int w = 0; w < kSplitFinalThreads / 32; ++w) {
        const uint32_t t = S.warp_sums[w];
        if (w < warp) before += t;
        nc += t;
    }
    if (static_cast<int>(threadIdx.x) < a.C) base[threadIdx.x] = before + incl - my_c;
    if (threadIdx.x == 0) base[a.C] = nc;
    __syncthreads();
    if (lane == 0) S.warp_sums[warp] = vsum;
    __syncthreads();
    uint32_t total = 0;
    for (int w = 0; w < kSplitFinalThreads / 32; ++w) total += S.warp_sums[w];
    __syncthreads();
    int32_t *out = a.idx + row * a.top_k;
    const bool decides = !overflow && nc <= static_cast<uint32_t>(kSplitCache) &&
                         (total <= k ? nc == total : nc >= k);
    if (decides) {
        // Join the slots: candidate g sits in the last slot c with base[c] <= g
        // (a binary search), so that all the copies are in flight at once.
        uint32_t kmn = 0xffffffffu, kmx = 0u;
        constexpr int J = 4;                              // candidates per thread in flight
        for (uint32_t g0 = 0; g0 < nc; g0 += J * kSplitFinalThreads) {
            uint2 e[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const uint32_t g = g0 + j * kSplitFinalThreads + threadIdx.x;
                e[j] = make_uint2(0u, 0u);
                if (g < nc) {
                    int lo = 0, hi = a.C;                 // base[lo] <= g < base[hi]
                    while (hi - lo > 1) {
                        const int mid = (lo + hi) >> 1;
                        if (base[mid] <= g) lo = mid; else hi = mid;
                    }
                    e[j] = a.cand[(row * a.C + lo) * static_cast<long long>(a.slot) + (g - base[lo])];
                }
            }
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const uint32_t g = g0 + j * kSplitFinalThreads + threadIdx.x;
                if (g < nc) {
                    cache[g] = e[j];
                    kmn = min(kmn, e[j].x);
                    kmx = max(kmx, e[j].x);
                }
            }
        }
        warp_fold_minmax(kmn, kmx, S);
        __syncthreads();
        select_from_list<kSplitFinalThreads>(cache, nc, total, k, sel, list, S, reinterpret_cast<uint32_t *>(cache),
                                             2 * kSplitCache, n, out, a.count + row);
    } else {
        select_exact_row<kSplitFinalThreads>(a.scores + row * a.N_cap, n, k, S, out, a.count + row);
    }
}

// ---------------------------------------------------------------- few rows: one cluster per row
// For up to kClusterMaxRows rows of more than kClusterMinRow scores: a
// thread-block cluster of kClusterRowCtas (8) CTAs per row, 16 for batches of
// up to kClusterWideRows rows.  CTA q filters chunk q
// of the row against the row's sampled threshold T0 (every CTA derives the
// same T0 from the same sample) into a candidate list in its own shared
// memory.  The CTAs then exchange what the exact selection needs through
// distributed shared memory, each CTA storing its part into every CTA of the
// cluster, so that every CTA reads only its own shared memory and takes the
// same decisions:
//   1. per CTA: candidate count, visible count, smallest and largest key;
//   2. per CTA: 32-bucket histogram of its candidates over the row's key range;
//   3. per CTA: the keys of the bucket holding the k-th key, in CTA order.
// Every CTA then knows the k-th key T, how many keys equal to T the selection
// takes and, for every CTA, how many rows it contributes: CTA q writes its
// rows above T and its share of the ties (lowest rows first: the chunks are in
// row order) in ascending order at its offset.  A row the lists cannot decide
// (a sample that missed, heavy ties) is selected by CTA 0 alone from the
// row's scores.  No global scratch; three cluster barriers.
constexpr int kClusterRowCtas = 8;        // CTAs per row (16 for batches of up to kClusterWideRows rows)
constexpr int kClusterThreads = 512;
constexpr int kClusterCap = 4096;          // candidates per CTA
constexpr int kClusterMaxRows = 16;       // more rows: one CTA per row is as fast
constexpr int kClusterMinRow = 4096;       // rows up to this long: one CTA per row (every row a candidate)
constexpr int kClusterAllBelow = 8192;     // rows up to this long need no sampled threshold

constexpr int kRingPiece = 8192;           // scores per bulk copy (32 KB)
constexpr int kRingStages = 4;             // copies in flight: the whole chunk of a row of up to 262,144 scores
// Up to this many rows the chunks go through the bulk-copy ring; more rows
// (more clusters of 182 KB CTAs to place at once) load through registers:
// 16 x 65,536 scores, step 78.9 vs 88.5 us; 8 x 16,384 35.7 vs 38.4 us and
// 4 x 262,144 75.0 vs 76.8 us the other way.
constexpr int kClusterRingRows = 8;
// Up to this many rows, sixteen CTAs per row (a non-portable cluster size):
// half the chunk per CTA, which the bulk copies bring in twice as fast
// (4 x 262,144 step 75.3 -> 73.4 us, 2 x 524,288 80.2 -> 74.3 us,
// 1 x 131,072 39.5 -> 37.8 us; without the ring sixteen were slower).
constexpr int kClusterWideRows = 4;

template <bool RING, int C = kClusterRowCtas>
struct __align__(16) ClusterSmem {
    float ring[RING ? kRingStages : 1][RING ? kRingPiece : 4];   // the CTA's chunk of scores, 32 KB at a time
    uint2 cand[kClusterCap];
    int32_t sel[kMaxTopK];                 // read as int4
    int32_t tie[kFastList];
    uint32_t list[kFastList];              // the crossing bucket's keys of every CTA, CTA-ordered; read as uint4
    uint32_t stat[C][4];                   // per CTA: candidates, visible rows, smallest key, largest key
    uint32_t hist[C][32];                  // per CTA: bucket counts
    uint32_t seg[C][2];                    // per CTA: crossing-bucket rows above T, rows equal to T
    uint32_t warp_cnt[kClusterThreads / 32][32];
    SelSmem S;
    uint64_t full[kRingStages];            // ring stage landed
    int abort;
};
using ClusterSmemWide = ClusterSmem<true, 16>;
static_assert(offsetof(ClusterSmem<true>, ring) % 16 == 0 && offsetof(ClusterSmem<true>, sel) % 16 == 0 &&
                  offsetof(ClusterSmem<true>, list) % 16 == 0 && offsetof(ClusterSmem<true>, S) % 16 == 0 &&
                  offsetof(ClusterSmem<true>, full) % 8 == 0 && offsetof(ClusterSmem<false>, sel) % 16 == 0 &&
                  offsetof(ClusterSmem<false>, list) % 16 == 0 && offsetof(ClusterSmem<false>, S) % 16 == 0 &&
                  offsetof(ClusterSmemWide, S) % 16 == 0 && offsetof(ClusterSmemWide, full) % 8 == 0,
              "bulk copies, vector loads and mbarriers need their alignment");

// Each of sel[0 .. m) (distinct rows) to out[base + its rank among them].
DS4A_DEV void rank_write(const int32_t *sel, uint32_t m, int32_t *out) {
    const int4 *s4 = reinterpret_cast<const int4 *>(sel);
    const int m4 = static_cast<int>(m) >> 2;
    for (uint32_t i = threadIdx.x; i < m; i += blockDim.x) {
        const int32_t e = sel[i];
        int r = 0;
        for (int j = 0; j < m4; ++j) {
            const int4 v = s4[j];
            r += (v.x < e) + (v.y < e) + (v.z < e) + (v.w < e);
        }
        for (int j = 4 * m4; j < static_cast<int>(m); ++j) r += sel[j] < e;
        out[r] = e;
    }
}

template <bool RING, int CL>
__global__ void __launch_bounds__(kClusterThreads) topk_cluster_kernel(const __grid_constant__ TopkArgs a, int chunk) {
    pdl_launch_dependents();
    extern __shared__ __align__(16) uint8_t cl_smem[];
    ClusterSmem<RING, CL> &M = *reinterpret_cast<ClusterSmem<RING, CL> *>(cl_smem);
    SelSmem &S = M.S;
    constexpr int C = CL, NT = kClusterThreads, NW = NT / 32;
    static_assert(C <= NW, "a warp per CTA of the cluster counts its crossing-bucket segment");
    const uint32_t q = cluster_rank();
    const long long row = blockIdx.x / C;
    const int u = static_cast<int>(row / a.Q);
    const int n_given = a.n_rows[u];                    // no kernel of this library writes n_rows
    const int n = clamp_rows(n_given, a.N_cap);
    pdl_wait();
    if (q == 0 && threadIdx.x == 0 && row % a.Q == 0 && n != n_given)
        report(a.status, DS4A_DEV_BOUNDS);
    const float *s = a.scores + row * a.N_cap;
    const uint32_t k = static_cast<uint32_t>(a.top_k);
    int32_t *out = a.idx + row * a.top_k;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int start = static_cast<int>(q) * chunk;          // chunk is a multiple of 4
    const int end = min(start + chunk, n);
    const bool vec4 = (a.N_cap & 3) == 0 && (reinterpret_cast<uintptr_t>(a.scores) & 15) == 0;
    // With the ring (RING: batches of up to kClusterRingRows rows) the chunk
    // goes into shared memory by bulk copies, 32 KB each, up to four in flight
    // from the start (an SM keeps far more bytes in flight this way than with
    // its threads' loads); the sample's loads run beside them.  The
    // last copy is rounded up to 16 bytes: still inside the row's N_cap
    // entries (N_cap is a multiple of 4 here), the excess is never looked at.
    const int len4 = end > start ? ((end - start + 3) & ~3) : 0;
    const int n_pieces = (len4 + kRingPiece - 1) / kRingPiece;
    auto issue = [&](int p) {
        const int off = p * kRingPiece;
        const uint32_t bytes = static_cast<uint32_t>(min(kRingPiece, len4 - off)) * 4u;
        uint64_t *bar = &M.full[p % kRingStages];
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(M.ring[p % kRingStages], s + start + off, bytes, bar);
    };
    if constexpr (RING) {
        if (vec4 && threadIdx.x == 0) {
            for (int i = 0; i < kRingStages; ++i) mbar_init(&M.full[i], 1);
            M.abort = 0;
            mbar_fence_init();
            for (int p = 0; p < min(kRingStages, n_pieces); ++p) issue(p);
        }
    }
    // Without the ring: eight float4 loads per thread in flight, the first
    // batch during the sample.
    constexpr int B = 8;
    const int g_beg = start / 4, g_end = end > start ? (end + 3) / 4 : g_beg;
    float4 v[B];
    auto load = [&](int g0) {
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int g = g0 + j * NT + static_cast<int>(threadIdx.x);
            v[j] = g < g_end ? __ldg(reinterpret_cast<const float4 *>(s) + g) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    if (!RING && vec4) load(g_beg);
    const uint32_t T0 = sample_threshold<NT, kSampleSplit>(s, n, k, kClusterAllBelow, S);
    sel_reset(S);
    __syncthreads();
    // ---- the chunk against T0: candidates, visible count, key range.  Plain
    // float compares (f >= the float of T0 is key(f) >= T0 for a visible f;
    // NaN and -inf fail both tests); keys only for the rare candidates.
    uint32_t my_vis = 0, kmn = 0xffffffffu, kmx = 0u;
    const bool take_all = T0 == 0u;
    const float T0f = key_float(T0);
    const float kNegInf = -__int_as_float(0x7f800000);
    // One float4 of scores (rows i .. i+3); every lane of the warp calls it.
    auto consume = [&](const float4 v, int i) {
        const float f[4] = {v.x, v.y, v.z, v.w};
        bool take[4];
        bool any = false;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const bool vis = i + c < end && f[c] > kNegInf;
            my_vis += vis ? 1u : 0u;
            take[c] = vis && (take_all || f[c] >= T0f);
            any |= take[c];
        }
        if (!__any_sync(0xffffffffu, any)) return;
        uint32_t key[4], bal[4], tot = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            key[c] = float_key(f[c]);
            kmn = take[c] ? min(kmn, key[c]) : kmn;
            kmx = take[c] ? max(kmx, key[c]) : kmx;
            bal[c] = __ballot_sync(0xffffffffu, take[c]);
            tot += __popc(bal[c]);
        }
        uint32_t pos = 0;                                     // one shared atomic per warp and float4
        if (lane == 0) pos = atomicAdd(&S.cnt[3], tot);
        pos = __shfl_sync(0xffffffffu, pos, 0);
        const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t p = pos + __popc(bal[c] & lt);
            if (take[c] && p < static_cast<uint32_t>(kClusterCap)) M.cand[p] = make_uint2(key[c], static_cast<uint32_t>(i + c));
            pos += __popc(bal[c]);
        }
    };
    if (RING && vec4) {
        if constexpr (RING) {
            bool ring_ok = true;
            for (int pc = 0; pc < n_pieces; ++pc) {           // block-uniform
                const int st = pc % kRingStages;
                // a copy that never lands is reported; the pass goes on (on what
                // the buffer holds) so that every CTA still meets the cluster barriers
                if (ring_ok && !mbar_wait(&M.full[st], static_cast<uint32_t>(pc / kRingStages) & 1u, &M.abort)) {
                    ring_ok = false;
                    *reinterpret_cast<volatile int *>(&M.abort) = 1;     // the others stop waiting too
                    if (threadIdx.x == 0) report(a.status, DS4A_DEV_TIMEOUT);
                }
                const int off = pc * kRingPiece;
                const int cnt4 = min(kRingPiece, len4 - off) / 4;
                const float4 *r4 = reinterpret_cast<const float4 *>(M.ring[st]);
#pragma unroll 2
                for (int g0 = 0; g0 < cnt4; g0 += NT) {      // block-uniform
                    const int g = g0 + static_cast<int>(threadIdx.x);
                    consume(g < cnt4 ? r4[g] : make_float4(0.f, 0.f, 0.f, 0.f), start + off + 4 * g);
                }
                __syncthreads();                              // stage st read by every thread
                if (threadIdx.x == 0 && pc + kRingStages < n_pieces) issue(pc + kRingStages);
            }
        }
    } else if (vec4) {
        for (int g0 = g_beg; g0 < g_end; g0 += B * NT) {     // block-uniform
            if (g0 != g_beg) load(g0);
#pragma unroll
            for (int j = 0; j < B; ++j) consume(v[j], 4 * (g0 + j * NT + static_cast<int>(threadIdx.x)));
        }
    } else {
        for (int b = start; b < end; b += NT) {              // block-uniform
            const int i = b + static_cast<int>(threadIdx.x);
            const float f = i < end ? s[i] : 0.f;
            const bool vis = i < end && score_visible(f);
            const uint32_t key = float_key(f);
            my_vis += vis ? 1u : 0u;
            const bool take = vis && key >= T0;
            kmn = take ? min(kmn, key) : kmn;
            kmx = take ? max(kmx, key) : kmx;
            warp_append<uint2>(M.cand, &S.cnt[3], kClusterCap, take, make_uint2(key, static_cast<uint32_t>(i)));
        }
    }
    warp_fold_minmax(kmn, kmx, S);
    {
        const uint32_t t = __reduce_add_sync(0xffffffffu, my_vis);
        if (lane == 0) S.warp_sums[warp] = t;
    }
    __syncthreads();
    const uint32_t nc_q = S.cnt[3];
    // ---- 1. counts and key range to every CTA
    if (threadIdx.x < C) {
        uint32_t vis_q = 0;
        for (int w = 0; w < NW; ++w) vis_q += S.warp_sums[w];
        const uint32_t b = smem_u32(&M.stat[q][0]);
        st_cluster_u32(b, threadIdx.x, nc_q);
        st_cluster_u32(b + 4, threadIdx.x, vis_q);
        st_cluster_u32(b + 8, threadIdx.x, S.mm[0]);
        st_cluster_u32(b + 12, threadIdx.x, S.mm[1]);
    }
    cluster_sync_all();                                       // (1 of 3)
    uint32_t nc = 0, total = 0, kmin = 0xffffffffu, kmax = 0u, below_q = 0;
    bool overflow = false;
#pragma unroll
    for (int j = 0; j < C; ++j) {
        const uint32_t cj = M.stat[j][0];
        overflow |= cj > static_cast<uint32_t>(kClusterCap);
        if (j < static_cast<int>(q)) below_q += cj;
        nc += cj;
        total += M.stat[j][1];
        kmin = min(kmin, M.stat[j][2]);
        kmax = max(kmax, M.stat[j][3]);
    }
    const bool decides = !overflow && (total <= k ? nc == total : nc >= k);
    if (!decides) {                                           // every CTA of the cluster agrees
        cluster_sync_all();
        cluster_sync_all();
        if (q == 0) select_exact_row<NT>(s, n, k, S, out, a.count + row);
        return;
    }
    if (total <= k) {
        // every visible row is a candidate: CTA q's rows, ascending, after those of CTAs 0 .. q-1
        for (uint32_t i = threadIdx.x; i < nc_q; i += NT) M.sel[i] = static_cast<int32_t>(M.cand[i].y);
        __syncthreads();
        rank_write(M.sel, nc_q, out + below_q);
        if (q == 0) {
            for (uint32_t i = total + threadIdx.x; i < k; i += NT) out[i] = -1;
            if (threadIdx.x == 0) a.count[row] = static_cast<int32_t>(total);
        }
        cluster_sync_all();
        cluster_sync_all();
        return;
    }
    // ---- 2. 32-bucket histogram of the candidates over [kmin, kmax], to every CTA
    const uint32_t range = kmax - kmin;
    const int sh = range > 31u ? 27 - __clz(range) : 0;      // (range >> sh) < 32
    {
        uint32_t mine = 0;
        for (uint32_t i0 = warp * 32; i0 < nc_q; i0 += NT) {  // warp-uniform trip count
            const uint32_t i = i0 + lane;
            const bool ok = i < nc_q;
            const uint32_t bk = ok ? (M.cand[i].x - kmin) >> sh : 0u;
            uint32_t match = __ballot_sync(0xffffffffu, ok);
#pragma unroll
            for (int bit = 0; bit < 5; ++bit) {
                const uint32_t mb = __ballot_sync(0xffffffffu, (bk >> bit) & 1u);
                match &= ((lane >> bit) & 1) ? mb : ~mb;
            }
            mine += __popc(match);
        }
        M.warp_cnt[warp][lane] = mine;
    }
    __syncthreads();
    if (warp == 0) {
        uint32_t cb = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) cb += M.warp_cnt[w][lane];
        const uint32_t b = smem_u32(&M.hist[q][lane]);
#pragma unroll
        for (int j = 0; j < C; ++j) st_cluster_u32(b, j, cb);
    }
    cluster_sync_all();                                       // (2 of 3)
    if (warp == 0) {
        uint32_t tb = 0;
#pragma unroll
        for (int j = 0; j < C; ++j) tb += M.hist[j][lane];
        uint32_t suf = tb;                                    // keys in buckets >= lane
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t t = __shfl_down_sync(0xffffffffu, suf, off);
            if (lane + off < 32) suf += t;
        }
        const uint32_t hit = __ballot_sync(0xffffffffu, suf >= k);
        const int bb = hit ? 31 - __clz(hit) : 0;             // hit != 0: nc >= k
        const uint32_t above = __shfl_sync(0xffffffffu, suf - tb, bb);
        if (lane == 0) {
            S.bc[0] = static_cast<uint32_t>(bb);
            S.bc[1] = above;
        }
    }
    __syncthreads();
    const uint32_t b0 = S.bc[0];
    const uint32_t need = k - S.bc[1];
    uint32_t L = 0, off_q = 0;
#pragma unroll
    for (int j = 0; j < C; ++j) {
        if (j < static_cast<int>(q)) off_q += M.hist[j][b0];
        L += M.hist[j][b0];
    }
    if (L > static_cast<uint32_t>(kFastList)) {               // every CTA agrees
        cluster_sync_all();
        if (q == 0) select_exact_row<NT>(s, n, k, S, out, a.count + row);
        return;
    }
    // ---- 3. the crossing bucket's keys, CTA q's at [off_q, off_q + hist[q][b0]), to every CTA
    if (sh > 0) {
        for (uint32_t i0 = 0; i0 < nc_q; i0 += NT) {          // block-uniform trip count
            const uint32_t i = i0 + threadIdx.x;
            const uint32_t key = i < nc_q ? M.cand[i].x : 0u;
            const bool in = i < nc_q && ((key - kmin) >> sh) == b0;
            const uint32_t bal = __ballot_sync(0xffffffffu, in);
            if (bal == 0u) continue;
            uint32_t p = 0;
            if (lane == 0) p = atomicAdd(&S.cnt[2], static_cast<uint32_t>(__popc(bal)));
            p = __shfl_sync(0xffffffffu, p, 0) + __popc(bal & ((1u << lane) - 1u));
            if (in) {
                const uint32_t b = smem_u32(&M.list[off_q + p]);
#pragma unroll
                for (int j = 0; j < C; ++j) st_cluster_u32(b, j, key);
            }
        }
    }
    cluster_sync_all();                                       // (3 of 3): no shared memory of another CTA is touched after this
    // ---- T, how many ties the selection takes, and every CTA's rows
    uint32_t T, need_eq;
    if (sh == 0) {                                            // one key per bucket
        T = kmin + b0;
        need_eq = need;
    } else if (L > 256u) {                                    // narrow the bucket 8 bits per round (one warp)
        if (warp == 0) warp_narrow(M.list, L, kmin + (b0 << sh), sh, need, S);
        __syncthreads();
        T = S.bc[2];
        need_eq = S.bc[3];
    } else {
        for (uint32_t i = threadIdx.x; i < L; i += NT) {
            const uint32_t vi = M.list[i];
            const uint4 *l4 = reinterpret_cast<const uint4 *>(M.list);
            uint32_t gt = 0, ge = 0;
            for (uint32_t j = 0; j < L / 4; ++j) {
                const uint4 o = l4[j];
                gt += (o.x > vi) + (o.y > vi) + (o.z > vi) + (o.w > vi);
                ge += (o.x >= vi) + (o.y >= vi) + (o.z >= vi) + (o.w >= vi);
            }
            for (uint32_t j = L & ~3u; j < L; ++j) {
                gt += M.list[j] > vi;
                ge += M.list[j] >= vi;
            }
            if (gt < need && ge >= need) {                    // every such thread holds the same key
                S.bc[2] = vi;
                S.bc[3] = need - gt;
            }
        }
        __syncthreads();
        T = S.bc[2];
        need_eq = S.bc[3];
    }
    // each CTA's rows above T (its buckets above the crossing one and its
    // crossing-bucket keys above T) and equal to T (warp j: CTA j)
    if (warp < C) {
        uint32_t o = 0;
        for (int j = 0; j < warp; ++j) o += M.hist[j][b0];
        const uint32_t cnt = M.hist[warp][b0];
        uint32_t g = lane > static_cast<int>(b0) ? M.hist[warp][lane] : 0u, e = 0;
        for (uint32_t i = lane; i < cnt; i += 32) {
            const uint32_t key = sh == 0 ? T : M.list[o + i];
            g += key > T;
            e += key == T;
        }
        g = __reduce_add_sync(0xffffffffu, g);
        e = __reduce_add_sync(0xffffffffu, e);
        if (lane == 0) {
            M.seg[warp][0] = g;
            M.seg[warp][1] = e;
        }
    }
    __syncthreads();
    uint32_t out_q = 0, ties_before = 0, gt_q = 0, eq_q = 0, taken_q = 0;
#pragma unroll
    for (int j = 0; j < C; ++j) {
        const uint32_t gj = M.seg[j][0];
        const uint32_t ej = M.seg[j][1];
        const uint32_t left = need_eq > ties_before ? need_eq - ties_before : 0u;
        const uint32_t tj = min(ej, left);
        if (j < static_cast<int>(q)) out_q += gj + tj;
        if (j == static_cast<int>(q)) {
            gt_q = gj;
            eq_q = ej;
            taken_q = tj;
        }
        ties_before += ej;
    }
    // ---- CTA q's rows: above T, and its share of the ties (its lowest rows)
    for (uint32_t i0 = 0; i0 < nc_q; i0 += NT) {              // block-uniform trip count
        const uint32_t i = i0 + threadIdx.x;
        const uint2 e = i < nc_q ? M.cand[i] : make_uint2(0u, 0u);
        warp_append<int32_t>(M.sel, &S.cnt[0], k, i < nc_q && e.x > T, static_cast<int32_t>(e.y));
        warp_append<int32_t>(M.tie, &S.cnt[1], kFastList, i < nc_q && e.x == T, static_cast<int32_t>(e.y));
    }
    __syncthreads();
    if (taken_q == eq_q) {
        for (uint32_t i = threadIdx.x; i < eq_q; i += NT) M.sel[gt_q + i] = M.tie[i];
    } else {
        int p2 = 1;
        while (p2 < static_cast<int>(eq_q)) p2 <<= 1;
        for (int i = static_cast<int>(eq_q) + threadIdx.x; i < p2; i += NT) M.tie[i] = 0x7fffffff;
        __syncthreads();
        block_bitonic_sort_asc(M.tie, p2);
        for (uint32_t i = threadIdx.x; i < taken_q; i += NT) M.sel[gt_q + i] = M.tie[i];
    }
    __syncthreads();
    rank_write(M.sel, gt_q + taken_q, out + out_q);
    if (q == 0 && threadIdx.x == 0) a.count[row] = static_cast<int32_t>(k);
}

// Split plan for R rows of N_cap scores: at most kTopkSplitMaxCtas CTAs in all
// (one wave), chunks of at least 1,024 scores (a multiple of 4), a slot of at
// most kTopkSplitSlot candidates per CTA (about 3k / C are expected; a slot
// also holds every candidate of a row whose top rows crowd into one chunk).
struct SplitPlan {
    int C, chunk, slot;
};
SplitPlan split_plan(long long R, int N_cap) {
    SplitPlan p;
    long long cmax = kTopkSplitMaxCtas / (R > 0 ? R : 1);
    if (cmax < 1) cmax = 1;
    long long c = (N_cap + 1023) / 1024;
    if (c > cmax) c = cmax;
    long long chunk = (N_cap + c - 1) / c;
    chunk = (chunk + 3) & ~3LL;
    p.chunk = static_cast<int>(chunk);
    p.C = static_cast<int>((N_cap + chunk - 1) / chunk);
    p.slot = p.chunk < kTopkSplitSlot ? p.chunk : kTopkSplitSlot;
    return p;
}
bool split_rows(long long R, int N_cap) { return 2 * R <= kTopkSplitMaxCtas && N_cap > kTopkSplitMinRow; }

// ---------------------------------------------------------------- candidates
// Exact top-k of one (u,q) row from the fused indexer's candidate list
// (order-preserving key, row): every row whose key is at or above the row's
// k-th key is in the list (the indexer's threshold never passed it), so the
// selection over the list is the selection over the row.  One CTA per row;
// the list is cached in shared memory when it fits, else used in place.
constexpr int kCandThreads = 512;
// 6,144 cached candidates (48 KB) let three CTAs share an SM; 12,288 (96 KB), two.
constexpr int kCandCacheSmall = 6144;
constexpr int kCandCacheLarge = 12288;

template <int kCandCache>
__global__ void __launch_bounds__(kCandThreads, kCandCache > 6144 ? 2 : 3)
    topk_cand_kernel(const __grid_constant__ TopkCandArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(16) uint8_t cand_smem[];
    uint2 *cache = reinterpret_cast<uint2 *>(cand_smem);                            // [kCandCache]
    int32_t *sel = reinterpret_cast<int32_t *>(cand_smem + kCandCache * 8);         // [kMaxTopK]
    uint32_t *list = reinterpret_cast<uint32_t *>(cand_smem + kCandCache * 8 + kMaxTopK * 4);   // [kFastList]
    SelSmem &S = *reinterpret_cast<SelSmem *>(cand_smem + kCandCache * 8 + kMaxTopK * 4 + kFastList * 4);
    sel_reset(S);
    __syncthreads();                                  // S.mm set before any warp folds its keys into it
    const long long row = blockIdx.x;
    const uint32_t k = static_cast<uint32_t>(a.top_k);
    uint32_t nc = a.cand_n[row];
    if (nc > static_cast<uint32_t>(a.N_cap)) nc = static_cast<uint32_t>(a.N_cap);
    const uint32_t total = a.vis_n[row];
    uint2 *gc = a.cand + row * a.N_cap;
    const bool cached = nc <= static_cast<uint32_t>(kCandCache);
    uint32_t kmn = 0xffffffffu, kmx = 0u;
    // Four loads per thread in flight per round trip (the list was just written
    // by the scan: L2 latency, not bandwidth, sets the pace).
    constexpr int kBatch = 4;
    for (uint32_t i0 = 0; i0 < nc; i0 += kBatch * kCandThreads) {    // block-uniform trip count
        uint2 e[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const uint32_t i = i0 + j * kCandThreads + threadIdx.x;
            e[j] = i < nc ? gc[i] : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const uint32_t i = i0 + j * kCandThreads + threadIdx.x;
            if (i < nc) {
                if (cached) cache[i] = e[j];
                kmn = min(kmn, e[j].x);
                kmx = max(kmx, e[j].x);
            }
        }
    }
    warp_fold_minmax(kmn, kmx, S);
    __syncthreads();
    select_from_list<kCandThreads>(cached ? cache : gc, nc, total, k, sel, list, S, reinterpret_cast<uint32_t *>(cache),
                                   cached ? 2 * kCandCache : 0, a.N_cap, a.idx + row * a.top_k, a.count + row);
}

}  // namespace

size_t topk_ws_bytes(long long R, int N_cap) {
    if (!split_rows(R, N_cap)) return 0;
    const SplitPlan p = split_plan(R, N_cap);
    const size_t slots = static_cast<size_t>(R) * p.C;
    return slots * p.slot * 8 + slots * 8;
}

cudaError_t launch_topk(const TopkArgs &a, int num_sms, cudaStream_t s) {
    const long long R = static_cast<long long>(a.U) * a.Q;
    if (R <= 0) return cudaSuccess;
    if (R <= kClusterMaxRows && a.N_cap > kClusterMinRow && a.N_cap <= kTopkSplitMinRow) {
        auto go = [&](auto kern, int smem, int cl) -> cudaError_t {
            int chunk = (a.N_cap + cl - 1) / cl;
            chunk = (chunk + 3) & ~3;
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            if (cl > 8) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e != cudaSuccess) return e;
            }
            return launch_k_cluster(kern, dim3(static_cast<unsigned>(R * cl)), dim3(kClusterThreads), smem, cl, s, a,
                                    chunk);
        };
        if (R <= kClusterWideRows)
            return go(topk_cluster_kernel<true, 16>, static_cast<int>(sizeof(ClusterSmemWide)), 16);
        if (R <= kClusterRingRows)
            return go(topk_cluster_kernel<true, 8>, static_cast<int>(sizeof(ClusterSmem<true>)), 8);
        return go(topk_cluster_kernel<false, 8>, static_cast<int>(sizeof(ClusterSmem<false>)), 8);
    }
    if (!split_rows(R, a.N_cap) || R >= num_sms) {
        // One CTA per row, no workspace.
        if (R > 0x7fffffffLL) return cudaErrorInvalidValue;
        auto go = [&](auto kern, int nt, int smem) -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            return launch_k(kern, dim3(static_cast<unsigned>(R)), dim3(nt), smem, s, a.scores, a.n_rows, a.Q, a.N_cap,
                            a.top_k, a.idx, a.count, a.status);
        };
        if (a.top_k <= kRowTinyMaxK && R >= 4LL * num_sms)
            return go(topk_row_kernel<128, 2048, kRowTinyMaxK>, 128, RowShape<128, 2048, kRowTinyMaxK>::kSmem);
        if (a.top_k <= kRowSmallMaxK)
            return go(topk_row_kernel<256, 4096, 1024>, 256, RowShape<256, 4096, 1024>::kSmem);
        return go(topk_row_kernel<512, 8192, kMaxTopK>, 512, RowShape<512, 8192, kMaxTopK>::kSmem);
    }
    const SplitPlan p = split_plan(R, a.N_cap);
    SplitArgs sa;
    sa.scores = a.scores;
    sa.n_rows = a.n_rows;
    sa.Q = a.Q;
    sa.N_cap = a.N_cap;
    sa.top_k = a.top_k;
    sa.C = p.C;
    sa.chunk = p.chunk;
    sa.slot = p.slot;
    uint8_t *w = static_cast<uint8_t *>(a.ws);
    const size_t slots = static_cast<size_t>(R) * p.C;
    sa.cand = reinterpret_cast<uint2 *>(w);
    sa.cnt = reinterpret_cast<uint32_t *>(w + slots * p.slot * 8);
    sa.vis = sa.cnt + slots;
    sa.idx = a.idx;
    sa.count = a.count;
    sa.status = a.status;
    cudaError_t e = launch_k(topk_split_kernel, dim3(static_cast<unsigned>(slots)), dim3(kSplitThreads), 0, s, sa);
    if (e != cudaSuccess) return e;
    const int smem = kSplitCache * 8 + kMaxTopK * 4 + kFastList * 4 + static_cast<int>(sizeof(SelSmem));
    e = cudaFuncSetAttribute(topk_split_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_k(topk_split_final_kernel, dim3(static_cast<unsigned>(R)), dim3(kSplitFinalThreads), smem, s, sa);
}

cudaError_t launch_topk_cand(const TopkCandArgs &a, cudaStream_t s) {
    if (a.R <= 0) return cudaSuccess;
    // top_k above 512 (the Pro shape's 1,024) leaves about twice the
    // candidates: a list of 12,288 pairs, two CTAs per SM, keeps them cached.
    auto go = [&](auto kern, int cache) -> cudaError_t {
        const int smem = cache * 8 + kMaxTopK * 4 + kFastList * 4 + static_cast<int>(sizeof(SelSmem));
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        return launch_k(kern, dim3(a.R), dim3(kCandThreads), smem, s, a);
    };
    if (a.top_k > 512) return go(topk_cand_kernel<kCandCacheLarge>, kCandCacheLarge);
    return go(topk_cand_kernel<kCandCacheSmall>, kCandCacheSmall);
}

}  // namespace ds4a
