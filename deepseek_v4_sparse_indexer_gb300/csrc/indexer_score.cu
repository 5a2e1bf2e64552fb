// Indexer score on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Computes, for every (unit u, query q, compressed row r):
//     scores[u,q,r] = sum_h w[u,q,h] * max(0, sum_d iq[u,q,h,d] * ik[u,r,d])
// The pages name the indexer (64 heads x 128 dims scoring every compressed
// row, "DwarfStar(ds4.c) のアーキテクチャを読む" §2 and §3-3) but print no
// formula; this is the library's specification of it.
//
// Mapping: one UMMA tile is D[128 rows x N] = ik_tile[128 x 128] * iq^T with
// rows on M and (query, head) pairs on N = 64*G (G queries share the rows of a
// tile: G = 1 in decode, 4 in a prefill chunk).  With rows on M, TMEM lane i
// holds all head sums of row i, so the ReLU-weighted head reduction is a
// per-thread loop after one tcgen05.ld, with no cross-thread traffic.
//
// Roles (warp specialised, one CTA per SM, persistent over work items):
//   warp 0      TMA producer: streams 32 KB key tiles through a K-stage ring
//               (L2 evict-first: each key is read once) and the G queries'
//               iq block per work item (L2 evict-last: shared by many CTAs);
//   warp 1      TMEM owner and UMMA issuer (one thread): 8 x (M128,N,K16)
//               per tile into a ring of TMEM accumulators;
//   warps 2..   epilogue: tcgen05.ld of the row's N accumulators, ReLU,
//               weight, sum over heads (packed fp32x2 FMAs, eight partial
//               sums), masked store of one fp32 per (q,row).
// The work is the list of (unit, query group, 128-row tile) triples, tile
// fastest; each CTA takes one contiguous, equal share of it, so the CTAs end
// together and a CTA reloads its iq block only where its share crosses into
// the next (unit, group).
//
// The decode scan is HBM-bound (256 B of keys per row for 16 kFLOP); the
// prefill chunk (G = 4) is tensor-bound.  Every wait is bounded: on timeout
// the kernel flags DS4A_DEV_TIMEOUT, waits (bounded) for its copies and
// UMMAs in flight, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"

namespace ds4a {
namespace {

constexpr int kTileRows = 128;   // UMMA M
// Key tiles per CTA put into L2 before the dependency wait.  Decode (G = 1):
// an eighth of the CTA's share, 4 to 24 (a long scan gains a deeper start;
// behind a partly idle GPU, a short one loses when its prefetch competes with
// the kernel still running: 4 x 262,144 step 71.8 us with 8 tiles, 73.6 with
// 16, 77.6 with 24; the 1,376-unit decode step 3,547 / 3,540 / 3,532 us).  A
// prefill chunk (G = 4), whose key tiles stay in L2 once read: 16 (24 cost
// 13 us on the 2,048-query step).
constexpr int kPrefetchMin = 4, kPrefetchMax = 24, kPrefetchGroups = 16;


template <int G>
struct IdxCfg {
    static constexpr int N = 64 * G;                      // UMMA N
    // Key-tile ring depth: four 32 KB stages.  The decode scan is HBM-bound and
    // best with ~18-20 MB in flight over the whole GPU; five stages on 152 SMs
    // (24 MB) ran 6 % slower (3.54 vs 3.33-3.35 ms on 1,376 x 65,536 rows).
    static constexpr int kStages = 4;
    static constexpr int kBBufs = (G == 1) ? 2 : 1;       // iq block buffers
    static constexpr int kAccBufs = (G == 1) ? 4 : 2;     // TMEM accumulators
    static constexpr int kEpiSplit = (G == 1) ? 1 : 2;    // epilogue warps per TMEM lane quarter
    static constexpr int kEpiWarps = 4 * kEpiSplit;
    static constexpr int kQPerEpiWarp = G / kEpiSplit;    // queries one epilogue thread reduces
    // G = 4 keeps two queries' 64 weights per epilogue thread in registers:
    // warps 0-3 (producer, issuer, two idle) give registers up and the two
    // epilogue warpgroups (warps 4-11) take them (setmaxnreg).
    static constexpr bool kSplitRegs = (G != 1);
    static constexpr int kFirstEpiWarp = kSplitRegs ? 4 : 2;
    static constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
    static constexpr int kLowRegs = 72, kHighRegs = 216;   // per thread after setmaxnreg
    static constexpr int kRegsNeeded = 128 * kLowRegs + 32 * kEpiWarps * kHighRegs;
    static constexpr uint32_t kTmemCols = kAccBufs * N;   // 256 or 512
    static constexpr int kASub = kTileRows * 128;         // one 64-element K half of a key tile
    static constexpr int kABytes = 2 * kASub;             // 32 KB
    static constexpr int kBSub = N * 128;
    static constexpr int kBBytes = 2 * kBSub;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kABytes;
    static constexpr int kWFloatsPerWarp = kQPerEpiWarp * 64;
    static constexpr int kOffW = kOffB + kBBufs * kBBytes;
    // Fused selection: one histogram of score keys per query of the group
    // (key bits 31..20 for G = 1, 31..22 for G = 4) and its threshold key.
    static constexpr int kHistShift = (G == 1) ? 20 : 22;
    static constexpr int kTauEvery = (G == 1) ? 16 : 8;    // tiles between threshold updates (a power of two)
    static constexpr int kCandQueue = (G == 1) ? 256 : 64; // candidates staged per epilogue warp and query
    static constexpr int kHistBins = 1 << (32 - kHistShift);
    static constexpr int kOffHist = kOffW + kEpiWarps * kWFloatsPerWarp * 4;
    static constexpr int kOffTau = kOffHist + G * kHistBins * 4;
    static constexpr int kOffQueue = ((kOffTau + G * 4 + 15) / 16) * 16;   // [kEpiWarps][kQPerEpiWarp][kCandQueue] uint2
    static constexpr int kOffBar = kOffQueue + kEpiWarps * kQPerEpiWarp * kCandQueue * 8;
    static constexpr int kNumBars = 2 * kStages + 2 * kBBufs + 2 * kAccBufs + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + slack to 1024-align the base
    static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation must be a power of two");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// One work item: tiles t0 .. t1-1 of (unit u, query group g).  first is the
// tile the item starts at before clamping to the unit's row count.
struct Item {
    int u, g, t0, t1, first;
};

// This CTA's share [lo, hi) of the U * n_groups * nt_cap tiles.
DS4A_DEV void cta_share(const IndexerArgs &a, long long &lo, long long &hi) {
    lo = a.total_tiles * blockIdx.x / gridDim.x;
    hi = a.total_tiles * (blockIdx.x + 1) / gridDim.x;
}

// The item starting at tile index lin (lin < hi), which runs to the end of its
// (unit, group) or of the share; advances lin past it.  Tiles beyond the
// unit's n_rows are clamped away (t0 >= t1: nothing to do).
DS4A_DEV Item next_item(const IndexerArgs &a, long long &lin, long long hi) {
    Item m;
    const long long per_unit = static_cast<long long>(a.n_groups) * a.nt_cap;
    m.u = static_cast<int>(lin / per_unit);
    const int rem = static_cast<int>(lin - static_cast<long long>(m.u) * per_unit);
    m.g = rem / a.nt_cap;
    m.first = rem - m.g * a.nt_cap;
    const long long left = hi - lin;
    const int end = left < a.nt_cap - m.first ? m.first + static_cast<int>(left) : a.nt_cap;
    lin += end - m.first;
    int nr = a.n_rows[m.u];
    nr = nr < 0 ? 0 : (nr > a.N_cap ? a.N_cap : nr);
    const int nt = (nr + kTileRows - 1) / kTileRows;
    m.t0 = m.first;
    m.t1 = min(end, nt);
    return m;
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
DS4A_DEV bool mbar_wait_drain(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// tcgen05.ld of 32 columns whose wait is tied to the destination registers,
// so no use of them can be scheduled before the load has completed.
DS4A_DEV void tmem_ld32_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
DS4A_DEV void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                   "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                   "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Two fp32 lanes as one 64-bit register pair, for the packed fp32x2 FMA.
DS4A_DEV unsigned long long pack_f2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
DS4A_DEV float2 unpack_f2(unsigned long long v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

// Accumulates sum_h w[h] * max(0, acc[h]) over 32 head sums v (heads
// 32*half .. 32*half + 31 of one query) into four packed fp32x2 partial sums.
// w2 holds the query's 64 weights as 32 (even, odd) pairs in registers, so the
// reduction reads no memory.  The ReLU is per element; the FMAs are packed.
DS4A_DEV void relu_weighted_acc(unsigned long long (&acc)[4], const unsigned long long (&w2)[32], int half,
                                const uint32_t (&v)[32]) {
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        const unsigned long long x =
            pack_f2(fmaxf(__uint_as_float(v[2 * p]), 0.f), fmaxf(__uint_as_float(v[2 * p + 1]), 0.f));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc[p & 3]) : "l"(w2[half * 16 + p]), "l"(x));
    }
}
// The bin b where the number of keys in bins >= b first reaches k; -1 when
// the histogram of NB bins (a multiple of 1024) holds fewer than k keys.  All
// lanes call it.  Lane l sums the NB/32 bins of segment 31 - l (lane 0: the
// top segment), reading them in a rotated order so that the lanes hit
// distinct banks; a prefix sum over the lanes finds the segment where the
// count from the top reaches k, and the warp walks that segment from its top.
template <int NB>
DS4A_DEV int hist_kth_bin(const uint32_t *h, uint32_t k, int lane) {
    constexpr int per = NB / 32;
    const uint32_t *hs = h + (31 - lane) * per;
    uint32_t sum = 0;
#pragma unroll 8
    for (int i = 0; i < per; ++i) sum += hs[(i + lane) & (per - 1)];
    uint32_t cum = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, cum, o);
        if (lane >= o) cum += v;
    }
    const uint32_t hit = __ballot_sync(0xffffffffu, cum >= k);
    if (!hit) return -1;
    const int L = __ffs(hit) - 1;
    uint32_t above = __shfl_sync(0xffffffffu, cum - sum, L);
    const int seg0 = (31 - L) * per;
    for (int top = per - 1; top >= 31; top -= 32) {
        uint32_t c = h[seg0 + top - lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, c, o);
            if (lane >= o) c += v;
        }
        const uint32_t tot = __shfl_sync(0xffffffffu, c, 31);
        if (above + tot >= k) return seg0 + top - (__ffs(__ballot_sync(0xffffffffu, above + c >= k)) - 1);
        above += tot;
    }
    return -1;
}

DS4A_DEV float sum_pairs(const unsigned long long (&acc)[4]) {
    const float2 s0 = unpack_f2(acc[0]), s1 = unpack_f2(acc[1]), s2 = unpack_f2(acc[2]), s3 = unpack_f2(acc[3]);
    return ((s0.x + s0.y) + (s1.x + s1.y)) + ((s2.x + s2.y) + (s3.x + s3.y));
}

// The first key tiles of a CTA's share and their query blocks go into L2
// before the kernel waits for the previous one: behind a partly idle GPU (a
// few-unit attention, a short select) the scan's first tiles then come from
// L2.  Tiles past a unit's n_rows are prefetched too (n_rows is read only
// after the wait).
DS4A_DEV void prefetch_share_head(const IndexerArgs &a, long long lo, long long hi, int G) {
    const long long per_unit = static_cast<long long>(a.n_groups) * a.nt_cap;
    const long long depth = G > 1 ? kPrefetchGroups
                                  : min(static_cast<long long>(kPrefetchMax), max(static_cast<long long>(kPrefetchMin), (hi - lo) / 8));
    const long long end = min(hi, lo + depth);
    int last_qrow = -1;
    for (long long lin = lo; lin < end; ++lin) {
        const int u = static_cast<int>(lin / per_unit);
        const int rem = static_cast<int>(lin - u * per_unit);
        const int g = rem / a.nt_cap, t = rem - g * a.nt_cap;
        const int qrow = (u * a.Q + g * G) * kNIdxHead;
        if (qrow != last_qrow) {
            tma_prefetch_l2_2d(&a.tm_iq, 0, qrow);
            tma_prefetch_l2_2d(&a.tm_iq, 64, qrow);
            last_qrow = qrow;
        }
        tma_prefetch_l2_3d(&a.tm_ik, 0, t * kTileRows, u);
        tma_prefetch_l2_3d(&a.tm_ik, 64, t * kTileRows, u);
    }
}

template <int G>
__global__ void __launch_bounds__(IdxCfg<G>::kThreads, 1)
    indexer_score_kernel(const __grid_constant__ IndexerArgs a) {
    pdl_launch_dependents();
    using C = IdxCfg<G>;
    extern __shared__ uint8_t smem_raw[];
    // Aligned by pointer arithmetic on the __shared__ array (not through an
    // integer), so that the compiler keeps shared-space accesses for it.
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem + C::kOffA;
    uint8_t *sB = smem + C::kOffB;
    float *sW = reinterpret_cast<float *>(smem + C::kOffW);
    uint64_t *a_full = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *a_empty = a_full + C::kStages;
    uint64_t *b_full = a_empty + C::kStages;
    uint64_t *b_empty = b_full + C::kBBufs;
    uint64_t *acc_full = b_empty + C::kBBufs;
    uint64_t *acc_empty = acc_full + C::kAccBufs;
    uint64_t *drain_bar = acc_empty + C::kAccBufs;
    uint64_t *epi_bar = drain_bar + 1;                 // epilogue-warp group sync (fused selection)
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + C::kOffHist);
    volatile uint32_t *tau_sh = reinterpret_cast<volatile uint32_t *>(smem + C::kOffTau);
    uint2 *cqueue = reinterpret_cast<uint2 *>(smem + C::kOffQueue);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
        }
        for (int b = 0; b < C::kBBufs; ++b) {
            mbar_init(&b_full[b], 1);
            mbar_init(&b_empty[b], 1);
        }
        for (int c = 0; c < C::kAccBufs; ++c) {
            mbar_init(&acc_full[c], 1);
            mbar_init(&acc_empty[c], C::kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        mbar_init(epi_bar, C::kEpiWarps);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&a.tm_ik);
        tma_prefetch_desc(&a.tm_iq);
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    long long share_lo, share_hi;
    cta_share(a, share_lo, share_hi);
    if (warp != 0) pdl_wait();                         // the set-up above reads no global memory
    const uint32_t tmem_base = *tmem_slot;

    if (warp < C::kFirstEpiWarp) {
        if constexpr (C::kSplitRegs) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kLowRegs));
    }
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) prefetch_share_head(a, share_lo, share_hi, G);
        pdl_wait();
        if (lane == 0) {
            // Decode (G = 1) reads every key tile once: stream it through L2.  A
            // prefill chunk's query groups all read the same key tiles: keep
            // them in L2 (evict-first keys were re-read from DRAM once the
            // scores written meanwhile had pushed them out).
            const uint64_t pol_stream = G == 1 ? l2_policy_evict_first() : l2_policy_evict_last();
            const uint64_t pol_keep = l2_policy_evict_last();
            int s = 0, bb = 0;
            uint32_t sph = 0, bph = 0;
            bool used_s[C::kStages] = {}, used_b[C::kBBufs] = {};
            uint32_t par_s[C::kStages] = {}, par_b[C::kBBufs] = {};
            bool ok = true;
            for (long long lin = share_lo; ok && lin < share_hi;) {
                const Item m = next_item(a, lin, share_hi);
                if (m.t0 >= m.t1) continue;
                if (!mbar_wait_hint(&b_empty[bb], bph ^ 1, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(&b_full[bb], C::kBBytes);
                const int qrow = (m.u * a.Q + m.g * G) * kNIdxHead;
                uint8_t *dstB = sB + bb * C::kBBytes;
                tma_load_2d(dstB, &a.tm_iq, &b_full[bb], 0, qrow, pol_keep);
                tma_load_2d(dstB + C::kBSub, &a.tm_iq, &b_full[bb], 64, qrow, pol_keep);
                used_b[bb] = true;
                par_b[bb] = bph;
                if (++bb == C::kBBufs) { bb = 0; bph ^= 1; }
                for (int t = m.t0; t < m.t1; ++t) {
                    if (!mbar_wait_hint(&a_empty[s], sph ^ 1, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&a_full[s], C::kABytes);
                    uint8_t *dstA = sA + s * C::kABytes;
                    tma_load_3d(dstA, &a.tm_ik, &a_full[s], 0, t * kTileRows, m.u, pol_stream);
                    tma_load_3d(dstA + C::kASub, &a.tm_ik, &a_full[s], 64, t * kTileRows, m.u, pol_stream);
                    used_s[s] = true;
                    par_s[s] = sph;
                    if (++s == C::kStages) { s = 0; sph ^= 1; }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                report(a.status, DS4A_DEV_TIMEOUT);
                // Let every copy already issued land before the CTA exits.
                for (int i = 0; i < C::kStages; ++i)
                    if (used_s[i]) mbar_wait_drain(&a_full[i], par_s[i]);
                for (int i = 0; i < C::kBBufs; ++i)
                    if (used_b[i]) mbar_wait_drain(&b_full[i], par_b[i]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kTileRows, C::N);
            int s = 0, bb = 0, ab = 0;
            uint32_t sph = 0, bph = 0, aph = 0;
            bool ok = true;
            for (long long lin = share_lo; ok && lin < share_hi;) {
                const Item m = next_item(a, lin, share_hi);
                if (m.t0 >= m.t1) continue;
                if (!mbar_wait_hint(&b_full[bb], bph, abort_flag)) { ok = false; break; }
                const uint32_t b_addr = smem_u32(sB + bb * C::kBBytes);
                for (int t = m.t0; t < m.t1; ++t) {
                    if (!mbar_wait_hint(&acc_empty[ab], aph ^ 1, abort_flag)) { ok = false; break; }
                    if (!mbar_wait_hint(&a_full[s], sph, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + s * C::kABytes);
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(ab * C::N);
#pragma unroll
                    for (int k = 0; k < kIdxDim / 16; ++k) {
                        const uint32_t ka = (k >> 2) * C::kASub + (k & 3) * 32;
                        const uint32_t kb = (k >> 2) * C::kBSub + (k & 3) * 32;
                        umma_bf16(d_tmem, sw128_kmajor_desc(a_addr + ka), sw128_kmajor_desc(b_addr + kb), idesc,
                                  k > 0 ? 1u : 0u);
                    }
                    umma_commit(&a_empty[s]);       // key tile may be overwritten once read
                    umma_commit(&acc_full[ab]);     // accumulator ready for the epilogue
                    if (++s == C::kStages) { s = 0; sph ^= 1; }
                    if (++ab == C::kAccBufs) { ab = 0; aph ^= 1; }
                }
                if (!ok) break;
                umma_commit(&b_empty[bb]);          // iq block free after this item's UMMAs
                if (++bb == C::kBBufs) { bb = 0; bph ^= 1; }
            }
            if (!ok) {
                *abort_flag = 1;
                report(a.status, DS4A_DEV_TIMEOUT);
            }
            // Every UMMA issued has completed once this commit arrives.
            umma_commit(drain_bar);
            mbar_wait_drain(drain_bar, 0);
        }
        __syncwarp();
    } else if (warp >= C::kFirstEpiWarp) {
        // ------------------------------------------------------------ epilogue
        if constexpr (C::kSplitRegs) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kHighRegs));
        const int e = warp - C::kFirstEpiWarp;
        const int quarter = warp & 3;             // TMEM lanes this warp may access
        const int half = e / 4;                   // which queries of the group
        const int row_in_tile = quarter * 32 + lane;
        float *wsm = sW + e * C::kWFloatsPerWarp;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        int ab = 0;
        uint32_t aph = 0, eph = 0;
        bool ok = true;
        // Barrier of the epilogue warps on an mbarrier (a wait that gives up
        // cannot leave the others stuck).
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(epi_bar);
            const bool r = __all_sync(0xffffffffu, mbar_wait_hint(epi_bar, eph, abort_flag));
            eph ^= 1;
            return r;
        };
        for (long long lin = share_lo; ok && lin < share_hi;) {
            const Item m = next_item(a, lin, share_hi);
            const int nr_raw = a.n_rows[m.u];
            // Reported once per unit: by the item holding its first tile.
            if ((nr_raw < 0 || nr_raw > a.N_cap) && e == 0 && lane == 0 && m.first == 0 && m.g == 0)
                report(a.status, DS4A_DEV_BOUNDS);
            if (m.t0 >= m.t1) continue;
            const int nr = nr_raw < 0 ? 0 : (nr_raw > a.N_cap ? a.N_cap : nr_raw);
            const int q0 = m.g * G + half * C::kQPerEpiWarp;
            if (a.fused) {
                // Fused selection: a fresh histogram per query of the group once
                // every epilogue warp is done with the previous item, and the
                // threshold other CTAs may already have raised for these rows.
                if (!(ok = epi_sync())) break;
                for (int i = e * 32 + lane; i < G * C::kHistBins; i += C::kEpiWarps * 32) hist[i] = 0u;
                const int gq = e * 32 + lane;
                if (gq < G) tau_sh[gq] = (m.g * G + gq < a.Q) ? a.tau[static_cast<long long>(m.u) * a.Q + m.g * G + gq] : 0u;
                if (!(ok = epi_sync())) break;
            }
            uint32_t my_vis[C::kQPerEpiWarp], qn[C::kQPerEpiWarp];
#pragma unroll
            for (int j = 0; j < C::kQPerEpiWarp; ++j) my_vis[j] = qn[j] = 0u;
            // Staged candidates of query j go out with one global atomic per batch.
            auto flush = [&](int j) {
                __syncwarp();
                const long long R = static_cast<long long>(m.u) * a.Q + q0 + j;
                uint32_t base = 0;
                if (lane == 0) base = atomicAdd(a.cand_n + R, qn[j]);
                base = __shfl_sync(0xffffffffu, base, 0);
                const uint2 *qq = cqueue + (e * C::kQPerEpiWarp + j) * C::kCandQueue;
                for (uint32_t i = lane; i < qn[j]; i += 32) a.cand[R * a.N_cap + base + i] = qq[i];
                qn[j] = 0;
                __syncwarp();
            };
            __syncwarp();
            for (int i = lane; i < C::kWFloatsPerWarp; i += 32) {
                const int qq = q0 + i / kNIdxHead;
                wsm[i] = (qq < a.Q) ? a.w[(static_cast<long long>(m.u) * a.Q + qq) * kNIdxHead + (i % kNIdxHead)]
                                    : 0.f;
            }
            __syncwarp();
            // The item's weights stay in registers for all of its tiles.
            unsigned long long w2[C::kQPerEpiWarp][32];
#pragma unroll
            for (int j = 0; j < C::kQPerEpiWarp; ++j) {
                const float4 *w4 = reinterpret_cast<const float4 *>(wsm + j * 64);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float4 ww = w4[i];
                    w2[j][2 * i] = pack_f2(ww.x, ww.y);
                    w2[j][2 * i + 1] = pack_f2(ww.z, ww.w);
                }
            }
            int qpos[C::kQPerEpiWarp];
#pragma unroll
            for (int j = 0; j < C::kQPerEpiWarp; ++j)
                qpos[j] = (a.q_pos && q0 + j < a.Q) ? a.q_pos[static_cast<long long>(m.u) * a.Q + q0 + j] : 0;

            // The row's position is loaded one tile ahead: its global-load
            // latency then hides behind a whole tile instead of stalling the
            // store at the end of each tile.
            const int32_t *rp = a.row_pos ? a.row_pos + static_cast<long long>(m.u) * a.N_cap : nullptr;
            int rpos_next = 0;
            if (rp && m.t0 * kTileRows + row_in_tile < nr) rpos_next = __ldg(rp + m.t0 * kTileRows + row_in_tile);
            for (int t = m.t0; t < m.t1; ++t) {
                const int row = t * kTileRows + row_in_tile;
                const int rpos = rpos_next;
                if (rp && t + 1 < m.t1 && row + kTileRows < nr) rpos_next = __ldg(rp + row + kTileRows);
                // Warp-uniform outcome: the tcgen05.ld below is .sync.aligned.
                if (!__all_sync(0xffffffffu, mbar_wait_hint(&acc_full[ab], aph, abort_flag))) { ok = false; break; }
                tc_fence_after();
                float sc[C::kQPerEpiWarp];
#pragma unroll
                for (int j = 0; j < C::kQPerEpiWarp; ++j) {
                    const uint32_t col = static_cast<uint32_t>(ab * C::N + (half * C::kQPerEpiWarp + j) * 64);
                    unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t v[32];
                        tmem_ld32_sync(tmem_base + lane_off + col + hh * 32, v);
                        tmem_wait_ld(v);
                        relu_weighted_acc(acc, w2[j], hh, v);
                    }
                    sc[j] = sum_pairs(acc);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[ab]);
                if (a.fused) {
                    // Keep the row as a candidate when its key reaches the query's
                    // threshold, and count it in the query's histogram.  The
                    // threshold is a bin edge with at least top_k counted keys at
                    // or above it, so it never passes the final k-th key: every
                    // row of the top k (ties included) is kept.  Rows below it
                    // need no count: the bin where the count from the top reaches
                    // top_k never lies below the threshold, and the bins at or
                    // above it hold only candidates.
#pragma unroll
                    for (int j = 0; j < C::kQPerEpiWarp; ++j) {
                        const int qq = q0 + j, slot = half * C::kQPerEpiWarp + j;
                        const bool vis = row < nr && qq < a.Q && !(a.q_pos && rpos > qpos[j]) && score_visible(sc[j]);
                        const uint32_t key = float_key(sc[j]);
                        my_vis[j] += vis ? 1u : 0u;
                        const bool emit = vis && key >= tau_sh[slot];
                        hist_add_warp(hist + slot * C::kHistBins, key >> C::kHistShift, emit);
                        const uint32_t bal = __ballot_sync(0xffffffffu, emit);
                        if (emit)
                            cqueue[(e * C::kQPerEpiWarp + j) * C::kCandQueue + qn[j] + __popc(bal & ((1u << lane) - 1u))] =
                                make_uint2(key, static_cast<uint32_t>(row));
                        qn[j] += __popc(bal);
                        if (qn[j] > C::kCandQueue - 32) flush(j);
                    }
                    // Every few tiles, warp e raises the threshold of query slot e.
                    if (e < G && ((t - m.t0) & (C::kTauEvery - 1)) == C::kTauEvery - 1 && m.g * G + e < a.Q) {
                        const int b = hist_kth_bin<C::kHistBins>(hist + e * C::kHistBins, static_cast<uint32_t>(a.top_k), lane);
                        if (b >= 0 && lane == 0) {
                            const uint32_t tk = static_cast<uint32_t>(b) << C::kHistShift;
                            const uint32_t old = atomicMax(a.tau + static_cast<long long>(m.u) * a.Q + m.g * G + e, tk);
                            tau_sh[e] = tk > old ? tk : old;
                        }
                    }
                } else if (row < nr) {
#pragma unroll
                    for (int j = 0; j < C::kQPerEpiWarp; ++j) {
                        const int qq = q0 + j;
                        if (qq < a.Q) {
                            float out = sc[j];
                            if (a.q_pos && rpos > qpos[j]) out = -__int_as_float(0x7f800000);
                            a.scores[(static_cast<long long>(m.u) * a.Q + qq) * a.N_cap + row] = out;
                        }
                    }
                }
                if (++ab == C::kAccBufs) { ab = 0; aph ^= 1; }
            }
            if (a.fused && ok) {
#pragma unroll
                for (int j = 0; j < C::kQPerEpiWarp; ++j) {
                    if (qn[j]) flush(j);
                    uint32_t v = my_vis[j];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0 && v && q0 + j < a.Q) atomicAdd(a.vis_n + static_cast<long long>(m.u) * a.Q + q0 + j, v);
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) report(a.status, DS4A_DEV_TIMEOUT);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int G>
cudaError_t launch_g(const IndexerArgs &a, cudaStream_t s) {
    using C = IdxCfg<G>;
    cudaError_t e = cudaFuncSetAttribute(indexer_score_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if constexpr (C::kSplitRegs) {
        // setmaxnreg.inc draws on the registers the block was launched with: the
        // split must fit in them, or the raising warps would wait forever.
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, indexer_score_kernel<G>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs * C::kThreads < C::kRegsNeeded) return cudaErrorInvalidConfiguration;
    }
    return launch_k(indexer_score_kernel<G>, dim3(a.grid), dim3(C::kThreads), C::kSmemBytes, s, a);
}

// Zeroes the fused selection's per-row counters.  A kernel rather than a
// memset, so that the scan launched behind it can start early (and put its
// first key tiles into L2) while the stream's previous kernels finish.  It
// waits for them first: the previous select over this workspace reads these
// counters.
__global__ void __launch_bounds__(256) clear_counters_kernel(uint32_t *c, long long n) {
    pdl_launch_dependents();
    pdl_wait();
    for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n; i += static_cast<long long>(gridDim.x) * 256)
        c[i] = 0u;
}

}  // namespace

cudaError_t launch_clear_counters(uint32_t *c, long long n, int num_sms, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const long long blocks = (n + 255) / 256;
    const int grid = static_cast<int>(blocks < 4LL * num_sms ? blocks : 4LL * num_sms);
    return launch_k(clear_counters_kernel, dim3(grid), dim3(256), 0, s, c, n);
}

int indexer_group_size(int Q) { return Q >= 4 ? 4 : 1; }

void indexer_plan(IndexerArgs &a, int num_sms) {
    a.G = indexer_group_size(a.Q);
    a.n_groups = (a.Q + a.G - 1) / a.G;
    a.nt_cap = (a.N_cap + kTileRows - 1) / kTileRows;
    a.total_tiles = static_cast<long long>(a.U) * a.n_groups * a.nt_cap;
    a.grid = static_cast<int>(a.total_tiles < num_sms ? a.total_tiles : num_sms);
}

cudaError_t launch_indexer_score(const IndexerArgs &a, cudaStream_t s) {
    if (a.G == 4) return launch_g<4>(a, s);
    return launch_g<1>(a, s);
}

}  // namespace ds4a
