// Sparse attention over the selected compressed rows and the raw window, on
// the 5th-generation tensor cores ("DwarfStar(ds4.c) のアーキテクチャを読む"
// §3: three tiers; §2: 64 query heads, one KV head whose 512-d rows are both
// key and value; §3-1: the raw window of the last 128 tokens kept rounded to
// f16).
//
// One CTA (persistent, one per SM) walks work items = (unit, split), where a
// unit is one decode query or one query of a prefill chunk.  The unit's row
// list [selected compressed rows..., raw-window rows...] is cut into 128-row
// tiles.  Per tile:
//   gather   warp 0: TMA tile::gather4 loads (4 rows x 64 columns each, 128B
//            swizzle) of the tile's rows into eight 16 KB column blocks;
//            a masked row uses an out-of-range coordinate and lands as zeros;
//   logits   warp 1 (one thread): S^T[128 rows x 64 heads] = X . q^T, 32
//            UMMAs (M=128, N=64, K=16) from the K-major row blocks and the
//            K-major q into TMEM;
//   softmax  warps 2-5 (thread i = row i): tcgen05.ld the row's 64 logits,
//            per-head tile max with redux.sync.max.f32 across the warp and a
//            4-way max across warps, p = exp2(l - m) written as P^T (the
//            16-bit MN-major operand) to shared memory, per-thread partial row
//            sums kept in registers;
//   values   warp 1: O^T[512 dims x 64 heads] += X^T . P^T as four M=128
//            chunks (X read as the MN-major operand), accumulating in TMEM;
//            each chunk's commit frees its two column blocks for the next tile.
// The running max per head is only raised when a tile exceeds it by more than
// 2^8 (then O^T and the partial sums are rescaled), so p <= 256 always and the
// rescale is rare.  Compressed tiles multiply in bf16; the raw tile in fp16
// with q converted in place to fp16 (exact for |q| in [2^-14, 65504]).
// Split items write unnormalised partials (O, m, l) that attn_merge_kernel
// combines by log-sum-exp.
//
// Every wait is bounded (DS4A_DEV_TIMEOUT); on timeout the CTA drains what it
// issued (bounded), frees TMEM and returns.
#include "common.cuh"
#include "internal.h"

namespace ds4a {
namespace {

constexpr int TR = 128;                       // rows per tile (UMMA M of the logit GEMM)
constexpr int kThreads = 192;                 // warp 0 gather, warp 1 UMMA/TMEM, warps 2-5 softmax
constexpr int kQBlk = kNHead * 128;           // 64 heads x 64 dims x 2 B = 8 KB
constexpr int kXBlk = TR * 128;               // 128 rows x 64 dims x 2 B = 16 KB
constexpr int kOffQ = 0;
constexpr int kOffX = kOffQ + 8 * kQBlk;      // 64 KB
constexpr int kOffP = kOffX + 8 * kXBlk;      // +128 KB
constexpr int kOffSmax = kOffP + TR * 128;    // +16 KB: P^T [128 rows][64 heads]
constexpr int kOffMused = kOffSmax + 4 * kNHead * 4;
constexpr int kOffAlpha = kOffMused + kNHead * 4;
constexpr int kOffInvL = kOffAlpha + kNHead * 4;
constexpr int kOffBar = kOffInvL + kNHead * 4;
constexpr int kNumBars = 8 + 8 + 10;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 32 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kTmemCols = 512;           // S^T: 64 columns, O^T: 4 x 64 columns
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 64;
constexpr int kMaxSplit = 16;
constexpr float kRescaleThreshold = 8.0f;     // log2 units

// UMMA instruction descriptors (see idesc_bf16_f32): logits with K-major A/B,
// values with MN-major A (rows x dims read as dims x rows) and MN-major B.
__host__ __device__ constexpr uint32_t idesc_f16(bool f16_inputs, bool mn_major) {
    const uint32_t fmt = f16_inputs ? 0u : 1u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (mn_major ? (1u << 15) | (1u << 16) : 0u) |
           (static_cast<uint32_t>(kNHead >> 3) << 17) | (static_cast<uint32_t>(TR >> 4) << 24);
}

// Shared-memory descriptor with explicit leading / stride byte offsets (128B swizzle).
DS4A_DEV uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

DS4A_DEV void gather4(void *dst, const void *map, uint64_t *bar, int col, int r0, int r1, int r2, int r3) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
        : "memory");
}
DS4A_DEV void tma_load_2d_nohint(void *dst, const void *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
DS4A_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
DS4A_DEV float warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

DS4A_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
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
DS4A_DEV void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
DS4A_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

DS4A_DEV bool wait_drain(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

// What one work item covers.
struct Item {
    int unit, split;
    int cnt;             // selected compressed rows (clamped to [0, top_k])
    int nrw;             // raw rows
    int ct;              // compressed tiles
    int t0, t1;          // tile range of this split
    long long raw_row0;  // row coordinate of raw row 0 in the raw map
    long long comp_row0; // row coordinate of compressed row 0 of the unit in the rows map
};

DS4A_DEV Item make_item(const AttnArgs &a, int it, int n_split) {
    Item m;
    m.unit = it / n_split;
    m.split = it - m.unit * n_split;
    int cnt = a.count[m.unit];
    cnt = cnt < 0 ? 0 : (cnt > a.top_k ? a.top_k : cnt);
    m.cnt = cnt;
    m.comp_row0 = static_cast<long long>(m.unit) * a.rows_per_unit;
    if (a.q_pos) {
        const long long p = a.q_pos[m.unit];
        const long long lo = max(p - (kNSwa - 1) - a.raw_pos0, 0LL);
        const long long hi = min(p - a.raw_pos0, static_cast<long long>(a.n_raw_rows) - 1);
        m.nrw = hi >= lo ? static_cast<int>(hi - lo + 1) : 0;
        m.raw_row0 = m.nrw ? lo : 0;
    } else {
        int n = a.n_raw[m.unit];
        n = n < 0 ? 0 : (n > kNSwa ? kNSwa : n);
        m.nrw = n;
        m.raw_row0 = static_cast<long long>(m.unit) * a.raw_per_unit;
    }
    m.ct = (m.cnt + TR - 1) / TR;
    const int nt = m.ct + (m.nrw + TR - 1) / TR;
    const int tps = (nt + n_split - 1) / n_split;
    m.t0 = m.split * tps;
    m.t1 = min(nt, m.t0 + tps);
    return m;
}

// Row j of tile t: valid?  (compressed rows need an index inside [0, N_cap)).
DS4A_DEV bool row_valid(const AttnArgs &a, const Item &m, int t, int j, int *coord) {
    if (t < m.ct) {
        const int jj = t * TR + j;
        if (jj >= m.cnt) return false;
        const int iv = __ldg(a.idx + static_cast<long long>(m.unit) * a.top_k + jj);
        if (iv < 0 || iv >= a.N_cap) return false;
        if (coord) *coord = static_cast<int>(m.comp_row0 + iv);
        return true;
    }
    const int jj = (t - m.ct) * TR + j;
    if (jj >= m.nrw) return false;
    if (coord) *coord = static_cast<int>(m.raw_row0 + jj);
    return true;
}

__global__ void __launch_bounds__(kThreads, 1) sparse_attn_kernel(const __grid_constant__ AttnArgs a, int n_split,
                                                                  int n_items) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem + kOffQ;
    uint8_t *sX = smem + kOffX;
    uint8_t *sP = smem + kOffP;
    float *sSmax = reinterpret_cast<float *>(smem + kOffSmax);
    float *sMused = reinterpret_cast<float *>(smem + kOffMused);
    float *sAlpha = reinterpret_cast<float *>(smem + kOffAlpha);
    float *sInvL = reinterpret_cast<float *>(smem + kOffInvL);
    uint64_t *slot_full = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *slot_empty = slot_full + 8;
    uint64_t *q_full = slot_empty + 8;
    uint64_t *q_free = q_full + 1;
    uint64_t *q16_ready = q_free + 1;
    uint64_t *s_full = q16_ready + 1;
    uint64_t *s_empty = s_full + 1;
    uint64_t *p_full = s_empty + 1;
    uint64_t *o_ready = p_full + 1;
    uint64_t *o_free = o_ready + 1;
    uint64_t *drain = o_free + 1;
    uint64_t *grp = drain + 1;                   // softmax-group barrier (4 warps)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    int *any_rescale = reinterpret_cast<int *>(smem + kOffMisc + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int b = 0; b < 8; ++b) {
            mbar_init(&slot_full[b], 1);
            mbar_init(&slot_empty[b], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_free, 1);
        mbar_init(q16_ready, 4);
        mbar_init(s_full, 1);
        mbar_init(s_empty, 4);
        mbar_init(p_full, 4);
        mbar_init(o_ready, 1);
        mbar_init(o_free, 4);
        mbar_init(drain, 1);
        mbar_init(grp, 4);
        *abort_flag = 0;
        *any_rescale = 0;
        mbar_fence_init();
        tma_prefetch_desc(&a.tm_q);
        tma_prefetch_desc(&a.tm_rows);
        tma_prefetch_desc(&a.tm_raw);
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const float NEG_INF = -__int_as_float(0x7f800000);

    if (warp == 0) {
        // ------------------------------------------------------------ gather producer
        uint32_t qph = 0, sph[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        bool ok = true;
        for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
            const Item m = make_item(a, it, n_split);
            if (m.t0 >= m.t1) continue;
            ok = __all_sync(0xffffffffu, mbar_wait(q_free, qph ^ 1, abort_flag));
            if (!ok) break;
            qph ^= 1;
            if (lane == 0) {
                mbar_arrive_expect_tx(q_full, 8 * kQBlk);
                for (int b = 0; b < 8; ++b) tma_load_2d_nohint(sQ + b * kQBlk, &a.tm_q, q_full, b * 64, m.unit * kNHead);
            }
            for (int t = m.t0; ok && t < m.t1; ++t) {
                int c[4];
                bool bad_idx = false;
                for (int i = 0; i < 4; ++i) {
                    c[i] = -1;                                   // out of range: loads zeros
                    int co = 0;
                    if (row_valid(a, m, t, 4 * lane + i, &co)) {
                        c[i] = co;
                    } else if (t < m.ct && t * TR + 4 * lane + i < m.cnt) {
                        bad_idx = true;                          // index outside [0, N_cap)
                    }
                }
                if (__any_sync(0xffffffffu, bad_idx) && lane == 0) report(a.status, DS4A_DEV_BOUNDS);
                const void *map = t < m.ct ? static_cast<const void *>(&a.tm_rows) : static_cast<const void *>(&a.tm_raw);
                for (int b = 0; b < 8; ++b) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&slot_empty[b], sph[b] ^ 1, abort_flag));
                    if (!ok) break;
                    sph[b] ^= 1;
                    if (lane == 0) mbar_arrive_expect_tx(&slot_full[b], kXBlk);
                    __syncwarp();
                    gather4(sX + b * kXBlk + lane * 512, map, &slot_full[b], b * 64, c[0], c[1], c[2], c[3]);
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) report(a.status, DS4A_DEV_TIMEOUT);
            // Let issued copies land: the last armed phase of every slot and of q.
            for (int b = 0; b < 8; ++b) wait_drain(&slot_full[b], sph[b] ^ 1);
            wait_drain(q_full, qph ^ 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            uint32_t qph = 0, q16ph = 0, sfph[8] = {0, 0, 0, 0, 0, 0, 0, 0}, seph = 0, pph = 0, ofph = 0;
            bool ok = true, first_item = true;
            constexpr uint32_t id_s_bf = idesc_f16(false, false), id_s_f16 = idesc_f16(true, false);
            constexpr uint32_t id_v_bf = idesc_f16(false, true), id_v_f16 = idesc_f16(true, true);
            const uint32_t aQ = smem_u32(sQ), aX = smem_u32(sX), aP = smem_u32(sP);
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const Item m = make_item(a, it, n_split);
                if (m.t0 >= m.t1) continue;
                if (!mbar_wait(q_full, qph, abort_flag)) { ok = false; break; }
                qph ^= 1;
                bool q16 = false, first_pv = true;
                for (int t = m.t0; ok && t < m.t1; ++t) {
                    const bool raw = t >= m.ct;
                    if (raw && !q16) {
                        if (!mbar_wait(q16_ready, q16ph, abort_flag)) { ok = false; break; }
                        q16ph ^= 1;
                        q16 = true;
                    }
                    // logits S^T = X . q^T
                    if (!mbar_wait(s_empty, seph ^ 1, abort_flag)) { ok = false; break; }
                    seph ^= 1;
                    for (int b = 0; b < 8 && ok; ++b) {
                        if (!mbar_wait(&slot_full[b], sfph[b], abort_flag)) { ok = false; break; }
                        sfph[b] ^= 1;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16(tmem + kTmemS, sw128_desc(aX + b * kXBlk + kk * 32, 16, 1024),
                                      sw128_desc(aQ + b * kQBlk + kk * 32, 16, 1024), raw ? id_s_f16 : id_s_bf,
                                      (b | kk) ? 1u : 0u);
                    }
                    if (!ok) break;
                    umma_commit(s_full);
                    if (t == m.t1 - 1) umma_commit(q_free);
                    // values O^T += X^T . P^T
                    if (!mbar_wait(p_full, pph, abort_flag)) { ok = false; break; }
                    pph ^= 1;
                    if (first_pv && !first_item) {
                        if (!mbar_wait(o_free, ofph, abort_flag)) { ok = false; break; }
                        ofph ^= 1;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int ks = 0; ks < TR / 16; ++ks)
                            umma_bf16(tmem + kTmemO + c * kNHead,
                                      sw128_desc(aX + 2 * c * kXBlk + ks * 2048, kXBlk, 1024),
                                      sw128_desc(aP + ks * 2048, 8192, 1024), raw ? id_v_f16 : id_v_bf,
                                      (first_pv && ks == 0) ? 0u : 1u);
                        umma_commit(&slot_empty[2 * c]);
                        umma_commit(&slot_empty[2 * c + 1]);
                    }
                    first_pv = false;
                }
                if (!ok) break;
                umma_commit(o_ready);
                first_item = false;
            }
            if (!ok) {
                *abort_flag = 1;
                report(a.status, DS4A_DEV_TIMEOUT);
            }
            umma_commit(drain);
            wait_drain(drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int q4 = warp & 3;                 // TMEM lane quarter
        const int i = q4 * 32 + lane;            // tile row (logits) / dim within a chunk (values)
        const int e = (warp - 2) * 32 + lane;    // 0..127 inside the softmax group
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        const float sl2 = a.scale * 1.4426950408889634f;
        uint32_t qph = 0, sfph = 0, orph = 0, gph = 0;
        bool ok = true;
        // Barrier of the four softmax warps on an mbarrier, so that a wait that
        // gives up (abort) cannot leave the other warps stuck.
        auto group_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(grp);
            const bool r = __all_sync(0xffffffffu, mbar_wait(grp, gph, abort_flag));
            gph ^= 1;
            return r;
        };
        for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
            const Item m = make_item(a, it, n_split);
            if (m.t0 >= m.t1) {
                // Empty row set: out = 0, lse = -inf (or an empty partial).
                if (n_split == 1) {
                    float *o = a.out + static_cast<long long>(m.unit) * kNHead * kHeadDim;
                    for (int k = e; k < kNHead * kHeadDim; k += 128) o[k] = 0.f;
                    if (a.lse && e < kNHead) a.lse[static_cast<long long>(m.unit) * kNHead + e] = NEG_INF;
                } else if (e < kNHead) {
                    float *ml = static_cast<float *>(a.ws) + static_cast<long long>(a.units) * n_split * kNHead * kHeadDim;
                    const long long slot = static_cast<long long>(m.unit) * n_split + m.split;
                    ml[(slot * kNHead + e) * 2] = NEG_INF;
                    ml[(slot * kNHead + e) * 2 + 1] = 0.f;
                }
                continue;
            }
            ok = __all_sync(0xffffffffu, mbar_wait(q_full, qph, abort_flag));
            if (!ok) break;
            qph ^= 1;
            if (e < kNHead) sMused[e] = NEG_INF;
            float lacc[kNHead];
#pragma unroll
            for (int h = 0; h < kNHead; ++h) lacc[h] = 0.f;
            bool q16 = false, first_pv = true;
            if (!(ok = group_sync())) break;
            for (int t = m.t0; ok && t < m.t1; ++t) {
                const bool raw = t >= m.ct;
                if (raw && !q16) {
                    // Previous logit GEMMs of this item have completed (their S
                    // was consumed); q -> fp16 in place for the fp16 raw tier.
                    uint4 *qv = reinterpret_cast<uint4 *>(sQ);
                    for (int k = e; k < 8 * kQBlk / 16; k += 128) {
                        uint4 v = qv[k];
                        uint32_t *w = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            w[j] = pack2<true>(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u));
                        qv[k] = v;
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(q16_ready);
                    q16 = true;
                }
                const bool valid = row_valid(a, m, t, i, nullptr);
                ok = __all_sync(0xffffffffu, mbar_wait(s_full, sfph, abort_flag));
                if (!ok) break;
                sfph ^= 1;
                tc_fence_after();
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lane_off + kTmemS, r0);
                tmem_ld32(tmem + lane_off + kTmemS + 32, r1);
                tmem_wait_ld(r0);
                tmem_wait_ld(r1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_empty);
                float x[kNHead];
#pragma unroll
                for (int h = 0; h < 32; ++h) {
                    x[h] = valid ? __uint_as_float(r0[h]) * sl2 : NEG_INF;
                    x[32 + h] = valid ? __uint_as_float(r1[h]) * sl2 : NEG_INF;
                }
                // per-head max over this warp's 32 rows, then over the 4 warps
#pragma unroll
                for (int h = 0; h < kNHead; ++h) {
                    const float mx = warp_max(x[h]);
                    if (lane == (h & 31)) sSmax[q4 * kNHead + h] = mx;
                }
                if (e == 0) *any_rescale = 0;
                if (!(ok = group_sync())) break;
                if (e < kNHead) {
                    const float mt = fmaxf(fmaxf(sSmax[e], sSmax[kNHead + e]),
                                           fmaxf(sSmax[2 * kNHead + e], sSmax[3 * kNHead + e]));
                    const float mo = sMused[e];
                    float alpha = 1.f;
                    if (mo == NEG_INF) {
                        sMused[e] = mt;                 // first finite max (O and sums are still 0)
                    } else if (mt > mo + kRescaleThreshold) {
                        sMused[e] = mt;
                        alpha = exp2f(mo - mt);
                        *any_rescale = 1;
                    }
                    sAlpha[e] = alpha;
                }
                if (!(ok = group_sync())) break;
                const bool rescale = *any_rescale != 0;
                uint32_t pk[32];
#pragma unroll
                for (int h = 0; h < kNHead; h += 2) {
                    const float m0 = sMused[h], m1 = sMused[h + 1];
                    const float p0 = exp2f(x[h] - (m0 == NEG_INF ? 0.f : m0));
                    const float p1 = exp2f(x[h + 1] - (m1 == NEG_INF ? 0.f : m1));
                    if (rescale) {
                        lacc[h] *= sAlpha[h];
                        lacc[h + 1] *= sAlpha[h + 1];
                    }
                    lacc[h] += p0;
                    lacc[h + 1] += p1;
                    pk[h >> 1] = raw ? pack2<true>(p0, p1) : pack2<false>(p0, p1);
                }
                // P^T row i: 64 heads = 8 chunks of 16 B, 128B swizzle.
                uint4 *prow = reinterpret_cast<uint4 *>(sP + i * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    prow[c ^ (i & 7)] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                fence_proxy_async();
                if (rescale && !first_pv) {
                    // The previous values GEMM is complete (this tile's logits needed
                    // every column block it freed): scale O^T column h by alpha_h.
                    tc_fence_after();
                    for (int c = 0; c < 4; ++c) {
                        for (int half = 0; half < 2; ++half) {
                            uint32_t v[32];
                            const uint32_t ta = tmem + lane_off + kTmemO + c * kNHead + half * 32;
                            tmem_ld32(ta, v);
                            tmem_wait_ld(v);
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                v[k] = __float_as_uint(__uint_as_float(v[k]) * sAlpha[half * 32 + k]);
                            tmem_st32(ta, v);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
                first_pv = false;
            }
            if (!ok) break;
            // ---- epilogue: row sums across the 128 rows, then O^T out
#pragma unroll
            for (int h = 0; h < kNHead; ++h) {
                float v = lacc[h];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                if (lane == (h & 31)) sSmax[q4 * kNHead + h] = v;
            }
            if (!(ok = group_sync())) break;
            const long long slot = static_cast<long long>(m.unit) * n_split + m.split;
            if (e < kNHead) {
                const float L = sSmax[e] + sSmax[kNHead + e] + sSmax[2 * kNHead + e] + sSmax[3 * kNHead + e];
                const float M = sMused[e];
                if (n_split == 1) {
                    sInvL[e] = L > 0.f ? 1.f / L : 0.f;
                    if (a.lse)
                        a.lse[static_cast<long long>(m.unit) * kNHead + e] =
                            L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : NEG_INF;
                } else {
                    sInvL[e] = 1.f;
                    float *ml = static_cast<float *>(a.ws) + static_cast<long long>(a.units) * n_split * kNHead * kHeadDim;
                    ml[(slot * kNHead + e) * 2] = L > 0.f ? M : NEG_INF;
                    ml[(slot * kNHead + e) * 2 + 1] = L;
                }
            }
            if (!(ok = group_sync())) break;
            ok = __all_sync(0xffffffffu, mbar_wait(o_ready, orph, abort_flag));
            if (!ok) break;
            orph ^= 1;
            tc_fence_after();
            float *obase = n_split == 1 ? a.out + static_cast<long long>(m.unit) * kNHead * kHeadDim
                                        : static_cast<float *>(a.ws) + slot * kNHead * kHeadDim;
            for (int c = 0; c < 4; ++c) {
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_off + kTmemO + c * kNHead + half * 32, v);
                    tmem_wait_ld(v);
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int h = half * 32 + k;
                        obase[static_cast<long long>(h) * kHeadDim + c * TR + i] = __uint_as_float(v[k]) * sInvL[h];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
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
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Combines the split partials of one (unit, head): O = sum_s 2^(m_s - M) O_s /
// sum_s 2^(m_s - M) l_s, lse = (M + log2 L) ln 2.
__global__ void __launch_bounds__(128) attn_merge_kernel(const __grid_constant__ AttnArgs a, int n_split) {
    const int unit = blockIdx.x / kNHead;
    const int h = blockIdx.x - unit * kNHead;
    const float *wo = static_cast<const float *>(a.ws);
    const float *ml = wo + static_cast<long long>(a.units) * n_split * kNHead * kHeadDim;
    const float NEG_INF = -__int_as_float(0x7f800000);
    float M = NEG_INF;
    for (int s = 0; s < n_split; ++s) {
        const long long slot = static_cast<long long>(unit) * n_split + s;
        const float2 v = *reinterpret_cast<const float2 *>(ml + (slot * kNHead + h) * 2);
        if (v.y > 0.f) M = fmaxf(M, v.x);
    }
    float wts[kMaxSplit];
    float L = 0.f;
    for (int s = 0; s < n_split; ++s) {
        const long long slot = static_cast<long long>(unit) * n_split + s;
        const float2 v = *reinterpret_cast<const float2 *>(ml + (slot * kNHead + h) * 2);
        wts[s] = v.y > 0.f ? exp2f(v.x - M) : 0.f;
        L += wts[s] * v.y;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int d = threadIdx.x * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < n_split; ++s) {
        if (wts[s] == 0.f) continue;
        const long long slot = static_cast<long long>(unit) * n_split + s;
        const float4 v = *reinterpret_cast<const float4 *>(wo + (slot * kNHead + h) * kHeadDim + d);
        acc.x += wts[s] * v.x;
        acc.y += wts[s] * v.y;
        acc.z += wts[s] * v.z;
        acc.w += wts[s] * v.w;
    }
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    *reinterpret_cast<float4 *>(a.out + (static_cast<long long>(unit) * kNHead + h) * kHeadDim + d) = acc;
    if (a.lse && threadIdx.x == 0)
        a.lse[static_cast<long long>(unit) * kNHead + h] =
            L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : NEG_INF;
}

}  // namespace

int attn_num_splits(int units, int top_k) {
    // Enough work items to cover 152 SMs; a split holds at least one 128-row tile.
    const int max_tiles = (top_k + TR - 1) / TR + (kNSwa + TR - 1) / TR;
    if (units >= 152) return 1;
    int s = (152 + units - 1) / units;
    if (s > max_tiles) s = max_tiles;
    if (s > kMaxSplit) s = kMaxSplit;
    return s < 1 ? 1 : s;
}

size_t attn_ws_bytes(int units, int top_k) {
    const int s = attn_num_splits(units, top_k);
    if (s == 1) return 0;
    return static_cast<size_t>(units) * s * kNHead * (kHeadDim + 2) * sizeof(float);
}

cudaError_t launch_sparse_attn(const AttnArgs &a, int num_sms, cudaStream_t s) {
    const int n_split = attn_num_splits(a.units, a.top_k);
    cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long items = static_cast<long long>(a.units) * n_split;
    if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
    const int grid = static_cast<int>(items < num_sms ? items : num_sms);
    sparse_attn_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, n_split, static_cast<int>(items));
    e = cudaGetLastError();
    if (e != cudaSuccess || n_split == 1) return e;
    attn_merge_kernel<<<static_cast<unsigned>(static_cast<long long>(a.units) * kNHead), 128, 0, s>>>(a, n_split);
    return cudaGetLastError();
}

}  // namespace ds4a
