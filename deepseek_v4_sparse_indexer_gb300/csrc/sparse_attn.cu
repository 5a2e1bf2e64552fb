// Sparse attention over the selected compressed rows and the raw window, on
// the 5th-generation tensor cores ("DwarfStar(ds4.c) のアーキテクチャを読む"
// §3: three tiers; §2: 64 query heads, one KV head whose 512-d rows are both
// key and value; §3-1: the raw window of the last 128 tokens kept rounded to
// f16).
//
// One CTA (persistent, one per SM) walks work items = (unit, split), where a
// unit is one decode query or one query of a prefill chunk.  The unit's row
// list [selected compressed rows..., raw-window rows...] is cut into 64-row
// tiles, double-buffered in shared memory:
//   gather   warps 6-13 (row lists; 6-9 for dense row lists, whose whole
//            tiles come by TMA): the warps share every tile (4-row groups dealt
//            round-robin) with 16-byte cp.async into eight 8 KB column
//            blocks in the 128B-swizzled layout; masked rows are zero-filled
//            and per-group row-validity bits go to shared memory; each
//            thread fences its copies into the async proxy before its warp
//            arrives on the buffer's barrier.  A whole tile of contiguous
//            rows (the raw window, or a dense row list) is instead eight TMA
//            tile loads (64 columns x 64 rows each) issued by one thread.
//            With the FP8 row store, a compressed row is 512 E4M3 codes and a
//            power-of-two scale: lane l loads codes 16l .. 16l+15 of a row (one
//            row per warp instruction, into registers), and the warp writes
//            them out as exact bf16 values (code * scale) into the same
//            swizzled tile, so the GEMMs below do not change;
//   logits   warp 4: S[64 heads x 64 rows] = q . X^T, 32 UMMAs
//            (M=64, N=64, K=16, both operands K-major) into one of two TMEM
//            buffers (head h of the M=64 accumulator sits in TMEM lane
//            32*(h/16) + h%16);
//   softmax  warps 0-3 (warp w reads TMEM lanes 32w..32w+15 = heads
//            16w..16w+15 with the 16x256b shape: thread t holds heads
//            16w + t/4 and 16w + t/4 + 8 for the 16 rows 8j + 2(t%4) + {0,1}).
//            The per-head tile max is a register max plus two shuffles;
//            p = exp2(l - m) goes to P[head][row] (the K-major operand of the
//            values GEMM), row sums stay in registers;
//   values   warp 5: O^T[512 dims x 64 heads] += X^T . P^T as four M=128
//            chunks (K = 64 rows; X read as the MN-major operand, P as the
//            K-major one), accumulating in TMEM; its commit frees the row
//            buffer and the P buffer.
// The running max per head is only raised when a tile exceeds it by more than
// 2^8, so p <= 256 always.  A raise needs O^T (whose TMEM lanes are the 512
// dims, spread over all four softmax warps) rescaled: the four warps exchange
// a flag and the factors once per tile, and all of them rescale their lanes
// when any head was raised (rare).  Compressed tiles multiply in bf16; raw
// tiles in fp16 with q converted in place to fp16 (exact for |q| in
// [2^-14, 65504]).  Split items write unnormalised partials (O, m, l) that
// attn_merge_kernel combines by log-sum-exp.
//
// The two GEMM streams have their own issuing warps, so that the values GEMM
// of a tile (which frees its row buffer) never queues behind the logits GEMMs
// of the next one.  A whole converged warp runs each issue loop and one
// elected lane issues: a lone lane inside a divergent branch issues a UMMA
// only every ~45 cycles, a converged warp as fast as the tensor core takes them
// (32 cycles for M=64, N=64, K=16).  Descriptors are advanced by adding the
// byte offset / 16 to a base descriptor.
//
// Every wait is bounded (DS4A_DEV_TIMEOUT); on timeout the CTA drains what it
// issued (bounded), frees TMEM and returns.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace ds4a {
namespace {

constexpr int TR = 64;                        // rows per tile (UMMA N of the logit GEMM)
constexpr int kSoftmaxWarps = 4;              // warps 0-3: softmax + epilogue (TMEM lane quarters)
constexpr int kMmaWarp = 4;                   // warp 4: TMEM owner + logits UMMA issuer
constexpr int kPvWarp = 5;                    // warp 5: values UMMA issuer
constexpr int kFirstGatherWarp = 6;           // warps 6..6+GW-1: row gather (cp.async)
constexpr int kRowGroups = TR / 4;            // 4-row groups of a tile, dealt round-robin to the gather warps
// Gather warps per CTA: eight for gathered row lists (two 4-row groups each:
// the copies and the FP8 expansion are the tile's critical path); four for
// dense row lists, whose tiles arrive by TMA and whose gather warps only
// arrive on the buffer barrier (640 x 8,192: 1.015 ms with four, 1.036 ms
// with six, 1.09 ms with eight).
constexpr int kGatherWarpsList = 8;
constexpr int kGatherWarpsDense = 4;
constexpr int attn_threads(int gw) { return (kFirstGatherWarp + gw) * 32; }
constexpr int kQBlk = kNHead * 128;           // 64 heads x 64 dims x 2 B = 8 KB
constexpr int kXBlk = TR * 128;               // 64 rows x 64 dims x 2 B = 8 KB
constexpr int kXBuf = 8 * kXBlk;              // one row tile: 64 KB
constexpr int kPBuf = kNHead * 128;           // P [64 heads][64 rows] 16-bit: 8 KB
constexpr int kOffQ = 0;
constexpr int kOffX = kOffQ + 8 * kQBlk;      // q: 64 KB
constexpr int kOffP = kOffX + 2 * kXBuf;      // two row tiles: 128 KB
constexpr int kOffValid = kOffP + 2 * kPBuf;  // two P buffers: 16 KB
constexpr int kOffAlpha = kOffValid + 2 * kRowGroups;  // [2][16] row-validity nibbles
constexpr int kOffFlag = kOffAlpha + 2 * kNHead * 4;
constexpr int kOffInvL = kOffFlag + 2 * kSoftmaxWarps * 4;
constexpr int kOffBar = kOffInvL + kNHead * 4;
constexpr int kNumBars = 18;                  // 17 used
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 32 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffBar % 8 == 0, "mbarrier alignment");
constexpr uint32_t kTmemCols = 512;           // S: 2 x 64 columns, O^T: 4 x 64 columns
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 128;
constexpr int kMaxAttnCtas = 160;            // grid cap (one persistent CTA per SM; 152 on GB300)
constexpr float kRescaleThreshold = 8.0f;     // log2 units

// UMMA instruction descriptors (see idesc_bf16_f32): logits (M = 64 heads,
// N = 64 rows, both K-major); values (M = 128 dims, N = 64 heads) with the
// MN-major A (row tile read as dims x rows) and the K-major B (P).
__host__ __device__ constexpr uint32_t idesc_f16(bool f16_inputs, bool values) {
    const uint32_t fmt = f16_inputs ? 0u : 1u;
    const uint32_t m = values ? 128u : static_cast<uint32_t>(kNHead);
    const uint32_t n = values ? static_cast<uint32_t>(kNHead) : static_cast<uint32_t>(TR);
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (values ? (1u << 15) : 0u) | ((n >> 3) << 17) | ((m >> 4) << 24);
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

DS4A_DEV void tma_load_2d_nohint(void *dst, const void *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
DS4A_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

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

// Eight E4M3 codes (two words) times a power-of-two scale as eight bf16
// (four words, dims in order).  E4M3 -> f16 is exact, and so are the scaling
// in fp32 and the rounding to bf16 of a value with at most four significant
// bits (down to 2^-133, the smallest bf16 subnormal).
DS4A_DEV void e4m3x8_to_bf16(uint32_t w0, uint32_t w1, float s, uint32_t (&o)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t w = j < 2 ? w0 : w1;
        const uint16_t pair = static_cast<uint16_t>(w >> (16 * (j & 1)));
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
        o[j] = pack2<false>(f.x * s, f.y * s);
    }
}
// 16-byte read-only load that bypasses L1 (rows are read once).  Volatile, so
// that it stays ahead of the buffer wait that follows it.
DS4A_DEV uint4 ld_nc_v4(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
DS4A_DEV void st_shared_v4(uint32_t addr, const uint32_t (&v)[4]) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
}

// 2^x by the MUFU approximation (relative error ~2^-22; -inf -> +0).
DS4A_DEV float ex2(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// UMMA / commit issued by the elected lane of a converged warp.
DS4A_DEV void umma_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
DS4A_DEV void commit_elect(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}
// Warp-wide bounded wait (hinted try_wait: a waiting issuer takes no issue slots).
DS4A_DEV bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return __all_sync(0xffffffffu, mbar_wait_hint(bar, parity, abort));
}

// Bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, multiple of 16 bytes).
DS4A_DEV void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

DS4A_DEV bool wait_drain(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

// What one work item covers: this CTA's piece of one unit.
struct Item {
    int unit;            // 64-head sub-unit (q, out, lse); ru: its row-side unit
    bool split;          // the unit's tiles are shared with another CTA: the piece is a partial
    long long slot;      // its partial's workspace slot
    int ru;
    int cnt;             // selected compressed rows (clamped to [0, top_k])
    int nrw;             // raw rows
    int ct;              // compressed tiles
    int t0, t1;          // tile range of this split
    long long raw_row0;  // row index of the unit's raw row 0 in the raw buffer
    long long comp_row0; // row index of the unit's compressed row 0 in the rows buffer
};

// Work schedule.  With G CTAs, the first R = floor(units / G) rounds of units
// are dealt whole and strided (CTA c: units c, c + G, ...), so that the CTAs
// work on neighbouring units at any time.  The remaining units' tiles (nt per
// unit: the most a unit can have, top_k compressed rows and the 128-row raw
// window) are cut into g_rem equal shares, one per CTA c < g_rem, so that
// every CTA ends with the same number of tiles to within one.  A unit cut by a
// share boundary is computed in pieces whose partials (unnormalised O, m, l)
// attn_merge_kernel combines.
struct Sched {
    int nt, R, n_pieces;
    int u_rem0;              // first remainder unit (R x G)
    long long rs, re;        // this CTA's remainder share: remainder tiles [rs, re)
    int v0;                  // its first remainder unit (relative to u_rem0)
};

DS4A_DEV Sched make_sched(const AttnArgs &a, int nt, int g_rem) {
    Sched sc;
    const int G = gridDim.x, c = blockIdx.x;
    sc.nt = nt;
    sc.R = a.units / G;
    sc.u_rem0 = sc.R * G;
    const long long t_rem = static_cast<long long>(a.units - sc.u_rem0) * nt;
    sc.rs = sc.re = 0;
    sc.v0 = 0;
    int n_rem = 0;
    if (c < g_rem) {
        sc.rs = static_cast<long long>(c) * t_rem / g_rem;
        sc.re = static_cast<long long>(c + 1) * t_rem / g_rem;
        if (sc.re > sc.rs) {
            sc.v0 = static_cast<int>(sc.rs / nt);
            n_rem = static_cast<int>((sc.re - 1) / nt) + 1 - sc.v0;
        }
    }
    sc.n_pieces = sc.R + n_rem;
    return sc;
}

// Piece i of this CTA's schedule.
DS4A_DEV Item make_piece(const AttnArgs &a, const Sched &sc, int i) {
    Item m;
    int lt0 = 0, lt1 = sc.nt;
    if (i < sc.R) {
        m.unit = blockIdx.x + i * gridDim.x;
        m.split = false;
        m.slot = 0;
    } else {
        const int v = sc.v0 + (i - sc.R);
        m.unit = sc.u_rem0 + v;
        const long long vs = static_cast<long long>(v) * sc.nt;
        lt0 = static_cast<int>(max(sc.rs - vs, 0LL));
        lt1 = static_cast<int>(min(sc.re - vs, static_cast<long long>(sc.nt)));
        m.split = lt0 > 0 || lt1 < sc.nt;
        m.slot = 2LL * blockIdx.x + (vs <= sc.rs ? 0 : 1);   // first piece of the share: slot 0, last: slot 1
    }
    m.ru = a.hsplit == 2 ? m.unit >> 1 : m.unit;     // 128 heads: two sub-units share the rows
    int cnt = a.count[m.ru];
    if (lt0 == 0 && (cnt < 0 || cnt > a.top_k) && threadIdx.x == 0) report(a.status, DS4A_DEV_BOUNDS);
    cnt = cnt < 0 ? 0 : (cnt > a.top_k ? a.top_k : cnt);
    m.cnt = cnt;
    m.comp_row0 = static_cast<long long>(m.ru) * a.rows_per_unit;
    if (a.q_pos) {
        const long long p = a.q_pos[m.ru];
        const long long lo = max(p - (kNSwa - 1) - a.raw_pos0, 0LL);
        const long long hi = min(p - a.raw_pos0, static_cast<long long>(a.n_raw_rows) - 1);
        m.nrw = hi >= lo ? static_cast<int>(hi - lo + 1) : 0;
        m.raw_row0 = m.nrw ? lo : 0;
    } else {
        int n = a.n_raw[m.ru];
        n = n < 0 ? 0 : (n > kNSwa ? kNSwa : n);
        m.nrw = n;
        m.raw_row0 = static_cast<long long>(m.ru) * a.raw_per_unit;
    }
    m.ct = (m.cnt + TR - 1) / TR;
    m.t0 = lt0;
    m.t1 = min(m.ct + (m.nrw + TR - 1) / TR, lt1);
    return m;
}

DS4A_DEV void tmem_ld16x256_x8(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

template <int GW>
__global__ void __launch_bounds__(attn_threads(GW), 1) sparse_attn_kernel(const __grid_constant__ AttnArgs a, int nt,
                                                                          int g_rem) {
    constexpr int kGatherWarps = GW;
    constexpr int kGroupsPerWarp = (kRowGroups + kGatherWarps - 1) / kGatherWarps;
    pdl_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    // Aligned by pointer arithmetic on the __shared__ array (not through an
    // integer), so that the compiler keeps shared-space accesses for it.
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem + kOffQ;
    uint8_t *sX = smem + kOffX;
    uint8_t *sP = smem + kOffP;
    uint8_t *sValid = smem + kOffValid;          // [2][16] bit i of byte g: tile row 4g + i is listed and in range
    float *sAlpha = reinterpret_cast<float *>(smem + kOffAlpha);        // [2][64] this tile's rescale factor per head
    uint32_t *sFlag = reinterpret_cast<uint32_t *>(smem + kOffFlag);    // [2][4] softmax warp raised a head's max
    float *sInvL = reinterpret_cast<float *>(smem + kOffInvL);
    uint64_t *x_full = reinterpret_cast<uint64_t *>(smem + kOffBar);   // [2] row tile landed
    uint64_t *x_empty = x_full + 2;                                    // [2] values GEMM done: row tile + P free
    uint64_t *s_full = x_empty + 2;                                    // [2] logits in TMEM
    uint64_t *s_empty = s_full + 2;                                    // [2] logits read
    uint64_t *p_full = s_empty + 2;                                    // [2] P written
    uint64_t *q_full = p_full + 2;
    uint64_t *q_free = q_full + 1;
    uint64_t *q16_ready = q_free + 1;
    uint64_t *o_free = q16_ready + 1;
    uint64_t *drain = o_free + 1;
    uint64_t *drain_v = drain + 1;
    uint64_t *grp = drain_v + 1;                                       // softmax-group barrier
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&x_full[b], kGatherWarps);
            mbar_init(&x_empty[b], 1);
            mbar_init(&s_full[b], 1);
            mbar_init(&s_empty[b], kSoftmaxWarps);
            mbar_init(&p_full[b], kSoftmaxWarps);
        }
        mbar_init(q_full, 1);
        mbar_init(q_free, 1 + kSoftmaxWarps);  // the item's last logits GEMM + each softmax warp past its q wait
        mbar_init(q16_ready, kSoftmaxWarps);
        mbar_init(o_free, kSoftmaxWarps);
        mbar_init(drain, 1);
        mbar_init(drain_v, 1);
        mbar_init(grp, kSoftmaxWarps);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&a.tm_q);
        if (a.tma_rows) tma_prefetch_desc(&a.tm_rows);
        if (a.tma_raw) tma_prefetch_desc(&a.tm_raw);
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const Sched sc = make_sched(a, nt, g_rem);
    if (threadIdx.x == 0 && sc.n_pieces > 0) {
        // q of the first piece into L2 while the previous kernel finishes
        // (a prefetch cannot go stale: L2 is the point of coherence)
        const long long u0 = sc.R > 0 ? blockIdx.x : sc.u_rem0 + sc.v0;
        prefetch_l2(a.q + u0 * kNHead * kHeadDim, kNHead * kHeadDim * 2);
    }
    pdl_wait();                                  // the set-up above reads no global memory
    const uint32_t tmem = *tmem_slot;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const int u_end = sc.n_pieces;               // pieces 0 .. n_pieces-1
    const long long n_slots = 2LL * gridDim.x;

    if (warp >= kFirstGatherWarp) {
        // ------------------------------------------------------------ row gather
        // All gather warps walk the CTA's (item, tile) sequence; warp g of GW
        // copies the 4-row groups g, g + GW, ... (< 16) of every tile.  Lane l
        // copies 16-byte chunk (l & 7) of row 4k + (l >> 3) of group k in
        // every 64-column block: a warp instruction moves four full 128-byte
        // row segments.  Destinations follow the 128B swizzle.
        const int gw = warp - kFirstGatherWarp;
        const int chunk = lane & 7, rsub = lane >> 3;
        uint32_t xeph[2] = {0, 0};
        bool ok = true;
        auto first_tile = [&](int u, Item &m) -> int {
            for (; u < u_end; ++u) {
                m = make_piece(a, sc, u);
                if (m.t0 < m.t1) return u;
            }
            return u_end;
        };
        int ordinal = 0;                                   // item ordinal within this CTA's sequence
        auto advance = [&](int &u, int &t, Item &m) {
            if (++t >= m.t1) {
                u = first_tile(u + 1, m);
                t = u < u_end ? m.t0 : 0;
                ++ordinal;
            }
        };
        // Row list entries of tile t for this lane (< 0: masked).
        auto fetch_rows = [&](const Item &m, int t, int (&rv)[kGroupsPerWarp]) {
#pragma unroll
            for (int k = 0; k < kGroupsPerWarp; ++k) {
                const int g = gw + k * kGatherWarps;
                const int r = 4 * g + rsub;
                if (g >= kRowGroups) {
                    rv[k] = -1;
                    continue;
                }
                if (t < m.ct) {
                    // no idx: the row list is 0 .. count-1 (dense attention)
                    const int jj = t * TR + r;
                    rv[k] = jj < m.cnt ? (a.idx ? __ldg(a.idx + static_cast<long long>(m.ru) * a.top_k + jj) : jj) : -1;
                } else {
                    const int jj = (t - m.ct) * TR + r;
                    rv[k] = jj < m.nrw ? jj : -1;
                }
            }
        };
        auto row_index = [&](const Item &m, int t, int v) -> int {
            if (t < m.ct) return (v < 0 || v >= a.N_cap) ? -1 : static_cast<int>(m.comp_row0 + v);
            return v < 0 ? -1 : static_cast<int>(m.raw_row0 + v);
        };
        // Dense row lists: the next whole tile of compressed rows goes into L2
        // ahead with one bulk prefetch, so that its TMA copy, issued once its
        // buffer is free, reads L2 (dense attention 1.10 -> 1.03 ms).  Gathered
        // tiles are not prefetched: per-row prefetches slow the gathers down,
        // and so did prefetching the raw-window tiles of a gathered unit.
        auto prefetch_next = [&](int u, int t, const Item &m) {
            if (u >= u_end || a.idx || a.rows8 || t >= m.ct) return;
            const int nfirst = t * TR;
            if (a.tma_rows && nfirst + TR <= m.cnt && gw == 0 && lane == 0)
                prefetch_l2(a.rows + (m.comp_row0 + nfirst) * kHeadDim, TR * kHeadDim * 2);
        };
        auto nibble = [](uint32_t bal) -> uint32_t {   // lanes 0, 8, 16, 24 -> bits 0..3
            return (bal & 1u) | ((bal >> 7) & 2u) | ((bal >> 14) & 4u) | ((bal >> 21) & 8u);
        };
        Item cm;
        int cit = first_tile(0, cm);
        int ct_ = cit < u_end ? cm.t0 : 0;
        uint32_t jt = 0;
        int rv[kGroupsPerWarp];
        if (cit < u_end) fetch_rows(cm, ct_, rv);
        while (ok && cit < u_end) {
            if (ct_ == cm.t0 && gw == 0) {
                // First tile of an item: q (bf16) by TMA once the previous item's
                // logits are done and every softmax warp has passed its q wait.
                // q_free completes once per item, so item k waits for phase k-1.
                if (ordinal > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait(q_free, (ordinal - 1) & 1, abort_flag));
                    if (!ok) break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(q_full, 8 * kQBlk);
                    for (int b = 0; b < 8; ++b)
                        tma_load_2d_nohint(sQ + b * kQBlk, &a.tm_q, q_full, b * 64, cm.unit * kNHead);
                }
            }
            int src[kGroupsPerWarp];
            bool bad_idx = false;
            const uint16_t *base = (ct_ < cm.ct ? a.rows : a.raw) + chunk * 8;
#pragma unroll
            for (int k = 0; k < kGroupsPerWarp; ++k) {
                const int g = gw + k * kGatherWarps;
                src[k] = g < kRowGroups ? row_index(cm, ct_, rv[k]) : -1;
                // A listed row whose index lies outside [0, N_cap) is masked and flagged.
                if (g < kRowGroups && ct_ < cm.ct && ct_ * TR + 4 * g + rsub < cm.cnt && src[k] < 0) bad_idx = true;
            }
            if (__any_sync(0xffffffffu, bad_idx) && lane == 0) report(a.status, DS4A_DEV_BOUNDS);
            // FP8 rows go to registers before their buffer is free, so that the
            // loads overlap the wait for the values GEMM two tiles back; bf16
            // rows are copied by cp.async once the buffer is free, and a whole
            // tile of contiguous rows (the raw window, or a dense row list) by
            // TMA (rows past the valid count must be zeros, so a partial tile is
            // gathered).
            const bool raw_tile = ct_ >= cm.ct;
            const int first = raw_tile ? (ct_ - cm.ct) * TR : ct_ * TR;
            const bool fp8_tile = !raw_tile && a.rows8 != nullptr;
            const bool tma_tile = !fp8_tile && (raw_tile ? (a.tma_raw && first + TR <= cm.nrw)
                                                         : (a.tma_rows && !a.idx && first + TR <= cm.cnt));
            // Lane l: codes 16l .. 16l+15 of each row of its groups, and the
            // rows' scales.
            uint4 rg[kGroupsPerWarp][4];
            float s8[kGroupsPerWarp][4];
            if (fp8_tile) {
#pragma unroll
                for (int k = 0; k < kGroupsPerWarp; ++k) {
                    const int g = gw + k * kGatherWarps;
                    if (g >= kRowGroups) continue;       // warp-uniform
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int sr = __shfl_sync(0xffffffffu, src[k], 8 * i);   // row 4g + i (lanes 8i.. hold it)
                        if (sr >= 0) {
                            rg[k][i] = ld_nc_v4(reinterpret_cast<const uint4 *>(a.rows8 + static_cast<long long>(sr) * kHeadDim) + lane);
                            s8[k][i] = __ldg(a.row_scale + sr);
                        } else {
                            rg[k][i] = make_uint4(0u, 0u, 0u, 0u);
                            s8[k][i] = 0.f;
                        }
                    }
                }
            }
            // The row list of the next tile: before the wait, except for a
            // cp.async tile, where it goes out right after the copies.
            const long long y_tma = (raw_tile ? cm.raw_row0 : cm.comp_row0) + first;
            const bool early_next = fp8_tile || tma_tile;
            if (early_next) {
                advance(cit, ct_, cm);
                if (cit < u_end) fetch_rows(cm, ct_, rv);
                prefetch_next(cit, ct_, cm);
            }
            const int xb = jt & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&x_empty[xb], xeph[xb] ^ 1, abort_flag));
            if (!ok) break;
            xeph[xb] ^= 1;
            // validity bits first: a warp's barrier arrival publishes them
#pragma unroll
            for (int k = 0; k < kGroupsPerWarp; ++k) {
                const int g = gw + k * kGatherWarps;
                const uint32_t bal = __ballot_sync(0xffffffffu, src[k] >= 0);
                if (lane == 0 && g < kRowGroups) sValid[xb * kRowGroups + g] = static_cast<uint8_t>(nibble(bal));
            }
            const uint32_t buf = smem_u32(sX) + xb * kXBuf;
            if (tma_tile && gw == 0 && lane == 0) {
                const int y = static_cast<int>(y_tma);
                mbar_arrive_expect_tx(&x_full[xb], kXBuf);      // also this warp's arrival
                for (int b = 0; b < 8; ++b)
                    tma_load_2d_nohint(sX + xb * kXBuf + b * kXBlk, raw_tile ? &a.tm_raw : &a.tm_rows, &x_full[xb], b * 64, y);
            }
            if (fp8_tile) {
                // dims 16l .. 16l+15 are 16-byte chunks 2(l%4) and 2(l%4)+1 of the
                // 64-column block l/4.  Lanes of odd blocks write their second
                // chunk first, so the eight lanes of a store phase hit eight
                // different 16-byte bank groups.
                const int blk = lane >> 2, c0 = 2 * (lane & 3), odd = blk & 1;
#pragma unroll
                for (int k = 0; k < kGroupsPerWarp; ++k) {
                    const int g = gw + k * kGatherWarps;
                    if (g >= kRowGroups) continue;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = 4 * g + i;
                        uint32_t lo[4], hi[4];
                        e4m3x8_to_bf16(rg[k][i].x, rg[k][i].y, s8[k][i], lo);
                        e4m3x8_to_bf16(rg[k][i].z, rg[k][i].w, s8[k][i], hi);
                        const uint32_t rowa = buf + blk * kXBlk + r * 128;
                        const uint32_t a0 = rowa + ((c0 ^ (r & 7)) << 4), a1 = rowa + (((c0 + 1) ^ (r & 7)) << 4);
                        if (odd) {
                            st_shared_v4(a1, hi);
                            st_shared_v4(a0, lo);
                        } else {
                            st_shared_v4(a0, lo);
                            st_shared_v4(a1, hi);
                        }
                    }
                }
            } else if (!tma_tile) {
                // 16-byte cp.async into the 128B-swizzled layout: lane l copies
                // chunk (l & 7) of row 4k' + (l >> 3) of each of its groups in
                // every 64-column block, so a warp instruction moves four whole
                // 128-byte row segments.  Masked rows are zero-filled.
#pragma unroll
                for (int b = 0; b < 8; ++b) {
#pragma unroll
                    for (int k = 0; k < kGroupsPerWarp; ++k) {
                        const int g = gw + k * kGatherWarps;
                        if (g >= kRowGroups) continue;
                        const int r = 4 * g + rsub;
                        cp_async16(buf + b * kXBlk + r * 128 + ((chunk ^ (r & 7)) << 4),
                                   src[k] >= 0 ? base + static_cast<long long>(src[k]) * kHeadDim + b * 64 : a.q,
                                   src[k] >= 0 ? 16u : 0u);
                    }
                }
                cp_async_commit();
                advance(cit, ct_, cm);
                if (cit < u_end) fetch_rows(cm, ct_, rv);
                prefetch_next(cit, ct_, cm);
                cp_async_wait<0>();
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0 && !(tma_tile && gw == 0)) mbar_arrive(&x_full[xb]);
            ++jt;
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) report(a.status, DS4A_DEV_TIMEOUT);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ logits issuer
        // S(t) once the row tile has landed and the softmax has read the
        // logits two tiles back; the first raw tile also waits for q in fp16.
        uint32_t qph = 0, q16ph = 0;
        uint32_t xfph[2] = {0, 0}, seph[2] = {0, 0};
        bool ok = true;
        constexpr uint32_t id_s_bf = idesc_f16(false, false), id_s_f16 = idesc_f16(true, false);
        const uint64_t dq = sw128_desc(smem_u32(sQ), 16, 1024), dx0 = sw128_desc(smem_u32(sX), 16, 1024);
        uint32_t js = 0;                                     // tile counter: buffers js & 1
        for (int i = 0; ok && i < sc.n_pieces; ++i) {
            const Item m = make_piece(a, sc, i);
            if (m.t0 >= m.t1) continue;
            if (!(ok = warp_wait(q_full, qph, abort_flag))) break;
            qph ^= 1;
            bool q16 = false;
            for (int t = m.t0; t < m.t1; ++t, ++js) {
                const bool raw = t >= m.ct;
                const int b = js & 1;
                if (raw && !q16) {
                    if (!(ok = warp_wait(q16_ready, q16ph, abort_flag))) break;
                    q16ph ^= 1;
                    q16 = true;
                }
                if (!(ok = warp_wait(&s_empty[b], seph[b] ^ 1, abort_flag))) break;
                seph[b] ^= 1;
                if (!(ok = warp_wait(&x_full[b], xfph[b], abort_flag))) break;
                xfph[b] ^= 1;
                tc_fence_after();
                const uint64_t dx = dx0 + static_cast<uint64_t>(b * (kXBuf >> 4));
#pragma unroll
                for (int blk = 0; blk < 8; ++blk) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_elect(tmem + kTmemS + b * TR, dq + static_cast<uint64_t>(blk * (kQBlk >> 4) + 2 * kk),
                                   dx + static_cast<uint64_t>(blk * (kXBlk >> 4) + 2 * kk), raw ? id_s_f16 : id_s_bf,
                                   (blk | kk) ? 1u : 0u);
                }
                commit_elect(&s_full[b]);
                if (t == m.t1 - 1) commit_elect(q_free);
            }
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) report(a.status, DS4A_DEV_TIMEOUT);
        }
        commit_elect(drain);
        wait_drain(drain, 0);
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------ values issuer
        // V(t) once the softmax has written P(t) (and rescaled O when a head's
        // max was raised); the first tile of an item also waits until the
        // epilogue has read the previous item's O.  Its commit frees the row
        // tile and the P buffer.
        uint32_t ofph = 0, pfph[2] = {0, 0};
        bool ok = true, first_item = true;
        constexpr uint32_t id_v_bf = idesc_f16(false, true), id_v_f16 = idesc_f16(true, true);
        const uint64_t dxv = sw128_desc(smem_u32(sX), kXBlk, 1024), dp = sw128_desc(smem_u32(sP), 16, 1024);
        uint32_t jv = 0;
        for (int i = 0; ok && i < sc.n_pieces; ++i) {
            const Item m = make_piece(a, sc, i);
            if (m.t0 >= m.t1) continue;
            for (int t = m.t0; t < m.t1; ++t, ++jv) {
                const int b = jv & 1;
                if (!(ok = warp_wait(&p_full[b], pfph[b], abort_flag))) break;
                pfph[b] ^= 1;
                if (t == m.t0 && !first_item) {
                    if (!(ok = warp_wait(o_free, ofph, abort_flag))) break;
                    ofph ^= 1;
                }
                tc_fence_after();
                const bool raw = t >= m.ct;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int ks = 0; ks < TR / 16; ++ks)
                        umma_elect(tmem + kTmemO + c * kNHead,
                                   dxv + static_cast<uint64_t>((b * kXBuf + 2 * c * kXBlk + ks * 2048) >> 4),
                                   dp + static_cast<uint64_t>((b * kPBuf + ks * 32) >> 4), raw ? id_v_f16 : id_v_bf,
                                   (t == m.t0 && ks == 0) ? 0u : 1u);
                }
                commit_elect(&x_empty[b]);               // row tile and P buffer free
            }
            if (!ok) break;
            first_item = false;
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) report(a.status, DS4A_DEV_TIMEOUT);
        }
        commit_elect(drain_v);
        wait_drain(drain_v, 0);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        // Warp w = TMEM lane quarter w.  Logits (16x256b loads): thread t holds
        // heads h0 = 16w + t/4 and h1 = h0 + 8 for tile rows 8j + 2(t%4) + {0,1},
        // j = 0..7 (registers 4j, 4j+1: h0; 4j+2, 4j+3: h1).  Values: lane = dim.
        const int q4 = warp;
        const int t4 = lane & 3;
        const int h0 = 16 * q4 + (lane >> 2), h1 = h0 + 8;
        const int e = threadIdx.x;                      // 0..127 inside the softmax group
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        const float sl2 = a.scale * 1.4426950408889634f;
        uint32_t qph = 0, gph = 0, sfph[2] = {0, 0};
        uint32_t jt = 0;
        bool ok = true;
        // Barrier of the softmax warps on an mbarrier, so that a wait that gives
        // up (abort) cannot leave the other warps stuck.
        auto group_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(grp);
            const bool r = __all_sync(0xffffffffu, mbar_wait(grp, gph, abort_flag));
            gph ^= 1;
            return r;
        };
        auto convert_q = [&]() {
            // q -> fp16 in place for the fp16 raw tier (no logit GEMM reads q now).
            uint4 *qv = reinterpret_cast<uint4 *>(sQ);
            for (int k = e; k < 8 * kQBlk / 16; k += kSoftmaxWarps * 32) {
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
        };
        for (int i = 0; ok && i < sc.n_pieces; ++i) {
            const Item m = make_piece(a, sc, i);
            if (m.t0 >= m.t1) {
                // Empty row set: out = 0, lse = -inf (or an empty partial).
                if (!m.split) {
                    float *o = a.out + static_cast<long long>(m.unit) * kNHead * kHeadDim;
                    for (int k = e; k < kNHead * kHeadDim; k += kSoftmaxWarps * 32) o[k] = 0.f;
                    if (a.lse && e < kNHead) a.lse[static_cast<long long>(m.unit) * kNHead + e] = NEG_INF;
                } else if (e < kNHead) {
                    float *ml = static_cast<float *>(a.ws) + n_slots * kNHead * kHeadDim;
                    ml[(m.slot * kNHead + e) * 2] = NEG_INF;
                    ml[(m.slot * kNHead + e) * 2 + 1] = 0.f;
                }
                continue;
            }
            ok = __all_sync(0xffffffffu, mbar_wait(q_full, qph, abort_flag));
            if (!ok) break;
            qph ^= 1;
            float M0 = NEG_INF, M1 = NEG_INF, l0 = 0.f, l1 = 0.f;   // running max (log2 units) and partial sums
            bool q16 = false;
            if (m.t0 >= m.ct) {                          // the item starts with a raw tile
                convert_q();
                q16 = true;
            }
            // The next item's q may overwrite this one only after every softmax
            // warp has seen this one land: q_full must never run two phases
            // ahead of a warp's wait (its parity could not tell them apart),
            // which one-tile items allowed when q_free counted only the logits
            // GEMMs.
            __syncwarp();
            if (lane == 0) mbar_arrive(q_free);
            for (int t = m.t0; ok && t < m.t1; ++t, ++jt) {
                const bool raw = t >= m.ct;
                const int b = jt & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(&s_full[b], sfph[b], abort_flag));
                if (!ok) break;
                sfph[b] ^= 1;
                // The next tile is the first raw one: its logits need q in fp16,
                // and every compressed logit GEMM has completed (this one too).
                if (!q16 && t + 1 < m.t1 && t + 1 >= m.ct) {
                    convert_q();
                    q16 = true;
                }
                tc_fence_after();
                uint32_t r[32];
                tmem_ld16x256_x8(tmem + lane_off + kTmemS + b * TR, r);
                tmem_wait_ld(r);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[b]);
                // Row validity of this tile (written by the gather before x_full).
                ok = __all_sync(0xffffffffu, mbar_wait(&x_full[b], (jt >> 1) & 1, abort_flag));
                if (!ok) break;
                // rows 8j + 2(t%4) + {0,1}: group 2j + (t%4)/2, bits 2(t%4 & 1) + {0,1}
                const uint4 vw = *reinterpret_cast<const uint4 *>(sValid + b * kRowGroups);
                // A tile whose rows are all listed, with a positive scale, keeps the
                // raw logits: the max is taken before scaling and p = 2^(s*c - M)
                // is one FMA and one ex2.  Otherwise masked rows are -inf and the
                // logits are scaled first (c = 1 below).
                const bool full = (vw.x & vw.y & vw.z & vw.w) == 0x0F0F0F0Fu && sl2 > 0.f;
                const float mul = full ? sl2 : 1.f;
                float x[32];
                if (full) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
                } else {
                    const uint32_t vsh = 8 * (t4 >> 1) + 2 * (t4 & 1);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t w = (j < 2 ? vw.x : j < 4 ? vw.y : j < 6 ? vw.z : vw.w) >> (16 * (j & 1) + vsh);
                        const bool va = w & 1u, vb = (w >> 1) & 1u;
                        x[4 * j] = va ? __uint_as_float(r[4 * j]) * sl2 : NEG_INF;
                        x[4 * j + 1] = vb ? __uint_as_float(r[4 * j + 1]) * sl2 : NEG_INF;
                        x[4 * j + 2] = va ? __uint_as_float(r[4 * j + 2]) * sl2 : NEG_INF;
                        x[4 * j + 3] = vb ? __uint_as_float(r[4 * j + 3]) * sl2 : NEG_INF;
                    }
                }
                float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    mx0 = fmaxf(mx0, fmaxf(x[4 * j], x[4 * j + 1]));
                    mx1 = fmaxf(mx1, fmaxf(x[4 * j + 2], x[4 * j + 3]));
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                mx0 *= mul;
                mx1 *= mul;
                // The running max is raised only when the tile exceeds it by more than 2^8.
                float al0 = 1.f, al1 = 1.f;
                if (M0 == NEG_INF) {
                    M0 = mx0;                            // first finite max: O and sums are still 0
                } else if (mx0 > M0 + kRescaleThreshold) {
                    al0 = ex2(M0 - mx0);
                    M0 = mx0;
                }
                if (M1 == NEG_INF) {
                    M1 = mx1;
                } else if (mx1 > M1 + kRescaleThreshold) {
                    al1 = ex2(M1 - mx1);
                    M1 = mx1;
                }
                // Any head raised in any warp: every warp rescales its O^T lanes.
                const int tb = jt & 1;
                const bool wresc = __any_sync(0xffffffffu, (al0 != 1.f) | (al1 != 1.f));
                if (t4 == 0) {
                    sAlpha[tb * kNHead + h0] = al0;
                    sAlpha[tb * kNHead + h1] = al1;
                }
                if (lane == 0) sFlag[tb * kSoftmaxWarps + q4] = wresc ? 1u : 0u;
                // Arrive now, wait after the exponentials: the exchange of the
                // rescale flags overlaps this warp's own work.
                __syncwarp();
                if (lane == 0) mbar_arrive(grp);
                const float nr0 = M0 == NEG_INF ? 0.f : -M0, nr1 = M1 == NEG_INF ? 0.f : -M1;
                float s0 = 0.f, s1 = 0.f;
                uint32_t pk0[8], pk1[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float pa = ex2(fmaf(x[4 * j], mul, nr0)), pb = ex2(fmaf(x[4 * j + 1], mul, nr0));
                    const float pc = ex2(fmaf(x[4 * j + 2], mul, nr1)), pd = ex2(fmaf(x[4 * j + 3], mul, nr1));
                    s0 += pa + pb;
                    s1 += pc + pd;
                    pk0[j] = raw ? pack2<true>(pa, pb) : pack2<false>(pa, pb);
                    pk1[j] = raw ? pack2<true>(pc, pd) : pack2<false>(pc, pd);
                }
                l0 = l0 * al0 + s0;
                l1 = l1 * al1 + s1;
                // P[h][row]: rows 8j + 2(t%4) + {0,1} are bytes 16j + 4(t%4) of the
                // 128-byte row of head h, 16-byte chunk j swizzled with h & 7.
                uint8_t *pbuf = sP + b * kPBuf;
                const int sw = h0 & 7;                   // == h1 & 7
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    *reinterpret_cast<uint32_t *>(pbuf + h0 * 128 + ((j ^ sw) << 4) + 4 * t4) = pk0[j];
                    *reinterpret_cast<uint32_t *>(pbuf + h1 * 128 + ((j ^ sw) << 4) + 4 * t4) = pk1[j];
                }
                fence_proxy_async();
                {
                    const bool r = __all_sync(0xffffffffu, mbar_wait(grp, gph, abort_flag));
                    gph ^= 1;
                    ok = r;
                    if (!ok) break;
                }
                const uint4 fl = *reinterpret_cast<const uint4 *>(sFlag + tb * kSoftmaxWarps);
                const bool any_resc = (fl.x | fl.y | fl.z | fl.w) != 0u;
                if (any_resc && t > m.t0) {
                    // O^T holds the sum up to the previous values GEMM (tile jt - 1): wait for it.
                    ok = __all_sync(0xffffffffu, mbar_wait(&x_empty[(jt - 1) & 1], ((jt - 1) >> 1) & 1, abort_flag));
                    if (!ok) break;
                    tc_fence_after();
                    for (int c = 0; c < 8; ++c) {
                        uint32_t v[32];
                        const uint32_t ta = tmem + lane_off + kTmemO + c * 32;
                        tmem_ld32(ta, v);
                        tmem_wait_ld(v);
                        const float *al = sAlpha + tb * kNHead + (c & 1) * 32;
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * al[k]);
                        tmem_st32(ta, v);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[b]);
            }
            if (!ok) break;
            // ---- epilogue: row sums over the four threads of a head, then O^T out
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            const long long slot = m.slot;
            if (t4 == 0) {
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int h = k ? h1 : h0;
                    const float L = k ? l1 : l0, M = k ? M1 : M0;
                    if (!m.split) {
                        sInvL[h] = L > 0.f ? 1.f / L : 0.f;
                        if (a.lse)
                            a.lse[static_cast<long long>(m.unit) * kNHead + h] =
                                L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : NEG_INF;
                    } else {
                        sInvL[h] = 1.f;
                        float *ml = static_cast<float *>(a.ws) + n_slots * kNHead * kHeadDim;
                        ml[(slot * kNHead + h) * 2] = L > 0.f ? M : NEG_INF;
                        ml[(slot * kNHead + h) * 2 + 1] = L;
                    }
                }
            }
            if (!(ok = group_sync())) break;
            // the item's last values GEMM (tile jt - 1)
            ok = __all_sync(0xffffffffu, mbar_wait(&x_empty[(jt - 1) & 1], ((jt - 1) >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            float *obase = !m.split ? a.out + static_cast<long long>(m.unit) * kNHead * kHeadDim
                                        : static_cast<float *>(a.ws) + slot * kNHead * kHeadDim;
            // 1/l of the 64 heads in registers: no shared load between the
            // global stores below.
            float il[kNHead];
#pragma unroll
            for (int h = 0; h < kNHead; ++h) il[h] = sInvL[h];
            for (int c = 0; c < 8; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_off + kTmemO + c * 32, v);
                tmem_wait_ld(v);
                const int d = (c >> 1) * 128 + q4 * 32 + lane;
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int h = (c & 1) * 32 + k;
                    obase[static_cast<long long>(h) * kHeadDim + d] = __uint_as_float(v[k]) * ((c & 1) ? il[32 + k] : il[k]);
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
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

constexpr int kMergeMaxPieces = 128;   // one per thread of the merge block; a unit has at most kMaxTopK / 64 + 2 tiles
static_assert((kMaxTopK + TR - 1) / TR + (kNSwa + TR - 1) / TR <= kMergeMaxPieces, "merge: one thread per piece");

// Combines the pieces of the remainder units that straddle a share boundary.
// Block (v, h): head h of remainder unit v, whose tiles [v nt, (v+1) nt) of the
// remainder tile space lie in the shares of CTAs c0 .. c1 (share c: tiles
// [c T / g, (c+1) T / g)); a unit inside one share was written directly.
// O = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k, lse = (M + log2 L) ln 2.
__global__ void __launch_bounds__(128) attn_merge_kernel(const __grid_constant__ AttnArgs a, int nt, int g_rem, int G) {
    pdl_launch_dependents();
    pdl_wait();
    const int v = blockIdx.x / kNHead;
    const int h = blockIdx.x - v * kNHead;
    const long long u_rem0 = static_cast<long long>(a.units / G) * G;
    const long long T = (a.units - u_rem0) * nt;
    const long long vs = static_cast<long long>(v) * nt, ve = vs + nt;
    auto share_of = [&](long long x) -> int { return static_cast<int>(((x + 1) * g_rem - 1) / T); };
    const int c0 = share_of(vs), c1 = share_of(ve - 1);
    if (c0 == c1) return;                                   // whole inside one share
    const float *wo = static_cast<const float *>(a.ws);
    const float *ml = wo + 2LL * G * kNHead * kHeadDim;    // (m, l) after the 2 G O slots
    // Share c0 holds the unit's start: its first piece (slot 0) when the share
    // starts exactly there, else its last (slot 1); later shares: their first.
    auto piece_slot = [&](int c) -> long long {
        return c == c0 ? 2LL * c + (static_cast<long long>(c) * T / g_rem == vs ? 0 : 1) : 2LL * c;
    };
    const float NEG_INF = -__int_as_float(0x7f800000);
    // One round trip for the first kEarly pieces: thread i < np loads piece
    // i's (m, l) and every thread its four dims of those pieces' O rows, all in
    // flight together; pieces past kEarly (top_k > 896) then load eight at a
    // time.  The sums run in piece order, as a sequential loop would.
    constexpr int kEarly = 16;
    __shared__ float s_w[kMergeMaxPieces], s_l[kMergeMaxPieces];
    __shared__ float s_max[4];
    const int np = c1 - c0 + 1;                              // <= tiles per unit <= kMergeMaxPieces
    const int d = threadIdx.x * 4;
    float4 oe[kEarly];
#pragma unroll
    for (int j = 0; j < kEarly; ++j)
        oe[j] = j < np ? *reinterpret_cast<const float4 *>(wo + (piece_slot(c0 + j) * kNHead + h) * kHeadDim + d)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    float mk = NEG_INF, lk = 0.f;
    if (threadIdx.x < np) {
        const float2 p = *reinterpret_cast<const float2 *>(ml + (piece_slot(c0 + threadIdx.x) * kNHead + h) * 2);
        if (p.y > 0.f) {
            mk = p.x;
            lk = p.y;
        }
    }
    float M = mk;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = M;
    __syncthreads();
    M = fmaxf(fmaxf(s_max[0], s_max[1]), fmaxf(s_max[2], s_max[3]));
    if (threadIdx.x < np) {
        s_w[threadIdx.x] = mk == NEG_INF ? 0.f : exp2f(mk - M);
        s_l[threadIdx.x] = lk;
    }
    __syncthreads();
    float L = 0.f;
    for (int i = 0; i < np; ++i) L += s_w[i] * s_l[i];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kEarly; ++j) {
        if (j >= np || s_w[j] == 0.f) continue;             // an empty piece's O was never written
        const float wk = s_w[j];
        acc.x += wk * oe[j].x;
        acc.y += wk * oe[j].y;
        acc.z += wk * oe[j].z;
        acc.w += wk * oe[j].w;
    }
    for (int i0 = kEarly; i0 < np; i0 += 8) {
        float4 o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = i0 + j;
            o[j] = (i < np && s_w[i] != 0.f)
                       ? *reinterpret_cast<const float4 *>(wo + (piece_slot(c0 + i) * kNHead + h) * kHeadDim + d)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = i0 + j;
            if (i >= np || s_w[i] == 0.f) continue;
            const float wk = s_w[i];
            acc.x += wk * o[j].x;
            acc.y += wk * o[j].y;
            acc.z += wk * o[j].z;
            acc.w += wk * o[j].w;
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    const long long u = u_rem0 + v;
    *reinterpret_cast<float4 *>(a.out + (u * kNHead + h) * kHeadDim + d) = acc;
    if (a.lse && threadIdx.x == 0)
        a.lse[u * kNHead + h] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : NEG_INF;
}

// Tiles per unit in the tile space: the top_k compressed rows and the raw window.
int attn_tiles_per_unit(int top_k) { return (top_k + TR - 1) / TR + (kNSwa + TR - 1) / TR; }

}  // namespace

size_t attn_ws_bytes(int units, int top_k) {
    // Two partial slots per CTA; the grid never exceeds kMaxAttnCtas.
    const long long T = static_cast<long long>(units) * attn_tiles_per_unit(top_k);
    const long long G = T < kMaxAttnCtas ? T : kMaxAttnCtas;
    if (G <= 1) return 0;                                   // one CTA: every unit whole
    return static_cast<size_t>(2 * G) * kNHead * (kHeadDim + 2) * sizeof(float);
}

cudaError_t launch_sparse_attn(const AttnArgs &a, int num_sms, cudaStream_t s) {
    const int gw = (a.idx == nullptr && a.rows8 == nullptr) ? kGatherWarpsDense : kGatherWarpsList;
    void (*kern)(AttnArgs, int, int) =
        gw == kGatherWarpsDense ? sparse_attn_kernel<kGatherWarpsDense> : sparse_attn_kernel<kGatherWarpsList>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int nt = attn_tiles_per_unit(a.top_k);
    const long long T = static_cast<long long>(a.units) * nt;
    if (T <= 0) return cudaSuccess;
    long long G = num_sms < kMaxAttnCtas ? num_sms : kMaxAttnCtas;
    if (T < G) G = T;
    // Remainder units (after the whole rounds) in one-tile-or-larger shares
    // over up to G CTAs.
    const long long u_rem = a.units - (a.units / G) * G;
    const long long t_rem = u_rem * nt;
    const int g_rem = static_cast<int>(t_rem < G ? t_rem : G);
    e = launch_k(kern, dim3(static_cast<unsigned>(G)), dim3(attn_threads(gw)), kSmemBytes, s, a, nt, g_rem);
    if (e != cudaSuccess || g_rem <= 1) return e;
    return launch_k(attn_merge_kernel, dim3(static_cast<unsigned>(u_rem * kNHead)), dim3(128), 0, s, a, nt, g_rem,
                    static_cast<int>(G));
}

}  // namespace ds4a
