// Sparse attention over the selected compressed rows and the raw window
// ("DwarfStar(ds4.c) のアーキテクチャを読む" §3: three tiers; §2: 64 query
// heads, one KV head whose 512-d rows are both key and value; §3-1: the raw
// window of the last 128 tokens is kept rounded to f16).
//
// One CTA handles one unit (a decode query, or one query of a prefill chunk),
// or one split of its row list when units are too few to fill the GPU.  The
// unit's row list is [selected compressed rows..., raw-window rows...] cut
// into 64-row tiles.  Per tile:
//   - gather: 64 rows x 1 KiB copied by cp.async (16 B per thread-op, 512 B
//     contiguous per warp) into an XOR-swizzled shared tile, double-buffered
//     so the next tile's gather overlaps this tile's math;
//   - S = q . x^T on the tensor cores (mma.sync m16n8k16, fp32 accumulate):
//     8 warps = 4 head groups x 2 halves of the 512 dims; the two halves'
//     partial logits are added through shared memory;
//   - online softmax in fp32 (exp2 domain), one joint softmax over all tiers;
//   - O += P . x on the tensor cores, P rounded to the tile's input type.
// Compressed rows are bf16; raw rows are fp16 and are multiplied in fp16, with
// q converted in place to fp16 (exact for |q| in [2^-14, 65504]).
// Split CTAs write unnormalised partials (O, m, l) that a merge kernel
// combines by their log-sum-exp.
#include "common.cuh"
#include "internal.h"

namespace ds4a {
namespace {

constexpr int kTile = 64;
constexpr int kThreads = 256;
constexpr int kRowBytes = kHeadDim * 2;                 // 1 KiB
constexpr int kTileBytes = kTile * kRowBytes;           // 64 KiB
constexpr int kOffQ = 0;
constexpr int kOffX = kOffQ + kNHead * kRowBytes;      // Q: 64 heads x 1 KiB
constexpr int kOffS = kOffX + 2 * kTileBytes;          // partial-logit exchange
constexpr int kOffValid = kOffS + 8 * 32 * 32 * 4;
constexpr int kSmemBytes = kOffValid + 2 * kTile;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr int kMaxSplit = 16;

// Byte offset of 16-byte chunk c (0..63) of row r in a [rows][512] 16-bit tile.
DS4A_DEV uint32_t swz(int r, int c) { return static_cast<uint32_t>(r * kRowBytes + ((c ^ (r & 7)) << 4)); }

DS4A_DEV void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

struct UnitRows {
    int cnt;            // selected compressed rows
    int nrw;            // raw rows
    const uint16_t *comp;
    const int32_t *idx;
    const uint16_t *raw;   // first raw row of this unit's window
};

DS4A_DEV UnitRows unit_rows(const AttnArgs &a, int unit, bool report_bounds) {
    UnitRows r;
    int cnt = a.count[unit];
    if (cnt < 0 || cnt > a.top_k) {
        if (report_bounds) report(a.status, DS4A_DEV_BOUNDS);
        cnt = cnt < 0 ? 0 : a.top_k;
    }
    r.cnt = cnt;
    r.comp = a.rows + static_cast<long long>(unit) * a.rows_unit_stride;
    r.idx = a.idx + static_cast<long long>(unit) * a.top_k;
    if (a.q_pos) {
        const int p = a.q_pos[unit];
        const long long lo = max(static_cast<long long>(p) - (kNSwa - 1) - a.raw_pos0, 0LL);
        const long long hi = min(static_cast<long long>(p) - a.raw_pos0, static_cast<long long>(a.n_raw_rows) - 1);
        r.nrw = hi >= lo ? static_cast<int>(hi - lo + 1) : 0;
        r.raw = a.raw + (r.nrw ? lo : 0) * kHeadDim;
    } else {
        int n = a.n_raw[unit];
        if (n < 0 || n > kNSwa) {
            if (report_bounds) report(a.status, DS4A_DEV_BOUNDS);
            n = n < 0 ? 0 : kNSwa;
        }
        r.nrw = n;
        r.raw = a.raw + static_cast<long long>(unit) * a.raw_unit_stride;
    }
    return r;
}

// Issues the cp.async gather of tile `ti` of the unit's row list into `dst`.
DS4A_DEV void gather_tile(const AttnArgs &a, const UnitRows &ur, int ct, int ti, uint8_t *dst, uint8_t *valid,
                          bool report_bounds) {
    const int c = threadIdx.x & 63;
    const uint32_t base = smem_u32(dst);
#pragma unroll 4
    for (int it = 0; it < kTile / 4; ++it) {
        const int r = it * 4 + (threadIdx.x >> 6);
        const uint16_t *src = a.q;   // any valid address when nothing is read
        bool ok;
        if (ti < ct) {
            const int j = ti * kTile + r;
            ok = j < ur.cnt;
            if (ok) {
                const int iv = __ldg(ur.idx + j);
                if (iv < 0 || iv >= a.N_cap) {
                    ok = false;
                    if (report_bounds && c == 0) report(a.status, DS4A_DEV_BOUNDS);
                } else {
                    src = ur.comp + static_cast<long long>(iv) * kHeadDim + c * 8;
                }
            }
        } else {
            const int j = (ti - ct) * kTile + r;
            ok = j < ur.nrw;
            if (ok) src = ur.raw + static_cast<long long>(j) * kHeadDim + c * 8;
        }
        cp_async16(base + swz(r, c), src, ok ? 16u : 0u);
        if (c == 0) valid[r] = ok ? 1 : 0;
    }
}

template <bool F16>
DS4A_DEV void tile_math(uint32_t sQ, uint32_t sX, const uint8_t *valid, float *sS, int warp, int lane, float sl2,
                        float (&O)[32][4], float &m0, float &m1, float &l0, float &l1) {
    const int hg = warp & 3, dh = warp >> 2;
    float S[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) S[i][0] = S[i][1] = S[i][2] = S[i][3] = 0.f;

    // ---- S (partial over this warp's 256 dims) = Q[16 heads] . X^T
#pragma unroll 2
    for (int kk = 0; kk < 16; ++kk) {
        const int kc = dh * 32 + kk * 2;
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sQ + swz(hg * 16 + (lane & 15), kc + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(sX + swz(np * 16 + (lane & 7) + ((lane >> 4) << 3), kc + ((lane >> 3) & 1)), b0, b1, b2, b3);
            mma_16816<F16>(S[2 * np], a0, a1, a2, a3, b0, b1);
            mma_16816<F16>(S[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
    }
    // ---- add the other dim-half's partial
    float *mine = sS + warp * 1024;
    const float *other = sS + (warp ^ 4) * 1024;
#pragma unroll
    for (int i = 0; i < 32; ++i) mine[i * 32 + lane] = S[i >> 2][i & 3];
    named_bar(1 + hg, 64);
#pragma unroll
    for (int i = 0; i < 32; ++i) S[i >> 2][i & 3] += other[i * 32 + lane];

    // ---- online softmax (log2 domain), rows g0 = lane/4 and g1 = g0 + 8
    const float NEG_INF = -__int_as_float(0x7f800000);
    float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int col = nt * 8 + 2 * (lane & 3) + (e & 1);
            const float x = valid[col] ? S[nt][e] * sl2 : NEG_INF;
            S[nt][e] = x;
            if (e < 2) mx0 = fmaxf(mx0, x); else mx1 = fmaxf(mx1, x);
        }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float base0 = mn0 == NEG_INF ? 0.f : mn0;
    const float base1 = mn1 == NEG_INF ? 0.f : mn1;
    const float al0 = exp2f(m0 - base0), al1 = exp2f(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        S[nt][0] = exp2f(S[nt][0] - base0);
        S[nt][1] = exp2f(S[nt][1] - base0);
        S[nt][2] = exp2f(S[nt][2] - base1);
        S[nt][3] = exp2f(S[nt][3] - base1);
        ps0 += S[nt][0] + S[nt][1];
        ps1 += S[nt][2] + S[nt][3];
    }
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        O[i][0] *= al0;
        O[i][1] *= al0;
        O[i][2] *= al1;
        O[i][3] *= al1;
    }

    // ---- O[16 heads x this warp's 256 dims] += P . X
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint32_t a0 = pack2<F16>(S[2 * kk][0], S[2 * kk][1]);
        const uint32_t a1 = pack2<F16>(S[2 * kk][2], S[2 * kk][3]);
        const uint32_t a2 = pack2<F16>(S[2 * kk + 1][0], S[2 * kk + 1][1]);
        const uint32_t a3 = pack2<F16>(S[2 * kk + 1][2], S[2 * kk + 1][3]);
        const int xr = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int dp = 0; dp < 16; ++dp) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(sX + swz(xr, dh * 32 + dp * 2 + (lane >> 4)), b0, b1, b2, b3);
            mma_16816<F16>(O[2 * dp], a0, a1, a2, a3, b0, b1);
            mma_16816<F16>(O[2 * dp + 1], a0, a1, a2, a3, b2, b3);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) sparse_attn_kernel(const __grid_constant__ AttnArgs a, int n_split) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int unit = blockIdx.x / n_split;
    const int split = blockIdx.x - unit * n_split;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool first_split = split == 0;
    const UnitRows ur = unit_rows(a, unit, first_split && threadIdx.x == 0);
    const int ct = (ur.cnt + kTile - 1) / kTile;
    const int rt = (ur.nrw + kTile - 1) / kTile;
    const int nt = ct + rt;
    const int tps = (nt + n_split - 1) / n_split;
    const int t0 = split * tps;
    const int t1 = min(nt, t0 + tps);

    uint8_t *sQ = smem + kOffQ;
    uint8_t *sX = smem + kOffX;
    float *sS = reinterpret_cast<float *>(smem + kOffS);
    uint8_t *sValid = smem + kOffValid;
    const uint32_t sQa = smem_u32(sQ), sXa = smem_u32(sX);
    const float sl2 = a.scale * 1.4426950408889634f;   // exp(x) = exp2(x * log2 e)

    float O[32][4];
#pragma unroll
    for (int i = 0; i < 32; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
    const float NEG_INF = -__int_as_float(0x7f800000);
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;

    if (t0 < t1) {
        // Q (bf16) + first tile.
        const uint16_t *qu = a.q + static_cast<long long>(unit) * kNHead * kHeadDim;
        {
            const int c = threadIdx.x & 63;
#pragma unroll 4
            for (int it = 0; it < kNHead / 4; ++it) {
                const int r = it * 4 + (threadIdx.x >> 6);
                cp_async16(sQa + swz(r, c), qu + r * kHeadDim + c * 8, 16u);
            }
        }
        gather_tile(a, ur, ct, t0, sX, sValid, first_split);
        cp_async_commit();
        bool q_f16 = false;
        for (int ti = t0; ti < t1; ++ti) {
            const int buf = (ti - t0) & 1;
            if (ti + 1 < t1) {
                gather_tile(a, ur, ct, ti + 1, sX + (buf ^ 1) * kTileBytes, sValid + (buf ^ 1) * kTile,
                            first_split);
                cp_async_commit();
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const bool raw_tile = ti >= ct;
            if (raw_tile && !q_f16) {
                // q -> fp16 in place for the fp16 raw tier.
                uint4 *qv = reinterpret_cast<uint4 *>(sQ);
                for (int i = threadIdx.x; i < kNHead * kRowBytes / 16; i += kThreads) {
                    uint4 v = qv[i];
                    uint32_t *w = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float lo = __uint_as_float(w[j] << 16);
                        const float hi = __uint_as_float(w[j] & 0xffff0000u);
                        w[j] = pack2<true>(lo, hi);
                    }
                    qv[i] = v;
                }
                q_f16 = true;
                __syncthreads();
            }
            const uint32_t xa = sXa + buf * kTileBytes;
            const uint8_t *vb = sValid + buf * kTile;
            if (raw_tile)
                tile_math<true>(sQa, xa, vb, sS, warp, lane, sl2, O, m0, m1, l0, l1);
            else
                tile_math<false>(sQa, xa, vb, sS, warp, lane, sl2, O, m0, m1, l0, l1);
            __syncthreads();
        }
    }

    // Row sums across the quad.
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    const int hg = warp & 3, dh = warp >> 2;
    const int g0 = hg * 16 + (lane >> 2), g1 = g0 + 8;
    const int dbase = dh * 256 + 2 * (lane & 3);
    if (n_split == 1) {
        const float i0 = l0 > 0.f ? 1.f / l0 : 0.f;
        const float i1 = l1 > 0.f ? 1.f / l1 : 0.f;
        float *o0 = a.out + (static_cast<long long>(unit) * kNHead + g0) * kHeadDim + dbase;
        float *o1 = a.out + (static_cast<long long>(unit) * kNHead + g1) * kHeadDim + dbase;
#pragma unroll
        for (int nt = 0; nt < 32; ++nt) {
            *reinterpret_cast<float2 *>(o0 + nt * 8) = make_float2(O[nt][0] * i0, O[nt][1] * i0);
            *reinterpret_cast<float2 *>(o1 + nt * 8) = make_float2(O[nt][2] * i1, O[nt][3] * i1);
        }
        if (a.lse && dh == 0 && (lane & 3) == 0) {
            const float LN2 = 0.6931471805599453f;
            a.lse[static_cast<long long>(unit) * kNHead + g0] = l0 > 0.f ? (m0 + log2f(l0)) * LN2 : NEG_INF;
            a.lse[static_cast<long long>(unit) * kNHead + g1] = l1 > 0.f ? (m1 + log2f(l1)) * LN2 : NEG_INF;
        }
    } else {
        float *wo = static_cast<float *>(a.ws);
        const long long slot = static_cast<long long>(unit) * n_split + split;
        float *o0 = wo + (slot * kNHead + g0) * kHeadDim + dbase;
        float *o1 = wo + (slot * kNHead + g1) * kHeadDim + dbase;
#pragma unroll
        for (int nt = 0; nt < 32; ++nt) {
            *reinterpret_cast<float2 *>(o0 + nt * 8) = make_float2(O[nt][0], O[nt][1]);
            *reinterpret_cast<float2 *>(o1 + nt * 8) = make_float2(O[nt][2], O[nt][3]);
        }
        if (dh == 0 && (lane & 3) == 0) {
            float *ml = wo + static_cast<long long>(a.units) * n_split * kNHead * kHeadDim;
            *reinterpret_cast<float2 *>(ml + (slot * kNHead + g0) * 2) = make_float2(m0, l0);
            *reinterpret_cast<float2 *>(ml + (slot * kNHead + g1) * 2) = make_float2(m1, l1);
        }
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
    // Enough CTAs to cover 152 SMs about twice; at most one 64-row tile per split.
    const int max_tiles = (top_k + kTile - 1) / kTile + (kNSwa + kTile - 1) / kTile;
    if (units >= 152) return 1;
    int s = (2 * 152 + units - 1) / units;
    if (s > max_tiles) s = max_tiles;
    if (s > kMaxSplit) s = kMaxSplit;
    return s < 1 ? 1 : s;
}

size_t attn_ws_bytes(int units, int top_k) {
    const int s = attn_num_splits(units, top_k);
    if (s == 1) return 0;
    return static_cast<size_t>(units) * s * kNHead * (kHeadDim + 2) * sizeof(float);
}

cudaError_t launch_sparse_attn(const AttnArgs &a, cudaStream_t s) {
    const int n_split = attn_num_splits(a.units, a.top_k);
    cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long blocks = static_cast<long long>(a.units) * n_split;
    sparse_attn_kernel<<<static_cast<unsigned>(blocks), kThreads, kSmemBytes, s>>>(a, n_split);
    e = cudaGetLastError();
    if (e != cudaSuccess || n_split == 1) return e;
    attn_merge_kernel<<<static_cast<unsigned>(static_cast<long long>(a.units) * kNHead), 128, 0, s>>>(a, n_split);
    return cudaGetLastError();
}

}  // namespace ds4a
