// Producer side of the caches ("DwarfStar(ds4.c) のアーキテクチャを読む"):
//   §3-1  the raw window keeps the last 128 tokens' rows rounded through f16;
//   §3-2  the compressor pools a frontier of `ratio` rows (4 or 128) into one
//         compressed row with a per-column softmax of learned scores.
//   §3-2  the new compressed row goes through an FP8 quantisation round trip
//         before it is stored: here its stored form, E4M3 codes with one
//         power-of-two scale per row (the pages name no format or scaling;
//         this is the library's reading), which keeps exactly the values the
//         round trip produces.
// The projections that produce kv and scores, the positional bias and the
// normalisation / RoPE steps after pooling need trained weights and are not
// part of this library; these kernels take their inputs as given.
//
// The raw window here is a ring: the row of position p goes to slot p % 128,
// so the window holds the same rows as the pages' oldest-first window (which
// slides its rows down one slot when full), in rotated order; the attention
// does not depend on slot order.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace ds4a {
namespace {

constexpr int kPushThreads = kHeadDim / 4;   // one thread per 4 elements of the row

__global__ void __launch_bounds__(kPushThreads) kv_push_raw_kernel(const float *__restrict__ kv, uint16_t *raw,
                                                                   long long raw_unit_stride,
                                                                   const int32_t *__restrict__ pos, int32_t *n_raw,
                                                                   uint32_t *status) {
    pdl_launch_dependents();
    pdl_wait();
    const int u = blockIdx.x;
    const int p = pos[u];
    if (p < 0) {                                  // no position: nothing is written
        if (threadIdx.x == 0) report(status, DS4A_DEV_BOUNDS);
        return;
    }
    const int slot = p % kNSwa;
    const float4 v = reinterpret_cast<const float4 *>(kv + static_cast<long long>(u) * kHeadDim)[threadIdx.x];
    const __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);   // round to nearest even
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t *>(&lo);
    o.y = *reinterpret_cast<const uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(raw + static_cast<long long>(u) * raw_unit_stride +
                              static_cast<long long>(slot) * kHeadDim)[threadIdx.x] = o;
    if (threadIdx.x == 0) n_raw[u] = p + 1 < kNSwa ? p + 1 : kNSwa;
}

// Four threads pool 4 consecutive columns of one unit: thread q of the four
// takes the frontier rows r = q (mod 4), eight rows of loads in flight at a
// time; the running column max is raised per group of eight rows (the sums so
// far are rescaled by e^(old max - new max)), then the group's weights
// e^(s - max) are added.  The four partial (max, sum of weights, weighted sum)
// are combined by two shuffles.  A column with no finite score gives 0.
// Lane l of a warp: row quarter l / 8, column group 8 * (warp index) + l % 8,
// so a warp load covers four 128-byte row segments.
constexpr int kPoolThreads = 64;
constexpr int kPoolGroup = 8;
constexpr int kPoolSplit = 4;

__global__ void __launch_bounds__(kPoolThreads) compressor_pool_kernel(const float *__restrict__ kv,
                                                                       const float *__restrict__ score, int ratio,
                                                                       int width, float *__restrict__ out, int U) {
    pdl_launch_dependents();
    pdl_wait();
    const int w4 = width >> 2;
    const int lane = threadIdx.x & 31, q = lane >> 3;
    const long long warp_g = (static_cast<long long>(blockIdx.x) * kPoolThreads + threadIdx.x) >> 5;
    const long long g = warp_g * 8 + (lane & 7);                  // column group over all units
    const bool live = g < static_cast<long long>(U) * w4;
    const long long u = live ? g / w4 : 0;
    const int c = live ? static_cast<int>(g - u * w4) : 0;
    const float4 *s4 = reinterpret_cast<const float4 *>(score + u * ratio * width) + c;
    const float4 *k4 = reinterpret_cast<const float4 *>(kv + u * ratio * width) + c;
    const float NEG_INF = -__int_as_float(0x7f800000);
    float m[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
    float num[4] = {0.f, 0.f, 0.f, 0.f}, den[4] = {0.f, 0.f, 0.f, 0.f};
    for (int r0 = q; live && r0 < ratio; r0 += kPoolSplit * kPoolGroup) {
        float4 s[kPoolGroup], k[kPoolGroup];
#pragma unroll
        for (int i = 0; i < kPoolGroup; ++i) {
            const int r = r0 + kPoolSplit * i;
            if (r < ratio) {
                s[i] = __ldg(s4 + static_cast<long long>(r) * w4);
                k[i] = __ldg(k4 + static_cast<long long>(r) * w4);
            } else {
                s[i] = make_float4(NEG_INF, NEG_INF, NEG_INF, NEG_INF);
                k[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int col = 0; col < 4; ++col) {
            float sv[kPoolGroup], kvv[kPoolGroup];
#pragma unroll
            for (int i = 0; i < kPoolGroup; ++i) {
                sv[i] = col == 0 ? s[i].x : col == 1 ? s[i].y : col == 2 ? s[i].z : s[i].w;
                kvv[i] = col == 0 ? k[i].x : col == 1 ? k[i].y : col == 2 ? k[i].z : k[i].w;
            }
            float gm = sv[0];
#pragma unroll
            for (int i = 1; i < kPoolGroup; ++i) gm = fmaxf(gm, sv[i]);
            if (gm > m[col]) {
                const float a = m[col] > NEG_INF ? expf(m[col] - gm) : 0.f;
                num[col] *= a;
                den[col] *= a;
                m[col] = gm;
            }
            if (m[col] > NEG_INF) {
#pragma unroll
                for (int i = 0; i < kPoolGroup; ++i) {
                    const float e = expf(sv[i] - m[col]);
                    den[col] += e;
                    num[col] += e * kvv[i];
                }
            }
        }
    }
    // combine the four row quarters (lanes l, l ^ 8, l ^ 16, l ^ 24)
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
        for (int col = 0; col < 4; ++col) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m[col], off);
            const float n2 = __shfl_xor_sync(0xffffffffu, num[col], off);
            const float d2 = __shfl_xor_sync(0xffffffffu, den[col], off);
            const float M = fmaxf(m[col], m2);
            if (M > NEG_INF) {
                const float a = m[col] > NEG_INF ? expf(m[col] - M) : 0.f;
                const float b = m2 > NEG_INF ? expf(m2 - M) : 0.f;
                num[col] = num[col] * a + n2 * b;
                den[col] = den[col] * a + d2 * b;
                m[col] = M;
            }
        }
    }
    if (!live || q != 0) return;
    float4 o;
    o.x = den[0] > 0.f ? num[0] / den[0] : 0.f;
    o.y = den[1] > 0.f ? num[1] / den[1] : 0.f;
    o.z = den[2] > 0.f ? num[2] / den[2] : 0.f;
    o.w = den[3] > 0.f ? num[3] / den[3] : 0.f;
    reinterpret_cast<float4 *>(out + u * width)[c] = o;
}

// One warp per row of 512 fp32 values; lane l owns elements 16l .. 16l+15.
//   amax  = max |x| over the row (fmaxf skips NaN);
//   e     = the smallest integer with amax <= 448 * 2^e, within [-126, 127]
//           (0 when amax is 0 or infinite): with amax = m * 2^k, m in [0.5, 1),
//           e = k - 9 if m <= 0.875 (448 = 0.875 * 2^9), else k - 8;
//   codes = E4M3 of x * 2^-e, rounded to nearest even, saturating at 448
//           (the scaling by a power of two is exact).
constexpr int kFp8RowsPerBlock = 4;

DS4A_DEV int fp8_row_exponent(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int field = static_cast<int>(b >> 23);
    if (amax == 0.f || field >= 255) return 0;            // zero, infinity
    if (field == 0) return -126;                           // subnormal: below 448 * 2^-127
    const int k = field - 126;                             // amax = m * 2^k, m in [0.5, 1)
    int e = (b & 0x7FFFFFu) <= 0x600000u ? k - 9 : k - 8;  // m <= 0.875 <=> fraction <= 0.75 * 2^23
    return e < -126 ? -126 : (e > 127 ? 127 : e);
}

DS4A_DEV uint32_t e4m3x4(float a, float b, float c, float d) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));   // a -> low byte
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__global__ void __launch_bounds__(32 * kFp8RowsPerBlock) rows_to_fp8_kernel(const float *__restrict__ x,
                                                                          long long n_rows, uint8_t *codes,
                                                                          float *row_scale) {
    pdl_launch_dependents();
    pdl_wait();
    const long long row = static_cast<long long>(blockIdx.x) * kFp8RowsPerBlock + (threadIdx.x >> 5);
    if (row >= n_rows) return;
    const int lane = threadIdx.x & 31;
    const float4 *src = reinterpret_cast<const float4 *>(x + row * kHeadDim) + lane * 4;
    float4 v[4];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i] = src[i];
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = fp8_row_exponent(amax);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);   // 2^-e (e <= 126 for finite amax)
    uint4 out;
    uint32_t *o = reinterpret_cast<uint32_t *>(&out);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = e4m3x4(v[i].x * inv, v[i].y * inv, v[i].z * inv, v[i].w * inv);
    reinterpret_cast<uint4 *>(codes + row * kHeadDim)[lane] = out;
    if (lane == 0) row_scale[row] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}

}  // namespace

cudaError_t launch_rows_to_fp8(const float *x, long long n_rows, uint8_t *codes, float *row_scale, cudaStream_t s) {
    const long long blocks = (n_rows + kFp8RowsPerBlock - 1) / kFp8RowsPerBlock;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    return launch_k(rows_to_fp8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(32 * kFp8RowsPerBlock), 0, s, x, n_rows,
                    codes, row_scale);
}

cudaError_t launch_kv_push_raw(const float *kv, uint16_t *raw, long long raw_unit_stride, const int32_t *pos,
                               int32_t *n_raw, int U, uint32_t *status, cudaStream_t s) {
    return launch_k(kv_push_raw_kernel, dim3(U), dim3(kPushThreads), 0, s, kv, raw, raw_unit_stride, pos, n_raw, status);
}

cudaError_t launch_compressor_pool(const float *kv, const float *score, int ratio, int width, float *out, int U,
                                   cudaStream_t s) {
    // a warp covers 8 column groups (4 threads each)
    const long long warps = (static_cast<long long>(U) * (width >> 2) + 7) / 8;
    const long long blocks = (warps * 32 + kPoolThreads - 1) / kPoolThreads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    return launch_k(compressor_pool_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kPoolThreads), 0, s, kv, score, ratio,
                    width, out, U);
}

}  // namespace ds4a
