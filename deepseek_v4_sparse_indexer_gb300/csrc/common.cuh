// Device helpers shared by the ds4a kernels: inline PTX for mbarriers, TMA,
// tcgen05 (UMMA + TMEM) and cp.async, plus the bounded
// waits every spin in this library goes through.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ds4a.h"

#define DS4A_DEV __device__ __forceinline__

namespace ds4a {

// A device-side wait gives up after this long and reports DS4A_DEV_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation (launch_k below): it lets the next kernel
// on the stream start launching at once (pdl_launch_dependents, the first
// thing each kernel does) and waits for the previous kernel to complete, with
// its memory visible, before touching global memory (pdl_wait).  Between
// dependent kernels the launch latency, the block scheduling and (tcgen05
// kernels) the barrier and TMEM set-up then overlap the previous kernel's
// tail; the data order is the stream order, as without it.  The one exception: the top-k kernels read the caller's row counts
// (n_rows) before the wait.  A kernel starts early only behind a kernel of this
// library; none of them writes n_rows, and the first kernel of such a chain
// started only once the stream's earlier work had completed.
DS4A_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
DS4A_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... Params, typename... Args>
inline cudaError_t launch_k(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args &&...args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

DS4A_DEV uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Thread-block cluster helpers.  Every thread of every CTA of the cluster
// must take part in cluster_sync_all (release/acquire at cluster scope orders
// the distributed shared-memory stores around it).
DS4A_DEV uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
DS4A_DEV void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Stores v at shared address `saddr` (this CTA's own layout) of CTA `rank` of the cluster.
DS4A_DEV void st_cluster_u32(uint32_t saddr, uint32_t rank, uint32_t v) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(r), "r"(v) : "memory");
}

// launch_k with a thread-block cluster of `cluster` CTAs along x.
template <typename... Params, typename... Args>
inline cudaError_t launch_k_cluster(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, int cluster,
                                    cudaStream_t s, Args &&...args) {
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

DS4A_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

DS4A_DEV void report(uint32_t *status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
DS4A_DEV void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
DS4A_DEV void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
DS4A_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
DS4A_DEV void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
DS4A_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up (returns
// false) after kWaitLimitNs, or early once *abort is set by another thread of
// the CTA that already gave up.
DS4A_DEV bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
}

// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps until it completes (or the hint runs out) instead of returning at
// once, so a waiting single-thread role takes no issue slots from the warps
// that share its SM sub-partition.
constexpr uint32_t kSuspendHintNs = 20000;
DS4A_DEV bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}
// mbar_wait through the hinted try_wait; same limits.
DS4A_DEV bool mbar_wait_hint(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait_hint(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_hint(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), no multicast
// ---------------------------------------------------------------------------
DS4A_DEV void tma_prefetch_desc(const void *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// global memory into this CTA's shared memory, completing on `bar`.
DS4A_DEV void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    uint64_t g;
    asm("cvta.to.global.u64 %0, %1;" : "=l"(g) : "l"(src));
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(g), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
// L2 prefetch of one box of a tensor map (no shared memory, no barrier).  L2 is
// the device's point of coherence, so a prefetch issued before the previous
// kernel has finished writing the tensor cannot leave a stale copy behind.
DS4A_DEV void tma_prefetch_l2_2d(const void *map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}
DS4A_DEV void tma_prefetch_l2_3d(const void *map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}
DS4A_DEV void tma_load_2d(void *dst, const void *map, uint64_t *bar, int x, int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
DS4A_DEV void tma_load_3d(void *dst, const void *map, uint64_t *bar, int x, int y, int z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
DS4A_DEV uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
DS4A_DEV uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, UMMA (kind::f16, cta_group::1), commit, loads
// ---------------------------------------------------------------------------
// Whole warp.  Writes the TMEM base address to *slot (shared memory).
DS4A_DEV void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
DS4A_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
DS4A_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DS4A_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.
DS4A_DEV void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on *bar when every UMMA this thread issued so far has completed.
DS4A_DEV void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 D, both K-major.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B format
// (1 = bf16), 15/16 A/B major (0 = K), [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a K-major operand stored as 128-byte
// rows with the 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B and a 64-element bf16 inner box): 8-row groups
// 1024 bytes apart.  The tile base must be 1024-byte aligned; a K offset
// inside the 128-byte row is applied by adding bytes to the start address.
DS4A_DEV uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);   // [0,14)  start address >> 4
    d |= static_cast<uint64_t>(1) << 16;                       // [16,30) leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;               // [32,46) stride byte offset >> 4
    d |= static_cast<uint64_t>(1) << 46;                       // [46,48) descriptor version 1
    d |= static_cast<uint64_t>(2) << 61;                       // [61,64) 128-byte swizzle
    return d;
}

// ---------------------------------------------------------------------------
// cp.async
// ---------------------------------------------------------------------------
// 16-byte async copy; src_bytes = 0 writes 16 zero bytes (src still valid).
DS4A_DEV void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
DS4A_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
DS4A_DEV void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Two fp32 -> packed pair (low half = x) in bf16 or fp16, round to nearest even.
template <bool IsF16>
DS4A_DEV uint32_t pack2(float x, float y) {
    uint32_t r;
    if constexpr (IsF16) {
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(y), "f"(x));
    } else {
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(y), "f"(x));
    }
    return r;
}

// Order-preserving map from fp32 to uint32: a > b (as floats, -0 == +0)
// implies key(a) > key(b).  -0 is folded onto +0 first.
DS4A_DEV uint32_t float_key(float f) {
    uint32_t b = __float_as_uint(f);
    if ((b << 1) == 0) b = 0;                  // -0 -> +0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// The float whose key is k (the inverse of float_key; key 0x80000000 gives +0).
DS4A_DEV float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// Visible = a real score: not -inf, not NaN.
DS4A_DEV bool score_visible(float f) { return f == f && f != -__int_as_float(0x7f800000); }

// Adds 1 to h[bin] for every lane with pred, one shared atomic per distinct
// bin in the warp (scores of one row often share a few bins).  All 32 lanes
// must call it.
DS4A_DEV void hist_add_warp(uint32_t *h, uint32_t bin, bool pred) {
    const uint32_t active = __ballot_sync(0xffffffffu, pred);
    if (!pred) return;
    const uint32_t peers = __match_any_sync(active, bin);
    if (static_cast<int>(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&h[bin], static_cast<uint32_t>(__popc(peers)));
}

}  // namespace ds4a
