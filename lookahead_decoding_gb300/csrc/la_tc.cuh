// Device helpers of the tcgen05 GEMMs (sm_103a): mbarriers, bulk and tensor
// copies, shared-memory and instruction descriptors, tcgen05.mma / commit /
// ld, the split-tile sums and the bounded counter wait.  Shared by the
// per-GEMM kernel (la_gemm_tc.cu) and the layer-chain kernel (la_mega.cu).
#pragma once
#include "la_common.cuh"
#include "la_kernels.h"

namespace latc {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN_MAX = 256;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int ROW_BYTES = BK * 2;         // 128 B per activation row per unit
constexpr uint32_t TMEM_COLS = 512;       // two accumulators of up to 256 fp32 columns


__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < LA_SPIN_LIMIT; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int x, int y,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(tm), "r"(bar), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// contiguous global -> shared copy completing on an mbarrier (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;                 // leading byte offset (unused with 128B swizzle, K-major)
    d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                 // descriptor version
    d |= (uint64_t)2 << 61;                 // 128-byte swizzle
    return d;
}

// instruction descriptor: kind::f16, A = B = bf16, D = f32, both K-major, M = 128
__device__ __forceinline__ uint32_t idesc_bf16(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// named barrier among the four epilogue warps; the warp reconverges first
// (bar.sync is warp-aligned: a warp with lanes still in a divergent branch
// must not reach it)
__device__ __forceinline__ void epi_sync() {
    __syncwarp();
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

__device__ __forceinline__ void better(float& v, int& i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
}

// the CTA that owns unit x when T units are split evenly over P CTAs
__device__ __forceinline__ int cta_of(long long x, long long T, int P) { return (int)(((x + 1) * P - 1) / T); }

// Sum of the partials of columns cb .. cb+NC-1 (clamped to c_hi - 1) over the
// nseg segments, in segment order.  All NS x NC loads of a group are issued
// before the first add; clamped indices keep every load on a written entry.
template <int NS, int NC>
__device__ __forceinline__ void sum_segments(const float* src0, size_t seg_stride, int nseg, int cb, int c_hi,
                                             float (&dst)[NC]) {
#pragma unroll
    for (int j = 0; j < NC; ++j) dst[j] = 0.f;
    for (int s0 = 0; s0 < nseg; s0 += NS) {
        float t[NS][NC];
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const float* src = src0 + (size_t)min(s0 + k, nseg - 1) * seg_stride;
#pragma unroll
            for (int j = 0; j < NC; ++j) t[k][j] = __ldcg(src + (size_t)min(cb + j, c_hi - 1) * BM);
        }
#pragma unroll
        for (int k = 0; k < NS; ++k)
            if (s0 + k < nseg) {
#pragma unroll
                for (int j = 0; j < NC; ++j) dst[j] = __fadd_rn(dst[j], t[k][j]);
            }
    }
}

// bounded wait until a split-tile arrival counter reaches `target` (acquire)
__device__ __forceinline__ bool spin_until64(const unsigned long long* ctr, unsigned long long target) {
    for (uint32_t i = 0; i < LA_SPIN_LIMIT; ++i) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        __nanosleep(32);
    }
    return false;
}

}  // namespace latc
