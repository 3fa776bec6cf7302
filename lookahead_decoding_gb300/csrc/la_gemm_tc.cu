// Tensor-core GEMM of the packed call on sm_103a: Y[q][n] = sum_k X[q][k] W[n][k]
// for the QKV, O, gate/up (SwiGLU) and down projections and the LM head.
//
// The call is a skinny contraction (Q packed rows against a weight matrix
// that is read once per call), so the weights take the MMA's M side:
//   - one CTA owns BM = 128 weight rows (n) and up to 256 packed rows (q);
//   - TMA streams 128 x 64 bf16 weight tiles and q x 64 activation tiles,
//     both 128-byte swizzled, through a multi-stage mbarrier pipeline;
//   - one thread issues tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in
//     TMEM, M = 128, N = q rounded up to 16, K = 16 per instruction);
//   - four warps read the accumulator back with tcgen05.ld and run the
//     epilogue (store, residual add, SwiGLU, or logits + argmax partials).
// Split-K is fixed per weight shape (never by Q) and reduced by the last
// arriving CTA in split order, so a row's result is independent of how many
// rows share the call.
//
// Every wait on an mbarrier is bounded; a wait that runs out sets the device
// error word (LA_ETIMEOUT) and the CTA skips its outputs, frees its TMEM and
// returns.
#include "la_common.cuh"
#include "la_kernels.h"

#include <cudaTypedefs.h>
#include <algorithm>

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN_MAX = 256;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int ROW_BYTES = BK * 2;         // 128 B per activation row per stage
constexpr int BOX_ROWS = 16;
constexpr int MAX_STAGES = 8;
constexpr int SMEM_BYTES = 200 * 1024;

struct TcParams {
    LaHdr* hdr;
    int sel, mode, K, Nout, k_tiles, splits, n_tiles, seg_tiles;
    void* out; int ldo;
    float* logits; int ld_logits;
    float* ws; int* counters;
    float* part_v; int* part_i; int part_stride;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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

__device__ __forceinline__ void better(float& v, int& i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
}

__global__ void __launch_bounds__(128, 1)
k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
          const __grid_constant__ CUtensorMap tmA3, const __grid_constant__ CUtensorMap tmB, TcParams p) {
    LaHdr* h = p.hdr;
    if (h->err != 0 || (p.sel != SEL_PREFILL && h->done != 0)) return;
    const int rows = p.sel == SEL_CALL ? h->Q : (p.sel == SEL_PREFILL ? h->prefill_rows : h->n_need);
    const int q0 = blockIdx.z * BN_MAX;
    if (q0 >= rows) return;
    const int nq = min(BN_MAX, rows - q0);
    const int BN = (nq + 15) & ~15;
    const int tile = blockIdx.x, split = blockIdx.y;
    const int swiglu = (p.mode == GEMM_SWIGLU);
    const int nA = swiglu ? 2 : 1;
    const int kt0 = (int)((long long)p.k_tiles * split / p.splits);
    const int kt1 = (int)((long long)p.k_tiles * (split + 1) / p.splits);
    const int nk = kt1 - kt0;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    // layout: [barriers 1 KB][stages ...]
    const uint32_t bar_full = base;                        // MAX_STAGES x 8 B
    const uint32_t bar_empty = base + 8 * MAX_STAGES;
    const uint32_t bar_acc = base + 16 * MAX_STAGES;
    uint32_t* tmem_slot = (uint32_t*)(gbase + 16 * MAX_STAGES + 8);
    int* s_flag = (int*)(gbase + 16 * MAX_STAGES + 16);
    float* red_v = (float*)(gbase + 1024 + 0);             // reuses stage memory after the mainloop
    const uint32_t stage0 = base + 1024;
    const uint32_t b_bytes = (uint32_t)BN * ROW_BYTES;
    const uint32_t stage_bytes = (((uint32_t)nA * A_BYTES + b_bytes) + 1023u) & ~1023u;
    int ns = (int)((SMEM_BYTES - 2048) / stage_bytes);
    ns = ns > MAX_STAGES ? MAX_STAGES : ns;
    const uint32_t tx_bytes = (uint32_t)nA * A_BYTES + b_bytes;
    const uint32_t ncols = swiglu ? 512u : 256u;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_acc, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *s_flag = 0;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0 && lane == 0) {
        // TMA producer
        // weight rows of this tile (segmented launches concatenate up to three matrices)
        const CUtensorMap* wmap = &tmA;
        int wrow = tile * BM;
        if (p.seg_tiles > 0) {
            const int seg = tile / p.seg_tiles;
            wmap = seg == 0 ? &tmA : (seg == 1 ? &tmA2 : &tmA3);
            wrow = (tile - seg * p.seg_tiles) * BM;
        }
        uint64_t pol_w, pol_x;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
        for (int it = 0; it < nk; ++it) {
            const int s = it % ns, u = it / ns;
            if (u > 0 && !mbar_wait(bar_empty + 8 * s, (uint32_t)((u - 1) & 1))) { ok = false; break; }
            const uint32_t st = stage0 + (uint32_t)s * stage_bytes;
            const uint32_t fb = bar_full + 8 * s;
            mbar_expect_tx(fb, tx_bytes);
            const int kx = (kt0 + it) * BK;
            tma_load_2d(st, wmap, fb, kx, wrow, pol_w);
            if (swiglu) tma_load_2d(st + A_BYTES, &tmA2, fb, kx, tile * BM, pol_w);
            const uint32_t bst = st + (uint32_t)nA * A_BYTES;
            for (int r = 0; r < BN; r += BOX_ROWS) tma_load_2d(bst + (uint32_t)r * ROW_BYTES, &tmB, fb, kx, q0 + r, pol_x);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        const uint32_t id = idesc_bf16(BN);
        for (int it = 0; it < nk; ++it) {
            const int s = it % ns, u = it / ns;
            if (!mbar_wait(bar_full + 8 * s, (uint32_t)(u & 1))) { ok = false; break; }
            tc_fence_after();
            const uint32_t st = stage0 + (uint32_t)s * stage_bytes;
            const uint32_t bst = st + (uint32_t)nA * A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t bdesc = sdesc(bst + kk * 32);
                mma_bf16(tmem, sdesc(st + kk * 32), bdesc, id, (it > 0 || kk > 0) ? 1u : 0u);
                if (swiglu) mma_bf16(tmem + (uint32_t)BN_MAX, sdesc(st + A_BYTES + kk * 32), bdesc, id,
                                     (it > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(bar_empty + 8 * s);
        }
        mma_commit(bar_acc);
    }
    __syncwarp();
    if (!__all_sync(0xffffffffu, ok)) la_set_err(h, LA_ETIMEOUT);
    // every thread waits for the accumulator
    bool acc_ok = mbar_wait(bar_acc, 0u);
    if (!acc_ok) la_set_err(h, LA_ETIMEOUT);
    tc_fence_after();

    const int n_local = warp * 32 + lane;
    const int n = tile * BM + n_local;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const int is_split = p.splits > 1;
    const bool last_ok = acc_ok && nk > 0;

    // ---- split-K: publish partial, let the last CTA of the tile finish
    if (is_split) {
        float* wsb = p.ws + ((size_t)(tile + (size_t)blockIdx.z * p.n_tiles) * p.splits + split) * (2 * BN_MAX * BM);
        for (int c0 = 0; c0 < BN; c0 += 16) {
            float v[16];
            tmem_ld16(trow + c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) wsb[(size_t)(c0 + j) * BM + n_local] = last_ok ? v[j] : 0.f;
            if (swiglu) {
                tmem_ld16(trow + BN_MAX + c0, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) wsb[(size_t)(BN_MAX + c0 + j) * BM + n_local] = last_ok ? v[j] : 0.f;
            }
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            int* ctr = p.counters + tile + blockIdx.z * p.n_tiles;
            int old = atomicAdd(ctr, 1);
            int last = (old == p.splits - 1);
            if (last) *ctr = 0;
            *s_flag = last;
        }
        __syncthreads();
        if (!*s_flag) goto done;
        __threadfence();
    }

    // ---- final epilogue, 16 packed rows at a time
    {
        const float* wst = p.ws + (size_t)(tile + (size_t)blockIdx.z * p.n_tiles) * p.splits * (2 * BN_MAX * BM);
        float* rv = (float*)red_v;                 // [4][BN] values
        int* ri = (int*)(red_v + 4 * BN_MAX);      // [4][BN] indices
        for (int c0 = 0; c0 < BN; c0 += 16) {
            float v[16], u[16];
            if (is_split) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float a = 0.f, b = 0.f;
                    for (int s = 0; s < p.splits; ++s) {
                        const float* w = wst + (size_t)s * (2 * BN_MAX * BM);
                        a = __fadd_rn(a, __ldcg(w + (size_t)(c0 + j) * BM + n_local));
                        if (swiglu) b = __fadd_rn(b, __ldcg(w + (size_t)(BN_MAX + c0 + j) * BM + n_local));
                    }
                    v[j] = a; u[j] = b;
                }
            } else {
                tmem_ld16(trow + c0, v);
                if (swiglu) tmem_ld16(trow + BN_MAX + c0, u);
            }
            if (!acc_ok) continue;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int q = q0 + c0 + j;
                const bool in = q < rows;
                const size_t o = (size_t)q * p.ldo + n;
                if (p.mode == GEMM_STORE) {
                    if (in) ((__nv_bfloat16*)p.out)[o] = __float2bfloat16_rn(v[j]);
                } else if (p.mode == GEMM_RESID) {
                    if (in) ((float*)p.out)[o] += v[j];
                } else if (p.mode == GEMM_SWIGLU) {
                    if (in) ((__nv_bfloat16*)p.out)[o] = __float2bfloat16_rn(v[j] / (1.0f + expf(-v[j])) * u[j]);
                } else {   // logits + argmax partials over this tile's 128 vocab entries
                    if (in && p.logits) p.logits[(size_t)q * p.ld_logits + n] = v[j];
                    float bv = v[j];
                    int bi = n;
#pragma unroll
                    for (int o2 = 16; o2 > 0; o2 >>= 1) {
                        float v2 = __shfl_xor_sync(0xffffffffu, bv, o2);
                        int i2 = __shfl_xor_sync(0xffffffffu, bi, o2);
                        better(bv, bi, v2, i2);
                    }
                    if (lane == 0) { rv[warp * BN_MAX + c0 + j] = bv; ri[warp * BN_MAX + c0 + j] = bi; }
                }
            }
        }
        if (p.mode == GEMM_LOGITS) {
            __syncthreads();
            for (int c = tid; c < nq; c += blockDim.x) {
                float bv = rv[c];
                int bi = ri[c];
                for (int w = 1; w < 4; ++w) better(bv, bi, rv[w * BN_MAX + c], ri[w * BN_MAX + c]);
                if (acc_ok) {
                    p.part_v[(size_t)tile * p.part_stride + q0 + c] = bv;
                    p.part_i[(size_t)tile * p.part_stride + q0 + c] = bi;
                }
            }
        }
    }
done:
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int la_tc_make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return -1;
        g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : (int)r;
}

// Fixed split-K per weight shape: enough CTAs to cover the SMs once.
int la_tc_split_for(int n_tiles, int k_tiles) {
    const int sms = 148;
    int s = sms / n_tiles;
    if (s < 1) s = 1;
    if (s > 8) s = 8;
    if (s > k_tiles) s = k_tiles;
    return s;
}

cudaError_t la_launch_gemm_tc(const LaDev& d, cudaStream_t st, const TcGemm& g, const TcWork& w, int sel) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES + 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    TcParams p;
    p.hdr = d.hdr;
    p.sel = sel;
    p.mode = g.mode;
    p.K = g.K;
    p.Nout = g.Nout;
    p.k_tiles = g.K / BK;
    p.splits = g.splits;
    p.n_tiles = g.Nout / BM;
    p.seg_tiles = g.seg_tiles;
    p.out = g.out;
    p.ldo = g.ldo;
    p.logits = g.logits;
    p.ld_logits = g.ld_logits;
    p.ws = w.ws;
    p.counters = w.counters;
    p.part_v = w.part_v;
    p.part_i = w.part_i;
    p.part_stride = w.part_stride;
    dim3 grid(p.n_tiles, g.splits, (g.rows_cap + BN_MAX - 1) / BN_MAX);
    k_gemm_tc<<<grid, 128, SMEM_BYTES + 1024, st>>>(g.tmA, g.tmA2, g.tmA3, g.tmB, p);
    return cudaGetLastError();
}
