// Masked attention of the packed call for bf16 models, in two kernels.
//
// Every row attends to one key per logical position 0..pos (M7.3 §0x04A:
// the committed prefix, then the row's own branch path).  The positions are
// split at t0(pos) = max(0, (floor(pos/32) - TB) * 32), a function of the
// row's position alone (TB is fixed per context so that pos - t0 covers
// every in-call offset):
//   * k_attn_blocks — keys [0, t0) are committed K/V; one CTA per (head,
//     128-position block) stages the block once and runs it for all rows on
//     tensor cores (mma.sync m16n8k16 -> fp32): S = Q K^T in bf16, a per-row
//     block maximum, P = exp(S - m) rounded to fp16, O = P V in fp16 (V
//     converts exactly from bf16; P keeps 10 mantissa bits).  The partial
//     (m, l, O) of each (row, head, block) goes to scratch.
//   * k_attn_combine — one warp per (row, head) merges the row's block
//     partials in block order, then walks the remaining positions [t0, pos]
//     in chunks of 32 with an online softmax on CUDA cores, taking each key
//     from the cache (committed) or from the call's temporary rows on the
//     row's path (in-call), and normalises.
// A row's arithmetic therefore depends only on its query, its position and
// the keys it sees — the same whether it is decoded alone or packed.
#include "la_common.cuh"
#include "la_kernels.h"

#include <cuda_fp16.h>
#include <math.h>

namespace {

constexpr int DH = 128;
constexpr int BLK = 128;          // positions per block
constexpr int RG = 128;           // rows per CTA (8 warps x 16)
constexpr int PAD = 8;            // bf16 padding per smem row (16 B): conflict-free fragment loads
constexpr int LDK = DH + PAD;     // K tile [key][dim]
constexpr int LDV = BLK + PAD;    // V tile transposed [dim][key]
constexpr int OOFF = 4;           // partial record: m, l, 2 pad, o[DH] (o 16-byte aligned)
constexpr int PSTR = DH + OOFF;

__device__ __forceinline__ int t0_of(int pos, int TB) {
    int b = (pos >> 5) - TB;
    return b > 0 ? (b << 5) : 0;
}

__device__ __forceinline__ int rows_sel(const LaHdr* h, int sel) {
    return sel == SEL_CALL ? h->Q : (sel == SEL_PREFILL ? h->prefill_rows : h->n_need);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void mma16816_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(256) k_attn_blocks(LaDev d, const __nv_bfloat16* qbuf, const __nv_bfloat16* kc,
                                                     const __nv_bfloat16* vc, float* part, int sel, int Qcap,
                                                     int max_ctx, int TB, int NS, int H) {
    const LaHdr* h = d.hdr;
    if (h->err != 0 || (sel != SEL_PREFILL && h->done != 0)) return;
    const int rows = rows_sel(h, sel);
    const int hh = blockIdx.x, blk = blockIdx.y, r0 = blockIdx.z * RG;
    if (r0 >= rows) return;
    const int key0 = blk * BLK;
    const int r1 = min(rows, r0 + RG);
    // skip the block if no row of this group sees committed keys in it
    int t0max = 0;
    for (int r = r0 + (int)threadIdx.x; r < r1; r += blockDim.x) t0max = max(t0max, t0_of(d.row_pos[r], TB));
    t0max = __reduce_max_sync(0xffffffffu, t0max);
    __shared__ int s_t0max[8];
    if ((threadIdx.x & 31) == 0) s_t0max[threadIdx.x >> 5] = t0max;
    __syncthreads();
    t0max = 0;
    for (int w = 0; w < 8; ++w) t0max = max(t0max, s_t0max[w]);
    if (t0max <= key0) return;

    extern __shared__ __align__(16) __nv_bfloat16 sm[];
    __nv_bfloat16* ks = sm;                                  // [BLK][LDK] bf16
    __half* vt = reinterpret_cast<__half*>(sm + BLK * LDK);  // [DH][LDV] fp16 (exact copies of bf16 V)
    const __nv_bfloat16* kh = kc + (size_t)hh * max_ctx * DH;
    const __nv_bfloat16* vh = vc + (size_t)hh * max_ctx * DH;
    // stage K [key][dim] and V transposed [dim][key]; positions past the cache read as zero
    for (int i = threadIdx.x; i < BLK * (DH / 8); i += blockDim.x) {
        const int key = i / (DH / 8), c8 = (i % (DH / 8)) * 8;
        const int p = key0 + key;
        int4 kv = make_int4(0, 0, 0, 0), vv = make_int4(0, 0, 0, 0);
        if (p < max_ctx) {
            kv = *reinterpret_cast<const int4*>(kh + (size_t)p * DH + c8);
            vv = *reinterpret_cast<const int4*>(vh + (size_t)p * DH + c8);
        }
        *reinterpret_cast<int4*>(ks + key * LDK + c8) = kv;
        const __nv_bfloat16* ve = reinterpret_cast<const __nv_bfloat16*>(&vv);
#pragma unroll
        for (int e = 0; e < 8; ++e) vt[(c8 + e) * LDV + key] = __float2half_rn(__bfloat162float(ve[e]));
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int rw = r0 + warp * 16;
    if (rw >= r1) return;
    const int ra = rw + g, rb = rw + g + 8;
    const int ta = ra < r1 ? t0_of(d.row_pos[ra], TB) : 0;
    const int tb = rb < r1 ? t0_of(d.row_pos[rb], TB) : 0;
    if (__all_sync(0xffffffffu, ta <= key0 && tb <= key0)) return;

    // Q fragments for 16 rows x 128 dims (8 k-steps)
    uint32_t qa[8][4];
    const __nv_bfloat16* qh = qbuf + (size_t)hh * Qcap * DH;
#pragma unroll
    for (int ks8 = 0; ks8 < 8; ++ks8) {
        const int c = ks8 * 16 + 2 * t;
        qa[ks8][0] = ra < r1 ? *reinterpret_cast<const uint32_t*>(qh + (size_t)ra * DH + c) : 0u;
        qa[ks8][1] = rb < r1 ? *reinterpret_cast<const uint32_t*>(qh + (size_t)rb * DH + c) : 0u;
        qa[ks8][2] = ra < r1 ? *reinterpret_cast<const uint32_t*>(qh + (size_t)ra * DH + c + 8) : 0u;
        qa[ks8][3] = rb < r1 ? *reinterpret_cast<const uint32_t*>(qh + (size_t)rb * DH + c + 8) : 0u;
    }
    // S = Q K^T over the 128 keys of the block (16 n-tiles of 8 keys)
    float s[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
        const __nv_bfloat16* krow = ks + (n * 8 + g) * LDK + 2 * t;
#pragma unroll
        for (int ks8 = 0; ks8 < 8; ++ks8) {
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow + ks8 * 16);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(krow + ks8 * 16 + 8);
            mma16816(s[n], qa[ks8], b0, b1);
        }
    }
    // mask (key position >= t0 of the row), scale, block maximum per row
    const float scale = 0.08838834764831845f;   // 1/sqrt(128)
    float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        const int kp = key0 + n * 8 + 2 * t;
        s[n][0] = (kp < ta) ? __fmul_rn(s[n][0], scale) : -INFINITY;
        s[n][1] = (kp + 1 < ta) ? __fmul_rn(s[n][1], scale) : -INFINITY;
        s[n][2] = (kp < tb) ? __fmul_rn(s[n][2], scale) : -INFINITY;
        s[n][3] = (kp + 1 < tb) ? __fmul_rn(s[n][3], scale) : -INFINITY;
        ma = fmaxf(ma, fmaxf(s[n][0], s[n][1]));
        mb = fmaxf(mb, fmaxf(s[n][2], s[n][3]));
    }
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    // P = exp(S - m) rounded to fp16 (the values the P V product uses); l sums them
    uint32_t pa[16][2];
    float la = 0.f, lb = 0.f;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        const float p0 = (s[n][0] == -INFINITY) ? 0.f : expf(__fsub_rn(s[n][0], ma));
        const float p1 = (s[n][1] == -INFINITY) ? 0.f : expf(__fsub_rn(s[n][1], ma));
        const float p2 = (s[n][2] == -INFINITY) ? 0.f : expf(__fsub_rn(s[n][2], mb));
        const float p3 = (s[n][3] == -INFINITY) ? 0.f : expf(__fsub_rn(s[n][3], mb));
        pa[n][0] = pack_f16(p0, p1);
        pa[n][1] = pack_f16(p2, p3);
        const __half2 q0 = *reinterpret_cast<__half2*>(&pa[n][0]);
        const __half2 q1 = *reinterpret_cast<__half2*>(&pa[n][1]);
        la = __fadd_rn(la, __fadd_rn(__low2float(q0), __high2float(q0)));
        lb = __fadd_rn(lb, __fadd_rn(__low2float(q1), __high2float(q1)));
    }
    la = __fadd_rn(la, __shfl_xor_sync(0xffffffffu, la, 1));
    la = __fadd_rn(la, __shfl_xor_sync(0xffffffffu, la, 2));
    lb = __fadd_rn(lb, __shfl_xor_sync(0xffffffffu, lb, 1));
    lb = __fadd_rn(lb, __shfl_xor_sync(0xffffffffu, lb, 2));
    // O = P V: 8 k-steps of 16 keys x 16 n-tiles of 8 dims
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a[4] = {pa[2 * kk][0], pa[2 * kk][1], pa[2 * kk + 1][0], pa[2 * kk + 1][1]};
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            const __half* vrow = vt + (n * 8 + g) * LDV + kk * 16 + 2 * t;
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(vrow);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(vrow + 8);
            mma16816_f16(o[n], a, b0, b1);
        }
    }
    // partial records for rows that see committed keys in this block
    if (ra < r1 && ta > key0) {
        float* pr = part + (((size_t)ra * H + hh) * NS + blk) * PSTR;
        if (t == 0) { pr[0] = ma; pr[1] = la; }
#pragma unroll
        for (int n = 0; n < 16; ++n) { pr[OOFF + n * 8 + 2 * t] = o[n][0]; pr[OOFF + n * 8 + 2 * t + 1] = o[n][1]; }
    }
    if (rb < r1 && tb > key0) {
        float* pr = part + (((size_t)rb * H + hh) * NS + blk) * PSTR;
        if (t == 0) { pr[0] = mb; pr[1] = lb; }
#pragma unroll
        for (int n = 0; n < 16; ++n) { pr[OOFF + n * 8 + 2 * t] = o[n][2]; pr[OOFF + n * 8 + 2 * t + 1] = o[n][3]; }
    }
}

__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// CW warps per CTA, one (row, head) per warp; each warp stages its row's
// 32-key chunks in shared memory with coalesced 16-byte loads.
constexpr int CW = 4;                 // warps per combine CTA
constexpr int LDC = DH + 8;           // staged key/value row (bf16), conflict-free 16-byte reads

__global__ void __launch_bounds__(CW * 32) k_attn_combine(LaDev d, const float* part, const __nv_bfloat16* qbuf,
                                                      const __nv_bfloat16* kc, const __nv_bfloat16* vc,
                                                      const __nv_bfloat16* kt, const __nv_bfloat16* vt,
                                                      __nv_bfloat16* out, int sel, int Qcap, int max_ctx, int Qmax,
                                                      int TB, int NS, int H) {
    const LaHdr* h = d.hdr;
    if (h->err != 0 || (sel != SEL_PREFILL && h->done != 0)) return;
    const int rows = rows_sel(h, sel);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hh = blockIdx.x;
    const int r = blockIdx.y * CW + warp;
    extern __shared__ __align__(16) uint8_t csm[];
    float (*q_s)[DH] = reinterpret_cast<float (*)[DH]>(csm);                                       // [CW][DH]
    __nv_bfloat16 (*k_s)[32][LDC] = reinterpret_cast<__nv_bfloat16 (*)[32][LDC]>(csm + CW * DH * 4);  // [CW][32][LDC]
    __nv_bfloat16 (*v_s)[32][DH] =
        reinterpret_cast<__nv_bfloat16 (*)[32][DH]>(csm + CW * DH * 4 + CW * 32 * LDC * 2);           // [CW][32][DH]
    if (r >= rows) return;
    for (int i = lane; i < DH; i += 32) q_s[warp][i] = __bfloat162float(qbuf[((size_t)hh * Qcap + r) * DH + i]);
    __syncwarp();
    const int prefill = (sel == SEL_PREFILL);
    const int pos = d.row_pos[r];
    const int t0 = t0_of(pos, TB);
    const int K = prefill ? 0 : h->K;
    const int Kr = prefill ? pos + 1 : K;        // positions below Kr are in the cache
    float m = -INFINITY, l = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
    // merge the committed blocks in block order
    const int nb = (t0 + BLK - 1) / BLK;
    for (int b = 0; b < nb; ++b) {
        const float* pr = part + (((size_t)r * H + hh) * NS + b) * PSTR;
        const float mj = pr[0], lj = pr[1];
        const float4 oj = *reinterpret_cast<const float4*>(pr + OOFF + lane * 4);
        const float mn = fmaxf(m, mj);
        const float ca = (m == -INFINITY) ? 0.f : expf(__fsub_rn(m, mn));
        const float cb = expf(__fsub_rn(mj, mn));
        l = fmaf(l, ca, __fmul_rn(lj, cb));
        o[0] = fmaf(o[0], ca, __fmul_rn(oj.x, cb));
        o[1] = fmaf(o[1], ca, __fmul_rn(oj.y, cb));
        o[2] = fmaf(o[2], ca, __fmul_rn(oj.z, cb));
        o[3] = fmaf(o[3], ca, __fmul_rn(oj.w, cb));
        m = mn;
    }
    // the remaining positions [t0, pos], 32 at a time
    const __nv_bfloat16* kch = kc + (size_t)hh * max_ctx * DH;
    const __nv_bfloat16* vch = vc + (size_t)hh * max_ctx * DH;
    const __nv_bfloat16* kth = kt + (size_t)hh * Qmax * DH;
    const __nv_bfloat16* vth = vt + (size_t)hh * Qmax * DH;
    const int* path = d.row_path + (size_t)r * d.PMAX;
    const float scale = 0.08838834764831845f;
    for (int c0 = t0; c0 <= pos; c0 += 32) {
        // stage the chunk: key j's source row (cache or the row's path), 16 bytes per lane per step
        const int p = c0 + lane;
        const bool valid = p <= pos;
        const __nv_bfloat16* kp = nullptr;
        const __nv_bfloat16* vp = nullptr;
        if (valid) {
            if (p < Kr) { kp = kch + (size_t)p * DH; vp = vch + (size_t)p * DH; }
            else {
                const int src = path[p - K];
                kp = kth + (size_t)src * DH; vp = vth + (size_t)src * DH;
            }
        }
        const int nvalid = min(32, pos - c0 + 1);
#pragma unroll 4
        for (int i = lane; i < 32 * (DH / 8); i += 32) {
            const int j = i >> 4, c8 = (i & 15) * 8;
            const __nv_bfloat16* kj = (const __nv_bfloat16*)__shfl_sync(0xffffffffu, (unsigned long long)kp, j);
            const __nv_bfloat16* vj = (const __nv_bfloat16*)__shfl_sync(0xffffffffu, (unsigned long long)vp, j);
            if (j < nvalid) {
                *reinterpret_cast<int4*>(&k_s[warp][j][c8]) = *reinterpret_cast<const int4*>(kj + c8);
                *reinterpret_cast<int4*>(&v_s[warp][j][c8]) = *reinterpret_cast<const int4*>(vj + c8);
            }
        }
        __syncwarp();
        float s = -INFINITY;
        if (valid) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < DH; i += 8) {
                const int4 kv = *reinterpret_cast<const int4*>(&k_s[warp][lane][i]);
                const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kv);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc = fmaf(q_s[warp][i + 2 * e], __low2float(k2[e]), acc);
                    acc = fmaf(q_s[warp][i + 2 * e + 1], __high2float(k2[e]), acc);
                }
            }
            s = __fmul_rn(acc, scale);
        }
        const float cmax = warp_max(valid ? s : -INFINITY);
        const float mn = fmaxf(m, cmax);
        const float pj_own = valid ? expf(__fsub_rn(s, mn)) : 0.f;
        const float corr = (m == -INFINITY) ? 0.f : expf(__fsub_rn(m, mn));
        l = fmaf(l, corr, warp_sum(pj_own));
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = __fmul_rn(o[e], corr);
        for (int j = 0; j < nvalid; ++j) {
            const float pj = __shfl_sync(0xffffffffu, pj_own, j);
            if (pj != 0.f) {
                const uint2 vv = *reinterpret_cast<const uint2*>(&v_s[warp][j][lane * 4]);
                const __nv_bfloat162 v01 = *reinterpret_cast<const __nv_bfloat162*>(&vv.x);
                const __nv_bfloat162 v23 = *reinterpret_cast<const __nv_bfloat162*>(&vv.y);
                o[0] = fmaf(pj, __low2float(v01), o[0]);
                o[1] = fmaf(pj, __high2float(v01), o[1]);
                o[2] = fmaf(pj, __low2float(v23), o[2]);
                o[3] = fmaf(pj, __high2float(v23), o[3]);
            }
        }
        m = mn;
        __syncwarp();
    }
    const float inv = 1.0f / l;
    __nv_bfloat16* op = out + (size_t)r * H * DH + hh * DH + lane * 4;
    *reinterpret_cast<__nv_bfloat162*>(op) = __floats2bfloat162_rn(__fmul_rn(o[0], inv), __fmul_rn(o[1], inv));
    *reinterpret_cast<__nv_bfloat162*>(op + 2) = __floats2bfloat162_rn(__fmul_rn(o[2], inv), __fmul_rn(o[3], inv));
}

}  // namespace

int la_attn_tail_blocks(int pmax) { return (pmax + 31) / 32; }
int la_attn_nblocks(int max_ctx) { return (max_ctx + BLK - 1) / BLK; }
int la_attn_record_floats() { return PSTR; }

cudaError_t la_launch_attention_bf16(const LaDev& d, cudaStream_t st, const void* qbuf, const void* kc, const void* vc,
                                     const void* kt, const void* vt, void* out, float* part, int H, int sel, int Qcap,
                                     int max_ctx, int Qmax, int rows_cap, int TB) {
    const int NS = la_attn_nblocks(max_ctx);
    const size_t smem = (size_t)(BLK * LDK + DH * LDV) * sizeof(__nv_bfloat16);
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_blocks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 g1(H, NS, (rows_cap + RG - 1) / RG);
    k_attn_blocks<<<g1, 256, smem, st>>>(d, (const __nv_bfloat16*)qbuf, (const __nv_bfloat16*)kc,
                                         (const __nv_bfloat16*)vc, part, sel, Qcap, max_ctx, TB, NS, H);
    const size_t csmem = (size_t)CW * DH * 4 + (size_t)CW * 32 * LDC * 2 + (size_t)CW * 32 * DH * 2;
    static bool cattr = false;
    if (!cattr) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_combine, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem);
        if (e != cudaSuccess) return e;
        cattr = true;
    }
    dim3 g2(H, (rows_cap + CW - 1) / CW);
    k_attn_combine<<<g2, CW * 32, csmem, st>>>(d, part, (const __nv_bfloat16*)qbuf, (const __nv_bfloat16*)kc,
                                       (const __nv_bfloat16*)vc, (const __nv_bfloat16*)kt, (const __nv_bfloat16*)vt,
                                       (__nv_bfloat16*)out, sel, Qcap, max_ctx, Qmax, TB, NS, H);
    return cudaGetLastError();
}
