// Masked attention of the packed call for bf16 models, in two kernels.
//
// Every row attends to one key per logical position 0..pos (M7.3 §0x04A:
// the committed prefix, then the row's own branch path).  The positions are
// split at t0(pos) = max(0, (floor(pos/32) - TB) * 32), a function of the
// row's position alone (TB is fixed per context so that pos - t0 covers
// every in-call offset):
//   * k_attn_blocks — keys [0, t0) are committed K/V; one CTA per (head,
//     128-position block) stages the block once (cp.async, [key][dim] bf16)
//     and runs it for all rows on tensor cores (mma.sync m16n8k16 -> fp32):
//     S = Q K^T in bf16, a per-row block maximum, P = exp(S - m) rounded to
//     fp16, O = P V in fp16 (V fragments by ldmatrix.trans, converted exactly
//     from bf16; P keeps 10 mantissa bits).  The partial (m, l, O) of each
//     (row, head, block) goes to scratch.
//   * k_attn_tail — one warp per (row, head) merges the row's block partials
//     in block order, then takes the remaining positions [t0, pos] (at most
//     128) as one softmax block on CUDA cores, one key per lane, each key
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
constexpr int LDK = DH + PAD;     // K and V tiles [key][dim]
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// two bf16 -> two fp16 (exact for |v| in the fp16 normal range)
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t x) {
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&x);
    return pack_f16(__low2float(b), __high2float(b));
}

__global__ void __launch_bounds__(256) k_attn_blocks(LaDev d, const __nv_bfloat16* qbuf, const __nv_bfloat16* kc,
                                                     const __nv_bfloat16* vc, float* part, int sel, int Qcap,
                                                     int max_ctx, int TB, int NS, int H) {
    la_pdl_wait();
    la_pdl_trigger();
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
    __nv_bfloat16* ks = sm;                 // [BLK][LDK] bf16 keys
    __nv_bfloat16* vs = sm + BLK * LDK;     // [BLK][LDK] bf16 values (same layout; fragments via ldmatrix.trans)
    const __nv_bfloat16* kh = kc + (size_t)hh * max_ctx * DH;
    const __nv_bfloat16* vh = vc + (size_t)hh * max_ctx * DH;
    // stage the block with 16-byte asynchronous copies; positions past the cache read as zero
    const uint32_t ks_a = (uint32_t)__cvta_generic_to_shared(ks), vs_a = (uint32_t)__cvta_generic_to_shared(vs);
    for (int i = threadIdx.x; i < BLK * (DH / 8); i += blockDim.x) {
        const int key = i >> 4, c8 = (i & 15) * 8;
        const int p = key0 + key;
        const int ok = p < max_ctx;
        const size_t src = (size_t)(ok ? p : 0) * DH + c8;
        const uint32_t off = (uint32_t)(key * LDK + c8) * 2u;
        cp_async16(ks_a + off, kh + src, ok ? 16 : 0);
        cp_async16(vs_a + off, vh + src, ok ? 16 : 0);
    }
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
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
    // O = P V: 8 k-steps of 16 keys x 16 n-tiles of 8 dims; V fragments by
    // transposing 8x8 tiles of the [key][dim] block, converted to fp16
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    // lane -> (matrix, row): matrices {keys 0-7, keys 8-15} x {dims n*8, dims n*8+8}
    const int mtx = lane >> 3, mrow = lane & 7;
    const int key_off = (mtx & 1) * 8 + mrow, dim_off = (mtx >> 1) * 8;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a[4] = {pa[2 * kk][0], pa[2 * kk][1], pa[2 * kk + 1][0], pa[2 * kk + 1][1]};
#pragma unroll
        for (int n = 0; n < 16; n += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(vs_a + (uint32_t)((kk * 16 + key_off) * LDK + n * 8 + dim_off) * 2u, b0, b1, b2, b3);
            mma16816_f16(o[n], a, bf2_to_h2(b0), bf2_to_h2(b1));
            mma16816_f16(o[n + 1], a, bf2_to_h2(b2), bf2_to_h2(b3));
        }
    }
    // partial records for rows that see committed keys in this block
    if (ra < r1 && ta > key0) {
        float* pr = part + (((size_t)ra * H + hh) * NS + blk) * PSTR;
        if (t == 0) { pr[0] = ma; pr[1] = la; }
#pragma unroll
        for (int n = 0; n < 16; ++n) *reinterpret_cast<float2*>(pr + OOFF + n * 8 + 2 * t) = make_float2(o[n][0], o[n][1]);
    }
    if (rb < r1 && tb > key0) {
        float* pr = part + (((size_t)rb * H + hh) * NS + blk) * PSTR;
        if (t == 0) { pr[0] = mb; pr[1] = lb; }
#pragma unroll
        for (int n = 0; n < 16; ++n) *reinterpret_cast<float2*>(pr + OOFF + n * 8 + 2 * t) = make_float2(o[n][2], o[n][3]);
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

// One warp per (row, head): merges the row's committed-block partials in
// block order, then the positions [t0, pos] — at most MAX_ROUNDS x 32 keys,
// one key per lane per round, each taken from the cache (committed) or from
// the call's temporary rows on the row's path (in-call) — as one softmax
// block, and normalises.  Every load of a stage is issued before its first
// use, so a warp spends a few memory round trips, not one per key.
constexpr int TW = 4;                 // warps per tail CTA
constexpr int MAX_ROUNDS = 4;         // tail keys <= 128 (TB <= 3)
constexpr int MAX_BLK = 8;            // block partials merged per batch

__global__ void __launch_bounds__(TW * 32) k_attn_tail(LaDev d, const float* part, const __nv_bfloat16* qbuf,
                                                     const __nv_bfloat16* kc, const __nv_bfloat16* vc,
                                                     const __nv_bfloat16* kt, const __nv_bfloat16* vt,
                                                     __nv_bfloat16* out, int sel, int Qcap, int max_ctx, int Qmax,
                                                     int TB, int NS, int H) {
    la_pdl_wait();
    la_pdl_trigger();
    const LaHdr* h = d.hdr;
    if (h->err != 0 || (sel != SEL_PREFILL && h->done != 0)) return;
    const int rows = rows_sel(h, sel);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hh = blockIdx.x;
    const int r = blockIdx.y * TW + warp;
    __shared__ __align__(16) float q_s[TW][DH];
    if (r >= rows) return;
    const int prefill = (sel == SEL_PREFILL);
    const int pos = d.row_pos[r];
    const int t0 = t0_of(pos, TB);
    const int K = prefill ? 0 : h->K;
    const int Kr = prefill ? pos + 1 : K;        // positions below Kr are in the cache
    {
        const uint2 qv = *reinterpret_cast<const uint2*>(qbuf + ((size_t)hh * Qcap + r) * DH + lane * 4);
        const __nv_bfloat162 q01 = *reinterpret_cast<const __nv_bfloat162*>(&qv.x);
        const __nv_bfloat162 q23 = *reinterpret_cast<const __nv_bfloat162*>(&qv.y);
        *reinterpret_cast<float4*>(&q_s[warp][lane * 4]) =
            make_float4(__low2float(q01), __high2float(q01), __low2float(q23), __high2float(q23));
    }
    // tail key sources: lane l owns the keys t0 + l + 32 i
    const int n = pos - t0 + 1;
    const __nv_bfloat16* kch = kc + (size_t)hh * max_ctx * DH;
    const __nv_bfloat16* vch = vc + (size_t)hh * max_ctx * DH;
    const __nv_bfloat16* kth = kt + (size_t)hh * Qmax * DH;
    const __nv_bfloat16* vth = vt + (size_t)hh * Qmax * DH;
    const int* path = d.row_path + (size_t)r * d.PMAX;
    size_t srow[MAX_ROUNDS];                 // element offset of the key's row; bit 63: in-call
#pragma unroll
    for (int i = 0; i < MAX_ROUNDS; ++i) {
        const int j = lane + 32 * i;
        const int p = t0 + j;
        srow[i] = 0;
        if (j < n) {
            if (p < Kr) srow[i] = (size_t)p * DH;
            else srow[i] = ((size_t)path[p - K] * DH) | (1ull << 63);
        }
    }
    // merge the committed blocks in block order (loads of a batch issued together)
    float m = -INFINITY, l = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
    const int nb = (t0 + BLK - 1) / BLK;
    for (int b0 = 0; b0 < nb; b0 += MAX_BLK) {
        float mj[MAX_BLK], lj[MAX_BLK];
        float4 oj[MAX_BLK];
#pragma unroll
        for (int k = 0; k < MAX_BLK; ++k) {
            const int b = min(b0 + k, nb - 1);
            const float* pr = part + (((size_t)r * H + hh) * NS + b) * PSTR;
            mj[k] = pr[0];
            lj[k] = pr[1];
            oj[k] = *reinterpret_cast<const float4*>(pr + OOFF + lane * 4);
        }
#pragma unroll
        for (int k = 0; k < MAX_BLK; ++k) {
            if (b0 + k >= nb) break;
            const float mn = fmaxf(m, mj[k]);
            const float ca = (m == -INFINITY) ? 0.f : expf(__fsub_rn(m, mn));
            const float cb = expf(__fsub_rn(mj[k], mn));
            l = fmaf(l, ca, __fmul_rn(lj[k], cb));
            o[0] = fmaf(o[0], ca, __fmul_rn(oj[k].x, cb));
            o[1] = fmaf(o[1], ca, __fmul_rn(oj[k].y, cb));
            o[2] = fmaf(o[2], ca, __fmul_rn(oj[k].z, cb));
            o[3] = fmaf(o[3], ca, __fmul_rn(oj[k].w, cb));
            m = mn;
        }
    }
    __syncwarp();
    // scores of the tail keys: one key per lane per round, 16-byte loads issued together
    const float scale = 0.08838834764831845f;
    float sc[MAX_ROUNDS];
#pragma unroll
    for (int i = 0; i < MAX_ROUNDS; ++i) {
        sc[i] = -INFINITY;
        if (32 * i >= n) continue;                       // warp-uniform
        const bool valid = lane + 32 * i < n;
        const __nv_bfloat16* kp = ((srow[i] >> 63) ? kth : kch) + (srow[i] & ~(1ull << 63));
        int4 kv[DH / 8];
#pragma unroll
        for (int c = 0; c < DH / 8; ++c) kv[c] = valid ? *reinterpret_cast<const int4*>(kp + c * 8) : make_int4(0, 0, 0, 0);
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < DH / 8; ++c) {
            const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kv[c]);
            const float4 qa = *reinterpret_cast<const float4*>(&q_s[warp][c * 8]);
            const float4 qb = *reinterpret_cast<const float4*>(&q_s[warp][c * 8 + 4]);
            acc = fmaf(qa.x, __low2float(k2[0]), acc);
            acc = fmaf(qa.y, __high2float(k2[0]), acc);
            acc = fmaf(qa.z, __low2float(k2[1]), acc);
            acc = fmaf(qa.w, __high2float(k2[1]), acc);
            acc = fmaf(qb.x, __low2float(k2[2]), acc);
            acc = fmaf(qb.y, __high2float(k2[2]), acc);
            acc = fmaf(qb.z, __low2float(k2[3]), acc);
            acc = fmaf(qb.w, __high2float(k2[3]), acc);
        }
        if (valid) sc[i] = __fmul_rn(acc, scale);
    }
    // one softmax block over the tail
    float tm = sc[0];
#pragma unroll
    for (int i = 1; i < MAX_ROUNDS; ++i) tm = fmaxf(tm, sc[i]);
    tm = warp_max(tm);
    float pj[MAX_ROUNDS], ps = 0.f;
#pragma unroll
    for (int i = 0; i < MAX_ROUNDS; ++i) {
        pj[i] = (sc[i] == -INFINITY) ? 0.f : expf(__fsub_rn(sc[i], tm));
        ps = __fadd_rn(ps, pj[i]);
    }
    const float tl = warp_sum(ps);
    // P V in key order: each lane accumulates its 4 dims over the tail keys, 16 keys' values in flight
    float to[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < n; j0 += 16) {
        uint2 vv[16];
        float pv[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int j = min(j0 + k, n - 1);
            const int i = j >> 5, src_lane = j & 31;
            size_t so = 0;
            float pk = 0.f;
#pragma unroll
            for (int ii = 0; ii < MAX_ROUNDS; ++ii)
                if (ii == i) {
                    so = __shfl_sync(0xffffffffu, srow[ii], src_lane);
                    pk = __shfl_sync(0xffffffffu, pj[ii], src_lane);
                }
            const __nv_bfloat16* vp = ((so >> 63) ? vth : vch) + (so & ~(1ull << 63));
            vv[k] = *reinterpret_cast<const uint2*>(vp + lane * 4);
            pv[k] = (j0 + k < n) ? pk : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (j0 + k >= n) break;
            const __nv_bfloat162 v01 = *reinterpret_cast<const __nv_bfloat162*>(&vv[k].x);
            const __nv_bfloat162 v23 = *reinterpret_cast<const __nv_bfloat162*>(&vv[k].y);
            to[0] = fmaf(pv[k], __low2float(v01), to[0]);
            to[1] = fmaf(pv[k], __high2float(v01), to[1]);
            to[2] = fmaf(pv[k], __low2float(v23), to[2]);
            to[3] = fmaf(pv[k], __high2float(v23), to[3]);
        }
    }
    // merge the tail block, normalise
    const float mn = fmaxf(m, tm);
    const float ca = (m == -INFINITY) ? 0.f : expf(__fsub_rn(m, mn));
    const float cb = expf(__fsub_rn(tm, mn));
    l = fmaf(l, ca, __fmul_rn(tl, cb));
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = fmaf(o[e], ca, __fmul_rn(to[e], cb));
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
    if (TB + 1 > MAX_ROUNDS) return cudaErrorInvalidValue;
    const int NS = la_attn_nblocks(max_ctx);
    const size_t smem = (size_t)(2 * BLK * LDK) * sizeof(__nv_bfloat16);
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_blocks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 g1(H, NS, (rows_cap + RG - 1) / RG);
    cudaError_t e = la_launch_pdl(k_attn_blocks, g1, dim3(256), smem, st, d, (const __nv_bfloat16*)qbuf,
                                  (const __nv_bfloat16*)kc, (const __nv_bfloat16*)vc, part, sel, Qcap, max_ctx, TB, NS, H);
    if (e != cudaSuccess) return e;
    dim3 g2(H, (rows_cap + TW - 1) / TW);
    return la_launch_pdl(k_attn_tail, g2, dim3(TW * 32), 0, st, d, (const float*)part, (const __nv_bfloat16*)qbuf,
                         (const __nv_bfloat16*)kc, (const __nv_bfloat16*)vc, (const __nv_bfloat16*)kt,
                         (const __nv_bfloat16*)vt, (__nv_bfloat16*)out, sel, Qcap, max_ctx, Qmax, TB, NS, H);
}
