// Model kernels of the packed target call: embedding, RMSNorm, RoPE + K/V
// write, masked attention, the CUDA-core GEMM (fp32 model and reference
// path), and the LM-head argmax reductions.
//
// Row invariance: every kernel computes a row's result with an arithmetic
// order that depends only on that row's inputs and logical position, never
// on how many rows share the call or where the row sits in the batch.  This
// makes a row packed with others bit-identical to the same token decoded
// alone, which is what lets the lookahead output equal autoregressive
// greedy decoding exactly (M7.3 §0x02A: the method's fixed point is the
// autoregressive result; the equality needs the same selector on the same
// logits).
#include "la_common.cuh"
#include "la_kernels.h"

#include <math.h>

// ---------------------------------------------------------------------------
// RoPE table: cos/sin(pos * theta^(-2i/dh)) evaluated in fp64, stored fp32
// ---------------------------------------------------------------------------
__global__ void k_rope_table(float* rcos, float* rsin, int n_pos, int half, double theta, int dh) {
    int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_pos * half) return;
    int p = idx / half, i = idx % half;
    double inv = pow(theta, -2.0 * (double)i / (double)dh);
    double ang = (double)p * inv;
    rcos[idx] = (float)cos(ang);
    rsin[idx] = (float)sin(ang);
}

__device__ __forceinline__ int rows_of(const LaHdr* h, int sel) {
    // sel: 0 = packed rows of the call, 1 = prefill chunk rows, 2 = needed rows
    return sel == 0 ? h->Q : (sel == 1 ? h->prefill_rows : h->n_need);
}
__device__ __forceinline__ bool skip_call(const LaHdr* h, int sel) {
    return h->err != 0 || (sel != 1 && h->done != 0);
}

// ---------------------------------------------------------------------------
// embedding: x[q][:] = E[tok[q]]  (fp32 residual stream)
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) { return *reinterpret_cast<const float4*>(p); }
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
}

template <typename T>
__global__ void k_embed(LaDev d, const T* emb, float* x, int dm, int sel) {
    LaTl la_tl_(LA_TL_EMBED, d.tl);
    la_pdl_wait();
    la_pdl_trigger();
    const LaHdr* h = d.hdr;
    if (skip_call(h, sel)) return;
    const int q = blockIdx.x;
    if (q >= rows_of(h, sel)) return;
    const int tok = d.row_tok[q];
    if (tok < 0 || tok >= d.V) { la_set_err(d.hdr, LA_EDEVICE); return; }
    const T* e = emb + (size_t)tok * dm;
    float* xr = x + (size_t)q * dm;
    // four float4 groups a thread in flight, then their stores
    constexpr int B = 4;
    for (int i0 = threadIdx.x * 4; i0 < dm; i0 += B * blockDim.x * 4) {
        float4 v[B];
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const int i = i0 + k * blockDim.x * 4;
            if (i < dm) v[k] = load4<T>(e + i);
        }
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const int i = i0 + k * blockDim.x * 4;
            if (i < dm) *reinterpret_cast<float4*>(xr + i) = v[k];
        }
    }
}

// ---------------------------------------------------------------------------
// RMSNorm: y = x / sqrt(mean(x^2) + eps) * g, one block per row, fixed
// reduction order.  gather=1 reads row need[i] and writes row i.  First, the
// split tiles the last residual GEMM left (resid) are added to x: x += the
// segments' partials in K order, and x is written back.
// ---------------------------------------------------------------------------
// the segments of a split tile summed in K order like la_split_sum4, the
// first eight loads issued together (a row of at most one float4 a thread
// has the registers for them)
__device__ __forceinline__ float4 split_sum4_wide(const LaSplit& s, int t, int y, size_t off, int nseg) {
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k < nseg) v[k] = __ldcg(reinterpret_cast<const float4*>(la_split_rec(s, t, y, k, 0) + off));
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k < nseg) {
            r.x = __fadd_rn(r.x, v[k].x);
            r.y = __fadd_rn(r.y, v[k].y);
            r.z = __fadd_rn(r.z, v[k].z);
            r.w = __fadd_rn(r.w, v[k].w);
        }
    for (int s0 = 8; s0 < nseg; s0 += 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (s0 + k < nseg) v[k] = __ldcg(reinterpret_cast<const float4*>(la_split_rec(s, t, y, s0 + k, 0) + off));
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (s0 + k < nseg) {
                r.x = __fadd_rn(r.x, v[k].x);
                r.y = __fadd_rn(r.y, v[k].y);
                r.z = __fadd_rn(r.z, v[k].z);
                r.w = __fadd_rn(r.w, v[k].w);
            }
    }
    return r;
}

template <typename T, int MAXV>
__global__ void __launch_bounds__(1024) k_rmsnorm(LaDev d, float* x, const T* g, T* y, int dm, float eps, int sel,
                                                 int gather, LaSplit resid) {
    LaTl la_tl_(LA_TL_RMSNORM, d.tl);
    const LaHdr* h = d.hdr;
    if (skip_call(h, sel)) return;       // header fields: readable before the wait (la_common.cuh)
    const int row = blockIdx.x;
    if (row >= rows_of(h, sel)) return;
    // the row stays in registers: up to MAXV float4 per thread (256 threads
    // for d_model <= 2048, 1024 threads up to 8192)
    float4 v[MAXV], add[MAXV], gv[MAXV];
    bool upd[MAXV];
    // the gains (weights) are read before the wait, the row after it
#pragma unroll
    for (int k = 0; k < MAXV; ++k) {
        const int i = (k * blockDim.x + threadIdx.x) * 4;
        if (i < dm) gv[k] = load4<T>(g + i);
    }
    la_pdl_wait();
    la_pdl_trigger();
    const int src = gather ? d.need[row] : row;
    float* xr = x + (size_t)src * dm;
    // every load of the row and its split partials is issued before the
    // first store of the updated row
#pragma unroll
    for (int k = 0; k < MAXV; ++k) {
        const int i = (k * blockDim.x + threadIdx.x) * 4;
        upd[k] = false;
        if (i < dm) {
            v[k] = *reinterpret_cast<const float4*>(xr + i);
            if (resid.ws) {
                const int tile = i >> 7;
                const int nseg = la_split_nseg(resid, tile);
                if (nseg > 1) {
                    const size_t off = (size_t)(src & 255) * 128 + (i & 127);
                    add[k] = MAXV == 1 ? split_sum4_wide(resid, tile, src >> 8, off, nseg)
                                       : la_split_sum4(resid, tile, src >> 8, off, nseg);
                    upd[k] = true;
                }
            }
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < MAXV; ++k) {
        const int i = (k * blockDim.x + threadIdx.x) * 4;
        if (i < dm) {
            if (upd[k]) {
                v[k].x = v[k].x + add[k].x;
                v[k].y = v[k].y + add[k].y;
                v[k].z = v[k].z + add[k].z;
                v[k].w = v[k].w + add[k].w;
                *reinterpret_cast<float4*>(xr + i) = v[k];
            }
            ss = fmaf(v[k].x, v[k].x, ss);
            ss = fmaf(v[k].y, v[k].y, ss);
            ss = fmaf(v[k].z, v[k].z, ss);
            ss = fmaf(v[k].w, v[k].w, ss);
        }
    }
    __shared__ float red[32];
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = ss;
    __syncthreads();
    if (w == 0) {
        float t = (l < (int)(blockDim.x >> 5)) ? red[l] : 0.f;
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (l == 0) red[0] = t;
    }
    __syncthreads();
    const float r = 1.0f / sqrtf(red[0] / (float)dm + eps);
    T* yr = y + (size_t)row * dm;
#pragma unroll
    for (int k = 0; k < MAXV; ++k) {
        const int i = (k * blockDim.x + threadIdx.x) * 4;
        if (i < dm) {
            yr[i + 0] = from_f<T>(v[k].x * r * gv[k].x);
            yr[i + 1] = from_f<T>(v[k].y * r * gv[k].y);
            yr[i + 2] = from_f<T>(v[k].z * r * gv[k].z);
            yr[i + 3] = from_f<T>(v[k].w * r * gv[k].w);
        }
    }
}

// ---------------------------------------------------------------------------
// RoPE (rotate-half) on q and k at each row's logical position; q goes to
// qbuf [H][Qcap][dh]; k, v go to kdst/vdst [H][stride][dh] at the row's
// packed index (temporary rows of the call) or, in a prefill, at its
// position in the cache.
// ---------------------------------------------------------------------------
// value n of row q of the QKV output: stored, or the sum of a split tile's
// segments rounded as the GEMM's store would round it
template <typename T>
__device__ __forceinline__ T qkv_at(const T* row, int q, int n, const LaSplit& sp) {
    const int nseg = sp.ws ? la_split_nseg(sp, n >> 7) : 1;
    if (nseg <= 1) return row[n];
    return from_f<T>(la_split_sum(sp, n >> 7, q >> 8, 0, (size_t)(q & 255) * 128 + (n & 127), nseg));
}

template <typename T>
__global__ void k_rope_kv(LaDev d, const T* qkv, const float* rcos, const float* rsin, T* qbuf, T* kdst, T* vdst,
                          int H, int dh, int sel, int Qcap, int stride, LaSplit sp) {
    LaTl la_tl_(LA_TL_ROPE_KV, d.tl);
    const LaHdr* h = d.hdr;
    if (skip_call(h, sel)) return;       // header fields: readable before the wait (la_common.cuh)
    const int q = blockIdx.x;
    if (q >= rows_of(h, sel)) return;
    const int half = dh >> 1;
    // blockDim = RH heads x half threads
    const int hh = blockIdx.y * (blockDim.x / half) + threadIdx.x / half, i = threadIdx.x % half;
    // the row's position (pack or chunk kernel) and its rotation (a table
    // written at init) are read before the wait; the QKV output after it
    const int pos = d.row_pos[q];
    const float c = rcos[(size_t)pos * half + i], s = rsin[(size_t)pos * half + i];
    la_pdl_wait();
    la_pdl_trigger();
    if (hh >= H) return;
    const int HD = H * dh;
    const T* row = qkv + (size_t)q * 3 * HD;
    const int nq = hh * dh, nk = HD + hh * dh, nv = 2 * HD + hh * dh;
    float qa = to_f(qkv_at(row, q, nq + i, sp)), qb = to_f(qkv_at(row, q, nq + i + half, sp));
    float ka = to_f(qkv_at(row, q, nk + i, sp)), kb = to_f(qkv_at(row, q, nk + i + half, sp));
    // all loads before the first store (the stores may alias them as far as the compiler knows)
    const T va = qkv_at(row, q, nv + i, sp), vb = qkv_at(row, q, nv + i + half, sp);
    T* qo = qbuf + ((size_t)hh * Qcap + q) * dh;
    qo[i] = from_f<T>(qa * c - qb * s);
    qo[i + half] = from_f<T>(qb * c + qa * s);
    int slot = (sel == 1) ? pos : q;
    T* ko = kdst + ((size_t)hh * stride + slot) * dh;
    T* vo = vdst + ((size_t)hh * stride + slot) * dh;
    ko[i] = from_f<T>(ka * c - kb * s);
    ko[i + half] = from_f<T>(kb * c + ka * s);
    vo[i] = va;
    vo[i + half] = vb;
}

// bf16 models: the same operation with eight dimensions per thread (four
// consecutive ones of the first half and their rotation partners), all
// partial loads as float4 and in flight before the first store, so the grid
// (a quarter of the threads of k_rope_kv) is resident at once.  Every output
// element takes the same arithmetic as in k_rope_kv.
// grid (rows, ceil(H / heads per CTA)); blockDim = heads per CTA x dh/8
__global__ void __launch_bounds__(256) k_rope_kv4(LaDev d, const __nv_bfloat16* qkv, const float* rcos,
                                                  const float* rsin, __nv_bfloat16* qbuf, __nv_bfloat16* kdst,
                                                  __nv_bfloat16* vdst, int H, int dh, int sel, int Qcap, int stride,
                                                  LaSplit sp) {
    LaTl la_tl_(LA_TL_ROPE_KV4, d.tl);
    const LaHdr* h = d.hdr;
    if (skip_call(h, sel)) return;       // header fields: readable before the wait (la_common.cuh)
    const int q = blockIdx.x;
    if (q >= rows_of(h, sel)) return;
    const int half = dh >> 1, tph = dh >> 3;
    const int hh = blockIdx.y * (blockDim.x / tph) + threadIdx.x / tph, i = (threadIdx.x % tph) * 4;
    const int pos = d.row_pos[q];
    const float4 c = *reinterpret_cast<const float4*>(rcos + (size_t)pos * half + i);
    const float4 s = *reinterpret_cast<const float4*>(rsin + (size_t)pos * half + i);
    // segments of the six column groups' tiles (the rotation partner sits in
    // the next tile when a head is wider than a tile)
    const int HD = H * dh, hc = hh < H ? hh : H - 1;
    const int nq = hc * dh, nk = HD + hc * dh, nv = 2 * HD + hc * dh;
    auto segs = [&](int n) { return sp.ws ? la_split_nseg(sp, n >> 7) : 1; };
    const int sqa = segs(nq + i), ska = segs(nk + i), sva = segs(nv + i);
    const int sqb = dh > 128 ? segs(nq + i + half) : sqa, skb = dh > 128 ? segs(nk + i + half) : ska;
    const int svb = dh > 128 ? segs(nv + i + half) : sva;
    la_pdl_wait();
    la_pdl_trigger();
    if (hh >= H) return;
    const __nv_bfloat16* row = qkv + (size_t)q * 3 * HD;
    const float4 qa = la_qkv_at4(row, q, nq + i, sp, sqa), qb = la_qkv_at4(row, q, nq + i + half, sp, sqb);
    const float4 ka = la_qkv_at4(row, q, nk + i, sp, ska), kb = la_qkv_at4(row, q, nk + i + half, sp, skb);
    const float4 va = la_qkv_at4(row, q, nv + i, sp, sva), vb = la_qkv_at4(row, q, nv + i + half, sp, svb);
    __nv_bfloat16* qo = qbuf + ((size_t)hh * Qcap + q) * dh;
    la_rope4_store(qo + i, qo + i + half, qa, qb, c, s);
    const int slot = (sel == 1) ? pos : q;
    __nv_bfloat16* ko = kdst + ((size_t)hh * stride + slot) * dh;
    __nv_bfloat16* vo = vdst + ((size_t)hh * stride + slot) * dh;
    la_rope4_store(ko + i, ko + i + half, ka, kb, c, s);
    *reinterpret_cast<uint2*>(vo + i) = la_pack_bf16x4(va.x, va.y, va.z, va.w);
    *reinterpret_cast<uint2*>(vo + i + half) = la_pack_bf16x4(vb.x, vb.y, vb.z, vb.w);
}

// SwiGLU of the gate/up GEMM's split tiles: act = silu(gate) * up with gate
// and up the sums of the segments' two accumulator planes.  One thread per
// four consecutive columns of a row (float4 partial loads, all in flight at once).
__global__ void __launch_bounds__(256) k_swiglu_split(LaDev d, LaSplit sp, __nv_bfloat16* act, int ldo, int sel) {
    LaTl la_tl_(LA_TL_SWIGLU, d.tl);
    const LaHdr* h = d.hdr;
    if (skip_call(h, sel)) return;       // header fields: readable before the wait (la_common.cuh)
    const int q = blockIdx.x;
    if (q >= rows_of(h, sel)) return;
    la_pdl_wait();
    la_pdl_trigger();
    const int n_cols = sp.n_tiles * 128;
    const int y = q >> 8;
    const size_t rowoff = (size_t)(q & 255) * 128;
    const int c4 = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
    if (c4 < n_cols) {
        const int tile = c4 >> 7;
        const int nseg = la_split_nseg(sp, tile);
        if (nseg <= 1) return;
        const size_t off = rowoff + (c4 & 127);
        const float4 v = la_split_sum4(sp, tile, y, off, nseg, 0);
        const float4 u = la_split_sum4(sp, tile, y, off, nseg, 1);
        __nv_bfloat162 r01 = __floats2bfloat162_rn(v.x / (1.0f + expf(-v.x)) * u.x, v.y / (1.0f + expf(-v.y)) * u.y);
        __nv_bfloat162 r23 = __floats2bfloat162_rn(v.z / (1.0f + expf(-v.z)) * u.z, v.w / (1.0f + expf(-v.w)) * u.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&r01);
        pk.y = *reinterpret_cast<uint32_t*>(&r23);
        *reinterpret_cast<uint2*>(act + (size_t)q * ldo + c4) = pk;
    }
}

// ---------------------------------------------------------------------------
// Masked attention (CUDA cores).  One CTA per (head, block of rows).  Every
// row sees one key per logical position 0..pos: positions below the
// committed length K come from the cache, positions K..pos from the call's
// temporary rows on the row's own path (row_path), which encodes the
// branch visibility of M7.3 §0x04A without a mask tensor.  Keys are taken in
// chunks of 32 aligned to absolute positions; chunks below every row's
// frontier are staged once in shared memory for all rows of the CTA.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int DPL, int RPW>
struct AttnState {
    float m[RPW], l[RPW], o[RPW][DPL];
};

// One online-softmax step over a chunk of 32 keys (lane j holds key j's
// score).  Both the shared-chunk and the gathered-key paths call this one
// function, and it uses only explicitly rounded operations, so a row's
// result does not depend on which path delivered its keys.
template <int DPL, typename VGet>
__device__ __forceinline__ void softmax_chunk(float s, bool valid, float& m, float& l, float (&o)[DPL], VGet vget) {
    const float cmax = warp_max(valid ? s : -INFINITY);
    const float mn = fmaxf(m, cmax);
    const float p = valid ? expf(__fsub_rn(s, mn)) : 0.f;
    const float corr = (m == -INFINITY) ? 0.f : expf(__fsub_rn(m, mn));
    l = fmaf(l, corr, warp_sum(p));
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = __fmul_rn(o[e], corr);
    for (int j = 0; j < 32; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
        if (pj != 0.f) {
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[e] = fmaf(pj, vget(j, e), o[e]);
        }
    }
    m = mn;
}

template <typename T, int DH, int RPW>
__global__ void __launch_bounds__(256) k_attention(LaDev d, const T* qbuf, const T* kc, const T* vc, const T* kt,
                                                   const T* vt, T* out, int H, int sel, int Qcap, int max_ctx,
                                                   int Qmax, float scale) {
    LaTl la_tl_(LA_TL_ATTENTION, d.tl);
    constexpr int DPL = DH / 32;
    constexpr int NW = 8;
    constexpr int RPC = NW * RPW;
    const LaHdr* h = d.hdr;
    if (skip_call(h, sel)) return;
    const int rows = rows_of(h, sel);
    const int hh = blockIdx.x;
    const int r0 = blockIdx.y * RPC;
    if (r0 >= rows) return;
    const int prefill = (sel == 1);
    const int K = prefill ? 0 : h->K;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    extern __shared__ float sm[];
    float* q_s = sm;                       // [RPC][DH]
    float* kt_s = q_s + RPC * DH;          // [DH][33]
    float* v_s = kt_s + DH * 33;           // [32][DH]

    const T* kc_h = kc + (size_t)hh * max_ctx * DH;
    const T* vc_h = vc + (size_t)hh * max_ctx * DH;
    const T* kt_h = kt + (size_t)hh * Qmax * DH;
    const T* vt_h = vt + (size_t)hh * Qmax * DH;

    int minpos = 0x7fffffff, maxpos = -1;
    for (int r = r0; r < min(rows, r0 + RPC); ++r) {
        int p = d.row_pos[r];
        minpos = min(minpos, p);
        maxpos = max(maxpos, p);
    }
    // queries into shared memory (fp32)
    for (int i = threadIdx.x; i < RPC * DH; i += blockDim.x) {
        int r = r0 + i / DH;
        q_s[i] = (r < rows) ? to_f(qbuf[((size_t)hh * Qcap + r) * DH + (i % DH)]) : 0.f;
    }
    // chunks below `shared_end` hold committed keys visible to every row here
    const int shared_end = prefill ? (minpos + 1) : K;
    const int n_shared = shared_end / 32;

    AttnState<DPL, RPW> st;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        st.m[i] = -INFINITY; st.l[i] = 0.f;
#pragma unroll
        for (int j = 0; j < DPL; ++j) st.o[i][j] = 0.f;
    }
    int myrow[RPW], mypos[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        int r = r0 + warp + i * NW;
        myrow[i] = r;
        mypos[i] = (r < rows) ? d.row_pos[r] : -1;
    }

    for (int c = 0; c < n_shared; ++c) {
        __syncthreads();
        for (int i = threadIdx.x; i < 32 * DH; i += blockDim.x) {
            int j = i / DH, dd = i % DH;
            size_t src = (size_t)(c * 32 + j) * DH + dd;
            kt_s[dd * 33 + j] = to_f(kc_h[src]);
            v_s[j * DH + dd] = to_f(vc_h[src]);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            if (mypos[i] < 0) continue;
            const float* qv = q_s + (myrow[i] - r0) * DH;
            float acc = 0.f;
#pragma unroll 8
            for (int dd = 0; dd < DH; ++dd) acc = fmaf(qv[dd], kt_s[dd * 33 + lane], acc);
            softmax_chunk<DPL>(__fmul_rn(acc, scale), true, st.m[i], st.l[i], st.o[i],
                               [&](int j, int e) { return v_s[j * DH + lane * DPL + e]; });
        }
    }
    // remaining chunks: keys gathered per row (committed or the row's own path)
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        if (mypos[i] < 0) continue;
        const int r = myrow[i], pos = mypos[i];
        const int Kr = prefill ? pos + 1 : K;       // keys below Kr are in the cache
        const int* path = d.row_path + (size_t)r * d.PMAX;
        const float* qv = q_s + (r - r0) * DH;
        for (int c = n_shared; c * 32 <= pos; ++c) {
            int p = c * 32 + lane;
            bool valid = p <= pos;
            const T* kp = nullptr;
            const T* vp = nullptr;
            if (valid) {
                if (p < Kr) { kp = kc_h + (size_t)p * DH; vp = vc_h + (size_t)p * DH; }
                else {
                    int src = path[p - K];
                    kp = kt_h + (size_t)src * DH; vp = vt_h + (size_t)src * DH;
                }
            }
            float s = -INFINITY;
            if (valid) {
                float acc = 0.f;
#pragma unroll 8
                for (int dd = 0; dd < DH; ++dd) acc = fmaf(qv[dd], to_f(kp[dd]), acc);
                s = __fmul_rn(acc, scale);
            }
            softmax_chunk<DPL>(s, valid, st.m[i], st.l[i], st.o[i], [&](int j, int e) {
                const T* vj = (const T*)__shfl_sync(0xffffffffu, (unsigned long long)vp, j);
                return to_f(vj[lane * DPL + e]);
            });
        }
        float inv = 1.0f / st.l[i];
        T* op = out + (size_t)r * H * DH + hh * DH + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) op[e] = from_f<T>(__fmul_rn(st.o[i][e], inv));
    }
}

// ---------------------------------------------------------------------------
// CUDA-core GEMM: Y[q][n] = sum_k X[q][k] W[n][k], k ascending per output
// (one FMA chain), tile 64 n x 32 q, fp32 accumulation.  Used for the fp32
// model and as the reference kernel of the tensor-core GEMM.
// ---------------------------------------------------------------------------
template <typename T, int MODE>
__global__ void __launch_bounds__(256) k_gemm_ffma(LaDev d, const T* X, int ldx, const T* Wm, const T* W2, int K,
                                                   int Nout, void* out, int ldo, int sel) {
    LaTl la_tl_(LA_TL_GEMM_FFMA, d.tl);
    const LaHdr* h = d.hdr;
    if (skip_call(h, sel)) return;
    const int rows = rows_of(h, sel);
    const int n0 = blockIdx.x * 64, q0 = blockIdx.y * 32;
    if (q0 >= rows) return;
    __shared__ float Ws[32][65];
    __shared__ float W2s[MODE == GEMM_SWIGLU ? 32 : 1][65];
    __shared__ float Xs[32][33];
    const int tid = threadIdx.x, nl = tid & 63, qg = tid >> 6;
    float acc[8], acc2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { acc[i] = 0.f; acc2[i] = 0.f; }
    for (int k0 = 0; k0 < K; k0 += 32) {
        for (int i = tid; i < 64 * 32; i += 256) {
            int n = i >> 5, k = i & 31;
            Ws[k][n] = to_f(Wm[(size_t)(n0 + n) * K + k0 + k]);
            if (MODE == GEMM_SWIGLU) W2s[k][n] = to_f(W2[(size_t)(n0 + n) * K + k0 + k]);
        }
        for (int i = tid; i < 32 * 32; i += 256) {
            int q = i >> 5, k = i & 31;
            Xs[q][k] = (q0 + q < rows) ? to_f(X[(size_t)(q0 + q) * ldx + k0 + k]) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < 32; ++kk) {
            float w = Ws[kk][nl];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, Xs[qg * 8 + i][kk], acc[i]);
            if (MODE == GEMM_SWIGLU) {
                float w2 = W2s[kk][nl];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc2[i] = fmaf(w2, Xs[qg * 8 + i][kk], acc2[i]);
            }
        }
        __syncthreads();
    }
    const int n = n0 + nl;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int q = q0 + qg * 8 + i;
        if (q >= rows) continue;
        size_t o = (size_t)q * ldo + n;
        if (MODE == GEMM_STORE) ((T*)out)[o] = from_f<T>(acc[i]);
        else if (MODE == GEMM_RESID) ((float*)out)[o] += acc[i];
        else if (MODE == GEMM_SWIGLU) {
            float g = acc[i];
            ((T*)out)[o] = from_f<T>(g / (1.0f + expf(-g)) * acc2[i]);
        } else if (MODE == GEMM_LOGITS) ((float*)out)[o] = acc[i];
    }
}

// ---------------------------------------------------------------------------
// argmax over fp32 logit rows, lowest id among maxima
// ---------------------------------------------------------------------------
__device__ __forceinline__ void better(float& v, int& i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
}
__global__ void k_argmax_rows(LaDev d, const float* logits, int V, int sel) {
    LaTl la_tl_(LA_TL_ARGMAX_ROWS, d.tl);
    la_pdl_wait();
    la_pdl_trigger();
    const LaHdr* h = d.hdr;
    if (skip_call(h, sel)) return;
    int row = blockIdx.x;
    if (row >= rows_of(h, sel)) return;
    const float* x = logits + (size_t)row * V;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int v = threadIdx.x; v < V; v += blockDim.x) better(bv, bi, x[v], v);
    for (int o = 16; o > 0; o >>= 1) {
        float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        better(bv, bi, v2, i2);
    }
    __shared__ float sv[32];
    __shared__ int si[32];
    int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) { sv[w] = bv; si[w] = bi; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int k = 1; k < (int)(blockDim.x >> 5); ++k) better(bv, bi, sv[k], si[k]);
        d.argmax[row] = bi;
    }
}

// partial (value, index) per (vocab tile, row) -> argmax per row
__global__ void k_argmax_reduce(LaDev d, const float* pv, const int* pi, int n_tiles, int stride, int sel) {
    LaTl la_tl_(LA_TL_ARGMAX_REDUCE, d.tl);
    la_pdl_wait();
    la_pdl_trigger();
    const LaHdr* h = d.hdr;
    if (skip_call(h, sel)) return;
    int row = blockIdx.x;
    if (row >= rows_of(h, sel)) return;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int t = threadIdx.x; t < n_tiles; t += blockDim.x) better(bv, bi, pv[(size_t)t * stride + row], pi[(size_t)t * stride + row]);
    for (int o = 16; o > 0; o >>= 1) {
        float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        better(bv, bi, v2, i2);
    }
    __shared__ float sv[32];
    __shared__ int si[32];
    int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) { sv[w] = bv; si[w] = bi; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int k = 1; k < (int)(blockDim.x >> 5); ++k) better(bv, bi, sv[k], si[k]);
        d.argmax[row] = bi;
    }
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
void la_launch_rope_table(float* rcos, float* rsin, int n_pos, int dh, double theta, cudaStream_t st) {
    int half = dh / 2, n = n_pos * half;
    k_rope_table<<<(n + 255) / 256, 256, 0, st>>>(rcos, rsin, n_pos, half, theta, dh);
}

template <typename T>
void la_launch_embed_t(const LaDev& d, cudaStream_t st, const void* emb, float* x, int dm, int sel, int rows_cap) {
    la_launch_pdl(k_embed<T>, dim3(rows_cap), dim3(256), 0, st, d, (const T*)emb, x, dm, sel);
}
void la_launch_embed(const LaDev& d, cudaStream_t st, int dtype, const void* emb, float* x, int dm, int sel, int rows_cap) {
    if (dtype == LA_F32) la_launch_embed_t<float>(d, st, emb, x, dm, sel, rows_cap);
    else la_launch_embed_t<__nv_bfloat16>(d, st, emb, x, dm, sel, rows_cap);
}

void la_launch_rmsnorm(const LaDev& d, cudaStream_t st, int dtype, float* x, const void* g, void* y, int dm,
                       float eps, int sel, int gather, int rows_cap, const LaSplit& resid) {
    const dim3 threads(dm > 2048 ? 1024 : 256);
    const bool one = dm <= 4 * (int)threads.x;           // one float4 a thread
    if (dtype == LA_F32)
        la_launch_pdl(one ? k_rmsnorm<float, 1> : k_rmsnorm<float, 2>, dim3(rows_cap), threads, 0, st, d, x,
                      (const float*)g, (float*)y, dm, eps, sel, gather, resid);
    else
        la_launch_pdl(one ? k_rmsnorm<__nv_bfloat16, 1> : k_rmsnorm<__nv_bfloat16, 2>, dim3(rows_cap), threads, 0,
                      st, d, x, (const __nv_bfloat16*)g, (__nv_bfloat16*)y, dm, eps, sel, gather, resid);
}

void la_launch_rope_kv(const LaDev& d, cudaStream_t st, int dtype, const void* qkv, const float* rcos, const float* rsin,
                       void* qbuf, void* kdst, void* vdst, int H, int dh, int sel, int Qcap, int stride, int rows_cap,
                       const LaSplit& sp) {
    if (dtype != LA_F32 && dh % 8 == 0 && dh <= 256) {
        const int hpc = H < 256 / (dh / 8) ? H : 256 / (dh / 8);   // heads per CTA
        la_launch_pdl(k_rope_kv4, dim3(rows_cap, (H + hpc - 1) / hpc), dim3(hpc * (dh / 8)), 0, st, d,
                      (const __nv_bfloat16*)qkv, rcos, rsin, (__nv_bfloat16*)qbuf, (__nv_bfloat16*)kdst,
                      (__nv_bfloat16*)vdst, H, dh, sel, Qcap, stride, sp);
        return;
    }
    const int rh = (H % 4 == 0) ? 4 : 1;      // heads per CTA
    dim3 g(rows_cap, H / rh);
    if (dtype == LA_F32) {
        k_rope_kv<float><<<g, rh * dh / 2, 0, st>>>(d, (const float*)qkv, rcos, rsin, (float*)qbuf, (float*)kdst,
                                                    (float*)vdst, H, dh, sel, Qcap, stride, sp);
        la_note_launch();
    } else
        la_launch_pdl(k_rope_kv<__nv_bfloat16>, g, dim3(rh * dh / 2), 0, st, d, (const __nv_bfloat16*)qkv, rcos, rsin,
                      (__nv_bfloat16*)qbuf, (__nv_bfloat16*)kdst, (__nv_bfloat16*)vdst, H, dh, sel, Qcap, stride, sp);
}

void la_launch_swiglu_split(const LaDev& d, cudaStream_t st, const LaSplit& sp, void* act, int ldo, int sel,
                            int rows_cap) {
    const int chunks = sp.n_tiles * 32;     // float4 columns per row
    la_launch_pdl(k_swiglu_split, dim3(rows_cap, (chunks + 255) / 256), dim3(256), 0, st, d, sp, (__nv_bfloat16*)act, ldo,
                  sel);
}

template <typename T, int DH, int RPW>
static cudaError_t attn_t(const LaDev& d, cudaStream_t st, const void* qbuf, const void* kc, const void* vc,
                          const void* kt, const void* vt, void* out, int H, int sel, int Qcap, int max_ctx, int Qmax,
                          int rows_cap) {
    constexpr int RPC = 8 * RPW;
    size_t smem = (size_t)(RPC * DH + DH * 33 + 32 * DH) * sizeof(float);
    auto kern = k_attention<T, DH, RPW>;
    static bool attr_done = false;     // set once, before any stream capture
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    dim3 g(H, (rows_cap + RPC - 1) / RPC);
    kern<<<g, 256, smem, st>>>(d, (const T*)qbuf, (const T*)kc, (const T*)vc, (const T*)kt, (const T*)vt, (T*)out, H,
                                sel, Qcap, max_ctx, Qmax, 1.0f / sqrtf((float)DH));
    la_note_launch();
    return cudaGetLastError();
}

cudaError_t la_launch_attention(const LaDev& d, cudaStream_t st, int dtype, int dh, const void* qbuf, const void* kc,
                                const void* vc, const void* kt, const void* vt, void* out, int H, int sel, int Qcap,
                                int max_ctx, int Qmax, int rows_cap) {
    if (dtype == LA_F32) {
        if (dh == 32) return attn_t<float, 32, 4>(d, st, qbuf, kc, vc, kt, vt, out, H, sel, Qcap, max_ctx, Qmax, rows_cap);
        if (dh == 128) return attn_t<float, 128, 4>(d, st, qbuf, kc, vc, kt, vt, out, H, sel, Qcap, max_ctx, Qmax, rows_cap);
    } else {
        if (dh == 32) return attn_t<__nv_bfloat16, 32, 4>(d, st, qbuf, kc, vc, kt, vt, out, H, sel, Qcap, max_ctx, Qmax, rows_cap);
        if (dh == 128) return attn_t<__nv_bfloat16, 128, 4>(d, st, qbuf, kc, vc, kt, vt, out, H, sel, Qcap, max_ctx, Qmax, rows_cap);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
static void gemm_ffma_t(const LaDev& d, cudaStream_t st, int mode, const void* X, int ldx, const void* Wm, const void* W2,
                        int K, int Nout, void* out, int ldo, int sel, int rows_cap) {
    dim3 g(Nout / 64, (rows_cap + 31) / 32);
    switch (mode) {
        case GEMM_STORE: k_gemm_ffma<T, GEMM_STORE><<<g, 256, 0, st>>>(d, (const T*)X, ldx, (const T*)Wm, nullptr, K, Nout, out, ldo, sel); break;
        case GEMM_RESID: k_gemm_ffma<T, GEMM_RESID><<<g, 256, 0, st>>>(d, (const T*)X, ldx, (const T*)Wm, nullptr, K, Nout, out, ldo, sel); break;
        case GEMM_SWIGLU: k_gemm_ffma<T, GEMM_SWIGLU><<<g, 256, 0, st>>>(d, (const T*)X, ldx, (const T*)Wm, (const T*)W2, K, Nout, out, ldo, sel); break;
        case GEMM_LOGITS: k_gemm_ffma<T, GEMM_LOGITS><<<g, 256, 0, st>>>(d, (const T*)X, ldx, (const T*)Wm, nullptr, K, Nout, out, ldo, sel); break;
    }
    la_note_launch();
}
void la_launch_gemm_ffma(const LaDev& d, cudaStream_t st, int dtype, int mode, const void* X, int ldx, const void* Wm,
                         const void* W2, int K, int Nout, void* out, int ldo, int sel, int rows_cap) {
    if (dtype == LA_F32) gemm_ffma_t<float>(d, st, mode, X, ldx, Wm, W2, K, Nout, out, ldo, sel, rows_cap);
    else gemm_ffma_t<__nv_bfloat16>(d, st, mode, X, ldx, Wm, W2, K, Nout, out, ldo, sel, rows_cap);
}

void la_launch_argmax_rows(const LaDev& d, cudaStream_t st, const float* logits, int V, int sel, int rows_cap) {
    k_argmax_rows<<<rows_cap, 256, 0, st>>>(d, logits, V, sel);
    la_note_launch();
}
void la_launch_argmax_reduce(const LaDev& d, cudaStream_t st, const float* pv, const int* pi, int n_tiles, int stride,
                             int sel, int rows_cap) {
    la_launch_pdl(k_argmax_reduce, dim3(rows_cap), dim3(256), 0, st, d, pv, pi, n_tiles, stride, sel);
}
