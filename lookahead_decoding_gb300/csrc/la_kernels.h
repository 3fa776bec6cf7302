// Host-side launchers of the liblookahead kernels (internal to the library).
#pragma once
#include <cuda_runtime.h>
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

struct LaDev;
struct LaHdr;
struct LaTlRec;

// epilogues of the GEMMs
#define GEMM_STORE 0   // out[q][n] = acc                       (element type of the model)
#define GEMM_RESID 1   // out[q][n] += acc                      (fp32 residual stream)
#define GEMM_SWIGLU 2  // out[q][n] = silu(acc_gate) * acc_up   (element type of the model)
#define GEMM_LOGITS 3  // out[q][n] = acc (fp32); tensor-core variant adds argmax partials

// row-count selectors read from the device header
#define SEL_CALL 0     // rows of the packed call (Q)
#define SEL_PREFILL 1  // rows of the current prefill chunk
#define SEL_NEED 2     // rows whose logits are read

void la_launch_begin(const LaDev& d, cudaStream_t st, int mode, int W, int N, int G, int sampling,
                     float temperature, float top_p, uint64_t seed, int max_out, int opts);
void la_launch_pack(const LaDev& d, cudaStream_t st);
void la_launch_publish(const LaDev& d, cudaStream_t st, int verdict_given);
void la_launch_commit(const LaDev& d, cudaStream_t st, void* cache, void* temp, int planes, int n_heads,
                      int head_bytes, int max_ctx, int Qmax);
void la_launch_inject_map(const LaDev& d, cudaStream_t st, const int32_t* argmax_rows, const float* logits_rows,
                          float* logits_need, int V);
void la_launch_prefill_rows(const LaDev& d, cudaStream_t st, int c0, int n);
void la_launch_prefill_need(const LaDev& d, cudaStream_t st, int last_local);
void la_launch_prefill_finish(const LaDev& d, cudaStream_t st, int P);

// Split tiles of a tensor-core GEMM left for its consumer.  A GEMM launched
// with `defer` writes each split tile's per-segment fp32 partials and stops;
// the kernel that reads the GEMM's output adds the segments in K order
// (starting from 0, the same additions the GEMM would have made) before its
// own epilogue: RoPE after QKV, the residual add + RMSNorm after O and down,
// SwiGLU after gate/up.  ws == nullptr: no split tiles to reduce.
struct LaSplit {
    const float* ws;      // partial records [unit tile + y * n_tiles][max_seg][nA][256][128]
    int n_tiles, k_tiles, P, max_seg, nA;
    int pair;             // 1: a unit tile is two adjacent output tiles (planes 0 and 1)
};

// segments of output tile t (1 = the GEMM wrote the tile itself)
__host__ __device__ __forceinline__ int la_split_nseg(const LaSplit& s, int t) {
    const int ut = s.pair ? (t >> 1) : t;
    const long long T = (long long)s.n_tiles * s.k_tiles;
    const long long u0 = (long long)ut * s.k_tiles, u1 = u0 + s.k_tiles - 1;
    const int c0 = (int)(((u0 + 1) * s.P - 1) / T), c1 = (int)(((u1 + 1) * s.P - 1) / T);
    return c1 - c0 + 1;
}
// the record of segment sg, accumulator plane pl, row chunk y of output tile
// t (a unit of two tiles: the plane is the tile's place in it)
__host__ __device__ __forceinline__ const float* la_split_rec(const LaSplit& s, int t, int y, int sg, int pl) {
    const int ut = s.pair ? (t >> 1) : t, plane = s.pair ? (t & 1) : pl;
    return s.ws + ((((size_t)ut + (size_t)y * s.n_tiles) * s.max_seg + sg) * s.nA + plane) * (size_t)(256 * 128);
}

#ifdef __CUDACC__
// Sum over the segments (K order, from 0) of the element at `off` of plane pl;
// the loads of the segments go out four at a time (only the tile's own
// segments: every request goes to L2), each group added in order.
__device__ __forceinline__ float la_split_sum(const LaSplit& s, int t, int y, int pl, size_t off, int nseg) {
    float r = 0.f;
    for (int s0 = 0; s0 < nseg; s0 += 4) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (s0 + k < nseg) v[k] = __ldcg(la_split_rec(s, t, y, s0 + k, pl) + off);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (s0 + k < nseg) r = __fadd_rn(r, v[k]);
    }
    return r;
}
// the same for four consecutive elements (off a multiple of 4)
__device__ __forceinline__ float4 la_split_sum4(const LaSplit& s, int t, int y, size_t off, int nseg, int pl = 0) {
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (k < nseg) v[k] = __ldcg(reinterpret_cast<const float4*>(la_split_rec(s, t, y, k, pl) + off));
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (k < nseg) {
            r.x = __fadd_rn(r.x, v[k].x);
            r.y = __fadd_rn(r.y, v[k].y);
            r.z = __fadd_rn(r.z, v[k].z);
            r.w = __fadd_rn(r.w, v[k].w);
        }
    for (int s0 = 4; s0 < nseg; s0 += 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (s0 + k < nseg) v[k] = __ldcg(reinterpret_cast<const float4*>(la_split_rec(s, t, y, s0 + k, pl) + off));
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

// RoPE of bf16 models on four consecutive dimensions i..i+3 (< dh/2) and
// their rotation partners, shared by the RoPE kernel and the attention that
// folds it in: values as the QKV GEMM's bf16 store would have rounded them,
// rotation with explicit roundings (no contraction), so every kernel that
// applies it gets the same bits.
__device__ __forceinline__ float la_bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// four consecutive values n .. n+3 (n % 4 == 0) of row q of the QKV output
__device__ __forceinline__ float4 la_qkv_at4(const __nv_bfloat16* row, int q, int n, const LaSplit& sp, int nseg) {
    if (nseg <= 1) {
        const uint2 u = *reinterpret_cast<const uint2*>(row + n);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
    const float4 s = la_split_sum4(sp, n >> 7, q >> 8, (size_t)(q & 255) * 128 + (n & 127), nseg);
    return make_float4(la_bf16_round(s.x), la_bf16_round(s.y), la_bf16_round(s.z), la_bf16_round(s.w));
}

__device__ __forceinline__ uint2 la_pack_bf16x4(float a, float b, float c, float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    return u;
}

__device__ __forceinline__ float la_rope_lo(float a, float b, float c, float s) {
    return __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s));
}
__device__ __forceinline__ float la_rope_hi(float a, float b, float c, float s) {
    return __fadd_rn(__fmul_rn(b, c), __fmul_rn(a, s));
}
// (a, b) = dimensions i.. and i+dh/2.. of one head; stores the rotated pair as bf16
__device__ __forceinline__ void la_rope4_store(__nv_bfloat16* lo, __nv_bfloat16* hi, float4 a, float4 b, float4 c,
                                               float4 s) {
    *reinterpret_cast<uint2*>(lo) = la_pack_bf16x4(la_rope_lo(a.x, b.x, c.x, s.x), la_rope_lo(a.y, b.y, c.y, s.y),
                                                   la_rope_lo(a.z, b.z, c.z, s.z), la_rope_lo(a.w, b.w, c.w, s.w));
    *reinterpret_cast<uint2*>(hi) = la_pack_bf16x4(la_rope_hi(a.x, b.x, c.x, s.x), la_rope_hi(a.y, b.y, c.y, s.y),
                                                   la_rope_hi(a.z, b.z, c.z, s.z), la_rope_hi(a.w, b.w, c.w, s.w));
}
#endif

void la_launch_rope_table(float* rcos, float* rsin, int n_pos, int dh, double theta, cudaStream_t st);
void la_launch_embed(const LaDev& d, cudaStream_t st, int dtype, const void* emb, float* x, int dm, int sel, int rows_cap);
// resid: split tiles of the GEMM that last added to x (O or down), summed into x first
void la_launch_rmsnorm(const LaDev& d, cudaStream_t st, int dtype, float* x, const void* g, void* y, int dm,
                       float eps, int sel, int gather, int rows_cap, const LaSplit& resid);
// sp: split tiles of the QKV GEMM
void la_launch_rope_kv(const LaDev& d, cudaStream_t st, int dtype, const void* qkv, const float* rcos, const float* rsin,
                       void* qbuf, void* kdst, void* vdst, int H, int dh, int sel, int Qcap, int stride, int rows_cap,
                       const LaSplit& sp);
// act[q][n] = silu(gate) * up for the split tiles of the gate/up GEMM
void la_launch_swiglu_split(const LaDev& d, cudaStream_t st, const LaSplit& sp, void* act, int ldo, int sel,
                            int rows_cap);
cudaError_t la_launch_attention(const LaDev& d, cudaStream_t st, int dtype, int dh, const void* qbuf, const void* kc,
                                const void* vc, const void* kt, const void* vt, void* out, int H, int sel, int Qcap,
                                int max_ctx, int Qmax, int rows_cap);
void la_launch_gemm_ffma(const LaDev& d, cudaStream_t st, int dtype, int mode, const void* X, int ldx, const void* Wm,
                         const void* W2, int K, int Nout, void* out, int ldo, int sel, int rows_cap);
void la_launch_argmax_rows(const LaDev& d, cudaStream_t st, const float* logits, int V, int sel, int rows_cap);
void la_launch_argmax_reduce(const LaDev& d, cudaStream_t st, const float* pv, const int* pi, int n_tiles, int stride,
                             int sel, int rows_cap);

// tensor-core (tcgen05) bf16 GEMM: Y[q][n] = sum_k X[q][k] W[n][k]
struct TcGemm {
    CUtensorMap tmA;      // weights [Nout][K], box 64 x 128, 128B swizzle
    CUtensorMap tmA2;     // second weight matrix (SwiGLU up, or segment 1), else a copy of tmA
    CUtensorMap tmA3;     // segment 2 (QKV), else a copy of tmA
    CUtensorMap tmB;      // activations [rows_alloc][K], box 64 x 16, 128B swizzle
    CUtensorMap tmB32, tmB64, tmB128, tmB256;   // the same activations with taller boxes
    int mode, K, Nout, rows_cap;
    int seg_tiles;        // >0: tiles per weight segment (output columns concatenate the segments)
    int n_cta;            // persistent CTAs (one per SM)
    int max_seg;          // largest number of CTAs sharing one tile's K range
    void* out; int ldo;
    float* logits; int ld_logits;   // GEMM_LOGITS: optional fp32 logits
    void* wpack;          // unit-contiguous weight images (la_tc_pack), or null: the tensor maps
    int defer;            // 1: split tiles left as partials for the consumer (LaSplit)
    int ctr_off;          // first split-tile counter of this GEMM (counters are per GEMM)
    const void* act;      // the activation rows [rows_alloc][K] the tensor maps cover
    int pair;             // 1: units of two adjacent 128-row output tiles x one 64-column atom
                          // (packed weights only; not with GEMM_SWIGLU or GEMM_LOGITS)
};
#define LA_TC_CTR_PER_TILE 2   // ints per split-tile arrival counter (one 64-bit word)
struct TcWork {
    float* ws;            // partial tiles of K ranges shared by several CTAs
    size_t ws_floats;
    int* counters;        // LA_TC_CTR_PER_TILE ints per (GEMM, tile, q-chunk), zero-initialised, 8-byte aligned
    int n_counters;
    float* part_v;        // argmax partials [n_tiles][part_stride]
    int* part_i;
    int part_stride;
};

int la_tc_make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows);
int la_tc_make_act_maps(TcGemm* g, const void* base, int rows, int K);
// rows_cap: the most rows any call of this launch (graph node) has
cudaError_t la_launch_gemm_tc(const LaDev& d, cudaStream_t st, const TcGemm& g, const TcWork& w, int sel,
                              int rows_cap);
// bytes of g's packed weights, and the packing of w1..w3 (the maps' matrices) into dst
size_t la_tc_packed_bytes(const TcGemm& g);
cudaError_t la_tc_pack(const TcGemm& g, const void* w1, const void* w2, const void* w3, void* dst, cudaStream_t st);
int la_tc_ctas();
// (tile, K) units per tile of a K-deep weight: 128-column units (64 for the gate/up pair)
int la_tc_k_units(int mode, int K, int pair = 0);
int la_tc_pick_ctas(int n_tiles, int k_tiles, int mode);
int la_tc_max_segments(int n_tiles, int k_tiles, int n_cta);
cudaError_t la_tc_prepare_device();
int la_tc_defer_default();
LaSplit la_tc_split(const TcGemm& g, const TcWork& w);
void la_tc_scratch_need(int mode, int n_out, int K, int rows, int n_cta, size_t* ws_floats, size_t* n_counters);

// exact sampling verifier (one CTA): reads the needed rows' fp32 logits and
// writes the verdict (a, winner, E, emitted) into the header; prefill=1 draws
// the first token of a request from row 0 (Philox step 0xFFFFFFFF)
cudaError_t la_launch_sample_verify(const LaDev& d, cudaStream_t st, const float* logits, int V, int prefill);
cudaError_t la_launch_sample_trials(cudaStream_t st, const float* logits, int V, const int32_t* cand, int Ct, int S,
                                    float T, float top_p, uint64_t seed, int n_trials, int32_t* out);

// bf16 attention: committed 128-position blocks on tensor cores + combine/tail
int la_attn_tail_blocks(int pmax);
// RoPE folded into the attention of a decode call: the QKV GEMM's output
// (and its split tiles) and the rotation tables; qkv == nullptr: the queries
// and temporary K/V come from the RoPE kernel
struct LaRope {
    const __nv_bfloat16* qkv;
    LaSplit sp;
    const float* rcos;
    const float* rsin;
};
size_t la_attn_smem_bytes(int TB, int tail_rows, int pmax, int qrows);
// the most temporary rows the paths of one attention tile (16 consecutive
// packed rows) can reach: base stripe and level 0 (<= W+N-3 cells), each
// row's own trajectory cells (<= N-2), the verification cells of the
// candidates the tile touches (<= 16 + N-1), bounded by the call's rows
inline int la_attn_tail_rows(int max_W, int max_N, int Qmax) {
    const int u = max_W + 20 * (max_N - 1);
    return u < Qmax ? u : Qmax;
}
cudaError_t la_launch_attention_bf16(const LaDev& d, cudaStream_t st, const void* qbuf, const void* kc, const void* vc,
                                     const void* kt, const void* vt, void* out, int H, int sel, int Qcap,
                                     int max_ctx, int Qmax, int rows_cap, int TB, int pmax, const CUtensorMap& cmap,
                                     int krow0, int vrow0, const LaHdr* const* req_hdr = nullptr, int qstride = 0,
                                     long long req_cache_elems = 0, int req_cache_rows = 0, int temp_stride = 0,
                                     int tail_rows = 0, const LaRope* rope = nullptr);

// ---------------------------------------------------------------------------
// Layer-chain kernel (la_mega.cu): one launch runs a chain of GEMM and row
// phases of a decode call on one CTA per SM (see la_mega.cu).
// ---------------------------------------------------------------------------
#define MG_MAX_PHASES 8
#define MG_MAX_GEMMS 4
#define MG_MAX_ROWS 4
#define MG_MAX_ROWS_PER_CALL 256      // packed rows a chain supports (one 256-row chunk)
enum { MG_PH_GEMM = 0, MG_PH_ROWS = 1 };
enum { MG_RMS = 0, MG_RMS_GATHER = 1, MG_SWIGLU = 2 };

struct MgGemm {
    const uint8_t* wpack;                 // unit-contiguous weight images (la_tc_pack)
    const __nv_bfloat16* act;             // activation rows [rows][K] (row stride K)
    int mode, K, n_tiles, k_tiles, ua, k_atoms, nA, max_seg, sel, defer, n_cta;
    float* ws;                            // split-tile partial records (LaSplit layout)
    unsigned long long* ctr;              // split-tile arrival counters (non-deferred GEMMs)
    void* out; int ldo;
    float* logits; int ld_logits;         // GEMM_LOGITS: optional fp32 logits
    float* part_v; int* part_i; int part_stride;   // GEMM_LOGITS: argmax partials per tile
};
struct MgRows {
    int kind, sel, dm;
    float eps;
    float* x;                             // RMS: the fp32 residual rows (updated in place)
    const __nv_bfloat16* g;               // RMS: gains
    __nv_bfloat16* y;                     // RMS: normalised rows; SWIGLU: the activation rows
    int ldo;                              // SWIGLU: row stride of y
    LaSplit split;                        // partials of the GEMM that wrote x (RMS) or gate/up (SWIGLU)
};
struct MgParams {
    LaHdr* hdr;
    LaTlRec* tl;                          // kernel timeline table, or nullptr
    const int32_t* need;                  // needed rows (MG_RMS_GATHER)
    unsigned long long* bar;              // this launch's phase counters [MG_MAX_PHASES] (zero at launch)
    int n_ph;
    int ph_kind[MG_MAX_PHASES], ph_idx[MG_MAX_PHASES];
    MgGemm g[MG_MAX_GEMMS];
    MgRows r[MG_MAX_ROWS];
    int rows_cap;                         // the most rows any call of this launch has
    int ns_pre;                           // ring stages whose weights are issued before the header is read
};
cudaError_t la_launch_mega(const MgParams& p, cudaStream_t st);
int la_mega_ring_stages(int rows);        // ring stages at `rows` packed rows
int la_tc_unit_atoms(int mode, int pair = 0);

