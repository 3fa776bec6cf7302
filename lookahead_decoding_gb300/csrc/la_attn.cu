// Masked attention of the packed call for bf16 models: one kernel, one CTA
// per (head, tile of 16 packed rows), 16 warps (8 for the committed blocks,
// all 16 for the tail).
//
// Every row attends to one key per logical position 0..pos (M7.3 §0x04A:
// the committed prefix, then the row's own branch path).  The positions are
// split at t0(pos) = max(0, (floor(pos/32) - TB) * 32), a function of the
// row's position alone (TB is fixed per context so that pos - t0 covers
// every in-call offset):
//   * committed keys [0, t0) — 128-position blocks of the cache stream
//     through a double-buffered shared-memory ring (TMA from one tensor map
//     over the whole cache: four 64-dimension boxes of 128-byte rows per
//     block, 128-byte swizzle, an mbarrier per buffer).  For each block the
//     8 block warps split the keys for S = Q K^T
//     (mma.sync m16n8k16 bf16 -> fp32), form the per-row block maximum m,
//     P = exp(S - m) rounded to fp16 and its row sum l, then split the
//     dimensions for O = P V (fp16 mma; V fragments by ldmatrix.trans,
//     converted exactly from bf16).  (m, l, O) of the block merges into the
//     row's running state in block order.
//   * positions [t0, pos] — at most 128 keys per row, from the cache
//     (committed) or the call's temporary rows on the row's path (in-call),
//     staged in shared memory once per tile.  S on tensor cores for every
//     (row, staged key) pair of the tile (an element of the mma depends only
//     on its query and its key); then one softmax block per row on CUDA
//     cores in fp32 over the row's own keys in position order (four
//     dimensions per lane for P V); merged after the blocks, then normalised.
// A row's arithmetic therefore depends only on its query, its position and
// the keys it sees — the same whether it is decoded alone or packed.
#include "la_common.cuh"
#include "la_kernels.h"

#include <cuda_fp16.h>
#include <math.h>

// la_split_sum4 with the first eight segments' loads issued together (same
// additions, K order), for callers with the registers for them
__device__ __forceinline__ float4 la_split_sum4_w8(const LaSplit& s, int t, int y, size_t off, int nseg) {
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
    for (int s0 = 8; s0 < nseg; ++s0) {
        const float4 q = __ldcg(reinterpret_cast<const float4*>(la_split_rec(s, t, y, s0, 0) + off));
        r.x = __fadd_rn(r.x, q.x);
        r.y = __fadd_rn(r.y, q.y);
        r.z = __fadd_rn(r.z, q.z);
        r.w = __fadd_rn(r.w, q.w);
    }
    return r;
}

// la_qkv_at4 with the wide segment loads
__device__ __forceinline__ float4 la_qkv_at4_w8(const __nv_bfloat16* row, int q, int n, const LaSplit& sp, int nseg) {
    if (nseg <= 1) {
        const uint2 u = *reinterpret_cast<const uint2*>(row + n);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
    const float4 s = la_split_sum4_w8(sp, n >> 7, q >> 8, (size_t)(q & 255) * 128 + (n & 127), nseg);
    return make_float4(la_bf16_round(s.x), la_bf16_round(s.y), la_bf16_round(s.z), la_bf16_round(s.w));
}

namespace {

constexpr int DH = 128;
constexpr int BLK = 128;          // positions per committed block
constexpr int FR = 16;            // packed rows per CTA (one m16 tile)
constexpr int FW = 8;             // warps of the committed blocks (S, P V on tensor cores)
constexpr int FT = 16;            // warps per CTA: the tail takes a row per warp
constexpr int KPW = BLK / FW;     // keys of a block per warp (S = Q K^T)
constexpr int DPW = DH / FW;      // dimensions per warp (O = P V)
constexpr int NTW = KPW / 8;      // n-tiles of 8 per warp (KPW == DPW)
constexpr int PAD = 8;            // bf16 padding per smem row (16 B): conflict-free fragment loads
constexpr int LDK = DH + PAD;     // K, V, Q and P rows in shared memory
constexpr int MAX_TAIL = 128;     // tail keys per row (TB <= 3)

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
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// bounded wait for phase `parity` of an mbarrier; false once the limit is spent
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < LA_SPIN_LIMIT; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
                 "l"(m), "r"(bar), "r"(x), "r"(y)
                 : "memory");
}
// byte offset of (key, dimension pair start) in a TMA-staged block: two
// 64-dimension boxes of BLK rows x 128 B, 16-byte chunks swizzled by key mod 8
__device__ __forceinline__ uint32_t blk_off(int key, int dim) {
    return (uint32_t)((dim >> 6) * (BLK * 128) + key * 128 + ((((dim & 63) >> 3) ^ (key & 7)) << 4) + ((dim & 7) << 1));
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

// barrier among the FW block warps (the helper warps are not in the block loop)
__device__ __forceinline__ void bar_blocks() { asm volatile("bar.sync 1, %0;" ::"n"(FW * 32) : "memory"); }

__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// shared memory (bytes): the K/V ring (reused for the tail keys), then fixed areas
// (offsets from the first 1024-byte boundary of the dynamic shared memory;
// the launch adds 1024 bytes of slack).  The ring holds two committed blocks
// as TMA leaves them (K then V, each two 64-dimension boxes of 128-byte rows,
// 64 KB per block) or, after the blocks, the tail keys in padded rows.
struct FusedLayout {
    uint32_t ring, ring_bytes, q, p, o, wmax, wl, rpos, rt0, pw, sw, bar, ssc, ssp, path, uslot, urow, misc, total;
    uint32_t tk, tv, ik, iv, ring_used;   // tail keys: committed (tk, tv) and, apart, in-call (ik, iv)
};
// ck: the committed tail keys a tile can stage (32 (TB + 1)).  sep: the
// in-call keys get a region of their own beside the block ring, so the warps
// that wait out the committed blocks can stage them meanwhile; the committed
// tail keys, the per-warp softmax rows and the tail scores then move into
// the ring, free once the blocks are done.
__host__ __device__ inline FusedLayout fused_layout(int ring_keys, int pmax, int qrows, int sep = 0, int ck = 0) {
    FusedLayout L;
    L.ring = 0;
    L.ssp = (uint32_t)ring_keys + 4;                                // tail scores: [FR][ssp] fp32
    if (!sep) {
        L.ring_bytes = (uint32_t)ring_keys * 2u * LDK * 2u;       // K and V rows, bf16
        if (L.ring_bytes < 2u * 4u * BLK * 128u) L.ring_bytes = 2u * 4u * BLK * 128u;
        L.tk = L.ring;
        L.tv = L.tk + (uint32_t)ring_keys * LDK * 2u;
        L.ik = L.tk;                                                // in-call keys follow the committed ones
        L.iv = L.tv;
        L.q = L.ring + L.ring_bytes;
    } else {
        L.ring_bytes = 2u * 4u * BLK * 128u;
        L.tk = L.ring;                                              // [ck][LDK] bf16, after the blocks
        L.tv = L.tk + (uint32_t)ck * LDK * 2u;
        L.pw = L.tv + (uint32_t)ck * LDK * 2u;                      // [FT][MAX_TAIL] fp32
        L.sw = L.pw + FT * MAX_TAIL * 4;                            // [FT][MAX_TAIL] int
        L.ssc = L.sw + FT * MAX_TAIL * 4;
        L.ring_used = L.ssc + FR * L.ssp * 4;                       // <= ring_bytes (checked by the launch)
        L.ik = L.ring + L.ring_bytes;                               // [ring_keys - ck][LDK] bf16
        L.iv = L.ik + (uint32_t)(ring_keys - ck) * LDK * 2u;
        L.q = L.iv + (uint32_t)(ring_keys - ck) * LDK * 2u;
    }
    L.p = L.q + FR * LDK * 2;                                       // [FR][LDK] fp16
    L.o = L.p + FR * LDK * 2;                                       // [FR][DH] fp32
    L.wmax = L.o + FR * DH * 4;                                     // [FW][FR] fp32
    L.wl = L.wmax + FW * FR * 4;                                    // [FW][FR] fp32
    L.rpos = L.wl + FW * FR * 4;                                    // [FR] int
    L.rt0 = L.rpos + FR * 4;                                        // [FR] int
    if (!sep) {
        L.pw = L.rt0 + FR * 4;                                      // [FT][MAX_TAIL] fp32
        L.sw = L.pw + FT * MAX_TAIL * 4;                            // [FT][MAX_TAIL] int
        L.bar = L.sw + FT * MAX_TAIL * 4;                           // 2 mbarriers
        L.ssc = L.bar + 16;
        L.path = L.ssc + FR * L.ssp * 4;                            // [FR][pmax] int
        L.ring_used = L.ring_bytes;
    } else {
        L.bar = L.rt0 + FR * 4;
        L.path = L.bar + 16;
    }
    L.uslot = L.path + (uint32_t)FR * pmax * 4;                     // [qrows] int: ring slot of a temporary row
    L.urow = L.uslot + (uint32_t)qrows * 4;                         // [qrows] int: temporary row of a slot
    L.misc = L.urow + (uint32_t)qrows * 4;                          // [4] int: the count of staged rows
    L.total = L.misc + 16;
    return L;
}

__global__ void __launch_bounds__(FT * 32) k_attn_fused(LaDev d, const __nv_bfloat16* qbuf, const __nv_bfloat16* kc,
                                                      const __nv_bfloat16* vc, const __nv_bfloat16* kt,
                                                      const __nv_bfloat16* vt, __nv_bfloat16* out, int sel, int Qcap,
                                                      int max_ctx, int temp_stride, int TB, int H, int ring_keys,
                                                      const __grid_constant__ CUtensorMap cmap, int krow0, int vrow0,
                                                      const LaHdr* const* req_hdr, int qstride,
                                                      long long req_cache_elems, int req_cache_rows, int qrows,
                                                      LaRope rope, int sep, int ck) {
    LaTl la_tl_(LA_TL_ATTN_FUSED, d.tl);
    const LaHdr* h = d.hdr;
    const int hh = blockIdx.x, r0 = blockIdx.y * FR;
    // A batched call stacks its requests' rows in slices of qstride rows (a
    // multiple of the tile): the tile's request has its own header
    // (committed length, row count), cache and temporary rows.
    const int req = qstride ? r0 / qstride : 0;
    const LaHdr* hr = qstride ? req_hdr[req] : h;
    krow0 += req * req_cache_rows;
    vrow0 += req * req_cache_rows;
    kc += (size_t)req * req_cache_elems;
    vc += (size_t)req * req_cache_elems;
    kt += (size_t)req * qstride * DH;
    vt += (size_t)req * qstride * DH;
    const int prefill = (sel == SEL_PREFILL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int PM = d.PMAX;

    extern __shared__ __align__(16) uint8_t smem_raw[];
    const FusedLayout LY = fused_layout(ring_keys, PM, qrows, sep, ck);
    const uint32_t sraw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - sraw);
    __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem + LY.q);
    __half* ps = reinterpret_cast<__half*>(smem + LY.p);
    float* os = reinterpret_cast<float*>(smem + LY.o);
    float* wmax = reinterpret_cast<float*>(smem + LY.wmax);
    float* wl = reinterpret_cast<float*>(smem + LY.wl);
    int* rpos = reinterpret_cast<int*>(smem + LY.rpos);
    int* rt0 = reinterpret_cast<int*>(smem + LY.rt0);
    float* pw = reinterpret_cast<float*>(smem + LY.pw);
    int* sw = reinterpret_cast<int*>(smem + LY.sw);
    int* spath = reinterpret_cast<int*>(smem + LY.path);
    const __nv_bfloat16* kh = kc + (size_t)hh * max_ctx * DH;
    const __nv_bfloat16* vh = vc + (size_t)hh * max_ctx * DH;

    // Committed block b (positions b*BLK ..) into ring buffer buf by TMA,
    // issued by thread 0, completing on barrier buf: rows krow0 + hh*max_ctx +
    // position of the cache (rows past this head's range read masked keys or
    // the zero fill past the end of the cache).
    const uint32_t bar0 = sbase + LY.bar;
    auto stage_block = [&](int b, int buf) {
        if (tid != 0) return;
        const uint32_t kb = sbase + LY.ring + (uint32_t)buf * (4u * BLK * 128u);
        const uint32_t vb = kb + 2u * BLK * 128u, bar = bar0 + 8u * buf;
        const int y = b * BLK + hh * max_ctx;
        mbar_arrive_tx(bar, 4u * BLK * 128u);
        tma_2d(kb, &cmap, bar, 0, krow0 + y);
        tma_2d(kb + BLK * 128u, &cmap, bar, 64, krow0 + y);
        tma_2d(vb, &cmap, bar, 0, vrow0 + y);
        tma_2d(vb + BLK * 128u, &cmap, bar, 64, vrow0 + y);
    };
    if (tid == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar0 + 8, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }

    // Before the wait (la_common.cuh): the header, and in a decode call the
    // tile's row positions and paths (written by the pack kernel) and, for
    // the first tile, which every call fills, committed block 0 of the cache
    // (written by earlier calls; cp.async group 1).  After the wait: the
    // queries, which the kernel before this one writes (group 2).  Every grid
    // row is below Qcap and block 0 lies in the cache, so all of it is in
    // bounds whatever the call's row count.
    const int h_err = h->err, h_done = h->done, rows = rows_sel(h, sel);
    if (h_err != 0 || (sel != SEL_PREFILL && (h_done != 0 || hr->done != 0)) || r0 >= rows) return;
    const bool spec0 = (blockIdx.y == 0) && !prefill;
    int pos_raw = 0;
    if (!prefill) {
        if (tid < FR) pos_raw = d.row_pos[r0 + tid];
        for (int i = tid; i < FR * PM; i += blockDim.x) spath[i] = d.row_path[(size_t)(r0 + i / PM) * PM + i % PM];
        if (spec0) stage_block(0, 0);
    }
    la_pdl_wait();
    la_pdl_trigger();
    if (prefill && tid < FR) pos_raw = d.row_pos[r0 + tid];
    const int nr = min(FR, rows - r0);
    // decode with RoPE folded in: the queries are computed below from the QKV output
    const bool fuse = rope.qkv != nullptr && !prefill;
    if (!fuse) {
        const __nv_bfloat16* qh = qbuf + (size_t)hh * Qcap * DH;
        for (int i = tid; i < FR * (DH / 8); i += blockDim.x) {
            const int r = i >> 4, c8 = (i & 15) * 8;
            cp_async16(sbase + LY.q + (uint32_t)(r * LDK + c8) * 2u, qh + (size_t)(r0 + r) * DH + c8, 16);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    const int K = prefill ? 0 : hr->K;
    const int Q = prefill ? 0 : hr->Q;                // the request's temporary K/V rows
    if (tid < FR) {
        const int pos = tid < nr ? pos_raw : -1;
        rpos[tid] = pos;
        rt0[tid] = pos >= 0 ? t0_of(pos, TB) : 0;
    }
    __syncthreads();
    // RoPE folded in: the tile's queries of head hh into shared memory and,
    // for the K/V commit, its rows' rotated K and V into the temporary rows
    // (each (row, head) is written by exactly one CTA; no CTA of this kernel
    // reads them).  Rows past the call's rows get zero queries.
    const int HD = H * DH, half = DH / 2;
    const int seg_q = (fuse && rope.sp.ws) ? la_split_nseg(rope.sp, hh) : 1;
    const int seg_k = (fuse && rope.sp.ws) ? la_split_nseg(rope.sp, H + hh) : 1;
    const int seg_v = (fuse && rope.sp.ws) ? la_split_nseg(rope.sp, 2 * H + hh) : 1;
    // item j of part 0 (the query: rotated into shared memory), 1 (the key:
    // rotated) or 2 (the value) of the tile's rows; keys and values go to the
    // temporary rows for the commit (no CTA of this kernel reads them)
    __nv_bfloat16* qs_w = reinterpret_cast<__nv_bfloat16*>(smem + LY.q);
    __nv_bfloat16* kt_w = const_cast<__nv_bfloat16*>(kt) + (size_t)hh * temp_stride * DH;
    __nv_bfloat16* vt_w = const_cast<__nv_bfloat16*>(vt) + (size_t)hh * temp_stride * DH;
    constexpr int RI = FR * (DH / 2 / 4);              // items of one part
    auto rope_item = [&](int part, int j) {
        const int r = j / (half / 4), c4 = (j % (half / 4)) * 4;
        if (r >= nr) {
            if (part == 0) {
                __nv_bfloat16* qd = qs_w + r * LDK + c4;
                *reinterpret_cast<uint2*>(qd) = make_uint2(0u, 0u);
                *reinterpret_cast<uint2*>(qd + half) = make_uint2(0u, 0u);
            }
            return;
        }
        const int row = r0 + r, pos = rpos[r], lrow = row - req * qstride;
        const __nv_bfloat16* x = rope.qkv + (size_t)row * 3 * HD;
        const int seg = part == 0 ? seg_q : (part == 1 ? seg_k : seg_v);
        const int n0 = part * HD + hh * DH + c4;
        const float4 a = la_qkv_at4(x, row, n0, rope.sp, seg);
        const float4 b = la_qkv_at4(x, row, n0 + half, rope.sp, seg);
        if (part == 2) {
            __nv_bfloat16* vo = vt_w + (size_t)lrow * DH + c4;
            *reinterpret_cast<uint2*>(vo) = la_pack_bf16x4(a.x, a.y, a.z, a.w);
            *reinterpret_cast<uint2*>(vo + half) = la_pack_bf16x4(b.x, b.y, b.z, b.w);
            return;
        }
        const float4 c = *reinterpret_cast<const float4*>(rope.rcos + (size_t)pos * half + c4);
        const float4 s = *reinterpret_cast<const float4*>(rope.rsin + (size_t)pos * half + c4);
        __nv_bfloat16* dst = part == 0 ? qs_w + r * LDK + c4 : kt_w + (size_t)lrow * DH + c4;
        la_rope4_store(dst, dst + half, a, b, c, s);
    };
    // the queries now; the keys and values for the commit by the warps that
    // wait out the committed blocks
    if (fuse) {
        // the queries: two lanes an item, one rotation partner each (its
        // segments' loads in one round), the pair exchanged by a shuffle
        for (int j = tid; j < 2 * RI; j += blockDim.x) {
            const int item = j >> 1, hf = j & 1;
            const int r = item / (half / 4), c4 = (item % (half / 4)) * 4;
            const bool live = r < nr;
            float4 own = make_float4(0.f, 0.f, 0.f, 0.f), c = own, sn = own;
            if (live) {
                const int row = r0 + r, pos = rpos[r];
                const __nv_bfloat16* x = rope.qkv + (size_t)row * 3 * HD;
                own = la_qkv_at4_w8(x, row, hh * DH + c4 + hf * half, rope.sp, seg_q);
                c = *reinterpret_cast<const float4*>(rope.rcos + (size_t)pos * half + c4);
                sn = *reinterpret_cast<const float4*>(rope.rsin + (size_t)pos * half + c4);
            }
            float4 oth;
            oth.x = __shfl_xor_sync(0xffffffffu, own.x, 1);
            oth.y = __shfl_xor_sync(0xffffffffu, own.y, 1);
            oth.z = __shfl_xor_sync(0xffffffffu, own.z, 1);
            oth.w = __shfl_xor_sync(0xffffffffu, own.w, 1);
            const float4 a = hf ? oth : own, b = hf ? own : oth;
            __nv_bfloat16* qd = qs_w + r * LDK + c4 + hf * half;
            if (!live) {
                *reinterpret_cast<uint2*>(qd) = make_uint2(0u, 0u);
            } else if (hf == 0) {
                *reinterpret_cast<uint2*>(qd) = la_pack_bf16x4(la_rope_lo(a.x, b.x, c.x, sn.x), la_rope_lo(a.y, b.y, c.y, sn.y),
                                                               la_rope_lo(a.z, b.z, c.z, sn.z), la_rope_lo(a.w, b.w, c.w, sn.w));
            } else {
                *reinterpret_cast<uint2*>(qd) = la_pack_bf16x4(la_rope_hi(a.x, b.x, c.x, sn.x), la_rope_hi(a.y, b.y, c.y, sn.y),
                                                               la_rope_hi(a.z, b.z, c.z, sn.z), la_rope_hi(a.w, b.w, c.w, sn.w));
            }
        }
    }
    int t0max = 0, t0min = 0x7fffffff, posmax = 0;
    for (int r = 0; r < nr; ++r) {
        t0max = max(t0max, rt0[r]);
        t0min = min(t0min, rt0[r]);
        posmax = max(posmax, rpos[r]);
    }
    const int nb = (t0max + BLK - 1) / BLK;
    if (!spec0 && nb > 0) stage_block(0, 0);
    const int ta = rt0[g], tb = rt0[g + 8];             // split points of this thread's two rows

    const bool sepm = sep && fuse;
    const int Kc = prefill ? posmax + 1 : K;
    const int nc = (nr > 0 && Kc > t0min) ? Kc - t0min : 0;
    int* uslot = reinterpret_cast<int*>(smem + LY.uslot);
    int* urow = reinterpret_cast<int*>(smem + LY.urow);
    int& s_nu = *reinterpret_cast<int*>(smem + LY.misc);
    const uint32_t tk_a = sbase + LY.tk, tv_a = sbase + LY.tv;
    // the temporary rows on the tile's rows' paths, each once, in row order
    // (uslot: a temporary row's slot among them; urow: the inverse; s_nu:
    // their count).  Called by every thread of the CTA (group 0) or by the
    // warps FW .. FT-1 alone (group 1, while the blocks run).
    auto mark_paths = [&](int group) {
        const int t = group ? tid - FW * 32 : tid, nthr = group ? (FT - FW) * 32 : (int)blockDim.x;
        auto sync = [&]() {
            if (group) asm volatile("bar.sync 2, %0;" ::"n"((FT - FW) * 32) : "memory");
            else __syncthreads();
        };
        if (t == 0) s_nu = 0;
        if (Q > 0) {
            for (int q = t; q < Q; q += nthr) uslot[q] = 0;
            sync();
            for (int i = t; i < nr * PM; i += nthr) {
                const int r = i / PM, e = i % PM, pos = rpos[r];
                if (pos >= K && e <= pos - K) {
                    const int pr = spath[i];
                    if (pr >= 0 && pr < Q) uslot[pr] = 1;
                }
            }
            sync();
            if (t < 32) {        // slots in row order: a ballot scan over the marks
                int run = 0;
                for (int base = 0; base < Q; base += 32) {
                    const int q = base + lane;
                    const bool m = q < Q && uslot[q] != 0;
                    const unsigned bal = __ballot_sync(0xffffffffu, m);
                    const int sl = run + __popc(bal & ((1u << lane) - 1u));
                    if (m) { uslot[q] = sl; urow[sl] = q; }
                    run += __popc(bal);
                }
                if (lane == 0) s_nu = run;
            }
        }
        sync();
    };
    if (sepm) mark_paths(0);
    // the in-call keys: rotated K and V of the request's row urow[s] at its
    // position, head hh, into in-call slot s (row nc + s of the tail keys, or
    // row s of the separate region), items from i0 in steps of di; one item
    // per (part, slot, four dimensions): part 0 the key, 1 the value
    auto stage_incall = [&](int i0, int di) {
        __nv_bfloat16* ik_w = reinterpret_cast<__nv_bfloat16*>(smem + LY.ik) + (sepm ? 0 : (size_t)nc * LDK);
        __nv_bfloat16* iv_w = reinterpret_cast<__nv_bfloat16*>(smem + LY.iv) + (sepm ? 0 : (size_t)nc * LDK);
        const int nk = s_nu * (half / 4);
        for (int i = i0; i < 2 * nk; i += di) {
            const int part = i / nk, j = i % nk;
            const int sl = j / (half / 4), c4 = (j % (half / 4)) * 4;
            const int row = req * qstride + urow[sl];
            const __nv_bfloat16* x = rope.qkv + (size_t)row * 3 * HD;
            const int n0 = (part + 1) * HD + hh * DH + c4;
            const float4 a = la_qkv_at4(x, row, n0, rope.sp, part == 0 ? seg_k : seg_v);
            const float4 b = la_qkv_at4(x, row, n0 + half, rope.sp, part == 0 ? seg_k : seg_v);
            if (part == 1) {
                __nv_bfloat16* vd = iv_w + (size_t)sl * LDK + c4;
                *reinterpret_cast<uint2*>(vd) = la_pack_bf16x4(a.x, a.y, a.z, a.w);
                *reinterpret_cast<uint2*>(vd + half) = la_pack_bf16x4(b.x, b.y, b.z, b.w);
                continue;
            }
            const int pos = d.row_pos[row];
            const float4 c = *reinterpret_cast<const float4*>(rope.rcos + (size_t)pos * half + c4);
            const float4 sn = *reinterpret_cast<const float4*>(rope.rsin + (size_t)pos * half + c4);
            __nv_bfloat16* kd = ik_w + (size_t)sl * LDK + c4;
            la_rope4_store(kd, kd + half, a, b, c, sn);
        }
    };

    // running state of rows g and g+8; O columns of this warp's dims
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    float o[NTW][4];
#pragma unroll
    for (int n = 0; n < NTW; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    // Q fragments (A operand of S = Q K^T) for the 8 k-steps, from shared memory
    asm volatile("cp.async.wait_group 0;" ::: "memory");     // the queries
    __syncthreads();
    uint32_t qa[8][4];
#pragma unroll
    for (int ks8 = 0; ks8 < 8; ++ks8)
        ldsm_x4(sbase + LY.q + (uint32_t)((lane & 15) * LDK + ks8 * 16 + (lane >> 4) * 8) * 2u, qa[ks8]);

    const float scale = 0.08838834764831845f;   // 1/sqrt(128)
    // (the paths are marked by the whole CTA first: the warps below would
    // otherwise outlast the blocks)
    if (fuse && warp >= FW) {
        for (int i = tid - FW * 32; i < 2 * RI; i += (FT - FW) * 32) rope_item(1 + i / RI, i % RI);
        if (sepm && s_nu <= ring_keys - ck) stage_incall(tid - FW * 32, (FT - FW) * 32);
    }
    // warps FW .. FT-1 wait for the blocks at the barrier before the tail
    for (int b = 0; b < (warp < FW ? nb : 0); ++b) {
        const int buf = b & 1;
        // buffer buf ^ 1 held block b - 1, which every block warp has finished
        if (b + 1 < nb) stage_block(b + 1, buf ^ 1);
        if (!mbar_wait(bar0 + 8u * buf, (uint32_t)((b >> 1) & 1)) && lane == 0) la_set_err(d.hdr, LA_ETIMEOUT);
        const uint8_t* kbb = smem + LY.ring + (size_t)buf * (4 * BLK * 128);
        const uint32_t vs_a = sbase + LY.ring + (uint32_t)buf * (4u * BLK * 128u) + 2u * BLK * 128u;
        const int key0 = b * BLK;
        // S for this warp's KPW keys (NTW n-tiles of 8)
        float s[NTW][4];
#pragma unroll
        for (int n = 0; n < NTW; ++n) {
            s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
            const int key = warp * KPW + n * 8 + g;
#pragma unroll
            for (int ks8 = 0; ks8 < 8; ++ks8) {
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kbb + blk_off(key, ks8 * 16 + 2 * t));
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kbb + blk_off(key, ks8 * 16 + 8 + 2 * t));
                mma16816(s[n], qa[ks8], b0, b1);
            }
        }
        float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
        for (int n = 0; n < NTW; ++n) {
            const int kp = key0 + warp * KPW + n * 8 + 2 * t;
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
        if (t == 0) { wmax[warp * FR + g] = ma; wmax[warp * FR + g + 8] = mb; }
        bar_blocks();
        // block maximum per row over the warps
        ma = wmax[g];
        mb = wmax[g + 8];
#pragma unroll
        for (int w = 1; w < FW; ++w) {
            ma = fmaxf(ma, wmax[w * FR + g]);
            mb = fmaxf(mb, wmax[w * FR + g + 8]);
        }
        // P = exp(S - m) rounded to fp16 into shared memory; l sums the rounded values
        float la = 0.f, lb = 0.f;
#pragma unroll
        for (int n = 0; n < NTW; ++n) {
            const float p0 = (s[n][0] == -INFINITY) ? 0.f : expf(__fsub_rn(s[n][0], ma));
            const float p1 = (s[n][1] == -INFINITY) ? 0.f : expf(__fsub_rn(s[n][1], ma));
            const float p2 = (s[n][2] == -INFINITY) ? 0.f : expf(__fsub_rn(s[n][2], mb));
            const float p3 = (s[n][3] == -INFINITY) ? 0.f : expf(__fsub_rn(s[n][3], mb));
            const uint32_t ua = pack_f16(p0, p1), ub = pack_f16(p2, p3);
            const int col = warp * KPW + n * 8 + 2 * t;
            *reinterpret_cast<uint32_t*>(ps + g * LDK + col) = ua;
            *reinterpret_cast<uint32_t*>(ps + (g + 8) * LDK + col) = ub;
            const __half2 q0 = *reinterpret_cast<const __half2*>(&ua);
            const __half2 q1 = *reinterpret_cast<const __half2*>(&ub);
            la = __fadd_rn(la, __fadd_rn(__low2float(q0), __high2float(q0)));
            lb = __fadd_rn(lb, __fadd_rn(__low2float(q1), __high2float(q1)));
        }
        la = __fadd_rn(la, __shfl_xor_sync(0xffffffffu, la, 1));
        la = __fadd_rn(la, __shfl_xor_sync(0xffffffffu, la, 2));
        lb = __fadd_rn(lb, __shfl_xor_sync(0xffffffffu, lb, 1));
        lb = __fadd_rn(lb, __shfl_xor_sync(0xffffffffu, lb, 2));
        if (t == 0) { wl[warp * FR + g] = la; wl[warp * FR + g + 8] = lb; }
        bar_blocks();
        la = wl[g];
        lb = wl[g + 8];
#pragma unroll
        for (int w = 1; w < FW; ++w) {
            la = __fadd_rn(la, wl[w * FR + g]);
            lb = __fadd_rn(lb, wl[w * FR + g + 8]);
        }
        // O of the block for this warp's DPW dims: 8 k-steps of 16 keys x NTW n-tiles
        float ob[NTW][4];
#pragma unroll
        for (int n = 0; n < NTW; ++n) ob[n][0] = ob[n][1] = ob[n][2] = ob[n][3] = 0.f;
        const int mtx = lane >> 3, mrow = lane & 7;
        const int key_off = (mtx & 1) * 8 + mrow, dim_off = (mtx >> 1) * 8;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t a[4];
            ldsm_x4(sbase + LY.p + (uint32_t)((lane & 15) * LDK + kk * 16 + (lane >> 4) * 8) * 2u, a);
#pragma unroll
            for (int n = 0; n < NTW; n += 2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(vs_a + blk_off(kk * 16 + key_off, warp * DPW + n * 8 + dim_off), b0, b1, b2, b3);
                mma16816_f16(ob[n], a, bf2_to_h2(b0), bf2_to_h2(b1));
                mma16816_f16(ob[n + 1], a, bf2_to_h2(b2), bf2_to_h2(b3));
            }
        }
        // merge the block into the running state (rows without committed keys here skip it)
        if (ma != -INFINITY) {
            const float mn = fmaxf(m_a, ma);
            const float ca = (m_a == -INFINITY) ? 0.f : expf(__fsub_rn(m_a, mn));
            const float cb = expf(__fsub_rn(ma, mn));
            l_a = fmaf(l_a, ca, __fmul_rn(la, cb));
#pragma unroll
            for (int n = 0; n < NTW; ++n) {
                o[n][0] = fmaf(o[n][0], ca, __fmul_rn(ob[n][0], cb));
                o[n][1] = fmaf(o[n][1], ca, __fmul_rn(ob[n][1], cb));
            }
            m_a = mn;
        }
        if (mb != -INFINITY) {
            const float mn = fmaxf(m_b, mb);
            const float ca = (m_b == -INFINITY) ? 0.f : expf(__fsub_rn(m_b, mn));
            const float cb = expf(__fsub_rn(mb, mn));
            l_b = fmaf(l_b, ca, __fmul_rn(lb, cb));
#pragma unroll
            for (int n = 0; n < NTW; ++n) {
                o[n][2] = fmaf(o[n][2], ca, __fmul_rn(ob[n][2], cb));
                o[n][3] = fmaf(o[n][3], ca, __fmul_rn(ob[n][3], cb));
            }
            m_b = mn;
        }
        bar_blocks();      // P, the warp maxima/sums and this buffer are reused
    }
    // the committed state to shared memory: O by (row, dim), m and l per row
    if (warp < FW) {
#pragma unroll
    for (int n = 0; n < NTW; ++n) {
        const int col = warp * DPW + n * 8 + 2 * t;
        *reinterpret_cast<float2*>(os + g * DH + col) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2*>(os + (g + 8) * DH + col) = make_float2(o[n][2], o[n][3]);
    }
    if (warp == 0 && t == 0) {
        wmax[g] = m_a; wmax[g + 8] = m_b;
        wl[g] = l_a; wl[g + 8] = l_b;
    }
    }
    // a first tile without committed blocks still had block 0 staged
    if (tid == 0 && spec0 && nb == 0 && !mbar_wait(bar0, 0)) la_set_err(d.hdr, LA_ETIMEOUT);
    __syncthreads();      // the ring is free for the tail keys

    // tail keys: committed positions [t0min, Kc), then (in a call) the
    // temporary rows on the tile's rows' paths, each once, in row order.
    // Which slot a key takes changes no arithmetic: every score depends only
    // on its query and key, and each row reads its own keys in position
    // order.  Separate layout: the in-call keys were marked and staged while
    // the blocks ran.
    if (!sepm) mark_paths(0);
    const int nt = nc + s_nu;
    if (nt > ring_keys || (sepm && (nc > ck || s_nu > ring_keys - ck))) {
        // beyond the ring the launch sized (bounded by construction)
        if (tid == 0) la_set_err(d.hdr, LA_ECAPACITY);
        return;
    }
    {
        const __nv_bfloat16* kth = kt + (size_t)hh * temp_stride * DH;
        const __nv_bfloat16* vth = vt + (size_t)hh * temp_stride * DH;
        const int nstage = sepm ? nc : nt;
        for (int i = tid; i < nstage * (DH / 8); i += blockDim.x) {
            const int j = i >> 4, c8 = (i & 15) * 8;
            const __nv_bfloat16* ksrc;
            const __nv_bfloat16* vsrc;
            if (j < nc) { ksrc = kh + (size_t)(t0min + j) * DH; vsrc = vh + (size_t)(t0min + j) * DH; }
            else if (fuse) continue;     // computed below from the QKV output
            else { const int row = urow[j - nc]; ksrc = kth + (size_t)row * DH; vsrc = vth + (size_t)row * DH; }
            const uint32_t off = (uint32_t)(j * LDK + c8) * 2u;
            cp_async16(tk_a + off, ksrc + c8, 16);
            cp_async16(tv_a + off, vsrc + c8, 16);
        }
        if (fuse && !sepm) stage_incall(tid, (int)blockDim.x);
        asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const __nv_bfloat16* TK = reinterpret_cast<const __nv_bfloat16*>(smem + LY.tk);
    const __nv_bfloat16* TV = reinterpret_cast<const __nv_bfloat16*>(smem + LY.tv);
    const __nv_bfloat16* IK = reinterpret_cast<const __nv_bfloat16*>(smem + LY.ik);
    const __nv_bfloat16* IV = reinterpret_cast<const __nv_bfloat16*>(smem + LY.iv);
    // row of tail slot j: committed keys first, then the in-call keys (in the
    // separate region in the separate layout)
    auto key_row = [&](int j) { return (sepm && j >= nc) ? IK + (size_t)(j - nc) * LDK : TK + (size_t)j * LDK; };
    auto val_row = [&](int j) { return (sepm && j >= nc) ? IV + (size_t)(j - nc) * LDK : TV + (size_t)j * LDK; };
    int* swr = sw + warp * MAX_TAIL;
    float* pwr = pw + warp * MAX_TAIL;
    // Tail scores on tensor cores: S = Q K^T for the tile's rows against every
    // staged tail key (the union of the rows' keys).  An output element of
    // the mma depends only on its query row and its key, so S[r][key] is the
    // same whichever rows share the tile; each row then reads its own keys.
    float* ssc = reinterpret_cast<float*>(smem + LY.ssc);
    const int SSP = (int)LY.ssp;
    for (int nti = warp; nti * 8 < nt; nti += FT) {
        float c4[4] = {0.f, 0.f, 0.f, 0.f};
        const int kr = min(nti * 8 + g, nt - 1);
        const __nv_bfloat16* krow = key_row(kr) + 2 * t;
#pragma unroll
        for (int ks8 = 0; ks8 < 8; ++ks8) {
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow + ks8 * 16);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(krow + ks8 * 16 + 8);
            mma16816(c4, qa[ks8], b0, b1);
        }
        const int col = nti * 8 + 2 * t;
        if (col < nt) { ssc[g * SSP + col] = c4[0]; ssc[(g + 8) * SSP + col] = c4[2]; }
        if (col + 1 < nt) { ssc[g * SSP + col + 1] = c4[1]; ssc[(g + 8) * SSP + col + 1] = c4[3]; }
    }
    __syncthreads();
    for (int r = warp; r < nr; r += FT) {
        const int pos = rpos[r], t0 = rt0[r];
        const int n = pos - t0 + 1;                  // tail keys, positions t0 .. pos
        const int Kr = prefill ? pos + 1 : K;
        // scores: lane owns keys t0 + lane + 32 i
        float sc[MAX_TAIL / 32];
        int slot[MAX_TAIL / 32];
#pragma unroll
        for (int i = 0; i < MAX_TAIL / 32; ++i) {
            const int j = lane + 32 * i;
            const int p = t0 + j;
            slot[i] = (j < n) ? ((p < Kr) ? (p - t0min) : (nc + uslot[spath[r * PM + (p - K)]])) : 0;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < MAX_TAIL / 32; ++i)
            sc[i] = (lane + 32 * i < n) ? __fmul_rn(ssc[r * SSP + slot[i]], scale) : -INFINITY;
        float tm = sc[0];
#pragma unroll
        for (int i = 1; i < MAX_TAIL / 32; ++i) tm = fmaxf(tm, sc[i]);
        tm = warp_max(tm);
        float psum = 0.f;
#pragma unroll
        for (int i = 0; i < MAX_TAIL / 32; ++i) {
            const float pv = (sc[i] == -INFINITY) ? 0.f : expf(__fsub_rn(sc[i], tm));
            psum = __fadd_rn(psum, pv);
            const int j = lane + 32 * i;
            if (j < n) { pwr[j] = pv; swr[j] = slot[i]; }
        }
        const float tl = warp_sum(psum);
        __syncwarp();
        // P V in key order; lane owns dims 4 lane .. 4 lane + 3
        float to[4] = {0.f, 0.f, 0.f, 0.f};
        int j = 0;
        for (; j + 4 <= n; j += 4) {
            uint2 vv[4];
            float pk[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                pk[u] = pwr[j + u];
                vv[u] = *reinterpret_cast<const uint2*>(val_row(swr[j + u]) + lane * 4);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                to[0] = fmaf(pk[u], __uint_as_float(vv[u].x << 16), to[0]);
                to[1] = fmaf(pk[u], __uint_as_float(vv[u].x & 0xffff0000u), to[1]);
                to[2] = fmaf(pk[u], __uint_as_float(vv[u].y << 16), to[2]);
                to[3] = fmaf(pk[u], __uint_as_float(vv[u].y & 0xffff0000u), to[3]);
            }
        }
        for (; j < n; ++j) {
            const float pk = pwr[j];
            const uint2 vv = *reinterpret_cast<const uint2*>(val_row(swr[j]) + lane * 4);
            to[0] = fmaf(pk, __uint_as_float(vv.x << 16), to[0]);
            to[1] = fmaf(pk, __uint_as_float(vv.x & 0xffff0000u), to[1]);
            to[2] = fmaf(pk, __uint_as_float(vv.y << 16), to[2]);
            to[3] = fmaf(pk, __uint_as_float(vv.y & 0xffff0000u), to[3]);
        }
        __syncwarp();
        // merge the tail block after the committed blocks, normalise
        const float m = wmax[r], l = wl[r];
        const float4 oc = *reinterpret_cast<const float4*>(os + r * DH + lane * 4);
        const float mn = fmaxf(m, tm);
        const float ca = (m == -INFINITY) ? 0.f : expf(__fsub_rn(m, mn));
        const float cb = expf(__fsub_rn(tm, mn));
        const float inv = 1.0f / fmaf(l, ca, __fmul_rn(tl, cb));
        const float o0 = fmaf(oc.x, ca, __fmul_rn(to[0], cb));
        const float o1 = fmaf(oc.y, ca, __fmul_rn(to[1], cb));
        const float o2 = fmaf(oc.z, ca, __fmul_rn(to[2], cb));
        const float o3 = fmaf(oc.w, ca, __fmul_rn(to[3], cb));
        __nv_bfloat16* op = out + (size_t)(r0 + r) * H * DH + hh * DH + lane * 4;
        *reinterpret_cast<__nv_bfloat162*>(op) = __floats2bfloat162_rn(__fmul_rn(o0, inv), __fmul_rn(o1, inv));
        *reinterpret_cast<__nv_bfloat162*>(op + 2) = __floats2bfloat162_rn(__fmul_rn(o2, inv), __fmul_rn(o3, inv));
    }
}

}  // namespace

int la_attn_tail_blocks(int pmax) { return (pmax + 31) / 32; }

// keys the ring must hold: two committed blocks, or the tail keys of a tile
// (committed positions [t0min, K) or a prefill tile's span, plus the call's rows)
static int ring_keys_for(int TB, int Qmax) {
    const int tail = 32 * (TB + 1) + FR + Qmax;
    return tail > 2 * BLK ? tail : 2 * BLK;
}

// tail_rows: the most temporary rows a tile's paths reach (the ring's share
// for them); qrows: the most temporary rows a request has
size_t la_attn_smem_bytes(int TB, int tail_rows, int pmax, int qrows) {
    return fused_layout(ring_keys_for(TB, tail_rows), pmax, qrows).total + 1024;   // + alignment slack
}

cudaError_t la_launch_attention_bf16(const LaDev& d, cudaStream_t st, const void* qbuf, const void* kc, const void* vc,
                                     const void* kt, const void* vt, void* out, int H, int sel, int Qcap,
                                     int max_ctx, int Qmax, int rows_cap, int TB, int pmax, const CUtensorMap& cmap,
                                     int krow0, int vrow0, const LaHdr* const* req_hdr, int qstride,
                                     long long req_cache_elems, int req_cache_rows, int temp_stride, int tail_rows,
                                     const LaRope* rope) {
    if (TB + 1 > MAX_TAIL / 32) return cudaErrorInvalidValue;
    if (tail_rows <= 0 || tail_rows > Qmax) tail_rows = Qmax;
    int ring_keys = ring_keys_for(TB, tail_rows);
    size_t smem = la_attn_smem_bytes(TB, tail_rows, pmax, Qmax);
    // the separate layout (in-call keys staged while the blocks run) where
    // it fits: decode calls with RoPE folded in (LA_ATTN_SEP=0: never)
    const char* sep_e = getenv("LA_ATTN_SEP");       // read per launch (graphs record it at capture)
    const int sep_env = (sep_e && sep_e[0] == '0') ? 0 : 1;
    // committed tail keys of a tile: K - t0min <= 31 + 32 TB; in-call keys:
    // at most tail_rows, plus a tile's slack
    const int ck = 32 * (TB + 1), keys_sep = ck + FR + tail_rows;
    int sep = 0;
    if (sep_env && rope && sel != SEL_PREFILL) {
        const FusedLayout L = fused_layout(keys_sep, pmax, Qmax, 1, ck);
        if (L.ring_used <= L.ring_bytes && (size_t)L.total + 1024 <= 227 * 1024) {
            sep = 1;
            smem = (size_t)L.total + 1024;
            ring_keys = keys_sep;
        }
    }
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    dim3 grid(H, (rows_cap + FR - 1) / FR);
    return la_launch_pdl(k_attn_fused, grid, dim3(FT * 32), smem, st, d, (const __nv_bfloat16*)qbuf,
                         (const __nv_bfloat16*)kc, (const __nv_bfloat16*)vc, (const __nv_bfloat16*)kt,
                         (const __nv_bfloat16*)vt, (__nv_bfloat16*)out, sel, Qcap, max_ctx,
                         temp_stride ? temp_stride : Qmax, TB, H, ring_keys,
                         cmap, krow0, vrow0, req_hdr, qstride, req_cache_elems, req_cache_rows, Qmax,
                         rope ? *rope : LaRope{nullptr, LaSplit{}, nullptr, nullptr}, sep, ck);
}
