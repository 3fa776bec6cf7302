// Tensor-core GEMM of the packed call on sm_103a: Y[q][n] = sum_k X[q][k] W[n][k]
// for the QKV, O, gate/up (SwiGLU) and down projections and the LM head.
//
// The call is a skinny contraction: Q packed rows against a weight matrix
// that streams from HBM once per call, so the kernel is built to keep every
// SM streaming weights:
//   - persistent stream-K: one CTA per SM; the (128-row weight tile, K slice
//     of two 64-column atoms, one for gate/up) units of the whole matrix are
//     split into equal contiguous ranges, one per CTA, so every SM moves the
//     same number of bytes;
//   - warp 0 streams units through a multi-stage mbarrier ring: the weights,
//     repacked once at init into unit-contiguous 128-byte-swizzled images,
//     by one bulk copy per unit (L2 evict-first), the q x 64 activation tiles
//     by TMA (128-byte swizzle); weight stages sit at fixed offsets,
//     activation stages are counted back from the ring's end and sized by
//     the call's rows; warp 1 issues tcgen05.mma (kind::f16, bf16 in, fp32 in
//     TMEM, M = 128 weight rows, N = q rounded up to 16); warps 2-5 drain the
//     accumulator with tcgen05.ld;
//   - two TMEM accumulators alternate between the K segments a CTA owns, so
//     the MMA warp starts the next tile while the epilogue drains the last;
//   - a tile whose K range spans several CTAs: each contributor publishes its
//     fp32 partial (L2) and goes on streaming.  The layer projections leave
//     the partials to the kernel that reads their output (`defer`: RoPE,
//     RMSNorm and SwiGLU add the segments in K order); otherwise (the LM
//     head) a contributor waits (bounded) after its last unit for the tile's
//     other partials and finishes its own slice of the tile's packed rows,
//     adding the partials in segment (K) order;
//   - all row chunks of a call (BN_MAX packed rows each) run inside the same
//     grid of at most one CTA per SM, so the contributors of a tile are
//     resident together.
// The partition depends only on the weight shape and the SM count, never on
// Q, so a row's result does not depend on how many rows share the call.
//
// Every wait on an mbarrier is bounded; a wait that runs out sets the device
// error word (LA_ETIMEOUT); the CTA then skips its outputs, frees its TMEM
// and returns.
#include "la_common.cuh"
#include "la_kernels.h"
#include "la_tc.cuh"

#include <cudaTypedefs.h>
#include <algorithm>
#include <cstdlib>

namespace {

using namespace latc;

constexpr int BOX_ROWS = 16;
constexpr int MAX_STAGES = 12;
constexpr int SMEM_BYTES = 220 * 1024;
constexpr int NTHREADS = 192;             // producer, MMA, 4 epilogue warps
constexpr int MAX_CHUNKS = 4;             // packed rows per launch <= MAX_CHUNKS * BN_MAX

struct TcParams {
    LaHdr* hdr;
    LaTlRec* tl;                     // kernel timeline table, or nullptr
    int sel, mode, K, Nout, k_tiles, n_tiles, seg_tiles, n_cta, max_seg;
    int ns, max_ns, rows_cap;        // stages at rows_cap rows (issued before the header), stage limit, rows per launch at most
    int ua, k_atoms;                 // 64-column atoms per unit (the last unit of a tile may hold fewer), K / 64
    const uint8_t* wpack;            // unit-contiguous weight images (la_tc_pack), or null: the tensor maps
    void* out; int ldo;
    float* logits; int ld_logits;
    float* ws; unsigned long long* ctr;   // this GEMM's split-tile arrival counters
    float* part_v; int* part_i; int part_stride;
    int max_chunks;
    int defer;            // split tiles left as partials for the consumer
    int pair;             // units of two adjacent output tiles (planes 0, 1) x one atom
};

__global__ void __launch_bounds__(NTHREADS, 1)
k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
          const __grid_constant__ CUtensorMap tmA3, const __grid_constant__ CUtensorMap tmB,
          const __grid_constant__ CUtensorMap tmB32, const __grid_constant__ CUtensorMap tmB64,
          const __grid_constant__ CUtensorMap tmB128, const __grid_constant__ CUtensorMap tmB256, TcParams p) {
    LaTl la_tl_(LA_TL_GEMM_TC, p.tl);
    LaHdr* h = p.hdr;
    const int swiglu = (p.mode == GEMM_SWIGLU);
    const int nA = (swiglu || p.pair) ? 2 : 1;     // weight matrices of a unit (accumulators)
    const long long T = (long long)p.n_tiles * p.k_tiles;
    // never more CTAs than units: every CTA then owns at least one unit and the
    // owners of one tile are consecutive CTAs
    const int P = (int)(T < (long long)p.n_cta ? T : (long long)p.n_cta), c = blockIdx.x;
    if (c >= P) return;
    const long long u_begin = T * c / P, u_end = T * (c + 1) / P;
    const int n_units = (int)(u_end - u_begin);
    const int tile0 = (int)(u_begin / p.k_tiles), kt0 = (int)(u_begin % p.k_tiles);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    // [barriers][flags][reduction scratch 8 KB][stages: weights][stages: activations]
    const uint32_t bar_full = base;                                   // MAX_STAGES x 8 B
    const uint32_t bar_empty = base + 8 * MAX_STAGES;
    const uint32_t bar_accf = base + 16 * MAX_STAGES;                 // 2 x 8 B
    const uint32_t bar_acce = bar_accf + 16;                          // 2 x 8 B
    uint8_t* flags = gbase + (bar_acce + 16 - base);
    uint32_t* tmem_slot = (uint32_t*)flags;
    int* s_flag = (int*)(flags + 8);
    int* s_rows = (int*)(flags + 12);                                 // header broadcast: rows, or -1 to skip the call
    float* rv = (float*)(gbase + 1024);                               // [4][BN_MAX] argmax values
    int* ri = (int*)(gbase + 1024 + 4 * BN_MAX * 4);                  // [4][BN_MAX] argmax ids
    const uint32_t a_stage = (uint32_t)(nA * p.ua) * A_BYTES;         // one unit's weight tiles (at most)
    // Weight stage s starts at wring + s * a_stage whatever the row count;
    // activation stage s ends at ring_end - s * b_stage, b_stage set by the
    // call's rows.  ns(rows) * (a_stage + b_stage) fits, and ns(rows) >=
    // p.ns = ns(rows_cap), so the weights of p.ns stages are issued before
    // the header is read and before the dependency wait.
    const uint32_t wring = base + 1024 + 8192;
    const uint32_t ring_end = base + SMEM_BYTES;
    const int n_pre = min(p.ns, n_units);

    // unit u = (tile, kt) covers atoms kt * ua .. + atoms_of(u) - 1 of its tile
    auto atoms_of = [&](long long u) { return min(p.ua, p.k_atoms - (int)(u % p.k_tiles) * p.ua); };
    // weight tiles of unit u into stage s (the stage's barrier already expects
    // them): atom i of matrix a at (i * nA + a) x 16 KB, the packed order
    auto load_w = [&](int s, long long u, uint64_t pol) {
        const uint32_t fb = bar_full + 8 * s, st = wring + (uint32_t)s * a_stage;
        const int tile = (int)(u / p.k_tiles), at0 = (int)(u % p.k_tiles) * p.ua, na = atoms_of(u);
        if (p.wpack) {
            bulk_load(st, p.wpack + ((size_t)tile * p.k_atoms + at0) * nA * A_BYTES, (uint32_t)(na * nA) * A_BYTES, fb,
                      pol);
        } else {
            const CUtensorMap* wmap = &tmA;
            int wrow = tile * BM;
            if (p.seg_tiles > 0) {
                const int seg = tile / p.seg_tiles;
                wmap = seg == 0 ? &tmA : (seg == 1 ? &tmA2 : &tmA3);
                wrow = (tile - seg * p.seg_tiles) * BM;
            }
            for (int i = 0; i < na; ++i) {
                tma_load_2d(st + (uint32_t)(i * nA) * A_BYTES, wmap, fb, (at0 + i) * BK, wrow, pol);
                if (swiglu) tma_load_2d(st + (uint32_t)(i * nA + 1) * A_BYTES, &tmA2, fb, (at0 + i) * BK, wrow, pol);
            }
        }
    };

    la_pdl_trigger();
    if (warp == 0) {
        int hdr_rows = 0;
        if (lane == 0) {
            for (int s = 0; s < MAX_STAGES; ++s) {
                mbar_init(bar_full + 8 * s, 1);
                mbar_init(bar_empty + 8 * s, 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(bar_accf + 8 * b, 1);
                mbar_init(bar_acce + 8 * b, 1);
            }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            uint64_t pol_w;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
            // expect_tx without arriving: a stage completes only once its
            // activation rows (registered with the arrival below) have landed too
            for (int i = 0; i < n_pre; ++i) {
                const uint32_t wb = (uint32_t)(atoms_of(u_begin + i) * nA) * A_BYTES;
                asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(bar_full + 8 * i), "r"(wb) : "memory");
                load_w(i, u_begin + i, pol_w);
            }
            // The weights depend on no earlier kernel, and neither do the
            // header fields read next (written at least three launches back,
            // la_common.cuh); the activations, written by the kernel before
            // this one, are loaded after the wait.
            const int h_err = h->err, h_done = h->done;
            const int h_n = p.sel == SEL_CALL ? h->Q : (p.sel == SEL_PREFILL ? h->prefill_rows : h->n_need);
            int rows = h_n;
            if (h_err != 0 || (p.sel != SEL_PREFILL && h_done != 0) || rows <= 0) rows = -1;
            if (rows > p.rows_cap || (rows > 0 && (rows + BN_MAX - 1) / BN_MAX > p.max_chunks)) {
                if (blockIdx.x == 0) la_set_err(h, LA_EDEVICE);
                rows = -1;
            }
            la_pdl_wait();
            *s_rows = rows;
            hdr_rows = rows;
        }
        __syncwarp();
        asm volatile("bar.arrive 2, 192;" ::: "memory");
        hdr_rows = __shfl_sync(0xffffffffu, hdr_rows, 0);
        if (lane == 0) {
            const int rows = hdr_rows;
            if (rows < 0) {
                // skipped call: let the weight loads already issued land before exiting
                for (int i = 0; i < n_pre; ++i) {
                    mbar_arrive(bar_full + 8 * i);
                    mbar_wait(bar_full + 8 * i, 0);
                }
            } else {
                // TMA producer: every (chunk, unit) of this CTA, in order
                const int n_chunks = (rows + BN_MAX - 1) / BN_MAX;
                const uint32_t b_atom = (uint32_t)((min(BN_MAX, rows) + 15) & ~15) * ROW_BYTES;
                const uint32_t b_stage = (uint32_t)p.ua * b_atom;
                const int ns = min(p.max_ns, (int)((SMEM_BYTES - 1024 - 8192) / (a_stage + b_stage)));
                uint64_t pol_w, pol_x;
                asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
                asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
                bool ok = true;
                int y = 0, iu = 0, s = 0, r = 0;
                const int n_items = n_chunks * n_units;
                for (int it = 0; it < n_items; ++it) {
                    const int q0 = y * BN_MAX;
                    const int BN = (min(BN_MAX, rows - q0) + 15) & ~15;
                    if (r > 0 && !mbar_wait(bar_empty + 8 * s, (uint32_t)((r - 1) & 1))) { ok = false; break; }
                    const uint32_t bst = ring_end - (uint32_t)(s + 1) * b_stage;
                    const uint32_t fb = bar_full + 8 * s;
                    const long long u = u_begin + iu;
                    const int at0 = (int)(u % p.k_tiles) * p.ua, na = atoms_of(u);
                    const uint32_t xb = (uint32_t)(na * BN) * ROW_BYTES;
                    if (it < n_pre) {
                        // the weight tiles are already on their way
                        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(xb) : "memory");
                    } else {
                        mbar_expect_tx(fb, (uint32_t)(na * nA) * A_BYTES + xb);
                        load_w(s, u, pol_w);
                    }
                    // per atom, the activation rows in at most four boxes (256/128/64/32/16 rows)
                    for (int i = 0; i < na; ++i) {
                        int rr = 0;
                        while (rr < BN) {
                            const int left = BN - rr;
                            const CUtensorMap* bm = left >= 256 ? &tmB256 : left >= 128 ? &tmB128 : left >= 64 ? &tmB64
                                                  : left >= 32 ? &tmB32 : &tmB;
                            const int hgt = left >= 256 ? 256 : left >= 128 ? 128 : left >= 64 ? 64 : left >= 32 ? 32 : 16;
                            tma_load_2d(bst + (uint32_t)i * b_atom + (uint32_t)rr * ROW_BYTES, bm, fb, (at0 + i) * BK,
                                        q0 + rr, pol_x);
                            rr += hgt;
                        }
                    }
                    if (++iu == n_units) { iu = 0; ++y; }
                    if (++s == ns) { s = 0; ++r; }
                }
                if (!ok) la_set_err(h, LA_ETIMEOUT);
            }
        }
    } else {
        if (warp == 1) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
        la_pdl_wait();
        tc_fence_before();
        asm volatile("bar.sync 2, 192;" ::: "memory");
        tc_fence_after();
    }
    const int rows = *s_rows;
    const uint32_t tmem = *tmem_slot;
    const int n_chunks = rows > 0 ? (rows + BN_MAX - 1) / BN_MAX : 0;
    const int BN0 = rows > 0 ? (min(BN_MAX, rows) + 15) & ~15 : 16;
    const int acc_cols = nA * BN0;                         // one accumulator: nA x BN fp32 columns
    const int nbuf = (2 * acc_cols <= TMEM_COLS) ? 2 : 1;
    const uint32_t b_atom = (uint32_t)BN0 * ROW_BYTES, b_stage = (uint32_t)p.ua * b_atom;
    const int ns = min(p.max_ns, (int)((SMEM_BYTES - 1024 - 8192) / (a_stage + b_stage)));

    if (warp == 0) {
        // producer (above)
    } else if (warp == 1) {
        if (lane == 0 && n_chunks > 0) {
            // MMA issuer: one accumulator per K segment, alternating buffers
            bool ok = true;
            int y = 0, iu = 0, kt = kt0, s = 0, r = 0, seg_i = 0;
            while (y < n_chunks && ok) {
                const int seg_len = min(n_units - iu, p.k_tiles - kt);
                const int BN = (min(BN_MAX, rows - y * BN_MAX) + 15) & ~15;
                const uint32_t id = idesc_bf16(BN);
                const int b = nbuf == 2 ? (seg_i & 1) : 0, ub = nbuf == 2 ? (seg_i >> 1) : seg_i;
                if (ub > 0 && !mbar_wait(bar_acce + 8 * b, (uint32_t)((ub - 1) & 1))) { ok = false; break; }
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * acc_cols);
                for (int j = 0; j < seg_len; ++j) {
                    if (!mbar_wait(bar_full + 8 * s, (uint32_t)(r & 1))) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t st = wring + (uint32_t)s * a_stage;
                    const uint32_t bst = ring_end - (uint32_t)(s + 1) * b_stage;
                    const int na = min(p.ua, p.k_atoms - (kt + j) * p.ua);
                    for (int i = 0; i < na; ++i) {
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t bdesc = sdesc(bst + (uint32_t)i * b_atom + kk * 32);
                            const uint32_t accum = (j == 0 && i == 0 && kk == 0) ? 0u : 1u;
                            const uint32_t sa = st + (uint32_t)(i * nA) * A_BYTES + kk * 32;
                            mma_bf16(acc, sdesc(sa), bdesc, id, accum);
                            if (nA == 2) mma_bf16(acc + (uint32_t)BN, sdesc(sa + A_BYTES), bdesc, id, accum);
                        }
                    }
                    mma_commit(bar_empty + 8 * s);
                    if (++s == ns) { s = 0; ++r; }
                }
                if (!ok) break;
                mma_commit(bar_accf + 8 * b);
                ++seg_i;
                iu += seg_len;
                kt += seg_len;
                if (kt == p.k_tiles) kt = 0;
                if (iu == n_units) { iu = 0; ++y; kt = kt0; }
            }
            if (!ok) la_set_err(h, LA_ETIMEOUT);
        }
    } else {
        // epilogue warps 2-5: TMEM lane quarter (warp % 4)
        const int quarter = warp & 3;
        const int et = quarter * 32 + lane;                // 0..127: the weight row within the tile
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const size_t plane = (size_t)BN_MAX * BM;          // floats of one accumulator in a partial record

        // Results of packed rows q0 + cb .. q0 + cb + ncol - 1 for weight row
        // tile * BM + et (v: the accumulator, w2: the SwiGLU up accumulator).
        // Loads of a group are issued together; lanes of a warp hold 32
        // consecutive weight rows, so every access is one coalesced line.
        auto emit_group = [&](int tile, int q0, int cb, int ncol, const float (&v)[16], const float (&w2)[16],
                              bool ok) {
            const int n = tile * BM + et;
            if (p.mode == GEMM_STORE) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (ok && j < ncol)
                        ((__nv_bfloat16*)p.out)[(size_t)(q0 + cb + j) * p.ldo + n] = __float2bfloat16_rn(v[j]);
            } else if (p.mode == GEMM_RESID) {
                float old[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    old[j] = ((const float*)p.out)[(size_t)(q0 + cb + min(j, ncol - 1)) * p.ldo + n];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (ok && j < ncol) ((float*)p.out)[(size_t)(q0 + cb + j) * p.ldo + n] = old[j] + v[j];
            } else if (p.mode == GEMM_SWIGLU) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (ok && j < ncol)
                        ((__nv_bfloat16*)p.out)[(size_t)(q0 + cb + j) * p.ldo + n] =
                            __float2bfloat16_rn(v[j] / (1.0f + expf(-v[j])) * w2[j]);
            } else {   // logits + argmax partials over this tile's 128 vocab entries
                if (ok && p.logits) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < ncol) p.logits[(size_t)(q0 + cb + j) * p.ld_logits + n] = v[j];
                }
                // 16 independent warp reductions, interleaved level by level
                float bv[16];
                int bi[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) { bv[j] = v[j]; bi[j] = n; }
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float vv = __shfl_xor_sync(0xffffffffu, bv[j], o2);
                        const int ii = __shfl_xor_sync(0xffffffffu, bi[j], o2);
                        better(bv[j], bi[j], vv, ii);
                    }
                }
                if (lane == 0) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < ncol) { rv[quarter * BN_MAX + cb + j] = bv[j]; ri[quarter * BN_MAX + cb + j] = bi[j]; }
                }
            }
        };
        // logits mode: combine the four lane quarters' argmax of columns [c_lo, c_hi)
        auto argmax_out = [&](int tile, int q0, int c_lo, int c_hi, bool ok) {
            if (p.mode != GEMM_LOGITS) return;
            epi_sync();
            for (int cc = c_lo + et; cc < c_hi; cc += 128) {
                float bv = rv[cc];
                int bi = ri[cc];
                for (int w = 1; w < 4; ++w) better(bv, bi, rv[w * BN_MAX + cc], ri[w * BN_MAX + cc]);
                if (ok) {
                    p.part_v[(size_t)tile * p.part_stride + q0 + cc] = bv;
                    p.part_i[(size_t)tile * p.part_stride + q0 + cc] = bi;
                }
            }
            epi_sync();
        };

        // split tiles this CTA contributed to, reduced after its last unit
        int d_tile[2 * MAX_CHUNKS], d_sg[2 * MAX_CHUNKS], d_nseg[2 * MAX_CHUNKS], d_y[2 * MAX_CHUNKS];
        unsigned long long d_target[2 * MAX_CHUNKS];         // the arrival count that completes the tile (leader)
        int nd = 0;
        int seg_i = 0;
        bool alive = true;
        int y = 0, iu = 0, tile = tile0, kt = kt0;
        while (y < n_chunks) {
            const int seg_len = min(n_units - iu, p.k_tiles - kt);
            const int q0 = y * BN_MAX;
            const int nq = min(BN_MAX, rows - q0);
            const int BN = (nq + 15) & ~15;
            const long long tile_u0 = (long long)tile * p.k_tiles, tile_u1 = tile_u0 + p.k_tiles;
            const int b = nbuf == 2 ? (seg_i & 1) : 0, ub = nbuf == 2 ? (seg_i >> 1) : seg_i;
            ++seg_i;
            const bool got = alive && mbar_wait(bar_accf + 8 * b, (uint32_t)(ub & 1));
            if (!got && alive) { alive = false; la_set_err(h, LA_ETIMEOUT); }
            tc_fence_after();
            const uint32_t acc = tmem + lane_base + (uint32_t)(b * acc_cols);
            const int c_first = cta_of(tile_u0, T, P), c_last = cta_of(tile_u1 - 1, T, P);
            const int nseg = c_last - c_first + 1;
            if (nseg > 1) {
                // publish this segment's partial (valid columns only) and free the accumulator
                const int sg = c - c_first;
                const size_t slot = (size_t)tile + (size_t)y * p.n_tiles;
                float* wsb = p.ws + ((slot * p.max_seg + sg) * nA) * plane;
                for (int c0 = 0; c0 < nq; c0 += 16) {
                    float v[16];
                    tmem_ld16(acc + c0, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < nq) __stcg(wsb + (size_t)(c0 + j) * BM + et, got ? v[j] : 0.f);
                    if (nA == 2) {
                        tmem_ld16(acc + BN + c0, v);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (c0 + j < nq) __stcg(wsb + plane + (size_t)(c0 + j) * BM + et, got ? v[j] : 0.f);
                    }
                }
                tc_fence_before();
                epi_sync();
                if (p.defer) {
                    // the consumer of this GEMM's output adds the segments
                    if (quarter == 0 && lane == 0) mbar_arrive(bar_acce + 8 * b);
                } else {
                    if (quarter == 0 && lane == 0) {
                        mbar_arrive(bar_acce + 8 * b);
                        // arrival (release: the CTA's partial stores, ordered before it by
                        // the barrier, are visible to whoever acquires the count).  The
                        // count only grows: arrival k completes launch k / nseg.
                        unsigned long long old;
                        asm volatile("atom.add.release.gpu.global.u64 %0, [%1], 1;"
                                     : "=l"(old)
                                     : "l"(p.ctr + slot)
                                     : "memory");
                        d_target[nd] = (old / (unsigned long long)nseg + 1ull) * (unsigned long long)nseg;
                    }
                    d_tile[nd] = tile; d_sg[nd] = sg; d_nseg[nd] = nseg; d_y[nd] = y;
                    ++nd;
                }
            } else {
                // a whole tile: straight from TMEM
                if (p.pair) {
                    // the unit's two output tiles in turn (the argmax scratch holds one)
                    for (int a = 0; a < 2; ++a) {
                        for (int c0 = 0; c0 < nq; c0 += 16) {
                            float v[16];
                            tmem_ld16(acc + (uint32_t)(a * BN) + c0, v);
                            emit_group(2 * tile + a, q0, c0, min(16, nq - c0), v, v, got);
                        }
                        if (a == 0) argmax_out(2 * tile, q0, 0, nq, got);
                    }
                } else {
                    for (int c0 = 0; c0 < nq; c0 += 16) {
                        float v[16], w2[16];
                        tmem_ld16(acc + c0, v);
                        if (nA == 2) tmem_ld16(acc + BN + c0, w2);
                        emit_group(tile, q0, c0, min(16, nq - c0), v, w2, got);
                    }
                }
                tc_fence_before();
                epi_sync();
                if (quarter == 0 && lane == 0) mbar_arrive(bar_acce + 8 * b);
                argmax_out(p.pair ? 2 * tile + 1 : tile, q0, 0, nq, got);
            }
            iu += seg_len;
            kt += seg_len;
            if (kt == p.k_tiles) { kt = 0; ++tile; }
            if (iu == n_units) { iu = 0; ++y; tile = tile0; kt = kt0; }
        }

        // Split tiles: once all nseg partials of this launch have arrived,
        // contributor sg sums columns [nq*sg/nseg, nq*(sg+1)/nseg) over the
        // segments in K order.
        for (int d = 0; d < nd; ++d) {
            const int tile = d_tile[d], sg = d_sg[d], nseg = d_nseg[d], y = d_y[d];
            const int q0 = y * BN_MAX;
            const int nq = min(BN_MAX, rows - q0);
            const size_t slot = (size_t)tile + (size_t)y * p.n_tiles;
            if (quarter == 0 && lane == 0) {
                bool ok = alive && spin_until64(p.ctr + slot, d_target[d]);
                if (!ok && alive) la_set_err(h, LA_ETIMEOUT);
                *s_flag = ok ? 1 : 0;
            }
            epi_sync();
            const bool ok = *s_flag != 0;
            alive = alive && ok;
            const int c_lo = nq * sg / nseg, c_hi = nq * (sg + 1) / nseg;
            const float* wst = p.ws + (slot * p.max_seg * nA) * plane + et;
            const size_t seg_stride = (size_t)nA * plane;
            if (p.pair) {
                // the unit's two output tiles in turn, each from its own plane
                for (int a = 0; a < 2; ++a) {
                    for (int cb = c_lo; cb < c_hi; cb += 16) {
                        float v[16];
                        const float* wa = wst + (size_t)a * plane;
                        if (nseg == 2) sum_segments<2, 16>(wa, seg_stride, nseg, cb, c_hi, v);
                        else if (nseg == 3) sum_segments<3, 16>(wa, seg_stride, nseg, cb, c_hi, v);
                        else sum_segments<4, 16>(wa, seg_stride, nseg, cb, c_hi, v);
                        emit_group(2 * tile + a, q0, cb, min(16, c_hi - cb), v, v, ok);
                    }
                    argmax_out(2 * tile + a, q0, c_lo, c_hi, ok);
                }
            } else {
                for (int cb = c_lo; cb < c_hi; cb += 16) {
                    float v[16], w2[16];
                    if (nseg == 2) {
                        sum_segments<2, 16>(wst, seg_stride, nseg, cb, c_hi, v);
                        if (nA == 2) sum_segments<2, 16>(wst + plane, seg_stride, nseg, cb, c_hi, w2);
                    } else if (nseg == 3) {
                        sum_segments<3, 16>(wst, seg_stride, nseg, cb, c_hi, v);
                        if (nA == 2) sum_segments<3, 16>(wst + plane, seg_stride, nseg, cb, c_hi, w2);
                    } else {
                        sum_segments<4, 16>(wst, seg_stride, nseg, cb, c_hi, v);
                        if (nA == 2) sum_segments<4, 16>(wst + plane, seg_stride, nseg, cb, c_hi, w2);
                    }
                    emit_group(tile, q0, cb, min(16, c_hi - cb), v, w2, ok);
                }
                argmax_out(tile, q0, c_lo, c_hi, ok);
            }
            // s_flag is rewritten by the next tile's leader only after this barrier
            epi_sync();
        }
    }
    // teardown: every warp reconverges (lane 0 of the producer and MMA warps
    // may still be finishing) before the CTA-wide barrier that frees TMEM
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
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

int la_tc_make_act_maps(TcGemm* g, const void* base, int rows, int K) {
    if (la_tc_make_map(&g->tmB, base, rows, K, 16) || la_tc_make_map(&g->tmB32, base, rows, K, 32) ||
        la_tc_make_map(&g->tmB64, base, rows, K, 64) || la_tc_make_map(&g->tmB128, base, rows, K, 128) ||
        la_tc_make_map(&g->tmB256, base, rows, K, 256))
        return -1;
    return 0;
}

// 1 unless LA_TC_DEFER=0 (A/B runs): the layer GEMMs leave split tiles to their consumers
int la_tc_defer_default() {
    static int v = -1;
    if (v < 0) {
        const char* e = getenv("LA_TC_DEFER");
        v = (e && e[0] == '0') ? 0 : 1;
    }
    return v;
}

// 64-column atoms per (tile, K) unit: two (one 32 KB copy) for a single
// weight matrix, one for the gate/up pair (already two 16 KB tiles)
static int unit_atoms(int mode, int pair = 0) { return (mode == GEMM_SWIGLU || pair) ? 1 : 2; }
int la_tc_unit_atoms(int mode, int pair) { return unit_atoms(mode, pair); }
int la_tc_k_units(int mode, int K, int pair) {
    const int atoms = K / BK, ua = unit_atoms(mode, pair);
    return (atoms + ua - 1) / ua;
}

LaSplit la_tc_split(const TcGemm& g, const TcWork& w) {
    LaSplit s;
    s.ws = g.defer ? w.ws : nullptr;
    s.n_tiles = g.Nout / BM / (g.pair ? 2 : 1);
    s.k_tiles = la_tc_k_units(g.mode, g.K, g.pair);
    const long long T = (long long)s.n_tiles * s.k_tiles;
    s.P = (int)std::min<long long>(g.n_cta, T);
    s.max_seg = g.max_seg;
    s.nA = (g.mode == GEMM_SWIGLU || g.pair) ? 2 : 1;
    s.pair = g.pair;
    return s;
}

// CTAs of the persistent kernel: one per SM of the current device
int la_tc_ctas() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 148;
    return sms;
}

// CTAs for a weight of n_tiles x k_tiles units: one per SM.  LA_TC_ALIGN=1
// (A/B runs) gives a weight whose tiles split into a whole number s of equal
// K ranges with at least 80 % of the SMs busy n_tiles * s CTAs instead (O and
// down: 128; measured 1.4 % slower per call than 152 with the packed-weight
// stream); LA_TC_SWIGLU_UNSPLIT=1 gives a gate/up pair with at least half as
// many tiles as SMs one CTA per tile.
int la_tc_pick_ctas(int n_tiles, int k_tiles, int mode) {
    const int sms = la_tc_ctas();
    static int unsplit = -1;
    if (unsplit < 0) {
        const char* e = getenv("LA_TC_SWIGLU_UNSPLIT");
        unsplit = (e && e[0] == '1') ? 1 : 0;
    }
    if (unsplit && mode == GEMM_SWIGLU && n_tiles <= sms && 2 * n_tiles >= sms) return n_tiles;
    static int align = -1;
    if (align < 0) {
        const char* e = getenv("LA_TC_ALIGN");
        align = (e && e[0] == '1') ? 1 : 0;
    }
    if (align && n_tiles <= sms) {
        const int s = std::min(sms / n_tiles, k_tiles);
        if (s >= 2 && n_tiles * s * 5 >= sms * 4) return n_tiles * s;
    }
    return sms;
}

// The largest number of CTAs that share one tile's K range (the partial
// segments the workspace must hold per tile).
int la_tc_max_segments(int n_tiles, int k_tiles, int n_cta) {
    const long long T = (long long)n_tiles * k_tiles;
    if ((long long)n_cta > T) n_cta = (int)T;
    int best = 1;
    for (int t = 0; t < n_tiles; ++t) {
        const long long u0 = (long long)t * k_tiles, u1 = u0 + k_tiles - 1;
        const int c0 = (int)(((u0 + 1) * n_cta - 1) / T), c1 = (int)(((u1 + 1) * n_cta - 1) / T);
        best = std::max(best, c1 - c0 + 1);
    }
    return best;
}

// Opt the kernel into its dynamic shared memory on the current device.
cudaError_t la_tc_prepare_device() {
    return cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES + 1024);
}

// Scratch the kernel needs for one problem: the split-tile partial sums
// (floats) and the per-tile arrival counters (ints).
void la_tc_scratch_need(int mode, int n_out, int K, int rows, int n_cta, size_t* ws_floats, size_t* n_counters) {
    const int tiles = n_out / BM, k_tiles = la_tc_k_units(mode, K), n_y = (rows + BN_MAX - 1) / BN_MAX;
    const int nA = mode == GEMM_SWIGLU ? 2 : 1;
    const int max_seg = la_tc_max_segments(tiles, k_tiles, n_cta);
    *ws_floats = (size_t)tiles * n_y * max_seg * nA * BN_MAX * BM;
    *n_counters = (size_t)LA_TC_CTR_PER_TILE * tiles * n_y;
}

// Ring stages at rows_cap rows (the weight stages issued before the header
// is read; a call with fewer rows gets more stages) and the stage limit.
// Each stage holds one unit's weight tiles and, per atom, the activation rows.
static void ring_shape(int mode, int pair, int rows_cap, int* ns, int* max_ns) {
    static int max_s = -1;
    if (max_s < 0) {
        const char* e = getenv("LA_TC_STAGES");   // pipeline-depth override for tuning runs
        max_s = e ? atoi(e) : MAX_STAGES;
        if (max_s < 2) max_s = 2;
        if (max_s > MAX_STAGES) max_s = MAX_STAGES;
    }
    const int bn = (std::min(BN_MAX, std::max(rows_cap, 1)) + 15) & ~15;
    const int ua = unit_atoms(mode, pair);
    const int a_stage = ((mode == GEMM_SWIGLU || pair) ? 2 : 1) * ua * A_BYTES;
    const int n = (SMEM_BYTES - 1024 - 8192) / (a_stage + ua * bn * ROW_BYTES);
    static int pre = -1;
    if (pre < 0) {
        const char* e = getenv("LA_TC_PRE");       // cap on the stages issued before the dependency wait (tuning runs)
        pre = e ? std::max(0, atoi(e)) : MAX_STAGES;
    }
    *max_ns = max_s;
    *ns = std::min(std::min(n, max_s), pre);
}

size_t la_tc_packed_bytes(const TcGemm& g) {
    return (size_t)g.Nout * g.K * 2 * (g.mode == GEMM_SWIGLU ? 2 : 1);
}

// Unit-contiguous weight images: unit (tile, kt) is nA blocks of 16 KB, each
// the 128 x 64 bf16 tile as the 128-byte-swizzled TMA load would leave it in
// shared memory (16-byte chunk c of row r at r * 128 + ((c ^ (r & 7)) * 16)).
// w0..w2: the segments (or gate, up) with seg_rows rows each.  pair: unit
// tile u holds output tiles 2u (block 0) and 2u + 1 (block 1).
__global__ void k_tc_pack(const uint4* w0, const uint4* w1, const uint4* w2, int seg_tiles, int nA, int n_tiles,
                          int K, int pair, uint4* dst) {
    const int k_tiles = K / BK;
    const long long total = (long long)n_tiles * k_tiles * nA * BM * 8;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        const int cc = (int)(i & 7), r = (int)((i >> 3) & 127);
        const long long ua = i >> 10;                     // unit * nA + a
        const int a = (int)(ua % nA);
        const long long u = ua / nA;
        const int tile = (int)(u / k_tiles), kt = (int)(u % k_tiles);
        const int out_tile = pair ? 2 * tile + a : tile;
        const uint4* src = w0;
        int row = out_tile * BM + r;
        if (nA == 2 && !pair) {
            src = a ? w1 : w0;
        } else if (seg_tiles > 0) {
            const int seg = out_tile / seg_tiles;
            src = seg == 0 ? w0 : (seg == 1 ? w1 : w2);
            row = (out_tile - seg * seg_tiles) * BM + r;
        }
        const uint4 v = src[((size_t)row * K + (size_t)kt * BK) / 8 + cc];
        dst[(size_t)ua * (A_BYTES / 16) + r * 8 + (cc ^ (r & 7))] = v;
    }
}

cudaError_t la_tc_pack(const TcGemm& g, const void* w1, const void* w2, const void* w3, void* dst, cudaStream_t st) {
    const int nA = (g.mode == GEMM_SWIGLU || g.pair) ? 2 : 1;
    const int n_tiles = g.Nout / BM / (g.pair ? 2 : 1);
    if (g.pair && (g.mode == GEMM_SWIGLU || (g.Nout / BM) % 2 || (g.seg_tiles % 2))) return cudaErrorInvalidValue;
    k_tc_pack<<<1024, 256, 0, st>>>((const uint4*)w1, (const uint4*)(w2 ? w2 : w1), (const uint4*)(w3 ? w3 : w1),
                                    g.seg_tiles, nA, n_tiles, g.K, g.pair, (uint4*)dst);
    return cudaGetLastError();
}

cudaError_t la_launch_gemm_tc(const LaDev& d, cudaStream_t st, const TcGemm& g, const TcWork& w, int sel,
                              int rows_cap) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES + 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    if (rows_cap < 1 || rows_cap > MAX_CHUNKS * BN_MAX) return cudaErrorInvalidValue;
    TcParams p;
    p.hdr = d.hdr;
    p.tl = d.tl;
    p.sel = sel;
    p.mode = g.mode;
    p.K = g.K;
    p.Nout = g.Nout;
    if (g.pair && (!g.wpack || g.mode == GEMM_SWIGLU || (g.Nout / BM) % 2))
        return cudaErrorInvalidValue;
    p.pair = g.pair;
    p.k_tiles = la_tc_k_units(g.mode, g.K, g.pair);
    p.ua = unit_atoms(g.mode, g.pair);
    p.k_atoms = g.K / BK;
    p.n_tiles = g.Nout / BM / (g.pair ? 2 : 1);
    p.seg_tiles = g.seg_tiles;
    p.n_cta = g.n_cta;
    p.max_seg = g.max_seg;
    ring_shape(g.mode, g.pair, rows_cap, &p.ns, &p.max_ns);
    p.rows_cap = rows_cap;
    p.wpack = (const uint8_t*)g.wpack;
    p.out = g.out;
    p.ldo = g.ldo;
    p.logits = g.logits;
    p.ld_logits = g.ld_logits;
    p.ws = w.ws;
    p.ctr = (unsigned long long*)w.counters + g.ctr_off;
    p.part_v = w.part_v;
    p.part_i = w.part_i;
    p.part_stride = w.part_stride;
    p.max_chunks = (rows_cap + BN_MAX - 1) / BN_MAX;
    p.defer = g.defer;
    const long long T = (long long)p.n_tiles * p.k_tiles;
    dim3 grid((unsigned)std::min<long long>(g.n_cta, T), 1);
    return la_launch_pdl(k_gemm_tc, grid, dim3(NTHREADS), (size_t)(SMEM_BYTES + 1024), st, g.tmA, g.tmA2, g.tmA3, g.tmB,
                         g.tmB32, g.tmB64, g.tmB128, g.tmB256, p);
}
