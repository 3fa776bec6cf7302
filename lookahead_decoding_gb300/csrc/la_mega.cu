// Layer-chain kernel of the packed decode call on sm_103a.
//
// Between two attention launches a decode call runs a fixed chain of dense
// phases: the O projection, the residual RMSNorm, the gate/up projection,
// SwiGLU, the down projection, the next layer's RMSNorm and its QKV
// projection (at the end of the call: the final RMSNorm of the needed rows
// and the LM head).  k_mega runs one such chain in a single launch of one CTA
// per SM:
//   - every GEMM phase is the stream-K tcgen05 GEMM of la_gemm_tc.cu: the
//     same (tile, K slice) units per CTA, the same MMA order into TMEM, the
//     same split-tile partial records (left to the consumer phase) and
//     epilogues;
//   - every row phase is the arithmetic of the RMSNorm or SwiGLU kernel of
//     la_model.cu in the same order (the RMSNorm sum of squares as 1024 or
//     256 virtual threads with the same butterflies), so each value equals
//     the multi-launch path bit for bit;
//   - warp 0 streams the weights of all GEMMs of the chain, in order, through
//     one mbarrier ring and never waits for activations: while a phase's
//     inputs are being produced elsewhere, the next GEMM's weights are
//     already arriving;
//   - warps 6-11 copy each unit's activation rows (L2) into the ring with
//     cp.async once the phase that writes them has completed on every CTA,
//     several units in flight; warp 1 issues tcgen05.mma; warps 2-5 drain
//     TMEM; all of warps 2-11 run the row phases;
//   - a phase completes grid-wide through its own arrival counter: each CTA
//     adds 1 once its part of the phase is in memory (release), and phase k
//     is complete when counter k reaches gridDim.x (acquire).  One counter
//     per phase, because a CTA with no part in phase k + 1 (no units of that
//     GEMM) arrives for it as soon as its own part of phase k is done, before
//     phase k is complete elsewhere.  The grid is one CTA per SM, resident
//     together.
// Every wait (mbarrier or counter) is bounded: on expiry the CTA sets the
// device error word (LA_ETIMEOUT), stops producing, frees its TMEM and
// returns; the waits of the other CTAs then run out too.
#include "la_common.cuh"
#include "la_kernels.h"
#include "la_tc.cuh"

#include <algorithm>

namespace {

using namespace latc;

constexpr int MG_THREADS = 384;            // 12 warps
constexpr int MG_SMEM = 220 * 1024;        // dynamic shared memory used (+1024 alignment slack)
constexpr int MG_SCRATCH = 1024 + 8192;    // barriers, flags, reductions; argmax scratch
constexpr int MG_MAX_STAGES = 12;
constexpr int MG_A_STAGE = 2 * A_BYTES;    // weights of one unit: 32 KB in every mode
constexpr int N_WORKERS = 320;             // warps 2..11
constexpr int BAR_EPI = 1, BAR_WORK = 4;

__device__ __forceinline__ void named_sync(int id, int n) {
    __syncwarp();
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// the units of GEMM g that CTA c streams (the partition of la_gemm_tc.cu)
struct Units {
    long long T, u0, u1;
    int P;
};
__device__ __forceinline__ Units units_of(const MgGemm& g, int c) {
    Units r;
    r.T = (long long)g.n_tiles * g.k_tiles;
    r.P = (int)(r.T < (long long)g.n_cta ? r.T : (long long)g.n_cta);
    if (c >= r.P) { r.u0 = r.u1 = 0; return r; }
    r.u0 = r.T * c / r.P;
    r.u1 = r.T * (c + 1) / r.P;
    return r;
}
__device__ __forceinline__ int atoms_of(const MgGemm& g, long long u) {
    return min(g.ua, g.k_atoms - (int)(u % g.k_tiles) * g.ua);
}
__device__ __forceinline__ int rows_for(int sel, int Q, int n_need) { return sel == SEL_NEED ? n_need : Q; }

// TMEM accumulator slots: columns [0, 256) and [256, 512), each with a
// full (MMA commit) and an empty (epilogue drained) barrier.  A segment whose
// accumulator fits 256 columns takes the next slot in turn; a wider one (the
// gate/up pair above 128 rows) takes both, with slot 0 as its primary.  The
// MMA warp and the epilogue walk the same segments and so the same slot
// sequence: `uses` counts the uses of each slot (one epilogue arrival on its
// empty barrier each), `fills` the segments whose primary it is (one MMA
// commit on its full barrier each).
struct AccUse {
    int primary, mask, fill;      // primary slot, slots used (bit mask), commits on the primary before this one
};
struct AccSlots {
    int next = 0, uses[2] = {0, 0}, fills[2] = {0, 0};
    __device__ __forceinline__ AccUse take(bool wide) {
        AccUse a;
        if (wide) {
            a.primary = 0;
            a.mask = 3;
        } else {
            a.primary = next;
            a.mask = 1 << next;
            next ^= 1;
        }
        a.fill = fills[a.primary]++;
        for (int q = 0; q < 2; ++q)
            if ((a.mask >> q) & 1) ++uses[q];
        return a;
    }
};

// bounded acquire wait until the phase counter reaches `target`
__device__ __forceinline__ bool wait_count(const unsigned long long* c, unsigned long long target) {
    for (uint32_t i = 0; i < LA_SPIN_LIMIT; ++i) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(c) : "memory");
        if (v >= target) return true;
        __nanosleep(64);
    }
    return false;
}
__device__ __forceinline__ void arrive_count(unsigned long long* c) {
    __threadfence();
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(c) : "memory");
}

__global__ void __launch_bounds__(MG_THREADS, 1) k_mega(const __grid_constant__ MgParams p) {
    LaTl la_tl_(LA_TL_CHAIN, p.tl);
    LaHdr* h = p.hdr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, NC = gridDim.x;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t bar_full = base;                                   // MG_MAX_STAGES x 8 B
    const uint32_t bar_empty = base + 8 * MG_MAX_STAGES;
    const uint32_t bar_accf = base + 16 * MG_MAX_STAGES;              // 2 x 8 B
    const uint32_t bar_acce = bar_accf + 16;
    volatile int* flags = reinterpret_cast<volatile int*>(gbase + 256);
    // flags[0] tmem base, [1] Q, [2] n_need, [3] skip, [4] items issued before the header,
    // [5] epilogue / [7] row-phase / [8..13] loader-warp wait results
    float* red = reinterpret_cast<float*>(gbase + 512);               // [32] + total at [32]
    float* rv = reinterpret_cast<float*>(gbase + 1024);               // [4][BN_MAX] argmax values
    int* ri = reinterpret_cast<int*>(gbase + 1024 + 4 * BN_MAX * 4);  // [4][BN_MAX] argmax ids
    const uint32_t wring = base + MG_SCRATCH;
    const uint32_t ring_end = base + MG_SMEM;

    // ---- item sequence: (GEMM phase, unit) in phase order ----------------------
    // Every role walks it in the same order; item `it` uses ring stage it % ns
    // in round it / ns.
    auto load_w = [&](uint32_t stage_addr, uint32_t full, const MgGemm& g, long long u, uint64_t pol) {
        const int tile = (int)(u / g.k_tiles), at0 = (int)(u % g.k_tiles) * g.ua, na = atoms_of(g, u);
        bulk_load(stage_addr, g.wpack + ((size_t)tile * g.k_atoms + at0) * g.nA * A_BYTES,
                  (uint32_t)(na * g.nA) * A_BYTES, full, pol);
    };

    la_pdl_trigger();
    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < MG_MAX_STAGES; ++s) {
                mbar_init(bar_full + 8 * s, 1 + 6);    // the weight copy (with its bytes), each loader warp
                mbar_init(bar_empty + 8 * s, 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(bar_accf + 8 * b, 1);
                mbar_init(bar_acce + 8 * b, 1);
            }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            uint64_t pol_w;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
            // the first ns_pre items' weights: they depend on no earlier kernel
            int it = 0;
            for (int ph = 0; ph < p.n_ph && it < p.ns_pre; ++ph) {
                if (p.ph_kind[ph] != MG_PH_GEMM) continue;
                const MgGemm& g = p.g[p.ph_idx[ph]];
                const Units U = units_of(g, c);
                for (long long u = U.u0; u < U.u1 && it < p.ns_pre; ++u, ++it) {
                    const uint32_t wb = (uint32_t)(atoms_of(g, u) * g.nA) * A_BYTES;
                    mbar_expect_tx(bar_full + 8 * it, wb);
                    load_w(wring + (uint32_t)it * MG_A_STAGE, bar_full + 8 * it, g, u, pol_w);
                }
            }
            flags[4] = it;            // items issued before the header (read back below)
            // header fields written at least three launches back (la_common.cuh)
            const int Q = h->Q, n_need = h->n_need;
            int skip = (h->err != 0 || h->done != 0) ? 1 : 0;
            if (!skip && (Q < 1 || Q > p.rows_cap || n_need > Q)) {
                if (c == 0) la_set_err(h, LA_EDEVICE);
                skip = 1;
            }
            flags[1] = Q;
            flags[2] = n_need;
            flags[3] = skip;
        }
    } else if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + 256),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else {
        // warps 2..11 read what the kernel before this one wrote (activations,
        // and, for the first GEMM's partial stores, its reads must be over)
        la_pdl_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = (uint32_t)flags[0];
    const int Q = flags[1], n_need = flags[2], skip = flags[3], n_pre = flags[4];
    const int BNmax = (min(max(Q, 1), MG_MAX_ROWS_PER_CALL) + 15) & ~15;
    const uint32_t b_atom = (uint32_t)BNmax * ROW_BYTES, b_stage = 2u * b_atom;
    const int ns = min(MG_MAX_STAGES, (int)((MG_SMEM - MG_SCRATCH) / (MG_A_STAGE + b_stage)));
    unsigned long long* bar = p.bar;

    if (warp == 0) {
        // ---- weight producer ----------------------------------------------------
        if (lane == 0) {
            if (skip) {
                // let the weight copies already issued land before exiting (the
                // loader threads add their arrivals below)
                for (int i = 0; i < n_pre; ++i) mbar_wait(bar_full + 8 * i, 0);
            } else {
                uint64_t pol_w;
                asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
                bool ok = true;
                int it = 0;
                for (int ph = 0; ph < p.n_ph && ok; ++ph) {
                    if (p.ph_kind[ph] != MG_PH_GEMM) continue;
                    const MgGemm& g = p.g[p.ph_idx[ph]];
                    const Units U = units_of(g, c);
                    for (long long u = U.u0; u < U.u1; ++u, ++it) {
                        if (it < n_pre) continue;                      // issued before the header
                        const int s = it % ns, r = it / ns;
                        if (r > 0 && !mbar_wait(bar_empty + 8 * s, (uint32_t)((r - 1) & 1))) { ok = false; break; }
                        mbar_expect_tx(bar_full + 8 * s, (uint32_t)(atoms_of(g, u) * g.nA) * A_BYTES);
                        load_w(wring + (uint32_t)s * MG_A_STAGE, bar_full + 8 * s, g, u, pol_w);
                    }
                }
                if (!ok) la_set_err(h, LA_ETIMEOUT);
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer ------------------------------------------------------------
        if (lane == 0 && !skip) {
            bool ok = true;
            int it = 0;
            AccSlots sl;
            for (int ph = 0; ph < p.n_ph && ok; ++ph) {
                if (p.ph_kind[ph] != MG_PH_GEMM) continue;
                const MgGemm& g = p.g[p.ph_idx[ph]];
                const Units U = units_of(g, c);
                const int BN = (rows_for(g.sel, Q, n_need) + 15) & ~15;
                const uint32_t id = idesc_bf16(BN);
                const bool swiglu = g.nA == 2;
                const bool wide = g.nA * BN > 256;
                long long u = U.u0;
                while (u < U.u1 && ok) {
                    const int kt = (int)(u % g.k_tiles);
                    const int seg_len = (int)min(U.u1 - u, (long long)(g.k_tiles - kt));
                    const AccUse au = sl.take(wide);
                    // the slots' previous contents must have been drained
                    for (int q = 0; q < 2 && ok; ++q)
                        if ((au.mask >> q) & 1) {
                            const int prior = sl.uses[q] - 1;        // uses before this one
                            if (prior > 0 && !mbar_wait(bar_acce + 8 * q, (uint32_t)((prior - 1) & 1))) ok = false;
                        }
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t acc = tmem + (uint32_t)(au.primary * 256);
                    for (int j = 0; j < seg_len; ++j, ++it) {
                        const int s = it % ns, r = it / ns;
                        if (!mbar_wait(bar_full + 8 * s, (uint32_t)(r & 1))) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t st = wring + (uint32_t)s * MG_A_STAGE;
                        const uint32_t bst = ring_end - (uint32_t)(s + 1) * b_stage;
                        const int na = atoms_of(g, u + j);
                        for (int i = 0; i < na; ++i) {
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk) {
                                const uint64_t bdesc = sdesc(bst + (uint32_t)i * b_atom + kk * 32);
                                const uint32_t accum = (j == 0 && i == 0 && kk == 0) ? 0u : 1u;
                                const uint32_t sa = st + (uint32_t)(i * g.nA) * A_BYTES + kk * 32;
                                mma_bf16(acc, sdesc(sa), bdesc, id, accum);
                                if (swiglu) mma_bf16(acc + (uint32_t)BN, sdesc(sa + A_BYTES), bdesc, id, accum);
                            }
                        }
                        mma_commit(bar_empty + 8 * s);
                    }
                    if (!ok) break;
                    mma_commit(bar_accf + 8 * au.primary);
                    u += seg_len;
                }
            }
            if (!ok) la_set_err(h, LA_ETIMEOUT);
        }
    } else if (skip) {
        if (warp >= 6 && lane == 0)
            for (int i = 0; i < n_pre; ++i) mbar_arrive(bar_full + 8 * i);
    } else {
        // ---- warps 2..11: epilogue (2-5) / activation loads (6-11), row phases (all)
        const int wt = tid - 64;                     // worker index 0..319
        const bool epi = warp < 6;
        bool alive = true;
        int it = 0;
        AccSlots sl;
        for (int ph = 0; ph < p.n_ph; ++ph) {
            // inputs of phase ph: every CTA's part of phase ph - 1
            const unsigned long long target = (unsigned long long)NC;
            unsigned long long* const prev = bar + (ph > 0 ? ph - 1 : 0);
            if (p.ph_kind[ph] == MG_PH_GEMM) {
                const MgGemm& g = p.g[p.ph_idx[ph]];
                const Units U = units_of(g, c);
                const int rows = rows_for(g.sel, Q, n_need);
                const int BN = (rows + 15) & ~15;
                if (!epi) {
                    // ---- activation rows of every unit, once the inputs are complete.
                    // Warps 6-11, each on every sixth group of four rows: cp.async
                    // (L2 only) into the stage's swizzled layout, up to D units in
                    // flight; once the warp's copies of a unit have landed it fences
                    // them for the tensor core (async proxy) and its lane 0 arrives
                    // on the stage's full barrier.
                    const int lw = warp - 6;             // loader warp 0..5
                    if (ph > 0) {
                        if (lane == 0) flags[8 + lw] = alive && wait_count(prev, target);
                        __syncwarp();
                        const bool ok = flags[8 + lw] != 0;
                        if (alive && !ok && lane == 0) la_set_err(h, LA_ETIMEOUT);
                        alive = alive && ok;
                        __syncwarp();
                    }
                    const int D = ns > 2 ? 2 : 1;        // units in flight beyond the one completing (< ns)
                    const int rsub = lane >> 3, cc = lane & 7;
                    int done = it;                       // first item not yet arrived on
                    for (long long u = U.u0; u < U.u1; ++u, ++it) {
                        const int s = it % ns, r = it / ns;
                        if (r > 0) {
                            bool ok = true;
                            if (lane == 0 && alive) ok = mbar_wait(bar_empty + 8 * s, (uint32_t)((r - 1) & 1));
                            ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
                            if (!ok && alive) {
                                alive = false;
                                if (lane == 0) la_set_err(h, LA_ETIMEOUT);
                            }
                        }
                        if (alive) {
                            const uint32_t bst = ring_end - (uint32_t)(s + 1) * b_stage;
                            const int at0 = (int)(u % g.k_tiles) * g.ua, na = atoms_of(g, u);
                            // 16-byte chunk cc of row q of atom i lands where a 128-byte
                            // swizzled TMA box would put it: q * 128 + ((cc ^ (q & 7)) * 16)
                            for (int i = 0; i < na; ++i) {
                                const __nv_bfloat16* src0 = g.act + (size_t)(at0 + i) * BK + cc * 8;
                                const uint32_t dst0 = bst + (uint32_t)i * b_atom;
                                for (int q = lw * 4 + rsub; q < BN; q += 24) {
                                    const uint32_t dst = dst0 + (uint32_t)q * 128u + (uint32_t)((cc ^ (q & 7)) * 16);
                                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                                                 "l"(src0 + (size_t)q * g.K)
                                                 : "memory");
                                }
                            }
                        }
                        asm volatile("cp.async.commit_group;" ::: "memory");
                        if (it - done + 1 > D) {
                            if (D == 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
                            else asm volatile("cp.async.wait_group 1;" ::: "memory");
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bar_full + 8 * (done % ns));
                            ++done;
                        }
                    }
                    asm volatile("cp.async.wait_group 0;" ::: "memory");
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    for (; done < it; ++done)
                        if (lane == 0) mbar_arrive(bar_full + 8 * (done % ns));
                } else {
                    // ---- epilogue: TMEM -> partial records / outputs
                    const int quarter = warp & 3;
                    const int et = quarter * 32 + lane;  // weight row within the tile
                    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
                    const size_t plane = (size_t)BN_MAX * BM;
                    const bool swiglu = g.nA == 2;
                    const bool wide = g.nA * BN > 256;
                    const int nA = g.nA;
                    auto emit_group = [&](int tile, int cb, int ncol, const float (&v)[16], const float (&w2)[16],
                                          bool ok) {
                        const int n = tile * BM + et;
                        if (g.mode == GEMM_STORE) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (ok && j < ncol)
                                    ((__nv_bfloat16*)g.out)[(size_t)(cb + j) * g.ldo + n] = __float2bfloat16_rn(v[j]);
                        } else if (g.mode == GEMM_RESID) {
                            float old[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                old[j] = __ldcg((const float*)g.out + (size_t)(cb + min(j, ncol - 1)) * g.ldo + n);
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (ok && j < ncol) ((float*)g.out)[(size_t)(cb + j) * g.ldo + n] = old[j] + v[j];
                        } else if (g.mode == GEMM_SWIGLU) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (ok && j < ncol)
                                    ((__nv_bfloat16*)g.out)[(size_t)(cb + j) * g.ldo + n] =
                                        __float2bfloat16_rn(v[j] / (1.0f + expf(-v[j])) * w2[j]);
                        } else {
                            if (ok && g.logits) {
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    if (j < ncol) g.logits[(size_t)(cb + j) * g.ld_logits + n] = v[j];
                            }
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
                                    if (vv > bv[j] || (vv == bv[j] && ii < bi[j])) { bv[j] = vv; bi[j] = ii; }
                                }
                            }
                            if (lane == 0) {
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    if (j < ncol) { rv[quarter * BN_MAX + cb + j] = bv[j]; ri[quarter * BN_MAX + cb + j] = bi[j]; }
                            }
                        }
                    };
                    auto argmax_out = [&](int tile, int c_lo, int c_hi, bool ok) {
                        if (g.mode != GEMM_LOGITS) return;
                        named_sync(BAR_EPI, 128);
                        for (int cc = c_lo + et; cc < c_hi; cc += 128) {
                            float bv = rv[cc];
                            int bi = ri[cc];
                            for (int w = 1; w < 4; ++w) {
                                const float v2 = rv[w * BN_MAX + cc];
                                const int i2 = ri[w * BN_MAX + cc];
                                if (v2 > bv || (v2 == bv && i2 < bi)) { bv = v2; bi = i2; }
                            }
                            if (ok) {
                                g.part_v[(size_t)tile * g.part_stride + cc] = bv;
                                g.part_i[(size_t)tile * g.part_stride + cc] = bi;
                            }
                        }
                        named_sync(BAR_EPI, 128);
                    };
                    int d_tile[2], d_sg[2], d_nseg[2];
                    unsigned long long d_target[2];
                    int nd = 0;
                    long long u = U.u0;
                    while (u < U.u1) {
                        const int tile = (int)(u / g.k_tiles), kt = (int)(u % g.k_tiles);
                        const int seg_len = (int)min(U.u1 - u, (long long)(g.k_tiles - kt));
                        const AccUse au = sl.take(wide);
                        const bool got = alive && mbar_wait(bar_accf + 8 * au.primary, (uint32_t)(au.fill & 1));
                        if (!got && alive) { alive = false; la_set_err(h, LA_ETIMEOUT); }
                        tc_fence_after();
                        const uint32_t acc = tmem + lane_base + (uint32_t)(au.primary * 256);
                        // drained: free every slot this segment used
                        auto release = [&]() {
                            if (quarter == 0 && lane == 0)
                                for (int q = 0; q < 2; ++q)
                                    if ((au.mask >> q) & 1) mbar_arrive(bar_acce + 8 * q);
                        };
                        const long long tile_u0 = (long long)tile * g.k_tiles, tile_u1 = tile_u0 + g.k_tiles;
                        const int c_first = (int)(((tile_u0 + 1) * U.P - 1) / U.T);
                        const int c_last = (int)(((tile_u1 - 1 + 1) * U.P - 1) / U.T);
                        const int nseg = c_last - c_first + 1;
                        if (nseg > 1) {
                            const int sg = c - c_first;
                            float* wsb = g.ws + (((size_t)tile * g.max_seg + sg) * nA) * plane;
                            for (int c0 = 0; c0 < rows; c0 += 16) {
                                float v[16];
                                tmem_ld16(acc + c0, v);
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    if (c0 + j < rows) __stcg(wsb + (size_t)(c0 + j) * BM + et, got ? v[j] : 0.f);
                                if (swiglu) {
                                    tmem_ld16(acc + BN + c0, v);
#pragma unroll
                                    for (int j = 0; j < 16; ++j)
                                        if (c0 + j < rows) __stcg(wsb + plane + (size_t)(c0 + j) * BM + et, got ? v[j] : 0.f);
                                }
                            }
                            tc_fence_before();
                            named_sync(BAR_EPI, 128);
                            release();
                            if (quarter == 0 && lane == 0) {
                                if (!g.defer) {
                                    unsigned long long old;
                                    asm volatile("atom.add.release.gpu.global.u64 %0, [%1], 1;"
                                                 : "=l"(old)
                                                 : "l"(g.ctr + tile)
                                                 : "memory");
                                    d_target[nd] = (old / (unsigned long long)nseg + 1ull) * (unsigned long long)nseg;
                                }
                            }
                            if (!g.defer) {
                                d_tile[nd] = tile; d_sg[nd] = sg; d_nseg[nd] = nseg;
                                ++nd;
                            }
                        } else {
                            for (int c0 = 0; c0 < rows; c0 += 16) {
                                float v[16], w2[16];
                                tmem_ld16(acc + c0, v);
                                if (swiglu) tmem_ld16(acc + BN + c0, w2);
                                emit_group(tile, c0, min(16, rows - c0), v, w2, got);
                            }
                            tc_fence_before();
                            named_sync(BAR_EPI, 128);
                            release();
                            argmax_out(tile, 0, rows, got);
                        }
                        u += seg_len;
                    }
                    // split tiles of a non-deferred GEMM (the LM head): once all
                    // partials are in, contributor sg sums its share of the rows in
                    // segment (K) order
                    for (int dd = 0; dd < nd; ++dd) {
                        const int tile = d_tile[dd], sg = d_sg[dd], nseg = d_nseg[dd];
                        if (quarter == 0 && lane == 0) {
                            const bool ok = alive && spin_until64(g.ctr + tile, d_target[dd]);
                            if (!ok && alive) la_set_err(h, LA_ETIMEOUT);
                            flags[5] = ok ? 1 : 0;
                        }
                        named_sync(BAR_EPI, 128);
                        const bool ok = flags[5] != 0;
                        alive = alive && ok;
                        const int c_lo = rows * sg / nseg, c_hi = rows * (sg + 1) / nseg;
                        const float* wst = g.ws + ((size_t)tile * g.max_seg * nA) * plane + et;
                        const size_t seg_stride = (size_t)nA * plane;
                        for (int cb = c_lo; cb < c_hi; cb += 16) {
                            float v[16], w2[16];
                            if (nseg == 2) {
                                sum_segments<2, 16>(wst, seg_stride, nseg, cb, c_hi, v);
                                if (swiglu) sum_segments<2, 16>(wst + plane, seg_stride, nseg, cb, c_hi, w2);
                            } else if (nseg == 3) {
                                sum_segments<3, 16>(wst, seg_stride, nseg, cb, c_hi, v);
                                if (swiglu) sum_segments<3, 16>(wst + plane, seg_stride, nseg, cb, c_hi, w2);
                            } else {
                                sum_segments<4, 16>(wst, seg_stride, nseg, cb, c_hi, v);
                                if (swiglu) sum_segments<4, 16>(wst + plane, seg_stride, nseg, cb, c_hi, w2);
                            }
                            emit_group(tile, cb, min(16, c_hi - cb), v, w2, ok);
                        }
                        argmax_out(tile, c_lo, c_hi, ok);
                        named_sync(BAR_EPI, 128);
                    }
                    // this CTA's part of the phase is in memory
                    named_sync(BAR_EPI, 128);
                    if (warp == 2 && lane == 0) arrive_count(bar + ph);
                }
            } else {
                // ---- row phase (all 320 workers) --------------------------------------
                const MgRows& R = p.r[p.ph_idx[ph]];
                if (ph > 0) {
                    if (wt == 0) flags[7] = alive && wait_count(prev, target);
                    named_sync(BAR_WORK, N_WORKERS);
                    if (alive && !flags[7] && wt == 0) la_set_err(h, LA_ETIMEOUT);
                    alive = alive && flags[7];
                    named_sync(BAR_WORK, N_WORKERS);
                }
                const int rows = rows_for(R.sel, Q, n_need);
                if (alive && R.kind == MG_SWIGLU) {
                    // k_swiglu_split's arithmetic per four consecutive columns
                    const int n_cols = R.split.n_tiles * 128;
                    const long long items = (long long)rows * (n_cols / 4);
                    for (long long i = (long long)c * N_WORKERS + wt; i < items; i += (long long)NC * N_WORKERS) {
                        const int q = (int)(i / (n_cols / 4)), c4 = (int)(i % (n_cols / 4)) * 4;
                        const int tile = c4 >> 7;
                        const int nseg = la_split_nseg(R.split, tile);
                        if (nseg <= 1) continue;
                        const size_t off = (size_t)(q & 255) * 128 + (c4 & 127);
                        const float4 v = la_split_sum4(R.split, tile, q >> 8, off, nseg, 0);
                        const float4 uu = la_split_sum4(R.split, tile, q >> 8, off, nseg, 1);
                        __nv_bfloat162 r01 = __floats2bfloat162_rn(v.x / (1.0f + expf(-v.x)) * uu.x,
                                                                   v.y / (1.0f + expf(-v.y)) * uu.y);
                        __nv_bfloat162 r23 = __floats2bfloat162_rn(v.z / (1.0f + expf(-v.z)) * uu.z,
                                                                   v.w / (1.0f + expf(-v.w)) * uu.w);
                        uint2 pk;
                        pk.x = *reinterpret_cast<uint32_t*>(&r01);
                        pk.y = *reinterpret_cast<uint32_t*>(&r23);
                        *reinterpret_cast<uint2*>(R.y + (size_t)q * R.ldo + c4) = pk;
                    }
                } else if (alive) {
                    // k_rmsnorm's arithmetic: VT virtual threads (1024 above 2048
                    // columns, else 256), one float4 per virtual thread and pass k,
                    // fmaf chain, butterfly per virtual warp, butterfly over warps
                    const int dm = R.dm;
                    const int VT = dm > 2048 ? 1024 : 256, VW = VT / 32;
                    const int ww = wt >> 5;                    // worker warp 0..9
                    for (int row = c; row < rows; row += NC) {
                        const int src = R.kind == MG_RMS_GATHER ? p.need[row] : row;
                        float* xr = R.x + (size_t)src * dm;
                        // every load of the row and its split partials is issued before
                        // the first sum (k_rmsnorm's order per virtual thread is kept)
                        float4 vv[4][2], add[4][2];
                        bool upd[4][2];
#pragma unroll
                        for (int jv = 0; jv < 4; ++jv) {
                            const int vw = ww + 10 * jv;
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                const int i = (k * VT + vw * 32 + lane) * 4;
                                upd[jv][k] = false;
                                if (vw < VW && i < dm) {
                                    vv[jv][k] = __ldcg(reinterpret_cast<const float4*>(xr + i));
                                    if (R.split.ws) {
                                        const int tile = i >> 7;
                                        const int nseg = la_split_nseg(R.split, tile);
                                        if (nseg > 1) {
                                            add[jv][k] = la_split_sum4(R.split, tile, src >> 8,
                                                                       (size_t)(src & 255) * 128 + (i & 127), nseg);
                                            upd[jv][k] = true;
                                        }
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int jv = 0; jv < 4; ++jv) {
                            const int vw = ww + 10 * jv;
                            if (vw >= VW) continue;
                            float ss = 0.f;
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                const int i = (k * VT + vw * 32 + lane) * 4;
                                if (i < dm) {
                                    if (upd[jv][k]) {
                                        vv[jv][k].x = vv[jv][k].x + add[jv][k].x;
                                        vv[jv][k].y = vv[jv][k].y + add[jv][k].y;
                                        vv[jv][k].z = vv[jv][k].z + add[jv][k].z;
                                        vv[jv][k].w = vv[jv][k].w + add[jv][k].w;
                                        *reinterpret_cast<float4*>(xr + i) = vv[jv][k];
                                    }
                                    ss = fmaf(vv[jv][k].x, vv[jv][k].x, ss);
                                    ss = fmaf(vv[jv][k].y, vv[jv][k].y, ss);
                                    ss = fmaf(vv[jv][k].z, vv[jv][k].z, ss);
                                    ss = fmaf(vv[jv][k].w, vv[jv][k].w, ss);
                                }
                            }
                            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                            if (lane == 0) red[vw] = ss;
                        }
                        named_sync(BAR_WORK, N_WORKERS);
                        if (ww == 0) {
                            float t = (lane < VW) ? red[lane] : 0.f;
                            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                            if (lane == 0) red[32] = t;
                        }
                        named_sync(BAR_WORK, N_WORKERS);
                        const float rs = 1.0f / sqrtf(red[32] / (float)dm + R.eps);
                        __nv_bfloat16* yr = R.y + (size_t)row * dm;
#pragma unroll
                        for (int jv = 0; jv < 4; ++jv) {
                            const int vw = ww + 10 * jv;
                            if (vw >= VW) continue;
                            const int vt = vw * 32 + lane;
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                const int i = (k * VT + vt) * 4;
                                if (i < dm) {
                                    const uint2 gr = *reinterpret_cast<const uint2*>(R.g + i);
                                    const float g0 = __uint_as_float(gr.x << 16), g1 = __uint_as_float(gr.x & 0xffff0000u);
                                    const float g2 = __uint_as_float(gr.y << 16), g3 = __uint_as_float(gr.y & 0xffff0000u);
                                    yr[i + 0] = __float2bfloat16_rn(vv[jv][k].x * rs * g0);
                                    yr[i + 1] = __float2bfloat16_rn(vv[jv][k].y * rs * g1);
                                    yr[i + 2] = __float2bfloat16_rn(vv[jv][k].z * rs * g2);
                                    yr[i + 3] = __float2bfloat16_rn(vv[jv][k].w * rs * g3);
                                }
                            }
                        }
                        // red[] is rewritten by the next row only after every worker read it
                        named_sync(BAR_WORK, N_WORKERS);
                    }
                }
                named_sync(BAR_WORK, N_WORKERS);
                if (wt == 0) arrive_count(bar + ph);
            }
        }
    }
    // teardown: every warp reconverges before the CTA-wide barrier that frees TMEM
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

}  // namespace

int la_mega_ring_stages(int rows) {
    const int bn = (std::min(std::max(rows, 1), MG_MAX_ROWS_PER_CALL) + 15) & ~15;
    return std::min(MG_MAX_STAGES, (MG_SMEM - MG_SCRATCH) / (MG_A_STAGE + 2 * bn * ROW_BYTES));
}

cudaError_t la_launch_mega(const MgParams& p, cudaStream_t st) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_mega, cudaFuncAttributeMaxDynamicSharedMemorySize, MG_SMEM + 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    if (p.rows_cap < 1 || p.rows_cap > MG_MAX_ROWS_PER_CALL || p.n_ph < 1 || p.n_ph > MG_MAX_PHASES)
        return cudaErrorInvalidValue;
    for (int i = 0; i < p.n_ph; ++i)
        if (p.ph_kind[i] == MG_PH_GEMM && p.g[p.ph_idx[i]].n_cta > la_tc_ctas()) return cudaErrorInvalidValue;
    return la_launch_pdl(k_mega, dim3(la_tc_ctas()), dim3(MG_THREADS), (size_t)(MG_SMEM + 1024), st, p);
}
