// Exact sampling verification of the packed call (one CTA per call).
//
// Target distribution (break the sequential dependency §2: greedy, top-K and
// top-P selectors; temperature and top-p shape p before verification):
//   p = softmax(logits / T), restricted to the top-p nucleus — probability
//   descending, ties by lower id, the shortest prefix whose mass reaches
//   top_p (crossing token kept) — and renormalised.
// Verifier (M7.3 §0x05B, disjoint one-hot proposals):
//   at each suffix offset, test the distinct tokens offered by the surviving
//   candidates in candidate order; accept token c with probability
//   residual(c) = p(c) / (1 - removed mass); on rejection remove its mass
//   once; if all are rejected, draw from the residual by inverse CDF in id
//   order and stop; after an acceptance keep the candidates carrying that
//   token and read the next distribution from the lowest-index survivor's
//   row; after S acceptances draw the bonus token from the last survivor row.
// Uniforms: Philox4x32-10 (Salmon et al., SC'11) with key (seed lo, seed hi)
// and counter (step, offset, test, purpose); word 0 >> 8 times 2^-24.
#include "la_common.cuh"
#include "la_kernels.h"

#include <math.h>

namespace {

constexpr int NT = 1024;
constexpr int NW = NT / 32;
constexpr uint32_t PURPOSE_ACCEPT = 0, PURPOSE_RESIDUAL = 1, PURPOSE_PLAIN = 2;

__device__ __forceinline__ float philox_uniform(uint32_t k0, uint32_t k1, uint32_t c0, uint32_t c1, uint32_t c2,
                                                uint32_t c3) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) { k0 += W0; k1 += W1; }
        const uint32_t hi0 = __umulhi(M0, c0), lo0 = M0 * c0;
        const uint32_t hi1 = __umulhi(M1, c2), lo1 = M1 * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    return (float)(c0 >> 8) * (1.0f / 16777216.0f);
}

// The distribution lives in shared memory in the blocked id layout (thread
// t owns ids [t per, (t + 1) per)), each thread's run starting at t * pstride
// with pstride odd: a warp's 32 threads stepping through their runs touch 32
// different banks (runs at t * per for even per hit one bank 32 times).
__host__ __device__ __forceinline__ int p_per(int V) { return (V + NT - 1) / NT; }
__host__ __device__ __forceinline__ int p_stride(int V) { return p_per(V) | 1; }
__device__ __forceinline__ int pidx(int i, int V) {
    const int per = p_per(V), q = i / per;
    return q * p_stride(V) + (i - q * per);
}

struct Red {
    float f[NW];
    int i[NW];
    float bcast_f;
    int bcast_i;
    float f2[2][NW];      // the one-barrier sums of a loop, alternating by iteration
};

__device__ float block_sum(float v, Red& r) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) r.f[w] = v;
    __syncthreads();
    if (w == 0) {
        float x = r.f[l];
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (l == 0) r.bcast_f = x;
    }
    __syncthreads();
    return r.bcast_f;
}
// The same sum as block_sum with one barrier: every warp adds the 32 warp
// partials in the same shuffle tree.  Consecutive calls must alternate ph (a
// warp cannot rewrite a slot until every warp has passed the next call's
// barrier, i.e. finished reading it).
__device__ float block_sum_1(float v, Red& r, int ph) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) r.f2[ph][w] = v;
    __syncthreads();
    float x = r.f2[ph][l];
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ float block_max(float v, Red& r) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) r.f[w] = v;
    __syncthreads();
    if (w == 0) {
        float x = r.f[l];
        for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        if (l == 0) r.bcast_f = x;
    }
    __syncthreads();
    return r.bcast_f;
}
__device__ int block_sum_i(int v, Red& r) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) r.i[w] = v;
    __syncthreads();
    if (w == 0) {
        int x = r.i[l];
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (l == 0) r.bcast_i = x;
    }
    __syncthreads();
    return r.bcast_i;
}
// exclusive prefix over threads (thread order = id order in the blocked layout)
__device__ float block_excl_scan(float v, Red& r, float* total) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    float x = v;
    for (int o = 1; o < 32; o <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, x, o);
        if (l >= o) x += y;
    }
    __syncthreads();
    if (l == 31) r.f[w] = x;
    __syncthreads();
    if (w == 0) {
        float t = r.f[l];
        for (int o = 1; o < 32; o <<= 1) {
            float y = __shfl_up_sync(0xffffffffu, t, o);
            if (l >= o) t += y;
        }
        r.f[l] = t;   // inclusive over warps
    }
    __syncthreads();
    const float before_warp = (w == 0) ? 0.f : r.f[w - 1];
    *total = r.f[NW - 1];
    const float res = before_warp + x - v;
    __syncthreads();
    return res;
}

// p[] <- nucleus-restricted softmax(logits / T), normalised (blocked id layout)
__device__ void warp_distribution(const float* logits, float* pall, int V, float T, float top_p, Red& r) {
    const int per = p_per(V);
    const int i0 = threadIdx.x * per, i1 = min(V, i0 + per);
    float* p = pall + threadIdx.x * p_stride(V) - i0;   // p[i] for this thread's ids
    // logits / T staged by coalesced reads (a thread's run of ids would
    // touch 32 lines a warp instruction, and the runs outgrow L1)
    for (int i = threadIdx.x; i < V; i += NT) pall[pidx(i, V)] = logits[i] / T;
    __syncthreads();
    float m = -INFINITY;
    for (int i = i0; i < i1; ++i) m = fmaxf(m, p[i]);
    m = block_max(m, r);
    float s = 0.f;
    for (int i = i0; i < i1; ++i) {
        const float e = expf(p[i] - m);
        p[i] = e;
        s += e;
    }
    const float Z = block_sum(s, r);
    float pmax = 0.f;
    for (int i = i0; i < i1; ++i) {
        p[i] = p[i] / Z;
        pmax = fmaxf(pmax, p[i]);
    }
    if (!(top_p < 1.0f)) return;
    pmax = block_max(pmax, r);
    // largest threshold tau (a float bit pattern) whose mass at-or-above reaches top_p
    uint32_t lo = 0u, hi = __float_as_uint(pmax) + 1u;
    int ph = 0;
    while (hi - lo > 1u) {
        const uint32_t mid = lo + ((hi - lo) >> 1);
        const float b = __uint_as_float(mid);
        float g = 0.f;
        for (int i = i0; i < i1; ++i)
            if (p[i] >= b) g += p[i];
        if (block_sum_1(g, r, ph) >= top_p) lo = mid;
        else hi = mid;
        ph ^= 1;
    }
    const float tau = __uint_as_float(lo);
    float a = 0.f;
    int nt = 0;
    for (int i = i0; i < i1; ++i) {
        if (p[i] > tau) a += p[i];
        else if (p[i] == tau) ++nt;
    }
    const float A = block_sum(a, r);
    const int n_ties = block_sum_i(nt, r);
    // ties at tau are kept in id order until the mass reaches top_p
    __shared__ int s_keep_ties;
    if (threadIdx.x == 0) {
        float acc = A;
        int j = 0;
        while (acc < top_p && j < n_ties) { acc += tau; ++j; }
        s_keep_ties = j;
    }
    __syncthreads();
    const int keep_ties = s_keep_ties;
    // rank of this thread's first tie among all ties (exclusive scan of counts)
    float tot;
    const int tie_rank0 = (int)block_excl_scan((float)nt, r, &tot);
    int rank = tie_rank0;
    float kept = 0.f;
    for (int i = i0; i < i1; ++i) {
        bool keep = p[i] > tau;
        if (p[i] == tau) keep = (rank++ < keep_ties);
        if (!keep) p[i] = 0.f;
        kept += p[i];
    }
    const float Zk = block_sum(kept, r);
    for (int i = i0; i < i1; ++i) p[i] = p[i] / Zk;
    __syncthreads();
}

// inverse CDF in id order: the first id whose cumulative mass exceeds u * total
__device__ int draw_index(const float* pall, int V, float u, Red& r) {
    const int per = p_per(V);
    const int i0 = threadIdx.x * per, i1 = min(V, i0 + per);
    const float* p = pall + threadIdx.x * p_stride(V) - i0;
    float s = 0.f;
    int last_nz = -1;
    for (int i = i0; i < i1; ++i) {
        s += p[i];
        if (p[i] > 0.f) last_nz = i;
    }
    float total;
    const float before = block_excl_scan(s, r, &total);
    const float target = u * total;
    __shared__ int s_pick, s_last;
    if (threadIdx.x == 0) { s_pick = 0x7fffffff; s_last = -1; }
    __syncthreads();
    atomicMax(&s_last, last_nz);
    float acc = before;
    for (int i = i0; i < i1; ++i) {
        acc += p[i];
        if (acc > target && p[i] > 0.f) { atomicMin(&s_pick, i); break; }
    }
    __syncthreads();
    int pick = s_pick;
    if (pick == 0x7fffffff) pick = s_last;   // rounding left the target above the total
    __syncthreads();
    return pick;
}

// Inputs of one verification: the needed-row logits ([rows][V], row 0 = the
// ordinary row, candidate c's offset s at row 1 + n_deep + c*S + s) and the
// candidates' tokens (cand[c*S + s]).
struct SvIn {
    const float* logits;
    int V;
    const int32_t* cand;
    int Ct, S, n_deep;
    uint32_t step, k0, k1;
    float T, top_p;
};
struct SvOut {
    int emitted[16];
    int E, a, w;
};

// One verification by the whole CTA; the result is valid in thread 0.
__device__ void sample_verify_core(const SvIn& in, float* p, Red& r, SvOut& o) {
    __shared__ int s_acc, s_row, s_tested[LA_MAX_G], s_ntested;
    __shared__ float s_removed;
    __shared__ unsigned s_surv;
    const int Ct = in.Ct, S = in.S, V = in.V;
    if (threadIdx.x == 0) {
        s_surv = Ct >= 32 ? 0xffffffffu : ((1u << Ct) - 1u);
        s_row = 0;
        o.E = 0; o.a = 0; o.w = -1;
    }
    __syncthreads();
    const int last_off = Ct > 0 ? S : 0;
    for (int off = 0; off <= last_off; ++off) {
        const int row = s_row;
        warp_distribution(in.logits + (size_t)row * V, p, V, in.T, in.top_p, r);
        if (off == last_off) {      // plain draw: no candidate is offered at this offset
            const float u = philox_uniform(in.k0, in.k1, in.step, (uint32_t)off, 0u, PURPOSE_PLAIN);
            const int tok = draw_index(p, V, u, r);
            if (threadIdx.x == 0) { o.emitted[o.E++] = tok; o.a = off; }
            break;
        }
        // sequential tests of the distinct offered tokens (one thread)
        if (threadIdx.x == 0) {
            s_ntested = 0;
            s_removed = 0.f;
            s_acc = -1;
            for (int c = 0; c < Ct && s_acc < 0; ++c) {
                if (!((s_surv >> c) & 1u)) continue;
                const int tok = in.cand[c * S + off];
                bool seen = false;
                for (int t = 0; t < s_ntested; ++t) seen |= (s_tested[t] == tok);
                if (seen) continue;
                const int t = s_ntested++;
                s_tested[t] = tok;
                const float rem = 1.0f - s_removed;
                const float u = philox_uniform(in.k0, in.k1, in.step, (uint32_t)off, (uint32_t)t, PURPOSE_ACCEPT);
                const float pt = p[pidx(tok, V)];
                if (u < pt / rem) { s_acc = tok; break; }
                s_removed += pt;
                if (!(1.0f - s_removed > 0.f)) { s_acc = tok; break; }   // all remaining mass was this token's
            }
        }
        __syncthreads();
        if (s_acc >= 0) {
            if (threadIdx.x == 0) {
                const int tok = s_acc;
                o.emitted[o.E++] = tok;
                unsigned sv = 0;
                for (int c = 0; c < Ct; ++c)
                    if (((s_surv >> c) & 1u) && in.cand[c * S + off] == tok) sv |= 1u << c;
                s_surv = sv;
                const int w = __ffs(sv) - 1;
                o.w = w;
                s_row = 1 + in.n_deep + w * S + off;
            }
            __syncthreads();
            continue;
        }
        // every offered token rejected: draw from the residual and stop
        if (threadIdx.x == 0)
            for (int t = 0; t < s_ntested; ++t) p[pidx(s_tested[t], V)] = 0.f;
        __syncthreads();
        const float u = philox_uniform(in.k0, in.k1, in.step, (uint32_t)off, 0u, PURPOSE_RESIDUAL);
        const int tok = draw_index(p, V, u, r);
        if (threadIdx.x == 0) { o.emitted[o.E++] = tok; o.a = off; }
        break;
    }
    __syncthreads();
    if (threadIdx.x == 0 && o.a == 0) o.w = -1;
}

__global__ void __launch_bounds__(NT) k_sample_verify(LaDev d, const float* logits, int V, int prefill) {
    LaTl la_tl_(LA_TL_SAMPLE_VERIFY, d.tl);
    la_pdl_wait();
    la_pdl_trigger();
    LaHdr* h = d.hdr;
    if (h->err || (!prefill && h->done)) return;
    extern __shared__ float p[];
    __shared__ Red r;
    __shared__ SvOut o;
    SvIn in;
    in.logits = logits;
    in.V = V;
    in.cand = d.row_tok + h->vstart;
    in.Ct = prefill ? 0 : h->C_t;
    in.S = h->S;
    in.n_deep = prefill ? 0 : h->n_deep;
    in.step = prefill ? 0xFFFFFFFFu : (uint32_t)h->step;
    in.k0 = h->seed_lo;
    in.k1 = h->seed_hi;
    in.T = h->temperature;
    in.top_p = h->top_p;
    sample_verify_core(in, p, r, o);
    if (threadIdx.x == 0) {
        h->a = o.a;
        h->winner = o.w;
        h->E = o.E;
        for (int i = 0; i < o.E; ++i) h->emitted[i] = o.emitted[i];
        if (prefill) d.argmax[0] = o.emitted[0];
    }
}

// Many independent verifications of the same rows and candidates, one per
// CTA, with Philox step index = trial (inspection entry point).
__global__ void __launch_bounds__(NT) k_sample_verify_trials(const float* logits, int V, const int32_t* cand, int Ct,
                                                             int S, float T, float top_p, uint32_t k0, uint32_t k1,
                                                             int n_trials, int32_t* out) {
    extern __shared__ float p[];
    __shared__ Red r;
    __shared__ SvOut o;
    for (int trial = blockIdx.x; trial < n_trials; trial += gridDim.x) {
        SvIn in{logits, V, cand, Ct, S, 0, (uint32_t)trial, k0, k1, T, top_p};
        sample_verify_core(in, p, r, o);
        if (threadIdx.x == 0) {
            int32_t* t = out + (size_t)trial * (S + 3);
            t[0] = o.E;
            t[1] = o.a;
            for (int i = 0; i <= S; ++i) t[2 + i] = i < o.E ? o.emitted[i] : -1;
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t la_launch_sample_trials(cudaStream_t st, const float* logits, int V, const int32_t* cand, int Ct, int S,
                                    float T, float top_p, uint64_t seed, int n_trials, int32_t* out) {
    const size_t smem = sizeof(float) * (size_t)NT * p_stride(V);
    cudaError_t e = cudaFuncSetAttribute(k_sample_verify_trials, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int grid = n_trials < 4096 ? n_trials : 4096;
    k_sample_verify_trials<<<grid, NT, smem, st>>>(logits, V, cand, Ct, S, T, top_p, (uint32_t)(seed & 0xffffffffu),
                                                    (uint32_t)(seed >> 32), n_trials, out);
    return cudaGetLastError();
}

cudaError_t la_launch_sample_verify(const LaDev& d, cudaStream_t st, const float* logits, int V, int prefill) {
    const size_t smem = sizeof(float) * (size_t)NT * p_stride(V);
    // the kernel's shared-memory allowance only grows: a context with a
    // larger vocabulary than the ones before raises it
    static size_t allowed = 0;
    if (smem > allowed) {
        cudaError_t e = cudaFuncSetAttribute(k_sample_verify, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        allowed = smem;
    }
    return la_launch_pdl(k_sample_verify, dim3(1), dim3(NT), smem, st, d, logits, V, prefill);
}
