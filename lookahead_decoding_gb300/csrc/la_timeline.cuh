// Per-CTA timeline of liblookahead's kernels (inspection only).
//
// When a timeline is open (la_timeline_start), thread 0 of every CTA of every
// library kernel reads the GPU's global nanosecond timer at entry and, when
// it returns, takes a record (atomic ticket) with the CTA's start and end,
// the kernel's id, the CTA's linear index and the grid's CTA count.  Every
// kernel of the library ends its CTAs with a block-wide barrier or a uniform
// return, so thread 0's return marks the CTA's end.  Grid ids
// (%gridid) repeat across launches here, so records carry no launch identity;
// the host splits the device time by which CTA is next to finish (see
// la_timeline_stop in include/lookahead.h).
//
// The table pointer travels in every kernel's parameters (LaDev::tl, or the
// GEMM's and layer chain's parameter blocks), so with no timeline open a
// kernel reads nothing but its parameters.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

// Kernel ids of the timeline (their kinds -- GEMM, attention, row-wise, state,
// layer chain -- are listed with la_timeline_start in include/lookahead.h).
enum {
    LA_TL_GEMM_TC = 0, LA_TL_GEMM_FFMA, LA_TL_ATTN_FUSED, LA_TL_ATTENTION, LA_TL_EMBED, LA_TL_RMSNORM,
    LA_TL_ROPE_KV, LA_TL_ROPE_KV4, LA_TL_SWIGLU, LA_TL_ARGMAX_ROWS, LA_TL_ARGMAX_REDUCE, LA_TL_SAMPLE_VERIFY,
    LA_TL_BEGIN, LA_TL_PACK, LA_TL_POOL_SEED, LA_TL_PUBLISH, LA_TL_COMMIT_KV, LA_TL_INJECT_MAP,
    LA_TL_PREFILL_ROWS, LA_TL_PREFILL_NEED, LA_TL_PREFILL_FINISH, LA_TL_CHAIN, LA_TL_IDS
};

// One CTA's record (32 bytes).
struct LaTlRec {
    unsigned long long start, end;
    unsigned int id, block, blocks, pad;
};

// Table layout: the first record's first two words hold the ticket counter
// and the capacity (records after the first); records follow.
struct LaTlHead {
    unsigned int count, cap;
};

__device__ __forceinline__ unsigned long long la_tl_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Declared first in a kernel body with the table pointer from the kernel's
// parameters (nullptr: no timeline; nothing is read then but the parameter).
// The destructor, which runs on every return path, takes the record.
struct LaTl {
    LaTlRec* t;
    unsigned long long start;
    unsigned int id;
    __device__ __forceinline__ LaTl(unsigned int kid, LaTlRec* tl) : t(tl), start(0), id(kid) {
        if (t != nullptr) start = la_tl_now();
    }
    __device__ __forceinline__ ~LaTl() {
        if (t == nullptr || threadIdx.x != 0 || threadIdx.y != 0 || threadIdx.z != 0) return;
        LaTlHead* hd = reinterpret_cast<LaTlHead*>(t);
        const unsigned int s = atomicAdd(&hd->count, 1u);
        if (s >= hd->cap) return;
        LaTlRec* r = t + 1 + s;
        r->start = start;
        r->end = la_tl_now();
        r->id = id;
        r->block = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        r->blocks = gridDim.x * gridDim.y * gridDim.z;
    }
};
