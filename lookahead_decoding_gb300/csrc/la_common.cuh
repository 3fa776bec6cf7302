// Shared device-side definitions of liblookahead (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda.h>
#include <stdint.h>

#include "../../include/lookahead.h"
#include "la_timeline.cuh"

#define LA_MAX_R 8            // trajectory levels: N <= 9
#define LA_MAX_G 32           // candidates per key (one warp lane each)
#define LA_MAX_W 64           // window columns
#define LA_MAX_L (LA_MAX_W + 8) // longest level: W+N-3
#define LA_HDR_STATS 16

// Roles in row metadata (M7.3 §0x04A "Row" record).
#define ROLE_ORDINARY 0
#define ROLE_LOOKAHEAD 1
#define ROLE_VERIFY 2

#define MODE_LOOKAHEAD 0
#define MODE_AR 1

// meta = role | level<<2 | column<<8 | candidate<<16 | offset<<24
__host__ __device__ __forceinline__ int32_t la_meta(int role, int level, int col, int cand, int off) {
    return (role & 3) | ((level & 63) << 2) | ((col & 255) << 8) | ((cand & 255) << 16) | ((off & 127) << 24);
}

// Per-request state that lives in device memory.  Everything a step needs to
// decide (row count, phase, verdict) is read from here by the kernels, so one
// captured graph serves every step.
struct LaHdr {
    int32_t err;            // device error word: 0 or an LA_E* code
    int32_t done;           // 1 once n_out >= max_out
    int32_t mode;           // MODE_LOOKAHEAD / MODE_AR
    int32_t sampling;       // 1 = sampling verifier
    int32_t K;              // committed K/V length == logical position of x_t
    int32_t x_t;            // ordinary input token of the next call
    int32_t W, N, G, S;     // knobs of this request (S = N-1)
    int32_t n_levels;       // materialised trajectory levels (d+1)
    int32_t level_len[LA_MAX_R];
    int32_t step;           // packed calls since the prefill (Philox step index)
    int32_t n_out, max_out; // out ring fill and cap
    int32_t prompt_len;
    // written by the pack kernel for the current call
    int32_t Q, C_t, steady, n_need, n_deep, deep_skip, vstart;
    int32_t lvl_off[LA_MAX_R + 1];
    // written by the verifier / publish kernel
    int32_t a, winner, E, commit_base, commit_n;
    int32_t emitted[16];
    // statistics since the prefill
    int32_t n_steps, n_steady;
    int64_t sum_Q, sum_Ct;
    int32_t hist[LA_HDR_STATS];
    // sampling policy
    float temperature, top_p;
    uint32_t seed_lo, seed_hi;
    int32_t prefill_rows;   // rows of the current prefill chunk
    int32_t opts;           // LA_OPT_* options of the request
    int32_t seed_next;      // next prompt index (mod prompt_len) of the refill cycle
    int32_t active;         // batch header only: requests of the batch not yet done
};

// Device pointers and sizes of one context, passed by value to kernels.
struct LaDev {
    LaHdr* hdr;
    int32_t* window;       // [Rmax][LMAX]
    int32_t* pool_tok;     // [V][Gmax][Smax]
    int32_t* pool_cnt;     // [V]
    int32_t* prompt;       // [max_ctx]
    int32_t* row_tok;      // [Qcap]
    int32_t* row_pos;      // [Qcap]
    int32_t* row_meta;     // [Qcap]
    int32_t* row_path;     // [Qcap][PMAX]: packed row of the in-call key at position K+t
    int32_t* need;         // [Qcap]: packed rows whose logits are read
    int32_t* argmax;       // [Qcap]: argmax per needed row (need order)
    int32_t* out;          // [out_cap]
    int32_t* commit_rows;  // [16]
    int32_t V, Gmax, Smax, Rmax, LMAX, PMAX, Qmax, Qcap, max_ctx, out_cap;
    // batched calls (several requests stacked in one call; all zero alone):
    // the row arrays above then point at this request's slice of the stacked
    // rows, need entries carry the slice's first stacked row, rows past the
    // request's own up to pad_to are filled as copies of its ordinary row,
    // and publication keeps the batch header's count of live requests.
    int32_t row_base;
    int32_t pad_to;
    LaHdr* batch;
    LaTlRec* tl;           // kernel timeline table (la_timeline.cuh), or nullptr
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ void la_set_err(LaHdr* h, int code) { atomicCAS(&h->err, 0, code); }

// Programmatic dependent launch.  Kernels of the step are launched so that
// each may start while its predecessor in the stream is still running; a
// kernel calls la_pdl_wait() before its first access to anything an earlier
// kernel wrote (it returns once the predecessor has completed and its writes
// are visible), and la_pdl_trigger() to let its own successor launch.  Both
// are no-ops for a kernel launched without the attribute.
//
// Every kernel except the tensor-core GEMM waits before it triggers, the GEMM
// triggers first, and no two GEMMs are adjacent in a step.  So when a kernel
// launches, every kernel three or more launches before it has completed and
// its writes are visible.  The header fields the layer kernels test (err,
// done, K and the row counts Q, n_need, prefill_rows, written by the pack or
// chunk kernels at the start of a call or by the publish kernel of the call
// before) are therefore read before la_pdl_wait() by every kernel from the
// first RMSNorm of a call on (an error flag a kernel sets in the same call
// may be seen late; it still reaches the host).  The embedding, right after
// the pack kernel, reads them after its wait.
__device__ __forceinline__ void la_pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void la_pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 1 unless LA_PDL=0 (A/B runs): launches below carry the attribute
int la_pdl_enabled();
int la_fuse_rope();      // decode calls of bf16 models: RoPE folded into the attention

// Process-wide count of kernel launches the library has enqueued outside
// graph capture (the launches recorded into a graph are taken back out once
// captured: they run, and are counted, with each launch of the graph).
void la_note_launch();
unsigned long long la_launch_count();

// kernel<<<grid, block, smem, st>>>(args...) with programmatic stream serialisation
template <typename... KArgs, typename... Args>
static inline cudaError_t la_launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                        cudaStream_t st, Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = la_pdl_enabled();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e == cudaSuccess) la_note_launch();
    return e;
}

// Spin limit of every bounded device wait (iterations of mbarrier.try_wait,
// each of which suspends for a hardware-defined interval).
#define LA_SPIN_LIMIT (1u << 22)
