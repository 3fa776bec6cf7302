// la_gemm_noalloc: the persistent tensor-core GEMM for callers that cannot
// allocate device memory.
//
// Who cannot allocate, and why: a serving engine or framework that has
// handed all free device memory to its own pool (a KV-cache arena, a caching
// allocator) has nothing left for cudaMalloc, and a caller with latency-bound
// work on other streams cannot afford cudaFree's implicit device-wide
// synchronisation.  The other GEMM entry points allocate their workspace per
// call (la_debug_gemm) or once per context (la_init); this one takes every
// byte it needs from a fixed array compiled into the library.
//
// The scratch is one file-scope __device__ array per device, of
// LA_NOALLOC_SCRATCH_BYTES.  Host code cannot use the array's name as a
// device address, so every call, with the caller's device current, asks the
// runtime for the array's address on that device (cudaGetSymbolAddress) and
// sets the kernel's shared-memory opt-in there.  Doing both on every call
// rather than caching them keeps a call correct after the caller resets the
// device (the module, and with it the array, may then load elsewhere).  The
// first call on a device loads the library's device code there.  A problem
// whose split-tile partial sums do not fit is rejected with LA_ECAPACITY
// before any device work.
//
// What must start at zero: the header's status word and the per-tile arrival
// counters.  The counters only grow during a launch (a tile's contributors
// each add to its counter and wait for the full count), so each call must
// zero both before its GEMM starts: a small kernel on the caller's stream
// does that before every launch.  The partial-sum region needs no
// initialisation, since every slot read in a launch is written earlier in
// the same launch.
//
// One scratch region per device means two executions that overlap on a
// device would race on its partial sums and counters.  The call therefore
// holds a process-wide lock and returns only after its work on the stream has
// finished, so calls through this entry point never overlap.
#include "la_common.cuh"
#include "la_kernels.h"

#include <cstdint>
#include <cstring>
#include <mutex>

#define LA_NOALLOC_SCRATCH_BYTES (64u << 20)
#define LA_NOALLOC_MAX_DEVICES 64

namespace {

static __device__ __align__(256) unsigned char g_scratch[LA_NOALLOC_SCRATCH_BYTES];

// layout: [LaHdr, padded to 256 B][counters, padded to 256 B][partial sums]
constexpr size_t HDR_BYTES = (sizeof(LaHdr) + 255) & ~(size_t)255;

std::mutex g_lock;

__global__ void k_noalloc_reset(LaHdr* h, int* counters, int n_counters, int rows) {
    int* w = (int*)h;
    for (int i = threadIdx.x; i < (int)(sizeof(LaHdr) / sizeof(int)); i += blockDim.x) w[i] = 0;
    for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0;
    __syncthreads();
    if (threadIdx.x == 0) h->n_need = rows;
}

// Per call, on the current device: the scratch array's device address and
// the GEMM's shared-memory opt-in.
int setup_device(int dev, void** base) {
    if (dev < 0 || dev >= LA_NOALLOC_MAX_DEVICES) return LA_ENOTSUP;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return LA_ECUDA;
    if (la_tc_prepare_device() != cudaSuccess) return LA_ECUDA;
    *base = p;
    return LA_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" {

int la_gemm_noalloc(int mode, const void* w, const void* w2, int n_out, int K, const void* x, int rows, void* y,
                    void* stream) {
    if (mode < GEMM_STORE || mode > GEMM_SWIGLU || !w || !x || !y || n_out < 128 || n_out % 128 || K < 64 ||
        K % 64 || rows < 1 || rows > 1024 || !aligned16(w) || !aligned16(x) || ((uintptr_t)y & 3u))
        return LA_EINVAL;
    if (mode == GEMM_SWIGLU && (!w2 || !aligned16(w2))) return LA_EINVAL;
    const int n_cta = la_tc_ctas();
    size_t ws_floats = 0, n_counters = 0;
    la_tc_scratch_need(mode, n_out, K, rows, n_cta, &ws_floats, &n_counters);
    const size_t ctr_bytes = (n_counters * sizeof(int) + 255) & ~(size_t)255;
    if (HDR_BYTES + ctr_bytes + ws_floats * sizeof(float) > (size_t)LA_NOALLOC_SCRATCH_BYTES) return LA_ECAPACITY;

    std::lock_guard<std::mutex> guard(g_lock);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LA_ECUDA;
    void* base = nullptr;
    int rc = setup_device(dev, &base);
    if (rc) return rc;
    LaHdr* hdr = (LaHdr*)base;
    int* counters = (int*)((char*)base + HDR_BYTES);
    float* ws = (float*)((char*)base + HDR_BYTES + ctr_bytes);
    cudaStream_t st = (cudaStream_t)stream;

    TcGemm g;
    memset(&g, 0, sizeof(g));
    if (la_tc_make_map(&g.tmA, w, n_out, K, 128) ||
        la_tc_make_map(&g.tmA2, mode == GEMM_SWIGLU ? w2 : w, n_out, K, 128) ||
        la_tc_make_map(&g.tmA3, w, n_out, K, 128) || la_tc_make_act_maps(&g, x, rows, K))
        return LA_ECUDA;
    g.mode = mode;
    g.K = K;
    g.Nout = n_out;
    g.seg_tiles = 0;
    g.n_cta = n_cta;
    g.max_seg = la_tc_max_segments(n_out / 128, la_tc_k_units(mode, K), n_cta);
    g.rows_cap = ((rows + 255) / 256) * 256;
    g.out = y;
    g.ldo = n_out;
    g.logits = nullptr;
    g.ld_logits = n_out;
    TcWork wk;
    memset(&wk, 0, sizeof(wk));
    wk.ws = ws;
    wk.ws_floats = ws_floats;
    wk.counters = counters;
    wk.n_counters = (int)n_counters;
    LaDev d{};
    memset(&d, 0, sizeof(d));
    d.hdr = hdr;

    // From the reset launch on, every return first waits for the stream, with
    // the lock still held, so that no work of this call can still be running
    // on the shared array when the next call resets it.
    auto fail = [&]() {
        cudaStreamSynchronize(st);
        return LA_ECUDA;
    };
    k_noalloc_reset<<<1, 256, 0, st>>>(hdr, counters, (int)n_counters, rows);
    if (cudaGetLastError() != cudaSuccess) return fail();
    // the GEMM reads the header's row count before its dependency wait, so
    // the reset must have completed before the GEMM launches
    if (cudaStreamSynchronize(st) != cudaSuccess) return fail();
    if (la_launch_gemm_tc(d, st, g, wk, SEL_NEED, rows) != cudaSuccess) return fail();
    int err = 0;
    if (cudaMemcpyAsync(&err, &hdr->err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return fail();
    if (cudaStreamSynchronize(st) != cudaSuccess) return fail();
    return err ? err : LA_OK;
}

}  // extern "C"
