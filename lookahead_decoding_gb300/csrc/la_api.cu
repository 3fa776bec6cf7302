// C ABI of liblookahead: context, device state, the step orchestrator and
// the CUDA-graph driven generate loop.  See include/lookahead.h for the
// contract of every entry point.
#include "la_common.cuh"
#include "la_kernels.h"

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

namespace {

constexpr int PREFILL_CHUNK = 256;

struct Graph {
    cudaGraph_t g = nullptr;
    cudaGraphExec_t x = nullptr;
    int prof_begin = 0, prof_end = 0;   // the graph's timing event pairs (kernel-timing graphs)
    long long n_kernels = 0;            // kernel launches one execution runs
    unsigned long long tl_epoch = 0;    // timeline session the graph's kernels record into (timeline graphs)
};

// kernel kinds of the kernel-timing mode
enum { PK_GEMM = 0, PK_ATTN = 1, PK_ROW = 2, PK_STATE = 3, PK_KINDS = 4 };

struct ProfPair {
    cudaEvent_t a = nullptr, b = nullptr;
    int kind = 0;
};

std::atomic<unsigned long long> g_launches{0};

// the open kernel timeline (la_timeline_start), process-wide
std::mutex g_tl_mu;
LaTlRec* g_tl_table = nullptr;
unsigned int g_tl_cap = 0;
unsigned long long g_tl_epoch = 0;      // changes at every open and close

}  // namespace

void la_note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
// launches recorded into a graph at capture run only when it is launched
static void la_unnote_launches(unsigned long long n) { g_launches.fetch_sub(n, std::memory_order_relaxed); }
unsigned long long la_launch_count() { return g_launches.load(std::memory_order_relaxed); }

struct la_ctx {
    la_model_cfg cfg{};
    int bf16 = 0;
    int tc = 0;                       // tensor-core GEMMs (bf16 models unless LA_GEMM=ffma)
    size_t esz = 4;
    int max_ctx = 0, max_W = 0, max_N = 0, max_G = 0;
    int Qmax = 0, Qcap = 0, PMAX = 0, LMAX = 0, Rmax = 0, Smax = 0, Gmax = 0, rope_len = 0, out_cap = 0;
    int HD = 0;
    cudaStream_t st = nullptr;
    bool own_stream = false;
    std::string last_err;

    // weights (borrowed)
    const void *emb = nullptr, *head = nullptr, *fnorm = nullptr;
    std::vector<const void*> attn_norm, wq, wk, wv, wo, mlp_norm, wg, wu, wd;

    // device state
    LaDev d{};
    std::vector<void*> allocs;
    float* x = nullptr;
    void *xn = nullptr, *qkv = nullptr, *qbuf = nullptr, *attn = nullptr, *act = nullptr, *hn = nullptr;
    void *cache = nullptr, *temp = nullptr;
    float *rcos = nullptr, *rsin = nullptr;
    float* logits = nullptr;          // [Qcap][V] fp32
    int attn_TB = 0;
    uint32_t opts = 0;                // LA_OPT_* for requests started from now on
    CUtensorMap cache_map;            // the K/V cache as [L*2*H*max_ctx][head_dim] rows, 64 x 128 boxes, 128B swizzle
    float* logits_in = nullptr;       // [Qmax][V] staging for injected logits
    int32_t* argmax_in = nullptr;     // [Qcap]
    TcWork work{};

    // tensor-core GEMM descriptors (bf16 models)
    std::vector<TcGemm> g_qkv, g_o, g_gu, g_down;
    TcGemm g_head{};
    // decode calls through the layer-chain kernel (la_mega.cu): one launch
    // per stretch between two attention launches; a phase counter each
    int mega = 0;
    unsigned long long* mg_bar = nullptr;   // [n_layers + 1][MG_MAX_PHASES]

    // batched calls: up to max_batch requests stacked in slices of Qstride
    // rows; request b's state and cache are its own (request 0's are the
    // single-request ones above), `bd` carries the batch header
    int max_batch = 1, Qstride = 0, temp_rows = 0;
    std::vector<LaDev> req;            // per request, row arrays at its slice
    std::vector<LaDev> req_pf;         // per request, row arrays at row 0 (prefill)
    LaDev bd{};
    const LaHdr** req_hdr = nullptr;   // device array of the requests' headers
    size_t cache_bytes_req = 0;

    // request state on the host side
    bool prefilled = false, begun = false;
    int W = 0, N = 0, G = 0, mode = 0, sampling = 0;
    int prompt_len = 0;
    int debug = 0;
    float* dbg_hidden = nullptr;      // [n_layers + 1][Qcap][d_model] fp32 (debug bit 3)
    // debug bit 3: per layer, the attention output, the normalised MLP input
    // and the SwiGLU output ([n_layers][Qcap][HD | d_model | d_ffn], model dtype)
    void *dbg_attn = nullptr, *dbg_hn = nullptr, *dbg_act = nullptr;
    std::map<int, Graph> graphs;

    // kernel-timing mode (debug bit 2): event pairs recorded inside the step graph
    bool prof_capture = false;
    std::vector<ProfPair> prof;
    double prof_ms[PK_KINDS] = {0, 0, 0, 0};
    long long prof_n[PK_KINDS] = {0, 0, 0, 0};
    long long prof_samples = 0;
};

// ---------------------------------------------------------------------------
// helpers
// ---------------------------------------------------------------------------
#define CK(expr)                                          \
    do {                                                  \
        cudaError_t _e = (expr);                          \
        if (_e != cudaSuccess) {                          \
            ctx->last_err = cudaGetErrorString(_e);       \
            return LA_ECUDA;                              \
        }                                                 \
    } while (0)

// Allocates and zeroes on the context's stream: the zeroing must be ordered
// before the first kernel of that stream (a non-blocking stream does not
// order against the legacy default stream).
static int dalloc(la_ctx* ctx, void** p, size_t bytes) {
    if (bytes == 0) bytes = 16;
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) { ctx->last_err = cudaGetErrorString(e); return LA_ECUDA; }
    ctx->allocs.push_back(*p);
    e = cudaMemsetAsync(*p, 0, bytes, ctx->st);
    if (e != cudaSuccess) { ctx->last_err = cudaGetErrorString(e); return LA_ECUDA; }
    return LA_OK;
}

static void* layer_plane(la_ctx* ctx, void* base, int l, int kv, int rows) {
    size_t plane = (size_t)ctx->cfg.n_heads * rows * ctx->cfg.head_dim * ctx->esz;
    return (char*)base + ((size_t)l * 2 + kv) * plane;
}

static int read_hdr(la_ctx* ctx, LaHdr* h) {
    CK(cudaMemcpyAsync(h, ctx->d.hdr, sizeof(LaHdr), cudaMemcpyDeviceToHost, ctx->st));
    CK(cudaStreamSynchronize(ctx->st));
    return LA_OK;
}

int la_fuse_rope() {
    static int on = -1;
    if (on < 0) {
        const char* e = getenv("LA_FUSE_ROPE");
        on = (e && e[0] == '0') ? 0 : 1;
    }
    return on;
}

int la_pdl_enabled() {
    static int on = -1;
    if (on < 0) {
        const char* e = getenv("LA_PDL");
        on = (e && e[0] == '0') ? 0 : 1;
    }
    return on;
}

// Kernel-timing mode: while a timing graph is being captured, an event pair
// brackets each timed launch on the context's stream.
static int prof_open(la_ctx* ctx, int kind) {
    if (!ctx->prof_capture) return -1;
    ProfPair pp;
    pp.kind = kind;
    if (cudaEventCreate(&pp.a) != cudaSuccess || cudaEventCreate(&pp.b) != cudaSuccess) return -1;
    ctx->prof.push_back(pp);
    const int i = (int)ctx->prof.size() - 1;
    if (cudaEventRecordWithFlags(ctx->prof[i].a, ctx->st, cudaEventRecordExternal) != cudaSuccess) return -1;
    return i;
}
static void prof_close(la_ctx* ctx, int i) {
    if (i >= 0) cudaEventRecordWithFlags(ctx->prof[i].b, ctx->st, cudaEventRecordExternal);
}
// adds the last execution of graph g to the per-kind totals
static void prof_collect(la_ctx* ctx, const Graph& g) {
    if (g.prof_end <= g.prof_begin) return;
    for (int i = g.prof_begin; i < g.prof_end; ++i) {
        float ms = 0;
        if (cudaEventElapsedTime(&ms, ctx->prof[i].a, ctx->prof[i].b) == cudaSuccess) {
            ctx->prof_ms[ctx->prof[i].kind] += ms;
            ctx->prof_n[ctx->prof[i].kind] += 1;
        }
    }
    ctx->prof_samples += 1;
}

static int make_gemm(la_ctx* ctx, TcGemm* g, int mode, const void* w1, const void* w2, const void* w3, int n_seg,
                     int Nout_seg, int K, void* X, void* out, int ldo, int pair = 0) {
    memset(g, 0, sizeof(*g));
    if (la_tc_make_map(&g->tmA, w1, Nout_seg, K, 128)) return LA_ECUDA;
    if (la_tc_make_map(&g->tmA2, w2 ? w2 : w1, Nout_seg, K, 128)) return LA_ECUDA;
    if (la_tc_make_map(&g->tmA3, w3 ? w3 : w1, Nout_seg, K, 128)) return LA_ECUDA;
    if (la_tc_make_act_maps(g, X, ctx->Qcap, K)) return LA_ECUDA;
    g->mode = mode;
    g->K = K;
    g->Nout = Nout_seg * n_seg;
    g->seg_tiles = n_seg > 1 ? Nout_seg / 128 : 0;
    g->pair = (pair && (g->Nout / 128) % 2 == 0 && g->seg_tiles % 2 == 0) ? 1 : 0;
    const int utiles = g->Nout / 128 / (g->pair ? 2 : 1), ku = la_tc_k_units(mode, K, g->pair);
    g->n_cta = la_tc_pick_ctas(utiles, ku, mode);
    g->max_seg = la_tc_max_segments(utiles, ku, g->n_cta);
    g->rows_cap = ctx->Qcap;
    g->out = out;
    g->ldo = ldo;
    g->act = X;
    return LA_OK;
}

// ---------------------------------------------------------------------------
// forward passes
// ---------------------------------------------------------------------------
// split tiles a GEMM leaves to its consumer (none for CUDA-core GEMMs)
static LaSplit split_of(const la_ctx* ctx, const TcGemm* g) {
    if (!ctx->tc || !g) {
        LaSplit none{};
        none.ws = nullptr;
        return none;
    }
    return la_tc_split(*g, ctx->work);
}

// What a pass runs on: the device view whose header gives the row counts,
// the K/V cache it reads (and a prefill writes), the temporary rows of a
// call, and for a batched call the requests' headers and slice size.
struct Lane {
    const LaDev* d;
    char* cache;                    // K/V cache [L][2][H][max_ctx][dh] of the lane's (first) request
    int cache_row0;                 // that cache's first row in the cache tensor map
    int temp_rows;                  // temporary K/V rows per (layer, k/v, head) plane
    int rows_call;                  // rows of a call (all stacked slices in a batch)
    const LaHdr* const* req_hdr;    // batched call: the requests' headers
    int qstride;                    // batched call: rows per request slice (0: one request)
};

static Lane solo_lane(la_ctx* ctx) {
    return Lane{&ctx->d, (char*)ctx->cache, 0, ctx->Qmax, ctx->Qmax, nullptr, 0};
}
// request b of a batched context, for its prefill (rows from row 0)
static Lane prefill_lane(la_ctx* ctx, int b) {
    const la_model_cfg& c = ctx->cfg;
    return Lane{&ctx->req_pf[b], (char*)ctx->cache + (size_t)b * ctx->cache_bytes_req,
                b * c.n_layers * 2 * c.n_heads * ctx->max_ctx, ctx->Qmax, ctx->Qmax, nullptr, 0};
}
// a batched call of B requests
static Lane batch_lane(la_ctx* ctx, int B) {
    return Lane{&ctx->bd, (char*)ctx->cache, 0, ctx->temp_rows, B * ctx->Qstride, ctx->req_hdr, ctx->Qstride};
}

// attention of layer l for a bf16 model (RoPE folded in when `rope` is given)
static int enqueue_attention_bf16(la_ctx* ctx, int l, int sel, const Lane& ln, int rc, const LaRope* rope) {
    const la_model_cfg& c = ctx->cfg;
    const int H = c.n_heads;
    CK(la_launch_attention_bf16(*ln.d, ctx->st, ctx->qbuf, layer_plane(ctx, ln.cache, l, 0, ctx->max_ctx),
                                layer_plane(ctx, ln.cache, l, 1, ctx->max_ctx),
                                layer_plane(ctx, ctx->temp, l, 0, ln.temp_rows),
                                layer_plane(ctx, ctx->temp, l, 1, ln.temp_rows), ctx->attn, H, sel, ctx->Qcap,
                                ctx->max_ctx, ctx->Qmax, rc, ctx->attn_TB, ctx->PMAX, ctx->cache_map,
                                ln.cache_row0 + (l * 2 + 0) * H * ctx->max_ctx,
                                ln.cache_row0 + (l * 2 + 1) * H * ctx->max_ctx, ln.req_hdr, ln.qstride,
                                (long long)(ctx->cache_bytes_req / ctx->esz), c.n_layers * 2 * H * ctx->max_ctx,
                                ln.temp_rows, la_attn_tail_rows(ctx->max_W, ctx->max_N, ctx->Qmax), rope));
    return LA_OK;
}

// ---- layer-chain kernel ---------------------------------------------------------

static MgGemm mg_gemm(la_ctx* ctx, const TcGemm& g, int sel) {
    MgGemm m;
    memset(&m, 0, sizeof(m));
    m.wpack = (const uint8_t*)g.wpack;
    m.act = (const __nv_bfloat16*)g.act;
    m.mode = g.mode;
    m.K = g.K;
    m.n_tiles = g.Nout / 128;
    m.k_tiles = la_tc_k_units(g.mode, g.K);
    m.ua = la_tc_unit_atoms(g.mode);
    m.k_atoms = g.K / 64;
    m.nA = g.mode == GEMM_SWIGLU ? 2 : 1;
    m.max_seg = g.max_seg;
    m.sel = sel;
    m.defer = g.defer;
    m.n_cta = g.n_cta;
    m.ws = ctx->work.ws;
    m.ctr = (unsigned long long*)ctx->work.counters + g.ctr_off;
    m.out = g.out;
    m.ldo = g.ldo;
    m.logits = g.logits;
    m.ld_logits = g.ld_logits;
    m.part_v = ctx->work.part_v;
    m.part_i = ctx->work.part_i;
    m.part_stride = ctx->work.part_stride;
    return m;
}
static MgRows mg_rms(la_ctx* ctx, int kind, int sel, const void* gain, void* y, const TcGemm* prev) {
    MgRows r;
    memset(&r, 0, sizeof(r));
    r.kind = kind;
    r.sel = sel;
    r.dm = ctx->cfg.d_model;
    r.eps = ctx->cfg.rms_eps;
    r.x = ctx->x;
    r.g = (const __nv_bfloat16*)gain;
    r.y = (__nv_bfloat16*)y;
    r.split = split_of(ctx, prev);
    return r;
}
struct MgChain {
    MgParams p;
    int ng = 0, nr = 0;
    explicit MgChain(la_ctx* ctx, unsigned long long* bar) {
        memset(&p, 0, sizeof(p));
        p.hdr = ctx->d.hdr;
        p.tl = ctx->d.tl;
        p.need = ctx->d.need;
        p.bar = bar;
        p.rows_cap = ctx->Qmax;
        p.ns_pre = la_mega_ring_stages(ctx->Qmax);
    }
    void gemm(const MgGemm& g) { p.ph_kind[p.n_ph] = MG_PH_GEMM; p.ph_idx[p.n_ph++] = ng; p.g[ng++] = g; }
    void rows(const MgRows& r) { p.ph_kind[p.n_ph] = MG_PH_ROWS; p.ph_idx[p.n_ph++] = nr; p.r[nr++] = r; }
};


// A decode call of a single-request bf16 context: embedding, then per layer
// one layer-chain launch and the attention, then the last chain (down of the
// last layer, final RMSNorm of the needed rows, LM head), then the argmax
// over the head's tiles.  The chains compute exactly what enqueue_forward and
// enqueue_head compute for SEL_CALL.
static int enqueue_call_mega(la_ctx* ctx, int keep_logits) {
    const la_model_cfg& c = ctx->cfg;
    const LaDev& d = ctx->d;
    cudaStream_t st = ctx->st;
    const int L = c.n_layers;
    const Lane ln = solo_lane(ctx);
    const int rc = ln.rows_call;
    CK(cudaMemsetAsync(ctx->mg_bar, 0, sizeof(unsigned long long) * (L + 1) * MG_MAX_PHASES, st));
    int pi = prof_open(ctx, PK_ROW);
    la_launch_embed(d, st, c.dtype, ctx->emb, ctx->x, c.d_model, SEL_CALL, rc);
    prof_close(ctx, pi);
    {
        MgChain ch(ctx, ctx->mg_bar);
        ch.rows(mg_rms(ctx, MG_RMS, SEL_CALL, ctx->attn_norm[0], ctx->xn, nullptr));
        ch.gemm(mg_gemm(ctx, ctx->g_qkv[0], SEL_CALL));
        pi = prof_open(ctx, PK_GEMM);
        CK(la_launch_mega(ch.p, st));
        prof_close(ctx, pi);
    }
    for (int l = 0; l < L; ++l) {
        const LaRope rope{(const __nv_bfloat16*)ctx->qkv, split_of(ctx, &ctx->g_qkv[l]), ctx->rcos, ctx->rsin};
        pi = prof_open(ctx, PK_ATTN);
        int r = enqueue_attention_bf16(ctx, l, SEL_CALL, ln, rc, &rope);
        prof_close(ctx, pi);
        if (r) return r;
        MgChain ch(ctx, ctx->mg_bar + (size_t)(l + 1) * MG_MAX_PHASES);
        ch.gemm(mg_gemm(ctx, ctx->g_o[l], SEL_CALL));
        ch.rows(mg_rms(ctx, MG_RMS, SEL_CALL, ctx->mlp_norm[l], ctx->xn, &ctx->g_o[l]));
        ch.gemm(mg_gemm(ctx, ctx->g_gu[l], SEL_CALL));
        if (ctx->g_gu[l].defer && ctx->g_gu[l].max_seg > 1) {
            MgRows sw;
            memset(&sw, 0, sizeof(sw));
            sw.kind = MG_SWIGLU;
            sw.sel = SEL_CALL;
            sw.y = (__nv_bfloat16*)ctx->act;
            sw.ldo = c.d_ffn;
            sw.split = la_tc_split(ctx->g_gu[l], ctx->work);
            ch.rows(sw);
        }
        ch.gemm(mg_gemm(ctx, ctx->g_down[l], SEL_CALL));
        if (l + 1 < L) {
            ch.rows(mg_rms(ctx, MG_RMS, SEL_CALL, ctx->attn_norm[l + 1], ctx->xn, &ctx->g_down[l]));
            ch.gemm(mg_gemm(ctx, ctx->g_qkv[l + 1], SEL_CALL));
        } else {
            ch.rows(mg_rms(ctx, MG_RMS_GATHER, SEL_NEED, ctx->fnorm, ctx->hn, &ctx->g_down[l]));
            TcGemm hg = ctx->g_head;
            hg.logits = keep_logits ? ctx->logits : nullptr;
            ch.gemm(mg_gemm(ctx, hg, SEL_NEED));
        }
        pi = prof_open(ctx, PK_GEMM);
        CK(la_launch_mega(ch.p, st));
        prof_close(ctx, pi);
    }
    pi = prof_open(ctx, PK_STATE);
    la_launch_argmax_reduce(d, st, ctx->work.part_v, ctx->work.part_i, c.vocab / 128, ctx->work.part_stride, SEL_NEED,
                            rc);
    prof_close(ctx, pi);
    CK(cudaGetLastError());
    return LA_OK;
}

static int enqueue_forward(la_ctx* ctx, int sel, const Lane& ln) {
    const la_model_cfg& c = ctx->cfg;
    const LaDev& d = *ln.d;
    cudaStream_t st = ctx->st;
    const int rc = (sel == SEL_PREFILL) ? PREFILL_CHUNK : ln.rows_call;
    const int dm = c.d_model, HD = ctx->HD, F = c.d_ffn, H = c.n_heads, dh = c.head_dim;
    int pi = prof_open(ctx, PK_ROW);
    la_launch_embed(d, st, c.dtype, ctx->emb, ctx->x, dm, sel, rc);
    prof_close(ctx, pi);
    for (int l = 0; l < c.n_layers; ++l) {
        pi = prof_open(ctx, PK_ROW);
        la_launch_rmsnorm(d, st, c.dtype, ctx->x, ctx->attn_norm[l], ctx->xn, dm, c.rms_eps, sel, 0, rc,
                          split_of(ctx, (ctx->tc && l > 0) ? &ctx->g_down[l - 1] : nullptr));
        prof_close(ctx, pi);
        if ((ctx->debug & 8) && ctx->dbg_hidden)     // layer l's input residual rows (complete after this RMSNorm)
            CK(cudaMemcpyAsync(ctx->dbg_hidden + (size_t)l * ctx->Qcap * dm, ctx->x, sizeof(float) * (size_t)rc * dm,
                               cudaMemcpyDeviceToDevice, st));
        if (ctx->tc) {
            pi = prof_open(ctx, PK_GEMM);
            CK(la_launch_gemm_tc(d, st, ctx->g_qkv[l], ctx->work, sel, rc));
            prof_close(ctx, pi);
        } else {
            char* q = (char*)ctx->qkv;
            la_launch_gemm_ffma(d, st, c.dtype, GEMM_STORE, ctx->xn, dm, ctx->wq[l], nullptr, dm, HD, q, 3 * HD, sel, rc);
            la_launch_gemm_ffma(d, st, c.dtype, GEMM_STORE, ctx->xn, dm, ctx->wk[l], nullptr, dm, HD, q + HD * ctx->esz,
                                3 * HD, sel, rc);
            la_launch_gemm_ffma(d, st, c.dtype, GEMM_STORE, ctx->xn, dm, ctx->wv[l], nullptr, dm, HD,
                                q + 2 * HD * ctx->esz, 3 * HD, sel, rc);
        }
        void* kdst = (sel == SEL_PREFILL) ? layer_plane(ctx, ln.cache, l, 0, ctx->max_ctx)
                                          : layer_plane(ctx, ctx->temp, l, 0, ln.temp_rows);
        void* vdst = (sel == SEL_PREFILL) ? layer_plane(ctx, ln.cache, l, 1, ctx->max_ctx)
                                          : layer_plane(ctx, ctx->temp, l, 1, ln.temp_rows);
        int stride = (sel == SEL_PREFILL) ? ctx->max_ctx : ln.temp_rows;
        // decode calls of bf16 models fold RoPE into the attention (LA_FUSE_ROPE=0: a kernel of its own)
        const bool fuse = ctx->bf16 && ctx->tc && sel != SEL_PREFILL && la_fuse_rope();
        const LaRope rope{(const __nv_bfloat16*)ctx->qkv, split_of(ctx, ctx->tc ? &ctx->g_qkv[l] : nullptr), ctx->rcos,
                          ctx->rsin};
        if (!fuse) {
            pi = prof_open(ctx, PK_ROW);
            la_launch_rope_kv(d, st, c.dtype, ctx->qkv, ctx->rcos, ctx->rsin, ctx->qbuf, kdst, vdst, H, dh, sel,
                              ctx->Qcap, stride, rc, split_of(ctx, ctx->tc ? &ctx->g_qkv[l] : nullptr));
            prof_close(ctx, pi);
        }
        pi = prof_open(ctx, PK_ATTN);
        if (ctx->bf16) {
            int r = enqueue_attention_bf16(ctx, l, sel, ln, rc, fuse ? &rope : nullptr);
            if (r) return r;
        } else {
            CK(la_launch_attention(d, st, c.dtype, dh, ctx->qbuf, layer_plane(ctx, ln.cache, l, 0, ctx->max_ctx),
                                   layer_plane(ctx, ln.cache, l, 1, ctx->max_ctx),
                                   layer_plane(ctx, ctx->temp, l, 0, ln.temp_rows),
                                   layer_plane(ctx, ctx->temp, l, 1, ln.temp_rows), ctx->attn, H, sel, ctx->Qcap,
                                   ctx->max_ctx, ln.temp_rows, rc));
        }
        prof_close(ctx, pi);
        const bool keep = (ctx->debug & 8) && ctx->dbg_attn;
        if (keep)
            CK(cudaMemcpyAsync((char*)ctx->dbg_attn + (size_t)l * ctx->Qcap * HD * ctx->esz, ctx->attn,
                               (size_t)rc * HD * ctx->esz, cudaMemcpyDeviceToDevice, st));
        if (ctx->tc) {
            pi = prof_open(ctx, PK_GEMM);
            CK(la_launch_gemm_tc(d, st, ctx->g_o[l], ctx->work, sel, rc));
            prof_close(ctx, pi);
        } else {
            la_launch_gemm_ffma(d, st, c.dtype, GEMM_RESID, ctx->attn, HD, ctx->wo[l], nullptr, HD, dm, ctx->x, dm, sel, rc);
        }
        pi = prof_open(ctx, PK_ROW);
        la_launch_rmsnorm(d, st, c.dtype, ctx->x, ctx->mlp_norm[l], ctx->xn, dm, c.rms_eps, sel, 0, rc,
                          split_of(ctx, ctx->tc ? &ctx->g_o[l] : nullptr));
        prof_close(ctx, pi);
        if (keep)
            CK(cudaMemcpyAsync((char*)ctx->dbg_hn + (size_t)l * ctx->Qcap * dm * ctx->esz, ctx->xn,
                               (size_t)rc * dm * ctx->esz, cudaMemcpyDeviceToDevice, st));
        if (ctx->tc) {
            pi = prof_open(ctx, PK_GEMM);
            CK(la_launch_gemm_tc(d, st, ctx->g_gu[l], ctx->work, sel, rc));
            prof_close(ctx, pi);
            if (ctx->g_gu[l].defer && ctx->g_gu[l].max_seg > 1) {
                pi = prof_open(ctx, PK_ROW);
                la_launch_swiglu_split(d, st, la_tc_split(ctx->g_gu[l], ctx->work), ctx->act, F, sel, rc);
                prof_close(ctx, pi);
            }
            if (keep)
                CK(cudaMemcpyAsync((char*)ctx->dbg_act + (size_t)l * ctx->Qcap * F * ctx->esz, ctx->act,
                                   (size_t)rc * F * ctx->esz, cudaMemcpyDeviceToDevice, st));
            pi = prof_open(ctx, PK_GEMM);
            CK(la_launch_gemm_tc(d, st, ctx->g_down[l], ctx->work, sel, rc));
            prof_close(ctx, pi);
        } else {
            la_launch_gemm_ffma(d, st, c.dtype, GEMM_SWIGLU, ctx->xn, dm, ctx->wg[l], ctx->wu[l], dm, F, ctx->act, F, sel, rc);
            if (keep)
                CK(cudaMemcpyAsync((char*)ctx->dbg_act + (size_t)l * ctx->Qcap * F * ctx->esz, ctx->act,
                                   (size_t)rc * F * ctx->esz, cudaMemcpyDeviceToDevice, st));
            la_launch_gemm_ffma(d, st, c.dtype, GEMM_RESID, ctx->act, F, ctx->wd[l], nullptr, F, dm, ctx->x, dm, sel, rc);
        }
    }
    CK(cudaGetLastError());
    return LA_OK;
}

// final norm on the needed rows, LM head, argmax (and fp32 logits when kept)
static int enqueue_head(la_ctx* ctx, int keep_logits, const Lane& ln) {
    const la_model_cfg& c = ctx->cfg;
    const LaDev& d = *ln.d;
    cudaStream_t st = ctx->st;
    const int rc = ln.rows_call;
    int pi = prof_open(ctx, PK_ROW);
    la_launch_rmsnorm(d, st, c.dtype, ctx->x, ctx->fnorm, ctx->hn, c.d_model, c.rms_eps, SEL_NEED, 1, rc,
                      split_of(ctx, ctx->tc ? &ctx->g_down[c.n_layers - 1] : nullptr));
    prof_close(ctx, pi);
    if ((ctx->debug & 8) && ctx->dbg_hidden)         // the final residual (complete on the needed rows)
        CK(cudaMemcpyAsync(ctx->dbg_hidden + (size_t)c.n_layers * ctx->Qcap * c.d_model, ctx->x,
                           sizeof(float) * (size_t)std::min(rc, ctx->Qcap) * c.d_model, cudaMemcpyDeviceToDevice, st));
    if (ctx->tc) {
        TcGemm g = ctx->g_head;
        g.logits = keep_logits ? ctx->logits : nullptr;
        pi = prof_open(ctx, PK_GEMM);
        CK(la_launch_gemm_tc(d, st, g, ctx->work, SEL_NEED, rc));
        prof_close(ctx, pi);
        pi = prof_open(ctx, PK_STATE);
        la_launch_argmax_reduce(d, st, ctx->work.part_v, ctx->work.part_i, c.vocab / 128, ctx->work.part_stride,
                                SEL_NEED, rc);
        prof_close(ctx, pi);
    } else {
        la_launch_gemm_ffma(d, st, c.dtype, GEMM_LOGITS, ctx->hn, c.d_model, ctx->head, nullptr, c.d_model, c.vocab,
                            ctx->logits, c.vocab, SEL_NEED, rc);
        la_launch_argmax_rows(d, st, ctx->logits, c.vocab, SEL_NEED, rc);
    }
    CK(cudaGetLastError());
    return LA_OK;
}

// publication and K/V commit of one request: `cache` is its cache, `temp`
// the first of its temporary rows in each plane of temp_rows rows
static int enqueue_publish_commit_req(la_ctx* ctx, const LaDev& d, int verdict_given, void* cache, char* temp,
                                      int temp_rows) {
    const la_model_cfg& c = ctx->cfg;
    const int pi = prof_open(ctx, PK_STATE);
    la_launch_publish(d, ctx->st, verdict_given);
    la_launch_commit(d, ctx->st, cache, temp, c.n_layers * 2 * c.n_heads, c.n_heads, (int)(c.head_dim * ctx->esz),
                     ctx->max_ctx, temp_rows);
    prof_close(ctx, pi);
    CK(cudaGetLastError());
    return LA_OK;
}

static int enqueue_publish_commit(la_ctx* ctx, int verdict_given) {
    return enqueue_publish_commit_req(ctx, ctx->d, verdict_given, ctx->cache, (char*)ctx->temp, ctx->Qmax);
}

static int enqueue_step(la_ctx* ctx) {
    int pi = prof_open(ctx, PK_STATE);
    la_launch_pack(ctx->d, ctx->st);
    prof_close(ctx, pi);
    const Lane ln = solo_lane(ctx);
    int r;
    if (ctx->mega && !(ctx->debug & (8 | 16))) {
        // the layer-chain schedule (debug bit 3 needs the per-layer hooks of
        // the multi-launch path; bit 4 forces it for comparisons)
        r = enqueue_call_mega(ctx, (ctx->debug & 1) | ctx->sampling);
        if (r) return r;
    } else {
        r = enqueue_forward(ctx, SEL_CALL, ln);
        if (r) return r;
        r = enqueue_head(ctx, (ctx->debug & 1) | ctx->sampling, ln);
        if (r) return r;
    }
    if (ctx->sampling) {
        pi = prof_open(ctx, PK_STATE);
        CK(la_launch_sample_verify(ctx->d, ctx->st, ctx->logits, ctx->cfg.vocab, 0));
        prof_close(ctx, pi);
    }
    return enqueue_publish_commit(ctx, ctx->sampling);
}

// Points every kernel-argument block of the context at the open timeline
// table (nullptr when none), before anything is launched or captured.
static void tl_sync(la_ctx* ctx) {
    LaTlRec* t = g_tl_table;
    ctx->d.tl = t;
    ctx->bd.tl = t;
    for (auto& e : ctx->req) e.tl = t;
    for (auto& e : ctx->req_pf) e.tl = t;
}

static void drop_graph(Graph& g) {
    if (g.x) cudaGraphExecDestroy(g.x);
    if (g.g) cudaGraphDestroy(g.g);
    g.x = nullptr;
    g.g = nullptr;
}

static int get_graph(la_ctx* ctx, Graph** out) {
    int key = (ctx->debug & 1) | (ctx->sampling << 1) | (ctx->debug & 4) | (ctx->debug & 8) | (ctx->debug & 16) |
              (g_tl_table ? 32 : 0);
    auto it = ctx->graphs.find(key);
    if (it != ctx->graphs.end()) {
        if (!g_tl_table || it->second.tl_epoch == g_tl_epoch) { *out = &it->second; return LA_OK; }
        drop_graph(it->second);     // captured into an earlier timeline's table
        ctx->graphs.erase(it);
    }
    tl_sync(ctx);
    Graph g;
    g.tl_epoch = g_tl_epoch;
    CK(cudaStreamBeginCapture(ctx->st, cudaStreamCaptureModeRelaxed));
    ctx->prof_capture = (ctx->debug & 4) != 0;
    g.prof_begin = (int)ctx->prof.size();
    const unsigned long long n0 = la_launch_count();
    int r = enqueue_step(ctx);
    g.n_kernels = (long long)(la_launch_count() - n0);
    la_unnote_launches((unsigned long long)g.n_kernels);
    ctx->prof_capture = false;
    g.prof_end = (int)ctx->prof.size();
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(ctx->st, &graph);
    if (r) { if (graph) cudaGraphDestroy(graph); return r; }
    CK(e);
    g.g = graph;
    CK(cudaGraphInstantiate(&g.x, graph, 0));
    ctx->graphs[key] = g;
    *out = &ctx->graphs[key];
    return LA_OK;
}

static int check_err_word(la_ctx* ctx, const LaHdr& h) {
    if (h.err) return h.err;
    return LA_OK;
}

// Clears the device error word before a call.  A GEMM CTA that gave up on a
// bounded wait may have left a split-K arrival counter short, so the counters
// are zeroed too.
static int clear_err(la_ctx* ctx) {
    CK(cudaMemsetAsync(&ctx->d.hdr->err, 0, sizeof(int32_t), ctx->st));
    if (ctx->work.counters) CK(cudaMemsetAsync(ctx->work.counters, 0, sizeof(int) * ctx->work.n_counters, ctx->st));
    return LA_OK;
}

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
extern "C" {

const char* la_strerror(int code) {
    switch (code) {
        case LA_OK: return "ok";
        case LA_EINVAL: return "invalid argument";
        case LA_ECAPACITY: return "capacity exceeded";
        case LA_ESTATE: return "call out of order";
        case LA_ECUDA: return "CUDA error";
        case LA_EDEVICE: return "device check failed";
        case LA_ETIMEOUT: return "device wait timed out";
        case LA_ENOTSUP: return "not supported";
        default: return "unknown error";
    }
}

const char* la_last_cuda_error(la_ctx* ctx) { return ctx ? ctx->last_err.c_str() : ""; }

void la_free(la_ctx* ctx) {
    if (!ctx) return;
    if (ctx->st) cudaStreamSynchronize(ctx->st);
    for (auto& kv : ctx->graphs) drop_graph(kv.second);
    for (auto& pp : ctx->prof) {
        if (pp.a) cudaEventDestroy(pp.a);
        if (pp.b) cudaEventDestroy(pp.b);
    }
    for (void* p : ctx->allocs) cudaFree(p);
    if (ctx->own_stream && ctx->st) cudaStreamDestroy(ctx->st);
    delete ctx;
}

int la_init(const la_model_cfg* cfg, const la_weights* w, int max_ctx, int max_W, int max_N, int max_G, void* stream,
            la_ctx** out) {
    return la_init_batch(cfg, w, max_ctx, max_W, max_N, max_G, 1, stream, out);
}

int la_init_batch(const la_model_cfg* cfg, const la_weights* w, int max_ctx, int max_W, int max_N, int max_G,
                  int max_batch, void* stream, la_ctx** out) {
    if (!cfg || !w || !out) return LA_EINVAL;
    if (max_batch < 1) return LA_EINVAL;
    *out = nullptr;
    const la_model_cfg& c = *cfg;
    if (c.n_layers < 1 || c.n_heads < 1 || c.vocab < 2 || c.d_model != c.n_heads * c.head_dim ||
        c.n_kv_heads != c.n_heads || !(c.rms_eps > 0.f) || !(c.rope_theta > 0.f))
        return LA_EINVAL;
    if (c.dtype != LA_F32 && c.dtype != LA_BF16) return LA_ENOTSUP;
    if (c.head_dim != 32 && c.head_dim != 128) return LA_ENOTSUP;
    if (c.d_model > 8192) return LA_ENOTSUP;
    if (c.dtype == LA_F32 && (c.d_model % 64 || c.d_ffn % 64 || c.vocab % 64)) return LA_ENOTSUP;
    if (c.dtype == LA_BF16 && (c.d_model % 128 || c.d_ffn % 128 || c.vocab % 128 || c.head_dim != 128)) return LA_ENOTSUP;
    if (max_N < 3 || max_N > LA_MAX_R + 1 || max_W < 1 || max_W > LA_MAX_W || max_G < 0 || max_G > LA_MAX_G ||
        max_ctx < 2)
        return LA_EINVAL;
    if (!w->tok_emb || !w->lm_head || !w->final_norm || !w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo ||
        !w->mlp_norm || !w->w_gate || !w->w_up || !w->w_down)
        return LA_EINVAL;

    // The weights may still be in flight on another stream (the caller's
    // allocator or generator): wait for all work already issued on the device.
    if (cudaDeviceSynchronize() != cudaSuccess) return LA_ECUDA;
    la_ctx* ctx = new la_ctx();
    ctx->cfg = c;
    ctx->bf16 = (c.dtype == LA_BF16);
    {
        const char* gsel = getenv("LA_GEMM");    // "ffma": CUDA-core reference GEMMs for every dtype
        ctx->tc = ctx->bf16 && !(gsel && strcmp(gsel, "ffma") == 0);
    }
    ctx->esz = ctx->bf16 ? 2 : 4;
    ctx->max_ctx = max_ctx;
    ctx->max_W = max_W;
    ctx->max_N = max_N;
    ctx->max_G = max_G;
    ctx->HD = c.n_heads * c.head_dim;
    ctx->Rmax = max_N - 1;
    ctx->Smax = max_N - 1;
    ctx->Gmax = std::max(1, max_G);
    ctx->LMAX = std::max(1, max_W + max_N - 3);
    ctx->PMAX = max_W + 2 * max_N;
    int steadyQ = (max_W + max_G) * (max_N - 1);
    int warmQ = 1 + (max_N - 1) * (max_W + max_N - 3);
    ctx->Qmax = std::max(steadyQ, warmQ) + 16;
    ctx->max_batch = max_batch;
    ctx->Qstride = (ctx->Qmax + 15) / 16 * 16;
    if (max_batch > 1 && (c.dtype != LA_BF16 || max_batch * ctx->Qstride > 1024)) { delete ctx; return LA_ENOTSUP; }
    ctx->temp_rows = max_batch > 1 ? max_batch * ctx->Qstride : ctx->Qmax;
    ctx->Qcap = ((std::max(std::max(ctx->Qmax, PREFILL_CHUNK), max_batch > 1 ? ctx->temp_rows : 0) + 255) / 256) * 256;
    ctx->rope_len = max_ctx + ctx->PMAX + 1;
    ctx->out_cap = max_ctx + 32;

    if (stream) ctx->st = (cudaStream_t)stream;
    else {
        if (cudaStreamCreateWithFlags(&ctx->st, cudaStreamNonBlocking) != cudaSuccess) { delete ctx; return LA_ECUDA; }
        ctx->own_stream = true;
    }
    ctx->emb = w->tok_emb;
    ctx->head = w->lm_head;
    ctx->fnorm = w->final_norm;
    for (int l = 0; l < c.n_layers; ++l) {
        ctx->attn_norm.push_back(w->attn_norm[l]);
        ctx->wq.push_back(w->wq[l]);
        ctx->wk.push_back(w->wk[l]);
        ctx->wv.push_back(w->wv[l]);
        ctx->wo.push_back(w->wo[l]);
        ctx->mlp_norm.push_back(w->mlp_norm[l]);
        ctx->wg.push_back(w->w_gate[l]);
        ctx->wu.push_back(w->w_up[l]);
        ctx->wd.push_back(w->w_down[l]);
    }

    int r = LA_OK;
    LaDev& d = ctx->d;
    auto A = [&](void** p, size_t bytes) { if (r == LA_OK) r = dalloc(ctx, p, bytes); };
    const size_t V = c.vocab;
    A((void**)&d.hdr, sizeof(LaHdr));
    A((void**)&d.window, sizeof(int32_t) * ctx->Rmax * ctx->LMAX);
    A((void**)&d.pool_tok, sizeof(int32_t) * V * ctx->Gmax * ctx->Smax);
    A((void**)&d.pool_cnt, sizeof(int32_t) * V);
    A((void**)&d.prompt, sizeof(int32_t) * max_ctx);
    A((void**)&d.row_tok, sizeof(int32_t) * ctx->Qcap);
    A((void**)&d.row_pos, sizeof(int32_t) * ctx->Qcap);
    A((void**)&d.row_meta, sizeof(int32_t) * ctx->Qcap);
    A((void**)&d.row_path, sizeof(int32_t) * ctx->Qcap * ctx->PMAX);
    A((void**)&d.need, sizeof(int32_t) * ctx->Qcap);
    A((void**)&d.argmax, sizeof(int32_t) * ctx->Qcap);
    A((void**)&d.out, sizeof(int32_t) * ctx->out_cap);
    A((void**)&d.commit_rows, sizeof(int32_t) * 16);
    A((void**)&ctx->argmax_in, sizeof(int32_t) * ctx->Qcap);
    d.V = c.vocab;
    d.Gmax = ctx->Gmax;
    d.Smax = ctx->Smax;
    d.Rmax = ctx->Rmax;
    d.LMAX = ctx->LMAX;
    d.PMAX = ctx->PMAX;
    d.Qmax = ctx->Qmax;
    d.Qcap = ctx->Qcap;
    d.max_ctx = max_ctx;
    d.out_cap = ctx->out_cap;

    const size_t dm = c.d_model, HD = ctx->HD, F = c.d_ffn, Qc = ctx->Qcap, es = ctx->esz;
    A((void**)&ctx->x, sizeof(float) * Qc * dm);
    A(&ctx->xn, es * Qc * dm);
    A(&ctx->qkv, es * Qc * 3 * HD);
    A(&ctx->qbuf, es * Qc * HD);
    A(&ctx->attn, es * Qc * HD);
    A(&ctx->act, es * Qc * F);
    A(&ctx->hn, es * Qc * dm);
    ctx->cache_bytes_req = es * (size_t)c.n_layers * 2 * HD * max_ctx;
    A(&ctx->cache, ctx->cache_bytes_req * max_batch);
    A(&ctx->temp, es * (size_t)c.n_layers * 2 * HD * ctx->temp_rows);
    A((void**)&ctx->rcos, sizeof(float) * (size_t)ctx->rope_len * (c.head_dim / 2));
    A((void**)&ctx->rsin, sizeof(float) * (size_t)ctx->rope_len * (c.head_dim / 2));
    A((void**)&ctx->logits, sizeof(float) * Qc * V);
    A((void**)&ctx->logits_in, sizeof(float) * (size_t)ctx->Qmax * V);
    if (ctx->bf16) {
        ctx->attn_TB = la_attn_tail_blocks(ctx->PMAX);
        if (!r && la_tc_make_map(&ctx->cache_map, ctx->cache, max_batch * c.n_layers * 2 * c.n_heads * max_ctx,
                                 c.head_dim, 128))
            r = LA_ECUDA;
        if (la_attn_smem_bytes(ctx->attn_TB, la_attn_tail_rows(max_W, max_N, ctx->Qmax), ctx->PMAX, ctx->Qmax) >
            227 * 1024)
            r = LA_ENOTSUP;
    }
    // batched calls: request 0 keeps the state above; requests 1.. get their
    // own header, window, pool, prompt, out ring and commit plan
    ctx->req_pf.assign(max_batch, d);
    for (int b = 1; b < max_batch && !r; ++b) {
        LaDev& e = ctx->req_pf[b];
        A((void**)&e.hdr, sizeof(LaHdr));
        A((void**)&e.window, sizeof(int32_t) * ctx->Rmax * ctx->LMAX);
        A((void**)&e.pool_tok, sizeof(int32_t) * V * ctx->Gmax * ctx->Smax);
        A((void**)&e.pool_cnt, sizeof(int32_t) * V);
        A((void**)&e.prompt, sizeof(int32_t) * max_ctx);
        A((void**)&e.out, sizeof(int32_t) * ctx->out_cap);
        A((void**)&e.commit_rows, sizeof(int32_t) * 16);
    }
    LaHdr* batch_hdr = nullptr;
    if (max_batch > 1) {
        A((void**)&batch_hdr, sizeof(LaHdr));
        A((void**)&ctx->req_hdr, sizeof(LaHdr*) * max_batch);
    }
    if (r) { la_free(ctx); return r; }
    if (max_batch > 1) {
        // the batch's view: shared rows and activations, the batch header
        ctx->bd = d;
        ctx->bd.hdr = batch_hdr;
        // the requests' views: their own state, their slice of the rows
        ctx->req = ctx->req_pf;
        std::vector<const LaHdr*> hs(max_batch);
        for (int b = 0; b < max_batch; ++b) {
            LaDev& e = ctx->req[b];
            const size_t o = (size_t)b * ctx->Qstride;
            e.row_tok = d.row_tok + o;
            e.row_pos = d.row_pos + o;
            e.row_meta = d.row_meta + o;
            e.row_path = d.row_path + o * ctx->PMAX;
            e.need = d.need + o;
            e.argmax = d.argmax + o;
            e.row_base = (int)o;
            e.pad_to = ctx->Qstride;
            e.batch = batch_hdr;
            hs[b] = e.hdr;
        }
        if (cudaMemcpyAsync(ctx->req_hdr, hs.data(), sizeof(LaHdr*) * max_batch, cudaMemcpyHostToDevice, ctx->st) !=
            cudaSuccess) {
            la_free(ctx);
            return LA_ECUDA;
        }
    }
    la_launch_rope_table(ctx->rcos, ctx->rsin, ctx->rope_len, c.head_dim, (double)c.rope_theta, ctx->st);

    if (ctx->tc) {
        // tensor-core GEMM descriptors and scratch
        ctx->g_qkv.resize(c.n_layers);
        ctx->g_o.resize(c.n_layers);
        ctx->g_gu.resize(c.n_layers);
        ctx->g_down.resize(c.n_layers);
        // QKV, O, down and the LM head stream units of two adjacent output tiles (one
        // 32 KB copy of one 64-column atom each, as gate/up does), which
        // halves a stage's activation bytes; packed weights only, and not
        // in the layer-chain kernel (LA_TC_PAIR=0: single-tile units)
        const char* pp = getenv("LA_TC_PAIR");      // bit 0 QKV, bit 1 O, bit 2 down, bit 3 LM head
        const char* pk = getenv("LA_TC_PACK");
        const char* mg = getenv("LA_MEGA");
        // (only where the rows every decode call stacks fit 128: above, a
        // unit's two accumulators fill TMEM and the kernel keeps one buffer.
        // A request's calls always carry the lookahead branch's W (N - 1)
        // rows and the ordinary row, and candidates add rows only to the calls
        // that have them; a batched call stacks every request's whole slice.)
        const int call_rows = max_batch > 1 ? max_batch * ctx->Qstride : max_W * (max_N - 1) + 1;
        const int pmask = (!(pk && pk[0] == '0') && !(mg && mg[0] == '1') && call_rows <= 128)
                              ? (pp ? atoi(pp) : 15) : 0;
        for (int l = 0; l < c.n_layers && !r; ++l) {
            r = make_gemm(ctx, &ctx->g_qkv[l], GEMM_STORE, ctx->wq[l], ctx->wk[l], ctx->wv[l], 3, (int)HD, (int)dm,
                          ctx->xn, ctx->qkv, (int)(3 * HD), pmask & 1);
            if (!r) r = make_gemm(ctx, &ctx->g_o[l], GEMM_RESID, ctx->wo[l], nullptr, nullptr, 1, (int)dm, (int)HD,
                                  ctx->attn, ctx->x, (int)dm, (pmask >> 1) & 1);
            if (!r) r = make_gemm(ctx, &ctx->g_gu[l], GEMM_SWIGLU, ctx->wg[l], ctx->wu[l], nullptr, 1, (int)F, (int)dm,
                                  ctx->xn, ctx->act, (int)F);
            if (!r) r = make_gemm(ctx, &ctx->g_down[l], GEMM_RESID, ctx->wd[l], nullptr, nullptr, 1, (int)dm, (int)F,
                                  ctx->act, ctx->x, (int)dm, (pmask >> 2) & 1);
        }
        if (!r) r = make_gemm(ctx, &ctx->g_head, GEMM_LOGITS, ctx->head, nullptr, nullptr, 1, (int)V, (int)dm, ctx->hn,
                              nullptr, 0, (pmask >> 3) & 1);
        if (r) { la_free(ctx); return r; }
        ctx->g_head.ld_logits = (int)V;
        // unit-contiguous weight images (one bulk copy per unit); LA_TC_PACK=0
        // (A/B runs) keeps the tensor-map loads of the row-major weights
        const char* pe = getenv("LA_TC_PACK");
        if (!(pe && pe[0] == '0')) {
            auto pack = [&](TcGemm& g, const void* w1, const void* w2, const void* w3) {
                if (r) return;
                void* dst = nullptr;
                r = dalloc(ctx, &dst, la_tc_packed_bytes(g));
                if (!r && la_tc_pack(g, w1, w2, w3, dst, ctx->st) != cudaSuccess) r = LA_ECUDA;
                if (!r) g.wpack = dst;
            };
            for (int l = 0; l < c.n_layers; ++l) {
                pack(ctx->g_qkv[l], ctx->wq[l], ctx->wk[l], ctx->wv[l]);
                pack(ctx->g_o[l], ctx->wo[l], nullptr, nullptr);
                pack(ctx->g_gu[l], ctx->wg[l], ctx->wu[l], nullptr);
                pack(ctx->g_down[l], ctx->wd[l], nullptr, nullptr);
            }
            pack(ctx->g_head, ctx->head, nullptr, nullptr);
            if (r) { la_free(ctx); return r; }
        }
        // the layer GEMMs leave their split tiles to RoPE, RMSNorm and SwiGLU
        const int defer = la_tc_defer_default();
        for (int l = 0; l < c.n_layers; ++l)
            ctx->g_qkv[l].defer = ctx->g_o[l].defer = ctx->g_gu[l].defer = ctx->g_down[l].defer = defer;
        size_t wsf = 0;
        int qchunks = ctx->Qcap / 256;
        auto need_ws = [&](const TcGemm& g) {
            const size_t planes = (g.mode == GEMM_SWIGLU || g.pair) ? 2 : 1;
            const size_t utiles = (size_t)(g.Nout / 128) / (g.pair ? 2 : 1);
            if (g.max_seg > 1) wsf = std::max(wsf, utiles * qchunks * g.max_seg * planes * 256 * 128);
        };
        need_ws(ctx->g_qkv[0]);
        need_ws(ctx->g_o[0]);
        need_ws(ctx->g_gu[0]);
        need_ws(ctx->g_down[0]);
        need_ws(ctx->g_head);
        ctx->work.ws_floats = wsf;
        A((void**)&ctx->work.ws, sizeof(float) * std::max<size_t>(wsf, 4));
        // split-tile counters: a region per GEMM (each tile's counter counts
        // arrivals over all launches of that GEMM)
        int slots = 0;
        auto give = [&](TcGemm& g) { g.ctr_off = slots; slots += (g.Nout / 128) * qchunks; };
        for (int l = 0; l < c.n_layers; ++l) {
            give(ctx->g_qkv[l]);
            give(ctx->g_o[l]);
            give(ctx->g_gu[l]);
            give(ctx->g_down[l]);
        }
        give(ctx->g_head);
        ctx->work.n_counters = LA_TC_CTR_PER_TILE * slots;
        A((void**)&ctx->work.counters, sizeof(int) * ctx->work.n_counters);
        ctx->work.part_stride = ctx->Qcap;
        A((void**)&ctx->work.part_v, sizeof(float) * (V / 128) * ctx->Qcap);
        A((void**)&ctx->work.part_i, sizeof(int) * (V / 128) * ctx->Qcap);
        if (r) { la_free(ctx); return r; }
        // decode calls through the layer-chain kernel: single-request bf16
        // contexts whose calls fit its accumulators, with packed weights, the
        // deferred split tiles and one GEMM CTA per SM (LA_MEGA=0: the
        // multi-launch schedule, for A/B runs)
        const char* me = getenv("LA_MEGA");
        bool mega = (me && me[0] == '1') && ctx->bf16 && max_batch == 1 && ctx->Qmax <= MG_MAX_ROWS_PER_CALL &&
                    defer && la_fuse_rope() && c.head_dim == 128;
        const int sms = la_tc_ctas();
        auto fits = [&](const TcGemm& g) { return g.wpack != nullptr && g.n_cta == sms; };
        for (int l = 0; l < c.n_layers && mega; ++l)
            mega = fits(ctx->g_qkv[l]) && fits(ctx->g_o[l]) && fits(ctx->g_gu[l]) && fits(ctx->g_down[l]);
        mega = mega && fits(ctx->g_head);
        if (mega) {
            A((void**)&ctx->mg_bar, sizeof(unsigned long long) * (c.n_layers + 1) * MG_MAX_PHASES);
            if (r) { la_free(ctx); return r; }
            ctx->mega = 1;
        }
    }
    if (cudaStreamSynchronize(ctx->st) != cudaSuccess) {
        ctx->last_err = cudaGetErrorString(cudaGetLastError());
        la_free(ctx);
        return LA_ECUDA;
    }
    *out = ctx;
    return LA_OK;
}

int la_query(la_ctx* ctx, int32_t* s) {
    if (!ctx || !s) return LA_EINVAL;
    s[0] = ctx->Qmax; s[1] = ctx->max_W; s[2] = ctx->max_N; s[3] = ctx->max_G;
    s[4] = ctx->max_ctx; s[5] = ctx->cfg.vocab; s[6] = ctx->LMAX; s[7] = ctx->PMAX;
    return LA_OK;
}

int la_set_debug(la_ctx* ctx, int flags) {
    if (!ctx || (flags & ~(1 | 4 | 8 | 16))) return LA_EINVAL;
    if ((flags & 8) && !ctx->dbg_hidden) {
        const la_model_cfg& c = ctx->cfg;
        const size_t rows = (size_t)ctx->Qcap;
        int r = dalloc(ctx, (void**)&ctx->dbg_hidden, sizeof(float) * (size_t)(c.n_layers + 1) * rows * c.d_model);
        if (!r) r = dalloc(ctx, &ctx->dbg_attn, ctx->esz * (size_t)c.n_layers * rows * ctx->HD);
        if (!r) r = dalloc(ctx, &ctx->dbg_hn, ctx->esz * (size_t)c.n_layers * rows * c.d_model);
        if (!r) r = dalloc(ctx, &ctx->dbg_act, ctx->esz * (size_t)c.n_layers * rows * c.d_ffn);
        if (r) return r;
    }
    ctx->debug = flags;
    return LA_OK;
}

int la_debug_layer(la_ctx* ctx, int layer, int what, void* host, int rows) {
    if (!ctx || !host || layer < 0 || layer > ctx->cfg.n_layers || rows < 1 || what < 0 || what > 3) return LA_EINVAL;
    if (what > 0 && layer == ctx->cfg.n_layers) return LA_EINVAL;
    if (!(ctx->debug & 8) || !ctx->dbg_hidden) return LA_ESTATE;
    if (rows > ctx->Qcap) return LA_ECAPACITY;
    const la_model_cfg& c = ctx->cfg;
    const size_t width[4] = {(size_t)c.d_model, (size_t)ctx->HD, (size_t)c.d_model, (size_t)c.d_ffn};
    const size_t esz = what == 0 ? sizeof(float) : ctx->esz;
    const char* base = what == 0 ? (const char*)ctx->dbg_hidden
                     : (const char*)(what == 1 ? ctx->dbg_attn : what == 2 ? ctx->dbg_hn : ctx->dbg_act);
    CK(cudaMemcpyAsync(host, base + (size_t)layer * ctx->Qcap * width[what] * esz, esz * (size_t)rows * width[what],
                       cudaMemcpyDeviceToHost, ctx->st));
    CK(cudaStreamSynchronize(ctx->st));
    return LA_OK;
}

int la_profile_read(la_ctx* ctx, double* ms4, int64_t* launches4, int64_t* samples) {
    if (!ctx || !ms4 || !launches4) return LA_EINVAL;
    for (int k = 0; k < PK_KINDS; ++k) {
        ms4[k] = ctx->prof_ms[k];
        launches4[k] = ctx->prof_n[k];
        ctx->prof_ms[k] = 0;
        ctx->prof_n[k] = 0;
    }
    if (samples) *samples = ctx->prof_samples;
    ctx->prof_samples = 0;
    return LA_OK;
}

// ---- kernel timeline (process-wide) ----
int la_timeline_start(int64_t max_ctas) {
    if (max_ctas < 1 || max_ctas > (int64_t(1) << 30)) return LA_EINVAL;
    std::lock_guard<std::mutex> lk(g_tl_mu);
    if (g_tl_table) return LA_EINVAL;
    if (cudaDeviceSynchronize() != cudaSuccess) return LA_ECUDA;
    LaTlRec* t = nullptr;
    const size_t bytes = sizeof(LaTlRec) * (size_t)(max_ctas + 1);
    if (cudaMalloc(&t, bytes) != cudaSuccess) return LA_ECUDA;
    const LaTlHead head{0u, (unsigned int)max_ctas};
    if (cudaMemset(t, 0, bytes) != cudaSuccess || cudaMemcpy(t, &head, sizeof(head), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(t);
        return LA_ECUDA;
    }
    g_tl_table = t;
    g_tl_cap = (unsigned int)max_ctas;
    ++g_tl_epoch;
    return LA_OK;
}

int la_timeline_stop(int64_t* rec, int64_t cap, int64_t* n) {
    if (!n || cap < 0 || (cap > 0 && !rec)) return LA_EINVAL;
    std::lock_guard<std::mutex> lk(g_tl_mu);
    if (!g_tl_table) return LA_ESTATE;
    std::vector<LaTlRec> h((size_t)g_tl_cap + 1);
    const cudaError_t e1 = cudaDeviceSynchronize();
    const cudaError_t e2 = cudaMemcpy(h.data(), g_tl_table, sizeof(LaTlRec) * h.size(), cudaMemcpyDeviceToHost);
    cudaFree(g_tl_table);
    g_tl_table = nullptr;
    g_tl_cap = 0;
    ++g_tl_epoch;
    if (e1 != cudaSuccess || e2 != cudaSuccess) return LA_ECUDA;
    LaTlHead head;
    std::memcpy(&head, &h[0], sizeof(head));
    const unsigned int kept = std::min(head.count, head.cap);
    std::vector<const LaTlRec*> used;
    used.reserve(kept);
    for (unsigned int i = 0; i < kept; ++i) used.push_back(&h[1 + i]);
    std::stable_sort(used.begin(), used.end(),
                     [](const LaTlRec* a, const LaTlRec* b) { return a->start < b->start; });
    *n = (int64_t)head.count;
    for (int64_t i = 0; i < (int64_t)used.size() && i < cap; ++i) {
        const LaTlRec* x = used[i];
        rec[5 * i + 0] = (int64_t)x->start;
        rec[5 * i + 1] = (int64_t)x->end;
        rec[5 * i + 2] = (int64_t)x->id;
        rec[5 * i + 3] = (int64_t)x->block;
        rec[5 * i + 4] = (int64_t)x->blocks;
    }
    return LA_OK;
}

// three timing events, destroyed on every return path
struct Events3 {
    cudaEvent_t e[3] = {nullptr, nullptr, nullptr};
    cudaError_t create() {
        for (auto& x : e) {
            cudaError_t r = cudaEventCreate(&x);
            if (r != cudaSuccess) return r;
        }
        return cudaSuccess;
    }
    ~Events3() {
        for (auto& x : e)
            if (x) cudaEventDestroy(x);
    }
};

static int check_sampling(const la_sampling* s) {
    if (!s) return LA_OK;
    if (!(s->temperature > 0.f) || !(s->top_p > 0.f) || !(s->top_p <= 1.f)) return LA_EINVAL;
    return LA_OK;
}

static int do_prefill(la_ctx* ctx, const int32_t* prompt, int n, const la_sampling* s, const Lane& ln) {
    const la_model_cfg& c = ctx->cfg;
    const LaDev& d = *ln.d;
    if (!prompt || n < 1) return LA_EINVAL;
    if (n > ctx->max_ctx - 1) return LA_ECAPACITY;
    for (int i = 0; i < n; ++i)
        if (prompt[i] < 0 || prompt[i] >= c.vocab) return LA_EINVAL;
    ctx->prefilled = false;
    ctx->begun = false;
    CK(cudaMemcpyAsync(d.prompt, prompt, sizeof(int32_t) * n, cudaMemcpyHostToDevice, ctx->st));
    LaHdr h0;
    memset(&h0, 0, sizeof(h0));
    h0.prompt_len = n;
    h0.max_out = 1;
    h0.S = 1;
    if (s) {
        h0.sampling = 1;
        h0.temperature = s->temperature;
        h0.top_p = s->top_p;
        h0.seed_lo = (uint32_t)(s->seed & 0xffffffffu);
        h0.seed_hi = (uint32_t)(s->seed >> 32);
    }
    CK(cudaMemcpyAsync(d.hdr, &h0, sizeof(h0), cudaMemcpyHostToDevice, ctx->st));
    CK(cudaMemsetAsync(d.pool_cnt, 0, sizeof(int32_t) * c.vocab, ctx->st));
    for (int c0 = 0; c0 < n; c0 += PREFILL_CHUNK) {
        int m = std::min(PREFILL_CHUNK, n - c0);
        la_launch_prefill_rows(d, ctx->st, c0, m);
        int r = enqueue_forward(ctx, SEL_PREFILL, ln);
        if (r) return r;
    }
    la_launch_prefill_need(d, ctx->st, (n - 1) % PREFILL_CHUNK);
    int r = enqueue_head(ctx, (ctx->debug & 1) | (s ? 1 : 0), ln);
    if (r) return r;
    if (s) CK(la_launch_sample_verify(d, ctx->st, ctx->logits, c.vocab, 1));
    la_launch_prefill_finish(d, ctx->st, n);
    CK(cudaGetLastError());
    ctx->prompt_len = n;
    return LA_OK;
}

int la_prefill(la_ctx* ctx, const int32_t* prompt, int n, const la_sampling* s, int32_t* first_token) {
    if (!ctx || !first_token) return LA_EINVAL;
    int r = check_sampling(s);
    if (r) return r;
    tl_sync(ctx);
    r = do_prefill(ctx, prompt, n, s, solo_lane(ctx));
    if (r) return r;
    LaHdr h;
    r = read_hdr(ctx, &h);
    if (r) return r;
    if (h.err) return h.err;
    *first_token = h.x_t;
    ctx->prefilled = true;
    return LA_OK;
}

int la_set_options(la_ctx* ctx, uint32_t flags) {
    if (!ctx || (flags & ~(LA_OPT_POOL_FROM_PROMPT | LA_OPT_POOL_FROM_OUTPUT | LA_OPT_SLICE_WINDOW))) return LA_EINVAL;
    ctx->opts = flags;
    return LA_OK;
}

static int begin_request(la_ctx* ctx, int mode, int W, int N, int G, const la_sampling* s, int max_out) {
    if (mode == MODE_LOOKAHEAD) {
        if (N < 3 || W < 1 || G < 0) return LA_EINVAL;
        if (N > ctx->max_N || W > ctx->max_W || G > ctx->max_G) return LA_ECAPACITY;
    }
    ctx->mode = mode;
    ctx->W = W; ctx->N = N; ctx->G = G;
    ctx->sampling = s ? 1 : 0;
    la_launch_begin(ctx->d, ctx->st, mode, W, N, G, ctx->sampling, s ? s->temperature : 1.f, s ? s->top_p : 1.f,
                    s ? s->seed : 0, max_out, (int)ctx->opts);
    CK(cudaGetLastError());
    ctx->begun = true;
    return LA_OK;
}

int la_step(la_ctx* ctx, int W, int N, int G, const la_sampling* s, int32_t* out, int* n_out) {
    if (!ctx || !out || !n_out) return LA_EINVAL;
    if (check_sampling(s)) return LA_EINVAL;
    if (!ctx->prefilled) return LA_ESTATE;
    if (N < 3 || W < 1 || G < 0) return LA_EINVAL;
    if (N > ctx->max_N || W > ctx->max_W || G > ctx->max_G) return LA_ECAPACITY;
    tl_sync(ctx);
    int r;
    if (!ctx->begun) {
        r = begin_request(ctx, MODE_LOOKAHEAD, W, N, G, s, ctx->out_cap);
        if (r) return r;
    } else if (ctx->mode != MODE_LOOKAHEAD || W != ctx->W || N != ctx->N || G != ctx->G ||
               ctx->sampling != (s ? 1 : 0)) {
        return LA_ESTATE;
    }
    r = clear_err(ctx);
    if (r) return r;
    r = enqueue_step(ctx);
    if (r) return r;
    LaHdr h;
    r = read_hdr(ctx, &h);
    if (r) return r;
    if (h.err) return h.err;
    for (int i = 0; i < h.E; ++i) out[i] = h.emitted[i];
    *n_out = h.E;
    return LA_OK;
}

int la_step_inject(la_ctx* ctx, int W, int N, int G, const la_sampling* s, int Q, const int32_t* argmax,
                   const float* logits, int32_t* out, int* n_out) {
    if (!ctx || !out || !n_out || !argmax) return LA_EINVAL;
    if (check_sampling(s) || (s && !logits)) return LA_EINVAL;
    if (!ctx->prefilled) return LA_ESTATE;
    if (N < 3 || W < 1 || G < 0) return LA_EINVAL;
    if (N > ctx->max_N || W > ctx->max_W || G > ctx->max_G) return LA_ECAPACITY;
    tl_sync(ctx);
    int r;
    if (!ctx->begun) {
        r = begin_request(ctx, MODE_LOOKAHEAD, W, N, G, s, ctx->out_cap);
        if (r) return r;
    } else if (ctx->mode != MODE_LOOKAHEAD || W != ctx->W || N != ctx->N || G != ctx->G ||
               ctx->sampling != (s ? 1 : 0)) {
        return LA_ESTATE;
    }
    r = clear_err(ctx);
    if (r) return r;
    la_launch_pack(ctx->d, ctx->st);
    LaHdr h;
    r = read_hdr(ctx, &h);
    if (r) return r;
    if (h.err) return h.err;
    if (h.Q != Q || Q > ctx->Qcap) return LA_ESTATE;
    for (int q = 0; q < Q; ++q)
        if (argmax[q] < 0 || argmax[q] >= ctx->cfg.vocab) return LA_EINVAL;
    CK(cudaMemcpyAsync(ctx->argmax_in, argmax, sizeof(int32_t) * Q, cudaMemcpyHostToDevice, ctx->st));
    if (s) {
        if (Q > ctx->Qmax) return LA_ECAPACITY;
        CK(cudaMemcpyAsync(ctx->logits_in, logits, sizeof(float) * (size_t)Q * ctx->cfg.vocab, cudaMemcpyHostToDevice,
                           ctx->st));
    }
    la_launch_inject_map(ctx->d, ctx->st, ctx->argmax_in, s ? ctx->logits_in : nullptr, ctx->logits, ctx->cfg.vocab);
    if (s) CK(la_launch_sample_verify(ctx->d, ctx->st, ctx->logits, ctx->cfg.vocab, 0));
    r = enqueue_publish_commit(ctx, s ? 1 : 0);
    if (r) return r;
    r = read_hdr(ctx, &h);
    if (r) return r;
    if (h.err) return h.err;
    for (int i = 0; i < h.E; ++i) out[i] = h.emitted[i];
    *n_out = h.E;
    return LA_OK;
}

static int run_generate(la_ctx* ctx, int mode, const int32_t* prompt, int n, int max_new, int W, int N, int G,
                        const la_sampling* s, int32_t* out, int* n_out, la_stats* stats) {
    if (!ctx || !out || !n_out || max_new < 1) return LA_EINVAL;
    if (check_sampling(s)) return LA_EINVAL;
    if (mode == MODE_LOOKAHEAD) {
        if (N < 3 || W < 1 || G < 0) return LA_EINVAL;
        if (N > ctx->max_N || W > ctx->max_W || G > ctx->max_G) return LA_ECAPACITY;
    }
    if (n + max_new > ctx->max_ctx) return LA_ECAPACITY;
    tl_sync(ctx);
    Events3 ev;
    CK(ev.create());
    cudaEvent_t e0 = ev.e[0], e1 = ev.e[1], e2 = ev.e[2];
    CK(cudaEventRecord(e0, ctx->st));
    const unsigned long long n0 = la_launch_count();
    int r = do_prefill(ctx, prompt, n, s, solo_lane(ctx));
    if (r) return r;
    ctx->prefilled = true;
    CK(cudaEventRecord(e1, ctx->st));
    r = begin_request(ctx, mode, W, N, G, s, max_new);
    if (r) return r;
    r = clear_err(ctx);
    if (r) return r;
    Graph* g = nullptr;
    r = get_graph(ctx, &g);
    if (r) return r;
    const int per_step_max = (mode == MODE_LOOKAHEAD) ? N : 1;
    const long long direct = (long long)(la_launch_count() - n0);
    long long graph_runs = 0;
    LaHdr h;
    r = read_hdr(ctx, &h);
    if (r) return r;
    int guard = 0;
    while (!h.done && !h.err) {
        int remaining = max_new - h.n_out;
        int launches = std::max(1, (remaining + per_step_max - 1) / per_step_max);
        for (int i = 0; i < launches; ++i) CK(cudaGraphLaunch(g->x, ctx->st));
        graph_runs += launches;
        r = read_hdr(ctx, &h);
        if (r) return r;
        prof_collect(ctx, *g);
        if (++guard > 4 * max_new + 16) return LA_EDEVICE;
    }
    CK(cudaEventRecord(e2, ctx->st));
    if (h.err) return h.err;
    CK(cudaMemcpyAsync(out, ctx->d.out, sizeof(int32_t) * max_new, cudaMemcpyDeviceToHost, ctx->st));
    CK(cudaStreamSynchronize(ctx->st));
    *n_out = max_new;
    if (stats) {
        float ms0 = 0, ms1 = 0;
        cudaEventElapsedTime(&ms0, e0, e1);
        cudaEventElapsedTime(&ms1, e1, e2);
        memset(stats, 0, sizeof(*stats));
        stats->steps = h.n_steps;
        stats->tokens = max_new;
        stats->prefill_ns = (int64_t)(ms0 * 1e6);
        stats->decode_ns = (int64_t)(ms1 * 1e6);
        for (int i = 0; i < 16; ++i) stats->emitted_hist[i] = h.hist[i];
        stats->mean_candidates = h.n_steady ? (double)h.sum_Ct / h.n_steady : 0.0;
        stats->mean_rows = h.n_steps ? (double)h.sum_Q / h.n_steps : 0.0;
        stats->kernel_launches = direct + graph_runs * g->n_kernels;
    }
    return LA_OK;
}

int la_generate(la_ctx* ctx, const int32_t* prompt, int n, int max_new, int W, int N, int G, const la_sampling* s,
                int32_t* out, int* n_out, la_stats* stats) {
    return run_generate(ctx, MODE_LOOKAHEAD, prompt, n, max_new, W, N, G, s, out, n_out, stats);
}

int la_generate_ar(la_ctx* ctx, const int32_t* prompt, int n, int max_new, const la_sampling* s, int32_t* out,
                   int* n_out, la_stats* stats) {
    return run_generate(ctx, MODE_AR, prompt, n, max_new, 1, 3, 0, s, out, n_out, stats);
}

// One batched call of B requests as a graph: every request's pack, one
// forward and LM head over the stacked slices, every request's publication
// and commit.
static int get_batch_graph(la_ctx* ctx, int B, int sampling, Graph** out) {
    const int keep = sampling | (ctx->debug & 1);
    const int key = 0x100 | B | (sampling << 12) | ((ctx->debug & 1) << 13) | (g_tl_table ? (1 << 14) : 0);
    auto it = ctx->graphs.find(key);
    if (it != ctx->graphs.end()) {
        if (!g_tl_table || it->second.tl_epoch == g_tl_epoch) { *out = &it->second; return LA_OK; }
        drop_graph(it->second);     // captured into an earlier timeline's table
        ctx->graphs.erase(it);
    }
    tl_sync(ctx);
    const la_model_cfg& c = ctx->cfg;
    const size_t head_bytes = (size_t)c.head_dim * ctx->esz;
    Graph g;
    g.tl_epoch = g_tl_epoch;
    CK(cudaStreamBeginCapture(ctx->st, cudaStreamCaptureModeRelaxed));
    const unsigned long long n0 = la_launch_count();
    int r = LA_OK;
    for (int b = 0; b < B; ++b) la_launch_pack(ctx->req[b], ctx->st);
    const Lane ln = batch_lane(ctx, B);
    r = enqueue_forward(ctx, SEL_CALL, ln);
    if (!r) r = enqueue_head(ctx, keep, ln);
    // sampling: each request's verifier on the logits of its slice of the needed rows
    for (int b = 0; b < B && !r && sampling; ++b)
        if (la_launch_sample_verify(ctx->req[b], ctx->st, ctx->logits + (size_t)b * ctx->Qstride * c.vocab, c.vocab, 0) !=
            cudaSuccess)
            r = LA_ECUDA;
    for (int b = 0; b < B && !r; ++b)
        r = enqueue_publish_commit_req(ctx, ctx->req[b], sampling,
                                       (char*)ctx->cache + (size_t)b * ctx->cache_bytes_req,
                                       (char*)ctx->temp + (size_t)b * ctx->Qstride * head_bytes, ctx->temp_rows);
    g.n_kernels = (long long)(la_launch_count() - n0);
    la_unnote_launches((unsigned long long)g.n_kernels);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(ctx->st, &graph);
    if (r) { if (graph) cudaGraphDestroy(graph); return r; }
    CK(e);
    g.g = graph;
    CK(cudaGraphInstantiate(&g.x, graph, 0));
    ctx->graphs[key] = g;
    *out = &ctx->graphs[key];
    return LA_OK;
}

int la_generate_batch(la_ctx* ctx, int B, const int32_t* prompts, const int32_t* lengths, int max_new, int W, int N,
                      int G, const la_sampling* s, int32_t* out, la_stats* stats) {
    if (!ctx || !prompts || !lengths || !out || B < 1 || max_new < 1) return LA_EINVAL;
    if (check_sampling(s)) return LA_EINVAL;
    if (ctx->max_batch < 2) return LA_ENOTSUP;
    if (B > ctx->max_batch) return LA_ECAPACITY;
    if (N < 3 || W < 1 || G < 0) return LA_EINVAL;
    if (N > ctx->max_N || W > ctx->max_W || G > ctx->max_G) return LA_ECAPACITY;
    for (int b = 0; b < B; ++b) {
        if (lengths[b] < 1) return LA_EINVAL;
        if (lengths[b] + max_new > ctx->max_ctx) return LA_ECAPACITY;
    }
    // request 0's single-request state is reused: a later la_step needs a new prefill
    ctx->prefilled = false;
    ctx->begun = false;
    tl_sync(ctx);
    Events3 ev;
    CK(ev.create());
    cudaEvent_t e0 = ev.e[0], e1 = ev.e[1], e2 = ev.e[2];
    CK(cudaEventRecord(e0, ctx->st));
    const unsigned long long n0 = la_launch_count();
    // sampling: request b draws with seed s->seed + b
    std::vector<la_sampling> sb(B);
    for (int b = 0; b < B && s; ++b) {
        sb[b] = *s;
        sb[b].seed = s->seed + (uint64_t)b;
    }
    size_t off = 0;
    for (int b = 0; b < B; ++b) {
        int r = do_prefill(ctx, prompts + off, lengths[b], s ? &sb[b] : nullptr, prefill_lane(ctx, b));
        if (r) return r;
        off += (size_t)lengths[b];
    }
    CK(cudaEventRecord(e1, ctx->st));
    for (int b = 0; b < B; ++b)
        la_launch_begin(ctx->req[b], ctx->st, MODE_LOOKAHEAD, W, N, G, s ? 1 : 0, s ? s->temperature : 1.f,
                        s ? s->top_p : 1.f, s ? sb[b].seed : 0, max_new, (int)ctx->opts);
    CK(cudaGetLastError());
    LaHdr hb;
    memset(&hb, 0, sizeof(hb));
    hb.mode = MODE_LOOKAHEAD;
    hb.W = W; hb.N = N; hb.G = G; hb.S = N - 1;
    hb.Q = B * ctx->Qstride;
    hb.n_need = B * ctx->Qstride;
    hb.active = B;
    hb.done = (max_new <= 1);
    CK(cudaMemcpyAsync(ctx->bd.hdr, &hb, sizeof(hb), cudaMemcpyHostToDevice, ctx->st));
    if (ctx->work.counters) CK(cudaMemsetAsync(ctx->work.counters, 0, sizeof(int) * ctx->work.n_counters, ctx->st));
    const long long direct = (long long)(la_launch_count() - n0);
    long long graph_runs = 0;
    Graph* g = nullptr;
    int r = get_batch_graph(ctx, B, s ? 1 : 0, &g);
    if (r) return r;
    LaHdr h;
    CK(cudaMemcpyAsync(&h, ctx->bd.hdr, sizeof(h), cudaMemcpyDeviceToHost, ctx->st));
    CK(cudaStreamSynchronize(ctx->st));
    int guard = 0, least = 1;     // tokens of the request that has the fewest
    std::vector<LaHdr> hr(B);
    while (!h.done && !h.err) {
        // a call appends 1 .. N tokens to every live request
        const int launches = std::max(1, (max_new - least + N - 1) / N);
        for (int i = 0; i < launches; ++i) CK(cudaGraphLaunch(g->x, ctx->st));
        graph_runs += launches;
        CK(cudaMemcpyAsync(&h, ctx->bd.hdr, sizeof(h), cudaMemcpyDeviceToHost, ctx->st));
        for (int b = 0; b < B; ++b)
            CK(cudaMemcpyAsync(&hr[b], ctx->req[b].hdr, sizeof(LaHdr), cudaMemcpyDeviceToHost, ctx->st));
        CK(cudaStreamSynchronize(ctx->st));
        least = max_new;
        for (int b = 0; b < B; ++b) least = std::min(least, (int)hr[b].n_out);
        if (++guard > 4 * max_new + 16) return LA_EDEVICE;
    }
    CK(cudaEventRecord(e2, ctx->st));
    if (h.err) return h.err;
    int64_t steps = 0;
    for (int b = 0; b < B; ++b) {
        CK(cudaMemcpyAsync(&hr[b], ctx->req[b].hdr, sizeof(LaHdr), cudaMemcpyDeviceToHost, ctx->st));
        CK(cudaMemcpyAsync(out + (size_t)b * max_new, ctx->req[b].out, sizeof(int32_t) * max_new,
                           cudaMemcpyDeviceToHost, ctx->st));
    }
    CK(cudaStreamSynchronize(ctx->st));
    for (int b = 0; b < B; ++b) {
        if (hr[b].err) return hr[b].err;
        if (hr[b].n_out < max_new) return LA_EDEVICE;
        steps = std::max<int64_t>(steps, hr[b].n_steps);
    }
    if (stats) {
        float ms0 = 0, ms1 = 0;
        cudaEventElapsedTime(&ms0, e0, e1);
        cudaEventElapsedTime(&ms1, e1, e2);
        memset(stats, 0, sizeof(*stats));
        stats->steps = steps;
        stats->tokens = (int64_t)B * max_new;
        stats->prefill_ns = (int64_t)(ms0 * 1e6);
        stats->decode_ns = (int64_t)(ms1 * 1e6);
        stats->mean_rows = (double)B * ctx->Qstride;
        stats->kernel_launches = direct + graph_runs * g->n_kernels;
    }
    return LA_OK;
}

int la_debug_logits(la_ctx* ctx, float* logits, int32_t* rows, int cap_rows, int* n_rows) {
    if (!ctx || !n_rows) return LA_EINVAL;
    if (!(ctx->debug & 1)) return LA_ESTATE;
    LaHdr h;
    int r = read_hdr(ctx, &h);
    if (r) return r;
    int n = h.n_need;
    *n_rows = n;
    if (n > cap_rows) return LA_ECAPACITY;
    if (logits) CK(cudaMemcpyAsync(logits, ctx->logits, sizeof(float) * n * ctx->cfg.vocab, cudaMemcpyDeviceToHost, ctx->st));
    if (rows) CK(cudaMemcpyAsync(rows, ctx->d.need, sizeof(int32_t) * n, cudaMemcpyDeviceToHost, ctx->st));
    CK(cudaStreamSynchronize(ctx->st));
    return LA_OK;
}

int la_debug_batch_logits(la_ctx* ctx, int b, float* logits, int32_t* rows, int cap_rows, int* n_rows) {
    if (!ctx || !n_rows || b < 0) return LA_EINVAL;
    if (ctx->max_batch < 2) return LA_ENOTSUP;
    if (b >= ctx->max_batch) return LA_EINVAL;
    if (!(ctx->debug & 1)) return LA_ESTATE;
    LaHdr h;
    CK(cudaMemcpyAsync(&h, ctx->req[b].hdr, sizeof(h), cudaMemcpyDeviceToHost, ctx->st));
    CK(cudaStreamSynchronize(ctx->st));
    const int n = h.n_need;
    *n_rows = n;
    if (n > cap_rows) return LA_ECAPACITY;
    const size_t o = (size_t)b * ctx->Qstride;
    if (logits)
        CK(cudaMemcpyAsync(logits, ctx->logits + o * ctx->cfg.vocab, sizeof(float) * (size_t)n * ctx->cfg.vocab,
                           cudaMemcpyDeviceToHost, ctx->st));
    if (rows) CK(cudaMemcpyAsync(rows, ctx->req[b].need, sizeof(int32_t) * n, cudaMemcpyDeviceToHost, ctx->st));
    CK(cudaStreamSynchronize(ctx->st));
    if (rows)
        for (int i = 0; i < n; ++i) rows[i] -= (int32_t)o;
    return LA_OK;
}

static int debug_state_of(la_ctx* ctx, const LaDev& v, int32_t* hdr, int32_t* levels, int32_t* level_len,
                          int32_t* row_tok, int32_t* row_pos, int32_t* row_meta) {
    LaHdr h;
    CK(cudaMemcpyAsync(&h, v.hdr, sizeof(h), cudaMemcpyDeviceToHost, ctx->st));
    CK(cudaStreamSynchronize(ctx->st));
    if (hdr) {
        int32_t v[16] = {h.K, h.x_t, h.W, h.N, h.G, h.n_levels, h.step, h.Q, h.C_t, h.a, h.winner, h.n_out,
                         h.err, h.steady, h.n_need, h.n_deep};
        memcpy(hdr, v, sizeof(v));
    }
    if (levels) CK(cudaMemcpyAsync(levels, v.window, sizeof(int32_t) * ctx->Rmax * ctx->LMAX, cudaMemcpyDeviceToHost, ctx->st));
    if (level_len)
        for (int i = 0; i < ctx->Rmax; ++i) level_len[i] = h.level_len[i];
    if (row_tok) CK(cudaMemcpyAsync(row_tok, v.row_tok, sizeof(int32_t) * ctx->Qmax, cudaMemcpyDeviceToHost, ctx->st));
    if (row_pos) CK(cudaMemcpyAsync(row_pos, v.row_pos, sizeof(int32_t) * ctx->Qmax, cudaMemcpyDeviceToHost, ctx->st));
    if (row_meta) CK(cudaMemcpyAsync(row_meta, v.row_meta, sizeof(int32_t) * ctx->Qmax, cudaMemcpyDeviceToHost, ctx->st));
    CK(cudaStreamSynchronize(ctx->st));
    return LA_OK;
}

int la_debug_state(la_ctx* ctx, int32_t* hdr, int32_t* levels, int32_t* level_len, int32_t* row_tok, int32_t* row_pos,
                   int32_t* row_meta) {
    if (!ctx) return LA_EINVAL;
    return debug_state_of(ctx, ctx->d, hdr, levels, level_len, row_tok, row_pos, row_meta);
}

int la_debug_batch_state(la_ctx* ctx, int b, int32_t* hdr, int32_t* levels, int32_t* level_len, int32_t* row_tok,
                         int32_t* row_pos, int32_t* row_meta) {
    if (!ctx || b < 0) return LA_EINVAL;
    if (ctx->max_batch < 2) return LA_ENOTSUP;
    if (b >= ctx->max_batch) return LA_EINVAL;
    return debug_state_of(ctx, ctx->req[b], hdr, levels, level_len, row_tok, row_pos, row_meta);
}

int la_debug_pool(la_ctx* ctx, int key, int32_t* suffixes, int* count) {
    if (!ctx || !count || key < 0 || key >= ctx->cfg.vocab) return LA_EINVAL;
    int32_t cnt = 0;
    CK(cudaMemcpyAsync(&cnt, ctx->d.pool_cnt + key, sizeof(int32_t), cudaMemcpyDeviceToHost, ctx->st));
    if (suffixes)
        CK(cudaMemcpyAsync(suffixes, ctx->d.pool_tok + (size_t)key * ctx->Gmax * ctx->Smax,
                           sizeof(int32_t) * ctx->Gmax * ctx->Smax, cudaMemcpyDeviceToHost, ctx->st));
    CK(cudaStreamSynchronize(ctx->st));
    *count = cnt;
    return LA_OK;
}

int la_debug_sample_verify(const float* logits, int rows, int V, const int32_t* cand, int Ct, int S,
                           const la_sampling* s, int n_trials, int32_t* out) {
    if (!logits || !s || !out || rows < 1 || V < 2 || Ct < 0 || Ct > LA_MAX_G || S < 1 || S > 15 || n_trials < 1)
        return LA_EINVAL;
    if (check_sampling(s)) return LA_EINVAL;
    if (Ct > 0 && !cand) return LA_EINVAL;
    if (rows < 1 + Ct * S) return LA_EINVAL;
    if ((size_t)V * sizeof(float) > 200 * 1024) return LA_ENOTSUP;
    for (int i = 0; i < Ct * S; ++i)
        if (cand[i] < 0 || cand[i] >= V) return LA_EINVAL;
    float* dl = nullptr;
    int32_t *dc = nullptr, *dout = nullptr;
    int rc = LA_OK;
    const size_t out_n = (size_t)n_trials * (S + 3);
    if (cudaMalloc(&dl, sizeof(float) * (size_t)rows * V) != cudaSuccess ||
        cudaMalloc(&dc, sizeof(int32_t) * (size_t)std::max(1, Ct * S)) != cudaSuccess ||
        cudaMalloc(&dout, sizeof(int32_t) * out_n) != cudaSuccess) {
        rc = LA_ECUDA;
    }
    if (!rc && cudaMemcpy(dl, logits, sizeof(float) * (size_t)rows * V, cudaMemcpyHostToDevice) != cudaSuccess) rc = LA_ECUDA;
    if (!rc && Ct > 0 && cudaMemcpy(dc, cand, sizeof(int32_t) * Ct * S, cudaMemcpyHostToDevice) != cudaSuccess) rc = LA_ECUDA;
    if (!rc && la_launch_sample_trials(0, dl, V, dc, Ct, S, s->temperature, s->top_p, s->seed, n_trials, dout) != cudaSuccess)
        rc = LA_ECUDA;
    if (!rc && cudaMemcpy(out, dout, sizeof(int32_t) * out_n, cudaMemcpyDeviceToHost) != cudaSuccess) rc = LA_ECUDA;
    cudaFree(dl);
    cudaFree(dc);
    cudaFree(dout);
    return rc;
}

int la_debug_gemm(int mode, const uint16_t* w, const uint16_t* w2, int n_seg, int n_out, int K, const uint16_t* x,
                  int rows, int n_cta, float* y) {
    const int pair = (mode & LA_GEMM_PAIR) ? 1 : 0;
    mode &= ~LA_GEMM_PAIR;
    if (!w || !x || !y || mode < GEMM_STORE || mode > GEMM_LOGITS || n_seg < 1 || n_seg > 3 || n_out < 128 ||
        n_out % (128 * n_seg) || K < 64 || K % 64 || rows < 1 || rows > 1024 || n_cta < 0 || n_cta > 4096)
        return LA_EINVAL;
    if (pair && (mode == GEMM_SWIGLU || (n_out / n_seg) % 256)) return LA_EINVAL;
    if (n_cta == 0) n_cta = la_tc_ctas();
    const int max_seg = la_tc_max_segments(n_out / 128 / (pair ? 2 : 1), la_tc_k_units(mode, K, pair), n_cta);
    if (mode == GEMM_SWIGLU && (!w2 || n_seg != 1)) return LA_EINVAL;
    if (mode == GEMM_LOGITS && n_seg != 1) return LA_EINVAL;
    const int rows_cap = ((rows + 255) / 256) * 256;
    const int n_seg_out = n_out / n_seg;
    void* dw[3] = {nullptr, nullptr, nullptr};
    void *dw2 = nullptr, *dx = nullptr, *dout = nullptr;
    float *ws = nullptr, *pv = nullptr;
    int *cnt = nullptr, *pi = nullptr;
    LaHdr* hdr = nullptr;
    int rc = LA_OK;
    const int tiles = n_out / 128, qchunks = rows_cap / 256;
    auto M = [&](void** p, size_t b) { if (!rc && cudaMalloc(p, b) != cudaSuccess) rc = LA_ECUDA; };
    for (int sgi = 0; sgi < n_seg; ++sgi) M(&dw[sgi], (size_t)n_seg_out * K * 2);
    if (mode == GEMM_SWIGLU) M(&dw2, (size_t)n_out * K * 2);
    M(&dx, (size_t)rows_cap * K * 2);
    M(&dout, (size_t)rows_cap * n_out * 4);
    M((void**)&ws, (size_t)tiles * qchunks * max_seg * 2 * 256 * 128 * 4);
    M((void**)&cnt, (size_t)LA_TC_CTR_PER_TILE * tiles * qchunks * 4);
    M((void**)&pv, (size_t)tiles * rows_cap * 4);
    M((void**)&pi, (size_t)tiles * rows_cap * 4);
    M((void**)&hdr, sizeof(LaHdr));
    const bool f32out = (mode == GEMM_RESID || mode == GEMM_LOGITS);
    if (!rc) {
        LaHdr h;
        memset(&h, 0, sizeof(h));
        h.n_need = rows;
        bool ok = cudaMemcpy(hdr, &h, sizeof(h), cudaMemcpyHostToDevice) == cudaSuccess;
        for (int sgi = 0; sgi < n_seg; ++sgi)
            ok = ok && cudaMemcpy(dw[sgi], w + (size_t)sgi * n_seg_out * K, (size_t)n_seg_out * K * 2,
                                  cudaMemcpyHostToDevice) == cudaSuccess;
        if (dw2) ok = ok && cudaMemcpy(dw2, w2, (size_t)n_out * K * 2, cudaMemcpyHostToDevice) == cudaSuccess;
        ok = ok && cudaMemset(dx, 0, (size_t)rows_cap * K * 2) == cudaSuccess;
        ok = ok && cudaMemcpy(dx, x, (size_t)rows * K * 2, cudaMemcpyHostToDevice) == cudaSuccess;
        ok = ok && cudaMemset(cnt, 0, (size_t)LA_TC_CTR_PER_TILE * tiles * qchunks * 4) == cudaSuccess;
        ok = ok && cudaMemset(dout, 0, (size_t)rows_cap * n_out * 4) == cudaSuccess;
        if (mode == GEMM_RESID) ok = ok && cudaMemcpy(dout, y, (size_t)rows * n_out * 4, cudaMemcpyHostToDevice) == cudaSuccess;
        if (!ok) rc = LA_ECUDA;
    }
    if (!rc) {
        TcGemm g;
        memset(&g, 0, sizeof(g));
        if (la_tc_make_map(&g.tmA, dw[0], n_seg_out, K, 128) ||
            la_tc_make_map(&g.tmA2, mode == GEMM_SWIGLU ? dw2 : (n_seg > 1 ? dw[1] : dw[0]), n_seg_out, K, 128) ||
            la_tc_make_map(&g.tmA3, n_seg > 2 ? dw[2] : dw[0], n_seg_out, K, 128) ||
            la_tc_make_act_maps(&g, dx, rows_cap, K))
            rc = LA_ECUDA;
        g.mode = mode;
        g.K = K;
        g.Nout = n_out;
        g.seg_tiles = n_seg > 1 ? n_seg_out / 128 : 0;
        g.pair = pair;
        g.n_cta = n_cta;
        g.max_seg = max_seg;
        g.rows_cap = rows_cap;
        g.out = dout;
        g.ldo = n_out;
        g.logits = mode == GEMM_LOGITS ? (float*)dout : nullptr;
        g.ld_logits = n_out;
        TcWork wk;
        memset(&wk, 0, sizeof(wk));
        wk.ws = ws;
        wk.counters = cnt;
        wk.part_v = pv;
        wk.part_i = pi;
        wk.part_stride = rows_cap;
        LaDev d{};
        memset(&d, 0, sizeof(d));
        d.hdr = hdr;
        // the weights as the model's GEMMs read them: unit-contiguous images
        void* wp = nullptr;
        if (!rc && cudaMalloc(&wp, la_tc_packed_bytes(g)) != cudaSuccess) rc = LA_ECUDA;
        if (!rc && la_tc_pack(g, dw[0], mode == GEMM_SWIGLU ? dw2 : dw[1], dw[2], wp, 0) != cudaSuccess) rc = LA_ECUDA;
        g.wpack = wp;
        if (!rc && la_launch_gemm_tc(d, 0, g, wk, SEL_NEED, rows) != cudaSuccess) rc = LA_ECUDA;
        if (!rc && cudaDeviceSynchronize() != cudaSuccess) rc = LA_ECUDA;
        if (wp) cudaFree(wp);
        LaHdr h;
        if (!rc && cudaMemcpy(&h, hdr, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) rc = LA_ECUDA;
        if (!rc && h.err) rc = h.err;
        if (!rc) {
            if (f32out) {
                if (cudaMemcpy(y, dout, (size_t)rows * n_out * 4, cudaMemcpyDeviceToHost) != cudaSuccess) rc = LA_ECUDA;
            } else {
                std::vector<uint16_t> tmpb((size_t)rows * n_out);
                if (cudaMemcpy(tmpb.data(), dout, tmpb.size() * 2, cudaMemcpyDeviceToHost) != cudaSuccess) rc = LA_ECUDA;
                for (size_t i = 0; i < tmpb.size() && !rc; ++i) {
                    uint32_t u = (uint32_t)tmpb[i] << 16;
                    memcpy(&y[i], &u, 4);
                }
            }
        }
    }
    for (int sgi = 0; sgi < 3; ++sgi) cudaFree(dw[sgi]);
    cudaFree(dw2); cudaFree(dx); cudaFree(dout); cudaFree(ws); cudaFree(cnt); cudaFree(pv); cudaFree(pi); cudaFree(hdr);
    return rc;
}

// fills a bf16 buffer with small deterministic values (timing inputs)
__global__ void k_fill_bf16(__nv_bfloat16* p, size_t n, uint32_t seed) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        uint32_t h = (uint32_t)i * 2654435761u ^ seed;
        h ^= h >> 15;
        h *= 2246822519u;
        h ^= h >> 13;
        p[i] = __float2bfloat16_rn(((float)(h & 0xffff) / 65536.0f - 0.5f) * 0.04f);
    }
}

int la_bench_gemm(int mode, int n_out, int K, int rows, int n_cta, int n_copies, int reps, int packed, float* us) {
    if (!us || mode < GEMM_STORE || mode > GEMM_LOGITS || n_out < 128 || n_out % 128 || K < 64 || K % 64 ||
        rows < 1 || rows > 1024 || n_cta < 0 || n_copies < 1 || n_copies > 64 || reps < 1 || packed < 0 || packed > 1)
        return LA_EINVAL;
    if (n_cta == 0) n_cta = la_tc_ctas();
    const int max_seg = la_tc_max_segments(n_out / 128, la_tc_k_units(mode, K), n_cta);
    const int rows_cap = ((rows + 255) / 256) * 256;
    const int tiles = n_out / 128, qchunks = rows_cap / 256;
    const int nA = mode == GEMM_SWIGLU ? 2 : 1;
    std::vector<void*> w(n_copies * nA, nullptr);
    void *dx = nullptr, *dout = nullptr;
    float *ws = nullptr, *pv = nullptr;
    int *cnt = nullptr, *pi = nullptr;
    LaHdr* hdr = nullptr;
    int rc = LA_OK;
    auto M = [&](void** p, size_t b) { if (!rc && cudaMalloc(p, b) != cudaSuccess) rc = LA_ECUDA; };
    for (auto& p : w) M(&p, (size_t)n_out * K * 2);
    M(&dx, (size_t)rows_cap * K * 2);
    M(&dout, (size_t)rows_cap * n_out * 4);
    M((void**)&ws, (size_t)tiles * qchunks * max_seg * 2 * 256 * 128 * 4);
    M((void**)&cnt, (size_t)LA_TC_CTR_PER_TILE * tiles * qchunks * 4);
    M((void**)&pv, (size_t)tiles * rows_cap * 4);
    M((void**)&pi, (size_t)tiles * rows_cap * 4);
    M((void**)&hdr, sizeof(LaHdr));
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (!rc) {
        for (size_t i = 0; i < w.size(); ++i) k_fill_bf16<<<512, 256>>>((__nv_bfloat16*)w[i], (size_t)n_out * K, 17u + (uint32_t)i);
        k_fill_bf16<<<512, 256>>>((__nv_bfloat16*)dx, (size_t)rows_cap * K, 99u);
        LaHdr h;
        memset(&h, 0, sizeof(h));
        h.n_need = rows;
        if (cudaMemcpy(hdr, &h, sizeof(h), cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemset(cnt, 0, (size_t)LA_TC_CTR_PER_TILE * tiles * qchunks * 4) != cudaSuccess || cudaMemset(dout, 0, (size_t)rows_cap * n_out * 4))
            rc = LA_ECUDA;
        if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) rc = LA_ECUDA;
    }
    std::vector<TcGemm> gs(n_copies);
    for (int i = 0; i < n_copies && !rc; ++i) {
        TcGemm& g = gs[i];
        memset(&g, 0, sizeof(g));
        void* a1 = w[i * nA];
        void* a2 = nA == 2 ? w[i * nA + 1] : a1;
        if (la_tc_make_map(&g.tmA, a1, n_out, K, 128) || la_tc_make_map(&g.tmA2, a2, n_out, K, 128) ||
            la_tc_make_map(&g.tmA3, a1, n_out, K, 128) || la_tc_make_act_maps(&g, dx, rows_cap, K))
            rc = LA_ECUDA;
        g.mode = mode; g.K = K; g.Nout = n_out; g.n_cta = n_cta; g.max_seg = max_seg; g.rows_cap = rows_cap;
        g.out = dout; g.ldo = n_out; g.logits = nullptr; g.ld_logits = n_out;
    }
    std::vector<void*> wp(n_copies, nullptr);
    for (int i = 0; i < n_copies && !rc && packed; ++i) {
        if (cudaMalloc(&wp[i], la_tc_packed_bytes(gs[i])) != cudaSuccess ||
            la_tc_pack(gs[i], w[i * nA], nA == 2 ? w[i * nA + 1] : nullptr, nullptr, wp[i], 0) != cudaSuccess)
            rc = LA_ECUDA;
        gs[i].wpack = wp[i];
    }
    TcWork wk;
    memset(&wk, 0, sizeof(wk));
    wk.ws = ws; wk.counters = cnt; wk.part_v = pv; wk.part_i = pi; wk.part_stride = rows_cap;
    LaDev d{};
    memset(&d, 0, sizeof(d));
    d.hdr = hdr;
    if (!rc) {
        for (int i = 0; i < 3 && !rc; ++i)
            if (la_launch_gemm_tc(d, 0, gs[i % n_copies], wk, SEL_NEED, rows) != cudaSuccess) rc = LA_ECUDA;
        if (!rc && cudaEventRecord(e0, 0) != cudaSuccess) rc = LA_ECUDA;
        for (int i = 0; i < reps && !rc; ++i)
            if (la_launch_gemm_tc(d, 0, gs[i % n_copies], wk, SEL_NEED, rows) != cudaSuccess) rc = LA_ECUDA;
        if (!rc && cudaEventRecord(e1, 0) != cudaSuccess) rc = LA_ECUDA;
        if (!rc && cudaEventSynchronize(e1) != cudaSuccess) rc = LA_ECUDA;
        float ms = 0;
        if (!rc) cudaEventElapsedTime(&ms, e0, e1);
        *us = ms * 1000.0f / reps;
        LaHdr h;
        if (!rc && cudaMemcpy(&h, hdr, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) rc = LA_ECUDA;
        if (!rc && h.err) rc = h.err;
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    for (auto p : wp) if (p) cudaFree(p);
    for (auto p : w) cudaFree(p);
    cudaFree(dx); cudaFree(dout); cudaFree(ws); cudaFree(cnt); cudaFree(pv); cudaFree(pi); cudaFree(hdr);
    return rc;
}

}  // extern "C"
