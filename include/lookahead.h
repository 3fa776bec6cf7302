/*
 * liblookahead — C ABI of the packed per-step target call of Lookahead decoding
 * on one GB300 (sm_103a).
 *
 * The method (Fu, Bailis, Stoica, Zhang, "Break the Sequential Dependency of
 * LLM Inference Using Lookahead Decoding", §3; "M7.3 – Lookahead Decoding",
 * §0x03–§0x07): every call runs one unchanged causal decoder over
 *   - the ordinary row (the last committed token x_t),
 *   - a lookahead branch: W window columns over N-1 Jacobi trajectory levels,
 *   - a verification branch: up to G candidate suffixes of N-1 tokens looked up
 *     in an n-gram pool under the key x_t,
 * packed into one batch of rows with a branch-structured attention mask; the
 * outputs feed a verifier (greedy, or exact sampling over disjoint one-hot
 * proposals), the n-gram pool update, the K/V commit and the window shift.
 *
 * Conventions for every entry point
 *   - Return value: LA_OK (0) or one of the LA_E* codes below.  la_strerror()
 *     names it.  Every call is fail-closed (M7.3 §0x07 "publication order
 *     should be fail-closed"): on any error no token is appended and the
 *     committed K/V length, the window and the pool keep their previous
 *     contents.
 *   - "host" pointers are ordinary CPU memory owned by the caller; the
 *     library copies from/into them before returning.  "device" pointers are
 *     CUDA global memory on the context's device, owned by the caller and
 *     borrowed for the lifetime of the context (weights).
 *   - All GPU work is enqueued on the CUDA stream given to la_init.  Calls
 *     that return host results (la_prefill, la_step, la_generate*,
 *     la_debug_*) synchronise that stream before returning.
 *   - A context is not thread-safe; use one context per thread.
 */
#ifndef LOOKAHEAD_H
#define LOOKAHEAD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define LA_OK        0
#define LA_EINVAL    1  /* bad argument: null pointer, N < 3, W < 1, G < 0, id out of range */
#define LA_ECAPACITY 2  /* exceeds a size fixed at la_init (context length, W, N, G, prompt) */
#define LA_ESTATE    3  /* call out of order: step before prefill, W/N/G changed without re-prefill */
#define LA_ECUDA     4  /* a CUDA runtime/driver call failed (details: la_last_cuda_error) */
#define LA_EDEVICE   5  /* a kernel set the device error word (bounds or invariant check) */
#define LA_ETIMEOUT  6  /* a bounded device wait ran out; the step's results were discarded */
#define LA_ENOTSUP   7  /* configuration not supported by this build (dtype, head_dim, ...) */

/* ---- element types ------------------------------------------------------- */
#define LA_F32  0       /* fp32 weights, activations and K/V */
#define LA_BF16 1       /* bf16 weights, activations and K/V; fp32 accumulation */

typedef struct la_ctx la_ctx;

/* Decoder-only Llama-style model: RMSNorm, RoPE (rotate-half, theta), SwiGLU
 * MLP, multi-head attention with n_kv_heads == n_heads, untied LM head, no
 * biases.  head_dim must be 32 or 128; d_model == n_heads * head_dim. */
typedef struct {
    int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, d_ffn, vocab;
    float   rms_eps;     /* e.g. 1e-5 */
    float   rope_theta;  /* e.g. 10000 */
    int32_t dtype;       /* LA_F32 or LA_BF16 */
} la_model_cfg;

/* Device pointers to the weights, row-major, element type cfg.dtype.
 *   tok_emb [vocab][d_model]   lm_head [vocab][d_model]   final_norm [d_model]
 * Per layer l (host arrays of n_layers device pointers):
 *   attn_norm[l], mlp_norm[l]  [d_model]
 *   wq[l], wk[l], wv[l]        [n_heads*head_dim][d_model]
 *   wo[l]                      [d_model][n_heads*head_dim]
 *   w_gate[l], w_up[l]         [d_ffn][d_model]
 *   w_down[l]                  [d_model][d_ffn]
 * Every matrix must be 16-byte aligned.  The caller keeps them alive and
 * unchanged until la_free.  The host pointer arrays are copied by la_init.
 * In bf16 mode la_init also copies every projection and the LM head into
 * context-owned device memory (the same size again) in the order the
 * tensor-core GEMM streams them: each 128 x 64 tile contiguous, already in
 * its shared-memory layout. */
typedef struct {
    const void* tok_emb;
    const void* lm_head;
    const void* final_norm;
    const void* const* attn_norm;
    const void* const* wq;
    const void* const* wk;
    const void* const* wv;
    const void* const* wo;
    const void* const* mlp_norm;
    const void* const* w_gate;
    const void* const* w_up;
    const void* const* w_down;
} la_weights;

/* Sampling policy (break the sequential dependency §2, §3.2; M7.3 §0x05B):
 * target p = softmax(logits / temperature) restricted to the top-p nucleus
 * (probability descending, ties by lower id, the crossing token kept),
 * renormalised.  Uniforms come from Philox4x32-10 keyed by seed with the
 * counter (step, offset, test, purpose).  Pass NULL for greedy decoding. */
typedef struct {
    float    temperature;  /* > 0 */
    float    top_p;        /* (0, 1] */
    uint64_t seed;
} la_sampling;

/* Pool seeding options (la_set_options), off by default.  Both feed the
 * same keyed LRU n-gram pool as the trajectory n-grams (M7.3 §0x03A
 * POOL_FROM_PROMPT, §0x06A generated-prefix insertion; break the sequential
 * dependency §5, prompt lookup).  The token sequence is the prompt followed
 * by every output token; the n-gram ending at sequence position k is keyed by
 * token k-(N-1) with suffix tokens k-(N-1)+1 .. k, upserted in increasing k.
 *   LA_OPT_POOL_FROM_PROMPT  every n-gram inside the prompt, when a request
 *                            starts
 *   LA_OPT_POOL_FROM_OUTPUT  the n-gram ending at each output token as it is
 *                            appended (the first token when the request
 *                            starts, after the prompt's n-grams; a call's
 *                            tokens after the call's trajectory n-grams)
 * Outputs are unchanged (greedy: still the AR tokens); only which candidates
 * are verified changes. */
#define LA_OPT_POOL_FROM_PROMPT 1u
#define LA_OPT_POOL_FROM_OUTPUT 2u

/* Window schedule option (la_set_options), off by default: ALWAYS_FWD_ONE=False
 * (M7.3 §0x03C, the alternative to the pinned one-column advance; §0x06,
 * sequence axis).  After a steady call that accepted a > 0 candidate tokens,
 * every level of the advanced window [u1[1:], u2, ..., z] also drops its first
 * a cells, the rest move left, and the vacated tail cells (level 0 first, each
 * level in column order) take the next tokens of the prompt cycle that seeded
 * level 0: refill cell c (counted from the request start) is
 * prompt[(W+N-3+c) mod prompt_len].  Level sizes stay [W-1, W, ..., W].
 * Outputs are unchanged (greedy: still the AR tokens); only the proposals
 * change. */
#define LA_OPT_SLICE_WINDOW 4u

/* Counters of the last la_generate / la_generate_ar call. */
typedef struct {
    int64_t steps;              /* packed target calls after the prefill */
    int64_t tokens;             /* tokens returned (including the prefill's) */
    int64_t prefill_ns;         /* device time of the prefill */
    int64_t decode_ns;          /* device time of all steps */
    int32_t emitted_hist[16];   /* calls that emitted 1, 2, ... tokens (E_t = a+1) */
    double  mean_candidates;    /* mean C_t over steady calls */
    double  mean_rows;          /* mean Q over calls */
    int64_t kernel_launches;    /* kernels of this library the call enqueued (a graph
                                   execution counts every kernel node it runs) */
} la_stats;

/* Create a context on the current CUDA device.
 * Defines the inputs of the method (break the sequential dependency, App. A,
 * the lookahead decoding algorithm: a model, the n-gram size N, the window
 * size W, the speculation limit G) and the state it keeps across calls
 * (M7.3 §0x07: the stable K/V prefix, the ordinary frontier and the packed
 * workspace of temporary rows; §0x03B: the keyed n-gram pool; §0x01A: the
 * window, pool and backend manifest fixed for a round).
 *   cfg, w        : model (see above); weights are borrowed device memory.
 *   max_ctx       : largest committed length (prompt + generated tokens).
 *   max_W, max_N, max_G : largest lookahead knobs any later call may use
 *                   (max_N >= 3, max_W >= 1, max_G >= 0); they size the
 *                   row buffers: Q <= (max_W + max_G) * (max_N - 1) + max_N.
 *   stream        : cudaStream_t to enqueue on (NULL: the context creates and
 *                   owns a non-blocking stream).
 *   out           : receives the context.
 * Allocates the K/V cache, the call's temporary K/V rows, the n-gram pool
 * ([vocab][max_G][max_N-1] ids), the window, the activations and scratch
 * with cudaMalloc.  la_init first waits for all work already issued on the
 * device, so weights still being written by another stream are complete
 * before any kernel of the context reads them; later writes to the weights
 * must be ordered before the context's calls by the caller.
 * Errors: LA_EINVAL, LA_ENOTSUP, LA_ECUDA. */
int la_init(const la_model_cfg* cfg, const la_weights* w, int max_ctx,
            int max_W, int max_N, int max_G, void* stream, la_ctx** out);

/* Pool seeding and window options (LA_OPT_* bits) for the requests that start after
 * this call (la_generate, or the first la_step after la_prefill).  Unknown
 * bits: LA_EINVAL.  Host-only; does not synchronise. */
int la_set_options(la_ctx* ctx, uint32_t flags);

/* Prefill the prompt (host ids, n >= 1, each in [0, vocab)) with one causal
 * forward; resets the K/V cache, the window, the pool and the step counter.
 * This is the state before the first target call of M7.3 §0x03A (window and
 * pool lifecycle) and §0x06B: the committed K/V covers the prompt and the
 * first output token is one ahead of it, to be the next call's ordinary
 * input.
 * *first_token (host) receives the first generated token (argmax of the last
 * prompt row, or a draw from it when `s` is not NULL).  Errors: LA_EINVAL,
 * LA_ECAPACITY (n > max_ctx - 1), LA_ECUDA, LA_EDEVICE. */
int la_prefill(la_ctx* ctx, const int32_t* prompt, int n, const la_sampling* s,
               int32_t* first_token);

/* One packed target call (M7.3 §0x03A steady-state lifecycle, steps 1-8):
 * lookup, pack, forward, verify, K/V commit, pool update, window shift.
 * The first call after la_prefill fixes W, N, G (1 <= W <= max_W,
 * 3 <= N <= max_N, 0 <= G <= max_G) and seeds window level 0 with
 * W+N-3 prompt tokens (cyclically); the first N-2 calls are warm-up fills
 * without a verification branch.  Later calls must pass the same W, N, G
 * (LA_ESTATE otherwise).  out (host, capacity >= N) receives the emitted
 * tokens, *n_out their number (1..N). */
int la_step(la_ctx* ctx, int W, int N, int G, const la_sampling* s,
            int32_t* out, int* n_out);

/* The whole decoding loop of M7.3 §0x06 (loop pseudocode; break the
 * sequential dependency §3 and App. A, the lookahead decoding algorithm with
 * prompt, model, N, W, G and a step limit): la_prefill, then the
 * warm-up fills and steady calls of la_step (M7.3 §0x03A, steps 1-8, each
 * published fail-closed, §0x06A, §0x07) until max_new tokens.
 * Prefill + lookahead steps until max_new tokens (the prefill's token
 * included) have been produced; out (host, capacity >= max_new) receives
 * exactly max_new tokens (*n_out = max_new).  Steps run as captured CUDA
 * graphs without host synchronisation between them.  stats may be NULL. */
int la_generate(la_ctx* ctx, const int32_t* prompt, int n, int max_new,
                int W, int N, int G, const la_sampling* s,
                int32_t* out, int* n_out, la_stats* stats);

/* The same as la_generate but with plain autoregressive decoding (one row
 * per call) on the same kernels: the baseline the method must equal
 * (greedy) and beat.  M7.3 §0x02A: greedy Jacobi iteration reaches the
 * autoregressive greedy fixed point, so lookahead output must equal this
 * call's output token for token; break the sequential dependency §1 and §5
 * measure speedup against this decoding; §3.3 and App. B make sampled
 * lookahead output follow this call's sampling distribution. */
int la_generate_ar(la_ctx* ctx, const int32_t* prompt, int n, int max_new,
                   const la_sampling* s, int32_t* out, int* n_out, la_stats* stats);

/* ---- several requests in one packed call ---------------------------------- */

/* As la_init, for contexts that also run batched calls of up to max_batch
 * requests (bf16 models; max_batch x the largest call's rows rounded up to
 * 16 must not exceed 1024).  Requests 1 .. max_batch-1 get their own
 * header, window, pool, prompt, out ring and K/V cache (max_batch x the
 * single-request cache).  la_init(...) is la_init_batch(..., 1, ...).
 * Errors: those of la_init; LA_ENOTSUP for max_batch > 1 with fp32 weights
 * or too many rows. */
int la_init_batch(const la_model_cfg* cfg, const la_weights* w, int max_ctx,
                  int max_W, int max_N, int max_G, int max_batch, void* stream,
                  la_ctx** out);

/* Lookahead decoding of B prompts together (M7.3 runs one request
 * per call in its pinned code, §0x04C, and calls that a property of the
 * code; the state is per request, §0x03B, §0x07).  prompts (host) holds the
 * B prompts back to back, lengths[b] (host) their lengths.  Each packed call
 * stacks every live request's rows (request b at rows b*Qs .. , Qs the
 * largest call's rows rounded up to 16; unused rows of a slice repeat the
 * request's ordinary row), runs one forward and LM head over them (one
 * weight stream for all requests), then verifies, publishes and advances
 * each request on its own; a request with max_new tokens leaves the batch.
 * Every request's rows see only its own cache and rows, so each output is
 * that request's la_generate output (greedy: its AR output).  s: NULL for
 * greedy, else every request samples with s's temperature and top-p and
 * request b with seed s->seed + b (its la_generate output with that seed).
 * out (host, B x max_new) gets
 * request b's tokens at out[b*max_new ..].  stats: steps = calls of the
 * request that needed most, tokens = B*max_new.
 * Errors: LA_EINVAL, LA_ECAPACITY (B > max_batch, a prompt + max_new >
 * max_ctx, knobs above the context's), LA_ENOTSUP (a context from la_init),
 * LA_ECUDA, device errors.  Resets request 0's single-request state: a
 * later la_step needs la_prefill first. */
int la_generate_batch(la_ctx* ctx, int B, const int32_t* prompts, const int32_t* lengths,
                      int max_new, int W, int N, int G, const la_sampling* s, int32_t* out,
                      la_stats* stats);

/* fp32 logits [*n_rows][vocab] of request b's needed rows in the last
 * batched call (la_set_debug bit 0 set before la_generate_batch) and their
 * packed row indices within the request's own rows.  A request that left the
 * batch before the last call keeps no logits of that call.  Errors:
 * LA_EINVAL, LA_ENOTSUP (a context from la_init), LA_ESTATE (bit 0 off),
 * LA_ECAPACITY (cap_rows < *n_rows), LA_ECUDA. */
int la_debug_batch_logits(la_ctx* ctx, int b, float* logits, int32_t* rows, int cap_rows, int* n_rows);

/* la_debug_state for request b of a batched context after the last batched
 * call: its header, window and its own packed rows (packed indices within
 * the request).  Errors: LA_EINVAL, LA_ENOTSUP (a context from la_init),
 * LA_ECUDA. */
int la_debug_batch_state(la_ctx* ctx, int b, int32_t* hdr, int32_t* levels, int32_t* level_len, int32_t* row_tok,
                         int32_t* row_pos, int32_t* row_meta);

/* ---- inspection (tests) -------------------------------------------------- */

/* flags bit 0: keep fp32 logits of the rows whose outputs the verifier reads
 * (the ordinary row, the deepest trajectory level, every verification row)
 * for la_debug_logits.
 * flags bit 2: kernel timing.  The step graph (a separate graph, captured on
 * first use) brackets every launch with a CUDA event pair on the context's
 * stream; at each host synchronisation la_generate adds the durations of the
 * last executed step to per-kind totals read by la_profile_read.  The event
 * records add a little time to every step: time whole steps with it off. */
int la_set_debug(la_ctx* ctx, int flags);

/* flags bit 3: keep, for la_debug_layer, every layer's values at the points
 * where the decoder stores them (the first call with it allocates them:
 * (n_layers+1) x rows x d_model floats and n_layers x rows x (HD + d_model +
 * d_ffn) elements of the model dtype).  Unknown bits: LA_EINVAL. */

/* Rows [0, rows) of the last pass (prefill chunk or packed call) of decoder
 * layer `layer`, at one of its storage points (host buffer of rows x width):
 *   what 0  the fp32 residual at the layer's input (width d_model); layer ==
 *           n_layers: the final residual before the final RMSNorm, complete
 *           only on the rows whose logits the call reads
 *   what 1  the attention output (width n_heads*head_dim, model dtype)
 *   what 2  the RMSNorm output that enters the gate/up projection (width
 *           d_model, model dtype)
 *   what 3  the SwiGLU output that enters the down projection (width d_ffn,
 *           model dtype)
 * Every packed row runs through the same decoder (break the sequential
 * dependency §2; M7.3 §0x04); tests feed these values to the oracle stage by
 * stage.  Requires la_set_debug bit 3 before the pass.  Errors: LA_EINVAL,
 * LA_ESTATE (bit 3 off), LA_ECAPACITY (rows above the row buffers), LA_ECUDA. */
int la_debug_layer(la_ctx* ctx, int layer, int what, void* host, int rows);

/* Per-kind kernel-timing totals since the last read (then reset):
 *   ms4[k], launches4[k] (host, 4 entries each): k = 0 tensor-core GEMMs,
 *   1 attention (block and combine kernels, timed together per layer),
 *   2 row-wise kernels (embedding, RMSNorm, RoPE), 3 state kernels (pack,
 *   argmax reduction, sampling verifier, publish, K/V commit);
 *   *samples (host, may be NULL): steps the totals cover.
 * Errors: LA_EINVAL. */
int la_profile_read(la_ctx* ctx, double* ms4, int64_t* launches4, int64_t* samples);

/* Kernel timeline (process-wide; every context's kernels are recorded).
 * la_timeline_start opens a table for up to max_ctas CTA records (32 bytes
 * each, device memory the library owns until la_timeline_stop); from then on
 * every CTA of every library kernel records its start and end on the GPU's
 * global nanosecond timer, the kernel's id, its linear CTA index and the
 * grid's CTA count.  Ids: 0 tensor-core GEMM, 1 CUDA-core GEMM, 2 fused
 * attention, 3 CUDA-core attention, 4 embedding, 5 RMSNorm, 6 and 7 RoPE,
 * 8 SwiGLU, 9 and 10 argmax, 11 sampling verifier, 12 request begin, 13 pack,
 * 14 pool seeding, 15 publish, 16 K/V commit, 17 injected outputs,
 * 18-20 prefill rows / needed row / finish, 21 layer chain.  The call
 * synchronises the device before and after.
 * la_timeline_stop synchronises, closes the table and writes up to cap
 * records to rec (host, 5 int64 each: start ns, end ns, id, CTA, CTAs of the
 * grid), ordered by start; *n (host) = CTAs that took a record, also when
 * above max_ctas or cap (the records beyond are lost).
 * Charging every instant of the device time to the running CTA that
 * finishes next splits the time of a call into kernels on its critical path
 * and adds up to that time.
 * Errors: LA_EINVAL (max_ctas < 1, null n, a second start), LA_ESTATE
 * (stop without start), LA_ECUDA. */
int la_timeline_start(int64_t max_ctas);
int la_timeline_stop(int64_t* rec, int64_t cap, int64_t* n);

/* fp32 logits [*n_rows][vocab] of the last call's needed rows and their
 * packed row indices.  host buffers of capacity cap_rows rows.
 * The needed rows are those whose outputs the step reads (M7.3 §0x04A row
 * compiler output slices; §0x05C row ledger): the ordinary row, the deepest
 * trajectory level's rows (the new n-gram ends) and every verification row.
 * Requires la_set_debug bit 0 before the call; *n_rows is set even when
 * the buffers are too small.  Errors: LA_EINVAL (null ctx or n_rows),
 * LA_ESTATE (debug bit 0 off), LA_ECAPACITY (cap_rows < *n_rows), LA_ECUDA. */
int la_debug_logits(la_ctx* ctx, float* logits, int32_t* rows, int cap_rows, int* n_rows);

/* Snapshot of the request state after the last call (host buffers):
 *   hdr[16]        : K (committed length), x_t, W, N, G, n_levels, step,
 *                    Q, C_t, a, winner, n_out, err, steady, n_need, n_deep
 *   levels         : [max_N-1][max_W+max_N-3] window ids, level_len[max_N-1]
 *   row_tok/pos/meta : [Qmax] ids, logical positions and metadata of the
 *                    last packed call (meta = role | level<<2 | column<<8 |
 *                    candidate<<16 | offset<<24; role 0 ordinary,
 *                    1 lookahead, 2 verify)
 * Any pointer may be NULL. */
int la_debug_state(la_ctx* ctx, int32_t* hdr, int32_t* levels, int32_t* level_len,
                   int32_t* row_tok, int32_t* row_pos, int32_t* row_meta);

/* The pool bucket of `key`: up to max_G suffixes of N-1 ids, oldest first
 * (host buffer [max_G][max_N-1]); *count receives the bucket size. */
int la_debug_pool(la_ctx* ctx, int key, int32_t* suffixes, int* count);

/* One call of the state machine with the model forward replaced by given
 * per-row outputs (host): argmax[q] for every packed row q of this call and,
 * in sampling mode, fp32 logits[q][vocab] (else NULL).  Q must equal the row
 * count the call packs (LA_ESTATE otherwise).  Everything else — lookup,
 * pack, verification, pool, window, out ring — is the product path; the K/V
 * commit copies whatever the temporary rows hold. */
int la_step_inject(la_ctx* ctx, int W, int N, int G, const la_sampling* s, int Q,
                   const int32_t* argmax, const float* logits, int32_t* out, int* n_out);

/* The exact sampling verifier alone (M7.3 §0x05B), for distribution tests:
 * n_trials independent verifications of the same rows, trial i drawing its
 * uniforms with Philox step index i.
 *   logits (host) [rows][V] fp32: row 0 the ordinary row, row 1 + c*S + s the
 *                  row whose input is candidate c's token s (rows >= 1 + Ct*S)
 *   cand   (host) [Ct][S] candidate suffix ids (Ct <= 32, 1 <= S <= 15)
 *   s      sampling policy (required)
 *   out    (host) [n_trials][S+3]: E (tokens emitted), a (accepted
 *                  candidate tokens), then the S+1 emitted ids (-1 padded).
 * Uses the current device; allocates its own temporary device buffers.
 * Errors: LA_EINVAL, LA_ENOTSUP (V * 4 bytes > 200 KB), LA_ECUDA. */
int la_debug_sample_verify(const float* logits, int rows, int V, const int32_t* cand, int Ct, int S,
                           const la_sampling* s, int n_trials, int32_t* out);

/* The tensor-core GEMM alone, for kernel tests: acc[q][n] = sum_k x[q][k] w[n][k]
 * with bf16 inputs (host, raw bf16 bit patterns) and fp32 accumulation on
 * n_cta persistent CTAs (0: one per SM; the (tile, K slice) units are split
 * evenly over them and a tile shared by several CTAs is reduced in K order),
 * followed by one epilogue:
 *   mode 0 store   y[q][n] = bf16(acc)                (w: n_seg stacked segments)
 *   mode 1 resid   y[q][n] += acc                     (y holds the input, fp32)
 *   mode 2 swiglu  y[q][n] = bf16(silu(acc_w) * acc_w2)
 *   mode 3 logits  y[q][n] = acc (fp32)
 * mode | LA_GEMM_PAIR (not with swiglu): the GEMM streams units of one
 * 64-column atom of two adjacent 128-row output tiles, as the model's QKV,
 * O, down and LM head GEMMs do (n_out / n_seg a multiple of 256).
 * w [n_out][K], w2 [n_out][K] (swiglu only), x [rows][K]; y (host)
 * [rows][n_out] fp32 (bf16 results widened).  n_out a multiple of
 * 128 * n_seg (n_seg 1..3), K of 64, 1 <= rows <= 1024, 0 <= n_cta <= 4096.
 * The weights are first packed into the unit-contiguous images the model's
 * GEMMs stream (la_init does the same for every projection).
 * Uses the current device and allocates its own temporary device buffers.
 * Errors: LA_EINVAL, LA_ECUDA, LA_ETIMEOUT. */
#define LA_GEMM_PAIR 16
int la_debug_gemm(int mode, const uint16_t* w, const uint16_t* w2, int n_seg, int n_out, int K,
                  const uint16_t* x, int rows, int n_cta, float* y);

/* Timing of the tensor-core GEMM alone (kernel tuning): n_copies weight
 * matrices of [n_out][K] (filled with small deterministic values) are used in
 * turn so that weights stream from HBM rather than L2; *us receives the mean
 * device time of one launch over `reps` launches after three warm-up
 * launches (CUDA events on the legacy default stream).  packed = 1 streams
 * the weights as the model's GEMMs do, from unit-contiguous images (one
 * 16 KB bulk copy per 128 x 64 tile); 0 loads the row-major matrices through
 * tensor maps, as la_gemm_noalloc does.  Arguments as for la_debug_gemm;
 * 1 <= n_copies <= 64, packed 0 or 1.  Errors: LA_EINVAL, LA_ECUDA,
 * LA_ETIMEOUT. */
int la_bench_gemm(int mode, int n_out, int K, int rows, int n_cta, int n_copies, int reps, int packed,
                  float* us);

/* The tensor-core GEMM for callers that cannot allocate device memory.  The
 * lookahead decoding pages have no counterpart to this call: it is a service
 * of this library.  Callers that cannot allocate: an engine whose own pool (a
 * KV-cache arena, a caching allocator) already holds all free device memory,
 * and callers that cannot accept the device-wide synchronisation cudaFree
 * implies.  The call allocates nothing: its workspace (status word, per-tile
 * arrival counters, split-tile partial sums) lives in a fixed 64 MiB array
 * compiled into the library, one per device.
 *   mode 0 store   y[q][n] = bf16(acc)            y bf16 [rows][n_out]
 *   mode 1 resid   y[q][n] += acc                 y fp32 [rows][n_out]
 *   mode 2 swiglu  y[q][n] = bf16(silu(acc_w) * acc_w2)
 * with acc[q][n] = sum_k x[q][k] w[n][k] (fp32 accumulation, K order, the
 * same kernel and reduction order as la_debug_gemm with n_cta 0).
 *   w, w2 (device) bf16 [n_out][K] row-major, 16-byte aligned (w2: swiglu only)
 *   x     (device) bf16 [rows][K] row-major, 16-byte aligned
 *   y     (device) as above, 4-byte aligned
 *   stream  cudaStream_t the work is ordered on (NULL: the legacy stream)
 * n_out a multiple of 128, K a multiple of 64 (>= 64), 1 <= rows <= 1024.  The call
 * returns once the result is in y.  Every call looks up the workspace's
 * address on the current device and sets the kernel's shared-memory limit
 * there; the first call on a device also loads the library's device code
 * there.  The counters
 * and status word must be zero when the GEMM starts: the call zeroes them
 * itself on `stream` before each launch.  There is one workspace per
 * device, so two executions overlapping on a device would race on it; calls
 * hold a process-wide lock until their work has finished, which keeps them
 * from overlapping.  Errors: LA_EINVAL (argument, alignment), LA_ECAPACITY
 * (the problem's partial sums exceed the 64 MiB workspace; checked before any
 * device work), LA_ENOTSUP (device index >= 64), LA_ECUDA, LA_ETIMEOUT. */
int la_gemm_noalloc(int mode, const void* w, const void* w2, int n_out, int K, const void* x, int rows, void* y,
                    void* stream);

/* Sizes fixed at la_init: [0]=Qmax [1]=max_W [2]=max_N [3]=max_G [4]=max_ctx
 * [5]=vocab [6]=window row length (max_W+max_N-3) [7]=path length bound. */
int la_query(la_ctx* ctx, int32_t* sizes8);

void        la_free(la_ctx* ctx);
const char* la_strerror(int code);
/* The last CUDA error string seen by this context (or "" if none). */
const char* la_last_cuda_error(la_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* LOOKAHEAD_H */
