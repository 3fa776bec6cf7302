// Integer state machine of one lookahead request on the GPU: window
// initialisation, the row compiler (pack), greedy verification, the out
// ring, the per-key LRU n-gram pool, the window advance and the K/V commit.
//
// Every rule here restates "M7.3 – Lookahead Decoding":
//   pack          §0x01A (row equations), §0x04/§0x04A (roles, positions,
//                 visibility, level-major order), §0x03C (lookup of G
//                 suffixes under the live key)
//   verification  §0x05A (longest accepted prefix, survivor order)
//   publication   §0x06B/§0x06C (ordinary row + h winner rows, next input)
//   pool          §0x03B (keyed extraction, per-key LRU)
//   window        §0x03A (warm-up fill), §0x03C (ALWAYS_FWD_ONE shift)
// All mutation happens only after a call's outputs are interpreted and only
// if the device error word is clear (fail-closed, §0x07).
#include "la_common.cuh"
#include "la_kernels.h"

// ---------------------------------------------------------------------------
// request start: seed level 0 with W+N-3 prompt tokens (cyclic), §0x03A
// ---------------------------------------------------------------------------
__global__ void k_begin(LaDev d, int mode, int W, int N, int G, int sampling,
                        float temperature, float top_p, uint32_t seed_lo, uint32_t seed_hi, int max_out, int opts) {
    LaTl la_tl_(LA_TL_BEGIN, d.tl);
    LaHdr* h = d.hdr;
    int t = threadIdx.x;
    if (t == 0) {
        h->mode = mode;
        h->opts = opts;
        h->sampling = sampling;
        h->W = W; h->N = N; h->G = G; h->S = N - 1;
        h->step = 0;
        h->done = (h->n_out >= max_out);
        h->max_out = max_out;
        h->temperature = temperature; h->top_p = top_p;
        h->seed_lo = seed_lo; h->seed_hi = seed_hi;
        h->n_steps = 0; h->n_steady = 0; h->sum_Q = 0; h->sum_Ct = 0;
        for (int i = 0; i < LA_HDR_STATS; ++i) h->hist[i] = 0;
        for (int r = 0; r < LA_MAX_R; ++r) h->level_len[r] = 0;
        if (mode == MODE_LOOKAHEAD) {
            h->n_levels = 1;
            h->level_len[0] = W + N - 3;
            h->seed_next = (W + N - 3) % h->prompt_len;
        } else {
            h->n_levels = 0;
        }
    }
    if (mode == MODE_LOOKAHEAD) {
        int P = h->prompt_len;
        for (int i = t; i < W + N - 3; i += blockDim.x) d.window[i] = d.prompt[i % P];
    }
}

// ---------------------------------------------------------------------------
// pack: token ids, logical positions, metadata, key paths, needed rows
// ---------------------------------------------------------------------------
__global__ void k_pack(LaDev d) {
    LaTl la_tl_(LA_TL_PACK, d.tl);
    la_pdl_wait();
    la_pdl_trigger();
    LaHdr* h = d.hdr;
    __shared__ int s_off[LA_MAX_R + 2];
    __shared__ int s_Q, s_Ct, s_vstart, s_ok, s_d, s_deep0;
    const int tid = threadIdx.x;
    if (h->err || h->done) {
        // a finished request of a batch: nothing of this call is committed
        if (tid == 0 && !h->err) h->commit_n = 0;
        return;
    }
    const int K = h->K, x_t = h->x_t, S = h->S;
    if (tid == 0) {
        int ok = 1;
        if (h->mode == MODE_AR) {
            s_Q = 1; s_Ct = 0; s_vstart = 1; s_d = -1; s_deep0 = 1;
            h->Q = 1; h->C_t = 0; h->steady = 0; h->n_deep = 0; h->deep_skip = 0; h->vstart = 1;
            h->n_need = 1;
            if (K + 1 > d.max_ctx) ok = 0;
        } else {
            int dl = h->n_levels - 1;
            int R = h->N - 1;
            int steady = (dl == R - 1);
            int Ct = 0;
            if (steady) {
                Ct = d.pool_cnt[x_t];
                if (Ct > h->G) Ct = h->G;
            }
            s_off[0] = 1;
            for (int r = 0; r <= dl; ++r) s_off[r + 1] = s_off[r] + h->level_len[r];
            int vstart = s_off[dl + 1];
            int Q = vstart + Ct * S;
            int n_deep = h->level_len[dl];
            int deep0 = s_off[dl];
            h->Q = Q; h->C_t = Ct; h->steady = steady; h->vstart = vstart;
            h->n_deep = n_deep; h->deep_skip = (!steady && dl >= 1) ? 1 : 0;
            h->n_need = 1 + n_deep + Ct * S;
            for (int r = 0; r <= dl + 1 && r <= LA_MAX_R; ++r) h->lvl_off[r] = s_off[r];
            s_Q = Q; s_Ct = Ct; s_vstart = vstart; s_d = dl; s_deep0 = deep0;
            // capacity: rows, key paths, positions of the call and the commit
            // largest offset pos-K of a row: level r cell j sits at j+r, v_{c,s} at 1+s
            int maxoff = h->level_len[0] + dl;
            if (steady && Ct > 0 && S > maxoff) maxoff = S;
            if (Q > d.Qmax || maxoff + 1 > d.PMAX || K + maxoff >= d.max_ctx + d.PMAX || K + 1 + S > d.max_ctx) ok = 0;
        }
        s_ok = ok;
        if (!ok) {
            la_set_err(h, LA_ECAPACITY);
            if (d.batch) la_set_err(d.batch, LA_ECAPACITY);
        }
    }
    __syncthreads();
    if (!s_ok) return;
    const int Q = s_Q, vstart = s_vstart, dl = s_d;
    const int P = d.PMAX;
    for (int q = tid; q < Q; q += blockDim.x) {
        int tok, pos, meta, plen = 0;
        int* path = d.row_path + (size_t)q * P;
        if (q == 0) {
            tok = x_t; pos = K; meta = la_meta(ROLE_ORDINARY, 0, 0, 0, 0);
            path[0] = 0; plen = 1;
        } else if (q < vstart) {
            int r = 0;
            while (q >= s_off[r + 1]) ++r;
            if (r == 0) {                       // base stripe b_j, j = q
                int j = q;
                tok = d.window[j - 1]; pos = K + j;
                meta = la_meta(ROLE_LOOKAHEAD, 0, j, 0, 0);
                for (int k = 0; k <= j; ++k) path[plen++] = k;
            } else {                            // u_{r,j}
                int j = q - s_off[r];
                tok = d.window[(size_t)r * d.LMAX + j]; pos = K + j + r;
                meta = la_meta(ROLE_LOOKAHEAD, r, j, 0, 0);
                for (int k = 0; k <= j; ++k) path[plen++] = k;
                for (int l = 1; l <= r; ++l) path[plen++] = s_off[l] + j;
            }
        } else {                                // v_{c,s}
            int c = (q - vstart) / S, s = (q - vstart) % S;
            tok = d.pool_tok[((size_t)x_t * d.Gmax + c) * d.Smax + s];
            pos = K + 1 + s;
            meta = la_meta(ROLE_VERIFY, 0, 0, c, s);
            path[plen++] = 0;
            for (int l = 0; l <= s; ++l) path[plen++] = vstart + c * S + l;
        }
        d.row_tok[q] = tok; d.row_pos[q] = pos; d.row_meta[q] = meta;
    }
    // batched call: the slice's remaining rows repeat the ordinary row
    for (int q = Q + tid; q < d.pad_to; q += blockDim.x) {
        d.row_tok[q] = x_t; d.row_pos[q] = K; d.row_meta[q] = la_meta(ROLE_ORDINARY, 0, 0, 0, 0);
        d.row_path[(size_t)q * P] = 0;
    }
    // needed rows: [0] + deepest level + verification rows (stacked-row
    // indices: the slice's first row added; a batch's slice padded with its
    // ordinary row)
    int n_need = 1;
    if (h->mode == MODE_AR) {
        if (tid == 0) d.need[0] = d.row_base;
    } else {
        int n_deep = h->level_len[dl];
        int nv = s_Ct * S;
        n_need = 1 + n_deep + nv;
        for (int i = tid; i < n_need; i += blockDim.x) {
            int r;
            if (i == 0) r = 0;
            else if (i <= n_deep) r = s_deep0 + (i - 1);
            else r = vstart + (i - 1 - n_deep);
            d.need[i] = d.row_base + r;
        }
    }
    for (int i = n_need + tid; i < d.pad_to; i += blockDim.x) d.need[i] = d.row_base;
}

// ---------------------------------------------------------------------------
// greedy verification + publication + pool + window (one CTA)
// ---------------------------------------------------------------------------
__device__ void pool_upsert_warp(const LaDev& d, int key, const int* suffix, int S, int G) {
    // One warp; lane g owns bucket entry g (G <= 32).  Entries are oldest first.
    const int lane = threadIdx.x & 31;
    int32_t* bucket = d.pool_tok + (size_t)key * d.Gmax * d.Smax;
    const int cnt = d.pool_cnt[key];
    bool match = false;
    if (lane < cnt) {
        match = true;
        for (int s = 0; s < S; ++s) match &= (bucket[lane * d.Smax + s] == suffix[s]);
    }
    const unsigned m = __ballot_sync(0xffffffffu, match);
    int from, last;
    if (m) { from = __ffs(m) - 1; last = cnt - 1; }   // reinsertion moves to the back
    else if (cnt >= G) { from = 0; last = cnt - 1; }  // full bucket evicts its oldest
    else { from = cnt; last = cnt; }                  // append
    int vals[LA_MAX_R];
    const bool sh = lane >= from && lane < last;      // entries after `from` move up one slot
    if (sh) for (int s = 0; s < S; ++s) vals[s] = bucket[(lane + 1) * d.Smax + s];
    __syncwarp();
    if (sh) for (int s = 0; s < S; ++s) bucket[lane * d.Smax + s] = vals[s];
    __syncwarp();
    if (lane == 0) {
        for (int s = 0; s < S; ++s) bucket[last * d.Smax + s] = suffix[s];
        d.pool_cnt[key] = last + 1;
    }
    __syncwarp();
}

// token at position k of the request's sequence: the prompt, then the out ring
__device__ __forceinline__ int seq_tok(const LaDev& d, int P, int k) { return k < P ? d.prompt[k] : d.out[k - P]; }

// the n-gram ending at sequence position k (k >= S): key token k-S, suffix k-S+1 .. k
__device__ __forceinline__ void upsert_seq_ngram_warp(const LaDev& d, int P, int k, int S, int G) {
    int suf[LA_MAX_R];
    const int key = seq_tok(d, P, k - S);
    for (int s = 0; s < S; ++s) suf[s] = seq_tok(d, P, k - S + 1 + s);
    pool_upsert_warp(d, key, suf, S, G);
}

// ---------------------------------------------------------------------------
// request start, optional pool seeding (POOL_FROM_PROMPT of M7.3 §0x03A,
// generated-prefix insertion of §0x06A): the n-grams ending at sequence
// positions S .. P-1 (inside the prompt) and/or P (the first output token),
// in increasing position.  Warp w applies the n-grams whose key is w modulo
// the warp count, so each key's upserts keep their order.
// ---------------------------------------------------------------------------
__global__ void k_pool_seed(LaDev d) {
    LaTl la_tl_(LA_TL_POOL_SEED, d.tl);
    const LaHdr* h = d.hdr;
    const int opts = h->opts, G = h->G, S = h->S, P = h->prompt_len;
    if (h->err || h->mode != MODE_LOOKAHEAD || G <= 0) return;
    const int k_lo = (opts & LA_OPT_POOL_FROM_PROMPT) ? S : P;
    const int k_hi = (opts & LA_OPT_POOL_FROM_OUTPUT) ? P + 1 : P;
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int k = k_lo > S ? k_lo : S; k < k_hi; ++k) {
        const int key = seq_tok(d, P, k - S);
        if (key % nw == warp) upsert_seq_ngram_warp(d, P, k, S, G);
    }
}

__global__ void k_publish(LaDev d, int verdict_given) {
    LaTl la_tl_(LA_TL_PUBLISH, d.tl);
    la_pdl_wait();
    la_pdl_trigger();
    LaHdr* h = d.hdr;
    __shared__ int s_best, s_emit[16], s_E, s_a, s_w, s_nout0, s_take;
    __shared__ int s_win[LA_MAX_R * LA_MAX_L];
    __shared__ int s_len[LA_MAX_R];
    __shared__ int s_z[LA_MAX_L];
    __shared__ int s_key[LA_MAX_L];
    __shared__ int s_suf[LA_MAX_L][LA_MAX_R];
    if (h->err || h->done) return;
    const int tid = threadIdx.x;
    const int S = h->S, Ct = h->C_t, vstart = h->vstart, n_deep = h->n_deep;
    const int mode = h->mode, steady = h->steady;
    const int x_old = h->x_t;
    if (tid == 0) s_best = -1;
    __syncthreads();
    // verdict
    if (!verdict_given) {
        if (tid < Ct) {
            int c = tid, a = 0, target = d.argmax[0];
            while (a < S && d.row_tok[vstart + c * S + a] == target) {
                target = d.argmax[1 + n_deep + c * S + a];
                ++a;
            }
            if (a > 0) atomicMax(&s_best, (a << 8) | (255 - c));
        }
        __syncthreads();
        if (tid == 0) {
            int a = 0, w = -1;
            if (s_best >= 0) { a = s_best >> 8; w = 255 - (s_best & 255); }
            if (a == 0) { s_emit[0] = d.argmax[0]; }
            else {
                for (int i = 0; i < a; ++i) s_emit[i] = d.row_tok[vstart + w * S + i];
                s_emit[a] = d.argmax[1 + n_deep + w * S + (a - 1)];
            }
            s_a = a; s_w = w; s_E = a + 1;
        }
    } else if (tid == 0) {   // sampling verdict written into the header
        s_a = h->a; s_w = h->winner; s_E = h->E;
        for (int i = 0; i < s_E; ++i) s_emit[i] = h->emitted[i];
    }
    __syncthreads();
    const int a = s_a, w = s_w, E = s_E;
    // stage the pre-shift window and z
    const int R = h->N - 1;
    const int nl = h->n_levels;
    if (mode == MODE_LOOKAHEAD) {
        if (tid < LA_MAX_R) s_len[tid] = (tid < nl) ? h->level_len[tid] : 0;
        for (int i = tid; i < nl * d.LMAX; i += blockDim.x) s_win[i] = d.window[i];
        int skip = h->deep_skip;
        for (int j = tid; j < n_deep - skip; j += blockDim.x) s_z[j] = d.argmax[1 + skip + j];
    }
    __syncthreads();
    // publication: out ring, commit plan, frontier
    if (tid == 0) {
        int n_out = h->n_out;
        int room = h->max_out - n_out;
        int take = E < room ? E : room;
        for (int i = 0; i < take; ++i) d.out[n_out + i] = s_emit[i];
        s_nout0 = n_out;
        s_take = take;
        h->n_out = n_out + take;
        if (h->n_out >= h->max_out) {
            h->done = 1;
            // the batch is done once its last live request is
            if (d.batch && atomicSub(&d.batch->active, 1) == 1) d.batch->done = 1;
        }
        h->a = a; h->winner = w; h->E = E;
        for (int i = 0; i < E; ++i) h->emitted[i] = s_emit[i];
        h->commit_base = h->K;
        h->commit_n = 1 + a;
        d.commit_rows[0] = 0;
        for (int i = 0; i < a; ++i) d.commit_rows[1 + i] = vstart + w * S + i;
        h->K = h->K + 1 + a;
        h->x_t = s_emit[E - 1];
        h->n_steps += 1;
        h->sum_Q += h->Q;
        if (steady) { h->n_steady += 1; h->sum_Ct += Ct; }
        h->hist[E < LA_HDR_STATS ? E - 1 : LA_HDR_STATS - 1] += 1;
        h->step += 1;
    }
    if (mode != MODE_LOOKAHEAD) return;
    // pool update from the pre-shift levels (steady calls only), §0x03B
    const int W = h->W, G = h->G;
    if (steady) {
        for (int j = tid; j < W; j += blockDim.x) {
            s_key[j] = (j == 0) ? x_old : s_win[j - 1];
            for (int r = 1; r < R; ++r) s_suf[j][r - 1] = s_win[r * d.LMAX + j];
            s_suf[j][R - 1] = s_z[j];
        }
        __syncthreads();
        // one warp per first occurrence of a key; it applies that key's upserts in column order
        const int warp = tid >> 5, nwarps = blockDim.x >> 5;
        if (G > 0) {
            for (int j = warp; j < W; j += nwarps) {
                int key = s_key[j];
                bool first = true;
                for (int k = 0; k < j; ++k) first &= (s_key[k] != key);
                if (!first) continue;
                for (int k = j; k < W; ++k)
                    if (s_key[k] == key) pool_upsert_warp(d, key, s_suf[k], S, G);
            }
        }
    }
    __syncthreads();
    // generated-prefix insertion (§0x06A): the n-grams ending at the tokens
    // this call appended, after the trajectory's, in increasing position
    if ((h->opts & LA_OPT_POOL_FROM_OUTPUT) && G > 0 && tid < 32) {
        const int P = h->prompt_len;
        for (int k = P + s_nout0; k < P + s_nout0 + s_take; ++k)
            if (k >= S) upsert_seq_ngram_warp(d, P, k, S, G);
    }
    __syncthreads();
    // window advance: steady §0x03C, warm-up §0x03A
    if (steady) {
        // new[0] = old[1][1:], new[r] = old[r+1] (1 <= r <= R-2), new[R-1] = z.
        // ALWAYS_FWD_ONE=False (LA_OPT_SLICE_WINDOW): every new level also drops
        // its first `sl` = a cells; the vacated tail cells, level 0 first and
        // each level in column order, take the next tokens of the prompt cycle.
        const int sl = (h->opts & LA_OPT_SLICE_WINDOW) ? a : 0;
        const int n0 = sl < W - 1 ? sl : W - 1;     // refills of level 0
        const int nr = sl < W ? sl : W;             // refills of each deeper level
        const int P = h->prompt_len, seed0 = h->seed_next;
        for (int i = tid; i < W - 1; i += blockDim.x)
            d.window[i] = (i < W - 1 - n0) ? s_win[1 * d.LMAX + 1 + sl + i]
                                           : d.prompt[(seed0 + i - (W - 1 - n0)) % P];
        for (int r = 1; r < R; ++r)
            for (int i = tid; i < W; i += blockDim.x) {
                const int c = n0 + (r - 1) * nr + i - (W - nr);   // refill index of this cell
                d.window[r * d.LMAX + i] = (i < W - nr) ? (r < R - 1 ? s_win[(r + 1) * d.LMAX + sl + i] : s_z[sl + i])
                                                        : d.prompt[(seed0 + c) % P];
            }
        __syncthreads();   // every thread has read seed_next (steady is block-uniform)
        if (tid == 0) {
            h->level_len[0] = W - 1;
            for (int r = 1; r < R; ++r) h->level_len[r] = W;
            h->seed_next = (seed0 + n0 + (R - 1) * nr) % P;
        }
    } else {
        int dl = nl - 1;
        int nz = n_deep - h->deep_skip;
        for (int r = 0; r <= dl; ++r)
            for (int i = tid; i < s_len[r] - 1; i += blockDim.x) d.window[r * d.LMAX + i] = s_win[r * d.LMAX + 1 + i];
        for (int i = tid; i < nz; i += blockDim.x) d.window[(dl + 1) * d.LMAX + i] = s_z[i];
        if (tid == 0) {
            for (int r = 0; r <= dl; ++r) h->level_len[r] = s_len[r] - 1;
            h->level_len[dl + 1] = nz;
            h->n_levels = nl + 1;
        }
    }
}

// ---------------------------------------------------------------------------
// K/V commit: temp rows commit_rows[i] -> cache position commit_base + i
// (the ordinary row and the winner's first a verification rows, §0x06C).
// grid.x = n_layers * 2 * n_heads; vectorised 16-byte copies.
// ---------------------------------------------------------------------------
__global__ void k_commit_kv(LaDev d, char* cache, char* temp, int n_heads, int head_bytes,
                            int max_ctx, int Qmax) {
    LaTl la_tl_(LA_TL_COMMIT_KV, d.tl);
    la_pdl_wait();
    la_pdl_trigger();
    LaHdr* h = d.hdr;
    if (h->err) return;
    // `done` may have been set by this very call's publication: the copy still runs
    const int n = h->commit_n, base = h->commit_base;
    const size_t plane = blockIdx.x;   // (layer, k/v, head)
    const char* src = temp + plane * (size_t)Qmax * head_bytes;
    char* dst = cache + plane * (size_t)max_ctx * head_bytes;
    const int vec = head_bytes / 16;
    for (int i = threadIdx.x; i < n * vec; i += blockDim.x) {
        int r = i / vec, c = i % vec;
        int srow = d.commit_rows[r];
        const int4* s = reinterpret_cast<const int4*>(src + (size_t)srow * head_bytes) + c;
        int4* t = reinterpret_cast<int4*>(dst + (size_t)(base + r) * head_bytes) + c;
        *t = *s;
    }
}

// ---------------------------------------------------------------------------
// injected outputs (la_step_inject): argmax by packed row -> need order
// ---------------------------------------------------------------------------
__global__ void k_inject_map(LaDev d, const int32_t* argmax_rows, const float* logits_rows,
                             float* logits_need, int V) {
    LaTl la_tl_(LA_TL_INJECT_MAP, d.tl);
    LaHdr* h = d.hdr;
    if (h->err || h->done) return;
    int n = h->n_need;
    for (int i = threadIdx.x; i < n; i += blockDim.x) d.argmax[i] = argmax_rows[d.need[i]];
    if (logits_rows) {
        for (int i = blockIdx.x; i < n; i += gridDim.x) {
            const float* s = logits_rows + (size_t)d.need[i] * V;
            float* t = logits_need + (size_t)i * V;
            for (int v = threadIdx.x; v < V; v += blockDim.x) t[v] = s[v];
        }
    }
}

// ---------------------------------------------------------------------------
// prefill rows of chunk [c0, c0+n): tokens and positions 0..P-1
// ---------------------------------------------------------------------------
__global__ void k_prefill_rows(LaDev d, int c0, int n) {
    LaTl la_tl_(LA_TL_PREFILL_ROWS, d.tl);
    LaHdr* h = d.hdr;
    if (threadIdx.x == 0 && blockIdx.x == 0) { h->Q = n; h->prefill_rows = n; }
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        d.row_tok[i] = d.prompt[c0 + i];
        d.row_pos[i] = c0 + i;
        d.row_meta[i] = 0;
    }
}

// the last prompt row is the only needed row of a prefill
__global__ void k_prefill_need(LaDev d, int last_local) {
    LaTl la_tl_(LA_TL_PREFILL_NEED, d.tl);
    LaHdr* h = d.hdr;
    h->n_need = 1;
    d.need[0] = last_local;
}

// after the prefill: the frontier is the prompt, x_t the first token
__global__ void k_prefill_finish(LaDev d, int P, int sampled_token_valid) {
    LaTl la_tl_(LA_TL_PREFILL_FINISH, d.tl);
    LaHdr* h = d.hdr;
    if (h->err) return;
    h->K = P;
    h->x_t = d.argmax[0];
    h->n_out = 1;
    d.out[0] = d.argmax[0];
    h->done = 0;
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
void la_launch_begin(const LaDev& d, cudaStream_t st, int mode, int W, int N, int G, int sampling,
                     float temperature, float top_p, uint64_t seed, int max_out, int opts) {
    k_begin<<<1, 128, 0, st>>>(d, mode, W, N, G, sampling, temperature, top_p,
                               (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32), max_out, opts); la_note_launch();
    if (mode == MODE_LOOKAHEAD && opts) {
        k_pool_seed<<<1, 1024, 0, st>>>(d);
        la_note_launch();
    }
}
void la_launch_pack(const LaDev& d, cudaStream_t st) { la_launch_pdl(k_pack, dim3(1), dim3(256), 0, st, d); }
void la_launch_publish(const LaDev& d, cudaStream_t st, int verdict_given) {
    la_launch_pdl(k_publish, dim3(1), dim3(256), 0, st, d, verdict_given);
}
void la_launch_commit(const LaDev& d, cudaStream_t st, void* cache, void* temp, int planes, int n_heads,
                      int head_bytes, int max_ctx, int Qmax) {
    la_launch_pdl(k_commit_kv, dim3(planes), dim3(128), 0, st, d, (char*)cache, (char*)temp, n_heads, head_bytes,
                  max_ctx, Qmax);
}
void la_launch_inject_map(const LaDev& d, cudaStream_t st, const int32_t* argmax_rows, const float* logits_rows,
                          float* logits_need, int V) {
    k_inject_map<<<logits_rows ? 64 : 1, 256, 0, st>>>(d, argmax_rows, logits_rows, logits_need, V); la_note_launch();
}
void la_launch_prefill_rows(const LaDev& d, cudaStream_t st, int c0, int n) {
    k_prefill_rows<<<(n + 255) / 256, 256, 0, st>>>(d, c0, n); la_note_launch();
}
void la_launch_prefill_need(const LaDev& d, cudaStream_t st, int last_local) {
    k_prefill_need<<<1, 1, 0, st>>>(d, last_local); la_note_launch();
}
void la_launch_prefill_finish(const LaDev& d, cudaStream_t st, int P) {
    k_prefill_finish<<<1, 1, 0, st>>>(d, P, 1); la_note_launch();
}
