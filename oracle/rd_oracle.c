/*
 * rd_oracle.c -- plain fp64 CPU oracle of the ReDrafter verification step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header or constant with the CUDA library.
 *
 * Every function is the plain definition of what the step computes, written
 * for a reader to check by eye, with no blocking, fusion or reordering:
 *
 *   oracle_pack            dynamic tree attention's prefix dedup
 *                          ("Recurrent Drafter for Fast Speculative Decoding in
 *                          LLMs", abstract: dynamic tree attention over beam
 *                          search results removes duplicated prefixes; Apple x
 *                          NVIDIA news page, section on dynamic tree attention:
 *                          shared prefixes are found and removed from the tokens
 *                          to verify).
 *   oracle_tree_attention  attention of the packed drafts over the KV cache and
 *                          their own tree ancestors (speculative-decoding survey
 *                          page, SpecInfer "Token Tree Verifier": one kernel with
 *                          a topology-aware causal mask replaces per-sequence
 *                          attention).
 *   oracle_tree_attention_paged  the same attention with the context read
 *                          through a paged KV cache (NVIDIA blog, introduction:
 *                          TensorRT-LLM's paged KV caching): position j of
 *                          request b lives in page block_table[b][j / page_size],
 *                          row j % page_size.
 *   oracle_tree_attention_fp8  the same attention with the context K/V stored
 *                          as e4m3 with one scale per tensor (NVIDIA blog,
 *                          introduction: TensorRT-LLM's FP8 quantisation).
 *   oracle_causal_attention  causal prefill of context-phase requests (NVIDIA
 *                          blog, "Inflight-batching Compatible Engine").
 *   oracle_beam_search_step  one step of the drafter's beam search (news page,
 *                          paragraph on the RNN draft model): the W best
 *                          (beam, token) candidates by cumulative log-probability.
 *   oracle_greedy_accept   greedy verification: argmax per packed position,
 *                          longest accepted draft prefix per beam, best beam
 *                          (NVIDIA blog introduction: verify and accept the best
 *                          path before drafting; news page: greedy decoding).
 *   oracle_sample_accept   stochastic verification of the draft tree by
 *                          multi-step speculative sampling (speculative-decoding
 *                          survey page: the rejection-sampling paragraph and
 *                          SpecInfer's "Token Tree Verifier").
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - position 0 of every beam is the anchor (already emitted by the LLM);
 *    positions 1..L-1 are drafts;
 *  - packed order = flattened beams (f = w*L + i) with every repeated prefix
 *    deleted, order kept; mask bits LSB-first within 32-bit words;
 *  - scale 1/sqrt(D) unless given; softmax with the maximum subtracted, in fp64;
 *  - argmax ties go to the lowest vocab index, beam ties to the lowest beam;
 *  - padded packed rows (p >= packed_len) give output 0 / argmax -1.
 *
 * bf16 inputs arrive as raw uint16 bit patterns and are widened exactly.
 * Return value: 0 on success, negative on an input the definition rejects.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_f64(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Two beams share the prefix of length i+1 iff their first i+1 tokens match. */
static int same_prefix(const int32_t* beam_a, const int32_t* beam_b, int i)
{
    for (int j = 0; j <= i; ++j)
        if (beam_a[j] != beam_b[j]) return 0;
    return 1;
}

int oracle_pack(const int32_t* beams, int B, int W, int L, int P_cap,
                int32_t* tokens, int32_t* packer, int32_t* unpacker,
                uint32_t* mask, int32_t* depth, int32_t* packed_len)
{
    if (B < 0 || W <= 0 || L <= 0 || P_cap <= 0) return -1;
    const int NW = (P_cap + 31) / 32;
    for (int b = 0; b < B; ++b) {
        const int32_t* bb = beams + (size_t)b * W * L;
        int32_t* tok = tokens + (size_t)b * P_cap;
        int32_t* pk = packer + (size_t)b * P_cap;
        int32_t* up = unpacker + (size_t)b * W * L;
        uint32_t* mk = mask + (size_t)b * P_cap * NW;
        int32_t* dp = depth + (size_t)b * P_cap;
        int P = 0;
        /* scan the flattened beams; a position whose prefix was seen before
         * maps to that earlier node, otherwise it becomes the next packed node */
        for (int f = 0; f < W * L; ++f) {
            int w = f / L, i = f % L, found = -1;
            for (int g = 0; g < P && found < 0; ++g) {
                int fw = pk[g] / L, fi = pk[g] % L;
                if (fi == i && same_prefix(bb + (size_t)fw * L, bb + (size_t)w * L, i))
                    found = g;
            }
            if (found >= 0) {
                up[w * L + i] = found;
            } else {
                if (P >= P_cap) return -2;
                pk[P] = f;
                tok[P] = bb[w * L + i];
                dp[P] = i;
                up[w * L + i] = P;
                ++P;
            }
        }
        packed_len[b] = P;
        /* ancestor mask: row p holds the nodes on the path root..p */
        memset(mk, 0, sizeof(uint32_t) * (size_t)P_cap * NW);
        for (int p = 0; p < P; ++p) {
            int w = pk[p] / L, i = pk[p] % L;
            for (int j = 0; j <= i; ++j) {
                int a = up[w * L + j];
                mk[(size_t)p * NW + a / 32] |= 1u << (a % 32);
            }
        }
        for (int p = P; p < P_cap; ++p) {
            tok[p] = 0;
            pk[p] = -1;
            dp[p] = 0;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* attention                                                                 */
/* ------------------------------------------------------------------------ */

/* softmax(scale * q.k) weighted sum of v over the keys the caller lists */
static void attend(const uint16_t* q, int D, double scale, int n_keys,
                   const uint16_t* const* keys, const uint16_t* const* vals,
                   double* s_buf, double* out)
{
    double m = -INFINITY;
    for (int j = 0; j < n_keys; ++j) {
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += bf16_to_f64(q[d]) * bf16_to_f64(keys[j][d]);
        s *= scale;
        s_buf[j] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int j = 0; j < n_keys; ++j) {
        double e = exp(s_buf[j] - m);
        l += e;
        for (int d = 0; d < D; ++d) out[d] += e * bf16_to_f64(vals[j][d]);
    }
    for (int d = 0; d < D; ++d) out[d] = (n_keys > 0) ? out[d] / l : 0.0;
}

typedef struct {
    int B, P_max, Hq, Hkv, D, NW;
    double scale;
    const uint16_t *q, *k_new, *v_new, *k_cache, *v_cache;
    const int64_t* ctx_offsets;
    const int32_t* packed_len;
    const uint32_t* mask;
    double* o;
    int next_task, n_tasks;
    pthread_mutex_t lock;
    int err;
    /* paged context (ctx_lens != NULL): rows of k_cache/v_cache are pool rows */
    const int32_t* ctx_lens;
    const int32_t* block_table;
    int max_pages, page_size;
} tree_job;

/* context length of request b */
static int64_t ctx_len(const tree_job* J, int b)
{
    if (J->ctx_lens) return J->ctx_lens[b];
    return J->ctx_offsets[b + 1] - J->ctx_offsets[b];
}

/* cache row holding context position j of request b */
static int64_t ctx_row(const tree_job* J, int b, int64_t j)
{
    if (J->ctx_lens) {
        int64_t page = J->block_table[(size_t)b * J->max_pages + j / J->page_size];
        return page * J->page_size + j % J->page_size;
    }
    return J->ctx_offsets[b] + j;
}

static void tree_task(tree_job* J, int task, const uint16_t** keys, const uint16_t** vals,
                      double* s_buf)
{
    int b = task / J->Hq, hq = task % J->Hq;
    int G = J->Hq / J->Hkv, h = hq / G;
    int64_t C = ctx_len(J, b);
    int Pb = J->packed_len[b];
    size_t qrow = (size_t)J->Hq * J->D, kvrow = (size_t)J->Hkv * J->D;
    for (int p = 0; p < J->P_max; ++p) {
        double* out = J->o + (((size_t)b * J->P_max + p) * J->Hq + hq) * J->D;
        if (p >= Pb) {
            for (int d = 0; d < J->D; ++d) out[d] = 0.0;
            continue;
        }
        int n = 0;
        for (int64_t j = 0; j < C; ++j) {     /* every context key is visible */
            int64_t r = ctx_row(J, b, j);
            keys[n] = J->k_cache + (size_t)r * kvrow + (size_t)h * J->D;
            vals[n] = J->v_cache + (size_t)r * kvrow + (size_t)h * J->D;
            ++n;
        }
        const uint32_t* row = J->mask + ((size_t)b * J->P_max + p) * J->NW;
        for (int k = 0; k < Pb; ++k) {        /* drafts: the node's ancestors and itself */
            if (row[k / 32] & (1u << (k % 32))) {
                keys[n] = J->k_new + ((size_t)b * J->P_max + k) * kvrow + (size_t)h * J->D;
                vals[n] = J->v_new + ((size_t)b * J->P_max + k) * kvrow + (size_t)h * J->D;
                ++n;
            }
        }
        attend(J->q + ((size_t)b * J->P_max + p) * qrow + (size_t)hq * J->D, J->D,
               J->scale, n, keys, vals, s_buf, out);
    }
}

static void* tree_worker(void* arg)
{
    tree_job* J = (tree_job*)arg;
    int64_t max_ctx = 0;
    for (int b = 0; b < J->B; ++b) {
        int64_t c = ctx_len(J, b);
        if (c > max_ctx) max_ctx = c;
    }
    size_t cap = (size_t)max_ctx + (size_t)J->P_max;
    const uint16_t** keys = malloc(sizeof(*keys) * (cap + 1));
    const uint16_t** vals = malloc(sizeof(*vals) * (cap + 1));
    double* s_buf = malloc(sizeof(double) * (cap + 1));
    if (!keys || !vals || !s_buf) {
        pthread_mutex_lock(&J->lock);
        J->err = -3;
        pthread_mutex_unlock(&J->lock);
    } else {
        for (;;) {
            pthread_mutex_lock(&J->lock);
            int t = J->next_task++;
            pthread_mutex_unlock(&J->lock);
            if (t >= J->n_tasks) break;
            tree_task(J, t, keys, vals, s_buf);
        }
    }
    free(keys); free(vals); free(s_buf);
    return NULL;
}

static int run_tree_job(tree_job* J, int n_threads)
{
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    pthread_t th[256];
    for (int t = 0; t < n_threads; ++t) pthread_create(&th[t], NULL, tree_worker, J);
    for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
    return J->err;
}

int oracle_tree_attention(int B, int P_max, int Hq, int Hkv, int D, double scale,
                          const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                          const uint16_t* k_cache, const uint16_t* v_cache,
                          const int64_t* ctx_offsets, const int32_t* packed_len,
                          const uint32_t* mask, int mask_words, double* o, int n_threads)
{
    if (B < 0 || P_max <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0) return -1;
    for (int b = 0; b < B; ++b)
        if (packed_len[b] < 0 || packed_len[b] > P_max ||
            ctx_offsets[b + 1] < ctx_offsets[b]) return -1;
    tree_job J = {B, P_max, Hq, Hkv, D, mask_words, scale > 0 ? scale : 1.0 / sqrt((double)D),
                  q, k_new, v_new, k_cache, v_cache, ctx_offsets, packed_len, mask, o,
                  0, B * Hq, PTHREAD_MUTEX_INITIALIZER, 0, NULL, NULL, 0, 1};
    return run_tree_job(&J, n_threads);
}

int oracle_tree_attention_paged(int B, int P_max, int Hq, int Hkv, int D, double scale,
                                const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                                const uint16_t* k_pool, const uint16_t* v_pool, int num_pages,
                                int page_size, const int32_t* block_table, int max_pages,
                                const int32_t* ctx_lens, const int32_t* packed_len,
                                const uint32_t* mask, int mask_words, double* o, int n_threads)
{
    if (B < 0 || P_max <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || page_size <= 0 ||
        max_pages < 0)
        return -1;
    for (int b = 0; b < B; ++b) {
        if (packed_len[b] < 0 || packed_len[b] > P_max || ctx_lens[b] < 0 ||
            (int64_t)ctx_lens[b] > (int64_t)max_pages * page_size)
            return -1;
        for (int64_t p = 0; p < ((int64_t)ctx_lens[b] + page_size - 1) / page_size; ++p) {
            int32_t pg = block_table[(size_t)b * max_pages + p];
            if (pg < 0 || pg >= num_pages) return -1;
        }
    }
    tree_job J = {B, P_max, Hq, Hkv, D, mask_words, scale > 0 ? scale : 1.0 / sqrt((double)D),
                  q, k_new, v_new, k_pool, v_pool, NULL, packed_len, mask, o,
                  0, B * Hq, PTHREAD_MUTEX_INITIALIZER, 0, ctx_lens, block_table, max_pages,
                  page_size};
    return run_tree_job(&J, n_threads);
}

typedef struct {
    int Bc, Hq, Hkv, D;
    double scale;
    const uint16_t *q, *k, *v;
    const int32_t* cu;
    double* o;
    int next_task, n_tasks, max_len;
    pthread_mutex_t lock;
    int err;
} causal_job;

static void* causal_worker(void* arg)
{
    causal_job* J = (causal_job*)arg;
    const uint16_t** keys = malloc(sizeof(*keys) * ((size_t)J->max_len + 1));
    const uint16_t** vals = malloc(sizeof(*vals) * ((size_t)J->max_len + 1));
    double* s_buf = malloc(sizeof(double) * ((size_t)J->max_len + 1));
    int G = J->Hq / J->Hkv;
    if (keys && vals && s_buf) {
        for (;;) {
            pthread_mutex_lock(&J->lock);
            int t = J->next_task++;
            pthread_mutex_unlock(&J->lock);
            if (t >= J->n_tasks) break;
            int b = t / J->Hq, hq = t % J->Hq, h = hq / G;
            int s0 = J->cu[b], T = J->cu[b + 1] - s0;
            for (int i = 0; i < T; ++i) {       /* query i sees keys 0..i */
                for (int j = 0; j <= i; ++j) {
                    keys[j] = J->k + ((size_t)(s0 + j) * J->Hkv + h) * J->D;
                    vals[j] = J->v + ((size_t)(s0 + j) * J->Hkv + h) * J->D;
                }
                attend(J->q + ((size_t)(s0 + i) * J->Hq + hq) * J->D, J->D, J->scale,
                       i + 1, keys, vals, s_buf,
                       J->o + ((size_t)(s0 + i) * J->Hq + hq) * J->D);
            }
        }
    } else {
        pthread_mutex_lock(&J->lock);
        J->err = -3;
        pthread_mutex_unlock(&J->lock);
    }
    free(keys); free(vals); free(s_buf);
    return NULL;
}

int oracle_causal_attention(int Bc, int Hq, int Hkv, int D, double scale,
                            const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            const int32_t* cu_seqlens, double* o, int n_threads)
{
    if (Bc < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0) return -1;
    int max_len = 0;
    for (int b = 0; b < Bc; ++b) {
        int T = cu_seqlens[b + 1] - cu_seqlens[b];
        if (T < 0) return -1;
        if (T > max_len) max_len = T;
    }
    causal_job J = {Bc, Hq, Hkv, D, scale > 0 ? scale : 1.0 / sqrt((double)D), q, k, v,
                    cu_seqlens, o, 0, Bc * Hq, max_len, PTHREAD_MUTEX_INITIALIZER, 0};
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    pthread_t th[256];
    for (int t = 0; t < n_threads; ++t) pthread_create(&th[t], NULL, causal_worker, &J);
    for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
    return J.err;
}

/* ------------------------------------------------------------------------ */
/* greedy acceptance                                                         */
/* ------------------------------------------------------------------------ */
int oracle_greedy_accept(const uint16_t* logits, int B, int P_max, int V,
                         const int32_t* beams, const int32_t* unpacker,
                         const int32_t* packed_len, int W, int L,
                         int32_t* argmax, int32_t* accept_len, int32_t* best_beam,
                         int32_t* n_accepted, int32_t* out_tokens)
{
    if (B < 0 || P_max <= 0 || V <= 0 || W <= 0 || L <= 0) return -1;
    for (int b = 0; b < B; ++b) {
        int Pb = packed_len[b];
        if (Pb < 0 || Pb > P_max) return -1;
        /* (i) greedy choice at every packed position; the first maximum wins */
        for (int p = 0; p < P_max; ++p) {
            int32_t* g = argmax + (size_t)b * P_max + p;
            if (p >= Pb) { *g = -1; continue; }
            const uint16_t* row = logits + ((size_t)b * P_max + p) * V;
            double best = bf16_to_f64(row[0]);
            int bi = 0;
            for (int v = 1; v < V; ++v) {
                double x = bf16_to_f64(row[v]);
                if (x > best) { best = x; bi = v; }
            }
            *g = bi;
        }
        /* (ii) per beam: drafts accepted while each equals the greedy choice
         * made at the position before it */
        const int32_t* bb = beams + (size_t)b * W * L;
        const int32_t* up = unpacker + (size_t)b * W * L;
        const int32_t* g = argmax + (size_t)b * P_max;
        int best_w = 0, best_a = -1;
        for (int w = 0; w < W; ++w) {
            int a = 0;
            for (int j = 1; j < L; ++j) {
                int prev = up[w * L + j - 1];
                if (prev < 0 || prev >= Pb) return -4;
                if (bb[w * L + j] != g[prev]) break;
                a = j;
            }
            accept_len[(size_t)b * W + w] = a;
            /* (iii) best beam: most accepted drafts, lowest beam on ties */
            if (a > best_a) { best_a = a; best_w = w; }
        }
        best_beam[b] = best_w;
        n_accepted[b] = best_a;
        /* (iv) emitted tokens: the accepted drafts, then the greedy token at the
         * last accepted node */
        int32_t* ot = out_tokens + (size_t)b * L;
        for (int j = 0; j < L; ++j) ot[j] = -1;
        for (int j = 1; j <= best_a; ++j) ot[j - 1] = bb[best_w * L + j];
        int last = up[best_w * L + best_a];
        if (last < 0 || last >= Pb) return -4;
        ot[best_a] = g[last];
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* drafter beam search                                                       */
/* ------------------------------------------------------------------------ */
/* One step of the drafter's beam search (Apple x NVIDIA news page, paragraph
 * on the RNN draft model: from the initial token and the LLM's last hidden
 * state the drafter runs a beam search that yields several candidate token
 * sequences).  Candidate (w, v) scores scores_in[w] + log softmax(logits[w])[v];
 * a beam with score -inf has no candidates.  The W best candidates, best first
 * (equal scores: lower w*V + v first), become the new beams. */
int oracle_beam_search_step(const uint16_t* logits, const double* scores_in,
                            const int32_t* beams_in, int B, int W, int V, int t,
                            int32_t* beams_out, double* scores_out, int32_t* parent)
{
    if (B < 0 || W <= 0 || V < W || t < 0) return -1;
    double* cand = malloc(sizeof(double) * (size_t)W * V);
    unsigned char* taken = malloc((size_t)W * V);
    if (!cand || !taken) { free(cand); free(taken); return -3; }
    for (int b = 0; b < B; ++b) {
        const uint16_t* lg = logits + (size_t)b * W * V;
        for (int w = 0; w < W; ++w) {
            const uint16_t* row = lg + (size_t)w * V;
            double mx = -INFINITY, sum = 0.0;
            for (int v = 0; v < V; ++v) {
                double x = bf16_to_f64(row[v]);
                if (x > mx) mx = x;
            }
            for (int v = 0; v < V; ++v) sum += exp(bf16_to_f64(row[v]) - mx);
            double lse = mx + log(sum);
            double s = scores_in[(size_t)b * W + w];
            for (int v = 0; v < V; ++v)
                cand[(size_t)w * V + v] = (s == -INFINITY) ? -INFINITY : s + bf16_to_f64(row[v]) - lse;
        }
        memset(taken, 0, (size_t)W * V);
        for (int r = 0; r < W; ++r) {
            int best = -1;
            for (int i = 0; i < W * V; ++i) {
                if (taken[i] || cand[i] == -INFINITY) continue;
                if (best < 0 || cand[i] > cand[best]) best = i;   /* first maximum: lower index */
            }
            if (best < 0) { free(cand); free(taken); return -4; }
            taken[best] = 1;
            int pw = best / V, tok = best % V;
            parent[(size_t)b * W + r] = pw;
            scores_out[(size_t)b * W + r] = cand[best];
            for (int j = 0; j < t; ++j)
                beams_out[((size_t)b * W + r) * (t + 1) + j] = beams_in[((size_t)b * W + pw) * t + j];
            beams_out[((size_t)b * W + r) * (t + 1) + t] = tok;
        }
    }
    free(cand);
    free(taken);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* FP8 (e4m3) context                                                        */
/* ------------------------------------------------------------------------ */
/* e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
 * subnormal (m/8 * 2^-6); S.1111.111 is NaN; there are no infinities. */
static double e4m3_to_f64(uint8_t x)
{
    int sgn = x >> 7, e = (x >> 3) & 15, m = x & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -v : v;
}

double oracle_e4m3_value(int code) { return e4m3_to_f64((uint8_t)code); }

int oracle_tree_attention_fp8(int B, int P_max, int Hq, int Hkv, int D, double scale,
                              const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                              const uint8_t* k_cache, const uint8_t* v_cache, double k_scale,
                              double v_scale, const int64_t* ctx_offsets,
                              const int32_t* packed_len, const uint32_t* mask, int mask_words,
                              double* o)
{
    if (B < 0 || P_max <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0) return -1;
    if (scale <= 0) scale = 1.0 / sqrt((double)D);
    int G = Hq / Hkv;
    int64_t max_n = 0;
    for (int b = 0; b < B; ++b) {
        if (packed_len[b] < 0 || packed_len[b] > P_max) return -1;
        int64_t c = ctx_offsets[b + 1] - ctx_offsets[b] + P_max;
        if (c > max_n) max_n = c;
    }
    double* s_buf = malloc(sizeof(double) * (size_t)(max_n + 1));
    if (!s_buf) return -3;
    for (int b = 0; b < B; ++b) {
        int64_t c0 = ctx_offsets[b], C = ctx_offsets[b + 1] - c0;
        int Pb = packed_len[b];
        for (int hq = 0; hq < Hq; ++hq) {
            int h = hq / G;
            for (int p = 0; p < P_max; ++p) {
                double* out = o + (((size_t)b * P_max + p) * Hq + hq) * D;
                for (int d = 0; d < D; ++d) out[d] = 0.0;
                if (p >= Pb) continue;
                const uint16_t* qv = q + (((size_t)b * P_max + p) * Hq + hq) * D;
                const uint32_t* row = mask + ((size_t)b * P_max + p) * mask_words;
                /* scores: context keys are k_scale * e4m3, drafts are bf16 */
                double m = -INFINITY;
                int64_t n = 0;
                for (int64_t j = 0; j < C; ++j, ++n) {
                    const uint8_t* kr = k_cache + ((size_t)(c0 + j) * Hkv + h) * D;
                    double sc = 0.0;
                    for (int d = 0; d < D; ++d) sc += bf16_to_f64(qv[d]) * (k_scale * e4m3_to_f64(kr[d]));
                    s_buf[n] = sc * scale;
                    if (s_buf[n] > m) m = s_buf[n];
                }
                for (int k = 0; k < Pb; ++k) {
                    if (!(row[k / 32] & (1u << (k % 32)))) continue;
                    const uint16_t* kr = k_new + (((size_t)b * P_max + k) * Hkv + h) * D;
                    double sc = 0.0;
                    for (int d = 0; d < D; ++d) sc += bf16_to_f64(qv[d]) * bf16_to_f64(kr[d]);
                    s_buf[n] = sc * scale;
                    if (s_buf[n] > m) m = s_buf[n];
                    ++n;
                }
                /* softmax-weighted values, in the same order */
                double l = 0.0;
                n = 0;
                for (int64_t j = 0; j < C; ++j, ++n) {
                    double e = exp(s_buf[n] - m);
                    const uint8_t* vr = v_cache + ((size_t)(c0 + j) * Hkv + h) * D;
                    l += e;
                    for (int d = 0; d < D; ++d) out[d] += e * (v_scale * e4m3_to_f64(vr[d]));
                }
                for (int k = 0; k < Pb; ++k) {
                    if (!(row[k / 32] & (1u << (k % 32)))) continue;
                    double e = exp(s_buf[n] - m);
                    const uint16_t* vr = v_new + (((size_t)b * P_max + k) * Hkv + h) * D;
                    l += e;
                    for (int d = 0; d < D; ++d) out[d] += e * bf16_to_f64(vr[d]);
                    ++n;
                }
                for (int d = 0; d < D; ++d) out[d] /= l;
            }
        }
    }
    free(s_buf);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* stochastic verification: multi-step speculative sampling over the tree    */
/* ------------------------------------------------------------------------ */
/*
 * Rejection sampling (speculative-decoding survey page, rejection-sampling
 * paragraph): a token x proposed by the draft distribution q is kept when
 * u < p(x) / q(x), u ~ U(0,1), p the target distribution.  Multi-step
 * speculative sampling (same page, SpecInfer "Token Tree Verifier"): the
 * children of the current tree node are tested in turn; after each rejection
 * the target becomes the normalised residual max(0, p - q); if every child is
 * rejected, or the node has no child, one token is drawn from the current
 * target and the walk ends.
 *
 * Readings (the pages leave these open):
 *  - p(.|n) = softmax(target_logits[n] / T), q(.|n) = softmax(draft_logits[n] / T):
 *    the LLM's and the drafter's next-token distributions after node n;
 *  - the walk starts at packed node 0 (beam 0's anchor); the children of node
 *    n are the packed nodes whose parent is n, tested in increasing packed
 *    index; the test u * q(x) < p(x) is the ratio test without the division;
 *  - a residual whose mass is 0 leaves the target unchanged;
 *  - a draw from a distribution R is the exponential race
 *    argmin_y E_y / R(y) with E_y = -ln(u_sample[b][y]) (lowest y on ties),
 *    which draws y with probability R(y) / sum R;
 *  - the emitted tokens are the accepted drafts and the drawn token;
 *    best_beam is the lowest beam whose prefix is the accepted walk;
 *    accept_len[w] is how many of beam w's leading drafts lie on the walk.
 * margin[b] (optional) returns the smallest relative gap of any decision taken
 * for request b (the two sides of a ratio test; the best and second-best race
 * keys), so that callers can tell a well-conditioned decision from a tie.
 */
static void softmax_row(const uint16_t* row, int V, double inv_T, double* out)
{
    double mx = -INFINITY, sum = 0.0;
    for (int v = 0; v < V; ++v) {
        double x = bf16_to_f64(row[v]) * inv_T;
        if (x > mx) mx = x;
    }
    for (int v = 0; v < V; ++v) {
        out[v] = exp(bf16_to_f64(row[v]) * inv_T - mx);
        sum += out[v];
    }
    for (int v = 0; v < V; ++v) out[v] /= sum;
}

static double rel_gap(double a, double b)
{
    double m = fabs(a) > fabs(b) ? fabs(a) : fabs(b);
    return m > 0.0 ? fabs(a - b) / m : 0.0;
}

int oracle_sample_accept(const uint16_t* target, const uint16_t* draft, int B, int P_max, int V,
                         double temperature, const int32_t* beams, const int32_t* packer,
                         const int32_t* unpacker, const int32_t* packed_len, int W, int L,
                         const float* u_accept, const float* u_sample, int32_t* accept_len,
                         int32_t* best_beam, int32_t* n_accepted, int32_t* out_tokens,
                         double* margin)
{
    if (B < 0 || P_max <= 0 || V <= 0 || W <= 0 || L <= 0 || !(temperature > 0.0)) return -1;
    const double inv_T = 1.0 / temperature;
    double* p = (double*)malloc(sizeof(double) * V);
    double* q = (double*)malloc(sizeof(double) * V);
    int32_t* walk = (int32_t*)malloc(sizeof(int32_t) * L);
    if (!p || !q || !walk) { free(p); free(q); free(walk); return -2; }
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        const int Pb = packed_len[b];
        if (Pb < 1 || Pb > P_max) { rc = -1; break; }
        const int32_t* bb = beams + (size_t)b * W * L;
        const int32_t* pk = packer + (size_t)b * P_max;
        const int32_t* up = unpacker + (size_t)b * W * L;
        double worst = 1.0;
        int node = 0, a = 0;
        walk[0] = 0;
        for (;;) {
            const uint16_t* trow = target + ((size_t)b * P_max + node) * V;
            const uint16_t* drow = draft + ((size_t)b * P_max + node) * V;
            softmax_row(trow, V, inv_T, p);          /* p: the current target */
            softmax_row(drow, V, inv_T, q);
            int accepted = -1;
            for (int c = node + 1; c < Pb && accepted < 0; ++c) {
                const int f = pk[c], w = f / L, i = f % L;
                if (i == 0 || up[w * L + i - 1] != node) continue;   /* not a child */
                const int x = bb[w * L + i];
                if (x < 0 || x >= V) { rc = -1; break; }
                const double lhs = (double)u_accept[(size_t)b * P_max + c] * q[x];
                const double g = rel_gap(lhs, p[x]);
                if (g < worst) worst = g;
                if (lhs < p[x]) {
                    accepted = c;
                } else {                              /* residual max(0, p - q) */
                    double Z = 0.0;
                    for (int v = 0; v < V; ++v) Z += (p[v] > q[v] ? p[v] - q[v] : 0.0);
                    if (Z > 0.0)
                        for (int v = 0; v < V; ++v) p[v] = (p[v] > q[v] ? p[v] - q[v] : 0.0) / Z;
                }
            }
            if (rc) break;
            if (accepted >= 0) {
                const int f = pk[accepted];
                out_tokens[(size_t)b * L + a] = bb[f];
                ++a;
                walk[a] = accepted;
                node = accepted;
                continue;
            }
            /* draw one token from p: the exponential race */
            const float* us = u_sample + (size_t)b * V;
            double k1 = INFINITY, k2 = INFINITY;
            int y1 = -1;
            for (int v = 0; v < V; ++v) {
                if (!(p[v] > 0.0)) continue;
                const double key = -log((double)us[v]) / p[v];
                if (key < k1) { k2 = k1; k1 = key; y1 = v; }
                else if (key < k2) k2 = key;
            }
            if (y1 < 0) { rc = -1; break; }
            if (isfinite(k2)) {
                const double g = (k2 - k1) / k2;
                if (g < worst) worst = g;
            }
            out_tokens[(size_t)b * L + a] = y1;
            break;
        }
        if (rc) break;
        for (int j = a + 1; j < L; ++j) out_tokens[(size_t)b * L + j] = -1;
        n_accepted[b] = a;
        int best = -1;
        for (int w = 0; w < W; ++w) {
            int n = -1;
            while (n + 1 <= a && up[w * L + n + 1] == walk[n + 1]) ++n;
            accept_len[(size_t)b * W + w] = n < 0 ? 0 : n;
            if (n == a && best < 0) best = w;
        }
        best_beam[b] = best;
        if (margin) margin[b] = worst;
    }
    free(p); free(q); free(walk);
    return rc;
}
