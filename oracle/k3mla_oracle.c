/*
 * k3mla_oracle.c -- plain, slow CPU oracle for absorbed multi-head latent
 * attention (MLA) decode over a paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only tests/, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes is taken from pegainfer PR #869, "K3: paged latent MLA KV +
 * absorbed decode":
 *   - cache geometry (M1 commit, "paged latent cache" paragraph): one
 *     page-first slab [page][mla_layer][64 tokens][576] bf16, each row the
 *     512-wide kv latent c_t followed by the 64-wide shared rope key; a per-slot
 *     int32 block table; a -1 entry reads as an all-zero latent;
 *   - the appended row lands at slab row ((page * L + layer) * 64 + pos % 64),
 *     with a size_t element index (M1 commit, "indexed row write" sentence);
 *   - the per-head math (M2 commit, first paragraph):
 *       score(t) = (W_UK[h]^T q_nope)^T c_t + q_rope^T k_rope_t,
 *       o[h]     = W_UV[h] (sum_t p_t c_t),
 *     with W_UK / W_UV read in place from w_kv_b;
 *   - the certified rounding chain (M2 commit, "rounding chain" sentence):
 *       1. q absorption lands bf16;
 *       2. f32 score dot over the 576 row entries in ascending order, lands bf16;
 *       3. that bf16 dot times the bf16 scale, landed bf16;
 *       4. f32 max and f32 sum of exp in a fixed order;
 *       5. probabilities land bf16 after normalising;
 *       6. f32 latent accumulation over ascending t, lands bf16;
 *       7. f32 W_UV expansion, lands bf16.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - w_kv_b is [96*256][512]; rows h*256 .. h*256+127 are W_UK[h] (row d,
 *     column j) and rows h*256+128 .. h*256+255 are W_UV[h] (row v, column j).
 *   - Every f32 sum not given an order by the pages runs in ascending index,
 *     one rounding per addition (no fused multiply-add: every product here is
 *     of two bf16 values and therefore exact in f32 anyway).
 *   - exp(x) is computed as (float)exp((double)x) with the C library's double
 *     exp, rounded once to f32.
 *   - Normalisation is the IEEE f32 quotient e_t / l, then rounded to bf16.
 *   - A -1 table entry inside the context is a token whose row is all zero: it
 *     takes part in the softmax with score 0 and adds nothing to the latent sum.
 *   - Rows at logical positions >= ctx_len are not read at all.
 *   - ctx_len == 0 gives an all-zero output row and argmax -1.
 *   - The argmax of the attention probabilities is the lowest logical t whose
 *     bf16 probability is the largest.
 *   - bf16 rounding is round-to-nearest-even from f32; NaN stays NaN.
 *
 * A "mutation" argument plants a known mistake so that tests can show each
 * pin catches it.  0 is the faithful oracle; any other value is wrong on
 * purpose and exists only for those negative-control tests.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define K3O_H 96
#define K3O_NOPE 128
#define K3O_ROPE 64
#define K3O_QDIM (K3O_NOPE + K3O_ROPE) /* 192 */
#define K3O_V 128
#define K3O_LORA 512
#define K3O_ROW (K3O_LORA + K3O_ROPE) /* 576 */
#define K3O_PAGE 64
#define K3O_WROWS_PER_HEAD (K3O_NOPE + K3O_V) /* 256 */

/* planted mistakes (negative controls only) */
enum {
    MUT_NONE = 0,
    MUT_DROP_ROPE = 1,      /* score ignores the rope half */
    MUT_SWAP_WUK_WUV = 2,   /* expansion reads W_UK rows instead of W_UV rows */
    MUT_NO_SCALE = 3,       /* scale multiply skipped */
    MUT_PAGE_OFF_BY_ONE = 4,/* logical page index shifted by one */
    MUT_DROP_LAST_IN_SUM = 5,/* normaliser misses the last token */
    MUT_TRANSPOSE_WUK = 6,  /* absorption indexes W_UK[h] as [j][d] */
    MUT_LAYER_IGNORED = 7,  /* slab row ignores the layer index */
    MUT_ROPE_SIGN = 8,      /* rope term subtracted */
};

/* ---- bf16 <-> f32 ---------------------------------------------------- */

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round-to-nearest, ties to even, from f32 to bf16.  NaN is kept NaN (quiet). */
static uint16_t f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    uint32_t rounded = u + 0x7FFFu + lsb;
    return (uint16_t)(rounded >> 16);
}

static float round_bf16(float f) { return bf16_to_f32(f32_to_bf16(f)); }

/* Exported for the pin that compares this rounding with a library routine. */
void k3o_f32_to_bf16(const float* x, uint16_t* y, size_t n)
{
    for (size_t i = 0; i < n; ++i) y[i] = f32_to_bf16(x[i]);
}

/* ---- step 1: q absorption -------------------------------------------- */

/* q      [B][96][192] bf16 (q_nope 0..127 | q_rope 128..191)
 * w_kv_b [96*256][512] bf16
 * q_abs  [B][96][576] bf16: [ bf16(W_UK[h]^T q_nope) (512) | q_rope (64) ]
 * q_abs[j] = bf16( sum_{d=0..127 ascending} W_UK[h][d][j] * q_nope[d] ) */
void k3o_absorb(const uint16_t* q, const uint16_t* w_kv_b, int B, uint16_t* q_abs, int mutation)
{
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < K3O_H; ++h) {
            const uint16_t* qn = q + ((size_t)b * K3O_H + h) * K3O_QDIM;
            const uint16_t* wuk = w_kv_b + (size_t)h * K3O_WROWS_PER_HEAD * K3O_LORA;
            uint16_t* qa = q_abs + ((size_t)b * K3O_H + h) * K3O_ROW;
            for (int j = 0; j < K3O_LORA; ++j) {
                float acc = 0.0f;
                for (int d = 0; d < K3O_NOPE; ++d) {
                    float w;
                    if (mutation == MUT_TRANSPOSE_WUK)
                        w = bf16_to_f32(wuk[(size_t)j * K3O_NOPE + d]);
                    else
                        w = bf16_to_f32(wuk[(size_t)d * K3O_LORA + j]);
                    float prod = w * bf16_to_f32(qn[d]);
                    acc = acc + prod;
                }
                qa[j] = f32_to_bf16(acc);
            }
            for (int r = 0; r < K3O_ROPE; ++r) qa[K3O_LORA + r] = qn[K3O_NOPE + r];
        }
    }
}

/* ---- cache row lookup ---------------------------------------------------- */

typedef struct {
    const uint16_t* slab;
    int n_pages;
    int n_layers;
    int layer;
    const int32_t* table;
    int max_pages;
} k3o_cache;

/* Row of logical token t of slot b, or NULL for a -1 (zero-latent) entry.
 * Returns -2 through *bad when the table holds an id outside [-1, n_pages). */
static const uint16_t* cache_row(const k3o_cache* c, int b, int t, int mutation, int* bad)
{
    int lp = t / K3O_PAGE;
    if (mutation == MUT_PAGE_OFF_BY_ONE) lp = (lp + 1) % c->max_pages;
    int32_t id = c->table[(size_t)b * c->max_pages + lp];
    if (id < 0) {
        if (id != -1) *bad = 1;
        return NULL;
    }
    if (id >= c->n_pages) {
        *bad = 1;
        return NULL;
    }
    int layer = (mutation == MUT_LAYER_IGNORED) ? 0 : c->layer;
    size_t row = ((size_t)id * (size_t)c->n_layers + (size_t)layer) * K3O_PAGE + (size_t)(t % K3O_PAGE);
    return c->slab + row * K3O_ROW;
}

/* ---- steps 2-7 for one (slot, head) ---------------------------------------- */

typedef struct {
    const uint16_t* q_abs;  /* [B][96][576] */
    k3o_cache cache;
    const int32_t* ctx_len; /* [B] */
    const uint16_t* w_kv_b;
    uint16_t scale;
    uint16_t* out;          /* [B][96][128] */
    int32_t* argmax;        /* [B][96] or NULL */
    uint16_t* o_lat;        /* [B][96][512] or NULL */
    uint16_t* probs;        /* [B][96][probs_stride] or NULL (bf16 p_t) */
    float* scores;          /* [B][96][probs_stride] or NULL (bf16-valued s_t) */
    int probs_stride;
    int mutation;
    int bad_table;          /* set if a table id was outside [-1, n_pages) */
} k3o_job;

static void decode_one(k3o_job* J, int b, int h)
{
    const int n = J->ctx_len[b];
    uint16_t* o = J->out + ((size_t)b * K3O_H + h) * K3O_V;
    uint16_t* ol_out = J->o_lat ? J->o_lat + ((size_t)b * K3O_H + h) * K3O_LORA : NULL;
    if (n <= 0) {
        for (int v = 0; v < K3O_V; ++v) o[v] = 0;
        if (ol_out)
            for (int j = 0; j < K3O_LORA; ++j) ol_out[j] = 0;
        if (J->argmax) J->argmax[(size_t)b * K3O_H + h] = -1;
        return;
    }
    const uint16_t* qa = J->q_abs + ((size_t)b * K3O_H + h) * K3O_ROW;
    float Q[K3O_ROW];
    for (int k = 0; k < K3O_ROW; ++k) Q[k] = bf16_to_f32(qa[k]);
    const float scale = bf16_to_f32(J->scale);
    int bad = 0;

    /* steps 2-3: s_t = bf16( bf16(dot_t) * scale ) */
    float* s = (float*)malloc(sizeof(float) * (size_t)n);
    for (int t = 0; t < n; ++t) {
        const uint16_t* row = cache_row(&J->cache, b, t, J->mutation, &bad);
        float acc = 0.0f;
        if (row) {
            const int kmax = (J->mutation == MUT_DROP_ROPE) ? K3O_LORA : K3O_ROW;
            for (int k = 0; k < kmax; ++k) {
                float prod = Q[k] * bf16_to_f32(row[k]);
                if (J->mutation == MUT_ROPE_SIGN && k >= K3O_LORA) prod = -prod;
                acc = acc + prod;
            }
        } else {
            /* zero latent: every product is +0 (or -0); the sum is +0 */
            acc = 0.0f;
        }
        float dot = round_bf16(acc);
        s[t] = (J->mutation == MUT_NO_SCALE) ? dot : round_bf16(dot * scale);
    }

    /* step 4: m = max_t s_t; e_t = exp(s_t - m); l = sum_t e_t (ascending t) */
    float m = s[0];
    for (int t = 1; t < n; ++t)
        if (s[t] > m) m = s[t];
    float* e = (float*)malloc(sizeof(float) * (size_t)n);
    float l = 0.0f;
    for (int t = 0; t < n; ++t) {
        float x = s[t] - m;
        e[t] = (float)exp((double)x);
        if (!(J->mutation == MUT_DROP_LAST_IN_SUM && t == n - 1)) l = l + e[t];
    }

    /* step 5: p_t = bf16(e_t / l); argmax = lowest t with the largest p_t */
    float* p = (float*)malloc(sizeof(float) * (size_t)n);
    int am = 0;
    for (int t = 0; t < n; ++t) {
        p[t] = round_bf16(e[t] / l);
        if (p[t] > p[am]) am = t;
    }
    if (J->argmax) J->argmax[(size_t)b * K3O_H + h] = am;
    if (J->probs) {
        uint16_t* pp = J->probs + ((size_t)b * K3O_H + h) * J->probs_stride;
        for (int t = 0; t < n && t < J->probs_stride; ++t) pp[t] = f32_to_bf16(p[t]);
    }
    if (J->scores) {
        float* ss = J->scores + ((size_t)b * K3O_H + h) * J->probs_stride;
        for (int t = 0; t < n && t < J->probs_stride; ++t) ss[t] = s[t];
    }

    /* step 6: ol[j] = bf16( sum_{t ascending} p_t * c_t[j] ), j < 512 */
    float ol[K3O_LORA];
    for (int j = 0; j < K3O_LORA; ++j) ol[j] = 0.0f;
    for (int t = 0; t < n; ++t) {
        const uint16_t* row = cache_row(&J->cache, b, t, J->mutation, &bad);
        for (int j = 0; j < K3O_LORA; ++j) {
            float c = row ? bf16_to_f32(row[j]) : 0.0f;
            float prod = p[t] * c;
            ol[j] = ol[j] + prod;
        }
    }
    for (int j = 0; j < K3O_LORA; ++j) {
        ol[j] = round_bf16(ol[j]);
        if (ol_out) ol_out[j] = f32_to_bf16(ol[j]);
    }

    /* step 7: out[v] = bf16( sum_{j ascending} W_UV[h][v][j] * ol[j] ) */
    const size_t uv_first_row = (J->mutation == MUT_SWAP_WUK_WUV)
                                    ? (size_t)h * K3O_WROWS_PER_HEAD
                                    : (size_t)h * K3O_WROWS_PER_HEAD + K3O_NOPE;
    for (int v = 0; v < K3O_V; ++v) {
        const uint16_t* w = J->w_kv_b + (uv_first_row + (size_t)v) * K3O_LORA;
        float acc = 0.0f;
        for (int j = 0; j < K3O_LORA; ++j) {
            float prod = bf16_to_f32(w[j]) * ol[j];
            acc = acc + prod;
        }
        o[v] = f32_to_bf16(acc);
    }
    if (bad) J->bad_table = 1;
    free(s);
    free(e);
    free(p);
}

/* ---- work distribution over (slot, head); arithmetic per pair is unchanged --- */

typedef struct {
    k3o_job* job;
    const int32_t* slots;
    int n_slots;
    int next;
    pthread_mutex_t mu;
} k3o_pool;

static void* worker(void* arg)
{
    k3o_pool* P = (k3o_pool*)arg;
    for (;;) {
        pthread_mutex_lock(&P->mu);
        int i = P->next++;
        pthread_mutex_unlock(&P->mu);
        if (i >= P->n_slots * K3O_H) break;
        decode_one(P->job, P->slots[i / K3O_H], i % K3O_H);
    }
    return NULL;
}

/* Decode the slots listed in slots[0..n_slots) (indices into the batch).
 * Outputs are written at those slots' rows only.  Returns 0, or 1 when a table
 * entry held an id outside [-1, n_pages) (that entry was read as zero). */
int k3o_decode(const uint16_t* q_abs, const uint16_t* slab, int n_pages, int n_layers, int layer,
               const int32_t* block_table, int max_pages, const int32_t* ctx_len,
               const uint16_t* w_kv_b, uint16_t scale_bf16,
               const int32_t* slots, int n_slots,
               uint16_t* out, int32_t* argmax, uint16_t* o_lat,
               uint16_t* probs, float* scores, int probs_stride,
               int nthreads, int mutation)
{
    k3o_job J;
    J.q_abs = q_abs;
    J.cache.slab = slab;
    J.cache.n_pages = n_pages;
    J.cache.n_layers = n_layers;
    J.cache.layer = layer;
    J.cache.table = block_table;
    J.cache.max_pages = max_pages;
    J.ctx_len = ctx_len;
    J.w_kv_b = w_kv_b;
    J.scale = scale_bf16;
    J.out = out;
    J.argmax = argmax;
    J.o_lat = o_lat;
    J.probs = probs;
    J.scores = scores;
    J.probs_stride = probs_stride;
    J.mutation = mutation;
    J.bad_table = 0;
    if (nthreads < 1) nthreads = 1;
    k3o_pool P;
    P.job = &J;
    P.slots = slots;
    P.n_slots = n_slots;
    P.next = 0;
    pthread_mutex_init(&P.mu, NULL);
    if (nthreads == 1) {
        worker(&P);
    } else {
        pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &P);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&P.mu);
    return J.bad_table;
}

/* ---- the append: two indexed writes into the mapped page ---------------------- */

/* For each b with pos[b] >= 0: the slab row of (page = table[b][pos/64], layer,
 * pos % 64) receives c_kv[b][0..511] then k_rope[b][0..63].  Row index is
 * ((page * L + layer) * 64 + pos % 64) and the element index is that row times
 * 576, both in size_t.  Returns the number of rows that could not be written
 * (unmapped entry or id out of range); those rows are skipped. */
int k3o_append(uint16_t* slab, int n_pages, int n_layers, int layer,
               const int32_t* block_table, int max_pages, const int32_t* pos,
               const uint16_t* c_kv, long long c_stride, const uint16_t* k_rope, long long r_stride,
               int B)
{
    int skipped = 0;
    for (int b = 0; b < B; ++b) {
        int p = pos[b];
        if (p < 0) continue;
        int lp = p / K3O_PAGE;
        if (lp >= max_pages) {
            ++skipped;
            continue;
        }
        int32_t id = block_table[(size_t)b * max_pages + lp];
        if (id < 0 || id >= n_pages) {
            ++skipped;
            continue;
        }
        size_t row = ((size_t)id * (size_t)n_layers + (size_t)layer) * K3O_PAGE + (size_t)(p % K3O_PAGE);
        size_t elem = row * K3O_ROW;
        for (int j = 0; j < K3O_LORA; ++j) slab[elem + j] = c_kv[(size_t)b * c_stride + j];
        for (int r = 0; r < K3O_ROPE; ++r) slab[elem + K3O_LORA + r] = k_rope[(size_t)b * r_stride + r];
    }
    return skipped;
}
