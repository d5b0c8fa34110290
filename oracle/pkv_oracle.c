/*
 * pkv_oracle.c -- plain, slow, fp64 CPU oracle for the paged-KV decode step
 * of a Qwen3-style attention layer (QK-norm -> RoPE -> page-slot append ->
 * grouped-query attention over the row's pages).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the reference the GPU path is
 * checked against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the product path never calls it and shares
 * no code, header, table or constant with it.
 *
 * Sources (web pages, cited by title and section):
 *   [NEST]  "qwen3-8b" model files on nest.franknoh.dev: README.md (Entries,
 *           Shards), src/attention.linnet (GroupedQueryAttention: decode_rows,
 *           decode_paged, prefill_paged, step_paged, split_heads),
 *           src/lib.linnet (Model entries decode_paged / prefill_paged /
 *           step_paged), src/norm.linnet (RmsNorm), src/rope.linnet (tables).
 *   [ZIG]   fantasma src/inference/model.zig: loadWeights (RoPE tables),
 *           fullAttentionForward (QK-norm, RoPE, GQA head map, softmax),
 *           applyRope (rotate-half form).
 *
 * Numerics: every bf16 input is widened exactly to double; all arithmetic is
 * in double; the only roundings are of the K values written to the pool
 * (round-to-nearest-even straight from double to bf16) and, for callers that
 * want it, of the output.  No intermediate is rounded to bf16 (the pages'
 * torch backend types intermediates as T; this oracle takes the exact
 * mathematical value, and the GPU path is held to a tolerance against it).
 *
 * Parity pins: every function here is pinned by tests that do not retype it
 * (closed forms, invariants, library routines such as torch's RMSNorm and
 * scaled-dot-product attention in fp64, brute force on tiny inputs).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int heads;        /* query heads (Heads) */
    int kv_heads;     /* key/value heads (KvHeads) */
    int head_dim;     /* HeadDim */
    int page_size;    /* PageSize */
    int max_seq;      /* MaxSeq: bound on positions */
    double rope_theta;
    double eps;
    int rotary_dim;   /* dims rotated by RoPE (the first rotary_dim); 0 = head_dim */
} orc_config;

/* Error bits reported for tokens the oracle skips (zero output, no write).
 * They describe the same conditions the library documents for its device
 * error word. */
enum {
    ORC_ERR_POSITION = 1u, /* position < 0, >= max_seq, or beyond the table */
    ORC_ERR_PAGE = 2u,     /* a table entry the token reads is not a pool page */
    ORC_ERR_ROW = 4u,      /* a prefill token names a row outside the table */
    ORC_ERR_SLOT = 8u      /* an explicit prefill slot is outside the pool */
};

/* ---- bf16 <-> double ------------------------------------------------- */

/* bf16 is the top 16 bits of an IEEE binary32; widening is exact. */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16, ties to even, in ONE step (no detour
 * through binary32, which could round twice).  bf16 keeps 8 significant bits
 * and binary32's exponent range: normal numbers >= 2^-126, subnormals with
 * quantum 2^-133, overflow to infinity at or above 2^128 after rounding. */
uint16_t orc_round_bf16(double x)
{
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (isinf(ax)) return sign | 0x7F80;
    if (ax == 0.0) return sign;
    double quantum;
    if (ax < ldexp(1.0, -126)) {
        quantum = ldexp(1.0, -133);
    } else {
        int e;
        frexp(ax, &e);              /* ax in [2^(e-1), 2^e) */
        quantum = ldexp(1.0, e - 8); /* 8 significant bits */
    }
    /* ax / quantum is exact (power of two); nearbyint rounds ties to even
     * under the default rounding mode. */
    double r = nearbyint(ax / quantum) * quantum;
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

void orc_round_bf16_array(const double* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = orc_round_bf16(x[i]);
}

/* ---- a2: per-head QK-norm ------------------------------------------------
 * [NEST] src/norm.linnet RmsNorm.forward = rms_norm(x, weight, 1e-6) over the
 * last axis; README.md: applied to every head's head_dim-wide slice after
 * split_heads, before rope.  [ZIG] fullAttentionForward normalises each q and
 * k head with the q_norm / k_norm weights.  Reading: y = x / sqrt(mean(x^2) +
 * eps) * w  (eps inside the root, weight after normalising). */
void orc_qk_norm(const orc_config* c, const uint16_t* x, const uint16_t* w, double* y)
{
    const int D = c->head_dim;
    double ss = 0.0;
    for (int i = 0; i < D; ++i) {
        double xi = orc_bf16_to_double(x[i]);
        ss += xi * xi;
    }
    double r = sqrt(ss / (double)D + c->eps);
    for (int i = 0; i < D; ++i) y[i] = (orc_bf16_to_double(x[i]) / r) * orc_bf16_to_double(w[i]);
}

/* ---- a3: rotate-half RoPE ------------------------------------------------
 * [NEST] src/rope.linnet tables: inv_freq[i] = theta^(-2i/D) for i < D/2,
 * angle = pos * inv_freq[i], tables are concat(angles, angles).  [ZIG]
 * applyRope: the rotate-half form, x*cos + rotate_half(x)*sin with
 * rotate_half(x) = concat(-x2, x1), over the first rotary_dim = R dims only
 * (Qwen3: R = D; the hybrid model of the Zig page rotates part of each head,
 * its tables built with inv_freq[i] = theta^(-2i/R)).  So for i < R/2:
 *   y[i]       = x[i]       cos(a_i) - x[i+R/2] sin(a_i)
 *   y[i+R/2]   = x[i+R/2]   cos(a_i) + x[i]     sin(a_i)
 * and y[d] = x[d] for d >= R.  Angles are formed in double (the pages use
 * f32; see the readings). */
void orc_rope(const orc_config* c, double* y, int pos)
{
    const int R = (c->rotary_dim > 0 && c->rotary_dim < c->head_dim) ? c->rotary_dim : c->head_dim, half = R / 2;
    for (int i = 0; i < half; ++i) {
        double inv_freq = pow(c->rope_theta, -2.0 * (double)i / (double)R);
        double a = (double)pos * inv_freq;
        double cs = cos(a), sn = sin(a);
        double x1 = y[i], x2 = y[i + half];
        y[i] = x1 * cs - x2 * sn;
        y[i + half] = x2 * cs + x1 * sn;
    }
}

/* ---- a1: page slot ---------------------------------------------------------
 * [NEST] README.md Entries (decode_paged): row b's positions lie in the pages
 * table[b] lists, PageSize positions each; attention.linnet decode_paged uses
 * page_slots(table, positions).  Position p of row b lives at slot
 * table[b][p / PageSize] * PageSize + p % PageSize of the pool. */
int64_t orc_page_slot(const orc_config* c, const int32_t* table, int pages, int row, int pos)
{
    int32_t page = table[(int64_t)row * pages + pos / c->page_size];
    return (int64_t)page * c->page_size + pos % c->page_size;
}

/* ---- a5: attention of one query over one row's pages ---------------------
 * [NEST] attention.linnet decode_paged: paged_attention(q, cache_k, cache_v,
 * table, positions, rsqrt(HeadDim)); decode_rows spells the mask as
 * seen[b, s] = s <= positions[b] (inclusive: the query sees the key it has
 * just written).  [ZIG] fullAttentionForward: scores q.k * scale, max-
 * subtracted exp, normalised, then the weighted sum of values.
 * Plain definition: gather the row's keys for s = 0..pos, then softmax. */
void orc_attend(const orc_config* c, const uint16_t* K, const uint16_t* V, int64_t num_slots,
                const int32_t* table, int pages, int row, int pos, int g,
                const double* qhat, double* out)
{
    const int D = c->head_dim;
    const int L = pos + 1;
    const double scale = 1.0 / sqrt((double)D);
    double* z = (double*)malloc(sizeof(double) * (size_t)L);
    int64_t* slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)L);
    double zmax = -INFINITY;
    for (int s = 0; s < L; ++s) {
        slot[s] = orc_page_slot(c, table, pages, row, s);
        const uint16_t* ks = K + ((int64_t)g * num_slots + slot[s]) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qhat[d] * orc_bf16_to_double(ks[d]);
        z[s] = dot * scale;
        if (z[s] > zmax) zmax = z[s];
    }
    double denom = 0.0;
    for (int s = 0; s < L; ++s) {
        z[s] = exp(z[s] - zmax);
        denom += z[s];
    }
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int s = 0; s < L; ++s) {
        const uint16_t* vs = V + ((int64_t)g * num_slots + slot[s]) * D;
        double wgt = z[s] / denom;
        for (int d = 0; d < D; ++d) out[d] += wgt * orc_bf16_to_double(vs[d]);
    }
    free(z);
    free(slot);
}

/* ---- a6 (second formulation, used by the pins) ----------------------------
 * The same attention computed page range by page range: each range r yields
 * its own max m_r, denominator l_r and normalised output o_r; the ranges are
 * merged by o = sum_r e^{m_r - M} l_r o_r / sum_r e^{m_r - M} l_r.  This is an
 * exact re-association of orc_attend (the split-KV decomposition); split[]
 * holds nsplit+1 increasing positions, split[0] = 0 and split[nsplit] = pos+1. */
void orc_attend_split(const orc_config* c, const uint16_t* K, const uint16_t* V, int64_t num_slots,
                      const int32_t* table, int pages, int row, int pos, int g,
                      const double* qhat, int nsplit, const int32_t* split, double* out)
{
    const int D = c->head_dim;
    const double scale = 1.0 / sqrt((double)D);
    double* m = (double*)malloc(sizeof(double) * (size_t)nsplit);
    double* l = (double*)malloc(sizeof(double) * (size_t)nsplit);
    double* o = (double*)calloc((size_t)nsplit * (size_t)D, sizeof(double));
    for (int r = 0; r < nsplit; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.0;
        int n = split[r + 1] - split[r];
        double* z = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        for (int s = split[r]; s < split[r + 1]; ++s) {
            int64_t sl = orc_page_slot(c, table, pages, row, s);
            const uint16_t* ks = K + ((int64_t)g * num_slots + sl) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qhat[d] * orc_bf16_to_double(ks[d]);
            z[s - split[r]] = dot * scale;
            if (z[s - split[r]] > m[r]) m[r] = z[s - split[r]];
        }
        for (int s = split[r]; s < split[r + 1]; ++s) {
            int64_t sl = orc_page_slot(c, table, pages, row, s);
            const uint16_t* vs = V + ((int64_t)g * num_slots + sl) * D;
            double e = exp(z[s - split[r]] - m[r]);
            l[r] += e;
            for (int d = 0; d < D; ++d) o[(int64_t)r * D + d] += e * orc_bf16_to_double(vs[d]);
        }
        if (l[r] > 0.0)
            for (int d = 0; d < D; ++d) o[(int64_t)r * D + d] /= l[r];
        free(z);
    }
    double M = -INFINITY;
    for (int r = 0; r < nsplit; ++r)
        if (m[r] > M) M = m[r];
    double den = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int r = 0; r < nsplit; ++r) {
        if (l[r] == 0.0) continue;
        double wr = exp(m[r] - M) * l[r];
        den += wr;
        for (int d = 0; d < D; ++d) out[d] += wr * o[(int64_t)r * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] /= den;
    free(m);
    free(l);
    free(o);
}

/* ---- validity of one token --------------------------------------------------
 * A token whose position or pages cannot be read is skipped: no write, a zero
 * output, and an error bit.  (The pages state no behaviour for bad inputs;
 * this is the library's documented contract.) */
static uint32_t token_check(const orc_config* c, const int32_t* table, int rows, int pages, int num_pages,
                            int row, int pos)
{
    if (row < 0 || row >= rows) return ORC_ERR_ROW;
    if (pos < 0 || pos >= c->max_seq || pos >= pages * c->page_size) return ORC_ERR_POSITION;
    for (int p = 0; p <= pos / c->page_size; ++p) {
        int32_t id = table[(int64_t)row * pages + p];
        if (id < 0 || id >= num_pages) return ORC_ERR_PAGE;
    }
    return 0;
}

/* ---- threaded attention over (token, head) tasks ------------------------- */
typedef struct {
    const orc_config* c;
    const uint16_t *K, *V, *q, *qw;
    int64_t num_slots;
    const int32_t* table;
    int pages;
    const int32_t* tok_row;
    const int32_t* tok_pos;
    const int32_t* tasks; /* token index per task (all heads of that token) */
    int ntasks;
    double* out;
    int next; /* shared counter */
} attend_job;

static void* attend_worker(void* arg)
{
    attend_job* J = (attend_job*)arg;
    const orc_config* c = J->c;
    const int H = c->heads, D = c->head_dim, group = c->heads / c->kv_heads;
    double* qhat = (double*)malloc(sizeof(double) * (size_t)D);
    for (;;) {
        int i = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (i >= J->ntasks * H) break;
        int t = J->tasks[i / H];
        int h = i % H;
        double* o = J->out + ((int64_t)t * H + h) * D;
        if (J->tok_pos[t] < 0) { /* skipped token: zero output */
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            continue;
        }
        /* [NEST] decode_paged: q = rope_rows(q_norm(split_heads(q))) */
        orc_qk_norm(c, J->q + ((int64_t)t * H + h) * D, J->qw, qhat);
        orc_rope(c, qhat, J->tok_pos[t]);
        /* [ZIG] fullAttentionForward: kv head = h / (heads / kv_heads) */
        orc_attend(c, J->K, J->V, J->num_slots, J->table, J->pages, J->tok_row[t], J->tok_pos[t],
                   h / group, qhat, o);
    }
    free(qhat);
    return NULL;
}

/* ---- a7/a8: step_paged ------------------------------------------------------
 * [NEST] attention.linnet step_paged: the P prompt tokens (token p at
 * positions[p] of row rows[p], written at slots[p]) and the Rows step tokens
 * (row b at step_positions[b], slot page_slots(table, step_positions)) are
 * normed, roped and ALL written to the pool first; then the prompt tokens
 * attend (paged_prefill_attention over table[rows[p]] up to positions[p]) and
 * the step rows attend (paged_attention up to step_positions[b]); the output
 * is concat(prompts, steps) in token order.  decode_paged is the case P = 0.
 *
 * Extension: step_positions[b] = -1 marks a row that takes no step (no
 * write, zero output, no error).  slots may be NULL: each prompt token's slot
 * is then derived from the table as for step rows.
 *
 * K, V: bf16 pools [kv_heads][num_pages * page_size][head_dim], updated in
 * place.  q [P+rows][heads][head_dim], k/v [P+rows][kv_heads][head_dim].
 * sel lists the token indices whose outputs are computed (NULL: all); out is
 * [P+rows][heads][head_dim] doubles (rows not selected are left untouched).
 * err_bits receives the OR of the error bits of skipped tokens.
 * Returns 0, or -1 on a malformed call. */
int orc_step(const orc_config* c, uint16_t* K, uint16_t* V, int num_pages,
             const uint16_t* q, const uint16_t* k, const uint16_t* v,
             const uint16_t* q_norm_w, const uint16_t* k_norm_w,
             const int32_t* positions, const int32_t* prow, const int32_t* slots,
             const int32_t* step_positions, const int32_t* table,
             int P, int rows, int pages,
             const int32_t* sel, int nsel, double* out, uint32_t* err_bits, int nthreads)
{
    if (!c || !K || !V || !q || !k || !v || !q_norm_w || !k_norm_w || !table || !out) return -1;
    if (P < 0 || rows < 0 || P + rows <= 0 || pages <= 0 || num_pages <= 0) return -1;
    if (c->heads % c->kv_heads != 0 || c->head_dim % 2 != 0) return -1;
    if (P > 0 && (!positions || !prow)) return -1;
    if (rows > 0 && !step_positions) return -1;
    const int N = P + rows, G = c->kv_heads, D = c->head_dim;
    const int64_t num_slots = (int64_t)num_pages * c->page_size;
    int32_t* tok_row = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    int32_t* tok_pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    uint32_t err = 0;
    double* kh = (double*)malloc(sizeof(double) * (size_t)D);

    /* Writes, in token order, before any attention. */
    for (int t = 0; t < N; ++t) {
        int row, pos;
        int64_t slot;
        if (t < P) {
            row = prow[t];
            pos = positions[t];
        } else {
            row = t - P;
            pos = step_positions[t - P];
            if (pos == -1) { /* row takes no step */
                tok_row[t] = row;
                tok_pos[t] = -1;
                continue;
            }
        }
        uint32_t e = token_check(c, table, rows, pages, num_pages, row, pos);
        if (!e) {
            if (t < P && slots) {
                slot = slots[t];
                if (slot < 0 || slot >= num_slots) e = ORC_ERR_SLOT;
            } else {
                slot = orc_page_slot(c, table, pages, row, pos);
            }
        }
        if (e) {
            err |= e;
            tok_row[t] = row;
            tok_pos[t] = -1;
            continue;
        }
        tok_row[t] = row;
        tok_pos[t] = pos;
        for (int g = 0; g < G; ++g) {
            /* [NEST] k = rope_rows(k_norm(split_heads(k))); write_tokens */
            orc_qk_norm(c, k + ((int64_t)t * G + g) * D, k_norm_w, kh);
            orc_rope(c, kh, pos);
            uint16_t* kd = K + ((int64_t)g * num_slots + slot) * D;
            uint16_t* vd = V + ((int64_t)g * num_slots + slot) * D;
            const uint16_t* vs = v + ((int64_t)t * G + g) * D;
            for (int d = 0; d < D; ++d) {
                kd[d] = orc_round_bf16(kh[d]);
                vd[d] = vs[d]; /* v is written as given */
            }
        }
    }
    free(kh);

    /* Attention for the selected tokens. */
    int32_t* tasks;
    int ntasks;
    if (sel) {
        tasks = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nsel > 0 ? nsel : 1));
        ntasks = 0;
        for (int i = 0; i < nsel; ++i)
            if (sel[i] >= 0 && sel[i] < N) tasks[ntasks++] = sel[i];
    } else {
        tasks = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
        for (int t = 0; t < N; ++t) tasks[t] = t;
        ntasks = N;
    }
    attend_job J = {c, K, V, q, q_norm_w, num_slots, table, pages, tok_row, tok_pos, tasks, ntasks, out, 0};
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&th[started], NULL, attend_worker, &J) == 0) ++started;
    attend_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);

    free(tasks);
    free(tok_row);
    free(tok_pos);
    if (err_bits) *err_bits = err;
    return 0;
}

/* decode_paged: step_paged with no prompt tokens.
 * [NEST] attention.linnet decode_paged / lib.linnet Model.decode_paged. */
int orc_decode(const orc_config* c, uint16_t* K, uint16_t* V, int num_pages,
               const uint16_t* q, const uint16_t* k, const uint16_t* v,
               const uint16_t* q_norm_w, const uint16_t* k_norm_w,
               const int32_t* positions, const int32_t* table, int rows, int pages,
               const int32_t* sel, int nsel, double* out, uint32_t* err_bits, int nthreads)
{
    return orc_step(c, K, V, num_pages, q, k, v, q_norm_w, k_norm_w, NULL, NULL, NULL, positions, table,
                    0, rows, pages, sel, nsel, out, err_bits, nthreads);
}
