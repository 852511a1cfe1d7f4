/*
 * sdpa_oracle.c -- plain fp64 CPU oracle for multi-head scaled dot-product
 * attention and the five-step multi-head layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference that the
 * CUDA path is checked against.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or helper with the CUDA library, and it includes nothing from it.
 *
 * What it computes (the plain definition, no tiling, no online softmax):
 *
 *   Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k) + M) V
 *     -- "04. Self-Attention：Transformer 的核心计算", section 四 (the four
 *        stages: scores, scale, row softmax, weighted sum) and section 七
 *        (the additive mask, -inf before the softmax);
 *     -- "attention-mechanism" page, sections "公式：为什么要除以 sqrt(d_k)"
 *        (scale is the per-head d_k) and "掩码：因果与 padding".
 *
 *   For each (b, head, query row i), in fp64, with n_b the keys of
 *   sequence b (kv_len[b] if PADDING, else Lk):
 *     J_i  = { j < n_b }  intersected with { j <= i } if CAUSAL
 *                         intersected with { j <= p_i } if CAUSAL_BR, where
 *                         p_i = n_b - Lq + i is the query's own position
 *     s_j  = scale * sum_c Q[i,c] K[j,c]          for j in J_i
 *     m    = max_j s_j                            (max subtraction, the
 *                                                  stable softmax form of the
 *                                                  "attention-mechanism" page,
 *                                                  section "最小实现")
 *     e_j  = exp(s_j - m),  l = sum_j e_j
 *     A_ij = e_j / l  (0 for j not in J_i)
 *     O[i] = sum_j e_j V[j] / l
 *     LSE[i] = m + log(l)
 *   A padded query row (PADDING without CAUSAL_BR, and i >= kv_len[b]) or a
 *   row whose J_i is empty (CAUSAL_BR and p_i < 0) has O[i] = 0 and
 *   LSE[i] = -inf.
 *
 *   Grouped-query attention ("Self-Attention 机制", section
 *   "MHA -> MQA -> GQA -> MLA"): with H query heads and Hkv key/value heads
 *   (H a multiple of Hkv), each run of H/Hkv consecutive query heads shares one
 *   K/V head: query head h reads K/V head h / (H/Hkv).  Hkv = H is ordinary
 *   multi-head attention, Hkv = 1 multi-query attention.
 *
 *   CAUSAL_BR is the causal mask aligned to the last key of each sequence
 *   instead of the first: the Lq queries are the sequence's last Lq tokens,
 *   so query i sits at position p_i = n_b - Lq + i and, by the look-ahead
 *   rule ("04. Self-Attention", section 七; "Self-Attention 机制", section
 *   "Causal Mask": a token never sees a later one), sees the keys j <= p_i.
 *   This is the reading for Lq new tokens decoded against a cache that
 *   already holds them (same page, the KV Cache of section
 *   "MHA -> MQA -> GQA -> MLA"): with per-sequence lengths (PADDING) each
 *   sequence's new tokens sit at its own end, and new token i never sees new
 *   token i + 1.  Without PADDING (n_b = Lk), and for Lq = Lk, it is the
 *   ordinary causal mask shifted by Lk - Lq.
 *
 *   The multi-head layer ("Self-Attention 机制", section "五步计算" and the
 *   shape trace in "维度全程跟踪"; "多模态大模型学习笔记（十四）", section 3.3):
 *     QKV = X W_QKV  (W_QKV is [d_model, 3 d_model], columns [Q | K | V])
 *     head i takes columns i*d_k .. (i+1)*d_k-1 of each block
 *     O_cat[:, i*d_k + c] = Attention(Q_i, K_i, V_i)[:, c]
 *     Y = O_cat W_O   (W_O is [d_model, d_model]); no biases.
 *   No intermediate is rounded: this is the mathematical result for the
 *   given bf16 inputs.
 *
 * Inputs are either bfloat16 bit patterns (uint16, widened exactly) or fp64.
 * Work is spread over POSIX threads by (batch, head, block of rows); each
 * row is computed independently in one thread, so results do not depend on
 * the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_MASK_CAUSAL 1
#define OR_MASK_PADDING 2
#define OR_MASK_CAUSAL_BR 4

#define OR_OK 0
#define OR_ERR_ARG (-1)
#define OR_ERR_NOMEM (-2)

static double widen_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double elem(const void *base, int is_bf16, size_t idx)
{
    if (is_bf16)
        return widen_bf16(((const uint16_t *)base)[idx]);
    return ((const double *)base)[idx];
}

/*
 * One query row against the keys [0, n_keys): the definition above.
 * q: d_k values; K, V: rows with strides k_stride / v_stride (doubles).
 * s: scratch of n_keys doubles.  Writes o[d_v], *lse, and (if a_row) the
 * n_keys weights.
 */
static void attend_row(const double *q, const double *K, size_t k_stride,
                       const double *V, size_t v_stride, int n_keys, int d_k, int d_v,
                       double scale, double *s, double *o, double *lse, double *a_row)
{
    int j, c;
    double m, l;
    if (n_keys <= 0) {
        for (c = 0; c < d_v; ++c)
            o[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    /* stage 1 + 2: scores and scale */
    for (j = 0; j < n_keys; ++j) {
        const double *k = K + (size_t)j * k_stride;
        double dot = 0.0;
        for (c = 0; c < d_k; ++c)
            dot += q[c] * k[c];
        s[j] = scale * dot;
    }
    /* stage 3: softmax with max subtraction */
    m = s[0];
    for (j = 1; j < n_keys; ++j)
        if (s[j] > m)
            m = s[j];
    l = 0.0;
    for (j = 0; j < n_keys; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    /* stage 4: weighted sum of values */
    for (c = 0; c < d_v; ++c)
        o[c] = 0.0;
    for (j = 0; j < n_keys; ++j) {
        const double *v = V + (size_t)j * v_stride;
        for (c = 0; c < d_v; ++c)
            o[c] += s[j] * v[c];
    }
    for (c = 0; c < d_v; ++c)
        o[c] /= l;
    if (a_row)
        for (j = 0; j < n_keys; ++j)
            a_row[j] = s[j] / l;
    *lse = m + log(l);
}

/*
 * Number of keys query row i of a sequence may attend to (J_i is always a
 * prefix).  kv_len is the sequence's own length when PADDING is set.
 */
static int valid_keys(int i, int Lq, int Lk, int mask_kind, int kv_len)
{
    const int padding = (mask_kind & OR_MASK_PADDING) != 0;
    const int n_seq = padding ? kv_len : Lk; /* keys of this sequence */
    int n = n_seq;
    if (mask_kind & OR_MASK_CAUSAL_BR) {
        /* the queries are the sequence's last Lq tokens: row i is at p_i */
        long long pos = (long long)n_seq - (long long)Lq + (long long)i;
        if (pos < 0)
            return 0; /* the query precedes the sequence: no keys, output 0 */
        /* keys 0..p_i; p_i < n_seq because i < Lq (the bound only guards the
           buffers against a wrong offset) */
        return (pos + 1 < n) ? (int)(pos + 1) : n;
    }
    if (padding && i >= kv_len)
        return 0; /* padded query row: output 0 */
    if (mask_kind & OR_MASK_CAUSAL)
        n = (i + 1 < n) ? i + 1 : n;
    return n;
}

/* ------------------------------------------------------------------------ */
/* attention over [B, H, L, d] heads                                         */
/* ------------------------------------------------------------------------ */
typedef struct {
    int is_bf16;
    const void *Q, *K, *V;
    int B, H, Hkv, Lq, Lk, dk, dv, mask_kind;
    const int32_t *kv_lens;
    double scale;
    const int64_t *rows; /* flat (b*H + h)*Lq + i, sorted by head, or NULL */
    int64_t nrows;
    double *O, *LSE, *A;
    /* work units: [unit_start[u], unit_start[u+1]) of the row list */
    int64_t *unit_start;
    int64_t n_units;
    int64_t next_unit; /* atomic */
    int err;
} attn_job;

static int64_t row_id(const attn_job *J, int64_t r)
{
    return J->rows ? J->rows[r] : r;
}

static void *attn_worker(void *arg)
{
    attn_job *J = (attn_job *)arg;
    double *Kd = NULL, *Vd = NULL, *q = NULL, *s = NULL;
    size_t cap_keys = 0;
    Kd = NULL;
    q = (double *)malloc(sizeof(double) * (size_t)J->dk);
    s = (double *)malloc(sizeof(double) * (size_t)(J->Lk > 0 ? J->Lk : 1));
    if (!q || !s) {
        __atomic_store_n(&J->err, OR_ERR_NOMEM, __ATOMIC_RELAXED);
        goto done;
    }
    for (;;) {
        int64_t u = __atomic_fetch_add(&J->next_unit, 1, __ATOMIC_RELAXED);
        int64_t r0, r1, r, bh, kvbh;
        int b, max_keys, kv_len, j, c;
        if (u >= J->n_units)
            break;
        r0 = J->unit_start[u];
        r1 = J->unit_start[u + 1];
        bh = row_id(J, r0) / J->Lq;
        b = (int)(bh / J->H);
        /* the K/V head this query head reads (grouped-query attention) */
        kvbh = (int64_t)b * J->Hkv + (int)(bh % J->H) / (J->H / J->Hkv);
        kv_len = (J->mask_kind & OR_MASK_PADDING) ? J->kv_lens[b] : J->Lk;
        /* widen the keys/values this block of rows needs */
        max_keys = 0;
        for (r = r0; r < r1; ++r) {
            int i = (int)(row_id(J, r) % J->Lq);
            int n = valid_keys(i, J->Lq, J->Lk, J->mask_kind, kv_len);
            if (n > max_keys)
                max_keys = n;
        }
        if ((size_t)max_keys > cap_keys) {
            free(Kd);
            free(Vd);
            Kd = (double *)malloc(sizeof(double) * (size_t)max_keys * (size_t)J->dk);
            Vd = (double *)malloc(sizeof(double) * (size_t)max_keys * (size_t)J->dv);
            cap_keys = (size_t)max_keys;
            if (!Kd || !Vd) {
                __atomic_store_n(&J->err, OR_ERR_NOMEM, __ATOMIC_RELAXED);
                goto done;
            }
        }
        for (j = 0; j < max_keys; ++j) {
            size_t kb = ((size_t)kvbh * (size_t)J->Lk + (size_t)j) * (size_t)J->dk;
            size_t vb = ((size_t)kvbh * (size_t)J->Lk + (size_t)j) * (size_t)J->dv;
            for (c = 0; c < J->dk; ++c)
                Kd[(size_t)j * J->dk + c] = elem(J->K, J->is_bf16, kb + c);
            for (c = 0; c < J->dv; ++c)
                Vd[(size_t)j * J->dv + c] = elem(J->V, J->is_bf16, vb + c);
        }
        for (r = r0; r < r1; ++r) {
            int64_t id = row_id(J, r);
            int i = (int)(id % J->Lq);
            int n = valid_keys(i, J->Lq, J->Lk, J->mask_kind, kv_len);
            size_t qb = (size_t)id * (size_t)J->dk;
            double *a_row = J->A ? J->A + (size_t)r * (size_t)J->Lk : NULL;
            for (c = 0; c < J->dk; ++c)
                q[c] = elem(J->Q, J->is_bf16, qb + c);
            if (a_row)
                for (j = 0; j < J->Lk; ++j)
                    a_row[j] = 0.0;
            attend_row(q, Kd, (size_t)J->dk, Vd, (size_t)J->dv, n, J->dk, J->dv, J->scale, s,
                       J->O + (size_t)r * (size_t)J->dv, J->LSE + r, a_row);
        }
    }
done:
    free(Kd);
    free(Vd);
    free(q);
    free(s);
    return NULL;
}

static int run_threads(void *(*fn)(void *), void *job, int nthreads)
{
    pthread_t *tid;
    int t, started = 0;
    if (nthreads < 1)
        nthreads = 1;
    tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tid)
        return OR_ERR_NOMEM;
    for (t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, fn, job) != 0)
            break;
        started = t;
    }
    fn(job);
    for (t = 1; t <= started; ++t)
        pthread_join(tid[t], NULL);
    free(tid);
    return OR_OK;
}

/*
 * oracle_attention: see the file header for the definition.
 *   elem_is_bf16: 1 -> Q/K/V are uint16 bf16 bit patterns, 0 -> fp64.
 *   Q [B,H,Lq,dk], K [B,Hkv,Lk,dk], V [B,Hkv,Lk,dv], contiguous; H % Hkv == 0.
 *   kv_lens: int32 [B], required when the PADDING bit is set; each in [0, Lk].
 *   scale <= 0 selects 1/sqrt(dk).
 *   rows: flat row ids (b*H + h)*Lq + i, in non-decreasing (b, h) order, or
 *         NULL for all B*H*Lq rows in order.
 *   O [nrows, dv], LSE [nrows], A [nrows, Lk] (optional, may be NULL).
 * Returns 0, or a negative error code.
 */
int oracle_attention(int elem_is_bf16, const void *Q, const void *K, const void *V, int B, int H,
                     int Hkv, int Lq, int Lk, int dk, int dv, int mask_kind,
                     const int32_t *kv_lens, double scale, const int64_t *rows, int64_t nrows,
                     double *O, double *LSE, double *A, int nthreads)
{
    attn_job J;
    int64_t r, n_units = 0;
    const int64_t block = 64;
    int rc;
    if (!Q || !K || !V || !O || !LSE || B < 0 || H < 0 || Lq < 0 || Lk < 0 || dk < 1 || dv < 1)
        return OR_ERR_ARG;
    if (Hkv < 1 || (H > 0 && H % Hkv != 0))
        return OR_ERR_ARG;
    if ((mask_kind & ~(OR_MASK_CAUSAL | OR_MASK_PADDING | OR_MASK_CAUSAL_BR)) != 0)
        return OR_ERR_ARG;
    if ((mask_kind & OR_MASK_CAUSAL) && (mask_kind & OR_MASK_CAUSAL_BR))
        return OR_ERR_ARG;
    if (mask_kind & OR_MASK_PADDING) {
        int b;
        if (!kv_lens)
            return OR_ERR_ARG;
        for (b = 0; b < B; ++b)
            if (kv_lens[b] < 0 || kv_lens[b] > Lk)
                return OR_ERR_ARG;
    }
    if (!rows)
        nrows = (int64_t)B * H * Lq;
    for (r = 0; r < nrows; ++r) {
        int64_t id = rows ? rows[r] : r;
        if (id < 0 || id >= (int64_t)B * H * Lq)
            return OR_ERR_ARG;
        if (r > 0 && rows && rows[r] / Lq < rows[r - 1] / Lq)
            return OR_ERR_ARG; /* must be grouped by head */
    }
    memset(&J, 0, sizeof J);
    J.is_bf16 = elem_is_bf16;
    J.Q = Q;
    J.K = K;
    J.V = V;
    J.B = B;
    J.H = H;
    J.Hkv = Hkv;
    J.Lq = Lq;
    J.Lk = Lk;
    J.dk = dk;
    J.dv = dv;
    J.mask_kind = mask_kind;
    J.kv_lens = kv_lens;
    J.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)dk);
    J.rows = rows;
    J.nrows = nrows;
    J.O = O;
    J.LSE = LSE;
    J.A = A;
    /* units: runs of at most `block` rows of the same head */
    J.unit_start = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nrows + 1));
    if (!J.unit_start)
        return OR_ERR_NOMEM;
    for (r = 0; r < nrows; ++r) {
        int64_t id = rows ? rows[r] : r;
        int64_t prev = r > 0 ? (rows ? rows[r - 1] : r - 1) : -1;
        int new_unit = (r == 0) || (id / Lq != prev / Lq) ||
                       (r - J.unit_start[n_units - 1] >= block);
        if (new_unit)
            J.unit_start[n_units++] = r;
    }
    J.unit_start[n_units] = nrows;
    J.n_units = n_units;
    J.next_unit = 0;
    rc = run_threads(attn_worker, &J, nthreads);
    free(J.unit_start);
    if (rc != OR_OK)
        return rc;
    return J.err;
}

/* ------------------------------------------------------------------------ */
/* the five-step multi-head layer                                            */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint16_t *X, *Wqkv, *Wo;
    int B, L, dm, H, mask_kind;
    const int32_t *kv_lens;
    double scale;
    const int64_t *rows;
    int64_t nrows;
    double *Y;
    /* K and V projections of the batches that are needed: [nb][L][dm] */
    int *batch_slot; /* b -> slot or -1 */
    int *slot_batch;
    int n_slots;
    int *slot_keys; /* keys needed per slot */
    double *Kp, *Vp;
    double *Wq_d, *Wk_d, *Wv_d, *Wo_d; /* widened weights [dm][dm] each */
    int64_t next; /* atomic work counter */
    int phase;
    int err;
} layer_job;

/* Phase 1 work item: one (slot, key row) -> K and V projections of that row. */
static void *layer_worker(void *arg)
{
    layer_job *J = (layer_job *)arg;
    const int dm = J->dm, dk = dm / J->H;
    double *x = (double *)malloc(sizeof(double) * (size_t)dm);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)dm);
    double *cat = (double *)malloc(sizeof(double) * (size_t)dm);
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->L > 0 ? J->L : 1));
    if (!x || !qrow || !cat || !s) {
        __atomic_store_n(&J->err, OR_ERR_NOMEM, __ATOMIC_RELAXED);
        goto done;
    }
    if (J->phase == 1) {
        int64_t total = (int64_t)J->n_slots * J->L;
        for (;;) {
            int64_t w = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
            int slot, l, b, c, n;
            double *kr, *vr;
            if (w >= total)
                break;
            slot = (int)(w / J->L);
            l = (int)(w % J->L);
            if (l >= J->slot_keys[slot])
                continue;
            b = J->slot_batch[slot];
            for (c = 0; c < dm; ++c)
                x[c] = widen_bf16(J->X[((size_t)b * J->L + l) * dm + c]);
            kr = J->Kp + ((size_t)slot * J->L + l) * dm;
            vr = J->Vp + ((size_t)slot * J->L + l) * dm;
            for (n = 0; n < dm; ++n) {
                kr[n] = 0.0;
                vr[n] = 0.0;
            }
            /* row of X times W_K, W_V (plain i-k-j loop) */
            for (c = 0; c < dm; ++c) {
                const double *wk = J->Wk_d + (size_t)c * dm;
                const double *wv = J->Wv_d + (size_t)c * dm;
                double xc = x[c];
                for (n = 0; n < dm; ++n) {
                    kr[n] += xc * wk[n];
                    vr[n] += xc * wv[n];
                }
            }
        }
    } else {
        for (;;) {
            int64_t r = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
            int64_t id;
            int b, l, slot, kv_len, n_keys, head, c, n;
            double lse;
            if (r >= J->nrows)
                break;
            id = J->rows ? J->rows[r] : r;
            b = (int)(id / J->L);
            l = (int)(id % J->L);
            slot = J->batch_slot[b];
            kv_len = (J->mask_kind & OR_MASK_PADDING) ? J->kv_lens[b] : J->L;
            n_keys = valid_keys(l, J->L, J->L, J->mask_kind, kv_len);
            /* step 1 for the query: q = x W_Q */
            for (c = 0; c < dm; ++c)
                x[c] = widen_bf16(J->X[((size_t)b * J->L + l) * dm + c]);
            for (n = 0; n < dm; ++n)
                qrow[n] = 0.0;
            for (c = 0; c < dm; ++c) {
                const double *wq = J->Wq_d + (size_t)c * dm;
                for (n = 0; n < dm; ++n)
                    qrow[n] += x[c] * wq[n];
            }
            /* steps 2-5 per head, written into the concatenated row */
            for (head = 0; head < J->H; ++head) {
                const double *Kh = J->Kp + (size_t)slot * J->L * dm + (size_t)head * dk;
                const double *Vh = J->Vp + (size_t)slot * J->L * dm + (size_t)head * dk;
                attend_row(qrow + (size_t)head * dk, Kh, (size_t)dm, Vh, (size_t)dm, n_keys, dk,
                           dk, J->scale, s, cat + (size_t)head * dk, &lse, NULL);
            }
            /* output projection y = cat W_O */
            {
                double *y = J->Y + (size_t)r * dm;
                for (n = 0; n < dm; ++n)
                    y[n] = 0.0;
                for (c = 0; c < dm; ++c) {
                    const double *wo = J->Wo_d + (size_t)c * dm;
                    double cc = cat[c];
                    for (n = 0; n < dm; ++n)
                        y[n] += cc * wo[n];
                }
            }
        }
    }
done:
    free(x);
    free(qrow);
    free(cat);
    free(s);
    return NULL;
}

/*
 * oracle_mha_layer: see the file header for the definition.
 *   X [B,L,dm], Wqkv [dm, 3*dm], Wo [dm, dm]: bf16 bit patterns, contiguous.
 *   H heads, d_k = dm / H (dm must be divisible by H).
 *   mask_kind: CAUSAL, CAUSAL_BR (exclusive with CAUSAL), PADDING, as for the
 *         attention (Lq = Lk = L).
 *   rows: flat ids b*L + l of the output rows wanted (any order), or NULL
 *         for all B*L rows.  Y [nrows, dm] fp64.
 */
int oracle_mha_layer(const uint16_t *X, const uint16_t *Wqkv, const uint16_t *Wo, int B, int L,
                     int dm, int H, int mask_kind, const int32_t *kv_lens, double scale,
                     const int64_t *rows, int64_t nrows, double *Y, int nthreads)
{
    layer_job J;
    int b, rc = OR_OK, c, n;
    int64_t r;
    if (!X || !Wqkv || !Wo || !Y || B < 0 || L < 0 || dm < 1 || H < 1 || dm % H != 0)
        return OR_ERR_ARG;
    if ((mask_kind & ~(OR_MASK_CAUSAL | OR_MASK_PADDING | OR_MASK_CAUSAL_BR)) != 0)
        return OR_ERR_ARG;
    if ((mask_kind & OR_MASK_CAUSAL) && (mask_kind & OR_MASK_CAUSAL_BR))
        return OR_ERR_ARG;
    if (mask_kind & OR_MASK_PADDING) {
        if (!kv_lens)
            return OR_ERR_ARG;
        for (b = 0; b < B; ++b)
            if (kv_lens[b] < 0 || kv_lens[b] > L)
                return OR_ERR_ARG;
    }
    if (!rows)
        nrows = (int64_t)B * L;
    for (r = 0; r < nrows; ++r) {
        int64_t id = rows ? rows[r] : r;
        if (id < 0 || id >= (int64_t)B * L)
            return OR_ERR_ARG;
    }
    memset(&J, 0, sizeof J);
    J.X = X;
    J.Wqkv = Wqkv;
    J.Wo = Wo;
    J.B = B;
    J.L = L;
    J.dm = dm;
    J.H = H;
    J.mask_kind = mask_kind;
    J.kv_lens = kv_lens;
    J.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)(dm / H));
    J.rows = rows;
    J.nrows = nrows;
    J.Y = Y;
    J.batch_slot = (int *)malloc(sizeof(int) * (size_t)(B > 0 ? B : 1));
    J.slot_batch = (int *)malloc(sizeof(int) * (size_t)(B > 0 ? B : 1));
    J.slot_keys = (int *)calloc((size_t)(B > 0 ? B : 1), sizeof(int));
    J.Wq_d = (double *)malloc(sizeof(double) * (size_t)dm * dm);
    J.Wk_d = (double *)malloc(sizeof(double) * (size_t)dm * dm);
    J.Wv_d = (double *)malloc(sizeof(double) * (size_t)dm * dm);
    J.Wo_d = (double *)malloc(sizeof(double) * (size_t)dm * dm);
    if (!J.batch_slot || !J.slot_batch || !J.slot_keys || !J.Wq_d || !J.Wk_d || !J.Wv_d ||
        !J.Wo_d) {
        rc = OR_ERR_NOMEM;
        goto out;
    }
    /* split W_QKV into its Q, K, V column blocks (widened) */
    for (c = 0; c < dm; ++c)
        for (n = 0; n < dm; ++n) {
            J.Wq_d[(size_t)c * dm + n] = widen_bf16(Wqkv[(size_t)c * 3 * dm + n]);
            J.Wk_d[(size_t)c * dm + n] = widen_bf16(Wqkv[(size_t)c * 3 * dm + dm + n]);
            J.Wv_d[(size_t)c * dm + n] = widen_bf16(Wqkv[(size_t)c * 3 * dm + 2 * dm + n]);
            J.Wo_d[(size_t)c * dm + n] = widen_bf16(Wo[(size_t)c * dm + n]);
        }
    /* which batches are needed, and how many key rows of each */
    for (b = 0; b < B; ++b)
        J.batch_slot[b] = -1;
    for (r = 0; r < nrows; ++r) {
        int64_t id = rows ? rows[r] : r;
        int bb = (int)(id / L), l = (int)(id % L);
        int kv_len = (mask_kind & OR_MASK_PADDING) ? kv_lens[bb] : L;
        int nk = valid_keys(l, L, L, mask_kind, kv_len);
        if (J.batch_slot[bb] < 0) {
            J.batch_slot[bb] = J.n_slots;
            J.slot_batch[J.n_slots] = bb;
            J.n_slots++;
        }
        if (nk > J.slot_keys[J.batch_slot[bb]])
            J.slot_keys[J.batch_slot[bb]] = nk;
    }
    J.Kp = (double *)malloc(sizeof(double) * (size_t)(J.n_slots > 0 ? J.n_slots : 1) * L * dm);
    J.Vp = (double *)malloc(sizeof(double) * (size_t)(J.n_slots > 0 ? J.n_slots : 1) * L * dm);
    if (!J.Kp || !J.Vp) {
        rc = OR_ERR_NOMEM;
        goto out;
    }
    J.phase = 1;
    J.next = 0;
    rc = run_threads(layer_worker, &J, nthreads);
    if (rc == OR_OK && J.err == OR_OK) {
        J.phase = 2;
        J.next = 0;
        rc = run_threads(layer_worker, &J, nthreads);
    }
    if (rc == OR_OK)
        rc = J.err;
out:
    free(J.batch_slot);
    free(J.slot_batch);
    free(J.slot_keys);
    free(J.Wq_d);
    free(J.Wk_d);
    free(J.Wv_d);
    free(J.Wo_d);
    free(J.Kp);
    free(J.Vp);
    return rc;
}
