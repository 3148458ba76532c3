/*
 * oracle.c -- plain, slow, fp64 CPU oracle for packed document-masked
 * attention, its worklist, zigzag context-parallel maps and the
 * online-softmax merge.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares no code, header
 * or table with the CUDA library; the only thing both sides share is the
 * seeded input generator (document lengths and bf16 tensors).
 *
 * Every function states the passage it follows.  Page titles:
 *   [P1] "03 · 长文负载均衡" (llm-infra-atlas, long-context load balancing)
 *   [P2] "数据并行负载均衡" (loongforge DP load balance)
 *   [P4] "长序列训练与上下文并行" (long-sequence training and context parallelism)
 *
 * Parity status: every function below is pinned by the CPU tests
 * (closed forms, brute force, library routines on tiny inputs, invariants).
 */
#include "oracle.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* bf16 -> double: the bf16 bit pattern is the top half of an fp32; the      */
/* widening to double is exact.                                              */
/* ------------------------------------------------------------------------ */
static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int32_t or_num_threads(void) {
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Zigzag shard map.  [P1] §1.2 and §4.2: the sequence is cut into 2*cp      */
/* chunks and rank i owns chunk i and chunk 2cp-1-i.  [P1] §4.3 (WLB-LLM     */
/* per-document sharding): every document is cut on its own, so each rank   */
/* gets a symmetric pair of chunks of every document.  Remainder rule (the   */
/* page only says "round-robin"): chunk c of a document of length L gets     */
/* floor(L/2cp) tokens plus one if c < L mod 2cp; chunks are contiguous in   */
/* chunk order.  Rank r's local rows are, document by document, chunk r      */
/* followed by chunk 2cp-1-r.                                                */
/* ------------------------------------------------------------------------ */
static void zz_chunk(int32_t len, int32_t cp, int32_t c, int32_t *off, int32_t *clen) {
    int32_t n = 2 * cp;
    int32_t base = len / n, rem = len % n;
    *clen = base + (c < rem ? 1 : 0);
    *off = c * base + (c < rem ? c : rem);
}

int32_t or_zigzag_map(const int32_t *cu, int32_t ndocs, int32_t cp, int32_t rank,
                      int32_t *map, int32_t *chunk_table) {
    if (cp <= 0 || rank < 0 || rank >= cp) return -1;
    int32_t local = 0;
    for (int32_t d = 0; d < ndocs; ++d) {
        int32_t len = cu[d + 1] - cu[d];
        int32_t chunks[2] = {rank, 2 * cp - 1 - rank};
        for (int e = 0; e < 2; ++e) {
            int32_t off, clen;
            zz_chunk(len, cp, chunks[e], &off, &clen);
            if (chunk_table) {
                int32_t *row = chunk_table + ((int64_t)d * 2 + e) * 4;
                row[0] = d;
                row[1] = chunks[e];
                row[2] = cu[d] + off;
                row[3] = clen;
            }
            for (int32_t i = 0; i < clen; ++i) {
                if (map) map[local] = cu[d] + off + i;
                ++local;
            }
        }
    }
    return local;
}

/* ------------------------------------------------------------------------ */
/* Mask predicate: which (query row, key row) pairs are allowed.             */
/*  - causal per document: [P1] §1.1 -- documents in a pack do not attend    */
/*    to each other, so the work is sum_j l_j^2 (not (sum l_j)^2).           */
/*  - sliding window and shared question: [P1] §1.2 (structured masks).      */
/*    Reading: window w keeps keys with q_pos - k_pos < w (w keys including  */
/*    the query itself).  Shared question: the first num_prefix documents   */
/*    are questions that attend causally to themselves; every other          */
/*    document (an answer) sees all question tokens and itself causally.    */
/*  - zigzag pair (q rank r, kv rank s): rows are rank-local (map above);    */
/*    allowed iff same document and k position <= q position ([P4] ring     */
/*    attention, each rank's Q against one KV shard).                        */
/*  - zigzag ring step t: every rank's shard at once, rows in ring order     */
/*    (rank 0's shard, then rank 1's, ...); a query row of rank r sees the   */
/*    key rows of rank (r - t) mod cp that hold the same document at a       */
/*    position <= its own ([P4] ring loop: at step t rank r works on the KV  */
/*    that started on rank r - t).                                           */
/*  - slices: [P1] §4.4 AttnSlice (QRange, KRange, MaskType).  The pages     */
/*    name FULL / CAUSAL / INV-CAUSAL / BI-CAUSAL without geometry; reading: */
/*    tests on the slice's token positions, CAUSAL k <= q and INV-CAUSAL     */
/*    k >= q (each with an optional window w: |q - k| < w), BI-CAUSAL        */
/*    k >= q and k_end - k >= q_end - q (inverse-causal from the start,      */
/*    causal from the end of the slice).                                     */
/* ------------------------------------------------------------------------ */
typedef struct {
    const int32_t *cu;
    int32_t ndocs;
    or_mask_t m;
    int32_t Tq, Tk;
    int32_t *doc_q, *doc_k; /* document id of every q / k row */
    int32_t *gq, *gk;       /* global token of every row (identity unless zigzag) */
    int32_t *kdoc_lo, *kdoc_hi; /* per document: range of k rows holding it */
    int32_t *rank_q, *rank_k;   /* ring step: rank of every q / k row */
    int32_t *krd_lo, *krd_hi;   /* ring step: per (rank, document), its k rows */
} ctx_t;

/* Ring order of all zigzag shards: map[i] = global token of row i, rank[i] =
 * the rank whose shard holds it (ranks 0..cp-1 in turn).  Returns the rows. */
static int32_t ring_order(const int32_t *cu, int32_t ndocs, int32_t cp, int32_t *map,
                          int32_t *rank) {
    int32_t n = 0;
    for (int32_t r = 0; r < cp; ++r) {
        int32_t nr = or_zigzag_map(cu, ndocs, cp, r, map ? map + n : NULL, NULL);
        if (rank)
            for (int32_t i = 0; i < nr; ++i) rank[n + i] = r;
        n += nr;
    }
    return n;
}

static int ctx_init(ctx_t *c, const int32_t *cu, int32_t ndocs, int32_t Tq, int32_t Tk,
                    const or_mask_t *m) {
    memset(c, 0, sizeof *c);
    c->cu = cu;
    c->ndocs = ndocs;
    c->m = *m;
    c->Tq = Tq;
    c->Tk = Tk;
    int32_t T = cu[ndocs];
    int32_t *doc_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    for (int32_t d = 0; d < ndocs; ++d)
        for (int32_t t = cu[d]; t < cu[d + 1]; ++t) doc_of[t] = d;
    c->gq = (int32_t *)malloc(sizeof(int32_t) * (size_t)(Tq > 0 ? Tq : 1));
    c->gk = (int32_t *)malloc(sizeof(int32_t) * (size_t)(Tk > 0 ? Tk : 1));
    if (m->kind == OR_MASK_ZIGZAG_PAIR) {
        int32_t tq = or_zigzag_map(cu, ndocs, m->cp, m->q_rank, NULL, NULL);
        int32_t tk = or_zigzag_map(cu, ndocs, m->cp, m->k_rank, NULL, NULL);
        if (tq != Tq || tk != Tk) {
            free(doc_of);
            free(c->gq);
            free(c->gk);
            return -1;
        }
        or_zigzag_map(cu, ndocs, m->cp, m->q_rank, c->gq, NULL);
        or_zigzag_map(cu, ndocs, m->cp, m->k_rank, c->gk, NULL);
    } else if (m->kind == OR_MASK_ZIGZAG_STEP) {
        if (m->cp <= 0 || m->ring_step < 0 || m->ring_step >= m->cp || Tq != T || Tk != T) {
            free(doc_of);
            free(c->gq);
            free(c->gk);
            return -1;
        }
        c->rank_q = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
        c->rank_k = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
        ring_order(cu, ndocs, m->cp, c->gq, c->rank_q);
        ring_order(cu, ndocs, m->cp, c->gk, c->rank_k);
    } else {
        if ((m->kind != OR_MASK_SLICES) && (Tq != T || Tk != T)) {
            free(doc_of);
            free(c->gq);
            free(c->gk);
            return -1;
        }
        for (int32_t i = 0; i < Tq; ++i) c->gq[i] = i;
        for (int32_t j = 0; j < Tk; ++j) c->gk[j] = j;
    }
    c->doc_q = (int32_t *)malloc(sizeof(int32_t) * (size_t)(Tq > 0 ? Tq : 1));
    c->doc_k = (int32_t *)malloc(sizeof(int32_t) * (size_t)(Tk > 0 ? Tk : 1));
    for (int32_t i = 0; i < Tq; ++i) c->doc_q[i] = (c->gq[i] < T) ? doc_of[c->gq[i]] : -1;
    for (int32_t j = 0; j < Tk; ++j) c->doc_k[j] = (c->gk[j] < T) ? doc_of[c->gk[j]] : -1;
    c->kdoc_lo = (int32_t *)malloc(sizeof(int32_t) * (size_t)(ndocs > 0 ? ndocs : 1));
    c->kdoc_hi = (int32_t *)malloc(sizeof(int32_t) * (size_t)(ndocs > 0 ? ndocs : 1));
    for (int32_t d = 0; d < ndocs; ++d) {
        c->kdoc_lo[d] = Tk;
        c->kdoc_hi[d] = 0;
    }
    for (int32_t j = 0; j < Tk; ++j) {
        int32_t d = c->doc_k[j];
        if (d < 0) continue;
        if (j < c->kdoc_lo[d]) c->kdoc_lo[d] = j;
        if (j + 1 > c->kdoc_hi[d]) c->kdoc_hi[d] = j + 1;
    }
    if (m->kind == OR_MASK_ZIGZAG_STEP) {
        int64_t nrd = (int64_t)m->cp * ndocs;
        c->krd_lo = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nrd > 0 ? nrd : 1));
        c->krd_hi = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nrd > 0 ? nrd : 1));
        for (int64_t x = 0; x < nrd; ++x) {
            c->krd_lo[x] = Tk;
            c->krd_hi[x] = 0;
        }
        for (int32_t j = 0; j < Tk; ++j) {
            int64_t x = (int64_t)c->rank_k[j] * ndocs + c->doc_k[j];
            if (j < c->krd_lo[x]) c->krd_lo[x] = j;
            if (j + 1 > c->krd_hi[x]) c->krd_hi[x] = j + 1;
        }
    }
    free(doc_of);
    return 0;
}

static void ctx_free(ctx_t *c) {
    free(c->doc_q);
    free(c->doc_k);
    free(c->gq);
    free(c->gk);
    free(c->kdoc_lo);
    free(c->kdoc_hi);
    free(c->rank_q);
    free(c->rank_k);
    free(c->krd_lo);
    free(c->krd_hi);
}

static int allowed(const ctx_t *c, int32_t i, int32_t j) {
    const or_mask_t *m = &c->m;
    switch (m->kind) {
    case OR_MASK_CAUSAL:
        return c->doc_q[i] == c->doc_k[j] && j <= i;
    case OR_MASK_SLIDING_WINDOW:
        return c->doc_q[i] == c->doc_k[j] && j <= i && (m->window <= 0 || i - j < m->window);
    case OR_MASK_SHARED_QUESTION: {
        int32_t dq = c->doc_q[i], dk = c->doc_k[j];
        if (dq < m->num_prefix) return dk == dq && j <= i;
        return dk < m->num_prefix || (dk == dq && j <= i);
    }
    case OR_MASK_ZIGZAG_PAIR:
        return c->doc_q[i] == c->doc_k[j] && c->gk[j] <= c->gq[i];
    case OR_MASK_ZIGZAG_STEP:
        return c->doc_q[i] == c->doc_k[j] &&
               c->rank_k[j] == (c->rank_q[i] - m->ring_step + m->cp) % m->cp &&
               c->gk[j] <= c->gq[i];
    case OR_MASK_SLICES:
        /* AttnSlice MaskTypes ("03 · 长文负载均衡" §4.4), tested on token positions:
         * CAUSAL k <= q, INV_CAUSAL k >= q (each with an optional window), and
         * BI_CAUSAL k >= q with k_end - k >= q_end - q (inverse-causal from the
         * slice start, causal from its end). */
        for (int32_t s = 0; s < m->num_slices; ++s) {
            const int32_t *sl = m->slices + 8 * s;
            if (i < sl[0] || i >= sl[0] + sl[1] || j < sl[3] || j >= sl[3] + sl[4]) continue;
            int64_t qp = (int64_t)sl[2] + (i - sl[0]);
            int64_t kp = (int64_t)sl[5] + (j - sl[3]);
            int64_t w = sl[7];
            switch (sl[6]) {
            case OR_SLICE_FULL:
                return 1;
            case OR_SLICE_CAUSAL:
                if (kp <= qp && (w <= 0 || qp - kp < w)) return 1;
                break;
            case OR_SLICE_INV_CAUSAL:
                if (kp >= qp && (w <= 0 || kp - qp < w)) return 1;
                break;
            case OR_SLICE_BI_CAUSAL: {
                int64_t q_end = (int64_t)sl[2] + sl[1], k_end = (int64_t)sl[5] + sl[4];
                if (kp >= qp && k_end - kp >= q_end - qp) return 1;
                break;
            }
            }
        }
        return 0;
    }
    return 0;
}

/* Candidate key rows for query row i: a superset of the allowed set, so    */
/* that large packs do not scan every key.  brute=1 scans all keys.          */
static int candidates(const ctx_t *c, int32_t i, int brute, int32_t lo[2], int32_t hi[2]) {
    if (brute || c->m.kind == OR_MASK_SLICES) {
        lo[0] = 0;
        hi[0] = c->Tk;
        return 1;
    }
    int32_t d = c->doc_q[i];
    if (d < 0) return 0;
    switch (c->m.kind) {
    case OR_MASK_CAUSAL:
    case OR_MASK_SLIDING_WINDOW:
        lo[0] = c->cu[d];
        hi[0] = i + 1;
        return 1;
    case OR_MASK_SHARED_QUESTION:
        if (d < c->m.num_prefix) {
            lo[0] = c->cu[d];
            hi[0] = i + 1;
            return 1;
        }
        lo[0] = 0;
        hi[0] = c->cu[c->m.num_prefix];
        lo[1] = c->cu[d];
        hi[1] = i + 1;
        return 2;
    case OR_MASK_ZIGZAG_PAIR:
        lo[0] = c->kdoc_lo[d];
        hi[0] = c->kdoc_hi[d];
        return lo[0] < hi[0] ? 1 : 0;
    case OR_MASK_ZIGZAG_STEP: {
        int64_t x = (int64_t)((c->rank_q[i] - c->m.ring_step + c->m.cp) % c->m.cp) * c->ndocs + d;
        lo[0] = c->krd_lo[x];
        hi[0] = c->krd_hi[x];
        return lo[0] < hi[0] ? 1 : 0;
    }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Attention, by definition, in fp64 from the bf16 inputs.                   */
/* For query row i and head h (kv head g = h / (Hq/Hkv), contiguous GQA      */
/* groups), with A(i) the allowed keys:                                      */
/*   s_j = scale * q_i . k_j,  LSE_i = ln sum_{j in A(i)} exp(s_j),          */
/*   O_i = sum_{j in A(i)} exp(s_j - LSE_i) v_j.                             */
/* The quadratic term of [P1] §1.1 (QK^T and PV), one row at a time.  Empty  */
/* A(i): O = 0 and LSE = -inf.  The max is subtracted before exp only to     */
/* keep fp64 in range; the value is the same.                                */
/* ------------------------------------------------------------------------ */
int or_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, int32_t Tq, int32_t Tk,
                 int32_t Hq, int32_t Hkv, int32_t d, const int32_t *cu, int32_t ndocs,
                 const or_mask_t *m, double scale, const int32_t *jobs, int64_t njobs,
                 int32_t brute, double *out, double *lse) {
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return -1;
    ctx_t c;
    if (ctx_init(&c, cu, ndocs, Tq, Tk, m) != 0) return -2;
    const int32_t G = Hq / Hkv;
    const int64_t n = jobs ? njobs : (int64_t)Tq * Hq;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
        int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(Tk > 0 ? Tk : 1));
        double *qi = (double *)malloc(sizeof(double) * (size_t)d);
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 8)
        for (int64_t job = 0; job < n; ++job) {
            int32_t i, h;
            if (jobs) {
                i = jobs[2 * job];
                h = jobs[2 * job + 1];
            } else {
                i = (int32_t)(job / Hq);
                h = (int32_t)(job % Hq);
            }
            if (i < 0 || i >= Tq || h < 0 || h >= Hq) {
                err = 1;
                continue;
            }
            const int32_t g = h / G;
            for (int32_t e = 0; e < d; ++e) qi[e] = bf16_to_double(q[((int64_t)i * Hq + h) * d + e]);
            int32_t lo[2], hi[2];
            int nr = candidates(&c, i, brute, lo, hi);
            int32_t cnt = 0;
            double mx = -INFINITY;
            for (int r = 0; r < nr; ++r) {
                for (int32_t j = lo[r]; j < hi[r]; ++j) {
                    if (!allowed(&c, i, j)) continue;
                    const uint16_t *kj = k + ((int64_t)j * Hkv + g) * d;
                    double dot = 0.0;
                    for (int32_t e = 0; e < d; ++e) dot += qi[e] * bf16_to_double(kj[e]);
                    s[cnt] = scale * dot;
                    idx[cnt] = j;
                    if (s[cnt] > mx) mx = s[cnt];
                    ++cnt;
                }
            }
            double *o = jobs ? out + job * d : out + ((int64_t)i * Hq + h) * d;
            double *l = jobs ? lse + job : lse + (int64_t)h * Tq + i;
            if (cnt == 0) {
                for (int32_t e = 0; e < d; ++e) o[e] = 0.0;
                *l = -INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int32_t e = 0; e < d; ++e) acc[e] = 0.0;
            for (int32_t t = 0; t < cnt; ++t) {
                double p = exp(s[t] - mx);
                sum += p;
                const uint16_t *vj = v + ((int64_t)idx[t] * Hkv + g) * d;
                for (int32_t e = 0; e < d; ++e) acc[e] += p * bf16_to_double(vj[e]);
            }
            for (int32_t e = 0; e < d; ++e) o[e] = acc[e] / sum;
            *l = mx + log(sum);
        }
        free(s);
        free(idx);
        free(qi);
        free(acc);
    }
    ctx_free(&c);
    return err ? -3 : 0;
}

/* ------------------------------------------------------------------------ */
/* Attention backward, by definition, in fp64 from bf16 inputs and the bf16  */
/* output gradient dO.  With A(i) the allowed keys of row i, s_ij =          */
/* scale q_i.k_j, P_ij = exp(s_ij - LSE_i) (the forward's probabilities):    */
/*   dP_ij = dO_i . v_j,   D_i = sum_{j in A(i)} P_ij dP_ij  (= dO_i . O_i), */
/*   dS_ij = P_ij (dP_ij - D_i),                                             */
/*   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,            */
/*   dV_j = sum_i P_ij dO_i,                                                 */
/* the gradients of the quadratic term of [P1] §1.1 (QK^T and PV); a kv head */
/* sums over the q heads of its group.  Rows with no key get no gradient.    */
/* dK and dV are gathered key by key over all query rows (brute force).      */
/* ------------------------------------------------------------------------ */
int or_attention_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const uint16_t *dout, int32_t Tq, int32_t Tk, int32_t Hq, int32_t Hkv,
                     int32_t d, const int32_t *cu, int32_t ndocs, const or_mask_t *m,
                     double scale, double *dq, double *dk, double *dv) {
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return -1;
    ctx_t c;
    if (ctx_init(&c, cu, ndocs, Tq, Tk, m) != 0) return -2;
    const int32_t G = Hq / Hkv;
    double *lse = (double *)malloc(sizeof(double) * (size_t)Tq * Hq + 1);
    double *Dv = (double *)malloc(sizeof(double) * (size_t)Tq * Hq + 1);
    /* pass 1, per (row, head): LSE, D and dQ */
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
        int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(Tk > 0 ? Tk : 1));
        double *qi = (double *)malloc(sizeof(double) * (size_t)d);
        double *gi = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 8)
        for (int64_t job = 0; job < (int64_t)Tq * Hq; ++job) {
            const int32_t i = (int32_t)(job / Hq), h = (int32_t)(job % Hq), g = h / G;
            for (int32_t e = 0; e < d; ++e) {
                qi[e] = bf16_to_double(q[((int64_t)i * Hq + h) * d + e]);
                gi[e] = bf16_to_double(dout[((int64_t)i * Hq + h) * d + e]);
            }
            double *dqi = dq + ((int64_t)i * Hq + h) * d;
            for (int32_t e = 0; e < d; ++e) dqi[e] = 0.0;
            int32_t cnt = 0;
            double mx = -INFINITY;
            for (int32_t j = 0; j < Tk; ++j) {
                if (!allowed(&c, i, j)) continue;
                const uint16_t *kj = k + ((int64_t)j * Hkv + g) * d;
                const uint16_t *vj = v + ((int64_t)j * Hkv + g) * d;
                double dot = 0.0, dd = 0.0;
                for (int32_t e = 0; e < d; ++e) {
                    dot += qi[e] * bf16_to_double(kj[e]);
                    dd += gi[e] * bf16_to_double(vj[e]);
                }
                s[cnt] = scale * dot;
                dp[cnt] = dd;
                idx[cnt] = j;
                if (s[cnt] > mx) mx = s[cnt];
                ++cnt;
            }
            if (cnt == 0) {
                lse[job] = -INFINITY;
                Dv[job] = 0.0;
                continue;
            }
            double sum = 0.0;
            for (int32_t t = 0; t < cnt; ++t) sum += exp(s[t] - mx);
            const double l = mx + log(sum);
            double D = 0.0;
            for (int32_t t = 0; t < cnt; ++t) D += exp(s[t] - l) * dp[t];
            lse[job] = l;
            Dv[job] = D;
            for (int32_t t = 0; t < cnt; ++t) {
                const double ds = exp(s[t] - l) * (dp[t] - D);
                const uint16_t *kj = k + ((int64_t)idx[t] * Hkv + g) * d;
                for (int32_t e = 0; e < d; ++e) dqi[e] += scale * ds * bf16_to_double(kj[e]);
            }
        }
        free(s);
        free(dp);
        free(idx);
        free(qi);
        free(gi);
    }
    /* pass 2, per (key, kv head): dK and dV over every query row of the group */
#pragma omp parallel
    {
        double *kj = (double *)malloc(sizeof(double) * (size_t)d);
        double *vj = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 8)
        for (int64_t job = 0; job < (int64_t)Tk * Hkv; ++job) {
            const int32_t j = (int32_t)(job / Hkv), g = (int32_t)(job % Hkv);
            for (int32_t e = 0; e < d; ++e) {
                kj[e] = bf16_to_double(k[((int64_t)j * Hkv + g) * d + e]);
                vj[e] = bf16_to_double(v[((int64_t)j * Hkv + g) * d + e]);
            }
            double *dkj = dk + ((int64_t)j * Hkv + g) * d;
            double *dvj = dv + ((int64_t)j * Hkv + g) * d;
            for (int32_t e = 0; e < d; ++e) dkj[e] = dvj[e] = 0.0;
            for (int32_t i = 0; i < Tq; ++i) {
                if (!allowed(&c, i, j)) continue;
                for (int32_t h = g * G; h < (g + 1) * G; ++h) {
                    const int64_t r = (int64_t)i * Hq + h;
                    const uint16_t *qi = q + r * d, *gi = dout + r * d;
                    double dot = 0.0, dd = 0.0;
                    for (int32_t e = 0; e < d; ++e) {
                        dot += bf16_to_double(qi[e]) * kj[e];
                        dd += bf16_to_double(gi[e]) * vj[e];
                    }
                    const double p = exp(scale * dot - lse[r]);
                    const double ds = p * (dd - Dv[r]);
                    for (int32_t e = 0; e < d; ++e) {
                        dkj[e] += scale * ds * bf16_to_double(qi[e]);
                        dvj[e] += p * bf16_to_double(gi[e]);
                    }
                }
            }
        }
        free(kj);
        free(vj);
    }
    free(lse);
    free(Dv);
    ctx_free(&c);
    return 0;
}

/* The same gradients on sampled outputs: dQ of (row, head) jobs and dK, dV  */
/* of (key, kv head) jobs, each from its definition (a key job visits every  */
/* query row that may see the key and recomputes that row's LSE and D).      */
/* Rows' statistics are computed by row_stats below.                         */
static void row_stats(const ctx_t *c, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const uint16_t *dout, int32_t Hq, int32_t Hkv, int32_t d, double scale,
                      int32_t i, int32_t h, double *lse, double *D) {
    const int32_t G = Hq / Hkv, g = h / G;
    const uint16_t *qi = q + ((int64_t)i * Hq + h) * d, *gi = dout + ((int64_t)i * Hq + h) * d;
    int32_t lo[2], hi[2];
    int nr = candidates(c, i, 0, lo, hi);
    double mx = -INFINITY;
    for (int r = 0; r < nr; ++r)
        for (int32_t j = lo[r]; j < hi[r]; ++j) {
            if (!allowed(c, i, j)) continue;
            const uint16_t *kj = k + ((int64_t)j * Hkv + g) * d;
            double dot = 0.0;
            for (int32_t e = 0; e < d; ++e) dot += bf16_to_double(qi[e]) * bf16_to_double(kj[e]);
            if (scale * dot > mx) mx = scale * dot;
        }
    if (mx == -INFINITY) {
        *lse = -INFINITY;
        *D = 0.0;
        return;
    }
    double sum = 0.0, acc = 0.0;
    for (int r = 0; r < nr; ++r)
        for (int32_t j = lo[r]; j < hi[r]; ++j) {
            if (!allowed(c, i, j)) continue;
            const uint16_t *kj = k + ((int64_t)j * Hkv + g) * d;
            const uint16_t *vj = v + ((int64_t)j * Hkv + g) * d;
            double dot = 0.0, dd = 0.0;
            for (int32_t e = 0; e < d; ++e) {
                dot += bf16_to_double(qi[e]) * bf16_to_double(kj[e]);
                dd += bf16_to_double(gi[e]) * bf16_to_double(vj[e]);
            }
            const double pexp = exp(scale * dot - mx);
            sum += pexp;
            acc += pexp * dd;
        }
    *lse = mx + log(sum);
    *D = acc / sum;
}

int or_attention_bwd_jobs(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const uint16_t *dout, int32_t Tq, int32_t Tk, int32_t Hq, int32_t Hkv,
                          int32_t d, const int32_t *cu, int32_t ndocs, const or_mask_t *m,
                          double scale, const int32_t *qjobs, int64_t nq, const int32_t *kjobs,
                          int64_t nk, double *dq, double *dk, double *dv) {
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return -1;
    ctx_t c;
    if (ctx_init(&c, cu, ndocs, Tq, Tk, m) != 0) return -2;
    const int32_t G = Hq / Hkv;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t job = 0; job < nq; ++job) {
        const int32_t i = qjobs[2 * job], h = qjobs[2 * job + 1], g = h / G;
        double *o = dq + job * d;
        for (int32_t e = 0; e < d; ++e) o[e] = 0.0;
        if (i < 0 || i >= Tq || h < 0 || h >= Hq) {
            err = 1;
            continue;
        }
        double lse, D;
        row_stats(&c, q, k, v, dout, Hq, Hkv, d, scale, i, h, &lse, &D);
        if (lse == -INFINITY) continue;
        const uint16_t *qi = q + ((int64_t)i * Hq + h) * d, *gi = dout + ((int64_t)i * Hq + h) * d;
        int32_t lo[2], hi[2];
        int nr = candidates(&c, i, 0, lo, hi);
        for (int r = 0; r < nr; ++r)
            for (int32_t j = lo[r]; j < hi[r]; ++j) {
                if (!allowed(&c, i, j)) continue;
                const uint16_t *kj = k + ((int64_t)j * Hkv + g) * d;
                const uint16_t *vj = v + ((int64_t)j * Hkv + g) * d;
                double dot = 0.0, dd = 0.0;
                for (int32_t e = 0; e < d; ++e) {
                    dot += bf16_to_double(qi[e]) * bf16_to_double(kj[e]);
                    dd += bf16_to_double(gi[e]) * bf16_to_double(vj[e]);
                }
                const double ds = exp(scale * dot - lse) * (dd - D);
                for (int32_t e = 0; e < d; ++e) o[e] += scale * ds * bf16_to_double(kj[e]);
            }
    }
    for (int64_t job = 0; job < nk; ++job) {
        const int32_t j = kjobs[2 * job], g = kjobs[2 * job + 1];
        double *ok = dk + job * d, *ov = dv + job * d;
        for (int32_t e = 0; e < d; ++e) ok[e] = ov[e] = 0.0;
        if (j < 0 || j >= Tk || g < 0 || g >= Hkv) {
            err = 1;
            continue;
        }
        const uint16_t *kj = k + ((int64_t)j * Hkv + g) * d, *vj = v + ((int64_t)j * Hkv + g) * d;
#pragma omp parallel
        {
            double *pk = (double *)calloc((size_t)d, sizeof(double));
            double *pv = (double *)calloc((size_t)d, sizeof(double));
#pragma omp for schedule(dynamic, 4)
            for (int32_t i = 0; i < Tq; ++i) {
                if (!allowed(&c, i, j)) continue;
                for (int32_t h = g * G; h < (g + 1) * G; ++h) {
                    double lse, D;
                    row_stats(&c, q, k, v, dout, Hq, Hkv, d, scale, i, h, &lse, &D);
                    const uint16_t *qi = q + ((int64_t)i * Hq + h) * d;
                    const uint16_t *gi = dout + ((int64_t)i * Hq + h) * d;
                    double dot = 0.0, dd = 0.0;
                    for (int32_t e = 0; e < d; ++e) {
                        dot += bf16_to_double(qi[e]) * bf16_to_double(kj[e]);
                        dd += bf16_to_double(gi[e]) * bf16_to_double(vj[e]);
                    }
                    const double p = exp(scale * dot - lse);
                    const double ds = p * (dd - D);
                    for (int32_t e = 0; e < d; ++e) {
                        pk[e] += scale * ds * bf16_to_double(qi[e]);
                        pv[e] += p * bf16_to_double(gi[e]);
                    }
                }
            }
#pragma omp critical
            for (int32_t e = 0; e < d; ++e) {
                ok[e] += pk[e];
                ov[e] += pv[e];
            }
            free(pk);
            free(pv);
        }
    }
    ctx_free(&c);
    return err ? -3 : 0;
}

/* Number of allowed (q row, k row) pairs, per head.  [P1] §1.1: this is     */
/* the work term W_attn ~ sum_j l_j^2 of a pack.                             */
int64_t or_pair_count(int32_t Tq, int32_t Tk, const int32_t *cu, int32_t ndocs,
                      const or_mask_t *m, int32_t brute) {
    ctx_t c;
    if (ctx_init(&c, cu, ndocs, Tq, Tk, m) != 0) return -1;
    int64_t total = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : total)
    for (int32_t i = 0; i < Tq; ++i) {
        int32_t lo[2], hi[2];
        int nr = candidates(&c, i, brute, lo, hi);
        for (int r = 0; r < nr; ++r)
            for (int32_t j = lo[r]; j < hi[r]; ++j) total += allowed(&c, i, j);
    }
    ctx_free(&c);
    return total;
}

/* Pairwise predicate exposed for tests (brute-force tile checks). */
int or_allowed_matrix(int32_t Tq, int32_t Tk, const int32_t *cu, int32_t ndocs,
                      const or_mask_t *m, uint8_t *out) {
    ctx_t c;
    if (ctx_init(&c, cu, ndocs, Tq, Tk, m) != 0) return -1;
    for (int32_t i = 0; i < Tq; ++i)
        for (int32_t j = 0; j < Tk; ++j) out[(int64_t)i * Tk + j] = (uint8_t)allowed(&c, i, j);
    ctx_free(&c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Online-softmax merge of two partial results over disjoint key sets.       */
/* [P1] §3.2 (DCP): partial outputs of several computation blocks of one O   */
/* block are reduced by online-softmax rescale-and-sum; [P4] ring attention: */
/* each step's local result is merged into the running state.                */
/*   lse = ln(e^{lse_a} + e^{lse_b}),  O = e^{lse_a-lse} O_a + e^{lse_b-lse} O_b */
/* Both -inf: O = 0, lse = -inf.  Layout O [tokens, heads, d], lse [heads,    */
/* tokens].                                                                  */
/* ------------------------------------------------------------------------ */
void or_merge(const double *oa, const double *la, const double *ob, const double *lb, double *o,
              double *l, int64_t tokens, int32_t heads, int32_t d) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < tokens; ++t) {
        for (int32_t h = 0; h < heads; ++h) {
            double a = la[(int64_t)h * tokens + t], b = lb[(int64_t)h * tokens + t];
            const double *xa = oa + (t * heads + h) * d, *xb = ob + (t * heads + h) * d;
            double *y = o + (t * heads + h) * d;
            if (a == -INFINITY && b == -INFINITY) {
                for (int32_t e = 0; e < d; ++e) y[e] = 0.0;
                l[(int64_t)h * tokens + t] = -INFINITY;
                continue;
            }
            double mx = a > b ? a : b;
            double lse = mx + log(exp(a - mx) + exp(b - mx));
            double wa = exp(a - lse), wb = exp(b - lse);
            for (int32_t e = 0; e < d; ++e) y[e] = wa * xa[e] + wb * xb[e];
            l[(int64_t)h * tokens + t] = lse;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Worklist.                                                                 */
/* [P1] §3.2: attention is cut into tiles; Libra TAP charges each tile its   */
/* exact causal query-key pair count, and DCP creates a computation block    */
/* only for (Q block, KV block) pairs whose mask is not all zero.            */
/* [P1] §2.1 (VRSP) and [P2] §4.4 phase 1: LPT -- sort by cost, descending,  */
/* and put each item on the currently lightest bin.  Here the bins are the   */
/* persistent CTAs of one GPU.                                               */
/*                                                                           */
/* Readings where the pages leave the step open:                             */
/*  - segments: a maximal group of slices with the same query range; q tiles */
/*    of tile_m rows are aligned at the segment start, kv tiles of tile_n    */
/*    rows at each slice's key start (document-local tiles).                 */
/*  - a slice's kv span for a q tile is [floor(min lo / tile_n),             */
/*    ceil(max hi / tile_n)) over the rows' allowed key intervals.           */
/*  - units: two query sub-tiles that share one kv head and the kv tiles.    */
/*    With G = Hq/Hkv: heads (2p, 2p+1) of a group on the same q tile; if G  */
/*    is odd the group's last head pairs consecutive q tiles (2u, 2u+1).     */
/*    Enumeration order: segment, kv head, head pair, q tile; then the odd  */
/*    head's tile pairs.                                                     */
/*  - unit cost = exact allowed pairs of both sub-tiles + c_tile * (sub-tiles */
/*    * kv tiles computed + sub-tiles); c_tile = 0 is pure pair counting.    */
/*    The last term is a fixed cost per query sub-tile (its Q load and its   */
/*    output rows), the analogue of the per-sample constant c*n of the      */
/*    fitted DP load model ([P2] §4.2).                                      */
/*  - LPT ties: sort is stable on the enumeration index; the lightest bin   */
/*    with the lowest id wins a tie.                                         */
/*  - LPT fixes which bin runs a unit, not when; a bin's list is in          */
/*    enumeration order (ascending unit id), so bins that run at the same   */
/*    time work on the same segments and kv heads.                           */
/* ------------------------------------------------------------------------ */
typedef struct {
    int32_t q_row0, q_len, q_pos0, k_row0, k_len, k_pos0, type, window;
    uint32_t dmask[4]; /* packed slices: bit r set when row r starts a document */
} slice_t;

typedef struct {
    int32_t q_row0, q_len, q_pos0, slice_begin, slice_count;
} seg_t;

typedef struct {
    slice_t *sl;
    int64_t nsl, cap_sl;
    seg_t *sg;
    int64_t nsg, cap_sg;
} plan_t;

static void push_slice(plan_t *p, slice_t s) {
    if (p->nsl == p->cap_sl) {
        p->cap_sl = p->cap_sl ? 2 * p->cap_sl : 64;
        p->sl = (slice_t *)realloc(p->sl, sizeof(slice_t) * (size_t)p->cap_sl);
    }
    p->sl[p->nsl++] = s;
}

static void push_seg(plan_t *p, int32_t q_row0, int32_t q_len, int32_t q_pos0, int64_t first) {
    if (p->nsg == p->cap_sg) {
        p->cap_sg = p->cap_sg ? 2 * p->cap_sg : 64;
        p->sg = (seg_t *)realloc(p->sg, sizeof(seg_t) * (size_t)p->cap_sg);
    }
    seg_t g = {q_row0, q_len, q_pos0, (int32_t)first, (int32_t)(p->nsl - first)};
    p->sg[p->nsg++] = g;
}

/* Slices of one zigzag pair (q rank r against the KV shard of rank s):     */
/* per document, each of r's two chunks is a segment, with a CAUSAL slice   */
/* (on positions) against each of s's chunks that has an allowed pair.     */
/* qbase / kbase: first row of r's / s's shard in the Q / K buffers.        */
static void derive_zigzag_pair(const int32_t *cu, int32_t ndocs, int32_t cp, int32_t r,
                               int32_t s, int32_t qbase, int32_t kbase, plan_t *p) {
    int32_t qloc = qbase, kloc = kbase;
    for (int32_t d = 0; d < ndocs; ++d) {
        int32_t len = cu[d + 1] - cu[d];
        int32_t qc[2] = {r, 2 * cp - 1 - r}, kc[2] = {s, 2 * cp - 1 - s};
        int32_t qoff[2], qlen[2], koff[2], klen[2], kl0[2];
        for (int e = 0; e < 2; ++e) {
            zz_chunk(len, cp, qc[e], &qoff[e], &qlen[e]);
            zz_chunk(len, cp, kc[e], &koff[e], &klen[e]);
        }
        kl0[0] = kloc;
        kl0[1] = kloc + klen[0];
        int32_t ql0 = qloc;
        for (int e = 0; e < 2; ++e) {
            if (qlen[e] > 0) {
                int64_t first = p->nsl;
                for (int f = 0; f < 2; ++f) {
                    if (klen[f] <= 0) continue;
                    if (koff[f] > qoff[e] + qlen[e] - 1) continue; /* no allowed pair */
                    slice_t sl = {ql0, qlen[e], qoff[e], kl0[f], klen[f], koff[f],
                                  OR_SLICE_CAUSAL, 0};
                    push_slice(p, sl);
                }
                /* kept even with no slice: its rows then read O = 0, LSE = -inf */
                push_seg(p, ql0, qlen[e], qoff[e], first);
            }
            ql0 += qlen[e];
        }
        qloc += qlen[0] + qlen[1];
        kloc += klen[0] + klen[1];
    }
}

/* Slices of every mask kind, in the order the worklist enumerates them.    */
/* pack_docs (causal and sliding-window masks): [P1] §4.1 notes that a block */
/* shorter than a tile is still charged as a whole tile.  Reading: walking   */
/* the documents in order, a group opens at a document shorter than tile_m   */
/* and takes the following documents while each is shorter than tile_m and  */
/* the group's rows stay <= tile_m.  A group with two or more non-empty      */
/* documents is one segment with one PACKED slice over its rows (positions   */
/* counted from its first row, every row seeing its own document causally);  */
/* otherwise its documents keep their own segments.                          */
static int derive_plan(const int32_t *cu, int32_t ndocs, const or_mask_t *m, plan_t *p,
                       int32_t pack_docs, int32_t tile_m) {
    memset(p, 0, sizeof *p);
    switch (m->kind) {
    case OR_MASK_CAUSAL:
    case OR_MASK_SLIDING_WINDOW: {
        int32_t w = m->kind == OR_MASK_SLIDING_WINDOW ? m->window : 0;
        int32_t d = 0;
        while (d < ndocs) {
            int32_t len = cu[d + 1] - cu[d];
            int32_t y = d + 1, rows = len, nonempty = len > 0;
            if (pack_docs && len < tile_m) {
                while (y < ndocs && cu[y + 1] - cu[y] < tile_m && rows + (cu[y + 1] - cu[y]) <= tile_m) {
                    rows += cu[y + 1] - cu[y];
                    nonempty += cu[y + 1] > cu[y];
                    ++y;
                }
            }
            if (nonempty >= 2) {
                slice_t s = {cu[d], rows, 0, cu[d], rows, 0, OR_SLICE_PACKED, w, {0, 0, 0, 0}};
                for (int32_t z = d; z < y; ++z)
                    if (cu[z + 1] > cu[z]) {
                        int32_t r = cu[z] - cu[d];
                        s.dmask[r / 32] |= 1u << (r % 32);
                    }
                int64_t first = p->nsl;
                push_slice(p, s);
                push_seg(p, cu[d], rows, 0, first);
            } else {
                for (int32_t z = d; z < y; ++z) {
                    int32_t l = cu[z + 1] - cu[z];
                    if (l <= 0) continue;
                    int64_t first = p->nsl;
                    slice_t s = {cu[z], l, 0, cu[z], l, 0, OR_SLICE_CAUSAL, w, {0, 0, 0, 0}};
                    push_slice(p, s);
                    push_seg(p, cu[z], l, 0, first);
                }
            }
            d = y;
        }
        return 0;
    }
    case OR_MASK_SHARED_QUESTION:
        if (m->num_prefix < 0 || m->num_prefix > ndocs) return -1;
        for (int32_t d = 0; d < ndocs; ++d) {
            int32_t len = cu[d + 1] - cu[d];
            if (len <= 0) continue;
            int64_t first = p->nsl;
            if (d >= m->num_prefix) {
                for (int32_t q = 0; q < m->num_prefix; ++q) {
                    int32_t ql = cu[q + 1] - cu[q];
                    if (ql <= 0) continue;
                    slice_t s = {cu[d], len, 0, cu[q], ql, 0, OR_SLICE_FULL, 0};
                    push_slice(p, s);
                }
            }
            slice_t s = {cu[d], len, 0, cu[d], len, 0, OR_SLICE_CAUSAL, 0};
            push_slice(p, s);
            push_seg(p, cu[d], len, 0, first);
        }
        return 0;
    case OR_MASK_ZIGZAG_PAIR: {
        int32_t cp = m->cp, r = m->q_rank, s = m->k_rank;
        if (cp <= 0 || r < 0 || r >= cp || s < 0 || s >= cp) return -1;
        derive_zigzag_pair(cu, ndocs, cp, r, s, 0, 0, p);
        return 0;
    }
    case OR_MASK_ZIGZAG_STEP: {
        /* rank r's Q rows start after the shards of ranks < r (ring order);   */
        /* at step t they meet the K rows of rank (r - t) mod cp, likewise     */
        int32_t cp = m->cp, t = m->ring_step;
        if (cp <= 0 || t < 0 || t >= cp) return -1;
        int32_t *base = (int32_t *)calloc((size_t)cp + 1, sizeof(int32_t));
        for (int32_t r = 0; r < cp; ++r)
            base[r + 1] = base[r] + or_zigzag_map(cu, ndocs, cp, r, NULL, NULL);
        for (int32_t r = 0; r < cp; ++r) {
            int32_t s = (r - t + cp) % cp;
            derive_zigzag_pair(cu, ndocs, cp, r, s, base[r], base[s], p);
        }
        free(base);
        return 0;
    }
    case OR_MASK_SLICES: {
        int64_t i = 0;
        while (i < m->num_slices) {
            const int32_t *a = m->slices + 8 * i;
            int64_t first = p->nsl;
            int64_t j = i;
            while (j < m->num_slices) {
                const int32_t *b = m->slices + 8 * j;
                if (b[0] != a[0] || b[1] != a[1] || b[2] != a[2]) break;
                slice_t s = {b[0], b[1], b[2], b[3], b[4], b[5], b[6], b[7]};
                push_slice(p, s);
                ++j;
            }
            push_seg(p, a[0], a[1], a[2], first);
            i = j;
        }
        /* q ranges of different segments must not overlap */
        for (int64_t x = 0; x < p->nsg; ++x)
            for (int64_t y = x + 1; y < p->nsg; ++y) {
                const seg_t *A = &p->sg[x], *B = &p->sg[y];
                if (A->q_row0 < B->q_row0 + B->q_len && B->q_row0 < A->q_row0 + A->q_len)
                    return -1;
            }
        return 0;
    }
    }
    return -1;
}

/* Allowed key interval [lo, hi) (slice-local key index) of one query row    */
/* r (slice-local): d is the index of the key at the query's position.       */
static void row_interval(const slice_t *s, int32_t r, int64_t *lo, int64_t *hi) {
    int64_t d = (int64_t)s->q_pos0 + r - s->k_pos0;
    int64_t l = 0, h = s->k_len;
    switch (s->type) {
    case OR_SLICE_CAUSAL:
        h = d + 1;
        if (s->window > 0) l = d - s->window + 1;
        break;
    case OR_SLICE_INV_CAUSAL:
        l = d;
        if (s->window > 0) h = d + s->window;
        break;
    case OR_SLICE_BI_CAUSAL:
        l = d;
        h = (int64_t)s->k_len - s->q_len + r + 1;
        break;
    case OR_SLICE_PACKED: {
        /* own document: from the nearest document start at or before row r */
        int32_t st = r;
        while (st > 0 && !((s->dmask[st / 32] >> (st % 32)) & 1u)) --st;
        l = st;
        h = d + 1;
        if (s->window > 0 && d - s->window + 1 > l) l = d - s->window + 1;
        break;
    }
    default: /* FULL */
        break;
    }
    if (l < 0) l = 0;
    if (h > s->k_len) h = s->k_len;
    *lo = l;
    *hi = h;
}

/* kv tile span and pair count of q tile t of segment g against slice s.    */
static void tile_span(const seg_t *g, const slice_t *s, int32_t t, int32_t tile_m, int32_t tile_n,
                      int32_t *lo_t, int32_t *hi_t, int64_t *pairs) {
    int64_t mn = INT64_MAX, mx = -1, cnt = 0;
    int32_t r0 = t * tile_m, r1 = r0 + tile_m;
    if (r1 > g->q_len) r1 = g->q_len;
    for (int32_t r = r0; r < r1; ++r) {
        int64_t lo, hi;
        row_interval(s, r, &lo, &hi);
        if (hi <= lo) continue;
        cnt += hi - lo;
        if (lo < mn) mn = lo;
        if (hi > mx) mx = hi;
    }
    if (cnt == 0) {
        *lo_t = *hi_t = 0;
    } else {
        *lo_t = (int32_t)(mn / tile_n);
        *hi_t = (int32_t)((mx + tile_n - 1) / tile_n);
    }
    *pairs = cnt;
}

typedef struct {
    int32_t seg, t0, t1, h0, h1, kvh;
    int64_t run_begin;
    int32_t run_count;
    int64_t pairs, cost, tiles;
} unit_t;

typedef struct {
    int64_t load;
    int32_t id;
} bin_t;

static int bin_less(const bin_t *a, const bin_t *b) {
    return a->load < b->load || (a->load == b->load && a->id < b->id);
}

static void heap_down(bin_t *h, int32_t n, int32_t i) {
    for (;;) {
        int32_t l = 2 * i + 1, r = l + 1, s = i;
        if (l < n && bin_less(&h[l], &h[s])) s = l;
        if (r < n && bin_less(&h[r], &h[s])) s = r;
        if (s == i) return;
        bin_t t = h[i];
        h[i] = h[s];
        h[s] = t;
        i = s;
    }
}

typedef struct {
    int64_t cost;
    int64_t idx;
} key_t_;

static int key_cmp(const void *a, const void *b) {
    const key_t_ *x = (const key_t_ *)a, *y = (const key_t_ *)b;
    if (x->cost != y->cost) return x->cost > y->cost ? -1 : 1; /* cost descending */
    return x->idx < y->idx ? -1 : (x->idx > y->idx ? 1 : 0);  /* then index ascending */
}

/* LPT with a binary min-heap over (load, id). [P1] §2.1, [P2] §4.4.       */
int or_lpt(const int64_t *cost, int64_t n, int32_t bins, int32_t *assign, int64_t *order,
           int64_t *loads) {
    if (bins <= 0) return -1;
    key_t_ *keys = (key_t_ *)malloc(sizeof(key_t_) * (size_t)(n > 0 ? n : 1));
    for (int64_t i = 0; i < n; ++i) {
        keys[i].cost = cost[i];
        keys[i].idx = i;
    }
    qsort(keys, (size_t)n, sizeof(key_t_), key_cmp);
    bin_t *h = (bin_t *)malloc(sizeof(bin_t) * (size_t)bins);
    for (int32_t b = 0; b < bins; ++b) {
        h[b].load = 0;
        h[b].id = b;
    }
    /* all loads zero: ids ascending already form a valid heap */
    for (int64_t i = 0; i < n; ++i) {
        int64_t u = keys[i].idx;
        assign[u] = h[0].id;
        if (order) order[i] = u;
        h[0].load += keys[i].cost;
        heap_down(h, bins, 0);
    }
    if (loads) {
        for (int32_t b = 0; b < bins; ++b) loads[h[b].id] = h[b].load;
    }
    free(h);
    free(keys);
    return 0;
}

/* Worklist: counts first (out arrays NULL), then fill. counts[0..4] =      */
/* segments, slices, units, runs, total pairs per head.                      */
/* Iterative move/swap refinement after LPT ("数据并行负载均衡" §4.4, phase 2), */
/* at most max_iters rounds.  Each round takes the most loaded bin (ties:    */
/* lower id) and the least loaded one (ties: lower id) and stops once their */
/* gap is under 5% of the largest load.  Candidates: move the costliest item */
/* of the heavy bin to the light one, or swap it with the cheapest item of  */
/* the light bin (ties between items: lower index).  The candidate leaving  */
/* the smaller gap between the two bins is applied (a move on a tie) if it  */
/* is smaller than the current gap; otherwise the refinement stops.         */
/* Returns the number of rounds applied; loads are updated with assign.     */
int or_refine_move_swap(const int64_t *cost, int64_t n, int32_t bins, int32_t *assign,
                        int64_t *loads, int32_t max_iters) {
    int32_t done = 0;
    for (int32_t it = 0; it < max_iters && bins > 1; ++it) {
        int32_t bmax = 0, bmin = 0;
        for (int32_t b = 1; b < bins; ++b) {
            if (loads[b] > loads[bmax]) bmax = b;
            if (loads[b] < loads[bmin]) bmin = b;
        }
        int64_t gap = loads[bmax] - loads[bmin];
        if (gap * 20 < loads[bmax] || gap == 0) break;
        int64_t x = -1, y = -1;
        for (int64_t u = 0; u < n; ++u) {
            if (assign[u] == bmax && (x < 0 || cost[u] > cost[x])) x = u;
            if (assign[u] == bmin && (y < 0 || cost[u] < cost[y])) y = u;
        }
        if (x < 0) break;
        int64_t g_move = gap - 2 * cost[x];
        if (g_move < 0) g_move = -g_move;
        int64_t g_swap = INT64_MAX;
        if (y >= 0) {
            g_swap = gap - 2 * (cost[x] - cost[y]);
            if (g_swap < 0) g_swap = -g_swap;
        }
        if (g_move >= gap && g_swap >= gap) break;
        if (g_move <= g_swap) {
            assign[x] = bmin;
            loads[bmax] -= cost[x];
            loads[bmin] += cost[x];
        } else {
            assign[x] = bmin;
            assign[y] = bmax;
            loads[bmax] += cost[y] - cost[x];
            loads[bmin] += cost[x] - cost[y];
        }
        ++done;
    }
    return done;
}

/* Non-negative least-squares fit of the per-tile cost to measured per-bin  */
/* times ("数据并行负载均衡" §4.2: the load model a·Σlen² + b·Σlen + c·n is     */
/* fitted to measured times with non-negative coefficients, no constant).    */
/* Per bin b with P_b allowed pairs and U_b = (sub-tile, kv tile) steps +    */
/* query sub-tiles:  t_b ~ a P_b + c U_b,  a, c >= 0.  With two unknowns the */
/* exact non-negative solution is the unconstrained one if it is feasible,   */
/* else the better (smaller residual) of (a, 0) and (0, c) fitted alone.     */
/* coef = {a, c}.  Returns round(c / a), the per-tile cost in pair units,   */
/* at most 2^24;                                                             */
/* a = 0 < c (time follows tiles alone) returns 2^24; -1 if both are zero    */
/* or there is no sample.                                                    */
#define OR_FIT_TILE_CAP (1LL << 24)

int64_t or_fit_tile_cost(const int64_t *P, const int64_t *U, const double *t, int32_t nb,
                         double *coef) {
    double pp = 0, uu = 0, pu = 0, pt = 0, ut = 0, tt = 0;
    for (int32_t b = 0; b < nb; ++b) {
        double p = (double)P[b], u = (double)U[b];
        pp += p * p;
        uu += u * u;
        pu += p * u;
        pt += p * t[b];
        ut += u * t[b];
        tt += t[b] * t[b];
    }
    double a = 0, c = 0;
    double det = pp * uu - pu * pu;
    int ok = 0;
    if (det > 0) {
        a = (pt * uu - pu * ut) / det;
        c = (pp * ut - pu * pt) / det;
        ok = a >= 0 && c >= 0;
    }
    if (!ok) {
        /* residual of t ~ x f: tt - 2 x ft + x^2 ff */
        double a1 = pp > 0 && pt > 0 ? pt / pp : 0, c1 = uu > 0 && ut > 0 ? ut / uu : 0;
        double r_a = tt - 2 * a1 * pt + a1 * a1 * pp;
        double r_c = tt - 2 * c1 * ut + c1 * c1 * uu;
        if (r_a <= r_c) {
            a = a1;
            c = 0;
        } else {
            a = 0;
            c = c1;
        }
    }
    if (coef) {
        coef[0] = a;
        coef[1] = c;
    }
    if (a > 0) {
        double r = c / a;
        return r >= (double)OR_FIT_TILE_CAP ? OR_FIT_TILE_CAP : (int64_t)llround(r);
    }
    return c > 0 ? OR_FIT_TILE_CAP : -1;
}

int or_worklist(const int32_t *cu, int32_t ndocs, const or_mask_t *m, int32_t tile_m,
                int32_t tile_n, int32_t Hq, int32_t Hkv, int32_t num_ctas, int64_t c_tile,
                int32_t refine_iters, int32_t pack_docs,
                int64_t *counts, int32_t *slices_out, uint32_t *slice_masks_out,
                int32_t *segs_out, int32_t *units_out,
                int64_t *unit_cost_out, int64_t *unit_pairs_out, int32_t *runs_out,
                int32_t *cta_off_out) {
    if (tile_m <= 0 || tile_n <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_ctas <= 0) return -1;
    if (pack_docs && tile_m > 128) return -1; /* a packed slice's rows fit one 128-bit mask */
    plan_t p;
    if (derive_plan(cu, ndocs, m, &p, pack_docs, tile_m) != 0) {
        free(p.sl);
        free(p.sg);
        return -2;
    }
    const int32_t G = Hq / Hkv;
    int64_t nunits = 0, nruns = 0, pairs_head = 0;
    for (int64_t g = 0; g < p.nsg; ++g) {
        int32_t nt = (p.sg[g].q_len + tile_m - 1) / tile_m;
        int64_t u = (int64_t)Hkv * ((int64_t)(G / 2) * nt + (G % 2) * ((nt + 1) / 2));
        nunits += u;
        nruns += u * p.sg[g].slice_count;
        for (int32_t sidx = 0; sidx < p.sg[g].slice_count; ++sidx)
            for (int32_t t = 0; t < nt; ++t) {
                int32_t a, b;
                int64_t pr;
                tile_span(&p.sg[g], &p.sl[p.sg[g].slice_begin + sidx], t, tile_m, tile_n, &a, &b,
                          &pr);
                pairs_head += pr;
            }
    }
    counts[0] = p.nsg;
    counts[1] = p.nsl;
    counts[2] = nunits;
    counts[3] = nruns;
    counts[4] = pairs_head;
    if (!units_out) {
        free(p.sl);
        free(p.sg);
        return 0;
    }
    for (int64_t i = 0; i < p.nsl; ++i) {
        const slice_t *s = &p.sl[i];
        int32_t *o = slices_out + 8 * i;
        o[0] = s->q_row0; o[1] = s->q_len; o[2] = s->q_pos0; o[3] = s->k_row0;
        o[4] = s->k_len; o[5] = s->k_pos0; o[6] = s->type; o[7] = s->window;
        if (slice_masks_out)
            for (int e = 0; e < 4; ++e) slice_masks_out[4 * i + e] = s->dmask[e];
    }
    for (int64_t g = 0; g < p.nsg; ++g) {
        int32_t *o = segs_out + 5 * g;
        o[0] = p.sg[g].q_row0; o[1] = p.sg[g].q_len; o[2] = p.sg[g].q_pos0;
        o[3] = p.sg[g].slice_begin; o[4] = p.sg[g].slice_count;
    }
    unit_t *U = (unit_t *)malloc(sizeof(unit_t) * (size_t)(nunits > 0 ? nunits : 1));
    int64_t ui = 0, ri = 0;
    for (int64_t g = 0; g < p.nsg; ++g) {
        const seg_t *sg = &p.sg[g];
        int32_t nt = (sg->q_len + tile_m - 1) / tile_m;
        for (int32_t kvh = 0; kvh < Hkv; ++kvh) {
            /* head pairs on the same q tile, then the odd head's tile pairs */
            int32_t npair = G / 2;
            int64_t total_here = (int64_t)npair * nt + (G % 2) * ((nt + 1) / 2);
            for (int64_t e = 0; e < total_here; ++e) {
                unit_t u;
                u.seg = (int32_t)g;
                u.kvh = kvh;
                if (e < (int64_t)npair * nt) {
                    int32_t pp = (int32_t)(e / nt), t = (int32_t)(e % nt);
                    u.t0 = u.t1 = t;
                    u.h0 = kvh * G + 2 * pp;
                    u.h1 = u.h0 + 1;
                } else {
                    int32_t uu = (int32_t)(e - (int64_t)npair * nt);
                    u.t0 = 2 * uu;
                    u.t1 = (2 * uu + 1 < nt) ? 2 * uu + 1 : -1;
                    u.h0 = kvh * G + G - 1;
                    u.h1 = (u.t1 >= 0) ? u.h0 : -1;
                }
                int nsub = (u.h1 >= 0) ? 2 : 1;
                u.run_begin = ri;
                u.run_count = sg->slice_count;
                u.pairs = 0;
                u.tiles = 0;
                for (int32_t sidx = 0; sidx < sg->slice_count; ++sidx) {
                    const slice_t *s = &p.sl[sg->slice_begin + sidx];
                    int32_t lo = 0, hi = 0, have = 0;
                    int32_t ts[2] = {u.t0, u.t1};
                    for (int k2 = 0; k2 < nsub; ++k2) {
                        int32_t a, b;
                        int64_t pr;
                        tile_span(sg, s, ts[k2], tile_m, tile_n, &a, &b, &pr);
                        u.pairs += pr;
                        if (b > a) {
                            if (!have || a < lo) lo = a;
                            if (!have || b > hi) hi = b;
                            have = 1;
                        }
                    }
                    int32_t *ro = runs_out + 3 * ri;
                    ro[0] = sg->slice_begin + sidx;
                    ro[1] = lo;
                    ro[2] = hi;
                    u.tiles += (int64_t)(hi - lo) * nsub;
                    ++ri;
                }
                u.cost = u.pairs + c_tile * (u.tiles + nsub);
                U[ui++] = u;
            }
        }
    }
    int64_t *cost = (int64_t *)calloc((size_t)(nunits > 0 ? nunits : 1), sizeof(int64_t));
    int32_t *assign = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nunits > 0 ? nunits : 1));
    for (int64_t i = 0; i < nunits; ++i) cost[i] = U[i].cost;
    int64_t *bload = (int64_t *)calloc((size_t)num_ctas, sizeof(int64_t));
    or_lpt(cost, nunits, num_ctas, assign, NULL, bload);
    if (refine_iters > 0) or_refine_move_swap(cost, nunits, num_ctas, assign, bload, refine_iters);
    free(bload);
    /* CSR: per bin, units in enumeration order */
    int32_t *fill = (int32_t *)calloc((size_t)num_ctas + 1, sizeof(int32_t));
    for (int64_t i = 0; i < nunits; ++i) fill[assign[i] + 1]++;
    for (int32_t b = 0; b < num_ctas; ++b) fill[b + 1] += fill[b];
    for (int32_t b = 0; b <= num_ctas; ++b) cta_off_out[b] = fill[b];
    for (int64_t u = 0; u < nunits; ++u) {
        int32_t pos = fill[assign[u]]++;
        int32_t *o = units_out + 10 * (int64_t)pos;
        o[0] = (int32_t)u; o[1] = U[u].seg; o[2] = U[u].t0; o[3] = U[u].t1; o[4] = U[u].h0;
        o[5] = U[u].h1; o[6] = U[u].kvh; o[7] = (int32_t)U[u].run_begin; o[8] = U[u].run_count;
        o[9] = assign[u];
        unit_cost_out[pos] = U[u].cost;
        unit_pairs_out[pos] = U[u].pairs;
    }
    free(fill);
    free(assign);
    free(cost);
    free(U);
    free(p.sl);
    free(p.sg);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Dispatch and sharding solvers ("03 · 长文负载均衡" §4.2-§4.4).              */
/* ------------------------------------------------------------------------ */

/* Mask area of equal query chunks (§4.4, MagiAttention's dispatch: the      */
/* global sequence is cut along the query dimension into chunks of           */
/* chunk_size rows, the last one possibly shorter; a chunk's area is the     */
/* number of allowed query-key pairs of its rows).  Masks over the whole     */
/* pack only (causal, sliding window, shared question).                      */
int or_chunk_areas(int32_t T, const int32_t *cu, int32_t ndocs, const or_mask_t *m,
                   int32_t chunk_size, int64_t *areas) {
    if (chunk_size <= 0 || T < 0) return -1;
    if (m->kind == OR_MASK_ZIGZAG_PAIR || m->kind == OR_MASK_ZIGZAG_STEP ||
        m->kind == OR_MASK_SLICES)
        return -1;
    ctx_t c;
    if (ctx_init(&c, cu, ndocs, T, T, m) != 0) return -2;
    int32_t n = (T + chunk_size - 1) / chunk_size;
    for (int32_t k = 0; k < n; ++k) areas[k] = 0;
    for (int32_t i = 0; i < T; ++i) {
        int32_t lo[2], hi[2];
        int nr = candidates(&c, i, 0, lo, hi);
        int64_t cnt = 0;
        for (int r = 0; r < nr; ++r)
            for (int32_t j = lo[r]; j < hi[r]; ++j) cnt += allowed(&c, i, j);
        areas[i / chunk_size] += cnt;
    }
    ctx_free(&c);
    return n;
}

/* Greedy dispatch of n chunks into cp buckets of exactly n/cp chunks each,  */
/* minimising the largest bucket area (§4.4): chunks are taken by area,      */
/* largest first (equal areas: lower chunk index first); each goes to the    */
/* bucket with the smallest area that still has room (equal areas: lower     */
/* bucket id), the buckets kept in a binary min-heap from which a full       */
/* bucket is removed.  bucket[n] gets each chunk's bucket, loads[cp] the     */
/* bucket areas.                                                             */
typedef struct {
    int64_t area;
    int32_t idx;
} chunk_key_t;

static int chunk_key_cmp(const void *a, const void *b) {
    const chunk_key_t *x = (const chunk_key_t *)a, *y = (const chunk_key_t *)b;
    if (x->area != y->area) return x->area > y->area ? -1 : 1;
    return x->idx < y->idx ? -1 : x->idx > y->idx;
}

int or_dispatch_minheap(const int64_t *areas, int32_t n, int32_t cp, int32_t *bucket,
                        int64_t *loads) {
    if (cp <= 0 || n < 0 || n % cp != 0) return -1;
    chunk_key_t *key = (chunk_key_t *)malloc(sizeof(chunk_key_t) * (size_t)(n > 0 ? n : 1));
    for (int32_t i = 0; i < n; ++i) {
        key[i].area = areas[i];
        key[i].idx = i;
    }
    qsort(key, (size_t)n, sizeof(chunk_key_t), chunk_key_cmp);
    bin_t *heap = (bin_t *)malloc(sizeof(bin_t) * (size_t)cp);
    int32_t *fill = (int32_t *)calloc((size_t)cp, sizeof(int32_t));
    for (int32_t b = 0; b < cp; ++b) {
        heap[b].load = 0;
        heap[b].id = b;
    }
    for (int32_t b = 0; b < cp; ++b) loads[b] = 0;
    int32_t hn = cp;  /* all loads 0 and ids ascending: already a heap */
    const int32_t cap = n / cp;
    for (int32_t t = 0; t < n; ++t) {
        bin_t top = heap[0];
        bucket[key[t].idx] = top.id;
        top.load += key[t].area;
        if (++fill[top.id] == cap) {
            heap[0] = heap[--hn];  /* full: leaves the heap */
        } else {
            heap[0] = top;
        }
        if (hn > 0) heap_down(heap, hn, 0);
        loads[top.id] = top.load;
    }
    free(fill);
    free(heap);
    free(key);
    return 0;
}

/* Striped sharding (§4.2: Striped Attention interleaves stripes of the      */
/* whole sequence across the ranks): token i belongs to rank                 */
/* (i / stripe) mod cp.  Writes rank r's tokens in order (map may be NULL)   */
/* and returns their count.                                                  */
int32_t or_striped_map(int32_t T, int32_t cp, int32_t rank, int32_t stripe, int32_t *map) {
    if (cp <= 0 || rank < 0 || rank >= cp || stripe <= 0 || T < 0) return -1;
    int32_t n = 0;
    for (int32_t i = 0; i < T; ++i)
        if ((i / stripe) % cp == rank) {
            if (map) map[n] = i;
            ++n;
        }
    return n;
}

/* Tile-rounded causal attention FLOPs of query positions [p0, p1) of one    */
/* document (§4.1 via §4.3: a block shorter than a tile is charged a whole   */
/* tile): q tiles of `tile` rows aligned at p0; q tile rows with last        */
/* position P see keys [0, P], i.e. ceil((P + 1) / tile) key tiles of        */
/* tile x tile pairs, each pair 4 d FLOPs.                                   */
static int64_t piece_flops(int32_t p0, int32_t p1, int32_t tile, int32_t d) {
    int64_t tiles = 0;
    for (int32_t r = p0; r < p1; r += tile) {
        int32_t last = r + tile < p1 ? r + tile - 1 : p1 - 1;
        tiles += (last + 1 + tile - 1) / tile;
    }
    return tiles * (int64_t)tile * tile * 4 * d;
}

/* WLB-LLM's per-micro-batch choice between per-sequence and per-document    */
/* zigzag sharding (§4.3): for each scheme, every CP worker's attention work  */
/* in tile-rounded FLOPs; the predicted latency of a scheme is its most      */
/* loaded worker and the smaller one wins (equal: per-sequence).             */
/*  - per-sequence: the whole pack is cut into 2 cp chunks by the zigzag     */
/*    chunk rule and worker r takes chunks r and 2 cp - 1 - r; each chunk's  */
/*    pieces inside documents are charged as above (positions are document  */
/*    positions, the causal mask never crosses documents).                   */
/*  - per-document: every document is cut into 2 cp chunks and worker r     */
/*    takes its chunks r and 2 cp - 1 - r.                                    */
/* costs[2 cp]: per worker, per-sequence then per-document.  Returns 0       */
/* (per-sequence) or 1 (per-document), -1 on bad arguments.                 */
int or_wlb_choose(const int32_t *cu, int32_t ndocs, int32_t cp, int32_t tile, int32_t d,
                  int64_t *costs) {
    if (cp <= 0 || tile <= 0 || d <= 0 || ndocs < 0) return -1;
    int32_t T = cu[ndocs];
    for (int32_t r = 0; r < 2 * cp; ++r) costs[r] = 0;
    for (int32_t r = 0; r < cp; ++r) {
        int32_t chunks[2] = {r, 2 * cp - 1 - r};
        for (int e = 0; e < 2; ++e) {
            int32_t off, len;
            zz_chunk(T, cp, chunks[e], &off, &len);
            for (int32_t dd = 0; dd < ndocs; ++dd) {
                int32_t a = off > cu[dd] ? off : cu[dd];
                int32_t b = off + len < cu[dd + 1] ? off + len : cu[dd + 1];
                if (a < b) costs[r] += piece_flops(a - cu[dd], b - cu[dd], tile, d);
            }
            for (int32_t dd = 0; dd < ndocs; ++dd) {
                zz_chunk(cu[dd + 1] - cu[dd], cp, chunks[e], &off, &len);
                if (len > 0) costs[cp + r] += piece_flops(off, off + len, tile, d);
            }
        }
    }
    int64_t mseq = 0, mdoc = 0;
    for (int32_t r = 0; r < cp; ++r) {
        if (costs[r] > mseq) mseq = costs[r];
        if (costs[cp + r] > mdoc) mdoc = costs[cp + r];
    }
    return mdoc < mseq ? 1 : 0;
}
