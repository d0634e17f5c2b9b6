/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY. The plain, slow, fp64 CPU definition of what the
 * context-parallel ring-attention forward computes. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the library's product path never does. It shares no
 * code, header or table with the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [CPC] "Context Parallelism (CP)" concept page (gunjandhanuka.github.io research hub):
 *         "Definition"; "Key math / How it works".
 *   [CPP] "primitive-context-parallel" skill page (skillsmp.com): "What it does"; "Memory".
 *   [CEX] "Context and expert parallelism" (zerotofrontier.app/distributed/context-expert):
 *         "Splitting the sequence, and the one layer that objects"; "What context
 *         parallelism communicates"; "When the ring hides its communication"; "The causal
 *         mask unbalances the sequence"; "Ulysses, splitting by heads instead".
 *
 * Readings where the pages are silent or garbled (each restated where it is used):
 *   causal mask includes the diagonal (key u visible to query t iff pos[u] <= pos[t]);
 *   scale defaults to 1/sqrt(d_k); lse is the natural log of the sum of exp(scaled scores);
 *   query head i reads KV head floor(i / (h / n_kv)); the contiguous interval is half-open;
 *   zigzag puts chunk r first, then chunk 2n_cp-1-r; striped is per token (t -> rank t mod
 *   n_cp, local index t div n_cp); at ring step s rank r holds the block of (r - s) mod n_cp.
 *
 * Parity status: every function below is pinned by the CPU tests (closed forms, the pages'
 * printed figures, brute force on small inputs, agreement of the ring simulation with the
 * definition, and a library softmax-attention routine; for the gradients also central finite
 * differences of the forward definition and a library's automatic differentiation). Nothing
 * here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { LAYOUT_CONTIGUOUS = 0, LAYOUT_ZIGZAG = 1, LAYOUT_STRIPED = 2 };
enum { CLASS_FULL = 0, CLASS_DIAG = 1, CLASS_SKIP = 2 };

static double bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------------------------- */
/* Token placement. [CEX] "Splitting the sequence...": contiguous chunks of T/n_cp.        */
/* [CEX] "The causal mask unbalances the sequence": zigzag = chunks r and 2n_cp-1-r of     */
/* 2n_cp; striped = round-robin tokens. [CPP] "What it does": rank i holds [i*N/cp,        */
/* (i+1)*N/cp), read as half-open.                                                         */
/* ------------------------------------------------------------------------------------- */

/* Natural token index held by rank r at local index j (0 <= j < T/n_cp); -1 on bad args. */
int64_t oracle_token_of(int64_t T, int n_cp, int layout, int r, int64_t j) {
    if (n_cp <= 0 || T % n_cp) return -1;
    int64_t n = T / n_cp;
    if (r < 0 || r >= n_cp || j < 0 || j >= n) return -1;
    if (layout == LAYOUT_CONTIGUOUS) return (int64_t)r * n + j;
    if (layout == LAYOUT_ZIGZAG) {
        if (T % (2 * n_cp)) return -1;
        int64_t m = T / (2 * n_cp);
        if (j < m) return (int64_t)r * m + j;                 /* chunk r, from the front   */
        return (int64_t)(2 * n_cp - 1 - r) * m + (j - m);     /* its mirror from the back  */
    }
    if (layout == LAYOUT_STRIPED) return j * n_cp + r;
    return -1;
}

/* map[r*n + j] = natural token of (rank r, local j). Returns 0 on success. */
int oracle_layout_map(int64_t T, int n_cp, int layout, int64_t* map) {
    if (n_cp <= 0 || T % n_cp) return 1;
    int64_t n = T / n_cp;
    for (int r = 0; r < n_cp; ++r)
        for (int64_t j = 0; j < n; ++j) {
            int64_t t = oracle_token_of(T, n_cp, layout, r, j);
            if (t < 0) return 1;
            map[(int64_t)r * n + j] = t;
        }
    return 0;
}

/* The chunks a rank holds, at chunk granularity: contiguous -> {r} of n_cp chunks; zigzag ->
 * {r, 2n_cp-1-r} of 2n_cp chunks. Writes up to 2 ids, returns how many (0 for striped, whose
 * unit is a single token). This is the exercise "chunk_assignment" of [CEX], done right. */
int oracle_chunk_assignment(int n_cp, int layout, int r, int* chunks) {
    if (layout == LAYOUT_CONTIGUOUS) { chunks[0] = r; return 1; }
    if (layout == LAYOUT_ZIGZAG) { chunks[0] = r; chunks[1] = 2 * n_cp - 1 - r; return 2; }
    return 0;
}

/* ------------------------------------------------------------------------------------- */
/* Attention, the definition. [CEX] "Splitting the sequence...": "the query of token i     */
/* must see the keys and values of every earlier token" (read inclusively); [CEX] "Pass    */
/* them around a ring" and [CPC] "Key math": the ring with online softmax is exact, so the */
/* result is full softmax attention:                                                        */
/*   lse[b,i,t] = ln sum_{u in V(t)} exp(s_u),  O[b,t,i,:] = sum_u exp(s_u - lse) v[b,u,kv,:] */
/*   s_u = scale * <q[b,t,i,:], k[b,u,kv,:]>,  kv = floor(i / (h/n_kv)),                     */
/*   V(t) = {u : pos[u] <= pos[t]} if causal, else all u.                                   */
/* Two passes per row (max, then sums), natural order, fp64 from exact bf16 values.        */
/* ------------------------------------------------------------------------------------- */

static int visible(const int32_t* pos, int64_t u, int64_t t, int causal) {
    if (!causal) return 1;
    int64_t pu = pos ? pos[u] : u;
    int64_t pt = pos ? pos[t] : t;
    return pu <= pt;
}

/* Document masks for packed sequences ([CEX] "What context parallelism communicates": the
 * all-gather variant "makes arbitrary masks, such as document masks for packed sequences, easy
 * to support"): with a document id per token, a query sees only keys of its own document (and,
 * causal, only those at or before it). doc NULL: one document. */
static int visible_doc(const int32_t* pos, const int32_t* doc, int64_t u, int64_t t, int causal) {
    if (doc && doc[u] != doc[t]) return 0;
    return visible(pos, u, t, causal);
}

/* q [B,T,h,d], k/v [B,T,n_kv,d] bf16 bits, natural order. rows: n_rows natural token ids or
 * NULL (all T, n_rows = T). keys: n_keys natural token ids the queries may attend to (one
 * block of the ring, or any key subset), or NULL for all T; a key outside the mask stays
 * hidden. o [B,n_rows,h,d] fp64, lse [B,h,n_rows] fp64 (-inf when a row sees no key, with
 * o = 0). Returns 0 on success. */
static int attention_impl(int B, int64_t T, int h, int n_kv, int d, const uint16_t* q, const uint16_t* k,
                          const uint16_t* v, const int32_t* pos, const int32_t* doc, int causal, double scale,
                          int64_t n_rows, const int64_t* rows, int64_t n_keys, const int64_t* keys, double* o,
                          double* lse) {
    if (B <= 0 || T <= 0 || h <= 0 || n_kv <= 0 || d <= 0 || h % n_kv) return 1;
    if (!rows) n_rows = T;
    if (!keys) n_keys = T;
    int g = h / n_kv;
    int64_t total = (int64_t)B * n_rows * h;
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        if (!s || !acc) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t w = 0; w < total; ++w) {
            if (!s || !acc) continue;
            int i = (int)(w % h);
            int64_t ri = (w / h) % n_rows;
            int b = (int)(w / ((int64_t)h * n_rows));
            int64_t t = rows ? rows[ri] : ri;
            int kv = i / g;
            const uint16_t* qrow = q + (((int64_t)b * T + t) * h + i) * d;
            /* pass 1: scores of the visible keys and their maximum */
            double mx = -INFINITY;
            for (int64_t ki = 0; ki < n_keys; ++ki) {
                int64_t u = keys ? keys[ki] : ki;
                if (!visible_doc(pos, doc, u, t, causal)) continue;
                const uint16_t* krow = k + (((int64_t)b * T + u) * n_kv + kv) * d;
                double dot = 0.0;
                for (int c = 0; c < d; ++c) dot += bf16_value(qrow[c]) * bf16_value(krow[c]);
                s[ki] = scale * dot;
                if (s[ki] > mx) mx = s[ki];
            }
            double* orow = o + (((int64_t)b * n_rows + ri) * h + i) * d;
            double* lrow = lse + ((int64_t)b * h + i) * n_rows + ri;
            if (mx == -INFINITY) {
                for (int c = 0; c < d; ++c) orow[c] = 0.0;
                *lrow = -INFINITY;
                continue;
            }
            /* pass 2: sum of exponentials and the exponential-weighted sum of values */
            double sum = 0.0;
            for (int c = 0; c < d; ++c) acc[c] = 0.0;
            for (int64_t ki = 0; ki < n_keys; ++ki) {
                int64_t u = keys ? keys[ki] : ki;
                if (!visible_doc(pos, doc, u, t, causal)) continue;
                double e = exp(s[ki] - mx);
                sum += e;
                const uint16_t* vrow = v + (((int64_t)b * T + u) * n_kv + kv) * d;
                for (int c = 0; c < d; ++c) acc[c] += e * bf16_value(vrow[c]);
            }
            for (int c = 0; c < d; ++c) orow[c] = acc[c] / sum;
            *lrow = mx + log(sum);
        }
        free(s);
        free(acc);
    }
    return err;
}

int oracle_attention(int B, int64_t T, int h, int n_kv, int d, const uint16_t* q, const uint16_t* k,
                     const uint16_t* v, const int32_t* pos, int causal, double scale, int64_t n_rows,
                     const int64_t* rows, int64_t n_keys, const int64_t* keys, double* o, double* lse) {
    return attention_impl(B, T, h, n_kv, d, q, k, v, pos, NULL, causal, scale, n_rows, rows, n_keys, keys, o, lse);
}

/* The same definition under a document mask: doc [T] int32 document id of each natural token. */
int oracle_attention_docs(int B, int64_t T, int h, int n_kv, int d, const uint16_t* q, const uint16_t* k,
                          const uint16_t* v, const int32_t* pos, const int32_t* doc, int causal, double scale,
                          int64_t n_rows, const int64_t* rows, double* o, double* lse) {
    return attention_impl(B, T, h, n_kv, d, q, k, v, pos, doc, causal, scale, n_rows, rows, 0, NULL, o, lse);
}

/* ------------------------------------------------------------------------------------- */
/* The ring, simulated literally. [CEX] "Pass them around a ring": in each of n_cp steps   */
/* every rank attends to the block it holds, sends it right and receives from the left, so */
/* at step s rank r holds the block of rank (r - s) mod n_cp. [CEX] same section, next     */
/* paragraph, and [CPC] "Key math": a running maximum, a running sum of exponentials and a */
/* running weighted sum of values, rescaled when a larger score arrives. Each held block   */
/* is consumed in key tiles of `block` tokens (blockwise attention). Output in natural     */
/* order like oracle_attention (all rows).                                                  */
/* ------------------------------------------------------------------------------------- */
int oracle_ring(int B, int64_t T, int h, int n_kv, int d, const uint16_t* q, const uint16_t* k,
                const uint16_t* v, const int32_t* pos, int causal, double scale, int n_cp, int layout,
                int block, double* o, double* lse) {
    if (B <= 0 || T <= 0 || h <= 0 || n_kv <= 0 || d <= 0 || h % n_kv || n_cp <= 0 || T % n_cp || block <= 0)
        return 1;
    if (layout == LAYOUT_ZIGZAG && T % (2 * n_cp)) return 1;
    int64_t n = T / n_cp;
    int64_t* map = (int64_t*)malloc(sizeof(int64_t) * (size_t)T);
    if (!map) return 1;
    if (oracle_layout_map(T, n_cp, layout, map)) { free(map); return 1; }
    int g = h / n_kv;
    int64_t total = (int64_t)B * T * h; /* (b, rank r, local j, head i) */
    int err = 0;
#pragma omp parallel
    {
        double* sc = (double*)malloc(sizeof(double) * (size_t)block);
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        if (!sc || !acc) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t w = 0; w < total; ++w) {
            if (!sc || !acc) continue;
            int i = (int)(w % h);
            int64_t rj = (w / h) % T;
            int b = (int)(w / ((int64_t)h * T));
            int r = (int)(rj / n), kv = i / g;
            int64_t t = map[rj];
            const uint16_t* qrow = q + (((int64_t)b * T + t) * h + i) * d;
            double m = -INFINITY, l = 0.0;
            for (int c = 0; c < d; ++c) acc[c] = 0.0;
            for (int s = 0; s < n_cp; ++s) {
                int src = ((r - s) % n_cp + n_cp) % n_cp;    /* block held at step s */
                for (int64_t k0 = 0; k0 < n; k0 += block) {
                    int64_t kn = (n - k0 < block) ? n - k0 : block;
                    double bm = -INFINITY;
                    for (int64_t jj = 0; jj < kn; ++jj) {
                        int64_t u = map[(int64_t)src * n + k0 + jj];
                        if (!visible(pos, u, t, causal)) { sc[jj] = -INFINITY; continue; }
                        const uint16_t* krow = k + (((int64_t)b * T + u) * n_kv + kv) * d;
                        double dot = 0.0;
                        for (int c = 0; c < d; ++c) dot += bf16_value(qrow[c]) * bf16_value(krow[c]);
                        sc[jj] = scale * dot;
                        if (sc[jj] > bm) bm = sc[jj];
                    }
                    if (bm == -INFINITY) continue;                 /* nothing visible here */
                    double m_new = bm > m ? bm : m;
                    double alpha = exp(m - m_new);                 /* 0 when m = -inf */
                    l *= alpha;
                    for (int c = 0; c < d; ++c) acc[c] *= alpha;
                    for (int64_t jj = 0; jj < kn; ++jj) {
                        if (sc[jj] == -INFINITY) continue;
                        double p = exp(sc[jj] - m_new);
                        int64_t u = map[(int64_t)src * n + k0 + jj];
                        const uint16_t* vrow = v + (((int64_t)b * T + u) * n_kv + kv) * d;
                        l += p;
                        for (int c = 0; c < d; ++c) acc[c] += p * bf16_value(vrow[c]);
                    }
                    m = m_new;
                }
            }
            double* orow = o + (((int64_t)b * T + t) * h + i) * d;
            double* lrow = lse + ((int64_t)b * h + i) * T + t;
            if (l == 0.0) {
                for (int c = 0; c < d; ++c) orow[c] = 0.0;
                *lrow = -INFINITY;
            } else {
                for (int c = 0; c < d; ++c) orow[c] = acc[c] / l;
                *lrow = m + log(l);
            }
        }
        free(sc);
        free(acc);
    }
    free(map);
    return err;
}

/* ------------------------------------------------------------------------------------- */
/* Combining partial results. [CEX] "Pass them around a ring" (online softmax): a partial  */
/* over a key subset is (O_x, lse_x); over the union, lse = ln sum_x exp(lse_x) and        */
/* O = sum_x exp(lse_x - lse) O_x. An empty partial has lse = -inf and is the identity.    */
/* o_parts [S][rows][h][d], lse_parts [S][h][rows]; o [rows][h][d], lse [h][rows].          */
/* ------------------------------------------------------------------------------------- */
void oracle_merge(int S, int64_t rows, int h, int d, const double* o_parts, const double* lse_parts, double* o,
                  double* lse) {
    for (int64_t r = 0; r < rows; ++r)
        for (int i = 0; i < h; ++i) {
            double mx = -INFINITY;
            for (int s = 0; s < S; ++s) {
                double x = lse_parts[((int64_t)s * h + i) * rows + r];
                if (x > mx) mx = x;
            }
            double* orow = o + (r * h + i) * d;
            if (mx == -INFINITY) {
                for (int c = 0; c < d; ++c) orow[c] = 0.0;
                lse[(int64_t)i * rows + r] = -INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int s = 0; s < S; ++s) sum += exp(lse_parts[((int64_t)s * h + i) * rows + r] - mx);
            double L = mx + log(sum);
            lse[(int64_t)i * rows + r] = L;
            for (int c = 0; c < d; ++c) {
                double a = 0.0;
                for (int s = 0; s < S; ++s) {
                    double x = lse_parts[((int64_t)s * h + i) * rows + r];
                    if (x == -INFINITY) continue;
                    a += exp(x - L) * o_parts[(((int64_t)s * rows + r) * h + i) * d + c];
                }
                orow[c] = a;
            }
        }
}

/* ------------------------------------------------------------------------------------- */
/* Block classes and work. [CEX] "The causal mask unbalances the sequence": a block whose  */
/* keys all precede its queries is fully computed, one whose keys all follow is skipped,   */
/* and the diagonal block is partly visible ("counting a diagonal block as half").         */
/* Brute force over every (query, key) pair of the tile.                                   */
/* ------------------------------------------------------------------------------------- */
int oracle_classify(int64_t nq, const int64_t* qpos, int64_t nk, const int64_t* kpos, int causal) {
    if (!causal) return CLASS_FULL;
    int any_vis = 0, any_hidden = 0;
    for (int64_t a = 0; a < nq; ++a)
        for (int64_t c = 0; c < nk; ++c) {
            if (kpos[c] <= qpos[a]) any_vis = 1; else any_hidden = 1;
            if (any_vis && any_hidden) return CLASS_DIAG;
        }
    return any_vis ? CLASS_FULL : CLASS_SKIP;
}

/* Per (rank r, step s) tile counts for one (batch element, query head), with query tiles of
 * bq rows and key tiles of bk keys taken over each rank's local order (the last tile of a
 * block may be shorter). full/diag/skip are [n_cp][n_cp] indexed r*n_cp + s. pairs[r] is the
 * exact number of visible (query, key) pairs of rank r over the whole ring. pos: position id
 * of each natural token, or NULL for 0..T-1. Returns 0 on success. */
int oracle_plan_counts(int64_t T, int n_cp, int layout, int causal, const int32_t* pos, int bq, int bk,
                       int64_t* full, int64_t* diag, int64_t* skip, int64_t* pairs) {
    if (n_cp <= 0 || T % n_cp || bq <= 0 || bk <= 0) return 1;
    if (layout == LAYOUT_ZIGZAG && T % (2 * n_cp)) return 1;
    int64_t n = T / n_cp;
    int64_t* lpos = (int64_t*)malloc(sizeof(int64_t) * (size_t)T);   /* position of (r, j) */
    if (!lpos) return 1;
    for (int r = 0; r < n_cp; ++r)
        for (int64_t j = 0; j < n; ++j) {
            int64_t t = oracle_token_of(T, n_cp, layout, r, j);
            if (t < 0) { free(lpos); return 1; }
            lpos[(int64_t)r * n + j] = pos ? pos[t] : t;
        }
    int64_t nqt = (n + bq - 1) / bq, nkt = (n + bk - 1) / bk;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int r = 0; r < n_cp; ++r)
        for (int s = 0; s < n_cp; ++s) {
            int src = ((r - s) % n_cp + n_cp) % n_cp;
            int64_t cf = 0, cd = 0, cs = 0;
            for (int64_t qt = 0; qt < nqt; ++qt)
                for (int64_t kt = 0; kt < nkt; ++kt) {
                    int64_t q0 = qt * bq, k0 = kt * bk;
                    int64_t qn = (n - q0 < bq) ? n - q0 : bq, kn = (n - k0 < bk) ? n - k0 : bk;
                    int c = oracle_classify(qn, lpos + (int64_t)r * n + q0, kn, lpos + (int64_t)src * n + k0, causal);
                    if (c == CLASS_FULL) ++cf; else if (c == CLASS_DIAG) ++cd; else ++cs;
                }
            full[r * n_cp + s] = cf;
            diag[r * n_cp + s] = cd;
            skip[r * n_cp + s] = cs;
        }
    /* exact visible pairs per rank: every query of the rank against every key of the sequence */
#pragma omp parallel for schedule(static)
    for (int r = 0; r < n_cp; ++r) {
        int64_t cnt = 0;
        for (int64_t j = 0; j < n; ++j) {
            int64_t pq = lpos[(int64_t)r * n + j];
            for (int64_t u = 0; u < T; ++u) cnt += (!causal || lpos[u] <= pq);
        }
        pairs[r] = cnt;
    }
    free(lpos);
    return 0;
}

/* Chunk-level work of [CEX] "The causal mask unbalances the sequence", in half-block units:
 * over the rank's query chunks and all key chunks, FULL counts 2, DIAG (partly visible)
 * counts 1, SKIP 0. Chunks: contiguous = n_cp of T/n_cp; zigzag = 2n_cp of T/(2n_cp) (a rank
 * holds two); striped = one stripe per rank. Classified by brute force over token pairs
 * (positions 0..T-1). out[r] for r < n_cp. */
int oracle_half_units(int64_t T, int n_cp, int layout, int causal, int64_t* out) {
    if (n_cp <= 0 || T % n_cp) return 1;
    if (layout == LAYOUT_ZIGZAG && T % (2 * n_cp)) return 1;
    int64_t n = T / n_cp;
    int nchunks = (layout == LAYOUT_ZIGZAG) ? 2 * n_cp : n_cp;
    int64_t csize = T / nchunks;
    int64_t* cpos = (int64_t*)malloc(sizeof(int64_t) * (size_t)T);   /* tokens of chunk c */
    if (!cpos) return 1;
    for (int c = 0; c < nchunks; ++c)
        for (int64_t j = 0; j < csize; ++j)
            cpos[(int64_t)c * csize + j] = (layout == LAYOUT_STRIPED) ? j * n_cp + c : (int64_t)c * csize + j;
    int rc = 0;
    for (int r = 0; r < n_cp && !rc; ++r) {
        int mine[2], nm;
        if (layout == LAYOUT_STRIPED) { mine[0] = r; nm = 1; }
        else nm = oracle_chunk_assignment(n_cp, layout, r, mine);
        int64_t units = 0;
        for (int a = 0; a < nm; ++a)
            for (int c = 0; c < nchunks; ++c) {
                int cls = oracle_classify(csize, cpos + (int64_t)mine[a] * csize, csize, cpos + (int64_t)c * csize,
                                          causal);
                units += (cls == CLASS_FULL) ? 2 : (cls == CLASS_DIAG) ? 1 : 0;
            }
        out[r] = units;
    }
    (void)n;
    free(cpos);
    return rc;
}

/* ------------------------------------------------------------------------------------- */
/* Communication and overlap, [CEX] "What context parallelism communicates", "When the     */
/* ring hides its communication" and "Ulysses, splitting by heads instead". The displayed  */
/* equations did not survive extraction; these are the readings that reproduce the pages' */
/* printed numbers (63 MB, 1.3 ms, ~2,200 and ~20,000 tokens, break-even 1 + h/n_kv).     */
/* ------------------------------------------------------------------------------------- */

/* Bytes one rank receives in the forward pass. method 0 = ring, 1 = all-gather: each
 * receives the other n_cp-1 blocks of keys and values, 2*n*d_kv numbers of 2 bytes each.
 * method 2 = Ulysses: an all-to-all keeps 1/n_cp of Q (width d), K, V (width d_kv) and the
 * output (width d) and sends the rest. d is the model width h*d_k, d_kv = n_kv*d_k. */
double oracle_cp_comm_bytes(double T, double d, double d_kv, double n_cp, int method) {
    double n = T / n_cp;
    if (method == 0 || method == 1) return 4.0 * n * d_kv * (n_cp - 1.0);
    if (method == 2) return 4.0 * n * (d + d_kv) * (n_cp - 1.0) / n_cp;
    return -1.0;
}

/* Group size above which Ulysses moves fewer bytes than the ring: ring bytes equal Ulysses
 * bytes when n_cp * d_kv = d + d_kv, i.e. n_cp = 1 + h/n_kv. */
double oracle_ulysses_breakeven(double h, double n_kv) { return 1.0 + h / n_kv; }

/* Smallest tokens per GPU for which a ring step's compute (4 n^2 d FLOPs for a fully
 * visible block) covers sending the next block (4 n d_kv bytes): n >= (F/B) * (n_kv/h). */
double oracle_overlap_min_tokens(double flops_per_s, double bytes_per_s, double h, double n_kv) {
    return flops_per_s / bytes_per_s * (n_kv / h);
}

/* Bytes of keys and values each rank receives around the ring in one forward pass: every
 * foreign block, skipped or not, for B sequences and all n_kv heads of width d_k. */
int64_t oracle_kv_bytes_recv(int B, int64_t n, int n_kv, int d_k, int n_cp) {
    return (int64_t)(n_cp - 1) * 2 /* K and V */ * (int64_t)B * n * n_kv * d_k * 2 /* bytes */;
}

/* ------------------------------------------------------------------------------------- */
/* Gradients. [CEX] "Splitting the sequence, and the one layer that objects" and "What    */
/* context parallelism communicates": the backward pass of the ring computes the same     */
/* gradients as plain attention; each rank keeps the gradient of its queries, and the key  */
/* and value gradients travel with the blocks back to their owners. The pages print no     */
/* gradient formulas; these are the derivatives of the forward definition above, for the   */
/* loss L = sum_{b,t,i} <O[b,t,i,:], dO[b,t,i,:]>:                                          */
/*   P_tu  = exp(s_tu - lse_t) for visible u, else 0                                        */
/*   dP_tu = <dO_t, v_u>,  D_t = sum_u P_tu dP_tu = <dO_t, O_t>                              */
/*   dS_tu = P_tu (dP_tu - D_t)                                                              */
/*   dQ_t  = scale sum_u dS_tu k_u                                                           */
/*   dK_u  = scale sum_{i in group} sum_t dS_tu q_t,  dV_u = sum_{i in group} sum_t P_tu dO_t */
/* (the KV head of a group receives the sum over the group's query heads).                 */
/* ------------------------------------------------------------------------------------- */

/* lse and D = <dO_t, O_t> of one (b, t, head i) row from the definition (two passes). */
static void row_stats(int64_t T, int h, int n_kv, int d, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      const uint16_t* dout, const int32_t* pos, const int32_t* doc, int causal, double scale, int b,
                      int64_t t, int i, double* acc, double* lse_out, double* d_out) {
    int kv = i / (h / n_kv);
    const uint16_t* qrow = q + (((int64_t)b * T + t) * h + i) * d;
    double mx = -INFINITY;
    for (int64_t u = 0; u < T; ++u) {
        if (!visible_doc(pos, doc, u, t, causal)) continue;
        const uint16_t* krow = k + (((int64_t)b * T + u) * n_kv + kv) * d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += bf16_value(qrow[c]) * bf16_value(krow[c]);
        if (scale * dot > mx) mx = scale * dot;
    }
    if (mx == -INFINITY) { *lse_out = -INFINITY; *d_out = 0.0; return; }
    double sum = 0.0;
    for (int c = 0; c < d; ++c) acc[c] = 0.0;
    for (int64_t u = 0; u < T; ++u) {
        if (!visible_doc(pos, doc, u, t, causal)) continue;
        const uint16_t* krow = k + (((int64_t)b * T + u) * n_kv + kv) * d;
        const uint16_t* vrow = v + (((int64_t)b * T + u) * n_kv + kv) * d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += bf16_value(qrow[c]) * bf16_value(krow[c]);
        double e = exp(scale * dot - mx);
        sum += e;
        for (int c = 0; c < d; ++c) acc[c] += e * bf16_value(vrow[c]);
    }
    const uint16_t* grow = dout + (((int64_t)b * T + t) * h + i) * d;
    double dd = 0.0;
    for (int c = 0; c < d; ++c) dd += bf16_value(grow[c]) * (acc[c] / sum);
    *lse_out = mx + log(sum);
    *d_out = dd;
}

/* The contribution of the pair (query t of head i, key u): P_tu and dS_tu. */
static void pair_terms(int64_t T, int h, int n_kv, int d, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const uint16_t* dout, double scale, int b, int64_t t, int i, int64_t u, double lse_t,
                       double d_t, double* p_out, double* ds_out) {
    int kv = i / (h / n_kv);
    const uint16_t* qrow = q + (((int64_t)b * T + t) * h + i) * d;
    const uint16_t* grow = dout + (((int64_t)b * T + t) * h + i) * d;
    const uint16_t* krow = k + (((int64_t)b * T + u) * n_kv + kv) * d;
    const uint16_t* vrow = v + (((int64_t)b * T + u) * n_kv + kv) * d;
    double dot = 0.0, dp = 0.0;
    for (int c = 0; c < d; ++c) {
        dot += bf16_value(qrow[c]) * bf16_value(krow[c]);
        dp += bf16_value(grow[c]) * bf16_value(vrow[c]);
    }
    double p = exp(scale * dot - lse_t);
    *p_out = p;
    *ds_out = p * (dp - d_t);
}

/* q [B,T,h,d], k/v [B,T,n_kv,d], dout [B,T,h,d] bf16 bits, natural order.
 * dq [B,n_rows,h,d] for the query rows `rows` (NULL: all T, n_rows = T; dq may be NULL);
 * dk, dv [B,n_keys,n_kv,d] for the keys `keys` (NULL: all T, n_keys = T; dk/dv may be NULL).
 * fp64 outputs. Returns 0 on success. */
static int backward_impl(int B, int64_t T, int h, int n_kv, int d, const uint16_t* q, const uint16_t* k,
                         const uint16_t* v, const uint16_t* dout, const int32_t* pos, const int32_t* doc, int causal,
                         double scale, int64_t n_rows, const int64_t* rows, int64_t n_keys, const int64_t* keys,
                         double* dq, double* dk, double* dv) {
    if (B <= 0 || T <= 0 || h <= 0 || n_kv <= 0 || d <= 0 || h % n_kv) return 1;
    if (!rows) n_rows = T;
    if (!keys) n_keys = T;
    int g = h / n_kv;
    int err = 0;
    /* dQ: every row is self-contained (its own lse and D, then one more pass over its keys) */
    if (dq) {
        int64_t total = (int64_t)B * n_rows * h;
#pragma omp parallel
        {
            double* acc = (double*)malloc(sizeof(double) * (size_t)d);
            if (!acc) {
#pragma omp atomic write
                err = 1;
            }
#pragma omp for schedule(dynamic, 4)
            for (int64_t w = 0; w < total; ++w) {
                if (!acc) continue;
                int i = (int)(w % h);
                int64_t ri = (w / h) % n_rows;
                int b = (int)(w / ((int64_t)h * n_rows));
                int64_t t = rows ? rows[ri] : ri;
                int kv = i / g;
                double lse_t, d_t;
                row_stats(T, h, n_kv, d, q, k, v, dout, pos, doc, causal, scale, b, t, i, acc, &lse_t, &d_t);
                double* out = dq + (((int64_t)b * n_rows + ri) * h + i) * d;
                for (int c = 0; c < d; ++c) out[c] = 0.0;
                if (lse_t == -INFINITY) continue;
                for (int64_t u = 0; u < T; ++u) {
                    if (!visible_doc(pos, doc, u, t, causal)) continue;
                    double p, ds;
                    pair_terms(T, h, n_kv, d, q, k, v, dout, scale, b, t, i, u, lse_t, d_t, &p, &ds);
                    const uint16_t* krow = k + (((int64_t)b * T + u) * n_kv + kv) * d;
                    for (int c = 0; c < d; ++c) out[c] += scale * ds * bf16_value(krow[c]);
                }
            }
            free(acc);
        }
        if (err) return err;
    }
    if (!dk && !dv) return 0;
    /* dK, dV: first lse and D of every row that sees one of the keys, then per key the sum
     * over those rows (and the query heads of its group). */
    double* lse = (double*)malloc(sizeof(double) * (size_t)B * h * T);
    double* dd = (double*)malloc(sizeof(double) * (size_t)B * h * T);
    unsigned char* need = (unsigned char*)calloc((size_t)B * T, 1);
    if (!lse || !dd || !need) { free(lse); free(dd); free(need); return 1; }
    for (int64_t t = 0; t < T; ++t)
        for (int64_t ki = 0; ki < n_keys; ++ki) {
            int64_t u = keys ? keys[ki] : ki;
            if (visible_doc(pos, doc, u, t, causal)) { for (int b = 0; b < B; ++b) need[(int64_t)b * T + t] = 1; break; }
        }
    int64_t total = (int64_t)B * T * h;
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        if (!acc) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t w = 0; w < total; ++w) {
            if (!acc) continue;
            int i = (int)(w % h);
            int64_t t = (w / h) % T;
            int b = (int)(w / ((int64_t)h * T));
            if (!need[(int64_t)b * T + t]) continue;
            row_stats(T, h, n_kv, d, q, k, v, dout, pos, doc, causal, scale, b, t, i, acc,
                      &lse[((int64_t)b * h + i) * T + t], &dd[((int64_t)b * h + i) * T + t]);
        }
        free(acc);
    }
    if (err) { free(lse); free(dd); free(need); return err; }
    int64_t kt = (int64_t)B * n_keys * n_kv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < kt; ++w) {
        int kvh = (int)(w % n_kv);
        int64_t ki = (w / n_kv) % n_keys;
        int b = (int)(w / ((int64_t)n_kv * n_keys));
        int64_t u = keys ? keys[ki] : ki;
        double* gk = dk ? dk + (((int64_t)b * n_keys + ki) * n_kv + kvh) * d : NULL;
        double* gv = dv ? dv + (((int64_t)b * n_keys + ki) * n_kv + kvh) * d : NULL;
        for (int c = 0; c < d; ++c) { if (gk) gk[c] = 0.0; if (gv) gv[c] = 0.0; }
        for (int i = kvh * g; i < (kvh + 1) * g; ++i)
            for (int64_t t = 0; t < T; ++t) {
                if (!visible_doc(pos, doc, u, t, causal)) continue;
                double lse_t = lse[((int64_t)b * h + i) * T + t];
                if (lse_t == -INFINITY) continue;
                double p, ds;
                pair_terms(T, h, n_kv, d, q, k, v, dout, scale, b, t, i, u, lse_t, dd[((int64_t)b * h + i) * T + t], &p, &ds);
                const uint16_t* qrow = q + (((int64_t)b * T + t) * h + i) * d;
                const uint16_t* grow = dout + (((int64_t)b * T + t) * h + i) * d;
                for (int c = 0; c < d; ++c) {
                    if (gk) gk[c] += scale * ds * bf16_value(qrow[c]);
                    if (gv) gv[c] += p * bf16_value(grow[c]);
                }
            }
    }
    free(lse);
    free(dd);
    free(need);
    return 0;
}

int oracle_attention_backward(int B, int64_t T, int h, int n_kv, int d, const uint16_t* q, const uint16_t* k,
                              const uint16_t* v, const uint16_t* dout, const int32_t* pos, int causal, double scale,
                              int64_t n_rows, const int64_t* rows, int64_t n_keys, const int64_t* keys, double* dq,
                              double* dk, double* dv) {
    return backward_impl(B, T, h, n_kv, d, q, k, v, dout, pos, NULL, causal, scale, n_rows, rows, n_keys, keys, dq,
                         dk, dv);
}

/* The gradients under a document mask (doc [T] document id per natural token): the derivatives
 * of oracle_attention_docs. */
int oracle_attention_backward_docs(int B, int64_t T, int h, int n_kv, int d, const uint16_t* q, const uint16_t* k,
                                   const uint16_t* v, const uint16_t* dout, const int32_t* pos, const int32_t* doc,
                                   int causal, double scale, int64_t n_rows, const int64_t* rows, int64_t n_keys,
                                   const int64_t* keys, double* dq, double* dk, double* dv) {
    return backward_impl(B, T, h, n_kv, d, q, k, v, dout, pos, doc, causal, scale, n_rows, rows, n_keys, keys, dq, dk,
                         dv);
}

/* The ring backward, simulated literally. [CEX] "What context parallelism communicates":   */
/* the key and value gradients travel back to their owners "as a second circulating block  */
/* in the ring". At step s rank r holds the key/value block of src = (r - s) mod n_cp and   */
/* that block's gradient accumulator; it adds the contribution of its own queries, tile by  */
/* tile (`block` keys), keeps its query gradient, and passes both blocks right. After n_cp  */
/* steps the accumulator has visited every rank and one more hop returns it to src. lse and */
/* D of every row come from the forward definition. Outputs in natural order, all rows.     */
int oracle_ring_backward(int B, int64_t T, int h, int n_kv, int d, const uint16_t* q, const uint16_t* k,
                         const uint16_t* v, const uint16_t* dout, const int32_t* pos, int causal, double scale,
                         int n_cp, int layout, int block, double* dq, double* dk, double* dv) {
    if (B <= 0 || T <= 0 || h <= 0 || n_kv <= 0 || d <= 0 || h % n_kv || n_cp <= 0 || T % n_cp || block <= 0)
        return 1;
    if (layout == LAYOUT_ZIGZAG && T % (2 * n_cp)) return 1;
    int64_t n = T / n_cp;
    int g = h / n_kv;
    int64_t* map = (int64_t*)malloc(sizeof(int64_t) * (size_t)T);
    double* lse = (double*)malloc(sizeof(double) * (size_t)B * h * T);
    double* dd = (double*)malloc(sizeof(double) * (size_t)B * h * T);
    if (!map || !lse || !dd || oracle_layout_map(T, n_cp, layout, map)) { free(map); free(lse); free(dd); return 1; }
    int err = 0;
    int64_t total = (int64_t)B * T * h;
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        if (!acc) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t w = 0; w < total; ++w) {
            if (!acc) continue;
            int i = (int)(w % h);
            int64_t t = (w / h) % T;
            int b = (int)(w / ((int64_t)h * T));
            row_stats(T, h, n_kv, d, q, k, v, dout, pos, NULL, causal, scale, b, t, i, acc,
                      &lse[((int64_t)b * h + i) * T + t], &dd[((int64_t)b * h + i) * T + t]);
        }
        free(acc);
    }
    if (err) { free(map); free(lse); free(dd); return err; }
    memset(dq, 0, sizeof(double) * (size_t)B * T * h * d);
    /* one independent ring per (batch element, KV head): its query heads and its KV blocks */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < (int64_t)B * n_kv; ++w) {
        int kvh = (int)(w % n_kv), b = (int)(w / n_kv);
        double* acc_k = (double*)calloc((size_t)T * d, sizeof(double));   /* [block src][n][d] */
        double* acc_v = (double*)calloc((size_t)T * d, sizeof(double));
        if (!acc_k || !acc_v) {
            free(acc_k); free(acc_v);
#pragma omp atomic write
            err = 1;
            continue;
        }
        for (int s = 0; s < n_cp; ++s)
            for (int r = 0; r < n_cp; ++r) {
                int src = ((r - s) % n_cp + n_cp) % n_cp;     /* block rank r holds at step s */
                for (int64_t j = 0; j < n; ++j) {
                    int64_t t = map[(int64_t)r * n + j];
                    for (int i = kvh * g; i < (kvh + 1) * g; ++i) {
                        double lse_t = lse[((int64_t)b * h + i) * T + t], d_t = dd[((int64_t)b * h + i) * T + t];
                        if (lse_t == -INFINITY) continue;
                        const uint16_t* qrow = q + (((int64_t)b * T + t) * h + i) * d;
                        const uint16_t* grow = dout + (((int64_t)b * T + t) * h + i) * d;
                        double* dqrow = dq + (((int64_t)b * T + t) * h + i) * d;
                        for (int64_t k0 = 0; k0 < n; k0 += block) {
                            int64_t kn = (n - k0 < block) ? n - k0 : block;
                            for (int64_t jj = 0; jj < kn; ++jj) {
                                int64_t u = map[(int64_t)src * n + k0 + jj];
                                if (!visible(pos, u, t, causal)) continue;
                                double p, ds;
                                pair_terms(T, h, n_kv, d, q, k, v, dout, scale, b, t, i, u, lse_t, d_t, &p, &ds);
                                const uint16_t* krow = k + (((int64_t)b * T + u) * n_kv + kvh) * d;
                                double* ak = acc_k + ((int64_t)src * n + k0 + jj) * d;
                                double* av = acc_v + ((int64_t)src * n + k0 + jj) * d;
                                for (int c = 0; c < d; ++c) {
                                    dqrow[c] += scale * ds * bf16_value(krow[c]);
                                    ak[c] += scale * ds * bf16_value(qrow[c]);
                                    av[c] += p * bf16_value(grow[c]);
                                }
                            }
                        }
                    }
                }
            }
        /* the accumulator of block src has made n_cp - 1 hops; the last returns it to src */
        for (int src = 0; src < n_cp; ++src)
            for (int64_t j = 0; j < n; ++j) {
                int64_t u = map[(int64_t)src * n + j];
                double* gk = dk + (((int64_t)b * T + u) * n_kv + kvh) * d;
                double* gv = dv + (((int64_t)b * T + u) * n_kv + kvh) * d;
                for (int c = 0; c < d; ++c) {
                    gk[c] = acc_k[((int64_t)src * n + j) * d + c];
                    gv[c] = acc_v[((int64_t)src * n + j) * d + c];
                }
            }
        free(acc_k);
        free(acc_v);
    }
    free(map);
    free(lse);
    free(dd);
    return err;
}

/* Bytes one rank receives in the backward ring: the key/value blocks of the n_cp - 1 other
 * ranks (as in the forward) plus the circulating key/value gradient blocks, which arrive
 * n_cp times (the last hop brings a rank its own block back). Gradient elements of
 * grad_bytes each. [CEX] "What context parallelism communicates": the backward roughly
 * doubles the traffic. */
int64_t oracle_bwd_bytes_recv(int B, int64_t n, int n_kv, int d_k, int n_cp, int grad_bytes) {
    int64_t blk = (int64_t)B * n * n_kv * d_k;
    return (int64_t)(n_cp - 1) * 2 * blk * 2 + (int64_t)n_cp * 2 * blk * grad_bytes;
}
