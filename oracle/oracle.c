/*
 * oracle.c -- plain fp64 CPU reference for tree verification through a gated
 * linear recurrence.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the benchmark's CPU-baseline leg call it; the library never does.  It shares
 * no code, header or table with the CUDA path.
 *
 * What it computes (Bole summary page, "Core techniques" §1 and §2; naive
 * baseline of "Comparison with existing approaches"): the naive tree walk that
 * keeps one full state matrix per draft node.
 *
 *   recurrence  h_{t+1} = S_t h_t + u_t   (§1), specialised to
 *               S_i = diag(exp g_i),  u_i = k_i v_i^T,  output o_i = H_i^T q_i
 *   tree        H_i = diag(exp g_i) H_{parent(i)} + k_i v_i^T,  H_{-1} = H0
 *
 * Every node state H_i (dk x dv) is materialised in index order (parents
 * precede children), exactly the "one state matrix per node, serial walk"
 * baseline whose memory the method removes (§2).
 *
 * Greedy acceptance (LLM Primer VI ch. 9, §9.1): the longest draft prefix that
 * matches the target is accepted; at the first mismatch the target's own token
 * is kept.  On a tree: start at the context with t = root_argmax; repeatedly
 * take the lowest-index child whose draft token equals t, set t to the target's
 * argmax after that child; stop when no child matches.  bonus = t.
 *
 * Commit (§2, "only the accepted path's state is restored"): replay the
 * recurrence from H0 along the accepted path; H_new = state of the last
 * accepted node (H0 when nothing is accepted).
 *
 * All arithmetic is double precision; inputs arrive as float (bf16 values are
 * exactly representable) and are widened element by element.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_TREE 1
#define ORC_ERR_NOMEM 2
#define ORC_ERR_ARG 3

/* parent[i] must be -1 or an earlier node. */
int orc_check_tree(int n, const int32_t *parent) {
    for (int i = 0; i < n; ++i)
        if (parent[i] < -1 || parent[i] >= i) return ORC_ERR_TREE;
    return ORC_OK;
}

/*
 * One (request, head): naive serial tree walk with per-node states.
 *   g:   n values (scalar decay) or n*dk (diagonal decay), row i = node i
 *   q,k: n*dk; v: n*dv; H0: dk*dv (row r = key channel, column c = value channel)
 *   out: n*dv
 *   states: n*dk*dv doubles of caller scratch, or NULL to allocate here.
 */
int orc_verify_unit(int n, const int32_t *parent, int dk, int dv, int diag,
                    const double *g, const double *q, const double *k,
                    const double *v, const double *H0, double *out, double *states) {
    if (orc_check_tree(n, parent) != ORC_OK) return ORC_ERR_TREE;
    int own = 0;
    if (!states && n > 0) {
        states = (double *)malloc(sizeof(double) * (size_t)n * dk * dv);
        if (!states) return ORC_ERR_NOMEM;
        own = 1;
    }
    for (int i = 0; i < n; ++i) {
        const double *prev = parent[i] < 0 ? H0 : states + (size_t)parent[i] * dk * dv;
        double *S = states + (size_t)i * dk * dv;
        for (int r = 0; r < dk; ++r) {
            double a = exp(diag ? g[(size_t)i * dk + r] : g[i]);
            for (int c = 0; c < dv; ++c)
                S[(size_t)r * dv + c] = a * prev[(size_t)r * dv + c]
                                      + k[(size_t)i * dk + r] * v[(size_t)i * dv + c];
        }
        for (int c = 0; c < dv; ++c) {
            double acc = 0.0;
            for (int r = 0; r < dk; ++r) acc += S[(size_t)r * dv + c] * q[(size_t)i * dk + r];
            out[(size_t)i * dv + c] = acc;
        }
    }
    if (own) free(states);
    return ORC_OK;
}

/* Greedy acceptance walk over one request's tree. path gets max_depth entries, -1 padded. */
int orc_accept(int n, const int32_t *parent, const int32_t *draft, const int32_t *target,
               int32_t root_tok, int max_depth, int32_t *len, int32_t *path, int32_t *bonus) {
    if (orc_check_tree(n, parent) != ORC_OK) return ORC_ERR_TREE;
    int cur = -1, L = 0;
    int32_t t = root_tok;
    for (;;) {
        int c = -1;
        for (int i = 0; i < n; ++i)
            if (parent[i] == cur && draft[i] == t) { c = i; break; }
        if (c < 0) break;
        if (L >= max_depth) return ORC_ERR_TREE;
        path[L++] = c;
        t = target[c];
        cur = c;
    }
    for (int m = L; m < max_depth; ++m) path[m] = -1;
    *len = L;
    *bonus = t;
    return ORC_OK;
}

/* Replay the recurrence from H0 along path[0..L) of one (request, head). */
int orc_commit_unit(int L, const int32_t *path, int dk, int dv, int diag, const double *g,
                    const double *k, const double *v, const double *H0, double *Hnew) {
    memcpy(Hnew, H0, sizeof(double) * (size_t)dk * dv);
    for (int m = 0; m < L; ++m) {
        int i = path[m];
        for (int r = 0; r < dk; ++r) {
            double a = exp(diag ? g[(size_t)i * dk + r] : g[i]);
            for (int c = 0; c < dv; ++c)
                Hnew[(size_t)r * dv + c] = a * Hnew[(size_t)r * dv + c]
                                         + k[(size_t)i * dk + r] * v[(size_t)i * dv + c];
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Batch drivers over packed inputs (layouts of the library's interface):
 *   q,k [T,H,dk], v [T,H,dv], g [T,H] or [T,H,dk], H0 [B,H,dk,dv] (float),
 *   node_offsets [B+1], parent [T] local to the request.
 * They gather one (request, head) unit into doubles and call the unit routine.
 * `units` lists u = b*H + h; outputs are written compactly in that order:
 *   verify: rows of sum_u N_b(u) x dv;  commit: n_units x dk x dv.
 * ---------------------------------------------------------------------- */

static void gather(double *dst, const float *src, int n, int off, int H, int h, int w) {
    for (int i = 0; i < n; ++i)
        for (int c = 0; c < w; ++c)
            dst[(size_t)i * w + c] = (double)src[((size_t)(off + i) * H + h) * w + c];
}

int orc_verify_batch(int B, int H, int dk, int dv, int diag, const int32_t *node_offsets,
                     const int32_t *parent, const float *g, const float *q, const float *k,
                     const float *v, const float *H0, int n_units, const int32_t *units,
                     double *out) {
    size_t row = 0;
    for (int s = 0; s < n_units; ++s) {
        int u = units[s], b = u / H, h = u % H;
        if (b < 0 || b >= B) return ORC_ERR_ARG;
        int off = node_offsets[b], n = node_offsets[b + 1] - off;
        int gw = diag ? dk : 1;
        double *gg = malloc(sizeof(double) * ((size_t)n * gw + 1));
        double *qq = malloc(sizeof(double) * ((size_t)n * dk + 1));
        double *kk = malloc(sizeof(double) * ((size_t)n * dk + 1));
        double *vv = malloc(sizeof(double) * ((size_t)n * dv + 1));
        double *hh = malloc(sizeof(double) * (size_t)dk * dv);
        if (!gg || !qq || !kk || !vv || !hh) return ORC_ERR_NOMEM;
        gather(gg, g, n, off, H, h, gw);
        gather(qq, q, n, off, H, h, dk);
        gather(kk, k, n, off, H, h, dk);
        gather(vv, v, n, off, H, h, dv);
        for (size_t e = 0; e < (size_t)dk * dv; ++e) hh[e] = (double)H0[(size_t)u * dk * dv + e];
        int rc = orc_verify_unit(n, parent + off, dk, dv, diag, gg, qq, kk, vv, hh,
                                 out + row * dv, NULL);
        free(gg); free(qq); free(kk); free(vv); free(hh);
        if (rc) return rc;
        row += (size_t)n;
    }
    return ORC_OK;
}

int orc_accept_batch(int B, const int32_t *node_offsets, const int32_t *parent,
                     const int32_t *draft, const int32_t *target, const int32_t *root_argmax,
                     int max_depth, int32_t *len, int32_t *path, int32_t *bonus) {
    for (int b = 0; b < B; ++b) {
        int off = node_offsets[b], n = node_offsets[b + 1] - off;
        int rc = orc_accept(n, parent + off, draft + off, target + off, root_argmax[b], max_depth,
                            len + b, path + (size_t)b * max_depth, bonus + b);
        if (rc) return rc;
    }
    return ORC_OK;
}

int orc_commit_batch(int B, int H, int dk, int dv, int diag, const int32_t *node_offsets,
                     const float *g, const float *k, const float *v, const float *H0,
                     const int32_t *len, const int32_t *path, int max_depth, int n_units,
                     const int32_t *units, double *Hnew) {
    for (int s = 0; s < n_units; ++s) {
        int u = units[s], b = u / H, h = u % H;
        if (b < 0 || b >= B) return ORC_ERR_ARG;
        int off = node_offsets[b], n = node_offsets[b + 1] - off, L = len[b];
        if (L < 0 || L > max_depth) return ORC_ERR_ARG;
        int gw = diag ? dk : 1;
        double *gg = malloc(sizeof(double) * ((size_t)n * gw + 1));
        double *kk = malloc(sizeof(double) * ((size_t)n * dk + 1));
        double *vv = malloc(sizeof(double) * ((size_t)n * dv + 1));
        double *hh = malloc(sizeof(double) * (size_t)dk * dv);
        if (!gg || !kk || !vv || !hh) return ORC_ERR_NOMEM;
        gather(gg, g, n, off, H, h, gw);
        gather(kk, k, n, off, H, h, dk);
        gather(vv, v, n, off, H, h, dv);
        for (size_t e = 0; e < (size_t)dk * dv; ++e) hh[e] = (double)H0[(size_t)u * dk * dv + e];
        for (int m = 0; m < L; ++m) {
            int p = path[(size_t)b * max_depth + m];
            if (p < 0 || p >= n) { free(gg); free(kk); free(vv); free(hh); return ORC_ERR_ARG; }
        }
        int rc = orc_commit_unit(L, path + (size_t)b * max_depth, dk, dv, diag, gg, kk, vv, hh,
                                 Hnew + (size_t)s * dk * dv);
        free(gg); free(kk); free(vv); free(hh);
        if (rc) return rc;
    }
    return ORC_OK;
}
