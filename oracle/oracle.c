/*
 * oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the batched
 * speculative-sampling verify step.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Every function below is the plain
 * definition of what the pages state, computed in double precision, one row at
 * a time, with no blocking, fusion or reordering beyond what the definition
 * states.  A library sort (qsort) serves as the ranking step.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11, "Parallel random numbers: as easy as */
/* 1, 2, 3").  Ten rounds of the 4x32 Philox S-box; between rounds the key   */
/* advances by the Weyl increments.                                         */
/* ------------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

double orc_u24(uint32_t w)
{
    return (double)(w >> 8) * (1.0 / 16777216.0);
}

void orc_philox_batch(uint64_t seed, const uint32_t* ctrs, int64_t n, uint32_t* out)
{
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    for (int64_t i = 0; i < n; ++i) orc_philox4x32_10(ctrs + 4 * i, key, out + 4 * i);
}

/* The verify step's uniforms: key = seed, counter = ((j << 2) | tag, b,
 * round_lo, round_hi).  Tag 0: word 0 is the accept uniform of slot j, word 1
 * the sampling uniform of slot j (residual at a rejection, or the bonus when
 * j = K_b).  Tag 1: word 0 draws the drafted token of slot j. */
static void verify_uniforms(uint64_t seed, uint64_t round, int32_t b, int32_t j,
                            uint32_t tag, double* u0, double* u1)
{
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {((uint32_t)j << 2) | tag, (uint32_t)b, (uint32_t)round,
                       (uint32_t)(round >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    if (u0) *u0 = orc_u24(w[0]);
    if (u1) *u1 = orc_u24(w[1]);
}

/* ------------------------------------------------------------------------ */
/* Element access: bf16 is widened to fp32 exactly (bits << 16), then to     */
/* double; fp32 is widened to double.                                       */
/* ------------------------------------------------------------------------ */
static double widen(const void* base, int32_t dtype, int64_t idx)
{
    if (dtype == ORC_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[idx];
}

static void load_row(const void* base, int32_t dtype, int64_t row, int32_t V, double* dst)
{
    for (int32_t v = 0; v < V; ++v) dst[v] = widen(base, dtype, row * (int64_t)V + v);
}

/* ------------------------------------------------------------------------ */
/* Sampling knobs and softmax of one row.                                   */
/* NOTE-159 ("Key results", "Recommendations" R3): temperature, top-k and    */
/* nucleus are applied to the probabilities before the rejection step.  The  */
/* order (temperature, top-k, top-p), the tie rule (lower id first) and the  */
/* strict prefix rule for the nucleus are this project's readings.          */
/* ------------------------------------------------------------------------ */
typedef struct {
    double l;
    int32_t v;
} rank_item;

static int rank_cmp(const void* a, const void* b)
{
    const rank_item* x = (const rank_item*)a;
    const rank_item* y = (const rank_item*)b;
    if (x->l > y->l) return -1;
    if (x->l < y->l) return 1;
    return (x->v < y->v) ? -1 : (x->v > y->v);
}

int orc_row_dist(const double* l, int32_t V, double T, int32_t top_k, double top_p,
                 double* P, orc_row_info* info)
{
    orc_row_info loc;
    if (!info) info = &loc;
    info->M = -INFINITY;
    info->S = 0.0;
    info->topp_margin = INFINITY;
    info->n_kept = 0;
    info->nonfinite = 0;

    int any_finite = 0;
    for (int32_t v = 0; v < V; ++v) {
        if (isnan(l[v]) || l[v] == INFINITY) info->nonfinite = 1;
        if (isfinite(l[v])) any_finite = 1;
    }
    if (!any_finite) info->nonfinite = 1;
    if (info->nonfinite) return -1;

    unsigned char* keep = (unsigned char*)malloc((size_t)V);
    double* e = (double*)malloc(sizeof(double) * (size_t)V);
    memset(keep, 1, (size_t)V);

    const int topk_on = (top_k > 0 && top_k < V);
    const int topp_on = (top_p < 1.0);
    rank_item* order = NULL;
    if (topk_on || topp_on) {
        order = (rank_item*)malloc(sizeof(rank_item) * (size_t)V);
        for (int32_t v = 0; v < V; ++v) {
            order[v].l = l[v];
            order[v].v = v;
        }
        qsort(order, (size_t)V, sizeof(rank_item), rank_cmp);
    }

    /* top-k: the first k tokens in rank order (l descending, id ascending) */
    if (topk_on) {
        memset(keep, 0, (size_t)V);
        for (int32_t r = 0; r < top_k; ++r) keep[order[r].v] = 1;
    }

    /* softmax of z = l / T over the kept set */
    double M = -INFINITY;
    for (int32_t v = 0; v < V; ++v)
        if (keep[v]) {
            double z = l[v] / T;
            if (z > M) M = z;
        }
    double S = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        e[v] = keep[v] ? exp(l[v] / T - M) : 0.0;
        S += e[v];
    }

    /* top-p: walk the kept tokens in rank order; the token at a rank is kept
     * iff the mass strictly before it is below top_p. */
    if (topp_on) {
        double prefix = 0.0;
        double last_kept = INFINITY, first_dropped = INFINITY;
        int dropped_any = 0;
        for (int32_t r = 0; r < V; ++r) {
            int32_t v = order[r].v;
            if (!keep[v]) continue;
            if (prefix < top_p) {
                /* a rank with nothing before it (prefix exactly 0) is kept by
                 * any top_p > 0: no rounding reaches that decision */
                if (prefix > 0.0) last_kept = top_p - prefix;
                prefix += e[v] / S;
            } else {
                if (!dropped_any) first_dropped = prefix - top_p;
                dropped_any = 1;
                keep[v] = 0;
                e[v] = 0.0;
            }
        }
        info->topp_margin = last_kept < first_dropped ? last_kept : first_dropped;
        S = 0.0;
        for (int32_t v = 0; v < V; ++v) S += e[v];
    }

    int32_t n_kept = 0;
    for (int32_t v = 0; v < V; ++v) {
        P[v] = keep[v] ? e[v] / S : 0.0;
        n_kept += keep[v];
    }
    info->M = M;
    info->S = S;
    info->n_kept = n_kept;

    free(order);
    free(e);
    free(keep);
    return 0;
}

int orc_row_probs(const void* row, int32_t dtype, int32_t V, double T, int32_t top_k,
                  double top_p, double* P, orc_row_info* info)
{
    double* l = (double*)malloc(sizeof(double) * (size_t)V);
    load_row(row, dtype, 0, V, l);
    int rc = orc_row_dist(l, V, T, top_k, top_p, P, info);
    free(l);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Residual distribution: max(0, p_target - p_draft), normalised by its sum  */
/* at sampling time ("The algorithm"; "The heart of it ... (2.3)").         */
/* ------------------------------------------------------------------------ */
double orc_residual(const double* Pt, const double* Pd, int32_t V, double* R)
{
    double Z = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        double d = Pt[v] - Pd[v];
        R[v] = d > 0.0 ? d : 0.0;
        Z += R[v];
    }
    return Z;
}

/* ------------------------------------------------------------------------ */
/* Inverse-CDF draw in ascending token order.                               */
/* ------------------------------------------------------------------------ */
static int32_t cdf_pick(const double* R, int32_t V, double t, double* c_before, double* c_at)
{
    double C = 0.0, prev = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        prev = C;
        C += R[v];
        if (C > t) {
            if (c_before) *c_before = prev;
            if (c_at) *c_at = C;
            return v;
        }
    }
    /* rounding left no v with C(v) > t: the largest token with mass */
    for (int32_t v = V - 1; v >= 0; --v)
        if (R[v] > 0.0) {
            if (c_before) *c_before = C - R[v];
            if (c_at) *c_at = C;
            return v;
        }
    return -1;
}

int32_t orc_inverse_cdf(const double* R, int32_t V, double u, double delta, double* Z_out,
                        double* margin, int32_t* v_lo, int32_t* v_hi)
{
    double Z = 0.0;
    for (int32_t v = 0; v < V; ++v) Z += R[v];
    if (Z_out) *Z_out = Z;
    if (!(Z > 0.0)) {
        if (margin) *margin = 0.0;
        if (v_lo) *v_lo = -1;
        if (v_hi) *v_hi = -1;
        return -1;
    }
    double t = u * Z;
    double cb = 0.0, ca = 0.0;
    int32_t tok = cdf_pick(R, V, t, &cb, &ca);
    if (margin) {
        double m0 = (t - cb) / Z, m1 = (ca - t) / Z;
        *margin = m0 < m1 ? m0 : m1;
    }
    if (v_lo) {
        double tl = t - delta * Z;
        *v_lo = cdf_pick(R, V, tl < 0.0 ? 0.0 : tl, NULL, NULL);
    }
    if (v_hi) *v_hi = cdf_pick(R, V, t + delta * Z, NULL, NULL);
    return tok;
}

/* ------------------------------------------------------------------------ */
/* The verify step for a batch of sequences.                                */
/* Walk the drafted tokens left to right; accept x_j iff u < p_t(x)/p_d(x)   */
/* (the listings in "57 Speculative Decoding" and "Speculative Decoding from */
/* Scratch" compare a uniform with min(1, p/q) strictly); stop at the first  */
/* rejection and resample it from norm(max(0, p_t - p_d)); when every draft  */
/* passes, sample one more token from the target at position K_b + 1        */
/* ("The big picture ... (2.1)", step 3; "How It Works", step 4).           */
/* ------------------------------------------------------------------------ */
static void put_d(double* p, int64_t i, double v)
{
    if (p) p[i] = v;
}
static void put_i(int32_t* p, int64_t i, int32_t v)
{
    if (p) p[i] = v;
}

static int probs_row_ok(const double* P, int32_t V)
{
    for (int32_t v = 0; v < V; ++v)
        if (!(P[v] >= 0.0) || P[v] == INFINITY) return 0;
    return 1;
}

/* Greedy verify (temperature 0): the limit T -> 0 of the knobs keeps only a
 * row's argmax, so the acceptance check p_t(x)/p_d(x) > u passes iff x is the
 * target's argmax, and the token after the accepted prefix is the argmax of
 * the target row there ("Speculative Decoding from Scratch", How much faster
 * in practice? (3.3, 4.1): "argmax" decoding).  The lowest id wins a tie, as
 * in top-k.  Returns -1 for a row the step refuses (NaN, +inf, no finite). */
static int32_t row_argmax(const double* l, int32_t V)
{
    int32_t a = -1;
    for (int32_t v = 0; v < V; ++v) {
        if (isnan(l[v]) || l[v] == INFINITY) return -1;
        if (isfinite(l[v]) && (a < 0 || l[v] > l[a])) a = v;
    }
    return a;
}

static void verify_greedy_seq(const orc_verify_in* in, orc_verify_out* out, int32_t b, int32_t Kb,
                              double* lrow)
{
    const int32_t V = in->V, Kmax = in->K_max;
    int32_t jstar = -1, tok = -1;
    for (int32_t j = 0; j <= Kb; ++j) {
        load_row(in->target, in->target_dtype, (int64_t)b * (Kmax + 1) + j, V, lrow);
        const int32_t a = row_argmax(lrow, V);
        if (a < 0) {
            put_i(out->row_status, b, ORC_ROW_NONFINITE);
            for (int32_t i = 0; i < Kmax; ++i) put_d(out->p_t_at_draft, (int64_t)b * Kmax + i, NAN);
            return;
        }
        if (j < Kb) {
            const int32_t x = in->draft_tokens[(int64_t)b * Kmax + j];
            put_d(out->p_t_at_draft, (int64_t)b * Kmax + j, x == a ? 1.0 : 0.0);
            if (jstar < 0 && x != a) {
                jstar = j;
                tok = a;
            }
        } else if (jstar < 0) {
            jstar = Kb;
            tok = a;
        }
    }
    for (int32_t j = 0; j < jstar; ++j)
        put_i(out->tokens, (int64_t)b * (Kmax + 1) + j, in->draft_tokens[(int64_t)b * Kmax + j]);
    put_i(out->tokens, (int64_t)b * (Kmax + 1) + jstar, tok);
    put_i(out->num_accepted, b, jstar);
}

int orc_verify(const orc_verify_in* in, const orc_sampling* s, orc_verify_out* out,
               int32_t b_begin, int32_t b_end)
{
    const int32_t V = in->V, Kmax = in->K_max;
    double* lrow = (double*)malloc(sizeof(double) * (size_t)V);
    double* Pt = (double*)malloc(sizeof(double) * (size_t)V);
    double* Pd = (double*)malloc(sizeof(double) * (size_t)V);
    double* Pt_star = (double*)malloc(sizeof(double) * (size_t)V);
    double* Pd_star = (double*)malloc(sizeof(double) * (size_t)V);
    double* R = (double*)malloc(sizeof(double) * (size_t)V);
    if (!lrow || !Pt || !Pd || !Pt_star || !Pd_star || !R) return -1;

    for (int32_t b = b_begin; b < b_end; ++b) {
        for (int32_t j = 0; j <= Kmax; ++j) {
            put_i(out->tokens, (int64_t)b * (Kmax + 1) + j, -1);
            put_d(out->target_lse, (int64_t)b * (Kmax + 1) + j, NAN);
            put_d(out->topp_margin_t, (int64_t)b * (Kmax + 1) + j, INFINITY);
            if (j < Kmax) put_d(out->topp_margin_d, (int64_t)b * Kmax + j, INFINITY);
        }
        for (int32_t j = 0; j < Kmax; ++j) {
            put_d(out->p_t_at_draft, (int64_t)b * Kmax + j, NAN);
            put_d(out->p_d_at_draft, (int64_t)b * Kmax + j, NAN);
            put_d(out->alpha, (int64_t)b * Kmax + j, NAN);
        }
        put_i(out->num_accepted, b, -1);
        put_i(out->row_status, b, ORC_ROW_OK);
        put_d(out->residual_mass, b, 0.0);
        put_d(out->margin_accept, b, INFINITY);
        put_d(out->margin_topp, b, INFINITY);
        put_d(out->margin_cdf, b, INFINITY);
        put_i(out->cdf_lo, b, -1);
        put_i(out->cdf_hi, b, -1);

        const int32_t Kb = in->k_per_row ? in->k_per_row[b] : Kmax;
        if (Kb < 0 || Kb > Kmax) {
            put_i(out->row_status, b, ORC_ROW_BAD_K);
            continue;
        }
        int bad_token = 0;
        for (int32_t j = 0; j < Kb; ++j) {
            int32_t x = in->draft_tokens[(int64_t)b * Kmax + j];
            if (x < 0 || x >= V) bad_token = 1;
        }
        if (bad_token) {
            put_i(out->row_status, b, ORC_ROW_BAD_TOKEN);
            continue;
        }
        if (s->temperature == 0.0) {
            verify_greedy_seq(in, out, b, Kb, lrow);
            continue;
        }

        int nonfinite = 0;
        int32_t jstar = -1;
        double u_smp_star = 0.0;
        double m_acc = INFINITY, m_topp = INFINITY;
        orc_row_info it, id;

        for (int32_t j = 0; j < Kb && !nonfinite; ++j) {
            const int64_t trow = (int64_t)b * (Kmax + 1) + j;
            const int64_t drow = (int64_t)b * Kmax + j;
            load_row(in->target, in->target_dtype, trow, V, lrow);
            if (orc_row_dist(lrow, V, s->temperature, s->top_k, s->top_p, Pt, &it)) {
                nonfinite = 1;
                break;
            }
            id.topp_margin = INFINITY;
            if (in->draft_kind == ORC_DRAFT_LOGITS) {
                load_row(in->draft, in->draft_dtype, drow, V, lrow);
                if (orc_row_dist(lrow, V, s->temperature, s->top_k, s->top_p, Pd, &id)) {
                    nonfinite = 1;
                    break;
                }
            } else {
                /* probabilities are used as given */
                load_row(in->draft, ORC_F32, drow, V, Pd);
            }
            const int32_t x = in->draft_tokens[drow];
            const double p = Pt[x], q = Pd[x];
            if (in->draft_kind == ORC_DRAFT_PROBS && (!(q >= 0.0) || q == INFINITY)) {
                nonfinite = 1;
                break;
            }
            put_d(out->p_t_at_draft, drow, p);
            put_d(out->p_d_at_draft, drow, q);
            put_d(out->topp_margin_t, trow, it.topp_margin);
            put_d(out->topp_margin_d, drow, id.topp_margin);
            put_d(out->target_lse, trow, it.M + log(it.S));
            if (out->alpha) {
                double a = 0.0;
                for (int32_t v = 0; v < V; ++v) a += Pt[v] < Pd[v] ? Pt[v] : Pd[v];
                out->alpha[drow] = a;
            }
            if (jstar < 0) {
                double u_acc, u_smp;
                verify_uniforms(s->seed, s->round, b, j, 0u, &u_acc, &u_smp);
                const double ratio = p / q; /* IEEE: q = 0 gives +inf or NaN */
                const int accept = (u_acc < ratio);
                if (isfinite(ratio)) {
                    double m = fabs(u_acc - ratio);
                    if (m < m_acc) m_acc = m;
                }
                if (it.topp_margin < m_topp) m_topp = it.topp_margin;
                if (id.topp_margin < m_topp) m_topp = id.topp_margin;
                if (!accept) {
                    jstar = j;
                    u_smp_star = u_smp;
                    memcpy(Pt_star, Pt, sizeof(double) * (size_t)V);
                    memcpy(Pd_star, Pd, sizeof(double) * (size_t)V);
                }
            }
        }

        /* the target row at position K_b + 1 (the bonus row) */
        if (!nonfinite) {
            const int64_t trow = (int64_t)b * (Kmax + 1) + Kb;
            load_row(in->target, in->target_dtype, trow, V, lrow);
            if (orc_row_dist(lrow, V, s->temperature, s->top_k, s->top_p, Pt, &it))
                nonfinite = 1;
            else {
                put_d(out->target_lse, trow, it.M + log(it.S));
                put_d(out->topp_margin_t, trow, it.topp_margin);
            }
        }
        if (!nonfinite && jstar >= 0 && in->draft_kind == ORC_DRAFT_PROBS &&
            !probs_row_ok(Pd_star, V))
            nonfinite = 1;
        if (nonfinite) {
            put_i(out->row_status, b, ORC_ROW_NONFINITE);
            continue;
        }

        int32_t status = ORC_ROW_OK;
        double Z, margin;
        int32_t lo, hi, tok;
        if (jstar < 0) {
            /* every draft accepted: the bonus token from the target at K_b */
            double u_smp;
            verify_uniforms(s->seed, s->round, b, Kb, 0u, NULL, &u_smp);
            if (it.topp_margin < m_topp) m_topp = it.topp_margin;
            tok = orc_inverse_cdf(Pt, V, u_smp, s->delta, &Z, &margin, &lo, &hi);
            jstar = Kb;
            put_d(out->residual_mass, b, 0.0);
        } else {
            Z = orc_residual(Pt_star, Pd_star, V, R);
            put_d(out->residual_mass, b, Z);
            if (!(Z > 0.0)) {
                /* only rounding can empty the residual after a rejection: fall
                 * back to the target row itself and say so */
                memcpy(R, Pt_star, sizeof(double) * (size_t)V);
                status = ORC_ROW_ZERO_RESIDUAL;
            }
            tok = orc_inverse_cdf(R, V, u_smp_star, s->delta, &Z, &margin, &lo, &hi);
        }
        for (int32_t j = 0; j < jstar; ++j)
            put_i(out->tokens, (int64_t)b * (Kmax + 1) + j,
                  in->draft_tokens[(int64_t)b * Kmax + j]);
        put_i(out->tokens, (int64_t)b * (Kmax + 1) + jstar, tok);
        put_i(out->num_accepted, b, jstar);
        put_i(out->row_status, b, status);
        put_d(out->margin_accept, b, m_acc);
        put_d(out->margin_topp, b, m_topp);
        put_d(out->margin_cdf, b, margin);
        put_i(out->cdf_lo, b, lo);
        put_i(out->cdf_hi, b, hi);
    }
    free(lrow);
    free(Pt);
    free(Pd);
    free(Pt_star);
    free(Pd_star);
    free(R);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Draft-side sampler: "q = draft.probs(...); x = sample(q)" of the listing  */
/* "One speculative decoding loop", with the knobs applied to logits and     */
/* the inverse CDF drawn with Philox tag 1.                                 */
/* ------------------------------------------------------------------------ */
int orc_draft_sample(const orc_verify_in* in, const orc_sampling* s, int32_t* tokens,
                     double* margin, int32_t b_begin, int32_t b_end)
{
    const int32_t V = in->V, Kmax = in->K_max;
    double* lrow = (double*)malloc(sizeof(double) * (size_t)V);
    double* P = (double*)malloc(sizeof(double) * (size_t)V);
    if (!lrow || !P) return -1;
    for (int32_t b = b_begin; b < b_end; ++b) {
        const int32_t Kb = in->k_per_row ? in->k_per_row[b] : Kmax;
        for (int32_t j = 0; j < Kmax; ++j) {
            const int64_t drow = (int64_t)b * Kmax + j;
            tokens[drow] = -1;
            if (margin) margin[drow] = INFINITY;
            if (Kb < 0 || Kb > Kmax || j >= Kb) continue;
            int ok;
            if (in->draft_kind == ORC_DRAFT_LOGITS && s->temperature == 0.0) {
                /* greedy drafting: the draft row's argmax (lowest id on ties) */
                load_row(in->draft, in->draft_dtype, drow, V, lrow);
                tokens[drow] = row_argmax(lrow, V);
                continue;
            }
            if (in->draft_kind == ORC_DRAFT_LOGITS) {
                load_row(in->draft, in->draft_dtype, drow, V, lrow);
                ok = orc_row_dist(lrow, V, s->temperature, s->top_k, s->top_p, P, NULL) == 0;
            } else {
                load_row(in->draft, ORC_F32, drow, V, P);
                ok = probs_row_ok(P, V);
            }
            if (!ok) continue;
            double u;
            verify_uniforms(s->seed, s->round, b, j, 1u, &u, NULL);
            double m;
            tokens[drow] = orc_inverse_cdf(P, V, u, s->delta, NULL, &m, NULL, NULL);
            if (margin) margin[drow] = m;
        }
    }
    free(lrow);
    free(P);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* LM head: logits = hidden x W_vocab, the textbook triple loop in double.  */
/* ------------------------------------------------------------------------ */
void orc_lmhead(const uint16_t* H, const uint16_t* W, int32_t N, int32_t K, int32_t m0,
                int32_t m1, double* out)
{
    for (int32_t m = m0; m < m1; ++m) {
        double* o = out + (int64_t)(m - m0) * N;
        for (int32_t n = 0; n < N; ++n) o[n] = 0.0;
        for (int32_t k = 0; k < K; ++k) {
            const double h = widen(H, ORC_BF16, (int64_t)m * K + k);
            const uint16_t* wrow = W + (int64_t)k * N;
            for (int32_t n = 0; n < N; ++n) o[n] += h * widen(wrow, ORC_BF16, n);
        }
    }
}
