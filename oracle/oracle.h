/*
 * oracle.h -- plain, slow, single-threaded fp64 CPU oracle for the batched
 * speculative-sampling verify step.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library. The product path (the CUDA
 * library under the package directory) shares no code, header, table or
 * constant with it, and never calls it.
 *
 * What it computes follows the pages this project is built from:
 *   - "Accelerating Large Language Model Decoding with Speculative Sampling"
 *     (zeroshotmind.com), sections "The algorithm" and "Why the output
 *     distribution is exactly the target's";
 *   - "57 Speculative Decoding" (ml-canon), section "Acceptance, and why the
 *     distribution is NOT distorted" and the listing "One speculative decoding
 *     loop";
 *   - "Speculative Decoding from Scratch" (ta-paperlens), sections "The big
 *     picture: draft -> verify in one batch -> patch (2.1)" and "The heart of
 *     it: an acceptance rule that never changes the output distribution (2.3)";
 *   - "Speculative Decoding: Getting 3x Speedups Without Changing the Model"
 *     (generalcompute), section "How It Works", steps 3 and 4;
 *   - "NOTE-159: Accelerating Large Language Model Decoding with Speculative
 *     Sampling" (dmarx), "Key results" (sampling knobs applied before the
 *     rejection step) and "Recommendations" R3.
 * Where the pages are silent the plainest reading is taken, and the comment at
 * the point of use says which reading it is.
 *
 * Pins (what this oracle is checked against, in tests/): curand's host
 * Philox4x32-10 stream, the logistic closed form at V = 2, counting
 * definitions of top-k / top-p, textbook greedy speculative decoding at
 * top-k = 1, exact residual identity, the E[tokens per pass] closed form, and
 * chi-square goodness of fit of the emitted tokens against the target
 * distribution.
 */
#ifndef SPEC_ORACLE_H
#define SPEC_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types of the input buffers (same codes as the product ABI, but
 * declared here independently) */
#define ORC_F32 0
#define ORC_BF16 1

#define ORC_DRAFT_LOGITS 0
#define ORC_DRAFT_PROBS 1

/* per-sequence status codes */
#define ORC_ROW_OK 0
#define ORC_ROW_BAD_TOKEN 1
#define ORC_ROW_BAD_K 2
#define ORC_ROW_NONFINITE 3
#define ORC_ROW_ZERO_RESIDUAL 4

/* Philox4x32-10 of Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3" (SC'11): out = bijection(ctr) keyed by key. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* u = (w >> 8) * 2^-24, a 24-bit uniform in [0, 1). */
double orc_u24(uint32_t w);

/* out[4*i .. 4*i+3] = Philox(ctrs[4*i .. 4*i+3]) keyed by (seed_lo, seed_hi),
 * for i in [0, n).  Used by the generator pins. */
void orc_philox_batch(uint64_t seed, const uint32_t* ctrs, int64_t n, uint32_t* out);

/* Diagnostics of one row distribution after the sampling knobs. */
typedef struct {
    double M;            /* max of z = l / T over the kept set              */
    double S;            /* sum over the kept set of exp(z - M)             */
    double topp_margin;  /* |prefix - top_p| at the nucleus boundary (inf if off) */
    int32_t n_kept;      /* size of the final kept set                      */
    int32_t nonfinite;   /* 1 when a logit is NaN or +inf, or none is finite */
} orc_row_info;

/* Temperature, then top-k, then top-p, then softmax of one logit row.
 *   l:  V logits (already widened to double)
 *   T:  temperature (> 0)
 *   top_k: 0 or >= V means off; else keep the k best by (l desc, id asc)
 *   top_p: >= 1 means off; else strict prefix rule in the same rank order
 *   P:  out, V probabilities (0 outside the kept set)
 * Returns 0, or -1 when the row is non-finite (P then untouched). */
int orc_row_dist(const double* l, int32_t V, double T, int32_t top_k, double top_p,
                 double* P, orc_row_info* info);

/* Inverse CDF in ascending token order: t = u * Z with Z = sum R; returns the
 * smallest v with C(v) > t, or the largest v with R(v) > 0 when rounding leaves
 * none; -1 when Z == 0.  margin = min(t - C(v-1), C(v) - t) / Z.  v_lo / v_hi
 * are the tokens chosen for t -/+ delta * Z (the near-tie neighbourhood). */
int32_t orc_inverse_cdf(const double* R, int32_t V, double u, double delta,
                        double* Z_out, double* margin, int32_t* v_lo, int32_t* v_hi);

/* Residual max(0, Pt - Pd) (unnormalised) into R; returns its sum Z. */
double orc_residual(const double* Pt, const double* Pd, int32_t V, double* R);

typedef struct {
    int32_t B, K_max, V;
    int32_t target_dtype;          /* ORC_F32 / ORC_BF16                   */
    const void* target;            /* [B, K_max+1, V]                      */
    int32_t draft_kind;            /* ORC_DRAFT_LOGITS / ORC_DRAFT_PROBS   */
    int32_t draft_dtype;           /* logits: ORC_F32/ORC_BF16; probs: ORC_F32 */
    const void* draft;             /* [B, K_max, V]                        */
    const int32_t* draft_tokens;   /* [B, K_max]                           */
    const int32_t* k_per_row;      /* [B] or NULL (all K_max)              */
} orc_verify_in;

typedef struct {
    double temperature;            /* > 0                                  */
    int32_t top_k;
    double top_p;
    uint64_t seed;
    uint64_t round;
    double delta;                  /* near-tie window for the margins      */
} orc_sampling;

typedef struct {
    int32_t* tokens;               /* [B, K_max+1], -1 padded              */
    int32_t* num_accepted;         /* [B]                                  */
    int32_t* row_status;           /* [B]                                  */
    double* p_t_at_draft;          /* [B, K_max] (NaN where not defined)   */
    double* p_d_at_draft;          /* [B, K_max]                           */
    double* residual_mass;         /* [B] Z at the first rejection, 0 if none */
    double* target_lse;            /* [B, K_max+1] M + log S over kept set */
    double* alpha;                 /* [B, K_max] sum_v min(Pt, Pd)         */
    double* margin_accept;         /* [B] min |u - ratio| over tested slots */
    double* margin_topp;           /* [B] min top-p margin over used rows  */
    double* margin_cdf;            /* [B] margin of the final inverse CDF  */
    int32_t* cdf_lo;               /* [B] near-tie neighbourhood of the    */
    int32_t* cdf_hi;               /* [B]   final sampled token            */
    double* topp_margin_t;         /* [B, K_max+1] top-p margin of each target row */
    double* topp_margin_d;         /* [B, K_max] top-p margin of each draft row    */
} orc_verify_out;

/* Verify sequences b in [b_begin, b_end).  Any output pointer may be NULL. */
int orc_verify(const orc_verify_in* in, const orc_sampling* s, orc_verify_out* out,
               int32_t b_begin, int32_t b_end);

/* Draft-side sampler: x[b, j] ~ P_d[b, j] (after the knobs when the draft is
 * logits, as given when it is probabilities) by inverse CDF with the Philox
 * stream tag 1.  tokens [B, K_max] (-1 for j >= K_b); margin [B, K_max]. */
int orc_draft_sample(const orc_verify_in* in, const orc_sampling* s, int32_t* tokens,
                     double* margin, int32_t b_begin, int32_t b_end);

/* One row's final distribution P (after knobs) as double, for tests. */
int orc_row_probs(const void* row, int32_t dtype, int32_t V, double T, int32_t top_k,
                  double top_p, double* P, orc_row_info* info);

/* LM head in fp64: out[m - m0][n] = sum_k H[m][k] * W[k][n] for m in [m0, m1).
 * H: [M, K] bf16 bits, W: [K, N] bf16 bits, row-major. */
void orc_lmhead(const uint16_t* H, const uint16_t* W, int32_t N, int32_t K,
                int32_t m0, int32_t m1, double* out);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_ORACLE_H */
