/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) batched speculative-sampling
 * verify step.
 *
 * The operation.  For each of B sequences with K_b drafted tokens x_0..x_{K_b-1}
 * (0 <= K_b <= K_max), the target gives logits at K_b + 1 positions and the
 * draft gives a distribution at K_b positions over one shared vocabulary of V
 * tokens.  The step:
 *   1. applies temperature, then top-k, then top-p to every target row and to
 *      every draft row given as logits, and softmaxes each row
 *      ("NOTE-159: Accelerating Large Language Model Decoding with Speculative
 *      Sampling", Key results: sampling knobs applied to the probabilities
 *      before the rejection step; Recommendations R3);
 *   2. walks the drafts left to right and accepts x_j iff u_j < p_t(x_j) /
 *      p_d(x_j), stopping at the first rejection j*
 *      ("Accelerating Large Language Model Decoding with Speculative Sampling",
 *      The algorithm; "57 Speculative Decoding", the listing "One speculative
 *      decoding loop");
 *   3. resamples position j* from max(0, p_t - p_d) renormalised, by inverse CDF
 *      in ascending token id, or, when every draft passed, samples one bonus
 *      token from the target row at position K_b + 1
 *      ("Speculative Decoding from Scratch", The big picture (2.1) step 3 and
 *      The heart of it (2.3); "Speculative Decoding: Getting 3x Speedups
 *      Without Changing the Model", How It Works, steps 3-4).
 * The output of a sequence is x_0..x_{j*-1} followed by the sampled token:
 * between 1 and K_b + 1 tokens.
 *
 * Greedy verify (temperature 0).  The limit T -> 0 of the knobs keeps one
 * token per row, its argmax (the lowest id among equal maxima); x_j is
 * accepted iff it is the argmax of target row j, and the emitted token is the
 * argmax of target row j* (or of row K_b when every draft matched): the
 * greedy ("argmax") decoding that "Speculative Decoding from Scratch", How
 * much faster in practice? (3.3, 4.1), measures beside temperature 1, taken as
 * the T -> 0 limit of the acceptance check.  No uniform is drawn, no draft row
 * is read (draft may be NULL), and top_k / top_p have no effect.
 *
 * Uniforms.  Philox4x32-10 (Salmon et al., SC'11) keyed by the 64-bit seed;
 * counter = ((j << 2) | tag, b, round_lo, round_hi); u = (word >> 8) * 2^-24.
 * Tag 0: word 0 is the accept uniform of slot j, word 1 the sampling uniform
 * of slot j (the resample at j*, or the bonus at j = K_b).  Tag 1, word 0:
 * the uniform of the draft-side sampler for slot j.
 *
 * Conventions.
 *  - Every tensor pointer is DEVICE memory owned by the caller, contiguous,
 *    row-major.  The library never frees or keeps caller memory.
 *  - A handle owns only its device workspace, sized at create time for
 *    max_batch x max_k x vocab.  One handle must not run on two streams at
 *    once; create one handle per concurrent stream.
 *  - spec_verify_run and spec_draft_sample are asynchronous on the given
 *    stream (a cudaStream_t passed as void*; NULL is the legacy default
 *    stream): no host synchronisation and no allocation.
 *  - Errors found on the host return a status and launch nothing.  Data
 *    errors found on the device are reported per sequence in row_status (see
 *    SPEC_ROW_*); such sequences get tokens = -1 and num_accepted = -1.
 *  - -inf logits are allowed (masked tokens, probability 0).  A NaN or +inf
 *    logit, or a row with no finite logit, in any row the step reads makes
 *    the sequence SPEC_ROW_NONFINITE.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct spec_verify* spec_verify_t; /* opaque handle */

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1, /* a NULL required pointer, a size out of range, a bad knob */
    SPEC_ERR_UNSUPPORTED = 2, /* a valid request the library does not implement        */
    SPEC_ERR_OOM = 3,         /* workspace allocation failed (create only)              */
    SPEC_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed            */
    SPEC_ERR_TIMEOUT = 5      /* a bounded device-side wait ran out (spec_verify_check) */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;
typedef enum { SPEC_TARGET_LOGITS = 0, SPEC_TARGET_HIDDEN_LMHEAD = 1 } spec_target_kind;
typedef enum { SPEC_DRAFT_LOGITS = 0, SPEC_DRAFT_PROBS = 1 } spec_draft_kind;

/* per-sequence row_status values */
enum {
    SPEC_ROW_OK = 0,
    SPEC_ROW_BAD_TOKEN = 1,     /* a drafted token at j < K_b outside [0, V)              */
    SPEC_ROW_BAD_K = 2,         /* K_b outside [0, K_max]                                 */
    SPEC_ROW_NONFINITE = 3,     /* NaN / +inf / no finite logit; or a negative, NaN or    */
                                /* +inf draft probability where one is read               */
    SPEC_ROW_ZERO_RESIDUAL = 4  /* the residual summed to 0 after a rejection (rounding   */
                                /* only): the token was drawn from p_t; output is valid   */
};

/* SPEC_TARGET_HIDDEN_LMHEAD (the fused round): `target` is the bf16 hidden
 * states [B * (k_max + 1), H] of the verified positions and `w_vocab` the bf16
 * LM head [H, V]; the run first computes the fp32 logits H x W_vocab (fp32
 * accumulation, tensor cores) into the handle's workspace and verifies them.
 * It needs target_dtype = SPEC_BF16, hidden = H, draft probabilities
 * (SPEC_DRAFT_PROBS, SPEC_F32) and H and V multiples of 8 (else create returns
 * SPEC_ERR_UNSUPPORTED); hidden and w_vocab must start on 16 bytes. */
typedef struct {
    int32_t device;       /* CUDA device ordinal                                     */
    int32_t max_batch;    /* largest B of any run                                    */
    int32_t max_k;        /* largest K_max of any run                                */
    int32_t vocab;        /* V (>= 1), shared by target and draft                    */
    int32_t hidden;       /* H of the fused LM head (SPEC_TARGET_HIDDEN_LMHEAD), else 0 */
    int32_t target_kind;  /* spec_target_kind                                        */
    int32_t target_dtype; /* spec_dtype of the target logits                         */
    int32_t draft_kind;   /* spec_draft_kind                                         */
    int32_t draft_dtype;  /* logits: equal to target_dtype; probabilities: SPEC_F32  */
} spec_verify_config;

typedef struct {
    float temperature; /* T > 0, or T == 0 for greedy verify (see above)            */
    int32_t top_k;     /* 0 or >= V: off; else keep the k highest logits, ties to   */
                       /* the lower token id                                         */
    float top_p;       /* >= 1: off; in (0, 1): keep the rank-ordered prefix whose   */
                       /* mass strictly before each kept token is < top_p            */
    int32_t reserved;  /* must be 0                                                  */
    uint64_t seed;     /* Philox key                                                 */
    uint64_t round;    /* Philox counter words 2-3 (one value per verify round)      */
} spec_sampling;

typedef struct {
    const void* target;          /* [B, k_max+1, V] logits of target_dtype; or, for the */
                                 /* LM head, hidden states [B*(k_max+1), H] bf16        */
    const void* w_vocab;         /* [H, V] bf16 for the LM head, else NULL              */
    const void* draft;           /* [B, k_max, V]: logits (draft_dtype) or f32 probs    */
    const int32_t* draft_tokens; /* [B, k_max]; slots j >= K_b are ignored              */
    const int32_t* k_per_row;    /* [B] per-sequence K_b, or NULL for K_b = k_max       */
    int32_t batch;               /* B, 0 <= B <= max_batch (0 is a no-op)               */
    int32_t k_max;               /* padded draft length of this run, <= max_k           */
} spec_verify_inputs;

typedef struct {
    int32_t* tokens;        /* [B, k_max+1] emitted tokens, -1 padded (required)      */
    int32_t* num_accepted;  /* [B] accepted drafts j* (required); emitted = j* + 1     */
    int32_t* row_status;    /* [B] SPEC_ROW_* or NULL                                 */
    float* p_t_at_draft;    /* [B, k_max] p_t(x_j) after knobs, NaN for j >= K_b; or NULL */
                            /* (greedy: 1 where x_j is the argmax, else 0)             */
    float* p_d_at_draft;    /* [B, k_max] p_d(x_j), NaN for j >= K_b (and greedy); or NULL */
    float* residual_mass;   /* [B] sum of max(0, p_t - p_d) at j*, 0 if all accepted   */
                            /* (and greedy); or NULL                                   */
    float* target_lse;      /* [B, k_max+1] log-sum-exp of l/T over the kept set, NaN  */
                            /* beyond K_b (and greedy); or NULL                        */
    float* alpha;           /* [B, k_max] acceptance statistic alpha_j = sum_v          */
                            /* min(p_t(v), p_d(v)) after the knobs ("Speculative       */
                            /* Decoding from Scratch", The acceptance rate alpha      */
                            /* decides everything (3.1-3.2)); NaN for j >= K_b, failed */
                            /* sequences and greedy; or NULL (not computed: one more  */
                            /* kernel, which re-reads the rows not kept as lists)      */
} spec_verify_outputs;

/* Allocate a handle and its device workspace on cfg->device (with the LM
 * head, also the fp32 logits [max_batch * (max_k + 1), V]).
 * Returns SPEC_ERR_INVALID_ARG for sizes < 1 (max_k may be 0) or a dtype/kind
 * combination outside the table above, SPEC_ERR_UNSUPPORTED for an LM-head
 * configuration outside the one described above, SPEC_ERR_OOM when the
 * workspace does not fit.  On error *out is NULL. */
spec_status spec_verify_create(const spec_verify_config* cfg, spec_verify_t* out);

/* One verify step for a batch (the operation described at the top).  All
 * outputs are written on `stream`; the call returns before they are ready. */
spec_status spec_verify_run(spec_verify_t h, const spec_verify_inputs* in,
                            const spec_sampling* s, const spec_verify_outputs* out,
                            void* stream);

/* The same verify with early exit (NEXT f2): for each sequence the target and
 * draft rows of position j are read only when every draft before j was
 * accepted, since the drafts after the first rejection are discarded
 * ("Accelerating Large Language Model Decoding with Speculative Sampling",
 * The algorithm), so the bytes read fall from 2 K_b + 1 rows to about
 * 2 sum_j alpha^j.  Each CTA walks whole sequences: it pays at large B, and
 * at small B (fewer sequences than SMs) the full verify is faster.
 * It applies to rows of logits on 16 bytes with 1 <= top-k <= 128 (or
 * greedy) and no LM head; otherwise it runs spec_verify_run.
 * Results are those of spec_verify_run except that
 *  - a NaN or +inf logit in a row after the first rejection is not seen;
 *  - p_t / p_d at the drafted tokens and target_lse are written for the
 *    positions read and NaN beyond; alpha is NaN.
 * Rows whose top-k candidates overflow its staging (heavy ties) make the
 * regular pipeline, enqueued behind it, recompute the whole batch. */
spec_status spec_verify_run_early_exit(spec_verify_t h, const spec_verify_inputs* in,
                                       const spec_sampling* s, const spec_verify_outputs* out,
                                       void* stream);

/* Draft-side sampler, the step before the verify: x = sample(q) of the listing
 * "One speculative decoding loop" ("57 Speculative Decoding").  For every
 * sequence b and slot j < K_b: draws draft_tokens[b, j] ~ P_d[b, j] (the draft
 * row after the knobs when it is logits, as given when it is probabilities) by
 * inverse CDF with the tag-1 uniform; slots j >= K_b get -1.  When draft_probs
 * is not NULL it receives the dense post-knob draft distribution [B, k_max, V]
 * (f32; rows j >= K_b untouched).  `draft` has the handle's draft kind/dtype. */
spec_status spec_draft_sample(spec_verify_t h, const void* draft, const int32_t* k_per_row,
                              int32_t batch, int32_t k_max, const spec_sampling* s,
                              int32_t* draft_tokens, float* draft_probs, void* stream);

/* The verify step for callers that cannot allocate device memory: a plugin
 * or operator interface that is handed only a stream at enqueue time, a
 * serving loop whose memory is a fixed arena owned by someone else, or code
 * that must not trigger the implicit device synchronisation an allocation can
 * cause.  The pages have no counterpart of this call: it is a deployment
 * variant of spec_verify_run.
 *
 * It takes no handle and allocates nothing.  Its workspace is one static
 * device array of SPEC_NOALLOC_SCRATCH_BYTES (16 MiB) inside the library,
 * which every GPU that loads the library holds until the process exits.
 * Inputs, outputs and their meaning are those of spec_verify_run; cfg gives
 * the device, vocabulary, kinds and dtypes (its max_batch / max_k are not
 * used: the sizes come from `in`).
 *  - The first call on a device looks up the array's device address on that
 *    device (once); make that first call before any stream capture begins.
 *  - A configuration with the fused LM head (SPEC_TARGET_HIDDEN_LMHEAD)
 *    returns SPEC_ERR_UNSUPPORTED: its fp32 logits alone exceed the array.
 *  - Sizes whose workspace would not fit the array return
 *    SPEC_ERR_INVALID_ARG and launch nothing.  The workspace is about
 *      per row slot (B * (2 K_max + 1) of them): 8244 bytes + 16 bytes per
 *        segment of 16 KB of the row + 2 bytes per 128-byte chunk of the row
 *        (but at least 256 bytes per 8192 tokens: the key histograms),
 *        i.e. 12.3 KiB at V = 128256 bf16 and 16.4 KiB at V = 128256 fp32;
 *      per drafted slot (B * K_max of them): 28 bytes + 40 bytes per 4096
 *        tokens, i.e. 1.28 KiB at V = 128256;
 *    so B = 64 with K_max = 8 at V = 128256 bf16 (1088 row slots, 512
 *    drafted slots) needs 14.4 MB.
 *  - Every call shares the one array and each call reuses the last call's
 *    contents (the counters that must start at zero are cleared on the
 *    stream first), so calls that overlap on the GPU race: issue them on one
 *    stream, or serialise them. */
#define SPEC_NOALLOC_SCRATCH_BYTES (16u << 20)
spec_status spec_verify_run_noalloc(const spec_verify_config* cfg, const spec_verify_inputs* in,
                                    const spec_sampling* s, const spec_verify_outputs* out,
                                    void* stream);

/* The LM head alone: logits[m, V] (fp32, row-major, row stride V) =
 * hidden[m, H] (bf16, row-major) x w_vocab[H, V] (bf16, row-major), fp32
 * accumulation on the tensor cores, asynchronous on `stream` (the current
 * device; all pointers device memory owned by the caller, 16-byte aligned).
 * m = 0 is a no-op.  Returns SPEC_ERR_INVALID_ARG for NULL pointers or sizes
 * < 1, SPEC_ERR_UNSUPPORTED when H or V is not a multiple of 8 or a pointer is
 * not on 16 bytes, SPEC_ERR_CUDA when the launch fails. */
spec_status spec_lmhead_logits(const void* hidden, const void* w_vocab, int32_t m, int32_t hidden_dim,
                               int32_t vocab, float* logits, void* stream);

/* Measurement hook (the pages have no counterpart): every later run of the
 * handle records ev_stage1_begin just before and ev_stage1_end just after the
 * kernel that reads the run's bulk input (the stage-1 stream kernel over the
 * logits, or the LM head over W_vocab when the target is hidden states) on the
 * run's stream,
 * so the caller can time that kernel with cudaEventElapsedTime; and when
 * launches_out is not NULL, each run stores there (host memory, written
 * before the call returns) the number of kernels it launched.  The events are
 * cudaEvent_t created by the caller on the handle's device and stay owned by
 * the caller, who must keep them valid while the hook is set.  Pass NULL for
 * all three to switch it off.  Returns SPEC_ERR_INVALID_ARG for a NULL handle
 * or when exactly one of the two events is NULL.  Recording the events may
 * stop the next kernel from being scheduled before the stream kernel ends, so
 * a run with the hook set can take slightly longer. */
spec_status spec_verify_set_profiling(spec_verify_t h, void* ev_stage1_begin, void* ev_stage1_end,
                                      int32_t* launches_out);

/* Device-side failure report (the pages have no counterpart).  Every wait
 * of the library's kernels on a copy or on another warp is bounded; a wait
 * that runs out records it in the handle's workspace and its kernel returns
 * early, which leaves that run's outputs undefined but the CUDA context
 * usable.  This call waits for the work queued on `stream` (a cudaStream_t
 * as void*, NULL the legacy default stream), reads the record and clears it.
 * Returns SPEC_ERR_TIMEOUT when a run of the handle since the last check ran
 * out of a wait, SPEC_OK when none did, SPEC_ERR_INVALID_ARG for a NULL
 * handle and SPEC_ERR_CUDA when the wait or the read fails. */
spec_status spec_verify_check(spec_verify_t h, void* stream);

/* Fault injection for tests of the failure report (the pages have no
 * counterpart); it acts on the host side only.  SPEC_FAULT_STALL_STREAM makes
 * the next spec_verify_run of the handle launch only its stage-1 stream
 * kernel, whose producer issues no copy, so that the consumers' waits run out
 * after a short limit (4096 polls) and record a timeout; no other kernel of
 * that run is launched and its outputs are not written.  It applies to one
 * run, then resets to SPEC_FAULT_NONE.  The run returns
 * SPEC_ERR_UNSUPPORTED (and the fault stays armed) when its rows do not take
 * the stream kernel (rows not on 16 bytes, the LM head).  Returns
 * SPEC_ERR_INVALID_ARG for a NULL handle or an unknown fault. */
enum { SPEC_FAULT_NONE = 0, SPEC_FAULT_STALL_STREAM = 1 };
spec_status spec_verify_inject_fault(spec_verify_t h, int32_t fault);

/* Workspace allocator (the pages have no counterpart).  By default a handle's
 * workspace comes from cudaMalloc and goes back with cudaFree.  A caller that
 * manages device memory itself (a pooled allocator, a memory budget) installs
 * alloc / release here: spec_verify_create then calls alloc(ctx, bytes,
 * device, &ptr) with `device` current, which returns 0 and a device pointer
 * aligned to 256 bytes on success and nonzero on failure (create then returns
 * SPEC_ERR_OOM); spec_verify_destroy calls release(ctx, ptr, device).  A
 * handle keeps the functions it was created with.  Passing NULL for both
 * restores cudaMalloc / cudaFree.  The setting is process-wide and applies to
 * handles created after the call.  Returns SPEC_ERR_INVALID_ARG when exactly
 * one of the two functions is NULL. */
typedef int (*spec_alloc_fn)(void* ctx, uint64_t bytes, int32_t device, void** ptr);
typedef void (*spec_release_fn)(void* ctx, void* ptr, int32_t device);
spec_status spec_verify_set_allocator(spec_alloc_fn alloc, spec_release_fn release, void* ctx);

/* Free the handle and its workspace (synchronises its device first). */
spec_status spec_verify_destroy(spec_verify_t h);

/* Static English text for a status code. */
const char* spec_verify_status_string(spec_status s);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
