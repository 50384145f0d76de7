// sv_api.cu -- the C ABI (include/spec_verify.h): argument checks, workspace,
// launch sequence.  Host code only; every step of the computation runs in the
// kernels of sv_rows.cu and sv_sample.cu.
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <new>

#include "sv_internal.cuh"
#include "spec_verify.h"

using namespace sv;

struct spec_verify {
    spec_verify_config cfg;
    int64_t rows_cap;     // max_batch * (2 * max_k + 1)
    int64_t jobs_cap;     // max_batch * max(1, max_k)
    int nseg_cap, nchunk_cap, nseg_sample;
    int chunk_stride;     // chunk keys per row slot (multiple of 8: 16-byte rows)
    int num_sms;          // streaming kernel: two CTAs per SM
    void* ws;
    size_t ws_bytes;
    SegStat* seg;
    uint16_t* chunk;
    RowStat* rstat;
    int32_t* kept_id;
    float* kept_l;
    unsigned* row_ticket;
    unsigned* seq_ticket;
    Job* jobs;
    unsigned long long* job_seg;
    unsigned long long* job_part;
    unsigned* job_ticket;
    unsigned* err;
    unsigned* seq_done;
    unsigned* exit_flag;  // early exit: a sequence was left to the regular pipeline
    // spec_verify_set_profiling: events around the stage-1 stream kernel and
    // where each run stores the number of kernels it launched (all optional)
    cudaEvent_t prof_begin;
    cudaEvent_t prof_end;
    int32_t* prof_launches;
    float* logits;        // the LM head's output (SPEC_TARGET_HIDDEN_LMHEAD), else NULL
    int fault;            // spec_verify_inject_fault: the fault armed for the next run
    // where the workspace came from (NULL: cudaMalloc / cudaFree)
    spec_alloc_fn alloc_fn;
    spec_release_fn release_fn;
    void* alloc_ctx;
};

namespace {

int elem_size(int dtype) { return dtype == SPEC_BF16 ? 2 : 4; }
int seg_elems(int dtype) { return SEG_BYTES / elem_size(dtype); }
int chunk_elems(int dtype) { return CHUNK_BYTES / elem_size(dtype); }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard()
    {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// spec_verify_set_allocator: the functions later handles take their workspace from
struct AllocHook {
    std::mutex mu;
    spec_alloc_fn alloc = nullptr;
    spec_release_fn release = nullptr;
    void* ctx = nullptr;
};
AllocHook& alloc_hook()
{
    static AllocHook hook;
    return hook;
}

// polls of a wait that runs out on purpose (SPEC_FAULT_STALL_STREAM)
constexpr uint32_t STALL_WAIT_POLLS = 4096;

// knobs of one launch; SPEC_OK or the error to return
spec_status fill_knobs(const spec_verify* h, const spec_sampling* s, Params& p)
{
    if (!s || s->reserved != 0) return SPEC_ERR_INVALID_ARG;
    const float T = s->temperature;
    if (!(T >= 0.f) || isinf(T)) return SPEC_ERR_INVALID_ARG;
    if (s->top_k < 0) return SPEC_ERR_INVALID_ARG;
    if (!(s->top_p > 0.f)) return SPEC_ERR_INVALID_ARG;  // also rejects NaN
    const int V = h->cfg.vocab;
    // temperature 0 is greedy: the kept set of every row is its argmax (the
    // lowest id among equal maxima), i.e. top-k = 1; top-k and top-p do not
    // change it; the verify reads no draft row
    p.greedy = T == 0.f ? 1 : 0;
    p.T = p.greedy ? 1.f : T;
    p.c = (float)(1.4426950408889634 / (double)p.T);
    p.c_lo = (float)(1.4426950408889634 / (double)p.T - (double)p.c);
    p.top_k = p.greedy ? (V > 1 ? 1 : 0) : (s->top_k > 0 && s->top_k < V) ? s->top_k : 0;
    p.top_p = p.greedy ? 1.f : s->top_p < 1.f ? s->top_p : 1.f;
    p.top_p_fix = !p.greedy && s->top_p < 1.f ? (uint64_t)((double)s->top_p * 72057594037927936.0) : 0;
    p.seed = s->seed;
    p.round = s->round;
    return SPEC_OK;
}

void fill_workspace(const spec_verify* h, Params& p)
{
    p.seg = h->seg;
    p.chunk = h->chunk;
    p.rstat = h->rstat;
    p.kept_id = h->kept_id;
    p.kept_l = h->kept_l;
    p.row_ticket = h->row_ticket;
    p.seq_ticket = h->seq_ticket;
    p.jobs = h->jobs;
    p.job_seg = h->job_seg;
    p.job_part = h->job_part;
    p.job_ticket = h->job_ticket;
    p.nseg_sample = h->nseg_sample;
    p.chunk_stride = h->chunk_stride;
    p.err = h->err;
    p.seq_done = h->seq_done;
}

// one workspace: 256-byte aligned sub-buffers for max_batch x max_k x vocab.
// Fills h's pointers when base is not NULL; returns the bytes needed.
size_t layout_workspace(spec_verify* h, void* base)
{
    const spec_verify_config* cfg = &h->cfg;
    const int64_t V = cfg->vocab;
    h->rows_cap = (int64_t)cfg->max_batch * (2 * (int64_t)cfg->max_k + 1);
    h->jobs_cap = (int64_t)cfg->max_batch * (cfg->max_k > 0 ? cfg->max_k : 1);
    int dts[2] = {cfg->target_dtype, cfg->draft_dtype};
    h->nseg_cap = 1;
    h->nchunk_cap = 1;
    for (int dt : dts) {
        h->nseg_cap = (int)std::max<int64_t>(h->nseg_cap, cdiv(V, seg_elems(dt)));
        h->nchunk_cap = (int)std::max<int64_t>(h->nchunk_cap, cdiv(V, chunk_elems(dt)));
    }
    // the LM head's softmax partials: one per 256-column tile
    if (cfg->target_kind == SPEC_TARGET_HIDDEN_LMHEAD)
        h->nseg_cap = (int)std::max<int64_t>(h->nseg_cap, cdiv(V, LM_STAT_COLS));
    h->nseg_sample = (int)cdiv(V, SAMPLE_SEG);
    // the chunk-key area of a row slot also holds its key histograms (bf16
    // rows with top-p alone): HIST_BINS bytes per 16 KB segment
    const int64_t hist_keys = cdiv(V, seg_elems(SPEC_BF16)) * HIST_BINS / 2;
    h->chunk_stride = (int)(cdiv(std::max<int64_t>(h->nchunk_cap, hist_keys), 8) * 8);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += (bytes + 255) & ~(size_t)255;
        return at;
    };
    const size_t o_seg = take(sizeof(SegStat) * h->rows_cap * h->nseg_cap);
    const size_t o_chunk = take(sizeof(uint16_t) * h->rows_cap * h->chunk_stride);
    const size_t o_rstat = take(sizeof(RowStat) * h->rows_cap);
    const size_t o_kid = take(sizeof(int32_t) * h->rows_cap * KCAP);
    const size_t o_kl = take(sizeof(float) * h->rows_cap * KCAP);
    const size_t o_rt = take(sizeof(unsigned) * h->rows_cap);
    const size_t o_st = take(sizeof(unsigned) * cfg->max_batch);
    const size_t o_jobs = take(sizeof(Job) * h->jobs_cap);
    const size_t o_jseg = take(sizeof(unsigned long long) * h->jobs_cap * h->nseg_sample);
    const size_t o_jpart = take(sizeof(unsigned long long) * h->jobs_cap * h->nseg_sample * SAMPLE_PARTS);
    const size_t o_jt = take(sizeof(unsigned) * h->jobs_cap);
    const size_t o_err = take(sizeof(unsigned));
    const size_t o_sd = take(sizeof(unsigned) * cfg->max_batch);
    const size_t o_xf = take(sizeof(unsigned));
    const bool lmhead = cfg->target_kind == SPEC_TARGET_HIDDEN_LMHEAD;
    const size_t o_logits =
        lmhead ? take(sizeof(float) * (size_t)cfg->max_batch * (cfg->max_k + 1) * (size_t)V) : 0;
    if (base) {
        char* b = (char*)base;
        h->ws = base;
        h->seg = (SegStat*)(b + o_seg);
        h->chunk = (uint16_t*)(b + o_chunk);
        h->rstat = (RowStat*)(b + o_rstat);
        h->kept_id = (int32_t*)(b + o_kid);
        h->kept_l = (float*)(b + o_kl);
        h->row_ticket = (unsigned*)(b + o_rt);
        h->seq_ticket = (unsigned*)(b + o_st);
        h->jobs = (Job*)(b + o_jobs);
        h->job_seg = (unsigned long long*)(b + o_jseg);
        h->job_part = (unsigned long long*)(b + o_jpart);
        h->job_ticket = (unsigned*)(b + o_jt);
        h->err = (unsigned*)(b + o_err);
        h->seq_done = (unsigned*)(b + o_sd);
        h->exit_flag = (unsigned*)(b + o_xf);
        h->logits = lmhead ? (float*)(b + o_logits) : nullptr;
    }
    return off;
}

// stage 1: stream every row (the persistent bulk-copy kernel when every row
// starts on a 16-byte boundary, else one CTA per segment); then merge the rows
// (one warp per row when the knobs allow, else one CTA per row) and decide the
// sequences, each grid a programmatic dependent launch of the one before
cudaError_t launch_stage1(spec_verify* h, Params& p, int dtype, bool vec, cudaStream_t s, int* launches,
                          bool timed = true)
{
    const bool rec = timed && h->prof_begin;
    if (rec && cudaEventRecord(h->prof_begin, s) != cudaSuccess) return cudaErrorUnknown;
    cudaError_t e = vec ? launch_rows_stream(p, dtype, STREAM_CTAS_PER_SM * h->num_sms, s)
                        : launch_rows(p, dtype, false, s);
    if (e != cudaSuccess) return e;
    if (rec && cudaEventRecord(h->prof_end, s) != cudaSuccess) return cudaErrorUnknown;
    // the merge grid, then (warp and top-k merges) the decision grid
    *launches += warp_merge_ok(p) ? 3 : 2;
    if (p.cand) return launch_merge_topk(p, dtype, s);
    return warp_merge_ok(p) ? launch_merge_warp(p, dtype, s) : launch_merge(p, dtype, s);
}

// the per-row merge keeps the kept set as an explicit list whenever top-k
// bounds it by KCAP; otherwise some target rows may need the stage-2 sampler
bool all_lists(const Params& p) { return p.top_k > 0 && p.top_k <= KCAP; }

void choose_seg_mode(Params& p, int dtype)
{
    p.nseg = (int)cdiv(p.V, seg_elems(dtype));
    p.nchunk = (int)cdiv(p.V, chunk_elems(dtype));
    const bool fast = p.top_k > 0 && p.top_k <= KCAP && p.top_k <= p.nchunk &&
                      p.nchunk <= MAX_CHUNKS;
    p.seg_mode = fast ? SEG_CHUNK : SEG_SUM;
}

// bf16 rows with top-p alone, streamed by the bulk-copy kernel: per-segment
// key histograms, from which the row merge cuts the nucleus without reading
// the row again
void use_key_histograms(Params& p, int dtype, bool vec)
{
    if (vec && dtype == SPEC_BF16 && p.seg_mode == SEG_SUM && p.top_k == 0 && p.top_p < 1.f && !p.greedy)
        p.seg_mode = SEG_HIST;
}

}  // namespace

extern "C" {

const char* spec_verify_status_string(spec_status s)
{
    switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported request";
    case SPEC_ERR_OOM: return "out of device memory";
    case SPEC_ERR_CUDA: return "CUDA error";
    case SPEC_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

spec_status spec_verify_create(const spec_verify_config* cfg, spec_verify_t* out)
{
    if (!out) return SPEC_ERR_INVALID_ARG;
    *out = nullptr;
    if (!cfg) return SPEC_ERR_INVALID_ARG;
    if (cfg->max_batch < 1 || cfg->max_k < 0 || cfg->vocab < 1 || cfg->device < 0)
        return SPEC_ERR_INVALID_ARG;
    if (cfg->target_dtype != SPEC_F32 && cfg->target_dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (cfg->draft_kind == SPEC_DRAFT_LOGITS) {
        if (cfg->draft_dtype != cfg->target_dtype) return SPEC_ERR_INVALID_ARG;
    } else if (cfg->draft_kind == SPEC_DRAFT_PROBS) {
        if (cfg->draft_dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
    } else {
        return SPEC_ERR_INVALID_ARG;
    }
    if (cfg->max_k > 255) return SPEC_ERR_UNSUPPORTED;  // a decision stages 2*K_max+1 rows
    if (cfg->target_kind == SPEC_TARGET_HIDDEN_LMHEAD) {
        // bf16 hidden states and W_vocab, fp32 draft probabilities; the tensor
        // maps want row strides on 16 bytes
        if (cfg->hidden < 1 || cfg->target_dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
        if (cfg->draft_kind != SPEC_DRAFT_PROBS || cfg->hidden % 8 || cfg->vocab % 8)
            return SPEC_ERR_UNSUPPORTED;
    } else if (cfg->target_kind != SPEC_TARGET_LOGITS) {
        return SPEC_ERR_INVALID_ARG;
    }
    // the stage-2 sampler scans at most NT segments per row
    if ((int64_t)cfg->vocab > (int64_t)NT * SAMPLE_SEG) return SPEC_ERR_UNSUPPORTED;
    if ((int64_t)cfg->max_batch * (2 * (int64_t)cfg->max_k + 1) > (int64_t)INT32_MAX / 4)
        return SPEC_ERR_INVALID_ARG;

    DeviceGuard g(cfg->device);
    if (!g.ok) return SPEC_ERR_CUDA;

    spec_verify* h = new (std::nothrow) spec_verify();
    if (!h) return SPEC_ERR_OOM;
    h->cfg = *cfg;
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, cfg->device) !=
        cudaSuccess) {
        delete h;
        return SPEC_ERR_CUDA;
    }
    layout_workspace(h, nullptr);
    // stage-1 work items (row slot, segment) are counted in 32-bit ints
    if (h->rows_cap * h->nseg_cap >= (int64_t)INT32_MAX) {
        delete h;
        return SPEC_ERR_INVALID_ARG;
    }
    h->ws_bytes = layout_workspace(h, nullptr);
    {
        AllocHook& hook = alloc_hook();
        std::lock_guard<std::mutex> lock(hook.mu);
        h->alloc_fn = hook.alloc;
        h->release_fn = hook.release;
        h->alloc_ctx = hook.ctx;
    }
    void* base = nullptr;
    if (h->alloc_fn) {
        if (h->alloc_fn(h->alloc_ctx, (uint64_t)h->ws_bytes, cfg->device, &base) != 0 || !base) {
            delete h;
            return SPEC_ERR_OOM;
        }
        if ((uintptr_t)base & 255u) {  // the sub-buffers need 256-byte alignment
            h->release_fn(h->alloc_ctx, base, cfg->device);
            delete h;
            return SPEC_ERR_INVALID_ARG;
        }
    } else if (cudaMalloc(&base, h->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return SPEC_ERR_OOM;
    }
    if (cudaMemset(base, 0, h->ws_bytes) != cudaSuccess) {
        if (h->alloc_fn) h->release_fn(h->alloc_ctx, base, cfg->device);
        else cudaFree(base);
        delete h;
        return SPEC_ERR_CUDA;
    }
    layout_workspace(h, base);
    *out = h;
    return SPEC_OK;
}

namespace {
spec_status run_verify(spec_verify_t h, const spec_verify_inputs* in, const spec_sampling* s,
                       const spec_verify_outputs* out, void* stream, bool early_exit)
{
    if (!h || !in || !s || !out) return SPEC_ERR_INVALID_ARG;
    const spec_verify_config& cfg = h->cfg;
    if (in->batch < 0 || in->batch > cfg.max_batch || in->k_max < 0 || in->k_max > cfg.max_k)
        return SPEC_ERR_INVALID_ARG;
    Params p;
    memset(&p, 0, sizeof p);
    spec_status st = fill_knobs(h, s, p);
    if (st != SPEC_OK) return st;
    if (in->batch == 0) return SPEC_OK;
    if (!in->target || (!in->draft && !p.greedy) || !out->tokens || !out->num_accepted)
        return SPEC_ERR_INVALID_ARG;
    if (in->k_max > 0 && !in->draft_tokens) return SPEC_ERR_INVALID_ARG;
    const bool lmhead = cfg.target_kind == SPEC_TARGET_HIDDEN_LMHEAD;
    const int m_rows = in->batch * (in->k_max + 1);  // verified positions (LM-head rows)
    if (lmhead && (!in->w_vocab || !lmhead_shape_ok(in->target, in->w_vocab, m_rows, cfg.vocab, cfg.hidden)))
        return SPEC_ERR_INVALID_ARG;

    p.B = in->batch;
    p.Kmax = in->k_max;
    p.V = cfg.vocab;
    p.rps = 2 * in->k_max + 1;
    p.draft_launch = 0;
    p.draft_kind = cfg.draft_kind;
    // with the LM head the verify reads the fp32 logits it writes to the workspace
    p.target = lmhead ? (const void*)h->logits : in->target;
    p.draft = in->draft;
    p.xin = in->draft_tokens;
    p.kpr = in->k_per_row;
    p.tokens = out->tokens;
    p.num_accepted = out->num_accepted;
    p.row_status = out->row_status;
    p.p_t_at = out->p_t_at_draft;
    p.p_d_at = out->p_d_at_draft;
    p.resid_mass = out->residual_mass;
    p.lse = out->target_lse;
    p.alpha = out->alpha;
    p.probs_out = nullptr;
    fill_workspace(h, p);
    const int dtype = lmhead ? SPEC_F32 : cfg.target_dtype;
    choose_seg_mode(p, dtype);
    const bool vec = ((int64_t)p.V * elem_size(dtype)) % 16 == 0 && aligned16(p.target) &&
                     (cfg.draft_kind == SPEC_DRAFT_PROBS || aligned16(in->draft));
    use_key_histograms(p, dtype, vec);
    // top-k rows: the chunks reaching the row's bound gathered by one CTA per row
    p.cand = vec && p.seg_mode == SEG_CHUNK && warp_merge_ok(p) && p.top_k >= 1 &&
             p.top_k <= CAND_TOPK_MAX;

    DeviceGuard g(cfg.device);
    if (!g.ok) return SPEC_ERR_CUDA;
    cudaStream_t cs = (cudaStream_t)stream;
    int launches = 0;
    if (h->fault == SPEC_FAULT_STALL_STREAM) {
        // the stream kernel alone, its producer idle: the consumers' waits run out
        if (!vec || lmhead) return SPEC_ERR_UNSUPPORTED;
        h->fault = SPEC_FAULT_NONE;
        p.stall = 1;
        p.wait_limit = STALL_WAIT_POLLS;
        if (launch_rows_stream(p, dtype, STREAM_CTAS_PER_SM * h->num_sms, cs) != cudaSuccess)
            return SPEC_ERR_CUDA;
        if (h->prof_launches) *h->prof_launches = 1;
        return SPEC_OK;
    }
    // rows without top-k / top-p after the LM head: its epilogue writes the
    // softmax partials per 256-column tile and no stream pass is needed
    const bool lm_stats = lmhead && p.seg_mode == SEG_SUM && warp_merge_ok(p);
    if (lmhead) {
        // the hook times the LM head, the kernel that reads W_vocab
        if (h->prof_begin && cudaEventRecord(h->prof_begin, cs) != cudaSuccess) return SPEC_ERR_CUDA;
        LmStats st{nullptr, 0, 1, 1, 0.f};
        if (lm_stats) {
            p.nseg = (int)cdiv(p.V, LM_STAT_COLS);
            st = LmStats{h->seg, p.nseg, in->k_max + 1, p.rps, p.c};
        }
        if (launch_lmhead(in->target, in->w_vocab, h->logits, m_rows, cfg.vocab, cfg.hidden, cfg.vocab,
                          h->err, cs, st) != cudaSuccess)
            return SPEC_ERR_CUDA;
        if (h->prof_end && cudaEventRecord(h->prof_end, cs) != cudaSuccess) return SPEC_ERR_CUDA;
        ++launches;
    }
    // early exit (top-k rows of logits): one kernel walks each sequence's
    // positions and stops at the first rejection; the regular pipeline after
    // it returns at once unless that kernel raised the flag
    const bool exit = early_exit && p.cand && !lmhead;
    if (exit) {
        p.exit_flag = h->exit_flag;
        if (cudaMemsetAsync(h->exit_flag, 0, sizeof(unsigned), cs) != cudaSuccess) return SPEC_ERR_CUDA;
        if (h->prof_begin && cudaEventRecord(h->prof_begin, cs) != cudaSuccess) return SPEC_ERR_CUDA;
        if (launch_verify_exit(p, dtype, h->num_sms, cs) != cudaSuccess) return SPEC_ERR_CUDA;
        if (h->prof_end && cudaEventRecord(h->prof_end, cs) != cudaSuccess) return SPEC_ERR_CUDA;
        ++launches;
    }
    if (lm_stats) {
        // the row merge (softmax partials of the LM head) and the decision grid
        launches += 2;
        if (launch_merge_warp(p, dtype, cs) != cudaSuccess) return SPEC_ERR_CUDA;
    } else if (launch_stage1(h, p, dtype, vec, cs, &launches, !lmhead && !exit) != cudaSuccess) {
        return SPEC_ERR_CUDA;
    }
    if (!all_lists(p) && launch_sample(p, dtype, p.B, cs, &launches) != cudaSuccess) return SPEC_ERR_CUDA;
    if (p.alpha) {
        if (launch_alpha(p, dtype, cs) != cudaSuccess) return SPEC_ERR_CUDA;
        ++launches;
    }
    if (h->prof_launches) *h->prof_launches = launches;
    return SPEC_OK;
}
}  // namespace

spec_status spec_verify_run(spec_verify_t h, const spec_verify_inputs* in, const spec_sampling* s,
                            const spec_verify_outputs* out, void* stream)
{
    return run_verify(h, in, s, out, stream, false);
}

spec_status spec_verify_run_early_exit(spec_verify_t h, const spec_verify_inputs* in, const spec_sampling* s,
                                       const spec_verify_outputs* out, void* stream)
{
    return run_verify(h, in, s, out, stream, true);
}

spec_status spec_draft_sample(spec_verify_t h, const void* draft, const int32_t* k_per_row,
                              int32_t batch, int32_t k_max, const spec_sampling* s,
                              int32_t* draft_tokens, float* draft_probs, void* stream)
{
    if (!h || !s) return SPEC_ERR_INVALID_ARG;
    const spec_verify_config& cfg = h->cfg;
    if (batch < 0 || batch > cfg.max_batch || k_max < 0 || k_max > cfg.max_k)
        return SPEC_ERR_INVALID_ARG;
    if (cfg.draft_kind != SPEC_DRAFT_LOGITS) return SPEC_ERR_UNSUPPORTED;
    Params p;
    memset(&p, 0, sizeof p);
    spec_status st = fill_knobs(h, s, p);
    if (st != SPEC_OK) return st;
    if (batch == 0 || k_max == 0) return SPEC_OK;
    if (!draft || !draft_tokens) return SPEC_ERR_INVALID_ARG;
    p.B = batch;
    p.Kmax = k_max;
    p.V = cfg.vocab;
    p.rps = k_max;
    p.draft_launch = 1;
    p.draft_kind = 0;
    p.greedy = 0;  // temperature 0 samples the argmax through the top-1 list
    p.target = nullptr;
    p.draft = draft;
    p.kpr = k_per_row;
    p.tokens = draft_tokens;
    p.probs_out = draft_probs;
    fill_workspace(h, p);
    const int dtype = cfg.draft_dtype;
    choose_seg_mode(p, dtype);
    const bool vec = ((int64_t)p.V * elem_size(dtype)) % 16 == 0 && aligned16(draft);
    use_key_histograms(p, dtype, vec);

    DeviceGuard g(cfg.device);
    if (!g.ok) return SPEC_ERR_CUDA;
    cudaStream_t cs = (cudaStream_t)stream;
    int launches = 0;
    if (launch_stage1(h, p, dtype, vec, cs, &launches) != cudaSuccess) return SPEC_ERR_CUDA;
    if (!all_lists(p) && launch_sample(p, dtype, p.B * p.Kmax, cs) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (draft_probs && launch_probs(p, dtype, cs) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}

spec_status spec_lmhead_logits(const void* hidden, const void* w_vocab, int32_t m, int32_t hidden_dim,
                               int32_t vocab, float* logits, void* stream)
{
    if (!hidden || !w_vocab || !logits || m < 0 || hidden_dim < 1 || vocab < 1) return SPEC_ERR_INVALID_ARG;
    if (m == 0) return SPEC_OK;
    if (!lmhead_shape_ok(hidden, w_vocab, m, vocab, hidden_dim) || ((uintptr_t)logits & 15u))
        return SPEC_ERR_UNSUPPORTED;
    if (launch_lmhead(hidden, w_vocab, logits, m, vocab, hidden_dim, vocab, nullptr, (cudaStream_t)stream) !=
        cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

spec_status spec_verify_set_profiling(spec_verify_t h, void* ev_stage1_begin, void* ev_stage1_end,
                                      int32_t* launches_out)
{
    if (!h || (!ev_stage1_begin) != (!ev_stage1_end)) return SPEC_ERR_INVALID_ARG;
    h->prof_begin = (cudaEvent_t)ev_stage1_begin;
    h->prof_end = (cudaEvent_t)ev_stage1_end;
    h->prof_launches = launches_out;
    return SPEC_OK;
}

spec_status spec_verify_check(spec_verify_t h, void* stream)
{
    if (!h) return SPEC_ERR_INVALID_ARG;
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return SPEC_ERR_CUDA;
    cudaStream_t cs = (cudaStream_t)stream;
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, h->err, sizeof word, cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
        cudaStreamSynchronize(cs) != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    if (word == 0) return SPEC_OK;
    // a run that gave up may leave tickets and chunk keys behind: clear them
    if (cudaMemsetAsync(h->err, 0, sizeof(unsigned), cs) != cudaSuccess ||
        cudaMemsetAsync(h->row_ticket, 0, sizeof(unsigned) * (size_t)h->rows_cap, cs) != cudaSuccess ||
        cudaMemsetAsync(h->seq_ticket, 0, sizeof(unsigned) * (size_t)h->cfg.max_batch, cs) != cudaSuccess ||
        cudaMemsetAsync(h->seq_done, 0, sizeof(unsigned) * (size_t)h->cfg.max_batch, cs) != cudaSuccess ||
        cudaMemsetAsync(h->job_ticket, 0, sizeof(unsigned) * (size_t)h->jobs_cap, cs) != cudaSuccess ||
        cudaStreamSynchronize(cs) != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    return SPEC_ERR_TIMEOUT;
}

spec_status spec_verify_inject_fault(spec_verify_t h, int32_t fault)
{
    if (!h || (fault != SPEC_FAULT_NONE && fault != SPEC_FAULT_STALL_STREAM)) return SPEC_ERR_INVALID_ARG;
    h->fault = fault;
    return SPEC_OK;
}

spec_status spec_verify_set_allocator(spec_alloc_fn alloc, spec_release_fn release, void* ctx)
{
    if ((!alloc) != (!release)) return SPEC_ERR_INVALID_ARG;
    AllocHook& hook = alloc_hook();
    std::lock_guard<std::mutex> lock(hook.mu);
    hook.alloc = alloc;
    hook.release = release;
    hook.ctx = alloc ? ctx : nullptr;
    return SPEC_OK;
}

spec_status spec_verify_destroy(spec_verify_t h)
{
    if (!h) return SPEC_ERR_INVALID_ARG;
    spec_status st = SPEC_OK;
    {
        DeviceGuard g(h->cfg.device);
        if (!g.ok) st = SPEC_ERR_CUDA;
        if (h->ws && h->release_fn) {
            if (cudaDeviceSynchronize() != cudaSuccess) st = SPEC_ERR_CUDA;
            h->release_fn(h->alloc_ctx, h->ws, h->cfg.device);
        } else if (h->ws && cudaFree(h->ws) != cudaSuccess) {
            st = SPEC_ERR_CUDA;
        }
    }
    delete h;
    return st;
}

}  // extern "C"

// ------------------------------------------------------------------------- //
// Workspace laid over caller-provided device memory (used by the entry point  //
// that allocates nothing, sv_noalloc.cu).  Same layout rules as create.       //
// ------------------------------------------------------------------------- //
namespace {

// fills h (workspace pointers into ws, when ws is not NULL) for a run of
// `batch` x `k_max`; returns the bytes needed, or 0 for invalid arguments
size_t layout_over(spec_verify* h, const spec_verify_config* cfg, int32_t batch, int32_t k_max,
                   void* ws, size_t ws_bytes)
{
    if (!cfg || batch < 0 || k_max < 0 || k_max > 255 || cfg->vocab < 1) return 0;
    if (cfg->target_dtype != SPEC_F32 && cfg->target_dtype != SPEC_BF16) return 0;
    if (cfg->draft_kind == SPEC_DRAFT_LOGITS) {
        if (cfg->draft_dtype != cfg->target_dtype) return 0;
    } else if (cfg->draft_kind == SPEC_DRAFT_PROBS) {
        if (cfg->draft_dtype != SPEC_F32) return 0;
    } else {
        return 0;
    }
    if (cfg->target_kind != SPEC_TARGET_LOGITS) return 0;
    if ((int64_t)cfg->vocab > (int64_t)NT * SAMPLE_SEG) return 0;
    const int64_t mb = batch > 0 ? batch : 1;
    h->cfg = *cfg;
    h->cfg.max_batch = (int32_t)mb;
    h->cfg.max_k = k_max;
    const size_t need = layout_workspace(h, nullptr);
    if (h->rows_cap * h->nseg_cap >= (int64_t)INT32_MAX) return 0;
    if (ws) layout_workspace(h, ws);
    return need;
}

}  // namespace

// bytes of workspace a run of these sizes needs (0: invalid arguments)
size_t sv_noalloc_bytes(const spec_verify_config* cfg, int32_t batch, int32_t k_max)
{
    spec_verify h{};  // value-initialised: no profiling hook, no pointers
    return layout_over(&h, cfg, batch, k_max, nullptr, 0);
}

// spec_verify_run over a workspace the caller provides (ws_bytes of device
// memory on cfg->device, which must be current); allocates nothing
spec_status sv_noalloc_run(void* ws, size_t ws_bytes, int num_sms, const spec_verify_config* cfg,
                           const spec_verify_inputs* in, const spec_sampling* s,
                           const spec_verify_outputs* out, void* stream)
{
    if (!ws || !in) return SPEC_ERR_INVALID_ARG;
    spec_verify h{};  // value-initialised: no profiling hook, no pointers
    const size_t need = layout_over(&h, cfg, in->batch, in->k_max, ws, ws_bytes);
    if (need == 0 || need > ws_bytes) return SPEC_ERR_INVALID_ARG;
    h.num_sms = num_sms;
    // the counters the kernels expect at zero (the array keeps the last call's contents)
    cudaStream_t cs = (cudaStream_t)stream;
    const size_t tickets = sizeof(unsigned) * (size_t)h.rows_cap;
    if (cudaMemsetAsync(h.row_ticket, 0, tickets, cs) != cudaSuccess ||
        cudaMemsetAsync(h.seq_ticket, 0, sizeof(unsigned) * (size_t)h.cfg.max_batch, cs) != cudaSuccess ||
        cudaMemsetAsync(h.job_ticket, 0, sizeof(unsigned) * (size_t)h.jobs_cap, cs) != cudaSuccess ||
        cudaMemsetAsync(h.err, 0, sizeof(unsigned), cs) != cudaSuccess ||
        cudaMemsetAsync(h.seq_done, 0, sizeof(unsigned) * (size_t)h.cfg.max_batch, cs) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return spec_verify_run(&h, in, s, out, stream);
}
