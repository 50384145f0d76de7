// sv_exit.cuh -- the early-exit verify of the top-k rows (included by
// sv_rows.cu after the row merge).
//
// The drafts of a sequence are checked left to right and the ones after the
// first rejection are discarded ("Accelerating Large Language Model Decoding
// with Speculative Sampling", The algorithm), so only the rows up to the
// first rejection matter: this kernel reads no others.  Each CTA owns whole
// sequences (b = blockIdx.x, + gridDim.x, ...) and walks their positions in
// order.  For position j one producer thread streams target row j and draft
// row j (bulk copies into the NSTAGE ring), the compute threads write their
// chunk keys and merge each row (merge_row_topk_core), and warp 0 takes the
// decision of position j: accept and go on, or stop with the residual sample
// (or the bonus sample at j = K_b).  The producer waits for that verdict
// before it reads the next position's rows.
//
// The tokens, accepted lengths and statuses are those of the full verify,
// with one difference: a non-finite logit in a row after the first rejection
// is not seen.  p_t / p_d at the drafted tokens and the target log-sum-exp
// are written for the positions read (NaN beyond); alpha is not computed
// (NaN).  A row whose candidates overflow the CTA's staging (ties) sets
// *p.exit_flag, and the regular pipeline that follows on the stream (which
// otherwise returns at once) recomputes every sequence.
#pragma once

namespace sv {

constexpr int EXIT_CTAS_PER_SM = 3;

// verdicts of the compute warps to the producer
enum : int { EXIT_GO = 1, EXIT_STOP = 0 };

// the outputs of a sequence that stops at position jstar with token tok
__device__ __forceinline__ void exit_emit(const Params& p, int b, int kb, int jstar, int tok, int status,
                                          float resid)
{
    const int K = p.Kmax, lane = threadIdx.x & 31;
    for (int j = lane; j <= K; j += 32) {
        int32_t v = -1;
        if (j < jstar) v = p.xin[(int64_t)b * K + j];
        else if (j == jstar) v = tok;
        p.tokens[(int64_t)b * (K + 1) + j] = v;
    }
    if (p.alpha)
        for (int j = lane; j < K; j += 32) p.alpha[(int64_t)b * K + j] = NAN;
    if (lane == 0) {
        p.num_accepted[b] = jstar;
        if (p.row_status) p.row_status[b] = status;
        if (p.resid_mass) p.resid_mass[b] = resid;
    }
}

// a sequence refused as a whole: every output -1 / NaN
__device__ __forceinline__ void exit_refuse(const Params& p, int b, int status)
{
    const int K = p.Kmax, lane = threadIdx.x & 31;
    for (int j = lane; j <= K; j += 32) {
        p.tokens[(int64_t)b * (K + 1) + j] = -1;
        if (p.lse) p.lse[(int64_t)b * (K + 1) + j] = NAN;
        if (j < K) {
            if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = NAN;
            if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = NAN;
            if (p.alpha) p.alpha[(int64_t)b * K + j] = NAN;
        }
    }
    if (lane == 0) {
        p.num_accepted[b] = -1;
        if (p.row_status) p.row_status[b] = status;
        if (p.resid_mass) p.resid_mass[b] = NAN;
    }
}

// warp 0: the decision of position j of sequence b from the merged records
// ts (target row j) and ds (draft row j, logits); EXIT_GO or EXIT_STOP
template <typename T>
__device__ int exit_decide(const Params& p, int b, int kb, int j, const RowStat& ts, const RowStat& ds,
                           unsigned char* stage)
{
    const int K = p.Kmax, V = p.V, lane = threadIdx.x & 31;
    const int64_t drow0 = (int64_t)b * K * V;
    const uint4 w = slot_words(p, b, j, 0u);
    if (lane == 0 && p.lse)
        p.lse[(int64_t)b * (K + 1) + j] = p.greedy ? NAN : ts.M / p.T + logf((float)ts.S);
    bool residual = false;
    if (j < kb) {
        const int x = p.xin[(int64_t)b * K + j];
        const float pt = ts.px;
        float pd = NAN;
        if (!p.greedy) pd = p.draft_kind == 1 ? __ldcg((const float*)p.draft + drow0 + (int64_t)j * V + x) : ds.px;
        if (p.draft_kind == 1 && !p.greedy && (!(pd >= 0.f) || pd == INFINITY)) {
            exit_refuse(p, b, ROW_NONFINITE);
            return EXIT_STOP;
        }
        if (lane == 0) {
            if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = pt;
            if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = pd;
        }
        // the same tests as the full verify (sv_warp.cuh)
        const bool rej = p.greedy ? !(pt > 0.f) : !(u24(w.x) < __fdiv_rn(pt, pd));
        if (!rej) return EXIT_GO;
        residual = !p.greedy;
    }
    // stop at j: the residual sample (or the bonus / greedy argmax); the
    // positions after j are not read
    for (int i = j + 1 + lane; i <= K; i += 32)
        if (p.lse) p.lse[(int64_t)b * (K + 1) + i] = NAN;
    for (int i = (j < kb ? j + 1 : kb) + lane; i < K; i += 32) {
        if (p.p_t_at) p.p_t_at[(int64_t)b * K + i] = NAN;
        if (p.p_d_at) p.p_d_at[(int64_t)b * K + i] = NAN;
    }
    DraftRef d;
    d.kind = p.draft_kind;
    d.r = residual ? draft_slot(p, b, j) : -1;
    if (residual && d.kind == 0) d.st = ds;
    d.row = residual ? (const void*)((const char*)p.draft +
                                     (drow0 + (int64_t)j * V) * (d.kind == 1 ? 4 : (int64_t)sizeof(T)))
                     : nullptr;
    unsigned long long Z;
    bool zero;
    const int tok = warp_sample_list<T>(p, target_slot(p, b, j), ts, residual, d, u24(w.y), stage, &Z, &zero);
    exit_emit(p, b, kb, j, tok, zero ? ROW_ZERO_RESIDUAL : ROW_OK, residual ? (float)from_fix56(Z) : 0.f);
    return EXIT_STOP;
}

template <typename T>
__global__ void __launch_bounds__(STREAM_THREADS, EXIT_CTAS_PER_SM) k_verify_exit(const Params p)
{
    extern __shared__ __align__(128) unsigned char smem_ring[];  // NSTAGE x SEG_BYTES
    __shared__ Ring ring;
    __shared__ __align__(8) uint64_t go;   // a verdict of the compute warps is ready
    __shared__ __align__(8) uint64_t ack;  // the producer has read it
    __shared__ McSmem sm;
    __shared__ float s_redf[NS / 32 + 1];
    __shared__ double s_redd[NS / 32 + 1];
    __shared__ int s_verdict;
    __shared__ int s_fail;  // a compute thread's bounded wait ran out (read after barriers only)
    __shared__ RowStat s_st[2];
    using G = SegGeom<T, NS>;
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&ring.full[s], 1);
            mbar_init(&ring.empty[s], 1);
        }
        mbar_init(&go, 1);
        mbar_init(&ack, 1);
        s_fail = 0;
        fence_barrier_init();
    }
    __syncthreads();  // the only barrier over all STREAM_THREADS threads
    const int64_t row_bytes = (int64_t)p.V * (int64_t)sizeof(T);
    const bool drafts = drafts_streamed(p);

    if (tid >= NS) {
        // ---------------- producer: the rows of each position, then the verdict
        if (tid != NS) return;
        int k = 0, nv = 0;  // copies issued, verdicts read
        bool failed = false;
        for (int b = blockIdx.x; b < p.B && !failed; b += gridDim.x) {
            const int kb = seq_k(p, b);
            // position -1 always (its verdict exists for every sequence)
            for (int j = -1; !failed && (j < 0 || j <= kb); ++j) {
                // position -1: the sequence check; then the rows of position j
                if (j >= 0) {
                    const int nr = (drafts && j < kb) ? 2 : 1;
                    for (int q = 0; q < nr && !failed; ++q) {
                        const int r = q == 0 ? target_slot(p, b, j) : draft_slot(p, b, j);
                        const RowRef rr = row_ref(p, r);
                        const char* rb = (const char*)(rr.is_draft ? p.draft : p.target) +
                                         row_elem_offset(p, rr) * (int64_t)sizeof(T);
                        for (int seg = 0; seg < p.nseg; ++seg, ++k) {
                            const int s = k % NSTAGE;
                            if (k >= NSTAGE && !mbar_wait(&ring.empty[s], ((k / NSTAGE) - 1) & 1)) {
                                failed = true;
                                break;
                            }
                            const uint32_t bytes =
                                (uint32_t)min((int64_t)SEG_BYTES, row_bytes - (int64_t)seg * SEG_BYTES);
                            mbar_arrive_expect_tx(&ring.full[s], bytes);
                            tma_load_1d(smem_ring + (size_t)s * SEG_BYTES, rb + (int64_t)seg * SEG_BYTES, bytes,
                                        &ring.full[s]);
                        }
                    }
                }
                if (failed || !mbar_wait(&go, nv & 1)) {
                    failed = true;
                    break;
                }
                ++nv;
                const int v = *(volatile int*)&s_verdict;
                mbar_arrive(&ack);  // the compute warps may post the next verdict
                if (v != EXIT_GO) break;
            }
        }
        if (failed) {
            atomicOr(p.err, 1u);
            for (int q = (k > NSTAGE ? k - NSTAGE : 0); q < k; ++q)
                mbar_wait(&ring.full[q % NSTAGE], (q / NSTAGE) & 1);
        }
        return;
    }

    // ---------------- compute threads
    const int warp = tid >> 5;
    int k = 0;        // segments consumed
    int nposted = 0;  // verdicts posted (thread 0)
    bool failed = false;
    auto verdict = [&](int v) {
        if (tid == 0) {
            // the previous verdict has been read before this one replaces it
            if (nposted > 0 && !mbar_wait(&ack, (nposted - 1) & 1)) atomicOr(p.err, 2u);
            s_verdict = v;
            mbar_arrive(&go);  // release: the producer reads the verdict after its wait
            ++nposted;
        }
    };
    for (int b = blockIdx.x; b < p.B && !failed; b += gridDim.x) {
        const int kb = seq_k(p, b);
        // position -1: K_b and the drafted tokens
        if (!k_ok(p, kb)) {
            if (tid == 0) report_skipped_row(p, row_ref(p, target_slot(p, b, 0)));
            ssync();
            verdict(EXIT_STOP);
            continue;
        }
        bool bad = false;
        for (int j = tid; j < kb; j += NS) {
            const int x = p.xin[(int64_t)b * p.Kmax + j];
            bad |= x < 0 || x >= p.V;
        }
        if (tid == 0) sm.flag = 0;
        ssync();
        if (bad) sm.flag = 1;
        ssync();
        if (sm.flag) {
            if (warp == 0) exit_refuse(p, b, ROW_BAD_TOKEN);
            ssync();
            verdict(EXIT_STOP);
            continue;
        }
        ssync();  // every thread has read sm.flag
        verdict(EXIT_GO);
        for (int j = 0; j <= kb; ++j) {
            const int nr = (drafts && j < kb) ? 2 : 1;
            for (int q = 0; q < nr; ++q) {
                const int r = q == 0 ? target_slot(p, b, j) : draft_slot(p, b, j);
                for (int seg = 0; seg < p.nseg; ++seg, ++k) {
                    const int s = k % NSTAGE;
                    // every thread takes the same branches: `failed` changes
                    // only from the shared flag, read after a barrier
                    if (!failed && !mbar_wait(&ring.full[s], (k / NSTAGE) & 1)) s_fail = 1;
                    if (!failed) {
                        const uint4* sv4 = reinterpret_cast<const uint4*>(smem_ring + (size_t)s * SEG_BYTES);
                        const int64_t base = (int64_t)seg * G::SEG;
                        segment_compute<T, SEG_CHUNK, NS>(
                            p,
                            [&](int i) {
                                const int64_t e0 = base + ((int64_t)i * NS + tid) * G::VW;
                                return e0 < p.V ? sv4[i * NS + tid] : Vec16<T>::neg_inf();
                            },
                            seg, r, tid, [] { ssync(); }, s_redf, s_redd);
                    }
                    ssync();  // every compute thread is done with the stage
                    // s_fail only ever goes from 0 to 1, so every thread reads
                    // the same value after the barrier
                    failed = *(volatile int*)&s_fail != 0;
                    if (tid == 0 && !failed) mbar_arrive(&ring.empty[s]);
                }
                // the row's chunk keys are written by this CTA: merge it
                __threadfence_block();
                ssync();
                const RowStat st = merge_row_topk_core<T>(p, r, sm);
                if (tid == 0) s_st[q] = st;
                ssync();
            }
            const RowStat ts = s_st[0];
            const RowStat ds = nr == 2 ? s_st[1] : s_st[0];
            int v = EXIT_STOP;
            if (failed) {
                v = EXIT_STOP;
            } else if ((ts.flags | (nr == 2 ? ds.flags : 0)) & FLAG_BLOCK_MERGE) {
                if (tid == 0) atomicOr(p.exit_flag, 1u);  // the regular pipeline recomputes everything
            } else if ((ts.flags | (nr == 2 ? ds.flags : 0)) & FLAG_NONFINITE) {
                if (warp == 0) exit_refuse(p, b, ROW_NONFINITE);
            } else if (warp == 0) {
                v = exit_decide<T>(p, b, kb, j, ts, ds, sm.u.stage);
                if (tid == 0) sm.flag = v;
            }
            ssync();
            if (!failed && !((ts.flags | (nr == 2 ? ds.flags : 0)) & (FLAG_BLOCK_MERGE | FLAG_NONFINITE)))
                v = sm.flag;
            ssync();  // every thread has read sm.flag
            verdict(v);
            if (v != EXIT_GO) break;
        }
    }
    if (failed && tid == 0) atomicOr(p.err, 2u);
}

template <typename T>
static cudaError_t launch_verify_exit_t(const Params& p, int num_sms, cudaStream_t s)
{
    static DeviceOnce once;  // the shared-memory opt-in, per device
    const cudaError_t e = cuda_once(once, nullptr, [](int, int*) {
        return cudaFuncSetAttribute(k_verify_exit<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, STREAM_SMEM);
    });
    if (e != cudaSuccess) return e;
    const int grid = std::min(p.B, EXIT_CTAS_PER_SM * num_sms);
    if (grid <= 0) return cudaSuccess;
    k_verify_exit<T><<<grid, STREAM_THREADS, STREAM_SMEM, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_verify_exit(const Params& p, int dtype, int num_sms, cudaStream_t s)
{
    return dtype == 1 ? launch_verify_exit_t<__nv_bfloat16>(p, num_sms, s)
                      : launch_verify_exit_t<float>(p, num_sms, s);
}

}  // namespace sv
