// sv_cand.cuh -- the candidate stream kernel (included by sv_rows.cu).
//
// For rows whose kept set is bounded by top-k (k <= CAND_TOPK_MAX) the row
// merge needs only the logits that can be in the top-k.  This kernel streams
// every row once, like k_stream, and while a piece is in shared memory it also
// collects those candidates:
//
//  * Work.  Each CTA is one warp that owns a contiguous run of pieces
//    (CS_PIECE bytes of one row slot; items in row-major order).  It walks the
//    run's rows from the last to the first, each row's pieces in order, so
//    consecutive pieces of a row pass through the same warp and a row split
//    between two runs is begun by the earlier run (as its first work) and
//    finished by the later one (as its last).  Lane 0 keeps CS_STAGES pieces
//    in flight with bulk (TMA) copies completing on mbarriers; there are no
//    block barriers.
//  * Chunk maxima.  Lane l reduces chunk l of the piece (128 bytes, eight
//    16-byte words), reading its words in a rotated order so the eight lanes
//    of a quarter-warp hit distinct banks; the 16-bit chunk keys go to the
//    workspace as in k_stream (the chunk-key merge runs when a row overflows).
//  * Threshold.  tau starts as the larger of the row's published threshold
//    (other runs' bounds for the same row) and, when none is published yet,
//    the k-th largest word maximum of the row's first piece in the run.  The
//    word maxima at or above tau are counted in a histogram of their 16-bit
//    keys over the window [tau, tau + 255] (the top
//    bin counts everything above), and tau
//    rises to the histogram's k-th largest key (once 32 maxima were added
//    since the last rise, and at the row's end) and the window slides.  Each
//    counted word maximum is a logit of the row and every count sits at or
//    below its logit's key, so at least k logits are >= tau throughout.  Each
//    raise is published (atomic max) in the row's control words.
//  * Candidates.  A lane whose chunk reaches tau checks its words; the logits
//    >= tau of a word whose maximum reaches tau go (order key, token id) to
//    the lane's own staging slots.  At the row's end in the run (or when a
//    lane's slots fill) the warp appends all staged candidates to the row's
//    candidate array with one atomic; the row's control words get the largest
//    tau and chunk key.
#pragma once

namespace sv {

constexpr int CS_STAGES = 4;
constexpr int CS_WARPS_PER_SM = 7;  // warps (CTAs) of the grid per SM
constexpr int CS_MIN_RUN = 16;      // fewest pieces per warp
constexpr int CS_SMEM = CS_STAGES * CS_PIECE;
constexpr int CS_WORDS = CS_PIECE / 16;             // 16-byte words per piece (256)
constexpr int CS_WPL = CS_WORDS / 32;               // words per lane: one chunk (8)
constexpr int LSTG = 16;                            // staged candidates per lane
constexpr int HBINS = 256;                          // threshold histogram bins
static_assert(CS_WPL * 16 == CHUNK_BYTES, "a lane reduces one chunk of the piece");
static_assert(HBINS == 32 * 8, "a lane owns eight histogram bins");

// element q (runtime) of a 16-byte word of T
template <typename T> __device__ __forceinline__ float word_elem_rt(uint4 w, int q);
template <> __device__ __forceinline__ float word_elem_rt<__nv_bfloat16>(uint4 w, int q)
{
    const uint32_t x = (q & 4) ? ((q & 2) ? w.w : w.z) : ((q & 2) ? w.y : w.x);
    return (q & 1) ? bf16_hi(x) : bf16_lo(x);
}
template <> __device__ __forceinline__ float word_elem_rt<float>(uint4 w, int q)
{
    return __uint_as_float((q & 2) ? ((q & 1) ? w.w : w.z) : ((q & 1) ? w.y : w.x));
}

// the k-th largest of the warp's keys (each lane holds N; key 0 = absent,
// present keys are >= 1): the largest t with #(keys >= t) >= k, or 0 when
// fewer than k keys are present
template <int N>
__device__ __forceinline__ uint32_t warp_kth_key(const uint32_t (&key)[N], int k)
{
    const unsigned FULL = 0xffffffffu;
    uint32_t hi = 0, lo = 0xFFFFFFFFu;
    int present = 0;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        hi = max(hi, key[i]);
        if (key[i]) {
            lo = min(lo, key[i]);
            ++present;
        }
    }
    if (__reduce_add_sync(FULL, present) < k) return 0;
    hi = __reduce_max_sync(FULL, hi);
    lo = __reduce_min_sync(FULL, lo);
    // #(keys >= lo) >= k holds throughout
    while (lo < hi) {
        const uint32_t mid = (lo + hi + 1) >> 1;
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < N; ++i) cnt += key[i] >= mid;
        if (__reduce_add_sync(FULL, cnt) >= k) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// the smallest non-NaN value whose order key is >= tau << 16 (tau = 0: every
// value); a logit x qualifies iff x >= this (false for NaN)
__device__ __forceinline__ float key16_floor(uint32_t tau)
{
    const uint32_t K = tau << 16;
    return K <= 0x007FFFFFu ? -INFINITY : val_of(K);
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// a work item: piece pc of row slot r (r < 0: the run is done)
struct PieceCur {
    int r, pc;
};

// per-warp state of the row being streamed
struct CandRow {
    int r;           // row slot (-1: none)
    uint32_t tau;    // current threshold key (0: every logit)
    bool tau_set;    // tau computed for this row
    int hist_n;      // word maxima counted in the histogram
    bool ovf;        // candidates were lost: the row takes the chunk path
    uint32_t kmax;   // this lane's largest chunk key of the row
};

// tau = the k-th largest counted key (the histogram holds at least k), and
// the window slides up to start at the new tau
__device__ __forceinline__ void raise_tau(CandRow& cr, uint32_t* s_hist, int k)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    __syncwarp();
    uint32_t h[8];
    int local = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        h[q] = s_hist[lane * 8 + q];
        local += (int)h[q];
    }
    // above = the count in the bins of the lanes above this one
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(FULL, incl, o);
        if (lane + o < 32) incl += y;
    }
    const int above = incl - local;
    // the highest bin whose count from the top reaches k
    const unsigned hit = __ballot_sync(FULL, incl >= k);
    const int L = 31 - __clz(hit);  // hit != 0: bin 0 covers all hist_n >= k
    int b = 0, from_b = 0;
    if (lane == L) {
        int run = above;
#pragma unroll
        for (int q = 7; q >= 0; --q) {
            run += (int)h[q];
            if (run >= k) {
                b = lane * 8 + q;
                from_b = run;
                break;
            }
        }
    }
    b = __shfl_sync(FULL, b, L);
    from_b = __shfl_sync(FULL, from_b, L);
    if (b > 0) {
        uint32_t nv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int src = lane * 8 + q + b;
            nv[q] = src < HBINS ? s_hist[src] : 0u;
        }
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 8; ++q) s_hist[lane * 8 + q] = nv[q];
        cr.tau += (uint32_t)b;
        cr.hist_n = from_b;
    }
    __syncwarp();
}

// append every lane's staged candidates (nl of them in its slots) to row
// cr.r's array with one atomic
__device__ __forceinline__ void flush_stage(const Params& p, const CandRow& cr,
                                            const unsigned long long* s_stage, int& nl)
{
    const int lane = threadIdx.x & 31;
    int tot;
    const int ex = warp_excl_scan(nl, &tot);
    if (tot == 0) return;
    unsigned base = 0;
    if (lane == 0) base = atomicAdd(p.rowctl + (int64_t)cr.r * 4 + CTL_COUNT, (unsigned)tot);
    base = __shfl_sync(0xffffffffu, base, 0) + (unsigned)ex;
    unsigned long long* dst = p.cand_rows + (int64_t)cr.r * RCAP_ROW;
    for (int i = 0; i < nl; ++i)
        if (base + (unsigned)i < (unsigned)RCAP_ROW) dst[base + i] = s_stage[i * 32 + lane];
    nl = 0;
    __syncwarp();
}

template <typename T>
__global__ void __launch_bounds__(32) k_stream_cand(const Params p)
{
    extern __shared__ __align__(128) unsigned char smem_cs[];  // CS_STAGES x CS_PIECE
    __shared__ __align__(8) uint64_t full[CS_STAGES];
    __shared__ unsigned long long s_stage[LSTG * 32];  // slot i of lane l at i * 32 + l
    __shared__ uint32_t s_hist[HBINS];
    using CM = ChunkMax<T>;
    using PM = typename CM::P;
    constexpr int VW = Vec16<T>::N;
    constexpr int PE = CS_PIECE / (int)sizeof(T);  // elements per piece
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x;
    // the merge grid may be scheduled as this grid drains; it waits for this
    // grid's completion before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (lane == 0) {
        for (int s = 0; s < CS_STAGES; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    const int npc = p.npiece;
    const int64_t total = (int64_t)p.B * p.rps * npc;
    const int64_t row_bytes = (int64_t)p.V * (int64_t)sizeof(T);
    const int k = p.top_k;
    // this warp's run of items [beg, end): rows r_first..r_last, pieces
    // [first_pc, npc) of r_first and [0, last_hi) of r_last (32-bit from here)
    int r_first, first_pc, r_last, last_hi;
    {
        const int64_t beg = total * blockIdx.x / gridDim.x;
        const int64_t end = total * (blockIdx.x + 1) / gridDim.x;
        if (end <= beg) return;
        r_first = (int)(beg / npc);
        first_pc = (int)(beg - (int64_t)r_first * npc);
        r_last = (int)((end - 1) / npc);
        last_hi = (int)(end - 1 - (int64_t)r_last * npc) + 1;
    }
    auto lo_pc = [&](int r) { return r == r_first ? first_pc : 0; };
    auto hi_pc = [&](int r) { return r == r_last ? last_hi : npc; };
    auto row_streamed = [&](int r) {
        const RowRef rr = row_ref(p, r);
        return rr.valid && !(rr.is_draft && p.draft_kind == 1);
    };
    // the first streamed row at or below r, entered at its first piece in the run
    auto enter_row = [&](int r) -> PieceCur {
        while (r >= r_first && !row_streamed(r)) --r;
        return r >= r_first ? PieceCur{r, lo_pc(r)} : PieceCur{-1, 0};
    };
    // the item after c in walking order (rows descending, pieces ascending)
    auto next_item = [&](PieceCur c) -> PieceCur {
        if (c.pc + 1 < hi_pc(c.r)) return PieceCur{c.r, c.pc + 1};
        return enter_row(c.r - 1);
    };
    int iss_row = -1;
    const char* iss_base = nullptr;
    auto issue = [&](PieceCur it, int s) {
        if (it.r != iss_row) {
            const RowRef rr = row_ref(p, it.r);
            iss_row = it.r;
            iss_base = (const char*)(rr.is_draft ? p.draft : p.target) +
                       row_elem_offset(p, rr) * (int64_t)sizeof(T);
        }
        const int64_t at = (int64_t)it.pc * CS_PIECE;
        const uint32_t bytes = (uint32_t)min((int64_t)CS_PIECE, row_bytes - at);
        mbar_arrive_expect_tx(&full[s], bytes);
        tma_load_1d(smem_cs + (size_t)s * CS_PIECE, iss_base + at, bytes, &full[s]);
    };

    // prime the ring
    PieceCur cur = enter_row(r_last);
    PieceCur tail = cur;
    int issued = 0;  // copies issued so far (copy i lands in stage i % CS_STAGES)
    if (cur.r >= 0) {
        if (lane == 0) issue(cur, 0);
        issued = 1;
        while (issued < CS_STAGES) {
            const PieceCur nx = next_item(tail);
            if (nx.r < 0) break;
            if (lane == 0) issue(nx, issued);
            tail = nx;
            ++issued;
        }
    }
    // this lane's word offsets within a piece: chunk `lane`, words rotated
    uint32_t woff[CS_WPL];
#pragma unroll
    for (int v = 0; v < CS_WPL; ++v) woff[v] = (uint32_t)(lane * CS_WPL + ((v + lane) & (CS_WPL - 1)));

    CandRow cr;
    bool failed = false;
    int kk = 0;
    while (cur.r >= 0 && !failed) {
        // ---------------- a row: its pieces in this run
        const int r = cur.r;
        unsigned* ctl = p.rowctl + (int64_t)r * 4;
        cr.r = r;
        cr.tau = __ldcg(ctl + CTL_TAU);  // published by other runs of this row, or 0
        cr.tau_set = cr.tau != 0u;
        cr.hist_n = 0;
        cr.ovf = false;
        cr.kmax = 0u;
#pragma unroll
        for (int q = 0; q < 8; ++q) s_hist[lane * 8 + q] = 0u;
        __syncwarp();
        int since = 0;  // word maxima counted since tau was last raised
        int nl = 0;     // this lane's staged candidates
        for (;;) {
            const int s = kk % CS_STAGES;
            if (!mbar_wait(&full[s], (kk / CS_STAGES) & 1)) {
                failed = true;
                break;
            }
            const int pc = cur.pc;
            const int e_base = pc * PE;  // < V
            const int nvec = min(CS_WORDS, (p.V - e_base) / VW);
            const uint4* sv4 = reinterpret_cast<const uint4*>(smem_cs + (size_t)s * CS_PIECE);

            // ---- word maxima and lane's chunk max
            PM pm[CS_WPL];
            PM cm = CM::lane(Vec16<T>::neg_inf());
            if (nvec == CS_WORDS) {
#pragma unroll
                for (int v = 0; v < CS_WPL; ++v) {
                    pm[v] = CM::lane(sv4[woff[v]]);
                    cm = CM::mx(cm, pm[v]);
                }
            } else {
#pragma unroll
                for (int v = 0; v < CS_WPL; ++v) {
                    pm[v] = CM::lane((int)woff[v] < nvec ? sv4[woff[v]] : Vec16<T>::neg_inf());
                    cm = CM::mx(cm, pm[v]);
                }
            }
            const bool chunk_here = lane * CS_WPL < nvec;
            const float cmax = CM::value(cm);
            const uint32_t ck = chunk_here ? key_of(cmax) >> 16 : 0u;
            if (chunk_here) p.chunk[(int64_t)r * p.chunk_stride + pc * 32 + lane] = (uint16_t)ck;
            cr.kmax = max(cr.kmax, ck);

            // ---- no bound yet for this row: the first piece's word maxima
            if (!cr.tau_set) {
                uint32_t wk[CS_WPL];
#pragma unroll
                for (int v = 0; v < CS_WPL; ++v)
                    wk[v] = (int)woff[v] < nvec ? key_of(CM::value(pm[v])) >> 16 : 0u;
                cr.tau = warp_kth_key(wk, k);
                cr.tau_set = true;
            }
            const float tf = key16_floor(cr.tau);
            const uint32_t tf2 = CM::thr2(tf);

            // ---- candidates: only lanes whose chunk reaches tau do any work;
            //      one word per lane per round
            if (__any_sync(FULL, chunk_here && cmax >= tf)) {
                uint32_t qm = 0;
                if (chunk_here && cmax >= tf) {
#pragma unroll
                    for (int v = 0; v < CS_WPL; ++v)
                        if ((int)woff[v] < nvec && CM::any_ge(pm[v], tf, tf2)) qm |= 1u << v;
                }
                const int nq = __reduce_add_sync(FULL, __popc(qm));
                while (__any_sync(FULL, qm != 0u)) {
                    uint32_t em = 0;
                    int vi = 0;
                    uint4 w = make_uint4(0, 0, 0, 0);
                    if (qm) {
                        const int v = __ffs(qm) - 1;
                        qm &= qm - 1u;
                        vi = lane * CS_WPL + ((v + lane) & (CS_WPL - 1));
                        w = sv4[vi];
                        const uint32_t wk16 = key_of(CM::value(CM::lane(w))) >> 16;
                        atomicAdd(&s_hist[min(wk16 - cr.tau, (uint32_t)(HBINS - 1))], 1u);
                        em = CM::elem_mask(w, tf, tf2);
                    }
                    if (__any_sync(FULL, nl + __popc(em) > LSTG)) {
                        __syncwarp();
                        flush_stage(p, cr, s_stage, nl);
                        if (__popc(em) > LSTG) cr.ovf = true;  // more than a lane's slots
                    }
                    while (em) {
                        const int q = __ffs(em) - 1;
                        em &= em - 1u;
                        if (nl < LSTG)
                            s_stage[nl * 32 + lane] = ((unsigned long long)key_of(word_elem_rt<T>(w, q)) << 32) |
                                                      (uint32_t)(e_base + vi * VW + q);
                        ++nl;
                    }
                    nl = min(nl, LSTG);
                }
                __syncwarp();
                cr.hist_n += nq;
                since += nq;
                if (cr.hist_n >= k && since >= 32) {
                    raise_tau(cr, s_hist, k);
                    since = 0;
                    if (lane == 0) atomicMax(ctl + CTL_TAU, cr.tau);
                }
            }

            // ---- the stage is free: refill it
            __syncwarp();
            const PieceCur nx = tail.r >= 0 ? next_item(tail) : tail;
            if (nx.r >= 0) {
                // every read of the stage has completed (its values are in
                // registers) before the warp synchronised, so the copy may
                // overwrite it
                if (lane == 0) issue(nx, s);
                ++issued;
            }
            tail = nx;
            ++kk;
            if (cur.pc + 1 >= hi_pc(r)) break;
            ++cur.pc;
        }
        if (failed) break;
        // ---------------- the row's end in this run
        if (cr.hist_n >= k && since > 0) raise_tau(cr, s_hist, k);
        __syncwarp();
        flush_stage(p, cr, s_stage, nl);
        const uint32_t km = __reduce_max_sync(FULL, cr.kmax);
        cr.ovf = __any_sync(FULL, cr.ovf);
        if (lane == 0) {
            atomicMax(ctl + CTL_TAU, cr.tau);
            atomicMax(ctl + CTL_MAXKEY, km);
            if (cr.ovf) atomicAdd(ctl + CTL_COUNT, (unsigned)RCAP_ROW + 1u);
        }
        __syncwarp();
        cur = enter_row(r - 1);
    }
    if (failed) {
        if (lane == 0) atomicOr(p.err, 4u);
        // wait (bounded) for the copies still in flight before leaving
        for (int kq = kk; kq < issued; ++kq) mbar_wait(&full[kq % CS_STAGES], (kq / CS_STAGES) & 1);
    }
}

template <typename T>
static cudaError_t launch_stream_cand_t(const Params& p, int num_sms, cudaStream_t s)
{
    static int ctas_per_sm = 0;
    if (!ctas_per_sm) {
        cudaError_t e = cudaFuncSetAttribute(k_stream_cand<T>,
                                             cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas_per_sm, k_stream_cand<T>, 32, CS_SMEM);
        if (e != cudaSuccess) return e;
        if (ctas_per_sm < 1) return cudaErrorInvalidConfiguration;
    }
    // up to CS_WARPS_PER_SM warps per SM, each with at least CS_MIN_RUN pieces
    const int64_t items = (int64_t)p.B * p.rps * p.npiece;
    int64_t grid = (int64_t)std::min(ctas_per_sm, CS_WARPS_PER_SM) * num_sms;
    const int64_t by_run = (items + CS_MIN_RUN - 1) / CS_MIN_RUN;
    if (grid > by_run) grid = by_run;
    if (grid <= 0) return cudaSuccess;
    k_stream_cand<T><<<(unsigned)grid, 32, CS_SMEM, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_stream_cand(const Params& p, int dtype, int num_sms, cudaStream_t s)
{
    return dtype == 1 ? launch_stream_cand_t<__nv_bfloat16>(p, num_sms, s)
                      : launch_stream_cand_t<float>(p, num_sms, s);
}

}  // namespace sv
