// sv_cand.cuh -- the candidate stream kernel (included by sv_rows.cu).
//
// For rows whose kept set is bounded by top-k (k <= CAND_TOPK_MAX) the row
// merge needs only the logits that can be in the top-k.  This kernel streams
// every row once, like k_stream, and while a piece is in shared memory it also
// collects those candidates:
//
//  * Work.  Each CTA (CW warps) owns a contiguous run of pieces (CS_PIECE
//    bytes of one row slot; items in row-major order).  It walks the run's
//    rows from the last to the first; the warps share a row, taking its pieces
//    in turn (piece lo + w + i * CW to warp w), and meet at a CTA barrier only
//    between rows.  A row split between two runs is begun by the earlier run
//    (as its first work) and finished by the later one (as its last).  Each
//    warp's lane 0 keeps CS_STAGES of the warp's pieces in flight with bulk
//    (TMA) copies completing on the warp's own mbarriers.
//  * Chunk maxima.  Lane l reduces chunk l of a piece (128 bytes, eight
//    16-byte words), reading its words in a rotated order so the eight lanes
//    of a quarter-warp hit distinct banks; the 16-bit chunk keys go to the
//    workspace as in k_stream (the chunk-key merge runs when a row overflows).
//  * Threshold.  tau, a lower bound of the row's k-th largest logit, starts as
//    the row's published bound (from the other run of the row) or else from
//    the warps' first pieces: base = the largest over the warps of the k-th
//    largest word maximum of the warp's first piece, then every word maximum
//    of those pieces at or above base is counted and tau = the k-th largest
//    counted key.  Every later word maximum at or above tau is counted in a
//    CTA-shared histogram of 16-bit keys over a window fixed for the row
//    ([base, base + HW - 1], the top bin counting everything above); after
//    every RAISE_EVERY counts one warp scans it and raises tau to its k-th
//    largest key.  Counted maxima are logits of the row and no count sits
//    above its logit's key (a scan racing with new counts misses some, which
//    only lowers the result), so at least k logits are >= tau throughout.
//    Raises are published (atomic max) in the row's control words.
//  * Candidates.  A lane whose chunk reaches tau checks its words; the logits
//    >= tau of a word whose maximum reaches tau go (order key, token id)
//    straight to slots of the row's candidate array that the warp reserved
//    RSV at a time (one atomic); slots it leaves unused hold CAND_EMPTY.  The
//    last warp to finish the row publishes the row's largest tau and chunk
//    key in its control words.
#pragma once

namespace sv {

constexpr int CW = 4;                               // warps of a CTA
constexpr int CS_STAGES = 2;                        // ring stages per warp
constexpr int CS_WORDS = CS_PIECE / 16;             // 16-byte words per piece (256)
constexpr int CS_WPL = CS_WORDS / 32;               // words per lane: one chunk (8)
constexpr int RSV = 64;                             // candidate slots a warp reserves at once
constexpr int HW = 512;                             // histogram window (16-bit keys)
constexpr int HPL = HW / 32;                        // histogram bins a lane scans
constexpr int RAISE_EVERY = 32;                     // a warp's counts between its raises
constexpr int CS_CTAS_PER_SM = 6;
constexpr int CS_MIN_RUN = 64;                      // fewest pieces per CTA
constexpr int CS_SMEM = CW * CS_STAGES * CS_PIECE;  // the warps' rings
constexpr unsigned long long CAND_EMPTY = 0xFFFFFFFFull;  // an unused slot (token id ~0)
static_assert(CS_WPL * 16 == CHUNK_BYTES, "a lane reduces one chunk of the piece");

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

// a work item: piece pc of row slot r (r < 0: none)
struct PieceCur {
    int r, pc;
};

// CTA-shared state of the row being streamed
struct CandShared {
    uint32_t hist[HW];  // counts of word maxima at key base + i (top bin: above)
    uint32_t base;      // the row's starting bound, the histogram window start
    uint32_t tau;       // raised bounds (atomic max; the bound is max(base, tau))
    uint32_t kmax;      // largest chunk key of the row in this run
    int ovf;            // candidates were lost: the row takes the chunk path
    int published;      // base came from the row's control words
    int arrived;        // warps done with the row
};

// by one warp: the highest key t = base + b with at least k counts at or
// above bin b, or 0 when fewer than k are counted
__device__ __forceinline__ uint32_t hist_kth(const uint32_t* hist, int k, uint32_t base)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    uint32_t h[HPL];
    int local = 0;
#pragma unroll
    for (int q = 0; q < HPL; ++q) {
        h[q] = *((volatile const uint32_t*)hist + lane * HPL + q);
        local += (int)h[q];
    }
    int incl = local;  // counts in this lane's bins and above
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(FULL, incl, o);
        if (lane + o < 32) incl += y;
    }
    const unsigned hit = __ballot_sync(FULL, incl >= k);
    if (!hit) return 0u;
    const int L = 31 - __clz(hit);
    int b = 0;
    if (lane == L) {
        int run = incl - local;
#pragma unroll
        for (int q = HPL - 1; q >= 0; --q) {
            run += (int)h[q];
            if (run >= k) {
                b = lane * HPL + q;
                break;
            }
        }
    }
    return base + (uint32_t)__shfl_sync(FULL, b, L);
}

// a warp's reserved candidate slots of the row being streamed
struct CandSlots {
    unsigned base;  // first reserved slot (~0u: none reserved)
    int used;       // slots filled
};

// fill the unused reserved slots with CAND_EMPTY
__device__ __forceinline__ void close_slots(const Params& p, int r, CandSlots& cs)
{
    const int lane = threadIdx.x & 31;
    if (cs.base == ~0u) return;
    unsigned long long* dst = p.cand_rows + (int64_t)r * RCAP_ROW;
    for (int i = cs.used + lane; i < RSV; i += 32)
        if (cs.base + (unsigned)i < (unsigned)RCAP_ROW) dst[cs.base + i] = CAND_EMPTY;
    cs.base = ~0u;
    cs.used = 0;
}

// RSV more slots of row r (the count may pass RCAP_ROW: the merge then takes
// the chunk path)
__device__ __forceinline__ void reserve_slots(const Params& p, int r, CandSlots& cs)
{
    unsigned b = 0;
    if ((threadIdx.x & 31) == 0) b = atomicAdd(p.rowctl + (int64_t)r * 4 + CTL_COUNT, (unsigned)RSV);
    cs.base = __shfl_sync(0xffffffffu, b, 0);
    cs.used = 0;
}

template <typename T>
__global__ void __launch_bounds__(CW * 32) k_stream_cand(const Params p)
{
    extern __shared__ __align__(128) unsigned char smem_cs[];  // rings, then staging
    __shared__ __align__(8) uint64_t full[CW][CS_STAGES];
    __shared__ CandShared sh;
    using CM = ChunkMax<T>;
    using PM = typename CM::P;
    constexpr int VW = Vec16<T>::N;
    constexpr int PE = CS_PIECE / (int)sizeof(T);  // elements per piece
    const unsigned FULL = 0xffffffffu;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* ring = smem_cs + (size_t)warp * CS_STAGES * CS_PIECE;
    // the merge grid may be scheduled as this grid drains; it waits for this
    // grid's completion before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int npc = p.npiece;
    const int64_t total = (int64_t)p.B * p.rps * npc;
    const int64_t row_bytes = (int64_t)p.V * (int64_t)sizeof(T);
    const int k = p.top_k;
    // this CTA's run of items [beg, end): rows r_first..r_last, pieces
    // [first_pc, npc) of r_first and [0, last_hi) of r_last (32-bit from here)
    int r_first, first_pc, r_last, last_hi;
    {
        const int64_t beg = total * blockIdx.x / gridDim.x;
        const int64_t end = total * (blockIdx.x + 1) / gridDim.x;
        if (end <= beg) return;  // the whole CTA
        r_first = (int)(beg / npc);
        first_pc = (int)(beg - (int64_t)r_first * npc);
        r_last = (int)((end - 1) / npc);
        last_hi = (int)(end - 1 - (int64_t)r_last * npc) + 1;
    }
    if (lane == 0) {
        for (int s = 0; s < CS_STAGES; ++s) mbar_init(&full[warp][s], 1);
        fence_barrier_init();
    }
    for (int i = threadIdx.x; i < HW; i += CW * 32) sh.hist[i] = 0u;
    __syncthreads();
    auto lo_pc = [&](int r) { return r == r_first ? first_pc : 0; };
    auto hi_pc = [&](int r) { return r == r_last ? last_hi : npc; };
    auto row_streamed = [&](int r) {
        const RowRef rr = row_ref(p, r);
        return rr.valid && !(rr.is_draft && p.draft_kind == 1);
    };
    // the first streamed row at or below r (r_first - 1: none)
    auto streamed_at_or_below = [&](int r) {
        while (r >= r_first && !row_streamed(r)) --r;
        return r;
    };
    // this warp's first item in the streamed rows at or below r
    auto warp_first = [&](int r) -> PieceCur {
        for (r = streamed_at_or_below(r); r >= r_first; r = streamed_at_or_below(r - 1)) {
            const int pc = lo_pc(r) + warp;
            if (pc < hi_pc(r)) return PieceCur{r, pc};
        }
        return PieceCur{-1, 0};
    };
    auto next_item = [&](PieceCur c) -> PieceCur {
        if (c.pc + CW < hi_pc(c.r)) return PieceCur{c.r, c.pc + CW};
        return warp_first(c.r - 1);
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
        mbar_arrive_expect_tx(&full[warp][s], bytes);
        tma_load_1d(ring + (size_t)s * CS_PIECE, iss_base + at, bytes, &full[warp][s]);
    };

    // prime this warp's ring; `tail` is the last item issued (r < 0: the
    // warp's items are all issued)
    PieceCur tail = warp_first(r_last);
    int issued = 0;  // copies issued so far (copy i lands in stage i % CS_STAGES)
    if (tail.r >= 0) {
        if (lane == 0) issue(tail, 0);
        issued = 1;
        while (issued < CS_STAGES) {
            const PieceCur nx = next_item(tail);
            if (nx.r < 0) break;
            if (lane == 0) issue(nx, issued);
            tail = nx;
            ++issued;
        }
    }
    int kk = 0;       // pieces consumed
    bool failed = false;

    // wait for this warp's next piece and reduce it: word maxima pm, the
    // lane's chunk max, its chunk key stored; the piece's words (NULL on a
    // timeout)
    auto take_piece = [&](int r, int pc, PM (&pm)[CS_WPL], float& cmax, bool& chunk_here,
                          uint32_t& kmax, int& nvec) -> const uint4* {
        const int s = kk % CS_STAGES;
        if (failed || !mbar_wait(&full[warp][s], (kk / CS_STAGES) & 1)) {
            failed = true;
            return nullptr;
        }
        const uint4* sv4 = reinterpret_cast<const uint4*>(ring + (size_t)s * CS_PIECE);
        nvec = min(CS_WORDS, (p.V - pc * PE) / VW);
        PM cm = CM::lane(Vec16<T>::neg_inf());
        if (nvec == CS_WORDS) {
#pragma unroll
            for (int v = 0; v < CS_WPL; ++v) {
                pm[v] = CM::lane(sv4[lane * CS_WPL + ((v + lane) & (CS_WPL - 1))]);
                cm = CM::mx(cm, pm[v]);
            }
        } else {
#pragma unroll
            for (int v = 0; v < CS_WPL; ++v) {
                const int vi = lane * CS_WPL + ((v + lane) & (CS_WPL - 1));
                pm[v] = CM::lane(vi < nvec ? sv4[vi] : Vec16<T>::neg_inf());
                cm = CM::mx(cm, pm[v]);
            }
        }
        chunk_here = lane * CS_WPL < nvec;
        cmax = CM::value(cm);
        const uint32_t ck = chunk_here ? key_of(cmax) >> 16 : 0u;
        if (chunk_here) p.chunk[(int64_t)r * p.chunk_stride + pc * 32 + lane] = (uint16_t)ck;
        kmax = max(kmax, ck);
        return sv4;
    };
    // the piece's stage is free: refill it with this warp's next item
    auto release_piece = [&]() {
        __syncwarp();
        // every read of the stage has completed (its values are in registers)
        // before the warp synchronised, so the copy may overwrite it
        if (tail.r >= 0 && !failed) {
            const PieceCur nx = next_item(tail);
            if (nx.r >= 0) {
                if (lane == 0) issue(nx, kk % CS_STAGES);
                ++issued;
            }
            tail = nx;
        }
        ++kk;
    };

    for (int r = streamed_at_or_below(r_last); r >= r_first; r = streamed_at_or_below(r - 1)) {
        const int hi = hi_pc(r);
        unsigned* ctl = p.rowctl + (int64_t)r * 4;
        // ---------------- row start: the previous row is done by every warp;
        // the published bound, then each warp's first piece: without a
        // published bound, base is the largest of the warps' k-th largest
        // word maxima of those pieces
        __syncthreads();
        for (int i = threadIdx.x; i < HW; i += CW * 32) sh.hist[i] = 0u;
        if (threadIdx.x == 0) {
            sh.base = __ldcg(ctl + CTL_TAU);
            sh.published = sh.base != 0u;
            sh.tau = 0u;
            sh.kmax = 0u;
            sh.ovf = 0;
            sh.arrived = 0;
        }
        __syncthreads();
        const bool published = sh.published != 0;  // uniform over the CTA
        uint32_t kmax = 0u;
        int pc = lo_pc(r) + warp;
        PM pm[CS_WPL];
        float cmax = -INFINITY;
        bool chunk_here = false;
        int nvec = 0;
        const uint4* sv4 = nullptr;
        uint32_t wk[CS_WPL];
        if (pc < hi) {
            sv4 = take_piece(r, pc, pm, cmax, chunk_here, kmax, nvec);
            if (sv4 && !published) {
#pragma unroll
                for (int v = 0; v < CS_WPL; ++v) {
                    const int vi = lane * CS_WPL + ((v + lane) & (CS_WPL - 1));
                    wk[v] = vi < nvec ? key_of(CM::value(pm[v])) >> 16 : 0u;
                }
                const uint32_t t = warp_kth_key(wk, k);
                if (lane == 0) atomicMax(&sh.base, t);
            }
        }
        __syncthreads();
        const uint32_t base = sh.base;  // fixed for the row from here on
        // without a published bound, every word maximum >= base of the first
        // pieces is counted now and tau starts at the k-th largest of them
        // (a warp's first piece is not counted again below)
        const bool precounted = !published && sv4 != nullptr && base != 0u;
        if (!published && base != 0u) {
            if (precounted) {
#pragma unroll
                for (int v = 0; v < CS_WPL; ++v)
                    if (wk[v] != 0u && wk[v] >= base)
                        atomicAdd(&sh.hist[min(wk[v] - base, (uint32_t)(HW - 1))], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                const uint32_t t = hist_kth(sh.hist, k, base);
                if (lane == 0) sh.tau = t;
            }
            __syncthreads();
        }

        // ---------------- this warp's pieces of the row
        CandSlots cs{~0u, 0};
        int own = 0;  // this warp's counts since its last raise
        for (bool first = precounted; pc < hi; pc += CW, first = false) {
            if (!sv4) sv4 = take_piece(r, pc, pm, cmax, chunk_here, kmax, nvec);
            if (!sv4) break;
            const uint32_t tau = max(base, *(volatile uint32_t*)&sh.tau);
            const float tf = key16_floor(tau);
            const uint32_t tf2 = CM::thr2(tf);
            const int e_base = pc * PE;  // < V
            // candidates: only lanes whose chunk reaches tau do any work; one
            // word per lane per round
            if (__any_sync(FULL, chunk_here && cmax >= tf)) {
                uint32_t qm = 0;
                if (chunk_here && cmax >= tf) {
#pragma unroll
                    for (int v = 0; v < CS_WPL; ++v) {
                        const int vi = lane * CS_WPL + ((v + lane) & (CS_WPL - 1));
                        if (vi < nvec && CM::any_ge(pm[v], tf, tf2)) qm |= 1u << v;
                    }
                }
                if (!first) own += __reduce_add_sync(FULL, __popc(qm));
                while (__any_sync(FULL, qm != 0u)) {
                    uint32_t em = 0;
                    int vi = 0;
                    uint4 w = make_uint4(0, 0, 0, 0);
                    if (qm) {
                        const int v = __ffs(qm) - 1;
                        qm &= qm - 1u;
                        vi = lane * CS_WPL + ((v + lane) & (CS_WPL - 1));
                        w = sv4[vi];
                        if (!first) {
                            const uint32_t wk16 = key_of(CM::value(CM::lane(w))) >> 16;
                            atomicAdd(&sh.hist[min(wk16 - base, (uint32_t)(HW - 1))], 1u);
                        }
                        em = CM::elem_mask(w, tf, tf2);
                    }
                    int tot;
                    const int ex = warp_excl_scan(__popc(em), &tot);
                    if (tot > RSV) {
                        // more candidates in one round than a reservation:
                        // the row takes the chunk path
                        if (lane == 0) sh.ovf = 1;
                        continue;
                    }
                    if (cs.base == ~0u || cs.used + tot > RSV) {
                        close_slots(p, r, cs);
                        reserve_slots(p, r, cs);
                    }
                    if (em) {
                        unsigned long long* dst = p.cand_rows + (int64_t)r * RCAP_ROW;
                        unsigned at = cs.base + (unsigned)(cs.used + ex);
                        while (em) {
                            const int q = __ffs(em) - 1;
                            em &= em - 1u;
                            if (at < (unsigned)RCAP_ROW)
                                dst[at] = ((unsigned long long)key_of(word_elem_rt<T>(w, q)) << 32) |
                                          (uint32_t)(e_base + vi * VW + q);
                            ++at;
                        }
                    }
                    cs.used += tot;
                }
                // raise tau after RAISE_EVERY of this warp's counts
                if (own >= RAISE_EVERY) {
                    own = 0;
                    __syncwarp();
                    const uint32_t t = hist_kth(sh.hist, k, base);
                    if (lane == 0 && t > tau) {
                        atomicMax(&sh.tau, t);
                        atomicMax(ctl + CTL_TAU, t);
                    }
                }
            }
            release_piece();
            sv4 = nullptr;
        }
        // ---------------- row end: the last warp to finish publishes the
        // row's bound (the final histogram scan) and largest chunk key
        close_slots(p, r, cs);
        const uint32_t km = __reduce_max_sync(FULL, kmax);
        int last = 0;
        if (lane == 0) {
            atomicMax(&sh.kmax, km);
            __threadfence_block();
            last = atomicAdd(&sh.arrived, 1) == CW - 1;
        }
        if (__shfl_sync(FULL, last, 0)) {
            __threadfence_block();
            const uint32_t t = hist_kth(sh.hist, k, base);
            if (lane == 0) {
                atomicMax(ctl + CTL_TAU, max(max(t, base), *(volatile uint32_t*)&sh.tau));
                atomicMax(ctl + CTL_MAXKEY, *(volatile uint32_t*)&sh.kmax);
                if (*(volatile int*)&sh.ovf) atomicAdd(ctl + CTL_COUNT, (unsigned)RCAP_ROW + 1u);
            }
        }
    }
    if (failed) {
        if (lane == 0) atomicOr(p.err, 4u);
        // wait (bounded) for the copies still in flight before leaving
        for (int kq = kk; kq < issued; ++kq) mbar_wait(&full[warp][kq % CS_STAGES], (kq / CS_STAGES) & 1);
    }
}

template <typename T>
static cudaError_t launch_stream_cand_t(const Params& p, int num_sms, cudaStream_t s)
{
    static int ctas_per_sm = 0;
    if (!ctas_per_sm) {
        cudaError_t e = cudaFuncSetAttribute(k_stream_cand<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, CS_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_stream_cand<T>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas_per_sm, k_stream_cand<T>, CW * 32,
                                                          CS_SMEM);
        if (e != cudaSuccess) return e;
        if (ctas_per_sm < 1) return cudaErrorInvalidConfiguration;
    }
    // up to CS_CTAS_PER_SM CTAs per SM, each with at least CS_MIN_RUN pieces
    const int64_t items = (int64_t)p.B * p.rps * p.npiece;
    int64_t grid = (int64_t)(ctas_per_sm < CS_CTAS_PER_SM ? ctas_per_sm : CS_CTAS_PER_SM) * num_sms;
    const int64_t by_run = (items + CS_MIN_RUN - 1) / CS_MIN_RUN;
    if (grid > by_run) grid = by_run;
    if (grid <= 0) return cudaSuccess;
    k_stream_cand<T><<<(unsigned)grid, CW * 32, CS_SMEM, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_stream_cand(const Params& p, int dtype, int num_sms, cudaStream_t s)
{
    return dtype == 1 ? launch_stream_cand_t<__nv_bfloat16>(p, num_sms, s)
                      : launch_stream_cand_t<float>(p, num_sms, s);
}

}  // namespace sv
