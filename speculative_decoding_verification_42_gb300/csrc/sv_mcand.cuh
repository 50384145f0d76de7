// sv_mcand.cuh -- the row merge of the top-k rows (1 <= k <= CAND_TOPK_MAX),
// one CTA per row slot after the chunk-key stream (included by sv_rows.cu
// after the streaming kernel and the warp code).
//
//  * bound: any value that k chunks reach bounds the row's k-th largest
//    logit from below (each of those chunks holds a logit at least that
//    large).  The first bound is the k-th largest of the threads' own
//    largest chunk keys (k <= MC_T threads each hold one), counted in a
//    window of MCG_HB keys below the row's largest; when it was not found,
//    or its chunks exceed one gather round, or their candidates the staging,
//    it is raised once to the k-th largest chunk key (the same count over
//    the keys at or above the first bound);
//  * candidates: the chunks reaching the bound are read back from HBM and
//    their logits at or above it kept, each list compacted with one
//    block-wide prefix sum;
//  * merge: the candidates are ranked in the exact order (logit descending,
//    token id ascending: one rank per thread by counting), the first k kept,
//    then the top-p prefix in rank order; the kept list goes out in ascending
//    id with M, S and P(x) at the drafted token.
//
// The last row of a sequence to be merged decides the sequence: warp 0 takes
// the accept tests (the head of the warp decision of sv_warp.cuh) while the
// other warps stage the sequence's kept lists, then the CTA draws the sample.
// Rows with more candidates than the CTA stages (ties), and sequences of more
// than 32 rows, are left to the decision grid.
#pragma once

namespace sv {

constexpr int MC_T = NS;         // threads of a row's CTA (its barrier is ssync)
constexpr int MC_CAP = 256;      // candidates a row can stage
constexpr int MCG_U4 = 4;        // 16-byte words of chunk keys per thread (8 keys each)
constexpr int MCG_QCAP = 256;    // qualifying chunks a row can stage
constexpr int MCG_LPT = 8;       // chunk words per thread per load round
constexpr int MCG_HB = 512;      // histogram bins (keys below the row's largest chunk key)
constexpr int MCG_QFAST = MC_T * MCG_LPT * 16 / CHUNK_BYTES;  // chunks one gather round reads
constexpr int MCG_BPT = MCG_HB / MC_T;  // bins a thread sums
constexpr int MC_STAGE = 4 * WM_CAND * 4;  // the decision's staged kept lists
static_assert(CAND_TOPK_MAX <= MC_T, "one kept rank per thread; k threads bound the k-th key");
static_assert(MC_T * MCG_U4 * 8 >= 4096, "the merge holds every chunk key of a warp-merge row");
static_assert(MC_T == 128, "the block sums add four warp sums");

struct __align__(16) McSmem {
    union {
        struct {
            uint32_t hist[MCG_HB];    // chunk keys at (largest key - bin)
            uint32_t qc[MCG_QCAP];    // qualifying chunks
        } g;
        unsigned char stage[MC_STAGE];
    } u;
    unsigned long long cand[MC_CAP];  // candidates: (~order key) << 32 | token id
    unsigned long long ord[MC_CAP];   // the candidates in rank order
    float redf[MC_T / 32];
    int redi[MC_T / 32];
    uint32_t sel[4];                  // the row's largest chunk key, a selected bound
    int stop;                         // first rank the top-p prefix drops
    int flag;                         // this CTA decides the sequence
    float px;
    int dstate;                       // the decision's head: DECIDE_*
    int tok;                          // the drawn token
    unsigned long long redu[MC_T / 32];
    DecidePending pend;               // the decision's pending sample
};
// after the merge, u, cand and ord (one 8 KB span) stage the kept lists of
// the deciding CTA's sequence
constexpr int MC_PRE_BYTES = MC_STAGE + 2 * MC_CAP * 8;
static_assert(offsetof(McSmem, u) == 0 && sizeof(McSmem::u) == MC_STAGE && offsetof(McSmem, cand) == MC_STAGE &&
                  offsetof(McSmem, ord) == MC_STAGE + MC_CAP * 8,
              "u, cand and ord are one span at the start");

__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

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

// block sum of one value per thread (a tree of fp32 additions: at
// most k <= 128 terms in [0, 1], relative error ~1e-7); all threads get it
__device__ __forceinline__ float mc_sum(float v, float* red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    ssync();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    ssync();
    return (red[0] + red[1]) + (red[2] + red[3]);
}

// block-wide exclusive prefix sum of one int per thread; *total gets
// the sum.  Two barriers; red may be reused after it returns.
__device__ __forceinline__ int mc_excl_scan(int v, int* red, int* total)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) red[warp] = x;
    ssync();
    int before = 0;
#pragma unroll
    for (int w = 0; w < MC_T / 32; ++w) before += w < warp ? red[w] : 0;
    *total = red[0] + red[1] + red[2] + red[3];
    ssync();
    return before + x - v;
}

// the merge of top-k row r by the MC_T threads: the row's record (also
// written to p.rstat) and its kept list; FLAG_BLOCK_MERGE when the CTA's
// staging overflows (ties)
template <typename T>
__device__ RowStat merge_row_topk_core(const Params& p, int r, McSmem& sm)
{
    const unsigned FULL = 0xffffffffu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // every load that does not depend on another goes out at once
    const int b = r / p.rps, slot = r - b * p.rps;
    const int jd = slot > p.Kmax ? slot - (p.Kmax + 1) : slot;  // position of the row
    const int x_raw = jd < p.Kmax ? __ldg(p.xin + (int64_t)b * p.Kmax + jd) : -1;
    const uint4* ksrc = reinterpret_cast<const uint4*>(p.chunk + (int64_t)r * p.chunk_stride);
    const int nch = p.nchunk;
    uint4 kw[MCG_U4];  // word g holds keys 8 (g MC_T + tid) .. + 7
    auto load_keys = [&]() {
#pragma unroll
        for (int g = 0; g < MCG_U4; ++g)
            kw[g] = (g * MC_T + tid) * 8 < nch ? __ldcg(ksrc + g * MC_T + tid) : make_uint4(0, 0, 0, 0);
    };
    load_keys();
    const RowRef rr = row_ref(p, r);
    const T* row = (const T*)(rr.is_draft ? p.draft : p.target) + row_elem_offset(p, rr);
    const int x = (rr.j < rr.kb && x_raw >= 0 && x_raw < p.V) ? x_raw : -1;
    const int k = p.top_k;
#pragma unroll
    for (int i = 0; i < MCG_BPT; ++i) sm.u.g.hist[i * MC_T + tid] = 0u;

    RowStat st;
    st.M = -INFINITY;
    st.kappa = 0;
    st.S = 0.0;
    st.i_kappa = p.V - 1;
    st.n_kept = p.V;
    st.mode = MODE_ALL;
    st.flags = 0;
    st.px = 0.f;
    st.pad[0] = st.pad[1] = st.pad[2] = 0;
    bool staged = false;  // candidates are in sm.cand (n of them)
    int n = 0;

    auto key_at = [&](int g, int i) -> uint32_t {
        const uint32_t u = (i >> 1) == 0 ? kw[g].x : (i >> 1) == 1 ? kw[g].y : (i >> 1) == 2 ? kw[g].z : kw[g].w;
        return (i & 1) ? (u >> 16) : (u & 0xFFFFu);
    };
    auto key_in = [&](int g, int i) { return (g * MC_T + tid) * 8 + i < nch; };
    uint32_t tmax = 0u;  // this thread's largest chunk key
#pragma unroll
    for (int g = 0; g < MCG_U4; ++g)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (key_in(g, i)) tmax = max(tmax, key_at(g, i));
    const uint32_t wmax = __reduce_max_sync(FULL, tmax);
    if (lane == 0) sm.redi[warp] = (int)wmax;
    ssync();  // the warps' maxima are posted, the histogram is cleared
    const uint32_t maxkey = max(max((uint32_t)sm.redi[0], (uint32_t)sm.redi[1]),
                                max((uint32_t)sm.redi[2], (uint32_t)sm.redi[3]));
    if (maxkey >= 0xFF80u || maxkey <= 0x007Fu) {  // NaN or +inf, or no finite logit
        st.flags = FLAG_NONFINITE;
    } else {
        // the k-th largest key counted in the histogram window (at maxkey -
        // key), at least `floor`; floor when the window holds fewer than k.
        // Clears the histogram.
        auto window_kth = [&](uint32_t floor) -> uint32_t {
            uint32_t hb[MCG_BPT];
            int local = 0;
#pragma unroll
            for (int i = 0; i < MCG_BPT; ++i) {
                hb[i] = sm.u.g.hist[tid * MCG_BPT + i];
                local += (int)hb[i];
            }
            int in_window;
            const int before = mc_excl_scan(local, sm.redi, &in_window);
            // (sel[3] is written by the thread holding the k-th key, read only
            // when the window holds k keys: it needs no reset)
            if (before < k && before + local >= k) {
                int run = before;
#pragma unroll
                for (int i = 0; i < MCG_BPT; ++i) {
                    run += (int)hb[i];
                    if (run >= k) {
                        sm.sel[3] = maxkey - (uint32_t)(tid * MCG_BPT + i);
                        break;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < MCG_BPT; ++i) sm.u.g.hist[tid * MCG_BPT + i] = 0u;
            ssync();
            const uint32_t t = in_window >= k ? sm.sel[3] : 0u;
            return max(t, floor);
        };
        // ---- a first bound: the k-th largest of the threads' largest keys
        //      (k <= MC_T threads each hold a key at least that large)
        {
            const uint32_t d = maxkey - tmax;
            if (tmax != 0u && d < (uint32_t)MCG_HB) atomicAdd(&sm.u.g.hist[d], 1u);
        }
        ssync();
        const uint32_t tau0 = window_kth(0u);
        // ---- the chunks reaching the bound (at least k of them), compacted,
        //      read back, and their logits at or above it kept.  tau0 serves
        //      when it was found, its chunks fit one gather round and their
        //      candidates the staging; otherwise the bound is raised once, to
        //      the k-th largest chunk key (counted among the keys >= tau0)
        auto reaching = [&](uint32_t tau) {
            uint32_t m = 0u;
#pragma unroll
            for (int g = 0; g < MCG_U4; ++g)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (key_in(g, i) && key_at(g, i) >= tau) m |= 1u << (g * 8 + i);
            return m;
        };
        auto raise_bound = [&]() {
#pragma unroll
            for (int g = 0; g < MCG_U4; ++g)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t key = key_at(g, i);
                    const uint32_t d = maxkey - key;
                    if (key_in(g, i) && key >= tau0 && d < (uint32_t)MCG_HB) atomicAdd(&sm.u.g.hist[d], 1u);
                }
            ssync();
            return window_kth(tau0);
        };
        uint32_t tau_c = tau0;
        bool raised = false;
        // nq, n and the bounds are the same in every thread
        for (;;) {
            uint32_t qmask = reaching(tau_c);
            int nq;
            int at = mc_excl_scan(__popc(qmask), sm.redi, &nq);
            if (!raised && (tau0 == 0u || nq > MCG_QFAST)) {
                tau_c = raise_bound();
                raised = true;
                continue;
            }
            while (qmask) {
                const int bit = __ffs(qmask) - 1;
                qmask &= qmask - 1u;
                if (at < MCG_QCAP) sm.u.g.qc[at] = (uint32_t)(((bit >> 3) * MC_T + tid) * 8 + (bit & 7));
                ++at;
            }
            ssync();
            if (nq > MCG_QCAP) break;
            constexpr int VW = Vec16<T>::N;
            constexpr int CWD = CHUNK_BYTES / 16;  // words per chunk
            const uint4* rowv = reinterpret_cast<const uint4*>(row);
            const int nw_row = p.V / VW;          // whole words: V s is a multiple of 16 here
            n = 0;
            for (int w0 = 0; w0 < nq * CWD; w0 += MC_T * MCG_LPT) {
                uint4 wv[MCG_LPT];
                int wi[MCG_LPT];
#pragma unroll
                for (int j = 0; j < MCG_LPT; ++j) {
                    const int i = w0 + j * MC_T + tid;
                    wi[j] = -1;
                    wv[j] = make_uint4(0, 0, 0, 0);
                    if (i < nq * CWD) {
                        const int word = (int)sm.u.g.qc[i / CWD] * CWD + i % CWD;
                        if (word < nw_row) {
                            wi[j] = word;
                            wv[j] = __ldcg(rowv + word);
                        }
                    }
                }
                uint32_t em[MCG_LPT];
                int cnt = 0;
                if constexpr (sizeof(T) == 2) {
                    // bf16: a value reaches the bound iff its key does; one
                    // packed compare per two values (-inf words never reach a
                    // finite bound; a -inf bound admits them by key as well)
                    const uint32_t thr2 = ChunkMax<T>::thr2(val_key16(tau_c));
#pragma unroll
                    for (int j = 0; j < MCG_LPT; ++j) {
                        em[j] = wi[j] >= 0 ? ChunkMax<T>::elem_mask(wv[j], 0.f, thr2) : 0u;
                        cnt += __popc(em[j]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < MCG_LPT; ++j) {
                        em[j] = 0u;
#pragma unroll
                        for (int q = 0; q < VW; ++q)
                            if (wi[j] >= 0 && (key_of(word_elem_rt<T>(wv[j], q)) >> 16) >= tau_c) em[j] |= 1u << q;
                        cnt += __popc(em[j]);
                    }
                }
                int tot;
                int pos = n + mc_excl_scan(cnt, sm.redi, &tot);
#pragma unroll
                for (int j = 0; j < MCG_LPT; ++j) {
                    uint32_t m = em[j];
                    while (m) {
                        const int q = __ffs(m) - 1;
                        m &= m - 1u;
                        const uint32_t key = key_of(word_elem_rt<T>(wv[j], q));
                        if (pos < MC_CAP)
                            sm.cand[pos] = ((unsigned long long)(~key) << 32) | (uint32_t)(wi[j] * VW + q);
                        ++pos;
                    }
                }
                n += tot;
            }
            ssync();  // the staging is read; qc and cand may be rewritten
            if (!raised && n > MC_CAP) {
                load_keys();  // again: the registers are not held through the gather
                tau_c = raise_bound();
                raised = true;
                continue;
            }
            staged = true;
            break;
        }
    }
    if (staged && n >= 1 && n <= MC_CAP) {
        // ---- exact rank of every candidate (keys are distinct: ids are)
        for (int i = tid; i < n; i += MC_T) {
            const unsigned long long v = sm.cand[i];
            int rank = 0;
            for (int j = 0; j < n; ++j) rank += sm.cand[j] < v;
            sm.ord[rank] = v;
        }
        if (tid == 0) sm.stop = INT_MAX;
        ssync();
        const int kk = min(k, n);
        const float M = val_of(~(uint32_t)(sm.ord[0] >> 32));
        const float c = p.c;
        const float lt = tid < kk ? val_of(~(uint32_t)(sm.ord[tid] >> 32)) : 0.f;
        const int idt = tid < kk ? (int)(uint32_t)sm.ord[tid] : -1;
        const float et = tid < kk ? ex2_fast((lt - M) * c) : 0.f;
        float S = mc_sum(et, sm.redf);
        int nk = kk;
        if (p.top_p < 1.0f) {
            // mass strictly before each rank, in rank order
            const float pv = tid < kk ? et / S : 0.f;
            float y = pv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float t = __shfl_up_sync(FULL, y, o);
                if (lane >= o) y += t;
            }
            ssync();
            if (lane == 31) sm.redf[warp] = y;
            ssync();
            float before = y - pv;
            for (int i = 0; i < warp; ++i) before += sm.redf[i];
            if (tid < kk && !(before < p.top_p)) atomicMin(&sm.stop, tid);
            ssync();
            nk = min(sm.stop, kk);  // the first rank whose mass before it reaches top_p
            S = mc_sum(tid < nk ? et : 0.f, sm.redf);
        }
        const float invS = 1.f / S;
        // ---- the kept list in ascending id, P(x)
        if (tid == 0) sm.px = 0.f;
        ssync();
        if (tid < nk) {
            int pos = 0;
            for (int j = 0; j < nk; ++j) pos += (int)(uint32_t)sm.ord[j] < idt;
            p.kept_id[(int64_t)r * KCAP + pos] = idt;
            p.kept_l[(int64_t)r * KCAP + pos] = lt;
            if (idt == x) sm.px = exp2f((lt - M) * c) * invS;
        }
        ssync();
        st.M = M;
        st.S = (double)S;
        st.n_kept = nk;
        st.mode = MODE_LIST;
        st.px = sm.px;
    } else if (!(st.flags & FLAG_NONFINITE)) {
        st.flags |= FLAG_BLOCK_MERGE;  // ties: more candidates than staged; the decision grid merges
    }
    if (tid == 0) p.rstat[r] = st;
    return st;
}

// block-wide inclusive prefix sum of one u64 per thread; *total gets the
// sum.  Two barriers; red may be reused after it returns.
__device__ __forceinline__ unsigned long long mc_incl_scan_u64(unsigned long long v, unsigned long long* red,
                                                               unsigned long long* total)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) red[warp] = x;
    ssync();
    unsigned long long before = 0ull;
#pragma unroll
    for (int w = 0; w < MC_T / 32; ++w) before += w < warp ? red[w] : 0ull;
    *total = (red[0] + red[1]) + (red[2] + red[3]);
    ssync();
    return before + x;
}

// the pending sample of a decision drawn by the CTA from staged lists, one
// kept token per thread (both lists hold at most MC_T): the same fixed-point
// masses, sums and inverse CDF as warp_sample_list, so the same token.
// sm.tok must be -1 before the barrier that ordered the staging.  Every
// thread gets the token (-1: no mass), *Zfix the first attempt's total and
// *zero whether the residual had no mass (the row itself was then sampled).
template <typename T>
__device__ int mc_sample_staged(const Params& p, const DecidePending& pe, const StagedList& tl,
                                const StagedList& dl, McSmem& sm, unsigned long long* Zfix, bool* zero)
{
    const int tid = threadIdx.x;
    const int n = tl.n;
    const float invSt = 1.f / (float)pe.ts.S;
    const float invSd = (pe.residual && pe.d.kind == 0) ? 1.f / (float)pe.d.st.S : 0.f;
    *zero = false;
    for (int attempt = 0; attempt < 2; ++attempt) {
        const bool res = pe.residual && attempt == 0;
        const unsigned long long part =
            tid < n ? list_r_fix<T>(p, pe.ts, tl, tid, res, pe.d, dl, invSt, invSd) : 0ull;
        unsigned long long Z;
        const unsigned long long ex = mc_incl_scan_u64(part, sm.redu, &Z) - part;
        if (attempt == 0) *Zfix = Z;
        if (Z == 0ull) {  // the same in every thread
            if (res) {
                *zero = true;
                continue;
            }
            return -1;
        }
        const unsigned long long t = cdf_target(pe.u, Z);
        if (ex <= t && t < ex + part) sm.tok = tl.ids[tid];  // one thread at most
        ssync();
        return sm.tok;
    }
    return -1;
}

// the same, staging the two lists from global memory first
template <typename T>
__device__ int mc_sample_list(const Params& p, const DecidePending& pe, McSmem& sm,
                              unsigned long long* Zfix, bool* zero)
{
    const int tid = threadIdx.x;
    const int n = pe.ts.n_kept;
    int32_t* ti = reinterpret_cast<int32_t*>(sm.u.stage);
    float* tv = reinterpret_cast<float*>(sm.u.stage) + MC_T;
    int32_t* di = reinterpret_cast<int32_t*>(sm.u.stage) + 2 * MC_T;
    float* dv = reinterpret_cast<float*>(sm.u.stage) + 3 * MC_T;
    static_assert(4 * MC_T * 4 <= MC_STAGE, "two staged lists fit the stage");
    const bool res_list = pe.residual && pe.d.kind == 0 && pe.d.st.mode == MODE_LIST;
    const StagedList tl{ti, tv, n}, dl{di, dv, res_list ? pe.d.st.n_kept : 0};
    if (tid < n) {
        ti[tid] = __ldcg(p.kept_id + (int64_t)pe.tr * KCAP + tid);
        tv[tid] = __ldcg(p.kept_l + (int64_t)pe.tr * KCAP + tid);
    }
    if (tid < dl.n) {
        di[tid] = __ldcg(p.kept_id + (int64_t)pe.d.r * KCAP + tid);
        dv[tid] = __ldcg(p.kept_l + (int64_t)pe.d.r * KCAP + tid);
    }
    if (tid == 0) sm.tok = -1;
    ssync();
    return mc_sample_staged<T>(p, pe, tl, dl, sm, Zfix, zero);
}

// the merge of top-k row r; then the sequence ticket and, for the last row of
// a sequence, the decision
template <typename T>
__device__ void merge_row_topk(const Params& p, int r, McSmem& sm)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const RowRef rr = row_ref(p, r);
    merge_row_topk_core<T>(p, r, sm);
    // sequence ticket: the barrier orders every thread's writes before thread
    // 0's fence, which makes them visible before the ticket is taken; the
    // last row's second fence, before the next barrier, orders the other
    // rows' records and lists before any thread of this CTA reads them
    ssync();
    if (tid == 0) {
        __threadfence();
        const int nrows = seq_rows(p, rr.kb);
        const bool last = atomicAdd(&p.seq_ticket[rr.b], 1u) == (unsigned)(nrows - 1);
        if (last) {
            p.seq_ticket[rr.b] = 0u;
            __threadfence();
        }
        sm.flag = last;
    }
    ssync();
    const bool last = sm.flag != 0;
    const int nrows_b = seq_rows(p, rr.kb);
    if (last && nrows_b <= 32) {
        // warp 0 takes the accept tests while the other warps stage the kept
        // list of every row of the sequence (when they fit); then the CTA
        // draws the sample.  A list holds at most top_k tokens.
        const int kb = rr.kb;
        const int klp = (p.top_k + 3) & ~3;  // a staged list, rounded to 16 bytes
        const bool pre = 2 * nrows_b * klp * 4 <= MC_PRE_BYTES;
        int32_t* pid = reinterpret_cast<int32_t*>(&sm);
        float* pl = reinterpret_cast<float*>(&sm) + nrows_b * klp;
        if (warp == 0) {
            DecidePending pe;
            const int h = warp_decide_lanes_head<T>(p, rr.b, kb, &pe);
            if (lane == 0) {
                sm.dstate = h;
                sm.tok = -1;
                if (h == DECIDE_SAMPLE) sm.pend = pe;
            }
        } else if (pre) {
            const int per = klp / 4;  // 16-byte words of a staged list
            const int nw = nrows_b * per;
            for (int e = tid - 32; e < 2 * nw; e += MC_T - 32) {
                const int half = e >= nw;  // 0: ids, 1: logits
                const int i = (e - half * nw) / per, q = (e - half * nw) - i * per;
                const int64_t row = i <= kb ? target_slot(p, rr.b, i) : draft_slot(p, rr.b, i - kb - 1);
                if (half) cp_async16(pl + i * klp + 4 * q, p.kept_l + row * KCAP + 4 * q);
                else cp_async16(pid + i * klp + 4 * q, p.kept_id + row * KCAP + 4 * q);
            }
            cp_async_wait_all();
        }
        ssync();
        const int h = sm.dstate;
        if (h == DECIDE_SAMPLE) {
            const DecidePending& pe = sm.pend;
            unsigned long long Z;
            bool zero;
            const bool res_list = pe.residual && pe.d.kind == 0 && pe.d.st.mode == MODE_LIST;
            const int nd = res_list ? pe.d.st.n_kept : 0;
            if (pre && pe.ts.n_kept <= min(klp, MC_T) && nd <= min(klp, MC_T)) {
                const int jt = pe.jstar, jd = kb + 1 + pe.jstar;
                const StagedList tl{pid + jt * klp, pl + jt * klp, pe.ts.n_kept};
                const StagedList dl{pid + (res_list ? jd : 0) * klp, pl + (res_list ? jd : 0) * klp, nd};
                const int tok = mc_sample_staged<T>(p, pe, tl, dl, sm, &Z, &zero);
                if (tid == 0) decide_finish(p, rr.b, pe, tok, Z, zero);
            } else if (pe.ts.n_kept <= MC_T && nd <= MC_T) {
                const int tok = mc_sample_list<T>(p, pe, sm, &Z, &zero);
                if (tid == 0) decide_finish(p, rr.b, pe, tok, Z, zero);
            } else if (warp == 0) {
                const int tok = warp_sample_list<T>(p, pe.tr, pe.ts, pe.residual != 0, pe.d, pe.u, sm.u.stage,
                                                    &Z, &zero);
                if (lane == 0) decide_finish(p, rr.b, pe, tok, Z, zero);
            }
        }
        if (h != DECIDE_LEFT && tid == 0) p.seq_done[rr.b] = 1u;
    }
    ssync();  // sm is free again
}

template <typename T>
__global__ void __launch_bounds__(MC_T, 8) k_merge_cand(const Params p)
{
    __shared__ McSmem sm;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream grid has completed
    if (exit_skip(p)) return;
    // the decision grid may be scheduled now; it waits for this grid's end
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int r = blockIdx.x;
    const RowRef rr = row_ref(p, r);
    if (!rr.valid) {
        if (threadIdx.x == 0) report_skipped_row(p, rr);
        return;
    }
    if (rr.is_draft && !drafts_streamed(p)) return;  // probabilities (or greedy): read only where needed
    merge_row_topk<T>(p, r, sm);
}

}  // namespace sv
