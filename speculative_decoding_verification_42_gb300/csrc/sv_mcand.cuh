// sv_mcand.cuh -- the row merge of the top-k rows, one CTA per row slot
// (included by sv_rows.cu after the candidate stream kernel).
//
// The CTA first gathers the row's candidates: every logit at or above a lower
// bound of its k-th largest.  Two sources:
//  * gather (after the chunk-key stream): the k-th largest of the row's
//    128-byte chunk maxima (their 16-bit order keys counted in a window of
//    MCG_HB keys below the largest) bounds the k-th largest logit from
//    below, since k chunks each hold a logit at least that large; the chunks
//    reaching it are read back from HBM and their logits at or above it
//    kept, each list compacted with one block-wide prefix sum;
//  * stream (after sv_cand.cuh): the candidates the stream wrote to the row's
//    flat array, kept if at or above the row's final bound.
// Then it ranks the survivors in the exact order (logit descending, token id
// ascending: one rank per thread by counting), takes the first k, the top-p
// prefix in rank order, and writes the kept list in ascending id with M, S and
// P(x) at the drafted token.  The last row of a sequence to finish decides
// the sequence (warp 0, the decision of sv_warp.cuh).  Rows with too many
// candidates (ties) take the chunk-key warp merge; rows that one cannot
// finish are left to the decision grid.
#pragma once

namespace sv {

constexpr int MC_T = 128;       // threads per row
constexpr int MC_CAP = 256;     // survivors a row can stage
constexpr int MC_PRE = 3;       // candidate words per thread loaded before the count is known
constexpr int MCG_U4 = 4;       // gather: 16-byte words of chunk keys per thread (8 keys each)
constexpr int MCG_QCAP = 512;   // gather: qualifying chunks a row can stage
constexpr int MCG_LPT = 4;      // gather: chunk words per thread per load round
constexpr int MCG_HB = 1024;    // gather: histogram bins (keys below the row's largest chunk key)
constexpr int MCG_BPT = MCG_HB / MC_T;  // bins a thread sums
static_assert(MC_T * MC_PRE * 2 >= 768, "the prefetch covers the usual candidate count");
static_assert(CAND_TOPK_MAX <= MC_T, "one kept rank per thread");
static_assert(MC_T * MCG_U4 * 8 >= 4096, "the gather holds every chunk key of a warp-merge row");

struct McSmem {
    WarpSmem ws;                      // warp 0: chunk-key merge and the decision
    unsigned long long cand[MC_CAP];  // survivors: (~order key) << 32 | token id
    unsigned long long ord[MC_CAP];   // the survivors in rank order
    float redf[MC_T / 32];
    uint32_t hist[MCG_HB];            // gather: chunk keys at (largest key - bin)
    uint32_t qc[MCG_QCAP];            // gather: qualifying chunks
    uint32_t sel[4];                  // gather: the row's largest chunk key, the bound
    int redi[MC_T / 32];
    int nq;                           // gather: qualifying chunks (may pass MCG_QCAP)
    int n;                            // survivors staged (may pass MC_CAP)
    int stop;                         // first rank the top-p prefix drops
    float px;
    int last;
    RowStat st;
};

// block sum of one value per thread (a tree of fp32 additions: at most k <=
// 128 terms in [0, 1], relative error ~1e-7); all threads get the sum
__device__ __forceinline__ float mc_sum(float v, float* red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    return (red[0] + red[1]) + (red[2] + red[3]);
}
static_assert(MC_T == 128, "mc_sum adds four warp sums");

// block-wide exclusive prefix sum of one int per thread (all MC_T threads);
// *total gets the sum.  Two barriers; red may be reused after it returns.
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
    __syncthreads();
    int before = 0;
#pragma unroll
    for (int w = 0; w < MC_T / 32; ++w) before += w < warp ? red[w] : 0;
    *total = red[0] + red[1] + red[2] + red[3];
    __syncthreads();
    return before + x - v;
}

// append v to arr (capacity cap) where take, one atomic per warp; every lane
// of the warp calls it
template <typename E>
__device__ __forceinline__ void mc_append(bool take, E v, int* count, E* arr, int cap)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const unsigned bal = __ballot_sync(FULL, take);
    if (!bal) return;
    const int leader = __ffs(bal) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(count, __popc(bal));
    base = __shfl_sync(FULL, base, leader);
    const int pos = base + __popc(bal & ((1u << lane) - 1u));
    if (take && pos < cap) arr[pos] = v;
}

template <typename T>
__global__ void __launch_bounds__(MC_T, 8) k_merge_cand(const Params p)
{
    __shared__ McSmem sm;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream grid has completed
    // the decision grid may be scheduled now; it waits for this grid's end
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const unsigned FULL = 0xffffffffu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x;
    const bool gather = p.gather != 0;
    // every load that does not depend on another goes out at once
    const int b = r / p.rps, slot = r - b * p.rps;
    const int jd = slot > p.Kmax ? slot - (p.Kmax + 1) : slot;  // position of the row
    const int x_raw = jd < p.Kmax ? __ldg(p.xin + (int64_t)b * p.Kmax + jd) : -1;
    unsigned* ctl = p.rowctl + (int64_t)r * 4;
    const uint4* src = reinterpret_cast<const uint4*>(p.cand_rows + (int64_t)r * RCAP_ROW);
    const uint4* ksrc = reinterpret_cast<const uint4*>(p.chunk + (int64_t)r * p.chunk_stride);
    const int nch = p.nchunk;
    uint4 c4 = make_uint4(0, 0, 0, 0);
    uint4 pre[MC_PRE];  // stream: candidate words; gather: chunk-key words
    static_assert(MC_PRE >= MCG_U4 - 1, "the prefetch registers hold the chunk keys");
    uint4 kq_last = make_uint4(0, 0, 0, 0);
    if (gather) {
#pragma unroll
        for (int g = 0; g < MC_PRE; ++g)
            pre[g] = (g * MC_T + tid) * 8 < nch ? __ldcg(ksrc + g * MC_T + tid) : make_uint4(0, 0, 0, 0);
        if ((MC_PRE * MC_T + tid) * 8 < nch) kq_last = __ldcg(ksrc + MC_PRE * MC_T + tid);
    } else {
        c4 = __ldcg(reinterpret_cast<const uint4*>(ctl));
#pragma unroll
        for (int g = 0; g < MC_PRE; ++g) pre[g] = __ldcg(src + g * MC_T + tid);
    }
    const RowRef rr = row_ref(p, r);
    if (!rr.valid) {
        if (tid == 0) report_skipped_row(p, rr);
        return;
    }
    if (rr.is_draft && p.draft_kind == 1) return;
    const T* row = (const T*)(rr.is_draft ? p.draft : p.target) + row_elem_offset(p, rr);
    const int x = (rr.j < rr.kb && x_raw >= 0 && x_raw < p.V) ? x_raw : -1;
    const int k = p.top_k;
    if (tid == 0) {
        sm.n = 0;
        sm.nq = 0;
        sm.sel[2] = 0u;
    }
    if (gather) {
#pragma unroll
        for (int i = 0; i < MCG_BPT; ++i) sm.hist[i * MC_T + tid] = 0u;
    }
    __syncthreads();  // every thread has its copy of the control words
    if (!gather && tid == 0) *reinterpret_cast<uint4*>(ctl) = make_uint4(0, 0, 0, 0);

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
    bool chunk_path = false;
    bool staged = false;  // survivors are in sm.cand (sm.n of them)
    if (gather) {
        // ---- the row's chunk keys: key 8 (g MC_T + tid) + i is half i of word g
        auto key_at = [&](int g, int i) -> uint32_t {
            const uint4 w = g < MC_PRE ? pre[g] : kq_last;
            const uint32_t u = (i >> 1) == 0 ? w.x : (i >> 1) == 1 ? w.y : (i >> 1) == 2 ? w.z : w.w;
            return (i & 1) ? (u >> 16) : (u & 0xFFFFu);
        };
        auto key_in = [&](int g, int i) { return (g * MC_T + tid) * 8 + i < nch; };
        uint32_t kmax = 0u;
#pragma unroll
        for (int g = 0; g < MCG_U4; ++g)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (key_in(g, i)) kmax = max(kmax, key_at(g, i));
        kmax = __reduce_max_sync(FULL, kmax);
        if (lane == 0) atomicMax(&sm.sel[2], kmax);
        __syncthreads();
        const uint32_t maxkey = sm.sel[2];
        if (maxkey >= 0xFF80u || maxkey <= 0x007Fu) {  // NaN or +inf, or no finite logit
            st.flags = FLAG_NONFINITE;
        } else {
            // ---- the k-th largest chunk key: keys counted at (maxkey - key)
#pragma unroll
            for (int g = 0; g < MCG_U4; ++g)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t d = maxkey - key_at(g, i);
                    if (key_in(g, i) && d < (uint32_t)MCG_HB) atomicAdd(&sm.hist[d], 1u);
                }
            __syncthreads();
            uint32_t hb[MCG_BPT];
            int local = 0;
#pragma unroll
            for (int i = 0; i < MCG_BPT; ++i) {
                hb[i] = sm.hist[tid * MCG_BPT + i];
                local += (int)hb[i];
            }
            int in_window;
            const int before = mc_excl_scan(local, sm.redi, &in_window);
            if (tid == 0) sm.sel[3] = 0u;
            __syncthreads();
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
            __syncthreads();
            // fewer than k chunks in the window: every chunk may hold a top-k logit
            const uint32_t tau_c = in_window >= k ? sm.sel[3] : 0u;
            // ---- the chunks reaching it (at least k of them), compacted
            uint32_t qmask = 0u;
#pragma unroll
            for (int g = 0; g < MCG_U4; ++g)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (key_in(g, i) && key_at(g, i) >= tau_c) qmask |= 1u << (g * 8 + i);
            int nq;
            int at = mc_excl_scan(__popc(qmask), sm.redi, &nq);
            while (qmask) {
                const int bit = __ffs(qmask) - 1;
                qmask &= qmask - 1u;
                if (at < MCG_QCAP) sm.qc[at] = (uint32_t)(((bit >> 3) * MC_T + tid) * 8 + (bit & 7));
                ++at;
            }
            __syncthreads();
            if (nq > MCG_QCAP) {
                chunk_path = true;  // ties: too many chunks reach the bound
            } else {
                // ---- read the chunks back; keep their logits at or above the bound
                constexpr int VW = Vec16<T>::N;
                constexpr int CWD = CHUNK_BYTES / 16;  // words per chunk
                const uint4* rowv = reinterpret_cast<const uint4*>(row);
                const int nw_row = p.V / VW;          // whole words: V s is a multiple of 16 here
                int nsurv = 0;
                for (int w0 = 0; w0 < nq * CWD; w0 += MC_T * MCG_LPT) {
                    uint4 wv[MCG_LPT];
                    int wi[MCG_LPT];
#pragma unroll
                    for (int j = 0; j < MCG_LPT; ++j) {
                        const int i = w0 + j * MC_T + tid;
                        wi[j] = -1;
                        wv[j] = make_uint4(0, 0, 0, 0);
                        if (i < nq * CWD) {
                            const int word = (int)sm.qc[i / CWD] * CWD + i % CWD;
                            if (word < nw_row) {
                                wi[j] = word;
                                wv[j] = __ldcg(rowv + word);
                            }
                        }
                    }
                    uint32_t em[MCG_LPT];
                    int cnt = 0;
#pragma unroll
                    for (int j = 0; j < MCG_LPT; ++j) {
                        em[j] = 0u;
#pragma unroll
                        for (int q = 0; q < VW; ++q)
                            if (wi[j] >= 0 && (key_of(word_elem_rt<T>(wv[j], q)) >> 16) >= tau_c)
                                em[j] |= 1u << q;
                        cnt += __popc(em[j]);
                    }
                    int tot;
                    int pos = nsurv + mc_excl_scan(cnt, sm.redi, &tot);
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
                    nsurv += tot;
                }
                if (tid == 0) sm.n = nsurv;
                __syncthreads();
                staged = true;
            }
        }
    } else {
        const uint32_t cnt = c4.x, tau = c4.y, maxkey = c4.z;
        if (maxkey >= 0xFF80u || maxkey <= 0x007Fu) {  // NaN or +inf, or no finite logit
            st.flags = FLAG_NONFINITE;
        } else if (cnt > (uint32_t)RCAP_ROW || cnt == 0u) {
            chunk_path = true;
        } else {
            // ---- survivors: candidates at or above the row's bound (unused
            //      slots have token id ~0), appended with warp-aggregated atomics
            const int nw = (int)((cnt + 1u) / 2u);
            auto append = [&](const uint4& w, int wi) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t key = h ? w.w : w.y;
                    const uint32_t id = h ? w.z : w.x;
                    const bool take = wi < nw && 2 * wi + h < (int)cnt && id < (uint32_t)p.V &&
                                      (key >> 16) >= tau;
                    mc_append<unsigned long long>(take, ((unsigned long long)(~key) << 32) | id, &sm.n,
                                                  sm.cand, MC_CAP);
                }
            };
#pragma unroll
            for (int g = 0; g < MC_PRE; ++g) append(pre[g], g * MC_T + tid);
            for (int w0 = MC_PRE * MC_T; w0 < nw; w0 += MC_T) {
                const int wi = w0 + tid;
                append(wi < nw ? __ldcg(src + wi) : make_uint4(0, 0, 0, 0), wi);
            }
            __syncthreads();
            staged = true;
        }
    }
    if (staged) {
        const int n = sm.n;
        if (n > MC_CAP || n < 1) {
            chunk_path = true;  // more survivors than staged (ties), or none
        } else {
            // ---- exact rank of every survivor (keys are distinct: ids are)
            for (int i = tid; i < n; i += MC_T) {
                const unsigned long long v = sm.cand[i];
                int rank = 0;
                for (int j = 0; j < n; ++j) rank += sm.cand[j] < v;
                sm.ord[rank] = v;
            }
            if (tid == 0) sm.stop = INT_MAX;
            __syncthreads();
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
                __syncthreads();
                if (lane == 31) sm.redf[warp] = y;
                __syncthreads();
                float before = y - pv;
                for (int i = 0; i < warp; ++i) before += sm.redf[i];
                if (tid < kk && !(before < p.top_p)) atomicMin(&sm.stop, tid);
                __syncthreads();
                nk = min(sm.stop, kk);  // the first rank whose mass before it reaches top_p
                S = mc_sum(tid < nk ? et : 0.f, sm.redf);
            }
            const float invS = 1.f / S;
            // ---- the kept list in ascending id, P(x)
            if (tid == 0) sm.px = 0.f;
            __syncthreads();
            if (tid < nk) {
                int pos = 0;
                for (int j = 0; j < nk; ++j) pos += (int)(uint32_t)sm.ord[j] < idt;
                p.kept_id[(int64_t)r * KCAP + pos] = idt;
                p.kept_l[(int64_t)r * KCAP + pos] = lt;
                if (idt == x) sm.px = exp2f((lt - M) * c) * invS;
            }
            __syncthreads();
            st.M = M;
            st.S = (double)S;
            st.n_kept = nk;
            st.mode = MODE_LIST;
            st.px = sm.px;
        }
    }
    if (chunk_path) {
        // the chunk-key merge by warp 0 (the candidates were lost or too many)
        if (warp == 0) {
            if (!warp_fast_topk<T>(p, row, r, x, sm.ws, st)) st.flags |= FLAG_BLOCK_MERGE;
            if (lane == 0) sm.st = st;
        }
        __syncthreads();
        st = sm.st;
    }
    if (tid == 0) p.rstat[r] = st;
    // sequence ticket: the barrier orders every thread's writes before thread
    // 0's fence, which makes them visible before the ticket is taken
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const int nrows = (rr.kb + 1) + (p.draft_kind == 0 ? rr.kb : 0);
        sm.last = atomicAdd(&p.seq_ticket[rr.b], 1u) == (unsigned)(nrows - 1);
        if (sm.last) p.seq_ticket[rr.b] = 0u;
    }
    __syncthreads();
    if (!sm.last || warp != 0) return;
    if (lane == 0) __threadfence();
    __syncwarp();
    const int nrows_b = p.draft_kind == 0 ? 2 * rr.kb + 1 : rr.kb + 1;
    if (nrows_b <= 32 ? warp_decide_lanes<T>(p, rr.b, rr.kb, sm.ws) : warp_decide<T>(p, rr.b, sm.ws)) {
        __syncwarp();
        if (lane == 0) p.seq_done[rr.b] = 1u;
    }
}

}  // namespace sv
