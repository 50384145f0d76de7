// sv_mcand.cuh -- the row merge of the candidate path, one CTA per row slot
// (included by sv_rows.cu after the candidate stream kernel).
//
// A row's candidates (every logit at or above a lower bound of its k-th
// largest, see sv_cand.cuh) sit in a flat array with the row's control words.
// MC_T threads load them in one round, keep those at or above the row's final
// bound, rank the survivors in the exact order (logit descending, token id
// ascending: one rank per thread by counting), take the first k, the top-p
// prefix in rank order, and write the kept list in ascending id with M, S and
// P(x) at the drafted token.  The last row of a sequence to finish decides
// the sequence (warp 0, the decision of sv_warp.cuh).  Rows whose candidates
// were lost take the chunk-key warp merge; rows that one cannot finish are
// left to the decision grid.
#pragma once

namespace sv {

constexpr int MC_T = 128;       // threads per row
constexpr int MC_CAP = 256;     // survivors a row can stage
constexpr int MC_PRE = 3;       // candidate words per thread loaded before the count is known
static_assert(MC_T * MC_PRE * 2 >= 768, "the prefetch covers the usual candidate count");
static_assert(CAND_TOPK_MAX <= MC_T, "one kept rank per thread");

struct McSmem {
    WarpSmem ws;                      // warp 0: chunk-key merge and the decision
    unsigned long long cand[MC_CAP];  // survivors: (~order key) << 32 | token id
    unsigned long long ord[MC_CAP];   // the survivors in rank order
    float redf[MC_T / 32];
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
    // every load that does not depend on another goes out at once
    const int b = r / p.rps, slot = r - b * p.rps;
    const int jd = slot > p.Kmax ? slot - (p.Kmax + 1) : slot;  // position of the row
    const int x_raw = jd < p.Kmax ? __ldg(p.xin + (int64_t)b * p.Kmax + jd) : -1;
    unsigned* ctl = p.rowctl + (int64_t)r * 4;
    const uint4 c4 = __ldcg(reinterpret_cast<const uint4*>(ctl));
    const uint4* src = reinterpret_cast<const uint4*>(p.cand_rows + (int64_t)r * RCAP_ROW);
    uint4 pre[MC_PRE];
#pragma unroll
    for (int g = 0; g < MC_PRE; ++g) pre[g] = __ldcg(src + g * MC_T + tid);
    const RowRef rr = row_ref(p, r);
    if (!rr.valid) {
        if (tid == 0) report_skipped_row(p, rr);
        return;
    }
    if (rr.is_draft && p.draft_kind == 1) return;
    const uint32_t cnt = c4.x, tau = c4.y, maxkey = c4.z;
    if (tid == 0) sm.n = 0;
    __syncthreads();  // every thread has its copy of the control words
    if (tid == 0) *reinterpret_cast<uint4*>(ctl) = make_uint4(0, 0, 0, 0);
    const T* row = (const T*)(rr.is_draft ? p.draft : p.target) + row_elem_offset(p, rr);
    const int x = (rr.j < rr.kb && x_raw >= 0 && x_raw < p.V) ? x_raw : -1;
    const int k = p.top_k;

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
                const unsigned bal = __ballot_sync(FULL, take);
                if (bal) {
                    const int leader = __ffs(bal) - 1;
                    int base = 0;
                    if (lane == leader) base = atomicAdd(&sm.n, __popc(bal));
                    base = __shfl_sync(FULL, base, leader);
                    const int pos = base + __popc(bal & ((1u << lane) - 1u));
                    if (take && pos < MC_CAP)
                        sm.cand[pos] = ((unsigned long long)(~key) << 32) | id;
                }
            }
        };
#pragma unroll
        for (int g = 0; g < MC_PRE; ++g) append(pre[g], g * MC_T + tid);
        for (int w0 = MC_PRE * MC_T; w0 < nw; w0 += MC_T) {
            const int wi = w0 + tid;
            append(wi < nw ? __ldcg(src + wi) : make_uint4(0, 0, 0, 0), wi);
        }
        __syncthreads();
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
