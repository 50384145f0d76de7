// sv_warp.cuh -- row merges by one warp per row, and the per-sequence
// decision grid (included by sv_rows.cu after the block-level merge code).
//
// A row merge is a chain of dependent steps (load the chunk keys, find the
// top-k threshold, gather the candidate chunks, sort, normalise).  Done by one
// warp with shuffles, ballots and __syncwarp there are no block barriers, and
// an SM holds many merges at once.  A row the warp cannot finish (more
// candidates or chunk keys than it stages) is flagged and merged by the block
// code in the decision grid.
#pragma once

namespace sv {

constexpr int WM_WARPS = 4;      // rows per CTA of the warp-merge grid
constexpr int WM_KEYS = 4096;    // chunk keys a warp stages
constexpr int WM_CAND = 256;     // candidates a warp sorts

struct __align__(16) WarpSmem {  // keys are written as 16-byte words
    uint16_t keys[WM_KEYS];
    unsigned long long cand[WM_CAND];
    unsigned long long srt[WM_CAND];
    int32_t qual[WM_CAND];
};
constexpr int WM_SMEM = WM_WARPS * (int)sizeof(WarpSmem);
static_assert(sizeof(WarpSmem) % 16 == 0, "every warp's staging must start on 16 bytes");

__device__ __forceinline__ void warp_bitonic_u64(unsigned long long* a, int n2)
{
    const int lane = threadIdx.x & 31;
    for (int k = 2; k <= n2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = lane; i < n2; i += 32) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long x = a[i], y = a[ixj];
                    if ((x > y) == ((i & k) == 0)) {
                        a[i] = y;
                        a[ixj] = x;
                    }
                }
            }
            __syncwarp();
        }
    }
}

// sort n distinct keys ascending from src to dst (per-warp shared memory)
__device__ __forceinline__ void warp_sort_keys(const unsigned long long* src, unsigned long long* dst,
                                               int n)
{
    const int lane = threadIdx.x & 31;
    if (n <= 64) {  // counting rank
        for (int i = lane; i < n; i += 32) {
            const unsigned long long x = src[i];
            int rk = 0;
            for (int j = 0; j < n; ++j) rk += src[j] < x;
            dst[rk] = x;
        }
        __syncwarp();
        return;
    }
    const int n2 = next_pow2(n);
    for (int i = lane; i < n2; i += 32) dst[i] = i < n ? src[i] : ~0ull;
    __syncwarp();
    warp_bitonic_u64(dst, n2);
}

// warp-level fast top-k (same result as fast_topk); false when the warp's
// staging overflows
template <typename T>
__device__ bool warp_fast_topk(const Params& p, const T* row, int r, WarpSmem& ws, RowStat& st)
{
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    const int V = p.V, k = p.top_k, nc = p.nchunk;
    const float c = p.c;
    using G = SegGeom<T, NT>;
    if (nc > WM_KEYS || k > WM_CAND) return false;

    // chunk keys into shared memory, 16-byte words (8 keys each), 8 loads in
    // flight per lane; each word's max (over 8 chunks, 512 bf16 / 256 f32
    // elements) stays in registers: lane l holds the maxima of words l + 32 i
    constexpr int WPL = WM_KEYS / 8 / 32;  // words per lane, at most
    const uint4* ckg = reinterpret_cast<const uint4*>(p.chunk + (int64_t)r * p.chunk_stride);
    uint4* kw = reinterpret_cast<uint4*>(ws.keys);
    const int nw = (nc + 7) / 8;
    uint32_t wm[WPL];
    uint32_t kmax = 0;
    bool bad = false;
#pragma unroll
    for (int i0 = 0; i0 < WPL; i0 += 8) {
        uint4 t[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = (i0 + q) * 32 + lane;
            t[q] = i < nw ? __ldcg(ckg + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = (i0 + q) * 32 + lane;
            uint32_t m = 0;
            if (i < nw) {
                kw[i] = t[q];
                const uint32_t w4[4] = {t[q].x, t[q].y, t[q].z, t[q].w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t key = i * 8 + e < nc ? (w4[e >> 1] >> ((e & 1) * 16)) & 0xFFFFu : 0u;
                    m = max(m, key);
                    bad |= key >= 0xFF80u;  // +inf or NaN
                }
            }
            wm[i0 + q] = m;
            kmax = max(kmax, m);
        }
        if ((i0 + 8) * 32 >= nw) {
#pragma unroll
            for (int q = i0 + 8; q < WPL; ++q) wm[q] = 0;
            break;
        }
    }
    kmax = __reduce_max_sync(FULL, kmax);
    if (__any_sync(FULL, bad) || kmax <= 0x007Fu) {
        st.flags = FLAG_NONFINITE;
        return true;
    }
    __syncwarp();
    // tau1 = the k-th largest word max: each word max is an element, so k
    // elements are >= tau1 and every top-k element is >= tau1 (binary search)
    uint32_t tau1 = 0;
    if (nw >= k) {
        uint32_t lo = 0, hi = kmax;
        while (lo < hi) {
            const uint32_t mid = (lo + hi + 1) >> 1;
            int cnt = 0;
#pragma unroll
            for (int q = 0; q < WPL; ++q) cnt += wm[q] >= mid;
            if (__reduce_add_sync(FULL, cnt) >= k) lo = mid;
            else hi = mid - 1;
        }
        tau1 = lo;
    }
    const uint32_t tau32 = tau1 << 16;
    // qualifying chunks: key >= tau1 inside the words whose max reaches tau1;
    // appends aggregated per warp with ballots
    int nq = 0;
#pragma unroll
    for (int q = 0; q < WPL; ++q) {
        if (q * 32 >= nw) break;  // warp-uniform
        const bool word_ok = wm[q] >= tau1 && wm[q] > 0;
        if (!__any_sync(FULL, word_ok)) continue;
        const int wi = q * 32 + lane;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const bool take = word_ok && wi * 8 + e < nc && ws.keys[wi * 8 + e] >= tau1;
            const unsigned bal = __ballot_sync(FULL, take);
            if (nq + __popc(bal) > WM_CAND) return false;
            if (take) ws.qual[nq + __popc(bal & ((1u << lane) - 1u))] = wi * 8 + e;
            nq += __popc(bal);
        }
    }
    __syncwarp();
    // gather the qualifying chunks as 16-byte words, 8 loads in flight per lane;
    // a word is checked whole, its kept elements appended with ballots
    constexpr int WPC = CHUNK_BYTES / 16;
    constexpr int EPW = 16 / (int)sizeof(T);
    const int nwords = nq * WPC;
    const bool aligned = ((uintptr_t)row & 15u) == 0;
    int n = 0;
#pragma unroll 1
    for (int b0 = 0; b0 < nwords; b0 += 32 * 8) {
        uint4 gw[8];
        int gi[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const int wi = b0 + g * 32 + lane;
            gi[g] = -1;
            gw[g] = make_uint4(0, 0, 0, 0);
            if (wi < nwords) {
                const int e0 = ws.qual[wi / WPC] * G::CHUNK_EL + (wi % WPC) * EPW;
                if (e0 < V) {
                    gi[g] = e0;
                    gw[g] = aligned ? __ldcg(reinterpret_cast<const uint4*>(row + e0))
                                    : Vec16<T>::load_scalar(row, e0, V);
                }
            }
        }
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const bool word_ok = gi[g] >= 0 && key_of(Vec16<T>::vmax(gw[g])) >= tau32;
            if (!__any_sync(FULL, word_ok)) continue;
#pragma unroll
            for (int q = 0; q < EPW; ++q) {
                const uint32_t key = key_of(word_elem<T>(gw[g], q));
                const bool take = word_ok && gi[g] + q < V && key >= tau32;
                const unsigned bal = __ballot_sync(FULL, take);
                if (n + __popc(bal) > WM_CAND) return false;
                if (take)
                    ws.cand[n + __popc(bal & ((1u << lane) - 1u))] =
                        ((unsigned long long)(~key) << 32) | (uint32_t)(gi[g] + q);
                n += __popc(bal);
            }
        }
    }
    __syncwarp();
    __syncwarp();
    // exact order: key descending, then id ascending
    warp_sort_keys(ws.cand, ws.srt, n);
    const int kk = min(k, n);
    const float M = val_of(~(uint32_t)(ws.srt[0] >> 32));
    float e_loc = 0.f;
    for (int i = lane; i < kk; i += 32) e_loc += ex2_fast((val_of(~(uint32_t)(ws.srt[i] >> 32)) - M) * c);
    double S = warp_sum_d((double)e_loc);
    int nk = kk;
    if (p.top_p < 1.0f) {
        double pre = 0.0;
        int stop = kk;
        for (int b0 = 0; b0 < kk; b0 += 32) {
            const int i = b0 + lane;
            const double pv =
                i < kk ? (double)ex2_fast((val_of(~(uint32_t)(ws.srt[i] >> 32)) - M) * c) / S : 0.0;
            double x = pv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(FULL, x, o);
                if (lane >= o) x += y;
            }
            const double before = pre + (x - pv);  // mass strictly before rank i
            const unsigned drop = __ballot_sync(FULL, i < kk && !(before < (double)p.top_p));
            if (drop) {
                stop = b0 + __ffs(drop) - 1;
                break;
            }
            pre += __shfl_sync(FULL, x, 31);
        }
        nk = stop;
        float e2 = 0.f;
        for (int i = lane; i < nk; i += 32) e2 += ex2_fast((val_of(~(uint32_t)(ws.srt[i] >> 32)) - M) * c);
        S = warp_sum_d((double)e2);
    }
    // the kept list in ascending id
    for (int i = lane; i < nk; i += 32) {
        const unsigned long long x = ws.srt[i];
        ws.cand[i] = ((unsigned long long)(uint32_t)x << 32) | (uint32_t)(~(uint32_t)(x >> 32));
    }
    __syncwarp();
    warp_sort_keys(ws.cand, ws.srt, nk);
    int32_t* kid = p.kept_id + (int64_t)r * KCAP;
    float* kl = p.kept_l + (int64_t)r * KCAP;
    for (int i = lane; i < nk; i += 32) {
        const unsigned long long x = ws.srt[i];
        kid[i] = (int32_t)(x >> 32);
        kl[i] = val_of((uint32_t)x);
    }
    st.M = M;
    st.S = S;
    st.n_kept = nk;
    st.mode = MODE_LIST;
    return true;
}

// statistics over all tokens (no knobs) from the segment records, by one warp
__device__ __forceinline__ void warp_all_stats(const Params& p, int r, RowStat& st)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    float m = -INFINITY;
    for (int i = lane; i < p.nseg; i += 32) m = fmax_nan(m, __ldcg(&p.seg[(int64_t)r * p.nseg + i].m));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmax_nan(m, __shfl_xor_sync(FULL, m, o));
    if (!(m > -INFINITY && m < INFINITY)) {
        st.flags = FLAG_NONFINITE;
        return;
    }
    double s = 0.0;
    for (int i = lane; i < p.nseg; i += 32) {
        const SegStat* g = p.seg + (int64_t)r * p.nseg + i;
        const float gm = __ldcg(&g->m);
        if (gm > -INFINITY) s += __ldcg(&g->s) * exp2(((double)gm - (double)m) * (double)p.c);
    }
    st.M = m;
    st.S = warp_sum_d(s);
    st.mode = MODE_ALL;
    st.n_kept = p.V;
}

// ------------------------------------------------------------------------- //
// k_merge_warp: one warp per row slot (after the stream grid)                //
// ------------------------------------------------------------------------- //
template <typename T>
__global__ void __launch_bounds__(WM_WARPS * 32) k_merge_warp(const Params p)
{
    extern __shared__ __align__(16) unsigned char smem_w[];
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream grid has completed
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * WM_WARPS + warp;
    if (r >= p.B * p.rps) return;
    const RowRef rr = row_ref(p, r);
    if (!rr.valid) {
        if (lane == 0) report_skipped_row(p, rr);
        return;
    }
    if (rr.is_draft && p.draft_kind == 1) return;
    WarpSmem& ws = reinterpret_cast<WarpSmem*>(smem_w)[warp];
    const T* row = (const T*)(rr.is_draft ? p.draft : p.target) + row_elem_offset(p, rr);
    RowStat st;
    st.M = -INFINITY;
    st.kappa = 0;
    st.S = 0.0;
    st.i_kappa = p.V - 1;
    st.n_kept = p.V;
    st.mode = MODE_ALL;
    st.flags = 0;
    if (p.seg_mode == SEG_CHUNK) {
        if (!warp_fast_topk<T>(p, row, r, ws, st)) st.flags |= FLAG_BLOCK_MERGE;
    } else {
        warp_all_stats(p, r, st);
    }
    if (lane == 0) p.rstat[r] = st;
}

// ------------------------------------------------------------------------- //
// k_decide: one CTA per sequence: rows the warp merge flagged are merged by  //
// the block code, then the sequence is decided                              //
// ------------------------------------------------------------------------- //
template <typename T>
__global__ void __launch_bounds__(NT) k_decide(const Params p)
{
    extern __shared__ __align__(16) unsigned char smem_scratch[];  // SCRATCH_BYTES
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the merge grid has completed
    const int b = blockIdx.x;
    const int kb = seq_k(p, b);
    if (!k_ok(p, kb)) return;  // reported by the merge grid
    const int nrows = p.draft_kind == 0 ? 2 * kb + 1 : kb + 1;
    // which rows the warps left to the block code (bitmask, one load round)
    __shared__ unsigned s_flagged[(2 * 255 + 1 + 31) / 32];
    for (int i = threadIdx.x; i < (nrows + 31) / 32; i += NT) s_flagged[i] = 0u;
    csync();
    for (int i = threadIdx.x; i < nrows; i += NT) {
        const int r = i <= kb ? target_slot(p, b, i) : draft_slot(p, b, i - kb - 1);
        if (load_rowstat(p.rstat + r).flags & FLAG_BLOCK_MERGE) atomicOr(&s_flagged[i >> 5], 1u << (i & 31));
    }
    csync();
    bool merged = false;
    for (int i = 0; i < nrows; ++i) {
        if (!(s_flagged[i >> 5] & (1u << (i & 31)))) continue;
        const int r = i <= kb ? target_slot(p, b, i) : draft_slot(p, b, i - kb - 1);
        const RowRef rr = row_ref(p, r);
        const T* row = (const T*)(rr.is_draft ? p.draft : p.target) + row_elem_offset(p, rr);
        merge_row<T>(p, row, r, smem_scratch);
        csync();
        merged = true;
    }
    if (merged) {
        if (threadIdx.x == 0) __threadfence();
        csync();
    }
    decide_sequence<T>(p, b, smem_scratch);
}

}  // namespace sv
