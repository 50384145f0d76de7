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
// a warp's share of the merge grid's shared memory: the whole WarpSmem for
// chunk-key rows (the top-k gather stages candidates), its key staging alone
// otherwise (histograms, the decision's lists), so that more rows fit an SM
__host__ __device__ constexpr int wm_stride(int seg_mode)
{
    return seg_mode == SEG_CHUNK ? (int)sizeof(WarpSmem) : (int)sizeof(WarpSmem::keys);
}
static_assert(sizeof(WarpSmem::keys) % 16 == 0, "every warp's staging must start on 16 bytes");
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
    if (n <= 128) {  // counting rank
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

// exclusive prefix sum over the warp; *total gets the sum of all lanes
__device__ __forceinline__ int warp_excl_scan(int v, int* total)
{
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if ((threadIdx.x & 31) >= o) x += y;
    }
    *total = __shfl_sync(0xffffffffu, x, 31);
    return x - v;
}

// P(x) of a merged row, the same arithmetic the decisions use
__device__ __forceinline__ float row_prob(const Params& p, float l, float M, double S)
{
    return (float)((double)exp2f((l - M) * p.c) / S);
}

// The n candidates in ws.cand (sort keys (~order key) << 32 | id, a superset
// of the top-k) become the row's kept list: exact order (key descending, id
// ascending), the first k, the top-p prefix, then the list in ascending id
// written to the workspace with M, S and P(x) of the drafted token x (x < 0:
// none).
__device__ void warp_topk_tail(const Params& p, int r, WarpSmem& ws, int n, int x, RowStat& st)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const float c = p.c;
    warp_sort_keys(ws.cand, ws.srt, n);
    const int kk = min(p.top_k, n);
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
            double y = pv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double t = __shfl_up_sync(FULL, y, o);
                if (lane >= o) y += t;
            }
            const double before = pre + (y - pv);  // mass strictly before rank i
            const unsigned drop = __ballot_sync(FULL, i < kk && !(before < (double)p.top_p));
            if (drop) {
                stop = b0 + __ffs(drop) - 1;
                break;
            }
            pre += __shfl_sync(FULL, y, 31);
        }
        nk = stop;
        float e2 = 0.f;
        for (int i = lane; i < nk; i += 32) e2 += ex2_fast((val_of(~(uint32_t)(ws.srt[i] >> 32)) - M) * c);
        S = warp_sum_d((double)e2);
    }
    // the kept list in ascending id
    for (int i = lane; i < nk; i += 32) {
        const unsigned long long v = ws.srt[i];
        ws.cand[i] = ((unsigned long long)(uint32_t)v << 32) | (uint32_t)(~(uint32_t)(v >> 32));
    }
    __syncwarp();
    warp_sort_keys(ws.cand, ws.srt, nk);
    int32_t* kid = p.kept_id + (int64_t)r * KCAP;
    float* kl = p.kept_l + (int64_t)r * KCAP;
    float lx = 0.f;
    bool found = false;
    for (int i = lane; i < nk; i += 32) {
        const unsigned long long v = ws.srt[i];
        const int id = (int)(v >> 32);
        const float l = val_of((uint32_t)v);
        kid[i] = id;
        kl[i] = l;
        if (id == x) {
            found = true;
            lx = l;
        }
    }
    const unsigned hit = __ballot_sync(FULL, found);
    lx = __shfl_sync(FULL, lx, hit ? __ffs(hit) - 1 : 0);
    st.M = M;
    st.S = S;
    st.n_kept = nk;
    st.mode = MODE_LIST;
    st.px = hit ? row_prob(p, lx, M, S) : 0.f;
}

// warp-level fast top-k (same result as fast_topk); false when the warp's
// staging overflows
template <typename T>
__device__ bool warp_fast_topk(const Params& p, const T* row, int r, int x, WarpSmem& ws, RowStat& st)
{
    const int lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    const int V = p.V, k = p.top_k, nc = p.nchunk;
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
    warp_topk_tail(p, r, ws, n, x, st);
    return true;
}

// statistics over all tokens (no knobs) from the segment records, by one warp
__device__ __forceinline__ void warp_all_stats(const Params& p, int r, RowStat& st)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    constexpr int PER = 16;  // segment records a lane holds (one round of loads)
    const uint4* seg = reinterpret_cast<const uint4*>(p.seg + (int64_t)r * p.nseg);
    float m = -INFINITY;
    double s = 0.0;
    for (int i0 = 0; i0 < p.nseg; i0 += 32 * PER) {
        uint4 w[PER];
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int i = i0 + k * 32 + lane;
            w[k] = i < p.nseg ? __ldcg(seg + i) : make_uint4(0xFF800000u, 0u, 0u, 0u);  // (-inf, 0)
        }
        float mb = -INFINITY;
#pragma unroll
        for (int k = 0; k < PER; ++k) mb = fmax_nan(mb, __uint_as_float(w[k].x));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mb = fmax_nan(mb, __shfl_xor_sync(FULL, mb, o));
        const float nm = fmax_nan(m, mb);
        if (!(nm > -INFINITY && nm < INFINITY)) {
            m = nm;
            continue;  // no finite maximum yet (or NaN / +inf: flagged below)
        }
        if (m > -INFINITY) s *= (double)exp2f((m - nm) * p.c);
        m = nm;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const float gm = __uint_as_float(w[k].x);
            const double gs = __hiloint2double((int)w[k].w, (int)w[k].z);
            if (gm > -INFINITY) s += gs * (double)exp2f((gm - m) * p.c);
        }
    }
    if (!(m > -INFINITY && m < INFINITY)) {
        st.flags = FLAG_NONFINITE;
        return;
    }
    st.M = m;
    st.S = warp_sum_d(s);
    st.mode = MODE_ALL;
    st.n_kept = p.V;
}

// ------------------------------------------------------------------------- //
// the decision of one sequence by one warp, inside the merge grid: every row //
// record carries P(x_j), so the accept tests need no lookups; the emitted    //
// token is drawn from the target's kept list (residual or bonus) by inverse  //
// CDF in fixed point, or posted as a job for the full-row sampler.           //
// ------------------------------------------------------------------------- //
template <typename T>
__device__ int warp_sample_list(const Params& p, int tr, const RowStat& ts, bool residual,
                                const DraftRef& d, float u, unsigned char* stage,
                                unsigned long long* Zfix, bool* zero)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int n = ts.n_kept;  // <= WM_CAND in the warp path
    // stage: 4 WM_CAND words (16-byte aligned) for the two lists
    int32_t* ti = reinterpret_cast<int32_t*>(stage);
    float* tv = reinterpret_cast<float*>(stage) + WM_CAND;
    int32_t* di = reinterpret_cast<int32_t*>(stage) + 2 * WM_CAND;
    float* dv = reinterpret_cast<float*>(stage) + 3 * WM_CAND;
    static_assert(4 * WM_CAND * 4 <= (int)sizeof(WarpSmem::keys), "two staged lists fit the key staging");
    StagedList tl{ti, tv, n}, dl{di, dv, 0};
    {
        const int32_t* gi = p.kept_id + (int64_t)tr * KCAP;
        const float* gv = p.kept_l + (int64_t)tr * KCAP;
        for (int i = lane; i < n; i += 32) {
            ti[i] = __ldcg(gi + i);
            tv[i] = __ldcg(gv + i);
        }
        if (residual && d.kind == 0 && d.st.mode == MODE_LIST) {
            dl.n = d.st.n_kept;
            const int32_t* hi = p.kept_id + (int64_t)d.r * KCAP;
            const float* hv = p.kept_l + (int64_t)d.r * KCAP;
            for (int i = lane; i < dl.n; i += 32) {
                di[i] = __ldcg(hi + i);
                dv[i] = __ldcg(hv + i);
            }
        }
        __syncwarp();
    }
    const float invSt = 1.f / (float)ts.S;
    const float invSd = (residual && d.kind == 0) ? 1.f / (float)d.st.S : 0.f;
    const int ept = (n + 31) / 32;
    const int i0 = lane * ept;
    *zero = false;
    for (int attempt = 0; attempt < 2; ++attempt) {
        const bool res = residual && attempt == 0;
        unsigned long long part = 0;
        for (int q = 0; q < ept; ++q) {
            const int i = i0 + q;
            if (i >= n) break;
            part += list_r_fix<T>(p, ts, tl, i, res, d, dl, invSt, invSd);
        }
        unsigned long long incl = part;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned long long Z = __shfl_sync(FULL, incl, 31);
        const unsigned long long ex = incl - part;
        if (attempt == 0) *Zfix = Z;
        if (Z == 0ull) {
            if (res) {
                *zero = true;
                continue;
            }
            return -1;
        }
        const unsigned long long t = cdf_target(u, Z);
        int tok = -1;
        if (ex <= t && t < ex + part) {
            unsigned long long acc = ex;
            for (int q = 0; q < ept; ++q) {
                const int i = i0 + q;
                if (i >= n) break;
                acc += list_r_fix<T>(p, ts, tl, i, res, d, dl, invSt, invSd);
                if (acc > t) {
                    tok = tl.ids[i];
                    break;
                }
            }
        }
        return __reduce_max_sync(FULL, tok);
    }
    return -1;
}

// a row record held in registers (three 16-byte words), as loaded by one lane
struct RecWords {
    uint4 a, b, c;
};
__device__ __forceinline__ RecWords load_rec(const RowStat* src)
{
    const uint4* s = reinterpret_cast<const uint4*>(src);
    return RecWords{__ldcg(s), __ldcg(s + 1), __ldcg(s + 2)};
}
__device__ __forceinline__ RecWords shfl_rec(const RecWords& w, int from)
{
    const unsigned FULL = 0xffffffffu;
    RecWords o;
    o.a = make_uint4(__shfl_sync(FULL, w.a.x, from), __shfl_sync(FULL, w.a.y, from),
                     __shfl_sync(FULL, w.a.z, from), __shfl_sync(FULL, w.a.w, from));
    o.b = make_uint4(__shfl_sync(FULL, w.b.x, from), __shfl_sync(FULL, w.b.y, from),
                     __shfl_sync(FULL, w.b.z, from), __shfl_sync(FULL, w.b.w, from));
    o.c = make_uint4(__shfl_sync(FULL, w.c.x, from), __shfl_sync(FULL, w.c.y, from),
                     __shfl_sync(FULL, w.c.z, from), __shfl_sync(FULL, w.c.w, from));
    return o;
}
__device__ __forceinline__ RowStat rec_stat(const RecWords& w)
{
    RowStat r;
    uint4* d = reinterpret_cast<uint4*>(&r);
    d[0] = w.a;
    d[1] = w.b;
    d[2] = w.c;
    return r;
}

// a decision that still needs its sample: the inverse CDF over the kept list
// of target row tr (its residual against the draft d, or the row itself) at u
struct DecidePending {
    int jstar;     // the emitted slot
    int tr;        // target row slot
    int residual;  // the residual of a rejection (else the bonus / greedy row)
    float u;
    RowStat ts;
    DraftRef d;
};

// the outputs of a pending decision once its sample tok is drawn (one thread)
__device__ __forceinline__ void decide_finish(const Params& p, int b, const DecidePending& pe, int tok,
                                              unsigned long long Z, bool zero)
{
    p.tokens[(int64_t)b * (p.Kmax + 1) + pe.jstar] = tok;
    p.num_accepted[b] = pe.jstar;
    if (p.row_status) p.row_status[b] = zero ? ROW_ZERO_RESIDUAL : ROW_OK;
    if (p.resid_mass) p.resid_mass[b] = pe.residual ? (float)from_fix56(Z) : 0.f;
    p.jobs[b].kind = JOB_NONE;
}

enum : int { DECIDE_LEFT = 0, DECIDE_DONE = 1, DECIDE_SAMPLE = 2 };

// the decision of sequence b by one warp when its rows fit one per lane
// (2 K_b + 1 <= 32): lane i holds row record i (target rows 0..K_b, then
// draft rows 0..K_b-1) and slot i's drafted token, all loaded in one round;
// the same arithmetic and outputs as warp_decide.  Up to the sample:
// DECIDE_LEFT (a row needs the decision grid), DECIDE_DONE, or DECIDE_SAMPLE
// with *pe (the same in every lane) to be drawn and passed to decide_finish
template <typename T>
__device__ int warp_decide_lanes_head(const Params& p, int b, int kb, DecidePending* pe)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int K = p.Kmax, V = p.V;
    const int nrows = seq_rows(p, kb);
    const int64_t drow0 = (int64_t)b * K * V;
    RecWords rw{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (lane < nrows)
        rw = load_rec(p.rstat + (lane <= kb ? target_slot(p, b, lane) : draft_slot(p, b, lane - kb - 1)));
    const int x = lane < kb ? p.xin[(int64_t)b * K + lane] : -1;
    const RowStat me = rec_stat(rw);
    const bool mine = lane < nrows;
    if (__any_sync(FULL, mine && ((me.flags & FLAG_BLOCK_MERGE) ||
                                  (me.mode == MODE_LIST && me.n_kept > WM_CAND))))
        return DECIDE_LEFT;
    bool nonf = __any_sync(FULL, mine && (me.flags & FLAG_NONFINITE));
    const bool bad = __any_sync(FULL, lane < kb && (x < 0 || x >= V));
    float q = 1.f;
    if (!bad && p.draft_kind == 1 && !p.greedy) {
        if (lane < kb) q = __ldcg((const float*)p.draft + drow0 + (int64_t)lane * V + x);
        nonf |= __any_sync(FULL, lane < kb && (!(q >= 0.f) || q == INFINITY));
    }
    if (bad || nonf) {
        for (int j = lane; j <= K; j += 32) {
            p.tokens[(int64_t)b * (K + 1) + j] = -1;
            if (p.lse) p.lse[(int64_t)b * (K + 1) + j] = NAN;
            if (j < K) {
                if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = NAN;
                if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = NAN;
            }
        }
        if (lane == 0) {
            p.num_accepted[b] = -1;
            if (p.row_status) p.row_status[b] = bad ? ROW_BAD_TOKEN : ROW_NONFINITE;
            if (p.resid_mass) p.resid_mass[b] = NAN;
            p.jobs[b].kind = JOB_NONE;
        }
        return DECIDE_DONE;
    }
    // accept tests, one slot per lane; the first rejection is the lowest
    // rejecting lane
    const float pd_row = __shfl_sync(FULL, me.px, min(kb + 1 + lane, 31));
    const uint4 wrd = lane <= kb ? slot_words(p, b, lane, 0u) : make_uint4(0, 0, 0, 0);
    bool rej = false;
    if (lane < kb) {
        const float pt = me.px;
        const float pd = p.greedy ? NAN : p.draft_kind == 1 ? q : pd_row;
        if (p.greedy) {
            rej = !(pt > 0.f);  // the kept set is the target's argmax alone
        } else {
            // IEEE: pd = 0 gives inf or NaN; rounding the ratio to fp32 moves
            // it by < 1e-7 relative, inside the near-tie window
            const float ratio = __fdiv_rn(pt, pd);
            rej = !(u24(wrd.x) < ratio);
        }
        if (p.p_t_at) p.p_t_at[(int64_t)b * K + lane] = pt;
        if (p.p_d_at) p.p_d_at[(int64_t)b * K + lane] = pd;
    }
    const unsigned rm = __ballot_sync(FULL, rej);
    const int jstar = rm ? __ffs(rm) - 1 : kb;
    for (int j = lane; j <= K; j += 32) {
        if (p.lse) {
            // lane j holds target row j for j <= kb (kb < 32 here)
            p.lse[(int64_t)b * (K + 1) + j] = j <= kb && !p.greedy ? me.M / p.T + logf((float)me.S) : NAN;
        }
        if (j >= kb && j < K) {
            if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = NAN;
            if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = NAN;
        }
        if (j != jstar) p.tokens[(int64_t)b * (K + 1) + j] = j < jstar ? x : -1;
    }
    // greedy: the emitted token is the argmax of target row j* (its kept list)
    const bool residual = jstar < kb && !p.greedy;
    const float u = u24(__shfl_sync(FULL, wrd.y, jstar));
    const int tr = target_slot(p, b, jstar);
    const RowStat ts = rec_stat(shfl_rec(rw, jstar));
    DraftRef d;
    d.kind = p.draft_kind;
    d.r = residual ? draft_slot(p, b, jstar) : -1;
    const RecWords dw = shfl_rec(rw, min(kb + 1 + jstar, 31));
    if (residual && d.kind == 0) d.st = rec_stat(dw);
    d.row = residual ? (const void*)((const char*)p.draft +
                                     (drow0 + (int64_t)jstar * V) * (d.kind == 1 ? 4 : (int64_t)sizeof(T)))
                     : nullptr;
    if (ts.mode == MODE_LIST) {
        pe->jstar = jstar;
        pe->tr = tr;
        pe->residual = residual;
        pe->u = u;
        pe->ts = ts;
        pe->d = d;
        return DECIDE_SAMPLE;
    }
    if (lane == 0) {
        p.tokens[(int64_t)b * (K + 1) + jstar] = -1;
        p.num_accepted[b] = jstar;
        if (p.row_status) p.row_status[b] = ROW_OK;
        if (p.resid_mass && !residual) p.resid_mass[b] = 0.f;
        Job jb;
        jb.kind = residual ? JOB_RESIDUAL : JOB_ROW;
        jb.trow = tr;
        jb.drow = residual ? d.r : -1;
        jb.out_idx = b * (K + 1) + jstar;
        jb.b = b;
        jb.u = u;
        p.jobs[b] = jb;
    }
    return DECIDE_DONE;
}

// the decision of sequence b by one warp (rows one per lane) with the warp's
// own sample; false leaves it to the decision grid
template <typename T>
__device__ bool warp_decide_lanes(const Params& p, int b, int kb, unsigned char* stage)
{
    DecidePending pe;
    const int h = warp_decide_lanes_head<T>(p, b, kb, &pe);
    if (h != DECIDE_SAMPLE) return h == DECIDE_DONE;
    unsigned long long Z;
    bool zero;
    const int tok = warp_sample_list<T>(p, pe.tr, pe.ts, pe.residual != 0, pe.d, pe.u, stage, &Z, &zero);
    if ((threadIdx.x & 31) == 0) decide_finish(p, b, pe, tok, Z, zero);
    return true;
}


// true when the warp decided sequence b; false leaves it to the decision grid
// (a row of it needs the block merge)
template <typename T>
__device__ bool warp_decide(const Params& p, int b, unsigned char* stage)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int K = p.Kmax, V = p.V;
    const int kb = seq_k(p, b);
    const int nrows = seq_rows(p, kb);
    const int64_t drow0 = (int64_t)b * K * V;
    bool bad = false, nonf = false, block = false;
    for (int i = lane; i < nrows; i += 32) {
        const int r = i <= kb ? target_slot(p, b, i) : draft_slot(p, b, i - kb - 1);
        const int fl = __ldcg(&p.rstat[r].flags);
        nonf |= (fl & FLAG_NONFINITE) != 0;
        // a kept list longer than the warp stages is sampled by the block code
        block |= (fl & FLAG_BLOCK_MERGE) != 0 ||
                 (__ldcg(&p.rstat[r].mode) == MODE_LIST && __ldcg(&p.rstat[r].n_kept) > WM_CAND);
    }
    if (__any_sync(FULL, block)) return false;
    for (int j = lane; j < kb; j += 32) {
        const int x = p.xin[(int64_t)b * K + j];
        if (x < 0 || x >= V) {
            bad = true;
        } else if (p.draft_kind == 1 && !p.greedy) {
            const float q = __ldcg((const float*)p.draft + drow0 + (int64_t)j * V + x);
            if (!(q >= 0.f) || q == INFINITY) nonf = true;
        }
    }
    bad = __any_sync(FULL, bad);
    nonf = __any_sync(FULL, nonf);
    if (bad || nonf) {
        for (int j = lane; j <= K; j += 32) {
            p.tokens[(int64_t)b * (K + 1) + j] = -1;
            if (p.lse) p.lse[(int64_t)b * (K + 1) + j] = NAN;
            if (j < K) {
                if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = NAN;
                if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = NAN;
            }
        }
        if (lane == 0) {
            p.num_accepted[b] = -1;
            if (p.row_status) p.row_status[b] = bad ? ROW_BAD_TOKEN : ROW_NONFINITE;
            if (p.resid_mass) p.resid_mass[b] = NAN;
            p.jobs[b].kind = JOB_NONE;
        }
        return true;
    }
    // accept tests, every slot; the first rejection is the smallest rejected j
    int jstar = kb;
    for (int j0 = 0; j0 < kb; j0 += 32) {
        const int j = j0 + lane;
        bool rej = false;
        if (j < kb) {
            const int x = p.xin[(int64_t)b * K + j];
            const float pt = __ldcg(&p.rstat[target_slot(p, b, j)].px);
            const float pd = p.greedy             ? NAN
                             : p.draft_kind == 1 ? __ldcg((const float*)p.draft + drow0 + (int64_t)j * V + x)
                                                 : __ldcg(&p.rstat[draft_slot(p, b, j)].px);
            if (p.greedy) {
                rej = !(pt > 0.f);  // the kept set is the target's argmax alone
            } else {
                const uint4 w = slot_words(p, b, j, 0u);
                const double ratio = (double)pt / (double)pd;  // IEEE: pd = 0 gives inf or NaN
                rej = !((double)u24(w.x) < ratio);
            }
            if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = pt;
            if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = pd;
        }
        const unsigned m = __ballot_sync(FULL, rej);
        if (m && jstar == kb) jstar = j0 + __ffs(m) - 1;
    }
    for (int j = lane; j <= K; j += 32) {
        if (p.lse) {
            float v = NAN;
            if (j <= kb && !p.greedy) {
                const RowStat* rs = p.rstat + target_slot(p, b, j);
                v = (float)((double)__ldcg(&rs->M) / (double)p.T + log(__ldcg(&rs->S)));
            }
            p.lse[(int64_t)b * (K + 1) + j] = v;
        }
        if (j >= kb && j < K) {
            if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = NAN;
            if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = NAN;
        }
        if (j != jstar) p.tokens[(int64_t)b * (K + 1) + j] = j < jstar ? p.xin[(int64_t)b * K + j] : -1;
    }
    // greedy: the emitted token is the argmax of target row j* (its kept list)
    const bool residual = jstar < kb && !p.greedy;
    const uint4 w = slot_words(p, b, jstar, 0u);
    const float u = u24(w.y);
    const int tr = target_slot(p, b, jstar);
    const RowStat ts = load_rowstat(p.rstat + tr);
    DraftRef d;
    d.kind = p.draft_kind;
    d.r = residual ? draft_slot(p, b, jstar) : -1;
    if (residual && d.kind == 0) d.st = load_rowstat(p.rstat + d.r);
    d.row = residual ? (const void*)((const char*)p.draft +
                                     (drow0 + (int64_t)jstar * V) * (d.kind == 1 ? 4 : (int64_t)sizeof(T)))
                     : nullptr;
    if (ts.mode == MODE_LIST) {
        unsigned long long Z;
        bool zero;
        const int tok = warp_sample_list<T>(p, tr, ts, residual, d, u, stage, &Z, &zero);
        if (lane == 0) {
            p.tokens[(int64_t)b * (K + 1) + jstar] = tok;
            p.num_accepted[b] = jstar;
            if (p.row_status) p.row_status[b] = zero ? ROW_ZERO_RESIDUAL : ROW_OK;
            if (p.resid_mass) p.resid_mass[b] = residual ? (float)from_fix56(Z) : 0.f;
            p.jobs[b].kind = JOB_NONE;
        }
    } else if (lane == 0) {
        p.tokens[(int64_t)b * (K + 1) + jstar] = -1;
        p.num_accepted[b] = jstar;
        if (p.row_status) p.row_status[b] = ROW_OK;
        if (p.resid_mass && !residual) p.resid_mass[b] = 0.f;
        Job jb;
        jb.kind = residual ? JOB_RESIDUAL : JOB_ROW;
        jb.trow = tr;
        jb.drow = residual ? d.r : -1;
        jb.out_idx = b * (K + 1) + jstar;
        jb.b = b;
        jb.u = u;
        p.jobs[b] = jb;
    }
    return true;
}

// a non-negative float below 2^20 as a fixed-point integer in 2^-40 units,
// rounded to nearest (zero, subnormals and anything below 2^-41 give 0)
__device__ __forceinline__ unsigned long long to_fix40(float w)
{
    const uint32_t u = __float_as_uint(w);
    const int ex = (int)(u >> 23);
    if ((u >> 31) || ex == 0) return 0ull;
    const unsigned long long m = (u & 0x7FFFFFu) | 0x800000u;  // w = m 2^(ex - 150)
    const int sh = ex - 110;                                   // w 2^40 = m 2^sh
    if (sh >= 0) return m << min(sh, 39);
    if (sh < -24) return 0ull;
    return (m + (1ull << (-sh - 1))) >> -sh;
}

// ------------------------------------------------------------------------- //
// k_merge_warp: one warp per row slot (after the stream grid).  The last row //
// of a sequence to finish (a ticket) decides the sequence.                   //
// ------------------------------------------------------------------------- //
// The nucleus (top-p after temperature, no top-k) of bf16 row r by one warp,
// from the segments' key histograms (SEG_HIST; sv_rows.cu's merge_row_hist
// does the same with a CTA): each bf16 key's mass is its count times
// exp2((v - M) c), the tokens below the two-binade window come from the
// stream's partial sums, and the rank prefix is cut where the mass before a
// token reaches top_p, ties at the cut key in ascending id (found in the one
// segment holding the boundary token).  Fills st (MODE_PREFIX, P(x) at the
// drafted token x) and returns true; false leaves the row to the block merge
// (a saturated bin, the cut below the window, or more than 32 segments).  A
// small nucleus stays a rank prefix too: its sample is drawn over the dense
// row like any other, with the same masses a kept list would give.
template <typename T>
__device__ bool warp_hist_nucleus(const Params& p, const T* row, int r, int x, WarpSmem& ws, RowStat& st)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int nseg = p.nseg;
    static_assert(sizeof(WarpSmem::keys) >= 32 * HIST_BINS, "32 segments' histograms fit the staging");
    if (nseg > 32) return false;
    uint8_t* H = reinterpret_cast<uint8_t*>(ws.keys);
    const SegStat* segs = p.seg + (int64_t)r * nseg;
    // segment `lane`'s record in this lane, every histogram in shared memory
    float ms = -INFINITY;
    double ss = 0.0;
    if (lane < nseg) {
        ms = __ldcg(&segs[lane].m);
        ss = __ldcg(&segs[lane].s);
    }
    const uint4* Hg = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.chunk) +
                                                     (int64_t)r * p.chunk_stride * 2);
    for (int i = lane; i < nseg * (HIST_BINS / 16); i += 32) reinterpret_cast<uint4*>(H)[i] = __ldcg(Hg + i);
    const float M = warp_reduce_f(ms, fmax_nan);
    if (!(M > -INFINITY && M < INFINITY)) {
        st.flags = FLAG_NONFINITE;
        return true;
    }
    __syncwarp();
    const uint32_t M16 = key16_bf16(__float_as_uint(M) >> 16);
    // masses in fixed point (2^-40 units of the max token's): exact integer
    // sums on the integer pipes, the per-key weights rounded once each
    // the tokens below each segment's own window (the stream's sums)
    unsigned long long below =
        (lane < nseg && ms > -INFINITY) ? to_fix40((float)ss * exp2f((ms - M) * p.c)) : 0ull;
    // lane l holds the row's bins 8 l .. 8 l + 7 (bin D: key M16 - D) and
    // the bins 256 + 8 l .. below the window (weighed once per bin, not per
    // segment); a segment whose window reaches below bin 511 weighs those
    // bins itself (rare: its max lies over two binades below the row's)
    // per window (the bins 8 l .., then 256 + 8 l ..) four packed 16-bit
    // sums of the lane's eight bins: bins 0 and 2, 1 and 3, 4 and 6, 5 and 7
    // (at most 32 segments of at most 255 each: no carry between halves)
    uint32_t acc[2][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[0][k] = acc[1][k] = 0u;
    bool sat = false;
    for (int i = 0; i < nseg; ++i) {
        const float mi = __shfl_sync(FULL, ms, i);
        if (!(mi > -INFINITY)) continue;
        const uint32_t m16 = key16_bf16(__float_as_uint(mi) >> 16);
        const uint32_t off = M16 - m16;  // segment bin d is the row's bin off + d
        const uint8_t* Hb = H + i * HIST_BINS;
        const uint32_t* Hi = reinterpret_cast<const uint32_t*>(Hb);
#pragma unroll
        for (int wd = 0; wd < 2; ++wd) {
            // the lane's row bins 8 l + 256 wd + q are the segment's bins
            // b + q, q < 8; those outside [0, HIST_BINS) count nothing.  The
            // eight bytes from three words of the segment's histogram (word
            // indices clamped to it: a clamped word only feeds bytes that
            // the mask drops), shifted into place, then masked
            const int b = 8 * lane + wd * HIST_BINS - (int)off;
            if (b + 8 <= 0 || b >= HIST_BINS) continue;
            const int w = b >> 2;  // floor: b may be negative
            const uint32_t sh = (uint32_t)(b & 3) * 8u;
            const uint32_t w0 = Hi[min(max(w, 0), HIST_BINS / 4 - 1)];
            const uint32_t w1 = Hi[min(max(w + 1, 0), HIST_BINS / 4 - 1)];
            const uint32_t w2 = Hi[min(max(w + 2, 0), HIST_BINS / 4 - 1)];
            const int cut_lo = max(0, -b), cut_hi = max(0, b + 8 - HIST_BINS);
            const unsigned long long keep = (~0ull << (8 * cut_lo)) & (~0ull >> (8 * cut_hi));
            const uint32_t lo = __funnelshift_r(w0, w1, sh) & (uint32_t)keep;
            const uint32_t hi = __funnelshift_r(w1, w2, sh) & (uint32_t)(keep >> 32);
            // a saturated bin (255) among them: a zero byte in the complement
            const uint32_t nl = ~lo, nh = ~hi;
            sat |= ((((nl - 0x01010101u) & ~nl) | ((nh - 0x01010101u) & ~nh)) & 0x80808080u) != 0u;
            acc[wd][0] += lo & 0x00FF00FFu;
            acc[wd][1] += (lo >> 8) & 0x00FF00FFu;
            acc[wd][2] += hi & 0x00FF00FFu;
            acc[wd][3] += (hi >> 8) & 0x00FF00FFu;
        }
        if (off > (uint32_t)HIST_BINS) {
            // segment bins d with off + d >= 512
            const uint32_t d0 = off >= 2u * HIST_BINS ? 0u : 2u * HIST_BINS - off;
            for (uint32_t d = d0 + lane; d < (uint32_t)HIST_BINS; d += 32) {
                const uint32_t c = Hb[d];
                sat |= c == 255u;
                if (c) below += (unsigned long long)c * to_fix40(hist_weight(p, m16 - d, M));
            }
        }
    }
    if (__any_sync(FULL, sat)) return false;
    uint32_t cnt[8], cntb[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        // sums k: bins (k & 1) + 4 (k >> 1) (low half) and that + 2 (high half)
        const int q = (k & 1) + 4 * (k >> 1);
        cnt[q] = acc[0][k] & 0xFFFFu;
        cnt[q + 2] = acc[0][k] >> 16;
        cntb[q] = acc[1][k] & 0xFFFFu;
        cntb[q + 2] = acc[1][k] >> 16;
    }
    unsigned long long mass[8], wq[8];
    unsigned long long lsum = 0ull;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint32_t key = M16 - (8u * lane + q);
        wq[q] = key >= 0x80u ? to_fix40(hist_weight(p, key, M)) : 0ull;
        mass[q] = (unsigned long long)cnt[q] * wq[q];
        lsum += mass[q];
        const uint32_t keyb = key - HIST_BINS;
        if (cntb[q] && key >= 0x80u + HIST_BINS)
            below += (unsigned long long)cntb[q] * to_fix40(hist_weight(p, keyb, M));
    }
    unsigned long long incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += y;
    }
    unsigned long long bsum = below;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bsum += __shfl_xor_sync(FULL, bsum, o);
    const unsigned long long S_all = __shfl_sync(FULL, incl, 31) + bsum;
    // the strict rule: a token is kept while the mass before it is below
    // top_p S; target = ceil(top_p S) in the same units (top_p_fix = top_p 2^56)
    unsigned long long target;
    {
        const unsigned long long lo = p.top_p_fix * S_all, hi = __umul64hi(p.top_p_fix, S_all);
        target = (hi << 8) | (lo >> 56);
        if (lo & ((1ull << 56) - 1ull)) ++target;
    }
    // the first bin whose inclusive mass reaches the target
    int cut = -1;
    unsigned long long above = 0ull, run = incl - lsum;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        if (cut < 0 && cnt[q] > 0 && run < target && run + mass[q] >= target) {
            cut = 8 * lane + q;
            above = run;
        }
        run += mass[q];
    }
    const unsigned has = __ballot_sync(FULL, cut >= 0);
    if (!has) return false;  // the cut lies below the window
    const int src = __ffs(has) - 1;
    cut = __shfl_sync(FULL, cut, src);
    above = __shfl_sync(FULL, above, src);
    int n_lane = 0, cntk = 0;
    unsigned long long wk = 0ull;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int d = 8 * lane + q;
        if (d < cut) n_lane += (int)cnt[q];
        if (d == cut) {
            cntk = (int)cnt[q];
            wk = wq[q];
        }
    }
    const int n_above = __reduce_add_sync(FULL, n_lane);
    cntk = __reduce_add_sync(FULL, cntk);
    wk = __shfl_sync(FULL, wk, src);
    const uint32_t kap16 = M16 - (uint32_t)cut;
    // the tokens of the cut key kept: the fewest whose mass reaches the target
    int nk = (int)((target - above + wk - 1ull) / wk);
    nk = max(1, min(nk, cntk));
    int32_t ik = p.V - 1;
    if (nk < cntk) {
        // the segment holding the nk-th token of key kap16 (in id order)
        int cs = 0;
        if (lane < nseg && ms > -INFINITY) {
            const uint32_t m16 = key16_bf16(__float_as_uint(ms) >> 16);
            if (m16 >= kap16 && m16 - kap16 < (uint32_t)HIST_BINS) cs = H[lane * HIST_BINS + (m16 - kap16)];
        }
        int ci = cs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, ci, o);
            if (lane >= o) ci += y;
        }
        const unsigned hit = __ballot_sync(FULL, ci - cs < nk && nk <= ci);
        const int sseg = hit ? __ffs(hit) - 1 : 0;
        const int need = nk - __shfl_sync(FULL, ci - cs, sseg);  // 1-based among the segment's
        // the segment in batches of eight rounds of coalesced loads (round j
        // of batch g: words 32 (8 g + j) .. + 31, lane l: word 32 (8 g + j)
        // + l), from its end when the token lies in the later half of the
        // segment's cs matches: the batch holding it is found from the
        // batches' match counts alone, then the round and the lane in it
        const unsigned short* rb = reinterpret_cast<const unsigned short*>(row);
        const int e_begin = sseg * (SEG_BYTES / 2);
        const int nwd = (min(p.V, e_begin + SEG_BYTES / 2) - e_begin) / 8;  // whole words (V % 8 == 0)
        const int nbat = (nwd + 255) / 256;
        const int csg = __shfl_sync(FULL, cs, sseg);  // the segment's tokens of key kap16
        const bool back = 2 * need > csg + 1;
        int want = back ? csg - need + 1 : need;  // 1-based, in the order the batches are read
        int found = -1;
        for (int i = 0; i < nbat; ++i) {
            const int g = back ? nbat - 1 - i : i;
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int w = (8 * g + j) * 32 + lane;
                v[j] = w < nwd ? __ldcg(reinterpret_cast<const uint4*>(rb + e_begin + 8 * w)) : make_uint4(0, 0, 0, 0);
            }
            uint32_t hm[8];
            int cl = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int w = (8 * g + j) * 32 + lane;
                const uint32_t xw[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                hm[j] = 0u;
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const uint32_t b16 = (h & 1) ? (xw[h >> 1] >> 16) : (xw[h >> 1] & 0xFFFFu);
                    if (w < nwd && key16_bf16(b16) == kap16) hm[j] |= 1u << h;
                }
                cl += __popc(hm[j]);
            }
            const int tb = __reduce_add_sync(FULL, cl);
            if (want > tb) {
                want -= tb;
                continue;
            }
            // this batch: the token is its need_b-th match in id order; the
            // round holding it (warp-uniform), then the lane and the bit
            int need_b = back ? tb - want + 1 : want;
            int js = -1;
            uint32_t mj = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int tot = __reduce_add_sync(FULL, __popc(hm[j]));
                if (js < 0) {
                    if (need_b <= tot) {
                        js = j;
                        mj = hm[j];
                    } else {
                        need_b -= tot;
                    }
                }
            }
            const int c = __popc(mj);
            int in = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(FULL, in, o);
                if (lane >= o) in += y;
            }
            int f = -1;
            if (js >= 0 && in - c < need_b && need_b <= in) {
                uint32_t m = mj;
                for (int q = 0; q < need_b - (in - c) - 1; ++q) m &= m - 1u;  // drop earlier hits
                f = e_begin + 8 * ((8 * g + js) * 32 + lane) + __ffs(m) - 1;
            }
            found = __reduce_max_sync(FULL, f);
            break;
        }
        if (found < 0) return false;  // not found (cannot happen with exact counts): the block merge
        ik = found;
    }
    st.M = M;
    st.S = (double)(above + (unsigned long long)nk * wk) * 0x1p-40;
    st.mode = MODE_PREFIX;
    st.kappa = key_of(val_key16(kap16));
    st.i_kappa = ik;
    st.n_kept = n_above + nk;
    st.flags = 0;
    if (x >= 0) {
        const float lx = Elem<T>::load_cg(row, x);
        st.px = kept_prefix(st, key_of(lx), x) ? row_prob(p, lx, M, st.S) : 0.f;
    }
    return true;
}

// The row slot of the g-th row the merge grid has work for, in sequence
// order: each sequence's valid rows (target rows 0..K_b, then its draft rows
// when they are streamed: seq_rows of them), or its slot 0 alone when K_b is
// out of range (to report it); -1 past the last.  With a ragged batch the
// valid rows then sit in the first warps of the grid, which fit the SMs at
// once, instead of spreading over every slot of the batch's largest K.
__device__ int warp_row_of(const Params& p, int g)
{
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    constexpr int PER = 8;  // sequences a lane counts per round
    int base = 0;           // rows of the sequences before this round's
    for (int b0 = 0; b0 < p.B; b0 += 32 * PER) {
        int cnt[PER], kbv[PER];
        int mine = 0;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int b = b0 + lane * PER + e;
            kbv[e] = b < p.B ? seq_k(p, b) : 0;
            cnt[e] = b < p.B ? (k_ok(p, kbv[e]) ? seq_rows(p, kbv[e]) : 1) : 0;
            mine += cnt[e];
        }
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += y;
        }
        const int tot = __shfl_sync(FULL, incl, 31);
        if (g < base + tot) {
            const int before = base + incl - mine;
            int r = -1;
            if (before <= g && g < before + mine) {
                int i = g - before;
#pragma unroll
                for (int e = 0; e < PER; ++e) {
                    if (r < 0 && i < cnt[e]) {
                        const int b = b0 + lane * PER + e, kb = kbv[e];
                        const int slot = !k_ok(p, kb) ? 0 : (i <= kb ? i : p.Kmax + 1 + (i - kb - 1));
                        r = b * p.rps + slot;
                    }
                    if (r < 0) i -= cnt[e];
                }
            }
            return __reduce_max_sync(FULL, r);
        }
        base += tot;
    }
    return -1;
}

template <typename T>
__global__ void __launch_bounds__(WM_WARPS * 32) k_merge_warp(const Params p)
{
    extern __shared__ __align__(16) unsigned char smem_w[];
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream grid has completed
    if (exit_skip(p)) return;
    // the decision grid may be scheduled now; it waits for this grid's end
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const unsigned FULL = 0xffffffffu;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int r = blockIdx.x * WM_WARPS + warp;
    if (p.kpr && !p.draft_launch) {
        r = warp_row_of(p, r);  // per-row K: the valid rows first
        if (r < 0) return;
    } else if (r >= p.B * p.rps) {
        return;
    }
    // every load that does not depend on another goes out at once: the
    // sequence's K_b and the row's drafted token
    const int b = r / p.rps, slot = r - b * p.rps;
    const int jd = slot > p.Kmax ? slot - (p.Kmax + 1) : slot;  // position of the row
    const int x_raw = jd < p.Kmax ? __ldg(p.xin + (int64_t)b * p.Kmax + jd) : -1;
    const RowRef rr = row_ref(p, r);
    if (!rr.valid) {
        if (lane == 0) report_skipped_row(p, rr);
        return;
    }
    if (rr.is_draft && !drafts_streamed(p)) return;
    // (only keys is touched outside chunk-key rows: see wm_stride)
    WarpSmem& ws = *reinterpret_cast<WarpSmem*>(smem_w + (size_t)warp * wm_stride(p.seg_mode));
    const T* row = (const T*)(rr.is_draft ? p.draft : p.target) + row_elem_offset(p, rr);
    // the drafted token this row's P(x) is needed at (the bonus row has none)
    int x = -1;
    if (rr.j < rr.kb && x_raw >= 0 && x_raw < p.V) x = x_raw;
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
    if (p.seg_mode == SEG_CHUNK) {
        if (!warp_fast_topk<T>(p, row, r, x, ws, st)) st.flags |= FLAG_BLOCK_MERGE;
    } else if (p.seg_mode == SEG_HIST) {
        bool ok = false;
        if constexpr (sizeof(T) == 2) ok = warp_hist_nucleus<T>(p, row, r, x, ws, st);
        if (!ok) st.flags |= FLAG_BLOCK_MERGE;
    } else {
        warp_all_stats(p, r, st);
        if (!st.flags && x >= 0) st.px = row_prob(p, Elem<T>::load_cg(row, x), st.M, st.S);
    }
    if (lane == 0) p.rstat[r] = st;
    // sequence ticket: the warp barrier orders every lane's writes before lane
    // 0's fence, which makes them visible before the ticket is taken
    __syncwarp();
    unsigned last = 0;
    if (lane == 0) {
        __threadfence();
        const int nrows = seq_rows(p, rr.kb);
        last = atomicAdd(&p.seq_ticket[rr.b], 1u) == (unsigned)(nrows - 1);
        if (last) p.seq_ticket[rr.b] = 0u;
    }
    last = __shfl_sync(FULL, last, 0);
    if (!last) return;
    if (lane == 0) __threadfence();
    __syncwarp();
    const int nrows_b = seq_rows(p, rr.kb);
    unsigned char* stage = reinterpret_cast<unsigned char*>(ws.keys);
    if (nrows_b <= 32 ? warp_decide_lanes<T>(p, rr.b, rr.kb, stage) : warp_decide<T>(p, rr.b, stage)) {
        __syncwarp();
        if (lane == 0) p.seq_done[rr.b] = 1u;
    }
}

// ------------------------------------------------------------------------- //
// k_decide: one CTA per sequence the merge grid did not decide: the rows the //
// warp merge flagged are merged by the block code, then the sequence is      //
// decided                                                                    //
// ------------------------------------------------------------------------- //
template <typename T>
__global__ void __launch_bounds__(NT) k_decide(const Params p)
{
    extern __shared__ __align__(16) unsigned char smem_scratch[];  // SCRATCH_BYTES
    __shared__ int s_done;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the merge grid has completed
    if (exit_skip(p)) return;
    const int b = blockIdx.x;
    const int kb = seq_k(p, b);
    if (!k_ok(p, kb)) return;  // reported by the merge grid
    if (threadIdx.x == 0) {
        s_done = (int)__ldcg(p.seq_done + b);
        if (s_done) p.seq_done[b] = 0u;
    }
    csync();
    if (s_done) return;
    const int nrows = seq_rows(p, kb);
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
