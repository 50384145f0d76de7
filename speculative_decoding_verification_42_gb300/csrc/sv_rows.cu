// sv_rows.cu -- stage 1 of the verify step: stream every valid row once, merge
// each row's statistics and kept set, decide each sequence.
//
// What a row needs (NOTE-159, "Key results": temperature, top-k and nucleus
// applied to the probabilities before the rejection step):
//   z = l / T; keep the top-k by (l desc, id asc); keep the rank prefix whose
//   mass strictly before each token is < top_p; P(v) = exp(z_v - M) / S over
//   the kept set.
// The accept test and the resample follow "Accelerating Large Language Model
// Decoding with Speculative Sampling" (The algorithm) and the listings of
// "57 Speculative Decoding" (One speculative decoding loop) and "Speculative
// Decoding from Scratch" (The heart of it, 2.3): accept x_j iff u < p_t/p_d;
// stop at the first rejection; resample it from max(0, p_t - p_d); when all
// pass, one more token from the target at K_b + 1 (The big picture, 2.1).
#include "sv_internal.cuh"

namespace sv {

// dynamic shared memory of k_rows
constexpr int SM_CK = MAX_CHUNKS * 2;        // chunk keys (u16)
constexpr int SM_CAND = CAND_CAP * 8;        // candidates (u64) / histogram (u64[NBINS])
constexpr int SM_QUAL = CAND_CAP * 4;        // qualifying chunk ids
constexpr int SM_HIST = 256 * 4 * 2;         // two 256-bin u32 histograms
constexpr int ROWS_SMEM = SM_CK + SM_CAND + SM_QUAL + SM_HIST;
static_assert(SM_CAND >= NBINS * 8, "histogram must fit the candidate region");

struct Smem {
    uint16_t* ck;
    unsigned long long* cand;  // also the u64 histogram of the general select
    int32_t* qual;
    uint32_t* h0;
    uint32_t* h1;
};

__device__ __forceinline__ Smem smem_layout(unsigned char* base)
{
    Smem s;
    s.ck = (uint16_t*)base;
    s.cand = (unsigned long long*)(base + SM_CK);
    s.qual = (int32_t*)(base + SM_CK + SM_CAND);
    s.h0 = (uint32_t*)(base + SM_CK + SM_CAND + SM_QUAL);
    s.h1 = s.h0 + 256;
    return s;
}

// ------------------------------------------------------------------------- //
// per-vector arithmetic of the streaming pass (16 bytes: 8 bf16 or 4 f32)     //
// ------------------------------------------------------------------------- //
template <typename T> struct Vec16;

template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ uint4 neg_inf() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
    static __device__ __forceinline__ float vmax(uint4 w)
    {
        float a = fmax_nan(fmax_nan(bf16_lo(w.x), bf16_hi(w.x)), fmax_nan(bf16_lo(w.y), bf16_hi(w.y)));
        float b = fmax_nan(fmax_nan(bf16_lo(w.z), bf16_hi(w.z)), fmax_nan(bf16_lo(w.w), bf16_hi(w.w)));
        return fmax_nan(a, b);
    }
    static __device__ __forceinline__ float vsumexp(uint4 w, float m, float c)
    {
        float s = 0.f;
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s += ex2_fast((bf16_lo(ws[i]) - m) * c);
            s += ex2_fast((bf16_hi(ws[i]) - m) * c);
        }
        return s;
    }
    static __device__ __forceinline__ uint4 load_scalar(const __nv_bfloat16* row, int64_t e0, int V)
    {
        uint16_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            h[i] = (e0 + i < V) ? __ldg((const unsigned short*)row + e0 + i) : (uint16_t)0xFF80u;
        return make_uint4(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16),
                          h[4] | ((uint32_t)h[5] << 16), h[6] | ((uint32_t)h[7] << 16));
    }
};

template <> struct Vec16<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ uint4 neg_inf() { return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u); }
    static __device__ __forceinline__ float vmax(uint4 w)
    {
        return fmax_nan(fmax_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                        fmax_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
    static __device__ __forceinline__ float vsumexp(uint4 w, float m, float c)
    {
        return ex2_fast((__uint_as_float(w.x) - m) * c) + ex2_fast((__uint_as_float(w.y) - m) * c) +
               ex2_fast((__uint_as_float(w.z) - m) * c) + ex2_fast((__uint_as_float(w.w) - m) * c);
    }
    static __device__ __forceinline__ uint4 load_scalar(const float* row, int64_t e0, int V)
    {
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            h[i] = (e0 + i < V) ? __float_as_uint(__ldg(row + e0 + i)) : 0xFF800000u;
        return make_uint4(h[0], h[1], h[2], h[3]);
    }
};

// ------------------------------------------------------------------------- //
// the streaming pass over one segment                                       //
// ------------------------------------------------------------------------- //
template <typename T, bool VEC, int MODE>
__device__ __forceinline__ void segment_pass(const Params& p, const T* row, int seg, int r,
                                             float* redf, double* redd)
{
    constexpr int VW = Vec16<T>::N;
    constexpr int SEG = SEG_BYTES / (int)sizeof(T);
    constexpr int ROUNDS = SEG / (NT * VW);
    constexpr int CHUNK_EL = CHUNK_BYTES / (int)sizeof(T);
    const int V = p.V;
    const int64_t base = (int64_t)seg * SEG;

    uint4 v[ROUNDS];
#pragma unroll
    for (int i = 0; i < ROUNDS; ++i) {
        const int64_t e0 = base + ((int64_t)i * NT + threadIdx.x) * VW;
        if (VEC)
            v[i] = (e0 < V) ? ld_stream16(row + e0) : Vec16<T>::neg_inf();
        else
            v[i] = (e0 < V) ? Vec16<T>::load_scalar(row, e0, V) : Vec16<T>::neg_inf();
    }

    if (MODE == SEG_CHUNK) {
        // 8 consecutive lanes hold one 128-byte chunk: its NaN-propagating max
        // becomes a 16-bit order key (a lower bound of every key in the chunk)
#pragma unroll
        for (int i = 0; i < ROUNDS; ++i) {
            float m = Vec16<T>::vmax(v[i]);
            m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, 4));
            const int64_t e0 = base + ((int64_t)i * NT + threadIdx.x) * VW;
            const int64_t ci = e0 / CHUNK_EL;
            if ((threadIdx.x & 7) == 0 && e0 < V)
                p.chunk[(int64_t)r * p.nchunk + ci] = (uint16_t)(key_of(m) >> 16);
        }
    } else {
        float m = Vec16<T>::vmax(v[0]);
#pragma unroll
        for (int i = 1; i < ROUNDS; ++i) m = fmax_nan(m, Vec16<T>::vmax(v[i]));
        m = block_max_nan(m, redf);
        float s = 0.f;
        if (m > -INFINITY && m < INFINITY) {
#pragma unroll
            for (int i = 0; i < ROUNDS; ++i) s += Vec16<T>::vsumexp(v[i], m, p.c);
        }
        const double tot = block_sum_d((double)s, redd);
        if (threadIdx.x == 0) {
            SegStat st;
            st.m = m;
            st.pad = 0.f;
            st.s = tot;
            p.seg[(int64_t)r * p.nseg + seg] = st;
        }
    }
}

// ------------------------------------------------------------------------- //
// general selection of a rank prefix by radix descent over the order keys    //
// ------------------------------------------------------------------------- //
struct SelCfg {
    bool mass;          // weight = fixed-point probability (2^-56 units), else 1
    float M, c;         // exponent reference and log2(e)/T
    float scale;        // 2^56 / S
    bool restricted;    // only tokens of the rank prefix rst
    RowStat rst;
};

__device__ __forceinline__ unsigned long long sel_weight(const SelCfg& cfg, float l)
{
    if (!cfg.mass) return 1ull;
    const float w = ex2_fast((l - cfg.M) * cfg.c) * cfg.scale;
    return __float2ull_rn(w);
}

// Finds the rank prefix {key > kappa} + {key == kappa, id <= i_kappa} whose last
// token is where the inclusive cumulative weight (from the top rank) first
// reaches `need`.  Returns false when the total weight is below `need` (then
// every token is kept).
template <typename T>
__device__ bool select_prefix(const T* row, int V, const SelCfg& cfg, unsigned long long need,
                              unsigned long long* hist, uint32_t* kappa_out, int32_t* ikappa_out)
{
    __shared__ unsigned long long s_red[NT / 32 + 1];
    __shared__ unsigned long long s_cum;
    __shared__ uint32_t s_bin;
    __shared__ int s_found;
    __shared__ int32_t s_ik;
    uint32_t pmask = 0, pval = 0;
    constexpr bool BF = sizeof(T) == 2;
    constexpr int LEVELS = BF ? 2 : 3;
    for (int lev = 0; lev < LEVELS; ++lev) {
        const int shift = lev == 0 ? 21 : (lev == 1 ? 10 : 0);
        const int nb = lev == 2 ? 1024 : 2048;
        for (int i = threadIdx.x; i < nb; i += NT) hist[i] = 0ull;
        if (threadIdx.x == 0) s_found = 0;
        __syncthreads();
        for (int e = threadIdx.x; e < V; e += NT) {
            const float l = Elem<T>::load_cg(row, e);
            const uint32_t k = key_of(l);
            if ((k & pmask) != pval) continue;
            if (cfg.restricted && !kept_prefix(cfg.rst, k, e)) continue;
            const unsigned long long w = sel_weight(cfg, l);
            if (w) atomicAdd(&hist[(k >> shift) & (uint32_t)(nb - 1)], w);
        }
        __syncthreads();
        const int per = nb / NT;
        unsigned long long local = 0;
        for (int q = 0; q < per; ++q) local += hist[nb - 1 - (threadIdx.x * per + q)];
        unsigned long long total;
        unsigned long long cum = block_excl_scan<unsigned long long>(local, s_red, &total);
        if (total < need) return false;  // uniform across the block
        for (int q = 0; q < per; ++q) {
            const int h = nb - 1 - (threadIdx.x * per + q);
            const unsigned long long w = hist[h];
            if (cum < need && need <= cum + w) {
                s_bin = (uint32_t)h;
                s_cum = cum;
                s_found = 1;
            }
            cum += w;
        }
        __syncthreads();
        need -= s_cum;
        pmask |= (uint32_t)(nb - 1) << shift;
        pval |= s_bin << shift;
        __syncthreads();
    }
    uint32_t kappa = pval;
    if (BF) kappa |= (pval & 0x80000000u) ? 0u : 0x3FFu;  // bf16 keys end in 0s or 1s

    // ties at kappa in ascending id: the first whose inclusive weight reaches need
    if (threadIdx.x == 0) s_ik = -1;
    unsigned long long running = 0;
    for (int tile = 0; tile < V; tile += NT * WALK_EPT) {
        const int e0 = tile + threadIdx.x * WALK_EPT;
        unsigned long long local = 0;
        for (int q = 0; q < WALK_EPT; ++q) {
            const int e = e0 + q;
            if (e >= V) break;
            const float l = Elem<T>::load_cg(row, e);
            const uint32_t k = key_of(l);
            if (k == kappa && (!cfg.restricted || kept_prefix(cfg.rst, k, e)))
                local += sel_weight(cfg, l);
        }
        unsigned long long total;
        const unsigned long long ex = block_excl_scan<unsigned long long>(local, s_red, &total);
        if (running + total >= need) {
            unsigned long long cum = running + ex;
            if (cum < need && need <= cum + local) {
                for (int q = 0; q < WALK_EPT; ++q) {
                    const int e = e0 + q;
                    if (e >= V) break;
                    const float l = Elem<T>::load_cg(row, e);
                    const uint32_t k = key_of(l);
                    if (k == kappa && (!cfg.restricted || kept_prefix(cfg.rst, k, e))) {
                        cum += sel_weight(cfg, l);
                        if (cum >= need) {
                            s_ik = e;
                            break;
                        }
                    }
                }
            }
            __syncthreads();
            break;
        }
        running += total;
    }
    __syncthreads();
    *kappa_out = kappa;
    *ikappa_out = s_ik < 0 ? V - 1 : s_ik;
    return true;
}

// max logit of a row (NaN-propagating), read from L2
template <typename T>
__device__ float row_max(const T* row, int V, float* redf)
{
    float m = -INFINITY;
    for (int e = threadIdx.x; e < V; e += NT) m = fmax_nan(m, Elem<T>::load_cg(row, e));
    return block_max_nan(m, redf);
}

// Sum over a rank prefix of exp2((l - M) c); writes the prefix as an ordered
// list when it has at most KCAP tokens.  Returns the kept count.
template <typename T>
__device__ int collect_prefix(const T* row, int V, const RowStat& fin, float M, float c,
                              int32_t* kid, float* kl, double* S_out)
{
    __shared__ int s_red_i[NT / 32 + 1];
    __shared__ double s_red_d[NT / 32 + 1];
    int offset = 0;
    float s = 0.f;
    for (int tile = 0; tile < V; tile += NT * WALK_EPT) {
        const int e0 = tile + threadIdx.x * WALK_EPT;
        int cnt = 0;
        for (int q = 0; q < WALK_EPT; ++q) {
            const int e = e0 + q;
            if (e >= V) break;
            const float l = Elem<T>::load_cg(row, e);
            if (kept_prefix(fin, key_of(l), e)) ++cnt;
        }
        int total;
        int off = offset + block_excl_scan<int>(cnt, s_red_i, &total);
        for (int q = 0; q < WALK_EPT && cnt; ++q) {
            const int e = e0 + q;
            if (e >= V) break;
            const float l = Elem<T>::load_cg(row, e);
            if (kept_prefix(fin, key_of(l), e)) {
                s += ex2_fast((l - M) * c);
                if (off < KCAP) {
                    kid[off] = e;
                    kl[off] = l;
                }
                ++off;
            }
        }
        offset += total;
    }
    *S_out = block_sum_d((double)s, s_red_d);
    return offset;
}

// ------------------------------------------------------------------------- //
// row merge: statistics and kept set of row slot r                          //
// ------------------------------------------------------------------------- //
template <typename T>
__device__ void merge_row(const Params& p, const T* row, int r, const Smem& sm)
{
    __shared__ float s_redf[NT / 32 + 1];
    __shared__ double s_redd[NT / 32 + 1];
    __shared__ RowStat s_st;
    __shared__ int s_cnt, s_nqual, s_fallback, s_nk;
    const int V = p.V;
    const float c = p.c;
    int32_t* kid = p.kept_id + (int64_t)r * KCAP;
    float* kl = p.kept_l + (int64_t)r * KCAP;
    const bool topk_on = p.top_k > 0 && p.top_k < V;
    const bool topp_on = p.top_p < 1.0f;

    RowStat st;
    st.M = -INFINITY;
    st.kappa = 0;
    st.S = 0.0;
    st.i_kappa = V - 1;
    st.n_kept = V;
    st.mode = MODE_ALL;
    st.flags = 0;
    bool have_stats = false;  // M (and the all-token S) known
    bool done = false;

    if (p.seg_mode == SEG_CHUNK) {
        // ---- fast top-k: the k-th largest chunk max bounds the k-th largest key
        const int nc = p.nchunk;
        const uint16_t* ckg = p.chunk + (int64_t)r * nc;
        uint32_t kmax = 0;
        bool bad = false;
        for (int i = threadIdx.x; i < nc; i += NT) {
            const uint16_t k = __ldcg(ckg + i);
            sm.ck[i] = k;
            kmax = max(kmax, (uint32_t)k);
            bad |= (k >= 0xFF80u);  // +inf or NaN
        }
        for (int i = threadIdx.x; i < 256; i += NT) {
            sm.h0[i] = 0;
            sm.h1[i] = 0;
        }
        if (threadIdx.x == 0) {
            s_cnt = 0;
            s_nqual = 0;
            s_fallback = 0;
        }
        bad = __syncthreads_or(bad);
        kmax = (uint32_t)__reduce_max_sync(0xffffffffu, kmax);
        __shared__ uint32_t s_kmax[NT / 32];
        if ((threadIdx.x & 31) == 0) s_kmax[threadIdx.x >> 5] = kmax;
        __syncthreads();
        kmax = 0;
        for (int i = 0; i < NT / 32; ++i) kmax = max(kmax, s_kmax[i]);
        if (bad || kmax <= 0x007Fu) {  // NaN / +inf, or no finite logit
            st.flags = FLAG_NONFINITE;
            done = true;
        } else {
            // radix select of the k-th largest 16-bit chunk key (two byte digits)
            const int k = p.top_k;
            for (int i = threadIdx.x; i < nc; i += NT) atomicAdd(&sm.h0[sm.ck[i] >> 8], 1u);
            __syncthreads();
            __shared__ uint32_t s_hi, s_lo, s_need;
            __shared__ int s_red_i[NT / 32 + 1];
            {
                const uint32_t cnt = sm.h0[255 - threadIdx.x];
                int total;
                const int ex = block_excl_scan<int>((int)cnt, s_red_i, &total);
                if (ex < k && k <= ex + (int)cnt) {
                    s_hi = 255 - threadIdx.x;
                    s_need = k - ex;
                }
            }
            __syncthreads();
            const uint32_t hi = s_hi;
            for (int i = threadIdx.x; i < nc; i += NT)
                if ((uint32_t)(sm.ck[i] >> 8) == hi) atomicAdd(&sm.h1[sm.ck[i] & 255], 1u);
            __syncthreads();
            {
                const int need = (int)s_need;
                const uint32_t cnt = sm.h1[255 - threadIdx.x];
                int total;
                const int ex = block_excl_scan<int>((int)cnt, s_red_i, &total);
                if (ex < need && need <= ex + (int)cnt) s_lo = 255 - threadIdx.x;
            }
            __syncthreads();
            const uint32_t tau16 = (hi << 8) | s_lo;
            const uint32_t tau32 = tau16 << 16;
            // chunks that can hold a top-k token
            for (int i = threadIdx.x; i < nc; i += NT)
                if (sm.ck[i] >= tau16) {
                    const int q = atomicAdd(&s_nqual, 1);
                    if (q < CAND_CAP) sm.qual[q] = i;
                }
            __syncthreads();
            const int nq = s_nqual;
            if (nq > CAND_CAP) {
                s_fallback = 1;
            } else {
                constexpr int CHUNK_EL = CHUNK_BYTES / (int)sizeof(T);
                const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
                for (int q = w; q < nq; q += NT / 32) {
                    const int e_base = sm.qual[q] * CHUNK_EL;
                    for (int e = e_base + lane; e < e_base + CHUNK_EL; e += 32) {
                        bool take = false;
                        uint32_t key = 0;
                        if (e < V) {
                            key = key_of(Elem<T>::load_cg(row, e));
                            take = key >= tau32;
                        }
                        const unsigned bal = __ballot_sync(0xffffffffu, take);
                        int slot0 = 0;
                        if (lane == 0 && bal) slot0 = atomicAdd(&s_cnt, __popc(bal));
                        slot0 = __shfl_sync(0xffffffffu, slot0, 0);
                        if (take) {
                            const int slot = slot0 + __popc(bal & ((1u << lane) - 1u));
                            if (slot < CAND_CAP)
                                sm.cand[slot] = ((unsigned long long)(~key) << 32) | (uint32_t)e;
                        }
                    }
                }
                __syncthreads();
                if (s_cnt > CAND_CAP) s_fallback = 1;
            }
            __syncthreads();
            if (!s_fallback) {
                // exact order: key descending, then id ascending
                const int n = s_cnt;
                const int n2 = next_pow2(n);
                for (int i = n + threadIdx.x; i < n2; i += NT) sm.cand[i] = ~0ull;
                __syncthreads();
                bitonic_sort_u64(sm.cand, n2);
                const int kk = min(k, n);
                const float M = val_of(~(uint32_t)(sm.cand[0] >> 32));
                // exponentials of the kept ranks (rank order) and their sum
                float e_loc = 0.f;
                for (int i = threadIdx.x; i < kk; i += NT) {
                    const float l = val_of(~(uint32_t)(sm.cand[i] >> 32));
                    e_loc += ex2_fast((l - M) * c);
                }
                double S = block_sum_d((double)e_loc, s_redd);
                int nk = kk;
                if (topp_on) {
                    // strict prefix rule over the kept ranks, in fp64
                    if (threadIdx.x == 0) {
                        double pre = 0.0;
                        int i = 0;
                        for (; i < kk; ++i) {
                            if (!(pre < (double)p.top_p)) break;
                            const float l = val_of(~(uint32_t)(sm.cand[i] >> 32));
                            pre += (double)ex2_fast((l - M) * c) / S;
                        }
                        s_nk = i;
                    }
                    __syncthreads();
                    nk = s_nk;
                    float e2 = 0.f;
                    for (int i = threadIdx.x; i < nk; i += NT) {
                        const float l = val_of(~(uint32_t)(sm.cand[i] >> 32));
                        e2 += ex2_fast((l - M) * c);
                    }
                    S = block_sum_d((double)e2, s_redd);
                }
                // the kept list in ascending id: re-key as (id << 32 | key)
                __syncthreads();
                for (int i = threadIdx.x; i < nk; i += NT) {
                    const unsigned long long x = sm.cand[i];
                    sm.cand[i] = ((unsigned long long)(uint32_t)x << 32) | (uint32_t)(~(uint32_t)(x >> 32));
                }
                const int nk2 = next_pow2(nk);
                for (int i = nk + threadIdx.x; i < nk2; i += NT) sm.cand[i] = ~0ull;
                __syncthreads();
                bitonic_sort_u64(sm.cand, nk2);
                for (int i = threadIdx.x; i < nk; i += NT) {
                    const unsigned long long x = sm.cand[i];
                    kid[i] = (int32_t)(x >> 32);
                    kl[i] = val_of((uint32_t)x);
                }
                st.M = M;
                st.S = S;
                st.n_kept = nk;
                st.mode = MODE_LIST;
                done = true;
            }
        }
        __syncthreads();
    } else {
        // ---- statistics over all tokens from the segment records
        float m = -INFINITY;
        for (int i = threadIdx.x; i < p.nseg; i += NT) m = fmax_nan(m, __ldcg(&p.seg[(int64_t)r * p.nseg + i].m));
        const float M = block_max_nan(m, s_redf);
        if (!(M > -INFINITY && M < INFINITY)) {
            st.flags = FLAG_NONFINITE;
            done = true;
        } else {
            double s = 0.0;
            for (int i = threadIdx.x; i < p.nseg; i += NT) {
                const SegStat* g = p.seg + (int64_t)r * p.nseg + i;
                const float gm = __ldcg(&g->m);
                if (gm > -INFINITY) s += __ldcg(&g->s) * exp2(((double)gm - (double)M) * (double)c);
            }
            st.M = M;
            st.S = block_sum_d(s, s_redd);
            have_stats = true;
            if (!topk_on && !topp_on) done = true;  // MODE_ALL
        }
    }

    if (!done) {
        // ---- general path: radix descent over the full row (read from L2)
        if (!have_stats) st.M = row_max<T>(row, V, s_redf);
        RowStat pre;  // the current kept rank prefix
        pre.mode = MODE_ALL;
        pre.kappa = 0;
        pre.i_kappa = V - 1;
        double S_pre = st.S;  // sum over the current kept set (valid if have_stats)
        if (topk_on) {
            SelCfg cfg;
            cfg.mass = false;
            cfg.M = st.M;
            cfg.c = c;
            cfg.scale = 0.f;
            cfg.restricted = false;
            uint32_t kap;
            int32_t ik;
            if (select_prefix<T>(row, V, cfg, (unsigned long long)p.top_k, sm.cand, &kap, &ik)) {
                pre.mode = MODE_PREFIX;
                pre.kappa = kap;
                pre.i_kappa = ik;
            }
            // sum over the top-k set (the list is rewritten below)
            collect_prefix<T>(row, V, pre, st.M, c, kid, kl, &S_pre);
        } else if (!have_stats) {
            collect_prefix<T>(row, V, pre, st.M, c, kid, kl, &S_pre);
        }
        if (topp_on) {
            SelCfg cfg;
            cfg.mass = true;
            cfg.M = st.M;
            cfg.c = c;
            cfg.scale = (float)(72057594037927936.0 / S_pre);  // 2^56 / S
            cfg.restricted = pre.mode == MODE_PREFIX;
            cfg.rst = pre;
            uint32_t kap;
            int32_t ik;
            if (select_prefix<T>(row, V, cfg, p.top_p_fix, sm.cand, &kap, &ik)) {
                pre.mode = MODE_PREFIX;
                pre.kappa = kap;
                pre.i_kappa = ik;
            }
        }
        double S;
        const int nk = collect_prefix<T>(row, V, pre, st.M, c, kid, kl, &S);
        st.S = S;
        st.n_kept = nk;
        st.kappa = pre.kappa;
        st.i_kappa = pre.i_kappa;
        st.mode = nk <= KCAP ? MODE_LIST : (pre.mode == MODE_ALL ? MODE_ALL : MODE_PREFIX);
    }
    if (threadIdx.x == 0) s_st = st;
    __syncthreads();
    if (threadIdx.x == 0) p.rstat[r] = s_st;
}

// ------------------------------------------------------------------------- //
// probability of one token under a merged row                               //
// ------------------------------------------------------------------------- //
template <typename T>
__device__ float token_logit(const Params& p, int r, const RowStat& st, const T* row, int x, bool* kept)
{
    if (st.mode == MODE_LIST) {
        const int32_t* ids = p.kept_id + (int64_t)r * KCAP;
        const int i = lower_bound_i32(ids, st.n_kept, x);
        *kept = i < st.n_kept && __ldcg(ids + i) == x;
        return *kept ? __ldcg(p.kept_l + (int64_t)r * KCAP + i) : -INFINITY;
    }
    const float l = Elem<T>::load_cg(row, x);
    *kept = kept_prefix(st, key_of(l), x);
    return l;
}

// P(x) of a merged row, in fp32 with an accurate exponential
template <typename T>
__device__ float token_prob(const Params& p, int r, const RowStat& st, const T* row, int x)
{
    bool kept;
    const float l = token_logit<T>(p, r, st, row, x, &kept);
    if (!kept) return 0.f;
    return (float)((double)exp2f((l - st.M) * p.c) / st.S);
}

// ------------------------------------------------------------------------- //
// inverse CDF over an explicit kept list (ascending id), in this CTA        //
// R(v) = max(0, P_t(v) - P_d(v)) for a residual, else P_t(v)                //
// ------------------------------------------------------------------------- //
struct DraftRef {
    int kind;           // 0: logits row (r >= 0), 1: probabilities row
    int r;
    RowStat st;
    const void* row;    // draft logits (T) or probabilities (float)
};

template <typename T>
__device__ __forceinline__ float draft_prob(const Params& p, const DraftRef& d, int v)
{
    if (d.kind == 1) return __ldcg((const float*)d.row + v);
    return token_prob<T>(p, d.r, d.st, (const T*)d.row, v);
}

template <typename T>
__device__ __forceinline__ unsigned long long list_r_fix(const Params& p, const RowStat& ts, float l,
                                                         int v, bool residual, const DraftRef& d)
{
    const float pt = ex2_fast((l - ts.M) * p.c) * (float)(1.0 / ts.S);
    const float r = residual ? fmaxf(pt - draft_prob<T>(p, d, v), 0.f) : pt;
    return to_fix56(r);
}

// Inverse CDF over the target's kept list in ascending id.  Returns the token;
// *Zfix the residual mass (2^-56 units) before any fallback; *zero when the
// residual summed to 0 and the target row itself was sampled.
template <typename T>
__device__ int sample_list(const Params& p, int tr, const RowStat& ts, bool residual,
                           const DraftRef& d, float u, unsigned long long* Zfix, bool* zero)
{
    __shared__ unsigned long long s_red[NT / 32 + 1];
    __shared__ int s_tok;
    const int n = ts.n_kept;
    const int32_t* ids = p.kept_id + (int64_t)tr * KCAP;
    const float* ls = p.kept_l + (int64_t)tr * KCAP;
    const int ept = (n + NT - 1) / NT;
    const int i0 = threadIdx.x * ept;
    *zero = false;
    for (int attempt = 0; attempt < 2; ++attempt) {
        const bool res = residual && attempt == 0;
        unsigned long long part = 0;
        for (int q = 0; q < ept; ++q) {
            const int i = i0 + q;
            if (i >= n) break;
            part += list_r_fix<T>(p, ts, __ldcg(ls + i), __ldcg(ids + i), res, d);
        }
        unsigned long long Z;
        const unsigned long long ex = block_excl_scan<unsigned long long>(part, s_red, &Z);
        if (attempt == 0) *Zfix = Z;
        if (Z == 0ull) {
            if (res) {
                *zero = true;
                continue;
            }
            return -1;
        }
        const unsigned long long t = cdf_target(u, Z);
        if (threadIdx.x == 0) s_tok = -1;
        __syncthreads();
        if (ex <= t && t < ex + part) {
            unsigned long long acc = ex;
            for (int q = 0; q < ept; ++q) {
                const int i = i0 + q;
                if (i >= n) break;
                acc += list_r_fix<T>(p, ts, __ldcg(ls + i), __ldcg(ids + i), res, d);
                if (acc > t) {
                    s_tok = __ldcg(ids + i);
                    break;
                }
            }
        }
        __syncthreads();
        return s_tok;
    }
    return -1;
}

// ------------------------------------------------------------------------- //
// the decision of one sequence (verify launch)                              //
// ------------------------------------------------------------------------- //
template <typename T>
__device__ void decide_sequence(const Params& p, int b)
{
    __shared__ int s_jstar, s_bad, s_nonfinite;
    const int K = p.Kmax, V = p.V;
    const int kb = seq_k(p, b);
    const T* target = (const T*)p.target;
    const int64_t trow0 = (int64_t)b * (K + 1) * V;
    const int64_t drow0 = (int64_t)b * K * V;
    if (threadIdx.x == 0) {
        s_jstar = kb;
        s_bad = 0;
        s_nonfinite = 0;
    }
    __syncthreads();
    for (int j = threadIdx.x; j < kb; j += NT) {
        const int x = p.xin[(int64_t)b * K + j];
        if (x < 0 || x >= V) s_bad = 1;
    }
    for (int j = threadIdx.x; j <= kb; j += NT) {
        if (load_rowstat(p.rstat + target_slot(p, b, j)).flags & FLAG_NONFINITE) s_nonfinite = 1;
        if (j < kb && p.draft_kind == 0 && (load_rowstat(p.rstat + draft_slot(p, b, j)).flags & FLAG_NONFINITE))
            s_nonfinite = 1;
    }
    __syncthreads();
    if (!s_bad && p.draft_kind == 1) {
        for (int j = threadIdx.x; j < kb; j += NT) {
            const int x = p.xin[(int64_t)b * K + j];
            const float q = __ldcg((const float*)p.draft + drow0 + (int64_t)j * V + x);
            if (!(q >= 0.f) || q == INFINITY) s_nonfinite = 1;
        }
    }
    __syncthreads();
    if (s_bad || s_nonfinite) {
        for (int j = threadIdx.x; j <= K; j += NT) {
            p.tokens[(int64_t)b * (K + 1) + j] = -1;
            if (p.lse) p.lse[(int64_t)b * (K + 1) + j] = NAN;
            if (j < K) {
                if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = NAN;
                if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = NAN;
            }
        }
        if (threadIdx.x == 0) {
            p.num_accepted[b] = -1;
            if (p.row_status) p.row_status[b] = s_bad ? ROW_BAD_TOKEN : ROW_NONFINITE;
            if (p.resid_mass) p.resid_mass[b] = NAN;
            p.jobs[b].kind = JOB_NONE;
        }
        return;
    }
    // accept tests of every slot (independent), first rejection by a min
    for (int j = threadIdx.x; j < kb; j += NT) {
        const int x = p.xin[(int64_t)b * K + j];
        const int tr = target_slot(p, b, j);
        const RowStat ts = load_rowstat(p.rstat + tr);
        const float pt = token_prob<T>(p, tr, ts, target + trow0 + (int64_t)j * V, x);
        float pd;
        if (p.draft_kind == 1) {
            pd = __ldcg((const float*)p.draft + drow0 + (int64_t)j * V + x);
        } else {
            const int dr = draft_slot(p, b, j);
            pd = token_prob<T>(p, dr, load_rowstat(p.rstat + dr), (const T*)p.draft + drow0 + (int64_t)j * V, x);
        }
        const uint4 w = slot_words(p, b, j, 0u);
        const float u_acc = u24(w.x);
        const double ratio = (double)pt / (double)pd;  // IEEE: pd = 0 gives inf or NaN
        const bool accept = (double)u_acc < ratio;
        if (!accept) atomicMin(&s_jstar, j);
        if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = pt;
        if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = pd;
    }
    for (int j = threadIdx.x; j <= K; j += NT) {
        if (p.lse) {
            float v = NAN;
            if (j <= kb) {
                const RowStat ts = load_rowstat(p.rstat + target_slot(p, b, j));
                v = (float)((double)ts.M / (double)p.T + log(ts.S));
            }
            p.lse[(int64_t)b * (K + 1) + j] = v;
        }
        if (j >= kb && j < K) {
            if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = NAN;
            if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = NAN;
        }
    }
    __syncthreads();
    const int jstar = s_jstar;
    for (int j = threadIdx.x; j <= K; j += NT)
        p.tokens[(int64_t)b * (K + 1) + j] = (j < jstar) ? p.xin[(int64_t)b * K + j] : -1;
    const bool residual = jstar < kb;
    const uint4 w = slot_words(p, b, jstar, 0u);
    const float u = u24(w.y);
    const int tr = target_slot(p, b, jstar);
    const RowStat ts = load_rowstat(p.rstat + tr);
    if (threadIdx.x == 0) {
        p.num_accepted[b] = jstar;
        if (p.row_status) p.row_status[b] = ROW_OK;
        if (p.resid_mass && !residual) p.resid_mass[b] = 0.f;
    }
    DraftRef d;
    d.kind = p.draft_kind;
    d.r = residual ? draft_slot(p, b, jstar) : -1;
    if (residual && d.kind == 0) d.st = load_rowstat(p.rstat + d.r);
    d.row = residual ? (const void*)((const char*)p.draft + (drow0 + (int64_t)jstar * V) *
                                                            (d.kind == 1 ? 4 : (int64_t)sizeof(T)))
                     : nullptr;
    if (ts.mode == MODE_LIST) {
        unsigned long long Z;
        bool zero;
        const int tok = sample_list<T>(p, tr, ts, residual, d, u, &Z, &zero);
        if (threadIdx.x == 0) {
            p.tokens[(int64_t)b * (K + 1) + jstar] = tok;
            if (residual && p.resid_mass) p.resid_mass[b] = (float)from_fix56(Z);
            if (zero && p.row_status) p.row_status[b] = ROW_ZERO_RESIDUAL;
            p.jobs[b].kind = JOB_NONE;
        }
    } else if (threadIdx.x == 0) {
        Job jb;
        jb.kind = residual ? JOB_RESIDUAL : JOB_ROW;
        jb.trow = tr;
        jb.drow = residual ? d.r : -1;
        jb.out_idx = b * (K + 1) + jstar;
        jb.b = b;
        jb.u = u;
        p.jobs[b] = jb;
    }
}

// the draft-side sampler: sample row r from its own distribution (tag 1)
template <typename T>
__device__ void sample_own_row(const Params& p, int r, const RowRef& rr)
{
    const RowStat st = load_rowstat(p.rstat + r);
    const int out = rr.b * p.Kmax + rr.j;
    const int jidx = rr.b * p.Kmax + rr.j;  // one job slot per draft row
    if (st.flags & FLAG_NONFINITE) {
        if (threadIdx.x == 0) {
            p.tokens[out] = -1;
            p.jobs[jidx].kind = JOB_NONE;
        }
        return;
    }
    const uint4 w = slot_words(p, rr.b, rr.j, 1u);
    const float u = u24(w.x);
    if (st.mode == MODE_LIST) {
        DraftRef d;
        d.kind = 0;
        d.r = -1;
        d.row = nullptr;
        unsigned long long Z;
        bool zero;
        const int tok = sample_list<T>(p, r, st, false, d, u, &Z, &zero);
        if (threadIdx.x == 0) {
            p.tokens[out] = tok;
            p.jobs[jidx].kind = JOB_NONE;
        }
    } else if (threadIdx.x == 0) {
        Job jb;
        jb.kind = JOB_ROW;
        jb.trow = r;
        jb.drow = -1;
        jb.out_idx = out;
        jb.b = rr.b;
        jb.u = u;
        p.jobs[jidx] = jb;
    }
}

// ------------------------------------------------------------------------- //
// stage-1 kernel: one CTA per (row slot, segment)                           //
// ------------------------------------------------------------------------- //
template <typename T, bool VEC, int MODE>
__global__ void __launch_bounds__(NT, 4) k_rows(const Params p)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ float s_redf[NT / 32 + 1];
    __shared__ double s_redd[NT / 32 + 1];
    __shared__ int s_last;
    const int r = blockIdx.x / p.nseg;
    const int seg = blockIdx.x - r * p.nseg;
    const RowRef rr = row_ref(p, r);
    if (!rr.valid) {
        if (seg == 0 && threadIdx.x == 0) {
            const int K = p.Kmax;
            if (!k_ok(p, rr.kb)) {
                // a sequence with K_b outside [0, K_max]: reported by its first slot
                const bool first = p.draft_launch ? rr.j == 0 : (!rr.is_draft && rr.j == 0);
                if (first) {
                    if (p.draft_launch) {
                        for (int j = 0; j < K; ++j) p.tokens[(int64_t)rr.b * K + j] = -1;
                    } else {
                        for (int j = 0; j <= K; ++j) {
                            p.tokens[(int64_t)rr.b * (K + 1) + j] = -1;
                            if (p.lse) p.lse[(int64_t)rr.b * (K + 1) + j] = NAN;
                            if (j < K && p.p_t_at) p.p_t_at[(int64_t)rr.b * K + j] = NAN;
                            if (j < K && p.p_d_at) p.p_d_at[(int64_t)rr.b * K + j] = NAN;
                        }
                        p.num_accepted[rr.b] = -1;
                        if (p.row_status) p.row_status[rr.b] = ROW_BAD_K;
                        if (p.resid_mass) p.resid_mass[rr.b] = NAN;
                        p.jobs[rr.b].kind = JOB_NONE;
                    }
                }
            } else if (p.draft_launch) {
                p.tokens[(int64_t)rr.b * K + rr.j] = -1;  // slot beyond K_b
                p.jobs[rr.b * K + rr.j].kind = JOB_NONE;
            }
        }
        return;
    }
    if (rr.is_draft && p.draft_kind == 1) return;  // probabilities: read only where needed

    const T* base = (const T*)(rr.is_draft ? p.draft : p.target);
    const T* row = base + row_elem_offset(p, rr);
    segment_pass<T, VEC, MODE>(p, row, seg, r, s_redf, s_redd);

    // last segment of the row merges it
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(&p.row_ticket[r], 1u) == (unsigned)(p.nseg - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0) p.row_ticket[r] = 0u;
    const Smem sm = smem_layout(smem_raw);
    merge_row<T>(p, row, r, sm);

    if (p.draft_launch) {
        __threadfence();
        __syncthreads();
        sample_own_row<T>(p, r, rr);
        return;
    }
    // last row of the sequence decides it
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int nrows = (rr.kb + 1) + (p.draft_kind == 0 ? rr.kb : 0);
        s_last = (atomicAdd(&p.seq_ticket[rr.b], 1u) == (unsigned)(nrows - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0) p.seq_ticket[rr.b] = 0u;
    decide_sequence<T>(p, rr.b);
}

template <typename T, bool VEC, int MODE>
static cudaError_t launch_rows_t(const Params& p, cudaStream_t s)
{
    const int64_t rows = (int64_t)p.B * p.rps;
    const int64_t grid = rows * p.nseg;
    if (grid <= 0) return cudaSuccess;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_rows<T, VEC, MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, ROWS_SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    k_rows<T, VEC, MODE><<<(unsigned)grid, NT, ROWS_SMEM, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_rows(const Params& p, int dtype, bool vec, cudaStream_t s)
{
    const bool chunk = p.seg_mode == SEG_CHUNK;
    if (dtype == 1) {
        if (vec) return chunk ? launch_rows_t<__nv_bfloat16, true, SEG_CHUNK>(p, s)
                              : launch_rows_t<__nv_bfloat16, true, SEG_SUM>(p, s);
        return chunk ? launch_rows_t<__nv_bfloat16, false, SEG_CHUNK>(p, s)
                     : launch_rows_t<__nv_bfloat16, false, SEG_SUM>(p, s);
    }
    if (vec) return chunk ? launch_rows_t<float, true, SEG_CHUNK>(p, s)
                          : launch_rows_t<float, true, SEG_SUM>(p, s);
    return chunk ? launch_rows_t<float, false, SEG_CHUNK>(p, s)
                 : launch_rows_t<float, false, SEG_SUM>(p, s);
}

}  // namespace sv
