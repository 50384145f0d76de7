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
//
// Two kernels run the same per-segment, per-row and per-sequence code:
//  * k_rows_tma (rows whose start is 16-byte aligned): persistent, two CTAs per
//    SM.  A producer warp takes work items from a global counter and streams
//    each 32 KB segment into a 3-stage shared-memory ring with bulk (TMA)
//    copies completing on mbarriers; eight compute warps consume the ring.
//    A merge runs in the stage it has just consumed, while the producer keeps
//    prefetching and the other CTA of the SM keeps streaming.
//  * k_rows: one CTA per segment, loads straight into registers (any V).
#include "sv_internal.cuh"

namespace sv {

// scratch layout of a merge (SCRATCH_BYTES)
constexpr int SC_CK = 0;                         // chunk keys, u16[MAX_CHUNKS]      (16 KB)
constexpr int SC_CAND = MAX_CHUNKS * 2;          // candidates, u64[CAND_CAP]        (8 KB)
constexpr int SC_QUAL = SC_CAND + CAND_CAP * 8;  // qualifying chunks, i32[CAND_CAP] (4 KB)
constexpr int SC_HIST = SC_QUAL + CAND_CAP * 4;  // two u32[256] histograms          (2 KB)
constexpr int SC_END = SC_HIST + 2 * 256 * 4;
static_assert(SC_END <= SCRATCH_BYTES, "merge scratch overflows");
static_assert(NBINS * 8 <= SCRATCH_BYTES, "radix histogram overflows the scratch");
static_assert(2 * KCAP * 8 <= SCRATCH_BYTES, "two staged kept lists overflow the scratch");

// ------------------------------------------------------------------------- //
// per-vector arithmetic (16 bytes: 8 bf16 or 4 f32)                           //
// ------------------------------------------------------------------------- //
template <typename T> struct Vec16;

template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ uint4 neg_inf() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
    // NaN-propagating max of two packed bf16 pairs, per half
    static __device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b)
    {
        uint32_t r;
        asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
    // the running packed max of a word's eight values (three paired maxima)
    static __device__ __forceinline__ uint32_t vmax2(uint4 w, uint32_t acc)
    {
        return max2(acc, max2(max2(w.x, w.y), max2(w.z, w.w)));
    }
    static __device__ __forceinline__ float unpack_max(uint32_t m2) { return fmax_nan(bf16_lo(m2), bf16_hi(m2)); }
    static __device__ __forceinline__ float vmax(uint4 w) { return unpack_max(max2(max2(w.x, w.y), max2(w.z, w.w))); }
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

template <typename T, int NTH> struct SegGeom {
    static constexpr int VW = Vec16<T>::N;
    static constexpr int SEG = SEG_BYTES / (int)sizeof(T);
    static constexpr int ROUNDS = SEG / (NTH * VW);
    static constexpr int CHUNK_EL = CHUNK_BYTES / (int)sizeof(T);
};

// NaN-propagating max of one lane's 16 bytes, kept packed for bf16 (two maxima
// per instruction), and its reduction over the 8 lanes of a 128-byte chunk
template <typename T> struct ChunkMax;

template <> struct ChunkMax<__nv_bfloat16> {
    using P = uint32_t;  // two bf16 maxima
    static __device__ __forceinline__ uint32_t mx(uint32_t a, uint32_t b)
    {
        __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
        __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
        __nv_bfloat162 z = __hmax2_nan(x, y);
        return *reinterpret_cast<uint32_t*>(&z);
    }
    static __device__ __forceinline__ P lane(uint4 w) { return mx(mx(w.x, w.y), mx(w.z, w.w)); }
    static __device__ __forceinline__ P shfl(P v, int o) { return mx(v, __shfl_xor_sync(0xffffffffu, v, o)); }
    static __device__ __forceinline__ float value(P v) { return fmax_nan(bf16_lo(v), bf16_hi(v)); }
    // threshold operand of the packed compares: a float threshold whose order
    // key has zero low bits compares like its upper 16 bits (a bf16) against
    // bf16 values; t2 holds that bf16 twice
    static __device__ __forceinline__ uint32_t thr2(float t)
    {
        const uint32_t h = __float_as_uint(t) >> 16;
        return h | (h << 16);
    }
    static __device__ __forceinline__ uint32_t ge2(uint32_t a, uint32_t t2)
    {
        return __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&a),
                           *reinterpret_cast<const __nv_bfloat162*>(&t2));
    }
    // does either packed maximum reach the threshold?
    static __device__ __forceinline__ bool any_ge(P v, float, uint32_t t2) { return ge2(v, t2) != 0u; }
    // bit q set iff element q of the word reaches the threshold
    static __device__ __forceinline__ uint32_t elem_mask(uint4 w, float, uint32_t t2)
    {
        const uint32_t m[4] = {ge2(w.x, t2), ge2(w.y, t2), ge2(w.z, t2), ge2(w.w, t2)};
        uint32_t e = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) e |= ((m[i] & 1u) | ((m[i] >> 15) & 2u)) << (2 * i);
        return e;
    }
};

template <> struct ChunkMax<float> {
    using P = float;
    static __device__ __forceinline__ float mx(float a, float b) { return fmax_nan(a, b); }
    static __device__ __forceinline__ P lane(uint4 w) { return Vec16<float>::vmax(w); }
    static __device__ __forceinline__ P shfl(P v, int o) { return fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o)); }
    static __device__ __forceinline__ float value(P v) { return v; }
    static __device__ __forceinline__ uint32_t thr2(float) { return 0u; }
    static __device__ __forceinline__ bool any_ge(P v, float t, uint32_t) { return v >= t; }
    static __device__ __forceinline__ uint32_t elem_mask(uint4 w, float t, uint32_t)
    {
        return (__uint_as_float(w.x) >= t ? 1u : 0u) | (__uint_as_float(w.y) >= t ? 2u : 0u) |
               (__uint_as_float(w.z) >= t ? 4u : 0u) | (__uint_as_float(w.w) >= t ? 8u : 0u);
    }
};

// ------------------------------------------------------------------------- //
// one segment: chunk-max keys (SEG_CHUNK) or (max, sum exp) (SEG_SUM), by a   //
// group of NTH threads (local index lt, barrier sync).  fetch(i) returns      //
// round i's 16-byte vector of this thread (or -inf padding).                 //
// ------------------------------------------------------------------------- //
template <typename T, int MODE, int NTH, typename F, typename SYNC>
__device__ __forceinline__ void segment_compute(const Params& p, F fetch, int seg, int r, int lt,
                                                SYNC sync, float* redf, double* redd,
                                                uint32_t* hist = nullptr)
{
    using G = SegGeom<T, NTH>;
    using CM = ChunkMax<T>;
    const int V = p.V;
    const int64_t base = (int64_t)seg * G::SEG;
    if constexpr (MODE == SEG_CHUNK) {
        // 8 consecutive lanes hold one 128-byte chunk: its NaN-propagating max
        // becomes a 16-bit order key (a lower bound of every key in the chunk)
        typename CM::P m[G::ROUNDS];
#pragma unroll
        for (int i = 0; i < G::ROUNDS; ++i) m[i] = CM::lane(fetch(i));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
#pragma unroll
            for (int i = 0; i < G::ROUNDS; ++i) m[i] = CM::shfl(m[i], o);
        }
        if ((lt & 7) == 0) {
#pragma unroll
            for (int i = 0; i < G::ROUNDS; ++i) {
                const int64_t e0 = base + ((int64_t)i * NTH + lt) * G::VW;
                if (e0 < V)
                    p.chunk[(int64_t)r * p.chunk_stride + e0 / G::CHUNK_EL] =
                        (uint16_t)(key_of(CM::value(m[i])) >> 16);
            }
        }
    } else if constexpr (MODE == SEG_HIST) {
        // bf16 rows with top-p alone: the segment max M; the count of tokens
        // at each key M16 - d, d < HIST_BINS (u8 per bin, 255 = "255 or
        // more"), into the row's histogram area (the chunk-key area); and the
        // sum of exp2((l - M) c) over the tokens below those keys.  The merge
        // rebuilds the row's mass per key from the counts (equal bf16 values
        // carry equal mass), so the nucleus cut needs no pass over the row.
        static_assert(sizeof(T) == 2, "the key histogram is for bf16 rows");
        const unsigned FULL = 0xffffffffu;
        uint4 w[G::ROUNDS];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < G::ROUNDS; ++i) {
            w[i] = fetch(i);
            m = fmax_nan(m, Vec16<T>::vmax(w[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmax_nan(m, __shfl_xor_sync(FULL, m, o));
        sync();  // the previous segment's reductions and histogram are read and cleared
        if ((lt & 31) == 0) redf[lt >> 5] = m;
        sync();
        float M = redf[0];
#pragma unroll
        for (int i = 1; i < NTH / 32; ++i) M = fmax_nan(M, redf[i]);
        float s = 0.f;
        if (M > -INFINITY && M < INFINITY) {
            const uint32_t m16 = key16_bf16(__float_as_uint(M) >> 16);
            // the lowest value counted (keys below 0x80 are -inf and NaNs)
            const uint32_t lo16 = m16 >= 0x7Fu + (HIST_BINS - 1) ? m16 - (HIST_BINS - 1) : 0x7Fu;
            const uint32_t thr = __float_as_uint(val_key16(lo16)) >> 16;
            const uint32_t thr2 = thr | (thr << 16);
            const float c = p.c, Mc = M * p.c;
            // pass 1, every token: exp2((l - M) c) summed over those below the
            // window, and a bit per token inside it (bit 8 i + 2 h + half)
            static_assert(G::ROUNDS * 8 <= 64, "a thread's tokens fit one 64-bit mask");
            uint64_t inmask = 0ull;
#pragma unroll
            for (int i = 0; i < G::ROUNDS; ++i) {
                const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const uint32_t x = ws[h];
                    const uint32_t in = ChunkMax<__nv_bfloat16>::ge2(x, thr2);  // 0xFFFF per counted half
                    const uint32_t two = (in & 1u) | ((in >> 15) & 2u);
                    inmask |= (uint64_t)two << (8 * i + 2 * h);
                    const float elo = ex2_fast(fmaf(bf16_lo(x), c, -Mc));
                    const float ehi = ex2_fast(fmaf(bf16_hi(x), c, -Mc));
                    s += (two & 1u) ? 0.f : elo;
                    s += (two & 2u) ? 0.f : ehi;
                }
            }
            // pass 2, the tokens inside the window (a few in ten): one count each
            while (inmask) {
                const int bit = __ffsll((long long)inmask) - 1;
                inmask &= inmask - 1ull;
                const uint4 v = fetch(bit >> 3);
                const int q = bit & 7;
                const uint32_t word = (q & 4) ? ((q & 2) ? v.w : v.z) : ((q & 2) ? v.y : v.x);
                const uint32_t b16 = (q & 1) ? (word >> 16) : (word & 0xFFFFu);
                atomicAdd(&hist[m16 - key16_bf16(b16)], 1u);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
        if ((lt & 31) == 0) redd[lt >> 5] = (double)s;
        sync();
        // the counts out, four u8 bins per word (saturating), and cleared
        uint32_t* out = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(p.chunk) +
                                                    (int64_t)r * p.chunk_stride * 2 + (int64_t)seg * HIST_BINS);
        for (int q = lt; q < HIST_BINS / 4; q += NTH) {
            uint32_t word = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                word |= min(hist[4 * q + j], 255u) << (8 * j);
                hist[4 * q + j] = 0u;
            }
            out[q] = word;
        }
        if (lt == 0) {
            double tot = 0.0;
#pragma unroll
            for (int i = 0; i < NTH / 32; ++i) tot += redd[i];
            SegStat st;
            st.m = M;
            st.pad = 0.f;
            st.s = tot;
            p.seg[(int64_t)r * p.nseg + seg] = st;
        }
    } else {
        // one read of the thread's words; each warp's (max, sum exp) in fp32
        // over its own max, the warps' pairs rescaled to the segment max and
        // added in fp64 by the first thread
        const unsigned FULL = 0xffffffffu;
        uint4 w[G::ROUNDS];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < G::ROUNDS; ++i) {
            w[i] = fetch(i);
            m = fmax_nan(m, Vec16<T>::vmax(w[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmax_nan(m, __shfl_xor_sync(FULL, m, o));
        float s = 0.f;
        if (m > -INFINITY && m < INFINITY) {
#pragma unroll
            for (int i = 0; i < G::ROUNDS; ++i) s += Vec16<T>::vsumexp(w[i], m, p.c);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
        sync();  // the previous segment's pairs are read
        if ((lt & 31) == 0) {
            redf[lt >> 5] = m;
            redd[lt >> 5] = (double)s;
        }
        sync();
        if (lt == 0) {
            float M = redf[0];
#pragma unroll
            for (int i = 1; i < NTH / 32; ++i) M = fmax_nan(M, redf[i]);
            double tot = 0.0;
            if (M > -INFINITY && M < INFINITY) {
#pragma unroll
                for (int i = 0; i < NTH / 32; ++i)
                    if (redf[i] > -INFINITY) tot += redd[i] * (double)exp2f((redf[i] - M) * p.c);
            }
            SegStat st;
            st.m = M;
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
    return __float2ull_rn(ex2_fast((l - cfg.M) * cfg.c) * cfg.scale);
}

// Finds the rank prefix {key > kappa} + {key == kappa, id <= i_kappa} whose last
// token is where the inclusive cumulative weight (from the top rank) first
// reaches `need`.  Returns false when the total weight is below `need` (then
// every token is kept).  hist: NBINS u64 of shared scratch.
template <typename T>
__device__ bool select_prefix(const T* row, int V, const SelCfg& cfg, unsigned long long need,
                              unsigned long long* hist, uint32_t* kappa_out, int32_t* ikappa_out)
{
    __shared__ unsigned long long s_red[NT / 32 + 1];
    __shared__ unsigned long long s_cum;
    __shared__ uint32_t s_bin;
    __shared__ int32_t s_ik;
    uint32_t pmask = 0, pval = 0;
    constexpr bool BF = sizeof(T) == 2;
    constexpr int LEVELS = BF ? 2 : 3;
    for (int lev = 0; lev < LEVELS; ++lev) {
        const int shift = lev == 0 ? 21 : (lev == 1 ? 10 : 0);
        const int nb = lev == 2 ? 1024 : 2048;
        for (int i = threadIdx.x; i < nb; i += NT) hist[i] = 0ull;
        csync();
        for (int e = threadIdx.x; e < V; e += NT) {
            const float l = Elem<T>::load_cg(row, e);
            const uint32_t k = key_of(l);
            if ((k & pmask) != pval) continue;
            if (cfg.restricted && !kept_prefix(cfg.rst, k, e)) continue;
            const unsigned long long w = sel_weight(cfg, l);
            if (w) atomicAdd(&hist[(k >> shift) & (uint32_t)(nb - 1)], w);
        }
        csync();
        const int per = nb / NT;
        unsigned long long local = 0;
        for (int q = 0; q < per; ++q) local += hist[nb - 1 - (threadIdx.x * per + q)];
        unsigned long long total;
        unsigned long long cum = block_excl_scan<unsigned long long>(local, s_red, &total);
        if (total < need) return false;  // uniform across the compute threads
        for (int q = 0; q < per; ++q) {
            const int h = nb - 1 - (threadIdx.x * per + q);
            const unsigned long long w = hist[h];
            if (cum < need && need <= cum + w) {
                s_bin = (uint32_t)h;
                s_cum = cum;
            }
            cum += w;
        }
        csync();
        need -= s_cum;
        pmask |= (uint32_t)(nb - 1) << shift;
        pval |= s_bin << shift;
        csync();
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
            break;
        }
        running += total;
    }
    csync();
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
            if (kept_prefix(fin, key_of(Elem<T>::load_cg(row, e)), e)) ++cnt;
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

template <typename T> __device__ __forceinline__ float word_elem(uint4 w, int q);

// The same for a row on 16 bytes, in one pass: coalesced rounds of LPT
// 16-byte words per thread in flight; every kept token goes to a staging
// list in shared memory (an atomic slot, id << 32 | logit bits) while the
// thread sums its mass; when the prefix has at most KCAP tokens the staging
// is sorted by id (bitonic) and written out as the ordered list.
constexpr int COLLECT_STAGE_OFF = 24576;  // staging offset in a merge's scratch (after the radix bins)
template <typename T>
__device__ int collect_prefix_vec(const T* row, int V, const RowStat& fin, float M, float c, int32_t* kid,
                                  float* kl, double* S_out, unsigned long long* stage)
{
    __shared__ int s_n;
    __shared__ double s_red_d[NT / 32 + 1];
    constexpr int VW = Vec16<T>::N;
    constexpr int LPT = 16;
    const int nw = V / VW;
    const uint4* rv = reinterpret_cast<const uint4*>(row);
    if (threadIdx.x == 0) s_n = 0;
    csync();
    float s = 0.f;
    for (int w0 = 0; w0 < nw; w0 += NT * LPT) {
        uint4 x[LPT];
#pragma unroll
        for (int j = 0; j < LPT; ++j) {
            const int w = w0 + j * NT + (int)threadIdx.x;
            x[j] = w < nw ? __ldcg(rv + w) : Vec16<T>::neg_inf();
        }
#pragma unroll
        for (int j = 0; j < LPT; ++j) {
            const int w = w0 + j * NT + (int)threadIdx.x;
#pragma unroll
            for (int q = 0; q < VW; ++q) {
                const float l = word_elem<T>(x[j], q);
                const int e = w * VW + q;
                if (w < nw && kept_prefix(fin, key_of(l), e)) {
                    s += ex2_fast((l - M) * c);
                    const int pos = atomicAdd(&s_n, 1);
                    if (pos < KCAP) stage[pos] = ((unsigned long long)(uint32_t)e << 32) | __float_as_uint(l);
                }
            }
        }
    }
    csync();
    const int total = s_n;
    *S_out = block_sum_d((double)s, s_red_d);
    if (total <= KCAP) {
        const int n2 = next_pow2(total);
        for (int i = total + (int)threadIdx.x; i < n2; i += NT) stage[i] = ~0ull;
        csync();
        bitonic_sort_u64(stage, n2);
        for (int i = threadIdx.x; i < total; i += NT) {
            kid[i] = (int32_t)(stage[i] >> 32);
            kl[i] = __uint_as_float((uint32_t)stage[i]);
        }
    }
    csync();  // the staging may be reused
    return total;
}

// the kept list of a rank prefix by whichever walk the row's alignment allows
template <typename T>
__device__ int collect_kept(const T* row, int V, const RowStat& fin, float M, float c, int32_t* kid, float* kl,
                            double* S_out, unsigned char* scratch)
{
    static_assert(COLLECT_STAGE_OFF + KCAP * 8 <= SCRATCH_BYTES && NBINS * 8 <= COLLECT_STAGE_OFF,
                  "the staging fits the scratch after the radix bins");
    if (((uintptr_t)row & 15u) == 0 && ((int64_t)V * (int64_t)sizeof(T)) % 16 == 0)
        return collect_prefix_vec<T>(row, V, fin, M, c, kid, kl, S_out,
                                     reinterpret_cast<unsigned long long*>(scratch + COLLECT_STAGE_OFF));
    return collect_prefix<T>(row, V, fin, M, c, kid, kl, S_out);
}

// ------------------------------------------------------------------------- //
// fast top-k from the chunk-max keys.  The k-th largest chunk max is a lower  //
// bound of the k-th largest key, so only chunks whose max reaches it can hold //
// a kept token; they are re-read from L2 (about k chunks of 128 bytes).       //
// Returns false when the candidates overflow (many ties): use the general     //
// path.  On success fills st (MODE_LIST, or the nonfinite flag) and the       //
// row's kept list.                                                           //
// ------------------------------------------------------------------------- //
constexpr int KEYQ = MAX_CHUNKS / 8 / NT;  // 16-byte words of chunk keys per thread
constexpr int RANK_MAX = 256;              // counting-rank sort up to this size

__device__ __forceinline__ int block_count(int v, int* red)
{
    v = __reduce_add_sync(0xffffffffu, v);
    csync();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    csync();
    int t = 0;
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) t += red[i];
    return t;
}

// sorts n distinct keys ascending from src into dst (shared): a counting rank
// for small n, a bitonic sort in place (src == dst allowed only then) otherwise
__device__ void sort_keys(const unsigned long long* src, unsigned long long* dst, int n)
{
    if (n <= RANK_MAX) {
        for (int i = threadIdx.x; i < n; i += NT) {
            const unsigned long long x = src[i];
            int rk = 0;
            for (int j = 0; j < n; ++j) rk += src[j] < x;
            dst[rk] = x;
        }
        csync();
        return;
    }
    const int n2 = next_pow2(n);
    for (int i = threadIdx.x; i < n; i += NT) dst[i] = src[i];
    for (int i = n + threadIdx.x; i < n2; i += NT) dst[i] = ~0ull;
    csync();
    bitonic_sort_u64(dst, n2);
}

// element q of a 16-byte word of T
template <typename T> __device__ __forceinline__ float word_elem(uint4 w, int q);
template <> __device__ __forceinline__ float word_elem<__nv_bfloat16>(uint4 w, int q)
{
    const uint32_t x = q < 2 ? w.x : q < 4 ? w.y : q < 6 ? w.z : w.w;
    return (q & 1) ? bf16_hi(x) : bf16_lo(x);
}
template <> __device__ __forceinline__ float word_elem<float>(uint4 w, int q)
{
    return __uint_as_float(q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w);
}

template <typename T>
__device__ bool fast_topk(const Params& p, const T* row, int r, unsigned char* scratch,
                          RowStat& st)
{
    __shared__ int s_cnt, s_nqual, s_flag, s_nk;
    __shared__ int s_red_i[NT / 32 + 1];
    unsigned long long* srt = (unsigned long long*)(scratch + SC_CK);   // sorted, CAND_CAP
    unsigned long long* cand = (unsigned long long*)(scratch + SC_CAND);
    int32_t* qual = (int32_t*)(scratch + SC_QUAL);
    const int V = p.V, k = p.top_k, nc = p.nchunk;
    const float c = p.c;
    using G = SegGeom<T, NT>;

    // chunk keys into registers, 8 per 16-byte load (row stride padded to 8)
    const uint4* ckg = reinterpret_cast<const uint4*>(p.chunk + (int64_t)r * p.chunk_stride);
    const int nw = (nc + 7) / 8;
    uint4 kv[KEYQ];
#pragma unroll
    for (int q = 0; q < KEYQ; ++q) {
        const int i = threadIdx.x + q * NT;
        kv[q] = i < nw ? __ldcg(ckg + i) : make_uint4(0, 0, 0, 0);
    }
    // key e of word q of this thread (0 for padding: below every real key)
    auto key_at = [&](int q, int e) -> uint32_t {
        const int idx = (threadIdx.x + q * NT) * 8 + e;
        const uint32_t w = e < 2 ? kv[q].x : e < 4 ? kv[q].y : e < 6 ? kv[q].z : kv[q].w;
        return idx < nc ? ((w >> ((e & 1) * 16)) & 0xFFFFu) : 0u;
    };
    const int lane = threadIdx.x & 31;
    uint32_t kmax = 0;
    bool bad = false;
#pragma unroll
    for (int q = 0; q < KEYQ; ++q)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t key = key_at(q, e);
            kmax = max(kmax, key);
            bad |= key >= 0xFF80u;  // +inf or NaN
        }
    if (threadIdx.x == 0) {
        s_cnt = 0;
        s_nqual = 0;
    }
    bad = csync_or(bad, &s_flag);
    kmax = (uint32_t)__reduce_max_sync(0xffffffffu, kmax);
    if ((threadIdx.x & 31) == 0) s_red_i[threadIdx.x >> 5] = (int)kmax;
    csync();
    kmax = 0;
    for (int i = 0; i < NT / 32; ++i) kmax = max(kmax, (uint32_t)s_red_i[i]);
    csync();
    if (bad || kmax <= 0x007Fu) {  // NaN / +inf, or no finite logit
        st.flags = FLAG_NONFINITE;
        return true;
    }
    // tau16 = max{t : count(key >= t) >= k}, one 4-bit digit per level: 15
    // counts per level, per-warp sums in a double-buffered table, no atomics
    const int warp = threadIdx.x >> 5;
    const int wbase = warp * 32;  // first key word of this warp at q = 0
    uint32_t tau16 = 0;
    {
        __shared__ int s_cnt15[2][NT / 32][16];
        for (int lev = 0; lev < 4; ++lev) {
            const int shift = 12 - 4 * lev;
            int cnt[15];
#pragma unroll
            for (int d = 0; d < 15; ++d) cnt[d] = 0;
#pragma unroll
            for (int q = 0; q < KEYQ; ++q) {
                if (wbase + q * NT >= nw) continue;  // warp-uniform: no keys here
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t key = key_at(q, e);
#pragma unroll
                    for (int d = 0; d < 15; ++d) cnt[d] += key >= tau16 + ((uint32_t)(d + 1) << shift);
                }
            }
#pragma unroll
            for (int d = 0; d < 15; ++d) {
                const int w = __reduce_add_sync(0xffffffffu, cnt[d]);
                if (lane == d) s_cnt15[lev & 1][warp][d] = w;
            }
            csync();
            int dsel = 0;
#pragma unroll
            for (int d = 0; d < 15; ++d) {
                int t = 0;
#pragma unroll
                for (int wi = 0; wi < NT / 32; ++wi) t += s_cnt15[lev & 1][wi][d];
                if (t >= k) dsel = d + 1;  // counts fall with d: the last that holds
            }
            tau16 += (uint32_t)dsel << shift;
        }
    }
    const uint32_t tau32 = tau16 << 16;
    // chunks that can hold a kept token, in ascending chunk order (block scan)
    {
        int mine = 0;
#pragma unroll
        for (int q = 0; q < KEYQ; ++q)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t key = key_at(q, e);
                mine += key >= tau16 && key > 0;
            }
        int tot;
        int off = block_excl_scan<int>(mine, s_red_i, &tot);
        if (threadIdx.x == 0) s_nqual = tot;
#pragma unroll
        for (int q = 0; q < KEYQ; ++q)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t key = key_at(q, e);
                if (key >= tau16 && key > 0) {
                    if (off < CAND_CAP) qual[off] = (threadIdx.x + q * NT) * 8 + e;
                    ++off;
                }
            }
    }
    csync();
    const int nq = s_nqual;
    if (nq > CAND_CAP) return false;

    // gather: the qualifying chunks as 16-byte words, all loads in flight at once
    constexpr int WPC = CHUNK_BYTES / 16;           // words per chunk
    constexpr int EPW = 16 / (int)sizeof(T);        // elements per word
    const int nwords = nq * WPC;
    const char* rowb = (const char*)row;
    const bool aligned = ((uintptr_t)row & 15u) == 0;  // else: element loads
    uint4 gw[4];
    int gi[4];
    for (int base = 0; base < nwords; base += NT * 4) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int wi = base + g * NT + threadIdx.x;
            gi[g] = -1;
            gw[g] = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
            if (wi < nwords) {
                const int e0 = qual[wi / WPC] * G::CHUNK_EL + (wi % WPC) * EPW;
                if (e0 < V) {
                    gi[g] = e0;
                    if (aligned)
                        gw[g] = __ldcg(reinterpret_cast<const uint4*>(rowb + (int64_t)e0 * (int64_t)sizeof(T)));
                    else
                        gw[g] = Vec16<T>::load_scalar(row, e0, V);
                }
            }
        }
        int cnt = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int q = 0; q < EPW; ++q)
                cnt += gi[g] >= 0 && gi[g] + q < V && key_of(word_elem<T>(gw[g], q)) >= tau32;
        int tot;
        int off = s_cnt + block_excl_scan<int>(cnt, s_red_i, &tot);
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int q = 0; q < EPW; ++q) {
                const uint32_t key = key_of(word_elem<T>(gw[g], q));
                if (gi[g] >= 0 && gi[g] + q < V && key >= tau32) {
                    if (off < CAND_CAP)
                        cand[off] = ((unsigned long long)(~key) << 32) | (uint32_t)(gi[g] + q);
                    ++off;
                }
            }
        csync();
        if (threadIdx.x == 0) s_cnt += tot;
        csync();
    }
    const int n = s_cnt;
    if (n > CAND_CAP) return false;

    // exact order: key descending, then id ascending
    sort_keys(cand, srt, n);
    const int kk = min(k, n);
    const float M = val_of(~(uint32_t)(srt[0] >> 32));
    // sum over the kept ranks by warp 0 (no block barrier)
    __shared__ double s_S;
    if (threadIdx.x < 32) {
        float e_loc = 0.f;
        for (int i = lane; i < kk; i += 32) e_loc += ex2_fast((val_of(~(uint32_t)(srt[i] >> 32)) - M) * c);
        const double t = warp_sum_d((double)e_loc);
        if (lane == 0) s_S = t;
    }
    csync();
    double S = s_S;
    int nk = kk;
    if (p.top_p < 1.0f) {
        // strict prefix rule over the kept ranks, in fp64 (one warp scans)
        if (threadIdx.x < 32) {
            double pre = 0.0;
            int stop = kk;
            for (int b0 = 0; b0 < kk; b0 += 32) {
                const int i = b0 + lane;
                const double pv =
                    i < kk ? (double)ex2_fast((val_of(~(uint32_t)(srt[i] >> 32)) - M) * c) / S : 0.0;
                double x = pv;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const double y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                const double before = pre + (x - pv);  // mass strictly before rank i
                const unsigned drop =
                    __ballot_sync(0xffffffffu, i < kk && !(before < (double)p.top_p));
                if (drop) {
                    stop = b0 + __ffs(drop) - 1;
                    break;
                }
                pre += __shfl_sync(0xffffffffu, x, 31);
            }
            if (lane == 0) s_nk = stop;
        }
        csync();
        nk = s_nk;
        if (threadIdx.x < 32) {
            float e2 = 0.f;
            for (int i = lane; i < nk; i += 32) e2 += ex2_fast((val_of(~(uint32_t)(srt[i] >> 32)) - M) * c);
            const double t = warp_sum_d((double)e2);
            if (lane == 0) s_S = t;
        }
        csync();
        S = s_S;
    }
    // the kept list in ascending id: re-key as (id << 32 | key) and sort again
    for (int i = threadIdx.x; i < nk; i += NT) {
        const unsigned long long x = srt[i];
        cand[i] = ((unsigned long long)(uint32_t)x << 32) | (uint32_t)(~(uint32_t)(x >> 32));
    }
    csync();
    sort_keys(cand, srt, nk);
    int32_t* kid = p.kept_id + (int64_t)r * KCAP;
    float* kl = p.kept_l + (int64_t)r * KCAP;
    for (int i = threadIdx.x; i < nk; i += NT) {
        const unsigned long long x = srt[i];
        kid[i] = (int32_t)(x >> 32);
        kl[i] = val_of((uint32_t)x);
    }
    st.M = M;
    st.S = S;
    st.n_kept = nk;
    st.mode = MODE_LIST;
    return true;
}

// ------------------------------------------------------------------------- //
// the nucleus of a bf16 row from its per-segment key histograms (SEG_HIST)  //
// ------------------------------------------------------------------------- //
// sum over the row of exp2((l - M) c), read from L2 / HBM (NT threads)
template <typename T>
__device__ double row_sumexp(const T* row, int V, float M, float c, double* red)
{
    float s = 0.f;
    for (int e = threadIdx.x; e < V; e += NT) s += ex2_fast((Elem<T>::load_cg(row, e) - M) * c);
    return block_sum_d((double)s, red);
}

// exp2((v - M) c) for the bf16 value of key k: the exponent in two parts (c +
// c_lo) so that it is exact to ~2^-40, its fractional part through exp2f
__device__ __forceinline__ float hist_weight(const Params& p, uint32_t k, float M)
{
    const float d = val_key16(k) - M;  // exact: two bf16 values
    if (!(d > -INFINITY)) return 0.f;
    const float x = d * p.c;
    const float x_lo = fmaf(d, p.c, -x) + d * p.c_lo;  // the rounding of d c, and d c_lo
    const float n = rintf(x);  // <= 0: v <= M
    if (n < -126.f) return 0.f;  // below 2^-126 of the max token's: no mass at fp32 range
    return exp2f((x - n) + x_lo) * __int_as_float(((int)n + 127) << 23);  // an exact power-of-two scale
}

// Finds the nucleus (top-p after temperature, no top-k) of row r from the
// segments' key histograms: the row's count per key in the HIST_BINS keys
// below its max, each key's mass count x exp2((v - M) c), the tokens below
// that window from the segments' partial sums; the rank prefix is cut where
// the mass before a token reaches top_p.  Ties at the cut key are kept in
// ascending id, found in the one segment that holds the boundary token.
// Returns 0 with st complete (MODE_PREFIX; the caller builds a list if small),
// 1 when the cut lies below the window (st.S then holds the row's total), 2
// when a bin saturated (the caller recomputes everything).  NT threads.
template <typename T>
__device__ int merge_row_hist(const Params& p, const T* row, int r, RowStat& st, unsigned char* scratch)
{
    static_assert(HIST_BINS == NT, "one row bin per thread");
    __shared__ double s_redd[NT / 32 + 1];
    __shared__ int s_redi[NT / 32 + 1];
    __shared__ int s_flag;
    __shared__ int s_cut;
    __shared__ double s_above;
    __shared__ int s_cnt_above;
    __shared__ int s_seg;
    __shared__ int s_before;
    __shared__ int s_id;
    __shared__ int s_cntk;
    const int t = threadIdx.x;
    const float M = st.M;
    const uint32_t M16 = key16_bf16(__float_as_uint(M) >> 16);
    const SegStat* segs = p.seg + (int64_t)r * p.nseg;
    // the segment maxima, partial sums and key histograms, staged in shared
    // memory with one round of loads
    float* s_m = reinterpret_cast<float*>(scratch);                       // [nseg]
    double* s_s = reinterpret_cast<double*>(scratch + 1024);              // [nseg]
    uint8_t* Hs = scratch + 2048;                                         // [nseg][HIST_BINS]
    static_assert(2048 + (NT / 2) * HIST_BINS <= SCRATCH_BYTES, "the histograms of a row fit the scratch");
    {
        const uint4* Hg = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.chunk) +
                                                         (int64_t)r * p.chunk_stride * 2);
        for (int i = t; i < p.nseg * (HIST_BINS / 16); i += NT) reinterpret_cast<uint4*>(Hs)[i] = __ldcg(Hg + i);
        for (int i = t; i < p.nseg; i += NT) {
            s_m[i] = __ldcg(&segs[i].m);
            s_s[i] = __ldcg(&segs[i].s);
        }
    }
    csync();
    uint32_t cnt = 0;      // tokens at key M16 - t
    double below = 0.0;    // mass of this thread's share of the tokens below the window
    bool sat = false;
    for (int s = 0; s < p.nseg; ++s) {
        const float ms = s_m[s];
        if (!(ms > -INFINITY)) continue;  // every token -inf
        const uint32_t m16 = key16_bf16(__float_as_uint(ms) >> 16);
        const uint32_t off = M16 - m16;  // the segment's window starts off keys below the row's
        if ((uint32_t)t >= off) {
            const uint32_t c = Hs[s * HIST_BINS + (t - off)];
            sat |= c == 255u;
            cnt += c;
        }
        if (off + (uint32_t)t >= (uint32_t)HIST_BINS) {
            const uint32_t c = Hs[s * HIST_BINS + t];
            sat |= c == 255u;
            if (c) below += (double)c * (double)hist_weight(p, m16 - (uint32_t)t, M);
        }
        if (t == 0) below += s_s[s] * (double)exp2f((ms - M) * p.c);
    }
    if (csync_or(sat, &s_flag)) return 2;
    const uint32_t key = M16 - (uint32_t)t;
    const float w = key >= 0x80u ? hist_weight(p, key, M) : 0.f;
    const double mass = (double)cnt * (double)w;
    double tot;
    const double cum_ex = block_excl_scan<double>(mass, s_redd, &tot);
    const double S_all = tot + block_sum_d(below, s_redd);
    const double target = (double)p.top_p * S_all;
    if (t == 0) s_cut = -1;
    csync();
    // the first key whose inclusive mass reaches the target (strict rule:
    // a token is kept while the mass before it is below top_p)
    if (cum_ex < target && cum_ex + mass >= target && cnt > 0) {
        s_cut = t;
        s_above = cum_ex;
    }
    int n_above_total;
    const int n_before = block_excl_scan<int>((int)cnt, s_redi, &n_above_total);
    csync();
    const int cut = s_cut;
    if (cut < 0) {
        st.S = S_all;
        return 1;
    }
    if (t == cut) s_cnt_above = n_before;
    csync();
    (void)n_above_total;
    const uint32_t kap16 = M16 - (uint32_t)cut;
    const float wk = hist_weight(p, kap16, M);
    const double above = s_above;
    if (t == cut) s_cntk = (int)cnt;
    csync();
    const int cntk = s_cntk;
    const double q = (target - above) / (double)wk;
    int nk = (int)ceil(q);
    nk = max(1, min(nk, cntk));
    int32_t ik = p.V - 1;
    if (nk < cntk) {
        // the nk-th token of key kap16 in ascending id: which segment holds it
        // (its count of that key is a bin of its histogram), then a walk of
        // that segment in id order
        using G = SegGeom<T, NT>;
        int cs = 0;
        if (t < p.nseg) {
            const float ms = s_m[t];
            if (ms > -INFINITY) {
                const uint32_t m16 = key16_bf16(__float_as_uint(ms) >> 16);
                if (m16 >= kap16 && m16 - kap16 < (uint32_t)HIST_BINS) cs = (int)Hs[t * HIST_BINS + (m16 - kap16)];
            }
        }
        static_assert(NT >= 64, "segments of a row fit one thread each up to NT");
        int dummy;
        if (t == 0) {
            s_seg = 0;
            s_before = 0;
        }
        const int cb = block_excl_scan<int>(cs, s_redi, &dummy);
        if (t < p.nseg && cb < nk && nk <= cb + cs) {
            s_seg = t;
            s_before = cb;
        }
        csync();
        const int sseg = s_seg;
        const int need = nk - s_before;  // 1-based rank of the boundary token in the segment
        const int e_begin = sseg * G::SEG;
        const int e_end = min(p.V, e_begin + G::SEG);
        constexpr int EPT = G::SEG / NT;  // contiguous elements per thread
        constexpr int WPT = EPT / 8;      // their 16-byte words, loaded in one round
        static_assert(EPT % 8 == 0, "a thread's tokens are whole words");
        const int e0 = e_begin + t * EPT;
        uint4 wv[WPT];
#pragma unroll
        for (int j = 0; j < WPT; ++j)
            wv[j] = e0 + 8 * j < e_end ? __ldcg(reinterpret_cast<const uint4*>((const unsigned short*)row + e0 + 8 * j))
                                       : make_uint4(0, 0, 0, 0);
        // bit 8 j + h: token e0 + 8 j + h has key kap16 (a row on 16 bytes
        // holds whole words up to e_end)
        uint32_t hit[WPT];
        int mine = 0;
#pragma unroll
        for (int j = 0; j < WPT; ++j) {
            const uint32_t xw[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
            hit[j] = 0u;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const uint32_t b16 = (h & 1) ? (xw[h >> 1] >> 16) : (xw[h >> 1] & 0xFFFFu);
                if (e0 + 8 * j + h < e_end && key16_bf16(b16) == kap16) hit[j] |= 1u << h;
            }
            mine += __popc(hit[j]);
        }
        const int mb = block_excl_scan<int>(mine, s_redi, &dummy);
        if (t == 0) s_id = p.V - 1;
        csync();
        if (mb < need && need <= mb + mine) {
            int seen = mb;
#pragma unroll
            for (int j = 0; j < WPT; ++j) {
                if (seen + __popc(hit[j]) >= need) {
                    uint32_t m = hit[j];
                    for (int q = 0; q < need - seen - 1; ++q) m &= m - 1u;  // drop the earlier hits
                    s_id = e0 + 8 * j + __ffs(m) - 1;
                    break;
                }
                seen += __popc(hit[j]);
            }
        }
        csync();
        ik = s_id;
    }
    st.mode = MODE_PREFIX;
    st.kappa = key_of(val_key16(kap16));
    st.i_kappa = ik;
    st.n_kept = s_cnt_above + nk;
    st.S = above + (double)nk * (double)wk;
    return 0;
}

// ------------------------------------------------------------------------- //
// row merge: statistics and kept set of row slot r                          //
// ------------------------------------------------------------------------- //
template <typename T>
__device__ void merge_row(const Params& p, const T* row, int r, unsigned char* scratch)
{
    __shared__ float s_redf[NT / 32 + 1];
    __shared__ double s_redd[NT / 32 + 1];
    __shared__ RowStat s_st;
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
        done = fast_topk<T>(p, row, r, scratch, st);
        csync();
    } else {
        // statistics over all tokens from the segment records
        float m = -INFINITY;
        for (int i = threadIdx.x; i < p.nseg; i += NT)
            m = fmax_nan(m, __ldcg(&p.seg[(int64_t)r * p.nseg + i].m));
        const float M = block_max_nan(m, s_redf);
        if (!(M > -INFINITY && M < INFINITY)) {
            st.flags = FLAG_NONFINITE;
            done = true;
        } else {
            // (the key-histogram path sums its own, from the histograms)
            const bool hist_path = sizeof(T) == 2 && p.seg_mode == SEG_HIST && topp_on && !topk_on;
            double s = 0.0;
            for (int i = threadIdx.x; i < p.nseg && !hist_path; i += NT) {
                const SegStat* g = p.seg + (int64_t)r * p.nseg + i;
                const float gm = __ldcg(&g->m);
                if (gm > -INFINITY)
                    s += __ldcg(&g->s) * exp2(((double)gm - (double)M) * (double)c);
            }
            st.M = M;
            st.S = hist_path ? 0.0 : block_sum_d(s, s_redd);
            have_stats = true;
            if (!topk_on && !topp_on) done = true;  // MODE_ALL
            if constexpr (sizeof(T) == 2) if (p.seg_mode == SEG_HIST && topp_on && !topk_on) {
                // the segment records hold only the mass below each key window:
                // the histograms give the rest and the nucleus itself
                const int h = merge_row_hist<T>(p, row, r, st, scratch);
                if (h == 0) {
                    if (st.n_kept <= KCAP) {  // a small nucleus becomes a list (one pass)
                        double S;
                        const int nk = collect_kept<T>(row, V, st, st.M, c, kid, kl, &S, scratch);
                        st.S = S;
                        st.n_kept = nk;
                        st.mode = MODE_LIST;
                    }
                    done = true;
                } else if (h == 2) {
                    st.S = row_sumexp<T>(row, V, st.M, c, s_redd);  // a bin saturated: the plain sum
                }
                // h == 1: st.S is the row's total; the radix descent below finds the cut
            }
        }
    }

    if (!done) {
        // general path: radix descent over the full row (read from L2)
        unsigned long long* hist = (unsigned long long*)scratch;
        if (!have_stats) {
            st.M = row_max<T>(row, V, s_redf);
            if (!(st.M > -INFINITY && st.M < INFINITY)) st.flags = FLAG_NONFINITE;
        }
        if (!st.flags) {
            RowStat pre;  // the current kept rank prefix
            pre.mode = MODE_ALL;
            pre.kappa = 0;
            pre.i_kappa = V - 1;
            double S_pre = st.S;
            if (topk_on) {
                SelCfg cfg;
                cfg.mass = false;
                cfg.M = st.M;
                cfg.c = c;
                cfg.scale = 0.f;
                cfg.restricted = false;
                uint32_t kap;
                int32_t ik;
                if (select_prefix<T>(row, V, cfg, (unsigned long long)p.top_k, hist, &kap, &ik)) {
                    pre.mode = MODE_PREFIX;
                    pre.kappa = kap;
                    pre.i_kappa = ik;
                }
                if (topp_on) collect_kept<T>(row, V, pre, st.M, c, kid, kl, &S_pre, scratch);
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
                if (select_prefix<T>(row, V, cfg, p.top_p_fix, hist, &kap, &ik)) {
                    pre.mode = MODE_PREFIX;
                    pre.kappa = kap;
                    pre.i_kappa = ik;
                }
            }
            double S;
            const int nk = collect_kept<T>(row, V, pre, st.M, c, kid, kl, &S, scratch);
            st.S = S;
            st.n_kept = nk;
            st.kappa = pre.kappa;
            st.i_kappa = pre.i_kappa;
            st.mode = nk <= KCAP ? MODE_LIST : (pre.mode == MODE_ALL ? MODE_ALL : MODE_PREFIX);
        }
    }
    if (threadIdx.x == 0) s_st = st;
    csync();
    if (threadIdx.x == 0) p.rstat[r] = s_st;
}

// ------------------------------------------------------------------------- //
// inverse CDF over the target's kept list (ascending id), in this CTA.       //
// R(v) = max(0, P_t(v) - P_d(v)) for a residual, else P_t(v).  Both lists   //
// are staged in shared scratch first.                                       //
// ------------------------------------------------------------------------- //
struct DraftRef {
    int kind;           // 0: logits row (merged stats st), 1: probabilities row
    int r;
    RowStat st;
    const void* row;    // draft logits (T) or probabilities (float)
};

struct StagedList {
    const int32_t* ids;
    const float* ls;
    int n;
};

__device__ __forceinline__ int lower_bound_smem(const int32_t* a, int n, int x)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

template <typename T>
__device__ __forceinline__ float staged_draft_prob(const Params& p, const DraftRef& d,
                                                   const StagedList& dl, float invSd, int v)
{
    if (d.kind == 1) return __ldcg((const float*)d.row + v);
    if (d.st.mode == MODE_LIST) {
        const int i = lower_bound_smem(dl.ids, dl.n, v);
        return (i < dl.n && dl.ids[i] == v) ? ex2_fast((dl.ls[i] - d.st.M) * p.c) * invSd : 0.f;
    }
    const float l = Elem<T>::load_cg((const T*)d.row, v);
    return kept_prefix(d.st, key_of(l), v) ? ex2_fast((l - d.st.M) * p.c) * invSd : 0.f;
}

template <typename T>
__device__ __forceinline__ unsigned long long list_r_fix(const Params& p, const RowStat& ts,
                                                         const StagedList& tl, int i, bool res,
                                                         const DraftRef& d, const StagedList& dl,
                                                         float invSt, float invSd)
{
    const float pt = ex2_fast((tl.ls[i] - ts.M) * p.c) * invSt;
    const float rv = res ? fmaxf(pt - staged_draft_prob<T>(p, d, dl, invSd, tl.ids[i]), 0.f) : pt;
    return to_fix56(rv);
}

template <typename T>
__device__ int sample_list(const Params& p, int tr, const RowStat& ts, bool residual,
                           const DraftRef& d, float u, unsigned char* scratch,
                           unsigned long long* Zfix, bool* zero)
{
    __shared__ unsigned long long s_red[NT / 32 + 1];
    __shared__ int s_tok;
    const int n = ts.n_kept;
    int32_t* ti = (int32_t*)scratch;
    float* tv = (float*)(scratch + KCAP * 4);
    int32_t* di = (int32_t*)(scratch + KCAP * 8);
    float* dv = (float*)(scratch + KCAP * 12);
    StagedList tl{ti, tv, n}, dl{di, dv, 0};
    {
        const int32_t* gi = p.kept_id + (int64_t)tr * KCAP;
        const float* gv = p.kept_l + (int64_t)tr * KCAP;
        for (int i = threadIdx.x; i < n; i += NT) {
            ti[i] = __ldcg(gi + i);
            tv[i] = __ldcg(gv + i);
        }
        if (residual && d.kind == 0 && d.st.mode == MODE_LIST) {
            dl.n = d.st.n_kept;
            const int32_t* hi = p.kept_id + (int64_t)d.r * KCAP;
            const float* hv = p.kept_l + (int64_t)d.r * KCAP;
            for (int i = threadIdx.x; i < dl.n; i += NT) {
                di[i] = __ldcg(hi + i);
                dv[i] = __ldcg(hv + i);
            }
        }
        csync();
    }
    const float invSt = 1.f / (float)ts.S;
    const float invSd = (residual && d.kind == 0) ? 1.f / (float)d.st.S : 0.f;
    const int ept = (n + NT - 1) / NT;
    const int i0 = threadIdx.x * ept;
    *zero = false;
    for (int attempt = 0; attempt < 2; ++attempt) {
        const bool res = residual && attempt == 0;
        unsigned long long part = 0;
        for (int q = 0; q < ept; ++q) {
            const int i = i0 + q;
            if (i >= n) break;
            part += list_r_fix<T>(p, ts, tl, i, res, d, dl, invSt, invSd);
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
        csync();
        if (ex <= t && t < ex + part) {
            unsigned long long acc = ex;
            for (int q = 0; q < ept; ++q) {
                const int i = i0 + q;
                if (i >= n) break;
                acc += list_r_fix<T>(p, ts, tl, i, res, d, dl, invSt, invSd);
                if (acc > t) {
                    s_tok = tl.ids[i];
                    break;
                }
            }
        }
        csync();
        return s_tok;
    }
    return -1;
}

// ------------------------------------------------------------------------- //
// the decision of one sequence (verify launch)                              //
// ------------------------------------------------------------------------- //
constexpr int DECIDE_ROWS_OFF = 2 * KCAP * 8;  // staged row records after the two lists
constexpr int MAX_DECIDE_ROWS = (SCRATCH_BYTES - DECIDE_ROWS_OFF) / (int)sizeof(RowStat);
static_assert(MAX_DECIDE_ROWS >= 2 * 255 + 1, "row records of K_max = 255 must fit");

// logit at token x of a merged row for one full warp: a kept list is scanned
// in 32-wide stripes with every stripe of ids and values loaded at once
template <typename T>
__device__ __forceinline__ float warp_lookup(const Params& p, int r, const RowStat& st, const T* row,
                                             int x, bool* kept)
{
    const int lane = threadIdx.x & 31;
    if (st.mode != MODE_LIST) {
        const float l = Elem<T>::load_cg(row, x);
        *kept = kept_prefix(st, key_of(l), x);
        return l;
    }
    const int32_t* ids = p.kept_id + (int64_t)r * KCAP;
    const float* ls = p.kept_l + (int64_t)r * KCAP;
    const int n = st.n_kept;
    for (int b0 = 0; b0 < n; b0 += 128) {
        int v[4];
        float w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = b0 + q * 32 + lane;
            v[q] = i < n ? __ldcg(ids + i) : -1;
            w[q] = i < n ? __ldcg(ls + i) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const unsigned m = __ballot_sync(0xffffffffu, v[q] == x);
            if (m) {
                *kept = true;
                return __shfl_sync(0xffffffffu, w[q], __ffs(m) - 1);
            }
        }
    }
    *kept = false;
    return -INFINITY;
}

template <typename T>
__device__ void decide_sequence(const Params& p, int b, unsigned char* scratch)
{
    __shared__ int s_jstar, s_bad, s_nonfinite;
    RowStat* rs = reinterpret_cast<RowStat*>(scratch + DECIDE_ROWS_OFF);  // [target 0..K, draft 0..K-1]
    const int K = p.Kmax, V = p.V;
    const int kb = seq_k(p, b);
    const T* target = (const T*)p.target;
    const int64_t trow0 = (int64_t)b * (K + 1) * V;
    const int64_t drow0 = (int64_t)b * K * V;
    const int nrows = seq_rows(p, kb);
    if (threadIdx.x == 0) {
        s_jstar = kb;
        s_bad = 0;
        s_nonfinite = 0;
    }
    csync();
    // one parallel round of loads: row records, drafted tokens (and q(x))
    for (int i = threadIdx.x; i < nrows; i += NT) {
        const int r = i <= kb ? target_slot(p, b, i) : draft_slot(p, b, i - kb - 1);
        rs[i] = load_rowstat(p.rstat + r);
        if (rs[i].flags & FLAG_NONFINITE) s_nonfinite = 1;
    }
    for (int j = threadIdx.x; j < kb; j += NT) {
        const int x = p.xin[(int64_t)b * K + j];
        if (x < 0 || x >= V) {
            s_bad = 1;
        } else if (p.draft_kind == 1 && !p.greedy) {
            const float q = __ldcg((const float*)p.draft + drow0 + (int64_t)j * V + x);
            if (!(q >= 0.f) || q == INFINITY) s_nonfinite = 1;
        }
    }
    csync();
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
    // accept tests of every slot (one warp per slot), first rejection by a min
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < kb; j += NT / 32) {
        const int x = p.xin[(int64_t)b * K + j];
        const RowStat ts = rs[j];
        bool kt, kd = true;
        const float lt = warp_lookup<T>(p, target_slot(p, b, j), ts, target + trow0 + (int64_t)j * V, x, &kt);
        float pd = NAN;  // greedy: the draft is not read
        if (p.greedy) {
        } else if (p.draft_kind == 1) {
            pd = __ldcg((const float*)p.draft + drow0 + (int64_t)j * V + x);
        } else {
            const RowStat ds = rs[kb + 1 + j];
            const float ld = warp_lookup<T>(p, draft_slot(p, b, j), ds,
                                            (const T*)p.draft + drow0 + (int64_t)j * V, x, &kd);
            pd = kd ? (float)((double)exp2f((ld - ds.M) * p.c) / ds.S) : 0.f;
        }
        const float pt = kt ? (float)((double)exp2f((lt - ts.M) * p.c) / ts.S) : 0.f;
        if (lane == 0) {
            bool rej;
            if (p.greedy) {
                rej = !(pt > 0.f);  // the kept set is the target's argmax alone
            } else {
                const uint4 w = slot_words(p, b, j, 0u);
                const double ratio = (double)pt / (double)pd;  // IEEE: pd = 0 gives inf or NaN
                rej = !((double)u24(w.x) < ratio);
            }
            if (rej) atomicMin(&s_jstar, j);
            if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = pt;
            if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = pd;
        }
    }
    for (int j = threadIdx.x; j <= K; j += NT) {
        if (p.lse) p.lse[(int64_t)b * (K + 1) + j] =
            j <= kb && !p.greedy ? (float)((double)rs[j].M / (double)p.T + log(rs[j].S)) : NAN;
        if (j >= kb && j < K) {
            if (p.p_t_at) p.p_t_at[(int64_t)b * K + j] = NAN;
            if (p.p_d_at) p.p_d_at[(int64_t)b * K + j] = NAN;
        }
    }
    csync();
    const int jstar = s_jstar;
    for (int j = threadIdx.x; j <= K; j += NT)
        p.tokens[(int64_t)b * (K + 1) + j] = (j < jstar) ? p.xin[(int64_t)b * K + j] : -1;
    // greedy: the emitted token is the argmax of target row j* (its kept list)
    const bool residual = jstar < kb && !p.greedy;
    const uint4 w = slot_words(p, b, jstar, 0u);
    const float u = u24(w.y);
    const int tr = target_slot(p, b, jstar);
    const RowStat ts = rs[jstar];
    if (threadIdx.x == 0) {
        p.num_accepted[b] = jstar;
        if (p.row_status) p.row_status[b] = ROW_OK;
        if (p.resid_mass && !residual) p.resid_mass[b] = 0.f;
    }
    DraftRef d;
    d.kind = p.draft_kind;
    d.r = residual ? draft_slot(p, b, jstar) : -1;
    if (residual && d.kind == 0) d.st = rs[kb + 1 + jstar];
    d.row = residual ? (const void*)((const char*)p.draft +
                                     (drow0 + (int64_t)jstar * V) * (d.kind == 1 ? 4 : (int64_t)sizeof(T)))
                     : nullptr;
    csync();  // the row records are read; sample_list reuses the front of the scratch
    if (ts.mode == MODE_LIST) {
        unsigned long long Z;
        bool zero;
        const int tok = sample_list<T>(p, tr, ts, residual, d, u, scratch, &Z, &zero);
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
__device__ void sample_own_row(const Params& p, int r, const RowRef& rr, unsigned char* scratch)
{
    const RowStat st = load_rowstat(p.rstat + r);
    const int out = rr.b * p.Kmax + rr.j;
    if (st.flags & FLAG_NONFINITE) {
        if (threadIdx.x == 0) {
            p.tokens[out] = -1;
            p.jobs[out].kind = JOB_NONE;
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
        const int tok = sample_list<T>(p, r, st, false, d, u, scratch, &Z, &zero);
        if (threadIdx.x == 0) {
            p.tokens[out] = tok;
            p.jobs[out].kind = JOB_NONE;
        }
    } else if (threadIdx.x == 0) {
        Job jb;
        jb.kind = JOB_ROW;
        jb.trow = r;
        jb.drow = -1;
        jb.out_idx = out;
        jb.b = rr.b;
        jb.u = u;
        p.jobs[out] = jb;
    }
}

// outputs of a row slot that is not read: a sequence with K_b outside
// [0, K_max] (reported by its first slot), or a draft slot beyond K_b
__device__ void report_skipped_row(const Params& p, const RowRef& rr)
{
    const int K = p.Kmax;
    if (!k_ok(p, rr.kb)) {
        const bool first = p.draft_launch ? rr.j == 0 : (!rr.is_draft && rr.j == 0);
        if (!first) return;
        if (p.draft_launch) {
            for (int j = 0; j < K; ++j) {
                p.tokens[(int64_t)rr.b * K + j] = -1;
                p.jobs[rr.b * K + j].kind = JOB_NONE;
            }
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
    } else if (p.draft_launch) {
        p.tokens[(int64_t)rr.b * K + rr.j] = -1;
        p.jobs[rr.b * K + rr.j].kind = JOB_NONE;
    }
}

// Row r, every segment streamed: merge it; then (draft launch) sample it, or
// (verify) take the sequence ticket, and the last row of the sequence decides
// it.  Called by NT threads; only thread 0 fences and takes the ticket.
template <typename T>
__device__ void finish_row(const Params& p, int r, const RowRef& rr, const T* row,
                           unsigned char* scratch)
{
    __shared__ int s_last_seq;
    merge_row<T>(p, row, r, scratch);
    if (p.draft_launch) {
        csync();
        if (threadIdx.x == 0) __threadfence();
        csync();
        sample_own_row<T>(p, r, rr, scratch);
        return;
    }
    csync();
    if (threadIdx.x == 0) {
        __threadfence();
        const int nrows = seq_rows(p, rr.kb);
        s_last_seq = atomicAdd(&p.seq_ticket[rr.b], 1u) == (unsigned)(nrows - 1);
        if (s_last_seq) {
            __threadfence();
            p.seq_ticket[rr.b] = 0u;
        }
    }
    csync();
    if (!s_last_seq) return;
    decide_sequence<T>(p, rr.b, scratch);
}

// ------------------------------------------------------------------------- //
// k_rows: one CTA per (row slot, segment), loads straight into registers     //
// (rows that do not start on a 16-byte boundary)                             //
// ------------------------------------------------------------------------- //
template <typename T, bool VEC, int MODE>
__global__ void __launch_bounds__(NT, 4) k_rows(const Params p)
{
    if (exit_skip(p)) return;
    __shared__ float s_redf[NT / 32 + 1];
    __shared__ double s_redd[NT / 32 + 1];
    using G = SegGeom<T, NT>;
    const int r = blockIdx.x / p.nseg;
    const int seg = blockIdx.x - r * p.nseg;
    const RowRef rr = row_ref(p, r);
    if (!rr.valid) {
        if (seg == 0 && threadIdx.x == 0) report_skipped_row(p, rr);
        return;
    }
    if (rr.is_draft && !drafts_streamed(p)) return;  // probabilities (or greedy): read only where needed

    const T* row = (const T*)(rr.is_draft ? p.draft : p.target) + row_elem_offset(p, rr);
    const int64_t base = (int64_t)seg * G::SEG;
    uint4 v[G::ROUNDS];
#pragma unroll
    for (int i = 0; i < G::ROUNDS; ++i) {
        const int64_t e0 = base + ((int64_t)i * NT + threadIdx.x) * G::VW;
        if (VEC)
            v[i] = (e0 < p.V) ? ld_stream16(row + e0) : Vec16<T>::neg_inf();
        else
            v[i] = (e0 < p.V) ? Vec16<T>::load_scalar(row, e0, p.V) : Vec16<T>::neg_inf();
    }
    segment_compute<T, MODE, NT>(p, [&](int i) { return v[i]; }, seg, r, (int)threadIdx.x,
                                 [] { csync(); }, s_redf, s_redd);
}

// ------------------------------------------------------------------------- //
// k_stream: persistent streaming kernel for rows that start on a 16-byte      //
// boundary.  One producer thread issues bulk (TMA) copies of its work items   //
// (row slot, segment), item = blockIdx.x + i * gridDim.x, into an NSTAGE ring //
// of SEG_BYTES completing on mbarriers; NS stream threads compute each        //
// segment's chunk-max keys or (max, sum) from shared memory.                 //
// ------------------------------------------------------------------------- //
struct Ring {
    uint64_t full[NSTAGE];
    uint64_t empty[NSTAGE];
    int item[NSTAGE];
};
constexpr int STREAM_SMEM = NSTAGE * SEG_BYTES;

// paired fp32 arithmetic (two lanes of a 64-bit register per instruction)
__device__ __forceinline__ unsigned long long f2_pack(float a, float b)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float f2_sum(unsigned long long r)
{
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
    return a + b;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// SEG_HIST for a segment whose window [val(lo16), M] holds positive values
// only: per token, exp2((l - M) c) is summed when l is below the window
// (exp2 of -inf adds 0 for the others) and its count is added to bin
// m16 - key = (m16 - 0x8000) - bits when it is inside (a positive bf16's key
// is its bits + 0x8000); -inf padding is below the window and adds 0.
template <bool FULLSEG>
__device__ __forceinline__ float warp_hist_pos(const uint4* sv4, int nvalid, int lane, float c, float Mc,
                                               uint32_t m16, uint32_t lo16, uint32_t* hist)
{
    constexpr int SEGE = SEG_BYTES / 2;
    constexpr int WPL = SEGE / 8 / 32;
    const uint32_t thr = __float_as_uint(val_key16(lo16)) >> 16;  // the window's lowest bf16
    const uint32_t thr2 = thr | (thr << 16);
    const unsigned long long c2 = f2_pack(c, c), nmc2 = f2_pack(-Mc, -Mc);
    const uint32_t hb = smem_u32(hist) + 4u * (m16 - 0x8000u);  // hb - 4 h: the bin of bits h
    // a token outside the window counts into the lane's own slot past the
    // bins (never read): every lane issues every count, no branch
    const uint32_t hdummy = smem_u32(hist) + 4u * (HIST_BINS + lane);
    unsigned long long s2[2] = {0ull, 0ull};  // four running sums, in two pairs
    // Per 32-bit word (two tokens): one packed bf16 compare gives both
    // window predicates, one paired FMA both exponents (l c - M c), -inf
    // where the token is counted instead, two ex2, one paired add, and the
    // two shared-memory counts.  (No memory clobber: the stage is
    // only read here, and the warp's __syncwarp orders the counts before the
    // histogram is read out.)
#pragma unroll 4
    for (int i = 0; i < WPL; ++i) {
        const int q = i * 32 + lane;
        const uint4 w = (FULLSEG || q * 8 < nvalid) ? sv4[q] : Vec16<__nv_bfloat16>::neg_inf();
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            asm volatile(
                "{\n\t"
                ".reg .pred plo, phi;\n\t"
                ".reg .b32 blo, bhi, t;\n\t"
                ".reg .f32 flo, fhi;\n\t"
                ".reg .b64 a2;\n\t"
                "setp.ge.bf16x2 plo|phi, %1, %2;\n\t"
                "shl.b32 blo, %1, 16;\n\t"
                "and.b32 bhi, %1, 0xFFFF0000;\n\t"
                "mov.b64 a2, {blo, bhi};\n\t"
                "fma.rn.f32x2 a2, a2, %3, %4;\n\t"
                "mov.b64 {flo, fhi}, a2;\n\t"
                "@plo mov.f32 flo, 0fFF800000;\n\t"
                "@phi mov.f32 fhi, 0fFF800000;\n\t"
                "ex2.approx.ftz.f32 flo, flo;\n\t"
                "ex2.approx.ftz.f32 fhi, fhi;\n\t"
                "mov.b64 a2, {flo, fhi};\n\t"
                "add.rn.f32x2 %0, %0, a2;\n\t"
                "and.b32 t, %1, 0xFFFF;\n\t"
                "mad.lo.s32 t, t, -4, %5;\n\t"
                "selp.b32 t, t, %6, plo;\n\t"
                "red.shared.add.u32 [t], 1;\n\t"
                "shr.u32 t, %1, 16;\n\t"
                "mad.lo.s32 t, t, -4, %5;\n\t"
                "selp.b32 t, t, %6, phi;\n\t"
                "red.shared.add.u32 [t], 1;\n\t"
                "}"
                : "+l"(s2[h >> 1])
                : "r"(ws[h]), "r"(thr2), "l"(c2), "l"(nmc2), "r"(hb), "r"(hdummy));
        }
    }
    return f2_sum(s2[0]) + f2_sum(s2[1]);
}

// One warp reduces a whole segment (SEG_SUM, SEG_HIST): no barrier with the
// other warps, so each of the CTA's stream warps keeps its own segment in
// flight.  Two reads of the segment in shared memory: its max M, then the sum
// of exp2((l - M) c) (SEG_HIST: over the tokens more than HIST_BINS keys below
// M, and a count per key for the others, in the warp's own histogram).
template <typename T, int MODE>
__device__ __forceinline__ void warp_segment(const Params& p, const uint4* sv4, int seg, int r, uint32_t* hist)
{
    constexpr int VW = Vec16<T>::N;
    constexpr int SEGE = SEG_BYTES / (int)sizeof(T);
    constexpr int WPL = SEGE / VW / 32;  // 16-byte words per lane
    const int lane = threadIdx.x & 31;
    const int64_t base = (int64_t)seg * SEGE;
    const int nvalid = (int)min((int64_t)SEGE, (int64_t)p.V - base);  // tokens of the segment
    auto word = [&](int i) {
        const int q = i * 32 + lane;
        return q * VW < nvalid ? sv4[q] : Vec16<T>::neg_inf();
    };
    float m = -INFINITY;
    if constexpr (sizeof(T) == 2) {
        uint32_t m2 = 0xFF80FF80u;  // -inf twice
#pragma unroll 8
        for (int i = 0; i < WPL; ++i) m2 = Vec16<T>::vmax2(word(i), m2);
        m = Vec16<T>::unpack_max(m2);
    } else {
#pragma unroll 8
        for (int i = 0; i < WPL; ++i) m = fmax_nan(m, Vec16<T>::vmax(word(i)));
    }
    const float M = warp_reduce_f(m, fmax_nan);
    float s = 0.f;
    if (M > -INFINITY && M < INFINITY) {
        const float c = p.c, Mc = M * p.c;
        if constexpr (MODE == SEG_HIST) {
            const uint32_t m16 = key16_bf16(__float_as_uint(M) >> 16);
            const uint32_t lo16 = m16 >= 0x7Fu + (HIST_BINS - 1) ? m16 - (HIST_BINS - 1) : 0x7Fu;
            if (lo16 > 0x8000u) {
                // the window holds positive values only: a token's bin is
                // (m16 - 0x8000) - its bf16 bits
                if (nvalid == SEGE) s = warp_hist_pos<true>(sv4, nvalid, lane, c, Mc, m16, lo16, hist);
                else s = warp_hist_pos<false>(sv4, nvalid, lane, c, Mc, m16, lo16, hist);
            } else {
                const uint32_t thr = __float_as_uint(val_key16(lo16)) >> 16;
                const uint32_t thr2 = thr | (thr << 16);
                float sh[4] = {0.f, 0.f, 0.f, 0.f};  // four running sums: shorter rounding chains
#pragma unroll 4
                for (int i = 0; i < WPL; ++i) {
                    const uint4 w = word(i);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const uint32_t x = ws[h];
                        const uint32_t in = ChunkMax<__nv_bfloat16>::ge2(x, thr2);  // 0xFFFF per counted half
                        const float elo = ex2_fast(fmaf(bf16_lo(x), c, -Mc));
                        const float ehi = ex2_fast(fmaf(bf16_hi(x), c, -Mc));
                        sh[h] += ((in & 0xFFFFu) ? 0.f : elo) + ((in >> 16) ? 0.f : ehi);
                        if (in & 0xFFFFu) atomicAdd(&hist[m16 - key16_bf16(x & 0xFFFFu)], 1u);
                        if (in >> 16) atomicAdd(&hist[m16 - key16_bf16(x >> 16)], 1u);
                    }
                }
                s = (sh[0] + sh[1]) + (sh[2] + sh[3]);
            }
        } else {
            float sh[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int i = 0; i < WPL; ++i) sh[i & 3] += Vec16<T>::vsumexp(word(i), M, c);
            s = (sh[0] + sh[1]) + (sh[2] + sh[3]);
        }
    }
    s = warp_reduce_f(s, [](float a, float b) { return a + b; });
    if constexpr (MODE == SEG_HIST) {
        __syncwarp();
        // the counts out, four u8 bins per word (saturating), and cleared
        uint32_t* out = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(p.chunk) +
                                                    (int64_t)r * p.chunk_stride * 2 + (int64_t)seg * HIST_BINS);
#pragma unroll
        for (int q = lane; q < HIST_BINS / 4; q += 32) {
            uint32_t wd = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                wd |= min(hist[4 * q + j], 255u) << (8 * j);
                hist[4 * q + j] = 0u;
            }
            out[q] = wd;
        }
        __syncwarp();
    }
    if (lane == 0) {
        SegStat st;
        st.m = M;
        st.pad = 0.f;
        st.s = (double)s;
        p.seg[(int64_t)r * p.nseg + seg] = st;
    }
}

template <typename T, int MODE>
__global__ void __launch_bounds__(STREAM_THREADS, 3) k_stream(const Params p)
{
    if (exit_skip(p)) return;
    extern __shared__ __align__(128) unsigned char smem_ring[];  // NSTAGE x SEG_BYTES
    __shared__ Ring ring;
    __shared__ float s_redf[NS / 32 + 1];
    __shared__ double s_redd[NS / 32 + 1];
    // SEG_SUM and SEG_HIST: each stream warp reduces whole segments on its own
    // (stage k belongs to warp k mod NSTAGE); SEG_CHUNK: the four warps share
    // every segment
    constexpr bool PERWARP = MODE != SEG_CHUNK;
    constexpr int NSENT = PERWARP ? NS / 32 : 1;  // end-of-work sentinels
    static_assert(!PERWARP || NSTAGE == NS / 32, "one stage per stream warp");
    constexpr int HSTRIDE = HIST_BINS + 32;  // a warp's bins, then one spare count per lane
    __shared__ uint32_t s_hist[MODE == SEG_HIST ? (NS / 32) * HSTRIDE : 1];
    using G = SegGeom<T, NS>;
    const int tid = threadIdx.x;
    if (MODE == SEG_HIST)
        for (int i = tid; i < (NS / 32) * HSTRIDE; i += STREAM_THREADS) s_hist[i] = 0u;
    // the merge kernel that follows may be scheduled as this grid drains; it
    // waits for this grid's completion before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&ring.full[s], 1);
            // SEG_CHUNK: each of the four warps releases the stage on its own
            mbar_init(&ring.empty[s], PERWARP ? 1 : NS / 32);
        }
        fence_barrier_init();
    }
    __syncthreads();  // the only barrier over all STREAM_THREADS threads
    const int64_t total_items = (int64_t)p.B * p.rps * p.nseg;
    const int64_t row_bytes = (int64_t)p.V * (int64_t)sizeof(T);

    if (tid >= NS) {
        // ---------------- producer
        if (tid != NS) return;
        if (p.stall) return;  // fault injection: no copy, so every consumer wait runs out
        const uint64_t pol = l2_evict_first();  // the rows are read once; the chunk keys stay in L2
        int k = 0;
        bool failed = false;
        for (int64_t item = blockIdx.x;; item += gridDim.x) {
            if (item >= total_items) {
                item = -1;
            } else {
                const RowRef rr = row_ref(p, (int)(item / p.nseg));
                if (!rr.valid) continue;
                if (rr.is_draft && !drafts_streamed(p)) continue;
            }
            const int s = k % NSTAGE;
            if (k >= NSTAGE && !mbar_wait_sleep(&ring.empty[s], ((k / NSTAGE) - 1) & 1, 0)) {
                atomicOr(p.err, 1u);
                failed = true;
                break;
            }
            ring.item[s] = (int)item;
            if (item < 0) {
                // the end-of-work sentinel, one per consumer (the next NSENT stages)
                mbar_arrive(&ring.full[s]);
                for (int g = 1; g < NSENT; ++g) {
                    ++k;
                    const int s2 = k % NSTAGE;
                    if (k >= NSTAGE && !mbar_wait_sleep(&ring.empty[s2], ((k / NSTAGE) - 1) & 1, 0)) {
                        atomicOr(p.err, 1u);
                        break;
                    }
                    ring.item[s2] = -1;
                    mbar_arrive(&ring.full[s2]);
                }
                break;
            }
            const int r = (int)(item / p.nseg), seg = (int)(item - (int64_t)r * p.nseg);
            const RowRef rr = row_ref(p, r);
            const char* src = (const char*)(rr.is_draft ? p.draft : p.target) +
                              row_elem_offset(p, rr) * (int64_t)sizeof(T) + (int64_t)seg * SEG_BYTES;
            const uint32_t bytes =
                (uint32_t)min((int64_t)SEG_BYTES, row_bytes - (int64_t)seg * SEG_BYTES);
            mbar_arrive_expect_tx(&ring.full[s], bytes);
            tma_load_1d_once(smem_ring + (size_t)s * SEG_BYTES, src, bytes, &ring.full[s], pol);
            ++k;
        }
        if (failed) {
            // wait (bounded) for the copies still in flight before leaving
            for (int q = (k > NSTAGE ? k - NSTAGE : 0); q < k; ++q)
                mbar_wait(&ring.full[q % NSTAGE], (q / NSTAGE) & 1);
        }
        return;
    }

    if constexpr (PERWARP) {
        // ---------------- stream warps, one segment each at a time
        const unsigned FULL = 0xffffffffu;
        const int w = tid >> 5;
        for (int k = w;; k += NS / 32) {
            const int s = k % NSTAGE;
            if (!__all_sync(FULL, mbar_wait_sleep(&ring.full[s], (k / NSTAGE) & 1, p.wait_limit))) {
                if ((tid & 31) == 0) atomicOr(p.err, 2u);
                break;
            }
            const int item = ring.item[s];
            if (item < 0) break;
            const int r = item / p.nseg, seg = item - r * p.nseg;
            warp_segment<T, MODE>(p, reinterpret_cast<const uint4*>(smem_ring + (size_t)s * SEG_BYTES), seg, r,
                                  s_hist + (MODE == SEG_HIST ? w * HSTRIDE : 0));
            __syncwarp();  // every lane is done with the stage
            if ((tid & 31) == 0) mbar_arrive(&ring.empty[s]);
        }
    } else {
        // ---------------- stream threads (SEG_CHUNK): the four warps share each
        // segment but need no barrier among them: a chunk's key is one lane group's
        // own, and every warp waits for, and releases, the stage by itself (so a
        // wait that runs out ends one warp without stranding the others)
        static_assert(PERWARP || MODE == SEG_CHUNK, "the shared-segment loop has no barriers");
        for (int k = 0;; ++k) {
            const int s = k % NSTAGE;
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(&ring.full[s], (k / NSTAGE) & 1, p.wait_limit))) {
                if ((tid & 31) == 0) atomicOr(p.err, 2u);
                break;
            }
            const int item = ring.item[s];
            if (item < 0) break;
            const int r = item / p.nseg, seg = item - r * p.nseg;
            const uint4* sv4 = reinterpret_cast<const uint4*>(smem_ring + (size_t)s * SEG_BYTES);
            const int64_t base = (int64_t)seg * G::SEG;
            segment_compute<T, MODE, NS>(
                p,
                [&](int i) {
                    const int64_t e0 = base + ((int64_t)i * NS + tid) * G::VW;
                    return e0 < p.V ? sv4[i * NS + tid] : Vec16<T>::neg_inf();
                },
                seg, r, tid, [] {}, s_redf, s_redd, s_hist);
            __syncwarp();  // the warp is done with the stage
            if ((tid & 31) == 0) mbar_arrive(&ring.empty[s]);
        }
    }
}

// ------------------------------------------------------------------------- //
// k_merge: one CTA per row slot, after the whole stream: merge the row, then  //
// the sequence ticket and the decision (verify) or the draft-row sample.     //
// ------------------------------------------------------------------------- //
template <typename T>
__global__ void __launch_bounds__(NT, 4) k_merge(const Params p)
{
    extern __shared__ __align__(16) unsigned char smem_scratch[];  // SCRATCH_BYTES
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream grid has completed
    if (exit_skip(p)) return;
    const int r = blockIdx.x;
    const RowRef rr = row_ref(p, r);
    if (!rr.valid) {
        if (threadIdx.x == 0) report_skipped_row(p, rr);
        return;
    }
    if (rr.is_draft && !drafts_streamed(p)) return;  // probabilities (or greedy): read only where needed
    const T* row = (const T*)(rr.is_draft ? p.draft : p.target) + row_elem_offset(p, rr);
    finish_row<T>(p, r, rr, row, smem_scratch);
}

}  // namespace sv

#include "sv_warp.cuh"
#include "sv_mcand.cuh"
#include "sv_exit.cuh"

namespace sv {

// ------------------------------------------------------------------------- //
// launchers                                                                 //
// ------------------------------------------------------------------------- //
template <typename T, bool VEC, int MODE>
static cudaError_t launch_rows_t(const Params& p, cudaStream_t s)
{
    const int64_t grid = (int64_t)p.B * p.rps * p.nseg;
    if (grid <= 0) return cudaSuccess;
    k_rows<T, VEC, MODE><<<(unsigned)grid, NT, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename T, int MODE>
static cudaError_t launch_stream_t(const Params& p, int ctas, cudaStream_t s)
{
    static DeviceOnce once;  // the shared-memory opt-in, per device
    const cudaError_t e = cuda_once(once, nullptr, [](int, int*) {
        return cudaFuncSetAttribute(k_stream<T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, STREAM_SMEM);
    });
    if (e != cudaSuccess) return e;
    k_stream<T, MODE><<<ctas, STREAM_THREADS, STREAM_SMEM, s>>>(p);
    return cudaGetLastError();
}

// a grid launched as a programmatic dependent of the previous one on the stream
template <typename K>
static cudaError_t launch_dependent(K kernel, const Params& p, unsigned grid, unsigned block,
                                    int smem, cudaStream_t s)
{
    if (grid == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_merge_t(const Params& p, cudaStream_t s)
{
    const int64_t rows = (int64_t)p.B * p.rps;
    return launch_dependent(k_merge<T>, p, (unsigned)rows, NT, SCRATCH_BYTES, s);
}

template <typename T>
static cudaError_t launch_merge_warp_t(const Params& p, cudaStream_t s)
{
    const int64_t rows = (int64_t)p.B * p.rps;
    static DeviceOnce once;  // the shared-memory opt-in, per device
    const cudaError_t e0 = cuda_once(once, nullptr, [](int, int*) {
        return cudaFuncSetAttribute(k_merge_warp<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, WM_SMEM);
    });
    if (e0 != cudaSuccess) return e0;
    cudaError_t e = launch_dependent(k_merge_warp<T>, p, (unsigned)((rows + WM_WARPS - 1) / WM_WARPS),
                                     WM_WARPS * 32, WM_WARPS * wm_stride(p.seg_mode), s);
    if (e != cudaSuccess) return e;
    return launch_dependent(k_decide<T>, p, (unsigned)p.B, NT, SCRATCH_BYTES, s);
}

template <typename T>
static cudaError_t launch_merge_topk_t(const Params& p, cudaStream_t s)
{
    cudaError_t e = launch_dependent(k_merge_cand<T>, p, (unsigned)(p.B * p.rps), MC_T, 0, s);
    if (e != cudaSuccess) return e;
    return launch_dependent(k_decide<T>, p, (unsigned)p.B, NT, SCRATCH_BYTES, s);
}

cudaError_t launch_merge_topk(const Params& p, int dtype, cudaStream_t s)
{
    return dtype == 1 ? launch_merge_topk_t<__nv_bfloat16>(p, s) : launch_merge_topk_t<float>(p, s);
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

cudaError_t launch_rows_stream(const Params& p, int dtype, int ctas, cudaStream_t s)
{
    if ((int64_t)p.B * p.rps * p.nseg <= 0) return cudaSuccess;
    if (p.seg_mode == SEG_HIST)
        return dtype == 1 ? launch_stream_t<__nv_bfloat16, SEG_HIST>(p, ctas, s) : cudaErrorInvalidValue;
    const bool chunk = p.seg_mode == SEG_CHUNK;
    if (dtype == 1)
        return chunk ? launch_stream_t<__nv_bfloat16, SEG_CHUNK>(p, ctas, s)
                     : launch_stream_t<__nv_bfloat16, SEG_SUM>(p, ctas, s);
    return chunk ? launch_stream_t<float, SEG_CHUNK>(p, ctas, s)
                 : launch_stream_t<float, SEG_SUM>(p, ctas, s);
}

cudaError_t launch_merge(const Params& p, int dtype, cudaStream_t s)
{
    return dtype == 1 ? launch_merge_t<__nv_bfloat16>(p, s) : launch_merge_t<float>(p, s);
}

cudaError_t launch_merge_warp(const Params& p, int dtype, cudaStream_t s)
{
    return dtype == 1 ? launch_merge_warp_t<__nv_bfloat16>(p, s) : launch_merge_warp_t<float>(p, s);
}

}  // namespace sv
