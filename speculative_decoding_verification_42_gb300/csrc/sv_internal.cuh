// sv_internal.cuh -- device-side building blocks of the verify step (sm_103a).
//
// Layout of one launch.  A "row" is one V-length logit row: for sequence b the
// verify launch has rows_per_seq = 2*K_max + 1 row slots, slot j <= K_max being
// target position j and slot K_max + 1 + j being draft position j.  The
// draft-sampler launch has rows_per_seq = K_max (draft rows only).  Row slots
// beyond a sequence's K_b are skipped.
//
// Stage 1 (k_rows): one CTA per (row, segment) streams SEG_BYTES of the row
// from HBM once.  The last segment CTA of a row (an atomic ticket, no waiting)
// merges the row: its max, its softmax normaliser over the kept set, and the
// kept set itself (explicit list, or a rank-prefix threshold).  The last row of
// a sequence (a second ticket) makes the accept decisions and either samples
// the emitted token directly (target kept set given as a list) or posts a
// sampling job.  Stage 2 (k_sample): segment-parallel inverse-CDF sampling of
// the posted jobs over full rows.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "sv_once.h"

namespace sv {

// the current device's one-time launch set-up (sv_once.h)
template <typename F>
inline cudaError_t cuda_once(DeviceOnce& o, int* value, F setup)
{
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return device_once(o, dev, cudaSuccess, cudaErrorInvalidDevice, value, setup);
}

constexpr int NT = 256;             // threads of every CTA
constexpr int SEG_BYTES = 16384;    // bytes of one stage-1 segment
constexpr int CHUNK_BYTES = 128;    // bytes of data behind one chunk-max key
constexpr int KCAP = 1024;          // largest kept set stored as an explicit list
constexpr int CAND_CAP = 1024;      // candidates of the fast top-k gather
constexpr int MAX_CHUNKS = 8192;    // chunk keys a row merge can hold in smem
constexpr int DIGIT_BITS = 11;      // radix digit of the general selection
constexpr int NBINS = 1 << DIGIT_BITS;
constexpr int SAMPLE_SEG = 4096;    // elements of one stage-2 segment
constexpr int SAMPLE_EPT = SAMPLE_SEG / NT;
constexpr int SAMPLE_PARTS = 4;      // per segment: partial masses of its rounds of 16-byte words
constexpr int WALK_EPT = 16;        // contiguous elements per thread in ordered walks
constexpr int SCRATCH_BYTES = 40960;  // shared scratch of a row merge / sequence decision
constexpr int NSTAGE = 4;           // ring stages of the streaming kernel
constexpr int NS = 128;             // stream threads of the streaming kernel
// streaming kernel layout: stream warps [0, NS), one producer warp [NS, NS + 32)
constexpr int STREAM_THREADS = NS + 32;
constexpr int STREAM_CTAS_PER_SM = 3;

// SEG_SUM: per-segment (max, sum exp); SEG_CHUNK: 16-bit chunk-max keys;
// SEG_HIST (bf16 rows with top-p alone): per-segment max, a count of tokens at
// each of the HIST_BINS order keys from the max down, and the sum of exp over
// the tokens below them
enum SegMode : int32_t { SEG_SUM = 0, SEG_CHUNK = 1, SEG_HIST = 2 };
constexpr int HIST_BINS = 256;      // bf16 keys counted below a segment's max (two binades)
enum RowMode : int32_t { MODE_ALL = 0, MODE_LIST = 1, MODE_PREFIX = 2 };
enum : int32_t { FLAG_NONFINITE = 1, FLAG_BLOCK_MERGE = 2 };  // 2: the warp merge gave up
enum : int32_t { JOB_NONE = 0, JOB_RESIDUAL = 1, JOB_ROW = 2 };

// status codes (same values as the public ABI)
enum : int32_t { ROW_OK = 0, ROW_BAD_TOKEN = 1, ROW_BAD_K = 2, ROW_NONFINITE = 3,
                 ROW_ZERO_RESIDUAL = 4 };

struct SegStat {
    float m;      // segment max (NaN-propagating)
    float pad;
    double s;     // sum of exp2((l - m) * c) over the segment
};

struct __align__(16) RowStat {
    float M;          // max logit of the kept set (rank 0 is always kept)
    uint32_t kappa;   // MODE_PREFIX: order key of the last kept rank
    double S;         // sum over the kept set of exp2((l - M) * c)
    int32_t i_kappa;  // MODE_PREFIX: largest kept token id among ties at kappa
    int32_t n_kept;   // size of the kept set
    int32_t mode;     // RowMode
    int32_t flags;    // FLAG_NONFINITE
    float px;         // warp merges: P(x) of the row at its drafted token x_j
                      // (0 when x_j is not kept or out of range)
    int32_t pad[3];
};

struct __align__(8) Job {
    int32_t kind;     // JOB_NONE / JOB_RESIDUAL / JOB_ROW
    int32_t trow;     // row slot sampled from (the target, or the draft row itself)
    int32_t drow;     // draft row slot of a residual, else -1
    int32_t out_idx;  // element of the token output written by the job
    int32_t b;        // sequence
    float u;          // sampling uniform
};

struct Params {
    // shape of this launch
    int32_t B, Kmax, V;
    int32_t rps;          // row slots per sequence
    int32_t nseg;         // stage-1 segments per row
    int32_t nchunk;       // chunk-max keys per row
    int32_t chunk_stride; // chunk keys per row in the workspace (multiple of 8)
    int32_t draft_launch; // 1: the draft-side sampler (rows are draft rows only)
    int32_t draft_kind;   // 0 logits, 1 probabilities (float)
    int32_t greedy;       // temperature 0: accept while x_j is the target's argmax; no draft row read
    int32_t seg_mode;     // SegMode of this launch
    // knobs
    float T;              // temperature
    float c;              // log2(e) / T (fp32, used by every exponential)
    float c_lo;           // log2(e) / T - c (fp32): c + c_lo carries the ratio to ~2^-48
    int32_t top_k;        // 0: off
    float top_p;          // >= 1: off
    uint64_t top_p_fix;   // top_p in units of 2^-56
    uint64_t seed, round;
    // inputs
    const void* target;       // [B, Kmax+1, V]
    const void* draft;        // [B, Kmax, V]
    const int32_t* xin;       // [B, Kmax] drafted tokens (verify)
    const int32_t* kpr;       // [B] or NULL
    // outputs
    int32_t* tokens;          // verify: [B, Kmax+1]; draft launch: [B, Kmax]
    int32_t* num_accepted;    // [B]
    int32_t* row_status;      // [B] or NULL
    float* p_t_at;            // [B, Kmax] or NULL
    float* p_d_at;            // [B, Kmax] or NULL
    float* resid_mass;        // [B] or NULL
    float* lse;               // [B, Kmax+1] or NULL
    float* alpha;             // [B, Kmax] acceptance statistic per slot, or NULL
    float* probs_out;         // draft launch: dense [B, Kmax, V] or NULL
    // workspace
    SegStat* seg;             // [rows, nseg]
    uint16_t* chunk;          // [rows, nchunk]
    RowStat* rstat;           // [rows]
    int32_t* kept_id;         // [rows, KCAP]
    float* kept_l;            // [rows, KCAP]
    unsigned* row_ticket;     // [rows]
    unsigned* seq_ticket;     // [B]
    Job* jobs;                // [njobs]
    unsigned long long* job_seg;  // [njobs, nseg_sample] fixed-point segment masses
    unsigned long long* job_part; // [njobs, nseg_sample, SAMPLE_PARTS] the segments' round masses
    unsigned* job_ticket;     // [njobs]
    int32_t nseg_sample;      // stage-2 segments per row
    int32_t sample_spc;       // stage-2 segments per CTA (set by the launcher)
    unsigned* err;            // bounded waits that ran out (0 = none)
    int32_t cand;             // 1: top-k rows (1 <= top-k <= CAND_TOPK_MAX) take k_merge_cand
    unsigned* exit_flag;      // early exit: the regular pipeline runs only when it is nonzero (NULL: always)
    unsigned* seq_done;       // [B] sequences decided inside the merge grid
    // fault injection (tests of the timeout report): the stream kernel's
    // producer issues no copy and its consumers' waits give up after
    // wait_limit polls; 0 / 0 in every ordinary run
    int32_t stall;
    uint32_t wait_limit;      // 0: WAIT_LIMIT
};

constexpr int CAND_TOPK_MAX = 128;  // largest top-k the row merge of sv_mcand.cuh serves

// ------------------------------------------------------------------------- //
// order keys: unsigned keys whose order is the order of the float values,    //
// with -0 folded onto +0 so that equal values give equal keys.               //
// ------------------------------------------------------------------------- //
__device__ __forceinline__ uint32_t key_of(float x)
{
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float val_of(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float ex2_fast(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// order key of a bf16 bit pattern (16 bits; -0 folded onto +0), and back
__device__ __forceinline__ uint32_t key16_bf16(uint32_t b)
{
    if (b == 0x8000u) b = 0u;
    return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}
__device__ __forceinline__ float val_key16(uint32_t k)
{
    const uint32_t b = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
    return __uint_as_float(b << 16);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float* p, int64_t i) { return __ldg(p + i); }
    static __device__ __forceinline__ float load_cg(const float* p, int64_t i) { return __ldcg(p + i); }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p, int64_t i)
    {
        return __uint_as_float((uint32_t)__ldg((const unsigned short*)p + i) << 16);
    }
    static __device__ __forceinline__ float load_cg(const __nv_bfloat16* p, int64_t i)
    {
        return __uint_as_float((uint32_t)__ldcg((const unsigned short*)p + i) << 16);
    }
};

__device__ __forceinline__ uint4 ld_stream16(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ------------------------------------------------------------------------- //
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of the 4x32   //
// S-box, the key advancing by the Weyl increments between rounds.            //
// ------------------------------------------------------------------------- //
__device__ __forceinline__ uint4 philox4x32_10(uint4 ctr, uint2 key)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * ctr.x, hi0 = __umulhi(0xD2511F53u, ctr.x);
        const uint32_t lo1 = 0xCD9E8D57u * ctr.z, hi1 = __umulhi(0xCD9E8D57u, ctr.z);
        ctr = make_uint4(hi1 ^ ctr.y ^ key.x, lo1, hi0 ^ ctr.w ^ key.y, lo0);
        key.x += 0x9E3779B9u;
        key.y += 0xBB67AE85u;
    }
    return ctr;
}

// the uniforms of slot j of sequence b: counter ((j << 2) | tag, b, round)
__device__ __forceinline__ uint4 slot_words(const Params& p, int b, int j, uint32_t tag)
{
    const uint4 ctr = make_uint4(((uint32_t)j << 2) | tag, (uint32_t)b, (uint32_t)p.round,
                                 (uint32_t)(p.round >> 32));
    return philox4x32_10(ctr, make_uint2((uint32_t)p.seed, (uint32_t)(p.seed >> 32)));
}

__device__ __forceinline__ float u24(uint32_t w) { return (float)(w >> 8) * 0x1p-24f; }

// Probability masses of the inverse CDF are summed as integers in units of
// 2^-56 (a row's masses sum to at most 1, so no sum overflows), which makes
// every partial sum exact and every scan order give the same CDF.
// r * 2^56 rounded to nearest (ties to even) for r >= 0, from r's bits with
// integer operations only (a float-to-u64 conversion runs on the fp64 pipe,
// which is slow on this part); negatives and NaN give 0, values >= 2^8
// saturate
__device__ __forceinline__ unsigned long long to_fix56(float r)
{
    const uint32_t u = __float_as_uint(r);
    if (u >> 31) return 0ull;                       // negative (or -0, -NaN)
    const int ex = (int)(u >> 23);                  // biased exponent
    if (ex == 0) return 0ull;                       // zero or subnormal: below 2^-70
    if (ex == 255) return (u & 0x7FFFFFu) ? 0ull : ~0ull;  // NaN, +inf
    const unsigned long long m = (u & 0x7FFFFFu) | 0x800000u;  // r = m 2^(ex - 150)
    const int sh = ex - 94;                         // r 2^56 = m 2^sh
    if (sh >= 0) return sh > 39 ? ~0ull : m << sh;
    if (sh < -24) return 0ull;                      // below 1/2
    const int d = -sh;
    const unsigned long long q = m >> d, rem = m & ((1ull << d) - 1ull), half = 1ull << (d - 1);
    return q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
}
__device__ __forceinline__ double from_fix56(unsigned long long z) { return (double)z * 0x1p-56; }

// floor(u * Z) for the 24-bit uniform u = m 2^-24, exactly
__device__ __forceinline__ unsigned long long cdf_target(float u, unsigned long long Z)
{
    const unsigned long long m = (unsigned long long)(u * 16777216.0f);
    const unsigned long long lo = m * Z, hi = __umul64hi(m, Z);
    return (hi << 40) | (lo >> 24);
}

// ------------------------------------------------------------------------- //
// block-wide helpers over the NT "compute" threads 0..NT-1.  They synchronise  //
// with named barrier 1 of NT threads, so a CTA may carry extra threads (the    //
// producer warp of the streaming kernel) that never join these barriers.       //
// ------------------------------------------------------------------------- //
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }

// barrier of the stream warps of the streaming kernel (named barrier 2)
__device__ __forceinline__ void ssync() { asm volatile("bar.sync 2, %0;" ::"n"(NS) : "memory"); }

// reductions over a thread group of NTH threads (local index lt) whose
// barrier is SYNC(); red holds NTH/32 values
template <int NTH, typename SYNC>
__device__ __forceinline__ float group_max_nan(float v, float* red, int lt, SYNC sync);
template <int NTH, typename SYNC>
__device__ __forceinline__ double group_sum_d(double v, double* red, int lt, SYNC sync);

// block-wide OR over the compute threads; flag: a shared int
__device__ __forceinline__ bool csync_or(bool v, int* flag)
{
    if (threadIdx.x == 0) *flag = 0;
    csync();
    if (v) *flag = 1;
    csync();
    return *flag != 0;
}
template <typename F>
__device__ __forceinline__ float warp_reduce_f(float v, F op)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ double warp_sum_d(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int NTH, typename SYNC>
__device__ __forceinline__ float group_max_nan(float v, float* red, int lt, SYNC sync)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    sync();
    if ((lt & 31) == 0) red[lt >> 5] = v;
    sync();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < NTH / 32; ++i) r = fmax_nan(r, red[i]);
    return r;
}

template <int NTH, typename SYNC>
__device__ __forceinline__ double group_sum_d(double v, double* red, int lt, SYNC sync)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    sync();
    if ((lt & 31) == 0) red[lt >> 5] = v;
    sync();
    double r = 0.0;
#pragma unroll
    for (int i = 0; i < NTH / 32; ++i) r += red[i];
    return r;
}

// all threads get the block max (NaN-propagating); red: >= NT/32 floats
__device__ __forceinline__ float block_max_nan(float v, float* red)
{
    v = warp_reduce_f(v, fmax_nan);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    csync();
    if (l == 0) red[w] = v;
    csync();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < NT / 32; ++i) r = fmax_nan(r, red[i]);
    return r;
}

// all threads get the block sum; red: >= NT/32 doubles
__device__ __forceinline__ double block_sum_d(double v, double* red)
{
    v = warp_sum_d(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    csync();
    if (l == 0) red[w] = v;
    csync();
    double r = 0.0;
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) r += red[i];
    return r;
}

// exclusive and inclusive block scans in thread order; red: >= NT/32 + 1 T
template <typename T>
__device__ __forceinline__ T block_excl_scan(T v, T* red, T* total)
{
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T y = __shfl_up_sync(0xffffffffu, x, o);
        if (l >= o) x += y;
    }
    csync();
    if (l == 31) red[w] = x;
    csync();
    T before = T(0), all = T(0);
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) {
        if (i < w) before += red[i];
        all += red[i];
    }
    if (total) *total = all;
    return before + x - v;
}

// bitonic sort (ascending) of n = power of two keys in shared memory
__device__ __forceinline__ void bitonic_sort_u64(unsigned long long* a, int n)
{
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += NT) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long x = a[i], y = a[ixj];
                    const bool up = ((i & k) == 0);
                    if ((x > y) == up) {
                        a[i] = y;
                        a[ixj] = x;
                    }
                }
            }
            csync();
        }
    }
}

__host__ __device__ __forceinline__ int next_pow2(int n)
{
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

// records written by another CTA of the same launch are read through L2
__device__ __forceinline__ RowStat load_rowstat(const RowStat* src)
{
    static_assert(sizeof(RowStat) == 48, "RowStat is three 16-byte words");
    const uint4 a = __ldcg(reinterpret_cast<const uint4*>(src));
    const uint4 b = __ldcg(reinterpret_cast<const uint4*>(src) + 1);
    const uint4 c = __ldcg(reinterpret_cast<const uint4*>(src) + 2);
    RowStat r;
    uint4* d = reinterpret_cast<uint4*>(&r);
    d[0] = a;
    d[1] = b;
    d[2] = c;
    return r;
}

__device__ __forceinline__ Job load_job(const Job* src)
{
    static_assert(sizeof(Job) == 24, "Job is three 8-byte words");
    const uint2* s = reinterpret_cast<const uint2*>(src);
    Job j;
    uint2* d = reinterpret_cast<uint2*>(&j);
    d[0] = __ldcg(s);
    d[1] = __ldcg(s + 1);
    d[2] = __ldcg(s + 2);
    return j;
}

// row slot helpers
struct RowRef {
    int b, j;          // sequence, position
    bool is_draft;
    bool valid;        // inside K_b (or K_b invalid -> false)
    int kb;            // K_b of the sequence (may be invalid)
};

__device__ __forceinline__ int seq_k(const Params& p, int b)
{
    return p.kpr ? p.kpr[b] : p.Kmax;
}

__device__ __forceinline__ bool k_ok(const Params& p, int kb) { return kb >= 0 && kb <= p.Kmax; }

__device__ __forceinline__ RowRef row_ref(const Params& p, int r)
{
    RowRef rr;
    rr.b = r / p.rps;
    const int slot = r - rr.b * p.rps;
    rr.kb = seq_k(p, rr.b);
    if (p.draft_launch) {
        rr.is_draft = true;
        rr.j = slot;
        rr.valid = k_ok(p, rr.kb) && rr.j < rr.kb;
    } else {
        rr.is_draft = slot > p.Kmax;
        rr.j = rr.is_draft ? slot - (p.Kmax + 1) : slot;
        rr.valid = k_ok(p, rr.kb) && (rr.is_draft ? rr.j < rr.kb : rr.j <= rr.kb);
    }
    return rr;
}

__device__ __forceinline__ int64_t row_elem_offset(const Params& p, const RowRef& rr)
{
    const int64_t V = p.V;
    return rr.is_draft ? ((int64_t)rr.b * p.Kmax + rr.j) * V
                       : ((int64_t)rr.b * (p.Kmax + 1) + rr.j) * V;
}

__device__ __forceinline__ int target_slot(const Params& p, int b, int j) { return b * p.rps + j; }
__device__ __forceinline__ int draft_slot(const Params& p, int b, int j)
{
    return p.draft_launch ? b * p.rps + j : b * p.rps + p.Kmax + 1 + j;
}

// is token x (with logit key k) in the kept set of a row?
__device__ __forceinline__ bool kept_prefix(const RowStat& st, uint32_t k, int x)
{
    return st.mode == MODE_ALL || k > st.kappa || (k == st.kappa && x <= st.i_kappa);
}

// lower_bound of x in a sorted id list
__device__ __forceinline__ int lower_bound_i32(const int32_t* a, int n, int x)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldcg(a + mid) < x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// ------------------------------------------------------------------------- //
// TMA bulk copies and mbarriers (sm_90+ PTX)                                 //
// ------------------------------------------------------------------------- //
__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// make initialised barriers visible to the async (TMA) proxy
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// a bounded wait: false when the barrier did not flip within the limit
constexpr uint32_t WAIT_LIMIT = 1u << 24;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity)
{
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// the same with a limit of `limit` polls (0: WAIT_LIMIT)
__device__ __forceinline__ bool mbar_wait_n(uint64_t* bar, uint32_t parity, uint32_t limit)
{
    const uint32_t n = limit ? limit : WAIT_LIMIT;
    for (uint32_t i = 0; i < n; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// polls that may sleep: the waiting thread is suspended for up to
// MBAR_SLEEP_NS until the phase completes, so a warp that waits (a producer
// for a free stage, a consumer for data) takes no issue slots from the
// warps that compute; at most `limit` polls (0: WAIT_LIMIT / 64)
constexpr uint32_t MBAR_SLEEP_NS = 2000;
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t limit)
{
    const uint32_t n = limit ? limit : WAIT_LIMIT / 64;
    for (uint32_t i = 0; i < n; ++i) {
        uint32_t ok;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "n"(MBAR_SLEEP_NS) : "memory");
        if (ok) return true;
    }
    return false;
}
// one-dimensional bulk copy global -> shared, completing on an mbarrier
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// the same copy with an L2 evict-first policy (from l2_evict_first()): data
// read once does not push out what later kernels read back
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_1d_once(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                 uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol) : "memory");
}

// launchers (defined in the .cu files)
cudaError_t launch_rows(const Params& p, int dtype, bool vec, cudaStream_t s);
cudaError_t launch_rows_stream(const Params& p, int dtype, int ctas, cudaStream_t s);
// top-k rows: the row merge (one CTA per row) and the decision grid for what
// it leaves, both programmatic dependents of the stream
cudaError_t launch_merge_topk(const Params& p, int dtype, cudaStream_t s);
// early-exit verify of the top-k rows (one CTA per sequence at a time)
cudaError_t launch_verify_exit(const Params& p, int dtype, int num_sms, cudaStream_t s);
cudaError_t launch_merge(const Params& p, int dtype, cudaStream_t s);
cudaError_t launch_merge_warp(const Params& p, int dtype, cudaStream_t s);
// rows whose merge the warp kernel handles: fast top-k rows, or rows without knobs
// the regular pipeline after the early-exit kernel: nothing to do unless
// that kernel left a sequence it could not finish (read after the stream's
// previous grids have completed)
__device__ __forceinline__ bool exit_skip(const Params& p)
{
    return p.exit_flag && __ldcg(p.exit_flag) == 0u;
}

// draft rows the verify streams and merges: logits, unless greedy
__host__ __device__ __forceinline__ bool drafts_streamed(const Params& p)
{
    return p.draft_kind == 0 && !p.greedy;
}
// rows of sequence b the merge grids count: K_b + 1 target rows (+ K_b drafts)
__host__ __device__ __forceinline__ int seq_rows(const Params& p, int kb)
{
    return drafts_streamed(p) ? 2 * kb + 1 : kb + 1;
}

__host__ __device__ __forceinline__ bool warp_merge_ok(const Params& p)
{
    return !p.draft_launch && ((p.seg_mode == SEG_CHUNK && p.top_k <= 256 && p.nchunk <= 4096) ||
                               (p.seg_mode == SEG_SUM && p.top_k == 0 && !(p.top_p < 1.0f)) ||
                               (p.seg_mode == SEG_HIST && p.top_k == 0 && p.nseg <= 32));
}
cudaError_t launch_sample(const Params& p, int dtype, int njobs, cudaStream_t s, int* launches = nullptr);
// alpha_j = sum_v min(p_t, p_d) of every slot (when p.alpha is set)
cudaError_t launch_alpha(const Params& p, int dtype, cudaStream_t s);
// the LM head: out[M, N] (row stride ldo) = hidden[M, K] x w[K, N], bf16 in, fp32 out
bool lmhead_shape_ok(const void* hidden, const void* w, int M, int N, int K);
// softmax partials the LM head's epilogue writes (seg NULL: none): per
// logits row m = b kp1 + j and 256-column tile n, (max, sum exp2((l - max)
// c)) at seg[(b rps + j) nseg + n]
constexpr int LM_STAT_COLS = 256;
struct LmStats {
    SegStat* seg;
    int nseg, kp1, rps;
    float c;
};
cudaError_t launch_lmhead(const void* hidden, const void* w, float* out, int M, int N, int K, int64_t ldo,
                          unsigned* err, cudaStream_t s, const LmStats& st = LmStats{nullptr, 0, 1, 1, 0.f});
cudaError_t launch_probs(const Params& p, int dtype, cudaStream_t s);

}  // namespace sv
