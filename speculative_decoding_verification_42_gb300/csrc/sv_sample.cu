// sv_sample.cu -- stage 2 of the verify step: inverse-CDF sampling over full
// rows, segment-parallel, for the jobs stage 1 posted (a target row whose kept
// set is not an explicit list).
//
// The resample: x ~ norm(max(0, p_t - p_d)) ("Accelerating Large Language
// Model Decoding with Speculative Sampling", The algorithm; "Speculative
// Decoding from Scratch", The heart of it, 2.3), or the bonus x ~ p_t at
// position K_b + 1 (The big picture, 2.1).  Inverse CDF in ascending token
// id: the smallest v with C(v) > u Z.  Masses are summed exactly as 2^-56
// fixed-point integers so the per-segment totals, the prefix over segments and
// the rescan of the crossing segment agree bit for bit.
#include <algorithm>

#include "sv_internal.cuh"

namespace sv {

struct DenseJob {
    bool residual;
    RowStat ts;            // target (or sampled) row
    const void* trow;
    float invSt;
    int dkind;             // 0 logits, 1 probabilities
    RowStat ds;            // draft row (logits)
    const void* drow;
    float invSd;
    const int32_t* dids;   // draft kept list (MODE_LIST)
    const float* dls;
    bool tvec, dvec;       // rows on 16 bytes: whole words are loaded at once
};

// p_t(v) from the target logit l at v
__device__ __forceinline__ float dense_pt(const DenseJob& J, float c, float l, int v)
{
    if (J.ts.mode != MODE_ALL && !kept_prefix(J.ts, key_of(l), v)) return 0.f;
    return ex2_fast((l - J.ts.M) * c) * J.invSt;
}

// A thread's elements of the segment at base come in SQ 16-byte words of
// the target row: element e of word q is base + (q NT + threadIdx.x) SW + e
// (consecutive threads read consecutive words).  All of them are loaded
// before any is used, so the loads share one round trip.
template <typename T> struct SampleGeom {
    static constexpr int SW = 16 / (int)sizeof(T);  // elements per word
    static constexpr int SQ = SAMPLE_EPT / SW;       // words per thread
};
static_assert(SampleGeom<float>::SQ <= SAMPLE_PARTS && SampleGeom<__nv_bfloat16>::SQ <= SAMPLE_PARTS,
              "a segment's rounds fit its partial masses");

template <typename T>
__device__ __forceinline__ int word_at(int base, int q, int t = (int)threadIdx.x)
{
    return base + (q * NT + t) * SampleGeom<T>::SW;
}

// SW elements of a row of U at v0 (16-byte aligned when vec) into out
template <typename U, int SW>
__device__ __forceinline__ void load_word(const U* row, int v0, int V, bool vec, float fill, float* out)
{
    if (vec && v0 + SW <= V) {
        constexpr int NV = SW * (int)sizeof(U) / 16;  // 16-byte loads
#pragma unroll
        for (int g = 0; g < NV; ++g) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(row + v0) + g);
            const uint32_t x[4] = {w.x, w.y, w.z, w.w};
            if (sizeof(U) == 4) {
#pragma unroll
                for (int i = 0; i < 4; ++i) out[g * 4 + i] = __uint_as_float(x[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    out[g * 8 + 2 * i] = bf16_lo(x[i]);
                    out[g * 8 + 2 * i + 1] = bf16_hi(x[i]);
                }
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < SW; ++e) out[e] = v0 + e < V ? Elem<U>::load(row, v0 + e) : fill;
    }
}

// the target logits and (when read densely) draft values of the word at v0
template <typename T>
__device__ __forceinline__ void load_word_vals(const DenseJob& J, int v0, int V, float* lt, float* dv)
{
    constexpr int SW = SampleGeom<T>::SW;
    load_word<T, SW>((const T*)J.trow, v0, V, J.tvec, -INFINITY, lt);
    if (!J.residual || (J.dkind == 0 && J.ds.mode == MODE_LIST)) {
#pragma unroll
        for (int e = 0; e < SW; ++e) dv[e] = 0.f;
    } else if (J.dkind == 1) {
        load_word<float, SW>((const float*)J.drow, v0, V, J.dvec, 0.f, dv);
    } else {
        load_word<T, SW>((const T*)J.drow, v0, V, J.dvec, -INFINITY, dv);
    }
}

// R(v) in fixed point from the target logit l and draft value d at v (v
// ascending over the calls of one walk); the draft list (if any) is walked
// with a pointer
__device__ __forceinline__ unsigned long long dense_r_fix(const DenseJob& J, float c, float l, float d, int v,
                                                          int& dptr)
{
    const float pt = dense_pt(J, c, l, v);
    if (!J.residual) return to_fix56(pt);
    if (!(pt > 0.f)) return 0ull;  // max(0, 0 - p_d) = 0: the draft need not be read
    float pd;
    if (J.dkind == 1) {
        pd = d;
    } else if (J.ds.mode == MODE_LIST) {
        const int n = J.ds.n_kept;
        while (dptr < n && __ldcg(J.dids + dptr) < v) ++dptr;
        pd = (dptr < n && __ldcg(J.dids + dptr) == v)
                 ? ex2_fast((__ldcg(J.dls + dptr) - J.ds.M) * c) * J.invSd
                 : 0.f;
    } else {
        pd = kept_prefix(J.ds, key_of(d), v) ? ex2_fast((d - J.ds.M) * c) * J.invSd : 0.f;
    }
    return to_fix56(fmaxf(pt - pd, 0.f));
}

// the fixed-point mass of each of the thread's words of the segment at base
// (all loads first)
template <typename T>
__device__ __forceinline__ void word_masses(const DenseJob& J, float c, int base, int V,
                                            unsigned long long (&wm)[SampleGeom<T>::SQ])
{
    using G = SampleGeom<T>;
    float lt[SAMPLE_EPT], dv[SAMPLE_EPT];
#pragma unroll
    for (int q = 0; q < G::SQ; ++q) load_word_vals<T>(J, word_at<T>(base, q), V, lt + q * G::SW, dv + q * G::SW);
    int dptr = 0;
    if (J.residual && J.dkind == 0 && J.ds.mode == MODE_LIST)
        dptr = lower_bound_i32(J.dids, J.ds.n_kept, min(word_at<T>(base, 0), V));
#pragma unroll
    for (int q = 0; q < G::SQ; ++q) {
        const int v0 = word_at<T>(base, q);
        wm[q] = 0ull;
#pragma unroll
        for (int e = 0; e < G::SW; ++e)
            if (v0 + e < V) wm[q] += dense_r_fix(J, c, lt[q * G::SW + e], dv[q * G::SW + e], v0 + e, dptr);
    }
}

template <typename T>
__device__ DenseJob make_job(const Params& p, const Job& jb, bool residual)
{
    DenseJob J;
    J.residual = residual;
    const int rps = p.rps;
    const int64_t V = p.V;
    J.ts = load_rowstat(p.rstat + jb.trow);
    J.invSt = 1.f / (float)J.ts.S;
    {
        const int b = jb.trow / rps, slot = jb.trow - b * rps;
        const bool is_draft = p.draft_launch || slot > p.Kmax;
        const int j = p.draft_launch ? slot : (is_draft ? slot - (p.Kmax + 1) : slot);
        const int64_t off = is_draft ? ((int64_t)b * p.Kmax + j) * V : ((int64_t)b * (p.Kmax + 1) + j) * V;
        J.trow = (const T*)(is_draft ? p.draft : p.target) + off;
    }
    J.tvec = ((uintptr_t)J.trow & 15u) == 0;
    J.dkind = p.draft_kind;
    J.drow = nullptr;
    J.dids = nullptr;
    J.dls = nullptr;
    J.invSd = 0.f;
    if (residual) {
        const int b = jb.drow / rps, slot = jb.drow - b * rps;
        const int j = slot - (p.Kmax + 1);
        const int64_t off = ((int64_t)b * p.Kmax + j) * V;
        if (J.dkind == 1) {
            J.drow = (const float*)p.draft + off;
        } else {
            J.drow = (const T*)p.draft + off;
            J.ds = load_rowstat(p.rstat + jb.drow);
            J.invSd = 1.f / (float)J.ds.S;
            J.dids = p.kept_id + (int64_t)jb.drow * KCAP;
            J.dls = p.kept_l + (int64_t)jb.drow * KCAP;
        }
    }
    J.dvec = J.drow && ((uintptr_t)J.drow & 15u) == 0;
    return J;
}

// one segment's pass: the fixed-point masses summed per round q (NT
// consecutive words) into parts[q] (smem s_part, then global), the segment
// total returned to thread 0 (integer sums: the order of the terms is free)
template <typename T>
__device__ unsigned long long segment_pass(const DenseJob& J, float c, int V, int seg,
                                           unsigned long long* parts, unsigned long long* s_part,
                                           unsigned long long* s_red)
{
    using G = SampleGeom<T>;
    unsigned long long wm[G::SQ];
    word_masses<T>(J, c, seg * SAMPLE_SEG, V, wm);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int q = 0; q < G::SQ; ++q) {
        unsigned long long w = wm[q];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        if (lane == 0) s_part[q * (NT / 32) + warp] = w;
    }
    csync();
    unsigned long long total = 0;
    if (threadIdx.x < G::SQ) {
        unsigned long long r = 0;
        for (int i = 0; i < NT / 32; ++i) r += s_part[threadIdx.x * (NT / 32) + i];
        parts[threadIdx.x] = r;
        s_red[threadIdx.x] = r;
    }
    csync();
    if (threadIdx.x == 0)
        for (int q = 0; q < G::SQ; ++q) total += s_red[q];
    csync();  // s_part and s_red may be reused
    return total;
}

// the scratch of a sampling CTA
struct SampleSmem {
    unsigned long long red[NT / 32 + 1];
    unsigned long long part[4 * (NT / 32)];
    unsigned long long base;
    int last, star, tok;
};

// the sample of job jid once every segment of it is summed (job_seg, job_part
// complete and visible), by every thread of the CTA: locate u Z, segment ->
// round -> element; the residual that summed to 0 falls back to p_t itself
template <typename T>
__device__ void sample_tail(const Params& p, int jid, const Job& jb, DenseJob J, SampleSmem& sm)
{
    using G = SampleGeom<T>;
    const int V = p.V, nseg = p.nseg_sample;
    const bool residual = jb.kind == JOB_RESIDUAL;
    unsigned long long* parts = p.job_part + (int64_t)jid * nseg * SAMPLE_PARTS;
    unsigned long long* s_red = sm.red;
    unsigned long long* s_part = sm.part;
    unsigned long long& s_base = sm.base;
    int& s_star = sm.star;
    int& s_tok = sm.tok;
    if (threadIdx.x == 0) {
        p.job_ticket[jid] = 0u;
        s_tok = -1;
    }
    unsigned long long* seg_tot = p.job_seg + (int64_t)jid * nseg;
    bool zero = false;
    unsigned long long Z0 = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        if (attempt == 1) {
            // the residual summed to 0 (rounding only): sample p_t itself
            zero = true;
            J.residual = false;
            for (int sg = 0; sg < nseg; ++sg) {
                const unsigned long long z =
                    segment_pass<T>(J, p.c, V, sg, parts + (int64_t)sg * SAMPLE_PARTS, s_part, s_red);
                if (threadIdx.x == 0) seg_tot[sg] = z;
            }
            __threadfence_block();
            csync();
        }
        const unsigned long long z = threadIdx.x < nseg ? __ldcg(seg_tot + threadIdx.x) : 0ull;
        unsigned long long Z;
        const unsigned long long exs = block_excl_scan<unsigned long long>(z, s_red, &Z);
        if (attempt == 0) Z0 = Z;
        if (Z == 0ull) {
            if (residual && attempt == 0) continue;
            break;  // nothing to sample (cannot happen for a finite row)
        }
        const unsigned long long t = cdf_target(jb.u, Z);
        if (threadIdx.x == 0) s_star = -1;
        csync();
        if (threadIdx.x < nseg && exs <= t && t < exs + z) {
            s_star = threadIdx.x;
            s_base = exs;
        }
        csync();
        const int star = s_star;
        if (star < 0) break;  // no segment holds u Z (cannot happen when Z > 0)
        // the round of the crossing segment holding u Z (thread 0, in order)
        if (threadIdx.x == 0) {
            unsigned long long acc = s_base;
            s_star = G::SQ - 1;
            for (int q = 0; q < G::SQ; ++q) {
                const unsigned long long rq = __ldcg(parts + (int64_t)star * SAMPLE_PARTS + q);
                if (t < acc + rq) {
                    s_star = q;
                    break;
                }
                acc += rq;
            }
            s_base = acc;  // the mass before that round
        }
        csync();
        const int qs = s_star;
        // that round again, one word per thread, then the thread and element
        const int v0 = word_at<T>(star * SAMPLE_SEG, qs);
        float lt[G::SW], dv[G::SW];
        load_word_vals<T>(J, v0, V, lt, dv);
        int dptr = 0;
        if (J.residual && J.dkind == 0 && J.ds.mode == MODE_LIST)
            dptr = lower_bound_i32(J.dids, J.ds.n_kept, min(v0, V));
        unsigned long long em[G::SW], mine = 0;
#pragma unroll
        for (int e = 0; e < G::SW; ++e) {
            em[e] = v0 + e < V ? dense_r_fix(J, p.c, lt[e], dv[e], v0 + e, dptr) : 0ull;
            mine += em[e];
        }
        unsigned long long rtot;
        const unsigned long long ex = block_excl_scan<unsigned long long>(mine, s_red, &rtot);
        unsigned long long acc = s_base + ex;
        if (mine > 0ull && acc <= t && t < acc + mine) {
#pragma unroll
            for (int e = 0; e < G::SW; ++e) {
                acc += em[e];
                if (acc > t) {
                    s_tok = v0 + e;
                    break;
                }
            }
        }
        csync();
        break;
    }
    if (threadIdx.x == 0) {
        p.tokens[jb.out_idx] = s_tok;
        if (!p.draft_launch) {
            if (residual && p.resid_mass) p.resid_mass[jb.b] = (float)from_fix56(Z0);
            if (zero && p.row_status) p.row_status[jb.b] = ROW_ZERO_RESIDUAL;
        }
        p.jobs[jid].kind = JOB_NONE;
    }
}

template <typename T>
__global__ void __launch_bounds__(NT, 4) k_sample(const Params p)
{
    if (exit_skip(p)) return;
    __shared__ SampleSmem sm;
    const int V = p.V, nseg = p.nseg_sample;
    // CTA c of a job takes the segments [c spc, (c + 1) spc)
    const int spc = p.sample_spc > 0 ? p.sample_spc : 1;
    const int nct = (nseg + spc - 1) / spc;
    const int jid = blockIdx.x / nct, cta = blockIdx.x - jid * nct;
    const Job jb = load_job(p.jobs + jid);
    if (jb.kind == JOB_NONE) return;
    const bool residual = jb.kind == JOB_RESIDUAL;
    DenseJob J = make_job<T>(p, jb, residual);
    unsigned long long* parts = p.job_part + (int64_t)jid * nseg * SAMPLE_PARTS;

    for (int seg = cta * spc; seg < min(nseg, (cta + 1) * spc); ++seg) {
        const unsigned long long zs =
            segment_pass<T>(J, p.c, V, seg, parts + (int64_t)seg * SAMPLE_PARTS, sm.part, sm.red);
        if (threadIdx.x == 0) p.job_seg[(int64_t)jid * nseg + seg] = zs;
    }
    if (threadIdx.x == 0) {
        __threadfence();  // the segments' masses are visible before the ticket
        sm.last = atomicAdd(&p.job_ticket[jid], 1u) == (unsigned)(nct - 1);
        if (sm.last) __threadfence();
    }
    __syncthreads();
    if (!sm.last) return;
    sample_tail<T>(p, jid, jb, J, sm);
}

// ------------------------------------------------------------------------- //
// k_sample_ring: the same sums for rows on 16 bytes, by a persistent grid    //
// that streams the jobs' segments through shared memory.  Item i (job       //
// i / nseg, segment i % nseg) goes to CTA i mod gridDim.  The CTA's copy warp //
// resolves each item's job and rows and keeps up to sr_stages() items in     //
// flight as bulk copies (the target segment, and the draft segment when the  //
// residual reads the draft densely), each landing on the stage's mbarrier;  //
// the NT sampling threads then sum their words of the stage in the same     //
// fixed point and rounds as segment_pass, weighing only the target's kept   //
// tokens.  The samples are drawn by k_sample_tail, one CTA per job, after   //
// the whole grid: a CTA that drew them as it summed a job's last segment    //
// fell behind the others and kept summing last segments (and drawing) for   //
// the rest of the grid.                                                      //
// ------------------------------------------------------------------------- //
constexpr int SR_STAGES = 4;
constexpr int SR_QUEUE = 64;  // kept tokens a warp weighs in one pass

// bytes of one stage: the target segment, then the draft segment
__host__ __device__ constexpr int sr_stage_bytes(int tsize, int dsize) { return SAMPLE_SEG * (tsize + dsize); }
// stages of the ring: 64 KB of them (two to SR_STAGES), so that three CTAs
// share an SM for every row type
__host__ __device__ constexpr int sr_stages(int stage_bytes)
{
    return 65536 / stage_bytes < 2 ? 2 : 65536 / stage_bytes > SR_STAGES ? SR_STAGES : 65536 / stage_bytes;
}

// the job's draft is read densely (a residual against draft logits not kept
// as a list, or draft probabilities)
__device__ __forceinline__ bool draft_dense(const DenseJob& J)
{
    return J.residual && (J.dkind == 1 || J.ds.mode != MODE_LIST);
}

// SW consecutive elements of a staged segment (element index i of the
// segment) into out, fill beyond n valid elements
template <typename U, int SW>
__device__ __forceinline__ void stage_word(const unsigned char* st, int i, int n, float fill, float* out)
{
    if (i + SW <= n) {
        constexpr int NV = SW * (int)sizeof(U) / 16;
#pragma unroll
        for (int g = 0; g < NV; ++g) {
            const uint4 w = reinterpret_cast<const uint4*>(st + (size_t)i * sizeof(U))[g];
            const uint32_t x[4] = {w.x, w.y, w.z, w.w};
            if (sizeof(U) == 4) {
#pragma unroll
                for (int k = 0; k < 4; ++k) out[g * 4 + k] = __uint_as_float(x[k]);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    out[g * 8 + 2 * k] = bf16_lo(x[k]);
                    out[g * 8 + 2 * k + 1] = bf16_hi(x[k]);
                }
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < SW; ++e) {
            if (i + e < n) {
                if (sizeof(U) == 4) out[e] = reinterpret_cast<const float*>(st)[i + e];
                else out[e] = __uint_as_float((uint32_t)reinterpret_cast<const unsigned short*>(st)[i + e] << 16);
            } else {
                out[e] = fill;
            }
        }
    }
}

constexpr int SR_THREADS = NT + 32;  // NT sampling threads, then the copy warp

// csync() returning whether v held in every sampling thread
__device__ __forceinline__ bool csync_and(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
                 "bar.red.and.pred p, 1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r) : "r"((uint32_t)v), "n"(NT) : "memory");
    return r != 0;
}

template <typename T>
__global__ void __launch_bounds__(SR_THREADS, 3) k_sample_ring(const Params p, int njobs)
{
    if (exit_skip(p)) return;
    using G = SampleGeom<T>;
    extern __shared__ __align__(128) unsigned char sr_ring[];
    __shared__ SampleSmem sm;
    __shared__ uint64_t s_full[SR_STAGES], s_empty[SR_STAGES];
    __shared__ int s_item[SR_STAGES];
    __shared__ Job s_jb[SR_STAGES];
    __shared__ DenseJob s_job[SR_STAGES];
    __shared__ int s_qv[NT / 32][SR_QUEUE];    // each warp's queue of kept tokens: id,
    __shared__ float s_ql[NT / 32][SR_QUEUE];  // target logit
    __shared__ float s_qd[NT / 32][SR_QUEUE];  // and draft value
    const int V = p.V, nseg = p.nseg_sample;
    const int dsize = p.draft_kind == 1 ? 4 : (int)sizeof(T);
    const int stage_bytes = sr_stage_bytes((int)sizeof(T), dsize);
    const int NST = sr_stages(stage_bytes);  // stages in the ring
    const int64_t n_items = (int64_t)njobs * nseg;
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&s_empty[s], NT / 32);  // each sampling warp frees the stage
        }
        fence_barrier_init();
    }
    __syncthreads();  // the only barrier over all SR_THREADS threads

    if (tid >= NT) {
        // ---------------- the copy warp (one thread): the CTA's items in
        // order, each job's record and rows resolved here and handed over
        // with the stage
        if (tid != NT) return;
        const uint64_t pol = l2_evict_first();
        int k = 0;
        for (int64_t i = blockIdx.x;; i += gridDim.x) {
            int jid = -1;
            Job jb;
            if (i < n_items) {
                jid = (int)(i / nseg);
                jb = load_job(p.jobs + jid);
                if (jb.kind == JOB_NONE) continue;
            }
            const int s = k % NST;
            if (k >= NST && !mbar_wait_sleep(&s_empty[s], ((k / NST) - 1) & 1, 0)) {
                atomicOr(p.err, 4u);
                // wait (bounded) for the copies still in flight before leaving
                for (int q = (k > NST ? k - NST : 0); q < k; ++q) mbar_wait(&s_full[q % NST], (q / NST) & 1);
                return;
            }
            if (jid < 0) {
                s_item[s] = -1;  // the end: one marker ends every sampling thread
                mbar_arrive(&s_full[s]);
                return;
            }
            const int seg = (int)(i - (int64_t)jid * nseg);
            const DenseJob J = make_job<T>(p, jb, jb.kind == JOB_RESIDUAL);
            s_item[s] = (int)i;
            s_jb[s] = jb;
            s_job[s] = J;
            const int n = min(SAMPLE_SEG, V - seg * SAMPLE_SEG);
            const uint32_t tb = (uint32_t)n * (uint32_t)sizeof(T);
            const uint32_t db = draft_dense(J) ? (uint32_t)n * (uint32_t)dsize : 0u;
            unsigned char* dst = sr_ring + (size_t)s * stage_bytes;
            mbar_arrive_expect_tx(&s_full[s], tb + db);  // releases the records above
            tma_load_1d_once(dst, (const T*)J.trow + (int64_t)seg * SAMPLE_SEG, tb, &s_full[s], pol);
            if (db)
                tma_load_1d_once(dst + SAMPLE_SEG * sizeof(T),
                                 (const char*)J.drow + (int64_t)seg * SAMPLE_SEG * dsize, db, &s_full[s], pol);
            ++k;
        }
    }

    // ---------------- the sampling threads
    const int lane = tid & 31, warp = tid >> 5;
    for (int k = 0;; ++k) {
        const int s = k % NST;
        if (!csync_and(mbar_wait_sleep(&s_full[s], (k / NST) & 1, p.wait_limit))) {
            if (tid == 0) atomicOr(p.err, 4u);
            break;
        }
        const int item = s_item[s];
        if (item < 0) break;
        const int jid = item / nseg, seg = item - jid * nseg;
        const Job jb = s_jb[s];
        DenseJob J = s_job[s];
        const unsigned char* st = sr_ring + (size_t)s * stage_bytes;
        const unsigned char* sd = st + SAMPLE_SEG * sizeof(T);
        const int n = min(SAMPLE_SEG, V - seg * SAMPLE_SEG);
        const int base = seg * SAMPLE_SEG;
        // this thread's words of the stage, one round at a time (word q:
        // elements (q NT + tid) SW ..)
        const bool dd = draft_dense(J);
        unsigned long long wm[G::SQ];
        int dptr = 0;
        if (J.residual && J.dkind == 0 && J.ds.mode == MODE_LIST)
            dptr = lower_bound_i32(J.dids, J.ds.n_kept, min(base + tid * G::SW, V));
#pragma unroll
        for (int q = 0; q < G::SQ; ++q) {
            const int i = (q * NT + tid) * G::SW;
            const int v0 = base + i;
            float lt[G::SW], dv[G::SW];
            stage_word<T, G::SW>(st, i, n, -INFINITY, lt);
            if (!dd) {
#pragma unroll
                for (int e = 0; e < G::SW; ++e) dv[e] = 0.f;
            } else if (J.dkind == 1) {
                stage_word<float, G::SW>(sd, i, n, 0.f, dv);
            } else {
                stage_word<T, G::SW>(sd, i, n, -INFINITY, dv);
            }
            wm[q] = 0ull;
            if (J.ts.mode == MODE_ALL) {
                // every token of the target is kept
#pragma unroll
                for (int e = 0; e < G::SW; ++e)
                    if (v0 + e < V) wm[q] += dense_r_fix(J, p.c, lt[e], dv[e], v0 + e, dptr);
            } else {
                // R(v) = 0 wherever p_t(v) = 0 (outside the target's kept
                // rank prefix): a mask of the word's kept tokens first
                uint32_t km = 0u;
                if (sizeof(T) == 2 && i + G::SW <= n) {
                    // bf16: kept iff l > val(kappa), or l = val(kappa) at an id
                    // <= i_kappa; packed compares, two values each
                    const uint4 w = *reinterpret_cast<const uint4*>(st + (size_t)i * sizeof(T));
                    const uint32_t kb = __float_as_uint(val_of(J.ts.kappa)) >> 16;
                    const uint32_t k2u = kb | (kb << 16);
                    const __nv_bfloat162 k2 = *reinterpret_cast<const __nv_bfloat162*>(&k2u);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                    uint32_t gt = 0u, eq = 0u;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&ws[h]);
                        const uint32_t mg = __hgt2_mask(x, k2), me = __heq2_mask(x, k2);
                        gt |= ((mg & 1u) | ((mg >> 15) & 2u)) << (2 * h);
                        eq |= ((me & 1u) | ((me >> 15) & 2u)) << (2 * h);
                    }
                    const int ties_ok = min(max(J.ts.i_kappa - v0 + 1, 0), G::SW);  // ids v0 .. i_kappa
                    km = gt | (eq & ((1u << ties_ok) - 1u));
                } else {
#pragma unroll
                    for (int e = 0; e < G::SW; ++e)
                        if (v0 + e < V && kept_prefix(J.ts, key_of(lt[e]), v0 + e)) km |= 1u << e;
                }
                if (!(J.residual && J.dkind == 0 && J.ds.mode == MODE_LIST)) {
                    // the warp's kept tokens of this round go to the warp's
                    // queue (in lane order) and are weighed one per lane, so a
                    // row with few kept tokens costs the warp about one pass;
                    // a lane keeps what overflows the queue
                    const unsigned FULL = 0xffffffffu;
                    const int cnt = __popc(km);
                    int incl = cnt;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(FULL, incl, o);
                        if (lane >= o) incl += y;
                    }
                    const int tot = __shfl_sync(FULL, incl, 31);
                    int pos = incl - cnt;
                    uint32_t own = 0u;  // kept tokens past the queue
#pragma unroll
                    for (int e = 0; e < G::SW; ++e) {
                        if ((km >> e) & 1u) {
                            if (pos < SR_QUEUE) {
                                s_qv[warp][pos] = v0 + e;
                                s_ql[warp][pos] = lt[e];
                                s_qd[warp][pos] = dv[e];
                            } else {
                                own |= 1u << e;
                            }
                            ++pos;
                        }
                    }
                    __syncwarp();
                    for (int i = lane; i < min(tot, SR_QUEUE); i += 32)
                        wm[q] += dense_r_fix(J, p.c, s_ql[warp][i], s_qd[warp][i], s_qv[warp][i], dptr);
                    __syncwarp();  // the queue may be refilled
                    km = own;
                }
                while (km) {
                    const int b = __ffs(km) - 1;
                    km &= km - 1u;
                    float l = 0.f, d = 0.f;  // element b, picked without indexing the arrays
#pragma unroll
                    for (int e = 0; e < G::SW; ++e)
                        if (e == b) {
                            l = lt[e];
                            d = dv[e];
                        }
                    wm[q] += dense_r_fix(J, p.c, l, d, v0 + b, dptr);
                }
            }
        }
        __syncwarp();  // the warp is done with the stage
        if (lane == 0) mbar_arrive(&s_empty[s]);
        // per round, then the segment (the samples are drawn by the next
        // grid, k_sample_tail, once every segment is summed)
        unsigned long long* parts = p.job_part + ((int64_t)jid * nseg + seg) * SAMPLE_PARTS;
#pragma unroll
        for (int q = 0; q < G::SQ; ++q) {
            unsigned long long w = wm[q];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
            if (lane == 0) sm.part[q * (NT / 32) + warp] = w;
        }
        csync();
        if (tid < G::SQ) {
            unsigned long long r = 0;
            for (int i = 0; i < NT / 32; ++i) r += sm.part[tid * (NT / 32) + i];
            parts[tid] = r;
            sm.red[tid] = r;
        }
        csync();
        if (tid == 0) {
            unsigned long long zs = 0;
            for (int q = 0; q < G::SQ; ++q) zs += sm.red[q];
            p.job_seg[(int64_t)jid * nseg + seg] = zs;
        }
        // sm.part and sm.red are next written after the next item's masses,
        // which every thread reaches only past the barrier above
    }
}

// the sample of each job after k_sample_ring: one CTA per job
template <typename T>
__global__ void __launch_bounds__(NT) k_sample_tail(const Params p)
{
    if (exit_skip(p)) return;
    __shared__ SampleSmem sm;
    const int jid = blockIdx.x;
    const Job jb = load_job(p.jobs + jid);
    if (jb.kind == JOB_NONE) return;
    sample_tail<T>(p, jid, jb, make_job<T>(p, jb, jb.kind == JOB_RESIDUAL), sm);
}

// dense post-knob distribution of every valid draft row (draft-side sampler)
template <typename T>
__global__ void __launch_bounds__(NT) k_probs(const Params p)
{
    const int r = blockIdx.x;
    const RowRef rr = row_ref(p, r);
    if (!rr.valid) return;
    const RowStat st = load_rowstat(p.rstat + r);
    if (st.flags & FLAG_NONFINITE) return;
    const int64_t off = row_elem_offset(p, rr);
    const T* row = (const T*)p.draft + off;
    float* out = p.probs_out + off;
    const float invS = 1.f / (float)st.S;
    const int32_t* ids = p.kept_id + (int64_t)r * KCAP;
    const float* ls = p.kept_l + (int64_t)r * KCAP;
    for (int v = threadIdx.x; v < p.V; v += NT) {
        float pr;
        if (st.mode == MODE_LIST) {
            const int i = lower_bound_i32(ids, st.n_kept, v);
            pr = (i < st.n_kept && __ldcg(ids + i) == v)
                     ? exp2f((__ldcg(ls + i) - st.M) * p.c) * invS
                     : 0.f;
        } else {
            const float l = Elem<T>::load(row, v);
            pr = kept_prefix(st, key_of(l), v) ? exp2f((l - st.M) * p.c) * invS : 0.f;
        }
        out[v] = pr;
    }
}

// ------------------------------------------------------------------------- //
// k_alpha: the acceptance statistic alpha_j = sum_v min(p_t(v), p_d(v)) of   //
// every drafted slot ("Speculative Decoding from Scratch", The acceptance     //
// rate alpha decides everything (3.1-3.2)), on request: one CTA per slot,    //
// summed exactly in 2^-56 fixed point.  A row kept as a list contributes     //
// only its list; otherwise the pass covers the vocabulary.  NaN where the    //
// slot is beyond K_b, the sequence failed, or the verify is greedy.          //
// ------------------------------------------------------------------------- //
template <typename T>
__global__ void __launch_bounds__(NT) k_alpha(const Params p)
{
    if (exit_skip(p)) return;
    __shared__ unsigned long long s_red[NT / 32 + 1];
    const int K = p.Kmax;
    const int b = blockIdx.x / K, j = blockIdx.x - b * K;
    const int kb = seq_k(p, b);
    float* dst = p.alpha + (int64_t)b * K + j;
    if (!k_ok(p, kb) || j >= kb || p.greedy || __ldcg(p.num_accepted + b) < 0) {
        if (threadIdx.x == 0) *dst = NAN;
        return;
    }
    const float c = p.c;
    const int V = p.V;
    const int tr = target_slot(p, b, j);
    const RowStat ts = load_rowstat(p.rstat + tr);
    const T* trow = (const T*)p.target + ((int64_t)b * (K + 1) + j) * V;
    const float invSt = 1.f / (float)ts.S;
    const bool dprobs = p.draft_kind == 1;
    const int dr = draft_slot(p, b, j);
    RowStat ds = ts;
    float invSd = 0.f;
    if (!dprobs) {
        ds = load_rowstat(p.rstat + dr);
        invSd = 1.f / (float)ds.S;
    }
    const int64_t doff = ((int64_t)b * K + j) * V;
    // p_t(v) of a target row not kept as a list
    auto pt_at = [&](int v) -> float {
        const float l = Elem<T>::load(trow, v);
        return kept_prefix(ts, key_of(l), v) ? ex2_fast((l - ts.M) * c) * invSt : 0.f;
    };
    auto pd_at = [&](int v) -> float {
        if (dprobs) return __ldg((const float*)p.draft + doff + v);
        if (ds.mode == MODE_LIST) {
            const int32_t* ids = p.kept_id + (int64_t)dr * KCAP;
            const int i = lower_bound_i32(ids, ds.n_kept, v);
            return (i < ds.n_kept && __ldcg(ids + i) == v)
                       ? ex2_fast((__ldcg(p.kept_l + (int64_t)dr * KCAP + i) - ds.M) * c) * invSd
                       : 0.f;
        }
        const float l = Elem<T>::load((const T*)p.draft + doff, v);
        return kept_prefix(ds, key_of(l), v) ? ex2_fast((l - ds.M) * c) * invSd : 0.f;
    };
    unsigned long long part = 0;
    if (ts.mode == MODE_LIST) {
        const int32_t* ids = p.kept_id + (int64_t)tr * KCAP;
        const float* ls = p.kept_l + (int64_t)tr * KCAP;
        for (int i = threadIdx.x; i < ts.n_kept; i += NT) {
            const float pt = ex2_fast((__ldcg(ls + i) - ts.M) * c) * invSt;
            part += to_fix56(fminf(pt, pd_at(__ldcg(ids + i))));
        }
    } else if (!dprobs && ds.mode == MODE_LIST) {
        const int32_t* ids = p.kept_id + (int64_t)dr * KCAP;
        const float* ls = p.kept_l + (int64_t)dr * KCAP;
        for (int i = threadIdx.x; i < ds.n_kept; i += NT) {
            const float pd = ex2_fast((__ldcg(ls + i) - ds.M) * c) * invSd;
            part += to_fix56(fminf(pt_at(__ldcg(ids + i)), pd));
        }
    } else {
        for (int v = threadIdx.x; v < V; v += NT) part += to_fix56(fminf(pt_at(v), pd_at(v)));
    }
    unsigned long long total;
    block_excl_scan<unsigned long long>(part, s_red, &total);
    if (threadIdx.x == 0) *dst = (float)from_fix56(total);
}

cudaError_t launch_alpha(const Params& p, int dtype, cudaStream_t s)
{
    const int64_t slots = (int64_t)p.B * p.Kmax;
    if (slots <= 0 || !p.alpha) return cudaSuccess;
    if (dtype == 1) k_alpha<__nv_bfloat16><<<(unsigned)slots, NT, 0, s>>>(p);
    else k_alpha<float><<<(unsigned)slots, NT, 0, s>>>(p);
    return cudaGetLastError();
}

// every row the samplers may read starts on 16 bytes and holds whole
// 16-byte words (the bulk copies of the ring kernel need both)
static bool rows_on_16(const Params& p, int dtype)
{
    const int64_t ts = dtype == 1 ? 2 : 4;
    if (((int64_t)p.V * ts) % 16 != 0 || ((int64_t)p.V * 4) % 16 != 0) return false;
    const void* t = p.draft_launch ? p.draft : p.target;
    return ((uintptr_t)t & 15u) == 0 && ((uintptr_t)p.draft & 15u) == 0;
}

template <typename T>
static cudaError_t launch_sample_ring(const Params& p, int njobs, cudaStream_t s)
{
    const int dsize = p.draft_kind == 1 ? 4 : (int)sizeof(T);
    const int smem = sr_stages(sr_stage_bytes((int)sizeof(T), dsize)) * sr_stage_bytes((int)sizeof(T), dsize);
    struct Geo {
        int sms, per_sm;
    };
    static DeviceOnce once[2];  // per device and draft kind: the opt-in and the CTAs per SM
    Geo g{0, 0};
    int packed = 0;
    const cudaError_t e = cuda_once(once[p.draft_kind == 1], &packed, [smem](int dev, int* out) {
        cudaError_t r = cudaFuncSetAttribute(k_sample_ring<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        int sms = 0, per = 0;
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (r == cudaSuccess) r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_sample_ring<T>, SR_THREADS, smem);
        *out = sms * 16 + (per < 1 ? 1 : per > 15 ? 15 : per);
        return r;
    });
    if (e != cudaSuccess) return e;
    g.sms = packed / 16;
    g.per_sm = packed % 16;
    const int64_t items = (int64_t)njobs * p.nseg_sample;
    const int grid = (int)std::min<int64_t>(items, (int64_t)g.sms * g.per_sm);
    k_sample_ring<T><<<grid, SR_THREADS, smem, s>>>(p, njobs);
    cudaError_t e2 = cudaGetLastError();
    if (e2 != cudaSuccess) return e2;
    k_sample_tail<T><<<njobs, NT, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_sample(const Params& p, int dtype, int njobs, cudaStream_t s, int* launches)
{
    if (njobs <= 0 || p.nseg_sample <= 0) return cudaSuccess;
    if (rows_on_16(p, dtype)) {
        if (launches) *launches += 2;
        return dtype == 1 ? launch_sample_ring<__nv_bfloat16>(p, njobs, s) : launch_sample_ring<float>(p, njobs, s);
    }
    if (launches) *launches += 1;
    // rows off 16 bytes: one CTA per (job, group of segments), about eight
    // CTAs per SM in all
    Params q = p;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t segs = (int64_t)njobs * p.nseg_sample;
    q.sample_spc = (int)std::max<int64_t>(1, (segs + 8LL * sms - 1) / (8LL * sms));
    const int nct = (p.nseg_sample + q.sample_spc - 1) / q.sample_spc;
    const unsigned grid = (unsigned)((int64_t)njobs * nct);
    if (dtype == 1) k_sample<__nv_bfloat16><<<grid, NT, 0, s>>>(q);
    else k_sample<float><<<grid, NT, 0, s>>>(q);
    return cudaGetLastError();
}

cudaError_t launch_probs(const Params& p, int dtype, cudaStream_t s)
{
    const int64_t rows = (int64_t)p.B * p.rps;
    if (rows <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)rows;
    if (dtype == 1) k_probs<__nv_bfloat16><<<grid, NT, 0, s>>>(p);
    else k_probs<float><<<grid, NT, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sv
