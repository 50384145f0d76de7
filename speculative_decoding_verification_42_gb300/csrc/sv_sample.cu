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
};

template <typename T>
__device__ __forceinline__ float dense_pt(const DenseJob& J, float c, int v)
{
    const float l = Elem<T>::load((const T*)J.trow, v);
    if (!kept_prefix(J.ts, key_of(l), v)) return 0.f;
    return ex2_fast((l - J.ts.M) * c) * J.invSt;
}

// R(v) of the element range [v0, v1) of one thread, in fixed point; the draft
// list (if any) is walked with a pointer
template <typename T>
__device__ __forceinline__ unsigned long long dense_r_fix(const DenseJob& J, float c, int v,
                                                          int& dptr)
{
    const float pt = dense_pt<T>(J, c, v);
    if (!J.residual) return to_fix56(pt);
    float pd;
    if (J.dkind == 1) {
        pd = __ldg((const float*)J.drow + v);
    } else if (J.ds.mode == MODE_LIST) {
        const int n = J.ds.n_kept;
        while (dptr < n && __ldcg(J.dids + dptr) < v) ++dptr;
        pd = (dptr < n && __ldcg(J.dids + dptr) == v)
                 ? ex2_fast((__ldcg(J.dls + dptr) - J.ds.M) * c) * J.invSd
                 : 0.f;
    } else {
        const float l = Elem<T>::load((const T*)J.drow, v);
        pd = kept_prefix(J.ds, key_of(l), v) ? ex2_fast((l - J.ds.M) * c) * J.invSd : 0.f;
    }
    return to_fix56(fmaxf(pt - pd, 0.f));
}

template <typename T>
__device__ __forceinline__ unsigned long long thread_part(const DenseJob& J, float c, int v0,
                                                          int v1)
{
    int dptr = 0;
    if (J.residual && J.dkind == 0 && J.ds.mode == MODE_LIST && v0 < v1)
        dptr = lower_bound_i32(J.dids, J.ds.n_kept, v0);
    unsigned long long part = 0;
    for (int v = v0; v < v1; ++v) part += dense_r_fix<T>(J, c, v, dptr);
    return part;
}

template <typename T>
__device__ DenseJob make_job(const Params& p, const Job& jb, bool residual)
{
    DenseJob J;
    J.residual = residual;
    const int rps = p.rps;
    const int64_t V = p.V;
    J.ts = load_rowstat(p.rstat + jb.trow);
    J.invSt = (float)(1.0 / J.ts.S);
    {
        const int b = jb.trow / rps, slot = jb.trow - b * rps;
        const bool is_draft = p.draft_launch || slot > p.Kmax;
        const int j = p.draft_launch ? slot : (is_draft ? slot - (p.Kmax + 1) : slot);
        const int64_t off = is_draft ? ((int64_t)b * p.Kmax + j) * V : ((int64_t)b * (p.Kmax + 1) + j) * V;
        J.trow = (const T*)(is_draft ? p.draft : p.target) + off;
    }
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
            J.invSd = (float)(1.0 / J.ds.S);
            J.dids = p.kept_id + (int64_t)jb.drow * KCAP;
            J.dls = p.kept_l + (int64_t)jb.drow * KCAP;
        }
    }
    return J;
}

// fixed-point mass of one segment (block total); every thread gets it
template <typename T>
__device__ unsigned long long segment_mass(const DenseJob& J, float c, int V, int seg,
                                           unsigned long long* red, unsigned long long* ex_out,
                                           unsigned long long* part_out, int* v0_out, int* v1_out)
{
    const int base = seg * SAMPLE_SEG;
    const int v0 = min(V, base + (int)threadIdx.x * SAMPLE_EPT);
    const int v1 = min(V, v0 + SAMPLE_EPT);
    const unsigned long long part = thread_part<T>(J, c, v0, v1);
    unsigned long long total;
    const unsigned long long ex = block_excl_scan<unsigned long long>(part, red, &total);
    if (ex_out) *ex_out = ex;
    if (part_out) *part_out = part;
    if (v0_out) *v0_out = v0;
    if (v1_out) *v1_out = v1;
    return total;
}

template <typename T>
__global__ void __launch_bounds__(NT) k_sample(const Params p)
{
    __shared__ unsigned long long s_red[NT / 32 + 1];
    __shared__ int s_last, s_star, s_tok;
    const int V = p.V, nseg = p.nseg_sample;
    const int jid = blockIdx.x / nseg, seg = blockIdx.x - jid * nseg;
    const Job jb = load_job(p.jobs + jid);
    if (jb.kind == JOB_NONE) return;
    const bool residual = jb.kind == JOB_RESIDUAL;
    DenseJob J = make_job<T>(p, jb, residual);

    const unsigned long long zs =
        segment_mass<T>(J, p.c, V, seg, s_red, nullptr, nullptr, nullptr, nullptr);
    if (threadIdx.x == 0) p.job_seg[(int64_t)jid * nseg + seg] = zs;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&p.job_ticket[jid], 1u) == (unsigned)(nseg - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
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
            for (int s = 0; s < nseg; ++s) {
                const unsigned long long z =
                    segment_mass<T>(J, p.c, V, s, s_red, nullptr, nullptr, nullptr, nullptr);
                if (threadIdx.x == 0) seg_tot[s] = z;
                __syncthreads();
            }
            __threadfence_block();
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
        if (threadIdx.x == 0) {
            s_star = -1;
            s_tok = -1;
        }
        __syncthreads();
        if (threadIdx.x < nseg && exs <= t && t < exs + z) s_star = threadIdx.x;
        __syncthreads();
        const int star = s_star;
        if (star < 0) break;  // no segment holds u Z (cannot happen when Z > 0)
        __shared__ unsigned long long s_base;
        if (threadIdx.x == star) s_base = exs;
        __syncthreads();
        // rescan the crossing segment: same per-thread partials, same order
        unsigned long long ex, part;
        int v0, v1;
        segment_mass<T>(J, p.c, V, star, s_red, &ex, &part, &v0, &v1);
        const unsigned long long before = s_base + ex;
        if (before <= t && t < before + part) {
            int dptr = 0;
            if (J.residual && J.dkind == 0 && J.ds.mode == MODE_LIST)
                dptr = lower_bound_i32(J.dids, J.ds.n_kept, v0);
            unsigned long long acc = before;
            for (int v = v0; v < v1; ++v) {
                acc += dense_r_fix<T>(J, p.c, v, dptr);
                if (acc > t) {
                    s_tok = v;
                    break;
                }
            }
        }
        __syncthreads();
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
    const float invS = (float)(1.0 / st.S);
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
    const float invSt = (float)(1.0 / ts.S);
    const bool dprobs = p.draft_kind == 1;
    const int dr = draft_slot(p, b, j);
    RowStat ds = ts;
    float invSd = 0.f;
    if (!dprobs) {
        ds = load_rowstat(p.rstat + dr);
        invSd = (float)(1.0 / ds.S);
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

cudaError_t launch_sample(const Params& p, int dtype, int njobs, cudaStream_t s)
{
    if (njobs <= 0 || p.nseg_sample <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)((int64_t)njobs * p.nseg_sample);
    if (dtype == 1) k_sample<__nv_bfloat16><<<grid, NT, 0, s>>>(p);
    else k_sample<float><<<grid, NT, 0, s>>>(p);
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
