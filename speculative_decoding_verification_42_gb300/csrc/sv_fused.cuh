// sv_fused.cuh -- the verify step of the top-k rows (1 <= k <= CAND_TOPK_MAX,
// rows on 16 bytes) as one persistent kernel (included by sv_rows.cu after
// the row merge of sv_mcand.cuh).
//
// Every CTA carries three roles that run at the same time:
//  * a producer thread (warp 8) streams the CTA's work items (row slot,
//    segment) into a six-stage shared-memory ring with bulk copies, item =
//    from a grid-wide counter, so that the rows complete in row order over
//    the whole stream;
//  * four stream warps (4..7) reduce each segment to its 16-bit chunk keys
//    (the largest logit of each 128-byte chunk);
//  * four merge warps (0..3) merge the rows blockIdx.x, blockIdx.x +
//    gridDim.x, ... as soon as their chunk keys are complete, while the
//    stream goes on: the bound on the k-th largest logit, the gather of the
//    chunks that reach it, the exact top-k, softmax and kept list; and the
//    last row of a sequence decides it (sv_mcand.cuh).
// A chunk key is never 0 once written (sv_rows.cu keeps 0 free), the
// workspace starts at 0, and the merge writes 0 back over a row's keys once
// it is done with them: a row is complete when none of its keys is 0, which
// needs no fence on the stream side.  The merge warps wait for other CTAs'
// stream warps, so the grid is launched cooperatively (every CTA resident)
// and each wait is bounded.
#pragma once

namespace sv {

constexpr int FZ_NSTAGE = 4;                       // ring stages per CTA
constexpr int FZ_GROUPS = 1;                       // stream groups: group g takes stages k = g mod FZ_GROUPS
constexpr int FZ_GT = 128 / FZ_GROUPS;             // threads of a stream group
constexpr int FZ_MERGE = MC_T;                     // merge threads: warps 0..3
constexpr int FZ_STREAM0 = FZ_MERGE;               // first stream thread
constexpr int FZ_PROD = FZ_STREAM0 + NS;           // the producer thread (warp 8, lane 0)
constexpr int FZ_THREADS = FZ_PROD + 32;
constexpr int FZ_CTAS_PER_SM = 3;
constexpr int FZ_SMEM = FZ_NSTAGE * SEG_BYTES;     // dynamic: the ring
constexpr uint32_t FZ_POLL_LIMIT = 1u << 22;       // polls of a row's keys (about a second)
static_assert(MC_T == 128 && NS == 128, "warps 0..3 merge, 4..7 stream");
static_assert(FZ_NSTAGE % FZ_GROUPS == 0 && FZ_GT % 32 == 0, "a stage always belongs to one group");

struct FzRing {
    uint64_t full[FZ_NSTAGE];
    uint64_t empty[FZ_NSTAGE];
    int item[FZ_NSTAGE];
};

// barrier of stream group g of the fused kernel (named barrier 3 + g; the
// merge warps use barrier 2 through the row merge's ssync)
__device__ __forceinline__ void fz_sync(int g) { asm volatile("bar.sync %0, %1;" ::"r"(3 + g), "n"(FZ_GT) : "memory"); }
__device__ __forceinline__ bool fz_sync_and(int g, bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
                 "bar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r) : "r"((uint32_t)v), "r"(3 + g), "n"(FZ_GT) : "memory");
    return r != 0;
}

// does any of the row's chunk keys still hold 0 (a chunk not streamed yet)?
// Every merge thread gets the answer.
__device__ __forceinline__ bool fz_row_pending(const Params& p, int r, int* flag)
{
    const uint4* k = reinterpret_cast<const uint4*>(p.chunk + (int64_t)r * p.chunk_stride);
    const int nw = (p.nchunk + 7) / 8;  // 16-byte words holding the row's keys
    bool zero = false;
    for (int w = threadIdx.x; w < nw; w += MC_T) {
        const uint4 v = __ldcg(k + w);
        const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = w * 8 + 2 * i;
            if (c < p.nchunk && (x[i] & 0xFFFFu) == 0u) zero = true;
            if (c + 1 < p.nchunk && (x[i] >> 16) == 0u) zero = true;
        }
    }
    if (threadIdx.x == 0) *flag = 0;
    ssync();
    if (zero) *flag = 1;
    ssync();
    return *flag != 0;
}

// writes 0 over the row's chunk keys (the next launch streams them again)
__device__ __forceinline__ void fz_clear_keys(const Params& p, int r)
{
    uint4* k = reinterpret_cast<uint4*>(p.chunk + (int64_t)r * p.chunk_stride);
    const int nw = p.chunk_stride / 8;
    for (int w = threadIdx.x; w < nw; w += MC_T) __stcg(k + w, make_uint4(0, 0, 0, 0));
}

template <typename T>
__global__ void __launch_bounds__(FZ_THREADS, FZ_CTAS_PER_SM) k_verify_topk(const Params p)
{
    extern __shared__ __align__(128) unsigned char fz_ring_smem[];  // FZ_NSTAGE x SEG_BYTES
    __shared__ FzRing ring;
    __shared__ McSmem sm;
    __shared__ int s_pending;
    // the item this CTA's stream warps finished last (every CTA goes through
    // the items at about the same pace, so it tells when a row can be near
    // complete), and whether they are done
    __shared__ volatile int s_stream_item;
    __shared__ volatile int s_stream_done;   // groups done
    using G = SegGeom<T, FZ_GT>;
    if (exit_skip(p)) return;
    // the decision grid that follows may be scheduled now; it waits for this
    // grid's completion before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == FZ_PROD) {
        for (int s = 0; s < FZ_NSTAGE; ++s) {
            mbar_init(&ring.full[s], 1);
            mbar_init(&ring.empty[s], 1);
        }
        fence_barrier_init();
        s_stream_item = -1;
        s_stream_done = 0;
    }
    __syncthreads();  // the only barrier over all FZ_THREADS threads
    const int64_t total_items = (int64_t)p.B * p.rps * p.nseg;
    const int64_t row_bytes = (int64_t)p.V * (int64_t)sizeof(T);

    if (threadIdx.x >= FZ_PROD) {
        // ---------------- producer
        if (threadIdx.x != FZ_PROD) return;
        // items come from a grid-wide counter in order, so that rows complete
        // in row order and a CTA slowed by its merges streams fewer of them;
        // the last producer out sets the counter back to 0
        int k = 0;
        bool failed = false;
        int64_t item = atomicAdd(p.work_ctr, 1u);
        for (;; item = atomicAdd(p.work_ctr, 1u)) {
            if (item >= total_items) {
                item = -1;
                if (atomicAdd(p.work_ctr + 1, 1u) == gridDim.x - 1) {
                    p.work_ctr[0] = 0u;
                    p.work_ctr[1] = 0u;
                }
            } else {
                const int r = (int)(item / p.nseg);
                const RowRef rr = row_ref(p, r);
                if (!rr.valid) continue;
                if (rr.is_draft && !drafts_streamed(p)) continue;
            }
            const int s = k % FZ_NSTAGE;
            if (k >= FZ_NSTAGE && !mbar_wait(&ring.empty[s], ((k / FZ_NSTAGE) - 1) & 1)) {
                atomicOr(p.err, 1u);
                failed = true;
                break;
            }
            ring.item[s] = (int)item;
            if (item < 0) {
                // the end-of-work sentinel, one for each group (the next
                // FZ_GROUPS stages)
                mbar_arrive(&ring.full[s]);
                bool ok = true;
                for (int g = 1; g < FZ_GROUPS && ok; ++g) {
                    ++k;
                    const int s2 = k % FZ_NSTAGE;
                    if (k >= FZ_NSTAGE && !mbar_wait(&ring.empty[s2], ((k / FZ_NSTAGE) - 1) & 1)) {
                        atomicOr(p.err, 1u);
                        ok = false;
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
            const uint32_t bytes = (uint32_t)min((int64_t)SEG_BYTES, row_bytes - (int64_t)seg * SEG_BYTES);
            mbar_arrive_expect_tx(&ring.full[s], bytes);
            // no cache hint: the merge re-reads a few chunks of each row soon after
            tma_load_1d(fz_ring_smem + (size_t)s * SEG_BYTES, src, bytes, &ring.full[s]);
            ++k;
        }
        if (failed) {
            // wait (bounded) for the copies still in flight before leaving
            for (int q = (k > FZ_NSTAGE ? k - FZ_NSTAGE : 0); q < k; ++q)
                mbar_wait(&ring.full[q % FZ_NSTAGE], (q / FZ_NSTAGE) & 1);
        }
        return;
    }

    if (threadIdx.x >= FZ_STREAM0) {
        // ---------------- stream groups: chunk keys of every segment; group g
        // takes the stages k = g, g + FZ_GROUPS, ...
        const int g = (threadIdx.x - FZ_STREAM0) / FZ_GT;
        const int lt = (threadIdx.x - FZ_STREAM0) - g * FZ_GT;
        for (int k = g;; k += FZ_GROUPS) {
            const int s = k % FZ_NSTAGE;
            if (!fz_sync_and(g, mbar_wait(&ring.full[s], (k / FZ_NSTAGE) & 1))) {
                if (lt == 0) {
                    atomicOr(p.err, 2u);
                    atomicAdd((int*)&s_stream_done, 1);
                }
                break;
            }
            const int item = ring.item[s];
            if (item < 0) {
                if (lt == 0) atomicAdd((int*)&s_stream_done, 1);
                break;
            }
            const int r = item / p.nseg, seg = item - r * p.nseg;
            const uint4* sv4 = reinterpret_cast<const uint4*>(fz_ring_smem + (size_t)s * SEG_BYTES);
            const int64_t base = (int64_t)seg * G::SEG;
            segment_compute<T, SEG_CHUNK, FZ_GT>(
                p,
                [&](int i) {
                    const int64_t e0 = base + ((int64_t)i * FZ_GT + lt) * G::VW;
                    return e0 < p.V ? sv4[i * FZ_GT + lt] : Vec16<T>::neg_inf();
                },
                seg, r, lt, [g] { fz_sync(g); }, nullptr, nullptr);
            fz_sync(g);  // every thread of the group is done with the stage
            if (lt == 0) {
                mbar_arrive(&ring.empty[s]);
                s_stream_item = item;
            }
        }
        return;
    }

    // ---------------- merge warps: rows blockIdx.x + i gridDim.x, each once
    // its chunk keys are complete
    const int nrows = p.B * p.rps;
    for (int r = blockIdx.x; r < nrows; r += gridDim.x) {
        const RowRef rr = row_ref(p, r);
        if (!rr.valid) {
            if (threadIdx.x == 0) report_skipped_row(p, rr);
            continue;
        }
        if (rr.is_draft && !drafts_streamed(p)) continue;  // probabilities (or greedy): not streamed
        // until this CTA's own stream is within a round of the row's last
        // item, the row cannot be complete: wait on shared memory only (the
        // stream warps' waits are bounded, and they mark themselves done on
        // every way out, so this loop ends)
        const int last_item = (r + 1) * p.nseg - 1;
        while (s_stream_done < FZ_GROUPS && s_stream_item + (int)gridDim.x < last_item) __nanosleep(500);
        uint32_t polls = 0;  // the same in every merge thread from here on
        while (fz_row_pending(p, r, &s_pending)) {
            if (++polls == FZ_POLL_LIMIT) break;
            __nanosleep(256);
        }
        if (polls == FZ_POLL_LIMIT) {
            // the row never completed (a stream wait ran out): give up; the
            // run reports the timeout and its outputs are undefined
            if (threadIdx.x == 0) atomicOr(p.err, 4u);
            break;
        }
        merge_row_topk<T>(p, r, sm);
        // the row's keys are read; a row left to the decision grid (ties)
        // keeps them for its block merge there
        if (threadIdx.x == 0) s_pending = __ldcg(&p.rstat[r].flags) & FLAG_BLOCK_MERGE;
        ssync();
        if (!s_pending) fz_clear_keys(p, r);
        ssync();
    }
}

template <typename T>
static cudaError_t launch_verify_topk_t(const Params& p, int num_sms, cudaStream_t s)
{
    static DeviceOnce once;  // the shared-memory opt-in and the resident CTAs per SM, per device
    int per_sm = 0;
    cudaError_t e = cuda_once(once, &per_sm, [](int, int* n) {
        cudaError_t e2 = cudaFuncSetAttribute(k_verify_topk<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              FZ_SMEM);
        if (e2 != cudaSuccess) return e2;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, k_verify_topk<T>, FZ_THREADS, FZ_SMEM);
    });
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const unsigned grid = (unsigned)(std::min(per_sm, FZ_CTAS_PER_SM) * num_sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(FZ_THREADS);
    cfg.dynamicSmemBytes = FZ_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the merges wait for the streams
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_verify_topk<T>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sv
