// sv_lmhead.cu -- the LM head of the fused verify round: logits = H x W.
//
// H [M, K] bf16 (row-major: the hidden states of the M = B (K_max + 1)
// verified positions), W [K, N] bf16 (row-major [hidden, vocab]) and fp32
// logits [M, N] with fp32 accumulation (the dense contraction of the fused
// workload; "Accelerating Large Language Model Decoding with Speculative
// Sampling", The cost of one token, is the target model's forward pass that
// produces these logits).
//
// Persistent pairs of CTAs (clusters of two) each own a 256 x 256 output tile
// per turn and issue one 2-SM MMA (tcgen05.mma.cta_group::2, M = 256, N =
// 256, K = 16): CTA r of the pair holds rows 128 r .. 128 r + 127 of the
// tile's H block (the A operand, K-major) and columns 128 r .. 128 r + 127 of
// the tile's W slice (the B operand, N-major) in its own shared memory, and
// its tensor memory receives its 128 rows x all 256 columns of the product.
// Every byte of W crosses HBM once and each CTA copies only its own half:
// lane 0 of warp 0 of each CTA fills a six-stage ring with tensor-map copies
// (128-byte swizzle) whose completion is counted on the even CTA's barrier;
// lane 0 of warp 1 of the even CTA issues the MMAs into one of two
// accumulators and commits each stage's release to both CTAs' barriers;
// warps 2..5 of each CTA read the other accumulator back (tcgen05.ld, one row
// per thread) and store the fp32 tile meanwhile.  On request the epilogue
// also writes, per row and 256-column tile, the softmax partials (max, sum
// exp2((l - max) c)) that the verify's row merge combines, so that no pass
// over the logits is needed for rows without top-k / top-p.
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched at run time)

#include <algorithm>

#include "sv_internal.cuh"
#include "spec_verify.h"

namespace sv {

constexpr int LM_BM = 128, LM_BN = 256, LM_BK = 64, LM_STAGES = 6;
constexpr int LM_BNH = LM_BN / 2;                  // W columns held by one CTA of the pair
constexpr int LM_A_BYTES = LM_BM * LM_BK * 2;      // 16 KB: 128 rows of one 128-byte swizzle row
constexpr int LM_BOX_B = LM_BK * 64 * 2;           // 8 KB: one W box (64 K-rows x 64 columns)
constexpr int LM_B_BYTES = LM_BK * LM_BNH * 2;     // 16 KB: two W boxes
constexpr int LM_STAGE_BYTES = LM_A_BYTES + LM_B_BYTES;
constexpr int LM_SMEM = LM_STAGES * LM_STAGE_BYTES + 1024;  // + slack for 1024-byte alignment
constexpr int LM_THREADS = 192;                     // producer, MMA, four epilogue warps
constexpr uint32_t LM_ACC_COLS = 256;               // fp32 accumulator: 128 lanes x 256 columns
constexpr uint32_t LM_TMEM_COLS = 2 * LM_ACC_COLS;  // two accumulators
static_assert(LM_BNH == 2 * 64, "each CTA of the pair copies two 64-column boxes of W");
static_assert(LM_BN == LM_STAT_COLS, "the softmax partials are per column tile");
static_assert(LM_SMEM <= 227 * 1024, "the ring fits one CTA's shared memory");

// ------------------------------------------------------------------------- //
// PTX wrappers                                                              //
// ------------------------------------------------------------------------- //
// the shared::cluster address of the same shared-memory location in CTA `rank`
__device__ __forceinline__ uint32_t lm_mapa(const void* p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// a tensor-map box into this CTA's shared memory; its bytes count on the
// mbarrier at cluster address bar (either CTA of the pair)
__device__ __forceinline__ void lm_tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                          uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_last()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (all in 16-byte units), descriptor version 1
__device__ __forceinline__ uint64_t lm_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A
// K-major, B N-major, M = 256 (the pair), N = 256
constexpr uint32_t LM_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                              ((uint32_t)(LM_BN >> 3) << 17) | ((uint32_t)((2 * LM_BM) >> 4) << 24);

__device__ __forceinline__ void lm_mma(uint32_t tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(tmem), "l"(adesc), "l"(bdesc), "r"(LM_IDESC), "r"(accumulate)
                 : "memory");
}
// arrive on the mbarrier at cluster address bar once every MMA issued so far
// by this thread completes
__device__ __forceinline__ void lm_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}
// arrive on the mbarrier at cluster address bar (either CTA of the pair)
__device__ __forceinline__ void lm_arrive_cluster(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// a bounded wait that also gives up once another role of the CTA has failed
__device__ __forceinline__ bool lm_wait(uint64_t* bar, uint32_t parity, const volatile int* failed)
{
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && *failed) return false;
    }
    return false;
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this warp's 32 accumulator lanes (thread =
// lane): v[i] = D[lane_base + lane][col + i]
__device__ __forceinline__ void lm_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------------- //
// k_lmhead: persistent CTA pairs; pair c takes the tiles c, c + C, c + 2C,   //
// ... of (256-row blocks of H) x (256-column blocks of W)                    //
// ------------------------------------------------------------------------- //
__global__ void __launch_bounds__(LM_THREADS, 1)
    k_lmhead(const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
             float* __restrict__ out, int M, int N, int K, int64_t ldo, unsigned* err, LmStats st)
{
    extern __shared__ unsigned char lm_smem_raw[];
    __shared__ __align__(8) uint64_t full[LM_STAGES];   // even CTA: the stage holds both CTAs' boxes
    __shared__ __align__(8) uint64_t empty[LM_STAGES];  // the MMAs have read this CTA's stage
    __shared__ __align__(8) uint64_t acc_full[2];       // the accumulator is complete
    __shared__ __align__(8) uint64_t acc_empty[2];      // even CTA: both CTAs read the accumulator back
    __shared__ uint32_t tmem_slot;
    __shared__ int failed;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    // stage buffers on a 1024-byte boundary (the period of the 128-byte
    // swizzle); the offset is the same in both CTAs of the pair, which the
    // 2-SM MMA needs (one descriptor addresses both CTAs' operands)
    const uint32_t raw = smem_u32(lm_smem_raw);
    unsigned char* base = lm_smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int nk = (K + LM_BK - 1) / LM_BK;
    const int n_mpair = (M + 2 * LM_BM - 1) / (2 * LM_BM);
    const int n_tiles = n_mpair * ((N + LM_BN - 1) / LM_BN);
    const int cid = blockIdx.x >> 1, n_cl = gridDim.x >> 1;
    const volatile int* vfailed = &failed;

    if (warp == 0) {
        // both CTAs of the pair allocate together (the same columns in each)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_slot)), "r"(LM_TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 32) {
        for (int s = 0; s < LM_STAGES; ++s) {
            mbar_init(&full[s], 1);   // the even CTA's producer (with both CTAs' bytes)
            mbar_init(&empty[s], 1);  // one commit of the MMA issuer
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 8);  // lane 0 of each epilogue warp of both CTAs
        }
        failed = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers are initialised before any copy or commit reaches them
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (threadIdx.x == 0) {
        // ---------------- producer (both CTAs): this CTA's half of each K slice
        const uint64_t pol_w = l2_evict_first(), pol_h = l2_evict_last();
        uint32_t it = 0;
        for (int t = cid; t < n_tiles && !*vfailed; t += n_cl) {
            const int m0 = ((t % n_mpair) * 2 + (int)rank) * LM_BM;
            const int n0 = (t / n_mpair) * LM_BN + (int)rank * LM_BNH;
            for (int kt = 0; kt < nk; ++kt, ++it) {
                const uint32_t s = it % LM_STAGES;
                if (it >= LM_STAGES && !lm_wait(&empty[s], ((it / LM_STAGES) - 1) & 1, vfailed)) {
                    failed = 1;
                    break;
                }
                unsigned char* a = base + s * LM_STAGE_BYTES;
                unsigned char* b = a + LM_A_BYTES;
                const uint32_t fb = lm_mapa(&full[s], 0);
                if (leader) mbar_arrive_expect_tx(&full[s], 2 * LM_STAGE_BYTES);
                lm_tma_2d(a, &tmap_h, kt * LM_BK, m0, fb, pol_h);
                lm_tma_2d(b, &tmap_w, n0, kt * LM_BK, fb, pol_w);
                lm_tma_2d(b + LM_BOX_B, &tmap_w, n0 + 64, kt * LM_BK, fb, pol_w);
            }
        }
        // drain: every stage this CTA filled has been read by the MMAs, so
        // no copy or commit is still on its way to either CTA's barriers
        for (uint32_t i = it; i < it + LM_STAGES && !*vfailed; ++i)
            if (i >= LM_STAGES && !lm_wait(&empty[i % LM_STAGES], ((i / LM_STAGES) - 1) & 1, vfailed))
                failed = 1;
    } else if (threadIdx.x == 32 && leader) {
        // ---------------- MMA issuer (even CTA)
        uint32_t it = 0, ti = 0;
        const uint32_t peer = 1;
        for (int t = cid; t < n_tiles && !*vfailed; t += n_cl, ++ti) {
            const uint32_t acc = ti & 1;
            if (ti >= 2 && !lm_wait(&acc_empty[acc], ((ti >> 1) - 1) & 1, vfailed)) {
                failed = 1;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + acc * LM_ACC_COLS;
            for (int kt = 0; kt < nk; ++kt, ++it) {
                const uint32_t s = it % LM_STAGES;
                if (!lm_wait(&full[s], (it / LM_STAGES) & 1, vfailed)) {
                    failed = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a = smem_u32(base + s * LM_STAGE_BYTES);
                const uint32_t b = a + LM_A_BYTES;
#pragma unroll
                for (int kk = 0; kk < LM_BK / 16; ++kk) {
                    // A: 16 K-elements = 32 bytes along the swizzled row; 8-row
                    // groups 1024 bytes apart.  B: 16 K-rows = 2048 bytes;
                    // 64-column boxes 8 KB apart, 8-row groups 1024 bytes apart.
                    const uint64_t ad = lm_sdesc(a + kk * 32, 16, 1024);
                    const uint64_t bd = lm_sdesc(b + kk * 2048, LM_BOX_B, 1024);
                    lm_mma(d, ad, bd, (kt | kk) != 0 ? 1u : 0u);
                }
                // the stage is free in both CTAs once the MMAs have read it
                lm_commit(smem_u32(&empty[s]));
                lm_commit(lm_mapa(&empty[s], peer));
            }
            // the accumulator is complete (or the loop gave up) in both CTAs
            lm_commit(smem_u32(&acc_full[acc]));
            lm_commit(lm_mapa(&acc_full[acc], peer));
        }
    } else if (warp >= 2) {
        // ---------------- epilogue: warp w reads accumulator lanes 32 (w % 4) ..
        const int q = warp & 3;
        uint32_t ti = 0;
        for (int t = cid; t < n_tiles && !*vfailed; t += n_cl, ++ti) {
            const uint32_t acc = ti & 1;
            const bool have = __all_sync(0xffffffffu, lm_wait(&acc_full[acc], (ti >> 1) & 1, vfailed));
            tc_fence_after();
            if (!have || *vfailed) {
                if (lane == 0) failed = 1;
                break;
            }
            const int m0 = ((t % n_mpair) * 2 + (int)rank) * LM_BM;
            const int n0 = (t / n_mpair) * LM_BN;
            const int row = m0 + q * 32 + lane;
            const uint32_t src = tmem + acc * LM_ACC_COLS + ((uint32_t)(q * 32) << 16);
            float tmx = -INFINITY, tsum = 0.f;  // the row's (max, sum exp2((l - max) c)) over the tile
#pragma unroll 1
            for (int c = 0; c < LM_BN; c += 32) {
                uint32_t v[32];
                lm_ld32(src + (uint32_t)c, v);
                if (st.seg) {
                    const int nvalid = min(32, N - (n0 + c));
                    float cm = -INFINITY;
#pragma unroll
                    for (int g = 0; g < 32; ++g)
                        if (g < nvalid) cm = fmax_nan(cm, __uint_as_float(v[g]));
                    const float nm = fmax_nan(tmx, cm);
                    if (nm > -INFINITY && nm < INFINITY) {
                        float add = 0.f;
#pragma unroll
                        for (int g = 0; g < 32; ++g)
                            if (g < nvalid) add += ex2_fast((__uint_as_float(v[g]) - nm) * st.c);
                        tsum = tsum * ex2_fast((tmx - nm) * st.c) + add;
                    }
                    tmx = nm;
                }
                if (row < M) {
                    float* o = out + (int64_t)row * ldo + n0 + c;
                    const int nvalid = min(32, N - (n0 + c));
                    if (nvalid == 32) {
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            reinterpret_cast<float4*>(o)[g] =
                                make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                            __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3]));
                    } else {
#pragma unroll
                        for (int g = 0; g < 32; ++g)
                            if (g < nvalid) o[g] = __uint_as_float(v[g]);
                    }
                }
            }
            if (st.seg && row < M && n0 < N) {
                // the verify's row slot of logits row `row` (position j of sequence b)
                const int b = row / st.kp1, j = row - b * st.kp1;
                SegStat ss;
                ss.m = tmx;
                ss.pad = 0.f;
                ss.s = (double)tsum;
                st.seg[((int64_t)b * st.rps + j) * st.nseg + n0 / LM_BN] = ss;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) lm_arrive_cluster(lm_mapa(&acc_empty[acc], 0));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && failed && err) atomicOr(err, 8u);  // a bounded wait ran out
    cluster_sync();  // neither CTA leaves (or frees its tensor memory) while the other may still reach it
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(LM_TMEM_COLS)
                     : "memory");
}

// ------------------------------------------------------------------------- //
// host side                                                                 //
// ------------------------------------------------------------------------- //
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

static EncodeTiled encoder()
{
    static EncodeTiled fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiled>(p);
    }
    return fn;
}

// a row-major bf16 matrix [rows, cols] as a 2-D tensor map with (box_cols,
// box_rows) boxes and 128-byte swizzle; false when the driver refuses it
static bool bf16_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_cols,
                     int box_rows)
{
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// shapes the kernel serves: row strides on 16 bytes, 16-byte-aligned bases
bool lmhead_shape_ok(const void* hidden, const void* w, int M, int N, int K)
{
    return M > 0 && N > 0 && K > 0 && (K % 8) == 0 && (N % 8) == 0 &&
           ((uintptr_t)hidden & 15u) == 0 && ((uintptr_t)w & 15u) == 0;
}

cudaError_t launch_lmhead(const void* hidden, const void* w, float* out, int M, int N, int K, int64_t ldo,
                          unsigned* err, cudaStream_t s, const LmStats& st)
{
    static DeviceOnce once;  // per device: the shared-memory opt-in and the resident pairs
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(LM_THREADS);
    cfg.dynamicSmemBytes = LM_SMEM;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int max_clusters = 0;
    cudaError_t e = cuda_once(once, &max_clusters, [&](int dev, int* n) {
        cudaError_t e2 = cudaFuncSetAttribute(k_lmhead, cudaFuncAttributeMaxDynamicSharedMemorySize, LM_SMEM);
        if (e2 != cudaSuccess) return e2;
        int sms = 0;
        if ((e2 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e2;
        cudaLaunchConfig_t q = cfg;
        q.gridDim = dim3((unsigned)(sms & ~1));
        if (cudaOccupancyMaxActiveClusters(n, k_lmhead, &q) != cudaSuccess || *n < 1) {
            (void)cudaGetLastError();
            *n = sms / 2;
        }
        return cudaSuccess;
    });
    if (e != cudaSuccess) return e;
    CUtensorMap mh, mw;
    if (!bf16_map(&mh, hidden, M, K, LM_BK, LM_BM) || !bf16_map(&mw, w, K, N, 64, LM_BK))
        return cudaErrorInvalidValue;
    const int n_mpair = (M + 2 * LM_BM - 1) / (2 * LM_BM);
    const int n_tiles = n_mpair * ((N + LM_BN - 1) / LM_BN);
    cfg.gridDim = dim3((unsigned)(2 * std::min(n_tiles, max_clusters)));
    return cudaLaunchKernelEx(&cfg, k_lmhead, mh, mw, out, M, N, K, ldo, err, st);
}

}  // namespace sv
