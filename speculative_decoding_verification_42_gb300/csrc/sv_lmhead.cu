// sv_lmhead.cu -- the LM head of the fused verify round: logits = H x W.
//
// H [M, K] bf16 (row-major: the hidden states of the M = B (K_max + 1)
// verified positions), W [K, N] bf16 (row-major [hidden, vocab]) and fp32
// logits [M, N] with fp32 accumulation (the dense contraction of the fused
// workload; "Accelerating Large Language Model Decoding with Speculative
// Sampling", The cost of one token, is the target model's forward pass that
// produces these logits).
//
// One CTA computes a 128 x 256 tile of logits on the 5th-generation tensor
// cores: lane 0 of warp 0 streams 64-deep K slices of H and W into a
// four-stage shared-memory ring with tensor-map bulk copies (128-byte
// swizzle); lane 0 of warp 1 issues tcgen05.mma (kind::f16, bf16 x bf16 ->
// fp32, M = 128, N = 256, K = 16 per instruction) into a tensor-memory
// accumulator and releases each stage with tcgen05.commit; after the last
// slice the four warps read the accumulator back (tcgen05.ld, one row per
// thread) and store the fp32 tile.  H is the K-major A operand; W, whose rows
// run along the vocabulary, is the N-major B operand.
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched at run time)

#include "sv_internal.cuh"
#include "spec_verify.h"

namespace sv {

constexpr int LM_BM = 128, LM_BN = 256, LM_BK = 64, LM_STAGES = 4;
constexpr int LM_A_BYTES = LM_BM * LM_BK * 2;      // 16 KB: 128 rows of one 128-byte swizzle row
constexpr int LM_B_BYTES = LM_BK * LM_BN * 2;      // 32 KB: four 64-column boxes of 64 K-rows
constexpr int LM_BOX_B = LM_BK * 64 * 2;           // 8 KB: one W box (64 K-rows x 64 columns)
constexpr int LM_STAGE_BYTES = LM_A_BYTES + LM_B_BYTES;
constexpr int LM_SMEM = LM_STAGES * LM_STAGE_BYTES + 1024;  // + slack for 1024-byte alignment
constexpr uint32_t LM_TMEM_COLS = 256;              // fp32 accumulator: 128 lanes x 256 columns

// ------------------------------------------------------------------------- //
// PTX wrappers                                                              //
// ------------------------------------------------------------------------- //
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (all in 16-byte units), descriptor version 1
__device__ __forceinline__ uint64_t lm_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A
// K-major, B N-major, M = 128, N = 256
constexpr uint32_t LM_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                              ((uint32_t)(LM_BN >> 3) << 17) | ((uint32_t)(LM_BM >> 4) << 24);

__device__ __forceinline__ void lm_mma(uint32_t tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(tmem), "l"(adesc), "l"(bdesc), "r"(LM_IDESC), "r"(accumulate)
                 : "memory");
}
// arrive on bar once every tcgen05.mma issued so far by this thread completes
__device__ __forceinline__ void lm_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
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
// k_lmhead: one 128 x 256 tile of logits per CTA (grid: N tiles x M tiles)  //
// ------------------------------------------------------------------------- //
__global__ void __launch_bounds__(128, 1)
    k_lmhead(const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
             float* __restrict__ out, int M, int N, int K, int64_t ldo, unsigned* err)
{
    extern __shared__ unsigned char lm_smem_raw[];
    __shared__ __align__(8) uint64_t full[LM_STAGES];
    __shared__ __align__(8) uint64_t empty[LM_STAGES];
    __shared__ __align__(8) uint64_t done;
    __shared__ uint32_t tmem_slot;
    __shared__ int failed;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // stage buffers on a 1024-byte boundary (the period of the 128-byte swizzle)
    const uint32_t raw = smem_u32(lm_smem_raw);
    unsigned char* base = lm_smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int m0 = blockIdx.y * LM_BM, n0 = blockIdx.x * LM_BN;
    const int nk = (K + LM_BK - 1) / LM_BK;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_slot)), "r"(LM_TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 32) {
        for (int s = 0; s < LM_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        failed = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (threadIdx.x == 0) {
        // ---------------- producer: K slices of H and W into the ring
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt % LM_STAGES;
            if (kt >= LM_STAGES && !mbar_wait(&empty[s], ((kt / LM_STAGES) - 1) & 1)) {
                failed = 1;
                break;
            }
            unsigned char* a = base + s * LM_STAGE_BYTES;
            unsigned char* b = a + LM_A_BYTES;
            mbar_arrive_expect_tx(&full[s], LM_STAGE_BYTES);
            tma_load_2d(a, &tmap_h, kt * LM_BK, m0, &full[s]);
#pragma unroll
            for (int j = 0; j < LM_BN / 64; ++j)
                tma_load_2d(b + j * LM_BOX_B, &tmap_w, n0 + 64 * j, kt * LM_BK, &full[s]);
        }
    } else if (threadIdx.x == 32) {
        // ---------------- MMA issuer
        bool ok = true;
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt % LM_STAGES;
            if (!mbar_wait(&full[s], (kt / LM_STAGES) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a = smem_u32(base + s * LM_STAGE_BYTES);
            const uint32_t b = a + LM_A_BYTES;
#pragma unroll
            for (int kk = 0; kk < LM_BK / 16; ++kk) {
                // A: 16 K-elements = 32 bytes along the swizzled row; 8-row
                // groups 1024 bytes apart.  B: 16 K-rows = 2048 bytes; 64-column
                // boxes 8 KB apart, 8-row groups 1024 bytes apart.
                const uint64_t ad = lm_sdesc(a + kk * 32, 16, 1024);
                const uint64_t bd = lm_sdesc(b + kk * 2048, LM_BOX_B, 1024);
                lm_mma(tmem, ad, bd, (kt | kk) != 0 ? 1u : 0u);
            }
            lm_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        if (!ok) failed = 1;
        lm_commit(&done);  // the accumulator is complete (or the loop gave up)
    }
    // ---------------- epilogue: one accumulator row per thread
    const bool have = __all_sync(0xffffffffu, mbar_wait(&done, 0));
    tc_fence_after();
    if (have && !*(volatile int*)&failed) {
        const int row = m0 + warp * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < LM_BN; c += 32) {
            uint32_t v[32];
            lm_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
            if (row < M) {
                float* o = out + (int64_t)row * ldo + n0 + c;
                const int nvalid = min(32, N - (n0 + c));
                if (nvalid == 32) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        reinterpret_cast<float4*>(o)[q] =
                            make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                        __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                } else {
                    for (int q = 0; q < nvalid; ++q) o[q] = __uint_as_float(v[q]);
                }
            }
        }
    } else if (threadIdx.x == 0 && err) {
        atomicOr(err, 8u);  // a bounded wait ran out: the tile was not written
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(LM_TMEM_COLS)
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
                          unsigned* err, cudaStream_t s)
{
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_lmhead, cudaFuncAttributeMaxDynamicSharedMemorySize, LM_SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    CUtensorMap mh, mw;
    if (!bf16_map(&mh, hidden, M, K, LM_BK, LM_BM) || !bf16_map(&mw, w, K, N, 64, LM_BK))
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((N + LM_BN - 1) / LM_BN), (unsigned)((M + LM_BM - 1) / LM_BM));
    k_lmhead<<<grid, 128, LM_SMEM, s>>>(mh, mw, out, M, N, K, ldo, err);
    return cudaGetLastError();
}

}  // namespace sv
