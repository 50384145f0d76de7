// sv_noalloc.cu -- the verify step for callers that cannot allocate device
// memory (see spec_verify_run_noalloc in include/spec_verify.h).
//
// The workspace is one file-scope device array.  Host code cannot use the
// array's name as a device address (on the host it names a stand-in object),
// so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current, checks the result and
// keeps it; every later call on the device reuses it.  Nothing here calls
// cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "spec_verify.h"
#include <cuda_runtime.h>

// every GPU that loads the library holds this array until the process exits
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

size_t sv_noalloc_bytes(const spec_verify_config* cfg, int32_t batch, int32_t k_max);
spec_status sv_noalloc_run(void* ws, size_t ws_bytes, int num_sms, const spec_verify_config* cfg,
                           const spec_verify_inputs* in, const spec_sampling* s,
                           const spec_verify_outputs* out, void* stream);

namespace {

constexpr int MAX_DEVICES = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[MAX_DEVICES];  // device address of the array, per device
int g_num_sms[MAX_DEVICES];

// once per device, with that device current
spec_status setup_device(int dev)
{
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_addr[dev]) return SPEC_OK;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    g_num_sms[dev] = sms;
    g_scratch_addr[dev] = ptr;
    return SPEC_OK;
}

// does a run of these sizes fit the array?
bool fits(const spec_verify_config* cfg, int32_t batch, int32_t k_max)
{
    const size_t need = sv_noalloc_bytes(cfg, batch, k_max);
    return need > 0 && need <= SPEC_NOALLOC_SCRATCH_BYTES;
}

}  // namespace

extern "C" {

spec_status spec_verify_run_noalloc(const spec_verify_config* cfg, const spec_verify_inputs* in,
                                    const spec_sampling* s, const spec_verify_outputs* out,
                                    void* stream)
{
    if (!cfg || !in || !s || !out) return SPEC_ERR_INVALID_ARG;
    if (cfg->device < 0 || cfg->device >= MAX_DEVICES) return SPEC_ERR_INVALID_ARG;
    // the fused LM head needs its fp32 logits in a workspace far larger than the array
    if (cfg->target_kind == SPEC_TARGET_HIDDEN_LMHEAD) return SPEC_ERR_UNSUPPORTED;
    if (!fits(cfg, in->batch, in->k_max)) return SPEC_ERR_INVALID_ARG;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return SPEC_ERR_CUDA;
    if (prev != cfg->device && cudaSetDevice(cfg->device) != cudaSuccess) return SPEC_ERR_CUDA;
    spec_status st = setup_device(cfg->device);
    if (st == SPEC_OK)
        st = sv_noalloc_run(g_scratch_addr[cfg->device], SPEC_NOALLOC_SCRATCH_BYTES,
                            g_num_sms[cfg->device], cfg, in, s, out, stream);
    if (prev != cfg->device) cudaSetDevice(prev);
    return st;
}

}  // extern "C"
