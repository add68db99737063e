// lola_prefill_noalloc: lola_prefill without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call into this library: code that
// runs inside a host runtime which owns the device allocator and fixes its memory budget at
// start-up, or a latency-critical path that must not call cudaMalloc/cudaFree (both can
// synchronise the whole device).  This entry point serves them: its scratch memory is one
// file-scope __device__ array of LOLA_NOALLOC_SCRATCH_BYTES bytes, created when the library
// is loaded on a device and held by every device that loads the library until the process
// exits.  It calls no allocating routine.
//
// Host code cannot use the array's name as a device address (in host code it names a
// host-side stand-in), so the address is looked up with cudaGetSymbolAddress, once per
// device, by the first call made on that device (with that device current), and cached for
// the life of the process: a cudaDeviceReset after that first call is not supported (the
// cached address would name memory of the destroyed context).
#include <mutex>

#include "lola_internal.cuh"

static __device__ __align__(256) unsigned char g_noalloc_scratch[LOLA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" {

int32_t lola_prefill_noalloc(const lola_config* cfg, int32_t n, const void* Q, const void* K, const void* V,
                             const float* W, int64_t w_head_stride, void* Y, void* state, int32_t* write_pos,
                             void* stream) {
    const int32_t chk = lola_check_config(cfg);
    if (chk != LOLA_OK) return chk;
    if (n < 1) return LOLA_ERR_INVALID_ARG;
    const size_t need = lola_prefill_workspace_bytes(cfg, n);
    if (need == 0) return LOLA_ERR_INVALID_ARG;
    if (need > (size_t)LOLA_NOALLOC_SCRATCH_BYTES) return LOLA_ERR_WORKSPACE;  // beyond the fixed array
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return lola::cuda_fail(e, "noalloc: current device");
    if (dev < 0 || dev >= kMaxDevices) return lola::cuda_fail(cudaErrorInvalidDevice, "noalloc: device ordinal");
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> g(g_mu);
        if (!g_scratch_ptr[dev]) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return lola::cuda_fail(e, "noalloc: scratch symbol address");
            if (!p) return lola::cuda_fail(cudaErrorInvalidSymbol, "noalloc: scratch symbol address");
            g_scratch_ptr[dev] = p;
        }
        scratch = g_scratch_ptr[dev];
    }
    // Every value lola_prefill reads from its workspace is written earlier in the same call
    // (its one flag that must start at zero is cleared there), so the array's contents
    // from a previous call do not matter.
    return lola_prefill(cfg, n, Q, K, V, W, w_head_stride, Y, state, write_pos, scratch,
                        (size_t)LOLA_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
