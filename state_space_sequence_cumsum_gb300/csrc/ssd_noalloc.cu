// ssd_fwd_noalloc: the whole SSD forward for callers that cannot allocate
// device memory.
//
// Who needs it: code that runs where cudaMalloc / cudaFree (or any caching
// allocator built on them) are off limits -- inside a custom allocator or
// memory-pool callback, a plugin host that owns every device allocation and
// forbids others, real-time loops where an allocation's implicit device
// synchronisation or latency is unacceptable, or a caller with no allocator
// of its own at hand.  ssd_fwd needs a caller-provided workspace; this entry
// point uses a fixed scratch array that lives in the library instead.
//
// The scratch array below is a file-scope __device__ array.  Its name in host
// code is only a host-side stand-in, so its device address is looked up with
// cudaGetSymbolAddress the first time the entry point runs on each device
// (with that device current) and cached; every call on that device then
// passes that address as ssd_fwd's workspace.  Nothing here allocates.
#include <mutex>

#include "ssd_internal.h"

namespace ssd {
namespace {

// Fixed scratch size: holds G_cum and dt_t for up to ~20.9M (batch x head x
// token) elements, plus whatever else ssd_fwd's chosen path needs.
constexpr size_t kNoAllocScratchBytes = 160ull << 20;  // 160 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch[kMaxDevices];

// Device address of the scratch array on the current device; nullptr on error.
void *scratch_for_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return nullptr;
        g_scratch[dev] = p;
    }
    return g_scratch[dev];
}

}  // namespace
}  // namespace ssd

extern "C" ssd_status_t ssd_fwd_noalloc(const void *x, const float *dt, const float *A,
                                        const void *Bm, const void *Cm, const float *D,
                                        const float *init_state, void *y, float *final_state,
                                        float *chunk_states, ssd_dims_t dims, ssd_dtype_t dtype,
                                        int chunk_size, void *stream)
{
    // the least the call runs with: the head-pair kernel falls back to its
    // hand-off plan when the scratch cannot hold the prefilled one
    const size_t need =
        ssd::fwd_workspace_min_size(dims, dtype, chunk_size, chunk_states != nullptr ? 1 : 0);
    if (need == 0)
        return SSD_ERR_INVALID_ARG;
    if (need > ssd::kNoAllocScratchBytes)
        return SSD_ERR_UNSUPPORTED;
    void *scratch = ssd::scratch_for_current_device();
    if (!scratch)
        return SSD_ERR_CUDA;
    // Nothing in the scratch needs to start at zero: every workspace region
    // ssd_fwd uses is written by an earlier kernel of the same call before
    // any kernel reads it.
    return ssd_fwd(x, dt, A, Bm, Cm, D, init_state, y, final_state, chunk_states, dims, dtype,
                   chunk_size, scratch, ssd::kNoAllocScratchBytes, stream);
}
