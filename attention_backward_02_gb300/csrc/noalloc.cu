// noalloc.cu -- sdpa_bwd for callers that cannot allocate device memory.
//
// Some callers cannot hand the backward a workspace: an engine or framework
// plugin that owns every byte of device memory and forbids side
// allocations, or a latency-critical loop that must not allocate once it is
// running.  sdpa_bwd_static_scratch serves them with a scratch area compiled
// into this library (a file-scope __device__ array), so the call itself
// allocates nothing.  It runs exactly the same kernels as sdpa_bwd, with the
// static array as their workspace.
#include <mutex>

#include "attnbwd.h"
#include "common.cuh"

namespace {

// The scratch area.  Every GPU that loads this library's code holds these
// bytes until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[ATTN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};  // device address of g_static_scratch, per device

// Once per device, with that device current: look up the device address of
// the array (host code only holds a host-side stand-in for the symbol).
attn_status_t scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t sdpa_bwd_static_scratch(const attn_sdpa_desc_t *desc, attn_view_t q, attn_view_t k,
                                                 attn_view_t v, attn_view_t o, attn_view_t dO, const float *lse,
                                                 attn_view_t dQ, attn_view_t dK, attn_view_t dV, void *stream)
{
    size_t need = 0;
    attn_status_t st = sdpa_workspace_size(desc, nullptr, &need);
    if (st) return st;
    if (need > size_t(ATTN_STATIC_SCRATCH_BYTES)) return ATTN_ERR_WORKSPACE;
    void *scratch = nullptr;
    if ((st = scratch_for_current_device(&scratch))) return st;
    // sdpa_bwd's first kernel rewrites every scratch byte the later kernels
    // read (status word, D, LSE * log2 e, the zeroed dQ accumulator), so what
    // an earlier call left in the array does not matter.
    return sdpa_bwd(desc, q, k, v, o, dO, lse, dQ, dK, dV, scratch, size_t(ATTN_STATIC_SCRATCH_BYTES), stream);
}
