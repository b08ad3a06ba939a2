// noalloc.cu -- sdpa_bwd for callers that cannot allocate device memory.
//
// Some callers cannot hand the backward a workspace: an engine or framework
// plugin that owns every byte of device memory and forbids side
// allocations, or a latency-critical loop that must not allocate once it is
// running.  sdpa_bwd_static_scratch serves them with a scratch area compiled
// into this library (a file-scope __device__ array), so the call itself
// allocates nothing.  It runs exactly the same kernels as sdpa_bwd, with the
// static array as their workspace.
#include "attnbwd.h"
#include "plan.h"

namespace {

// The scratch area.  Every GPU that loads this library's code holds these
// bytes until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[ATTN_STATIC_SCRATCH_BYTES];

// Device address of the array in the current context.  In host code the
// array's name is only a host-side stand-in for the symbol, never a device
// address, so it is looked up on every call (a host-side table lookup once
// the module is loaded).  Nothing is cached: after cudaDeviceReset, or with
// another context current, the address may differ.  The first call in a
// context loads the module, which is why that call must come before any
// stream capture.
attn_status_t scratch_for_current_context(void **out)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return attn::record_cuda_error(e);
    if (!p) return attn::record_cuda_error(cudaErrorInvalidSymbol);
    *out = p;
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
    if ((st = scratch_for_current_context(&scratch))) return st;
    // sdpa_bwd's first kernel rewrites every scratch byte the later kernels
    // read (status word, D, LSE * log2 e, the zeroed dQ accumulator), so what
    // an earlier call left in the array does not matter.
    return sdpa_bwd(desc, q, k, v, o, dO, lse, dQ, dK, dV, scratch, size_t(ATTN_STATIC_SCRATCH_BYTES), stream);
}

extern "C" attn_status_t attn_static_scratch_status(void *stream, uint32_t *device_flags)
{
    if (!device_flags) return ATTN_ERR_NULLPTR;
    void *scratch = nullptr;
    attn_status_t st = scratch_for_current_context(&scratch);
    if (st) return st;
    return attn_query_status(scratch, stream, device_flags);
}
