// selftest.cu -- a check of the device failure path that every tensor-core
// kernel here relies on: a bounded mbarrier wait that runs out sets
// ATTN_DEV_TIMEOUT in the workspace status word and the kernel returns, so the
// context stays usable and the host reads the flag back with
// attn_query_status (the Ascend page "aclnnNsaSelectedAttentionGrad", Return Value, reports
// failures as status codes; this library reports device-side ones the same way).
//
// One block, one thread: it arms an mbarrier that nothing ever completes and
// waits on it with the same bounded wait (sm103::mbar_wait) and the same
// abort path (tc::flag_abort) the backward kernels use.
#include "plan.h"
#include "sm103.cuh"
#include "tc_util.cuh"

namespace attn {

__global__ void selftest_wait_timeout_kernel(uint32_t *status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    sm103::mbar_init(&bar, 1);
    sm103::fence_mbar_init();
    // phase 0 never completes: no thread arrives and no copy is in flight
    if (!sm103::mbar_wait(&bar, 0, &abort_flag, limit_ns)) tc::flag_abort(&abort_flag, status);
}

// Holds its SM for `ns` nanoseconds with `dynamicSmem` bytes of shared memory
// reserved (so a large-footprint kernel cannot share the SM), then exits.
// Touches no memory.
__global__ void selftest_occupy_kernel(uint64_t ns)
{
    extern __shared__ uint8_t occupy_smem[];
    if (threadIdx.x != 0) return;
    const uint64_t t0 = sm103::globaltimer_ns();
    while (sm103::globaltimer_ns() - t0 < ns) __nanosleep(10000);
    if (ns == 0) occupy_smem[0] = 0;  // keeps the allocation referenced
}

}  // namespace attn

extern "C" attn_status_t attn_selftest_occupy(int blocks, size_t smem_bytes, double seconds, void *stream)
{
    using namespace attn;
    if (blocks < 1 || blocks > 4096 || smem_bytes > 200 * 1024 || !(seconds > 0.0) || seconds > 5.0)
        return ATTN_ERR_INVALID;
    cudaError_t e = cudaFuncSetAttribute(selftest_occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem_bytes));
    if (e != cudaSuccess) return record_cuda_error(e);
    selftest_occupy_kernel<<<blocks, 32, smem_bytes, static_cast<cudaStream_t>(stream)>>>(uint64_t(seconds * 1e9));
    return record_cuda_error(cudaGetLastError());
}

extern "C" attn_status_t attn_selftest_wait_timeout(void *workspace, size_t workspace_bytes, double limit_s,
                                                    void *stream)
{
    using namespace attn;
    if (!workspace) return ATTN_ERR_NULLPTR;
    if (workspace_bytes < sizeof(uint32_t) || (reinterpret_cast<uintptr_t>(workspace) & 3u)) return ATTN_ERR_WORKSPACE;
    if (!(limit_s > 0.0) || limit_s > 2.0) return ATTN_ERR_INVALID;  // short waits only
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    selftest_wait_timeout_kernel<<<1, 32, 0, s>>>(static_cast<uint32_t *>(workspace), uint64_t(limit_s * 1e9));
    return record_cuda_error(cudaGetLastError());
}
