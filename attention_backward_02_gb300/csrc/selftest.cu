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

}  // namespace attn

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
