// common.cuh -- types and small device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attnbwd.h"

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSeq = 256;  // sequences a packed (varlen) call may hold

// ---------------------------------------------------------------- 16-bit I/O
template <class T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <class T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// two floats -> packed pair of 16-bit values (low half = a), round to nearest even
template <class T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b)
{
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// packed pair -> two floats
template <class T> __device__ __forceinline__ float2 unpack2(uint32_t u);
template <> __device__ __forceinline__ float2 unpack2<__half>(uint32_t u)
{
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(h);
}
template <> __device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t u)
{
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(h);
}

// ------------------------------------------------------- sequence geometry
// A fixed-length batch: sequence b covers query rows [b*s_q, (b+1)*s_q) of the
// token-major index space.  Packed: starts from inclusive cumulative lengths.
// Workspace rows (per-query-row stats and the fp32 dQ accumulator) give
// every sequence a run of rows rounded up to a multiple of kWsRowAlign, so a
// query tile never straddles two sequences there and every tile starts on a
// 256-byte boundary.
constexpr int64_t kWsRowAlign = 128;
__host__ __device__ constexpr int64_t ws_round(int64_t n) { return (n + kWsRowAlign - 1) / kWsRowAlign * kWsRowAlign; }

struct FixedGeo {
    int64_t nseq, s_q, s_kv;
    __host__ __device__ int64_t q_start(int64_t b) const { return b * s_q; }
    __host__ __device__ int64_t kv_start(int64_t b) const { return b * s_kv; }
    __host__ __device__ int64_t q_len(int64_t) const { return s_q; }
    __host__ __device__ int64_t kv_len(int64_t) const { return s_kv; }
    __host__ __device__ int64_t ws_start(int64_t b) const { return b * ws_round(s_q); }
    __host__ __device__ int64_t ws_rows() const { return nseq * ws_round(s_q); }
    // workspace row -> (sequence, position); false on padding rows
    __host__ __device__ bool ws_locate(int64_t r, int64_t *b, int64_t *i) const
    {
        const int64_t per = ws_round(s_q);
        *b = r / per;
        *i = r - *b * per;
        return *i < s_q;
    }
};

struct PackedGeo {
    int64_t nseq;
    int64_t cu_q[kMaxSeq + 1];   // cu_q[0] = 0, cu_q[b+1] = end of sequence b
    int64_t cu_kv[kMaxSeq + 1];
    int64_t ws_q[kMaxSeq + 1];   // first workspace row of sequence b; ws_q[nseq] = total
    __host__ __device__ int64_t q_start(int64_t b) const { return cu_q[b]; }
    __host__ __device__ int64_t kv_start(int64_t b) const { return cu_kv[b]; }
    __host__ __device__ int64_t q_len(int64_t b) const { return cu_q[b + 1] - cu_q[b]; }
    __host__ __device__ int64_t kv_len(int64_t b) const { return cu_kv[b + 1] - cu_kv[b]; }
    __host__ __device__ int64_t ws_start(int64_t b) const { return ws_q[b]; }
    __host__ __device__ int64_t ws_rows() const { return ws_q[nseq]; }
    __host__ __device__ bool ws_locate(int64_t r, int64_t *b, int64_t *i) const
    {
        int64_t lo = 0, hi = nseq - 1;  // last b with ws_q[b] <= r
        while (lo < hi) {
            int64_t mid = (lo + hi + 1) / 2;
            if (ws_q[mid] <= r) lo = mid;
            else hi = mid - 1;
        }
        *b = lo;
        *i = r - ws_q[lo];
        return *i < q_len(lo);
    }
};

// Visibility of key j to query i (both local to their sequence).
__host__ __device__ __forceinline__ bool visible(int mask, int64_t i, int64_t j, int64_t lq, int64_t lkv)
{
    if (mask == ATTN_CAUSAL_TOP_LEFT) return j <= i;
    if (mask == ATTN_CAUSAL_BOTTOM_RIGHT) return j <= i + (lkv - lq);
    return true;
}

// Largest key index visible to query i, or lkv-1 with no mask (may be < 0).
__host__ __device__ __forceinline__ int64_t last_visible_key(int mask, int64_t i, int64_t lq, int64_t lkv)
{
    if (mask == ATTN_CAUSAL_TOP_LEFT) return i < lkv - 1 ? i : lkv - 1;
    if (mask == ATTN_CAUSAL_BOTTOM_RIGHT) {
        int64_t j = i + (lkv - lq);
        return j < lkv - 1 ? j : lkv - 1;
    }
    return lkv - 1;
}

// First query that sees key j (queries before it see nothing of column j).
__host__ __device__ __forceinline__ int64_t first_query_seeing(int mask, int64_t j, int64_t lq, int64_t lkv)
{
    if (mask == ATTN_CAUSAL_TOP_LEFT) return j;
    if (mask == ATTN_CAUSAL_BOTTOM_RIGHT) {
        int64_t i = j - (lkv - lq);
        return i > 0 ? i : 0;
    }
    return 0;
}

// ------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may start while
// the previous kernel of the stream still runs; it must wait here before it
// touches anything that kernel writes.  (A no-op for an ordinary launch.)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel of the stream start launching (its blocks then wait
// in pdl_wait until this grid has completed).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launches k on stream s, optionally with programmatic stream serialization
// and optionally as a cooperative launch (all blocks resident at once, or
// the launch fails).
template <class... KArgs, class... Args>
inline cudaError_t launch_kernel_ex(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                                    bool coop, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n++].val.programmaticStreamSerializationAllowed = 1;
    }
    if (coop) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n++].val.cooperative = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, k, static_cast<Args &&>(args)...);
}

template <class... KArgs, class... Args>
inline cudaError_t launch_kernel(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                                 Args &&...args)
{
    return launch_kernel_ex(k, grid, block, smem, s, pdl, false, static_cast<Args &&>(args)...);
}

// ----------------------------------------------------------- status word
__device__ __forceinline__ void raise_flag(uint32_t *status, uint32_t bit)
{
    if (status) atomicOr(status, bit);
}

}  // namespace attn
