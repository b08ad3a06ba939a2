// tc_util.cuh -- small device helpers shared by the tensor-core kernels:
// fast exp2, shared-memory vector accesses, named-barrier reductions, the
// 128-byte-swizzle descriptors for K-major and MN-major operand tiles, and
// the packed P / dS computation.
#pragma once

#include "common.cuh"
#include "sm103.cuh"

namespace attn {
namespace tc {
using namespace sm103;

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// P = exp2(x) and dS = P (dP - D) for two adjacent columns, packed as two
// 16-bit values each (low half = first column).  x = S scale log2 e - LSE
// log2 e (-inf where masked), g = dP - D.  fp16: the two exponentials run as
// one f16x2 MUFU operation and dS as one f16x2 multiply, at the precision P
// and dS are rounded to anyway.  bf16: fp32 exponentials and products,
// rounded once.
template <class T> __device__ __forceinline__ uint32_t p_and_ds(float x0, float x1, float g0, float g1, uint32_t *ds);
template <> __device__ __forceinline__ uint32_t p_and_ds<__half>(float x0, float x1, float g0, float g1, uint32_t *ds)
{
    const uint32_t xh = pack2<__half>(x0, x1), gh = pack2<__half>(g0, g1);
    uint32_t ph, dh;
    asm("ex2.approx.f16x2 %0, %1;" : "=r"(ph) : "r"(xh));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(dh) : "r"(ph), "r"(gh));
    *ds = dh;
    return ph;
}
template <>
__device__ __forceinline__ uint32_t p_and_ds<__nv_bfloat16>(float x0, float x1, float g0, float g1, uint32_t *ds)
{
    const float p0 = ex2(x0), p1 = ex2(x1);
    *ds = pack2<__nv_bfloat16>(p0 * g0, p1 * g1);
    return pack2<__nv_bfloat16>(p0, p1);
}

// AND of `pred` over the threads of named barrier `id` (also a barrier).
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t nthreads, bool pred)
{
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %3, 0;\n\t"
        "bar.red.and.pred q, %1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"(id), "r"(nthreads), "r"(uint32_t(pred))
        : "memory");
    return out != 0;
}

// K-major SW128 tile of `rows` rows stored in 64-column blocks; K step kk (16 elements).
__device__ __forceinline__ uint64_t desc_kmaj(uint32_t base, uint32_t rows, int kk)
{
    return smem_desc_sw128(base + uint32_t(kk >> 2) * rows * 128u + uint32_t(kk & 3) * 32u, 16, 1024);
}

// MN-major SW128 tile whose rows are the K dimension (`krows` of them) and
// whose 64-column blocks run along M/N; K step kk (16 rows).
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, uint32_t krows, int kk)
{
    return smem_desc_sw128(base + uint32_t(kk) * 2048u, krows * 128u, 1024);
}

// The same descriptors advanced to K step kk from their step-0 value: only
// the start-address field (address >> 4, 14 bits, no carry for shared
// memory addresses) changes, so a step is one add.
__device__ __forceinline__ uint64_t kmaj_step(uint64_t d0, uint32_t rows, int kk)
{
    return d0 + uint64_t((uint32_t(kk >> 2) * rows * 128u + uint32_t(kk & 3) * 32u) >> 4);
}
__device__ __forceinline__ uint64_t mn_step(uint64_t d0, int kk) { return d0 + uint64_t(uint32_t(kk) * 128u); }

__device__ __forceinline__ void flag_abort(volatile int *abort, uint32_t *status)
{
    *abort = 1;
    raise_flag(status, ATTN_DEV_TIMEOUT);
}

}  // namespace tc
}  // namespace attn
