// dense.cu -- dense SDPA kernels other than the tensor-core backward:
//   preprocess  (D = rowsum(dO * O), LSE * log2 e, zeroed fp32 dQ accumulator)
//   dq_finalize (dQ = cast(scale * sum of the partial dQ buffers, in index
//                order); chained behind the main kernel)
//
// Definitions: cuDNN-frontend sample "51_scaled_dot_product_attention_backward"
// (FlashAttention-2 backward from the (B,H,S,1) fp32 stats; D, P, dP, dS are
// that algorithm's intermediates), and the Ascend page
// "aclnnNsaSelectedAttentionGrad", Function / Formula, for dQ = scale dS K.
#include <math.h>

#include "plan.h"

namespace attn {

// Element offset of position i of sequence b, head h, in a query-side view.
__device__ __forceinline__ int64_t seq_off(const View &v, const FixedGeo &, int64_t b, int64_t i, int64_t h)
{
    return b * v.sb + h * v.sh + i * v.ss;
}
__device__ __forceinline__ int64_t seq_off(const View &v, const PackedGeo &g, int64_t b, int64_t i, int64_t h)
{
    return h * v.sh + (g.cu_q[b] + i) * v.ss;
}
__device__ __forceinline__ int64_t seq_lse(const DenseArgs &a, const FixedGeo &g, int64_t b, int64_t i, int64_t h)
{
    return (b * a.h + h) * g.s_q + i;
}
__device__ __forceinline__ int64_t seq_lse(const DenseArgs &a, const PackedGeo &g, int64_t b, int64_t i, int64_t h)
{
    return h * a.t_q + g.cu_q[b] + i;
}

// Rows of a preprocess / finalize work unit: half the workspace row alignment,
// so a unit lies within one sequence, each thread has two (d = 64) or four
// (d = 128) rows' loads in flight, and workload-sized grids fit one wave.
constexpr int kUnitRows = int(kWsRowAlign) / 2;

// ------------------------------------------------------------- preprocess
// Work unit = (head, 64 workspace rows); a unit lies within one sequence, so
// it is located once.  d/8 threads per row (8 elements each),
// 256-thread blocks striding over the units in one resident wave.  Covers
// every workspace row: padding rows get LSE2 = +inf (so P = 0) and D = 0.
// Then zeroes every partial dQ buffer (and, in ordered dQ mode, the per-tile
// add counters).  Launched normally (it overwrites what
// the previous call's last kernel reads); lets the main kernel launch behind it.
template <class T, class Geo, int D>
__global__ void __launch_bounds__(256) dense_preprocess_kernel(DenseArgs a, Geo geo)
{
    constexpr int TPR = D / 8, RPP = 256 / TPR, RPT = kUnitRows / RPP;  // rows per pass / per thread
    pdl_trigger();
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0u;
    const int lane_in_row = threadIdx.x % TPR, k0 = threadIdx.x / TPR;
    const int ntile = int(a.t_pad / kUnitRows);
    const int nunit = int(a.h) * ntile;
    for (int u = blockIdx.x; u < nunit; u += gridDim.x) {
        // heads fastest: blocks running together read the same tokens' rows (one DRAM page run)
        const int wt = u / int(a.h), h = u - wt * int(a.h);
        int64_t b = 0, i0 = 0;
        geo.ws_locate(int64_t(wt) * kUnitRows, &b, &i0);
        const int64_t lq = geo.q_len(b);
        const int64_t row0 = int64_t(h) * a.t_pad + int64_t(wt) * kUnitRows;
        uint4 ov[RPT], dv[RPT];  // all loads of this thread first
        float lse[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int64_t i = i0 + k0 + r * RPP;
            ov[r] = dv[r] = make_uint4(0, 0, 0, 0);
            lse[r] = 0.f;
            if (i < lq) {
                ov[r] = *reinterpret_cast<const uint4 *>(static_cast<const T *>(a.o.ptr) + seq_off(a.o, geo, b, i, h) +
                                                         lane_in_row * 8);
                dv[r] = *reinterpret_cast<const uint4 *>(static_cast<const T *>(a.dO.ptr) + seq_off(a.dO, geo, b, i, h) +
                                                         lane_in_row * 8);
                if (lane_in_row == 0) lse[r] = a.lse[seq_lse(a, geo, b, i, h)];
            }
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int k = k0 + r * RPP;
            const bool real = i0 + k < lq;
            const uint32_t *op = &ov[r].x, *dp = &dv[r].x;
            float dsum = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float2 of = unpack2<T>(op[e]), df = unpack2<T>(dp[e]);
                dsum += of.x * df.x + of.y * df.y;
            }
#pragma unroll
            for (int off = TPR / 2; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
            if (lane_in_row == 0) {
                a.dvec[row0 + k] = real ? dsum : 0.f;
                a.lse2[row0 + k] = real ? lse[r] * kLog2e : INFINITY;
            }
        }
    }
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 *acc = reinterpret_cast<float4 *>(a.dqacc);
    const int64_t n4 = int64_t(a.n_part) * a.h * a.t_pad * D / 4;
    for (int64_t k = int64_t(blockIdx.x) * 256 + threadIdx.x; k < n4; k += int64_t(gridDim.x) * 256) acc[k] = z;
    if (a.ordered)  // no query tile has received an add yet
        for (int64_t k = int64_t(blockIdx.x) * 256 + threadIdx.x; k < a.h * a.sem_stride; k += int64_t(gridDim.x) * 256)
            a.sem[k] = 0u;
}

// ------------------------------------------------------------ dq finalize
// dQ = cast(scale * sum over the partial buffers, in index order).  Same
// units as the preprocess; launched behind the main kernel and waits for it.
template <class T, class Geo, int D>
__global__ void __launch_bounds__(256) dq_finalize_kernel(DenseArgs a, Geo geo)
{
    constexpr int TPR = D / 8, RPP = 256 / TPR, RPT = kUnitRows / RPP;
    const int lane_in_row = threadIdx.x % TPR, k0 = threadIdx.x / TPR;
    const int ntile = int(a.t_pad / kUnitRows);
    const int nunit = int(a.h) * ntile;
    const int64_t part_stride = a.h * a.t_pad * D;
    pdl_wait();
    for (int u = blockIdx.x; u < nunit; u += gridDim.x) {
        // heads fastest: blocks running together read the same tokens' rows (one DRAM page run)
        const int wt = u / int(a.h), h = u - wt * int(a.h);
        int64_t b = 0, i0 = 0;
        geo.ws_locate(int64_t(wt) * kUnitRows, &b, &i0);
        const int64_t lq = geo.q_len(b);
        const int64_t row0 = int64_t(h) * a.t_pad + int64_t(wt) * kUnitRows;
        float acc[RPT][8];
#pragma unroll
        for (int r = 0; r < RPT; ++r)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[r][e] = 0.f;
        for (int p = 0; p < a.n_part; ++p) {  // fixed order: bitwise reproducible
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const float4 *src = reinterpret_cast<const float4 *>(a.dqacc + p * part_stride +
                                                                     (row0 + k0 + r * RPP) * D + lane_in_row * 8);
                const float4 x0 = src[0], x1 = src[1];
                acc[r][0] += x0.x; acc[r][1] += x0.y; acc[r][2] += x0.z; acc[r][3] += x0.w;
                acc[r][4] += x1.x; acc[r][5] += x1.y; acc[r][6] += x1.z; acc[r][7] += x1.w;
            }
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int64_t i = i0 + k0 + r * RPP;
            if (i >= lq) continue;
            uint4 out;
            out.x = pack2<T>(acc[r][0] * a.scale, acc[r][1] * a.scale);
            out.y = pack2<T>(acc[r][2] * a.scale, acc[r][3] * a.scale);
            out.z = pack2<T>(acc[r][4] * a.scale, acc[r][5] * a.scale);
            out.w = pack2<T>(acc[r][6] * a.scale, acc[r][7] * a.scale);
            *reinterpret_cast<uint4 *>(static_cast<T *>(a.dQ.ptr) + seq_off(a.dQ, geo, b, i, h) + lane_in_row * 8) = out;
        }
    }
}

// ------------------------------------------------------------- launchers
namespace {

// One wave of 256-thread blocks (8 per SM), or fewer when there are fewer rows.
unsigned row_grid(const DenseArgs &a)
{
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0)
            sms = 1;
    }
    const int64_t need = a.h * (a.t_pad / kUnitRows);  // (head, 32-row) units
    const int64_t wave = int64_t(sms) * 8;
    return unsigned(need < 1 ? 1 : (need < wave ? need : wave));
}

template <class Geo> cudaError_t preprocess(const DenseArgs &a, const Geo &g, cudaStream_t s)
{
    const dim3 grid(row_grid(a));
    if (a.d == 64)
        return a.dtype == ATTN_F16
                   ? launch_kernel(dense_preprocess_kernel<__half, Geo, 64>, grid, 256, 0, s, false, a, g)
                   : launch_kernel(dense_preprocess_kernel<__nv_bfloat16, Geo, 64>, grid, 256, 0, s, false, a, g);
    return a.dtype == ATTN_F16 ? launch_kernel(dense_preprocess_kernel<__half, Geo, 128>, grid, 256, 0, s, false, a, g)
                               : launch_kernel(dense_preprocess_kernel<__nv_bfloat16, Geo, 128>, grid, 256, 0, s, false, a, g);
}

template <class Geo> cudaError_t finalize(const DenseArgs &a, const Geo &g, cudaStream_t s)
{
    if (a.t_q == 0) return cudaSuccess;
    const dim3 grid(row_grid(a));
    if (a.d == 64)
        return a.dtype == ATTN_F16 ? launch_kernel(dq_finalize_kernel<__half, Geo, 64>, grid, 256, 0, s, true, a, g)
                                   : launch_kernel(dq_finalize_kernel<__nv_bfloat16, Geo, 64>, grid, 256, 0, s, true, a, g);
    return a.dtype == ATTN_F16 ? launch_kernel(dq_finalize_kernel<__half, Geo, 128>, grid, 256, 0, s, true, a, g)
                               : launch_kernel(dq_finalize_kernel<__nv_bfloat16, Geo, 128>, grid, 256, 0, s, true, a, g);
}

}  // namespace

cudaError_t launch_dense_preprocess(const DenseArgs &a, const FixedGeo &g, cudaStream_t s) { return preprocess(a, g, s); }
cudaError_t launch_dense_preprocess(const DenseArgs &a, const PackedGeo &g, cudaStream_t s) { return preprocess(a, g, s); }
cudaError_t launch_dq_finalize(const DenseArgs &a, const FixedGeo &g, cudaStream_t s) { return finalize(a, g, s); }
cudaError_t launch_dq_finalize(const DenseArgs &a, const PackedGeo &g, cudaStream_t s) { return finalize(a, g, s); }

}  // namespace attn
