// dense.cu -- dense SDPA kernels other than the tensor-core backward:
//   preprocess  (D = rowsum(dO * O), LSE * log2 e, zeroed fp32 dQ accumulator)
//   dq_finalize (dQ = cast(scale * sum of the partial dQ buffers, in index
//                order); chained behind the main kernel)
//   fwd         (O and LSE; CUDA-core kernel, not on the timed path)
//
// Definitions: cuDNN-frontend sample "51_scaled_dot_product_attention_backward"
// (FlashAttention-2 backward from the (B,H,S,1) fp32 stats; D, P, dP, dS are
// that algorithm's intermediates), and the Ascend page
// "aclnnNsaSelectedAttentionGrad", Function / Formula, for dQ = scale dS K.
#include <math.h>

#include "plan.h"

namespace attn {

// Element offset of token t (packed index space) of head h in a view.
__device__ __forceinline__ int64_t tok_off(const View &v, const FixedGeo &g, int64_t t, int64_t h)
{
    int64_t b = t / g.s_q, i = t - b * g.s_q;
    return b * v.sb + h * v.sh + i * v.ss;
}
__device__ __forceinline__ int64_t tok_off(const View &v, const PackedGeo &, int64_t t, int64_t h)
{
    return h * v.sh + t * v.ss;
}
__device__ __forceinline__ int64_t kv_off(const View &v, const FixedGeo &g, int64_t t, int64_t h)
{
    int64_t b = t / g.s_kv, i = t - b * g.s_kv;
    return b * v.sb + h * v.sh + i * v.ss;
}
__device__ __forceinline__ int64_t kv_off(const View &v, const PackedGeo &, int64_t t, int64_t h)
{
    return h * v.sh + t * v.ss;
}
// Caller's stats layout: [B][h][s_q] (fixed) or [h][T_q] (packed).
__device__ __forceinline__ int64_t lse_index(const DenseArgs &a, const FixedGeo &g, int64_t t, int64_t h)
{
    int64_t b = t / g.s_q, i = t - b * g.s_q;
    return (b * a.h + h) * g.s_q + i;
}
__device__ __forceinline__ int64_t lse_index(const DenseArgs &a, const PackedGeo &, int64_t t, int64_t h)
{
    return h * a.t_q + t;
}

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

// Rows of a preprocess / finalize work unit: a quarter of the workspace row
// alignment, so a unit lies within one sequence and the grid has enough blocks.
constexpr int kUnitRows = int(kWsRowAlign) / 4;

// ------------------------------------------------------------- preprocess
// Work unit = (head, 32 workspace rows); a unit lies within one sequence, so
// it is located once.  d/8 threads per row (8 elements each),
// 256-thread blocks striding over the units in one resident wave.  Covers
// every workspace row: padding rows get LSE2 = +inf (so P = 0) and D = 0.
// Then zeroes every partial dQ buffer.  Launched normally (it overwrites what
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

// ------------------------------------------------------------- forward
// CUDA-core forward, two passes over the keys: (1) row max and sum of
// exp2, (2) O = sum P V with the final LSE.  One CTA per (32-row query
// tile, query head, sequence), 256 threads.
template <class T, class Geo, int D>
__global__ void __launch_bounds__(256) dense_fwd_kernel(DenseArgs a, Geo geo)
{
    constexpr int BM = 32, BN = 32, LD = D + 1;
    extern __shared__ float fwd_smem[];
    float(*Qs)[LD] = reinterpret_cast<float(*)[LD]>(fwd_smem);
    float(*Ks)[LD] = reinterpret_cast<float(*)[LD]>(fwd_smem + BM * LD);
    float(*Vs)[LD] = reinterpret_cast<float(*)[LD]>(fwd_smem + (BM + BN) * LD);
    float(*Ss)[BN + 1] = reinterpret_cast<float(*)[BN + 1]>(fwd_smem + (BM + 2 * BN) * LD);
    float *row_m = fwd_smem + (BM + 2 * BN) * LD + BM * (BN + 1);
    float *row_l = row_m + BM;
    const int64_t b = blockIdx.z, hq = blockIdx.y, g = hq / (a.h / a.h_kv);
    const int64_t lq = geo.q_len(b), lkv = geo.kv_len(b);
    const int64_t i0 = int64_t(blockIdx.x) * BM;
    if (i0 >= lq) return;
    const int64_t q0 = geo.q_start(b), k0 = geo.kv_start(b);
    const int tid = threadIdx.x;
    const float c = a.scale * kLog2e;
    const T *Q = static_cast<const T *>(a.q.ptr);
    const T *K = static_cast<const T *>(a.k.ptr);
    const T *V = static_cast<const T *>(a.v.ptr);

    for (int e = tid; e < BM * D; e += 256) {
        int r = e / D, x = e % D;
        Qs[r][x] = (i0 + r < lq) ? to_f32(Q[tok_off(a.q, geo, q0 + i0 + r, hq) + x]) : 0.f;
    }
    if (tid < BM) { row_m[tid] = -INFINITY; row_l[tid] = 0.f; }
    const int64_t i_last = (i0 + BM - 1 < lq - 1) ? i0 + BM - 1 : lq - 1;
    const int64_t j_end = last_visible_key(a.mask, i_last, lq, lkv) + 1;  // keys beyond are masked for all rows

    const int r = tid / 8, part = tid % 8;  // row r, 4 columns / (D/8) features per thread
    float o_acc[D / 8];
    for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
        for (int e = 0; e < D / 8; ++e) o_acc[e] = 0.f;
        for (int64_t j0 = 0; j0 < j_end; j0 += BN) {
            __syncthreads();
            for (int e = tid; e < BN * D; e += 256) {
                int rr = e / D, x = e % D;
                bool in = j0 + rr < lkv;
                Ks[rr][x] = in ? to_f32(K[kv_off(a.k, geo, k0 + j0 + rr, g) + x]) : 0.f;
                Vs[rr][x] = in ? to_f32(V[kv_off(a.v, geo, k0 + j0 + rr, g) + x]) : 0.f;
            }
            __syncthreads();
            for (int cc = part; cc < BN; cc += 8) {
                float s = 0.f;
#pragma unroll 8
                for (int x = 0; x < D; ++x) s += Qs[r][x] * Ks[cc][x];
                bool vis = (i0 + r < lq) && (j0 + cc < lkv) && visible(a.mask, i0 + r, j0 + cc, lq, lkv);
                Ss[r][cc] = vis ? s * c : -INFINITY;
            }
            __syncthreads();
            if (pass == 0) {
                float m = -INFINITY;
                for (int cc = part; cc < BN; cc += 8) m = fmaxf(m, Ss[r][cc]);
                for (int off = 4; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                float m_new = fmaxf(row_m[r], m);
                float l = 0.f;
                if (m_new != -INFINITY)
                    for (int cc = part; cc < BN; cc += 8) l += exp2f(Ss[r][cc] - m_new);
                for (int off = 4; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
                __syncwarp();
                if (part == 0) {
                    float l_old = row_m[r] == -INFINITY ? 0.f : row_l[r] * exp2f(row_m[r] - m_new);
                    row_l[r] = l_old + l;
                    row_m[r] = m_new;
                }
            } else {
                const float lse2 = row_m[r] == -INFINITY ? INFINITY : row_m[r] + log2f(row_l[r]);
                for (int cc = 0; cc < BN; ++cc) {
                    float p = (lse2 == INFINITY) ? 0.f : exp2f(Ss[r][cc] - lse2);
#pragma unroll
                    for (int e = 0; e < D / 8; ++e) o_acc[e] += p * Vs[cc][part * (D / 8) + e];
                }
            }
        }
        __syncthreads();
    }
    if (i0 + r < lq) {
        T *O = static_cast<T *>(a.o.ptr);
        int64_t off = tok_off(a.o, geo, q0 + i0 + r, hq) + part * (D / 8);
#pragma unroll
        for (int e = 0; e < D / 8; ++e) O[off + e] = from_f32<T>(o_acc[e]);
        if (part == 0) {
            float lse = row_m[r] == -INFINITY ? INFINITY : (row_m[r] + log2f(row_l[r])) / kLog2e;
            int64_t idx = a.packed ? hq * a.t_q + (q0 + i0 + r) : (b * a.h + hq) * lq + (i0 + r);
            a.lse_out[idx] = lse;
        }
    }
}

// ------------------------------------------------------------- launchers
namespace {

template <class Geo> int64_t max_len_q(const DenseArgs &a, const Geo &g);
template <> int64_t max_len_q(const DenseArgs &, const FixedGeo &g) { return g.s_q; }
template <> int64_t max_len_q(const DenseArgs &, const PackedGeo &g)
{
    int64_t m = 0;
    for (int64_t b = 0; b < g.nseq; ++b) m = g.q_len(b) > m ? g.q_len(b) : m;
    return m;
}

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

template <class T, class Geo, int D> cudaError_t fwd_run(const DenseArgs &a, const Geo &g, dim3 grid, cudaStream_t s)
{
    constexpr int BM = 32, BN = 32, LD = D + 1;
    const size_t smem = sizeof(float) * ((BM + 2 * BN) * LD + BM * (BN + 1) + 2 * BM);
    auto k = dense_fwd_kernel<T, Geo, D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    k<<<grid, 256, smem, s>>>(a, g);
    return cudaGetLastError();
}

template <class Geo> cudaError_t fwd(const DenseArgs &a, const Geo &g, cudaStream_t s)
{
    int64_t ml = max_len_q(a, g);
    if (ml == 0) return cudaSuccess;
    dim3 grid(unsigned((ml + 31) / 32), unsigned(a.h), unsigned(g.nseq));
    if (a.d == 64)
        return a.dtype == ATTN_F16 ? fwd_run<__half, Geo, 64>(a, g, grid, s) : fwd_run<__nv_bfloat16, Geo, 64>(a, g, grid, s);
    return a.dtype == ATTN_F16 ? fwd_run<__half, Geo, 128>(a, g, grid, s) : fwd_run<__nv_bfloat16, Geo, 128>(a, g, grid, s);
}

}  // namespace

cudaError_t launch_dense_preprocess(const DenseArgs &a, const FixedGeo &g, cudaStream_t s) { return preprocess(a, g, s); }
cudaError_t launch_dense_preprocess(const DenseArgs &a, const PackedGeo &g, cudaStream_t s) { return preprocess(a, g, s); }
cudaError_t launch_dq_finalize(const DenseArgs &a, const FixedGeo &g, cudaStream_t s) { return finalize(a, g, s); }
cudaError_t launch_dq_finalize(const DenseArgs &a, const PackedGeo &g, cudaStream_t s) { return finalize(a, g, s); }
cudaError_t launch_dense_fwd(const DenseArgs &a, const FixedGeo &g, cudaStream_t s) { return fwd(a, g, s); }
cudaError_t launch_dense_fwd(const DenseArgs &a, const PackedGeo &g, cudaStream_t s) { return fwd(a, g, s); }

}  // namespace attn
