// bwd_simt.cu -- CUDA-core dense backward (FlashAttention-2 form).
//
// One CTA per (key tile of 32 rows, kv head, sequence); in deterministic mode
// one CTA per (split, kv head, sequence) that walks the key tiles
// j = split, split + n_part, ... in order and is the only writer of partial
// dQ buffer `split`.  Inside, the CTA loops over the query heads of its
// group and the query tiles that see the key tile:
//   S = scale Q K^T, P = exp2(S log2 e - LSE log2 e), dP = dO V^T,
//   dS = P (dP - D), dV += P^T dO, dK += dS^T Q, dQ += dS K (fp32 reduce).
// All arithmetic is fp32.  Formulas: cuDNN-frontend SDPA-backward sample
// (FlashAttention-2) and the Ascend aclnnNsaSelectedAttentionGrad page,
// Function / Formula.
#include <math.h>

#include "plan.h"

namespace attn {

namespace {
__device__ __forceinline__ int64_t off_q(const View &v, const FixedGeo &g, int64_t b, int64_t i, int64_t h)
{
    return b * v.sb + h * v.sh + i * v.ss;
}
__device__ __forceinline__ int64_t off_q(const View &v, const PackedGeo &g, int64_t b, int64_t i, int64_t h)
{
    return h * v.sh + (g.cu_q[b] + i) * v.ss;
}
__device__ __forceinline__ int64_t off_kv(const View &v, const FixedGeo &g, int64_t b, int64_t j, int64_t h)
{
    return b * v.sb + h * v.sh + j * v.ss;
}
__device__ __forceinline__ int64_t off_kv(const View &v, const PackedGeo &g, int64_t b, int64_t j, int64_t h)
{
    return h * v.sh + (g.cu_kv[b] + j) * v.ss;
}
}  // namespace

template <class T, class Geo, int D>
__global__ void __launch_bounds__(256) dense_bwd_simt_kernel(DenseArgs a, Geo geo)
{
    constexpr int BM = 32, BN = 32, LD = D + 1, F = D / 8;
    extern __shared__ float smem[];
    float(*Ks)[LD] = reinterpret_cast<float(*)[LD]>(smem);
    float(*Vs)[LD] = reinterpret_cast<float(*)[LD]>(smem + BN * LD);
    float(*Qs)[LD] = reinterpret_cast<float(*)[LD]>(smem + 2 * BN * LD);
    float(*dOs)[LD] = reinterpret_cast<float(*)[LD]>(smem + 2 * BN * LD + BM * LD);
    float(*Ps)[BM + 1] = reinterpret_cast<float(*)[BM + 1]>(smem + 2 * BN * LD + 2 * BM * LD);
    float(*dSs)[BM + 1] = reinterpret_cast<float(*)[BM + 1]>(smem + 2 * BN * LD + 2 * BM * LD + BN * (BM + 1));
    float *lse_s = smem + 2 * BN * LD + 2 * BM * LD + 2 * BN * (BM + 1);
    float *d_s = lse_s + BM;

    const int64_t b = blockIdx.z, g = blockIdx.y, G = a.h / a.h_kv;
    const int64_t lq = geo.q_len(b), lkv = geo.kv_len(b);
    const int64_t ntiles = (lkv + BN - 1) / BN;
    const int64_t q0 = geo.q_start(b);
    const int tid = threadIdx.x;
    const float c = a.scale * kLog2e;
    const T *Q = static_cast<const T *>(a.q.ptr);
    const T *K = static_cast<const T *>(a.k.ptr);
    const T *V = static_cast<const T *>(a.v.ptr);
    const T *dO = static_cast<const T *>(a.dO.ptr);
    const int64_t step = a.deterministic ? a.n_part : ntiles;
    const int64_t part = a.deterministic ? blockIdx.x : 0;
    float *dqacc = a.dqacc + part * a.h * a.t_pad * a.d;

    for (int64_t jt = blockIdx.x; jt < ntiles; jt += step) {
        const int64_t j0 = jt * BN;
        __syncthreads();
        for (int e = tid; e < BN * D; e += 256) {
            int r = e / D, x = e % D;
            bool in = j0 + r < lkv;
            Ks[r][x] = in ? to_f32(K[off_kv(a.k, geo, b, j0 + r, g) + x]) : 0.f;
            Vs[r][x] = in ? to_f32(V[off_kv(a.v, geo, b, j0 + r, g) + x]) : 0.f;
        }
        const int rr = tid / 8, x0 = (tid % 8) * F;  // owner of dK/dV row rr, features x0..x0+F
        float dk[F], dv[F];
#pragma unroll
        for (int e = 0; e < F; ++e) dk[e] = dv[e] = 0.f;
        const int64_t i_lo = first_query_seeing(a.mask, j0, lq, lkv);
        for (int64_t hq = g * G; hq < (g + 1) * G; ++hq) {
            for (int64_t i0 = (i_lo / BM) * BM; i0 < lq; i0 += BM) {
                __syncthreads();
                for (int e = tid; e < BM * D; e += 256) {
                    int r = e / D, x = e % D;
                    bool in = i0 + r < lq;
                    Qs[r][x] = in ? to_f32(Q[off_q(a.q, geo, b, i0 + r, hq) + x]) : 0.f;
                    dOs[r][x] = in ? to_f32(dO[off_q(a.dO, geo, b, i0 + r, hq) + x]) : 0.f;
                }
                if (tid < BM) {
                    int64_t row = hq * a.t_pad + q0 + i0 + tid;
                    lse_s[tid] = a.lse2[row];
                    d_s[tid] = a.dvec[row];
                }
                __syncthreads();
                for (int e = tid; e < BN * BM; e += 256) {
                    int r = e / BM, cq = e % BM;  // key row r, query column cq
                    bool vis = (j0 + r < lkv) && (i0 + cq < lq) && visible(a.mask, i0 + cq, j0 + r, lq, lkv);
                    float s = 0.f, dp = 0.f;
                    if (vis) {
#pragma unroll 8
                        for (int x = 0; x < D; ++x) {
                            s += Ks[r][x] * Qs[cq][x];
                            dp += Vs[r][x] * dOs[cq][x];
                        }
                    }
                    float p = vis ? exp2f(s * c - lse_s[cq]) : 0.f;
                    Ps[r][cq] = p;
                    dSs[r][cq] = vis ? p * (dp - d_s[cq]) : 0.f;
                }
                __syncthreads();
                for (int cq = 0; cq < BM; ++cq) {
                    float p = Ps[rr][cq], ds = dSs[rr][cq];
#pragma unroll
                    for (int e = 0; e < F; ++e) {
                        dv[e] += p * dOs[cq][x0 + e];
                        dk[e] += ds * Qs[cq][x0 + e];
                    }
                }
                // dQ rows of this query tile: thread owns query row rr, features x0..
                if (i0 + rr < lq) {
                    float dq[F];
#pragma unroll
                    for (int e = 0; e < F; ++e) dq[e] = 0.f;
                    for (int r = 0; r < BN; ++r) {
                        float ds = dSs[r][rr];
#pragma unroll
                        for (int e = 0; e < F; ++e) dq[e] += ds * Ks[r][x0 + e];
                    }
                    float *dst = dqacc + (hq * a.t_pad + q0 + i0 + rr) * a.d + x0;
#pragma unroll
                    for (int e = 0; e < F; ++e) {
                        if (a.deterministic) dst[e] += dq[e];
                        else atomicAdd(dst + e, dq[e]);
                    }
                }
            }
        }
        if (j0 + rr < lkv) {
            T *dK = static_cast<T *>(a.dK.ptr);
            T *dV = static_cast<T *>(a.dV.ptr);
            int64_t ok = off_kv(a.dK, geo, b, j0 + rr, g) + x0, ov = off_kv(a.dV, geo, b, j0 + rr, g) + x0;
#pragma unroll
            for (int e = 0; e < F; ++e) {
                dK[ok + e] = from_f32<T>(dk[e] * a.scale);
                dV[ov + e] = from_f32<T>(dv[e]);
            }
        }
    }
}

namespace {
template <class Geo> int64_t max_len_kv(const Geo &g);
template <> int64_t max_len_kv(const FixedGeo &g) { return g.s_kv; }
template <> int64_t max_len_kv(const PackedGeo &g)
{
    int64_t m = 0;
    for (int64_t b = 0; b < g.nseq; ++b) m = g.kv_len(b) > m ? g.kv_len(b) : m;
    return m;
}

template <class T, class Geo, int D> cudaError_t run(const DenseArgs &a, const Geo &g, cudaStream_t s)
{
    constexpr int BM = 32, BN = 32, LD = D + 1;
    size_t smem = sizeof(float) * (2 * BN * LD + 2 * BM * LD + 2 * BN * (BM + 1) + 2 * BM);
    auto k = dense_bwd_simt_kernel<T, Geo, D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    int64_t ntiles = (max_len_kv(g) + BN - 1) / BN;
    if (ntiles == 0) return cudaSuccess;
    dim3 grid(unsigned(a.deterministic ? a.n_part : ntiles), unsigned(a.h_kv), unsigned(g.nseq));
    k<<<grid, 256, smem, s>>>(a, g);
    return cudaGetLastError();
}

template <class Geo> cudaError_t dispatch(const DenseArgs &a, const Geo &g, cudaStream_t s)
{
    if (a.d == 64)
        return a.dtype == ATTN_F16 ? run<__half, Geo, 64>(a, g, s) : run<__nv_bfloat16, Geo, 64>(a, g, s);
    return a.dtype == ATTN_F16 ? run<__half, Geo, 128>(a, g, s) : run<__nv_bfloat16, Geo, 128>(a, g, s);
}
}  // namespace

cudaError_t launch_dense_bwd_main(const DenseArgs &a, const FixedGeo &g, cudaStream_t s) { return dispatch(a, g, s); }
cudaError_t launch_dense_bwd_main(const DenseArgs &a, const PackedGeo &g, cudaStream_t s) { return dispatch(a, g, s); }

}  // namespace attn
