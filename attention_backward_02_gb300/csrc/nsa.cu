// nsa.cu -- NSA selected-attention backward (Ascend CANN page
// "aclnnNsaSelectedAttentionGrad", Function / Formula):
//   selectedKey = Gather(key, topkIndices), selectedValue = Gather(value, ...)
//   then the attention backward on the gathered rows, with dK / dV of every
//   gathered row added back to the key / value row it came from.
//
// Kernels:
//   nsa_init         zeroes the status word and the block bitmap
//   preprocess       LSE2 = (softmaxMax + ln softmaxSum) * log2 e (lane 0 of the
//                    8-wide stats), D = rowsum(dO * O); zeroes the dK/dV and
//                    (tensor-core path) dQ accumulators.  It runs as extra blocks
//                    of the emit launch, without waiting, so it overlaps the
//                    block-list kernels.
// The kernels after init are chained with programmatic dependent launch: each
// waits for its predecessor on entry (the preprocess blocks excepted).
//   block lists      per (sequence, kv head, block): ascending list of the
//                    tokens that selected the block and see at least one of
//                    its keys (bitmap -> count -> scan -> ordered emit), with
//                    validation of every index (range, duplicates)
//   nsa_bwd_simt     CUDA-core backward: one CTA per (token, kv head)
//   nsa_finalize     dK, dV = cast(fp32 accumulators)
#include <math.h>

#include "plan.h"

namespace attn {

__device__ __forceinline__ int64_t seq_of_token(const PackedGeo &g, int64_t t)
{
    int64_t lo = 0, hi = g.nseq - 1;  // first b with t < cu_q[b+1]
    while (lo < hi) {
        int64_t mid = (lo + hi) / 2;
        if (t < g.cu_q[mid + 1]) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

// ------------------------------------------------------------- preprocess
// grid (ceil(t1_pad / 128), n1), 256 threads, 16 threads per 128-wide row.
__device__ __forceinline__ void zero_words(uint32_t *p, int64_t n, int64_t tid, int64_t nthr)
{
    // 16-byte stores over the 256-byte aligned region, then the tail
    uint4 *p4 = reinterpret_cast<uint4 *>(p);
    const int64_t n4 = n / 4;
    for (int64_t k = tid; k < n4; k += nthr) p4[k] = make_uint4(0, 0, 0, 0);
    for (int64_t k = n4 * 4 + tid; k < n; k += nthr) p[k] = 0u;
}

// Blocks of the preprocess: (ceil(t1_pad / 128) x n1) row blocks, 16 threads
// per 128-wide row; they also zero the accumulators the main kernel adds into.
inline int64_t nsa_pre_blocks(const NsaArgs &a) { return (a.t1 > 0 ? (a.t1_pad + 127) / 128 : 1) * a.n1; }

// Preprocess block pb of nblk (256 threads).
template <class T>
__device__ __forceinline__ void nsa_preprocess_block(const NsaArgs &a, int64_t pb, int64_t nblk)
{
    {   // buffers the main kernel adds into
        const int64_t nthr = nblk * blockDim.x, tid = pb * blockDim.x + threadIdx.x;
        zero_words(reinterpret_cast<uint32_t *>(a.dkacc), a.t2 * a.n2 * a.d, tid, nthr);
        zero_words(reinterpret_cast<uint32_t *>(a.dvacc), a.t2 * a.n2 * a.dv, tid, nthr);
        if (a.zero_dq) zero_words(reinterpret_cast<uint32_t *>(a.dqacc), a.t1 * a.n1 * a.d, tid, nthr);
        if (a.deterministic == 2) zero_words(a.sem, a.t1 * a.n2, tid, nthr);  // no dQ add has landed yet
    }
    const int64_t gx = nblk / a.n1, bx = pb % gx, h = pb / gx;
    const int lane = threadIdx.x % 16;
    for (int r = threadIdx.x / 16; r < 128; r += 16) {
        const int64_t t = bx * 128 + r;
        const bool live = t < a.t1_pad;  // no early exit: the row's threads shuffle below
        const int64_t row = t * a.n1 + h;  // token-major
        float dsum = 0.f;
        if (t < a.t1)  // D = rowsum(dO * O) over the value head dim, 8 elements per chunk
            for (int64_t ch = lane; ch < a.dv / 8; ch += 16) {
                const int64_t off = (t * a.n1 + h) * a.dv + ch * 8;
                uint4 ov = *reinterpret_cast<const uint4 *>(static_cast<const T *>(a.o) + off);
                uint4 dv = *reinterpret_cast<const uint4 *>(static_cast<const T *>(a.dO) + off);
                const uint32_t *op = &ov.x, *dp = &dv.x;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 of = unpack2<T>(op[e]), df = unpack2<T>(dp[e]);
                    dsum += of.x * df.x + of.y * df.y;
                }
            }
        for (int off = 8; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
        if (!live) continue;
        if (lane == 0) {
            float lse2 = INFINITY;
            if (t < a.t1) {
                const float mx = a.smax[(t * a.n1 + h) * 8], sm = a.ssum[(t * a.n1 + h) * 8];
                if (sm > 0.f && mx != -INFINITY) lse2 = (mx + logf(sm)) * kLog2e;
            }
            a.lse2[row] = lse2;
            a.dvec[row] = t < a.t1 ? dsum : 0.f;
        }
    }
}

// Init: the status word and the block bitmap (launched first, ordinarily).
__global__ void __launch_bounds__(256) nsa_init_kernel(NsaArgs a)
{
    pdl_trigger();  // the block lists may start launching; they wait for this grid
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0u;
    zero_words(a.bitmap, a.nrows * a.words_max, int64_t(blockIdx.x) * blockDim.x + threadIdx.x,
               int64_t(gridDim.x) * blockDim.x);
}

// ------------------------------------------------------------ block lists
// Mark: one thread per (token, kv head, slot).  A slot that repeats an earlier
// slot's block is flagged and skipped; the earlier one is kept.
__global__ void nsa_mark_kernel(NsaArgs a, PackedGeo geo)
{
    pdl_trigger();  // the next kernel may be placed now; it waits for this grid before it reads anything
    pdl_wait();     // the bitmap has been zeroed
    const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (gid >= a.t1 * a.n2 * a.cnt) return;
    const int64_t idx = gid / a.cnt, c = gid - idx * a.cnt;  // (token, kv head), slot
    const int64_t t = idx / a.n2, g = idx % a.n2;
    const int64_t b = seq_of_token(geo, t);
    const int64_t i = t - geo.cu_q[b], lq = geo.q_len(b), lkv = geo.kv_len(b);
    const int64_t nblk = lkv / a.bs;
    const int32_t *ids = a.topk + idx * a.cnt;
    const int32_t blk = ids[c];
    if (blk < 0 || blk >= nblk) {
        raise_flag(a.status, ATTN_DEV_INDEX_RANGE);
        return;
    }
    bool dup = false;
    for (int64_t c2 = 0; c2 < c; ++c2) dup |= ids[c2] == blk;
    if (dup) {
        raise_flag(a.status, ATTN_DEV_INDEX_DUP);
        return;
    }
    // the block's first key is the one most likely to be visible
    if (a.sparse_mode == 2 && !visible(ATTN_CAUSAL_BOTTOM_RIGHT, i, int64_t(blk) * a.bs, lq, lkv)) return;
    const int64_t row = (b * a.n2 + g) * a.nblk_max + blk;
    atomicOr(a.bitmap + row * a.words_max + i / 32, 1u << (i % 32));
    if (a.deterministic == 2) {  // ordered dQ: the token's kept blocks above this one add before it
        int32_t above = 0;
        for (int64_t c2 = 0; c2 < a.cnt; ++c2) {
            const int32_t id = ids[c2];
            if (id <= blk || int64_t(id) >= nblk) continue;
            bool first = true;
            for (int64_t c3 = 0; c3 < c2 && first; ++c3) first = ids[c3] != id;
            if (first && (a.sparse_mode != 2 || visible(ATTN_CAUSAL_BOTTOM_RIGHT, i, int64_t(id) * a.bs, lq, lkv)))
                ++above;
        }
        a.rank[idx * a.cnt + c] = above;
    }
}

// Count: one warp per row; counts land in offsets[row + 1].
__global__ void nsa_count_kernel(NsaArgs a)
{
    pdl_trigger();
    pdl_wait();
    const int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    if (row >= a.nrows) return;
    int n = 0;
    for (int64_t w = lane; w < a.words_max; w += 32) n += __popc(a.bitmap[row * a.words_max + w]);
    for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
    if (lane == 0) a.offsets[row + 1] = n;
    if (row == 0 && lane == 0) a.offsets[0] = 0;
}

// Scan: one CTA of 1024 threads, inclusive scan of offsets[1..nrows] in chunks.
__global__ void __launch_bounds__(1024) nsa_scan_kernel(NsaArgs a)
{
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
    for (int64_t base = 0; base < a.nrows; base += 1024) {
        const int64_t r = base + threadIdx.x;
        int32_t v = r < a.nrows ? a.offsets[r + 1] : 0;
        for (int off = 1; off < 32; off <<= 1) {
            int32_t u = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += u;
        }
        if (lane == 31) warp_tot[wid] = v;
        __syncthreads();
        if (wid == 0) {
            int32_t w = warp_tot[lane];
            for (int off = 1; off < 32; off <<= 1) {
                int32_t u = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += u;
            }
            warp_tot[lane] = w;
        }
        __syncthreads();
        const int32_t prefix = carry + (wid ? warp_tot[wid - 1] : 0);
        if (r < a.nrows) a.offsets[r + 1] = prefix + v;
        __syncthreads();
        if (threadIdx.x == 1023) carry = prefix + v;
        __syncthreads();
    }
}

// Emit: one warp per (row, 32-word segment of its bitmap), in token order
// within the row; a segment starts after the tokens of the row's earlier words.
// Blocks from emit_blocks on run the preprocess instead (pre = 1): it needs
// nothing from the block lists, so they do not wait and run while the
// earlier block-list kernels do; the kernels after this one wait for both.
template <class T>
__global__ void __launch_bounds__(256) nsa_emit_kernel(NsaArgs a, PackedGeo geo, int64_t emit_blocks, int pre)
{
    if (int64_t(blockIdx.x) >= emit_blocks) {
        pdl_trigger();
        if (pre) nsa_preprocess_block<T>(a, int64_t(blockIdx.x) - emit_blocks, int64_t(gridDim.x) - emit_blocks);
        return;
    }
    pdl_trigger();
    pdl_wait();
    const int64_t nseg = (a.words_max + 31) / 32;
    const int64_t wid = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    if (wid >= a.nrows * nseg) return;
    const int64_t row = wid / nseg, w0 = (wid - row * nseg) * 32;
    const int64_t b = row / (a.n2 * a.nblk_max);
    const uint32_t *bits_row = a.bitmap + row * a.words_max;
    int before = 0;  // tokens of the row's words before this segment
    for (int64_t w = lane; w < w0; w += 32) before += __popc(bits_row[w]);
    for (int off = 16; off > 0; off >>= 1) before += __shfl_xor_sync(0xffffffffu, before, off);
    const int64_t w = w0 + lane;
    uint32_t bits = w < a.words_max ? bits_row[w] : 0u;
    int n = __popc(bits), incl = n;
    for (int off = 1; off < 32; off <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += u;
    }
    int32_t my = a.offsets[row] + before + incl - n;
    while (bits) {
        int bit = __ffs(bits) - 1;
        bits &= bits - 1;
        a.tokens[my++] = int32_t(geo.cu_q[b] + w * 32 + bit);
    }
}

// ------------------------------------------------------------ main (CUDA cores)
// One CTA per (token, kv head); loops over the selected blocks, KB keys at a
// time, masking by the sparse mode and attenMaskOptional (if given).  dQ rows of the token are owned by the CTA; dK / dV go to fp32
// accumulators.  DQK: query / key head dim, DV: value head dim.
constexpr int kNsaKB = 32;  // keys per pass of the CUDA-core kernels
inline size_t nsa_simt_smem(int64_t G, int dqk, int dv)
{
    return sizeof(float) * size_t(kNsaKB * (dqk + 1) + kNsaKB * (dv + 1) + G * (dqk + 1) + G * (dv + 1) +
                                  2 * G * kNsaKB + 2 * G);
}

template <class OutT> __device__ __forceinline__ OutT out_cast(float x);
template <> __device__ __forceinline__ float out_cast<float>(float x) { return x; }
template <> __device__ __forceinline__ __half out_cast<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 out_cast<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <class T, class OutT, int DQK, int DV>
__global__ void __launch_bounds__(256) nsa_bwd_simt_kernel(NsaArgs a, PackedGeo geo)
{
    pdl_wait();
    pdl_trigger();
    constexpr int KB = kNsaKB, LDQ = DQK + 1, LDV = DV + 1;
    constexpr int PER = (32 * DQK + 255) / 256;  // dQ features per thread at G = 32
    extern __shared__ float smem[];
    const int G = int(a.n1 / a.n2);
    float(*Ks)[LDQ] = reinterpret_cast<float(*)[LDQ]>(smem);
    float(*Vs)[LDV] = reinterpret_cast<float(*)[LDV]>(smem + KB * LDQ);
    float(*Qs)[LDQ] = reinterpret_cast<float(*)[LDQ]>(smem + KB * LDQ + KB * LDV);
    float(*dOs)[LDV] = reinterpret_cast<float(*)[LDV]>(smem + KB * LDQ + KB * LDV + G * LDQ);
    float *Ps = smem + KB * LDQ + KB * LDV + G * LDQ + G * LDV;  // [G][KB]
    float *dSs = Ps + G * KB;
    float *lse_s = dSs + G * KB;
    float *d_s = lse_s + G;

    const int64_t t = blockIdx.x, g = blockIdx.y;
    const int64_t b = seq_of_token(geo, t);
    const int64_t i = t - geo.cu_q[b], lq = geo.q_len(b), lkv = geo.kv_len(b), k0 = geo.cu_kv[b];
    const int tid = threadIdx.x;
    const float c = a.scale * kLog2e;
    const T *Q = static_cast<const T *>(a.q), *K = static_cast<const T *>(a.k);
    const T *V = static_cast<const T *>(a.v), *dO = static_cast<const T *>(a.dO);

    for (int e = tid; e < G * DQK; e += 256) {
        const int hh = e / DQK, x = e % DQK;
        Qs[hh][x] = to_f32(Q[(t * a.n1 + g * G + hh) * DQK + x]);
    }
    for (int e = tid; e < G * DV; e += 256) {
        const int hh = e / DV, x = e % DV;
        dOs[hh][x] = to_f32(dO[(t * a.n1 + g * G + hh) * DV + x]);
    }
    if (tid < G) {
        lse_s[tid] = a.lse2[t * a.n1 + g * G + tid];
        d_s[tid] = a.dvec[t * a.n1 + g * G + tid];
    }
    float dq[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) dq[e] = 0.f;
    const int32_t *ids = a.topk + (t * a.n2 + g) * a.cnt;
    const int64_t nblk = lkv / a.bs;
    for (int64_t cc = 0; cc < a.cnt; ++cc) {
        const int64_t blk = ids[cc];
        if (blk < 0 || blk >= nblk) continue;  // flagged by the mark kernel
        bool dup = false;
        for (int64_t c2 = 0; c2 < cc; ++c2) dup |= ids[c2] == blk;
        if (dup) continue;
        for (int64_t sub = 0; sub < a.bs; sub += KB) {
            const int64_t j0 = blk * a.bs + sub;
            const int nk = int(a.bs - sub < KB ? a.bs - sub : KB);
            __syncthreads();
            for (int e = tid; e < nk * DQK; e += 256) {
                const int r = e / DQK, x = e % DQK;
                Ks[r][x] = to_f32(K[((k0 + j0 + r) * a.n2 + g) * DQK + x]);
            }
            for (int e = tid; e < nk * DV; e += 256) {
                const int r = e / DV, x = e % DV;
                Vs[r][x] = to_f32(V[((k0 + j0 + r) * a.n2 + g) * DV + x]);
            }
            __syncthreads();
            for (int e = tid; e < G * nk; e += 256) {
                const int hh = e / nk, r = e % nk;
                const bool vis = (a.sparse_mode != 2 || visible(ATTN_CAUSAL_BOTTOM_RIGHT, i, j0 + r, lq, lkv)) &&
                                 !(a.mask && a.mask[i * a.mask_cols + j0 + r]);
                float sv = 0.f, dp = 0.f;
                if (vis) {
#pragma unroll 8
                    for (int x = 0; x < DQK; ++x) sv += Qs[hh][x] * Ks[r][x];
#pragma unroll 8
                    for (int x = 0; x < DV; ++x) dp += dOs[hh][x] * Vs[r][x];
                }
                const float pv = (vis && lse_s[hh] != INFINITY) ? exp2f(sv * c - lse_s[hh]) : 0.f;
                Ps[hh * KB + r] = pv;
                dSs[hh * KB + r] = pv * (dp - d_s[hh]);
            }
            __syncthreads();
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                const int f = tid + e * 256;
                if (f >= G * DQK) break;
                const int hh = f / DQK, x = f % DQK;
                float acc = 0.f;
                for (int r = 0; r < nk; ++r) acc += dSs[hh * KB + r] * Ks[r][x];
                dq[e] += acc;
            }
            for (int f = tid; f < nk * DQK; f += 256) {
                const int r = f / DQK, x = f % DQK;
                float dk = 0.f;
                for (int hh = 0; hh < G; ++hh) dk += dSs[hh * KB + r] * Qs[hh][x];
                atomicAdd(a.dkacc + ((k0 + j0 + r) * a.n2 + g) * DQK + x, dk * a.scale);
            }
            for (int f = tid; f < nk * DV; f += 256) {
                const int r = f / DV, x = f % DV;
                float dv = 0.f;
                for (int hh = 0; hh < G; ++hh) dv += Ps[hh * KB + r] * dOs[hh][x];
                atomicAdd(a.dvacc + ((k0 + j0 + r) * a.n2 + g) * DV + x, dv);
            }
        }
    }
    OutT *dQ = static_cast<OutT *>(a.dq);
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        const int f = tid + e * 256;
        if (f >= G * DQK) break;
        const int hh = f / DQK, x = f % DQK;
        dQ[(t * a.n1 + g * G + hh) * DQK + x] = out_cast<OutT>(dq[e] * a.scale);
    }
}

// ------------------------------------------------------------- forward (CUDA cores)
// NSA selected-attention forward: one CTA per (token, kv head), KB keys of the
// selected blocks at a time, online softmax per query head (max in log2 units).
// A key is used when the sparse mode and attenMaskOptional (if given) keep it.
// O = sum_j exp(s_j - max) v_j / sum; softmaxMax = max_j s_j (natural units),
// softmaxSum = sum_j exp(s_j - max), both written to all 8 lanes.
template <class T, int DQK, int DV>
__global__ void __launch_bounds__(256) nsa_fwd_simt_kernel(NsaArgs a, PackedGeo geo)
{
    constexpr int KB = kNsaKB, LDQ = DQK + 1, LDV = DV + 1;
    constexpr int PER = (32 * DV + 255) / 256;  // O features per thread at G = 32
    extern __shared__ float smem[];
    const int G = int(a.n1 / a.n2);
    float(*Ks)[LDQ] = reinterpret_cast<float(*)[LDQ]>(smem);
    float(*Vs)[LDV] = reinterpret_cast<float(*)[LDV]>(smem + KB * LDQ);
    float(*Qs)[LDQ] = reinterpret_cast<float(*)[LDQ]>(smem + KB * LDQ + KB * LDV);
    float *Ps = smem + KB * LDQ + KB * LDV + G * LDQ;  // [G][KB]
    float *m_s = Ps + G * KB, *l_s = m_s + G, *al_s = l_s + G;

    const int64_t t = blockIdx.x, g = blockIdx.y;
    const int64_t b = seq_of_token(geo, t);
    const int64_t i = t - geo.cu_q[b], lq = geo.q_len(b), lkv = geo.kv_len(b), k0 = geo.cu_kv[b];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const float c = a.scale * kLog2e;
    const T *Q = static_cast<const T *>(a.q), *K = static_cast<const T *>(a.k), *V = static_cast<const T *>(a.v);

    for (int e = tid; e < G * DQK; e += 256) {
        const int hh = e / DQK, x = e % DQK;
        Qs[hh][x] = to_f32(Q[(t * a.n1 + g * G + hh) * DQK + x]);
    }
    if (tid < G) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.f;
    }
    float o[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = 0.f;
    const int32_t *ids = a.topk + (t * a.n2 + g) * a.cnt;
    const int64_t nblk = lkv / a.bs;
    for (int64_t cc = 0; cc < a.cnt; ++cc) {
        const int64_t blk = ids[cc];
        if (blk < 0 || blk >= nblk) {
            if (tid == 0) raise_flag(a.status, ATTN_DEV_INDEX_RANGE);
            continue;
        }
        bool dup = false;
        for (int64_t c2 = 0; c2 < cc; ++c2) dup |= ids[c2] == blk;
        if (dup) {
            if (tid == 0) raise_flag(a.status, ATTN_DEV_INDEX_DUP);
            continue;
        }
        for (int64_t sub = 0; sub < a.bs; sub += KB) {
            const int64_t j0 = blk * a.bs + sub;
            const int nk = int(a.bs - sub < KB ? a.bs - sub : KB);
            __syncthreads();
            for (int e = tid; e < nk * DQK; e += 256) {
                const int r = e / DQK, x = e % DQK;
                Ks[r][x] = to_f32(K[((k0 + j0 + r) * a.n2 + g) * DQK + x]);
            }
            for (int e = tid; e < nk * DV; e += 256) {
                const int r = e / DV, x = e % DV;
                Vs[r][x] = to_f32(V[((k0 + j0 + r) * a.n2 + g) * DV + x]);
            }
            __syncthreads();
            for (int e = tid; e < G * KB; e += 256) {  // scores, log2 units; -inf where masked
                const int hh = e / KB, r = e % KB;
                float sv = -INFINITY;
                if (r < nk && (a.sparse_mode != 2 || visible(ATTN_CAUSAL_BOTTOM_RIGHT, i, j0 + r, lq, lkv)) &&
                    !(a.mask && a.mask[i * a.mask_cols + j0 + r])) {
                    sv = 0.f;
#pragma unroll 8
                    for (int x = 0; x < DQK; ++x) sv += Qs[hh][x] * Ks[r][x];
                    sv *= c;
                }
                Ps[hh * KB + r] = sv;
            }
            __syncthreads();
            for (int hh = warp; hh < G; hh += 8) {  // one warp per head: raise the max, P, the sum
                const float sv = Ps[hh * KB + lane];
                float mb = sv;
                for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
                const float m_old = m_s[hh], m_new = fmaxf(m_old, mb);
                const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_old - m_new);
                const float pv = sv == -INFINITY ? 0.f : exp2f(sv - m_new);
                float ps = pv;
                for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
                Ps[hh * KB + lane] = pv;
                __syncwarp();
                if (lane == 0) {
                    l_s[hh] = l_s[hh] * alpha + ps;
                    m_s[hh] = m_new;
                    al_s[hh] = alpha;
                }
            }
            __syncthreads();
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                const int f = tid + e * 256;
                if (f >= G * DV) break;
                const int hh = f / DV, x = f % DV;
                float acc = 0.f;
                for (int r = 0; r < nk; ++r) acc += Ps[hh * KB + r] * Vs[r][x];
                o[e] = o[e] * al_s[hh] + acc;
            }
        }
    }
    __syncthreads();
    T *O = static_cast<T *>(a.o_out);
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        const int f = tid + e * 256;
        if (f >= G * DV) break;
        const int hh = f / DV, x = f % DV;
        const float l = l_s[hh];
        O[(t * a.n1 + g * G + hh) * DV + x] = from_f32<T>(l > 0.f ? o[e] / l : 0.f);
    }
    for (int e = tid; e < G * 8; e += 256) {
        const int hh = e / 8;
        const int64_t row = t * a.n1 + g * G + hh;
        const float m = m_s[hh];
        a.smax_out[row * 8 + e % 8] = m == -INFINITY ? -INFINITY : m / kLog2e;
        a.ssum_out[row * 8 + e % 8] = l_s[hh];
    }
}

// Four fp32 values to OutT (16-bit: packed, round to nearest even).
template <class OutT> __device__ __forceinline__ void store4(OutT *p, float4 v);
template <> __device__ __forceinline__ void store4<float>(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
template <> __device__ __forceinline__ void store4<__half>(__half *p, float4 v)
{
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack2<__half>(v.x, v.y), pack2<__half>(v.z, v.w));
}
template <> __device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *p, float4 v)
{
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack2<__nv_bfloat16>(v.x, v.y), pack2<__nv_bfloat16>(v.z, v.w));
}

// dK, dV = cast(fp32 accumulators), 4 elements per step (head dims are multiples of 8).
template <class OutT>
__device__ __forceinline__ void convert_dkdv4(const NsaArgs &a)
{
    const int64_t nk = a.t2 * a.n2 * a.d, nv = a.t2 * a.n2 * a.dv;
    OutT *dK = static_cast<OutT *>(a.dk), *dV = static_cast<OutT *>(a.dv_out());
    const int64_t step = int64_t(gridDim.x) * blockDim.x * 4;
    for (int64_t e = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) * 4; e < nk; e += step)
        store4<OutT>(dK + e, *reinterpret_cast<const float4 *>(a.dkacc + e));
    for (int64_t e = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) * 4; e < nv; e += step)
        store4<OutT>(dV + e, *reinterpret_cast<const float4 *>(a.dvacc + e));
}

// dQ = cast(scale * fp32 accumulator), tensor-core path
template <class OutT>
__global__ void nsa_dq_finalize_kernel(NsaArgs a, int with_kv)
{
    pdl_wait();
    pdl_trigger();
    const int64_t n = a.t1 * a.n1 * a.d;
    OutT *dQ = static_cast<OutT *>(a.dq);
    for (int64_t e = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) * 4; e < n; e += int64_t(gridDim.x) * blockDim.x * 4) {
        const float4 v = *reinterpret_cast<const float4 *>(a.dqacc + e);
        store4<OutT>(dQ + e, make_float4(v.x * a.scale, v.y * a.scale, v.z * a.scale, v.w * a.scale));
    }
    if (with_kv) convert_dkdv4<OutT>(a);  // dK / dV in the same launch
}

// Deterministic dQ: per (token, query head) the partial rows of the selected
// slots, summed in slot order; slots whose block was never processed (out of
// range, a repeat, or fully masked by sparse mode 2) are skipped.  (d = 128:
// 32 threads x 4 floats per row.)
template <class OutT>
__global__ void nsa_dq_finalize_det_kernel(NsaArgs a, PackedGeo geo, int with_kv)
{
    pdl_wait();
    pdl_trigger();
    const int64_t rows = a.t1 * a.n1;
    const int G = int(a.n1 / a.n2);
    for (int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) / 32; w < rows;
         w += int64_t(gridDim.x) * blockDim.x / 32) {
        const int lane = threadIdx.x % 32;
        const int64_t t = w / a.n1, h = w % a.n1, g = h / G, hh = h % G;
        const int64_t b = seq_of_token(geo, t);
        const int64_t i = t - geo.cu_q[b], lq = geo.q_len(b), lkv = geo.kv_len(b);
        const int32_t *ids = a.topk + (t * a.n2 + g) * a.cnt;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int64_t c = 0; c < a.cnt; ++c) {
            const int32_t blk = ids[c];
            bool use = blk >= 0 && int64_t(blk) < lkv / a.bs;
            for (int64_t c2 = 0; use && c2 < c; ++c2) use = ids[c2] != blk;
            if (use && a.sparse_mode == 2) use = visible(ATTN_CAUSAL_BOTTOM_RIGHT, i, int64_t(blk) * a.bs, lq, lkv);
            if (!use) continue;
            const float4 v = reinterpret_cast<const float4 *>(a.dqpart + (((t * a.n2 + g) * a.cnt + c) * G + hh) * a.d)[lane];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        store4<OutT>(static_cast<OutT *>(a.dq) + w * a.d + lane * 4,
                     make_float4(acc.x * a.scale, acc.y * a.scale, acc.z * a.scale, acc.w * a.scale));
    }
    if (with_kv) convert_dkdv4<OutT>(a);  // dK / dV in the same launch
}

// Deterministic mode 1: each block's dK / dV rows are the sum of its pieces' rows, taken in piece
// order (one thread per block-list row, key and 4 of the d + d_v columns).
__global__ void __launch_bounds__(256) nsa_kv_sum_kernel(NsaArgs a, PackedGeo geo)
{
    pdl_wait();
    pdl_trigger();
    const int64_t w = (a.d + a.dv) / 4;
    const int64_t n = a.nrows * a.bs * w;
    for (int64_t x = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; x < n; x += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = x / (a.bs * w), key = (x / w) % a.bs, c4 = x % w;
        const int32_t p0 = a.pieces[row], p1 = a.pieces[row + 1];
        if (p0 == p1) continue;  // no token selected the block: its rows stay zero
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t pc = p0; pc < p1; ++pc) {
            const float4 v = reinterpret_cast<const float4 *>(a.kvpart + (int64_t(pc) * a.bs + key) * (a.d + a.dv))[c4];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        const int64_t b = row / (a.n2 * a.nblk_max), g = (row / a.nblk_max) % a.n2, blk = row % a.nblk_max;
        const int64_t krow = (geo.cu_kv[b] + blk * a.bs + key) * a.n2 + g;
        float *dst = c4 < a.d / 4 ? a.dkacc + krow * a.d + c4 * 4 : a.dvacc + krow * a.dv + (c4 - a.d / 4) * 4;
        *reinterpret_cast<float4 *>(dst) = acc;
    }
}

template <class OutT>
__global__ void nsa_finalize_kernel(NsaArgs a)
{
    pdl_wait();
    convert_dkdv4<OutT>(a);
}

namespace {
// bitmap must be zero on entry.  pdl: chained behind a kernel (else behind a memset, ordinarily).
// pre: the emit kernel also runs the preprocess (its extra blocks).
template <class T>
cudaError_t block_lists(const NsaArgs &a, const PackedGeo &g, cudaStream_t s, bool pdl, bool pre)
{
    cudaError_t e = cudaSuccess;
    if (a.t1 > 0 && (e = launch_kernel(nsa_mark_kernel, dim3(unsigned((a.t1 * a.n2 * a.cnt + 255) / 256)), dim3(256), 0,
                                       s, pdl, a, g)) != cudaSuccess)
        return e;
    int64_t emit_blocks = 0;
    if (a.nrows > 0) {
        const dim3 grid(unsigned((a.nrows * 32 + 255) / 256));
        if ((e = launch_kernel(nsa_count_kernel, grid, dim3(256), 0, s, pdl || a.t1 > 0, a)) != cudaSuccess) return e;
        if ((e = launch_kernel(nsa_scan_kernel, dim3(1), dim3(1024), 0, s, true, a)) != cudaSuccess) return e;
        emit_blocks = (a.nrows * ((a.words_max + 31) / 32) * 32 + 255) / 256;
    }
    const int64_t blocks = emit_blocks + (pre ? nsa_pre_blocks(a) : 0);
    if (blocks > 0 &&
        (e = launch_kernel(nsa_emit_kernel<T>, dim3(unsigned(blocks)), dim3(256), 0, s, pdl || a.t1 > 0 || a.nrows > 0,
                           a, g, emit_blocks, pre ? 1 : 0)) != cudaSuccess)
        return e;
    return cudaSuccess;
}

template <class T, class OutT>
cudaError_t launch_simt_bwd(const NsaArgs &a, const PackedGeo &g, cudaStream_t s)
{
    const int64_t G = a.n1 / a.n2;
    void (*k)(NsaArgs, PackedGeo) = nullptr;
    if (a.d == 128 && a.dv == 128) k = nsa_bwd_simt_kernel<T, OutT, 128, 128>;
    else if (a.d == 192 && a.dv == 128) k = nsa_bwd_simt_kernel<T, OutT, 192, 128>;
    else if (a.d == 128 && a.dv == 192) k = nsa_bwd_simt_kernel<T, OutT, 128, 192>;
    else k = nsa_bwd_simt_kernel<T, OutT, 192, 192>;
    const size_t smem = nsa_simt_smem(G, int(a.d), int(a.dv));
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    return launch_kernel(k, dim3(unsigned(a.t1), unsigned(a.n2)), dim3(256), smem, s, true, a, g);
}

template <class T, class OutT>
cudaError_t run_nsa(const NsaArgs &a0, const PackedGeo &g, cudaStream_t s, cudaEvent_t before, cudaEvent_t after)
{
    cudaError_t e;
    const bool tc = nsa_tc_supported(a0);
    NsaArgs a = a0;
    a.zero_dq = tc && a.deterministic != 1 ? 1 : 0;
    // init (status word, bitmap) first, ordinarily; then the block lists with the preprocess riding in
    // the emit launch; every kernel after init is chained with programmatic dependent launch
    {
        const int64_t words = a.nrows * a.words_max;
        const unsigned blocks = unsigned(words > 0 ? (words / 4 + 255) / 256 < 1024 ? (words / 4 + 255) / 256 : 1024 : 1);
        nsa_init_kernel<<<blocks > 0 ? blocks : 1, 256, 0, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = block_lists<T>(a, g, s, true, true)) != cudaSuccess) return e;
    if (tc) {
        if (before && (e = cudaEventRecord(before, s)) != cudaSuccess) return e;
        if ((e = launch_nsa_tc(a, g, s)) != cudaSuccess) return e;
        if (after && (e = cudaEventRecord(after, s)) != cudaSuccess) return e;
        if (a.t1 > 0 && a.deterministic == 1 &&
            (e = launch_kernel(nsa_kv_sum_kernel, dim3(1024), dim3(256), 0, s, true, a, g)) != cudaSuccess)
            return e;
        // the dQ finalize converts dK / dV too
        if (a.t1 > 0 && a.deterministic == 1)
            e = launch_kernel(nsa_dq_finalize_det_kernel<OutT>, dim3(1024), dim3(256), 0, s, true, a, g, 1);
        else if (a.t1 > 0)
            e = launch_kernel(nsa_dq_finalize_kernel<OutT>, dim3(1024), dim3(256), 0, s, true, a, 1);
        if (e != cudaSuccess) return e;
    } else if (a.t1 > 0) {
        if (before && (e = cudaEventRecord(before, s)) != cudaSuccess) return e;
        if ((e = launch_simt_bwd<T, OutT>(a, g, s)) != cudaSuccess) return e;
        if (after && (e = cudaEventRecord(after, s)) != cudaSuccess) return e;
    }
    const bool kv_done = tc && a.t1 > 0;  // converted by the dQ finalize
    if (a.t2 > 0 && !kv_done &&
        (e = launch_kernel(nsa_finalize_kernel<OutT>, dim3(1024), dim3(256), 0, s, true, a)) != cudaSuccess)
        return e;
    return cudaSuccess;
}

// ------------------------------------------------- forward on the tensor cores
// Before the two passes: every row's maximum at -inf (as the order-preserving
// int of the atomicMax), its sum and the fp32 O accumulator at 0.
__global__ void __launch_bounds__(256) nsa_fwd_init_kernel(NsaArgs a)
{
    pdl_wait();
    pdl_trigger();
    const int64_t nthr = int64_t(gridDim.x) * blockDim.x, tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int32_t neg_inf = int32_t(0x807FFFFF);  // -inf (0xFF800000) with its magnitude bits flipped
    for (int64_t r = tid; r < a.t1 * a.n1; r += nthr) {
        reinterpret_cast<int32_t *>(a.lse2)[r] = neg_inf;
        a.dvec[r] = 0.f;
    }
    zero_words(reinterpret_cast<uint32_t *>(a.dqacc), a.t1 * a.n1 * a.dv, tid, nthr);
}

// After them: O = O_acc / sum (0 where the row sees no key), softmaxMax = the maximum in natural units
// (-inf where none), softmaxSum = the sum, the stats in all 8 lanes.  A warp per (token, query head) row.
template <class T>
__global__ void __launch_bounds__(256) nsa_fwd_finalize_kernel(NsaArgs a)
{
    pdl_wait();
    const int lane = threadIdx.x % 32;
    for (int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) / 32; w < a.t1 * a.n1;
         w += int64_t(gridDim.x) * blockDim.x / 32) {
        const float sum = a.dvec[w], inv = sum > 0.f ? 1.f / sum : 0.f;
        for (int64_t x = lane * 4; x < a.dv; x += 128) {
            const float4 v = *reinterpret_cast<const float4 *>(a.dqacc + w * a.dv + x);
            T *o = static_cast<T *>(a.o_out) + w * a.dv + x;
            *reinterpret_cast<uint2 *>(o) = make_uint2(pack2<T>(v.x * inv, v.y * inv), pack2<T>(v.z * inv, v.w * inv));
        }
        if (lane < 8) {
            const int32_t mi = reinterpret_cast<const int32_t *>(a.lse2)[w];
            const float m = __int_as_float(mi >= 0 ? mi : mi ^ 0x7FFFFFFF);
            a.smax_out[w * 8 + lane] = m == -INFINITY ? -INFINITY : m / kLog2e;
            a.ssum_out[w * 8 + lane] = sum;
        }
    }
}

template <class T, int DQK, int DV> cudaError_t run_nsa_fwd_t(const NsaArgs &a, const PackedGeo &g, cudaStream_t s)
{
    auto k = nsa_fwd_simt_kernel<T, DQK, DV>;
    const int64_t G = a.n1 / a.n2;
    const size_t smem = sizeof(float) * size_t(kNsaKB * (DQK + 1) + kNsaKB * (DV + 1) + G * (DQK + 1) + G * kNsaKB + 3 * G);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s)) != cudaSuccess) return e;
    k<<<dim3(unsigned(a.t1), unsigned(a.n2)), 256, smem, s>>>(a, g);
    return cudaGetLastError();
}

template <class T> cudaError_t run_nsa_fwd(const NsaArgs &a0, const PackedGeo &g, cudaStream_t s)
{
    if (nsa_tc_supported(a0)) {  // tensor cores: block lists, init, row maxima, sums and O, finalize
        NsaArgs a = a0;
        a.zero_dq = 0;
        cudaError_t e;
        const int64_t words = a.nrows * a.words_max;
        const unsigned blocks = unsigned(words > 0 ? (words / 4 + 255) / 256 < 1024 ? (words / 4 + 255) / 256 : 1024 : 1);
        nsa_init_kernel<<<blocks > 0 ? blocks : 1, 256, 0, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = block_lists<T>(a, g, s, true, false)) != cudaSuccess) return e;
        if ((e = launch_kernel(nsa_fwd_init_kernel, dim3(1024), dim3(256), 0, s, true, a)) != cudaSuccess) return e;
        if ((e = launch_nsa_tc(a, g, s, true)) != cudaSuccess) return e;
        return launch_kernel(nsa_fwd_finalize_kernel<T>, dim3(1024), dim3(256), 0, s, true, a);
    }
    const NsaArgs &a = a0;
    if (a.d == 128 && a.dv == 128) return run_nsa_fwd_t<T, 128, 128>(a, g, s);
    if (a.d == 192 && a.dv == 128) return run_nsa_fwd_t<T, 192, 128>(a, g, s);
    if (a.d == 128 && a.dv == 192) return run_nsa_fwd_t<T, 128, 192>(a, g, s);
    return run_nsa_fwd_t<T, 192, 192>(a, g, s);
}
}  // namespace

cudaError_t launch_nsa_block_lists(const NsaArgs &a, const PackedGeo &g, cudaStream_t s)
{
    cudaError_t e;
    if ((e = cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s)) != cudaSuccess) return e;
    size_t bitmap_bytes = size_t(a.nrows) * size_t(a.words_max) * sizeof(uint32_t);
    if (bitmap_bytes && (e = cudaMemsetAsync(a.bitmap, 0, bitmap_bytes, s)) != cudaSuccess) return e;
    // no preprocess here: the emit kernel's type argument only names an instantiation
    return block_lists<__nv_bfloat16>(a, g, s, false, false);
}

cudaError_t launch_nsa_bwd(const NsaArgs &a, const PackedGeo &g, cudaStream_t s, cudaEvent_t before,
                           cudaEvent_t after)
{
    if (a.grad_fp32)
        return a.dtype == ATTN_F16 ? run_nsa<__half, float>(a, g, s, before, after)
                                   : run_nsa<__nv_bfloat16, float>(a, g, s, before, after);
    return a.dtype == ATTN_F16 ? run_nsa<__half, __half>(a, g, s, before, after)
                               : run_nsa<__nv_bfloat16, __nv_bfloat16>(a, g, s, before, after);
}

cudaError_t launch_nsa_fwd(const NsaArgs &a, const PackedGeo &g, cudaStream_t s)
{
    return a.dtype == ATTN_F16 ? run_nsa_fwd<__half>(a, g, s) : run_nsa_fwd<__nv_bfloat16>(a, g, s);
}

}  // namespace attn
