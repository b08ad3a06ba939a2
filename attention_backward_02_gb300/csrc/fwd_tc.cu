// fwd_tc.cu -- tensor-core SDPA forward in training mode (O and the fp32
// log-sum-exp stats) for sm_103a: tcgen05 MMAs with TMEM accumulators, TMA
// tile loads, mbarrier pipelines.
//
// The forward graph of the cuDNN-frontend sample
// "51_scaled_dot_product_attention_backward" (sdpa with is_inference=False:
// O and the (B,H,S,1) float32 stats, attn_scale, causal mask), computed the
// FlashAttention way: key tiles stream past a resident query tile and the
// softmax is accumulated online.
//
// One CTA per (sequence, query head, tile of BM = 128 queries), longest tiles
// first.  Query rows are the MMA M dimension and the TMEM lanes:
//   S = Q K^T      M=128 (queries) N=128 (keys) K=D   A=Q (smem, K-major) B=K (smem, K-major)
//   O += P V       M=128           N=D          K=128 A=P (TMEM, 16-bit)  B=V (smem, MN-major)
// S goes to two alternating TMEM buffers, so the MMA of key tile j+1 runs
// while the softmax warps work on tile j; P goes to TMEM (two buffers) as
// 16-bit pairs and is read there by the O GEMM.  TMEM: S 2 x 128 + P 2 x 64 +
// O D columns.
//
// Online softmax: two warps per TMEM lane quadrant (warps 2..9), each thread
// one query row and half of the tile's 128 key columns (and half of O's
// columns).  Each row keeps a reference max m (log2 units, scale folded in)
// and the sum l of exp2(x - m); the two halves of a row swap their tile
// maxima through shared memory (a named barrier per tile), so both take the
// same m.  m is raised only when a tile's max exceeds it by more than 8, and
// then l and the row of O in TMEM are scaled by exp2(m_old - m_new), so
// P = exp2(x - m) <= 2^8 fits both 16-bit types and the rescale is rare.
// O / l and LSE = (m + log2 l) / log2 e come out at the end (the halves add
// their sums first); a row that sees no key has O = 0 and LSE = +inf.
//
// Roles (11 warps): warp 0 issues the TMA loads of Q (once) and K (through an
// NSK-stage ring), warp 10 those of V (an NSV-stage ring of its own: a K stage
// is free once S has read it, a V stage only once O += P V has), warp 1 the
// MMAs, warps 2..9 the softmax and the epilogue.  Every
// barrier wait is bounded; a wait that runs out sets ATTN_DEV_TIMEOUT in the
// status word and the CTA skips the rest of its work, drains its copies and
// MMAs, and frees its TMEM.
#include <climits>
#include <type_traits>

#include "plan.h"
#include "sm103.cuh"
#include "tc_util.cuh"
#include "tmap.h"

namespace attn {
using namespace sm103;
using namespace tc;

template <int D>
struct FwdCfg {
    static constexpr int BM = 128, BN = 128;
    static constexpr int NSK = D == 64 ? 4 : 3;      // K ring stages
    static constexpr int NSV = D == 64 ? 4 : 2;      // V ring stages
    static constexpr int THREADS = 32 * 11;          // TMA (Q, K), MMA, 8 softmax warps (two per quadrant), TMA (V)
    static constexpr int TILE_BYTES = BN * D * 2;    // a K or V tile, and the Q tile (BM = BN)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + TILE_BYTES;          // NSK stages
    static constexpr int OFF_V = OFF_K + NSK * TILE_BYTES;    // NSV stages
    static constexpr int OFF_BAR = OFF_V + NSV * TILE_BYTES;
    static constexpr int OFF_MISC = OFF_BAR + 32 * 8;
    static constexpr int OFF_XM = OFF_MISC + 64;        // [2 tile parities][2 halves][128 rows] floats
    static constexpr int SMEM = OFF_XM + 2 * 2 * 128 * 4;
    // room to align the base to 1024; at least half the SM's shared memory, so one CTA (holding all
    // 512 TMEM columns) runs per SM
    static constexpr int SMEM_ALLOC = SMEM + 1024 > 116 * 1024 ? SMEM + 1024 : 116 * 1024;
    static constexpr int T_S = 0, T_P = 256, T_O = 384;
    static constexpr int T_COLS = 512;
    static_assert(T_O + D <= T_COLS, "TMEM budget");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(2 + 2 * NSK + 2 * NSV + 10 <= 32, "barrier slots");
};

struct FwdParams {
    CUtensorMap tm_q, tm_k, tm_v;
    DenseArgs a;
};

template <class Geo> struct FwdPacked : std::false_type {};
template <> struct FwdPacked<PackedGeo> : std::true_type {};

template <class T, int D, class Geo>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
    dense_fwd_tc_kernel(const __grid_constant__ FwdParams p, const Geo geo)
{
    using Cfg = FwdCfg<D>;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, NSK = Cfg::NSK, NSV = Cfg::NSV;
    constexpr bool kPacked = FwdPacked<Geo>::value;
    constexpr int kType = std::is_same<T, __half>::value ? 0 : 1;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *q_full = bars + 0, *drain = bars + 1;
    uint64_t *k_full = bars + 2, *k_empty = k_full + NSK, *v_full = k_empty + NSK, *v_empty = v_full + NSV;
    uint64_t *s_full = v_empty + NSV;      // [2] S of a key tile written
    uint64_t *s_free = s_full + 2;         // [2] S read out by the softmax warps
    uint64_t *p_full = s_full + 4;         // [2] P written (and O rescaled if needed)
    uint64_t *p_free = s_full + 6;         // [2] the O GEMM has read P
    uint64_t *o_done = s_full + 8;         // the O GEMMs issued so far have completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + Cfg::OFF_MISC + 8);
    const DenseArgs &a = p.a;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // ---- the unit: (sequence b, query head hq, query tile qt), longest first
    int64_t b, hq, qt;
    {
        const int64_t u = blockIdx.x;
        if (!kPacked) {
            const int64_t nqt = (geo.q_len(0) + BM - 1) / BM, per = a.h * geo.nseq;
            qt = nqt - 1 - u / per;
            const int64_t rest = u - (u / per) * per;
            b = rest / a.h;
            hq = rest - b * a.h;
        } else {  // 128-row tiles of the packed workspace rows, each sequence's last tile first
            const int64_t tile = u / a.h;
            hq = u - tile * a.h;
            int64_t i0w = 0;
            geo.ws_locate(tile * BM, &b, &i0w);
            const int64_t nqt = (geo.q_len(b) + BM - 1) / BM;
            qt = nqt - 1 - i0w / BM;
        }
    }
    const int64_t G = a.h / a.h_kv, g = hq / G;
    const int64_t lq = geo.q_len(b), lkv = geo.kv_len(b);
    const int64_t q_row0 = kPacked ? geo.q_start(b) : 0, kv_row0 = kPacked ? geo.kv_start(b) : 0;
    const int q_b = kPacked ? 0 : int(b);
    const int64_t i0 = qt * BM;
    const int64_t i_last = (i0 + BM - 1 < lq - 1) ? i0 + BM - 1 : lq - 1;
    const int64_t key_last = lkv > 0 ? last_visible_key(a.mask, i_last, lq, lkv) : -1;
    const int n_kt = key_last < 0 ? 0 : int(key_last / BN + 1);  // key tiles any row of the tile sees

    if (threadIdx.x == 0) {
        *abort = 0;
        mbar_init(q_full, 1);
        mbar_init(drain, 1);
        for (int s = 0; s < NSK; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s_full[k], 1);
            mbar_init(&s_free[k], 8);
            mbar_init(&p_full[k], 8);
            mbar_init(&p_free[k], 1);
        }
        mbar_init(o_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, Cfg::T_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    uint8_t *sQ = smem + Cfg::OFF_Q;
    auto sK = [&](int s) { return smem + Cfg::OFF_K + s * Cfg::TILE_BYTES; };
    auto sV = [&](int s) { return smem + Cfg::OFF_V + s * Cfg::TILE_BYTES; };

    if (warp == 0 || warp == 10) {
        // ================================================= TMA producers: Q and K (warp 0), V (warp 10)
        if (elect_one() && n_kt > 0) {
            const bool isk = warp == 0;
            const int nst = isk ? NSK : NSV;
            uint64_t *full = isk ? k_full : v_full, *empty = isk ? k_empty : v_empty;
            const CUtensorMap *tm = isk ? &p.tm_k : &p.tm_v;
            prefetch_tmap(tm);
            bool ok = true;
            int armed = 0;
            if (isk) {
                prefetch_tmap(&p.tm_q);
                mbar_arrive_expect_tx(q_full, Cfg::TILE_BYTES);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(sQ + c * BM * 128, &p.tm_q, q_full, c * 64, int(q_row0 + i0), int(hq), q_b);
            }
            for (int j = 0; j < n_kt; ++j) {
                const int s = j % nst, use = j / nst;
                if (use > 0 && ok && !(ok = mbar_wait(&empty[s], uint32_t(use - 1) & 1, abort)))
                    flag_abort(abort, a.status);
                if (!ok) break;
                armed = j + 1;
                mbar_arrive_expect_tx(&full[s], Cfg::TILE_BYTES);
                uint8_t *dst = isk ? sK(s) : sV(s);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(dst + c * BN * 128, tm, &full[s], c * 64, int(kv_row0 + j * BN), int(g), q_b);
            }
            // let every copy this thread started land before the CTA exits
            volatile int never = 0;
            if (isk) mbar_wait(q_full, 0, &never, 100000000ull);
            for (int j = armed - nst; j < armed; ++j)
                if (j >= 0) mbar_wait(&full[j % nst], uint32_t(j / nst) & 1, &never, 100000000ull);
        }
    } else if (warp == 1) {
        // ================================================= MMA issuer
        if (elect_one() && n_kt > 0) {
            constexpr uint32_t idS = idesc_f16(128, BN, kType, 0, 0);
            constexpr uint32_t idO = idesc_f16(128, D, kType, 0, 1);
            bool ok = true;
            auto wait = [&](uint64_t *bar, uint32_t parity) {
                if (ok && !(ok = mbar_wait(bar, parity, abort))) flag_abort(abort, a.status);
                tc_fence_after();
            };
            const uint64_t kQ = desc_kmaj(smem_u32(sQ), BM, 0);
            // O += P V for key tile x, once its P is in TMEM
            auto pv = [&](int x) {
                const int pb = x & 1, s = x % NSV;
                wait(&p_full[pb], uint32_t(x >> 1) & 1);
                wait(&v_full[s], uint32_t(x / NSV) & 1);
                if (ok) {
                    const uint64_t mV = desc_mn(smem_u32(sV(s)), BN, 0);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_f16_ts(tmem + Cfg::T_O, tmem + Cfg::T_P + pb * 64 + kk * 8, mn_step(mV, kk), idO,
                                   x > 0 || kk > 0);
                    mma_commit(o_done);
                    mma_commit(&v_empty[s]);
                    mma_commit(&p_free[pb]);
                }
            };
            wait(q_full, 0);
            for (int j = 0; j < n_kt; ++j) {
                const int s = j % NSK, sb = j & 1;
                wait(&k_full[s], uint32_t(j / NSK) & 1);
                if (j >= 2) wait(&s_free[sb], uint32_t((j >> 1) - 1) & 1);
                if (ok) {
                    const uint64_t kK = desc_kmaj(smem_u32(sK(s)), BN, 0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_f16_ss(tmem + Cfg::T_S + sb * 128, kmaj_step(kQ, BM, kk), kmaj_step(kK, BN, kk), idS,
                                   kk > 0);
                    mma_commit(&s_full[sb]);
                    mma_commit(&k_empty[s]);  // S has read this K stage
                }
                if (j >= 1) pv(j - 1);
            }
            pv(n_kt - 1);
            volatile int never = 0;
            mma_commit(drain);
            mbar_wait(drain, 0, &never, 100000000ull);
        }
    } else {
        // ================================================= softmax and epilogue (warps 2..9)
        const int qd = warp & 3, half = (warp - 2) >> 2;  // TMEM lane quadrant, half of the columns
        const uint32_t lane_addr = uint32_t(qd * 32) << 16;
        const int r = qd * 32 + lane;
        constexpr int HC = BN / 2, HD = D / 2;  // key columns and O columns per half
        float *xm = reinterpret_cast<float *>(smem + Cfg::OFF_XM);  // the halves' exchange
        const int64_t i = i0 + r;  // query position in the sequence
        const float c = a.scale * kLog2e;
        const int64_t kmax = lkv > 0 && i < lq ? last_visible_key(a.mask, i, lq, lkv) : -1;  // last key it sees
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        auto wait = [&](uint64_t *bar, uint32_t parity) {
            if (ok && !(ok = mbar_wait(bar, parity, abort))) flag_abort(abort, a.status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
        };
        for (int j = 0; j < n_kt; ++j) {
            const int sb = j & 1;
            const uint32_t tS = tmem + lane_addr + Cfg::T_S + sb * 128;
            const int64_t lim64 = kmax - int64_t(j) * BN;  // columns <= lim are visible
            const int lim = int(lim64 < -1 ? -1 : (lim64 > BN ? BN : lim64));
            wait(&s_full[sb], uint32_t(j >> 1) & 1);
            // this half row of S, scaled to log2 units and masked, into registers; the S buffer is free
            // for the tile after next as soon as it has been read.  Then the row max (this half, then both
            // halves through shared memory).
            static_assert(HC == 64, "two chunks of 32 columns per half row");
            float x[HC];
            float mx = -INFINITY;
            if (ok) {
                uint32_t v0[32], v1[32];
                tmem_ld32(tS + half * HC, v0);
                tmem_ld32(tS + half * HC + 32, v1);
                tmem_ld_wait_regs(v0);
                tmem_ld_wait_regs(v1);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    x[e] = half * HC + e <= lim ? __uint_as_float(v0[e]) * c : -INFINITY;
                    x[32 + e] = half * HC + 32 + e <= lim ? __uint_as_float(v1[e]) * c : -INFINITY;
                }
#pragma unroll
                for (int e = 0; e < HC; ++e) mx = fmaxf(mx, x[e]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[sb]);
            {
                float *slot = xm + (j & 1) * 256;  // alternate by tile: the other half may still read the last
                slot[half * 128 + r] = mx;
                named_bar_sync(1, 256);
                mx = fmaxf(slot[r], slot[128 + r]);
            }
            const float m_new = fmaxf(m_ref, mx);
            const bool need = m_new > m_ref + 8.f;  // also the first finite max
            if (__any_sync(0xffffffffu, need)) {
                const float f = need ? ex2(m_ref - m_new) : 1.f;  // exp2(-inf) = 0 on the first raise
                if (j > 0) {  // O holds earlier tiles: scale this row once their GEMMs have completed
                    wait(o_done, uint32_t(j - 1) & 1);
                    if (ok) {  // this half's columns of the row of O
#pragma unroll
                        for (int ch = 0; ch < HD / 32; ++ch) {
                            const int o0 = half * HD + ch * 32;
                            uint32_t v[32];
                            tmem_ld32(tmem + lane_addr + Cfg::T_O + o0, v);
                            tmem_ld_wait_regs(v);
#pragma unroll
                            for (int e0 = 0; e0 < 32; e0 += 8) {
                                uint32_t w[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(__uint_as_float(v[e0 + e]) * f);
                                tmem_st8(tmem + lane_addr + Cfg::T_O + o0 + e0, w);
                            }
                        }
                        tmem_st_wait();
                    }
                }
                if (need) {
                    l *= f;
                    m_ref = m_new;
                }
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;  // no visible key yet: every P is 0
            // pass 2: P = exp2(x - m) into TMEM, once the O GEMM two tiles back has read its buffer
            if (j >= 2) wait(&p_free[sb], uint32_t((j >> 1) - 1) & 1);
            if (ok) {
#pragma unroll
                for (int ch = 0; ch < HC / 32; ++ch) {
                    const int c0 = half * HC + ch * 32;
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float p0 = ex2(x[ch * 32 + e] - m_use), p1 = ex2(x[ch * 32 + e + 1] - m_use);
                        l += p0 + p1;
                        pk[e / 2] = pack2<T>(p0, p1);
                    }
                    uint32_t w0[8], w1[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        w0[e] = pk[e];
                        w1[e] = pk[8 + e];
                    }
                    tmem_st8(tmem + lane_addr + Cfg::T_P + sb * 64 + c0 / 2, w0);
                    tmem_st8(tmem + lane_addr + Cfg::T_P + sb * 64 + c0 / 2 + 8, w1);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[sb]);
        }
        // ---- epilogue: O / l (16-bit, row per thread, this half's columns) and LSE (natural log)
        {
            float *slot = xm + (n_kt & 1) * 256;  // not the slot the last tile's maxima went through
            slot[half * 128 + r] = l;
            named_bar_sync(1, 256);
            l = slot[r] + slot[128 + r];
        }
        if (n_kt > 0) wait(o_done, uint32_t(n_kt - 1) & 1);
        const bool row_ok = i < lq;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T *O = static_cast<T *>(a.o.ptr) + (kPacked ? 0 : int64_t(q_b) * a.o.sb) + hq * a.o.sh + (q_row0 + i) * a.o.ss;
#pragma unroll
        for (int ch = 0; ch < HD / 32; ++ch) {
            const int o0 = half * HD + ch * 32;
            uint32_t v[32];
            if (n_kt > 0 && ok) {
                tmem_ld32(tmem + lane_addr + Cfg::T_O + o0, v);
                tmem_ld_wait_regs(v);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
            if (row_ok) {
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint4 o;
                    o.x = pack2<T>(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
                    o.y = pack2<T>(__uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv);
                    o.z = pack2<T>(__uint_as_float(v[e + 4]) * inv, __uint_as_float(v[e + 5]) * inv);
                    o.w = pack2<T>(__uint_as_float(v[e + 6]) * inv, __uint_as_float(v[e + 7]) * inv);
                    *reinterpret_cast<uint4 *>(O + o0 + e) = o;
                }
            }
        }
        if (row_ok && half == 0) {
            const float lse = l > 0.f ? (m_ref + __log2f(l)) / kLog2e : INFINITY;
            const int64_t idx = kPacked ? hq * a.t_q + q_row0 + i : (int64_t(q_b) * a.h + hq) * lq + i;
            a.lse_out[idx] = lse;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::T_COLS);
    }
}

// ===================================================================== host

namespace {

template <class T, int D, class Geo> cudaError_t run_fwd(const DenseArgs &a, const Geo &g, cudaStream_t s)
{
    using Cfg = FwdCfg<D>;
    constexpr bool packed = FwdPacked<Geo>::value;
    int64_t units;
    if (packed) units = (g.ws_rows() / Cfg::BM) * a.h;
    else units = (g.q_len(0) + Cfg::BM - 1) / Cfg::BM * a.h * a.nseq;
    if (units == 0) return cudaSuccess;
    if (units > INT32_MAX) return cudaErrorInvalidValue;
    FwdParams prm;
    prm.a = a;
    const int64_t nb = packed ? 1 : a.nseq;
    const int64_t sq = packed ? a.t_q : g.q_len(0), skv = packed ? a.t_kv : g.kv_len(0);
    if (!tmap_view16(&prm.tm_q, a.q, a.dtype, D, sq, a.h, nb, Cfg::BM)) return cudaErrorInvalidValue;
    if (skv > 0) {
        if (!tmap_view16(&prm.tm_k, a.k, a.dtype, D, skv, a.h_kv, nb, Cfg::BN) ||
            !tmap_view16(&prm.tm_v, a.v, a.dtype, D, skv, a.h_kv, nb, Cfg::BN))
            return cudaErrorInvalidValue;
    } else {
        prm.tm_k = prm.tm_v = prm.tm_q;  // never read: no key tiles
    }
    auto k = dense_fwd_tc_kernel<T, D, Geo>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s)) != cudaSuccess) return e;
    return launch_kernel(k, dim3(unsigned(units)), dim3(Cfg::THREADS), Cfg::SMEM_ALLOC, s, false, prm, g);
}

template <class Geo> cudaError_t fwd(const DenseArgs &a, const Geo &g, cudaStream_t s)
{
    if (a.d == 64)
        return a.dtype == ATTN_F16 ? run_fwd<__half, 64>(a, g, s) : run_fwd<__nv_bfloat16, 64>(a, g, s);
    return a.dtype == ATTN_F16 ? run_fwd<__half, 128>(a, g, s) : run_fwd<__nv_bfloat16, 128>(a, g, s);
}

}  // namespace

cudaError_t launch_dense_fwd(const DenseArgs &a, const FixedGeo &g, cudaStream_t s) { return fwd(a, g, s); }
cudaError_t launch_dense_fwd(const DenseArgs &a, const PackedGeo &g, cudaStream_t s) { return fwd(a, g, s); }

}  // namespace attn
