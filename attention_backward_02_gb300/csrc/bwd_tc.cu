// bwd_tc.cu -- tensor-core SDPA backward for sm_103a (tcgen05 + TMA + TMEM).
//
// FlashAttention-2 backward (cuDNN-frontend sample
// "51_scaled_dot_product_attention_backward": backward from the saved
// (B,H,S,1) stats, no stored P), with the gradient formulas of the Ascend page
// "aclnnNsaSelectedAttentionGrad", Function / Formula (dV = P^T dY,
// dQ = dS K scale, dK = dS^T Q scale).
//
// One CTA owns a tile of BN = 128 key/value rows of one (sequence, kv head)
// and walks every (query head of the group, query tile of BM rows) that sees
// it.  Everything is computed transposed, so the 128 key rows are the MMA M
// dimension and the TMEM lanes:
//   S^T  = K Q^T           M=128 (keys) N=BM  K=D    A=K  (smem, K-major) B=Q  (K-major)
//   dP^T = V dO^T          M=128        N=BM  K=D    A=V  (smem, K-major) B=dO (K-major)
//   P^T  = exp2(S^T scale log2 e - LSE log2 e),  dS^T = P^T (dP^T - D)   (CUDA cores)
//   dV  += P^T dO          M=128        N=D   K=BM   A=P^T (TMEM, 16-bit)   B=dO (MN-major)
//   dK  += dS^T Q          M=128        N=D   K=BM   A=dS^T (smem, K-major) B=Q  (MN-major)
//   dQ   = dS K     (D=64) M=BM=128     N=64  K=128  A=dS (MN-major)       B=K  (MN-major)
//   dQ^T = K^T dS^T (D=128) M=D=128     N=BM=64 K=128 A=K^T (MN-major)     B=dS^T (MN-major)
// dV, dK stay in TMEM for the whole tile and are written once; each dQ tile
// is staged in shared memory and added into the fp32 accumulator with a TMA
// reduce-add.  TMEM: S^T BM + dP^T BM + P^T BM/2 + dV D + dK D + dQ 64 columns
// (512 at D = 64, 480 at D = 128).
//
// Pipeline.  The MMA warp issues S/dP of query tile i and then dV/dK/dQ of
// tile i-1, so the tensor cores run tile i-1's three GEMMs while the softmax
// warps turn tile i's S/dP into P/dS.  Two 32 KB shared buffers alternate
// per query tile: tile i writes its dS into one while tile i-1's GEMMs read
// their dS from the other, which, once they complete, stages tile i-1's dQ
// for the reduce-add.  P (16-bit, packed) waits in registers until tile
// i-1's dV GEMM has released the P columns of TMEM.  Q, dO and the LSE / D
// vectors stream through a 3-stage ring.
//
// Roles (320 threads): warp 0 issues TMA loads, warp 1 issues the MMAs,
// warps 2..9 do the element-wise work (warp w reads TMEM lanes
// 32 (w % 4) .. + 31; the two warps on the same lanes split the columns), the
// dQ staging and the dK / dV epilogue.
//
// Causal masking: query tiles entirely before the first query that sees the
// key tile are skipped; the rest are masked per element when needed.  Key
// rows past the sequence end are masked by row; query rows past it have
// LSE = +inf in the workspace and so P = 0.
//
// Every barrier wait is bounded (about a second).  On a timeout the thread
// sets ATTN_DEV_TIMEOUT in the status word and an abort flag in shared
// memory; from then on every wait of the CTA fails fast and all work is
// skipped while the control flow (and so every named barrier) stays the same;
// the CTA drains its in-flight copies and MMAs, frees its TMEM and exits.
#include <cudaTypedefs.h>

#include <climits>
#include <type_traits>

#include "plan.h"
#include "sm103.cuh"
#include "tc_util.cuh"

namespace attn {
using namespace sm103;

template <int D>
struct TcCfg {
    static constexpr int BN = 128;                  // key rows per CTA tile
    static constexpr int BM = D == 64 ? 128 : 64;   // query rows per iteration
    static constexpr int NST = 3;                   // Q / dO ring stages
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int DS_BYTES = BN * BM * 2;
    static constexpr int DQ_BYTES = BM * D * 4;
    static constexpr int X_BYTES = DS_BYTES > DQ_BYTES ? DS_BYTES : DQ_BYTES;  // dS / dQ buffer
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KV_BYTES;
    static constexpr int OFF_Q = OFF_V + KV_BYTES;            // NST stages
    static constexpr int OFF_DO = OFF_Q + NST * Q_BYTES;      // NST stages
    static constexpr int OFF_X = OFF_DO + NST * Q_BYTES;      // 2 dS / dQ buffers
    static constexpr int OFF_LSE = OFF_X + 2 * X_BYTES;       // NST x BM floats
    static constexpr int OFF_DVEC = OFF_LSE + NST * BM * 4;   // NST x BM floats
    static constexpr int OFF_BAR = OFF_DVEC + NST * BM * 4;
    static constexpr int OFF_MISC = OFF_BAR + 24 * 8;
    static constexpr int SMEM = OFF_MISC + 64;
    static constexpr int SMEM_ALLOC = SMEM + 1024;            // room to align the base to 1024
    static constexpr int T_S = 0, T_DP = BM, T_P = 2 * BM, T_DV = 2 * BM + BM / 2, T_DK = T_DV + D,
                         T_DQ = T_DK + D;
    static constexpr int T_COLS = 512;
    static_assert(T_DQ + 64 <= T_COLS, "TMEM budget");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_dq, tm_dk, tm_dv;
    DenseArgs a;
};

using namespace tc;

namespace {

// Query tiles that see the key tile starting at j0: [qt0, qt0 + nq).
template <int BM>
__device__ __forceinline__ void query_tiles(int mask, int64_t j0, int64_t lq, int64_t lkv, int *qt0, int *nq)
{
    const int64_t i_lo = first_query_seeing(mask, j0, lq, lkv);
    if (lq <= 0 || lkv <= 0 || i_lo >= lq) {
        *qt0 = 0;
        *nq = 0;
        return;
    }
    *qt0 = int(i_lo / BM);
    *nq = int((lq + BM - 1) / BM) - *qt0;
}

template <class Geo> struct IsPacked : std::false_type {};
template <> struct IsPacked<PackedGeo> : std::true_type {};

}  // namespace

template <class T, int D, class Geo>
__global__ void __launch_bounds__(320, 1) dense_bwd_tc_kernel(const __grid_constant__ TcParams p, const Geo geo)
{
    using Cfg = TcCfg<D>;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, NST = Cfg::NST;
    constexpr int HC = BM / 2;  // query columns per softmax thread
    constexpr bool kPacked = IsPacked<Geo>::value;
    constexpr int kType = std::is_same<T, __half>::value ? 0 : 1;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *kv_full = bars + 0, *kv_empty = bars + 1, *q_full = bars + 2, *q_empty = bars + 2 + NST;
    uint64_t *s_full = bars + 2 + 2 * NST, *s_free = s_full + 1, *p_ready = s_full + 2, *mma_done = s_full + 3;
    uint64_t *drain = s_full + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + Cfg::OFF_MISC + 8);
    const DenseArgs &a = p.a;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        *abort = 0;
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, 8);
        mbar_init(p_ready, 8);
        mbar_init(mma_done, 1);
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, Cfg::T_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // the preprocess (LSE, D, zeroed dQ accumulator) has completed

    // ---- work units: (sequence b, kv head g) and its key tiles; unit
    // index = first tile * (nseq * h_kv) + (b * h_kv + g), so for a causal
    // fixed-length batch the units come heaviest first.  The CTA takes units
    // c, 2C-1-c, 2C+c, ... (C CTAs), which evens out their total work.
    const int64_t nheads = a.nseq * a.h_kv;
    const int64_t tile_step = a.deterministic ? a.n_part : INT64_MAX / 2;
    const int G = int(a.h / a.h_kv);
#define ATTN_FOR_EACH_UNIT                                                                                    \
    for (int64_t round_ = 0;; ++round_) {                                                                     \
        const int64_t unit = round_ * gridDim.x +                                                             \
                             ((round_ & 1) ? int64_t(gridDim.x) - 1 - blockIdx.x : int64_t(blockIdx.x));      \
        if (unit >= a.tc_units) break;                                                                        \
        const int64_t bg = unit % nheads, first_tile = unit / nheads;                                         \
        const int64_t b = bg / a.h_kv, g = bg % a.h_kv;                                                       \
        const int64_t part = a.deterministic ? first_tile : 0;                                                \
        const int64_t lq = geo.q_len(b), lkv = geo.kv_len(b);                                                 \
        const int64_t ntiles = (lkv + BN - 1) / BN;                                                           \
        const int q_b = kPacked ? 0 : int(b), kv_b = q_b;                                                     \
        const int64_t q_row0 = kPacked ? geo.q_start(b) : 0, kv_row0 = kPacked ? geo.kv_start(b) : 0;         \
        (void)part;                                                                                           \
        (void)q_row0;                                                                                         \
        (void)kv_row0;
#define ATTN_END_UNITS }

    uint8_t *sK = smem + Cfg::OFF_K, *sV = smem + Cfg::OFF_V, *sX = smem + Cfg::OFF_X;

    if (warp == 0) {
        // ================================================= TMA producer
        if (elect_one()) {
            prefetch_tmap(&p.tm_q); prefetch_tmap(&p.tm_k); prefetch_tmap(&p.tm_v); prefetch_tmap(&p.tm_do);
            bool ok = true;
            int64_t kt = 0, qi = 0, q_armed = 0, kv_armed = 0;  // loads started (for the drain below)
            ATTN_FOR_EACH_UNIT
            for (int64_t jt = first_tile; jt < ntiles; jt += tile_step) {
                const int64_t j0 = jt * BN;
                int qt0, nq;
                query_tiles<BM>(a.mask, j0, lq, lkv, &qt0, &nq);
                const int n_iter = G * nq;
                if (n_iter == 0) continue;
                // Q / dO of query tile `it` (global iteration index x) into its ring stage
                auto load_q = [&](int it, int64_t x) {
                    const int st = int(x % NST);
                    const int64_t use = x / NST;
                    if (use > 0 && ok && !(ok = mbar_wait(&q_empty[st], uint32_t(use - 1) & 1, abort)))
                        flag_abort(abort, a.status);
                    if (!ok) return;
                    const int64_t hq = g * G + it / nq, i0 = int64_t(qt0 + it % nq) * BM;
                    uint8_t *sQ = smem + Cfg::OFF_Q + st * Cfg::Q_BYTES, *sdO = smem + Cfg::OFF_DO + st * Cfg::Q_BYTES;
                    q_armed = x + 1;
                    mbar_arrive_expect_tx(&q_full[st], 2 * Cfg::Q_BYTES + 2 * BM * 4);
                    for (int c = 0; c < D / 64; ++c) {
                        tma_load_4d(sQ + c * BM * 128, &p.tm_q, &q_full[st], c * 64, int(q_row0 + i0), int(hq), q_b);
                        tma_load_4d(sdO + c * BM * 128, &p.tm_do, &q_full[st], c * 64, int(q_row0 + i0), int(hq), q_b);
                    }
                    const int64_t wrow = hq * a.t_pad + geo.ws_start(b) + i0;
                    bulk_load(smem + Cfg::OFF_LSE + st * BM * 4, a.lse2 + wrow, BM * 4, &q_full[st]);
                    bulk_load(smem + Cfg::OFF_DVEC + st * BM * 4, a.dvec + wrow, BM * 4, &q_full[st]);
                };
                // the first query tile does not need the key tile: load it before waiting for K / V
                load_q(0, qi);
                if (kt > 0 && ok && !(ok = mbar_wait(kv_empty, uint32_t(kt - 1) & 1, abort))) flag_abort(abort, a.status);
                if (ok) {
                    kv_armed = kt + 1;
                    mbar_arrive_expect_tx(kv_full, 2 * Cfg::KV_BYTES);
                    for (int c = 0; c < D / 64; ++c) {
                        tma_load_4d(sK + c * BN * 128, &p.tm_k, kv_full, c * 64, int(kv_row0 + j0), int(g), kv_b);
                        tma_load_4d(sV + c * BN * 128, &p.tm_v, kv_full, c * 64, int(kv_row0 + j0), int(g), kv_b);
                    }
                }
                ++qi;
                for (int it = 1; it < n_iter; ++it, ++qi) load_q(it, qi);
                ++kt;
            }
            ATTN_END_UNITS
            if (!ok) {
                // let every copy this thread started land before the CTA exits
                volatile int never = 0;
                for (int64_t x = q_armed - NST; x < q_armed; ++x)
                    if (x >= 0) mbar_wait(&q_full[x % NST], uint32_t(x / NST) & 1, &never, 100000000ull);
                if (kv_armed > 0) mbar_wait(kv_full, uint32_t(kv_armed - 1) & 1, &never, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ================================================= MMA issuer
        if (elect_one()) {
            constexpr uint32_t idS = idesc_f16(128, BM, kType, 0, 0);
            constexpr uint32_t idDV = idesc_f16(128, D, kType, 0, 1);
            constexpr uint32_t idDQ = idesc_f16(128, 64, kType, 1, 1);
            const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
            bool ok = true;
            int64_t kt = 0, qi = 0;
            // dV, dK, dQ of query tile x (global index) whose P / dS are ready
            auto grads = [&](int64_t x, bool first) {
                const int st = int(x % NST);
                const uint32_t adS = smem_u32(sX + (x & 1) * Cfg::X_BYTES);
                const uint32_t aQ = smem_u32(smem + Cfg::OFF_Q + st * Cfg::Q_BYTES);
                const uint32_t adO = smem_u32(smem + Cfg::OFF_DO + st * Cfg::Q_BYTES);
                for (int kk = 0; kk < BM / 16; ++kk)
                    mma_f16_ts(tmem + Cfg::T_DV, tmem + Cfg::T_P + kk * 8, desc_mn(adO, BM, kk), idDV, !first || kk > 0);
                for (int kk = 0; kk < BM / 16; ++kk)
                    mma_f16_ss(tmem + Cfg::T_DK, desc_kmaj(adS, BN, kk), desc_mn(aQ, BM, kk), idDV, !first || kk > 0);
                for (int kk = 0; kk < BN / 16; ++kk) {
                    if (D == 64)
                        mma_f16_ss(tmem + Cfg::T_DQ, desc_mn(adS, BN, kk), desc_mn(aK, BN, kk), idDQ, kk > 0);
                    else
                        mma_f16_ss(tmem + Cfg::T_DQ, desc_mn(aK, BN, kk), desc_mn(adS, BN, kk), idDQ, kk > 0);
                }
                mma_commit(mma_done);
                mma_commit(&q_empty[st]);
            };
            ATTN_FOR_EACH_UNIT
            for (int64_t jt = first_tile; jt < ntiles; jt += tile_step) {
                const int64_t j0 = jt * BN;
                int qt0, nq;
                query_tiles<BM>(a.mask, j0, lq, lkv, &qt0, &nq);
                const int n_iter = G * nq;
                if (n_iter == 0) continue;
                if (ok && !(ok = mbar_wait(kv_full, uint32_t(kt) & 1, abort))) flag_abort(abort, a.status);
                tc_fence_after();
                for (int it = 0; it < n_iter; ++it, ++qi) {
                    const int st = int(qi % NST);
                    const uint32_t aQ = smem_u32(smem + Cfg::OFF_Q + st * Cfg::Q_BYTES);
                    const uint32_t adO = smem_u32(smem + Cfg::OFF_DO + st * Cfg::Q_BYTES);
                    if (ok && !(ok = mbar_wait(&q_full[st], uint32_t(qi / NST) & 1, abort))) flag_abort(abort, a.status);
                    // S^T / dP^T of the previous query tile have been read out of TMEM
                    if (qi > 0 && ok && !(ok = mbar_wait(s_free, uint32_t(qi - 1) & 1, abort)))
                        flag_abort(abort, a.status);
                    tc_fence_after();
                    if (ok) {
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_f16_ss(tmem + Cfg::T_S, desc_kmaj(aK, BN, kk), desc_kmaj(aQ, BM, kk), idS, kk > 0);
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_f16_ss(tmem + Cfg::T_DP, desc_kmaj(aV, BN, kk), desc_kmaj(adO, BM, kk), idS, kk > 0);
                        mma_commit(s_full);
                    }
                    if (it > 0) {
                        if (ok && !(ok = mbar_wait(p_ready, uint32_t(qi - 1) & 1, abort))) flag_abort(abort, a.status);
                        tc_fence_after();
                        if (ok) grads(qi - 1, it == 1);
                    }
                }
                if (ok && !(ok = mbar_wait(p_ready, uint32_t(qi - 1) & 1, abort))) flag_abort(abort, a.status);
                tc_fence_after();
                if (ok) {
                    grads(qi - 1, n_iter == 1);
                    mma_commit(kv_empty);  // K / V free for the next tile once these GEMMs finish
                }
                ++kt;
            }
            ATTN_END_UNITS
            // wait for every MMA this thread issued before TMEM is freed
            volatile int never = 0;
            mma_commit(drain);
            mbar_wait(drain, 0, &never, 100000000ull);
        }
    } else {
        // ================================================= P / dS, dQ, dK / dV
        const int lg = warp & 3, half = (warp - 2) >> 2;
        const uint32_t lane_addr = uint32_t(lg * 32) << 16;
        const int r = lg * 32 + lane;  // TMEM lane of this thread
        const float sc = a.scale * kLog2e;
        const bool leader = warp == 2 && lane == 0;
        const uint32_t aX = smem_u32(sX);
        T *dK = static_cast<T *>(a.dK.ptr), *dV = static_cast<T *>(a.dV.ptr);
        bool ok = true;
        int64_t kt = 0, qi = 0;

        // dQ of query tile x (head hq, first row i0), whose GEMMs just completed and released
        // dS buffer x & 1 -> staged there -> TMA add-reduce into the fp32 accumulator
        auto stage_dq = [&](int64_t x, int64_t hq, int64_t row_base, int64_t i0) {
            const uint32_t adQ = aX + uint32_t(x & 1) * Cfg::X_BYTES;
            uint8_t *sdQ = sX + (x & 1) * Cfg::X_BYTES;
            ok = bar_and(1, 256, ok);
            if (ok) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_addr + Cfg::T_DQ + half * 32, v);
                tmem_ld_wait();
                if (D == 64) {  // lane = query row r, columns = head dims [32 half, 32 half + 32)
                    const uint32_t base = adQ + uint32_t(half * BM * 128 + r * 128);
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        st_shared_v4(base + (uint32_t(ch ^ (r & 7)) << 4), v[4 * ch], v[4 * ch + 1], v[4 * ch + 2],
                                     v[4 * ch + 3]);
                } else {  // lane = head dim r, columns = query rows [32 half, 32 half + 32)
                    const uint32_t base = adQ + uint32_t(lg * BM * 128) + uint32_t((lane & 3) << 2);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int c = half * 32 + e;
                        st_shared_f32(base + uint32_t(c * 128) + (uint32_t((lane >> 2) ^ (c & 7)) << 4), v[e]);
                    }
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 256);
            if (leader && ok) {
                const int64_t row0 = row_base + hq * a.t_pad + i0;
                for (int box = 0; box < D / 32; ++box)
                    tma_reduce_add_2d(&p.tm_dq, sdQ + box * BM * 128, box * 32, int(row0));
                bulk_commit();
            }
        };

        ATTN_FOR_EACH_UNIT
        const int64_t shift = a.mask == ATTN_CAUSAL_BOTTOM_RIGHT ? lkv - lq : 0;
        for (int64_t jt = first_tile; jt < ntiles; jt += tile_step) {
            const int64_t j0 = jt * BN, j = j0 + r;
            const bool row_ok = j < lkv;
            const int64_t kv_tok = kv_row0 + j;
            const int64_t offk = kv_b * a.dK.sb + g * a.dK.sh + kv_tok * a.dK.ss;
            const int64_t offv = kv_b * a.dV.sb + g * a.dV.sh + kv_tok * a.dV.ss;
            int qt0, nq;
            query_tiles<BM>(a.mask, j0, lq, lkv, &qt0, &nq);
            const int n_iter = G * nq;
            if (n_iter == 0) {  // no query sees these keys: dK = dV = 0
                if (row_ok)
                    for (int x = half * (D / 2); x < (half + 1) * (D / 2); x += 8) {
                        *reinterpret_cast<uint4 *>(dK + offk + x) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(dV + offv + x) = make_uint4(0, 0, 0, 0);
                    }
                continue;
            }
            int64_t prev_hq = 0, prev_i0 = 0;
            for (int it = 0; it < n_iter; ++it, ++qi) {
                const int st = int(qi % NST);
                const int64_t hq = g * G + it / nq, i0 = int64_t(qt0 + it % nq) * BM;
                if (ok && !(ok = mbar_wait(&q_full[st], uint32_t(qi / NST) & 1, abort))) flag_abort(abort, a.status);
                if (ok && !(ok = mbar_wait(s_full, uint32_t(qi) & 1, abort))) flag_abort(abort, a.status);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                // dS buffer qi & 1 last staged dQ of tile qi - 2: that reduce must have read it
                if (leader) bulk_wait_read0();
                named_bar_sync(1, 256);
                const uint32_t adS = aX + uint32_t(qi & 1) * Cfg::X_BYTES;
                // ---- P^T (kept packed until TMEM frees) and dS^T (to shared memory now)
                uint32_t pk[HC / 2];
                if (ok) {
                    const uint32_t a_lse = smem_u32(smem + Cfg::OFF_LSE + st * BM * 4);
                    const uint32_t a_dv = smem_u32(smem + Cfg::OFF_DVEC + st * BM * 4);
                    // first visible query column of this key row; everything is masked past the sequence
                    const int64_t cmin64 = !row_ok ? INT64_MAX : (a.mask ? j - shift - i0 : INT64_MIN);
                    const int cmin = int(cmin64 < -1 ? -1 : (cmin64 > BM ? BM : cmin64));
                    const bool any_mask = __any_sync(0xffffffffu, cmin > half * HC);
                    // chunks of 16 columns; the TMEM loads of chunk cc + 1 are issued before
                    // chunk cc is computed
                    constexpr int NCH = HC / 16;
                    uint32_t sbuf[2][16], dbuf[2][16];
                    tmem_ld16(tmem + lane_addr + Cfg::T_S + half * HC, sbuf[0]);
                    tmem_ld16(tmem + lane_addr + Cfg::T_DP + half * HC, dbuf[0]);
#pragma unroll
                    for (int cc = 0; cc < NCH; ++cc) {
                        const int col0 = half * HC + cc * 16, cur = cc & 1;
                        tmem_ld_wait_regs(sbuf[cur], dbuf[cur]);
                        if (cc + 1 < NCH) {
                            tmem_ld16(tmem + lane_addr + Cfg::T_S + col0 + 16, sbuf[cur ^ 1]);
                            tmem_ld16(tmem + lane_addr + Cfg::T_DP + col0 + 16, dbuf[cur ^ 1]);
                        }
                        uint32_t dk[8];
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const float4 l4 = ld_shared_f4(a_lse + uint32_t(col0 + 4 * q4) * 4);
                            const float4 d4 = ld_shared_f4(a_dv + uint32_t(col0 + 4 * q4) * 4);
                            const float lse4[4] = {l4.x, l4.y, l4.z, l4.w}, dv4[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const int e = 4 * q4 + 2 * h2, c = col0 + e;
                                float x0 = fmaf(__uint_as_float(sbuf[cur][e]), sc, -lse4[2 * h2]);
                                float x1 = fmaf(__uint_as_float(sbuf[cur][e + 1]), sc, -lse4[2 * h2 + 1]);
                                if (any_mask) {
                                    x0 = c >= cmin ? x0 : -INFINITY;
                                    x1 = c + 1 >= cmin ? x1 : -INFINITY;
                                }
                                const float g0 = __uint_as_float(dbuf[cur][e]) - dv4[2 * h2];
                                const float g1 = __uint_as_float(dbuf[cur][e + 1]) - dv4[2 * h2 + 1];
                                pk[cc * 8 + 2 * q4 + h2] = p_and_ds<T>(x0, x1, g0, g1, &dk[2 * q4 + h2]);
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const uint32_t off = sw128_offset(uint32_t(r), uint32_t(col0 + 8 * q), BN);
                            st_shared_v4(adS + off, dk[4 * q], dk[4 * q + 1], dk[4 * q + 2], dk[4 * q + 3]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free);  // S^T / dP^T may be overwritten
                // ---- the previous query tile's GEMMs have released P (TMEM) and dS (smem); its dQ is ready
                if (it > 0) {
                    if (ok && !(ok = mbar_wait(mma_done, uint32_t(qi - 1) & 1, abort))) flag_abort(abort, a.status);
                    ok = __all_sync(0xffffffffu, ok);
                    tc_fence_after();
                    stage_dq(qi - 1, prev_hq, part * a.h * a.t_pad + geo.ws_start(b), prev_i0);
                }
                if (ok) {
#pragma unroll
                    for (int c8 = 0; c8 < HC / 16; ++c8) {
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[e] = pk[c8 * 8 + e];
                        tmem_st8(tmem + lane_addr + Cfg::T_P + half * (HC / 2) + c8 * 8, w);
                    }
                    tmem_st_wait();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_ready);
                prev_hq = hq;
                prev_i0 = i0;
            }
            // ---- last query tile of this key tile: its dQ, then dK and dV
            if (ok && !(ok = mbar_wait(mma_done, uint32_t(qi - 1) & 1, abort))) flag_abort(abort, a.status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            stage_dq(qi - 1, prev_hq, part * a.h * a.t_pad + geo.ws_start(b), prev_i0);
            // dK, dV tiles: staged in the two dS / dQ buffers (swizzled like the loads) and
            // written by TMA, unless the tile runs past a packed sequence's end (per-row stores)
            const bool tma_out = !kPacked || j0 + BN <= lkv;
            if (tma_out) {
                if (leader) bulk_wait_read0();  // the last dQ reduce has read its buffer
                ok = bar_and(1, 256, ok);
            }
            if (ok) {
#pragma unroll
                for (int cc = 0; cc < D / 64; ++cc) {
                    const int col0 = half * (D / 2) + cc * 32;
                    uint32_t vv[32], kk[32];
                    tmem_ld32(tmem + lane_addr + Cfg::T_DV + col0, vv);
                    tmem_ld32(tmem + lane_addr + Cfg::T_DK + col0, kk);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 ov, ok4;
                        ov.x = pack2<T>(__uint_as_float(vv[8 * q + 0]), __uint_as_float(vv[8 * q + 1]));
                        ov.y = pack2<T>(__uint_as_float(vv[8 * q + 2]), __uint_as_float(vv[8 * q + 3]));
                        ov.z = pack2<T>(__uint_as_float(vv[8 * q + 4]), __uint_as_float(vv[8 * q + 5]));
                        ov.w = pack2<T>(__uint_as_float(vv[8 * q + 6]), __uint_as_float(vv[8 * q + 7]));
                        ok4.x = pack2<T>(__uint_as_float(kk[8 * q + 0]) * a.scale, __uint_as_float(kk[8 * q + 1]) * a.scale);
                        ok4.y = pack2<T>(__uint_as_float(kk[8 * q + 2]) * a.scale, __uint_as_float(kk[8 * q + 3]) * a.scale);
                        ok4.z = pack2<T>(__uint_as_float(kk[8 * q + 4]) * a.scale, __uint_as_float(kk[8 * q + 5]) * a.scale);
                        ok4.w = pack2<T>(__uint_as_float(kk[8 * q + 6]) * a.scale, __uint_as_float(kk[8 * q + 7]) * a.scale);
                        if (tma_out) {
                            const uint32_t off = sw128_offset(uint32_t(r), uint32_t(col0 + 8 * q), BN);
                            st_shared_v4(aX + off, ov.x, ov.y, ov.z, ov.w);
                            st_shared_v4(aX + Cfg::X_BYTES + off, ok4.x, ok4.y, ok4.z, ok4.w);
                        } else if (row_ok) {
                            *reinterpret_cast<uint4 *>(dV + offv + col0 + 8 * q) = ov;
                            *reinterpret_cast<uint4 *>(dK + offk + col0 + 8 * q) = ok4;
                        }
                    }
                }
            }
            if (tma_out) {
                fence_proxy_async_smem();
                named_bar_sync(1, 256);
                if (leader && ok) {
                    for (int c = 0; c < D / 64; ++c) {
                        tma_store_4d(&p.tm_dv, sX + c * BN * 128, c * 64, int(kv_row0 + j0), int(g), kv_b);
                        tma_store_4d(&p.tm_dk, sX + Cfg::X_BYTES + c * BN * 128, c * 64, int(kv_row0 + j0), int(g), kv_b);
                    }
                    bulk_commit();
                }
            }
            // deterministic mode: this tile's dQ adds land before the next tile's (fixed order)
            if (leader && a.deterministic) bulk_wait0();
            ++kt;
        }
        ATTN_END_UNITS
        if (leader) bulk_wait0();
        pdl_trigger();  // the dQ finalize may start launching; it waits for this grid
    }

#undef ATTN_FOR_EACH_UNIT
#undef ATTN_END_UNITS
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::T_COLS);
    }
}

// ===================================================================== host

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// 16-bit [B][H][S][D] view (element strides) as a 4-D map (d, s, h, b), box (64, rows, 1, 1).
bool map_view(CUtensorMap *m, const View &v, int dtype, int64_t d, int64_t s, int64_t h, int64_t b, uint32_t rows)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {cuuint64_t(d), cuuint64_t(s), cuuint64_t(h), cuuint64_t(b)};
    const int64_t sb = b > 1 ? v.sb : s * v.ss;  // unused extent-1 dim: any legal stride
    cuuint64_t strides[3] = {cuuint64_t(v.ss * 2), cuuint64_t(v.sh * 2), cuuint64_t((sb > 0 ? sb : 8) * 2)};
    cuuint32_t box[4] = {64, rows, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(m, dtype == ATTN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                     v.ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool map_dqacc(CUtensorMap *m, float *base, int64_t d, int64_t rows, uint32_t box_rows)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cuuint64_t(d), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(d * 4)};
    cuuint32_t box[2] = {32, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int64_t sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

template <class Geo> int64_t max_kv_len(const Geo &g)
{
    int64_t m = 0;
    for (int64_t b = 0; b < g.nseq; ++b) m = g.kv_len(b) > m ? g.kv_len(b) : m;
    return m;
}

template <class T, int D, class Geo> cudaError_t run_tc(const DenseArgs &a, const Geo &g, cudaStream_t s)
{
    using Cfg = TcCfg<D>;
    constexpr bool packed = IsPacked<Geo>::value;
    const int64_t ntiles = (max_kv_len(g) + Cfg::BN - 1) / Cfg::BN;
    if (ntiles == 0) return cudaSuccess;
    TcParams prm;
    prm.a = a;
    const int64_t nb = packed ? 1 : a.nseq;
    const int64_t sq = packed ? a.t_q : (a.t_q / (a.nseq ? a.nseq : 1));
    const int64_t skv = packed ? a.t_kv : (a.t_kv / (a.nseq ? a.nseq : 1));
    if (sq > 0 && (!map_view(&prm.tm_q, a.q, a.dtype, D, sq, a.h, nb, Cfg::BM) ||
                   !map_view(&prm.tm_do, a.dO, a.dtype, D, sq, a.h, nb, Cfg::BM)))
        return cudaErrorInvalidValue;
    if (!map_view(&prm.tm_k, a.k, a.dtype, D, skv, a.h_kv, nb, Cfg::BN) ||
        !map_view(&prm.tm_v, a.v, a.dtype, D, skv, a.h_kv, nb, Cfg::BN) ||
        !map_view(&prm.tm_dk, a.dK, a.dtype, D, skv, a.h_kv, nb, Cfg::BN) ||
        !map_view(&prm.tm_dv, a.dV, a.dtype, D, skv, a.h_kv, nb, Cfg::BN))
        return cudaErrorInvalidValue;
    if (!map_dqacc(&prm.tm_dq, a.dqacc, D, int64_t(a.n_part) * a.h * a.t_pad, Cfg::BM)) return cudaErrorInvalidValue;
    if (sq == 0) prm.tm_q = prm.tm_do = prm.tm_k;  // never read: no query tiles
    auto k = dense_bwd_tc_kernel<T, D, Geo>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    prm.a.tc_units = (a.deterministic ? a.n_part : ntiles) * a.nseq * a.h_kv;
    const int64_t units = prm.a.tc_units < sm_count() ? prm.a.tc_units : sm_count();
    return launch_kernel(k, dim3(unsigned(units)), dim3(320), Cfg::SMEM_ALLOC, s, true, prm, g);
}

template <class Geo> cudaError_t dispatch(const DenseArgs &a, const Geo &g, cudaStream_t s)
{
    if (a.d == 64)
        return a.dtype == ATTN_F16 ? run_tc<__half, 64>(a, g, s) : run_tc<__nv_bfloat16, 64>(a, g, s);
    return a.dtype == ATTN_F16 ? run_tc<__half, 128>(a, g, s) : run_tc<__nv_bfloat16, 128>(a, g, s);
}

}  // namespace

cudaError_t launch_dense_bwd_main(const DenseArgs &a, const FixedGeo &g, cudaStream_t s) { return dispatch(a, g, s); }
cudaError_t launch_dense_bwd_main(const DenseArgs &a, const PackedGeo &g, cudaStream_t s) { return dispatch(a, g, s); }

}  // namespace attn
