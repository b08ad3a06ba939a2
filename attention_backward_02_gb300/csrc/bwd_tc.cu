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
// dV, dK stay in TMEM for the whole key tile and are written once; each dQ
// tile is read out of TMEM, staged in shared memory half a tile at a time and
// added into the fp32 accumulator with a TMA reduce-add; a kernel chained
// behind this one converts the accumulator into dQ.  Bitwise reproducible dQ
// either way: split (n_part partial buffers, each with one chain of key tiles
// adding in a fixed order) or ordered (one buffer; the adds into a query tile
// go in decreasing key-tile order, each waiting on a per-tile counter in the
// workspace).  TMEM: S^T BM + dP^T BM + P^T BM/2 + dV D + dK D + dQ 64 columns
// (512 at D = 64, 480 at D = 128).
//
// Pipeline.  The MMA warp issues S/dP of query tile i and then dV/dK/dQ of
// tile i-1, so the tensor cores run tile i-1's three GEMMs while the softmax
// warps turn tile i's S/dP into P/dS.  Two 32 KB shared buffers alternate
// per query tile: tile i writes its dS into one while tile i-1's GEMMs read
// their dS from the other.  P (16-bit, packed) waits in registers until tile
// i-1's dV GEMM has released the P columns of TMEM.  At d = 128 the softmax
// warps copy S^T / dP^T into registers and release them before computing, so
// tile i+1's S/dP GEMMs run during tile i's element-wise work.  Q, dO and the
// LSE / D vectors stream through a 3-stage ring.  Fixed-length batches take
// their work units in a longest-first order planned on the host.
//
// Roles (14 warps): warp 0 issues TMA loads, warp 1 the MMAs, warps 2..9 do
// the element-wise work (warp w reads TMEM lanes 32 (w % 4) .. + 31; the two
// warps on the same lanes split the columns), warps 10..13 the dQ staging and
// the dK / dV epilogue.  The ordered dQ mode adds warp 14, which publishes the
// per-tile add counts.
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

#include <algorithm>
#include <climits>
#include <queue>
#include <type_traits>
#include <utility>
#include <vector>

#include "plan.h"
#include "sm103.cuh"
#include "tc_util.cuh"

namespace attn {
using namespace sm103;

template <int D>
struct TcCfg {
    static constexpr int BN = 128;                  // key rows per CTA tile
    static constexpr int BM = D == 64 ? 128 : 64;   // query rows per iteration
    static constexpr int NG = D == 64 ? 2 : 1;      // column groups of 32 per softmax thread
#ifndef ATTN_SDP_RELEASE_GROUPS
    static constexpr int NH = NG;                   // groups of S^T / dP^T columns released one by one
#else
    static constexpr int NH = ATTN_SDP_RELEASE_GROUPS;
#endif
    static constexpr int NST = 3;                   // Q / dO ring stages
#ifndef ATTN_SOFTMAX_WARPS
    static constexpr int NSW = 8;                   // P / dS warps (two or four per TMEM lane quadrant)
#else
    static constexpr int NSW = ATTN_SOFTMAX_WARPS;
#endif
    static constexpr int THREADS = 32 * (2 + NSW + 4);  // TMA, MMA, P / dS, dQ + dK / dV
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int DS_BYTES = BN * BM * 2;
    static constexpr int X_BYTES = DS_BYTES;
    static constexpr int DQS_BYTES = BM * D * 2;             // fp32 dQ, half of the columns
    static constexpr int DQ_BOX_ROWS = D == 64 ? BM : 32;    // rows of one dQ reduce box (32 fp32 wide)
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KV_BYTES;
    static constexpr int OFF_Q = OFF_V + KV_BYTES;            // NST stages
    static constexpr int OFF_DO = OFF_Q + NST * Q_BYTES;      // NST stages
    static constexpr int OFF_X = OFF_DO + NST * Q_BYTES;      // 2 dS buffers
    static constexpr int OFF_DQS = OFF_X + 2 * X_BYTES;       // dQ staging, half a tile
    static constexpr int OFF_LSE = OFF_DQS + DQS_BYTES;       // NST x BM floats
    static constexpr int OFF_DVEC = OFF_LSE + NST * BM * 4;   // NST x BM floats
    static constexpr int OFF_BAR = OFF_DVEC + NST * BM * 4;
    static constexpr int OFF_MISC = OFF_BAR + 32 * 8;
    static constexpr int SMEM = OFF_MISC + 64;
    static constexpr int SMEM_ALLOC = SMEM + 1024;            // room to align the base to 1024
    static constexpr int T_S = 0, T_DP = BM, T_P = 2 * BM, T_DV = 2 * BM + BM / 2, T_DK = T_DV + D,
                         T_DQ = T_DK + D;
    static constexpr int T_COLS = 512;
    static_assert(T_DQ + 64 <= T_COLS, "TMEM budget");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static constexpr int GW = BM / NG / (NSW / 4);  // query columns per P / dS thread and column group
    static_assert(GW % 16 == 0 && (NSW == 8 || NSW == 16), "P / dS work split");
    static_assert(NH == 1 || NH == NG, "release groups");
};

// Work units of each CTA, chosen on the host (see plan_units).  on = 0: the CTAs
// take the units in snake order instead.
constexpr int kSchedCtas = 160;
constexpr int kMailbox = 4;  // ordered dQ mode: counters in flight from the dQ leader to the publishing warp
constexpr int kSchedUnits = 4096;
struct TcSched {
    int32_t on;
    uint16_t off[kSchedCtas + 1];  // CTA c takes unit[off[c]] .. unit[off[c + 1] - 1], in this order
    uint16_t unit[kSchedUnits];
};

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_dq, tm_dk, tm_dv;
    DenseArgs a;
    TcSched sched;
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

// Unit this CTA takes in its round r, or -1 once it has none left.
__device__ __forceinline__ int64_t cta_unit(const TcParams &p, int64_t r)
{
    if (p.sched.on) {
        const int k = int(p.sched.off[blockIdx.x]) + int(r);
        return k < int(p.sched.off[blockIdx.x + 1]) ? int64_t(p.sched.unit[k]) : -1;
    }
    const int64_t u = r * gridDim.x + ((r & 1) ? int64_t(gridDim.x) - 1 - blockIdx.x : int64_t(blockIdx.x));
    return u < p.a.tc_units ? u : -1;
}

template <class Geo> struct IsPacked : std::false_type {};
template <> struct IsPacked<PackedGeo> : std::true_type {};

}  // namespace

// kOrdered: ordered dQ mode (one accumulator, each query tile's adds in a fixed order; needs the planned
// unit order and a cooperative launch).  A template parameter, so the other modes carry none of its code.
template <class T, int D, class Geo, bool kOrdered>
__global__ void __launch_bounds__(TcCfg<D>::THREADS + (kOrdered ? 32 : 0), 1)
    dense_bwd_tc_kernel(const __grid_constant__ TcParams p, const Geo geo)
{
    using Cfg = TcCfg<D>;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, NST = Cfg::NST, NH = Cfg::NH, NG = Cfg::NG;
    constexpr int GW = Cfg::GW;      // query columns per softmax thread and column group
    constexpr bool kPacked = IsPacked<Geo>::value;
    constexpr int kType = std::is_same<T, __half>::value ? 0 : 1;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *kv_full = bars + 0, *kv_empty = bars + 1, *q_full = bars + 2, *q_empty = bars + 2 + NST;
    uint64_t *s_full = bars + 2 + 2 * NST;   // [NH] S^T / dP^T column group written
    uint64_t *s_free = s_full + 2;           // [NH] column group read out by the softmax warps
    uint64_t *p_ready = s_full + 4;          // P^T in TMEM and dS^T in shared memory
    uint64_t *p_free = s_full + 5;           // the dV GEMM has read P^T
    uint64_t *mma_done = s_full + 6;         // all GEMMs of a query tile have completed
    uint64_t *dq_free = s_full + 7;          // the dQ accumulator has been read out
    uint64_t *ds_free = s_full + 8;          // [2] dS buffer: the GEMMs that read it have completed
    uint64_t *acc_free = s_full + 10;        // the dK / dV accumulators have been read out
    uint64_t *drain = s_full + 11;
    // ordered dQ mode: counters handed from the dQ leader to the warp that publishes them
    uint64_t *mb_full = s_full + 12, *mb_empty = s_full + 12 + kMailbox;  // [kMailbox]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + Cfg::OFF_MISC + 8);
    uint32_t **mailbox = reinterpret_cast<uint32_t **>(smem + Cfg::OFF_MISC + 16);  // [kMailbox]
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
        for (int q = 0; q < NH; ++q) {
            mbar_init(&s_full[q], 1);
            mbar_init(&s_free[q], Cfg::NSW);
        }
        mbar_init(p_ready, Cfg::NSW);
        mbar_init(p_free, 1);
        mbar_init(mma_done, 1);
        mbar_init(dq_free, 4);
        mbar_init(&ds_free[0], 1);
        mbar_init(&ds_free[1], 1);
        mbar_init(acc_free, 4);
        mbar_init(drain, 1);
        if (kOrdered)
            for (int k = 0; k < kMailbox; ++k) {
                mbar_init(&mb_full[k], 1);
                mbar_init(&mb_empty[k], 1);
            }
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, Cfg::T_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The preprocess (LSE, D, zeroed dQ accumulator) may still be running: only the loads of
    // LSE / D and the dQ reduce-adds wait for it (pdl_wait below), the Q / K / V / dO loads do not.

    // ---- work units: (sequence b, kv head g) and its key tiles; unit
    // index = first tile * (nseq * h_kv) + (b * h_kv + g).  Each CTA takes
    // the units the host planned for it (cta_unit).
    const int64_t nheads = a.nseq * a.h_kv;
    const int64_t tile_step = a.deterministic ? a.n_part : INT64_MAX / 2;
    const int G = int(a.h / a.h_kv);
#define ATTN_FOR_EACH_UNIT                                                                                    \
    for (int64_t round_ = 0;; ++round_) {                                                                     \
        const int64_t unit = cta_unit(p, round_);                                                             \
        if (unit < 0) break;                                                                                  \
        /* 32-bit divisions: the unit count fits (checked at launch) */                                       \
        const uint32_t ft_ = uint32_t(unit) / uint32_t(nheads), bg_ = uint32_t(unit) - ft_ * uint32_t(nheads);  \
        const uint32_t b_ = bg_ / uint32_t(a.h_kv);                                                           \
        const int64_t bg = bg_, first_tile = ft_;                                                             \
        const int64_t b = b_, g = int64_t(bg_ - b_ * uint32_t(a.h_kv));                                       \
        const int64_t part = a.deterministic ? first_tile : 0;                                                \
        const int64_t lq = geo.q_len(b), lkv = geo.kv_len(b);                                                 \
        const int64_t ntiles = (lkv + BN - 1) / BN;                                                           \
        const int q_b = kPacked ? 0 : int(b), kv_b = q_b;                                                     \
        const int64_t q_row0 = kPacked ? geo.q_start(b) : 0, kv_row0 = kPacked ? geo.kv_start(b) : 0;         \
        (void)part;                                                                                           \
        (void)bg;                                                                                             \
        (void)g;                                                                                              \
        (void)kv_b;                                                                                           \
        (void)q_row0;                                                                                         \
        (void)kv_row0;
#define ATTN_END_UNITS }

    uint8_t *sK = smem + Cfg::OFF_K, *sV = smem + Cfg::OFF_V, *sX = smem + Cfg::OFF_X;

    if (warp == 0) {
        // ================================================= TMA producer
        if (elect_one()) {
            prefetch_tmap(&p.tm_q); prefetch_tmap(&p.tm_k); prefetch_tmap(&p.tm_v); prefetch_tmap(&p.tm_do);
            bool ok = true, pre_done = false;
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
                    // the CTA's first tile gets its inputs before the rest of the ring is filled: every
                    // CTA starts by loading at once, and the later stages would compete for the memory
                    if (x == 1 && ok && !(ok = mbar_wait(&q_full[0], 0, abort))) flag_abort(abort, a.status);
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
                    if (!pre_done) {  // LSE / D come from the preprocess
                        pdl_wait();
                        pre_done = true;
                    }
                    bulk_load(smem + Cfg::OFF_LSE + st * BM * 4, a.lse2 + wrow, BM * 4, &q_full[st]);
                    bulk_load(smem + Cfg::OFF_DVEC + st * BM * 4, a.dvec + wrow, BM * 4, &q_full[st]);
                };
                // the first query tile does not need the key tile: load it before waiting for K / V
                // (except on the very first tile, whose K / V load should start first)
                auto load_kv = [&]() {
                    if (kt > 0 && ok && !(ok = mbar_wait(kv_empty, uint32_t(kt - 1) & 1, abort)))
                        flag_abort(abort, a.status);
                    if (ok) {
                        kv_armed = kt + 1;
                        mbar_arrive_expect_tx(kv_full, 2 * Cfg::KV_BYTES);
                        for (int c = 0; c < D / 64; ++c) {
                            tma_load_4d(sK + c * BN * 128, &p.tm_k, kv_full, c * 64, int(kv_row0 + j0), int(g), kv_b);
                            tma_load_4d(sV + c * BN * 128, &p.tm_v, kv_full, c * 64, int(kv_row0 + j0), int(g), kv_b);
                        }
                    }
                };
                if (kt == 0) load_kv();
                load_q(0, qi);
                // warm L2 with the K / V tile this CTA takes next, so its load does not stall the next unit
                // (on the CTA's first tile only after its second query tile: the first tile's own loads
                // go first)
                auto prefetch_next = [&]() {
                    int64_t nb = b, ng = g, njt = jt + tile_step, nrow0 = kv_row0;
                    int nkv_b = kv_b;
                    bool has = njt < ntiles;
                    if (!has) {
                        const int64_t u2 = cta_unit(p, round_ + 1);
                        if (u2 >= 0) {
                            const uint32_t njt_ = uint32_t(u2) / uint32_t(nheads);
                            const uint32_t bg2 = uint32_t(u2) - njt_ * uint32_t(nheads);
                            nb = bg2 / uint32_t(a.h_kv);
                            ng = int64_t(bg2) - nb * a.h_kv;
                            njt = njt_;
                            nrow0 = kPacked ? geo.kv_start(nb) : 0;
                            nkv_b = kPacked ? 0 : int(nb);
                            has = njt * BN < geo.kv_len(nb);
                        }
                    }
                    if (has)
                        for (int c = 0; c < D / 64; ++c) {
                            tma_prefetch_4d(&p.tm_k, c * 64, int(nrow0 + njt * BN), int(ng), nkv_b);
                            tma_prefetch_4d(&p.tm_v, c * 64, int(nrow0 + njt * BN), int(ng), nkv_b);
                        }
                };
                if (kt > 0 || n_iter == 1) prefetch_next();
                if (kt > 0) load_kv();
                ++qi;
                for (int it = 1; it < n_iter; ++it, ++qi) {
                    load_q(it, qi);
                    if (kt == 0 && it == 1) prefetch_next();
                }
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
            constexpr uint32_t idS = idesc_f16(128, BM / NH, kType, 0, 0);
            constexpr uint32_t idDV = idesc_f16(128, D, kType, 0, 1);
            constexpr uint32_t idDQ = idesc_f16(128, 64, kType, 1, 1);
            const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
            bool ok = true;
            int64_t kt = 0;
            uint32_t qi = 0, st_par = 0;
            int st = 0;
            auto wait = [&](uint64_t *bar, uint32_t parity) {
                if (ok && !(ok = mbar_wait(bar, parity, abort))) flag_abort(abort, a.status);
                tc_fence_after();
            };
            // step-0 descriptors of the K / V tile (K-major for S / dP, MN-major for dQ)
            const uint64_t kK = desc_kmaj(aK, BN, 0), kV = desc_kmaj(aV, BN, 0), mK = desc_mn(aK, BN, 0);
            // dV, dK, dQ of query tile x (global index) whose P / dS are ready
            // x: global index of the query tile, xs: its ring stage
            // last: the key tile's last query tile; its dQ GEMM, the only one of the three that reads K,
            // goes first, so the K / V reload for the next key tile can start as early as possible
            auto grads = [&](uint32_t x, int xs, bool first, bool last) {
                const int st = xs;
                const uint32_t adS = smem_u32(sX + (x & 1) * Cfg::X_BYTES);
                const uint64_t mdO = desc_mn(smem_u32(smem + Cfg::OFF_DO + st * Cfg::Q_BYTES), BM, 0);
                const uint64_t mQ = desc_mn(smem_u32(smem + Cfg::OFF_Q + st * Cfg::Q_BYTES), BM, 0);
                const uint64_t kdS = desc_kmaj(adS, BN, 0), mdS = desc_mn(adS, BN, 0);
                auto dq_gemm = [&]() {
                    if (x > 0) wait(dq_free, (x - 1) & 1);
                    if (ok) {
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk) {
                            if (D == 64)
                                mma_f16_ss(tmem + Cfg::T_DQ, mn_step(mdS, kk), mn_step(mK, kk), idDQ, kk > 0);
                            else
                                mma_f16_ss(tmem + Cfg::T_DQ, mn_step(mK, kk), mn_step(mdS, kk), idDQ, kk > 0);
                        }
                        if (last) mma_commit(kv_empty);  // K / V are no longer read once these GEMMs finish
                    }
                };
                if (last) dq_gemm();
                // a new key tile overwrites dV / dK: the previous tile's epilogue has read them
                if (first && kt > 0) wait(acc_free, uint32_t(kt - 1) & 1);
                if (ok) {
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_f16_ts(tmem + Cfg::T_DV, tmem + Cfg::T_P + kk * 8, mn_step(mdO, kk), idDV, !first || kk > 0);
                    mma_commit(p_free);
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_f16_ss(tmem + Cfg::T_DK, kmaj_step(kdS, BN, kk), mn_step(mQ, kk), idDV, !first || kk > 0);
                    mma_commit(&q_empty[st]);  // the Q / dO stage may be refilled once dV / dK have read it
                }
                if (!last) dq_gemm();
                if (ok) {
                    mma_commit(mma_done);
                    mma_commit(&ds_free[x & 1]);
                }
            };
            ATTN_FOR_EACH_UNIT
            for (int64_t jt = first_tile; jt < ntiles; jt += tile_step) {
                const int64_t j0 = jt * BN;
                int qt0, nq;
                query_tiles<BM>(a.mask, j0, lq, lkv, &qt0, &nq);
                const int n_iter = G * nq;
                if (n_iter == 0) continue;
                wait(kv_full, uint32_t(kt) & 1);
                int prev_st = 0;
                for (int it = 0; it < n_iter; ++it, ++qi) {
                    const uint64_t kQ = desc_kmaj(smem_u32(smem + Cfg::OFF_Q + st * Cfg::Q_BYTES), BM, 0);
                    const uint64_t kdO = desc_kmaj(smem_u32(smem + Cfg::OFF_DO + st * Cfg::Q_BYTES), BM, 0);
                    wait(&q_full[st], st_par);
#pragma unroll
                    for (int q = 0; q < NH; ++q) {
                        // this column group of the previous tile has been read out of TMEM
                        if (qi > 0) wait(&s_free[q], (qi - 1) & 1);
                        if (ok) {
                            const uint32_t qoff = uint32_t(q * (BM / NH) * 128 / 16);  // query rows, in 16 B
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_f16_ss(tmem + Cfg::T_S + q * (BM / NH), kmaj_step(kK, BN, kk),
                                           kmaj_step(kQ + qoff, BM, kk), idS, kk > 0);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_f16_ss(tmem + Cfg::T_DP + q * (BM / NH), kmaj_step(kV, BN, kk),
                                           kmaj_step(kdO + qoff, BM, kk), idS, kk > 0);
                            mma_commit(&s_full[q]);
                        }
                    }
                    if (it > 0) {
                        wait(p_ready, (qi - 1) & 1);
                        grads(qi - 1, prev_st, it == 1, false);
                    }
                    prev_st = st;
                    if (++st == NST) {
                        st = 0;
                        st_par ^= 1;
                    }
                }
                wait(p_ready, (qi - 1) & 1);
                grads(qi - 1, prev_st, n_iter == 1, true);
                ++kt;
            }
            ATTN_END_UNITS
            // wait for every MMA this thread issued before TMEM is freed
            volatile int never = 0;
            mma_commit(drain);
            mbar_wait(drain, 0, &never, 100000000ull);
        }
    } else if (warp < 2 + Cfg::NSW) {
        // ================================================= P^T / dS^T (warps 2 .. 1 + NSW)
        const int lg = warp & 3, half = (warp - 2) >> 2;  // lane quadrant, column slice
        const uint32_t lane_addr = uint32_t(lg * 32) << 16;
        const int r = lg * 32 + lane;  // TMEM lane of this thread = key row of the tile
        const float sc = a.scale * kLog2e;
        const uint32_t aX = smem_u32(sX);
        bool ok = true;
        uint32_t qi = 0;            // query tiles done by this CTA
        int st = 0;                 // their Q / dO ring stage ...
        uint32_t st_par = 0;        // ... and its phase parity
        // tc: the wait orders later TMEM accesses (else it only guards shared memory)
        auto wait = [&](uint64_t *bar, uint32_t parity, bool tc) {
            if (ok && !(ok = mbar_wait(bar, parity, abort))) flag_abort(abort, a.status);
            ok = __all_sync(0xffffffffu, ok);
            if (tc) tc_fence_after();
        };

        ATTN_FOR_EACH_UNIT
        const int64_t shift = a.mask == ATTN_CAUSAL_BOTTOM_RIGHT ? lkv - lq : 0;
        for (int64_t jt = first_tile; jt < ntiles; jt += tile_step) {
            const int64_t j0 = jt * BN, j = j0 + r;
            const bool row_ok = j < lkv;
            int qt0, nq;
            query_tiles<BM>(a.mask, j0, lq, lkv, &qt0, &nq);
            const int n_iter = G * nq;
            int iq = 0;  // query tile within the head
            for (int it = 0; it < n_iter; ++it, ++qi) {
                const int64_t i0 = int64_t(qt0 + iq) * BM;
                // Usually LSE / D of this tile have landed (q_full), the GEMMs of tile qi - 2 that read
                // dS buffer qi & 1 have completed (ds_free) and the first S^T / dP^T group is written
                // (s_full): test all three at once and wait one by one only if one is not.
                const uint32_t t_q = mbar_test_wait(&q_full[st], st_par);
                const uint32_t t_d = qi >= 2 ? mbar_test_wait(&ds_free[qi & 1], ((qi >> 1) - 1) & 1) : 1u;
                const uint32_t t_s = mbar_test_wait(&s_full[0], qi & 1);
                const bool ready0 = __all_sync(0xffffffffu, t_q && t_d && t_s);
                if (!ready0) {
                    wait(&q_full[st], st_par, false);
                    if (qi >= 2) wait(&ds_free[qi & 1], ((qi >> 1) - 1) & 1, false);
                }
                bool ready1 = false;  // the previous tile's dV has read P^T and the second group is written
                const uint32_t adS = aX + uint32_t(qi & 1) * Cfg::X_BYTES;
                const uint32_t a_lse = smem_u32(smem + Cfg::OFF_LSE + st * BM * 4);
                const uint32_t a_dv = smem_u32(smem + Cfg::OFF_DVEC + st * BM * 4);
                // first visible query column of this key row; everything is masked past the sequence
                const int64_t cmin64 = !row_ok ? INT64_MAX : (a.mask ? j - shift - i0 : INT64_MIN);
                const int cmin = int(cmin64 < -1 ? -1 : (cmin64 > BM ? BM : cmin64));
#pragma unroll
                for (int q = 0; q < NG; ++q) {
                    const int rel = NH == NG ? q : 0;  // release group of these columns
                    if (q == 0 ? !ready0 : (NH == NG && !ready1)) wait(&s_full[rel], qi & 1, true);
                    else if (q == 0) tc_fence_after();
                    const int c0 = q * (BM / NG) + half * GW;
                    uint32_t pk[GW / 2];  // P^T of this column group, packed
                    // S^T / dP^T of the group in chunks of 16 columns.  With one group a thread (d = 128)
                    // the whole group is loaded at once and its TMEM columns released before P / dS are
                    // computed, so the next tile's S^T / dP^T GEMMs overlap this tile's element-wise work;
                    // with two (d = 64) chunk cc + 1 is loaded while chunk cc is computed and the columns
                    // are released after the group (the early release measured slower there)
                    constexpr int NCH = GW / 16;
                    constexpr bool kEarlyFree = NG == 1 && NCH == 2;
                    uint32_t sbuf[2][16], dbuf[2][16];
                    auto release = [&]() {
                        if (NH == NG || q == NG - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&s_free[rel]);  // these columns may be overwritten
                        }
                    };
                    if (kEarlyFree) {
                        if (ok) {
#pragma unroll
                            for (int cc = 0; cc < NCH; ++cc) {
                                tmem_ld16(tmem + lane_addr + Cfg::T_S + c0 + 16 * cc, sbuf[cc & 1]);
                                tmem_ld16(tmem + lane_addr + Cfg::T_DP + c0 + 16 * cc, dbuf[cc & 1]);
                            }
                            tmem_ld_wait_regs(sbuf[0], dbuf[0]);
                            tmem_ld_wait_regs(sbuf[1], dbuf[1]);
                        }
                        release();
                    } else if (ok) {
                        tmem_ld16(tmem + lane_addr + Cfg::T_S + c0, sbuf[0]);
                        tmem_ld16(tmem + lane_addr + Cfg::T_DP + c0, dbuf[0]);
                    }
                    if (ok) {
                        const bool any_mask = __any_sync(0xffffffffu, cmin > c0);
#pragma unroll
                        for (int cc = 0; cc < NCH; ++cc) {
                            const int col0 = c0 + cc * 16, cur = cc & 1;
                            if (!kEarlyFree) {
                                tmem_ld_wait_regs(sbuf[cur], dbuf[cur]);
                                if (cc + 1 < NCH) {
                                    tmem_ld16(tmem + lane_addr + Cfg::T_S + col0 + 16, sbuf[cur ^ 1]);
                                    tmem_ld16(tmem + lane_addr + Cfg::T_DP + col0 + 16, dbuf[cur ^ 1]);
                                }
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
                            for (int q2 = 0; q2 < 2; ++q2) {
                                const uint32_t off = sw128_offset(uint32_t(r), uint32_t(col0 + 8 * q2), BN);
                                st_shared_v4(adS + off, dk[4 * q2], dk[4 * q2 + 1], dk[4 * q2 + 2], dk[4 * q2 + 3]);
                            }
                        }
                    }
                    if (!kEarlyFree) release();
                    // P^T into TMEM once the previous tile's dV GEMM has read it
                    if (q == 0) {
                        const uint32_t t_p = qi > 0 ? mbar_test_wait(p_free, (qi - 1) & 1) : 1u;
                        const uint32_t t_s1 = NH == NG && NG > 1 ? mbar_test_wait(&s_full[NG > 1 ? 1 : 0], qi & 1) : 1u;
                        ready1 = __all_sync(0xffffffffu, t_p && t_s1);
                        if (!ready1 && qi > 0) wait(p_free, (qi - 1) & 1, true);
                        else tc_fence_after();
                    }
                    if (ok) {
#pragma unroll
                        for (int cc = 0; cc < GW / 16; ++cc) {
                            uint32_t w[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) w[e] = pk[cc * 8 + e];
                            tmem_st8(tmem + lane_addr + Cfg::T_P + c0 / 2 + cc * 8, w);
                        }
                    }
                }
                if (ok) tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_ready);
                if (++st == NST) {
                    st = 0;
                    st_par ^= 1;
                }
                if (++iq == nq) iq = 0;
            }
        }
        ATTN_END_UNITS
        pdl_trigger();
    } else if (kOrdered && warp == 2 + Cfg::NSW + 4) {
        // ================================================= ordered dQ mode: add counts (warp 14)
        // A GPU-scope release stalls the warp that issues it for about a microsecond; the dQ leader
        // hands each counter over (after its adds have landed and a proxy fence) and goes on, and
        // this warp publishes it.  A null counter ends the list.
        if (lane == 0) {
            for (uint32_t n = 0;; ++n) {
                const int k = int(n % kMailbox);
                if (!mbar_wait(&mb_full[k], (n / kMailbox) & 1, abort)) {
                    if (!*abort) flag_abort(abort, a.status);
                    break;
                }
                uint32_t *const ctr = mailbox[k];
                mbar_arrive(&mb_empty[k]);
                if (!ctr) break;
                red_release_gpu_add(ctr, 1u);
            }
        }
    } else {
        // ================================================= dQ reduce, dK / dV epilogue (warps 10..13)
        const int lg = warp & 3;
        const uint32_t lane_addr = uint32_t(lg * 32) << 16;
        const int r = lg * 32 + lane;  // TMEM lane of this thread
        const bool leader = warp == 2 + Cfg::NSW && lane == 0;
        uint8_t *sDQS = smem + Cfg::OFF_DQS;
        const uint32_t aDQS = smem_u32(sDQS);
        T *dK = static_cast<T *>(a.dK.ptr), *dV = static_cast<T *>(a.dV.ptr);
        bool ok = true;
        uint32_t qi = 0;
        uint32_t *pend = nullptr;  // ordered dQ mode: counter of the tile whose adds are still to be counted
        uint32_t n_post = 0;       // ... and the counters handed to the publishing warp so far
        auto post = [&](uint32_t *ctr) {
            const int k = int(n_post % kMailbox);
            if (n_post >= kMailbox && ok && !(ok = mbar_wait(&mb_empty[k], ((n_post / kMailbox) - 1) & 1, abort)))
                flag_abort(abort, a.status);
            if (ok) {
                mailbox[k] = ctr;
                mbar_arrive(&mb_full[k]);
            }
            ++n_post;
        };
        pdl_wait();  // the dQ accumulator (and the ordered mode's counters) have been zeroed

        ATTN_FOR_EACH_UNIT
        for (int64_t jt = first_tile; jt < ntiles; jt += tile_step) {
            const int64_t j0 = jt * BN, j = j0 + r;
            const bool row_ok = j < lkv;
            // element offsets of this thread's dK / dV row (recomputed where used: fewer live registers)
            auto offk = [&]() { return kv_b * a.dK.sb + g * a.dK.sh + (kv_row0 + j) * a.dK.ss; };
            auto offv = [&]() { return kv_b * a.dV.sb + g * a.dV.sh + (kv_row0 + j) * a.dV.ss; };
            int qt0, nq;
            query_tiles<BM>(a.mask, j0, lq, lkv, &qt0, &nq);
            const int n_iter = G * nq;
            if (n_iter == 0) {  // no query sees these keys: dK = dV = 0
                if (row_ok)
                    for (int x = 0; x < D; x += 8) {
                        *reinterpret_cast<uint4 *>(dK + offk() + x) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(dV + offv() + x) = make_uint4(0, 0, 0, 0);
                    }
                continue;
            }
            // dK (scaled) and dV of this key tile, once its last GEMMs have completed.  When TMA may
            // store the tile whole (fixed-length layout, whose extent clips the last tile; or a packed
            // tile inside its sequence), dV, then dK, is staged as 16-bit rows in the dQ staging buffer
            // and written by a TMA store
            // (d = 64 only: at d = 128 the 64 KB of dK / dV would pass through the 16 KB buffer in four
            // serial rounds, slower than the row stores)
            const bool tma_epi = D == 64 && (!kPacked || j0 + BN <= lkv);
            auto epilogue_tma = [&]() {
                constexpr int NBOX = D / 64;
#pragma unroll 1
                for (int t = 0; t < 2 * NBOX; ++t) {
                    const bool isk = t >= NBOX;
                    const int cb = t % NBOX;
                    const uint32_t tcol = (isk ? Cfg::T_DK : Cfg::T_DV) + cb * 64;
                    const float mul = isk ? a.scale : 1.f;
                    if (leader) bulk_wait_read0();  // the buffer's previous reader (reduce or store) is done
                    named_bar_sync(2, 128);
                    if (ok) {
#pragma unroll
                        for (int c16 = 0; c16 < 4; ++c16) {  // 16 columns at a time, two 16-byte chunks
                            uint32_t w[16];
                            tmem_ld16(tmem + lane_addr + tcol + c16 * 16, w);
                            tmem_ld_wait_regs(w);
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const uint32_t off = sw128_offset(uint32_t(r), uint32_t(c16 * 16 + h2 * 8), BN);
                                st_shared_v4(aDQS + off,
                                             pack2<T>(__uint_as_float(w[8 * h2 + 0]) * mul, __uint_as_float(w[8 * h2 + 1]) * mul),
                                             pack2<T>(__uint_as_float(w[8 * h2 + 2]) * mul, __uint_as_float(w[8 * h2 + 3]) * mul),
                                             pack2<T>(__uint_as_float(w[8 * h2 + 4]) * mul, __uint_as_float(w[8 * h2 + 5]) * mul),
                                             pack2<T>(__uint_as_float(w[8 * h2 + 6]) * mul, __uint_as_float(w[8 * h2 + 7]) * mul));
                            }
                        }
                    }
                    if (t == 2 * NBOX - 1) {  // every accumulator column has been read
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(acc_free);
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(2, 128);
                    if (leader && ok) {
                        tma_store_4d(isk ? &p.tm_dk : &p.tm_dv, sDQS, cb * 64, int(kv_row0 + j0), int(g), kv_b);
                        bulk_commit();
                    }
                }
            };
            // otherwise: read out of TMEM first (the accumulators are released right after the last
            // read, so the next key tile's first GEMMs need not wait for the dQ reduce), then stored
            // row by row
            auto epilogue = [&]() {
#pragma unroll 1
                for (int cc = 0; cc < D / 8; ++cc) {
                    uint32_t w[8], u[8];
                    if (ok) {
                        tmem_ld8(tmem + lane_addr + Cfg::T_DV + cc * 8, w);
                        tmem_ld8(tmem + lane_addr + Cfg::T_DK + cc * 8, u);
                        tmem_ld_wait_regs(w, u);
                    }
                    if (cc == D / 8 - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(acc_free);
                    }
                    if (ok && row_ok) {
                        uint4 ov, ok4;
                        ov.x = pack2<T>(__uint_as_float(w[0]), __uint_as_float(w[1]));
                        ov.y = pack2<T>(__uint_as_float(w[2]), __uint_as_float(w[3]));
                        ov.z = pack2<T>(__uint_as_float(w[4]), __uint_as_float(w[5]));
                        ov.w = pack2<T>(__uint_as_float(w[6]), __uint_as_float(w[7]));
                        ok4.x = pack2<T>(__uint_as_float(u[0]) * a.scale, __uint_as_float(u[1]) * a.scale);
                        ok4.y = pack2<T>(__uint_as_float(u[2]) * a.scale, __uint_as_float(u[3]) * a.scale);
                        ok4.z = pack2<T>(__uint_as_float(u[4]) * a.scale, __uint_as_float(u[5]) * a.scale);
                        ok4.w = pack2<T>(__uint_as_float(u[6]) * a.scale, __uint_as_float(u[7]) * a.scale);
                        *reinterpret_cast<uint4 *>(dV + offv() + cc * 8) = ov;
                        *reinterpret_cast<uint4 *>(dK + offk() + cc * 8) = ok4;
                    }
                }
            };
            int iq = 0, hg = 0;  // query tile within the head, head within the group
            for (int it = 0; it < n_iter; ++it, ++qi) {
                const int64_t hq = g * G + hg, i0 = int64_t(qt0 + iq) * BM;
                if (++iq == nq) {
                    iq = 0;
                    ++hg;
                }
                if (ok && !(ok = mbar_wait(mma_done, qi & 1, abort))) flag_abort(abort, a.status);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                if (it == n_iter - 1) {
                    if (tma_epi) epilogue_tma();
                    else epilogue();
                }
                // dQ of tile qi, half of its columns at a time, through the staging buffer
                const int64_t row0 = part * a.h * a.t_pad + geo.ws_start(b) + hq * a.t_pad + i0;
                // ordered dQ mode: this query tile's add counter
                auto sem_of = [&]() { return a.sem + hq * a.sem_stride + (geo.ws_start(b) + i0) / 64; };
                // read the whole accumulator first, so the next tile's dQ GEMM is not held up by the
                // reduce (whose rate the L2 sets)
                uint32_t v[2][32];
                if (ok) {
                    tmem_ld32(tmem + lane_addr + Cfg::T_DQ, v[0]);
                    tmem_ld32(tmem + lane_addr + Cfg::T_DQ + 32, v[1]);
                    tmem_ld_wait_regs(v[0]);
                    tmem_ld_wait_regs(v[1]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dq_free);
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {  // half of the columns at a time through the staging buffer
                    if (leader) bulk_wait_read0();  // the previous reduce has read the staging buffer
                    named_bar_sync(2, 128);
                    if (ok) {
                        if (D == 64) {  // lane = query row r, columns = head dims 32 hb ..
                            const uint32_t base = aDQS + uint32_t(r * 128);
#pragma unroll
                            for (int ch = 0; ch < 8; ++ch)
                                st_shared_v4(base + (uint32_t(ch ^ (r & 7)) << 4), v[hb][4 * ch], v[hb][4 * ch + 1],
                                             v[hb][4 * ch + 2], v[hb][4 * ch + 3]);
                        } else {  // lane = head dim r (box lg), columns = query rows 32 hb ..
                            const uint32_t base = aDQS + uint32_t(lg * 32 * 128) + uint32_t((lane & 3) << 2);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                st_shared_f32(base + uint32_t(e * 128) + (uint32_t((lane >> 2) ^ (e & 7)) << 4), v[hb][e]);
                        }
                    }
                    fence_proxy_async_smem();
                    ok = bar_and(2, 128, ok);
                    if (kOrdered && leader && ok && hb == 0) {
                        // the key tiles with work for this query tile are 0 .. J (whether a key tile has
                        // work for it does not increase with the key tile: J by bisection) and they add
                        // in the order J, J - 1, .., 0, so this add waits until J - jt adds have landed
                        const int qtile = int(i0 / BM);
                        int64_t lo = jt, hi = ntiles - 1;
                        while (lo < hi) {
                            const int64_t mid = (lo + hi + 1) / 2;
                            int q0, n;
                            query_tiles<BM>(a.mask, mid * BN, lq, lkv, &q0, &n);
                            if (n > 0 && q0 <= qtile) lo = mid;
                            else hi = mid - 1;
                        }
                        if (!(ok = wait_count(sem_of(), uint32_t(lo - jt), abort))) flag_abort(abort, a.status);
                        fence_proxy_async_global();
                    }
                    if (leader && ok) {
                        if (D == 64)
                            tma_reduce_add_2d(&p.tm_dq, sDQS, hb * 32, int(row0));
                        else
                            for (int box = 0; box < 4; ++box)
                                tma_reduce_add_2d(&p.tm_dq, sDQS + box * 32 * 128, box * 32, int(row0 + hb * 32));
                        bulk_commit();
                    }
                    if (kOrdered && leader && ok && hb == 1) {
                        // count the previous tile's adds once they have landed (this tile's two groups may
                        // still be in flight); the key tile's last tile is counted at once, so a unit
                        // leaves nothing pending behind it
                        if (pend) {
                            bulk_wait2();
                            fence_proxy_async_global();
                            post(pend);
                            pend = nullptr;
                        }
                        if (it == n_iter - 1) {
                            bulk_wait0();
                            fence_proxy_async_global();
                            post(sem_of());
                        } else {
                            pend = sem_of();
                        }
                    }
                }
            }
            // deterministic mode: this tile's dQ adds land before the next tile's (fixed order)
            if (leader && a.deterministic) bulk_wait0();
        }
        ATTN_END_UNITS
        if (kOrdered && leader) post(nullptr);  // the publishing warp may exit
        if (leader) bulk_wait0();  // the reduce-adds have read the staging buffer (and landed) before the exit
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

// Ordered dQ mode: the adds into each query tile's dQ go in decreasing key-tile order, each one
// waiting until the adds of all higher key tiles have landed.  Units are dealt in decreasing key-tile
// order (longest first among equal ones) to the least loaded CTA, and every CTA takes its units in
// the order dealt, so the key tiles a CTA works on never increase.  A wait then depends only on
// units of higher key tiles, which their CTAs take before any lower one; with every CTA resident
// (cooperative launch) no cycle of waits can form.  Leaves on = 0 when the units do not fit (the API
// refuses such problems).
template <int BM, int BN, class Geo>
void plan_ordered(TcSched &S, const DenseArgs &a, const Geo &g, int64_t units, int64_t ctas)
{
    S.on = 0;
    if (units > kSchedUnits || ctas > kSchedCtas || ctas < 1) return;
    const int64_t nheads = a.nseq * a.h_kv, G = a.h / a.h_kv;
    const int n = int(ctas), nu = int(units);
    static thread_local int32_t cost[kSchedUnits], order[kSchedUnits], cta_of[kSchedUnits];
    for (int u = 0; u < nu; ++u) {
        const int64_t jt = u / nheads, b = (u % nheads) / a.h_kv;
        const int64_t lq = g.q_len(b), lkv = g.kv_len(b);
        int64_t nq = 0;
        if (jt * BN < lkv) {
            const int64_t i_lo = first_query_seeing(a.mask, jt * BN, lq, lkv);
            nq = lq <= 0 || i_lo >= lq ? 0 : (lq + BM - 1) / BM - i_lo / BM;
        }
        cost[u] = jt * BN >= lkv ? 0 : nq > 0 ? int32_t(2 * G * nq + 2) : 1;
        order[u] = u;
    }
    std::stable_sort(order, order + nu, [&](int32_t x, int32_t y) {
        const int64_t jx = x / nheads, jy = y / nheads;
        return jx != jy ? jx > jy : cost[x] > cost[y];
    });
    // least loaded CTA first (lowest index among equals): a min-heap of (load, cta)
    std::priority_queue<std::pair<int64_t, int>, std::vector<std::pair<int64_t, int>>,
                        std::greater<std::pair<int64_t, int>>> heap;
    for (int c = 0; c < n; ++c) heap.push({0, c});
    int cnt[kSchedCtas];
    for (int c = 0; c < n; ++c) cnt[c] = 0;
    for (int k = 0; k < nu; ++k) {
        const int u = order[k];
        cta_of[u] = -1;
        if (cost[u] == 0) continue;  // past the sequence's keys: nothing to do
        const auto top = heap.top();
        heap.pop();
        cta_of[u] = top.second;
        ++cnt[top.second];
        heap.push({top.first + cost[u], top.second});
    }
    S.off[0] = 0;
    for (int c = 0; c < n; ++c) S.off[c + 1] = uint16_t(S.off[c] + cnt[c]);
    for (int c = 0; c < n; ++c) cnt[c] = S.off[c];
    for (int k = 0; k < nu; ++k) {
        const int u = order[k];
        if (cta_of[u] >= 0) S.unit[cnt[cta_of[u]]++] = uint16_t(u);
    }
    S.on = 1;
}

// Assigns the work units of a fixed-length batch to `ctas` CTAs.  A unit's cost is its query tiles
// plus one for its start (loading K / V, the pipeline refill, the dK / dV epilogue), in half tiles;
// units without work cost one (they write zero dK / dV rows).  Two plans: greedy (each unit,
// longest first, to the least loaded CTA) and bin packing, first fit decreasing (with a capacity
// starting at the mean load per CTA, at least the largest unit, units longest first go to the
// first CTA they fit in; the capacity grows until ctas CTAs suffice).  The packing finds the
// balanced groupings of the causal workloads' regular unit sizes that greedy misses by up to a
// tile; it is used when its makespan is at least 3 % shorter.  Each CTA takes its units longest
// first.  The plan of the last shape is kept
// (planning is host work on every call).  Varlen batches take only the head-local plan below, when
// its makespan is within 5 % of the snake order's; otherwise, in the split deterministic mode or
// when the plan does not fit, on = 0 (snake order).
template <int BM, int BN, class Geo>
void plan_units(TcSched &S, const DenseArgs &a, const Geo &g, int64_t units, int64_t ctas)
{
    S.on = 0;
    if (a.ordered) {
        plan_ordered<BM, BN>(S, a, g, units, ctas);
        return;
    }
    constexpr bool packed = IsPacked<Geo>::value;
    if (a.deterministic || units > kSchedUnits || ctas > kSchedCtas || ctas < 1) return;
    struct Key {
        int64_t nseq, h, h_kv, s_q, s_kv, units, ctas;
        int mask;
        uint64_t lens;  // packed batches: a hash of the sequence lengths
        bool operator==(const Key &o) const
        {
            return nseq == o.nseq && h == o.h && h_kv == o.h_kv && s_q == o.s_q && s_kv == o.s_kv && units == o.units &&
                   ctas == o.ctas && mask == o.mask && lens == o.lens;
        }
    };
    uint64_t lens = 1469598103934665603ull;  // FNV-1a over the (query, key) lengths
    if (packed)
        for (int64_t b = 0; b < a.nseq; ++b)
            for (const int64_t l : {g.q_len(b), g.kv_len(b)}) {
                lens ^= uint64_t(l);
                lens *= 1099511628211ull;
            }
    static thread_local Key last_key = {-1, 0, 0, 0, 0, 0, 0, 0, 0};
    static thread_local TcSched last_plan;
    const Key key = {a.nseq, a.h, a.h_kv, g.q_len(0), g.kv_len(0), units, ctas, a.mask, lens};
    if (key == last_key) {
        S = last_plan;
        return;
    }
    const int64_t nheads = a.nseq * a.h_kv, G = a.h / a.h_kv;
    const int n = int(ctas), nu = int(units);
    static thread_local int32_t cost[kSchedUnits], order[kSchedUnits], cta_of[kSchedUnits];
    int64_t load[kSchedCtas];
    int64_t total = 0, biggest = 0;
    for (int u = 0; u < nu; ++u) {
        const int64_t jt = u / nheads, b = (u % nheads) / a.h_kv;
        const int64_t lq = g.q_len(b), lkv = g.kv_len(b);
        int64_t nq = 0;
        if (jt * BN < lkv) {
            const int64_t i_lo = first_query_seeing(a.mask, jt * BN, lq, lkv);
            nq = lq <= 0 || i_lo >= lq ? 0 : (lq + BM - 1) / BM - i_lo / BM;
        }
        cost[u] = jt * BN >= lkv ? 0 : nq > 0 ? int32_t(2 * G * nq + 2) : 1;
        order[u] = u;
        total += cost[u];
        biggest = cost[u] > biggest ? cost[u] : biggest;
    }
    std::stable_sort(order, order + nu, [&](int32_t x, int32_t y) { return cost[x] > cost[y]; });
    // greedy: each unit, longest first, to the least loaded CTA
    static thread_local int32_t greedy_of[kSchedUnits];
    int64_t greedy_max = 0;
    {
        for (int c = 0; c < n; ++c) load[c] = 0;
        for (int k = 0; k < nu; ++k) {
            const int u = order[k];
            greedy_of[u] = -1;
            if (cost[u] == 0) continue;
            int c = 0;
            for (int d = 1; d < n; ++d)
                if (load[d] < load[c]) c = d;
            greedy_of[u] = c;
            load[c] += cost[u];
            greedy_max = load[c] > greedy_max ? load[c] : greedy_max;
        }
    }
    int64_t cap = (total + n - 1) / n;
    cap = cap > biggest ? cap : biggest;
    for (;; ++cap) {
        int used = 0;
        bool fits = true;
        for (int k = 0; k < nu && fits; ++k) {
            const int u = order[k];
            cta_of[u] = -1;
            if (cost[u] == 0) continue;  // past the keys: nothing to do
            int c = 0;
            while (c < used && load[c] + cost[u] > cap) ++c;
            if (c == used) {
                if (used == n) {
                    fits = false;
                    break;
                }
                load[used++] = 0;
            }
            cta_of[u] = c;
            load[c] += cost[u];
        }
        if (fits) break;
    }
    // the packing is kept only where it shortens the planned makespan clearly
    bool use_ffd = 100 * cap <= 97 * greedy_max;
    int64_t best = use_ffd ? cap : greedy_max;
    // head-local plan, for problems whose inputs and dQ accumulator do not fit in L2: the key tiles of
    // one (sequence, kv head) are paired (jt, n - 1 - jt), equal in cost under a causal mask; pairs
    // go out head by head in full rounds of `ctas` (all rounds but the last full one), so the CTAs
    // running together share a few heads' Q / dO rows and dQ accumulator rows; the remaining units
    // go greedily, longest first, to the least loaded CTA
    static thread_local int32_t local_of[kSchedUnits], local_rank[kSchedUnits], tail[kSchedUnits];
    bool use_local = false;
    const int64_t ws_bytes = (a.t_q * a.h * a.d * 2 + a.t_kv * a.h_kv * a.d) * 2 + a.h * a.t_pad * a.d * 4;
    if (ws_bytes > (int64_t(64) << 20)) {
        // the (sequence, kv head) heads, largest first (packed batches: their lengths differ), each with
        // its key tiles in pairs (jt, n_b - 1 - jt)
        static thread_local int32_t heads[kSchedUnits];
        static thread_local int64_t head_cost[kSchedUnits];
        for (int64_t hd = 0; hd < nheads; ++hd) {
            heads[hd] = int32_t(hd);
            head_cost[hd] = 0;
        }
        for (int u = 0; u < nu; ++u) head_cost[u % nheads] += cost[u];
        std::stable_sort(heads, heads + nheads, [&](int32_t x, int32_t y) { return head_cost[x] > head_cost[y]; });
        int64_t njobs = 0;
        for (int64_t hd = 0; hd < nheads; ++hd) {
            const int64_t nt = (g.kv_len(hd / a.h_kv) + BN - 1) / BN;
            njobs += (nt + 1) / 2;
        }
        const int64_t full = njobs / n > 1 ? njobs / n - 1 : 0;
        for (int c = 0; c < n; ++c) load[c] = 0;
        for (int u = 0; u < nu; ++u) local_of[u] = -1;
        int32_t rank = 0;
        int ntail = 0;
        int64_t job = 0;
        for (int64_t k = 0; k < nheads; ++k) {
            const int64_t head = heads[k];
            const int64_t nt = (g.kv_len(head / a.h_kv) + BN - 1) / BN;
            for (int64_t pj = 0; pj < (nt + 1) / 2; ++pj, ++job) {
                const int64_t ua = pj * nheads + head, ub = (nt - 1 - pj) * nheads + head;
                for (int kk = 0; kk < (ua == ub ? 1 : 2); ++kk) {
                    const int64_t u = kk == 0 ? ua : ub;
                    if (cost[u] == 0) continue;
                    if (job < full * n) {
                        const int c = int(job % n);
                        local_of[u] = c;
                        local_rank[u] = rank++;
                        load[c] += cost[u];
                    } else {
                        tail[ntail++] = int32_t(u);
                    }
                }
            }
        }
        std::stable_sort(tail, tail + ntail, [&](int32_t x, int32_t y) { return cost[x] > cost[y]; });
        for (int k = 0; k < ntail; ++k) {
            const int u = tail[k];
            int c = 0;
            for (int d = 1; d < n; ++d)
                if (load[d] < load[c]) c = d;
            local_of[u] = c;
            local_rank[u] = rank++;
            load[c] += cost[u];
        }
        int64_t local_max = 0;
        for (int c = 0; c < n; ++c) local_max = load[c] > local_max ? load[c] : local_max;
        use_local = 100 * local_max <= 105 * best;
        if (packed) {  // against the snake order packed batches take otherwise
            for (int c = 0; c < n; ++c) load[c] = 0;
            for (int u = 0; u < nu; ++u) {
                const int r = u / n, c = u % n;
                load[(r & 1) ? n - 1 - c : c] += cost[u];
            }
            int64_t snake_max = 0;
            for (int c = 0; c < n; ++c) snake_max = load[c] > snake_max ? load[c] : snake_max;
            use_local = 100 * local_max <= 105 * snake_max;
        }
    }
    if (packed && !use_local) {  // snake order (units running together would add into one long sequence's rows)
        last_plan = S;
        last_key = key;
        return;
    }
    if (use_local)
        for (int u = 0; u < nu; ++u) cta_of[u] = local_of[u];
    else if (!use_ffd)
        for (int u = 0; u < nu; ++u) cta_of[u] = greedy_of[u];
    int cnt[kSchedCtas];
    for (int c = 0; c < n; ++c) cnt[c] = 0;
    for (int u = 0; u < nu; ++u)
        if (cta_of[u] >= 0) ++cnt[cta_of[u]];
    S.off[0] = 0;
    for (int c = 0; c < n; ++c) S.off[c + 1] = uint16_t(S.off[c] + cnt[c]);
    for (int c = 0; c < n; ++c) cnt[c] = S.off[c];
    if (use_local) {  // each CTA's units in the order they were dealt
        std::stable_sort(order, order + nu, [&](int32_t x, int32_t y) {
            const int32_t rx = cta_of[x] >= 0 ? local_rank[x] : INT32_MAX, ry = cta_of[y] >= 0 ? local_rank[y] : INT32_MAX;
            return rx < ry;
        });
    }
    for (int k = 0; k < nu; ++k) {  // each CTA's units longest first (head-local plan: as dealt)
        const int u = order[k];
        if (cta_of[u] >= 0) S.unit[cnt[cta_of[u]]++] = uint16_t(u);
    }
    S.on = 1;
    last_plan = S;
    last_key = key;
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
    if (!map_dqacc(&prm.tm_dq, a.dqacc, D, int64_t(a.n_part) * a.h * a.t_pad, Cfg::DQ_BOX_ROWS))
        return cudaErrorInvalidValue;
    if (sq == 0) prm.tm_q = prm.tm_do = prm.tm_k;  // never read: no query tiles
    auto k = a.ordered ? dense_bwd_tc_kernel<T, D, Geo, true> : dense_bwd_tc_kernel<T, D, Geo, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    prm.a.tc_units = (a.deterministic ? a.n_part : ntiles) * a.nseq * a.h_kv;
    if (prm.a.tc_units > INT32_MAX) return cudaErrorInvalidValue;  // the kernel splits units in 32 bits
    const int64_t units = prm.a.tc_units < sm_count() ? prm.a.tc_units : sm_count();
    plan_units<Cfg::BM, Cfg::BN>(prm.sched, prm.a, g, prm.a.tc_units, units);
    if (a.ordered && !prm.sched.on) return cudaErrorNotSupported;  // the waits need the planned order
    // ordered dQ mode waits across CTAs: a cooperative launch puts all of them on the GPU at once
    return launch_kernel_ex(k, dim3(unsigned(units)), dim3(Cfg::THREADS + (a.ordered ? 32 : 0)), Cfg::SMEM_ALLOC, s,
                            true, a.ordered != 0, prm, g);
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
