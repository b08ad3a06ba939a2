// nsa_tc.cu -- tensor-core NSA selected-attention backward for sm_103a.
//
// Ascend CANN page "aclnnNsaSelectedAttentionGrad", Function / Formula:
// every query token gathers selectedBlockCount blocks of selectedBlockSize
// keys / values through topkIndices, runs the attention backward on them
// (dV = P^T dY, dQ = dS K scale, dK = dS^T Q scale) and the gathered dK / dV
// rows go back to the key / value rows they came from.
//
// Block-centric: a work unit ("piece") is one (sequence, kv head, key block)
// and up to kPieceChunks chunks of the ascending list of tokens that selected
// the block (built by the block-list kernels).  A chunk is 128 rows: 128 / R
// tokens x R rows, where a token's G query heads of the kv head (contiguous
// in TND) fill the first G of its R = 8 ceil(G / 8) rows, so one TMA box per
// token brings its G rows to a 1024-byte aligned start (empty slots load out
// of bounds and arrive as zeros; the R - G padding rows, and the rows past
// 128 / R tokens, are zeroed once and masked).  Any G from 1 to 32 runs here;
// G = 8, 16, 32 fill every row.  Per chunk:
//   S   = Q K_blk^T        M=128 rows  N=64 keys K=128  A=Q (K-major)   B=K (K-major)
//   dP  = dO V_blk^T       M=128       N=64      K=128  A=dO (K-major)  B=V (K-major)
//   P   = exp2(S scale log2 e - LSE log2 e), dS = P (dP - D)     (LSE from max/sum)
//   dV^T += dO^T P         M=128 (d)   N=64      K=128  A=dO (MN-major) B=P (MN-major)
//   dK^T += Q^T dS         M=128 (d)   N=64      K=128  A=Q (MN-major)  B=dS (MN-major)
//   dQ   = dS K_blk        M=128 rows  N=128 (d) K=64   A=dS (K-major)  B=K (MN-major)
// dQ of each token is added into an fp32 accumulator with TMA reduce-adds
// (one box of G rows per token), staged 64 head dims at a time in a buffer of
// its own, so a Q / dO stage is free as soon as the chunk's GEMMs are done;
// dK^T / dV^T stay in TMEM for the piece and are added into fp32
// accumulators at its end.  The chunk's token list travels through a 4-deep
// ring in shared memory with its own barriers.
// TMEM: S 64 + dP 64 + dV^T 64 + dK^T 64 + dQ 128 = 384 columns.
//
// The same kernel runs the NSA forward (the Function / Formula's attention over
// the gathered blocks) in two passes over the same work units, since a
// token's softmax spans blocks that different CTAs hold: kFwdMax computes S
// and each row's maximum over the block (atomicMax into the workspace);
// kFwdSum computes P = exp2(S scale log2 e - max), adds each row's sum of P
// into the workspace (atomicAdd) and O += P V_blk (M=128 rows, N=128, K=64,
// A=P K-major, B=V MN-major) through the dQ path's TMA reduce-adds; a finalize
// divides O by the sum.
//
// Roles (448 threads): warp 0 TMA producer, warp 1 MMA issuer, warps 2..9
// element-wise work (warp w reads TMEM lanes 32 (w % 4) .. + 31; two warps
// per lane group split the columns) and the piece's dK / dV, warps 10..13 the
// dQ of each chunk (TMEM -> its stage -> reduce), so the element-wise warps go
// straight on to the next chunk.  Bounded waits as in the dense kernel.
// Deterministic mode 1 stores each piece's dK / dV rows for a kernel that sums
// them per block in piece order (in place of the fp32 atomics), and each
// (token, slot)'s dQ rows for a finalize to sum in slot order.  Mode 2 (kOrd)
// takes whole block lists as work units (one writer per dK / dV row) and adds
// dQ into the one accumulator in decreasing block order per token:
// before its first add for a token the issuer lane waits until the token's
// counter equals the number of its kept blocks above this one (worked out with
// the block lists), and once the adds have landed (one chunk later, at once
// for a piece's last chunk) a 15th warp increments the counters with
// GPU-scope releases.  Pieces go to the CTAs in decreasing block order, so
// every wait is for a higher block and none can close a cycle; the launch is
// cooperative, so every CTA is resident.
#include <cudaTypedefs.h>

#include <climits>
#include <type_traits>

#include "plan.h"
#include "sm103.cuh"
#include "tc_util.cuh"

namespace attn {
using namespace sm103;
using namespace tc;

namespace {

constexpr int kD = 128, kBS = 64, kRows = 128, kNst = 2, kMaxSlots = 16, kSlotInts = 4, kSlotRing = 4;
constexpr int kMailbox = 2;  // ordered mode: chunks of add counters in flight to the publishing warp
enum : int { kBwd = 0, kFwdMax = 1, kFwdSum = 2 };  // what a launch of the kernel computes

// Order-preserving map of a float onto int32 (an involution), for atomicMax on floats.
__device__ __forceinline__ int32_t ord_f32(float x)
{
    const int32_t b = __float_as_int(x);
    return b >= 0 ? b : b ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float unord_f32(int32_t v) { return __int_as_float(v >= 0 ? v : v ^ 0x7FFFFFFF); }
constexpr int kPieceChunks = kNsaPieceChunks;  // chunks per work unit at most

struct NsaCfg {
    static constexpr int KV_BYTES = kBS * kD * 2;       // 16 KB
    static constexpr int Q_BYTES = kRows * kD * 2;      // 32 KB
    static constexpr int PS_BYTES = kRows * kBS * 2;    // 16 KB
    static constexpr int DQS_BYTES = kRows * 64 * 4;    // fp32 dQ: two buffers of one 32-wide box each
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KV_BYTES;
    static constexpr int OFF_Q = OFF_V + KV_BYTES;          // kNst stages
    static constexpr int OFF_DO = OFF_Q + kNst * Q_BYTES;   // kNst stages
    static constexpr int OFF_P = OFF_DO + kNst * Q_BYTES;
    static constexpr int OFF_DS = OFF_P + PS_BYTES;
    static constexpr int OFF_DQS = OFF_DS + PS_BYTES;
    static constexpr int OFF_SLOT = OFF_DQS + DQS_BYTES;    // kSlotRing x kMaxSlots x {local index, token, topk slot, -}
    static constexpr int OFF_MBOX = OFF_SLOT + kSlotRing * kMaxSlots * kSlotInts * 4;  // ordered mode: counters
    static constexpr int OFF_BAR = OFF_MBOX + kMailbox * kMaxSlots * 8;
    static constexpr int OFF_MISC = OFF_BAR + 24 * 8;
    static constexpr int THREADS = 448;
    static constexpr int SMEM = OFF_MISC + 64;
    static constexpr int SMEM_ALLOC = SMEM + 1024;
    static constexpr int T_S = 0, T_DP = 64, T_DV = 128, T_DK = 192, T_DQ = 256;
    static constexpr int T_COLS = 512;
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

}  // namespace

struct NsaTcParams {
    CUtensorMap tm_q, tm_do, tm_k, tm_v, tm_dq, tm_dqpart;
    NsaArgs a;
};

// piece index -> row of the block lists (binary search over the piece offsets)
__device__ __forceinline__ int64_t piece_row(const int32_t *piece_off, int64_t nrows, int64_t p)
{
    int64_t lo = 0, hi = nrows - 1;  // last row with piece_off[row] <= p
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) / 2;
        if (piece_off[mid] <= p) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// kOrd: backward in the ordered deterministic mode (a publishing warp, pieces in decreasing order)
template <class T, int kMode, bool kOrd>
__global__ void __launch_bounds__(kOrd ? 480 : 448, 1)
    nsa_tc_kernel(const __grid_constant__ NsaTcParams p, const PackedGeo geo)
{
    using Cfg = NsaCfg;
    constexpr int kType = std::is_same<T, __half>::value ? 0 : 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *kv_full = bars + 0, *kv_empty = bars + 1, *q_full = bars + 2, *q_empty = bars + 2 + kNst;
    uint64_t *s_full = bars + 2 + 2 * kNst, *p_ready = s_full + 1, *mma_done = s_full + 2, *drain = s_full + 3;
    uint64_t *dq_free = s_full + 4;  // the dQ warps have read the dQ accumulator
    uint64_t *slot_full = s_full + 5, *slot_empty = s_full + 5 + kSlotRing;  // [kSlotRing] token lists
    // ordered mode: chunks of add counters from the dQ issuer to the publishing warp
    uint64_t *mb_full = s_full + 5 + 2 * kSlotRing, *mb_empty = mb_full + kMailbox;  // [kMailbox]
    uint32_t **mbox = reinterpret_cast<uint32_t **>(smem + Cfg::OFF_MBOX);           // [kMailbox][kMaxSlots]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + Cfg::OFF_MISC + 8);
    int32_t *slots = reinterpret_cast<int32_t *>(smem + Cfg::OFF_SLOT);  // [ring][slot][kSlotInts]
    const NsaArgs &a = p.a;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // query heads per kv head, rows per token (a multiple of 8), tokens per chunk
    const int G = int(a.n1 / a.n2), R = (G + 7) / 8 * 8, tpc = kRows / R;
    // rows of the Q / dO stages no box writes (padding of each token, and past tpc tokens): zero
    // once, so the MMAs read finite values there (their P and dS are zero)
    if (R != G || tpc * R != kRows) {
        for (int x = threadIdx.x; x < 2 * kNst * 2 * kRows * 8; x += blockDim.x) {
            const int chunk16 = x % 8, row = (x / 8) % kRows, cb = (x / (8 * kRows)) % 2, buf = x / (16 * kRows);
            if (row / R < tpc && row % R < G) continue;
            const int off = (buf < kNst ? Cfg::OFF_Q + buf * Cfg::Q_BYTES : Cfg::OFF_DO + (buf - kNst) * Cfg::Q_BYTES) +
                            cb * kRows * 128 + row * 128 + chunk16 * 16;
            *reinterpret_cast<uint4 *>(smem + off) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // the tensor cores (async proxy) read these rows
    }
    pdl_wait();     // statistics, block lists, pieces and the zeroed accumulators are ready
    pdl_trigger();  // the finalize kernels may start launching; they wait for this grid
    // Work units: the pieces, in block-list row order; in the ordered mode the rows go in decreasing block
    // order (then sequence and kv head; a.pieces is scanned in that order), so each CTA's units have
    // non-increasing blocks, every wait is for a higher block, and no cycle of waits can form.
    const int64_t n_pieces = a.pieces[a.nrows];

    if (threadIdx.x == 0) {
        *abort = 0;
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s = 0; s < kNst; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_ready, 8);
        mbar_init(mma_done, 1);
        mbar_init(drain, 1);
        mbar_init(dq_free, 4);
        for (int k = 0; k < kSlotRing; ++k) {
            mbar_init(&slot_full[k], 1);
            mbar_init(&slot_empty[k], 8 + 4);  // P / dS warps, dQ warps
        }
        if (kOrd)
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

    uint8_t *sK = smem + Cfg::OFF_K, *sV = smem + Cfg::OFF_V, *sP = smem + Cfg::OFF_P, *sdS = smem + Cfg::OFF_DS;

    // the work unit of piece pc: block-list row, token range, sequence / head / block
#define NSA_PIECE_DECODE                                                                         \
    const int64_t qrow_ = piece_row(a.pieces, a.nrows, pc);                                     \
    const int64_t row = kOrd ? nsa_ord_row(a, qrow_) : qrow_;                                       \
    const int64_t lp = pc - a.pieces[qrow_];                                                    \
    const int64_t tok_begin = a.offsets[row] + lp * a.piece_tokens;                            \
    const int64_t tok_end_full = a.offsets[row + 1];                                            \
    const int64_t tok_end = tok_begin + a.piece_tokens < tok_end_full ? tok_begin + a.piece_tokens : tok_end_full; \
    const int nchunks = int((tok_end - tok_begin + tpc - 1) / tpc);                            \
    const int64_t b = row / (a.n2 * a.nblk_max), g = (row / a.nblk_max) % a.n2, blk = row % a.nblk_max; \
    (void)b; (void)g; (void)blk; (void)nchunks;

    if (warp == 0) {
        // ================================================= TMA producer (the whole warp: lane u
        // takes token u of a chunk, so the chunk's many small copies are issued in parallel)
        {
            if (lane == 0) {
                prefetch_tmap(&p.tm_q); prefetch_tmap(&p.tm_do); prefetch_tmap(&p.tm_k); prefetch_tmap(&p.tm_v);
            }
            bool ok = true;
            int64_t kt = 0, ci = 0, q_armed = 0, kv_armed = 0;
            for (int64_t pc = blockIdx.x; pc < n_pieces; pc += gridDim.x) {
                NSA_PIECE_DECODE
                if (kt > 0 && ok && !(ok = mbar_wait(kv_empty, uint32_t(kt - 1) & 1, abort))) flag_abort(abort, a.status);
                ok = __all_sync(0xffffffffu, ok);
                if (ok && lane == 0) {
                    kv_armed = kt + 1;
                    const int krow = int(geo.cu_kv[b] + blk * kBS);
                    mbar_arrive_expect_tx(kv_full, (kMode == kFwdMax ? 1 : 2) * Cfg::KV_BYTES);
                    for (int c = 0; c < kD / 64; ++c) {
                        tma_load_3d(sK + c * kBS * 128, &p.tm_k, kv_full, c * 64, int(g), krow);
                        if (kMode != kFwdMax) tma_load_3d(sV + c * kBS * 128, &p.tm_v, kv_full, c * 64, int(g), krow);
                    }
                }
                // lane u's token of the next chunk, loaded one chunk ahead
                int32_t t_next = -1;
                if (lane < tpc) {
                    const int64_t idx = tok_begin + lane;
                    t_next = idx < tok_end ? a.tokens[idx] : -1;
                }
                for (int ch = 0; ch < nchunks; ++ch, ++ci) {
                    const int st = int(ci % kNst), rs = int(ci % kSlotRing);
                    const int64_t use = ci / kNst, ruse = ci / kSlotRing;
                    if (use > 0 && ok && !(ok = mbar_wait(&q_empty[st], uint32_t(use - 1) & 1, abort)))
                        flag_abort(abort, a.status);
                    if (ruse > 0 && ok && !(ok = mbar_wait(&slot_empty[rs], uint32_t(ruse - 1) & 1, abort)))
                        flag_abort(abort, a.status);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) continue;
                    const int u = lane;  // this lane's token slot
                    const int32_t t = t_next;
                    if (u < tpc) {
                        // deterministic mode 1: position of this block in the token's topk (its first
                        // occurrence, the one the block lists keep); mode 2: how many of the token's kept
                        // blocks above this one add before it (worked out with the block lists)
                        int32_t slot = -1;
                        if (a.deterministic != 0 && t >= 0) {
                            const int32_t *ids = a.topk + (int64_t(t) * a.n2 + g) * a.cnt;
                            for (int64_t c = a.cnt - 1; c >= 0; --c)
                                if (ids[c] == blk) slot = int32_t(c);
                            if (kOrd && slot >= 0) slot = a.rank[(int64_t(t) * a.n2 + g) * a.cnt + slot];
                        }
                        int32_t *sl = slots + (rs * kMaxSlots + u) * kSlotInts;
                        sl[0] = t >= 0 ? int32_t(t - geo.cu_q[b]) : -1;
                        sl[1] = t;
                        sl[2] = slot;
                        const int64_t idx = tok_begin + int64_t(ch + 1) * tpc + u;
                        t_next = idx < tok_end ? a.tokens[idx] : -1;
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&slot_full[rs]);  // the token list is written
                        q_armed = ci + 1;
                        // Q (and dO in the backward): d = 128, 16-bit
                        mbar_arrive_expect_tx(&q_full[st], uint32_t(tpc * G * (kMode == kBwd ? 512 : 256)));
                    }
                    __syncwarp();  // the expected bytes are registered before any copy lands
                    uint8_t *sQ = smem + Cfg::OFF_Q + st * Cfg::Q_BYTES, *sdO = smem + Cfg::OFF_DO + st * Cfg::Q_BYTES;
                    if (u < tpc) {
                        const int qrow = t >= 0 ? int(int64_t(t) * a.n1 + g * G) : int(a.t1 * a.n1);  // past the end: zeros
                        for (int c = 0; c < kD / 64; ++c) {
                            tma_load_2d(sQ + c * kRows * 128 + u * R * 128, &p.tm_q, &q_full[st], c * 64, qrow);
                            if (kMode == kBwd)
                                tma_load_2d(sdO + c * kRows * 128 + u * R * 128, &p.tm_do, &q_full[st], c * 64, qrow);
                        }
                    }
                }
                ++kt;
            }
            if (!ok && lane == 0) {
                volatile int never = 0;
                for (int64_t x = q_armed - kNst; x < q_armed; ++x)
                    if (x >= 0) mbar_wait(&q_full[x % kNst], uint32_t(x / kNst) & 1, &never, 100000000ull);
                if (kv_armed > 0) mbar_wait(kv_full, uint32_t(kv_armed - 1) & 1, &never, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ================================================= MMA issuer
        if (elect_one()) {
            constexpr uint32_t idS = idesc_f16(128, kBS, kType, 0, 0);     // S, dP
            constexpr uint32_t idT = idesc_f16(128, kBS, kType, 1, 1);     // dV^T, dK^T
            constexpr uint32_t idQ = idesc_f16(128, kD, kType, 0, 1);      // dQ
            // step-0 descriptors (a K step adds a constant to the start address field)
            const uint64_t kK = desc_kmaj(smem_u32(sK), kBS, 0), kV = desc_kmaj(smem_u32(sV), kBS, 0);
            const uint64_t mK = desc_mn(smem_u32(sK), kBS, 0);
            const uint64_t mP = desc_mn(smem_u32(sP), kRows, 0), mdS = desc_mn(smem_u32(sdS), kRows, 0);
            const uint64_t kdS = desc_kmaj(smem_u32(sdS), kRows, 0);
            const uint64_t kP = desc_kmaj(smem_u32(sP), kRows, 0), mV = desc_mn(smem_u32(sV), kBS, 0);
            bool ok = true;
            int64_t kt = 0, ci = 0;
            for (int64_t pc = blockIdx.x; pc < n_pieces; pc += gridDim.x) {
                NSA_PIECE_DECODE
                if (ok && !(ok = mbar_wait(kv_full, uint32_t(kt) & 1, abort))) flag_abort(abort, a.status);
                tc_fence_after();
                for (int ch = 0; ch < nchunks; ++ch, ++ci) {
                    const int st = int(ci % kNst);
                    const uint32_t aQ = smem_u32(smem + Cfg::OFF_Q + st * Cfg::Q_BYTES);
                    const uint32_t adO = smem_u32(smem + Cfg::OFF_DO + st * Cfg::Q_BYTES);
                    const uint64_t kQ = desc_kmaj(aQ, kRows, 0), kdO = desc_kmaj(adO, kRows, 0);
                    const uint64_t mQ = desc_mn(aQ, kRows, 0), mdO = desc_mn(adO, kRows, 0);
                    if (ok && !(ok = mbar_wait(&q_full[st], uint32_t(ci / kNst) & 1, abort))) flag_abort(abort, a.status);
                    tc_fence_after();
                    if (ok) {
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk)
                            mma_f16_ss(tmem + Cfg::T_S, kmaj_step(kQ, kRows, kk), kmaj_step(kK, kBS, kk), idS, kk > 0);
                        if (kMode == kBwd)
#pragma unroll
                            for (int kk = 0; kk < kD / 16; ++kk)
                                mma_f16_ss(tmem + Cfg::T_DP, kmaj_step(kdO, kRows, kk), kmaj_step(kV, kBS, kk), idS,
                                           kk > 0);
                        mma_commit(s_full);
                    }
                    if (ok && !(ok = mbar_wait(p_ready, uint32_t(ci) & 1, abort))) flag_abort(abort, a.status);
                    tc_fence_after();
                    if (kMode == kFwdMax) {  // the row maxima are all this pass needs
                        if (ok) {
                            mma_commit(&q_empty[st]);
                            if (ch == nchunks - 1) mma_commit(kv_empty);
                        }
                        continue;
                    }
                    if (kMode == kBwd && ok) {
#pragma unroll
                        for (int kk = 0; kk < kRows / 16; ++kk)
                            mma_f16_ss(tmem + Cfg::T_DV, mn_step(mdO, kk), mn_step(mP, kk), idT, ch > 0 || kk > 0);
#pragma unroll
                        for (int kk = 0; kk < kRows / 16; ++kk)
                            mma_f16_ss(tmem + Cfg::T_DK, mn_step(mQ, kk), mn_step(mdS, kk), idT, ch > 0 || kk > 0);
                    }
                    // the dQ warps have read the previous chunk's dQ
                    if (ci > 0 && ok && !(ok = mbar_wait(dq_free, uint32_t(ci - 1) & 1, abort))) flag_abort(abort, a.status);
                    tc_fence_after();
                    if (ok) {  // backward: dQ = dS K; forward: O = P V
#pragma unroll
                        for (int kk = 0; kk < kBS / 16; ++kk) {
                            if (kMode == kBwd)
                                mma_f16_ss(tmem + Cfg::T_DQ, kmaj_step(kdS, kRows, kk), mn_step(mK, kk), idQ, kk > 0);
                            else
                                mma_f16_ss(tmem + Cfg::T_DQ, kmaj_step(kP, kRows, kk), mn_step(mV, kk), idQ, kk > 0);
                        }
                        mma_commit(mma_done);
                        mma_commit(&q_empty[st]);  // this Q / dO stage may be refilled
                        if (ch == nchunks - 1) mma_commit(kv_empty);
                    }
                }
                ++kt;
            }
            volatile int never = 0;
            mma_commit(drain);
            mbar_wait(drain, 0, &never, 100000000ull);
        }
    } else if (warp < 10) {
        // ================================================= P / dS, and dK / dV at the end of a piece
        const int lg = warp & 3, half = (warp - 2) >> 2;
        const uint32_t lane_addr = uint32_t(lg * 32) << 16;
        const int r = lg * 32 + lane;  // TMEM lane: chunk row (S, dP, dQ) or head dim (dV^T, dK^T)
        const float sc = a.scale * kLog2e;
        const uint32_t aP = smem_u32(sP), adS = smem_u32(sdS);
        bool ok = true;
        int64_t kt = 0, ci = 0;
        for (int64_t pc = blockIdx.x; pc < n_pieces; pc += gridDim.x) {
            NSA_PIECE_DECODE
            const int64_t shift = geo.kv_len(b) - geo.q_len(b);
            for (int ch = 0; ch < nchunks; ++ch, ++ci) {
                const int rs = int(ci % kSlotRing);
                // this row's token (empty slot: -1), then its LSE and D straight from the workspace
                if (ok && !(ok = mbar_wait(&slot_full[rs], uint32_t(ci / kSlotRing) & 1, abort)))
                    flag_abort(abort, a.status);
                const bool row_used = r / R < tpc && r % R < G;  // else a padding row
                const int32_t *sl = slots + (rs * kMaxSlots + (row_used ? r / R : 0)) * kSlotInts;
                const int32_t i_loc = ok && row_used ? sl[0] : -1, tok = ok && row_used ? sl[1] : -1;
                __syncwarp();
                if (lane == 0) mbar_arrive(&slot_empty[rs]);
                const int64_t qrow = int64_t(tok) * a.n1 + g * G + r % R;
                // backward: LSE (log2 units); forward sum pass: the row's maximum over all its blocks
                // (+inf where there is none, so every P is 0)
                float lse = INFINITY, dvv = 0.f;
                if (kMode == kBwd && i_loc >= 0) {
                    lse = a.lse2[qrow];
                    dvv = a.dvec[qrow];
                } else if (kMode == kFwdSum && i_loc >= 0) {
                    const float m = unord_f32(reinterpret_cast<const int32_t *>(a.lse2)[qrow]);
                    lse = m == -INFINITY ? INFINITY : m;
                }
                float rmax = -INFINITY, rsum = 0.f;  // forward: this thread's part of the row
                if (ok && !(ok = mbar_wait(s_full, uint32_t(ci) & 1, abort))) flag_abort(abort, a.status);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                if (ok) {
                    // empty slot -> everything masked; sparse mode 2 -> keys past (local index + S2 - S1) masked
                    const int64_t cmax64 =
                        i_loc < 0 ? -1 : (a.sparse_mode == 2 ? int64_t(i_loc) + shift - blk * kBS : int64_t(kBS));
                    const int cmax = int(cmax64 < -1 ? -1 : (cmax64 > kBS ? kBS : cmax64));
                    const bool any_mask = a.mask || __any_sync(0xffffffffu, cmax < (half + 1) * 32 - 1);
                    // attenMaskOptional: this query's row of the mask, from the block's first key
                    const uint8_t *mrow = a.mask && i_loc >= 0 ? a.mask + int64_t(i_loc) * a.mask_cols + blk * kBS : nullptr;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int col0 = half * 32 + cc * 16;
                        if (kMode != kBwd) {  // forward passes: S only
                            uint32_t s[16];
                            tmem_ld16(tmem + lane_addr + Cfg::T_S + col0, s);
                            tmem_ld_wait_regs(s);
                            uint32_t pk[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int c = col0 + 2 * e;
                                float x0 = __uint_as_float(s[2 * e]) * sc, x1 = __uint_as_float(s[2 * e + 1]) * sc;
                                if (any_mask) {
                                    x0 = c <= cmax && !(mrow && mrow[c]) ? x0 : -INFINITY;
                                    x1 = c + 1 <= cmax && !(mrow && mrow[c + 1]) ? x1 : -INFINITY;
                                }
                                if (kMode == kFwdMax) {
                                    rmax = fmaxf(rmax, fmaxf(x0, x1));
                                } else {
                                    const float p0 = ex2(x0 - lse), p1 = ex2(x1 - lse);
                                    rsum += p0 + p1;
                                    pk[e] = pack2<T>(p0, p1);
                                }
                            }
                            if (kMode == kFwdSum)
#pragma unroll
                                for (int q = 0; q < 2; ++q) {
                                    const uint32_t off = sw128_offset(uint32_t(r), uint32_t(col0 + 8 * q), kRows);
                                    st_shared_v4(aP + off, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                                }
                            continue;
                        }
                        uint32_t s[16], dp[16];
                        tmem_ld16(tmem + lane_addr + Cfg::T_S + col0, s);
                        tmem_ld16(tmem + lane_addr + Cfg::T_DP + col0, dp);
                        tmem_ld_wait_regs(s, dp);
                        uint32_t pk[8], dk[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int c = col0 + 2 * e;
                            float x0 = fmaf(__uint_as_float(s[2 * e]), sc, -lse);
                            float x1 = fmaf(__uint_as_float(s[2 * e + 1]), sc, -lse);
                            if (any_mask) {
                                x0 = c <= cmax && !(mrow && mrow[c]) ? x0 : -INFINITY;
                                x1 = c + 1 <= cmax && !(mrow && mrow[c + 1]) ? x1 : -INFINITY;
                            }
                            pk[e] = p_and_ds<T>(x0, x1, __uint_as_float(dp[2 * e]) - dvv,
                                                __uint_as_float(dp[2 * e + 1]) - dvv, &dk[e]);
                        }
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const uint32_t off = sw128_offset(uint32_t(r), uint32_t(col0 + 8 * q), kRows);
                            st_shared_v4(aP + off, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                            st_shared_v4(adS + off, dk[4 * q], dk[4 * q + 1], dk[4 * q + 2], dk[4 * q + 3]);
                        }
                    }
                }
                // forward: fold this half row into the row's maximum / sum over all blocks
                if (kMode == kFwdMax && i_loc >= 0 && rmax != -INFINITY)
                    atomicMax(reinterpret_cast<int32_t *>(a.lse2) + qrow, ord_f32(rmax));
                if (kMode == kFwdSum && i_loc >= 0 && rsum > 0.f) atomicAdd(a.dvec + qrow, rsum);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_ready);
            }
            // ---- dV^T, dK^T of this piece (this thread: head dim r, 32 of the 64 keys), once its
            // last chunk's GEMMs have completed (backward only)
            if (kMode != kBwd) {
                ++kt;
                continue;
            }
            if (ok && !(ok = mbar_wait(mma_done, uint32_t(ci - 1) & 1, abort))) flag_abort(abort, a.status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            if (ok) {
                uint32_t vv[32], kk[32];
                tmem_ld32(tmem + lane_addr + Cfg::T_DV + half * 32, vv);
                tmem_ld32(tmem + lane_addr + Cfg::T_DK + half * 32, kk);
                tmem_ld_wait();
                if (a.deterministic == 1) {  // this piece's rows, summed per block in piece order afterwards
                    float *dst = a.kvpart + (pc * kBS + half * 32) * (2 * kD) + r;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        dst[e * 2 * kD] = __uint_as_float(kk[e]) * a.scale;
                        dst[e * 2 * kD + kD] = __uint_as_float(vv[e]);
                    }
                } else {
                    const int64_t key0 = geo.cu_kv[b] + blk * kBS + half * 32;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int64_t off = ((key0 + e) * a.n2 + g) * kD + r;
                        atomicAdd(a.dvacc + off, __uint_as_float(vv[e]));
                        atomicAdd(a.dkacc + off, __uint_as_float(kk[e]) * a.scale);
                    }
                }
            }
            tc_fence_before();
            ++kt;
        }
    } else if (kOrd && warp == 14) {
        // ================================================= ordered mode: add counts (warp 14)
        // A GPU-scope release stalls the warp that issues it for about a microsecond; the dQ issuer
        // hands each chunk's counters over once their adds have landed, and this warp publishes them.
        uint32_t *const end_mark = reinterpret_cast<uint32_t *>(uintptr_t(1));
        for (uint32_t n = 0;; ++n) {
            const int k = int(n % kMailbox);
            const bool got = __all_sync(0xffffffffu, mbar_wait(&mb_full[k], (n / kMailbox) & 1, abort));
            if (!got) {
                if (lane == 0 && !*abort) flag_abort(abort, a.status);
                break;
            }
            uint32_t *const ctr = lane < kMaxSlots ? mbox[k * kMaxSlots + lane] : nullptr;
            const bool end = mbox[k * kMaxSlots] == end_mark;
            __syncwarp();
            if (lane == 0) mbar_arrive(&mb_empty[k]);
            if (end) break;
            if (ctr) red_release_gpu_add(ctr, 1u);
        }
    } else {
        // ================================================= dQ of each chunk (warps 10..13)
        const int lg = warp & 3;
        const uint32_t lane_addr = uint32_t(lg * 32) << 16;
        const int r = lg * 32 + lane;        // TMEM lane = chunk row
        const bool issuer = warp == 10;      // lane u of this warp adds token u's rows
        uint8_t *sDQS = smem + Cfg::OFF_DQS;
        const uint32_t aDQS = smem_u32(sDQS);
        bool ok = true;
        int64_t ci = 0;
        // ordered mode (issuer warp): the counter of this lane's token in the previous chunk, whose
        // adds are still to be counted, and the chunks handed to the publishing warp so far
        uint32_t *pend = nullptr;
        bool pend_set = false;
        uint32_t n_post = 0;
        auto post = [&](uint32_t *ctr) {  // the whole issuer warp; lanes past the chunk's tokens pass null
            const int k = int(n_post % kMailbox);
            bool free_ok = true;
            if (n_post >= kMailbox) free_ok = mbar_wait(&mb_empty[k], ((n_post / kMailbox) - 1) & 1, abort);
            if (!__all_sync(0xffffffffu, free_ok)) {
                if (lane == 0 && !*abort) flag_abort(abort, a.status);
                ok = false;
            } else {
                if (lane < kMaxSlots) mbox[k * kMaxSlots + lane] = ctr;
                __syncwarp();
                if (lane == 0) mbar_arrive(&mb_full[k]);
            }
            ++n_post;
        };
        for (int64_t pc = blockIdx.x; pc < n_pieces; pc += gridDim.x) {
            NSA_PIECE_DECODE
            for (int ch = 0; ch < nchunks; ++ch, ++ci) {
                const int rs = int(ci % kSlotRing);
                if (ok && !(ok = mbar_wait(&slot_full[rs], uint32_t(ci / kSlotRing) & 1, abort)))
                    flag_abort(abort, a.status);
                int32_t t = -1, slot = -1;  // this lane's token and its topk position (ordered: blocks above)
                if (ok && issuer && lane < tpc) {
                    const int32_t *sl = slots + (rs * kMaxSlots + lane) * kSlotInts;
                    t = sl[1];
                    slot = sl[2];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&slot_empty[rs]);
                if (kMode == kFwdMax) continue;  // no GEMM output to add in this pass
                if (ok && !(ok = mbar_wait(mma_done, uint32_t(ci) & 1, abort))) flag_abort(abort, a.status);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {  // head dims 64 hr .. + 63
                    uint32_t v[2][32];
                    if (ok) {
                        tmem_ld32(tmem + lane_addr + Cfg::T_DQ + hr * 64, v[0]);
                        tmem_ld32(tmem + lane_addr + Cfg::T_DQ + hr * 64 + 32, v[1]);
                        tmem_ld_wait_regs(v[0]);
                        tmem_ld_wait_regs(v[1]);
                    }
                    if (hr == 1) {  // the accumulator has been read out
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(dq_free);
                    }
#pragma unroll
                    for (int bx = 0; bx < 2; ++bx) {  // one 32-wide box per round, alternating buffers
                        // the adds issued two rounds ago (same buffer) have read it
                        if (issuer) bulk_wait_read1();
                        named_bar_sync(2, 128);
                        if (ok) {
                            const uint32_t base = aDQS + uint32_t(bx * kRows * 128 + r * 128);
#pragma unroll
                            for (int c4 = 0; c4 < 8; ++c4)
                                st_shared_v4(base + (uint32_t(c4 ^ (r & 7)) << 4), v[bx][4 * c4], v[bx][4 * c4 + 1],
                                             v[bx][4 * c4 + 2], v[bx][4 * c4 + 3]);
                        }
                        fence_proxy_async_smem();
                        ok = bar_and(2, 128, ok);
                        if (issuer) {
                            bool add = ok && t >= 0;
                            if (kOrd && add && hr == 0 && bx == 0) {
                                // this token's adds from its selected blocks above this one have landed
                                if (wait_count(a.sem + int64_t(t) * a.n2 + g, uint32_t(slot), abort)) {
                                    fence_proxy_async_global();
                                } else {
                                    flag_abort(abort, a.status);
                                    ok = add = false;
                                }
                            }
                            if (add) {
                                const int box = hr * 2 + bx;
                                const uint8_t *src = sDQS + bx * (kRows * 128) + lane * R * 128;
                                if (kMode == kBwd && a.deterministic == 1) {  // own partial rows (summed in slot order later)
                                    const int prow = int(((int64_t(t) * a.n2 + g) * a.cnt + slot) * G);
                                    tma_store_2d(&p.tm_dqpart, src, box * 32, prow);
                                } else {
                                    tma_reduce_add_2d(&p.tm_dq, src, box * 32, int(int64_t(t) * a.n1 + g * G));
                                }
                            }
                            bulk_commit();  // one group per round and lane, possibly empty
                            if (kOrd && hr == 1 && bx == 1) {
                                // count the previous chunk's adds once they have landed (all but this
                                // chunk's four groups complete); a piece's last chunk is counted at once,
                                // so the next piece (a lower block) never waits on an uncounted add here
                                uint32_t *const cur = ok && t >= 0 ? a.sem + int64_t(t) * a.n2 + g : nullptr;
                                if (pend_set) {
                                    bulk_wait4();
                                    fence_proxy_async_global();
                                    post(pend);
                                }
                                if (ch == nchunks - 1) {
                                    bulk_wait0();
                                    fence_proxy_async_global();
                                    post(cur);
                                    pend_set = false;
                                } else {
                                    pend = cur;
                                    pend_set = true;
                                }
                            }
                        }
                    }
                }
            }
        }
        if (kOrd && issuer) post(reinterpret_cast<uint32_t *>(uintptr_t(lane == 0)));  // the publisher may exit
        if (issuer) bulk_wait0();
    }
#undef NSA_PIECE_DECODE

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::T_COLS);
    }
}

// ===================================================================== host

namespace {

PFN_cuTensorMapEncodeTiled_v12000 nsa_encode_fn()
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

bool encode(CUtensorMap *m, CUtensorMapDataType type, int rank, const void *base, const cuuint64_t *dims,
            const cuuint64_t *strides, const cuuint32_t *box)
{
    auto enc = nsa_encode_fn();
    if (!enc) return false;
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, type, rank, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int nsa_sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

// Pieces per block-list row and their exclusive scan (one CTA).
__global__ void __launch_bounds__(1024) nsa_piece_scan_kernel(NsaArgs a)
{
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    pdl_wait();  // the block lists are complete
    pdl_trigger();
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int per_piece = int(a.piece_tokens);
    const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
    if (threadIdx.x == 0) a.pieces[0] = 0;
    for (int64_t base = 0; base < a.nrows; base += 1024) {
        const int64_t r = base + threadIdx.x;  // position; the ordered mode takes the rows in its own order
        const int64_t rr = r < a.nrows && a.deterministic == 2 ? nsa_ord_row(a, r) : r;
        const int32_t len = r < a.nrows ? a.offsets[rr + 1] - a.offsets[rr] : 0;
        int32_t v = (len + per_piece - 1) / per_piece;
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
        if (r < a.nrows) a.pieces[r + 1] = prefix + v;
        __syncthreads();
        if (threadIdx.x == 1023) carry = prefix + v;
        __syncthreads();
    }
}

}  // namespace

bool nsa_tc_supported(const NsaArgs &a)
{
    const int64_t G = a.n1 / a.n2;
    return a.d == kD && a.dv == kD && a.bs == kBS && G >= 1 && G <= 32;
}

cudaError_t launch_nsa_tc(const NsaArgs &a, const PackedGeo &g, cudaStream_t s, bool forward)
{
    NsaTcParams prm;
    prm.a = a;
    const int G = int(a.n1 / a.n2);
    // The block lists are split into pieces, except in the ordered mode, which takes each whole (one
    // writer per dK / dV row; split, the pieces of a block run beside those of the blocks above it and
    // wait on them: 1.86 against 1.30 ms at 4 x 4096 tokens).  Mode 1 stores each piece's dK / dV rows
    // for a sum in piece order.
    prm.a.piece_tokens = a.deterministic == 2 && !forward ? (int64_t(1) << 30) : nsa_piece_tokens(G);
    cudaError_t e = launch_kernel(nsa_piece_scan_kernel, dim3(1), dim3(1024), 0, s, true, prm.a);
    if (e != cudaSuccess) return e;
    if (a.t1 == 0) return cudaSuccess;
    const CUtensorMapDataType dt = a.dtype == ATTN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    {   // Q, dO: rows (token, head) x d; box 64 x G (one token's heads of a kv head)
        cuuint64_t dims[2] = {cuuint64_t(kD), cuuint64_t(a.t1 * a.n1)};
        cuuint64_t strides[1] = {cuuint64_t(kD * 2)};
        cuuint32_t box[2] = {64, cuuint32_t(G)};
        if (!encode(&prm.tm_q, dt, 2, a.q, dims, strides, box) ||
            !encode(&prm.tm_do, dt, 2, forward ? a.q : a.dO, dims, strides, box))  // the forward reads no dO
            return cudaErrorInvalidValue;
    }
    {   // K, V: (d, kv head, token); box 64 x 1 x block
        cuuint64_t dims[3] = {cuuint64_t(kD), cuuint64_t(a.n2), cuuint64_t(a.t2)};
        cuuint64_t strides[2] = {cuuint64_t(kD * 2), cuuint64_t(a.n2 * kD * 2)};
        cuuint32_t box[3] = {64, 1, cuuint32_t(kBS)};
        if (!encode(&prm.tm_k, dt, 3, a.k, dims, strides, box) || !encode(&prm.tm_v, dt, 3, a.v, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    {   // fp32 dQ accumulator: rows (token, head) x d; box 32 x G
        cuuint64_t dims[2] = {cuuint64_t(kD), cuuint64_t(a.t1 * a.n1)};
        cuuint64_t strides[1] = {cuuint64_t(kD * 4)};
        cuuint32_t box[2] = {32, cuuint32_t(G)};
        if (!encode(&prm.tm_dq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.dqacc, dims, strides, box))
            return cudaErrorInvalidValue;
        prm.tm_dqpart = prm.tm_dq;
        if (!forward && a.deterministic == 1) {  // fp32 partials: rows (token, kv head, slot, head of group) x d
            cuuint64_t pdims[2] = {cuuint64_t(kD), cuuint64_t(a.t1 * a.n1 * a.cnt)};
            if (!encode(&prm.tm_dqpart, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.dqpart, pdims, strides, box))
                return cudaErrorInvalidValue;
        }
    }
    const dim3 grid = dim3(unsigned(nsa_sm_count()));
    if (!forward) {
        // ordered deterministic mode: a CTA waits for adds other CTAs make, so all of them must be resident
        // (a cooperative launch), and a 15th warp publishes the counts
        const bool ord = a.deterministic == 2;
        auto k = ord ? (a.dtype == ATTN_F16 ? nsa_tc_kernel<__half, kBwd, true> : nsa_tc_kernel<__nv_bfloat16, kBwd, true>)
                     : (a.dtype == ATTN_F16 ? nsa_tc_kernel<__half, kBwd, false> : nsa_tc_kernel<__nv_bfloat16, kBwd, false>);
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, NsaCfg::SMEM_ALLOC)) != cudaSuccess)
            return e;
        return launch_kernel_ex(k, grid, dim3(NsaCfg::THREADS + (ord ? 32 : 0)), NsaCfg::SMEM_ALLOC, s, true, ord, prm, g);
    }
    // forward: the row maxima, then the sums and O, over the same work units
    auto k1 = a.dtype == ATTN_F16 ? nsa_tc_kernel<__half, kFwdMax, false> : nsa_tc_kernel<__nv_bfloat16, kFwdMax, false>;
    auto k2 = a.dtype == ATTN_F16 ? nsa_tc_kernel<__half, kFwdSum, false> : nsa_tc_kernel<__nv_bfloat16, kFwdSum, false>;
    if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, NsaCfg::SMEM_ALLOC)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, NsaCfg::SMEM_ALLOC)) != cudaSuccess)
        return e;
    if ((e = launch_kernel(k1, grid, dim3(NsaCfg::THREADS), NsaCfg::SMEM_ALLOC, s, true, prm, g)) != cudaSuccess) return e;
    return launch_kernel(k2, grid, dim3(NsaCfg::THREADS), NsaCfg::SMEM_ALLOC, s, true, prm, g);
}

}  // namespace attn
