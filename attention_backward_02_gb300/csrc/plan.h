// plan.h -- host-side argument bundles handed from the C ABI (api.cu) to the
// kernel launchers.  Private to the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace attn {

// A 16-bit tensor: element offset of (b, h, token) is
//   b * sb + h * sh + (start_b + i) * ss
// with sb = 0 and start_b from the cumulative lengths in packed mode, and
// start_b = 0 in fixed-length mode.
struct View {
    void *ptr;
    int64_t sb, sh, ss;
};

// Workspace of sdpa_bwd (all offsets 256-byte aligned):
//   status   uint32[64]              [0] device flags
//   lse2     f32 [h][t_pad]          LSE * log2(e); +inf on padding rows
//   dvec     f32 [h][t_pad]          D = rowsum(dO * O); 0 on padding rows
//   dqacc    f32 [n_part][h][t_pad][d]
//   sem      u32 [h][t_pad / 64]     ordered dQ mode: adds done per query tile
// t_pad = sum over sequences of their query length rounded up to 128
// (Geo::ws_start / ws_rows); the row of (head hq, sequence b, position i) is
// hq * t_pad + ws_start(b) + i.
struct DenseArgs {
    int dtype;                  // ATTN_F16 / ATTN_BF16
    int64_t nseq, h, h_kv, d;
    int64_t t_q, t_kv, t_pad;   // total query / key tokens, padded row count
    float scale;
    int mask;
    int deterministic, n_part;  // n_part partial dQ buffers (1 unless deterministic)
    int ordered;                // one dQ buffer, each query tile's adds in a fixed order (sem)
    uint32_t *sem;              // ordered: adds done per (head, 64-row workspace tile)
    int64_t sem_stride;         // sem words per head (t_pad / 64)
    bool packed;
    View q, k, v, o, dO, dQ, dK, dV;
    const float *lse;           // caller's stats ([B][h][s_q] or [h][T_q])
    float *lse_out;             // forward: where the stats go
    uint32_t *status;
    float *lse2, *dvec, *dqacc;
    int64_t tc_units;           // main kernel: work units (set by its launcher)
};

// Ordered dQ mode: the host plans every work unit (key tile of a sequence and kv head) up front.
constexpr int64_t kOrderedMaxUnits = 4096;

struct Workspace {
    static constexpr size_t kAlign = 256;
    static size_t align(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
};

// NSA workspace (all offsets 256-byte aligned):
//   status   uint32[64]
//   lse2     f32 [t1_pad][n1]       (max + ln sum) * log2(e), token-major
//   dvec     f32 [t1_pad][n1]
//   bitmap   uint32 [nseq][n2][nblk_max][words_max]   token bits per block
//   counts   int32 [nrows + 1]      then offsets (exclusive scan), in place
//   pieces   int32 [nrows + 1]      tensor-core work units per row (exclusive scan)
//   tokens   int32 [t1 * n2 * cnt]  block lists, ascending token ids
//   dqacc    f32 [t1_pad][n1][d]
//   dkacc    f32 [t2][n2][d], dvacc f32 [t2][n2][dv]
//   dqpart   f32 [t1][n2][cnt][G][d]   deterministic mode 1: dQ per (token, selected slot)
//   sem      uint32 [t1][n2]           deterministic mode 2: dQ adds landed per (token, kv head)
//   rank     int32 [t1][n2][cnt]       deterministic mode 2: per kept (token, slot), the token's kept
//                                      blocks above the slot's block (the adds that go before its own)
//   kvpart   f32 [pieces][bs][dK d | dV dv]   deterministic mode 1: each piece's dK / dV rows, summed
//                                      per block in piece order
// Chunks of 128 rows per work unit ("piece") of the tensor-core NSA kernel, and the most units a call
// can have: every block-list row's tokens in pieces of kNsaPieceChunks chunks of 128 / R tokens
// (R = 8 ceil(G / 8) rows per token).
constexpr int kNsaPieceChunks = 32;
inline int64_t nsa_piece_tokens(int64_t G) { return int64_t(kNsaPieceChunks) * (128 / ((G + 7) / 8 * 8)); }
inline int64_t nsa_max_pieces(int64_t nrows, int64_t t1, int64_t n2, int64_t cnt, int64_t G)
{
    const int64_t pt = nsa_piece_tokens(G);
    return nrows + (t1 * n2 * cnt + pt - 1) / pt;
}

struct NsaArgs {
    int dtype;
    int grad_fp32;              // dq, dk, dv are fp32 (else the input dtype)
    int64_t nseq, n1, n2, d, dv, bs, cnt;   // d: query / key head dim, dv: value head dim
    int64_t t1, t2, t1_pad;
    int64_t nblk_max, words_max, nrows;   // nrows = nseq * n2 * nblk_max
    float scale;
    int sparse_mode, n_part;
    int deterministic;          // 0: atomic adds; 1: per-slot dQ partials; 2: ordered adds behind counters
    const void *q, *k, *v, *o, *dO;
    const uint8_t *mask;        // attenMaskOptional [..][mask_cols], nonzero = removed (NULL: none)
    int64_t mask_cols;
    void *o_out;                // forward: O
    float *smax_out, *ssum_out; // forward: softmaxMax / softmaxSum [T1][n1][8]
    const float *smax, *ssum;
    const int32_t *topk;
    void *dq, *dk, *dvp;         // gradients (dvp: dV)
    __host__ __device__ void *dv_out() const { return dvp; }
    uint32_t *status;
    float *lse2, *dvec;
    uint32_t *bitmap;
    int32_t *offsets, *tokens, *pieces;
    float *dqacc, *dkacc, *dvacc, *dqpart;
    uint32_t *sem;
    int32_t *rank;
    float *kvpart;
    int64_t piece_tokens;       // tokens per work unit of the tensor-core kernel (whole lists when deterministic)
    int zero_dq;                // the preprocess also zeroes dqacc (tensor-core path, one dQ accumulator)
};

// Ordered deterministic NSA mode: the block-list rows in decreasing block order (then sequence and kv
// head); the row at position q.
__host__ __device__ inline int64_t nsa_ord_row(const NsaArgs &a, int64_t q)
{
    const int64_t nbg = a.nseq * a.n2;
    return (q % nbg) * a.nblk_max + (a.nblk_max - 1 - q / nbg);
}

// Maps a CUDA error to ATTN_ERR_CUDA and keeps its text for attn_last_error
// (this host thread); cudaSuccess maps to ATTN_OK.
attn_status_t record_cuda_error(cudaError_t e);

// ------------------------------------------------------------ launchers
// Each returns cudaGetLastError() of its launches.
cudaError_t launch_dense_preprocess(const DenseArgs &a, const FixedGeo &g, cudaStream_t s);
cudaError_t launch_dense_preprocess(const DenseArgs &a, const PackedGeo &g, cudaStream_t s);
cudaError_t launch_dense_bwd_main(const DenseArgs &a, const FixedGeo &g, cudaStream_t s);
cudaError_t launch_dense_bwd_main(const DenseArgs &a, const PackedGeo &g, cudaStream_t s);
cudaError_t launch_dq_finalize(const DenseArgs &a, const FixedGeo &g, cudaStream_t s);
cudaError_t launch_dq_finalize(const DenseArgs &a, const PackedGeo &g, cudaStream_t s);
cudaError_t launch_dense_fwd(const DenseArgs &a, const FixedGeo &g, cudaStream_t s);
cudaError_t launch_dense_fwd(const DenseArgs &a, const PackedGeo &g, cudaStream_t s);

cudaError_t launch_nsa_bwd(const NsaArgs &a, const PackedGeo &g, cudaStream_t s, cudaEvent_t before,
                           cudaEvent_t after);
cudaError_t launch_nsa_block_lists(const NsaArgs &a, const PackedGeo &g, cudaStream_t s);
bool nsa_tc_supported(const NsaArgs &a);
// forward: the two forward passes (row maxima; sums and O into a.lse2 / a.dvec / a.dqacc)
cudaError_t launch_nsa_tc(const NsaArgs &a, const PackedGeo &g, cudaStream_t s, bool forward = false);
// NSA forward: a.o, a.smax, a.ssum are written (o is the output here).
cudaError_t launch_nsa_fwd(const NsaArgs &a, const PackedGeo &g, cudaStream_t s);

}  // namespace attn
