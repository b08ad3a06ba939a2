// api.cu -- the C ABI: argument checks, workspace layout, launch order.
//
// Every check runs on the host before the first launch, so a call that
// returns an error has launched nothing.  Launch order on the caller's
// stream: preprocess -> main backward -> dQ finalize (dense), and
// preprocess -> block lists -> main -> finalizes (NSA); each kernel is
// chained to its predecessor with programmatic dependent launch.
#include <cmath>
#include <cstring>

#include "attnbwd.h"
#include "plan.h"

using namespace attn;

namespace {

constexpr int64_t kTilePad = 128;       // NSA: rows a tile may run past the last token
constexpr int kDefaultDqSplits = 8;     // deterministic dense dQ partial buffers

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Element strides of a 16-bit tensor must be multiples of 8 (16 bytes).
bool strides_ok(const attn_view_t &v) { return v.sb % 8 == 0 && v.sh % 8 == 0 && v.ss % 8 == 0; }

struct DenseShape {
    bool packed;
    int64_t nseq, t_q, t_kv;
};

attn_status_t check_cu(const int64_t *cu, int64_t n, int64_t *total)
{
    int64_t prev = 0;
    for (int64_t b = 0; b < n; ++b) {
        if (cu[b] < prev) return ATTN_ERR_INVALID;
        prev = cu[b];
    }
    *total = prev;
    return ATTN_OK;
}

attn_status_t check_dense_desc(const attn_sdpa_desc_t *d, DenseShape *sh)
{
    if (!d) return ATTN_ERR_NULLPTR;
    if (d->dtype != ATTN_F16 && d->dtype != ATTN_BF16) return ATTN_ERR_INVALID;
    if (d->b < 1 || d->h < 1 || d->h_kv < 1 || d->h % d->h_kv != 0 || d->d < 1) return ATTN_ERR_INVALID;
    if (!std::isfinite(d->scale)) return ATTN_ERR_INVALID;
    if (d->mask != ATTN_MASK_NONE && d->mask != ATTN_CAUSAL_TOP_LEFT && d->mask != ATTN_CAUSAL_BOTTOM_RIGHT)
        return ATTN_ERR_INVALID;
    if ((d->cu_seqlens_q == nullptr) != (d->cu_seqlens_kv == nullptr)) return ATTN_ERR_NULLPTR;
    if (d->deterministic < 0 || d->deterministic > 2) return ATTN_ERR_INVALID;
    if (d->dq_splits < 0) return ATTN_ERR_INVALID;
    sh->packed = d->cu_seqlens_q != nullptr;
    sh->nseq = d->b;
    if (sh->packed) {
        if (d->b > kMaxSeq) return ATTN_ERR_UNSUPPORTED;
        attn_status_t st = check_cu(d->cu_seqlens_q, d->b, &sh->t_q);
        if (st) return st;
        st = check_cu(d->cu_seqlens_kv, d->b, &sh->t_kv);
        if (st) return st;
    } else {
        if (d->s_q < 0 || d->s_kv < 0) return ATTN_ERR_INVALID;
        if (d->b > 65535) return ATTN_ERR_UNSUPPORTED;  // grid z
        sh->t_q = d->b * d->s_q;
        sh->t_kv = d->b * d->s_kv;
    }
    if (d->d != 64 && d->d != 128) return ATTN_ERR_UNSUPPORTED;
    // 32-bit row indices inside the kernels
    if (sh->t_q * d->h >= (int64_t(1) << 31) || sh->t_kv * d->h_kv >= (int64_t(1) << 31))
        return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

int dense_parts(const attn_sdpa_desc_t *d)
{
    if (d->deterministic != 1) return 1;
    return d->dq_splits > 0 ? d->dq_splits : kDefaultDqSplits;
}

struct DenseLayout {
    size_t status, lse2, dvec, dqacc, sem, total;
    int64_t t_pad;
};

// Workspace rows: every sequence's query rows rounded up to kWsRowAlign.
int64_t ws_rows(const attn_sdpa_desc_t *d, const DenseShape &sh)
{
    if (!sh.packed) return d->b * ws_round(d->s_q);
    int64_t n = 0;
    for (int64_t b = 0; b < d->b; ++b) n += ws_round(d->cu_seqlens_q[b] - (b ? d->cu_seqlens_q[b - 1] : 0));
    return n;
}

DenseLayout dense_layout(const attn_sdpa_desc_t *d, const DenseShape &sh)
{
    DenseLayout L;
    L.t_pad = ws_rows(d, sh);
    size_t rows = size_t(d->h) * size_t(L.t_pad);
    L.status = 0;
    L.lse2 = Workspace::align(64 * sizeof(uint32_t));
    L.dvec = L.lse2 + Workspace::align(rows * sizeof(float));
    L.dqacc = L.dvec + Workspace::align(rows * sizeof(float));
    L.sem = L.dqacc + Workspace::align(size_t(dense_parts(d)) * rows * size_t(d->d) * sizeof(float));
    // ordered dQ mode: one add counter per (head, 64 workspace rows)
    L.total = L.sem + (d->deterministic == 2 ? Workspace::align(rows / 64 * sizeof(uint32_t)) : 0);
    return L;
}

View to_view(const attn_view_t &v, bool packed)
{
    View w;
    w.ptr = v.ptr;
    w.sb = packed ? 0 : v.sb;
    w.sh = v.sh;
    w.ss = v.ss;
    return w;
}

attn_status_t check_view(const attn_view_t &v, int64_t rows)
{
    if (rows == 0) return ATTN_OK;
    if (!v.ptr) return ATTN_ERR_NULLPTR;
    if (!aligned16(v.ptr) || !strides_ok(v)) return ATTN_ERR_ALIGN;
    return ATTN_OK;
}

attn_status_t check_ws(const void *ws, size_t have, size_t need)
{
    if (need == 0) return ATTN_OK;
    if (!ws || have < need || (reinterpret_cast<uintptr_t>(ws) & (Workspace::kAlign - 1))) return ATTN_ERR_WORKSPACE;
    return ATTN_OK;
}

void fill_geo(const attn_sdpa_desc_t *d, const DenseShape &sh, FixedGeo *fg, PackedGeo *pg)
{
    fg->nseq = d->b;
    fg->s_q = d->s_q;
    fg->s_kv = d->s_kv;
    if (sh.packed) {
        pg->nseq = d->b;
        pg->cu_q[0] = pg->cu_kv[0] = pg->ws_q[0] = 0;
        for (int64_t b = 0; b < d->b; ++b) {
            pg->cu_q[b + 1] = d->cu_seqlens_q[b];
            pg->cu_kv[b + 1] = d->cu_seqlens_kv[b];
            pg->ws_q[b + 1] = pg->ws_q[b] + ws_round(pg->cu_q[b + 1] - pg->cu_q[b]);
        }
    }
}

// Text of the CUDA error behind the last ATTN_ERR_CUDA of this host thread.
thread_local const char *g_last_error = "";

attn_status_t cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return ATTN_OK;
    g_last_error = cudaGetErrorString(e);
    return ATTN_ERR_CUDA;
}

thread_local cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;

// Records a timing event; under stream capture as an external event node, so replays record it.
cudaError_t mark(cudaEvent_t ev, cudaStream_t s)
{
    if (!ev) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    return cudaEventRecordWithFlags(ev, s, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0);
}

}  // namespace

attn_status_t attn::record_cuda_error(cudaError_t e) { return cuda_status(e); }

extern "C" {

const char *attn_last_error(void) { return g_last_error; }

const char *attn_status_string(attn_status_t s)
{
    switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_NULLPTR: return "ATTN_ERR_NULLPTR";
    case ATTN_ERR_INVALID: return "ATTN_ERR_INVALID";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_ALIGN: return "ATTN_ERR_ALIGN";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE: return "ATTN_ERR_DEVICE";
    }
    return "ATTN_ERR_UNKNOWN";
}

attn_status_t sdpa_workspace_size(const attn_sdpa_desc_t *desc, size_t *fwd_bytes, size_t *bwd_bytes)
{
    DenseShape sh;
    attn_status_t st = check_dense_desc(desc, &sh);
    if (st) return st;
    if (fwd_bytes) *fwd_bytes = Workspace::align(64 * sizeof(uint32_t));
    if (bwd_bytes) *bwd_bytes = dense_layout(desc, sh).total;
    return ATTN_OK;
}

attn_status_t sdpa_fwd_stats(const attn_sdpa_desc_t *desc, attn_view_t q, attn_view_t k, attn_view_t v,
                             attn_view_t o, float *lse, void *workspace, size_t workspace_bytes, void *stream)
{
    DenseShape sh;
    attn_status_t st = check_dense_desc(desc, &sh);
    if (st) return st;
    if ((st = check_view(q, sh.t_q)) || (st = check_view(o, sh.t_q)) || (st = check_view(k, sh.t_kv)) ||
        (st = check_view(v, sh.t_kv)))
        return st;
    if (sh.t_q && !lse) return ATTN_ERR_NULLPTR;
    if ((st = check_ws(workspace, workspace_bytes, Workspace::align(64 * sizeof(uint32_t))))) return st;
    if (sh.t_q == 0) return ATTN_OK;

    DenseArgs a;
    std::memset(&a, 0, sizeof a);
    a.dtype = desc->dtype;
    a.nseq = desc->b; a.h = desc->h; a.h_kv = desc->h_kv; a.d = desc->d;
    a.t_q = sh.t_q; a.t_kv = sh.t_kv; a.t_pad = ws_rows(desc, sh);
    a.scale = float(desc->scale);
    a.mask = desc->mask;
    a.packed = sh.packed;
    a.q = to_view(q, sh.packed); a.k = to_view(k, sh.packed); a.v = to_view(v, sh.packed);
    a.o = to_view(o, sh.packed);
    a.lse_out = lse;
    a.status = static_cast<uint32_t *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FixedGeo fg;
    static thread_local PackedGeo pg;
    fill_geo(desc, sh, &fg, &pg);
    return cuda_status(sh.packed ? launch_dense_fwd(a, pg, s) : launch_dense_fwd(a, fg, s));
}

attn_status_t sdpa_bwd(const attn_sdpa_desc_t *desc, attn_view_t q, attn_view_t k, attn_view_t v, attn_view_t o,
                       attn_view_t dO, const float *lse, attn_view_t dQ, attn_view_t dK, attn_view_t dV,
                       void *workspace, size_t workspace_bytes, void *stream)
{
    DenseShape sh;
    attn_status_t st = check_dense_desc(desc, &sh);
    if (st) return st;
    if ((st = check_view(q, sh.t_q)) || (st = check_view(o, sh.t_q)) || (st = check_view(dO, sh.t_q)) ||
        (st = check_view(dQ, sh.t_q)) || (st = check_view(k, sh.t_kv)) || (st = check_view(v, sh.t_kv)) ||
        (st = check_view(dK, sh.t_kv)) || (st = check_view(dV, sh.t_kv)))
        return st;
    if (sh.t_q && !lse) return ATTN_ERR_NULLPTR;
    DenseLayout L = dense_layout(desc, sh);
    // 32-bit row coordinates of the fp32 dQ accumulator inside the kernels
    if (int64_t(dense_parts(desc)) * desc->h * L.t_pad >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
    if (desc->deterministic == 2) {  // ordered dQ: every work unit is planned on the host
        int64_t max_kv = desc->s_kv;
        if (sh.packed) {
            max_kv = 0;
            for (int64_t b = 0; b < desc->b; ++b) {
                const int64_t l = desc->cu_seqlens_kv[b] - (b ? desc->cu_seqlens_kv[b - 1] : 0);
                max_kv = l > max_kv ? l : max_kv;
            }
        }
        if ((max_kv + 127) / 128 * desc->b * desc->h_kv > kOrderedMaxUnits) return ATTN_ERR_UNSUPPORTED;
    }
    if ((st = check_ws(workspace, workspace_bytes, L.total))) return st;

    DenseArgs a;
    std::memset(&a, 0, sizeof a);
    a.dtype = desc->dtype;
    a.nseq = desc->b; a.h = desc->h; a.h_kv = desc->h_kv; a.d = desc->d;
    a.t_q = sh.t_q; a.t_kv = sh.t_kv; a.t_pad = L.t_pad;
    a.scale = float(desc->scale);
    a.mask = desc->mask;
    a.deterministic = desc->deterministic == 1;
    a.ordered = desc->deterministic == 2;
    a.n_part = dense_parts(desc);
    a.packed = sh.packed;
    a.q = to_view(q, sh.packed); a.k = to_view(k, sh.packed); a.v = to_view(v, sh.packed);
    a.o = to_view(o, sh.packed); a.dO = to_view(dO, sh.packed);
    a.dQ = to_view(dQ, sh.packed); a.dK = to_view(dK, sh.packed); a.dV = to_view(dV, sh.packed);
    a.lse = lse;
    char *ws = static_cast<char *>(workspace);
    a.status = reinterpret_cast<uint32_t *>(ws + L.status);
    a.lse2 = reinterpret_cast<float *>(ws + L.lse2);
    a.dvec = reinterpret_cast<float *>(ws + L.dvec);
    a.dqacc = reinterpret_cast<float *>(ws + L.dqacc);
    a.sem = reinterpret_cast<uint32_t *>(ws + L.sem);
    a.sem_stride = L.t_pad / 64;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (sh.t_q == 0 && sh.t_kv == 0) return ATTN_OK;

    FixedGeo fg;
    static thread_local PackedGeo pg;
    fill_geo(desc, sh, &fg, &pg);
    cudaError_t e;
    if (sh.packed) {
        if ((e = launch_dense_preprocess(a, pg, s)) != cudaSuccess) return cuda_status(e);
        if ((e = mark(g_ev_before, s)) != cudaSuccess) return cuda_status(e);
        if ((e = launch_dense_bwd_main(a, pg, s)) != cudaSuccess) return cuda_status(e);
        if ((e = mark(g_ev_after, s)) != cudaSuccess) return cuda_status(e);
        if ((e = launch_dq_finalize(a, pg, s)) != cudaSuccess) return cuda_status(e);
    } else {
        if ((e = launch_dense_preprocess(a, fg, s)) != cudaSuccess) return cuda_status(e);
        if ((e = mark(g_ev_before, s)) != cudaSuccess) return cuda_status(e);
        if ((e = launch_dense_bwd_main(a, fg, s)) != cudaSuccess) return cuda_status(e);
        if ((e = mark(g_ev_after, s)) != cudaSuccess) return cuda_status(e);
        if ((e = launch_dq_finalize(a, fg, s)) != cudaSuccess) return cuda_status(e);
    }
    return ATTN_OK;
}

// ------------------------------------------------------------------- NSA

namespace {

struct NsaShape {
    int64_t t1, t2, nblk_max, words_max, maxlen_q, dv;
};

attn_status_t check_nsa_desc(const attn_nsa_desc_t *d, NsaShape *sh)
{
    if (!d) return ATTN_ERR_NULLPTR;
    if (!d->cu_seqlens_q || !d->cu_seqlens_kv) return ATTN_ERR_NULLPTR;
    if (d->dtype != ATTN_F16 && d->dtype != ATTN_BF16) return ATTN_ERR_INVALID;
    if (d->b < 1) return ATTN_ERR_INVALID;
    if (d->b > kMaxSeq) return ATTN_ERR_UNSUPPORTED;
    if (d->n1 < 1 || d->n2 < 1 || d->n1 > 128 || d->n2 > 128 || d->n1 % d->n2 != 0 || d->n1 / d->n2 > 32)
        return ATTN_ERR_INVALID;
    if (!std::isfinite(d->scale)) return ATTN_ERR_INVALID;
    if (d->block_size < 16 || d->block_size > 128 || d->block_size % 16 != 0) return ATTN_ERR_INVALID;
    if (d->block_count < 1 || d->block_count > 128 || d->block_count * d->block_size >= 8192)
        return ATTN_ERR_INVALID;
    if (d->sparse_mode != 0 && d->sparse_mode != 2) return ATTN_ERR_INVALID;
    if (d->deterministic < 0 || d->deterministic > 2) return ATTN_ERR_INVALID;
    if (d->d != 128 && d->d != 192) return ATTN_ERR_INVALID;
    if (d->d_v != 0 && d->d_v != 128 && d->d_v != 192) return ATTN_ERR_INVALID;
    if (d->grad_fp32 != 0 && d->grad_fp32 != 1) return ATTN_ERR_INVALID;
    if (check_cu(d->cu_seqlens_q, d->b, &sh->t1) || check_cu(d->cu_seqlens_kv, d->b, &sh->t2))
        return ATTN_ERR_INVALID;
    sh->nblk_max = 0;
    sh->maxlen_q = 0;
    for (int64_t b = 0; b < d->b; ++b) {
        int64_t lkv = d->cu_seqlens_kv[b] - (b ? d->cu_seqlens_kv[b - 1] : 0);
        int64_t lq = d->cu_seqlens_q[b] - (b ? d->cu_seqlens_q[b - 1] : 0);
        if (lkv % d->block_size != 0 || lkv < d->block_count * d->block_size) return ATTN_ERR_INVALID;
        if (lkv / d->block_size > sh->nblk_max) sh->nblk_max = lkv / d->block_size;
        if (lq > sh->maxlen_q) sh->maxlen_q = lq;
    }
    sh->words_max = (sh->maxlen_q + 31) / 32;
    sh->dv = d->d_v ? d->d_v : d->d;
    if (d->atten_mask) {  // the mask covers every sequence's local positions
        if (d->mask_rows < sh->maxlen_q || d->mask_cols < 0) return ATTN_ERR_INVALID;
        for (int64_t b = 0; b < d->b; ++b)
            if (d->cu_seqlens_kv[b] - (b ? d->cu_seqlens_kv[b - 1] : 0) > d->mask_cols) return ATTN_ERR_INVALID;
    }
    if (sh->t1 * d->n1 >= (int64_t(1) << 31) || sh->t2 * d->n2 >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

struct NsaLayout {
    size_t status, lse2, dvec, bitmap, offsets, pieces, tokens, dqacc, dkacc, dvacc, dqpart, sem, rank, kvpart, total;
    int64_t t1_pad, nrows;
};

NsaLayout nsa_layout(const attn_nsa_desc_t *d, const NsaShape &sh)
{
    NsaLayout L;
    L.t1_pad = sh.t1 + kTilePad;
    L.nrows = d->b * d->n2 * sh.nblk_max;
    size_t rows = size_t(d->n1) * size_t(L.t1_pad);
    L.status = 0;
    L.lse2 = Workspace::align(64 * sizeof(uint32_t));
    L.dvec = L.lse2 + Workspace::align(rows * sizeof(float));
    L.bitmap = L.dvec + Workspace::align(rows * sizeof(float));
    L.offsets = L.bitmap + Workspace::align(size_t(L.nrows) * size_t(sh.words_max) * sizeof(uint32_t));
    L.pieces = L.offsets + Workspace::align(size_t(L.nrows + 1) * sizeof(int32_t));
    L.tokens = L.pieces + Workspace::align(size_t(L.nrows + 1) * sizeof(int32_t));
    L.dqacc = L.tokens + Workspace::align(size_t(sh.t1) * size_t(d->n2 * d->block_count) * sizeof(int32_t) + 4);
    L.dkacc = L.dqacc + Workspace::align(rows * size_t(d->d) * sizeof(float));
    L.dvacc = L.dkacc + Workspace::align(size_t(sh.t2) * size_t(d->n2 * d->d) * sizeof(float));
    L.dqpart = L.dvacc + Workspace::align(size_t(sh.t2) * size_t(d->n2 * sh.dv) * sizeof(float));
    // deterministic 1: dQ per (token, selected slot); 2: one add counter per (token, kv head)
    const size_t part_bytes = d->deterministic == 1
                                  ? size_t(sh.t1) * size_t(d->n1) * size_t(d->block_count) * size_t(d->d) * sizeof(float)
                                  : 0;
    L.sem = L.dqpart + Workspace::align(part_bytes);
    const bool ord = d->deterministic == 2;
    L.rank = L.sem + (ord ? Workspace::align(size_t(sh.t1) * size_t(d->n2) * sizeof(uint32_t)) : 0);
    L.kvpart = L.rank + (ord ? Workspace::align(size_t(sh.t1) * size_t(d->n2 * d->block_count) * sizeof(int32_t)) : 0);
    // deterministic mode 1: each work unit's dK / dV rows (block_size keys x (d + d_v) fp32)
    const size_t kv_bytes = d->deterministic == 1 ? size_t(nsa_max_pieces(L.nrows, sh.t1, d->n2, d->block_count,
                                                                           d->n1 / d->n2)) *
                                                        size_t(d->block_size) * size_t(d->d + sh.dv) * sizeof(float)
                                                  : 0;
    L.total = L.kvpart + Workspace::align(kv_bytes);
    return L;
}

// The forward runs on the tensor cores for d = d_v = 128 and blocks of 64 (the backward's block lists,
// its lse2 / dvec rows for the row maxima and sums and its dQ accumulator for O); otherwise on CUDA
// cores, which need the status word alone.
bool nsa_fwd_on_tc(const attn_nsa_desc_t *d, const NsaShape &sh)
{
    return d->d == 128 && sh.dv == 128 && d->block_size == 64;
}

NsaLayout nsa_fwd_layout(const attn_nsa_desc_t *d, const NsaShape &sh)
{
    attn_nsa_desc_t c = *d;
    c.deterministic = 0;  // no per-slot partials or add counters in the forward
    return nsa_layout(&c, sh);
}

size_t nsa_fwd_bytes(const attn_nsa_desc_t *d, const NsaShape &sh)
{
    return nsa_fwd_on_tc(d, sh) ? nsa_fwd_layout(d, sh).total : Workspace::align(64 * sizeof(uint32_t));
}

void nsa_ws_pointers(NsaArgs *a, const NsaLayout &L, void *workspace)
{
    char *ws = static_cast<char *>(workspace);
    a->status = reinterpret_cast<uint32_t *>(ws + L.status);
    a->lse2 = reinterpret_cast<float *>(ws + L.lse2);
    a->dvec = reinterpret_cast<float *>(ws + L.dvec);
    a->bitmap = reinterpret_cast<uint32_t *>(ws + L.bitmap);
    a->offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    a->tokens = reinterpret_cast<int32_t *>(ws + L.tokens);
    a->pieces = reinterpret_cast<int32_t *>(ws + L.pieces);
    a->dqacc = reinterpret_cast<float *>(ws + L.dqacc);
    a->dkacc = reinterpret_cast<float *>(ws + L.dkacc);
    a->dvacc = reinterpret_cast<float *>(ws + L.dvacc);
    a->dqpart = reinterpret_cast<float *>(ws + L.dqpart);
    a->sem = reinterpret_cast<uint32_t *>(ws + L.sem);
    a->rank = reinterpret_cast<int32_t *>(ws + L.rank);
    a->kvpart = reinterpret_cast<float *>(ws + L.kvpart);
}

}  // namespace

attn_status_t nsa_workspace_size(const attn_nsa_desc_t *desc, size_t *bytes)
{
    NsaShape sh;
    attn_status_t st = check_nsa_desc(desc, &sh);
    if (st) return st;
    if (!bytes) return ATTN_ERR_NULLPTR;
    *bytes = nsa_layout(desc, sh).total;
    return ATTN_OK;
}

attn_status_t nsa_selected_attn_bwd(const attn_nsa_desc_t *desc, const void *q, const void *k, const void *v,
                                    const void *o, const void *dO, const float *softmax_max,
                                    const float *softmax_sum, const int32_t *topk, void *dq, void *dk, void *dv,
                                    void *workspace, size_t workspace_bytes, void *stream)
{
    NsaShape sh;
    attn_status_t st = check_nsa_desc(desc, &sh);
    if (st) return st;
    if (sh.t1 > 0 && (!q || !o || !dO || !softmax_max || !softmax_sum || !topk || !dq)) return ATTN_ERR_NULLPTR;
    if (sh.t2 > 0 && (!k || !v || !dk || !dv)) return ATTN_ERR_NULLPTR;
    for (const void *p : {q, k, v, o, dO, (const void *)dq, (const void *)dk, (const void *)dv})
        if (p && !aligned16(p)) return ATTN_ERR_ALIGN;
    if ((topk && (reinterpret_cast<uintptr_t>(topk) & 3)) || (softmax_max && !aligned16(softmax_max)) ||
        (softmax_sum && !aligned16(softmax_sum)))
        return ATTN_ERR_ALIGN;
    NsaLayout L = nsa_layout(desc, sh);
    if ((st = check_ws(workspace, workspace_bytes, L.total))) return st;
    if (sh.t1 == 0 && sh.t2 == 0) return ATTN_OK;

    NsaArgs a;
    std::memset(&a, 0, sizeof a);
    a.dtype = desc->dtype;
    a.nseq = desc->b; a.n1 = desc->n1; a.n2 = desc->n2; a.d = desc->d; a.dv = sh.dv;
    a.grad_fp32 = desc->grad_fp32;
    a.bs = desc->block_size; a.cnt = desc->block_count;
    a.mask = desc->atten_mask; a.mask_cols = desc->mask_cols;
    a.t1 = sh.t1; a.t2 = sh.t2; a.t1_pad = L.t1_pad;
    a.nblk_max = sh.nblk_max; a.words_max = sh.words_max; a.nrows = L.nrows;
    a.scale = float(desc->scale);
    a.sparse_mode = desc->sparse_mode;
    a.deterministic = desc->deterministic;
    a.n_part = 1;
    a.q = q; a.k = k; a.v = v; a.o = o; a.dO = dO;
    a.smax = softmax_max; a.ssum = softmax_sum; a.topk = topk;
    a.dq = dq; a.dk = dk; a.dvp = dv;
    char *ws = static_cast<char *>(workspace);
    a.status = reinterpret_cast<uint32_t *>(ws + L.status);
    a.lse2 = reinterpret_cast<float *>(ws + L.lse2);
    a.dvec = reinterpret_cast<float *>(ws + L.dvec);
    a.bitmap = reinterpret_cast<uint32_t *>(ws + L.bitmap);
    a.offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    a.tokens = reinterpret_cast<int32_t *>(ws + L.tokens);
    a.pieces = reinterpret_cast<int32_t *>(ws + L.pieces);
    a.dqacc = reinterpret_cast<float *>(ws + L.dqacc);
    a.dkacc = reinterpret_cast<float *>(ws + L.dkacc);
    a.dvacc = reinterpret_cast<float *>(ws + L.dvacc);
    a.dqpart = reinterpret_cast<float *>(ws + L.dqpart);
    a.sem = reinterpret_cast<uint32_t *>(ws + L.sem);
    a.rank = reinterpret_cast<int32_t *>(ws + L.rank);
    a.kvpart = reinterpret_cast<float *>(ws + L.kvpart);
    // the CUDA-core kernel (a head dim of 192) adds dK / dV atomically from many blocks
    if (a.deterministic && !nsa_tc_supported(a)) return ATTN_ERR_UNSUPPORTED;
    static thread_local PackedGeo pg;
    pg.nseq = desc->b;
    pg.cu_q[0] = pg.cu_kv[0] = 0;
    for (int64_t b = 0; b < desc->b; ++b) {
        pg.cu_q[b + 1] = desc->cu_seqlens_q[b];
        pg.cu_kv[b + 1] = desc->cu_seqlens_kv[b];
    }
    return cuda_status(launch_nsa_bwd(a, pg, static_cast<cudaStream_t>(stream), g_ev_before, g_ev_after));
}

attn_status_t nsa_fwd_workspace_size(const attn_nsa_desc_t *desc, size_t *bytes)
{
    NsaShape sh;
    attn_status_t st = check_nsa_desc(desc, &sh);
    if (st) return st;
    if (!bytes) return ATTN_ERR_NULLPTR;
    *bytes = nsa_fwd_bytes(desc, sh);
    return ATTN_OK;
}

attn_status_t nsa_selected_attn_fwd(const attn_nsa_desc_t *desc, const void *q, const void *k, const void *v,
                                    const int32_t *topk, void *o, float *softmax_max, float *softmax_sum,
                                    void *workspace, size_t workspace_bytes, void *stream)
{
    NsaShape sh;
    attn_status_t st = check_nsa_desc(desc, &sh);
    if (st) return st;
    if (sh.t1 > 0 && (!q || !o || !softmax_max || !softmax_sum || !topk)) return ATTN_ERR_NULLPTR;
    if (sh.t2 > 0 && (!k || !v)) return ATTN_ERR_NULLPTR;
    for (const void *p : {q, k, v, (const void *)o})
        if (p && !aligned16(p)) return ATTN_ERR_ALIGN;
    if ((topk && (reinterpret_cast<uintptr_t>(topk) & 3)) || (softmax_max && !aligned16(softmax_max)) ||
        (softmax_sum && !aligned16(softmax_sum)))
        return ATTN_ERR_ALIGN;
    if ((st = check_ws(workspace, workspace_bytes, nsa_fwd_bytes(desc, sh)))) return st;
    if (sh.t1 == 0) return ATTN_OK;
    NsaArgs a;
    std::memset(&a, 0, sizeof a);
    if (nsa_fwd_on_tc(desc, sh)) {
        const NsaLayout L = nsa_fwd_layout(desc, sh);
        a.t1_pad = L.t1_pad;
        a.nblk_max = sh.nblk_max; a.words_max = sh.words_max; a.nrows = L.nrows;
        nsa_ws_pointers(&a, L, workspace);
    } else {
        a.status = static_cast<uint32_t *>(workspace);
    }
    a.dtype = desc->dtype;
    a.nseq = desc->b; a.n1 = desc->n1; a.n2 = desc->n2; a.d = desc->d; a.dv = sh.dv;
    a.bs = desc->block_size; a.cnt = desc->block_count;
    a.mask = desc->atten_mask; a.mask_cols = desc->mask_cols;
    a.t1 = sh.t1; a.t2 = sh.t2;
    a.scale = float(desc->scale);
    a.sparse_mode = desc->sparse_mode;
    a.q = q; a.k = k; a.v = v; a.topk = topk;
    a.o_out = o; a.smax_out = softmax_max; a.ssum_out = softmax_sum;
    static thread_local PackedGeo pg;
    pg.nseq = desc->b;
    pg.cu_q[0] = pg.cu_kv[0] = 0;
    for (int64_t b = 0; b < desc->b; ++b) {
        pg.cu_q[b + 1] = desc->cu_seqlens_q[b];
        pg.cu_kv[b + 1] = desc->cu_seqlens_kv[b];
    }
    return cuda_status(launch_nsa_fwd(a, pg, static_cast<cudaStream_t>(stream)));
}

attn_status_t nsa_block_lists(const attn_nsa_desc_t *desc, const int32_t *topk, int32_t *offsets, int32_t *tokens,
                              int64_t *nblk_max_out, void *workspace, size_t workspace_bytes, void *stream)
{
    NsaShape sh;
    attn_status_t st = check_nsa_desc(desc, &sh);
    if (st) return st;
    if (!offsets || !tokens || !nblk_max_out || (sh.t1 > 0 && !topk)) return ATTN_ERR_NULLPTR;
    if (reinterpret_cast<uintptr_t>(topk) & 3) return ATTN_ERR_ALIGN;
    NsaLayout L = nsa_layout(desc, sh);
    if ((st = check_ws(workspace, workspace_bytes, L.total))) return st;
    *nblk_max_out = sh.nblk_max;
    NsaArgs a;
    std::memset(&a, 0, sizeof a);
    a.dtype = desc->dtype;
    a.nseq = desc->b; a.n1 = desc->n1; a.n2 = desc->n2; a.d = desc->d; a.dv = sh.dv;
    a.grad_fp32 = desc->grad_fp32;
    a.bs = desc->block_size; a.cnt = desc->block_count;
    a.mask = desc->atten_mask; a.mask_cols = desc->mask_cols;
    a.t1 = sh.t1; a.t2 = sh.t2; a.t1_pad = L.t1_pad;
    a.nblk_max = sh.nblk_max; a.words_max = sh.words_max; a.nrows = L.nrows;
    a.sparse_mode = desc->sparse_mode;
    a.topk = topk;
    char *ws = static_cast<char *>(workspace);
    a.status = reinterpret_cast<uint32_t *>(ws + L.status);
    a.bitmap = reinterpret_cast<uint32_t *>(ws + L.bitmap);
    a.offsets = offsets;
    a.tokens = tokens;
    static thread_local PackedGeo pg;
    pg.nseq = desc->b;
    pg.cu_q[0] = pg.cu_kv[0] = 0;
    for (int64_t b = 0; b < desc->b; ++b) {
        pg.cu_q[b + 1] = desc->cu_seqlens_q[b];
        pg.cu_kv[b + 1] = desc->cu_seqlens_kv[b];
    }
    return cuda_status(launch_nsa_block_lists(a, pg, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_set_main_kernel_events(void *before, void *after)
{
    g_ev_before = static_cast<cudaEvent_t>(before);
    g_ev_after = static_cast<cudaEvent_t>(after);
    return ATTN_OK;
}

attn_status_t attn_query_status(void *workspace, void *stream, uint32_t *device_flags)
{
    if (!workspace || !device_flags) return ATTN_ERR_NULLPTR;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_status(e);
    uint32_t flags = 0;
    if ((e = cudaMemcpy(&flags, workspace, sizeof flags, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_status(e);
    if (flags && (e = cudaMemset(workspace, 0, sizeof flags)) != cudaSuccess) return cuda_status(e);
    *device_flags = flags;
    return flags ? ATTN_ERR_DEVICE : ATTN_OK;
}

}  // extern "C"
