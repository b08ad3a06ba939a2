/*
 * attnbwd.h -- C ABI of the GB300 (sm_103a) attention-backward library.
 *
 * Three computations, each a stateless, asynchronous call on the caller's
 * CUDA stream (passed as void*; NULL is the legacy default stream):
 *
 *   sdpa_fwd_stats          O and the fp32 log-sum-exp stats of scaled dot
 *                           product attention (training-mode forward).
 *   sdpa_bwd                dQ, dK, dV of the same attention, FlashAttention-2
 *                           form: P is recomputed from the saved stats.
 *   nsa_selected_attn_bwd   dQ, dK, dV of NSA selected attention, where every
 *                           query token attends to selectedBlockCount blocks of
 *                           selectedBlockSize keys chosen by int32 topkIndices.
 *
 * Definitions.  With s_ij = scale * q_i . k_j over the visible keys,
 *   LSE_i = log sum_j exp(s_ij),  P_ij = exp(s_ij - LSE_i),  O_i = sum_j P_ij v_j,
 *   D_i = rowsum(dO_i * O_i),  dP = dO V^T,  dS = P * (dP - D),
 *   dV = P^T dO,  dQ = scale dS K,  dK = scale dS^T Q.
 * Pages cited below by title and section:
 *   [cuDNN]  cuDNN-frontend sample "51_scaled_dot_product_attention_backward"
 *   [Ascend] Ascend CANN page "aclnnNsaSelectedAttentionGrad"
 *   [PR]     PyTorch PR #94729 (matmul -> scale -> softmax -> matmul pattern)
 * Each call below names the passage that defines it.
 *
 * Conventions shared by every call.
 *  - Tensors are caller-owned device memory.  The library allocates nothing,
 *    keeps no state between calls, and fully overwrites its outputs.
 *  - The workspace is caller-owned device memory of at least the size the
 *    matching *_workspace_size call returns, 256-byte aligned.  Its contents
 *    need not be initialised.  Two calls in flight at once must not share it.
 *  - Every argument check runs on the host before anything is launched; a
 *    call that returns an error has launched nothing.  Errors the device
 *    finds (an index out of range, a duplicate selected block, a bounded wait
 *    that ran out) never trap: they set bits in a status word inside the
 *    workspace that attn_query_status reads back.
 *  - 16-bit tensors (fp16 or bf16, one type per call) must start on a 16-byte
 *    boundary and have element strides that are multiples of 8 (16 bytes);
 *    the innermost (head-dim) stride is 1.  Otherwise ATTN_ERR_ALIGN.
 *  - Query head hq uses key/value head hq / (h / h_kv).
 *  - A query row that sees no key (possible only when a bottom-right causal
 *    mask meets s_q > s_kv) has O = 0, LSE = +inf and zero gradients.
 */
#ifndef ATTNBWD_H
#define ATTNBWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  [Ascend] "Return Value" table: a call returns a code; the
 * page's parameter-check failures map to NULLPTR / INVALID here, and its
 * run-time failure code to ATTN_ERR_CUDA.  Deviation from a single
 * "timeout" code: device-side failures (a wait that ran out, a bad index)
 * cannot be returned by an asynchronous call, so they set bits of a device
 * status word (ATTN_DEV_*), and attn_query_status returns ATTN_ERR_DEVICE
 * with those bits in *device_flags.                                          */
typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULLPTR = 1,     /* a required pointer is NULL                    */
    ATTN_ERR_INVALID = 2,     /* a size, dtype, mode or stride is not valid    */
    ATTN_ERR_UNSUPPORTED = 3, /* valid, but outside what the kernels cover     */
    ATTN_ERR_WORKSPACE = 4,   /* workspace NULL, too small or misaligned       */
    ATTN_ERR_ALIGN = 5,       /* a tensor breaks the 16-byte rule above        */
    ATTN_ERR_CUDA = 6,        /* a CUDA runtime / driver call failed           */
    ATTN_ERR_DEVICE = 7       /* attn_query_status: the device flagged an error */
} attn_status_t;

/* Bits of the device status word (attn_query_status).                        */
#define ATTN_DEV_TIMEOUT      0x1u  /* a bounded barrier wait ran out; the CTA quit */
#define ATTN_DEV_INDEX_RANGE  0x2u  /* a topk index outside [0, S2_b / block_size)   */
#define ATTN_DEV_INDEX_DUP    0x4u  /* a block listed twice for one (token, kv head) */

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1 } attn_dtype_t;

/* Causal alignment.  Top-left: key j is visible to query i iff j <= i.
 * Bottom-right: iff j <= i + (s_kv - s_q).  Both coincide when s_q == s_kv.   */
typedef enum {
    ATTN_MASK_NONE = 0,
    ATTN_CAUSAL_TOP_LEFT = 1,
    ATTN_CAUSAL_BOTTOM_RIGHT = 2
} attn_mask_t;

/* A 16-bit tensor seen as logical [B, H, S, D] with element strides
 * (sb, sh, ss, 1).  The sample's BSHD storage viewed as BHSD has
 * (S*H*D, D, H*D, 1).  In packed (varlen, TND) mode token t of head h is at
 * ptr + t*ss + h*sh and sb is ignored.                                       */
typedef struct {
    void *ptr;
    int64_t sb, sh, ss;
} attn_view_t;

typedef struct {
    attn_dtype_t dtype;
    int64_t b;              /* batch size (number of sequences)                */
    int64_t h;              /* query heads                                     */
    int64_t h_kv;           /* key/value heads; h % h_kv == 0                  */
    int64_t s_q, s_kv;      /* fixed lengths; ignored in packed mode           */
    int64_t d;              /* head dim: 64 or 128                             */
    double scale;           /* multiplies q.k, e.g. 1/sqrt(d)                  */
    attn_mask_t mask;
    /* Packed mode: host arrays of b inclusive cumulative lengths, no leading
     * zero (the Ascend page's actualSeqQLen / actualSeqKvLen form), b <= 256.
     * Both NULL: fixed-length mode.                                          */
    const int64_t *cu_seqlens_q;
    const int64_t *cu_seqlens_kv;
    /* sdpa_bwd only: an attn_dq_mode_t.  ATTN_DQ_ATOMIC: dQ accumulated with
     * fp32 reductions whose order varies from run to run.  ATTN_DQ_SPLIT:
     * bitwise reproducible dQ; each of dq_splits partial fp32 buffers (0: a
     * default) has one writer that adds in a fixed order, and the buffers are
     * summed in index order.  ATTN_DQ_ORDERED: bitwise reproducible dQ with
     * one fp32 buffer; the key tiles of each query tile add in decreasing
     * order, each waiting for a per-tile counter in the workspace (bounded
     * wait: ATTN_DEV_TIMEOUT), under a cooperative launch (every block of the
     * kernel resident at once); problems of more than 4096 work units (key
     * tiles of 128 rows x sequences x kv heads) return ATTN_ERR_UNSUPPORTED.
     * [Ascend] "Constraints": deterministic computation is opt-in.          */
    int deterministic;
    int dq_splits;
} attn_sdpa_desc_t;

typedef enum { ATTN_DQ_ATOMIC = 0, ATTN_DQ_SPLIT = 1, ATTN_DQ_ORDERED = 2 } attn_dq_mode_t;

/* Workspace bytes for sdpa_fwd_stats and for sdpa_bwd with this descriptor.
 * Either output pointer may be NULL.  Host only; no CUDA call.
 * [cuDNN] workspace cell (the caller queries the graph's workspace size and
 * allocates it); [Ascend] "Function Prototype" (first phase of the two-phase
 * API returns workspaceSize).                                               */
attn_status_t sdpa_workspace_size(const attn_sdpa_desc_t *desc, size_t *fwd_bytes, size_t *bwd_bytes);

/* Forward in training mode.  [cuDNN] forward-graph cell (sdpa with
 * is_inference=False, attn_scale, causal mask, emitting O and the (B,H,S,1)
 * float32 stats); [PR] the attention formula (softmax of scaled scores times
 * V).  q, o: [B,h,s_q,d] views; k, v: [B,h_kv,s_kv,d].
 * lse (fp32, natural log, contiguous): [B][h][s_q] in fixed-length mode,
 * [h][T_q] in packed mode (T_q = total query tokens).                        */
attn_status_t sdpa_fwd_stats(const attn_sdpa_desc_t *desc, attn_view_t q, attn_view_t k, attn_view_t v,
                             attn_view_t o, float *lse, void *workspace, size_t workspace_bytes,
                             void *stream);

/* Backward.  [cuDNN] backward-graph cell (sdpa_backward from Q, K, V, O, dO
 * and the stats, FlashAttention-2, attn_scale, causal mask; dQ, dK, dV
 * allocated like the inputs); [Ascend] "Function / Formula" for the
 * gradient formulas; [Ascend] "Constraints" for opt-in deterministic
 * computation.  q, o, dO, dQ: [B,h,s_q,d] views; k, v, dK, dV: [B,h_kv,s_kv,d];
 * lse as sdpa_fwd_stats writes it.  dQ / dK / dV may have any strides that
 * follow the 16-byte rule (the sample allocates them empty_like the inputs).
 * Outputs have the input dtype, rounded to nearest even.  No block of any
 * kernel waits for another block (in ATTN_DQ_ORDERED, blocks wait for one
 * another under a cooperative launch, which starts once all of them can be
 * resident), so the call is safe next to other work on the device (other
 * streams, other processes).                                                */
attn_status_t sdpa_bwd(const attn_sdpa_desc_t *desc, attn_view_t q, attn_view_t k, attn_view_t v,
                       attn_view_t o, attn_view_t dO, const float *lse, attn_view_t dQ, attn_view_t dK,
                       attn_view_t dV, void *workspace, size_t workspace_bytes, void *stream);

/* Allocation-free variant of sdpa_bwd.  The pages this library follows
 * have no counterpart to it; it exists for callers that cannot allocate
 * device memory when they run the backward (an engine or plugin that owns
 * all device memory and forbids side allocations, a loop that must not
 * allocate once running).  Instead of a caller workspace it uses a static
 * scratch array of ATTN_STATIC_SCRATCH_BYTES compiled into the library;
 * every GPU that loads the library holds those bytes until the process exits.
 * Arguments and results are those of sdpa_bwd; the call allocates nothing.
 *  - Problems whose sdpa_workspace_size exceeds ATTN_STATIC_SCRATCH_BYTES
 *    are rejected with ATTN_ERR_WORKSPACE before anything is launched.
 *  - The first call on a device looks up the array's device address (once
 *    per device, with that device current); make that first call before any
 *    stream capture begins.
 *  - All calls share the one array, so calls that overlap on the GPU (other
 *    streams, other host threads) race and corrupt each other's results;
 *    serialise them.  Each call re-initialises the scratch it reads, so what
 *    an earlier call left there does not matter.
 *  - Device status flags land in the static array; attn_static_scratch_status
 *    reads them back (and clears them) like attn_query_status.
 *  - The array's device address is looked up on every call (nothing is
 *    cached across contexts or cudaDeviceReset); errors of that lookup return
 *    ATTN_ERR_CUDA with the text in attn_last_error.                         */
#define ATTN_STATIC_SCRATCH_BYTES (16u << 20)
attn_status_t sdpa_bwd_static_scratch(const attn_sdpa_desc_t *desc, attn_view_t q, attn_view_t k, attn_view_t v,
                                      attn_view_t o, attn_view_t dO, const float *lse, attn_view_t dQ,
                                      attn_view_t dK, attn_view_t dV, void *stream);

/* Waits for the stream, then reads and clears the device status word that
 * the static scratch of sdpa_bwd_static_scratch holds (bits ATTN_DEV_*).
 * Returns ATTN_ERR_DEVICE when any bit was set.  No counterpart on the
 * pages.                                                                    */
attn_status_t attn_static_scratch_status(void *stream, uint32_t *device_flags);

typedef struct {
    attn_dtype_t dtype;
    int64_t b;              /* sequences; b <= 256                             */
    const int64_t *cu_seqlens_q;   /* host, b inclusive cumulative lengths   */
    const int64_t *cu_seqlens_kv;  /* host, b inclusive cumulative lengths   */
    int64_t n1;             /* query heads (headNum)                          */
    int64_t n2;             /* key/value heads; n1 % n2 == 0, n1/n2 <= 32     */
    int64_t d;              /* head dim of q and k: 128 or 192                */
    double scale;           /* scaleValue                                     */
    int64_t block_size;     /* selectedBlockSize: 64                          */
    int64_t block_count;    /* selectedBlockCount in [1, 128], count*size < 8192 */
    int sparse_mode;        /* 0: only the selection; 2: also causal,
                               bottom-right aligned per sequence              */
    int deterministic;      /* bitwise reproducible dQ, dK, dV, needing
                               d = d_v = 128 (ATTN_ERR_UNSUPPORTED otherwise):
                               0 off; 1 dQ per (token, selected slot) in the
                               workspace, summed in slot order (T1 n1
                               block_count d 4 bytes, plus the dK / dV rows of
                               every work unit); 2 one dQ accumulator
                               whose adds for a token go in decreasing block
                               order behind a counter per (token, kv head)
                               (T1 n2 (block_count + 1) 4 bytes; a
                               cooperative launch)                            */
    int64_t d_v;            /* head dim of v, O, dO and dv: 128 or 192; 0 means
                               d ([Ascend] Constraints: D is 192 or 128, and K
                               and V may differ)                              */
    int grad_fp32;          /* 1: dq, dk, dv are fp32; 0: the input dtype
                               ([Ascend] parameter table: FLOAT16, BFLOAT16,
                               FLOAT32 outputs)                               */
    /* attenMaskOptional ([Ascend] function prototype and parameter table: a
     * 2-D BOOL / UINT8 mask that no formula on the page uses).  Read here as:
     * device array [mask_rows][mask_cols] of uint8, row-major; entry (i, j)
     * nonzero removes key j for query i (positions local to the sequence),
     * on top of the selection and the sparse mode; it must cover every
     * sequence (mask_rows >= its query length, mask_cols >= its key length).
     * NULL: no mask.                                                       */
    const uint8_t *atten_mask;
    int64_t mask_rows, mask_cols;
} attn_nsa_desc_t;

/* NSA selected-attention forward (training mode): O and the softmax stats the
 * backward reads.  [Ascend] "Function / Formula" (gather of the selected
 * blocks, then attention over them) and parameter table (softmaxMax /
 * softmaxSum [T1, N1, 8]).  For query token t, kv head g and query head
 * h of g, over the keys of the selected blocks that the sparse mode leaves
 * visible: softmax_max = max_j s_j with s_j = scale q.k_j, softmax_sum =
 * sum_j exp(s_j - softmax_max), O = sum_j exp(s_j - softmax_max) v_j /
 * softmax_sum; all 8 lanes of a stats row hold the same value.  A row that
 * sees no key has O = 0, softmax_max = -inf, softmax_sum = 0.
 *   q : [T1][n1][d]  k : [T2][n2][d]  v : [T2][n2][d_v]  o : [T1][n1][d_v]
 *   topk : as for the backward; invalid indices are skipped and flagged.
 * Workspace: nsa_fwd_workspace_size bytes (d = d_v = 128 with blocks of 64
 * runs on the tensor cores and needs the backward's block lists and fp32
 * row / O accumulators; other shapes need the device status word alone). */
attn_status_t nsa_fwd_workspace_size(const attn_nsa_desc_t *desc, size_t *bytes);
attn_status_t nsa_selected_attn_fwd(const attn_nsa_desc_t *desc, const void *q, const void *k, const void *v,
                                    const int32_t *topk, void *o, float *softmax_max, float *softmax_sum,
                                    void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes for nsa_selected_attn_bwd.  Host only; no CUDA call.
 * [Ascend] "Function Prototype": aclnnNsaSelectedAttentionGradGetWorkspaceSize. */
attn_status_t nsa_workspace_size(const attn_nsa_desc_t *desc, size_t *bytes);

/* NSA selected-attention backward.  [Ascend] "Function / Formula" (gather of
 * the selected blocks, then the attention backward; dK / dV scattered back
 * through the indices), parameter table (TND layout, actualSeqQLen /
 * actualSeqKvLen, softmaxMax / softmaxSum, topkIndices, scaleValue,
 * selectedBlockSize / Count, sparseMode) and "Constraints".  Layout, all
 * contiguous (d_v = value head dim):
 *   q, dq : [T1][n1][d]    o, dO : [T1][n1][d_v]
 *   k, dk : [T2][n2][d]    v, dv : [T2][n2][d_v]
 *   dq, dk, dv are fp32 when grad_fp32 is set, else the input dtype.
 *   softmax_max, softmax_sum : [T1][n1][8] fp32 (the 8 lanes hold one value;
 *       lane 0 is read): P = exp(scale q.k - max) / sum over the selection.
 *   topk : [T1][n2][block_count] int32 block ids local to the token's
 *       sequence, each in [0, S2_b / block_size), distinct per (token, head).
 * Every selected block must lie inside its sequence: S2_b % block_size == 0
 * and S2_b >= block_count * block_size for every sequence.  As for sdpa_bwd,
 * blocks wait for one another only in deterministic mode 2, under a
 * cooperative launch.                                                        */
attn_status_t nsa_selected_attn_bwd(const attn_nsa_desc_t *desc, const void *q, const void *k,
                                    const void *v, const void *o, const void *dO,
                                    const float *softmax_max, const float *softmax_sum,
                                    const int32_t *topk, void *dq, void *dk, void *dv,
                                    void *workspace, size_t workspace_bytes, void *stream);

/* [Ascend] "Function / Formula" (Gather(key, topkIndices)), read in the
 * backward direction: which tokens selected each block.
 * The inverted index the NSA backward builds internally, exposed so callers
 * (and tests) can use or check it: for every (sequence b, kv head g, block k)
 * in that order, row r = (b * n2 + g) * nblk_max + k with
 * nblk_max = max_b S2_b / block_size, tokens[offsets[r] .. offsets[r+1]) are
 * the ascending global ids of the query tokens whose topk lists block k and
 * see at least one of its keys under the sparse mode.  offsets (int32,
 * nblk_max * n2 * b + 1 entries) and tokens (int32, T1 * n2 * block_count
 * entries) are device memory; *nblk_max_out (host) receives nblk_max.
 * Invalid indices are skipped and flagged in the device status word.        */
attn_status_t nsa_block_lists(const attn_nsa_desc_t *desc, const int32_t *topk, int32_t *offsets,
                              int32_t *tokens, int64_t *nblk_max_out, void *workspace, size_t workspace_bytes,
                              void *stream);

/* Waits for the stream, then reads the device status word of a workspace a
 * previous call used (bits ATTN_DEV_*; 0 when clean) and clears it.
 * Returns ATTN_ERR_DEVICE when any bit was set.  [Ascend] "Return Value"
 * (failures reported as codes); see the deviation note above the enum.     */
attn_status_t attn_query_status(void *workspace, void *stream, uint32_t *device_flags);

/* Self-test of the device failure path: launches one block whose bounded
 * mbarrier wait (the same wait every tensor-core kernel uses) can never
 * complete, so after about limit_s seconds (0 < limit_s <= 2) it gives up,
 * sets ATTN_DEV_TIMEOUT in the status word at `workspace` (at least 4 bytes,
 * 4-byte aligned) and returns; the context stays usable.  Read the flag with
 * attn_query_status.  [Ascend] "Return Value" (failures as codes, never a
 * crash).                                                                   */
attn_status_t attn_selftest_wait_timeout(void *workspace, size_t workspace_bytes, double limit_s, void *stream);

/* Test aid: launches `blocks` blocks of 32 threads that each reserve
 * smem_bytes (<= 200 KiB) of shared memory and hold their SM for `seconds`
 * (0 < seconds <= 5) without touching memory, so a test can run the
 * backward while other work occupies part of the GPU.  No counterpart on the
 * pages.                                                                    */
attn_status_t attn_selftest_occupy(int blocks, size_t smem_bytes, double seconds, void *stream);

/* Optional instrumentation for benchmarks.  While set, every sdpa_bwd and
 * nsa_selected_attn_bwd call made from this host thread records the CUDA
 * event `before` on its stream just before its main backward kernel and
 * `after` just after it, so the main kernel can be timed alone.  Events are
 * cudaEvent_t handles passed as void*; NULL, NULL clears.  Never fails.    */
attn_status_t attn_set_main_kernel_events(void *before, void *after);

/* Text of the CUDA runtime / driver error behind the most recent
 * ATTN_ERR_CUDA returned to this host thread ("" if none).  Static storage. */
const char *attn_last_error(void);

/* Human-readable name of a status code (static storage).                    */
const char *attn_status_string(attn_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* ATTNBWD_H */
