// Host-only check of the dense backward's work-unit plans (no GPU needed; built by
// tests/test_plan_host.py with nvcc, which compiles the kernels alongside but never launches them).
// For each shape it prints: name, plan on/off, units planned, units with work, units planned twice,
// and whether every CTA's list in the ordered dQ mode takes key tiles in non-increasing order (the
// condition under which the ordered mode's waits cannot form a cycle).
#include <cstdio>
#include <cstring>
#include <vector>

#include "bwd_tc.cu"
using namespace attn;

template <int BM, int BN, class Geo>
void check(const char *name, DenseArgs a, const Geo &g, int64_t units, int64_t ctas)
{
    static TcSched S;
    plan_units<BM, BN>(S, a, g, units, ctas);
    const int64_t nheads = a.nseq * a.h_kv;
    std::vector<int> seen(size_t(units), 0);
    int64_t planned = 0, with_work = 0, twice = 0;
    bool ordered_ok = true;
    for (int64_t u = 0; u < units; ++u) {
        const int64_t jt0 = u / nheads, b = (u % nheads) / a.h_kv;
        with_work += jt0 * BN < g.kv_len(b) ? 1 : 0;  // a unit with a key tile in its sequence
    }
    if (S.on)
        for (int64_t c = 0; c < ctas; ++c) {
            int64_t prev_jt = INT64_MAX;
            for (int k = S.off[c]; k < S.off[c + 1]; ++k) {
                const int u = S.unit[k];
                ++planned;
                if (++seen[size_t(u)] > 1) ++twice;
                const int64_t jt = u / nheads;
                if (a.ordered && jt > prev_jt) ordered_ok = false;
                prev_jt = jt;
            }
        }
    printf("%s on %d planned %lld work %lld twice %lld ordered_ok %d\n", name, S.on, (long long)planned,
           (long long)with_work, (long long)twice, ordered_ok ? 1 : 0);
}

PackedGeo packed(const std::vector<int64_t> &lq, const std::vector<int64_t> &lkv)
{
    PackedGeo g;
    memset(&g, 0, sizeof g);
    g.nseq = int64_t(lq.size());
    for (size_t b = 0; b < lq.size(); ++b) {
        g.cu_q[b + 1] = g.cu_q[b] + lq[b];
        g.cu_kv[b + 1] = g.cu_kv[b] + lkv[b];
        g.ws_q[b + 1] = g.ws_q[b] + (lq[b] + 127) / 128 * 128;
    }
    return g;
}

// The NSA ordered deterministic mode's unit order (nsa_ord_row): a permutation of the block-list rows in
// which blocks never increase, so the pieces dealt to a CTA (every grid-th one, in that order) take
// non-increasing blocks and every wait points to a block above.
void check_nsa_order(int64_t nseq, int64_t n2, int64_t nblk)
{
    NsaArgs a;
    memset(&a, 0, sizeof a);
    a.nseq = nseq; a.n2 = n2; a.nblk_max = nblk; a.nrows = nseq * n2 * nblk;
    std::vector<int> seen(size_t(a.nrows), 0);
    bool perm = true, mono = true;
    int64_t prev_blk = INT64_MAX;
    for (int64_t q = 0; q < a.nrows; ++q) {
        const int64_t row = nsa_ord_row(a, q);
        if (row < 0 || row >= a.nrows || seen[size_t(row)]++) perm = false;
        const int64_t blk = row % nblk;
        if (blk > prev_blk) mono = false;
        prev_blk = blk;
    }
    printf("nsa_order_%lldx%lldx%lld on 1 perm %d mono %d\n", (long long)nseq, (long long)n2, (long long)nblk,
           perm ? 1 : 0, mono ? 1 : 0);
}

int main()
{
    check_nsa_order(4, 1, 64);
    check_nsa_order(3, 2, 17);
    check_nsa_order(1, 8, 5);
    DenseArgs a;
    for (int mode = 0; mode < 3; ++mode) {  // atomic, split (8 partial buffers), ordered
        const char *tag = mode == 0 ? "atomic" : mode == 1 ? "split" : "ordered";
        char name[64];
        memset(&a, 0, sizeof a);
        a.deterministic = mode == 1;
        a.ordered = mode == 2;
        a.n_part = mode == 1 ? 8 : 1;
        // b4 h12 s1024 d64, causal top-left
        a.nseq = 4; a.h = 12; a.h_kv = 12; a.d = 64; a.mask = ATTN_CAUSAL_TOP_LEFT;
        a.t_q = a.t_kv = a.t_pad = 4096;
        const FixedGeo g1{4, 1024, 1024};
        snprintf(name, sizeof name, "w1_%s", tag);
        check<128, 128>(name, a, g1, 8 * 48, 152);
        // b2 h32 s4096 d128, causal top-left
        a.nseq = 2; a.h = 32; a.h_kv = 32; a.d = 128;
        a.t_q = a.t_kv = a.t_pad = 8192;
        const FixedGeo g2{2, 4096, 4096};
        snprintf(name, sizeof name, "w2_%s", tag);
        check<64, 128>(name, a, g2, (mode == 1 ? 8 : 32) * 64, 152);
        // non-causal, GQA 8 / 2, s_q 300, s_kv 700 (ragged tiles)
        a.nseq = 3; a.h = 8; a.h_kv = 2; a.d = 64; a.mask = ATTN_MASK_NONE;
        a.t_q = 900; a.t_kv = 2100; a.t_pad = 3 * 384;
        const FixedGeo g3{3, 300, 700};
        snprintf(name, sizeof name, "ragged_gqa_%s", tag);
        check<128, 128>(name, a, g3, (mode == 1 ? 8 : 6) * 6, 36);
        // varlen, GQA 32 / 8, causal bottom-right, 8 sequences of 2285 .. 3807 tokens
        const std::vector<int64_t> lens = {2285, 3807, 2900, 3100, 2500, 3600, 2700, 2550};
        const PackedGeo g4 = packed(lens, lens);
        a.nseq = 8; a.h = 32; a.h_kv = 8; a.d = 128; a.mask = ATTN_CAUSAL_BOTTOM_RIGHT;
        a.t_q = a.t_kv = g4.cu_q[8]; a.t_pad = g4.ws_q[8];
        snprintf(name, sizeof name, "varlen_gqa_%s", tag);
        check<64, 128>(name, a, g4, (mode == 1 ? 8 : 30) * 64, 152);
        // varlen with a sequence without keys and one without queries
        const PackedGeo g5 = packed({0, 513, 129}, {384, 0, 1000});
        a.nseq = 3; a.h = 4; a.h_kv = 4; a.d = 64; a.mask = ATTN_CAUSAL_TOP_LEFT;
        a.t_q = g5.cu_q[3]; a.t_kv = g5.cu_kv[3]; a.t_pad = g5.ws_q[3];
        snprintf(name, sizeof name, "varlen_empty_%s", tag);
        check<128, 128>(name, a, g5, 8 * 12, 64);
    }
    return 0;
}
