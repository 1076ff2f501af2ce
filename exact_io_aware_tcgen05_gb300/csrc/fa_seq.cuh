// fa_seq.cuh -- sequence geometry shared by the attention kernels: where a
// sequence lives in the token dimension, which keys a query row sees
// (causal / sliding-window / sequence end), and the mapping from a CTA index
// to a (sequence, head, block) work item.
#pragma once

#include "fa_kernels.h"

namespace fa {

// Clamped to the token dimension, so malformed cu_seqlens can never send a
// load or store outside [0, total_tokens).
__device__ __forceinline__ void seq_bounds(const SeqInfo& s, int b, int& start, int& len) {
    if (s.cu_seqlens) {
        start = min(max(__ldg(s.cu_seqlens + b), 0), s.total_tokens);
        const int end = min(max(__ldg(s.cu_seqlens + b + 1), start), s.total_tokens);
        len = end - start;
    } else {
        start = b * s.N;
        len = s.N;
    }
}

// Visible keys of query row q (position within its sequence of length len):
// kv in [key_lo(q), key_hi(q)].  Causal: kv <= q; window W: q - kv < W.
__device__ __forceinline__ int key_lo(const SeqInfo& s, int q) {
    return s.window > 0 ? q - s.window + 1 : 0;
}
__device__ __forceinline__ int key_hi(const SeqInfo& s, int q, int len) {
    return s.causal ? min(q, len - 1) : len - 1;
}
// Query rows that see key kv: q in [query_lo(kv), query_hi(kv)].
__device__ __forceinline__ int query_lo(const SeqInfo& s, int kv) { return s.causal ? kv : 0; }
__device__ __forceinline__ int query_hi(const SeqInfo& s, int kv, int len) {
    return s.window > 0 ? min(kv + s.window - 1, len - 1) : len - 1;
}

// Index of (sequence b, head h, row q) in the logsumexp / delta arrays:
// dense [B, Hq, N], packed [Hq, total_tokens].
__device__ __forceinline__ long long row_stat_index(const SeqInfo& s, int b, int h, int start,
                                                    int q) {
    if (s.cu_seqlens) return static_cast<long long>(h) * s.total_tokens + start + q;
    return (static_cast<long long>(b) * s.Hq + h) * s.N + q;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Maps CTA index w to (sequence b, head h, block index blk of `rows` rows).
// The work items of one (sequence, head) are consecutive, so the CTAs in
// flight at any moment touch few heads and the tiles they share stay in L2;
// within a (sequence, head) the most expensive block comes first: its last
// block for query blocks under a causal mask (`from_end`), its first for key
// blocks.  Returns false for CTAs beyond the real work (packed batches launch
// an upper bound).
__device__ __forceinline__ bool map_work(const SeqInfo& s, int w, int rows, int heads,
                                         bool from_end, int& b, int& h, int& blk) {
    if (!s.cu_seqlens) {
        const int nblk = ceil_div(s.N, rows);
        if (w >= nblk * heads * s.B) return false;
        const int t = w % nblk, bh = w / nblk;
        h = bh % heads;
        b = bh / heads;
        blk = from_end ? nblk - 1 - t : t;
        return true;
    }
    int base = 0;
    for (b = 0; b < s.B; ++b) {
        int st, len;
        seq_bounds(s, b, st, len);
        const int n = ceil_div(len, rows);
        if (w < base + n * heads) {
            const int r = w - base;
            h = r / n;
            const int t = r % n;
            blk = from_end ? n - 1 - t : t;
            return true;
        }
        base += n * heads;
    }
    return false;
}

}  // namespace fa
