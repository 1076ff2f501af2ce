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

// Number of work items of "level" below V: sum_b min(nblk_b, V), where
// nblk_b = ceil(len_b / rows).
__device__ __forceinline__ int items_below_level(const SeqInfo& s, int rows, int V) {
    int c = 0;
    for (int b = 0; b < s.B; ++b) {
        int st, len;
        seq_bounds(s, b, st, len);
        c += min(ceil_div(len, rows), V);
    }
    return c;
}

// Maps CTA index w to (sequence b, head h, block index blk of `rows` rows).
// Heads vary fastest.  Blocks are ordered by level: level 0 holds the most
// expensive block of every sequence, level 1 the next, and so on, so the
// heaviest work items start first.  `from_end` selects whether the most
// expensive block of a sequence is its last (query blocks under a causal
// mask) or its first (key blocks under a causal mask).  Returns false for
// CTAs beyond the real work (packed batches launch an upper bound).
__device__ __forceinline__ bool map_work(const SeqInfo& s, int w, int rows, int heads,
                                         bool from_end, int& b, int& h, int& blk) {
    h = w % heads;
    int r = w / heads;
    if (!s.cu_seqlens) {
        int nblk = ceil_div(s.N, rows);
        if (r >= nblk * s.B) return false;
        b = r % s.B;
        int v = r / s.B;
        blk = from_end ? nblk - 1 - v : v;
        return true;
    }
    const int max_level = ceil_div(s.N, rows);
    if (r >= items_below_level(s, rows, max_level)) return false;
    // largest v with items_below_level(v) <= r
    int lo = 0, hi = max_level;  // invariant: below(lo) <= r < below(hi)
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (items_below_level(s, rows, mid) <= r) lo = mid;
        else hi = mid;
    }
    const int v = lo;
    int idx = r - items_below_level(s, rows, v);
    for (b = 0; b < s.B; ++b) {
        int st, len;
        seq_bounds(s, b, st, len);
        int n = ceil_div(len, rows);
        if (n > v) {
            if (idx == 0) break;
            --idx;
        }
    }
    if (b >= s.B) return false;
    int st, len;
    seq_bounds(s, b, st, len);
    int n = ceil_div(len, rows);
    blk = from_end ? n - 1 - v : v;
    return true;
}

}  // namespace fa
