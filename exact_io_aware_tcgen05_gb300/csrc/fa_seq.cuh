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

// fp8 layouts: the column of sequence b's first 128-token block in a [heads, nb]
// block-scale array (the blocks of the earlier sequences, ceil(len / 128) each);
// 128 times it is the column of its first key in the transposed V layout, where
// every sequence is padded to a multiple of 128 keys.
__device__ __forceinline__ int seq_block_col(const SeqInfo& s, int b) {
    if (!s.cu_seqlens) return b * ceil_div(s.N, 128);
    int acc = 0;
    for (int i = 0; i < b; ++i) {
        int st, len;
        seq_bounds(s, i, st, len);
        acc += ceil_div(len, 128);
    }
    return acc;
}

// Heads per scheduling chunk (see map_work) unless the launcher picks another.
constexpr int kHeadChunk = 8;

// Maps CTA index w to (sequence b, head h, block index blk of `rows` rows).
// Heads are taken in chunks of `chunk`: all work items of a chunk are launched
// before the next chunk's, so the CTAs in flight touch few heads and the tiles
// they share stay in L2.  Within a chunk the order is by "level": level 0 is the
// most expensive block of every head of the chunk, level 1 the next, and so on
// (longest first); the most expensive block is the last one for query blocks
// under a causal mask (`from_end`), the first for key blocks.  A wider chunk
// shortens the tail (the last chunk's long items start earlier) at the price of
// a larger working set.  Returns false for CTAs beyond the real work (packed
// batches launch an upper bound).
__device__ __forceinline__ bool map_work(const SeqInfo& s, int w, int rows, int heads,
                                         bool from_end, int& b, int& h, int& blk,
                                         int chunk = kHeadChunk) {
    int n, first_bh, nbh, r;   // blocks per head, first (seq, head) pair of the range, pairs, index
    if (!s.cu_seqlens) {
        n = ceil_div(s.N, rows);
        const int pairs = s.B * heads;
        if (w >= n * pairs) return false;
        const int c = w / (n * chunk);
        first_bh = c * chunk;
        nbh = min(chunk, pairs - first_bh);
        r = w - first_bh * n;
    } else {
        // sequences in order; within a sequence its heads in chunks
        int base = 0;
        for (b = 0; b < s.B; ++b) {
            int st, len;
            seq_bounds(s, b, st, len);
            n = ceil_div(len, rows);
            if (w < base + n * heads) break;
            base += n * heads;
        }
        if (b >= s.B) return false;
        const int idx = w - base;
        const int c = idx / (n * chunk);
        first_bh = b * heads + c * chunk;
        nbh = min(chunk, heads - c * chunk);
        r = idx - c * chunk * n;
    }
    const int level = r / nbh;
    const int bh = first_bh + r % nbh;
    b = bh / heads;
    h = bh % heads;
    blk = from_end ? n - 1 - level : level;
    return true;
}

}  // namespace fa
