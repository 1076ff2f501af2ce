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

// First block slot of sequence b of a packed batch for blocks of `rows` rows:
// floor(start_b / rows) + b.  The slot ranges [first(b), first(b) + ceil(len_b /
// rows)) are disjoint, increase with b and lie below ceil(T / rows) + B, so the
// sequence that owns a slot is found by a search over cu_seqlens rather than a walk
// over all earlier sequences.
__device__ __forceinline__ int seq_first_slot(const SeqInfo& s, int b, int rows) {
    const int start = min(max(__ldg(s.cu_seqlens + b), 0), s.total_tokens);   // as seq_bounds
    return start / rows + b;
}

// The sequence b whose slot range may hold `slot`: the last b with first(b) <= slot
// (first() strictly increases with b; first(0) = 0).  A 32-way search by the whole
// warp, which must call it converged with the same arguments: each round the lanes
// test 32 evenly spaced candidates with one load each, and the count of those at
// or below `slot` (a prefix of the lanes) narrows the range 32-fold.  One round of
// loads for up to 33 sequences, two up to 1057; a binary search by one thread
// would wait for about log2(B) dependent loads.
__device__ __forceinline__ int seq_of_slot(const SeqInfo& s, int slot, int rows) {
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = s.B - 1;   // the answer lies in [lo, hi]
    while (lo < hi) {
        const int step = (hi - lo + 31) / 32;
        const int cand = lo + (lane + 1) * step;
        const bool below = cand <= hi && seq_first_slot(s, cand, rows) <= slot;
        const int k = __popc(__ballot_sync(0xffffffffu, below));
        const int nlo = lo + k * step;
        hi = min(hi, nlo + step - 1);
        lo = nlo;
    }
    return lo;
}

// fp8 layouts: the column of sequence b's first 128-token block in a [heads, nb]
// block-scale array: b ceil(N / 128) for dense batches, first(b) (above) for packed
// ones; 128 times it is the column of its first key in the transposed V layout,
// where every sequence is padded to a multiple of 128 keys.
__device__ __forceinline__ int seq_block_col(const SeqInfo& s, int b) {
    if (!s.cu_seqlens) return b * ceil_div(s.N, 128);
    return seq_first_slot(s, b, 128);
}

// Heads per scheduling chunk (see map_work) unless the launcher picks another.
constexpr int kHeadChunk = 8;

// Maps CTA index w to (sequence b, head h, block index blk of `rows` rows).  Called
// by every thread of the CTA at entry (whole warps: the packed search is per warp).
// Heads are taken in chunks of `chunk`: all work items of a chunk are launched
// before the next chunk's, so the CTAs in flight touch few heads and the tiles
// they share stay in L2.  Within a chunk the order is by "level": level 0 is the
// most expensive block of every head of the chunk, level 1 the next, and so on
// (longest first); the most expensive block is the last one for query blocks
// under a causal mask (`from_end`), the first for key blocks.  A wider chunk
// shortens the tail (the last chunk's long items start earlier) at the price of
// a larger working set.  Packed batches: sequence b owns CTA indices
// [first(b) heads, (first(b) + blocks) heads) (see seq_first_slot), sequences in
// order, within a sequence its heads in chunks.  Returns false for CTAs beyond
// the real work (packed batches launch an upper bound, with gaps).
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
        const int slot = w / heads;
        b = seq_of_slot(s, slot, rows);
        int st, len;
        seq_bounds(s, b, st, len);
        n = ceil_div(len, rows);
        const int base = seq_first_slot(s, b, rows);
        if (slot >= base + n) return false;   // a gap between sequences
        const int idx = w - base * heads;
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
