// fa_fp8.cu -- quantisation of attention operands to e4m3 for the fp8 forward.
//
// The pages name block quantisation of the FP8 inputs as a FlashAttention-3
// capability ("FlashAttention: How IO-Aware Tiling and Online Softmax Solved
// Transformer Memory Bottlenecks", "FlashAttention-3" bullets) without a
// format or scale rule; the library's rule:
//   * Q, K: per (sequence, head, 128-token block of the sequence) -- the tiles of
//     the attention kernels -- scale = amax / 448 in float32 (1 for an all-zero
//     block), code = e4m3(x / scale), the division rounded to nearest in float32
//     and the code rounded to nearest even, saturating at +-448.  Scales [H, nb]:
//     block kb of sequence b at column (blocks of the sequences before b) + kb.
//   * V: per (sequence, head) one scale (the P V product sums all key blocks in
//     one accumulator), codes stored transposed, V^T [H, d, vt_tokens], sequence b
//     from column 128 * (blocks of the sequences before b), padded with zero codes
//     to a multiple of 128 keys, so every tile the attention kernel loads starts
//     on a 128-byte boundary.  Scales [H, B].
//   * Incoherent processing (Q and K, optional; the same bullets name it, again
//     undefined): every row x becomes R x = (1/sqrt d) H_d diag(sigma) x before the
//     block quantisation, H_d the Sylvester Hadamard matrix and sigma in {+1, -1}^d
//     (-1 where bit c % 32 of word c / 32 of Philox4x32-10 at counter
//     (0, 2^32 - 1, 2^32 - 1, 0), keyed by the seed, is set).  R is orthogonal, so
//     Q K^T is unchanged, while a channel much larger than the rest is spread over
//     all d.  The float32 arithmetic has one fixed order (sign flips; butterflies
//     (a, b) -> (a + b, a - b) on channel pairs (c, c + h), c & h = 0, for
//     h = 1, 2, ..., d/2, each sum rounded to nearest; one rounded product with
//     float32(1/sqrt d)), so the codes are reproducible bit for bit.
#include "fa_kernels.h"
#include "fa_ptx.cuh"
#include "fa_seq.cuh"

namespace fa {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float amax8(const uint4& v) {
    float m = fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x)));
    m = fmax3(m, fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)));
    m = fmax3(m, fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z)));
    return fmax3(m, fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w)));
}

// eight bf16 values / scale -> eight e4m3 codes (value order = byte order)
__device__ __forceinline__ uint2 quant8(const uint4& v, float scale) {
    uint2 r;
    r.x = pack4_e4m3(__fdiv_rn(bf16_lo(v.x), scale), __fdiv_rn(bf16_hi(v.x), scale),
                     __fdiv_rn(bf16_lo(v.y), scale), __fdiv_rn(bf16_hi(v.y), scale));
    r.y = pack4_e4m3(__fdiv_rn(bf16_lo(v.z), scale), __fdiv_rn(bf16_hi(v.z), scale),
                     __fdiv_rn(bf16_lo(v.w), scale), __fdiv_rn(bf16_hi(v.w), scale));
    return r;
}

// max over the CTA (blockDim.x threads, a multiple of 32); every thread gets it
__device__ __forceinline__ float cta_max(float m, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int warp = threadIdx.x / 32, nw = blockDim.x / 32;
    if ((threadIdx.x & 31) == 0) red[warp] = m;
    __syncthreads();
    float r = red[0];
    for (int w = 1; w < nw; ++w) r = fmaxf(r, red[w]);
    __syncthreads();
    return r;
}

__device__ __forceinline__ float block_scale(float amax) {
    return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
}

constexpr int kQuantThreads = 256;

// The 128 x D block of (sequence b, head h, 128-token block blk) as 16-byte units:
// thread t takes units u = t % (D / 8) of rows t / (D / 8) + k * (256 / (D / 8)),
// so a warp reads whole rows (coalesced).  Returns the block's largest magnitude
// over the CTA; `v` holds this thread's units (zero past the sequence end).
template <int D>
__device__ __forceinline__ float load_block(const uint16_t* x, int heads, int start, int len, int h,
                                            int blk, uint4 (&v)[kBlockM * D / 8 / kQuantThreads],
                                            float* red) {
    constexpr int kU = D / 8, kRows = kQuantThreads / kU, kN = kBlockM / kRows;
    const int u = threadIdx.x % kU, r0 = threadIdx.x / kU;
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < kN; ++k) {
        const int row = blk * kBlockM + r0 + k * kRows;
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        if (row < len) {
            v[k] = *reinterpret_cast<const uint4*>(
                x + (static_cast<long long>(start + row) * heads + h) * D + 8 * u);
            m = fmaxf(m, amax8(v[k]));
        }
    }
    return cta_max(m, red);
}

// Q or K: one CTA per (sequence, 128-token block, head).
template <int D>
__global__ void __launch_bounds__(kQuantThreads) fp8_quant_qk_kernel(const __grid_constant__ Fp8QuantParams p) {
    __shared__ float red[kQuantThreads / 32];
    int b, h, blk;
    if (!map_work(p.seq, blockIdx.x, kBlockM, p.heads, false, b, h, blk)) return;
    int start, len;
    seq_bounds(p.seq, b, start, len);
    constexpr int kU = D / 8, kRows = kQuantThreads / kU, kN = kBlockM / kRows;
    uint4 v[kN];
    const float scale = block_scale(load_block<D>(static_cast<const uint16_t*>(p.x), p.heads, start,
                                                  len, h, blk, v, red));
    const long long sidx = static_cast<long long>(h) * p.nb + seq_block_col(p.seq, b) + blk;
    if (threadIdx.x == 0 && fa_index_ok(sidx, static_cast<long long>(p.heads) * p.nb, p.status))
        p.scales[sidx] = scale;
    const int u = threadIdx.x % kU, r0 = threadIdx.x / kU;
    uint8_t* out = static_cast<uint8_t*>(p.out);
#pragma unroll
    for (int k = 0; k < kN; ++k) {
        const int row = blk * kBlockM + r0 + k * kRows;
        if (row < len && fa_index_ok(static_cast<long long>(start + row) * p.heads + h,
                                     static_cast<long long>(p.seq.total_tokens) * p.heads, p.status))
            *reinterpret_cast<uint2*>(out + (static_cast<long long>(start + row) * p.heads + h) * D +
                                      8 * u) = quant8(v[k], scale);
    }
}

// Q or K with incoherent processing: one CTA per (sequence, 128-token block, head).
// Thread t takes the four 16-byte units u = q + kQ j (j = 0..3, q = t % kQ,
// kQ = D / 32) of rows t / kQ + k (256 / kQ): channel c = 8 u + e is element e of
// unit u.  Butterflies with h < 8 pair elements of one unit; h = 8 m pairs units u
// and u ^ m, which for m < kQ sit in lanes q and q ^ m of the row's lane group and
// otherwise in the thread's own units j and j ^ (m / kQ).  Either way the stages run
// in the order h = 1, 2, ..., D/2, as the definition fixes.
template <int D>
__global__ void __launch_bounds__(kQuantThreads) fp8_quant_qk_rot_kernel(const __grid_constant__ Fp8QuantParams p) {
    constexpr int kQ = D / 32, kRows = kQuantThreads / kQ, kN = kBlockM / kRows;
    constexpr float kInvSqrtD = D == 64 ? 0x1p-3f : 0x1.6a09e6p-4f;   // float32(1 / sqrt D)
    static_assert(D == 64 || D == 128, "d in {64, 128}");
    __shared__ float red[kQuantThreads / 32];
    int b, h, blk;
    if (!map_work(p.seq, blockIdx.x, kBlockM, p.heads, false, b, h, blk)) return;
    int start, len;
    seq_bounds(p.seq, b, start, len);
    const int q = threadIdx.x % kQ, r0 = threadIdx.x / kQ;
    const Philox4 w = philox4x32_10(0u, 0xFFFFFFFFu, 0xFFFFFFFFu, 0u, p.seed_lo, p.seed_hi);
    const uint16_t* x = static_cast<const uint16_t*>(p.x);
    float f[kN][4][8];
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < kN; ++k) {
        const int row = blk * kBlockM + r0 + k * kRows;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int u = q + kQ * j;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);   // rows past the sequence: zeros, no codes
            if (row < len)
                v = *reinterpret_cast<const uint4*>(x + (static_cast<long long>(start + row) * p.heads + h) * D +
                                                    8 * u);
            // sign bits of channels 8u .. 8u + 7: byte u % 4 of word u / 4 (= kQ j / 4, as q < kQ)
            const int wi = (kQ * j) >> 2;
            const uint32_t word = wi == 0 ? w.x : wi == 1 ? w.y : wi == 2 ? w.z : w.w;
            const uint32_t sb = word >> (8 * (u & 3));
            const uint32_t raw[8] = {v.x << 16, v.x & 0xFFFF0000u, v.y << 16, v.y & 0xFFFF0000u,
                                     v.z << 16, v.z & 0xFFFF0000u, v.w << 16, v.w & 0xFFFF0000u};
#pragma unroll
            for (int e = 0; e < 8; ++e) f[k][j][e] = __uint_as_float(raw[e] ^ (((sb >> e) & 1u) << 31));
#pragma unroll
            for (int s = 1; s < 8; s <<= 1)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if ((e & s) == 0) {
                        const float a = f[k][j][e], c = f[k][j][e + s];
                        f[k][j][e] = __fadd_rn(a, c);
                        f[k][j][e + s] = __fsub_rn(a, c);
                    }
        }
#pragma unroll
        for (int mu = 1; mu < D / 8; mu <<= 1) {
            if (mu < kQ) {
                const bool upper = (q & mu) != 0;
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float o = __shfl_xor_sync(0xffffffffu, f[k][j][e], mu);
                        f[k][j][e] = upper ? __fsub_rn(o, f[k][j][e]) : __fadd_rn(f[k][j][e], o);
                    }
            } else {
                const int dj = mu / kQ;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if ((j & dj) == 0)
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float a = f[k][j][e], c = f[k][j + dj][e];
                            f[k][j][e] = __fadd_rn(a, c);
                            f[k][j + dj][e] = __fsub_rn(a, c);
                        }
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                f[k][j][e] = __fmul_rn(f[k][j][e], kInvSqrtD);
                m = fmaxf(m, fabsf(f[k][j][e]));
            }
    }
    const float scale = block_scale(cta_max(m, red));
    const long long sidx = static_cast<long long>(h) * p.nb + seq_block_col(p.seq, b) + blk;
    if (threadIdx.x == 0 && fa_index_ok(sidx, static_cast<long long>(p.heads) * p.nb, p.status))
        p.scales[sidx] = scale;
    uint8_t* out = static_cast<uint8_t*>(p.out);
#pragma unroll
    for (int k = 0; k < kN; ++k) {
        const int row = blk * kBlockM + r0 + k * kRows;
        if (row >= len || !fa_index_ok(static_cast<long long>(start + row) * p.heads + h,
                                       static_cast<long long>(p.seq.total_tokens) * p.heads, p.status))
            continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float* g = f[k][j];
            uint2 c;
            c.x = pack4_e4m3(__fdiv_rn(g[0], scale), __fdiv_rn(g[1], scale), __fdiv_rn(g[2], scale),
                             __fdiv_rn(g[3], scale));
            c.y = pack4_e4m3(__fdiv_rn(g[4], scale), __fdiv_rn(g[5], scale), __fdiv_rn(g[6], scale),
                             __fdiv_rn(g[7], scale));
            *reinterpret_cast<uint2*>(out + (static_cast<long long>(start + row) * p.heads + h) * D +
                                      8 * (q + kQ * j)) = c;
        }
    }
}

// V, in three passes over (sequence, 128-token block, head) CTAs and a fourth over
// (sequence, head): the scale slots start at zero, take the atomic max of the
// blocks' largest magnitudes (float bits compare like ints for non-negative
// values), then every block quantises with amax / 448, and last the slots turn
// from amax into the scale.
__global__ void fp8_v_slots_kernel(float* slots, int n, bool to_scale) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) slots[i] = to_scale ? block_scale(slots[i]) : 0.f;
}

template <int D>
__global__ void __launch_bounds__(kQuantThreads) fp8_v_amax_kernel(const __grid_constant__ Fp8QuantParams p) {
    __shared__ float red[kQuantThreads / 32];
    int b, h, blk;
    if (!map_work(p.seq, blockIdx.x, kBlockN, p.heads, false, b, h, blk)) return;
    int start, len;
    seq_bounds(p.seq, b, start, len);
    uint4 v[kBlockM * D / 8 / kQuantThreads];
    const float m = load_block<D>(static_cast<const uint16_t*>(p.x), p.heads, start, len, h, blk, v, red);
    if (threadIdx.x == 0 && fa_index_ok(static_cast<long long>(h) * p.seq.B + b,
                                        static_cast<long long>(p.heads) * p.seq.B, p.status))
        atomicMax(reinterpret_cast<int*>(p.scales + static_cast<long long>(h) * p.seq.B + b),
                  __float_as_int(m));
}

// Quantise one block of V and write it transposed: thread i takes channels
// 8 (i % (D / 8)) .. + 7 of the block's tokens (i / (D / 8)) * kT .. + kT - 1 (one
// 16-byte load per token, a warp reading whole rows), and after the quantisation
// regroups the bytes per channel in registers (byte permutes) into kT keys of one
// V^T row, stored as one piece.
template <int D>
__global__ void __launch_bounds__(128) fp8_v_quant_kernel(const __grid_constant__ Fp8QuantParams p) {
    constexpr int kU = D / 8;              // channel groups
    constexpr int kT = kBlockN * kU / 128; // tokens per thread: 16 (d = 128) or 8 (d = 64)
    static_assert(kT % 4 == 0, "whole words of keys");
    int b, h, blk;
    if (!map_work(p.seq, blockIdx.x, kBlockN, p.heads, false, b, h, blk)) return;
    int start, len;
    seq_bounds(p.seq, b, start, len);
    const float scale = block_scale(p.scales[static_cast<long long>(h) * p.seq.B + b]);
    const int u = threadIdx.x % kU, t0 = (threadIdx.x / kU) * kT;
    const uint16_t* x = static_cast<const uint16_t*>(p.x);
    uint2 c[kT];
#pragma unroll
    for (int t = 0; t < kT; ++t) {
        const int tok = blk * kBlockN + t0 + t;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);   // padding keys: zero values, zero codes
        if (tok < len)
            v = *reinterpret_cast<const uint4*>(x + (static_cast<long long>(start + tok) * p.heads + h) * D +
                                                8 * u);
        c[t] = quant8(v, scale);
    }
    uint8_t* out = static_cast<uint8_t*>(p.out);
    const long long col = 128LL * seq_block_col(p.seq, b) + static_cast<long long>(blk) * kBlockN + t0;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint32_t sel = (ch & 3) | (((ch & 3) + 4) << 4);   // byte ch of two words
        uint32_t w[kT / 4];
#pragma unroll
        for (int q = 0; q < kT / 4; ++q) {
            const uint32_t a0 = ch < 4 ? c[4 * q].x : c[4 * q].y, a1 = ch < 4 ? c[4 * q + 1].x : c[4 * q + 1].y;
            const uint32_t a2 = ch < 4 ? c[4 * q + 2].x : c[4 * q + 2].y, a3 = ch < 4 ? c[4 * q + 3].x : c[4 * q + 3].y;
            w[q] = __byte_perm(__byte_perm(a0, a1, sel), __byte_perm(a2, a3, sel), 0x5410);
        }
        const long long di = (static_cast<long long>(h) * D + 8 * u + ch) * p.vt_tokens + col;
        if (!fa_index_ok(di + kT - 1, static_cast<long long>(p.heads) * D * p.vt_tokens, p.status)) continue;
        uint8_t* dst = out + di;
        if constexpr (kT == 16)
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1 % (kT / 4)], w[2 % (kT / 4)], w[3 % (kT / 4)]);
        else
            *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1 % (kT / 4)]);
    }
}

}  // namespace

cudaError_t launch_fp8_quant_qk(const Fp8QuantParams& p, int d, int grid, cudaStream_t stream) {
    if (grid <= 0) return cudaSuccess;
    if (p.rotate) {
        if (d == 128) fp8_quant_qk_rot_kernel<128><<<grid, kQuantThreads, 0, stream>>>(p);
        else fp8_quant_qk_rot_kernel<64><<<grid, kQuantThreads, 0, stream>>>(p);
    } else if (d == 128) fp8_quant_qk_kernel<128><<<grid, kQuantThreads, 0, stream>>>(p);
    else fp8_quant_qk_kernel<64><<<grid, kQuantThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fp8_quant_v(const Fp8QuantParams& p, int d, int grid, cudaStream_t stream) {
    const int n = p.seq.B * p.heads;
    if (grid <= 0 || n <= 0) return cudaSuccess;
    fp8_v_slots_kernel<<<(n + 255) / 256, 256, 0, stream>>>(p.scales, n, false);
    if (d == 128) {
        fp8_v_amax_kernel<128><<<grid, kQuantThreads, 0, stream>>>(p);
        fp8_v_quant_kernel<128><<<grid, 128, 0, stream>>>(p);
    } else {
        fp8_v_amax_kernel<64><<<grid, kQuantThreads, 0, stream>>>(p);
        fp8_v_quant_kernel<64><<<grid, 128, 0, stream>>>(p);
    }
    fp8_v_slots_kernel<<<(n + 255) / 256, 256, 0, stream>>>(p.scales, n, true);
    return cudaGetLastError();
}

}  // namespace fa
