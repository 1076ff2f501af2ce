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

// Q or K: thread r of a 128-thread CTA owns token row r of the block.
template <int D>
__global__ void __launch_bounds__(128) fp8_quant_qk_kernel(const __grid_constant__ Fp8QuantParams p) {
    __shared__ float red[4];
    int b, h, blk;
    if (!map_work(p.seq, blockIdx.x, kBlockM, p.heads, false, b, h, blk)) return;
    int start, len;
    seq_bounds(p.seq, b, start, len);
    const int row = blk * kBlockM + threadIdx.x;
    const bool valid = row < len;
    const long long base = (static_cast<long long>(start + row) * p.heads + h) * D;
    uint4 v[D / 8];
    float m = 0.f;
    if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) + base);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            v[i] = src[i];
            m = fmaxf(m, amax8(v[i]));
        }
    }
    const float scale = block_scale(cta_max(m, red));
    if (threadIdx.x == 0)
        p.scales[static_cast<long long>(h) * p.nb + seq_block_col(p.seq, b) + blk] = scale;
    if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + base);
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
            const uint2 lo = quant8(v[2 * i], scale), hi = quant8(v[2 * i + 1], scale);
            dst[i] = make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
    }
}

// V: one CTA of 256 threads per (sequence, head): the sequence's amax, then per
// 128-token block the codes into shared memory [token][d] and out transposed, a
// row of 128 keys (128 bytes) per d.
template <int D>
__global__ void __launch_bounds__(256) fp8_quant_v_kernel(const __grid_constant__ Fp8QuantParams p) {
    __shared__ float red[8];
    __shared__ __align__(16) uint8_t tile[kBlockN][D];
    const int b = blockIdx.x / p.heads, h = blockIdx.x % p.heads;
    if (b >= p.seq.B) return;
    int start, len;
    seq_bounds(p.seq, b, start, len);
    const uint16_t* x = static_cast<const uint16_t*>(p.x);
    constexpr int kU = D / 8;   // 16-byte units per token row
    float m = 0.f;
    for (int i = threadIdx.x; i < len * kU; i += blockDim.x) {
        const int t = i / kU, u = i % kU;
        m = fmaxf(m, amax8(*reinterpret_cast<const uint4*>(
                         x + (static_cast<long long>(start + t) * p.heads + h) * D + 8 * u)));
    }
    const float scale = block_scale(cta_max(m, red));
    if (threadIdx.x == 0) p.scales[static_cast<long long>(h) * p.seq.B + b] = scale;
    uint8_t* out = static_cast<uint8_t*>(p.out);
    const long long col0 = 128LL * seq_block_col(p.seq, b);
    const int nblk = ceil_div(len, kBlockN);
    for (int kb = 0; kb < nblk; ++kb) {
        for (int i = threadIdx.x; i < kBlockN * kU; i += blockDim.x) {
            const int t = i / kU, u = i % kU;
            const int tok = kb * kBlockN + t;
            uint2 c = make_uint2(0u, 0u);   // padding keys: zero codes
            if (tok < len)
                c = quant8(*reinterpret_cast<const uint4*>(
                               x + (static_cast<long long>(start + tok) * p.heads + h) * D + 8 * u),
                           scale);
            *reinterpret_cast<uint2*>(&tile[t][8 * u]) = c;
        }
        __syncthreads();
        // d rows of 128 keys: 8 units of 16 keys each
        for (int i = threadIdx.x; i < D * 8; i += blockDim.x) {
            const int dd = i / 8, k16 = i % 8;
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int t0 = 16 * k16 + 4 * q;
                w[q] = static_cast<uint32_t>(tile[t0][dd]) | (static_cast<uint32_t>(tile[t0 + 1][dd]) << 8) |
                       (static_cast<uint32_t>(tile[t0 + 2][dd]) << 16) |
                       (static_cast<uint32_t>(tile[t0 + 3][dd]) << 24);
            }
            *reinterpret_cast<uint4*>(out + (static_cast<long long>(h) * D + dd) * p.vt_tokens + col0 +
                                      kb * kBlockN + 16 * k16) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_fp8_quant_qk(const Fp8QuantParams& p, int d, int grid, cudaStream_t stream) {
    if (grid <= 0) return cudaSuccess;
    if (d == 128) fp8_quant_qk_kernel<128><<<grid, 128, 0, stream>>>(p);
    else fp8_quant_qk_kernel<64><<<grid, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fp8_quant_v(const Fp8QuantParams& p, int d, cudaStream_t stream) {
    const int grid = p.seq.B * p.heads;
    if (grid <= 0) return cudaSuccess;
    if (d == 128) fp8_quant_v_kernel<128><<<grid, 256, 0, stream>>>(p);
    else fp8_quant_v_kernel<64><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace fa
