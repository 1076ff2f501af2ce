// fa_bwd.cu -- backward pass of exact attention on sm_103a, by recomputation.
//
// "FlashAttention: How IO-Aware Tiling and Online Softmax Solved Transformer
// Memory Bottlenecks", section "3. Recomputation in the Backward Pass": the
// forward pass keeps only O and per-row statistics (here the logsumexp, as in
// "Flash Attention -- Fast Memory-Efficient Exact Attention", "Architecture
// Overview"); the backward pass reloads Q, K, V tiles, rebuilds each score
// tile S_ij on chip and forms the gradients from it.  The gradient formulas
// are the calculus of softmax (the pages give none):
//   P_ij = exp(S_ij - LSE_i)         D_i = dO_i . O_i
//   dP_ij = dO_i . v_j               dS_ij = P_ij (dP_ij - D_i)
//   dV_j = sum_i P_ij dO_i           dK_j = scale sum_i dS_ij q_i
//   dQ_i = scale sum_j dS_ij k_j
//
// Three kernels, all deterministic (no atomics, no cross-CTA accumulation):
//   fa_bwd_preprocess  D_i for every query row and head (HBM-bound)
//   fa_bwd_dkdv        one CTA per (sequence, key/value head, 128-key tile);
//                      loops over the query heads of the group and the query
//                      tiles that see the key tile; S^T and dP^T are built in
//                      TMEM with keys on the TMEM lanes, P^T and dS^T go back
//                      to TMEM as bf16 and feed dV += P^T dO and dK += dS^T Q
//   fa_bwd_dq          one CTA per (sequence, query head, 128-row tile); loops
//                      over the key tiles; S and dP in TMEM, dS (bf16) back to
//                      TMEM feeds dQ += dS K
// Warp roles in both tensor-core kernels: warp 0 TMA producer, warp 1 tcgen05
// issuer (one thread, owns TMEM), warps 4..7 element-wise work + epilogue
// (TMEM lane = row).
#include "fa_kernels.h"
#include "fa_ptx.cuh"
#include "fa_seq.cuh"

#include <cuda_bf16.h>

namespace fa {
namespace {

constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kPosInf = __builtin_huge_valf();

// ------------------------------------------------------------- preprocess

// D_i = sum_c dO_ic O_ic in fp32 for every (token, query head).  A group of
// D/8 lanes handles one row, 8 bf16 (16 bytes) per lane.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_kernel(const __grid_constant__ BwdParams p) {
    constexpr int kLanesPerRow = D / 8;
    const SeqInfo& s = p.seq;
    const long long rows = static_cast<long long>(s.total_tokens) * s.Hq;
    const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / kLanesPerRow;
    const int sub = threadIdx.x % kLanesPerRow;
    float acc = 0.f;
    if (row < rows) {
        const uint4 o4 = reinterpret_cast<const uint4*>(p.o)[row * kLanesPerRow + sub];
        const uint4 d4 = reinterpret_cast<const uint4*>(p.dout)[row * kLanesPerRow + sub];
        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o4);
        const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&d4);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = __bfloat1622float2(o2[i]);
            const float2 c = __bfloat1622float2(d2[i]);
            acc = fmaf(a.x, c.x, acc);
            acc = fmaf(a.y, c.y, acc);
        }
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off, kLanesPerRow);
    if (row < rows && sub == 0) {
        const int token = static_cast<int>(row / s.Hq), h = static_cast<int>(row % s.Hq);
        long long idx;
        if (s.cu_seqlens) idx = static_cast<long long>(h) * s.total_tokens + token;
        else idx = (static_cast<long long>(token / s.N) * s.Hq + h) * s.N + token % s.N;
        p.delta[idx] = acc;
    }
}

// ------------------------------------------------------------ shared bits

template <int D>
struct BwdCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kChunkBytes = kBlockM * 128;
    static constexpr int kTileBytes = kBlockM * D * 2;
    static constexpr int kStages = 2;
    static constexpr int kThreads = 256;
    static constexpr int kTmemCols = 512;
    static constexpr int kColS = 0;          // S (or S^T), 128 fp32 columns
    static constexpr int kColDP = 128;       // dP (or dP^T), 128 fp32 columns
    static constexpr int kColAcc = 256;      // accumulators: dQ, or dV then dK (D each)
    // resident pair (Q,dO or K,V) + kStages streamed pairs + row statistics
    static constexpr int kTilesBytes = (2 + 2 * kStages) * kTileBytes;
    static constexpr int kStatBytes = kStages * 2 * kBlockM * 4;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmemBytes = kTilesBytes + kStatBytes + kBarBytes + 1024;
    static constexpr uint32_t kIdescSS = idesc_bf16_f32(kBlockM, kBlockN, false, false);
    static constexpr uint32_t kIdescTS = idesc_bf16_f32(kBlockM, D, false, true);
};

struct BwdBars {
    uint64_t res_full;      // resident pair landed
    uint64_t s_full;        // S and dP tiles computed
    uint64_t ds_full;       // element-wise results written back to TMEM
    uint64_t acc_full;      // all accumulation done
    uint64_t st_full[2];    // streamed pair landed
    uint64_t st_empty[2];   // streamed pair consumed
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
}

// a[rows: K-major 128 x D] . b[rows: K-major 128 x D]^T -> tmem (128 x 128 fp32)
template <int D>
__device__ __forceinline__ void issue_ss(uint32_t d_tmem, uint32_t a, uint32_t b) {
    using C = BwdCfg<D>;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * C::kChunkBytes + (kk % 4) * 32;
        mma_ss(d_tmem, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + off, 16, 1024), C::kIdescSS,
               kk > 0);
    }
}

// tmem bf16 A (128 x 128, packed at a_tmem) . b[smem rows: 128 x D, MN-major] -> d_tmem (128 x D)
template <int D>
__device__ __forceinline__ void issue_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b, bool acc) {
    using C = BwdCfg<D>;
#pragma unroll
    for (int kk = 0; kk < kBlockN / 16; ++kk)
        mma_ts(d_tmem, a_tmem + kk * 8, sdesc_sw128(b + kk * 2048, C::kChunkBytes, 1024),
               C::kIdescTS, (acc || kk > 0) ? 1u : 0u);
}

// TMEM accumulator row (D fp32 columns) * mul -> bf16 row in global memory.
template <int D>
__device__ __forceinline__ void store_acc_row(uint32_t t_acc, float mul, __nv_bfloat16* dst,
                                              bool valid) {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(t_acc + c * 32, r);
        tmem_ld_wait();
        reg_fence(r);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
        if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
    }
}

template <int D>
__device__ __forceinline__ void init_bwd_cta(BwdBars* bars, int warp) {
    if (threadIdx.x == 0) {
        bars->abort = 0;
        mbar_init(smem_addr(&bars->res_full), 1);
        mbar_init(smem_addr(&bars->s_full), 1);
        mbar_init(smem_addr(&bars->ds_full), kBlockM);
        mbar_init(smem_addr(&bars->acc_full), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&bars->st_full[i]), 1);
            mbar_init(smem_addr(&bars->st_empty[i]), 1);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&bars->tmem_base), BwdCfg<D>::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

template <int D>
__device__ __forceinline__ void teardown_bwd_cta(BwdBars* bars, int warp, long long limit) {
    if (bars->abort && threadIdx.x == 32)
        mbar_wait_drain(smem_addr(&bars->acc_full), 0, limit);  // no tcgen05 op left in flight
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(bars->tmem_base, BwdCfg<D>::kTmemCols);
    }
}

// ------------------------------------------------------------------ dK, dV

template <int D>
__global__ void __launch_bounds__(256, 1) fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdCfg<D>;
    const SeqInfo& s = p.seq;
    int b, g, kblk;
    if (!map_work(s, blockIdx.x, kBlockN, s.Hkv, false, b, g, kblk)) return;
    int seq_start, len;
    seq_bounds(s, b, seq_start, len);
    const int kb = kblk * kBlockN;
    const int k_last = min(kb + kBlockN - 1, len - 1);
    const int qt_first = query_lo(s, kb) / kBlockM;
    const int qt_last = query_hi(s, k_last, len) / kBlockM;
    const int nq = qt_last - qt_first + 1;
    const int nsteps = s.group * nq;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* sK = smem;
    uint8_t* sV = smem + C::kTileBytes;
    uint8_t* sQ = smem + 2 * C::kTileBytes;                       // [stage][tile]
    uint8_t* sDO = sQ + C::kStages * C::kTileBytes;                // [stage][tile]
    float* sStat = reinterpret_cast<float*>(smem + C::kTilesBytes);  // [stage][lse2|delta][128]
    BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kTilesBytes + C::kStatBytes);
    volatile int* abort_flag = &bars->abort;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    init_bwd_cta<D>(bars, warp);
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------ producer
        const uint64_t keep = make_l2_policy_evict_last();
        if (lane == 0) {
            const uint32_t rb = smem_addr(&bars->res_full);
            mbar_arrive_expect_tx(rb, 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(smem_addr(sK + c * C::kChunkBytes), &p.tm_k, rb, c * 64, g, seq_start + kb);
                tma_load_3d(smem_addr(sV + c * C::kChunkBytes), &p.tm_v, rb, c * 64, g, seq_start + kb);
            }
        }
        int issued = 0;
        for (int n = 0; n < nsteps; ++n) {
            const int st = n % C::kStages, use = n / C::kStages;
            const int h = g * s.group + n / nq;
            const int q0 = (qt_first + n % nq) * kBlockM;
            // lane 0 waits for the stage, the warp follows its verdict (uniform exit)
            int free_ok = 1;
            if (lane == 0 && use > 0)
                free_ok = mbar_wait(smem_addr(&bars->st_empty[st]), (use - 1) & 1, abort_flag,
                                    p.timeout_cycles, p.status);
            if (!__shfl_sync(0xffffffffu, free_ok, 0)) break;
            // row statistics of the 128 query rows: LSE in log2 units and D;
            // rows past the sequence end get +inf / 0 so they contribute nothing
            float* stat = sStat + st * 2 * kBlockM;
#pragma unroll
            for (int i = 0; i < kBlockM / 32; ++i) {
                const int r = i * 32 + lane, q = q0 + r;
                float l2 = kPosInf, dl = 0.f;
                if (q < len) {
                    const long long idx = row_stat_index(s, b, h, seq_start, q);
                    l2 = __ldg(p.lse + idx) * kLog2eF;
                    dl = p.delta[idx];
                }
                stat[r] = l2;
                stat[kBlockM + r] = dl;
            }
            __syncwarp();
            if (lane == 0) {
                const uint32_t fb = smem_addr(&bars->st_full[st]);
                mbar_arrive_expect_tx(fb, 2 * C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d_hint(smem_addr(sQ + st * C::kTileBytes + c * C::kChunkBytes), &p.tm_q,
                                     fb, c * 64, h, seq_start + q0, keep);
                    tma_load_3d_hint(smem_addr(sDO + st * C::kTileBytes + c * C::kChunkBytes),
                                     &p.tm_do, fb, c * 64, h, seq_start + q0, keep);
                }
            }
            issued = n + 1;
        }
        if (*abort_flag && lane == 0) {
            mbar_wait_drain(smem_addr(&bars->res_full), 0, p.timeout_cycles);
            for (int n = max(0, issued - C::kStages); n < issued; ++n)
                mbar_wait_drain(smem_addr(&bars->st_full[n % C::kStages]), (n / C::kStages) & 1,
                                p.timeout_cycles);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait(smem_addr(&bars->res_full), 0, abort_flag, p.timeout_cycles, p.status);
            const uint32_t aK = smem_addr(sK), aV = smem_addr(sV);
            for (int n = 0; ok && n < nsteps; ++n) {
                const int st = n % C::kStages;
                if (!(ok = mbar_wait(smem_addr(&bars->st_full[st]), (n / C::kStages) & 1, abort_flag,
                                     p.timeout_cycles, p.status)))
                    break;
                tc_fence_after();
                const uint32_t aQ = smem_addr(sQ + st * C::kTileBytes);
                const uint32_t aDO = smem_addr(sDO + st * C::kTileBytes);
                issue_ss<D>(tmem + C::kColS, aK, aQ);     // S^T = K Q^T
                issue_ss<D>(tmem + C::kColDP, aV, aDO);   // dP^T = V dO^T
                mma_commit(smem_addr(&bars->s_full));
                if (!(ok = mbar_wait(smem_addr(&bars->ds_full), n & 1, abort_flag, p.timeout_cycles,
                                     p.status)))
                    break;
                tc_fence_after();
                issue_ts<D>(tmem + C::kColAcc, tmem + C::kColS, aDO, n > 0);       // dV += P^T dO
                issue_ts<D>(tmem + C::kColAcc + D, tmem + C::kColDP, aQ, n > 0);   // dK += dS^T Q
                mma_commit(smem_addr(&bars->st_empty[st]));
            }
            mma_commit(smem_addr(&bars->acc_full));
        }
    } else if (warp >= 4) {
        // ------------------------------------------- element-wise + epilogue
        const int quad = warp % 4;
        const int r = quad * 32 + lane;  // key row within the tile = TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const int kpos = kb + r;
        // queries that see this key: [qlo, qhi]; none if the key is past the end
        const int qlo = query_lo(s, kpos);
        const int qhi = (kpos < len) ? query_hi(s, kpos, len) : -1;
        const float sl2 = p.scale_log2;
        bool ok = true;
        for (int n = 0; n < nsteps; ++n) {
            const int st = n % C::kStages;
            const int q0 = (qt_first + n % nq) * kBlockM;
            const float* lse2 = sStat + st * 2 * kBlockM;
            const float* dlt = lse2 + kBlockM;
            ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bars->s_full), n & 1, abort_flag,
                                                   p.timeout_cycles, p.status));
            if (!ok) break;  // warp-uniform: the TMEM accesses below are warp-collective
            tc_fence_after();
            const bool need_mask = !(q0 >= qlo && q0 + kBlockM - 1 <= qhi);
            const int clo = qlo - q0, chi = qhi - q0;
#pragma unroll
            for (int c = 0; c < kBlockM / 32; ++c) {
                uint32_t sr[32], dr[32];
                tmem_ld32(tmem + lane_addr + C::kColS + c * 32, sr);
                tmem_ld32(tmem + lane_addr + C::kColDP + c * 32, dr);
                tmem_ld_wait();
                reg_fence(sr);
                reg_fence(dr);
                uint32_t pw[16], dw[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float pv[2], dv2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int col = c * 32 + 2 * i + e;
                        float pe = ex2_approx(fmaf(__uint_as_float(sr[2 * i + e]), sl2, -lse2[col]));
                        if (need_mask && (col < clo || col > chi)) pe = 0.f;
                        pv[e] = pe;
                        dv2[e] = pe * (__uint_as_float(dr[2 * i + e]) - dlt[col]);
                    }
                    pw[i] = pack_bf16x2(pv[0], pv[1]);
                    dw[i] = pack_bf16x2(dv2[0], dv2[1]);
                }
                // P^T and dS^T overwrite columns already consumed (16c .. 16c+15 < 32c+32)
                tmem_st16(tmem + lane_addr + C::kColS + c * 16, pw);
                tmem_st16(tmem + lane_addr + C::kColDP + c * 16, dw);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_addr(&bars->ds_full));
        }
        if (ok)
            ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bars->acc_full), 0, abort_flag,
                                                   p.timeout_cycles, p.status));
        if (ok) {
            tc_fence_after();
            const bool valid = kpos < len;
            const long long row = (static_cast<long long>(seq_start + kpos) * s.Hkv + g) * D;
            store_acc_row<D>(tmem + lane_addr + C::kColAcc, 1.f,
                             reinterpret_cast<__nv_bfloat16*>(p.dv) + row, valid);
            store_acc_row<D>(tmem + lane_addr + C::kColAcc + D, p.scale,
                             reinterpret_cast<__nv_bfloat16*>(p.dk) + row, valid);
        }
    }
    teardown_bwd_cta<D>(bars, warp, p.timeout_cycles);
}

// ---------------------------------------------------------------------- dQ

template <int D>
__global__ void __launch_bounds__(256, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdCfg<D>;
    const SeqInfo& s = p.seq;
    int b, h, qblk;
    if (!map_work(s, blockIdx.x, kBlockM, s.Hq, true, b, h, qblk)) return;
    int seq_start, len;
    seq_bounds(s, b, seq_start, len);
    const int g = h / s.group;
    const int q0 = qblk * kBlockM;
    const int q_last = min(q0 + kBlockM - 1, len - 1);
    const int kt_first = max(key_lo(s, q0), 0) / kBlockN;
    const int kt_last = key_hi(s, q_last, len) / kBlockN;
    const int nk = kt_last - kt_first + 1;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* sQ = smem;
    uint8_t* sDO = smem + C::kTileBytes;
    uint8_t* sK = smem + 2 * C::kTileBytes;          // [stage][tile]
    uint8_t* sV = sK + C::kStages * C::kTileBytes;   // [stage][tile]
    BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kTilesBytes + C::kStatBytes);
    volatile int* abort_flag = &bars->abort;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    init_bwd_cta<D>(bars, warp);
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t keep = make_l2_policy_evict_last();
            const uint32_t rb = smem_addr(&bars->res_full);
            mbar_arrive_expect_tx(rb, 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(smem_addr(sQ + c * C::kChunkBytes), &p.tm_q, rb, c * 64, h, seq_start + q0);
                tma_load_3d(smem_addr(sDO + c * C::kChunkBytes), &p.tm_do, rb, c * 64, h, seq_start + q0);
            }
            int issued = 0;
            for (int j = 0; j < nk; ++j) {
                const int st = j % C::kStages, use = j / C::kStages;
                if (use > 0 && !mbar_wait(smem_addr(&bars->st_empty[st]), (use - 1) & 1, abort_flag,
                                          p.timeout_cycles, p.status))
                    break;
                const uint32_t fb = smem_addr(&bars->st_full[st]);
                mbar_arrive_expect_tx(fb, 2 * C::kTileBytes);
                const int row = seq_start + (kt_first + j) * kBlockN;
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d_hint(smem_addr(sK + st * C::kTileBytes + c * C::kChunkBytes), &p.tm_k,
                                     fb, c * 64, g, row, keep);
                    tma_load_3d_hint(smem_addr(sV + st * C::kTileBytes + c * C::kChunkBytes), &p.tm_v,
                                     fb, c * 64, g, row, keep);
                }
                issued = j + 1;
            }
            if (*abort_flag) {
                mbar_wait_drain(rb, 0, p.timeout_cycles);
                for (int j = max(0, issued - C::kStages); j < issued; ++j)
                    mbar_wait_drain(smem_addr(&bars->st_full[j % C::kStages]), (j / C::kStages) & 1,
                                    p.timeout_cycles);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = mbar_wait(smem_addr(&bars->res_full), 0, abort_flag, p.timeout_cycles, p.status);
            const uint32_t aQ = smem_addr(sQ), aDO = smem_addr(sDO);
            for (int j = 0; ok && j < nk; ++j) {
                const int st = j % C::kStages;
                if (!(ok = mbar_wait(smem_addr(&bars->st_full[st]), (j / C::kStages) & 1, abort_flag,
                                     p.timeout_cycles, p.status)))
                    break;
                tc_fence_after();
                const uint32_t aK = smem_addr(sK + st * C::kTileBytes);
                const uint32_t aV = smem_addr(sV + st * C::kTileBytes);
                issue_ss<D>(tmem + C::kColS, aQ, aK);     // S = Q K^T
                issue_ss<D>(tmem + C::kColDP, aDO, aV);   // dP = dO V^T
                mma_commit(smem_addr(&bars->s_full));
                if (!(ok = mbar_wait(smem_addr(&bars->ds_full), j & 1, abort_flag, p.timeout_cycles,
                                     p.status)))
                    break;
                tc_fence_after();
                issue_ts<D>(tmem + C::kColAcc, tmem + C::kColS, aK, j > 0);   // dQ += dS K
                mma_commit(smem_addr(&bars->st_empty[st]));
            }
            mma_commit(smem_addr(&bars->acc_full));
        }
    } else if (warp >= 4) {
        const int quad = warp % 4;
        const int r = quad * 32 + lane;  // query row within the tile = TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const int q = q0 + r;
        const bool valid = q < len;
        float lse2 = kPosInf, dlt = 0.f;
        if (valid) {
            const long long idx = row_stat_index(s, b, h, seq_start, q);
            lse2 = __ldg(p.lse + idx) * kLog2eF;
            dlt = p.delta[idx];
        }
        const int lo_q = key_lo(s, q), hi_q = valid ? key_hi(s, q, len) : -1;
        const int full_lo = key_lo(s, q0 + kBlockM - 1);
        const int full_hi = key_hi(s, q0, len);
        const float sl2 = p.scale_log2;
        bool ok = true;
        for (int j = 0; j < nk; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bars->s_full), j & 1, abort_flag,
                                                   p.timeout_cycles, p.status));
            if (!ok) break;  // warp-uniform: the TMEM accesses below are warp-collective
            tc_fence_after();
            const int kb = (kt_first + j) * kBlockN;
            const bool need_mask = !(kb >= full_lo && kb + kBlockN - 1 <= full_hi) || !valid;
            const int clo = lo_q - kb, chi = hi_q - kb;
#pragma unroll
            for (int c = 0; c < kBlockN / 32; ++c) {
                uint32_t sr[32], dr[32];
                tmem_ld32(tmem + lane_addr + C::kColS + c * 32, sr);
                tmem_ld32(tmem + lane_addr + C::kColDP + c * 32, dr);
                tmem_ld_wait();
                reg_fence(sr);
                reg_fence(dr);
                uint32_t dw[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float ds[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int col = c * 32 + 2 * i + e;
                        float pe = ex2_approx(fmaf(__uint_as_float(sr[2 * i + e]), sl2, -lse2));
                        if (need_mask && (col < clo || col > chi)) pe = 0.f;
                        ds[e] = pe * (__uint_as_float(dr[2 * i + e]) - dlt);
                    }
                    dw[i] = pack_bf16x2(ds[0], ds[1]);
                }
                tmem_st16(tmem + lane_addr + C::kColS + c * 16, dw);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_addr(&bars->ds_full));
        }
        if (ok)
            ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bars->acc_full), 0, abort_flag,
                                                   p.timeout_cycles, p.status));
        if (ok) {
            tc_fence_after();
            const long long row = (static_cast<long long>(seq_start + q) * s.Hq + h) * D;
            store_acc_row<D>(tmem + lane_addr + C::kColAcc, p.scale,
                             reinterpret_cast<__nv_bfloat16*>(p.dq) + row, valid);
        }
    }
    teardown_bwd_cta<D>(bars, warp, p.timeout_cycles);
}

template <typename K>
cudaError_t launch_tc(K kern, int grid, int smem, const BwdParams& p, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 256, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdParams& p, int d, cudaStream_t stream) {
    const long long rows = static_cast<long long>(p.seq.total_tokens) * p.seq.Hq;
    const int lanes = d / 8;
    const long long threads = rows * lanes;
    const int grid = static_cast<int>((threads + 255) / 256);
    if (grid <= 0) return cudaSuccess;
    if (d == 128) fa_bwd_preprocess_kernel<128><<<grid, 256, 0, stream>>>(p);
    else fa_bwd_preprocess_kernel<64><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const BwdParams& p, int d, cudaStream_t stream) {
    if (p.num_work_dkdv <= 0) return cudaSuccess;
    return d == 128 ? launch_tc(fa_bwd_dkdv_kernel<128>, p.num_work_dkdv, BwdCfg<128>::kSmemBytes, p, stream)
                    : launch_tc(fa_bwd_dkdv_kernel<64>, p.num_work_dkdv, BwdCfg<64>::kSmemBytes, p, stream);
}

cudaError_t launch_bwd_dq(const BwdParams& p, int d, cudaStream_t stream) {
    if (p.num_work_dq <= 0) return cudaSuccess;
    return d == 128 ? launch_tc(fa_bwd_dq_kernel<128>, p.num_work_dq, BwdCfg<128>::kSmemBytes, p, stream)
                    : launch_tc(fa_bwd_dq_kernel<64>, p.num_work_dq, BwdCfg<64>::kSmemBytes, p, stream);
}

}  // namespace fa
