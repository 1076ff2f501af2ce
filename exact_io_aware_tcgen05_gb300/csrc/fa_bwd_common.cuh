// fa_bwd_common.cuh -- pieces shared by the backward kernels (fa_bwd.cu: the
// preprocess and the split dK/dV and dQ kernels; fa_bwd_fused.cu: the single
// fused kernel): tile geometry, barrier blocks, tcgen05 issue helpers for the
// products, TMEM row loads and packed stores, the streamed-tile slot ring and
// its producer loop, and the launch helpers.  Internal to the library.
#pragma once

#include "fa_kernels.h"
#include "fa_ptx.cuh"
#include "fa_seq.cuh"

#include <cuda_bf16.h>

#include <type_traits>

namespace fa {
namespace {

constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kPosInf = __builtin_huge_valf();

// ------------------------------------------------------------ shared bits

template <int D>
struct BwdCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kChunkBytes = kBlockM * 128;
    static constexpr int kTileBytes = kBlockM * D * 2;
    // dK/dV kernel: ring of single-tile slots for the streamed Q_n and dO_n
    static constexpr int kSlots = (D == 128) ? 5 : 8;
    // The streamed items alternate between two rings of slots: even items (Q_n,
    // K_j) are held from their first product to their last, about one and a half
    // steps; odd items (dO_n, V_j) about half a step.  Separate rings give each
    // kind a prefetch distance of its own.
    static constexpr int kSlotsOdd = (D == 128) ? 2 : 3;
    // The dQ kernel keeps Q and dO in TMEM (below), so every tile of shared memory
    // belongs to its ring: 7 (d = 128) or 10 (d = 64) slots, of which the odd items
    // (each head's dO, then its V_j) take kSlotsOddDq and the even ones (Q, K_j) the rest.
    static constexpr int kSlotsDq = kSlots + 2;
    static constexpr int kSlotsOddDq = (D == 128) ? 2 : 3;
    // element-wise warpgroups, each owning kEwCols of the 128 tile columns.  Two at
    // both head dimensions: four of 32 columns at d = 64 (640 threads, 96 registers at
    // launch) spilled in the dK/dV kernel and measured slower than two of 64
    static constexpr int kEwWG = 2;
    static constexpr int kEwCols = 128 / kEwWG;
    static constexpr int kEwThreads = 128 * kEwWG;
    static constexpr int kThreads = 128 + kEwThreads;   // warp 0 TMA, warp 1 MMA, warp 2 relay, warps 4.. element-wise
    static constexpr int kBarCount = kEwThreads + 64;   // named barriers: element-wise + issuer + relay warps
    // registers per thread: the launch reserves kRegsLaunch for every thread (one CTA
    // per SM); the warpgroup of warps 0..3 then drops to kRegsCtl and the
    // element-wise warpgroups rise to kRegsEw (setmaxnreg)
    static constexpr int kRegsLaunch = (65536 / kThreads) & ~7;
    static constexpr int kRegsCtl = 152;
    static constexpr int kRegsEw = 176;
    static_assert(128 * kRegsCtl + kEwThreads * kRegsEw <= kThreads * kRegsLaunch,
                  "register split exceeds the launch's registers");
    static constexpr int kTmemCols = 512;
    static constexpr int kColS = 0;          // S (or S^T), 128 fp32 columns
    static constexpr int kColDP = 128;       // dP (or dP^T), 128 fp32 columns
    static constexpr int kColAcc = 256;      // accumulators: dQ, or dV then dK (D each)
    // dQ kernel: Q and dO of the query tile, the A operands of S and dP, packed two
    // elements per 32-bit column (D/2 columns each) after the dQ accumulator
    static constexpr int kColQ = kColAcc + D;
    static constexpr int kColDO = kColQ + D / 2;
    static_assert(kColDO + D / 2 <= kTmemCols, "TMEM columns");
    // [barriers 512 B][row statistics: warpgroups x 2 buffers x 2 kEwCols fp32][pad] then
    // tiles: dK/dV kernel, the resident pair (K, V) followed by its slot ring; dQ
    // kernel, all of them its slot ring
    static constexpr int kBarBytes = 512;
    static constexpr int kStatOffset = kBarBytes;
    static constexpr int kHeadBytes = 3072;
    static constexpr int kTilesBytes = (2 + kSlots) * kTileBytes;
    static constexpr int kSmemBytes = kHeadBytes + kTilesBytes;
};
static_assert(BwdCfg<128>::kSmemBytes <= 232448, "shared memory budget");
static_assert(BwdCfg<64>::kSmemBytes <= 232448, "shared memory budget");

// named barrier ids (0 is __syncthreads): element-wise results (and streamed
// tiles) ready for the issuer's next products
constexpr int kBarP = 1;     // P (P^T) written / S read
constexpr int kBarDS0 = 2;   // dS (dS^T) written
constexpr int kBarOperands = 3;  // dQ kernel: Q and dO copied into TMEM
constexpr int kBarEpi = 4;   // element-wise warps among themselves: the epilogue
constexpr int kBarStat = 5;  // + warpgroup: a dK/dV element-wise warpgroup's row statistics staged

struct BwdBars {
    uint64_t res_full;        // resident pair landed
    uint64_t s_full;          // S (S^T) tile computed
    uint64_t dp_full[2];      // dP (dP^T) tile computed, per dP buffer
    uint64_t acc_full;        // all accumulation done
    uint64_t dq_full;         // fused kernel: a dQ partial tile computed
    uint64_t slot_full[10];   // streamed tile landed in slot
    uint64_t slot_empty[10];  // streamed tile consumed
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(BwdBars) <= BwdCfg<128>::kBarBytes, "barrier block");
static_assert(kBarStat + BwdCfg<64>::kEwWG - 1 <= 15, "named barrier ids");
static_assert(BwdCfg<128>::kStatOffset + 2 * 2 * kBlockM * 4 <= BwdCfg<128>::kHeadBytes, "stats");
static_assert(BwdCfg<64>::kStatOffset + 2 * 2 * kBlockM * 4 <= BwdCfg<64>::kHeadBytes, "stats");

// Fixed-point scale of the fused backward's dQ sums: 2^(15 - e) with 2^e >= x
// (x >= 0), the largest power of two that keeps 2^(15 - e) x <= 2^15, clamped to
// 2^[-60, 60] (x = 0: 2^60; x infinite or NaN: 2^-60).
__device__ __forceinline__ float fixed_point_scale(float x) {
    int e = -45;
    if (!(x <= 3.0e38f)) e = 75;
    else if (x > 0.f) (void)frexpf(x, &e);   // x = m 2^e, m in [0.5, 1)
    const int f = max(-60, min(60, 15 - e));
    return ldexpf(1.f, f);
}

// 2^Fc of channel c of key/value head g: fixed_point_scale of the bound
// 2 r (1 + 2^-5) max_j ||v_j||_2 max_j |k_jc| on the dQ contributions per unit of
// ||dO_i||_2 (|dS_ij| sums to at most 2 ||dO_i|| max_j ||v_j||, times the dropout
// factor r; the margin covers the roundings of P, dS and the products), from
// the preprocess's per-slot maxima.
template <int D>
__device__ __forceinline__ float channel_scale(const float* kv_bound, int g, int c, float r) {
    const float* kb = kv_bound + static_cast<long long>(g) * kBoundSlots * (D + 1);
    float km = 0.f, vm = 0.f;
    for (int sl = 0; sl < kBoundSlots; ++sl) {
        km = fmaxf(km, kb[sl * (D + 1) + c]);
        vm = fmaxf(vm, kb[sl * (D + 1) + D]);
    }
    return fixed_point_scale(2.f * r * 1.03125f * vm * km);
}

// a[rows: K-major 128 x D] . b[rows: K-major 128 x D]^T -> tmem (128 x 128 fp32);
// E: element type of both operands
template <int D, int E>
__device__ __forceinline__ void issue_ss(uint32_t d_tmem, uint32_t a, uint32_t b) {
    using C = BwdCfg<D>;
    constexpr uint32_t kIdescSS = idesc_f32acc(kBlockM, kBlockN, false, false, E);
    // descriptor of the tile base; a k-step adds its byte offset >> 4
    const uint64_t ad = sdesc_sw128(a, 16, 1024), bd = sdesc_sw128(b, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk / 4) * C::kChunkBytes + (kk % 4) * 32) >> 4;
        mma_ss(d_tmem, ad + off, bd + off, kIdescSS, kk > 0);
    }
}

// A = 16-bit operand written back to TMEM by the element-wise warpgroups: the W =
// kEwCols tile columns of warpgroup w sit, packed two per 32-bit column, in the
// first W/2 TMEM columns of that warpgroup's own range (region + W w).
// D (128 x D fp32) (+)= A (128 x 128) . b[smem rows: 128 x D, MN-major].
// W: the warpgroups' column width (the split kernels' BwdCfg<D>::kEwCols unless given).
template <int D, int E, int W = BwdCfg<D>::kEwCols>
__device__ __forceinline__ void issue_ts(uint32_t d_tmem, uint32_t a_region, uint32_t b, bool acc) {
    using C = BwdCfg<D>;
    constexpr uint32_t kIdescTS = idesc_f32acc(kBlockM, D, false, true, E);
    const uint64_t bd = sdesc_sw128(b, C::kChunkBytes, 1024);
#pragma unroll
    for (int kk = 0; kk < kBlockN / 16; ++kk)
        mma_ts(d_tmem, a_region + (16 * kk / W) * W + (16 * kk % W) / 2,
               bd + ((kk * 2048) >> 4),
               kIdescTS, (acc || kk > 0) ? 1u : 0u);
}

// N consecutive 32-bit TMEM columns of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_st_words(uint32_t taddr, const uint32_t (&w)[N]) {
    static_assert(N == 8 || N == 16 || N == 32, "TMEM store width");
    if constexpr (N == 32) tmem_st32(taddr, w);
    else if constexpr (N == 16) tmem_st16(taddr, w);
    else tmem_st8(taddr, w);
}

// A = 16-bit operand held whole in TMEM (128 rows x D, packed two per 32-bit
// column, D/2 contiguous columns) . b[smem rows: K-major 128 x D]^T -> tmem
// (128 x 128 fp32): the dQ kernel's S = Q K^T and dP = dO V^T.
template <int D, int E>
__device__ __forceinline__ void issue_ts_k(uint32_t d_tmem, uint32_t a_tmem, uint32_t b) {
    using C = BwdCfg<D>;
    constexpr uint32_t kIdesc = idesc_f32acc(kBlockM, kBlockN, false, false, E);
    const uint64_t bd = sdesc_sw128(b, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk / 4) * C::kChunkBytes + (kk % 4) * 32) >> 4;
        mma_ts(d_tmem, a_tmem + 8 * kk, bd + off, kIdesc, kk > 0 ? 1u : 0u);
    }
}

// NC fp32 columns of a TMEM accumulator row * mul -> element type E in global memory.
template <int NC, int E>
__device__ __forceinline__ void store_acc_row(uint32_t t_acc, float mul, uint16_t* dst,
                                              bool valid) {
#pragma unroll
    for (int c = 0; c < NC / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(t_acc + c * 32, r);
        tmem_ld_wait();
        reg_fence(r);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i] = pack2<E>(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
        if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
    }
}

// Loads this warpgroup's W (32 or 64) fp32 columns of one TMEM row.
template <int W>
__device__ __forceinline__ void tmem_ldw(uint32_t taddr, float (&v)[W]) {
    uint32_t a[32], b[32];
    tmem_ld32(taddr, a);
    if (W == 64) tmem_ld32(taddr + 32, b);
    tmem_ld_wait();
    reg_fence(a);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(a[i]);
    if (W == 64) {
        reg_fence(b);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[(32 + i) % W] = __uint_as_float(b[i]);
    }
}

// Packs W fp32 values to pairs of element type E and stores them in the first W/2 columns at taddr.
template <int W, int E>
__device__ __forceinline__ void tmem_st_pk(uint32_t taddr, const float (&v)[W]) {
    if (W == 64) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = pack2<E>(v[(2 * i) % W], v[(2 * i + 1) % W]);
        tmem_st32(taddr, w);
    } else {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack2<E>(v[2 * i], v[2 * i + 1]);
        tmem_st16(taddr, w);
    }
}

// v[c] with the dropped columns cleared (m: the row's keep masks, 4 columns a word)
template <int W>
__device__ __forceinline__ float kept(const uint32_t (&m)[W / 4], const float (&v)[W], int c) {
    return __uint_as_float(__float_as_uint(v[c]) & keep_mask32(m[c >> 2], c));
}

// tmem_st_pk of v with the dropped columns cleared (the 1 / keep-probability factor is
// left to the fp32 side: the dV epilogue, the dS arithmetic)
template <int W, int E>
__device__ __forceinline__ void tmem_st_pk_dropped(uint32_t taddr, const float (&v)[W],
                                                   const uint32_t (&m)[W / 4]) {
    uint32_t w[W / 2];
#pragma unroll
    for (int i = 0; i < W / 2; ++i)
        w[i] = pack2<E>(v[2 * i], v[2 * i + 1]) & keep_mask_pair(m[i >> 1], 2 * i);
    if constexpr (W == 64)
        tmem_st32(taddr, w);
    else
        tmem_st16(taddr, w);
}

// Returns false (uniformly for the CTA) if the dynamic shared memory base is not
// 1024-byte aligned, which the 128-byte-swizzled tiles and the exact shared
// memory budget rely on.
__device__ __forceinline__ bool smem_base_ok(const uint8_t* base, int* status) {
    if (smem_addr(base) & 1023u) {
        if (threadIdx.x == 0) atomicExch(status, kDevBadSmem);
        return false;
    }
    return true;
}

template <int D>
__device__ __forceinline__ void init_bwd_cta(BwdBars* bars, int warp, int slots) {
    if (threadIdx.x == 0) {
        bars->abort = 0;
        mbar_init(smem_addr(&bars->res_full), 1);
        mbar_init(smem_addr(&bars->s_full), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&bars->dp_full[i]), 1);
        }
        mbar_init(smem_addr(&bars->acc_full), 1);
        mbar_init(smem_addr(&bars->dq_full), 1);
        for (int i = 0; i < slots; ++i) {
            mbar_init(smem_addr(&bars->slot_full[i]), 1);
            mbar_init(smem_addr(&bars->slot_empty[i]), 1);
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
__device__ __forceinline__ void teardown_bwd_cta(BwdBars* bars, int warp) {
    if (bars->abort && threadIdx.x == 32)
        mbar_wait_drain(smem_addr(&bars->acc_full), 0, kDrainCycles);  // no tcgen05 op left in flight
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(bars->tmem_base, BwdCfg<D>::kTmemCols);
    }
}

// Slot ring of SLOTS tiles for a stream of items that alternate between two
// kinds: the odd items take ODD slots, the even ones the rest.  index(i) is item
// i's slot, use(i) how many items used that slot before it.  Each kind gets at
// least two slots: with one, a wait for item i + 2 on the slot's mbarrier could
// complete on the phase of item i if that item had not landed yet.
template <int SLOTS, int ODD>
struct Ring {
    static constexpr int kSlots = SLOTS;
    static constexpr int kEven = SLOTS - ODD;
    static_assert(ODD >= 2 && kEven >= 2, "two slots per kind of item");
    __device__ static __forceinline__ int index(int i) {
        const int k = i >> 1;
        return (i & 1) ? kEven + k % ODD : k % kEven;
    }
    __device__ static __forceinline__ int use(int i) {
        const int k = i >> 1;
        return (i & 1) ? k / ODD : k / kEven;
    }
};

// Warp-uniform bounded wait (the TMEM accesses that follow are warp-collective).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          long long limit, int* status) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, limit, status));
}

// Producer loop shared by the kernels: streams `items` tiles through the slot
// ring R (item i from map (i & 1) ? odd : even); `coords(i, head, row)` gives the
// head and token row of item i and may return another tensor map for it (void or
// nullptr: the one its parity names).  `resident`: the CTA also loaded a resident
// pair on res_full, which an abort has to wait for too.
template <int D, typename R, typename Coords>
__device__ __forceinline__ void stream_tiles(BwdBars* bars, uint8_t* slots, int items,
                                             const CUtensorMap* even, const CUtensorMap* odd,
                                             Coords coords, volatile int* abort_flag,
                                             const BwdParams& p, bool resident) {
    using C = BwdCfg<D>;
    const uint64_t keep = make_l2_policy_evict_last();
    int issued = 0;
    for (int i = 0; i < items; ++i) {
        const int sl = R::index(i), use = R::use(i);
        if (use > 0 && !mbar_wait(smem_addr(&bars->slot_empty[sl]), (use - 1) & 1, abort_flag,
                                  p.timeout_cycles, p.status))
            break;
        const uint32_t fb = smem_addr(&bars->slot_full[sl]);
        mbar_arrive_expect_tx(fb, C::kTileBytes);
        int head, row;
        const CUtensorMap* map = (i & 1) ? odd : even;
        if constexpr (std::is_void_v<decltype(coords(i, head, row))>) {
            coords(i, head, row);
        } else {
            const CUtensorMap* m = coords(i, head, row);
            if (m) map = m;
        }
        for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d_hint(smem_addr(slots + sl * C::kTileBytes + c * C::kChunkBytes), map, fb,
                             c * 64, head, row, keep);
        issued = i + 1;
    }
    if (*abort_flag) {
        if (resident) mbar_wait_drain(smem_addr(&bars->res_full), 0, kDrainCycles);
        // the last item issued into each slot
        unsigned seen = 0;
        for (int i = issued - 1; i >= 0 && i >= issued - 2 * R::kSlots; --i) {
            const int sl = R::index(i);
            if (seen & (1u << sl)) continue;
            seen |= 1u << sl;
            mbar_wait_drain(smem_addr(&bars->slot_full[sl]), R::use(i) & 1, kDrainCycles);
        }
    }
}

// The register split inside the tensor-core kernels needs the launch's full
// per-thread count: a build that gave a kernel fewer would make its element-wise
// warps wait forever, so such a kernel is refused.
template <typename K>
cudaError_t check_regs(K kern, int need) {
    cudaFuncAttributes fa;
    const cudaError_t r = cudaFuncGetAttributes(&fa, kern);
    if (r != cudaSuccess) return r;
    return fa.numRegs >= need ? cudaSuccess : cudaErrorInvalidKernelImage;
}

template <typename K>
cudaError_t launch_tc(K kern, int grid, int threads, int smem, const BwdParams& p, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, threads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace
}  // namespace fa
