// fa_bwd_fused.cu -- the backward pass of exact attention with ONE tensor-core
// kernel on sm_103a: dQ, dK and dV from a single rebuild of each score tile.
//
// "FlashAttention: How IO-Aware Tiling and Online Softmax Solved Transformer
// Memory Bottlenecks", "3. Recomputation in the Backward Pass": each score tile is
// rebuilt once from Q, K and the saved logsumexp, and every gradient comes from
// that one rebuild.  The split backward (fa_bwd.cu) rebuilds S and dP a second
// time in a query-major dQ kernel; here the key-major CTA of the dK/dV pass also
// forms each tile's dQ contribution, dQ_i += scale sum_j dS_ij k_j.
//
// One CTA per (sequence, key/value head, 128-key tile), looping over the query
// heads of the group and the query tiles that see the key tile (all of them
// without a causal mask; under one, those from the key tile's diagonal on, up to
// the window's end).  Per step n the issuer runs
//   dV += P^T_n dO_n | S^T_{n+1} = K Q_{n+1}^T      (after P^T_n is written)
//   dQ_n = (dS_n K)  | dK += dS^T_n Q_n              (after dS_n is written)
//   dP^T_{n+1} = V dO_{n+1}^T                        (after dQ_n has been read out)
// P^T goes back to TMEM in place of S^T (the A operand of dV); dS_n goes to a
// 128 x 128 shared-memory tile, the operand of both dK (read K-major) and dQ
// (read MN-major).  d = 128: the dQ tile is formed transposed, dQ^T_n = K^T dS^T_n
// (TMEM lanes = the d channels), in the dP^T columns, which are free from the
// moment the dS pass has read them until dP^T_{n+1}; d = 64: dQ_n = dS_n K (lanes =
// query rows) in TMEM columns of its own.  Either way the layout of the
// accumulator in global memory puts a warp's 32 lanes on 32 consecutive words, so
// every reduction instruction covers one full 128-byte line.
//
// Warps: 0 TMA producer, 1 tcgen05 issuer (lane 0; owns TMEM), 2 relay (waits for
// streamed tiles and passes that on through the issuer's named barriers), 3 idle,
// 4..11 two element-wise warpgroups (64 query columns each; P^T and dS), 12..15 the
// dQ warpgroup: it copies each dQ tile from TMEM into registers (which frees the
// columns) and adds it into the accumulator.
//
// Deterministic sums without any order among CTAs.  Several key-tile CTAs add into
// each dQ row.  fp32 sums would depend on the order of those additions, and a fixed
// order costs a hand-off between CTAs per tile, measured at several times the
// tile's compute.  So each contribution is rounded to fixed point, an int32
// multiple of 2^-F_ic with F_ic = Fr_i + Fc_c: 2^Fr_i ||dO_i||_2 <= 2^15 (the
// preprocess, per query row) and 2^Fc_c times a bound on the contributions per
// unit of ||dO_i|| <= 2^15 (per key/value head and channel, from the maxima of
// |k_jc| and ||v_j||), so that every partial sum of an element stays below 2^30 in
// magnitude.  Integer additions commute, so the sums are the same whatever the
// order of the reductions.  A conversion kernel scales the sums back and rounds
// them to the output type; its error is at most (contributions / 2) 2^-F_ic.
#include "fa_bwd_common.cuh"

namespace fa {
namespace {

template <int D>
struct FusedCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kChunkBytes = kBlockM * 128;       // one 128-row x 128-byte block
    static constexpr int kTileBytes = kBlockM * D * 2;      // a 128-row tile of Q, K, V or dO
    static constexpr int kDSBytes = kBlockN * kBlockM * 2;  // dS^T: 128 keys x 128 queries
    static constexpr int kEwWG = 2;                         // element-wise warpgroups
    static constexpr int kEwCols = 64;                      // query columns of each
    static constexpr int kEwThreads = 128 * kEwWG;
    static constexpr int kThreads = 128 + kEwThreads + 128; // + the dQ warpgroup
    static constexpr int kRegsLaunch = 65536 / kThreads;    // 128
    // the dQ warps hold a whole 128-value row (d = 128) of the tile in registers
    static constexpr int kRegsCtl = (D == 128) ? 56 : 48;
    static constexpr int kRegsEw = 144;
    static constexpr int kRegsDq = (D == 128) ? 168 : 176;
    static_assert(128 * kRegsCtl + kEwThreads * kRegsEw + 128 * kRegsDq <= kThreads * kRegsLaunch,
                  "register split exceeds the launch's registers");
    // streamed tiles: Q_n (even items) and dO_n (odd items).  Q_n is held from S^T_n
    // to dK_n, about one and a half steps, dO_n from dP^T_n to dV_n, about half a
    // step; the shared memory left after K, V and dS buys 4 slots at d = 128.
    static constexpr int kSlots = (D == 128) ? 4 : 10;
    static constexpr int kSlotsOdd = (D == 128) ? 1 : 3;
    static constexpr int kTmemCols = 512;
    static constexpr int kColS = 0;                         // S^T, then P^T (bf16 pairs)
    static constexpr int kColDP = 128;                      // dP^T
    static constexpr int kColDV = 256;
    static constexpr int kColDK = 256 + D;
    static constexpr int kColDQ = (D == 128) ? kColDP : kColDK + D;   // d = 128: shares dP^T's
    static_assert(kColDQ + 128 <= kTmemCols || D == 64, "TMEM columns");
    static_assert(D == 128 || kColDQ + D <= kTmemCols, "TMEM columns");
    static constexpr int kBarBytes = 512;
    static constexpr int kStatOffset = kBarBytes;           // [wg][buf][2 x 64] fp32
    static constexpr int kFcOffset = kStatOffset + 2 * 2 * 2 * kEwCols * 4;   // d = 64: 2^Fc per channel
    static constexpr int kHeadBytes = 3072;
    static constexpr int kSmemBytes = kHeadBytes + 2 * kTileBytes + kDSBytes + kSlots * kTileBytes;
};
static_assert(FusedCfg<128>::kSmemBytes <= 232448, "shared memory budget");
static_assert(FusedCfg<64>::kSmemBytes <= 232448, "shared memory budget");
static_assert(FusedCfg<64>::kFcOffset + 64 * 4 <= FusedCfg<64>::kHeadBytes, "stats and channel scales");

// named barriers (0 is __syncthreads)
constexpr int kFBarP = 1;      // P^T_n written (element-wise) + Q_{n+1} landed (relay)
constexpr int kFBarDS = 2;     // dS_n written (element-wise)
constexpr int kFBarDQ = 3;     // dQ_n read out (dQ warps) + dO_{n+1} landed (relay)
constexpr int kFBarEpi = 4;    // element-wise warps among themselves: the dK/dV epilogue
constexpr int kFBarStat = 5;   // + warpgroup (5, 6): a warpgroup's row statistics staged
constexpr int kFBarDqw = 7;    // the dQ warps among themselves: channel scales staged (d = 64)
constexpr int kCountP = 256 + 64;    // element-wise + issuer + relay
constexpr int kCountDS = 256 + 32;   // element-wise + issuer
constexpr int kCountDQ = 128 + 64;   // dQ warps + issuer + relay

// Slot ring of the streamed tiles: even items (Q_n) take the first SLOTS - ODD
// slots, odd items (dO_n) the last ODD.  One odd slot is enough here: the relay
// waits for the odd items in order, each only after a barrier that the issuer
// passes after having seen the previous one land, so no wait can complete on the
// phase of an earlier item.
template <int SLOTS, int ODD>
struct FusedRing {
    static constexpr int kSlots = SLOTS;
    static constexpr int kEven = SLOTS - ODD;
    static_assert(ODD >= 1 && kEven >= 2, "slots per kind of item");
    __device__ static __forceinline__ int index(int i) {
        const int k = i >> 1;
        return (i & 1) ? kEven + k % ODD : k % kEven;
    }
    __device__ static __forceinline__ int use(int i) {
        const int k = i >> 1;
        return (i & 1) ? k / ODD : k / kEven;
    }
};

// D (128 x N fp32) = A . B with A and B both MN-major 128-byte-swizzled tiles of
// 128 rows along K (keys): d = 128, A = K (d contiguous: K^T), B = dS^T (queries
// contiguous) -> dQ^T; d = 64, A = dS^T read as dS (queries contiguous), B = K -> dQ.
template <int N, int E>
__device__ __forceinline__ void issue_mn_mn(uint32_t d_tmem, uint32_t a, uint32_t b) {
    constexpr uint32_t kIdesc = idesc_f32acc(kBlockM, N, true, true, E);
    const uint64_t ad = sdesc_sw128(a, kBlockM * 128, 1024), bd = sdesc_sw128(b, kBlockM * 128, 1024);
#pragma unroll
    for (int kk = 0; kk < kBlockN / 16; ++kk)
        mma_ss(d_tmem, ad + ((kk * 2048) >> 4), bd + ((kk * 2048) >> 4), kIdesc, kk > 0 ? 1u : 0u);
}

// dK (128 keys x D) (+)= dS^T (K-major: each key row's 128 queries contiguous) . Q_n
// (MN-major: each query row's D channels contiguous).
template <int D, int E>
__device__ __forceinline__ void issue_dk(uint32_t d_tmem, uint32_t ds, uint32_t q, bool acc) {
    constexpr uint32_t kIdesc = idesc_f32acc(kBlockM, D, false, true, E);
    constexpr int kChunk = kBlockM * 128;
    const uint64_t ad = sdesc_sw128(ds, 16, 1024), bd = sdesc_sw128(q, kChunk, 1024);
#pragma unroll
    for (int kk = 0; kk < kBlockM / 16; ++kk) {
        const uint32_t a_off = ((kk / 4) * kChunk + (kk % 4) * 32) >> 4;
        mma_ss(d_tmem, ad + a_off, bd + ((kk * 2048) >> 4), kIdesc, (acc || kk > 0) ? 1u : 0u);
    }
}

template <int D, int E, bool DROP>
__global__ void __launch_bounds__(FusedCfg<D>::kThreads, 1) fa_bwd_fused_kernel(const __grid_constant__ BwdParams p) {
    using C = FusedCfg<D>;
    using R = FusedRing<C::kSlots, C::kSlotsOdd>;   // Q_n (even), dO_n (odd)
    constexpr int W = C::kEwCols;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (!smem_base_ok(smem_raw, p.status)) return;
    const SeqInfo& s = p.seq;
    int b, g, kblk;
    // most expensive key tiles first (the sums need no order)
    if (!map_work(s, blockIdx.x, kBlockN, s.Hkv, false, b, g, kblk)) return;
    int seq_start, len;
    seq_bounds(s, b, seq_start, len);
    const int kb = kblk * kBlockN;
    const int k_last = min(kb + kBlockN - 1, len - 1);
    const int qt_first = query_lo(s, kb) / kBlockM;
    const int qt_last = query_hi(s, k_last, len) / kBlockM;
    const int nq = qt_last - qt_first + 1;
    const int nsteps = s.group * nq;

    BwdBars* bars = reinterpret_cast<BwdBars*>(smem_raw);
    float* sStat = reinterpret_cast<float*>(smem_raw + C::kStatOffset);
    uint8_t* sK = smem_raw + C::kHeadBytes;
    uint8_t* sV = sK + C::kTileBytes;
    uint8_t* sDS = sV + C::kTileBytes;
    uint8_t* sSlots = sDS + C::kDSBytes;
    volatile int* abort_flag = &bars->abort;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    init_bwd_cta<D>(bars, warp, C::kSlots);
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        regs_lower<C::kRegsCtl>();
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t rb = smem_addr(&bars->res_full);
            mbar_arrive_expect_tx(rb, 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(smem_addr(sK + c * C::kChunkBytes), &p.tm_k, rb, c * 64, g, seq_start + kb);
                tma_load_3d(smem_addr(sV + c * C::kChunkBytes), &p.tm_v, rb, c * 64, g, seq_start + kb);
            }
            stream_tiles<D, R>(bars, sSlots, 2 * nsteps, &p.tm_q, &p.tm_do,
                               [&](int i, int& head, int& row) {
                                   const int n = i / 2;
                                   head = g * s.group + n / nq;
                                   row = seq_start + (qt_first + n % nq) * kBlockM;
                               },
                               abort_flag, p, true);
        }
    } else if (warp == 1) {
        regs_lower<C::kRegsCtl>();
        // ------------------------------------------------------ MMA issuer
        // The whole warp walks the steps (named barriers are warp-collective); lane 0
        // issues.  No mbarrier wait inside the loop, no look at the abort flag: after
        // an abort it keeps issuing on stale data so that every phase completes.
        auto slot = [&](int i) { return smem_addr(sSlots + R::index(i) * C::kTileBytes); };
        auto free_slot = [&](int i) { mma_commit(smem_addr(&bars->slot_empty[R::index(i)])); };
        const uint32_t aK = smem_addr(sK), aV = smem_addr(sV), aDS = smem_addr(sDS);
        if (lane == 0) {
            auto wait = [&](uint64_t& bar, int parity) {
                return mbar_wait(smem_addr(&bar), parity, abort_flag, p.timeout_cycles, p.status);
            };
            if (wait(bars->res_full, 0) && wait(bars->slot_full[R::index(0)], 0) &&
                wait(bars->slot_full[R::index(1)], 0)) {}
            tc_fence_after();
            issue_ss<D, E>(tmem + C::kColS, aK, slot(0));      // S^T_0 = K Q_0^T
            mma_commit(smem_addr(&bars->s_full));
            issue_ss<D, E>(tmem + C::kColDP, aV, slot(1));     // dP^T_0 = V dO_0^T
            mma_commit(smem_addr(&bars->dp_full[0]));
        }
        __syncwarp();
        for (int n = 0; n < nsteps; ++n) {
            const bool more = n + 1 < nsteps;
            named_bar_sync(kFBarP, kCountP);            // P^T_n written, Q_{n+1} landed
            if (lane == 0) {
                tc_fence_after();
                issue_ts<D, E, W>(tmem + C::kColDV, tmem + C::kColS, slot(2 * n + 1), n > 0);  // dV += P^T dO
                free_slot(2 * n + 1);
                if (more) {
                    issue_ss<D, E>(tmem + C::kColS, aK, slot(2 * n + 2));                  // S^T_{n+1}
                    mma_commit(smem_addr(&bars->s_full));
                }
            }
            __syncwarp();
            named_bar_sync(kFBarDS, kCountDS);          // dS_n written
            if (lane == 0) {
                tc_fence_after();
                if constexpr (D == 128)
                    issue_mn_mn<128, E>(tmem + C::kColDQ, aK, aDS);   // dQ^T_n = K^T dS^T_n
                else
                    issue_mn_mn<D, E>(tmem + C::kColDQ, aDS, aK);     // dQ_n = dS_n K
                mma_commit(smem_addr(&bars->dq_full));
                issue_dk<D, E>(tmem + C::kColDK, aDS, slot(2 * n), n > 0);                  // dK += dS^T Q
                free_slot(2 * n);
            }
            __syncwarp();
            named_bar_sync(kFBarDQ, kCountDQ);          // dQ_n read out, dO_{n+1} landed
            if (lane == 0 && more) {
                tc_fence_after();
                issue_ss<D, E>(tmem + C::kColDP, aV, slot(2 * n + 3));                      // dP^T_{n+1}
                mma_commit(smem_addr(&bars->dp_full[0]));
            }
            __syncwarp();
        }
        if (lane == 0) mma_commit(smem_addr(&bars->acc_full));
    } else if (warp == 2) {
        regs_lower<C::kRegsCtl>();
        // ------------------------------------------------------ slot relay
        auto wait_item = [&](int i) {
            mbar_wait(smem_addr(&bars->slot_full[R::index(i)]), R::use(i) & 1, abort_flag,
                      p.timeout_cycles, p.status);
        };
        if (lane == 0) wait_item(1);   // dO_0: the odd items are waited for in order
        __syncwarp();
        for (int n = 0; n < nsteps; ++n) {
            const bool more = n + 1 < nsteps;
            if (lane == 0 && more) wait_item(2 * n + 2);   // Q_{n+1}
            __syncwarp();
            named_bar_sync(kFBarP, kCountP);
            if (lane == 0 && more) wait_item(2 * n + 3);   // dO_{n+1}
            __syncwarp();
            named_bar_sync(kFBarDQ, kCountDQ);
        }
    } else if (warp == 3) {
        regs_lower<C::kRegsCtl>();   // idle; its warpgroup gives registers away
    } else if (warp < 12) {
        regs_raise<C::kRegsEw>();
        // ------------------------------------------- element-wise + epilogue
        const int wg = (warp - 4) / 4;      // query columns [W wg, W wg + W) of each tile
        const int quad = warp % 4;
        const int r = quad * 32 + lane;     // key row within the tile = TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_addr + C::kColS + W * wg;
        const uint32_t tDP = tmem + lane_addr + C::kColDP + W * wg;
        uint8_t* ds_chunk = sDS + wg * C::kChunkBytes;   // dS^T columns [W wg, W wg + W)
        const int kpos = kb + r;
        const int qlo = query_lo(s, kpos);
        const int qhi = (kpos < len) ? query_hi(s, kpos, len) : -1;
        const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
        // row statistics of step m for this warpgroup's W query columns, negated:
        // thread r fetches -LSE (log2 units) of column r (r < W) or -D of column r - W
        auto fetch_stat = [&](int m) -> float {
            const int h = g * s.group + m / nq;
            const int q = (qt_first + m % nq) * kBlockM + W * wg + (r % W);
            if (q >= len) return r < W ? -kPosInf : 0.f;
            const long long idx = row_stat_index(s, b, h, seq_start, q);
            if (!fa_index_ok(idx, static_cast<long long>(s.total_tokens) * s.Hq, p.status)) return 0.f;
            return r < W ? -__ldg(p.lse + idx) * kLog2eF : -__ldg(p.delta + idx);
        };
        float next_stat = fetch_stat(0);
        uint32_t dw[DROP ? W / 4 : 1];
        auto draw = [&](int n) {
            dropout_words_cols<W / 4>(*reinterpret_cast<uint32_t(*)[W / 4]>(dw),
                                      ((qt_first + n % nq) * kBlockM + W * wg) >> 2, kpos >> 2,
                                      static_cast<uint32_t>(b * s.Hq + g * s.group + n / nq),
                                      p.drop.offset, p.drop.seed_lo, p.drop.seed_hi, lane);
            keep_masks(*reinterpret_cast<uint32_t(*)[W / 4]>(dw), p.drop.thresh);
        };
        if (DROP) draw(0);
        bool ok = true;
        for (int n = 0; n < nsteps; ++n) {
            const int buf = n & 1;
            float* sb = sStat + (wg * 2 + buf) * (2 * W);
            const int q0 = (qt_first + n % nq) * kBlockM + W * wg;
            const bool need_mask = !(q0 >= qlo && q0 + W - 1 <= qhi);
            const int clo = qlo - q0, chi = qhi - q0;
            const float4* nlse4 = reinterpret_cast<const float4*>(sb);
            const float4* ndlt4 = reinterpret_cast<const float4*>(sb + W);
            if (ok) sb[r] = next_stat;
            named_bar_sync(kFBarStat + wg, 128);
            if (ok && n + 1 < nsteps) next_stat = fetch_stat(n + 1);
            // P^T = exp(S^T - LSE), written back as 16-bit pairs in place (with dropout
            // the kept entries only; dV takes the inverse keep probability at the end)
            if (ok) ok = warp_wait(smem_addr(&bars->s_full), n & 1, abort_flag, p.timeout_cycles, p.status);
            float pv[W];
            if (ok) {
                tc_fence_after();
                tmem_ldw<W>(tS, pv);
#pragma unroll
                for (int c4 = 0; c4 < W / 4; ++c4) {
                    const float4 nl = nlse4[c4];
                    const float2 a = f2_unpack(f2_fma(f2_pack(pv[4 * c4], pv[4 * c4 + 1]), sl2x2,
                                                      f2_pack(nl.x, nl.y)));
                    const float2 e = f2_unpack(f2_fma(f2_pack(pv[4 * c4 + 2], pv[4 * c4 + 3]), sl2x2,
                                                      f2_pack(nl.z, nl.w)));
                    pv[4 * c4] = ex2_approx(a.x);
                    pv[4 * c4 + 1] = ex2_approx(a.y);
                    pv[4 * c4 + 2] = ex2_approx(e.x);
                    pv[4 * c4 + 3] = ex2_approx(e.y);
                }
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < W; ++c)
                        if (c < clo || c > chi) pv[c] = 0.f;
                }
                if (DROP)
                    tmem_st_pk_dropped<W, E>(tS, pv, *reinterpret_cast<const uint32_t(*)[W / 4]>(dw));
                else
                    tmem_st_pk<W, E>(tS, pv);
                tmem_st_wait();
                tc_fence_before();
            }
            named_bar_signal(kFBarP, kCountP, ok);
            // dS = P (dP - D) into the shared dS^T tile (key row r, this warpgroup's
            // columns), 32 columns at a time
            if (ok) ok = warp_wait(smem_addr(&bars->dp_full[0]), n & 1, abort_flag, p.timeout_cycles, p.status);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t raw[32];
                    tmem_ld32(tDP + 32 * half, raw);
                    tmem_ld_wait();
                    reg_fence(raw);
                    // with dropout dS = P (r keep dZ - D): the dropped columns cleared by
                    // their masks, r folded into the multiply-add
                    float dp[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        dp[i] = __uint_as_float(raw[i]);
                        if (DROP)
                            dp[i] = __uint_as_float(raw[i] & keep_mask32(dw[(32 * half + i) >> 2], i));
                    }
                    const uint64_t rr = f2_pack(p.drop.rscale, p.drop.rscale);
                    uint32_t wds[16];
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 nd = ndlt4[8 * half + c4];
                        const int c = 32 * half + 4 * c4;
                        const uint64_t z0 = DROP ? f2_fma(rr, f2_pack(dp[4 * c4], dp[4 * c4 + 1]), f2_pack(nd.x, nd.y))
                                                 : f2_add(f2_pack(dp[4 * c4], dp[4 * c4 + 1]), f2_pack(nd.x, nd.y));
                        const uint64_t z1 = DROP ? f2_fma(rr, f2_pack(dp[4 * c4 + 2], dp[4 * c4 + 3]), f2_pack(nd.z, nd.w))
                                                 : f2_add(f2_pack(dp[4 * c4 + 2], dp[4 * c4 + 3]), f2_pack(nd.z, nd.w));
                        const float2 a = f2_unpack(f2_mul(f2_pack(pv[c], pv[c + 1]), z0));
                        const float2 e = f2_unpack(f2_mul(f2_pack(pv[c + 2], pv[c + 3]), z1));
                        wds[2 * c4] = pack2<E>(a.x, a.y);
                        wds[2 * c4 + 1] = pack2<E>(e.x, e.y);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        *swizzled_unit(ds_chunk, r, 4 * half + u) =
                            make_uint4(wds[4 * u], wds[4 * u + 1], wds[4 * u + 2], wds[4 * u + 3]);
                }
                tc_fence_before();
                fence_proxy_async_smem();   // the generic-proxy writes, before the MMAs read them
            }
            named_bar_signal(kFBarDS, kCountDS, ok);
            if (DROP && ok && n + 1 < nsteps) draw(n + 1);
        }
        if (ok)
            ok = warp_wait(smem_addr(&bars->acc_full), 0, abort_flag, p.timeout_cycles, p.status);
        // dV (first warpgroup) and dK (second, scaled) leave through the idle slot
        // ring and TMA stores; a key tile cut by the sequence end row by row
        const bool is_dk = wg == 1;
        const uint32_t t_acc = tmem + lane_addr + (is_dk ? C::kColDK : C::kColDV);
        const float mul = is_dk ? p.scale : (DROP ? p.drop.rscale : 1.f);
        if (named_bar_all(kFBarEpi, C::kEwThreads, ok && kb + kBlockN <= len)) {
            tc_fence_after();
            stage_acc_row<D, E>(t_acc, mul, sSlots + (is_dk ? C::kTileBytes : 0), C::kChunkBytes, r, 0);
            fence_proxy_async_smem();
            named_bar_sync(kFBarEpi, C::kEwThreads);
            if (warp == 4 && lane == 0) {
                if (fa_box_ok(seq_start + kb, kBlockN, s.total_tokens, g, s.Hkv, p.status))
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_store_3d(&p.tm_dv, smem_addr(sSlots + c * C::kChunkBytes), c * 64, g,
                                     seq_start + kb);
                        tma_store_3d(&p.tm_dk, smem_addr(sSlots + C::kTileBytes + c * C::kChunkBytes),
                                     c * 64, g, seq_start + kb);
                    }
                bulk_commit_group();
                bulk_wait_read_all();
            }
        } else if (ok) {
            tc_fence_after();
            const long long row = (static_cast<long long>(seq_start + kpos) * s.Hkv + g) * D;
            store_acc_row<D, E>(t_acc, mul, static_cast<uint16_t*>(is_dk ? p.dk : p.dv) + row,
                                kpos < len && fa_index_ok(static_cast<long long>(seq_start + kpos) * s.Hkv + g,
                                                          static_cast<long long>(s.total_tokens) * s.Hkv, p.status));
        }
    } else {
        regs_raise<C::kRegsDq>();
        // ------------------------------------------------------ dQ warps
        // d = 128: thread = channel c (TMEM lane) of dQ^T, its 128 values the tile's
        //          query rows; accumulator [Hq, tokens, 128].
        // d = 64:  thread = query row of dQ, its 64 values the channels; accumulator
        //          [Hq, 64, tokens].
        // Each value goes in as the int32 round(v 2^Fr_i 2^Fc_c) (both factors powers
        // of two, so the products are exact): no order among the CTAs is needed.
        constexpr int NV = (D == 128) ? kBlockM : D;
        const int quad = warp % 4;
        const int ln = quad * 32 + lane;
        const uint32_t tDQ = tmem + (static_cast<uint32_t>(quad * 32) << 16) + C::kColDQ;
        const long long T = s.total_tokens;
        const float r = DROP ? p.drop.rscale : 1.f;
        float* sFc = reinterpret_cast<float*>(smem_raw + C::kFcOffset);
        float fc = 1.f;
        if constexpr (D == 128) {
            fc = channel_scale<D>(p.kv_bound, g, ln, r);
        } else {
            if (ln < D) sFc[ln] = channel_scale<D>(p.kv_bound, g, ln, r);
            named_bar_sync(kFBarDqw, 128);
        }
        bool ok = true;
        for (int n = 0; n < nsteps; ++n) {
            const int h = g * s.group + n / nq;
            const int q0 = (qt_first + n % nq) * kBlockM;
            const int rows = min(kBlockM, len - q0);
            // the tile's row scales (fetched before the wait); d = 128: lane l holds those
            // of rows l, l + 32, l + 64, l + 96
            float rs[D == 128 ? 4 : 1];
#pragma unroll
            for (int m = 0; m < (D == 128 ? 4 : 1); ++m) {
                const int q = q0 + (D == 128 ? 32 * m + lane : ln);
                rs[m] = (q < len && fa_index_ok(row_stat_index(s, b, h, seq_start, q), T * s.Hq, p.status))
                            ? __ldg(p.row_scale + row_stat_index(s, b, h, seq_start, q)) : 0.f;
            }
            float acc[NV];
            if (ok) ok = warp_wait(smem_addr(&bars->dq_full), n & 1, abort_flag, p.timeout_cycles, p.status);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < NV / 32; ++c)
                    tmem_ld32(tDQ + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&acc[32 * c]));
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < NV / 32; ++c) reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&acc[32 * c]));
                tc_fence_before();
            }
            named_bar_signal(kFBarDQ, kCountDQ, ok);    // the columns may be overwritten
            if (!ok) continue;
            if constexpr (D == 128) {
                int* accg = p.dq_acc + (static_cast<long long>(h) * T + seq_start + q0) * 128 + ln;
#pragma unroll
                for (int j = 0; j < NV; ++j) {
                    const float sj = __shfl_sync(0xffffffffu, rs[j / 32], j % 32);
                    if (j < rows && fa_index_ok((static_cast<long long>(h) * T + seq_start + q0 + j) * 128 + ln,
                                                T * s.Hq * 128, p.status))
                        red_add_s32(accg + j * 128, __float2int_rn(acc[j] * sj * fc));
                }
            } else if (ln < rows && fa_index_ok(static_cast<long long>(h) * D * T + (D - 1) * T + seq_start + q0 + ln,
                                                T * s.Hq * D, p.status)) {
                int* accg = p.dq_acc + static_cast<long long>(h) * D * T + seq_start + q0 + ln;
#pragma unroll
                for (int c = 0; c < NV; ++c) red_add_s32(accg + c * T, __float2int_rn(acc[c] * rs[0] * sFc[c]));
            }
        }
    }
    teardown_bwd_cta<D>(bars, warp);
}

// dQ_ic = scale 2^-(Fr_i + Fc_c) (sum of the contributions), rounded to E: one CTA
// per (query head, 64 tokens).  d = 128 reads the accumulator [Hq, tokens, 128]
// row by row; d = 64 transposes [Hq, 64, tokens] through shared memory.
constexpr int kConvTokens = 64;
constexpr int kConvThreads = 256;

template <int D, int E, bool DROP>
__global__ void __launch_bounds__(kConvThreads) fa_bwd_dq_convert_kernel(const __grid_constant__ BwdParams p) {
    __shared__ float sInvFc[D];
    __shared__ int sT[D == 64 ? 64 : 1][65];
    const SeqInfo& s = p.seq;
    const int h = blockIdx.y, g = h / s.group;
    const long long T = s.total_tokens;
    const long long t0 = static_cast<long long>(blockIdx.x) * kConvTokens;
    if (threadIdx.x < D) sInvFc[threadIdx.x] = 1.f / channel_scale<D>(p.kv_bound, g, threadIdx.x, DROP ? p.drop.rscale : 1.f);
    // row-statistics index of token t: dense [B, Hq, N], packed [Hq, T]
    auto stat_index = [&](long long t) -> long long {
        if (s.cu_seqlens) return static_cast<long long>(h) * T + t;
        return (t / s.N * s.Hq + h) * s.N + t % s.N;
    };
    if constexpr (D == 64) {
        // accumulator columns t0 .. t0 + 63 of the head's 64 channel rows
#pragma unroll
        for (int k = 0; k < kConvTokens * D / kConvThreads; ++k) {
            const int idx = k * kConvThreads + threadIdx.x;
            const int c = idx / kConvTokens, j = idx % kConvTokens;
            sT[c][j] = (t0 + j < T && fa_index_ok((static_cast<long long>(h) * D + c) * T + t0 + j,
                                                  T * s.Hq * D, p.status))
                           ? p.dq_acc[(static_cast<long long>(h) * D + c) * T + t0 + j] : 0;
        }
    }
    __syncthreads();
    constexpr int kItems = kConvTokens * (D / 8);   // (token, 8 channels)
#pragma unroll
    for (int k = 0; k < kItems / kConvThreads; ++k) {
        const int idx = k * kConvThreads + threadIdx.x;
        const int j = idx / (D / 8), c8 = (idx % (D / 8)) * 8;
        const long long t = t0 + j;
        if (t >= T || !fa_index_ok(t * s.Hq + h, T * s.Hq, p.status)) continue;
        int v[8];
        if constexpr (D == 128) {
            const int4* src = reinterpret_cast<const int4*>(p.dq_acc + (static_cast<long long>(h) * T + t) * D + c8);
            const int4 a = src[0], b2 = src[1];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b2.x; v[5] = b2.y; v[6] = b2.z; v[7] = b2.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = sT[c8 + i][j];
        }
        const float inv_r = p.scale / p.row_scale[stat_index(t)];
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = pack2<E>(static_cast<float>(v[2 * i]) * sInvFc[c8 + 2 * i] * inv_r,
                            static_cast<float>(v[2 * i + 1]) * sInvFc[c8 + 2 * i + 1] * inv_r);
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dq) + (t * s.Hq + h) * D + c8) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int D, int E, bool DROP>
cudaError_t launch_convert_d(const BwdParams& p, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>((p.seq.total_tokens + kConvTokens - 1) / kConvTokens),
                    static_cast<unsigned>(p.seq.Hq));
    fa_bwd_dq_convert_kernel<D, E, DROP><<<grid, kConvThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int D, int E>
cudaError_t launch_convert_de(const BwdParams& p, cudaStream_t stream) {
    return p.drop.thresh ? launch_convert_d<D, E, true>(p, stream) : launch_convert_d<D, E, false>(p, stream);
}

template <int D, int E, bool DROP>
cudaError_t launch_fused_d(const BwdParams& p, cudaStream_t stream) {
    static const cudaError_t regs_ok = check_regs(fa_bwd_fused_kernel<D, E, DROP>, FusedCfg<D>::kRegsLaunch);
    if (regs_ok != cudaSuccess) return regs_ok;
    return launch_tc(fa_bwd_fused_kernel<D, E, DROP>, p.num_work_dkdv, FusedCfg<D>::kThreads,
                     FusedCfg<D>::kSmemBytes, p, stream);
}

template <int D, int E>
cudaError_t launch_fused_de(const BwdParams& p, cudaStream_t stream) {
    return p.drop.thresh ? launch_fused_d<D, E, true>(p, stream) : launch_fused_d<D, E, false>(p, stream);
}

}  // namespace

cudaError_t launch_bwd_dq_convert(const BwdParams& p, int d, cudaStream_t stream) {
    if (p.seq.total_tokens <= 0) return cudaSuccess;
    if (p.elem == kElemF16)
        return d == 128 ? launch_convert_de<128, kElemF16>(p, stream) : launch_convert_de<64, kElemF16>(p, stream);
    return d == 128 ? launch_convert_de<128, kElemBf16>(p, stream) : launch_convert_de<64, kElemBf16>(p, stream);
}

cudaError_t launch_bwd_fused(const BwdParams& p, int d, cudaStream_t stream) {
    if (p.num_work_dkdv <= 0) return cudaSuccess;
    if (p.elem == kElemF16)
        return d == 128 ? launch_fused_de<128, kElemF16>(p, stream) : launch_fused_de<64, kElemF16>(p, stream);
    return d == 128 ? launch_fused_de<128, kElemBf16>(p, stream) : launch_fused_de<64, kElemBf16>(p, stream);
}

}  // namespace fa
