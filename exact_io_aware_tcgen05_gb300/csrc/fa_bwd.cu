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
//                      over the key tiles; Q and dO held in TMEM as the A
//                      operands of S and dP, dS (bf16) back to TMEM feeds
//                      dQ += dS K
// Warp roles in both tensor-core kernels: warp 0 TMA producer, warp 1 tcgen05
// issuer (one thread, owns TMEM), warps 4.. element-wise work + epilogue as two
// (d = 128) or four (d = 64) warpgroups, each owning 64 or 32 of the 128 tile
// columns (TMEM lane = row).
#include "fa_bwd_common.cuh"

namespace fa {
namespace {

// ------------------------------------------------------------- preprocess

// D_i = sum_c dO_ic O_ic in fp32 for every (token, query head).  A group of
// D/8 lanes handles one row, 8 elements (16 bytes) per lane; a CTA takes
// kPrePasses passes of 256 / (D/8) consecutive rows, all of whose loads are
// issued before the first sum, so that every thread keeps 2 kPrePasses
// 16-byte loads in flight.  E: element type.
//
// For the fused backward the same launch also prepares its fixed-point dQ sums:
// the row CTAs write 2^Fr_i per row (Fr_i = 15 - e_i with 2^e_i >= ||dO_i||_2,
// so that 2^Fr_i ||dO_i||_2 <= 2^15) and zero the int32 accumulator; the CTAs
// after them (kBoundSlots per key/value head) take the maxima of |k_jc| per
// channel and of ||v_j||_2 over their slot of tokens.
constexpr int kPrePasses = 4;
constexpr int kPreThreads = 256;

template <int D>
constexpr int pre_rows_per_cta() { return kPrePasses * (kPreThreads / (D / 8)); }

template <int D, int E>
__device__ __forceinline__ void kv_bound_cta(const BwdParams& p, int bi) {
    constexpr int kLanesPerRow = D / 8;
    constexpr int kRowsPerPass = kPreThreads / kLanesPerRow;
    __shared__ unsigned int s_max[D + 1];   // non-negative floats as bits: order-preserving
    const SeqInfo& s = p.seq;
    const int g = bi / kBoundSlots, slot = bi % kBoundSlots;
    const long long T = s.total_tokens;
    const long long t0 = T * slot / kBoundSlots, t1 = T * (slot + 1) / kBoundSlots;
    for (int i = threadIdx.x; i <= D; i += kPreThreads) s_max[i] = 0u;
    __syncthreads();
    const int sub = threadIdx.x % kLanesPerRow;
    float kmax[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float vmax = 0.f;
    // the same number of trips for every thread (the row sums shuffle across the warp)
    const long long trips = (t1 - t0 + kRowsPerPass - 1) / kRowsPerPass;
    for (long long it = 0; it < trips; ++it) {
        const long long t = t0 + it * kRowsPerPass + threadIdx.x / kLanesPerRow;
        const bool in = t < t1;
        const long long off = (t * s.Hkv + g) * kLanesPerRow + sub;
        const uint4 k4 = in ? reinterpret_cast<const uint4*>(p.k_ptr)[off] : make_uint4(0u, 0u, 0u, 0u);
        const uint4 v4 = in ? reinterpret_cast<const uint4*>(p.v_ptr)[off] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t kw[4] = {k4.x, k4.y, k4.z, k4.w}, vw[4] = {v4.x, v4.y, v4.z, v4.w};
        float vsq = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = unpack2<E>(kw[i]), c = unpack2<E>(vw[i]);
            kmax[2 * i] = fmaxf(kmax[2 * i], fabsf(a.x));
            kmax[2 * i + 1] = fmaxf(kmax[2 * i + 1], fabsf(a.y));
            vsq = fmaf(c.x, c.x, fmaf(c.y, c.y, vsq));
        }
#pragma unroll
        for (int o = kLanesPerRow / 2; o > 0; o >>= 1) vsq += __shfl_xor_sync(0xffffffffu, vsq, o, kLanesPerRow);
        vmax = fmaxf(vmax, sqrtf(vsq));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) atomicMax(&s_max[8 * sub + i], __float_as_uint(kmax[i]));
    if (sub == 0) atomicMax(&s_max[D], __float_as_uint(vmax));
    __syncthreads();
    const long long o0 = (static_cast<long long>(g) * kBoundSlots + slot) * (D + 1);
    for (int i = threadIdx.x; i <= D; i += kPreThreads)
        if (fa_index_ok(o0 + i, static_cast<long long>(s.Hkv) * kBoundSlots * (D + 1), p.status))
            p.kv_bound[o0 + i] = __uint_as_float(s_max[i]);
}

template <int D, int E>
__global__ void __launch_bounds__(kPreThreads) fa_bwd_preprocess_kernel(const __grid_constant__ BwdParams p) {
    constexpr int kLanesPerRow = D / 8;
    constexpr int kRowsPerPass = kPreThreads / kLanesPerRow;
    const SeqInfo& s = p.seq;
    if (p.dq_acc && static_cast<int>(blockIdx.x) >= p.pre_row_ctas) {
        kv_bound_cta<D, E>(p, blockIdx.x - p.pre_row_ctas);
        return;
    }
    const long long rows = static_cast<long long>(s.total_tokens) * s.Hq;
    if (p.dq_acc) {
        // the fused backward's int32 dQ accumulator starts at zero
        const long long n4 = rows * D / 4;
        uint4* acc4 = reinterpret_cast<uint4*>(p.dq_acc);
        for (long long i = static_cast<long long>(blockIdx.x) * kPreThreads + threadIdx.x; i < n4;
             i += static_cast<long long>(p.pre_row_ctas) * kPreThreads)
            acc4[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    const long long row0 = static_cast<long long>(blockIdx.x) * pre_rows_per_cta<D>() +
                           threadIdx.x / kLanesPerRow;
    const int sub = threadIdx.x % kLanesPerRow;
    uint4 o4[kPrePasses], d4[kPrePasses];
#pragma unroll
    for (int k = 0; k < kPrePasses; ++k) {
        const long long row = row0 + k * kRowsPerPass;
        o4[k] = d4[k] = make_uint4(0u, 0u, 0u, 0u);
        if (row < rows) {
            o4[k] = reinterpret_cast<const uint4*>(p.o)[row * kLanesPerRow + sub];
            d4[k] = reinterpret_cast<const uint4*>(p.dout)[row * kLanesPerRow + sub];
        }
    }
#pragma unroll
    for (int k = 0; k < kPrePasses; ++k) {
        const long long row = row0 + k * kRowsPerPass;
        const uint32_t ow[4] = {o4[k].x, o4[k].y, o4[k].z, o4[k].w};
        const uint32_t dw[4] = {d4[k].x, d4[k].y, d4[k].z, d4[k].w};
        float acc = 0.f, dsq = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = unpack2<E>(ow[i]);
            const float2 c = unpack2<E>(dw[i]);
            acc = fmaf(a.x, c.x, acc);
            acc = fmaf(a.y, c.y, acc);
            dsq = fmaf(c.x, c.x, fmaf(c.y, c.y, dsq));
        }
#pragma unroll
        for (int off = kLanesPerRow / 2; off > 0; off >>= 1) {
            acc += __shfl_xor_sync(0xffffffffu, acc, off, kLanesPerRow);
            dsq += __shfl_xor_sync(0xffffffffu, dsq, off, kLanesPerRow);
        }
        if (row < rows && sub == 0) {
            const int token = static_cast<int>(row / s.Hq), h = static_cast<int>(row % s.Hq);
            long long idx;
            if (s.cu_seqlens) idx = static_cast<long long>(h) * s.total_tokens + token;
            else idx = (static_cast<long long>(token / s.N) * s.Hq + h) * s.N + token % s.N;
            if (fa_index_ok(idx, rows, p.status)) {
                p.delta[idx] = acc;
                if (p.dq_acc) p.row_scale[idx] = fixed_point_scale(sqrtf(dsq));
            }
        }
    }
}

// ------------------------------------------------------------------ dK, dV
//
// Per step n (one query head of the group, one 128-row query tile) the issuer
// runs   dV += P^T_n dO_n | S^T_{n+1} = K Q_{n+1}^T | dK += dS^T_n Q_n |
//        dP^T_{n+1} = V dO_{n+1}^T
// so the element-wise warps turn S^T_{n+1} into P^T_{n+1} while dK_n and
// dP^T_{n+1} run, and dP^T_n into dS^T_n while dV_n and S^T_{n+1} run.
// P^T overwrites S^T and dS^T overwrites dP^T in place; each product that
// overwrites a region is issued after the product reading it (tcgen05 ops of
// one thread execute in issue order).  Q_n and dO_n stream through the slot
// ring as items 2n and 2n+1; the element-wise warps fetch the row statistics
// (LSE, D) of step n+1 from global memory while they work on step n.
//
// Synchronisation: the issuer learns of the element-wise results (and, through
// a relay warp that waits on the slot mbarriers, of the streamed tiles) from
// two named barriers, kBarP and kBarDS0, one phase each per step; the
// element-wise warps learn of finished products from tcgen05.commit mbarriers.
// Each signal that would open phase n+1 of a named barrier depends on a product
// issued after phase n completed, so no participant gets a phase ahead.

template <int D, int E, bool DROP>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1) fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdCfg<D>;
    using R = Ring<C::kSlots, C::kSlotsOdd>;   // Q_n (even) and dO_n (odd)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the dQ kernel reads nothing this kernel writes: let it start on SMs this
    // grid's last CTAs leave idle
    grid_launch_dependents();
    if (!smem_base_ok(smem_raw, p.status)) return;
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

    BwdBars* bars = reinterpret_cast<BwdBars*>(smem_raw);
    float* sStat = reinterpret_cast<float*>(smem_raw + C::kStatOffset);   // [wg][buf][2 W]
    uint8_t* sK = smem_raw + C::kHeadBytes;
    uint8_t* sV = sK + C::kTileBytes;
    uint8_t* sSlots = sV + C::kTileBytes;
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
        // The whole warp walks the step sequence (the named barriers are
        // warp-collective); lane 0 issues.  It never waits on an mbarrier inside
        // the loop and does not look at the abort flag: after an abort it keeps
        // issuing (on stale data) so that every barrier phase still completes.
        auto slot = [&](int i) { return smem_addr(sSlots + R::index(i) * C::kTileBytes); };
        auto free_slot = [&](int i) { mma_commit(smem_addr(&bars->slot_empty[R::index(i)])); };
        const uint32_t aK = smem_addr(sK), aV = smem_addr(sV);
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
            named_bar_sync(kBarP, C::kBarCount);          // P^T_n written, Q_{n+1} landed
            if (lane == 0) {
                tc_fence_after();
                issue_ts<D, E>(tmem + C::kColAcc, tmem + C::kColS, slot(2 * n + 1), n > 0);   // dV += P^T dO
                free_slot(2 * n + 1);
                if (more) {
                    issue_ss<D, E>(tmem + C::kColS, aK, slot(2 * n + 2));                     // S^T_{n+1}
                    mma_commit(smem_addr(&bars->s_full));
                }
            }
            __syncwarp();
            named_bar_sync(kBarDS0, C::kBarCount);        // dS^T_n written, dO_{n+1} landed
            if (lane == 0) {
                tc_fence_after();
                issue_ts<D, E>(tmem + C::kColAcc + D, tmem + C::kColDP, slot(2 * n), n > 0);  // dK += dS^T Q
                free_slot(2 * n);
                if (more) {
                    issue_ss<D, E>(tmem + C::kColDP, aV, slot(2 * n + 3));                    // dP^T_{n+1}
                    mma_commit(smem_addr(&bars->dp_full[0]));
                }
            }
            __syncwarp();
        }
        if (lane == 0) mma_commit(smem_addr(&bars->acc_full));
    } else if (warp == 2) {
        regs_lower<C::kRegsCtl>();
        // ------------------------------------------------------ slot relay
        // Waits for the streamed tiles the next products read and passes that on
        // through the issuer's named barriers.
        for (int n = 0; n < nsteps; ++n) {
            const bool more = n + 1 < nsteps;
            if (lane == 0 && more)
                mbar_wait(smem_addr(&bars->slot_full[R::index(2 * n + 2)]),
                          R::use(2 * n + 2) & 1, abort_flag, p.timeout_cycles, p.status);
            __syncwarp();
            named_bar_sync(kBarP, C::kBarCount);
            if (lane == 0 && more)
                mbar_wait(smem_addr(&bars->slot_full[R::index(2 * n + 3)]),
                          R::use(2 * n + 3) & 1, abort_flag, p.timeout_cycles, p.status);
            __syncwarp();
            named_bar_sync(kBarDS0, C::kBarCount);
        }
    } else if (warp == 3) {
        regs_lower<C::kRegsCtl>();   // idle; its warpgroup gives registers away
    } else if (warp >= 4) {
        regs_raise<C::kRegsEw>();
        // ------------------------------------------- element-wise + epilogue
        constexpr int W = C::kEwCols;
        const int wg = (warp - 4) / 4;      // query columns [W wg, W wg + W) of each tile
        const int quad = warp % 4;
        const int r = quad * 32 + lane;     // key row within the tile = TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_addr + C::kColS + W * wg;
        const uint32_t tDP = tmem + lane_addr + C::kColDP + W * wg;
        const int kpos = kb + r;
        // queries that see this key: [qlo, qhi]; none if the key is past the end
        const int qlo = query_lo(s, kpos);
        const int qhi = (kpos < len) ? query_hi(s, kpos, len) : -1;
        const float sl2 = p.scale_log2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        // Row statistics of step m for this warpgroup's W query columns, negated:
        // thread r fetches -LSE (in log2 units) of column r (r < W) or -D of
        // column r - W (r < 2W); rows past the sequence end get -inf / 0 so they
        // contribute nothing.
        auto fetch_stat = [&](int m) -> float {
            if (r >= 2 * W) return 0.f;
            const int h = g * s.group + m / nq;
            const int q = (qt_first + m % nq) * kBlockM + W * wg + (r % W);
            if (q >= len) return r < W ? -kPosInf : 0.f;
            const long long idx = row_stat_index(s, b, h, seq_start, q);
            if (!fa_index_ok(idx, static_cast<long long>(s.total_tokens) * s.Hq, p.status)) return 0.f;
            return r < W ? -__ldg(p.lse + idx) * kLog2eF : -__ldg(p.delta + idx);
        };
        float next_stat = fetch_stat(0);
        // Dropout bytes of this key row for the current step, 4 queries a word.  They
        // do not depend on the products, so the next step's are drawn at the end of
        // each step, while the tensor cores work on that step's S^T.
        uint32_t dw[DROP ? W / 4 : 1];
        auto draw = [&](int n) {
            dropout_words_cols<W / 4>(*reinterpret_cast<uint32_t(*)[W / 4]>(dw),
                                      ((qt_first + n % nq) * kBlockM + W * wg) >> 2, kpos >> 2,
                                      static_cast<uint32_t>(b * s.Hq + g * s.group + n / nq),
                                      p.drop.offset, p.drop.seed_lo, p.drop.seed_hi, lane);
            keep_masks(*reinterpret_cast<uint32_t(*)[W / 4]>(dw), p.drop.thresh);
        };
        if (DROP) draw(0);
        // `ok` turns false (warp-uniformly) when a wait gives up; the warp then
        // skips the work but keeps taking part in every named-barrier phase,
        // blocking (bar.sync) instead of arriving so it cannot run a phase ahead.
        bool ok = true;
        for (int n = 0; n < nsteps; ++n) {
            const int buf = n & 1;
            float* sb = sStat + (wg * 2 + buf) * (2 * W);
            const int q0 = (qt_first + n % nq) * kBlockM + W * wg;   // first query of my columns
            const bool need_mask = !(q0 >= qlo && q0 + W - 1 <= qhi);
            const int clo = qlo - q0, chi = qhi - q0;
            const float4* nlse4 = reinterpret_cast<const float4*>(sb);
            const float4* ndlt4 = reinterpret_cast<const float4*>(sb + W);
            // The four warps of the warpgroup stage the step's statistics and meet at a
            // named barrier (every step, whatever `ok`): a hardware barrier, where 128
            // mbarrier arrivals and their polls had cost 0.5% (d = 128) to 1.3% (d = 64)
            // of the backward.  A buffer is written again two steps later, after every
            // warp of the warpgroup has passed the barrier in between.
            if (ok && r < 2 * W) sb[r] = next_stat;
            named_bar_sync(kBarStat + wg, 128);
            if (ok && n + 1 < nsteps) next_stat = fetch_stat(n + 1);   // in flight during this step
            // P^T = exp(S^T - LSE) (keys x queries), written back as bf16 in place (with
            // dropout: the kept entries only, the operand of dV; dV is scaled by the
            // inverse keep probability in its epilogue)
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
            named_bar_signal(kBarP, C::kBarCount, ok);
            // dS^T = P^T (dP^T - D), written back as bf16 in place
            if (ok) ok = warp_wait(smem_addr(&bars->dp_full[0]), n & 1, abort_flag, p.timeout_cycles, p.status);
            if (ok) {
                tc_fence_after();
                float dp[W];
                tmem_ldw<W>(tDP, dp);
                // with dropout dS = P (r keep dZ - D), dZ the product's dP: the dropped
                // columns cleared by their masks, r folded into the multiply-add
                const uint32_t(&km)[W / 4] = *reinterpret_cast<const uint32_t(*)[W / 4]>(dw);
                const uint64_t rr = f2_pack(p.drop.rscale, p.drop.rscale);
#pragma unroll
                for (int c4 = 0; c4 < W / 4; ++c4) {
                    const float4 nd = ndlt4[c4];
                    const int c = 4 * c4;
                    const uint64_t z0 = DROP ? f2_fma(rr, f2_pack(kept<W>(km, dp, c), kept<W>(km, dp, c + 1)), f2_pack(nd.x, nd.y))
                                             : f2_add(f2_pack(dp[c], dp[c + 1]), f2_pack(nd.x, nd.y));
                    const uint64_t z1 = DROP ? f2_fma(rr, f2_pack(kept<W>(km, dp, c + 2), kept<W>(km, dp, c + 3)), f2_pack(nd.z, nd.w))
                                             : f2_add(f2_pack(dp[c + 2], dp[c + 3]), f2_pack(nd.z, nd.w));
                    const float2 a = f2_unpack(f2_mul(f2_pack(pv[c], pv[c + 1]), z0));
                    const float2 e = f2_unpack(f2_mul(f2_pack(pv[c + 2], pv[c + 3]), z1));
                    dp[4 * c4] = a.x;
                    dp[4 * c4 + 1] = a.y;
                    dp[4 * c4 + 2] = e.x;
                    dp[4 * c4 + 3] = e.y;
                }
                tmem_st_pk<W, E>(tDP, dp);
                tmem_st_wait();
                tc_fence_before();
            }
            named_bar_signal(kBarDS0, C::kBarCount, ok);
            if (DROP && ok && n + 1 < nsteps) draw(n + 1);
        }
        if (ok)
            ok = warp_wait(smem_addr(&bars->acc_full), 0, abort_flag, p.timeout_cycles, p.status);
        // The first half of the warpgroups stores dV, the second dK (scaled), each
        // warpgroup kSC columns of the row.  A tile of 128 keys inside the sequence
        // leaves through shared memory (the idle slot ring) and TMA stores, coalesced
        // and asynchronous; a tile cut by the sequence end is stored row by row.
        // The choice is made uniform over the element-wise warps.
        constexpr int kHalf = C::kEwWG / 2;
        constexpr int kSC = D / kHalf;
        const bool is_dk = wg >= kHalf;
        const int c0 = kSC * (wg % kHalf);
        const uint32_t t_acc = tmem + lane_addr + C::kColAcc + (is_dk ? D : 0) + c0;
        const float mul = is_dk ? p.scale : (DROP ? p.drop.rscale : 1.f);   // dV = r (keep P)^T dO
        if (named_bar_all(kBarEpi, C::kEwThreads, ok && kb + kBlockN <= len)) {
            tc_fence_after();
            stage_acc_row<kSC, E>(t_acc, mul, sSlots + (is_dk ? C::kTileBytes : 0), C::kChunkBytes,
                                  r, c0);
            fence_proxy_async_smem();
            named_bar_sync(kBarEpi, C::kEwThreads);
            if (warp == 4 && lane == 0) {
                if (fa_box_ok(seq_start + kb, kBlockN, s.total_tokens, g, s.Hkv, p.status))
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_store_3d(&p.tm_dv, smem_addr(sSlots + c * C::kChunkBytes), c * 64, g,
                                     seq_start + kb);
                        tma_store_3d(&p.tm_dk, smem_addr(sSlots + C::kTileBytes + c * C::kChunkBytes),
                                     c * 64, g, seq_start + kb);
                    }
                bulk_commit_group();
                bulk_wait_read_all();   // the CTA's shared memory outlives the reads
            }
        } else if (ok) {
            tc_fence_after();
            const long long row = (static_cast<long long>(seq_start + kpos) * s.Hkv + g) * D;
            store_acc_row<kSC, E>(t_acc, mul,
                                  static_cast<uint16_t*>(is_dk ? p.dk : p.dv) + row + c0,
                                  kpos < len && fa_index_ok(static_cast<long long>(seq_start + kpos) * s.Hkv + g,
                                                            static_cast<long long>(s.total_tokens) * s.Hkv, p.status));
        }
    }
    teardown_bwd_cta<D>(bars, warp);
}

// ---------------------------------------------------------------------- dQ
//
// Q and dO of the CTA's query tile live in TMEM, as the A operands of S_j = Q K_j^T
// and dP_j = dO V_j^T.  Shared memory holds one slot ring (7 slots at d = 128: 5 for
// even items, 2 for odd ones; 10 at d = 64: 7 and 3).  Per query head it streams Q
// and dO (items 0 and 1, whole tiles by TMA), then K_j and V_j as items 2 + 2j and
// 3 + 2j.  The element-wise warps copy their rows of Q and dO from the ring into TMEM
// (whole-tile loads, then conflict-free reads of the swizzled rows: a warp-wide load
// of 32 scattered rows from global memory took about 3 us per tile) and the issuer
// hands the two slots back.  K_j is held from S_j to dQ_j, about one and a half
// steps, and the deeper even ring lets its load start well before it is needed.
//
// Per key tile j: as soon as the element-wise warps have read S_j into registers the
// issuer runs S_{j+1}; when dS_j is back in TMEM (over dP_j) it runs dQ += dS_j K_j
// and then dP_{j+1} into the same columns (tcgen05 ops of one thread execute in issue
// order, so dQ_j has read dS_j first).  V_j's slot is released after dP_j, K_j's
// after dQ_j.  Every signal waits for its waiter's previous phase: S_{j+1} needs S_j
// read, dP_{j+1} needs dS_j written, so no mbarrier or named barrier runs two phases
// ahead.
//
// A CTA may serve several query heads of one key/value group (p.dq_heads, chosen
// at launch so that enough CTAs remain): their K/V tiles are the same, so the ring
// streams them head after head without a break and the CTA's fixed costs (barrier
// set-up, TMEM allocation, the first loads) are paid once.  Steps are counted over
// all heads (J = t nk + j for head t), ring items too (2 nk + 2 per head), and so are
// the mbarrier phases.  Head t+1's Q and dO go into TMEM once acc_full has shown that
// every product of head t is complete; its first dQ product overwrites the
// accumulator only after all element-wise warps have passed head t's epilogue (they
// signal dS_0 of head t+1 after it).  Only the last head's epilogue stages through the
// ring's shared memory, which is idle by then; earlier heads store their dQ rows
// directly.

template <int D, int E, bool DROP, bool HL>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdCfg<D>;
    using R = Ring<C::kSlotsDq, C::kSlotsOddDq>;   // Q and K_j (even), dO and V_j (odd)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Launched as a programmatic dependent of the dK/dV kernel: it may start while
    // that grid finishes.  Before exiting, every CTA waits for that grid, so the
    // completion of this kernel still implies the completion of all earlier work.
    struct WaitPrimaryOnExit {
        __device__ ~WaitPrimaryOnExit() { grid_dependency_wait(); }
    } wait_on_exit;
    if (!smem_base_ok(smem_raw, p.status)) return;
    const SeqInfo& s = p.seq;
    // query heads of this CTA (a divisor of the group); the instances without the heads
    // loop fix it at one at compile time
    static_assert(!(HL && DROP), "the heads loop serves the backward without dropout");
    const int hpc = HL ? p.dq_heads : 1;
    int b, hc, qblk;
    if (!map_work(s, blockIdx.x, kBlockM, s.Hq / hpc, true, b, hc, qblk)) return;
    int seq_start, len;
    seq_bounds(s, b, seq_start, len);
    const int h0 = hc * hpc;      // first query head
    const int g = h0 / s.group;
    const int q0 = qblk * kBlockM;
    const int q_last = min(q0 + kBlockM - 1, len - 1);
    const int kt_first = max(key_lo(s, q0), 0) / kBlockN;
    const int kt_last = key_hi(s, q_last, len) / kBlockN;
    const int nk = kt_last - kt_first + 1;
    const int steps = hpc * nk;   // key-tile steps over all heads of the CTA
    // ring items per head: Q, dO, then K_j, V_j; K_j of head t is item k_item(t, j)
    const int P = 2 * nk + 2;
    auto k_item = [&](int t, int j) { return t * P + 2 + 2 * j; };

    BwdBars* bars = reinterpret_cast<BwdBars*>(smem_raw);
    uint8_t* sSlots = smem_raw + C::kHeadBytes;
    volatile int* abort_flag = &bars->abort;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    init_bwd_cta<D>(bars, warp, C::kSlotsDq);
    const uint32_t tmem = bars->tmem_base;
    constexpr int kOperandBar = C::kEwThreads + 32;   // element-wise warps + the issuer

    if (warp == 0) {
        regs_lower<C::kRegsCtl>();
        if (lane == 0)
            stream_tiles<D, R>(bars, sSlots, P * hpc, &p.tm_k, &p.tm_v,
                               [&](int i, int& head, int& row) -> const CUtensorMap* {
                                   const int t = i / P, k = i % P;
                                   if (k < 2) {            // Q and dO of query head t
                                       head = h0 + t;
                                       row = seq_start + q0;
                                       return k == 0 ? &p.tm_q : &p.tm_do;
                                   }
                                   head = g;
                                   row = seq_start + (kt_first + (k - 2) / 2) * kBlockN;
                                   // with head t's first K tile, head t+1's Q and dO tiles
                                   // into L2, so that their ring loads are short
                                   if (k == 2 && t + 1 < hpc)
                                       for (int c = 0; c < C::kChunks; ++c) {
                                           tma_prefetch_l2_3d(&p.tm_q, c * 64, h0 + t + 1, seq_start + q0);
                                           tma_prefetch_l2_3d(&p.tm_do, c * 64, h0 + t + 1, seq_start + q0);
                                       }
                                   return nullptr;         // K_j (even) or V_j (odd)
                               },
                               abort_flag, p, false);
    } else if (warp == 1) {
        regs_lower<C::kRegsCtl>();
        // ------------------------------------------------------ MMA issuer
        // (whole warp walks the tiles, lane 0 issues; as in the dK/dV kernel it
        // never waits on an mbarrier inside the loop)
        auto slot = [&](int i) { return smem_addr(sSlots + R::index(i) * C::kTileBytes); };
        auto free_slot = [&](int i) { mma_commit(smem_addr(&bars->slot_empty[R::index(i)])); };
        const uint32_t tQ = tmem + C::kColQ, tDO = tmem + C::kColDO, tDP = tmem + C::kColDP;
        auto wait = [&](int i) {
            return mbar_wait(smem_addr(&bars->slot_full[R::index(i)]), R::use(i) & 1, abort_flag,
                             p.timeout_cycles, p.status);
        };
        for (int t = 0; t < hpc; ++t) {
            named_bar_sync(kBarOperands, kOperandBar);    // Q and dO of head t are in TMEM
            if (lane == 0) {
                // the element-wise warps read Q and dO from their slots before the
                // barrier: the slots go back to the producer
                mbar_arrive(smem_addr(&bars->slot_empty[R::index(t * P)]));
                mbar_arrive(smem_addr(&bars->slot_empty[R::index(t * P + 1)]));
                const int k0 = k_item(t, 0);
                if (wait(k0) && wait(k0 + 1)) {}
                tc_fence_after();
                issue_ts_k<D, E>(tmem + C::kColS, tQ, slot(k0));        // S_0 = Q K_0^T
                mma_commit(smem_addr(&bars->s_full));
                issue_ts_k<D, E>(tDP, tDO, slot(k0 + 1));               // dP_0 = dO V_0^T
                mma_commit(smem_addr(&bars->dp_full[0]));
                free_slot(k0 + 1);
            }
            __syncwarp();
            for (int j = 0; j < nk; ++j) {
                const int kj = k_item(t, j);                    // K_j; V_j is kj + 1
                named_bar_sync(kBarP, C::kBarCount);            // S_j read, K_{j+1} landed
                if (lane == 0 && j + 1 < nk) {
                    tc_fence_after();
                    issue_ts_k<D, E>(tmem + C::kColS, tQ, slot(kj + 2));   // S_{j+1}
                    mma_commit(smem_addr(&bars->s_full));
                }
                __syncwarp();
                named_bar_sync(kBarDS0, C::kBarCount);          // dS_j written, V_{j+1} landed
                if (lane == 0) {
                    tc_fence_after();
                    issue_ts<D, E>(tmem + C::kColAcc, tDP, slot(kj), j > 0);   // dQ += dS_j K_j
                    free_slot(kj);
                    if (j + 1 < nk) {
                        issue_ts_k<D, E>(tDP, tDO, slot(kj + 3));   // dP_{j+1}, after dQ_j read dS_j
                        mma_commit(smem_addr(&bars->dp_full[0]));
                        free_slot(kj + 3);
                    }
                }
                __syncwarp();
            }
            if (lane == 0) mma_commit(smem_addr(&bars->acc_full));   // head t's products done
        }
    } else if (warp == 2) {
        regs_lower<C::kRegsCtl>();
        // ------------------------------------------------------ slot relay
        auto wait_item = [&](int i) {
            mbar_wait(smem_addr(&bars->slot_full[R::index(i)]), R::use(i) & 1, abort_flag,
                      p.timeout_cycles, p.status);
        };
        for (int J = 0; J < steps; ++J) {
            const int t = J / nk, j = J % nk;
            const bool more = j + 1 < nk;                        // head t has a next tile
            if (lane == 0 && more) wait_item(k_item(t, j + 1));      // K_{j+1}
            __syncwarp();
            named_bar_sync(kBarP, C::kBarCount);
            if (lane == 0 && more) wait_item(k_item(t, j + 1) + 1);  // V_{j+1}
            __syncwarp();
            named_bar_sync(kBarDS0, C::kBarCount);
        }
    } else if (warp == 3) {
        regs_lower<C::kRegsCtl>();   // idle; its warpgroup gives registers away
    } else if (warp >= 4) {
        regs_raise<C::kRegsEw>();
        constexpr int W = C::kEwCols;
        const int wg = (warp - 4) / 4;      // key columns [W wg, W wg + W) of each tile
        const int quad = warp % 4;
        const int r = quad * 32 + lane;     // query row within the tile = TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_addr + C::kColS + W * wg;
        const uint32_t tDP = tmem + lane_addr + C::kColDP + W * wg;
        const int q = q0 + r;
        const bool valid = q < len;
        const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
        const int lo_q = key_lo(s, q), hi_q = valid ? key_hi(s, q, len) : -1;
        // The warpgroups share the dQ row store: kSC (>= 32) columns each, as far as it
        // goes.
        constexpr int kSC = (D / C::kEwWG >= 32) ? D / C::kEwWG : 32;
        const bool mine = wg * kSC < D;
        const uint32_t t_acc = tmem + lane_addr + C::kColAcc + kSC * wg;
        // `ok`: as in the dK/dV kernel, a warp that gave up keeps taking part in
        // every named-barrier phase
        bool ok = true;
        for (int t = 0; t < hpc; ++t) {
            const int h = h0 + t;
            {
                // Q and dO of row q into TMEM, two elements per 32-bit column as they lie
                // in memory (the A-operand layout of S and dP), from their ring slots: each
                // warpgroup copies kQW of the D/2 columns, whole 16-byte units of the
                // 128-byte-swizzled row; rows past the sequence end are zero.  For t > 0
                // the previous head's products are complete (acc_full, below).
                constexpr int kQW = D / 2 / C::kEwWG;   // 32 (d = 128) or 16 (d = 64)
                static_assert(kQW % 4 == 0 && 4 * kQW <= 128, "whole units of one 64-column chunk");
                uint32_t wq[kQW], wd[kQW];
#pragma unroll
                for (int i = 0; i < kQW; ++i) wq[i] = wd[i] = 0u;
                const int qi = t * P;                   // Q's item; dO's is qi + 1
                if (ok) ok = warp_wait(smem_addr(&bars->slot_full[R::index(qi)]), R::use(qi) & 1,
                                       abort_flag, p.timeout_cycles, p.status);
                if (ok) ok = warp_wait(smem_addr(&bars->slot_full[R::index(qi + 1)]), R::use(qi + 1) & 1,
                                       abort_flag, p.timeout_cycles, p.status);
                if (ok && valid) {
                    const int byte0 = 4 * kQW * wg;     // this warpgroup's first byte of the row
                    const int off = (byte0 / 128) * C::kChunkBytes;
                    const int u0 = (byte0 % 128) / 16;
                    uint8_t* tq = sSlots + R::index(qi) * C::kTileBytes + off;
                    uint8_t* td = sSlots + R::index(qi + 1) * C::kTileBytes + off;
#pragma unroll
                    for (int i = 0; i < kQW / 4; ++i) {
                        const uint4 a = *swizzled_unit(tq, r, u0 + i), c = *swizzled_unit(td, r, u0 + i);
                        wq[4 * i] = a.x; wq[4 * i + 1] = a.y; wq[4 * i + 2] = a.z; wq[4 * i + 3] = a.w;
                        wd[4 * i] = c.x; wd[4 * i + 1] = c.y; wd[4 * i + 2] = c.z; wd[4 * i + 3] = c.w;
                    }
                }
                tmem_st_words<kQW>(tmem + lane_addr + C::kColQ + kQW * wg, wq);
                tmem_st_words<kQW>(tmem + lane_addr + C::kColDO + kQW * wg, wd);
                tmem_st_wait();
                tc_fence_before();
                named_bar_arrive(kBarOperands, kOperandBar);
            }
            float lse2 = kPosInf, dlt = 0.f;
            if (valid && fa_index_ok(row_stat_index(s, b, h, seq_start, q),
                                     static_cast<long long>(s.total_tokens) * s.Hq, p.status)) {
                const long long idx = row_stat_index(s, b, h, seq_start, q);
                lse2 = __ldg(p.lse + idx) * kLog2eF;
                dlt = __ldg(p.delta + idx);
            }
            const uint64_t nlse2 = f2_pack(-lse2, -lse2), ndlt2 = f2_pack(-dlt, -dlt);
            // dropout bytes of this query row for the current key tile, 4 keys a word; as
            // in the dK/dV kernel the next tile's are drawn at the end of each step
            uint32_t dw[DROP ? W / 4 : 1];
            auto draw = [&](int j) {
                dropout_words_rows<W / 4>(*reinterpret_cast<uint32_t(*)[W / 4]>(dw), q >> 2,
                                          ((kt_first + j) * kBlockN + W * wg) >> 2,
                                          static_cast<uint32_t>(b * s.Hq + h), p.drop.offset,
                                          p.drop.seed_lo, p.drop.seed_hi, lane);
                keep_masks(*reinterpret_cast<uint32_t(*)[W / 4]>(dw), p.drop.thresh);
            };
            if (DROP) draw(0);
            for (int j = 0; j < nk; ++j) {
                const int J = t * nk + j;                               // step over all heads
                const int kc = (kt_first + j) * kBlockN + W * wg;      // first key of my columns
                const bool need_mask = !(kc >= lo_q && kc + W - 1 <= hi_q);
                const int clo = lo_q - kc, chi = hi_q - kc;
                if (ok) ok = warp_wait(smem_addr(&bars->s_full), J & 1, abort_flag, p.timeout_cycles, p.status);
                float pv[W];
                if (ok) {
                    tc_fence_after();
                    tmem_ldw<W>(tS, pv);
                    tc_fence_before();
                }
                named_bar_signal(kBarP, C::kBarCount, ok);   // S_j consumed: the next S may be issued
                if (ok) {
#pragma unroll
                    for (int i = 0; i < W / 2; ++i) {
                        const float2 a = f2_unpack(f2_fma(f2_pack(pv[2 * i], pv[2 * i + 1]), sl2x2, nlse2));
                        pv[2 * i] = ex2_approx(a.x);
                        pv[2 * i + 1] = ex2_approx(a.y);
                    }
                    if (need_mask) {
#pragma unroll
                        for (int c = 0; c < W; ++c)
                            if (c < clo || c > chi) pv[c] = 0.f;
                    }
                    ok = warp_wait(smem_addr(&bars->dp_full[0]), J & 1, abort_flag, p.timeout_cycles,
                                   p.status);
                }
                if (ok) {
                    tc_fence_after();
                    float dp[W];
                    tmem_ldw<W>(tDP, dp);
                    // with dropout dS = P (r keep dZ - D), as in the dK/dV kernel
                    const uint32_t(&km)[W / 4] = *reinterpret_cast<const uint32_t(*)[W / 4]>(dw);
                    const uint64_t rr = f2_pack(p.drop.rscale, p.drop.rscale);
#pragma unroll
                    for (int i = 0; i < W / 2; ++i) {
                        const uint64_t z = DROP ? f2_fma(rr, f2_pack(kept<W>(km, dp, 2 * i), kept<W>(km, dp, 2 * i + 1)), ndlt2)
                                                : f2_add(f2_pack(dp[2 * i], dp[2 * i + 1]), ndlt2);
                        const float2 a = f2_unpack(f2_mul(f2_pack(pv[2 * i], pv[2 * i + 1]), z));
                        dp[2 * i] = a.x;
                        dp[2 * i + 1] = a.y;
                    }
                    tmem_st_pk<W, E>(tDP, dp);
                    tmem_st_wait();
                    tc_fence_before();
                }
                named_bar_signal(kBarDS0, C::kBarCount, ok);
                if (DROP && ok && j + 1 < nk) draw(j + 1);
            }
            if (ok)
                ok = warp_wait(smem_addr(&bars->acc_full), t & 1, abort_flag, p.timeout_cycles, p.status);
            // The last head's whole query tile leaves through shared memory (the ring is
            // idle once every product is complete) and TMA stores; an earlier head's, while
            // the ring streams the next head's tiles, and a tile cut by the sequence end,
            // row by row (see the dK/dV epilogue).
            if (t == hpc - 1 && named_bar_all(kBarEpi, C::kEwThreads, ok && q0 + kBlockM <= len)) {
                if (mine) {
                    tc_fence_after();
                    stage_acc_row<kSC, E>(t_acc, p.scale, sSlots, C::kChunkBytes, r, kSC * wg);
                }
                fence_proxy_async_smem();
                named_bar_sync(kBarEpi, C::kEwThreads);
                if (warp == 4 && lane == 0) {
                    if (fa_box_ok(seq_start + q0, kBlockM, s.total_tokens, h, s.Hq, p.status))
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_store_3d(&p.tm_dq, smem_addr(sSlots + c * C::kChunkBytes), c * 64, h,
                                         seq_start + q0);
                    bulk_commit_group();
                    bulk_wait_read_all();
                }
            } else if (ok && mine) {
                tc_fence_after();
                const long long row = (static_cast<long long>(seq_start + q) * s.Hq + h) * D;
                store_acc_row<kSC, E>(t_acc, p.scale, static_cast<uint16_t*>(p.dq) + row + kSC * wg,
                                      valid && fa_index_ok(static_cast<long long>(seq_start + q) * s.Hq + h,
                                                           static_cast<long long>(s.total_tokens) * s.Hq,
                                                           p.status));
            }
        }
    }
    teardown_bwd_cta<D>(bars, warp);
}

}  // namespace

int bwd_preprocess_row_ctas(const BwdParams& p, int d) {
    const long long rows = static_cast<long long>(p.seq.total_tokens) * p.seq.Hq;
    const int per_cta = d == 128 ? pre_rows_per_cta<128>() : pre_rows_per_cta<64>();
    return static_cast<int>((rows + per_cta - 1) / per_cta);
}

cudaError_t launch_bwd_preprocess(const BwdParams& p, int d, cudaStream_t stream) {
    // row CTAs (p.pre_row_ctas of them, from bwd_preprocess_row_ctas), then for the
    // fused backward the K/V bound CTAs
    const int grid = p.pre_row_ctas + (p.dq_acc ? p.seq.Hkv * kBoundSlots : 0);
    if (p.pre_row_ctas <= 0) return cudaSuccess;
    const bool f16 = p.elem == kElemF16;
    if (d == 128) {
        if (f16) fa_bwd_preprocess_kernel<128, kElemF16><<<grid, kPreThreads, 0, stream>>>(p);
        else fa_bwd_preprocess_kernel<128, kElemBf16><<<grid, kPreThreads, 0, stream>>>(p);
    } else {
        if (f16) fa_bwd_preprocess_kernel<64, kElemF16><<<grid, kPreThreads, 0, stream>>>(p);
        else fa_bwd_preprocess_kernel<64, kElemBf16><<<grid, kPreThreads, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

template <int D, int E, bool DROP>
cudaError_t launch_bwd_dkdv_d(const BwdParams& p, cudaStream_t stream) {
    static const cudaError_t regs_ok = check_regs(fa_bwd_dkdv_kernel<D, E, DROP>, BwdCfg<D>::kRegsLaunch);
    if (regs_ok != cudaSuccess) return regs_ok;
    return launch_tc(fa_bwd_dkdv_kernel<D, E, DROP>, p.num_work_dkdv, BwdCfg<D>::kThreads,
                     BwdCfg<D>::kSmemBytes, p, stream);
}

template <int D, int E>
cudaError_t launch_bwd_dkdv_de(const BwdParams& p, cudaStream_t stream) {
    return p.drop.thresh ? launch_bwd_dkdv_d<D, E, true>(p, stream) : launch_bwd_dkdv_d<D, E, false>(p, stream);
}

cudaError_t launch_bwd_dkdv(const BwdParams& p, int d, cudaStream_t stream) {
    if (p.num_work_dkdv <= 0) return cudaSuccess;
    if (p.elem == kElemF16)
        return d == 128 ? launch_bwd_dkdv_de<128, kElemF16>(p, stream) : launch_bwd_dkdv_de<64, kElemF16>(p, stream);
    return d == 128 ? launch_bwd_dkdv_de<128, kElemBf16>(p, stream) : launch_bwd_dkdv_de<64, kElemBf16>(p, stream);
}

// The dQ kernel is launched as a programmatic dependent of the dK/dV kernel
// (see fa_bwd_dq_kernel).
template <typename K>
cudaError_t launch_dependent(K kern, int grid, int threads, int smem, const BwdParams& p,
                             cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int D, int E, bool DROP, bool HL>
cudaError_t launch_bwd_dq_d(const BwdParams& p, cudaStream_t stream) {
    static const cudaError_t regs_ok = check_regs(fa_bwd_dq_kernel<D, E, DROP, HL>, BwdCfg<D>::kRegsLaunch);
    if (regs_ok != cudaSuccess) return regs_ok;
    return launch_dependent(fa_bwd_dq_kernel<D, E, DROP, HL>, p.num_work_dq, BwdCfg<D>::kThreads,
                            BwdCfg<D>::kSmemBytes, p, stream);
}

template <int D, int E>
cudaError_t launch_bwd_dq_de(const BwdParams& p, cudaStream_t stream) {
    if (p.drop.thresh) return launch_bwd_dq_d<D, E, true, false>(p, stream);
    return p.dq_heads > 1 ? launch_bwd_dq_d<D, E, false, true>(p, stream)
                          : launch_bwd_dq_d<D, E, false, false>(p, stream);
}

cudaError_t launch_bwd_dq(const BwdParams& p, int d, cudaStream_t stream) {
    if (p.num_work_dq <= 0) return cudaSuccess;
    if (p.elem == kElemF16)
        return d == 128 ? launch_bwd_dq_de<128, kElemF16>(p, stream) : launch_bwd_dq_de<64, kElemF16>(p, stream);
    return d == 128 ? launch_bwd_dq_de<128, kElemBf16>(p, stream) : launch_bwd_dq_de<64, kElemBf16>(p, stream);
}

}  // namespace fa
