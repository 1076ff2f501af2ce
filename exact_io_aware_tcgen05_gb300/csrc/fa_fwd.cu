// fa_fwd.cu -- forward pass of exact attention on sm_103a.
//
// Computes, per query row i, O_i = sum_j softmax_j(scale * q_i . k_j) v_j over
// the visible keys and LSE_i = ln sum_j exp(scale * q_i . k_j), tile by tile,
// without writing the score matrix anywhere.  The block loop is the online
// softmax of "FlashAttention: How IO-Aware Tiling and Online Softmax Solved
// Transformer Memory Bottlenecks" (section "1. IO-Aware Tiling": a query block
// stays on chip while key/value blocks stream past; section "2. Online Softmax
// Reduction": running max m, running normaliser l, rescale of the partial
// output by exp(m_old - m_new), final division by l).  The saved statistic is
// the logsumexp of "Flash Attention -- Fast Memory-Efficient Exact Attention"
// ("Architecture Overview").
//
// One CTA owns 256 query rows of one (sequence, head) as two 128-row tiles and
// streams the 128-key K/V tiles they need:
//   warp 0        TMA producer: both Q tiles once, then K_j, V_j into a ring
//   warp 1        tcgen05 issuer (lane 0 issues); owns the TMEM allocation
//   warp 2        relay: waits for the K/V tiles the next products read
//   warps 4..7    softmax + epilogue of query tile 0 (one TMEM lane = one row)
//   warps 8..11   softmax + epilogue of query tile 1
// TMEM (512 columns): S_0 [0,128)  S_1 [128,256)  O_0 and O_1 (D columns each)
// from 256.  P_t (bf16 or fp16, the input type; e4m3 in the fp8 instance, four
// keys per column) overwrites the first 64 (32) columns of S_t and feeds the
// P.V product straight from TMEM.  The fp8 instance runs both products as
// kind::f8f6f4 on e4m3 Q, K and transposed V, with the Q and K block scales
// folded into the exponent scale and V's scale into 1/l.  The issuer interleaves the two tiles so the
// tensor cores work on one tile while the softmax warps work on the other:
//   S0=Q0K0 S1=Q1K0 | O0+=P0V0 S0=Q0K1 | O1+=P1V0 S1=Q1K1 | O0+=P0V1 ...
// Scores are kept in log2 units (scale * log2 e folded in) and exponentiated
// with ex2.  The running max used for exponentiation is only raised when the
// block max exceeds it by more than 8 (a factor 256); O and l always share
// that reference, so the result is exact and most blocks skip the O rescale.
//
// The issuer hears from the softmax warps (and, through the relay warp, from
// the K/V ring) by named barriers, one per query tile and one phase per key
// block: an mbarrier wait is a shared-memory load, and one by the issuing warp
// would hold back its next MMAs until those in flight drained.  The softmax
// warps hear from the issuer by tcgen05.commit mbarriers.  The signal opening
// phase j+1 of tile t's barrier needs S_t(j+1), issued after phase j completed,
// so no one runs a phase ahead.
#include "fa_kernels.h"
#include "fa_ptx.cuh"
#include "fa_seq.cuh"


namespace fa {
static_assert(kElemBf16 == kElemBf16Code && kElemF16 == kElemF16Code && kElemFp8 == kElemFp8Code,
              "element-type codes");
namespace {

// E: element type of the operands (kElemBf16, kElemF16, or kElemFp8: e4m3 Q, K and
// transposed V, bf16 O)
template <int D, int E>
struct FwdCfg {
    static constexpr bool kF8 = (E == kElemFp8);
    static constexpr int kElemBytes = kF8 ? 1 : 2;
    static constexpr int kChunks = D * kElemBytes / 128;   // 128-byte swizzle column blocks
    static constexpr int kChunkElems = 128 / kElemBytes;
    static constexpr int kChunkBytes = kBlockM * 128;      // 128 rows x 128 bytes
    static constexpr int kTileBytes = kBlockM * D * kElemBytes;
    static constexpr int kOTileBytes = kBlockM * D * 2;    // a 16-bit output tile
    static constexpr int kOChunks = D / 64;
    static constexpr int kStages = (kTileBytes == 32768) ? 4 : 8;   // K/V ring depth
    static_assert(2 * kOTileBytes <= kStages * kTileBytes, "output staging in the ring");
    static constexpr int kThreads = 384;
    static constexpr int kTmemCols = 512;
    static constexpr int kColS = 0;                        // S_t at kColS + 128 t
    static constexpr int kColO = 256;                      // O_t at kColO + D t
    static constexpr int kTilesBytes = (kFwdQTiles + kStages) * kTileBytes;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmemBytes = kTilesBytes + kBarBytes + 1024;  // + alignment slack
    // dropout only: the random words of each softmax row for its next key block
    // (32 words per row of 128 keys), after the barrier block
    static constexpr int kDropBytes = kFwdQTiles * kBlockM * (kBlockN / 4) * 4;
    static constexpr int kSmemBytesDrop = kSmemBytes + kDropBytes;
    static_assert(kSmemBytesDrop <= 232448, "shared memory per CTA");
};

// Registers per thread: the kernel is built for 384 threads at 168 (one CTA per
// SM); at the start the warpgroup of warps 0..3 (producer, issuer, relay, idle)
// drops to kFwdRegsCtl and the two softmax warpgroups rise to kFwdRegsSoftmax,
// which keeps a row of 128 scores and its P in registers without spilling.
constexpr int kFwdRegsLaunch = 168;
constexpr int kFwdRegsCtl = 152;
constexpr int kFwdRegsSoftmax = 176;
static_assert(128 * kFwdRegsCtl + 256 * kFwdRegsSoftmax <= 384 * kFwdRegsLaunch,
              "register split exceeds the launch's registers");

// named barrier of query tile t: kFwdBarP + t (0 is __syncthreads); softmax
// warpgroup t + issuer warp + relay warp
constexpr int kFwdBarP = 1;
constexpr int kFwdBarCount = kBlockM + 64;
constexpr int kFwdBarEpi = 3;   // + t: softmax warpgroup t among itself, the epilogue

struct FwdBars {
    uint64_t q_full;
    uint64_t q_empty;   // heads loop: the head's last Q K^T products are complete
    uint64_t s_full[kFwdQTiles];
    uint64_t o_full;
    uint64_t kv_full[8];
    uint64_t kv_empty[8];
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(FwdBars) <= 256, "barrier block");

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// E: element type of q, k, v and o (kElemBf16 or kElemF16); DROP: dropout of P; HL: the
// CTA serves p.heads consecutive query heads in turn (16-bit, no dropout).  The ring
// streams each head's K/V tiles after the previous head's (the same tiles, read again
// from L2, for the heads of one key/value group) and the CTA's fixed costs (set-up, the
// first loads, the exit) are paid once.  Ring items, S and O
// phases are counted over all the CTA's heads.  Head t+1's Q tiles load once q_empty
// shows head t's last Q K^T complete; its first P V overwrites O only after the
// softmax warps have left head t's epilogue (they hand P of head t+1 over after it).
// Only the last head's O tiles leave through the ring's shared memory; the earlier
// ones are stored row by row, because the ring is then streaming the next head's tiles.
template <int D, int E, bool DROP, bool HL>
__global__ void __launch_bounds__(384, 1) fa_fwd_kernel(const __grid_constant__ FwdParams p) {
    using C = FwdCfg<D, E>;
    constexpr bool F8 = C::kF8;
    constexpr int EO = F8 ? kElemBf16 : E;   // element type of O
    static_assert(!(F8 && (DROP || D != 128)), "the fp8 forward: d = 128, no dropout");
    constexpr uint32_t kIdescQK = idesc_f32acc(kBlockM, kBlockN, false, false, E);
    // fp8: V^T tiles, K-major like K; 16-bit: V tiles read MN-major
    constexpr uint32_t kIdescPV = idesc_f32acc(kBlockM, D, false, !F8, E);
    const SeqInfo& s = p.seq;
    static_assert(!HL || (!F8 && !DROP), "the heads loop serves the 16-bit forward without dropout");
    const int hpc = HL ? p.heads : 1;   // query heads of this CTA (a divisor of the group)

    int b, hc, qblk;
    if (!map_work(s, blockIdx.x, kFwdQTiles * kBlockM, s.Hq / hpc, true, b, hc, qblk, p.head_chunk))
        return;
    int seq_start, len;
    seq_bounds(s, b, seq_start, len);
    const int h0 = hc * hpc;            // first query head
    const int g = h0 / s.group;
    const int q0 = qblk * kFwdQTiles * kBlockM;  // first query row of the CTA (in-sequence)
    const int q_last = min(q0 + kFwdQTiles * kBlockM - 1, len - 1);
    const int kv_first = max(key_lo(s, q0), 0) / kBlockN;
    const int kv_last = key_hi(s, q_last, len) / kBlockN;
    const int nkv = kv_last - kv_first + 1;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;                                   // [2][tile]
    uint8_t* sKV = smem + kFwdQTiles * C::kTileBytes;     // [stages][tile]
    FwdBars* bars = reinterpret_cast<FwdBars*>(smem + C::kTilesBytes);
    volatile int* abort_flag = &bars->abort;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        bars->abort = 0;
        mbar_init(smem_addr(&bars->q_full), 1);
        mbar_init(smem_addr(&bars->q_empty), 1);
        mbar_init(smem_addr(&bars->o_full), 1);
        for (int t = 0; t < kFwdQTiles; ++t) {
            mbar_init(smem_addr(&bars->s_full[t]), 1);
        }
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(smem_addr(&bars->kv_full[i]), 1);
            mbar_init(smem_addr(&bars->kv_empty[i]), 1);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&bars->tmem_base), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        regs_lower<kFwdRegsCtl>();
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            const uint64_t keep = make_l2_policy_evict_last();
            const uint32_t qbar = smem_addr(&bars->q_full);
            // fp8: V^T rows are the d dimension, columns this sequence's keys from
            // its padded start (a multiple of 128, so the TMA x coordinate is aligned)
            const int vt_col = F8 ? 128 * seq_block_col(s, b) : 0;
            int issued = 0, q_issued = 0;   // ring items (over all heads), Q loads
            bool stop = false;
            for (int hd = 0; hd < hpc && !stop; ++hd) {
                if (hd > 0 && !mbar_wait(smem_addr(&bars->q_empty), (hd - 1) & 1, abort_flag,
                                         p.timeout_cycles, p.status))
                    break;
                mbar_arrive_expect_tx(qbar, kFwdQTiles * C::kTileBytes);
                for (int t = 0; t < kFwdQTiles; ++t)
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(smem_addr(sQ + t * C::kTileBytes + c * C::kChunkBytes), &p.tm_q,
                                    qbar, c * C::kChunkElems, h0 + hd, seq_start + q0 + t * kBlockM);
                q_issued = hd + 1;
                for (int i = 0; i < 2 * nkv; ++i) {
                    const int ig = hd * 2 * nkv + i;
                    const int st = ig % C::kStages, use = ig / C::kStages;
                    if (use > 0 && !mbar_wait(smem_addr(&bars->kv_empty[st]), (use - 1) & 1,
                                              abort_flag, p.timeout_cycles, p.status)) {
                        stop = true;
                        break;
                    }
                    const uint32_t fb = smem_addr(&bars->kv_full[st]);
                    mbar_arrive_expect_tx(fb, C::kTileBytes);
                    const CUtensorMap* map = (i & 1) ? &p.tm_v : &p.tm_k;
                    const int row = seq_start + (kv_first + i / 2) * kBlockN;
                    const int gh = (h0 + hd) / s.group;   // this head's key/value head
                    if (F8 && (i & 1))
                        tma_load_3d_hint(smem_addr(sKV + st * C::kTileBytes), map, fb,
                                         vt_col + (kv_first + i / 2) * kBlockN, 0, gh, keep);
                    else
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_3d_hint(smem_addr(sKV + st * C::kTileBytes + c * C::kChunkBytes),
                                             map, fb, c * C::kChunkElems, gh, row, keep);
                    issued = ig + 1;
                }
            }
            if (*abort_flag) {
                // let copies already in flight land before the CTA exits
                if (q_issued > 0) mbar_wait_drain(qbar, (q_issued - 1) & 1, kDrainCycles);
                for (int i = max(0, issued - C::kStages); i < issued; ++i)
                    mbar_wait_drain(smem_addr(&bars->kv_full[i % C::kStages]),
                                    (i / C::kStages) & 1, kDrainCycles);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        regs_lower<kFwdRegsCtl>();
        // The whole warp walks the blocks (named barriers are warp-collective);
        // lane 0 issues.  No mbarrier wait and no look at the abort flag inside
        // the loop: after an abort it keeps issuing on stale data, so every
        // barrier phase still completes.
        auto kv_stage = [&](int i) { return i % C::kStages; };
        auto issue_qk = [&](int t, int st) {
            // descriptor of the tile base; a k-step adds its byte offset >> 4
            const uint64_t qd = sdesc_sw128(smem_addr(sQ + t * C::kTileBytes), 16, 1024);
            const uint64_t kd = sdesc_sw128(smem_addr(sKV + st * C::kTileBytes), 16, 1024);
            if constexpr (F8) {
                // one 128-byte chunk per row; K = 32 e4m3 (32 bytes) per product
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk)
                    mma_ss_f8(tmem + C::kColS + t * kBlockN, qd + 2 * kk, kd + 2 * kk, kIdescQK, kk > 0);
            } else {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk / 4) * C::kChunkBytes + (kk % 4) * 32) >> 4;
                    mma_ss(tmem + C::kColS + t * kBlockN, qd + off, kd + off, kIdescQK, kk > 0);
                }
            }
        };
        auto issue_pv = [&](int t, int st, bool acc) {
            if constexpr (F8) {
                // P_t: 4 e4m3 per TMEM column, 32 keys (8 columns) per product; V^T K-major
                const uint64_t vd = sdesc_sw128(smem_addr(sKV + st * C::kTileBytes), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kBlockN / 32; ++kk)
                    mma_ts_f8(tmem + C::kColO + t * D, tmem + C::kColS + t * kBlockN + kk * 8,
                              vd + 2 * kk, kIdescPV, (acc || kk > 0) ? 1u : 0u);
            } else {
                const uint64_t vd = sdesc_sw128(smem_addr(sKV + st * C::kTileBytes),
                                                C::kChunkBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk) {
                    mma_ts(tmem + C::kColO + t * D, tmem + C::kColS + t * kBlockN + kk * 8,
                           vd + ((kk * 2048) >> 4), kIdescPV, (acc || kk > 0) ? 1u : 0u);
                }
            }
        };
        for (int hd = 0; hd < hpc; ++hd) {
            const int base = hd * 2 * nkv;   // ring item of this head's K_0
            if (lane == 0) {
                if (mbar_wait(smem_addr(&bars->q_full), hd & 1, abort_flag, p.timeout_cycles, p.status))
                    mbar_wait(smem_addr(&bars->kv_full[kv_stage(base)]), (base / C::kStages) & 1,
                              abort_flag, p.timeout_cycles, p.status);
                tc_fence_after();
                for (int t = 0; t < kFwdQTiles; ++t) {
                    issue_qk(t, kv_stage(base));
                    mma_commit(smem_addr(&bars->s_full[t]));
                }
                mma_commit(smem_addr(&bars->kv_empty[kv_stage(base)]));
                if (HL && nkv == 1) mma_commit(smem_addr(&bars->q_empty));   // Q is free
            }
            __syncwarp();
            for (int j = 0; j < nkv; ++j) {
                const int iv = base + 2 * j + 1, ik = base + 2 * j + 2;
                for (int t = 0; t < kFwdQTiles; ++t) {
                    named_bar_sync(kFwdBarP + t, kFwdBarCount);   // P_t(j) written (V_j, K_{j+1} landed)
                    if (lane == 0) {
                        tc_fence_after();
                        issue_pv(t, kv_stage(iv), j > 0);
                        if (j + 1 < nkv) {
                            issue_qk(t, kv_stage(ik));
                            mma_commit(smem_addr(&bars->s_full[t]));
                            if (t == kFwdQTiles - 1) {
                                mma_commit(smem_addr(&bars->kv_empty[kv_stage(ik)]));
                                if (HL && j + 2 == nkv) mma_commit(smem_addr(&bars->q_empty));
                            }
                        }
                    }
                    __syncwarp();
                }
                if (lane == 0) mma_commit(smem_addr(&bars->kv_empty[kv_stage(iv)]));
            }
            // o_full: head hd's products are complete (and, for the last head, tells the
            // teardown that no MMA is still running)
            if (lane == 0) mma_commit(smem_addr(&bars->o_full));
        }
    } else if (warp == 2) {
        // ------------------------------------------------------ K/V relay
        regs_lower<kFwdRegsCtl>();
        for (int hd = 0; hd < hpc; ++hd) {
            const int base = hd * 2 * nkv;
            for (int j = 0; j < nkv; ++j) {
                if (lane == 0) {
                    for (int i = 2 * j + 1; i <= 2 * j + 2 && i < 2 * nkv; ++i)
                        mbar_wait(smem_addr(&bars->kv_full[(base + i) % C::kStages]),
                                  ((base + i) / C::kStages) & 1, abort_flag, p.timeout_cycles,
                                  p.status);
                }
                __syncwarp();
                for (int t = 0; t < kFwdQTiles; ++t) named_bar_sync(kFwdBarP + t, kFwdBarCount);
            }
        }
    } else if (warp == 3) {
        regs_lower<kFwdRegsCtl>();   // idle; its warpgroup gives registers away
    } else if (warp >= 4) {
        // ------------------------------------------------- softmax + epilogue
        regs_raise<kFwdRegsSoftmax>();
        const int t = (warp - 4) / 4;
        const int quad = warp % 4;
        const int r = quad * 32 + lane;               // row within the tile = TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_addr + C::kColS + t * kBlockN;
        const uint32_t tO = tmem + lane_addr + C::kColO + t * D;
        const int q = q0 + t * kBlockM + r;           // query position in the sequence
        const int lo_q = key_lo(s, q), hi_q = key_hi(s, q, len);
        const int tile_q_first = q0 + t * kBlockM, tile_q_last = tile_q_first + kBlockM - 1;
        const int full_lo = key_lo(s, tile_q_last);            // keys >= this are >= every row's lo
        const int full_hi = key_hi(s, tile_q_first, len);      // keys <= this are <= every row's hi
        const float sl2 = p.scale_log2;
        // fp8: the scores of key block j are (Q8 K8^T) s_q s_k with s_q the scale of this
        // query tile and s_k that of the key block; both fold into the exponent scale
        const int blk_col = F8 ? seq_block_col(s, b) : 0;
        // (a tile wholly past the sequence end reads its last block's scale; its rows
        // are never stored)
        const long long sq_idx = static_cast<long long>(h0) * p.nb + blk_col +
                                 min(q0 / kBlockM + t, ceil_div(len, kBlockM) - 1);
        const float sq = (F8 && fa_index_ok(sq_idx, static_cast<long long>(s.Hq) * p.nb, p.status))
                             ? __ldg(p.q_scale + sq_idx) : 1.f;
        const float* ks_row = F8 ? p.k_scale + static_cast<long long>(g) * p.nb + blk_col : nullptr;
        const uint32_t hs = static_cast<uint32_t>(b * s.Hq + h0);   // dropout counter word

        // Dropout: the Philox words of a key block do not depend on the scores, so each
        // row draws those of its next block right after handing P over, while the tensor
        // cores compute that block's scores, turns them into keep masks and parks them in
        // shared memory (its own 128-byte row; 16-byte chunks XOR-swizzled by the row so
        // that a warp's accesses spread over the banks).
        uint4* drop_row = reinterpret_cast<uint4*>(smem + C::kTilesBytes + C::kBarBytes) +
                          (t * kBlockM + r) * (kBlockN / 16);
        auto draw_block = [&](int jj) {
            uint32_t dw[kBlockN / 4];
            dropout_words_rows<kBlockN / 4>(dw, q >> 2, ((kv_first + jj) * kBlockN) >> 2, hs,
                                            p.drop.offset, p.drop.seed_lo, p.drop.seed_hi, lane);
            keep_masks(dw, p.drop.thresh);
#pragma unroll
            for (int c = 0; c < kBlockN / 16; ++c)
                drop_row[c ^ (r & 7)] = make_uint4(dw[4 * c], dw[4 * c + 1], dw[4 * c + 2], dw[4 * c + 3]);
        };
        if (DROP) draw_block(0);

        // `ok` turns false (warp-uniformly: the TMEM accesses are warp-collective)
        // when a wait gives up; the warp then skips the work but keeps taking part
        // in every named-barrier phase, blocking instead of arriving.
        bool ok = true;
        for (int hd = 0; hd < hpc; ++hd) {
            const int h = h0 + hd;
            float m_ref = kNegInf;  // exponent reference (log2 units), shared by O and l
            float l = 0.f;
            for (int j = 0; j < nkv; ++j) {
                if (ok)
                    ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bars->s_full[t]), (hd * nkv + j) & 1,
                                                           abort_flag, p.timeout_cycles, p.status));
                if (ok) {
                    tc_fence_after();
                    uint32_t sr[kBlockN];
#pragma unroll
                    for (int c = 0; c < kBlockN / 32; ++c)
                        tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
                    tmem_ld_wait();
                    reg_fence(sr);
                    float sv[kBlockN];
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c) sv[c] = __uint_as_float(sr[c]);
                    const int kb = (kv_first + j) * kBlockN;
                    if (!(kb >= full_lo && kb + kBlockN - 1 <= full_hi)) {
                        const int clo = lo_q - kb, chi = hi_q - kb;
#pragma unroll
                        for (int c = 0; c < kBlockN; ++c)
                            if (c < clo || c > chi) sv[c] = kNegInf;
                    }
                    // row max in 8 independent chains (short latency) of three-input maxima
                    // (half the instructions of two-input ones)
                    float mx8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = sv[i];
#pragma unroll
                    for (int c = 8; c + 16 <= kBlockN; c += 16)
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], sv[c + i], sv[c + 8 + i]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], sv[kBlockN - 8 + i]);
                    const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                           fmaxf(mx8[6], mx8[7]));
                    const float sl2b =
                        (F8 && fa_index_ok(static_cast<long long>(g) * p.nb + blk_col + kv_first + j,
                                           static_cast<long long>(s.Hkv) * p.nb, p.status))
                            ? sl2 * sq * __ldg(ks_row + kv_first + j) : sl2;
                    const float m_blk = mx * sl2b;
                    float alpha = 1.f;
                    bool rescale = false;
                    if (m_blk > m_ref + kRescaleThreshold) {
                        alpha = ex2_approx(m_ref - m_blk);  // 0 on the first visible block
                        rescale = (j > 0);
                        m_ref = m_blk;
                        l *= alpha;
                    }
                    const float neg_ref = (m_ref == kNegInf) ? 0.f : -m_ref;
                    const uint64_t sl2x2 = f2_pack(sl2b, sl2b), nref2 = f2_pack(neg_ref, neg_ref);
                    uint64_t rs2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
                    // P (16-bit pairs) goes to the first 64 columns of S_t in two halves; every
                    // S value is already in registers, so the overwrite is safe.  fp8: P as
                    // e4m3, four keys per column, the first 32 columns.
#pragma unroll
                    for (int half = 0; half < 2 && F8; ++half) {
                        uint32_t pk[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int kc = 64 * half + 4 * c;
                            const float2 a = f2_unpack(f2_fma(f2_pack(sv[kc], sv[kc + 1]), sl2x2, nref2));
                            const float2 e = f2_unpack(f2_fma(f2_pack(sv[kc + 2], sv[kc + 3]), sl2x2, nref2));
                            const float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
                            const float p2 = ex2_approx(e.x), p3 = ex2_approx(e.y);
                            rs2[c & 1] = f2_add(rs2[c & 1], f2_add(f2_pack(p0, p1), f2_pack(p2, p3)));
                            pk[c] = pack4_e4m3(p0, p1, p2, p3);
                        }
                        tmem_st16(tS + 16 * half, pk);
                    }
#pragma unroll
                    // (an eighth of the row per TMEM store, 16 keys in 8 packed words, and two
                    // row-sum chains keep the live registers of the pass within the 168 the
                    // compiler allocates to every warp: no spills in the 16-bit instances)
                    for (int qtr = 0; qtr < 4 && !F8; ++qtr) {
                        // dropout: the keep masks of keys kb + 32 qtr .. + 31 of this row;
                        // l sums the probabilities before dropout, the product takes the kept
                        // ones (the 1 / keep-probability factor is applied to O in fp32 at the
                        // end, so the 16-bit P carries no extra rounding)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            // the keep masks of these 16 keys: one 16-byte chunk of the row
                            uint32_t dw[DROP ? 4 : 1];
                            if (DROP) {
                                const uint4 v = drop_row[(2 * qtr + hh) ^ (r & 7)];
                                dw[0] = v.x;
                                dw[1 % (DROP ? 4 : 1)] = v.y;
                                dw[2 % (DROP ? 4 : 1)] = v.z;
                                dw[3 % (DROP ? 4 : 1)] = v.w;
                            }
                            uint32_t pk8[8];
#pragma unroll
                            for (int c8 = 0; c8 < 8; ++c8) {
                                const int c = 8 * hh + c8;
                                const int k = 32 * qtr + 2 * c;
                                const float2 a = f2_unpack(f2_fma(f2_pack(sv[k], sv[k + 1]), sl2x2, nref2));
                                const float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
                                rs2[c & 1] = f2_add(rs2[c & 1], f2_pack(p0, p1));
                                pk8[c8] = pack2<E>(p0, p1);
                                if (DROP) pk8[c8] &= keep_mask_pair(dw[(c8 >> 1) % (DROP ? 4 : 1)], 2 * c);
                            }
                            tmem_st8(tS + 16 * qtr + 8 * hh, pk8);
                        }
                    }
                    const float2 rsum = f2_unpack(f2_add(rs2[0], rs2[1]));
                    l += rsum.x + rsum.y;
                    if (__any_sync(0xffffffffu, rescale)) {
                        // O_t was last written by O_t += P V_{j-1}, complete before S_t(j) was
                        // signalled; scale it in place before the next product accumulates.
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t orow[32];
                            tmem_ld32(tO + c * 32, orow);
                            tmem_ld_wait();
                            reg_fence(orow);
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                orow[i] = __float_as_uint(__uint_as_float(orow[i]) * alpha);
                            tmem_st32(tO + c * 32, orow);
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                }
                named_bar_signal(kFwdBarP + t, kFwdBarCount, ok);
                if (DROP && ok && j + 1 < nkv) draw_block(j + 1);
            }
            // ------------------------------------------------------------ epilogue
            if (ok)
                ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bars->o_full), hd & 1, abort_flag,
                                                       p.timeout_cycles, p.status));
            // A tile of 128 query rows inside the sequence leaves through shared memory
            // (its K/V stage, idle by now) and TMA stores, coalesced and asynchronous; a
            // tile cut by the sequence end, and any head but the CTA's last (the ring is
            // streaming the next head's tiles), row by row.  The choice is made uniform over
            // the warpgroup.
            const bool valid = q < len;
            // fp8: O carries the scale of V (per sequence and key/value head)
            const float vs = (F8 && fa_index_ok(static_cast<long long>(g) * s.B + b,
                                                static_cast<long long>(s.Hkv) * s.B, p.status))
                                 ? __ldg(p.v_scale + static_cast<long long>(g) * s.B + b) : 1.f;
            const float inv_l = (l > 0.f) ? (DROP ? p.drop.rscale : 1.f) * vs / l : 0.f;
            if (hd == hpc - 1 && named_bar_all(kFwdBarEpi + t, kBlockM, ok && tile_q_first + kBlockM <= len)) {
                tc_fence_after();
                uint8_t* stage = sKV + t * C::kOTileBytes;
                stage_acc_row<D, EO>(tO, inv_l, stage, C::kChunkBytes, r, 0);
                fence_proxy_async_smem();
                named_bar_sync(kFwdBarEpi + t, kBlockM);
                if (quad == 0 && lane == 0) {
                    if (fa_box_ok(seq_start + tile_q_first, kBlockM, s.total_tokens, h, s.Hq, p.status))
                        for (int c = 0; c < C::kOChunks; ++c)
                            tma_store_3d(&p.tm_o, smem_addr(stage + c * C::kChunkBytes), c * 64, h,
                                         seq_start + tile_q_first);
                    bulk_commit_group();
                    bulk_wait_read_all();   // the CTA's shared memory outlives the reads
                }
            } else if (ok) {
                tc_fence_after();
                uint16_t* orow_g = static_cast<uint16_t*>(p.o) +
                                   (static_cast<long long>(seq_start + q) * s.Hq + h) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t orow[32];
                    tmem_ld32(tO + c * 32, orow);
                    tmem_ld_wait();
                    reg_fence(orow);
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack2<EO>(__uint_as_float(orow[2 * i]) * inv_l,
                                         __uint_as_float(orow[2 * i + 1]) * inv_l);
                    if (valid && fa_index_ok(static_cast<long long>(seq_start + q) * s.Hq + h,
                                             static_cast<long long>(s.total_tokens) * s.Hq, p.status)) {
                        uint4* dst = reinterpret_cast<uint4*>(orow_g + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                }
            }
            if (ok && valid && fa_index_ok(row_stat_index(s, b, h, seq_start, q),
                                           static_cast<long long>(s.total_tokens) * s.Hq, p.status))
                p.lse[row_stat_index(s, b, h, seq_start, q)] =
                    (l > 0.f) ? m_ref * kLn2 + logf(l) : kNegInf;
        }
    }

    // ------------------------------------------------------------ teardown
    if (*abort_flag && warp == 1 && lane == 0) {
        // o_full was committed last: once it fires no tcgen05 op still uses TMEM
        mbar_wait_drain(smem_addr(&bars->o_full), (hpc - 1) & 1, kDrainCycles);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// Heads per scheduling chunk of the forward (map_work): as many as keep the
// chunk's K and V at the longest sequence within 16 MB of L2, at least
// kHeadChunk.  At 1 MB of K and V per head (d = 128, 2048 keys) 16 heads per
// chunk ran 7% faster than 8 (the tail of longest-first items is shorter); at
// 4 MB per head and more every chunk wider than 8 was slower.
int fwd_head_chunk(int n_keys, int d, int elem_bytes) {
    const long long per_head = 2LL * n_keys * d * elem_bytes;
    const long long fit = (16LL << 20) / (per_head > 0 ? per_head : 1);
    return static_cast<int>(fit < kHeadChunk ? kHeadChunk : fit > 4096 ? 4096 : fit);
}

template <int D, int E, bool DROP, bool HL = false>
cudaError_t launch_fwd_d(const FwdParams& params, cudaStream_t stream) {
    using C = FwdCfg<D, E>;
    FwdParams p = params;
    p.head_chunk = fwd_head_chunk(p.seq.N, D, C::kElemBytes);
    auto kern = fa_fwd_kernel<D, E, DROP, HL>;
    // the register split needs the launch's full 168 registers per thread: a
    // build that gave the kernel fewer would make the softmax warps wait forever
    static const cudaError_t regs_ok = [&] {
        cudaFuncAttributes fa;
        const cudaError_t r = cudaFuncGetAttributes(&fa, kern);
        if (r != cudaSuccess) return r;
        return fa.numRegs >= kFwdRegsLaunch ? cudaSuccess : cudaErrorInvalidKernelImage;
    }();
    if (regs_ok != cudaSuccess) return regs_ok;
    constexpr int smem = DROP ? C::kSmemBytesDrop : C::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<p.num_work, C::kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdParams& p, int d, cudaStream_t stream) {
    if (p.num_work <= 0) return cudaSuccess;
    if (p.elem == kElemFp8) return d == 128 ? launch_fwd_d<128, kElemFp8, false>(p, stream) : cudaErrorInvalidValue;
    const bool f16 = p.elem == kElemF16, drop = p.drop.thresh != 0;
    if (drop) {
        if (f16) return d == 128 ? launch_fwd_d<128, kElemF16, true>(p, stream) : launch_fwd_d<64, kElemF16, true>(p, stream);
        return d == 128 ? launch_fwd_d<128, kElemBf16, true>(p, stream) : launch_fwd_d<64, kElemBf16, true>(p, stream);
    }
    if (p.heads > 1) {   // several query heads per CTA (16-bit, no dropout)
        if (f16) return d == 128 ? launch_fwd_d<128, kElemF16, false, true>(p, stream) : launch_fwd_d<64, kElemF16, false, true>(p, stream);
        return d == 128 ? launch_fwd_d<128, kElemBf16, false, true>(p, stream) : launch_fwd_d<64, kElemBf16, false, true>(p, stream);
    }
    if (f16) return d == 128 ? launch_fwd_d<128, kElemF16, false>(p, stream) : launch_fwd_d<64, kElemF16, false>(p, stream);
    return d == 128 ? launch_fwd_d<128, kElemBf16, false>(p, stream) : launch_fwd_d<64, kElemBf16, false>(p, stream);
}

}  // namespace fa
