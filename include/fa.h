/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library libfa_gb300.so.
 *
 * The library computes exact scaled dot-product attention tile by tile with an
 * online softmax, so the N x N score / probability matrix never reaches HBM,
 * and the backward pass by recomputation from the saved logsumexp:
 *
 *   "FlashAttention: How IO-Aware Tiling and Online Softmax Solved Transformer
 *    Memory Bottlenecks" -- "Naive Attention Execution Profile" (S = QK^T,
 *    P = softmax(S), O = PV), "1. IO-Aware Tiling", "2. Online Softmax
 *    Reduction" (running max / normaliser, rescale, final division) and
 *    "3. Recomputation in the Backward Pass";
 *   "Flash Attention -- Fast Memory-Efficient Exact Attention" -- "What Flash
 *    Attention Does" (causal masking, variable-length sequences, GQA/MQA),
 *    "Key Features" (sliding window), "Architecture Overview" (backward from
 *    the saved output and logsumexp statistics), "Self-Hosting &
 *    Configuration" (FP16 and BF16).
 *
 * Conventions for every entry point
 * ---------------------------------
 * Pointers marked "device" are CUDA device pointers owned by the caller; the
 * library never allocates, frees or keeps them, and never synchronises the
 * stream (fa_device_status excepted).  Every tensor is contiguous, bf16 unless
 * stated (fa_fwd_typed / fa_bwd_typed also take fp16), and 16-byte aligned
 * (TMA requirement).
 *
 *   dense batch (cu_seqlens == NULL): B sequences of N tokens each
 *     q, o, dout, dq   [B, N, Hq, d]      k, v, dk, dv   [B, N, Hkv, d]
 *     lse, workspace rows  [B, Hq, N] fp32
 *   packed batch (cu_seqlens != NULL): B sequences concatenated, T tokens
 *     q, o, dout, dq   [T, Hq, d]         k, v, dk, dv   [T, Hkv, d]
 *     lse              [Hq, T] fp32
 *     cu_seqlens       device int32[B + 1], cu_seqlens[0] = 0,
 *                      cu_seqlens[B] = T, non-decreasing; sequence b holds
 *                      tokens cu_seqlens[b] .. cu_seqlens[b+1]-1.
 *     N must be >= the longest sequence and total_tokens must equal T: the
 *     library cannot read cu_seqlens on the host without a synchronisation,
 *     and uses them to bound its TMA descriptors and grids.
 *
 *   Scores are S_ij = scale * q_i . k_j (the page's S = QK^T with the usual
 *   softmax scale made explicit; pass scale = 1/sqrt(d) for the standard
 *   form).  Key j is visible to query i of the same sequence iff
 *     causal == 0:  always;
 *     causal != 0:  j <= i, and if window > 0 also i - j < window, i.e. each
 *                   query sees at most `window` keys including itself.
 *   window > 0 requires causal != 0.  Query head h reads key/value head
 *   h / (Hq / Hkv) (consecutive grouping); Hkv == 1 is multi-query attention.
 *   lse holds the natural-log logsumexp LSE_i = ln sum_{j visible} exp(S_ij).
 *   A row with no visible key (impossible with the masks above unless a
 *   sequence is empty) gets O = 0 and LSE = -inf.
 *
 * Supported: d in {64, 128}; 1 <= Hkv <= Hq, Hq % Hkv == 0.  Outputs are
 * written in full (no accumulate mode), rounded to the input element type
 * (bf16 unless stated) by round-to-nearest-even from fp32 accumulators.
 *
 * Errors: argument checks run before anything is enqueued and return
 * FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED / FA_ERR_WORKSPACE; a failed launch
 * returns FA_ERR_CUDA.  fa_last_error() gives a message for the calling
 * thread's last non-OK status.  Kernels never trap: every wait inside them is
 * bounded, and a wait that gives up records FA_ERR_TIMEOUT in a library-owned
 * device status word, read (and cleared) by fa_device_status().
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the 16-bit tensors (q, k, v, o, dout, dq, dk, dv); products
 * accumulate in fp32 either way and lse / workspace stay fp32. */
typedef enum fa_dtype {
    FA_DTYPE_BF16 = 0,       /* bfloat16 (the type of fa_fwd / fa_bwd)             */
    FA_DTYPE_F16 = 1         /* IEEE binary16                                       */
} fa_dtype;

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad size or flag          */
    FA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. d not in {64, 128})  */
    FA_ERR_WORKSPACE = 3,    /* workspace null, misaligned or below fa_bwd_workspace_size_min */
    FA_ERR_CUDA = 4,         /* a CUDA call failed; see fa_last_error()               */
    FA_ERR_TIMEOUT = 5       /* a kernel's bounded wait gave up (fa_device_status)    */
} fa_status;

/*
 * Forward pass: O = softmax(scale * Q K^T, masked) V and LSE.
 *   q, k, v       device, read only (layouts above)
 *   o             device, written: bf16, layout of q
 *   lse           device, written: fp32 [B, Hq, N] dense, [Hq, T] packed
 *   B, Hq, Hkv, N, d, causal, window, cu_seqlens, total_tokens: see above
 *                 (total_tokens is ignored for dense batches)
 *   scale         softmax scale, finite and > 0
 *   stream        CUDA stream the kernel is enqueued on (0: legacy default)
 * Enqueues one kernel; returns without waiting for it.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int N, int d, int causal, int window, const int* cu_seqlens,
                 int total_tokens, float scale, cudaStream_t stream);

/*
 * Query heads per CTA of the forward (per calling thread).  One CTA may serve several
 * consecutive query heads in turn and pay its fixed costs (set-up, the first loads,
 * the exit) once; the heads of one key/value group also read the same K and V tiles.
 * 0, the default, lets fa_fwd choose: the largest divisor of the group Hq / Hkv that
 * still leaves at least 4 CTAs per SM; where that is 1 (always without GQA), 2 when no
 * sequence is longer than 2048 tokens and at least 1.5 CTAs per SM remain.  A positive
 * value forces that many; fa_fwd then fails with FA_ERR_INVALID_ARG (before any launch)
 * if it does not divide Hq.  The forward with dropout and the fp8 forward always serve
 * one head per CTA.  Results do not depend on the choice (each head's products, their
 * order and the epilogue's arithmetic are the same).  FA_ERR_INVALID_ARG for heads < 0.
 */
fa_status fa_fwd_set_heads(int heads);

/*
 * How many query heads per CTA fa_fwd (16-bit, no dropout) would serve on the calling
 * thread for these sizes: the fa_fwd_set_heads value if one is set, else the library's
 * choice above.  total_tokens: T for a packed batch, 0 for a dense one (the choice needs
 * only the token and sequence counts, not cu_seqlens).  The SM count is the current
 * device's, 152 (GB300) when none can be queried.  -1 for invalid sizes or a set value
 * that does not divide Hq (fa_fwd would fail).  No device work.
 */
int fa_fwd_heads(int B, int Hq, int Hkv, int N, int d, int causal, int window, int total_tokens);

/*
 * Backward paths.  fa_bwd runs one of two:
 *   split  the row statistics D_i = sum_c dO_ic O_ic, a dK/dV kernel, then a dQ
 *          kernel that rebuilds S and dP a second time (any mask);
 *   fused  (any mask) D_i and the fixed-point scales, ONE kernel that forms
 *          dQ, dK and dV from a single rebuild of each score tile, then a
 *          kernel that converts the dQ sums.  Several CTAs add into each dQ row;
 *          each contribution is rounded to fixed point (an int32 multiple of
 *          2^-F for an F chosen per row and channel from ||dO_i||_2, max_j ||v_j||_2
 *          and max_j |k_jc|, so that no partial sum exceeds 2^30), and integer sums
 *          do not depend on the order of the additions.  The rounding adds at most
 *          (contributing 128-key tiles / 2) 2^-F to an element: about 1e-7 of the
 *          bound 2 ||dO_i|| max||v_j|| max|k_jc| on |dQ_ic| / scale per tile.
 * Both are deterministic (the same inputs, workspace size and path give the same
 * bits); their dQ differ in the last bits.
 *
 * Workspace (total_tokens: T for a packed batch, 0 for a dense one, whose B * N
 * rows are used; 0 for invalid sizes):
 *   fa_bwd_workspace_size_min    the split backward's: D, one fp32 per query row
 *                                and head, padded to 256 bytes;
 *   fa_bwd_workspace_size_fused  the fused backward's: D, the row scales (one
 *                                fp32 per row and head), the K/V bounds (32 x
 *                                (d + 1) fp32 per key/value head) and the int32
 *                                dQ sums (d per row and head), each padded;
 *   fa_bwd_workspace_size        what the default choice below needs for this d.
 *
 * Choice (per calling thread, fa_bwd_set_path): FA_BWD_AUTO, the default, runs
 * the fused backward where it measured faster on GB300 (d = 64, with or without a
 * causal mask), given at least fa_bwd_workspace_size_fused bytes, and the split
 * one otherwise; FA_BWD_SPLIT always runs the split one; FA_BWD_FUSED always runs
 * the fused one and fails with FA_ERR_WORKSPACE given a smaller workspace.
 * fa_bwd_path tells which one fa_bwd would run on the calling thread (-1: it
 * would fail).
 */
typedef enum fa_bwd_path_kind {
    FA_BWD_AUTO = -1,
    FA_BWD_SPLIT = 0,        /* row statistics; dK/dV kernel; dQ kernel (3 kernels) */
    FA_BWD_FUSED = 1         /* row statistics; fused kernel; dQ conversion (3 kernels) */
} fa_bwd_path_kind;
size_t fa_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d, int total_tokens);
size_t fa_bwd_workspace_size_min(int B, int Hq, int Hkv, int N, int d, int total_tokens);
size_t fa_bwd_workspace_size_fused(int B, int Hq, int Hkv, int N, int d, int total_tokens);
void fa_bwd_set_path(int path);
int fa_bwd_path(int B, int Hq, int Hkv, int N, int d, int causal, int window, int total_tokens,
                size_t workspace_bytes);

/*
 * Query heads per CTA of the split backward's dQ kernel (per calling thread).  The
 * query heads of one key/value group read the same K and V tiles, so one CTA may
 * serve several of them in turn and pay its fixed costs (set-up, the first loads)
 * once.  0, the default, lets fa_bwd choose: the largest divisor of the group
 * Hq / Hkv that still leaves at least 4 CTAs per SM (1 without GQA).  A positive
 * value forces that many; fa_bwd then fails with FA_ERR_INVALID_ARG (before any
 * launch) if it does not divide the group.  The backward with dropout always serves
 * one head per dQ CTA.  Results do not depend on the choice: each head's products
 * and their order are the same, so the bits are too.  FA_ERR_INVALID_ARG for
 * heads < 0.
 */
fa_status fa_bwd_set_dq_heads(int heads);

/*
 * How many query heads per dQ CTA the split backward (no dropout) would serve on the
 * calling thread for these sizes: the fa_bwd_set_dq_heads value if one is set, else the
 * library's choice above.  Arguments as for fa_fwd_heads; -1 for invalid sizes or a set
 * value that does not divide the group (fa_bwd would fail).  No device work.
 */
int fa_bwd_dq_heads(int B, int Hq, int Hkv, int N, int d, int causal, int window, int total_tokens);

/*
 * fa_fwd and fa_bwd for an explicit element type: `dtype` gives the type of
 * every 16-bit tensor of the call (all of them share it; "Flash Attention --
 * Fast Memory-Efficient Exact Attention", "Self-Hosting & Configuration", lists
 * FP16 and BF16).  The probabilities P
 * and the gradient dS that feed the second products are rounded to the same
 * type.  fa_fwd and fa_bwd are these with FA_DTYPE_BF16.  A dtype outside
 * fa_dtype returns FA_ERR_UNSUPPORTED before anything is enqueued; all other
 * arguments and errors are those of fa_fwd / fa_bwd.
 */
fa_status fa_fwd_typed(fa_dtype dtype, const void* q, const void* k, const void* v, void* o,
                       float* lse, int B, int Hq, int Hkv, int N, int d, int causal, int window,
                       const int* cu_seqlens, int total_tokens, float scale, cudaStream_t stream);
fa_status fa_bwd_typed(fa_dtype dtype, const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int N, int d, int causal, int window,
                       const int* cu_seqlens, int total_tokens, float scale, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream);

/*
 * Forward and backward with dropout on the attention probabilities.  The pages
 * give dropout no semantics; this library defines them.  With P the softmax
 * probabilities (computed before dropout, so LSE is that of fa_fwd),
 *   O_i = sum_j Z_ij v_j,    Z_ij = P_ij * keep_ij * r,
 * keep_ij in {0, 1}, r = 256 / (256 - t) and t = floor(256 * p_drop + 1/2) (in
 * float; p_drop in [0, 1), t <= 255), so a pair is dropped with probability
 * t / 256 and kept pairs are scaled to keep the expectation.  The backward pass
 * is the gradient of that O for the same keep mask:
 *   dV_j = sum_i Z_ij dO_i,  dP_ij = keep_ij * r * (dO_i . v_j),
 *   dS_ij = P_ij (dP_ij - D_i) with D_i = dO_i . O_i, dQ and dK from dS as in fa_bwd.
 * keep_ij comes from Philox4x32-10 (Salmon, Moraes, Dror, Shaw: "Parallel
 * Random Numbers: As Easy as 1, 2, 3", SC 2011) with key (seed & 0xffffffff,
 * seed >> 32): for query i and key j of sequence b (positions within the
 * sequence) and query head h, the call with counter
 *   (j / 4, i / 4, b * Hq + h, offset)
 * returns four 32-bit words; byte (j % 4) (bits 8 (j%4) .. +7) of word (i % 4)
 * is the pair's random byte, and keep_ij = (byte >= t).  fa_bwd_dropout must be
 * called with the p_drop, seed and offset of the matching fa_fwd_dropout.
 * p_drop == 0 gives exactly fa_fwd_typed / fa_bwd_typed.  Errors: p_drop
 * outside [0, 1) is FA_ERR_INVALID_ARG, t == 256 FA_ERR_UNSUPPORTED; the rest
 * as fa_fwd / fa_bwd.
 */
fa_status fa_fwd_dropout(fa_dtype dtype, float p_drop, unsigned long long seed,
                         unsigned int offset, const void* q, const void* k, const void* v, void* o,
                         float* lse, int B, int Hq, int Hkv, int N, int d, int causal, int window,
                         const int* cu_seqlens, int total_tokens, float scale,
                         cudaStream_t stream);
fa_status fa_bwd_dropout(fa_dtype dtype, float p_drop, unsigned long long seed,
                         unsigned int offset, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout, void* dq, void* dk,
                         void* dv, int B, int Hq, int Hkv, int N, int d, int causal, int window,
                         const int* cu_seqlens, int total_tokens, float scale, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/*
 * FP8 (e4m3) forward.  "FlashAttention: How IO-Aware Tiling and Online Softmax
 * Solved Transformer Memory Bottlenecks" ("FlashAttention-3" bullets) names
 * FP8 with block quantisation of the inputs but gives no format, block or scale
 * rule; this library defines them.
 *
 * e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
 * largest finite value 448; a code is a value rounded to nearest (ties to even)
 * and saturated to +-448.
 *
 * Layouts (tokens as in fa_fwd: dense b * N + i, packed cu_seqlens[b] + i):
 *   q8, k8   e4m3 [tokens, Hq or Hkv, d], scales [heads, nb]: one per (head,
 *            128-token block of a sequence, ceil(L / 128) blocks for length L);
 *            block kb of sequence b is column c_b + kb, with c_b = b ceil(N / 128)
 *            for a dense batch and c_b = floor(cu_seqlens[b] / 128) + b for a
 *            packed one (columns between sequences unused).
 *            nb >= fa_fp8_scale_blocks(...).
 *   vt8      e4m3 V^T [Hkv, d, vt_tokens]: key i of sequence b (and channel c)
 *            at column 128 c_b + i, row c; the columns past a sequence's length
 *            up to its next multiple of 128 hold zero codes.
 *            vt_tokens >= fa_fp8_vt_tokens(...), a multiple of 128.
 *   v_scale  [Hkv, B]: one per (key/value head, sequence).
 * The values are code * scale.  fa_fp8_quantize_qk / fa_fp8_quantize_v write
 * these from bf16 tensors in the layouts of fa_fwd: per block (Q, K) or per
 * (sequence, head) (V), scale = amax / 448 in float (1 for an all-zero block,
 * and for the V of an empty sequence) and code = e4m3(x / scale) with the
 * division rounded to nearest in float.
 *
 * fa_fwd_fp8 computes O (bf16, layout of fa_fwd) and LSE (fp32, layout of
 * fa_fwd) of exact attention on those values, with the arguments and masks of
 * fa_fwd.  The products run on e4m3 operands with fp32 accumulation; the
 * probabilities are rounded to e4m3 for the P V product (the row sums use them
 * unrounded), so each O element is within 2^-4 sum_j P_ij |V_jc| plus 2^-10 per
 * key with P_ij < 2^-6 of the exact value (plus the bf16 rounding of O); LSE is
 * as accurate as fa_fwd's.  Only d = 128 (FA_ERR_UNSUPPORTED otherwise); no
 * dropout.  Pointers: tensors 16-byte aligned, scale arrays 4-byte aligned.
 * Errors otherwise as fa_fwd.  The quantisers take d in {64, 128} and the
 * geometry arguments of fa_fwd (H heads); they only enqueue work.
 *
 * fa_fp8_scale_blocks / fa_fp8_vt_tokens return the minimum nb / vt_tokens for
 * a batch (dense: B ceil(N / 128) blocks; packed != 0: ceil(total_tokens / 128)
 * + B, the column space above), or 0 for invalid arguments.
 */
int fa_fp8_scale_blocks(int B, int N, int total_tokens, int packed);
int fa_fp8_vt_tokens(int B, int N, int total_tokens, int packed);
fa_status fa_fp8_quantize_qk(const void* x, void* x8, float* scales, int nb, int B, int H, int N,
                             int d, const int* cu_seqlens, int total_tokens, cudaStream_t stream);
fa_status fa_fp8_quantize_v(const void* v, void* vt8, float* scales, int vt_tokens, int B, int H,
                            int N, int d, const int* cu_seqlens, int total_tokens,
                            cudaStream_t stream);

/*
 * Incoherent processing, the other FP8 technique the same bullets name without
 * defining it.  This library's reading: a random orthogonal rotation R of the
 * head dimension applied to Q and to K before the block quantisation.  Because
 * (R q) . (R k) = q . k, fa_fwd_fp8 needs no change (Q and K must be rotated with
 * the same seed; V is not rotated), while a channel much larger than the rest is
 * spread over all d, so the e4m3 rounding errors of the score terms average out.
 *
 *   R x = (1/sqrt d) H_d diag(sigma) x on each row x (d channels), H_d the
 *   Sylvester Hadamard matrix, H[i][c] = (-1)^popcount(i & c); sigma_c = -1 where
 *   bit c % 32 of word c / 32 of Philox4x32-10 (defined with the dropout entry
 *   points) at counter (0, 0xFFFFFFFF, 0xFFFFFFFF, 0), key (seed mod 2^32,
 *   seed / 2^32), is set, else +1.
 *   The float32 arithmetic has one order, so the codes are reproducible bit for
 *   bit: the sign flips; for h = 1, 2, 4, ..., d/2 in turn, every channel pair
 *   (c, c + h) with c & h = 0 becomes (a + b, a - b), each rounded to nearest; one
 *   product with float32(1/sqrt d), rounded to nearest.  The amax, scale and codes
 *   of each block are then taken from those float32 values as in
 *   fa_fp8_quantize_qk (arguments, layouts and errors as there).
 */
fa_status fa_fp8_quantize_qk_incoherent(const void* x, void* x8, float* scales, int nb, int B,
                                        int H, int N, int d, const int* cu_seqlens,
                                        int total_tokens, unsigned long long seed,
                                        cudaStream_t stream);
fa_status fa_fwd_fp8(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                     const void* vt8, const float* v_scale, int nb, int vt_tokens, void* o,
                     float* lse, int B, int Hq, int Hkv, int N, int d, int causal, int window,
                     const int* cu_seqlens, int total_tokens, float scale, cudaStream_t stream);

/*
 * Backward pass of fa_fwd for the loss gradient dO, recomputing S and P from
 * the saved logsumexp ("3. Recomputation in the Backward Pass"):
 *   D_i = dO_i . O_i,  P_ij = exp(S_ij - LSE_i),  dP_ij = dO_i . v_j,
 *   dS_ij = P_ij (dP_ij - D_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
 *   dV_j = sum_i P_ij dO_i,
 * with dK and dV summed over the query heads that share a key/value head.
 * (The pages give no backward formulas; these are the calculus of softmax.)
 *   q, k, v, o, lse, dout   device, read only; o and lse as written by fa_fwd
 *   dq, dk, dv              device, written (bf16, layouts of q, k, v)
 *   workspace               device, >= fa_bwd_workspace_size_min(...) bytes
 *                           (see "Backward paths" for the fused backward's),
 *                           256-byte aligned, contents on entry ignored; it
 *                           must not be shared by calls in flight together
 * dQ, dK and dV are deterministic: the same inputs, workspace size and path
 * give the same bits.  Enqueues three kernels on `stream` (either path);
 * returns without waiting.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                 int d, int causal, int window, const int* cu_seqlens, int total_tokens,
                 float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Backward pass with a built-in workspace, for callers that cannot allocate
 * device memory.  The pages have no counterpart to this entry point.
 *
 * fa_bwd needs device scratch (fa_bwd_workspace_size() bytes for its fused
 * backward, at least fa_bwd_workspace_size_min()), normally allocated by the
 * caller.  Some callers cannot call cudaMalloc where they
 * run the backward pass (a framework whose allocator owns all device memory,
 * a plugin that may not allocate behind its host, code that must not
 * allocate because allocation synchronises or may fail mid-step).  This
 * variant takes the same arguments as fa_bwd minus the workspace, and uses a
 * fixed array of FA_STATIC_WORKSPACE_BYTES bytes that the library image
 * places in device memory (every GPU that loads the library holds it until
 * the process exits).  It calls no allocating routine.
 *
 *   - The array is fa_bwd's workspace: a call runs exactly what fa_bwd runs
 *     on the calling thread with a caller workspace of
 *     FA_STATIC_WORKSPACE_BYTES bytes (so the fused backward only where its
 *     workspace fits in the array) and gives the same bits.
 *   - Sizes whose least workspace exceeds the array (fa_bwd_workspace_size_min:
 *     Hq * tokens fp32 row statistics, i.e. Hq * T <= 4,194,304 rows) are
 *     rejected with FA_ERR_WORKSPACE and a message, before anything is
 *     enqueued; other argument errors are those of fa_bwd.
 *   - The first call on a device looks up the array's device address on
 *     that device (cudaGetSymbolAddress, with that device current); make
 *     that first call before any stream capture.  The address is looked up
 *     again on the first call after the device's context has changed (for
 *     instance after cudaDeviceReset); that call, too, belongs before any
 *     capture.
 *   - A call rejected for its size uses up the timing events armed for it
 *     by fa_set_launch_events, as fa_bwd's own argument errors do.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls whose work
 *     overlaps on the GPU race on it: serialise them.
 */
#define FA_STATIC_WORKSPACE_BYTES (16 * 1024 * 1024)
fa_status fa_bwd_static_workspace(const void* q, const void* k, const void* v, const void* o,
                                  const float* lse, const void* dout, void* dq, void* dk,
                                  void* dv, int B, int Hq, int Hkv, int N, int d, int causal,
                                  int window, const int* cu_seqlens, int total_tokens,
                                  float scale, cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device: FA_OK, or FA_ERR_TIMEOUT if a kernel gave up a
 * bounded wait since the last call (its outputs are then incomplete), or
 * FA_ERR_CUDA if the synchronisation itself failed.
 */
fa_status fa_device_status(cudaStream_t stream);

/*
 * Cycle budget of every bounded wait inside the kernels (default about two
 * seconds of SM clock).  Values <= 0 restore the default.  Host-side setting,
 * read at each launch.
 */
void fa_set_wait_limit_cycles(long long cycles);

/*
 * Per-kernel timing hook.  Arms the calling thread's NEXT fa_fwd or fa_bwd
 * call (one call, then it disarms itself): events[i] is recorded on that
 * call's stream just before the call enqueues its i-th kernel, and events[L]
 * just after the last one, L being the number of kernels the call enqueues
 * (fa_fwd: 1; fa_bwd: 3 -- row statistics D, then dK/dV and dQ on the split
 * path, or the fused kernel and the dQ conversion on the fused one).  The
 * events are created and owned by the caller (cudaEventCreate); count must be
 * >= L + 1, otherwise that call fails with FA_ERR_INVALID_ARG before enqueuing
 * anything.  events == NULL disarms.
 */
void fa_set_launch_events(const cudaEvent_t* events, int count);

/*
 * Bounds-checking build.  The library built with FA_DEBUG_CHECKS defined
 * (exact_io_aware_tcgen05_gb300.build.build(debug=True), libfa_gb300_debug.so)
 * checks, inside every kernel, each computed global index and TMA store box
 * against its tensor; a failing check skips the access and records device
 * status 7, which fa_device_status() reports as FA_ERR_CUDA with a message.
 * Nothing traps.  (A stand-in for a memory checker; the kernels are otherwise
 * identical.)
 *   fa_debug_checks_enabled: 1 in that build, 0 in the normal one.
 *   fa_debug_check_selftest: enqueues one thread that tests an index one past
 *     its range without touching memory, so that fa_device_status() must then
 *     report the failed check; FA_ERR_UNSUPPORTED in the normal build.
 */
int fa_debug_checks_enabled(void);
fa_status fa_debug_check_selftest(cudaStream_t stream);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* fa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
