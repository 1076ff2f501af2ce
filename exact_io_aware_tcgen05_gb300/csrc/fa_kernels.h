// fa_kernels.h -- parameter blocks and launchers shared by the host API
// (fa_api.cu) and the kernels (fa_fwd.cu, fa_bwd.cu).  Internal to the
// library; the public interface is include/fa.h.
#pragma once

#include "../../include/fa.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fa {

constexpr int kBlockM = 128;   // rows of one MMA tile (TMEM lanes)
constexpr int kBlockN = 128;   // keys per key/value tile
constexpr int kFwdQTiles = 2;  // query tiles per forward CTA (ping-pong)
// element-type codes of FwdParams::elem / BwdParams::elem (the values of fa_dtype;
// the kernels name them kElemBf16 / kElemF16)
constexpr int kElemBf16Code = 0;
constexpr int kElemF16Code = 1;
constexpr int kElemFp8Code = 2;   // the fp8 forward: e4m3 Q, K, V^T and bf16 O
constexpr long long kDefaultTimeoutCycles = 4000000000LL;  // ~2 s at 2 GHz

// Token / sequence geometry common to all kernels.  Dense batches are the
// packed case with sequence b starting at token b*N and length N.
struct SeqInfo {
    const int* cu_seqlens;  // device int32[B+1], or nullptr for dense
    int B;                  // sequences
    int N;                  // dense: length of every sequence; packed: longest
    int total_tokens;       // rows of the token dimension (dense: B*N)
    int Hq, Hkv, group;     // group = Hq / Hkv
    int causal, window;     // window <= 0: none
};

// Dropout of the attention probabilities (see fa_fwd_dropout in fa.h): a pair is
// kept iff its random byte is >= thresh (thresh == 0: no dropout, the kernels
// compiled without it run); kept probabilities are scaled by rscale.
struct DropoutParams {
    uint32_t thresh;    // 0 .. 255
    float rscale;       // 256 / (256 - thresh)
    uint32_t seed_lo, seed_hi, offset;
};

struct FwdParams {
    CUtensorMap tm_q;  // [total_tokens, Hq, d] bf16 or fp16, box 64 x 1 x 128, 128B swizzle
    CUtensorMap tm_k;  // [total_tokens, Hkv, d]
    CUtensorMap tm_v;
    CUtensorMap tm_o;  // output, same layout as tm_q (stores of whole tiles)
    SeqInfo seq;
    void* o;            // [tokens, Hq, d], element type of q
    float* lse;         // fp32 dense [B, Hq, N]; packed [Hq, total_tokens]
    float scale_log2;   // softmax scale * log2(e)
    int num_work;       // launched CTAs (upper bound on work items)
    int head_chunk;     // heads per scheduling chunk (map_work); set by launch_fwd
    int heads;          // query heads per CTA, a divisor of the GQA group (1: fp8, dropout)
    int elem;           // element type of q, k, v, o (kElemBf16Code / kElemF16Code), or
                        // kElemFp8Code: e4m3 q, k and transposed v (tm_v over [Hkv, d,
                        // vt_tokens]), bf16 o
    DropoutParams drop;
    // fp8 only: block scales of q [Hq, nb] and k [Hkv, nb], per-sequence scales of v [Hkv, B]
    const float* q_scale;
    const float* k_scale;
    const float* v_scale;
    int nb;
    long long timeout_cycles;
    int* status;        // device status word
};

struct BwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;  // as in FwdParams; dO like Q
    CUtensorMap tm_dq, tm_dk, tm_dv;      // outputs (stores of whole tiles)
    SeqInfo seq;
    const void* q;      // Q (the dQ kernel copies its query tile's rows into TMEM)
    const void* k_ptr;  // K, V (the fused backward's preprocess bounds them)
    const void* v_ptr;
    const void* o;      // forward output (for the preprocess)
    const void* dout;   // dO (for the preprocess)
    const float* lse;   // forward logsumexp, layout as FwdParams::lse
    float* delta;       // fp32 D_i = rowsum(dO * O), same layout as lse
    // fused backward only (null for the split one).  dQ is summed across CTAs as
    // fixed-point int32: element (i, c) of every contribution is rounded to a
    // multiple of 2^-F_ic with F_ic = Fr_i + Fc_gc, where 2^Fr_i = row_scale (from
    // ||dO_i||) and 2^Fc_gc comes from the K and V bounds (kBoundSlots slots of
    // tokens per key/value head: max_j |k_jc| for c < d, max_j ||v_j||_2 at d), so
    // that every partial sum of row i stays below 2^30 in magnitude; integer sums
    // do not depend on the order of the additions.
    int* dq_acc;        // d = 128: [Hq, tokens, d]; d = 64: [Hq, d, tokens]
    float* row_scale;   // 2^Fr_i, layout of lse
    float* kv_bound;    // [Hkv, kBoundSlots, d + 1]
    int pre_row_ctas;   // preprocess CTAs over the rows (the bound CTAs follow them)
    void* dq;           // outputs, element type of q
    void* dk;
    void* dv;
    float scale;        // softmax scale
    float scale_log2;
    int num_work_dq, num_work_dkdv;
    int dq_heads;       // query heads per dQ CTA, a divisor of the GQA group (dq_heads_per_cta)
    int elem;           // element type of every 16-bit tensor (kElemBf16Code / kElemF16Code)
    DropoutParams drop;
    long long timeout_cycles;
    int* status;
};

// Quantisation of one attention operand to e4m3 (fa_fp8.cu).
struct Fp8QuantParams {
    SeqInfo seq;        // only B, N, total_tokens and cu_seqlens are used
    const void* x;      // bf16 [tokens, heads, d]
    void* out;          // Q/K: e4m3 [tokens, heads, d]; V: e4m3 V^T [heads, d, vt_tokens]
    float* scales;      // Q/K: [heads, nb]; V: [heads, B]
    int heads;
    int nb;             // Q/K: columns of the scale array
    long long vt_tokens;  // V: columns of V^T
    int* status;          // device status word (the debug build's bounds checks)
    int rotate;           // Q/K: incoherent processing (sign-randomised Hadamard rotation)
    uint32_t seed_lo, seed_hi;  // its seed, the Philox key
};

// Launchers (defined in the kernel translation units).  They only enqueue on
// `stream` and return the launch error.
cudaError_t launch_fwd(const FwdParams& p, int d, cudaStream_t stream);
int bwd_preprocess_row_ctas(const BwdParams& p, int d);
cudaError_t launch_bwd_preprocess(const BwdParams& p, int d, cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdParams& p, int d, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const BwdParams& p, int d, cudaStream_t stream);
cudaError_t launch_bwd_fused(const BwdParams& p, int d, cudaStream_t stream);
cudaError_t launch_bwd_dq_convert(const BwdParams& p, int d, cudaStream_t stream);

// Slots of tokens per key/value head over which the preprocess takes the maxima
// of |k_jc| and ||v_j||_2 for the fused backward's fixed-point scales.
constexpr int kBoundSlots = 32;
cudaError_t launch_fp8_quant_qk(const Fp8QuantParams& p, int d, int grid, cudaStream_t stream);
cudaError_t launch_fp8_quant_v(const Fp8QuantParams& p, int d, int grid, cudaStream_t stream);

int* device_status_word();  // library-owned device status word (fa_api.cu)

// Byte layout of the backward workspace (fa_api.cu): D at 0 (`delta` bytes; all
// the split backward needs), then for the fused backward the row scales, the
// K/V bound slots and the int32 dQ accumulator; `full` bytes in all.
struct BwdWorkspace {
    size_t delta;                     // row statistics D (all the split backward needs)
    size_t scale_offset, bound_offset, acc_offset;
    size_t full;                      // + row scales, K/V bound slots, int32 dQ accumulator
};
bool bwd_workspace(int B, int Hq, int Hkv, int N, int d, int total_tokens, BwdWorkspace* w);

// Identifier of the calling thread's current CUDA context, unique for the life
// of the process (0 if no context is current or the driver cannot say).  Device
// addresses of the library's own __device__ arrays are cached per device and
// looked up again when this changes, e.g. after cudaDeviceReset.
unsigned long long current_context_id();

// Records `fmt` as the calling thread's fa_last_error() message; returns st.
fa_status report_error(fa_status st, const char* fmt, ...);

}  // namespace fa
