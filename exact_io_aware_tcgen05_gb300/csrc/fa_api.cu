// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument
// checks, TMA descriptor encoding, the device status word and kernel launches.
#include "../../include/fa.h"
#include "fa_kernels.h"
#include "fa_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

namespace fa {

__device__ int g_status_word;  // written by kernels when a bounded wait gives up

namespace {

thread_local char t_last_error[512] = "";
thread_local const cudaEvent_t* t_events = nullptr;  // armed by fa_set_launch_events
thread_local int t_event_count = 0;
thread_local int t_bwd_path = FA_BWD_AUTO;          // fa_bwd_set_path
thread_local int t_dq_heads = 0;                     // fa_bwd_set_dq_heads (0: automatic)
thread_local int t_fwd_heads = 0;                    // fa_fwd_set_heads (0: automatic)

// Takes (and disarms) the events armed for this call, with their count.
void take_events_any(const cudaEvent_t** out, int* count) {
    *out = t_events;
    *count = t_event_count;
    t_events = nullptr;
    t_event_count = 0;
}

// Takes (and disarms) the events armed for this call; fails if too few.
fa_status take_events(int kernels, const cudaEvent_t** out) {
    int count = 0;
    take_events_any(out, &count);
    if (*out && count < kernels + 1) {
        *out = nullptr;
        return FA_ERR_INVALID_ARG;
    }
    return FA_OK;
}

cudaError_t record(const cudaEvent_t* ev, int i, cudaStream_t stream) {
    return ev ? cudaEventRecord(ev[i], stream) : cudaSuccess;
}
std::atomic<long long> g_wait_limit{kDefaultTimeoutCycles};

fa_status fail(fa_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return st;
}

fa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(FA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// [tokens, heads, d] 16-bit elements (bf16 or fp16) viewed as a 3-D tensor (d,
// heads, tokens); the box is 64 elements of d (128 bytes, the swizzle span) x 1
// head x 128 tokens.
fa_status make_token_map(CUtensorMap* map, const void* base, int tokens, int heads, int d,
                         fa_dtype dtype, const char* name) {
    auto enc = encode_fn();
    if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                          static_cast<cuuint64_t>(tokens)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(heads) * d * 2};
    cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kBlockM)};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType type = dtype == FA_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = enc(map, type, 3, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name,
                    static_cast<int>(r));
    return FA_OK;
}

using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

}  // namespace

unsigned long long current_context_id() {
    static PfnCtxGetCurrent get_current = nullptr;
    static PfnCtxGetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PfnCtxGetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PfnCtxGetId>(f);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

namespace {

int* status_word_ptr() {
    // one address per device and context: looked up again when the device's
    // context has changed (after cudaDeviceReset the old address is stale)
    static std::mutex mu;
    static int* ptrs[64] = {nullptr};
    static unsigned long long ctx_ids[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_context_id();
    if (!ptrs[dev] || id == 0 || id != ctx_ids[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int*>(p);
        ctx_ids[dev] = current_context_id();
    }
    return ptrs[dev];
}

struct Geometry {
    SeqInfo seq;
    int tokens;  // rows of the token dimension
};

fa_status check_common(int B, int Hq, int Hkv, int N, int d, int causal, int window,
                       const int* cu_seqlens, int total_tokens, float scale, Geometry* g) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1)
        return fail(FA_ERR_INVALID_ARG, "B, Hq, Hkv and N must be >= 1 (got %d, %d, %d, %d)", B,
                    Hq, Hkv, N);
    if (Hq % Hkv != 0)
        return fail(FA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
    if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d not in {64, 128}", d);
    if (window < 0) return fail(FA_ERR_INVALID_ARG, "window must be >= 0 (got %d)", window);
    if (window > 0 && !causal)
        return fail(FA_ERR_INVALID_ARG, "a sliding window requires causal != 0");
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
    long long tokens;
    if (cu_seqlens) {
        if (total_tokens < 0)
            return fail(FA_ERR_INVALID_ARG, "total_tokens must be >= 0 for a packed batch");
        if (!aligned16(cu_seqlens) && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
            return fail(FA_ERR_INVALID_ARG, "cu_seqlens must be 4-byte aligned");
        tokens = total_tokens;
    } else {
        tokens = static_cast<long long>(B) * N;
    }
    if (tokens > INT_MAX / 2)
        return fail(FA_ERR_UNSUPPORTED, "token count %lld too large", tokens);
    if (static_cast<long long>(B) * Hq * ((N + 127) / 128) > INT_MAX / 2)
        return fail(FA_ERR_UNSUPPORTED, "problem too large for one launch");
    g->seq.cu_seqlens = cu_seqlens;
    g->seq.B = B;
    g->seq.N = N;
    g->seq.total_tokens = static_cast<int>(tokens);
    g->seq.Hq = Hq;
    g->seq.Hkv = Hkv;
    g->seq.group = Hq / Hkv;
    g->seq.causal = causal ? 1 : 0;
    g->seq.window = window;
    g->tokens = static_cast<int>(tokens);
    return FA_OK;
}

// CTAs to launch for blocks of `rows` rows per sequence and head: exact for
// dense batches; for packed ones the slot space of map_work, ceil(T / rows) + B
// slots per head (sequence b's blocks start at slot floor(start_b / rows) + b).
int num_blocks(const Geometry& g, int rows, int heads) {
    long long per_head;
    if (g.seq.cu_seqlens)
        per_head = (static_cast<long long>(g.tokens) + rows - 1) / rows + g.seq.B;
    else
        per_head = static_cast<long long>(g.seq.B) * ((g.seq.N + rows - 1) / rows);
    return static_cast<int>(per_head * heads);
}

constexpr float kLog2e = 1.4426950408889634f;

// Query heads per CTA of the forward kernel and of the split backward's dQ kernel.
// The heads of one key/value group read the same K/V tiles, so one CTA can serve
// several of them in turn and pay its fixed costs (set-up, the first loads) once.
// The largest divisor of the group that still leaves at least kMinWaves CTAs per SM
// is taken (1 without GQA).
constexpr int kMinWaves = 4;

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        sms = 152;
    return sms;
}

int heads_per_cta(const Geometry& g, int rows, int Hq, int Hkv) {
    const int sms = sm_count();
    const int group = Hq / Hkv;
    int best = 1;
    for (int c = 2; c <= group; ++c)
        if (group % c == 0 &&
            static_cast<long long>(num_blocks(g, rows, Hq / c)) >= static_cast<long long>(kMinWaves) * sms)
            best = c;
    return best;
}

// The forward's choice: heads_per_cta (GQA groups on large grids), and where that gives
// one head, the fixed costs alone decide: short sequences (at most 2048 tokens, 16 key
// blocks per query tile) take 2 heads per CTA while at least 1.5 CTAs per SM remain.
// Measured on GB300 without GQA: B4 H16 N2048 causal 0.0783 -> 0.0758 ms with 2 heads,
// 0.116 ms with 4 (128 CTAs); at N = 8192 (items 4x longer) 2 heads were 2.6% slower.
int fwd_heads_per_cta(const Geometry& g, int Hq, int Hkv) {
    constexpr int rows = kFwdQTiles * kBlockM;
    const int c = heads_per_cta(g, rows, Hq, Hkv);
    if (c > 1 || g.seq.N > 2048 || Hq % 2 != 0) return c;
    return 2LL * num_blocks(g, rows, Hq / 2) >= 3LL * sm_count() ? 2 : 1;
}

// The geometry of a query about sizes alone (no tensors): total_tokens > 0 marks a packed
// batch, whose block counts need only T and B, so a non-null stand-in takes cu_seqlens'
// place.  False where the sizes are invalid (the calls would fail).
bool query_geometry(int B, int Hq, int Hkv, int N, int d, int causal, int window,
                    int total_tokens, Geometry* g) {
    static const int kPacked = 0;
    return check_common(B, Hq, Hkv, N, d, causal, window, total_tokens > 0 ? &kPacked : nullptr,
                        total_tokens, 1.f, g) == FA_OK;
}

fa_status check_dtype(fa_dtype dtype, const char* who) {
    if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16)
        return fail(FA_ERR_UNSUPPORTED, "%s: element type %d is neither FA_DTYPE_BF16 nor FA_DTYPE_F16",
                    who, static_cast<int>(dtype));
    return FA_OK;
}

// the kernels' element-type codes are the ABI's
static_assert(FA_DTYPE_BF16 == kElemBf16Code && FA_DTYPE_F16 == kElemF16Code, "element codes");

// Dropout parameters of a call: a pair is dropped with probability thresh / 256,
// thresh = round(256 p_drop) (p_drop as float; see fa_fwd_dropout in fa.h).
fa_status make_dropout(float p_drop, unsigned long long seed, unsigned int offset,
                       DropoutParams* d, const char* who) {
    if (!(p_drop >= 0.f) || !(p_drop < 1.f))
        return fail(FA_ERR_INVALID_ARG, "%s: p_drop must be in [0, 1) (got %g)", who,
                    static_cast<double>(p_drop));
    const float t = std::floor(p_drop * 256.0f + 0.5f);
    if (t > 255.f)
        return fail(FA_ERR_UNSUPPORTED, "%s: p_drop %g rounds to 256/256; the largest is 255/256",
                    who, static_cast<double>(p_drop));
    d->thresh = static_cast<uint32_t>(t);
    d->rscale = 256.0f / static_cast<float>(256u - d->thresh);
    d->seed_lo = static_cast<uint32_t>(seed & 0xffffffffull);
    d->seed_hi = static_cast<uint32_t>(seed >> 32);
    d->offset = offset;
    return FA_OK;
}

fa_status fwd_impl(fa_dtype dtype, const DropoutParams& drop, const void* q, const void* k,
                   const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N, int d,
                   int causal, int window, const int* cu_seqlens, int total_tokens, float scale,
                   cudaStream_t stream);
fa_status bwd_impl(fa_dtype dtype, const DropoutParams& drop, const void* q, const void* k,
                   const void* v, const void* o, const float* lse, const void* dout, void* dq,
                   void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal,
                   int window, const int* cu_seqlens, int total_tokens, float scale,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

}  // namespace

int* device_status_word() { return status_word_ptr(); }

fa_status report_error(fa_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return st;
}

// Workspace of the backward pass for these sizes (false for invalid ones): the
// fp32 row statistics D, then (fused backward only) the fp32 row scales, the
// K/V bound slots and the int32 dQ accumulator; each part padded to 256 bytes.
bool bwd_workspace(int B, int Hq, int Hkv, int N, int d, int total_tokens, BwdWorkspace* w) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || (d != 64 && d != 128) || total_tokens < 0)
        return false;
    auto pad = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    // rows of the token dimension: packed T (total_tokens > 0); dense B * N
    const long long rows = total_tokens > 0 ? total_tokens : static_cast<long long>(B) * N;
    w->delta = pad(static_cast<size_t>(rows) * Hq * sizeof(float));
    w->scale_offset = w->delta;
    w->bound_offset = w->scale_offset + w->delta;
    w->acc_offset = w->bound_offset + pad(static_cast<size_t>(Hkv) * kBoundSlots * (d + 1) * sizeof(float));
    w->full = w->acc_offset + pad(static_cast<size_t>(rows) * Hq * d * sizeof(int));
    return true;
}

// The backward fa_bwd runs by default for head dimension d when the workspace allows
// the fused one (the path measured faster on GB300, with and without a causal mask).
bool prefer_fused(int d) { return d == 64; }

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_last_error(void) { return t_last_error; }

void fa_set_launch_events(const cudaEvent_t* events, int count) {
    t_events = (events && count > 0) ? events : nullptr;
    t_event_count = t_events ? count : 0;
}

void fa_set_wait_limit_cycles(long long cycles) {
    g_wait_limit.store(cycles > 0 ? cycles : kDefaultTimeoutCycles);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int N, int d, int causal, int window, const int* cu_seqlens,
                 int total_tokens, float scale, cudaStream_t stream) {
    return fa_fwd_typed(FA_DTYPE_BF16, q, k, v, o, lse, B, Hq, Hkv, N, d, causal, window,
                        cu_seqlens, total_tokens, scale, stream);
}

fa_status fa_fwd_typed(fa_dtype dtype, const void* q, const void* k, const void* v, void* o,
                       float* lse, int B, int Hq, int Hkv, int N, int d, int causal, int window,
                       const int* cu_seqlens, int total_tokens, float scale, cudaStream_t stream) {
    t_last_error[0] = '\0';
    const DropoutParams none{};
    return fwd_impl(dtype, none, q, k, v, o, lse, B, Hq, Hkv, N, d, causal, window, cu_seqlens,
                    total_tokens, scale, stream);
}

fa_status fa_fwd_dropout(fa_dtype dtype, float p_drop, unsigned long long seed,
                         unsigned int offset, const void* q, const void* k, const void* v, void* o,
                         float* lse, int B, int Hq, int Hkv, int N, int d, int causal, int window,
                         const int* cu_seqlens, int total_tokens, float scale,
                         cudaStream_t stream) {
    t_last_error[0] = '\0';
    DropoutParams drop{};
    const fa_status st = make_dropout(p_drop, seed, offset, &drop, "fa_fwd_dropout");
    if (st != FA_OK) return st;
    return fwd_impl(dtype, drop, q, k, v, o, lse, B, Hq, Hkv, N, d, causal, window, cu_seqlens,
                    total_tokens, scale, stream);
}

}  // extern "C"

namespace fa {
namespace {

fa_status fwd_impl(fa_dtype dtype, const DropoutParams& drop, const void* q, const void* k,
                   const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N, int d,
                   int causal, int window, const int* cu_seqlens, int total_tokens, float scale,
                   cudaStream_t stream) {
    const cudaEvent_t* ev = nullptr;
    if (take_events(1, &ev) != FA_OK)
        return fail(FA_ERR_INVALID_ARG, "fa_fwd: fa_set_launch_events needs >= 2 events");
    if (!q || !k || !v || !o || !lse)
        return fail(FA_ERR_INVALID_ARG, "fa_fwd: q, k, v, o and lse must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return fail(FA_ERR_INVALID_ARG, "fa_fwd: tensors must be 16-byte aligned");
    fa_status st = check_dtype(dtype, "fa_fwd");
    if (st != FA_OK) return st;
    Geometry g;
    st = check_common(B, Hq, Hkv, N, d, causal, window, cu_seqlens, total_tokens, scale, &g);
    if (st != FA_OK) return st;
    if (drop.thresh == 0 && t_fwd_heads > 0 && Hq % t_fwd_heads != 0)
        return fail(FA_ERR_INVALID_ARG, "fa_fwd: %d query heads per CTA (fa_fwd_set_heads) do not "
                    "divide Hq = %d", t_fwd_heads, Hq);
    if (g.tokens == 0) return FA_OK;

    FwdParams p;
    if ((st = make_token_map(&p.tm_q, q, g.tokens, Hq, d, dtype, "q")) != FA_OK) return st;
    if ((st = make_token_map(&p.tm_k, k, g.tokens, Hkv, d, dtype, "k")) != FA_OK) return st;
    if ((st = make_token_map(&p.tm_v, v, g.tokens, Hkv, d, dtype, "v")) != FA_OK) return st;
    if ((st = make_token_map(&p.tm_o, o, g.tokens, Hq, d, dtype, "o")) != FA_OK) return st;
    p.elem = static_cast<int>(dtype);
    p.drop = drop;
    p.seq = g.seq;
    p.o = o;
    p.lse = lse;
    p.scale_log2 = scale * kLog2e;
    // several query heads per CTA for the 16-bit forward without dropout
    p.heads = drop.thresh != 0 ? 1 : t_fwd_heads > 0 ? t_fwd_heads : fwd_heads_per_cta(g, Hq, Hkv);
    p.num_work = num_blocks(g, kFwdQTiles * kBlockM, Hq / p.heads);
    p.timeout_cycles = g_wait_limit.load();
    p.status = status_word_ptr();
    if (!p.status) return fail(FA_ERR_CUDA, "fa_fwd: cannot resolve the device status word");
    cudaError_t e = record(ev, 0, stream);
    if (e == cudaSuccess) e = launch_fwd(p, d, stream);
    if (e == cudaSuccess) e = record(ev, 1, stream);
    if (e != cudaSuccess) return cuda_fail(e, "fa_fwd launch");
    return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

size_t fa_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d, int total_tokens) {
    fa::BwdWorkspace w;
    if (!fa::bwd_workspace(B, Hq, Hkv, N, d, total_tokens, &w)) return 0;
    return fa::prefer_fused(d) ? w.full : w.delta;
}

size_t fa_bwd_workspace_size_min(int B, int Hq, int Hkv, int N, int d, int total_tokens) {
    fa::BwdWorkspace w;
    return fa::bwd_workspace(B, Hq, Hkv, N, d, total_tokens, &w) ? w.delta : 0;
}

size_t fa_bwd_workspace_size_fused(int B, int Hq, int Hkv, int N, int d, int total_tokens) {
    fa::BwdWorkspace w;
    return fa::bwd_workspace(B, Hq, Hkv, N, d, total_tokens, &w) ? w.full : 0;
}

void fa_bwd_set_path(int path) {
    t_bwd_path = (path == FA_BWD_SPLIT || path == FA_BWD_FUSED) ? path : FA_BWD_AUTO;
}

fa_status fa_fwd_set_heads(int heads) {
    t_last_error[0] = '\0';
    if (heads < 0) return fa::fail(FA_ERR_INVALID_ARG, "fa_fwd_set_heads: heads = %d < 0", heads);
    t_fwd_heads = heads;
    return FA_OK;
}

fa_status fa_bwd_set_dq_heads(int heads) {
    t_last_error[0] = '\0';
    if (heads < 0) return fa::fail(FA_ERR_INVALID_ARG, "fa_bwd_set_dq_heads: heads = %d < 0", heads);
    t_dq_heads = heads;
    return FA_OK;
}

int fa_fwd_heads(int B, int Hq, int Hkv, int N, int d, int causal, int window, int total_tokens) {
    fa::Geometry g;
    if (!fa::query_geometry(B, Hq, Hkv, N, d, causal, window, total_tokens, &g)) return -1;
    if (t_fwd_heads > 0) return Hq % t_fwd_heads == 0 ? t_fwd_heads : -1;
    return fa::fwd_heads_per_cta(g, Hq, Hkv);
}

int fa_bwd_dq_heads(int B, int Hq, int Hkv, int N, int d, int causal, int window, int total_tokens) {
    fa::Geometry g;
    if (!fa::query_geometry(B, Hq, Hkv, N, d, causal, window, total_tokens, &g)) return -1;
    if (t_dq_heads > 0) return (Hq / Hkv) % t_dq_heads == 0 ? t_dq_heads : -1;
    return fa::heads_per_cta(g, kBlockM, Hq, Hkv);
}

int fa_bwd_path(int B, int Hq, int Hkv, int N, int d, int causal, int window, int total_tokens,
                size_t workspace_bytes) {
    fa::BwdWorkspace w;
    if (!fa::bwd_workspace(B, Hq, Hkv, N, d, total_tokens, &w) || workspace_bytes < w.delta)
        return -1;
    (void)causal;
    (void)window;
    const bool can_fuse = workspace_bytes >= w.full;
    if (t_bwd_path == FA_BWD_SPLIT) return FA_BWD_SPLIT;
    if (t_bwd_path == FA_BWD_FUSED) return can_fuse ? FA_BWD_FUSED : -1;
    return (can_fuse && fa::prefer_fused(d)) ? FA_BWD_FUSED : FA_BWD_SPLIT;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                 int d, int causal, int window, const int* cu_seqlens, int total_tokens,
                 float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return fa_bwd_typed(FA_DTYPE_BF16, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal,
                        window, cu_seqlens, total_tokens, scale, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_typed(fa_dtype dtype, const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int N, int d, int causal, int window,
                       const int* cu_seqlens, int total_tokens, float scale, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
    t_last_error[0] = '\0';
    const DropoutParams none{};
    return bwd_impl(dtype, none, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal,
                    window, cu_seqlens, total_tokens, scale, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_dropout(fa_dtype dtype, float p_drop, unsigned long long seed,
                         unsigned int offset, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout, void* dq, void* dk,
                         void* dv, int B, int Hq, int Hkv, int N, int d, int causal, int window,
                         const int* cu_seqlens, int total_tokens, float scale, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
    t_last_error[0] = '\0';
    DropoutParams drop{};
    const fa_status st = make_dropout(p_drop, seed, offset, &drop, "fa_bwd_dropout");
    if (st != FA_OK) return st;
    return bwd_impl(dtype, drop, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal,
                    window, cu_seqlens, total_tokens, scale, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace fa {
namespace {

fa_status bwd_impl(fa_dtype dtype, const DropoutParams& drop, const void* q, const void* k,
                   const void* v, const void* o, const float* lse, const void* dout, void* dq,
                   void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal,
                   int window, const int* cu_seqlens, int total_tokens, float scale,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    // the events armed for this call are used up by it, whatever happens
    const cudaEvent_t* ev = nullptr;
    int ev_count = 0;
    take_events_any(&ev, &ev_count);
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv)
        return fail(FA_ERR_INVALID_ARG, "fa_bwd: tensor pointers must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return fail(FA_ERR_INVALID_ARG, "fa_bwd: tensors must be 16-byte aligned");
    fa_status st = check_dtype(dtype, "fa_bwd");
    if (st != FA_OK) return st;
    Geometry g;
    st = check_common(B, Hq, Hkv, N, d, causal, window, cu_seqlens, total_tokens, scale, &g);
    if (st != FA_OK) return st;
    BwdWorkspace wl;
    bwd_workspace(B, Hq, Hkv, N, d, cu_seqlens ? total_tokens : 0, &wl);
    if (!workspace || workspace_bytes < wl.delta)
        return fail(FA_ERR_WORKSPACE, "fa_bwd: workspace of at least %zu bytes needed (%zu for the "
                    "fused backward), got %zu%s", wl.delta, wl.full, workspace_bytes,
                    workspace ? "" : " (null)");
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(FA_ERR_WORKSPACE, "fa_bwd: workspace must be 256-byte aligned");
    // the fused backward (one tensor-core kernel, any mask) when the workspace holds
    // its dQ accumulator and the thread's preference allows it; otherwise the split
    // backward (dK/dV, then dQ)
    const bool can_fuse = workspace_bytes >= wl.full;
    if (t_bwd_path == FA_BWD_FUSED && !can_fuse)
        return fail(FA_ERR_WORKSPACE, "fa_bwd: the fused backward needs a workspace of %zu bytes, got %zu",
                    wl.full, workspace_bytes);
    const bool fused = t_bwd_path == FA_BWD_FUSED ||
                       (t_bwd_path == FA_BWD_AUTO && can_fuse && prefer_fused(d));
    if (!fused && drop.thresh == 0 && t_dq_heads > 0 && (Hq / Hkv) % t_dq_heads != 0)
        return fail(FA_ERR_INVALID_ARG, "fa_bwd: %d query heads per dQ CTA (fa_bwd_set_dq_heads) do "
                    "not divide the group of %d", t_dq_heads, Hq / Hkv);
    const int kernels = 3;
    if (ev && ev_count < kernels + 1)
        return fail(FA_ERR_INVALID_ARG, "fa_bwd: fa_set_launch_events needs >= %d events", kernels + 1);
    if (g.tokens == 0) return FA_OK;

    BwdParams p;
    if ((st = make_token_map(&p.tm_q, q, g.tokens, Hq, d, dtype, "q")) != FA_OK) return st;
    if ((st = make_token_map(&p.tm_k, k, g.tokens, Hkv, d, dtype, "k")) != FA_OK) return st;
    if ((st = make_token_map(&p.tm_v, v, g.tokens, Hkv, d, dtype, "v")) != FA_OK) return st;
    if ((st = make_token_map(&p.tm_do, dout, g.tokens, Hq, d, dtype, "dout")) != FA_OK) return st;
    if ((st = make_token_map(&p.tm_dq, dq, g.tokens, Hq, d, dtype, "dq")) != FA_OK) return st;
    if ((st = make_token_map(&p.tm_dk, dk, g.tokens, Hkv, d, dtype, "dk")) != FA_OK) return st;
    if ((st = make_token_map(&p.tm_dv, dv, g.tokens, Hkv, d, dtype, "dv")) != FA_OK) return st;
    p.elem = static_cast<int>(dtype);
    p.drop = drop;
    p.seq = g.seq;
    p.q = q;
    p.o = o;
    p.dout = dout;
    p.lse = lse;
    p.delta = static_cast<float*>(workspace);
    p.k_ptr = k;
    p.v_ptr = v;
    p.dq_acc = nullptr;
    p.row_scale = nullptr;
    p.kv_bound = nullptr;
    if (fused) {
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        p.row_scale = reinterpret_cast<float*>(ws + wl.scale_offset);
        p.kv_bound = reinterpret_cast<float*>(ws + wl.bound_offset);
        p.dq_acc = reinterpret_cast<int*>(ws + wl.acc_offset);
    }
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    // several query heads per dQ CTA for the backward without dropout
    p.dq_heads = drop.thresh != 0 ? 1 : t_dq_heads > 0 ? t_dq_heads : heads_per_cta(g, kBlockM, Hq, Hkv);
    p.num_work_dq = num_blocks(g, kBlockM, Hq / p.dq_heads);
    p.num_work_dkdv = num_blocks(g, kBlockN, Hkv);
    p.timeout_cycles = g_wait_limit.load();
    p.status = status_word_ptr();
    if (!p.status) return fail(FA_ERR_CUDA, "fa_bwd: cannot resolve the device status word");
    p.pre_row_ctas = bwd_preprocess_row_ctas(p, d);
    cudaError_t e = record(ev, 0, stream);
    if (e == cudaSuccess) e = launch_bwd_preprocess(p, d, stream);
    if (e == cudaSuccess) e = record(ev, 1, stream);
    if (e != cudaSuccess) return cuda_fail(e, "fa_bwd preprocess launch");
    if (fused) {
        e = launch_bwd_fused(p, d, stream);
        if (e == cudaSuccess) e = record(ev, 2, stream);
        if (e != cudaSuccess) return cuda_fail(e, "fa_bwd fused launch");
        e = launch_bwd_dq_convert(p, d, stream);
        if (e == cudaSuccess) e = record(ev, 3, stream);
        if (e != cudaSuccess) return cuda_fail(e, "fa_bwd dq conversion launch");
        return FA_OK;
    }
    e = launch_bwd_dkdv(p, d, stream);
    if (e == cudaSuccess) e = record(ev, 2, stream);
    if (e != cudaSuccess) return cuda_fail(e, "fa_bwd dk/dv launch");
    e = launch_bwd_dq(p, d, stream);
    if (e == cudaSuccess) e = record(ev, 3, stream);
    if (e != cudaSuccess) return cuda_fail(e, "fa_bwd dq launch");
    return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_device_status(cudaStream_t stream) {
    t_last_error[0] = '\0';
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "fa_device_status: stream synchronisation");
    int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "fa_device_status: reading the status word");
    if (word != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "fa_device_status: clearing the status word");
        if (word == 5)
            return fail(FA_ERR_TIMEOUT, "a kernel gave up a bounded wait (device status %d)", word);
        if (word == 7)
            return fail(FA_ERR_CUDA, "a kernel of the bounds-checking build found a global index "
                        "out of its tensor and skipped the access (device status %d)", word);
        return fail(FA_ERR_CUDA, "a kernel reported device status %d (misaligned shared memory)",
                    word);
    }
    return FA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ fp8 forward

namespace fa {
namespace {

// [tokens, heads, d] e4m3 viewed as (d, heads, tokens); the box is one 128-byte row
// of d (d = 128) x 1 head x 128 tokens.
fa_status make_u8_token_map(CUtensorMap* map, const void* base, int tokens, int heads, int d,
                            const char* name) {
    auto enc = encode_fn();
    if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                          static_cast<cuuint64_t>(tokens)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads) * d};
    cuuint32_t box[3] = {128, 1, static_cast<cuuint32_t>(kBlockM)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name,
                    static_cast<int>(r));
    return FA_OK;
}

// V^T [heads, d, vt_tokens] e4m3 viewed as (vt_tokens, d, heads); the box is 128 keys
// (one 128-byte row) x 128 rows of d x 1 head.
fa_status make_vt_map(CUtensorMap* map, const void* base, int vt_tokens, int d, int heads) {
    auto enc = encode_fn();
    if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(vt_tokens), static_cast<cuuint64_t>(d),
                          static_cast<cuuint64_t>(heads)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(vt_tokens),
                             static_cast<cuuint64_t>(d) * vt_tokens};
    cuuint32_t box[3] = {128, static_cast<cuuint32_t>(d), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(vt) failed with CUresult %d",
                    static_cast<int>(r));
    return FA_OK;
}

// Columns of the fp8 block-scale arrays: exact for dense batches (B ceil(N / 128));
// packed, the column space of seq_block_col: ceil(T / 128) + B.
long long fp8_blocks(int B, int N, int total_tokens, bool packed) {
    if (!packed) return static_cast<long long>(B) * ((static_cast<long long>(N) + 127) / 128);
    // packed: sequence b's blocks start at column floor(cu_seqlens[b] / 128) + b
    return (static_cast<long long>(total_tokens) + 127) / 128 + B;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

fa_status fp8_geometry(int B, int H, int N, int d, const int* cu_seqlens, int total_tokens,
                       const char* who, Geometry* g) {
    if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "%s: head dim %d not in {64, 128}", who, d);
    return check_common(B, H, H, N, d, 0, 0, cu_seqlens, total_tokens, 1.f, g);
}

fa_status fp8_quantize_qk(const char* name, bool rotate, unsigned long long seed, const void* x,
                          void* x8, float* scales, int nb, int B, int H, int N, int d,
                          const int* cu_seqlens, int total_tokens, cudaStream_t stream) {
    t_last_error[0] = '\0';
    if (!x || !x8 || !scales)
        return fail(FA_ERR_INVALID_ARG, "%s: x, x8 and scales must be non-null", name);
    if (!aligned16(x) || !aligned16(x8) || !aligned4(scales))
        return fail(FA_ERR_INVALID_ARG,
                    "%s: x and x8 must be 16-byte aligned, scales 4-byte aligned", name);
    Geometry g;
    fa_status st = fp8_geometry(B, H, N, d, cu_seqlens, total_tokens, name, &g);
    if (st != FA_OK) return st;
    if (nb < fp8_blocks(B, N, g.tokens, cu_seqlens != nullptr))
        return fail(FA_ERR_INVALID_ARG, "%s: nb = %d below fa_fp8_scale_blocks", name, nb);
    if (g.tokens == 0) return FA_OK;
    Fp8QuantParams p{};
    p.seq = g.seq;
    p.x = x;
    p.out = x8;
    p.scales = scales;
    p.heads = H;
    p.status = status_word_ptr();
    if (!p.status) return fail(FA_ERR_CUDA, "fp8 quantisation: cannot resolve the device status word");
    p.nb = nb;
    p.rotate = rotate ? 1 : 0;
    p.seed_lo = static_cast<uint32_t>(seed);
    p.seed_hi = static_cast<uint32_t>(seed >> 32);
    const cudaError_t e = launch_fp8_quant_qk(p, d, num_blocks(g, kBlockM, H), stream);
    if (e != cudaSuccess) return fail(FA_ERR_CUDA, "%s launch: %s", name, cudaGetErrorString(e));
    return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_fp8_scale_blocks(int B, int N, int total_tokens, int packed) {
    if (B < 1 || N < 1 || total_tokens < 0) return 0;
    const long long nb = fa::fp8_blocks(B, N, total_tokens, packed != 0);
    return nb > INT_MAX ? 0 : static_cast<int>(nb);
}

int fa_fp8_vt_tokens(int B, int N, int total_tokens, int packed) {
    if (B < 1 || N < 1 || total_tokens < 0) return 0;
    const long long t = 128 * fa::fp8_blocks(B, N, total_tokens, packed != 0);
    return t > INT_MAX / 2 ? 0 : static_cast<int>(t);
}

fa_status fa_fp8_quantize_qk(const void* x, void* x8, float* scales, int nb, int B, int H, int N,
                             int d, const int* cu_seqlens, int total_tokens, cudaStream_t stream) {
    return fa::fp8_quantize_qk("fa_fp8_quantize_qk", false, 0, x, x8, scales, nb, B, H, N, d,
                           cu_seqlens, total_tokens, stream);
}

fa_status fa_fp8_quantize_qk_incoherent(const void* x, void* x8, float* scales, int nb, int B,
                                        int H, int N, int d, const int* cu_seqlens,
                                        int total_tokens, unsigned long long seed,
                                        cudaStream_t stream) {
    return fa::fp8_quantize_qk("fa_fp8_quantize_qk_incoherent", true, seed, x, x8, scales, nb, B, H,
                           N, d, cu_seqlens, total_tokens, stream);
}

fa_status fa_fp8_quantize_v(const void* v, void* vt8, float* scales, int vt_tokens, int B, int H,
                            int N, int d, const int* cu_seqlens, int total_tokens,
                            cudaStream_t stream) {
    using namespace fa;
    t_last_error[0] = '\0';
    if (!v || !vt8 || !scales)
        return fail(FA_ERR_INVALID_ARG, "fa_fp8_quantize_v: v, vt8 and scales must be non-null");
    if (!aligned16(v) || !aligned16(vt8) || !aligned4(scales))
        return fail(FA_ERR_INVALID_ARG,
                    "fa_fp8_quantize_v: v and vt8 must be 16-byte aligned, scales 4-byte aligned");
    Geometry g;
    fa_status st = fp8_geometry(B, H, N, d, cu_seqlens, total_tokens, "fa_fp8_quantize_v", &g);
    if (st != FA_OK) return st;
    if (vt_tokens % 128 != 0 || vt_tokens < 128 * fp8_blocks(B, N, g.tokens, cu_seqlens != nullptr))
        return fail(FA_ERR_INVALID_ARG,
                    "fa_fp8_quantize_v: vt_tokens = %d must be a multiple of 128 and at least "
                    "fa_fp8_vt_tokens", vt_tokens);
    if (g.tokens == 0) return FA_OK;
    Fp8QuantParams p{};
    p.seq = g.seq;
    p.x = v;
    p.out = vt8;
    p.scales = scales;
    p.heads = H;
    p.status = status_word_ptr();
    if (!p.status) return fail(FA_ERR_CUDA, "fp8 quantisation: cannot resolve the device status word");
    p.vt_tokens = vt_tokens;
    const cudaError_t e = launch_fp8_quant_v(p, d, num_blocks(g, kBlockN, H), stream);
    if (e != cudaSuccess) return cuda_fail(e, "fa_fp8_quantize_v launch");
    return FA_OK;
}

fa_status fa_fwd_fp8(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                     const void* vt8, const float* v_scale, int nb, int vt_tokens, void* o,
                     float* lse, int B, int Hq, int Hkv, int N, int d, int causal, int window,
                     const int* cu_seqlens, int total_tokens, float scale, cudaStream_t stream) {
    using namespace fa;
    t_last_error[0] = '\0';
    const cudaEvent_t* ev = nullptr;
    if (take_events(1, &ev) != FA_OK)
        return fail(FA_ERR_INVALID_ARG, "fa_fwd_fp8: fa_set_launch_events needs >= 2 events");
    if (!q8 || !k8 || !vt8 || !q_scale || !k_scale || !v_scale || !o || !lse)
        return fail(FA_ERR_INVALID_ARG, "fa_fwd_fp8: every pointer must be non-null");
    if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o) || !aligned16(lse) ||
        !aligned4(q_scale) || !aligned4(k_scale) || !aligned4(v_scale))
        return fail(FA_ERR_INVALID_ARG,
                    "fa_fwd_fp8: tensors must be 16-byte aligned, scales 4-byte aligned");
    if (d != 128) return fail(FA_ERR_UNSUPPORTED, "fa_fwd_fp8: head dim %d (only 128)", d);
    Geometry g;
    fa_status st = check_common(B, Hq, Hkv, N, d, causal, window, cu_seqlens, total_tokens, scale, &g);
    if (st != FA_OK) return st;
    const long long blocks = fp8_blocks(B, N, g.tokens, cu_seqlens != nullptr);
    if (nb < blocks) return fail(FA_ERR_INVALID_ARG, "fa_fwd_fp8: nb = %d below fa_fp8_scale_blocks", nb);
    if (vt_tokens % 128 != 0 || vt_tokens < 128 * blocks)
        return fail(FA_ERR_INVALID_ARG,
                    "fa_fwd_fp8: vt_tokens = %d must be a multiple of 128 and at least "
                    "fa_fp8_vt_tokens", vt_tokens);
    if (g.tokens == 0) return FA_OK;

    FwdParams p;
    if ((st = make_u8_token_map(&p.tm_q, q8, g.tokens, Hq, d, "q8")) != FA_OK) return st;
    if ((st = make_u8_token_map(&p.tm_k, k8, g.tokens, Hkv, d, "k8")) != FA_OK) return st;
    if ((st = make_vt_map(&p.tm_v, vt8, vt_tokens, d, Hkv)) != FA_OK) return st;
    if ((st = make_token_map(&p.tm_o, o, g.tokens, Hq, d, FA_DTYPE_BF16, "o")) != FA_OK) return st;
    p.elem = kElemFp8Code;
    p.drop = DropoutParams{};
    p.q_scale = q_scale;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.nb = nb;
    p.seq = g.seq;
    p.o = o;
    p.lse = lse;
    p.scale_log2 = scale * kLog2e;
    p.heads = 1;
    p.num_work = num_blocks(g, kFwdQTiles * kBlockM, Hq);
    p.timeout_cycles = g_wait_limit.load();
    p.status = status_word_ptr();
    if (!p.status) return fail(FA_ERR_CUDA, "fa_fwd_fp8: cannot resolve the device status word");
    cudaError_t e = record(ev, 0, stream);
    if (e == cudaSuccess) e = launch_fwd(p, d, stream);
    if (e == cudaSuccess) e = record(ev, 1, stream);
    if (e != cudaSuccess) return cuda_fail(e, "fa_fwd_fp8 launch");
    return FA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ debug checks

namespace fa {
namespace {

// One thread tests an index one past a three-element range: a build with the bounds
// checks records kDevBadIndex; no memory is touched either way.
__global__ void debug_check_selftest_kernel(int* status) {
    (void)fa_index_ok(3, 3, status);
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_debug_checks_enabled(void) {
#ifdef FA_DEBUG_CHECKS
    return 1;
#else
    return 0;
#endif
}

fa_status fa_debug_check_selftest(cudaStream_t stream) {
    using namespace fa;
    t_last_error[0] = '\0';
    if (!fa_debug_checks_enabled())
        return fail(FA_ERR_UNSUPPORTED, "fa_debug_check_selftest: not a bounds-checking build");
    int* st = status_word_ptr();
    if (!st) return fail(FA_ERR_CUDA, "fa_debug_check_selftest: cannot resolve the device status word");
    debug_check_selftest_kernel<<<1, 1, 0, stream>>>(st);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "fa_debug_check_selftest launch");
    return FA_OK;
}

}  // extern "C"
