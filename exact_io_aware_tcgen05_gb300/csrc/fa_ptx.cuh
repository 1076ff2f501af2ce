// fa_ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the attention
// kernels are built on: mbarriers, TMA tensor loads, tcgen05 (TMEM allocation,
// MMA, commit, TMEM loads/stores) and the shared-memory / instruction
// descriptors of tcgen05.mma.  Nothing here is attention-specific.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace fa {

// ------------------------------------------------------------------ basics

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ bool elect_lane0() { return lane_id() == 0; }

// Device-wide status word, written (never read) by kernels when a bounded wait
// gives up (kDevTimeout), a launch finds its shared memory misaligned
// (kDevBadSmem), or -- in a build with FA_DEBUG_CHECKS -- a computed global index
// or TMA store box falls outside its tensor (kDevBadIndex).  Host code reads it
// with fa_device_status().
enum : int { kDevOk = 0, kDevTimeout = 5, kDevBadSmem = 6, kDevBadIndex = 7 };

// Bounds checks of the debug build.  With FA_DEBUG_CHECKS defined, fa_index_ok
// tests 0 <= idx < size; a failing check records kDevBadIndex and the caller skips
// the access (nothing traps).  Without it the checks are compiled away.
#ifdef FA_DEBUG_CHECKS
__device__ __forceinline__ bool fa_index_ok(long long idx, long long size, int* status) {
    if (idx >= 0 && idx < size) return true;
    atomicExch(status, kDevBadIndex);
    return false;
}
#else
__device__ __forceinline__ bool fa_index_ok(long long, long long, int*) { return true; }
#endif

// A TMA store box of `rows` token rows from `row` and one head: it must lie inside
// [0, tokens) x [0, heads) (stores may not start at negative coordinates).
__device__ __forceinline__ bool fa_box_ok(long long row, int rows, long long tokens, int head,
                                          int heads, int* status) {
    return fa_index_ok(row, tokens - rows + 1, status) && fa_index_ok(head, heads, status);
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on phase `parity` of an mbarrier.  Gives up (returns false) when
// `*abort` becomes non-zero or after `limit` SM clock cycles; in the latter
// case it raises the CTA-wide abort flag and the device status word, so the
// other roles of the CTA stop waiting too.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          long long limit, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit) {
            *abort = 1;
            atomicExch(status, kDevTimeout);
            return false;
        }
    }
}

// Cycle budget of the teardown drains below (about 1 s): independent of the
// configurable wait limit, so a short limit never lets a CTA exit while its
// own copies or MMAs are still in flight.
constexpr long long kDrainCycles = 2000000000LL;

// Wait used only while tearing down: ignores the abort flag and gives up
// silently after `limit` cycles.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

// ------------------------------------------------------------ named barriers
//
// Hardware barrier `id` (1..15; 0 is __syncthreads) that completes when `count`
// threads have arrived; whole warps take part (warp-collective).  They link the
// tcgen05 issuer with the warps feeding it: an mbarrier wait is a shared-memory
// load, and a shared-memory load by the issuing warp holds back the MMAs it
// issues next until those already in flight have drained.  A named barrier
// does not.

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void named_bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ANDs a predicate over its `count` threads: every
// participant gets the same verdict (a way to make a choice uniform).
__device__ __forceinline__ bool named_bar_all(int id, int count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pin, pout;\n\t"
        "setp.ne.u32 pin, %1, 0;\n\t"
        "bar.red.and.pred pout, %2, %3, pin;\n\t"
        "selp.u32 %0, 1, 0, pout;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// A producer warp's signal: arrive while running normally; once it has given up
// (`live` false, warp-uniform) it blocks instead, so a warp that skips its work
// can never get a phase ahead of the barrier's other participants.
__device__ __forceinline__ void named_bar_signal(int id, int count, bool live) {
    if (live) named_bar_arrive(id, count);
    else named_bar_sync(id, count);
}

// ---------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled prefetch of one box into L2: no shared memory, no completion signal.  The
// coordinates follow the rules of a load (x (c0) * element size a multiple of 16 bytes;
// rows past the tensor's end are allowed).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// 3-D tiled load; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Same, with an L2 eviction-priority policy (from make_l2_policy_*).
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int c0, int c1, int c2,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
        : "memory");
}

// 3-D tiled store shared -> global, tracked by the thread's bulk groups.  The
// shared tile uses the tensor map's layout (128-byte swizzle); the coordinates
// must not be negative and x (c0) * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every bulk store this thread committed has finished reading shared
// memory (the source may then be reused, or the CTA exit).
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Orders this thread's earlier shared-memory writes before later async-proxy
// (TMA) accesses issued after a thread synchronisation.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t make_l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t make_l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------- register budgets
//
// setmaxnreg: every warp of a warpgroup lowers (or raises) its per-thread
// register count to N together, moving registers between the warpgroups of a
// CTA.  A raise waits until the registers are free, so the counts summed over
// the CTA's threads must not exceed what the launch reserved (threads x the
// kernel's register count); the launcher checks the kernel's count.

template <int N>
__device__ __forceinline__ void regs_lower() {
    static_assert(N % 8 == 0 && N >= 24 && N <= 256, "register count");
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void regs_raise() {
    static_assert(N % 8 == 0 && N >= 24 && N <= 256, "register count");
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ tcgen05

// TMEM allocation: executed by one full warp; the base address is written to
// shared memory at `dst`.  ncols is a power of two in [32, 512].
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]  (bf16 x bf16 -> f32, shape from idesc)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on `bar` when all previously issued tcgen05 async ops of this
// thread have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// TMEM -> registers, 32 lanes x 32 consecutive 32-bit columns: thread t of the
// warp receives lane (lane_base + t), columns col .. col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// 16-column variant.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Registers filled by tmem_ld* are valid only after tmem_ld_wait(); passing
// them through this empty asm after the wait keeps the compiler from moving
// their uses above it.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// The same products on e4m3 operands (kind::f8f6f4; K = 32 per instruction;
// the instruction descriptor's A and B format fields 0 = E4M3).
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                     taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------- programmatic dependent launch

// Lets grids launched as programmatic dependents of this grid start once every
// CTA of this grid has executed this (or exited).
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Blocks until the grids this grid programmatically depends on have completed
// and their memory operations are visible.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------- global reductions

// *p += v in L2 (32-bit integer), no return value
__device__ __forceinline__ void red_add_s32(int* p, int v) {
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle (the
// layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).  Fields: start address
// >> 4 in bits 0-13, leading-dimension byte offset >> 4 in bits 16-29,
// stride-dimension byte offset >> 4 in bits 32-45, fixed version 1 in bits
// 46-47, base offset 0 (tiles are 1024-byte aligned), swizzle mode 2
// (128B) in bits 61-63.
//   K-major operand: rows of 128 bytes, 8-row core groups `sbo` bytes apart;
//                    `lbo` unused.
//   MN-major operand: `lbo` = bytes between 64-element column blocks along
//                    M/N, `sbo` = bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Element type of the operands and outputs (accumulation is always fp32); the
// codes of the C ABI's fa_dtype.
constexpr int kElemBf16 = 0;
constexpr int kElemF16 = 1;
constexpr int kElemFp8 = 2;   // e4m3 operands (kind::f8f6f4), bf16 output

// Instruction descriptor of tcgen05.mma.kind::f16 with an f32 accumulator and
// A, B both of element type `elem`: D format bits 4-5 = 1 (f32), A format bits
// 7-9 and B format bits 10-12 (1 = bf16, 0 = fp16; one kind::f16 product takes
// one type for both), A / B major bits 15 / 16 (0 = K-major, 1 = MN-major),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f32acc(int M, int N, bool a_mn_major,
                                                    bool b_mn_major, int elem) {
    return (1u << 4) | ((elem == kElemBf16 ? 1u : 0u) << 7) |
           ((elem == kElemBf16 ? 1u : 0u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// -------------------------------------------------------------- conversions

// Two fp32 values rounded (to nearest even) to element type E and packed, `lo`
// in the low half.
template <int E>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    // cvt packs its first source operand into the upper half.
    if (E == kElemBf16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Row r of a [128 rows x 64 elements] 16-bit tile in the 128-byte-swizzled layout
// TMA uses: 16-byte unit u of the row sits at unit position u ^ (r % 8).
__device__ __forceinline__ uint4* swizzled_unit(uint8_t* tile, int r, int u) {
    return reinterpret_cast<uint4*>(tile + r * 128 + ((u ^ (r & 7)) << 4));
}

// A packed pair of element type E widened to fp32 (exact).
template <int E>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if (E == kElemBf16)
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    float lo, hi;
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(w));
    return make_float2(lo, hi);
}

// Packed fp32 pairs for the f32x2 instructions (two fp32 lanes per 64-bit
// register, the first value in the low half).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 f2_unpack(uint64_t r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}

// a * b + c, lane-wise
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Four floats -> four e4m3 codes (round to nearest even, finite values beyond
// 448 saturated), a in the lowest byte (cvt packs its first source operand into
// the upper byte of each pair).
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

// max(a, b, c) in one instruction (sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- epilogues

// NC fp32 columns of a TMEM accumulator row * mul, rounded to element type E, into
// row r of a 128-row staging tile of the output (128-byte swizzle, chunks of 64
// columns `chunk_bytes` apart); c0 is the output column of the first one.
template <int NC, int E>
__device__ __forceinline__ void stage_acc_row(uint32_t t_acc, float mul, uint8_t* stage,
                                              int chunk_bytes, int r, int c0) {
#pragma unroll
    for (int c = 0; c < NC / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(t_acc + c * 32, v);
        tmem_ld_wait();
        reg_fence(v);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int col = c0 + 32 * c + 8 * u;
            uint4 w;
            w.x = pack2<E>(__uint_as_float(v[8 * u]) * mul, __uint_as_float(v[8 * u + 1]) * mul);
            w.y = pack2<E>(__uint_as_float(v[8 * u + 2]) * mul, __uint_as_float(v[8 * u + 3]) * mul);
            w.z = pack2<E>(__uint_as_float(v[8 * u + 4]) * mul, __uint_as_float(v[8 * u + 5]) * mul);
            w.w = pack2<E>(__uint_as_float(v[8 * u + 6]) * mul, __uint_as_float(v[8 * u + 7]) * mul);
            *swizzled_unit(stage + (col / 64) * chunk_bytes, r, (col % 64) / 8) = w;
        }
    }
}

// ------------------------------------------------------------------ dropout
//
// Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3" (SC 2011): ten rounds of
// (c0, c1, c2, c3) -> (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))
// with the key bumped by the Weyl constants between rounds.
struct Philox4 {
    uint32_t x, y, z, w;
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
    constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
    constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += kW0;
            k1 += kW1;
        }
        // one 32 x 32 -> 64-bit product each (its high and low words)
        const uint64_t m0 = static_cast<uint64_t>(kM0) * c0, m1 = static_cast<uint64_t>(kM1) * c2;
        const uint32_t hi0 = static_cast<uint32_t>(m0 >> 32), lo0 = static_cast<uint32_t>(m0);
        const uint32_t hi1 = static_cast<uint32_t>(m1 >> 32), lo1 = static_cast<uint32_t>(m1);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return Philox4{c0, c1, c2, c3};
}

__device__ __forceinline__ uint32_t pick4(const Philox4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// The dropout draw of one 4 x 4 block of (query, key) pairs -- queries 4 I .. 4 I + 3,
// keys 4 J .. 4 J + 3 of one (sequence, query head) -- is one Philox call with
// counter (J, I, head_seq, offset) and key (seed low, seed high): output word w
// belongs to query 4 I + w, its byte k (bits 8k .. 8k + 7) to key 4 J + k.  A pair
// is kept iff its byte is >= the threshold.
//
// Four consecutive lanes 4m .. 4m + 3 of a warp form a group.  gather_rows: the
// lanes hold 4 consecutive query rows (lane 4m + a = query 4 I + a) and want the
// 4 keys of each block J in a list; gather_cols: the lanes hold 4 consecutive key
// rows (lane 4m + a = key 4 J + a) and want the 4 queries of each block I.  In
// round r lane 4m + a draws the block of index 4 r + a of the list and the group
// transposes the four draws, so every lane gets, for each of the 4 list entries
// of the round, one 32-bit word with the 4 bytes of its own row.
__device__ __forceinline__ void group_transpose4(const uint32_t (&mine)[4], uint32_t (&out)[4],
                                                 int lane) {
    // Two butterfly stages over the 4 x 4 block (lane a holds row a, wants column
    // a): first with lane a ^ 1 on the entries whose index differs from a in bit 0,
    // then with lane a ^ 2 on bit 1.  Constant register indices only, so nothing
    // goes to local memory.
    const bool b0 = lane & 1, b1 = lane & 2;
    uint32_t u[4];
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
        const uint32_t lo = mine[2 * pr], hi = mine[2 * pr + 1];
        const uint32_t got = __shfl_xor_sync(0xffffffffu, b0 ? lo : hi, 1);
        u[2 * pr] = b0 ? got : lo;
        u[2 * pr + 1] = b0 ? hi : got;
    }
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
        const uint32_t lo = u[pr], hi = u[pr + 2];
        const uint32_t got = __shfl_xor_sync(0xffffffffu, b1 ? lo : hi, 2);
        out[pr] = b1 ? got : lo;
        out[pr + 2] = b1 ? hi : got;
    }
}

// Rows are queries: word (query row) of the block's draw, per block J of the list
template <int NB>   // list length, a multiple of 4
__device__ __forceinline__ void dropout_words_rows(uint32_t (&words)[NB], int I, int J0, uint32_t hs,
                                                   uint32_t offset, uint32_t k0, uint32_t k1,
                                                   int lane) {
#pragma unroll
    for (int r = 0; r < NB / 4; ++r) {
        const Philox4 v = philox4x32_10(static_cast<uint32_t>(J0 + 4 * r + (lane & 3)),
                                        static_cast<uint32_t>(I), hs, offset, k0, k1);
        const uint32_t mine[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[4];
        group_transpose4(mine, out, lane);
#pragma unroll
        for (int u = 0; u < 4; ++u) words[4 * r + u] = out[u];
    }
}

// Rows are keys: per block I of the list, the 4 bytes of this key row (byte w =
// query 4 I + w), gathered from the four words of the draw.
template <int NB>
__device__ __forceinline__ void dropout_words_cols(uint32_t (&words)[NB], int I0, int J, uint32_t hs,
                                                   uint32_t offset, uint32_t k0, uint32_t k1,
                                                   int lane) {
#pragma unroll
    for (int r = 0; r < NB / 4; ++r) {
        const Philox4 v = philox4x32_10(static_cast<uint32_t>(J),
                                        static_cast<uint32_t>(I0 + 4 * r + (lane & 3)), hs, offset,
                                        k0, k1);
        // byte k of words 0..3 packed: the bytes key 4 J + k needs from this block
        // (byte permutes: bytes k of x and y, bytes k of z and w, then the two pairs)
        uint32_t mine[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t xy = __byte_perm(v.x, v.y, k | ((k + 4) << 4));
            const uint32_t zw = __byte_perm(v.z, v.w, k | ((k + 4) << 4));
            mine[k] = __byte_perm(xy, zw, 0x5410);
        }
        uint32_t out[4];
        group_transpose4(mine, out, lane);
#pragma unroll
        for (int u = 0; u < 4; ++u) words[4 * r + u] = out[u];
    }
}

// Dropout keep masks.  keep_masks turns a row's dropout words into byte masks once
// per step (byte k of a mask is 0xff iff byte k of the word, the random byte of the
// column, is >= the threshold); the element-wise passes then clear dropped values
// with a byte permute and an AND: a kept value passes unchanged, a dropped one
// becomes +0.
template <int N>
__device__ __forceinline__ void keep_masks(uint32_t (&w)[N], uint32_t thresh) {
    const uint32_t t4 = thresh * 0x01010101u;
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = __vcmpgeu4(w[i], t4);
}

// all 32 bits of column c's mask byte (the AND mask of an fp32 value)
__device__ __forceinline__ uint32_t keep_mask32(uint32_t m, int c) {
    return __byte_perm(m, 0u, static_cast<uint32_t>(c & 3) * 0x1111u);
}

// the AND mask of a 16-bit pair, columns c (low half) and c + 1 (high half), c even
__device__ __forceinline__ uint32_t keep_mask_pair(uint32_t m, int c) {
    const uint32_t a = c & 3, b = (c + 1) & 3;
    return __byte_perm(m, 0u, a | (a << 4) | (b << 8) | (b << 12));
}

}  // namespace fa
