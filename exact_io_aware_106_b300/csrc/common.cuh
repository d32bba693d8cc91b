// common.cuh -- inline-PTX building blocks for the sm_103a kernels:
// mbarriers with bounded waits, bulk / tensor (TMA) copies, tcgen05 tensor
// memory, MMA issue and shared-memory matrix descriptors, numeric packing.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// Bits of the per-device error word.
enum : unsigned { DERR_TIMEOUT = 1u, DERR_INDEX = 2u };

// The error word is the first of CTL_WORDS per-device control words that
// every kernel receives as `err`:
//   [CTL_ERR]     error bits, set by kernels, read and cleared by the host;
//   [CTL_WAIT_US] limit of the bounded waits in microseconds (0: the default
//                 kWaitTimeoutNs); set only by the test entry point;
//   [CTL_HOOKS]   test hooks (HOOK_WITHHOLD_Q: the dense prefill's producer
//                 does not issue the Q copy, so the first wait on it expires;
//                 HOOK_WITHHOLD_KV: the decode split kernel's producer issues
//                 no K/V copy, so its consumers' first wait expires).
enum : int { CTL_ERR = 0, CTL_WAIT_US = 1, CTL_HOOKS = 2, CTL_WORDS = 4 };
enum : unsigned { HOOK_WITHHOLD_Q = 1u, HOOK_WITHHOLD_KV = 2u, HOOK_ALL = 3u };

// A bounded wait gives up after this long (a healthy wait in these kernels
// lasts microseconds).  On expiry the waiter sets DERR_TIMEOUT and the CTA's
// abort flag, and every role unwinds to the common exit.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

__device__ __forceinline__ unsigned long long wait_limit_ns(const unsigned *ctl) {
    const unsigned us = *reinterpret_cast<const volatile unsigned *>(ctl + CTL_WAIT_US);
    return us != 0u ? 1000ull * us : kWaitTimeoutNs;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------- mbarriers

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            bar),
        "r"(bytes)
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false if
// the CTA is aborting (another role gave up) or this wait expired.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned *err) {
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = globaltimer();
    unsigned long long limit = 0; // read once the wait has spun a while
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((n & 31u) == 0) {
            if (*abort_flag)
                return false;
            if (limit == 0)
                limit = wait_limit_ns(err);
            if (globaltimer() - t0 > limit) {
                atomicOr(err, DERR_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Three waits at once: the three try_waits are issued back to back, so that
// when all phases have already completed (the common case in a pipeline
// whose producers run ahead) their latencies overlap instead of adding up;
// otherwise each one not yet seen complete is waited for (bounded) in turn.
// A barrier with `need` false is not tested.
__device__ __forceinline__ bool mbar_wait3(uint32_t b0, uint32_t p0, bool need0, uint32_t b1,
                                           uint32_t p1, bool need1, uint32_t b2, uint32_t p2,
                                           bool need2, volatile int *abort_flag,
                                           unsigned *err) {
    const bool d0 = !need0 || mbar_try_wait(b0, p0);
    const bool d1 = !need1 || mbar_try_wait(b1, p1);
    const bool d2 = !need2 || mbar_try_wait(b2, p2);
    if (d0 && d1 && d2)
        return true;
    return (d0 || mbar_wait(b0, p0, abort_flag, err)) && (d1 || mbar_wait(b1, p1, abort_flag, err)) &&
           (d2 || mbar_wait(b2, p2, abort_flag, err));
}

// mbar_wait by a whole warp whose next instructions are warp-wide
// (.sync.aligned tensor-memory loads, ldmatrix, mma.sync): the result is the
// same in every lane, so a wait that gives up in one lane never leaves the
// others to enter a warp-wide instruction alone.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               volatile int *abort_flag, unsigned *err) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, err));
}

// Wait used only while unwinding after an abort: ignores the abort flag so
// that copies already in flight land before the CTA exits; bounded by the
// default limit (never the test's shorter one, so that copies in flight
// always land).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kWaitTimeoutNs)
            return;
}

// ------------------------------------------------------- bulk / TMA copies

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// src, dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 3-D tiled tensor copy global -> shared (box and swizzle from the map).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y, int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}

// 3-D tiled tensor copy shared -> global (box and swizzle from the map);
// rows past the tensor's extent are not written.  Completion is tracked by
// the bulk async-group of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int x, int y,
                                             int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::
                     "l"(map),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk store of this thread has finished reading
// its shared-memory source.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
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
// Arrive once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], 8-bit operands (kind::f8f6f4;
// the instruction descriptor's A/B format fields are 0 for E4M3).
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor, kind::f16 with fp32 accumulation.
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format (0 f16,
//   1 bf16), 15/16 A/B major (0 = K-major, 1 = MN-major), 17-22 N>>3,
//   24-28 M>>4.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool a_mn_major,
                                                 bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
//   bits 0-13 start address >> 4, 16-29 leading byte offset >> 4,
//   32-45 stride byte offset >> 4, 46-47 descriptor version (1),
//   61-63 layout (2 = 128-byte swizzle).
// K-major: rows of 128 bytes, 8-row atoms SBO apart (LBO unused).
// MN-major: 64-element (128-byte) MN chunks LBO apart, 8-row K groups SBO
// apart.  Tiles start on 1024-byte boundaries.
// The descriptor splits into a low word that depends on the address
// (start address, leading byte offset) and a high word fixed by the layout
// (stride byte offset, version, swizzle): kernels that step through an
// operand keep the low word (32 bits) and attach the constant high word per
// MMA.
__host__ __device__ constexpr uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo) {
    return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t sdesc_hi(uint32_t sbo, uint32_t layout) {
    return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (layout << 29);
}
__device__ __forceinline__ uint64_t sdesc(uint32_t lo, uint32_t hi) {
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
// high words of the two layouts below
__host__ __device__ constexpr uint32_t sdesc_sw128_hi(uint32_t sbo) { return sdesc_hi(sbo, 2u); }
__host__ __device__ constexpr uint32_t sdesc_kmajor_hi(int row_bytes) {
    return sdesc_hi(8u * row_bytes, row_bytes == 128 ? 2u : 4u);
}

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return sdesc(sdesc_lo(saddr, lbo), sdesc_sw128_hi(sbo));
}

// Shared-memory matrix descriptor for a K-major operand whose rows are
// `row_bytes` (128 or 64) long and swizzled over that span by TMA: 8-row
// atoms SBO = 8 * row_bytes apart; layout 2 = 128-byte, 4 = 64-byte swizzle;
// the leading byte offset (unused when swizzled) is 16.
__device__ __forceinline__ uint64_t sdesc_kmajor(uint32_t saddr, int row_bytes) {
    return sdesc(sdesc_lo(saddr, 16u), sdesc_kmajor_hi(row_bytes));
}

#define ATTN_R32_OUT(r)                                                                          \
    "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),          \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),  \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),            \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),            \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define ATTN_R32_IN(r)                                                                           \
    "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),      \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),        \
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),      \
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),      \
        "r"(r[29]), "r"(r[30]), "r"(r[31])
#define ATTN_REGS32_0                                                                            \
    "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, " \
    "%20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}"
#define ATTN_REGS32_1                                                                            \
    "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, "    \
    "%20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32}"

// Thread i of the warp reads 32 consecutive 32-bit columns of TMEM lane
// (lane base + i).  The load and its completion wait are one asm statement
// so no use of the registers can be scheduled before the data arrives.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " ATTN_REGS32_0
                 ", [%32];\n\ttcgen05.wait::ld.sync.aligned;"
                 : ATTN_R32_OUT(r)
                 : "r"(taddr)
                 : "memory");
}
// Thread i reads 64 consecutive 32-bit columns of TMEM lane (lane base + i)
// with one load and one completion wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
                 "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
                 "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
                 "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63"
                 "}, [%64];\n\ttcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                 "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                 "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                 "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                 "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
                 "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
                 "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
                 "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]),
                 "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]),
                 "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr)
                 : "memory");
}
// Thread i reads 128 consecutive 32-bit columns of TMEM lane (lane base +
// i) with one load and one completion wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
                 "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
                 "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
                 "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, "
                 "%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
                 "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, "
                 "%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, "
                 "%112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}"
                 ", [%128];\n\ttcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                 "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
                 "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
                 "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]),
                 "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
                 "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
                 "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
                 "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]),
                 "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]),
                 "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]),
                 "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]),
                 "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]),
                 "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]),
                 "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
                 "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]),
                 "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]),
                 "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]),
                 "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
                 : "r"(taddr)
                 : "memory");
}
// Two loads of 32 consecutive 32-bit columns each (thread i reads TMEM lane
// base + i) under one completion wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t a0, uint32_t (&r0)[32], uint32_t a1,
                                            uint32_t (&r1)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : ATTN_R32_OUT(r0), ATTN_R32_OUT(r1)
                 : "r"(a0), "r"(a1)
                 : "memory");
}
// Two loads of 64 consecutive 32-bit columns each (thread i reads TMEM lane
// base + i) under one completion wait.
__device__ __forceinline__ void tmem_ld64x2(uint32_t a0, uint32_t (&r0)[64], uint32_t a1,
                                            uint32_t (&r1)[64]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%128];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%129];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r0[0]), "=r"(r0[1]), "=r"(r0[2]), "=r"(r0[3]), "=r"(r0[4]), "=r"(r0[5]), "=r"(r0[6]), "=r"(r0[7]), "=r"(r0[8]), "=r"(r0[9]), "=r"(r0[10]), "=r"(r0[11]), "=r"(r0[12]), "=r"(r0[13]), "=r"(r0[14]), "=r"(r0[15]), "=r"(r0[16]), "=r"(r0[17]), "=r"(r0[18]), "=r"(r0[19]), "=r"(r0[20]), "=r"(r0[21]), "=r"(r0[22]), "=r"(r0[23]), "=r"(r0[24]), "=r"(r0[25]), "=r"(r0[26]), "=r"(r0[27]), "=r"(r0[28]), "=r"(r0[29]), "=r"(r0[30]), "=r"(r0[31]), "=r"(r0[32]), "=r"(r0[33]), "=r"(r0[34]), "=r"(r0[35]), "=r"(r0[36]), "=r"(r0[37]), "=r"(r0[38]), "=r"(r0[39]), "=r"(r0[40]), "=r"(r0[41]), "=r"(r0[42]), "=r"(r0[43]), "=r"(r0[44]), "=r"(r0[45]), "=r"(r0[46]), "=r"(r0[47]), "=r"(r0[48]), "=r"(r0[49]), "=r"(r0[50]), "=r"(r0[51]), "=r"(r0[52]), "=r"(r0[53]), "=r"(r0[54]), "=r"(r0[55]), "=r"(r0[56]), "=r"(r0[57]), "=r"(r0[58]), "=r"(r0[59]), "=r"(r0[60]), "=r"(r0[61]), "=r"(r0[62]), "=r"(r0[63]),
                   "=r"(r1[0]), "=r"(r1[1]), "=r"(r1[2]), "=r"(r1[3]), "=r"(r1[4]), "=r"(r1[5]), "=r"(r1[6]), "=r"(r1[7]), "=r"(r1[8]), "=r"(r1[9]), "=r"(r1[10]), "=r"(r1[11]), "=r"(r1[12]), "=r"(r1[13]), "=r"(r1[14]), "=r"(r1[15]), "=r"(r1[16]), "=r"(r1[17]), "=r"(r1[18]), "=r"(r1[19]), "=r"(r1[20]), "=r"(r1[21]), "=r"(r1[22]), "=r"(r1[23]), "=r"(r1[24]), "=r"(r1[25]), "=r"(r1[26]), "=r"(r1[27]), "=r"(r1[28]), "=r"(r1[29]), "=r"(r1[30]), "=r"(r1[31]), "=r"(r1[32]), "=r"(r1[33]), "=r"(r1[34]), "=r"(r1[35]), "=r"(r1[36]), "=r"(r1[37]), "=r"(r1[38]), "=r"(r1[39]), "=r"(r1[40]), "=r"(r1[41]), "=r"(r1[42]), "=r"(r1[43]), "=r"(r1[44]), "=r"(r1[45]), "=r"(r1[46]), "=r"(r1[47]), "=r"(r1[48]), "=r"(r1[49]), "=r"(r1[50]), "=r"(r1[51]), "=r"(r1[52]), "=r"(r1[53]), "=r"(r1[54]), "=r"(r1[55]), "=r"(r1[56]), "=r"(r1[57]), "=r"(r1[58]), "=r"(r1[59]), "=r"(r1[60]), "=r"(r1[61]), "=r"(r1[62]), "=r"(r1[63])
                 : "r"(a0), "r"(a1)
                 : "memory");
}
// Thread i writes 32 consecutive columns of TMEM lane (lane base + i).
// Completion is awaited separately with tmem_st_wait().
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], " ATTN_REGS32_1 ";" ::"r"(taddr),
                 ATTN_R32_IN(r)
                 : "memory");
}
// Thread i writes 16 consecutive columns of TMEM lane (lane base + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(
                     taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
                 "r"(r[14]), "r"(r[15])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------- warp-level MMA (mma.sync)

// Four 8x8 16-bit matrices from shared memory; lanes 8j..8j+7 give the row
// addresses of matrix j, register j receives matrix j (lane i: row i/4,
// elements 2(i%4), 2(i%4)+1).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
// Same, transposed: lane i receives elements (2(i%4), i/4) and (2(i%4)+1, i/4).
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// D (16x8 fp32) += A (16x16, row) * B (16x8, col), 16-bit inputs.
//   A regs: {(g, 2t..2t+1), (g+8, 2t..), (g, 2t+8..), (g+8, 2t+8..)}
//   B regs: {(k 2t..2t+1, n g), (k 2t+8..2t+9, n g)}
//   D regs: {(g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)}
// with g = lane / 4, t = lane % 4.
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    if constexpr (BF16)
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                     "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
                     "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `ch` of row `row` in a TMA-swizzled panel
// whose rows are PW bytes (128: chunk ^= row mod 8; 64: chunk ^= row/2 mod 4).
template <int PW>
__device__ __forceinline__ uint32_t swz_offset(int row, int ch) {
    if constexpr (PW == 128)
        return static_cast<uint32_t>(row * 128 + ((ch ^ (row & 7)) << 4));
    else
        return static_cast<uint32_t>(row * 64 + ((ch ^ ((row >> 1) & 3)) << 4));
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Two E4M3 codes (low byte first) widened exactly to f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<unsigned short>(v & 0xFFFFu)));
    return r;
}

// Per-warpgroup register budget (all four warps of the warpgroup execute
// it): dec gives registers back to the CTA's pool, inc waits until the pool
// can grant the new count.  The counts must add up to the launch's
// allocation or inc never returns.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------- numerics

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (three-input max, sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

// Pack two floats as 16-bit values, `lo` in the low half.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (BF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <bool BF16>
__device__ __forceinline__ float lo16(uint32_t v) {
    if constexpr (BF16)
        return __uint_as_float(v << 16);
    else
        return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}
template <bool BF16>
__device__ __forceinline__ float hi16(uint32_t v) {
    if constexpr (BF16)
        return __uint_as_float(v & 0xFFFF0000u);
    else
        return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
}

} // namespace attn
