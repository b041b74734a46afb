// Shared device helpers of libidx: status bits, the order-preserving fp32 key,
// bounded mbarrier waits, TMA and tcgen05 (5th-generation tensor core) PTX.
// Everything here targets sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/idx.h"

#define IDX_DEVI __device__ __forceinline__

namespace idx {

// ---------------------------------------------------------------- status

// OR a bit into the caller's optional device status word.
IDX_DEVI void raise_status(int* d_status, int bit) {
    if (d_status) atomicOr(d_status, bit);
}

// ------------------------------------------------------ order-preserving key

// Maps an fp32 value to a uint32 whose unsigned order is the float order.
// -0.0 is first folded onto +0.0 so that the two compare equal (an exact tie).
IDX_DEVI uint32_t fkey(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The float whose order key is L: for every non-NaN f, f >= it exactly when
// fkey(f) >= L (fkey is monotone and folds -0 onto +0).  Keys below the one of
// -inf admit every non-NaN value.
IDX_DEVI float key_floor_float(uint32_t L) {
    if (L <= 0x007fffffu) return -INFINITY;
    return __uint_as_float((L & 0x80000000u) ? (L & 0x7fffffffu) : ~L);
}

// --------------------------------------------------------------- smem/ptx

IDX_DEVI uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous global -> shared copy (L2 only), and the wait for
// every copy this thread issued.
IDX_DEVI void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
                 : "memory");
}
IDX_DEVI void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

IDX_DEVI void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Programmatic dependent launch.  A kernel launched with the attribute (see
// launch_k) is launched as the kernel before it on the stream finishes, its
// CTAs taking SMs as that kernel's CTAs leave them: pdl_wait blocks until that
// kernel has completed and its memory is visible (at once for a launch without
// the attribute).  (No kernel here signals its dependents early: measured on
// GB300, letting the next grid launch from the start of this one slowed the
// long scoring passes it overlapped.)
IDX_DEVI void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

IDX_DEVI void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

IDX_DEVI void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

IDX_DEVI void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One test of the phase (the thread may be suspended in hardware for a
// system-dependent time while the phase is incomplete).
IDX_DEVI bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most ~`limit`
// SM clock cycles.  Returns false when the wait gave up.  `abort` (shared) is
// polled so that one timed-out role releases every other role of the CTA.
IDX_DEVI bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                        long long limit = (1ll << 32)) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort && *abort) return false;
        if (clock64() - t0 > limit) return false;
    }
}

// ------------------------------------------------------------------- TMA

IDX_DEVI void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

IDX_DEVI void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar, int c0, int c1,
                          int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from global to shared memory, both
// 16-byte aligned, completing on `bar` (transaction bytes).
IDX_DEVI void bulk_g2s(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
        "r"(smem_u32(bar))
        : "memory");
}

IDX_DEVI void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// --------------------------------------------------------------- tcgen05

IDX_DEVI void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(smem_slot)),
                 "r"(ncols)
                 : "memory");
}

IDX_DEVI void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

IDX_DEVI void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

IDX_DEVI void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
IDX_DEVI void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one CTA, bf16 inputs, fp32 accumulator.
IDX_DEVI void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same with e4m3 inputs (kind::f8f6f4).
IDX_DEVI void mma_fp8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
IDX_DEVI void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 16x256b shape, R repetitions along the columns (R in {1, 2, 4, 8}): thread t
// gets, for repetition j, lanes t/4 and t/4 + 8 (relative to taddr's lane) at
// columns 8j + 2(t%4) and 8j + 2(t%4) + 1, in the order (lane t/4, col even),
// (t/4, odd), (t/4 + 8, even), (t/4 + 8, odd).
template <int R>
IDX_DEVI void tmem_ld16x256b(uint32_t taddr, float* v) {
    uint32_t r[4 * R];
    if constexpr (R == 1) {
        asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr));
    } else if constexpr (R == 2) {
        asm volatile(
            "tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7])
            : "r"(taddr));
    } else if constexpr (R == 8) {
        asm volatile(
            "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
            "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, "
            "%26, %27, %28, %29, %30, %31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
              "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
              "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
              "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
              "=r"(r[31])
            : "r"(taddr));
    } else {
        static_assert(R == 4, "1, 2, 4 or 8 repetitions");
        asm volatile(
            "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
            "%10, %11, %12, %13, %14, %15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
              "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
    }
#pragma unroll
    for (int i = 0; i < 4 * R; ++i) v[i] = __uint_as_float(r[i]);
}

// 32x32b shape, N repetitions along the columns (N in {8, 16, 32}): thread t
// gets lane t (relative to taddr's lane) at columns 0 .. N-1.
template <int N>
IDX_DEVI void tmem_ld32x32b(uint32_t taddr, float* v) {
    uint32_t r[N];
    if constexpr (N == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                       "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr));
    } else if constexpr (N == 16) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
            "%10, %11, %12, %13, %14, %15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
              "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
    } else {
        static_assert(N == 32, "8, 16 or 32 repetitions");
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
            "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, "
            "%26, %27, %28, %29, %30, %31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
              "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
              "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
              "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
              "=r"(r[31])
            : "r"(taddr));
    }
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

IDX_DEVI void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

IDX_DEVI void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------- descriptors

// Shared-memory matrix descriptor of a K-major operand tile whose rows are
// `row_bytes` (64 or 128) long and swizzled at that width by TMA; groups of 8
// rows are `8 * row_bytes` apart.  Field layout per the PTX ISA tcgen05
// "shared memory descriptor": start address >> 4 in bits 0-13, leading byte
// offset >> 4 in 16-29 (unused for swizzled K-major), stride byte offset >> 4
// in 32-45, the fixed version value 1 in 46-47, base offset 0 (1024-byte
// aligned tiles) in 49-51, swizzle mode in 61-63 (2 = 128 B, 4 = 64 B).
IDX_DEVI uint64_t smem_desc(uint32_t saddr, uint32_t row_bytes) {
    const uint64_t sbo = 8ull * row_bytes;
    const uint64_t swz = row_bytes == 128 ? 2ull : 4ull;
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
           ((sbo >> 4) & 0x3FFFull) << 32 | (1ull << 46) | (swz << 61);
}

// Instruction descriptor for a dense M x N MMA with fp32 accumulation, both
// operands K-major.  a/b format: kind::f16 1 = bf16; kind::f8f6f4 0 = e4m3.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t ab_format, uint32_t M, uint32_t N) {
    return (1u << 4)                 // D format f32
           | (ab_format << 7)        // A format
           | (ab_format << 10)       // B format
           | ((N >> 3) << 17)        // N / 8
           | ((M >> 4) << 24);       // M / 16
}


// Launch `kern` on stream s; with pdl the launch may overlap the tail of the
// kernel before it (the kernel must begin with pdl_wait before it touches that
// kernel's results).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace idx
