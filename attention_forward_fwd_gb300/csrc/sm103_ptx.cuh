// sm103_ptx.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100a /
// sm_103a) data path used by the attention kernel: mbarriers, TMA tensor
// copies, tensor memory (TMEM) allocation / load / store, and tcgen05.mma with
// its shared-memory and instruction descriptors.  Everything here follows the
// PTX ISA; nothing is taken from a compiled library.
#pragma once

#include <cstdint>

namespace fa {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders generic-proxy shared-memory writes before later async-proxy reads
// (a TMA store that reads what the threads wrote).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One probe of the phase with the given parity; true once that phase completed.
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, P1;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier over `nthreads` threads that also returns the OR of `pred`
// over them.
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t nthreads, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred P1, P2;\n\tsetp.ne.u32 P1, %1, 0;\n\t"
        "bar.red.or.pred P2, %2, %3, P1;\n\tselp.u32 %0, 1, 0, P2;\n\t}"
        : "=r"(out)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return out != 0;
}

// Named barrier over `nthreads` threads that also returns the AND of `pred`
// over them.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t nthreads, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred P1, P2;\n\tsetp.ne.u32 P1, %1, 0;\n\t"
        "bar.red.and.pred P2, %2, %3, P1;\n\tselp.u32 %0, 1, 0, P2;\n\t}"
        : "=r"(out)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return out != 0;
}

// --------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_map(const void* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled load global -> shared; completion is counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* map, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// 4-D tiled store shared -> global (elements outside the tensor are dropped).
__device__ __forceinline__ void tma_store_4d(const void* map, uint32_t src, int c0, int c1, int c2,
                                             int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk group has finished reading its shared
// memory source (the writes to global memory may still be in flight).
__device__ __forceinline__ void bulk_wait_group_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_group_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------ tensor memory
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
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

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// 32 lanes x 32 columns of 32-bit words: thread t of the warp receives lane
// (warp's lane quarter + t), columns [col, col + 32) of `taddr`.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t* r) {
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

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Ties N registers to a point after tmem_ld_wait(): the empty volatile asm
// redefines them, so no use can be scheduled between the load and its wait.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t* r) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// ------------------------------------------------------------ tcgen05.mma
// Shared-memory matrix descriptor (tcgen05 format), 128-byte swizzle.
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride-dimension byte offset >> 4
//   bits 46-47 descriptor version (1 on sm_10x)
//   bits 49-51 base offset (0: every tile here starts 1024-byte aligned)
//   bits 61-63 swizzle mode (2 = 128-byte swizzle)
// K-major operand: rows of 128 bytes, 8-row groups SBO apart (LBO unused).
// MN-major operand: 64 contiguous MN elements per 128-byte row, one row per
// K index, 8-row groups SBO apart along K, 64-element MN chunks LBO apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor for tcgen05.mma.kind::f16 with fp32 accumulation.
//   bits  4-5  D format (1 = f32)
//   bits  7-9  A format (0 = f16, 1 = bf16); bits 10-12 B format (same)
//   bit  15    A major (0 = K-major); bit 16 B major (1 = MN-major)
//   bits 17-22 N >> 3; bits 24-28 M >> 4
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool bf16, bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one K=16 step.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred P1;\n\tsetp.ne.b32 P1, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, P1;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Issue forms for a whole converged warp: every lane runs the issuing code
// (so that descriptors and loop state are warp-uniform), one lane elected by
// elect.sync issues the instruction.  With all 32 lanes active the elected
// lane is the same every time, so its commits track the MMAs it issued.
// (Issuing from a loop that only lane 0 runs was measured to slow the tensor
// pipe to 88-123 cycles per M128 N128 K16 MMA when the SM sub-partition also
// runs busy warps, against 64 cycles from a converged warp.)
__device__ __forceinline__ void mma_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred E, P1;\n\telect.sync _|E, 0xffffffff;\n\t"
        "setp.ne.b32 P1, %4, 0;\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, P1;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same two issue forms with each shared-memory descriptor given as its low
// word (start address and leading byte offset, which vary per K step) and
// one high word shared by both operands (stride byte offset, version and
// swizzle, fixed for the kernel): 32-bit values keep the issuing warp's
// unrolled loops within a small register budget.
__host__ __device__ constexpr uint32_t sdesc_sw128_hi(uint32_t sbo_bytes) {
    return ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}
__device__ __forceinline__ uint32_t sdesc_sw128_lo(uint32_t saddr, uint32_t lbo_bytes) {
    return ((saddr >> 4) & 0x3FFFu) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
__device__ __forceinline__ void mma_ss_warp_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred E, P1;\n\t.reg .b64 DA, DB;\n\t"
        "mov.b64 DA, {%1, %3};\n\tmov.b64 DB, {%2, %3};\n\t"
        "elect.sync _|E, 0xffffffff;\n\tsetp.ne.b32 P1, %5, 0;\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %4, P1;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts_warp_lo(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred E, P1;\n\t.reg .b64 DB;\n\t"
        "mov.b64 DB, {%2, %3};\n\t"
        "elect.sync _|E, 0xffffffff;\n\tsetp.ne.b32 P1, %5, 0;\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], DB, %4, P1;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Four K=16 steps issued under one elect.sync (the per-instruction election
// and predicate set-up are paid once).  SS form: both descriptors (low words
// over the shared high word) advance by `step` 16-byte units per K step, the
// first step accumulates iff `acc_first`, the others always.
__device__ __forceinline__ void mma_ss_x4_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                             uint32_t step, uint32_t idesc, uint32_t acc_first) {
    asm volatile(
        "{\n\t.reg .pred E, P1, T;\n\t.reg .b64 DA, DB;\n\t.reg .b32 A1, B1;\n\t"
        "setp.ne.b32 P1, %6, 0;\n\tsetp.eq.b32 T, %6, %6;\n\t"
        "elect.sync _|E, 0xffffffff;\n\t"
        "mov.b64 DA, {%1, %3};\n\tmov.b64 DB, {%2, %3};\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %4, P1;\n\t"
        "add.u32 A1, %1, %5;\n\tadd.u32 B1, %2, %5;\n\t"
        "mov.b64 DA, {A1, %3};\n\tmov.b64 DB, {B1, %3};\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %4, T;\n\t"
        "add.u32 A1, A1, %5;\n\tadd.u32 B1, B1, %5;\n\t"
        "mov.b64 DA, {A1, %3};\n\tmov.b64 DB, {B1, %3};\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %4, T;\n\t"
        "add.u32 A1, A1, %5;\n\tadd.u32 B1, B1, %5;\n\t"
        "mov.b64 DA, {A1, %3};\n\tmov.b64 DB, {B1, %3};\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], DA, DB, %4, T;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(step), "r"(acc_first)
        : "memory");
}

// TS form of the same: A from tensor memory advancing by `a_step` columns,
// B's descriptor low word by `b_step` 16-byte units per K step.
__device__ __forceinline__ void mma_ts_x4_lo(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi,
                                             uint32_t a_step, uint32_t b_step, uint32_t idesc,
                                             uint32_t acc_first) {
    asm volatile(
        "{\n\t.reg .pred E, P1, T;\n\t.reg .b64 DB;\n\t.reg .b32 A1, B1;\n\t"
        "setp.ne.b32 P1, %7, 0;\n\tsetp.eq.b32 T, %7, %7;\n\t"
        "elect.sync _|E, 0xffffffff;\n\t"
        "mov.b64 DB, {%2, %3};\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], DB, %4, P1;\n\t"
        "add.u32 A1, %1, %5;\n\tadd.u32 B1, %2, %6;\n\tmov.b64 DB, {B1, %3};\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], [A1], DB, %4, T;\n\t"
        "add.u32 A1, A1, %5;\n\tadd.u32 B1, B1, %6;\n\tmov.b64 DB, {B1, %3};\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], [A1], DB, %4, T;\n\t"
        "add.u32 A1, A1, %5;\n\tadd.u32 B1, B1, %6;\n\tmov.b64 DB, {B1, %3};\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], [A1], DB, %4, T;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(a_step), "r"(b_step), "r"(acc_first)
        : "memory");
}

__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred E, P1;\n\telect.sync _|E, 0xffffffff;\n\t"
        "setp.ne.b32 P1, %4, 0;\n\t"
        "@E tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, P1;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit_warp(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred E;\n\telect.sync _|E, 0xffffffff;\n\t"
        "@E tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred E;\n\telect.sync _|E, 0xffffffff;\n\t"
        "@E mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], one K=16 step (A read from tensor memory).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred P1;\n\tsetp.ne.b32 P1, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, P1;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// --------------------------------------------- programmatic dependent launch
// Lets a dependent grid launched with programmatic stream serialisation be
// scheduled once every CTA of this grid has issued this (or exited).
__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Waits until the grids this one depends on have completed and their memory
// operations are visible (a no-op without such a dependency).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------ register budget
// Move this warpgroup's per-thread register budget up / down (all four warps
// of the warpgroup execute it; the CTA's total stays what it launched with).
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// The value of x, hidden from the optimiser (it cannot reuse a computation
// made from x before this point).
__device__ __forceinline__ int opaque(int x) {
    asm volatile("" : "+r"(x));
    return x;
}

// ----------------------------------------------------------------- math
// max of three floats (one instruction on sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace ptx
}  // namespace fa
