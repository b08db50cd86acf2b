// Inline-PTX wrappers for sm_103a: mbarrier, TMA tensor loads, tcgen05
// (tensor memory allocation, MMA, loads/stores, commits and fences).
//
// Everything here is a thin, literal wrapper around one PTX instruction (or a
// bounded wait loop around one); the attention logic lives in the kernel.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace attn {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------- dependent grid launch

// Wait until the grids this one depends on have completed and their memory
// operations are visible (a no-op when launched without a dependency).
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the grids that depend on this one to be scheduled.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------ register reallocation

// Warpgroup-collective: raise (inc) or lower (dec) this warpgroup's per-thread
// register count to N.  The registers come from the pool the block was
// launched with (threads x registers per thread at launch); an increase waits
// until other warpgroups have released enough.
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Warp-collective issue: the wrappers marked "(warp)" are called by all 32
// lanes of a converged warp and one lane, chosen by elect.sync, issues the
// instruction.  Keeping the issuing warp converged lets the compiler hold
// loop state, descriptors and addresses in uniform registers.

// (warp) arrive on `bar` and add `bytes` to its expected transaction count.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
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

// Non-blocking probe of the same phase condition as mbar_try_wait.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// (warp) 3-D tiled load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *m, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// (warp) the same load with an L2 "evict last" cache policy (kept in L2 in
// preference to other lines).
__device__ __forceinline__ void tma_load_3d_keep(uint32_t dst, const CUtensorMap *m, int c0, int c1,
                                                 int c2, uint32_t bar) {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(pol)
        : "memory");
}

// (one thread) 3-D tiled store of one box from shared memory into the tensor,
// in the thread's bulk async-group; the part of the box outside the tensor is
// not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *m, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// The thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// The thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's earlier generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// ------------------------------------------------------------------ tcgen05

// (warp) 1-D bulk copy global -> shared of `bytes` (a multiple of 16; both
// addresses 16-byte aligned), counted on the mbarrier's transaction bytes.
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

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

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// The MMA and commit wrappers touch no memory the compiler tracks (operands
// are named by descriptors and TMEM addresses); being volatile they keep their
// order relative to every other volatile asm, including the mbarrier waits
// that carry the memory ordering.

// (warp) D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16, one CTA.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// (warp) D[tmem] (+)= A[tmem] * B[smem desc], kind::f16, one CTA.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// (warp) D[tmem] (+)= A[tmem] * B[smem desc], kind::f8f6f4 (8-bit operands,
// K = 32 per instruction), one CTA.
__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Batches of four MMAs issued by one elected lane.  The issuing warp shares its
// SM sub-partition with compute warps, so the instructions it spends per MMA
// bound the MMA rate; one elect and the descriptor steps inside one block keep
// them few.  A descriptor's start address is its low 14 bits (16-byte units),
// so a step within one operand buffer is a 32-bit add to the low word.  The
// first MMA of a batch accumulates if `accumulate` != 0, the others always do.

// (warp) four SS MMAs: A_k, B_k = a_desc, b_desc advanced by k * a_step, k * b_step.
__device__ __forceinline__ void mma_ss_x4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t a_step,
                                          uint32_t b_step, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t.reg .b32 al, ah, bl, bh;\n\t.reg .b64 a1, b1, a2, b2, a3, b3;\n\t"
        "setp.ne.b32 p, %6, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"
        "mov.b64 {al, ah}, %1;\n\tmov.b64 {bl, bh}, %2;\n\t"
        "add.u32 al, al, %3;\n\tadd.u32 bl, bl, %4;\n\tmov.b64 a1, {al, ah};\n\tmov.b64 b1, {bl, bh};\n\t"
        "add.u32 al, al, %3;\n\tadd.u32 bl, bl, %4;\n\tmov.b64 a2, {al, ah};\n\tmov.b64 b2, {bl, bh};\n\t"
        "add.u32 al, al, %3;\n\tadd.u32 bl, bl, %4;\n\tmov.b64 a3, {al, ah};\n\tmov.b64 b3, {bl, bh};\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %5, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %5, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %5, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %5, q;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(a_step), "r"(b_step), "r"(idesc), "r"(accumulate));
}

// (warp) four TS MMAs: A from TMEM at a0..a3, B_k = b_desc advanced by k * b_step.
__device__ __forceinline__ void mma_ts_x4(uint32_t d_tmem, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint64_t b_desc, uint32_t b_step, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t.reg .b32 bl, bh;\n\t.reg .b64 b1, b2, b3;\n\t"
        "setp.ne.b32 p, %8, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"
        "mov.b64 {bl, bh}, %5;\n\t"
        "add.u32 bl, bl, %6;\n\tmov.b64 b1, {bl, bh};\n\t"
        "add.u32 bl, bl, %6;\n\tmov.b64 b2, {bl, bh};\n\t"
        "add.u32 bl, bl, %6;\n\tmov.b64 b3, {bl, bh};\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %7, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], b1, %7, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], b2, %7, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], b3, %7, q;\n\t}" ::"r"(d_tmem),
        "r"(a0), "r"(a1), "r"(a2), "r"(a3), "l"(b_desc), "r"(b_step), "r"(idesc), "r"(accumulate));
}

// (warp) eight TS MMAs with A from consecutive 8-column steps of TMEM (a_tmem +
// 8k) and B_k = b_desc advanced by k * b_step, then a commit of the issuing
// lane's MMAs to `bar`, all from one elected lane.
__device__ __forceinline__ void mma_ts_x8_commit(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t b_step,
                                                 uint32_t idesc, uint32_t accumulate, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t.reg .b32 bl, bh, a;\n\t.reg .b64 b;\n\t"
        "setp.ne.b32 p, %5, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"
        "mov.b64 {bl, bh}, %2;\n\tmov.b32 a, %1;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], %2, %4, p;\n\t"
        "add.u32 a, a, 8;\n\tadd.u32 bl, bl, %3;\n\tmov.b64 b, {bl, bh};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.u32 bl, bl, %3;\n\tmov.b64 b, {bl, bh};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.u32 bl, bl, %3;\n\tmov.b64 b, {bl, bh};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.u32 bl, bl, %3;\n\tmov.b64 b, {bl, bh};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.u32 bl, bl, %3;\n\tmov.b64 b, {bl, bh};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.u32 bl, bl, %3;\n\tmov.b64 b, {bl, bh};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.u32 bl, bl, %3;\n\tmov.b64 b, {bl, bh};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(b_step), "r"(idesc), "r"(accumulate), "r"(bar));
}

// (warp) the same with 8-bit operands (kind::f8f6f4, K = 32 per MMA).
__device__ __forceinline__ void mma_ts_f8_x4(uint32_t d_tmem, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint64_t b_desc, uint32_t b_step, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t.reg .b32 bl, bh;\n\t.reg .b64 b1, b2, b3;\n\t"
        "setp.ne.b32 p, %8, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"
        "mov.b64 {bl, bh}, %5;\n\t"
        "add.u32 bl, bl, %6;\n\tmov.b64 b1, {bl, bh};\n\t"
        "add.u32 bl, bl, %6;\n\tmov.b64 b2, {bl, bh};\n\t"
        "add.u32 bl, bl, %6;\n\tmov.b64 b3, {bl, bh};\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %5, %7, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%2], b1, %7, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%3], b2, %7, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%4], b3, %7, q;\n\t}" ::"r"(d_tmem),
        "r"(a0), "r"(a1), "r"(a2), "r"(a3), "l"(b_desc), "r"(b_step), "r"(idesc), "r"(accumulate));
}

// (warp) arrive once on `bar` when every tcgen05 operation the issuing lane
// issued before has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            bar));
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bits, 32 consecutive columns: thread t of the warp gets
// columns [col, col+32) of TMEM lane (lane_base + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
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

// 32 lanes x 32 bits, 8 consecutive columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
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

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// 16 columns of zeros (one zero register for every operand of the store).
__device__ __forceinline__ void tmem_st16_zero(uint32_t taddr) {
    asm volatile(
        "{\n\t.reg .b32 z;\n\tmov.b32 z, 0;\n\t"
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {z, z, z, z, z, z, z, z, z, z, z, z, z, z, z, z};\n\t}"
        ::"r"(taddr)
        : "memory");
}

// ------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor of a tcgen05 operand stored with the
// 128-byte swizzle: start address, leading/stride byte offsets (16-byte
// units), descriptor version 1 (bit 46), swizzle mode 2 = 128B (bits 61-63).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with an fp32 accumulator:
// A and B both fp16 (0) or both bf16 (1); A K-major; B K-major or MN-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32acc(bool bf16, int M, int N, bool b_mn_major) {
    return (1u << 4)                                   // D format: f32
           | ((bf16 ? 1u : 0u) << 7)                    // A format
           | ((bf16 ? 1u : 0u) << 10)                   // B format
           | ((b_mn_major ? 1u : 0u) << 16)             // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)      // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);     // M / 16
}

// Instruction descriptor of a kind::f8f6f4 MMA with both operands float8 e5m2
// (format code 1), both K-major, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_e5m2_f32acc(int M, int N) {
    return (1u << 4)                                   // D format: f32
           | (1u << 7)                                  // A format: e5m2
           | (1u << 10)                                 // B format: e5m2
           | (static_cast<uint32_t>(N >> 3) << 17)      // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);     // M / 16
}

// ----------------------------------------------------------------- numerics

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two fp32 values rounded to nearest-even into one packed pair; `lo` lands
// in bits 0-15 (the lower-indexed element).
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (BF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four fp32 values rounded to float8 e5m2 (nearest, saturating to the largest
// finite value) in one word, a in the lowest byte.
// Two 16-bit values of a 32-bit word (lower half first) widened to fp32.
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if constexpr (BF16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        float lo, hi;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
            : "=f"(lo), "=f"(hi)
            : "r"(w));
        return make_float2(lo, hi);
    }
}

__device__ __forceinline__ uint32_t pack4_e5m2(float a, float b, float c, float d) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

}  // namespace attn
