// tcgen05 (5th-generation tensor core) helpers in inline PTX, shared by the
// tensor-core kernels: shared-memory operand descriptors, the kind::tf32
// MMA, commits, TMEM loads, the split of an fp32 value into its tf32 part
// and remainder, and a bounded mbarrier wait with a CTA-local abort.
#pragma once
#include "cn_common.cuh"
#include "cn_internal.h"

namespace cn {

// ---- tcgen05 / UMMA helpers (inline PTX) --------------------------------------

// Shared-memory matrix descriptor: start address, leading-dimension byte
// offset (between the two K core matrices), stride byte offset (between
// 8-row core-matrix groups), descriptor version 1, no swizzle.
CN_DEV uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor of kind::tf32: fp32 accumulator, tf32 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
CN_DEV uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
CN_DEV void umma_tf32(uint32_t dtmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
        "l"(ad), "l"(bd), "r"(idesc), "r"(accum));
}
// Arrives on bar once every MMA this thread issued so far has completed.
CN_DEV void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
            smem_u32(bar))
        : "memory");
}
CN_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
CN_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// 32 lanes x 32 consecutive columns of TMEM: thread i gets lane (base + i).
CN_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
// The tf32 part the tensor cores read (low 13 mantissa bits dropped) and
// the exact remainder.
CN_DEV float tf32_trunc(float v) { return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u); }
CN_DEV float tf32_rest(float v) { return v - tf32_trunc(v); }
// 32 lanes x 16 consecutive columns, without the wait (tmem_wait_ld).
CN_DEV void tmem_ld16(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// 32 lanes x 8 consecutive columns, without the wait (tmem_wait_ld).
CN_DEV void tmem_ld8(uint32_t taddr, uint32_t *r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
// 32 lanes x 4 consecutive columns, without the wait (tmem_wait_ld).
CN_DEV void tmem_ld4(uint32_t taddr, uint32_t *r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}
// 32 lanes x 2 consecutive columns, without the wait (tmem_wait_ld).
CN_DEV void tmem_ld2(uint32_t taddr, uint32_t *r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];\n"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(taddr));
}
CN_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }


// Bounded wait with a CTA-local abort: after one wait gives up (limit_ns of
// GPU wall time without the phase completing), every role stops at its next
// wait instead of running into further timeouts.
CN_DEV bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *abort, int *err,
                    uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                flag_error(err, ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

// The same bounded wait with the thread suspended in hardware between polls
// (up to 20 us each, woken when the phase completes): for roles that wait
// most of the time, so their polling does not take issue slots from the
// warps that work.  The abort flag and the limit are checked after every
// poll.
CN_DEV bool tc_wait_sleep(uint64_t *bar, uint32_t parity, volatile int *abort, int *err,
                          uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            flag_error(err, ERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

}  // namespace cn
