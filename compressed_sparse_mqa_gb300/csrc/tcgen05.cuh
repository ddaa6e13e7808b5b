// tcgen05.cuh -- thin inline-PTX wrappers for the 5th-generation tensor cores
// (tcgen05.mma with the accumulator in tensor memory), mbarriers and the
// shared-memory matrix descriptors, as used by the ds4a tensor-core kernels.
#pragma once

#include <stdint.h>

#include "ds4a_common.cuh"

namespace ds4a {
namespace tc {

DS4A_DEVINL uint32_t smem_u32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// Shared-memory matrix descriptor, 128-byte swizzle.  K-major operands: rows of
// 64 fp16 (128 B) per swizzle atom, 8-row groups SBO bytes apart; the start
// address advances 32 B per K=16 step inside an atom.  MN-major operands: rows
// are K, 64 fp16 of M/N per atom, atoms along M/N LBO bytes apart, 8-row (K)
// groups SBO bytes apart.
DS4A_DEVINL uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;   // descriptor version
    d |= static_cast<uint64_t>(2) << 61;   // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16 with fp16 A and B, fp32 D.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (static_cast<uint32_t>(a_mn_major) << 15) | (static_cast<uint32_t>(b_mn_major) << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// byte offset of fp16 element c (0..63) of row r inside a 128-byte-swizzled atom column
DS4A_DEVINL uint32_t sw128(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((((c >> 3) ^ (r & 7)) << 4) | ((c & 7) * 2)));
}
// byte offset of 16-byte chunk ch (0..7) of row r inside a 128-byte-swizzled atom column
DS4A_DEVINL uint32_t sw128_chunk(int r, int ch) { return static_cast<uint32_t>(r * 128 + ((ch ^ (r & 7)) << 4)); }

DS4A_DEVINL void mma_f16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(da), "l"(db), "r"(idesc), "r"(accumulate));
}

DS4A_DEVINL void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

DS4A_DEVINL void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
DS4A_DEVINL void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }

DS4A_DEVINL uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Each try_wait may suspend the thread in hardware (woken when the phase
// completes) for up to this long, so waiting warps do not spin on issue slots
// that the warps doing the work need.
constexpr uint32_t kSuspendHintNs = 20000;

// Bounded wait for the phase with the given parity to complete.  The bound is
// wall-clock time (try_wait may itself suspend for a while, so a poll count is
// no bound); returns false if the phase did not complete within `limit_ns`.
DS4A_DEVINL bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns = 1000000000ull) {
    const uint32_t a = smem_u32(bar);
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(parity), "r"(kSuspendHintNs)
            : "memory");
        if (done) return true;
        const uint64_t now = globaltimer_ns();
        if (it == 0) t0 = now;
        else if (now - t0 > limit_ns) return false;
    }
}

DS4A_DEVINL void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
DS4A_DEVINL void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// make generic-proxy shared-memory writes (st.shared, cp.async) visible to the tensor cores
DS4A_DEVINL void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// Tensor-memory allocation: one full warp executes these.
DS4A_DEVINL void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}
DS4A_DEVINL void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols));
}

// 32 lanes x 16 consecutive 32-bit columns: lane i of the warp gets row (lane base + i).
DS4A_DEVINL void ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
DS4A_DEVINL void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

}  // namespace tc
}  // namespace ds4a
