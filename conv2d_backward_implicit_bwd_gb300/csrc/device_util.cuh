// device_util.cuh -- small device helpers shared by the kernels: shared-memory
// barriers with bounded waits, and the status word protocol.
//
// Every blocking wait in this library is bounded: it spins on
// mbarrier.try_wait for at most `budget` SM clock cycles, then records a
// status code in the plan's device status word (first writer wins), raises a
// block-local abort flag so the other roles stop waiting too, and returns
// false.  Nothing traps; the host reads the status word afterwards.
#pragma once
#include <stdint.h>

namespace cbd {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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

__device__ __forceinline__ void record_status(int32_t *status, int32_t code) {
    if (status) atomicCAS(status, 0, code);
}

// Wait until the barrier's phase with the given parity has completed.  Gives
// up after `budget` cycles or as soon as *abort is set by another role.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int64_t budget,
                                                  volatile int32_t *abort, int32_t *status, int32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (abort && *abort) return false;
            if (clock64() - t0 > budget) {
                record_status(status, code);
                if (abort) *abort = 1;
                return false;
            }
        }
    }
}

// Timeline stamp of the instrumented build (-DCBD_PHASE_TIMES): globaltimer
// (ns) into slot `slot` of this CTA's row of `log`.  Compiles to nothing
// otherwise.
#ifdef CBD_PHASE_TIMES
#define CBD_PHASE(params, slot)                                                                 \
    do {                                                                                        \
        if ((params).phase_log) {                                                               \
            unsigned long long t_;                                                              \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                              \
            (params).phase_log[(size_t)blockIdx.x * kPhaseSlots + (slot)] = t_;                 \
        }                                                                                       \
    } while (0)
#else
#define CBD_PHASE(params, slot) \
    do {                        \
    } while (0)
#endif

}  // namespace cbd
