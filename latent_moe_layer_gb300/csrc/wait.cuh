// Bounded mbarrier waits shared by the warp-specialised kernels (the prefill expert
// GEMMs and the decode GEMVs): every wait gives up after an iteration limit or
// kWaitCapNs of wall time, records an error status and raises the CTA's abort flag.
#pragma once

#include "k3moe_internal.h"
#include "ptx.cuh"

namespace k3 {

// try_wait with a suspend-time hint of 20 us: a waiting thread sleeps until the phase
// completes (or the hint runs out) instead of spinning on the issue slots its warp shares
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// Wait with the CTA abort flag: returns false on timeout or abort (after recording
// K3MOE_ERR_TIMEOUT with the caller's site code and raising the flag).
__device__ __forceinline__ bool role_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          uint32_t limit, int *status, int where)
{
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer();
    for (uint32_t i = 1; i < limit; ++i) {
        if (mbar_try_wait_hint(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((i & 255u) == 0 && globaltimer() - t0 > kWaitCapNs) break;
    }
    set_status(status, K3MOE_ERR_TIMEOUT, where);
    *abort_flag = 1;
    return false;
}

// Drain: wait (wall-clock bounded) for the last min(n, ring) uses of a TMA ring.
__device__ __forceinline__ void drain_ring(uint64_t *full, uint32_t issued, int ring)
{
    const uint32_t n = issued < (uint32_t)ring ? issued : (uint32_t)ring;
    for (uint32_t q = 0; q < n; ++q) {
        const uint32_t i2 = issued - 1 - q;
        mbar_wait(smem_u32(full + i2 % ring), (i2 / ring) & 1, 0xFFFFFFFFu);
    }
}

}  // namespace k3
