// Bounded mbarrier wait shared by the streaming kernels.
#pragma once
#include "mhcpb_internal.h"
#include "ptx.cuh"

namespace mhcpb {

// Returns false when the CTA is aborting (another role timed out) or when this
// wait exceeded the time limit; in the latter case it raises the CTA's abort
// flag and records the timeout in the status word.  With honor_abort == false
// it keeps waiting (still bounded) while aborting: used to drain a role's own
// in-flight copies and MMAs before exit.
static __device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity,
                                             volatile uint32_t* abort_flag, uint32_t* status,
                                             uint64_t timeout_ns, bool honor_abort) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0) {
            if (honor_abort && *abort_flag) return false;
            if (ptx::globaltimer() - t0 > timeout_ns) {
                *abort_flag = 1u;
                atomicCAS(status, kDevOk, kDevTimeout);
                return false;
            }
        }
    }
}

}  // namespace mhcpb
