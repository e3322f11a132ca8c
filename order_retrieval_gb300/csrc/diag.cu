// diag.cu -- a check of the bounded mbarrier wait that the TMA-fed and tcgen05
// kernels rely on: one thread waits on a shared-memory mbarrier that is (or is
// not) completed, with a given poll limit; a wait that gives up writes
// ZETA_ERR_DEVICE_TIMEOUT to the status word and the kernel returns normally,
// so the context stays usable.  Nothing faults, traps or spins without a limit.
#include "mma.cuh"

namespace zeta {
namespace {

__global__ void bounded_wait_check(uint32_t limit, int arrive, int32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (arrive)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&bar)) : "memory");
    if (!mbar_wait_limit(&bar, 0, limit)) set_status(status, ZETA_ERR_DEVICE_TIMEOUT);
}

}  // namespace

cudaError_t launch_bounded_wait_check(uint32_t limit, int arrive, int32_t *status,
                                      cudaStream_t st) {
    bounded_wait_check<<<1, 32, 0, st>>>(limit, arrive, status);
    return cudaGetLastError();
}

}  // namespace zeta
