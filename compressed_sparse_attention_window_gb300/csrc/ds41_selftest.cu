// ds41_selftest.cu - the failure path of the bounded device-side waits, run on
// purpose: a kernel that holds tensor memory waits on an mbarrier that nobody
// arrives on, with a short poll bound, gives up, raises DS41_E_TIMEOUT, frees
// its tensor memory and returns.  Every mbarrier wait of the tensor-core
// kernels goes through the same tc::wait_bar.
#include "ds41_tc.cuh"

namespace ds41 {

__global__ void __launch_bounds__(64) wait_timeout_kernel(uint32_t polls, int arrive,
                                                          unsigned int* status, int32_t* out) {
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_f;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_f = 0;
        mbar_init_fence();
    }
    if (warp == 0) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;\n" ::"r"(
                smem_u32(&tmem_slot))
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    int done = 1;
    if (threadIdx.x == 0) {
        if (arrive) tc::mbar_arrive(&bar);
        done = tc::wait_bar(&bar, 0, &abort_f, status, polls) ? 1 : 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) out[0] = done;
    if (threadIdx.x == 32) out[1] = abort_f;  // seen by another warp after the barrier
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;\n" ::"r"(tmem_slot)
                     : "memory");
    }
}

}  // namespace ds41

extern "C" int ds41_selftest_wait_timeout(uint32_t polls, int arrive, int32_t* result,
                                          ds41_stream_t stream) {
    const char* name = "ds41_selftest_wait_timeout";
    DS41_REQUIRE(result && ds41::aligned16(result), DS41_E_ARG,
                 "%s: result must be a 16-byte aligned device pointer", name);
    DS41_REQUIRE(polls >= 1 && polls <= (1u << 22), DS41_E_ARG, "%s: polls=%u out of 1..2^22",
                 name, polls);
    unsigned int* status = nullptr;
    int rc = ds41::status_word(&status);
    if (rc) return rc;
    ds41::wait_timeout_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(polls, arrive ? 1 : 0, status,
                                                                   result);
    return ds41::launch_check(name);
}
