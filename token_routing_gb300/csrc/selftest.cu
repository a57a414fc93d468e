// Self-test of the device-side bounded waits: a kernel waits on an object that nothing
// signals, with a short cycle budget, through the wait helper the layer's kernels use (an
// mbarrier phase wait, as in the tensor-core pipelines). The wait runs out, records
// MOE_ERR_DEVICE_TIMEOUT in the device error word and the kernel returns normally, so the
// context stays usable. No fault, trap or endless loop is involved.
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

// One thread waits for phase 0 of a fresh mbarrier that expects one arrival (none comes).
__global__ void __launch_bounds__(32) wait_timeout_kernel(long long budget, int* err, int* done) {
    __shared__ uint64_t mb;
    if (threadIdx.x == 0) {
        tc::mbar_init(&mb, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool ok = tc::mbar_wait(&mb, 0, err, budget);
        atomicAdd(done, ok ? 0 : 1);
    }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_selftest_wait_timeout(int32_t mode, int64_t budget_cycles, int32_t* timed_out, void* scratch,
                                       moe_stream_t stream) {
    (void)scratch;
    if (mode != 0 || budget_cycles < 1000 || budget_cycles > kSpinBudgetCycles || !timed_out)
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(timed_out, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, s>>>((long long)budget_cycles, device_error_word(), timed_out);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
