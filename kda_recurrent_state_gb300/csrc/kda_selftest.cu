// kda_selftest.cu -- a diagnostic for the library's failure detection: one CTA waits, with the
// same bounded mbarrier wait every kernel of the library uses, on a barrier that nothing ever
// arrives at.  The wait gives up after its deadline (about 2 s), records KDA_ERR_TIMEOUT in the
// device status word, raises the CTA's abort flag so the other threads leave too, and the
// kernel returns: the context stays usable and the host reads the status.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

__global__ void __launch_bounds__(128) bounded_wait_selftest_kernel(int* status) {
    __shared__ uint64_t bar;
    __shared__ sm100::Abort ab;
    if (threadIdx.x == 0) {
        ab.flag = 0;
        sm100::mbar_init(&bar, 1);  // expects one arrival, which never comes
    }
    __syncthreads();
    sm100::mbar_wait(&bar, 0, &ab, status);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int* status, cudaStream_t st) {
    bounded_wait_selftest_kernel<<<1, 128, 0, st>>>(status);
    return cudaGetLastError();
}

}  // namespace kda
