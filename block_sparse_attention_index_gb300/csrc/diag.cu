// Diagnostics: the bounded wait that every barrier wait of the library uses,
// made to run out on purpose.  One thread waits on a barrier that nothing
// arrives on; after limit_ns it gives up, sets the timeout bit of the error
// word and returns, and the context stays usable.  No copy, no tensor memory
// and no other CTA is involved.
#include "common.cuh"
#include "internal.h"

namespace msa {

__global__ void wait_timeout_check_kernel(uint32_t* err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait(&bar, 0, err, limit_ns);  // nothing arrives: gives up after limit_ns
}

cudaError_t run_wait_timeout_check(uint32_t* err, uint64_t limit_ns, cudaStream_t stream) {
    wait_timeout_check_kernel<<<1, 1, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace msa
