// tcgen05 tensor-core qdot_t (placeholder until the kernel lands).
#include "pq_internal.h"

namespace pq {

__device__ unsigned g_pq_status;

cudaError_t launch_qdot_tc(const QdotArgs&, cudaStream_t) { return cudaErrorNotSupported; }

cudaError_t read_and_clear_status(unsigned* status) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_pq_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_pq_status, &zero, sizeof(unsigned));
}

}  // namespace pq
