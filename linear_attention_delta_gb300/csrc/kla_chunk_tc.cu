// Tensor-core (tcgen05) chunkwise KLA forward pass -- placeholder until the
// kernel lands; not eligible for any shape yet.
#include "kla_internal.cuh"

namespace kla {

namespace {
__device__ unsigned int g_fault_word = 0;
}

bool chunk_tc_eligible(const FwdArgs&) { return false; }

cudaError_t launch_chunk_tc(const FwdArgs&, cudaStream_t) {
    return cudaErrorNotSupported;
}

cudaError_t read_and_clear_fault(cudaStream_t stream, unsigned int* word) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(word, g_fault_word, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(unsigned int));
}

}  // namespace kla
