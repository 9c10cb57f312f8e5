// kda_chunk.cu -- chunkwise KDA prefill on tcgen05 tensor cores (chunk = 64).
#include "kda_internal.cuh"

namespace kda {

size_t chunk_prefill_workspace(int N, int H) { (void)N; (void)H; return 0; }

cudaError_t launch_chunk_prefill(const SeqProblem& p, int in_dtype, int out_dtype, void* workspace,
                                 size_t ws_bytes, cudaStream_t st) {
    (void)p; (void)in_dtype; (void)out_dtype; (void)workspace; (void)ws_bytes; (void)st;
    return cudaErrorNotSupported;
}

}  // namespace kda
