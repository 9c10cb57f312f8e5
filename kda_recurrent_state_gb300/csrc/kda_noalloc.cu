// kda_noalloc.cu -- kda_bwd with the library's own static scratch instead of a caller
// workspace.  The array lives in this translation unit alone.  Under lazy module loading
// (CUDA_MODULE_LOADING=LAZY, the CUDA 12+ default) it is reserved on a device only when this
// entry point is first used there; with CUDA_MODULE_LOADING=EAGER every context that loads
// libkda reserves it when the context is created.
#include "kda_internal.cuh"

static __device__ __align__(256) unsigned char g_bwd_scratch[KDA_NOALLOC_SCRATCH_BYTES];

namespace {
// Device address of the static scratch on the current device.  Looked up on every call, not
// cached: after a cudaDeviceReset the module is loaded again and a cached address would point
// into memory the library no longer owns.  The first lookup on a device loads the module
// (lazy loading), so the first call should come before any stream capture.
void* scratch_ptr() {
    void* p = nullptr;
    return cudaGetSymbolAddress(&p, g_bwd_scratch) == cudaSuccess ? p : nullptr;
}
}  // namespace

extern "C" int kda_bwd_noalloc(const void* q, const void* k, const void* v, const float* log_alpha, int gate,
                               const float* beta, const float* init_states, const float* d_out,
                               const float* d_final_states, const int64_t* cu_seqlens, int N, int64_t T, int H,
                               int dk, int dv, float* dq, float* dk_out, float* dv_out, float* dlog_alpha,
                               float* dbeta, float* d_init_states, int in_dtype, void* stream) {
    if (N < 0 || T < 0 || H < 0) return KDA_ERR_INVALID_ARG;
    const int64_t T_total = cu_seqlens ? T : (int64_t)N * T;
    if (N > 0 && H > 0 && kda_workspace_size(KDA_OP_BWD, N, T_total, H, dk, dv, 64) > KDA_NOALLOC_SCRATCH_BYTES)
        return KDA_ERR_SCRATCH_TOO_SMALL;
    void* ws = scratch_ptr();
    if (!ws) return KDA_ERR_CUDA;
    return kda_bwd(q, k, v, log_alpha, gate, beta, init_states, d_out, d_final_states, cu_seqlens, N, T, H, dk, dv,
                   dq, dk_out, dv_out, dlog_alpha, dbeta, d_init_states, in_dtype, ws, KDA_NOALLOC_SCRATCH_BYTES,
                   stream);
}
