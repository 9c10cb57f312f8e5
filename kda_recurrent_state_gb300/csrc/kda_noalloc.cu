// kda_noalloc.cu -- kda_bwd with the library's own static scratch instead of a caller
// workspace.  The array lives in this translation unit alone, so it is reserved only when
// this entry point is first used on a device (lazy module loading), not by every user of
// the library.
#include <mutex>

#include "kda_internal.cuh"

static __device__ __align__(256) unsigned char g_bwd_scratch[KDA_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the static scratch on the current device, looked up once per device.
void* scratch_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
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
