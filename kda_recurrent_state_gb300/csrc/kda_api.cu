// kda_api.cu -- the C ABI of libkda: host-side validation, the device status
// word and dispatch to the kernels.  Declarations and the contract of every
// entry point are in include/kda.h.
#include <nvtx3/nvToolsExt.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

// Device status word: kernels record the first fault they see (a bounded wait
// that ran out, a gate out of range) here instead of trapping.
__device__ int g_status;

// Device address of the status word on the current device, looked up on every call (not
// cached, so that it stays valid across a cudaDeviceReset, which reloads the module).
int* status_ptr() {
    void* p = nullptr;
    return cudaGetSymbolAddress(&p, g_status) == cudaSuccess ? static_cast<int*>(p) : nullptr;
}

// An NVTX range over one entry point, so that a profiler's timeline shows the library's calls.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool dtype_ok(int d) { return d == KDA_BF16 || d == KDA_F32; }

// Shape/dtype/alignment checks shared by the prefill entry points.
int check_common(int dk, int dv, int chunk, int in_dtype, int out_dtype) {
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return KDA_ERR_INVALID_ARG;
    if (dk != kD || dv != kD) return KDA_ERR_UNSUPPORTED;
    if (chunk != 1 && chunk != 64) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

int run_prefill(const SeqProblem& p, const PoolSlots& pool, bool pool_bf16, int gate, int chunk, int in_dtype,
                int out_dtype, void* ws, size_t ws_bytes, cudaStream_t st) {
    cudaError_t e = chunk == 1
                        ? launch_serial_prefill(p, pool, pool_bf16, gate, in_dtype, out_dtype, st)
                        : launch_chunk_prefill(p, pool, pool_bf16, gate, in_dtype, out_dtype, ws, ws_bytes, st);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" {

const char* kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: null pointer, negative size or bad enum";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: only dk = dv = 128 and chunk in {1, 64}";
        case KDA_ERR_MISALIGNED: return "KDA_ERR_MISALIGNED: pointers must be 16-byte aligned";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA call or kernel launch failed";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded wait inside a kernel expired";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace missing or too small";
        case KDA_STATUS_GATE_RANGE:
            return "KDA_STATUS_GATE_RANGE: no longer raised (units whose gates leave the chunked kernels' range are "
                   "recomputed exactly within the same call)";
        case KDA_STATUS_SLOT_RANGE:
            return "KDA_STATUS_SLOT_RANGE: a state-pool slot index was out of range and skipped";
        case KDA_ERR_SCRATCH_TOO_SMALL:
            return "KDA_ERR_SCRATCH_TOO_SMALL: the problem needs more scratch than the library's static 128 MiB";
        default: return "unknown kda status";
    }
}

int64_t kda_snapshot_count(int64_t seqlen, int64_t interval) {
    if (interval <= 0 || seqlen < 0) return 0;
    return seqlen / interval;
}

int kda_snapshot_offsets(const int64_t* cu_seqlens_host, int N, int64_t interval, int64_t* offsets_host) {
    if (!cu_seqlens_host || !offsets_host || N < 0 || interval < 0) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens_host[0] != 0) return KDA_ERR_INVALID_ARG;
    offsets_host[0] = 0;
    for (int s = 0; s < N; ++s) {
        const int64_t len = cu_seqlens_host[s + 1] - cu_seqlens_host[s];
        if (len < 0) return KDA_ERR_INVALID_ARG;
        offsets_host[s + 1] = offsets_host[s] + kda_snapshot_count(len, interval);
    }
    return KDA_OK;
}

int64_t kda_snapshot_lookup(const int64_t* offsets_host, int N, int seq, int64_t interval, int64_t prefix_len,
                            int64_t* covered_host) {
    if (!offsets_host || !covered_host || seq < 0 || seq >= N || interval <= 0 || prefix_len < 0) return -2;
    const int64_t have = offsets_host[seq + 1] - offsets_host[seq];
    int64_t m = prefix_len / interval;
    if (m > have) m = have;
    *covered_host = m * interval;
    return m > 0 ? offsets_host[seq] + m - 1 : -1;
}

size_t kda_workspace_size(int op, int B, int64_t T, int H, int dk, int dv, int chunk) {
    (void)dk; (void)dv;
    if (op == KDA_OP_BWD) return (B <= 0 || H <= 0 || T < 0) ? 0 : bwd_workspace(B, T, H);
    if (op == KDA_OP_CHUNK_BWD) {
        if (B <= 0 || H <= 0 || T < 0) return 0;
        return chunk == 64 ? chunk_bwd_workspace(B, T, H, true) : chunk == 1 ? bwd_workspace(B, T, H) : 0;
    }
    if (op == KDA_OP_DECODE || B <= 0 || H <= 0 || chunk != 64) return 0;
    return chunk_prefill_workspace(B, H);
}

int kda_get_device_status(void* stream) {
    int* addr = status_ptr();
    if (!addr) return KDA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int host = 0;
    if (cudaMemcpyAsync(&host, addr, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaMemsetAsync(addr, 0, sizeof(int), st) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ERR_CUDA;
    return host;
}

// The gates: per channel (16-byte aligned, TMA), per head (4-byte aligned) or none (null).
static bool gate_ok(const float* log_alpha, int gate, bool required) {
    if (gate == kGateNone) return log_alpha == nullptr;
    return log_alpha ? true : !required;
}
static bool gate_aligned(const float* log_alpha, int gate) {
    return !log_alpha || (gate == kGateChannel ? aligned16(log_alpha) : aligned(log_alpha, 4));
}

static int chunk_common(const void* q, const void* k, const void* v, const float* log_alpha, int gate,
                        const float* beta, const float* init_state, void* out, float* final_state, int B,
                        int64_t T, int H, int dk, int dv, int chunk, int in_dtype, int out_dtype, void* workspace,
                        size_t ws_bytes, void* stream) {
    if (B < 0 || T < 0 || H < 0) return KDA_ERR_INVALID_ARG;
    int rc = check_common(dk, dv, chunk, in_dtype, out_dtype);
    if (rc != KDA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (B == 0 || H == 0) return KDA_OK;
    const size_t state_bytes = (size_t)B * H * kD * kD * sizeof(float);
    if (T == 0) {  // nothing to run: the final state is the initial state
        if (!final_state) return KDA_OK;
        if (!aligned16(final_state) || (init_state && !aligned16(init_state))) return KDA_ERR_MISALIGNED;
        cudaError_t e = init_state ? (init_state == final_state
                                          ? cudaSuccess
                                          : cudaMemcpyAsync(final_state, init_state, state_bytes,
                                                            cudaMemcpyDeviceToDevice, st))
                                   : cudaMemsetAsync(final_state, 0, state_bytes, st);
        return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    }
    if (!q || !k || !v || !gate_ok(log_alpha, gate, true) || !beta || !out) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, init_state, out, final_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    if (!aligned(beta, 4) || !gate_aligned(log_alpha, gate)) return KDA_ERR_MISALIGNED;
    const size_t need = kda_workspace_size(KDA_OP_CHUNK, B, T, H, dk, dv, chunk);
    if (need > 0 && (!workspace || ws_bytes < need)) return KDA_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return KDA_ERR_MISALIGNED;

    SeqProblem p{};
    p.q = q; p.k = k; p.v = v; p.log_alpha = log_alpha; p.beta = beta;
    p.init = init_state; p.final_state = final_state; p.out = out;
    p.cu_seqlens = nullptr; p.T_uniform = T; p.T_total = (int64_t)B * T;
    p.N = B; p.H = H;
    p.snap_interval = 0; p.snap_offsets = nullptr; p.snapshots = nullptr;
    p.status = status_ptr();
    if (!p.status) return KDA_ERR_CUDA;
    return run_prefill(p, PoolSlots{nullptr, nullptr, 0}, false, gate, chunk, in_dtype, out_dtype, workspace, ws_bytes,
                       st);
}

int kda_chunk_fwd(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                  const float* init_state, void* out, float* final_state, int B, int64_t T, int H, int dk,
                  int dv, int chunk, int in_dtype, int out_dtype, void* workspace, size_t ws_bytes,
                  void* stream) {
    NvtxRange nvtx_range("kda_chunk_fwd");
    return chunk_common(q, k, v, log_alpha, kGateChannel, beta, init_state, out, final_state, B, T, H, dk, dv,
                        chunk, in_dtype, out_dtype, workspace, ws_bytes, stream);
}

int kda_gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                      const float* init_state, void* out, float* final_state, int B, int64_t T, int H, int dk,
                      int dv, int chunk, int in_dtype, int out_dtype, void* workspace, size_t ws_bytes,
                      void* stream) {
    NvtxRange nvtx_range("kda_gdn_chunk_fwd");
    return chunk_common(q, k, v, log_alpha, log_alpha ? kGateHead : kGateNone, beta, init_state, out, final_state,
                        B, T, H, dk, dv, chunk, in_dtype, out_dtype, workspace, ws_bytes, stream);
}

// `pool.init_slots` / `pool.snap_slots` select the pool layout: init_states and snapshots
// are then the same pool of pool.n_slots slots.
static int varlen_common(const void* q, const void* k, const void* v, const float* log_alpha, int gate,
                         const float* beta, const int64_t* cu_seqlens, int N, int64_t T_total, int H, int dk,
                         int dv, int chunk, const float* init_states, float* final_states,
                         int64_t snapshot_interval, const int64_t* snap_offsets, float* snapshots, void* out,
                         int in_dtype, int out_dtype, void* workspace, size_t ws_bytes, void* stream,
                         const PoolSlots& pool, bool pool_bf16) {
    if (N < 0 || T_total < 0 || H < 0 || snapshot_interval < 0) return KDA_ERR_INVALID_ARG;
    int rc = check_common(dk, dv, chunk, in_dtype, out_dtype);
    if (rc != KDA_OK) return rc;
    if (N == 0 || H == 0) return KDA_OK;
    if (!cu_seqlens || !final_states) return KDA_ERR_INVALID_ARG;
    if (!gate_ok(log_alpha, gate, T_total > 0)) return KDA_ERR_INVALID_ARG;
    if (T_total > 0 && (!q || !k || !v || !beta || !out)) return KDA_ERR_INVALID_ARG;
    if (snapshot_interval > 0) {
        if (snapshot_interval % chunk != 0) return KDA_ERR_INVALID_ARG;
        if (!snap_offsets) return KDA_ERR_INVALID_ARG;
    }
    const void* ptrs[] = {q, k, v, init_states, final_states, snapshots, out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    if ((beta && !aligned(beta, 4)) || !gate_aligned(log_alpha, gate) || !aligned(cu_seqlens, 8) ||
        (snap_offsets && !aligned(snap_offsets, 8)) || (pool.init_slots && !aligned(pool.init_slots, 8)) ||
        (pool.snap_slots && !aligned(pool.snap_slots, 8)))
        return KDA_ERR_MISALIGNED;
    const size_t need = kda_workspace_size(KDA_OP_VARLEN, N, T_total, H, dk, dv, chunk);
    if (need > 0 && (!workspace || ws_bytes < need)) return KDA_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return KDA_ERR_MISALIGNED;

    SeqProblem p{};
    p.q = q; p.k = k; p.v = v; p.log_alpha = log_alpha; p.beta = beta;
    p.init = init_states; p.final_state = final_states; p.out = out;
    p.cu_seqlens = cu_seqlens; p.T_uniform = 0; p.T_total = T_total;
    p.N = N; p.H = H;
    p.snap_interval = snapshot_interval; p.snap_offsets = snap_offsets; p.snapshots = snapshots;
    p.status = status_ptr();
    if (!p.status) return KDA_ERR_CUDA;
    return run_prefill(p, pool, pool_bf16, gate, chunk, in_dtype, out_dtype, workspace, ws_bytes,
                       static_cast<cudaStream_t>(stream));
}

int kda_varlen_fwd(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                   const int64_t* cu_seqlens, int N, int64_t T_total, int H, int dk, int dv, int chunk,
                   const float* init_states, float* final_states, int64_t snapshot_interval,
                   const int64_t* snap_offsets, float* snapshots, void* out, int in_dtype, int out_dtype,
                   void* workspace, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_range("kda_varlen_fwd");
    return varlen_common(q, k, v, log_alpha, kGateChannel, beta, cu_seqlens, N, T_total, H, dk, dv, chunk,
                         init_states, final_states, snapshot_interval, snap_offsets, snapshots, out, in_dtype,
                         out_dtype, workspace, ws_bytes, stream, PoolSlots{nullptr, nullptr, 0}, false);
}

int kda_gdn_varlen_fwd(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                       const int64_t* cu_seqlens, int N, int64_t T_total, int H, int dk, int dv, int chunk,
                       const float* init_states, float* final_states, int64_t snapshot_interval,
                       const int64_t* snap_offsets, float* snapshots, void* out, int in_dtype, int out_dtype,
                       void* workspace, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_range("kda_gdn_varlen_fwd");
    return varlen_common(q, k, v, log_alpha, log_alpha ? kGateHead : kGateNone, beta, cu_seqlens, N, T_total, H,
                         dk, dv, chunk, init_states, final_states, snapshot_interval, snap_offsets, snapshots, out,
                         in_dtype, out_dtype, workspace, ws_bytes, stream, PoolSlots{nullptr, nullptr, 0}, false);
}

int kda_varlen_fwd_pool(const void* q, const void* k, const void* v, const float* log_alpha, int gate,
                        const float* beta, const int64_t* cu_seqlens, int N, int64_t T_total, int H, int dk, int dv,
                        int chunk, void* pool, int64_t pool_slots, int pool_dtype, const int64_t* init_slots,
                        int64_t snapshot_interval, const int64_t* snap_offsets, const int64_t* snap_slots,
                        float* final_states, void* out, int in_dtype, int out_dtype, void* workspace,
                        size_t ws_bytes, void* stream) {
    NvtxRange nvtx_range("kda_varlen_fwd_pool");
    if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_HEAD && gate != KDA_GATE_NONE) return KDA_ERR_INVALID_ARG;
    if (pool_slots < 0 || !dtype_ok(pool_dtype)) return KDA_ERR_INVALID_ARG;
    if (snapshot_interval > 0 && !snap_slots) snapshot_interval = 0;  // no slot table: nothing is stored
    if ((init_slots || snapshot_interval > 0) && !pool) return KDA_ERR_INVALID_ARG;
    if (gate == KDA_GATE_HEAD && !log_alpha && T_total > 0) return KDA_ERR_INVALID_ARG;
    const int g = gate == KDA_GATE_CHANNEL ? kGateChannel : gate == KDA_GATE_HEAD ? kGateHead : kGateNone;
    float* pool_f = static_cast<float*>(pool);  // element type per pool_dtype; the kernels cast back
    return varlen_common(q, k, v, log_alpha, g, beta, cu_seqlens, N, T_total, H, dk, dv, chunk,
                         init_slots ? pool_f : nullptr, final_states, snapshot_interval, snap_offsets,
                         snapshot_interval > 0 ? pool_f : nullptr, out, in_dtype, out_dtype, workspace, ws_bytes,
                         stream, PoolSlots{init_slots, snapshot_interval > 0 ? snap_slots : nullptr, pool_slots},
                         pool_dtype == KDA_BF16);
}

static int decode_common(const void* q, const void* k, const void* v, const float* log_alpha, int gate,
                         const float* beta, void* state, int state_dtype, void* out, int B, int H, int dk, int dv,
                         int in_dtype, int out_dtype, void* stream) {
    if (B < 0 || H < 0) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return KDA_ERR_INVALID_ARG;
    if (dk != kD || dv != kD) return KDA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0) return KDA_OK;
    if (!q || !k || !v || !gate_ok(log_alpha, gate, true) || !beta || !state || !out) return KDA_ERR_INVALID_ARG;
    const uintptr_t in_al = in_dtype == KDA_BF16 ? 2 : 4, out_al = out_dtype == KDA_BF16 ? 2 : 4;
    if (!aligned16(state) || !aligned(q, in_al) || !aligned(k, in_al) || !aligned(v, in_al) ||
        (log_alpha && !aligned(log_alpha, 4)) || !aligned(beta, 4) || !aligned(out, out_al))
        return KDA_ERR_MISALIGNED;
    DecodeProblem p{q, k, v, log_alpha, beta, state, out, B, H, status_ptr(), gate};
    if (!p.status) return KDA_ERR_CUDA;
    return launch_decode(p, in_dtype, out_dtype, state_dtype, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

int kda_decode_step(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                    float* state, void* out, int B, int H, int dk, int dv, int in_dtype, int out_dtype,
                    void* stream) {
    NvtxRange nvtx_range("kda_decode_step");
    return decode_common(q, k, v, log_alpha, kGateChannel, beta, state, KDA_F32, out, B, H, dk, dv, in_dtype,
                         out_dtype, stream);
}

int kda_gdn_decode_step(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                        float* state, void* out, int B, int H, int dk, int dv, int in_dtype, int out_dtype,
                        void* stream) {
    NvtxRange nvtx_range("kda_gdn_decode_step");
    return decode_common(q, k, v, log_alpha, log_alpha ? kGateHead : kGateNone, beta, state, KDA_F32, out, B, H,
                         dk, dv, in_dtype, out_dtype, stream);
}

int kda_gdn_decode_step_bf16state(const void* q, const void* k, const void* v, const float* log_alpha,
                                  const float* beta, void* state, void* out, int B, int H, int dk, int dv,
                                  int in_dtype, int out_dtype, void* stream) {
    NvtxRange nvtx_range("kda_gdn_decode_step_bf16state");
    return decode_common(q, k, v, log_alpha, log_alpha ? kGateHead : kGateNone, beta, state, KDA_BF16, out, B, H,
                         dk, dv, in_dtype, out_dtype, stream);
}

int kda_decode_step_bf16state(const void* q, const void* k, const void* v, const float* log_alpha,
                              const float* beta, void* state, void* out, int B, int H, int dk, int dv,
                              int in_dtype, int out_dtype, void* stream) {
    NvtxRange nvtx_range("kda_decode_step_bf16state");
    return decode_common(q, k, v, log_alpha, kGateChannel, beta, state, KDA_BF16, out, B, H, dk, dv, in_dtype,
                         out_dtype, stream);
}

static int bwd_common(const void* q, const void* k, const void* v, const float* log_alpha, int gate,
                      const float* beta, const float* init_states, const float* d_out, const float* d_final_states,
                      const int64_t* cu_seqlens, int N, int64_t T, int H, int dk, int dv, int chunk, float* dq,
                      float* dk_out, float* dv_out, float* dlog_alpha, float* dbeta, float* d_init_states,
                      int in_dtype, void* workspace, size_t ws_bytes, void* stream) {
    if (N < 0 || T < 0 || H < 0) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(in_dtype)) return KDA_ERR_INVALID_ARG;
    if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_HEAD && gate != KDA_GATE_NONE) return KDA_ERR_INVALID_ARG;
    if (dk != kD || dv != kD || (chunk != 1 && chunk != 64)) return KDA_ERR_UNSUPPORTED;
    if (N == 0 || H == 0) return KDA_OK;
    const int64_t T_total = cu_seqlens ? T : (int64_t)N * T;
    const bool gated = gate != KDA_GATE_NONE;
    if (T_total > 0 && (!q || !k || !v || !beta || !d_out || !dq || !dk_out || !dv_out || !dbeta))
        return KDA_ERR_INVALID_ARG;
    if (T_total > 0 && gated != (log_alpha != nullptr)) return KDA_ERR_INVALID_ARG;
    if (T_total > 0 && gated != (dlog_alpha != nullptr)) return KDA_ERR_INVALID_ARG;
    const uintptr_t in_al = in_dtype == KDA_BF16 ? 2 : 4;
    const void* al4[] = {log_alpha, beta, d_out, dq, dk_out, dv_out, dlog_alpha, dbeta};
    for (const void* p : al4)
        if (p && !aligned(p, 4)) return KDA_ERR_MISALIGNED;
    if (!aligned(q, in_al) || !aligned(k, in_al) || !aligned(v, in_al) || (cu_seqlens && !aligned(cu_seqlens, 8)))
        return KDA_ERR_MISALIGNED;
    const void* al16[] = {init_states, d_final_states, d_init_states, workspace};
    for (const void* p : al16)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    if (chunk == 64 && !(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(d_out)))
        return KDA_ERR_MISALIGNED;  // read as 16-byte (fp32) or 8-byte (bf16) vectors
    const size_t need = kda_workspace_size(KDA_OP_CHUNK_BWD, N, T_total, H, dk, dv, chunk);
    if (need > 0 && (!workspace || ws_bytes < need)) return KDA_ERR_WORKSPACE;
    BwdProblem p{};
    p.q = q; p.k = k; p.v = v; p.log_alpha = log_alpha; p.beta = beta; p.init = init_states;
    p.dout = d_out; p.dfinal = d_final_states;
    p.dq = dq; p.dk = dk_out; p.dv = dv_out; p.dlog_alpha = dlog_alpha; p.dbeta = dbeta; p.dinit = d_init_states;
    p.cu_seqlens = cu_seqlens; p.T_uniform = cu_seqlens ? 0 : T; p.T_total = T_total; p.N = N; p.H = H;
    p.gate = gate == KDA_GATE_CHANNEL ? kGateChannel : gate == KDA_GATE_HEAD ? kGateHead : kGateNone;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (chunk == 1) return launch_bwd(p, in_dtype, workspace, st) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    int* status = status_ptr();
    if (!status) return KDA_ERR_CUDA;
    return launch_chunk_bwd(p, in_dtype, workspace, status, st) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_bwd(const void* q, const void* k, const void* v, const float* log_alpha, int gate, const float* beta,
            const float* init_states, const float* d_out, const float* d_final_states, const int64_t* cu_seqlens,
            int N, int64_t T, int H, int dk, int dv, float* dq, float* dk_out, float* dv_out, float* dlog_alpha,
            float* dbeta, float* d_init_states, int in_dtype, void* workspace, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_range("kda_bwd");
    return bwd_common(q, k, v, log_alpha, gate, beta, init_states, d_out, d_final_states, cu_seqlens, N, T, H, dk,
                      dv, 1, dq, dk_out, dv_out, dlog_alpha, dbeta, d_init_states, in_dtype, workspace, ws_bytes,
                      stream);
}

int kda_chunk_bwd(const void* q, const void* k, const void* v, const float* log_alpha, int gate, const float* beta,
                  const float* init_states, const float* d_out, const float* d_final_states,
                  const int64_t* cu_seqlens, int N, int64_t T, int H, int dk, int dv, int chunk, float* dq,
                  float* dk_out, float* dv_out, float* dlog_alpha, float* dbeta, float* d_init_states, int in_dtype,
                  void* workspace, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_range("kda_chunk_bwd");
    return bwd_common(q, k, v, log_alpha, gate, beta, init_states, d_out, d_final_states, cu_seqlens, N, T, H, dk,
                      dv, chunk, dq, dk_out, dv_out, dlog_alpha, dbeta, d_init_states, in_dtype, workspace,
                      ws_bytes, stream);
}

int kda_selftest_bounded_wait(void* stream) {
    NvtxRange nvtx_range("kda_selftest_bounded_wait");
    int* st = status_ptr();
    if (!st) return KDA_ERR_CUDA;
    return launch_bounded_wait_selftest(st, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
