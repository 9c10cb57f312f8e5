// kda_host.cu -- the chunked prefill streamed from host memory: the sequence is cut into
// segments of whole chunks, and each segment's host-to-device copy, kernel and
// device-to-host copy run on three streams, so that the copies of one segment overlap the
// work on its neighbours.  A run resumed at a chunk boundary reproduces the unsplit run bit
// for bit, so the result equals kda_chunk_fwd on the whole sequence.
#include <nvtx3/nvToolsExt.h>

#include "kda_internal.cuh"

namespace {

constexpr int64_t kDefaultSegment = 4096;  // tokens per segment when the caller passes 0

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Staging layout of one segment buffer (all pieces 16-byte aligned).
struct SegLayout {
    size_t q, k, v, la, beta, out, bytes;
};

SegLayout seg_layout(int B, int H, int64_t L, int es, int oes) {
    const size_t th = (size_t)B * (size_t)L * (size_t)H;  // token-heads in a segment
    SegLayout s{};
    size_t o = 0;
    s.q = o; o += align16(th * kda::kD * es);
    s.k = o; o += align16(th * kda::kD * es);
    s.v = o; o += align16(th * kda::kD * es);
    s.la = o; o += align16(th * kda::kD * 4);
    s.beta = o; o += align16(th * 4);
    s.out = o; o += align16(th * kda::kD * oes);
    s.bytes = o;
    return s;
}

struct Range {
    explicit Range(const char* n) { nvtxRangePushA(n); }
    ~Range() { nvtxRangePop(); }
};

}  // namespace

extern "C" size_t kda_host_fwd_workspace_size(int B, int H, int dk, int dv, int64_t segment_tokens, int in_dtype,
                                              int out_dtype) {
    if (B <= 0 || H <= 0 || dk != kda::kD || dv != kda::kD || segment_tokens < 0) return 0;
    const int64_t L = segment_tokens ? segment_tokens : kDefaultSegment;
    const SegLayout s = seg_layout(B, H, L, in_dtype == KDA_BF16 ? 2 : 4, out_dtype == KDA_BF16 ? 2 : 4);
    return 2 * s.bytes + 2 * align16((size_t)B * H * kda::kD * kda::kD * 4) + kda::chunk_prefill_workspace(B, H);
}

extern "C" int kda_chunk_fwd_host(const void* q, const void* k, const void* v, const float* log_alpha,
                                  const float* beta, const float* init_state, void* out, float* final_state,
                                  int B, int64_t T, int H, int dk, int dv, int in_dtype, int out_dtype,
                                  int64_t segment_tokens, void* workspace, size_t ws_bytes, void* stream) {
    Range nvtx_range("kda_chunk_fwd_host");
    if (B < 0 || T < 0 || H < 0 || segment_tokens < 0) return KDA_ERR_INVALID_ARG;
    if ((in_dtype != KDA_BF16 && in_dtype != KDA_F32) || (out_dtype != KDA_BF16 && out_dtype != KDA_F32))
        return KDA_ERR_INVALID_ARG;
    if (dk != kda::kD || dv != kda::kD) return KDA_ERR_UNSUPPORTED;
    const int64_t L = segment_tokens ? segment_tokens : kDefaultSegment;
    if (L % 64 != 0) return KDA_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return KDA_OK;
    if (T > 0 && (!q || !k || !v || !log_alpha || !beta || !out)) return KDA_ERR_INVALID_ARG;
    const size_t need = kda_host_fwd_workspace_size(B, H, dk, dv, L, in_dtype, out_dtype);
    if (!workspace || ws_bytes < need) return KDA_ERR_WORKSPACE;
    const bool ws_misaligned = (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0;
    if (ws_misaligned || (init_state && (reinterpret_cast<uintptr_t>(init_state) & 15u))) return KDA_ERR_MISALIGNED;

    const int es = in_dtype == KDA_BF16 ? 2 : 4, oes = out_dtype == KDA_BF16 ? 2 : 4;
    const SegLayout lay = seg_layout(B, H, L, es, oes);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t state_bytes = (size_t)B * H * kda::kD * kda::kD * 4;
    float* states[2] = {reinterpret_cast<float*>(ws + 2 * lay.bytes),
                        reinterpret_cast<float*>(ws + 2 * lay.bytes + align16(state_bytes))};
    // the prefill's own workspace (a flag per (sequence, head)), reused by every segment in order
    uint8_t* kws = ws + 2 * lay.bytes + 2 * align16(state_bytes);
    const size_t kws_bytes = kda::chunk_prefill_workspace(B, H);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    cudaStream_t hs = nullptr, ds = nullptr;  // host-to-device and device-to-host copy streams
    cudaEvent_t ev[8] = {};                   // in_ready[2], comp_done[2], out_done[2], entry, end
    bool ok = cudaStreamCreateWithFlags(&hs, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&ds, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; i < 8 && ok; ++i) ok = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
    cudaEvent_t *in_ready = ev, *comp_done = ev + 2, *out_done = ev + 4, entry = ev[6], end = ev[7];
    int rc = ok ? KDA_OK : KDA_ERR_CUDA;
    auto chk = [&](cudaError_t e) {
        if (e != cudaSuccess && rc == KDA_OK) rc = KDA_ERR_CUDA;
        return rc == KDA_OK;
    };
    // the staging buffers may still be in use by earlier work on the caller's stream
    if (rc == KDA_OK) chk(cudaEventRecord(entry, cs)) && chk(cudaStreamWaitEvent(hs, entry, 0)) &&
                          chk(cudaStreamWaitEvent(ds, entry, 0));

    const int64_t nseg = (T + L - 1) / L;
    const size_t row_in = (size_t)H * kda::kD * es, row_la = (size_t)H * kda::kD * 4, row_b = (size_t)H * 4;
    const size_t row_out = (size_t)H * kda::kD * oes;
    if (rc == KDA_OK && nseg == 0) {  // no tokens: the final state is the initial state
        const int r = kda_chunk_fwd(nullptr, nullptr, nullptr, nullptr, nullptr, init_state, nullptr, states[0], B, 0,
                                    H, dk, dv, 64, in_dtype, out_dtype, nullptr, 0, stream);
        if (r != KDA_OK) rc = r;
        if (rc == KDA_OK) chk(cudaEventRecord(comp_done[0], cs));
    }
    for (int64_t s = 0; s < nseg && rc == KDA_OK; ++s) {
        const int b = (int)(s & 1);
        const int64_t s0 = s * L, Ls = (T - s0) < L ? (T - s0) : L;
        uint8_t* buf = ws + b * lay.bytes;
        // host -> device: one 2-D copy per tensor (rows = batch entries of the segment)
        auto h2d = [&](size_t off, const void* src, size_t row) {
            const uint8_t* from = static_cast<const uint8_t*>(src) + (size_t)s0 * row;
            return chk(cudaMemcpy2DAsync(buf + off, (size_t)Ls * row, from, (size_t)T * row, (size_t)Ls * row, (size_t)B,
                                         cudaMemcpyHostToDevice, hs));
        };
        if (s >= 2 && !chk(cudaStreamWaitEvent(hs, comp_done[b], 0))) break;
        if (!(h2d(lay.q, q, row_in) && h2d(lay.k, k, row_in) && h2d(lay.v, v, row_in) &&
              h2d(lay.la, log_alpha, row_la) && h2d(lay.beta, beta, row_b) && chk(cudaEventRecord(in_ready[b], hs))))
            break;
        // the kernel, on the caller's stream
        if (!chk(cudaStreamWaitEvent(cs, in_ready[b], 0))) break;
        if (s >= 2 && !chk(cudaStreamWaitEvent(cs, out_done[b], 0))) break;
        const float* s_in = s == 0 ? init_state : states[(s - 1) & 1];
        const int r = kda_chunk_fwd(buf + lay.q, buf + lay.k, buf + lay.v, reinterpret_cast<const float*>(buf + lay.la),
                                    reinterpret_cast<const float*>(buf + lay.beta), s_in, buf + lay.out, states[s & 1],
                                    B, Ls, H, dk, dv, 64, in_dtype, out_dtype, kws, kws_bytes, stream);
        if (r != KDA_OK) {
            rc = r;
            break;
        }
        if (!chk(cudaEventRecord(comp_done[b], cs))) break;
        // device -> host
        if (!(chk(cudaStreamWaitEvent(ds, comp_done[b], 0)) &&
              chk(cudaMemcpy2DAsync(static_cast<uint8_t*>(out) + (size_t)s0 * row_out, (size_t)T * row_out,
                                    buf + lay.out, (size_t)Ls * row_out, (size_t)Ls * row_out, (size_t)B,
                                    cudaMemcpyDeviceToHost, ds)) &&
              chk(cudaEventRecord(out_done[b], ds))))
            break;
    }
    if (rc == KDA_OK && final_state) {  // after the last kernel (or the no-token copy) wrote it
        const int last = nseg > 0 ? (int)((nseg - 1) & 1) : 0;
        chk(cudaStreamWaitEvent(ds, comp_done[last], 0)) &&
            chk(cudaMemcpyAsync(final_state, states[last], state_bytes, cudaMemcpyDeviceToHost, ds));
    }
    // the call is complete on the caller's stream once both copy streams are
    if (rc == KDA_OK)
        chk(cudaEventRecord(end, ds)) && chk(cudaStreamWaitEvent(cs, end, 0)) && chk(cudaEventRecord(entry, hs)) &&
            chk(cudaStreamWaitEvent(cs, entry, 0));
    for (int i = 0; i < 8; ++i)
        if (ev[i]) cudaEventDestroy(ev[i]);
    if (hs) cudaStreamDestroy(hs);
    if (ds) cudaStreamDestroy(ds);
    return rc;
}
