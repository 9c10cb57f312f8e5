// kda_internal.cuh -- declarations shared by the libkda translation units.
// Not installed; the public interface is include/kda.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kD = 128;  // d_k = d_v supported by every kernel

// Layout of the decay gates log_alpha:
//   kGateChannel: one per key channel, [.., H, d_k] (KDA)
//   kGateHead:    one per head, [.., H] (Gated DeltaNet's scalar gate)
//   kGateNone:    no gates, alpha = 1 (DeltaNet); log_alpha is null
enum GateMode { kGateChannel = 0, kGateHead = 1, kGateNone = 2 };

// One prefill problem: N sequences x H heads.  Sequence s covers packed tokens
// [start(s), start(s) + len(s)).  With cu_seqlens == nullptr the sequences are
// uniform: start = s * T_uniform, len = T_uniform (the batched [B, T] layout).
struct SeqProblem {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const float* beta;
    const float* init;    // [N, H, D, D] or nullptr (zeros)
    float* final_state;   // [N, H, D, D] or nullptr
    void* out;            // [tokens, H, D]
    const int64_t* cu_seqlens;  // device [N+1] or nullptr
    int64_t T_uniform;
    int64_t T_total;
    int N;
    int H;
    int64_t snap_interval;        // 0 = none
    const int64_t* snap_offsets;  // device [N+1]
    float* snapshots;             // [snap_offsets[N], H, D, D]
    int* status;                  // device status word
};

struct DecodeProblem {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const float* beta;
    void* state;  // [B, H, D, D] fp32 or bf16
    void* out;
    int B;
    int H;
    int* status;  // device status word
    int gate;     // GateMode
};

__host__ __device__ inline void seq_bounds(const SeqProblem& p, int s, int64_t& start, int64_t& len) {
    if (p.cu_seqlens) {
        start = p.cu_seqlens[s];
        len = p.cu_seqlens[s + 1] - start;
    } else {
        start = (int64_t)s * p.T_uniform;
        len = p.T_uniform;
    }
}

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_decode(const DecodeProblem& p, int in_dtype, int out_dtype, int state_dtype, cudaStream_t st);
// `gate` (a GateMode) travels beside the problem: the chunk kernel takes it as a template
// argument, so it is not part of the kernel's parameter block.
cudaError_t launch_serial_prefill(const SeqProblem& p, int gate, int in_dtype, int out_dtype, cudaStream_t st);
cudaError_t launch_chunk_prefill(const SeqProblem& p, int gate, int in_dtype, int out_dtype, void* workspace,
                                 size_t ws_bytes, cudaStream_t st);
size_t chunk_prefill_workspace(int N, int H);

}  // namespace kda
