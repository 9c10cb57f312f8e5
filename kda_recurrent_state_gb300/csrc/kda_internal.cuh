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
    float* snapshots;             // [snap_offsets[N], H, D, D], or the pool when snap_slots is set
    int* status;                  // device status word
};

// State pool (both null for the packed layout): sequence s starts from pool slot
// init_slots[s] of SeqProblem::init (-1: zeros), and its snapshot k = snap_offsets[s] + m - 1
// goes to slot snap_slots[k] of SeqProblem::snapshots (-1: not stored).  A slot is [H, D, D].
// Kept out of SeqProblem so that the chunk kernel's parameter block keeps its size.
// A slot index outside [-1, n_slots) is skipped and raises KDA_STATUS_SLOT_RANGE.
// A bf16 pool (the launchers' pool_bf16) holds bf16 states: read widened exactly, snapshots
// stored rounded to nearest (the arithmetic stays fp32).
struct PoolSlots {
    const int64_t* init_slots;
    const int64_t* snap_slots;
    int64_t n_slots;
    int* claim;  // chunk kernel only: [2] unit counters (first pass, exact pass), or null (unit = CTA index)
};

// Pool slot `i` checked against the pool: -1 (none) passes through, anything else outside
// [0, n) becomes -1 and records KDA_STATUS_SLOT_RANGE.
__device__ inline int64_t checked_slot(int64_t i, int64_t n, int* status) {
    if (i < -1 || i >= n) {
        atomicCAS(status, 0, (int)KDA_STATUS_SLOT_RANGE);
        return -1;
    }
    return i;
}

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

// Gradients of L = sum_t <dout_t, o_t> + <dfinal, S_T> (training).  Sequences as in
// SeqProblem; gradients in the layouts of their inputs (dlog_alpha per the gate mode).
struct BwdProblem {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const float* beta;
    const float* init;    // [N, H, D, D] or nullptr
    const float* dout;    // [tokens, H, D]
    const float* dfinal;  // [N, H, D, D] or nullptr
    float* dq;
    float* dk;
    float* dv;
    float* dlog_alpha;
    float* dbeta;
    float* dinit;         // [N, H, D, D] or nullptr
    const int64_t* cu_seqlens;
    int64_t T_uniform;
    int64_t T_total;
    int N;
    int H;
    int gate;
    float* ckpt;          // set by launch_bwd from the workspace
    float* scratch;
    int64_t ckpt_slots;
    const int* redo;      // token-serial backward: nullptr, or [N*H] with only units u, redo[u] != 0, computed
};
size_t bwd_workspace(int N, int64_t T_total, int H);
cudaError_t launch_bwd(BwdProblem p, int in_dtype, void* workspace, cudaStream_t st);
// The chunked backward (C = 64): workspace bytes for N sequences, T_total tokens, H heads
// (varlen: packed by cu_seqlens), and its launch sequence.
size_t chunk_bwd_workspace(int N, int64_t T_total, int H, bool varlen);
cudaError_t launch_chunk_bwd(const BwdProblem& p, int in_dtype, void* workspace, int* status, cudaStream_t st);

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_decode(const DecodeProblem& p, int in_dtype, int out_dtype, int state_dtype, cudaStream_t st);
// `gate` (a GateMode) travels beside the problem: the chunk kernel takes it as a template
// argument, so it is not part of the kernel's parameter block.
cudaError_t launch_serial_prefill(const SeqProblem& p, const PoolSlots& pool, bool pool_bf16, int gate, int in_dtype,
                                  int out_dtype, cudaStream_t st);
cudaError_t launch_chunk_prefill(const SeqProblem& p, const PoolSlots& pool, bool pool_bf16, int gate, int in_dtype,
                                 int out_dtype, void* workspace, size_t ws_bytes, cudaStream_t st);
size_t chunk_prefill_workspace(int N, int H);
cudaError_t launch_bounded_wait_selftest(int* status, cudaStream_t st);

}  // namespace kda
