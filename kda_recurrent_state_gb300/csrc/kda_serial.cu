// kda_serial.cu -- token-serial KDA prefill on CUDA cores (the chunk = 1 path).
//
// Evaluates the "Kimi K3" article's (lshu.cn/news/263999) §四 recurrence one
// token at a time, i.e. the §六 chunking with chunks of one token.  It is the
// plain GPU formulation of the operator: no WY factors, no decay ratios, the
// fp32 state never leaves registers.  Columns of S evolve independently, so a
// work unit is (sequence, head, block of 32 value columns); a CTA of 8 warps
// holds the 128 x 32 block as 16 rows per warp x 32 lanes (one column each).
// Per token: decay, column prediction p = S'^T k (a cross-warp reduction),
// u = beta (v - p), rank-one write, read o = S^T q (a second reduction).
// Snapshots (hubwiz.com "Kimi K3 混合线性注意力", §5) are taken after every
// `interval` tokens of a sequence.  The decay is per key channel (KDA), one
// scalar per head (Gated DeltaNet) or absent (DeltaNet, alpha = 1).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int NJ = 32;  // value columns per work unit
constexpr int TB = 16;  // tokens staged in shared memory at a time

__device__ __forceinline__ float ldin(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float ldin(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ void stout(__nv_bfloat16* p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }
__device__ __forceinline__ void stout(float* p, size_t i, float x) { p[i] = x; }

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) serial_kernel(SeqProblem p, PoolSlots pool, int pool_bf16, int gate) {
    const int nblk = kD / NJ;
    const int jb = blockIdx.x % nblk;
    const int h = (blockIdx.x / nblk) % p.H;
    const int s = blockIdx.x / (nblk * p.H);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = jb * NJ + lane;
    int64_t t0, len;
    seq_bounds(p, s, t0, len);

    __shared__ float sk[TB][kD], sq[TB][kD], sa[TB][kD], sv[TB][NJ], sb[TB];
    __shared__ float red[2][8][NJ];

    const size_t sbase = ((size_t)s * p.H + h) * kD * kD;
    int64_t S0 = p.init ? (int64_t)sbase : -1;  // element offset of the initial state (-1: zeros)
    if (pool.init_slots) {
        const int64_t slot = checked_slot(pool.init_slots[s], pool.n_slots, p.status);
        S0 = slot >= 0 ? (slot * p.H + h) * kD * kD : -1;
    }
    float S[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const size_t e = (size_t)S0 + (size_t)(w * 16 + i) * kD + j;
        S[i] = S0 < 0 ? 0.f
             : pool_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.init)[e])
                         : p.init[e];
    }

    const Tin* q = static_cast<const Tin*>(p.q);
    const Tin* k = static_cast<const Tin*>(p.k);
    const Tin* v = static_cast<const Tin*>(p.v);
    Tout* out = static_cast<Tout*>(p.out);

    for (int64_t tb = 0; tb < len; tb += TB) {
        const int nt = (int)((len - tb) < TB ? (len - tb) : TB);
        __syncthreads();
        for (int idx = threadIdx.x; idx < TB * kD; idx += blockDim.x) {
            const int r = idx / kD, c = idx % kD;
            if (r < nt) {
                const size_t off = ((size_t)(t0 + tb + r) * p.H + h) * kD + c;
                sk[r][c] = ldin(k, off);
                sq[r][c] = ldin(q, off);
                sa[r][c] = gate == kGateChannel ? expf(p.log_alpha[off])
                           : gate == kGateHead  ? expf(p.log_alpha[(size_t)(t0 + tb + r) * p.H + h])
                                                : 1.f;
            }
        }
        for (int idx = threadIdx.x; idx < TB * NJ; idx += blockDim.x) {
            const int r = idx / NJ, c = idx % NJ;
            if (r < nt) sv[r][c] = ldin(v, ((size_t)(t0 + tb + r) * p.H + h) * kD + jb * NJ + c);
        }
        if (threadIdx.x < TB && (int)threadIdx.x < nt)
            sb[threadIdx.x] = p.beta[(size_t)(t0 + tb + threadIdx.x) * p.H + h];
        __syncthreads();

        for (int r = 0; r < nt; ++r) {
            float pp = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = w * 16 + i;
                S[i] *= sa[r][c];
                pp += sk[r][c] * S[i];
            }
            red[0][w][lane] = pp;
            __syncthreads();
            float pt = 0.f;
#pragma unroll
            for (int g = 0; g < 8; ++g) pt += red[0][g][lane];
            const float u = sb[r] * (sv[r][lane] - pt);
            float oo = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = w * 16 + i;
                S[i] += sk[r][c] * u;
                oo += sq[r][c] * S[i];
            }
            red[1][w][lane] = oo;
            __syncthreads();
            const int64_t t = tb + r;  // position within the sequence
            if (w == 0) {
                float ot = 0.f;
#pragma unroll
                for (int g = 0; g < 8; ++g) ot += red[1][g][lane];
                stout(out, ((size_t)(t0 + t) * p.H + h) * kD + j, ot);
            }
            if (p.snap_interval > 0 && (t + 1) % p.snap_interval == 0) {
                int64_t slot = p.snap_offsets[s] + (t + 1) / p.snap_interval - 1;
                if (pool.snap_slots) slot = checked_slot(pool.snap_slots[slot], pool.n_slots, p.status);
                if (slot >= 0 && p.snapshots) {
                    const size_t off = ((size_t)slot * p.H + h) * kD * kD;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const size_t e = off + (size_t)(w * 16 + i) * kD + j;
                        if (pool_bf16)
                            reinterpret_cast<__nv_bfloat16*>(p.snapshots)[e] = __float2bfloat16_rn(S[i]);
                        else
                            p.snapshots[e] = S[i];
                    }
                }
            }
        }
    }
    if (p.final_state) {
#pragma unroll
        for (int i = 0; i < 16; ++i) p.final_state[sbase + (size_t)(w * 16 + i) * kD + j] = S[i];
    }
}

}  // namespace

cudaError_t launch_serial_prefill(const SeqProblem& p, const PoolSlots& pool, bool pool_bf16, int gate, int in_dtype,
                                  int out_dtype, cudaStream_t st) {
    const int64_t units = (int64_t)p.N * p.H * (kD / NJ);
    if (units == 0) return cudaSuccess;
    const unsigned grid = (unsigned)units;
    if (in_dtype == KDA_BF16 && out_dtype == KDA_BF16)
        serial_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, st>>>(p, pool, pool_bf16 ? 1 : 0, gate);
    else if (in_dtype == KDA_BF16)
        serial_kernel<__nv_bfloat16, float><<<grid, 256, 0, st>>>(p, pool, pool_bf16 ? 1 : 0, gate);
    else if (out_dtype == KDA_BF16)
        serial_kernel<float, __nv_bfloat16><<<grid, 256, 0, st>>>(p, pool, pool_bf16 ? 1 : 0, gate);
    else
        serial_kernel<float, float><<<grid, 256, 0, st>>>(p, pool, pool_bf16 ? 1 : 0, gate);
    return cudaGetLastError();
}

}  // namespace kda
