// kda_bwd.cu -- gradients of the KDA recurrence (training), token by token on CUDA cores.
//
// The forward step is the "Kimi K3" article's (lshu.cn/news/263999) §四 update with the
// §二.1 read; the pages give no backward, so it is the reverse mode of that step, one
// operation at a time.  From S = S_{t-1}:
//     a = exp(log_alpha_t)    S' = Diag(a) S    p = S'^T k    e = v - p    u = beta e
//     S_t = S' + k u^T        o_t = S_t^T q
// and backwards, with dS = dL/dS_t carried from the later tokens:
//     dS += q do^T                     dq = S_t do
//     du = dS^T k                      dbeta = du . e        dv = beta du     dp = -beta du
//     dk = dS u + S' dp                dS' = dS + k dp^T
//     dlog_alpha_i = a_i sum_j dS'_ij S_ij                   dS_{t-1} = Diag(a) dS'
// for L = sum_t <do_t, o_t> + <dS_T, S_T>.
//
// One CTA of 512 threads walks one (sequence, head).  Thread (c, i) holds row i (key
// channel) of value columns 32c .. 32c+31 of both S and dS in registers.  Sums over key
// channels (p, du) stay inside one column block: a warp reduce-scatter and a 4-warp pass
// through shared memory behind a 128-thread barrier, so the four blocks run on their own.
// Sums over value columns (dq, dk, dlog_alpha, dbeta) add the four column blocks in a
// fixed order once per 8-token piece, so the result is bit-reproducible.
//
// States for the reverse sweep: a forward sweep stores S every 64 tokens (checkpoints,
// workspace).  Then, segment by segment from the end, the segment is recomputed from its
// checkpoint keeping S every 8 tokens (per-CTA scratch, small enough to stay in L2), and
// each 8-token piece is recomputed once more keeping every S_{t-1}, e_t and u_t before
// its tokens are undone in reverse order.  3 forward steps and 1 backward step per token.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int SEG = 64;         // tokens per checkpoint
constexpr int SUB = 8;          // tokens per recomputed piece
constexpr int NT = 512;         // threads: 4 column blocks x 128 rows
constexpr int BLK = kD * kD;    // floats per state image, laid out [column][row]

__device__ __forceinline__ float ldin(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float ldin(const float* p, size_t i) { return p[i]; }

// Reduce-scatter over a warp: lane l returns the sum over all 32 lanes of x[l].
__device__ __forceinline__ float warp_reduce_scatter(float (&x)[32], int lane) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        const bool up = (lane & d) != 0;  // this lane keeps the upper half of the live values
#pragma unroll
        for (int m = 0; m < d; ++m) {
            const float send = up ? x[m] : x[m + d];
            const float keep = up ? x[m + d] : x[m];
            x[m] = keep + __shfl_xor_sync(0xffffffffu, send, d);
        }
    }
    return x[0];
}

struct Shared {
    float q[SUB][kD], k[SUB][kD], a[SUB][kD], v[SUB][kD], dout[SUB][kD];
    float e[SUB][kD], u[SUB][kD];
    float beta[SUB];
    float red[2][4][4][32];    // [parity][column block][warp][lane]: per-warp column partials
    float rs[SUB][4][3][kD];   // [token][column block][dq, dk, dlog_alpha][row]: row partials
    float bpart[SUB][4];       // [token][column block]: dbeta partials
};

// Barrier of the 128 threads (4 warps) of column block c; the column sums need no more.
__device__ __forceinline__ void wg_sync(int c) { asm volatile("bar.sync %0, 128;" ::"r"(c + 1) : "memory"); }

template <typename Tin>
__global__ void __launch_bounds__(NT, 1) bwd_kernel(BwdProblem P) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Shared& sm = *reinterpret_cast<Shared*>(smem_raw);
    const int tid = threadIdx.x;
    const int c = tid >> 7, i = tid & 127, w = (tid >> 5) & 3, lane = tid & 31;
    const int h = blockIdx.x % P.H, s = blockIdx.x / P.H;
    if (P.redo && !P.redo[(size_t)s * P.H + h]) return;  // as the chunked backward's exact second pass
    int64_t t0, len;
    if (P.cu_seqlens) {
        t0 = P.cu_seqlens[s];
        len = P.cu_seqlens[s + 1] - t0;
    } else {
        t0 = (int64_t)s * P.T_uniform;
        len = P.T_uniform;
    }
    const size_t sbase = ((size_t)s * P.H + h) * BLK;  // row-major [D][D] states of this unit
    const Tin* gq = static_cast<const Tin*>(P.q);
    const Tin* gk = static_cast<const Tin*>(P.k);
    const Tin* gv = static_cast<const Tin*>(P.v);
    // workspace: checkpoints of this head, and this CTA's two 8-slot scratch areas
    const int64_t slot0 = t0 / SEG + s;  // first checkpoint slot of the sequence (slots never overlap)
    float* ckpt = P.ckpt + (size_t)h * P.ckpt_slots * BLK;
    float* sub = P.scratch + (size_t)blockIdx.x * 2 * SUB * BLK;
    float* st = sub + SUB * BLK;
    auto img = [&](float* base, int jj) -> float* { return base + (size_t)(c * 32 + jj) * kD + i; };
    int par = 0;  // parity of the column-partial buffer (the same sequence of steps in every warp)

    // S and dS of this thread's row, value columns in pairs (2p, 2p+1): the element-wise
    // work runs on packed fp32 pairs
    float2 S[16], dS[16];
#pragma unroll
    for (int p = 0; p < 16; ++p)
        S[p] = P.init ? *reinterpret_cast<const float2*>(P.init + sbase + (size_t)i * kD + c * 32 + 2 * p)
                      : make_float2(0.f, 0.f);

    // inputs of tokens [p0, p0 + n) of the sequence into shared memory
    auto stage = [&](int64_t p0, int n, bool with_dout) {
        __syncthreads();
        for (int idx = tid; idx < SUB * kD; idx += NT) {
            const int tl = idx >> 7, ch = idx & 127;
            if (tl < n) {
                const size_t r = (size_t)(t0 + p0 + tl) * P.H + h;
                const size_t off = r * kD + ch;
                sm.q[tl][ch] = ldin(gq, off);
                sm.k[tl][ch] = ldin(gk, off);
                sm.v[tl][ch] = ldin(gv, off);
                sm.a[tl][ch] = P.gate == kGateChannel ? expf(P.log_alpha[off])
                             : P.gate == kGateHead  ? expf(P.log_alpha[r])
                                                    : 1.f;
                if (with_dout) sm.dout[tl][ch] = P.dout[off];
            }
        }
        if (tid < n) sm.beta[tid] = P.beta[(size_t)(t0 + p0 + tid) * P.H + h];
        __syncthreads();
    };
    // column sum over this block's 128 rows of x[jj] (column 32c + jj): every lane gets
    // the total of its own column `32c + lane`
    auto col_sum = [&](float (&x)[32]) -> float {
        sm.red[par][c][w][lane] = warp_reduce_scatter(x, lane);
        wg_sync(c);
        const float t = ((sm.red[par][c][0][lane] + sm.red[par][c][1][lane]) + sm.red[par][c][2][lane]) +
                        sm.red[par][c][3][lane];
        par ^= 1;
        return t;
    };
    // one forward step on S (token tl of the staged piece); with `keep`, also S_{t-1}
    // into the scratch and e, u into shared memory for the backward steps
    auto fwd_step = [&](int tl, float* keep) {
        const float2 a2 = make_float2(sm.a[tl][i], sm.a[tl][i]), k2 = make_float2(sm.k[tl][i], sm.k[tl][i]);
        float x[32];
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            if (keep) {
                *img(keep, 2 * p) = S[p].x;
                *img(keep, 2 * p + 1) = S[p].y;
            }
            S[p] = __fmul2_rn(S[p], a2);
            const float2 kx = __fmul2_rn(S[p], k2);
            x[2 * p] = kx.x;
            x[2 * p + 1] = kx.y;
        }
        const int j = 32 * c + lane;
        const float e = sm.v[tl][j] - col_sum(x);
        const float u = sm.beta[tl] * e;
        if (keep && w == 0) {
            sm.e[tl][j] = e;
            sm.u[tl][j] = u;
        }
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            const float2 u2 = make_float2(__shfl_sync(0xffffffffu, u, 2 * p), __shfl_sync(0xffffffffu, u, 2 * p + 1));
            S[p] = __ffma2_rn(k2, u2, S[p]);
        }
    };
    // one backward step for token tl of the staged piece (token `pos` of the sequence);
    // row partials go to sm.rs / sm.bpart and are combined once per piece
    auto bwd_step = [&](int tl, int64_t pos) {
        const size_t r = (size_t)(t0 + pos) * P.H + h;
        float* stt = st + (size_t)tl * BLK;
#pragma unroll
        for (int p = 0; p < 16; ++p) S[p] = make_float2(*img(stt, 2 * p), *img(stt, 2 * p + 1));  // S_{t-1}
        const float ai = sm.a[tl][i], ki = sm.k[tl][i], qi = sm.q[tl][i];
        const float2 a2 = make_float2(ai, ai), k2 = make_float2(ki, ki), q2 = make_float2(qi, qi);
        const float2* dout2 = reinterpret_cast<const float2*>(&sm.dout[tl][32 * c]);
        const float2* u2s = reinterpret_cast<const float2*>(&sm.u[tl][32 * c]);
        float2 dq2 = make_float2(0.f, 0.f);
        float x[32];
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            const float2 do2 = dout2[p];
            dS[p] = __ffma2_rn(q2, do2, dS[p]);
            dq2 = __ffma2_rn(__ffma2_rn(k2, u2s[p], __fmul2_rn(a2, S[p])), do2, dq2);  // S_t do
            const float2 kx = __fmul2_rn(dS[p], k2);
            x[2 * p] = kx.x;
            x[2 * p + 1] = kx.y;
        }
        const float dq = dq2.x + dq2.y;
        const int j = 32 * c + lane;
        const float du = col_sum(x);
        const float b = sm.beta[tl];
        const float dp = -b * du;
        if (w == 0) {
            P.dv[r * kD + j] = b * du;
            float bp = du * sm.e[tl][j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) bp += __shfl_xor_sync(0xffffffffu, bp, o);
            if (lane == 0) sm.bpart[tl][c] = bp;
        }
        float2 dk2 = make_float2(0.f, 0.f), da2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            const float2 dp2 =
                make_float2(__shfl_sync(0xffffffffu, dp, 2 * p), __shfl_sync(0xffffffffu, dp, 2 * p + 1));
            dk2 = __ffma2_rn(dS[p], u2s[p], dk2);
            dk2 = __ffma2_rn(__fmul2_rn(a2, S[p]), dp2, dk2);
            const float2 dsp = __ffma2_rn(k2, dp2, dS[p]);
            da2 = __ffma2_rn(dsp, S[p], da2);
            dS[p] = __fmul2_rn(a2, dsp);
        }
        const float dk = dk2.x + dk2.y, da = da2.x + da2.y;
        sm.rs[tl][c][0][i] = dq;
        sm.rs[tl][c][1][i] = dk;
        sm.rs[tl][c][2][i] = ai * da;
    };
    // sums over the four column blocks, in a fixed order, for tokens [p0, p0 + n)
    auto combine = [&](int64_t p0, int n) {
        __syncthreads();
        for (int idx = tid; idx < n * 3 * kD; idx += NT) {
            const int tl = idx / (3 * kD), kind = (idx >> 7) % 3, row = idx & 127;
            const float val = ((sm.rs[tl][0][kind][row] + sm.rs[tl][1][kind][row]) + sm.rs[tl][2][kind][row]) +
                              sm.rs[tl][3][kind][row];
            const size_t o = ((size_t)(t0 + p0 + tl) * P.H + h) * kD + row;
            if (kind == 0)
                P.dq[o] = val;
            else if (kind == 1)
                P.dk[o] = val;
            else if (P.gate == kGateChannel)
                P.dlog_alpha[o] = val;
        }
        if (P.gate == kGateHead && (tid >> 5) < n) {  // warp tl: the head's gate gradient of token tl
            const int tl = tid >> 5;
            float hs = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int row = lane + 32 * m;
                hs += ((sm.rs[tl][0][2][row] + sm.rs[tl][1][2][row]) + sm.rs[tl][2][2][row]) + sm.rs[tl][3][2][row];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) hs += __shfl_xor_sync(0xffffffffu, hs, o);
            if (lane == 0) P.dlog_alpha[(size_t)(t0 + p0 + tl) * P.H + h] = hs;
        }
        if (tid < n)
            P.dbeta[(size_t)(t0 + p0 + tid) * P.H + h] =
                ((sm.bpart[tid][0] + sm.bpart[tid][1]) + sm.bpart[tid][2]) + sm.bpart[tid][3];
    };

    // forward sweep: checkpoints every SEG tokens
    for (int64_t t = 0; t < len; t += SUB) {
        const int n = (int)((len - t) < SUB ? (len - t) : SUB);
        if (t % SEG == 0) {
            float* ck = ckpt + (size_t)(slot0 + t / SEG) * BLK;
#pragma unroll
            for (int p = 0; p < 16; ++p) {
                *img(ck, 2 * p) = S[p].x;
                *img(ck, 2 * p + 1) = S[p].y;
            }
        }
        stage(t, n, false);
        for (int tl = 0; tl < n; ++tl) fwd_step(tl, nullptr);
    }

    // reverse sweep
#pragma unroll
    for (int p = 0; p < 16; ++p)
        dS[p] = P.dfinal ? *reinterpret_cast<const float2*>(P.dfinal + sbase + (size_t)i * kD + c * 32 + 2 * p)
                         : make_float2(0.f, 0.f);
    const int64_t nseg = (len + SEG - 1) / SEG;
    for (int64_t g = nseg - 1; g >= 0; --g) {
        const int64_t seg0 = g * SEG;
        const int seg_len = (int)((len - seg0) < SEG ? (len - seg0) : SEG);
        const int nsub = (seg_len + SUB - 1) / SUB;
        float* ck = ckpt + (size_t)(slot0 + g) * BLK;
#pragma unroll
        for (int p = 0; p < 16; ++p) S[p] = make_float2(*img(ck, 2 * p), *img(ck, 2 * p + 1));
        for (int m = 0; m < nsub; ++m) {  // S every SUB tokens of the segment
#pragma unroll
            for (int p = 0; p < 16; ++p) {
                *img(sub + (size_t)m * BLK, 2 * p) = S[p].x;
                *img(sub + (size_t)m * BLK, 2 * p + 1) = S[p].y;
            }
            if (m + 1 < nsub) {
                stage(seg0 + m * SUB, SUB, false);
                for (int tl = 0; tl < SUB; ++tl) fwd_step(tl, nullptr);
            }
        }
        for (int m = nsub - 1; m >= 0; --m) {
            const int64_t p0 = seg0 + m * SUB;
            const int n = (int)((seg0 + seg_len - p0) < SUB ? (seg0 + seg_len - p0) : SUB);
            float* sm_ = sub + (size_t)m * BLK;
#pragma unroll
            for (int p = 0; p < 16; ++p) S[p] = make_float2(*img(sm_, 2 * p), *img(sm_, 2 * p + 1));
            stage(p0, n, true);
            for (int tl = 0; tl < n; ++tl) fwd_step(tl, st + (size_t)tl * BLK);
            wg_sync(c);  // e, u of the piece (written by warp 0 of the block) before they are read
            for (int tl = n - 1; tl >= 0; --tl) bwd_step(tl, p0 + tl);
            combine(p0, n);
        }
    }
    if (P.dinit) {
#pragma unroll
        for (int p = 0; p < 16; ++p)
            *reinterpret_cast<float2*>(P.dinit + sbase + (size_t)i * kD + c * 32 + 2 * p) = dS[p];
    }
}

}  // namespace

size_t bwd_workspace(int N, int64_t T_total, int H) {
    const size_t slots = (size_t)(T_total / SEG) + (size_t)N + 1;
    return ((size_t)H * slots + (size_t)N * H * 2 * SUB) * BLK * sizeof(float);
}

cudaError_t launch_bwd(BwdProblem p, int in_dtype, void* workspace, cudaStream_t st) {
    const int64_t units = (int64_t)p.N * p.H;
    if (units == 0) return cudaSuccess;
    const size_t slots = (size_t)(p.T_total / SEG) + (size_t)p.N + 1;
    p.ckpt_slots = (int64_t)slots;
    p.ckpt = static_cast<float*>(workspace);
    p.scratch = p.ckpt + (size_t)p.H * slots * BLK;
    const int smem = (int)sizeof(Shared);
    auto kern = in_dtype == KDA_BF16 ? bwd_kernel<__nv_bfloat16> : bwd_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)units, NT, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
