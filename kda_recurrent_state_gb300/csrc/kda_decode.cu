// kda_decode.cu -- single-token KDA state update for B sessions, in place.
//
// "Kimi K3" article (lshu.cn/news/263999), §四, applied to one token:
//   S' = Diag(alpha) S                (alpha = exp(log_alpha), per key channel)
//   p  = S'^T k                       (§三: the memory's prediction for key k)
//   u  = beta (v - p)                 (§三: beta times the prediction error)
//   S  = S' + k u^T                   (= (I - beta k k^T) S' + beta k v^T)
//   o  = S^T q = S'^T q + (q . k) u   (§二.1: read after the update)
//
// Roofline: HBM.  Per (session, head) the 128 x 128 fp32 state is read once
// and written once (131,072 bytes); everything else is < 2 KB.  One CTA of
// 256 threads owns one (session, head): thread (rg, cg) holds rows
// 16*rg .. 16*rg+15 and columns 4*cg .. 4*cg+3 as 16 float4 registers, so
// each warp moves whole 512-byte rows (coalesced, 128-bit accesses) and all
// 16 loads of a thread are in flight before the first use.
#include "kda_internal.cuh"

namespace kda {
namespace {

__device__ __forceinline__ float ldin(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float ldin(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ void stout(__nv_bfloat16* p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }
__device__ __forceinline__ void stout(float* p, size_t i, float x) { p[i] = x; }

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) decode_kernel(DecodeProblem p) {
    const int bh = blockIdx.x;
    const int tid = threadIdx.x;
    const int cg = tid & 31;  // column group: columns 4cg..4cg+3
    const int rg = tid >> 5;  // row group: rows 16rg..16rg+15

    __shared__ float s_q[kD], s_k[kD], s_a[kD], s_v[kD];
    __shared__ float s_redp[8][kD], s_redo[8][kD];
    __shared__ float s_qk[4];
    __shared__ float s_beta;

    float4* S4 = reinterpret_cast<float4*>(p.state + (size_t)bh * kD * kD);
    float4 st[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) st[i] = S4[(rg * 16 + i) * (kD / 4) + cg];

    const Tin* q = static_cast<const Tin*>(p.q) + (size_t)bh * kD;
    const Tin* k = static_cast<const Tin*>(p.k) + (size_t)bh * kD;
    const Tin* v = static_cast<const Tin*>(p.v) + (size_t)bh * kD;
    if (tid < kD) {
        s_q[tid] = ldin(q, tid);
        s_k[tid] = ldin(k, tid);
        s_v[tid] = ldin(v, tid);
        s_a[tid] = expf(p.log_alpha[(size_t)bh * kD + tid]);
    }
    if (tid == 0) s_beta = p.beta[bh];
    __syncthreads();

    if (tid < kD) {  // q . k over the key channels
        float x = s_q[tid] * s_k[tid];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if ((tid & 31) == 0) s_qk[tid >> 5] = x;
    }

    float4 pp = make_float4(0.f, 0.f, 0.f, 0.f), oo = pp;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = rg * 16 + i;
        const float a = s_a[r], kk = s_k[r], qq = s_q[r];
        st[i].x *= a; st[i].y *= a; st[i].z *= a; st[i].w *= a;
        pp.x += kk * st[i].x; pp.y += kk * st[i].y; pp.z += kk * st[i].z; pp.w += kk * st[i].w;
        oo.x += qq * st[i].x; oo.y += qq * st[i].y; oo.z += qq * st[i].z; oo.w += qq * st[i].w;
    }
    reinterpret_cast<float4*>(s_redp[rg])[cg] = pp;
    reinterpret_cast<float4*>(s_redo[rg])[cg] = oo;
    __syncthreads();

    const float qk = s_qk[0] + s_qk[1] + s_qk[2] + s_qk[3];
    float u[4], o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int j = 4 * cg + c;
        float ps = 0.f, os = 0.f;
#pragma unroll
        for (int g = 0; g < 8; ++g) { ps += s_redp[g][j]; os += s_redo[g][j]; }
        u[c] = s_beta * (s_v[j] - ps);
        o[c] = os + qk * u[c];
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float kk = s_k[rg * 16 + i];
        st[i].x += kk * u[0]; st[i].y += kk * u[1]; st[i].z += kk * u[2]; st[i].w += kk * u[3];
        S4[(rg * 16 + i) * (kD / 4) + cg] = st[i];
    }
    if (rg == 0) {
        Tout* out = static_cast<Tout*>(p.out) + (size_t)bh * kD;
#pragma unroll
        for (int c = 0; c < 4; ++c) stout(out, 4 * cg + c, o[c]);
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeProblem& p, int in_dtype, int out_dtype, cudaStream_t st) {
    const unsigned grid = (unsigned)((int64_t)p.B * p.H);
    if (grid == 0) return cudaSuccess;
    if (in_dtype == KDA_BF16 && out_dtype == KDA_BF16)
        decode_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, st>>>(p);
    else if (in_dtype == KDA_BF16)
        decode_kernel<__nv_bfloat16, float><<<grid, 256, 0, st>>>(p);
    else if (out_dtype == KDA_BF16)
        decode_kernel<float, __nv_bfloat16><<<grid, 256, 0, st>>>(p);
    else
        decode_kernel<float, float><<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
