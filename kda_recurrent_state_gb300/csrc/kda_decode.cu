// kda_decode.cu -- single-token KDA state update for B sessions, in place.
//
// "Kimi K3" article (lshu.cn/news/263999), §四, applied to one token:
//   S' = Diag(alpha) S                (alpha = exp(log_alpha), per key channel)
//   p  = S'^T k                       (§三: the memory's prediction for key k)
//   u  = beta (v - p)                 (§三: beta times the prediction error)
//   S  = S' + k u^T                   (= (I - beta k k^T) S' + beta k v^T)
//   o  = S^T q = S'^T q + (q . k) u   (§二.1: read after the update)
//
// Roofline: HBM.  Per (session, head) the 128 x 128 state is read once and
// written once; everything else is < 2 KB.
//
// fp32 state (131,072 bytes moved): one CTA of 256 threads owns one (session,
// head): thread (rg, cg) holds rows 16*rg .. 16*rg+15 and columns 4*cg ..
// 4*cg+3 as 16 float4 registers, so each warp moves whole 512-byte rows
// (coalesced, 128-bit accesses) and all 16 loads of a thread are in flight
// before the first use.  2 CTAs per SM (register-bound) keep 128 KB of state
// loads in flight per SM.
//
// bf16 state (65,536 bytes moved; kda_decode_step_bf16state): held in registers
// the same way it would keep only 64 KB in flight per SM, so instead one thread
// copies the CTA's 32 KB state into shared memory with a single bulk copy
// (completion on an mbarrier), and 5 CTAs per SM keep 160 KB in flight.  The
// entries are widened exactly to fp32, the step runs in fp32, the output is read
// from the unrounded new state, and the new state is stored rounded to nearest
// bf16.  The decay is folded into the per-row weights of the first pass
// (p = S^T (alpha*k), and S'^T q = S^T (alpha*q)), so S' is never formed there.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

__device__ __forceinline__ float ldin(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float ldin(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ void stout(__nv_bfloat16* p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }
__device__ __forceinline__ void stout(float* p, size_t i, float x) { p[i] = x; }
// alpha of key channel c: per channel (KDA), one per head (Gated DeltaNet) or 1 (DeltaNet).
__device__ __forceinline__ float gate_alpha(const DecodeProblem& p, int bh, int c) {
    if (p.gate == kGateChannel) return expf(p.log_alpha[(size_t)bh * kD + c]);
    if (p.gate == kGateHead) return expf(p.log_alpha[bh]);
    return 1.f;
}
// Four bf16 (two packed words) widened exactly to fp32.
__device__ __forceinline__ float4 widen_bf16x4(uint2 w) {
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xFFFF0000u));
}

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

    float4* S4 = reinterpret_cast<float4*>(static_cast<float*>(p.state) + (size_t)bh * kD * kD);
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
        s_a[tid] = gate_alpha(p, bh, tid);
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

// ---------------------------------------------------------------- bf16 state
constexpr int kBf16StateBytes = kD * kD * 2;  // one (session, head)
constexpr int kBf16Smem = kBf16StateBytes + 2 * 8 * kD * 4 + 6 * kD * 4;

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256, 5) decode_bf16state_kernel(DecodeProblem p) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ uint64_t bar;
    __shared__ sm100::Abort ab;
    __shared__ float s_qk[4];
    __shared__ float s_beta;
    const uint2* s_S = reinterpret_cast<const uint2*>(dsm);  // [128 rows][32 groups of 4 bf16]
    float(*s_redp)[kD] = reinterpret_cast<float(*)[kD]>(dsm + kBf16StateBytes);
    float(*s_redo)[kD] = reinterpret_cast<float(*)[kD]>(dsm + kBf16StateBytes + 8 * kD * 4);
    float* s_ak = reinterpret_cast<float*>(dsm + kBf16StateBytes + 16 * kD * 4);  // alpha * k
    float* s_aq = s_ak + kD;                                                      // alpha * q
    float* s_a = s_aq + kD;
    float* s_k = s_a + kD;
    float* s_v = s_k + kD;

    const int bh = blockIdx.x;
    const int tid = threadIdx.x;
    const int cg = tid & 31;  // columns 4cg..4cg+3
    const int rg = tid >> 5;  // rows 16rg..16rg+15
    __nv_bfloat16* S = static_cast<__nv_bfloat16*>(p.state) + (size_t)bh * kD * kD;

    if (tid == 0) {
        ab.flag = 0;
        sm100::mbar_init(&bar, 1);
        sm100::fence_proxy_async_smem();
        sm100::mbar_arrive_expect_tx(&bar, kBf16StateBytes);
        sm100::bulk_load(dsm, S, kBf16StateBytes, &bar);
    }
    const Tin* q = static_cast<const Tin*>(p.q) + (size_t)bh * kD;
    const Tin* k = static_cast<const Tin*>(p.k) + (size_t)bh * kD;
    const Tin* v = static_cast<const Tin*>(p.v) + (size_t)bh * kD;
    float qk = 0.f;
    if (tid < kD) {
        const float qq = ldin(q, tid), kk = ldin(k, tid), a = gate_alpha(p, bh, tid);
        s_k[tid] = kk;
        s_v[tid] = ldin(v, tid);
        s_a[tid] = a;
        s_ak[tid] = a * kk;
        s_aq[tid] = a * qq;
        qk = qq * kk;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, o);
        if ((tid & 31) == 0) s_qk[tid >> 5] = qk;
    }
    if (tid == 0) s_beta = p.beta[bh];
    __syncthreads();  // also publishes the mbarrier's initialisation
    if (!sm100::mbar_wait(&bar, 0, &ab, p.status)) return;  // timed out: status recorded

    float4 pp = make_float4(0.f, 0.f, 0.f, 0.f), oo = pp;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = rg * 16 + i;
        const float4 x = widen_bf16x4(s_S[r * 32 + cg]);
        const float ak = s_ak[r], aq = s_aq[r];
        pp.x += ak * x.x; pp.y += ak * x.y; pp.z += ak * x.z; pp.w += ak * x.w;
        oo.x += aq * x.x; oo.y += aq * x.y; oo.z += aq * x.z; oo.w += aq * x.w;
    }
    reinterpret_cast<float4*>(s_redp[rg])[cg] = pp;
    reinterpret_cast<float4*>(s_redo[rg])[cg] = oo;
    __syncthreads();

    qk = s_qk[0] + s_qk[1] + s_qk[2] + s_qk[3];
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
    uint2* S2 = reinterpret_cast<uint2*>(S);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = rg * 16 + i;
        float4 x = widen_bf16x4(s_S[r * 32 + cg]);
        const float a = s_a[r], kk = s_k[r];
        x.x = a * x.x + kk * u[0]; x.y = a * x.y + kk * u[1];
        x.z = a * x.z + kk * u[2]; x.w = a * x.w + kk * u[3];
        const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
        S2[r * 32 + cg] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
    if (rg == 0) {
        Tout* out = static_cast<Tout*>(p.out) + (size_t)bh * kD;
#pragma unroll
        for (int c = 0; c < 4; ++c) stout(out, 4 * cg + c, o[c]);
    }
}

template <typename Tin, typename Tout>
cudaError_t launch_bf16state(const DecodeProblem& p, unsigned grid, cudaStream_t st) {
    auto* fn = decode_bf16state_kernel<Tin, Tout>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kBf16Smem);
    if (e == cudaSuccess)  // shared memory over L1, so that 5 CTAs fit on an SM
        e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    fn<<<grid, 256, kBf16Smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeProblem& p, int in_dtype, int out_dtype, int state_dtype, cudaStream_t st) {
    const unsigned grid = (unsigned)((int64_t)p.B * p.H);
    if (grid == 0) return cudaSuccess;
    if (state_dtype == KDA_BF16) {
        if (in_dtype == KDA_BF16 && out_dtype == KDA_BF16)
            return launch_bf16state<__nv_bfloat16, __nv_bfloat16>(p, grid, st);
        if (in_dtype == KDA_BF16) return launch_bf16state<__nv_bfloat16, float>(p, grid, st);
        if (out_dtype == KDA_BF16) return launch_bf16state<float, __nv_bfloat16>(p, grid, st);
        return launch_bf16state<float, float>(p, grid, st);
    }
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
