// kda_bwd_chunk.cu -- gradients of the KDA recurrence in chunked form (C = 64).
//
// The forward is the "Kimi K3" article's (lshu.cn/news/263999) §四 update with the §二.1 read,
// rewritten per chunk in the WY form of §六.2.  With the chunk's start state S_0, the in-chunk
// cumulative log-decay g_r (per key channel) and the reference ref = g_31:
//     Q~ = q e^{g-ref}   K~ = k e^{g-ref}   K^ = k e^{ref-g}      (row r of each)
//     T  = (I + strict_lower(diag(beta) K~ K^^T))^-1
//     U' = T diag(beta) V          W~ = T diag(beta) K~          P = lower_incl(Q~ K^^T)
//     X  = Diag(e^ref) S_0         U  = U' - W~ X
//     O  = Q~ X + P U              S_C = Diag(e^{g_C - ref}) (X + K^^T U)
// The pages give no backward; this is the reverse mode of those products, one at a time.  The
// output does not depend on ref, so its adjoint is zero and is not formed.  Four passes:
//   local   (chunk-parallel)  g, Q~, K~, K^, T, W~, U', P, and the chunk's output-gradient term
//                             E = Q~^T dO - W~^T (P^T dO) of the state gradient
//   states  (serial per head: tcgen05 products, or warp-level ones split over value columns when
//            the heads leave most SMs idle)
//                             S_{n+1} = Diag(e^{g_C-ref}) (X + K^^T (U' - W~ X)), every S_n and U kept
//   dstates (the same)        dS_n = Diag(e^ref) (dD - W~^T (K^ dD) + E), dD = Diag(e^{g_C-ref}) dS_{n+1}
//   grads   (chunk-parallel, two kernels) every input gradient of the chunk from S_n and dS_{n+1}
// Every product is a small dense GEMM computed on the tensor cores with each operand split into
// bf16 hi + lo (three products per tile, fp32 accumulation: about 2^-16 relative error per
// product, against the 2e-3 gradient bar), instead of the token-serial path's per-token reduction
// latency: warp-level MMAs over shared-memory tiles in the chunk-parallel passes, tcgen05 MMAs with
// TMEM accumulators in the serial ones.  Every element-wise
// step is fp32; sums are in a fixed order, so the result is bit-reproducible.  e^{g-ref} must stay in fp32
// range: a (sequence, head) with a chunk whose half-chunk log-decay sum is below -80 is flagged,
// and after these passes the token-serial backward (which has no such limit) recomputes exactly
// those units.
#include <type_traits>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

constexpr int C = 64;          // chunk
constexpr int NT = 512;        // 16 warps
// Row strides of the shared tiles: multiples of 4 floats (16-byte rows for 128-bit loads) and
// 8 more than a multiple of 32.  A tensor-core fragment reads a pair along k from each of 8 rows
// (rows g, lanes 4g..4g+3): at that stride the 4 rows of a half-warp cover the 32 banks once, and
// a transposed read (one float from each of 8 rows at 4 k) is conflict-free as well.
constexpr int LD = kD + 8;     // C x D and D x D tiles
constexpr int LC = C + 8;      // C x C tiles
constexpr int TILE_CD = C * LD;
constexpr int TILE_DD = kD * LD;
constexpr int TILE_CC = C * LC;
constexpr float kExpLimit = 80.f;  // |g - ref| beyond this leaves fp32 range in e^{+-(g-ref)}

// Per chunk-head workspace records (floats) and the state arrays.
constexpr size_t REC_CD = (size_t)C * kD, REC_DD = (size_t)kD * kD, REC_CC = (size_t)C * C;

struct CBwd {
    BwdProblem p;
    int* status;
    const int64_t* co;  // [N+1] first chunk index of each sequence
    int64_t* co_w;
    int* redo;          // [N * H]: 1 where a chunk of the unit left the fp32 range of e^{+-(g-ref)}
    // per chunk-head (index (cg * H + h)):
    float* Wt;  // W~ [C][D]; after the first gradient kernel: dW~
    float* Up;  // U' [C][D]; then U (states pass); then dU
    float* Kh;  // K^ [C][D]
    float* Ej;  // E [D][D]; then dQ~ (first half) and dK^ (second half), partial
    float* Tm;  // T [C][C]
    float* Pq;  // P [C][C]; then dP
    float* sc;  // [3][D]: e^ref, e^{g_C - ref}, and the final-decay gradient sum_j S_C dS_C
    float* dS;  // [D][D] gradient w.r.t. the chunk's end state
    float* S;   // per (sequence, n) for n = 0..chunks: S_n at slot (co[s] + s + n) * H + h
};

// Register fragment of an M x N product spread over the 16 warps, in the accumulator layout of
// the warp-level tensor-core product m16n8k16: warp w owns MT = M/64 tiles of 16 rows starting at
// row 16 MT (w % 4) and NTL = N/32 tiles of 8 columns starting at column 8 NTL (w / 4); lane
// (g, t) = (lane / 4, lane % 4) holds rows g and g + 8 and columns 2t and 2t + 1 of each tile.
// v[i][j] is row(i), col(j): the element-wise code addresses it through these alone.
template <int M, int N>
struct Frag {
    static constexpr int MT = M / 64, NTL = N / 32, MR = 2 * MT, NJ = 2 * NTL;
    static_assert(M % 64 == 0 && N % 32 == 0, "fragment shape");
    float v[MR][NJ];
    __device__ __forceinline__ static int row(int i) {
        return (int)((threadIdx.x >> 5) & 3) * MT * 16 + 16 * (i >> 1) + 8 * (i & 1) + (int)((threadIdx.x & 31) >> 2);
    }
    __device__ __forceinline__ static int col(int j) {
        return (int)(threadIdx.x >> 7) * NTL * 8 + 8 * (j >> 1) + 2 * (int)(threadIdx.x & 3) + (j & 1);
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < MR; ++i)
#pragma unroll
            for (int j = 0; j < NJ; ++j) v[i][j] = 0.f;
    }
};

// Two fp32 values as bf16 pairs hi + lo (x ~ hi + lo to 16 significant bits): hi rounded to
// nearest, lo the rounded remainder.  Lower k index in the low half, as the MMA fragments want.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
    lo = *reinterpret_cast<const uint32_t*>(&l);
}
// d (16x8 fp32) += a (16x16 bf16, row fragment) x b (16x8 bf16, column fragment)
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// f (+/-)= A B, A(m, k) = A[m * ARS + k * ACS], B(k, n) = B[k * BRS + n * BCS], k in [0, K).
// One of ARS, ACS is 1 (A is stored k-contiguous or m-contiguous) and one of BRS, BCS is 1.
// On the tensor cores with fp32-level accuracy from bf16 operands: every operand is split into
// bf16 hi + lo as its fragment is loaded, and each 16 x 8 x 16 tile takes the three products
// hi.hi + hi.lo + lo.hi (the dropped lo.lo term and the rounding of lo are below 2^-16 of the
// product), accumulated in fp32.  Pairs along k are loaded 8 bytes at a time where they are
// contiguous.
template <bool NEG, int K, int ARS, int ACS, int BRS, int BCS, int M, int N>
__device__ __forceinline__ void gemm(Frag<M, N>& f, const float* A, const float* B) {
    using F = Frag<M, N>;
    constexpr int MT = F::MT, NTL = F::NTL;
    constexpr bool A_KC = ACS == 1, B_KC = BRS == 1;
    static_assert((A_KC || ARS == 1) && (B_KC || BCS == 1) && K % 16 == 0, "layout");
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int mb = (int)((threadIdx.x >> 5) & 3) * MT * 16, nb = (int)(threadIdx.x >> 7) * NTL * 8;
    auto ldA = [&](int m, int k) -> float2 {
        if constexpr (A_KC) return *reinterpret_cast<const float2*>(A + m * ARS + k);
        else return make_float2(A[m + k * ACS], A[m + (k + 1) * ACS]);
    };
    auto ldB = [&](int k, int n) -> float2 {
        if constexpr (B_KC) return *reinterpret_cast<const float2*>(B + k + n * BCS);
        else return make_float2(B[k * BRS + n], B[(k + 1) * BRS + n]);
    };
#pragma unroll 2
    for (int k0 = 0; k0 < K; k0 += 16) {
        uint32_t ah[MT][4], al[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int r0 = mb + 16 * mt + g, ka = k0 + 2 * t;
            const float2 x0 = ldA(r0, ka), x1 = ldA(r0 + 8, ka), x2 = ldA(r0, ka + 8), x3 = ldA(r0 + 8, ka + 8);
            split_bf16(x0.x, x0.y, ah[mt][0], al[mt][0]);
            split_bf16(x1.x, x1.y, ah[mt][1], al[mt][1]);
            split_bf16(x2.x, x2.y, ah[mt][2], al[mt][2]);
            split_bf16(x3.x, x3.y, ah[mt][3], al[mt][3]);
            if (NEG) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    ah[mt][q] ^= 0x80008000u;
                    al[mt][q] ^= 0x80008000u;
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt) {
            const int cn = nb + 8 * nt + g, kk = k0 + 2 * t;
            const float2 y0 = ldB(kk, cn), y1 = ldB(kk + 8, cn);
            uint32_t bh[2], bl[2];
            split_bf16(y0.x, y0.y, bh[0], bl[0]);
            split_bf16(y1.x, y1.y, bh[1], bl[1]);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                float d[4] = {f.v[2 * mt][2 * nt], f.v[2 * mt][2 * nt + 1], f.v[2 * mt + 1][2 * nt],
                              f.v[2 * mt + 1][2 * nt + 1]};
                mma_bf16(d, ah[mt], bh);
                mma_bf16(d, ah[mt], bl);
                mma_bf16(d, al[mt], bh);
                f.v[2 * mt][2 * nt] = d[0];
                f.v[2 * mt][2 * nt + 1] = d[1];
                f.v[2 * mt + 1][2 * nt] = d[2];
                f.v[2 * mt + 1][2 * nt + 1] = d[3];
            }
        }
    }
}

template <int M, int N>
__device__ __forceinline__ void to_smem(const Frag<M, N>& f, float* dst, int ld) {
#pragma unroll
    for (int i = 0; i < Frag<M, N>::MR; ++i)
#pragma unroll
        for (int j = 0; j < Frag<M, N>::NJ; ++j) dst[Frag<M, N>::row(i) * ld + Frag<M, N>::col(j)] = f.v[i][j];
}
// Global copies of a fragment: row r of the block at dst + r * ld (a column slice when ld > N).
// Columns col(2i) and col(2i + 1) are adjacent (and the first is even), so they move as one 8-byte
// access (ld and the base offset are even).
template <int M, int N>
__device__ __forceinline__ void to_global(const Frag<M, N>& f, float* dst, int ld = N) {
#pragma unroll
    for (int i = 0; i < Frag<M, N>::MR; ++i)
#pragma unroll
        for (int j = 0; j < Frag<M, N>::NJ; j += 2)
            *reinterpret_cast<float2*>(dst + (size_t)Frag<M, N>::row(i) * ld + Frag<M, N>::col(j)) =
                make_float2(f.v[i][j], f.v[i][j + 1]);
}
template <int M, int N>
__device__ __forceinline__ void from_global(Frag<M, N>& f, const float* src, int ld = N) {
#pragma unroll
    for (int i = 0; i < Frag<M, N>::MR; ++i)
#pragma unroll
        for (int j = 0; j < Frag<M, N>::NJ; j += 2) {
            const float2 x = *reinterpret_cast<const float2*>(src + (size_t)Frag<M, N>::row(i) * ld + Frag<M, N>::col(j));
            f.v[i][j] = x.x;
            f.v[i][j + 1] = x.y;
        }
}

// Dense [ROWS][D] record in global memory -> shared tile with row stride LD, optionally scaled per
// row.  Every thread issues all of its 16-byte loads before it stores any.
template <int ROWS>
__device__ __forceinline__ void load_tile(float* dst, const float* src, const float* row_scale = nullptr) {
    constexpr int PER = ROWS * (kD / 4) / NT;  // float4 per thread
    float4 x[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) x[i] = reinterpret_cast<const float4*>(src)[threadIdx.x + i * NT];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int g = threadIdx.x + i * NT, r = g >> 5, c4 = (g & 31) * 4;
        float4 v = x[i];
        if (row_scale) {
            const float sc = row_scale[r];
            v.x *= sc; v.y *= sc; v.z *= sc; v.w *= sc;
        }
        *reinterpret_cast<float4*>(dst + r * LD + c4) = v;
    }
}

// Asynchronous 16-byte global -> shared copies (cp.async), committed and awaited in groups.
__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
// A vector of 2 D scales.
__device__ __forceinline__ void scales_async(float* dst, const float* src) {
    if (threadIdx.x < 2 * kD / 4) cp_async16(dst + 4 * threadIdx.x, src + 4 * threadIdx.x);
}

// Four consecutive elements as fp32 (bf16 widens exactly: it is the high half of an fp32).
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ float4 scale4(float4 v, float s) { return make_float4(v.x * s, v.y * s, v.z * s, v.w * s); }

// ---- operands stored pre-split: a tile held as two bf16 arrays hi and lo (x ~ hi + lo, split as
// by split_bf16) with row stride RS elements, so that the fragments of every product are read with
// ldmatrix and no warp splits an element again.  RS = width + 8: the 8 rows of an ldmatrix read
// start 16 bytes apart modulo 128, so a read is free of bank conflicts.
constexpr int RSD = kD + 8;  // rows of D elements
constexpr int RSC = C + 8;   // rows of C elements
struct Split {
    __nv_bfloat16* hi;
    __nv_bfloat16* lo;
};
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t a) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a) : "memory");
}
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], uint32_t a) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a) : "memory");
}
__device__ __forceinline__ void ldsm2(uint32_t (&r)[4], uint32_t a) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(a) : "memory");
}
__device__ __forceinline__ void ldsm2t(uint32_t (&r)[4], uint32_t a) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(a)
                 : "memory");
}
// Four consecutive elements of a row into the split tile (8-byte stores of hi and of lo).
__device__ __forceinline__ void split_store4(const Split& t, int off, float4 v) {
    uint2 h, l;
    split_bf16(v.x, v.y, h.x, l.x);
    split_bf16(v.z, v.w, h.y, l.y);
    *reinterpret_cast<uint2*>(t.hi + off) = h;
    *reinterpret_cast<uint2*>(t.lo + off) = l;
}
// Dense [ROWS][D] record in global memory -> split tile, optionally scaled per row.  Every thread
// issues all of its 16-byte loads before it stores any.
template <int ROWS>
__device__ __forceinline__ void load_tile_split(const Split& dst, const float* src, const float* row_scale = nullptr) {
    constexpr int PER = ROWS * (kD / 4) / NT;
    float4 x[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) x[i] = reinterpret_cast<const float4*>(src)[threadIdx.x + i * NT];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int g = threadIdx.x + i * NT, r = g >> 5, c4 = (g & 31) * 4;
        split_store4(dst, r * RSD + c4, row_scale ? scale4(x[i], row_scale[r]) : x[i]);
    }
}
__device__ __forceinline__ void load_cc_split(const Split& dst, const float* src) {
    constexpr int PER = C * C / 4 / NT;
    float4 x[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) x[i] = reinterpret_cast<const float4*>(src)[threadIdx.x + i * NT];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int g = threadIdx.x + i * NT;
        split_store4(dst, (g >> 4) * RSC + (g & 15) * 4, x[i]);
    }
}
// Split records in the workspace: a [C][D] record held as its bf16 hi array followed by its lo
// array (the bytes of one fp32 record).  Copied into a split tile of row stride RSD with cp.async.
__device__ __forceinline__ Split record_split(float* rec) {
    __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(rec);
    return Split{b, b + C * kD};
}
__device__ __forceinline__ void cp_async16b(void* dst, const void* src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void tile_async_split(const Split& dst, const float* rec) {
    const __nv_bfloat16* hi = reinterpret_cast<const __nv_bfloat16*>(rec);
    const __nv_bfloat16* lo = hi + C * kD;
#pragma unroll
    for (int i = 0; i < C * kD / 8 / NT; ++i) {  // 16-byte pieces (8 elements) of each array
        const int g = threadIdx.x + i * NT, r = g >> 4, c8 = (g & 15) * 8;
        cp_async16b(dst.hi + r * RSD + c8, hi + g * 8);
        cp_async16b(dst.lo + r * RSD + c8, lo + g * 8);
    }
}
// A split record into a split tile with plain loads (all of a thread's loads issued first).
__device__ __forceinline__ void load_record_split(const Split& dst, const float* rec) {
    const uint4* hi = reinterpret_cast<const uint4*>(rec);
    const uint4* lo = hi + C * kD / 8;
    constexpr int PER = C * kD / 8 / NT;
    uint4 xh[PER], xl[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        xh[i] = hi[threadIdx.x + i * NT];
        xl[i] = lo[threadIdx.x + i * NT];
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int g = threadIdx.x + i * NT, r = g >> 4, c8 = (g & 15) * 8;
        *reinterpret_cast<uint4*>(dst.hi + r * RSD + c8) = xh[i];
        *reinterpret_cast<uint4*>(dst.lo + r * RSD + c8) = xl[i];
    }
}
// A [C][D] fragment into a split record in global memory.
template <int M, int N>
__device__ __forceinline__ void to_global_split(const Frag<M, N>& f, float* rec) {
    const Split t = record_split(rec);
#pragma unroll
    for (int i = 0; i < Frag<M, N>::MR; ++i)
#pragma unroll
        for (int j = 0; j < Frag<M, N>::NJ; j += 2) {
            uint32_t h, l;
            split_bf16(f.v[i][j], f.v[i][j + 1], h, l);
            const int off = Frag<M, N>::row(i) * N + Frag<M, N>::col(j);
            *reinterpret_cast<uint32_t*>(t.hi + off) = h;
            *reinterpret_cast<uint32_t*>(t.lo + off) = l;
        }
}
// A fragment into a split tile: adjacent column pairs (col(2i), col(2i+1)) as bf16x2 stores.
template <int M, int N>
__device__ __forceinline__ void to_smem_split(const Frag<M, N>& f, const Split& t, int rs) {
#pragma unroll
    for (int i = 0; i < Frag<M, N>::MR; ++i)
#pragma unroll
        for (int j = 0; j < Frag<M, N>::NJ; j += 2) {
            uint32_t h, l;
            split_bf16(f.v[i][j], f.v[i][j + 1], h, l);
            const int off = Frag<M, N>::row(i) * rs + Frag<M, N>::col(j);
            *reinterpret_cast<uint32_t*>(t.hi + off) = h;
            *reinterpret_cast<uint32_t*>(t.lo + off) = l;
        }
}
// Product operands: a tile stored pre-split (Split) or in fp32 (split as its fragments are loaded),
// each with its row stride in elements.
struct OpS {
    Split t;
    int rs;
};
struct OpF {
    const float* p;
    int rs;
};
// f (+/-)= A B with each operand pre-split or fp32, the same three products per tile in the same
// order as gemm() (so the same result bit for bit).  A_KC: A stored [m][k] (else [k][m]); B_KC:
// B stored [n][k] (else [k][n]).
template <bool NEG, int K, bool A_KC, bool B_KC, int M, int N, class AO, class BO>
__device__ __forceinline__ void gemm_mx(Frag<M, N>& f, const AO& A, const BO& B) {
    using F = Frag<M, N>;
    constexpr int MT = F::MT, NTL = F::NTL;
    constexpr bool AS = std::is_same<AO, OpS>::value, BS = std::is_same<BO, OpS>::value;
    static_assert(K % 16 == 0 && (NTL == 1 || NTL % 2 == 0), "layout");
    constexpr int NP = NTL == 1 ? 1 : NTL / 2, NH = NTL == 1 ? 1 : 2;  // n-tile pairs, tiles per pair
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int mb = (int)((threadIdx.x >> 5) & 3) * MT * 16, nb = (int)(threadIdx.x >> 7) * NTL * 8;
    const int l7 = lane & 7, l8 = (lane >> 3) & 1, l16 = lane >> 4;
#pragma unroll 2
    for (int k0 = 0; k0 < K; k0 += 16) {
        uint32_t fa[MT][4], fl[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int m0 = mb + 16 * mt;
            if constexpr (AS) {  // matrices (m 0-7|8-15) x (k 0-7|8-15), m-minor first
                const int ras = A.rs;
                const uint32_t o = A_KC ? (uint32_t)(((m0 + l7 + 8 * l8) * ras + k0 + 8 * l16) * 2)
                                        : (uint32_t)(((k0 + l7 + 8 * l16) * ras + m0 + 8 * l8) * 2);
                if (A_KC) {
                    ldsm4(fa[mt], smem_addr(A.t.hi) + o);
                    ldsm4(fl[mt], smem_addr(A.t.lo) + o);
                } else {
                    ldsm4t(fa[mt], smem_addr(A.t.hi) + o);
                    ldsm4t(fl[mt], smem_addr(A.t.lo) + o);
                }
            } else {
                auto ldA = [&](int m, int k) -> float2 {
                    if constexpr (A_KC) return *reinterpret_cast<const float2*>(A.p + m * A.rs + k);
                    else return make_float2(A.p[m + k * A.rs], A.p[m + (k + 1) * A.rs]);
                };
                const int r0 = m0 + g, ka = k0 + 2 * t;
                const float2 x0 = ldA(r0, ka), x1 = ldA(r0 + 8, ka), x2 = ldA(r0, ka + 8), x3 = ldA(r0 + 8, ka + 8);
                split_bf16(x0.x, x0.y, fa[mt][0], fl[mt][0]);
                split_bf16(x1.x, x1.y, fa[mt][1], fl[mt][1]);
                split_bf16(x2.x, x2.y, fa[mt][2], fl[mt][2]);
                split_bf16(x3.x, x3.y, fa[mt][3], fl[mt][3]);
            }
            if (NEG) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    fa[mt][q] ^= 0x80008000u;
                    fl[mt][q] ^= 0x80008000u;
                }
            }
        }
#pragma unroll
        for (int np = 0; np < NP; ++np) {
            uint32_t gh[4], gl[4];  // (b0, b1) of n-tiles 2 np and 2 np + 1
            if constexpr (BS) {  // matrices (k 0-7, n0), (k 8-15, n0), (k 0-7, n0+8), (k 8-15, n0+8)
                const int n0 = nb + 16 * np, rbs = B.rs;
                const uint32_t o = B_KC ? (uint32_t)(((n0 + l7 + 8 * l16) * rbs + k0 + 8 * l8) * 2)
                                        : (uint32_t)(((k0 + l7 + 8 * l8) * rbs + n0 + 8 * l16) * 2);
                if constexpr (NTL == 1) {  // one n-tile: the first two matrices (lanes 0-15 address them)
                    if (B_KC) {
                        ldsm2(gh, smem_addr(B.t.hi) + o);
                        ldsm2(gl, smem_addr(B.t.lo) + o);
                    } else {
                        ldsm2t(gh, smem_addr(B.t.hi) + o);
                        ldsm2t(gl, smem_addr(B.t.lo) + o);
                    }
                } else if (B_KC) {
                    ldsm4(gh, smem_addr(B.t.hi) + o);
                    ldsm4(gl, smem_addr(B.t.lo) + o);
                } else {
                    ldsm4t(gh, smem_addr(B.t.hi) + o);
                    ldsm4t(gl, smem_addr(B.t.lo) + o);
                }
            } else {
                auto ldB = [&](int k, int n) -> float2 {
                    if constexpr (B_KC) return *reinterpret_cast<const float2*>(B.p + k + n * B.rs);
                    else return make_float2(B.p[k * B.rs + n], B.p[(k + 1) * B.rs + n]);
                };
#pragma unroll
                for (int h2 = 0; h2 < NH; ++h2) {
                    const int cn = nb + 8 * (2 * np + h2) + g, kk = k0 + 2 * t;
                    const float2 y0 = ldB(kk, cn), y1 = ldB(kk + 8, cn);
                    split_bf16(y0.x, y0.y, gh[2 * h2], gl[2 * h2]);
                    split_bf16(y1.x, y1.y, gh[2 * h2 + 1], gl[2 * h2 + 1]);
                }
            }
#pragma unroll
            for (int h2 = 0; h2 < NH; ++h2) {
                const int nt = 2 * np + h2;
                const uint32_t bhi[2] = {gh[2 * h2], gh[2 * h2 + 1]}, blo[2] = {gl[2 * h2], gl[2 * h2 + 1]};
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    float d[4] = {f.v[2 * mt][2 * nt], f.v[2 * mt][2 * nt + 1], f.v[2 * mt + 1][2 * nt],
                                  f.v[2 * mt + 1][2 * nt + 1]};
                    mma_bf16(d, fa[mt], bhi);
                    mma_bf16(d, fa[mt], blo);
                    mma_bf16(d, fl[mt], bhi);
                    f.v[2 * mt][2 * nt] = d[0];
                    f.v[2 * mt][2 * nt + 1] = d[1];
                    f.v[2 * mt + 1][2 * nt] = d[2];
                    f.v[2 * mt + 1][2 * nt + 1] = d[3];
                }
            }
        }
    }
}
template <bool NEG, int K, bool A_KC, bool B_KC, int M, int N>
__device__ __forceinline__ void gemm_ps(Frag<M, N>& f, const Split& A, int ras, const Split& B, int rbs) {
    gemm_mx<NEG, K, A_KC, B_KC>(f, OpS{A, ras}, OpS{B, rbs});
}

__device__ __forceinline__ void seq_of(const BwdProblem& P, int s, int64_t& start, int64_t& len) {
    if (P.cu_seqlens) {
        start = P.cu_seqlens[s];
        len = P.cu_seqlens[s + 1] - start;
    } else {
        start = (int64_t)s * P.T_uniform;
        len = P.T_uniform;
    }
}

struct ChunkAt {
    int s;
    int64_t n, tok0;
    int L;  // valid rows
};

// The chunk's rows of a token-major [.., H, D] tensor at head h, in groups of 4 elements (rows >= L:
// zero).  Group i of thread t is row (t + i NT) / 32, columns 4 ((t + i NT) % 32) .. +3.
template <typename Tin>
__device__ __forceinline__ void load_rows(float4 (&x)[4], const Tin* src, const ChunkAt& c, int H, int h) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int g = threadIdx.x + i * NT, r = g >> 5, c4 = (g & 31) * 4;
        x[i] = r < c.L ? ld4(src + ((size_t)(c.tok0 + r) * H + h) * kD + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// The chunk with global index cg: the last sequence s with co[s] <= cg (empty sequences own no chunk).
__device__ __forceinline__ bool locate_chunk(const CBwd& W, int64_t cg, ChunkAt& c) {
    const int N = W.p.N;
    if (cg >= W.co[N]) return false;
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (W.co[mid] <= cg) lo = mid; else hi = mid - 1;
    }
    int64_t start, len;
    seq_of(W.p, lo, start, len);
    c.s = lo;
    c.n = cg - W.co[lo];
    c.tok0 = start + c.n * C;
    const int64_t rem = len - c.n * C;
    c.L = rem < C ? (int)rem : C;
    return true;
}

__global__ void chunk_offsets_kernel(CBwd W) {
    __shared__ int64_t part[1024];
    const int N = W.p.N, t = threadIdx.x;
    const int per = (N + 1023) / 1024;
    const int s0 = min(N, t * per), s1 = min(N, s0 + per);
    auto nch = [&](int s) {
        int64_t start, len;
        seq_of(W.p, s, start, len);
        return (len + C - 1) / C;
    };
    int64_t sum = 0;
    for (int s = s0; s < s1; ++s) sum += nch(s);
    part[t] = sum;
    __syncthreads();
    if (t == 0) {
        int64_t run = 0;
        for (int i = 0; i < 1024; ++i) {
            const int64_t x = part[i];
            part[i] = run;
            run += x;
        }
        W.co_w[N] = run;
    }
    __syncthreads();
    int64_t run = part[t];
    for (int s = s0; s < s1; ++s) {
        W.co_w[s] = run;
        run += nch(s);
    }
    for (int64_t u = t; u < (int64_t)N * W.p.H; u += 1024) W.redo[u] = 0;
}

// Cumulative log-decay of the chunk into g (rows >= L: no decay), and beta (rows >= L: 0).  Thread t
// scans rows 16 sg .. 16 sg + 15 of channel ch (sg = t / 128, ch = t % 128) in registers; each
// segment is then offset by the totals of the segments before it (`tot`: 4 x D scratch).
__device__ __forceinline__ void load_gates(const CBwd& W, const ChunkAt& c, int h, float* g, float* beta, float* tot) {
    const BwdProblem& P = W.p;
    const int ch = threadIdx.x & 127, sg = threadIdx.x >> 7;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = sg * 16 + i;
        float la = 0.f;
        if (r < c.L) {
            const size_t row = (size_t)(c.tok0 + r) * P.H + h;
            la = P.gate == kGateChannel ? P.log_alpha[row * kD + ch] : P.gate == kGateHead ? P.log_alpha[row] : 0.f;
        }
        x[i] = la;
    }
#pragma unroll
    for (int i = 1; i < 16; ++i) x[i] += x[i - 1];
    tot[sg * kD + ch] = x[15];
    if (beta && threadIdx.x < C)
        beta[threadIdx.x] = (int)threadIdx.x < c.L ? P.beta[(size_t)(c.tok0 + threadIdx.x) * P.H + h] : 0.f;
    __syncthreads();
    float off = 0.f;
    for (int k = 0; k < sg; ++k) off += tot[k * kD + ch];
#pragma unroll
    for (int i = 0; i < 16; ++i) g[(sg * 16 + i) * LD + ch] = x[i] + off;
    __syncthreads();
}

// Q~, K~, K^ of the chunk from q, k and the cumulative decay g (rows >= L: zero).  SPLIT: Q~ and
// K^ are stored pre-split (sQ and sH then hold Split tiles of row stride RSD).
template <typename Tin, bool SPLIT = false>
__device__ __forceinline__ void scaled_qk(const CBwd& W, const ChunkAt& c, int h, const float* g, float* sQ,
                                          float* sK, float* sH, float* Kh_out) {
    float4 q4[4], k4[4];
    load_rows(q4, static_cast<const Tin*>(W.p.q), c, W.p.H, h);
    load_rows(k4, static_cast<const Tin*>(W.p.k), c, W.p.H, h);
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int gi = threadIdx.x + i * NT, r = gi >> 5, c4 = (gi & 31) * 4;
        const float4 gr = *reinterpret_cast<const float4*>(g + r * LD + c4);
        const float4 g31 = *reinterpret_cast<const float4*>(g + 31 * LD + c4);
        const float x[4] = {gr.x - g31.x, gr.y - g31.y, gr.z - g31.z, gr.w - g31.w};
        const float qa[4] = {q4[i].x, q4[i].y, q4[i].z, q4[i].w}, ka[4] = {k4[i].x, k4[i].y, k4[i].z, k4[i].w};
        float qo[4], ko[4], ho[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            bad |= fabsf(x[e]) > kExpLimit;
            const float ee = expf(x[e]), ff = expf(-x[e]);
            qo[e] = qa[e] * ee;
            ko[e] = ka[e] * ee;
            ho[e] = ka[e] * ff;
        }
        const float4 qv = make_float4(qo[0], qo[1], qo[2], qo[3]), hv = make_float4(ho[0], ho[1], ho[2], ho[3]);
        *reinterpret_cast<float4*>(sK + r * LD + c4) = make_float4(ko[0], ko[1], ko[2], ko[3]);
        if constexpr (SPLIT) {
            __nv_bfloat16* q16 = reinterpret_cast<__nv_bfloat16*>(sQ);
            __nv_bfloat16* h16 = reinterpret_cast<__nv_bfloat16*>(sH);
            split_store4(Split{q16, q16 + C * RSD}, r * RSD + c4, qv);
            split_store4(Split{h16, h16 + C * RSD}, r * RSD + c4, hv);
        } else {
            *reinterpret_cast<float4*>(sQ + r * LD + c4) = qv;
            *reinterpret_cast<float4*>(sH + r * LD + c4) = hv;
        }
        if (Kh_out) split_store4(record_split(Kh_out), r * kD + c4, hv);  // the K^ record, pre-split
    }
    if (bad) W.redo[(size_t)c.s * W.p.H + h] = 1;
}

// In place: the strictly lower C x C matrix A (stride LC) becomes T = (I + A)^-1, by 16 x 16 blocks:
// diagonal blocks by substitution, then T_ab = -Dg_a sum_{k=b}^{a-1} A_ak T_kb block row by block row.
// `y` is scratch for 3 blocks.
__device__ void invert_unit_lower(float* A, float* y) {
    const int t = threadIdx.x;
    float x[16];
    if (t < 64) {  // column j of diagonal block a
        const int a = t >> 4, j = t & 15;
        const float* Ab = A + (a * 16) * LC + a * 16;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float s = r == j ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < r; ++i) s = fmaf(-Ab[r * LC + i], x[i], s);
            x[r] = s;
        }
    }
    __syncthreads();
    if (t < 64) {
        const int a = t >> 4, j = t & 15;
        float* Ab = A + (a * 16) * LC + a * 16;
#pragma unroll
        for (int r = 0; r < 16; ++r) Ab[r * LC + j] = x[r];
    }
    __syncthreads();
    for (int a = 1; a < 4; ++a) {
        for (int idx = t; idx < a * 256; idx += NT) {  // Y_ab = sum_{k=b}^{a-1} A_ak T_kb
            const int b = idx >> 8, r = (idx >> 4) & 15, cc = idx & 15;
            float s = 0.f;
            for (int k = b; k < a; ++k) {
                const float* Ar = A + (a * 16 + r) * LC + k * 16;
                const float* Tk = A + (k * 16) * LC + b * 16 + cc;
#pragma unroll
                for (int m = 0; m < 16; ++m) s = fmaf(Ar[m], Tk[m * LC], s);
            }
            y[idx] = s;
        }
        __syncthreads();
        for (int idx = t; idx < a * 256; idx += NT) {  // T_ab = -Dg_a Y_ab
            const int b = idx >> 8, r = (idx >> 4) & 15, cc = idx & 15;
            const float* Dr = A + (a * 16 + r) * LC + a * 16;
            const float* Yb = y + b * 256 + cc;
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) s = fmaf(Dr[m], Yb[m * 16], s);
            A[(a * 16 + r) * LC + b * 16 + cc] = -s;
        }
        __syncthreads();
    }
}

// ---- pass 1: the chunk's local terms ------------------------------------------------------
constexpr int SMEM_LOCAL = (5 * TILE_CD + 2 * TILE_CC + 3 * 256 + C) * 4;

template <typename Tin>
__global__ void __launch_bounds__(NT, 1) cbwd_local(CBwd W) {
    extern __shared__ __align__(16) float sm[];
    float* sA = sm;              // g, then beta V, then W~ (both pre-split)
    float* sQ = sA + TILE_CD;    // Q~ (pre-split)
    float* sK = sQ + TILE_CD;    // K~, then beta K~, then P^T dO (pre-split)
    float* sH = sK + TILE_CD;    // K^ (pre-split)
    float* sO = sH + TILE_CD;    // dO (pre-split)
    float* sP = sO + TILE_CD;    // P (pre-split)
    float* sT = sP + TILE_CC;    // strict_lower(beta K~ K^^T), then T
    float* sY = sT + TILE_CC;    // inverse scratch
    float* sB = sY + 3 * 256;    // beta
    auto split_of = [](float* t, int rows, int rs) {
        __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(t);
        return Split{b, b + (size_t)rows * rs};
    };
    const Split xA = split_of(sA, C, RSD), xQ = split_of(sQ, C, RSD), xK = split_of(sK, C, RSD),
                xH = split_of(sH, C, RSD), xO = split_of(sO, C, RSD), xP = split_of(sP, C, RSC);
    const BwdProblem& P = W.p;
    const int h = blockIdx.x % P.H;
    const int64_t cg = blockIdx.x / P.H;
    ChunkAt c;
    if (!locate_chunk(W, cg, c)) return;
    const size_t ch = (size_t)cg * P.H + h;

    load_gates(W, c, h, sA, sB, sY);
    scaled_qk<Tin, true>(W, c, h, sA, sQ, sK, sH, W.Kh + ch * REC_CD);
    if (threadIdx.x < kD) {
        const float ref = sA[31 * LD + threadIdx.x];
        W.sc[ch * 3 * kD + threadIdx.x] = expf(ref);
        W.sc[ch * 3 * kD + kD + threadIdx.x] = expf(sA[63 * LD + threadIdx.x] - ref);
    }
    __syncthreads();
    {
        float4 v4[4], o4[4];
        load_rows(v4, static_cast<const Tin*>(P.v), c, P.H, h);
        load_rows(o4, P.dout, c, P.H, h);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gi = threadIdx.x + i * NT, r = gi >> 5, c4 = (gi & 31) * 4;
            split_store4(xA, r * RSD + c4, scale4(v4[i], sB[r]));
            split_store4(xO, r * RSD + c4, o4[i]);
        }
    }
    {
        Frag<C, C> gk, pq;
        gk.zero();
        pq.zero();
        gemm_mx<false, kD, true, true>(gk, OpF{sK, LD}, OpS{xH, RSD});  // K~ K^^T
        gemm_ps<false, kD, true, true>(pq, xQ, RSD, xH, RSD);          // Q~ K^^T
#pragma unroll
        for (int i = 0; i < Frag<C, C>::MR; ++i)
#pragma unroll
            for (int j = 0; j < Frag<C, C>::NJ; ++j) {
                const int r = Frag<C, C>::row(i), cc = Frag<C, C>::col(j);
                sT[r * LC + cc] = cc < r ? sB[r] * gk.v[i][j] : 0.f;
                if (cc > r) pq.v[i][j] = 0.f;
            }
        to_smem_split(pq, xP, RSC);
        to_global(pq, W.Pq + ch * REC_CC);
    }
    __syncthreads();
    invert_unit_lower(sT, sY);
    for (int idx = threadIdx.x; idx < C * C; idx += NT) W.Tm[ch * REC_CC + idx] = sT[(idx >> 6) * LC + (idx & 63)];
    {
        Frag<C, kD> u;
        u.zero();
        gemm_mx<false, C, true, false>(u, OpF{sT, LC}, OpS{xA, RSD});  // U' = T (beta V)
        to_global(u, W.Up + ch * REC_CD);
    }
    for (int idx = threadIdx.x; idx < C * kD; idx += NT) sK[(idx >> 7) * LD + (idx & 127)] *= sB[idx >> 7];
    __syncthreads();
    {
        Frag<C, kD> w;
        w.zero();
        gemm<false, C, LC, 1, LD, 1>(w, sT, sK);  // W~ = T (beta K~)
        to_smem_split(w, xA, RSD);
        to_global_split(w, W.Wt + ch * REC_CD);  // the W~ record, pre-split
    }
    __syncthreads();
    {
        Frag<C, kD> pd;
        pd.zero();
        gemm_ps<false, C, false, false>(pd, xP, RSC, xO, RSD);  // P^T dO
        to_smem_split(pd, xK, RSD);
    }
    __syncthreads();
    {
        Frag<kD, kD> e;
        e.zero();
        gemm_ps<false, C, false, false>(e, xQ, RSD, xO, RSD);  // Q~^T dO
        gemm_ps<true, C, false, false>(e, xA, RSD, xK, RSD);   // - W~^T (P^T dO)
        to_global(e, W.Ej + ch * REC_DD);
    }
}

// ---- passes 2 and 3: the serial recurrences, warp-level form ------------------------------------
// Used when the (sequence, head) units would leave most SMs idle (otherwise the tcgen05 form below
// runs).  Value columns are independent in both recurrences, so a unit is split over kD / NCOL
// CTAs, each carrying NCOL columns of the state (or its gradient).  Every output element sums over
// k in the same order at every NCOL, so the split changes no bit of the result.
// Every tile of these passes is a product operand only, stored pre-split: the state (or its
// gradient) slice and U (or K^ dD) with row stride NCOL + 8, W~ and K^ copied from their split
// records (row stride RSD).
template <int NCOL>
constexpr int smem_serial() {
    return (kD * (NCOL + 8) + C * (NCOL + 8) + 2 * C * RSD) * 4 + 4 * kD * 4;
}

// Pass 2: chunk-start states.  W~ and the scales of chunk n+1 are copied in while K^^T U of
// chunk n runs, and K^ of chunk n+1 while the next chunk's W~ X runs (cp.async groups; the
// scales are double-buffered).
template <int NCOL>
__global__ void __launch_bounds__(NT, 1) cbwd_states(CBwd W) {
    constexpr int RS = NCOL + 8;  // row stride of the column-slice tiles (elements)
    extern __shared__ __align__(16) float sm[];
    __nv_bfloat16* b16 = reinterpret_cast<__nv_bfloat16*>(sm);
    const Split xX{b16, b16 + kD * RS};                        // X = Diag(e^ref) S, this CTA's columns
    const Split xU{xX.lo + kD * RS, xX.lo + kD * RS + C * RS};  // U, this CTA's columns
    const Split xW{xU.lo + C * RS, xU.lo + C * RS + C * RSD};  // W~
    const Split xH{xW.lo + C * RSD, xW.lo + 2 * C * RSD};      // K^
    float* sE = reinterpret_cast<float*>(xH.lo + C * RSD);     // [2][e^ref, e^{g_C - ref}]
    const BwdProblem& P = W.p;
    constexpr int PARTS = kD / NCOL;
    const int unit = blockIdx.x / PARTS, c0 = (blockIdx.x % PARTS) * NCOL;
    const int h = unit % P.H, s = unit / P.H;
    int64_t start, len;
    seq_of(P, s, start, len);
    const int64_t nc = (len + C - 1) / C, base = W.co[s];
    using F = Frag<kD, NCOL>;
    F S;
    if (P.init) from_global(S, P.init + ((size_t)s * P.H + h) * REC_DD + c0, kD);
    else S.zero();
    if (nc > 0) {
        const size_t ch0 = (size_t)base * P.H + h;
        tile_async_split(xW, W.Wt + ch0 * REC_CD);
        scales_async(sE, W.sc + ch0 * 3 * kD);
        cp_commit();
        tile_async_split(xH, W.Kh + ch0 * REC_CD);
        cp_commit();
    }
    for (int64_t n = 0; n <= nc; ++n) {
        to_global(S, W.S + ((size_t)(base + s + n) * P.H + h) * REC_DD + c0, kD);
        if (n == nc) break;
        const size_t ch = (size_t)(base + n) * P.H + h;
        const float* e = sE + (n & 1) * 2 * kD;
        Frag<C, NCOL> u;
        from_global(u, W.Up + ch * REC_CD + c0, kD);
        cp_wait<1>();  // W~ and the scales of this chunk
        __syncthreads();
#pragma unroll
        for (int i = 0; i < F::MR; ++i)
#pragma unroll
            for (int j = 0; j < F::NJ; ++j) S.v[i][j] *= e[F::row(i)];
        to_smem_split(S, xX, RS);
        __syncthreads();
        gemm_ps<true, kD, true, false>(u, xW, RSD, xX, RS);  // U = U' - W~ X
        to_smem_split(u, xU, RS);
        to_global(u, W.Up + ch * REC_CD + c0, kD);  // U replaces U' (read back by the gradient pass)
        __syncthreads();
        if (n + 1 < nc) {
            tile_async_split(xW, W.Wt + (ch + P.H) * REC_CD);
            scales_async(sE + ((n + 1) & 1) * 2 * kD, W.sc + (ch + P.H) * 3 * kD);
            cp_commit();
            cp_wait<1>();  // K^ of this chunk
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        gemm_ps<false, C, false, false>(S, xH, RSD, xU, RS);  // X + K^^T U
#pragma unroll
        for (int i = 0; i < F::MR; ++i)
#pragma unroll
            for (int j = 0; j < F::NJ; ++j) S.v[i][j] *= e[kD + F::row(i)];
        __syncthreads();
        if (n + 1 < nc) {
            tile_async_split(xH, W.Kh + (ch + P.H) * REC_CD);
            cp_commit();
        }
    }
}

// Pass 3: state gradients at chunk ends, last chunk first.  K^ and the scales of chunk n-1 are
// copied in while W~^T Z of chunk n runs, and W~ of chunk n-1 while the next chunk's K^ dD runs.
template <int NCOL>
__global__ void __launch_bounds__(NT, 1) cbwd_dstates(CBwd W) {
    constexpr int RS = NCOL + 8;
    extern __shared__ __align__(16) float sm[];
    __nv_bfloat16* b16 = reinterpret_cast<__nv_bfloat16*>(sm);
    const Split xD{b16, b16 + kD * RS};                        // dD = Diag(e^{g_C - ref}) dS, this CTA's columns
    const Split xZ{xD.lo + kD * RS, xD.lo + kD * RS + C * RS};  // K^ dD, this CTA's columns
    const Split xW{xZ.lo + C * RS, xZ.lo + C * RS + C * RSD};  // W~
    const Split xH{xW.lo + C * RSD, xW.lo + 2 * C * RSD};      // K^
    float* sE = reinterpret_cast<float*>(xH.lo + C * RSD);     // [2][e^ref, e^{g_C - ref}]
    const BwdProblem& P = W.p;
    constexpr int PARTS = kD / NCOL;
    const int unit = blockIdx.x / PARTS, c0 = (blockIdx.x % PARTS) * NCOL;
    const int h = unit % P.H, s = unit / P.H;
    int64_t start, len;
    seq_of(P, s, start, len);
    const int64_t nc = (len + C - 1) / C, base = W.co[s];
    using F = Frag<kD, NCOL>;
    F dS;
    if (P.dfinal) from_global(dS, P.dfinal + ((size_t)s * P.H + h) * REC_DD + c0, kD);
    else dS.zero();
    if (nc > 0) {
        const size_t chl = (size_t)(base + nc - 1) * P.H + h;
        tile_async_split(xH, W.Kh + chl * REC_CD);
        scales_async(sE + ((nc - 1) & 1) * 2 * kD, W.sc + chl * 3 * kD);
        cp_commit();
        tile_async_split(xW, W.Wt + chl * REC_CD);
        cp_commit();
    }
    for (int64_t n = nc - 1; n >= 0; --n) {
        const size_t ch = (size_t)(base + n) * P.H + h;
        const float* e = sE + (n & 1) * 2 * kD;
        to_global(dS, W.dS + ch * REC_DD + c0, kD);
        cp_wait<1>();  // K^ and the scales of this chunk
        __syncthreads();
#pragma unroll
        for (int i = 0; i < F::MR; ++i)
#pragma unroll
            for (int j = 0; j < F::NJ; ++j) dS.v[i][j] *= e[kD + F::row(i)];
        to_smem_split(dS, xD, RS);
        __syncthreads();
        Frag<C, NCOL> z;
        z.zero();
        gemm_ps<false, kD, true, false>(z, xH, RSD, xD, RS);  // K^ dD
        to_smem_split(z, xZ, RS);
        __syncthreads();
        if (n > 0) {
            tile_async_split(xH, W.Kh + (ch - P.H) * REC_CD);
            scales_async(sE + ((n - 1) & 1) * 2 * kD, W.sc + (ch - P.H) * 3 * kD);
            cp_commit();
            cp_wait<1>();  // W~ of this chunk
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        gemm_ps<true, C, false, false>(dS, xW, RSD, xZ, RS);  // dD - W~^T (K^ dD)
        const float* E = W.Ej + ch * REC_DD + c0;
#pragma unroll
        for (int i = 0; i < F::MR; ++i)
#pragma unroll
            for (int j = 0; j < F::NJ; ++j)
                dS.v[i][j] = (dS.v[i][j] + E[(size_t)F::row(i) * kD + F::col(j)]) * e[F::row(i)];
        __syncthreads();
        if (n > 0) {
            tile_async_split(xW, W.Wt + (ch - P.H) * REC_CD);
            cp_commit();
        }
    }
    if (P.dinit) to_global(dS, P.dinit + ((size_t)s * P.H + h) * REC_DD + c0, kD);
}

// ---- passes 2 and 3 on the tcgen05 tensor cores -----------------------------------------------------
// One CTA of 256 threads per (sequence, head) carries all 128 value columns of the chain.  The chain
// matrix lives in TMEM in fp32 (lanes = value columns j, columns = key channels c), next to its bf16
// hi/lo split, which is the A operand of the chunk's first product.  W~ and K^ (split records written
// by the local pass) are copied with cp.async into 128-byte-swizzled tiles, rows t with the 128 key
// channels in two 64-channel atoms; the same bytes are the K-major B operand of a product over c and
// the MN-major B operand of a product over t.  Per chunk (TMEM holds the transposes):
//   states  (REV = false): D_U = U'^T - X^T W~^T    (A: X split, negated; B: W~, over c); U stored
//                          D_S = X^T + U^T K^       (A: U split;          B: K^, over t)
//                          S_{n+1} = D_S e^{g_C - ref} stored; X_{n+1} = S_{n+1} e^{ref'} into D_S, split
//   dstates (REV = true):  D_U = dD^T K^^T          (A: dD split;         B: K^, over c)
//                          D_S = dD^T - Z^T W~      (A: Z split, negated; B: W~, over t)
//                          dS_n = (D_S + E^T) e^{ref} stored; dD' = dS_n e^{g_C' - ref'} into D_S, split
// Each product is three bf16 MMAs (hi.hi + hi.lo + lo.hi) accumulating in fp32, the operand split of
// the warp-level passes.  Thread 0 issues the products; all threads do the element-wise work, warps
// w and w + 4 sharing TMEM lanes 32 (w % 4) .. + 31 and splitting the columns in halves.  U' and E are
// read straight from global memory, asked of L2 one chunk ahead.  Every wait is bounded.
namespace tcs {
constexpr int NTS = 256;
constexpr uint32_t T_S = 0, T_XH = 128, T_XL = 192, T_U = 256, T_UH = 320, T_UL = 352;  // TMEM columns
constexpr uint32_t HALF = 16384;               // one bf16 array of a split record as a swizzled tile
constexpr uint32_t OFF_SC = 8 * HALF;          // [3][2][D] fp32: e^ref, e^{g_C - ref} by chunk % 3
constexpr uint32_t OFF_BAR = OFF_SC + 3 * 2 * kD * 4;
constexpr uint32_t SMEM = OFF_BAR + 64 + 1024;  // + alignment slack
constexpr uint32_t ID_C = sm100::idesc_bf16(128, 64, 0, 0);   // over c: M = 128, N = 64, B K-major
constexpr uint32_t ID_T = sm100::idesc_bf16(128, 128, 0, 1);  // over t: M = 128, N = 128, B MN-major

// Split record (hi [C][D] bf16, then lo) -> two swizzled tiles (hi, lo): element (t, c) of a tile at
// atom c / 64, row t, 16-byte chunk ((c % 64) / 8) ^ (t % 8).
__device__ __forceinline__ void stage_record(uint8_t* tiles, const float* rec) {
    const uint8_t* src = reinterpret_cast<const uint8_t*>(rec);
#pragma unroll
    for (int k = 0; k < 2 * C * 16 / NTS; ++k) {
        const int i = threadIdx.x + k * NTS, p = i >> 10, t = (i >> 4) & 63, ck = i & 15;
        cp_async16b(tiles + p * HALF + (ck >> 3) * 8192 + t * 128 + (((ck & 7) ^ (t & 7)) << 4),
                    src + p * 16384 + t * 256 + ck * 16);
    }
}
// L2 prefetch hint of every 128-byte line of `bytes` bytes
__device__ __forceinline__ void l2_prefetch(const float* p, int bytes) {
    for (int i = threadIdx.x * 128; i < bytes; i += NTS * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(p) + i));
}
}  // namespace tcs

template <bool REV>
__global__ void __launch_bounds__(tcs::NTS, 1) cbwd_serial_tc(CBwd W) {
    using namespace tcs;
    extern __shared__ uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);  // [0] first product, [1] second, [2] CTA
    sm100::Abort* ab = reinterpret_cast<sm100::Abort*>(sm + OFF_BAR + 24);
    uint32_t* holder = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 32);
    float* ssc = reinterpret_cast<float*>(sm + OFF_SC);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int hf = warp >> 2;                    // column half of the element-wise work
    const int j = 32 * (warp & 3) + (tid & 31);  // value column = TMEM lane
    const BwdProblem& P = W.p;
    const int h = blockIdx.x % P.H, s = blockIdx.x / P.H;
    int64_t start, len;
    seq_of(P, s, start, len);
    const int nc = (int)((len + C - 1) / C);
    const int64_t base = W.co[s];
    const size_t unit_dd = ((size_t)s * P.H + h) * REC_DD;
    auto chi = [&](int n) -> size_t { return (size_t)(base + n) * P.H + h; };
    auto slot = [&](int n) -> float* { return W.S + ((size_t)(base + s + n) * P.H + h) * REC_DD; };
    if (tid == 0) {
        sm100::mbar_init(&bar[0], 1);
        sm100::mbar_init(&bar[1], 1);
        sm100::mbar_init(&bar[2], NTS);
        ab->flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) sm100::tmem_alloc(holder, 512);
    sm100::tc_fence_before();
    __syncthreads();
    sm100::tc_fence_after();
    const uint32_t tm = *holder, tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t sb = sm100::smem_u32(sm);
    uint32_t ph_sync = 0;
    auto cta_sync = [&]() -> bool {
        sm100::tc_fence_before();
        sm100::mbar_arrive(&bar[2]);
        const bool r = sm100::mbar_wait(&bar[2], (ph_sync++) & 1, ab, W.status);
        sm100::tc_fence_after();
        return r;
    };
    // the records of chunk n into buffer b; the scales of chunk n into slot n % 3
    auto stage = [&](int n, int b) {
        const size_t ch = chi(n);
        stage_record(sm + (4 * b + 0) * HALF, W.Wt + ch * REC_CD);
        stage_record(sm + (4 * b + 2) * HALF, W.Kh + ch * REC_CD);
    };
    auto stage_sc = [&](int n) {
        if (tid < 2 * kD / 4) cp_async16b(ssc + (n % 3) * 2 * kD + 4 * tid, W.sc + chi(n) * 3 * kD + 4 * tid);
    };
    // the cp.async data of every thread, visible to all threads and to the tensor cores
    auto staged = [&]() -> bool {
        cp_wait<0>();
        sm100::fence_proxy_async_smem();
        return cta_sync();
    };
    // this thread's 64 columns of D_S <- v, and its split beside it (negated for the states pass)
    auto put_chain = [&](uint32_t (&v)[2][32]) {
#pragma unroll
        for (int pc = 0; pc < 2; ++pc) {
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float x0 = __uint_as_float(v[pc][2 * e]), x1 = __uint_as_float(v[pc][2 * e + 1]);
                split_bf16(REV ? x0 : -x0, REV ? x1 : -x1, hi[e], lo[e]);
            }
            sm100::tmem_st32(tl + T_S + 64 * hf + 32 * pc, v[pc]);
            sm100::tmem_st16(tl + T_XH + 32 * hf + 16 * pc, hi);
            sm100::tmem_st16(tl + T_XL + 32 * hf + 16 * pc, lo);
        }
        sm100::tmem_st_wait();
    };
    auto col = [&](int pc, int e) { return 64 * hf + 32 * pc + e; };  // key channel of v[pc][e]
    const int n0 = REV ? nc - 1 : 0, dn = REV ? -1 : 1;  // first chunk of the chain, direction
    uint32_t un[32];  // states: U' of the coming chunk (this thread's 32 tokens)
    bool ok = true;
    if (nc > 0) {
        stage(n0, 0);
        stage_sc(n0);
        if (nc > 1) stage_sc(n0 + dn);
        if (!REV)
#pragma unroll
            for (int e = 0; e < 32; ++e) un[e] = __float_as_uint(W.Up[chi(n0) * REC_CD + (size_t)(32 * hf + e) * kD + j]);
    }
    cp_commit();
    {  // the chain's start, S_0 (states) or the cotangent of the end state (dstates): stored, then scaled
        const float* src = REV ? P.dfinal : P.init;
        uint32_t v[2][32];
#pragma unroll
        for (int pc = 0; pc < 2; ++pc)
#pragma unroll
            for (int e = 0; e < 32; ++e) v[pc][e] = __float_as_uint(src ? src[unit_dd + (size_t)col(pc, e) * kD + j] : 0.f);
        float* dst = !REV ? slot(0) : nc > 0 ? W.dS + chi(nc - 1) * REC_DD : P.dinit ? P.dinit + unit_dd : nullptr;
        if (dst)
#pragma unroll
            for (int pc = 0; pc < 2; ++pc)
#pragma unroll
                for (int e = 0; e < 32; ++e) dst[(size_t)col(pc, e) * kD + j] = __uint_as_float(v[pc][e]);
        if (nc > 0) {
            ok = staged();
            const float* sc = ssc + (n0 % 3) * 2 * kD + (REV ? kD : 0);  // e^{g_C - ref} or e^{ref} of chunk n0
#pragma unroll
            for (int pc = 0; pc < 2; ++pc)
#pragma unroll
                for (int e = 0; e < 32; ++e) v[pc][e] = __float_as_uint(__uint_as_float(v[pc][e]) * sc[col(pc, e)]);
            put_chain(v);
            if (ok) ok = cta_sync();
        }
    }
    for (int k = 0; ok && k < nc; ++k) {
        const int n = n0 + dn * k, b = k & 1;
        const size_t ch = chi(n);
        const bool more = k + 1 < nc;
        if (more) {  // the next chunk's records, the scales of the one after it, U' / E of the next chunk to L2
            stage(n + dn, b ^ 1);
            if (k + 2 < nc) stage_sc(n + 2 * dn);
            if (REV)
                l2_prefetch(W.Ej + chi(n + dn) * REC_DD, REC_DD * 4);
            else
                l2_prefetch(W.Up + chi(n + dn) * REC_CD, REC_CD * 4);
        }
        cp_commit();
        if (!REV) {  // D_U <- U'
            sm100::tmem_st32(tl + T_U + 32 * hf, un);
            sm100::tmem_st_wait();
            if (!(ok = cta_sync())) break;
        }
        const uint32_t tw = sb + (4 * b + 0) * HALF, th = sb + (4 * b + 2) * HALF;  // W~, K^ (hi; lo at + HALF)
        if (tid == 0) {  // first product, over the key channels
            const uint32_t t1 = REV ? th : tw;
#pragma unroll
            for (int st = 0; st < 8; ++st) {
                const uint64_t bh = sm100::sdesc(t1 + (st >> 2) * 8192, 16, 1024) + 2u * (st & 3);
                const uint64_t bl = sm100::sdesc(t1 + HALF + (st >> 2) * 8192, 16, 1024) + 2u * (st & 3);
                sm100::mma_ts(tm + T_U, tm + T_XH + 8 * st, bh, ID_C, REV ? (st > 0) : 1);
                sm100::mma_ts(tm + T_U, tm + T_XH + 8 * st, bl, ID_C, 1);
                sm100::mma_ts(tm + T_U, tm + T_XL + 8 * st, bh, ID_C, 1);
            }
            sm100::mma_commit(&bar[0]);
        }
        if (!(ok = sm100::mbar_wait(&bar[0], k & 1, ab, W.status))) break;
        sm100::tc_fence_after();
        {  // U (stored; its split is the next A operand) or Z (its split negated)
            uint32_t u[32], hi[16], lo[16];
            sm100::tmem_ld32(tl + T_U + 32 * hf, u);
            sm100::tmem_ld_wait();
            if (!REV)
#pragma unroll
                for (int e = 0; e < 32; ++e) W.Up[ch * REC_CD + (size_t)(32 * hf + e) * kD + j] = __uint_as_float(u[e]);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float x0 = __uint_as_float(u[2 * e]), x1 = __uint_as_float(u[2 * e + 1]);
                split_bf16(REV ? -x0 : x0, REV ? -x1 : x1, hi[e], lo[e]);
            }
            sm100::tmem_st16(tl + T_UH + 16 * hf, hi);
            sm100::tmem_st16(tl + T_UL + 16 * hf, lo);
            sm100::tmem_st_wait();
        }
        if (!(ok = cta_sync())) break;
        if (tid == 0) {  // second product, over the tokens
            const uint32_t t2 = REV ? tw : th;
#pragma unroll
            for (int st = 0; st < 4; ++st) {
                const uint64_t bh = sm100::sdesc(t2, 8192, 1024) + 128u * st;
                const uint64_t bl = sm100::sdesc(t2 + HALF, 8192, 1024) + 128u * st;
                sm100::mma_ts(tm + T_S, tm + T_UH + 8 * st, bh, ID_T, 1);
                sm100::mma_ts(tm + T_S, tm + T_UH + 8 * st, bl, ID_T, 1);
                sm100::mma_ts(tm + T_S, tm + T_UL + 8 * st, bh, ID_T, 1);
            }
            sm100::mma_commit(&bar[1]);
        }
        // loaded while the product runs: E^T of this chunk (dstates), U' of the next (states)
        float ev[2][32];
        if (REV) {
#pragma unroll
            for (int pc = 0; pc < 2; ++pc)
#pragma unroll
                for (int e = 0; e < 32; ++e) ev[pc][e] = W.Ej[ch * REC_DD + (size_t)col(pc, e) * kD + j];
        } else if (more) {
#pragma unroll
            for (int e = 0; e < 32; ++e) un[e] = __float_as_uint(W.Up[chi(n + 1) * REC_CD + (size_t)(32 * hf + e) * kD + j]);
        }
        if (!(ok = sm100::mbar_wait(&bar[1], k & 1, ab, W.status))) break;
        sm100::tc_fence_after();
        {
            const float* e_ref = ssc + (n % 3) * 2 * kD;                               // e^{ref} of this chunk
            const float* e_dec = e_ref + kD;                                           // e^{g_C - ref}
            const float* nxt = ssc + ((n + dn + 3) % 3) * 2 * kD + (REV ? kD : 0);  // the next chunk's factor
            uint32_t v[2][32];
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
                sm100::tmem_ld32(tl + T_S + 64 * hf + 32 * pc, v[pc]);
                sm100::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float x = __uint_as_float(v[pc][e]);
                    v[pc][e] = __float_as_uint(REV ? (x + ev[pc][e]) * e_ref[col(pc, e)] : x * e_dec[col(pc, e)]);
                }
            }
            // S_{n+1} into its slot; dS_n into the record of chunk n - 1, or d_init after the first chunk
            float* dst = !REV ? slot(n + 1) : more ? W.dS + chi(n - 1) * REC_DD : P.dinit ? P.dinit + unit_dd : nullptr;
            if (dst)
#pragma unroll
                for (int pc = 0; pc < 2; ++pc)
#pragma unroll
                    for (int e = 0; e < 32; ++e) dst[(size_t)col(pc, e) * kD + j] = __uint_as_float(v[pc][e]);
            if (more) {
#pragma unroll
                for (int pc = 0; pc < 2; ++pc)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        v[pc][e] = __float_as_uint(__uint_as_float(v[pc][e]) * nxt[col(pc, e)]);
                put_chain(v);
            }
        }
        if (!(ok = staged())) break;
    }
    sm100::tc_fence_before();
    __syncthreads();
    sm100::tc_fence_after();
    if (ab->flag) {  // aborted: let any product still in flight drain before TMEM goes away
        const long long t0 = clock64();
        while (clock64() - t0 < 2000000) {
        }
    }
    if (warp == 0) sm100::tmem_dealloc(tm, 512);
}

// ---- pass 4a: the state-dependent gradient products of each chunk --------------------------------
constexpr int SMEM_GRAD_A = (TILE_DD + 4 * TILE_CD + TILE_CC + 2 * kD) * 4;

__global__ void __launch_bounds__(NT, 1) cbwd_grad_state(CBwd W) {
    extern __shared__ __align__(16) float sm[];
    // Every tile of this pass is only ever a product operand, so each is stored pre-split.
    uint8_t* base = reinterpret_cast<uint8_t*>(sm);
    auto split_at = [&](size_t off, int rows, int rs) {
        __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(base + off);
        return Split{b, b + (size_t)rows * rs};
    };
    constexpr size_t BD = 4ull * kD * RSD, BC = 4ull * C * RSD, BCC = 4ull * C * RSC;  // bytes: hi and lo
    static_assert(BD + 4 * BC + BCC + 8 * kD == SMEM_GRAD_A, "split tiles take the fp32 tiles' room");
    const Split sR = split_at(0, kD, RSD);               // dD, then X
    const Split s1 = split_at(BD, C, RSD);               // K^
    const Split s2 = split_at(BD + BC, C, RSD);          // U
    const Split s3 = split_at(BD + 2 * BC, C, RSD);      // dU
    const Split s4 = split_at(BD + 3 * BC, C, RSD);      // dO
    const Split s5 = split_at(BD + 4 * BC, C, RSC);      // P, then dP
    float* sE = reinterpret_cast<float*>(base + BD + 4 * BC + BCC);
    const BwdProblem& P = W.p;
    const int h = blockIdx.x % P.H;
    const int64_t cg = blockIdx.x / P.H;
    ChunkAt c;
    if (!locate_chunk(W, cg, c)) return;
    const size_t ch = (size_t)cg * P.H + h;
    const size_t s_slot = ((size_t)(W.co[c.s] + c.s + c.n) * P.H + h) * REC_DD;
    const float* S0 = W.S + s_slot;
    const float* SC = W.S + s_slot + (size_t)P.H * REC_DD;  // the next state of the same sequence
    const float* dSC = W.dS + ch * REC_DD;
    if (threadIdx.x < 2 * kD) sE[threadIdx.x] = W.sc[ch * 3 * kD + threadIdx.x];
    load_tile_split<C>(s2, W.Up + ch * REC_CD);  // U, stored by the states pass
    {  // final-decay gradient: sum_j S_C[c][j] dS_C[c][j], one warp per row, every load of the
       // warp's 8 rows issued before the first is used
        const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
        float sv[8][4], dv[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                sv[i][j] = SC[(w + 16 * i) * kD + l + 32 * j];
                dv[i][j] = dSC[(w + 16 * i) * kD + l + 32 * j];
            }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float a = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) a = fmaf(sv[i][j], dv[i][j], a);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (l == 0) W.sc[ch * 3 * kD + 2 * kD + w + 16 * i] = a;
        }
    }
    __syncthreads();
    load_tile_split<kD>(sR, dSC, sE + kD);  // dD
    load_record_split(s1, W.Kh + ch * REC_CD);
    {
        float4 o4[4];
        load_rows(o4, P.dout, c, P.H, h);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gi = threadIdx.x + i * NT;
            split_store4(s4, (gi >> 5) * RSD + (gi & 31) * 4, o4[i]);
        }
    }
    load_cc_split(s5, W.Pq + ch * REC_CC);
    __syncthreads();
    Frag<C, kD> du, acc;
    du.zero();
    gemm_ps<false, kD, true, false>(du, s1, RSD, sR, RSD);  // K^ dD
    gemm_ps<false, C, false, false>(du, s5, RSC, s4, RSD);  // + P^T dO
    to_smem_split(du, s3, RSD);
    to_global(du, W.Up + ch * REC_CD);
    acc.zero();
    gemm_ps<false, kD, true, true>(acc, s2, RSD, sR, RSD);  // dK^ = U dD^T
    to_global(acc, W.Ej + ch * REC_DD + REC_CD);
    Frag<C, C> dp;
    dp.zero();
    gemm_ps<false, kD, true, true>(dp, s4, RSD, s2, RSD);  // dP = lower(dO U^T)
#pragma unroll
    for (int i = 0; i < Frag<C, C>::MR; ++i)
#pragma unroll
        for (int j = 0; j < Frag<C, C>::NJ; ++j)
            if (Frag<C, C>::col(j) > Frag<C, C>::row(i)) dp.v[i][j] = 0.f;
    __syncthreads();
    load_tile_split<kD>(sR, S0, sE);  // X again
    to_smem_split(dp, s5, RSC);
    to_global(dp, W.Pq + ch * REC_CC);
    __syncthreads();
    acc.zero();
    gemm_ps<false, kD, true, true>(acc, s4, RSD, sR, RSD);  // dQ~ = dO X^T
    gemm_ps<false, C, true, false>(acc, s5, RSC, s1, RSD);  //      + dP K^
    to_global(acc, W.Ej + ch * REC_DD);
    acc.zero();
    gemm_ps<true, kD, true, true>(acc, s3, RSD, sR, RSD);  // dW~ = -dU X^T
    to_global(acc, W.Wt + ch * REC_CD);
}

// ---- pass 4b: the chunk's local gradient products and the input gradients ----------------------
constexpr int SMEM_GRAD_B = (5 * TILE_CD + 3 * TILE_CC + C + kD) * 4;

template <typename Tin>
__global__ void __launch_bounds__(NT, 1) cbwd_grad_local(CBwd W) {
    extern __shared__ __align__(16) float sm[];
    float* s0 = sm;              // g, then V, then d(g - ref)
    float* sQ = s0 + TILE_CD;    // Q~
    float* sK = sQ + TILE_CD;    // K~
    float* sH = sK + TILE_CD;    // K^
    float* sX = sH + TILE_CD;    // dU, then dW~ (pre-split), then g
    float* sT = sX + TILE_CD;    // T (pre-split)
    float* sP = sT + TILE_CC;    // dP, then Y = dT T^T (pre-split)
    float* sM = sP + TILE_CC;    // dT, then dA, then diag(beta) dA (pre-split)
    float* sB = sM + TILE_CC;    // beta
    float* sG = sB + C;          // final-decay gradient
    // tiles that are only product operands are stored pre-split in the fp32 tiles' room
    auto split_of = [](float* t, int rows, int rs) {
        __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(t);
        return Split{b, b + (size_t)rows * rs};
    };
    static_assert(TILE_CD == C * RSD && TILE_CC == C * RSC, "a split tile (2 x 2 bytes per element) fills an fp32 tile");
    const Split xX = split_of(sX, C, RSD), xT = split_of(sT, C, RSC), xP = split_of(sP, C, RSC),
                xM = split_of(sM, C, RSC);
    const BwdProblem& P = W.p;
    const int h = blockIdx.x % P.H;
    const int64_t cg = blockIdx.x / P.H;
    ChunkAt c;
    if (!locate_chunk(W, cg, c)) return;
    const size_t ch = (size_t)cg * P.H + h;
    using F = Frag<C, kD>;
    using FC = Frag<C, C>;

    load_gates(W, c, h, s0, sB, sM);
    scaled_qk<Tin>(W, c, h, s0, sQ, sK, sH, nullptr);
    if (threadIdx.x < kD) sG[threadIdx.x] = W.sc[ch * 3 * kD + 2 * kD + threadIdx.x];
    load_cc_split(xT, W.Tm + ch * REC_CC);
    load_cc_split(xP, W.Pq + ch * REC_CC);
    load_tile_split<C>(xX, W.Up + ch * REC_CD);  // dU
    __syncthreads();
    {
        float4 v4[4];
        load_rows(v4, static_cast<const Tin*>(P.v), c, P.H, h);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gi = threadIdx.x + i * NT;
            *reinterpret_cast<float4*>(s0 + (gi >> 5) * LD + (gi & 31) * 4) = v4[i];
        }
    }
    __syncthreads();

    float db[F::MR];  // per-lane partial sums of dbeta for this warp's rows
#pragma unroll
    for (int i = 0; i < F::MR; ++i) db[i] = 0.f;
    F dKh, dKt, t;
    from_global(dKh, W.Ej + ch * REC_DD + REC_CD);
    gemm_mx<false, C, false, false>(dKh, OpS{xP, RSC}, OpF{sQ, LD});  // + dP^T Q~
    FC dT;
    dT.zero();
    gemm_mx<false, kD, true, true>(dT, OpS{xX, RSD}, OpF{s0, LD});  // dU V^T
    t.zero();
    gemm_ps<false, C, false, false>(t, xT, RSC, xX, RSD);  // T^T dU
    // dv, dq, dk: adjacent column pairs as 8-byte stores where the arrays allow it
    const bool pairs = ((reinterpret_cast<uintptr_t>(P.dv) | reinterpret_cast<uintptr_t>(P.dq) |
                         reinterpret_cast<uintptr_t>(P.dk)) & 7u) == 0;
#pragma unroll
    for (int i = 0; i < F::MR; ++i) {
        const int r = F::row(i);
#pragma unroll
        for (int j = 0; j < F::NJ; j += 2) {
            db[i] = fmaf(t.v[i][j], s0[r * LD + F::col(j)], db[i]);
            db[i] = fmaf(t.v[i][j + 1], s0[r * LD + F::col(j + 1)], db[i]);
            if (r < c.L) {
                float* dst = P.dv + ((size_t)(c.tok0 + r) * P.H + h) * kD + F::col(j);
                const float a0 = sB[r] * t.v[i][j], a1 = sB[r] * t.v[i][j + 1];
                if (pairs) {
                    *reinterpret_cast<float2*>(dst) = make_float2(a0, a1);
                } else {
                    dst[0] = a0;
                    dst[1] = a1;
                }
            }
        }
    }
    __syncthreads();
    load_tile_split<C>(xX, W.Wt + ch * REC_CD);  // dW~
    __syncthreads();
    gemm_mx<false, kD, true, true>(dT, OpS{xX, RSD}, OpF{sK, LD});  // + dW~ K~^T
#pragma unroll
    for (int i = 0; i < FC::MR; ++i)
#pragma unroll
        for (int j = 0; j < FC::NJ; ++j) dT.v[i][j] *= sB[FC::col(j)];
    to_smem_split(dT, xM, RSC);
    t.zero();
    gemm_ps<false, C, false, false>(t, xT, RSC, xX, RSD);  // T^T dW~
#pragma unroll
    for (int i = 0; i < F::MR; ++i) {
        const int r = F::row(i);
#pragma unroll
        for (int j = 0; j < F::NJ; ++j) {
            db[i] = fmaf(t.v[i][j], sK[r * LD + F::col(j)], db[i]);
            dKt.v[i][j] = sB[r] * t.v[i][j];
        }
    }
    __syncthreads();
    {
        FC y;
        y.zero();
        gemm_ps<false, C, true, true>(y, xM, RSC, xT, RSC);  // Y = dT T^T
        to_smem_split(y, xP, RSC);
    }
    __syncthreads();
    FC a;  // dA = -T^T Y, strictly lower part
    a.zero();
    gemm_ps<true, C, false, false>(a, xT, RSC, xP, RSC);
#pragma unroll
    for (int i = 0; i < FC::MR; ++i)
#pragma unroll
        for (int j = 0; j < FC::NJ; ++j)
            if (FC::col(j) >= FC::row(i)) a.v[i][j] = 0.f;
    to_smem_split(a, xM, RSC);
    __syncthreads();
    t.zero();
    gemm_mx<false, C, true, false>(t, OpS{xM, RSC}, OpF{sH, LD});  // dA K^
#pragma unroll
    for (int i = 0; i < F::MR; ++i) {
        const int r = F::row(i);
#pragma unroll
        for (int j = 0; j < F::NJ; ++j) {
            db[i] = fmaf(t.v[i][j], sK[r * LD + F::col(j)], db[i]);
            dKt.v[i][j] = fmaf(sB[r], t.v[i][j], dKt.v[i][j]);
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < FC::MR; ++i)
#pragma unroll
        for (int j = 0; j < FC::NJ; ++j) a.v[i][j] *= sB[FC::row(i)];  // diag(beta) dA
    to_smem_split(a, xM, RSC);
    __syncthreads();
    gemm_mx<false, C, false, false>(dKh, OpS{xM, RSC}, OpF{sK, LD});  // + (diag(beta) dA)^T K~

    // beta gradient: a row's columns are spread over the 4 lanes of a quad (t) and the 4 warps w / 4;
    // sum over the quad, then over the warps in a fixed order (s0 rows 0..3 hold the partials)
    __syncthreads();
#pragma unroll
    for (int i = 0; i < F::MR; ++i) {
        float x = db[i];
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        if ((threadIdx.x & 3) == 0) s0[(threadIdx.x >> 7) * LD + F::row(i)] = x;
    }
    __syncthreads();
    if (threadIdx.x < c.L)
        P.dbeta[(size_t)(c.tok0 + threadIdx.x) * P.H + h] =
            ((s0[threadIdx.x] + s0[LD + threadIdx.x]) + s0[2 * LD + threadIdx.x]) + s0[3 * LD + threadIdx.x];
    // decay gradient and dq, dk
    __syncthreads();
    load_gates(W, c, h, sX, nullptr, sM);  // g again
    F dQt;
    from_global(dQt, W.Ej + ch * REC_DD);
#pragma unroll
    for (int i = 0; i < F::MR; ++i) {
        const int r = F::row(i);
#pragma unroll
        for (int j = 0; j < F::NJ; j += 2) {
            float gq[2], gk[2];
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int col = F::col(j + e2);
                const int o = r * LD + col;
                const float x = sX[o] - sX[31 * LD + col];
                const float e = expf(x), f = expf(-x);
                gq[e2] = dQt.v[i][j + e2] * e;
                gk[e2] = fmaf(dKt.v[i][j + e2], e, dKh.v[i][j + e2] * f);
                float dl = fmaf(dQt.v[i][j + e2], sQ[o], fmaf(dKt.v[i][j + e2], sK[o], -dKh.v[i][j + e2] * sH[o]));
                if (r == C - 1) dl += sG[col];
                s0[o] = dl;
            }
            if (r < c.L) {
                const size_t off = ((size_t)(c.tok0 + r) * P.H + h) * kD + F::col(j);
                if (pairs) {
                    *reinterpret_cast<float2*>(P.dq + off) = make_float2(gq[0], gq[1]);
                    *reinterpret_cast<float2*>(P.dk + off) = make_float2(gk[0], gk[1]);
                } else {
                    P.dq[off] = gq[0];
                    P.dq[off + 1] = gq[1];
                    P.dk[off] = gk[0];
                    P.dk[off + 1] = gk[1];
                }
            }
        }
    }
    __syncthreads();
    if (P.gate == kGateNone) return;
    if (threadIdx.x < kD) {  // reverse cumulative sum over the chunk's rows
        float run = 0.f;
        for (int r = C - 1; r >= 0; --r) {
            run += s0[r * LD + threadIdx.x];
            s0[r * LD + threadIdx.x] = run;
        }
    }
    __syncthreads();
    if (P.gate == kGateChannel) {
        for (int idx = threadIdx.x; idx < c.L * kD; idx += NT) {
            const int r = idx >> 7, col = idx & 127;
            P.dlog_alpha[((size_t)(c.tok0 + r) * P.H + h) * kD + col] = s0[r * LD + col];
        }
    } else {  // one gate per head: the sum over key channels, one warp per row
        const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
        for (int r = w; r < c.L; r += 16) {
            float a = ((s0[r * LD + l] + s0[r * LD + l + 32]) + s0[r * LD + l + 64]) + s0[r * LD + l + 96];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (l == 0) P.dlog_alpha[(size_t)(c.tok0 + r) * P.H + h] = a;
        }
    }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Upper bound on the number of chunks: sum_s ceil(len_s / C) <= T_total / C + N.
int64_t chunk_bound(int N, int64_t T_total, bool varlen, int64_t T_uniform) {
    return varlen ? T_total / C + N : (int64_t)N * ((T_uniform + C - 1) / C);
}

}  // namespace

// Layout: chunk offsets [N+1] | redo flags [N*H] | records | states.  The token-serial backward
// that recomputes flagged units runs after the chunked passes and reuses everything from the
// records on, so that part is at least bwd_workspace() long.
size_t chunk_bwd_workspace(int N, int64_t T_total, int H, bool varlen) {
    const int64_t T_uniform = varlen || N == 0 ? 0 : T_total / N;
    const size_t nch = (size_t)chunk_bound(N, T_total, varlen, T_uniform) * H;
    const size_t per = 3 * REC_CD + 2 * REC_DD + 2 * REC_CC + 3 * kD;  // Wt Up Kh, Ej dS, Tm Pq, sc
    const size_t states = ((size_t)chunk_bound(N, T_total, varlen, T_uniform) + N) * H * REC_DD;
    size_t tail = align256(nch * per * 4) + align256(states * 4);
    const size_t serial = bwd_workspace(N, T_total, H);
    if (tail < serial) tail = align256(serial);
    return align256((size_t)(N + 1) * 8) + align256((size_t)N * H * 4) + tail;
}

cudaError_t launch_chunk_bwd(const BwdProblem& p, int in_dtype, void* workspace, int* status, cudaStream_t st) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    const bool varlen = p.cu_seqlens != nullptr;
    const int64_t ncb = chunk_bound(p.N, p.T_total, varlen, p.T_uniform);
    const size_t nch = (size_t)ncb * p.H;
    CBwd W{};
    W.p = p;
    W.status = status;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    W.co_w = reinterpret_cast<int64_t*>(ws);
    W.co = W.co_w;
    W.redo = reinterpret_cast<int*>(ws + align256((size_t)(p.N + 1) * 8));
    uint8_t* tail = ws + align256((size_t)(p.N + 1) * 8) + align256((size_t)p.N * p.H * 4);
    float* f = reinterpret_cast<float*>(tail);
    W.Wt = f; f += nch * REC_CD;
    W.Up = f; f += nch * REC_CD;
    W.Kh = f; f += nch * REC_CD;
    W.Ej = f; f += nch * REC_DD;
    W.dS = f; f += nch * REC_DD;
    W.Tm = f; f += nch * REC_CC;
    W.Pq = f; f += nch * REC_CC;
    W.sc = f; f += nch * 3 * kD;
    W.S = reinterpret_cast<float*>(tail + align256(nch * (3 * REC_CD + 2 * REC_DD + 2 * REC_CC + 3 * kD) * 4));
    chunk_offsets_kernel<<<1, 1024, 0, st>>>(W);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const bool bf = in_dtype == KDA_BF16;
    auto local = bf ? cbwd_local<__nv_bfloat16> : cbwd_local<float>;
    auto grad_local = bf ? cbwd_grad_local<__nv_bfloat16> : cbwd_grad_local<float>;
    struct K {
        const void* fn;
        int smem;
    };
    // The serial passes: one CTA per (sequence, head) on tcgen05 (256 threads) while the units fill
    // more than a quarter of the SMs; with fewer, the warp-level form with each unit's value columns
    // split over 4 CTAs of 32 columns (measured faster there: 1.49 against 1.64 ms at B=1, H=8).
    int sms = 0, dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const int64_t units = (int64_t)p.N * p.H;
    const bool tc = units * 4 > sms;
    const int parts = tc ? 1 : 4;
    const void* states = tc ? (const void*)cbwd_serial_tc<false> : (const void*)cbwd_states<32>;
    const void* dstates = tc ? (const void*)cbwd_serial_tc<true> : (const void*)cbwd_dstates<32>;
    const int smem_ser = tc ? (int)tcs::SMEM : smem_serial<32>();
    const int nt_ser = tc ? tcs::NTS : NT;
    const K ks[] = {{(const void*)local, SMEM_LOCAL},
                    {states, smem_ser},
                    {dstates, smem_ser},
                    {(const void*)cbwd_grad_state, SMEM_GRAD_A},
                    {(const void*)grad_local, SMEM_GRAD_B}};
    for (const K& k : ks)
        if ((e = cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem)) != cudaSuccess)
            return e;
    const unsigned chunk_ctas = (unsigned)nch, seq_ctas = (unsigned)(units * parts);
    if (chunk_ctas > 0) local<<<chunk_ctas, NT, SMEM_LOCAL, st>>>(W);
    void* args[] = {&W};
    if ((e = cudaLaunchKernel(states, dim3(seq_ctas), dim3(nt_ser), args, (size_t)smem_ser, st)) != cudaSuccess) return e;
    if ((e = cudaLaunchKernel(dstates, dim3(seq_ctas), dim3(nt_ser), args, (size_t)smem_ser, st)) != cudaSuccess) return e;
    if (chunk_ctas > 0) {
        cbwd_grad_state<<<chunk_ctas, NT, SMEM_GRAD_A, st>>>(W);
        grad_local<<<chunk_ctas, NT, SMEM_GRAD_B, st>>>(W);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the flagged units, exactly, by the token-serial backward (its CTAs for the others return)
    BwdProblem q = p;
    q.redo = W.redo;
    return launch_bwd(q, in_dtype, tail, st);
}

}  // namespace kda
