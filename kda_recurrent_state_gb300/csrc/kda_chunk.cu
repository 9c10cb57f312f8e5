// kda_chunk.cu -- chunkwise KDA prefill on tcgen05 tensor cores (chunk = 64).
//
// What it computes: the "Kimi K3" article's (lshu.cn/news/263999) §四 recurrence
//   S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,  o_t = S_t^T q_t,
// evaluated as in §六: recurrent between chunks of C = 64 tokens, and inside a
// chunk the product of the rank-one factors is rewritten in WY form so that the
// work becomes a few dense products.  For a chunk with start state S0, rows
// r = 0..63 and g_r = sum_{s<=r} log alpha_s (per key channel c):
//   A[r][i]  = beta_r sum_c k_r[c] k_i[c] e^{g_r[c]-g_i[c]}  (i < r),  T = (I + A)^-1
//   W        = T diag(beta) Ktil,   U' = T diag(beta) V,   U = U' - W S0
//   O        = Qtil S0 + lower_incl(Qtil Khat^T) U
//   S_C      = Diag(e^{g_C}) S0 + Kend^T U           (= (D - Kend^T W) S0 + Kend^T U')
// with Ktil = k e^{g}, Qtil = q e^{g}, Khat = k e^{-g}, Kend = k e^{g_C - g}.
//
// Scaling (so fp16 operands never overflow): every decay factor is taken
// relative to a per-channel reference ref = g_31 (the log-decay after the
// chunk's first 32 tokens): Ktil_p = k e^{g-ref}, Qtil_p = q e^{g-ref},
// Khat_p = k e^{ref-g}; the pairwise products e^{g_r - g_i} are unchanged and
// each factor stays within e^{max(|g_31|, |g_63 - g_31|)}.  The state is carried
// as X = Diag(e^{ref}) S0 (what the products with Ktil_p / Qtil_p need), and the
// state accumulator holds D = X + Khat_p^T U, so S_C = Diag(e^{g_63 - ref}) D.
//
// The triangular inverse on the tensor cores: split A = A_d + A_o into its
// 16x16 diagonal blocks and the rest.  With Dg = (I + A_d)^-1 (four small
// inverses, CUDA cores) and N = Dg A_o (strictly block-lower, N^4 = 0):
//   I + A = (I + A_d)(I + N)   =>   T = (I + N)^-1 Dg = (I - N)(I + N^2) Dg,
// evaluated as four 64x64x64 products: N = Dg A_o, N2 = N N, M = Dg + N2 Dg,
// T = M - N M.
//
// Data layout on chip (one CTA = one (sequence, head), all of d_v = 128):
//   TMEM (fp32 accumulators, lanes = the M rows):
//     D_S [j][c] state (128 cols)   X16 [j][c] fp16 A operand   D_U [j][r] U'/U
//     U16 [j][r] fp16 A operand (over D_U)   D_O [j][r] output   D_G [r|64+r][i] Gram
//     D_W [c][r] W^T, and before that the four M = 64 products of the inverse
//     V16 [2][j][i] fp16 A operand (v^T), by chunk parity
//   SMEM (fp16, 128-byte swizzled rows of 64 elements):
//     KT[c][r] = Ktil_p, QT[c][r] = Qtil_p (adjacent: together the M = 128 A
//     operand of the Gram), KH[c][r] = Khat_p, PP[r][i] = P, WT[c][r] = -W^T,
//     DT[m][r] = Dg^T, B1 = A_o -> N2 -> -M (row-major), NR = N -> T diag(beta)
//     (row-major); fp32 diagonal blocks of A and of Dg; a ring of 16-token
//     input slots filled by TMA.
//   The products (all tcgen05.mma, fp16 operands, fp32 accumulation):
//     Gram  D_G = [KT;QT] x KH                 M=128 N=64  K=128
//     S1..4 D_W = DT x B1, NR x NR, B1 x DT, NR x B1 (accumulate)   M=64 N=64 K=64
//     WY    D_W = KT x T,  D_U = V16 x T       M=128 N=64  K=64
//     (i)   D_U += X16 x WT                    M=128 N=64  K=128
//     (iii) D_O = X16 x QT + U16 x PP          M=128 N=64  K=128+64
//     (ii)  D_S += U16 x KH                    M=128 N=128 K=64
//
// Warp roles (16 warps): 0 TMA producer, 1 MMA issuer (+ TMEM allocation),
// 2-3 the 16x16 diagonal-block inverses, 4-7 "prep" warpgroup (decay cumsum,
// operand tiles, Gram readout), 8-11 "state" warpgroup (W and U conversion,
// outputs, state rescale, snapshots), 12-15 "tri" warpgroup (readout of the
// four inverse products).  Roles hand work to each other through mbarriers;
// every wait is bounded.
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {
using namespace sm100;

constexpr int C = 64;   // chunk length
constexpr int QR = 16;  // token rows per input slot
constexpr int NTHREADS = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxExp2 = 15.0f;  // |g - ref| bound (log2 units) for fp16 operands

// TMEM column map (512 columns allocated).  The fp16 U operand is written over
// the first 32 columns of the U accumulator once that has been read out; V16
// (the fp16 v^T operand) is double-buffered by chunk parity.
constexpr uint32_t TM_S = 0, TM_X16 = 128, TM_U = 192, TM_U16 = 192, TM_O = 256, TM_G = 320, TM_W = 384,
                   TM_V16 = 448;

template <typename Tin>
struct Cfg {
    static constexpr int ES = sizeof(Tin);
    static constexpr int NSLOT = ES == 2 ? 3 : 2;
    static constexpr int NPP = ES == 2 ? 2 : 1;  // P buffers (fp32 inputs trade overlap for smem)
    static constexpr uint32_t SLOT_Q = 0;
    static constexpr uint32_t SLOT_K = QR * 128 * ES;
    static constexpr uint32_t SLOT_V = 2 * QR * 128 * ES;
    static constexpr uint32_t SLOT_LA = 3 * QR * 128 * ES;
    static constexpr uint32_t SLOT_BYTES = 3 * QR * 128 * ES + QR * 128 * 4;
    // shared memory map (offsets from a 1024-byte aligned base)
    static constexpr uint32_t OFF_KQ = 0;                    // [2] x (KT 16K | QT 16K)
    static constexpr uint32_t OFF_KH = 65536;                // [2] x 16K
    static constexpr uint32_t OFF_PP = 98304;                // [NPP] x 8K
    static constexpr uint32_t OFF_WT = OFF_PP + NPP * 8192;  // 16K
    static constexpr uint32_t OFF_DT = OFF_WT + 16384;       // 8K
    static constexpr uint32_t OFF_B1 = OFF_DT + 8192;        // 8K
    static constexpr uint32_t OFF_NR = OFF_B1 + 8192;        // 8K
    static constexpr uint32_t OFF_LDG = OFF_NR + 8192;       // fp32 [4][16][17]
    static constexpr uint32_t OFF_DFP = OFF_LDG + 4 * 16 * 17 * 4;  // fp32 [4][16][16]
    static constexpr uint32_t OFF_RING = OFF_DFP + 4 * 16 * 16 * 4;
    static constexpr uint32_t OFF_VEC = OFF_RING + NSLOT * SLOT_BYTES;  // a[2][128], b[2][128]
    static constexpr uint32_t OFF_BETA = OFF_VEC + 4 * 128 * 4;         // [4][64]
    static constexpr uint32_t OFF_BAR = OFF_BETA + 4 * 64 * 4;
    static constexpr uint32_t NBAR = 44;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
};
static_assert(Cfg<__nv_bfloat16>::SMEM_BYTES <= 232448, "smem budget (bf16)");
static_assert(Cfg<float>::SMEM_BYTES <= 232448, "smem budget (fp32)");
static_assert(Cfg<__nv_bfloat16>::OFF_RING % 128 == 0 && Cfg<float>::OFF_RING % 128 == 0, "TMA destinations");

// barrier indices
enum {
    B_FULL = 0,     // [NSLOT] input slot landed
    B_EMPTY = 3,    // [NSLOT] input slot consumed
    B_PREPD = 6,    // [2] KT/QT/KH, vectors, beta of a chunk ready
    B_GDONE = 9,    // Gram complete
    B_P2D = 10,     // Gram read out: D_G free; A blocks, A_o and P written
    B_AFREE = 11,   // diagonal-block inverses done reading their input
    B_DRDY = 12,    // DT and the fp32 diagonal inverses written
    B_S1D = 13, B_C1 = 14, B_S2D = 15, B_C2 = 16, B_S3D = 17, B_C3 = 18,  // inverse products / readouts
    B_TDONE = 19,   // last inverse product complete
    B_TRDY = 20,    // T diag(beta) written
    B_WYDONE = 21,  // WY products complete
    B_WRDY = 22,    // WT written, D_W free
    B_XRDY = 23,    // X16 / D_S ready for the chunk
    B_UIDONE = 24,  // (i) and (iii-a) complete
    B_URDY = 25,    // U16 written, D_U free
    B_SDONE = 26,   // (ii) and (iii-b) complete
    B_KQFREE = 27,  // [2] chunk's KT/QT/KH/PP buffers free again
    B_OFREE = 29,   // D_O read out
    B_VFREE = 30,   // [2] vector buffers free again
    B_BFULL = 33,   // [4] beta of a chunk loaded (ring of 4, by chunk index mod 4)
    B_STG = 37,     // output staging tile written by the whole state warpgroup
    B_STGR = 38,    // output staging buffer free again (thread 0 -> state warpgroup)
    B_BFREE = 39,   // [4] beta ring slot read by all its users
    B_COUNT = 43
};

#ifdef KDA_TRACE
// Debug timeline (compiled only with -DKDA_TRACE): clock64 stamps of each
// role's milestones for the first 64 chunks of CTA 0.
constexpr int kTrEv = 40;
__device__ unsigned long long g_trace[64 * kTrEv];
#define KDA_TR(n, ev)                                                                                    \
    do {                                                                                                 \
        if (blockIdx.x == 0 && (n) < 64) g_trace[(n) * kTrEv + (ev)] = (unsigned long long)clock64(); \
    } while (0)
#else
#define KDA_TR(n, ev) \
    do {              \
    } while (0)
#endif

__device__ __forceinline__ float ld_in(const __nv_bfloat16* s, uint32_t idx) { return __bfloat162float(s[idx]); }
__device__ __forceinline__ float ld_in(const float* s, uint32_t idx) { return s[idx]; }

// Writes 64 fp32 values (r0: columns 0..31, r1: 32..63) as one 128-byte
// swizzled fp16 row.
__device__ __forceinline__ void store_row16(uint8_t* tile, uint32_t row, const uint32_t (&r0)[32],
                                            const uint32_t (&r1)[32]) {
#pragma unroll
    for (int c16 = 0; c16 < 8; ++c16) {
        const uint32_t* s = c16 < 4 ? &r0[8 * c16] : &r1[8 * (c16 - 4)];
        *reinterpret_cast<uint4*>(tile + sw128(row, c16)) =
            make_uint4(pack_half2(__uint_as_float(s[0]), __uint_as_float(s[1])),
                       pack_half2(__uint_as_float(s[2]), __uint_as_float(s[3])),
                       pack_half2(__uint_as_float(s[4]), __uint_as_float(s[5])),
                       pack_half2(__uint_as_float(s[6]), __uint_as_float(s[7])));
    }
}

// Adds the 16 values `d` to columns 16a .. 16a+15 of a 64-wide row held as (r0, r1).
__device__ __forceinline__ void add_block16(uint32_t (&r0)[32], uint32_t (&r1)[32], int a, const float* d) {
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const float dm = d[m];
#pragma unroll
        for (int aa = 0; aa < 4; ++aa)
            if (aa == a) {
                uint32_t& e = aa < 2 ? r0[16 * aa + m] : r1[16 * (aa - 2) + m];
                e = __float_as_uint(__uint_as_float(e) + dm);
            }
    }
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(NTHREADS, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_la,
                 const __grid_constant__ CUtensorMap tm_out, const SeqProblem P) {
    using L = Cfg<Tin>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::OFF_MISC);
    Abort* ab = reinterpret_cast<Abort*>(sm + L::OFF_MISC + 16);
    float* vec_a = reinterpret_cast<float*>(sm + L::OFF_VEC);         // [2][128]
    float* vec_b = reinterpret_cast<float*>(sm + L::OFF_VEC + 1024);  // [2][128]
    float* sbeta = reinterpret_cast<float*>(sm + L::OFF_BETA);        // [4][64]
    float* ldg = reinterpret_cast<float*>(sm + L::OFF_LDG);           // [4][16][17] diagonal blocks of A
    float* dfp = reinterpret_cast<float*>(sm + L::OFF_DFP);           // [4][16][16] their inverses

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const int h = unit % P.H, s = unit / P.H;
    int64_t t0, len;
    seq_bounds(P, s, t0, len);
    const int nch = (int)((len + C - 1) / C);
    const size_t sbase = ((size_t)s * P.H + h) * kD * kD;

    if (nch == 0) {  // empty sequence: the final state is the initial state
        if (P.final_state)
            for (int i = tid; i < kD * kD; i += NTHREADS) P.final_state[sbase + i] = P.init ? P.init[sbase + i] : 0.f;
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < L::NSLOT; ++i) {
            mbar_init(&bar[B_FULL + i], 1);
            mbar_init(&bar[B_EMPTY + i], 128);
        }
        const int c128[] = {B_PREPD, B_PREPD + 1, B_P2D, B_C1, B_C2, B_C3, B_TRDY, B_WRDY, B_XRDY, B_URDY,
                            B_OFREE, B_VFREE, B_VFREE + 1};
        for (int i : c128) mbar_init(&bar[i], 128);
        const int c1[] = {B_GDONE, B_S1D, B_S2D, B_S3D, B_TDONE, B_WYDONE, B_UIDONE, B_SDONE, B_KQFREE, B_KQFREE + 1};
        for (int i : c1) mbar_init(&bar[i], 1);
        mbar_init(&bar[B_AFREE], 64);
        mbar_init(&bar[B_DRDY], 64);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&bar[B_BFULL + i], 32);
            mbar_init(&bar[B_BFREE + i], 64 + 128);
        }
        mbar_init(&bar[B_STG], 128);
        mbar_init(&bar[B_STGR], 1);
        ab->flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    int* status = P.status;

    const uint32_t sm_base = smem_u32(sm);
    // MN-major operand: the stride between 64-element atoms along M/N goes in
    // the leading-byte-offset field, the 1024-byte stride between 8-row groups
    // in the stride field.  K-major operand: only the 8-row group stride.
    auto mn_desc = [&](uint32_t addr, uint32_t atom_stride) -> uint64_t { return sdesc(addr, atom_stride, 1024); };
    auto k_desc = [&](uint32_t addr) -> uint64_t { return sdesc(addr, 16, 1024); };
    constexpr uint32_t ID_G = idesc_f16(128, 64, 1, 1);
    constexpr uint32_t ID_MN = idesc_f16(128, 64, 0, 1);
    constexpr uint32_t ID_KK = idesc_f16(128, 64, 0, 0);
    constexpr uint32_t ID_S = idesc_f16(128, 128, 0, 0);
    constexpr uint32_t ID_T1 = idesc_f16(64, 64, 1, 1);
    constexpr uint32_t ID_T2 = idesc_f16(64, 64, 0, 1);
    constexpr uint32_t ID_T3 = idesc_f16(64, 64, 0, 0);
    const uint32_t sdt = sm_base + L::OFF_DT, sb1 = sm_base + L::OFF_B1, snr = sm_base + L::OFF_NR;
    // Every product group is issued by thread 0 of the role that completes its last
    // input, after waiting for that input and for the previous reader of its
    // accumulator; the commits below are what the other roles wait on.

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v); prefetch_tmap(&tm_la);
            prefetch_tmap(&tm_out);
            int issued = 0;
            bool ok = true;
            for (int n = 0; n < nch && ok; ++n)
                for (int q = 0; q < 4 && ok; ++q) {
                    const int g = 4 * n + q, sl = g % L::NSLOT, use = g / L::NSLOT;
                    if (use > 0 && !(ok = mbar_wait(&bar[B_EMPTY + sl], (use - 1) & 1, ab, status))) break;
                    uint8_t* slot = sm + L::OFF_RING + sl * L::SLOT_BYTES;
                    mbar_arrive_expect_tx(&bar[B_FULL + sl], L::SLOT_BYTES);
                    const int z = (int)(t0 + (int64_t)C * n + QR * q);
                    tma_load_3d(slot + L::SLOT_Q, &tm_q, &bar[B_FULL + sl], 0, h, z);
                    tma_load_3d(slot + L::SLOT_K, &tm_k, &bar[B_FULL + sl], 0, h, z);
                    tma_load_3d(slot + L::SLOT_V, &tm_v, &bar[B_FULL + sl], 0, h, z);
                    tma_load_3d(slot + L::SLOT_LA, &tm_la, &bar[B_FULL + sl], 0, h, z);
                    KDA_TR(n, 32 + q);
                    ++issued;
                }
            if (!ok) {  // let the copies already issued land before the CTA can exit
                for (int g = (issued > L::NSLOT ? issued - L::NSLOT : 0); g < issued; ++g) {
                    const long long tstart = clock64();
                    while (!mbar_try_wait(&bar[B_FULL + g % L::NSLOT], (g / L::NSLOT) & 1) &&
                           clock64() - tstart < kWaitCycles) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ beta loader
        // beta of chunk m into ring slot m % 4 (0 past the sequence end).  Plain loads in a
        // warp of their own, so that no other role's barrier arrive or proxy fence waits on
        // them.  (This warp also owns the TMEM allocation.)
        for (int m = 0; m < nch; ++m) {
            const int k4 = m & 3;
            if (m >= 4 && !mbar_wait(&bar[B_BFREE + k4], ((m - 4) >> 2) & 1, ab, status)) break;
            const int64_t vld = len - (int64_t)C * m;
            for (int i = lane; i < C; i += 32)
                sbeta[k4 * 64 + i] = i < vld ? P.beta[(size_t)(t0 + (int64_t)C * m + i) * P.H + h] : 0.f;
            mbar_arrive(&bar[B_BFULL + k4]);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ 16x16 diagonal-block inverses
        // Thread (a, jj) solves column jj of (I + A_aa)^-1 by right-looking substitution.
        const int t = tid - 64, a = t >> 4, jj = t & 15;
        const float* blk = ldg + a * 16 * 17;
        for (int n = 0; n < nch; ++n) {
            if (!mbar_wait(&bar[B_P2D], n & 1, ab, status)) break;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = 0.f;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float xr = (r == jj) ? 1.f : (r > jj ? x[r] : 0.f);
                x[r] = xr;
#pragma unroll
                for (int i = r + 1; i < 16; ++i) x[i] -= blk[i * 17 + r] * xr;
            }
            mbar_arrive(&bar[B_AFREE]);
            if (n > 0 && !mbar_wait(&bar[B_TRDY], (n - 1) & 1, ab, status)) break;
#pragma unroll
            for (int i = 0; i < 16; ++i) dfp[(a * 16 + i) * 16 + jj] = x[i];
            uint8_t* dt = sm + L::OFF_DT;  // row (16a + jj) holds column 16a+jj of Dg
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16) {
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (c16 == 2 * a)
                    w = make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]),
                                   pack_half2(x[6], x[7]));
                if (c16 == 2 * a + 1)
                    w = make_uint4(pack_half2(x[8], x[9]), pack_half2(x[10], x[11]), pack_half2(x[12], x[13]),
                                   pack_half2(x[14], x[15]));
                *reinterpret_cast<uint4*>(dt + sw128(16 * a + jj, c16)) = w;
            }
            fence_proxy_async_smem();
            mbar_arrive(&bar[B_DRDY]);
            KDA_TR(n, 7);
            if (t == 0) {  // S1: D_W = Dg A_o, once D_W's previous contents (W of chunk n-1) were read
                if (!mbar_wait(&bar[B_DRDY], n & 1, ab, status)) break;
                if (n > 0 && !mbar_wait(&bar[B_WRDY], (n - 1) & 1, ab, status)) break;
                tc_fence_after();
                for (int st = 0; st < 4; ++st)
                    mma_ss(tmem + TM_W, mn_desc(sdt + st * 2048, 8192), mn_desc(sb1 + st * 2048, 8192), ID_T1, st > 0);
                mma_commit(&bar[B_S1D]);
                KDA_TR(n, 12);
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ prep warpgroup
        const int c = tid - 128;  // key channel (and TMEM lane) of this thread
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        float max_x = 0.f;  // largest |g - ref| seen (log2 units), for the range check

        // prep1(n): decay cumsum, operand tiles KT/QT/KH, V16, vectors, beta.
        // Rows past the end of a sequence get log alpha = 0 and k = 0 (their beta
        // is 0 too), which makes them identity steps; q and v of such rows only
        // reach outputs that are never stored.
        auto prep1 = [&](int n) -> bool {
            const int b = n & 1;
            if (c == 0) KDA_TR(n, 0);
            if (n >= 2) {
                if (!mbar_wait(&bar[B_KQFREE + b], ((n - 2) >> 1) & 1, ab, status)) return false;
                if (!mbar_wait(&bar[B_VFREE + b], ((n - 2) >> 1) & 1, ab, status)) return false;
            }
            tc_fence_after();  // V16[b] was last read by the WY product of chunk n - 2
            const int valid = (int)((len - (int64_t)C * n) < C ? (len - (int64_t)C * n) : C);
            uint8_t* kt = sm + L::OFF_KQ + b * 32768;
            uint8_t* qt = kt + 16384;
            uint8_t* kh = sm + L::OFF_KH + b * 16384;
            auto slot_ptr = [&](int q) { return sm + L::OFF_RING + ((4 * n + q) % L::NSLOT) * L::SLOT_BYTES; };
            auto wait_slot = [&](int q) {
                const int g = 4 * n + q;
                return mbar_wait(&bar[B_FULL + g % L::NSLOT], (g / L::NSLOT) & 1, ab, status);
            };
            // pass A over rows 0..31: the reference ref = g_31
            if (!wait_slot(0) || !wait_slot(1)) return false;
            if (c == 0) KDA_TR(n, 1);
            float g2 = 0.f;
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const uint8_t* sl = slot_ptr(r >> 4);
                const float la = reinterpret_cast<const float*>(sl + L::SLOT_LA)[(r & 15) * 128 + c];
                g2 += (r < valid) ? la * kLog2e : 0.f;
            }
            const float ref = g2;
            // pass B, one 16-row quarter at a time
            g2 = 0.f;
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                if (q >= 2 && !wait_slot(q)) return false;
                if (c == 0) KDA_TR(n, 34 + q);
                const uint8_t* sl = slot_ptr(q);
                const float* sla = reinterpret_cast<const float*>(sl + L::SLOT_LA);
                const Tin* sk = reinterpret_cast<const Tin*>(sl + L::SLOT_K);
                const Tin* sq = reinterpret_cast<const Tin*>(sl + L::SLOT_Q);
                const Tin* sv = reinterpret_cast<const Tin*>(sl + L::SLOT_V);
                const int vq = valid - QR * q;  // rows of this quarter inside the sequence
                uint32_t pk[8], pq[8], ph[8], pv[8];
#pragma unroll
                for (int rp = 0; rp < QR / 2; ++rp) {
                    float kv2[2], qv2[2], hv2[2], vv2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int rr = 2 * rp + e;
                        const bool on = rr < vq;
                        const float la = on ? sla[rr * 128 + c] : 0.f;
                        const float kk = on ? ld_in(sk, rr * 128 + c) : 0.f;
                        const float qq = ld_in(sq, rr * 128 + c);
                        vv2[e] = ld_in(sv, rr * 128 + c);
                        g2 = fmaf(la, kLog2e, g2);
                        const float x = g2 - ref;
                        max_x = fmaxf(max_x, fabsf(x));
                        const float e1 = fast_exp2(x), e2 = fast_exp2(-x);
                        kv2[e] = kk * e1;
                        qv2[e] = qq * e1;
                        hv2[e] = kk * e2;
                    }
                    pk[rp] = pack_half2(kv2[0], kv2[1]);
                    pq[rp] = pack_half2(qv2[0], qv2[1]);
                    ph[rp] = pack_half2(hv2[0], hv2[1]);
                    pv[rp] = pack_half2(vv2[0], vv2[1]);
                }
                mbar_arrive(&bar[B_EMPTY + (4 * n + q) % L::NSLOT]);
#pragma unroll
                for (int g8 = 0; g8 < 2; ++g8) {
                    const uint32_t off = sw128(c, 2 * q + g8);
                    *reinterpret_cast<uint4*>(kt + off) = make_uint4(pk[4 * g8], pk[4 * g8 + 1], pk[4 * g8 + 2], pk[4 * g8 + 3]);
                    *reinterpret_cast<uint4*>(qt + off) = make_uint4(pq[4 * g8], pq[4 * g8 + 1], pq[4 * g8 + 2], pq[4 * g8 + 3]);
                    *reinterpret_cast<uint4*>(kh + off) = make_uint4(ph[4 * g8], ph[4 * g8 + 1], ph[4 * g8 + 2], ph[4 * g8 + 3]);
                }
                tmem_st8(tmem + lane_base + TM_V16 + b * 32 + q * 8, pv);
                if (c == 0) KDA_TR(n, 22 + q);
            }
            const float an = fast_exp2(ref);
            vec_a[b * 128 + c] = an;
            vec_b[b * 128 + c] = fast_exp2(g2 - ref);
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar[B_PREPD + b]);
            if (c == 0) {  // the Gram of this chunk, once all operand rows and D_G (read by P2(n-1)) are ready
                KDA_TR(n, 2);
                if (!mbar_wait(&bar[B_PREPD + b], (n >> 1) & 1, ab, status)) return false;
                if (n > 0 && !mbar_wait(&bar[B_P2D], (n - 1) & 1, ab, status)) return false;
                tc_fence_after();
                const uint32_t kq = sm_base + L::OFF_KQ + b * 32768, khb = sm_base + L::OFF_KH + b * 16384;
                for (int st = 0; st < 8; ++st)
                    mma_ss(tmem + TM_G, mn_desc(kq + st * 2048, 16384), mn_desc(khb + st * 2048, 8192), ID_G, st > 0);
                mma_commit(&bar[B_GDONE]);
                KDA_TR(n, 8);
            }
            return true;
        };
        // P2(n): read the Gram accumulator.  Rows 0..63 (A, beta_r applied): the
        // 16x16 diagonal blocks (fp32) and A_o (fp16); rows 64..127: P (fp16).
        auto p2 = [&](int n) -> bool {
            const int b = n & 1;
            if (!mbar_wait(&bar[B_GDONE], n & 1, ab, status)) return false;
            if (!mbar_wait(&bar[B_BFULL + (n & 3)], (n >> 2) & 1, ab, status)) return false;
            tc_fence_after();
            if (c == 0) KDA_TR(n, 3);
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + lane_base + TM_G, r0);
            tmem_ld32(tmem + lane_base + TM_G + 32, r1);
            tmem_ld_wait();
            if (c == 0) KDA_TR(n, 29);
            if (c < 64) {  // row r = c of A
                if (n > 0) {
                    if (!mbar_wait(&bar[B_AFREE], (n - 1) & 1, ab, status)) return false;
                    if (!mbar_wait(&bar[B_TDONE], (n - 1) & 1, ab, status)) return false;
                }

                const float br = c < len - (int64_t)C * n ? sbeta[(n & 3) * 64 + c] : 0.f;
                const int a = c >> 4, i = c & 15;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    r0[e] = __float_as_uint(e < c ? br * __uint_as_float(r0[e]) : 0.f);
                    r1[e] = __float_as_uint(e + 32 < c ? br * __uint_as_float(r1[e]) : 0.f);
                }
                // row i of diagonal block a: columns 16a .. 16a+15
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    float v = 0.f;
#pragma unroll
                    for (int aa = 0; aa < 4; ++aa)
                        if (aa == a) v = __uint_as_float(aa < 2 ? r0[16 * aa + m] : r1[16 * (aa - 2) + m]);
                    ldg[(a * 16 + i) * 17 + m] = v;
                }

                mbar_arrive(&bar[B_BFREE + (n & 3)]);
                // A_o: keep the columns left of the diagonal block
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    if (e >= 16 * a) r0[e] = 0u;
                    if (e + 32 >= 16 * a) r1[e] = 0u;
                }
                store_row16(sm + L::OFF_B1, c, r0, r1);
                if (c == 0) KDA_TR(n, 26);
            } else {  // row r = c - 64 of P (lower triangle including the diagonal)
                if (n >= L::NPP) {
                    const int m = n - L::NPP;
                    if (!mbar_wait(&bar[B_KQFREE + (m & 1)], (m >> 1) & 1, ab, status)) return false;
                }
                const int r = c - 64;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    if (e > r) r0[e] = 0u;
                    if (e + 32 > r) r1[e] = 0u;
                }
                store_row16(sm + L::OFF_PP + (n % L::NPP) * 8192, r, r0, r1);
            }
            fence_proxy_async_smem();
            if (c == 0) KDA_TR(n, 27);
            tc_fence_before();
            mbar_arrive(&bar[B_P2D]);
            if (c == 0) KDA_TR(n, 4);
            return true;
        };
        for (int n = 0; n < nch; ++n)
            if (!prep1(n) || !p2(n)) break;
        if (max_x > kMaxExp2) atomicCAS(status, 0, (int)KDA_STATUS_GATE_RANGE);
    } else if (warp < 12) {
        // ------------------------------------------------------------ state warpgroup
        const int j = tid - 256;  // value column (and TMEM lane) of this thread
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        Tout* out = static_cast<Tout*>(P.out);
        bool ok = true;
        // Staging buffer hand-offs within the warpgroup (every thread follows the same
        // sequence, so the phase counters agree).  Thread 0 owns the bulk stores.
        uint32_t ph_stg = 0, ph_rd = 0;
        auto staging_free = [&](bool all_read) -> bool {  // wait until WT may be rewritten
            if (j == 0) {
                if (all_read) bulk_wait_read<0>(); else bulk_wait_read<1>();
                mbar_arrive(&bar[B_STGR]);
            }
            return mbar_wait(&bar[B_STGR], (ph_rd++) & 1, ab, status);
        };
        {  // X_0 = Diag(a_0) S_0 into D_S and X16
            if (!(ok = mbar_wait(&bar[B_PREPD], 0, ab, status))) goto state_done;
#pragma unroll 1
            for (int piece = 0; piece < 4; ++piece) {
                uint32_t xs[32], x16[16];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int cc = piece * 32 + e;
                    const float s0 = P.init ? P.init[sbase + (size_t)cc * kD + j] : 0.f;
                    xs[e] = __float_as_uint(s0 * vec_a[cc]);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    x16[e] = pack_half2(__uint_as_float(xs[2 * e]), __uint_as_float(xs[2 * e + 1]));
                tmem_st32(tmem + lane_base + TM_S + piece * 32, xs);
                tmem_st16(tmem + lane_base + TM_X16 + piece * 16, x16);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar[B_XRDY]);
        }
        for (int n = 0; n < nch; ++n) {
            const int b = n & 1;
            const int valid = (int)((len - (int64_t)C * n) < C ? (len - (int64_t)C * n) : C);
            // P4(n): WT = -W^T as fp16 (WT also stages the previous chunk's outputs)
            if (!(ok = staging_free(true))) break;
            if (!(ok = mbar_wait(&bar[B_WYDONE], n & 1, ab, status))) break;
            tc_fence_after();
            if (j == 0) KDA_TR(n, 16);
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lane_base + TM_W, r0);
                tmem_ld32(tmem + lane_base + TM_W + 32, r1);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    r0[e] ^= 0x80000000u;
                    r1[e] ^= 0x80000000u;
                }
                store_row16(sm + L::OFF_WT, j, r0, r1);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bar[B_WRDY]);
                if (j == 0) {  // C: U = U' - W S0 and O = Qtil S0
                    KDA_TR(n, 17);
                    if (!(ok = mbar_wait(&bar[B_WRDY], n & 1, ab, status))) break;
                    if (!(ok = mbar_wait(&bar[B_XRDY], n & 1, ab, status))) break;
                    if (n > 0 && !(ok = mbar_wait(&bar[B_OFREE], (n - 1) & 1, ab, status))) break;
                    tc_fence_after();
                    const uint32_t wt = sm_base + L::OFF_WT, qt = sm_base + L::OFF_KQ + (n & 1) * 32768 + 16384;
                    for (int st = 0; st < 8; ++st)
                        mma_ts(tmem + TM_U, tmem + TM_X16 + st * 8, mn_desc(wt + st * 2048, 8192), ID_MN, 1);
                    for (int st = 0; st < 8; ++st)
                        mma_ts(tmem + TM_O, tmem + TM_X16 + st * 8, mn_desc(qt + st * 2048, 8192), ID_MN, st > 0);
                    mma_commit(&bar[B_UIDONE]);
                    KDA_TR(n, 10);
                }
            }
            // S2(n): U16 = fp16(U^T)
            if (!(ok = mbar_wait(&bar[B_UIDONE], n & 1, ab, status))) break;
            tc_fence_after();
            if (j == 0) KDA_TR(n, 18);
            {
                uint32_t r0[32], r1[32], u16[32];
                tmem_ld32(tmem + lane_base + TM_U, r0);
                tmem_ld32(tmem + lane_base + TM_U + 32, r1);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    u16[e] = pack_half2(__uint_as_float(r0[2 * e]), __uint_as_float(r0[2 * e + 1]));
                    u16[16 + e] = pack_half2(__uint_as_float(r1[2 * e]), __uint_as_float(r1[2 * e + 1]));
                }
                tmem_st32(tmem + lane_base + TM_U16, u16);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bar[B_URDY]);
                if (j == 0) {  // D: state update and the intra-chunk part of the output
                    if (!(ok = mbar_wait(&bar[B_URDY], n & 1, ab, status))) break;
                    tc_fence_after();
                    const uint32_t kh = sm_base + L::OFF_KH + b * 16384, pp = sm_base + L::OFF_PP + (n % L::NPP) * 8192;
                    for (int st = 0; st < 4; ++st)
                        mma_ts(tmem + TM_S, tmem + TM_U16 + st * 8, k_desc(kh + st * 32), ID_S, 1);
                    for (int st = 0; st < 4; ++st)
                        mma_ts(tmem + TM_O, tmem + TM_U16 + st * 8, k_desc(pp + st * 32), ID_KK, 1);
                    mma_commit(&bar[B_SDONE]);
                    mma_commit(&bar[B_KQFREE + b]);
                    KDA_TR(n, 11);
                }
                if (j == 0) KDA_TR(n, 19);
            }
            // S3(n): outputs and state.  Order: rows 0..31 of the output (staged and
            // stored), the state (snapshots, next X: the chain continues from there),
            // then rows 32..63.  No 32-wide register array stays live across the state
            // update, which keeps it free of register spills.
            if (!(ok = mbar_wait(&bar[B_SDONE], n & 1, ab, status))) break;
            tc_fence_after();
            if (j == 0) KDA_TR(n, 20);
            constexpr uint32_t QB = QR * kD * sizeof(Tout);  // one 16-row output quarter
            const bool full = valid == C;
            // Writes rows 32*half .. 32*half+31 of the output: staged through WT and
            // stored by bulk tensor copies for full chunks, plain stores otherwise.
            auto emit_half = [&](const uint32_t (&o)[32], int half) -> bool {
                if (!full) {
                    const size_t obase = ((size_t)(t0 + (int64_t)C * n) * P.H + h) * kD + j;
                    const size_t ostride = (size_t)P.H * kD;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int r = 32 * half + e;
                        if (r < valid) {
                            if constexpr (sizeof(Tout) == 2)
                                out[obase + r * ostride] = __float2bfloat16_rn(__uint_as_float(o[e]));
                            else
                                out[obase + r * ostride] = __uint_as_float(o[e]);
                        }
                    }
                    return true;
                }
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const int q = 2 * half + qq;
                    Tout* buf = reinterpret_cast<Tout*>(sm + L::OFF_WT + qq * QB);
                    if (half == 1 && !staging_free(false)) return false;
#pragma unroll
                    for (int rr = 0; rr < QR; ++rr) {
                        const float v = __uint_as_float(o[QR * qq + rr]);
                        if constexpr (sizeof(Tout) == 2)
                            buf[rr * kD + j] = __float2bfloat16_rn(v);
                        else
                            buf[rr * kD + j] = v;
                    }
                    // Every thread waits, so no thread can arrive for the next quarter
                    // before all have arrived for this one.
                    fence_proxy_async_smem();
                    mbar_arrive(&bar[B_STG]);
                    if (!mbar_wait(&bar[B_STG], (ph_stg++) & 1, ab, status)) return false;
                    if (j == 0) {
                        tma_store_3d(&tm_out, buf, 0, h, (int)(t0 + (int64_t)C * n + QR * q));
                        bulk_commit();
                    }
                }
                return true;
            };
            {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + TM_O, o);
                tmem_ld_wait();
                if (!(ok = emit_half(o, 0))) break;
            }
            if (j == 0) KDA_TR(n, 5);
            {
                const bool last = (n + 1 == nch);
                const int64_t end_pos = (int64_t)C * n + valid;  // tokens of the sequence consumed so far
                float* snap = nullptr;
                if (P.snap_interval > 0 && full && end_pos % P.snap_interval == 0)
                    snap = P.snapshots + ((size_t)(P.snap_offsets[s] + end_pos / P.snap_interval - 1) * P.H + h) *
                                             kD * kD;
                float* fin = (last && P.final_state) ? P.final_state + sbase : nullptr;
                if (!last && !(ok = mbar_wait(&bar[B_PREPD + ((n + 1) & 1)], ((n + 1) >> 1) & 1, ab, status)))
                    break;
                const float* bv = vec_b + b * 128;
                if (snap || fin) {  // true state S = Diag(b_n) D, at snapshot positions and the end
#pragma unroll 1
                    for (int piece = 0; piece < 4; ++piece) {
                        uint32_t d[32];
                        tmem_ld32(tmem + lane_base + TM_S + piece * 32, d);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int cc = piece * 32 + e;
                            const float sv = __uint_as_float(d[e]) * bv[cc];
                            if (snap) snap[(size_t)cc * kD + j] = sv;
                            if (fin) fin[(size_t)cc * kD + j] = sv;
                        }
                    }
                }
                if (!last) {  // X_{n+1} = Diag(a_{n+1}) (Diag(b_n) D) into D_S (fp32) and X16 (fp16)
                    // (the same two roundings as a run resumed from the returned state)
                    const float* an = vec_a + ((n + 1) & 1) * 128;
                    uint32_t da[32], db[32];
                    tmem_ld32(tmem + lane_base + TM_S, da);
                    tmem_ld_wait();
#pragma unroll
                    for (int piece = 0; piece < 4; ++piece) {
                        uint32_t(&d)[32] = (piece & 1) ? db : da;
                        uint32_t(&dn)[32] = (piece & 1) ? da : db;
                        if (piece < 3) tmem_ld32(tmem + lane_base + TM_S + (piece + 1) * 32, dn);
                        uint32_t x16[16];
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            d[e] = __float_as_uint(__uint_as_float(d[e]) * bv[piece * 32 + e] * an[piece * 32 + e]);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            x16[e] = pack_half2(__uint_as_float(d[2 * e]), __uint_as_float(d[2 * e + 1]));
                        tmem_st32(tmem + lane_base + TM_S + piece * 32, d);
                        tmem_st16(tmem + lane_base + TM_X16 + piece * 16, x16);
                        if (piece < 3) tmem_ld_wait();
                    }
                }
                if (j == 0) KDA_TR(n, 30);
                if (!last) {
                    tmem_st_wait();
                    if (j == 0) KDA_TR(n, 31);
                    tc_fence_before();
                    mbar_arrive(&bar[B_XRDY]);
                }
                mbar_arrive(&bar[B_VFREE + b]);
                if (j == 0) KDA_TR(n, 21);
            }
            {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + TM_O + 32, o);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&bar[B_OFREE]);
                if (!(ok = emit_half(o, 1))) break;
            }
            if (j == 0) KDA_TR(n, 28);
        }
        if (j == 0) bulk_wait_all();  // the CTA's shared memory must outlive the bulk stores
    state_done:;
    } else {
        // ------------------------------------------------------------ tri warpgroup
        // Reads the four M = 64 products of the inverse (row r of a product sits in
        // TMEM lane 32*(r/16) + r%16, so lanes 0..15 of each warp hold rows).
        const int q = warp & 3, r = 16 * q + (lane & 15);
        const bool act = lane < 16;
        const int a = r >> 4;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        uint8_t* b1 = sm + L::OFF_B1;
        uint8_t* nr = sm + L::OFF_NR;
        const float* dblk = dfp + r * 16;  // row r of its 16x16 diagonal inverse block
        for (int n = 0; n < nch; ++n) {
            uint32_t r0[32], r1[32];
            // readout 1: N -> NR
            if (!mbar_wait(&bar[B_S1D], n & 1, ab, status)) break;
            tc_fence_after();
            tmem_ld32(tmem + lane_base + TM_W, r0);
            tmem_ld32(tmem + lane_base + TM_W + 32, r1);
            tmem_ld_wait();
            if (act) store_row16(nr, r, r0, r1);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar[B_C1]);
            if (tid == 384) {  // S2: D_W = N N
                if (!mbar_wait(&bar[B_C1], n & 1, ab, status)) break;
                tc_fence_after();
                for (int st = 0; st < 4; ++st)
                    mma_ss(tmem + TM_W, k_desc(snr + st * 32), mn_desc(snr + st * 2048, 8192), ID_T2, st > 0);
                mma_commit(&bar[B_S2D]);
                KDA_TR(n, 13);
            }
            // readout 2: N2 -> B1
            if (!mbar_wait(&bar[B_S2D], n & 1, ab, status)) break;
            tc_fence_after();
            tmem_ld32(tmem + lane_base + TM_W, r0);
            tmem_ld32(tmem + lane_base + TM_W + 32, r1);
            tmem_ld_wait();
            if (act) store_row16(b1, r, r0, r1);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar[B_C2]);
            if (tid == 384) {  // S3: D_W = N2 Dg
                if (!mbar_wait(&bar[B_C2], n & 1, ab, status)) break;
                tc_fence_after();
                for (int st = 0; st < 4; ++st)
                    mma_ss(tmem + TM_W, k_desc(sb1 + st * 32), k_desc(sdt + st * 32), ID_T3, st > 0);
                mma_commit(&bar[B_S3D]);
                KDA_TR(n, 14);
            }
            // readout 3: M = Dg + N2 Dg; -M -> B1
            if (!mbar_wait(&bar[B_S3D], n & 1, ab, status)) break;
            tc_fence_after();
            tmem_ld32(tmem + lane_base + TM_W, r0);
            tmem_ld32(tmem + lane_base + TM_W + 32, r1);
            tmem_ld_wait();
            if (act) {
                add_block16(r0, r1, a, dblk);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    r0[e] ^= 0x80000000u;
                    r1[e] ^= 0x80000000u;
                }
                store_row16(b1, r, r0, r1);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar[B_C3]);
            if (tid == 384) {  // S4: D_W += N (-M)
                if (!mbar_wait(&bar[B_C3], n & 1, ab, status)) break;
                tc_fence_after();
                for (int st = 0; st < 4; ++st)
                    mma_ss(tmem + TM_W, k_desc(snr + st * 32), mn_desc(sb1 + st * 2048, 8192), ID_T2, 1);
                mma_commit(&bar[B_TDONE]);
                KDA_TR(n, 15);
            }
            // readout 4: T = Dg + (N2 Dg - N M); T diag(beta) -> NR (K-major B of the WY products)
            if (!mbar_wait(&bar[B_TDONE], n & 1, ab, status)) break;
            tc_fence_after();
            tmem_ld32(tmem + lane_base + TM_W, r0);
            tmem_ld32(tmem + lane_base + TM_W + 32, r1);
            tmem_ld_wait();
            if (!mbar_wait(&bar[B_BFULL + (n & 3)], (n >> 2) & 1, ab, status)) break;
            if (act) {
                add_block16(r0, r1, a, dblk);
                const float* bt = sbeta + (n & 3) * 64;
                const int64_t vld = len - (int64_t)C * n;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    r0[e] = __float_as_uint(e < vld ? __uint_as_float(r0[e]) * bt[e] : 0.f);
                    r1[e] = __float_as_uint(e + 32 < vld ? __uint_as_float(r1[e]) * bt[e + 32] : 0.f);
                }
                store_row16(nr, r, r0, r1);
            }
            mbar_arrive(&bar[B_BFREE + (n & 3)]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar[B_TRDY]);
            KDA_TR(n, 6);
            if (tid == 384) {  // WY products, once U16 of chunk n-1 (over D_U) has been consumed
                if (!mbar_wait(&bar[B_TRDY], n & 1, ab, status)) break;
                if (!mbar_wait(&bar[B_PREPD + (n & 1)], (n >> 1) & 1, ab, status)) break;
                if (n > 0 && !mbar_wait(&bar[B_SDONE], (n - 1) & 1, ab, status)) break;
                tc_fence_after();
                const uint32_t kt = sm_base + L::OFF_KQ + (n & 1) * 32768, v16 = TM_V16 + (n & 1) * 32;
                for (int st = 0; st < 4; ++st) {
                    const uint64_t bd = k_desc(snr + st * 32);
                    mma_ss(tmem + TM_W, k_desc(kt + st * 32), bd, ID_KK, st > 0);
                    mma_ts(tmem + TM_U, tmem + v16 + st * 8, bd, ID_KK, st > 0);
                }
                mma_commit(&bar[B_WYDONE]);
                KDA_TR(n, 9);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (ab->flag) {  // aborted: let any product group still in flight drain before TMEM goes away
        const long long tstart = clock64();
        while (clock64() - tstart < 2000000) {
        }
    }
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [T_total][H][128] token-major tensor, box = 16 tokens x 1 head x 128 channels.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int es, int64_t T_total, int H) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T_total};
    cuuint64_t strides[2] = {(cuuint64_t)kD * es, (cuuint64_t)kD * es * H};
    cuuint32_t box[3] = {(cuuint32_t)kD, 1, (cuuint32_t)QR};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Tin, typename Tout>
cudaError_t launch_t(const SeqProblem& p, cudaStream_t st) {
    CUtensorMap mq, mk, mv, ml, mo;
    const CUtensorMapDataType dt = sizeof(Tin) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int64_t Tt = p.T_total > 0 ? p.T_total : 1;
    if (Tt > (int64_t)0x7FFFFFFF - 2 * C) return cudaErrorInvalidValue;  // tensor-map coordinates are 32-bit
    if (!make_map(&mq, p.q, dt, sizeof(Tin), Tt, p.H) || !make_map(&mk, p.k, dt, sizeof(Tin), Tt, p.H) ||
        !make_map(&mv, p.v, dt, sizeof(Tin), Tt, p.H) ||
        !make_map(&ml, p.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Tt, p.H) ||
        !make_map(&mo, p.out, sizeof(Tout) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  sizeof(Tout), Tt, p.H))
        return cudaErrorInvalidValue;
    auto kern = chunk_kernel<Tin, Tout>;
    const int smem = (int)Cfg<Tin>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((int64_t)p.N * p.H);
    kern<<<grid, NTHREADS, smem, st>>>(mq, mk, mv, ml, mo, p);
    return cudaGetLastError();
}

}  // namespace

#ifdef KDA_TRACE
extern "C" int kda_trace_read(unsigned long long* host, int n) {
    const size_t cnt = (size_t)(n < 64 * kTrEv ? n : 64 * kTrEv);
    return cudaMemcpyFromSymbol(host, g_trace, sizeof(unsigned long long) * cnt) == cudaSuccess ? 0 : 1;
}
#endif

size_t chunk_prefill_workspace(int N, int H) {
    (void)N;
    (void)H;
    return 0;
}

cudaError_t launch_chunk_prefill(const SeqProblem& p, int in_dtype, int out_dtype, void* workspace,
                                 size_t ws_bytes, cudaStream_t st) {
    (void)workspace;
    (void)ws_bytes;
    if ((int64_t)p.N * p.H == 0) return cudaSuccess;
    if (in_dtype == KDA_BF16 && out_dtype == KDA_BF16) return launch_t<__nv_bfloat16, __nv_bfloat16>(p, st);
    if (in_dtype == KDA_BF16) return launch_t<__nv_bfloat16, float>(p, st);
    if (out_dtype == KDA_BF16) return launch_t<float, __nv_bfloat16>(p, st);
    return launch_t<float, float>(p, st);
}

}  // namespace kda
