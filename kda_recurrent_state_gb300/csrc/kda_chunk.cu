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
// Data layout on chip (one CTA = one (sequence, head), all of d_v = 128):
//   TMEM (fp32 accumulators, lanes = the M rows):
//     D_S [j][c] state (128 cols)   X16 [j][c] fp16 A operand   D_U [j][r] U'/U
//     U16 [j][r] fp16 A operand     D_O [j][r] output           D_G [r|64+r][i] Gram
//     D_W [c][r] W^T                V16 [j][i] fp16 A operand (v^T)
//   SMEM (fp16, 128-byte swizzled rows of 64 elements):
//     KT[c][r] = Ktil_p, QT[c][r] = Qtil_p (adjacent: together the M = 128 A
//     operand of the Gram), KH[c][r] = Khat_p, PP[r][i] = P, TT[i][r] =
//     T[r][i] beta_i, WT[c][r] = -W^T; a ring of 16-token input slots (TMA).
//   Every product is one M = 128 tcgen05.mma chain:
//     Gram  D_G = [KT;QT] (MN-major) x KH (MN-major)        128x64x128
//     WY    D_W = KT (K-major) x TT (MN-major)               128x64x64
//           D_U = V16 (TMEM) x TT                            128x64x64
//     (i)   D_U += X16 x WT (MN-major)                       128x64x128
//     (iii) D_O = X16 x QT (MN-major) + U16 x PP (K-major)   128x64x192
//     (ii)  D_S += U16 x KH (K-major)                        128x128x64
//
// Warp roles (12 warps): 0 TMA producer, 1 MMA issuer (+ TMEM allocation),
// 2-3 triangular solve (one column of T per thread), 4-7 "prep" warpgroup
// (decay cumsum, operand tiles, Gram readout), 8-11 "state" warpgroup (W
// conversion, U conversion, outputs, state rescale, snapshots).  Roles hand
// work to each other through mbarriers; every wait is bounded.
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {
using namespace sm100;

constexpr int C = 64;     // chunk length
constexpr int QR = 16;    // token rows per input slot
constexpr int NTHREADS = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxExp2 = 15.0f;  // |g - ref| bound (log2 units) for fp16 operands

// TMEM column map (512 columns allocated)
constexpr uint32_t TM_S = 0, TM_X16 = 128, TM_U = 192, TM_U16 = 256, TM_O = 288, TM_G = 352, TM_W = 416,
                   TM_V16 = 480;

// MN-major descriptors: which field carries the stride between 64-element
// atoms along M/N (the other carries the 1024-byte stride between 8-row groups).
constexpr bool kMnAtomInLbo = true;

template <typename Tin>
struct Cfg {
    static constexpr int ES = sizeof(Tin);
    static constexpr int NSLOT = ES == 2 ? 3 : 2;
    static constexpr uint32_t SLOT_Q = 0;
    static constexpr uint32_t SLOT_K = QR * 128 * ES;
    static constexpr uint32_t SLOT_V = 2 * QR * 128 * ES;
    static constexpr uint32_t SLOT_LA = 3 * QR * 128 * ES;
    static constexpr uint32_t SLOT_BYTES = 3 * QR * 128 * ES + QR * 128 * 4;
    // shared memory map (offsets from a 1024-byte aligned base)
    static constexpr uint32_t OFF_KQ = 0;            // [2] x (KT 16K | QT 16K)
    static constexpr uint32_t OFF_KH = 65536;        // [2] x 16K
    static constexpr uint32_t OFF_PP = 98304;        // [2] x 8K
    static constexpr uint32_t OFF_TT = 114688;       // 8K
    static constexpr uint32_t OFF_WT = 122880;       // 16K
    static constexpr uint32_t OFF_AS = 139264;       // fp32 [64][68]
    static constexpr uint32_t AS_STRIDE = 68;
    static constexpr uint32_t OFF_RING = OFF_AS + 64 * AS_STRIDE * 4;  // 156672
    static constexpr uint32_t OFF_VEC = OFF_RING + NSLOT * SLOT_BYTES;  // a[2][128], b[2][128]
    static constexpr uint32_t OFF_BETA = OFF_VEC + 4 * 128 * 4;         // [2][64]
    static constexpr uint32_t OFF_BAR = OFF_BETA + 2 * 64 * 4;
    static constexpr uint32_t NBAR = 64;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
};
static_assert(Cfg<__nv_bfloat16>::SMEM_BYTES <= 232448, "smem budget (bf16)");
static_assert(Cfg<float>::SMEM_BYTES <= 232448, "smem budget (fp32)");

// barrier indices
enum {
    B_FULL = 0,       // [NSLOT] (up to 3)
    B_EMPTY = 4,      // [NSLOT]
    B_PREPD = 8,      // [2] prep outputs (KT/QT/KH, vectors, beta) of a chunk ready
    B_VRDY = 10,      // V16 written
    B_GDONE = 11,     // Gram complete
    B_P2D = 12,       // Gram read out (A scratch, PP written; D_G free)
    B_AFREE = 13,     // solver finished reading the A scratch
    B_TRDY = 14,      // TT written
    B_WYDONE = 15,    // WY products complete
    B_WRDY = 16,      // WT written, D_W free
    B_XRDY = 17,      // X16 / D_S ready for the chunk
    B_UIDONE = 18,    // (i) and (iii-a) complete
    B_URDY = 19,      // U16 written, D_U free
    B_SDONE = 20,     // (ii) and (iii-b) complete
    B_KQFREE = 21,    // [2] chunk's KT/QT/KH/PP buffers free again
    B_OFREE = 23,     // D_O read out
    B_VFREE = 24,     // [2] vector buffers free again
    B_DRAIN = 26,     // MMA drain on abort
    B_COUNT = 27
};


__device__ __forceinline__ float ld_in(const __nv_bfloat16* s, uint32_t idx) { return __bfloat162float(s[idx]); }
__device__ __forceinline__ float ld_in(const float* s, uint32_t idx) { return s[idx]; }

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(NTHREADS, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_la,
                 const SeqProblem P) {
    using L = Cfg<Tin>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::OFF_MISC);
    Abort* ab = reinterpret_cast<Abort*>(sm + L::OFF_MISC + 16);
    float* vec_a = reinterpret_cast<float*>(sm + L::OFF_VEC);            // [2][128]
    float* vec_b = reinterpret_cast<float*>(sm + L::OFF_VEC + 1024);     // [2][128]
    float* sbeta = reinterpret_cast<float*>(sm + L::OFF_BETA);           // [2][64]
    float* ascr = reinterpret_cast<float*>(sm + L::OFF_AS);

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
        mbar_init(&bar[B_PREPD], 128);
        mbar_init(&bar[B_PREPD + 1], 128);
        mbar_init(&bar[B_VRDY], 128);
        mbar_init(&bar[B_GDONE], 1);
        mbar_init(&bar[B_P2D], 128);
        mbar_init(&bar[B_AFREE], 64);
        mbar_init(&bar[B_TRDY], 64);
        mbar_init(&bar[B_WYDONE], 1);
        mbar_init(&bar[B_WRDY], 128);
        mbar_init(&bar[B_XRDY], 128);
        mbar_init(&bar[B_UIDONE], 1);
        mbar_init(&bar[B_URDY], 128);
        mbar_init(&bar[B_SDONE], 1);
        mbar_init(&bar[B_KQFREE], 1);
        mbar_init(&bar[B_KQFREE + 1], 1);
        mbar_init(&bar[B_OFREE], 128);
        mbar_init(&bar[B_VFREE], 128);
        mbar_init(&bar[B_VFREE + 1], 128);
        mbar_init(&bar[B_DRAIN], 1);
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
    auto mn_desc = [&](uint32_t addr, uint32_t atom_stride) -> uint64_t {
        return kMnAtomInLbo ? sdesc(addr, atom_stride, 1024) : sdesc(addr, 1024, atom_stride);
    };
    auto k_desc = [&](uint32_t addr) -> uint64_t { return sdesc(addr, 16, 1024); };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v); prefetch_tmap(&tm_la);
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
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_G = idesc_f16(128, 64, 1, 1);
            constexpr uint32_t ID_MN = idesc_f16(128, 64, 0, 1);
            constexpr uint32_t ID_S = idesc_f16(128, 128, 0, 0);
            constexpr uint32_t ID_P = idesc_f16(128, 64, 0, 0);
            auto gram = [&](int n) {
                const uint32_t kq = sm_base + L::OFF_KQ + (n & 1) * 32768, kh = sm_base + L::OFF_KH + (n & 1) * 16384;
                for (int st = 0; st < 8; ++st)
                    mma_ss(tmem + TM_G, mn_desc(kq + st * 2048, 16384), mn_desc(kh + st * 2048, 8192), ID_G, st > 0);
                mma_commit(&bar[B_GDONE]);
            };
            bool ok = mbar_wait(&bar[B_PREPD], 0, ab, status);
            if (ok) { tc_fence_after(); gram(0); }
            for (int n = 0; n < nch && ok; ++n) {
                const int b = n & 1;
                // B(n): Gram of the next chunk
                if (n + 1 < nch) {
                    if (!(ok = mbar_wait(&bar[B_PREPD + ((n + 1) & 1)], ((n + 1) >> 1) & 1, ab, status))) break;
                    if (!(ok = mbar_wait(&bar[B_P2D], n & 1, ab, status))) break;
                    tc_fence_after();
                    gram(n + 1);
                }
                // A(n): WY products
                if (!(ok = mbar_wait(&bar[B_TRDY], n & 1, ab, status))) break;
                if (!(ok = mbar_wait(&bar[B_VRDY], n & 1, ab, status))) break;
                tc_fence_after();
                {
                    const uint32_t kt = sm_base + L::OFF_KQ + b * 32768, tt = sm_base + L::OFF_TT;
                    for (int st = 0; st < 4; ++st) {
                        const uint64_t bd = mn_desc(tt + st * 2048, 8192);
                        mma_ss(tmem + TM_W, k_desc(kt + st * 32), bd, ID_MN, st > 0);
                        mma_ts(tmem + TM_U, tmem + TM_V16 + st * 8, bd, ID_MN, st > 0);
                    }
                    mma_commit(&bar[B_WYDONE]);
                }
                // C(n): U = U' - W S0 and O = Qtil S0
                if (!(ok = mbar_wait(&bar[B_WRDY], n & 1, ab, status))) break;
                if (!(ok = mbar_wait(&bar[B_XRDY], n & 1, ab, status))) break;
                if (n > 0 && !(ok = mbar_wait(&bar[B_OFREE], (n - 1) & 1, ab, status))) break;
                tc_fence_after();
                {
                    const uint32_t wt = sm_base + L::OFF_WT, qt = sm_base + L::OFF_KQ + b * 32768 + 16384;
                    for (int st = 0; st < 8; ++st)
                        mma_ts(tmem + TM_U, tmem + TM_X16 + st * 8, mn_desc(wt + st * 2048, 8192), ID_MN, 1);
                    for (int st = 0; st < 8; ++st)
                        mma_ts(tmem + TM_O, tmem + TM_X16 + st * 8, mn_desc(qt + st * 2048, 8192), ID_MN, st > 0);
                    mma_commit(&bar[B_UIDONE]);
                }
                // D(n): state update and the intra-chunk part of the output
                if (!(ok = mbar_wait(&bar[B_URDY], n & 1, ab, status))) break;
                tc_fence_after();
                {
                    const uint32_t kh = sm_base + L::OFF_KH + b * 16384, pp = sm_base + L::OFF_PP + b * 8192;
                    for (int st = 0; st < 4; ++st)
                        mma_ts(tmem + TM_S, tmem + TM_U16 + st * 8, k_desc(kh + st * 32), ID_S, 1);
                    for (int st = 0; st < 4; ++st)
                        mma_ts(tmem + TM_O, tmem + TM_U16 + st * 8, k_desc(pp + st * 32), ID_P, 1);
                    mma_commit(&bar[B_SDONE]);
                    mma_commit(&bar[B_KQFREE + b]);
                }
            }
            if (!ok) {  // wait for every MMA already issued before the CTA can release TMEM
                mma_commit(&bar[B_DRAIN]);
                const long long tstart = clock64();
                while (!mbar_try_wait(&bar[B_DRAIN], 0) && clock64() - tstart < kWaitCycles) {
                }
            }
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ triangular solve
        // Thread j owns column j of T = (I + A)^-1 (A strictly lower triangular):
        // x_j = 1, x_r = -sum_{i<r} A[r][i] x_i for r > j, x_r = 0 for r < j.
        const int j = tid - 64;
        for (int n = 0; n < nch; ++n) {
            if (!mbar_wait(&bar[B_P2D], n & 1, ab, status)) break;
            float x[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float acc = 0.f;
                const float4* row = reinterpret_cast<const float4*>(ascr + r * L::AS_STRIDE);
#pragma unroll
                for (int i4 = 0; i4 < (r + 3) / 4; ++i4) {
                    const float4 a = row[i4];
                    acc += a.x * x[4 * i4];
                    if (4 * i4 + 1 < r) acc += a.y * x[4 * i4 + 1];
                    if (4 * i4 + 2 < r) acc += a.z * x[4 * i4 + 2];
                    if (4 * i4 + 3 < r) acc += a.w * x[4 * i4 + 3];
                }
                x[r] = (r == j) ? 1.f : (r > j ? -acc : 0.f);
            }
            mbar_arrive(&bar[B_AFREE]);
            if (n > 0 && !mbar_wait(&bar[B_WYDONE], (n - 1) & 1, ab, status)) break;
            const float bj = sbeta[(n & 1) * 64 + j];
            uint8_t* tt = sm + L::OFF_TT;
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16) {
                uint4 w;
                w.x = pack_half2(x[8 * c16 + 0] * bj, x[8 * c16 + 1] * bj);
                w.y = pack_half2(x[8 * c16 + 2] * bj, x[8 * c16 + 3] * bj);
                w.z = pack_half2(x[8 * c16 + 4] * bj, x[8 * c16 + 5] * bj);
                w.w = pack_half2(x[8 * c16 + 6] * bj, x[8 * c16 + 7] * bj);
                *reinterpret_cast<uint4*>(tt + sw128(j, c16)) = w;
            }
            fence_proxy_async_smem();
            mbar_arrive(&bar[B_TRDY]);
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ prep warpgroup
        const int c = tid - 128;  // key channel (and TMEM lane) of this thread
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        bool range_bad = false;
        uint32_t v16[32];  // this channel's 64 values of v as packed fp16 (V16 row c)
        float beta_next = 0.f;
        auto load_beta = [&](int n) -> float {
            const int64_t vld = len - (int64_t)C * n;
            return (c < 64 && c < vld) ? P.beta[(size_t)(t0 + (int64_t)C * n + c) * P.H + h] : 0.f;
        };
        beta_next = load_beta(0);

        // prep1(n): decay cumsum, operand tiles KT/QT/KH, vectors, beta.
        auto prep1 = [&](int n) -> bool {
            const int b = n & 1;
            if (n >= 2) {
                if (!mbar_wait(&bar[B_KQFREE + b], ((n - 2) >> 1) & 1, ab, status)) return false;
                if (!mbar_wait(&bar[B_VFREE + b], ((n - 2) >> 1) & 1, ab, status)) return false;
            }
            const int valid = (int)((len - (int64_t)C * n) < C ? (len - (int64_t)C * n) : C);
            if (c < 64) sbeta[b * 64 + c] = beta_next;
            if (n + 1 < nch) beta_next = load_beta(n + 1);
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
            float g2 = 0.f;
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const uint8_t* sl = slot_ptr(r >> 4);
                const float la = reinterpret_cast<const float*>(sl + L::SLOT_LA)[(r & 15) * 128 + c];
                g2 += (r < valid) ? la * kLog2e : 0.f;
            }
            const float ref = g2;
            // pass B: operand rows
            g2 = 0.f;
            uint32_t pk[4], pq[4], ph[4];
            float kprev = 0.f, qprev = 0.f, hprev = 0.f, vprev = 0.f;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                if (r == 32) {  // rows 0..31 consumed: release their slots, fetch rows 32..47
                    mbar_arrive(&bar[B_EMPTY + (4 * n + 0) % L::NSLOT]);
                    mbar_arrive(&bar[B_EMPTY + (4 * n + 1) % L::NSLOT]);
                    if (!wait_slot(2)) return false;
                }
                if (r == 48) {
                    mbar_arrive(&bar[B_EMPTY + (4 * n + 2) % L::NSLOT]);
                    if (!wait_slot(3)) return false;
                }
                const uint8_t* sl = slot_ptr(r >> 4);
                const int rr = r & 15;
                const bool on = r < valid;
                const float la = on ? reinterpret_cast<const float*>(sl + L::SLOT_LA)[rr * 128 + c] : 0.f;
                const float kk = on ? ld_in(reinterpret_cast<const Tin*>(sl + L::SLOT_K), rr * 128 + c) : 0.f;
                const float qq = on ? ld_in(reinterpret_cast<const Tin*>(sl + L::SLOT_Q), rr * 128 + c) : 0.f;
                const float vv = on ? ld_in(reinterpret_cast<const Tin*>(sl + L::SLOT_V), rr * 128 + c) : 0.f;
                g2 += la * kLog2e;
                const float x = g2 - ref;
                range_bad |= fabsf(x) > kMaxExp2;
                const float e1 = exp2f(x), e2 = exp2f(-x);
                const float kv = kk * e1, qv = qq * e1, hv = kk * e2;
                if (r & 1) {
                    pk[(r >> 1) & 3] = pack_half2(kprev, kv);
                    pq[(r >> 1) & 3] = pack_half2(qprev, qv);
                    ph[(r >> 1) & 3] = pack_half2(hprev, hv);
                    v16[r >> 1] = pack_half2(vprev, vv);
                } else {
                    kprev = kv; qprev = qv; hprev = hv; vprev = vv;
                }
                if ((r & 7) == 7) {
                    const uint32_t off = sw128(c, r >> 3);
                    *reinterpret_cast<uint4*>(kt + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    *reinterpret_cast<uint4*>(qt + off) = make_uint4(pq[0], pq[1], pq[2], pq[3]);
                    *reinterpret_cast<uint4*>(kh + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                }
            }
            mbar_arrive(&bar[B_EMPTY + (4 * n + 3) % L::NSLOT]);
            vec_a[b * 128 + c] = exp2f(ref);
            vec_b[b * 128 + c] = exp2f(g2 - ref);
            fence_proxy_async_smem();
            mbar_arrive(&bar[B_PREPD + b]);
            return true;
        };
        // prep2(n): V16 into TMEM once the previous chunk's WY product has read it
        auto prep2 = [&](int n) -> bool {
            if (n > 0 && !mbar_wait(&bar[B_WYDONE], (n - 1) & 1, ab, status)) return false;
            tc_fence_after();
            tmem_st32(tmem + lane_base + TM_V16, v16);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar[B_VRDY]);
            return true;
        };
        // P2(n): read the Gram accumulator: A rows to the solver's scratch, P rows to PP
        auto p2 = [&](int n) -> bool {
            const int b = n & 1;
            if (!mbar_wait(&bar[B_GDONE], n & 1, ab, status)) return false;
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + lane_base + TM_G, r0);
            tmem_ld32(tmem + lane_base + TM_G + 32, r1);
            tmem_ld_wait();
            if (c < 64) {  // row r = c of A (beta_r applied here)
                if (n > 0 && !mbar_wait(&bar[B_AFREE], (n - 1) & 1, ab, status)) return false;
                const float br = sbeta[b * 64 + c];
                float* row = ascr + c * L::AS_STRIDE;
#pragma unroll
                for (int i4 = 0; i4 < 16; ++i4) {
                    float4 w;
                    const uint32_t* src = i4 < 8 ? &r0[4 * i4] : &r1[4 * (i4 - 8)];
                    w.x = (4 * i4 + 0 < c) ? br * __uint_as_float(src[0]) : 0.f;
                    w.y = (4 * i4 + 1 < c) ? br * __uint_as_float(src[1]) : 0.f;
                    w.z = (4 * i4 + 2 < c) ? br * __uint_as_float(src[2]) : 0.f;
                    w.w = (4 * i4 + 3 < c) ? br * __uint_as_float(src[3]) : 0.f;
                    reinterpret_cast<float4*>(row)[i4] = w;
                }
            } else {  // row r = c - 64 of P (lower triangle including the diagonal)
                if (n >= 2 && !mbar_wait(&bar[B_KQFREE + b], ((n - 2) >> 1) & 1, ab, status)) return false;
                const int r = c - 64;
                uint8_t* pp = sm + L::OFF_PP + b * 8192;
#pragma unroll
                for (int c16 = 0; c16 < 8; ++c16) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int i = 8 * c16 + e;
                        const uint32_t u = i < 32 ? r0[i] : r1[i - 32];
                        f[e] = (i <= r) ? __uint_as_float(u) : 0.f;
                    }
                    *reinterpret_cast<uint4*>(pp + sw128(r, c16)) =
                        make_uint4(pack_half2(f[0], f[1]), pack_half2(f[2], f[3]), pack_half2(f[4], f[5]),
                                   pack_half2(f[6], f[7]));
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(&bar[B_P2D]);
            return true;
        };
        bool ok = prep1(0) && prep2(0) && p2(0);
        for (int n = 0; n + 1 < nch && ok; ++n) ok = prep1(n + 1) && p2(n + 1) && prep2(n + 1);
        if (range_bad) atomicCAS(status, 0, (int)KDA_STATUS_GATE_RANGE);
    } else {
        // ------------------------------------------------------------ state warpgroup
        const int j = tid - 256;  // value column (and TMEM lane) of this thread
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        Tout* out = static_cast<Tout*>(P.out);
        bool ok = true;
        {  // X_0 = Diag(a_0) S_0 into D_S and X16
            if (!(ok = mbar_wait(&bar[B_PREPD], 0, ab, status))) goto state_done;
            const float* a0 = vec_a;
            uint32_t x16[64];
#pragma unroll
            for (int piece = 0; piece < 4; ++piece) {
                uint32_t xs[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int cc = piece * 32 + e;
                    const float s0 = P.init ? P.init[sbase + (size_t)cc * kD + j] : 0.f;
                    xs[e] = __float_as_uint(s0 * a0[cc]);
                }
                tmem_st32(tmem + lane_base + TM_S + piece * 32, xs);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    x16[piece * 16 + e] = pack_half2(__uint_as_float(xs[2 * e]), __uint_as_float(xs[2 * e + 1]));
            }
            tmem_st32(tmem + lane_base + TM_X16, *reinterpret_cast<uint32_t(*)[32]>(&x16[0]));
            tmem_st32(tmem + lane_base + TM_X16 + 32, *reinterpret_cast<uint32_t(*)[32]>(&x16[32]));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar[B_XRDY]);
        }
        for (int n = 0; n < nch; ++n) {
            const int b = n & 1;
            const int valid = (int)((len - (int64_t)C * n) < C ? (len - (int64_t)C * n) : C);
            // P4(n): WT = -W^T as fp16
            if (!(ok = mbar_wait(&bar[B_WYDONE], n & 1, ab, status))) break;
            tc_fence_after();
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lane_base + TM_W, r0);
                tmem_ld32(tmem + lane_base + TM_W + 32, r1);
                tmem_ld_wait();
                uint8_t* wt = sm + L::OFF_WT;
#pragma unroll
                for (int c16 = 0; c16 < 8; ++c16) {
                    const uint32_t* src = c16 < 4 ? &r0[8 * c16] : &r1[8 * (c16 - 4)];
                    *reinterpret_cast<uint4*>(wt + sw128(j, c16)) = make_uint4(
                        pack_half2(-__uint_as_float(src[0]), -__uint_as_float(src[1])),
                        pack_half2(-__uint_as_float(src[2]), -__uint_as_float(src[3])),
                        pack_half2(-__uint_as_float(src[4]), -__uint_as_float(src[5])),
                        pack_half2(-__uint_as_float(src[6]), -__uint_as_float(src[7])));
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bar[B_WRDY]);
            }
            // S2(n): U16 = fp16(U^T)
            if (!(ok = mbar_wait(&bar[B_UIDONE], n & 1, ab, status))) break;
            tc_fence_after();
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
            }
            // S3(n): outputs, state, snapshots, next X
            if (!(ok = mbar_wait(&bar[B_SDONE], n & 1, ab, status))) break;
            tc_fence_after();
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lane_base + TM_O, r0);
                tmem_ld32(tmem + lane_base + TM_O + 32, r1);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&bar[B_OFREE]);
                const size_t obase = ((size_t)(t0 + (int64_t)C * n) * P.H + h) * kD + j;
                const size_t ostride = (size_t)P.H * kD;
#pragma unroll
                for (int r = 0; r < C; ++r) {
                    if (r < valid) {
                        const float o = __uint_as_float(r < 32 ? r0[r] : r1[r - 32]);
                        if constexpr (sizeof(Tout) == 2)
                            out[obase + r * ostride] = __float2bfloat16_rn(o);
                        else
                            out[obase + r * ostride] = o;
                    }
                }
            }
            {
                const bool last = (n + 1 == nch);
                const int64_t end_pos = (int64_t)C * n + valid;  // tokens of the sequence consumed so far
                float* snap = nullptr;
                if (P.snap_interval > 0 && valid == C && end_pos % P.snap_interval == 0)
                    snap = P.snapshots + ((size_t)(P.snap_offsets[s] + end_pos / P.snap_interval - 1) * P.H + h) *
                                             kD * kD;
                float* fin = (last && P.final_state) ? P.final_state + sbase : nullptr;
                if (!last && !(ok = mbar_wait(&bar[B_PREPD + ((n + 1) & 1)], ((n + 1) >> 1) & 1, ab, status)))
                    break;
                const float* bv = vec_b + b * 128;
                const float* an = vec_a + ((n + 1) & 1) * 128;
                uint32_t x16[64];
#pragma unroll
                for (int piece = 0; piece < 4; ++piece) {
                    uint32_t d[32];
                    tmem_ld32(tmem + lane_base + TM_S + piece * 32, d);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int cc = piece * 32 + e;
                        const float sv = __uint_as_float(d[e]) * bv[cc];  // true state S[cc][j]
                        if (snap) snap[(size_t)cc * kD + j] = sv;
                        if (fin) fin[(size_t)cc * kD + j] = sv;
                        d[e] = __float_as_uint(last ? 0.f : sv * an[cc]);
                    }
                    if (!last) {
                        tmem_st32(tmem + lane_base + TM_S + piece * 32, d);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            x16[piece * 16 + e] =
                                pack_half2(__uint_as_float(d[2 * e]), __uint_as_float(d[2 * e + 1]));
                    }
                }
                if (!last) {
                    tmem_st32(tmem + lane_base + TM_X16, *reinterpret_cast<uint32_t(*)[32]>(&x16[0]));
                    tmem_st32(tmem + lane_base + TM_X16 + 32, *reinterpret_cast<uint32_t(*)[32]>(&x16[32]));
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&bar[B_XRDY]);
                }
                mbar_arrive(&bar[B_VFREE + b]);
            }
        }
    state_done:;
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
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
    CUtensorMap mq, mk, mv, ml;
    const CUtensorMapDataType dt = sizeof(Tin) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int64_t Tt = p.T_total > 0 ? p.T_total : 1;
    if (Tt > (int64_t)0x7FFFFFFF - 2 * C) return cudaErrorInvalidValue;  // tensor-map coordinates are 32-bit
    if (!make_map(&mq, p.q, dt, sizeof(Tin), Tt, p.H) || !make_map(&mk, p.k, dt, sizeof(Tin), Tt, p.H) ||
        !make_map(&mv, p.v, dt, sizeof(Tin), Tt, p.H) ||
        !make_map(&ml, p.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Tt, p.H))
        return cudaErrorInvalidValue;
    auto kern = chunk_kernel<Tin, Tout>;
    const int smem = (int)Cfg<Tin>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((int64_t)p.N * p.H);
    kern<<<grid, NTHREADS, smem, st>>>(mq, mk, mv, ml, p);
    return cudaGetLastError();
}

}  // namespace

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
