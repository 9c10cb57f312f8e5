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
// Gates beyond that range: a chunk in which some key channel decays by more than
// 2^kMaxExp2 over either half (a channel that forgets within a few tokens, down to
// alpha = 0) cannot be factored this way.  The kernel runs in two instantiations.
// The first (ROB = false, the hot one) processes every (sequence, head) and only
// marks the units that met such a chunk; the second (ROB = true) recomputes exactly
// those units: a chunk within range goes through the same products in the same
// order (bit-identical to the first), a chunk beyond it skips its state products
// and the state warpgroup applies its tokens one at a time in fp32 to the state held
// in TMEM instead (the §四 recurrence itself, exact for any alpha in [0, 1]).  The
// path of a chunk depends on its own gates only, so a run resumed at a chunk
// boundary still reproduces the unsplit run bit for bit.
//
// The triangular inverse (the WY solve of §六) is a blocked substitution: A is
// split into 16x16 blocks; the diagonal blocks are inverted in fp32 on CUDA cores
// (Dg_a = (I + A_aa)^-1, one thread per column), and the blocks below the diagonal
// follow block column by block column from
//   T_ab = -Dg_a sum_{k=b}^{a-1} A_ak T_kb      (T_bb = Dg_b),
// as warp-level 16x16 products (fp16 operands, fp32 accumulation), one warp per
// block column.  They are computed transposed, S_ba = T_ab^T, so that every result
// is directly the left operand of the next product.  T diag(beta) is rounded to
// fp16 as the operand of the WY products.
//
// Data layout on chip (one CTA = one (sequence, head), all of d_v = 128):
//   TMEM (fp32 accumulators, lanes = the M rows):
//     D_S [j][c] state (128 cols)   D_O [j][r] output (right after D_S)   X16 [j][c] fp16 A operand
//     D_U [j][r] U'/U   U16 [j][r] fp16 A operand (over D_U)   D_G [r|64+r][i] Gram
//     D_W [c][r] W^T    V16 [2][j][i] fp16 A operand (v^T), by chunk parity
//   SMEM (fp16 operand tiles, 128-byte swizzled rows of 64 elements):
//     KT[c][r] = Ktil_p, QT[c][r] = Qtil_p (adjacent: together the M = 128 A
//     operand of the Gram; once a chunk's products are done the pair stages
//     its output for the TMA store), KH[c][r] = Khat_p followed by PP[r][i] = P (one
//     N = 192 operand),
//     WT[c][r] = -W^T, NR[r][i] = T diag(beta); the 16x16 blocks of A (diagonal
//     ones fp32, the rest fp16) and of Dg (fp16);
//     a ring of 16-token input slots filled by TMA.
//   The products (all tcgen05.mma, fp16 operands, fp32 accumulation):
//     Gram  D_G = [KT;QT] x KH                 M=128 N=64  K=128
//     WY    D_W = KT x NR,  D_U = V16 x NR     M=128 N=64  K=64
//     (i)   D_U += X16 x WT                    M=128 N=64  K=128
//     (iii-a) D_O = X16 x QT                   M=128 N=64  K=128
//     (ii) + (iii-b)  [D_S | D_O] += U16 x [KH | PP]   M=128 N=192 K=64 (one product)
//
// Warp roles (16 warps): 0 TMA producer, 1 beta loader (+ TMEM allocation),
// 2 issues the Gram, 3 issues the WY products (in the exact second pass the tri
// warpgroup issues them itself), 4-7 "prep" warpgroup (decay cumsum, operand
// tiles), 8-11 "state" warpgroup (U conversion, state rescale, snapshots, outputs;
// issues (i)-(iii)), 12-15 "tri" warpgroup (Gram readout, the inverse, W readout).
// A product group is issued by a thread whose warp has nothing else to do, so that
// no warp of the working roles stalls behind the issue.  Roles hand work to each
// other through mbarriers; every wait is bounded.
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {
using namespace sm100;

constexpr int C = 64;   // chunk length
constexpr int QR = 16;  // token rows per input slot
constexpr int NTHREADS = 512;
constexpr int kLptMax = 256;  // most packed sequences the kernel orders by length itself
constexpr long long kClaimDelay = 4000;  // cycles a CTA on a higher-numbered SM waits before it claims a unit
// Launches of at most this many (sequence, head) units place them on the lowest-numbered SMs.  The
// scheduler starts a launch on SMs 148..151 and then pairs of SMs across the chip; for the 96 heads
// of the long prefill that placement (SMs 0..91 and 148..151) ran 15% slower than SMs 0..95 (8.73
// against 10.24 ms, bit-identical), while at 16 and 64 units the two were within 1% and at 128 units
// the scheduler's placement was 12% faster, so the rule stops at 96.
constexpr int kPackUnits = 96;
constexpr float kLog2e = 1.4426950408889634f;
// |g - ref| bound (log2 units) of the fp16 operand path.  An element scaled down by 2^-|g-ref|
// can land in the fp16 subnormals, where its absolute rounding error is 2^-25, and the factor
// on the other side of its product scales that error by up to 2^|g-ref|.  At 10 the worst such
// term is 2^-15 of an O(1) operand, below the fp16 rounding of the products themselves; chunks
// beyond it take the exact fp32 path.
constexpr float kMaxExp2 = 10.0f;
constexpr int kRowH = 48;          // row stride (bytes) of a 16x16 fp16 block (ldmatrix: no bank conflicts)
constexpr int kBlkH = 16 * kRowH;  // bytes per fp16 block

// TMEM column map (512 columns allocated).  D_O follows D_S, so that the state update and
// the intra-chunk output term are one N = 192 product.  The fp16 U operand is written over
// the first 32 columns of the U accumulator once that has been read out; V16
// (the fp16 v^T operand) is double-buffered by chunk parity.
constexpr uint32_t TM_S = 0, TM_O = 128, TM_X16 = 192, TM_U = 256, TM_U16 = 256, TM_G = 320, TM_W = 384,
                   TM_V16 = 448;

template <typename Tin>
struct Cfg {
    static constexpr int ES = sizeof(Tin);
#ifndef KDA_CFG_NSLOT
#define KDA_CFG_NSLOT 2
#endif
#ifndef KDA_CFG_STG_OWN
#define KDA_CFG_STG_OWN 1
#endif
    static constexpr int NSLOT = ES == 2 ? KDA_CFG_NSLOT : 2;  // input ring slots (tiles are pulled into L2 ahead)
    static constexpr bool STG_OWN = ES == 2 && KDA_CFG_STG_OWN;  // own staging buffer for the output (else KT/QT)
    static constexpr uint32_t SLOT_Q = 0;
    static constexpr uint32_t SLOT_K = QR * 128 * ES;
    static constexpr uint32_t SLOT_V = 2 * QR * 128 * ES;
    static constexpr uint32_t SLOT_LA = 3 * QR * 128 * ES;
    static constexpr uint32_t SLOT_BYTES = 3 * QR * 128 * ES + QR * 128 * 4;
    // shared memory map (offsets from a 1024-byte aligned base)
    static constexpr uint32_t OFF_KQ = 0;                    // [2] x (KT 16K | QT 16K)
    static constexpr uint32_t OFF_KH = 65536;                // [2] x (KH 16K | PP 8K)
    static constexpr uint32_t KHP = 24576;                   // stride of the KH/PP pairs
    static constexpr uint32_t OFF_WT = OFF_KH + 2 * KHP;     // 16K
    static constexpr uint32_t OFF_NR = OFF_WT + 16384;       // 8K
    static constexpr uint32_t OFF_INV = OFF_NR + 8192;  // A diagonal blocks (fp32), A below them and Dg (fp16)
    static constexpr uint32_t INV_BYTES = 4 * 1024 + 10 * kBlkH;
    static constexpr uint32_t OFF_STG = OFF_INV + INV_BYTES;  // 64 output rows (STG_OWN)
    static constexpr uint32_t OFF_RING = OFF_STG + (STG_OWN ? 64 * 128 * 4 : 0);
    static constexpr uint32_t OFF_VEC = OFF_RING + NSLOT * SLOT_BYTES;  // a[3][128], b[3][128]
    static constexpr uint32_t OFF_BETA = OFF_VEC + 6 * 128 * 4;         // [4][64]
    static constexpr uint32_t OFF_GATE = OFF_BETA + 4 * 64 * 4;         // [4][64] scalar gates
    static constexpr uint32_t OFF_ONES = OFF_GATE + 4 * 64 * 4;         // [128] 1.0f
    static constexpr uint32_t OFF_CBAD = OFF_ONES + 128 * 4;            // [3][4] chunk beyond the fp16 range
    static constexpr uint32_t OFF_BAR = OFF_CBAD + 3 * 4 * 4;
    static constexpr uint32_t NBAR = 40;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
#ifdef KDA_TRACE
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 32 * 24 * 4 + 1024;
#else
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
#endif
};
static_assert(Cfg<__nv_bfloat16>::SMEM_BYTES <= 232448, "smem budget (bf16)");
static_assert(Cfg<float>::SMEM_BYTES <= 232448, "smem budget (fp32)");
static_assert(Cfg<__nv_bfloat16>::OFF_RING % 128 == 0 && Cfg<float>::OFF_RING % 128 == 0, "TMA destinations");
static_assert(Cfg<__nv_bfloat16>::OFF_STG % 128 == 0, "TMA store source");
static_assert(Cfg<__nv_bfloat16>::OFF_BAR % 8 == 0 && Cfg<float>::OFF_BAR % 8 == 0, "mbarrier alignment");

// barrier indices
enum {
    B_FULL = 0,      // [NSLOT] input slot landed
    B_EMPTY = 3,     // [NSLOT] input slot consumed
    B_PREPD = 6,     // [2] KT/QT/KH, V16, vectors of a chunk ready
    B_GDONE = 8,     // Gram complete
    B_P2D = 9,       // Gram read out: D_G free
    B_TB = 10,       // tri warpgroup's own barrier
    B_WYDONE = 11,   // WY products complete
    B_V16FREE = 12,  // [2] V16 of a chunk consumed (WY complete)
    B_WRDY = 14,     // WT and PP written
    B_XRDY = 15,     // X16 / D_S ready for the chunk
    B_UIDONE = 16,   // (i) complete: U readable, WT free
    B_URDY = 17,     // U16 written
    B_SDONE = 18,    // (ii) and (iii) complete
    B_KQFREE = 19,   // [2] KH and PP of a chunk consumed
    B_OFREE = 21,    // D_O read out
    B_STG = 22,      // output staging tile written by the whole state warpgroup
    B_STGFREE = 23,  // [2] KT/QT pair free again (staged output read by the bulk store; !STG_OWN)
    B_BFULL = 25,    // [4] beta of a chunk loaded (ring of 4, by chunk index mod 4)
    B_BFREE = 29,    // [4] beta ring slot consumed
    B_VFREE = 33,    // [3] decay vectors of a chunk consumed (ring of 3, by chunk index mod 3)
    B_STGR = 36,     // own staging buffer read by the previous bulk store (STG_OWN)
    B_PDONE = 37,    // prep has seen every chunk (the unit's range flag is final); ROB = false
    B_SER = 38,      // the exact path's coefficient buffers written (state warpgroup; ROB = true)
    B_NRD = 39,      // NR = T diag(beta) written by the tri warpgroup (ROB = false)
    B_COUNT = 40
};
static_assert(B_COUNT <= (int)Cfg<float>::NBAR, "barrier space");

#ifdef KDA_TRACE
// Debug timeline (compiled only with -DKDA_TRACE): clock() stamps of each role's
// milestones for chunks 16..47 of CTA 0, kept in shared memory (a global store
// would delay the next barrier arrive) and copied out when the CTA ends.
#ifndef KDA_TRACE_FIRST
#define KDA_TRACE_FIRST 16
#endif
constexpr int kTrEv = 32, kTrN0 = KDA_TRACE_FIRST, kTrN = 24;
__device__ unsigned int g_trace[kTrN * kTrEv];
#define KDA_TR(n, ev)                                                                       \
    do {                                                                                    \
        if (blockIdx.x == 0 && (n) >= kTrN0 && (n) < kTrN0 + kTrN)                          \
            trace_sm[((n) - kTrN0) * kTrEv + (ev)] = (unsigned int)clock();                 \
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
// `sign` is XORed into every packed pair (0x80008000 negates both halves).
__device__ __forceinline__ void store_row16(uint8_t* tile, uint32_t row, const uint32_t (&r0)[32],
                                            const uint32_t (&r1)[32], uint32_t sign = 0u) {
#pragma unroll
    for (int c16 = 0; c16 < 8; ++c16) {
        const uint32_t* s = c16 < 4 ? &r0[8 * c16] : &r1[8 * (c16 - 4)];
        *reinterpret_cast<uint4*>(tile + sw128(row, c16)) =
            make_uint4(pack_half2(__uint_as_float(s[0]), __uint_as_float(s[1])) ^ sign,
                       pack_half2(__uint_as_float(s[2]), __uint_as_float(s[3])) ^ sign,
                       pack_half2(__uint_as_float(s[4]), __uint_as_float(s[5])) ^ sign,
                       pack_half2(__uint_as_float(s[6]), __uint_as_float(s[7])) ^ sign);
    }
}

// Writes 32 packed fp16 pairs (columns 0..63) as one 128-byte swizzled row.
__device__ __forceinline__ void store_row16_packed(uint8_t* tile, uint32_t row, const uint32_t (&p)[32]) {
#pragma unroll
    for (int c16 = 0; c16 < 8; ++c16)
        *reinterpret_cast<uint4*>(tile + sw128(row, c16)) =
            make_uint4(p[4 * c16], p[4 * c16 + 1], p[4 * c16 + 2], p[4 * c16 + 3]);
}

// fp32 16x16 diagonal blocks of A (read by the substitution): row r holds its 16
// values as four 16-byte chunks, chunk k stored at position k ^ ((r >> 1) & 3).
__device__ __forceinline__ int bsw(int r, int k4) { return r * 16 + ((k4 ^ ((r >> 1) & 3)) << 2); }

// Warp-level 16x16 block products of the triangular solve (fp16 in, fp32 accumulate).
// ldmatrix: lanes 8m .. 8m+7 give the rows of 8x8 matrix m; .trans delivers its transpose.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t saddr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t saddr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr)
                 : "memory");
}
// d (16x8 fp32) += a (16x16 fp16, row-major fragment) x b (16x8 fp16, column fragment)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void st4(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void st_half(uint8_t* p, float v) {
    *reinterpret_cast<__half*>(p) = __float2half_rn(v);
}

// One block column B of T = (I + A)^-1 (T_aa = Dg_a), with T_aB = -Dg_a sum_{k=B}^{a-1} A_ak T_kB,
// computed transposed, S_Ba = T_aB^T = -(sum_k S_Bk A_ak^T) Dg_a^T, so that each result's
// accumulator fragment is directly the A fragment of the next product.  The blocks
// below the diagonal go to NR as T diag(beta) (fp16, 128-byte swizzled rows).  One warp.
template <int B>
__device__ __forceinline__ void tri_column(uint32_t a16, uint32_t dg16, uint8_t* nr, const float* bt, int lane) {
    // lane l supplies the row address (l & 7) + 8 (l >> 4), column half (l >> 3) & 1 of a block
    const uint32_t lrow = (uint32_t)(((lane & 7) + 8 * (lane >> 4)) * kRowH + 16 * ((lane >> 3) & 1));
    const int g = lane >> 2, t = lane & 3;
    uint32_t sf[4][4];
    {  // S_BB = Dg_B^T: matrices (rows 0-7 | 8-15) x (cols 0-7 | 8-15) of Dg_B, transposed
        const uint32_t trow = (uint32_t)(((lane & 7) + 8 * ((lane >> 4) & 1)) * kRowH + 16 * ((lane >> 3) & 1));
        uint32_t m[4];
        ldsm_x4_t(m, dg16 + B * kBlkH + trow);
        // fragment order: (rows 0-7, k 0-7), (rows 8-15, k 0-7), (rows 0-7, k 8-15), (rows 8-15, k 8-15)
        sf[B][0] = m[0];
        sf[B][1] = m[1];
        sf[B][2] = m[2];
        sf[B][3] = m[3];
    }
    const float bg = bt[16 * B + g], bg8 = bt[16 * B + g + 8];
#pragma unroll
    for (int a = B + 1; a < 4; ++a) {
        float z0[4] = {0.f, 0.f, 0.f, 0.f}, z1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = B; k < a; ++k) {  // Z += S_Bk A_ak^T
            uint32_t bA[4];
            ldsm_x4(bA, a16 + (a * (a - 1) / 2 + k) * kBlkH + lrow);
            mma16816(z0, sf[k], bA[0], bA[1]);
            mma16816(z1, sf[k], bA[2], bA[3]);
        }
        const uint32_t zf[4] = {pack_half2(z0[0], z0[1]), pack_half2(z0[2], z0[3]), pack_half2(z1[0], z1[1]),
                                pack_half2(z1[2], z1[3])};
        uint32_t bD[4];
        ldsm_x4(bD, dg16 + a * kBlkH + lrow);
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(s0, zf, bD[0], bD[1]);
        mma16816(s1, zf, bD[2], bD[3]);
        if (a < 3) {  // S_Ba = -Z Dg_a^T, kept as the A fragment of later levels
            sf[a][0] = pack_half2(-s0[0], -s0[1]);
            sf[a][1] = pack_half2(-s0[2], -s0[3]);
            sf[a][2] = pack_half2(-s1[0], -s1[1]);
            sf[a][3] = pack_half2(-s1[2], -s1[3]);
        }
        // S_Ba[i][r] = T_aB[r][i]: this lane holds i in {g, g+8}, r in {2t, 2t+1, 2t+8, 2t+9}
        const int row = 16 * a + 2 * t, col = 16 * B + g;
        st_half(nr + sw128(row, col >> 3) + (col & 7) * 2, -s0[0] * bg);
        st_half(nr + sw128(row + 1, col >> 3) + (col & 7) * 2, -s0[1] * bg);
        st_half(nr + sw128(row, (col + 8) >> 3) + (col & 7) * 2, -s0[2] * bg8);
        st_half(nr + sw128(row + 1, (col + 8) >> 3) + (col & 7) * 2, -s0[3] * bg8);
        st_half(nr + sw128(row + 8, col >> 3) + (col & 7) * 2, -s1[0] * bg);
        st_half(nr + sw128(row + 9, col >> 3) + (col & 7) * 2, -s1[1] * bg);
        st_half(nr + sw128(row + 8, (col + 8) >> 3) + (col & 7) * 2, -s1[2] * bg8);
        st_half(nr + sw128(row + 9, (col + 8) >> 3) + (col & 7) * 2, -s1[3] * bg8);
    }
}

// The true state Diag(b) D of column j (TMEM lane) rounded to bf16 into a bf16 pool slot.
// Out of line: rare (snapshots only) and kept out of the kernel's hot code.
__device__ __noinline__ void store_state_bf16(__nv_bfloat16* dst, uint32_t taddr, const float* bv, int j) {
#pragma unroll 1
    for (int piece = 0; piece < 4; ++piece) {
        uint32_t d[32];
        tmem_ld32(taddr + piece * 32, d);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int cc = piece * 32 + e;
            dst[(size_t)cc * kD + j] = __float2bfloat16_rn(__uint_as_float(d[e]) * bv[cc]);
        }
    }
}

// The exact path for one chunk whose gates leave the fp16 operand range: its tokens applied in
// fp32, in order, to the state held in TMEM (taddr: D_S of this warp's 32 lanes, lanes = value
// columns, columns = key channels).  Per token ("Kimi K3" article §四 with the §二.1 read):
//   u_t = beta_t (v_t - (alpha_t . k_t)^T S_{t-1}),  S_t = alpha_t . S_{t-1} + k_t u_t,  o_t = S_t^T q_t.
// kG tokens are folded into one read pass and one write pass over the state.  With the group's
// start state S, A_t = alpha_0 ... alpha_t and B_{s,t} = alpha_{s+1} ... alpha_t (B_{t,t} = 1),
// products of gates, so every factor is in [0, 1] whatever the gates:
//   (alpha_t . k_t)^T S_{t-1} = (k_t A_t)^T S + sum_{s<t} [(k_t B_{s,t})^T k_s] u_s
//   o_t = (q_t A_t)^T S + sum_{s<=t} [(q_t B_{s,t})^T k_s] u_s
//   S_{kG-1} = A_{kG-1} . S + sum_s (k_s B_{s,kG-1}) u_s.
// The bracketed scalars are the same for every column; the 128 threads reduce them together.
// The state is accessed with 16x256b TMEM loads, so that a thread holds two key channels of four
// value columns at a time and each coefficient it reads from shared memory serves four columns;
// the four threads that share columns (lane % 4) sum their partial dot products with two shuffles.
// Called by the 128 threads of the state warpgroup; `stage` (two buffers of kSerBuf floats) is
// shared memory the warpgroup owns for the call; `sbar` (128 arrivals per use, phase count in
// `sph`) orders its use, with bounded waits.  row0: the chunk's first packed token.  The output
// rows go straight to global memory.  Out of line: it runs only for such chunks.  Returns false
// if a wait gave up.
constexpr int kG = 4;                                     // tokens per pass pair
constexpr int kSerVec = 4 * kG + 1;                       // coefficient (and v) vectors of a group
constexpr int kSerM = kG * (kG - 1) / 2, kSerN = kG * (kG + 1) / 2;  // scalars (s < t), (s <= t)
constexpr int kSerBuf = kSerVec * 128 + 4 * (kSerM + kSerN);  // + one partial sum per warp
static_assert(2 * kSerBuf * 4 <= 32768 && (kSerBuf * 4) % 16 == 0, "exact path buffers fit the output staging / KT-QT pair");
template <typename Tin, typename Tout, bool SG>
__device__ __noinline__ bool serial_chunk(uint32_t taddr, int j, int64_t row0, int valid, int h, int H,
                                          const Tin* __restrict__ q, const Tin* __restrict__ k,
                                          const Tin* __restrict__ v, const float* __restrict__ log_alpha,
                                          const float* __restrict__ beta, Tout* __restrict__ out, float* stage,
                                          uint64_t* sbar, uint32_t& sph, Abort* ab, int* status) {
    // vectors of a buffer: [t] k_t A_t, [kG + t] q_t A_t, [2 kG] A_{kG-1}, [2 kG + 1 + s] k_s B_{s,kG-1},
    // [3 kG + 1 + t] v_t (by value column)
    constexpr int KA = 0, QA = kG, AL = 2 * kG, KB = 2 * kG + 1, VV = 3 * kG + 1, PART = kSerVec * 128;
    const int lane = j & 31, wq = j >> 5;
    // 16x256b layout: this thread's value columns jc(i) = 32 wq + lane / 4 + 8 i (i = 0, 1 from the
    // warp's first 16 lanes, 2, 3 from the next 16), its key channels 8 b + cq and 8 b + cq + 1 of
    // every block b of 8
    const int cq = 2 * (lane & 3), j0 = 32 * wq + (lane >> 2);
    const uint32_t tA = taddr, tB = taddr + (16u << 16);
    // this thread's channel c = j of every token of a group (and value column j)
    float kk[kG], qq[kG], la[kG], vv[kG], bb[kG];
    auto load = [&](int r0) {
#pragma unroll
        for (int t = 0; t < kG; ++t) {
            kk[t] = qq[t] = la[t] = vv[t] = bb[t] = 0.f;  // past the chunk: identity steps
            if (r0 + t < valid) {
                const size_t tok = (size_t)(row0 + r0 + t) * H + h, off = tok * kD + j;
                kk[t] = ld_in(k, off);
                qq[t] = ld_in(q, off);
                vv[t] = ld_in(v, off);
                bb[t] = beta[tok];
                if constexpr (SG)
                    la[t] = log_alpha ? log_alpha[tok] : 0.f;
                else
                    la[t] = log_alpha[off];
            }
        }
    };
    load(0);
#pragma unroll 1
    for (int r0 = 0, g = 0; r0 < valid; r0 += kG, ++g) {
        float* buf = stage + (g & 1) * kSerBuf;
        float bt[kG];
        {  // coefficients of this group (channel j), and v (column j)
            float al[kG];
#pragma unroll
            for (int t = 0; t < kG; ++t) al[t] = expf(la[t]);
            float A = 1.f;  // A_t
#pragma unroll
            for (int t = 0; t < kG; ++t) {
                A *= al[t];
                buf[(KA + t) * 128 + j] = kk[t] * A;
                buf[(QA + t) * 128 + j] = qq[t] * A;
                buf[(VV + t) * 128 + j] = vv[t];
                bt[t] = bb[t];
            }
            buf[AL * 128 + j] = A;
            // Per-channel terms of the scalars, each summed over the warp (xor tree); lane 0 keeps
            // one partial per warp.  b runs through B_{s,t} for t = s, s + 1, ...
#pragma unroll
            for (int s = 0; s < kG; ++s) {
                float b = 1.f;
#pragma unroll
                for (int t = s; t < kG; ++t) {
                    if (t > s) b *= al[t];
                    const float kb = kk[s] * b;
                    float nq = qq[t] * kb, mk = kk[t] * kb;
#pragma unroll
                    for (int m = 16; m >= 1; m >>= 1) {
                        nq += __shfl_xor_sync(0xffffffffu, nq, m);
                        if (t > s) mk += __shfl_xor_sync(0xffffffffu, mk, m);
                    }
                    if (lane == 0) {
                        float* pw = buf + PART + wq * (kSerM + kSerN);
                        pw[kSerM + t * (t + 1) / 2 + s] = nq;
                        if (t > s) pw[t * (t - 1) / 2 + s] = mk;
                    }
                }
                buf[(KB + s) * 128 + j] = kk[s] * b;  // k_s B_{s,kG-1}
            }
        }
        mbar_arrive(sbar);
        if (!mbar_wait(sbar, (sph++) & 1, ab, status)) return false;
        // read pass: x_t = (k_t A_t)^T S and y_t = (q_t A_t)^T S for the four columns (partial over
        // this thread's channels, then summed over the four threads sharing the columns)
        float acc[2 * kG][4];
#pragma unroll
        for (int w = 0; w < 2 * kG; ++w)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[w][i] = 0.f;
#pragma unroll 1
        for (int p = 0; p < 4; ++p) {
            uint32_t ra[16], rb[16];
            tmem_ld16x256_x4(tA + 32 * p, ra);
            tmem_ld16x256_x4(tB + 32 * p, rb);
            tmem_ld_wait();
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int c = 32 * p + 8 * b + cq;
                // sv[e][i]: channel c + e of column jc(i)
                const float sv[2][4] = {{__uint_as_float(ra[4 * b]), __uint_as_float(ra[4 * b + 2]),
                                         __uint_as_float(rb[4 * b]), __uint_as_float(rb[4 * b + 2])},
                                        {__uint_as_float(ra[4 * b + 1]), __uint_as_float(ra[4 * b + 3]),
                                         __uint_as_float(rb[4 * b + 1]), __uint_as_float(rb[4 * b + 3])}};
#pragma unroll
                for (int w = 0; w < 2 * kG; ++w) {  // vector w: KA then QA rows of the buffer
                    const float2 cf = *reinterpret_cast<const float2*>(buf + w * 128 + c);
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[w][i] = fmaf(cf.y, sv[1][i], fmaf(cf.x, sv[0][i], acc[w][i]));
                }
            }
        }
#pragma unroll
        for (int w = 0; w < 2 * kG; ++w)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[w][i] += __shfl_xor_sync(0xffffffffu, acc[w][i], 1);
                acc[w][i] += __shfl_xor_sync(0xffffffffu, acc[w][i], 2);
            }
        if (r0 + kG < valid) load(r0 + kG);  // the next group's inputs in flight during the write pass
        // the tokens in order: u_t, o_t for the four columns (scalar i: the four warps' partials,
        // summed in a fixed order); the thread with lane % 4 = i stores column jc(i)
        float sc[kSerM + kSerN];
#pragma unroll
        for (int i = 0; i < kSerM + kSerN; ++i) {
            const float* pt = buf + PART + i;
            sc[i] = (pt[0] + pt[kSerM + kSerN]) + (pt[2 * (kSerM + kSerN)] + pt[3 * (kSerM + kSerN)]);
        }
        float u[kG][4];
#pragma unroll
        for (int t = 0; t < kG; ++t) {
            float o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float z = acc[t][i];
#pragma unroll
                for (int s = 0; s < t; ++s) z = fmaf(sc[t * (t - 1) / 2 + s], u[s][i], z);
                u[t][i] = bt[t] * (buf[(VV + t) * 128 + j0 + 8 * i] - z);
                o[i] = acc[kG + t][i];
#pragma unroll
                for (int s = 0; s <= t; ++s) o[i] = fmaf(sc[kSerM + t * (t + 1) / 2 + s], u[s][i], o[i]);
            }
            if (r0 + t < valid) {
                const int sel = lane & 3;
                const float os = sel == 0 ? o[0] : sel == 1 ? o[1] : sel == 2 ? o[2] : o[3];
                const size_t off = ((size_t)(row0 + r0 + t) * H + h) * kD + j0 + 8 * sel;
                if constexpr (sizeof(Tout) == 2)
                    out[off] = __float2bfloat16_rn(os);
                else
                    out[off] = os;
            }
        }
        // write pass: S <- A_{kG-1} . S + sum_s (k_s B_{s,kG-1}) u_s
#pragma unroll 1
        for (int p = 0; p < 4; ++p) {
            uint32_t ra[16], rb[16];
            tmem_ld16x256_x4(tA + 32 * p, ra);
            tmem_ld16x256_x4(tB + 32 * p, rb);
            tmem_ld_wait();
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int c = 32 * p + 8 * b + cq;
                const float2 a = *reinterpret_cast<const float2*>(buf + AL * 128 + c);
                float2 kb[kG];
#pragma unroll
                for (int s2 = 0; s2 < kG; ++s2) kb[s2] = *reinterpret_cast<const float2*>(buf + (KB + s2) * 128 + c);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t* r = i < 2 ? ra : rb;
                    const int o0 = 4 * b + 2 * (i & 1);  // channel c of column jc(i); c + 1 follows
                    float s0 = a.x * __uint_as_float(r[o0]), s1 = a.y * __uint_as_float(r[o0 + 1]);
#pragma unroll
                    for (int s2 = 0; s2 < kG; ++s2) {
                        s0 = fmaf(kb[s2].x, u[s2][i], s0);
                        s1 = fmaf(kb[s2].y, u[s2][i], s1);
                    }
                    r[o0] = __float_as_uint(s0);
                    r[o0 + 1] = __float_as_uint(s1);
                }
            }
            tmem_st16x256_x4(tA + 32 * p, ra);
            tmem_st16x256_x4(tB + 32 * p, rb);
        }
        tmem_st_wait();  // the next group reads these columns back
    }
    return true;
}

// ROB: the instantiation that recomputes the units the first pass marked in `redo`
// (every other unit returns at once), taking each chunk beyond the fp16 range through
// the exact per-token path; without it, the kernel marks such units in `redo`.
// SG: one log-decay per (token, head) (the scalar gate of Gated DeltaNet), or none at
// all (DeltaNet, alpha = 1) when P.log_alpha is null.  The gates then come in with beta
// through the beta loader, and the TMA ring carries q, k and v only.
// PB: the state pool holds bf16 states (a separate instantiation, so that the common
// kernels' code is not touched by it).
template <typename Tin, typename Tout, bool SG, bool PB, bool ROB>
__global__ void __launch_bounds__(NTHREADS, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_la,
                 const __grid_constant__ CUtensorMap tm_out, const SeqProblem P, const PoolSlots pool,
                 int* __restrict__ redo) {
    using L = Cfg<Tin>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::OFF_MISC);
    volatile int* range_bad = reinterpret_cast<volatile int*>(sm + L::OFF_MISC + 8);  // ROB = false
    Abort* ab = reinterpret_cast<Abort*>(sm + L::OFF_MISC + 16);
    float* vec_a = reinterpret_cast<float*>(sm + L::OFF_VEC);         // [3][128] e^{ref}
    float* vec_b = reinterpret_cast<float*>(sm + L::OFF_VEC + 1536);  // [3][128] e^{g_63 - ref}
    float* sbeta = reinterpret_cast<float*>(sm + L::OFF_BETA);        // [4][64]
    float* sgate = reinterpret_cast<float*>(sm + L::OFF_GATE);        // [4][64] (SG)
    float* ones = reinterpret_cast<float*>(sm + L::OFF_ONES);         // [128] 1.0f
    int* cbad = reinterpret_cast<int*>(sm + L::OFF_CBAD);             // [3][4]: per prep warp, by chunk % 3
#ifdef KDA_TRACE
    unsigned int* trace_sm = reinterpret_cast<unsigned int*>(sm + L::OFF_MISC + 64);
#endif

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int unit = blockIdx.x;
    if (pool.claim) {
        // A launch of at most kPackUnits units, one CTA per SM: each CTA claims the next unit, and
        // CTAs on SMs with an ID of at least the unit count wait a moment first, so that the units
        // land on the SMs with the lowest IDs.  Every CTA claims once, so every unit is taken
        // whatever the placement.
        __shared__ int claimed;
        if (tid == 0) {
            unsigned id;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
            if (id >= (unsigned)(P.N * P.H)) {
                const long long tw = clock64();
                while (clock64() - tw < kClaimDelay) {
                }
            }
            claimed = atomicAdd(pool.claim + (ROB ? 1 : 0), 1);
        }
        __syncthreads();
        unit = claimed;
        if (unit >= P.N * P.H) return;
    }
    const int h = unit % P.H;
    // Packed sequences of different lengths: CTAs are handed out longest sequence first
    // (CTA u takes the sequence of length rank u / H), so that the longest chains start
    // first and the short ones fill in behind them.  Every CTA ranks the lengths itself
    // (up to kLptMax sequences; beyond that, in order of appearance).
    int s = unit / P.H;
    if (P.cu_seqlens && P.N > 1 && P.N <= kLptMax) {
        int64_t* cul = reinterpret_cast<int64_t*>(sm + L::OFF_RING);  // scratch before the ring is used
        int* pick = reinterpret_cast<int*>(sm + L::OFF_RING + 8 * (kLptMax + 1));
        for (int i = threadIdx.x; i <= P.N; i += NTHREADS) cul[i] = P.cu_seqlens[i];
        __syncthreads();
        for (int i = threadIdx.x; i < P.N; i += NTHREADS) {
            const int64_t li = cul[i + 1] - cul[i];
            int rank = 0;
            for (int q = 0; q < P.N; ++q) {
                const int64_t lq = cul[q + 1] - cul[q];
                rank += (lq > li) || (lq == li && q < i);
            }
            if (rank == s) *pick = i;
        }
        __syncthreads();
        s = *pick;
        __syncthreads();
    }
    if constexpr (ROB)
        if (!redo[(size_t)s * P.H + h]) return;  // every chunk of this unit was within range
    int64_t t0, len;
    seq_bounds(P, s, t0, len);
    const int nch = (int)((len + C - 1) / C);
    const size_t sbase = ((size_t)s * P.H + h) * kD * kD;
    // this unit's initial state (null: zeros), looked up where it is read; with a bf16 pool
    // the pointer addresses bf16 entries, which init_at widens
    auto init_state = [&]() -> const float* {
        if (!pool.init_slots) return P.init ? P.init + sbase : nullptr;
        const int64_t slot = checked_slot(pool.init_slots[s], pool.n_slots, P.status);
        if constexpr (PB)
            return slot >= 0 ? reinterpret_cast<const float*>(reinterpret_cast<const __nv_bfloat16*>(P.init) +
                                                              ((size_t)slot * P.H + h) * kD * kD)
                             : nullptr;
        else
            return slot >= 0 ? P.init + ((size_t)slot * P.H + h) * kD * kD : nullptr;
    };
    auto init_at = [&](const float* S0, size_t i) -> float {
        if constexpr (PB)
            return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(S0)[i]);
        else
            return S0[i];
    };

    if (nch == 0) {  // empty sequence: the final state is the initial state
        if constexpr (!ROB)
            if (tid == 0) redo[(size_t)s * P.H + h] = 0;
        if (P.final_state) {
            const float* S0 = init_state();
            for (int i = tid; i < kD * kD; i += NTHREADS) P.final_state[sbase + i] = S0 ? init_at(S0, i) : 0.f;
        }
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < L::NSLOT; ++i) {
            mbar_init(&bar[B_FULL + i], 1);
            mbar_init(&bar[B_EMPTY + i], 128);
        }
        const int c128[] = {B_PREPD, B_PREPD + 1, B_P2D, B_TB, B_WRDY, B_XRDY, B_URDY, B_OFREE, B_STG};
        for (int i : c128) mbar_init(&bar[i], 128);
        const int c1[] = {B_GDONE,  B_WYDONE,   B_V16FREE,    B_V16FREE + 1, B_UIDONE,
                          B_SDONE,  B_KQFREE,   B_KQFREE + 1, B_STGFREE,     B_STGFREE + 1};
        for (int i : c1) mbar_init(&bar[i], 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&bar[B_BFULL + i], 32);
            mbar_init(&bar[B_BFREE + i], SG ? 256 : 128);  // SG: prep reads the gates too
        }
        for (int i = 0; i < 3; ++i) mbar_init(&bar[B_VFREE + i], 128);
        mbar_init(&bar[B_STGR], 1);
        mbar_init(&bar[B_PDONE], 128);
        mbar_init(&bar[B_SER], 128);
        mbar_init(&bar[B_NRD], 128);
        ab->flag = 0;
        *range_bad = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(tmem_holder, 512);
    if constexpr (ROB)
        if (tid < 128) ones[tid] = 1.f;
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
    constexpr uint32_t ID_SO = idesc_f16(128, 192, 0, 0);  // [D_S | D_O]: D_O follows D_S in TMEM
    // Every product group is issued by one thread after waiting for its inputs and for the
    // previous reader of its accumulator; the commits below are what the other roles wait on.
    // WY products of chunk n, once V16/KT of the chunk are ready and the state update of
    // chunk n - 1 has consumed U16 (NR complete is the caller's wait).
    auto issue_wy = [&](int n) -> bool {
        const int b = n & 1;
        if (!mbar_wait(&bar[B_PREPD + b], (n >> 1) & 1, ab, status)) return false;
        if (n > 0 && !mbar_wait(&bar[B_SDONE], (n - 1) & 1, ab, status)) return false;
        tc_fence_after();
        KDA_TR(n, 22);
        const uint64_t dkt = k_desc(sm_base + L::OFF_KQ + b * 32768), dnr = k_desc(sm_base + L::OFF_NR);
        const uint32_t v16 = tmem + TM_V16 + b * 32;
#pragma unroll
        for (int st = 0; st < 4; ++st) {
            mma_ss(tmem + TM_W, dkt + 2u * st, dnr + 2u * st, ID_KK, st > 0);
            mma_ts(tmem + TM_U, v16 + st * 8, dnr + 2u * st, ID_KK, st > 0);
        }
        mma_commit(&bar[B_WYDONE]);
        mma_commit(&bar[B_V16FREE + b]);
        KDA_TR(n, 8);
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v);
            if constexpr (!SG) prefetch_tmap(&tm_la);
            prefetch_tmap(&tm_out);
            int issued = 0;
            bool ok = true;
            // The ring holds only a few slots, so every tile is first pulled into L2
            // kPf quarters ahead of its load (DRAM latency would otherwise stall prep).
            constexpr int kPf = 8;
            const int nq = (int)((len + QR - 1) / QR);
            auto prefetch = [&](int g) {
                const int z = (int)(t0 + (int64_t)QR * g);
                tma_prefetch_3d(&tm_q, 0, h, z);
                tma_prefetch_3d(&tm_k, 0, h, z);
                tma_prefetch_3d(&tm_v, 0, h, z);
                if constexpr (!SG) tma_prefetch_3d(&tm_la, 0, h, z);
            };
            for (int g = L::NSLOT; g < kPf && g < nq; ++g) prefetch(g);
            for (int n = 0; n < nch && ok; ++n)
                for (int i = 0; i < 4 && ok; ++i) {
                    const int q = i < 2 ? 1 - i : i;  // the order prep consumes them: 1, 0, 2, 3
                    const int g = 4 * n + i, sl = g % L::NSLOT, use = g / L::NSLOT;
                    if (g + kPf < nq) prefetch(g + kPf);
                    if (use > 0 && !(ok = mbar_wait(&bar[B_EMPTY + sl], (use - 1) & 1, ab, status))) break;
                    uint8_t* slot = sm + L::OFF_RING + sl * L::SLOT_BYTES;
                    mbar_arrive_expect_tx(&bar[B_FULL + sl], SG ? L::SLOT_LA : L::SLOT_BYTES);
                    const int z = (int)(t0 + (int64_t)C * n + QR * q);
                    tma_load_3d(slot + L::SLOT_Q, &tm_q, &bar[B_FULL + sl], 0, h, z);
                    tma_load_3d(slot + L::SLOT_K, &tm_k, &bar[B_FULL + sl], 0, h, z);
                    tma_load_3d(slot + L::SLOT_V, &tm_v, &bar[B_FULL + sl], 0, h, z);
                    if constexpr (!SG) tma_load_3d(slot + L::SLOT_LA, &tm_la, &bar[B_FULL + sl], 0, h, z);
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
            for (int i = lane; i < C; i += 32) {
                const size_t row = (size_t)(t0 + (int64_t)C * m + i) * P.H + h;
                sbeta[k4 * 64 + i] = i < vld ? P.beta[row] : 0.f;
                if constexpr (SG) sgate[k4 * 64 + i] = (i < vld && P.log_alpha) ? P.log_alpha[row] : 0.f;
            }
            mbar_arrive(&bar[B_BFULL + k4]);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ Gram issuer
        // the Gram of each chunk, once all its operand rows are ready and the tri warpgroup has
        // read out the previous one (D_G free)
        if (lane == 0)
            for (int n = 0; n < nch; ++n) {
                const int b = n & 1;
                if (!mbar_wait(&bar[B_PREPD + b], (n >> 1) & 1, ab, status)) break;
                if (n > 0 && !mbar_wait(&bar[B_P2D], (n - 1) & 1, ab, status)) break;
                tc_fence_after();
                const uint64_t da = mn_desc(sm_base + L::OFF_KQ + b * 32768, 16384);
                const uint64_t db = mn_desc(sm_base + L::OFF_KH + b * L::KHP, 8192);
#pragma unroll
                for (int st = 0; st < 8; ++st) mma_ss(tmem + TM_G, da + 128u * st, db + 128u * st, ID_G, st > 0);
                mma_commit(&bar[B_GDONE]);
                KDA_TR(n, 3);
            }
    } else if (warp == 3) {
        // ------------------------------------------------------------ WY issuer (first pass)
        // the WY products of each chunk, once NR is written, V16/KT of the chunk are ready and
        // the state update of the previous chunk has consumed U16
        if constexpr (!ROB)
            if (lane == 0)
                for (int n = 0; n < nch; ++n) {
                    if (!mbar_wait(&bar[B_NRD], n & 1, ab, status)) break;
                    if (!issue_wy(n)) break;
                }
    } else if (warp < 8) {
        // ------------------------------------------------------------ prep warpgroup
        const int c = tid - 128;  // key channel (and TMEM lane) of this thread
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        float max_x = 0.f;  // largest |g - ref| of the chunk (log2 units), for the range check

        // prep1(n): decay cumsum, operand tiles KT/QT/KH, V16, decay vectors.
        // Rows past the end of a sequence get log alpha = 0 and k = 0 (their beta
        // is 0 too), which makes them identity steps; q and v of such rows only
        // reach outputs that are never stored.
        auto prep1 = [&](int n) -> bool {
            const int b = n & 1, v3 = n % 3;
            if (c == 0) KDA_TR(n, 0);
            if (n >= 2) {  // the buffers of chunk n - 2
                const uint32_t par = ((n - 2) >> 1) & 1;
                if (!mbar_wait(&bar[B_KQFREE + b], par, ab, status)) return false;  // KT/QT/KH (products)
                if (c == 0) KDA_TR(n, 18);
                if constexpr (!L::STG_OWN)  // KT/QT also staged the output of chunk n - 2
                    if (!mbar_wait(&bar[B_STGFREE + b], par, ab, status)) return false;
                if (c == 0) KDA_TR(n, 19);
                if (!mbar_wait(&bar[B_V16FREE + b], par, ab, status)) return false;  // V16 (WY products)
                if (c == 0) KDA_TR(n, 20);
            }
            if (n >= 3 && !mbar_wait(&bar[B_VFREE + v3], ((n - 3) / 3) & 1, ab, status)) return false;
            if (c == 0) KDA_TR(n, 21);
            tc_fence_after();
            const int valid = (int)((len - (int64_t)C * n) < C ? (len - (int64_t)C * n) : C);
            uint8_t* kt = sm + L::OFF_KQ + b * 32768;
            uint8_t* qt = kt + 16384;
            uint8_t* kh = sm + L::OFF_KH + b * L::KHP;
            // Quarters in the order 1, 0 (rows 31 down to 0), 2, 3 (rows 32 up to 63), one ring
            // slot each.  Relative to ref = g_31: rows r <= 31 use x_r = g_r - ref =
            // -(L_{r+1} + .. + L_31), accumulated downwards from row 31 (which also yields
            // ref = L_0 + .. + L_31); rows r >= 32 use x_r = L_32 + .. + L_r (L = log2 alpha).
            const float* sg = sgate + (n & 3) * 64;  // SG: this chunk's gates
            if constexpr (SG)
                if (!mbar_wait(&bar[B_BFULL + (n & 3)], (n >> 2) & 1, ab, status)) return false;
            auto wait_slot = [&](int i) {
                const int g = 4 * n + i;
                return mbar_wait(&bar[B_FULL + g % L::NSLOT], (g / L::NSLOT) & 1, ab, status);
            };
            const bool full = valid == C;
            float x = 0.f;
            if constexpr (ROB) max_x = 0.f;  // per chunk; otherwise over the whole unit
            // g decreases monotonically (log alpha <= 0), so |x| is largest at a quarter's
            // first or last row: the range check looks at those.
            auto quarter = [&](int i, auto full_chunk, auto reverse) {
                constexpr bool FULL = decltype(full_chunk)::value, REV = decltype(reverse)::value;
                const int q = REV ? 1 - i : i;
                const uint8_t* sl = sm + L::OFF_RING + ((4 * n + i) % L::NSLOT) * L::SLOT_BYTES;
                [[maybe_unused]] const float* sla = reinterpret_cast<const float*>(sl + L::SLOT_LA);  // !SG only
                const Tin* sk = reinterpret_cast<const Tin*>(sl + L::SLOT_K);
                const Tin* sq = reinterpret_cast<const Tin*>(sl + L::SLOT_Q);
                const Tin* sv = reinterpret_cast<const Tin*>(sl + L::SLOT_V);
                const int vq = valid - QR * q;  // rows of this quarter inside the sequence
                uint32_t pk[8], pq[8], ph[8], pv[8];
#pragma unroll
                for (int ps = 0; ps < QR / 2; ++ps) {
                    const int rp = REV ? QR / 2 - 1 - ps : ps;
                    float kk[2], qq[2], e1[2], e2[2], vv2[2];
#pragma unroll
                    for (int es = 0; es < 2; ++es) {
                        const int e = REV ? 1 - es : es;
                        const int rr = 2 * rp + e;
                        const bool on = FULL || rr < vq;
                        float la;
                        if constexpr (SG)
                            la = on ? sg[QR * q + rr] : 0.f;
                        else
                            la = on ? sla[rr * 128 + c] : 0.f;
                        kk[e] = on ? ld_in(sk, rr * 128 + c) : 0.f;
                        qq[e] = ld_in(sq, rr * 128 + c);
                        vv2[e] = ld_in(sv, rr * 128 + c);
                        float xu;
                        if (REV) {
                            xu = x;
                            x = fmaf(-la, kLog2e, x);
                        } else {
                            x = fmaf(la, kLog2e, x);
                            xu = x;
                        }
                        if ((ps == 0 && es == 0) || (ps == QR / 2 - 1 && es == 1)) max_x = fmaxf(max_x, fabsf(xu));
                        e1[e] = fast_exp2(xu);
                        e2[e] = fast_exp2(-xu);
                    }
                    pk[rp] = pack_half2(kk[0] * e1[0], kk[1] * e1[1]);
                    pq[rp] = pack_half2(qq[0] * e1[0], qq[1] * e1[1]);
                    ph[rp] = pack_half2(kk[0] * e2[0], kk[1] * e2[1]);
                    pv[rp] = pack_half2(vv2[0], vv2[1]);
                }
                mbar_arrive(&bar[B_EMPTY + (4 * n + i) % L::NSLOT]);
#pragma unroll
                for (int g8 = 0; g8 < 2; ++g8) {
                    const uint32_t off = sw128(c, 2 * q + g8);
                    *reinterpret_cast<uint4*>(kt + off) = make_uint4(pk[4 * g8], pk[4 * g8 + 1], pk[4 * g8 + 2], pk[4 * g8 + 3]);
                    *reinterpret_cast<uint4*>(qt + off) = make_uint4(pq[4 * g8], pq[4 * g8 + 1], pq[4 * g8 + 2], pq[4 * g8 + 3]);
                    *reinterpret_cast<uint4*>(kh + off) = make_uint4(ph[4 * g8], ph[4 * g8 + 1], ph[4 * g8 + 2], ph[4 * g8 + 3]);
                }
                tmem_st8(tmem + lane_base + TM_V16 + b * 32 + q * 8, pv);
            };
            float ref = 0.f;
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                if (!wait_slot(i)) return false;
                if (i == 2) {  // first half done: ref = -x, and the second half restarts at row 32
                    ref = -x;
                    x = 0.f;
                }
                if (i < 2) {
                    if (full)
                        quarter(i, std::true_type{}, std::true_type{});
                    else
                        quarter(i, std::false_type{}, std::true_type{});
                } else {
                    if (full)
                        quarter(i, std::true_type{}, std::false_type{});
                    else
                        quarter(i, std::false_type{}, std::false_type{});
                }
                if (c == 0 && i == 1) KDA_TR(n, 29);
            }
            if constexpr (SG) mbar_arrive(&bar[B_BFREE + (n & 3)]);  // done with this chunk's gates
            vec_a[v3 * 128 + c] = fast_exp2(ref);
            vec_b[v3 * 128 + c] = fast_exp2(x);  // e^{g_63 - ref}
            if constexpr (ROB) {  // does any key channel of this warp leave the fp16 range in this chunk?
                const unsigned bad = __ballot_sync(0xffffffffu, !(max_x <= kMaxExp2));  // (NaN: yes)
                if ((c & 31) == 0) cbad[v3 * 4 + (warp & 3)] = bad != 0u;
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar[B_PREPD + b]);
            if (c == 0) KDA_TR(n, 2);
            return true;
        };
        for (int n = 0; n < nch; ++n)
            if (!prep1(n)) break;
        if constexpr (!ROB) {  // mark the unit for the exact pass (NaN: yes), before the state reads it
            if (!(max_x <= kMaxExp2)) *range_bad = 1;
            mbar_arrive(&bar[B_PDONE]);
        }
    } else if (warp < 12) {
        // ------------------------------------------------------------ state warpgroup
        const int j = tid - 256;  // value column (and TMEM lane) of this thread
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        Tout* out = static_cast<Tout*>(P.out);
        bool ok = true;
        uint32_t ph_stg = 0;    // phase of the staging barrier (every thread waits on it)
        uint32_t ph_ser = 0;    // phase of the exact path's barrier
        bool u_issued = false;  // (i) of the coming chunk already issued (thread 0)
        // chunk m goes the exact per-token way (read once prep(m) has arrived on B_PREPD)
        auto bad_chunk = [&](int m) -> bool {
            if constexpr (!ROB) return false;
            const volatile int* cb = cbad + (m % 3) * 4;
            return (cb[0] | cb[1] | cb[2] | cb[3]) != 0;
        };
        // (i): U += X16 x WT for chunk m, once X_m and WT(m) are ready (thread 0)
        auto issue_u = [&](int m) -> bool {
            if (!mbar_wait(&bar[B_XRDY], m & 1, ab, status)) return false;
            if (!mbar_wait(&bar[B_WRDY], m & 1, ab, status)) return false;
            tc_fence_after();
            KDA_TR(m, 24);
            const uint64_t db = mn_desc(sm_base + L::OFF_WT, 8192);
            if (!bad_chunk(m)) {
#pragma unroll
                for (int st = 0; st < 8; ++st) mma_ts(tmem + TM_U, tmem + TM_X16 + st * 8, db + 128u * st, ID_MN, 1);
            }
            mma_commit(&bar[B_UIDONE]);
            KDA_TR(m, 10);
            return true;
        };
        // (iii-a): O = X16 x QT for chunk m, once O of chunk m - 1 has been read out (thread 0)
        auto issue_o = [&](int m) -> bool {
            if (m > 0 && !mbar_wait(&bar[B_OFREE], (m - 1) & 1, ab, status)) return false;
            tc_fence_after();
            const uint64_t db = mn_desc(sm_base + L::OFF_KQ + (m & 1) * 32768 + 16384, 8192);
            if (!bad_chunk(m)) {
#pragma unroll
                for (int st = 0; st < 8; ++st)
                    mma_ts(tmem + TM_O, tmem + TM_X16 + st * 8, db + 128u * st, ID_MN, st > 0);
            }
            KDA_TR(m, 11);
            return true;
        };
        {  // X_0 = Diag(a_0) S_0 into D_S and X16
            const float* S0 = init_state();
            if (!(ok = mbar_wait(&bar[B_PREPD], 0, ab, status))) goto state_done;
            const float* a0 = ROB && bad_chunk(0) ? ones : vec_a;  // the exact path works on S itself
#pragma unroll 1
            for (int piece = 0; piece < 4; ++piece) {
                uint32_t xs[32], x16[16];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int cc = piece * 32 + e;
                    const float s0 = S0 ? init_at(S0, (size_t)cc * kD + j) : 0.f;
                    xs[e] = __float_as_uint(s0 * a0[cc]);
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
            if (j == 0 && !(ok = issue_u(0) && issue_o(0))) goto state_done;
        }
        for (int n = 0; n < nch; ++n) {
            const int b = n & 1;
            const int valid = (int)((len - (int64_t)C * n) < C ? (len - (int64_t)C * n) : C);
            const bool last = (n + 1 == nch);
            // S2(n): U16 = fp16(U^T).  Thread 0 first hands back the buffer that staged
            // the previous chunk's output, once the bulk store has read it, and issues
            // (i) of this chunk if WT was not ready earlier.
            if (j == 0 && n > 0) {
                bulk_wait_read<0>();
                if constexpr (L::STG_OWN)
                    mbar_arrive(&bar[B_STGR]);
                else
                    mbar_arrive(&bar[B_STGFREE + ((n - 1) & 1)]);
                if (!u_issued && !(ok = issue_u(n))) break;
                u_issued = false;
            }
            if (!(ok = mbar_wait(&bar[B_UIDONE], n & 1, ab, status))) break;
            tc_fence_after();
            if (j == 0) KDA_TR(n, 12);
            {
                uint32_t r0[32], r1[32], u16[32];
                tmem_ld32(tmem + lane_base + TM_U, r0);
                tmem_ld32(tmem + lane_base + TM_U + 32, r1);
                tmem_ld_wait();
                if (j == 0) KDA_TR(n, 25);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    u16[e] = pack_half2(__uint_as_float(r0[2 * e]), __uint_as_float(r0[2 * e + 1]));
                    u16[16 + e] = pack_half2(__uint_as_float(r1[2 * e]), __uint_as_float(r1[2 * e + 1]));
                }
                tmem_st32(tmem + lane_base + TM_U16, u16);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bar[B_URDY]);
                if (j == 0) {  // (ii) state update and (iii-b) the intra-chunk part of the output
                    if (!(ok = mbar_wait(&bar[B_URDY], n & 1, ab, status))) break;
                    tc_fence_after();
                    // one product: [D_S | D_O] += U16 x [KH | PP] (N = 192; PP follows KH)
                    const uint64_t dkp = k_desc(sm_base + L::OFF_KH + b * L::KHP);
                    if (!bad_chunk(n)) {
#pragma unroll
                        for (int st = 0; st < 4; ++st)
                            mma_ts(tmem + TM_S, tmem + TM_U16 + st * 8, dkp + 2u * st, ID_SO, 1);
                    }
                    mma_commit(&bar[B_SDONE]);
                    mma_commit(&bar[B_KQFREE + b]);
                    KDA_TR(n, 13);
                }
            }
            // S3(n): the state (snapshots, final state, next X: the chain continues from
            // there), then the output of the chunk.
            if (!(ok = mbar_wait(&bar[B_SDONE], n & 1, ab, status))) break;
            tc_fence_after();
            if (j == 0) KDA_TR(n, 14);
            const bool bad = ROB && bad_chunk(n);
            if (bad) {  // the exact per-token path on D_S = S (no product of this chunk touched it)
                uint8_t* stage = sm + (L::STG_OWN ? L::OFF_STG : L::OFF_KQ + b * 32768);
                if constexpr (L::STG_OWN)  // the previous chunk's bulk store has read the buffer
                    if (n > 0 && !(ok = mbar_wait(&bar[B_STGR], (n - 1) & 1, ab, status))) break;
                if (j == 0) KDA_TR(n, 1);
                if (!(ok = serial_chunk<Tin, Tout, SG>(tmem + lane_base + TM_S, j, t0 + (int64_t)C * n, valid, h,
                                                       P.H, static_cast<const Tin*>(P.q),
                                                       static_cast<const Tin*>(P.k), static_cast<const Tin*>(P.v),
                                                       P.log_alpha, P.beta, static_cast<Tout*>(P.out),
                                                       reinterpret_cast<float*>(stage), &bar[B_SER], ph_ser, ab,
                                                       status)))
                    break;
                if (j == 0) KDA_TR(n, 28);
            }
            {
                const int64_t end_pos = (int64_t)C * n + valid;  // tokens of the sequence consumed so far
                float* snap = nullptr;
                __nv_bfloat16* snap16 = nullptr;  // snapshot into a bf16 pool
                if (P.snap_interval > 0 && valid == C && end_pos % P.snap_interval == 0) {
                    int64_t slot = P.snap_offsets[s] + end_pos / P.snap_interval - 1;
                    if (pool.snap_slots) slot = checked_slot(pool.snap_slots[slot], pool.n_slots, P.status);
                    if constexpr (PB) {
                        if (slot >= 0 && P.snapshots)
                            snap16 = reinterpret_cast<__nv_bfloat16*>(P.snapshots) + ((size_t)slot * P.H + h) * kD * kD;
                    } else {
                        if (slot >= 0 && P.snapshots) snap = P.snapshots + ((size_t)slot * P.H + h) * kD * kD;
                    }
                }
                float* fin = (last && P.final_state) ? P.final_state + sbase : nullptr;
                if constexpr (!ROB) {
                    // A unit marked for the exact pass is recomputed from its initial state, which
                    // the final state may alias: it must not be overwritten here.
                    if (last && !(ok = mbar_wait(&bar[B_PDONE], 0, ab, status))) break;
                    if (*range_bad) fin = nullptr;
                }
                const float* bv = ROB && bad ? ones : vec_b + (n % 3) * 128;
                if constexpr (PB)
                    if (snap16) store_state_bf16(snap16, tmem + lane_base + TM_S, bv, j);
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
                    if (!(ok = mbar_wait(&bar[B_PREPD + ((n + 1) & 1)], ((n + 1) >> 1) & 1, ab, status))) break;
                    const float* an = ROB && bad_chunk(n + 1) ? ones : vec_a + ((n + 1) % 3) * 128;
                    // 16x256b accesses: per block of 8 key channels a thread holds channels cq, cq + 1
                    // of four value columns (lanes lane/4 + {0, 8} of the warp's two 16-lane halves), so
                    // each pair of factors it reads serves eight elements; the fp16 pairs go back with
                    // the matching 16x128b stores (X16 column = channel / 2)
                    const int cq = 2 * (lane & 3);
                    const uint32_t tA = tmem + lane_base, tB = tA + (16u << 16);
#pragma unroll 1
                    for (int p = 0; p < 4; ++p) {
                        uint32_t ra[16], rb[16], xa[8], xb[8];
                        tmem_ld16x256_x4(tA + TM_S + 32 * p, ra);
                        tmem_ld16x256_x4(tB + TM_S + 32 * p, rb);
                        tmem_ld_wait();
                        if (j == 0 && p == 0) KDA_TR(n, 26);
#pragma unroll
                        for (int bk = 0; bk < 4; ++bk) {
                            const int cc = 32 * p + 8 * bk + cq;
                            const float2 b2 = *reinterpret_cast<const float2*>(bv + cc);
                            const float2 a2 = *reinterpret_cast<const float2*>(an + cc);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {  // e & 1: channel cc + 1
                                const float bb = (e & 1) ? b2.y : b2.x, aa = (e & 1) ? a2.y : a2.x;
                                ra[4 * bk + e] = __float_as_uint(__uint_as_float(ra[4 * bk + e]) * bb * aa);
                                rb[4 * bk + e] = __float_as_uint(__uint_as_float(rb[4 * bk + e]) * bb * aa);
                            }
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                xa[2 * bk + hh] = pack_half2(__uint_as_float(ra[4 * bk + 2 * hh]),
                                                             __uint_as_float(ra[4 * bk + 2 * hh + 1]));
                                xb[2 * bk + hh] = pack_half2(__uint_as_float(rb[4 * bk + 2 * hh]),
                                                             __uint_as_float(rb[4 * bk + 2 * hh + 1]));
                            }
                        }
                        tmem_st16x256_x4(tA + TM_S + 32 * p, ra);
                        tmem_st16x256_x4(tB + TM_S + 32 * p, rb);
                        tmem_st16x128_x4(tA + TM_X16 + 16 * p, xa);
                        tmem_st16x128_x4(tB + TM_X16 + 16 * p, xb);
                    }
                    if (j == 0) KDA_TR(n, 27);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&bar[B_XRDY]);
                    if (j == 0) KDA_TR(n, 15);
                }
                mbar_arrive(&bar[B_VFREE + (n % 3)]);
                // (i) of the next chunk now if its inputs are ready; otherwise after this
                // chunk's output is out (so that the output never waits on WT)
                if (!last && j == 0 && mbar_test(&bar[B_XRDY], (n + 1) & 1) &&
                    mbar_test(&bar[B_WRDY], (n + 1) & 1)) {
                    if (!(ok = issue_u(n + 1))) break;
                    u_issued = true;
                }
            }
            if (bad) {  // its output rows are stored already
                tc_fence_before();
                mbar_arrive(&bar[B_OFREE]);
            } else {  // O(n): read out, hand D_O back to (iii-a) of the next chunk, store
                uint32_t o0[32], o1[32];
                tmem_ld32(tmem + lane_base + TM_O, o0);
                tmem_ld32(tmem + lane_base + TM_O + 32, o1);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&bar[B_OFREE]);
                if (j == 0) KDA_TR(n, 16);
                {  // staged in shared memory; full chunks are stored by the TMA
                    Tout* stg = reinterpret_cast<Tout*>(sm + (L::STG_OWN ? L::OFF_STG : L::OFF_KQ + b * 32768));
                    if constexpr (L::STG_OWN)  // the previous chunk's bulk store has read the buffer
                        if (n > 0 && !(ok = mbar_wait(&bar[B_STGR], (n - 1) & 1, ab, status))) break;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        if constexpr (sizeof(Tout) == 2) {
                            stg[e * kD + j] = __float2bfloat16_rn(__uint_as_float(o0[e]));
                            stg[(32 + e) * kD + j] = __float2bfloat16_rn(__uint_as_float(o1[e]));
                        } else {
                            stg[e * kD + j] = __uint_as_float(o0[e]);
                            stg[(32 + e) * kD + j] = __uint_as_float(o1[e]);
                        }
                    }
                    if (valid == C) {
                        // Every thread waits, so no thread can arrive for the next chunk before
                        // all have arrived for this one.
                        fence_proxy_async_smem();
                        mbar_arrive(&bar[B_STG]);
                        if (!(ok = mbar_wait(&bar[B_STG], (ph_stg++) & 1, ab, status))) break;
                        if (j == 0) {
                            for (int q = 0; q < 4; ++q)
                                tma_store_3d(&tm_out, stg + q * QR * kD, 0, h, (int)(t0 + (int64_t)C * n + QR * q));
                            bulk_commit();
                        }
                    } else {  // partial last chunk: this thread's column of the rows inside the sequence
                        Tout* dst = out + ((size_t)(t0 + (int64_t)C * n) * P.H + h) * kD + j;
#pragma unroll 1
                        for (int e = 0; e < valid; ++e) dst[(size_t)e * P.H * kD] = stg[e * kD + j];
                    }
                }
                if (j == 0) KDA_TR(n, 17);
            }
            if (!last && j == 0 && !(ok = issue_o(n + 1))) break;  // (iii-a) of the next chunk
        }
        if (j == 0) bulk_wait_all();  // the CTA's shared memory must outlive the bulk stores
    state_done:;
    } else {
        // ------------------------------------------------------------ tri warpgroup
        const int c = tid - 384;  // TMEM lane: Gram row / key channel
        const int wi = warp - 12;
        const uint32_t lane_base = (uint32_t)(wi * 32) << 16;
        // Workspace of the inverse: the diagonal blocks A_aa in fp32 (for the substitution),
        // the blocks below them A_ab (b < a, block a(a-1)/2 + b) and Dg_a in fp16 rows of
        // kRowH bytes (for the warp-level products).
        float* adiag = reinterpret_cast<float*>(sm + L::OFF_INV);
        uint8_t* a16p = sm + L::OFF_INV + 4096;
        uint8_t* dg16p = a16p + 6 * kBlkH;
        uint8_t* nr = sm + L::OFF_NR;
        uint32_t ph_tb = 0;
        auto wg_sync = [&]() -> bool {
            tc_fence_before();
            mbar_arrive(&bar[B_TB]);
            const bool r = mbar_wait(&bar[B_TB], (ph_tb++) & 1, ab, status);
            tc_fence_after();
            return r;
        };
        // NR blocks above the diagonal are never written again: zero them once.
        for (int i = c; i < 8192 / 16; i += 128) reinterpret_cast<uint4*>(nr)[i] = make_uint4(0u, 0u, 0u, 0u);
        for (int n = 0; n < nch; ++n) {
            const int b = n & 1;
            const float* bt = sbeta + (n & 3) * 64;
            // ---- P2: read the Gram; rows 0..63 -> A (beta_r applied, strictly lower, fp32
            // blocks), rows 64..127 -> P (lower triangle including the diagonal, fp16)
            if (!mbar_wait(&bar[B_GDONE], n & 1, ab, status)) break;
            if (!mbar_wait(&bar[B_BFULL + (n & 3)], (n >> 2) & 1, ab, status)) break;
            tc_fence_after();
            if (c == 0) KDA_TR(n, 4);
            uint32_t pr[32];  // P row (c >= 64), packed fp16, written after the WY issue
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lane_base + TM_G, r0);
                tmem_ld32(tmem + lane_base + TM_G + 32, r1);
                tmem_ld_wait();
                if (c == 0) KDA_TR(n, 30);
                tc_fence_before();
                mbar_arrive(&bar[B_P2D]);
                if (c < 64) {
                    // Row c of A = beta_c G[c][:]: the blocks left of the diagonal in fp16, the
                    // diagonal block in fp32.  Only entries left of the diagonal are ever read,
                    // so nothing is masked.
                    const float br = bt[c];
                    const int a = c >> 4, i = c & 15;
#pragma unroll
                    for (int bb = 0; bb < 3; ++bb) {
                        if (bb < a) {
                            uint32_t h[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int e0 = 16 * bb + 2 * e;
                                h[e] = pack_half2(br * __uint_as_float(e0 < 32 ? r0[e0] : r1[e0 - 32]),
                                                  br * __uint_as_float(e0 + 1 < 32 ? r0[e0 + 1] : r1[e0 + 1 - 32]));
                            }
                            uint8_t* dst = a16p + (a * (a - 1) / 2 + bb) * kBlkH + i * kRowH;
                            *reinterpret_cast<uint4*>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
                            *reinterpret_cast<uint4*>(dst + 16) = make_uint4(h[4], h[5], h[6], h[7]);
                        }
                    }
#pragma unroll
                    for (int aa = 0; aa < 4; ++aa) {
                        if (aa == a) {
#pragma unroll
                            for (int e4 = 0; e4 < 4; ++e4) {
                                float w[4];
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const int e = 16 * aa + 4 * e4 + q;
                                    w[q] = br * __uint_as_float(e < 32 ? r0[e] : r1[e - 32]);
                                }
                                st4(adiag + aa * 256 + bsw(i, e4), w);
                            }
                        }
                    }
                } else {
                    const int rr = c - 64;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int e0 = 2 * e, e1 = 2 * e + 1;
                        const float v0 = __uint_as_float(e0 < 32 ? r0[e0] : r1[e0 - 32]);
                        const float v1 = __uint_as_float(e1 < 32 ? r0[e1] : r1[e1 - 32]);
                        pr[e] = pack_half2(e0 <= rr ? v0 : 0.f, e1 <= rr ? v1 : 0.f);
                    }
                }
            }
            if (!wg_sync()) break;  // A written
            if (c == 0) KDA_TR(n, 5);
            if ((c & 31) < 16) {
                // ---- diagonal blocks: column jj of Dg_a = (I + A_aa)^-1 (lane jj of warp 12 + a)
                // by right-looking substitution, one block per warp so that the four run on
                // four sub-partitions
                const int a = c >> 5, jj = c & 15;
                const float* blk = adiag + a * 256;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = (i == jj) ? 1.f : 0.f;
#pragma unroll
                for (int rr = 0; rr < 15; ++rr) {
                    const float xr = x[rr];
#pragma unroll
                    for (int i = rr + 1; i < 16; ++i) x[i] = fmaf(-blk[bsw(i, rr >> 2) + (rr & 3)], xr, x[i]);
                }
                // Dg_a in fp16 for the block products, and T diag(beta) of the diagonal block
                const int col = 16 * a + jj;
                const float bcol = bt[col];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    st_half(dg16p + a * kBlkH + i * kRowH + jj * 2, x[i]);
                    st_half(nr + sw128(16 * a + i, col >> 3) + (col & 7) * 2, x[i] * bcol);
                }
            }
            if (!wg_sync()) break;  // Dg written
            if (c == 0) KDA_TR(n, 6);
            // ---- blocks below the diagonal: warp 12 + B takes block column B (warp-level products)
            {
                const uint32_t a16 = smem_u32(a16p), dg16 = smem_u32(dg16p);
                if (wi == 0)
                    tri_column<0>(a16, dg16, nr, bt, lane);
                else if (wi == 1)
                    tri_column<1>(a16, dg16, nr, bt, lane);
                else if (wi == 2)
                    tri_column<2>(a16, dg16, nr, bt, lane);
                if (c == 0) KDA_TR(n, 31);
            }
            fence_proxy_async_smem();
            if constexpr (!ROB) {  // NR = T diag(beta) complete: warp 3 issues the WY products
                tc_fence_before();
                mbar_arrive(&bar[B_NRD]);
                if (c == 0) KDA_TR(n, 7);
                mbar_arrive(&bar[B_BFREE + (n & 3)]);
            } else {  // the exact pass issues them here (2% faster there, where every chunk takes it)
                if (!wg_sync()) break;
                if (c == 0) KDA_TR(n, 7);
                mbar_arrive(&bar[B_BFREE + (n & 3)]);
                if (c == 0 && !issue_wy(n)) break;
            }
            if (c >= 64) {  // P of this chunk beside its KH, once the products of chunk n - 2 are done with the pair
                if (n >= 2) {
                    const int m = n - 2;
                    if (!mbar_wait(&bar[B_KQFREE + (m & 1)], (m >> 1) & 1, ab, status)) break;
                }
                store_row16_packed(sm + L::OFF_KH + b * L::KHP + 16384, c - 64, pr);
            }
            // ---- P4: WT = -W^T (fp16), once the WY products are complete and (i) of
            // chunk n - 1 has consumed the previous WT
            if (!mbar_wait(&bar[B_WYDONE], n & 1, ab, status)) break;
            tc_fence_after();
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lane_base + TM_W, r0);
                tmem_ld32(tmem + lane_base + TM_W + 32, r1);
                tmem_ld_wait();
                if (c == 0) KDA_TR(n, 23);
                if (n > 0 && !mbar_wait(&bar[B_UIDONE], (n - 1) & 1, ab, status)) break;
                store_row16(sm + L::OFF_WT, c, r0, r1, 0x80008000u);  // -W^T
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar[B_WRDY]);
            if (c == 0) KDA_TR(n, 9);
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
    if constexpr (!ROB)
        if (tid == 0) redo[(size_t)s * P.H + h] = *range_bad;
#ifdef KDA_TRACE
    if (blockIdx.x == 0)
        for (int i = tid; i < kTrN * kTrEv; i += NTHREADS) g_trace[i] = trace_sm[i];
#endif
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

template <typename Tin, typename Tout, bool SG, bool PB>
cudaError_t launch_t(const SeqProblem& p, const PoolSlots& pool, int* redo, int* claim, cudaStream_t st) {
    CUtensorMap mq, mk, mv, ml, mo;
    const CUtensorMapDataType dt = sizeof(Tin) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int64_t Tt = p.T_total > 0 ? p.T_total : 1;
    if (Tt > (int64_t)0x7FFFFFFF - 2 * C) return cudaErrorInvalidValue;  // tensor-map coordinates are 32-bit
    if (!make_map(&mq, p.q, dt, sizeof(Tin), Tt, p.H) || !make_map(&mk, p.k, dt, sizeof(Tin), Tt, p.H) ||
        !make_map(&mv, p.v, dt, sizeof(Tin), Tt, p.H) ||
        (!SG && !make_map(&ml, p.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Tt, p.H)) ||
        !make_map(&mo, p.out, sizeof(Tout) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  sizeof(Tout), Tt, p.H))
        return cudaErrorInvalidValue;
    if (SG) ml = mq;  // not read
    // the pass over every unit, then the exact pass over the units it marked (its CTAs for the
    // others return at once)
    auto kern = chunk_kernel<Tin, Tout, SG, PB, false>;
    auto rob = chunk_kernel<Tin, Tout, SG, PB, true>;
    const int smem = (int)Cfg<Tin>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(rob, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)p.N * p.H;
    unsigned grid = (unsigned)units;
    PoolSlots pl = pool;
    pl.claim = nullptr;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if (units <= kPackUnits && units < sms) {  // one CTA per SM; units claimed by the lowest-numbered SMs
        if ((e = cudaMemsetAsync(claim, 0, 2 * sizeof(int), st)) != cudaSuccess) return e;
        grid = (unsigned)sms;
        pl.claim = claim;
    }
    kern<<<grid, NTHREADS, smem, st>>>(mq, mk, mv, ml, mo, p, pl, redo);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    rob<<<grid, NTHREADS, smem, st>>>(mq, mk, mv, ml, mo, p, pl, redo);
    return cudaGetLastError();
}

}  // namespace

#ifdef KDA_TRACE
extern "C" int kda_trace_read(unsigned int* host, int n) {
    const size_t cnt = (size_t)(n < kTrN * kTrEv ? n : kTrN * kTrEv);
    return cudaMemcpyFromSymbol(host, g_trace, sizeof(unsigned int) * cnt) == cudaSuccess ? 0 : 1;
}
#endif

// One int per (sequence, head): set by the first pass when the unit met a chunk beyond the
// fp16 operand range, read by the exact pass.
// [N * H] exact-pass flags, then (in the last 256 bytes) the two unit counters of a launch with
// fewer units than SMs
size_t chunk_prefill_workspace(int N, int H) {
    const size_t b = (size_t)N * H * sizeof(int);
    return ((b + 255) & ~(size_t)255) + 256;
}

template <typename Tin, typename Tout>
cudaError_t launch_gate(const SeqProblem& p, const PoolSlots& pool, bool pool_bf16, int gate, int* redo, int* claim,
                        cudaStream_t st) {
    if (pool_bf16)
        return gate != kGateChannel ? launch_t<Tin, Tout, true, true>(p, pool, redo, claim, st)
                                    : launch_t<Tin, Tout, false, true>(p, pool, redo, claim, st);
    return gate != kGateChannel ? launch_t<Tin, Tout, true, false>(p, pool, redo, claim, st)
                                : launch_t<Tin, Tout, false, false>(p, pool, redo, claim, st);
}

cudaError_t launch_chunk_prefill(const SeqProblem& p, const PoolSlots& pool, bool pool_bf16, int gate, int in_dtype,
                                 int out_dtype, void* workspace, size_t ws_bytes, cudaStream_t st) {
    if ((int64_t)p.N * p.H == 0) return cudaSuccess;
    if (!workspace || ws_bytes < chunk_prefill_workspace(p.N, p.H)) return cudaErrorInvalidValue;
    int* redo = static_cast<int*>(workspace);
    int* claim = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + chunk_prefill_workspace(p.N, p.H) - 256);
    if (in_dtype == KDA_BF16 && out_dtype == KDA_BF16)
        return launch_gate<__nv_bfloat16, __nv_bfloat16>(p, pool, pool_bf16, gate, redo, claim, st);
    if (in_dtype == KDA_BF16) return launch_gate<__nv_bfloat16, float>(p, pool, pool_bf16, gate, redo, claim, st);
    if (out_dtype == KDA_BF16) return launch_gate<float, __nv_bfloat16>(p, pool, pool_bf16, gate, redo, claim, st);
    return launch_gate<float, float>(p, pool, pool_bf16, gate, redo, claim, st);
}

}  // namespace kda
