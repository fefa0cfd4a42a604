// vc_attn.cu -- FP8 attention forward with ExpCast-FP8 and the V-Smooth mean
// restore, on tcgen05 tensor cores (sm_103a).
//
// What it computes: paper summary (paper.rainbus.top), 前置知识 "在线 softmax"
// (running max m_i, normaliser l_i, numerator A_i, rescale alpha_i) and
// 方法步骤详情 steps 3-4 (A_i <- alpha_i A_i + P_q,ij R_q,j + r_ij mu_j^T with
// r_ij the row sum of the quantized probabilities; ExpCast byte
// c = clip(Round(8(u+8)+56+beta), 0, 120)); dimensionstp.github.io 2-3 / 2-4.
//
// One CTA = two 128-row query tiles (A and B) of one (b, h), processed as two
// independent pipelines that share the K/V stages and the tensor core, so the
// softmax of one tile overlaps the matrix products of the other.  12 warps:
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: thread q*32+lane
//              of a warpgroup owns one query row (its TMEM lane) and all 128
//              keys of every key tile, so the row max needs no exchange.
//   warp 8, 9  MMA issuers of tile A and tile B (one elected lane each; the
//              first also owns TMEM).
//   warp 10    K loader: TMA loads of the two Q tiles (once) and of the K tiles
//              (ring of NSK stages).
//   warp 11    V loader: TMA loads of the V^T tiles (ring of NSV stages), the
//              row-sum operand rows and the block means (bf16 hi/lo parts).
// Tensor memory (512 columns), per tile X at base_X = X * (d + 128):
//   O_X  [base, base+d)       fp32 accumulator in residual-code units.
//   S_X  [base+d, base+d+128) fp32 scores of the current key tile.  After the
//        softmax has read them: column 0 is zeroed and receives the row sum
//        r_ij (the PV MMA has width d + 16, so its last 16 columns land on
//        S_X[0..16) and the V stage's operand row d holds E4M3 1.0); columns
//        [32, 64) hold the probability bytes (4 per column), the A operand of
//        P V.
// Per key tile j and tile X: QK^T -> softmax (max, ExpCast bytes, O rescale)
// -> P V + row sum -> softmax reads r_ij back (l, batch history) and releases
// S_X -> QK^T of tile j+1.
// Mean restore, batched: after every 16 key tiles the softmax rescales the
// batch's row sums to the current running max, splits them into bf16 hi/lo
// parts and writes them into a shared-memory A operand; the MMA warp adds
// sum_t r_t mu_t^T to O with one bf16 MMA of depth 48 (terms r_hi mu_hi +
// r_lo mu_hi + r_hi mu_lo per tile), ahead of the next QK^T, so O is complete
// before the softmax rescales it again.  The means enter in units of the
// channel's residual scale g_c (g_c = s_v[c], or 1 for a channel whose
// residual is identically 0; mu' = mu * fp32(1/g_c)), so O = g (.) A / l at
// the end.
//
// The row max of a key tile comes from the TMEM loads themselves
// (tcgen05.ld.red with max: each 32-column load also returns the maximum of
// this lane's 32 values), so the first read costs four loads and three max
// instructions; only the last, masked tile reduces in registers.
//
// ExpCast inner loop, per score: ts = sat(acc * sigma/16 + C/128) (one FFMA
// with saturation = clip to [0, 128] of t/128, exact because /128 and /16 are
// powers of two), then b = ts*128 + 1.5*2^23 (packed FFMA2) whose low byte is
// rint(t); three byte permutes pack four codes.
// The upper clip at 120 is implied while |m'| < 2^19 (t <= 119.65 + 2^-1);
// warps with a row beyond take a path with an explicit min.
#include <cstdio>
#include <type_traits>

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "vc_device.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr int kMmaWarp0 = 8;           // + X
constexpr int kKLoadWarp = 10;
constexpr int kVLoadWarp = 11;
constexpr int kThreads = 12 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kBatch = 16;             // key tiles per batched mean restore
constexpr int kMeanK = 3 * kBatch;     // bf16 depth of the mean MMA
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer in the low mantissa bits

template <int D>
struct Cfg {
    static constexpr int NSK = (D == 128) ? 3 : 5;      // K stages
    static constexpr int NSV = (D == 128) ? 3 : 5;      // V stages
    static constexpr int QB = 128 * D;
    static constexpr int KB = 128 * D;
    static constexpr int VB = (D + 16) * 128;           // d channel rows + 16 row-sum operand rows
    static constexpr uint32_t QK_SWZ = (D == 128) ? kSwizzle128B : kSwizzle64B;
    static constexpr uint32_t QK_SBO = 8 * D;  // bytes per group of 8 rows
    static constexpr int MG = 6 * 128;                  // 8 rows x 48 bf16, stored as 6 core matrices
    static constexpr int BMB = (D / 8) * MG;            // one mean-operand (B) buffer
    static constexpr int AMB = (128 / 8) * MG;          // one row-sum-operand (A) buffer
    static constexpr int OFF_Q = 0;                     // [2] Q tiles
    static constexpr int OFF_K = OFF_Q + 2 * QB;
    static constexpr int OFF_V = OFF_K + NSK * KB;
    static constexpr int OFF_BM = OFF_V + NSV * VB;     // [2] by batch parity
    static constexpr int OFF_AM = OFF_BM + 2 * BMB;     // [2] by tile X
    static constexpr int OFF_HIST = OFF_AM + 2 * AMB;   // [X][r, m][slot][row] floats
    static constexpr int OFF_BAR = OFF_HIST + 2 * 2 * kBatch * 128 * 4;
    static constexpr int NBAR = 40;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int USED = OFF_MISC + 64;
    // at least 116 KB so that exactly one CTA (and one 512-column TMEM owner) sits on an SM
    static constexpr int SMEM = ((USED > 118784) ? USED : 118784) + 1024;
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(VB % 1024 == 0 && KB % 1024 == 0 && OFF_K % 1024 == 0 && OFF_V % 1024 == 0,
                  "stages keep the swizzle alignment");
    // barrier indices
    static constexpr int B_Q = 0;
    static constexpr int B_KF = 1;               // [NSK] K stage loaded
    static constexpr int B_KE = B_KF + NSK;      // [NSK] K stage read by both QK MMAs
    static constexpr int B_VF = B_KE + NSK;      // [NSV] V stage loaded, operand rows written
    static constexpr int B_VE = B_VF + NSV;      // [NSV] V stage read by both PV MMAs
    static constexpr int B_SF = B_VE + NSV;      // [2] scores of tile X in S_X
    static constexpr int B_PF = B_SF + 2;        // [2] bytes in S_X, O_X rescaled (4 warps)
    static constexpr int B_OD = B_PF + 2;        // [2] P V of tile X complete
    static constexpr int B_SE = B_OD + 2;        // [2] row sum read back, S_X free (4 warps)
    static constexpr int B_OF = B_SE + 2;        // [2] last mean restore of tile X complete
    static constexpr int B_TD = B_OF + 2;        // [2] every MMA of tile X's issuer complete
    static constexpr int B_AMF = B_TD + 2;       // [2] mean-restore A operand of tile X written (4 warps)
    static constexpr int B_MD = B_AMF + 2;       // [2] mean-restore MMA of tile X complete
    static constexpr int NBAR_USED = B_MD + 2;
    static_assert(NBAR_USED <= NBAR, "barrier area");
    // TMEM columns
    __host__ __device__ static constexpr uint32_t base(int X) { return (uint32_t)X * (D + 128); }
    static constexpr uint32_t COL_S = D;         // S_X = base + COL_S
    static constexpr uint32_t COL_P = D + 32;    // probability bytes, 32 columns
    static_assert(2 * (D + 128) <= (int)kTmemCols, "tmem budget");
};

struct AttnParams {
    const float* sq;
    const float* sk;
    const float* sv;
    const uint16_t* mu;
    uint16_t* O;
    int64_t o_sb, o_sn, o_sh;
    int H, N, nblk;
    int64_t Npad;
    float kscale;
    float exact_margin;  // hybrid: a tile is exact if some row's tile max is within this of its running max (log2)
    int32_t* dev_status;
    uint64_t timeout_ns;
    int skip_k_tile;     // test hook: the K loader never loads (nor signals) this key tile; -1 = off
    int dbg_bh, dbg_qtile;
    float* S_dump;
    uint8_t* P_dump;
};

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Byte offset of element (n, k) of a 48-deep bf16 operand buffer: K-major, no
// swizzle, core matrices of 8 rows x 8 bf16 (16 bytes), 6 along K per group of
// 8 rows.
__device__ __forceinline__ uint32_t mo_offset(int n, int k) {
    return (uint32_t)((n >> 3) * (6 * 128) + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2);
}

// Four ExpCast bytes, packed little-endian.  ts = sat(acc k1 + k2) is t/128
// clipped to [0, 1]; ts*128 + 1.5*2^23 puts rint(t) in the low byte.
template <bool CLIP>
__device__ __forceinline__ uint32_t expcast4(const float* a, float k1, float k2) {
    const float t0 = fma_sat(a[0], k1, k2);
    const float t1 = fma_sat(a[1], k1, k2);
    const float t2 = fma_sat(a[2], k1, k2);
    const float t3 = fma_sat(a[3], k1, k2);
    const float2 b01 = __ffma2_rn(make_float2(t0, t1), make_float2(128.f, 128.f), make_float2(kMagic, kMagic));
    const float2 b23 = __ffma2_rn(make_float2(t2, t3), make_float2(128.f, 128.f), make_float2(kMagic, kMagic));
    uint32_t u0 = __float_as_uint(b01.x), u1 = __float_as_uint(b01.y);
    uint32_t u2 = __float_as_uint(b23.x), u3 = __float_as_uint(b23.y);
    if (CLIP) {
        u0 = min(u0 & 0xFFu, 120u);
        u1 = min(u1 & 0xFFu, 120u);
        u2 = min(u2 & 0xFFu, 120u);
        u3 = min(u3 & 0xFFu, 120u);
    }
    // byte permutes gather the four low bytes (c0 | c1 << 8, c2 | c3 << 8, then
    // both halves), keeping the packing off the FMA pipes
    return prmt(prmt(u0, u1, 0x0040u), prmt(u2, u3, 0x0040u), 0x5410u);
}

// Range-adaptive ExpCast (expcast = 3): beta chosen by which pair of codes of
// its octave rint(t0) falls on, t0 = acc 8 sigma + 120 - 8 m' (ExpCast's t
// without beta); each beta maximises agreement with the exp-then-cast byte
// over its piece.
constexpr float kBetaPiece0 = -0.195f, kBetaPiece1 = -0.635f, kBetaPiece2 = -0.685f, kBetaPiece3 = -0.535f;

// u: bits of rint(t0) + 1.5 * 2^23, so bits 1-2 hold the piece.
__device__ __forceinline__ float piece_beta(uint32_t u) {
    const float lo = (u & 2u) ? kBetaPiece1 : kBetaPiece0;
    const float hi = (u & 2u) ? kBetaPiece3 : kBetaPiece2;
    return (u & 4u) ? hi : lo;
}

// Four range-adaptive bytes, packed little-endian.  ts = sat(acc k1 + k2) is
// t0/128 clipped to [0, 1]; ts*128 + magic gives rint(t0) (the piece), then
// fl(ts*128 + beta) + magic gives rint(t0 + beta) in the low byte.  With
// t0 >= 0, t0 + beta > -0.5, so the byte never wraps below zero.
template <bool CLIP>
__device__ __forceinline__ uint32_t expcast4_pieces(const float* a, float k1, float k2) {
    const float t0 = fma_sat(a[0], k1, k2);
    const float t1 = fma_sat(a[1], k1, k2);
    const float t2 = fma_sat(a[2], k1, k2);
    const float t3 = fma_sat(a[3], k1, k2);
    const float2 mg = make_float2(kMagic, kMagic), c128 = make_float2(128.f, 128.f), one = make_float2(1.f, 1.f);
    const float2 k01 = __ffma2_rn(make_float2(t0, t1), c128, mg);
    const float2 k23 = __ffma2_rn(make_float2(t2, t3), c128, mg);
    const float2 b01 = make_float2(piece_beta(__float_as_uint(k01.x)), piece_beta(__float_as_uint(k01.y)));
    const float2 b23 = make_float2(piece_beta(__float_as_uint(k23.x)), piece_beta(__float_as_uint(k23.y)));
    const float2 r01 = __ffma2_rn(__ffma2_rn(make_float2(t0, t1), c128, b01), one, mg);
    const float2 r23 = __ffma2_rn(__ffma2_rn(make_float2(t2, t3), c128, b23), one, mg);
    uint32_t u0 = __float_as_uint(r01.x), u1 = __float_as_uint(r01.y);
    uint32_t u2 = __float_as_uint(r23.x), u3 = __float_as_uint(r23.y);
    if (CLIP) {
        u0 = min(u0 & 0xFFu, 120u);
        u1 = min(u1 & 0xFFu, 120u);
        u2 = min(u2 & 0xFFu, 120u);
        u3 = min(u3 & 0xFFu, 120u);
    }
    return prmt(prmt(u0, u1, 0x0040u), prmt(u2, u3, 0x0040u), 0x5410u);
}

__device__ __forceinline__ uint16_t bf16_rn_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

// This thread's 64 scores of half `hf` of the key tile, from TMEM.
__device__ __forceinline__ void load_half(uint32_t taddr, float (&a)[64]) {
    uint32_t r0[32], r1[32];
    tmem_ld32(taddr, r0);
    tmem_ld32(taddr + 32, r1);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        a[i] = __uint_as_float(r0[i]);
        a[32 + i] = __uint_as_float(r1[i]);
    }
}

// 32 columns of this thread's TMEM lane and their maximum (tcgen05.ld.red).
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float& mx) {
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31]), "=f"(mx)
        : "r"(taddr));
}

__device__ __forceinline__ float max64(const float (&a)[64]) {
    float t[22];
#pragma unroll
    for (int i = 0; i < 21; ++i) t[i] = max3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
    t[21] = a[63];
    float u[8];
#pragma unroll
    for (int i = 0; i < 7; ++i) u[i] = max3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
    u[7] = t[21];
    return max3(max3(u[0], u[1], u[2]), max3(u[3], u[4], u[5]), fmaxf(u[6], u[7]));
}

// EC: 0 exp-then-cast, 1 ExpCast, 2 hybrid (exp-then-cast on the key tiles
// that are high-weight for the warp's 32 query rows, ExpCast elsewhere),
// 3 range-adaptive ExpCast (a beta per pair of codes of the octave).
template <int D, int EC, bool VSMOOTH, bool DBG>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using C = Cfg<D>;
    constexpr int NSK = C::NSK, NSV = C::NSV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    const int bh = b * p.H + h;
    const int J = p.nblk;
    // query tiles of this CTA; with an odd tile count the last CTA's tile B
    // repeats tile A and is not stored
    const int qt0 = 2 * (int)blockIdx.x, qt1 = min(2 * (int)blockIdx.x + 1, J - 1);
    const bool has_b = 2 * (int)blockIdx.x + 1 < J;
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_Q), 1);
        for (int s = 0; s < NSK; ++s) {
            mbar_init(bar(C::B_KF + s), 1);
            mbar_init(bar(C::B_KE + s), 2);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(bar(C::B_VF + s), 1);
            mbar_init(bar(C::B_VE + s), 2);
        }
        for (int X = 0; X < 2; ++X) {
            mbar_init(bar(C::B_SF + X), 1);
            mbar_init(bar(C::B_PF + X), 4);
            mbar_init(bar(C::B_OD + X), 1);
            mbar_init(bar(C::B_SE + X), 4);
            mbar_init(bar(C::B_OF + X), 1);
            mbar_init(bar(C::B_TD + X), 1);
            mbar_init(bar(C::B_AMF + X), 4);
            mbar_init(bar(C::B_MD + X), 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    {
        // The mean operand buffers start zeroed; the 16 row-sum operand rows of
        // every V stage are constant: row d is E4M3 1.0 (0x38), rows d+1.. are 0
        // (a uniform 128-byte row is the same under the 128-byte swizzle).
        uint4* bm = reinterpret_cast<uint4*>(smem + C::OFF_BM);
        for (int i = threadIdx.x; i < (2 * C::BMB + 2 * C::AMB) / 16; i += kThreads) bm[i] = make_uint4(0, 0, 0, 0);
        for (int i = threadIdx.x; i < NSV * 128; i += kThreads) {
            const int s = i / 128, idx = i % 128;  // 16-byte chunk of the 2 KB operand rows, 8 per row
            const uint32_t v = (idx < 8) ? 0x38383838u : 0u;
            *reinterpret_cast<uint4*>(smem + C::OFF_V + s * C::VB + D * 128 + idx * 16) = make_uint4(v, v, v, v);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
    const int32_t row0 = (int32_t)((int64_t)bh * p.Npad);

    if (warp == kKLoadWarp) {
        // ------------------------------------------------------------ K loader
        if (lane == 0) {
            prefetch_tensormap(&tmQ);
            prefetch_tensormap(&tmK);
            mbar_expect_tx(bar(C::B_Q), 2 * C::QB);
            tma_load_2d(sbase + C::OFF_Q, &tmQ, 0, row0 + qt0 * 128, bar(C::B_Q));
            tma_load_2d(sbase + C::OFF_Q + C::QB, &tmQ, 0, row0 + qt1 * 128, bar(C::B_Q));
            mbar_arrive(bar(C::B_Q));
        }
        int issued = 0;
        for (int j = 0; j < J; ++j) {
            const int s = j % NSK;
            if (j >= NSK && !mbar_wait_warp(bar(C::B_KE + s), (j / NSK - 1) & 1, abort_flag, p.dev_status, tmo))
                break;
            if (lane == 0 && j != p.skip_k_tile) {
                mbar_expect_tx(bar(C::B_KF + s), C::KB);
                tma_load_2d(sbase + C::OFF_K + s * C::KB, &tmK, 0, row0 + j * 128, bar(C::B_KF + s));
                mbar_arrive(bar(C::B_KF + s));
            }
            issued = j + 1;
        }
        // let this CTA's own copies in flight land before the CTA can exit
        for (int j = (issued > NSK ? issued - NSK : 0); j < issued; ++j)
            if (j != p.skip_k_tile) drain_wait(bar(C::B_KF + j % NSK), (j / NSK) & 1, tmo);
        drain_wait(bar(C::B_Q), 0, tmo);
    } else if (warp == kVLoadWarp) {
        // ------------------------------------------------------------ V loader
        constexpr int PER = D / 32;  // channels per lane for the mean operand
        float ginv[PER];             // 1 / g_c, g_c = s_v[c] (1 for an all-zero residual channel)
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const float sv = __ldg(p.sv + (int64_t)bh * D + lane * PER + e);
            ginv[e] = __frcp_rn(sv > 0.f ? sv : 1.f);
        }
        if (lane == 0) prefetch_tensormap(&tmV);
        // Mean operand of batch bt (key tiles 16 bt .. 16 bt + 15) into buffer
        // bt & 1: for channel n the 48 bf16 at k = 3t, 3t+1, 3t+2 hold
        // (mu'_hi, mu'_hi, mu'_lo) of tile t, mu' = mu / g; tiles past the
        // last are 0.  Written in halves of 8 tiles (3 chunks of 16 bytes per
        // channel each), with one proxy fence per batch.
        auto write_batch = [&](int bt) {
            uint8_t* bmb = smem + C::OFF_BM + (bt & 1) * C::BMB;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                uint32_t mw[8][PER / 2];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int jt = bt * kBatch + hb * 8 + t;
                    const uint32_t* src =
                        reinterpret_cast<const uint32_t*>(p.mu + ((int64_t)bh * p.nblk + jt) * D + lane * PER);
#pragma unroll
                    for (int e = 0; e < PER / 2; ++e) mw[t][e] = (jt < J) ? __ldg(src + e) : 0u;
                }
#pragma unroll
                for (int e = 0; e < PER; ++e) {
                    uint16_t v[24];  // k = 24 hb .. 24 hb + 23
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const uint32_t bits = (e & 1) ? (mw[t][e / 2] >> 16) : (mw[t][e / 2] & 0xFFFFu);
                        const float mp = __fmul_rn(bf16_bits_to_f32(bits), ginv[e]);
                        const uint16_t hi = bf16_rn_bits(mp);
                        const uint16_t lo = bf16_rn_bits(__fsub_rn(mp, bf16_bits_to_f32(hi)));
                        v[3 * t] = hi;
                        v[3 * t + 1] = hi;
                        v[3 * t + 2] = lo;
                    }
                    const int n_ch = lane * PER + e;
#pragma unroll
                    for (int c = 0; c < 3; ++c) {
                        uint32_t w4[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) w4[q] = (uint32_t)v[8 * c + 2 * q] | ((uint32_t)v[8 * c + 2 * q + 1] << 16);
                        *reinterpret_cast<uint4*>(bmb + mo_offset(n_ch, 24 * hb + 8 * c)) =
                            make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
            fence_proxy_async_smem();  // the generic-proxy writes above are read by the MMAs
        };
        int issued = 0;
        for (int j = 0; j < J; ++j) {
            const int s = j % NSV;
            if (j >= NSV && !mbar_wait_warp(bar(C::B_VE + s), (j / NSV - 1) & 1, abort_flag, p.dev_status, tmo))
                break;
            if (lane == 0) {
                mbar_expect_tx(bar(C::B_VF + s), D * 128);
                tma_load_2d(sbase + C::OFF_V + s * C::VB, &tmV, j * 128, bh * D, bar(C::B_VF + s));
            }
            // Batch 0 goes out with tile 0, batch b+1 with tile 16 b + 8: by then
            // the V stage of tile 16 b + 5 has been released, so both tiles' P V
            // up to it -- and the mean MMA of batch b-1 issued before them, the
            // last reader of buffer (b+1) & 1 -- have completed.  The batch's own
            // mean MMA comes after the MMA warp has waited for this stage.
            if (VSMOOTH) {
                if (j == 0) write_batch(0);
                else if (j % kBatch == kBatch / 2 && (j / kBatch + 1) * kBatch < J) write_batch(j / kBatch + 1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_VF + s));
            issued = j + 1;
        }
        for (int j = (issued > NSV ? issued - NSV : 0); j < issued; ++j)
            drain_wait(bar(C::B_VF + j % NSV), (j / NSV) & 1, tmo);
    } else if (warp == kMmaWarp0 || warp == kMmaWarp0 + 1) {
        // ------------------------------------------------------------ MMA issuer of tile X
        // The whole warp runs this loop (uniform control flow); each tensor-core
        // instruction is issued by one elected lane.  Per key tile j: QK^T into
        // S_X once the softmax has released it, then P V (+ row sum) once the
        // probability bytes are in place.  The batch's mean restore goes in
        // after the next QK^T, once the softmax has written its operand.
        const int X = warp - kMmaWarp0;
        const uint32_t tb = tmem + C::base(X);
        {
            constexpr uint32_t IDESC_QK = idesc_f8_e4m3(128, 128);
            constexpr uint32_t IDESC_PVR = idesc_f8_e4m3(128, D + 16);  // O and the row sum together
            constexpr uint32_t IDESC_MEAN = idesc_bf16(128, D);
            auto issue_qk = [&](int j) {
                const int s = j % NSK;
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
                    const uint64_t ad = smem_desc(sbase + C::OFF_Q + X * C::QB + kk * 32, C::QK_SBO, C::QK_SWZ);
                    const uint64_t bd = smem_desc(sbase + C::OFF_K + s * C::KB + kk * 32, C::QK_SBO, C::QK_SWZ);
                    mma_f8_ss_w(tb + C::COL_S, ad, bd, IDESC_QK, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int j) {
                const uint32_t vbase = sbase + C::OFF_V + (j % NSV) * C::VB;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bd = smem_desc(vbase + kk * 32, 1024, kSwizzle128B);
                    mma_f8_ts_w(tb, tb + C::COL_P + kk * 8, bd, IDESC_PVR, (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            auto issue_mean = [&](int batch) {
                const uint32_t bmb = sbase + C::OFF_BM + (batch & 1) * C::BMB;
                const uint32_t amb = sbase + C::OFF_AM + X * C::AMB;
#pragma unroll
                for (int i = 0; i < kMeanK / 16; ++i) {
                    const uint64_t ad = smem_desc_lbo(amb + i * 256, 128, C::MG, kSwizzleNone);
                    const uint64_t bd = smem_desc_lbo(bmb + i * 256, 128, C::MG, kSwizzleNone);
                    mma_bf16_ss_w(tb, ad, bd, IDESC_MEAN, 1u);
                }
            };
            bool ok = mbar_wait_warp(bar(C::B_Q), 0, abort_flag, p.dev_status, tmo);
            // tile B starts half a step behind tile A
            if (X == 1 && ok) ok = mbar_wait_warp(bar(C::B_PF + 0), 0, abort_flag, p.dev_status, tmo);
            // The waits for data that is normally already there (the K stage of the
            // next tile, the V stage of this one) sit where this warp would idle
            // anyway, so that after a softmax hand-off only the MMA issue remains.
            ok = ok && mbar_wait_warp(bar(C::B_KF), 0, abort_flag, p.dev_status, tmo);
            for (int j = 0; ok && j < J; ++j) {
                if (j > 0) {
                    // S_X free: the softmax has read the row sum of tile j-1 back
                    if (!mbar_wait_warp(bar(C::B_SE + X), (j - 1) & 1, abort_flag, p.dev_status, tmo)) {
                        ok = false;
                        break;
                    }
                }
                tc_fence_after();
                issue_qk(j);
                mma_commit_w(bar(C::B_SF + X));
                mma_commit_w(bar(C::B_KE + j % NSK));
                if (VSMOOTH && j > 0 && (j - 1) % kBatch == kBatch - 1) {
                    // the batch that ended with tile j-1: its row-sum operand is
                    // written after S_X was released, and the softmax of tile j
                    // waits for this product before it rescales O
                    const int bi = (j - 1) / kBatch;
                    if (!mbar_wait_warp(bar(C::B_AMF + X), bi & 1, abort_flag, p.dev_status, tmo)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_mean(bi);
                    mma_commit_w(bar(C::B_MD + X));
                }
                if (!mbar_wait_warp(bar(C::B_VF + j % NSV), (j / NSV) & 1, abort_flag, p.dev_status, tmo) ||
                    !mbar_wait_warp(bar(C::B_PF + X), j & 1, abort_flag, p.dev_status, tmo)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_pv(j);
                mma_commit_w(bar(C::B_OD + X));
                mma_commit_w(bar(C::B_VE + j % NSV));
                if (j + 1 < J &&
                    !mbar_wait_warp(bar(C::B_KF + (j + 1) % NSK), ((j + 1) / NSK) & 1, abort_flag, p.dev_status, tmo)) {
                    ok = false;
                    break;
                }
            }
            if (ok && mbar_wait_warp(bar(C::B_SE + X), (J - 1) & 1, abort_flag, p.dev_status, tmo) &&
                (!VSMOOTH || mbar_wait_warp(bar(C::B_AMF + X), ((J - 1) / kBatch) & 1, abort_flag, p.dev_status, tmo))) {
                tc_fence_after();
                if (VSMOOTH) issue_mean((J - 1) / kBatch);
                mma_commit_w(bar(C::B_OF + X));
            }
            // every MMA this warp issued has completed once this phase flips
            mma_commit_w(bar(C::B_TD + X));
            drain_wait(bar(C::B_TD + X), 0, tmo);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax of tile X
        const int X = warp >> 2, q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16) + C::base(X);
        const int qtile = X ? qt1 : qt0;
        const int qrow = qtile * 128 + row;
        const float sq_i = __ldg(p.sq + (int64_t)bh * p.nblk + qtile);
        const float* skp = p.sk + (int64_t)bh * p.nblk;
        const int tail = p.N - (J - 1) * 128;  // valid keys of the last tile, 1..128
        const bool dbg_cta = DBG && bh == p.dbg_bh && qtile == p.dbg_qtile && (X == 0 || has_b);
        // row sums and running maxima of the current batch, [r | m][slot][row]
        float* hist = reinterpret_cast<float*>(smem + C::OFF_HIST) + X * (2 * kBatch * 128) + row;
        uint8_t* amb = smem + C::OFF_AM + X * C::AMB;
        float m = -INFINITY, l = 0.f;
        float sk_pref = __ldg(skp);
        bool ok = true;

        // Mean-restore operand of a batch of `nslots` tiles: each row sum, rescaled
        // to the running max m_now, as bf16 hi/lo at k = 3t (hi), 3t+1 (lo), 3t+2 (hi).
        auto close_batch = [&](float m_now, int nslots) {
            float rh[kBatch];
#pragma unroll
            for (int t = 0; t < kBatch; ++t)
                rh[t] = (t < nslots) ? hist[t * 128] * ex2_approx(hist[(kBatch + t) * 128] - m_now) : 0.f;
            uint32_t w[kMeanK / 2];
#pragma unroll
            for (int t = 0; t < kBatch; t += 2) {
                // k = 3t .. 3t+5 for the pair of tiles (t, t+1): hi0 lo0 hi0 hi1 lo1 hi1
                const uint32_t h0 = bf16_rn_bits(rh[t]);
                const uint32_t l0 = bf16_rn_bits(__fsub_rn(rh[t], bf16_bits_to_f32(h0)));
                const uint32_t h1 = bf16_rn_bits(rh[t + 1]);
                const uint32_t l1 = bf16_rn_bits(__fsub_rn(rh[t + 1], bf16_bits_to_f32(h1)));
                const int wi = 3 * t / 2;  // word index of k = 3t
                w[wi] = h0 | (l0 << 16);
                w[wi + 1] = h0 | (h1 << 16);
                w[wi + 2] = l1 | (h1 << 16);
            }
            // row `row` of the operand: 6 core-matrix rows of 16 bytes
#pragma unroll
            for (int c = 0; c < kMeanK / 8; ++c)
                *reinterpret_cast<uint4*>(amb + mo_offset(row, 8 * c)) =
                    make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
            fence_proxy_async_smem();
        };

        // Key tile j.  LAST marks the last tile, the only one with keys to mask.
        auto step = [&](int j, auto last_tag) -> bool {
            constexpr bool LAST = decltype(last_tag)::value;
            const bool masked = LAST && tail < 128;
            const int slot = j % kBatch;
            const float sk_j = sk_pref;  // loaded one tile ahead
            sk_pref = (j + 1 < J) ? __ldg(skp + j + 1) : 0.f;
            if (!mbar_wait_warp(bar(C::B_SF + X), j & 1, abort_flag, p.dev_status, tmo)) return false;
            tc_fence_after();
            // first read: the row max over all 128 keys
            float mx;
            if (!masked) {
                // the loads reduce as they read: the row max comes with the data
                uint32_t r0[32], r1[32], r2[32], r3[32];
                float m0, m1, m2, m3;
                tmem_ld32_max(lane_addr + C::COL_S, r0, m0);
                tmem_ld32_max(lane_addr + C::COL_S + 32, r1, m1);
                tmem_ld32_max(lane_addr + C::COL_S + 64, r2, m2);
                tmem_ld32_max(lane_addr + C::COL_S + 96, r3, m3);
                tmem_wait_ld();
                mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
                if (dbg_cta) {
                    float* dst = p.S_dump + (int64_t)row * p.Npad + j * 128;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        dst[i] = __uint_as_float(r0[i]);
                        dst[32 + i] = __uint_as_float(r1[i]);
                        dst[64 + i] = __uint_as_float(r2[i]);
                        dst[96 + i] = __uint_as_float(r3[i]);
                    }
                }
            } else {
                float a[64];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    load_half(lane_addr + C::COL_S + hf * 64, a);
                    if (dbg_cta) {
                        float* dst = p.S_dump + (int64_t)row * p.Npad + j * 128 + hf * 64;
#pragma unroll
                        for (int i = 0; i < 64; ++i) dst[i] = a[i];
                    }
                    if (masked) {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if (hf * 64 + i >= tail) a[i] = -INFINITY;
                    }
                    const float mh = max64(a);
                    mx = hf ? fmaxf(mx, mh) : mh;
                }
            }
            const float sigma = __fmul_rn(__fmul_rn(sq_i, sk_j), p.kscale);
            const float smx = __fmul_rn(sigma, mx);
            const float m_new = fmaxf(m, smx);
            // hybrid: the warp's 32 rows take exp-then-cast on this tile if one
            // of its valid rows holds a probability >= 2^-margin of its running max
            bool exact_tile = (EC == 0);
            if constexpr (EC == 2)
                exact_tile = __any_sync(0xffffffffu, qrow < p.N && __fsub_rn(smx, m_new) >= -p.exact_margin);
            const float alpha = ex2_approx(m - m_new);
            const float Cc = __fmaf_rn(-8.f, m_new, EC == 3 ? 120.f : 119.65f);
            const float k1 = sigma * 0.0625f;
            const float k2 = Cc * 0.0078125f;
            const float off = __fsub_rn(8.f, m_new);
            // |m'| < 2^19 in every row of the warp: the clip at 120 is implied
            // (t stays below 120.5 + beta for ExpCast, below 120.5 for the
            // adaptive t0, whose piece at 120 then carries beta = -0.195)
            const bool fast = __all_sync(0xffffffffu, fabsf(m_new) < 524288.f);
            // second read: probability bytes, half by half, into columns [32, 64)
            // of S_X, whose scores (keys 32..63) were read by then
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float a[64];
                load_half(lane_addr + C::COL_S + hf * 64, a);
                if (masked) {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        if (hf * 64 + i >= tail) a[i] = -INFINITY;
                }
                uint32_t pw[16];
                if constexpr (EC == 3) {
                    if (fast) {
#pragma unroll
                        for (int w = 0; w < 16; ++w) pw[w] = expcast4_pieces<false>(a + 4 * w, k1, k2);
                    } else {
#pragma unroll
                        for (int w = 0; w < 16; ++w) pw[w] = expcast4_pieces<true>(a + 4 * w, k1, k2);
                    }
                } else if (!exact_tile) {
                    if (fast) {
#pragma unroll
                        for (int w = 0; w < 16; ++w) pw[w] = expcast4<false>(a + 4 * w, k1, k2);
                    } else {
#pragma unroll
                        for (int w = 0; w < 16; ++w) pw[w] = expcast4<true>(a + 4 * w, k1, k2);
                    }
                } else {
#pragma unroll
                    for (int w = 0; w < 16; ++w) {
                        const float e0 = ex2_approx(__fmaf_rn(a[4 * w + 0], sigma, off));
                        const float e1 = ex2_approx(__fmaf_rn(a[4 * w + 1], sigma, off));
                        const float e2 = ex2_approx(__fmaf_rn(a[4 * w + 2], sigma, off));
                        const float e3 = ex2_approx(__fmaf_rn(a[4 * w + 3], sigma, off));
                        pw[w] = cvt_e4m3x2(e0, e1) | (cvt_e4m3x2(e2, e3) << 16);
                    }
                }
                if (masked) {
#pragma unroll
                    for (int w = 0; w < 16; ++w) {
                        uint32_t keep = 0;
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (hf * 64 + 4 * w + e < tail) keep |= 0xFFu << (8 * e);
                        pw[w] &= keep;
                    }
                }
                if (dbg_cta) {
                    uint32_t* dst = reinterpret_cast<uint32_t*>(p.P_dump + (int64_t)row * p.Npad + j * 128 + hf * 64);
#pragma unroll
                    for (int w = 0; w < 16; ++w) dst[w] = pw[w];
                }
                tmem_st16(lane_addr + C::COL_P + hf * 16, pw);
                if (hf == 0) {
                    // column 0 of S_X receives the row sum: start it at zero
                    const uint32_t zero[1] = {0u};
                    tmem_st1(lane_addr + C::COL_S, zero);
                }
            }
            tmem_wait_st();
            // O holds every product up to tile j-1: the completion of the P V of
            // tile j-1 and of the QK^T of tile j were both observed above.  The
            // mean restore of the batch that ended with tile j-1 is issued after
            // this QK^T, so a rescale here first awaits it; without a rescale
            // nothing touches O before this tile's P V, which the MMA warp
            // issues after the mean MMA, and the next QK^T's commit covers it
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                if (VSMOOTH && slot == 0) {
                    if (!mbar_wait_warp(bar(C::B_MD + X), ((j - 1) / kBatch) & 1, abort_flag, p.dev_status, tmo))
                        return false;
                    tc_fence_after();
                }
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                                    make_float2(alpha, alpha));
                        o[i] = __float_as_uint(v.x);
                        o[i + 1] = __float_as_uint(v.y);
                    }
                    tmem_st32(lane_addr + c0, o);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_PF + X));
            // row sum of tile j, once its P V has completed
            if (!mbar_wait_warp(bar(C::B_OD + X), j & 1, abort_flag, p.dev_status, tmo)) return false;
            tc_fence_after();
            uint32_t rbits;
            tmem_ld1(lane_addr + C::COL_S, rbits);
            tmem_wait_ld();
            const float r = __uint_as_float(rbits);
            l = __fmaf_rn(l, alpha, r);
            m = m_new;
            if (VSMOOTH) {
                hist[slot * 128] = r;
                hist[(kBatch + slot) * 128] = m_new;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_SE + X));
            // the batch's row-sum operand is built after S_X is released, off
            // the path to the next QK^T
            if (VSMOOTH && (slot == kBatch - 1 || LAST)) {
                close_batch(m_new, slot + 1);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_AMF + X));
            }
            return true;
        };

        for (int j = 0; j < J - 1; ++j)
            if (!step(j, std::false_type{})) {
                ok = false;
                break;
            }
        if (ok && !step(J - 1, std::true_type{})) ok = false;
        if (ok && mbar_wait_warp(bar(C::B_OF + X), 0, abort_flag, p.dev_status, tmo) && (X == 0 || has_b)) {
            tc_fence_after();
            const float inv_l = __frcp_rn(l);
            const float* svp = p.sv + (int64_t)bh * D;
            uint16_t* dst = p.O + (int64_t)b * p.o_sb + (int64_t)qrow * p.o_sn + (int64_t)h * p.o_sh;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(lane_addr + c0, o);
                tmem_wait_ld();
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float s0 = __ldg(svp + c0 + i), s1 = __ldg(svp + c0 + i + 1);
                    const float g0 = s0 > 0.f ? s0 : 1.f, g1 = s1 > 0.f ? s1 : 1.f;
                    const float v0 = g0 * __uint_as_float(o[i]) * inv_l;
                    const float v1 = g1 * __uint_as_float(o[i + 1]) * inv_l;
                    const __nv_bfloat162 pr = __floats2bfloat162_rn(v0, v1);
                    packed[i / 2] = *reinterpret_cast<const uint32_t*>(&pr);
                }
                if (qrow < p.N) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        d4[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

bool make_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                 uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, int E, bool S, bool G>
vc_status launch_one(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p,
                     dim3 grid, cudaStream_t st) {
    auto kern = attn_fwd_kernel<D, E, S, G>;
    vc_status a = ensure_smem_attr(reinterpret_cast<const void*>(kern), Cfg<D>::SMEM);
    if (a != VC_OK) return a;
    kern<<<grid, kThreads, Cfg<D>::SMEM, st>>>(mq, mk, mv, p);
    return cuda_status(cudaGetLastError());
}

template <int D, int E, bool G>
vc_status launch_e(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p,
                   dim3 grid, cudaStream_t st, int vsmooth) {
    return vsmooth ? launch_one<D, E, true, G>(mq, mk, mv, p, grid, st)
                   : launch_one<D, E, false, G>(mq, mk, mv, p, grid, st);
}

template <int D, bool G>
vc_status launch_g(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p,
                   dim3 grid, cudaStream_t st, int expcast, int vsmooth) {
    if (expcast == 1) return launch_e<D, 1, G>(mq, mk, mv, p, grid, st, vsmooth);
    if (expcast == 2) return launch_e<D, 2, G>(mq, mk, mv, p, grid, st, vsmooth);
    if (expcast == 3) return launch_e<D, 3, G>(mq, mk, mv, p, grid, st, vsmooth);
    return launch_e<D, 0, G>(mq, mk, mv, p, grid, st, vsmooth);
}

template <int D>
vc_status launch_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p,
                   dim3 grid, cudaStream_t st, int expcast, int vsmooth, bool dbg) {
    return dbg ? launch_g<D, true>(mq, mk, mv, p, grid, st, expcast, vsmooth)
               : launch_g<D, false>(mq, mk, mv, p, grid, st, expcast, vsmooth);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

vc_status launch_attn(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk, const uint8_t* V8T,
                      const float* sv, const uint16_t* mu, const vc_shape& s, float softmax_scale, int expcast,
                      float exact_margin, int vsmooth, uint16_t* O, int32_t* dev_status, cudaStream_t st,
                      const AttnDebug* dbg) {
    const int nblk = nblk_of(s.N);
    const int64_t Npad = npad_of(s.N);
    const uint64_t rows_qk = (uint64_t)s.B * s.H * Npad;
    const uint64_t rows_v = (uint64_t)s.B * s.H * s.d;
    CUtensorMap mq, mk, mv;
    const CUtensorMapSwizzle qk_swz = (s.d == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!make_map_2d(&mq, Q8, s.d, rows_qk, s.d, s.d, 128, qk_swz) ||
        !make_map_2d(&mk, K8, s.d, rows_qk, s.d, s.d, 128, qk_swz) ||
        !make_map_2d(&mv, V8T, Npad, rows_v, Npad, 128, s.d, CU_TENSOR_MAP_SWIZZLE_128B))
        return VC_ERR_CUDA;
    AttnParams p{};
    p.sq = sq;
    p.sk = sk;
    p.sv = sv;
    p.mu = mu;
    p.O = O;
    p.o_sb = s.s_b;
    p.o_sn = s.s_n;
    p.o_sh = s.s_h;
    p.H = s.H;
    p.N = s.N;
    p.nblk = nblk;
    p.Npad = Npad;
    const double sc = softmax_scale > 0.f ? (double)softmax_scale : (double)(float)(1.0 / __builtin_sqrt((double)s.d));
    p.kscale = (float)(sc * 1.4426950408889634);
    p.exact_margin = exact_margin;
    p.dev_status = dev_status;
    p.timeout_ns = (dbg && dbg->timeout_ns) ? dbg->timeout_ns : 4000000000ull;
    p.skip_k_tile = dbg ? dbg->skip_k_tile : -1;
    const bool dumps = dbg && dbg->S;
    p.dbg_bh = dumps ? dbg->bh : -1;
    p.dbg_qtile = dumps ? dbg->qtile : -1;
    p.S_dump = dumps ? dbg->S : nullptr;
    p.P_dump = dumps ? dbg->P : nullptr;
    const dim3 grid((nblk + 1) / 2, s.H, s.B);  // two query tiles per CTA
    if (s.d == 128) return launch_d<128>(mq, mk, mv, p, grid, st, expcast, vsmooth, dumps);
    return launch_d<64>(mq, mk, mv, p, grid, st, expcast, vsmooth, dumps);
}

}  // namespace vc
