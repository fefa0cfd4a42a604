// vc_attn.cu -- FP8 attention forward with ExpCast-FP8 and the V-Smooth mean
// restore, on tcgen05 tensor cores (sm_103a).
//
// What it computes: paper summary (paper.rainbus.top), 前置知识 "在线 softmax"
// (running max m_i, normaliser l_i, numerator A_i, rescale alpha_i) and
// 方法步骤详情 steps 3-4 (A_i <- alpha_i A_i + P_q,ij R_q,j + r_ij mu_j^T with
// r_ij the row sum of the quantized probabilities; ExpCast byte
// c = clip(Round(8(u+8)+56+beta), 0, 120)); dimensionstp.github.io 2-3 / 2-4.
//
// One CTA = 128 query rows of one (b, h); 10 warps:
//   warps 0-7  softmax: two warpgroups; thread (wg, row) owns query row `row`,
//              key columns [64 wg, 64 wg + 64) of each 128-key tile and output
//              channels [wg d/2, (wg+1) d/2).  The halves of a row exchange
//              partial maxima through shared memory.
//   warp 8     producer: TMA loads of the K and V^T tiles (ring of NS
//              stages); per tile it also writes the key scale, the
//              row-sum operand and the block mean (bf16 hi/lo parts) into
//              shared memory.
//   warp 9     MMA issuer (one elected lane) and TMEM owner.
// Tensor memory (512 columns):
//   S0, S1  [0,256)        fp32 scores of key tile j (double-buffered), QK^T.
//   P       inside S       probability bytes of tile j overwrite the first 16
//                          columns of each half of the score buffer.
//   O       [256, 256+d)   fp32 accumulator in residual-code units.
//   R       16 columns     row sums r_ij of the last 16 tiles, directly after O.
//   AM      24 columns     bf16 A operand of the batched mean restore.
//   Q       d/4 columns    the CTA's Q codes (A operand of every QK MMA),
//                          written once by the softmax warps.
// Row sums: each V^T stage carries 16 operand rows after its d channel rows;
// row d + (j mod 16) holds E4M3 1.0 and the others 0, so the PV MMA of width
// d + 16 adds P_j V_j into O and r_j into column j mod 16 of R.  The first
// tile of a batch restarts R with a separate width-16 MMA.
// Mean restore, batched: every 16 tiles the softmax warps read the 16 row
// sums, rescale each to the current running max, split them into bf16 hi/lo
// parts and the MMA thread adds sum_t r_t mu_t^T to O with one bf16 MMA of
// depth 48 (terms r_hi mu_hi + r_lo mu_hi + r_hi mu_lo per tile).  The means
// enter in units of the channel's residual scale g_c (g_c = s_v[c], or 1 for a
// channel whose residual is identically 0; mu' = mu * fp32(1/g_c)), so
// O = g (.) A / l at the end.
// The normaliser l is kept in registers, updated from the same row sums.
//
// ExpCast inner loop, per score: ts = sat(acc * sigma/16 + C/128) (one FFMA
// with saturation = clip to [0, 128] of t/128, exact because /128 and /16 are
// powers of two), then b = ts*128 + 1.5*2^23 (packed FFMA2) whose low byte is
// rint(t); two integer multiply-adds and one byte permute pack four codes.
// The upper clip at 120 is implied while |m'| < 2^19 (t <= 119.65 + 2^-1);
// rows beyond take a path with an explicit min.
#include <cstdio>
#include <type_traits>

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "vc_device.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr int kBatch = 16;             // key tiles per batched mean restore
constexpr int kMeanK = 3 * kBatch;     // bf16 depth of the mean MMA
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer in the low mantissa bits

template <int D>
struct Cfg {
    static constexpr int NS = (D == 128) ? 5 : 6;
    static constexpr int KB = 128 * D;
    static constexpr int VB = (D + 16) * 128;           // d channel rows + 16 row-sum operand rows
    static constexpr uint32_t QK_SWZ = (D == 128) ? kSwizzle128B : kSwizzle64B;
    static constexpr uint32_t QK_SBO = 8 * D;  // bytes per group of 8 rows
    static constexpr int BM_ROW_GROUP = 6 * 128;        // 8 rows x 48 bf16, stored as 6 core matrices
    static constexpr int BMB = (D / 8) * BM_ROW_GROUP;  // one mean-operand buffer
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + NS * KB;
    static constexpr int OFF_BM = OFF_V + NS * VB;
    static constexpr int OFF_SK = OFF_BM + 2 * BMB;
    static constexpr int OFF_MT = OFF_SK + NS * 16;      // running max per (wg, slot, row)
    static constexpr int OFF_XCH = OFF_MT + 2 * kBatch * 128 * 4;
    static constexpr int OFF_BAR = OFF_XCH + 2 * 2 * 128 * 4;
    static constexpr int NBAR = 32;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int USED = OFF_MISC + 64;
    // at least 116 KB so that exactly one CTA (and one 512-column TMEM owner) sits on an SM
    static constexpr int SMEM = ((USED > 118784) ? USED : 118784) + 1024;
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(VB % 1024 == 0 && KB % 1024 == 0 && OFF_V % 1024 == 0, "stages keep the swizzle alignment");
    // barrier indices
    static constexpr int B_Q = 0;
    static constexpr int B_KVF = 1;
    static constexpr int B_KVE = B_KVF + NS;
    static constexpr int B_SF = B_KVE + NS;
    static constexpr int B_PF = B_SF + 2;
    static constexpr int B_OD = B_PF + 2;
    static constexpr int B_XCH = B_OD + 1;
    static constexpr int B_PL = B_XCH + 2;
    static constexpr int B_OF = B_PL + 1;
    static constexpr int B_TD = B_OF + 1;
    static constexpr int NBAR_USED = B_TD + 1;
    static_assert(NBAR_USED <= NBAR, "barrier area");
    // TMEM columns
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256, COL_R = 256 + D, COL_AM = 256 + D + 16;
    static constexpr uint32_t COL_Q = COL_AM + kMeanK / 2;  // Q codes, 4 per column, D / 4 columns
    static_assert(COL_Q + D / 4 <= kTmemCols, "tmem budget");
};

struct AttnParams {
    const uint8_t* Q8;
    const float* sq;
    const float* sk;
    const float* sv;
    const uint16_t* mu;
    uint16_t* O;
    int64_t o_sb, o_sn, o_sh;
    int H, N, nblk;
    int64_t Npad;
    float kscale;
    int32_t* dev_status;
    uint64_t timeout_ns;
    int dbg_bh, dbg_qtile;
    float* S_dump;
    uint8_t* P_dump;
};

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bounded wait that ignores the abort flag: used at teardown to let this
// CTA's own copies and MMAs in flight finish before their memory is released.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns) return;
    }
}

// Byte offset of element (n, k) of a mean operand buffer: K-major, no swizzle,
// core matrices of 8 rows x 8 bf16 (16 bytes), 6 along K per group of 8 rows.
__device__ __forceinline__ uint32_t bm_offset(int n, int k) {
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
    // low 16 bits of u0 + 256 u1 are c0 | c1 << 8 (the magic's low 16 bits are 0)
    return prmt(mad_lo(u1, 256u, u0), mad_lo(u3, 256u, u2), 0x5410u);
}

__device__ __forceinline__ uint16_t bf16_rn_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

template <int D, bool EXPCAST, bool VSMOOTH, bool DBG>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const AttnParams p) {
    using C = Cfg<D>;
    constexpr int NS = C::NS;
    constexpr int HD = D / 2;  // output channels per softmax thread
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
    const int qtile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int bh = b * p.H + h;
    const int J = p.nblk;
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_Q), 8);  // the eight softmax warps have written Q into TMEM
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(C::B_KVF + s), 1);
            mbar_init(bar(C::B_KVE + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::B_SF + i), 1);
            mbar_init(bar(C::B_PF + i), 8);
            mbar_init(bar(C::B_XCH + i), 256);
        }
        mbar_init(bar(C::B_OD), 1);
        mbar_init(bar(C::B_PL), 8);
        mbar_init(bar(C::B_OF), 1);
        mbar_init(bar(C::B_TD), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    {
        // The mean operand buffers start zeroed.
        uint4* bm = reinterpret_cast<uint4*>(smem + C::OFF_BM);
        for (int i = threadIdx.x; i < 2 * C::BMB / 16; i += kThreads) bm[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        const int32_t row0 = (int32_t)((int64_t)bh * p.Npad);
        constexpr int PER = D / 32;  // channels per lane for the mean operand
        float ginv[PER];             // 1 / g_c, g_c = s_v[c] (1 for an all-zero residual channel)
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const float sv = __ldg(p.sv + (int64_t)bh * D + lane * PER + e);
            ginv[e] = __frcp_rn(sv > 0.f ? sv : 1.f);
        }
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
        }
        int issued = 0;
        for (int j = 0; j < J; ++j) {
            const int s = j % NS, n = j / NS;
            // global loads for this tile go out before the wait for a free stage,
            // so their latency overlaps it
            const float sk_j = (lane == 0) ? __ldg(p.sk + (int64_t)bh * p.nblk + j) : 0.f;
            uint32_t mu_w[PER / 2];
            if (VSMOOTH) {
                const uint32_t* src =
                    reinterpret_cast<const uint32_t*>(p.mu + ((int64_t)bh * p.nblk + j) * D + lane * PER);
#pragma unroll
                for (int e = 0; e < PER / 2; ++e) mu_w[e] = __ldg(src + e);
            }
            if (j >= NS && !mbar_wait_warp(bar(C::B_KVE + s), (n - 1) & 1, abort_flag, p.dev_status, tmo)) break;
            if (lane == 0) {
                mbar_expect_tx(bar(C::B_KVF + s), C::KB + D * 128);
                tma_load_2d(sbase + C::OFF_K + s * C::KB, &tmK, 0, row0 + j * 128, bar(C::B_KVF + s));
                tma_load_2d(sbase + C::OFF_V + s * C::VB, &tmV, j * 128, bh * D, bar(C::B_KVF + s));
                *reinterpret_cast<float*>(smem + C::OFF_SK + s * 16) = sk_j;
            }
            {
                // row-sum operand rows D..D+15 of the stage: row D + (j mod 16) is
                // E4M3 1.0 (0x38), the others 0, so the PV MMA adds r_j to column
                // j mod 16 of R.  A uniform 128-byte row is the same under the
                // 128-byte swizzle.
                uint4* ones = reinterpret_cast<uint4*>(smem + C::OFF_V + s * C::VB + D * 128);
                const int slot = j % kBatch;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int idx = lane * 4 + i;  // 16-byte chunk, 8 per row
                    const uint32_t v = ((idx >> 3) == slot) ? 0x38383838u : 0u;
                    ones[idx] = make_uint4(v, v, v, v);
                }
            }
            if (VSMOOTH) {
                // mean operand rows: k = 3t, 3t+1, 3t+2 hold (mu'_hi, mu'_hi, mu'_lo), mu' = mu / g
                uint8_t* bmb = smem + C::OFF_BM + ((j / kBatch) & 1) * C::BMB;
                const int k0 = 3 * (j % kBatch);
#pragma unroll
                for (int e = 0; e < PER; ++e) {
                    const int n_ch = lane * PER + e;
                    const uint32_t bits = (e & 1) ? (mu_w[e / 2] >> 16) : (mu_w[e / 2] & 0xFFFFu);
                    const float mp = __fmul_rn(bf16_bits_to_f32(bits), ginv[e]);
                    const uint16_t hi = bf16_rn_bits(mp);
                    const uint16_t lo = bf16_rn_bits(__fsub_rn(mp, bf16_bits_to_f32(hi)));
                    *reinterpret_cast<uint16_t*>(bmb + bm_offset(n_ch, k0)) = hi;
                    *reinterpret_cast<uint16_t*>(bmb + bm_offset(n_ch, k0 + 1)) = hi;
                    *reinterpret_cast<uint16_t*>(bmb + bm_offset(n_ch, k0 + 2)) = lo;
                }
            }
            fence_proxy_async_smem();  // the generic-proxy writes above are read by the MMAs
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_KVF + s));
            issued = j + 1;
        }
        // let this CTA's own copies in flight land before the CTA can exit
        for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
            drain_wait(bar(C::B_KVF + j % NS), (j / NS) & 1, tmo);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop (uniform control flow); each tensor-core
        // instruction is issued by one elected lane.
        {
            constexpr uint32_t IDESC_QK = idesc_f8_e4m3(128, 128);
            constexpr uint32_t IDESC_PV = idesc_f8_e4m3(128, D);
            constexpr uint32_t IDESC_PVR = idesc_f8_e4m3(128, D + 16);  // O and R together
            constexpr uint32_t IDESC_RS = idesc_f8_e4m3(128, 16);
            constexpr uint32_t IDESC_MEAN = idesc_bf16(128, D);
            auto issue_qk = [&](int j) {
                const int s = j % NS;
                const uint32_t d = tmem + ((j & 1) ? C::COL_S1 : C::COL_S0);
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
                    const uint64_t bd = smem_desc(sbase + C::OFF_K + s * C::KB + kk * 32, C::QK_SBO, C::QK_SWZ);
                    mma_f8_ts_w(d, tmem + C::COL_Q + kk * 8, bd, IDESC_QK, kk > 0 ? 1u : 0u);
                }
            };
            // P_j V_j into O and the row sums into R: one MMA of width d + 16 per
            // K-step reads the stage's channel rows and its row-sum operand rows.
            // The first tile of a batch restarts R with separate width-d and
            // width-16 MMAs.
            auto issue_pv_rs = [&](int j) {
                const int s = j % NS;
                const uint32_t pbase = tmem + ((j & 1) ? C::COL_S1 : C::COL_S0);
                const uint32_t vbase = sbase + C::OFF_V + s * C::VB;
                if (j % kBatch != 0) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t a = pbase + (kk < 2 ? kk * 8 : 64 + (kk - 2) * 8);
                        const uint64_t bd = smem_desc(vbase + kk * 32, 1024, kSwizzle128B);
                        mma_f8_ts_w(tmem + C::COL_O, a, bd, IDESC_PVR, 1u);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t a = pbase + (kk < 2 ? kk * 8 : 64 + (kk - 2) * 8);
                        const uint64_t bd = smem_desc(vbase + kk * 32, 1024, kSwizzle128B);
                        mma_f8_ts_w(tmem + C::COL_O, a, bd, IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t a = pbase + (kk < 2 ? kk * 8 : 64 + (kk - 2) * 8);
                        const uint64_t bd = smem_desc(vbase + D * 128 + kk * 32, 1024, kSwizzle128B);
                        mma_f8_ts_w(tmem + C::COL_R, a, bd, IDESC_RS, kk > 0 ? 1u : 0u);
                    }
                }
            };
            auto issue_mean = [&](int batch) {
                const uint32_t bmb = sbase + C::OFF_BM + (batch & 1) * C::BMB;
#pragma unroll
                for (int i = 0; i < kMeanK / 16; ++i) {
                    const uint64_t bd = smem_desc_lbo(bmb + i * 256, 128, C::BM_ROW_GROUP, kSwizzleNone);
                    mma_bf16_ts_w(tmem + C::COL_O, tmem + C::COL_AM + i * 8, bd, IDESC_MEAN, 1u);
                }
            };
            bool ok = mbar_wait_warp(bar(C::B_Q), 0, abort_flag, p.dev_status, tmo) &&
                      mbar_wait_warp(bar(C::B_KVF), 0, abort_flag, p.dev_status, tmo);
            if (ok) {
                tc_fence_after();
                issue_qk(0);
                mma_commit_w(bar(C::B_SF + 0));
            }
            for (int j = 0; ok && j < J; ++j) {
                if (j + 1 < J) {
                    const int s1 = (j + 1) % NS;
                    if (!mbar_wait_warp(bar(C::B_KVF + s1), ((j + 1) / NS) & 1, abort_flag, p.dev_status, tmo)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_qk(j + 1);
                    mma_commit_w(bar(C::B_SF + ((j + 1) & 1)));
                }
                if (!mbar_wait_warp(bar(C::B_PF + (j & 1)), (j >> 1) & 1, abort_flag, p.dev_status, tmo)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (VSMOOTH && j > 0 && (j % kBatch) == 0) issue_mean(j / kBatch - 1);
                issue_pv_rs(j);
                mma_commit_w(bar(C::B_OD));
                mma_commit_w(bar(C::B_KVE + j % NS));
            }
            if (VSMOOTH && ok && mbar_wait_warp(bar(C::B_PL), 0, abort_flag, p.dev_status, tmo)) {
                tc_fence_after();
                issue_mean((J - 1) / kBatch);
                mma_commit_w(bar(C::B_OF));
            }
            // every MMA this thread issued has completed once this phase flips
            mma_commit_w(bar(C::B_TD));
            drain_wait(bar(C::B_TD), 0, tmo);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax / correction / epilogue
        const int wg = warp >> 2, q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        const int qrow = qtile * 128 + row;
        const float sq_i = __ldg(p.sq + (int64_t)bh * p.nblk + qtile);
        const int tail = p.N - (J - 1) * 128;  // valid keys of the last tile, 1..128
        const bool dbg_cta = DBG && bh == p.dbg_bh && qtile == p.dbg_qtile;
        float* xch = reinterpret_cast<float*>(smem + C::OFF_XCH);
        float* mt = reinterpret_cast<float*>(smem + C::OFF_MT) + wg * kBatch * 128 + row;  // [slot * 128]
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        {
            // Q codes of this row into TMEM (column c holds bytes 4c..4c+3), read
            // by every QK MMA as its A operand; each warpgroup writes half the row.
            const uint4* src = reinterpret_cast<const uint4*>(
                p.Q8 + ((int64_t)bh * p.Npad + (int64_t)qtile * 128 + row) * D + wg * (D / 2));
            uint32_t w[D / 8];
#pragma unroll
            for (int i = 0; i < D / 32; ++i) {
                const uint4 v = __ldg(src + i);
                w[4 * i] = v.x;
                w[4 * i + 1] = v.y;
                w[4 * i + 2] = v.z;
                w[4 * i + 3] = v.w;
            }
            if constexpr (D == 128) tmem_st16(lane_addr + C::COL_Q + wg * (D / 8), w);
            else tmem_st8(lane_addr + C::COL_Q + wg * (D / 8), w);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_Q));
        }

        // Closes a batch of `nslots` tiles: their row sums, rescaled to the running
        // max m_now, go into l and (warpgroup 0, V-Smooth) into the bf16 A operand
        // of the mean MMA as hi/lo pairs: k = 3t -> hi, 3t+1 -> lo, 3t+2 -> hi.
        auto close_batch = [&](float m_now, int nslots) {
            uint32_t r[16];
            tmem_ld16(lane_addr + C::COL_R, r);
            tmem_wait_ld();
            float rh[kBatch];
            float lsum = 0.f;
#pragma unroll
            for (int t = 0; t < kBatch; ++t) {
                rh[t] = (t < nslots) ? __uint_as_float(r[t]) * ex2_approx(mt[t * 128] - m_now) : 0.f;
                lsum += rh[t];
            }
            l += lsum;
            if (VSMOOTH && wg == 0) {
                uint32_t e[kMeanK];
#pragma unroll
                for (int t = 0; t < kBatch; ++t) {
                    const uint32_t hi = bf16_rn_bits(rh[t]);
                    const uint32_t lo = bf16_rn_bits(__fsub_rn(rh[t], bf16_bits_to_f32(hi)));
                    e[3 * t] = hi;
                    e[3 * t + 1] = lo;
                    e[3 * t + 2] = hi;
                }
                uint32_t a0[16], a1[8];
#pragma unroll
                for (int w = 0; w < 16; ++w) a0[w] = e[2 * w] | (e[2 * w + 1] << 16);
#pragma unroll
                for (int w = 0; w < 8; ++w) a1[w] = e[32 + 2 * w] | (e[33 + 2 * w] << 16);
                tmem_st16(lane_addr + C::COL_AM, a0);
                tmem_st8(lane_addr + C::COL_AM + 16, a1);
                tmem_wait_st();
            }
        };

        // One key tile.  MASKED is set only for the last tile, so the hot loop
        // carries no masking code.  Returns false when a wait gave up.
        auto step = [&](int j, auto masked_tag) -> bool {
            constexpr bool MASKED = decltype(masked_tag)::value;
            const int sb = j & 1, slot = j % kBatch;
            const uint32_t colS = sb ? C::COL_S1 : C::COL_S0;
            if (!mbar_wait_warp(bar(C::B_SF + sb), (j >> 1) & 1, abort_flag, p.dev_status, tmo) ||
                !mbar_wait_warp(bar(C::B_KVF + j % NS), (j / NS) & 1, abort_flag, p.dev_status, tmo)) {
                return false;
            }
            tc_fence_after();
            const float sk_j = *reinterpret_cast<const float*>(smem + C::OFF_SK + (j % NS) * 16);
            float a[64];
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(lane_addr + colS + wg * 64, r0);
                tmem_ld32(lane_addr + colS + wg * 64 + 32, r1);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    a[i] = __uint_as_float(r0[i]);
                    a[32 + i] = __uint_as_float(r1[i]);
                }
            }
            if (dbg_cta) {
                float* dst = p.S_dump + (int64_t)row * p.Npad + j * 128 + wg * 64;
#pragma unroll
                for (int i = 0; i < 64; ++i) dst[i] = a[i];
            }
            const bool masked = MASKED && (tail < 128);
            if (masked) {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (wg * 64 + i >= tail) a[i] = -INFINITY;
            }
            // partial row max over this thread's 64 keys, exchanged with the other half
            float mx;
            {
                float t[22];
#pragma unroll
                for (int i = 0; i < 21; ++i) t[i] = max3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
                t[21] = a[63];
                float u[8];
#pragma unroll
                for (int i = 0; i < 7; ++i) u[i] = max3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
                u[7] = t[21];
                mx = max3(max3(u[0], u[1], u[2]), max3(u[3], u[4], u[5]), fmaxf(u[6], u[7]));
            }
            xch[sb * 256 + wg * 128 + row] = mx;
            mbar_arrive(bar(C::B_XCH + sb));
            if (!mbar_wait_warp(bar(C::B_XCH + sb), (j >> 1) & 1, abort_flag, p.dev_status, tmo)) {
                return false;
            }
            const float mx_all = fmaxf(mx, xch[sb * 256 + (1 - wg) * 128 + row]);
            const float sigma = __fmul_rn(__fmul_rn(sq_i, sk_j), p.kscale);
            const float m_new = fmaxf(m, __fmul_rn(sigma, mx_all));
            const float alpha = ex2_approx(m - m_new);
            uint32_t pw[16];
            if (EXPCAST) {
                const float Cc = __fmaf_rn(-8.f, m_new, 119.65f);
                const float k1 = sigma * 0.0625f;
                const float k2 = Cc * 0.0078125f;
                // |m'| < 2^19 in every row of the warp: the clip at 120 is implied
                if (__all_sync(0xffffffffu, fabsf(m_new) < 524288.f)) {
#pragma unroll
                    for (int w = 0; w < 16; ++w) pw[w] = expcast4<false>(a + 4 * w, k1, k2);
                } else {
#pragma unroll
                    for (int w = 0; w < 16; ++w) pw[w] = expcast4<true>(a + 4 * w, k1, k2);
                }
            } else {
                const float off = __fsub_rn(8.f, m_new);
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
                        if (wg * 64 + 4 * w + e < tail) keep |= 0xFFu << (8 * e);
                    pw[w] &= keep;
                }
            }
            if (dbg_cta) {
                uint32_t* dst = reinterpret_cast<uint32_t*>(p.P_dump + (int64_t)row * p.Npad + j * 128 + wg * 64);
#pragma unroll
                for (int w = 0; w < 16; ++w) dst[w] = pw[w];
            }
            tmem_st16(lane_addr + colS + wg * 64, pw);
            tmem_wait_st();
            // O must hold every product up to tile j-1 before it is rescaled, and
            // the row sums of a finished batch are read after their MMAs complete.
            const bool resc = (j > 0) && __any_sync(0xffffffffu, alpha != 1.f);
            const bool bend = (j > 0) && slot == 0;
            if (resc || bend) {
                if (!mbar_wait_warp(bar(C::B_OD), (j - 1) & 1, abort_flag, p.dev_status, tmo)) {
                    return false;
                }
                tc_fence_after();
            }
            if (resc) {
#pragma unroll
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + C::COL_O + wg * HD + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                                    make_float2(alpha, alpha));
                        o[i] = __float_as_uint(v.x);
                        o[i + 1] = __float_as_uint(v.y);
                    }
                    tmem_st32(lane_addr + C::COL_O + wg * HD + c0, o);
                }
                tmem_wait_st();
            }
            l *= alpha;
            if (bend) close_batch(m_new, kBatch);
            mt[slot * 128] = m_new;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_PF + sb));
            m = m_new;
            return true;
        };
        for (int j = 0; j < J - 1; ++j)
            if (!step(j, std::false_type{})) {
                ok = false;
                break;
            }
        if (ok && !step(J - 1, std::true_type{})) ok = false;
        if (ok && mbar_wait_warp(bar(C::B_OD), (J - 1) & 1, abort_flag, p.dev_status, tmo)) {
            tc_fence_after();
            close_batch(m, (J - 1) % kBatch + 1);
            bool fin = true;
            if (VSMOOTH) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_PL));
                fin = mbar_wait_warp(bar(C::B_OF), 0, abort_flag, p.dev_status, tmo);
                tc_fence_after();
            }
            if (fin) {
                const float inv_l = __frcp_rn(l);
                const float* svp = p.sv + (int64_t)bh * D + wg * HD;
                uint16_t* dst =
                    p.O + (int64_t)b * p.o_sb + (int64_t)qrow * p.o_sn + (int64_t)h * p.o_sh + wg * HD;
#pragma unroll
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + C::COL_O + wg * HD + c0, o);
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
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

// cuTensorMapEncodeTiled is a driver API; it is looked up through the runtime
// so that the library does not link against libcuda directly.
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

template <int D, bool E, bool S, bool G>
vc_status launch_one(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p,
                     dim3 grid, cudaStream_t st) {
    auto kern = attn_fwd_kernel<D, E, S, G>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
        if (e != cudaSuccess) return cuda_status(e);
        attr = true;
    }
    kern<<<grid, kThreads, Cfg<D>::SMEM, st>>>(mk, mv, p);
    return cuda_status(cudaGetLastError());
}

template <int D>
vc_status launch_d(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p,
                   dim3 grid, cudaStream_t st, int expcast, int vsmooth, bool dbg) {
    if (dbg) {
        if (expcast)
            return vsmooth ? launch_one<D, true, true, true>(mk, mv, p, grid, st)
                           : launch_one<D, true, false, true>(mk, mv, p, grid, st);
        return vsmooth ? launch_one<D, false, true, true>(mk, mv, p, grid, st)
                       : launch_one<D, false, false, true>(mk, mv, p, grid, st);
    }
    if (expcast)
        return vsmooth ? launch_one<D, true, true, false>(mk, mv, p, grid, st)
                       : launch_one<D, true, false, false>(mk, mv, p, grid, st);
    return vsmooth ? launch_one<D, false, true, false>(mk, mv, p, grid, st)
                   : launch_one<D, false, false, false>(mk, mv, p, grid, st);
}

}  // namespace

vc_status launch_attn(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk, const uint8_t* V8T,
                      const float* sv, const uint16_t* mu, const vc_shape& s, float softmax_scale, int expcast,
                      int vsmooth, uint16_t* O, int32_t* dev_status, cudaStream_t st, const AttnDebug* dbg) {
    const int nblk = nblk_of(s.N);
    const int64_t Npad = npad_of(s.N);
    const uint64_t rows_qk = (uint64_t)s.B * s.H * Npad;
    const uint64_t rows_v = (uint64_t)s.B * s.H * s.d;
    CUtensorMap mk, mv;
    const CUtensorMapSwizzle qk_swz = (s.d == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!make_map_2d(&mk, K8, s.d, rows_qk, s.d, s.d, 128, qk_swz) ||
        !make_map_2d(&mv, V8T, Npad, rows_v, Npad, 128, s.d, CU_TENSOR_MAP_SWIZZLE_128B))
        return VC_ERR_CUDA;
    AttnParams p{};
    p.Q8 = Q8;
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
    p.dev_status = dev_status;
    p.timeout_ns = 4000000000ull;
    p.dbg_bh = dbg ? dbg->bh : -1;
    p.dbg_qtile = dbg ? dbg->qtile : -1;
    p.S_dump = dbg ? dbg->S : nullptr;
    p.P_dump = dbg ? dbg->P : nullptr;
    const dim3 grid(nblk, s.H, s.B);
    if (s.d == 128) return launch_d<128>(mk, mv, p, grid, st, expcast, vsmooth, dbg != nullptr);
    return launch_d<64>(mk, mv, p, grid, st, expcast, vsmooth, dbg != nullptr);
}

}  // namespace vc
