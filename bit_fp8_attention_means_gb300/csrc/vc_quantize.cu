// vc_quantize.cu -- the fused quantizer of the V-Smooth path.
//
// Paper summary (paper.rainbus.top), 方法步骤详情 step 2 and 前置知识 "低比特
// 量化与离群值"; dimensionstp.github.io section 2-2:
//   Q, K' = K[pi]: one fp32 scale per 128-token block, codes = E4M3(x * 448/amax).
//   V' = V[pi]:   mu_j = bf16(block mean), R = V' - mu_j, residual codes with
//                 one scale per channel over the whole head.
// vc_quantize: three memory-bound kernels per call:
//   quant_qk_kernel      Q and K' blocks (gathered rows for K'), one CTA per
//                        (head, block), heads fastest.
//   quant_v_stats_kernel block means of V' and the per-channel residual amax
//                        (atomicMax on the fp32 bit pattern, values are >= 0).
//   quant_v_codes_kernel residual codes, written token-contiguous per channel
//                        (V8T [B,H,d,Npad]) so that the attention kernel can
//                        read V as a K-major MMA operand.
// The two V kernels stage each block's gathered rows in shared memory with
// 16-byte loads; the per-channel scale needs the whole head, hence two passes.
// vc_quantize_ex replaces quant_qk_kernel with quant_qk_pre_kernel, which
// also applies the rotary transform and the Hadamard rotation to Q and K'
// (the rest of the pages' fused preprocessing chain: paper summary 核心方法,
// dimensionstp.github.io 3-1 and 3-3); vc_quantize_staged runs the same
// computation as separate kernels with fp32 intermediates (rope_stage,
// gather_stage, hadamard_stage, then the quantizers) to measure the fusion.
// Every rounding step is written with an explicit _rn intrinsic so that the
// codes are bit-reproducible: fp32 block sum in token order, IEEE division,
// round-to-nearest-even conversions (cvt.rn.satfinite.e4m3x2).
#include <algorithm>

#include <cuda_bf16.h>

#include "vc_device.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr int kQkThreads = 256;

struct QkArgs {
    const void* X;        // rows of bf16 (uint16 bits) or fp32, by the kernel's input type
    int64_t s_b, s_n, s_h;
    const int32_t* perm;  // may be null
    const float* rope;    // [N, D/2, 2] (cos, sin) per position and channel pair; read only when rotating
    float s_mul;          // factor on the block scale: 1/D on Q when the Hadamard rotation is applied, else 1
    uint8_t* X8;
    float* sx;
    int H, N, nblk;
    int64_t Npad;
};

// Rotation of the channel pair (x0, x1) by the angle with cosine c and sine s,
// (x0 + i x1)(c + i s): the four products rounded, then the difference and sum.
__device__ __forceinline__ void rotate_pair(float& x0, float& x1, float c, float s) {
    const float a = __fmul_rn(x0, c), b = __fmul_rn(x1, s);
    const float e = __fmul_rn(x0, s), f = __fmul_rn(x1, c);
    x0 = __fsub_rn(a, b);
    x1 = __fadd_rn(e, f);
}

// Rotates the consecutive channel pairs x[0..n) with the (cos, sin) pairs at tab.
template <int n>
__device__ __forceinline__ void rotate_pairs(float (&x)[n], const float* tab) {
    const float4* t4 = reinterpret_cast<const float4*>(tab);
#pragma unroll
    for (int v = 0; v < n / 4; ++v) {
        const float4 r = __ldg(t4 + v);
        rotate_pair(x[4 * v], x[4 * v + 1], r.x, r.y);
        rotate_pair(x[4 * v + 2], x[4 * v + 3], r.z, r.w);
    }
}

// Walsh-Hadamard butterfly stages of stride 1 .. n/2 over x[0..n), stride 1
// first: (a, b) -> (a + b, a - b), each result rounded.
template <int n, int st>
__device__ __forceinline__ void hadamard_stage(float (&x)[n]) {
#pragma unroll
    for (int p = 0; p < n / 2; ++p) {
        const int i = (p / st) * (2 * st) + (p % st);
        const float a = x[i], b = x[i + st];
        x[i] = __fadd_rn(a, b);
        x[i + st] = __fsub_rn(a, b);
    }
    if constexpr (2 * st < n) hadamard_stage<n, 2 * st>(x);
}

template <int n>
__device__ __forceinline__ void hadamard_local(float (&x)[n]) {
    hadamard_stage<n, 1>(x);
}

// One butterfly stage whose partners sit in the lane that differs in `mask`:
// the lower lane keeps a + b, the upper lane a - b (a = lower's value).  Every
// lane of the warp must take part.
template <int n>
__device__ __forceinline__ void hadamard_cross(float (&x)[n], int mask, bool upper) {
#pragma unroll
    for (int c = 0; c < n; ++c) {
        const float o = __shfl_xor_sync(0xffffffffu, x[c], mask);
        x[c] = upper ? __fsub_rn(o, x[c]) : __fadd_rn(x[c], o);
    }
}

template <int n>
__device__ __forceinline__ void load_row_part(const uint16_t* p, float (&x)[n]) {
    const uint4* p4 = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int v = 0; v < n / 8; ++v) {
        const uint4 w = __ldg(p4 + v);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[v * 8 + 2 * e] = bf16_bits_to_f32(ws[e] & 0xFFFFu);
            x[v * 8 + 2 * e + 1] = bf16_bits_to_f32(ws[e] >> 16);
        }
    }
}

template <int n>
__device__ __forceinline__ void load_row_part(const float* p, float (&x)[n]) {
    const float4* p4 = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int v = 0; v < n / 4; ++v) {
        const float4 w = __ldg(p4 + v);
        x[4 * v] = w.x;
        x[4 * v + 1] = w.y;
        x[4 * v + 2] = w.z;
        x[4 * v + 3] = w.w;
    }
}

// Plain Q/K block quantizer (no rotation): one CTA per (head h, block j,
// batch b, tensor which), heads fastest; 2 threads per token row, each holding
// D/2 channels.  In: uint16_t (bf16) or float rows.
template <int D, typename In>
__global__ void __launch_bounds__(kQkThreads) quant_qk_kernel(QkArgs q, QkArgs k) {
    constexpr int CH = D / 2;           // channels per thread
    const QkArgs& a = (blockIdx.z & 1) ? k : q;
    const int b = blockIdx.z >> 1;
    const int h = (int)(blockIdx.x % (unsigned)a.H), j = (int)(blockIdx.x / (unsigned)a.H);
    const int bh = b * a.H + h;
    const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int t = j * kBlock + row;
    const bool valid = t < a.N;

    float x[CH];
    float amax = 0.f;
    if (valid) {
        const int src = a.perm ? __ldg(a.perm + (int64_t)bh * a.N + t) : t;
        load_row_part<CH>(static_cast<const In*>(a.X) + (int64_t)b * a.s_b + (int64_t)src * a.s_n +
                              (int64_t)h * a.s_h + half * CH,
                          x);
#pragma unroll
        for (int c = 0; c < CH; ++c) amax = fmaxf(amax, fabsf(x[c]));
    }
    __shared__ float red[kQkThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < kQkThreads / 32; ++w) amax = fmaxf(amax, red[w]);

    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
    if (threadIdx.x == 0) a.sx[(int64_t)bh * a.nblk + j] = __fmul_rn(__fdiv_rn(amax, 448.f), a.s_mul);

    uint4* out = reinterpret_cast<uint4*>(a.X8 + ((int64_t)bh * a.Npad + t) * D + half * CH);
#pragma unroll
    for (int v = 0; v < CH / 16; ++v) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (valid) {
                const int c = v * 16 + 4 * e;
                uint32_t lo = cvt_e4m3x2(__fmul_rn(x[c], inv), __fmul_rn(x[c + 1], inv));
                uint32_t hi = cvt_e4m3x2(__fmul_rn(x[c + 2], inv), __fmul_rn(x[c + 3], inv));
                w[e] = lo | (hi << 16);
            } else {
                w[e] = 0u;
            }
        }
        out[v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ------------------------------------------------------------------ fused rotary + Hadamard
//
// Q/K block quantizer with the rotary transform and the Hadamard rotation in
// registers.  Persistent: one CTA of 128 * kPreTpr threads per SM walks the
// (tensor, batch, block, head) tiles, heads fastest so that the CTAs running
// at the same time share the rows of the rotary table, and stages every tile
// in shared memory with 16-byte cp.async copies one tile ahead: the copies of
// tile i+1 (the gathered bf16 rows and their table rows) run while tile i is
// computed; the perm entries are loaded a further tile ahead.  kPreTpr
// threads per token row, each holding D/kPreTpr channels (2 and D/2 here; 4
// measured the same): warp w computes rows (32/kPreTpr) w .. and also copies
// them (lane l holds the source index of one of them and hands it out by
// shuffle), whole rows per instruction so that every sector is read once.
// Shared rows are stored with a row- and part-dependent rotation of the
// 16-byte chunks inside each group of 8, so that the compute reads (the eight
// lanes of a shared-memory phase) are free of bank conflicts.
// Arithmetic is that of the plain path plus, per row: rotation of each channel
// pair (four products, then difference and sum) and the Walsh-Hadamard stages
// of stride 1 .. D/(2 kPreTpr) in the thread and D/kPreTpr .. D/2 across the
// row's lanes, each result rounded as the definition states; packed fp32
// instructions carry two of them at once.

constexpr int kPreTpr = 2;                    // threads per token row
constexpr int kPreThreads = kBlock * kPreTpr;

template <int D, bool ROPE>
struct PreCfg {
    static constexpr int CPD = D / 8;                   // 16-byte chunks per bf16 row
    static constexpr int CPT = ROPE ? D / 4 : 0;        // 16-byte chunks per table row
    static constexpr int DATA = kBlock * CPD * 16;
    static constexpr int TAB = kBlock * CPT * 16;
    static constexpr int STAGE = DATA + TAB;
    static constexpr int SMEM = 2 * STAGE;
};

// Physical chunk of logical chunk c in row r, for rows of `cpr` chunks read by
// kPreTpr threads as equal parts of cq = cpr/kPreTpr chunks.  Within each
// aligned group of 8 chunks the chunk index is rotated by an amount that
// differs for the eight (row, part) readers of one shared-memory phase.
template <int cpr>
__device__ __forceinline__ int chunk_swz(int r, int c) {
    constexpr int cq = cpr / kPreTpr;
    int rot;
    if constexpr (kPreTpr == 2) {
        // a phase = 4 rows x 2 halves
        rot = (cq >= 8) ? 2 * (r & 3) + ((c / cq) & 1) : (r & 3);
    } else {
        // a phase = 2 rows x 4 quarters
        if constexpr (cq >= 8)
            rot = ((c / cq) & 3) + 4 * (r & 1);       // c & 7 = v
        else if constexpr (cq == 4)
            rot = 2 * (r & 1) + ((c >> 3) & 1);       // c & 7 = 4 (q & 1) + v
        else
            rot = (r & 1);                             // c & 7 = 2 q + v
    }
    return (c & ~7) | ((c + rot) & 7);
}

// 16-byte asynchronous copy global -> shared, cached in L2 only.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

struct PreTile {
    int which, b, j, h;
};

// Tile coordinates of work item `item` = ((which*B + b)*nblk + j)*H + h
// (items < 2^25, so 32-bit arithmetic suffices; decoded once per item).
__device__ __forceinline__ PreTile pre_tile(int item, int H, int nblk, int B) {
    uint32_t r = (uint32_t)item;
    PreTile t;
    t.h = (int)(r % (uint32_t)H);
    r /= (uint32_t)H;
    t.j = (int)(r % (uint32_t)nblk);
    r /= (uint32_t)nblk;
    t.b = (int)(r % (uint32_t)B);
    t.which = (int)(r / (uint32_t)B);
    return t;
}

// Walsh-Hadamard stage of stride st over x[0..n): stride 1 with scalar
// instructions, wider strides two butterflies per packed instruction; a - b
// is fma(b, -1, a), which rounds the difference once as a subtraction does.
template <int n, int st>
__device__ __forceinline__ void hadamard_stage_packed(float (&x)[n]) {
    if constexpr (st == 1) {
#pragma unroll
        for (int i = 0; i < n; i += 2) {
            const float a = x[i], b = x[i + 1];
            x[i] = __fadd_rn(a, b);
            x[i + 1] = __fsub_rn(a, b);
        }
    } else {
#pragma unroll
        for (int p = 0; p < n / 4; ++p) {
            const int i = ((2 * p) / st) * (2 * st) + ((2 * p) % st);
            const float2 A = make_float2(x[i], x[i + 1]), Bv = make_float2(x[i + st], x[i + st + 1]);
            const float2 S = __fadd2_rn(A, Bv);
            const float2 Df = __ffma2_rn(Bv, make_float2(-1.f, -1.f), A);
            x[i] = S.x;
            x[i + 1] = S.y;
            x[i + st] = Df.x;
            x[i + st + 1] = Df.y;
        }
    }
    if constexpr (2 * st < n) hadamard_stage_packed<n, 2 * st>(x);
}

// Butterfly stage with the partner in lane ^ mask: the lower lane keeps a + b,
// the upper lane a - b (a = lower's value), both as fma(own, +-1, other).
template <int n>
__device__ __forceinline__ void hadamard_cross_packed(float (&x)[n], int mask, bool upper) {
    const float sgn = upper ? -1.f : 1.f;
#pragma unroll
    for (int c = 0; c < n; c += 2) {
        const float o0 = __shfl_xor_sync(0xffffffffu, x[c], mask);
        const float o1 = __shfl_xor_sync(0xffffffffu, x[c + 1], mask);
        const float2 y = __ffma2_rn(make_float2(x[c], x[c + 1]), make_float2(sgn, sgn), make_float2(o0, o1));
        x[c] = y.x;
        x[c + 1] = y.y;
    }
}

template <int D, bool ROPE, bool HAD>
__global__ void __launch_bounds__(kPreThreads, 1) quant_qk_pre_kernel(QkArgs q, QkArgs k, int B, int items) {
    using C = PreCfg<D, ROPE>;
    constexpr int CH = D / kPreTpr;       // channels per thread
    constexpr int RPW = 32 / kPreTpr;     // rows per warp
    constexpr int NW = kPreThreads / 32;
    extern __shared__ __align__(16) uint8_t smem_pre[];
    __shared__ float red[NW];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = q.H, nblk = q.nblk, N = q.N;
    const int stride = gridDim.x;

    // source token of row RPW*warp + (lane % RPW) of a tile (perm entry or the row itself)
    auto src_of = [&](const PreTile& tl) -> int {
        const QkArgs& a = tl.which ? k : q;
        const int t = tl.j * kBlock + RPW * warp + (lane % RPW);
        if (t >= N) return 0;
        return a.perm ? __ldg(a.perm + (int64_t)(tl.b * H + tl.h) * N + t) : t;
    };
    // copies of this warp's rows of one tile into stage `st`
    auto issue = [&](const PreTile& tl, int srcv, int st) {
        const QkArgs& a = tl.which ? k : q;
        const int cnt = min(kBlock, N - tl.j * kBlock);
        const uint32_t base = smem_u32(smem_pre) + st * C::STAGE;
        const uint16_t* X = static_cast<const uint16_t*>(a.X) + (int64_t)tl.b * a.s_b + (int64_t)tl.h * a.s_h;
        constexpr int RPI = 32 / C::CPD;  // bf16 rows per instruction
#pragma unroll
        for (int i = 0; i < RPW / RPI; ++i) {
            const int rl = i * RPI + lane / C::CPD, c = lane % C::CPD;
            const int src = __shfl_sync(0xffffffffu, srcv, rl);
            const int r = RPW * warp + rl;
            if (r < cnt)
                cp_async16(base + r * (C::CPD * 16) + chunk_swz<C::CPD>(r, c) * 16,
                           X + (int64_t)src * a.s_n + c * 8);
        }
        if constexpr (ROPE) {
            constexpr int TRPI = (C::CPT >= 32) ? 1 : 32 / C::CPT;  // table rows per instruction
#pragma unroll
            for (int i = 0; i < RPW / TRPI; ++i) {
#pragma unroll
                for (int u = 0; u < (C::CPT >= 32 ? C::CPT / 32 : 1); ++u) {
                    const int rl = i * TRPI + (C::CPT >= 32 ? 0 : lane / C::CPT);
                    const int c = (C::CPT >= 32) ? u * 32 + lane : lane % C::CPT;
                    const int src = __shfl_sync(0xffffffffu, srcv, rl);
                    const int r = RPW * warp + rl;
                    if (r < cnt)
                        cp_async16(base + C::DATA + r * (C::CPT * 16) + chunk_swz<C::CPT>(r, c) * 16,
                                   a.rope + (int64_t)src * D + c * 4);
                }
            }
        }
    };

    int item = blockIdx.x;
    PreTile tl = pre_tile(item, H, nblk, B), tl_next = pre_tile(item + stride, H, nblk, B);
    if (item < items) issue(tl, src_of(tl), 0);
    cp_async_commit();
    int src_next = (item + stride < items) ? src_of(tl_next) : 0;
    const int r = tid / kPreTpr, qd = tid % kPreTpr;
    for (int it = 0; item < items; ++it, item += stride) {
        // copies of the next tile, then the perm entries of the one after it
        const PreTile tl_after = pre_tile(item + 2 * stride, H, nblk, B);
        if (item + stride < items) issue(tl_next, src_next, (it + 1) & 1);
        cp_async_commit();
        if (item + 2 * stride < items) src_next = src_of(tl_after);
        cp_async_wait1();
        __syncthreads();

        const QkArgs& a = tl.which ? k : q;
        const int bh = tl.b * H + tl.h;
        const int t = tl.j * kBlock + r;
        const bool valid = t < N;
        const uint8_t* stg = smem_pre + (it & 1) * C::STAGE;
        float x[CH];
        if (valid) {
            const uint8_t* drow = stg + r * (C::CPD * 16);
#pragma unroll
            for (int v = 0; v < CH / 8; ++v) {
                const uint4 w = *reinterpret_cast<const uint4*>(drow + chunk_swz<C::CPD>(r, qd * (CH / 8) + v) * 16);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    x[v * 8 + 2 * e] = __uint_as_float(ws[e] << 16);
                    x[v * 8 + 2 * e + 1] = __uint_as_float(ws[e] & 0xFFFF0000u);
                }
            }
            if constexpr (ROPE) {
                const uint8_t* trow = stg + C::DATA + r * (C::CPT * 16);
#pragma unroll
                for (int v = 0; v < CH / 4; ++v) {
                    const float4 cs =
                        *reinterpret_cast<const float4*>(trow + chunk_swz<C::CPT>(r, qd * (CH / 4) + v) * 16);
                    const float2 p0 = __fmul2_rn(make_float2(x[4 * v], x[4 * v + 1]), make_float2(cs.x, cs.x));
                    const float2 q0 = __fmul2_rn(make_float2(x[4 * v], x[4 * v + 1]), make_float2(cs.y, cs.y));
                    const float2 p1 = __fmul2_rn(make_float2(x[4 * v + 2], x[4 * v + 3]), make_float2(cs.z, cs.z));
                    const float2 q1 = __fmul2_rn(make_float2(x[4 * v + 2], x[4 * v + 3]), make_float2(cs.w, cs.w));
                    x[4 * v] = __fsub_rn(p0.x, q0.y);
                    x[4 * v + 1] = __fadd_rn(q0.x, p0.y);
                    x[4 * v + 2] = __fsub_rn(p1.x, q1.y);
                    x[4 * v + 3] = __fadd_rn(q1.x, p1.y);
                }
            }
        } else {
#pragma unroll
            for (int c = 0; c < CH; ++c) x[c] = 0.f;
        }
        if constexpr (HAD) {
            hadamard_stage_packed<CH, 1>(x);
            // strides D/kPreTpr .. D/2 across the lanes of the row
#pragma unroll
            for (int m = 1; m < kPreTpr; m <<= 1) hadamard_cross_packed<CH>(x, m, (qd & m) != 0);
        }
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) amax = fmaxf(amax, fabsf(x[c]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) red[warp] = amax;
        __syncthreads();
        amax = red[0];
#pragma unroll
        for (int w = 1; w < NW; ++w) amax = fmaxf(amax, red[w]);
        const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
        if (tid == 0) a.sx[(int64_t)bh * nblk + tl.j] = __fmul_rn(__fdiv_rn(amax, 448.f), a.s_mul);
        uint4* out = reinterpret_cast<uint4*>(a.X8 + ((int64_t)bh * a.Npad + t) * D + qd * CH);
#pragma unroll
        for (int v = 0; v < CH / 16; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = v * 16 + 4 * e;
                const float2 lo = __fmul2_rn(make_float2(x[c], x[c + 1]), make_float2(inv, inv));
                const float2 hi = __fmul2_rn(make_float2(x[c + 2], x[c + 3]), make_float2(inv, inv));
                w[e] = valid ? (cvt_e4m3x2(lo.x, lo.y) | (cvt_e4m3x2(hi.x, hi.y) << 16)) : 0u;
            }
            out[v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        // every thread is done with this stage and with red[] before they are reused
        __syncthreads();
        tl = tl_next;
        tl_next = tl_after;
    }
    cp_async_wait0();
}

struct VArgs {
    const uint16_t* V;
    int64_t s_b, s_n, s_h;
    const int32_t* perm;
    int H, N, nblk;
    int64_t Npad;
    int vsmooth;
    uint16_t* mu;       // [B,H,nblk,D]
    uint32_t* amax_ws;  // [B,H,D] fp32 bit patterns
    uint8_t* V8T;       // [B,H,D,Npad]
    float* sv;          // [B,H,D]
};

constexpr int kVThreads = 256;

// Stages the block's rows of V' (gathered through pi) into shared memory as
// bf16 [128][D] with 16-byte loads; rows beyond the valid count are zero.
// Returns the number of valid rows.
template <int D>
__device__ __forceinline__ int stage_v_block(const VArgs& a, int b, int h, int j, uint16_t* vs, int32_t* src_s) {
    const int bh = b * a.H + h;
    const int t0 = j * kBlock;
    const int cnt = min(kBlock, a.N - t0);
    if (threadIdx.x < kBlock) {
        const int i = threadIdx.x;
        src_s[i] = (i < cnt) ? (a.perm ? __ldg(a.perm + (int64_t)bh * a.N + t0 + i) : t0 + i) : 0;
    }
    __syncthreads();
    const uint16_t* base = a.V + (int64_t)b * a.s_b + (int64_t)h * a.s_h;
    constexpr int CH = D / 8;                     // 16-byte chunks per row
    constexpr int PER = kBlock * CH / kVThreads;  // chunks per thread: all loads in flight, then the stores
    uint4 w[PER];
#pragma unroll
    for (int r = 0; r < PER; ++r) {
        const int e = threadIdx.x + r * kVThreads;
        const int t = e / CH, q = e % CH;
        w[r] = (t < cnt) ? __ldg(reinterpret_cast<const uint4*>(base + (int64_t)src_s[t] * a.s_n) + q)
                         : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int r = 0; r < PER; ++r) {
        const int e = threadIdx.x + r * kVThreads;
        *reinterpret_cast<uint4*>(vs + (e / CH) * D + (e % CH) * 8) = w[r];
    }
    __syncthreads();
    return cnt;
}

// Block means (fp32 sum in token order, one thread per channel) and the
// per-channel maximum of |V' - mu| (atomicMax on the fp32 bit pattern, values
// are >= 0).  One CTA per (block, head, batch).
template <int D>
__global__ void __launch_bounds__(kVThreads) quant_v_stats_kernel(VArgs a) {
    __shared__ __align__(16) uint16_t vs[kBlock * D];
    __shared__ int32_t src_s[kBlock];
    __shared__ float mu_s[D];
    __shared__ float part_s[kVThreads];
    const int b = blockIdx.z, h = blockIdx.y, j = blockIdx.x;
    const int bh = b * a.H + h;
    const int cnt = stage_v_block<D>(a, b, h, j, vs, src_s);
    if (threadIdx.x < D) {
        const int c = threadIdx.x;
        float m = 0.f;
        if (a.vsmooth) {
            float sum = 0.f;
            for (int i = 0; i < cnt; ++i) sum = __fadd_rn(sum, bf16_bits_to_f32(vs[i * D + c]));
            const uint16_t bits = __bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(sum, (float)cnt)));
            a.mu[((int64_t)bh * a.nblk + j) * D + c] = bits;
            m = bf16_bits_to_f32(bits);
        }
        mu_s[c] = m;
    }
    __syncthreads();
    constexpr int PARTS = kVThreads / D;
    const int c = threadIdx.x % D, part = threadIdx.x / D;
    const float m = mu_s[c];
    float amax = 0.f;
    for (int i = part; i < cnt; i += PARTS) amax = fmaxf(amax, fabsf(__fsub_rn(bf16_bits_to_f32(vs[i * D + c]), m)));
    part_s[threadIdx.x] = amax;
    __syncthreads();
    if (threadIdx.x < D) {
        for (int p2 = 1; p2 < PARTS; ++p2) amax = fmaxf(amax, part_s[p2 * D + c]);
        atomicMax(a.amax_ws + (int64_t)bh * D + c, __float_as_uint(amax));
    }
}

// E2M1 value nearest to |y| <= 8 (0, 0.5, 1, 1.5, 2, 3, 4, 6), ties to the
// even code (the one whose mantissa bit is 0), saturating at 6.
__device__ __forceinline__ float e2m1_rne_abs(float y) {
    return y <= 0.25f ? 0.f : y < 0.75f ? 0.5f : y <= 1.25f ? 1.f : y < 1.75f ? 1.5f
         : y <= 2.5f ? 2.f : y < 3.5f ? 3.f : y <= 5.f ? 4.f : 6.f;
}

// Residual codes, written token-contiguous per channel (V8T [B,H,D,Npad]).
// Thread (c, part) converts the block's tokens [part*T, part*T + T) of channel c.
// V4: the residual in the 4-bit form -- E2M1 with a power-of-two scale per 32
// tokens of a channel (the OCP MX rule: the group's largest |x| lands in
// [4, 8), exponent clamped to [-8, 0]) under the channel scale amax/6 -- each
// value stored as its (equal) E4M3 byte.
template <int D, bool V4>
__global__ void __launch_bounds__(kVThreads) quant_v_codes_kernel(VArgs a) {
    __shared__ __align__(16) uint16_t vs[kBlock * D];
    __shared__ int32_t src_s[kBlock];
    const int b = blockIdx.z, h = blockIdx.y, j = blockIdx.x;
    const int bh = b * a.H + h;
    const int cnt = stage_v_block<D>(a, b, h, j, vs, src_s);
    constexpr int PARTS = kVThreads / D;
    constexpr int T = kBlock / PARTS;  // tokens per thread
    const int c = threadIdx.x % D, part = threadIdx.x / D;
    const float m = a.vsmooth ? bf16_bits_to_f32(a.mu[((int64_t)bh * a.nblk + j) * D + c]) : 0.f;
    const float amax = __uint_as_float(a.amax_ws[(int64_t)bh * D + c]);
    constexpr float QMAX = V4 ? 6.f : 448.f;
    const float inv = amax > 0.f ? __fdiv_rn(QMAX, amax) : 0.f;
    if (j == 0 && part == 0) a.sv[(int64_t)bh * D + c] = __fdiv_rn(amax, QMAX);
    uint4* out =
        reinterpret_cast<uint4*>(a.V8T + ((int64_t)bh * D + c) * a.Npad + (int64_t)j * kBlock + part * T);
    if constexpr (V4) {
#pragma unroll
        for (int grp = 0; grp < T / 32; ++grp) {
            const int i0 = part * T + grp * 32;
            float x[32];
            float gmax = 0.f;
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                x[u] = (i0 + u < cnt) ? __fmul_rn(__fsub_rn(bf16_bits_to_f32(vs[(i0 + u) * D + c]), m), inv) : 0.f;
                gmax = fmaxf(gmax, fabsf(x[u]));
            }
            int e = -8;
            if (gmax > 0.f) {
                int ex;
                frexpf(gmax, &ex);  // gmax = f 2^ex, f in [0.5, 1): floor(log2 gmax) = ex - 1
                e = min(max(ex - 3, -8), 0);
            }
            const float up = __int_as_float((127 - e) << 23), down = __int_as_float((127 + e) << 23);  // 2^-e, 2^e
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                uint32_t w[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float xv = x[g * 16 + q4 * 4 + u];
                        v[u] = copysignf(__fmul_rn(e2m1_rne_abs(fabsf(__fmul_rn(xv, up))), down), xv);
                    }
                    w[q4] = cvt_e4m3x2(v[0], v[1]) | (cvt_e4m3x2(v[2], v[3]) << 16);
                }
                out[grp * 2 + g] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        return;
    }
#pragma unroll
    for (int g = 0; g < T / 16; ++g) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = part * T + g * 16 + 4 * e;
            float r[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                r[u] = (i + u < cnt) ? __fmul_rn(__fsub_rn(bf16_bits_to_f32(vs[(i + u) * D + c]), m), inv) : 0.f;
            w[e] = cvt_e4m3x2(r[0], r[1]) | (cvt_e4m3x2(r[2], r[3]) << 16);
        }
        out[g] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ------------------------------------------------------------------ staged chain
//
// The same computation as separate kernels, each writing its result to HBM:
// rotary transform (bf16 -> fp32 [B,N,H,D]), gather of K' and V' into
// [B,H,N,D], Hadamard rotation in place, V block means and residual maxima,
// Q/K block quantization of the fp32 rows, V residual codes.  Every kernel
// rounds in the order the fused kernels do, so the outputs are bit-identical;
// it exists to measure what the fusion saves.

constexpr int kStageThreads = 256;

// Rotary transform of Q (blockIdx.y = 0) and K (1), or a plain conversion
// without a table; one thread per 8 channels of a row, output [B,N,H,D] fp32.
template <int D>
__global__ void __launch_bounds__(kStageThreads)
    rope_stage_kernel(const uint16_t* Q, const uint16_t* K, vc_shape s, const float* rope, float* Qr, float* Kr) {
    constexpr int CPR = D / 8;
    const uint16_t* X = blockIdx.y ? K : Q;
    float* Y = blockIdx.y ? Kr : Qr;
    const int64_t i = (int64_t)blockIdx.x * kStageThreads + threadIdx.x;
    if (i >= (int64_t)s.B * s.N * s.H * CPR) return;
    const int ch = (int)(i % CPR);
    int64_t r = i / CPR;
    const int h = (int)(r % s.H);
    r /= s.H;
    const int n = (int)(r % s.N), b = (int)(r / s.N);
    float x[8];
    load_row_part<8>(X + (int64_t)b * s.s_b + (int64_t)n * s.s_n + (int64_t)h * s.s_h + ch * 8, x);
    if (rope) rotate_pairs<8>(x, rope + (int64_t)n * D + ch * 8);
    float4* o = reinterpret_cast<float4*>(Y + i * 8);
    o[0] = make_float4(x[0], x[1], x[2], x[3]);
    o[1] = make_float4(x[4], x[5], x[6], x[7]);
}

// Gather into cluster order: Kg[b,h,t] = Kr[b,pi(t),h] (fp32 rows, blockIdx.y
// = 0) and Vg[b,h,t] = V[b,pi(t),h] (bf16 rows, 1); one thread per 16 bytes.
template <int D>
__global__ void __launch_bounds__(kStageThreads)
    gather_stage_kernel(const float* Kr, const uint16_t* V, vc_shape s, const int32_t* perm, float* Kg,
                        uint16_t* Vg) {
    const bool isv = blockIdx.y != 0;
    const int cpr = isv ? D / 8 : D / 4;  // 16-byte chunks per row
    const int64_t i = (int64_t)blockIdx.x * kStageThreads + threadIdx.x;
    if (i >= (int64_t)s.B * s.H * s.N * cpr) return;
    const int ch = (int)(i % cpr);
    const int64_t r = i / cpr;  // (b*H + h)*N + t
    const int t = (int)(r % s.N);
    const int64_t bh = r / s.N;
    const int h = (int)(bh % s.H), b = (int)(bh / s.H);
    const int src = perm ? __ldg(perm + r) : t;
    if (isv) {
        const uint4* p = reinterpret_cast<const uint4*>(V + (int64_t)b * s.s_b + (int64_t)src * s.s_n +
                                                        (int64_t)h * s.s_h);
        reinterpret_cast<uint4*>(Vg + r * D)[ch] = __ldg(p + ch);
    } else {
        const uint4* p = reinterpret_cast<const uint4*>(Kr + (((int64_t)b * s.N + src) * s.H + h) * D);
        reinterpret_cast<uint4*>(Kg + r * D)[ch] = __ldg(p + ch);
    }
}

// Hadamard rotation in place of `rows` contiguous fp32 rows of D values in X
// (blockIdx.y = 0) and Y (1): 8 values per thread, D/8 consecutive lanes per
// row; strides 1, 2, 4 inside the thread, 8 .. D/2 across lanes.
template <int D>
__global__ void __launch_bounds__(kStageThreads) hadamard_stage_kernel(float* X, float* Y, int64_t rows) {
    constexpr int CPR = D / 8;
    float* A = blockIdx.y ? Y : X;
    const int64_t i = (int64_t)blockIdx.x * kStageThreads + threadIdx.x;
    const bool valid = i < rows * CPR;  // lanes past the end still join the shuffles
    const int ch = (int)(i % CPR);
    float x[8];
    if (valid) {
        load_row_part<8>(A + i * 8, x);
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) x[c] = 0.f;
    }
    hadamard_local<8>(x);
#pragma unroll
    for (int m = 1; m < CPR; m <<= 1) hadamard_cross<8>(x, m, (ch & m) != 0);
    if (valid) {
        float4* o = reinterpret_cast<float4*>(A + i * 8);
        o[0] = make_float4(x[0], x[1], x[2], x[3]);
        o[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
}

inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t quantize_workspace(const vc_shape& s) { return (size_t)s.B * s.H * s.d * sizeof(uint32_t); }

size_t quantize_staged_workspace(const vc_shape& s) {
    const size_t elems = (size_t)s.B * s.N * s.H * s.d;
    return round256(quantize_workspace(s)) + 3 * round256(elems * sizeof(float)) + round256(elems * 2);
}

template <int D, typename In>
static cudaError_t launch_qk(const QkArgs& qa, const QkArgs& ka, const vc_shape& s, cudaStream_t st) {
    quant_qk_kernel<D, In><<<dim3(s.H * nblk_of(s.N), 1, 2 * s.B), kQkThreads, 0, st>>>(qa, ka);
    return cudaGetLastError();
}

template <int D, bool ROPE, bool HAD>
static cudaError_t launch_qk_pre(const QkArgs& qa, const QkArgs& ka, const vc_shape& s, cudaStream_t st) {
    constexpr int smem = PreCfg<D, ROPE>::SMEM;
    if (ensure_smem_attr(reinterpret_cast<const void*>(quant_qk_pre_kernel<D, ROPE, HAD>), smem) != VC_OK)
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int items = 2 * s.B * s.H * nblk_of(s.N);  // < 2^25 (B*H*Npad < 2^31)
    const int grid = std::min(items, sms > 0 ? sms : 1);
    quant_qk_pre_kernel<D, ROPE, HAD><<<grid, kPreThreads, smem, st>>>(qa, ka, s.B, items);
    return cudaGetLastError();
}

template <int D>
static vc_status launch_v(const uint16_t* V, int64_t s_b, int64_t s_n, int64_t s_h, const vc_shape& s,
                          const int32_t* perm, int vsmooth, uint8_t* V8T, float* sv, uint16_t* mu, void* ws,
                          cudaStream_t st, bool v4 = false) {
    const int nblk = nblk_of(s.N);
    uint32_t* amax_ws = static_cast<uint32_t*>(ws);
    cudaError_t e = cudaMemsetAsync(amax_ws, 0, quantize_workspace(s), st);
    if (e != cudaSuccess) return cuda_status(e);
    VArgs va{V, s_b, s_n, s_h, perm, s.H, s.N, nblk, npad_of(s.N), vsmooth, mu, amax_ws, V8T, sv};
    quant_v_stats_kernel<D><<<dim3(nblk, s.H, s.B), kVThreads, 0, st>>>(va);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
    if (v4) quant_v_codes_kernel<D, true><<<dim3(nblk, s.H, s.B), kVThreads, 0, st>>>(va);
    else quant_v_codes_kernel<D, false><<<dim3(nblk, s.H, s.B), kVThreads, 0, st>>>(va);
    return cuda_status(cudaGetLastError());
}

template <int D>
static vc_status launch_quantize_d(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const vc_shape& s,
                                   const int32_t* perm, int vsmooth, const Preproc& pp, uint8_t* Q8, float* sq,
                                   uint8_t* K8, float* sk, uint8_t* V8T, float* sv, uint16_t* mu, void* ws,
                                   cudaStream_t st) {
    const int nblk = nblk_of(s.N);
    const int64_t Npad = npad_of(s.N);
    const float qmul = pp.hadamard ? 1.0f / (float)D : 1.0f;
    QkArgs qa{Q, s.s_b, s.s_n, s.s_h, nullptr, pp.rope, qmul, Q8, sq, s.H, s.N, nblk, Npad};
    QkArgs ka{K, s.s_b, s.s_n, s.s_h, perm, pp.rope, 1.0f, K8, sk, s.H, s.N, nblk, Npad};
    cudaError_t e;
    if (pp.rope)
        e = pp.hadamard ? launch_qk_pre<D, true, true>(qa, ka, s, st) : launch_qk_pre<D, true, false>(qa, ka, s, st);
    else
        e = pp.hadamard ? launch_qk_pre<D, false, true>(qa, ka, s, st) : launch_qk<D, uint16_t>(qa, ka, s, st);
    if (e != cudaSuccess) return cuda_status(e);
    return launch_v<D>(V, s.s_b, s.s_n, s.s_h, s, perm, vsmooth, V8T, sv, mu, ws, st, pp.v4 != 0);
}

vc_status launch_quantize(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const vc_shape& s,
                          const int32_t* perm, int vsmooth, const Preproc& pp, uint8_t* Q8, float* sq, uint8_t* K8,
                          float* sk, uint8_t* V8T, float* sv, uint16_t* mu, void* ws, cudaStream_t st) {
    if (s.d == 128)
        return launch_quantize_d<128>(Q, K, V, s, perm, vsmooth, pp, Q8, sq, K8, sk, V8T, sv, mu, ws, st);
    return launch_quantize_d<64>(Q, K, V, s, perm, vsmooth, pp, Q8, sq, K8, sk, V8T, sv, mu, ws, st);
}

template <int D>
static vc_status launch_staged_d(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const vc_shape& s,
                                 const int32_t* perm, int vsmooth, const Preproc& pp, uint8_t* Q8, float* sq,
                                 uint8_t* K8, float* sk, uint8_t* V8T, float* sv, uint16_t* mu, void* ws,
                                 cudaStream_t st) {
    const size_t elems = (size_t)s.B * s.N * s.H * D;
    uint8_t* w = static_cast<uint8_t*>(ws);
    void* amax_ws = w;
    w += round256(quantize_workspace(s));
    float* Qr = reinterpret_cast<float*>(w);
    w += round256(elems * sizeof(float));
    float* Kr = reinterpret_cast<float*>(w);
    w += round256(elems * sizeof(float));
    float* Kg = reinterpret_cast<float*>(w);
    w += round256(elems * sizeof(float));
    uint16_t* Vg = reinterpret_cast<uint16_t*>(w);

    const int64_t chunks8 = (int64_t)elems / 8;
    rope_stage_kernel<D><<<dim3((unsigned)((chunks8 + kStageThreads - 1) / kStageThreads), 2), kStageThreads, 0,
                           st>>>(Q, K, s, pp.rope, Qr, Kr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
    const int64_t chunks16 = (int64_t)elems / 4;  // K rows in 16-byte chunks (V rows need half as many)
    gather_stage_kernel<D><<<dim3((unsigned)((chunks16 + kStageThreads - 1) / kStageThreads), 2), kStageThreads,
                             0, st>>>(Kr, V, s, perm, Kg, Vg);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
    if (pp.hadamard) {
        hadamard_stage_kernel<D><<<dim3((unsigned)((chunks8 + kStageThreads - 1) / kStageThreads), 2),
                                   kStageThreads, 0, st>>>(Qr, Kg, (int64_t)elems / D);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_status(e);
    }
    // V' is now contiguous [B,H,N,D] in cluster order
    const int64_t vs_b = (int64_t)s.H * s.N * D, vs_n = D, vs_h = (int64_t)s.N * D;
    vc_status vst = launch_v<D>(Vg, vs_b, vs_n, vs_h, s, nullptr, vsmooth, V8T, sv, mu, amax_ws, st);
    if (vst != VC_OK) return vst;
    const int nblk = nblk_of(s.N);
    const int64_t Npad = npad_of(s.N);
    const float qmul = pp.hadamard ? 1.0f / (float)D : 1.0f;
    QkArgs qa{Qr, (int64_t)s.N * s.H * D, (int64_t)s.H * D, D, nullptr, nullptr, qmul, Q8, sq, s.H, s.N, nblk, Npad};
    QkArgs ka{Kg, vs_b, vs_n, vs_h, nullptr, nullptr, 1.0f, K8, sk, s.H, s.N, nblk, Npad};
    return cuda_status(launch_qk<D, float>(qa, ka, s, st));
}

vc_status launch_quantize_staged(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const vc_shape& s,
                                 const int32_t* perm, int vsmooth, const Preproc& pp, uint8_t* Q8, float* sq,
                                 uint8_t* K8, float* sk, uint8_t* V8T, float* sv, uint16_t* mu, void* ws,
                                 cudaStream_t st) {
    if (s.d == 128)
        return launch_staged_d<128>(Q, K, V, s, perm, vsmooth, pp, Q8, sq, K8, sk, V8T, sv, mu, ws, st);
    return launch_staged_d<64>(Q, K, V, s, perm, vsmooth, pp, Q8, sq, K8, sk, V8T, sv, mu, ws, st);
}

}  // namespace vc

// ------------------------------------------------------------------ fixed-scratch variant
//
// vc_quantize needs B*H*d words of device scratch for the per-channel residual
// maxima.  Some callers cannot hand it any: a host that embeds this library
// inside a framework whose memory pool owns all device memory (a raw
// cudaMalloc would bypass its accounting), or code that runs where an
// allocation would synchronize the device or is simply not permitted.  For
// them vc_quantize_static keeps that scratch in a fixed array inside this
// library instead.
#include <mutex>

namespace vc {
namespace {

constexpr size_t kStaticScratchWords = 65536;  // B*H*d <= 65536 (256 KB, held by every GPU that loads the library)
__device__ __align__(256) uint32_t g_quantize_scratch[kStaticScratchWords];

constexpr int kMaxContexts = 64;
std::mutex g_scratch_mutex;
struct ScratchEntry {
    CtxKey key;
    void* addr;
};
ScratchEntry g_scratch_addr[kMaxContexts] = {};
int g_scratch_n = 0;

// Device address of g_quantize_scratch in the current context; looked up once
// per context, with that context's device current (the host-side name is only
// a stand-in, never a device pointer).  Keyed by the context handle, so a
// context destroyed by a device reset and recreated gets a fresh lookup.
vc_status static_scratch(void** out) {
    CtxKey key;
    if (current_ctx(&key) != VC_OK) return VC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (key.ctx) {
        for (int i = 0; i < g_scratch_n; ++i)
            if (g_scratch_addr[i].key == key) {
                *out = g_scratch_addr[i].addr;
                return VC_OK;
            }
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_quantize_scratch) != cudaSuccess || !p) return VC_ERR_CUDA;
    // the lookup initialises the context if none was current yet
    if (!key.ctx && current_ctx(&key) != VC_OK) return VC_ERR_CUDA;
    if (key.ctx) {
        if (g_scratch_n < kMaxContexts) g_scratch_addr[g_scratch_n++] = ScratchEntry{key, p};
        else g_scratch_addr[kMaxContexts - 1] = ScratchEntry{key, p};
    }
    *out = p;
    return VC_OK;
}

}  // namespace
}  // namespace vc

extern "C" vc_status vc_quantize_static(const void* Q, const void* K, const void* V, vc_shape shape,
                                        const int32_t* perm, int vsmooth, uint8_t* Q8, float* sq, uint8_t* K8,
                                        float* sk, uint8_t* V8T, float* sv, void* mu, vc_stream_t stream) {
    using namespace vc;
    vc_status st = quantize_args(Q, K, V, shape, vsmooth, nullptr, 0, Q8, sq, K8, sk, V8T, sv, mu);
    if (st != VC_OK) return st;
    if ((size_t)shape.B * shape.H * shape.d > kStaticScratchWords) return VC_ERR_WORKSPACE;
    void* scratch = nullptr;
    st = static_scratch(&scratch);
    if (st != VC_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t *q = static_cast<const uint16_t*>(Q), *k = static_cast<const uint16_t*>(K),
                   *v = static_cast<const uint16_t*>(V);
    uint16_t* m = static_cast<uint16_t*>(mu);
    return launch_quantize(q, k, v, shape, perm, vsmooth, Preproc{}, Q8, sq, K8, sk, V8T, sv, m, scratch, cs);
}
