// vc_quantize.cu -- the fused quantizer of the V-Smooth path.
//
// Paper summary (paper.rainbus.top), 方法步骤详情 step 2 and 前置知识 "低比特
// 量化与离群值"; dimensionstp.github.io section 2-2:
//   Q, K' = K[pi]: one fp32 scale per 128-token block, codes = E4M3(x * 448/amax).
//   V' = V[pi]:   mu_j = bf16(block mean), R = V' - mu_j, residual codes with
//                 one scale per channel over the whole head.
// Three memory-bound kernels per call:
//   quant_qk_kernel      Q and K' blocks (gathered rows for K'), one CTA per block.
//   quant_v_stats_kernel block means of V' and the per-channel residual amax
//                        (atomicMax on the fp32 bit pattern, values are >= 0).
//   quant_v_codes_kernel residual codes, written token-contiguous per channel
//                        (V8T [B,H,d,Npad]) so that the attention kernel can
//                        read V as a K-major MMA operand.
// The two V kernels stage each block's gathered rows in shared memory with
// 16-byte loads; the per-channel scale needs the whole head, hence two passes.
// Every rounding step is written with an explicit _rn intrinsic so that the
// codes are bit-reproducible: fp32 block sum in token order, IEEE division,
// round-to-nearest-even conversions (cvt.rn.satfinite.e4m3x2).
#include <cuda_bf16.h>

#include "vc_device.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr int kQkThreads = 256;

struct QkArgs {
    const uint16_t* X;
    int64_t s_b, s_n, s_h;
    const int32_t* perm;  // may be null
    uint8_t* X8;
    float* sx;
    int H, N, nblk;
    int64_t Npad;
};

// One CTA per (block j, head h, batch b, tensor which); 2 threads per token row.
template <int D>
__global__ void __launch_bounds__(kQkThreads) quant_qk_kernel(QkArgs q, QkArgs k) {
    constexpr int CH = D / 2;           // channels per thread
    constexpr int NV = CH / 8;          // 16-byte vectors per thread
    const QkArgs& a = (blockIdx.z & 1) ? k : q;
    const int b = blockIdx.z >> 1, h = blockIdx.y, j = blockIdx.x;
    const int bh = b * a.H + h;
    const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int t = j * kBlock + row;
    const bool valid = t < a.N;

    float x[CH];
    float amax = 0.f;
    if (valid) {
        const int src = a.perm ? __ldg(a.perm + (int64_t)bh * a.N + t) : t;
        const uint4* p = reinterpret_cast<const uint4*>(a.X + (int64_t)b * a.s_b + (int64_t)src * a.s_n +
                                                        (int64_t)h * a.s_h + half * CH);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            uint4 w = __ldg(p + v);
            uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[v * 8 + 2 * e] = bf16_bits_to_f32(ws[e] & 0xFFFFu);
                x[v * 8 + 2 * e + 1] = bf16_bits_to_f32(ws[e] >> 16);
            }
        }
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
    if (threadIdx.x == 0) a.sx[(int64_t)bh * a.nblk + j] = __fdiv_rn(amax, 448.f);

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
    constexpr int CH = D / 8;  // 16-byte chunks per row
#pragma unroll 4
    for (int e = threadIdx.x; e < kBlock * CH; e += kVThreads) {
        const int t = e / CH, q = e % CH;
        uint4 w = make_uint4(0, 0, 0, 0);
        if (t < cnt) w = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)src_s[t] * a.s_n) + q);
        *reinterpret_cast<uint4*>(vs + t * D + q * 8) = w;
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

// Residual codes, written token-contiguous per channel (V8T [B,H,D,Npad]).
// Thread (c, part) converts the block's tokens [part*T, part*T + T) of channel c.
template <int D>
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
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
    if (j == 0 && part == 0) a.sv[(int64_t)bh * D + c] = __fdiv_rn(amax, 448.f);
    uint4* out =
        reinterpret_cast<uint4*>(a.V8T + ((int64_t)bh * D + c) * a.Npad + (int64_t)j * kBlock + part * T);
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

}  // namespace

size_t quantize_workspace(const vc_shape& s) { return (size_t)s.B * s.H * s.d * sizeof(uint32_t); }

template <int D>
static vc_status launch_quantize_d(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const vc_shape& s,
                                   const int32_t* perm, int vsmooth, uint8_t* Q8, float* sq, uint8_t* K8,
                                   float* sk, uint8_t* V8T, float* sv, uint16_t* mu, void* ws, cudaStream_t st) {
    const int nblk = nblk_of(s.N);
    const int64_t Npad = npad_of(s.N);
    QkArgs qa{Q, s.s_b, s.s_n, s.s_h, nullptr, Q8, sq, s.H, s.N, nblk, Npad};
    QkArgs ka{K, s.s_b, s.s_n, s.s_h, perm, K8, sk, s.H, s.N, nblk, Npad};
    quant_qk_kernel<D><<<dim3(nblk, s.H, 2 * s.B), kQkThreads, 0, st>>>(qa, ka);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
    uint32_t* amax_ws = static_cast<uint32_t*>(ws);
    e = cudaMemsetAsync(amax_ws, 0, quantize_workspace(s), st);
    if (e != cudaSuccess) return cuda_status(e);
    VArgs va{V, s.s_b, s.s_n, s.s_h, perm, s.H, s.N, nblk, Npad, vsmooth, mu, amax_ws, V8T, sv};
    quant_v_stats_kernel<D><<<dim3(nblk, s.H, s.B), kVThreads, 0, st>>>(va);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
    quant_v_codes_kernel<D><<<dim3(nblk, s.H, s.B), kVThreads, 0, st>>>(va);
    return cuda_status(cudaGetLastError());
}

vc_status launch_quantize(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const vc_shape& s,
                          const int32_t* perm, int vsmooth, uint8_t* Q8, float* sq, uint8_t* K8, float* sk,
                          uint8_t* V8T, float* sv, uint16_t* mu, void* ws, cudaStream_t st) {
    if (s.d == 128)
        return launch_quantize_d<128>(Q, K, V, s, perm, vsmooth, Q8, sq, K8, sk, V8T, sv, mu, ws, st);
    return launch_quantize_d<64>(Q, K, V, s, perm, vsmooth, Q8, sq, K8, sk, V8T, sv, mu, ws, st);
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

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_quantize_scratch on the current device; looked up once
// per device (the host-side name is only a stand-in, never a device pointer).
vc_status static_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_quantize_scratch) != cudaSuccess || !p) return VC_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return VC_OK;
}

bool aligned16_q(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace vc

extern "C" vc_status vc_quantize_static(const void* Q, const void* K, const void* V, vc_shape shape,
                                        const int32_t* perm, int vsmooth, uint8_t* Q8, float* sq, uint8_t* K8,
                                        float* sk, uint8_t* V8T, float* sv, void* mu, vc_stream_t stream) {
    using namespace vc;
    vc_status st = check_shape(shape);
    if (st != VC_OK) return st;
    if (vsmooth != 0 && vsmooth != 1) return VC_ERR_INVALID_ARG;
    if (!Q || !K || !V || !Q8 || !sq || !K8 || !sk || !V8T || !sv || (vsmooth && !mu)) return VC_ERR_INVALID_ARG;
    if (!aligned16_q(Q) || !aligned16_q(K) || !aligned16_q(V) || !aligned16_q(Q8) || !aligned16_q(K8) ||
        !aligned16_q(V8T))
        return VC_ERR_INVALID_ARG;
    if ((size_t)shape.B * shape.H * shape.d > kStaticScratchWords) return VC_ERR_WORKSPACE;
    void* scratch = nullptr;
    st = static_scratch(&scratch);
    if (st != VC_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t *q = static_cast<const uint16_t*>(Q), *k = static_cast<const uint16_t*>(K),
                   *v = static_cast<const uint16_t*>(V);
    uint16_t* m = static_cast<uint16_t*>(mu);
    if (shape.d == 128) return launch_quantize_d<128>(q, k, v, shape, perm, vsmooth, Q8, sq, K8, sk, V8T, sv, m, scratch, cs);
    return launch_quantize_d<64>(q, k, v, shape, perm, vsmooth, Q8, sq, K8, sk, V8T, sv, m, scratch, cs);
}
