// vc_cluster.cu -- the grouping step of V-Smooth.
//
// Paper summary (paper.rainbus.top), 方法步骤详情 step 1: online (inference-time)
// k-means on the value tokens of each (batch, head), warm-started from the
// previous denoising step's centroids, then pi = argsort(z); dimensionstp.github.io
// section 2-1 (K' = K[pi], V' = V[pi]).
//
// One Lloyd iteration = four launches:
//   centroid_norms   |c_i|^2 in fp32.
//   assign_kernel    z_t = argmin_i |c_i|^2 - 2 v_t.c_i (fp32 CUDA-core tiles:
//                    128 tokens x 64 centroids per step, 8x4 register blocking).
//   seg_hist / seg_scan / seg_scatter
//                    stable counting sort of z in segments of kSeg tokens:
//                    per-segment histograms, one exclusive scan per head in
//                    (label, segment) order, then an in-order scatter where each
//                    warp ranks equal labels with __match_any_sync.  The result
//                    is the stable argsort pi (ascending label, token order).
//   update_kernel    centroid i = fp32 mean of its members, read contiguously
//                    through pi; empty clusters keep their centroid.
// Labels and pi of the last assignment are the outputs.
#include "vc_device.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr int kSeg = 4096;      // tokens per sort segment
constexpr int kTokTile = 128;   // tokens per assign CTA
constexpr int kCenTile = 64;    // centroids per assign step
constexpr int kAssignThreads = 256;

struct ClusterWs {
    float* cnorm;       // [BH, k]
    int32_t* seg;       // [BH, nseg, k]: counts, then exclusive offsets
    int32_t* count;     // [BH, k]
    int32_t* start;     // [BH, k]
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

ClusterWs carve(void* ws, const vc_shape& s, int k) {
    const size_t BH = (size_t)s.B * s.H;
    const size_t nseg = (s.N + kSeg - 1) / kSeg;
    char* p = static_cast<char*>(ws);
    ClusterWs w;
    w.cnorm = reinterpret_cast<float*>(p);
    p += align256(BH * k * sizeof(float));
    w.seg = reinterpret_cast<int32_t*>(p);
    p += align256(BH * nseg * k * sizeof(int32_t));
    w.count = reinterpret_cast<int32_t*>(p);
    p += align256(BH * k * sizeof(int32_t));
    w.start = reinterpret_cast<int32_t*>(p);
    return w;
}

__device__ __forceinline__ const uint16_t* tok_ptr(const uint16_t* V, const vc_shape& s, int b, int h, int n) {
    return V + (int64_t)b * s.s_b + (int64_t)n * s.s_n + (int64_t)h * s.s_h;
}

// Cold start: centroid i = token floor(i*N/k).
__global__ void init_centroids(const uint16_t* V, vc_shape s, int k, float* cent) {
    const int i = blockIdx.x, bh = blockIdx.y;
    const int b = bh / s.H, h = bh % s.H;
    const int src = (int)(((int64_t)i * s.N) / k);
    const uint16_t* v = tok_ptr(V, s, b, h, src);
    for (int c = threadIdx.x; c < s.d; c += blockDim.x)
        cent[((int64_t)bh * k + i) * s.d + c] = bf16_bits_to_f32(v[c]);
}

__global__ void centroid_norms(const float* cent, int k, int d, float* cnorm) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x, bh = blockIdx.y;
    if (i >= k) return;
    const float* c = cent + ((int64_t)bh * k + i) * d;
    float acc = 0.f;
    for (int e = 0; e < d; ++e) acc = __fmaf_rn(c[e], c[e], acc);
    cnorm[(int64_t)bh * k + i] = acc;
}

// z_t = argmin_i (|c_i|^2 - 2 v_t . c_i), ties to the lowest index.
template <int D>
__global__ void __launch_bounds__(kAssignThreads) assign_kernel(const uint16_t* V, vc_shape s, int k,
                                                                const float* cent, const float* cnorm,
                                                                int32_t* labels) {
    extern __shared__ __align__(16) float sm[];
    float* vt = sm;                                // [D][kTokTile + 4]
    float* ct = vt + D * (kTokTile + 4);           // [D][kCenTile + 4]
    __shared__ float best_s[16][kTokTile];
    __shared__ int arg_s[16][kTokTile];
    const int bh = blockIdx.y, b = bh / s.H, h = bh % s.H;
    const int t0 = blockIdx.x * kTokTile;
    const int tid = threadIdx.x;
    // token tile, transposed to [channel][token]
    for (int e = tid; e < kTokTile * (D / 8); e += kAssignThreads) {
        const int t = e / (D / 8), c8 = (e % (D / 8)) * 8;
        float f[8];
        if (t0 + t < s.N) {
            const uint4 w = *reinterpret_cast<const uint4*>(tok_ptr(V, s, b, h, t0 + t) + c8);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                f[2 * q] = bf16_bits_to_f32(ws[q] & 0xFFFFu);
                f[2 * q + 1] = bf16_bits_to_f32(ws[q] >> 16);
            }
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) vt[(c8 + q) * (kTokTile + 4) + t] = f[q];
    }
    const int tg = tid / 16, cg = tid % 16;   // 16 token groups of 8, 16 centroid groups of 4
    float best[8];
    int arg[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) { best[r] = INFINITY; arg[r] = 0; }
    const float* cb = cent + (int64_t)bh * k * D;
    for (int i0 = 0; i0 < k; i0 += kCenTile) {
        __syncthreads();
        for (int e = tid; e < kCenTile * D; e += kAssignThreads) {
            const int i = e / D, c = e % D;
            ct[c * (kCenTile + 4) + i] = (i0 + i < k) ? cb[(int64_t)(i0 + i) * D + c] : 0.f;
        }
        __syncthreads();
        float acc[8][4];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[r][q] = 0.f;
#pragma unroll 4
        for (int c = 0; c < D; ++c) {
            const float4 va = *reinterpret_cast<const float4*>(vt + c * (kTokTile + 4) + tg * 8);
            const float4 vb = *reinterpret_cast<const float4*>(vt + c * (kTokTile + 4) + tg * 8 + 4);
            const float4 cc = *reinterpret_cast<const float4*>(ct + c * (kCenTile + 4) + cg * 4);
            const float vv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
            const float cv[4] = {cc.x, cc.y, cc.z, cc.w};
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[r][q] = __fmaf_rn(vv[r], cv[q], acc[r][q]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = i0 + cg * 4 + q;
            if (i < k) {
                const float cn = cnorm[(int64_t)bh * k + i];
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const float dist = __fmaf_rn(-2.f, acc[r][q], cn);
                    if (dist < best[r]) { best[r] = dist; arg[r] = i; }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        best_s[cg][tg * 8 + r] = best[r];
        arg_s[cg][tg * 8 + r] = arg[r];
    }
    __syncthreads();
    if (tid < kTokTile && t0 + tid < s.N) {
        float bv = best_s[0][tid];
        int ba = arg_s[0][tid];
        for (int g = 1; g < 16; ++g) {
            const float v = best_s[g][tid];
            const int a = arg_s[g][tid];
            if (v < bv || (v == bv && a < ba)) { bv = v; ba = a; }
        }
        labels[(int64_t)bh * s.N + t0 + tid] = ba;
    }
}

// Per-segment label histograms.
__global__ void seg_hist(const int32_t* labels, int N, int k, int nseg, int32_t* seg) {
    extern __shared__ int32_t hist[];
    const int sgi = blockIdx.x, bh = blockIdx.y;
    for (int i = threadIdx.x; i < k; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int t0 = sgi * kSeg, t1 = min(N, t0 + kSeg);
    for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) atomicAdd(&hist[labels[(int64_t)bh * N + t]], 1);
    __syncthreads();
    for (int i = threadIdx.x; i < k; i += blockDim.x) seg[((int64_t)bh * nseg + sgi) * k + i] = hist[i];
}

// Exclusive scan per head over (label, segment) in label-major order.
__global__ void seg_scan(int k, int nseg, int32_t* seg, int32_t* count, int32_t* start) {
    const int bh = blockIdx.x;
    __shared__ int32_t tot[1024];
    for (int i = threadIdx.x; i < k; i += blockDim.x) {
        int acc = 0;
        for (int g = 0; g < nseg; ++g) acc += seg[((int64_t)bh * nseg + g) * k + i];
        tot[i] = acc;
        count[(int64_t)bh * k + i] = acc;
    }
    __syncthreads();
    // exclusive scan of tot[0..k) by one warp (k <= 1024)
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = (k + 31) / 32;
        int local = 0;
        for (int e = 0; e < per; ++e) {
            const int i = lane * per + e;
            if (i < k) local += tot[i];
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int e = 0; e < per; ++e) {
            const int i = lane * per + e;
            if (i < k) {
                const int v = tot[i];
                tot[i] = run;
                run += v;
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < k; i += blockDim.x) {
        int run = tot[i];
        start[(int64_t)bh * k + i] = run;
        for (int g = 0; g < nseg; ++g) {
            int32_t* p = seg + ((int64_t)bh * nseg + g) * k + i;
            const int v = *p;
            *p = run;
            run += v;
        }
    }
}

// Stable scatter: one warp walks its segment in token order, 32 tokens at a time.
__global__ void seg_scatter(const int32_t* labels, int N, int k, int nseg, const int32_t* seg, int32_t* perm) {
    extern __shared__ int32_t cursor[];
    const int sgi = blockIdx.x, bh = blockIdx.y, lane = threadIdx.x;
    for (int i = lane; i < k; i += 32) cursor[i] = seg[((int64_t)bh * nseg + sgi) * k + i];
    __syncwarp();
    const int t0 = sgi * kSeg, t1 = min(N, t0 + kSeg);
    for (int base = t0; base < t1; base += 32) {
        const int t = base + lane;
        const bool valid = t < t1;
        const int lab = valid ? labels[(int64_t)bh * N + t] : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, lab);
        const unsigned lower = peers & ((1u << lane) - 1u);
        int pos = 0;
        if (valid) {
            pos = cursor[lab] + __popc(lower);
            perm[(int64_t)bh * N + pos] = t;
        }
        __syncwarp();
        // the highest lane of each group advances the cursor
        if (valid && (peers >> lane) == 1u) cursor[lab] = pos + 1;
        __syncwarp();
    }
}

// Centroid i = mean of its members (fp32 sum through pi); empty keeps the old value.
template <int D>
__global__ void __launch_bounds__(D) update_kernel(const uint16_t* V, vc_shape s, int k, const int32_t* perm,
                                                   const int32_t* count, const int32_t* start, float* cent) {
    const int i = blockIdx.x, bh = blockIdx.y, b = bh / s.H, h = bh % s.H, c = threadIdx.x;
    const int n = count[(int64_t)bh * k + i];
    if (n == 0) return;
    const int st = start[(int64_t)bh * k + i];
    const int32_t* p = perm + (int64_t)bh * s.N + st;
    float acc = 0.f;
    int e = 0;
    for (; e + 4 <= n; e += 4) {
        const int t0 = p[e], t1 = p[e + 1], t2 = p[e + 2], t3 = p[e + 3];
        const float v0 = bf16_bits_to_f32(tok_ptr(V, s, b, h, t0)[c]);
        const float v1 = bf16_bits_to_f32(tok_ptr(V, s, b, h, t1)[c]);
        const float v2 = bf16_bits_to_f32(tok_ptr(V, s, b, h, t2)[c]);
        const float v3 = bf16_bits_to_f32(tok_ptr(V, s, b, h, t3)[c]);
        acc = __fadd_rn(__fadd_rn(acc, v0), __fadd_rn(v1, __fadd_rn(v2, v3)));
    }
    for (; e < n; ++e) acc = __fadd_rn(acc, bf16_bits_to_f32(tok_ptr(V, s, b, h, p[e])[c]));
    cent[((int64_t)bh * k + i) * D + c] = __fdiv_rn(acc, (float)n);
}

}  // namespace

size_t cluster_workspace(const vc_shape& s, int k) {
    const size_t BH = (size_t)s.B * s.H;
    const size_t nseg = (s.N + kSeg - 1) / kSeg;
    return align256(BH * k * 4) + align256(BH * nseg * k * 4) + align256(BH * k * 4) + align256(BH * k * 4);
}

template <int D>
static vc_status launch_cluster_d(const uint16_t* V, const vc_shape& s, int k, int iters, int warm, float* cent,
                                  int32_t* labels, int32_t* perm, void* ws, cudaStream_t st) {
    const int BH = s.B * s.H;
    const int nseg = (s.N + kSeg - 1) / kSeg;
    ClusterWs w = carve(ws, s, k);
    if (!warm) init_centroids<<<dim3(k, BH), 128, 0, st>>>(V, s, k, cent);
    const size_t assign_smem = (size_t)D * (kTokTile + 4) * 4 + (size_t)D * (kCenTile + 4) * 4;
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(assign_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)assign_smem);
        attr_set = true;
    }
    for (int it = 0; it < iters; ++it) {
        centroid_norms<<<dim3((unsigned)((k + 127) / 128), BH), 128, 0, st>>>(cent, k, D, w.cnorm);
        assign_kernel<D><<<dim3((s.N + kTokTile - 1) / kTokTile, BH), kAssignThreads, assign_smem, st>>>(
            V, s, k, cent, w.cnorm, labels);
        seg_hist<<<dim3(nseg, BH), 256, k * 4, st>>>(labels, s.N, k, nseg, w.seg);
        seg_scan<<<BH, 256, 0, st>>>(k, nseg, w.seg, w.count, w.start);
        seg_scatter<<<dim3(nseg, BH), 32, k * 4, st>>>(labels, s.N, k, nseg, w.seg, perm);
        update_kernel<D><<<dim3(k, BH), D, 0, st>>>(V, s, k, perm, w.count, w.start, cent);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_status(e);
    }
    return VC_OK;
}

vc_status launch_cluster(const uint16_t* V, const vc_shape& s, int k, int iters, int warm, float* cent,
                         int32_t* labels, int32_t* perm, void* ws, int32_t* dev_status, cudaStream_t st) {
    (void)dev_status;  // no device-side waits in these kernels
    if (s.d == 128) return launch_cluster_d<128>(V, s, k, iters, warm, cent, labels, perm, ws, st);
    return launch_cluster_d<64>(V, s, k, iters, warm, cent, labels, perm, ws, st);
}

}  // namespace vc
