// vc_cluster.cu -- the grouping step of V-Smooth.
//
// Paper summary (paper.rainbus.top), 方法步骤详情 step 1: online (inference-time)
// k-means on the value tokens of each (batch, head), warm-started from the
// previous denoising step's centroids, then pi = argsort(z); dimensionstp.github.io
// section 2-1 (K' = K[pi], V' = V[pi]).
//
// One Lloyd iteration = an assignment, the counting sort and the update:
//   assign_tc_kernel (k <= 256, the case the workloads use)
//                    z_t = argmin_i |c_i|^2 - 2 v_t.c_i with v.c on tcgen05
//                    (bf16 token tiles by TMA against the centroids split into
//                    two bf16 parts, fp32 accumulators in TMEM; |c|^2 and the
//                    argmin in the epilogue warps); one persistent launch.
//   centroid_norms + assign_kernel (k > 256)
//                    |c_i|^2 in fp32, then the same argmin on fp32 CUDA-core
//                    tiles (128 tokens x 64 centroids per step, 8x4 register
//                    blocking).
//   seg_hist / seg_scan / seg_scatter
//                    stable counting sort of z in segments of kSeg tokens:
//                    per-segment histograms, one exclusive scan per head in
//                    (label, segment) order, then an in-order scatter where each
//                    warp ranks equal labels with __match_any_sync.  The result
//                    is the stable argsort pi (ascending label, token order).
//   update_kernel    centroid i = fp32 mean of its members, read contiguously
//                    through pi; empty clusters keep their centroid.
// Labels and pi of the last assignment are the outputs.
//
// Block fill (optional, after the last iteration): the permutation that keeps
// each cluster's whole 128-token blocks together (label order) and then places
// the clusters' leftovers along a greedy nearest-centroid chain -- the cheap
// balancing the paper summary's own analysis proposes (独立分析的弱点, weakness
// one: greedy backfill instead of balanced k-means).
//   fill_chain_kernel    one CTA per head: whole-block prefix sums in label
//                        order, the greedy chain over the clusters with
//                        leftovers (fp32 squared distances summed over the
//                        channels in order, ties to the lower label), the
//                        leftover prefix sums in chain order.
//   fill_scatter_kernel  moves every entry of the stable argsort to its place.
#include <algorithm>

#include <cuda_bf16.h>

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
    int32_t* fdst;      // [BH, k] block fill: destination of a cluster's whole blocks
    int32_t* ldst;      // [BH, k] block fill: destination of a cluster's leftovers
    int32_t* pi_sort;   // [BH, N] block fill: the stable argsort before the fill
    float* cT;          // [BH, d, k] block fill: centroids transposed (coalesced chain reads)
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
    p += align256(BH * k * sizeof(int32_t));
    w.fdst = reinterpret_cast<int32_t*>(p);
    p += align256(BH * k * sizeof(int32_t));
    w.ldst = reinterpret_cast<int32_t*>(p);
    p += align256(BH * k * sizeof(int32_t));
    w.pi_sort = reinterpret_cast<int32_t*>(p);
    p += align256(BH * (size_t)s.N * sizeof(int32_t));
    w.cT = reinterpret_cast<float*>(p);
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

// Centroid i = mean of its members (fp32 sums through pi); empty keeps the old
// value.  A CTA per (centroid, head): D/8 lanes each own 8 channels (one
// 16-byte load per member row), 256/(D/8) member groups stride over the
// members, then the groups' partial sums are added in shared memory.
constexpr int kUpdThreads = 256;

template <int D>
__global__ void __launch_bounds__(kUpdThreads) update_kernel(const uint16_t* V, vc_shape s, int k,
                                                             const int32_t* perm, const int32_t* count,
                                                             const int32_t* start, float* cent) {
    constexpr int LANES = D / 8;
    constexpr int GROUPS = kUpdThreads / LANES;
    __shared__ float red[GROUPS][D];
    const int i = blockIdx.x, bh = blockIdx.y, b = bh / s.H, h = bh % s.H;
    const int n = count[(int64_t)bh * k + i];
    if (n == 0) return;
    const int st = start[(int64_t)bh * k + i];
    const int32_t* p = perm + (int64_t)bh * s.N + st;
    const int lane = threadIdx.x % LANES, grp = threadIdx.x / LANES;
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    auto add_row = [&](const uint4 w) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc[2 * q] = __fadd_rn(acc[2 * q], bf16_bits_to_f32(ws[q] & 0xFFFFu));
            acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], bf16_bits_to_f32(ws[q] >> 16));
        }
    };
    int e = grp;
    for (; e + 3 * GROUPS < n; e += 4 * GROUPS) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            w[u] = __ldg(reinterpret_cast<const uint4*>(tok_ptr(V, s, b, h, __ldg(p + e + u * GROUPS)) + lane * 8));
#pragma unroll
        for (int u = 0; u < 4; ++u) add_row(w[u]);
    }
    for (; e < n; e += GROUPS)
        add_row(__ldg(reinterpret_cast<const uint4*>(tok_ptr(V, s, b, h, __ldg(p + e)) + lane * 8)));
#pragma unroll
    for (int q = 0; q < 8; ++q) red[grp][lane * 8 + q] = acc[q];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += kUpdThreads) {
        float sum = 0.f;
#pragma unroll 8
        for (int g = 0; g < GROUPS; ++g) sum = __fadd_rn(sum, red[g][c]);
        cent[((int64_t)bh * k + i) * D + c] = __fdiv_rn(sum, (float)n);
    }
}

// ------------------------------------------------------------ assignment on the tensor cores
//
// z_t = argmin_i (|c_i|^2 - 2 v_t . c_i) with v . c on tcgen05: A = a tile of
// 128 tokens (bf16, exact), B = the centroids split into two bf16 parts
// c = c_hi + c_lo (c_lo = bf16(c - c_hi); the pair keeps ~16 significant bits,
// so |v . c - v . (c_hi + c_lo)| <= 2^-17 |v||c|), accumulated in fp32 in
// TMEM; the epilogue adds |c|^2 (fp32, as centroid_norms) and takes the
// argmin with ties to the lowest index.  Used for k <= 256.
//
// Persistent CTAs, each over a contiguous range of (head, token-tile) pairs;
// a range spans few heads, and the centroids of a head are split into shared
// memory once per head.  6 warps: warp 0 TMA producer (token tiles, 2
// stages), warp 1 MMA issuer and TMEM owner (2 accumulators of 256 columns),
// warps 2-5 epilogue (one TMEM lane quadrant each).
constexpr int kAsThreads = 192;
constexpr int kAsMaxK = 256;

template <int D>
struct AsCfg {
    static constexpr int KBLK = D / 64;                 // 64-channel K blocks (128-byte swizzled rows)
    static constexpr int TILE_BYTES = KBLK * 128 * 128; // one token tile
    static constexpr int CPART = KBLK * kAsMaxK * 128;  // one centroid part
    static constexpr int OFF_C = 0;                     // [2 parts]
    static constexpr int OFF_V = OFF_C + 2 * CPART;     // [2 stages]
    static constexpr int OFF_N = OFF_V + 2 * TILE_BYTES;  // |c|^2, kAsMaxK floats
    static constexpr int OFF_BAR = OFF_N + kAsMaxK * 4;
    static constexpr int OFF_MISC = OFF_BAR + 8 * 8;
    static constexpr int SMEM = OFF_MISC + 64 + 1024;
    static_assert(SMEM <= 232448, "shared memory budget");
    // barriers: VF[2] tile loaded, VE[2] tile read, DF[2] accumulator ready, DE[2] accumulator read
    static constexpr int B_VF = 0, B_VE = 2, B_DF = 4, B_DE = 6;
};

template <int D>
__global__ void __launch_bounds__(kAsThreads, 1)
    assign_tc_kernel(const __grid_constant__ CUtensorMap tmV, vc_shape s, int k, int kpad, int tiles_per_head,
                     int total, const float* cent, int32_t* labels, int32_t* dev_status, uint64_t tmo) {
    using C = AsCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
    float* cn_s = reinterpret_cast<float*>(smem + C::OFF_N);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::B_VF + i), 1);
            mbar_init(bar(C::B_VE + i), 1);
            mbar_init(bar(C::B_DF + i), 1);
            mbar_init(bar(C::B_DE + i), 4);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);

    const int per = (total + gridDim.x - 1) / gridDim.x;
    const int g0 = blockIdx.x * per, g1 = min(total, g0 + per);
    const uint32_t idesc = idesc_bf16(128, (uint32_t)kpad);
    int n = 0;  // tiles this CTA has processed (barrier phases)
    bool ok = true;
    for (int seg = g0; seg < g1 && ok;) {
        const int bh = seg / tiles_per_head;
        const int seg_end = min(g1, (bh + 1) * tiles_per_head);
        const int b = bh / s.H, h = bh % s.H;
        // ---- centroids of head bh: two bf16 parts in the 128-byte swizzled
        // K-major layout of the B operand, and |c|^2
        const float* cb = cent + (int64_t)bh * k * D;
        for (int e = threadIdx.x; e < kpad * (D / 8); e += kAsThreads) {
            const int c = e / (D / 8), kc = e % (D / 8);  // centroid, 8-channel chunk
            float x[8];
            if (c < k) {
                const float4 x0 = *reinterpret_cast<const float4*>(cb + (int64_t)c * D + kc * 8);
                const float4 x1 = *reinterpret_cast<const float4*>(cb + (int64_t)c * D + kc * 8 + 4);
                x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
                x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) x[q] = 0.f;
            }
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const __nv_bfloat16 h0 = __float2bfloat16_rn(x[2 * q]), h1 = __float2bfloat16_rn(x[2 * q + 1]);
                const __nv_bfloat16 l0 = __float2bfloat16_rn(__fsub_rn(x[2 * q], __bfloat162float(h0)));
                const __nv_bfloat16 l1 = __float2bfloat16_rn(__fsub_rn(x[2 * q + 1], __bfloat162float(h1)));
                hi[q] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                lo[q] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
            }
            const int kb = kc / 8, chunk = kc % 8;
            const uint32_t off = kb * (kAsMaxK * 128) + (c >> 3) * 1024 + (c & 7) * 128 + ((chunk ^ (c & 7)) << 4);
            *reinterpret_cast<uint4*>(smem + C::OFF_C + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(smem + C::OFF_C + C::CPART + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        // |c|^2 for the real centroids, +inf for the padding up to kAsMaxK, so
        // that a padded column can never be the minimum
        for (int c = threadIdx.x; c < kAsMaxK; c += kAsThreads) {
            float acc = INFINITY;
            if (c < k) {
                acc = 0.f;
                for (int e = 0; e < D; ++e) acc = __fmaf_rn(cb[(int64_t)c * D + e], cb[(int64_t)c * D + e], acc);
            }
            cn_s[c] = acc;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const int ntile = seg_end - seg;
        if (warp == 0) {
            // ---- producer: token tiles of this head
            for (int i = 0; i < ntile; ++i) {
                const int m = n + i, st = m & 1;
                if (m >= 2 && !mbar_wait_warp(bar(C::B_VE + st), ((m >> 1) - 1) & 1, abort_flag, dev_status, tmo)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int t0 = (seg + i - bh * tiles_per_head) * 128;
                    mbar_arrive_expect_tx(bar(C::B_VF + st), C::TILE_BYTES);
#pragma unroll
                    for (int kb = 0; kb < C::KBLK; ++kb)
                        tma_load_4d(sbase + C::OFF_V + st * C::TILE_BYTES + kb * 16384, &tmV, kb * 64, h, t0, b,
                                    bar(C::B_VF + st));
                }
                __syncwarp();
            }
        } else if (warp == 1) {
            // ---- MMA issuer
            for (int i = 0; i < ntile; ++i) {
                const int m = n + i, st = m & 1, buf = m & 1;
                if (!mbar_wait_warp(bar(C::B_VF + st), (m >> 1) & 1, abort_flag, dev_status, tmo) ||
                    (m >= 2 && !mbar_wait_warp(bar(C::B_DE + buf), ((m >> 1) - 1) & 1, abort_flag, dev_status, tmo))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + buf * 256;
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int kb = kk / 4, kin = (kk % 4) * 32;
                        const uint64_t ad =
                            smem_desc(sbase + C::OFF_V + st * C::TILE_BYTES + kb * 16384 + kin, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(sbase + C::OFF_C + part * C::CPART + kb * (kAsMaxK * 128) + kin,
                                                      1024, kSwizzle128B);
                        mma_bf16_ss_w(d_tmem, ad, bd, idesc, (part > 0 || kk > 0) ? 1u : 0u);
                    }
                mma_commit_w(bar(C::B_DF + buf));
                mma_commit_w(bar(C::B_VE + st));
            }
        } else {
            // ---- epilogue: argmin over the centroids for one token row
            const int q = warp & 3, row = q * 32 + lane;
            const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
            for (int i = 0; i < ntile; ++i) {
                const int m = n + i, buf = m & 1;
                if (!mbar_wait_warp(bar(C::B_DF + buf), (m >> 1) & 1, abort_flag, dev_status, tmo)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // 64 columns per TMEM round trip; four independent running minima
                // (columns c = 4i + q), each keeping its first minimum, merged at
                // the end with ties to the lower column: the same argmin as one
                // pass in column order.  Columns past k (stale TMEM past kpad
                // included) meet |c|^2 = +inf and never win.
                float best[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
                int arg[4] = {0, 0, 0, 0};
                const float4* cn4 = reinterpret_cast<const float4*>(cn_s);
                for (int c0 = 0; c0 < kpad; c0 += 64) {
                    uint32_t r[64];
                    tmem_ld32(lane_addr + buf * 256 + c0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                    if (c0 + 32 < kpad) tmem_ld32(lane_addr + buf * 256 + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                    tmem_wait_ld();
                    const int nq = (c0 + 32 < kpad) ? 16 : 8;  // float4 groups of columns in this round
#pragma unroll
                    for (int g = 0; g < 16; ++g) {
                        if (g < nq) {
                            const float4 cn = cn4[(c0 >> 2) + g];
                            const float cv[4] = {cn.x, cn.y, cn.z, cn.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float dist = __fmaf_rn(-2.f, __uint_as_float(r[4 * g + q]), cv[q]);
                                if (dist < best[q]) {
                                    best[q] = dist;
                                    arg[q] = c0 + 4 * g + q;
                                }
                            }
                        }
                    }
                }
                float bestv = best[0];
                int argv = arg[0];
#pragma unroll
                for (int q = 1; q < 4; ++q)
                    if (best[q] < bestv || (best[q] == bestv && arg[q] < argv)) {
                        bestv = best[q];
                        argv = arg[q];
                    }
                const int arg_final = argv;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_DE + buf));
                const int t = (seg + i - bh * tiles_per_head) * 128 + row;
                if (t < s.N) labels[(int64_t)bh * s.N + t] = arg_final;
            }
        }
        // every role has finished this head's tiles (the epilogue waited for the
        // last accumulator, so every MMA reading the centroid parts is complete)
        n += ntile;
        seg = seg_end;
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        ok = ok && (*abort_flag == 0);
    }
    // let the producer's copies in flight land before the CTA exits
    if (warp == 0 && n > 0) {
        for (int m = (n > 2 ? n - 2 : 0); m < n; ++m) drain_wait(bar(C::B_VF + (m & 1)), (m >> 1) & 1, tmo);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------ block fill

constexpr int kFillThreads = 256;
constexpr size_t kFillSmemT = 200 * 1024;  // dynamic shared memory limit for the in-smem centroid copy

// Exclusive scan of x[0..k) in place (k <= 1024) by the whole CTA; returns the total.
__device__ int cta_exclusive_scan(int32_t* x, int k, int32_t* tmp) {
    // each warp scans a 32-entry slice; warp totals in tmp[0..32)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int total = 0;
    for (int base = 0; base < k; base += kFillThreads) {
        const int i = base + tid;
        int v = (i < k) ? x[i] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        if (lane == 31) tmp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = (lane < kFillThreads / 32) ? tmp[lane] : 0;
            int wi = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += u;
            }
            if (lane < kFillThreads / 32) tmp[lane] = wi - w;  // exclusive warp offsets
            if (lane == kFillThreads / 32 - 1) tmp[32] = wi;  // chunk total
        }
        __syncthreads();
        if (i < k) x[i] = total + tmp[warp] + incl - v;
        total += tmp[32];
        __syncthreads();
    }
    return total;
}

// One CTA per head.  count: cluster sizes of the last assignment.
// fdst[c] = start of cluster c's whole blocks; ldst[c] = start of its leftovers.
// The head's centroids are read transposed (T[e * k + c] = C[c][e], so a warp
// reads channel e of 32 clusters at once) from shared memory when they fit
// (SMEM_T), else from a transposed copy in global memory.
template <int D, bool SMEM_T>
__global__ void __launch_bounds__(kFillThreads) fill_chain_kernel(const int32_t* count, const float* cent, int k,
                                                                  float* cT, int32_t* fdst, int32_t* ldst) {
    extern __shared__ __align__(16) uint8_t fsm_raw[];
    __shared__ int32_t tmp[33];
    __shared__ float lastc[D];
    __shared__ float wmin[kFillThreads / 32];
    __shared__ int32_t warg[kFillThreads / 32];
    __shared__ int32_t cur_s;
    int32_t* f = reinterpret_cast<int32_t*>(fsm_raw);     // [k] whole-block sizes, then starts
    int32_t* lft = f + k;                                  // [k] leftover sizes (0: not in the chain)
    int32_t* order = f + 2 * k;                            // [k] chain: position -> cluster
    int32_t* lsz = f + 3 * k;                              // [k] leftover sizes in chain order
    uint8_t* used = reinterpret_cast<uint8_t*>(f + 4 * k);  // [k]
    const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t* n = count + (int64_t)bh * k;
    const float* C = cent + (int64_t)bh * k * D;
    float* T;
    if constexpr (SMEM_T)
        T = reinterpret_cast<float*>(fsm_raw + (((size_t)4 * k * 4 + k + 15) & ~size_t(15)));
    else
        T = cT + (int64_t)bh * D * k;
    for (int i = tid; i < k * D; i += kFillThreads) T[(i % D) * k + i / D] = C[i];
    for (int c = tid; c < k; c += kFillThreads) {
        const int nc = n[c];
        f[c] = nc - nc % kBlock;
        lft[c] = nc % kBlock;
        used[c] = (nc % kBlock) == 0;  // clusters without leftovers never join the chain
    }
    __syncthreads();
    const int base = cta_exclusive_scan(f, k, tmp);  // f[] now holds the whole-block starts
    for (int c = tid; c < k; c += kFillThreads) fdst[(int64_t)bh * k + c] = f[c];
    // chain start: the lowest label with leftovers
    if (tid < 32) {
        int c0 = 0x7fffffff;
        for (int c = lane; c < k; c += 32)
            if (!used[c]) {
                c0 = c;
                break;
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c0 = min(c0, __shfl_xor_sync(0xffffffffu, c0, o));
        if (lane == 0) cur_s = (c0 == 0x7fffffff) ? -1 : c0;
    }
    __syncthreads();
    int nch = 0;
    while (true) {
        const int cur = cur_s;
        if (cur < 0) break;
        if (tid == 0) {
            order[nch] = cur;
            lsz[nch] = lft[cur];
            used[cur] = 1;
        }
        for (int e = tid; e < D; e += kFillThreads) lastc[e] = T[e * k + cur];
        ++nch;
        __syncthreads();
        // nearest unvisited cluster with leftovers: fp32, channels in order, no contraction
        float best = INFINITY;
        int arg = 0x7fffffff;
        for (int c = tid; c < k; c += kFillThreads) {
            if (used[c]) continue;
            float sum = 0.f;
#pragma unroll 16
            for (int e = 0; e < D; ++e) {
                const float df = __fsub_rn(T[e * k + c], lastc[e]);
                sum = __fadd_rn(sum, __fmul_rn(df, df));
            }
            if (sum < best) {  // candidates visited in increasing label order: ties keep the lower
                best = sum;
                arg = c;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oa = __shfl_xor_sync(0xffffffffu, arg, o);
            if (ob < best || (ob == best && oa < arg)) {
                best = ob;
                arg = oa;
            }
        }
        if (lane == 0) {
            wmin[warp] = best;
            warg[warp] = arg;
        }
        __syncthreads();
        if (warp == 0) {
            float b = (lane < kFillThreads / 32) ? wmin[lane] : INFINITY;
            int a = (lane < kFillThreads / 32) ? warg[lane] : 0x7fffffff;
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) {
                const float ob = __shfl_xor_sync(0xffffffffu, b, o);
                const int oa = __shfl_xor_sync(0xffffffffu, a, o);
                if (ob < b || (ob == b && oa < a)) {
                    b = ob;
                    a = oa;
                }
            }
            if (lane == 0) cur_s = (a == 0x7fffffff) ? -1 : a;
        }
        __syncthreads();
    }
    // leftover starts in chain order, after all whole blocks
    cta_exclusive_scan(lsz, nch, tmp);
    for (int i = tid; i < nch; i += kFillThreads) ldst[(int64_t)bh * k + order[i]] = base + lsz[i];
}

// Entry i of the stable argsort (cluster c, rank r = i - start[c]) goes to
// fdst[c] + r if r < f_c, else to ldst[c] + r - f_c.
__global__ void fill_scatter_kernel(const int32_t* pi_sort, const int32_t* labels, const int32_t* count,
                                    const int32_t* start, const int32_t* fdst, const int32_t* ldst, int N, int k,
                                    int32_t* perm) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N) return;
    const int64_t off = (int64_t)bh * N;
    const int t = pi_sort[off + i];
    const int c = labels[off + t];
    const int64_t ko = (int64_t)bh * k + c;
    const int r = i - start[ko];
    const int f = count[ko] - count[ko] % kBlock;
    perm[off + (r < f ? fdst[ko] + r : ldst[ko] + (r - f))] = t;
}

}  // namespace

size_t cluster_workspace(const vc_shape& s, int k) {
    const size_t BH = (size_t)s.B * s.H;
    const size_t nseg = (s.N + kSeg - 1) / kSeg;
    return align256(BH * k * 4) + align256(BH * nseg * k * 4) + 4 * align256(BH * k * 4) +
           align256(BH * (size_t)s.N * 4) + align256(BH * (size_t)s.d * k * 4);
}

// Tensor map over V [B, N, H, d] (bf16) for the assignment kernel: boxes of
// 64 channels x 1 head x 128 tokens, 128-byte swizzled.
static bool make_v_map(CUtensorMap* map, const uint16_t* V, const vc_shape& s) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)s.d, (cuuint64_t)s.H, (cuuint64_t)s.N, (cuuint64_t)s.B};
    const cuuint64_t strides[3] = {(cuuint64_t)s.s_h * 2, (cuuint64_t)s.s_n * 2, (cuuint64_t)s.s_b * 2};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(V), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static vc_status launch_cluster_d(const uint16_t* V, const vc_shape& s, int k, int iters, int warm, int fill,
                                  float* cent, int32_t* labels, int32_t* perm, void* ws, int32_t* dev_status,
                                  cudaStream_t st) {
    const int BH = s.B * s.H;
    const int nseg = (s.N + kSeg - 1) / kSeg;
    ClusterWs w = carve(ws, s, k);
    if (!warm) init_centroids<<<dim3(k, BH), 128, 0, st>>>(V, s, k, cent);
    const size_t assign_smem = (size_t)D * (kTokTile + 4) * 4 + (size_t)D * (kCenTile + 4) * 4;
    const bool tc = k <= kAsMaxK;
    {
        vc_status a = tc ? ensure_smem_attr(reinterpret_cast<const void*>(assign_tc_kernel<D>), AsCfg<D>::SMEM)
                         : ensure_smem_attr(reinterpret_cast<const void*>(assign_kernel<D>), (int)assign_smem);
        if (a != VC_OK) return a;
    }
    CUtensorMap vmap;
    int grid_tc = 0;
    const int tiles_per_head = (s.N + 127) / 128;
    if (tc) {
        if (!make_v_map(&vmap, V, s)) return VC_ERR_CUDA;
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        grid_tc = (int)std::min<int64_t>((int64_t)BH * tiles_per_head, sms > 0 ? sms : 1);
    }
    const int kpad = (k + 15) & ~15;
    for (int it = 0; it < iters; ++it) {
        if (tc) {
            assign_tc_kernel<D><<<grid_tc, kAsThreads, AsCfg<D>::SMEM, st>>>(
                vmap, s, k, kpad, tiles_per_head, BH * tiles_per_head, cent, labels, dev_status, 4000000000ull);
        } else {
            centroid_norms<<<dim3((unsigned)((k + 127) / 128), BH), 128, 0, st>>>(cent, k, D, w.cnorm);
            assign_kernel<D><<<dim3((s.N + kTokTile - 1) / kTokTile, BH), kAssignThreads, assign_smem, st>>>(
                V, s, k, cent, w.cnorm, labels);
        }
        seg_hist<<<dim3(nseg, BH), 256, k * 4, st>>>(labels, s.N, k, nseg, w.seg);
        seg_scan<<<BH, 256, 0, st>>>(k, nseg, w.seg, w.count, w.start);
        int32_t* pi = fill ? w.pi_sort : perm;
        seg_scatter<<<dim3(nseg, BH), 32, k * 4, st>>>(labels, s.N, k, nseg, w.seg, pi);
        update_kernel<D><<<dim3(k, BH), kUpdThreads, 0, st>>>(V, s, k, pi, w.count, w.start, cent);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (fill) {
        const size_t fbase = ((size_t)4 * k * sizeof(int32_t) + k + 15) & ~size_t(15);
        const size_t tbytes = (size_t)k * D * sizeof(float);
        if (fbase + tbytes <= kFillSmemT) {
            vc_status a = ensure_smem_attr(reinterpret_cast<const void*>(fill_chain_kernel<D, true>), (int)kFillSmemT);
            if (a != VC_OK) return a;
            fill_chain_kernel<D, true><<<BH, kFillThreads, fbase + tbytes, st>>>(w.count, cent, k, w.cT, w.fdst,
                                                                                 w.ldst);
        } else {
            fill_chain_kernel<D, false><<<BH, kFillThreads, fbase, st>>>(w.count, cent, k, w.cT, w.fdst, w.ldst);
        }
        fill_scatter_kernel<<<dim3((s.N + 255) / 256, BH), 256, 0, st>>>(w.pi_sort, labels, w.count, w.start, w.fdst,
                                                                       w.ldst, s.N, k, perm);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_status(e);
    }
    return VC_OK;
}

vc_status launch_cluster(const uint16_t* V, const vc_shape& s, int k, int iters, int warm, int fill, float* cent,
                         int32_t* labels, int32_t* perm, void* ws, int32_t* dev_status, cudaStream_t st) {
    if (s.d == 128)
        return launch_cluster_d<128>(V, s, k, iters, warm, fill, cent, labels, perm, ws, dev_status, st);
    return launch_cluster_d<64>(V, s, k, iters, warm, fill, cent, labels, perm, ws, dev_status, st);
}

}  // namespace vc
