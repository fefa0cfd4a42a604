// vc_api.cu -- the extern "C" entry points declared in include/vc.h.
// Argument checks happen here, on the host, before anything is enqueued.
#include <cstdint>
#include <mutex>
#include <vector>

#include "vc.h"
#include "vc_internal.h"

namespace vc {

vc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? VC_OK : VC_ERR_CUDA; }

vc_status check_shape(const vc_shape& s) {
    if (s.B < 1 || s.H < 1 || s.N < 1 || s.d < 1) return VC_ERR_INVALID_ARG;
    if (s.d != 64 && s.d != 128) return VC_ERR_UNSUPPORTED;
    if (s.N > (1 << 24)) return VC_ERR_UNSUPPORTED;
    if (s.s_b <= 0 || s.s_n <= 0 || s.s_h <= 0) return VC_ERR_INVALID_ARG;
    if ((s.s_b % 8) || (s.s_n % 8) || (s.s_h % 8)) return VC_ERR_INVALID_ARG;
    // TMA row coordinates are 32-bit
    if ((int64_t)s.B * s.H * npad_of(s.N) >= (int64_t(1) << 31)) return VC_ERR_UNSUPPORTED;
    return VC_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetCurrentFn>(ptr);
        return static_cast<CtxGetCurrentFn>(nullptr);
    }();
    return fn;
}

CtxAttrCache g_smem_attr;
}  // namespace

vc_status current_ctx(CtxKey* out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return VC_ERR_CUDA;
    CUcontext ctx = nullptr;
    CtxGetCurrentFn fn = ctx_get_current_fn();
    if (fn && fn(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    out->device = dev;
    out->ctx = ctx;
    return VC_OK;
}

vc_status ensure_smem_attr(const void* kern, int bytes) {
    CtxKey key;
    vc_status st = current_ctx(&key);
    if (st != VC_OK) return st;
    return g_smem_attr.ensure(key, kern, bytes, [&](CtxKey* k) -> vc_status {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return cuda_status(e);
        // a context created by this call's own runtime initialisation is known only now
        if (!k->ctx) current_ctx(k);
        return VC_OK;
    });
}

vc_status quantize_args(const void* Q, const void* K, const void* V, const vc_shape& shape, int vsmooth,
                        const float* rope, int hadamard, const uint8_t* Q8, const float* sq, const uint8_t* K8,
                        const float* sk, const uint8_t* V8T, const float* sv, const void* mu) {
    vc_status st = check_shape(shape);
    if (st != VC_OK) return st;
    if ((vsmooth != 0 && vsmooth != 1) || (hadamard != 0 && hadamard != 1)) return VC_ERR_INVALID_ARG;
    if (!Q || !K || !V || !Q8 || !sq || !K8 || !sk || !V8T || !sv || (vsmooth && !mu)) return VC_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(Q8) || !aligned16(K8) || !aligned16(V8T) ||
        !aligned16(rope))
        return VC_ERR_INVALID_ARG;
    return VC_OK;
}

}  // namespace vc

using namespace vc;

extern "C" {

const char* vc_status_string(vc_status s) {
    switch (s) {
        case VC_OK: return "VC_OK";
        case VC_ERR_INVALID_ARG: return "VC_ERR_INVALID_ARG";
        case VC_ERR_UNSUPPORTED: return "VC_ERR_UNSUPPORTED";
        case VC_ERR_WORKSPACE: return "VC_ERR_WORKSPACE";
        case VC_ERR_CUDA: return "VC_ERR_CUDA";
        case VC_ERR_TIMEOUT: return "VC_ERR_TIMEOUT";
    }
    return "VC_ERR_UNKNOWN";
}

int vc_version(void) { return 101; }

size_t vc_cluster_workspace(vc_shape shape, int k) {
    if (check_shape(shape) != VC_OK || k < 1) return 0;
    return cluster_workspace(shape, k);
}

vc_status vc_cluster(const void* V, vc_shape shape, int k, int iters, int warm_start, float* centroids,
                     int32_t* labels, int32_t* perm, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                     vc_stream_t stream) {
    return vc_cluster_ex(V, shape, k, iters, warm_start, 0, centroids, labels, perm, workspace, workspace_bytes,
                         dev_status, stream);
}

vc_status vc_cluster_ex(const void* V, vc_shape shape, int k, int iters, int warm_start, int block_fill,
                        float* centroids, int32_t* labels, int32_t* perm, void* workspace, size_t workspace_bytes,
                        int32_t* dev_status, vc_stream_t stream) {
    vc_status st = check_shape(shape);
    if (st != VC_OK) return st;
    if (!V || !centroids || !labels || !perm) return VC_ERR_INVALID_ARG;
    if (!aligned16(V) || !aligned16(centroids)) return VC_ERR_INVALID_ARG;
    if (iters < 1 || (warm_start != 0 && warm_start != 1) || (block_fill != 0 && block_fill != 1))
        return VC_ERR_INVALID_ARG;
    if (k < 1 || k > 1024) return VC_ERR_UNSUPPORTED;
    if (k > shape.N) return VC_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < cluster_workspace(shape, k) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return VC_ERR_WORKSPACE;
    return launch_cluster(static_cast<const uint16_t*>(V), shape, k, iters, warm_start, block_fill, centroids, labels,
                          perm, workspace, dev_status, reinterpret_cast<cudaStream_t>(stream));
}

size_t vc_quantize_workspace(vc_shape shape) {
    if (check_shape(shape) != VC_OK) return 0;
    return quantize_workspace(shape);
}

static bool workspace_ok(const void* ws, size_t bytes, size_t need) {
    return ws && bytes >= need && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0;
}

vc_status vc_quantize(const void* Q, const void* K, const void* V, vc_shape shape, const int32_t* perm, int vsmooth,
                      uint8_t* Q8, float* sq, uint8_t* K8, float* sk, uint8_t* V8T, float* sv, void* mu,
                      void* workspace, size_t workspace_bytes, vc_stream_t stream) {
    return vc_quantize_ex(Q, K, V, shape, perm, vsmooth, nullptr, 0, Q8, sq, K8, sk, V8T, sv, mu, workspace,
                          workspace_bytes, stream);
}

vc_status vc_quantize_ex(const void* Q, const void* K, const void* V, vc_shape shape, const int32_t* perm,
                         int vsmooth, const float* rope, int hadamard, uint8_t* Q8, float* sq, uint8_t* K8,
                         float* sk, uint8_t* V8T, float* sv, void* mu, void* workspace, size_t workspace_bytes,
                         vc_stream_t stream) {
    vc_status st = quantize_args(Q, K, V, shape, vsmooth, rope, hadamard, Q8, sq, K8, sk, V8T, sv, mu);
    if (st != VC_OK) return st;
    if (!workspace_ok(workspace, workspace_bytes, quantize_workspace(shape))) return VC_ERR_WORKSPACE;
    Preproc pp;
    pp.rope = rope;
    pp.hadamard = hadamard;
    return launch_quantize(static_cast<const uint16_t*>(Q), static_cast<const uint16_t*>(K),
                           static_cast<const uint16_t*>(V), shape, perm, vsmooth, pp, Q8, sq, K8, sk, V8T, sv,
                           static_cast<uint16_t*>(mu), workspace, reinterpret_cast<cudaStream_t>(stream));
}

vc_status vc_quantize_v4(const void* Q, const void* K, const void* V, vc_shape shape, const int32_t* perm,
                         int vsmooth, uint8_t* Q8, float* sq, uint8_t* K8, float* sk, uint8_t* V8T, float* sv,
                         void* mu, void* workspace, size_t workspace_bytes, vc_stream_t stream) {
    vc_status st = quantize_args(Q, K, V, shape, vsmooth, nullptr, 0, Q8, sq, K8, sk, V8T, sv, mu);
    if (st != VC_OK) return st;
    if (!workspace_ok(workspace, workspace_bytes, quantize_workspace(shape))) return VC_ERR_WORKSPACE;
    Preproc pp;
    pp.v4 = 1;
    return launch_quantize(static_cast<const uint16_t*>(Q), static_cast<const uint16_t*>(K),
                           static_cast<const uint16_t*>(V), shape, perm, vsmooth, pp, Q8, sq, K8, sk, V8T, sv,
                           static_cast<uint16_t*>(mu), workspace, reinterpret_cast<cudaStream_t>(stream));
}

size_t vc_quantize_staged_workspace(vc_shape shape) {
    if (check_shape(shape) != VC_OK) return 0;
    return quantize_staged_workspace(shape);
}

vc_status vc_quantize_staged(const void* Q, const void* K, const void* V, vc_shape shape, const int32_t* perm,
                             int vsmooth, const float* rope, int hadamard, uint8_t* Q8, float* sq, uint8_t* K8,
                             float* sk, uint8_t* V8T, float* sv, void* mu, void* workspace, size_t workspace_bytes,
                             vc_stream_t stream) {
    vc_status st = quantize_args(Q, K, V, shape, vsmooth, rope, hadamard, Q8, sq, K8, sk, V8T, sv, mu);
    if (st != VC_OK) return st;
    if (!workspace_ok(workspace, workspace_bytes, quantize_staged_workspace(shape))) return VC_ERR_WORKSPACE;
    Preproc pp;
    pp.rope = rope;
    pp.hadamard = hadamard;
    return launch_quantize_staged(static_cast<const uint16_t*>(Q), static_cast<const uint16_t*>(K),
                                  static_cast<const uint16_t*>(V), shape, perm, vsmooth, pp, Q8, sq, K8, sk, V8T,
                                  sv, static_cast<uint16_t*>(mu), workspace, reinterpret_cast<cudaStream_t>(stream));
}

static vc_status attn_common(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk,
                             const uint8_t* V8T, const float* sv, const void* mu, const vc_shape& shape,
                             int expcast, int vsmooth, void* O) {
    vc_status st = check_shape(shape);
    if (st != VC_OK) return st;
    if ((expcast < 0 || expcast > 3) || (vsmooth != 0 && vsmooth != 1)) return VC_ERR_INVALID_ARG;
    if (!Q8 || !sq || !K8 || !sk || !V8T || !sv || !O || (vsmooth && !mu)) return VC_ERR_INVALID_ARG;
    if (!aligned16(Q8) || !aligned16(K8) || !aligned16(V8T) || !aligned16(O)) return VC_ERR_INVALID_ARG;
    return VC_OK;
}

vc_status vc_attn_fwd(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk, const uint8_t* V8T,
                      const float* sv, const void* mu, vc_shape shape, float softmax_scale, int expcast, int vsmooth,
                      void* O, int32_t* dev_status, vc_stream_t stream) {
    if (expcast == 2) return VC_ERR_INVALID_ARG;  // the hybrid has its own entry point
    vc_status st = attn_common(Q8, sq, K8, sk, V8T, sv, mu, shape, expcast, vsmooth, O);
    if (st != VC_OK) return st;
    return launch_attn(Q8, sq, K8, sk, V8T, sv, static_cast<const uint16_t*>(mu), shape, softmax_scale, expcast, 0.f,
                       vsmooth, static_cast<uint16_t*>(O), dev_status, reinterpret_cast<cudaStream_t>(stream),
                       nullptr);
}

vc_status vc_attn_fwd_hybrid(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk,
                             const uint8_t* V8T, const float* sv, const void* mu, vc_shape shape,
                             float softmax_scale, float exact_margin, int vsmooth, void* O, int32_t* dev_status,
                             vc_stream_t stream) {
    if (exact_margin != exact_margin) return VC_ERR_INVALID_ARG;  // NaN
    vc_status st = attn_common(Q8, sq, K8, sk, V8T, sv, mu, shape, 2, vsmooth, O);
    if (st != VC_OK) return st;
    return launch_attn(Q8, sq, K8, sk, V8T, sv, static_cast<const uint16_t*>(mu), shape, softmax_scale, 2,
                       exact_margin, vsmooth, static_cast<uint16_t*>(O), dev_status,
                       reinterpret_cast<cudaStream_t>(stream), nullptr);
}

vc_status vc_attn_fwd_debug(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk,
                            const uint8_t* V8T, const float* sv, const void* mu, vc_shape shape, float softmax_scale,
                            int expcast, int vsmooth, void* O, int32_t* dev_status, vc_stream_t stream, int dbg_bh,
                            int dbg_qtile, float* S_dump, uint8_t* P_dump, float exact_margin) {
    if (exact_margin != exact_margin) return VC_ERR_INVALID_ARG;
    vc_status st = attn_common(Q8, sq, K8, sk, V8T, sv, mu, shape, expcast, vsmooth, O);
    if (st != VC_OK) return st;
    if (!S_dump || !P_dump || dbg_bh < 0 || dbg_bh >= shape.B * shape.H || dbg_qtile < 0 ||
        dbg_qtile >= nblk_of(shape.N))
        return VC_ERR_INVALID_ARG;
    AttnDebug dbg;
    dbg.bh = dbg_bh;
    dbg.qtile = dbg_qtile;
    dbg.S = S_dump;
    dbg.P = P_dump;
    return launch_attn(Q8, sq, K8, sk, V8T, sv, static_cast<const uint16_t*>(mu), shape, softmax_scale, expcast,
                       exact_margin, vsmooth, static_cast<uint16_t*>(O), dev_status,
                       reinterpret_cast<cudaStream_t>(stream), &dbg);
}

vc_status vc_debug_attn_timeout(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk,
                                const uint8_t* V8T, const float* sv, const void* mu, vc_shape shape, int vsmooth,
                                void* O, int32_t* dev_status, vc_stream_t stream, int skip_k_tile,
                                uint32_t timeout_us) {
    vc_status st = attn_common(Q8, sq, K8, sk, V8T, sv, mu, shape, 1, vsmooth, O);
    if (st != VC_OK) return st;
    if (!dev_status || skip_k_tile < 0 || skip_k_tile >= nblk_of(shape.N) || timeout_us == 0 ||
        timeout_us > 10000000u)
        return VC_ERR_INVALID_ARG;
    AttnDebug dbg;
    dbg.skip_k_tile = skip_k_tile;
    dbg.timeout_ns = (uint64_t)timeout_us * 1000ull;
    return launch_attn(Q8, sq, K8, sk, V8T, sv, static_cast<const uint16_t*>(mu), shape, 0.f, 1, 0.f, vsmooth,
                       static_cast<uint16_t*>(O), dev_status, reinterpret_cast<cudaStream_t>(stream), &dbg);
}

}  // extern "C"
