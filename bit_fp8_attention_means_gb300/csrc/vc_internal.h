// vc_internal.h -- host-side declarations shared by the library's translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "vc.h"
#include "vc_ctx_cache.h"

namespace vc {

constexpr int kBlock = 128;  // tokens per block (B_v) and per attention tile

inline int nblk_of(int N) { return (N + kBlock - 1) / kBlock; }
inline int64_t npad_of(int N) { return (int64_t)nblk_of(N) * kBlock; }

vc_status check_shape(const vc_shape& s);
vc_status cuda_status(cudaError_t e);

// The CUDA context current on this host thread and its device (CtxKey, in
// vc_ctx_cache.h): the key of every per-context cache below.
vc_status current_ctx(CtxKey* out);

// Raises the dynamic shared-memory limit of kernel `kern` to `bytes` once per
// context (cudaFuncSetAttribute acts on the current context only).  Thread
// safe: host threads may launch on one or several devices concurrently.
vc_status ensure_smem_attr(const void* kern, int bytes);

// Argument checks shared by the quantizer entry points (vc_quantize,
// vc_quantize_ex, vc_quantize_staged, vc_quantize_static).
vc_status quantize_args(const void* Q, const void* K, const void* V, const vc_shape& shape, int vsmooth,
                        const float* rope, int hadamard, const uint8_t* Q8, const float* sq, const uint8_t* K8,
                        const float* sk, const uint8_t* V8T, const float* sv, const void* mu);

// cuTensorMapEncodeTiled, looked up through the runtime so that the library
// does not link against the driver library directly; null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn();

// quantizer (vc_quantize.cu)
struct Preproc {
    const float* rope = nullptr;  // [N, d/2, 2] (cos, sin), or null: no rotary transform
    int hadamard = 0;             // 1: Walsh-Hadamard transform of Q and K rows, 1/d on the Q scale
    int v4 = 0;                   // 1: the V residual in the 4-bit form (E2M1, power-of-two scale per 32 tokens)
};
size_t quantize_workspace(const vc_shape& s);
size_t quantize_staged_workspace(const vc_shape& s);
vc_status launch_quantize(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const vc_shape& s,
                          const int32_t* perm, int vsmooth, const Preproc& pp, uint8_t* Q8, float* sq, uint8_t* K8,
                          float* sk, uint8_t* V8T, float* sv, uint16_t* mu, void* ws, cudaStream_t st);
vc_status launch_quantize_staged(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const vc_shape& s,
                                 const int32_t* perm, int vsmooth, const Preproc& pp, uint8_t* Q8, float* sq,
                                 uint8_t* K8, float* sk, uint8_t* V8T, float* sv, uint16_t* mu, void* ws,
                                 cudaStream_t st);

// grouping (vc_cluster.cu)
size_t cluster_workspace(const vc_shape& s, int k);
vc_status launch_cluster(const uint16_t* V, const vc_shape& s, int k, int iters, int warm, int fill, float* cent,
                         int32_t* labels, int32_t* perm, void* ws, int32_t* dev_status, cudaStream_t st);

// attention (vc_attn.cu)
struct AttnDebug {
    int bh = -1, qtile = -1;       // the query tile whose scores and bytes are dumped (with S, P)
    float* S = nullptr;
    uint8_t* P = nullptr;
    int skip_k_tile = -1;          // >= 0: the K loader never loads nor signals this key tile
    uint64_t timeout_ns = 0;       // bound of every device wait (0: the default, 4 s)
};
vc_status launch_attn(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk, const uint8_t* V8T,
                      const float* sv, const uint16_t* mu, const vc_shape& s, float softmax_scale, int expcast,
                      float exact_margin, int vsmooth, uint16_t* O, int32_t* dev_status, cudaStream_t st,
                      const AttnDebug* dbg);

}  // namespace vc
