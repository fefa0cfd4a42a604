/*
 * vc.h -- C ABI of the VC-Attention hot path for one GB300 (sm_103a).
 *
 * Non-causal attention O = softmax(Q K^T * scale) V computed in FP8 with the
 * two techniques of "VC-Attention: Value Smoothing and Softmax Casting for
 * Low-bit Attention":
 *   V-Smooth  -- value tokens of each (batch, head) are grouped by online
 *                k-means, K and V are gathered jointly into cluster order
 *                (exact for non-causal attention, P'V' = PV), every 128-token
 *                block mean mu_j is kept in 16 bits and only the residual is
 *                quantized to E4M3 with per-channel scales; the mean is added
 *                back inside the online softmax from the row sums r_ij.
 *   ExpCast   -- each E4M3 probability byte is written from the log-domain
 *                score by one FMA: c = clip(Round(8(u+8) + 56 + beta), 0, 120),
 *                beta = -0.35, replacing the FP32 exp and the cast.
 * Passages: paper summary on paper.rainbus.top (方法步骤详情, steps 1-4;
 * 前置知识 "在线 softmax", "E4M3 浮点格式"); study note on
 * dimensionstp.github.io (sections 2-1 .. 2-4); wire.sakhanda.co article
 * (sections "V-Smooth", "ExpCast-FP8").
 *
 * Conventions shared by every entry point
 *   - Every pointer is device memory owned by the caller unless stated.  The
 *     library never allocates or frees memory and keeps no per-call state;
 *     calls on different streams with disjoint buffers may run concurrently,
 *     from one or several host threads and on one or several devices (the
 *     one-time launch set-up is done per CUDA context, under a lock).
 *   - All work is enqueued asynchronously on `stream` (NULL = legacy default
 *     stream).  A return of VC_OK means the launches were enqueued.
 *   - Argument and shape errors are detected on the host before anything is
 *     launched and return VC_ERR_INVALID_ARG / VC_ERR_UNSUPPORTED /
 *     VC_ERR_WORKSPACE.  A failed launch returns VC_ERR_CUDA.
 *   - Every wait inside a kernel is bounded.  A wait that runs out writes
 *     VC_ERR_TIMEOUT to *dev_status (an int32 in device memory, nullable;
 *     the caller zeroes it beforehand and reads it after synchronising); the
 *     kernel then releases what it holds and returns instead of hanging.
 *   - Token blocks are 128 tokens; nblk = ceil(N/128), Npad = 128*nblk.
 *   - NaN or Inf inputs are outside the contract.
 */
#ifndef VC_H_
#define VC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-identical to cudaStream_t; declared here so this header needs no CUDA headers. */
typedef struct CUstream_st* vc_stream_t;

typedef enum {
    VC_OK = 0,
    VC_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad stride, bad flag */
    VC_ERR_UNSUPPORTED = 2, /* d not in {64, 128}, k outside [1, 1024], N > 2^24 */
    VC_ERR_WORKSPACE = 3,   /* workspace pointer null or smaller than the query says */
    VC_ERR_CUDA = 4,        /* a CUDA launch or driver call failed */
    VC_ERR_TIMEOUT = 5      /* a bounded device wait ran out (written to *dev_status) */
} vc_status;

/*
 * Shape and strides of a bf16 tensor laid out [B, N, H, d] (channel stride 1).
 * Strides are in elements; the usual contiguous layout has
 * s_b = N*H*d, s_n = H*d, s_h = d.  Every stride must be a multiple of 8
 * (16-byte rows) and every bf16 base pointer 16-byte aligned.
 */
typedef struct {
    int32_t B, H, N, d;
    int64_t s_b, s_n, s_h;
} vc_shape;

/* Human-readable name of a status code (static storage, never NULL). */
const char* vc_status_string(vc_status s);

/* Library ABI version (major*100 + minor). */
int vc_version(void);

/*
 * Grouping step, paper summary 方法步骤详情 step 1 (online k-means on the value
 * tokens of each batch/head, pi = argsort(z)); dimensionstp.github.io 2-1.
 *
 *   V          bf16 [B,N,H,d] with `shape` strides (read only).
 *   k          number of centroids, 1 <= k <= 1024, k <= N.
 *   iters      Lloyd iterations, >= 1.  Each iteration assigns every token to
 *              its nearest centroid (squared Euclidean distance) and moves each
 *              centroid to the mean of its members; an empty cluster keeps its
 *              centroid.
 *   warm_start 1: start from `centroids` as given (previous step's state);
 *              0: centroid i starts at token floor(i*N/k).
 *   centroids  fp32 [B,H,k,d], in/out (the warm-start state the caller keeps),
 *              16-byte aligned.
 *   labels     int32 [B,H,N], out: label of every token from the last
 *              assignment (the centroids are the means of these groups).
 *   perm       int32 [B,H,N], out: pi, the stable argsort of labels (ascending
 *              label, equal labels in token order).  Row t of K' and V' is
 *              token perm[t].
 *   workspace  device scratch of at least vc_cluster_workspace(shape, k) bytes,
 *              256-byte aligned; contents on entry are ignored.
 *   dev_status nullable device int32; a device-side wait that gives up writes
 *              VC_ERR_TIMEOUT there.
 * The distances are |c|^2 - 2 v.c.  For k <= 256 the products v.c run on the
 * tensor cores with each centroid split into two bf16 parts (about 16
 * significant bits, |error| <= 2^-17 |v||c|) and fp32 accumulation; for
 * larger k they are fp32 on the CUDA cores.  Label choice between
 * near-equidistant centroids therefore follows that rounding and is not
 * guaranteed to be bit-reproducible across hardware.
 * Errors: VC_ERR_INVALID_ARG (null or misaligned pointers, iters < 1, k > N),
 * VC_ERR_UNSUPPORTED (k outside 1..1024, d not 64 or 128), VC_ERR_WORKSPACE,
 * VC_ERR_CUDA (launch failure).
 */
size_t vc_cluster_workspace(vc_shape shape, int k);
vc_status vc_cluster(const void* V, vc_shape shape, int k, int iters, int warm_start,
                     float* centroids, int32_t* labels, int32_t* perm,
                     void* workspace, size_t workspace_bytes,
                     int32_t* dev_status, vc_stream_t stream);

/*
 * vc_cluster with an optional block-fill permutation.  The paper summary's own
 * analysis (独立分析的弱点, weakness one) observes that balanced k-means lowers
 * the V error but costs 2.8x the grouping time, and proposes cheap balancing
 * of the block fill instead (greedy backfill, or exchanges at block
 * boundaries).  With block_fill = 1, perm is instead:
 *   1. every cluster's whole 128-token blocks -- its first n_c - (n_c mod 128)
 *      members in token order -- with the clusters in label order;
 *   2. then the clusters' leftovers (their last n_c mod 128 members, token
 *      order), the clusters ordered by a greedy chain: start at the lowest
 *      label that has leftovers, then repeatedly the unvisited cluster with
 *      leftovers whose centroid is nearest to the last one (squared distance
 *      over the channels in order, each difference, square and sum rounded
 *      to fp32; ties to the lower label), using the returned centroids.
 * Any order of K and V leaves attention exact (P'V' = PV); this one puts
 * similar tokens into the partial blocks, so their means remove more.  With
 * every cluster size a multiple of 128 it equals the stable argsort.
 * block_fill = 0 is vc_cluster.  Same workspace query and errors as
 * vc_cluster, plus VC_ERR_INVALID_ARG for block_fill not in {0, 1}.
 */
vc_status vc_cluster_ex(const void* V, vc_shape shape, int k, int iters, int warm_start, int block_fill,
                        float* centroids, int32_t* labels, int32_t* perm,
                        void* workspace, size_t workspace_bytes,
                        int32_t* dev_status, vc_stream_t stream);

/*
 * Fused quantizer, paper summary 方法步骤详情 step 2 and 前置知识 "低比特量化与
 * 离群值"; dimensionstp.github.io 2-2 (mu_j = (1/B_v) V'_j^T 1, R_j = V'_j - 1 mu_j^T).
 *
 *   Q, K, V    bf16 [B,N,H,d] with `shape` strides (read only).
 *   perm       int32 [B,H,N] or NULL (identity).  K' = K[perm], V' = V[perm]
 *              (the joint gather); Q keeps its order.  Each (b,h) row must be
 *              a permutation of 0..N-1 (vc_cluster's output is); the entries
 *              are not checked, and a value outside 0..N-1 is out of contract.
 *   vsmooth    1: subtract each 128-token block mean of V' (kept as bf16 in
 *              `mu`) and quantize the residual; 0: quantize V' directly
 *              (`mu` may be NULL and is not written).
 *   Q8, K8     E4M3 [B,H,Npad,d]: code = E4M3_RNE_sat(x * (448/amax)), one
 *              scale per 128-token block; rows >= N are written as 0.
 *   sq, sk     fp32 [B,H,nblk]: amax/448 of each block (0 for an all-zero block).
 *   V8T        E4M3 [B,H,d,Npad] (token-contiguous per channel): residual
 *              codes with one scale per channel over the whole sequence;
 *              tokens >= N are 0.
 *   sv         fp32 [B,H,d]: per-channel scale amax_t|R[t,c]|/448.
 *   mu         bf16 [B,H,nblk,d]: bf16_RNE(fp32 sum in token order / count).
 *   workspace  >= vc_quantize_workspace(shape) bytes, 256-byte aligned.
 * Output pointers must be 16-byte aligned.  Codes and scales are
 * deterministic and bit-reproducible.
 * Errors, all returned before any launch: VC_ERR_INVALID_ARG (a null pointer
 * -- mu may be NULL only with vsmooth = 0 --, a misaligned Q, K, V, Q8, K8 or
 * V8T, vsmooth not in {0,1}, a non-positive size, or a stride that is not a
 * positive multiple of 8), VC_ERR_UNSUPPORTED (d not 64 or 128, N > 2^24, or
 * B*H*Npad >= 2^31), VC_ERR_WORKSPACE (workspace null, unaligned or too
 * small); VC_ERR_CUDA if a launch fails.
 */
size_t vc_quantize_workspace(vc_shape shape);
vc_status vc_quantize(const void* Q, const void* K, const void* V, vc_shape shape,
                      const int32_t* perm, int vsmooth,
                      uint8_t* Q8, float* sq, uint8_t* K8, float* sk,
                      uint8_t* V8T, float* sv, void* mu,
                      void* workspace, size_t workspace_bytes, vc_stream_t stream);

/*
 * vc_quantize with the rotary transform and the Hadamard rotation of Q and K
 * fused in: the rest of the preprocessing chain that the paper's fused
 * quantization kernel absorbs together with the block means, the gather and
 * the quantizers (paper summary 核心方法; dimensionstp.github.io 3-1 "Fused
 * CuTe kernel" and 3-3 "Kernel fusion"; the Q/K Hadamard rotation is the one
 * FlashAttention-3 applies before FP8, paper summary 研究动机).  Neither
 * formula is printed in the paper's pages; this library computes, per Q row
 * and K' row, in fp32 and in this order:
 *
 *   rope      fp32 [N, d/2, 2], 16-byte aligned, or NULL (no rotation): the
 *             (cos, sin) of the rotary angle of every token position and
 *             channel pair -- the memory layout of a complex64 [N, d/2]
 *             table, shared by all batches and heads.  Channels (2i, 2i+1)
 *             of a row holding token n become
 *               y0 = fl(fl(x0 cos) - fl(x1 sin)),  y1 = fl(fl(x0 sin) + fl(x1 cos))
 *             with (cos, sin) = rope[n][i]; row t of K' = K[perm] holds token
 *             perm[t] and is rotated at that position (as if K were rotated
 *             before the gather).
 *   hadamard  1: then y <- H_d y with the Sylvester Hadamard matrix
 *             (H_d)_ij = (-1)^popcount(i & j) (entries +-1, H_d H_d = d I),
 *             evaluated as log2(d) butterfly stages (a, b) -> (a + b, a - b),
 *             stride 1 first, each result rounded to fp32.  (H q).(H k) =
 *             d q.k, so sq carries the 1/d: sq = fl(amax/448) * (1/d), exact
 *             for d a power of two, and vc_attn_fwd needs no change.
 *             0: no rotation.
 *
 * The transformed rows are then quantized exactly as in vc_quantize (block
 * amax, codes E4M3_RNE_sat(y * 448/amax)); V is not transformed.  With
 * rope = NULL and hadamard = 0 the call is vc_quantize, bit for bit.  Same
 * workspace as vc_quantize (vc_quantize_workspace).
 * Errors: as vc_quantize, plus VC_ERR_INVALID_ARG for hadamard not in {0,1}
 * or a misaligned `rope`.
 */
vc_status vc_quantize_ex(const void* Q, const void* K, const void* V, vc_shape shape,
                         const int32_t* perm, int vsmooth, const float* rope, int hadamard,
                         uint8_t* Q8, float* sq, uint8_t* K8, float* sk,
                         uint8_t* V8T, float* sv, void* mu,
                         void* workspace, size_t workspace_bytes, vc_stream_t stream);

/*
 * The computation of vc_quantize_ex run as the unfused chain: one kernel per
 * step, each step's result written to device memory and read back by the
 * next -- rotary transform (Q and K to fp32 [B,N,H,d]), gather of K' (fp32)
 * and V' (bf16) into [B,H,N,d], Hadamard rotation in place, V block means
 * and residual maxima, Q/K block quantization, V residual codes.  Every step
 * rounds as the fused kernels do, so all outputs are bit-identical to
 * vc_quantize_ex; it is there to measure what the fusion saves (the paper
 * reports its fused chain against the unfused one, paper summary 核心方法).
 * The workspace holds the intermediates: vc_quantize_staged_workspace(shape)
 * = the vc_quantize workspace + 14 B*N*H*d bytes (+ alignment), 256-byte
 * aligned.  Same arguments, errors and results as vc_quantize_ex.
 */
size_t vc_quantize_staged_workspace(vc_shape shape);
vc_status vc_quantize_staged(const void* Q, const void* K, const void* V, vc_shape shape,
                             const int32_t* perm, int vsmooth, const float* rope, int hadamard,
                             uint8_t* Q8, float* sq, uint8_t* K8, float* sk,
                             uint8_t* V8T, float* sv, void* mu,
                             void* workspace, size_t workspace_bytes, vc_stream_t stream);

/*
 * vc_quantize with the V residual in 4 bits: the pages' 4-bit path keeps the
 * residual R = V' - mu_j in 4 bits with a per-block scale (paper summary
 * 方法步骤详情 step 2, "4 比特 NVFP4"; the summary's own analysis, weakness
 * three, and the wire.sakhanda.co section "ExpCast-FP8" note that the
 * probabilities must stay FP8 beside it).  This library's form of it, for FP8
 * probabilities on the tensor core: E2M1 codes with a power-of-two scale per
 * 32 consecutive tokens of a channel (the OCP MX rule), under a per-channel
 * fp32 scale; per (b, h, channel c):
 *   g_c = amax_t |R[t,c]| / 6 (sv),  x_t = fl(R[t,c] * fl(6 / amax));
 *   per group of 32 tokens (t = 32 i .. 32 i + 31): e = floor(log2 max |x_t|) - 2
 *   clamped to [-8, 0] (-8 for an all-zero group);
 *   q_t = E2M1_RNE_sat(x_t * 2^-e) (0, 0.5, 1, 1.5, 2, 3, 4, 6; ties to the
 *   even code), value q_t * 2^e.
 * Every such value is an E4M3 value, so V8T holds its E4M3 byte and
 * vc_attn_fwd runs unchanged: the FP8 product computes exactly what a
 * block-scaled E4M3 x E2M1 product computes, at the same tensor-core rate.
 * Q, K and the block means are as in vc_quantize; same arguments, workspace
 * and errors.
 */
vc_status vc_quantize_v4(const void* Q, const void* K, const void* V, vc_shape shape,
                         const int32_t* perm, int vsmooth,
                         uint8_t* Q8, float* sq, uint8_t* K8, float* sk,
                         uint8_t* V8T, float* sv, void* mu,
                         void* workspace, size_t workspace_bytes, vc_stream_t stream);

/*
 * vc_quantize without a workspace argument, for callers that cannot allocate
 * device memory: a host that embeds this library inside a framework whose
 * memory pool owns all device memory, or code running where an allocation
 * would synchronize the device or is not allowed.  (The paper has no
 * counterpart; this is a deployment convenience of this library.)
 *
 * Same arguments, outputs and results as vc_quantize (bit-identical codes,
 * scales and means).  The per-channel scratch lives in a fixed array compiled
 * into the library: 65536 32-bit words (256 KB), which every GPU that loads
 * the library holds until the process exits.  Limit: B*H*d <= 65536 (for
 * example H <= 512 heads at d = 128 with B = 1); larger shapes return
 * VC_ERR_WORKSPACE without launching.  Nothing is allocated: no cudaMalloc,
 * no cudaFree, no allocating library routine.
 *
 * The first call in each CUDA context (normally one per device: the primary
 * context) looks up the array's device address, with that context current,
 * and caches it; make that first call before any stream capture begins.
 * After a device reset the next call looks it up again.  Every call shares the one array and clears what it needs
 * at its start, so calls whose work overlaps on the GPU (different streams,
 * or different host threads on one device) race and must be serialized by
 * the caller.
 */
vc_status vc_quantize_static(const void* Q, const void* K, const void* V, vc_shape shape,
                             const int32_t* perm, int vsmooth,
                             uint8_t* Q8, float* sq, uint8_t* K8, float* sk,
                             uint8_t* V8T, float* sv, void* mu, vc_stream_t stream);

/*
 * FP8 attention forward, paper summary 前置知识 "在线 softmax" and 方法步骤详情
 * steps 3-4; dimensionstp.github.io 2-3 (P_ij V'_j = P_ij R_j + r_ij mu_j^T)
 * and 2-4.  Takes the outputs of vc_quantize.
 *
 * For each query row i, keys are visited in 128-token tiles in stored order
 * with an exact running max m' (scores in log2 units):
 *   acc    = sum_c q8*k8 (tcgen05 FP8 MMA, fp32 accumulate)
 *   sigma  = fp32(fp32(sq_i*sk_j) * kscale), kscale = fp32(scale * log2 e)
 *   m'     = max(m, sigma * max_k acc)
 *   expcast=1: c = clamp(rint(fmaf(acc, 8 sigma, fmaf(-8, m', 119.65f))), 0, 120)
 *   expcast=0: c = E4M3_RNE_sat(exp2(fmaf(acc, sigma, 8 - m')))
 *   expcast=3: range-adaptive ExpCast (the paper summary's own analysis,
 *              独立分析的弱点 weakness two: beta chosen by score range).
 *              t0 = fmaf(acc, 8 sigma, fmaf(-8, m', 120)),
 *              p  = (rint(t0) >> 1) & 3  (the pair of codes of its octave),
 *              c  = clamp(rint(fl(t0 + beta_p)), 0, 120), c = 0 for t0 < 0,
 *              beta = {-0.195, -0.635, -0.685, -0.535} (fp32 constants).
 *   r_ij   = sum_k decode(c)            (row sum of the quantized P)
 *   l     <- alpha l + r_ij,  alpha = exp2(m - m')
 *   A     <- alpha A + P_q V8_res * s_v + r_ij mu_j   (mu term only if vsmooth)
 *   O      = A / l, stored as bf16.
 *
 *   softmax_scale  > 0, or <= 0 for 1/sqrt(d).
 *   O        bf16 [B,N,H,d] with `shape` strides (rows in original query order).
 *   dev_status  nullable; receives VC_ERR_TIMEOUT if a device wait ran out.
 * Q8/K8/V8T must be 16-byte aligned (they are read with TMA), and so must O
 * (rows are written 16 bytes at a time).
 * Errors, all returned before any launch: VC_ERR_INVALID_ARG (a null pointer
 * -- mu may be NULL only with vsmooth = 0 --, a misaligned Q8, K8, V8T or O,
 * expcast not in {0,1,3}, vsmooth not in {0,1}, a non-positive size, or a stride that is
 * not a positive multiple of 8), VC_ERR_UNSUPPORTED (d not 64 or 128,
 * N > 2^24, or B*H*Npad >= 2^31); VC_ERR_CUDA if a tensor map cannot be
 * encoded or the launch fails.
 */
vc_status vc_attn_fwd(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk,
                      const uint8_t* V8T, const float* sv, const void* mu, vc_shape shape,
                      float softmax_scale, int expcast, int vsmooth,
                      void* O, int32_t* dev_status, vc_stream_t stream);

/*
 * vc_attn_fwd with hybrid probability bytes: the exact exponent on the key
 * tiles that carry high weight, ExpCast elsewhere.  The paper summary's own
 * analysis (独立分析的弱点, weakness two) notes that ExpCast's fixed beta costs
 * 0.7-2.1 dB and proposes keeping the exact exponent on high-weight tiles (a
 * mixed-precision softmax).  This library's rule: query rows are taken in
 * groups of 32 consecutive rows of a 128-row query tile (rows >= N do not
 * count); key tile j is exact for a group if, for some row of it,
 *   fl(sigma * max_k acc) - m' >= -exact_margin      (fp32, log2 units)
 * i.e. the tile holds a probability >= 2^-exact_margin of that row's running
 * maximum m'.  Exact tiles take the exp-then-cast byte of vc_attn_fwd with
 * expcast = 0 for every row of the group, the others the ExpCast byte.
 * exact_margin < 0 with |exact_margin| large gives vc_attn_fwd(expcast = 1),
 * a large positive one vc_attn_fwd(expcast = 0).  Other arguments, layouts
 * and errors as vc_attn_fwd; VC_ERR_INVALID_ARG for a NaN margin.
 */
vc_status vc_attn_fwd_hybrid(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk,
                             const uint8_t* V8T, const float* sv, const void* mu, vc_shape shape,
                             float softmax_scale, float exact_margin, int vsmooth,
                             void* O, int32_t* dev_status, vc_stream_t stream);

/*
 * Test hook for the ExpCast byte check: runs vc_attn_fwd and additionally,
 * for the single query tile `dbg_qtile` of head-slot `dbg_bh` (= b*H + h),
 * writes the fp32 scores acc it computed, S_dump fp32 [128, Npad], and the
 * probability bytes it fed to the PV product, P_dump uint8 [128, Npad]
 * (rows = the tile's 128 query rows, columns = keys in stored order).
 * expcast = 2 runs the hybrid bytes of vc_attn_fwd_hybrid with exact_margin
 * (ignored for 0, 1 and 3).  Same contract as vc_attn_fwd otherwise; slower
 * (a separate instantiation).
 */
vc_status vc_attn_fwd_debug(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk,
                            const uint8_t* V8T, const float* sv, const void* mu, vc_shape shape,
                            float softmax_scale, int expcast, int vsmooth,
                            void* O, int32_t* dev_status, vc_stream_t stream,
                            int dbg_bh, int dbg_qtile, float* S_dump, uint8_t* P_dump,
                            float exact_margin);

/*
 * Test hook: the device conversion the quantizer uses to write E4M3 codes
 * (round to nearest even, saturating to +-448), applied to n fp32 values.
 * x: fp32 [n], out: uint8 [n], both device memory.  Lets tests compare the
 * hardware conversion with an independent encoder over all fp32 patterns.
 */
vc_status vc_debug_e4m3_encode(const float* x, int64_t n, uint8_t* out, vc_stream_t stream);

/*
 * Test hook: launches one CTA whose mbarrier wait can never complete (two
 * arrivals expected, one made).  The library's bounded wait gives up after
 * timeout_us microseconds (1 .. 10^7), writes VC_ERR_TIMEOUT to *dev_status
 * and the kernel returns; the CUDA context stays usable.
 */
vc_status vc_debug_wait_timeout(int32_t* dev_status, uint32_t timeout_us, vc_stream_t stream);

/*
 * Test hook for the attention kernel's own failure path: runs vc_attn_fwd
 * (expcast = 1) except that its K loader never loads, nor signals, key tile
 * `skip_k_tile` (0 <= skip_k_tile < nblk), and every device wait is bounded
 * by timeout_us microseconds (1 .. 10^7) instead of 4 s.  The wait for that
 * tile runs out: the kernel writes VC_ERR_TIMEOUT to *dev_status (required
 * here), every warp of the CTA stops waiting, the CTA's own copies and MMAs
 * in flight drain, its tensor memory is freed and the kernel returns; O is
 * left unspecified.  The CUDA context stays usable.  Same other arguments as
 * vc_attn_fwd.
 */
vc_status vc_debug_attn_timeout(const uint8_t* Q8, const float* sq, const uint8_t* K8, const float* sk,
                                const uint8_t* V8T, const float* sv, const void* mu, vc_shape shape,
                                int vsmooth, void* O, int32_t* dev_status, vc_stream_t stream,
                                int skip_k_tile, uint32_t timeout_us);

#ifdef __cplusplus
}
#endif

#endif /* VC_H_ */
