// vc_selftest.cu -- test hooks: the device E4M3 conversion the quantizer uses,
// and a kernel whose wait can never complete, to check that the library's
// bounded waits end with VC_ERR_TIMEOUT instead of hanging.
#include "vc_device.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

__global__ void e4m3_encode_kernel(const float* x, int64_t n, uint8_t* out) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 2;
    if (i + 1 < n) {
        const uint32_t c = cvt_e4m3x2(x[i], x[i + 1]);
        out[i] = (uint8_t)(c & 0xFFu);
        out[i + 1] = (uint8_t)(c >> 8);
    } else if (i < n) {
        out[i] = (uint8_t)(cvt_e4m3x2(x[i], 0.f) & 0xFFu);
    }
}

// One mbarrier expecting two arrivals; only one ever arrives.
__global__ void wait_timeout_kernel(int32_t* dev_status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 2);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_arrive(b);
    mbar_wait(b, 0, &abort_flag, dev_status, timeout_ns);
}

}  // namespace
}  // namespace vc

extern "C" vc_status vc_debug_e4m3_encode(const float* x, int64_t n, uint8_t* out, vc_stream_t stream) {
    if (!x || !out || n < 0) return VC_ERR_INVALID_ARG;
    if (n == 0) return VC_OK;
    const int64_t pairs = (n + 1) / 2;
    const int threads = 256;
    const int64_t blocks = (pairs + threads - 1) / threads;
    if (blocks > 0x7FFFFFFF) return VC_ERR_UNSUPPORTED;
    vc::e4m3_encode_kernel<<<(unsigned)blocks, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(x, n, out);
    return vc::cuda_status(cudaGetLastError());
}

extern "C" vc_status vc_debug_wait_timeout(int32_t* dev_status, uint32_t timeout_us, vc_stream_t stream) {
    if (!dev_status || timeout_us == 0 || timeout_us > 10000000u) return VC_ERR_INVALID_ARG;
    vc::wait_timeout_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev_status,
                                                                                 (uint64_t)timeout_us * 1000ull);
    return vc::cuda_status(cudaGetLastError());
}
