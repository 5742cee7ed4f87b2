// Support for the FP8 forward (Inference Cookbook FAQ Q20: FP8 inputs, BF16
// output).  Q and K stay E4M3 and feed the tensor cores directly
// (kind::f8f6f4, fwd_sm103.cu); V is widened once to bf16 here, which is
// exact (every E4M3 value is a bf16 value), so P V runs at 16 bits like the
// 16-bit forward and P keeps 8 significant bits rather than 4.
#include <cuda_fp8.h>

#include "kernels.h"

namespace attn {
namespace {

// 16 E4M3 bytes -> 16 bf16 values per thread and step.
__global__ void __launch_bounds__(256) widen_e4m3_kernel(const uint4 *src, uint4 *dst,
                                                         int64_t n16) {
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n16;
       x += (int64_t)gridDim.x * blockDim.x) {
    const uint4 u = src[x];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        // two E4M3 bytes -> two halves (exact) -> two floats -> bf16 pair (exact)
        const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(
            (__nv_fp8x2_storage_t)((w[e] >> (16 * hh)) & 0xFFFFu), __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
        o[2 * e + hh] = Elem<__nv_bfloat16>::from_f2(f.x, f.y);
      }
    }
    dst[2 * x] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[2 * x + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace

cudaError_t launch_widen_e4m3(const void *src, void *dst, int64_t n, int sms, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  if (n % 16) return cudaErrorInvalidValue;
  const int64_t n16 = n / 16;
  const int blocks = (int)std::min<int64_t>((n16 + 255) / 256, (int64_t)sms * 8);
  widen_e4m3_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint4 *>(src),
                                            static_cast<uint4 *>(dst), n16);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace attn
