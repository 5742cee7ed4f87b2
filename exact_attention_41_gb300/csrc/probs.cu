// Two small CUDA-core kernels beside the attention path.
//
// probs_kernel: the probability matrix of a forward call for debugging
// (Inference Cookbook FAQ Q9, return_attn_probs).  P_ij = exp(s_ij - LSE_i)
// for visible pairs, where s is the scaled, soft-capped score (FAQ Q22 order)
// and the mask is the bottom-right causal / sliding-window one of the
// forward (FAQ Q6, Q21).  One thread per key; the query row is staged in
// shared memory as fp32.  It materialises O(sq * sk) values per head, which
// is the point of the debug output and the reason it is off the hot path.
//
// advance_kernel: cache_seqlens += s_new on the device (FAQ Q17), so a decode
// step can be captured in a CUDA graph with the length update inside it
// (FAQ Q19).
#include "kernels.h"

namespace attn {
namespace {

constexpr int kKeysPerBlock = 128;

template <typename T>
__global__ void __launch_bounds__(kKeysPerBlock) probs_kernel(FwdArgs a, float *p) {
  __shared__ float qs[256];
  const int d = a.d;
  const int i = blockIdx.y;
  const int bh = blockIdx.z;
  const int bi = bh / a.hq, h = bh % a.hq;
  const int sq = a.seqs.sq, sk = a.seqs.sk;
  const int kvh = h / (a.hq / a.hkv);
  const T *qrow = static_cast<const T *>(a.q) + (((int64_t)bi * sq + i) * a.hq + h) * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) qs[c] = Elem<T>::to_f(qrow[c]);
  __syncthreads();
  const int j = blockIdx.x * kKeysPerBlock + threadIdx.x;
  if (j >= sk) return;
  const uint4 *krow = reinterpret_cast<const uint4 *>(
      static_cast<const T *>(a.k) + (((int64_t)bi * sk + j) * a.hkv + kvh) * d);
  float acc = 0.f;
  for (int c8 = 0; c8 < d / 8; ++c8) {
    const uint4 u = krow[c8];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 kv = Elem<T>::to_f2(w[e]);
      acc = fmaf(qs[8 * c8 + 2 * e], kv.x, acc);
      acc = fmaf(qs[8 * c8 + 2 * e + 1], kv.y, acc);
    }
  }
  float s = acc * a.scale;
  if (a.softcap > 0.f) s = a.softcap * tanhf(s / a.softcap);
  int lo, hi;
  key_range(i, sq, sk, a.win_l, a.win_r, lo, hi);
  const float lse = a.lse[((int64_t)bi * a.hq + h) * sq + i];
  const bool vis = j >= lo && j <= hi && lse > -INFINITY;
  p[(((int64_t)bi * a.hq + h) * sq + i) * sk + j] = vis ? expf(s - lse) : 0.f;
}

__global__ void advance_kernel(int32_t *cache_seqlens, int b, int s_new) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < b) cache_seqlens[i] += s_new;
}

}  // namespace

cudaError_t launch_probs(const FwdArgs &a, float *p, cudaStream_t st) {
  const int sq = a.seqs.sq, sk = a.seqs.sk;
  if (a.batch == 0 || sq == 0) return cudaSuccess;
  if (sk == 0) return cudaSuccess;  // (b, hq, sq, 0): nothing to write
  const int64_t bh = (int64_t)a.batch * a.hq;
  if (bh > 65535 || sq > 65535) return cudaErrorInvalidValue;  // grid y/z limits
  const dim3 grid((sk + kKeysPerBlock - 1) / kKeysPerBlock, sq, (unsigned)bh);
  if (a.dtype == ATTN_BF16)
    probs_kernel<__nv_bfloat16><<<grid, kKeysPerBlock, 0, st>>>(a, p);
  else
    probs_kernel<__half><<<grid, kKeysPerBlock, 0, st>>>(a, p);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_kvcache_advance(int32_t *cache_seqlens, int b, int s_new, cudaStream_t st) {
  if (b == 0) return cudaSuccess;
  advance_kernel<<<(b + 255) / 256, 256, 0, st>>>(cache_seqlens, b, s_new);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace attn
