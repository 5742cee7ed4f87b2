// Shared device-side definitions for the libattn kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/libattn.h"

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Bits of the sticky device error word (attn_get_device_error's `detail`).
enum : int {
  kErrPageOutOfRange = 1,   // block_table entry outside [0, num_pages)
  kErrCacheOverflow = 2,    // cache_seqlens + s_new exceeds the cache capacity
  kErrVarlenTooLong = 4,    // a varlen sequence exceeds max_seqlen_q/k
  kErrTimeout = 8,          // a bounded wait gave up
  kErrBadSeqlen = 16,       // negative length or offsets out of order
};

__device__ __forceinline__ void raise_error(int *err, int bit) {
  if (err) atomicOr(err, bit);
}

template <typename T> struct Elem;
template <> struct Elem<__half> {
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
  static __device__ __forceinline__ float2 to_f2(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(h);
  }
  static __device__ __forceinline__ uint32_t from_f2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
  }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ float2 to_f2(uint32_t u) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(h);
  }
  static __device__ __forceinline__ uint32_t from_f2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
  }
};

// Load N (2, 4 or 8) consecutive elements as floats (aligned vector load).
template <typename T, int N>
__device__ __forceinline__ void load_vec(const T *p, float *out) {
  static_assert(N == 2 || N == 4 || N == 8, "vector width");
  if constexpr (N == 2) {
    uint32_t u = *reinterpret_cast<const uint32_t *>(p);
    float2 f = Elem<T>::to_f2(u);
    out[0] = f.x; out[1] = f.y;
  } else if constexpr (N == 4) {
    uint2 u = *reinterpret_cast<const uint2 *>(p);
    float2 a = Elem<T>::to_f2(u.x), b = Elem<T>::to_f2(u.y);
    out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
  } else {
    uint4 u = *reinterpret_cast<const uint4 *>(p);
    float2 a = Elem<T>::to_f2(u.x), b = Elem<T>::to_f2(u.y);
    float2 c = Elem<T>::to_f2(u.z), e = Elem<T>::to_f2(u.w);
    out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
    out[4] = c.x; out[5] = c.y; out[6] = e.x; out[7] = e.y;
  }
}

template <typename T, int N>
__device__ __forceinline__ void store_vec(T *p, const float *in) {
  if constexpr (N == 2) {
    *reinterpret_cast<uint32_t *>(p) = Elem<T>::from_f2(in[0], in[1]);
  } else if constexpr (N == 4) {
    uint2 u{Elem<T>::from_f2(in[0], in[1]), Elem<T>::from_f2(in[2], in[3])};
    *reinterpret_cast<uint2 *>(p) = u;
  } else {
    uint4 u{Elem<T>::from_f2(in[0], in[1]), Elem<T>::from_f2(in[2], in[3]),
            Elem<T>::from_f2(in[4], in[5]), Elem<T>::from_f2(in[6], in[7])};
    *reinterpret_cast<uint4 *>(p) = u;
  }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Sequence geometry shared by the dense and the varlen (packed) problems.
// Dense: sequence b owns rows b*sq .. b*sq+sq-1 of the (rows, heads, d) view.
// Varlen: rows cu_q[b] .. cu_q[b+1]-1 (Inference Cookbook FAQ Q8).
struct Seqs {
  const int32_t *cu_q;  // nullptr for dense
  const int32_t *cu_k;
  int sq, sk;           // dense lengths, or the stated maxima for varlen
  int total_q;          // varlen LSE row stride (hq, total_q); dense: unused
  int total_k;          // varlen key rows; dense: unused
  int hq;

  // Returns false if the sequence is malformed (and raises the error word).
  __device__ __forceinline__ bool get(int b, int &q0, int &lq, int &k0, int &lk,
                                      int *err) const {
    if (!cu_q) {
      q0 = b * sq; lq = sq; k0 = b * sk; lk = sk;
      return true;
    }
    q0 = cu_q[b]; lq = cu_q[b + 1] - q0;
    k0 = cu_k[b]; lk = cu_k[b + 1] - k0;
    // offsets must stay inside the packed tensors: a sequence ending past
    // total_q / total_k would make the output and gradient stores run off
    // the end of the caller's buffers
    if (lq < 0 || lk < 0 || q0 < 0 || k0 < 0 || q0 + lq > total_q || k0 + lk > total_k) {
      raise_error(err, kErrBadSeqlen);
      return false;
    }
    if (lq > sq || lk > sk) { raise_error(err, kErrVarlenTooLong); return false; }
    return true;
  }
  // Index of LSE(b, h, row i): dense (b, hq, sq), varlen (hq, total_q).
  __device__ __forceinline__ int64_t lse_index(int b, int h, int q0, int i) const {
    if (!cu_q) return ((int64_t)b * hq + h) * sq + i;
    return (int64_t)h * total_q + q0 + i;
  }
};

// Visible key range [lo, hi] of query row i (bottom-right alignment,
// Inference Cookbook FAQ Q6; window bounds FAQ Q21).  win_r already carries
// causal (= 0).  Empty when hi < lo.
__device__ __forceinline__ void key_range(int i, int lq, int lk, int win_l, int win_r,
                                          int &lo, int &hi) {
  const int pos = i + (lk - lq);
  hi = (win_r < 0) ? lk - 1 : min(lk - 1, pos + win_r);
  lo = (win_l < 0) ? 0 : max(0, pos - win_l);
}

// Query rows [lo, hi] that see key j (the transpose of key_range).
__device__ __forceinline__ void query_range(int j, int lq, int lk, int win_l, int win_r,
                                            int &lo, int &hi) {
  const int off = lk - lq;
  lo = (win_r < 0) ? 0 : max(0, j - off - win_r);
  hi = (win_l < 0) ? lq - 1 : min(lq - 1, j - off + win_l);
}

}  // namespace attn
