// Decode against a paged KV cache: append, split-KV attention, LSE combine.
//
// Inference Cookbook FAQ Q17 (the call appends k_new/v_new but does not
// advance cache_seqlens), Q18 (paged cache, 256-token pages), Q14 (split the
// key range across CTAs when batch x heads is small, then merge).  Split s of
// batch entry i covers keys [s*chunk, (s+1)*chunk) of its L_i keys; each
// split produces a normalised partial output and its LSE, and the combine
// step merges them: lse = ln sum_s exp(lse_s), O = sum_s exp(lse_s - lse) O_s.
#include "kernels.h"

namespace attn {
namespace {

constexpr int kWarps = 4;

// Physical row of logical position t of batch entry bi, or -1 (and the error
// word raised) when the page table points outside the pool.
__device__ __forceinline__ int64_t cache_row(const DecodeArgs &a, int bi, int t) {
  const int pg_idx = t / a.page_size;
  if (pg_idx >= a.max_pages) { raise_error(a.err, kErrCacheOverflow); return -1; }
  const int page = a.block_table ? a.block_table[(int64_t)bi * a.max_pages + pg_idx] : bi;
  if (page < 0 || page >= a.num_pages) { raise_error(a.err, kErrPageOutOfRange); return -1; }
  return (int64_t)page * a.page_size + (t % a.page_size);
}

// Writes k_new/v_new into their cache slots.  grid (s_new, b), 128 threads.
template <typename T>
__global__ void append_kernel(DecodeArgs a) {
  const int t = blockIdx.x, bi = blockIdx.y;
  const int pos = a.cache_seqlens[bi] + t;
  if (pos < 0) { if (threadIdx.x == 0) raise_error(a.err, kErrBadSeqlen); return; }
  const int64_t row = cache_row(a, bi, pos);
  if (row < 0) return;
  const int n16 = a.hkv * a.d / 8;  // 16-byte chunks per token
  const int64_t src = ((int64_t)bi * a.s_new + t) * a.hkv * a.d;
  const int64_t dst = row * a.hkv * a.d;
  for (int c = threadIdx.x; c < n16; c += blockDim.x) {
    reinterpret_cast<uint4 *>(static_cast<T *>(a.k_cache) + dst)[c] =
        reinterpret_cast<const uint4 *>(static_cast<const T *>(a.k_new) + src)[c];
    reinterpret_cast<uint4 *>(static_cast<T *>(a.v_cache) + dst)[c] =
        reinterpret_cast<const uint4 *>(static_cast<const T *>(a.v_new) + src)[c];
  }
}

// Result of a row whose keys could not be read (bad length or page): O = 0
// and LSE = -inf, the result of an empty key set, so that the combine step
// gives the split no weight and the output does not depend on stale scratch
// contents.  The device error word says what happened.  One warp.
template <typename T, int D>
__device__ __forceinline__ void store_empty_row(const DecodeArgs &a, int split, int bi, int r,
                                                int h, int lane) {
  constexpr int V = D / 32;
  float z[V];
#pragma unroll
  for (int u = 0; u < V; ++u) z[u] = 0.f;
  if (a.num_splits == 1) {
    store_vec<T, V>(static_cast<T *>(a.o) + (((int64_t)bi * a.sq + r) * a.hq + h) * D + lane * V, z);
    if (lane == 0) a.lse[((int64_t)bi * a.hq + h) * a.sq + r] = -INFINITY;
  } else {
    float *op = a.o_part + (((((int64_t)split * a.b + bi) * a.sq + r) * a.hq + h) * D) + lane * V;
#pragma unroll
    for (int u = 0; u < V; ++u) op[u] = 0.f;
    if (lane == 0) a.lse_part[(((int64_t)split * a.b + bi) * a.hq + h) * a.sq + r] = -INFINITY;
  }
}

// One warp per (batch entry, query head, query row, split).
// grid (splits, hq, b); the 4 warps of a block take rows r = warp, warp+4, ...
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) decode_rows_kernel(DecodeArgs a) {
  constexpr int V = D / 32;
  __shared__ float qs[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, h = blockIdx.y, bi = blockIdx.z;
  const int L = a.cache_seqlens[bi] + a.s_new;
  if (L < 0 || L > a.max_pages * a.page_size) {
    if (threadIdx.x == 0) raise_error(a.err, L < 0 ? kErrBadSeqlen : kErrCacheOverflow);
    for (int r = warp; r < a.sq; r += kWarps) store_empty_row<T, D>(a, split, bi, r, h, lane);
    return;
  }
  const int kvh = h / (a.hq / a.hkv);
  const int64_t rs = (int64_t)a.hkv * D;
  const T *kc = static_cast<const T *>(a.k_cache) + (int64_t)kvh * D;
  const T *vc = static_cast<const T *>(a.v_cache) + (int64_t)kvh * D;
  const float sl2 = a.scale * kLog2e;
  for (int r = warp; r < a.sq; r += kWarps) {
    const int64_t qoff = (((int64_t)bi * a.sq + r) * a.hq + h) * D;
    for (int c = lane; c < D; c += 32) qs[warp][c] = Elem<T>::to_f(static_cast<const T *>(a.q)[qoff + c]);
    __syncwarp();
    int lo, hi;
    key_range(r, a.sq, L, a.win_l, a.win_r, lo, hi);
    lo = max(lo, split * a.split_chunk);
    hi = min(hi, (split + 1) * a.split_chunk - 1);
    float m = -INFINITY, l = 0.f, acc[V];
#pragma unroll
    for (int u = 0; u < V; ++u) acc[u] = 0.f;
    bool bad = false;
    for (int j0 = lo; j0 <= hi && !bad; j0 += 32) {
      const int j = j0 + lane;
      float s = -INFINITY;
      int64_t row = 0;
      if (j <= hi) {
        row = cache_row(a, bi, j);
        if (row >= 0) {
          const T *kr = kc + row * rs;
          float dot = 0.f;
#pragma unroll
          for (int c = 0; c < D; c += 8) {
            float e[8];
            load_vec<T, 8>(kr + c, e);
#pragma unroll
            for (int u = 0; u < 8; ++u) dot = fmaf(qs[warp][c + u], e[u], dot);
          }
          s = a.softcap > 0.f ? a.softcap * tanhf(dot * a.scale / a.softcap) * kLog2e : dot * sl2;
        }
      }
      bad = __any_sync(0xffffffffu, j <= hi && row < 0);
      if (bad) break;
      const float mnew = fmaxf(m, warp_max(s));
      const float alpha = exp2f(m - mnew);
      const float p = exp2f(s - mnew);
      l = l * alpha + warp_sum(p);
#pragma unroll
      for (int u = 0; u < V; ++u) acc[u] *= alpha;
      const int n = min(32, hi - j0 + 1);
      for (int jj = 0; jj < n; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
        const int64_t rj = __shfl_sync(0xffffffffu, row, jj);
        float vv[V];
        load_vec<T, V>(vc + rj * rs + lane * V, vv);
#pragma unroll
        for (int u = 0; u < V; ++u) acc[u] = fmaf(pj, vv[u], acc[u]);
      }
      m = mnew;
    }
    if (bad) {
      store_empty_row<T, D>(a, split, bi, r, h, lane);
      __syncwarp();
      continue;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int u = 0; u < V; ++u) acc[u] *= inv;
    const float lse = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    if (a.num_splits == 1) {
      store_vec<T, V>(static_cast<T *>(a.o) + qoff + lane * V, acc);
      if (lane == 0) a.lse[((int64_t)bi * a.hq + h) * a.sq + r] = lse;
    } else {
      float *op = a.o_part + (((((int64_t)split * a.b + bi) * a.sq + r) * a.hq + h) * D) + lane * V;
#pragma unroll
      for (int u = 0; u < V; ++u) op[u] = acc[u];
      if (lane == 0) a.lse_part[(((int64_t)split * a.b + bi) * a.hq + h) * a.sq + r] = lse;
    }
    __syncwarp();
  }
}

// Merge the splits of one (batch, head, row): one warp each; grid (sq, hq, b).
template <typename T, int D>
__global__ void __launch_bounds__(32) combine_kernel(DecodeArgs a) {
  constexpr int V = D / 32;
  const int lane = threadIdx.x;
  const int r = blockIdx.x, h = blockIdx.y, bi = blockIdx.z;
  const int64_t stride_l = (int64_t)a.b * a.hq * a.sq;
  const int64_t li = ((int64_t)bi * a.hq + h) * a.sq + r;
  // splits whose key range holds no key any query row may see were not
  // written (same test as the split kernels); they are skipped
  const int L = a.cache_seqlens[bi] + a.s_new;
  int lo0, hi0, lo1, hi1;
  key_range(0, a.sq, L, a.win_l, a.win_r, lo0, hi0);
  key_range(a.sq - 1, a.sq, L, a.win_l, a.win_r, lo1, hi1);
  auto used = [&](int s) {
    const int kb = max(lo0, s * a.split_chunk);
    const int ke = min(hi1 + 1, min(L, (s + 1) * a.split_chunk));
    return ke > kb;
  };
  float m = -INFINITY;
  for (int s = lane; s < a.num_splits; s += 32)
    if (used(s)) m = fmaxf(m, a.lse_part[s * stride_l + li]);
  m = warp_max(m);
  float acc[V];
#pragma unroll
  for (int u = 0; u < V; ++u) acc[u] = 0.f;
  float wsum = 0.f;
  if (m > -INFINITY) {
    const int64_t stride_o = (int64_t)a.b * a.sq * a.hq * D;
    const int64_t oi = (((int64_t)bi * a.sq + r) * a.hq + h) * D + lane * V;
    for (int s = 0; s < a.num_splits; ++s) {
      if (!used(s)) continue;
      const float w = exp2f((a.lse_part[s * stride_l + li] - m) * kLog2e);
      if (w == 0.f) continue;
      wsum += w;
      const float *op = a.o_part + s * stride_o + oi;
#pragma unroll
      for (int u = 0; u < V; ++u) acc[u] = fmaf(w, op[u], acc[u]);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int u = 0; u < V; ++u) acc[u] *= inv;
  store_vec<T, V>(static_cast<T *>(a.o) + (((int64_t)bi * a.sq + r) * a.hq + h) * D + lane * V, acc);
  if (lane == 0) a.lse[li] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

template <typename T, int D>
cudaError_t decode(const DecodeArgs &a, cudaStream_t st) {
  if (a.s_new > 0) {
    append_kernel<T><<<dim3(a.s_new, a.b), 128, 0, st>>>(a);
  }
  count_launches(a.s_new > 0);
  // tensor-core kernel (g * sq <= 32, pages of 128-token multiples); warp-per-row kernel otherwise
  cudaError_t e = launch_decode_tc(a, st);
  if (e == cudaErrorNotSupported) {
    debug_log("decode: decode_rows_kernel (CUDA cores, one warp per query row) d=%d, "
              "num_splits=%d (%d keys each)", D, a.num_splits, a.split_chunk);
    decode_rows_kernel<T, D><<<dim3(a.num_splits, a.hq, a.b), kWarps * 32, 0, st>>>(a);
    count_launches(1);
  } else if (e != cudaSuccess) {
    return e;
  }
  if (a.num_splits > 1) {
    combine_kernel<T, D><<<dim3(a.sq, a.hq, a.b), 32, 0, st>>>(a);
    count_launches(1);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st) {
  const bool bf = a.dtype == ATTN_BF16;
  switch (a.d) {
    case 64: return bf ? decode<__nv_bfloat16, 64>(a, st) : decode<__half, 64>(a, st);
    case 128: return bf ? decode<__nv_bfloat16, 128>(a, st) : decode<__half, 128>(a, st);
    case 256: return bf ? decode<__nv_bfloat16, 256>(a, st) : decode<__half, 256>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
