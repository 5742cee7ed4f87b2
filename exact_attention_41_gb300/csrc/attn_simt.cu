// Warp-per-row forward (CUDA cores, fp32 math).
//
// One warp owns one query row.  Lanes take 32 keys at a time for the dot
// products, and 32 column slices of the head dimension for the
// accumulation, exchanging the per-key scalars with warp shuffles: the
// online softmax of "FlashAttention完整说明" §二.1 with key blocks of 32.
// Used only where the tensor-core forward does not apply: a problem with no
// keys at all (every row empty: O = 0, LSE = -inf).
#include "kernels.h"

namespace attn {
namespace {

constexpr int kWarps = 4;

template <typename T, int D>
__device__ __forceinline__ float dot_row(const float *x_s, const T *row) {
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < D; c += 8) {
    float e[8];
    load_vec<T, 8>(row + c, e);
#pragma unroll
    for (int u = 0; u < 8; ++u) acc = fmaf(x_s[c + u], e[u], acc);
  }
  return acc;
}

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) fwd_rows_kernel(FwdArgs a) {
  constexpr int V = D / 32;
  __shared__ float qs[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h = blockIdx.y;
  const int i = blockIdx.x * kWarps + warp;
  int q0, lq, k0, lk;
  if (!a.seqs.get(b, q0, lq, k0, lk, a.err) || i >= lq) return;
  const int kvh = h / (a.hq / a.hkv);
  const int64_t krs = a.k_rs, vrs = a.v_rs;
  const T *qrow = static_cast<const T *>(a.q) + (int64_t)(q0 + i) * a.q_rs + (int64_t)h * D;
  const T *kb = static_cast<const T *>(a.k) + (int64_t)k0 * krs + (int64_t)kvh * D;
  const T *vb = static_cast<const T *>(a.v) + (int64_t)k0 * vrs + (int64_t)kvh * D;
  for (int c = lane; c < D; c += 32) qs[warp][c] = Elem<T>::to_f(qrow[c]);
  __syncwarp();
  int lo, hi;
  key_range(i, lq, lk, a.win_l, a.win_r, lo, hi);
  const float sl2 = a.scale * kLog2e;
  float m = -INFINITY, l = 0.f, acc[V];
#pragma unroll
  for (int u = 0; u < V; ++u) acc[u] = 0.f;
  for (int j0 = lo; j0 <= hi; j0 += 32) {
    const int j = j0 + lane;
    float s = -INFINITY;
    if (j <= hi) {
      const float dot = dot_row<T, D>(qs[warp], kb + (int64_t)j * krs);
      s = a.softcap > 0.f ? a.softcap * tanhf(dot * a.scale / a.softcap) * kLog2e : dot * sl2;
    }
    const float mnew = fmaxf(m, warp_max(s));
    const float alpha = exp2f(m - mnew);
    const float p = exp2f(s - mnew);
    l = l * alpha + warp_sum(p);
#pragma unroll
    for (int u = 0; u < V; ++u) acc[u] *= alpha;
    const int n = min(32, hi - j0 + 1);
    for (int jj = 0; jj < n; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      float vv[V];
      load_vec<T, V>(vb + (int64_t)(j0 + jj) * vrs + lane * V, vv);
#pragma unroll
      for (int u = 0; u < V; ++u) acc[u] = fmaf(pj, vv[u], acc[u]);
    }
    m = mnew;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int u = 0; u < V; ++u) acc[u] *= inv;
  store_vec<T, V>(static_cast<T *>(a.o) + ((int64_t)(q0 + i) * a.hq + h) * D + lane * V, acc);
  if (lane == 0)
    a.lse[a.seqs.lse_index(b, h, q0, i)] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

template <typename T, int D>
cudaError_t fwd_rows(const FwdArgs &a, cudaStream_t st) {
  dim3 grid((a.seqs.sq + kWarps - 1) / kWarps, a.hq, a.batch);
  fwd_rows_kernel<T, D><<<grid, kWarps * 32, 0, st>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs &a, cudaStream_t st) {
  debug_log("forward: row kernel on CUDA cores (one warp per query row), d=%d", a.d);
  const bool bf = a.dtype == ATTN_BF16;
  switch (a.d) {
    case 64: return bf ? fwd_rows<__nv_bfloat16, 64>(a, st) : fwd_rows<__half, 64>(a, st);
    case 128: return bf ? fwd_rows<__nv_bfloat16, 128>(a, st) : fwd_rows<__half, 128>(a, st);
    case 256: return bf ? fwd_rows<__nv_bfloat16, 256>(a, st) : fwd_rows<__half, 256>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
