// Warp-per-row forward and backward kernels (CUDA cores, fp32 math).
//
// One warp owns one query row (forward, dQ) or one key row (dK/dV).  Lanes
// take 32 keys (or 32 query rows) at a time for the dot products, and 32
// column slices of the head dimension for the accumulations, exchanging the
// per-key scalars with warp shuffles.  The forward is the online softmax of
// "FlashAttention完整说明" §二.1 with key blocks of 32; the backward
// recomputes P from Q, K and the saved LSE (§二.2).  Used where the
// tensor-core kernels do not apply: the backward for d = 64 and d = 256, and
// the forward of a problem with no keys at all.
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

// D_i = sum_c dO_ic * O_ic, stored in the LSE layout.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_dsum_kernel(BwdArgs a) {
  constexpr int V = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h = blockIdx.y;
  const int i = blockIdx.x * kWarps + warp;
  int q0, lq, k0, lk;
  if (!a.f.seqs.get(b, q0, lq, k0, lk, a.f.err) || i >= lq) return;
  const int64_t off = ((int64_t)(q0 + i) * a.f.hq + h) * D + lane * V;
  float o[V], g[V];
  load_vec<T, V>(static_cast<const T *>(a.f.o) + off, o);
  load_vec<T, V>(static_cast<const T *>(a.dout) + off, g);
  float acc = 0.f;
#pragma unroll
  for (int u = 0; u < V; ++u) acc = fmaf(o[u], g[u], acc);
  acc = warp_sum(acc);
  if (lane == 0) a.dsum[a.f.seqs.lse_index(b, h, q0, i)] = acc;
}

// dQ_i = scale * sum_j dS_ij k_j, one warp per query row (no atomics).
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_dq_rows_kernel(BwdArgs a) {
  constexpr int V = D / 32;
  __shared__ float qs[kWarps][D];
  __shared__ float gs[kWarps][D];
  const FwdArgs &f = a.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h = blockIdx.y;
  const int i = blockIdx.x * kWarps + warp;
  int q0, lq, k0, lk;
  if (!f.seqs.get(b, q0, lq, k0, lk, f.err) || i >= lq) return;
  const int kvh = h / (f.hq / f.hkv);
  const int64_t krs = f.k_rs, vrs = f.v_rs;
  const int64_t qoff = (int64_t)(q0 + i) * f.q_rs + (int64_t)h * D;      // q
  const int64_t goff = ((int64_t)(q0 + i) * f.hq + h) * D;             // dO (contiguous)
  const T *kb = static_cast<const T *>(f.k) + (int64_t)k0 * krs + (int64_t)kvh * D;
  const T *vb = static_cast<const T *>(f.v) + (int64_t)k0 * vrs + (int64_t)kvh * D;
  for (int c = lane; c < D; c += 32) {
    qs[warp][c] = Elem<T>::to_f(static_cast<const T *>(f.q)[qoff + c]);
    gs[warp][c] = Elem<T>::to_f(static_cast<const T *>(a.dout)[goff + c]);
  }
  __syncwarp();
  const int64_t li = f.seqs.lse_index(b, h, q0, i);
  const float lse2 = f.lse[li] * kLog2e, dsum = a.dsum[li];
  int lo, hi;
  key_range(i, lq, lk, f.win_l, f.win_r, lo, hi);
  float acc[V];
#pragma unroll
  for (int u = 0; u < V; ++u) acc[u] = 0.f;
  for (int j0 = lo; j0 <= hi; j0 += 32) {
    const int j = j0 + lane;
    float ds = 0.f;
    if (j <= hi) {
      const float s_raw = dot_row<T, D>(qs[warp], kb + (int64_t)j * krs) * f.scale;
      float s = s_raw, dcap = 1.f;
      if (f.softcap > 0.f) {
        const float t = tanhf(s_raw / f.softcap);
        s = f.softcap * t;
        dcap = 1.f - t * t;
      }
      const float p = exp2f(s * kLog2e - lse2);
      const float dp = dot_row<T, D>(gs[warp], vb + (int64_t)j * vrs);
      ds = p * (dp - dsum) * dcap;
    }
    const int n = min(32, hi - j0 + 1);
    for (int jj = 0; jj < n; ++jj) {
      const float dj = __shfl_sync(0xffffffffu, ds, jj);
      float kk[V];
      load_vec<T, V>(kb + (int64_t)(j0 + jj) * krs + lane * V, kk);
#pragma unroll
      for (int u = 0; u < V; ++u) acc[u] = fmaf(dj, kk[u], acc[u]);
    }
  }
#pragma unroll
  for (int u = 0; u < V; ++u) acc[u] *= f.scale;
  store_vec<T, V>(static_cast<T *>(a.dq) + (int64_t)(q0 + i) * a.dq_rs + (int64_t)h * D + lane * V,
                  acc);
}

// dV_j = sum_{h in group} sum_i P_ij dO_i and dK_j = scale * sum dS_ij q_i,
// one warp per key row, summing the group's query heads in a fixed order.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_dkdv_rows_kernel(BwdArgs a) {
  constexpr int V = D / 32;
  __shared__ float ks[kWarps][D];
  __shared__ float vs[kWarps][D];
  const FwdArgs &f = a.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int j = blockIdx.x * kWarps + warp;
  int q0, lq, k0, lk;
  if (!f.seqs.get(b, q0, lq, k0, lk, f.err) || j >= lk) return;
  const int g = f.hq / f.hkv;
  const int64_t krow = (int64_t)(k0 + j), col = (int64_t)kvh * D;
  for (int c = lane; c < D; c += 32) {
    ks[warp][c] = Elem<T>::to_f(static_cast<const T *>(f.k)[krow * f.k_rs + col + c]);
    vs[warp][c] = Elem<T>::to_f(static_cast<const T *>(f.v)[krow * f.v_rs + col + c]);
  }
  __syncwarp();
  int lo, hi;
  query_range(j, lq, lk, f.win_l, f.win_r, lo, hi);
  float dk[V], dv[V];
#pragma unroll
  for (int u = 0; u < V; ++u) dk[u] = dv[u] = 0.f;
  for (int t = 0; t < g; ++t) {
    const int h = kvh * g + t;
    const T *qb = static_cast<const T *>(f.q) + (int64_t)q0 * f.q_rs + (int64_t)h * D;
    const T *gb = static_cast<const T *>(a.dout) + ((int64_t)q0 * f.hq + h) * D;
    const int64_t qrs = f.q_rs, grs = (int64_t)f.hq * D;
    for (int i0 = lo; i0 <= hi; i0 += 32) {
      const int i = i0 + lane;
      float p = 0.f, ds = 0.f;
      if (i <= hi) {
        const int64_t li = f.seqs.lse_index(b, h, q0, i);
        const float s_raw = dot_row<T, D>(ks[warp], qb + (int64_t)i * qrs) * f.scale;
        float s = s_raw, dcap = 1.f;
        if (f.softcap > 0.f) {
          const float tt = tanhf(s_raw / f.softcap);
          s = f.softcap * tt;
          dcap = 1.f - tt * tt;
        }
        p = exp2f(s * kLog2e - f.lse[li] * kLog2e);
        const float dp = dot_row<T, D>(vs[warp], gb + (int64_t)i * grs);
        ds = p * (dp - a.dsum[li]) * dcap;
      }
      const int n = min(32, hi - i0 + 1);
      for (int ii = 0; ii < n; ++ii) {
        const float pi = __shfl_sync(0xffffffffu, p, ii);
        const float di = __shfl_sync(0xffffffffu, ds, ii);
        float gg[V], qq[V];
        load_vec<T, V>(gb + (int64_t)(i0 + ii) * grs + lane * V, gg);
        load_vec<T, V>(qb + (int64_t)(i0 + ii) * qrs + lane * V, qq);
#pragma unroll
        for (int u = 0; u < V; ++u) {
          dv[u] = fmaf(pi, gg[u], dv[u]);
          dk[u] = fmaf(di, qq[u], dk[u]);
        }
      }
    }
  }
#pragma unroll
  for (int u = 0; u < V; ++u) dk[u] *= f.scale;
  store_vec<T, V>(static_cast<T *>(a.dk) + krow * a.dk_rs + col + lane * V, dk);
  store_vec<T, V>(static_cast<T *>(a.dv) + krow * a.dv_rs + col + lane * V, dv);
}

template <typename T, int D>
cudaError_t fwd_rows(const FwdArgs &a, cudaStream_t st) {
  dim3 grid((a.seqs.sq + kWarps - 1) / kWarps, a.hq, a.batch);
  fwd_rows_kernel<T, D><<<grid, kWarps * 32, 0, st>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_rows(const BwdArgs &a, cudaStream_t st) {
  const FwdArgs &f = a.f;
  dim3 gq((f.seqs.sq + kWarps - 1) / kWarps, f.hq, f.batch);
  bwd_dsum_kernel<T, D><<<gq, kWarps * 32, 0, st>>>(a);
  bwd_dq_rows_kernel<T, D><<<gq, kWarps * 32, 0, st>>>(a);
  dim3 gk((f.seqs.sk + kWarps - 1) / kWarps, f.hkv, f.batch);
  bwd_dkdv_rows_kernel<T, D><<<gk, kWarps * 32, 0, st>>>(a);
  count_launches(3);
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

cudaError_t launch_bwd_simt(const BwdArgs &a, cudaStream_t st) {
  debug_log("backward: row kernels on CUDA cores (one warp per query / key row), d=%d", a.f.d);
  const bool bf = a.f.dtype == ATTN_BF16;
  switch (a.f.d) {
    case 64: return bf ? bwd_rows<__nv_bfloat16, 64>(a, st) : bwd_rows<__half, 64>(a, st);
    case 128: return bf ? bwd_rows<__nv_bfloat16, 128>(a, st) : bwd_rows<__half, 128>(a, st);
    case 256: return bf ? bwd_rows<__nv_bfloat16, 256>(a, st) : bwd_rows<__half, 256>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
