// Backward attention on the 5th-generation tensor cores (sm_103a), d = 128.
//
// "FlashAttention完整说明" §二.2: the forward keeps only O and the softmax
// statistics; the backward recomputes S and P tile by tile from Q, K and the
// saved LSE.  With D_i = sum_c dO_ic O_ic (the preprocess kernel):
//
//   P = exp(s - LSE),  dV += P^T dO,  dP = dO V^T,
//   dS = P * (dP - D) [* (1 - tanh^2) under softcap],
//   dK += dS^T Q,  dQ += dS K          (dK, dQ scaled by `scale` at the end)
//
// One CTA owns a block of 128 keys of one (batch, KV head) and loops over the
// query heads of its GQA group and the 64-row query chunks that can see those
// keys.  Roles:
//
//   warp 0       TMA producer: K and V once, Q and dO chunks into a 3-stage ring.
//   warp 1       MMA issuer: S^T = K Q^T and dP^T = V dO^T into TMEM, then
//                dV += P^T dO, dK += dS^T Q and dQ^T = K^T dS^T (P^T and dS^T
//                from shared memory).
//   warps 2-9    two warpgroups, one thread per (key row, half of the chunk's
//                queries): P^T and dS^T from S^T and dP^T, written to shared
//                memory as a high and a low 16-bit part each, so the dV and dK
//                products see P and dS to about 16 significant bits; finally
//                dK and dV out of TMEM.
//   warps 10-13  one thread per head-dim column: dQ^T out of TMEM, added into
//                an fp32 accumulator in global memory (`red.global.add`).
//                In deterministic mode (Inference Cookbook FAQ Q11) this
//                kernel skips dQ and the query-stationary kernel of
//                bwd_dq_sm103.cu computes it without atomics.
//
// TMEM (512 columns): dV [0,128), dK [128,256), S^T [256,320), dP^T [320,384),
// dQ^T buffers [384,448) and [448,512).
#include <cudaTypedefs.h>

#include <algorithm>

#include "kernels.h"
#include "sm103.cuh"

namespace attn {

namespace {
using namespace sm103;

constexpr int D = 128;
constexpr int BN = 128;   // keys per CTA
constexpr int BQ = 64;    // query rows per iteration
constexpr int ST = 3;     // Q/dO ring stages
constexpr int kThreads = 448;
constexpr int kTileK = BN * D * 2;       // 32 KB
constexpr int kChunk = BQ * D * 2;       // 16 KB
constexpr int kPT = BN * BQ * 2;         // 16 KB
constexpr int kSmemData = 2 * kTileK + ST * 2 * kChunk + 4 * kPT;  // 224 KB
constexpr int kSmem = kSmemData + 1024;
constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 320, kColDQ = 384;

struct Shared {
  uint64_t kv_full;
  uint64_t qd_full[ST], qd_empty[ST];
  uint64_t sdp_full, st_free, pds_full;
  uint64_t mma_done[2], dq_free[2];
  uint64_t grp_p[2], grp_q;  // bounded barriers of each P^T warpgroup and of the dQ warpgroup
  uint32_t tmem_base;
  int abort;
  float lse2[2][2][BQ / 2];  // [warpgroup][buffer][column]
  float dsum[2][2][BQ / 2];
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool wait_bar(Shared &sh, uint64_t *bar, uint32_t parity, int *err) {
  const uint32_t a = smem_u32(bar);
  if (mbar_test(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_test(a, parity)) return true;
    if ((spin & 255) == 0) {
      if (*(volatile int *)&sh.abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        raise_error(err, kErrTimeout);
        *(volatile int *)&sh.abort = 1;
        return false;
      }
    }
  }
}

// The same wait taken by a whole warp with one answer, so warp-collective
// tcgen05 loads/stores that follow are never reached by part of a warp.
__device__ __forceinline__ bool wait_warp(Shared &sh, uint64_t *bar, uint32_t parity, int *err) {
  return __all_sync(0xffffffffu, wait_bar(sh, bar, parity, err));
}

template <typename T> struct IsBf16 { static constexpr int v = 0; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr int v = 1; };

// Fire-and-forget fp32 add to global memory (no value returned).
__device__ __forceinline__ void red_add(float *p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// x = hi + lo with hi, lo 16-bit: packed pairs of the high parts and of the
// low parts.  bf16: hi is x with its low 16 bits cleared (truncation), so
// lo = x - hi is exact in fp32 and only lo is rounded; fp16: hi rounded to
// nearest, lo the rounded remainder.
template <typename T>
__device__ __forceinline__ void split_hi_lo(const float (&x)[2], uint32_t &hi, uint32_t &lo) {
  if constexpr (IsBf16<T>::v) {
    const uint32_t a = __float_as_uint(x[0]) & 0xFFFF0000u, b = __float_as_uint(x[1]) & 0xFFFF0000u;
    hi = __byte_perm(a, b, 0x7632);  // high halves of a and b -> (a, b) packed
    lo = Elem<T>::from_f2(x[0] - __uint_as_float(a), x[1] - __uint_as_float(b));
  } else {
    hi = Elem<T>::from_f2(x[0], x[1]);
    const float2 h = Elem<T>::to_f2(hi);
    lo = Elem<T>::from_f2(x[0] - h.x, x[1] - h.y);
  }
}

// Query chunks [c_lo, c_lo + nch) that can see any key of block nb.
__device__ __forceinline__ void chunk_range(int nb, int lq, int lk, int win_l, int win_r,
                                            int &c_lo, int &nch) {
  const int key0 = nb * BN, key1 = min(key0 + BN, lk) - 1;
  int lo0, hi0, lo1, hi1;
  query_range(key0, lq, lk, win_l, win_r, lo0, hi0);
  query_range(key1, lq, lk, win_l, win_r, lo1, hi1);
  if (key1 < key0 || hi1 < lo0 || hi1 < 0 || lo0 > lq - 1) {
    c_lo = 0;
    nch = 0;
    return;
  }
  c_lo = lo0 / BQ;
  nch = hi1 / BQ - c_lo + 1;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const BwdArgs a, const int n_blocks, int *sem, const int sem_per_head) {
  const FwdArgs &f = a.f;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *k_s = smem;
  uint8_t *v_s = smem + kTileK;
  uint8_t *qd_s = smem + 2 * kTileK;           // [stage][Q | dO]
  uint8_t *pt_s = qd_s + ST * 2 * kChunk;      // [P high | P low | dS high | dS low], each [key][query]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA -> (key block, kv head, batch): key blocks fastest, so the CTAs of one
  // (batch, kv head) run together and share Q/dO in L2; lower key blocks (the
  // heaviest under a causal mask) are dispatched first.
  const int bid = blockIdx.x;
  const int nb = bid % n_blocks;
  const int kvh = (bid / n_blocks) % f.hkv;
  const int b = bid / (n_blocks * f.hkv);
  int q0, lq, k0, lk;
  if (!f.seqs.get(b, q0, lq, k0, lk, f.err)) return;
  const int key0 = nb * BN;
  if (key0 >= lk) return;
  const int g = f.hq / f.hkv;
  int c_lo, nch;
  chunk_range(nb, lq, lk, f.win_l, f.win_r, c_lo, nch);
  const int n_iter = g * nch;
  // deterministic mode: dQ comes from the query-stationary kernel instead
  const bool with_dq = !a.deterministic;

  if (threadIdx.x == 0) {
    mbar_init(&sh.kv_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&sh.qd_full[s], 1);
      mbar_init(&sh.qd_empty[s], 1);
    }
    mbar_init(&sh.sdp_full, 1);
    mbar_init(&sh.st_free, 256);
    mbar_init(&sh.pds_full, 256);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.mma_done[s], 1);
      mbar_init(&sh.dq_free[s], 128);
      mbar_init(&sh.grp_p[s], 128);
    }
    mbar_init(&sh.grp_q, 128);
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one() && n_iter > 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      mbar_expect_tx(&sh.kv_full, 2 * kTileK);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(k_s + c * BN * 128, &tk, &sh.kv_full, c * 64, kvh, k0 + key0);
        tma_load_3d(v_s + c * BN * 128, &tv, &sh.kv_full, c * 64, kvh, k0 + key0);
      }
      int issued = 0;
      for (int it = 0; it < n_iter; ++it) {
        const int st = it % ST;
        const int h = kvh * g + it / nch;
        const int row = q0 + (c_lo + it % nch) * BQ;
        if (!wait_bar(sh, &sh.qd_empty[st], ((it / ST) & 1) ^ 1, f.err)) break;
        mbar_expect_tx(&sh.qd_full[st], 2 * kChunk);
        uint8_t *dst = qd_s + st * 2 * kChunk;
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(dst + c * BQ * 128, &tq, &sh.qd_full[st], c * 64, h, row);
          tma_load_3d(dst + kChunk + c * BQ * 128, &tdo, &sh.qd_full[st], c * 64, h, row);
        }
        issued = it + 1;
      }
      if (*(volatile int *)&sh.abort) {
        int *noerr = nullptr;
        mbar_wait(&sh.kv_full, 0, noerr);
        for (int it = max(0, issued - ST); it < issued; ++it)
          mbar_wait(&sh.qd_full[it % ST], (it / ST) & 1, noerr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one() && n_iter > 0) {
      constexpr int ab = IsBf16<T>::v;
      constexpr uint32_t id_s = idesc_f16(128, BQ, ab, 0, 0);   // S^T, dP^T
      constexpr uint32_t id_kv = idesc_f16(128, D, ab, 0, 1);   // dV, dK (B = dO/Q, MN-major)
      constexpr uint32_t id_q = idesc_f16(128, BQ, ab, 1, 1);   // dQ^T (A = K^T, B = dS^T)
      const uint32_t k_addr = smem_u32(k_s), v_addr = smem_u32(v_s);
      const uint32_t qd_addr = smem_u32(qd_s), pt_addr = smem_u32(pt_s);
      // descriptor bases; every operand below is base + constant offset
      const uint64_t k_kd = smem_desc(k_addr, 16, 1024), v_kd = smem_desc(v_addr, 16, 1024);
      const uint64_t k_mn = smem_desc(k_addr, BN * 128, 1024);
      const uint64_t qd_k = smem_desc(qd_addr, 16, 1024), qd_mn = smem_desc(qd_addr, BQ * 128, 1024);
      const uint64_t pt_k = smem_desc(pt_addr, 16, 1024), pt_mn = smem_desc(pt_addr, BQ * 128, 1024);
      auto issue_sdp = [&](int it) -> bool {
        const int st = it % ST;
        if (!wait_bar(sh, &sh.qd_full[st], (it / ST) & 1, f.err)) return false;
        tc_fence_after();
        const uint32_t q_o = st * 2 * kChunk, do_o = q_o + kChunk;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk / 4) * (BN * 128) + (kk % 4) * 32;
          const uint32_t qo = (kk / 4) * (BQ * 128) + (kk % 4) * 32;
          mma_ss(tmem + kColS, desc_add(k_kd, ko), desc_add(qd_k, q_o + qo), id_s, kk > 0);
          mma_ss(tmem + kColDP, desc_add(v_kd, ko), desc_add(qd_k, do_o + qo), id_s, kk > 0);
        }
        mma_commit(&sh.sdp_full);
        return true;
      };
      bool ok = wait_bar(sh, &sh.kv_full, 0, f.err) && issue_sdp(0);
      for (int it = 0; ok && it < n_iter; ++it) {
        if (it + 1 < n_iter) {
          if (!wait_bar(sh, &sh.st_free, it & 1, f.err)) break;
          if (!issue_sdp(it + 1)) break;
        }
        const int buf = it & 1, st = it % ST;
        if (!wait_bar(sh, &sh.pds_full, it & 1, f.err)) break;
        tc_fence_after();
        const uint32_t q_o = st * 2 * kChunk, do_o = q_o + kChunk;
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          const uint64_t do_d = desc_add(qd_mn, do_o + kk * 16 * 128);
          const uint64_t q_d = desc_add(qd_mn, q_o + kk * 16 * 128);
          // dV += (P_high + P_low)^T dO,  dK += (dS_high + dS_low)^T Q
          mma_ss(tmem + kColDV, desc_add(pt_k, 0 * kPT + kk * 32), do_d, id_kv, acc);
          mma_ss(tmem + kColDV, desc_add(pt_k, 1 * kPT + kk * 32), do_d, id_kv, 1u);
          mma_ss(tmem + kColDK, desc_add(pt_k, 2 * kPT + kk * 32), q_d, id_kv, acc);
          mma_ss(tmem + kColDK, desc_add(pt_k, 3 * kPT + kk * 32), q_d, id_kv, 1u);
        }
        mma_commit(&sh.qd_empty[st]);  // Q and dO of this chunk are no longer read
        if (with_dq) {
          if (it >= 2 && !wait_bar(sh, &sh.dq_free[buf], ((it >> 1) - 1) & 1, f.err)) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ss(tmem + kColDQ + buf * BQ, desc_add(k_mn, kk * 16 * 128),
                   desc_add(pt_mn, 2 * kPT + kk * 16 * 128), id_q, kk > 0);
        }
        mma_commit(&sh.mma_done[buf]);
      }
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ P^T, dS^T
    const int sw = (warp - 2) >> 2;         // which half of the chunk's 64 queries
    const int tid = threadIdx.x - 64 - 128 * sw;
    const int j = 32 * (warp & 3) + lane;  // TMEM lane = key row of the block
    const int kj = key0 + j;
    const uint32_t row_t = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    int qlo, qhi;
    query_range(kj, lq, lk, f.win_l, f.win_r, qlo, qhi);
    if (kj >= lk) qhi = -1;
    const bool cap = f.softcap > 0.f;
    const float sl2 = f.scale * kLog2e, cap_in = cap ? f.scale / f.softcap : 0.f;
    bool ok = true;
    // thread tid < 32 fetches the LSE of query column 32*sw + tid of a chunk,
    // 32 <= tid < 64 its D; the fetch for iteration it+1 is issued during it
    auto fetch = [&](int it) -> float {
      if (it >= n_iter || tid >= 64) return 0.f;
      const int h = kvh * g + it / nch;
      const int i = (c_lo + it % nch) * BQ + 32 * sw + (tid & 31);
      if (i >= lq) return 0.f;
      const int64_t li = f.seqs.lse_index(b, h, q0, i);
      return tid < 32 ? f.lse[li] * kLog2e : a.dsum[li];
    };
    float next = fetch(0);
    for (int it = 0; it < n_iter; ++it) {
      const int buf = it & 1;
      const int i0 = (c_lo + it % nch) * BQ + 32 * sw;
      if (tid < 32)
        sh.lse2[sw][buf][tid] = next;
      else if (tid < 64)
        sh.dsum[sw][buf][tid - 32] = next;
      next = fetch(it + 1);
      mbar_arrive(&sh.grp_p[sw]);  // this half's LSE and D are in shared memory
      if (!wait_warp(sh, &sh.grp_p[sw], it & 1, f.err)) { ok = false; break; }
      if (!wait_warp(sh, &sh.sdp_full, it & 1, f.err)) { ok = false; break; }
      tc_fence_after();
      uint32_t su[32], du[32];
      tmem_ld32(row_t + kColS + 32 * sw, su);
      tmem_ld32(row_t + kColDP + 32 * sw, du);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&sh.st_free);
      // the MMAs of the previous chunk must be done reading the P/dS buffers
      if (it >= 1 && !wait_warp(sh, &sh.mma_done[(it - 1) & 1], ((it - 1) >> 1) & 1, f.err)) {
        ok = false;
        break;
      }
      // two halves of 16 columns: compute, split into high and low 16-bit
      // parts, store (each row is 128 bytes; this warpgroup owns 64 of them)
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        uint32_t w[4][8];  // [P high, P low, dS high, dS low][8 packed pairs]
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          float pv[2], dv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col = 16 * hv + e + u;
            const int i = i0 + col;
            const float s = __uint_as_float(su[col]);
            float x, dcap = 1.f;
            if (cap) {
              const float t = tanhf(s * cap_in);
              x = f.softcap * t * kLog2e;
              dcap = 1.f - t * t;
            } else {
              x = s * sl2;
            }
            const bool vis = i >= qlo && i <= qhi;
            const float p = vis ? ex2(x - sh.lse2[sw][buf][col]) : 0.f;
            pv[u] = p;
            dv[u] = p * (__uint_as_float(du[col]) - sh.dsum[sw][buf][col]) * dcap;
          }
          split_hi_lo<T>(pv, w[0][e / 2], w[1][e / 2]);
          split_hi_lo<T>(dv, w[2][e / 2], w[3][e / 2]);
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int chunk = 4 * sw + 2 * hv + cc;  // 16-byte chunk of the 128-byte row
            const uint32_t off = j * 128 + ((chunk ^ (j & 7)) << 4);
            *reinterpret_cast<uint4 *>(pt_s + m * kPT + off) =
                make_uint4(w[m][4 * cc], w[m][4 * cc + 1], w[m][4 * cc + 2], w[m][4 * cc + 3]);
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&sh.pds_full);
    }
    // dK, dV out of TMEM: each warpgroup writes half of the head-dim columns
    if (ok && n_iter > 0)
      ok = wait_warp(sh, &sh.mma_done[(n_iter - 1) & 1], ((n_iter - 1) >> 1) & 1, f.err);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    // tcgen05.ld is warp-collective: every lane loads, only real keys store
    if (ok) {
      const int64_t off = ((int64_t)(k0 + kj) * f.hkv + kvh) * D;
      T *dvr = static_cast<T *>(a.dv) + off;
      T *dkr = static_cast<T *>(a.dk) + off;
#pragma unroll 1
      for (int c = 2 * sw; c < 2 * sw + 2; ++c) {
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          uint32_t u[32];
          if (n_iter > 0) {
            tmem_ld32(row_t + (which ? kColDK : kColDV) + c * 32, u);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = 0u;
          }
          const float sc = which ? f.scale : 1.f;
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = Elem<T>::from_f2(__uint_as_float(u[2 * e]) * sc, __uint_as_float(u[2 * e + 1]) * sc);
          if (kj < lk) {
            uint4 *dst = reinterpret_cast<uint4 *>((which ? dkr : dvr) + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
        }
      }
    }
  } else if (!with_dq) {
    // dQ warpgroup idle: the query-stationary kernel computes dQ
  } else {
    // ------------------------------------------------------------ dQ
    const int tid = threadIdx.x - 320;
    const int dl = 32 * (warp & 3) + lane;  // TMEM lane = head-dim column
    const uint32_t row_t = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    uint32_t grp_phase = 0;
    auto group_sync = [&]() -> bool {
      mbar_arrive(&sh.grp_q);
      return wait_warp(sh, &sh.grp_q, (grp_phase++) & 1, f.err);
    };
    for (int it = 0; it < n_iter; ++it) {
      const int buf = it & 1;
      const int h = kvh * g + it / nch;
      const int c = c_lo + it % nch;
      const int i0 = c * BQ;
      if (!wait_warp(sh, &sh.mma_done[buf], (it >> 1) & 1, f.err)) break;
      tc_fence_after();
      uint32_t u[BQ];
      tmem_ld32(row_t + kColDQ + buf * BQ, *reinterpret_cast<uint32_t(*)[32]>(u));
      tmem_ld32(row_t + kColDQ + buf * BQ + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&sh.dq_free[buf]);
      int *turn_ctr = nullptr;
      if (a.deterministic) {
        // key blocks below this one that also add into chunk c go first
        turn_ctr = sem + (int64_t)h * sem_per_head + (q0 / BQ + b) + c;
        if (tid == 0) {
          int turn = 0;
          for (int nb2 = 0; nb2 < nb; ++nb2) {
            int cl, nc;
            chunk_range(nb2, lq, lk, f.win_l, f.win_r, cl, nc);
            turn += (c >= cl && c < cl + nc) ? 1 : 0;
          }
          const uint64_t t0 = globaltimer();
          int seen;
          for (uint32_t spin = 0;; ++spin) {
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(turn_ctr) : "memory");
            if (seen >= turn) break;
            if ((spin & 63) == 63 && (globaltimer() - t0 > kWaitLimitNs || *(volatile int *)&sh.abort)) {
              raise_error(f.err, kErrTimeout);
              *(volatile int *)&sh.abort = 1;
              break;
            }
          }
        }
        if (!group_sync()) break;  // thread 0 has seen this key block's turn
      }
      float *acc = a.dq_acc + ((int64_t)(q0 + i0) * f.hq + h) * D + dl;
      const int rows = min(BQ, lq - i0);
#pragma unroll
      for (int e = 0; e < BQ; ++e)
        if (e < rows) red_add(acc + (int64_t)e * f.hq * D, __uint_as_float(u[e]));
      if (a.deterministic) {
        __threadfence();
        if (!group_sync()) break;  // every add of this key block is performed
        if (tid == 0) atomicAdd(turn_ctr, 1);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// D_i = rowsum(dO_i * O_i) (fp32, LSE layout); zero the dQ accumulator and
// the turn counters.  One warp per (row, head).
template <typename T>
__global__ void __launch_bounds__(256) bwd_prep_kernel(BwdArgs a, int *sem, int64_t sem_count,
                                                       int64_t rows) {
  const FwdArgs &f = a.f;
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t x = w; x < rows * f.hq; x += nw) {
    const int64_t row = x / f.hq;
    const int h = (int)(x % f.hq);
    const int64_t off = x * D + lane * 4;
    float o[4], g[4];
    load_vec<T, 4>(static_cast<const T *>(f.o) + off, o);
    load_vec<T, 4>(static_cast<const T *>(a.dout) + off, g);
    float s = o[0] * g[0] + o[1] * g[1] + o[2] * g[2] + o[3] * g[3];
    s = warp_sum(s);
    if (!a.deterministic)
      reinterpret_cast<float4 *>(a.dq_acc + off)[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane == 0) {
      int64_t li;
      if (f.seqs.cu_q) {
        li = (int64_t)h * f.seqs.total_q + row;
      } else {
        const int64_t bb = row / f.seqs.sq, i = row % f.seqs.sq;
        li = (bb * f.hq + h) * f.seqs.sq + i;
      }
      a.dsum[li] = s;
    }
  }
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t x = t; x < sem_count; x += (int64_t)gridDim.x * blockDim.x) sem[x] = 0;
}

// dQ = scale * dQ_acc -> dtype.
template <typename T>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(BwdArgs a, int64_t n4) {
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n4;
       x += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = reinterpret_cast<const float4 *>(a.dq_acc)[x];
    const float s = a.f.scale;
    uint2 out{Elem<T>::from_f2(v.x * s, v.y * s), Elem<T>::from_f2(v.z * s, v.w * s)};
    reinterpret_cast<uint2 *>(a.dq)[x] = out;
  }
}

template <typename T>
cudaError_t bwd_tc(const BwdArgs &a, int *sem, int sem_per_head, int sms, cudaStream_t st) {
  const FwdArgs &f = a.f;
  const int64_t rows_q = f.seqs.cu_q ? f.seqs.total_q : (int64_t)f.batch * f.seqs.sq;
  const int64_t rows_k = f.seqs.cu_k ? f.seqs.total_k : (int64_t)f.batch * f.seqs.sk;
  const int64_t sem_count = (int64_t)sem_per_head * f.hq;
  const int prep_blocks = (int)std::min<int64_t>((rows_q * f.hq + 7) / 8, (int64_t)sms * 16);
  if (rows_q > 0) {
    bwd_prep_kernel<T><<<std::max(prep_blocks, 1), 256, 0, st>>>(a, sem, sem_count, rows_q);
    count_launches(1);
  }
  if (rows_k > 0 && rows_q > 0) {
    CUtensorMap tq, tk, tv, tdo;
    if (!make_map_3d(&tq, f.q, f.dtype, rows_q, f.hq, D, BQ) ||
        !make_map_3d(&tdo, a.dout, f.dtype, rows_q, f.hq, D, BQ) ||
        !make_map_3d(&tk, f.k, f.dtype, rows_k, f.hkv, D, BN) ||
        !make_map_3d(&tv, f.v, f.dtype, rows_k, f.hkv, D, BN))
      return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    const int n_blocks = (f.seqs.sk + BN - 1) / BN;
    const int64_t grid = (int64_t)n_blocks * f.hkv * f.batch;
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
    bwd_tc_kernel<T><<<(unsigned)grid, kThreads, kSmem, st>>>(tq, tk, tv, tdo, a, n_blocks, sem,
                                                              sem_per_head);
    count_launches(1);
  } else if (rows_k > 0) {  // no queries: the key gradients are zero
    const size_t bytes = (size_t)rows_k * f.hkv * D * 2;
    cudaError_t e = cudaMemsetAsync(a.dk, 0, bytes, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dv, 0, bytes, st);
    if (e != cudaSuccess) return e;
  }
  if (a.deterministic) {
    // dQ from the query-stationary kernel: no atomics, the same bits every run
    cudaError_t e = launch_bwd_dq_tc(a, st);
    if (e != cudaSuccess) return e;
  } else if (rows_q > 0) {
    const int64_t n4 = rows_q * f.hq * D / 4;
    const int blocks = (int)std::min<int64_t>((n4 + 255) / 256, (int64_t)sms * 16);
    bwd_dq_convert_kernel<T><<<std::max(blocks, 1), 256, 0, st>>>(a, n4);
    count_launches(1);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdArgs &a, int *sem, int sem_per_head, int sms,
                          cudaStream_t st) {
  if (a.f.d != D) return cudaErrorInvalidValue;
  return a.f.dtype == ATTN_BF16 ? bwd_tc<__nv_bfloat16>(a, sem, sem_per_head, sms, st)
                                : bwd_tc<__half>(a, sem, sem_per_head, sms, st);
}

}  // namespace attn
