// dQ of the backward, query-stationary, on the tensor cores (sm_103a), d = 128.
//
// dQ_i = scale * sum_j dS_ij k_j with dS = P * (dP - D), P = exp(s - LSE),
// dP = dO V^T ("FlashAttention完整说明" §二.2: S and P are recomputed from
// Q, K and the saved LSE).  A CTA owns two 128-row query tiles of one
// (batch, head) and walks the 64-key tiles they can see; dQ stays in TMEM
// for the whole walk and is written once, so no atomics are needed and the
// result is the same bit for bit on every run (Inference Cookbook FAQ Q11).
//
//   warpgroup 0   warp 0: TMA (Q, dO of both tiles once; K, V tiles into a
//                 3-stage ring); warp 1: MMA issuer and TMEM owner.
//   warpgroups 1, 2   one per query tile, one thread per query row: P and dS
//                 from S and dP (TMEM), dS (fp16/bf16) written back into the
//                 S columns as the A operand of dQ += dS K.
//
// TMEM (512 columns): S_0 [0,64), S_1 [64,128), dP_0 [128,192),
// dP_1 [192,256), dQ_0 [256,384), dQ_1 [384,512).  The MMA warp alternates
// between the tiles, so one tile's P/dS work overlaps the other's MMAs.
#include <cudaTypedefs.h>

#include "kernels.h"
#include "sm103.cuh"

namespace attn {
namespace {
using namespace sm103;

constexpr int D = 128;
constexpr int BM = 128;  // query rows per tile
constexpr int NT = 2;    // query tiles per CTA
constexpr int BN = 64;   // keys per step
constexpr int ST = 3;
constexpr int kThreads = 384;
constexpr int kQBytes = BM * D * 2;    // 32 KB, one tile of Q (and of dO)
constexpr int kKVBytes = BN * D * 2;   // 16 KB
constexpr int kSmemData = 2 * NT * kQBytes + 2 * ST * kKVBytes;  // 224 KB
constexpr int kSmem = kSmemData + 1024;
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;

struct Shared {
  uint64_t q_full;
  uint64_t kv_full[ST], kv_empty[ST];
  uint64_t s_full[NT], ds_full[NT], dq_done[NT];
  uint64_t all_done;  // every MMA of the CTA has completed
  uint64_t wait_ns;   // wall-clock limit of a wait
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool wait_bar(Shared &sh, uint64_t *bar, uint32_t parity, int *err) {
  return mbar_wait_bounded(smem_u32(bar), parity, &sh.abort, err, sh.wait_ns);
}

__device__ __forceinline__ bool wait_warp(Shared &sh, uint64_t *bar, uint32_t parity, int *err) {
  return __all_sync(0xffffffffu, wait_bar(sh, bar, parity, err));
}

template <typename T> struct IsBf16 { static constexpr int v = 0; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr int v = 1; };

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const BwdArgs a, const int m_blocks) {
  const FwdArgs &f = a.f;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *q_s = smem;                      // [tile] 32 KB each
  uint8_t *do_s = smem + NT * kQBytes;      // [tile]
  uint8_t *k_s = do_s + NT * kQBytes;       // [stage] 16 KB
  uint8_t *v_s = k_s + ST * kKVBytes;       // [stage]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA -> (query block, batch, head): heaviest blocks first, heads fastest
  const int bid = blockIdx.x;
  const int h = bid % f.hq;
  const int b = (bid / f.hq) % f.batch;
  const int mb = m_blocks - 1 - bid / (f.hq * f.batch);
  int q0, lq, k0, lk;
  if (!f.seqs.get(b, q0, lq, k0, lk, f.err)) return;
  const int m0 = mb * (BM * NT);
  if (m0 >= lq) return;
  const int kvh = h / (f.hq / f.hkv);
  const int m_last = min(m0 + BM * NT, lq) - 1;
  int lo_first, hi_first, lo_last, hi_last;
  key_range(m0, lq, lk, f.win_l, f.win_r, lo_first, hi_first);
  key_range(m_last, lq, lk, f.win_l, f.win_r, lo_last, hi_last);
  int n_lo = 0, nt = 0;
  if (hi_last >= lo_first && hi_last >= 0) {
    n_lo = lo_first / BN;
    nt = hi_last / BN - n_lo + 1;
  }

  if (threadIdx.x == 0) {
    mbar_init(&sh.q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&sh.kv_full[s], 1);
      mbar_init(&sh.kv_empty[s], 1);
    }
    for (int t = 0; t < NT; ++t) {
      mbar_init(&sh.s_full[t], 1);
      mbar_init(&sh.ds_full[t], BM);
      mbar_init(&sh.dq_done[t], 1);
    }
    mbar_init(&sh.all_done, 1);
    sh.wait_ns = f.wait_ns;
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
  // launched at 168 registers a thread (12 warps); 128 * 112 + 256 * 192 <= 384 * 168
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      if (elect_one() && nt > 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        prefetch_tmap(&tdo);
        mbar_expect_tx(&sh.q_full, 2 * NT * kQBytes);
        for (int t = 0; t < NT; ++t)
          for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(q_s + t * kQBytes + c * BM * 128, &tq, &sh.q_full, c * 64, h,
                        q0 + m0 + t * BM);
            tma_load_3d(do_s + t * kQBytes + c * BM * 128, &tdo, &sh.q_full, c * 64, h,
                        q0 + m0 + t * BM);
          }
        int issued = 0;
        for (int j = 0; j < nt; ++j) {
          const int st = j % ST;
          const int krow = k0 + (n_lo + j) * BN;
          if (!wait_bar(sh, &sh.kv_empty[st], ((j / ST) & 1) ^ 1, f.err)) break;
          mbar_expect_tx(&sh.kv_full[st], 2 * kKVBytes);
          for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(k_s + st * kKVBytes + c * BN * 128, &tk, &sh.kv_full[st], c * 64, kvh, krow);
            tma_load_3d(v_s + st * kKVBytes + c * BN * 128, &tv, &sh.kv_full[st], c * 64, kvh, krow);
          }
          issued = j + 1;
        }
        if (*(volatile int *)&sh.abort) {
          int *noerr = nullptr;
          mbar_wait(&sh.q_full, 0, noerr);
          for (int j = max(0, issued - ST); j < issued; ++j)
            mbar_wait(&sh.kv_full[j % ST], (j / ST) & 1, noerr);
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (elect_one() && nt > 0) {
        constexpr int ab = IsBf16<T>::v;
        constexpr uint32_t id_s = idesc_f16(BM, BN, ab, 0, 0);  // S, dP (K-major A and B)
        constexpr uint32_t id_q = idesc_f16(BM, D, ab, 0, 1);   // dQ (A = dS in TMEM, B = K MN-major)
        const uint64_t q_d = smem_desc(smem_u32(q_s), 16, 1024);
        const uint64_t do_d = smem_desc(smem_u32(do_s), 16, 1024);
        const uint64_t k_d = smem_desc(smem_u32(k_s), 16, 1024);
        const uint64_t v_d = smem_desc(smem_u32(v_s), 16, 1024);
        const uint64_t k_mn = smem_desc(smem_u32(k_s), BN * 128, 1024);
        auto mma_sdp = [&](int t, int j) {
          const uint32_t ko = (j % ST) * kKVBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qo = t * kQBytes + (kk / 4) * (BM * 128) + (kk % 4) * 32;
            const uint32_t kvo = ko + (kk / 4) * (BN * 128) + (kk % 4) * 32;
            mma_ss(tmem + kColS + t * BN, desc_add(q_d, qo), desc_add(k_d, kvo), id_s, kk > 0);
            mma_ss(tmem + kColDP + t * BN, desc_add(do_d, qo), desc_add(v_d, kvo), id_s, kk > 0);
          }
          mma_commit(&sh.s_full[t]);
        };
        auto mma_dq = [&](int t, int j) {
          const uint32_t ko = (j % ST) * kKVBytes;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + kColDQ + t * D, tmem + kColS + t * BN + kk * 8,
                   desc_add(k_mn, ko + kk * 16 * 128), id_q, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&sh.dq_done[t]);
        };
        // test hook: all_done completes only after this thread's last
        // commit, so this wait can only run out
        bool ok = !(f.stall && !wait_bar(sh, &sh.all_done, 0, f.err));
        ok = ok && wait_bar(sh, &sh.q_full, 0, f.err) && wait_bar(sh, &sh.kv_full[0], 0, f.err);
        tc_fence_after();
        if (ok)
          for (int t = 0; t < NT; ++t) mma_sdp(t, 0);
        // S_0, dP_0, S_1, dP_1 | dQ_0(j) S_0/dP_0(j+1) dQ_1(j) S_1/dP_1(j+1) | ...
        for (int j = 0; ok && j < nt; ++j) {
          for (int t = 0; t < NT; ++t) {
            if (!wait_bar(sh, &sh.ds_full[t], j & 1, f.err)) { ok = false; break; }
            tc_fence_after();
            mma_dq(t, j);
            if (t == NT - 1) mma_commit(&sh.kv_empty[j % ST]);
            if (j + 1 < nt) {
              if (t == 0) {
                if (!wait_bar(sh, &sh.kv_full[(j + 1) % ST], ((j + 1) / ST) & 1, f.err)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              mma_sdp(t, j + 1);
            }
          }
        }
        // after an abort, no MMA may still run when the TMEM is released
        mma_commit(&sh.all_done);
        if (*(volatile int *)&sh.abort) {
          int *noerr = nullptr;
          mbar_wait(&sh.all_done, 0, noerr);
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    // ------------------------------------------------------------ P, dS
    const int t = (warp - 4) >> 2;
    const int r = 32 * (warp & 3) + lane;  // TMEM lane = query row of the tile
    const int i = m0 + t * BM + r;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    int lo_i, hi_i;
    key_range(i, lq, lk, f.win_l, f.win_r, lo_i, hi_i);
    int lo_tile_max, hi_tile_min, dummy;
    key_range(m0 + t * BM + BM - 1, lq, lk, f.win_l, f.win_r, lo_tile_max, dummy);
    key_range(m0 + t * BM, lq, lk, f.win_l, f.win_r, dummy, hi_tile_min);
    const bool valid = i < lq;
    const int64_t li = f.seqs.lse_index(b, h, q0, valid ? i : 0);
    const float nlse2 = valid ? a.nlse2[li] : 0.f;  // -LSE * log2(e)
    const float dsum = valid ? a.dsum[li] : 0.f;
    const bool cap = f.softcap > 0.f;
    const float sl2 = f.scale * kLog2e, cap_in = cap ? f.scale / f.softcap : 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int key0 = (n_lo + j) * BN;
      if (!wait_warp(sh, &sh.s_full[t], j & 1, f.err)) { ok = false; break; }
      tc_fence_after();
      uint32_t su[BN], du[BN];
      tmem_ld32(lane_off + tmem + kColS + t * BN, *reinterpret_cast<uint32_t(*)[32]>(su));
      tmem_ld32(lane_off + tmem + kColS + t * BN + 32, *reinterpret_cast<uint32_t(*)[32]>(su + 32));
      tmem_ld32(lane_off + tmem + kColDP + t * BN, *reinterpret_cast<uint32_t(*)[32]>(du));
      tmem_ld32(lane_off + tmem + kColDP + t * BN + 32, *reinterpret_cast<uint32_t(*)[32]>(du + 32));
      tmem_wait_ld();
      const bool need_mask = !valid || key0 < lo_tile_max || key0 + BN - 1 > hi_tile_min;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int e = 0; e < BN; e += 2) {
        float ds[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int col = e + u;
          const float s = __uint_as_float(su[col]);
          float p, dcap = 1.f;
          if (cap) {
            const float tt = tanh_fast(s * cap_in);
            p = ex2(fmaf(f.softcap * kLog2e, tt, nlse2));
            dcap = 1.f - tt * tt;
          } else {
            p = ex2(fmaf(s, sl2, nlse2));
          }
          if (need_mask) {
            const int kj = key0 + col;
            if (!valid || kj < lo_i || kj > hi_i) p = 0.f;
          }
          ds[u] = p * (__uint_as_float(du[col]) - dsum) * dcap;
        }
        pk[e / 2] = Elem<T>::from_f2(ds[0], ds[1]);
      }
      // dS (16-bit) over the first BN/2 columns of S: the A operand of dQ += dS K
      tmem_st16(lane_off + tmem + kColS + t * BN, pk);
      tmem_st16(lane_off + tmem + kColS + t * BN + 16, pk + 16);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sh.ds_full[t]);
    }
    // epilogue: dQ = scale * accumulated dS K
    if (ok && nt > 0) ok = wait_warp(sh, &sh.dq_done[t], (nt - 1) & 1, f.err);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
      T *row = static_cast<T *>(a.dq) + (int64_t)(q0 + (valid ? i : 0)) * a.dq_rs + (int64_t)h * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        if (nt > 0) {
          tmem_ld32(lane_off + tmem + kColDQ + t * D + c * 32, u);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = Elem<T>::from_f2(__uint_as_float(u[2 * e]) * f.scale,
                                  __uint_as_float(u[2 * e + 1]) * f.scale);
        if (valid) {
          uint4 *dst = reinterpret_cast<uint4 *>(row + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <typename T>
cudaError_t bwd_dq(const BwdArgs &a, cudaStream_t st) {
  const FwdArgs &f = a.f;
  const int64_t rows_q = f.seqs.cu_q ? f.seqs.total_q : (int64_t)f.batch * f.seqs.sq;
  const int64_t rows_k = f.seqs.cu_k ? f.seqs.total_k : (int64_t)f.batch * f.seqs.sk;
  if (rows_q == 0) return cudaSuccess;
  if (rows_k == 0)
    return cudaMemset2DAsync(a.dq, (size_t)a.dq_rs * 2, 0, (size_t)f.hq * D * 2, (size_t)rows_q, st);
  CUtensorMap tq, tk, tv, tdo;
  if (!make_map_3d(&tq, f.q, f.dtype, rows_q, f.hq, D, BM, f.q_rs) ||
      !make_map_3d(&tdo, a.dout, f.dtype, rows_q, f.hq, D, BM) ||
      !make_map_3d(&tk, f.k, f.dtype, rows_k, f.hkv, D, BN, f.k_rs) ||
      !make_map_3d(&tv, f.v, f.dtype, rows_k, f.hkv, D, BN, f.v_rs))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_once<bwd_dq_kernel<T>>(kSmem);
  if (e != cudaSuccess) return e;
  const int m_blocks = (f.seqs.sq + BM * NT - 1) / (BM * NT);
  const int64_t grid = (int64_t)m_blocks * f.hq * f.batch;
  if (grid == 0) return cudaSuccess;
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  debug_log("backward dQ (deterministic): bwd_dq_kernel d=128, %d query tiles of %d rows per "
            "CTA, %d-key tiles, grid=%lld CTAs x %d threads, smem=%d B", NT, BM, BN,
            (long long)grid, kThreads, kSmem);
  bwd_dq_kernel<T><<<(unsigned)grid, kThreads, kSmem, st>>>(tq, tk, tv, tdo, a, m_blocks);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_tc(const BwdArgs &a, cudaStream_t st) {
  if (a.f.d != D) return cudaErrorInvalidValue;
  return a.f.dtype == ATTN_BF16 ? bwd_dq<__nv_bfloat16>(a, st) : bwd_dq<__half>(a, st);
}

}  // namespace attn
