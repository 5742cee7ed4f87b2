// dQ of the backward, query-stationary, on the tensor cores (sm_103a), d = 64,
// 128 or 256.
//
// dQ_i = scale * sum_j dS_ij k_j with dS = P * (dP - D), P = exp(s - LSE),
// dP = dO V^T ("FlashAttention完整说明" §二.2: S and P are recomputed from
// Q, K and the saved LSE).  A CTA owns one 128-row query tile of one (batch,
// head) and walks the 128-key tiles it can see; dQ stays in TMEM for the
// whole walk and is written once, so no atomics are needed and the result is
// the same bit for bit on every run (Inference Cookbook FAQ Q11).
//
//   warp 0        TMA producer: Q and dO of the tile once; K tiles into a
//                 3-stage ring, V tiles into a 2-stage ring (a V tile is
//                 released as soon as its dP product is done, a K tile only
//                 after its dQ product).
//   warp 1        MMA issuer and TMEM owner.
//   warpgroups    one thread per query row; warpgroup w takes keys
//   1 and 2       [64 w, 64 w + 64) of every key tile: P and dS from S and dP
//                 (TMEM), dS (fp16/bf16) written back over its own S columns
//                 as the A operand of dQ += dS K.  At the end warpgroup w
//                 writes dQ columns [64 w, 64 w + 64).
//
// TMEM (512 columns): S of key tile j in buffer j % 2 at [0,128) / [128,256),
// dP at [256,384), dQ at [384,512).  Issue order: S(0) dP(0) S(1) |
// dP(j+1) once both warpgroups have read dP(j); dQ(j) once dS(j) is written;
// S(j+2) into the buffer dQ(j) reads, behind it in issue order.  So while the
// softmax works on tile j the tensor pipe runs dQ(j-1), S(j+1) and dP(j+1).
//
// d = 256: Q and dO of the tile take 128 KB, so keys come in steps of 64
// (K and V tiles of 32 KB; 2 K stages, 1 V stage) and each CTA produces one
// 128-column half of dQ (two CTAs per query tile, each recomputing S and
// dP).  TMEM: S buffers at [0,64) / [64,128), dP at [128,192), dQ at
// [192,320).
#include <cudaTypedefs.h>

#include "kernels.h"
#include "sm103.cuh"

namespace attn {
namespace {
using namespace sm103;

constexpr int BM = 128;  // query rows per CTA
constexpr int kThreads = 384;

// Tile shape for head dimension D (64, 128 or 256).
template <int D>
struct DqCfg {
  static constexpr int BN = D == 256 ? 64 : 128;   // keys per step
  static constexpr int KST = D == 256 ? 2 : 3;     // K ring stages
  static constexpr int VST = D == 256 ? 1 : 2;     // V ring stages
  static constexpr int DO = D < 128 ? D : 128;     // dQ columns of one CTA
  static constexpr int NH = D / DO;                // CTAs per query tile
  static constexpr uint32_t kColS = 0, kColDP = 2 * BN, kColDQ = 3 * BN;
  static constexpr int kQTile = BM * D * 2;        // Q or dO of the tile: 32 KB at d = 128
  static constexpr int kKTile = BN * D * 2;        // one K or V tile
  static constexpr int kSmemData = 2 * kQTile + (KST + VST) * kKTile;  // 224 KB at d = 128, 256
  static constexpr int kSmem = kSmemData + 1024;
  static_assert(kSmem <= 227 * 1024 - 1024, "shared memory");
  static_assert(kColDQ + DO <= 512, "TMEM");
};

template <int KST, int VST>
struct Shared {
  uint64_t q_full;
  uint64_t k_full[KST], k_empty[KST], v_full[VST], v_empty[VST];
  uint64_t s_full[2];  // S(j) of buffer j % 2 is in TMEM
  uint64_t dp_full;    // dP(j) is in TMEM
  uint64_t dp_free;    // both warpgroups have read dP(j)
  uint64_t ds_full[2]; // dS(j) is written over its S columns
  uint64_t all_done;   // every MMA of the CTA has completed
  uint64_t wait_ns;    // wall-clock limit of a wait
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename Sh>
__device__ __forceinline__ bool wait_bar(Sh &sh, uint64_t *bar, uint32_t parity, int *err) {
  return mbar_wait_bounded(smem_u32(bar), parity, &sh.abort, err, sh.wait_ns);
}

template <typename Sh>
__device__ __forceinline__ bool wait_warp(Sh &sh, uint64_t *bar, uint32_t parity, int *err) {
  return __all_sync(0xffffffffu, wait_bar(sh, bar, parity, err));
}

template <typename T> struct IsBf16 { static constexpr int v = 0; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr int v = 1; };

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const BwdArgs a, const int m_blocks) {
  using C = DqCfg<D>;
  constexpr int BN = C::BN, KST = C::KST, VST = C::VST, DO = C::DO;
  constexpr int kQTile = C::kQTile, kKTile = C::kKTile;
  constexpr uint32_t kColS = C::kColS, kColDP = C::kColDP, kColDQ = C::kColDQ;
  const FwdArgs &f = a.f;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared<KST, VST> sh;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *q_s = smem;
  uint8_t *do_s = smem + kQTile;
  uint8_t *k_s = smem + 2 * kQTile;       // [KST]
  uint8_t *v_s = k_s + KST * kKTile;      // [VST]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA -> (column half, query block, batch, head): heaviest blocks first,
  // heads fastest; dh selects the dQ columns [dh DO, dh DO + DO)
  const int dh = blockIdx.x % C::NH;
  const int bid = blockIdx.x / C::NH;
  const int h = bid % f.hq;
  const int b = (bid / f.hq) % f.batch;
  const int mb = m_blocks - 1 - bid / (f.hq * f.batch);
  int q0, lq, k0, lk;
  if (!f.seqs.get(b, q0, lq, k0, lk, f.err)) return;
  const int m0 = mb * BM;
  if (m0 >= lq) return;
  const int kvh = h / (f.hq / f.hkv);
  const int m_last = min(m0 + BM, lq) - 1;
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
    for (int s = 0; s < KST; ++s) {
      mbar_init(&sh.k_full[s], 1);
      mbar_init(&sh.k_empty[s], 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(&sh.v_full[s], 1);
      mbar_init(&sh.v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.s_full[s], 1);
      mbar_init(&sh.ds_full[s], 8);  // warps
    }
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.dp_free, 8);       // warps
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
  // launched at 168 registers a thread (12 warps); 128 * 88 + 256 * 208 = 384 * 168
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      if (elect_one() && nt > 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        prefetch_tmap(&tdo);
        mbar_expect_tx(&sh.q_full, 2 * kQTile);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(q_s + c * BM * 128, &tq, &sh.q_full, c * 64, h, q0 + m0);
          tma_load_3d(do_s + c * BM * 128, &tdo, &sh.q_full, c * 64, h, q0 + m0);
        }
        int k_issued = 0, v_issued = 0;
        for (int j = 0; j < nt; ++j) {
          const int krow = k0 + (n_lo + j) * BN;
          const int ks = j % KST, vs = j % VST;
          if (!wait_bar(sh, &sh.k_empty[ks], ((j / KST) & 1) ^ 1, f.err)) break;
          mbar_expect_tx(&sh.k_full[ks], kKTile);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(k_s + ks * kKTile + c * BN * 128, &tk, &sh.k_full[ks], c * 64, kvh, krow);
          k_issued = j + 1;
          if (!wait_bar(sh, &sh.v_empty[vs], ((j / VST) & 1) ^ 1, f.err)) break;
          mbar_expect_tx(&sh.v_full[vs], kKTile);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(v_s + vs * kKTile + c * BN * 128, &tv, &sh.v_full[vs], c * 64, kvh, krow);
          v_issued = j + 1;
        }
        if (*(volatile int *)&sh.abort) {
          // let this CTA's copies in flight land before the CTA exits
          int *noerr = nullptr;
          mbar_wait(&sh.q_full, 0, noerr);
          for (int j = max(0, k_issued - KST); j < k_issued; ++j)
            mbar_wait(&sh.k_full[j % KST], (j / KST) & 1, noerr);
          for (int j = max(0, v_issued - VST); j < v_issued; ++j)
            mbar_wait(&sh.v_full[j % VST], (j / VST) & 1, noerr);
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (elect_one() && nt > 0) {
        constexpr int ab = IsBf16<T>::v;
        constexpr uint32_t id_s = idesc_f16(BM, BN, ab, 0, 0);  // S, dP (K-major A and B)
        constexpr uint32_t id_q = idesc_f16(BM, DO, ab, 0, 1);  // dQ (A = dS in TMEM, B = K MN-major)
        const uint64_t q_d = smem_desc(smem_u32(q_s), 16, 1024);
        const uint64_t do_d = smem_desc(smem_u32(do_s), 16, 1024);
        const uint64_t k_d = smem_desc(smem_u32(k_s), 16, 1024);
        const uint64_t v_d = smem_desc(smem_u32(v_s), 16, 1024);
        // K as dQ's B operand: this CTA's column half (64-column blocks 2 dh, 2 dh + 1)
        const uint64_t k_mn = smem_desc(smem_u32(k_s) + dh * 2 * (BN * 128), BN * 128, 1024);
        // X (Q or dO) times the key tile's K or V rows, K = d
        // (at d = 256 one 64-column block of d per outer step, not unrolled:
        // 16 unrolled steps would keep too many descriptors live)
        auto mma_xk = [&](uint32_t dcol, uint64_t a_d, uint64_t b_d, uint32_t b_off) {
          if constexpr (D == 256) {
#pragma unroll 1
            for (int cb = 0; cb < D / 64; ++cb) {
              const uint64_t ab = desc_add(a_d, cb * (BM * 128));
              const uint64_t bb = desc_add(b_d, b_off + cb * (BN * 128));
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4)
                mma_ss(dcol, desc_add(ab, k4 * 32), desc_add(bb, k4 * 32), id_s, (cb | k4) > 0);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t oa = (kk / 4) * (BM * 128) + (kk % 4) * 32;
              const uint32_t ob = (kk / 4) * (BN * 128) + (kk % 4) * 32;
              mma_ss(dcol, desc_add(a_d, oa), desc_add(b_d, b_off + ob), id_s, kk > 0);
            }
          }
        };
        auto k_ready = [&](int j) {
          const bool r = wait_bar(sh, &sh.k_full[j % KST], (j / KST) & 1, f.err);
          tc_fence_after();
          return r;
        };
        auto v_ready = [&](int j) {
          const bool r = wait_bar(sh, &sh.v_full[j % VST], (j / VST) & 1, f.err);
          tc_fence_after();
          return r;
        };
        auto issue_s = [&](int j) {  // S(j) = Q K_j^T into buffer j % 2
          mma_xk(tmem + kColS + (j & 1) * BN, q_d, k_d, (j % KST) * kKTile);
          mma_commit(&sh.s_full[j & 1]);
        };
        auto issue_dp = [&](int j) {  // dP(j) = dO V_j^T
          mma_xk(tmem + kColDP, do_d, v_d, (j % VST) * kKTile);
          mma_commit(&sh.dp_full);
          mma_commit(&sh.v_empty[j % VST]);  // V_j is no longer read
        };
        // test hook: all_done completes only after this thread's last
        // commit, so this wait can only run out
        bool ok = !(f.stall && !wait_bar(sh, &sh.all_done, 0, f.err));
        ok = ok && wait_bar(sh, &sh.q_full, 0, f.err) && k_ready(0);
        if (ok) issue_s(0);
        ok = ok && v_ready(0);
        if (ok) issue_dp(0);
        if (ok && nt > 1 && (ok = k_ready(1))) issue_s(1);
        for (int j = 0; ok && j < nt; ++j) {
          if (j + 1 < nt) {
            // dP(j+1) overwrites dP(j): both warpgroups must have read it
            if (!wait_bar(sh, &sh.dp_free, j & 1, f.err) || !v_ready(j + 1)) break;
            issue_dp(j + 1);
          }
          if (!wait_bar(sh, &sh.ds_full[j & 1], (j >> 1) & 1, f.err)) break;
          tc_fence_after();
          // dQ += dS(j) K_j: A = dS (warpgroup w's BN/2 keys packed at the
          // buffer's columns BN/2 w + [0, BN/4)), B = K_j with d as N
          const uint32_t sbuf = tmem + kColS + (j & 1) * BN;
          const uint32_t ko = (j % KST) * kKTile;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + kColDQ, sbuf + (BN / 2) * (16 * kk / (BN / 2)) + 8 * ((16 * kk % (BN / 2)) / 16),
                   desc_add(k_mn, ko + kk * 16 * 128), id_q, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&sh.k_empty[j % KST]);  // K_j is no longer read
          if (j + 2 < nt) {
            if (!k_ready(j + 2)) break;
            issue_s(j + 2);  // into the buffer dQ(j) reads: behind it in issue order
          }
        }
        // completes when every MMA above has; the epilogue reads dQ after it,
        // and after an abort no MMA may still run when the TMEM is released
        mma_commit(&sh.all_done);
        if (*(volatile int *)&sh.abort) {
          int *noerr = nullptr;
          mbar_wait(&sh.all_done, 0, noerr);
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 208;" ::: "memory");
    // ------------------------------------------------------------ P, dS
    const int w = (warp - 4) >> 2;          // key half of every tile
    const int r = 32 * (warp & 3) + lane;   // TMEM lane = query row of the tile
    const int i = m0 + r;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    int lo_i, hi_i;
    key_range(i, lq, lk, f.win_l, f.win_r, lo_i, hi_i);
    int lo_tile_max, hi_tile_min, dummy;
    key_range(m_last, lq, lk, f.win_l, f.win_r, lo_tile_max, dummy);
    key_range(m0, lq, lk, f.win_l, f.win_r, dummy, hi_tile_min);
    const bool valid = i < lq;
    const int64_t li = f.seqs.lse_index(b, h, q0, valid ? i : 0);
    const float nlse = valid ? a.nlse2[li] : 0.f;  // -LSE * log2(e)
    const float dsum = valid ? a.dsum[li] : 0.f;
    const bool cap = f.softcap > 0.f;
    const float sl2 = f.scale * kLog2e, cap_in = cap ? f.scale / f.softcap : 0.f;
    const float cap_l2 = f.softcap * kLog2e;
    const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2 = f2_pack(nlse, nlse), dd2 = f2_pack(dsum, dsum);
    const uint64_t capx2 = f2_pack(cap_l2, cap_l2);
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int key0 = (n_lo + j) * BN + (BN / 2) * w;  // first key of this warpgroup's half
      if (!wait_warp(sh, &sh.s_full[j & 1], (j >> 1) & 1, f.err) ||
          !wait_warp(sh, &sh.dp_full, j & 1, f.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      constexpr int HK = BN / 2;  // keys of this warpgroup per step
      const uint32_t scol = lane_off + tmem + kColS + (j & 1) * BN + HK * w;
      const uint32_t dcol = lane_off + tmem + kColDP + HK * w;
      uint32_t su[HK], du[HK];
      // written out rather than as a loop over 32-column pieces: the loop
      // form measured 15% slower at d = 128 (same registers, same spills)
      if constexpr (HK == 64) {
        tmem_ld32(scol, *reinterpret_cast<uint32_t(*)[32]>(su));
        tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(su + 32));
        tmem_ld32(dcol, *reinterpret_cast<uint32_t(*)[32]>(du));
        tmem_ld32(dcol + 32, *reinterpret_cast<uint32_t(*)[32]>(du + 32));
      } else {
        tmem_ld32(scol, su);
        tmem_ld32(dcol, du);
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(&sh.dp_free);  // dP(j+1) may overwrite the dP columns
      const bool need_mask = !valid || key0 < lo_tile_max || key0 + HK - 1 > hi_tile_min;
      uint32_t pk[HK / 2];
#pragma unroll
      for (int q = 0; q < HK / 2; ++q) {
        const int c = 2 * q;
        const uint64_t s2 = f2_pack(__uint_as_float(su[c]), __uint_as_float(su[c + 1]));
        const uint64_t dp2 = f2_pack(__uint_as_float(du[c]), __uint_as_float(du[c + 1]));
        float t0, t1;
        uint64_t dcap = 0;
        if (cap) {
          // capped score c tanh(s / c); its derivative factor is 1 - tanh^2
          const float h0 = tanh_fast(__uint_as_float(su[c]) * cap_in);
          const float h1 = tanh_fast(__uint_as_float(su[c + 1]) * cap_in);
          f2_unpack(f2_fma(capx2, f2_pack(h0, h1), nl2), t0, t1);
          dcap = f2_pack(fmaf(-h0, h0, 1.f), fmaf(-h1, h1, 1.f));
        } else {
          f2_unpack(f2_fma(s2, sl2x2, nl2), t0, t1);
        }
        float p0 = ex2(t0), p1 = ex2(t1);
        if (need_mask) {
          const int kj = key0 + c;
          if (!valid || kj < lo_i || kj > hi_i) p0 = 0.f;
          if (!valid || kj + 1 < lo_i || kj + 1 > hi_i) p1 = 0.f;
        }
        uint64_t ds2 = f2_mul(f2_pack(p0, p1), f2_sub(dp2, dd2));
        if (cap) ds2 = f2_mul(ds2, dcap);
        float d0, d1;
        f2_unpack(ds2, d0, d1);
        pk[q] = Elem<T>::from_f2(d0, d1);
      }
      // dS (16-bit) over the first half of this warpgroup's S columns: the A
      // operand of dQ += dS K
      tmem_st16(scol, pk);
      if constexpr (HK == 64) tmem_st16(scol + 16, pk + 16);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&sh.ds_full[j & 1]);
    }
    // epilogue: dQ = scale * accumulated dS K; warpgroup w writes columns
    // [DO/2 w, DO/2 w + DO/2) of this CTA's half
    if (ok && nt > 0) ok = wait_warp(sh, &sh.all_done, 0, f.err);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
      T *row = static_cast<T *>(a.dq) + (int64_t)(q0 + (valid ? i : 0)) * a.dq_rs +
               (int64_t)h * D + dh * DO;
#pragma unroll 1
      for (int c = w * (DO / 64); c < (w + 1) * (DO / 64); ++c) {
        uint32_t u[32];
        if (nt > 0) {
          tmem_ld32(lane_off + tmem + kColDQ + c * 32, u);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = 0u;
        }
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          o[e] = Elem<T>::from_f2(__uint_as_float(u[2 * e]) * f.scale,
                                  __uint_as_float(u[2 * e + 1]) * f.scale);
        if (valid) {
          uint4 *dst = reinterpret_cast<uint4 *>(row + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <typename T, int D>
cudaError_t bwd_dq(const BwdArgs &a, cudaStream_t st) {
  using C = DqCfg<D>;
  constexpr int kSmem = C::kSmem, BN = C::BN;
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
  cudaError_t e = set_smem_once<bwd_dq_kernel<T, D>>(kSmem);
  if (e == cudaSuccess)  // 128 * 88 + 256 * 208 after setmaxnreg
    e = check_regs_once<bwd_dq_kernel<T, D>>(kThreads, 128 * 88 + 256 * 208);
  if (e != cudaSuccess) return e;
  const int m_blocks = (f.seqs.sq + BM - 1) / BM;
  const int64_t grid = (int64_t)C::NH * m_blocks * f.hq * f.batch;
  if (grid == 0) return cudaSuccess;
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  debug_log("backward dQ (deterministic): bwd_dq_kernel d=%d, one %d-row query tile and %d dQ "
            "columns per CTA, %d-key steps, grid=%lld CTAs x %d threads, smem=%d B", D, BM, C::DO,
            BN, (long long)grid, kThreads, kSmem);
  bwd_dq_kernel<T, D><<<(unsigned)grid, kThreads, kSmem, st>>>(tq, tk, tv, tdo, a, m_blocks);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_tc(const BwdArgs &a, cudaStream_t st) {
  const bool bf = a.f.dtype == ATTN_BF16;
  switch (a.f.d) {
    case 64: return bf ? bwd_dq<__nv_bfloat16, 64>(a, st) : bwd_dq<__half, 64>(a, st);
    case 128: return bf ? bwd_dq<__nv_bfloat16, 128>(a, st) : bwd_dq<__half, 128>(a, st);
    case 256: return bf ? bwd_dq<__nv_bfloat16, 256>(a, st) : bwd_dq<__half, 256>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
