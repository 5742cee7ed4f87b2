// Backward attention on the 5th-generation tensor cores (sm_103a), d = 64, 128
// or 256.
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
// keys.  Two chunks are in flight: chunk `it` uses TMEM buffer it % 2, so
// the exponentials of one chunk overlap the matrix products of the previous
// one.  Roles (16 warps):
//
//   warp 0         TMA producer: K and V once, Q and dO chunks into a 3-stage
//                  ring.
//   warp 1         MMA issuer and TMEM owner: S^T = K Q^T and dP^T = V dO^T
//                  into the chunk's buffer; then dQ^T = K^T dS^T into the dP^T
//                  columns (already read), dV += P^T dO with P^T read from
//                  TMEM, dK += dS^T Q with dS^T from shared memory.
//   warps 4-7,     two softmax warpgroups, one thread per (key row, half of
//   warps 8-11     the chunk's 64 queries): P^T and dS^T, each split into a
//                  high and a low 16-bit part (so the dV and dK products see
//                  P and dS to about 16 significant bits); P^T goes back into
//                  the S^T columns, dS^T into shared memory.  At the end each
//                  warpgroup writes half of the dK and dV columns.
//   warps 12-15    one thread per head-dim column: dQ^T out of TMEM, added
//                  into an fp32 accumulator in global memory
//                  (`red.global.add`).  In deterministic mode (Inference
//                  Cookbook FAQ Q11) this kernel skips dQ and the
//                  query-stationary kernel of bwd_dq_sm103.cu computes it
//                  without atomics.
//
// TMEM (512 columns): dV [0,128), dK [128,256), buffer b at 256 + 128 b:
// S^T, then P^T high/low, in [0,64); dP^T, then dQ^T, in [64,128).  The MMAs
// of one thread run in issue order, so the products that read P^T from a
// buffer finish before the next S^T overwrites it.
//
// d = 256 keeps this structure with three changes that make it fit.  Each
// CTA produces one 128-column half of dK, dV and dQ (two CTAs per key
// block, each recomputing S and dP over all 256 columns), so dV and dK stay
// at 128 TMEM columns.  Chunks are 32 queries (buffers of 64 columns; the
// dS^T arrays have 64-byte rows in the 64-byte swizzle), and the Q/dO ring
// has 2 stages, so K and V (64 KB each), the ring and dS fit in 224 KB;
// with 2 stages S^T of chunk it+2 is issued after dK of chunk it, which
// frees the stage it loads into.
#include <cudaTypedefs.h>

#include <algorithm>

#include "kernels.h"
#include "sm103.cuh"

namespace attn {

namespace {
using namespace sm103;

constexpr int BN = 128;   // keys per CTA
constexpr int kThreads = 512;

// Tile shape for head dimension D (64, 128 or 256).
template <int D>
struct BwdCfg {
  static constexpr int BQ = D == 256 ? 32 : 64;  // query rows per chunk
  static constexpr int QH = BQ / 2;              // queries of a softmax thread
  static constexpr int ST = D == 256 ? 2 : 3;    // Q/dO ring stages
  static constexpr int DO = D < 128 ? D : 128;   // dK/dV/dQ columns of one CTA
  static constexpr int NH = D / DO;              // CTAs per key block
  static constexpr int kTileK = BN * D * 2;      // one K or V tile: 32 KB at d = 128
  static constexpr int kChunk = BQ * D * 2;      // one Q or dO chunk: 16 KB at d = 128
  static constexpr int kDsRow = BQ * 2;          // bytes per key row of a dS^T array
  static constexpr int kDS = BN * kDsRow;        // one 16-bit [key][query] array
  static constexpr uint32_t kDsSwizzle = BQ == 64 ? 2 : 4;  // descriptor: 128- / 64-byte swizzle
  static constexpr int kSmemData = 2 * kTileK + ST * 2 * kChunk + 2 * 2 * kDS;  // 224 KB at d = 128, 256
  static constexpr int kSmem = kSmemData + 1024;
  static_assert(kSmem <= 227 * 1024 - 1024, "shared memory");
};
constexpr uint32_t kColDV = 0, kColDK = 128, kColBuf = 256;

template <int ST, int BQ>
struct Shared {
  uint64_t kv_full;
  uint64_t qd_full[ST], qd_empty[ST];
  uint64_t sdp_full[2];  // S^T, dP^T of the buffer's chunk are in TMEM
  uint64_t pds_full[2];  // its P^T (TMEM) and dS^T (shared memory) are written
  uint64_t dq_full[2], dq_free[2];
  uint64_t all_done;     // every MMA of the CTA has completed
  uint64_t wait_ns;      // wall-clock limit of a wait
  uint32_t tmem_base;
  int abort;
  // -LSE * log2(e) and D of each ring stage's 64 queries, copied with the
  // stage; per pair of queries (2p, 2p+1): {-LSE_2p, -LSE_2p+1, D_2p, D_2p+1}
  // (log2 units), so a 16-byte load gives both packed pairs
  alignas(16) float lsd[ST][2 * BQ];
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

// The same wait taken by a whole warp with one answer, so warp-collective
// tcgen05 loads/stores that follow are never reached by part of a warp.
template <typename Sh>
__device__ __forceinline__ bool wait_warp(Sh &sh, uint64_t *bar, uint32_t parity, int *err) {
  return __all_sync(0xffffffffu, wait_bar(sh, bar, parity, err));
}

template <typename T> struct IsBf16 { static constexpr int v = 0; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr int v = 1; };

// Fire-and-forget fp32 add to global memory (no value returned).
__device__ __forceinline__ void red_add(float *p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// x = hi + lo with hi, lo 16-bit, for the two values of a packed pair: hi
// and lo are the packed 16-bit pairs.  bf16: hi is x with its low 16 bits
// cleared (truncation), so lo = x - hi is exact in fp32 and only lo is
// rounded; fp16: hi rounded to nearest, lo the rounded remainder.
template <typename T>
__device__ __forceinline__ void split_hi_lo(uint64_t x2, uint32_t &hi, uint32_t &lo) {
  float x0, x1;
  f2_unpack(x2, x0, x1);
  uint64_t h2;
  if constexpr (IsBf16<T>::v) {
    const uint32_t a = __float_as_uint(x0), b = __float_as_uint(x1);
    hi = __byte_perm(a, b, 0x7632);  // high halves of a and b -> (a, b) packed
    h2 = f2_pack(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(b & 0xFFFF0000u));
  } else {
    hi = Elem<T>::from_f2(x0, x1);
    const float2 h = Elem<T>::to_f2(hi);
    h2 = f2_pack(h.x, h.y);
  }
  float l0, l1;
  f2_unpack(f2_sub(x2, h2), l0, l1);
  lo = Elem<T>::from_f2(l0, l1);
}

// Query chunks [c_lo, c_lo + nch) of BQ rows that can see any key of block nb.
template <int BQ>
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

// P^T and dS^T of 16 queries of one key row: the high/low parts of P as 8 + 8
// packed words, of dS as 8 + 8.  Pairs of queries go through packed f32x2
// arithmetic.  `masked` selects the per-element visibility test (rows whose
// whole chunk is visible skip it).  lsd4: the pairs' {-LSE, -LSE, D, D}.
template <typename T, bool kCap>
__device__ __forceinline__ void p_ds_16(const uint32_t *su, const uint32_t *du, const float4 *lsd4,
                                        int i, int qlo, int qhi, bool masked,
                                        float sl2, float cap_in, float cap_l2, uint32_t *ph,
                                        uint32_t *pl, uint32_t *dh, uint32_t *dl) {
  const uint64_t sl2x2 = f2_pack(sl2, sl2), cap_l2x2 = f2_pack(cap_l2, cap_l2);
  const float capk = cap_in * 2.8853900817779268f;  // 2 log2(e) / c, times scale
  const uint64_t capk2 = f2_pack(capk, capk), one2 = f2_pack(1.f, 1.f), mone2 = f2_pack(-1.f, -1.f);
  const uint64_t two2 = f2_pack(2.f, 2.f), mtwo2 = f2_pack(-2.f, -2.f);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int c = 2 * q;
    const float4 v = lsd4[q];
    const uint64_t nl = f2_pack(v.x, v.y), dd = f2_pack(v.z, v.w);
    const uint64_t s2 = f2_pack(__uint_as_float(su[c]), __uint_as_float(su[c + 1]));
    const uint64_t dp2 = f2_pack(__uint_as_float(du[c]), __uint_as_float(du[c + 1]));
    float t0, t1;
    uint64_t dcap = 0;
    if constexpr (kCap) {
      // capped score c tanh(s / c), two at a time: tanh(u) = 1 - 2 r with
      // r = 1 / (e^{2u} + 1) (MUFU exponential and reciprocal); its
      // derivative factor is 1 - tanh^2
      float a0, a1, y0, y1;
      f2_unpack(f2_mul(s2, capk2), a0, a1);  // 2 u log2(e)
      f2_unpack(f2_add(f2_pack(ex2(a0), ex2(a1)), one2), y0, y1);
      const uint64_t r2 = f2_pack(rcp_approx(y0), rcp_approx(y1));
      const uint64_t h2 = f2_fma(r2, mtwo2, one2), nh2 = f2_fma(r2, two2, mone2);
      f2_unpack(f2_fma(cap_l2x2, h2, nl), t0, t1);
      dcap = f2_fma(nh2, h2, one2);
    } else {
      f2_unpack(f2_fma(s2, sl2x2, nl), t0, t1);
    }
    float p0 = ex2(t0), p1 = ex2(t1);
    if (masked) {
      if (i + c < qlo || i + c > qhi) p0 = 0.f;
      if (i + c + 1 < qlo || i + c + 1 > qhi) p1 = 0.f;
    }
    const uint64_t p2 = f2_pack(p0, p1);
    uint64_t ds2 = f2_mul(p2, f2_sub(dp2, dd));
    if constexpr (kCap) ds2 = f2_mul(ds2, dcap);
    split_hi_lo<T>(p2, ph[q], pl[q]);
    split_hi_lo<T>(ds2, dh[q], dl[q]);
  }
}

// Byte offset of 16-byte chunk `c` of row j in a swizzled [row][16-bit]
// array with `row_bytes`-byte rows: the 128-byte swizzle XORs the chunk
// index with (row mod 8), the 64-byte one with ((row / 2) mod 4).
template <int row_bytes>
__device__ __forceinline__ uint32_t swz_off(int j, int c) {
  if constexpr (row_bytes == 128) return j * 128 + ((c ^ (j & 7)) << 4);
  else return j * 64 + ((c ^ ((j >> 1) & 3)) << 4);
}

// Half a chunk of one softmax thread (key row j; row_t = TMEM base + its
// lane): the QH = BQ/2 queries [QH hq, QH hq + QH) of the chunk in buffer
// `buf` (S^T at [0, BQ), dP^T at [BQ, 2 BQ)).  P^T high/low go back over the
// S^T columns just read (high at QH hq + [0, QH/2), low at QH hq + [QH/2,
// QH)); dS^T high/low into the two [key][query] arrays at ds_hi and
// ds_hi + kDS.
template <typename T, bool kCap, typename C>
__device__ __forceinline__ void half_p_ds(uint32_t row_t, uint32_t buf, int hq, uint8_t *ds_hi,
                                          int j, const float4 *lsd4, int i0, int qlo, int qhi,
                                          float sl2, float cap_in, float cap_l2) {
  constexpr int QH = C::QH;
  uint32_t su[QH], du[QH];
  if constexpr (QH == 32) {
    tmem_ld32(row_t + buf + 32 * hq, *reinterpret_cast<uint32_t(*)[32]>(su));
    tmem_ld32(row_t + buf + C::BQ + 32 * hq, *reinterpret_cast<uint32_t(*)[32]>(du));
  } else {
    tmem_ld16(row_t + buf + QH * hq, su);
    tmem_ld16(row_t + buf + C::BQ + QH * hq, du);
  }
  tmem_wait_ld();
  const bool masked = i0 < qlo || i0 + QH - 1 > qhi;
  uint32_t pp[QH];  // P^T high parts in [0, QH/2), low parts in [QH/2, QH)
#pragma unroll
  for (int hv = 0; hv < QH / 16; ++hv) {
    const int c0 = 16 * hv;
    uint32_t dh[8], dl[8];
    p_ds_16<T, kCap>(su + c0, du + c0, lsd4 + c0 / 2, i0 + c0, qlo, qhi, masked, sl2, cap_in, cap_l2,
                     pp + 8 * hv, pp + QH / 2 + 8 * hv, dh, dl);
    // dS^T: 16 queries = two 16-byte chunks of the key's row
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const uint32_t off = swz_off<C::kDsRow>(j, (QH * hq + c0) / 8 + cc);
      *reinterpret_cast<uint4 *>(ds_hi + off) =
          make_uint4(dh[4 * cc], dh[4 * cc + 1], dh[4 * cc + 2], dh[4 * cc + 3]);
      *reinterpret_cast<uint4 *>(ds_hi + C::kDS + off) =
          make_uint4(dl[4 * cc], dl[4 * cc + 1], dl[4 * cc + 2], dl[4 * cc + 3]);
    }
  }
#pragma unroll
  for (int x = 0; x < QH / 16; ++x) tmem_st16(row_t + buf + QH * hq + 16 * x, pp + 16 * x);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const BwdArgs a, const int n_blocks) {
  using C = BwdCfg<D>;
  constexpr int kTileK = C::kTileK, kChunk = C::kChunk, kDS = C::kDS;
  constexpr int BQ = C::BQ, QH = C::QH, ST = C::ST, DO = C::DO;
  const FwdArgs &f = a.f;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared<ST, BQ> sh;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *k_s = smem;
  uint8_t *v_s = smem + kTileK;
  uint8_t *qd_s = smem + 2 * kTileK;           // [stage][Q | dO]
  uint8_t *ds_s = qd_s + ST * 2 * kChunk;      // [buffer][dS high | dS low], each [key][query]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA -> (column half, key block, kv head, batch): halves, then key blocks
  // fastest, so the CTAs of one (batch, kv head) run together and share
  // Q/dO in L2; lower key blocks (the heaviest under a causal mask) are
  // dispatched first.  dh selects the head-dim columns [dh DO, dh DO + DO)
  // of dK, dV and dQ this CTA produces (always 0 below d = 256).
  const int dh = blockIdx.x % C::NH;
  const int bid = blockIdx.x / C::NH;
  const int nb = bid % n_blocks;
  const int kvh = (bid / n_blocks) % f.hkv;
  const int b = bid / (n_blocks * f.hkv);
  int q0, lq, k0, lk;
  if (!f.seqs.get(b, q0, lq, k0, lk, f.err)) return;
  const int key0 = nb * BN;
  if (key0 >= lk) return;
  const int g = f.hq / f.hkv;
  int c_lo, nch;
  chunk_range<BQ>(nb, lq, lk, f.win_l, f.win_r, c_lo, nch);
  const int n_iter = g * nch;
  // deterministic mode: dQ comes from the query-stationary kernel instead
  const bool with_dq = !a.deterministic;

  if (threadIdx.x == 0) {
    mbar_init(&sh.kv_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&sh.qd_full[s], 1);
      mbar_init(&sh.qd_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.sdp_full[s], 1);
      mbar_init(&sh.pds_full[s], 8);   // warps
      mbar_init(&sh.dq_full[s], 1);
      mbar_init(&sh.dq_free[s], 4);
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
  const uint32_t row_t = tmem + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's TMEM lanes

  // launched at 128 registers a thread (16 warps):
  // 128 * (104 + 104 + 2 * 152) <= 512 * 128
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 104;" ::: "memory");
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      // the whole warp copies (LSE * log2(e), D) of each chunk's queries
      // into the stage with cp.async (zeros past the sequence end); lane 0
      // issues the TMA loads.  Both complete the stage's qd_full phase.
      if (n_iter > 0) {
        if (lane == 0) {
          prefetch_tmap(&tq);
          prefetch_tmap(&tk);
          prefetch_tmap(&tv);
          prefetch_tmap(&tdo);
          mbar_expect_tx(&sh.kv_full, 2 * kTileK);
          for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(k_s + c * BN * 128, &tk, &sh.kv_full, c * 64, kvh, k0 + key0);
            tma_load_3d(v_s + c * BN * 128, &tv, &sh.kv_full, c * 64, kvh, k0 + key0);
          }
        }
        int issued = 0;
        for (int it = 0; it < n_iter; ++it) {
          const int st = it % ST;
          const int h = kvh * g + it / nch;
          const int i0 = (c_lo + it % nch) * BQ;
          if (!wait_warp(sh, &sh.qd_empty[st], ((it / ST) & 1) ^ 1, f.err)) break;
#pragma unroll
          for (int r = lane; r < BQ; r += 32) {
            const int i = i0 + r;
            const bool in = i < lq;
            const int64_t li = f.seqs.lse_index(b, h, q0, in ? i : 0);
            float *dst = &sh.lsd[st][(r >> 1) * 4 + (r & 1)];
            cp_async_4(dst, a.nlse2 + li, in ? 4u : 0u);
            cp_async_4(dst + 2, a.dsum + li, in ? 4u : 0u);
          }
          cp_async_mbar_arrive(&sh.qd_full[st]);
          __syncwarp();
          if (lane == 0) {
            mbar_expect_tx(&sh.qd_full[st], 2 * kChunk);
            uint8_t *dst = qd_s + st * 2 * kChunk;
            for (int c = 0; c < D / 64; ++c) {
              tma_load_3d(dst + c * BQ * 128, &tq, &sh.qd_full[st], c * 64, h, q0 + i0);
              tma_load_3d(dst + kChunk + c * BQ * 128, &tdo, &sh.qd_full[st], c * 64, h, q0 + i0);
            }
          }
          issued = it + 1;
        }
        cp_async_wait_all();
        if (lane == 0 && *(volatile int *)&sh.abort) {
          // let this CTA's copies in flight land before the CTA exits
          int *noerr = nullptr;
          mbar_wait(&sh.kv_full, 0, noerr);
          for (int it = max(0, issued - ST); it < issued; ++it)
            mbar_wait(&sh.qd_full[it % ST], (it / ST) & 1, noerr);
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (elect_one() && n_iter > 0) {
        constexpr int ab = IsBf16<T>::v;
        constexpr uint32_t id_s = idesc_f16(128, BQ, ab, 0, 0);   // S^T, dP^T
        constexpr uint32_t id_kv = idesc_f16(128, DO, ab, 0, 1);  // dV, dK (B = dO/Q, MN-major)
        constexpr uint32_t id_q = idesc_f16(128, BQ, ab, 1, 1);   // dQ^T (A = K^T, B = dS^T)
        const uint32_t k_addr = smem_u32(k_s), v_addr = smem_u32(v_s);
        const uint32_t qd_addr = smem_u32(qd_s), ds_addr = smem_u32(ds_s);
        // descriptor bases; every operand below is base + constant offset
        const uint64_t k_kd = smem_desc(k_addr, 16, 1024), v_kd = smem_desc(v_addr, 16, 1024);
        // the MN-major views start at this CTA's column half (64-column blocks 2 dh, 2 dh + 1)
        const uint64_t k_mn = smem_desc(k_addr + dh * 2 * (BN * 128), BN * 128, 1024);
        const uint64_t qd_k = smem_desc(qd_addr, 16, 1024);
        const uint64_t qd_mn = smem_desc(qd_addr + dh * 2 * (BQ * 128), BQ * 128, 1024);
        // dS^T arrays: rows of BQ queries, 8-row groups 8 * kDsRow bytes apart
        const uint64_t ds_k = smem_desc(ds_addr, 16, 8 * C::kDsRow, C::kDsSwizzle);
        const uint64_t ds_mn = smem_desc(ds_addr, 8 * C::kDsRow, 8 * C::kDsRow, C::kDsSwizzle);
        // S^T = K Q^T (which = 0) or dP^T = V dO^T (which = 1) of chunk `it`
        // into its buffer; the Q/dO stage must have landed
        auto issue_s_or_dp = [&](int it, int which) {
          const int st = it % ST;
          const uint32_t buf = tmem + kColBuf + 2 * BQ * (it & 1) + BQ * which;
          const uint64_t a_d = which ? v_kd : k_kd;
          const uint32_t b_o = st * 2 * kChunk + which * kChunk;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = (kk / 4) * (BN * 128) + (kk % 4) * 32;
            const uint32_t qo = (kk / 4) * (BQ * 128) + (kk % 4) * 32;
            mma_ss(buf, desc_add(a_d, ko), desc_add(qd_k, b_o + qo), id_s, kk > 0);
          }
        };
        auto stage_ready = [&](int it) -> bool {
          const bool r = wait_bar(sh, &sh.qd_full[it % ST], (it / ST) & 1, f.err);
          tc_fence_after();
          return r;
        };
        // test hook: all_done completes only after this thread's last
        // commit, so this wait can only run out
        bool ok = !(f.stall && !wait_bar(sh, &sh.all_done, 0, f.err));
        ok = ok && wait_bar(sh, &sh.kv_full, 0, f.err);
        for (int it = 0; ok && it < min(2, n_iter); ++it) {
          if (!(ok = stage_ready(it))) break;
          issue_s_or_dp(it, 0);
          issue_s_or_dp(it, 1);
          mma_commit(&sh.sdp_full[it]);
        }
        // S/dP(0) S/dP(1) | dQ(it) dV(it) S(it+2) dK(it) dP(it+2) | ...
        // S(it+2) needs only dV(it) to have read P^T(it) (issue order);
        // dP(it+2) waits until dQ^T(it) has left the dP^T columns.  With a
        // 2-stage ring, S(it+2) comes after dK(it), whose completion frees
        // the stage chunk it+2 is loaded into.
        for (int it = 0; ok && it < n_iter; ++it) {
          const int bf = it & 1, st = it % ST;
          const uint32_t par = (it >> 1) & 1;
          const uint32_t buf = tmem + kColBuf + 2 * BQ * bf;
          const uint32_t dso = bf * 2 * kDS;
          if (!wait_bar(sh, &sh.pds_full[bf], par, f.err)) break;
          tc_fence_after();
          if (with_dq) {
            // dQ^T = K^T dS^T (high part) into the dP^T columns, already read
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ss(buf + BQ, desc_add(k_mn, kk * 16 * 128),
                     desc_add(ds_mn, dso + kk * 16 * C::kDsRow), id_q, kk > 0);
            mma_commit(&sh.dq_full[bf]);
          }
          const uint32_t q_o = st * 2 * kChunk, do_o = q_o + kChunk;
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk) {
            // dV += (P_high + P_low)^T dO
            const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
            const uint64_t do_d = desc_add(qd_mn, do_o + kk * 16 * 128);
            // queries 16 kk.. of the chunk: softmax half 16 kk / QH, its
            // 16-query step (16 kk % QH) / 16; low parts QH / 2 columns on
            const uint32_t pc = buf + QH * (16 * kk / QH) + 8 * ((16 * kk % QH) / 16);
            mma_ts(tmem + kColDV, pc, do_d, id_kv, acc);
            mma_ts(tmem + kColDV, pc + QH / 2, do_d, id_kv, 1u);
          }
          const bool next = it + 2 < n_iter;
          if constexpr (ST >= 3) {
            if (next) {
              if (!stage_ready(it + 2)) break;
              issue_s_or_dp(it + 2, 0);
            }
          }
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk) {
            // dK += (dS_high + dS_low)^T Q
            const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
            const uint64_t q_d = desc_add(qd_mn, q_o + kk * 16 * 128);
            mma_ss(tmem + kColDK, desc_add(ds_k, dso + kk * 32), q_d, id_kv, acc);
            mma_ss(tmem + kColDK, desc_add(ds_k, dso + kDS + kk * 32), q_d, id_kv, 1u);
          }
          mma_commit(&sh.qd_empty[st]);  // Q and dO of this chunk are no longer read
          if (next) {
            if constexpr (ST < 3) {
              if (!stage_ready(it + 2)) break;
              issue_s_or_dp(it + 2, 0);
            }
            if (with_dq && !wait_bar(sh, &sh.dq_free[bf], par, f.err)) break;
            tc_fence_after();
            issue_s_or_dp(it + 2, 1);
            mma_commit(&sh.sdp_full[bf]);
          }
        }
        // completes when every MMA above has; on abort, wait (bounded) so
        // no MMA is in flight when the TMEM is released
        mma_commit(&sh.all_done);
        if (*(volatile int *)&sh.abort) {
          int *noerr = nullptr;
          mbar_wait(&sh.all_done, 0, noerr);
        }
      }
    }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 152;" ::: "memory");
    // ------------------------------------------------------------ P^T, dS^T
    const int w = (warp - 4) >> 2;          // which half of every chunk's queries
    const int j = 32 * (warp & 3) + lane;  // TMEM lane = key row of the block
    const int kj = key0 + j;
    int qlo, qhi;
    query_range(kj, lq, lk, f.win_l, f.win_r, qlo, qhi);
    if (kj >= lk) qhi = -1;
    const bool cap = f.softcap > 0.f;
    const float sl2 = f.scale * kLog2e, cap_in = cap ? f.scale / f.softcap : 0.f;
    const float cap_l2 = f.softcap * kLog2e;
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int bf = it & 1, st = it % ST;
      const uint32_t par = (it >> 1) & 1;
      const int i0 = (c_lo + it % nch) * BQ + QH * w;
      // S^T, dP^T of this chunk; the commit behind it also covers the MMAs of
      // this buffer's previous chunk, so its dS^T arrays are free.  The
      // stage's (LSE, D) copies landed before its S^T was computed; the wait
      // on qd_full (already complete) makes them visible to this warp.
      if (!wait_warp(sh, &sh.sdp_full[bf], par, f.err) ||
          !wait_warp(sh, &sh.qd_full[st], (it / ST) & 1, f.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint8_t *ds_hi = ds_s + bf * 2 * kDS;
      const uint32_t buf = kColBuf + 2 * BQ * bf;
      const float4 *lsd4 = reinterpret_cast<const float4 *>(sh.lsd[st]) + (QH / 2) * w;
      if (cap)
        half_p_ds<T, true, C>(row_t, buf, w, ds_hi, j, lsd4, i0, qlo, qhi, sl2, cap_in, cap_l2);
      else
        half_p_ds<T, false, C>(row_t, buf, w, ds_hi, j, lsd4, i0, qlo, qhi, sl2, cap_in, cap_l2);
      tmem_wait_st();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive_warp(&sh.pds_full[bf]);
    }
    // dK, dV out of TMEM: each warpgroup writes half of this CTA's columns
    if (ok && n_iter > 0) ok = wait_warp(sh, &sh.all_done, 0, f.err);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    // tcgen05.ld is warp-collective: every lane loads, only real keys store
    if (ok) {
      const int64_t col0 = (int64_t)kvh * D + dh * DO;
      T *dvr = static_cast<T *>(a.dv) + (int64_t)(k0 + kj) * a.dv_rs + col0;
      T *dkr = static_cast<T *>(a.dk) + (int64_t)(k0 + kj) * a.dk_rs + col0;
#pragma unroll 1
      for (int c = w * (DO / 64); c < (w + 1) * (DO / 64); ++c) {
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
          uint32_t o[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            o[e] = Elem<T>::from_f2(__uint_as_float(u[2 * e]) * sc, __uint_as_float(u[2 * e + 1]) * sc);
          if (kj < lk) {
            uint4 *dst = reinterpret_cast<uint4 *>((which ? dkr : dvr) + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
          }
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 104;" ::: "memory");
    // ------------------------------------------------------------ dQ
    const int dl = 32 * (warp & 3) + lane;  // TMEM lane = column dh DO + dl
    // at d = 64 the dQ^T product still has 128 rows (lanes 64-127 hold
    // nothing of use); those two warps only keep the barrier counts
    const bool dq_rows = 32 * (warp & 3) < DO;
    // the accumulator is (hq, rows, d): a chunk's rows are D floats apart
    const int64_t rows_all = f.seqs.cu_q ? f.seqs.total_q : (int64_t)f.batch * f.seqs.sq;
    for (int it = 0; with_dq && it < n_iter; ++it) {
      const int bf = it & 1;
      const int h = kvh * g + it / nch;
      const int i0 = (c_lo + it % nch) * BQ;
      if (!wait_warp(sh, &sh.dq_full[bf], (it >> 1) & 1, f.err)) break;
      tc_fence_after();
      uint32_t u[BQ];
      const uint32_t col = kColBuf + 2 * BQ * bf + BQ;
      if (dq_rows) {
#pragma unroll
        for (int x = 0; x < BQ / 32; ++x)
          tmem_ld32(row_t + col + 32 * x, *reinterpret_cast<uint32_t(*)[32]>(u + 32 * x));
        tmem_wait_ld();
      }
      tc_fence_before();
      mbar_arrive_relaxed_warp(&sh.dq_free[bf]);  // not behind the previous chunk's adds
      if (!dq_rows) continue;
      float *acc = a.dq_acc + ((int64_t)h * rows_all + q0 + i0) * D + dh * DO + dl;
      const int rows = min(BQ, lq - i0);
#pragma unroll
      for (int e = 0; e < BQ; ++e)
        if (e < rows) red_add(acc + e * D, __uint_as_float(u[e]));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// (LSE_i * log2(e), D_i = rowsum(dO_i * O_i)) per row (fp32, LSE layout);
// zero the dQ accumulator of the atomic mode.  One warp per (row, head).
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(BwdArgs a, int64_t rows) {
  // four (row, head) pairs per warp, eight lanes each: D/8 values a lane in
  // 16-byte loads, so each warp keeps several loads of both streams in flight
  constexpr int V = D / 8;  // values per lane
  const FwdArgs &f = a.f;
  const int lane = threadIdx.x & 31, sub = lane & 7;
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t n = rows * f.hq;
  for (int64_t x0 = w * 4; x0 < n; x0 += nw * 4) {
    const int64_t x = x0 + (lane >> 3);
    const bool live = x < n;
    const int64_t off = (live ? x : 0) * D + sub * V;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < V; c += 8) {
      float o[8], g[8];
      load_vec<T, 8>(static_cast<const T *>(f.o) + off + c, o);
      load_vec<T, 8>(static_cast<const T *>(a.dout) + off + c, g);
#pragma unroll
      for (int e = 0; e < 8; ++e) s = fmaf(o[e], g[e], s);
    }
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    if (!live) continue;
    if (!a.deterministic) {
      float4 *z = reinterpret_cast<float4 *>(a.dq_acc + off);
#pragma unroll
      for (int c = 0; c < V / 4; ++c) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (sub == 0) {
      const int64_t row = x / f.hq;
      const int h = (int)(x % f.hq);
      int64_t li;
      if (f.seqs.cu_q) {
        li = (int64_t)h * f.seqs.total_q + row;
      } else {
        const int64_t bb = row / f.seqs.sq, i = row % f.seqs.sq;
        li = (bb * f.hq + h) * f.seqs.sq + i;
      }
      a.dsum[li] = s;
      a.nlse2[li] = -(f.lse[li] * kLog2e);
    }
  }
}

// dQ = scale * dQ_acc -> dtype: the accumulator is (hq, rows, d), dQ
// (rows, hq, d) with rows dq_rs elements apart.  One thread per 8 values
// (two 16-byte loads, one 16-byte store).
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(BwdArgs a, int64_t rows, int64_t n8) {
  const int hq = a.f.hq;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n8;
       x += (int64_t)gridDim.x * blockDim.x) {
    // x walks dQ in (row, head, d / 8) order
    const int c8 = (int)(x % (D / 8));
    const int64_t rh = x / (D / 8);
    const int h = (int)(rh % hq);
    const int64_t row = rh / hq;
    const float4 *src = reinterpret_cast<const float4 *>(a.dq_acc) + ((h * rows + row) * (D / 8) + c8) * 2;
    const float4 v0 = src[0], v1 = src[1];
    const float s = a.f.scale;
    const uint4 out{Elem<T>::from_f2(v0.x * s, v0.y * s), Elem<T>::from_f2(v0.z * s, v0.w * s),
                    Elem<T>::from_f2(v1.x * s, v1.y * s), Elem<T>::from_f2(v1.z * s, v1.w * s)};
    *reinterpret_cast<uint4 *>(static_cast<T *>(a.dq) + row * a.dq_rs + (int64_t)h * D + c8 * 8) =
        out;
  }
}

template <typename T, int D>
cudaError_t bwd_tc(const BwdArgs &a, int sms, cudaStream_t st) {
  using C = BwdCfg<D>;
  constexpr int kSmem = C::kSmem, BQ = C::BQ;
  const FwdArgs &f = a.f;
  const int64_t rows_q = f.seqs.cu_q ? f.seqs.total_q : (int64_t)f.batch * f.seqs.sq;
  const int64_t rows_k = f.seqs.cu_k ? f.seqs.total_k : (int64_t)f.batch * f.seqs.sk;
  const int prep_blocks = (int)std::min<int64_t>((rows_q * f.hq + 31) / 32, (int64_t)sms * 16);
  if (rows_q > 0) {
    bwd_prep_kernel<T, D><<<std::max(prep_blocks, 1), 256, 0, st>>>(a, rows_q);
    count_launches(1);
  }
  if (rows_k > 0 && rows_q > 0) {
    CUtensorMap tq, tk, tv, tdo;
    if (!make_map_3d(&tq, f.q, f.dtype, rows_q, f.hq, D, BQ, f.q_rs) ||
        !make_map_3d(&tdo, a.dout, f.dtype, rows_q, f.hq, D, BQ) ||
        !make_map_3d(&tk, f.k, f.dtype, rows_k, f.hkv, D, BN, f.k_rs) ||
        !make_map_3d(&tv, f.v, f.dtype, rows_k, f.hkv, D, BN, f.v_rs))
      return cudaErrorInvalidValue;
    cudaError_t e = set_smem_once<bwd_tc_kernel<T, D>>(kSmem);
    if (e == cudaSuccess)  // 128 * (104 + 2 * 152 + 104) after setmaxnreg
      e = check_regs_once<bwd_tc_kernel<T, D>>(kThreads, 128 * (104 + 2 * 152 + 104));
    if (e != cudaSuccess) return e;
    const int n_blocks = (f.seqs.sk + BN - 1) / BN;
    const int64_t grid = (int64_t)C::NH * n_blocks * f.hkv * f.batch;
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
    debug_log("backward: bwd_tc_kernel d=%d, %d keys per CTA, %d output columns per CTA, "
              "%d-query chunks, %d-stage ring, dQ %s, grid=%lld CTAs x %d threads, smem=%d B",
              D, BN, C::DO, BQ, C::ST,
              a.deterministic ? "by the query-stationary kernel (deterministic)" : "atomic fp32 adds",
              (long long)grid, kThreads, kSmem);
    bwd_tc_kernel<T, D><<<(unsigned)grid, kThreads, kSmem, st>>>(tq, tk, tv, tdo, a, n_blocks);
    count_launches(1);
  } else if (rows_k > 0) {  // no queries: the key gradients are zero
    const size_t w = (size_t)f.hkv * D * 2;
    cudaError_t e = cudaMemset2DAsync(a.dk, (size_t)a.dk_rs * 2, 0, w, (size_t)rows_k, st);
    if (e == cudaSuccess) e = cudaMemset2DAsync(a.dv, (size_t)a.dv_rs * 2, 0, w, (size_t)rows_k, st);
    if (e != cudaSuccess) return e;
  }
  if (a.deterministic) {
    // dQ from the query-stationary kernel: no atomics, the same bits every run
    cudaError_t e = launch_bwd_dq_tc(a, st);
    if (e != cudaSuccess) return e;
  } else if (rows_q > 0) {
    const int64_t n8 = rows_q * f.hq * D / 8;
    const int blocks = (int)std::min<int64_t>((n8 + 255) / 256, (int64_t)sms * 16);
    bwd_dq_convert_kernel<T, D><<<std::max(blocks, 1), 256, 0, st>>>(a, rows_q, n8);
    count_launches(1);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdArgs &a, int sms, cudaStream_t st) {
  const bool bf = a.f.dtype == ATTN_BF16;
  switch (a.f.d) {
    case 64: return bf ? bwd_tc<__nv_bfloat16, 64>(a, sms, st) : bwd_tc<__half, 64>(a, sms, st);
    case 128: return bf ? bwd_tc<__nv_bfloat16, 128>(a, sms, st) : bwd_tc<__half, 128>(a, sms, st);
    case 256: return bf ? bwd_tc<__nv_bfloat16, 256>(a, sms, st) : bwd_tc<__half, 256>(a, sms, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
