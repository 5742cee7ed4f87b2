// Split-KV paged decode on the 5th-generation tensor cores (sm_103a), d = 64,
// 128 or 256.
//
// Inference Cookbook FAQ Q14/Q17/Q18.  One CTA owns one key range (split) of
// one (batch entry, KV head) and all R = g * sq query rows that read that KV
// head (GQA packing: the g query heads of the group and the sq new tokens
// share every K/V tile; FAQ Q15).  The contraction is done transposed so the
// 128 keys of a tile sit on the TMEM lanes and the few query rows are the
// MMA's N dimension:
//
//   S^T [128 keys x RP] = K_tile Q^T              (A = K, B = Q; both K-major)
//   O^T [d x RP]       += V_tile^T P^T            (A = V as MN-major, B = P K-major)
//
// with RP = R padded to 16 or 32.  K/V tiles are 128 consecutive keys of one
// page (page_size % 128 == 0), fetched by TMA from the page pool at the
// physical row the block table gives.  Roles:
//
//   warp 0     TMA producer (Q once, then K and V tiles through 3-stage
//              rings; other depths at d = 64 and 256, below)
//   warp 1     MMA issuer
//   warps 2-5  one thread per key (TMEM lane): mask, column max across the
//              CTA, exp, P into shared memory; the same threads own the d
//              rows of O^T for the rescale and the epilogue.
//
// The output is the split's normalised partial O and its LSE (or the final
// output when there is one split); decode.cu merges the splits.
//
// Head dims: at d = 64 the O^T product keeps M = 128 (its rows 64-127 read
// the 16 KB after the V tile, padding included in the shared memory, and are
// never stored; with 16 query rows two CTAs share an SM, each with 2-stage
// rings); at d = 256 O^T is two M = 128 products, one per half of d, and the
// 64 KB K and V tiles come through a 1-stage K ring and a 2-stage V ring.
#include <cudaTypedefs.h>

#include "kernels.h"
#include "sm103.cuh"

namespace attn {

namespace {
using namespace sm103;

constexpr int BK = 128;  // keys per tile
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;

// Shapes for head dim D and RP (query rows padded to 16 or 32).
template <int D, int RP>
struct DecCfg {
  // two CTAs per SM at d = 64 with 16 query rows (its registers allow it):
  // the per-tile chain of one overlaps the other's
  static constexpr int kCtas = (D == 64 && RP == 16) ? 2 : 1;
  static constexpr int KST = D == 256 ? 1 : kCtas == 2 ? 2 : 3;  // K ring stages
  static constexpr int VST = D == 256 ? 2 : kCtas == 2 ? 2 : 3;  // V ring stages
  static constexpr int kTile = BK * D * 2;           // one K or V tile: 32 KB at d = 128
  static constexpr int kQBytes = RP * D * 2;
  static constexpr int kPBytes = RP * BK * 2;
  static constexpr int kPad = D == 64 ? kTile : 0;   // read past the last V tile by O^T's rows 64-127
  static constexpr int kSmemData = kQBytes + (KST + VST) * kTile + 2 * kPBytes + kPad;
  static constexpr int kSmem = kSmemData + 1024;
  static constexpr int kOHalves = D == 256 ? 2 : 1;  // O^T products of 128 rows
  static constexpr uint32_t kColS = 0;               // two S^T buffers of RP columns
  static constexpr uint32_t kColO = 2 * RP;          // O^T: kOHalves blocks of RP columns
  static constexpr uint32_t kTmemCols = (2 + kOHalves) * RP <= 64 ? 64 : 128;
  static_assert(kSmem + 2048 <= 227 * 1024, "shared memory");
  static_assert(kCtas == 1 || 2 * (kSmem + 2048) <= 228 * 1024, "shared memory of two CTAs");
};

template <int KST, int VST>
struct DecShared {
  uint64_t q_full;
  uint64_t k_full[KST], k_empty[KST], v_full[VST], v_empty[VST];
  uint64_t s_full[2], p_full[2], o_done;
  uint64_t grp;  // bounded barrier of the 128 softmax threads (one phase per use)
  uint64_t all_done;  // every MMA of the CTA has completed
  uint64_t wait_ns;   // wall-clock limit of a wait
  uint32_t tmem_base;
  int abort;
  alignas(16) float wmax[2][4][32];
  alignas(16) float wsum[4][32];
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Maximum of v over the 32 lanes of the warp (all lanes active).
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

template <typename Sh>
__device__ __forceinline__ bool wait_bar(Sh &sh, uint64_t *bar, uint32_t parity, int *err) {
  return mbar_wait_bounded(smem_u32(bar), parity, &sh.abort, err, sh.wait_ns);
}

// The result of a split whose keys could not be read (a bad length, a page
// outside the pool, or an abandoned wait): O = 0 and LSE = -inf, what an
// empty key set gives, so the combine step gives the split no weight and no
// stale scratch value reaches the output.  The device error word records
// the cause.  Thread `tid` of `nthreads` writes its share of the R rows.
template <typename T, int D>
__device__ __forceinline__ void store_empty_split(const DecodeArgs &a, int split, int bi, int kvh,
                                                  int R, int tid, int nthreads) {
  const int g = a.hq / a.hkv;
  for (int x = tid; x < R * D; x += nthreads) {
    const int q = x / D, dcol = x % D;
    const int r = q / g, h = kvh * g + q % g;
    if (a.num_splits == 1) {
      static_cast<T *>(a.o)[(((int64_t)bi * a.sq + r) * a.hq + h) * D + dcol] = Elem<T>::from_f(0.f);
      if (dcol == 0) a.lse[((int64_t)bi * a.hq + h) * a.sq + r] = -INFINITY;
    } else {
      a.o_part[((((int64_t)split * a.b + bi) * a.sq + r) * a.hq + h) * D + dcol] = 0.f;
      if (dcol == 0) a.lse_part[(((int64_t)split * a.b + bi) * a.hq + h) * a.sq + r] = -INFINITY;
    }
  }
}

// The same wait taken by a whole warp with one answer, so warp-collective
// tcgen05 loads/stores that follow are never reached by part of a warp.
template <typename Sh>
__device__ __forceinline__ bool wait_warp(Sh &sh, uint64_t *bar, uint32_t parity, int *err) {
  return __all_sync(0xffffffffu, wait_bar(sh, bar, parity, err));
}

template <typename T> struct IsBf16 { static constexpr int v = 0; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr int v = 1; };

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11,"
      " %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

template <int RP>
__device__ __forceinline__ void tmem_ld_rp(uint32_t taddr, uint32_t (&r)[RP]) {
  if constexpr (RP == 16) {
    tmem_ld16(taddr, r);
  } else {
    tmem_ld32(taddr, r);
  }
}

template <int RP>
__device__ __forceinline__ void tmem_st_rp(uint32_t taddr, uint32_t (&r)[RP]) {
  if constexpr (RP == 16) {
    tmem_st16(taddr, r);
  } else {
    tmem_st32(taddr, r);
  }
}

template <typename T, int D, int RP>
__global__ void __launch_bounds__(kThreads, DecCfg<D, RP>::kCtas)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const DecodeArgs a) {
  using C = DecCfg<D, RP>;
  constexpr int KST = C::KST, VST = C::VST, kTile = C::kTile;
  extern __shared__ uint8_t smem_raw[];
  __shared__ DecShared<KST, VST> sh;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *q_s = smem;
  uint8_t *k_s = smem + C::kQBytes;
  uint8_t *v_s = k_s + KST * kTile;
  uint8_t *p_s = v_s + VST * kTile;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = a.hq / a.hkv;
  const int R = g * a.sq;
  // CTA -> (split, kv head, batch entry), splits fastest
  const int split = blockIdx.x % a.num_splits;
  const int kvh = (blockIdx.x / a.num_splits) % a.hkv;
  const int bi = blockIdx.x / (a.num_splits * a.hkv);
  const int L = a.cache_seqlens[bi] + a.s_new;
  if (L < 0 || L > a.max_pages * a.page_size) {
    if (threadIdx.x == 0) raise_error(a.err, L < 0 ? kErrBadSeqlen : kErrCacheOverflow);
    store_empty_split<T, D>(a, split, bi, kvh, R, threadIdx.x, kThreads);
    return;
  }
  // keys any query row may see, clipped to this split
  int lo0, hi0, lo1, hi1;
  key_range(0, a.sq, L, a.win_l, a.win_r, lo0, hi0);
  key_range(a.sq - 1, a.sq, L, a.win_l, a.win_r, lo1, hi1);
  const int k_begin = max(lo0, split * a.split_chunk);
  const int k_end = min(hi1 + 1, min(L, (split + 1) * a.split_chunk));  // exclusive
  const int t_first = k_begin / BK;
  const int n = k_end > k_begin ? (k_end - 1) / BK - t_first + 1 : 0;
  // an empty split writes nothing: the combine step skips it by the same test
  if (n == 0 && a.num_splits > 1) return;

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
      mbar_init(&sh.p_full[s], 128);
    }
    mbar_init(&sh.o_done, 1);
    mbar_init(&sh.grp, 128);
    mbar_init(&sh.all_done, 1);
    sh.wait_ns = a.wait_ns;
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  // rows R..RP-1 of the Q tile are padding: zero them once (all D/64
  // column blocks, D/8 16-byte chunks a row)
  for (int x = threadIdx.x; x < (RP - R) * (D / 8); x += kThreads) {
    const int row = R + x / (D / 8), chunk = x % (D / 8);
    *reinterpret_cast<uint4 *>(q_s + (chunk / 8) * (RP * 128) + row * 128 + (chunk % 8) * 16) =
        make_uint4(0, 0, 0, 0);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one() && n > 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      mbar_expect_tx(&sh.q_full, R * D * 2);
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(q_s + c * RP * 128, &tq, &sh.q_full, c * 64, kvh * g, bi * a.sq);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n; ++j) {
        const int pos = (t_first + j) * BK;
        const int pg = pos / a.page_size;
        const int page = a.block_table ? a.block_table[(int64_t)bi * a.max_pages + pg] : bi;
        if (pg >= a.max_pages || page < 0 || page >= a.num_pages) {
          raise_error(a.err, kErrPageOutOfRange);
          *(volatile int *)&sh.abort = 1;
          break;
        }
        const int row = page * a.page_size + pos % a.page_size;
        const int ks = j % KST, vs = j % VST;
        if (!wait_bar(sh, &sh.k_empty[ks], ((j / KST) & 1) ^ 1, a.err)) break;
        mbar_expect_tx(&sh.k_full[ks], kTile);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(k_s + ks * kTile + c * BK * 128, &tk, &sh.k_full[ks], c * 64, kvh, row);
        k_issued = j + 1;
        if (!wait_bar(sh, &sh.v_empty[vs], ((j / VST) & 1) ^ 1, a.err)) break;
        mbar_expect_tx(&sh.v_full[vs], kTile);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(v_s + vs * kTile + c * BK * 128, &tv, &sh.v_full[vs], c * 64, kvh, row);
        v_issued = j + 1;
      }
      if (*(volatile int *)&sh.abort) {
        int *noerr = nullptr;
        mbar_wait(&sh.q_full, 0, noerr);
        for (int j = max(0, k_issued - KST); j < k_issued; ++j)
          mbar_wait(&sh.k_full[j % KST], (j / KST) & 1, noerr);
        for (int j = max(0, v_issued - VST); j < v_issued; ++j)
          mbar_wait(&sh.v_full[j % VST], (j / VST) & 1, noerr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one() && n > 0) {
      constexpr int ab = IsBf16<T>::v;
      constexpr uint32_t id_s = idesc_f16(128, RP, ab, 0, 0);
      constexpr uint32_t id_o = idesc_f16(128, RP, ab, 1, 0);
      const uint32_t q_addr = smem_u32(q_s), k_addr = smem_u32(k_s), v_addr = smem_u32(v_s);
      const uint32_t p_addr = smem_u32(p_s);
      auto issue_s = [&](int j) -> bool {
        const int st = j % KST;
        if (!wait_bar(sh, &sh.k_full[st], (j / KST) & 1, a.err)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = smem_desc(k_addr + st * kTile + (kk / 4) * (BK * 128) + (kk % 4) * 32,
                                        16, 1024);
          const uint64_t bd = smem_desc(q_addr + (kk / 4) * (RP * 128) + (kk % 4) * 32, 16, 1024);
          mma_ss(tmem + C::kColS + (j & 1) * RP, ad, bd, id_s, kk > 0);
        }
        mma_commit(&sh.s_full[j & 1]);
        mma_commit(&sh.k_empty[st]);
        return true;
      };
      // test hook: all_done completes only after this thread's last commit,
      // so this wait can only run out
      bool ok = !(a.stall && !wait_bar(sh, &sh.all_done, 0, a.err));
      ok = ok && wait_bar(sh, &sh.q_full, 0, a.err) && issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n && !issue_s(j + 1)) break;
        if (!wait_bar(sh, &sh.p_full[j & 1], (j >> 1) & 1, a.err)) break;
        const int st = j % VST;
        if (!wait_bar(sh, &sh.v_full[st], (j / VST) & 1, a.err)) break;
        tc_fence_after();
        const uint32_t pb = p_addr + (j & 1) * C::kPBytes;
#pragma unroll
        for (int h2 = 0; h2 < C::kOHalves; ++h2) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A = V^T (M = 128 rows of d from column block 2 h2 on, MN-major:
            // 64-column blocks BK*128 bytes apart)
            const uint64_t ad = smem_desc(v_addr + st * kTile + h2 * 2 * (BK * 128) + kk * 16 * 128,
                                          BK * 128, 1024);
            const uint64_t bd = smem_desc(pb + (kk / 4) * (RP * 128) + (kk % 4) * 32, 16, 1024);
            mma_ss(tmem + C::kColO + h2 * RP, ad, bd, id_o, (j > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&sh.o_done);
        mma_commit(&sh.v_empty[st]);
      }
      // after an abort, no MMA may still run when the TMEM is released
      mma_commit(&sh.all_done);
      if (*(volatile int *)&sh.abort) {
        int *noerr = nullptr;
        mbar_wait(&sh.all_done, 0, noerr);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int w4 = warp & 3;
    const int jl = 32 * w4 + lane;  // TMEM lane: key of the tile, and row d of O^T
    const uint32_t lane_off = (uint32_t)(32 * w4) << 16;
    const float sl2 = a.scale * kLog2e;
    const bool cap = a.softcap > 0.f;
    const float cap_in = cap ? a.scale / a.softcap : 0.f, cap_out = a.softcap * kLog2e;
    // visible key range of each query row q = r * g + t (r = new-token index)
    int qlo[RP], qhi[RP];
#pragma unroll
    for (int q = 0; q < RP; ++q) {
      const int r = q < R ? q / g : 0;
      key_range(r, a.sq, L, a.win_l, a.win_r, qlo[q], qhi[q]);
      if (q >= R) qhi[q] = -1;
      qlo[q] = max(qlo[q], k_begin);
      qhi[q] = min(qhi[q], k_end - 1);
    }
    // tiles inside [qlo_max, qhi_min] are seen whole by every live row
    int qlo_max = k_begin, qhi_min = k_end - 1;
#pragma unroll
    for (int q = 0; q < RP; ++q) {
      if (q < R) {
        qlo_max = max(qlo_max, qlo[q]);
        qhi_min = min(qhi_min, qhi[q]);
      }
    }
    float m_run[RP], l_part[RP];
#pragma unroll
    for (int q = 0; q < RP; ++q) {
      m_run[q] = -INFINITY;
      l_part[q] = 0.f;
    }
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int key = (t_first + j) * BK + jl;
      if (!wait_warp(sh, &sh.s_full[j & 1], (j >> 1) & 1, a.err)) { ok = false; break; }
      tc_fence_after();
      uint32_t su[RP];
      tmem_ld_rp<RP>(tmem + lane_off + C::kColS + (j & 1) * RP, su);
      tmem_wait_ld();
      float x[RP];
      float tmax[RP];
      const int t0 = key - jl;
      if (RP <= 16 && !cap && t0 >= qlo_max && t0 + BK - 1 <= qhi_min) {
        // every live row sees the whole tile: no mask (the padding columns
        // past R get scores of their zero rows, which touch only their own
        // O^T columns and are never stored)
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
        for (int q = 0; q < RP; q += 2)
          f2_unpack(f2_mul(f2_pack(__uint_as_float(su[q]), __uint_as_float(su[q + 1])), sl2x2),
                    x[q], x[q + 1]);
      } else {
#pragma unroll
        for (int q = 0; q < RP; ++q) {
          const float s = __uint_as_float(su[q]);
          const bool vis = key >= qlo[q] && key <= qhi[q];
          x[q] = vis ? (cap ? cap_out * tanh_fast(s * cap_in) : s * sl2) : -INFINITY;
        }
      }
#pragma unroll
      for (int q = 0; q < RP; ++q) tmax[q] = x[q];
      // column max over the 128 keys of the tile: one warp reduction per
      // column, then across warps
#pragma unroll
      for (int q = 0; q < RP; ++q) tmax[q] = warp_max(tmax[q]);
      // lane 0 publishes the warp's column maxima (every lane holds them);
      // the buffer alternates per tile, so the barrier of tile j also ends
      // every read of tile j-1's buffer
      float(*wm)[32] = sh.wmax[j & 1];
      if (lane == 0) {
#pragma unroll
        for (int q = 0; q < RP; q += 4)
          *reinterpret_cast<float4 *>(&wm[w4][q]) = make_float4(tmax[q], tmax[q + 1], tmax[q + 2], tmax[q + 3]);
      }
      mbar_arrive(&sh.grp);
      if (!wait_warp(sh, &sh.grp, j & 1, a.err)) { ok = false; break; }
      float alpha[RP];
      bool any_rescale = false;
      float tms[RP];
      if constexpr (RP <= 16) {
#pragma unroll
        for (int q = 0; q < RP; q += 4) {
          const float4 w0 = *reinterpret_cast<const float4 *>(&wm[0][q]);
          const float4 w1 = *reinterpret_cast<const float4 *>(&wm[1][q]);
          const float4 w2 = *reinterpret_cast<const float4 *>(&wm[2][q]);
          const float4 w3 = *reinterpret_cast<const float4 *>(&wm[3][q]);
          tms[q] = fmaxf(fmax3(w0.x, w1.x, w2.x), w3.x);
          tms[q + 1] = fmaxf(fmax3(w0.y, w1.y, w2.y), w3.y);
          tms[q + 2] = fmaxf(fmax3(w0.z, w1.z, w2.z), w3.z);
          tms[q + 3] = fmaxf(fmax3(w0.w, w1.w, w2.w), w3.w);
        }
      }
#pragma unroll
      for (int q = 0; q < RP; ++q) {
        // (32 columns: read one at a time, to stay within the registers)
        const float tm = RP <= 16 ? tms[q] : fmaxf(fmax3(wm[0][q], wm[1][q], wm[2][q]), wm[3][q]);
        const float m_new = fmaxf(m_run[q], tm);
        alpha[q] = 1.f;
        if (m_new > m_run[q] + kRescaleThreshold) {
          alpha[q] = ex2(m_run[q] - m_new);
          m_run[q] = m_new;
          l_part[q] *= alpha[q];
          any_rescale = true;
        }
      }
      uint16_t pv[RP];
#pragma unroll
      for (int q = 0; q < RP; ++q) {
        const float p = x[q] == -INFINITY ? 0.f : ex2(x[q] - m_run[q]);
        l_part[q] += p;
        const uint32_t pk = Elem<T>::from_f2(p, 0.f);
        pv[q] = (uint16_t)(pk & 0xFFFF);
      }
      // PV(j-1) must be done before its P buffer's twin is rewritten and O^T rescaled
      if (j > 0) {
        if (!wait_warp(sh, &sh.o_done, (j - 1) & 1, a.err)) { ok = false; break; }
        tc_fence_after();
      }
      uint8_t *pb = p_s + (j & 1) * C::kPBytes + (jl / 64) * (RP * 128);
#pragma unroll
      for (int q = 0; q < RP; ++q) {
        const uint32_t off = q * 128 + (jl % 64) * 2;
        *reinterpret_cast<uint16_t *>(pb + (off ^ (((off >> 7) & 7) << 4))) = pv[q];
      }
      if (j > 0 && any_rescale) {  // all threads agree: the maxima are shared
#pragma unroll
        for (int h2 = 0; h2 < C::kOHalves; ++h2) {
          uint32_t ou[RP];
          tmem_ld_rp<RP>(tmem + lane_off + C::kColO + h2 * RP, ou);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < RP; ++q) ou[q] = __float_as_uint(__uint_as_float(ou[q]) * alpha[q]);
          tmem_st_rp<RP>(tmem + lane_off + C::kColO + h2 * RP, ou);
        }
        tmem_wait_st();
      }
      if (__any_sync(0xffffffffu, key >= L)) {
        // keys past the cache end: their V rows may hold anything, and 0 * NaN
        // would poison O^T, so zero them (the TMA load must have landed)
        if (!wait_warp(sh, &sh.v_full[j % VST], (j / VST) & 1, a.err)) { ok = false; break; }
        if (key >= L) {
          uint8_t *vr = v_s + (j % VST) * kTile + jl * 128;
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4 *>(vr + c * BK * 128 + u * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(&sh.p_full[j & 1]);
    }
    // epilogue: column sums across the CTA, then O^T / l
    if (ok && n > 0) ok = wait_warp(sh, &sh.o_done, (n - 1) & 1, a.err);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
#pragma unroll
      for (int q = 0; q < RP; ++q) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l_part[q] += __shfl_xor_sync(0xffffffffu, l_part[q], o);
      }
      float mine = 0.f;
#pragma unroll
      for (int q = 0; q < RP; ++q)
        if (lane == q) mine = l_part[q];
      if (lane < RP) sh.wsum[w4][lane] = mine;
      mbar_arrive(&sh.grp);
      ok = wait_warp(sh, &sh.grp, n & 1, a.err);
    }
    if (ok) {
#pragma unroll 1
      for (int h2 = 0; h2 < C::kOHalves; ++h2) {
      uint32_t ou[RP];
      if (n > 0) {  // warp-collective: every lane loads, only real columns store
        tmem_ld_rp<RP>(tmem + lane_off + C::kColO + h2 * RP, ou);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int q = 0; q < RP; ++q) ou[q] = 0u;
      }
      const int dcol = jl + 128 * h2;  // O^T row = head-dim column
      if (dcol >= D) continue;         // d = 64: rows 64-127 of O^T are not used
#pragma unroll
      for (int q = 0; q < RP; ++q) {
        if (q >= R) continue;
        const float lsum = sh.wsum[0][q] + sh.wsum[1][q] + sh.wsum[2][q] + sh.wsum[3][q];
        const float o = lsum > 0.f ? __uint_as_float(ou[q]) / lsum : 0.f;
        const int r = q / g, h = kvh * g + q % g;
        const float lse = lsum > 0.f ? (m_run[q] + __log2f(lsum)) * kLn2 : -INFINITY;
        if (a.num_splits == 1) {
          static_cast<T *>(a.o)[(((int64_t)bi * a.sq + r) * a.hq + h) * D + dcol] = Elem<T>::from_f(o);
          if (dcol == 0) a.lse[((int64_t)bi * a.hq + h) * a.sq + r] = lse;
        } else {
          a.o_part[((((int64_t)split * a.b + bi) * a.sq + r) * a.hq + h) * D + dcol] = o;
          if (dcol == 0) a.lse_part[(((int64_t)split * a.b + bi) * a.hq + h) * a.sq + r] = lse;
        }
      }
      }
    } else {
      store_empty_split<T, D>(a, split, bi, kvh, R, jl, 128);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

template <typename T, int D, int RP>
cudaError_t decode_tc(const DecodeArgs &a, cudaStream_t st) {
  using C = DecCfg<D, RP>;
  CUtensorMap tq, tk, tv;
  const int64_t pool_rows = (int64_t)a.num_pages * a.page_size;
  const int g = a.hq / a.hkv;
  // Q as (d, hq, b*sq) with a box of g heads x sq tokens: rows r*g + t
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.hq, (cuuint64_t)a.b * a.sq};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.hq * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)a.sq};
  cuuint32_t es[3] = {1, 1, 1};
  auto enc = tensor_map_encoder();
  if (!enc ||
      enc(&tq, a.dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
          3, const_cast<void *>(a.q), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (!make_map_3d(&tk, a.k_cache, a.dtype, pool_rows, a.hkv, D, BK) ||
      !make_map_3d(&tv, a.v_cache, a.dtype, pool_rows, a.hkv, D, BK))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_once<decode_tc_kernel<T, D, RP>>(C::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t grid = (int64_t)a.num_splits * a.hkv * a.b;
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  debug_log("decode: decode_tc_kernel d=%d, %d query rows (g*sq) padded to %d, %d-key tiles, "
            "K/V rings of %d/%d stages, num_splits=%d (%d keys each), grid=%lld CTAs x %d threads",
            D, (a.hq / a.hkv) * a.sq, RP, BK, C::KST, C::VST, a.num_splits, a.split_chunk,
            (long long)grid, kThreads);
  decode_tc_kernel<T, D, RP><<<(unsigned)grid, kThreads, C::kSmem, st>>>(tq, tk, tv, a);
  count_launches(1);
  return cudaGetLastError();
}

template <int D>
cudaError_t decode_tc_d(const DecodeArgs &a, int R, cudaStream_t st) {
  const bool bf = a.dtype == ATTN_BF16;
  if (R <= 16) return bf ? decode_tc<__nv_bfloat16, D, 16>(a, st) : decode_tc<__half, D, 16>(a, st);
  return bf ? decode_tc<__nv_bfloat16, D, 32>(a, st) : decode_tc<__half, D, 32>(a, st);
}

}  // namespace

// Returns cudaErrorNotSupported when the shape is outside what this kernel
// handles (d not 64, 128 or 256, g * sq > 32, page_size % 128 != 0).
cudaError_t launch_decode_tc(const DecodeArgs &a, cudaStream_t st) {
  const int R = (a.hq / a.hkv) * a.sq;
  if (R > 32 || a.page_size % BK != 0 || a.sq > 256 || a.hq / a.hkv > 256)
    return cudaErrorNotSupported;
  switch (a.d) {
    case 64: return decode_tc_d<64>(a, R, st);
    case 128: return decode_tc_d<128>(a, R, st);
    case 256: return decode_tc_d<256>(a, R, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace attn
