// Forward attention on the 5th-generation tensor cores (sm_103a).
//
// One CTA owns two 128-row query tiles (one for d = 256) of one (batch,
// head) and streams the key/value tiles they may see ("FlashAttention完整说明"
// §二.1: tiling plus an online softmax, so S and P never reach global
// memory).  With PackGQA (Inference Cookbook FAQ Q15) a tile holds 128/g
// query positions of all g query heads of one KV head instead.  The FP8
// variant (QB = 1, FAQ Q20) reads E4M3 Q and K and computes S with
// kind::f8f6f4; V is bf16 there too.  Roles:
//
//   warp 0      TMA producer: Q once, then K and V tiles into a smem ring.
//   warp 1      MMA issuer (one elected lane): S_j = Q K_j^T into TMEM,
//               O += P_j V_j with P_j read from TMEM; also owns the TMEM
//               allocation.
//   softmax     one warpgroup per 128-row query tile (warps 4-11 for two
//               tiles, 2-5 for one), one thread per query row: loads S_j from
//               TMEM, applies scale -> softcap -> mask (Inference Cookbook
//               FAQ Q22 order; bottom-right causal FAQ Q6; window FAQ Q21),
//               runs the online max/sum update, writes P_j (fp16/bf16) back
//               into the S_j columns, rescales O in TMEM when the running max
//               grows by more than 2^8, and finally writes O / l and the LSE.
//
// TMEM (512 columns): O at [0, D), two S/P buffers at [D, D+BN) and
// [D+BN, D+2BN), so S_{j+1} is computed while the softmax works on S_j.
// The CTA order puts the heaviest causal query tiles first (longest job
// first) and keeps the query heads of one KV head adjacent, so their K/V
// tiles are shared through L2.
#include <cudaTypedefs.h>

#include <algorithm>

#include "kernels.h"
#include "sm103.cuh"

namespace attn {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// (rows, heads, D) tensor, box {64, 1, box_rows}, 128-byte swizzle.
bool make_map_3d(CUtensorMap *m, const void *base, int dtype, int64_t rows, int heads, int d,
              int box_rows, int64_t row_stride, int box_heads) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  if (row_stride == 0) row_stride = (int64_t)heads * d;
  // E4M3 tensors: 1-byte elements, so a 128-byte box row is 128 of them
  const int eb = dtype == kDtypeE4M3 ? 1 : 2;
  cuuint64_t strides[2] = {(cuuint64_t)d * eb, (cuuint64_t)row_stride * eb};
  cuuint32_t box[3] = {(cuuint32_t)(128 / eb), (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dtype == kDtypeE4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
             : dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
             3, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
using namespace sm103;

constexpr int kBM = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when max grows > 256x

// NT query tiles of 128 rows per CTA.  NT = 2 (d <= 128): one softmax
// warpgroup per tile, TMEM = [O_0 | O_1 | S_0 | S_1]; the MMA warp alternates
// between the tiles so one tile's softmax overlaps the other tile's MMAs, and
// every K/V tile staged in shared memory serves 256 query rows.  NT = 1
// (d = 256, d = 64, and d = 128 over at most 1024 keys): TMEM = [O | S_a
// | S_b], S double-buffered instead; at d = 128 with 64-key steps that is 256
// TMEM columns and ~97 KB of shared memory, so two CTAs share an SM.
// QB: bytes per Q/K element (2, or 1 for the E4M3 forward, whose V is bf16).
template <int D, int BN, int NT, int QB = 2>
struct FwdCfg {
  static constexpr int kStages = (D == 64) ? 3 : 2;
  static constexpr int kQBytes = kBM * D * QB;  // one tile
  static constexpr int kKBytes = BN * D * QB;   // one K tile
  static constexpr int kKVBytes = BN * D * 2;   // one stage slot (V is 16-bit)
  static constexpr int kQKCols = D * QB / 128;  // 128-byte column blocks of Q / K
  static constexpr int kSmemData = NT * kQBytes + 2 * kStages * kKVBytes;
  // CTAs per SM: one tile with 64-key steps at d <= 128 fits two CTAs (TMEM
  // O + 2 S = 256 columns, ~97 KB of shared memory), so one CTA's set-up,
  // pipeline fill and epilogue overlap the other's work -- the short key
  // ranges of a sliding window gain from that.  Otherwise one CTA owns the
  // SM: at least ~120 KB of shared memory, all 512 TMEM columns.
  static constexpr int kCtas = (NT == 1 && D <= 128) ? 2 : 1;
  static constexpr int kSmem =
      kCtas == 2 ? kSmemData + 1024
                 : (kSmemData + 1024 > 120 * 1024 ? kSmemData + 1024 : 120 * 1024);
  static constexpr int kSCol0 = NT * D;
  static constexpr uint32_t kTmemCols = kCtas == 2 ? 256 : 512;
  // NT = 2: warpgroup 0 = producer, MMA and two idle warps; warpgroups 1-2 =
  // softmax.  NT = 1: warps 0-1 = producer, MMA; warps 2-5 = softmax.
  static constexpr int kThreads = NT == 2 ? 384 : 192;
  static constexpr int kSoftmaxWarp0 = NT == 2 ? 4 : 2;
  static_assert(NT * D + 2 * BN <= (int)kTmemCols, "TMEM budget");
  static_assert(kCtas == 1 || 2 * kSmem <= 227 * 1024, "shared memory of two CTAs");
};

struct Shared {
  uint64_t q_full;
  uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];
  uint64_t s_full[2], p_full[2], o_done[2];
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

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_bar(Shared &sh, uint64_t *bar, uint32_t parity, int *err) {
  return mbar_wait_bounded(smem_u32(bar), parity, &sh.abort, err, sh.wait_ns);
}

// The same wait taken by a whole warp with one answer, so warp-collective
// tcgen05 loads/stores that follow are never reached by part of a warp.
__device__ __forceinline__ bool wait_warp(Shared &sh, uint64_t *bar, uint32_t parity, int *err) {
  return __all_sync(0xffffffffu, wait_bar(sh, bar, parity, err));
}

template <typename T> struct IsBf16 { static constexpr int v = 0; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr int v = 1; };

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b) { return Elem<T>::from_f2(a, b); }

template <typename T, int D, int BN, int NT, int QB>
__global__ void __launch_bounds__(FwdCfg<D, BN, NT, QB>::kThreads, FwdCfg<D, BN, NT, QB>::kCtas)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdArgs a, const int m_blocks) {
  using C = FwdCfg<D, BN, NT, QB>;
  constexpr int ST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *q_s = smem;
  uint8_t *k_s = smem + NT * C::kQBytes;
  uint8_t *v_s = k_s + ST * C::kKVBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // PackGQA (Inference Cookbook FAQ Q15): with pg = g, tile row r holds
  // position r / pg of the tile and query head r % pg of the KV head's group.
  const int pg = a.pack > 1 ? a.pack : 1;
  const int tile_pos = kBM / pg;  // query positions per 128-row tile
  // CTA -> (query block, batch, head or KV head): heaviest blocks first,
  // heads fastest.
  const int nh = pg > 1 ? a.hkv : a.hq;
  const int bid = blockIdx.x;
  const int hh = bid % nh;
  const int b = (bid / nh) % a.batch;
  const int mb = m_blocks - 1 - bid / (nh * a.batch);
  int q0, lq, k0, lk;
  if (!a.seqs.get(b, q0, lq, k0, lk, a.err)) return;
  const int m0 = mb * (tile_pos * NT);  // first query position of the CTA
  if (m0 >= lq) return;
  const int kvh = pg > 1 ? hh : hh / (a.hq / a.hkv);
  const int h = pg > 1 ? kvh * pg : hh;  // (first) query head of the tile rows

  // Key tiles each query tile may see: [t_lo, t_hi] from its first and last
  // valid rows (the visible range's ends never decrease down the rows), and
  // their union [n_lo, n_lo + nt), which the producer streams.  Tile t runs
  // the steps [ta, tb) of the union, so a tile never computes a key tile
  // that none of its rows sees (e.g. the diagonal tile of the next query
  // tile under a causal mask, or the tiles left of a sliding window).
  auto tile_keys = [&](int t, int &t_lo, int &t_hi) {
    const int first = m0 + t * tile_pos, last = min(first + tile_pos, lq) - 1;
    t_lo = 0;
    t_hi = -1;
    if (first < lq) {
      int lo_f, hi_f, lo_l, hi_l;
      key_range(first, lq, lk, a.win_l, a.win_r, lo_f, hi_f);
      key_range(last, lq, lk, a.win_l, a.win_r, lo_l, hi_l);
      if (hi_l >= lo_f && hi_l >= 0) {
        t_lo = lo_f / BN;
        t_hi = hi_l / BN;
      }
    }
  };
  int n_lo = 0, nt = 0;
  {
    int u_lo = INT_MAX, u_hi = -1;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      int t_lo, t_hi;
      tile_keys(t, t_lo, t_hi);
      if (t_hi >= t_lo) {
        u_lo = min(u_lo, t_lo);
        u_hi = max(u_hi, t_hi);
      }
    }
    if (u_hi >= 0) {
      n_lo = u_lo;
      nt = u_hi - u_lo + 1;
    }
  }
  // steps [ta, tb) of the union that tile t takes part in
  auto tile_steps = [&](int t, int &ta, int &tb) {
    int t_lo, t_hi;
    tile_keys(t, t_lo, t_hi);
    ta = t_hi >= t_lo ? t_lo - n_lo : 0;
    tb = t_hi >= t_lo ? t_hi - n_lo + 1 : 0;
  };

  if (threadIdx.x == 0) {
    mbar_init(&sh.q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&sh.k_full[s], 1);
      mbar_init(&sh.k_empty[s], 1);
      mbar_init(&sh.v_full[s], 1);
      mbar_init(&sh.v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.s_full[s], 1);
      mbar_init(&sh.p_full[s], kBM);
      mbar_init(&sh.o_done[s], 1);
    }
    mbar_init(&sh.all_done, 1);
    sh.wait_ns = a.wait_ns;
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  // NT = 2 is launched at 168 registers a thread (12 warps).  The producer/MMA
  // warpgroup gives registers to the softmax warpgroups, which hold a whole
  // 128-score row: 128 * 88 + 256 * 208 = 384 * 168 (88 is the least at
  // which the MMA issuer's loop needs no spill).  Each setmaxnreg sits at the
  // head of its warpgroup's branch, so every role's code is compiled for its
  // own register budget.
  if (warp < C::kSoftmaxWarp0) {
  if constexpr (NT == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // (no key tile visible: nothing is loaded, so no copy outlives the CTA)
    if (elect_one() && nt > 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      mbar_expect_tx(&sh.q_full, NT * C::kQBytes);
      for (int t = 0; t < NT; ++t)
        for (int c = 0; c < C::kQKCols; ++c)  // 128-byte column blocks
          tma_load_3d(q_s + t * C::kQBytes + c * kBM * 128, &tq, &sh.q_full, c * (128 / QB), h,
                      q0 + m0 + t * tile_pos);
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int st = j % ST;
        const uint32_t ph = (j / ST) & 1;
        const int krow = k0 + (n_lo + j) * BN;
        if (!wait_bar(sh, &sh.k_empty[st], ph ^ 1, a.err)) break;
        mbar_expect_tx(&sh.k_full[st], C::kKBytes);
        for (int c = 0; c < C::kQKCols; ++c)
          tma_load_3d(k_s + st * C::kKVBytes + c * BN * 128, &tk, &sh.k_full[st], c * (128 / QB),
                      kvh, krow);
        if (!wait_bar(sh, &sh.v_empty[st], ph ^ 1, a.err)) { issued = 2 * j + 1; break; }
        mbar_expect_tx(&sh.v_full[st], C::kKVBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(v_s + st * C::kKVBytes + c * BN * 128, &tv, &sh.v_full[st], c * 64, kvh,
                      krow);
        issued = 2 * j + 2;
      }
      if (*(volatile int *)&sh.abort) {
        // let this CTA's copies in flight land before the CTA exits
        int *noerr = nullptr;
        mbar_wait(&sh.q_full, 0, noerr);
        for (int x = max(0, issued - 2 * ST); x < issued; ++x) {
          const int j = x / 2, st = j % ST;
          mbar_wait(x % 2 ? &sh.v_full[st] : &sh.k_full[st], (j / ST) & 1, noerr);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr int ab = IsBf16<T>::v;
      constexpr uint32_t id_s = QB == 1 ? idesc_e4m3(kBM, BN) : idesc_f16(kBM, BN, ab, 0, 0);
      constexpr uint32_t id_o = idesc_f16(kBM, D, ab, 0, 1);
      const uint32_t q_addr = smem_u32(q_s), k_addr = smem_u32(k_s), v_addr = smem_u32(v_s);
      // descriptor bases; every operand below is base + constant offset
      const uint64_t q_d = smem_desc(q_addr, 16, 1024), k_d = smem_desc(k_addr, 16, 1024);
      const uint64_t v_d = smem_desc(v_addr, BN * 128, 1024);
      // S_t = Q_t K_j^T into TMEM column `dcol`
      // (each instruction takes 32 bytes of every row: 16 elements at 16 bits,
      // 32 at 8 bits)
      auto mma_s = [&](int t, int j, uint32_t dcol) {
        const uint32_t ko = (j % ST) * C::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < D * QB / 32; ++kk) {
          const uint64_t ad = desc_add(q_d, t * C::kQBytes + (kk / 4) * (kBM * 128) + (kk % 4) * 32);
          const uint64_t bd = desc_add(k_d, ko + (kk / 4) * (BN * 128) + (kk % 4) * 32);
          if constexpr (QB == 1)
            mma_ss_e4m3(dcol, ad, bd, id_s, kk > 0);
          else
            mma_ss(dcol, ad, bd, id_s, kk > 0);
        }
      };
      // O_t (+)= P V_j with P read from TMEM column `pcol`; `first`: the
      // tile's first key tile, which starts the accumulation
      auto mma_pv = [&](int t, int j, uint32_t pcol, bool first) {
        const uint32_t vo = (j % ST) * C::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bd = desc_add(v_d, vo + kk * 16 * 128);
          mma_ts(tmem + t * D, pcol + kk * 8, bd, id_o, (!first || kk > 0) ? 1u : 0u);
        }
      };
      auto k_ready = [&](int j) {
        const bool r = wait_bar(sh, &sh.k_full[j % ST], (j / ST) & 1, a.err);
        tc_fence_after();
        return r;
      };
      auto v_ready = [&](int j) {
        const bool r = wait_bar(sh, &sh.v_full[j % ST], (j / ST) & 1, a.err);
        tc_fence_after();
        return r;
      };
      int ta[NT], tb[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) tile_steps(t, ta[t], tb[t]);
      // test hook: all_done completes only after this thread's last commit,
      // so this wait can only run out (then every role takes the abort path)
      const bool stalled = a.stall && !wait_bar(sh, &sh.all_done, 0, a.err);
      if (stalled) {
      } else if (NT == 2) {
        // S_0(0) S_1(0) | PV_0(j) S_0(j+1) PV_1(j) S_1(j+1) | ..., where a
        // tile takes part in step j only inside its own range [ta, tb).
        // Every K and V tile of the union is waited for once before its
        // stage is released, whether or not a tile used it.
        bool ok = nt == 0 || (wait_bar(sh, &sh.q_full, 0, a.err) && k_ready(0));
        if (ok && nt > 0) {
          for (int t = 0; t < NT; ++t) {
            if (ta[t] == 0 && tb[t] > 0) {
              mma_s(t, 0, tmem + C::kSCol0 + t * BN);
              mma_commit(&sh.s_full[t]);
            }
          }
          mma_commit(&sh.k_empty[0]);
        }
        for (int j = 0; ok && j < nt; ++j) {
          const bool k_next = j + 1 < nt;
          // the last tile that reads V_j / K_{j+1} releases its stage
          const int last_pv = (j >= ta[1] && j < tb[1]) ? 1 : 0;
          const int last_s = (j + 1 >= ta[1] && j + 1 < tb[1]) ? 1 : 0;
          bool v_in = false, k_in = false;
          for (int t = 0; t < NT && ok; ++t) {
            const uint32_t scol = tmem + C::kSCol0 + t * BN;
            if (j >= ta[t] && j < tb[t]) {
              if (!wait_bar(sh, &sh.p_full[t], (j - ta[t]) & 1, a.err)) { ok = false; break; }
              tc_fence_after();
              if (!v_in && !(v_in = v_ready(j))) { ok = false; break; }
              mma_pv(t, j, scol, j == ta[t]);
              mma_commit(&sh.o_done[t]);
              if (t == last_pv) mma_commit(&sh.v_empty[j % ST]);
            }
            if (k_next && j + 1 >= ta[t] && j + 1 < tb[t]) {
              if (!k_in && !(k_in = k_ready(j + 1))) { ok = false; break; }
              mma_s(t, j + 1, scol);
              mma_commit(&sh.s_full[t]);
              if (t == last_s) mma_commit(&sh.k_empty[(j + 1) % ST]);
            }
          }
          // a tile of the union that no query tile read still has to land
          // before its stage is handed back
          if (ok && !v_in) {
            if (!v_ready(j)) break;
            mma_commit(&sh.v_empty[j % ST]);
          }
          if (ok && k_next && !k_in) {
            if (!k_ready(j + 1)) break;
            mma_commit(&sh.k_empty[(j + 1) % ST]);
          }
        }
      } else {
        bool ok = nt == 0 || (wait_bar(sh, &sh.q_full, 0, a.err) && k_ready(0));
        if (ok && nt > 0) {
          mma_s(0, 0, tmem + C::kSCol0);
          mma_commit(&sh.s_full[0]);
          mma_commit(&sh.k_empty[0]);
        }
        for (int j = 0; ok && j < nt; ++j) {
          if (j + 1 < nt) {
            if (!k_ready(j + 1)) break;
            mma_s(0, j + 1, tmem + C::kSCol0 + ((j + 1) & 1) * BN);
            mma_commit(&sh.s_full[(j + 1) & 1]);
            mma_commit(&sh.k_empty[(j + 1) % ST]);
          }
          if (!wait_bar(sh, &sh.p_full[j & 1], (j >> 1) & 1, a.err)) break;
          tc_fence_after();
          if (!v_ready(j)) break;
          mma_pv(0, j, tmem + C::kSCol0 + (j & 1) * BN, j == 0);
          mma_commit(&sh.o_done[0]);
          mma_commit(&sh.v_empty[j % ST]);
        }
      }
      // completes when every MMA above has; after an abort, wait for it so
      // that no MMA still reads shared memory or writes TMEM when the CTA
      // releases its TMEM and exits
      mma_commit(&sh.all_done);
      if (*(volatile int *)&sh.abort) {
        int *noerr = nullptr;
        mbar_wait(&sh.all_done, 0, noerr);
      }
    }
  }
  } else {
    if constexpr (NT == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 208;" ::: "memory");
    // ------------------------------------------------------------ softmax
    const int t = (warp - C::kSoftmaxWarp0) >> 2;  // query tile of this warpgroup
    const int r = 32 * (warp & 3) + lane;  // TMEM lane = row in the tile
    const int i = m0 + t * tile_pos + r / pg;  // its query position
    const int hr = h + r % pg;                 // and query head
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t o_t = tmem + lane_off + t * D;
    int lo_i, hi_i;
    key_range(i, lq, lk, a.win_l, a.win_r, lo_i, hi_i);
    const uint32_t n_vis = (uint32_t)max(hi_i - lo_i + 1, 0);  // keys this row sees
    // tiles that need no mask: every row of the tile sees every key in them
    int lo_tile_max, hi_tile_min, dummy;
    key_range(m0 + t * tile_pos + tile_pos - 1, lq, lk, a.win_l, a.win_r, lo_tile_max, dummy);
    key_range(m0 + t * tile_pos, lq, lk, a.win_l, a.win_r, dummy, hi_tile_min);
    const float sl2 = a.scale * kLog2e;
    const bool cap = a.softcap > 0.f;
    const float cap_in = cap ? a.scale / a.softcap : 0.f, cap_out = a.softcap * kLog2e;
    const float cap_k = cap_in * 2.8853900817779268f;  // 2 log2(e) cap_in
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    // this tile's own key tiles: n_lo + ta + j for j in [0, ntt)
    int ta, tb;
    tile_steps(t, ta, tb);
    const int ntt = tb - ta;
    for (int j = 0; j < ntt; ++j) {
      const int key0 = (n_lo + ta + j) * BN;
      const int sb = NT == 2 ? t : (j & 1);                 // S/P buffer and its barriers
      const uint32_t s_par = NT == 2 ? (j & 1) : ((j >> 1) & 1);
      if (!wait_warp(sh, &sh.s_full[sb], s_par, a.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t scol = tmem + lane_off + C::kSCol0 + sb * BN;
      float x[BN];
      {
        uint32_t u[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          tmem_ld32(scol + c * 32, *reinterpret_cast<uint32_t(*)[32]>(u + c * 32));
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < BN; ++e) x[e] = __uint_as_float(u[e]);
      }
      // softcap, then the mask (Inference Cookbook FAQ Q22 order)
      if (cap) {
        // c tanh(x cap_in) in log2 units = cap_out - 2 cap_out / (e^{2 x cap_in} + 1),
        // two scores at a time (the exponential and the reciprocal on MUFU)
        const uint64_t k2 = f2_pack(cap_k, cap_k), one2 = f2_pack(1.f, 1.f);
        const uint64_t co2 = f2_pack(cap_out, cap_out), mco2 = f2_pack(-2.f * cap_out, -2.f * cap_out);
#pragma unroll
        for (int e = 0; e < BN; e += 2) {
          float a0, a1, y0, y1;
          f2_unpack(f2_mul(f2_pack(x[e], x[e + 1]), k2), a0, a1);
          f2_unpack(f2_add(f2_pack(ex2(a0), ex2(a1)), one2), y0, y1);
          f2_unpack(f2_fma(f2_pack(rcp_approx(y0), rcp_approx(y1)), mco2, co2), x[e], x[e + 1]);
        }
      }
      const bool need_mask = key0 < lo_tile_max || key0 + BN - 1 > hi_tile_min;
      if (need_mask) {
        // visible: e - (lo_i - key0) in [0, n_vis), one unsigned compare per key
        const int e_lo = lo_i - key0;
#pragma unroll
        for (int e = 0; e < BN; ++e)
          if ((uint32_t)(e - e_lo) >= n_vis) x[e] = -INFINITY;
      }
      // raw-score max: scale and softcap preserve the order (scale >= 0);
      // eight independent partial maxima of three-input maxes keep the
      // dependency chains short
      float mp[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mp[u] = x[u];
#pragma unroll
      for (int e = 8; e + 16 <= BN; e += 16) {
#pragma unroll
        for (int u = 0; u < 8; ++u) mp[u] = fmax3(mp[u], x[e + u], x[e + 8 + u]);
      }
      if constexpr ((BN - 8) % 16 != 0) {
#pragma unroll
        for (int u = 0; u < 8; ++u) mp[u] = fmaxf(mp[u], x[BN - 8 + u]);
      }
      const float mt = fmaxf(fmax3(mp[0], mp[1], mp[2]),
                             fmax3(fmax3(mp[3], mp[4], mp[5]), mp[6], mp[7]));
      const float f = cap ? 1.f : sl2;  // x * f is the score in log2 units
      const float m_new = fmaxf(m_ref, mt * f);
      const bool rescale = m_new > m_ref + kRescaleThreshold;
      float alpha = 1.f;
      if (rescale) {
        alpha = ex2(m_ref - m_new);
        l *= alpha;
        m_ref = m_new;
      }
      const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
      // t = x f - m and the row sums two at a time (packed f32x2)
      const uint64_t f2 = f2_pack(f, f), nm2 = f2_pack(neg_m, neg_m);
      uint64_t rs[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) rs[u] = 0ull;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int el = c * 32 + 2 * e;
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(x[el], x[el + 1]), f2, nm2), t0, t1);
          const float p0 = ex2(t0), p1 = ex2(t1);
          rs[e & 3] = f2_add(rs[e & 3], f2_pack(p0, p1));
          pk[e] = pack2<T>(p0, p1);
        }
        tmem_st16(scol + c * 16, pk);
      }
      {
        float r[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) f2_unpack(rs[u], r[2 * u], r[2 * u + 1]);
        l += ((r[0] + r[1]) + (r[2] + r[3])) + ((r[4] + r[5]) + (r[6] + r[7]));
      }
      tmem_wait_st();
      if (j > 0) {
        // O holds P_{j-1} V_{j-1} once this completes; only then may it be rescaled
        if (!wait_warp(sh, &sh.o_done[t], (j - 1) & 1, a.err)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld32(o_t + c * 32, u);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            tmem_st32(o_t + c * 32, u);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(&sh.p_full[sb]);
    }
    // epilogue: O / l -> dtype, LSE = ln(sum exp(s))
    if (ok && ntt > 0) ok = wait_warp(sh, &sh.o_done[t], (ntt - 1) & 1, a.err);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
      // (out_scale: the V descale of the FP8 forward)
      const float inv = l > 0.f ? (a.out_scale > 0.f ? a.out_scale : 1.f) / l : 0.f;
      T *orow = static_cast<T *>(a.o) + ((int64_t)(q0 + i) * a.hq + hr) * D;
      const bool valid = i < lq;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        if (ntt > 0) {
          tmem_ld32(o_t + c * 32, u);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack2<T>(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
        if (valid) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      if (valid) {
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        a.lse[a.seqs.lse_index(b, hr, q0, i)] = l > 0.f ? (m_use + __log2f(l)) * kLn2 : -INFINITY;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

template <typename T, int D, int BN, int NT, int QB = 2>
cudaError_t fwd_tc(const FwdArgs &a, cudaStream_t st) {
  using C = FwdCfg<D, BN, NT, QB>;
  const int qk_dtype = QB == 1 ? kDtypeE4M3 : a.dtype;
  const int64_t rows_q = a.seqs.cu_q ? a.seqs.total_q : (int64_t)a.batch * a.seqs.sq;
  const int64_t rows_k = a.seqs.cu_k ? a.seqs.total_k : (int64_t)a.batch * a.seqs.sk;
  if (rows_k == 0) return launch_fwd_simt(a, st);  // no keys: every row is empty
  CUtensorMap tq, tk, tv;
  const int pg = a.pack > 1 ? a.pack : 1;
  if (kBM % pg != 0) return cudaErrorInvalidValue;
  if (!make_map_3d(&tq, a.q, qk_dtype, rows_q, a.hq, D, kBM / pg, a.q_rs, pg) ||
      !make_map_3d(&tk, a.k, qk_dtype, rows_k, a.hkv, D, BN, a.k_rs) ||
      !make_map_3d(&tv, a.v, a.dtype, rows_k, a.hkv, D, BN, a.v_rs))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_once<fwd_tc_kernel<T, D, BN, NT, QB>>(C::kSmem);
  if (e == cudaSuccess && NT == 2)  // 128 * 88 + 256 * 208 after setmaxnreg
    e = check_regs_once<fwd_tc_kernel<T, D, BN, NT, QB>>(C::kThreads, 128 * 88 + 256 * 208);
  if (e != cudaSuccess) return e;
  const int block_pos = kBM / pg * NT;  // query positions per CTA
  const int m_blocks = (a.seqs.sq + block_pos - 1) / block_pos;
  const int64_t grid = (int64_t)m_blocks * (pg > 1 ? a.hkv : a.hq) * a.batch;
  if (grid == 0) return cudaSuccess;
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  debug_log("forward: fwd_tc_kernel d=%d, %d query tile(s) of 128 rows per CTA, %d-key tiles, "
            "%d-stage K/V ring, QK^T %s, pack_gqa=%d, grid=%lld CTAs x %d threads, smem=%d B",
            D, NT, BN, C::kStages, QB == 1 ? "e4m3 (kind::f8f6f4)" : "16-bit (kind::f16)", pg,
            (long long)grid, C::kThreads, C::kSmem);
  fwd_tc_kernel<T, D, BN, NT, QB><<<(unsigned)grid, C::kThreads, C::kSmem, st>>>(tq, tk, tv, a,
                                                                          m_blocks);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs &a, cudaStream_t st) {
  const bool bf = a.dtype == ATTN_BF16;
  switch (a.d) {
    // d = 64: one tile with 64-key steps and two CTAs per SM at every length
    // (measured 4-6% faster than two tiles per CTA on long sequences, ~20%
    // on short or windowed ones)
    case 64: return bf ? fwd_tc<__nv_bfloat16, 64, 64, 1>(a, st) : fwd_tc<__half, 64, 64, 1>(a, st);
    case 128:
      if (a.qk_fp8) return bf ? fwd_tc<__nv_bfloat16, 128, 128, 2, 1>(a, st) : cudaErrorInvalidValue;
      // a window of at most 1024 keys (besides the tile itself) or sequences
      // of at most 1024 keys: short key ranges, one 128-row tile per CTA and
      // two CTAs per SM
      if ((a.win_l >= 0 && a.win_r >= 0 && a.win_l + a.win_r <= 1024) || a.seqs.sk <= 1024)
        return bf ? fwd_tc<__nv_bfloat16, 128, 64, 1>(a, st) : fwd_tc<__half, 128, 64, 1>(a, st);
      return bf ? fwd_tc<__nv_bfloat16, 128, 128, 2>(a, st) : fwd_tc<__half, 128, 128, 2>(a, st);
    case 256: return bf ? fwd_tc<__nv_bfloat16, 256, 64, 1>(a, st) : fwd_tc<__half, 256, 64, 1>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
