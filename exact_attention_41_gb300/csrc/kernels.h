// Internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"

namespace attn {

// One dense or packed (varlen) attention problem.
struct FwdArgs {
  const void *q, *k, *v;
  void *o;
  float *lse;
  Seqs seqs;
  int batch, hq, hkv, d, dtype;
  float scale, softcap;  // softcap <= 0: off
  int win_l, win_r;      // -1 = unbounded; causal already folded into win_r = 0
  int *err;              // device error word
  // elements between consecutive tokens of q, k, v (row r of head h starts
  // at r * stride + h * d); hq*d / hkv*d when contiguous, larger for packed
  // qkv / kv layouts.  Set by the C ABI before any launch.
  int64_t q_rs, k_rs, v_rs;
  // PackGQA: 1, or g = hq / hkv when the g query heads of one KV head share
  // every 128-row tile (128 / g positions x g heads).  Set by the C ABI.
  int pack;
  // FP8 forward: q and k hold E4M3 values (S runs as kind::f8f6f4), v is the
  // bf16 widening of E4M3 values, and the output is multiplied by out_scale
  // (the V descale).  0 / 0.f: the plain 16-bit forward.
  int qk_fp8;
  float out_scale;
  // wall-clock limit of a device-side wait (ns); set by the C ABI
  uint64_t wait_ns;
  // test hook (attn_set_test_stall): the MMA issuer first waits on a barrier
  // that nothing completes, so the wait limit runs out
  int stall;
};

// Storage code of E4M3 tensors for make_map_3d (beside ATTN_F16 / ATTN_BF16).
constexpr int kDtypeE4M3 = 2;

struct BwdArgs {
  FwdArgs f;             // f.o / f.lse are the forward's outputs (read only)
  const void *dout;
  void *dq, *dk, *dv;
  float *dsum;           // workspace: D_i = rowsum(dO * O), LSE layout
  float *nlse2;          // workspace: -LSE_i * log2(e), LSE layout (tensor-core path)
  float *dq_acc;         // workspace: fp32 dQ accumulator (hq, rows, d) (atomic mode)
  int deterministic;
  int64_t dq_rs, dk_rs, dv_rs;  // token strides of the gradients (as q_rs ...)
};

struct DecodeArgs {
  const void *q;
  void *k_cache, *v_cache;
  const void *k_new, *v_new;
  const int32_t *cache_seqlens, *block_table;
  int num_pages, page_size, max_pages;
  void *o;
  float *lse;
  int dtype, b, sq, s_new, hq, hkv, d;
  float scale, softcap;
  int win_l, win_r;
  int num_splits, split_chunk;  // keys per split (multiple of 128)
  float *o_part;                // (splits, b, sq, hq, d) fp32 when num_splits > 1
  float *lse_part;              // (splits, b, hq, sq)
  int *err;
  uint64_t wait_ns;             // wall-clock limit of a device-side wait (ns)
  int stall;                    // test hook, as FwdArgs::stall
};

// cuTensorMapEncodeTiled from the driver (looked up once), or nullptr.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
// 3-D (rows, heads, d) tensor map, box {64, box_heads, box_rows}, 128-byte
// swizzle (a box lands as box_rows * box_heads rows of 128 bytes, head-minor).
// row_stride: elements between consecutive rows (0: heads * d, contiguous).
bool make_map_3d(CUtensorMap *m, const void *base, int dtype, int64_t rows, int heads, int d,
                 int box_rows, int64_t row_stride = 0, int box_heads = 1);
// Tensor-core decode; cudaErrorNotSupported for shapes it does not handle.
cudaError_t launch_decode_tc(const DecodeArgs &a, cudaStream_t st);

// Adds n to the library's launch counter (attn_launch_count).
void count_launches(int n);

// LIBATTN_DEBUG set to a non-zero number in the environment (read once, at
// the first use) makes every launcher print the kernel, tile shape, pack
// factor or split count and grid it chose, one line on stderr per launch
// decision (the counterpart of FLASH_ATTN_DEBUG in Inference Cookbook FAQ
// Q13).  debug_log is printf-like and does nothing when it is off.
bool debug_enabled();
void debug_log(const char *fmt, ...);

// Raises `Kernel`'s dynamic shared memory limit to `bytes`, once per device:
// later calls (including ones made during CUDA graph capture) only read a
// flag.
template <auto Kernel>
cudaError_t set_smem_once(int bytes) {
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Kernels whose warpgroups move registers between them with setmaxnreg need
// the CTA to be launched with at least `needed` registers in all (threads x
// registers a thread, the latter as compiled, rounded up to 8): a split
// above that would leave an increase waiting forever.  Checked once per
// process from the compiled kernel; a kernel that fails it is not launched.
template <auto Kernel>
cudaError_t check_regs_once(int threads, int needed) {
  static std::atomic<int> state{0};  // 0 unknown, 1 fits, 2 does not
  int s = state.load(std::memory_order_acquire);
  if (s == 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, Kernel);
    if (e != cudaSuccess) return e;
    const int regs = (fa.numRegs + 7) / 8 * 8;
    s = regs * threads >= needed ? 1 : 2;
    if (s == 2)
      debug_log("register split of %d needs %d registers a CTA; compiled with %d a thread x %d",
                needed, needed, fa.numRegs, threads);
    state.store(s, std::memory_order_release);
  }
  return s == 1 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t launch_fwd_simt(const FwdArgs &a, cudaStream_t st);
cudaError_t launch_fwd_tc(const FwdArgs &a, cudaStream_t st);
// dQ of the backward, query-stationary (d = 64, 128, 256): written once, no atomics.
cudaError_t launch_bwd_dq_tc(const BwdArgs &a, cudaStream_t st);
// Backward on the tensor cores (d = 64, 128, 256): preprocess, key-stationary
// dK/dV kernel (with atomic dQ unless deterministic), dQ finish.
cudaError_t launch_bwd_tc(const BwdArgs &a, int sms, cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st);
// E4M3 -> bf16 widening of n (a multiple of 16) contiguous values.
cudaError_t launch_widen_e4m3(const void *src, void *dst, int64_t n, int sms, cudaStream_t st);
// Debug probability matrix p (b, hq, sq, sk) fp32 from q, k and a.lse.
cudaError_t launch_probs(const FwdArgs &a, float *p, cudaStream_t st);
// cache_seqlens[i] += s_new for i < b.
cudaError_t launch_kvcache_advance(int32_t *cache_seqlens, int b, int s_new, cudaStream_t st);

}  // namespace attn
