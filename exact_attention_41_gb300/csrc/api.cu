// The libattn C ABI: argument validation, workspace sizing and dispatch.
// Declarations and the contract of every entry point are in include/libattn.h.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>

#include "kernels.h"

namespace attn {
namespace {

// Sticky device error word, one per device that loads the library.
__device__ int g_device_error;

// Wall-clock limit of one device-side wait, read by every call
// (attn_set_wait_limit_ns).
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

// attn_set_test_stall: read by every call into its kernel arguments.
std::atomic<int> g_test_stall{0};
int test_stall() { return g_test_stall.load(std::memory_order_relaxed); }

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int sms = 0;
  int *err = nullptr;
  bool ready = false;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Per-device facts, looked up once (thread safe).  Does not allocate or
// synchronise, so it is safe inside stream capture after the first call.
const DeviceInfo *device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo &di = g_dev[dev];
  if (!di.ready) {
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return nullptr;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    di.err = static_cast<int *>(p);
    di.ready = true;
  }
  return &di;
}

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Checks shared by every entry point.  win_r is normalised (causal -> 0).
attn_status check_common(int dtype, int hq, int hkv, int d, float scale, int win_l, int &win_r,
                         int causal, float softcap) {
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return ATTN_ERR_INVALID;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (!isfinite(scale) || scale < 0.f) return ATTN_ERR_INVALID;
  if (isnan(softcap)) return ATTN_ERR_INVALID;
  if (win_l < -1 || win_r < -1) return ATTN_ERR_INVALID;
  if (causal) win_r = 0;
  return ATTN_OK;
}

// Token strides in elements; 0 means contiguous (heads * d).  A given stride
// must hold a whole row of heads and keep 16-byte alignment (TMA).
bool stride_ok(int64_t rs, int heads, int d) {
  return rs == 0 || (rs >= (int64_t)heads * d && rs % 8 == 0 && rs <= (int64_t)1 << 40);
}
void set_strides(FwdArgs &a, int64_t q_rs, int64_t k_rs, int64_t v_rs) {
  a.q_rs = q_rs ? q_rs : (int64_t)a.hq * a.d;
  a.k_rs = k_rs ? k_rs : (int64_t)a.hkv * a.d;
  a.v_rs = v_rs ? v_rs : (int64_t)a.hkv * a.d;
}
void set_grad_strides(BwdArgs &a, int64_t dq_rs, int64_t dk_rs, int64_t dv_rs) {
  a.dq_rs = dq_rs ? dq_rs : (int64_t)a.f.hq * a.f.d;
  a.dk_rs = dk_rs ? dk_rs : (int64_t)a.f.hkv * a.f.d;
  a.dv_rs = dv_rs ? dv_rs : (int64_t)a.f.hkv * a.f.d;
}

// PackGQA (Inference Cookbook FAQ Q15): the g = hq / hkv query heads of a
// KV head share every 128-row tile of the forward.  pack_gqa < 0: automatic
// -- on when the query sequences are short (<= 128 rows, where an unpacked
// 256-row query block is mostly empty), off for long ones, where the FAQ
// notes packing can be slightly slower; 0: off; > 0: on.  Returns the pack
// factor, or 0 when packing is asked for but g does not divide 128.
int resolve_pack(int pack_gqa, int hq, int hkv, int max_sq) {
  const int g = hq / hkv;
  const bool can = g > 1 && 128 % g == 0;
  if (pack_gqa == 0 || g == 1) return 1;
  if (pack_gqa > 0) return can ? g : 0;
  return can && max_sq <= 128 ? g : 1;
}

attn_status launched(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// Backward workspace for `rows` query rows in total: D_i and -LSE_i log2(e)
// (fp32, LSE layout each) and, unless deterministic, the fp32 dQ
// accumulator of the key-stationary kernel's atomic adds.
size_t bwd_ws_bytes(int64_t rows, int hq, int d, int deterministic) {
  return 2 * align256(sizeof(float) * rows * hq) +
         (deterministic ? 0 : align256(sizeof(float) * rows * hq * d));
}

// Splits a backward workspace and launches the backward kernels.
attn_status run_bwd(BwdArgs &a, int64_t rows, void *workspace, const DeviceInfo *di,
                    cudaStream_t stream) {
  char *ws = static_cast<char *>(workspace);
  const int hq = a.f.hq;
  a.dsum = reinterpret_cast<float *>(ws);
  ws += align256(sizeof(float) * rows * hq);
  a.nlse2 = reinterpret_cast<float *>(ws);
  ws += align256(sizeof(float) * rows * hq);
  a.dq_acc = a.deterministic ? nullptr : reinterpret_cast<float *>(ws);
  a.f.wait_ns = wait_limit_ns();
  a.f.stall = test_stall();
  return launched(launch_bwd_tc(a, di->sms, stream));
}

int resolve_splits(int b, int hkv, int max_seqlen_k, int num_splits, int sms) {
  const int max_useful = max(1, (max_seqlen_k + 127) / 128);
  if (num_splits > 0) return min(num_splits, min(max_useful, 256));
  // Inference Cookbook FAQ Q14: enough (batch, kv head) units -> one split;
  // fewer units than SMs -> split until near the SM count; long caches ->
  // split so each piece streams a bounded key range.
  const int units = max(1, b * hkv);
  // A piece of 8192 keys (64 tiles) amortises a CTA's start and epilogue;
  // on the paged decode workload (b=64, hkv=8, caches up to 32K) 4-5 splits
  // stream at ~6 TB/s and 17 splits of 2048 keys at 5.2 TB/s.
  if (units >= sms && max_seqlen_k <= 8192) return 1;
  int s = (max_seqlen_k + 8191) / 8192;
  s = max(s, (sms + units - 1) / units);
  return max(1, min(min(s, 64), max_useful));
}

std::atomic<unsigned long long> g_launches{0};

}  // namespace

void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

bool debug_enabled() {
  static const bool on = [] {
    const char *e = getenv("LIBATTN_DEBUG");
    return e != nullptr && atoi(e) != 0;
  }();
  return on;
}

void debug_log(const char *fmt, ...) {
  if (!debug_enabled()) return;
  char line[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(line, sizeof line, fmt, ap);
  va_end(ap);
  fprintf(stderr, "libattn: %s\n", line);
}

}  // namespace attn

using namespace attn;

extern "C" {

const char *attn_version(void) { return "libattn 0.1.0 (sm_103a)"; }

const char *attn_status_str(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
    case ATTN_ERR_DEVICE: return "device-side data check failed";
  }
  return "unknown status";
}

attn_status attn_fwd_strided(const void *q, const void *k, const void *v, void *out, float *lse,
                             int64_t q_row_stride, int64_t k_row_stride, int64_t v_row_stride,
                             int dtype, int b, int sq, int sk, int hq, int hkv, int d,
                             float scale, int causal, int win_l, int win_r, float softcap,
                             int pack_gqa, attn_stream_t stream) {
  attn_status st = check_common(dtype, hq, hkv, d, scale, win_l, win_r, causal, softcap);
  if (st != ATTN_OK) return st;
  if (!stride_ok(q_row_stride, hq, d) || !stride_ok(k_row_stride, hkv, d) ||
      !stride_ok(v_row_stride, hkv, d))
    return ATTN_ERR_INVALID;
  if (b < 0 || sq < 0 || sk < 0) return ATTN_ERR_INVALID;
  if (b == 0 || sq == 0) return ATTN_OK;
  if (!q || !out || !lse || (sk > 0 && (!k || !v))) return ATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return ATTN_ERR_INVALID;
  if ((int64_t)b * sq * hq > INT32_MAX || (int64_t)b * sk * hkv > INT32_MAX)
    return ATTN_ERR_UNSUPPORTED;
  const int pack = resolve_pack(pack_gqa, hq, hkv, sq);
  if (pack == 0) return ATTN_ERR_UNSUPPORTED;
  const DeviceInfo *di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  FwdArgs a{q, k, v, out, lse, Seqs{nullptr, nullptr, sq, sk, 0, 0, hq}, b, hq, hkv, d, dtype,
            scale, softcap > 0.f ? softcap : 0.f, win_l, win_r, di->err};
  set_strides(a, q_row_stride, k_row_stride, v_row_stride);
  a.wait_ns = wait_limit_ns();
  a.stall = test_stall();
  a.pack = pack;
  return launched(launch_fwd_tc(a, stream));
}

attn_status attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                     int dtype, int b, int sq, int sk, int hq, int hkv, int d, float scale,
                     int causal, int win_l, int win_r, float softcap, attn_stream_t stream) {
  return attn_fwd_strided(q, k, v, out, lse, 0, 0, 0, dtype, b, sq, sk, hq, hkv, d, scale, causal,
                          win_l, win_r, softcap, -1, stream);
}

size_t attn_bwd_workspace_size(int b, int sq, int sk, int hq, int hkv, int d, int deterministic) {
  (void)sk; (void)hkv;
  if (b <= 0 || sq <= 0 || hq <= 0 || d <= 0) return 0;
  return bwd_ws_bytes((int64_t)b * sq, hq, d, deterministic);
}

attn_status attn_bwd_strided(const void *q, const void *k, const void *v, const void *out,
                             const float *lse, const void *dout, void *dq, void *dk, void *dv,
                             int64_t q_row_stride, int64_t k_row_stride, int64_t v_row_stride,
                             int64_t dq_row_stride, int64_t dk_row_stride,
                             int64_t dv_row_stride, int dtype, int b, int sq, int sk, int hq,
                             int hkv, int d, float scale, int causal, int win_l, int win_r,
                             float softcap, int deterministic, void *workspace,
                             size_t workspace_bytes, attn_stream_t stream) {
  attn_status st = check_common(dtype, hq, hkv, d, scale, win_l, win_r, causal, softcap);
  if (st != ATTN_OK) return st;
  if (!stride_ok(q_row_stride, hq, d) || !stride_ok(k_row_stride, hkv, d) ||
      !stride_ok(v_row_stride, hkv, d) || !stride_ok(dq_row_stride, hq, d) ||
      !stride_ok(dk_row_stride, hkv, d) || !stride_ok(dv_row_stride, hkv, d))
    return ATTN_ERR_INVALID;
  if (b < 0 || sq < 0 || sk < 0) return ATTN_ERR_INVALID;
  if (b == 0 || (sq == 0 && sk == 0)) return ATTN_OK;
  if ((sq > 0 && (!q || !out || !lse || !dout || !dq)) || (sk > 0 && (!k || !v || !dk || !dv)))
    return ATTN_ERR_INVALID;
  for (const void *p : {q, k, v, out, (const void *)lse, dout, (const void *)dq, (const void *)dk,
                        (const void *)dv, (const void *)workspace})
    if (!aligned16(p)) return ATTN_ERR_INVALID;
  if ((int64_t)b * sq * hq > INT32_MAX || (int64_t)b * sk * hkv > INT32_MAX)
    return ATTN_ERR_UNSUPPORTED;
  const size_t need = attn_bwd_workspace_size(b, sq, sk, hq, hkv, d, deterministic);
  if (need > 0 && (!workspace || workspace_bytes < need)) return ATTN_ERR_WORKSPACE;
  const DeviceInfo *di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  BwdArgs a{FwdArgs{q, k, v, const_cast<void *>(out), const_cast<float *>(lse),
                    Seqs{nullptr, nullptr, sq, sk, 0, 0, hq}, b, hq, hkv, d, dtype, scale,
                    softcap > 0.f ? softcap : 0.f, win_l, win_r, di->err},
            dout, dq, dk, dv};
  a.deterministic = deterministic;
  set_strides(a.f, q_row_stride, k_row_stride, v_row_stride);
  set_grad_strides(a, dq_row_stride, dk_row_stride, dv_row_stride);
  return run_bwd(a, (int64_t)b * sq, workspace, di, stream);
}

attn_status attn_bwd(const void *q, const void *k, const void *v, const void *out,
                     const float *lse, const void *dout, void *dq, void *dk, void *dv,
                     int dtype, int b, int sq, int sk, int hq, int hkv, int d, float scale,
                     int causal, int win_l, int win_r, float softcap, int deterministic,
                     void *workspace, size_t workspace_bytes, attn_stream_t stream) {
  return attn_bwd_strided(q, k, v, out, lse, dout, dq, dk, dv, 0, 0, 0, 0, 0, 0, dtype, b, sq,
                          sk, hq, hkv, d, scale, causal, win_l, win_r, softcap, deterministic,
                          workspace, workspace_bytes, stream);
}

attn_status attn_fwd_varlen(const void *q, const void *k, const void *v, void *out, float *lse,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            int batch, int max_seqlen_q, int max_seqlen_k, int total_q,
                            int total_k, int dtype, int hq, int hkv, int d, float scale,
                            int causal, int win_l, int win_r, float softcap,
                            attn_stream_t stream) {
  attn_status st = check_common(dtype, hq, hkv, d, scale, win_l, win_r, causal, softcap);
  if (st != ATTN_OK) return st;
  if (batch < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_k < 0)
    return ATTN_ERR_INVALID;
  if (batch == 0 || total_q == 0 || max_seqlen_q == 0) return ATTN_OK;
  if (!q || !out || !lse || !cu_seqlens_q || !cu_seqlens_k || (total_k > 0 && (!k || !v)))
    return ATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return ATTN_ERR_INVALID;
  if ((int64_t)total_q * hq > INT32_MAX || (int64_t)total_k * hkv > INT32_MAX)
    return ATTN_ERR_UNSUPPORTED;
  const DeviceInfo *di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  FwdArgs a{q, k, v, out, lse,
            Seqs{cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, total_q, total_k, hq},
            batch, hq, hkv, d, dtype, scale, softcap > 0.f ? softcap : 0.f, win_l, win_r,
            di->err};
  set_strides(a, 0, 0, 0);
  a.wait_ns = wait_limit_ns();
  a.stall = test_stall();
  a.pack = resolve_pack(-1, hq, hkv, max_seqlen_q);
  return launched(launch_fwd_tc(a, stream));
}

size_t attn_bwd_varlen_workspace_size(int batch, int max_seqlen_q, int max_seqlen_k,
                                      int total_q, int total_k, int hq, int hkv, int d,
                                      int deterministic) {
  (void)max_seqlen_q; (void)max_seqlen_k; (void)total_k; (void)hkv;
  if (batch <= 0 || total_q <= 0 || hq <= 0 || d <= 0) return 0;
  return bwd_ws_bytes(total_q, hq, d, deterministic);
}

attn_status attn_bwd_varlen(const void *q, const void *k, const void *v, const void *out,
                            const float *lse, const void *dout, void *dq, void *dk, void *dv,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            int batch, int max_seqlen_q, int max_seqlen_k, int total_q,
                            int total_k, int dtype, int hq, int hkv, int d, float scale,
                            int causal, int win_l, int win_r, float softcap, int deterministic,
                            void *workspace, size_t workspace_bytes, attn_stream_t stream) {
  attn_status st = check_common(dtype, hq, hkv, d, scale, win_l, win_r, causal, softcap);
  if (st != ATTN_OK) return st;
  if (batch < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_k < 0)
    return ATTN_ERR_INVALID;
  if (batch == 0 || (total_q == 0 && total_k == 0)) return ATTN_OK;
  if (!cu_seqlens_q || !cu_seqlens_k) return ATTN_ERR_INVALID;
  if ((total_q > 0 && (!q || !out || !lse || !dout || !dq)) ||
      (total_k > 0 && (!k || !v || !dk || !dv)))
    return ATTN_ERR_INVALID;
  for (const void *p : {q, k, v, out, (const void *)lse, dout, (const void *)dq, (const void *)dk,
                        (const void *)dv, (const void *)workspace})
    if (!aligned16(p)) return ATTN_ERR_INVALID;
  if ((int64_t)total_q * hq > INT32_MAX || (int64_t)total_k * hkv > INT32_MAX)
    return ATTN_ERR_UNSUPPORTED;
  const size_t need = attn_bwd_varlen_workspace_size(batch, max_seqlen_q, max_seqlen_k, total_q,
                                                     total_k, hq, hkv, d, deterministic);
  if (need > 0 && (!workspace || workspace_bytes < need)) return ATTN_ERR_WORKSPACE;
  const DeviceInfo *di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  BwdArgs a{FwdArgs{q, k, v, const_cast<void *>(out), const_cast<float *>(lse),
                    Seqs{cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, total_q, total_k, hq},
                    batch, hq, hkv, d, dtype, scale, softcap > 0.f ? softcap : 0.f, win_l, win_r,
                    di->err},
            dout, dq, dk, dv};
  a.deterministic = deterministic;
  set_strides(a.f, 0, 0, 0);
  set_grad_strides(a, 0, 0, 0);
  return run_bwd(a, total_q, workspace, di, stream);
}

int attn_kvcache_num_splits(int b, int sq, int hq, int hkv, int d, int max_seqlen_k,
                            int num_splits) {
  (void)sq; (void)hq; (void)d;
  if (b <= 0 || hkv <= 0 || max_seqlen_k <= 0 || num_splits < 0) return 1;
  const DeviceInfo *di = device_info();
  return resolve_splits(b, hkv, max_seqlen_k, num_splits, di ? di->sms : 152);
}

size_t attn_kvcache_workspace_size(int b, int sq, int hq, int hkv, int d, int max_seqlen_k,
                                   int num_splits) {
  if (b <= 0 || sq <= 0 || hq <= 0 || d <= 0) return 0;
  const int s = attn_kvcache_num_splits(b, sq, hq, hkv, d, max_seqlen_k, num_splits);
  if (s <= 1) return 0;
  return align256(sizeof(float) * (size_t)s * b * sq * hq * d) +
         align256(sizeof(float) * (size_t)s * b * hq * sq);
}

attn_status attn_fwd_kvcache(const void *q, void *k_cache, void *v_cache, const void *k_new,
                             const void *v_new, const int32_t *cache_seqlens,
                             const int32_t *block_table, int num_pages, int page_size,
                             int max_pages_per_seq, void *out, float *lse, int dtype, int b,
                             int sq, int s_new, int hq, int hkv, int d, float scale, int causal,
                             int win_l, int win_r, float softcap, int num_splits,
                             void *workspace, size_t workspace_bytes, attn_stream_t stream) {
  attn_status st = check_common(dtype, hq, hkv, d, scale, win_l, win_r, causal, softcap);
  if (st != ATTN_OK) return st;
  if (b < 0 || sq < 0 || s_new < 0 || num_splits < 0 || num_pages < 0 || page_size <= 0 ||
      max_pages_per_seq <= 0)
    return ATTN_ERR_INVALID;
  if (b == 0 || sq == 0) return ATTN_OK;
  if (!q || !k_cache || !v_cache || !cache_seqlens || !out || !lse) return ATTN_ERR_INVALID;
  if (s_new > 0 && (!k_new || !v_new)) return ATTN_ERR_INVALID;
  if (block_table) {
    if (page_size % 128 != 0) return ATTN_ERR_INVALID;
  } else if (num_pages != b || max_pages_per_seq != 1) {
    return ATTN_ERR_INVALID;
  }
  for (const void *p : {q, (const void *)k_cache, (const void *)v_cache, k_new, v_new,
                        (const void *)out, (const void *)lse, (const void *)workspace})
    if (!aligned16(p)) return ATTN_ERR_INVALID;
  const int64_t cap = (int64_t)max_pages_per_seq * page_size;
  if (cap > INT32_MAX / 2 || (int64_t)num_pages * page_size * hkv > INT32_MAX)
    return ATTN_ERR_UNSUPPORTED;
  const DeviceInfo *di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  const int splits = resolve_splits(b, hkv, (int)cap, num_splits, di->sms);
  const size_t need = attn_kvcache_workspace_size(b, sq, hq, hkv, d, (int)cap, num_splits);
  if (need > 0 && (!workspace || workspace_bytes < need)) return ATTN_ERR_WORKSPACE;
  int chunk = (int)((cap + splits - 1) / splits);
  chunk = (chunk + 127) / 128 * 128;
  char *ws = static_cast<char *>(workspace);
  DecodeArgs a{q, k_cache, v_cache, k_new, v_new, cache_seqlens, block_table, num_pages,
               page_size, max_pages_per_seq, out, lse, dtype, b, sq, s_new, hq, hkv, d, scale,
               softcap > 0.f ? softcap : 0.f, win_l, win_r, splits, chunk,
               splits > 1 ? reinterpret_cast<float *>(ws) : nullptr,
               splits > 1 ? reinterpret_cast<float *>(
                                ws + align256(sizeof(float) * (size_t)splits * b * sq * hq * d))
                          : nullptr,
               di->err};
  a.wait_ns = wait_limit_ns();
  a.stall = test_stall();
  return launched(launch_decode(a, stream));
}

attn_status attn_fwd_probs(const void *q, const void *k, const float *lse, float *p, int dtype,
                           int b, int sq, int sk, int hq, int hkv, int d, float scale,
                           int causal, int win_l, int win_r, float softcap,
                           attn_stream_t stream) {
  attn_status st = check_common(dtype, hq, hkv, d, scale, win_l, win_r, causal, softcap);
  if (st != ATTN_OK) return st;
  if (b < 0 || sq < 0 || sk < 0) return ATTN_ERR_INVALID;
  if (b == 0 || sq == 0 || sk == 0) return ATTN_OK;
  if (!q || !k || !lse || !p) return ATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(lse) || !aligned16(p)) return ATTN_ERR_INVALID;
  if ((int64_t)b * hq > 65535 || sq > 65535) return ATTN_ERR_UNSUPPORTED;
  const DeviceInfo *di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  FwdArgs a{q, k, nullptr, nullptr, const_cast<float *>(lse),
            Seqs{nullptr, nullptr, sq, sk, 0, 0, hq}, b, hq, hkv, d, dtype, scale,
            softcap > 0.f ? softcap : 0.f, win_l, win_r, di->err};
  set_strides(a, 0, 0, 0);
  a.wait_ns = wait_limit_ns();
  a.stall = test_stall();
  return launched(launch_probs(a, p, stream));
}

size_t attn_fwd_fp8_workspace_size(int b, int sk, int hkv, int d) {
  if (b <= 0 || sk <= 0 || hkv <= 0 || d <= 0) return 0;
  return align256(sizeof(uint16_t) * (size_t)b * sk * hkv * d);  // v widened to bf16
}

attn_status attn_fwd_fp8(const void *q, const void *k, const void *v, void *out, float *lse,
                         float descale_q, float descale_k, float descale_v, int b, int sq, int sk,
                         int hq, int hkv, int d, float scale, int causal, int win_l, int win_r,
                         float softcap, void *workspace, size_t workspace_bytes,
                         attn_stream_t stream) {
  attn_status st = check_common(ATTN_BF16, hq, hkv, d, scale, win_l, win_r, causal, softcap);
  if (st != ATTN_OK) return st;
  for (float s : {descale_q, descale_k, descale_v})
    if (!isfinite(s) || !(s > 0.f)) return ATTN_ERR_INVALID;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if (b < 0 || sq < 0 || sk < 0) return ATTN_ERR_INVALID;
  if (b == 0 || sq == 0) return ATTN_OK;
  if (sk == 0) return ATTN_ERR_UNSUPPORTED;
  if (!q || !k || !v || !out || !lse) return ATTN_ERR_INVALID;
  for (const void *p : {q, k, v, (const void *)out, (const void *)lse, (const void *)workspace})
    if (!aligned16(p)) return ATTN_ERR_INVALID;
  if ((int64_t)b * sq * hq > INT32_MAX || (int64_t)b * sk * hkv > INT32_MAX)
    return ATTN_ERR_UNSUPPORTED;
  const float eff = scale * descale_q * descale_k;
  if (!isfinite(eff)) return ATTN_ERR_INVALID;
  const size_t need = attn_fwd_fp8_workspace_size(b, sk, hkv, d);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  const DeviceInfo *di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  cudaError_t e = launch_widen_e4m3(v, workspace, (int64_t)b * sk * hkv * d, di->sms, stream);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  FwdArgs a{q, k, workspace, out, lse, Seqs{nullptr, nullptr, sq, sk, 0, 0, hq}, b, hq, hkv, d,
            ATTN_BF16, eff, softcap > 0.f ? softcap : 0.f, win_l, win_r, di->err};
  set_strides(a, 0, 0, 0);
  a.wait_ns = wait_limit_ns();
  a.stall = test_stall();
  a.pack = resolve_pack(-1, hq, hkv, sq);
  a.qk_fp8 = 1;
  a.out_scale = descale_v;
  return launched(launch_fwd_tc(a, stream));
}

attn_status attn_kvcache_advance(int32_t *cache_seqlens, int b, int s_new, attn_stream_t stream) {
  if (b < 0 || s_new < 0) return ATTN_ERR_INVALID;
  if (b == 0) return ATTN_OK;
  if (!cache_seqlens || (reinterpret_cast<uintptr_t>(cache_seqlens) & 3)) return ATTN_ERR_INVALID;
  return launched(launch_kvcache_advance(cache_seqlens, b, s_new, stream));
}

unsigned long long attn_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

unsigned long long attn_set_wait_limit_ns(unsigned long long ns) {
  return g_wait_ns.exchange(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
}

int attn_set_test_stall(int on) { return g_test_stall.exchange(on != 0, std::memory_order_relaxed); }

attn_status attn_get_device_error(attn_stream_t stream, int *detail) {
  const DeviceInfo *di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyAsync(&word, di->err, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyAsync(di->err, &zero, sizeof(int), cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  if (detail) *detail = word;
  if (word & kErrTimeout) return ATTN_ERR_TIMEOUT;
  return word ? ATTN_ERR_DEVICE : ATTN_OK;
}

}  // extern "C"
