// C-ABI entry points: argument validation, workspace carving, tensor-map
// construction (in the launchers) and the per-device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#ifdef FA_DEBUG
#include "fa_debug.h"
#endif

namespace {

// Per-device word the kernels write when a bounded wait runs out or an
// in-kernel check fails: code, wait site, blockIdx.x, blockIdx.y.
__device__ int g_status[4];
fa::SymbolCache g_status_cache;

int* device_status(int* err) {
  return static_cast<int*>(fa::symbol_on_current_device(g_status, g_status_cache, "status word", err));
}

// The current CUDA context (driver handle), through the driver entry point the runtime hands
// out, so that the library needs no link-time dependency on libcuda.
bool current_context(void** out) {
  using Fn = CUresult (*)(CUcontext*);
  static Fn fn = []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (Fn) nullptr;
    return reinterpret_cast<Fn>(p);
  }();
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return false;
  *out = c;
  return true;
}

std::mutex g_symbol_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

struct WsLayout {
  size_t lse2, dvec, dqacc, total;
};

WsLayout ws_layout(int B, int H, int N, int d) {
  const long long BH = (long long)B * H;
  const long long Npad = round_up(N, 128);
  WsLayout w;
  w.lse2 = 0;
  w.dvec = (size_t)round_up(w.lse2 + BH * Npad * 4, 256);
  w.dqacc = (size_t)round_up(w.dvec + BH * Npad * 4, 256);
  w.total = (size_t)round_up(w.dqacc + BH * Npad * d * 4, 256);
  return w;
}

thread_local char g_last_error[256] = "";

}  // namespace

namespace fa {
int check_common(int B, int H, int Nq, int Nk, int d, float scale, int causal) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  if (BH > 65535) return FA_ERR_UNSUPPORTED;  // documented limit on B*H
  for (const int n : {Nq, Nk}) {
    if ((long long)n + 255 > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    if ((n + 127) / 128 > 65535) return FA_ERR_UNSUPPORTED;  // key tiles / query pairs on the grid's y axis
  }
  if (BH > 0 && (Nq == 0) != (Nk == 0)) return FA_ERR_UNSUPPORTED;  // queries without keys or keys without queries
  return FA_OK;
}

void* symbol_on_current_device(const void* symbol, SymbolCache& cache, const char* what, int* rc) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *rc = cuda_fail("cudaGetDevice", (int)e, cudaGetErrorName(e));
    return nullptr;
  }
  if (dev < 0 || dev >= SymbolCache::kMaxDevices) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "device ordinal %d: this library serves devices 0 .. %d", dev,
                  SymbolCache::kMaxDevices - 1);
    set_error_detail(msg);
    *rc = FA_ERR_UNSUPPORTED;
    return nullptr;
  }
  // the address belongs to the module loaded in the current context: a new context on the same
  // device (after cudaDeviceReset, say) gets its own lookup
  void* ctx = nullptr;
  if (!current_context(&ctx)) {
    *rc = cuda_fail("cuCtxGetCurrent", 0, "no current context");
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_symbol_mu);
  if (cache.ptr[dev] == nullptr || cache.ctx[dev] != ctx) {
    void* p = nullptr;
    const cudaError_t e2 = cudaGetSymbolAddress(&p, symbol);
    if (e2 != cudaSuccess || p == nullptr) {
      char where[96];
      std::snprintf(where, sizeof(where), "cudaGetSymbolAddress(%s)", what);
      *rc = cuda_fail(where, (int)e2, cudaGetErrorName(e2));
      return nullptr;
    }
    cache.ptr[dev] = p;
    cache.ctx[dev] = ctx;
  }
  return cache.ptr[dev];
}

int cuda_fail(const char* where, int code, const char* what) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s failed: %s (code %d)", where, what ? what : "", code);
  return FA_ERR_CUDA;
}
void set_error_detail(const char* text) { std::snprintf(g_last_error, sizeof(g_last_error), "%s", text); }
bool sm_count(int* out) {
  static int cache[64] = {0};  // benign race: every writer stores the same value
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", (int)e, cudaGetErrorName(e)) == FA_OK;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    *out = cache[dev];
    return true;
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess || n <= 0) {
    cuda_fail("cudaDeviceGetAttribute(MultiProcessorCount)", (int)e, cudaGetErrorName(e));
    return false;
  }
  if (dev >= 0 && dev < 64) cache[dev] = n;
  *out = n;
  return true;
}

int check_launch(const char* kernel) {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return FA_OK;
  return cuda_fail(kernel, (int)e, cudaGetErrorName(e));
}
#ifdef FA_DEBUG
namespace {
std::atomic<int> g_check_slack{0};
}
int debug_check_slack() { return g_check_slack.load(std::memory_order_relaxed); }
#endif
}  // namespace fa

extern "C" {

const char* fa_last_error_detail(void) { return g_last_error; }

#ifdef FA_DEBUG
int fa_debug_set_check_slack(int rows) {
  if (rows < 0) return FA_ERR_INVALID_ARG;
  fa::g_check_slack.store(rows, std::memory_order_relaxed);
  return FA_OK;
}
#endif

int fa_version(void) { return 100; }

const char* fa_status_string(int s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported shape (d must be 64 or 128, B*H <= 65535)";
    case FA_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "CUDA call failed";
    case FA_ERR_TIMEOUT: return "bounded wait inside a kernel ran out";
    case FA_ERR_DEVICE_CHECK: return "in-kernel consistency check failed";
    default: return "unknown status";
  }
}

int fa_forward_qk(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                  int d, float scale, int causal, const int32_t* kv_len, fa_stream_t stream) {
  int rc = fa::check_common(B, H, Nq, Nk, d, scale, causal);
  if (rc != FA_OK) return rc;
  if ((long long)B * H * Nq == 0) return FA_OK;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  int err = FA_OK;
  int* status = device_status(&err);
  if (!status) return err;
  fa::FwdArgs a;
  a.H = H;
  a.N = Nq;
  a.Nk = Nk;
  a.coff = Nk - Nq;
  a.n_pairs = (Nq + 255) / 256;
  a.causal = causal;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.kv_len = kv_len;
  a.lse = lse;
  a.o = static_cast<uint16_t*>(o);
  a.cu_seqlens = nullptr;
  a.T = 0;
  a.max_seqlen = 0;
  a.n_split = 1;
  a.part_o = nullptr;
  a.part_lse = nullptr;
  a.status = status;
  FA_DEBUG_ARGS(a, B);
  return fa::launch_fwd(q, k, v, o, a, B * H, d, reinterpret_cast<cudaStream_t>(stream));
}

int fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens,
                      int B, int H, int T, int max_seqlen, int d, float scale, int causal, fa_stream_t stream) {
  if (B < 0 || T < 0 || max_seqlen < 0) return FA_ERR_INVALID_ARG;
  int rc = fa::check_common(B, H, max_seqlen, max_seqlen, d, scale, causal);
  if (rc != FA_OK) return rc;
  if ((long long)B * H == 0 || T == 0 || max_seqlen == 0) return FA_OK;
  if (!q || !k || !v || !o || !lse || !cu_seqlens) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  if ((long long)H * T > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  int err = FA_OK;
  int* status = device_status(&err);
  if (!status) return err;
  fa::FwdArgs a;
  a.H = H;
  a.N = max_seqlen;
  a.Nk = max_seqlen;
  a.coff = 0;
  a.n_pairs = (max_seqlen + 255) / 256;
  a.causal = causal;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.kv_len = nullptr;
  a.lse = lse;
  a.o = static_cast<uint16_t*>(o);
  a.cu_seqlens = cu_seqlens;
  a.T = T;
  a.max_seqlen = max_seqlen;
  a.n_split = 1;
  a.part_o = nullptr;
  a.part_lse = nullptr;
  a.status = status;
  FA_DEBUG_ARGS(a, B);
  return fa::launch_fwd_varlen(q, k, v, o, a, B * H, d, reinterpret_cast<cudaStream_t>(stream));
}

size_t fa_forward_split_workspace_size(int B, int H, int Nq, int d, int n_split) {
  if (B < 0 || H < 0 || Nq < 0 || (d != 64 && d != 128) || n_split < 1) return 0;
  const long long rows = 2LL * n_split * B * H * Nq;  // two partial slots per share
  return (size_t)(round_up(rows * d * 4, 256) + round_up(rows * 4, 256));
}

int fa_forward_split_count(int B, int H, int Nq, int Nk, int d) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128)) return 1;
  int sms = 0;
  if (!fa::sm_count(&sms)) return 1;
  if (Nq <= 8) {
    // the streaming decode kernel: with heads for at least half the SMs, whole heads a CTA
    // (n_split = 1, no join: the stream is memory-bound there already); fewer heads are cut
    // between min(#SMs, n_split B H) CTAs, enough shares for one CTA per SM
    const long long bh = (long long)B * H;
    if (2 * bh >= sms) return 1;
    return (int)std::max<long long>(1, std::min<long long>((sms + bh - 1) / bh, 64));
  }
  const long long items = (long long)B * H * ((Nq + 255) / 256);
  if (items >= sms) return 1;
  // the most shares whose CTAs still fit in two waves (a partly filled last wave costs as
  // much as a full one), each share at least four 128-key tiles, at most 64 shares
  long long n = (2LL * sms) / items;
  n = std::min<long long>(n, std::max(1, ((Nk + 127) / 128) / 4));
  return (int)std::max<long long>(1, std::min<long long>(n, 64));
}

int fa_forward_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                     int d, float scale, int causal, const int32_t* kv_len, int n_split, void* workspace,
                     size_t workspace_bytes, fa_stream_t stream) {
  int rc = fa::check_common(B, H, Nq, Nk, d, scale, causal);
  if (rc != FA_OK) return rc;
  if (n_split < 1) return FA_ERR_INVALID_ARG;
  if (n_split > 1024) return FA_ERR_UNSUPPORTED;
  // one share with an LSE to write: the plain forward (no workspace used); decode rows (Nq <= 8)
  // keep the streaming decode kernel, which then writes o and lse itself
  if (n_split == 1 && lse && Nq > 8)
    return fa_forward_qk(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, kv_len, stream);
  if ((long long)B * H * Nq == 0) return FA_OK;
  if (!q || !k || !v || !o || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
    return FA_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_MISALIGNED;
  if (workspace_bytes < fa_forward_split_workspace_size(B, H, Nq, d, n_split)) return FA_ERR_INVALID_ARG;
  int err = FA_OK;
  int* status = device_status(&err);
  if (!status) return err;
  const long long rows = 2LL * n_split * B * H * Nq;
  fa::FwdArgs a;
  a.H = H;
  a.N = Nq;
  a.Nk = Nk;
  a.coff = Nk - Nq;
  a.n_pairs = (Nq + 255) / 256;
  a.causal = causal;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.kv_len = kv_len;
  a.lse = lse;
  a.o = static_cast<uint16_t*>(o);
  a.cu_seqlens = nullptr;
  a.T = 0;
  a.max_seqlen = 0;
  a.n_split = n_split;
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + round_up(rows * d * 4, 256));
  a.status = status;
  FA_DEBUG_ARGS(a, B);
  return fa::launch_fwd_split(q, k, v, o, a, B * H, d, reinterpret_cast<cudaStream_t>(stream));
}

int fa_forward_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                  float scale, int causal, const int32_t* kv_len, fa_stream_t stream) {
  return fa_forward_qk(q, k, v, o, lse, B, H, N, N, d, scale, causal, kv_len, stream);
}

int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
               float scale, int causal, fa_stream_t stream) {
  return fa_forward_ex(q, k, v, o, lse, B, H, N, d, scale, causal, nullptr, stream);
}

size_t fa_backward_workspace_size(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N < 0 || (d != 64 && d != 128)) return 0;
  return ws_layout(B, H, N, d).total;
}

int fa_backward_stage_qk(int stage, const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                         float scale, int causal, const int32_t* kv_len, void* workspace, size_t workspace_bytes,
                         fa_stream_t stream) {
  if (stage < 0 || stage > 2) return FA_ERR_INVALID_ARG;
  int rc = fa::check_common(B, H, Nq, Nk, d, scale, causal);
  if (rc != FA_OK) return rc;
  if ((long long)B * H * Nq == 0) return FA_OK;
  const int N = Nq;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_MISALIGNED;
  const WsLayout w = ws_layout(B, H, N, d);
  if (workspace_bytes < w.total) return FA_ERR_INVALID_ARG;
  int err = FA_OK;
  int* status = device_status(&err);
  if (!status) return err;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  fa::BwdArgs a;
  a.H = H;
  a.N = N;
  a.Npad = (int)round_up(N, 128);
  a.Nk = Nk;
  a.coff = Nk - Nq;
  a.causal = causal;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.kv_len = kv_len;
  a.o = static_cast<const uint16_t*>(o);
  a.dO = static_cast<const uint16_t*>(dO);
  a.lse = lse;
  a.lse2 = reinterpret_cast<float*>(ws + w.lse2);
  a.dvec = reinterpret_cast<float*>(ws + w.dvec);
  a.dq_acc = reinterpret_cast<float*>(ws + w.dqacc);
  a.dq = static_cast<uint16_t*>(dq);
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  a.status = status;
  FA_DEBUG_ARGS(a, B);
  return fa::launch_bwd_stage(stage, q, k, v, a, B * H, d, reinterpret_cast<cudaStream_t>(stream));
}

int fa_backward_stage(int stage, const void* q, const void* k, const void* v, const void* o, const void* dO,
                      const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                      int causal, const int32_t* kv_len, void* workspace, size_t workspace_bytes,
                      fa_stream_t stream) {
  return fa_backward_stage_qk(stage, q, k, v, o, dO, lse, dq, dk, dv, B, H, N, N, d, scale, causal, kv_len,
                              workspace, workspace_bytes, stream);
}

int fa_backward_qk(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                   const int32_t* kv_len, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  for (int stage = 0; stage < 3; ++stage) {
    const int rc = fa_backward_stage_qk(stage, q, k, v, o, dO, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, causal,
                                        kv_len, workspace, workspace_bytes, stream);
    if (rc != FA_OK) return rc;
  }
  return FA_OK;
}

int fa_backward_ex(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                   const int32_t* kv_len, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return fa_backward_qk(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, N, d, scale, causal, kv_len, workspace,
                        workspace_bytes, stream);
}

int fa_backward(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, void* workspace,
                size_t workspace_bytes, fa_stream_t stream) {
  return fa_backward_ex(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, nullptr, workspace,
                        workspace_bytes, stream);
}

size_t fa_backward_varlen_workspace_size(int B, int H, int T, int d) {
  if (B < 0 || H < 0 || T < 0 || (d != 64 && d != 128)) return 0;
  const long long Lpad = round_up((long long)T + 4LL * B, 128) + 128, Tpad = round_up(T, 128);
  const long long l2 = round_up((long long)H * Lpad * 4, 256);
  return (size_t)(2 * l2 + round_up((long long)H * Tpad * d * 4, 256));
}

int fa_backward_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                       void* dq, void* dk, void* dv, const int32_t* cu_seqlens, int B, int H, int T, int max_seqlen,
                       int d, float scale, int causal, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (B < 0 || T < 0 || max_seqlen < 0) return FA_ERR_INVALID_ARG;
  int rc = fa::check_common(B, H, max_seqlen, max_seqlen, d, scale, causal);
  if (rc != FA_OK) return rc;
  if ((long long)B * H == 0 || T == 0 || max_seqlen == 0) return FA_OK;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || !cu_seqlens || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_MISALIGNED;
  if ((long long)H * (T + 4LL * B + 256) > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (workspace_bytes < fa_backward_varlen_workspace_size(B, H, T, d)) return FA_ERR_INVALID_ARG;
  int err = FA_OK;
  int* status = device_status(&err);
  if (!status) return err;
  const long long Lpad = round_up((long long)T + 4LL * B, 128) + 128;
  const long long l2 = round_up((long long)H * Lpad * 4, 256);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  fa::BwdArgs a;  // packed sequences: kv_len, N, Nk and coff carry cu_seqlens, max_seqlen, T, Lpad
  a.H = H;
  a.N = max_seqlen;
  a.Npad = (int)round_up(T, 128);  // dQ accumulator rows per head
  a.Nk = T;
  a.coff = (int)Lpad;
  a.kv_len = cu_seqlens;
  a.BH = B * H;
  a.causal = causal;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.o = static_cast<const uint16_t*>(o);
  a.dO = static_cast<const uint16_t*>(dO);
  a.lse = lse;
  a.lse2 = reinterpret_cast<float*>(ws);
  a.dvec = reinterpret_cast<float*>(ws + l2);
  a.dq_acc = reinterpret_cast<float*>(ws + 2 * l2);
  a.dq = static_cast<uint16_t*>(dq);
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  a.status = status;
  FA_DEBUG_ARGS(a, B);
  for (int stage = 0; stage < 3; ++stage) {
    rc = fa::launch_bwd_varlen_stage(stage, q, k, v, a, B, H, d, reinterpret_cast<cudaStream_t>(stream));
    if (rc != FA_OK) return rc;
  }
  return FA_OK;
}

int fa_get_last_device_status_detail(fa_stream_t stream, int* detail) {
  int err = FA_OK;
  int* status = device_status(&err);
  if (!status) return err;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fa::cuda_fail("cudaStreamSynchronize", (int)e, cudaGetErrorName(e));
  int h[4] = {0, 0, 0, 0};
  e = cudaMemcpy(h, status, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fa::cuda_fail("cudaMemcpy(status word)", (int)e, cudaGetErrorName(e));
  if (h[0] != 0) {
    const int zero[4] = {0, 0, 0, 0};
    e = cudaMemcpy(status, zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fa::cuda_fail("cudaMemcpy(status word)", (int)e, cudaGetErrorName(e));
  }
  if (detail)
    for (int i = 0; i < 4; ++i) detail[i] = h[i];
  return h[0];
}

int fa_get_last_device_status(fa_stream_t stream) { return fa_get_last_device_status_detail(stream, nullptr); }

}  // extern "C"
