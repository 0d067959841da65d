// Backward pass for callers that cannot allocate device memory.
//
// fa_backward_ex needs a caller-provided workspace (D, LSE in base 2 and the
// fp32 dQ accumulator). Some callers have no way to provide one: a host
// runtime that reserves all device memory up front and hands plugins only
// their input and output buffers, or code running where a cudaMalloc is not
// permitted. For them, fa_backward_noalloc uses a fixed scratch array that
// lives in this library's device image instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds kScratchBytes of it until the process exits. In host code the
// name g_scratch is only a host-side stand-in, not a device address; the
// device address is obtained once per device (and context) with
// cudaGetSymbolAddress and passed to the kernels as their workspace pointer.
#include <cuda_runtime.h>

#include <cstdio>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB
__device__ __align__(256) unsigned char g_scratch[kScratchBytes];
fa::SymbolCache g_scratch_cache;

}  // namespace

extern "C" {

size_t fa_backward_noalloc_max_bytes(void) { return kScratchBytes; }

int fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                        const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                        int causal, const int32_t* kv_len, fa_stream_t stream) {
  // the checks of fa_backward_ex, in its order, before the size of this entry point's array
  const int rc0 = fa::check_common(B, H, N, N, d, scale, causal);
  if (rc0 != FA_OK) return rc0;
  if ((long long)B * H * N == 0)  // nothing to compute; same result as fa_backward_ex
    return fa_backward_ex(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, kv_len, nullptr, 0, stream);
  const size_t need = fa_backward_workspace_size(B, H, N, d);
  if (need > kScratchBytes) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "fa_backward_noalloc: this shape needs %zu bytes of scratch, the fixed array has %zu",
                  need, kScratchBytes);
    fa::set_error_detail(msg);
    return FA_ERR_UNSUPPORTED;
  }
  int rc = FA_OK;
  void* scratch = fa::symbol_on_current_device(g_scratch, g_scratch_cache, "scratch", &rc);
  if (!scratch) return rc;
  // The first stage overwrites D and LSE and zeroes the dQ accumulator, so
  // whatever an earlier call left in the array does not matter.
  return fa_backward_ex(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, kv_len, scratch, kScratchBytes,
                        stream);
}

}  // extern "C"
