// Launch descriptions shared between the entry points and the kernels.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace fa {

struct FwdArgs {
  int H, N;            // heads per batch, query rows N_q (rows of Q, O, LSE)
  int Nk;              // key rows N_k (rows of K, V)
  int coff;            // N_k - N_q: causal query row i keeps keys j <= i + coff
  int n_pairs;         // ceil(N_q / 256): work items per head (two 128-row query tiles each)
  int causal;
  float scale_log2;    // scale * log2(e)
  const int* kv_len;   // [B] device, or null
  float* lse;          // [B*H, N]; null only with a split (the combine then writes none)
  uint16_t* o;         // [B*H, N, d] bf16 (also written through the tensor map)
  const int* cu_seqlens;  // packed sequences: device [B + 1] row offsets, else null
  int T, max_seqlen;   // packed sequences: rows per head, and an upper bound of every length
  int n_split;         // split-KV forward: key-tile shares per work item (1 = no split)
  float* part_o;       // split-KV: [2 n_split, B*H, N, d] fp32 partial O (two slots per share),
                       // each normalised by its own l
  float* part_lse;     // split-KV: [2 n_split, B*H, N] fp32 LSE of each slot (-inf: no key)
  int* status;         // device status word (4 ints)
#ifdef FA_DEBUG
  int dbg_B;           // batch count B, for the extents the debug build checks against
  int dbg_slack;       // rows taken off those extents (fa_debug_set_check_slack)
#endif
};

// Packed sequences ([H, T, d], cu_seqlens) reuse four fields that mean nothing there (no key
// padding, no causal offset): kv_len holds cu_seqlens, N the longest sequence, Nk the rows per
// head T and coff the -LSE2 / -D rows per head. The accessors below name them. (The backward
// kernels measured 2 % slower with four more fields in this struct.)
struct BwdArgs {
  int H, N, Npad;      // query rows N_q (rows of Q, O, dO, LSE, dQ); Npad = N_q rounded up to 128
  int Nk;              // key rows N_k (rows of K, V, dK, dV)
  int coff;            // N_k - N_q: causal query row i keeps keys j <= i + coff
  int BH;              // B * H (set by the launcher of the persistent d = 64 kernel)
  int causal;
  float scale;         // softmax scale s
  float scale_log2;    // s * log2(e)
  const int* kv_len;   // [B] device, or null
  const uint16_t* o;   // [B*H, N, d]
  const uint16_t* dO;  // [B*H, N, d]
  const float* lse;    // [B*H, N]
  float* lse2;         // workspace [B*H, Npad]: -LSE * log2(e), -inf on padding rows
  float* dvec;         // workspace [B*H, Npad]: -D = -rowsum(dO * O), 0 on padding rows
  float* dq_acc;       // workspace [B*H, Npad, d] fp32
  uint16_t* dq;        // [B*H, N, d] bf16
  uint16_t* dk;        // [B*H, N, d] bf16
  uint16_t* dv;        // [B*H, N, d] bf16
  int* status;
#ifdef FA_DEBUG
  int dbg_B;           // batch count B, for the extents the debug build checks against
  int dbg_slack;       // rows taken off those extents (fa_debug_set_check_slack)
#endif
};
__host__ __device__ inline const int* vl_cu(const BwdArgs& a) { return a.kv_len; }
__host__ __device__ inline int vl_maxlen(const BwdArgs& a) { return a.N; }
__host__ __device__ inline int vl_T(const BwdArgs& a) { return a.Nk; }
__host__ __device__ inline int vl_Lpad(const BwdArgs& a) { return a.coff; }


// Debug build: the batch count and the current check slack into the kernels' arguments (no-op in
// every other build).
#ifdef FA_DEBUG
int debug_check_slack();
#define FA_DEBUG_ARGS(args, B)            \
  do {                                    \
    (args).dbg_B = (B);                   \
    (args).dbg_slack = ::fa::debug_check_slack(); \
  } while (0)
#else
#define FA_DEBUG_ARGS(args, B) \
  do {                         \
  } while (0)
#endif

// Argument checks shared by every entry point: sizes non-negative, causal 0 or 1, scale finite
// and positive (FA_ERR_INVALID_ARG); d in {64, 128}, B * H <= 65535, lengths within 32-bit
// indexing and the grid's y axis, and no queries without keys or the reverse
// (FA_ERR_UNSUPPORTED). FA_OK otherwise.
int check_common(int B, int H, int Nq, int Nk, int d, float scale, int causal);

// Device address of a file-scope __device__ variable (`symbol`, its host-side stand-in) on the
// current device, looked up with cudaGetSymbolAddress on the first call for each (device,
// context) pair and cached in `cache`. Returns null with *rc set (FA_ERR_UNSUPPORTED for a
// device ordinal of 64 or more, FA_ERR_CUDA for a failed CUDA call, detail recorded).
struct SymbolCache {
  static constexpr int kMaxDevices = 64;
  void* ctx[kMaxDevices] = {};
  void* ptr[kMaxDevices] = {};
};
void* symbol_on_current_device(const void* symbol, SymbolCache& cache, const char* what, int* rc);

// Records, for this host thread, which CUDA call failed and why (read back by
// fa_last_error_detail). Returns FA_ERR_CUDA for convenience.
int cuda_fail(const char* where, int code, const char* what);
// Records a free-form reason for this host thread (read back by fa_last_error_detail).
void set_error_detail(const char* text);
// Number of SMs of the current device (cached per device); false, with the CUDA error
// recorded, when it cannot be read.
bool sm_count(int* out);
// After a launch: FA_OK, or FA_ERR_CUDA with the launch error recorded.
int check_launch(const char* kernel);

// Launches `kernel` with programmatic stream serialization (programmatic dependent launch): its
// CTAs may start while the previous grid in the stream finishes, and wait for it in
// griddep_wait() before touching global memory. Returns FA_OK or FA_ERR_CUDA.
template <typename... Params, typename... Args>
int launch_pdl(const char* name, void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
  if (e != cudaSuccess) return cuda_fail(name, (int)e, cudaGetErrorName(e));
  return check_launch(name);
}

int launch_fwd(const void* q, const void* k, const void* v, void* o, const FwdArgs& args, int BH, int d,
               cudaStream_t stream);
// Packed sequences ([H, T, d], args.cu_seqlens): fwd_kernel over (sequence x head, query pair).
int launch_fwd_varlen(const void* q, const void* k, const void* v, void* o, const FwdArgs& args, int BH, int d,
                      cudaStream_t stream);
// Split-KV forward: fwd_kernel over (head, query pair, share) writing per-share partial
// results to args.part_o / args.part_lse, then fwd_combine_kernel joining them into o (and lse).
int launch_fwd_split(const void* q, const void* k, const void* v, void* o, const FwdArgs& args, int BH, int d,
                     cudaStream_t stream);
// stage 0: D, base-2 LSE, zeroed dQ accumulator; 1: main kernel (dK, dV, dQ accumulator);
// 2: dQ accumulator -> bf16 dQ
// Packed sequences ([H, T, d], args.cu_seqlens): the same three stages.
int launch_bwd_varlen_stage(int stage, const void* q, const void* k, const void* v, const BwdArgs& args, int B, int H,
                            int d, cudaStream_t stream);
int launch_bwd_stage(int stage, const void* q, const void* k, const void* v, const BwdArgs& args, int BH, int d,
                     cudaStream_t stream);

}  // namespace fa
