/*
 * Exact IO-aware softmax attention for NVIDIA GB300 (sm_103a): C ABI.
 *
 * What is computed (per batch b and head h, with s = `scale`):
 *   S = s Q K^T, masked;  P = softmax_rows(S);  O = P V;  LSE = logsumexp_rows(S)
 * and, for an upstream gradient dO of O,
 *   D = rowsum(dO * O), dV = P^T dO, dP = dO V^T, dS = P * (dP - D),
 *   dQ = s dS K, dK = s dS^T Q.
 *
 * How it is computed follows the FlashAttention practice record ("Why
 * recomputation is cheaper here than storing", Anthology of the SOTA): score
 * tiles live only in on-chip memory and are consumed at once with a running
 * row maximum and normaliser, the N x N matrix is never written to HBM, and the
 * backward pass rebuilds every S/P tile from Q, K, V and the saved per-row
 * statistics. Those statistics are the running maximum m and normaliser l of
 * "FlashAttention Algorithm > Recomputation Strategy" (section "What Gets
 * Stored vs Recomputed"), folded here into one value LSE = m + ln l.
 *
 * Conventions shared by every entry point (the _qk, _varlen and _split entry
 * points below state how their shapes differ):
 *  - Tensors Q, K, V, O, dO, dQ, dK, dV are contiguous [B, H, N, d] bf16 in
 *    device memory, d innermost; every base pointer 16-byte aligned.
 *    LSE is contiguous [B, H, N] fp32 (natural log). kv_len, when given, is
 *    a device int32 [B]: key j of batch b is valid iff j < kv_len[b].
 *  - d must be 64 or 128. N >= 0 (any value; N = 0 is a no-op). B, H >= 1.
 *    causal = 1 keeps key j for query i iff j <= i (with N_q query and N_k key
 *    rows, fa_forward_qk: iff j <= i + N_k - N_q).
 *  - All memory is owned by the caller. The library allocates nothing and
 *    frees nothing; outputs are fully overwritten.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream). A non-OK return means nothing was launched, except FA_ERR_CUDA
 *    after a failed launch.
 *  - Inside the kernels every wait is bounded; a wait that runs out records
 *    FA_ERR_TIMEOUT in a per-device status word that
 *    fa_get_last_device_status() reads (fa_get_last_device_status_detail()
 *    also says where). An argument that only the kernels can
 *    check (a packed sequence longer than max_seqlen) records
 *    FA_ERR_DEVICE_CHECK there; so does a failed bounds check in the
 *    bounds-checked build of this library (fa_debug.h).
 *  - Entry points are reentrant; calls that share output buffers race.
 */
#ifndef IO_AWARE_EXACT_FA_H
#define IO_AWARE_EXACT_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

typedef struct CUstream_st* fa_stream_t; /* identical to cudaStream_t */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad flag, too-small workspace */
  FA_ERR_UNSUPPORTED = 2,  /* d not in {64, 128}, B*H > 65535, or N beyond 32-bit indexing */
  FA_ERR_MISALIGNED = 3,   /* a tensor base pointer not 16-byte aligned */
  FA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
  FA_ERR_TIMEOUT = 5,      /* (device status) a bounded wait inside a kernel ran out */
  FA_ERR_DEVICE_CHECK = 6  /* (device status) an in-kernel consistency check failed */
} fa_status;

/* Forward pass: O and LSE from Q, K, V.
 * Defined by the practice record's account of the tiled kernel (scores kept on
 * chip and consumed immediately, blockwise running-maximum softmax) and by the
 * handbook's list of what is stored for the backward pass (O plus the per-row
 * running statistics). Returns an fa_status. */
FA_API int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
               float scale, int causal, fa_stream_t stream);

/* As fa_forward, with optional key padding: kv_len is NULL or a device int32
 * [B] of valid key counts (values are clamped to [0, N]). A query row with no
 * valid key gets O = 0 and LSE = -inf. */
FA_API int fa_forward_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                  float scale, int causal, const int32_t* kv_len, fa_stream_t stream);

/* As fa_forward_ex, with query and key lengths that may differ: q and o are
 * [B, H, Nq, d], k and v [B, H, Nk, d], lse [B, H, Nq]; kv_len values are
 * clamped to [0, Nk]. With causal = 1 the queries stand for the last Nq
 * positions of the keys' sequence: query row i keeps key j iff
 * j <= i + Nk - Nq (for Nq = Nk the pages' rule j <= i; the pages state only
 * that case). When Nq > Nk the first Nq - Nk rows keep no key and get O = 0,
 * LSE = -inf. Nq = 0 with Nk > 0 or the reverse returns FA_ERR_UNSUPPORTED;
 * both 0 is FA_OK with nothing to do. fa_forward_ex(.., N, ..) is exactly
 * fa_forward_qk(.., N, N, ..). */
FA_API int fa_forward_qk(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                         int Nk, int d, float scale, int causal, const int32_t* kv_len, fa_stream_t stream);

/* Forward pass over packed sequences of different lengths (variable-length
 * batches with no padding): B sequences, each its own attention problem with
 * N = len_b query and key rows (the pages' masks per sequence: causal j <= i).
 *  - Layout: q, k, v, o are [H, T, d] bf16 with every head's rows of all
 *    sequences packed back to back; lse is [H, T] fp32. Sequence b has rows
 *    [cu_seqlens[b], cu_seqlens[b + 1]) of every head.
 *  - cu_seqlens: device int32 [B + 1], non-decreasing, cu_seqlens[0] = 0,
 *    cu_seqlens[B] = T. max_seqlen: host upper bound of every length; it sizes
 *    the grid. A longer sequence is not fully computed and records
 *    FA_ERR_DEVICE_CHECK in the device status word.
 *  - A sequence of length 0 writes nothing. */
FA_API int fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int32_t* cu_seqlens, int B, int H, int T, int max_seqlen, int d, float scale,
                             int causal, fa_stream_t stream);

/* Backward of fa_forward_varlen: q, k, v, o, dO, dq, dk, dv are [H, T, d] bf16,
 * lse [H, T] fp32, sequences as in the forward call (same cu_seqlens,
 * max_seqlen, scale and causal). workspace: fa_backward_varlen_workspace_size
 * bytes, 256-byte aligned, contents on entry irrelevant. A sequence longer
 * than max_seqlen records FA_ERR_DEVICE_CHECK. */
FA_API int fa_backward_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_seqlens, int B, int H,
                              int T, int max_seqlen, int d, float scale, int causal, void* workspace,
                              size_t workspace_bytes, fa_stream_t stream);

/* Workspace bytes of fa_backward_varlen: per head, -D and a base-2 LSE for
 * T + 4 B + 256 rows (each sequence's rows start on a 16-byte boundary) and
 * an fp32 dQ accumulator of T rows rounded up to 128. 0 for invalid arguments. */
FA_API size_t fa_backward_varlen_workspace_size(int B, int H, int T, int d);

/* Forward pass for inference shapes: few query rows over many keys, where one
 * CTA per (head, query-tile pair) leaves most SMs idle (the pages: inference
 * workloads are mostly memory-bound). The key tiles of each work item are cut
 * into n_split near-equal shares run by separate CTAs. Each writes its share's O
 * (divided by its own normaliser, fp32) and LSE into `workspace`. A second
 * kernel joins the shares with the running-maximum rescaling that the tiled
 * softmax applies between key blocks. Shapes, masks and results as
 * fa_forward_qk. With Nq <= 8 (decode) a streaming kernel on the CUDA cores
 * runs instead (one query row would waste a 128-row tensor-core tile). It
 * takes the 128-key tiles of all heads as one sequence. With n_split = 1 each
 * CTA takes ceil(B * H / min(#SMs, 256)) whole heads and writes their O and LSE
 * directly (no second kernel, the workspace is not touched). With n_split > 1
 * each of G = min(#SMs, 256, n_split * B * H) CTAs takes an equal run of the
 * sequence; a head whose tiles all fall to one CTA is written directly, the
 * partial results of a head split between CTAs go to the workspace and a
 * second kernel joins them. That second kernel runs whenever kv_len is given
 * (the tile counts are on the device) or some CTA's run starts inside a head.
 *  - lse may be NULL: then no LSE is written.
 *  - workspace: at least fa_forward_split_workspace_size(B, H, Nq, d, n_split)
 *    bytes, 256-byte aligned; its contents on entry do not matter.
 *  - n_split >= 1 (more than 1024 returns FA_ERR_UNSUPPORTED). With
 *    n_split = 1, Nq > 8 and lse non-NULL this is fa_forward_qk and the
 *    workspace is not touched. */
FA_API int fa_forward_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                            int Nk, int d, float scale, int causal, const int32_t* kv_len, int n_split,
                            void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Workspace bytes of fa_forward_split: 2 * n_split * B * H * Nq rows of d + 1 fp32
 * (the decode kernel uses 2 G * Nq of them, G <= n_split * B * H).
 * Returns 0 for invalid arguments. */
FA_API size_t fa_forward_split_workspace_size(int B, int H, int Nq, int d, int n_split);

/* The library's choice of n_split for a shape on the current device. For
 * Nq <= 8 (the decode kernel): 1 (whole heads a CTA) when 2 * B * H >= SMs, else
 * ceil(SMs / (B * H)), at most 64, so that the decode kernel runs one CTA per SM.
 * Otherwise it is 1 when B * H * ceil(Nq / 256) work items
 * already reach the SM count, else the largest count whose CTAs fit in two
 * waves (floor(2 * SMs / items)), capped at ceil(Nk / 128) / 4 (four key tiles
 * a share) and at 64. */
FA_API int fa_forward_split_count(int B, int H, int Nq, int Nk, int d);

/* Bytes of device workspace fa_backward needs: per (b, h), D and a base-2
 * copy of LSE for every query row and an fp32 dQ accumulator, each padded to
 * a multiple of 128 rows. Linear in N. Returns 0 for unsupported d. */
FA_API size_t fa_backward_workspace_size(int B, int H, int N, int d);

/* Backward pass: dQ, dK, dV from Q, K, V, O, dO and the LSE saved by the
 * forward pass. No N x N input exists: every S and P tile is recomputed from
 * Q, K and LSE, as the practice record and the handbook ("What Gets Stored vs
 * Recomputed", and the closing paragraph of that section: tiles rebuilt with
 * the forward's tiling, gradients computed per block and accumulated) describe.
 * `workspace` is caller-owned device memory of at least
 * fa_backward_workspace_size(B, H, N, d) bytes, 256-byte aligned; its
 * contents on entry do not matter. `scale` and `causal` must equal the
 * forward call's. */
FA_API int fa_backward(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, void* workspace,
                size_t workspace_bytes, fa_stream_t stream);

/* As fa_backward, with the same optional key padding as fa_forward_ex. */
FA_API int fa_backward_ex(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                   const int32_t* kv_len, void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Backward of fa_forward_qk: q, o, dO, dq are [B, H, Nq, d], k, v, dk, dv
 * [B, H, Nk, d], lse [B, H, Nq]; the same masking as the forward call. The
 * workspace is fa_backward_workspace_size(B, H, Nq, d) bytes (it holds
 * per-query-row data only). fa_backward_ex(.., N, ..) is exactly
 * fa_backward_qk(.., N, N, ..). */
FA_API int fa_backward_qk(const void* q, const void* k, const void* v, const void* o, const void* dO,
                          const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                          float scale, int causal, const int32_t* kv_len, void* workspace, size_t workspace_bytes,
                          fa_stream_t stream);

/* One stage of fa_backward_ex, same arguments; running stages 0, 1, 2 in
 * order on one stream is exactly fa_backward_ex. Exposed so that each kernel
 * can be timed on its own.
 *   0: -D = -rowsum(dO * O) and -LSE in base 2 per query row, into the workspace;
 *      zeroes the fp32 dQ accumulator.
 *   1: the recomputing kernel: dK and dV written, dQ accumulated in fp32.
 *   2: the fp32 dQ accumulator rounded to bf16 into dq.
 * Any other stage value returns FA_ERR_INVALID_ARG. */
FA_API int fa_backward_stage(int stage, const void* q, const void* k, const void* v, const void* o, const void* dO,
                             const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                             float scale, int causal, const int32_t* kv_len, void* workspace,
                             size_t workspace_bytes, fa_stream_t stream);

/* One stage of fa_backward_qk (stages as for fa_backward_stage). */
FA_API int fa_backward_stage_qk(int stage, const void* q, const void* k, const void* v, const void* o,
                                const void* dO, const float* lse, void* dq, void* dk, void* dv, int B, int H,
                                int Nq, int Nk, int d, float scale, int causal, const int32_t* kv_len,
                                void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Backward pass for callers that cannot allocate device memory: no workspace
 * argument. The pages have no counterpart of this entry point; it exists for
 * callers that are handed only their input and output buffers and may not
 * call cudaMalloc (for example a runtime that reserves all device memory up
 * front and gives a plugin nothing else). Instead of a caller's workspace it
 * uses one fixed scratch array compiled into the library, of
 * fa_backward_noalloc_max_bytes() bytes (32 MiB) on every GPU that loads the
 * library, held until the process exits.
 *  - Same arguments and results as fa_backward_ex without the workspace; the
 *    same argument checks come first, in the same order.
 *  - A valid shape whose workspace (fa_backward_workspace_size) exceeds the
 *    array returns FA_ERR_UNSUPPORTED before anything runs;
 *    fa_last_error_detail() then says how many bytes it needed.
 *  - Allocates nothing. The first call on each device (and context) looks up
 *    the array's device address (cudaGetSymbolAddress) with that device
 *    current; make that first call before any stream capture. A device
 *    ordinal of 64 or more returns FA_ERR_UNSUPPORTED.
 *  - All calls on a device share the one array: calls whose kernels overlap on
 *    the GPU (other streams, other host threads) race and corrupt each other's
 *    gradients. Serialise them. Each call re-initialises what it needs. */
FA_API int fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                               const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                               float scale, int causal, const int32_t* kv_len, fa_stream_t stream);

/* Size in bytes of the scratch array fa_backward_noalloc uses. */
FA_API size_t fa_backward_noalloc_max_bytes(void);

/* Static text for an fa_status value. */
FA_API const char* fa_status_string(int status);

/* Synchronises `stream`, then returns and clears the current device's status
 * word: FA_OK if no kernel recorded an error, else the first error a kernel
 * recorded (FA_ERR_TIMEOUT or FA_ERR_DEVICE_CHECK). A failure of the CUDA
 * calls this makes returns FA_ERR_CUDA (fa_last_error_detail names it); a
 * device ordinal of 64 or more returns FA_ERR_UNSUPPORTED. The word's device
 * address is looked up once per device and context; after cudaDeviceReset the
 * next call looks it up again. */
FA_API int fa_get_last_device_status(fa_stream_t stream);

/* As fa_get_last_device_status; if detail is non-NULL it also receives 4 ints
 * describing the first recorded error: code, site (which wait or check),
 * blockIdx.x, blockIdx.y (all 0 when none was recorded). */
FA_API int fa_get_last_device_status_detail(fa_stream_t stream, int* detail);

/* For the calling host thread: text naming the CUDA call that made the last
 * FA_ERR_CUDA return and its error (or the reason for a size rejection by
 * fa_backward_noalloc), or "" if none has. Static storage. */
FA_API const char* fa_last_error_detail(void);

/* Library version as major*10000 + minor*100 + patch. */
FA_API int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IO_AWARE_EXACT_FA_H */
