/*
 * Hardware self-checks for the sm_103a building blocks of the attention
 * kernels (libfa_selftest.so). These are not part of the attention method;
 * they isolate one fact each so that a failing attention parity test can be
 * traced to a tcgen05 operand layout or to the bounded-wait machinery.
 */
#ifndef IO_AWARE_EXACT_FA_SELFTEST_H
#define IO_AWARE_EXACT_FA_SELFTEST_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

#define FA_SELFTEST_A_MN 1   /* A stored [K][128] (M contiguous) instead of [128][K] */
#define FA_SELFTEST_B_MN 2   /* B stored [K][N] (N contiguous) instead of [N][K] */
#define FA_SELFTEST_A_TMEM 4 /* A copied to tensor memory, read by the MMA from there ([128][K] storage) */

/* d[128][N] (fp32, device) = A (128 x K) * B (K x N), one CTA, bf16 operands
 * in device memory (16-byte aligned), N and K in {64, 128}. The layouts are
 * selected by `mode` as above. `status` is a device int[4], zeroed by the
 * caller; a wait that runs out writes FA_ERR_TIMEOUT there. */
FA_API int fa_selftest_mma(const void* a, const void* b, float* d, int N, int K, int mode, int* status,
                    fa_stream_t stream);

/* Launches one thread that waits on a shared-memory barrier nothing arrives
 * on, with a limit of limit_us microseconds (1 .. 5e6). Afterwards status[0]
 * (device int[4], zeroed by the caller) must read FA_ERR_TIMEOUT. */
FA_API int fa_selftest_wait_timeout(int* status, unsigned int limit_us, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif
