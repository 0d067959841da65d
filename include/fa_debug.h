/*
 * Debug build of the attention library (libfa_debug.so): the C ABI of fa.h
 * unchanged, plus the one entry point below. It stands in for a memory checker.
 *
 * Built from the same sources with FA_DEBUG defined, every kernel checks the
 * following before use:
 *  - the index of each direct global load and store;
 *  - the index of each metadata read (kv_len, cu_seqlens, partial slots);
 *  - the coordinates of each TMA or bulk copy: x inside the row on a 16-byte
 *    boundary, the head inside the tensor, and a box that overlaps the
 *    tensor's rows. A store or a reduce-add must also start at a row >= 0;
 *  - the shared-memory range of each copy and each MMA operand tile;
 *  - the TMEM lane quarter and columns of each warp's accumulators.
 * A failed check does not fault. It records FA_ERR_DEVICE_CHECK in the status
 * word, with one of the sites below in detail[1] of
 * fa_get_last_device_status_detail(), and skips the access. The CTA then gives
 * up its remaining waits and leaves, as after a timeout. Outputs that the
 * failed CTA did not write are then undefined.
 *
 * The checks cost time. libfa.so compiles none of them and is the library to
 * use; this build is for tests and for chasing a suspected out-of-bounds
 * access.
 */
#ifndef IO_AWARE_EXACT_FA_DEBUG_H
#define IO_AWARE_EXACT_FA_DEBUG_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Sites recorded with FA_ERR_DEVICE_CHECK (detail[1]). */
typedef enum {
  FA_DBG_META = 100,         /* kv_len / cu_seqlens index */
  FA_DBG_TMA_LOAD = 101,     /* TMA load: coordinates or shared-memory destination */
  FA_DBG_TMA_STORE = 102,    /* TMA store or reduce-add: coordinates or shared-memory source */
  FA_DBG_BULK = 103,         /* bulk row copy: global source range or shared-memory destination */
  FA_DBG_GLOBAL_LOAD = 104,  /* direct global load */
  FA_DBG_GLOBAL_STORE = 105, /* direct global store */
  FA_DBG_SMEM = 106,         /* shared-memory operand or staging index */
  FA_DBG_TMEM = 107          /* TMEM lane quarter or column range */
} fa_debug_site;

/* Takes `rows` rows off every row extent that the checks compare against,
 * for all later calls in the process (0, the default, checks the real
 * extents). The kernels still touch only memory that is there. A check near
 * the end of a tensor then fails and is reported, so a test can see the
 * checks work without an out-of-bounds access. rows < 0 returns
 * FA_ERR_INVALID_ARG. Not thread-safe against calls in flight on other
 * threads, which may see either value. */
FA_API int fa_debug_set_check_slack(int rows);

#ifdef __cplusplus
}
#endif

#endif /* IO_AWARE_EXACT_FA_DEBUG_H */
