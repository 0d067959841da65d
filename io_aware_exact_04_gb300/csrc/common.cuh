// Device-side helpers shared by the attention kernels: bounded mbarrier waits
// that record a status instead of hanging, and 128-byte-swizzled smem address
// arithmetic matching what TMA writes with CU_TENSOR_MAP_SWIZZLE_128B.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_debug.h"
#include "ptx.cuh"

namespace fa {

// Upper bound for any single wait inside a kernel. Every wait in these kernels
// normally completes within microseconds; after this long the CTA gives up,
// records FA_ERR_TIMEOUT in the status word and exits cleanly. A test build
// may set a shorter limit (FA_WAIT_LIMIT_NS).
#ifndef FA_WAIT_LIMIT_NS
#define FA_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr uint64_t kWaitLimitNs = FA_WAIT_LIMIT_NS;

// Test build only (FA_TEST_WITHHOLD, never the library's own build): every CTA leaves out one
// of its TMA copies (the forward's second K/V tile, the backward's second or third Q/dO step),
// so that the wait for it runs out; the test then checks that the kernel reports
// FA_ERR_TIMEOUT, stops cleanly and leaves the CUDA context usable.
#ifdef FA_TEST_WITHHOLD
constexpr bool kWithhold = true;
#else
constexpr bool kWithhold = false;
#endif

// status[0]: first error code, status[1]: wait site, status[2..3]: block index.
struct DevStatus {
  int* word;        // global, 4 ints
  int* abort_smem;  // this CTA's abort flag
};

__device__ __forceinline__ void record_error(const DevStatus& st, int code, int site) {
  if (atomicCAS(st.word, 0, code) == 0) {
    st.word[1] = site;
    st.word[2] = blockIdx.x;
    st.word[3] = blockIdx.y;
  }
  *(volatile int*)st.abort_smem = 1;
}

// A failed argument check inside a kernel, found before the CTA's pipeline exists: records
// FA_ERR_DEVICE_CHECK (code 6) and the site once; the caller carries on or returns.
__device__ __forceinline__ void record_check(int* word, int site) {
  if (atomicCAS(word, 0, 6) == 0) {
    word[1] = site;
    word[2] = blockIdx.x;
    word[3] = blockIdx.y;
  }
}

// ---------------------------------------------------------------------------------------------
// Debug build (FA_DEBUG: libfa_debug.so, never the library's own build). Before use, the kernels
// check the indices of their direct global loads and stores and of the metadata they read
// (kv_len, cu_seqlens). They also check the coordinates and the shared-memory range of every TMA
// or bulk copy, the shared-memory operands of their MMAs, and the TMEM lanes and columns of each
// warp's accumulators. A failed check records FA_ERR_DEVICE_CHECK with its site (fa_debug.h) in
// the status word and raises the CTA's abort flag where the CTA has one, so that the CTA's
// waits give up and it leaves through the same path as after a timeout. The access is skipped.
// In every other build FA_CHECK is the literal `true` and its condition is not compiled.
// FA_SLACK(args) is the debug-only shrink of the row extents the checks compare against (0 in
// every other build); a test sets it so that a check fails on memory that is really there.
#ifdef FA_DEBUG
constexpr bool kDebugChecks = true;
#define FA_CHECK(cond, st, site) ::fa::dbg_check((cond), (st), (site))
#define FA_SLACK(args) ((args).dbg_slack)
#else
constexpr bool kDebugChecks = false;
#define FA_CHECK(cond, st, site) true
#define FA_SLACK(args) 0
#endif

// Check sites recorded with FA_ERR_DEVICE_CHECK.
enum { DBG_META = FA_DBG_META, DBG_TMA_LOAD = FA_DBG_TMA_LOAD, DBG_TMA_STORE = FA_DBG_TMA_STORE,
       DBG_BULK = FA_DBG_BULK, DBG_GLOBAL_LOAD = FA_DBG_GLOBAL_LOAD, DBG_GLOBAL_STORE = FA_DBG_GLOBAL_STORE,
       DBG_SMEM = FA_DBG_SMEM, DBG_TMEM = FA_DBG_TMEM };

__device__ __forceinline__ bool dbg_check(bool ok, const DevStatus& st, int site) {
  if (!ok) {
    if (atomicCAS(st.word, 0, FA_ERR_DEVICE_CHECK) == 0) {
      st.word[1] = site;
      st.word[2] = blockIdx.x;
      st.word[3] = blockIdx.y;
    }
    *(volatile int*)st.abort_smem = 1;
  }
  return ok;
}
__device__ __forceinline__ bool dbg_check(bool ok, int* word, int site) {
  if (!ok) record_check(word, site);
  return ok;
}

// Index idx of a buffer of n elements.
__device__ __forceinline__ bool in_range(long long idx, long long n) { return idx >= 0 && idx < n; }
// The elements [idx, idx + len) of a buffer of n elements.
__device__ __forceinline__ bool span_in(long long idx, long long len, long long n) {
  return idx >= 0 && len >= 0 && idx + len <= n;
}
// A tiled TMA copy at (x, row, z) of a 3-D tensor [outer][rows][inner], box_rows rows high:
// x inside the row on a 16-byte boundary, z inside [0, outer), and the box overlapping rows
// [0, rows). A load may start above row 0 (the rows there read as zero); a store or a
// reduce-add must start at a row of the tensor.
__device__ __forceinline__ bool tma_coords_ok(int x, int row, int z, int inner, int rows, int outer, int elem_bytes,
                                              int box_rows, bool store) {
  if (x < 0 || x >= inner || (x * elem_bytes) % 16 != 0 || z < 0 || z >= outer) return false;
  return store ? (row >= 0 && row < rows) : (row > -box_rows && row < rows);
}
// The shared-memory bytes [addr, addr + bytes) inside [lo, hi).
__device__ __forceinline__ bool smem_in(uint32_t addr, uint32_t bytes, uint32_t lo, uint32_t hi) {
  return addr >= lo && addr + bytes <= hi;
}
// An access of `cols` TMEM columns at taddr by a warp: its lane quarter, and the columns inside
// the allocation of ncols columns at base.
__device__ __forceinline__ bool tmem_in(uint32_t taddr, uint32_t cols, uint32_t base, uint32_t ncols) {
  const uint32_t lane = taddr >> 16, col = taddr & 0xFFFFu, c0 = base & 0xFFFFu;
  return lane < 128 && (lane & 31) == 0 && col >= c0 && col + cols <= c0 + ncols;
}

// Single-thread bounded wait. Returns false if the CTA must abort. SLEEP: after the first
// test, each poll may suspend the thread in hardware for up to 20 us (it resumes as soon as the
// phase completes), so a waiting warp takes no issue slots from the warps still computing.
template <bool SLEEP = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, DevStatus st, int site,
                                             uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t spins = 1;; ++spins) {
    if (SLEEP ? mbar_try_wait_sleep(bar, parity, 20000u) : mbar_try_wait(bar, parity)) return true;
    if ((spins & (SLEEP ? 7u : 63u)) == 0) {
      if (*(volatile int*)st.abort_smem) return false;
      if (*(volatile int*)st.word != 0) {
        *(volatile int*)st.abort_smem = 1;
        return false;
      }
      if (globaltimer_ns() - t0 > limit_ns) {
        record_error(st, FA_ERR_TIMEOUT, site);
        return false;
      }
    }
  }
}

// Whole-warp bounded wait; the result is warp-uniform so that the .sync.aligned
// tcgen05 instructions that follow stay converged.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, DevStatus st, int site) {
  bool ok = wait_bounded(bar, parity, st, site);
  return __all_sync(0xffffffffu, ok);
}
// The same with hardware-suspended polls (the forward kernels, whose softmax warps are
// bound by issue: measured long32768 forward -1.3 %; the backward measured 0.6 % slower).
__device__ __forceinline__ bool wait_warp_sleep(uint32_t bar, uint32_t parity, DevStatus st, int site) {
  bool ok = wait_bounded<true>(bar, parity, st, site);
  return __all_sync(0xffffffffu, ok);
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile whose
// rows are 128 bytes and which TMA fills with 128-byte swizzling (1024-byte atoms).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace fa
