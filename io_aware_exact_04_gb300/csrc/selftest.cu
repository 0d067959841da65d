// Self-checks of the sm_103a building blocks the attention kernels rely on,
// each small enough to isolate one fact:
//  - a single-CTA tcgen05 GEMM, D[128 x N] = A[128 x K] B[K x N], with A from
//    K-major or MN-major smem or from TMEM and B K-major or MN-major, loaded
//    by TMA with 128-byte swizzling; compared on the host with a plain matmul;
//  - the bounded mbarrier wait: a wait nothing will satisfy gives up after a
//    short limit and records FA_ERR_TIMEOUT, leaving the context usable.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "fa_selftest.h"
#include "tmap.h"

namespace fa {

struct GemmArgs {
  const uint32_t* a_words;  // A as packed bf16 pairs, [128][K] (TMEM mode)
  float* d;
  int N, K, mode;
  int* status;
};

__global__ void __launch_bounds__(128, 1)
    selftest_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                         GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const uint32_t sbase = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool a_mn = g.mode & FA_SELFTEST_A_MN, b_mn = g.mode & FA_SELFTEST_B_MN, a_tm = g.mode & FA_SELFTEST_A_TMEM;
  const int K = g.K, N = g.N;
  // smem: A region 32 KB, B region 32 KB, barriers after
  const uint32_t A0 = sbase, B0 = sbase + 32768;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + 65536);
  const uint32_t load_bar = smem_u32(bars), mma_bar = smem_u32(bars + 1);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 2);
  int* abort_flag = reinterpret_cast<int*>(slot + 1);
  DevStatus st{g.status, abort_flag};
  if (threadIdx.x == 0) {
    mbar_init(load_bar, 1);
    mbar_init(mma_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  if (threadIdx.x == 0) {
    int bytes = 0;
    if (!a_tm) {
      if (!a_mn) {  // [128 rows][K]: K/64 blocks of [128][64]
        for (int c = 0; c < K / 64; ++c) tma_load_2d(A0 + c * 16384, &tm_a, c * 64, 0, load_bar);
      } else {      // [K rows][128]: 2 blocks of [K][64]
        for (int c = 0; c < 2; ++c) tma_load_2d(A0 + c * K * 128, &tm_a, c * 64, 0, load_bar);
      }
      bytes += 128 * K * 2;
    }
    if (!b_mn) {  // [N rows][K]: K/64 blocks of [N][64]
      for (int c = 0; c < K / 64; ++c) tma_load_2d(B0 + c * N * 128, &tm_b, c * 64, 0, load_bar);
    } else {      // [K rows][N]: N/64 blocks of [K][64]
      for (int c = 0; c < N / 64; ++c) tma_load_2d(B0 + c * K * 128, &tm_b, c * 64, 0, load_bar);
    }
    bytes += N * K * 2;
    mbar_arrive_expect_tx(load_bar, bytes);
  }
  if (a_tm) {
    // thread t writes row t of A (K/2 packed words) into TMEM columns [256, 256 + K/2)
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t* row = g.a_words + (size_t)threadIdx.x * (K / 2);
    for (int c = 0; c < K / 2; c += 16) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = row[c + i];
      tmem_st16(tmem + lane_off + 256 + c, w);
    }
    tmem_wait_st();
    tc_fence_before();
  }
  __syncthreads();
  bool ok = true;
  if (threadIdx.x == 0) {
    ok = wait_bounded(load_bar, 0, st, 100);
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, N, a_mn ? 1 : 0, b_mn ? 1 : 0);
      for (int k = 0; k < K / 16; ++k) {
        uint64_t bd = b_mn ? sdesc_sw128(B0 + k * 2048, K * 128, 1024)
                           : sdesc_sw128(B0 + (k >> 2) * N * 128 + (k & 3) * 32, 16, 1024);
        if (a_tm) {
          mma_ts(tmem, tmem + 256 + k * 8, bd, idesc, k > 0);
        } else {
          uint64_t ad = a_mn ? sdesc_sw128(A0 + k * 2048, K * 128, 1024)
                             : sdesc_sw128(A0 + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
          mma_ss(tmem, ad, bd, idesc, k > 0);
        }
      }
      mma_commit(mma_bar);
    }
  }
  ok = wait_warp(mma_bar, 0, st, 101) && ok;
  if (ok) {
    tc_fence_after();
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int r = warp * 32 + lane;
    for (int c = 0; c < N; c += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + c, v);
      tmem_wait_ld();
      for (int i = 0; i < 32; ++i) g.d[(size_t)r * N + c + i] = __uint_as_float(v[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__global__ void selftest_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    DevStatus st{status, &abort_flag};
    // nothing arrives on this barrier: the wait must give up and report
    (void)wait_bounded(smem_u32(&bar), 0, st, 99, limit_ns);
  }
}

}  // namespace fa

extern "C" {

int fa_selftest_mma(const void* a, const void* b, float* d, int N, int K, int mode, int* status,
                    fa_stream_t stream) {
  if (!a || !b || !d || !status) return FA_ERR_INVALID_ARG;
  if ((N != 64 && N != 128) || (K != 64 && K != 128) || (mode & ~7)) return FA_ERR_UNSUPPORTED;
  const bool a_mn = mode & FA_SELFTEST_A_MN, b_mn = mode & FA_SELFTEST_B_MN, a_tm = mode & FA_SELFTEST_A_TMEM;
  if (a_tm && a_mn) return FA_ERR_UNSUPPORTED;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap ma, mb;
  bool ok = true;
  if (a_mn)
    ok = ok && fa::make_tmap_2d(&ma, a, BF, 2, 128, K, 64, K, SW);
  else
    ok = ok && fa::make_tmap_2d(&ma, a, BF, 2, K, 128, 64, 128, SW);
  if (b_mn)
    ok = ok && fa::make_tmap_2d(&mb, b, BF, 2, N, K, 64, K, SW);
  else
    ok = ok && fa::make_tmap_2d(&mb, b, BF, 2, K, N, 64, N, SW);
  if (!ok) return FA_ERR_CUDA;
  const int smem = 65536 + 256 + 1024;
  if (cudaFuncSetAttribute(fa::selftest_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  fa::GemmArgs g{static_cast<const uint32_t*>(a), d, N, K, mode, status};
  fa::selftest_gemm_kernel<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(ma, mb, g);
  return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_selftest_wait_timeout(int* status, unsigned int limit_us, fa_stream_t stream) {
  if (!status || limit_us == 0 || limit_us > 5000000u) return FA_ERR_INVALID_ARG;
  fa::selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      status, (unsigned long long)limit_us * 1000ull);
  return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
