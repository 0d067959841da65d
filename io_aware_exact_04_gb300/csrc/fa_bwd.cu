// Backward pass of exact tiled attention on sm_103a, by recomputation.
//
// Method (practice record "Why recomputation is cheaper here than storing";
// handbook "FlashAttention Algorithm > Recomputation Strategy", section "What
// Gets Stored vs Recomputed"): no attention matrix is read; each block of S
// and P is rebuilt from Q, K and the saved per-row statistic, with the same
// tiling as the forward pass, and the gradients of each block are formed at
// once and accumulated. Gradient formulas (softmax-attention Jacobian):
//   D = rowsum(dO * O); P = exp(s Q K^T - LSE); dV += P^T dO; dP = dO V^T;
//   dS = P * (dP - D); dK += s dS^T Q; dQ += s dS K.
//
// Three kernels:
//   bwd_pre_kernel     -D and -LSE (base 2) per query row, zeroed fp32 dQ accumulator
//   main kernel        one CTA per 128-key tile of one head, looping over query steps
//                      (bwd_kernel_d64 for d = 64, bwd_kernel<128> for d = 128). Keys are
//                      the M dimension of every MMA but dQ's:
//                        S^T = K Q_i^T, dP^T = V dO_i^T          (smem x smem)
//                        dV += P^T dO_i, dK += dS^T Q_i           (P^T, dS^T from TMEM)
//                        d=64:  dQ = dS K per pair of steps       (M = 128 query rows)
//                        d=128: dQ_i^T = K^T dS^T                 (M = 128 head dims)
//                      One TMA producer warp, MMA-issuing warp(s), two warpgroups whose
//                      thread r owns key r (TMEM lane r) and forms P^T and dS^T in
//                      registers, and a dQ epilogue warpgroup (TMEM -> scaled fp32 ->
//                      swizzled smem -> TMA reduce-add into the fp32 accumulator).
//   dq_convert_kernel  fp32 accumulator -> bf16 dQ
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "fa_internal.h"
#include "tmap.h"

namespace fa {

#ifdef FA_DEBUG
// Extents that the debug build checks the backward's accesses against, each less the check
// slack. Per tensor-map head: rows of Q / O / dO / dQ, of K / V / dK / dV and of the dQ
// accumulator, and the maps' outer extent. In all: those rows, and the -LSE2 / -D rows. Plain
// [B H, N, d] or packed [H, T, d] (vl) tensors.
struct BwdExt {
  int rows_q, rows_k, rows_acc, heads;
  long long q_rows, k_rows, acc_rows, stat_rows;
};
__device__ __forceinline__ BwdExt bwd_ext(const BwdArgs& a, bool vl) {
  const long long bh = (long long)a.dbg_B * a.H;
  const int sl = a.dbg_slack;
  BwdExt e;
  e.rows_q = (vl ? vl_T(a) : a.N) - sl;
  e.rows_k = (vl ? vl_T(a) : a.Nk) - sl;
  e.rows_acc = a.Npad - sl;
  e.heads = vl ? a.H : (int)bh;
  e.q_rows = (vl ? (long long)a.H * vl_T(a) : bh * a.N) - sl;
  e.k_rows = (vl ? (long long)a.H * vl_T(a) : bh * a.Nk) - sl;
  e.acc_rows = (vl ? (long long)a.H : bh) * a.Npad - sl;
  e.stat_rows = (vl ? (long long)a.H * vl_Lpad(a) : bh * a.Npad) - sl;
  return e;
}
#endif

// ---------------------------------------------------------------------------------------------
// Stored negated, so that the main kernels add them with no extra instruction:
// dvec_i = -D_i = -sum_k dO_ik O_ik; lse2_i = -LSE_i * log2(e) (-inf where no row or
// LSE = -inf, so that recomputed P is 0 there); dq_acc row zeroed. Grid (row blocks, heads):
// one group of D/8 lanes per row, 16 B each, so no index needs a division.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(BwdArgs a, int BH) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int LPR = D / 8;         // lanes per row
  constexpr int RPB = 256 / LPR;     // rows per block
  const int part = threadIdx.x % LPR;
  const int n = blockIdx.x * RPB + threadIdx.x / LPR;
  const int bh = blockIdx.y;
  if (n >= a.Npad) return;  // whole row groups leave together: RPB divides the 128-row padding
  float acc = 0.f;
  if (n < a.N && FA_CHECK(in_range((long long)bh * a.N + n, bwd_ext(a, false).q_rows), a.status, DBG_GLOBAL_LOAD)) {
    const size_t off = ((size_t)bh * a.N + n) * D + part * 8;
    const uint4 ov = *reinterpret_cast<const uint4*>(a.o + off);
    const uint4 gv = *reinterpret_cast<const uint4*>(a.dO + off);
    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
    const uint32_t gw4[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(ow[i] << 16), __uint_as_float(gw4[i] << 16), acc);
      acc = fmaf(__uint_as_float(ow[i] & 0xFFFF0000u), __uint_as_float(gw4[i] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int m = LPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  const size_t r = (size_t)bh * a.Npad + n;
  if (!FA_CHECK(in_range(r, bwd_ext(a, false).acc_rows) && in_range(r, bwd_ext(a, false).stat_rows), a.status,
                DBG_GLOBAL_STORE))
    return;
  float4* dq = reinterpret_cast<float4*>(a.dq_acc + r * D + part * 8);
  dq[0] = make_float4(0.f, 0.f, 0.f, 0.f);
  dq[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (part == 0) {
    a.dvec[r] = -acc;
    float l2 = -INFINITY;
    if (n < a.N) {
      const float l = a.lse[(size_t)bh * a.N + n];
      if (l != -INFINITY) l2 = l * -1.4426950408889634f;
    }
    a.lse2[r] = l2;
  }
}

// fp32 dQ accumulator -> bf16 dQ. Grid (row blocks, heads), each thread two rows' worth of
// 16-byte outputs with both rows' loads in flight before the stores.
template <int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(BwdArgs a, int BH) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int LPR = D / 8;         // threads per row (8 outputs each)
  constexpr int RPB = 256 / LPR;     // rows per block and pass
  const int part = threadIdx.x % LPR;
  const int bh = blockIdx.y;
  const int n0 = blockIdx.x * (2 * RPB) + threadIdx.x / LPR;
  float4 x[2][2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int n = n0 + u * RPB;
    if (n < a.N &&
        FA_CHECK(in_range((long long)bh * a.Npad + n, bwd_ext(a, false).acc_rows), a.status, DBG_GLOBAL_LOAD)) {
      const float4* src = reinterpret_cast<const float4*>(a.dq_acc + ((size_t)bh * a.Npad + n) * D + part * 8);
      x[u][0] = src[0];
      x[u][1] = src[1];
    }
  }
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int n = n0 + u * RPB;
    if (n < a.N && FA_CHECK(in_range((long long)bh * a.N + n, bwd_ext(a, false).q_rows), a.status, DBG_GLOBAL_STORE)) {
      uint4 o;
      o.x = pack_bf16x2(x[u][0].x, x[u][0].y);
      o.y = pack_bf16x2(x[u][0].z, x[u][0].w);
      o.z = pack_bf16x2(x[u][1].x, x[u][1].y);
      o.w = pack_bf16x2(x[u][1].z, x[u][1].w);
      *reinterpret_cast<uint4*>(a.dq + ((size_t)bh * a.N + n) * D + part * 8) = o;
    }
  }
}

// Packed sequences ([H, T, d], cu_seqlens): -D and -LSE2 of sequence b of head h go to rows
// [base_b, base_{b+1}) of the head's Lpad rows, base_b = (cu[b] + 4 b) rounded down to a multiple
// of 4 (16-byte aligned for the main kernels' bulk copies; bases still increase past each
// sequence's end). The rows between a sequence's end and the next base, and the last sequence's
// rows up to Lpad, get -LSE2 = -inf and -D = 0, so a step that reads past a sequence finds
// values that its mask turns into P = 0. Grid (row blocks, sequence x head); the dQ
// accumulator rows of the packed tensor are zeroed as well.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_varlen_kernel(BwdArgs a, int B) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int LPR = D / 8;
  constexpr int RPB = 256 / LPR;
  const int part = threadIdx.x % LPR;
  const int n = blockIdx.x * RPB + threadIdx.x / LPR;  // row within the sequence's slots
  const int b = blockIdx.y / a.H, h = blockIdx.y - b * a.H;
  if (!FA_CHECK(in_range(b + 1, a.dbg_B + 1LL), a.status, DBG_META)) return;
  const int rb = vl_cu(a)[b];
  const int len = vl_cu(a)[b + 1] - rb;
  const int base = (rb + 4 * b) & ~3;
  if (len > vl_maxlen(a) && blockIdx.x == 0 && threadIdx.x == 0) record_check(a.status, 40);  // grid too small
  const int slots = (b + 1 < B) ? (((vl_cu(a)[b + 1] + 4 * (b + 1)) & ~3) - base) : (vl_Lpad(a) - base);
  const bool valid = n < len;
  float acc = 0.f;
  if (valid && FA_CHECK(in_range((long long)h * vl_T(a) + rb + n, bwd_ext(a, true).q_rows) &&
                            in_range((long long)h * a.Npad + rb + n, bwd_ext(a, true).acc_rows),
                        a.status, DBG_GLOBAL_LOAD)) {
    const size_t off = ((size_t)h * vl_T(a) + rb + n) * D + part * 8;
    const uint4 ov = *reinterpret_cast<const uint4*>(a.o + off);
    const uint4 gv = *reinterpret_cast<const uint4*>(a.dO + off);
    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
    const uint32_t gw4[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(ow[i] << 16), __uint_as_float(gw4[i] << 16), acc);
      acc = fmaf(__uint_as_float(ow[i] & 0xFFFF0000u), __uint_as_float(gw4[i] & 0xFFFF0000u), acc);
    }
    float4* dq = reinterpret_cast<float4*>(a.dq_acc + ((size_t)h * a.Npad + rb + n) * D + part * 8);
    dq[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    dq[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int m = LPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (part == 0 && n < slots &&
      FA_CHECK(in_range((long long)h * vl_Lpad(a) + base + n, bwd_ext(a, true).stat_rows), a.status, DBG_GLOBAL_STORE)) {
    const size_t r = (size_t)h * vl_Lpad(a) + base + n;
    a.dvec[r] = valid ? -acc : 0.f;
    float l2 = -INFINITY;
    if (valid && FA_CHECK(in_range((long long)h * vl_T(a) + rb + n, bwd_ext(a, true).q_rows), a.status, DBG_GLOBAL_LOAD)) {
      const float l = a.lse[(size_t)h * vl_T(a) + rb + n];
      if (l != -INFINITY) l2 = l * -1.4426950408889634f;
    }
    a.lse2[r] = l2;
  }
}

// ---------------------------------------------------------------------------------------------
// d = 128 (the d = 64 kernel has its own layout, Bwd64 below). A step is 64 query rows; the
// two warpgroups split its columns. S^T is double-buffered (the next step's S^T is formed while
// the warpgroups still turn the current one into P^T and dS^T); the Q / dO ring has three
// stages so that the copy for step i + 1 lands before its S^T is wanted.
template <int D>
struct BwdCfg {
  static_assert(D == 128, "BwdCfg serves the d = 128 kernel");
  static constexpr int BR = 64;                    // query rows per step
  static constexpr int NSUB = D / 64;
  static constexpr int KSUB = 128 * 128;           // [128 keys][64] bf16 block
  static constexpr int KTILE = NSUB * KSUB;        // K or V tile
  static constexpr int QSUB = BR * 128;            // [BR rows][64] bf16 block
  static constexpr int QTILE = NSUB * QSUB;        // Q_i or dO_i tile
  static constexpr int NSTQ = 3;
  static constexpr int DS_BYTES = 128 * BR * 2;    // dS: [128 keys][BR queries] bf16, 64-query blocks
  static constexpr int DQ_STAGE = BR * D * 4;      // fp32 dQ staging tile (one)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KTILE;
  static constexpr int OFF_Q = OFF_V + KTILE;                 // NSTQ stages, contiguous
  static constexpr int OFF_DO = OFF_Q + NSTQ * QTILE;         // NSTQ stages, contiguous
  static constexpr int OFF_DS = OFF_DO + NSTQ * QTILE;
  static constexpr int OFF_DQ = OFF_DS + DS_BYTES;            // one staging buffer
  static constexpr int OFF_LSE = OFF_DQ + DQ_STAGE;           // NSTQ x BR floats
  static constexpr int OFF_DV = OFF_LSE + NSTQ * BR * 4;      // NSTQ x BR floats
  static constexpr int OFF_BAR = OFF_DV + NSTQ * BR * 4;
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
  // TMEM columns: S^T buffer b at BR b (P^T packed into it), dP^T (dS^T packed into it), dV, dK
  // and one dQ^T buffer (BR query columns of 128 head-dim lanes)
  static constexpr uint32_t TM_ST = 0, TM_DPT = 2 * BR, TM_DV = 3 * BR, TM_DK = 3 * BR + D, TM_DQ = 3 * BR + 2 * D;
  static constexpr uint32_t DQ_COLS = 64;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int THREADS = 448;
  // Each warpgroup owns BR/2 query columns of S^T (and dP^T) in TMEM and packs
  // its bf16 P^T (dS^T) pairs into the first half of its own range, so neither
  // warpgroup overwrites fp32 values the other has not read yet.
  static constexpr int HC = BR / 2;
  __host__ __device__ static constexpr uint32_t pcol(int qc) { return (qc / HC) * HC + (qc % HC) / 2; }
};
static_assert(BwdCfg<128>::TM_DQ + BwdCfg<128>::DQ_COLS <= BwdCfg<128>::TM_COLS, "d = 128 backward: TMEM columns");
static_assert(BwdCfg<128>::SMEM_BYTES <= 232448, "d = 128 backward: shared memory above the 227 KB per-CTA limit");

enum { SITE_B_KV_FULL = 20, SITE_B_QDO_EMPTY, SITE_B_QDO_FULL, SITE_B_S_FULL, SITE_B_DP_FULL, SITE_B_P_READY,
       SITE_B_DS_READY, SITE_B_DQ_EMPTY, SITE_B_DQ_FULL, SITE_B_FINAL, SITE_B_SMEM_ALIGN };

// VL (packed sequences, [H, T, d]): the item is sequence b of head h. Each statement that
// addresses rows has its packed form in an if-constexpr branch beside the plain [BH, N, d]
// one, so the plain kernel compiles exactly as it does without packing.
template <bool VL>
struct SeqD128 {  // packed only: TMA row base and head, row count, -LSE2 / -D and dK / dV row bases
  int rb, nq, zh;
  size_t lrow, krow;
};
template <>
struct SeqD128<false> {};

template <int D, bool VL = false>
__global__ void __launch_bounds__(448, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
               const __grid_constant__ CUtensorMap tm_dqacc, BwdArgs a) {
  griddep_wait();  // before any access to global memory
  griddep_launch_dependents();
  using C = BwdCfg<D>;
  constexpr int BR = C::BR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const uint32_t sbase = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  const uint32_t b0 = smem_u32(bars);
  auto BAR = [&](int i) { return b0 + 8u * i; };
  constexpr int NSTQ = C::NSTQ;
  const uint32_t kv_full = BAR(0);
  auto qdo_full = [&](int s) { return BAR(1 + s); };
  auto qdo_empty = [&](int s) { return BAR(1 + NSTQ + s); };
  auto s_full = [&](int b) { return BAR(1 + 2 * NSTQ + b); };  // S^T buffer b
  const uint32_t dp_full = BAR(3 + 2 * NSTQ), p_ready = BAR(4 + 2 * NSTQ), ds_ready = BAR(5 + 2 * NSTQ);
  const uint32_t dq_full = BAR(6 + 2 * NSTQ), dq_empty = BAR(7 + 2 * NSTQ), final_bar = BAR(8 + 2 * NSTQ);
  static_assert(9 + 2 * NSTQ <= 16, "d = 128 backward: barrier area");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * 16);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  DevStatus st{a.status, abort_flag};

  // blocks launch x-fastest: every head's longest causal key tile (j = 0) goes first
  const int j = blockIdx.y;  // key tile
  const int bh = blockIdx.x;
  const int b = bh / a.H;
  const int k0 = j * 128;
  [[maybe_unused]] SeqD128<VL> sq;
  int kv, n_qt, i_start;
  if constexpr (VL) {
    const int h = bh - b * a.H;
    if (!FA_CHECK(in_range(b + 1, a.dbg_B + 1LL), a.status, DBG_META)) return;
    sq.rb = vl_cu(a)[b];
    sq.nq = vl_cu(a)[b + 1] - sq.rb;
    sq.zh = h;
    sq.lrow = (size_t)h * vl_Lpad(a) + ((sq.rb + 4 * b) & ~3);  // 16-byte aligned for the bulk copies
    sq.krow = (size_t)h * vl_T(a) + sq.rb;
    if (k0 >= sq.nq) return;  // past the sequence: these rows are another sequence's
    kv = sq.nq;
    n_qt = (sq.nq + BR - 1) / BR;
    i_start = a.causal ? k0 / BR : 0;
  } else {
    kv = a.Nk;
    if (a.kv_len && FA_CHECK(in_range(b, a.dbg_B), a.status, DBG_META)) kv = min(max(a.kv_len[b], 0), a.Nk);
    n_qt = (a.N + BR - 1) / BR;
    // causal: the first query row that sees key k0 is k0 - coff
    i_start = a.causal ? max(0, k0 - a.coff) / BR : 0;
  }
  const int n_it = (k0 >= kv || i_start >= n_qt) ? 0 : (n_qt - i_start);

  if (n_it == 0) {
    // no valid key in this tile, or no query sees it: its dK and dV rows are zero
    int rows;
    size_t row0;
    if constexpr (VL) {
      rows = min(128, sq.nq - k0);
      row0 = sq.krow + k0;
    } else {
      rows = min(128, a.Nk - k0);
      row0 = (size_t)bh * a.Nk + k0;
    }
    if (!FA_CHECK(span_in(row0, rows, bwd_ext(a, VL).k_rows), a.status, DBG_GLOBAL_STORE)) return;
    for (int idx = threadIdx.x; idx < rows * (D / 8); idx += blockDim.x) {
      const size_t off = (row0 + idx / (D / 8)) * D + (idx % (D / 8)) * 8;
      *reinterpret_cast<uint4*>(a.dk + off) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(a.dv + off) = make_uint4(0, 0, 0, 0);
    }
    return;
  }

  const float* lse2_h;
  const float* dvec_h;
  if constexpr (VL) {
    lse2_h = a.lse2 + sq.lrow;
    dvec_h = a.dvec + sq.lrow;
  } else {
    lse2_h = a.lse2 + (size_t)bh * a.Npad;
    dvec_h = a.dvec + (size_t)bh * a.Npad;
  }
  // The producer warp initialises the barriers and starts the first copies (K, V and the first
  // NSTQ query steps, whose slots are free) before the CTA-wide setup, hiding their latency. It
  // runs its code with the whole warp and lets one elected lane issue each copy.
  const int n_pre = min(NSTQ, n_it);
  auto load_qdo = [&](int it) {  // whole warp
    if (kWithhold && it == 1) return;  // test build: this copy never arrives
    const int s = it % NSTQ, i = i_start + it;
    const uint32_t bar = qdo_full(s);
    const float* lsrc = lse2_h + (size_t)i * BR;
    const float* dsrc = dvec_h + (size_t)i * BR;
    if (elect_one()) mbar_arrive_expect_tx(bar, 2 * C::QTILE + 2 * BR * 4);
    for (int c = 0; c < C::NSUB; ++c) {
      const bool in =
          FA_CHECK(tma_coords_ok(c * 64, VL ? i * BR + vl_cu(a)[b] : i * BR, VL ? bh - b * a.H : bh, D,
                                 bwd_ext(a, VL).rows_q, bwd_ext(a, VL).heads, 2, BR, false) &&
                       smem_in(sbase + C::OFF_Q + s * C::QTILE + c * C::QSUB, C::QSUB, sbase + C::OFF_Q,
                               sbase + C::OFF_DO) &&
                       smem_in(sbase + C::OFF_DO + s * C::QTILE + c * C::QSUB, C::QSUB, sbase + C::OFF_DO,
                               sbase + C::OFF_DS),
                   st, DBG_TMA_LOAD);
      if constexpr (VL) {
        if (in && elect_one())
          tma_load_3d(sbase + C::OFF_Q + s * C::QTILE + c * C::QSUB, &tm_q, c * 64, sq.rb + i * BR, sq.zh, bar);
        if (in && elect_one())
          tma_load_3d(sbase + C::OFF_DO + s * C::QTILE + c * C::QSUB, &tm_do, c * 64, sq.rb + i * BR, sq.zh, bar);
      } else {
        if (in && elect_one())
          tma_load_3d(sbase + C::OFF_Q + s * C::QTILE + c * C::QSUB, &tm_q, c * 64, i * BR, bh, bar);
        if (in && elect_one())
          tma_load_3d(sbase + C::OFF_DO + s * C::QTILE + c * C::QSUB, &tm_do, c * 64, i * BR, bh, bar);
      }
    }
    // the -LSE2 and -D rows of the step: inside the workspace, 16-byte aligned
    const bool rows_in = FA_CHECK(
        span_in(lsrc - a.lse2, BR, bwd_ext(a, VL).stat_rows) && span_in(dsrc - a.dvec, BR, bwd_ext(a, VL).stat_rows) &&
            ((reinterpret_cast<uintptr_t>(lsrc) | reinterpret_cast<uintptr_t>(dsrc)) & 15) == 0 &&
            smem_in(sbase + C::OFF_LSE + s * BR * 4, BR * 4, sbase + C::OFF_LSE, sbase + C::OFF_DV) &&
            smem_in(sbase + C::OFF_DV + s * BR * 4, BR * 4, sbase + C::OFF_DV, sbase + C::OFF_BAR),
        st, DBG_BULK);
    if (rows_in && elect_one()) bulk_load(sbase + C::OFF_LSE + s * BR * 4, lsrc, BR * 4, bar);
    if (rows_in && elect_one()) bulk_load(sbase + C::OFF_DV + s * BR * 4, dsrc, BR * 4, bar);
    __syncwarp();
  };
  if (warp == 12) {
    if (lane == 0) {
      mbar_init(kv_full, 1);
      for (int s = 0; s < NSTQ; ++s) {
        mbar_init(qdo_full(s), 1);
        mbar_init(qdo_empty(s), 1);
      }
      mbar_init(s_full(0), 1);
      mbar_init(s_full(1), 1);
      mbar_init(dq_full, 1);
      mbar_init(dq_empty, 4);
      mbar_init(dp_full, 1);
      mbar_init(p_ready, 8);
      mbar_init(ds_ready, 8);
      mbar_init(final_bar, 1);
      *abort_flag = 0;
      fence_mbar_init();
    }
    __syncwarp();
    if (elect_one()) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_do);
    }
    if (elect_one()) mbar_arrive_expect_tx(kv_full, 2 * C::KTILE);
    for (int c = 0; c < C::NSUB; ++c) {
      const bool in = FA_CHECK(tma_coords_ok(c * 64, VL ? k0 + vl_cu(a)[b] : k0, VL ? bh - b * a.H : bh, D,
                                             bwd_ext(a, VL).rows_k, bwd_ext(a, VL).heads, 2, 128, false) &&
                                   smem_in(sbase + C::OFF_K + c * C::KSUB, C::KSUB, sbase + C::OFF_K, sbase + C::OFF_V) &&
                                   smem_in(sbase + C::OFF_V + c * C::KSUB, C::KSUB, sbase + C::OFF_V, sbase + C::OFF_Q),
                               st, DBG_TMA_LOAD);
      if constexpr (VL) {
        if (in && elect_one()) tma_load_3d(sbase + C::OFF_K + c * C::KSUB, &tm_k, c * 64, sq.rb + k0, sq.zh, kv_full);
        if (in && elect_one()) tma_load_3d(sbase + C::OFF_V + c * C::KSUB, &tm_v, c * 64, sq.rb + k0, sq.zh, kv_full);
      } else {
        if (in && elect_one()) tma_load_3d(sbase + C::OFF_K + c * C::KSUB, &tm_k, c * 64, k0, bh, kv_full);
        if (in && elect_one()) tma_load_3d(sbase + C::OFF_V + c * C::KSUB, &tm_v, c * 64, k0, bh, kv_full);
      }
    }
    for (int it = 0; it < n_pre; ++it) load_qdo(it);
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    {
      int issued = n_pre;
      for (int it = n_pre; it < n_it; ++it) {
        if (!wait_warp(qdo_empty(it % NSTQ), ((it / NSTQ) & 1) ^ 1, st, SITE_B_QDO_EMPTY)) break;
        load_qdo(it);
        issued = it + 1;
      }
      if (*(volatile int*)abort_flag) {
        // let copies already in flight land before the CTA's smem is released
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(kv_full, 0) && globaltimer_ns() - t0 < 100000000ull) {
        }
        for (int it = max(0, issued - NSTQ); it < issued; ++it)
          while (!mbar_try_wait(qdo_full(it % NSTQ), (it / NSTQ) & 1) && globaltimer_ns() - t0 < 100000000ull) {
          }
      }
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer (whole warp runs
    // the loop; one elected lane issues each MMA and commit)
    {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BR, 0, 0);  // K (or V) x Q_i (or dO_i), K-major
      constexpr uint32_t IDESC_G = idesc_bf16_f32(128, D, 0, 1);   // TMEM A x MN-major B
      constexpr uint32_t IDESC_Q = idesc_bf16_f32(128, 64, 1, 1);  // both operands MN-major
      // Descriptors are formed once; each MMA only adds a constant to the low word.
      constexpr uint32_t HI = sdesc_hi(1024);
      constexpr uint32_t QT16 = C::QTILE >> 4;
      const uint32_t k_lo = sdesc_lo(sbase + C::OFF_K, 16), v_lo = sdesc_lo(sbase + C::OFF_V, 16);
      const uint32_t q_lo = sdesc_lo(sbase + C::OFF_Q, 16), do_lo = sdesc_lo(sbase + C::OFF_DO, 16);
      const uint32_t qmn_lo = sdesc_lo(sbase + C::OFF_Q, C::QSUB), domn_lo = sdesc_lo(sbase + C::OFF_DO, C::QSUB);
      const uint32_t ds_lo = sdesc_lo(sbase + C::OFF_DS, 128 * 128), kmn_lo = sdesc_lo(sbase + C::OFF_K, C::KSUB);
      auto issue_kmajor = [&](uint32_t dst, uint32_t a_lo, uint32_t b_lo) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t oa = ((k >> 2) * C::KSUB + (k & 3) * 32) >> 4;
          const uint32_t ob = ((k >> 2) * C::QSUB + (k & 3) * 32) >> 4;
          if (elect_one()) mma_ss(tmem + dst, sdesc_join(a_lo + oa, HI), sdesc_join(b_lo + ob, HI), IDESC_S, k > 0);
        }
      };
      auto issue_grad = [&](uint32_t dst, uint32_t a_tm, uint32_t b_lo, uint32_t acc) {
#pragma unroll
        for (int k = 0; k < BR / 16; ++k)
          if (elect_one())
            mma_ts(tmem + dst, tmem + a_tm + C::pcol(16 * k), sdesc_join(b_lo + k * (2048 >> 4), HI), IDESC_G,
                   (acc | k) != 0);
      };
      auto commit = [&](uint32_t bar) {
        if (elect_one()) mma_commit(bar);
        __syncwarp();
      };
      auto issue_dq = [&](uint32_t dst) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // 128 keys
          if (!elect_one()) continue;
          if (D == 64)  // dQ = dS K: A = dS (M = queries), B = K (N = head dims)
            mma_ss(tmem + dst, sdesc_join(ds_lo + k * (2048 >> 4), HI), sdesc_join(kmn_lo + k * (2048 >> 4), HI),
                   IDESC_Q, k > 0);
          else  // dQ^T = K^T dS^T: A = K^T (M = head dims), B = dS^T (N = queries)
            mma_ss(tmem + dst, sdesc_join(kmn_lo + k * (2048 >> 4), HI), sdesc_join(ds_lo + k * (2048 >> 4), HI),
                   IDESC_Q, k > 0);
        }
      };
      // Step i: once P^T(i) is complete, S^T(i + 1) goes into the other S^T buffer (whose
      // P^T(i - 1) has been read by dV(i - 1), issued before, and by the warpgroups' dS^T(i - 1),
      // waited for), where it forms while the warpgroups turn dP^T(i) into dS^T(i); then
      // dV(i), dK(i), dQ^T(i) as P^T(i) and dS^T(i) arrive, and dP^T(i + 1) after dK(i) has read
      // dS^T(i) out of the dP^T columns. S^T(i + 1) must not start earlier: both warpgroups
      // count into one p_ready barrier, and a warpgroup that reached P^T(i + 1) first would
      // complete phase i with its second arrivals while the other's P^T(i) is still being
      // stored (dV(i) then reads unfinished columns).
      // the TMEM layout inside this CTA's allocation
      bool ok = FA_CHECK(tmem_in(tmem + C::TM_ST, 2 * BR, tmem, C::TM_COLS) &&
                             tmem_in(tmem + C::TM_DPT, BR, tmem, C::TM_COLS) &&
                             tmem_in(tmem + C::TM_DV, D, tmem, C::TM_COLS) &&
                             tmem_in(tmem + C::TM_DK, D, tmem, C::TM_COLS) &&
                             tmem_in(tmem + C::TM_DQ, C::DQ_COLS, tmem, C::TM_COLS),
                         st, DBG_TMEM) &&
                wait_warp(kv_full, 0, st, SITE_B_KV_FULL) && wait_warp(qdo_full(0), 0, st, SITE_B_QDO_FULL);
      if (ok) {
        tc_fence_after();
        issue_kmajor(C::TM_ST, k_lo, q_lo);
        commit(s_full(0));
        issue_kmajor(C::TM_DPT, v_lo, do_lo);
        commit(dp_full);
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int s = it % NSTQ, sb = it & 1;
        const uint32_t so = s * QT16;
        const bool next = it + 1 < n_it;
        const int s1 = (it + 1) % NSTQ;
        if (!(ok = wait_warp(p_ready, it & 1, st, SITE_B_P_READY))) break;
        // S^T(i + 1) only now: both warpgroups count into the one p_ready barrier, so neither
        // may reach P^T(i + 1), and arrive again, before phase i has completed here
        if (next) {
          if (!(ok = wait_warp(qdo_full(s1), ((it + 1) / NSTQ) & 1, st, SITE_B_QDO_FULL))) break;
          tc_fence_after();
          issue_kmajor(C::TM_ST + (sb ^ 1) * BR, k_lo, q_lo + s1 * QT16);
          commit(s_full(sb ^ 1));
        }
        tc_fence_after();
        issue_grad(C::TM_DV, C::TM_ST + sb * BR, domn_lo + so, it > 0);
        if (!(ok = wait_warp(ds_ready, it & 1, st, SITE_B_DS_READY))) break;
        tc_fence_after();
        issue_grad(C::TM_DK, C::TM_DPT, qmn_lo + so, it > 0);
        // one dQ^T buffer: the epilogue has read out the previous step's
        if (!(ok = wait_warp(dq_empty, (it & 1) ^ 1, st, SITE_B_DQ_EMPTY))) break;
        tc_fence_after();
        issue_dq(C::TM_DQ);
        commit(dq_full);
        commit(qdo_empty(s));  // last readers of Q_i and dO_i issued
        if (next) {
          issue_kmajor(C::TM_DPT, v_lo, do_lo + s1 * QT16);
          commit(dp_full);
        }
      }
      commit(final_bar);  // also the drain: completes after every MMA issued above
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(final_bar, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ epilogue
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // TMEM lane: query row (d=64) or head dim (d=128)
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int tid = threadIdx.x - 256;
    for (int it = 0; it < n_it; ++it) {
      const int i = i_start + it;
      // the four warps leave the loop together, so the named barriers below never wait on a missing warp
      if (!named_bar_and(3, 128, wait_warp(dq_full, it & 1, st, SITE_B_DQ_FULL))) break;
      tc_fence_after();
      uint32_t v[2][32];
      tmem_ld32(tmem + lane_off + C::TM_DQ, v[0]);
      tmem_ld32(tmem + lane_off + C::TM_DQ + 32, v[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_empty);
      // the reduce issued from the staging buffer one step ago has finished reading it
      if (tid == 0) bulk_wait_read0();
      named_bar_sync(3, 128);
      uint8_t* stg = sm + C::OFF_DQ;
      const float sc = a.scale;
      if (D == 64) {
        // row r of a [128 queries][64 dims] fp32 tile, two 32-column swizzled boxes
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float4 x = make_float4(__uint_as_float(v[h][4 * c]) * sc, __uint_as_float(v[h][4 * c + 1]) * sc,
                                   __uint_as_float(v[h][4 * c + 2]) * sc, __uint_as_float(v[h][4 * c + 3]) * sc);
            *reinterpret_cast<float4*>(stg + h * (128 * 128) + sw128_offset(r, c)) = x;
          }
      } else {
        // column r of a [64 queries][128 dims] fp32 tile, four 32-column swizzled boxes
        const int box = r >> 5, within = r & 31;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int q = h * 32 + c;
            *reinterpret_cast<float*>(stg + box * (BR * 128) + sw128_offset(q, within >> 2) + (within & 3) * 4) =
                __uint_as_float(v[h][c]) * sc;
          }
      }
      fence_proxy_async_smem();
      named_bar_sync(3, 128);
      if (tid == 0) {
        constexpr int NBOX = D / 32;
        constexpr int BOX_BYTES = BR * 128;
        for (int x = 0; x < NBOX; ++x) {
          if (!FA_CHECK(tma_coords_ok(x * 32, VL ? i * BR + vl_cu(a)[b] : i * BR, VL ? bh - b * a.H : bh, D,
                                      bwd_ext(a, VL).rows_acc, bwd_ext(a, VL).heads, 4, BR, true) &&
                            smem_in(smem_u32(stg + x * BOX_BYTES), BOX_BYTES, sbase + C::OFF_DQ, sbase + C::OFF_LSE),
                        st, DBG_TMA_STORE))
            continue;
          if constexpr (VL)
            tma_reduce_add_3d(&tm_dqacc, smem_u32(stg + x * BOX_BYTES), x * 32, sq.rb + i * BR, sq.zh);
          else
            tma_reduce_add_3d(&tm_dqacc, smem_u32(stg + x * BOX_BYTES), x * 32, i * BR, bh);
        }
        bulk_commit();
      }
    }
    if (tid == 0) bulk_wait_read0();
  } else {
    // ------------------------------------------------------------ P^T / dS^T warpgroups
    const int wg = warp >> 2;  // which half of the BR query columns
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key within the tile (TMEM lane)
    const int key = k0 + r;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    constexpr int HC = C::HC;      // query columns per warpgroup (64 or 32)
    constexpr int NCH = HC / 32;   // 32-column chunks per warpgroup
    const int c0 = wg * HC;        // first query column of this warpgroup
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it % NSTQ, sb = it & 1;
      const uint32_t tST = C::TM_ST + sb * BR;  // this step's S^T buffer (P^T packed into it)
      const int i = i_start + it;
      const int q0 = i * BR;
      const float* lse_s = reinterpret_cast<const float*>(sm + C::OFF_LSE + s * BR * 4);
      const float* dv_s = reinterpret_cast<const float*>(sm + C::OFF_DV + s * BR * 4);
      if (!(ok = wait_warp(qdo_full(s), (it / NSTQ) & 1, st, SITE_B_QDO_FULL))) break;
      if (!(ok = wait_warp(s_full(sb), (it >> 1) & 1, st, SITE_B_S_FULL))) break;
      tc_fence_after();
      bool need_mask;
      if constexpr (VL)
        need_mask = (k0 + 127 >= kv) || (a.causal && k0 + 127 > q0) || (q0 + BR > sq.nq);
      else
        need_mask = (k0 + 127 >= kv) || (a.causal && k0 + 127 > q0 + a.coff);
      // ---- P^T = exp2(S^T s log2e + lse2), bf16 into the S^T columns (lse2 = -LSE log2e)
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        const int cb = c0 + ch * 32;  // query column base within the tile
        uint32_t sv[32];
        tmem_ld32(tmem + lane_off + tST + cb, sv);
        float lz[32];  // LSE of the 32 queries, broadcast loads
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 t4 = reinterpret_cast<const float4*>(lse_s + cb)[e];
          lz[4 * e] = t4.x, lz[4 * e + 1] = t4.y, lz[4 * e + 2] = t4.z, lz[4 * e + 3] = t4.w;
        }
        tmem_wait_ld();
        if (need_mask) {  // only steps on the diagonal or past kv_len: masked S -> -inf, so P = 0
          if constexpr (VL) {
            const int lim = key >= kv ? 32 : (a.causal ? key - q0 - cb : 0);  // columns [0, lim)
            const int hi = sq.nq - q0 - cb;  // columns [hi, 32) are past the sequence
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c < lim || c >= hi) sv[c] = 0xff800000u;
          } else {
            const int lim = key >= kv ? 32 : (a.causal ? key - a.coff - q0 - cb : 0);  // columns [0, lim)
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c < lim) sv[c] = 0xff800000u;
          }
        }
        uint32_t pk[16];
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float x[2];
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), sl2x2,
                           f2_pack(lz[2 * e], lz[2 * e + 1])),
                    x[0], x[1]);
          pk[e] = pack_bf16x2(ex2_approx(x[0]), ex2_approx(x[1]));
        }
        tmem_st16(tmem + lane_off + tST + C::pcol(cb), pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready);
      // ---- dS^T = P^T * (dP^T + dvec), bf16 into the dP^T columns and into smem (dvec = -D)
      if (!(ok = wait_warp(dp_full, it & 1, st, SITE_B_DP_FULL))) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        const int cb = c0 + ch * 32;
        uint32_t dp[32], pp[16];
        tmem_ld32(tmem + lane_off + C::TM_DPT + cb, dp);
        tmem_ld16(tmem + lane_off + tST + C::pcol(cb), pp);
        float dz[32];  // D of the 32 queries, broadcast loads
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 t4 = reinterpret_cast<const float4*>(dv_s + cb)[e];
          dz[4 * e] = t4.x, dz[4 * e + 1] = t4.y, dz[4 * e + 2] = t4.z, dz[4 * e + 3] = t4.w;
        }
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = __uint_as_float(pp[e] << 16), p1 = __uint_as_float(pp[e] & 0xFFFF0000u);
          // dS = P (dP - D), two columns per paired instruction (dz holds -D)
          const uint64_t t2 = f2_add(f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])),
                                     f2_pack(dz[2 * e], dz[2 * e + 1]));
          float d0, d1;
          f2_unpack(f2_mul(t2, f2_pack(p0, p1)), d0, d1);
          pk[e] = pack_bf16x2(d0, d1);
        }
        tmem_st16(tmem + lane_off + C::TM_DPT + C::pcol(cb), pk);
        // smem dS: row = key r, 64-query blocks of 128 B, 16-byte chunks of 8 queries
        uint8_t* dsb = sm + C::OFF_DS + (cb >> 6) * (128 * 128);
        const int chunk0 = (cb & 63) >> 3;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(dsb + sw128_offset(r, chunk0 + q)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_ready);
    }
    // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes s * dK
    if (ok) ok = wait_warp(final_bar, 0, st, SITE_B_FINAL);
    ok = named_bar_and(1 + wg, 128, ok);  // reached by every warp of the warpgroup
    if (ok) {
      tc_fence_after();
      const uint32_t src = wg == 0 ? C::TM_DV : C::TM_DK;
      const float mul = wg == 0 ? 1.f : a.scale;
      uint8_t* stage = sm + (wg == 0 ? C::OFF_Q : C::OFF_DO);  // both free once every MMA is done
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t x[32];
        tmem_ld32(tmem + lane_off + src + c * 32, x);
        tmem_wait_ld();
        const int blk = (c * 32) >> 6;
        const int chunk0 = ((c * 32) & 63) >> 3;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(x[q * 8 + 0]) * mul, __uint_as_float(x[q * 8 + 1]) * mul);
          v.y = pack_bf16x2(__uint_as_float(x[q * 8 + 2]) * mul, __uint_as_float(x[q * 8 + 3]) * mul);
          v.z = pack_bf16x2(__uint_as_float(x[q * 8 + 4]) * mul, __uint_as_float(x[q * 8 + 5]) * mul);
          v.w = pack_bf16x2(__uint_as_float(x[q * 8 + 6]) * mul, __uint_as_float(x[q * 8 + 7]) * mul);
          if constexpr (VL) {
            if (k0 + 128 > sq.nq) {  // the tile runs past its sequence: rows written directly
              if (k0 + r < sq.nq &&
                  FA_CHECK(in_range(sq.krow + k0 + r, bwd_ext(a, VL).k_rows), st, DBG_GLOBAL_STORE))
                *reinterpret_cast<uint4*>((wg == 0 ? a.dv : a.dk) + (sq.krow + k0 + r) * D + c * 32 + q * 8) = v;
              continue;
            }
          }
          *reinterpret_cast<uint4*>(stage + blk * C::KSUB + sw128_offset(r, chunk0 + q)) = v;
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + wg, 128);
      bool tma_out = wq == 0 && lane == 0;
      if constexpr (VL) tma_out = tma_out && k0 + 128 <= sq.nq;
      if (tma_out) {
        for (int c = 0; c < C::NSUB; ++c) {
          if (!FA_CHECK(tma_coords_ok(c * 64, VL ? k0 + vl_cu(a)[b] : k0, VL ? bh - b * a.H : bh, D,
                                      bwd_ext(a, VL).rows_k, bwd_ext(a, VL).heads, 2, 128, true) &&
                            smem_in(smem_u32(stage + c * C::KSUB), C::KSUB, sbase + C::OFF_Q, sbase + C::OFF_DS),
                        st, DBG_TMA_STORE))
            continue;
          if constexpr (VL)
            tma_store_3d(wg == 0 ? &tm_dv : &tm_dk, smem_u32(stage + c * C::KSUB), c * 64, sq.rb + k0, sq.zh);
          else
            tma_store_3d(wg == 0 ? &tm_dv : &tm_dk, smem_u32(stage + c * C::KSUB), c * 64, k0, bh);
        }
        bulk_commit();
        bulk_wait_read0();  // the staging tile must outlive the copy's reads
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// ---------------------------------------------------------------------------------------------
// d = 64 backward, persistent: G CTAs (one per SM) loop over the 128-key tiles of every head.
// Tile t is key tile j = t / BH of head t % BH, so for causal attention the longest tiles come
// first; CTA c takes tile r G + c in even rounds r and r G + G - 1 - c in odd ones. Within a
// tile the 64-query steps are double-buffered: warpgroup w (w = 0, 1) owns TMEM buffer w of
// S^T and dP^T and the steps of global index parity w, so the tensor core forms S^T, dP^T of
// the next step while a warpgroup turns the current one into P^T and dS^T; dQ is formed per pair
// of steps (128 queries, M = 128) from a double-buffered dS tile in shared memory. The global
// step index runs on across tiles, so MMA issue flows from one tile into the next; K and V are
// double-buffered, and the dV / dK epilogue (TMEM -> bf16 -> TMA store, then the accumulators
// zeroed for the next tile) runs on the dQ epilogue warps while the warpgroups move on.
struct Bwd64 {
  static constexpr int D = 64, BR = 64;           // queries per step
  // Q/dO ring depth: four stages keep the copy of step g+2 clear of the readers of step g-1
  // (three measured 40 % slower); the epilogue warps need one staging buffer.
  static constexpr int NQS = 5;
  static constexpr int NSTG = 1;
  static constexpr int KTILE = 128 * 128;          // K or V tile: [128 keys][64] bf16
  static constexpr int QTILE = BR * 128;           // Q_i or dO_i: [64 rows][64] bf16
  static constexpr int DS_BYTES = 128 * 128 * 2;   // dS of a pair: [128 keys][2 blocks of 64 queries]
  static constexpr int STG_BYTES = 16384;          // staging: [128][32] fp32 dQ, or [128][64] bf16 dV / dK
  static constexpr int OFF_KV = 0;                           // 2 buffers, each K then V
  static constexpr int OFF_Q = 4 * KTILE;                    // NQS stages
  static constexpr int OFF_DO = OFF_Q + NQS * QTILE;         // NQS stages
  static constexpr int OFF_DS = OFF_DO + NQS * QTILE;        // 2 buffers (even / odd pairs)
  static constexpr int OFF_STG = OFF_DS + 2 * DS_BYTES;
  static constexpr int OFF_LSE = OFF_STG + NSTG * STG_BYTES; // NQS x BR floats
  static constexpr int OFF_DV = OFF_LSE + NQS * BR * 4;      // NQS x BR floats
  static constexpr int OFF_BAR = OFF_DV + NQS * BR * 4;
  // no alignment slack: the kernel checks that dynamic shared memory starts 1024-byte aligned
  static constexpr int BAR_BYTES = 272;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES;
  __host__ __device__ static constexpr int off_k(int b) { return OFF_KV + b * 2 * KTILE; }
  __host__ __device__ static constexpr int off_v(int b) { return OFF_KV + b * 2 * KTILE + KTILE; }
  // TMEM: S^T buffer w at 64 w (P^T packed in its first 32 columns), dP^T buffer w at
  // 128 + 64 w (dS^T packed likewise), dV 256, dK 320, dQ buffer c at 384 + 64 c.
  static constexpr uint32_t TM_ST = 0, TM_DPT = 128, TM_DV = 256, TM_DK = 320, TM_DQ = 384;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int THREADS = 480;
};
static_assert(Bwd64::SMEM_BYTES <= 232448, "d = 64 backward: shared memory above the 227 KB per-CTA limit");
static_assert(8 * (4 + 2 * Bwd64::NQS + 17) + 12 <= Bwd64::BAR_BYTES, "d = 64 backward: barrier area");

// One key tile of the persistent schedule.
struct TileD64 {
  int bh, k0, kv, n_it, i_start;
};
// Where work item bh's rows live. VL (packed sequences, [H, T, d]): item bh is sequence
// b = bh / H of head h, its rows start at TMA row rb of head zh and it has nq query (and key)
// rows; its -LSE2 / -D rows start at lrow and its dK / dV rows at krow. Without VL these are
// the plain [BH, N, d] offsets (rb = 0), so that code compiles as it did without packing.
struct SeqD64 {
  int rb, nq, zh;
  size_t lrow, krow;
};
template <bool VL>
__device__ __forceinline__ SeqD64 seq_d64(int bh, const BwdArgs& a) {
  SeqD64 q;
  if (VL) {
    const int b = bh / a.H, h = bh - b * a.H;
    if (FA_CHECK(in_range(b + 1, a.dbg_B + 1LL), a.status, DBG_META)) {
      q.rb = vl_cu(a)[b];
      q.nq = vl_cu(a)[b + 1] - q.rb;
    } else {
      q.rb = 0;
      q.nq = 0;
    }
    q.zh = h;
    q.lrow = (size_t)h * vl_Lpad(a) + ((q.rb + 4 * b) & ~3);  // 16-byte aligned for the bulk copies
    q.krow = (size_t)h * vl_T(a) + q.rb;
  } else {
    q.rb = 0;
    q.nq = a.N;
    q.zh = bh;
    q.lrow = (size_t)bh * a.Npad;
    q.krow = (size_t)bh * a.Nk;
  }
  return q;
}
template <bool VL>
__device__ __forceinline__ TileD64 tile_d64(int t, const BwdArgs& a) {
  TileD64 r;
  const int j = t / a.BH;
  r.bh = t - j * a.BH;
  r.k0 = j * 128;
  int nq = a.N;
  if (VL) {
    nq = seq_d64<VL>(r.bh, a).nq;
    r.kv = nq;  // a tile past its sequence gets no work (and writes nothing: see the epilogue)
  } else {
    r.kv = a.Nk;
    if (a.kv_len && FA_CHECK(in_range(r.bh / a.H, a.dbg_B), a.status, DBG_META))
      r.kv = min(max(a.kv_len[r.bh / a.H], 0), a.Nk);
  }
  const int n_qt = (nq + Bwd64::BR - 1) / Bwd64::BR;
  // causal: the first query row that sees key k0 is k0 - coff; steps start on a 128-row
  // boundary (even) so that dQ pairs cover whole 128-row blocks
  r.i_start = a.causal ? (max(0, r.k0 - (VL ? 0 : a.coff)) >> 7) << 1 : 0;
  const int n = (r.k0 >= r.kv || r.i_start >= n_qt) ? 0 : (n_qt - r.i_start);
  // whole pairs: a trailing step past the last query reads masked (or zero) Q / dO rows and adds nothing
  r.n_it = n + (n & 1);
  return r;
}
// Tile of round r for CTA c of G, or -1 past the end (later rounds are past it too).
__device__ __forceinline__ int sched_d64(int r, int c, int G, int T) {
  const int t = r * G + ((r & 1) ? (G - 1 - c) : c);
  return t < T ? t : -1;
}
// First tile with work at or after round r; returns its round, or -1.
template <bool VL>
__device__ __forceinline__ int next_work_d64(int r, int c, int G, int T, const BwdArgs& a, TileD64& out) {
  for (;; ++r) {
    const int t = sched_d64(r, c, G, T);
    if (t < 0) return -1;
    out = tile_d64<VL>(t, a);
    if (out.n_it > 0) return r;
  }
}

template <bool VL>
__global__ void __launch_bounds__(480, 1)
    bwd_kernel_d64(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                   const __grid_constant__ CUtensorMap tm_dqacc, BwdArgs a) {
  griddep_wait();  // before any access to global memory
  griddep_launch_dependents();
  using C = Bwd64;
  constexpr int BR = C::BR, NQS = C::NQS;
  extern __shared__ uint8_t smem_raw[];
  // the layout has no room for alignment slack: dynamic shared memory must start on a 1024-byte
  // boundary (the 128-byte swizzle atoms); otherwise record a device check and do nothing
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_check(a.status, SITE_B_SMEM_ALIGN);
    return;
  }
  uint8_t* sm = smem_raw;
  const uint32_t sbase = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  const uint32_t b0 = smem_u32(bars);
  auto BAR = [&](int i) { return b0 + 8u * i; };
  auto kv_full = [&](int b) { return BAR(b); };
  auto kv_empty = [&](int b) { return BAR(2 + b); };
  auto qdo_full = [&](int s) { return BAR(4 + s); };
  auto qdo_empty = [&](int s) { return BAR(4 + NQS + s); };
  constexpr int nb = 4 + 2 * NQS;
  auto s_full = [&](int w) { return BAR(nb + w); };
  auto dp_full = [&](int w) { return BAR(nb + 2 + w); };
  auto p_ready = [&](int w) { return BAR(nb + 4 + w); };
  auto ds_ready = [&](int w) { return BAR(nb + 6 + w); };
  auto dq_full = [&](int c) { return BAR(nb + 8 + c); };
  auto dq_empty = [&](int c) { return BAR(nb + 10 + c); };
  auto dq_done = [&](int c) { return BAR(nb + 12 + c); };
  const uint32_t tile_done = BAR(nb + 14);  // every MMA of a tile complete (one commit per issuing warp)
  const uint32_t acc_free = BAR(nb + 15);   // dV / dK read out and zeroed (one arrival per epilogue warp)
  const uint32_t final_bar = BAR(nb + 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * (nb + 17));
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  // number of dS^T steps warpgroup 0 has finished, times 4 (one add per warp)
  const uint32_t ds0_count = smem_u32(tmem_slot + 2);
  DevStatus st{a.status, abort_flag};

  const int T = a.BH * (((VL ? vl_maxlen(a) : a.Nk) + 127) >> 7);
  const int G = gridDim.x, cta = blockIdx.x;

  // The producer warp initialises the barriers and starts the first copies (K, V and the first
  // NQS steps of this CTA's first tile, whose slots are free) before the CTA-wide setup, hiding
  // their latency. It runs its code with the whole warp and lets one elected lane issue each copy.
  auto load_kv = [&](int b, const TileD64& tl) {  // whole warp
    const SeqD64 sq = seq_d64<VL>(tl.bh, a);
    const bool in = FA_CHECK(tma_coords_ok(0, sq.rb + tl.k0, sq.zh, C::D, bwd_ext(a, VL).rows_k, bwd_ext(a, VL).heads,
                                           2, 128, false) &&
                                 smem_in(sbase + C::off_k(b), C::KTILE, sbase + C::OFF_KV, sbase + C::OFF_Q) &&
                                 smem_in(sbase + C::off_v(b), C::KTILE, sbase + C::OFF_KV, sbase + C::OFF_Q),
                             st, DBG_TMA_LOAD);
    if (elect_one()) mbar_arrive_expect_tx(kv_full(b), 2 * C::KTILE);
    if (in && elect_one()) tma_load_3d(sbase + C::off_k(b), &tm_k, 0, sq.rb + tl.k0, sq.zh, kv_full(b));
    if (in && elect_one()) tma_load_3d(sbase + C::off_v(b), &tm_v, 0, sq.rb + tl.k0, sq.zh, kv_full(b));
    __syncwarp();
  };
  auto load_qdo = [&](int gs, const TileD64& tl, int it) {  // whole warp
    if (kWithhold && gs == 2) return;  // test build: this copy never arrives
    const int s = gs % NQS, i = tl.i_start + it;
    const uint32_t bar = qdo_full(s);
    const SeqD64 sq = seq_d64<VL>(tl.bh, a);
    const float* lsrc = a.lse2 + sq.lrow + (size_t)i * BR;
    const float* dsrc = a.dvec + sq.lrow + (size_t)i * BR;
    // (a step that completes the tile's last pair may start up to one step past the last row:
    // TMA reads zeros there, and its columns are masked)
    const bool in = FA_CHECK(tma_coords_ok(0, sq.rb + i * BR, sq.zh, C::D, bwd_ext(a, VL).rows_q + BR,
                                           bwd_ext(a, VL).heads, 2, BR, false) &&
                                 smem_in(sbase + C::OFF_Q + s * C::QTILE, C::QTILE, sbase + C::OFF_Q, sbase + C::OFF_DO) &&
                                 smem_in(sbase + C::OFF_DO + s * C::QTILE, C::QTILE, sbase + C::OFF_DO, sbase + C::OFF_DS),
                             st, DBG_TMA_LOAD);
    // the -LSE2 and -D rows of the step: inside the workspace, 16-byte aligned
    const bool rows_in = FA_CHECK(
        span_in(lsrc - a.lse2, BR, bwd_ext(a, VL).stat_rows) && span_in(dsrc - a.dvec, BR, bwd_ext(a, VL).stat_rows) &&
            ((reinterpret_cast<uintptr_t>(lsrc) | reinterpret_cast<uintptr_t>(dsrc)) & 15) == 0 &&
            smem_in(sbase + C::OFF_LSE + s * BR * 4, BR * 4, sbase + C::OFF_LSE, sbase + C::OFF_DV) &&
            smem_in(sbase + C::OFF_DV + s * BR * 4, BR * 4, sbase + C::OFF_DV, sbase + C::OFF_BAR),
        st, DBG_BULK);
    if (elect_one()) mbar_arrive_expect_tx(bar, 2 * C::QTILE + 2 * BR * 4);
    if (in && elect_one()) tma_load_3d(sbase + C::OFF_Q + s * C::QTILE, &tm_q, 0, sq.rb + i * BR, sq.zh, bar);
    if (in && elect_one()) tma_load_3d(sbase + C::OFF_DO + s * C::QTILE, &tm_do, 0, sq.rb + i * BR, sq.zh, bar);
    if (rows_in && elect_one()) bulk_load(sbase + C::OFF_LSE + s * BR * 4, lsrc, BR * 4, bar);
    if (rows_in && elect_one()) bulk_load(sbase + C::OFF_DV + s * BR * 4, dsrc, BR * 4, bar);
    __syncwarp();
  };
  int pre_steps = 0;  // steps of the first tile issued before the setup
  if (warp == 12) {
    if (lane == 0) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(kv_full(b), 1);
        mbar_init(kv_empty(b), 2);  // one commit per MMA-issuing warp
      }
      for (int s = 0; s < NQS; ++s) {
        mbar_init(qdo_full(s), 1);
        mbar_init(qdo_empty(s), 1);
      }
      for (int w = 0; w < 2; ++w) {
        mbar_init(s_full(w), 1);
        mbar_init(dp_full(w), 1);
        mbar_init(p_ready(w), 4);
        mbar_init(ds_ready(w), 4);
        mbar_init(dq_full(w), 1);
        mbar_init(dq_empty(w), 4);
        mbar_init(dq_done(w), 1);
      }
      mbar_init(tile_done, 2);
      mbar_init(acc_free, 4);
      mbar_init(final_bar, 2);
      *abort_flag = 0;
      tmem_slot[2] = 0;
      fence_mbar_init();
    }
    __syncwarp();
    TileD64 tl;
    if (next_work_d64<VL>(0, cta, G, T, a, tl) >= 0) {
      if (elect_one()) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_do);
      }
      load_kv(0, tl);
      pre_steps = min(NQS, tl.n_it);
      for (int it = 0; it < pre_steps; ++it) load_qdo(it, tl, it);
    }
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp < 8) {
    // dV (warpgroup 0) and dK (warpgroup 1) start at zero: the two MMA-issuing warps then
    // always accumulate, whichever reaches a tile first (the epilogue zeroes them per tile)
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0;
    const uint32_t base = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (warp < 4 ? C::TM_DV : C::TM_DK);
    tmem_st32(base, z);
    tmem_st32(base + 32, z);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    int gs0 = 0, tu = 0, issued = 0, kv_loads = 0;
    bool ok = true;
    TileD64 tl;
    for (int r = next_work_d64<VL>(0, cta, G, T, a, tl); ok && r >= 0; r = next_work_d64<VL>(r + 1, cta, G, T, a, tl)) {
      const int b = tu & 1;
      if (tu > 0) {  // the first tile's K and V went out before the setup
        if (!(ok = wait_warp(kv_empty(b), ((tu >> 1) & 1) ^ 1, st, SITE_B_QDO_EMPTY))) break;
        load_kv(b, tl);
      }
      ++kv_loads;
      for (int it = (tu == 0 ? pre_steps : 0); it < tl.n_it; ++it) {
        const int gs = gs0 + it;
        if (!(ok = wait_warp(qdo_empty(gs % NQS), ((gs / NQS) & 1) ^ 1, st, SITE_B_QDO_EMPTY))) break;
        load_qdo(gs, tl, it);
      }
      gs0 += tl.n_it;
      issued = gs0;
      ++tu;
    }
    if (*(volatile int*)abort_flag) {
      // let copies already in flight land before the CTA's smem is released
      const uint64_t t0 = globaltimer_ns();
      for (int u = max(0, kv_loads - 2); u < kv_loads; ++u)
        while (!mbar_try_wait(kv_full(u & 1), (u >> 1) & 1) && globaltimer_ns() - t0 < 100000000ull) {
        }
      for (int gs = max(0, issued - NQS); gs < issued; ++gs)
        while (!mbar_try_wait(qdo_full(gs % NQS), (gs / NQS) & 1) && globaltimer_ns() - t0 < 100000000ull) {
        }
    }
  } else if (warp == 13 || warp == 14) {
    // ------------------------------------------------------------ MMA issuers: warp 13 serves
    // warpgroup 0 (even global steps), warp 14 warpgroup 1 (odd steps) and forms dQ. The whole
    // warp runs the loop; one elected lane issues each MMA and commit.
    const int w = warp - 13;
    constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BR, 0, 0);  // K (V) x Q_i (dO_i), K-major
    constexpr uint32_t IDESC_G = idesc_bf16_f32(128, 64, 0, 1);  // TMEM A x MN-major B
    constexpr uint32_t IDESC_Q = idesc_bf16_f32(128, 64, 1, 1);  // dS x K, both MN-major
    constexpr uint32_t HI = sdesc_hi(1024);
    constexpr uint32_t QT16 = C::QTILE >> 4;
    const uint32_t q_lo = sdesc_lo(sbase + C::OFF_Q, 16), do_lo = sdesc_lo(sbase + C::OFF_DO, 16);
    const uint32_t qmn_lo = sdesc_lo(sbase + C::OFF_Q, C::QTILE), domn_lo = sdesc_lo(sbase + C::OFF_DO, C::QTILE);
    const uint32_t ds_lo = sdesc_lo(sbase + C::OFF_DS, 128 * 128);
    auto k_lo = [&](int b) { return sdesc_lo(sbase + C::off_k(b), 16); };
    auto v_lo = [&](int b) { return sdesc_lo(sbase + C::off_v(b), 16); };
    auto kmn_lo = [&](int b) { return sdesc_lo(sbase + C::off_k(b), C::KTILE); };
    auto commit = [&](uint32_t bar) {
      if (elect_one()) mma_commit(bar);
      __syncwarp();
    };
    auto issue_s = [&](int gs, int b) {  // S^T of global step gs into buffer gs % 2
      const uint32_t so = (gs % NQS) * QT16, kl = k_lo(b);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (elect_one())
          mma_ss(tmem + C::TM_ST + 64 * (gs & 1), sdesc_join(kl + 2 * k, HI), sdesc_join(q_lo + so + 2 * k, HI),
                 IDESC_S, k > 0);
      commit(s_full(gs & 1));
    };
    auto issue_dp = [&](int gs, int b) {  // dP^T of global step gs into buffer gs % 2
      const uint32_t so = (gs % NQS) * QT16, vl = v_lo(b);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (elect_one())
          mma_ss(tmem + C::TM_DPT + 64 * (gs & 1), sdesc_join(vl + 2 * k, HI), sdesc_join(do_lo + so + 2 * k, HI),
                 IDESC_S, k > 0);
      commit(dp_full(gs & 1));
    };
    // dV (dK) += P^T (dS^T) [128 keys x 64 queries, TMEM] x dO_i (Q_i) [64 queries x 64 dims]
    auto issue_grad = [&](uint32_t dst, uint32_t a_tm, uint32_t b_lo) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (elect_one())
          mma_ts(tmem + dst, tmem + a_tm + 8 * k, sdesc_join(b_lo + k * (2048 >> 4), HI), IDESC_G, 1);
    };
    // This warp's first step starts its buffers. Afterwards S^T(g+2) follows dV(g) as soon as the
    // warpgroup has P^T(g) (it keeps P in registers for dS, so S^T's columns are free), and
    // dP^T(g+2) follows dK(g) once dS^T(g) is written; step g+2 may belong to the next tile.
    bool ok = true;
    int gs0 = 0, tu = 0;
    TileD64 cur, nxt;
    int r = next_work_d64<VL>(0, cta, G, T, a, cur);
    if (r >= 0) {
      // the TMEM layout inside this CTA's allocation, then the first copies
      ok = FA_CHECK(tmem_in(tmem + C::TM_ST, 128, tmem, C::TM_COLS) && tmem_in(tmem + C::TM_DPT, 128, tmem, C::TM_COLS) &&
                        tmem_in(tmem + C::TM_DV, C::D, tmem, C::TM_COLS) &&
                        tmem_in(tmem + C::TM_DK, C::D, tmem, C::TM_COLS) &&
                        tmem_in(tmem + C::TM_DQ, 128, tmem, C::TM_COLS),
                    st, DBG_TMEM) &&
           wait_warp(kv_full(0), 0, st, SITE_B_KV_FULL) && wait_warp(qdo_full(w), 0, st, SITE_B_QDO_FULL);
      if (ok) {
        tc_fence_after();
        issue_s(w, 0);
        issue_dp(w, 0);
      }
    }
    while (ok && r >= 0) {
      const int b = tu & 1;
      const int r2 = next_work_d64<VL>(r + 1, cta, G, T, a, nxt);
      for (int it = w; ok && it < cur.n_it; it += 2) {
        const int gs = gs0 + it;
        const uint32_t par = (gs >> 1) & 1;
        const uint32_t so = (gs % NQS) * QT16;
        const bool in_tile = it + 2 < cur.n_it;
        const bool succ = in_tile || r2 >= 0;
        const int b2 = in_tile ? b : (b ^ 1);
        if (!(ok = wait_warp(p_ready(w), par, st, SITE_B_P_READY))) break;
        if (it == w && tu > 0) {  // the epilogue has read and zeroed the previous tile's dV, dK
          if (!(ok = wait_warp(acc_free, (tu - 1) & 1, st, SITE_B_FINAL))) break;
        }
        tc_fence_after();
        issue_grad(C::TM_DV, C::TM_ST + 64 * w, domn_lo + so);
        if (succ) {
          if (!in_tile && !(ok = wait_warp(kv_full(b2), ((tu + 1) >> 1) & 1, st, SITE_B_KV_FULL))) break;
          if (!(ok = wait_warp(qdo_full((gs + 2) % NQS), ((gs + 2) / NQS) & 1, st, SITE_B_QDO_FULL))) break;
          tc_fence_after();
          issue_s(gs + 2, b2);
        }
        if (!(ok = wait_warp(ds_ready(w), par, st, SITE_B_DS_READY))) break;
        tc_fence_after();
        issue_grad(C::TM_DK, C::TM_DPT + 64 * w, qmn_lo + so);
        commit(qdo_empty(gs % NQS));  // last readers of Q_i and dO_i issued
        if (succ) issue_dp(gs + 2, b2);
        if (w == 1) {  // the pair (gs-1, gs) is complete once warpgroup 0's dS of step gs-1 is in smem
          const int pg = gs >> 1, c = pg & 1;
          const uint32_t need = 4u * (uint32_t)(pg + 1);
          if (lane == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (smem_ld_acquire(ds0_count) < need) {
              if (*(volatile int*)abort_flag || *(volatile int*)a.status != 0) {
                *(volatile int*)abort_flag = 1;
                ok = false;
                break;
              }
              if (globaltimer_ns() - t0 > kWaitLimitNs) {
                record_error(st, FA_ERR_TIMEOUT, SITE_B_DS_READY);
                ok = false;
                break;
              }
            }
          }
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
          if (!(ok = wait_warp(dq_empty(c), ((pg >> 1) & 1) ^ 1, st, SITE_B_DQ_EMPTY))) break;
          tc_fence_after();
          const uint32_t dsb = ds_lo + c * (C::DS_BYTES >> 4), kb = kmn_lo(b);
#pragma unroll
          for (int k = 0; k < 8; ++k)  // 128 keys
            if (elect_one())
              mma_ss(tmem + C::TM_DQ + 64 * c, sdesc_join(dsb + k * (2048 >> 4), HI),
                     sdesc_join(kb + k * (2048 >> 4), HI), IDESC_Q, k > 0);
          commit(dq_full(c));
          commit(dq_done(c));
        }
      }
      if (!ok) break;
      commit(tile_done);    // every MMA of this tile issued by this warp
      commit(kv_empty(b));  // ... and with them the last readers of this tile's K and V
      gs0 += cur.n_it;
      ++tu;
      cur = nxt;
      r = r2;
    }
    commit(final_bar);  // also the drain: completes after every MMA issued above
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(final_bar, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ epilogue warps: dQ of each pair
    // (reduced into the fp32 accumulator), then each tile's dV and dK
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int tid = threadIdx.x - 256;
    const float sc = a.scale;
    // Staging buffers are used in strict rotation (dQ halves, then a tile's dV and dK); before
    // writing one, the copy that last read it (NSTG copies back) must have finished reading.
    int ng = 0;
    auto stage_acquire = [&]() -> uint8_t* {
      if (tid == 0) {
        if (C::NSTG == 1)
          bulk_wait_read0();
        else
          asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
      }
      named_bar_sync(3, 128);
      return sm + C::OFF_STG + (ng++ % C::NSTG) * C::STG_BYTES;
    };
    bool ok = true;
    int gs0 = 0, tu = 0;
    for (int rr = 0; ok; ++rr) {
      const int t = sched_d64(rr, cta, G, T);
      if (t < 0) break;
      const TileD64 tl = tile_d64<VL>(t, a);
      const SeqD64 sq = seq_d64<VL>(tl.bh, a);
      if (tl.n_it == 0) {  // no valid key in this tile: its dK and dV rows are zero
        if (VL && tl.k0 >= sq.nq) continue;  // past its sequence: those rows are another sequence's
        const int rows = min(128, (VL ? sq.nq : a.Nk) - tl.k0);
        if (!FA_CHECK(span_in(sq.krow + tl.k0, rows, bwd_ext(a, VL).k_rows), st, DBG_GLOBAL_STORE)) continue;
        for (int idx = tid; idx < rows * (C::D / 8); idx += 128) {
          const size_t off = (sq.krow + tl.k0 + idx / (C::D / 8)) * C::D + (idx % (C::D / 8)) * 8;
          *reinterpret_cast<uint4*>(a.dk + off) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(a.dv + off) = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      for (int p = 0; p < tl.n_it / 2; ++p) {
        const int pg = (gs0 >> 1) + p, c = pg & 1;
        if (!(ok = named_bar_and(3, 128, wait_warp(dq_full(c), (pg >> 1) & 1, st, SITE_B_DQ_FULL)))) break;
        tc_fence_after();
        uint32_t v[2][32];
        tmem_ld32(tmem + lane_off + C::TM_DQ + 64 * c, v[0]);
        tmem_ld32(tmem + lane_off + C::TM_DQ + 64 * c + 32, v[1]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dq_empty(c));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint8_t* stg = stage_acquire();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 x = make_float4(__uint_as_float(v[h][4 * k]) * sc, __uint_as_float(v[h][4 * k + 1]) * sc,
                                         __uint_as_float(v[h][4 * k + 2]) * sc, __uint_as_float(v[h][4 * k + 3]) * sc);
            *reinterpret_cast<float4*>(stg + sw128_offset(r, k)) = x;
          }
          fence_proxy_async_smem();
          named_bar_sync(3, 128);
          if (tid == 0) {
            if (FA_CHECK(tma_coords_ok(h * 32, sq.rb + (tl.i_start + 2 * p) * BR, sq.zh, C::D, bwd_ext(a, VL).rows_acc,
                                       bwd_ext(a, VL).heads, 4, 128, true) &&
                             smem_in(smem_u32(stg), C::STG_BYTES, sbase + C::OFF_STG, sbase + C::OFF_LSE),
                         st, DBG_TMA_STORE))
              tma_reduce_add_3d(&tm_dqacc, smem_u32(stg), h * 32, sq.rb + (tl.i_start + 2 * p) * BR, sq.zh);
            bulk_commit();
          }
        }
      }
      if (!ok) break;
      // ---- this tile's dV and s * dK -> bf16 -> staging -> TMA store. dV is staged and stored
      //      first; once dK is in registers both accumulators are zeroed and handed back to
      //      the issuers (the next tile's first dV / dK MMAs wait for that), before dK waits
      //      for the staging buffer.
      if (!(ok = named_bar_and(3, 128, wait_warp(tile_done, tu & 1, st, SITE_B_FINAL)))) break;
      tc_fence_after();
      auto load_packed = [&](uint32_t col, float mul, uint32_t (&out)[32]) {
        uint32_t x[2][32];
        tmem_ld32(tmem + lane_off + col, x[0]);
        tmem_ld32(tmem + lane_off + col + 32, x[1]);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          out[e] = pack_bf16x2(__uint_as_float(x[e >> 4][(2 * e) & 31]) * mul,
                               __uint_as_float(x[e >> 4][(2 * e + 1) & 31]) * mul);
      };
      auto stage_store = [&](const uint32_t (&pk)[32], const CUtensorMap* map, uint16_t* gdst) {
        if (VL && tl.k0 + 128 > sq.nq) {  // the tile runs past its sequence: rows written directly
          if (tl.k0 + r < sq.nq &&
              FA_CHECK(in_range(sq.krow + tl.k0 + r, bwd_ext(a, VL).k_rows), st, DBG_GLOBAL_STORE)) {
            uint4* dst = reinterpret_cast<uint4*>(gdst + (sq.krow + tl.k0 + r) * C::D);
#pragma unroll
            for (int q = 0; q < 8; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
          return;
        }
        uint8_t* stg = stage_acquire();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(stg + sw128_offset(r, q)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        fence_proxy_async_smem();
        named_bar_sync(3, 128);
        if (tid == 0) {
          if (FA_CHECK(tma_coords_ok(0, sq.rb + tl.k0, sq.zh, C::D, bwd_ext(a, VL).rows_k, bwd_ext(a, VL).heads, 2, 128,
                                     true) &&
                           smem_in(smem_u32(stg), C::STG_BYTES, sbase + C::OFF_STG, sbase + C::OFF_LSE),
                       st, DBG_TMA_STORE))
            tma_store_3d(map, smem_u32(stg), 0, sq.rb + tl.k0, sq.zh);
          bulk_commit();
        }
      };
      {
        uint32_t pk[32];
        load_packed(C::TM_DV, 1.f, pk);
        stage_store(pk, &tm_dv, a.dv);
      }
      {
        uint32_t pk[32];
        load_packed(C::TM_DK, sc, pk);
        uint32_t z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0;
        tmem_st32(tmem + lane_off + C::TM_DV, z);
        tmem_st32(tmem + lane_off + C::TM_DV + 32, z);
        tmem_st32(tmem + lane_off + C::TM_DK, z);
        tmem_st32(tmem + lane_off + C::TM_DK + 32, z);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_free);
        stage_store(pk, &tm_dk, a.dk);
      }
      gs0 += tl.n_it;
      ++tu;
    }
    if (tid == 0) bulk_wait_read0();  // the staging buffer must outlive the copies' reads
  } else {
    // ------------------------------------------------------------ P^T / dS^T warpgroups
    const int w = warp >> 2;       // this warpgroup's steps: global index % 2 == w
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key within the tile (TMEM lane)
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float sl2 = a.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    const uint32_t tST = tmem + lane_off + C::TM_ST + 64 * w, tDPT = tmem + lane_off + C::TM_DPT + 64 * w;
    bool ok = true;
    int gs0 = 0;
    TileD64 tl;
    for (int rr = next_work_d64<VL>(0, cta, G, T, a, tl); ok && rr >= 0; rr = next_work_d64<VL>(rr + 1, cta, G, T, a, tl)) {
      const int key = tl.k0 + r;
      const int nq = VL ? seq_d64<VL>(tl.bh, a).nq : 0;  // VL: query columns past it are masked
      for (int it = w; it < tl.n_it; it += 2) {
        const int gs = gs0 + it;
        const int s = gs % NQS;
        const uint32_t par = (gs >> 1) & 1;
        const int q0 = (tl.i_start + it) * BR;
        const float* lse_s = reinterpret_cast<const float*>(sm + C::OFF_LSE + s * BR * 4);
        const float* dv_s = reinterpret_cast<const float*>(sm + C::OFF_DV + s * BR * 4);
        if (!(ok = wait_warp(qdo_full(s), (gs / NQS) & 1, st, SITE_B_QDO_FULL))) break;
        if (!(ok = wait_warp(s_full(w), par, st, SITE_B_S_FULL))) break;
        tc_fence_after();
        const bool need_mask = (tl.k0 + 127 >= tl.kv) || (a.causal && tl.k0 + 127 > q0 + (VL ? 0 : a.coff)) ||
                               (VL && q0 + BR > nq);
        // ---- P^T = exp2(S^T s log2e + lse2) (lse2 = -LSE log2e) -> bf16 pairs in the first 32
        //      columns of this buffer, kept in registers too: S^T's columns are overwritten by
        //      the next step once P^T is out
        // Both 32-column halves are loaded before one wait, so the TMEM load latency is paid once.
        uint32_t pkeep[32];
        {
          uint32_t sv[2][32];
          tmem_ld32(tST, sv[0]);
          tmem_ld32(tST + 32, sv[1]);
          tmem_wait_ld();
          if (need_mask) {  // only steps on the diagonal or past kv_len: masked S -> -inf, so P = 0
            const int lim = key >= tl.kv ? 64 : (a.causal ? key - (VL ? 0 : a.coff) - q0 : 0);  // columns [0, lim)
            const int hi = VL ? nq - q0 : 64;  // VL: columns [hi, 64) are past the sequence
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c < lim || c >= hi) sv[c >> 5][c & 31] = 0xff800000u;
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            // lse2 of the 64 queries: 16-byte broadcast loads (one shared-memory wavefront each)
            const float4 l4 = reinterpret_cast<const float4*>(lse_s)[e >> 1];
            float x0, x1;
            const uint32_t* se = &sv[e >> 4][(2 * e) & 31];
            const uint64_t s2 = f2_pack(__uint_as_float(se[0]), __uint_as_float(se[1]));
            f2_unpack(f2_fma(s2, sl2x2, (e & 1) ? f2_pack(l4.z, l4.w) : f2_pack(l4.x, l4.y)), x0, x1);
            pkeep[e] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
          }
          tmem_st32(tST, pkeep);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready(w));
        // ---- dS^T = P^T * (dP^T + dvec) -> bf16 pairs in this dP^T buffer and into the pair's dS tile
        if (!(ok = wait_warp(dp_full(w), par, st, SITE_B_DP_FULL))) break;
        tc_fence_after();
        const int pg = gs >> 1;
        uint8_t* dsb = sm + C::OFF_DS + (pg & 1) * C::DS_BYTES + w * (128 * 128);
        if (w == 0 && pg >= 2) {  // dQ of the pair that last used this dS tile has read it
          if (!(ok = wait_warp(dq_done(pg & 1), ((pg - 2) >> 1) & 1, st, SITE_B_DQ_EMPTY))) break;
        }
        {
          // dP^T in two halves, each waited for on its own: loading both before one wait needs
          // 32 more live registers than the 128 this kernel has per thread
          uint32_t dp[2][32];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tmem_ld32(tDPT + 32 * h, dp[h]);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int g = 16 * h + e;
              const float4 d4 = reinterpret_cast<const float4*>(dv_s)[g >> 1];
              const float2 d2 = (g & 1) ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
              const float p0 = __uint_as_float(pkeep[g] << 16), p1 = __uint_as_float(pkeep[g] & 0xFFFF0000u);
              const uint64_t t2 = f2_add(f2_pack(__uint_as_float(dp[h][2 * e]), __uint_as_float(dp[h][2 * e + 1])),
                                         f2_pack(d2.x, d2.y));
              float d0, d1;
              f2_unpack(f2_mul(t2, f2_pack(p0, p1)), d0, d1);
              pk[e] = pack_bf16x2(d0, d1);
            }
            tmem_st16(tDPT + 16 * h, pk);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(dsb + sw128_offset(r, 4 * h + q)) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(ds_ready(w));
          if (w == 0) smem_add_release(ds0_count, 1);
        }
      }
      gs0 += tl.n_it;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

template <int D>
static int launch_bwd_pre_d(const BwdArgs& a, int BH, cudaStream_t stream) {
  constexpr int RPB = 256 / (D / 8);
  const dim3 grid((unsigned)((a.Npad + RPB - 1) / RPB), (unsigned)BH);
  return launch_pdl(__func__, bwd_pre_kernel<D>, grid, dim3(256), 0, stream, a, BH);
}

// BH = B * H work items per key tile. VL: tensors are [H, T, d] (all sequences' rows packed
// per head): the maps span T rows (the dQ accumulator Npad) and H heads.
template <int D, bool VL = false>
static int launch_bwd_main_d(const void* q, const void* k, const void* v, const BwdArgs& a, int BH,
                             cudaStream_t stream) {
  constexpr int BR = 64;  // query rows per step of both main kernels (Bwd64::BR, BwdCfg<128>::BR)
  static_assert(Bwd64::BR == BR && BwdCfg<128>::BR == BR, "query rows per step");
  const uint64_t N = (uint64_t)(VL ? vl_T(a) : a.N), Nk = (uint64_t)(VL ? vl_T(a) : a.Nk);
  const uint64_t Z = (uint64_t)(VL ? a.H : BH);
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap mq, mk, mv, mdo, mdk, mdv, mdq;
  if (!make_tmap_3d(&mq, q, BF, 2, D, N, Z, 64, BR, SW) || !make_tmap_3d(&mdo, a.dO, BF, 2, D, N, Z, 64, BR, SW) ||
      !make_tmap_3d(&mk, k, BF, 2, D, Nk, Z, 64, 128, SW) || !make_tmap_3d(&mv, v, BF, 2, D, Nk, Z, 64, 128, SW) ||
      !make_tmap_3d(&mdk, a.dk, BF, 2, D, Nk, Z, 64, 128, SW) ||
      !make_tmap_3d(&mdv, a.dv, BF, 2, D, Nk, Z, 64, 128, SW) ||
      !make_tmap_3d(&mdq, a.dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, (uint64_t)a.Npad, Z, 32,
                    (D == 64) ? 128 : BR, SW))
    return cuda_fail("cuTensorMapEncodeTiled", 0, "tensor map rejected");
  static bool attr_set = false;  // benign race: idempotent
  const int n_kt = ((VL ? vl_maxlen(a) : a.Nk) + 127) / 128;
  dim3 grid(BH, n_kt);
  if constexpr (D == 64) {
    if (!attr_set) {
      const cudaError_t e = cudaFuncSetAttribute(bwd_kernel_d64<VL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Bwd64::SMEM_BYTES);
      if (e != cudaSuccess) return cuda_fail("cudaFuncSetAttribute", (int)e, cudaGetErrorName(e));
      attr_set = true;
    }
    // persistent: one CTA per SM (at most one per key tile)
    int sms = 0;
    if (!sm_count(&sms)) return FA_ERR_CUDA;
    const long long tiles = (long long)BH * n_kt;
    BwdArgs ap = a;
    ap.BH = BH;
    return launch_pdl(__func__, bwd_kernel_d64<VL>, dim3((unsigned)std::min<long long>(tiles, sms)),
                      dim3(Bwd64::THREADS), Bwd64::SMEM_BYTES, stream, mq, mk, mv, mdo, mdk, mdv, mdq, ap);
  } else {
    using C = BwdCfg<D>;
    if (!attr_set) {
      const cudaError_t e =
          cudaFuncSetAttribute(bwd_kernel<D, VL>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
      if (e != cudaSuccess) return cuda_fail("cudaFuncSetAttribute", (int)e, cudaGetErrorName(e));
      attr_set = true;
    }
    return launch_pdl(__func__, bwd_kernel<D, VL>, grid, dim3(C::THREADS), C::SMEM_BYTES, stream, mq, mk, mv, mdo,
                      mdk, mdv, mdq, a);
  }
}

template <int D>
static int launch_bwd_convert_d(const BwdArgs& a, int BH, cudaStream_t stream) {
  constexpr int RPB = 256 / (D / 8);
  const dim3 grid((unsigned)((a.N + 2 * RPB - 1) / (2 * RPB)), (unsigned)BH);
  return launch_pdl(__func__, dq_convert_kernel<D>, grid, dim3(256), 0, stream, a, BH);
}

int launch_bwd_stage(int stage, const void* q, const void* k, const void* v, const BwdArgs& a, int BH, int d,
                     cudaStream_t stream) {
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  switch (stage) {
    case 0: return d == 64 ? launch_bwd_pre_d<64>(a, BH, stream) : launch_bwd_pre_d<128>(a, BH, stream);
    case 1:
      return d == 64 ? launch_bwd_main_d<64>(q, k, v, a, BH, stream) : launch_bwd_main_d<128>(q, k, v, a, BH, stream);
    case 2: return d == 64 ? launch_bwd_convert_d<64>(a, BH, stream) : launch_bwd_convert_d<128>(a, BH, stream);
    default: return FA_ERR_INVALID_ARG;
  }
}

// Packed sequences: stage 0 the -D / -LSE2 rows (aligned per sequence) and the zeroed dQ
// accumulator, 1 the main kernel over (sequence x head, key tile), 2 the dQ rounding over
// all H * T rows. args.BH = B * H.
int launch_bwd_varlen_stage(int stage, const void* q, const void* k, const void* v, const BwdArgs& a, int B, int H,
                            int d, cudaStream_t stream) {
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  switch (stage) {
    case 0: {
      const int rpb = 256 / (d / 8);
      const dim3 grid((unsigned)((vl_maxlen(a) + 262 + rpb - 1) / rpb), (unsigned)(B * H));
      return d == 64 ? launch_pdl("bwd_pre_varlen_kernel", bwd_pre_varlen_kernel<64>, grid, dim3(256), 0, stream, a, B)
                     : launch_pdl("bwd_pre_varlen_kernel", bwd_pre_varlen_kernel<128>, grid, dim3(256), 0, stream, a,
                                  B);
    }
    case 1:
      return d == 64 ? launch_bwd_main_d<64, true>(q, k, v, a, B * H, stream)
                     : launch_bwd_main_d<128, true>(q, k, v, a, B * H, stream);
    case 2: {
      BwdArgs c = a;  // rows of the packed tensor: H items of T rows
      c.N = vl_T(a);
      return d == 64 ? launch_bwd_convert_d<64>(c, H, stream) : launch_bwd_convert_d<128>(c, H, stream);
    }
    default: return FA_ERR_INVALID_ARG;
  }
}

}  // namespace fa
