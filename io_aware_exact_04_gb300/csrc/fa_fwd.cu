// Forward pass of exact tiled attention on sm_103a.
//
// Method (practice record "Why recomputation is cheaper here than storing"):
// each block of scores is formed in on-chip memory, consumed at once by a
// blockwise softmax with a running row maximum and normaliser, and never
// written to HBM; only O and the per-row statistics leave the chip
// (handbook "FlashAttention Algorithm > Recomputation Strategy", section
// "What Gets Stored vs Recomputed"; here m and l are folded into LSE).
//
// GB300 mapping (one CTA = two 128-row query tiles of one head):
//   warp 8      TMA producer: Q tiles once, then K_j / V_j 128-key tiles
//               through an NST-stage ring of 128-byte-swizzled smem tiles.
//   warp 9      TMEM allocator and single-thread tcgen05.mma issuer:
//               S_t = Q_t K_j^T (smem x smem -> TMEM fp32, M=128, N=128),
//               O_t += P_t V_j (P from TMEM as bf16, V from smem, N=d).
//   warps 0-3   softmax for query tile 0, warps 4-7 for tile 1; thread r of a
//               warpgroup owns row r (TMEM lane r): running max/normaliser in
//               registers, P written back over S in TMEM, O rescaled in TMEM
//               only when the row maximum grows by more than 2^8 (exact: O and
//               l always share the same reference maximum).
// The issuer alternates the two tiles (PV_0, S_0 next, PV_1, S_1 next) so one
// warpgroup's softmax overlaps the other's tensor-core work.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "fa_internal.h"
#include "tmap.h"

namespace fa {

template <int D, bool SPLIT = false>
struct FwdCfg {
  static constexpr int NSUB = D / 64;              // 128-byte column blocks per row
  static constexpr int SUB_BYTES = 128 * 128;      // one [128 rows][64 bf16] block
  static constexpr int TILE_BYTES = NSUB * SUB_BYTES;
  // K/V ring depth. The split d = 64 kernel may give alternate ring tiles to its two query
  // lanes (dual mode), so each lane sees only half of the ring ahead: six stages there.
  static constexpr int NST = (D == 64) ? (SPLIT ? 6 : 3) : 2;
  static constexpr int OFF_Q = 0;                  // two query tiles
  static constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NST * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NST * TILE_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // barriers + alignment slack
  // TMEM columns. d = 64: S_t at 128 t, P_t (bf16 pairs) at 256 + 64 t, O_t at 384 + 64 t,
  // so S_t is free again as soon as its values are in registers. d = 128: S_t at
  // 128 t with P_t written over its first 64 columns, O_t at 256 + 128 t.
  static constexpr bool SEP_P = (D == 64);
  __device__ static constexpr uint32_t tm_s(int t) { return 128u * t; }
  __device__ static constexpr uint32_t tm_p(int t) { return SEP_P ? 256u + 64u * t : 128u * t; }
  __device__ static constexpr uint32_t tm_o(int t) { return SEP_P ? 384u + 64u * t : 256u + (uint32_t)D * t; }
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int THREADS = 352;
  // MMA-issuing threads: d = 64 one per query tile (warps 9, 10); d = 128 one
  // (warp 9) for both tiles, P_t over S_t forcing S_t(j+1) behind PV_t(j) anyway.
  static constexpr int NMMA = SEP_P ? 2 : 1;
};

static_assert(FwdCfg<64, true>::SMEM_BYTES <= 232448, "split d = 64 forward: shared memory above 227 KB");
static_assert(8 * (1 + 3 * FwdCfg<64, true>::NST + 9) + 8 <= 256, "split d = 64 forward: barrier area");

// Wait-site identifiers recorded with FA_ERR_TIMEOUT.
enum { SITE_F_KV_EMPTY = 1, SITE_F_Q_FULL, SITE_F_K_FULL, SITE_F_V_FULL, SITE_F_P_READY, SITE_F_S_FULL,
       SITE_F_O_DONE, SITE_F_DRAIN, SITE_F_S_FREE, SITE_F_SEQLEN };

// Key tiles that the query tile of rows [qs, qs + 128) needs: those below kv (the valid keys)
// that some row of the tile may see. Causal row i sees keys j <= i + coff.
__device__ __forceinline__ int key_tiles(int qs, int nq, int nkt, int causal, int coff) {
  if (qs >= nq) return 0;
  if (!causal) return nkt;
  const int lim = min(qs + 128, nq) + coff;  // keys [0, lim) are visible to some row
  return lim <= 0 ? 0 : min(nkt, (lim + 127) >> 7);
}

#ifdef FA_DEBUG
// Extents that the debug build checks the forward's accesses against, each less the check slack:
// rows per tensor-map head of Q / O and of K / V, the maps' outer extent, and the rows of O and
// LSE and of the split partials in all; plain [B H, N, d] or packed [H, T, d] (vl) tensors.
struct FwdExt {
  int rows_q, rows_k, heads;
  long long o_rows, part_rows;
};
__device__ __forceinline__ FwdExt fwd_ext(const FwdArgs& a, bool vl) {
  const long long bh = (long long)a.dbg_B * a.H;
  FwdExt e;
  e.rows_q = (vl ? a.T : a.N) - a.dbg_slack;
  e.rows_k = (vl ? a.T : a.Nk) - a.dbg_slack;
  e.heads = vl ? a.H : (int)bh;
  e.o_rows = (vl ? (long long)a.H * a.T : bh * a.N) - a.dbg_slack;
  e.part_rows = 2LL * a.n_split * bh * a.N - a.dbg_slack;
  return e;
}
#endif

// ONE (plain rows only): the CTA takes one 128-row query tile instead of a pair (a.n_pairs then
// counts tiles), its second lane idle; for grids of pairs too small to fill the SMs, where
// one lane alone runs a tile faster than two sharing an SM.
// SPLIT: the CTA (head, query pair, share z) runs key tiles [jb, je) of its item, the
// z-th of a.n_split near-equal shares, and writes normalised partial O (fp32) and LSE to
// slots 2z and 2z + 1 of a.part_o / a.part_lse for fwd_combine_kernel; the same
// running-maximum rescaling that joins key tiles inside a CTA then joins the slots.
template <int D, bool SPLIT, bool VL = false, bool ONE = false>
__global__ void __launch_bounds__(352, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, FwdArgs a) {
  griddep_wait();  // before any access to global memory
  griddep_launch_dependents();
  using C = FwdCfg<D, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const uint32_t sbase = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // barriers
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  const uint32_t b0 = smem_u32(bars);
  auto BAR = [&](int i) { return b0 + 8u * i; };
  const uint32_t q_full = BAR(0);
  auto k_full = [&](int s) { return BAR(1 + s); };
  auto v_full = [&](int s) { return BAR(1 + C::NST + s); };
  auto kv_empty = [&](int s) { return BAR(1 + 2 * C::NST + s); };
  const int nb = 1 + 3 * C::NST;
  auto s_full = [&](int t) { return BAR(nb + t); };
  auto p_ready = [&](int t) { return BAR(nb + 2 + t); };
  auto o_done = [&](int t) { return BAR(nb + 4 + t); };
  auto s_free = [&](int t) { return BAR(nb + 6 + t); };
  const uint32_t drain = BAR(nb + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * (nb + 9));
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  DevStatus st{a.status, abort_flag};

  // work description
  // blocks launch x-fastest: every head's longest causal query pair goes first
  const int pair = a.n_pairs - 1 - (int)blockIdx.y;
  const int bh = blockIdx.x;
  const int b = bh / a.H;
  // VL (packed sequences, layout [H, T, d]): this CTA's sequence b has rows [cu[b], cu[b+1])
  // of head h; NQ is its query count, rbase the TMA row of its first row, zh the TMA head
  // coordinate and obase the index of its row 0 among the O / LSE rows
  int NQ = a.N, rbase = 0, zh = bh;
  size_t obase = (size_t)bh * a.N;
  if (VL) {
    const int h = bh - b * a.H;
    if (FA_CHECK(in_range(b + 1, a.dbg_B + 1LL), a.status, DBG_META)) {
      rbase = a.cu_seqlens[b];
      NQ = a.cu_seqlens[b + 1] - rbase;
    } else {
      NQ = 0;
    }
    zh = h;
    obase = (size_t)h * a.T + rbase;
    if (NQ > a.max_seqlen && threadIdx.x == 0 && blockIdx.y == 0) record_check(a.status, SITE_F_SEQLEN);
    if ((a.n_pairs - 1 - (int)blockIdx.y) * 256 >= NQ) return;  // this pair lies past the sequence
  }
  int kv = VL ? NQ : a.Nk;
  if (!VL && a.kv_len && FA_CHECK(in_range(b, a.dbg_B), a.status, DBG_META)) kv = min(max(a.kv_len[b], 0), a.Nk);
  const int nkt = (kv + 127) >> 7;
  static_assert(!ONE || (!SPLIT && !VL), "one query tile per CTA: plain rows only");
  const int q0 = pair * (ONE ? 128 : 256);
  int n_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t)
    n_t[t] = (ONE && t == 1) ? 0 : key_tiles(q0 + t * 128, NQ, nkt, a.causal, VL ? 0 : a.coff);
  // key tiles run here: [jb, jb + nmax), all of them without a split; loops count from 0.
  // dual (split only): the item's second query tile lies past N, so query lane 1 takes the
  // same rows as lane 0 and the two lanes split the share's key tiles, even ones to lane 0
  // and odd ones to lane 1; each lane's result is a partial of its own for the combine.
  int jb = 0, nmax;
  const bool dual = SPLIT && D == 64 && q0 + 128 >= NQ && n_t[0] > 0;
  if (SPLIT) {
    const int nall = max(n_t[0], n_t[1]);
    const int z = blockIdx.z;
    jb = (int)((long long)z * nall / a.n_split);
    const int je = (int)((long long)(z + 1) * nall / a.n_split);
    if (dual) {
      n_t[0] = (je - jb + 1) >> 1;
      n_t[1] = (je - jb) >> 1;
      nmax = je - jb;  // ring tiles of both lanes
    } else {
#pragma unroll
      for (int t = 0; t < 2; ++t) n_t[t] = max(0, min(n_t[t], je) - jb);
      nmax = max(n_t[0], n_t[1]);
    }
  } else {
    nmax = max(n_t[0], n_t[1]);
  }

  // The producer warp initialises the barriers and starts the first copies (Q and the first
  // NST K/V stages, whose slots are free) before the CTA-wide setup, hiding their latency. It
  // runs its code with the whole warp and lets one elected lane issue each copy.
  const int n_pre = min(C::NST, nmax);
  auto load_kv = [&](int j) {  // whole warp
    if (kWithhold && j == 1) return;  // test build: this copy never arrives
    const int s = j % C::NST;
    const uint32_t kf = k_full(s), vf = v_full(s);
    const uint32_t kd = sbase + C::OFF_K + s * C::TILE_BYTES, vd = sbase + C::OFF_V + s * C::TILE_BYTES;
    if (elect_one()) mbar_arrive_expect_tx(kf, C::TILE_BYTES);
    for (int c = 0; c < C::NSUB; ++c)
      if (FA_CHECK(tma_coords_ok(c * 64, rbase + (jb + j) * 128, zh, D, fwd_ext(a, VL).rows_k, fwd_ext(a, VL).heads, 2,
                                 128, false) &&
                       smem_in(kd + c * C::SUB_BYTES, C::SUB_BYTES, sbase + C::OFF_K, sbase + C::OFF_V),
                   st, DBG_TMA_LOAD) &&
          elect_one())
        tma_load_3d(kd + c * C::SUB_BYTES, &tm_k, c * 64, rbase + (jb + j) * 128, zh, kf);
    if (elect_one()) mbar_arrive_expect_tx(vf, C::TILE_BYTES);
    for (int c = 0; c < C::NSUB; ++c)
      if (FA_CHECK(tma_coords_ok(c * 64, rbase + (jb + j) * 128, zh, D, fwd_ext(a, VL).rows_k, fwd_ext(a, VL).heads, 2,
                                 128, false) &&
                       smem_in(vd + c * C::SUB_BYTES, C::SUB_BYTES, sbase + C::OFF_V, sbase + C::OFF_BAR),
                   st, DBG_TMA_LOAD) &&
          elect_one())
        tma_load_3d(vd + c * C::SUB_BYTES, &tm_v, c * 64, rbase + (jb + j) * 128, zh, vf);
    __syncwarp();
  };
  if (warp == 8) {
    if (lane == 0) {
      mbar_init(q_full, 1);
      for (int s = 0; s < C::NST; ++s) {
        mbar_init(k_full(s), 1);
        mbar_init(v_full(s), 1);
        mbar_init(kv_empty(s), C::NMMA);  // one arrival per MMA-issuing warp
      }
      for (int t = 0; t < 2; ++t) {
        mbar_init(s_full(t), 1);
        mbar_init(p_ready(t), 4);
        mbar_init(o_done(t), 1);
        mbar_init(s_free(t), 4);
      }
      mbar_init(drain, C::NMMA);
      *abort_flag = 0;
      fence_mbar_init();
    }
    __syncwarp();
    if (nmax > 0) {
      if (elect_one()) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
      }
      const int nq = (n_t[1] > 0) ? 2 : 1;
      if (elect_one()) mbar_arrive_expect_tx(q_full, nq * C::TILE_BYTES);
      for (int t = 0; t < nq; ++t)
        for (int s = 0; s < C::NSUB; ++s) {
          const uint32_t dst = sbase + C::OFF_Q + t * C::TILE_BYTES + s * C::SUB_BYTES;
          const int row = rbase + q0 + (dual ? 0 : t * 128);
          if (FA_CHECK(tma_coords_ok(s * 64, row, zh, D, fwd_ext(a, VL).rows_q, fwd_ext(a, VL).heads, 2, 128, false) &&
                           smem_in(dst, C::SUB_BYTES, sbase, sbase + C::OFF_K),
                       st, DBG_TMA_LOAD) &&
              elect_one())
            tma_load_3d(dst, &tm_q, s * 64, row, zh, q_full);
        }
      for (int j = 0; j < n_pre; ++j) load_kv(j);
    }
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (nmax > 0) {
      int issued = n_pre;
      for (int j = n_pre; j < nmax; ++j) {
        if (!wait_warp_sleep(kv_empty(j % C::NST), ((j / C::NST) & 1) ^ 1, st, SITE_F_KV_EMPTY)) break;
        load_kv(j);
        issued = j + 1;
      }
      if (*(volatile int*)abort_flag) {
        // let copies already in flight land before the CTA's smem is released
        for (int j = max(0, issued - C::NST); j < issued; ++j) {
          const int s = j % C::NST;
          const uint32_t par = (j / C::NST) & 1;
          const uint64_t t0 = globaltimer_ns();
          while (!(mbar_try_wait(k_full(s), par) && mbar_try_wait(v_full(s), par)) &&
                 globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers: for d = 64 warp 9
    // serves query tile 0 and warp 10 query tile 1, each in its own order; for d = 128
    // warp 9 serves both, alternating. The whole warp runs the loop; one elected lane issues.
    if (nmax > 0 && warp - 9 < C::NMMA) {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, 0, 0);  // Q, K both K-major
      constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, 0, 1);    // P from TMEM, V MN-major
      // Descriptors are formed once; each MMA only adds a constant to the low word.
      constexpr uint32_t HI = sdesc_hi(1024);
      const uint32_t q_lo = sdesc_lo(sbase + C::OFF_Q, 16);
      const uint32_t k_lo = sdesc_lo(sbase + C::OFF_K, 16);
      const uint32_t v_lo = sdesc_lo(sbase + C::OFF_V, C::SUB_BYTES);
      constexpr uint32_t TILE16 = C::TILE_BYTES >> 4;
      auto issue_s = [&](int t, int kst) {  // S_t = Q_t K^T (K from stage kst)
        const uint32_t qa = q_lo + t * TILE16, ka = k_lo + kst * TILE16, d = tmem + C::tm_s(t);
        if (!FA_CHECK(smem_in(sbase + C::OFF_Q + t * C::TILE_BYTES, C::TILE_BYTES, sbase, sbase + C::OFF_K) &&
                          smem_in(sbase + C::OFF_K + kst * C::TILE_BYTES, C::TILE_BYTES, sbase + C::OFF_K,
                                  sbase + C::OFF_V),
                      st, DBG_SMEM) ||
            !FA_CHECK(tmem_in(d, 128, tmem, C::TM_COLS), st, DBG_TMEM))
          return;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * C::SUB_BYTES + (k & 3) * 32) >> 4;
          if (elect_one()) mma_ss(d, sdesc_join(qa + off, HI), sdesc_join(ka + off, HI), IDESC_S, k > 0);
        }
      };
      auto issue_pv = [&](int t, int vst, uint32_t acc) {  // O_t += P_t V (V from stage vst)
        const uint32_t va = v_lo + vst * TILE16, d = tmem + C::tm_o(t), pa = tmem + C::tm_p(t);
        if (!FA_CHECK(smem_in(sbase + C::OFF_V + vst * C::TILE_BYTES, C::TILE_BYTES, sbase + C::OFF_V,
                              sbase + C::OFF_BAR),
                      st, DBG_SMEM) ||
            !FA_CHECK(tmem_in(d, D, tmem, C::TM_COLS) && tmem_in(pa, 64, tmem, C::TM_COLS), st, DBG_TMEM))
          return;
#pragma unroll
        for (int k = 0; k < 8; ++k)  // 128 keys, 16 per MMA
          if (elect_one()) mma_ts(d, pa + k * 8, sdesc_join(va + k * (2048 >> 4), HI), IDESC_O, (acc | k) != 0);
      };
      auto commit = [&](uint32_t bar) {
        if (elect_one()) mma_commit(bar);
        __syncwarp();
      };
      bool ok = wait_warp_sleep(q_full, 0, st, SITE_F_Q_FULL) && wait_warp_sleep(k_full(0), 0, st, SITE_F_K_FULL);
      const int t_lo = C::SEP_P ? warp - 9 : 0, t_hi = C::SEP_P ? warp - 9 : 1;  // query tiles served
      if (ok) {
        tc_fence_after();
        for (int t = t_lo; t <= t_hi && ok; ++t)
          if (n_t[t] > 0) {
            if (dual && t == 1) {  // lane 1 starts at ring tile 1
              if (!C::SEP_P) continue;  // the single issuer starts it inside the loop
              if (!(ok = wait_warp_sleep(k_full(1 % C::NST), (1 / C::NST) & 1, st, SITE_F_K_FULL))) break;
              issue_s(1, 1 % C::NST);
            } else {
              issue_s(t, 0);
            }
            commit(s_full(t));
          }
      }
      int s = 0, ph = 0;  // ring stage and phase of tile j
      for (int j = 0; ok && j < nmax; ++j) {
        const int s2 = (s + 1 == C::NST) ? 0 : s + 1;
        const int ph2 = (s + 1 == C::NST) ? ph ^ 1 : ph;
        bool used = false;
        if (dual) {
          // ring tile j is lane (j & 1)'s tile j >> 1
          if (!C::SEP_P && j + 1 < nmax) {
            // one issuer for both lanes: the other lane's next S as soon as its K has landed
            // (ring tile j + 1 is another stage than j: no wait on this tile's release)
            if (!(ok = wait_warp_sleep(k_full(s2), ph2, st, SITE_F_K_FULL))) break;
            issue_s((j + 1) & 1, s2);
            commit(s_full((j + 1) & 1));
          }
          for (int t = t_lo; t <= t_hi && ok; ++t) {
            if ((j & 1) != t) continue;
            used = true;
            const int kk = j >> 1;
            if (C::SEP_P && kk + 1 < n_t[t]) {  // this lane's next tile is ring tile j + 2
              const int sn = (j + 2) % C::NST;
              const uint32_t phn = ((j + 2) / C::NST) & 1;
              if (!(ok = wait_warp_sleep(k_full(sn), phn, st, SITE_F_K_FULL))) break;
              if (!(ok = wait_warp_sleep(s_free(t), kk & 1, st, SITE_F_S_FREE))) break;
              tc_fence_after();
              issue_s(t, sn);
              commit(s_full(t));
            }
            if (!(ok = wait_warp_sleep(v_full(s), ph, st, SITE_F_V_FULL))) break;
            if (!(ok = wait_warp_sleep(p_ready(t), kk & 1, st, SITE_F_P_READY))) break;
            tc_fence_after();
            issue_pv(t, s, kk > 0);
            commit(o_done(t));
          }
        } else
        for (int t = t_lo; t <= t_hi && ok; ++t) {
          const int n = n_t[t];
          if (j >= n) continue;
          used = true;
          if (C::SEP_P && j + 1 < n) {
            // S_t(j+1) as soon as the warpgroup has S_t(j) in registers
            if (!(ok = wait_warp_sleep(k_full(s2), ph2, st, SITE_F_K_FULL))) break;
            if (!(ok = wait_warp_sleep(s_free(t), j & 1, st, SITE_F_S_FREE))) break;
            tc_fence_after();
            issue_s(t, s2);
            commit(s_full(t));
          }
          if (!(ok = wait_warp_sleep(v_full(s), ph, st, SITE_F_V_FULL))) break;
          if (!(ok = wait_warp_sleep(p_ready(t), j & 1, st, SITE_F_P_READY))) break;
          tc_fence_after();
          issue_pv(t, s, j > 0);
          commit(o_done(t));
          if (!C::SEP_P && j + 1 < n) {  // P_t(j) lives over S_t(j): S_t(j+1) follows PV_t(j)
            if (!(ok = wait_warp_sleep(k_full(s2), ph2, st, SITE_F_K_FULL))) break;
            issue_s(t, s2);
            commit(s_full(t));
          }
        }
        if (!ok) break;
        if (used) {
          commit(kv_empty(s));  // this warp's readers of K_j, V_j are issued
        } else {
          // tile j is not this warp's: once it has landed (so its stage's previous use
          // is released), add this warp's arrival without waiting for anything else
          if (!(ok = wait_warp_sleep(v_full(s), ph, st, SITE_F_V_FULL))) break;
          if (elect_one()) mbar_arrive(kv_empty(s));
          __syncwarp();
        }
        s = s2;
        ph = ph2;
      }
      // every MMA issued by either warp has completed before TMEM is released
      commit(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // TMEM lane == row within the query tile
    const int qs = q0 + (dual ? 0 : t * 128);
    const int grow = qs + row;
    const int n = n_t[t];
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::tm_s(t);
    const uint32_t tP = tmem + lane_off + C::tm_p(t);
    const uint32_t tO = tmem + lane_off + C::tm_o(t);
    const float sl2 = a.scale_log2;
    float* lse_row = a.lse + obase;
    // split: this lane's partial slot (two per share: lanes of a dual CTA, or the tile's
    // own result and an empty second slot)
    const size_t plane = (size_t)gridDim.x * a.N;
    const size_t prow = (size_t)(2 * blockIdx.z + (dual ? t : 0)) * plane + obase + grow;
    if (SPLIT && !dual && grow < NQ && qs < NQ &&
        FA_CHECK(in_range(prow + plane, fwd_ext(a, VL).part_rows), st, DBG_GLOBAL_STORE))
      a.part_lse[prow + plane] = -INFINITY;
    if ((!ONE || t == 0) && qs < NQ && n == 0) {  // (ONE: lane 1's rows are another CTA's)
      // no valid key for any row of this tile (in this share): O = 0, LSE = -inf
      if (grow < NQ) {
        if (SPLIT) {
          if (FA_CHECK(in_range(prow, fwd_ext(a, VL).part_rows), st, DBG_GLOBAL_STORE))
            a.part_lse[prow] = -INFINITY;  // the combine skips this slot's O
        } else if (FA_CHECK(in_range(obase + grow, fwd_ext(a, VL).o_rows), st, DBG_GLOBAL_STORE)) {
          uint4* orow = reinterpret_cast<uint4*>(a.o + (obase + grow) * D);
          for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
          lse_row[grow] = -INFINITY;
        }
      }
    } else if (n > 0 && FA_CHECK(tmem_in(tmem + C::tm_s(t), 128, tmem, C::TM_COLS) &&
                                     tmem_in(tmem + C::tm_p(t), 64, tmem, C::TM_COLS) &&
                                     tmem_in(tmem + C::tm_o(t), D, tmem, C::TM_COLS),
                                 st, DBG_TMEM)) {
      float m_run = -INFINITY;  // running maximum of s*S*log2(e)
      float l_run = 0.f;        // running normaliser
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        ok = wait_warp_sleep(s_full(t), j & 1, st, SITE_F_S_FULL);
        if (!ok) break;
        tc_fence_after();
        float sv[128];
        {
          uint32_t r[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, r[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(r[c][i]);
        }
        if (C::SEP_P) {  // S_t is in registers: the MMA may overwrite it with S_t(j+1)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free(t));
        }
        const int k0 = (jb + (dual ? 2 * j + t : j)) * 128;
        const bool need_mask = (k0 + 127 >= kv) || (a.causal && k0 + 127 > qs + a.coff);
        if (need_mask) {
          const int lim = a.causal ? min(kv, grow + 1 + a.coff) : kv;  // keys [0, lim) are valid
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (k0 + c >= lim) sv[c] = -INFINITY;
        }
        // row maximum: four independent partial maxima (three-input max), then a short tree
        float pm[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) pm[u] = sv[u];
#pragma unroll
        for (int c = 4; c < 124; c += 8)
#pragma unroll
          for (int u = 0; u < 4; ++u) pm[u] = fmax3(pm[u], sv[c + 2 * u], sv[c + 2 * u + 1]);
        const float mx = fmax3(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]), fmax3(sv[124], sv[125], fmaxf(sv[126], sv[127])));
        const float m_tile = mx * sl2;
        // lazy rescale: move the reference maximum only when it grows by > 2^8
        float f = 1.f;
        bool rescale_warp = false;
        if (j == 0) {
          m_run = m_tile;
        } else {
          const bool grow_m = m_tile > m_run + 8.0f;
          rescale_warp = __any_sync(0xffffffffu, grow_m);
          if (grow_m) {
            f = ex2_approx(m_run - m_tile);
            m_run = m_tile;
          }
        }
        const float base = (m_run == -INFINITY) ? 0.f : m_run;
        // P = exp2(S s log2e - base): the argument of two columns per fma.f32x2,
        // the row sum in two paired partial sums
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nbase2 = f2_pack(-base, -base);
        uint64_t ps2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
        uint32_t pk[4][16];
#pragma unroll
        for (int h = 0; h < 4; ++h) {  // 32 columns -> 16 packed bf16x2 words per store
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(sv[h * 32 + 2 * i], sv[h * 32 + 2 * i + 1]), sl2x2, nbase2), x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            ps2[i & 1] = f2_add(ps2[i & 1], f2_pack(p0, p1));
            pk[h][i] = pack_bf16x2(p0, p1);
          }
          if (C::SEP_P && h == 1) {
            // separate P buffer: half of P is formed before PV_t(j-1) must be done with it
            if (j > 0) {
              if (!(ok = wait_warp_sleep(o_done(t), (j - 1) & 1, st, SITE_F_O_DONE))) break;
              tc_fence_after();
            }
            tmem_st16(tP, pk[0]);
            tmem_st16(tP + 16, pk[1]);
          }
          if (!C::SEP_P || h >= 2) tmem_st16(tP + h * 16, pk[h]);
        }
        if (!ok) break;
        float ps[4];
        f2_unpack(ps2[0], ps[0], ps[1]);
        f2_unpack(ps2[1], ps[2], ps[3]);
        const float lsum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
        l_run = l_run * f + lsum;
        if (rescale_warp) {
          if (!C::SEP_P) {  // PV_{j-1} must have landed in O before it is rescaled
            if (!(ok = wait_warp_sleep(o_done(t), (j - 1) & 1, st, SITE_F_O_DONE))) break;
            tc_fence_after();
          }
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            tmem_ld32(tO + c * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
            tmem_st32(tO + c * 32, r);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready(t));
      }
      if (ok) ok = wait_warp_sleep(o_done(t), (n - 1) & 1, st, SITE_F_O_DONE);
      // every warp of the warpgroup reaches this vote, aborted or not, so the
      // named barrier of the epilogue below is entered by all four or by none
      ok = named_bar_and(1 + t, 128, ok);
      if (ok && SPLIT) {
        tc_fence_after();
        // this share's O / l (fp32) and LSE, one row per thread
        const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
        float4* dst = reinterpret_cast<float4*>(a.part_o + prow * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tO + c * 32, r);
          tmem_wait_ld();
          if (grow < a.N && FA_CHECK(in_range(prow, fwd_ext(a, VL).part_rows), st, DBG_GLOBAL_STORE)) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[c * 8 + q] = make_float4(__uint_as_float(r[4 * q]) * inv, __uint_as_float(r[4 * q + 1]) * inv,
                                           __uint_as_float(r[4 * q + 2]) * inv, __uint_as_float(r[4 * q + 3]) * inv);
          }
        }
        if (grow < a.N && FA_CHECK(in_range(prow, fwd_ext(a, VL).part_rows), st, DBG_GLOBAL_STORE))
          a.part_lse[prow] = (l_run > 0.f) ? (m_run + lg2_approx(l_run)) * 0.6931471805599453f : -INFINITY;
      } else if (ok) {
        tc_fence_after();
        // epilogue: O / l -> bf16 -> swizzled smem (this tile's Q buffer) -> TMA store; a VL
        // tile that runs past its sequence writes its rows directly (the next sequence's
        // rows follow in the same tensor)
        const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
        uint8_t* stage = sm + C::OFF_Q + t * C::TILE_BYTES;
        const bool direct = VL && qs + 128 > NQ;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tO + c * 32, r);
          tmem_wait_ld();
          // columns c*32 .. c*32+31 = 4 chunks of 8 bf16 in column block (c*32)/64
          const int blk = (c * 32) >> 6;
          const int chunk0 = ((c * 32) & 63) >> 3;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(r[q * 8 + 0]) * inv, __uint_as_float(r[q * 8 + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(r[q * 8 + 2]) * inv, __uint_as_float(r[q * 8 + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(r[q * 8 + 4]) * inv, __uint_as_float(r[q * 8 + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(r[q * 8 + 6]) * inv, __uint_as_float(r[q * 8 + 7]) * inv);
            if (direct) {
              if (grow < NQ && FA_CHECK(in_range(obase + grow, fwd_ext(a, VL).o_rows), st, DBG_GLOBAL_STORE))
                *reinterpret_cast<uint4*>(a.o + (obase + grow) * D + c * 32 + q * 8) = v;
            } else if (FA_CHECK(smem_in(smem_u32(stage + blk * C::SUB_BYTES + sw128_offset(row, chunk0 + q)), 16,
                                        sbase + C::OFF_Q, sbase + C::OFF_K),
                                st, DBG_SMEM)) {
              *reinterpret_cast<uint4*>(stage + blk * C::SUB_BYTES + sw128_offset(row, chunk0 + q)) = v;
            }
          }
        }
        if (grow < NQ && FA_CHECK(in_range(obase + grow, fwd_ext(a, VL).o_rows), st, DBG_GLOBAL_STORE))
          lse_row[grow] = (l_run > 0.f) ? (m_run + lg2_approx(l_run)) * 0.6931471805599453f : -INFINITY;
        fence_proxy_async_smem();
        named_bar_sync(1 + t, 128);
        if (wq == 0 && lane == 0 && !direct) {
          for (int c = 0; c < C::NSUB; ++c)
            if (FA_CHECK(tma_coords_ok(c * 64, rbase + qs, zh, D, fwd_ext(a, VL).rows_q, fwd_ext(a, VL).heads, 2, 128,
                                       true) &&
                             smem_in(smem_u32(stage + c * C::SUB_BYTES), C::SUB_BYTES, sbase + C::OFF_Q,
                                     sbase + C::OFF_K),
                         st, DBG_TMA_STORE))
              tma_store_3d(&tm_o, smem_u32(stage + c * C::SUB_BYTES), c * 64, rbase + qs, zh);
          bulk_commit();
          bulk_wait_read0();  // the staging tile must outlive the copy's reads
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// ---------------------------------------------------------------------------------------------
// d = 64 forward, persistent: G CTAs (one per SM) loop over work items = (pair of 128-row query
// tiles, head), longest causal pairs first with heads fastest, in the snake order of the
// backward (CTA c takes item r G + c in even rounds r and r G + G - 1 - c in odd ones). Inside
// an item the pipeline is that of fwd_kernel<64>; across items the K/V ring, the TMEM buffers
// and every barrier phase run on, Q is double-buffered by item (the next item's Q loads while
// this one runs; a set doubles as its item's O staging and is released once the O stores have
// read it), S_t(0) of the next item is issued as soon as S_t is free, and PV_t(0) of the next
// item waits until the epilogue has read O_t out of TMEM.
struct FwdP64 {
  static constexpr int D = 64, NST = 3;
  static constexpr int TILE_BYTES = 128 * 128;         // [128 rows][64] bf16
  static constexpr int OFF_Q = 0;                      // 2 sets x 2 query tiles
  static constexpr int OFF_K = OFF_Q + 4 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NST * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NST * TILE_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
  // TMEM columns as fwd_kernel<64>: S_t 128 t, P_t 256 + 64 t, O_t 384 + 64 t
  __device__ static constexpr uint32_t tm_s(int t) { return 128u * t; }
  __device__ static constexpr uint32_t tm_p(int t) { return 256u + 64u * t; }
  __device__ static constexpr uint32_t tm_o(int t) { return 384u + 64u * t; }
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int THREADS = 352;  // 0-7 softmax, 8 TMA, 9-10 MMA (one per query tile)
  __host__ __device__ static constexpr int off_q(int set, int t) { return OFF_Q + (2 * set + t) * TILE_BYTES; }
};
static_assert(8 * (10 + 3 * FwdP64::NST + 1) + 8 <= 256, "persistent forward: barrier area");

struct ItemF64 {
  int bh, kv, q0, n[2], nmax;
};
// Where item bh's rows live. Plain [BH, N, d]: rows start at TMA row 0 of head bh, N query
// rows, O / LSE row index base bh N. Packed sequences (VL, [H, T, d]): item bh is sequence
// b = bh / H of head h, its rows start at TMA row cu[b] of head h, it has cu[b + 1] - cu[b]
// rows, and its O / LSE rows start at h T + cu[b].
struct RowsF64 {
  int rb, nq, zh;
  size_t obase;
};
template <bool VL>
__device__ __forceinline__ RowsF64 rows_f64(int bh, const FwdArgs& a) {
  RowsF64 r;
  if (VL) {
    const int b = bh / a.H, h = bh - b * a.H;
    if (FA_CHECK(in_range(b + 1, a.dbg_B + 1LL), a.status, DBG_META)) {
      r.rb = a.cu_seqlens[b];
      r.nq = a.cu_seqlens[b + 1] - r.rb;
    } else {
      r.rb = 0;
      r.nq = 0;
    }
    r.zh = h;
    r.obase = (size_t)h * a.T + r.rb;
  } else {
    r.rb = 0;
    r.nq = a.N;
    r.zh = bh;
    r.obase = (size_t)bh * a.N;
  }
  return r;
}
template <bool VL>
__device__ __forceinline__ ItemF64 item_f64(int t, const FwdArgs& a, int BH) {
  ItemF64 it;
  const int p = t / BH;
  it.bh = t - p * BH;
  it.q0 = (a.n_pairs - 1 - p) * 256;
  int nq = a.N;
  if (VL) {  // a pair past its sequence has no work (and writes nothing: the rows are another's)
    nq = rows_f64<VL>(it.bh, a).nq;
    it.kv = nq;
  } else {
    it.kv = a.Nk;
    if (a.kv_len && FA_CHECK(in_range(it.bh / a.H, a.dbg_B), a.status, DBG_META))
      it.kv = min(max(a.kv_len[it.bh / a.H], 0), a.Nk);
  }
  const int nkt = (it.kv + 127) >> 7;
#pragma unroll
  for (int u = 0; u < 2; ++u) it.n[u] = key_tiles(it.q0 + u * 128, nq, nkt, a.causal, VL ? 0 : a.coff);
  it.nmax = max(it.n[0], it.n[1]);
  return it;
}
__device__ __forceinline__ int sched_f64(int r, int c, int G, int T) {
  const int t = r * G + ((r & 1) ? (G - 1 - c) : c);
  return t < T ? t : -1;
}

// The rows of an item with no valid key (kv_len = 0): O = 0 and LSE = -inf. Kept out of
// line: inlined into the producer's loop it made the register allocator spill in the
// softmax warpgroups.
__device__ __noinline__ void zero_rows_f64(uint16_t* o, float* lse, int N, int bh, int q0, int lane) {
  constexpr int D = FwdP64::D;
  for (int idx = lane; idx < 256 * (D / 8); idx += 32) {
    const int grow = q0 + idx / (D / 8);
    if (grow < N) {
      const size_t off = ((size_t)bh * N + grow) * D + (idx % (D / 8)) * 8;
      *reinterpret_cast<uint4*>(o + off) = make_uint4(0, 0, 0, 0);
      if (idx % (D / 8) == 0) lse[(size_t)bh * N + grow] = -INFINITY;
    }
  }
}

template <bool VL>
__global__ void __launch_bounds__(352, 1)
    fwd_kernel_p64(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, FwdArgs a,
                   int BH) {
  griddep_wait();  // before any access to global memory
  griddep_launch_dependents();
  using C = FwdP64;
  constexpr int D = C::D, NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const uint32_t sbase = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  const uint32_t b0 = smem_u32(bars);
  auto BAR = [&](int i) { return b0 + 8u * i; };
  auto q_full = [&](int set) { return BAR(set); };
  auto q_empty = [&](int set) { return BAR(2 + set); };  // one arrival per query tile
  auto k_full = [&](int s) { return BAR(4 + s); };
  auto v_full = [&](int s) { return BAR(4 + NST + s); };
  auto kv_empty = [&](int s) { return BAR(4 + 2 * NST + s); };
  constexpr int nb = 4 + 3 * NST;
  auto s_full = [&](int t) { return BAR(nb + t); };
  auto p_ready = [&](int t) { return BAR(nb + 2 + t); };
  auto o_done = [&](int t) { return BAR(nb + 4 + t); };
  auto s_free = [&](int t) { return BAR(nb + 6 + t); };
  auto o_free = [&](int t) { return BAR(nb + 8 + t); };  // O_t read out by the epilogue
  const uint32_t drain = BAR(nb + 10);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 8 * (nb + 11));
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  DevStatus st{a.status, abort_flag};

  const int T = BH * a.n_pairs;
  const int G = gridDim.x, cta = blockIdx.x;
  // the next item with work at or after round r (its round, or -1)
  auto next_item = [&](int r, ItemF64& out) -> int {
    for (;; ++r) {
      const int t = sched_f64(r, cta, G, T);
      if (t < 0) return -1;
      out = item_f64<VL>(t, a, BH);
      if (out.nmax > 0) return r;
    }
  };

  // Producer warp: barriers, then the first item's Q and first K/V stages before the setup.
  auto load_kv = [&](int g, int j, int bh) {  // whole warp; ring index g, key tile j
    if (kWithhold && g == 1) return;  // test build: this copy never arrives
    const int s = g % NST;
    const uint32_t kf = k_full(s), vf = v_full(s);
    const RowsF64 rw = rows_f64<VL>(bh, a);
    if (elect_one()) mbar_arrive_expect_tx(kf, C::TILE_BYTES);
    if (FA_CHECK(tma_coords_ok(0, rw.rb + j * 128, rw.zh, D, fwd_ext(a, VL).rows_k, fwd_ext(a, VL).heads, 2, 128,
                               false) &&
                     smem_in(sbase + C::OFF_K + s * C::TILE_BYTES, C::TILE_BYTES, sbase + C::OFF_K, sbase + C::OFF_V),
                 st, DBG_TMA_LOAD) &&
        elect_one())
      tma_load_3d(sbase + C::OFF_K + s * C::TILE_BYTES, &tm_k, 0, rw.rb + j * 128, rw.zh, kf);
    if (elect_one()) mbar_arrive_expect_tx(vf, C::TILE_BYTES);
    if (FA_CHECK(tma_coords_ok(0, rw.rb + j * 128, rw.zh, D, fwd_ext(a, VL).rows_k, fwd_ext(a, VL).heads, 2, 128,
                               false) &&
                     smem_in(sbase + C::OFF_V + s * C::TILE_BYTES, C::TILE_BYTES, sbase + C::OFF_V,
                             sbase + C::OFF_BAR),
                 st, DBG_TMA_LOAD) &&
        elect_one())
      tma_load_3d(sbase + C::OFF_V + s * C::TILE_BYTES, &tm_v, 0, rw.rb + j * 128, rw.zh, vf);
    __syncwarp();
  };
  auto load_q = [&](int set, const ItemF64& it) {  // whole warp
    const int nq = (it.n[1] > 0) ? 2 : 1;
    const RowsF64 rw = rows_f64<VL>(it.bh, a);
    if (elect_one()) mbar_arrive_expect_tx(q_full(set), nq * C::TILE_BYTES);
    for (int u = 0; u < nq; ++u)
      if (FA_CHECK(tma_coords_ok(0, rw.rb + it.q0 + u * 128, rw.zh, D, fwd_ext(a, VL).rows_q, fwd_ext(a, VL).heads, 2,
                                 128, false) &&
                       smem_in(sbase + C::off_q(set, u), C::TILE_BYTES, sbase + C::OFF_Q, sbase + C::OFF_K),
                   st, DBG_TMA_LOAD) &&
          elect_one())
        tma_load_3d(sbase + C::off_q(set, u), &tm_q, 0, rw.rb + it.q0 + u * 128, rw.zh, q_full(set));
    __syncwarp();
  };
  int n_pre = 0;  // K/V stages of the first item issued before the setup (producer warp)
  if (warp == 8) {
    if (lane == 0) {
      for (int u = 0; u < 2; ++u) {
        mbar_init(q_full(u), 1);
        mbar_init(q_empty(u), 2);
      }
      for (int s = 0; s < NST; ++s) {
        mbar_init(k_full(s), 1);
        mbar_init(v_full(s), 1);
        mbar_init(kv_empty(s), 2);  // one arrival per MMA-issuing warp
      }
      for (int t = 0; t < 2; ++t) {
        mbar_init(s_full(t), 1);
        mbar_init(p_ready(t), 4);
        mbar_init(o_done(t), 1);
        mbar_init(s_free(t), 4);
        mbar_init(o_free(t), 4);
      }
      mbar_init(drain, 2);
      *abort_flag = 0;
      fence_mbar_init();
    }
    __syncwarp();
    ItemF64 it;
    if (next_item(0, it) >= 0) {
      if (elect_one()) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
      }
      load_q(0, it);
      n_pre = min(NST, it.nmax);
      for (int j = 0; j < n_pre; ++j) load_kv(j, j, it.bh);
    }
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    bool ok = true;
    int iu = 0, g0 = 0, issued = 0, q_loads = 1;  // the first item's Q went out before the setup
    for (int r = 0; ok; ++r) {
      const int tt = sched_f64(r, cta, G, T);
      if (tt < 0) break;
      const ItemF64 it = item_f64<VL>(tt, a, BH);
      if (VL && lane == 0 && it.q0 == 0 && rows_f64<VL>(it.bh, a).nq > a.max_seqlen)
        record_check(a.status, SITE_F_SEQLEN);  // the grid (sized by max_seqlen) misses rows of it
      if (it.nmax == 0) {
        if (!VL && FA_CHECK(span_in((long long)it.bh * a.N + it.q0, min(256, a.N - it.q0), fwd_ext(a, VL).o_rows), st,
                            DBG_GLOBAL_STORE))
          zero_rows_f64(a.o, a.lse, a.N, it.bh, it.q0, lane);
        continue;
      }
      const int set = iu & 1;
      if (iu > 0) {
        if (!(ok = wait_warp_sleep(q_empty(set), ((iu >> 1) & 1) ^ 1, st, SITE_F_Q_FULL))) break;
        load_q(set, it);
        ++q_loads;
      }
      for (int j = (iu == 0 ? n_pre : 0); j < it.nmax; ++j) {
        const int g = g0 + j;
        if (!(ok = wait_warp_sleep(kv_empty(g % NST), ((g / NST) & 1) ^ 1, st, SITE_F_KV_EMPTY))) break;
        load_kv(g, j, it.bh);
        issued = g + 1;
      }
      g0 += it.nmax;
      ++iu;
    }
    if (*(volatile int*)abort_flag) {
      // let copies already in flight land before the CTA's smem is released
      const uint64_t t0 = globaltimer_ns();
      for (int g = max(0, issued - NST); g < issued; ++g)
        while (!(mbar_try_wait(k_full(g % NST), (g / NST) & 1) && mbar_try_wait(v_full(g % NST), (g / NST) & 1)) &&
               globaltimer_ns() - t0 < 100000000ull) {
        }
      for (int u = max(0, q_loads - 2); u < q_loads; ++u)
        while (!mbar_try_wait(q_full(u & 1), (u >> 1) & 1) && globaltimer_ns() - t0 < 100000000ull) {
        }
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuer of query tile t
    // (whole warp; one elected lane issues)
    const int t = warp - 9;
    constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, 0, 0);  // Q, K both K-major
    constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, 0, 1);    // P from TMEM, V MN-major
    constexpr uint32_t HI = sdesc_hi(1024);
    constexpr uint32_t TILE16 = C::TILE_BYTES >> 4;
    const uint32_t k_lo = sdesc_lo(sbase + C::OFF_K, 16);
    const uint32_t v_lo = sdesc_lo(sbase + C::OFF_V, C::TILE_BYTES);
    auto issue_s = [&](int set, int kst) {  // S_t = Q_t K^T (Q from set, K from stage kst)
      const uint32_t qa = sdesc_lo(sbase + C::off_q(set, t), 16), ka = k_lo + kst * TILE16, d = tmem + C::tm_s(t);
      if (!FA_CHECK(smem_in(sbase + C::off_q(set, t), C::TILE_BYTES, sbase + C::OFF_Q, sbase + C::OFF_K) &&
                        smem_in(sbase + C::OFF_K + kst * C::TILE_BYTES, C::TILE_BYTES, sbase + C::OFF_K,
                                sbase + C::OFF_V),
                    st, DBG_SMEM) ||
          !FA_CHECK(tmem_in(d, 128, tmem, C::TM_COLS), st, DBG_TMEM))
        return;
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        if (elect_one()) mma_ss(d, sdesc_join(qa + 2 * k, HI), sdesc_join(ka + 2 * k, HI), IDESC_S, k > 0);
    };
    auto issue_pv = [&](int vst, uint32_t acc) {  // O_t += P_t V (V from stage vst)
      const uint32_t va = v_lo + vst * TILE16, d = tmem + C::tm_o(t), pa = tmem + C::tm_p(t);
      if (!FA_CHECK(smem_in(sbase + C::OFF_V + vst * C::TILE_BYTES, C::TILE_BYTES, sbase + C::OFF_V,
                            sbase + C::OFF_BAR),
                    st, DBG_SMEM) ||
          !FA_CHECK(tmem_in(d, D, tmem, C::TM_COLS) && tmem_in(pa, 64, tmem, C::TM_COLS), st, DBG_TMEM))
        return;
#pragma unroll
      for (int k = 0; k < 8; ++k)  // 128 keys, 16 per MMA
        if (elect_one()) mma_ts(d, pa + k * 8, sdesc_join(va + k * (2048 >> 4), HI), IDESC_O, (acc | k) != 0);
    };
    auto commit = [&](uint32_t bar) {
      if (elect_one()) mma_commit(bar);
      __syncwarp();
    };
    bool ok = true;
    int iu = 0, g0 = 0, gj = 0, ep = 0;  // items, ring index, S_t count, epilogues of tile t
    bool s0_issued = false;              // S_t(0) of the current item already issued ahead
    ItemF64 it, nx;
    for (int r = next_item(0, it); ok && r >= 0;) {
      const int set = iu & 1;
      const int n = (t == 0 ? it.n[0] : it.n[1]);
      const int r2 = next_item(r + 1, nx);
      if (n > 0 && !s0_issued) {  // S_t(0) of this item (S_t is free once its last one was read)
        if (!(ok = wait_warp_sleep(q_full(set), (iu >> 1) & 1, st, SITE_F_Q_FULL))) break;
        if (!(ok = wait_warp_sleep(k_full(g0 % NST), (g0 / NST) & 1, st, SITE_F_K_FULL))) break;
        if (gj > 0 && !(ok = wait_warp_sleep(s_free(t), (gj - 1) & 1, st, SITE_F_S_FREE))) break;
        tc_fence_after();
        issue_s(set, g0 % NST);
        commit(s_full(t));
      }
      s0_issued = false;
      for (int j = 0; ok && j < it.nmax; ++j) {
        const int g = g0 + j, s = g % NST;
        const uint32_t ph = (g / NST) & 1;
        if (j < n) {
          if (j + 1 < n) {  // S_t(j+1) as soon as the warpgroup has S_t(j) in registers
            if (!(ok = wait_warp_sleep(k_full((g + 1) % NST), ((g + 1) / NST) & 1, st, SITE_F_K_FULL))) break;
            if (!(ok = wait_warp_sleep(s_free(t), (gj + j) & 1, st, SITE_F_S_FREE))) break;
            tc_fence_after();
            issue_s(set, (g + 1) % NST);
            commit(s_full(t));
          } else if (r2 >= 0 && (t == 0 ? nx.n[0] : nx.n[1]) > 0) {
            // ... and S_t(0) of the next item, if its Q and first K tile have landed already.
            // Waiting for them here would hold up PV_t(j), and with it this item's epilogue;
            // otherwise S_t(0) is issued at the next item's start.
            const int g2 = g0 + it.nmax;
            bool rdy = false;
            if (lane == 0)
              rdy = mbar_test_wait(q_full(set ^ 1), ((iu + 1) >> 1) & 1) &&
                    mbar_test_wait(k_full(g2 % NST), (g2 / NST) & 1);
            if (__shfl_sync(0xffffffffu, rdy, 0)) {
              if (!(ok = wait_warp_sleep(s_free(t), (gj + j) & 1, st, SITE_F_S_FREE))) break;
              tc_fence_after();
              issue_s(set ^ 1, g2 % NST);
              commit(s_full(t));
              s0_issued = true;
            }
          }
          if (!(ok = wait_warp_sleep(v_full(s), ph, st, SITE_F_V_FULL))) break;
          if (!(ok = wait_warp_sleep(p_ready(t), (gj + j) & 1, st, SITE_F_P_READY))) break;
          if (j == 0 && ep > 0) {  // the epilogue has read O_t of the previous item
            if (!(ok = wait_warp_sleep(o_free(t), (ep - 1) & 1, st, SITE_F_O_DONE))) break;
          }
          tc_fence_after();
          issue_pv(s, j > 0);
          commit(o_done(t));
          commit(kv_empty(s));  // this warp's readers of K_j, V_j are issued
        } else {
          // tile j is not this warp's: once it has landed (so its stage's previous use is
          // released), add this warp's arrival without waiting for anything else
          if (!(ok = wait_warp_sleep(v_full(s), ph, st, SITE_F_V_FULL))) break;
          if (elect_one()) mbar_arrive(kv_empty(s));
          __syncwarp();
        }
      }
      if (!ok) break;
      gj += n;
      if (n > 0) ++ep;
      g0 += it.nmax;
      ++iu;
      it = nx;
      r = r2;
    }
    commit(drain);  // completes after every MMA issued above
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax warpgroup of tile t
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // TMEM lane == row within the query tile
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::tm_s(t);
    const uint32_t tP = tmem + lane_off + C::tm_p(t);
    const uint32_t tO = tmem + lane_off + C::tm_o(t);
    const float sl2 = a.scale_log2;
    bool ok = FA_CHECK(tmem_in(tmem + C::tm_s(t), 128, tmem, C::TM_COLS) &&
                           tmem_in(tmem + C::tm_p(t), 64, tmem, C::TM_COLS) &&
                           tmem_in(tmem + C::tm_o(t), D, tmem, C::TM_COLS),
                       st, DBG_TMEM);
    int iu = 0, gj = 0;
    // Q_t set whose O store (issued by warp 0 of this warpgroup) may still be reading it: the
    // wait for those reads, and the set's release to the producer, come after the warpgroup's
    // next S wait, off the path from one item to the next
    int pend = -1;
    auto release_pending = [&]() {
      if (pend >= 0 && wq == 0 && lane == 0) {
        bulk_wait_read0();
        mbar_arrive(q_empty(pend));
      }
      __syncwarp();
      pend = -1;
    };
    ItemF64 it;
    for (int r = next_item(0, it); ok && r >= 0; r = next_item(r + 1, it)) {
      // only n, qs and kv live through the key loop; the rest of the item is recomputed for
      // the epilogue (fewer live registers in the softmax)
      const int n = (t == 0 ? it.n[0] : it.n[1]);
      const int qs = it.q0 + t * 128;
      const int kvv = it.kv;
      const int grow = qs + row;
      bool stored = false;
      if (!VL && qs < a.N && n == 0) {
        // no valid key for any row of this tile: O = 0, LSE = -inf (packed: no such tile, the
        // rows past a sequence belong to the next one)
        if (grow < a.N &&
            FA_CHECK(in_range((long long)it.bh * a.N + grow, fwd_ext(a, VL).o_rows), st, DBG_GLOBAL_STORE)) {
          uint4* orow = reinterpret_cast<uint4*>(a.o + ((size_t)it.bh * a.N + grow) * D);
          for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
          a.lse[(size_t)it.bh * a.N + grow] = -INFINITY;
        }
      } else if (n > 0) {
        float m_run = -INFINITY;  // running maximum of s*S*log2(e)
        float l_run = 0.f;        // running normaliser
        for (int j = 0; j < n; ++j) {
          const uint32_t par = (gj + j) & 1;
          ok = wait_warp_sleep(s_full(t), par, st, SITE_F_S_FULL);
          if (!ok) break;
          if (pend >= 0) release_pending();
          tc_fence_after();
          float sv[128];
          {
            uint32_t rr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, rr[c]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(rr[c][i]);
          }
          // S_t is in registers: the MMA may overwrite it with the next S_t
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free(t));
          const int k0 = j * 128;
          const bool need_mask = (k0 + 127 >= kvv) || (a.causal && k0 + 127 > qs + a.coff);
          if (need_mask) {
            const int lim = a.causal ? min(kvv, grow + 1 + a.coff) : kvv;  // keys [0, lim) are valid
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (k0 + c >= lim) sv[c] = -INFINITY;
          }
          // row maximum: four independent partial maxima (three-input max), then a short tree
          float pm[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) pm[u] = sv[u];
#pragma unroll
          for (int c = 4; c < 124; c += 8)
#pragma unroll
            for (int u = 0; u < 4; ++u) pm[u] = fmax3(pm[u], sv[c + 2 * u], sv[c + 2 * u + 1]);
          const float mx =
              fmax3(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]), fmax3(sv[124], sv[125], fmaxf(sv[126], sv[127])));
          const float m_tile = mx * sl2;
          // lazy rescale: move the reference maximum only when it grows by > 2^8
          float f = 1.f;
          bool rescale_warp = false;
          if (j == 0) {
            m_run = m_tile;
          } else {
            const bool grow_m = m_tile > m_run + 8.0f;
            rescale_warp = __any_sync(0xffffffffu, grow_m);
            if (grow_m) {
              f = ex2_approx(m_run - m_tile);
              m_run = m_tile;
            }
          }
          const float base = (m_run == -INFINITY) ? 0.f : m_run;
          // P = exp2(S s log2e - base): the argument of two columns per fma.f32x2,
          // the row sum in two paired partial sums
          const uint64_t sl2x2 = f2_pack(sl2, sl2), nbase2 = f2_pack(-base, -base);
          uint64_t ps2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
          uint32_t pk[4][16];
#pragma unroll
          for (int h = 0; h < 4; ++h) {  // 32 columns -> 16 packed bf16x2 words per store
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(sv[h * 32 + 2 * i], sv[h * 32 + 2 * i + 1]), sl2x2, nbase2), x0, x1);
              const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              ps2[i & 1] = f2_add(ps2[i & 1], f2_pack(p0, p1));
              pk[h][i] = pack_bf16x2(p0, p1);
            }
            if (h == 1) {
              // half of P is formed before PV_t(j-1) must be done with P_t
              if (j > 0) {
                if (!(ok = wait_warp_sleep(o_done(t), par ^ 1, st, SITE_F_O_DONE))) break;
                tc_fence_after();
              }
              tmem_st16(tP, pk[0]);
              tmem_st16(tP + 16, pk[1]);
            }
            if (h >= 2) tmem_st16(tP + h * 16, pk[h]);
          }
          if (!ok) break;
          float ps[4];
          f2_unpack(ps2[0], ps[0], ps[1]);
          f2_unpack(ps2[1], ps[2], ps[3]);
          const float lsum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
          l_run = l_run * f + lsum;
          if (rescale_warp) {
            uint32_t rr[32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              tmem_ld32(tO + c * 32, rr);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * f);
              tmem_st32(tO + c * 32, rr);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_ready(t));
        }
        if (ok) ok = wait_warp_sleep(o_done(t), (gj + n - 1) & 1, st, SITE_F_O_DONE);
        // every warp of the warpgroup reaches this vote, aborted or not, so the
        // named barrier of the epilogue below is entered by all four or by none
        ok = named_bar_and(1 + t, 128, ok);
        if (!ok) break;
        tc_fence_after();
        const RowsF64 rw = rows_f64<VL>(item_f64<VL>(sched_f64(r, cta, G, T), a, BH).bh, a);
        const int set = iu & 1;
        // a packed sequence's partial last tile is written row by row: a TMA box would run into
        // the next sequence's rows
        const bool direct = VL && qs + 128 > rw.nq;
        // epilogue: O_t out of TMEM (then released to the next item's PV), O / l -> bf16 ->
        // swizzled smem (this item's Q_t buffer, which no MMA reads any more) -> TMA store
        uint32_t ov[2][32];
        tmem_ld32(tO, ov[0]);
        tmem_ld32(tO + 32, ov[1]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free(t));
        const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
        uint8_t* stage = sm + C::off_q(set, t);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t* x = &ov[q >> 2][(q & 3) * 8];
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(x[0]) * inv, __uint_as_float(x[1]) * inv);
          v.y = pack_bf16x2(__uint_as_float(x[2]) * inv, __uint_as_float(x[3]) * inv);
          v.z = pack_bf16x2(__uint_as_float(x[4]) * inv, __uint_as_float(x[5]) * inv);
          v.w = pack_bf16x2(__uint_as_float(x[6]) * inv, __uint_as_float(x[7]) * inv);
          if (direct) {
            if (grow < rw.nq && FA_CHECK(in_range(rw.obase + grow, fwd_ext(a, VL).o_rows), st, DBG_GLOBAL_STORE))
              *reinterpret_cast<uint4*>(a.o + (rw.obase + grow) * D + q * 8) = v;
          } else if (FA_CHECK(smem_in(smem_u32(stage + sw128_offset(row, q)), 16, sbase + C::OFF_Q, sbase + C::OFF_K),
                              st, DBG_SMEM)) {
            *reinterpret_cast<uint4*>(stage + sw128_offset(row, q)) = v;
          }
        }
        if (grow < rw.nq && FA_CHECK(in_range(rw.obase + grow, fwd_ext(a, VL).o_rows), st, DBG_GLOBAL_STORE))
          a.lse[rw.obase + grow] = (l_run > 0.f) ? (m_run + lg2_approx(l_run)) * 0.6931471805599453f : -INFINITY;
        fence_proxy_async_smem();
        named_bar_sync(1 + t, 128);
        if (!direct) {
          if (wq == 0 && lane == 0) {
            if (FA_CHECK(tma_coords_ok(0, rw.rb + qs, rw.zh, D, fwd_ext(a, VL).rows_q, fwd_ext(a, VL).heads, 2, 128,
                                       true) &&
                             smem_in(smem_u32(stage), C::TILE_BYTES, sbase + C::OFF_Q, sbase + C::OFF_K),
                         st, DBG_TMA_STORE))
              tma_store_3d(&tm_o, smem_u32(stage), 0, rw.rb + qs, rw.zh);
            bulk_commit();
          }
          pend = set;  // the Q_t buffer is free again once the store has read it
        } else if (wq == 0 && lane == 0) {
          mbar_arrive(q_empty(set));
        }
        stored = true;
      }
      if (!stored) {  // nothing staged in Q_t; a pending set is released first (the producer may need it)
        release_pending();
        if (wq == 0 && lane == 0) mbar_arrive(q_empty(iu & 1));
      }
      gj += n;
      ++iu;
    }
    release_pending();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// Joins the partial results of each query row (2 n_split slots: two per share). With L_z the
// slots' LSEs and M their maximum: LSE = M + ln sum_z e^(L_z - M), O = sum_z e^(L_z - LSE) O_z,
// each O_z already divided by its own normaliser; slots with no key (L_z = -inf) drop out. Grid (row blocks,
// heads), one group of D/8 lanes per row, 8 outputs per lane.
template <int D>
__global__ void __launch_bounds__(256) fwd_combine_kernel(FwdArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int LPR = D / 8;
  constexpr int RPB = 256 / LPR;
  constexpr int G = 16;  // slots whose loads are issued together
  const int part = threadIdx.x % LPR;
  const int n = blockIdx.x * RPB + threadIdx.x / LPR;
  const int bh = blockIdx.y;
  if (n >= a.N) return;
  const size_t row = (size_t)bh * a.N + n, plane = (size_t)gridDim.y * a.N;
  const int nz = 2 * a.n_split;
  float mx = -INFINITY;
  for (int z0 = 0; z0 < nz; z0 += G) {
    float l[G];
#pragma unroll
    for (int g = 0; g < G; ++g)
      l[g] = (z0 + g < nz && FA_CHECK(in_range((z0 + g) * plane + row, fwd_ext(a, false).part_rows), a.status,
                                      DBG_GLOBAL_LOAD))
                 ? a.part_lse[(z0 + g) * plane + row]
                 : -INFINITY;
#pragma unroll
    for (int g = 0; g < G; ++g) mx = fmaxf(mx, l[g]);
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int z0 = 0; z0 < nz; z0 += G) {
      float w[G];
      float4 x0[G], x1[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        // a slot out of range reads as one without keys (its O is then not read either)
        const float lz = (z0 + g < nz && FA_CHECK(in_range((z0 + g) * plane + row, fwd_ext(a, false).part_rows),
                                                  a.status, DBG_GLOBAL_LOAD))
                             ? a.part_lse[(z0 + g) * plane + row]
                             : -INFINITY;
        w[g] = (lz == -INFINITY) ? 0.f : ex2_approx((lz - mx) * 1.4426950408889634f);
        const float4* src = reinterpret_cast<const float4*>(a.part_o + ((z0 + g) * plane + row) * D + part * 8);
        // a slot without keys holds no O: read nothing there
        x0[g] = (w[g] > 0.f) ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f);
        x1[g] = (w[g] > 0.f) ? src[1] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        wsum += w[g];
        acc[0] = fmaf(w[g], x0[g].x, acc[0]), acc[1] = fmaf(w[g], x0[g].y, acc[1]);
        acc[2] = fmaf(w[g], x0[g].z, acc[2]), acc[3] = fmaf(w[g], x0[g].w, acc[3]);
        acc[4] = fmaf(w[g], x1[g].x, acc[4]), acc[5] = fmaf(w[g], x1[g].y, acc[5]);
        acc[6] = fmaf(w[g], x1[g].z, acc[6]), acc[7] = fmaf(w[g], x1[g].w, acc[7]);
      }
    }
  }
  const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
  uint4 out;
  out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
  out.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
  out.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
  if (!FA_CHECK(in_range(row, fwd_ext(a, false).o_rows), a.status, DBG_GLOBAL_STORE)) return;
  *reinterpret_cast<uint4*>(a.o + row * D + part * 8) = out;
  if (part == 0 && a.lse) a.lse[row] = (wsum > 0.f) ? mx + lg2_approx(wsum) * 0.6931471805599453f : -INFINITY;
}

// Decode: few query rows (N_q <= 8) over many keys, the inference shape the pages call memory
// bound. Such a problem has no dense contraction worth the tensor cores (one query row would
// fill an M = 128 MMA with padding), so it streams K and V from HBM at copy speed and reduces
// on the CUDA cores.
//
// Work decomposition: the 128-key tiles of all heads, head after head, form one sequence of T
// tiles, of which each CTA takes a contiguous run. With hpc > 0, CTA c takes the hpc whole
// heads [hpc c, hpc (c + 1)). With hpc = 0 (stream-K), CTA c of G takes tiles
// [c T / G, (c + 1) T / G), so every SM gets the same number of tiles whatever the head count.
// The tiles of one head inside a CTA's run form a segment. A segment that covers its whole head
// writes the head's O (bf16) and LSE directly; otherwise it is a partial result (O / l in fp32
// and its LSE) in partial slot 2c (the CTA's first segment) or 2c + 1 (its last), and
// decode_combine_kernel joins the segments of each such head. Heads with no valid key are
// written O = 0, LSE = -inf here.
//
// Within a CTA, warp 8 streams the segments' 128-key K and V tiles by TMA (128-byte swizzle)
// through an NS-stage ring, running ahead across segment boundaries. Each of warps 0-7 owns
// 16 keys of every tile and keeps its own running maximum, normaliser and O, so a tile needs
// no block-wide synchronisation: lane l scores key l % 16 over half the head dimensions (the
// halves joined by one shuffle), the warp's maximum and sum go through shuffles, and for P V
// lane l owns D / 32 dimensions of the warp's 16 keys. The running maximum rescales O and the
// normaliser between tiles, as between key blocks of the tiled forward. At a segment's end
// the eight warps' states are joined with the same rescaling through shared memory. 288
// threads; NQ >= N_q rows (1, 2, 4 or 8).
constexpr int kDecodeMaxRows = 8;
constexpr int kDecodeMaxCtas = 256;  // CTAs of the decode kernel at most (the join's slot list)
template <int D, int NQ>
struct DecCfg {
  static constexpr int NSUB = D / 64;
  static constexpr int TILE = NSUB * 128 * 128;   // one 128-key tile of K (or V), bf16
  // static shared memory of the kernel: the queries, the warps' states (m, l, O)
  static constexpr int STATIC_BYTES = NQ * (D * 4 + 8 * (2 + D) * 4);
  // ring stages (K and V each): as many as fit beside the static arrays, at most 5
  static constexpr int NS_FIT = (232448 - STATIC_BYTES - 128 - 1024) / (2 * TILE);
  static constexpr int NS = NS_FIT < 5 ? NS_FIT : 5;
  static constexpr int OFF_K = 0, OFF_V = NS * TILE, OFF_BAR = 2 * NS * TILE;
  static constexpr int SMEM_BYTES = OFF_BAR + 128 + 1024;
  static_assert(NS >= 2, "decode: at least two ring stages");
};
enum { SITE_D_FULL = 11, SITE_D_EMPTY, SITE_D_SYNC };

// 128-key tiles of each head of batch b: its valid keys, rounded up.
__device__ __forceinline__ int dec_tiles(const FwdArgs& a, int b) {
  int kv = a.Nk;
  if (a.kv_len && FA_CHECK(in_range(b, a.dbg_B), a.status, DBG_META)) kv = min(max(a.kv_len[b], 0), a.Nk);
  return (kv + 127) >> 7;
}

// Position in the tile sequence of all heads: head h of batch b has tb tiles, its tile 0 is
// global tile gbase. b == B: past the last head.
struct DecCursor {
  int b, h, tb;
  long long gbase;
};

// The head that holds global tile g (g < T).
__device__ DecCursor dec_seek(const FwdArgs& a, int B, long long g) {
  DecCursor c{0, 0, 0, 0};
  for (; c.b < B; ++c.b) {
    c.tb = dec_tiles(a, c.b);
    const long long span = (long long)a.H * c.tb;
    if (g < c.gbase + span) {
      c.h = (int)((g - c.gbase) / c.tb);
      c.gbase += (long long)c.h * c.tb;
      return c;
    }
    c.gbase += span;
  }
  c.tb = 0;
  return c;
}

// The next head that has tiles.
__device__ void dec_next_head(const FwdArgs& a, int B, DecCursor& c) {
  c.gbase += c.tb;
  if (++c.h < a.H) return;
  c.h = 0;
  do {
    ++c.b;
    c.tb = (c.b < B) ? dec_tiles(a, c.b) : 0;
  } while (c.b < B && c.tb == 0);
}

// T, the tiles of all heads.
__device__ long long dec_total(const FwdArgs& a, int B) {
  if (!a.kv_len) return (long long)B * a.H * ((a.Nk + 127) >> 7);
  long long t = 0;
  for (int b = 0; b < B; ++b) t += dec_tiles(a, b);
  return t * a.H;
}

// Global index of the first tile of head bh (bh = B H: T).
__device__ long long dec_head_base(const FwdArgs& a, int B, int bh) {
  const int b = bh / a.H, h = bh - b * a.H;
  if (!a.kv_len) return (long long)bh * ((a.Nk + 127) >> 7);
  long long t = 0;
  for (int bb = 0; bb < b; ++bb) t += dec_tiles(a, bb);
  return t * a.H + (b < B ? (long long)h * dec_tiles(a, b) : 0);
}

template <int D, int NQ>
__global__ void __launch_bounds__(288, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const uint16_t* __restrict__ q, FwdArgs a, int B, int hpc) {
  griddep_wait();
  griddep_launch_dependents();
  using C = DecCfg<D, NQ>;
  constexpr int NS = C::NS, DPL = D / 32, HD = D / 2;  // dims a lane takes in P V; half a row
  // key-major lanes (each lane its own key's O half-row) while NQ half-rows of O fit in registers
  constexpr bool KM = NQ * D <= 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const uint32_t sbase = smem_u32(sm);
  __shared__ float4 qs[NQ][D / 4];        // the segment's queries x s log2(e)
  __shared__ float wm[8][NQ], wl[8][NQ];  // the warps' running maxima and normalisers
  __shared__ float wo[8][NQ][D];          // ... and O
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  const uint32_t b0 = smem_u32(bars);
  auto full = [&](int s) { return b0 + 8u * s; };
  auto empty = [&](int s) { return b0 + 8u * (NS + s); };
  int* abort_flag = reinterpret_cast<int*>(sm + C::OFF_BAR + 8 * 2 * NS);
  DevStatus st{a.status, abort_flag};
  const int G = gridDim.x, cta = blockIdx.x;
  const int BH = B * a.H, nq = a.N;
  // this CTA's tiles [g0, g1) of the sequence of all heads' tiles: heads [hpc c, hpc (c + 1))
  // whole, or (hpc = 0) the c-th of G equal runs
  long long g0, g1;
  if (hpc > 0) {
    g0 = dec_head_base(a, B, min(cta * hpc, BH));
    g1 = dec_head_base(a, B, min((cta + 1) * hpc, BH));
  } else {
    const long long T = dec_total(a, B);
    g0 = (long long)cta * T / G, g1 = (long long)(cta + 1) * T / G;
  }
  if (warp == 8) {
    if (lane == 0) {
      for (int s = 0; s < NS; ++s) {
        mbar_init(full(s), 1);
        mbar_init(empty(s), 8);  // one arrival per consumer warp
      }
      *abort_flag = 0;
      fence_mbar_init();
    }
  }
  __syncthreads();
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    int g = 0;  // ring tiles issued
    bool ok = true;
    if (g0 < g1) {
      DecCursor cur = dec_seek(a, B, g0);
      for (long long gt = g0; ok && gt < g1;) {
        const int bh = cur.b * a.H + cur.h;
        const int ta = (int)(gt - cur.gbase), te = (int)min(g1 - cur.gbase, (long long)cur.tb);
        for (int t = ta; t < te; ++t, ++g) {
          const int s = g % NS;
          if (!(ok = wait_warp_sleep(empty(s), ((g / NS) & 1) ^ 1, st, SITE_D_EMPTY))) break;
          if (elect_one()) mbar_arrive_expect_tx(full(s), 2 * C::TILE);
          for (int c = 0; c < C::NSUB; ++c) {
            const bool in = FA_CHECK(
                tma_coords_ok(c * 64, t * 128, bh, D, fwd_ext(a, false).rows_k, fwd_ext(a, false).heads, 2, 128, false) &&
                    smem_in(sbase + C::OFF_K + s * C::TILE + c * 16384, 16384, sbase + C::OFF_K, sbase + C::OFF_V) &&
                    smem_in(sbase + C::OFF_V + s * C::TILE + c * 16384, 16384, sbase + C::OFF_V, sbase + C::OFF_BAR),
                st, DBG_TMA_LOAD);
            if (in && elect_one()) tma_load_3d(sbase + C::OFF_K + s * C::TILE + c * 16384, &tm_k, c * 64, t * 128, bh, full(s));
            if (in && elect_one()) tma_load_3d(sbase + C::OFF_V + s * C::TILE + c * 16384, &tm_v, c * 64, t * 128, bh, full(s));
          }
          __syncwarp();
        }
        gt = cur.gbase + te;
        if (te == cur.tb) dec_next_head(a, B, cur);
      }
    }
    if (*(volatile int*)abort_flag) {
      // let copies already in flight land before the CTA's smem is released
      const uint64_t t0 = globaltimer_ns();
      for (int gg = max(0, g - NS); gg < g; ++gg)
        while (!mbar_try_wait(full(gg % NS), (gg / NS) & 1) && globaltimer_ns() - t0 < 100000000ull) {
        }
    }
  } else {
    // ------------------------------------------------------------ consumers (warps 0-7)
    // heads without a valid key: O = 0, LSE = -inf (heads cta, cta + G, ...)
    for (int bh = cta; bh < BH; bh += G) {
      if (dec_tiles(a, bh / a.H) > 0) continue;
      for (int idx = tid; idx < nq * D; idx += 256) {
        const size_t row = (size_t)bh * nq + idx / D;
        if (!FA_CHECK(in_range(row, fwd_ext(a, false).o_rows), st, DBG_GLOBAL_STORE)) continue;
        a.o[row * D + idx % D] = 0;
        if (idx % D == 0 && a.lse) a.lse[row] = -INFINITY;
      }
    }
    const int kl = lane & 15, half = lane >> 4;  // score phase: key of the warp, half of the row
    const int key = 16 * warp + kl;              // ... within the tile
    int g = 0;
    bool ok = true;
    DecCursor cur{};
    if (g0 < g1) cur = dec_seek(a, B, g0);
    for (long long gt = g0, seg = 0; ok && gt < g1; ++seg) {
      const int bh = cur.b * a.H + cur.h;
      const int ta = (int)(gt - cur.gbase), te = (int)min(g1 - cur.gbase, (long long)cur.tb);
      const int kv = (a.kv_len && FA_CHECK(in_range(cur.b, a.dbg_B), st, DBG_META))
                         ? min(max(a.kv_len[cur.b], 0), a.Nk)
                         : a.Nk;
      const int j1 = min(te * 128, kv);  // the segment's keys end here
      for (int idx = tid; idx < NQ * (D / 4); idx += 256) {
        const int i = idx / (D / 4), c = idx % (D / 4);
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < nq && FA_CHECK(in_range((size_t)bh * nq + i, fwd_ext(a, false).o_rows), st, DBG_GLOBAL_LOAD)) {
          const uint2 w = *reinterpret_cast<const uint2*>(q + ((size_t)bh * nq + i) * D + 4 * c);
          f = make_float4(__uint_as_float(w.x << 16) * a.scale_log2, __uint_as_float(w.x & 0xFFFF0000u) * a.scale_log2,
                          __uint_as_float(w.y << 16) * a.scale_log2, __uint_as_float(w.y & 0xFFFF0000u) * a.scale_log2);
        }
        qs[i][c] = f;
      }
      if (!(ok = named_bar_and(1, 256, ok))) break;
      bool wok = true;  // this warp's waits (voted at the segment's end)
      if constexpr (KM) {
        // ---- key-major: lane (kl, half) owns key kl of the warp's 16 in every tile and the
        //      head dimensions [half HD, half HD + HD) of its O. Each lane keeps its own
        //      reference maximum, normaliser and O (lazily rescaled: the reference moves only when
        //      a score exceeds it by more than 8, i.e. a factor 256), so a tile needs no reduction
        //      across lanes; the 16 lanes of each half are joined once, at the segment's end.
        float m[NQ], l[NQ], o[NQ][HD];
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          m[i] = -INFINITY, l[i] = 0.f;
#pragma unroll
          for (int e = 0; e < HD; ++e) o[i][e] = 0.f;
        }
        for (int t = ta; t < te; ++t, ++g) {
          const int s = g % NS;
          if (!(wok = wait_warp_sleep(full(s), (g / NS) & 1, st, SITE_D_FULL))) break;
          wok = FA_CHECK(smem_in(sbase + C::OFF_K + s * C::TILE, C::TILE, sbase + C::OFF_K, sbase + C::OFF_V) &&
                             smem_in(sbase + C::OFF_V + s * C::TILE, C::TILE, sbase + C::OFF_V, sbase + C::OFF_BAR),
                         st, DBG_SMEM);
          if (!wok) break;
          const uint8_t* kt = sm + C::OFF_K + s * C::TILE;
          const uint8_t* vt = sm + C::OFF_V + s * C::TILE;
          const int jj = t * 128 + key;
          const bool valid = jj < j1;
          uint4 kr[HD / 8], vr[HD / 8];
#pragma unroll
          for (int c = 0; c < HD / 8; ++c) {
            const int cc = half * (HD / 8) + c;  // 16-byte chunk of the row
            const int off = (cc >> 3) * 16384 + sw128_offset(key, cc & 7);
            kr[c] = *reinterpret_cast<const uint4*>(kt + off);
            vr[c] = *reinterpret_cast<const uint4*>(vt + off);
          }
          // this lane's K and V rows are in registers: the stage may be refilled
          __syncwarp();
          if (lane == 0) mbar_arrive(empty(s));
#pragma unroll
          for (int i = 0; i < NQ; ++i) {
            uint64_t acc2 = f2_pack(0.f, 0.f);
            if (i < nq) {
#pragma unroll
              for (int c = 0; c < HD / 8; ++c) {
                const float4 q0 = qs[i][half * (HD / 4) + 2 * c], q1 = qs[i][half * (HD / 4) + 2 * c + 1];
                const uint32_t w[4] = {kr[c].x, kr[c].y, kr[c].z, kr[c].w};
                acc2 = f2_fma(f2_pack(q0.x, q0.y), f2_pack(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u)), acc2);
                acc2 = f2_fma(f2_pack(q0.z, q0.w), f2_pack(__uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u)), acc2);
                acc2 = f2_fma(f2_pack(q1.x, q1.y), f2_pack(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u)), acc2);
                acc2 = f2_fma(f2_pack(q1.z, q1.w), f2_pack(__uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u)), acc2);
              }
            }
            float a0, a1;
            f2_unpack(acc2, a0, a1);
            float acc = a0 + a1;
            acc += __shfl_xor_sync(0xffffffffu, acc, 16);
            // causal: query i keeps keys j <= i + N_k - N_q; past the head's valid keys: none
            const float sc = (i < nq && valid && !(a.causal && jj > i + a.coff)) ? acc : -INFINITY;
            if (sc > m[i] + 8.f) {  // both lanes of a key take the same branch
              const float alpha = (m[i] == -INFINITY) ? 0.f : ex2_approx(m[i] - sc);
              l[i] *= alpha;
#pragma unroll
              for (int e = 0; e < HD; ++e) o[i][e] *= alpha;
              m[i] = sc;
            }
            const float p = (sc == -INFINITY) ? 0.f : ex2_approx(sc - m[i]);
            l[i] += p;
            const uint64_t p2 = f2_pack(p, p);
#pragma unroll
            for (int c = 0; c < HD / 8; ++c) {
              const uint32_t w[4] = {vr[c].x, vr[c].y, vr[c].z, vr[c].w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint64_t r2 = f2_fma(p2, f2_pack(__uint_as_float(w[u] << 16), __uint_as_float(w[u] & 0xFFFF0000u)),
                                           f2_pack(o[i][8 * c + 2 * u], o[i][8 * c + 2 * u + 1]));
                f2_unpack(r2, o[i][8 * c + 2 * u], o[i][8 * c + 2 * u + 1]);
              }
            }
          }
        }
        // ---- join the 16 lanes of each half (same dimensions, different keys), then publish
        //      the warp's state: lane 0 the maximum and normaliser, lanes 0 and 16 their halves of O
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          float mx = m[i];
#pragma unroll
          for (int sh = 1; sh < 16; sh <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
          const float f = (m[i] == -INFINITY) ? 0.f : ex2_approx(m[i] - mx);
          float ls = l[i] * f;
#pragma unroll
          for (int sh = 1; sh < 16; sh <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, sh);
#pragma unroll
          for (int e = 0; e < HD; ++e) {
            float x = o[i][e] * f;
#pragma unroll
            for (int sh = 1; sh < 16; sh <<= 1) x += __shfl_xor_sync(0xffffffffu, x, sh);
            if (kl == 0) wo[warp][i][half * HD + e] = x;
          }
          if (lane == 0) wm[warp][i] = mx, wl[warp][i] = ls;
        }
      } else {
        float m[NQ], l[NQ], o[NQ][DPL];
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          m[i] = -INFINITY, l[i] = 0.f;
#pragma unroll
          for (int e = 0; e < DPL; ++e) o[i][e] = 0.f;
        }
        for (int t = ta; t < te; ++t, ++g) {
          const int s = g % NS;
          const int jb = t * 128;
          if (!(wok = wait_warp_sleep(full(s), (g / NS) & 1, st, SITE_D_FULL))) break;
          wok = FA_CHECK(smem_in(sbase + C::OFF_K + s * C::TILE, C::TILE, sbase + C::OFF_K, sbase + C::OFF_V) &&
                             smem_in(sbase + C::OFF_V + s * C::TILE, C::TILE, sbase + C::OFF_V, sbase + C::OFF_BAR),
                         st, DBG_SMEM);
          if (!wok) break;
          const uint8_t* kt = sm + C::OFF_K + s * C::TILE;
          const uint8_t* vt = sm + C::OFF_V + s * C::TILE;
          const int jj = jb + key;
          const bool valid = jj < j1;
          // ---- half-row partial scores of this lane's key, joined across the two halves
          uint4 kr[HD / 8];
#pragma unroll
          for (int c = 0; c < HD / 8; ++c) {
            const int cc = half * (HD / 8) + c;  // 16-byte chunk of the row
            kr[c] = *reinterpret_cast<const uint4*>(kt + (cc >> 3) * 16384 + sw128_offset(key, cc & 7));
          }
          float sc[NQ];
#pragma unroll
          for (int i = 0; i < NQ; ++i) {
            float acc = 0.f;
            if (i < nq) {
#pragma unroll
              for (int c = 0; c < HD / 8; ++c) {
                const float4 q0 = qs[i][half * (HD / 4) + 2 * c], q1 = qs[i][half * (HD / 4) + 2 * c + 1];
                const uint32_t w[4] = {kr[c].x, kr[c].y, kr[c].z, kr[c].w};
                acc = fmaf(q0.x, __uint_as_float(w[0] << 16), acc);
                acc = fmaf(q0.y, __uint_as_float(w[0] & 0xFFFF0000u), acc);
                acc = fmaf(q0.z, __uint_as_float(w[1] << 16), acc);
                acc = fmaf(q0.w, __uint_as_float(w[1] & 0xFFFF0000u), acc);
                acc = fmaf(q1.x, __uint_as_float(w[2] << 16), acc);
                acc = fmaf(q1.y, __uint_as_float(w[2] & 0xFFFF0000u), acc);
                acc = fmaf(q1.z, __uint_as_float(w[3] << 16), acc);
                acc = fmaf(q1.w, __uint_as_float(w[3] & 0xFFFF0000u), acc);
              }
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 16);
            // causal: query i keeps keys j <= i + N_k - N_q; past the head's valid keys: none
            sc[i] = (i < nq && valid && !(a.causal && jj > i + a.coff)) ? acc : -INFINITY;
          }
          // ---- the warp's maximum and sum over its 16 keys; rescale; O += P V
          float p[NQ];
#pragma unroll
          for (int i = 0; i < NQ; ++i) {
            float x = sc[i];
#pragma unroll
            for (int sh = 8; sh > 0; sh >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, sh));
            const float mnew = fmaxf(m[i], x);
            const float alpha = (mnew == -INFINITY) ? 1.f : ex2_approx(m[i] - mnew);
            p[i] = (sc[i] == -INFINITY) ? 0.f : ex2_approx(sc[i] - mnew);
            float y = p[i];
#pragma unroll
            for (int sh = 8; sh > 0; sh >>= 1) y += __shfl_xor_sync(0xffffffffu, y, sh);
            l[i] = l[i] * alpha + y;
            m[i] = mnew;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[i][e] *= alpha;
          }
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const int r = 16 * warp + kk;           // V row
            const int d0 = lane * DPL;              // this lane's first dimension
            const int cc = d0 >> 3;                 // its 16-byte chunk
            const uint8_t* src = vt + (cc >> 3) * 16384 + sw128_offset(r, cc & 7) + (d0 & 7) * 2;
            uint32_t w[DPL / 2];
            if (DPL == 2) {
              w[0] = *reinterpret_cast<const uint32_t*>(src);
            } else {
              const uint2 t2 = *reinterpret_cast<const uint2*>(src);
              w[0] = t2.x;
              w[DPL / 2 - 1] = t2.y;
            }
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
              const float pk = __shfl_sync(0xffffffffu, p[i], kk);
#pragma unroll
              for (int e = 0; e < DPL / 2; ++e) {
                o[i][2 * e] = fmaf(pk, __uint_as_float(w[e] << 16), o[i][2 * e]);
                o[i][2 * e + 1] = fmaf(pk, __uint_as_float(w[e] & 0xFFFF0000u), o[i][2 * e + 1]);
              }
            }
          }
          // this warp is done with the stage's K and V
          __syncwarp();
          if (lane == 0) mbar_arrive(empty(s));
        }
        // ---- join the eight warps' states; whole head: O and LSE, else partial slot 2c or 2c + 1
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          if (lane == 0) wm[warp][i] = m[i], wl[warp][i] = l[i];
#pragma unroll
          for (int e = 0; e < DPL; ++e) wo[warp][i][lane * DPL + e] = o[i][e];
        }
      }
      if (!(ok = named_bar_and(1, 256, wok))) break;
      const bool whole = (ta == 0 && te == cur.tb);
      const int slot = 2 * cta + (seg == 0 ? 0 : 1);
      for (int idx = tid; idx < nq * D; idx += 256) {
        const int i = idx / D, d = idx % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < 8; ++w) mx = fmaxf(mx, wm[w][i]);
        float lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const float f = (wm[w][i] == -INFINITY) ? 0.f : ex2_approx(wm[w][i] - mx);
          lsum = fmaf(wl[w][i], f, lsum);
          acc = fmaf(wo[w][i][d], f, acc);
        }
        const float lse = (lsum > 0.f) ? (mx + lg2_approx(lsum)) * 0.6931471805599453f : -INFINITY;
        const float ov = (lsum > 0.f) ? acc / lsum : 0.f;
        if (whole) {
          const size_t row = (size_t)bh * nq + i;
          if (!FA_CHECK(in_range(row, fwd_ext(a, false).o_rows), st, DBG_GLOBAL_STORE)) continue;
          a.o[row * D + d] = (uint16_t)(pack_bf16x2(ov, 0.f) & 0xFFFFu);
          if (d == 0 && a.lse) a.lse[row] = lse;
        } else {
          const size_t row = (size_t)slot * nq + i;
          if (!FA_CHECK(in_range(row, fwd_ext(a, false).part_rows), st, DBG_GLOBAL_STORE)) continue;
          a.part_o[row * D + d] = ov;
          if (d == 0) a.part_lse[row] = lse;
        }
      }
      if (!(ok = named_bar_and(1, 256, ok))) break;  // qs and the warps' states are rewritten next
      gt = cur.gbase + te;
      if (te == cur.tb) dec_next_head(a, B, cur);
    }
  }
}

// Joins the segments of each head that decode_kernel split between CTAs (grid: one block per
// head). The head's tiles are global tiles [gs, ge); CTA c of G took [c T / G, (c + 1) T / G),
// so the owner of tile g is ((g + 1) G - 1) / T. The first owner's segment is in its slot 2c
// when its range starts at gs, else in 2c + 1 (its last segment); every later CTA with tiles up
// to the owner of ge - 1 holds its first segment in slot 2c. With L_z the segments' LSEs and
// M their maximum: LSE = M + ln sum_z e^(L_z - M), O = sum_z e^(L_z - LSE) O_z, each O_z
// already divided by its own normaliser; segments with no visible key (L_z = -inf) drop out.
// The slot list and the LSEs go through shared memory, so each thread's loads of O_z are
// independent of one another (two memory round trips in all). G <= kDecodeMaxCtas.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(FwdArgs a, int B, int G) {
  griddep_wait();
  griddep_launch_dependents();
  const int bh = blockIdx.x, b = bh / a.H, h = bh - b * a.H, tid = threadIdx.x;
  const int tb = dec_tiles(a, b);
  if (tb == 0) return;
  // T and the tiles of the batches before b, summed over the block
  __shared__ long long part[2][8];
  __shared__ int slots[kDecodeMaxCtas];
  __shared__ float lses[kDecodeMaxCtas][kDecodeMaxRows];
  __shared__ float wmax[kDecodeMaxRows];
  long long sT = 0, sB = 0;
  if (a.kv_len) {
    for (int bb = tid; bb < B; bb += 256) {
      const long long x = (long long)a.H * dec_tiles(a, bb);
      sT += x;
      if (bb < b) sB += x;
    }
  } else if (tid == 0) {
    sT = (long long)B * a.H * tb;
    sB = (long long)b * a.H * tb;
  }
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) {
    sT += __shfl_xor_sync(0xffffffffu, sT, sh);
    sB += __shfl_xor_sync(0xffffffffu, sB, sh);
  }
  if ((tid & 31) == 0) part[0][tid >> 5] = sT, part[1][tid >> 5] = sB;
  __syncthreads();
  long long T = 0, gs = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) T += part[0][w], gs += part[1][w];
  gs += (long long)h * tb;
  const long long ge = gs + tb;
  const int clo = (int)(((gs + 1) * G - 1) / T), chi = (int)((ge * G - 1) / T);
  if (clo == chi) return;  // one CTA held the whole head and wrote it
  const int nseg = chi - clo + 1, nq = a.N;
  // entry e: CTA clo + e, its slot (or -1: a CTA without tiles)
  if (!FA_CHECK(nseg <= kDecodeMaxCtas && nq <= kDecodeMaxRows, a.status, DBG_SMEM)) return;
  if (tid < nseg) {
    const int c = clo + tid;
    const long long st0 = (long long)c * T / G, st1 = (long long)(c + 1) * T / G;
    slots[tid] = (tid > 0 && st0 == st1) ? -1 : (tid == 0 && st0 < gs) ? 2 * c + 1 : 2 * c;
  }
  __syncthreads();
  for (int idx = tid; idx < nseg * nq; idx += 256) {
    const int e = idx / nq, i = idx - e * nq;
    lses[e][i] = (slots[e] < 0 || !FA_CHECK(in_range((size_t)slots[e] * nq + i, fwd_ext(a, false).part_rows),
                                            a.status, DBG_GLOBAL_LOAD))
                     ? -INFINITY
                     : a.part_lse[(size_t)slots[e] * nq + i];
  }
  __syncthreads();
  if (tid < nq) {
    float mx = -INFINITY;
    for (int e = 0; e < nseg; ++e) mx = fmaxf(mx, lses[e][tid]);
    wmax[tid] = mx;
  }
  __syncthreads();
  for (int idx = tid; idx < nq * D; idx += 256) {
    const int i = idx / D, d = idx - i * D;
    const float mx = wmax[i];
    float wsum = 0.f, acc = 0.f;
    if (mx != -INFINITY) {
#pragma unroll 4
      for (int e = 0; e < nseg; ++e) {
        const float lz = lses[e][i];
        const float w = (lz == -INFINITY) ? 0.f : ex2_approx((lz - mx) * 1.4426950408889634f);
        const float oz = (w > 0.f) ? a.part_o[((size_t)slots[e] * nq + i) * D + d] : 0.f;
        wsum += w;
        acc = fmaf(w, oz, acc);
      }
    }
    const size_t row = (size_t)bh * nq + i;
    if (!FA_CHECK(in_range(row, fwd_ext(a, false).o_rows), a.status, DBG_GLOBAL_STORE)) continue;
    a.o[row * D + d] = (uint16_t)(pack_bf16x2(wsum > 0.f ? acc / wsum : 0.f, 0.f) & 0xFFFFu);
    if (d == 0 && a.lse) a.lse[row] = (wsum > 0.f) ? mx + lg2_approx(wsum) * 0.6931471805599453f : -INFINITY;
  }
}

// BH = B * H work items per query pair. VL: the tensors are [H, T, d] (rows of all sequences
// packed per head), so the maps span T rows and H heads.
template <int D, bool SPLIT = false, bool VL = false, bool ONE = false>
static int launch_fwd_d(const void* q, const void* k, const void* v, void* o, const FwdArgs& args, int BH,
                        cudaStream_t stream) {
  using C = FwdCfg<D, SPLIT>;
  CUtensorMap mq, mk, mv, mo;
  const uint64_t N = (uint64_t)(VL ? args.T : args.N), Nk = (uint64_t)(VL ? args.T : args.Nk);
  const uint64_t Z = (uint64_t)(VL ? args.H : BH);
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_tmap_3d(&mq, q, BF, 2, D, N, Z, 64, 128, SW) || !make_tmap_3d(&mk, k, BF, 2, D, Nk, Z, 64, 128, SW) ||
      !make_tmap_3d(&mv, v, BF, 2, D, Nk, Z, 64, 128, SW) || !make_tmap_3d(&mo, o, BF, 2, D, N, Z, 64, 128, SW))
    return cuda_fail("cuTensorMapEncodeTiled", 0, "tensor map rejected");
  static bool attr_set = false;  // benign race: idempotent
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D, SPLIT, VL, ONE>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_fail("cudaFuncSetAttribute", (int)e, cudaGetErrorName(e));
    attr_set = true;
  }
  FwdArgs a = args;
  if (ONE) a.n_pairs = (args.N + 127) / 128;  // query tiles along y
  dim3 grid(BH, a.n_pairs, SPLIT ? args.n_split : 1);
  return launch_pdl(__func__, fwd_kernel<D, SPLIT, VL, ONE>, grid, dim3(C::THREADS), C::SMEM_BYTES, stream, mq, mk,
                    mv, mo, a);
}

// d = 64: the persistent kernel, one CTA per SM (at most one per work item). VL: packed
// sequences, [H, T, d] tensors; BH = B * H items per query pair.
template <bool VL = false>
static int launch_fwd_p64(const void* q, const void* k, const void* v, void* o, const FwdArgs& args, int BH,
                          cudaStream_t stream) {
  using C = FwdP64;
  CUtensorMap mq, mk, mv, mo;
  const uint64_t N = (uint64_t)(VL ? args.T : args.N), Nk = (uint64_t)(VL ? args.T : args.Nk);
  const uint64_t Z = (uint64_t)(VL ? args.H : BH);
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_tmap_3d(&mq, q, BF, 2, 64, N, Z, 64, 128, SW) || !make_tmap_3d(&mk, k, BF, 2, 64, Nk, Z, 64, 128, SW) ||
      !make_tmap_3d(&mv, v, BF, 2, 64, Nk, Z, 64, 128, SW) || !make_tmap_3d(&mo, o, BF, 2, 64, N, Z, 64, 128, SW))
    return cuda_fail("cuTensorMapEncodeTiled", 0, "tensor map rejected");
  static bool attr_set = false;  // benign race: idempotent
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(fwd_kernel_p64<VL>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_fail("cudaFuncSetAttribute", (int)e, cudaGetErrorName(e));
    attr_set = true;
  }
  int sms = 0;
  if (!sm_count(&sms)) return FA_ERR_CUDA;
  const long long items = (long long)BH * args.n_pairs;
  const dim3 grid((unsigned)std::min<long long>(items, sms));
  return launch_pdl(__func__, fwd_kernel_p64<VL>, grid, dim3(C::THREADS), C::SMEM_BYTES, stream, mq, mk, mv, mo,
                    args, BH);
}

int launch_fwd(const void* q, const void* k, const void* v, void* o, const FwdArgs& args, int BH, int d,
               cudaStream_t stream) {
  // Short rows (at most 4 query-tile pairs and 1024 keys): the persistent kernel, whose
  // per-CTA setup and item epilogues overlap the next item's MMAs. Longer rows: one CTA per
  // item, where the hardware's block dispatch balances the causal work at least as well as
  // the static order and the per-item setup is amortised over many key tiles.
  if (d == 64 && args.n_pairs <= 4 && args.Nk <= 1024) return launch_fwd_p64<false>(q, k, v, o, args, BH, stream);
  // Fewer pairs than SMs: one query tile per CTA, so that more SMs work and each lane runs
  // alone (a lane alone takes ~1700 cycles a key tile, two sharing an SM ~2175 each).
  int sms = 0;
  const bool one = sm_count(&sms) && (long long)BH * args.n_pairs < sms;
  if (d == 64) return one ? launch_fwd_d<64, false, false, true>(q, k, v, o, args, BH, stream)
                          : launch_fwd_d<64>(q, k, v, o, args, BH, stream);
  if (d == 128) return one ? launch_fwd_d<128, false, false, true>(q, k, v, o, args, BH, stream)
                           : launch_fwd_d<128>(q, k, v, o, args, BH, stream);
  return FA_ERR_UNSUPPORTED;
}

int launch_fwd_varlen(const void* q, const void* k, const void* v, void* o, const FwdArgs& args, int BH, int d,
                      cudaStream_t stream) {
  // sequences of at most 1024 rows: the persistent kernel over (query pair, sequence x head)
  if (d == 64 && args.n_pairs <= 4) return launch_fwd_p64<true>(q, k, v, o, args, BH, stream);
  if (d == 64) return launch_fwd_d<64, false, true>(q, k, v, o, args, BH, stream);
  if (d == 128) return launch_fwd_d<128, false, true>(q, k, v, o, args, BH, stream);
  return FA_ERR_UNSUPPORTED;
}

// The CTAs of the decode kernel. n_split = 1: whole heads, hpc = ceil(B H / min(#SMs, 256))
// of them a CTA, never a join. n_split > 1: stream-K over G = min(#SMs, 256, n_split B H, T_max)
// CTAs (T_max: the tiles of all heads at N_k keys each), so that the 2 G partial slots fit the
// workspace of n_split shares; whether some head may be split between CTAs is written to
// *split (always, with key padding: the tile counts are on the device).
static int decode_grid(const FwdArgs& args, int BH, int sms, int* hpc, bool* split) {
  const long long cap = std::min(sms, kDecodeMaxCtas);
  if (args.n_split == 1) {
    *hpc = (int)((BH + cap - 1) / cap);
    *split = false;
    return (BH + *hpc - 1) / *hpc;
  }
  *hpc = 0;
  const long long t_head = (args.Nk + 127) / 128;
  const long long t_max = std::max<long long>(1, BH * t_head);
  const int G = (int)std::max<long long>(1, std::min<long long>({cap, (long long)args.n_split * BH, t_max}));
  *split = args.kv_len != nullptr;
  for (int c = 1; c < G && !*split; ++c)  // without padding a head splits where a CTA starts inside it
    if ((long long)c * t_max / G % t_head != 0) *split = true;
  return G;
}

int launch_fwd_split(const void* q, const void* k, const void* v, void* o, const FwdArgs& args, int BH, int d,
                     cudaStream_t stream) {
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  int rc;
  if (args.N <= kDecodeMaxRows) {
    // decode: the streaming stream-K kernel over all heads' key tiles, then (if a head was split
    // between CTAs) the join of its segments
    CUtensorMap mk, mv;
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_tmap_3d(&mk, k, BF, 2, d, (uint64_t)args.Nk, BH, 64, 128, SW) ||
        !make_tmap_3d(&mv, v, BF, 2, d, (uint64_t)args.Nk, BH, 64, 128, SW))
      return cuda_fail("cuTensorMapEncodeTiled", 0, "tensor map rejected");
    int sms = 0;
    if (!sm_count(&sms)) return FA_ERR_CUDA;
    bool split = false;
    int hpc = 0;
    const int G = decode_grid(args, BH, sms, &hpc, &split);
    const int B = BH / args.H;
    const auto* qq = static_cast<const uint16_t*>(q);
    auto go = [&](auto kernel, int smem) {
      const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return cuda_fail("cudaFuncSetAttribute", (int)e, cudaGetErrorName(e));
      return launch_pdl("decode_kernel", kernel, dim3(G), dim3(288), (size_t)smem, stream, mk, mv, qq, args, B,
                        hpc);
    };
    const int r = args.N;
#define FA_DEC(DD, NN) go(decode_kernel<DD, NN>, DecCfg<DD, NN>::SMEM_BYTES)
    if (d == 64)
      rc = r <= 1 ? FA_DEC(64, 1) : r <= 2 ? FA_DEC(64, 2) : r <= 4 ? FA_DEC(64, 4) : FA_DEC(64, 8);
    else
      rc = r <= 1 ? FA_DEC(128, 1) : r <= 2 ? FA_DEC(128, 2) : r <= 4 ? FA_DEC(128, 4) : FA_DEC(128, 8);
#undef FA_DEC
    if (rc != FA_OK || !split) return rc;
    return (d == 64) ? launch_pdl("decode_combine_kernel", decode_combine_kernel<64>, dim3(BH), dim3(256), 0, stream,
                                  args, B, G)
                     : launch_pdl("decode_combine_kernel", decode_combine_kernel<128>, dim3(BH), dim3(256), 0, stream,
                                  args, B, G);
  }
  rc = (d == 64) ? launch_fwd_d<64, true>(q, k, v, o, args, BH, stream)
                 : launch_fwd_d<128, true>(q, k, v, o, args, BH, stream);
  if (rc != FA_OK) return rc;
  const int rpb = 256 / (d / 8);
  const dim3 grid((unsigned)((args.N + rpb - 1) / rpb), (unsigned)BH);
  return (d == 64) ? launch_pdl("fwd_combine_kernel", fwd_combine_kernel<64>, grid, dim3(256), 0, stream, args)
                   : launch_pdl("fwd_combine_kernel", fwd_combine_kernel<128>, grid, dim3(256), 0, stream, args);
}

}  // namespace fa
