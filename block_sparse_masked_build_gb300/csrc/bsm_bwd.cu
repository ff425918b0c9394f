// Block-sparse masked attention backward for sm_103a (GB300): dQ, dK, dV of
// sum(dO * out) for both score paths, over the same mask info as the
// forward.
//
// Softmax path (the forward of the splash notes section 15, differentiated):
// with s = scale * q.k over the visible keys, P = exp(s - lse) (lse of the
// forward), D_q = sum_d dO[q, d] * out[q, d]:
//     dV = P^T dO,  dS = P * (dO V^T - D_q),  dQ = scale dS K,
//     dK = scale dS^T Q.
// Pointwise path (hstu_ops `_pointwise_splash_attention_bwd_kernel_impl`):
// with x = scale * q.k, sig = logistic(x), p = x sig / Sq (0 where masked),
//     dV = p^T dO,  dS = (dO V^T) sig (1 + x (1 - sig)) / Sq,
//     dQ = scale dS K,  dK = scale dS^T Q.
// As in hstu_ops' backward, p (and dS) are rounded to the input type (bf16)
// for the products; accumulation is f32 in TMEM.
//
// Two kernels, no atomics:
//   dK/dV: one CTA per (batch, K/V head, 128-key tile); it walks the query
//          tiles the mask info marks nonzero for its key tile (the
//          transposed walk of the forward's), for every query head of the
//          K/V head's group, and accumulates dV and dK in TMEM.
//   dQ:    one CTA per (batch, head, 128-row query tile); it walks the key
//          tiles of its row, as the forward does, and accumulates dQ.
// A third, small kernel computes D_q (softmax path only).
//
// Warp roles (320 threads): warp 0 loads with TMA (the CTA's fixed pair of
// tiles once, then the streamed pair of every step through a two-stage
// ring), warp 1 issues the tcgen05 MMAs (the whole warp runs the issuing
// code, the lane elect.sync picks sends each MMA) and owns the TMEM
// allocation, warps 2-9 do the elementwise work, a thread per TMEM lane (a
// row of the fixed tiles) and column half.  Per step, with F0/F1 the fixed tiles and
// T0/T1 the streamed ones (dK/dV: F = K, V and T = Q, dO; dQ: F = Q, dO and
// T = K, V):
//     S  = F0 T0^T   -> TMEM [0, 128)      (both operands K-major in smem)
//     dP = F1 T1^T   -> TMEM [128, 256)
//     elementwise: P (dK/dV only) over S's columns, dS over dP's, as bf16
//     dK/dV: dV += P T1, dK += dS T0 (A from TMEM, B = the streamed tile
//            read MN-major) -> TMEM [256, 256 + D), [384, 384 + D)
//     dQ:    dQ += dS T0 -> TMEM [256, 256 + D)
// Every mbarrier wait is bounded; a role that gives up records the error
// (read by bsm_device_status) and every role stops.
#include <cstdint>

#include "bsm_internal.h"
#include "bsm_ptx.cuh"

namespace bsm {

// Error record of the backward kernels: [0] code, [1] block, [2] role,
// [3] phase.
__device__ int g_bwd_error[4];

namespace {

constexpr int kBwdThreads = 320;  // warps 0-1 roles, 2-9 elementwise
constexpr int kBwdBand = 16;      // tiles per band of the causal block order
constexpr uint32_t kBwdTmemCols = 512;
constexpr int kRoleBLoad = 11, kRoleBMma = 12, kRoleBElem = 13;

template <int D>
struct BwdCfg {
  static constexpr int kKBlocks = D / 64;            // 128-byte k-blocks
  static constexpr int kTileBytes = kTileM * D * 2;  // one 128-row tile
  static constexpr int kOffF = 0;                    // fixed F0, F1
  static constexpr int kOffT = 2 * kTileBytes;       // ring: 2 x (T0, T1)
  static constexpr int kOffList = kOffT + 4 * kTileBytes;
  static constexpr int kOffBar = kOffList + kMaxKvTiles * 2;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
};
static_assert(BwdCfg<128>::kSmemBytes <= 232448, "shared memory budget");

struct BwdBars {
  uint64_t f_full;
  uint64_t t_full[2], t_empty[2];
  uint64_t s_full, dp_full, acc_done, mma_done;
  // elementwise -> MMA: P stored (dK/dV) or S read (dQ); dS stored
  uint64_t p_ready, ds_ready;
  // the first column half has read S, and dP
  uint64_t h0_s, h0_dp;
  uint32_t tmem_base;
  int abort;
  int n_list;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block");

__device__ __forceinline__ void record_bwd_timeout(int role, int phase) {
  if (atomicCAS(&g_bwd_error[0], 0, 1) == 0) {
    g_bwd_error[1] = blockIdx.x;
    g_bwd_error[2] = role;
    g_bwd_error[3] = phase;
  }
}

__device__ __forceinline__ bool bwarp_wait(uint64_t* bar, uint32_t parity,
                                           volatile int* abort_flag,
                                           uint64_t timeout_ns) {
  const bool ok = mbar_wait(bar, parity, abort_flag, timeout_ns);
  return __all_sync(0xffffffffu, ok);
}

// Class of (128-row query tile starting at row R0) x (key tile jt) from the
// mask-info blocks covering it: 2 if all are full, 0 if all are empty, else
// 1; a key tile cut by the end of the keys is never full (the same
// combination as the forward's).
__device__ __forceinline__ int bwd_tile_class(const BwdParams& p, int table,
                                              int R0, int jt) {
  if (R0 >= p.Sq) return 0;
  const int R1 = min(p.Sq, R0 + kTileM) - 1;
  const int C0 = jt * kTileN;
  const int C1 = min(p.Skv, C0 + kTileN) - 1;
  const int i0 = R0 / p.bq, i1 = R1 / p.bq;
  const int j0 = C0 / p.bkv, j1 = C1 / p.bkv;
  const int8_t* bm =
      p.block_mask + static_cast<int64_t>(table) * p.mi_nq * p.mi_nk;
  bool all_full = true, any = false;
  for (int i = i0; i <= i1; ++i)
    for (int j = j0; j <= j1; ++j) {
      const int c = bm[static_cast<int64_t>(i) * p.mi_nk + j];
      all_full = all_full && (c == 2);
      any = any || (c != 0);
    }
  if (!any) return 0;
  if (all_full && C0 + kTileN <= p.Skv) return 2;
  return 1;
}

// Bits of the columns [lo, hi] within the 32 columns starting at c0.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int c0) {
  const int lb = min(max(lo - c0, 0), 32), hb = min(max(hi - c0 + 1, 0), 32);
  const uint32_t below_hi = hb >= 32 ? 0xffffffffu : (1u << hb) - 1u;
  const uint32_t below_lo = lb >= 32 ? 0xffffffffu : (1u << lb) - 1u;
  return below_hi & ~below_lo;
}

// Visibility bits of one thread's row against 32 consecutive columns
// starting at c0 (a multiple of 32), under every predicate of the mask (the
// ones the mask-info builder applies).  DKDV: the row is key `row` and the
// columns are queries; dQ: the row is query `row` and the columns are keys.
// Causal/local/band and the sequence ends are a range of columns; segment
// ids and arbitrary-mask words of the 32 columns are loaded one per lane
// and passed around with shuffles.  Whole warp.
template <bool DKDV>
__device__ __forceinline__ uint32_t chunk_visible(const BwdParams& p, int b,
                                                  int row, int row_seg,
                                                  int c0) {
  const int lane = threadIdx.x % 32;
  int lo, hi;
  if (DKDV) {  // queries q that see key k = row
    const int k = row;
    lo = 0;
    hi = p.Sq - 1;
    if (p.flags & BSM_MASK_CAUSAL) lo = max(lo, k);
    if (p.flags & BSM_MASK_LOCAL) hi = min(hi, k + p.window - 1);
    if (p.flags & BSM_MASK_BAND) lo = max(lo, k - p.window + 1);
    if (k >= p.Skv) hi = -1;
  } else {  // keys k that query q = row sees
    const int q = row;
    lo = 0;
    hi = p.Skv - 1;
    if (p.flags & BSM_MASK_CAUSAL) hi = min(hi, q);
    if (p.flags & BSM_MASK_LOCAL) lo = max(lo, q - p.window + 1);
    if (p.flags & BSM_MASK_BAND) hi = min(hi, q + p.window - 1);
    if (q >= p.Sq) hi = -1;
  }
  uint32_t bits = range_bits(lo, hi, c0);
  const int col = c0 + lane;  // this lane's column
  if (p.flags & BSM_MASK_SEGMENT) {
    int cs = 0;
    if (DKDV ? col < p.Sq : col < p.Skv)
      cs = DKDV ? p.q_seg[static_cast<int64_t>(b) * p.Sq + col]
                : p.kv_seg[static_cast<int64_t>(b) * p.Skv + col];
    uint32_t same = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      same |= (__shfl_sync(0xffffffffu, cs, j) == row_seg ? 1u : 0u) << j;
    bits &= same;
  }
  if (p.dense != nullptr) {
    if (DKDV) {
      // word (query col, keys of this warp): the warp's 32 keys share it
      const int kw = (row - lane) >> 5;
      uint32_t w = 0;
      if (col < p.Sq && kw * 32 < p.Skv)
        w = __ldg(p.dense + static_cast<int64_t>(col) * p.dense_words + kw);
      uint32_t keep = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        keep |= ((__shfl_sync(0xffffffffu, w, j) >> lane) & 1u) << j;
      bits &= keep;
    } else {
      uint32_t w = 0;
      if (row < p.Sq && c0 < p.Skv)
        w = __ldg(p.dense + static_cast<int64_t>(row) * p.dense_words +
                  (c0 >> 5));
      bits &= w;
    }
  }
  return bits;
}

// The CTA's list of nonzero tiles (uint16: tile << 2 | class), built by one
// warp into shared memory.  DKDV: the query tiles of key tile `fixed_tile`;
// dQ: the key tiles of query tile `fixed_tile`.
template <bool DKDV>
__device__ __forceinline__ int build_bwd_list(const BwdParams& p, int table,
                                              int fixed_tile, uint16_t* list) {
  const int lane = threadIdx.x % 32;
  const int n_tiles = DKDV ? (p.Sq + kTileM - 1) / kTileM
                           : (p.Skv + kTileN - 1) / kTileN;
  int n = 0;
  for (int base = 0; base < n_tiles; base += 32) {
    const int x = base + lane;
    int c = 0;
    if (x < n_tiles)
      c = DKDV ? bwd_tile_class(p, table, x * kTileM, fixed_tile)
               : bwd_tile_class(p, table, fixed_tile * kTileM, x);
    const unsigned m = __ballot_sync(0xffffffffu, c != 0);
    if (c) list[n + __popc(m & ((1u << lane) - 1u))] =
        static_cast<uint16_t>((x << 2) | c);
    n += __popc(m);
  }
  return n;
}

template <int D, bool DKDV>
__device__ __forceinline__ void bwd_load_role(
    const BwdParams& p, const CUtensorMap* tq, const CUtensorMap* tk,
    const CUtensorMap* tv, const CUtensorMap* tdo, uint8_t* smem,
    BwdBars* bars, const uint16_t* list, int b, int hq_or_hkv, int fixed_tile,
    int n_iter) {
  using C = BwdCfg<D>;
  const int lane = threadIdx.x % 32;
  volatile int* abort_flag = &bars->abort;
  const int G = p.H / p.Hkv;
  const int n_list = bars->n_list;
  const uint64_t pol_fixed = l2_policy_evict_first();
  const uint64_t pol_stream = l2_policy_evict_last();
  bool ok = true;
  uint32_t issued = 0;
  if (lane == 0) {
    // fixed pair: dK/dV: K, V of (b, hkv, key tile); dQ: Q, dO of
    // (b, h, query tile)
    mbar_arrive_expect_tx(&bars->f_full, 2 * C::kTileBytes);
    const int row0 = fixed_tile * kTileM;
    for (int kb = 0; kb < C::kKBlocks; ++kb) {
      tma_load_4d(DKDV ? tk : tq, &bars->f_full,
                  smem + C::kOffF + kb * kTileM * 128, kb * 64, row0,
                  hq_or_hkv, b, pol_fixed);
      tma_load_4d(DKDV ? tv : tdo, &bars->f_full,
                  smem + C::kOffF + C::kTileBytes + kb * kTileM * 128,
                  kb * 64, row0, hq_or_hkv, b, pol_fixed);
    }
  }
  for (int it = 0; ok && it < n_iter; ++it) {
    const int s = it & 1;
    ok = bwarp_wait(&bars->t_empty[s], ((it >> 1) & 1) ^ 1, abort_flag,
                    p.timeout_ns);
    if (!ok) {
      if (lane == 0) record_bwd_timeout(kRoleBLoad, 0);
      break;
    }
    if (lane == 0) {
      const int e = it % n_list;
      const int tile = list[e] >> 2;
      // dK/dV: Q and dO of query head hkv * G + it / n_list; dQ: K and V
      // of the query head's K/V head
      const int head = DKDV ? hq_or_hkv * G + it / n_list : hq_or_hkv / G;
      uint8_t* dst = smem + C::kOffT + s * 2 * C::kTileBytes;
      mbar_arrive_expect_tx(&bars->t_full[s], 2 * C::kTileBytes);
      for (int kb = 0; kb < C::kKBlocks; ++kb) {
        tma_load_4d(DKDV ? tq : tk, &bars->t_full[s], dst + kb * kTileM * 128,
                    kb * 64, tile * kTileM, head, b, pol_stream);
        tma_load_4d(DKDV ? tdo : tv, &bars->t_full[s],
                    dst + C::kTileBytes + kb * kTileM * 128, kb * 64,
                    tile * kTileM, head, b, pol_stream);
      }
    }
    ++issued;
  }
  __syncwarp();
  // Drain: the loads already issued land before the CTA exits.
  if (lane == 0) {
    if (!mbar_wait_drain(&bars->f_full, 0, p.timeout_ns) && ok)
      record_bwd_timeout(kRoleBLoad, 1);
    for (int s = 0; s < 2; ++s) {
      const uint32_t n = issued > static_cast<uint32_t>(s)
                             ? (issued - 1 - s) / 2 + 1 : 0;
      if (n > 0 && !mbar_wait_drain(&bars->t_full[s], (n - 1) & 1,
                                    p.timeout_ns) && ok)
        record_bwd_timeout(kRoleBLoad, 2);
    }
  }
  __syncwarp();
}

template <int D, bool DKDV>
__device__ __forceinline__ void bwd_mma_role(const BwdParams& p, uint8_t* smem,
                                             BwdBars* bars, uint32_t tmem,
                                             int n_iter) {
  using C = BwdCfg<D>;
  const bool leader = (threadIdx.x % 32) == 0;
  volatile int* abort_flag = &bars->abort;
  constexpr uint32_t idesc_s = idesc_bf16_f32(kTileM, kTileN, false);
  constexpr uint32_t idesc_acc = idesc_bf16_f32(kTileM, D, true);
  constexpr uint32_t kTileUnits = C::kTileBytes >> 4;
  // K-major descriptors of the fixed tiles (A) and the ring (B), and the
  // MN-major form of the ring's tiles for the accumulating products
  const uint64_t da = sdesc_sw128(smem_u32(smem + C::kOffF), 16, 1024);
  const uint64_t db = sdesc_sw128(smem_u32(smem + C::kOffT), 16, 1024);
  const uint64_t dbm =
      sdesc_sw128(smem_u32(smem + C::kOffT), kTileN * 128, 1024);
  const uint32_t t_s = tmem, t_dp = tmem + 128;
  const uint32_t t_acc0 = tmem + 256, t_acc1 = tmem + 384;
  // S = F0 T0^T and dP = F1 T1^T of step `it` from ring slot it & 1
  auto issue_s = [&](int it) {
    const uint64_t t0 = db + (it & 1) * 2 * kTileUnits;
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k >> 2) * (kTileM * 128 / 16) + (k & 3) * 2;
      mma_ss_elect(t_s, da + off, t0 + off, idesc_s, k > 0 ? 1u : 0u);
    }
    mma_commit_elect(&bars->s_full);
  };
  auto issue_dp = [&](int it) {
    const uint64_t t1 = db + (it & 1) * 2 * kTileUnits + kTileUnits;
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k >> 2) * (kTileM * 128 / 16) + (k & 3) * 2;
      mma_ss_elect(t_dp, da + kTileUnits + off, t1 + off, idesc_s,
                   k > 0 ? 1u : 0u);
    }
    mma_commit_elect(&bars->dp_full);
  };
  // Per step: once P is stored (dK/dV) or S has been read (dQ), dV += P T1
  // and the next step's S go in; once dS is stored, dK += dS T0 (dQ += dS
  // T0) and the next step's dP.  The next S and dP overwrite the TMEM
  // columns that P and dS occupy; tcgen05 MMAs of one thread run in issue
  // order, so they come after the products that read them, and the
  // elementwise warps work on the next S while dS, dK and dP are in flight.
  bool ok = bwarp_wait(&bars->f_full, 0, abort_flag, p.timeout_ns);
  if (!ok && leader) record_bwd_timeout(kRoleBMma, 0);
  if (ok && n_iter > 0) {
    ok = bwarp_wait(&bars->t_full[0], 0, abort_flag, p.timeout_ns);
    if (!ok && leader) record_bwd_timeout(kRoleBMma, 1);
    if (ok) {
      tc_fence_after();
      issue_s(0);
      issue_dp(0);
    }
  }
  for (int it = 0; ok && it < n_iter; ++it) {
    const int s = it & 1;
    const uint64_t m0 = dbm + s * 2 * kTileUnits;  // T0 read MN-major
    const uint64_t m1 = m0 + kTileUnits;           // T1 read MN-major
    const uint32_t first = it == 0 ? 0u : 1u;
    ok = bwarp_wait(&bars->p_ready, it & 1, abort_flag, p.timeout_ns);
    if (!ok) {
      if (leader) record_bwd_timeout(kRoleBMma, 2);
      break;
    }
    tc_fence_after();
    // bf16 A from TMEM: rows 16kk..16kk+15 of the K dimension in columns
    // 8kk..8kk+7
    if (DKDV) {
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)  // dV += P T1
        mma_ts_elect(t_acc0, t_s + kk * 8, m1 + kk * (16 * 128 / 16),
                     idesc_acc, (kk > 0 || first) ? 1u : 0u);
    }
    const bool more = it + 1 < n_iter;
    if (more) {
      ok = bwarp_wait(&bars->t_full[(it + 1) & 1], ((it + 1) >> 1) & 1,
                      abort_flag, p.timeout_ns);
      if (!ok) {
        if (leader) record_bwd_timeout(kRoleBMma, 1);
        break;
      }
      tc_fence_after();
      issue_s(it + 1);
    }
    ok = bwarp_wait(&bars->ds_ready, it & 1, abort_flag, p.timeout_ns);
    if (!ok) {
      if (leader) record_bwd_timeout(kRoleBMma, 4);
      break;
    }
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < kTileN / 16; ++kk)  // dK (or dQ) += dS T0
      mma_ts_elect(DKDV ? t_acc1 : t_acc0, t_dp + kk * 8,
                   m0 + kk * (16 * 128 / 16), idesc_acc,
                   (kk > 0 || first) ? 1u : 0u);
    mma_commit_elect(&bars->t_empty[s]);
    if (more) issue_dp(it + 1);
  }
  __syncwarp();
  mma_commit_elect(&bars->acc_done);
  mma_commit_elect(&bars->mma_done);
  if (leader && !mbar_wait_drain(&bars->mma_done, 0, p.timeout_ns) && ok)
    record_bwd_timeout(kRoleBMma, 3);
  __syncwarp();
}

// Elementwise warps: two per TMEM lane quarter (one thread per row of the
// fixed tiles), warps 2-5 taking columns [0, 64) of S and dP, warps 6-9
// columns [64, 128).  The packed P and dS of the second half go over
// columns [32, 64), which the first half reads: the second half writes only
// after the first half has read (h0_read).
template <int D, int SCORE, bool DKDV>
__device__ __forceinline__ void bwd_elem_role(const BwdParams& p,
                                              BwdBars* bars,
                                              const uint16_t* list,
                                              uint32_t tmem, int b,
                                              int hq_or_hkv, int fixed_tile,
                                              int n_iter) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4;  // TMEM lanes this warp may access
  const int half = (warp - 2) / 4;  // column half of S and dP
  const int r = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t t_s = tmem + lane_off, t_dp = tmem + lane_off + 128;
  volatile int* abort_flag = &bars->abort;
  const int G = p.H / p.Hkv;
  const int n_list = bars->n_list;
  const float kLog2e = 1.4426950408889634f;
  // the thread's row: a key (dK/dV) or a query (dQ)
  const int row = fixed_tile * kTileM + r;
  // the row's segment id (the thread's key or query)
  int row_seg = 0;
  if ((p.flags & BSM_MASK_SEGMENT) && (DKDV ? row < p.Skv : row < p.Sq))
    row_seg = DKDV ? p.kv_seg[static_cast<int64_t>(b) * p.Skv + row]
                   : p.q_seg[static_cast<int64_t>(b) * p.Sq + row];
  // dQ: the row's lse (log2 units) and D_q are fixed
  float lse2_row = 0.f, delta_row = 0.f;
  if (!DKDV && SCORE == BSM_SCORE_SOFTMAX && row < p.Sq) {
    const int64_t i = (static_cast<int64_t>(b) * p.H + hq_or_hkv) * p.Sq + row;
    lse2_row = p.lse[i] * kLog2e;
    delta_row = p.delta[i];
  }
  // dK/dV softmax: the lse (log2 units) and D_q of the step's query
  // columns, loaded a step ahead so that their latency hides behind the
  // current step
  auto load_stats = [&](int it, float (&l2)[2], float (&dl)[2]) {
    const int tile = list[it % n_list] >> 2;
    const int hd = hq_or_hkv * G + it / n_list;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int qc = tile * kTileM + half * 64 + c * 32 + lane;
      l2[c] = 0.f;
      dl[c] = 0.f;
      if (qc < p.Sq) {
        const int64_t i = (static_cast<int64_t>(b) * p.H + hd) * p.Sq + qc;
        l2[c] = p.lse[i] * kLog2e;
        dl[c] = p.delta[i];
      }
    }
  };
  constexpr bool kStats = DKDV && SCORE == BSM_SCORE_SOFTMAX;
  float lse2_n[2] = {0.f, 0.f}, delta_n[2] = {0.f, 0.f};
  if (kStats && n_iter > 0) load_stats(0, lse2_n, delta_n);
  bool ok = true;
  for (int it = 0; it < n_iter; ++it) {
    const int e = it % n_list;
    const int tile = list[e] >> 2, cls = list[e] & 3;
    const int col0 = tile * kTileM + half * 64;  // first column of the half
    float lse2_c[2] = {lse2_n[0], lse2_n[1]}, delta_c[2] = {delta_n[0], delta_n[1]};
    if (kStats && it + 1 < n_iter) load_stats(it + 1, lse2_n, delta_n);
    ok = bwarp_wait(&bars->s_full, it & 1, abort_flag, p.timeout_ns);
    if (!ok) {
      record_bwd_timeout(kRoleBElem, 0);
      break;
    }
    tc_fence_after();
    uint32_t sraw[64];
    tmem_ld32(t_s + half * 64, sraw);
    tmem_ld32(t_s + half * 64 + 32, sraw + 32);
    // visibility of the half's 64 columns
    uint32_t vis[2] = {0xffffffffu, 0xffffffffu};
#pragma unroll
    for (int c = 0; c < 2; ++c)
      if (cls == 1) vis[c] = chunk_visible<DKDV>(p, b, row, row_seg, col0 + c * 32);
    tmem_ld_wait();
    tc_fence_before();
    if (!DKDV) mbar_arrive(&bars->p_ready);  // S read: the next S may go in
    else if (half == 0) mbar_arrive(&bars->h0_s);
    // P, and the per-element factor dS needs: softmax dS = P (dP - D_q),
    // pointwise dS = dP sig (1 + x (1 - sig)) / Sq
    float f[64];
    uint32_t pw[32];
#pragma unroll
    for (int j = 0; j < 64; j += 2) {
      float pv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = (j + u) >> 5, jj = (j + u) & 31;
        const float sv = __uint_as_float(sraw[j + u]);
        const bool v = (vis[c] >> jj) & 1u;
        if (SCORE == BSM_SCORE_SOFTMAX) {
          const float l2 = DKDV ? __shfl_sync(0xffffffffu, lse2_c[c], jj)
                                : lse2_row;
          const float pr = v ? ex2_approx(fmaf(sv, p.scale_log2, -l2)) : 0.f;
          pv[u] = pr;
          f[j + u] = pr;
        } else {
          const float x = sv * p.scale;
          const float sig = fmaf(0.5f, tanh_approx(0.5f * x), 0.5f);
          pv[u] = v ? x * sig * p.inv_sq : 0.f;
          f[j + u] = v ? sig * fmaf(x, 1.f - sig, 1.f) * p.inv_sq : 0.f;
        }
      }
      pw[j / 2] = pack_bf16x2(pv[0], pv[1]);
    }
    if (DKDV) {
      // P over S's columns: the half's 64 columns pack into columns
      // 32 * half .. 32 * half + 31; [32, 64) are the first half's S
      if (half == 1) {
        if (!bwarp_wait(&bars->h0_s, it & 1, abort_flag, p.timeout_ns)) {
          record_bwd_timeout(kRoleBElem, 2);
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st32(t_s + half * 32, pw);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_ready);
    }
    ok = bwarp_wait(&bars->dp_full, it & 1, abort_flag, p.timeout_ns);
    if (!ok) {
      record_bwd_timeout(kRoleBElem, 3);
      break;
    }
    tc_fence_after();
    uint32_t dpraw[64];
    tmem_ld32(t_dp + half * 64, dpraw);
    tmem_ld32(t_dp + half * 64 + 32, dpraw + 32);
    tmem_ld_wait();
    if (half == 0) {
      tc_fence_before();
      mbar_arrive(&bars->h0_dp);
    }
    uint32_t dsw[32];
#pragma unroll
    for (int j = 0; j < 64; j += 2) {
      float dsv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float dpv = __uint_as_float(dpraw[j + u]);
        if (SCORE == BSM_SCORE_SOFTMAX) {
          const int c = (j + u) >> 5, jj = (j + u) & 31;
          const float dl = DKDV ? __shfl_sync(0xffffffffu, delta_c[c], jj)
                                : delta_row;
          dsv[u] = f[j + u] * (dpv - dl);
        } else {
          dsv[u] = dpv * f[j + u];
        }
      }
      dsw[j / 2] = pack_bf16x2(dsv[0], dsv[1]);
    }
    if (half == 1) {  // columns [32, 64) of dP are the first half's input
      if (!bwarp_wait(&bars->h0_dp, it & 1, abort_flag, p.timeout_ns)) {
        record_bwd_timeout(kRoleBElem, 2);
        ok = false;
        break;
      }
      tc_fence_after();
    }
    tmem_st32(t_dp + half * 32, dsw);
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&bars->ds_ready);
  }
  if (!ok) return;
  // ---- results: dK/dV rows (keys) or dQ rows, bf16; dK and dQ scaled;
  // each half stores half of the D columns
  const bool row_ok = DKDV ? row < p.Skv : row < p.Sq;
  if (n_iter > 0) {
    if (!bwarp_wait(&bars->acc_done, 0, abort_flag, p.timeout_ns)) {
      record_bwd_timeout(kRoleBElem, 1);
      return;
    }
    tc_fence_after();
  }
#pragma unroll 1
  for (int a = 0; a < (DKDV ? 2 : 1); ++a) {
    // dK/dV: a = 0 is dV (TMEM 256), a = 1 dK (TMEM 384); dQ: a = 0
    uint16_t* dst;
    float mul;
    if (DKDV) {
      dst = (a == 0 ? p.dv : p.dk) +
            static_cast<int64_t>(b) * (a == 0 ? p.dv_sb : p.dk_sb) +
            static_cast<int64_t>(hq_or_hkv) * (a == 0 ? p.dv_sh : p.dk_sh) +
            static_cast<int64_t>(row) * (a == 0 ? p.dv_ss : p.dk_ss);
      mul = a == 0 ? 1.f : p.scale;
    } else {
      dst = p.dq + static_cast<int64_t>(b) * p.dq_sb +
            static_cast<int64_t>(hq_or_hkv) * p.dq_sh +
            static_cast<int64_t>(row) * p.dq_ss;
      mul = p.scale;
    }
#pragma unroll 1
    for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
      uint32_t o[32];
      if (n_iter > 0) {
        tmem_ld32(tmem + lane_off + 256 + a * 128 + c * 32, o);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = 0u;
      }
      if (row_ok) {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          w[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * mul,
                             __uint_as_float(o[2 * j + 1]) * mul);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          st_global_v4(dst + c * 32 + v * 8, w[4 * v], w[4 * v + 1],
                       w[4 * v + 2], w[4 * v + 3]);
      }
    }
  }
}

template <int D, int SCORE, bool DKDV>
__global__ void __launch_bounds__(kBwdThreads, 1)
    splash_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_do,
                      const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kOffBar);
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + C::kOffList);
  const int warp = threadIdx.x / 32;
  // grid: (tile, head, batch); dK/dV: key tile and K/V head; dQ: query tile
  // and query head.  Blocks start in linear order.  Under a causal mask
  // (without a window) a walk is longest for the first key tiles (dK/dV)
  // and the last query tiles (dQ), so the linear index is dealt out in
  // bands of kBwdBand tiles, longest band first, every (head, batch) of a
  // band before the next band: long walks start early, and the CTAs in
  // flight still share a few heads' tiles in L2.
  int fixed_tile = blockIdx.x, head = blockIdx.y, b = blockIdx.z;
  if ((p.flags & BSM_MASK_CAUSAL) &&
      !(p.flags & (BSM_MASK_LOCAL | BSM_MASK_BAND))) {
    const int X = gridDim.x, G = gridDim.y * gridDim.z;
    const int lin = blockIdx.x + X * (blockIdx.y + gridDim.y * blockIdx.z);
    const int band = lin / (kBwdBand * G);
    const int width = min(kBwdBand, X - band * kBwdBand);
    const int within = lin - band * kBwdBand * G;
    const int g = within / width, k = within - g * width;
    const int rank = band * kBwdBand + k;  // 0 = the longest walk
    fixed_tile = DKDV ? rank : X - 1 - rank;
    head = g % gridDim.y;
    b = g / gridDim.y;
  }
  const int table = (p.flags & BSM_MASK_SEGMENT) ? b : 0;
  // The dQ grid reads nothing the dK/dV grid writes, so it is launched as
  // its programmatic dependent: once every dK/dV CTA has started, dQ CTAs
  // take the SMs the dK/dV grid's last CTAs leave.
  if (DKDV && threadIdx.x == 0)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    mbar_init(&bars->f_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->t_full[s], 1);
      mbar_init(&bars->t_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, 256);
    mbar_init(&bars->ds_ready, 256);
    mbar_init(&bars->h0_s, 128);
    mbar_init(&bars->h0_dp, 128);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 0) {
    const int n = build_bwd_list<DKDV>(p, table, fixed_tile, list);
    if (threadIdx.x == 0) bars->n_list = n;
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int n_iter = bars->n_list * (DKDV ? p.H / p.Hkv : 1);

  if (warp == 0) {
    if (n_iter > 0)
      bwd_load_role<D, DKDV>(p, &tm_q, &tm_k, &tm_v, &tm_do, smem, bars, list,
                             b, head, fixed_tile, n_iter);
  } else if (warp == 1) {
    if (n_iter > 0) bwd_mma_role<D, DKDV>(p, smem, bars, tmem, n_iter);
  } else {
    bwd_elem_role<D, SCORE, DKDV>(p, bars, list, tmem, b, head, fixed_tile,
                                  n_iter);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kBwdTmemCols);
  // a dQ grid ends only after the dK/dV grid it overlapped, so work queued
  // after the backward on the stream sees both
  if (!DKDV && threadIdx.x == 0)
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// D_q = sum_d dO[q, d] * out[q, d]: D / 8 threads per (batch, head, row),
// each with one 16-byte load of out and of dO (rows and strides are 16-byte
// aligned), a warp covering 32 / (D / 8) rows per pass of a grid-stride
// loop.
__global__ void __launch_bounds__(256) bwd_delta_kernel(const BwdParams p) {
  const int gs = p.D / 8;  // threads per row: 16 (D = 128) or 8 (D = 64)
  const int lane = threadIdx.x % 32, sub = lane % gs;
  const int rpw = 32 / gs;  // rows per warp and pass
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.Sq;
  const int64_t warp0 =
      (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * blockDim.x / 32;
#pragma unroll 2
  for (int64_t base = warp0 * rpw; base < rows; base += nwarps * rpw) {
    const int64_t r = base + lane / gs;
    float acc = 0.f;
    if (r < rows) {
      const int q = static_cast<int>(r % p.Sq);
      const int64_t bh = r / p.Sq;
      const int h = static_cast<int>(bh % p.H), b = static_cast<int>(bh / p.H);
      const uint4 ov = __ldg(reinterpret_cast<const uint4*>(
          p.out + b * p.o_sb + h * p.o_sh + q * p.o_ss + sub * 8));
      const uint4 dv = __ldg(reinterpret_cast<const uint4*>(
          p.dout + b * p.do_sb + h * p.do_sh + q * p.do_ss + sub * 8));
      const uint32_t o4[4] = {ov.x, ov.y, ov.z, ov.w};
      const uint32_t d4[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc = fmaf(__uint_as_float(o4[i] << 16), __uint_as_float(d4[i] << 16),
                   acc);
        acc = fmaf(__uint_as_float(o4[i] & 0xffff0000u),
                   __uint_as_float(d4[i] & 0xffff0000u), acc);
      }
    }
    for (int s = gs / 2; s > 0; s >>= 1)
      acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (r < rows && sub == 0) p.delta[r] = acc;
  }
}

template <int D, int SCORE, bool DKDV>
cudaError_t launch_bwd_one(const BwdParams& p, const CUtensorMap& tq,
                           const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, cudaStream_t stream) {
  using C = BwdCfg<D>;
  auto kern = splash_bwd_kernel<D, SCORE, DKDV>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid = DKDV ? dim3((p.Skv + kTileN - 1) / kTileN, p.Hkv, p.B)
                         : dim3((p.Sq + kTileM - 1) / kTileM, p.H, p.B);
  if (DKDV) {
    kern<<<grid, kBwdThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, p);
    return cudaGetLastError();
  }
  // dQ: a programmatic dependent of the launch before it (the dK/dV grid,
  // which lets it start early; or D_q's, which does not, so dQ then starts
  // after it as usual)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, p);
}

template <int D, int SCORE>
cudaError_t launch_bwd_d(const BwdParams& p, const CUtensorMap& tq,
                         const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (p.Skv > 0) e = launch_bwd_one<D, SCORE, true>(p, tq, tk, tv, tdo, stream);
  if (e != cudaSuccess) return e;
  if (p.Sq > 0) e = launch_bwd_one<D, SCORE, false>(p, tq, tk, tv, tdo, stream);
  return e;
}

}  // namespace

cudaError_t launch_splash_bwd(const BwdParams& p, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, cudaStream_t stream) {
  cudaError_t e;
  if (p.score == BSM_SCORE_SOFTMAX) {
    const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.Sq;
    if (rows > 0) {
      int dev = 0, sms = 0;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      const int64_t need = (rows * (p.D / 8) + 255) / 256;
      const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 8;
      bwd_delta_kernel<<<static_cast<unsigned>(need < cap ? need : cap), 256,
                         0, stream>>>(p);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  const bool pw = p.score == BSM_SCORE_POINTWISE;
  if (p.D == 128)
    return pw ? launch_bwd_d<128, BSM_SCORE_POINTWISE>(p, tq, tk, tv, tdo, stream)
              : launch_bwd_d<128, BSM_SCORE_SOFTMAX>(p, tq, tk, tv, tdo, stream);
  if (p.D == 64)
    return pw ? launch_bwd_d<64, BSM_SCORE_POINTWISE>(p, tq, tk, tv, tdo, stream)
              : launch_bwd_d<64, BSM_SCORE_SOFTMAX>(p, tq, tk, tv, tdo, stream);
  return cudaErrorInvalidValue;
}

cudaError_t read_bwd_error(int32_t out[4]) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_bwd_error, 4 * sizeof(int32_t));
  if (e != cudaSuccess) return e;
  const int32_t zero[4] = {0, 0, 0, 0};
  return cudaMemcpyToSymbol(g_bwd_error, zero, 4 * sizeof(int32_t));
}

}  // namespace bsm
