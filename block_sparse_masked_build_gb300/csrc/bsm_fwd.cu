// Block-sparse masked attention forward for sm_103a (GB300).
//
// One persistent CTA per SM walks work units of (batch, head, 256 query
// rows).  A unit is two 128-row query tiles that share one stream of
// 128-key KV tiles: the union of the nonzero blocks of both tiles, read from
// the mask-info block classes (hstu_ops `_next_nonzero`: 0 empty, 1
// partial, 2 full).  Empty KV tiles are never loaded (splash notes section
// 21); the element mask is evaluated on partial tiles only.
//
// Warp roles (320 threads):
//   warp 0      builds the unit's KV-tile list in shared memory, then issues
//               TMA loads: Q once per unit, K and V tiles through a ring of
//               shared-memory slots (128-byte swizzle).
//   warp 1      allocates the 512 TMEM columns and, from one lane, issues the
//               tcgen05 MMAs: S_t = Q_t K^T (both operands in shared memory)
//               and O_t += P_t V (P_t read from TMEM, V from shared memory).
//   warps 2-5   score warpgroup of query tile 0, warps 6-9 of tile 1: one
//               thread per query row (its TMEM lane).  Softmax: online
//               max/sum with the correction of the splash notes section 15
//               (O is rescaled in TMEM only when the running max grew by more
//               than 2^8, which leaves the final O / l exact).  Pointwise:
//               x * sigmoid(x) / Sq with x = scale * q.k, masked -> 0
//               (hstu_ops fwd kernel).  P goes back to TMEM as bf16 over S.
// TMEM: S0/P0 cols [0,128), S1/P1 [128,256), O0 [256,256+D), O1 [384,384+D).
#include <cstdint>

#include "bsm_internal.h"
#include "bsm_ptx.cuh"

namespace bsm {

// Error record: [0] code (1 = wait timed out), [1] block, [2] role, [3] phase.
__device__ int g_fwd_error[4];

namespace {

constexpr int kThreads = 320;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr int kRoleLoad = 1, kRoleMma = 2, kRoleScore = 3;

template <int D>
struct Cfg {
  static constexpr int kKBlocks = D / 64;            // 128-byte k-blocks
  static constexpr int kTileBytes = kTileM * D * 2;  // Q, K or V tile
  static constexpr int kSlots = (D == 128) ? 4 : 8;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kTileBytes;
  static constexpr int kOffList = kOffKV + kSlots * kTileBytes;
  static constexpr int kOffBar = kOffList + 2 * kMaxKvTiles * 4;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;
};

struct Bars {
  uint64_t list_full[2], list_free[2];
  uint64_t q_full, q_empty;
  uint64_t kv_full[8], kv_empty[8];
  uint64_t s_full[2], p_full[2], pv_done[2], o_free[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int list_count[2];
  int list_unit[2];
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

__device__ __forceinline__ void record_timeout(int role, int phase) {
  if (atomicCAS(&g_fwd_error[0], 0, 1) == 0) {
    g_fwd_error[1] = blockIdx.x;
    g_fwd_error[2] = role;
    g_fwd_error[3] = phase;
  }
}

// Warp-wide bounded wait: every lane polls, and the outcome is made uniform
// so that no lane runs a .sync.aligned instruction its siblings skip.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag,
                                          uint64_t timeout_ns) {
  const bool ok = mbar_wait(bar, parity, abort_flag, timeout_ns);
  return __all_sync(0xffffffffu, ok);
}

struct UnitCoord {
  int b, h, st;
};

__device__ __forceinline__ UnitCoord decode_unit(const FwdParams& p, int u) {
  // Heaviest super-tiles first: under a causal mask the last rows see the
  // most keys.
  const int bh_count = p.B * p.H;
  UnitCoord c;
  c.st = p.n_super - 1 - u / bh_count;
  const int bh = u % bh_count;
  c.b = bh / p.H;
  c.h = bh % p.H;
  return c;
}

// Class of (128-row query tile starting at row R0) x (KV tile jt), combined
// from the mask-info blocks that cover it: 2 if all are full, 0 if all are
// empty, else 1.  A KV tile cut by the end of the keys is never full.
__device__ __forceinline__ int tile_class(const FwdParams& p, int table,
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

template <int D>
__device__ __forceinline__ void load_role(const FwdParams& p,
                                          const CUtensorMap* tq,
                                          const CUtensorMap* tk,
                                          const CUtensorMap* tv, uint8_t* smem,
                                          Bars* bars, uint32_t* lists) {
  using C = Cfg<D>;
  const int lane = threadIdx.x % 32;
  volatile int* abort_flag = &bars->abort;
  const uint64_t pol_q = l2_policy_evict_first();
  const uint64_t pol_kv = l2_policy_evict_last();
  uint32_t kv_it = 0, q_it = 0;
  int ui = 0;
  for (int unit = blockIdx.x; unit < p.num_units; unit += gridDim.x, ++ui) {
    const int buf = ui & 1;
    if (!warp_wait(&bars->list_free[buf], ((ui >> 1) & 1) ^ 1, abort_flag,
                   p.timeout_ns)) {
      if (lane == 0) record_timeout(kRoleLoad, 0);
      break;
    }
    const UnitCoord uc = decode_unit(p, unit);
    const int table = (p.flags & BSM_MASK_SEGMENT) ? uc.b : 0;
    const int row0 = uc.st * kUnitRows;
    uint32_t* list = lists + buf * kMaxKvTiles;
    int n = 0;
    for (int base = 0; base < p.n_kvtiles; base += 32) {
      const int jt = base + lane;
      int c0 = 0, c1 = 0;
      if (jt < p.n_kvtiles) {
        c0 = tile_class(p, table, row0, jt);
        c1 = tile_class(p, table, row0 + kTileM, jt);
      }
      const bool nz = (c0 | c1) != 0;
      const unsigned m = __ballot_sync(0xffffffffu, nz);
      if (nz) {
        list[n + __popc(m & ((1u << lane) - 1u))] =
            (static_cast<uint32_t>(jt) << 4) | (c0 << 2) | c1;
      }
      n += __popc(m);
    }
    __syncwarp();
    if (lane == 0) {
      bars->list_count[buf] = n;
      bars->list_unit[buf] = unit;
      mbar_arrive(&bars->list_full[buf]);
    }
    if (lane == 0 && n > 0) {
      bool ok = mbar_wait(&bars->q_empty, (q_it & 1) ^ 1, abort_flag,
                          p.timeout_ns);
      if (!ok) {
        record_timeout(kRoleLoad, 1);
      } else {
        const int nt = (row0 + kTileM < p.Sq) ? 2 : 1;
        mbar_arrive_expect_tx(&bars->q_full, nt * C::kTileBytes);
        for (int t = 0; t < nt; ++t)
          for (int kb = 0; kb < C::kKBlocks; ++kb)
            tma_load_4d(tq, &bars->q_full,
                        smem + C::kOffQ + t * C::kTileBytes + kb * kTileM * 128,
                        kb * 64, row0 + t * kTileM, uc.h, uc.b, pol_q);
        ++q_it;
        const int hkv = uc.h / (p.H / p.Hkv);
        for (int e = 0; e < n && ok; ++e) {
          const int jt = static_cast<int>(list[e] >> 4);
          for (int which = 0; which < 2 && ok; ++which) {
            const int slot = kv_it % C::kSlots;
            const uint32_t ph = (kv_it / C::kSlots) & 1;
            ok = mbar_wait(&bars->kv_empty[slot], ph ^ 1, abort_flag,
                           p.timeout_ns);
            if (!ok) {
              record_timeout(kRoleLoad, 2);
              break;
            }
            mbar_arrive_expect_tx(&bars->kv_full[slot], C::kTileBytes);
            uint8_t* dst = smem + C::kOffKV + slot * C::kTileBytes;
            for (int kb = 0; kb < C::kKBlocks; ++kb)
              tma_load_4d(which == 0 ? tk : tv, &bars->kv_full[slot],
                          dst + kb * kTileN * 128, kb * 64, jt * kTileN, hkv,
                          uc.b, pol_kv);
            ++kv_it;
          }
        }
      }
    }
    __syncwarp();
    if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
  }
}

template <int D>
__device__ __forceinline__ void mma_role(const FwdParams& p, uint8_t* smem,
                                         Bars* bars, const uint32_t* lists,
                                         uint32_t tmem) {
  using C = Cfg<D>;
  volatile int* abort_flag = &bars->abort;
  const uint32_t q_base = smem_u32(smem + C::kOffQ);
  const uint32_t kv_base = smem_u32(smem + C::kOffKV);
  constexpr uint32_t idesc_s = idesc_bf16_f32(kTileM, kTileN, false);
  constexpr uint32_t idesc_o = idesc_bf16_f32(kTileM, D, true);
  uint32_t kv_it = 0, q_it = 0;
  uint32_t s_cnt[2] = {0, 0}, pv_cnt[2] = {0, 0};
  int ui = 0;
  bool ok = true;
  for (int unit = blockIdx.x; unit < p.num_units && ok;
       unit += gridDim.x, ++ui) {
    const int buf = ui & 1;
    ok = mbar_wait(&bars->list_full[buf], (ui >> 1) & 1, abort_flag,
                   p.timeout_ns);
    if (!ok) {
      record_timeout(kRoleMma, 0);
      break;
    }
    const int n = bars->list_count[buf];
    const uint32_t* list = lists + buf * kMaxKvTiles;
    if (n > 0) {
      ok = mbar_wait(&bars->q_full, q_it & 1, abort_flag, p.timeout_ns);
      if (!ok) {
        record_timeout(kRoleMma, 1);
        break;
      }
      tc_fence_after();
      bool first_pv[2] = {true, true};
      for (int e = 0; e < n && ok; ++e) {
        const uint32_t ent = list[e];
        const int cls[2] = {static_cast<int>((ent >> 2) & 3u),
                            static_cast<int>(ent & 3u)};
        // ---- S_t = Q_t K^T
        const int kslot = kv_it % C::kSlots;
        ok = mbar_wait(&bars->kv_full[kslot], (kv_it / C::kSlots) & 1,
                       abort_flag, p.timeout_ns);
        if (!ok) {
          record_timeout(kRoleMma, 2);
          break;
        }
        ++kv_it;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!cls[t] || !ok) continue;
          if (pv_cnt[t] > 0) {  // P_t (aliasing S_t) consumed by the last PV
            ok = mbar_wait(&bars->pv_done[t], (pv_cnt[t] - 1) & 1, abort_flag,
                           p.timeout_ns);
            if (!ok) {
              record_timeout(kRoleMma, 3);
              break;
            }
            tc_fence_after();
          }
          const uint32_t a0 = q_base + t * C::kTileBytes;
          const uint32_t b0 = kv_base + kslot * C::kTileBytes;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * (kTileM * 128) + (k & 3) * 32;
            mma_ss(tmem + t * 128, sdesc_sw128(a0 + off, 16, 1024),
                   sdesc_sw128(b0 + off, 16, 1024), idesc_s, k > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[t]);
          ++s_cnt[t];
        }
        if (!ok) break;
        mma_commit(&bars->kv_empty[kslot]);
        // ---- O_t += P_t V
        const int vslot = kv_it % C::kSlots;
        ok = mbar_wait(&bars->kv_full[vslot], (kv_it / C::kSlots) & 1,
                       abort_flag, p.timeout_ns);
        if (!ok) {
          record_timeout(kRoleMma, 4);
          break;
        }
        ++kv_it;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!cls[t] || !ok) continue;
          ok = mbar_wait(&bars->p_full[t], (s_cnt[t] - 1) & 1, abort_flag,
                         p.timeout_ns);
          if (ok && first_pv[t])
            ok = mbar_wait(&bars->o_free[t], (ui & 1) ^ 1, abort_flag,
                           p.timeout_ns);
          if (!ok) {
            record_timeout(kRoleMma, 5);
            break;
          }
          tc_fence_after();
          const uint32_t b0 = kv_base + vslot * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk) {
            mma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8,
                   sdesc_sw128(b0 + kk * 16 * 128, kTileN * 128, 1024),
                   idesc_o, (first_pv[t] && kk == 0) ? 0u : 1u);
          }
          first_pv[t] = false;
          mma_commit(&bars->pv_done[t]);
          ++pv_cnt[t];
        }
        if (!ok) break;
        mma_commit(&bars->kv_empty[vslot]);
      }
      if (!ok) break;
      mma_commit(&bars->q_empty);
      ++q_it;
    }
    mbar_arrive(&bars->list_free[buf]);
  }
  // Drain: every MMA issued above has completed once this arrives.
  mma_commit(&bars->mma_done);
  if (!mbar_wait(&bars->mma_done, 0, abort_flag, p.timeout_ns) && ok)
    record_timeout(kRoleMma, 6);
}

// Element mask of a partial tile for one query row (hstu_ops `_apply_mask`:
// the computed causal/local predicate AND q_seg == kv_seg, with key indices
// taken from the true KV position of the tile, not its list position).
struct RowMask {
  int lo_c, hi_c;  // visible columns c of the tile satisfy lo_c <= c <= hi_c
  int segq;
  const int32_t* segk;  // kv segment ids of the tile's first key, or null
};

__device__ __forceinline__ RowMask row_mask(const FwdParams& p, int qrow, int b,
                                            int jt) {
  const int kbase = jt * kTileN;
  int hi_k = p.Skv - 1;
  int lo_k = 0;
  if (p.flags & BSM_MASK_CAUSAL) hi_k = min(hi_k, qrow);
  if (p.flags & BSM_MASK_LOCAL) lo_k = max(lo_k, qrow - p.window + 1);
  RowMask m;
  m.lo_c = lo_k - kbase;
  m.hi_c = hi_k - kbase;
  m.segq = 0;
  m.segk = nullptr;
  if (p.flags & BSM_MASK_SEGMENT) {
    m.segk = p.kv_seg + static_cast<int64_t>(b) * p.Skv + kbase;
  }
  return m;
}

// Visibility of the 4 columns c..c+3 as bits (segment ids read 4 at a time;
// the last KV tile is only read below hi_c, which stays inside the keys).
__device__ __forceinline__ uint32_t vis4(const RowMask& m, int c) {
  uint32_t bits = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    bits |= ((c + u >= m.lo_c) && (c + u <= m.hi_c)) ? (1u << u) : 0u;
  if (m.segk != nullptr && bits) {
    int4 s;
    if (c + 3 <= m.hi_c &&
        (reinterpret_cast<uintptr_t>(m.segk + c) & 15u) == 0) {
      s = __ldg(reinterpret_cast<const int4*>(m.segk + c));
    } else {
      s.x = m.segk[c];
      s.y = (c + 1 <= m.hi_c) ? m.segk[c + 1] : 0;
      s.z = (c + 2 <= m.hi_c) ? m.segk[c + 2] : 0;
      s.w = (c + 3 <= m.hi_c) ? m.segk[c + 3] : 0;
    }
    bits &= (s.x == m.segq ? 1u : 0u) | (s.y == m.segq ? 2u : 0u) |
            (s.z == m.segq ? 4u : 0u) | (s.w == m.segq ? 8u : 0u);
  }
  return bits;
}

template <int D, int SCORE>
__device__ __forceinline__ void score_role(const FwdParams& p, Bars* bars,
                                           const uint32_t* lists,
                                           uint32_t tmem) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = (warp - 2) / 4;  // query tile of this warpgroup
  const int quarter = warp % 4;  // TMEM lane quarter this warp may access
  const int r = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t s_addr = tmem + lane_off + t * 128;
  const uint32_t o_addr = tmem + lane_off + 256 + t * 128;
  volatile int* abort_flag = &bars->abort;
  const float NEG_INF = __int_as_float(0xff800000);
  uint32_t s_cnt = 0, pv_cnt = 0;
  int ui = 0;
  for (int unit = blockIdx.x; unit < p.num_units; unit += gridDim.x, ++ui) {
    const int buf = ui & 1;
    if (!warp_wait(&bars->list_full[buf], (ui >> 1) & 1, abort_flag,
                   p.timeout_ns)) {
      record_timeout(kRoleScore, 0);
      break;
    }
    const int n = bars->list_count[buf];
    const UnitCoord uc = decode_unit(p, bars->list_unit[buf]);
    const uint32_t* list = lists + buf * kMaxKvTiles;
    const int qrow = uc.st * kUnitRows + t * kTileM + r;
    int segq = 0;
    if ((p.flags & BSM_MASK_SEGMENT) && qrow < p.Sq)
      segq = p.q_seg[static_cast<int64_t>(uc.b) * p.Sq + qrow];
    float m_used = NEG_INF, l_sum = 0.f;
    uint32_t unit_pv = 0;
    bool ok = true;
    for (int e = 0; e < n; ++e) {
      const uint32_t ent = list[e];
      const int cls = t == 0 ? static_cast<int>((ent >> 2) & 3u)
                             : static_cast<int>(ent & 3u);
      if (!cls) continue;
      const int jt = static_cast<int>(ent >> 4);
      ok = warp_wait(&bars->s_full[t], s_cnt & 1, abort_flag, p.timeout_ns);
      if (!ok) {
        record_timeout(kRoleScore, 1);
        break;
      }
      ++s_cnt;
      tc_fence_after();
      uint32_t sraw[kTileN];
#pragma unroll
      for (int q = 0; q < kTileN / 32; ++q) tmem_ld32(s_addr + q * 32, sraw + q * 32);
      tmem_ld_wait();
      float* s = reinterpret_cast<float*>(sraw);

      uint32_t pk[kTileN / 2];
      if (SCORE == BSM_SCORE_SOFTMAX) {
        if (cls == 1) {
          RowMask mk = row_mask(p, qrow, uc.b, jt);
          mk.segq = segq;
#pragma unroll
          for (int c = 0; c < kTileN; c += 4) {
            const uint32_t bits = vis4(mk, c);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (!(bits & (1u << u))) s[c + u] = NEG_INF;
          }
        }
        float mx = s[0];
#pragma unroll
        for (int c = 1; c < kTileN; ++c) mx = fmaxf(mx, s[c]);
        const float m_blk = mx * p.scale_log2;
        bool rescale = false;
        float alpha = 1.f;
        if (m_blk > m_used + kRescaleLog2) {
          if (m_used != NEG_INF) {
            alpha = ex2_approx(m_used - m_blk);
            rescale = true;
          }
          l_sum *= alpha;
          m_used = m_blk;
        }
        const float neg_m = (m_used == NEG_INF) ? 0.f : -m_used;
        float lsum = 0.f;
#pragma unroll
        for (int c = 0; c < kTileN; c += 2) {
          const float p0 = ex2_approx(fmaf(s[c], p.scale_log2, neg_m));
          const float p1 = ex2_approx(fmaf(s[c + 1], p.scale_log2, neg_m));
          lsum += p0 + p1;
          pk[c / 2] = pack_bf16x2(p0, p1);
        }
        l_sum += lsum;
#pragma unroll
        for (int q = 0; q < kTileN / 32; ++q) tmem_st16(s_addr + q * 16, pk + q * 16);
        // Rescale O_t (needs the previous PV of this tile to have landed).
        if (__any_sync(0xffffffffu, rescale) && unit_pv > 0) {
          ok = warp_wait(&bars->pv_done[t], (pv_cnt - 1) & 1, abort_flag,
                         p.timeout_ns);
          if (!ok) {
            record_timeout(kRoleScore, 2);
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            tmem_ld32(o_addr + q * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c)
              o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(o_addr + q * 32, o);
          }
        }
      } else {
        // pointwise: x = scale*qk; p = x*sigmoid(x)/Sq; masked -> 0
        RowMask mk;
        if (cls == 1) {
          mk = row_mask(p, qrow, uc.b, jt);
          mk.segq = segq;
        }
#pragma unroll
        for (int c = 0; c < kTileN; c += 4) {
          const uint32_t bits = (cls == 1) ? vis4(mk, c) : 0xfu;
          float pv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float x = s[c + u] * p.scale;
            const float sg = rcp_approx(1.f + ex2_approx(-1.4426950408889634f * x));
            pv[u] = (bits & (1u << u)) ? x * sg * p.inv_sq : 0.f;
          }
          pk[c / 2] = pack_bf16x2(pv[0], pv[1]);
          pk[c / 2 + 1] = pack_bf16x2(pv[2], pv[3]);
        }
#pragma unroll
        for (int q = 0; q < kTileN / 32; ++q) tmem_st16(s_addr + q * 16, pk + q * 16);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_full[t]);
      ++pv_cnt;
      ++unit_pv;
    }
    if (!ok) break;

    // ---- epilogue: out = O / l (softmax) or O (pointwise), bf16
    const bool row_ok = qrow < p.Sq;
    uint16_t* orow = p.out + static_cast<int64_t>(uc.b) * p.o_sb +
                     static_cast<int64_t>(uc.h) * p.o_sh +
                     static_cast<int64_t>(qrow) * p.o_ss;
    if (unit_pv > 0) {
      if (!warp_wait(&bars->pv_done[t], (pv_cnt - 1) & 1, abort_flag,
                     p.timeout_ns)) {
        record_timeout(kRoleScore, 3);
        break;
      }
      tc_fence_after();
      float inv = 1.f;
      if (SCORE == BSM_SCORE_SOFTMAX) inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
#pragma unroll 1
      for (int q = 0; q < D / 32; ++q) {
        uint32_t o[32];
        tmem_ld32(o_addr + q * 32, o);
        tmem_ld_wait();
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv,
                             __uint_as_float(o[2 * c + 1]) * inv);
        if (row_ok) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st_global_v4(orow + q * 32 + v * 8, w[4 * v], w[4 * v + 1],
                         w[4 * v + 2], w[4 * v + 3]);
        }
      }
    } else if (row_ok) {
#pragma unroll
      for (int v = 0; v < D / 8; ++v) st_global_v4(orow + v * 8, 0u, 0u, 0u, 0u);
    }
    if (SCORE == BSM_SCORE_SOFTMAX && p.lse != nullptr && row_ok) {
      const float lse = l_sum > 0.f
                            ? (m_used + log2f(l_sum)) * 0.6931471805599453f
                            : NEG_INF;
      p.lse[(static_cast<int64_t>(uc.b) * p.H + uc.h) * p.Sq + qrow] = lse;
    }
    tc_fence_before();
    mbar_arrive(&bars->o_free[t]);
    mbar_arrive(&bars->list_free[buf]);
  }
}

template <int D, int SCORE>
__global__ void __launch_bounds__(kThreads, 1)
    splash_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);
  uint32_t* lists = reinterpret_cast<uint32_t*>(smem + C::kOffList);
  const int warp = threadIdx.x / 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->list_full[i], 1);
      mbar_init(&bars->list_free[i], 1 + 2 * kTileM);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], kTileM);
      mbar_init(&bars->pv_done[i], 1);
      mbar_init(&bars->o_free[i], kTileM);
    }
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    load_role<D>(p, &tm_q, &tm_k, &tm_v, smem, bars, lists);
  } else if (warp == 1) {
    if ((threadIdx.x % 32) == 0) mma_role<D>(p, smem, bars, lists, tmem);
    __syncwarp();
  } else {
    score_role<D, SCORE>(p, bars, lists, tmem);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int D, int SCORE>
cudaError_t launch_one(const FwdParams& p, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv,
                       int num_sms, cudaStream_t stream) {
  using C = Cfg<D>;
  auto kern = splash_fwd_kernel<D, SCORE>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = p.num_units < num_sms ? p.num_units : num_sms;
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

// Self test of the bounded wait: nothing ever arrives on this barrier.
__global__ void wait_selftest_kernel(uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&bar, 0, &abort_flag, timeout_ns)) record_timeout(0, 7);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_splash_fwd(const FwdParams& p, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv,
                              int num_sms, cudaStream_t stream) {
  const bool pw = p.score == BSM_SCORE_POINTWISE;
  if (p.D == 128)
    return pw ? launch_one<128, BSM_SCORE_POINTWISE>(p, tq, tk, tv, num_sms, stream)
              : launch_one<128, BSM_SCORE_SOFTMAX>(p, tq, tk, tv, num_sms, stream);
  if (p.D == 64)
    return pw ? launch_one<64, BSM_SCORE_POINTWISE>(p, tq, tk, tv, num_sms, stream)
              : launch_one<64, BSM_SCORE_SOFTMAX>(p, tq, tk, tv, num_sms, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns);
  return cudaGetLastError();
}

cudaError_t read_device_error(int32_t out[4], cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_fwd_error, 4 * sizeof(int32_t));
  if (e != cudaSuccess) return e;
  const int32_t zero[4] = {0, 0, 0, 0};
  return cudaMemcpyToSymbol(g_fwd_error, zero, 4 * sizeof(int32_t));
}

}  // namespace bsm
