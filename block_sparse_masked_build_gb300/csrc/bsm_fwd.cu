// Block-sparse masked attention forward for sm_103a (GB300).  Two kernels:
// the lockstep one described here, and, at head dim 128 for packed
// sequences (segment ids) and for any mask below 4096 keys, a variant whose
// two query tiles run as independent pipelines (see "Decoupled query
// tiles" below).
//
// One persistent CTA per SM takes work units of (batch, head, 256 query
// rows) from a counter in the caller's workspace, longest units first.  A
// unit is two 128-row query tiles that share one stream of
// 128-key KV tiles: the union of the nonzero blocks of both tiles, read from
// the mask-info block classes (hstu_ops `_next_nonzero`: 0 empty, 1
// partial, 2 full).  Empty KV tiles are never loaded (splash notes section
// 21); the element mask is evaluated on partial tiles only.
//
// Warp roles (384 threads, three warpgroups; the first gives registers to
// the other two with setmaxnreg):
//   warp 3      takes work units from the counter and builds each unit's
//               KV-tile list, up to two units ahead (three list buffers).
//   warp 0      issues TMA loads: Q per query tile, K and V tiles through a
//               ring of shared-memory slots (128-byte swizzle).
//   warps 1,2   one MMA issuer per query tile (warp 1 also allocates the 512
//               TMEM columns): the whole warp waits and issues, each
//               tcgen05 MMA going out from the lane elect.sync picks:
//               S_t = Q_t K^T (both operands in shared memory) and
//               O_t += P_t V (P_t read from TMEM, V from shared memory).
//   warps 4-7   score warpgroup of query tile 0, warps 8-11 of tile 1: one
//               thread per query row (its TMEM lane).  Softmax: online
//               max/sum with the correction of the splash notes section 15
//               (O is rescaled in TMEM only when the running max grew by more
//               than 2^8, which leaves the final O / l exact).  Pointwise:
//               x * sigmoid(x) / Sq with x = scale * q.k, masked -> 0
//               (hstu_ops fwd kernel).  P goes back to TMEM as bf16 over S.
//               In the instance used for long units without segment ids
//               the two score warps of each SM sub-partition take their
//               softmax turns alternately (see score_role).
// TMEM: S0/P0 cols [0,128), S1/P1 [128,256), O0 [256,256+D), O1 [384,384+D).
//
// Element mask of a partial tile (hstu_ops `_apply_mask`): each row's visible
// keys under causal / local / band masks -- and under segment ids when the kv
// ids are sorted, via the mask-info's per-row segment ranges -- are one
// interval, so the mask is a column-range test; unsorted segment ids are
// compared element by element and an arbitrary mask contributes its bits
// (both as per-column keep bits).  Key indices are the tile's true KV
// position.
#include <cstdint>

#include "bsm_internal.h"
#include "bsm_ptx.cuh"

namespace bsm {

// Error record: [0] code (1 = wait timed out), [1] block, [2] role, [3] phase.
__device__ int g_fwd_error[4];

namespace {

constexpr int kThreads = 384;
// Register split: warpgroup 0 (load, MMA, list) drops to kRegsLight per
// thread, the two score warpgroups rise to kRegsScore.  Their sum must stay
// within what the CTA was launched with (kThreads x the kernel's register
// count), which the launcher checks.
constexpr uint32_t kRegsLight = 80, kRegsScore = 208;
constexpr int kRegsNeeded = 128 * kRegsLight + 256 * kRegsScore;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kPingPongMin = 12;  // see score_role
// K/V ring slots at head dim 128, each holding one 128 x 128 K or V tile.
// Five (224 KB of shared memory with the two Q tiles) keep the long units'
// loads ahead of the alternating softmax turns; three were as fast on
// packed sequences but 9-12 % slower on long causal and local-window units.
constexpr int kSlots128 = 5;
constexpr uint32_t kTmemCols = 512;
constexpr int kRoleLoad = 1, kRoleMma = 2, kRoleScore = 3, kRoleList = 4;

template <int D>
struct Cfg {
  static constexpr int kKBlocks = D / 64;            // 128-byte k-blocks
  static constexpr int kTileBytes = kTileM * D * 2;  // Q, K or V tile
  static constexpr int kSlots = (D == 128) ? kSlots128 : 8;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kTileBytes;
  static constexpr int kOffBar = kOffKV + kSlots * kTileBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;
};
static_assert(Cfg<128>::kSmemBytes <= 232448, "shared memory budget");

struct ListMeta {
  int n;          // entries (KV tiles) of the unit
  int n_t[2];     // entries used by query tile t
  int last_t[2];  // index of the last entry used by query tile t (-1: none)
  int unit;
  int b, h, st;   // the unit's batch row, head and 256-row super-tile
};

struct Bars {
  uint64_t list_full[kListBufs], list_free[kListBufs];
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[8], kv_empty[8];  // up to 8 ring slots
  uint64_t s_full[2], p_full[2], pv_done[2], o_free[2];
  // softmax turn of each score warp: [query tile][TMEM lane quarter]
  uint64_t sm_turn[2][4];
  uint64_t mma_done[2];
  uint32_t tmem_base;
  int abort;
  uint32_t trace_n[6];
  ListMeta meta[kListBufs];
};
static_assert(sizeof(Bars) <= 512, "barrier block");

__device__ __forceinline__ void record_timeout(int role, int phase) {
  if (atomicCAS(&g_fwd_error[0], 0, 1) == 0) {
    g_fwd_error[1] = blockIdx.x;
    g_fwd_error[2] = role;
    g_fwd_error[3] = phase;
  }
}

// Optional event trace.  CTA c owns records [c*(cap+2), (c+1)*(cap+2)):
// records 0-1 hold the event counts of the six recording threads (uint32
// each: load, MMA tile 0, score tile 0, score tile 1, list, MMA tile 1), then
// come six equal regions, each written by one thread with a plain counter.  A record is
// {globaltimer ns, role<<28 | event<<24 | tile<<20 | entry, unit}.
struct TraceRec {
  uint64_t t;
  uint32_t a, b;
};
enum : uint32_t {
  kEvListBuilt = 1, kEvQIssued = 2, kEvMmaUnit = 3, kEvMmaLastPv = 4,
  kEvSFull = 5, kEvPFull = 6, kEvEpiBegin = 7, kEvEpiEnd = 8, kEvRescale = 9,
  kEvEpiPvLanded = 10, kEvSIssued = 11, kEvPReady = 12, kEvPVIssued = 13,
  kEvEpiOLoaded = 14, kEvTmaIssued = 15
};

__device__ __forceinline__ void trace(const FwdParams& p, Bars* bars,
                                      uint32_t role, uint32_t ev, uint32_t tile,
                                      uint32_t entry, uint32_t unit) {
  if (p.trace == nullptr) return;
  const uint32_t slot = role == kRoleScore ? 2 + tile
                        : role == kRoleMma   ? (tile == 0 ? 1 : 5)
                        : role == kRoleList  ? 4
                                             : 0;
  const uint32_t per = p.trace_cap / 6;
  const uint32_t i = bars->trace_n[slot]++;
  if (i < per) {
    TraceRec* r = reinterpret_cast<TraceRec*>(p.trace) +
                  static_cast<size_t>(blockIdx.x) * (p.trace_cap + 2) + 2 +
                  slot * per + i;
    r->t = globaltimer_ns();
    r->a = (role << 28) | (ev << 24) | (tile << 20) | (entry & 0xFFFFFu);
    r->b = unit;
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

// Work unit u -> (batch, head, super-tile).  Units come in groups that
// share one (mask table, super-tile) pair: all heads of that batch row with
// one table per batch row, else all batch rows and heads.  The pairs are
// taken longest first when the mask info carries that order; otherwise the
// last super-tiles go first (under a causal mask the last rows see the most
// keys).
__device__ __forceinline__ UnitCoord decode_unit(const FwdParams& p, int u) {
  const int per = p.tables == 1 ? p.B * p.H : p.H;
  const int rank = u / per, r = u % per;
  int table, st;
  if (p.super_order != nullptr) {
    const int pr = p.super_order[rank];
    table = pr / p.n_super;
    st = pr % p.n_super;
  } else {
    table = rank % p.tables;
    st = p.n_super - 1 - rank / p.tables;
  }
  UnitCoord c;
  c.st = st;
  c.b = p.tables == 1 ? r / p.H : table;
  c.h = p.tables == 1 ? r % p.H : r;
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

// Takes the next work unit from the launch's counter and builds its list
// into buffer ui % 3 (whole warp).  Entries are uint16: kv tile << 4 | class
// of query tile 0 << 2 | class of tile 1.  When no unit is left the buffer
// carries unit = -1, which ends every role's loop.
__device__ __forceinline__ bool build_list(const FwdParams& p, Bars* bars,
                                           uint16_t* lists, int ui) {
  const int lane = threadIdx.x % 32;
  const int buf = ui % kListBufs;
  if (!warp_wait(&bars->list_free[buf], ((ui / kListBufs) & 1) ^ 1,
                 &bars->abort, p.timeout_ns)) {
    if (lane == 0) record_timeout(kRoleList, 0);
    return false;
  }
  int unit = 0;
  if (lane == 0) unit = atomicAdd(p.unit_counter, 1);
  unit = __shfl_sync(0xffffffffu, unit, 0);
  if (unit >= p.num_units) {
    if (lane == 0) {
      bars->meta[buf].unit = -1;
      bars->meta[buf].n = 0;
      mbar_arrive(&bars->list_full[buf]);
    }
    __syncwarp();
    return true;
  }
  const UnitCoord uc = decode_unit(p, unit);
  const int table = (p.flags & BSM_MASK_SEGMENT) ? uc.b : 0;
  const int row0 = uc.st * kUnitRows;
  uint16_t* list = lists + buf * kMaxKvTiles;
  int n = 0, n0 = 0, n1 = 0, last0 = -1, last1 = -1;
  for (int base = 0; base < p.n_kvtiles; base += 64) {
    // two chunks of 32 tiles per pass so that their loads overlap
    int c[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int jt = base + 32 * h + lane;
      c[h][0] = c[h][1] = 0;
      if (jt < p.n_kvtiles) {
        c[h][0] = tile_class(p, table, row0, jt);
        c[h][1] = tile_class(p, table, row0 + kTileM, jt);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int jt = base + 32 * h + lane;
      const int c0 = c[h][0], c1 = c[h][1];
      const unsigned m = __ballot_sync(0xffffffffu, (c0 | c1) != 0);
      const int pos = n + __popc(m & ((1u << lane) - 1u));
      if (c0 | c1)
        list[pos] = static_cast<uint16_t>((jt << 4) | (c0 << 2) | c1);
      n0 += __popc(__ballot_sync(0xffffffffu, c0 != 0));
      n1 += __popc(__ballot_sync(0xffffffffu, c1 != 0));
      last0 = max(last0, __reduce_max_sync(0xffffffffu, c0 ? pos : -1));
      last1 = max(last1, __reduce_max_sync(0xffffffffu, c1 ? pos : -1));
      n += __popc(m);
    }
  }
  __syncwarp();
  if (lane == 0) {
    ListMeta& mt = bars->meta[buf];
    mt.n = n;
    mt.n_t[0] = n0;
    mt.n_t[1] = n1;
    mt.last_t[0] = last0;
    mt.last_t[1] = last1;
    mt.unit = unit;
    mt.b = uc.b;
    mt.h = uc.h;
    mt.st = uc.st;
    trace(p, bars, kRoleList, kEvListBuilt, 0, n, unit);
    mbar_arrive(&bars->list_full[buf]);
  }
  __syncwarp();
  return true;
}

// List-builder warp: stays up to two units ahead of the consumers.
__device__ __forceinline__ void list_role(const FwdParams& p, Bars* bars,
                                         uint16_t* lists) {
  for (int ui = 0;; ++ui) {
    if (!build_list(p, bars, lists, ui)) break;
    if (bars->meta[ui % kListBufs].unit < 0) break;  // sentinel written
  }
}

template <int D>
__device__ __forceinline__ void load_role(const FwdParams& p,
                                          const CUtensorMap* tq,
                                          const CUtensorMap* tk,
                                          const CUtensorMap* tv, uint8_t* smem,
                                          Bars* bars, uint16_t* lists) {
  using C = Cfg<D>;
  const int lane = threadIdx.x % 32;
  volatile int* abort_flag = &bars->abort;
  const uint64_t pol_q = l2_policy_evict_first();
  const uint64_t pol_kv = l2_policy_evict_last();
  uint32_t kv_it = 0;
  uint32_t q_it[2] = {0, 0};
  bool ok = true;
  for (int ui = 0; ok; ++ui) {
    const int buf = ui % kListBufs;
    ok = warp_wait(&bars->list_full[buf], (ui / kListBufs) & 1, abort_flag,
                   p.timeout_ns);
    if (!ok) {
      if (lane == 0) record_timeout(kRoleLoad, 0);
      break;
    }
    const ListMeta mt = bars->meta[buf];
    if (mt.unit < 0) break;
    const int unit = mt.unit;
    const uint16_t* list = lists + buf * kMaxKvTiles;
    const UnitCoord uc{mt.b, mt.h, mt.st};
    const int row0 = uc.st * kUnitRows;
    // Q, per query tile that has work in this unit
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (!ok || mt.n_t[t] == 0) continue;
      ok = warp_wait(&bars->q_empty[t], (q_it[t] & 1) ^ 1, abort_flag,
                     p.timeout_ns);
      if (!ok) {
        if (lane == 0) record_timeout(kRoleLoad, 1);
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->q_full[t], C::kTileBytes);
        for (int kb = 0; kb < C::kKBlocks; ++kb)
          tma_load_4d(tq, &bars->q_full[t],
                      smem + C::kOffQ + t * C::kTileBytes + kb * kTileM * 128,
                      kb * 64, row0 + t * kTileM, uc.h, uc.b, pol_q);
        trace(p, bars, kRoleLoad, kEvQIssued, t, 0, unit);
      }
      ++q_it[t];
    }
    const int hkv = uc.h / (p.H / p.Hkv);
    for (int e = 0; ok && e < mt.n; ++e) {
      const int jt = static_cast<int>(list[e] >> 4);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        if (!ok) break;
        const int slot = kv_it % C::kSlots;
        const uint32_t ph = (kv_it / C::kSlots) & 1;
        ok = warp_wait(&bars->kv_empty[slot], ph ^ 1, abort_flag,
                       p.timeout_ns);
        if (!ok) {
          if (lane == 0) record_timeout(kRoleLoad, 2);
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->kv_full[slot], C::kTileBytes);
          uint8_t* dst = smem + C::kOffKV + slot * C::kTileBytes;
          for (int kb = 0; kb < C::kKBlocks; ++kb)
            tma_load_4d(which == 0 ? tk : tv, &bars->kv_full[slot],
                        dst + kb * kTileN * 128, kb * 64, jt * kTileN, hkv,
                        uc.b, pol_kv);
          trace(p, bars, kRoleLoad, kEvTmaIssued, which, e, unit);
        }
        ++kv_it;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->list_free[buf]);
  }
  // Drain: wait for the loads already issued (after an abort some may still
  // be landing in shared memory); the last load into each barrier completes
  // the phase of parity (loads issued into it - 1) & 1.
  if (lane == 0) {
    for (int s = 0; s < C::kSlots; ++s) {
      const uint32_t n = kv_it > static_cast<uint32_t>(s)
                             ? (kv_it - 1 - s) / C::kSlots + 1 : 0;
      if (n > 0 && !mbar_wait_drain(&bars->kv_full[s], (n - 1) & 1,
                                    p.timeout_ns) && ok)
        record_timeout(kRoleLoad, 3);
    }
    for (int t = 0; t < 2; ++t)
      if (q_it[t] > 0 && !mbar_wait_drain(&bars->q_full[t], (q_it[t] - 1) & 1,
                                          p.timeout_ns) && ok)
        record_timeout(kRoleLoad, 4);
  }
  __syncwarp();
}

// MMA issuer of query tile t: warp 1 (tile 0) or warp 11 (tile 1).  The
// whole warp runs the loop, waits and issues together: each MMA and commit
// goes out from the lane elect.sync picks, the same lane every time (a
// commit tracks the MMAs of the thread that issues it).  The
// two issuers share the K/V ring: every slot is released by both (kv_empty
// counts two arrivals), and an issuer whose tile skips an entry still waits
// for that slot to be filled before releasing it, so the two never drift
// more than one ring cycle apart.
template <int D, int SCORE>
__device__ __forceinline__ void mma_role(const FwdParams& p, uint8_t* smem,
                                         Bars* bars, const uint16_t* lists,
                                         uint32_t tmem, const int t) {
  using C = Cfg<D>;
  const bool leader = (threadIdx.x % 32) == 0;
  volatile int* abort_flag = &bars->abort;
  constexpr uint32_t idesc_s = idesc_bf16_f32(kTileM, kTileN, false);
  constexpr uint32_t idesc_o = idesc_bf16_f32(kTileM, D, true);
  constexpr uint32_t kTileUnits = C::kTileBytes >> 4;
  // Descriptors of the tile bases; a K-step only adds to the start-address
  // field (16-byte units), which never carries into the upper fields.
  const uint64_t dq =
      sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024) + t * kTileUnits;
  const uint64_t dkv0 = sdesc_sw128(smem_u32(smem + C::kOffKV), 16, 1024);
  const uint64_t dv0 =
      sdesc_sw128(smem_u32(smem + C::kOffKV), kTileN * 128, 1024);
  const uint32_t s_acc = tmem + t * 128;        // S_t, and P_t over it
  const uint32_t o_acc = tmem + 256 + t * 128;  // O_t
  uint32_t kv_it = 0, q_it = 0, s_cnt = 0;
  bool ok = true;

  auto wait_slot = [&](int& slot) -> bool {
    slot = kv_it % C::kSlots;
    const bool r = warp_wait(&bars->kv_full[slot], (kv_it / C::kSlots) & 1,
                             abort_flag, p.timeout_ns);
    ++kv_it;
    return r;
  };
  // S_t = Q_t K^T for the K tile in `kslot` (the whole warp; one lane
  // issues).
  auto issue_s = [&](int kslot) {
    const uint64_t b = dkv0 + kslot * kTileUnits;
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k >> 2) * (kTileM * 128 / 16) + (k & 3) * 2;
      mma_ss_elect(s_acc, dq + off, b + off, idesc_s, k > 0 ? 1u : 0u);
    }
    mma_commit_elect(&bars->s_full[t]);
  };
  auto fail = [&](int where) {
    if (leader) record_timeout(kRoleMma, where);
  };

  for (int ui = 0; ok; ++ui) {
    const int buf = ui % kListBufs;
    ok = warp_wait(&bars->list_full[buf], (ui / kListBufs) & 1, abort_flag,
                   p.timeout_ns);
    if (!ok) {
      fail(0);
      break;
    }
    const ListMeta mt = bars->meta[buf];
    if (mt.unit < 0) break;
    const int unit = mt.unit;
    const uint16_t* list = lists + buf * kMaxKvTiles;
    const int shift = t == 0 ? 2 : 0;
    if (leader) trace(p, bars, kRoleMma, kEvMmaUnit, t, mt.n, unit);
    bool q_ready = false, first_pv = true;
    bool s_ahead = false;  // S_t of the current entry already issued
    int kslot_ahead = -1;  // K slot of the current entry if waited ahead
    uint32_t nxt = mt.n > 0 ? list[0] : 0u;  // list entries are read one ahead
    for (int e = 0; e < mt.n && ok; ++e) {
      const bool use = ((nxt >> shift) & 3u) != 0;
      nxt = (e + 1 < mt.n) ? list[e + 1] : 0u;
      const bool use_next = (e + 1 < mt.n) && ((nxt >> shift) & 3u) != 0;
      // ---- K of this entry
      int kslot = kslot_ahead;
      if (kslot < 0 && !(ok = wait_slot(kslot))) {
        fail(2);
        break;
      }
      kslot_ahead = -1;
      if (use && !s_ahead) {
        if (!q_ready) {
          q_ready = true;
          if (!(ok = warp_wait(&bars->q_full[t], q_it & 1, abort_flag,
                               p.timeout_ns))) {
            fail(1);
            break;
          }
        }
        tc_fence_after();
        issue_s(kslot);
        if (leader) trace(p, bars, kRoleMma, kEvSIssued, t, e, unit);
        ++s_cnt;
      }
      if (use && e == mt.last_t[t])  // Q_t of this unit no longer needed
        mma_commit_elect(&bars->q_empty[t]);
      // release the K slot once the S MMA that read it has completed
      if (use)
        mma_commit_elect(&bars->kv_empty[kslot]);
      else if (leader)
        mbar_arrive(&bars->kv_empty[kslot]);
      if (use && e == mt.last_t[t]) ++q_it;
      __syncwarp();
      // ---- V of this entry: O_t += P_t V, then S_t of the next entry
      int vslot;
      if (!(ok = wait_slot(vslot))) {
        fail(4);
        break;
      }
      s_ahead = false;
      if (!use) {
        if (leader) mbar_arrive(&bars->kv_empty[vslot]);
        __syncwarp();
        continue;
      }
      ok = warp_wait(&bars->p_full[t], (s_cnt - 1) & 1, abort_flag,
                     p.timeout_ns);
      if (ok && first_pv)
        ok = warp_wait(&bars->o_free[t], (ui & 1) ^ 1, abort_flag,
                       p.timeout_ns);
      if (!ok) {
        fail(5);
        break;
      }
      {
        if (leader) trace(p, bars, kRoleMma, kEvPReady, t, e, unit);
        tc_fence_after();
        const uint64_t b = dv0 + vslot * kTileUnits;
        if (SCORE == BSM_SCORE_SOFTMAX) {
          // P: key 16kk..16kk+15 in TMEM columns 8kk..8kk+7
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            mma_ts_elect(o_acc, s_acc + kk * 8, b + kk * (16 * 128 / 16),
                         idesc_o, (kk > 0 || !first_pv) ? 1u : 0u);
        } else {
          // P = hi + lo, per 64-key half h: hi in columns 64h..64h+31, lo in
          // 64h+32..64h+63
#pragma unroll 2
          for (int kk = 0; kk < kTileN / 16; ++kk) {
            const uint32_t col = (kk >> 2) * 64 + (kk & 3) * 8;
            mma_ts_elect(o_acc, s_acc + col, b + kk * (16 * 128 / 16),
                         idesc_o, (kk > 0 || !first_pv) ? 1u : 0u);
            mma_ts_elect(o_acc, s_acc + col + 32, b + kk * (16 * 128 / 16),
                         idesc_o, 1u);
          }
        }
        mma_commit_elect(&bars->pv_done[t]);
        if (leader) trace(p, bars, kRoleMma, kEvPVIssued, t, e, unit);
      }
      first_pv = false;
      // S_t of the next entry goes right behind this P.V.  It overwrites the
      // TMEM columns the P.V just read: tcgen05.mma instructions of one
      // thread run in the order they were issued.
      if (use_next) {
        if (!(ok = wait_slot(kslot_ahead))) {
          fail(2);
          break;
        }
        tc_fence_after();
        issue_s(kslot_ahead);
        if (leader) trace(p, bars, kRoleMma, kEvSIssued, t, e + 1, unit);
        ++s_cnt;
        s_ahead = true;
      }
      mma_commit_elect(&bars->kv_empty[vslot]);
      __syncwarp();
    }
    if (!ok) break;
    if (leader) {
      trace(p, bars, kRoleMma, kEvMmaLastPv, t, mt.n, unit);
      mbar_arrive(&bars->list_free[buf]);
    }
    __syncwarp();
  }
  // Drain: every MMA issued above has completed once this arrives (waited
  // for also after an abort, before the CTA frees TMEM).
  __syncwarp();
  mma_commit_elect(&bars->mma_done[t]);
  if (leader && !mbar_wait_drain(&bars->mma_done[t], 0, p.timeout_ns) && ok)
    record_timeout(kRoleMma, 6);
  __syncwarp();
}

// "Same segment" bits of the 128 keys of a tile for one row (unsorted
// segment ids), one 32-bit word per 32 keys.  Computed before S is loaded
// from TMEM, so the loads never compete with S for registers.
__device__ __forceinline__ void segment_bits(uint32_t keep[4],
                                             const int32_t* segk, int nvalid,
                                             int segq) {
  const bool vec =
      nvalid == kTileN && (reinterpret_cast<uintptr_t>(segk) & 15u) == 0;
#pragma unroll 1
  for (int w = 0; w < kTileN / 32; ++w) {
    uint32_t bits = 0;
    if (vec) {
      const int4* s4 = reinterpret_cast<const int4*>(segk + 32 * w);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const int4 v = __ldg(s4 + c4);
        bits |= (v.x == segq ? 1u : 0u) << (4 * c4);
        bits |= (v.y == segq ? 1u : 0u) << (4 * c4 + 1);
        bits |= (v.z == segq ? 1u : 0u) << (4 * c4 + 2);
        bits |= (v.w == segq ? 1u : 0u) << (4 * c4 + 3);
      }
    } else {
#pragma unroll 8
      for (int c = 0; c < 32; ++c) {
        const int k = 32 * w + c;
        if (k < nvalid && __ldg(segk + k) == segq) bits |= 1u << c;
      }
    }
    keep[0] = w == 0 ? bits : keep[0];
    keep[1] = w == 1 ? bits : keep[1];
    keep[2] = w == 2 ? bits : keep[2];
    keep[3] = w == 3 ? bits : keep[3];
  }
}

// Masks S of a partial tile in place: columns outside [lo_c, hi_c] (and,
// with use_keep, columns whose keep bit is clear) become -inf.  Each thread
// holds one row.  Per 32-column chunk the row's visible columns are built as
// one bit word from the two bounds; a chunk that all 32 rows of the warp see
// whole (a warp-uniform test) is left alone, the others cost one bit test
// and one select per column.  Under causal and packed-segment masks most
// chunks of a partial tile are whole for the warp.
__device__ __forceinline__ void mask_tile(float* s, int lo_c, int hi_c,
                                          const uint32_t keep[4],
                                          bool use_keep) {
  const float NEG_INF = __int_as_float(0xff800000);
#pragma unroll
  for (int q = 0; q < kTileN / 32; ++q) {
    const int c0 = 32 * q;
    // visible columns of this chunk as bits: [lo_c, hi_c] cut to the chunk
    const int lb = min(max(lo_c - c0, 0), 32), hb = min(max(hi_c - c0 + 1, 0), 32);
    const uint32_t below_hi = hb >= 32 ? 0xffffffffu : (1u << hb) - 1u;
    const uint32_t below_lo = lb >= 32 ? 0xffffffffu : (1u << lb) - 1u;
    uint32_t vm = below_hi & ~below_lo;
    if (use_keep) vm &= keep[q];
    if (!__all_sync(0xffffffffu, vm == 0xffffffffu)) {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        s[c0 + c] = (vm & (1u << c)) ? s[c0 + c] : NEG_INF;
    }
  }
}

// KEEP: partial tiles also carry per-element "keep" bits -- from segment ids
// compared element by element (some key-id row is not sorted) and/or from
// an arbitrary bit-packed mask; otherwise every mask is a key range per row.
template <int D, int SCORE, bool KEEP, bool PINGPONG>
__device__ __forceinline__ void score_role(const FwdParams& p, Bars* bars,
                                           const uint16_t* lists,
                                           uint32_t tmem) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = (warp - 4) / 4;  // query tile of this warpgroup
  const int quarter = warp % 4;  // TMEM lane quarter this warp may access
  const int r = quarter * 32 + lane;
  const bool tracer = (r == 0);
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t s_addr = tmem + lane_off + t * 128;
  const uint32_t o_addr = tmem + lane_off + 256 + t * 128;
  volatile int* abort_flag = &bars->abort;
  const float NEG_INF = __int_as_float(0xff800000);
  const bool seg = (p.flags & BSM_MASK_SEGMENT) != 0;
  const bool seg_elem = KEEP && seg && (*p.seg_flags & 1) != 0;
  const bool dense = KEEP && p.dense != nullptr;
  uint32_t s_cnt = 0, pv_cnt = 0, turns = 0;
  auto pass_turn = [&]() {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->sm_turn[1 - t][quarter]);
  };
  for (int ui = 0;; ++ui) {
    const int buf = ui % kListBufs;
    if (!warp_wait(&bars->list_full[buf], (ui / kListBufs) & 1, abort_flag,
                   p.timeout_ns)) {
      record_timeout(kRoleScore, 0);
      break;
    }
    const int unit = bars->meta[buf].unit;
    if (unit < 0) break;
    const int n_ent = bars->meta[buf].n;
    const UnitCoord uc{bars->meta[buf].b, bars->meta[buf].h,
                       bars->meta[buf].st};
    const uint16_t* list = lists + buf * kMaxKvTiles;
    const int qrow = uc.st * kUnitRows + t * kTileM + r;
    const bool row_ok = qrow < p.Sq;
    // visible keys of this row form [rlo, rhi] (plus the element compare of
    // unsorted segment ids)
    int rlo = 0, rhi = p.Skv - 1;
    if (p.flags & BSM_MASK_CAUSAL) rhi = min(rhi, qrow);
    if (p.flags & BSM_MASK_LOCAL) rlo = max(rlo, qrow - p.window + 1);
    if (p.flags & BSM_MASK_BAND) rhi = min(rhi, qrow + p.window - 1);
    int segq = 0;
    if (seg && row_ok) {
      const int64_t qi = static_cast<int64_t>(uc.b) * p.Sq + qrow;
      if (seg_elem) {
        segq = p.q_seg[qi];
      } else {
        const int2 sr = reinterpret_cast<const int2*>(p.seg_range)[qi];
        rlo = max(rlo, sr.x);
        rhi = min(rhi, sr.y);
      }
    }
    const int32_t* segk_b =
        seg_elem ? p.kv_seg + static_cast<int64_t>(uc.b) * p.Skv : nullptr;
    float m_used = NEG_INF, l_sum = 0.f;
    uint32_t unit_pv = 0;
    bool ok = true;
    for (int e = 0; e < n_ent; ++e) {
      const uint32_t ent = list[e];
      const int cls = t == 0 ? static_cast<int>((ent >> 2) & 3u)
                             : static_cast<int>(ent & 3u);
      if (!cls) continue;
      // On entries both tiles use, softmax turns alternate between the two
      // score warps that share an SM sub-partition (same lane quarter,
      // tiles 0 and 1; tile 0 first): one works while the tensor core runs
      // the other tile's P.V and next S, instead of both competing for the
      // same issue slots and MUFU at once.
      // (only in units of at least kPingPongMin entries: in a short unit
      // the two tiles would spend a softmax setting up the alternation)
      const bool shared = PINGPONG && n_ent >= kPingPongMin &&
                          ((ent >> 2) & 3u) != 0 && (ent & 3u) != 0;
      if (shared) {
        ok = warp_wait(&bars->sm_turn[t][quarter],
                       (turns & 1) ^ (t == 0 ? 1u : 0u), abort_flag,
                       p.timeout_ns);
        if (!ok) {
          record_timeout(kRoleScore, 6);
          break;
        }
        ++turns;
      }
      const int jt = static_cast<int>(ent >> 4);
      const int kbase = jt * kTileN;
      uint32_t keep[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
      if (KEEP && cls == 1) {
        if (seg_elem)
          segment_bits(keep, segk_b + kbase, min(kTileN, p.Skv - kbase), segq);
        if (dense) {  // the row's mask words for these 128 keys
          const int64_t w0 = kbase >> 5;
          const uint32_t* dw =
              p.dense + static_cast<int64_t>(row_ok ? qrow : 0) * p.dense_words;
#pragma unroll
          for (int w = 0; w < 4; ++w)
            keep[w] &= (row_ok && w0 + w < p.dense_words) ? __ldg(dw + w0 + w)
                                                          : 0u;
        }
      }
      ok = warp_wait(&bars->s_full[t], s_cnt & 1, abort_flag, p.timeout_ns);
      if (!ok) {
        record_timeout(kRoleScore, 1);
        break;
      }
      ++s_cnt;
      if (tracer) trace(p, bars, kRoleScore, kEvSFull, t, e, unit);
      tc_fence_after();
      uint32_t sraw[kTileN];
#pragma unroll
      for (int q = 0; q < kTileN / 32; ++q)
        tmem_ld32(s_addr + q * 32, sraw + q * 32);
      tmem_ld_wait();
      float* s = reinterpret_cast<float*>(sraw);
      if (cls == 1) mask_tile(s, rlo - kbase, rhi - kbase, keep, KEEP);

      uint32_t pk[16];
      if (SCORE == BSM_SCORE_SOFTMAX) {
        // row max: three-input max, four independent chains
        float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
        float mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
        for (int c = 8; c < kTileN; c += 8) {
          mx0 = fmax3(mx0, s[c], s[c + 1]);
          mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
          mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
          mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
        }
        const float mx = fmax3(mx0, mx1, fmaxf(mx2, mx3));
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
        float ls0 = 0.f, ls1 = 0.f, ls2 = 0.f, ls3 = 0.f;
#pragma unroll
        for (int q = 0; q < kTileN / 32; ++q) {  // 32 columns at a time
#pragma unroll
          for (int c = 32 * q; c < 32 * q + 32; c += 4) {
            // paired f32 FMA/add: the same roundings as one element at a time
            float x0, x1, x2, x3;
            ffma2(x0, x1, s[c], s[c + 1], p.scale_log2, neg_m);
            ffma2(x2, x3, s[c + 2], s[c + 3], p.scale_log2, neg_m);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            fadd2(ls0, ls1, ls0, ls1, p0, p1);
            fadd2(ls2, ls3, ls2, ls3, p2, p3);
            pk[(c & 31) / 2] = pack_bf16x2(p0, p1);
            pk[(c & 31) / 2 + 1] = pack_bf16x2(p2, p3);
          }
          tmem_st16(s_addr + q * 16, pk);
        }
        l_sum += (ls0 + ls1) + (ls2 + ls3);
        // Rescale O_t (needs the previous PV of this tile to have landed).
        if (__any_sync(0xffffffffu, rescale) && unit_pv > 0) {
          ok = warp_wait(&bars->pv_done[t], (pv_cnt - 1) & 1, abort_flag,
                         p.timeout_ns);
          if (!ok) {
            record_timeout(kRoleScore, 2);
            break;
          }
          if (tracer) trace(p, bars, kRoleScore, kEvRescale, t, e, unit);
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
        // pointwise: x = scale*qk; p = x*sigmoid(x)/Sq; masked (-inf) -> 0.
        // With sigmoid(x) = (1 + tanh(x/2)) / 2 this is g + g*tanh(x/2),
        // g = x / (2 Sq): one tanh per element, the rest on paired f32.
        // hstu_ops multiplies the f32 scores by f32 v, so p is kept to about
        // 16 bits: p = hi + lo, both bf16 (lo = p - hi is exact in f32).
        // Each 64-key half's hi and lo (32 columns each) go back over that
        // half's own 64 columns of S; the MMA warp adds both products into O.
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t pl[16];
#pragma unroll
            for (int c = 64 * hf + 32 * q; c < 64 * hf + 32 * q + 32; c += 2) {
              float h0, h1, g0, g1, p0, p1;
              fmul2(h0, h1, s[c], s[c + 1], p.pw_half);
              fmul2(g0, g1, s[c], s[c + 1], p.pw_g);
              ffma2v(p0, p1, g0, g1, tanh_approx(h0), tanh_approx(h1), g0,
                     g1);
              p0 = s[c] != NEG_INF ? p0 : 0.f;
              p1 = s[c + 1] != NEG_INF ? p1 : 0.f;
              const uint32_t hi = pack_bf16x2(p0, p1);
              pk[(c & 31) / 2] = hi;
              pl[(c & 31) / 2] =
                  pack_bf16x2(p0 - __uint_as_float(hi << 16),
                              p1 - __uint_as_float(hi & 0xffff0000u));
            }
            tmem_st16(s_addr + hf * 64 + q * 16, pk);
            tmem_st16(s_addr + hf * 64 + 32 + q * 16, pl);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_full[t]);
      if (shared) pass_turn();
      if (tracer) trace(p, bars, kRoleScore, kEvPFull, t, e, unit);
      ++pv_cnt;
      ++unit_pv;
    }
    if (!ok) break;

    // ---- epilogue: out = O / l (softmax) or O (pointwise), bf16
    if (tracer) trace(p, bars, kRoleScore, kEvEpiBegin, t, 0, unit);
    uint16_t* orow = p.out + static_cast<int64_t>(uc.b) * p.o_sb +
                     static_cast<int64_t>(uc.h) * p.o_sh +
                     static_cast<int64_t>(qrow) * p.o_ss;
    if (unit_pv > 0) {
      if (!warp_wait(&bars->pv_done[t], (pv_cnt - 1) & 1, abort_flag,
                     p.timeout_ns)) {
        record_timeout(kRoleScore, 3);
        break;
      }
      if (tracer) trace(p, bars, kRoleScore, kEvEpiPvLanded, t, 0, unit);
      tc_fence_after();
      // all of O_t into registers with one wait; the next unit's first P.V
      // may then overwrite it while the stores go out
      uint32_t o[D];
#pragma unroll
      for (int q = 0; q < D / 32; ++q) tmem_ld32(o_addr + q * 32, o + q * 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bars->o_free[t]);
      if (tracer) trace(p, bars, kRoleScore, kEvEpiOLoaded, t, 0, unit);
      float inv = 1.f;
      if (SCORE == BSM_SCORE_SOFTMAX) inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      if (row_ok) {
        // 32 bytes per store where the row alignment allows: each warp
        // store touches 32 rows, so fewer, wider stores cost fewer requests
        const bool v8 = p.o_vec8 != 0;
#pragma unroll
        for (int v = 0; v < D / 16; ++v) {
          uint32_t w[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            w[c] = pack_bf16x2(__uint_as_float(o[16 * v + 2 * c]) * inv,
                               __uint_as_float(o[16 * v + 2 * c + 1]) * inv);
          if (v8) {
            st_global_v8(orow + v * 16, w);
          } else {
            st_global_v4(orow + v * 16, w[0], w[1], w[2], w[3]);
            st_global_v4(orow + v * 16 + 8, w[4], w[5], w[6], w[7]);
          }
        }
      }
    } else {
      if (row_ok) {
#pragma unroll
        for (int v = 0; v < D / 8; ++v)
          st_global_v4(orow + v * 8, 0u, 0u, 0u, 0u);
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free[t]);
    }
    if (SCORE == BSM_SCORE_SOFTMAX && p.lse != nullptr && row_ok) {
      const float lse = l_sum > 0.f
                            ? (m_used + log2f(l_sum)) * 0.6931471805599453f
                            : NEG_INF;
      p.lse[(static_cast<int64_t>(uc.b) * p.H + uc.h) * p.Sq + qrow] = lse;
    }
    mbar_arrive(&bars->list_free[buf]);
    if (tracer) trace(p, bars, kRoleScore, kEvEpiEnd, t, 0, unit);
  }
}

template <int D, int SCORE, bool PINGPONG>
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
  uint16_t* lists = p.lists + static_cast<size_t>(blockIdx.x) * kListBufs *
                                  kMaxKvTiles;
  const int warp = threadIdx.x / 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kListBufs; ++i) {
      mbar_init(&bars->list_full[i], 1);
      mbar_init(&bars->list_free[i], 3 + 2 * kTileM);  // load, 2 MMA, score
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], kTileM);
      mbar_init(&bars->pv_done[i], 1);
      mbar_init(&bars->o_free[i], kTileM);
      for (int q = 0; q < 4; ++q) mbar_init(&bars->sm_turn[i][q], 1);
    }
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 2);  // both MMA issuers
    }
    mbar_init(&bars->mma_done[0], 1);
    mbar_init(&bars->mma_done[1], 1);
    bars->abort = 0;
    for (int i = 0; i < 6; ++i) bars->trace_n[i] = 0;
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

  if (warp < 4) {
    setmaxnreg_dec<kRegsLight>();
    if (warp == 0)
      load_role<D>(p, &tm_q, &tm_k, &tm_v, smem, bars, lists);
    else if (warp == 3)
      list_role(p, bars, lists);
    else
      mma_role<D, SCORE>(p, smem, bars, lists, tmem, warp - 1);
  } else {
    setmaxnreg_inc<kRegsScore>();
    // one path per launch: per-element keep bits only when segment ids are
    // unsorted or an arbitrary mask is given (read once; the same for every
    // thread).  The alternating-turn instance is never launched for either.
    if (!PINGPONG && (((p.flags & BSM_MASK_SEGMENT) && (*p.seg_flags & 1) != 0) ||
                      p.dense != nullptr))
      score_role<D, SCORE, !PINGPONG, PINGPONG>(p, bars, lists, tmem);
    else
      score_role<D, SCORE, false, PINGPONG>(p, bars, lists, tmem);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (p.trace != nullptr && threadIdx.x == 0) {
    uint32_t* hdr = reinterpret_cast<uint32_t*>(
        reinterpret_cast<TraceRec*>(p.trace) +
        static_cast<size_t>(blockIdx.x) * (p.trace_cap + 2));
    const uint32_t per = p.trace_cap / 6;
    for (int i = 0; i < 8; ++i) hdr[i] = i < 6 ? min(bars->trace_n[i], per) : 0;
  }
}

// ---------------------------------------------------------------------------
// Decoupled query tiles, for packed sequences (segment ids).  There the
// units are short and the two query tiles of a unit often need different KV
// tiles, so the lockstep pipeline above spends much of its time at unit
// boundaries and on entries one tile skips.  Here the two 128-row query
// tiles of an SM are two independent pipelines: each takes its own work
// units (one query tile of one (batch, head)), builds its own KV-tile list,
// and has its own Q buffer and two-slot K/V ring, so one pipeline's unit
// boundary overlaps the other's work on the tensor core.  K/V tiles are not
// shared between the tiles (L2 carries the reuse).  Masks without segment
// ids take this kernel too below 4096 keys, where units are short as well.
//
// Warp roles (384 threads, three warpgroups, registers split as above):
// warps 0/1 take pipeline 0/1's units, build their lists and load their
// tiles; warps 2/3 issue its MMAs (warp 2 also owns the TMEM); warps 4-7
// and 8-11 are the score warpgroups of pipeline 0 and 1.  TMEM as above:
// S_t/P_t at [128 t, +128), O_t at [256 + 128 t, +128).  Head dim 128,
// softmax or pointwise.
constexpr int kDtThreads = 384;
constexpr int kDtTile = kTileM * 128 * 2;  // one 128 x 128 bf16 tile
constexpr int kDtOffQ = 0;                 // Q of pipeline t at t tiles
constexpr int kDtOffKV = 2 * kDtTile;      // ring slot s of pipeline t
constexpr int kDtOffBar = kDtOffKV + 4 * kDtTile;
constexpr int kDtSmemBytes = kDtOffBar + 1024 + 1024;
static_assert(kDtSmemBytes <= 232448, "shared memory budget");

struct DtMeta {
  int n;     // entries (KV tiles) of the unit
  int unit;  // -1: no unit left
  int b, h;  // batch row and head
  int qt;    // 128-row query tile
};

struct DtBars {
  uint64_t list_full[2][kListBufs], list_free[2][kListBufs];
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[2][2], kv_empty[2][2];  // [pipeline][slot]: K, V
  uint64_t s_full[2], p_full[2], pv_done[2], o_free[2], mma_done[2];
  uint32_t tmem_base;
  int abort;
  uint32_t trace_n[6];
  DtMeta meta[2][kListBufs];
};
static_assert(sizeof(DtBars) <= 1024, "barrier block");

// Optional event trace, in the layout of `trace` above; the six recording
// threads are: loader 0, MMA 0, score 0, score 1, loader 1, MMA 1.
template <bool TRACE>
__device__ __forceinline__ void dt_trace(const FwdParams& p, DtBars* bars,
                                         uint32_t role, uint32_t ev,
                                         uint32_t tile, uint32_t entry,
                                         uint32_t unit) {
  if (!TRACE) return;
  const uint32_t slot = role == kRoleScore ? 2 + tile
                        : role == kRoleMma   ? (tile == 0 ? 1 : 5)
                                             : (tile == 0 ? 0 : 4);
  const uint32_t per = p.trace_cap / 6;
  const uint32_t i = bars->trace_n[slot]++;
  if (i < per) {
    TraceRec* r = reinterpret_cast<TraceRec*>(p.trace) +
                  static_cast<size_t>(blockIdx.x) * (p.trace_cap + 2) + 2 +
                  slot * per + i;
    r->t = globaltimer_ns();
    r->a = (role << 28) | (ev << 24) | (tile << 20) | (entry & 0xFFFFFu);
    r->b = unit;
  }
}

// Takes pipeline t's next unit from the counter and writes its KV-tile
// list (uint16: tile << 2 | class) into buffer ui % kListBufs (whole warp);
// unit -1 when none is left.  Units are numbered two per 256-row unit of
// the lockstep kernel's order (its two query tiles), longest first.
template <bool TRACE>
__device__ __forceinline__ bool dt_build_list(const FwdParams& p, DtBars* bars,
                                              uint16_t* lists, const int t,
                                              const int ui) {
  const int lane = threadIdx.x % 32;
  volatile int* abort_flag = &bars->abort;
  const int n_units = 2 * p.num_units;
  {
    const int buf = ui % kListBufs;
    if (!warp_wait(&bars->list_free[t][buf], ((ui / kListBufs) & 1) ^ 1,
                   abort_flag, p.timeout_ns)) {
      if (lane == 0) record_timeout(kRoleList, 0);
      return false;
    }
    int unit = 0;
    if (lane == 0) unit = atomicAdd(p.unit_counter, 1);
    unit = __shfl_sync(0xffffffffu, unit, 0);
    DtMeta& mt = bars->meta[t][buf];
    if (unit >= n_units) {
      if (lane == 0) {
        mt.unit = -1;
        mt.n = 0;
        mbar_arrive(&bars->list_full[t][buf]);
      }
      __syncwarp();
      return true;
    }
    const UnitCoord uc = decode_unit(p, unit >> 1);
    const int qt = uc.st * 2 + (unit & 1);
    const int table = (p.flags & BSM_MASK_SEGMENT) ? uc.b : 0;
    uint16_t* list = lists + buf * kMaxKvTiles;
    int n = 0;
    for (int base = 0; base < p.n_kvtiles; base += 64) {
      int c[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int jt = base + 32 * h + lane;
        c[h] = jt < p.n_kvtiles ? tile_class(p, table, qt * kTileM, jt) : 0;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int jt = base + 32 * h + lane;
        const unsigned m = __ballot_sync(0xffffffffu, c[h] != 0);
        if (c[h]) list[n + __popc(m & ((1u << lane) - 1u))] =
            static_cast<uint16_t>((jt << 2) | c[h]);
        n += __popc(m);
      }
    }
    __syncwarp();
    if (lane == 0) {
      mt.n = n;
      mt.unit = unit;
      mt.b = uc.b;
      mt.h = uc.h;
      mt.qt = qt;
      dt_trace<TRACE>(p, bars, kRoleList, kEvListBuilt, t, n, unit);
      mbar_arrive(&bars->list_full[t][buf]);
    }
    __syncwarp();
  }
  return true;
}

// Pipeline t's loader: builds the next unit's list, then loads its Q and
// the K and V of every entry through the pipeline's two slots (K in slot
// 0, V in slot 1).  The next list is built once this unit's last loads are
// issued, i.e. while the unit's last entries still run (building it after
// the first entry's loads measured slower).
template <bool TRACE>
__device__ __forceinline__ void dt_load_role(const FwdParams& p,
                                             const CUtensorMap* tq,
                                             const CUtensorMap* tk,
                                             const CUtensorMap* tv,
                                             uint8_t* smem, DtBars* bars,
                                             uint16_t* lists, const int t) {
  const int lane = threadIdx.x % 32;
  volatile int* abort_flag = &bars->abort;
  const uint64_t pol_q = l2_policy_evict_first();
  const uint64_t pol_kv = l2_policy_evict_last();
  uint32_t kv_it = 0, q_it = 0;
  bool ok = true;
  for (int ui = 0; ok; ++ui) {
    const int buf = ui % kListBufs;
    ok = dt_build_list<TRACE>(p, bars, lists, t, ui);
    if (!ok) break;
    const DtMeta mt = bars->meta[t][buf];
    if (mt.unit < 0) break;
    const uint16_t* list = lists + buf * kMaxKvTiles;
    if (mt.n > 0) {
      ok = warp_wait(&bars->q_empty[t], (q_it & 1) ^ 1, abort_flag,
                     p.timeout_ns);
      if (!ok) {
        if (lane == 0) record_timeout(kRoleLoad, 1);
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->q_full[t], kDtTile);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_4d(tq, &bars->q_full[t],
                      smem + kDtOffQ + t * kDtTile + kb * kTileM * 128,
                      kb * 64, mt.qt * kTileM, mt.h, mt.b, pol_q);
        dt_trace<TRACE>(p, bars, kRoleLoad, kEvQIssued, t, 0, mt.unit);
      }
      ++q_it;
    }
    const int hkv = mt.h / (p.H / p.Hkv);
    for (int e = 0; ok && e < mt.n; ++e) {
      const int jt = static_cast<int>(list[e] >> 2);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        if (!ok) break;
        const uint32_t ph = (kv_it >> 1) & 1;
        ok = warp_wait(&bars->kv_empty[t][which], ph ^ 1, abort_flag,
                       p.timeout_ns);
        if (!ok) {
          if (lane == 0) record_timeout(kRoleLoad, 2);
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->kv_full[t][which], kDtTile);
          uint8_t* dst = smem + kDtOffKV + (2 * t + which) * kDtTile;
          for (int kb = 0; kb < 2; ++kb)
            tma_load_4d(which == 0 ? tk : tv, &bars->kv_full[t][which],
                        dst + kb * kTileN * 128, kb * 64, jt * kTileN, hkv,
                        mt.b, pol_kv);
          dt_trace<TRACE>(p, bars, kRoleLoad, kEvTmaIssued, t, e * 2 + which, mt.unit);
        }
        ++kv_it;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->list_free[t][buf]);
  }
  // Drain the loads already issued (each slot received kv_it / 2 loads).
  if (lane == 0) {
    for (int s = 0; s < 2; ++s) {
      const uint32_t n = (kv_it + 1 - s) >> 1;  // loads slot s received
      if (n > 0 && !mbar_wait_drain(&bars->kv_full[t][s], (n - 1) & 1,
                                    p.timeout_ns) && ok)
        record_timeout(kRoleLoad, 3);
    }
    if (q_it > 0 && !mbar_wait_drain(&bars->q_full[t], (q_it - 1) & 1,
                                     p.timeout_ns) && ok)
      record_timeout(kRoleLoad, 4);
  }
  __syncwarp();
}

// Pipeline t's MMA warp: S(e) = Q K(e)^T, then O += P(e) V(e) and S(e + 1)
// right behind it (tcgen05 MMAs of one thread run in issue order, so
// S(e + 1) overwrites the columns P(e) V read only after that product).
// The K slot is released once the S that read it completed, the V slot
// once the P.V did.  The whole warp runs the issuing code and each MMA and
// commit goes out from the lane elect.sync picks (the same lane every
// time: the warp is converged there); issued that way the pipeline's MMAs
// measured ~5 % faster than from a branch lane 0 takes alone.
template <int SCORE, bool TRACE>
__device__ __forceinline__ void dt_mma_role(const FwdParams& p, uint8_t* smem,
                                            DtBars* bars, uint32_t tmem,
                                            const int t) {
  const bool leader = (threadIdx.x % 32) == 0;
  volatile int* abort_flag = &bars->abort;
  constexpr uint32_t idesc_s = idesc_bf16_f32(kTileM, kTileN, false);
  constexpr uint32_t idesc_o = idesc_bf16_f32(kTileM, 128, true);
  const uint64_t dq =
      sdesc_sw128(smem_u32(smem + kDtOffQ + t * kDtTile), 16, 1024);
  const uint64_t dk =
      sdesc_sw128(smem_u32(smem + kDtOffKV + (2 * t) * kDtTile), 16, 1024);
  const uint64_t dv = sdesc_sw128(
      smem_u32(smem + kDtOffKV + (2 * t + 1) * kDtTile), kTileN * 128, 1024);
  const uint32_t s_acc = tmem + t * 128;
  const uint32_t o_acc = tmem + 256 + t * 128;
  uint32_t k_it = 0, v_it = 0, q_it = 0, s_cnt = 0;
  bool ok = true;
  auto fail = [&](int where) {
    if (leader) record_timeout(kRoleMma, where);
  };
  auto issue_s = [&]() {
#pragma unroll
    for (int k = 0; k < 128 / 16; ++k) {
      const uint32_t off = (k >> 2) * (kTileM * 128 / 16) + (k & 3) * 2;
      mma_ss_elect(s_acc, dq + off, dk + off, idesc_s, k > 0 ? 1u : 0u);
    }
    mma_commit_elect(&bars->s_full[t]);
  };
  for (int ui = 0; ok; ++ui) {
    const int buf = ui % kListBufs;
    ok = warp_wait(&bars->list_full[t][buf], (ui / kListBufs) & 1, abort_flag,
                   p.timeout_ns);
    if (!ok) {
      fail(0);
      break;
    }
    const DtMeta mt = bars->meta[t][buf];
    if (mt.unit < 0) break;
    const int n = mt.n;
    if (n > 0) {
      ok = warp_wait(&bars->q_full[t], q_it & 1, abort_flag, p.timeout_ns) &&
           warp_wait(&bars->kv_full[t][0], k_it & 1, abort_flag, p.timeout_ns);
      if (!ok) {
        fail(1);
        break;
      }
      ++q_it;
      ++k_it;
      tc_fence_after();
      issue_s();
      if (leader) dt_trace<TRACE>(p, bars, kRoleMma, kEvSIssued, t, 0, mt.unit);
      if (n == 1) mma_commit_elect(&bars->q_empty[t]);
      mma_commit_elect(&bars->kv_empty[t][0]);
      ++s_cnt;
    }
    for (int e = 0; ok && e < n; ++e) {
      ok = warp_wait(&bars->kv_full[t][1], v_it & 1, abort_flag,
                     p.timeout_ns) &&
           warp_wait(&bars->p_full[t], (s_cnt - 1) & 1, abort_flag,
                     p.timeout_ns);
      if (ok && e == 0)
        ok = warp_wait(&bars->o_free[t], (ui & 1) ^ 1, abort_flag,
                       p.timeout_ns);
      if (!ok) {
        fail(5);
        break;
      }
      ++v_it;
      if (leader) dt_trace<TRACE>(p, bars, kRoleMma, kEvPReady, t, e, mt.unit);
      tc_fence_after();
      if (SCORE == BSM_SCORE_SOFTMAX) {
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)
          mma_ts_elect(o_acc, s_acc + kk * 8, dv + kk * (16 * 128 / 16),
                       idesc_o, (kk > 0 || e > 0) ? 1u : 0u);
      } else {
#pragma unroll 2
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          const uint32_t col = (kk >> 2) * 64 + (kk & 3) * 8;
          mma_ts_elect(o_acc, s_acc + col, dv + kk * (16 * 128 / 16), idesc_o,
                       (kk > 0 || e > 0) ? 1u : 0u);
          mma_ts_elect(o_acc, s_acc + col + 32, dv + kk * (16 * 128 / 16),
                       idesc_o, 1u);
        }
      }
      mma_commit_elect(&bars->pv_done[t]);
      mma_commit_elect(&bars->kv_empty[t][1]);
      if (leader)
        dt_trace<TRACE>(p, bars, kRoleMma, kEvPVIssued, t, e, mt.unit);
      if (e + 1 < n) {
        ok = warp_wait(&bars->kv_full[t][0], k_it & 1, abort_flag,
                       p.timeout_ns);
        if (!ok) {
          fail(2);
          break;
        }
        ++k_it;
        tc_fence_after();
        issue_s();
        if (leader)
          dt_trace<TRACE>(p, bars, kRoleMma, kEvSIssued, t, e + 1, mt.unit);
        if (e + 1 == n - 1) mma_commit_elect(&bars->q_empty[t]);
        mma_commit_elect(&bars->kv_empty[t][0]);
        ++s_cnt;
      }
    }
    if (!ok) break;
    if (leader) mbar_arrive(&bars->list_free[t][buf]);
    __syncwarp();
  }
  __syncwarp();
  mma_commit_elect(&bars->mma_done[t]);
  if (leader && !mbar_wait_drain(&bars->mma_done[t], 0, p.timeout_ns) && ok)
    record_timeout(kRoleMma, 6);
  __syncwarp();
}

template <int SCORE, bool KEEP, bool TRACE>
__device__ __forceinline__ void dt_score_role(const FwdParams& p, DtBars* bars,
                                              const uint16_t* lists,
                                              uint32_t tmem, const int t) {
  constexpr int D = 128;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4;  // TMEM lane quarter this warp may access
  const int r = quarter * 32 + lane;
  const bool tracer = (r == 0);
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t s_addr = tmem + lane_off + t * 128;
  const uint32_t o_addr = tmem + lane_off + 256 + t * 128;
  volatile int* abort_flag = &bars->abort;
  const float NEG_INF = __int_as_float(0xff800000);
  const bool seg = (p.flags & BSM_MASK_SEGMENT) != 0;
  const bool seg_elem = KEEP && seg && (*p.seg_flags & 1) != 0;
  const bool dense = KEEP && p.dense != nullptr;
  uint32_t s_cnt = 0, pv_cnt = 0;
  for (int ui = 0;; ++ui) {
    const int buf = ui % kListBufs;
    if (!warp_wait(&bars->list_full[t][buf], (ui / kListBufs) & 1, abort_flag,
                   p.timeout_ns)) {
      record_timeout(kRoleScore, 0);
      break;
    }
    const int unit = bars->meta[t][buf].unit;
    if (unit < 0) break;
    const int n_ent = bars->meta[t][buf].n;
    const UnitCoord uc{bars->meta[t][buf].b, bars->meta[t][buf].h, 0};
    const uint16_t* list = lists + buf * kMaxKvTiles;
    const int qrow = bars->meta[t][buf].qt * kTileM + r;
    const bool row_ok = qrow < p.Sq;
    // visible keys of this row form [rlo, rhi] (plus the element compare of
    // unsorted segment ids)
    int rlo = 0, rhi = p.Skv - 1;
    if (p.flags & BSM_MASK_CAUSAL) rhi = min(rhi, qrow);
    if (p.flags & BSM_MASK_LOCAL) rlo = max(rlo, qrow - p.window + 1);
    if (p.flags & BSM_MASK_BAND) rhi = min(rhi, qrow + p.window - 1);
    int segq = 0;
    if (seg && row_ok) {
      const int64_t qi = static_cast<int64_t>(uc.b) * p.Sq + qrow;
      if (seg_elem) {
        segq = p.q_seg[qi];
      } else {
        const int2 sr = reinterpret_cast<const int2*>(p.seg_range)[qi];
        rlo = max(rlo, sr.x);
        rhi = min(rhi, sr.y);
      }
    }
    const int32_t* segk_b =
        seg_elem ? p.kv_seg + static_cast<int64_t>(uc.b) * p.Skv : nullptr;
    float m_used = NEG_INF, l_sum = 0.f;
    uint32_t unit_pv = 0;
    bool ok = true;
    for (int e = 0; e < n_ent; ++e) {
      const uint32_t ent = list[e];
      const int cls = static_cast<int>(ent & 3u);
      if (!cls) continue;
      const int jt = static_cast<int>(ent >> 2);
      const int kbase = jt * kTileN;
      uint32_t keep[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
      if (KEEP && cls == 1) {
        if (seg_elem)
          segment_bits(keep, segk_b + kbase, min(kTileN, p.Skv - kbase), segq);
        if (dense) {  // the row's mask words for these 128 keys
          const int64_t w0 = kbase >> 5;
          const uint32_t* dw =
              p.dense + static_cast<int64_t>(row_ok ? qrow : 0) * p.dense_words;
#pragma unroll
          for (int w = 0; w < 4; ++w)
            keep[w] &= (row_ok && w0 + w < p.dense_words) ? __ldg(dw + w0 + w)
                                                          : 0u;
        }
      }
      ok = warp_wait(&bars->s_full[t], s_cnt & 1, abort_flag, p.timeout_ns);
      if (!ok) {
        record_timeout(kRoleScore, 1);
        break;
      }
      ++s_cnt;
      if (tracer) dt_trace<TRACE>(p, bars, kRoleScore, kEvSFull, t, e, unit);
      tc_fence_after();
      uint32_t sraw[kTileN];
#pragma unroll
      for (int q = 0; q < kTileN / 32; ++q)
        tmem_ld32(s_addr + q * 32, sraw + q * 32);
      tmem_ld_wait();
      float* s = reinterpret_cast<float*>(sraw);
      if (cls == 1) mask_tile(s, rlo - kbase, rhi - kbase, keep, KEEP);

      uint32_t pk[16];
      if (SCORE == BSM_SCORE_SOFTMAX) {
        // row max: three-input max, four independent chains
        float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
        float mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
        for (int c = 8; c < kTileN; c += 8) {
          mx0 = fmax3(mx0, s[c], s[c + 1]);
          mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
          mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
          mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
        }
        const float mx = fmax3(mx0, mx1, fmaxf(mx2, mx3));
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
        float ls0 = 0.f, ls1 = 0.f, ls2 = 0.f, ls3 = 0.f;
#pragma unroll
        for (int q = 0; q < kTileN / 32; ++q) {  // 32 columns at a time
#pragma unroll
          for (int c = 32 * q; c < 32 * q + 32; c += 4) {
            // paired f32 FMA/add: the same roundings as one element at a time
            float x0, x1, x2, x3;
            ffma2(x0, x1, s[c], s[c + 1], p.scale_log2, neg_m);
            ffma2(x2, x3, s[c + 2], s[c + 3], p.scale_log2, neg_m);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            fadd2(ls0, ls1, ls0, ls1, p0, p1);
            fadd2(ls2, ls3, ls2, ls3, p2, p3);
            pk[(c & 31) / 2] = pack_bf16x2(p0, p1);
            pk[(c & 31) / 2 + 1] = pack_bf16x2(p2, p3);
          }
          tmem_st16(s_addr + q * 16, pk);
        }
        l_sum += (ls0 + ls1) + (ls2 + ls3);
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
        // pointwise: x = scale*qk; p = x*sigmoid(x)/Sq; masked (-inf) -> 0.
        // With sigmoid(x) = (1 + tanh(x/2)) / 2 this is g + g*tanh(x/2),
        // g = x / (2 Sq): one tanh per element, the rest on paired f32.
        // hstu_ops multiplies the f32 scores by f32 v, so p is kept to about
        // 16 bits: p = hi + lo, both bf16 (lo = p - hi is exact in f32).
        // Each 64-key half's hi and lo (32 columns each) go back over that
        // half's own 64 columns of S; the MMA warp adds both products into O.
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t pl[16];
#pragma unroll
            for (int c = 64 * hf + 32 * q; c < 64 * hf + 32 * q + 32; c += 2) {
              float h0, h1, g0, g1, p0, p1;
              fmul2(h0, h1, s[c], s[c + 1], p.pw_half);
              fmul2(g0, g1, s[c], s[c + 1], p.pw_g);
              ffma2v(p0, p1, g0, g1, tanh_approx(h0), tanh_approx(h1), g0,
                     g1);
              p0 = s[c] != NEG_INF ? p0 : 0.f;
              p1 = s[c + 1] != NEG_INF ? p1 : 0.f;
              const uint32_t hi = pack_bf16x2(p0, p1);
              pk[(c & 31) / 2] = hi;
              pl[(c & 31) / 2] =
                  pack_bf16x2(p0 - __uint_as_float(hi << 16),
                              p1 - __uint_as_float(hi & 0xffff0000u));
            }
            tmem_st16(s_addr + hf * 64 + q * 16, pk);
            tmem_st16(s_addr + hf * 64 + 32 + q * 16, pl);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_full[t]);
      if (tracer) dt_trace<TRACE>(p, bars, kRoleScore, kEvPFull, t, e, unit);
      ++pv_cnt;
      ++unit_pv;
    }
    if (!ok) break;

    // ---- epilogue: out = O / l (softmax) or O (pointwise), bf16
    if (tracer) dt_trace<TRACE>(p, bars, kRoleScore, kEvEpiBegin, t, 0, unit);
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
      // all of O_t into registers with one wait; the next unit's first P.V
      // may then overwrite it while the stores go out
      uint32_t o[D];
#pragma unroll
      for (int q = 0; q < D / 32; ++q) tmem_ld32(o_addr + q * 32, o + q * 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bars->o_free[t]);
      float inv = 1.f;
      if (SCORE == BSM_SCORE_SOFTMAX) inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      if (row_ok) {
        // 32 bytes per store where the row alignment allows: each warp
        // store touches 32 rows, so fewer, wider stores cost fewer requests
        const bool v8 = p.o_vec8 != 0;
#pragma unroll
        for (int v = 0; v < D / 16; ++v) {
          uint32_t w[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            w[c] = pack_bf16x2(__uint_as_float(o[16 * v + 2 * c]) * inv,
                               __uint_as_float(o[16 * v + 2 * c + 1]) * inv);
          if (v8) {
            st_global_v8(orow + v * 16, w);
          } else {
            st_global_v4(orow + v * 16, w[0], w[1], w[2], w[3]);
            st_global_v4(orow + v * 16 + 8, w[4], w[5], w[6], w[7]);
          }
        }
      }
    } else {
      if (row_ok) {
#pragma unroll
        for (int v = 0; v < D / 8; ++v)
          st_global_v4(orow + v * 8, 0u, 0u, 0u, 0u);
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free[t]);
    }
    if (SCORE == BSM_SCORE_SOFTMAX && p.lse != nullptr && row_ok) {
      const float lse = l_sum > 0.f
                            ? (m_used + log2f(l_sum)) * 0.6931471805599453f
                            : NEG_INF;
      p.lse[(static_cast<int64_t>(uc.b) * p.H + uc.h) * p.Sq + qrow] = lse;
    }
    mbar_arrive(&bars->list_free[t][buf]);
    if (tracer) dt_trace<TRACE>(p, bars, kRoleScore, kEvEpiEnd, t, 0, unit);
  }
}


template <int SCORE, bool TRACE>
__global__ void __launch_bounds__(kDtThreads, 1)
    splash_fwd_dt_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  DtBars* bars = reinterpret_cast<DtBars*>(smem + kDtOffBar);
  // the CTA's lists: kListBufs per pipeline
  uint16_t* lists = p.lists + static_cast<size_t>(blockIdx.x) * 2 * kListBufs *
                                  kMaxKvTiles;
  const int warp = threadIdx.x / 32;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      for (int i = 0; i < kListBufs; ++i) {
        mbar_init(&bars->list_full[t][i], 1);
        mbar_init(&bars->list_free[t][i], 2 + kTileM);  // load, MMA, score
      }
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->q_empty[t], 1);
      for (int s = 0; s < 2; ++s) {
        mbar_init(&bars->kv_full[t][s], 1);
        mbar_init(&bars->kv_empty[t][s], 1);
      }
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], kTileM);
      mbar_init(&bars->pv_done[t], 1);
      mbar_init(&bars->o_free[t], kTileM);
      mbar_init(&bars->mma_done[t], 1);
    }
    bars->abort = 0;
    for (int i = 0; i < 6; ++i) bars->trace_n[i] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 2) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < 4) {
    setmaxnreg_dec<kRegsLight>();
    const int t = warp & 1;
    uint16_t* lt = lists + t * kListBufs * kMaxKvTiles;
    if (warp < 2)
      dt_load_role<TRACE>(p, &tm_q, &tm_k, &tm_v, smem, bars, lt, t);
    else
      dt_mma_role<SCORE, TRACE>(p, smem, bars, tmem, t);
  } else {
    setmaxnreg_inc<kRegsScore>();
    const int t = (warp - 4) / 4;
    const uint16_t* lt = lists + t * kListBufs * kMaxKvTiles;
    // per-element keep bits only when segment ids are unsorted or an
    // arbitrary mask is given (read once; the same for every thread)
    if (((p.flags & BSM_MASK_SEGMENT) && (*p.seg_flags & 1) != 0) ||
        p.dense != nullptr)
      dt_score_role<SCORE, true, TRACE>(p, bars, lt, tmem, t);
    else
      dt_score_role<SCORE, false, TRACE>(p, bars, lt, tmem, t);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
  if (TRACE && threadIdx.x == 0) {
    uint32_t* hdr = reinterpret_cast<uint32_t*>(
        reinterpret_cast<TraceRec*>(p.trace) +
        static_cast<size_t>(blockIdx.x) * (p.trace_cap + 2));
    const uint32_t per = p.trace_cap / 6;
    for (int i = 0; i < 8; ++i) hdr[i] = i < 6 ? min(bars->trace_n[i], per) : 0;
  }
}

template <int SCORE>
cudaError_t launch_dt(const FwdParams& p, const CUtensorMap& tq,
                      const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                      cudaStream_t stream) {
  // the instance that records the event trace is launched only with one
  auto kern = p.trace != nullptr ? splash_fwd_dt_kernel<SCORE, true>
                                 : splash_fwd_dt_kernel<SCORE, false>;
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs * kDtThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kDtSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kDtThreads, kDtSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

template <int D, int SCORE, bool PINGPONG>
cudaError_t launch_one(const FwdParams& p, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv,
                       int grid, cudaStream_t stream) {
  using C = Cfg<D>;
  auto kern = splash_fwd_kernel<D, SCORE, PINGPONG>;
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  // the setmaxnreg split must fit the registers the CTA is launched with,
  // else the score warps would wait for registers forever
  if (attr.numRegs * kThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes);
  if (e != cudaSuccess) return e;
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

int fwd_grid_size(const FwdParams& p, int num_sms) {
  return p.num_units < num_sms ? p.num_units : num_sms;
}

cudaError_t launch_splash_fwd(const FwdParams& p, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv,
                              int num_sms, cudaStream_t stream) {
  const int grid = fwd_grid_size(p, num_sms);
  const bool pw = p.score == BSM_SCORE_POINTWISE;
  // Softmax turns alternate between the tiles only where work units are
  // long: no segment ids and at least 4096 keys.  Packed sequences and
  // short sequences give short units, where the alternation costs more
  // than it saves.  Arbitrary masks take the other instance too, which
  // keeps the alternating one free of per-element keep bits; head dim 64
  // is built without it.
  const bool pp = (p.flags & BSM_MASK_SEGMENT) == 0 && p.Skv >= 4096 &&
                  p.dense == nullptr && p.D == 128;
  // Packed sequences (segment ids, no arbitrary mask) at head dim 128 take
  // the kernel with decoupled query tiles, and so do the other masks below
  // 4096 keys (causal S=2048: 11 % faster there; from 4096 keys on, the
  // lockstep kernel's shared K/V stream is 2-6 % faster).
  const bool dt = p.dense == nullptr && p.D == 128 &&
                  ((p.flags & BSM_MASK_SEGMENT) != 0 || p.Skv < 4096);
  if (dt)
    return pw ? launch_dt<BSM_SCORE_POINTWISE>(p, tq, tk, tv, grid, stream)
              : launch_dt<BSM_SCORE_SOFTMAX>(p, tq, tk, tv, grid, stream);
  if (p.D == 128) {
    if (pw)
      return pp ? launch_one<128, BSM_SCORE_POINTWISE, true>(p, tq, tk, tv, grid, stream)
                : launch_one<128, BSM_SCORE_POINTWISE, false>(p, tq, tk, tv, grid, stream);
    return pp ? launch_one<128, BSM_SCORE_SOFTMAX, true>(p, tq, tk, tv, grid, stream)
              : launch_one<128, BSM_SCORE_SOFTMAX, false>(p, tq, tk, tv, grid, stream);
  }
  if (p.D == 64) {  // head dim 64 uses the instance without alternation
    return pw ? launch_one<64, BSM_SCORE_POINTWISE, false>(p, tq, tk, tv, grid, stream)
              : launch_one<64, BSM_SCORE_SOFTMAX, false>(p, tq, tk, tv, grid, stream);
  }
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
