// Device mask-info builder.
//
// Classifies every (q-block, kv-block) of the mask as empty (0), partial (1)
// or full (2) -- the encoding of hstu_ops `_next_nonzero` -- and emits the
// next-block table (splash notes section 21: an empty step points at the
// next nonzero block) plus per-row CSR lists of the nonzero blocks.
//
// Two launches for masks of up to 2^20 block cells (every workload here):
//   classify: one CTA per (table, q-block row).  Causal/local blocks are
//      classified exactly from the range of q - k over the block.  With
//      segment ids the CTA first stages the table's kv ids in shared memory
//      (up to kStagedKeys of them), checks that they are non-decreasing, and
//      finds for each of its query rows the first and last key with the
//      row's id (binary search; exact for sorted ids, as for packed
//      sequences).  With sorted ids every row's visible keys form one
//      interval, so a block is classified from its rows' intervals; with
//      unsorted ids the min/max of the ids settle most blocks and the rest
//      are scanned element by element.  Writes block_mask, data_next, the
//      row's nonzero count, the rows' segment ranges, the table's "not
//      sorted" bit and the row's nonzero list, compacted, into a staging
//      area.  Then it takes a ticket; the CTA that finishes last turns the
//      counts into CSR row offsets, ORs the tables' "not sorted" bits into
//      seg_flags[0] and orders the super-tiles (finish_tables).  The ticket
//      word is (epoch, count): each build brings a new epoch, installed by
//      the first CTA to start, so a stale word from an earlier build, or
//      garbage, is never counted; the last CTA puts the count back to zero,
//      so a replay of the same launch (same epoch) starts from zero too.
//   copy: a warp per row moves the staged list to its CSR place.  Launched
//      with programmatic stream serialization, so it is scheduled while
//      classify runs and waits (griddepcontrol.wait) for its completion.
// Larger masks take three launches: classify, then one CTA for the offsets
// and the order (finish_tables), then one CTA per row writes the ascending
// nonzero list from block_mask.
#include <cstdint>

#include "bsm_internal.h"

namespace bsm {
namespace {

constexpr int kMiThreads = 512;
constexpr int kStagedKeys = 32768;  // kv ids staged in shared memory (128 KB)
// Masks of at most this many block cells (and fewer than 2^24 rows) are
// built in one launch.
constexpr int64_t kFusedCells = int64_t{1} << 20;
constexpr int kTicketBits = 24;  // count bits of the (epoch, count) word

__host__ __device__ constexpr int cls_bytes(int nk) { return (nk + 15) & ~15; }

// First index in ks[0, n) whose id is >= v (or > v with `after`).
__device__ __forceinline__ int id_search(const int32_t* ks, int n, int v,
                                         bool after) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int x = ks[mid];
    if (x < v || (after && x == v)) lo = mid + 1; else hi = mid;
  }
  return lo;
}
constexpr int kNegInf = -(1 << 30);
constexpr int kPosInf = (1 << 30);

struct BlockRange {
  int r0, r1, c0, c1;  // inclusive, clipped to the sequence
  bool ragged;
};

__device__ __forceinline__ BlockRange block_range(const MaskInfoParams& p,
                                                  int i, int j) {
  BlockRange br;
  br.r0 = i * p.bq;
  br.r1 = min(p.Sq, br.r0 + p.bq) - 1;
  br.c0 = j * p.bkv;
  br.c1 = min(p.Skv, br.c0 + p.bkv) - 1;
  br.ragged = (br.r1 - br.r0 + 1 != p.bq) || (br.c1 - br.c0 + 1 != p.bkv);
  return br;
}

// Causal/local part: every integer d = q - k in [r0 - c1, r1 - c0] occurs in
// the (clipped) block; the allowed set is [lo, hi].
__device__ __forceinline__ int base_class(const MaskInfoParams& p,
                                          const BlockRange& br) {
  const int lo = (p.flags & BSM_MASK_CAUSAL) ? 0
                 : (p.flags & BSM_MASK_BAND) ? 1 - p.window
                                             : kNegInf;
  const int hi = (p.flags & BSM_MASK_LOCAL) ? p.window - 1 : kPosInf;
  const int dmin = br.r0 - br.c1, dmax = br.r1 - br.c0;
  if (dmax < lo || dmin > hi) return 0;
  return (dmin >= lo && dmax <= hi && !br.ragged) ? 2 : 1;
}

__device__ __forceinline__ bool base_visible(const MaskInfoParams& p, int q,
                                             int k) {
  bool v = true;
  if (p.flags & BSM_MASK_CAUSAL) v = v && (k <= q);
  if (p.flags & BSM_MASK_LOCAL) v = v && (q - k < p.window);
  if (p.flags & BSM_MASK_BAND) v = v && (k - q < p.window);
  return v;
}

// Shared scratch of finish_tables.
struct FinishScratch {
  int warp_sums[32];
  int carry;
  uint32_t wmax;
  int any_unsorted;
};

// Run by one CTA (any multiple of 32 threads): inclusive scan of the row
// counts in row_ptr[1..R] in place (row_ptr[0] = 0), giving the CSR
// offsets; the OR of the tables' "not sorted" bits; then, if requested, the
// order in which the forward should take its 256-row super-tiles: by
// decreasing work (sum over the super-tile's rows of the nonzero blocks they
// see), so that the longest units start first and the short ones fill in at
// the end.  `keys` holds kMaxSuperOrder words of shared memory; the work of
// each (table, super-tile) pair is summed there while the counts are scanned
// and then turned into its sort key in place.
__device__ __forceinline__ void finish_tables(const MaskInfoParams& p,
                                              FinishScratch& fs,
                                              uint32_t* keys) {
  int32_t* row_ptr = p.row_ptr;
  const int R = p.tables * p.nq;
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int nwarps = blockDim.x / 32;
  const bool order = p.super_order != nullptr;
  const int pairs = p.tables * p.n_super;  // <= kMaxSuperOrder when ordered
  // the "not sorted" bits are read alongside the first counts
  int unsorted = 0;
  if (p.flags & BSM_MASK_SEGMENT)
    for (int tb = threadIdx.x; tb < p.tables; tb += blockDim.x)
      unsorted |= p.seg_flags[1 + tb];
  if (order)
    for (int i = threadIdx.x; i < pairs; i += blockDim.x) keys[i] = 0;
  if (threadIdx.x == 0) {
    row_ptr[0] = 0;
    fs.carry = 0;
    fs.wmax = 0;
  }
  fs.any_unsorted = 0;
  __syncthreads();
  if (unsorted) fs.any_unsorted = 1;
  for (int base = 0; base < R; base += blockDim.x) {
    const int idx = base + threadIdx.x;
    const int cnt = idx < R ? row_ptr[idx + 1] : 0;
    if (order && idx < R && cnt > 0) {
      // this block row's share of each super-tile it overlaps
      const int t = idx / p.nq, i = idx - t * p.nq;
      const int r0 = i * p.bq, r1 = min(p.Sq, r0 + p.bq);  // [r0, r1)
      for (int st = r0 / kUnitRows; st * kUnitRows < r1; ++st) {
        const int rows = min(r1, (st + 1) * kUnitRows) - max(r0, st * kUnitRows);
        atomicAdd(&keys[t * p.n_super + st], static_cast<uint32_t>(cnt * rows));
      }
    }
    int v = cnt;
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    if (lane == 31) fs.warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int sum = lane < nwarps ? fs.warp_sums[lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, sum, o);
        if (lane >= o) sum += n;
      }
      fs.warp_sums[lane] = sum;
    }
    __syncthreads();
    const int carry = fs.carry;
    const int prefix = (warp > 0 ? fs.warp_sums[warp - 1] : 0) + carry;
    if (idx < R) row_ptr[idx + 1] = v + prefix;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) fs.carry = carry + fs.warp_sums[nwarps - 1];
    __syncthreads();
  }
  __syncthreads();
  if ((p.flags & BSM_MASK_SEGMENT) && threadIdx.x == 0)
    p.seg_flags[0] = fs.any_unsorted;
  if (!order) return;

  // ---- longest-first order of the (table, super-tile) pairs
  uint32_t wm = 0;
  for (int pr = threadIdx.x; pr < pairs; pr += blockDim.x) wm = max(wm, keys[pr]);
  for (int o = 16; o > 0; o >>= 1) wm = max(wm, __shfl_xor_sync(0xffffffffu, wm, o));
  if (lane == 0 && wm > 0) atomicMax(&fs.wmax, wm);
  __syncthreads();
  const unsigned long long wmax = fs.wmax > 0 ? fs.wmax : 1;
  int n2 = 1;
  while (n2 < pairs) n2 <<= 1;
  // key: complemented 19-bit work above the complemented 13-bit index, so
  // an ascending sort gives decreasing work and, among equals, decreasing
  // index (later rows first, as for a causal mask)
  for (int i = threadIdx.x; i < n2; i += blockDim.x) {
    uint32_t key = 0xffffffffu;
    if (i < pairs) {
      const unsigned long long q = keys[i] * 0x7ffffull / wmax;
      key = (static_cast<uint32_t>(0x7ffffull - q) << 13) |
            (0x1fffu - static_cast<uint32_t>(i));
    }
    keys[i] = key;
  }
  __syncthreads();
  if (pairs <= static_cast<int>(blockDim.x)) {
    // few pairs: each key's rank is the number of smaller keys (the index
    // bits make the keys of distinct pairs distinct); one pass, no barriers
    if (static_cast<int>(threadIdx.x) < pairs) {
      const uint32_t mine = keys[threadIdx.x];
      int rank = 0;
#pragma unroll 8
      for (int j = 0; j < pairs; ++j) rank += keys[j] < mine ? 1 : 0;
      p.super_order[rank] = static_cast<int32_t>(threadIdx.x);
    }
    return;
  }
  // bitonic sort of keys[0..n2)
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int l = i ^ j;
        if (l > i) {
          const uint32_t a = keys[i], b = keys[l];
          const bool up = (i & k) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < pairs; i += blockDim.x)
    p.super_order[i] = static_cast<int32_t>(0x1fffu - (keys[i] & 0x1fffu));
}

__global__ void __launch_bounds__(kMiThreads)
    mi_classify_kernel(const MaskInfoParams p) {
  extern __shared__ __align__(16) uint8_t dyn_s[];
  int8_t* cls_s = reinterpret_cast<int8_t*>(dyn_s);  // [nk]
  __shared__ int qseg_s[512];
  __shared__ int2 sr_s[512];
  __shared__ int red_min[kMiThreads / 32], red_max[kMiThreads / 32];
  __shared__ int cnt_s;

  const int i = blockIdx.x, t = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const bool seg = (p.flags & BSM_MASK_SEGMENT) != 0;
  const int r0 = i * p.bq, r1 = min(p.Sq, r0 + p.bq) - 1;
  // the copy kernel that follows may be scheduled now: it waits for this
  // grid's completion before reading anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Ticket, part one: install this build's epoch if the word still holds
  // another one.  Issued first so that its round trips overlap the loads
  // below; the same thread counts this CTA at the end, after it.
  if (p.fused && threadIdx.x == 0) {
    const unsigned long long mine = p.epoch << kTicketBits;
    const unsigned long long cur =
        *reinterpret_cast<volatile unsigned long long*>(p.ticket);
    if ((cur >> kTicketBits) != p.epoch) atomicCAS(p.ticket, cur, mine);
  }

  // The kv ids of this table are staged in shared memory when they fit; their
  // loads are issued together with the row block's q ids, so that one
  // barrier covers both.
  const int32_t* ks = nullptr;
  const bool staged = seg && p.Skv <= kStagedKeys;
  if (seg) {
    const int32_t* ks_g = p.kv_seg + static_cast<int64_t>(t) * p.Skv;
    ks = ks_g;
    if (staged) {
      int32_t* ks_s = reinterpret_cast<int32_t*>(dyn_s + cls_bytes(p.nk));
      // 16-byte loads, unrolled so that all of a thread's loads are in
      // flight at once (the ids of a table are read by every row's CTA)
      int k0 = 0;
      if ((reinterpret_cast<uintptr_t>(ks_g) & 15u) == 0) {
        const int n4 = p.Skv / 4;
        const int4* g4 = reinterpret_cast<const int4*>(ks_g);
        int4* s4 = reinterpret_cast<int4*>(ks_s);
#pragma unroll 8
        for (int k = threadIdx.x; k < n4; k += blockDim.x) s4[k] = __ldg(g4 + k);
        k0 = 4 * n4;
      }
      for (int k = k0 + threadIdx.x; k < p.Skv; k += blockDim.x)
        ks_s[k] = ks_g[k];
      ks = ks_s;
    }
  }

  int qmin = kPosInf, qmax = kNegInf;
  if (seg) {
    const int32_t* qs = p.q_seg + static_cast<int64_t>(t) * p.Sq;
    for (int r = r0 + threadIdx.x; r <= r1; r += blockDim.x) {
      const int v = qs[r];
      qseg_s[r - r0] = v;
      qmin = min(qmin, v);
      qmax = max(qmax, v);
    }
    for (int o = 16; o > 0; o >>= 1) {
      qmin = min(qmin, __shfl_xor_sync(0xffffffffu, qmin, o));
      qmax = max(qmax, __shfl_xor_sync(0xffffffffu, qmax, o));
    }
    if (lane == 0) {
      red_min[warp] = qmin;
      red_max[warp] = qmax;
    }
  }
  if (threadIdx.x == 0) cnt_s = 0;
  __syncthreads();
  if (seg) {
    qmin = red_min[0];
    qmax = red_max[0];
    for (int w = 1; w < kMiThreads / 32; ++w) {
      qmin = min(qmin, red_min[w]);
      qmax = max(qmax, red_max[w]);
    }
  }

  bool sorted = true;
  if (seg) {
    bool unsorted = false;
#pragma unroll 8
    for (int k = threadIdx.x; k + 1 < p.Skv; k += blockDim.x)
      unsorted |= ks[k] > ks[k + 1];
    sorted = !__syncthreads_or(unsorted);
    if (i == 0 && threadIdx.x == 0) p.seg_flags[1 + t] = sorted ? 0 : 1;
    // each row's [first, last] key with its id (first > last: none); the
    // two searches of a row run on different threads
    const int nrows = r1 - r0 + 1;
    for (int e = threadIdx.x; e < 2 * nrows; e += blockDim.x) {
      const bool after = e >= nrows;
      const int r = after ? e - nrows : e;
      const int x = id_search(ks, p.Skv, qseg_s[r], after);
      if (after) sr_s[r].y = x - 1; else sr_s[r].x = x;
    }
    __syncthreads();
    int2* sr_g = reinterpret_cast<int2*>(p.seg_range) +
                 static_cast<int64_t>(t) * p.Sq;
    for (int r = threadIdx.x; r < nrows; r += blockDim.x) sr_g[r0 + r] = sr_s[r];
  }
  const bool ranges = seg && sorted;

  // One warp per block (i, j).
  int my_count = 0;
  for (int j = warp; j < p.nk; j += kMiThreads / 32) {
    const BlockRange br = block_range(p, i, j);
    int c = base_class(p, br);
    if (p.dense != nullptr && c != 0 && (!seg || ranges)) {
      // arbitrary mask, every other predicate a key interval per row: count
      // the row's mask bits inside its interval, a word at a time
      bool any = false, all = !br.ragged;
      for (int q = br.r0 + lane; q <= br.r1; q += 32) {
        int lo = br.c0, hi = br.c1;
        if (ranges) {
          lo = max(lo, sr_s[q - br.r0].x);
          hi = min(hi, sr_s[q - br.r0].y);
        }
        if (p.flags & BSM_MASK_CAUSAL) hi = min(hi, q);
        if (p.flags & BSM_MASK_LOCAL) lo = max(lo, q - p.window + 1);
        if (p.flags & BSM_MASK_BAND) hi = min(hi, q + p.window - 1);
        int n = 0;
        if (hi >= lo) {
          const uint32_t* row = p.dense + static_cast<int64_t>(q) * p.dense_words;
          for (int wd = lo >> 5; wd <= (hi >> 5); ++wd) {
            const int base = wd << 5;
            const int lb = max(lo - base, 0);        // < 32
            const int hb = min(hi - base + 1, 32);   // >= 1
            const uint32_t m = (hb >= 32 ? 0xffffffffu : (1u << hb) - 1u) &
                               ~((1u << lb) - 1u);
            n += __popc(__ldg(row + wd) & m);
          }
        }
        any |= n > 0;
        all &= n == p.bkv;
      }
      any = __any_sync(0xffffffffu, any);
      all = __all_sync(0xffffffffu, all);
      c = any ? (all ? 2 : 1) : 0;
    } else if (p.dense != nullptr && c != 0) {
      // arbitrary mask with unsorted segment ids: exact element scan with
      // every predicate (columns past Skv and rows past Sq are invisible)
      bool any = false, all = !br.ragged;
      for (int cb = 0; cb < p.bkv; cb += 32) {
        const int k = br.c0 + cb + lane;
        const bool kin = (cb + lane < p.bkv) && (k <= br.c1);
        const int kv = (seg && kin) ? ks[k] : 0;
        for (int r = br.r0; r <= br.r1; ++r) {
          bool v = kin && base_visible(p, r, k) &&
                   ((p.dense[static_cast<int64_t>(r) * p.dense_words +
                             (k >> 5)] >>
                     (k & 31)) &
                    1u);
          if (seg) v = v && qseg_s[r - br.r0] == kv;
          any |= v;
          all &= v || (cb + lane >= p.bkv);
        }
        const bool wany = __any_sync(0xffffffffu, any);
        const bool wall = __all_sync(0xffffffffu, all);
        if (wany && !wall) break;  // already known to be partial
      }
      any = __any_sync(0xffffffffu, any);
      all = __all_sync(0xffffffffu, all);
      c = any ? (all ? 2 : 1) : 0;
    } else if (ranges && c != 0) {
      // each row sees one interval of keys: count it inside the block
      bool any = false, all = !br.ragged;
      for (int q = br.r0 + lane; q <= br.r1; q += 32) {
        int lo = max(br.c0, sr_s[q - br.r0].x),
            hi = min(br.c1, sr_s[q - br.r0].y);
        if (p.flags & BSM_MASK_CAUSAL) hi = min(hi, q);
        if (p.flags & BSM_MASK_LOCAL) lo = max(lo, q - p.window + 1);
        if (p.flags & BSM_MASK_BAND) hi = min(hi, q + p.window - 1);
        const int n = hi >= lo ? hi - lo + 1 : 0;
        any |= n > 0;
        all &= n == p.bkv;
      }
      any = __any_sync(0xffffffffu, any);
      all = __all_sync(0xffffffffu, all);
      c = any ? (all ? 2 : 1) : 0;
    } else if (seg && c != 0) {
      int kmin = kPosInf, kmax = kNegInf;
      for (int k = br.c0 + lane; k <= br.c1; k += 32) {
        const int v = ks[k];
        kmin = min(kmin, v);
        kmax = max(kmax, v);
      }
      for (int o = 16; o > 0; o >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
        kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
      }
      if (qmax < kmin || qmin > kmax) {
        c = 0;  // no id occurs on both sides
      } else if (qmin == qmax && kmin == kmax) {
        // one segment covers the whole block: the causal/local class stands
      } else {
        // exact element scan; columns past Skv and rows past Sq are
        // invisible, so a ragged block is never full
        bool any = false, all = !br.ragged;
        for (int cb = 0; cb < p.bkv; cb += 32) {
          const int k = br.c0 + cb + lane;
          const bool kin = (cb + lane < p.bkv) && (k <= br.c1);
          const int kv = kin ? ks[k] : 0;
          for (int r = br.r0; r <= br.r1; ++r) {
            const bool v = kin && base_visible(p, r, k) && qseg_s[r - br.r0] == kv;
            any |= v;
            all &= v || (cb + lane >= p.bkv);
          }
          const bool wany = __any_sync(0xffffffffu, any);
          const bool wall = __all_sync(0xffffffffu, all);
          if (wany && !wall) break;  // already known to be partial
        }
        any = __any_sync(0xffffffffu, any);
        all = __all_sync(0xffffffffu, all);
        c = any ? (all ? 2 : 1) : 0;
      }
    }
    if (lane == 0) {
      cls_s[j] = static_cast<int8_t>(c);
      my_count += (c != 0);
    }
  }
  if (lane == 0 && my_count) atomicAdd(&cnt_s, my_count);
  __syncthreads();

  const int64_t row = static_cast<int64_t>(t) * p.nq + i;
  int8_t* bm = p.block_mask + row * p.nk;
  for (int j = threadIdx.x; j < p.nk; j += blockDim.x) bm[j] = cls_s[j];
  if (threadIdx.x == 0) p.row_ptr[row + 1] = cnt_s;

  // The row's nonzero list (ascending, uint16 `j << 2 | class`), staged at
  // row * nk for the finishing CTA, warp 1.
  if (p.fused && warp == 1) {
    uint16_t* st = p.staged + row * p.nk;
    int base = 0;
    for (int j0 = 0; j0 < p.nk; j0 += 32) {
      const int j = j0 + lane;
      const int c = j < p.nk ? cls_s[j] : 0;
      const unsigned m = __ballot_sync(0xffffffffu, c != 0);
      if (c != 0)
        st[base + __popc(m & ((1u << lane) - 1u))] =
            static_cast<uint16_t>((j << 2) | c);
      base += __popc(m);
    }
  }
  // Next-block table, warp 0, right to left in chunks of 32.
  if (warp == 0) {
    int32_t* dn = p.data_next + row * p.nk;
    const int nchunks = (p.nk + 31) / 32;
    int last_nz = -1;
    for (int ch = nchunks - 1; ch >= 0 && last_nz < 0; --ch) {
      const int j = ch * 32 + lane;
      const unsigned m = __ballot_sync(0xffffffffu, j < p.nk && cls_s[j] != 0);
      if (m) last_nz = ch * 32 + 31 - __clz(m);
    }
    int carry = -1;  // nearest nonzero to the right of the current chunk
    for (int ch = nchunks - 1; ch >= 0; --ch) {
      const int j = ch * 32 + lane;
      const unsigned m = __ballot_sync(0xffffffffu, j < p.nk && cls_s[j] != 0);
      const unsigned hi = m & (0xffffffffu << lane);
      int nxt = hi ? ch * 32 + __ffs(hi) - 1 : carry;
      if (nxt < 0) nxt = last_nz < 0 ? 0 : last_nz;
      if (j < p.nk) dn[j] = nxt;
      if (m) carry = ch * 32 + __ffs(m) - 1;
    }
  }
  if (!p.fused) return;

  // ---- ticket, part two: the CTA that finishes last completes the tables.
  // Every thread's writes are made visible device-wide before the CTA counts
  // itself; the word holds (epoch << kTicketBits) | CTAs counted, so a word
  // from an earlier build (another epoch) counts as zero.  Each CTA installed
  // the epoch (or found it installed) before counting, and within a build
  // only that swap changes the epoch, so no count is lost to it.  The last
  // CTA puts the count back to zero, so that a replay of the same launch
  // (same epoch) counts from zero as well.
  __shared__ int last_s;
  __shared__ FinishScratch fs;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int total = p.nq * p.tables;
    const unsigned long long got = atomicAdd(p.ticket, 1ull);
    const bool ok = (got >> kTicketBits) == p.epoch;
    last_s = (ok && static_cast<int>(got & ((1ull << kTicketBits) - 1)) ==
                        total - 1) ? 1 : 0;
    __threadfence();
  }
  __syncthreads();
  if (!last_s) return;
  if (threadIdx.x == 0) atomicExch(p.ticket, p.epoch << kTicketBits);
  finish_tables(p, fs, reinterpret_cast<uint32_t*>(dyn_s));
}

// Moves each row's staged nonzero list to its CSR place, a warp per row
// (second launch of the build; it waits for the first, whose last CTA wrote
// the offsets).
__global__ void __launch_bounds__(kMiThreads)
    mi_copy_kernel(const MaskInfoParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int R = p.tables * p.nq;
  const int row = blockIdx.x * (kMiThreads / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= R) return;
  const int start = p.row_ptr[row], cnt = p.row_ptr[row + 1] - start;
  const uint16_t* st = p.staged + static_cast<int64_t>(row) * p.nk;
  for (int k = lane; k < cnt; k += 32) {
    const uint32_t e = st[k];
    p.kv_idx[start + k] = static_cast<int32_t>(e >> 2);
    p.kv_cls[start + k] = static_cast<int8_t>(e & 3u);
  }
}

// Offsets and order of a mask too large for the one-launch build.
__global__ void __launch_bounds__(1024) mi_scan_kernel(const MaskInfoParams p) {
  __shared__ FinishScratch fs;
  __shared__ uint32_t keys[kMaxSuperOrder];
  finish_tables(p, fs, keys);
}

// Ascending list of the nonzero blocks of one row.
__global__ void __launch_bounds__(kMiThreads)
    mi_compact_kernel(const MaskInfoParams p) {
  __shared__ int warp_cnt[kMiThreads / 32];
  const int i = blockIdx.x, t = blockIdx.y;
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int64_t row = static_cast<int64_t>(t) * p.nq + i;
  const int8_t* bm = p.block_mask + row * p.nk;
  int base = p.row_ptr[row];
  for (int j0 = 0; j0 < p.nk; j0 += blockDim.x) {
    const int j = j0 + threadIdx.x;
    const int8_t c = j < p.nk ? bm[j] : 0;
    const unsigned m = __ballot_sync(0xffffffffu, c != 0);
    if (lane == 0) warp_cnt[warp] = __popc(m);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kMiThreads / 32; ++w) {
      before += (w < warp) ? warp_cnt[w] : 0;
      total += warp_cnt[w];
    }
    if (c != 0) {
      const int pos = base + before + __popc(m & ((1u << lane) - 1u));
      p.kv_idx[pos] = j;
      p.kv_cls[pos] = c;
    }
    base += total;
    __syncthreads();
  }
}

// Bit-packs a boolean mask, one thread per output word: bit i of word w of
// row q is mask[q][32 w + i] != 0 (zero past Skv and in row padding).  With
// 16-byte aligned rows a word's 32 bytes are two 16-byte loads, and each
// 4-byte lane becomes 4 bits through a per-byte compare.
__global__ void __launch_bounds__(256)
    pack_dense_kernel(const uint8_t* __restrict__ mask, int64_t stride,
                      int32_t Sq, int32_t Skv, uint32_t* __restrict__ words,
                      int32_t row_words, int vec16) {
  const int64_t total = static_cast<int64_t>(Sq) * row_words;
  for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       w < total; w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t q = w / row_words;
    const int k0 = static_cast<int>(w - q * row_words) * 32;
    const uint8_t* row = mask + q * stride;
    uint32_t bits = 0;
    if (k0 + 32 <= Skv && vec16) {
      const uint4* src = reinterpret_cast<const uint4*>(row + k0);
      const uint4 a = __ldg(src), b = __ldg(src + 1);
      const uint32_t lanes[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t ne = __vcmpne4(lanes[i], 0u);  // 0xff per nonzero byte
        const uint32_t nib = ((ne >> 7) & 1u) | ((ne >> 14) & 2u) |
                             ((ne >> 21) & 4u) | ((ne >> 28) & 8u);
        bits |= nib << (4 * i);
      }
    } else {
      const int n = min(32, Skv - k0);  // <= 0 in the row padding
      for (int i = 0; i < n; ++i) bits |= (row[k0 + i] != 0 ? 1u : 0u) << i;
    }
    words[w] = bits;
  }
}

}  // namespace

cudaError_t launch_pack_dense(const uint8_t* mask, int64_t stride, int32_t Sq,
                              int32_t Skv, uint32_t* words, int32_t row_words,
                              int num_sms, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(Sq) * row_words;
  if (total == 0) return cudaSuccess;
  const int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(blocks < cap ? blocks : cap);
  const int vec16 = ((reinterpret_cast<uintptr_t>(mask) & 15u) == 0 &&
                     (stride & 15) == 0) ? 1 : 0;
  pack_dense_kernel<<<grid, 256, 0, stream>>>(mask, stride, Sq, Skv, words,
                                              row_words, vec16);
  return cudaGetLastError();
}

bool mask_info_fused(int64_t tables, int64_t nq, int64_t nk) {
  return tables * nq < (int64_t{1} << kTicketBits) &&
         tables * nq * nk <= kFusedCells;
}

cudaError_t launch_mask_info(const MaskInfoParams& p, cudaStream_t stream) {
  const int R = p.tables * p.nq;
  if (R == 0) {
    return cudaMemsetAsync(p.row_ptr, 0, sizeof(int32_t), stream);
  }
  cudaError_t e;
  // All of the build's kernels ask for the largest shared-memory carveout,
  // the one the forward runs with, so an SM need not be reconfigured
  // between the build and the forward that follows it.
  for (const void* k : {reinterpret_cast<const void*>(mi_classify_kernel),
                        reinterpret_cast<const void*>(mi_scan_kernel),
                        reinterpret_cast<const void*>(mi_compact_kernel),
                        reinterpret_cast<const void*>(mi_copy_kernel)}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  size_t smem = static_cast<size_t>(cls_bytes(p.nk > 0 ? p.nk : 1));
  if ((p.flags & BSM_MASK_SEGMENT) && p.Skv <= kStagedKeys)
    smem += static_cast<size_t>(p.Skv) * sizeof(int32_t);
  if (p.fused && p.super_order != nullptr) {
    // the finishing CTA sorts the super-tile keys in the same space
    size_t n2 = 1;
    while (n2 < static_cast<size_t>(p.tables) * p.n_super) n2 <<= 1;
    smem = smem > 4 * n2 ? smem : 4 * n2;
  }
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(mi_classify_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  mi_classify_kernel<<<dim3(p.nq, p.tables), kMiThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.fused) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((R + kMiThreads / 32 - 1) / (kMiThreads / 32));
    cfg.blockDim = dim3(kMiThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mi_copy_kernel, p);
  }
  mi_scan_kernel<<<1, 1024, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mi_compact_kernel<<<dim3(p.nq, p.tables), kMiThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace bsm
