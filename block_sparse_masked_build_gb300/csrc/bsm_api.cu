// Host side of the C ABI declared in include/bsm.h: argument validation,
// layout of the caller's mask-info buffer, TMA tensor-map encoding and the
// kernel launches.  Allocates no device memory.
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "bsm_internal.h"

namespace {

thread_local std::string g_last_error;

bsm_status fail(bsm_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

bsm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(BSM_ERR_CUDA,
              std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                  cudaGetErrorString(e) + ")");
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool is_block_size(int32_t b) {
  return b >= 16 && b <= 512 && (b & (b - 1)) == 0;
}

struct MiLayout {
  size_t off_bm, off_dn, off_rp, off_idx, off_cls, off_sr, off_sf, off_so,
      off_stage, off_ticket, total;
};

// seg_rows = B * Sq with segment ids, else 0.
int64_t super_pairs(int64_t tables, int64_t Sq) {
  return tables * ((Sq + bsm::kUnitRows - 1) / bsm::kUnitRows);
}

MiLayout mi_layout(int64_t tables, int64_t nq, int64_t nk, int64_t seg_rows,
                   int64_t pairs) {
  const size_t cells = static_cast<size_t>(tables * nq * nk);
  const size_t rows = static_cast<size_t>(tables * nq);
  MiLayout L;
  size_t o = 0;
  L.off_bm = o;
  o = align_up(o + cells, 256);
  L.off_dn = o;
  o = align_up(o + cells * 4, 256);
  L.off_rp = o;
  o = align_up(o + (rows + 1) * 4, 256);
  L.off_idx = o;
  o = align_up(o + cells * 4, 256);
  L.off_cls = o;
  o = align_up(o + cells, 256);
  L.off_sr = o;
  o = align_up(o + static_cast<size_t>(seg_rows) * 8, 256);
  L.off_sf = o;  // [0]: any table unsorted; [1 + t]: table t (builder scratch)
  o = align_up(o + 4 * (1 + (seg_rows > 0 ? tables : 0)), 256);
  L.off_so = o;
  if (pairs <= bsm::kMaxSuperOrder)
    o = align_up(o + static_cast<size_t>(pairs) * 4, 256);
  // one-launch build: the rows' staged lists and the (epoch, count) ticket
  L.off_stage = o;
  L.off_ticket = o;
  if (bsm::mask_info_fused(tables, nq, nk)) {
    o = align_up(o + cells * 2, 256);
    L.off_ticket = o;
    o = align_up(o + 8, 256);
  }
  L.total = o;
  return L;
}

bsm_status check_spec(const bsm_mask_spec* spec) {
  if (spec == nullptr) return fail(BSM_ERR_INVALID_ARG, "mask spec is NULL");
  const uint32_t known = BSM_MASK_CAUSAL | BSM_MASK_LOCAL | BSM_MASK_SEGMENT |
                         BSM_MASK_BAND | BSM_MASK_DENSE;
  if (spec->flags & ~known)
    return fail(BSM_ERR_INVALID_ARG, "unknown mask flag bits");
  if ((spec->flags & BSM_MASK_BAND) && !(spec->flags & BSM_MASK_LOCAL))
    return fail(BSM_ERR_INVALID_ARG, "BSM_MASK_BAND needs BSM_MASK_LOCAL");
  if ((spec->flags & BSM_MASK_LOCAL) && spec->window < 1)
    return fail(BSM_ERR_INVALID_ARG, "local window must be >= 1");
  return BSM_OK;
}

bsm_status check_mi_shape(const bsm_mask_spec* spec, int32_t B, int32_t Sq,
                          int32_t Skv, int32_t bq, int32_t bkv) {
  bsm_status s = check_spec(spec);
  if (s != BSM_OK) return s;
  if (B < 0 || Sq < 0 || Skv < 0)
    return fail(BSM_ERR_INVALID_ARG, "negative size");
  if (Sq > bsm::kMaxSeq || Skv > bsm::kMaxSeq)
    return fail(BSM_ERR_UNSUPPORTED, "sequence length above 262144");
  if (!is_block_size(bq) || !is_block_size(bkv))
    return fail(BSM_ERR_INVALID_ARG,
                "block_q and block_kv must be powers of two in [16, 512]");
  return BSM_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 4-D bf16 map over [B][H][S][D] storage with element strides (sb, sh, ss);
// box = 64 head-dim elements (128 bytes, 128-byte swizzle) x 128 rows.
bsm_status make_map(CUtensorMap* map, const void* ptr, int32_t B, int32_t H,
                    int32_t S, int32_t D, const int64_t strides[3],
                    const char* name) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr)
    return fail(BSM_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  // Strides of size-1 dimensions are never used; give them a valid value.
  const int64_t ss = S > 1 ? strides[2] : D;
  const int64_t sh = H > 1 ? strides[1] : ss * S;
  const int64_t sb = B > 1 ? strides[0] : sh * H;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t gstr[3] = {static_cast<cuuint64_t>(ss * 2),
                        static_cast<cuuint64_t>(sh * 2),
                        static_cast<cuuint64_t>(sb * 2)};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(bsm::kTileM), 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void*>(ptr), dims, gstr, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(BSM_ERR_INVALID_ARG,
                std::string("tensor map for ") + name +
                    " rejected (strides must be multiples of 8 elements)");
  return BSM_OK;
}

bsm_status check_device(int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3)
    return fail(BSM_ERR_UNSUPPORTED,
                "libbsm is built for sm_103a (GB300) only; device is sm_" +
                    std::to_string(major) + std::to_string(minor));
  if (num_sms) *num_sms = sms;
  return BSM_OK;
}

uint64_t wait_timeout_ns() {
  static uint64_t v = [] {
    const char* s = std::getenv("BSM_WAIT_TIMEOUT_NS");
    if (s != nullptr) {
      const unsigned long long x = std::strtoull(s, nullptr, 10);
      if (x >= 1000ull && x <= 100000000000ull) return static_cast<uint64_t>(x);
    }
    return static_cast<uint64_t>(2000000000ull);  // 2 s
  }();
  return v;
}

std::mutex g_trace_mu;
void* g_trace_buf = nullptr;
size_t g_trace_bytes = 0;

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// A new epoch for every mask-info build (40 bits, never 0), starting at a
// value that differs between processes, so that a ticket word left in a
// reused buffer by an earlier build never matches.
uint64_t next_build_epoch() {
  static std::atomic<uint64_t> counter{
      (static_cast<uint64_t>(
           std::chrono::steady_clock::now().time_since_epoch().count()) *
       0x9E3779B97F4A7C15ull) ^
      static_cast<uint64_t>(reinterpret_cast<uintptr_t>(&counter))};
  constexpr uint64_t kMask = (uint64_t{1} << 40) - 1;
  uint64_t e = 0;
  while (e == 0) e = counter.fetch_add(1, std::memory_order_relaxed) & kMask;
  return e;
}

}  // namespace

namespace bsm {
void set_last_error(const char* msg) { g_last_error = msg; }
}  // namespace bsm

extern "C" {

size_t bsm_mask_info_bytes(const bsm_mask_spec* spec, int32_t B, int32_t Sq,
                           int32_t Skv, int32_t block_q, int32_t block_kv) {
  if (check_mi_shape(spec, B, Sq, Skv, block_q, block_kv) != BSM_OK) return 0;
  const bool seg = (spec->flags & BSM_MASK_SEGMENT) != 0;
  const int64_t tables = seg ? B : 1;
  const int64_t nq = (Sq + block_q - 1) / block_q;
  const int64_t nk = (Skv + block_kv - 1) / block_kv;
  return mi_layout(tables, nq, nk, seg ? static_cast<int64_t>(B) * Sq : 0,
                   super_pairs(tables, Sq))
      .total;
}

bsm_status bsm_build_mask_info(const bsm_mask_spec* spec,
                               const int32_t* q_segment_ids,
                               const int32_t* kv_segment_ids, int32_t B,
                               int32_t Sq, int32_t Skv, int32_t block_q,
                               int32_t block_kv, void* buffer,
                               size_t buffer_bytes, bsm_mask_info* info,
                               void* stream) {
  g_last_error.clear();
  bsm_status s = check_mi_shape(spec, B, Sq, Skv, block_q, block_kv);
  if (s != BSM_OK) return s;
  if (info == nullptr) return fail(BSM_ERR_INVALID_ARG, "info is NULL");
  const bool seg = (spec->flags & BSM_MASK_SEGMENT) != 0;
  if (seg && (q_segment_ids == nullptr || kv_segment_ids == nullptr))
    return fail(BSM_ERR_INVALID_ARG,
                "BSM_MASK_SEGMENT needs both q and kv segment ids");
  if (!seg && (q_segment_ids != nullptr || kv_segment_ids != nullptr))
    return fail(BSM_ERR_INVALID_ARG,
                "segment ids given without BSM_MASK_SEGMENT");
  if (seg && B < 1) return fail(BSM_ERR_INVALID_ARG, "B must be >= 1");
  const bool dense = (spec->flags & BSM_MASK_DENSE) != 0;
  if (dense && (spec->dense_bits == nullptr ||
                spec->dense_row_words < (static_cast<int64_t>(Skv) + 31) / 32))
    return fail(BSM_ERR_INVALID_ARG,
                "BSM_MASK_DENSE needs dense_bits and dense_row_words >= "
                "ceil(Skv / 32)");
  const int64_t tables = seg ? B : 1;
  const int64_t nq = (Sq + block_q - 1) / block_q;
  const int64_t nk = (Skv + block_kv - 1) / block_kv;
  if (tables > 65535)
    return fail(BSM_ERR_UNSUPPORTED, "too many mask tables");
  const int64_t pairs = super_pairs(tables, Sq);
  const MiLayout L = mi_layout(
      tables, nq, nk, seg ? static_cast<int64_t>(B) * Sq : 0, pairs);
  if (buffer == nullptr) return fail(BSM_ERR_INVALID_ARG, "buffer is NULL");
  if ((reinterpret_cast<uintptr_t>(buffer) & 255u) != 0)
    return fail(BSM_ERR_INVALID_ARG, "buffer must be 256-byte aligned");
  if (buffer_bytes < L.total)
    return fail(BSM_ERR_INVALID_ARG,
                "buffer too small: need " + std::to_string(L.total) +
                    " bytes");
  s = check_device(nullptr);
  if (s != BSM_OK) return s;

  uint8_t* base = static_cast<uint8_t*>(buffer);
  bsm_mask_info mi;
  mi.flags = spec->flags;
  mi.window = (spec->flags & BSM_MASK_LOCAL) ? spec->window : 0;
  mi.num_tables = static_cast<int32_t>(tables);
  mi.Sq = Sq;
  mi.Skv = Skv;
  mi.block_q = block_q;
  mi.block_kv = block_kv;
  mi.nq = static_cast<int32_t>(nq);
  mi.nk = static_cast<int32_t>(nk);
  mi.block_mask = reinterpret_cast<int8_t*>(base + L.off_bm);
  mi.data_next = reinterpret_cast<int32_t*>(base + L.off_dn);
  mi.row_ptr = reinterpret_cast<int32_t*>(base + L.off_rp);
  mi.kv_idx = reinterpret_cast<int32_t*>(base + L.off_idx);
  mi.kv_cls = reinterpret_cast<int8_t*>(base + L.off_cls);
  mi.seg_range = reinterpret_cast<int32_t*>(base + L.off_sr);
  mi.seg_flags = reinterpret_cast<int32_t*>(base + L.off_sf);
  mi.num_super = static_cast<int32_t>((Sq + bsm::kUnitRows - 1) / bsm::kUnitRows);
  mi.dense_bits = dense ? spec->dense_bits : nullptr;
  mi.dense_row_words = dense ? spec->dense_row_words : 0;
  mi.super_order = pairs <= bsm::kMaxSuperOrder
                       ? reinterpret_cast<int32_t*>(base + L.off_so)
                       : nullptr;

  bsm::MaskInfoParams p;
  p.flags = mi.flags;
  p.window = mi.window;
  p.Sq = Sq;
  p.Skv = Skv;
  p.bq = block_q;
  p.bkv = block_kv;
  p.nq = mi.nq;
  p.nk = mi.nk;
  p.tables = mi.num_tables;
  p.q_seg = q_segment_ids;
  p.kv_seg = kv_segment_ids;
  p.block_mask = mi.block_mask;
  p.data_next = mi.data_next;
  p.row_ptr = mi.row_ptr;
  p.kv_idx = mi.kv_idx;
  p.kv_cls = mi.kv_cls;
  p.seg_range = mi.seg_range;
  p.seg_flags = mi.seg_flags;
  p.n_super = mi.num_super;
  p.super_order = mi.super_order;
  p.dense = mi.dense_bits;
  p.dense_words = mi.dense_row_words;
  p.fused = bsm::mask_info_fused(tables, nq, nk) ? 1 : 0;
  p.staged = reinterpret_cast<uint16_t*>(base + L.off_stage);
  p.ticket = reinterpret_cast<unsigned long long*>(base + L.off_ticket);
  p.epoch = next_build_epoch();
  cudaError_t e =
      bsm::launch_mask_info(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mask-info launch");
  *info = mi;
  return BSM_OK;
}

bsm_status bsm_splash_fwd(const void* q, const void* k, const void* v,
                          const int64_t q_strides[3],
                          const int64_t k_strides[3],
                          const int64_t v_strides[3],
                          const int64_t o_strides[3], int32_t B, int32_t H,
                          int32_t H_kv, int32_t Sq, int32_t Skv, int32_t D,
                          const bsm_mask_info* info,
                          const int32_t* q_segment_ids,
                          const int32_t* kv_segment_ids, float scale,
                          int32_t score, void* out, float* lse,
                          void* workspace, size_t workspace_bytes,
                          void* stream) {
  g_last_error.clear();
  if (B < 0 || H < 0 || H_kv < 0 || Sq < 0 || Skv < 0)
    return fail(BSM_ERR_INVALID_ARG, "negative size");
  if (H_kv == 0 ? H != 0 : (H % H_kv) != 0)
    return fail(BSM_ERR_INVALID_ARG, "H must be a multiple of H_kv");
  if (D != 64 && D != 128)
    return fail(BSM_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (Sq > bsm::kMaxSeq || Skv > bsm::kMaxSeq)
    return fail(BSM_ERR_UNSUPPORTED, "sequence length above 262144");
  if (score != BSM_SCORE_SOFTMAX && score != BSM_SCORE_POINTWISE)
    return fail(BSM_ERR_INVALID_ARG, "unknown score path");
  if (score == BSM_SCORE_POINTWISE && lse != nullptr)
    return fail(BSM_ERR_INVALID_ARG,
                "the pointwise score path has no logsumexp; pass lse = NULL");
  if (!std::isfinite(scale)) return fail(BSM_ERR_INVALID_ARG, "scale not finite");
  if (info == nullptr) return fail(BSM_ERR_INVALID_ARG, "mask info is NULL");
  if (info->Sq != Sq || info->Skv != Skv)
    return fail(BSM_ERR_INVALID_ARG,
                "mask info was built for other sequence lengths");
  const bool seg = (info->flags & BSM_MASK_SEGMENT) != 0;
  if (info->num_tables != (seg ? B : 1))
    return fail(BSM_ERR_INVALID_ARG,
                "mask info was built for another batch size");
  if (!is_block_size(info->block_q) || !is_block_size(info->block_kv) ||
      info->nq != (Sq + info->block_q - 1) / info->block_q ||
      info->nk != (Skv + info->block_kv - 1) / info->block_kv ||
      info->num_super != (Sq + bsm::kUnitRows - 1) / bsm::kUnitRows)
    return fail(BSM_ERR_INVALID_ARG, "inconsistent mask info");
  if (seg && (q_segment_ids == nullptr || kv_segment_ids == nullptr))
    return fail(BSM_ERR_INVALID_ARG,
                "BSM_MASK_SEGMENT needs both q and kv segment ids");
  if (!seg && (q_segment_ids != nullptr || kv_segment_ids != nullptr))
    return fail(BSM_ERR_INVALID_ARG,
                "segment ids given without BSM_MASK_SEGMENT");
  if ((info->flags & BSM_MASK_DENSE) &&
      (info->dense_bits == nullptr ||
       info->dense_row_words < (static_cast<int64_t>(Skv) + 31) / 32))
    return fail(BSM_ERR_INVALID_ARG, "mask info lacks its dense mask");
  if (seg && (info->seg_range == nullptr || info->seg_flags == nullptr))
    return fail(BSM_ERR_INVALID_ARG, "mask info lacks segment ranges");
  const int64_t n_super = (Sq + bsm::kUnitRows - 1) / bsm::kUnitRows;
  const int64_t units = static_cast<int64_t>(B) * H * n_super;
  if (units == 0) return BSM_OK;
  if (units > 0x7fffffff) return fail(BSM_ERR_UNSUPPORTED, "too many tiles");
  if (q == nullptr || out == nullptr || (Skv > 0 && (k == nullptr || v == nullptr)))
    return fail(BSM_ERR_INVALID_ARG, "NULL tensor");
  if (workspace == nullptr || workspace_bytes < bsm::kFwdWorkspaceBytes ||
      !aligned16(workspace))
    return fail(BSM_ERR_INVALID_ARG,
                "workspace must be >= bsm_splash_fwd_workspace_bytes() bytes, "
                "16-byte aligned");
  if (q_strides == nullptr || k_strides == nullptr || v_strides == nullptr ||
      o_strides == nullptr)
    return fail(BSM_ERR_INVALID_ARG, "NULL strides");
  if (!aligned16(q) || !aligned16(out) || (Skv > 0 && (!aligned16(k) || !aligned16(v))))
    return fail(BSM_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  const int64_t sizes_q[3] = {B, H, Sq};
  const int64_t sizes_kv[3] = {B, H_kv, Skv};
  for (int d = 0; d < 3; ++d) {
    if (sizes_q[d] > 1 && ((q_strides[d] % 8) != 0 || q_strides[d] <= 0))
      return fail(BSM_ERR_INVALID_ARG, "q strides must be positive multiples of 8");
    if (sizes_q[d] > 1 && ((o_strides[d] % 8) != 0 || o_strides[d] <= 0))
      return fail(BSM_ERR_INVALID_ARG, "out strides must be positive multiples of 8");
    if (Skv > 0 && sizes_kv[d] > 1 && ((k_strides[d] % 8) != 0 || k_strides[d] <= 0 ||
                            (v_strides[d] % 8) != 0 || v_strides[d] <= 0))
      return fail(BSM_ERR_INVALID_ARG, "k/v strides must be positive multiples of 8");
  }
  int num_sms = 0;
  bsm_status s = check_device(&num_sms);
  if (s != BSM_OK) return s;

  CUtensorMap tq, tk, tv;
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  s = make_map(&tq, q, B, H, Sq, D, q_strides, "q");
  if (s != BSM_OK) return s;
  if (Skv > 0) {
    s = make_map(&tk, k, B, H_kv, Skv, D, k_strides, "k");
    if (s != BSM_OK) return s;
    s = make_map(&tv, v, B, H_kv, Skv, D, v_strides, "v");
    if (s != BSM_OK) return s;
  }

  bsm::FwdParams p;
  p.B = B;
  p.H = H;
  p.Hkv = H_kv;
  p.Sq = Sq;
  p.Skv = Skv;
  p.D = D;
  p.n_super = static_cast<int32_t>(n_super);
  p.n_kvtiles = (Skv + bsm::kTileN - 1) / bsm::kTileN;
  p.num_units = static_cast<int32_t>(units);
  p.flags = info->flags;
  p.window = info->window;
  p.block_mask = info->block_mask;
  p.mi_nq = info->nq;
  p.mi_nk = info->nk;
  p.bq = info->block_q;
  p.bkv = info->block_kv;
  p.tables = info->num_tables;
  p.q_seg = q_segment_ids;
  p.kv_seg = kv_segment_ids;
  p.seg_range = info->seg_range;
  p.seg_flags = info->seg_flags;
  p.super_order = info->super_order;
  p.dense = (info->flags & BSM_MASK_DENSE) ? info->dense_bits : nullptr;
  p.dense_words = info->dense_row_words;
  p.score = score;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.scale = scale;
  p.inv_sq = Sq > 0 ? static_cast<float>(1.0 / static_cast<double>(Sq)) : 0.f;
  // pointwise: x sigmoid(x) / Sq = g (1 + tanh(x / 2)), x = scale s,
  // g = x / (2 Sq)
  p.pw_half = static_cast<float>(0.5 * static_cast<double>(scale));
  p.pw_g = Sq > 0 ? static_cast<float>(0.5 * static_cast<double>(scale) /
                                        static_cast<double>(Sq))
                  : 0.f;
  p.out = static_cast<uint16_t*>(out);
  p.o_sb = o_strides[0];
  p.o_sh = o_strides[1];
  p.o_ss = o_strides[2];
  p.o_vec8 = (reinterpret_cast<uintptr_t>(out) % 32 == 0 &&
              o_strides[0] % 16 == 0 && o_strides[1] % 16 == 0 &&
              o_strides[2] % 16 == 0)
                 ? 1
                 : 0;
  p.lse = lse;
  p.unit_counter = static_cast<int32_t*>(workspace);
  p.lists = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + 256);
  if (bsm::fwd_grid_size(p, num_sms) > bsm::kMaxCtas)
    return fail(BSM_ERR_UNSUPPORTED, "more than 256 SMs");
  p.timeout_ns = wait_timeout_ns();
  p.trace = nullptr;
  p.trace_cap = 0;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    const int grid = bsm::fwd_grid_size(p, num_sms);
    if (g_trace_buf != nullptr && grid > 0) {
      const size_t per = g_trace_bytes / 16 / static_cast<size_t>(grid);
      if (per >= 8) {
        p.trace = g_trace_buf;
        p.trace_cap = static_cast<uint32_t>(per - 2);
      }
    }
  }
  cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(int32_t),
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "workspace reset");
  e = bsm::launch_splash_fwd(p, tq, tk, tv, num_sms,
                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "splash_fwd launch");
  return BSM_OK;
}

bsm_status bsm_pack_dense_mask(const uint8_t* mask, int64_t mask_row_stride,
                               int32_t Sq, int32_t Skv, uint32_t* words,
                               int32_t row_words, void* stream) {
  g_last_error.clear();
  if (Sq < 0 || Skv < 0)
    return fail(BSM_ERR_INVALID_ARG, "Sq and Skv must be >= 0");
  if (row_words < (static_cast<int64_t>(Skv) + 31) / 32)
    return fail(BSM_ERR_INVALID_ARG, "row_words must be >= ceil(Skv / 32)");
  if (mask_row_stride < Skv)
    return fail(BSM_ERR_INVALID_ARG, "mask_row_stride must be >= Skv");
  if (static_cast<int64_t>(Sq) * row_words == 0) return BSM_OK;
  if (mask == nullptr || words == nullptr)
    return fail(BSM_ERR_INVALID_ARG, "mask and words must be non-NULL");
  int num_sms = 0;
  bsm_status s = check_device(&num_sms);
  if (s != BSM_OK) return s;
  const cudaError_t e = bsm::launch_pack_dense(
      mask, mask_row_stride, Sq, Skv, words, row_words, num_sms,
      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "pack_dense launch");
  return BSM_OK;
}

size_t bsm_splash_fwd_workspace_bytes(void) { return bsm::kFwdWorkspaceBytes; }

size_t bsm_splash_bwd_workspace_bytes(int32_t B, int32_t H, int32_t Sq,
                                      int32_t score) {
  if (B < 0 || H < 0 || Sq < 0) return 0;
  if (score != BSM_SCORE_SOFTMAX) return 0;
  return align_up(static_cast<size_t>(B) * H * Sq * sizeof(float), 256);
}

bsm_status bsm_splash_bwd(const bsm_tensor* q, const bsm_tensor* k,
                          const bsm_tensor* v, const bsm_tensor* out,
                          const float* lse, const bsm_tensor* dout, int32_t B,
                          int32_t H, int32_t H_kv, int32_t Sq, int32_t Skv,
                          int32_t D, const bsm_mask_info* info,
                          const int32_t* q_segment_ids,
                          const int32_t* kv_segment_ids, float scale,
                          int32_t score, const bsm_tensor* dq,
                          const bsm_tensor* dk, const bsm_tensor* dv,
                          void* workspace, size_t workspace_bytes,
                          void* stream) {
  g_last_error.clear();
  if (B < 0 || H < 0 || H_kv < 0 || Sq < 0 || Skv < 0)
    return fail(BSM_ERR_INVALID_ARG, "negative size");
  if (H_kv == 0 ? H != 0 : (H % H_kv) != 0)
    return fail(BSM_ERR_INVALID_ARG, "H must be a multiple of H_kv");
  if (D != 64 && D != 128)
    return fail(BSM_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (Sq > bsm::kMaxSeq || Skv > bsm::kMaxSeq)
    return fail(BSM_ERR_UNSUPPORTED, "sequence length above 262144");
  if (score != BSM_SCORE_SOFTMAX && score != BSM_SCORE_POINTWISE)
    return fail(BSM_ERR_INVALID_ARG, "unknown score path");
  if (!std::isfinite(scale)) return fail(BSM_ERR_INVALID_ARG, "scale not finite");
  const bool sm = score == BSM_SCORE_SOFTMAX;
  if (q == nullptr || k == nullptr || v == nullptr || dout == nullptr ||
      dq == nullptr || dk == nullptr || dv == nullptr || (sm && out == nullptr))
    return fail(BSM_ERR_INVALID_ARG, "NULL tensor view");
  if (sm && lse == nullptr)
    return fail(BSM_ERR_INVALID_ARG,
                "the softmax backward needs the forward's out and lse");
  if (info == nullptr) return fail(BSM_ERR_INVALID_ARG, "mask info is NULL");
  if (info->Sq != Sq || info->Skv != Skv)
    return fail(BSM_ERR_INVALID_ARG,
                "mask info was built for other sequence lengths");
  const bool seg = (info->flags & BSM_MASK_SEGMENT) != 0;
  if (info->num_tables != (seg ? B : 1))
    return fail(BSM_ERR_INVALID_ARG,
                "mask info was built for another batch size");
  if (!is_block_size(info->block_q) || !is_block_size(info->block_kv) ||
      info->nq != (Sq + info->block_q - 1) / info->block_q ||
      info->nk != (Skv + info->block_kv - 1) / info->block_kv)
    return fail(BSM_ERR_INVALID_ARG, "inconsistent mask info");
  if (seg && (q_segment_ids == nullptr || kv_segment_ids == nullptr))
    return fail(BSM_ERR_INVALID_ARG,
                "BSM_MASK_SEGMENT needs both q and kv segment ids");
  if (!seg && (q_segment_ids != nullptr || kv_segment_ids != nullptr))
    return fail(BSM_ERR_INVALID_ARG,
                "segment ids given without BSM_MASK_SEGMENT");
  if ((info->flags & BSM_MASK_DENSE) &&
      (info->dense_bits == nullptr ||
       info->dense_row_words < (static_cast<int64_t>(Skv) + 31) / 32))
    return fail(BSM_ERR_INVALID_ARG, "mask info lacks its dense mask");
  if (static_cast<int64_t>(B) * H * Sq == 0 &&
      static_cast<int64_t>(B) * H_kv * Skv == 0)
    return BSM_OK;
  const size_t ws_need = bsm_splash_bwd_workspace_bytes(B, H, Sq, score);
  if (ws_need > 0 && (workspace == nullptr || workspace_bytes < ws_need ||
                      !aligned16(workspace)))
    return fail(BSM_ERR_INVALID_ARG,
                "workspace must be >= bsm_splash_bwd_workspace_bytes() bytes, "
                "16-byte aligned");
  // every view: aligned data, positive strides that are multiples of 8
  struct View {
    const bsm_tensor* t;
    int64_t heads, S;
    const char* name;
  };
  const View views[] = {{q, H, Sq, "q"},       {k, H_kv, Skv, "k"},
                        {v, H_kv, Skv, "v"},   {dout, H, Sq, "dout"},
                        {dq, H, Sq, "dq"},     {dk, H_kv, Skv, "dk"},
                        {dv, H_kv, Skv, "dv"}, {sm ? out : dout, H, Sq, "out"}};
  for (const View& w : views) {
    if (w.S == 0) continue;
    if (w.t->data == nullptr || !aligned16(w.t->data))
      return fail(BSM_ERR_INVALID_ARG,
                  std::string(w.name) + " must be non-NULL and 16-byte aligned");
    const int64_t sizes[3] = {B, w.heads, w.S};
    for (int d = 0; d < 3; ++d)
      if (sizes[d] > 1 && (w.t->strides[d] <= 0 || w.t->strides[d] % 8 != 0))
        return fail(BSM_ERR_INVALID_ARG,
                    std::string(w.name) +
                        " strides must be positive multiples of 8");
  }
  int num_sms = 0;
  bsm_status s = check_device(&num_sms);
  if (s != BSM_OK) return s;
  CUtensorMap tq, tk, tv, tdo;
  std::memset(&tq, 0, sizeof(tq));
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  std::memset(&tdo, 0, sizeof(tdo));
  if (Sq > 0) {
    s = make_map(&tq, q->data, B, H, Sq, D, q->strides, "q");
    if (s != BSM_OK) return s;
    s = make_map(&tdo, dout->data, B, H, Sq, D, dout->strides, "dout");
    if (s != BSM_OK) return s;
  }
  if (Skv > 0) {
    s = make_map(&tk, k->data, B, H_kv, Skv, D, k->strides, "k");
    if (s != BSM_OK) return s;
    s = make_map(&tv, v->data, B, H_kv, Skv, D, v->strides, "v");
    if (s != BSM_OK) return s;
  }
  bsm::BwdParams p;
  p.B = B;
  p.H = H;
  p.Hkv = H_kv;
  p.Sq = Sq;
  p.Skv = Skv;
  p.D = D;
  p.flags = info->flags;
  p.window = info->window;
  p.block_mask = info->block_mask;
  p.mi_nq = info->nq;
  p.mi_nk = info->nk;
  p.bq = info->block_q;
  p.bkv = info->block_kv;
  p.q_seg = q_segment_ids;
  p.kv_seg = kv_segment_ids;
  p.dense = (info->flags & BSM_MASK_DENSE) ? info->dense_bits : nullptr;
  p.dense_words = info->dense_row_words;
  p.score = score;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.inv_sq = Sq > 0 ? static_cast<float>(1.0 / static_cast<double>(Sq)) : 0.f;
  p.lse = lse;
  p.delta = static_cast<float*>(workspace);
  p.out = sm ? static_cast<const uint16_t*>(out->data) : nullptr;
  p.o_sb = sm ? out->strides[0] : 0;
  p.o_sh = sm ? out->strides[1] : 0;
  p.o_ss = sm ? out->strides[2] : 0;
  p.dout = static_cast<const uint16_t*>(dout->data);
  p.do_sb = dout->strides[0];
  p.do_sh = dout->strides[1];
  p.do_ss = dout->strides[2];
  p.dq = static_cast<uint16_t*>(dq->data);
  p.dq_sb = dq->strides[0];
  p.dq_sh = dq->strides[1];
  p.dq_ss = dq->strides[2];
  p.dk = static_cast<uint16_t*>(dk->data);
  p.dk_sb = dk->strides[0];
  p.dk_sh = dk->strides[1];
  p.dk_ss = dk->strides[2];
  p.dv = static_cast<uint16_t*>(dv->data);
  p.dv_sb = dv->strides[0];
  p.dv_sh = dv->strides[1];
  p.dv_ss = dv->strides[2];
  p.timeout_ns = wait_timeout_ns();
  cudaError_t e = bsm::launch_splash_bwd(p, tq, tk, tv, tdo,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "splash_bwd launch");
  return BSM_OK;
}

bsm_status bsm_device_status(void* stream, int32_t* detail) {
  g_last_error.clear();
  int32_t rec[4] = {0, 0, 0, 0}, brec[4] = {0, 0, 0, 0};
  cudaError_t e = bsm::read_device_error(rec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "device status");
  e = bsm::read_bwd_error(brec);
  if (e != cudaSuccess) return cuda_fail(e, "device status");
  if (rec[0] == 0 && brec[0] != 0) std::memcpy(rec, brec, sizeof(rec));
  if (detail != nullptr) std::memcpy(detail, rec, sizeof(rec));
  if (rec[0] != 0)
    return fail(BSM_ERR_DEVICE_TIMEOUT,
                "a kernel gave up on a bounded wait (block " +
                    std::to_string(rec[1]) + ", role " + std::to_string(rec[2]) +
                    ", phase " + std::to_string(rec[3]) + ")");
  return BSM_OK;
}

bsm_status bsm_selftest_wait_timeout(int64_t timeout_ns, void* stream) {
  g_last_error.clear();
  if (timeout_ns < 1000 || timeout_ns > 10000000000LL)
    return fail(BSM_ERR_INVALID_ARG, "timeout_ns must be in [1e3, 1e10]");
  bsm_status s = check_device(nullptr);
  if (s != BSM_OK) return s;
  cudaError_t e = bsm::launch_wait_selftest(static_cast<uint64_t>(timeout_ns),
                                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return BSM_OK;
}

bsm_status bsm_debug_set_trace(void* buffer, size_t bytes) {
  g_last_error.clear();
  if (buffer != nullptr && (reinterpret_cast<uintptr_t>(buffer) & 15u) != 0)
    return fail(BSM_ERR_INVALID_ARG, "trace buffer must be 16-byte aligned");
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_buf = bytes >= 32 ? buffer : nullptr;
  g_trace_bytes = g_trace_buf != nullptr ? bytes : 0;
  return BSM_OK;
}

int32_t bsm_debug_fwd_grid(int32_t B, int32_t H, int32_t Sq) {
  int num_sms = 0;
  if (check_device(&num_sms) != BSM_OK) return -1;
  bsm::FwdParams p;
  p.num_units = B * H * ((Sq + bsm::kUnitRows - 1) / bsm::kUnitRows);
  return bsm::fwd_grid_size(p, num_sms);
}

const char* bsm_last_error(void) { return g_last_error.c_str(); }

int32_t bsm_version(void) { return 302; }

}  // extern "C"
