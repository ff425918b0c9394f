// Internal declarations shared by the host C ABI (bsm_api.cu) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/bsm.h"

namespace bsm {

// Query tile (rows of one tcgen05 accumulator) and KV tile of the forward
// kernel; one work unit is two query tiles (256 rows) of one (batch, head).
constexpr int kTileM = 128;
constexpr int kTileN = 128;
constexpr int kUnitRows = 2 * kTileM;
constexpr int kMaxSeq = 262144;
constexpr int kMaxKvTiles = kMaxSeq / kTileN;  // list capacity per unit
// Forward workspace: 256 bytes of counters, then per CTA two sets (one per
// query-tile pipeline of the packed-sequence kernel; the other kernel uses
// the first) of three unit lists of kMaxKvTiles uint16 entries (up to
// kMaxCtas CTAs).
constexpr int kMaxCtas = 256;
constexpr int kMaxSuperOrder = 8192;  // longest-first table size limit
constexpr int kListBufs = 3;
constexpr size_t kListBytes = static_cast<size_t>(kMaxKvTiles) * 2;
constexpr size_t kFwdWorkspaceBytes =
    256 + static_cast<size_t>(kMaxCtas) * 2 * kListBufs * kListBytes;

struct MaskInfoParams {
  uint32_t flags;
  int32_t window;
  int32_t Sq, Skv, bq, bkv, nq, nk, tables;
  const int32_t* q_seg;   // [tables][Sq] (SEGMENT only)
  const int32_t* kv_seg;  // [tables][Skv]
  int8_t* block_mask;
  int32_t* data_next;
  int32_t* row_ptr;
  int32_t* kv_idx;
  int8_t* kv_cls;
  int32_t* seg_range;  // [tables][Sq][2] (SEGMENT only)
  int32_t* seg_flags;  // [1]: bit 0 = some kv id row is not sorted
  int32_t n_super;        // ceil(Sq / kUnitRows)
  int32_t* super_order;   // [tables * n_super] or null
  const uint32_t* dense;  // DENSE: [Sq][dense_words] bit-packed, else null
  int64_t dense_words;
  // one-launch build: staged row lists [tables * nq][nk] and the ticket word
  int32_t fused;
  uint16_t* staged;
  unsigned long long* ticket;
  unsigned long long epoch;  // 1 .. 2^40 - 1, new for every build
};

struct FwdParams {
  int32_t B, H, Hkv, Sq, Skv, D;
  int32_t n_super;    // ceil(Sq / 256)
  const int32_t* super_order;  // longest-first (table, super-tile) or null
  const uint32_t* dense;       // DENSE: [Sq][dense_words] bit-packed, else null
  int64_t dense_words;
  int32_t n_kvtiles;  // ceil(Skv / 128)
  int32_t num_units;  // B * H * n_super
  // mask
  uint32_t flags;
  int32_t window;
  const int8_t* block_mask;  // [tables][mi_nq][mi_nk]
  int32_t mi_nq, mi_nk, bq, bkv, tables;
  const int32_t* q_seg;      // [B][Sq]
  const int32_t* kv_seg;     // [B][Skv]
  const int32_t* seg_range;  // [B][Sq][2] from the mask-info
  const int32_t* seg_flags;  // bit 0: kv ids not sorted
  // scores
  int32_t score;     // bsm_score
  float scale_log2;  // softmax: scale * log2(e)
  float scale;       // pointwise
  float inv_sq;      // pointwise: 1 / Sq
  float pw_half;     // pointwise: scale / 2
  float pw_g;        // pointwise: scale / (2 Sq)
  // outputs
  uint16_t* out;  // bf16 bits
  int64_t o_sb, o_sh, o_ss;
  int32_t o_vec8;  // out and its strides allow 32-byte row stores
  float* lse;
  int32_t* unit_counter;  // workspace: next work unit (zeroed per launch)
  uint16_t* lists;        // workspace: [grid][kListBufs][kMaxKvTiles]
  uint64_t timeout_ns;
  // optional event trace (records of 16 bytes, cap per CTA), else null
  void* trace;
  uint32_t trace_cap;
};

struct BwdParams {
  int32_t B, H, Hkv, Sq, Skv, D;
  // mask
  uint32_t flags;
  int32_t window;
  const int8_t* block_mask;  // [tables][mi_nq][mi_nk]
  int32_t mi_nq, mi_nk, bq, bkv;
  const int32_t* q_seg;   // [B][Sq] (SEGMENT only)
  const int32_t* kv_seg;  // [B][Skv]
  const uint32_t* dense;  // DENSE: [Sq][dense_words] bit-packed, else null
  int64_t dense_words;
  // scores
  int32_t score;
  float scale, scale_log2, inv_sq;
  const float* lse;  // forward logsumexp [B][H][Sq] (softmax)
  float* delta;      // workspace: D_q = sum_d dO * out, [B][H][Sq] (softmax)
  const uint16_t* out;   // forward output (softmax), bf16
  int64_t o_sb, o_sh, o_ss;
  const uint16_t* dout;  // gradient of the output, bf16
  int64_t do_sb, do_sh, do_ss;
  // gradients, bf16
  uint16_t* dq;
  int64_t dq_sb, dq_sh, dq_ss;
  uint16_t* dk;
  int64_t dk_sb, dk_sh, dk_ss;
  uint16_t* dv;
  int64_t dv_sb, dv_sh, dv_ss;
  uint64_t timeout_ns;
};

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_mask_info(const MaskInfoParams& p, cudaStream_t stream);
cudaError_t launch_pack_dense(const uint8_t* mask, int64_t stride, int32_t Sq,
                              int32_t Skv, uint32_t* words, int32_t row_words,
                              int num_sms, cudaStream_t stream);
// Whether a mask of these sizes is built in one launch.
bool mask_info_fused(int64_t tables, int64_t nq, int64_t nk);
int fwd_grid_size(const FwdParams& p, int num_sms);
cudaError_t launch_splash_fwd(const FwdParams& p, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv,
                              int num_sms, cudaStream_t stream);
cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t stream);
// D_q (softmax), then the dK/dV and dQ kernels.
cudaError_t launch_splash_bwd(const BwdParams& p, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, cudaStream_t stream);
// Reads and clears the device error record of the backward kernels.
cudaError_t read_bwd_error(int32_t out[4]);
// Sets the thread-local text returned by bsm_last_error().
void set_last_error(const char* msg);
// Reads and clears the device error record of the forward kernel TU.
cudaError_t read_device_error(int32_t out[4], cudaStream_t stream);

}  // namespace bsm
