// Forward entry point that allocates nothing.
//
// Some callers cannot allocate device memory when they run the attention:
// plugins or language runtimes that are handed finished device buffers by a
// host framework and have no allocator of their own, serving engines that
// reserve all free HBM for their KV cache up front, or real-time loops in
// which the implicit device synchronisation of cudaMalloc is not acceptable.
// bsm_splash_fwd needs a caller-provided workspace; this variant uses a
// workspace that lives in the library itself instead: a file-scope device
// array of bsm::kFwdWorkspaceBytes (3 MiB), held by every GPU that loads the
// library until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "bsm_internal.h"

namespace {

// The forward's scratch: the work-unit counter (first 256 bytes) and each
// CTA's KV-tile lists.  Shared by every call on a device.
static __device__ __align__(256) uint8_t g_fwd_scratch[bsm::kFwdWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_fwd_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
bsm_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    bsm::set_last_error("bsm_splash_fwd_noalloc: cudaGetDevice failed");
    return BSM_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    bsm::set_last_error("bsm_splash_fwd_noalloc: device ordinal above 63");
    return BSM_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fwd_scratch);
    if (e != cudaSuccess || p == nullptr) {
      bsm::set_last_error(
          "bsm_splash_fwd_noalloc: cudaGetSymbolAddress of the scratch "
          "array failed");
      return BSM_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return BSM_OK;
}

}  // namespace

extern "C" bsm_status bsm_splash_fwd_noalloc(
    const void* q, const void* k, const void* v, const int64_t q_strides[3],
    const int64_t k_strides[3], const int64_t v_strides[3],
    const int64_t o_strides[3], int32_t B, int32_t H, int32_t H_kv, int32_t Sq,
    int32_t Skv, int32_t D, const bsm_mask_info* info,
    const int32_t* q_segment_ids, const int32_t* kv_segment_ids, float scale,
    int32_t score, void* out, float* lse, void* stream) {
  // The scratch holds lists for up to bsm::kMaxCtas CTAs of at most
  // bsm::kMaxKvTiles KV tiles: reject anything longer before touching it.
  if (Sq > bsm::kMaxSeq || Skv > bsm::kMaxSeq) {
    bsm::set_last_error(
        "bsm_splash_fwd_noalloc: sequence length above 262144 does not fit "
        "the library's 3 MiB scratch");
    return BSM_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  const bsm_status s = scratch_address(&scratch);
  if (s != BSM_OK) return s;
  return bsm_splash_fwd(q, k, v, q_strides, k_strides, v_strides, o_strides,
                        B, H, H_kv, Sq, Skv, D, info, q_segment_ids,
                        kv_segment_ids, scale, score, out, lse, scratch,
                        sizeof(g_fwd_scratch), stream);
}
