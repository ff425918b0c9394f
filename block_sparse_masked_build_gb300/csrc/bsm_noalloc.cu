// Forward entry point that allocates nothing.
//
// Some callers cannot allocate device memory when they run the attention:
// plugins or language runtimes that are handed finished device buffers by a
// host framework and have no allocator of their own, serving engines that
// reserve all free HBM for their KV cache up front, or real-time loops in
// which the implicit device synchronisation of cudaMalloc is not acceptable.
// bsm_splash_fwd needs a caller-provided workspace; this variant uses a
// workspace that lives in the library itself instead: a file-scope device
// array of bsm::kFwdWorkspaceBytes (6 MiB).
//
// The array is part of this file's device code.  CUDA loads a library's
// device code into a context lazily by default (on the first use of one of
// its kernels or symbols), and that load is when the array's 6 MiB are
// taken.  So the first call on a device -- which looks the array up -- may
// take device memory and synchronise; every later call in the same context
// takes none.  Callers that reserve all free memory make one call first.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "bsm_internal.h"

namespace {

// The forward's scratch: the work-unit counter (first 256 bytes) and each
// CTA's KV-tile lists.  Shared by every call on a device.
static __device__ __align__(256) uint8_t g_fwd_scratch[bsm::kFwdWorkspaceBytes];

constexpr int kMaxDevices = 64;

// Address of g_fwd_scratch per device, valid for the CUDA context it was
// looked up in (a cudaDeviceReset makes a new primary context with a new
// id, and the stale address is then looked up again).
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
std::mutex g_mu;
ScratchEntry g_scratch[kMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

bool driver_fns() {
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return g_ctx_current != nullptr && g_ctx_id != nullptr;
}

// Device address of g_fwd_scratch in the current device's context.  In host
// code the array's name is only a host-side stand-in, so the address is
// looked up with cudaGetSymbolAddress once per device and context, with that
// device current, and kept.
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
  if (!driver_fns()) {
    bsm::set_last_error(
        "bsm_splash_fwd_noalloc: cuCtxGetCurrent/cuCtxGetId unavailable");
    return BSM_ERR_CUDA;
  }
  // Id of the context bound to this thread (none yet: id 0, never cached).
  auto context_id = [](unsigned long long* id) {
    CUcontext ctx = nullptr;
    *id = 0;
    return g_ctx_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
           g_ctx_id(ctx, id) == CUDA_SUCCESS;
  };
  unsigned long long id = 0;
  const bool bound = context_id(&id);
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchEntry& ent = g_scratch[dev];
  if (!bound || ent.addr == nullptr || ent.ctx_id != id) {
    // binds the device's primary context to this thread if needed
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fwd_scratch);
    if (e != cudaSuccess || p == nullptr) {
      bsm::set_last_error(
          "bsm_splash_fwd_noalloc: cudaGetSymbolAddress of the scratch "
          "array failed");
      return BSM_ERR_CUDA;
    }
    if (!context_id(&id)) {
      bsm::set_last_error(
          "bsm_splash_fwd_noalloc: cannot identify the CUDA context");
      return BSM_ERR_CUDA;
    }
    ent.addr = p;
    ent.ctx_id = id;
  }
  *out = ent.addr;
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
        "the library's 6 MiB scratch");
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
