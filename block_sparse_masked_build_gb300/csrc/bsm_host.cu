// Forward on host buffers: the end-to-end call.
//
// q, k, v (and the segment ids) live in host memory and out/lse go back
// there.  The call copies them in, builds the mask info, runs the forward
// and copies the results out, pipelined over chunks of K/V heads: the
// host->device copies of chunk c + 1 run on one copy stream, the forward of
// chunk c on the caller's stream and the device->host copies of chunk c - 1
// on a second copy stream, so the host link carries both directions while
// the kernels run.  A chunk is a range of heads of every batch row, moved
// with one strided copy per tensor (cudaMemcpy2DAsync: B rows of one
// head-range slab each).  Everything is enqueued; the call returns without
// waiting, and the caller's stream waits for the last copy.
//
// The two copy streams and the events that chain the chunks belong to the
// library: created on a device's first call (per CUDA context) and kept.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>

#include "bsm_internal.h"

namespace {

constexpr int kMaxHostChunks = 16;
constexpr int kDefaultHostChunks = 4;
constexpr int kMaxDevices = 64;

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Offsets of the pieces of the caller's device buffer.
struct HostLayout {
  size_t q, k, v, o, lse, qs, ks, mi, ws, total;
};

bool host_layout(const bsm_mask_spec* spec, int32_t B, int32_t H,
                 int32_t H_kv, int32_t Sq, int32_t Skv, int32_t D,
                 int32_t block_q, int32_t block_kv, int32_t score,
                 HostLayout* L) {
  if (spec == nullptr || B < 0 || H < 0 || H_kv < 0 || Sq < 0 || Skv < 0 ||
      D <= 0)
    return false;
  const size_t mi = bsm_mask_info_bytes(spec, B, Sq, Skv, block_q, block_kv);
  if (mi == 0) return false;
  const bool seg = (spec->flags & BSM_MASK_SEGMENT) != 0;
  const size_t qo = static_cast<size_t>(B) * H * Sq * D * 2;
  const size_t kv = static_cast<size_t>(B) * H_kv * Skv * D * 2;
  size_t o = 0;
  L->q = o;
  o = up256(o + qo);
  L->k = o;
  o = up256(o + kv);
  L->v = o;
  o = up256(o + kv);
  L->o = o;
  o = up256(o + qo);
  L->lse = o;
  if (score == BSM_SCORE_SOFTMAX)
    o = up256(o + static_cast<size_t>(B) * H * Sq * 4);
  L->qs = o;
  if (seg) o = up256(o + static_cast<size_t>(B) * Sq * 4);
  L->ks = o;
  if (seg) o = up256(o + static_cast<size_t>(B) * Skv * 4);
  L->mi = o;
  o = up256(o + mi);
  L->ws = o;
  o = up256(o + bsm::kFwdWorkspaceBytes);
  L->total = o;
  return true;
}

// The library's copy streams and chunk events on one device, valid for
// the CUDA context they were made in.
struct CopyRes {
  unsigned long long ctx_id = 0;
  bool made = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, finish = nullptr;
  cudaEvent_t loaded[kMaxHostChunks] = {}, done[kMaxHostChunks] = {};
};
std::mutex g_res_mu;
CopyRes g_res[kMaxDevices];

PFN_cuCtxGetCurrent_v4000 g_get_ctx = nullptr;
PFN_cuCtxGetId_v12000 g_get_ctx_id = nullptr;

bool context_id(unsigned long long* id) {
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_get_ctx = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_get_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (g_get_ctx == nullptr || g_get_ctx_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (g_get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return g_get_ctx_id(ctx, id) == CUDA_SUCCESS;
}

bsm_status cuda_error(cudaError_t e, const char* what) {
  const std::string msg = std::string("bsm_splash_fwd_host: ") + what +
                          ": " + cudaGetErrorName(e);
  bsm::set_last_error(msg.c_str());
  return BSM_ERR_CUDA;
}

// The current device's streams and events, made on first use in a context.
bsm_status copy_resources(CopyRes** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    bsm::set_last_error("bsm_splash_fwd_host: device ordinal above 63");
    return BSM_ERR_UNSUPPORTED;
  }
  // the runtime makes the device's primary context current on first use
  e = cudaFree(nullptr);
  if (e != cudaSuccess) return cuda_error(e, "context set-up");
  unsigned long long id = 0;
  if (!context_id(&id)) {
    bsm::set_last_error("bsm_splash_fwd_host: no current CUDA context");
    return BSM_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_res_mu);
  CopyRes& r = g_res[dev];
  if (!r.made || r.ctx_id != id) {
    // a new context (first call, or after a device reset): the old handles
    // died with the old context and are not destroyed here
    r = CopyRes{};
    const unsigned ef = cudaEventDisableTiming;
    e = cudaStreamCreateWithFlags(&r.in, cudaStreamNonBlocking);
    if (e == cudaSuccess)
      e = cudaStreamCreateWithFlags(&r.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.start, ef);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.finish, ef);
    for (int c = 0; e == cudaSuccess && c < kMaxHostChunks; ++c) {
      e = cudaEventCreateWithFlags(&r.loaded[c], ef);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.done[c], ef);
    }
    if (e != cudaSuccess) return cuda_error(e, "copy streams and events");
    r.ctx_id = id;
    r.made = true;
  }
  *out = &r;
  return BSM_OK;
}

// Rows [0, rows) of `width` bytes, at `dpitch` / `spitch` byte strides:
// one strided copy, or one copy per row where a pitch is above what a
// strided copy takes (`max_pitch`, the device's cudaDevAttrMaxPitch).
cudaError_t copy_rows(void* dst, size_t dpitch, const void* src,
                      size_t spitch, size_t width, size_t rows,
                      size_t max_pitch, cudaMemcpyKind kind,
                      cudaStream_t s) {
  if (width == 0 || rows == 0) return cudaSuccess;
  if (rows == 1 || (dpitch == width && spitch == width))
    return cudaMemcpyAsync(dst, src, width * rows, kind, s);
  if (dpitch <= max_pitch && spitch <= max_pitch)
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s);
  for (size_t r = 0; r < rows; ++r) {
    const cudaError_t e = cudaMemcpyAsync(
        static_cast<uint8_t*>(dst) + r * dpitch,
        static_cast<const uint8_t*>(src) + r * spitch, width, kind, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t bsm_splash_fwd_host_bytes(const bsm_mask_spec* spec, int32_t B,
                                 int32_t H, int32_t H_kv, int32_t Sq,
                                 int32_t Skv, int32_t D, int32_t block_q,
                                 int32_t block_kv, int32_t score) {
  HostLayout L;
  if (!host_layout(spec, B, H, H_kv, Sq, Skv, D, block_q, block_kv, score,
                   &L))
    return 0;
  return L.total;
}

bsm_status bsm_splash_fwd_host(const bsm_mask_spec* spec, const void* q,
                               const void* k, const void* v,
                               const int32_t* q_segment_ids,
                               const int32_t* kv_segment_ids, int32_t B,
                               int32_t H, int32_t H_kv, int32_t Sq,
                               int32_t Skv, int32_t D, int32_t block_q,
                               int32_t block_kv, float scale, int32_t score,
                               void* out, float* lse, void* device_buffer,
                               size_t device_bytes, int32_t n_chunks,
                               void* stream) {
  bsm::set_last_error("");
  if (spec == nullptr) {
    bsm::set_last_error("bsm_splash_fwd_host: mask spec is NULL");
    return BSM_ERR_INVALID_ARG;
  }
  if (B < 0 || H < 0 || H_kv < 0 || Sq < 0 || Skv < 0) {
    bsm::set_last_error("bsm_splash_fwd_host: negative size");
    return BSM_ERR_INVALID_ARG;
  }
  if (H_kv == 0 ? H != 0 : (H % H_kv) != 0) {
    bsm::set_last_error("bsm_splash_fwd_host: H must be a multiple of H_kv");
    return BSM_ERR_INVALID_ARG;
  }
  if (D != 64 && D != 128) {
    bsm::set_last_error("bsm_splash_fwd_host: head_dim must be 64 or 128");
    return BSM_ERR_UNSUPPORTED;
  }
  if (score != BSM_SCORE_SOFTMAX && score != BSM_SCORE_POINTWISE) {
    bsm::set_last_error("bsm_splash_fwd_host: unknown score path");
    return BSM_ERR_INVALID_ARG;
  }
  if (score == BSM_SCORE_POINTWISE && lse != nullptr) {
    bsm::set_last_error(
        "bsm_splash_fwd_host: the pointwise score path has no logsumexp; "
        "pass lse = NULL");
    return BSM_ERR_INVALID_ARG;
  }
  const bool seg = (spec->flags & BSM_MASK_SEGMENT) != 0;
  if (seg != (q_segment_ids != nullptr && kv_segment_ids != nullptr) ||
      (!seg && (q_segment_ids != nullptr || kv_segment_ids != nullptr))) {
    bsm::set_last_error(
        "bsm_splash_fwd_host: segment ids are needed (both) iff "
        "BSM_MASK_SEGMENT");
    return BSM_ERR_INVALID_ARG;
  }
  HostLayout L;
  if (!host_layout(spec, B, H, H_kv, Sq, Skv, D, block_q, block_kv, score,
                   &L)) {
    bsm::set_last_error(
        "bsm_splash_fwd_host: bad mask spec, sizes or block sizes");
    return BSM_ERR_INVALID_ARG;
  }
  if (B == 0 || H == 0 || Sq == 0) return BSM_OK;
  if (q == nullptr || out == nullptr ||
      (Skv > 0 && (k == nullptr || v == nullptr))) {
    bsm::set_last_error("bsm_splash_fwd_host: NULL host tensor");
    return BSM_ERR_INVALID_ARG;
  }
  if (device_buffer == nullptr || device_bytes < L.total ||
      (reinterpret_cast<uintptr_t>(device_buffer) & 255) != 0) {
    bsm::set_last_error(
        "bsm_splash_fwd_host: device buffer must be >= "
        "bsm_splash_fwd_host_bytes(...) bytes, 256-byte aligned");
    return BSM_ERR_INVALID_ARG;
  }
  CopyRes* r = nullptr;
  bsm_status st = copy_resources(&r);
  if (st != BSM_OK) return st;
  int dev = 0, pitch_attr = 0;
  cudaError_t ae = cudaGetDevice(&dev);
  if (ae == cudaSuccess)
    ae = cudaDeviceGetAttribute(&pitch_attr, cudaDevAttrMaxPitch, dev);
  if (ae != cudaSuccess) return cuda_error(ae, "device attributes");
  const size_t max_pitch = pitch_attr > 0 ? static_cast<size_t>(pitch_attr) : 0;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(device_buffer);
  uint8_t* qd = base + L.q;
  uint8_t* kd = base + L.k;
  uint8_t* vd = base + L.v;
  uint8_t* od = base + L.o;
  float* lsed = score == BSM_SCORE_SOFTMAX
                    ? reinterpret_cast<float*>(base + L.lse)
                    : nullptr;
  int32_t* qsd = seg ? reinterpret_cast<int32_t*>(base + L.qs) : nullptr;
  int32_t* ksd = seg ? reinterpret_cast<int32_t*>(base + L.ks) : nullptr;

  const int g = H / H_kv;
  int chunks = n_chunks > 0 ? n_chunks : kDefaultHostChunks;
  if (chunks > kMaxHostChunks) chunks = kMaxHostChunks;
  if (chunks > H_kv) chunks = H_kv;
  const size_t q_head = static_cast<size_t>(Sq) * D * 2;   // bytes
  const size_t kv_head = static_cast<size_t>(Skv) * D * 2;
  const size_t q_pitch = q_head * H, kv_pitch = kv_head * H_kv;
  const uint8_t* qh = static_cast<const uint8_t*>(q);
  const uint8_t* kh = static_cast<const uint8_t*>(k);
  const uint8_t* vh = static_cast<const uint8_t*>(v);
  uint8_t* oh = static_cast<uint8_t*>(out);

  // the copy streams start after the work already on the caller's stream
  // (an earlier call on the same device buffer may still read it)
  cudaError_t e = cudaEventRecord(r->start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(r->in, r->start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(r->out, r->start, 0);
  if (e != cudaSuccess) return cuda_error(e, "stream fork");
  // After a failure part-way the caller's stream still waits for the
  // copies already enqueued, so the device buffer is free once it is
  // synchronised (best effort: the failure may be the stream's own).
  auto join_fail = [&](bsm_status status) {
    for (cudaStream_t c : {r->in, r->out})
      if (cudaEventRecord(r->finish, c) == cudaSuccess)
        cudaStreamWaitEvent(s, r->finish, 0);
    return status;
  };

  // segment ids in and the mask info, on the caller's stream
  if (seg) {
    e = cudaMemcpyAsync(qsd, q_segment_ids, static_cast<size_t>(B) * Sq * 4,
                        cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ksd, kv_segment_ids,
                          static_cast<size_t>(B) * Skv * 4,
                          cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return join_fail(cuda_error(e, "segment ids"));
  }
  bsm_mask_info info;
  st = bsm_build_mask_info(spec, qsd, ksd, B, Sq, Skv, block_q, block_kv,
                           base + L.mi, L.ws - L.mi, &info, stream);
  if (st != BSM_OK) return join_fail(st);

  const int64_t q_strides[3] = {static_cast<int64_t>(H) * Sq * D,
                                static_cast<int64_t>(Sq) * D, D};
  const int64_t kv_strides[3] = {static_cast<int64_t>(H_kv) * Skv * D,
                                 static_cast<int64_t>(Skv) * D, D};
  for (int c = 0; c < chunks; ++c) {
    const int a = static_cast<int>(static_cast<int64_t>(H_kv) * c / chunks);
    const int b = static_cast<int>(static_cast<int64_t>(H_kv) * (c + 1) / chunks);
    const int nkv = b - a, nq = nkv * g, qa = a * g;
    // in: the chunk's heads of every batch row
    e = copy_rows(qd + qa * q_head, q_pitch, qh + qa * q_head, q_pitch,
                  nq * q_head, B, max_pitch, cudaMemcpyHostToDevice, r->in);
    if (e == cudaSuccess)
      e = copy_rows(kd + a * kv_head, kv_pitch, kh + a * kv_head, kv_pitch,
                    nkv * kv_head, B, max_pitch, cudaMemcpyHostToDevice, r->in);
    if (e == cudaSuccess)
      e = copy_rows(vd + a * kv_head, kv_pitch, vh + a * kv_head, kv_pitch,
                    nkv * kv_head, B, max_pitch, cudaMemcpyHostToDevice, r->in);
    if (e == cudaSuccess) e = cudaEventRecord(r->loaded[c], r->in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, r->loaded[c], 0);
    if (e != cudaSuccess)
      return join_fail(cuda_error(e, "host-to-device copies"));
    // the chunk's forward; its lse goes to [B][nq][Sq] at B * qa * Sq
    float* lse_c = lsed ? lsed + static_cast<size_t>(B) * qa * Sq : nullptr;
    st = bsm_splash_fwd(qd + qa * q_head, kd + a * kv_head, vd + a * kv_head,
                        q_strides, kv_strides, kv_strides, q_strides, B, nq,
                        nkv, Sq, Skv, D, &info, qsd, ksd, scale, score,
                        od + qa * q_head, lse_c, base + L.ws,
                        bsm::kFwdWorkspaceBytes, stream);
    if (st != BSM_OK) return join_fail(st);
    e = cudaEventRecord(r->done[c], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(r->out, r->done[c], 0);
    // out: the chunk's rows of out and lse
    if (e == cudaSuccess)
      e = copy_rows(oh + qa * q_head, q_pitch, od + qa * q_head, q_pitch,
                    nq * q_head, B, max_pitch, cudaMemcpyDeviceToHost, r->out);
    if (e == cudaSuccess && lse != nullptr)
      e = copy_rows(lse + static_cast<size_t>(qa) * Sq,
                    static_cast<size_t>(H) * Sq * 4, lse_c,
                    static_cast<size_t>(nq) * Sq * 4,
                    static_cast<size_t>(nq) * Sq * 4, B,
                    max_pitch, cudaMemcpyDeviceToHost, r->out);
    if (e != cudaSuccess)
      return join_fail(cuda_error(e, "device-to-host copies"));
  }
  // the caller's stream ends after the last copy out; the copy-in stream
  // has nothing left after the last chunk's forward waited for it
  e = cudaEventRecord(r->finish, r->out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, r->finish, 0);
  if (e != cudaSuccess) return cuda_error(e, "stream join");
  return BSM_OK;
}

}  // extern "C"
