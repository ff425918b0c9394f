/*
 * bsm.h -- block-sparse masked attention (Splash-style) on GB300: the
 * forward and its backward.
 *
 * C ABI of libbsm.so.  All compute runs in hand-written CUDA kernels for
 * sm_103a; there is no CPU path.  The library allocates no device memory:
 * the caller owns every buffer (inputs, outputs and the mask-info buffer).
 * Pointers marked "device" must be device (or managed) memory of the current
 * CUDA device; `stream` is a cudaStream_t passed as void* (NULL = the legacy
 * default stream).  Work is enqueued asynchronously; argument errors are
 * returned synchronously, before anything is enqueued, with a message in
 * bsm_last_error().  No function falls back to another algorithm silently.
 *
 * Sources (page title, section):
 *   [HSTU]   RecML "recml/core/ops/hstu_ops.py" -- pointwise splash attention:
 *            _next_nonzero (block classes), _apply_mask (element mask),
 *            _pointwise_splash_attention_fwd_kernel_impl (pointwise scores),
 *            pointwise_splash_attention (API, defaults, argument checks).
 *   [NOTES]  "JAX 到 VLIW, Pallas / Splash Attention 复习笔记" -- section 12
 *            (naive attention), 15 (online softmax m/l/o), 18-19 (grid
 *            h, i, j), 21 (sparse K/V indirection via data_next).
 *   [KERNELS] "Attention Kernels -- Splash, Flash, SDPA on TPU" -- section
 *            "Splash Attention via call_jax" (make_splash_mha(mask) then
 *            kernel(q, k, v)).
 */
#ifndef BSM_H_
#define BSM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bsm_status {
  BSM_OK = 0,
  BSM_ERR_INVALID_ARG = -1,    /* bad shape, pointer, stride or size */
  BSM_ERR_UNSUPPORTED = -2,    /* valid but not built (e.g. head_dim 96) */
  BSM_ERR_CUDA = -3,           /* a CUDA runtime/driver call failed */
  BSM_ERR_DEVICE_TIMEOUT = -4  /* a kernel gave up waiting (see below) */
} bsm_status;

/* Score path.  SOFTMAX: out = softmax(scale * q k^T restricted to the
 * visible keys) v, plus the per-row logsumexp ([NOTES] section 15).
 * POINTWISE: out = sum over visible keys of x*sigmoid(x)/Sq * v with
 * x = scale * q.k, no normalisation ([HSTU] fwd kernel impl). */
typedef enum bsm_score {
  BSM_SCORE_SOFTMAX = 0,
  BSM_SCORE_POINTWISE = 1
} bsm_score;

/* Mask predicates, AND-ed; flags == 0 is the full mask ([HSTU]
 * pointwise_splash_attention: MaskType.CAUSAL / FULL, segment ids).
 *   CAUSAL : key k visible from query q iff k <= q
 *   LOCAL  : iff q - k < window            (window >= 1)
 *   BAND   : with LOCAL only, the window also bounds the keys after q:
 *            iff k - q < window, so LOCAL|BAND is the symmetric sliding
 *            window |q - k| < window (hstu_ops LocalMask((w, w)) with
 *            MaskType.FULL)
 *   SEGMENT: iff q_segment_ids[b][q] == kv_segment_ids[b][k]
 *   DENSE  : iff bit k % 32 of word dense_bits[q * dense_row_words + k / 32]
 *            is set: an arbitrary mask ([HSTU]'s NumpyMask), bit-packed,
 *            one row of dense_row_words >= ceil(Skv / 32) uint32 words per
 *            query row, shared by every batch row and head; device memory
 *            owned by the caller, read by bsm_build_mask_info and again by
 *            bsm_splash_fwd (keep it alive while the mask info is used)
 * Elements past Sq or Skv (a ragged last block) are never visible. */
#define BSM_MASK_CAUSAL 1u
#define BSM_MASK_LOCAL 2u
#define BSM_MASK_SEGMENT 4u
#define BSM_MASK_BAND 8u
#define BSM_MASK_DENSE 16u

typedef struct bsm_mask_spec {
  uint32_t flags;
  int32_t window;  /* used with BSM_MASK_LOCAL only */
  const uint32_t* dense_bits; /* BSM_MASK_DENSE only, else NULL */
  int64_t dense_row_words;    /* BSM_MASK_DENSE only */
} bsm_mask_spec;

/* Mask-info tables ([HSTU] _next_nonzero; [NOTES] section 21), filled by
 * bsm_build_mask_info.  All arrays are device memory inside the caller's
 * buffer.  num_tables is B when SEGMENT is set (one table per batch row),
 * else 1 (shared by all batch rows and heads).  Row r = t*nq + i.
 *   block_mask[t][i][j] int8: 0 empty (never loaded), 1 partial (element
 *                       mask applied), 2 full (no mask)
 *   data_next[t][i][j]  int32: smallest nonzero j' >= j of row i; if none,
 *                       the largest nonzero j' < j; 0 for an empty row
 *   row_ptr[r]          int32, num_tables*nq + 1 entries, CSR offsets
 *   kv_idx[row_ptr[r]..row_ptr[r+1])  nonzero j of row r, ascending
 *   kv_cls[...]         their classes (1 or 2)
 *   seg_range[b][q][2]  int32 (SEGMENT only): first and last key index whose
 *                       segment id equals q's, valid when every kv segment-id
 *                       row is non-decreasing (packed sequences); first > last
 *                       when no key has q's id
 *   seg_flags[0]        int32 (SEGMENT only): bit 0 set if some kv segment-id
 *                       row is not non-decreasing (then seg_range is unused and
 *                       segments are compared element by element); entries
 *                       1..num_tables are the builder's per-table scratch
 *   super_order[k]      int32, num_tables*num_super entries: the pairs
 *                       (table t, super-tile s) as t*num_super + s, ordered by
 *                       decreasing work (query rows times nonzero blocks
 *                       they see, quantised to 19 bits of the largest),
 *                       ties by decreasing index.  A super-tile is 256 query
 *                       rows, the forward's work unit; bsm_splash_fwd hands
 *                       its units out in this order (longest first).  NULL
 *                       when num_tables*num_super > 8192 (the forward then
 *                       takes the last super-tiles first).  Scheduling only:
 *                       no result depends on it.  No counterpart on the
 *                       pages, whose grid walks the query blocks in order.
 * kv_idx/kv_cls have capacity num_tables*nq*nk. */
typedef struct bsm_mask_info {
  uint32_t flags;
  int32_t window;
  int32_t num_tables;
  int32_t Sq, Skv;
  int32_t block_q, block_kv;
  int32_t nq, nk; /* ceil(Sq / block_q), ceil(Skv / block_kv) */
  int8_t* block_mask;
  int32_t* data_next;
  int32_t* row_ptr;
  int32_t* kv_idx;
  int8_t* kv_cls;
  int32_t* seg_range;
  int32_t* seg_flags;
  int32_t num_super; /* ceil(Sq / 256) */
  int32_t* super_order;
  const uint32_t* dense_bits; /* the spec's, for the forward (DENSE only) */
  int64_t dense_row_words;
} bsm_mask_info;

/* Bytes the caller must allocate for bsm_build_mask_info (0 on bad
 * arguments).  B is the batch size (only used with BSM_MASK_SEGMENT). */
size_t bsm_mask_info_bytes(const bsm_mask_spec* spec, int32_t B, int32_t Sq,
                           int32_t Skv, int32_t block_q, int32_t block_kv);

/* Build the mask-info tables on the device ([HSTU] process_mask call in
 * pointwise_splash_attention; class encoding of _next_nonzero; next-block
 * table of [NOTES] section 21).  Exact: block classes come from the same
 * per-element predicate the forward kernel applies.
 *   q_segment_ids  device int32 [B][Sq], contiguous; required iff SEGMENT
 *   kv_segment_ids device int32 [B][Skv]; required iff SEGMENT
 *   block_q, block_kv in {16, 32, 64, 128, 256, 512}
 *   buffer         device, >= bsm_mask_info_bytes(...) bytes, 256-aligned
 *   info           host struct, filled with the shape and pointers into
 *                  `buffer` (valid once the enqueued work has run)
 * Returns BSM_ERR_INVALID_ARG for non-positive/inconsistent sizes, a
 * missing or superfluous segment-id array ([HSTU]: both or neither),
 * window < 1 with LOCAL, or a buffer that is too small or misaligned. */
bsm_status bsm_build_mask_info(const bsm_mask_spec* spec,
                               const int32_t* q_segment_ids,
                               const int32_t* kv_segment_ids, int32_t B,
                               int32_t Sq, int32_t Skv, int32_t block_q,
                               int32_t block_kv, void* buffer,
                               size_t buffer_bytes, bsm_mask_info* info,
                               void* stream);

/* Bit-pack a boolean mask into the BSM_MASK_DENSE layout (the role of
 * [HSTU]'s dense mask array, stored as bits): bit k % 32 of word
 * words[q * row_words + k / 32] is (mask[q * mask_row_stride + k] != 0) for
 * k < Skv; the rest of each row's words are zero.
 *   mask             device uint8 [Sq][mask_row_stride] (torch.bool bytes)
 *   words            device uint32 [Sq][row_words], row_words >=
 *                    ceil(Skv / 32); pass it as bsm_mask_spec.dense_bits
 * One kernel launch on `stream`.  Returns BSM_ERR_INVALID_ARG for negative
 * sizes, row_words or mask_row_stride too small, or a NULL pointer with a
 * nonempty mask. */
bsm_status bsm_pack_dense_mask(const uint8_t* mask, int64_t mask_row_stride,
                               int32_t Sq, int32_t Skv, uint32_t* words,
                               int32_t row_words, void* stream);

/* Block-sparse masked attention forward ([NOTES] sections 15, 18, 21;
 * [HSTU] _pointwise_splash_attention_fwd_kernel_impl).  For each (batch,
 * head, 128-row query tile) the kernel walks only the KV tiles the mask-info
 * marks nonzero; full tiles skip the element mask.
 *   q           device bf16, logical [B][H][Sq][D], head_dim contiguous
 *   k, v        device bf16, logical [B][H_kv][Skv][D], head_dim contiguous
 *   *_strides   element strides of the batch, head and sequence dims
 *               (so [B,H,S,D] and [B,S,H,D] storage both work); every
 *               stride and pointer must be a multiple of 16 bytes
 *   H % H_kv == 0: query head h reads K/V head h / (H / H_kv)
 *   D           64 or 128 (else BSM_ERR_UNSUPPORTED)
 *   info        from bsm_build_mask_info with the same Sq, Skv, mask and
 *               (with SEGMENT) the same B; block_q and block_kv must divide
 *               or be multiples of 128
 *   q/kv_segment_ids  as for bsm_build_mask_info (required iff SEGMENT)
 *   scale       logits are scale * q.k ([HSTU] default 1/sqrt(D))
 *   score       bsm_score
 *   out         device bf16 [B][H][Sq][D] at o_strides, rounded to nearest
 *   lse         SOFTMAX: device f32 [B][H][Sq] contiguous, natural-log
 *               logsumexp of the visible scaled logits (-inf for a row that
 *               sees no key), or NULL; POINTWISE: must be NULL
 *   workspace   device, >= bsm_splash_fwd_workspace_bytes(), 16-aligned:
 *               the persistent CTAs take work units (batch, head, 256 query
 *               rows; heaviest rows first) from a counter kept there and
 *               write the units' KV-tile lists there
 * Rows that see no key get out = 0.  Returns BSM_ERR_UNSUPPORTED for
 * Sq > 262144 or Skv > 262144. */
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
                          void* stream);

/* Bytes of the forward's device workspace (about 6 MiB): the work-unit
 * counter and each CTA's lists of the KV tiles of its next units.  The
 * counter is zeroed on `stream` before each launch; the launch overwrites
 * the rest.  Two forward calls that may run at the same time need separate
 * workspaces. */
size_t bsm_splash_fwd_workspace_bytes(void);

/* Bytes of the device buffer bsm_splash_fwd_host needs (0 on bad
 * arguments): device copies of q, k, v, out, lse (SOFTMAX) and the segment
 * ids (SEGMENT), the mask info and the forward's workspace. */
size_t bsm_splash_fwd_host_bytes(const bsm_mask_spec* spec, int32_t B,
                                 int32_t H, int32_t H_kv, int32_t Sq,
                                 int32_t Skv, int32_t D, int32_t block_q,
                                 int32_t block_kv, int32_t score);

/* The forward on host buffers, end to end (this entry point has no
 * counterpart in the pages; it is a property of this library): copies the
 * inputs to the device, builds the mask info, runs bsm_splash_fwd and
 * copies out (and lse) back, pipelined over n_chunks ranges of K/V heads
 * (their query heads follow): the host-to-device copies of one range, the
 * forward of the previous one and the device-to-host copies of the one
 * before that run at the same time, on two copy streams the library keeps
 * per device (made on the first call in a CUDA context) and the caller's
 * stream.  Each range moves as one strided copy per tensor.
 *   spec, block_q, block_kv, scale, score  as for bsm_build_mask_info and
 *               bsm_splash_fwd (spec->dense_bits, if any, is device memory)
 *   q           host bf16 [B][H][Sq][D], contiguous
 *   k, v        host bf16 [B][H_kv][Skv][D], contiguous
 *   q/kv_segment_ids  host int32 [B][Sq] / [B][Skv]; both iff SEGMENT
 *   out         host bf16 [B][H][Sq][D]; lse host f32 [B][H][Sq] or NULL
 *               (NULL for POINTWISE)
 *   device_buffer  device, >= bsm_splash_fwd_host_bytes(...) bytes,
 *               256-byte aligned, owned by the caller; two calls that may
 *               run at the same time need separate buffers
 *   n_chunks    1..16 head ranges, capped at H_kv; <= 0 picks 4
 * Host memory should be page-locked (cudaHostAlloc / cudaHostRegister):
 * copies from or to pageable memory are correct but do not overlap.
 * Everything is enqueued: the call returns once the work is issued and
 * `stream` waits for the last copy, so out and lse are ready after the
 * stream is synchronised.  Argument errors as for bsm_splash_fwd, found
 * before anything is enqueued; a failure part-way returns its status with
 * the work enqueued until then left to run, `stream` still waiting for it
 * (so the device buffer is free once `stream` is synchronised). */
bsm_status bsm_splash_fwd_host(const bsm_mask_spec* spec, const void* q,
                               const void* k, const void* v,
                               const int32_t* q_segment_ids,
                               const int32_t* kv_segment_ids, int32_t B,
                               int32_t H, int32_t H_kv, int32_t Sq,
                               int32_t Skv, int32_t D, int32_t block_q,
                               int32_t block_kv, float scale, int32_t score,
                               void* out, float* lse, void* device_buffer,
                               size_t device_bytes, int32_t n_chunks,
                               void* stream);

/* bsm_splash_fwd for callers that cannot allocate device memory (this entry
 * point has no counterpart in the pages; it is a property of this library).
 * Plugins handed finished buffers by a host framework, serving engines that
 * reserve all free HBM up front, and loops that cannot afford cudaMalloc's
 * implicit synchronisation can call it: it takes the same arguments as
 * bsm_splash_fwd minus the workspace and allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library routine).  Its workspace is a 6 MiB
 * (bsm_splash_fwd_workspace_bytes()) array in the library's own device
 * code, held on a device from the moment that code is loaded there until
 * the process exits.
 * Limits: Sq, Skv <= 262144 (else BSM_ERR_UNSUPPORTED), at most 256 CTAs
 * (every supported GPU).
 * Set-up: the first call on a device (per CUDA context) looks up the
 * array's device address (cudaGetSymbolAddress, with that device current)
 * and keeps it for later calls in that context.  Under CUDA's default lazy
 * module loading that first call is also where the library's device code,
 * with the array, is loaded into the context, which takes device memory
 * and may synchronise: make it once, before reserving the device's free
 * memory and before any stream capture.  Later calls take no device memory.
 * Sharing: every call on a device uses the same array.  The work-unit
 * counter in it is zeroed on `stream` before each launch (the rest is
 * overwritten), so a call never depends on what an earlier call left there;
 * calls that overlap on the GPU (e.g. on two streams) race on it and must
 * not be issued. */
bsm_status bsm_splash_fwd_noalloc(const void* q, const void* k, const void* v,
                                  const int64_t q_strides[3],
                                  const int64_t k_strides[3],
                                  const int64_t v_strides[3],
                                  const int64_t o_strides[3], int32_t B,
                                  int32_t H, int32_t H_kv, int32_t Sq,
                                  int32_t Skv, int32_t D,
                                  const bsm_mask_info* info,
                                  const int32_t* q_segment_ids,
                                  const int32_t* kv_segment_ids, float scale,
                                  int32_t score, void* out, float* lse,
                                  void* stream);

/* A bf16 tensor in device memory, logical [B][heads][S][D] with head_dim
 * contiguous; strides are in elements for the batch, head and sequence
 * dims (multiples of 8, positive), data 16-byte aligned.  `data` is read
 * for inputs and written for outputs. */
typedef struct bsm_tensor {
  void* data;
  int64_t strides[3];
} bsm_tensor;

/* Bytes of bsm_splash_bwd's device workspace: B*H*Sq floats (the softmax
 * path's per-row D_q = sum_d dO * out), 0 for the pointwise path. */
size_t bsm_splash_bwd_workspace_bytes(int32_t B, int32_t H, int32_t Sq,
                                      int32_t score);

/* Backward of bsm_splash_fwd: dQ, dK, dV of sum(dout * out) over the same
 * mask ([HSTU] _pointwise_splash_attention_bwd_kernel_impl and its
 * launcher, which accumulate dK/dV over query blocks and dQ over key
 * blocks; for the softmax path the forward of [NOTES] section 15,
 * differentiated: with P = exp(scale q.k - lse) over the visible keys and
 * D_q = sum_d dout[q, d] out[q, d],
 *     dV = P^T dout,  dS = P * (dout V^T - D_q),
 *     dQ = scale dS K,  dK = scale dS^T Q;
 * pointwise: with x = scale q.k and sig = logistic(x),
 *     dV = (x sig / Sq)^T dout,  dS = (dout V^T) sig (1 + x (1 - sig)) / Sq,
 *     dQ = scale dS K,  dK = scale dS^T Q).
 * P and dS are rounded to bf16 for the products (as [HSTU]'s backward
 * casts p to the input type); accumulation is f32.
 *   q, k, v, info, segment ids, scale, score: as given to bsm_splash_fwd
 *   out, lse     the forward's output and logsumexp (SOFTMAX; NULL allowed
 *                for POINTWISE)
 *   dout         device bf16 [B][H][Sq][D]: gradient of the output
 *   dq           device bf16 [B][H][Sq][D], written
 *   dk, dv       device bf16 [B][H_kv][Skv][D], written; with H_kv < H the
 *                gradient of a K/V head sums over its group of query heads
 *   workspace    device, >= bsm_splash_bwd_workspace_bytes(B, H, Sq, score)
 *                bytes, 16-byte aligned (may be NULL when that is 0)
 * Rows and keys that see nothing get zero gradients.  Returns the same
 * argument errors as bsm_splash_fwd. */
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
                          void* stream);

/* Synchronise `stream` and report whether a kernel of this library gave up
 * on a bounded wait since the last call (then BSM_ERR_DEVICE_TIMEOUT; the
 * affected outputs are undefined, the CUDA context stays usable).  If
 * `detail` is non-NULL it receives 4 ints: code, block, role, phase. */
bsm_status bsm_device_status(void* stream, int32_t* detail);

/* Failure-detection self test: enqueue one tiny kernel that waits on an
 * mbarrier nothing ever arrives on, with the given limit in nanoseconds
 * (1e3..1e10), so that the bounded wait must run out.  A later
 * bsm_device_status() then returns BSM_ERR_DEVICE_TIMEOUT. */
bsm_status bsm_selftest_wait_timeout(int64_t timeout_ns, void* stream);

/* Tracing (diagnostics).  With a non-NULL device buffer, every following
 * bsm_splash_fwd launch records timestamped events into it: the buffer is
 * split evenly over the launch's CTAs (see bsm_debug_fwd_grid) into
 * 16-byte records; a CTA's records 0-1 hold the event counts of its six
 * recording threads as uint32 {load, mma tile 0, score tile 0, score tile 1,
 * list, mma tile 1, 0, 0}, then come six equal regions, one per thread, of
 * records {uint64 %globaltimer ns, uint32 role<<28 | event<<24 | tile<<20 |
 * entry, uint32 unit}.  NULL (or bytes too small) switches tracing off.  The
 * buffer stays owned by the caller; it must outlive the launches. */
bsm_status bsm_debug_set_trace(void* buffer, size_t bytes);

/* Number of CTAs bsm_splash_fwd launches for these sizes (-1 on error). */
int32_t bsm_debug_fwd_grid(int32_t B, int32_t H, int32_t Sq);

/* Thread-local text of the last error of this thread ("" if none). */
const char* bsm_last_error(void);

/* ABI version (major*10000 + minor*100 + patch): 302 = 0.3.2, adding
 * bsm_splash_fwd_host and bsm_splash_fwd_host_bytes to 0.3.1 (which added
 * bsm_pack_dense_mask to 0.3.0: the backward entry points and bsm_tensor
 * added to 0.2.0's forward, mask spec and mask info). */
int32_t bsm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSM_H_ */
