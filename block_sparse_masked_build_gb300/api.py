"""Python binding of the C ABI (same names as include/bsm.h) plus two thin
conveniences that allocate with torch and call it.

Every step of the computation runs in the CUDA kernels of libbsm.so; this
module only marshals arguments (pointers, strides, the stream) and uses
torch for device memory, pinned host memory and streams.
"""

from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import MaskInfoStruct, MaskSpec, I64x3, TensorView

MASK_CAUSAL = 1
MASK_LOCAL = 2
MASK_SEGMENT = 4
MASK_BAND = 8  # with MASK_LOCAL: |q - k| < window
MASK_DENSE = 16  # arbitrary mask, bit-packed uint32 words per query row
SCORE_SOFTMAX = 0
SCORE_POINTWISE = 1


class BsmError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        name = _lib.STATUS_NAMES.get(status, str(status))
        super().__init__(f"{name}: {message}")


def _check(status: int) -> None:
    if status != _lib.BSM_OK:
        raise BsmError(status, _lib.last_error())


def _stream_handle(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


# --------------------------------------------------------------- C ABI names

def bsm_version() -> int:
    return int(_lib.lib().bsm_version())


def bsm_last_error() -> str:
    return _lib.last_error()


def bsm_mask_info_bytes(flags: int, window: int, B: int, Sq: int, Skv: int,
                        block_q: int, block_kv: int) -> int:
    spec = MaskSpec(flags, window)
    return int(_lib.lib().bsm_mask_info_bytes(ctypes.byref(spec), B, Sq, Skv,
                                              block_q, block_kv))


@dataclass
class MaskInfo:
    """Mask-info tables living in ``buffer`` (a CUDA uint8 tensor)."""

    struct: MaskInfoStruct
    buffer: torch.Tensor
    dense_bits: object = None  # keeps a MASK_DENSE mask alive with the info

    def _view(self, ptr: int, dtype, count: int) -> torch.Tensor:
        off = ptr - self.buffer.data_ptr()
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        return self.buffer[off:off + nbytes].view(dtype)

    @property
    def num_tables(self) -> int:
        return self.struct.num_tables

    @property
    def nq(self) -> int:
        return self.struct.nq

    @property
    def nk(self) -> int:
        return self.struct.nk

    @property
    def block_mask(self) -> torch.Tensor:
        s = self.struct
        return self._view(s.block_mask, torch.int8,
                          s.num_tables * s.nq * s.nk).view(
                              s.num_tables, s.nq, s.nk)

    @property
    def data_next(self) -> torch.Tensor:
        s = self.struct
        return self._view(s.data_next, torch.int32,
                          s.num_tables * s.nq * s.nk).view(
                              s.num_tables, s.nq, s.nk)

    @property
    def row_ptr(self) -> torch.Tensor:
        s = self.struct
        return self._view(s.row_ptr, torch.int32, s.num_tables * s.nq + 1)

    @property
    def seg_range(self) -> torch.Tensor:
        """[B, Sq, 2] first/last key with the row's segment id (SEGMENT)."""
        s = self.struct
        return self._view(s.seg_range, torch.int32,
                          s.num_tables * s.Sq * 2).view(s.num_tables, s.Sq, 2)

    @property
    def seg_flags(self) -> torch.Tensor:
        return self._view(self.struct.seg_flags, torch.int32, 1)

    @property
    def super_order(self):
        """[num_tables * num_super] longest-first (table, 256-row super-tile)
        pairs as table * num_super + super_tile, or None when not built."""
        s = self.struct
        if not s.super_order:
            return None
        return self._view(s.super_order, torch.int32,
                          s.num_tables * s.num_super)

    def kv_lists(self) -> tuple[torch.Tensor, torch.Tensor]:
        """(kv_idx, kv_cls) trimmed to row_ptr[-1] entries (synchronises)."""
        s = self.struct
        nnz = int(self.row_ptr[-1].item())
        idx = self._view(s.kv_idx, torch.int32, s.num_tables * s.nq * s.nk)
        cls = self._view(s.kv_cls, torch.int8, s.num_tables * s.nq * s.nk)
        return idx[:nnz], cls[:nnz]


def bsm_build_mask_info(flags: int, window: int, q_segment_ids, kv_segment_ids,
                        B: int, Sq: int, Skv: int, block_q: int, block_kv: int,
                        buffer: torch.Tensor, stream=None,
                        dense_bits=None) -> MaskInfo:
    """dense_bits: with MASK_DENSE, a device int32/uint32-bits tensor
    [Sq, W] (W >= ceil(Skv / 32), row-major); it must stay alive while the
    mask info is used, since the forward reads it too."""
    spec = MaskSpec(flags, window)
    if dense_bits is not None:
        if dense_bits.dim() != 2 or dense_bits.stride(1) != 1 or \
                dense_bits.element_size() != 4:
            raise ValueError("dense_bits must be a [Sq, W] 32-bit tensor with "
                             "contiguous rows")
        spec.dense_bits = dense_bits.data_ptr()
        spec.dense_row_words = dense_bits.stride(0)
    info = MaskInfoStruct()
    _check(_lib.lib().bsm_build_mask_info(
        ctypes.byref(spec), _ptr(q_segment_ids), _ptr(kv_segment_ids), B, Sq,
        Skv, block_q, block_kv, buffer.data_ptr(),
        buffer.numel() * buffer.element_size(), ctypes.byref(info),
        _stream_handle(stream)))
    return MaskInfo(info, buffer, dense_bits)


def _strides3(t: torch.Tensor):
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("tensors must be 4-D [B, H, S, D] views with a "
                         "contiguous head dimension")
    return I64x3(t.stride(0), t.stride(1), t.stride(2))


def bsm_splash_fwd_workspace_bytes() -> int:
    return int(_lib.lib().bsm_splash_fwd_workspace_bytes())


_workspaces: dict = {}


def _default_workspace(device, stream_handle):
    """One workspace per (device, stream): calls on one stream run in
    order, so they can share it."""
    key = (device, stream_handle)
    ws = _workspaces.get(key)
    if ws is None:
        ws = torch.empty(bsm_splash_fwd_workspace_bytes(), dtype=torch.uint8,
                         device=device)
        _workspaces[key] = ws
    return ws


def bsm_splash_fwd(q, k, v, mask_info: MaskInfo, q_segment_ids,
                   kv_segment_ids, scale: float, score: int, out,
                   lse=None, stream=None, workspace=None) -> None:
    """q [B,H,Sq,D], k/v [B,H_kv,Skv,D], out [B,H,Sq,D] (bf16, CUDA)."""
    B, H, Sq, D = q.shape
    H_kv, Skv = k.shape[1], k.shape[2]
    sh = _stream_handle(stream)
    if workspace is None:
        workspace = _default_workspace(q.device, sh)
    _check(_lib.lib().bsm_splash_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), _strides3(q), _strides3(k),
        _strides3(v), _strides3(out), B, H, H_kv, Sq, Skv, D,
        ctypes.byref(mask_info.struct), _ptr(q_segment_ids),
        _ptr(kv_segment_ids), float(scale), int(score), out.data_ptr(),
        _ptr(lse), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), sh))


def bsm_splash_fwd_host_bytes(flags: int, window: int, B: int, H: int,
                              H_kv: int, Sq: int, Skv: int, D: int,
                              block_q: int, block_kv: int, score: int) -> int:
    spec = MaskSpec(flags, window)
    return int(_lib.lib().bsm_splash_fwd_host_bytes(
        ctypes.byref(spec), B, H, H_kv, Sq, Skv, D, block_q, block_kv, score))


def bsm_splash_fwd_host(flags: int, window: int, q, k, v, q_segment_ids,
                        kv_segment_ids, block_q: int, block_kv: int,
                        scale: float, score: int, out, lse, device_buffer,
                        n_chunks: int = 0, stream=None) -> None:
    """The forward on contiguous CPU tensors (pinned for overlap): q
    [B,H,Sq,D], k/v [B,H_kv,Skv,D] bf16, segment ids int32 [B,S], out
    [B,H,Sq,D] bf16 and lse [B,H,Sq] f32 (or None); device_buffer a CUDA
    uint8 tensor of bsm_splash_fwd_host_bytes(...) bytes.  Enqueued on
    `stream`; out and lse are ready once it is synchronised."""
    B, H, Sq, D = q.shape
    H_kv, Skv = k.shape[1], k.shape[2]
    spec = MaskSpec(flags, window)
    _check(_lib.lib().bsm_splash_fwd_host(
        ctypes.byref(spec), q.data_ptr(), k.data_ptr(), v.data_ptr(),
        _ptr(q_segment_ids), _ptr(kv_segment_ids), B, H, H_kv, Sq, Skv, D,
        block_q, block_kv, float(scale), int(score), out.data_ptr(),
        _ptr(lse), device_buffer.data_ptr(),
        device_buffer.numel() * device_buffer.element_size(), int(n_chunks),
        _stream_handle(stream)))


def bsm_splash_fwd_noalloc(q, k, v, mask_info: MaskInfo, q_segment_ids,
                           kv_segment_ids, scale: float, score: int, out,
                           lse=None, stream=None) -> None:
    """bsm_splash_fwd using the library's own device scratch (allocates
    nothing; calls that overlap on the GPU must not be issued)."""
    B, H, Sq, D = q.shape
    H_kv, Skv = k.shape[1], k.shape[2]
    _check(_lib.lib().bsm_splash_fwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), _strides3(q), _strides3(k),
        _strides3(v), _strides3(out), B, H, H_kv, Sq, Skv, D,
        ctypes.byref(mask_info.struct), _ptr(q_segment_ids),
        _ptr(kv_segment_ids), float(scale), int(score), out.data_ptr(),
        _ptr(lse), _stream_handle(stream)))


def _view(t):
    """bsm_tensor of a 4-D [B, heads, S, D] CUDA tensor view (or None)."""
    if t is None:
        return None
    st = _strides3(t)
    return TensorView(t.data_ptr(), st)


def bsm_splash_bwd_workspace_bytes(B: int, H: int, Sq: int,
                                   score: int) -> int:
    return int(_lib.lib().bsm_splash_bwd_workspace_bytes(B, H, Sq, score))


def bsm_splash_bwd(q, k, v, out, lse, dout, mask_info: MaskInfo,
                   q_segment_ids, kv_segment_ids, scale: float, score: int,
                   dq, dk, dv, stream=None, workspace=None) -> None:
    """Gradients of sum(dout * out): dq [B,H,Sq,D], dk/dv [B,H_kv,Skv,D]
    (bf16, CUDA), from the forward's q, k, v and (softmax) out and lse."""
    B, H, Sq, D = q.shape
    H_kv, Skv = k.shape[1], k.shape[2]
    sh = _stream_handle(stream)
    need = bsm_splash_bwd_workspace_bytes(B, H, Sq, score)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    views = [_view(t) for t in (q, k, v, out, dout, dq, dk, dv)]
    refs = [None if x is None else ctypes.byref(x) for x in views]
    _check(_lib.lib().bsm_splash_bwd(
        refs[0], refs[1], refs[2], refs[3], _ptr(lse), refs[4], B, H, H_kv,
        Sq, Skv, D, ctypes.byref(mask_info.struct), _ptr(q_segment_ids),
        _ptr(kv_segment_ids), float(scale), int(score), refs[5], refs[6],
        refs[7], _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        sh))


def bsm_device_status(stream=None) -> tuple[int, list[int]]:
    detail = (ctypes.c_int32 * 4)()
    st = _lib.lib().bsm_device_status(_stream_handle(stream), detail)
    return int(st), list(detail)


def bsm_selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(_lib.lib().bsm_selftest_wait_timeout(int(timeout_ns),
                                                _stream_handle(stream)))


def bsm_debug_set_trace(buffer) -> None:
    """Trace the following forward launches into ``buffer`` (a CUDA tensor,
    16-byte aligned) or switch tracing off with None."""
    if buffer is None:
        _check(_lib.lib().bsm_debug_set_trace(None, 0))
    else:
        _check(_lib.lib().bsm_debug_set_trace(
            buffer.data_ptr(), buffer.numel() * buffer.element_size()))


def bsm_debug_fwd_grid(B: int, H: int, Sq: int) -> int:
    return int(_lib.lib().bsm_debug_fwd_grid(B, H, Sq))


def decode_trace(buffer, grid: int):
    """Records of a trace buffer as a list per CTA of
    (t_ns, role, event, tile, entry, unit), sorted by time."""
    raw = buffer.cpu().numpy().view("<u8").reshape(-1, 2)
    per = raw.shape[0] // grid
    region = (per - 2) // 6
    out = []
    for c in range(grid):
        blk = raw[c * per:(c + 1) * per]
        counts = blk[0:2].reshape(-1).view("<u4")[:6]
        recs = []
        for r, n in enumerate(counts):
            for i in range(int(n)):
                row = blk[2 + r * region + i]
                a = int(row[1] & 0xFFFFFFFF)
                recs.append((int(row[0]), a >> 28, (a >> 24) & 15,
                             (a >> 20) & 15, a & 0xFFFFF, int(row[1] >> 32)))
        recs.sort()
        out.append(recs)
    return out


# ------------------------------------------------------------ conveniences

def build_mask_info(flags: int, B: int, Sq: int, Skv: int, block_q: int = 128,
                    block_kv: int = 128, window: int = 0, q_segment_ids=None,
                    kv_segment_ids=None, device=None, stream=None,
                    dense_bits=None) -> MaskInfo:
    """Allocate the mask-info buffer with torch and build the tables."""
    nbytes = bsm_mask_info_bytes(flags, window, B, Sq, Skv, block_q, block_kv)
    if nbytes == 0:
        raise BsmError(_lib.BSM_ERR_INVALID_ARG, bsm_last_error())
    if device is None:
        device = (q_segment_ids.device if q_segment_ids is not None
                  else torch.device("cuda"))
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return bsm_build_mask_info(flags, window, q_segment_ids, kv_segment_ids, B,
                               Sq, Skv, block_q, block_kv, buf, stream,
                               dense_bits)


def bsm_pack_dense_mask(mask: torch.Tensor, words: torch.Tensor,
                        stream=None) -> None:
    """Bit-pack a boolean CUDA mask [Sq, Skv] (rows contiguous) into the
    int32/uint32 CUDA tensor words [Sq, W], W >= ceil(Skv / 32): bit k % 32
    of word k // 32 of row q is mask[q, k] (the layout MASK_DENSE reads)."""
    if not (mask.is_cuda and words.is_cuda):
        raise ValueError("mask and words must be CUDA tensors")
    if mask.dim() != 2 or mask.stride(1) != 1 or mask.element_size() != 1:
        raise ValueError("mask must be a [Sq, Skv] bool/uint8 tensor with "
                         "contiguous rows")
    if words.dim() != 2 or words.stride(1) != 1 or words.element_size() != 4:
        raise ValueError("words must be a [Sq, W] 32-bit tensor with "
                         "contiguous rows")
    Sq, Skv = mask.shape
    if words.shape[0] != Sq:
        raise ValueError("words must have one row per mask row")
    _check(_lib.lib().bsm_pack_dense_mask(
        mask.data_ptr(), mask.stride(0), Sq, Skv, words.data_ptr(),
        words.stride(0), _stream_handle(stream)))


def pack_dense_mask(mask: torch.Tensor, stream=None) -> torch.Tensor:
    """bsm_pack_dense_mask into a new int32 tensor [Sq, ceil(Skv / 32)]."""
    Sq, Skv = mask.shape
    if mask.dtype != torch.bool and mask.dtype != torch.uint8:
        mask = mask != 0
    mask = mask.contiguous()
    words = torch.empty((Sq, (Skv + 31) // 32), dtype=torch.int32,
                        device=mask.device)
    bsm_pack_dense_mask(mask, words, stream)
    return words


def splash_attention_bwd(q, k, v, out, lse, dout, *,
                         mask_flags: int = MASK_CAUSAL, window: int = 0,
                         q_segment_ids=None, kv_segment_ids=None,
                         scale: float | None = None,
                         score: int = SCORE_SOFTMAX, block_q: int = 128,
                         block_kv: int = 128,
                         mask_info: MaskInfo | None = None, stream=None,
                         dense_mask=None):
    """Backward of :func:`splash_attention` on CUDA tensors: returns
    (dq, dk, dv) for the gradient ``dout`` of the output.  ``out`` and
    ``lse`` are the forward's (softmax path; ignored for the pointwise
    path)."""
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if mask_info is None:
        bits = None
        if dense_mask is not None:
            bits = pack_dense_mask(dense_mask.to(q.device))
        mask_info = build_mask_info(mask_flags, B, Sq, Skv, block_q, block_kv,
                                    window, q_segment_ids, kv_segment_ids,
                                    device=q.device, stream=stream,
                                    dense_bits=bits)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    sm = score == SCORE_SOFTMAX
    bsm_splash_bwd(q, k, v, out if sm else None, lse if sm else None, dout,
                   mask_info, q_segment_ids, kv_segment_ids, scale, score, dq,
                   dk, dv, stream)
    return dq, dk, dv


def _can_pipeline(q, k, v, out, lse, q_seg, kv_seg, stream, mask_info,
                  dense_mask):
    """Host inputs go through bsm_splash_fwd_host (chunked copies that
    overlap the forward when the memory is pinned) when they and any given
    outputs are contiguous CPU tensors, and no prebuilt mask info or
    arbitrary mask is involved."""
    ts = [q, k, v] + [t for t in (out, lse, q_seg, kv_seg) if t is not None]
    return (all(t.device.type == "cpu" and t.is_contiguous() for t in ts)
            and mask_info is None and dense_mask is None
            and (stream is None or isinstance(stream, torch.cuda.Stream))
            and k.shape[1] > 0 and q.shape[1] % k.shape[1] == 0)


def _splash_host_pipelined(q, k, v, flags, window, q_seg, kv_seg, scale,
                           score, block_q, block_kv, want_lse, out, lse,
                           stream, dev):
    """Host tensors through bsm_splash_fwd_host: one call that copies in,
    builds the mask info, runs the forward and copies out, pipelined over
    ranges of heads on the library's copy streams."""
    B, H, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    comp = torch.cuda.current_stream(dev) if stream is None else stream
    nbytes = bsm_splash_fwd_host_bytes(flags, window, B, H, Hkv, Sq, Skv, D,
                                       block_q, block_kv, score)
    if nbytes == 0:
        raise BsmError(_lib.BSM_ERR_INVALID_ARG,
                       "bsm_splash_fwd_host_bytes: bad arguments")
    with torch.cuda.stream(comp):
        buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty((B, H, Sq, D), dtype=torch.bfloat16,
                          pin_memory=True)
    if want_lse and lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, pin_memory=True)
    qs = None if q_seg is None else q_seg.to(torch.int32).contiguous()
    ks = None if kv_seg is None else kv_seg.to(torch.int32).contiguous()
    bsm_splash_fwd_host(flags, window, q, k, v, qs, ks, block_q, block_kv,
                        scale, score, out, lse if want_lse else None, buf,
                        0, comp)
    comp.synchronize()
    return out, (lse if want_lse else None)


def splash_attention(q, k, v, *, mask_flags: int = MASK_CAUSAL,
                     window: int = 0, q_segment_ids=None, kv_segment_ids=None,
                     scale: float | None = None, score: int = SCORE_SOFTMAX,
                     block_q: int = 128, block_kv: int = 128,
                     mask_info: MaskInfo | None = None,
                     return_lse: bool = True, out=None, lse=None,
                     stream=None, dense_mask=None):
    """Block-sparse masked attention forward, q/k/v [B, H, S, D] bf16.

    Defaults follow hstu_ops ``pointwise_splash_attention``: scale =
    1/sqrt(D).  With CUDA inputs everything stays on the device.  With CPU
    inputs (ideally pinned) the inputs are copied to the current device,
    the kernels run there, and ``out``/``lse`` are copied back into host
    tensors (``out``/``lse`` may be given, pinned, to be reused).
    Returns (out, lse); lse is None for the pointwise path or when
    ``return_lse`` is False.  ``dense_mask`` (with MASK_DENSE) is a boolean
    [Sq, Skv] tensor, an arbitrary mask shared by every batch row and head;
    it is bit-packed on the device here.
    """
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    host = q.device.type == "cpu"
    dev = torch.device("cuda", torch.cuda.current_device()) if host \
        else q.device
    want_lse = return_lse and score == SCORE_SOFTMAX
    if host and _can_pipeline(q, k, v, out, lse, q_segment_ids,
                              kv_segment_ids, stream, mask_info, dense_mask):
        return _splash_host_pipelined(
            q, k, v, mask_flags, window, q_segment_ids, kv_segment_ids,
            scale, score, block_q, block_kv, want_lse, out, lse, stream, dev)
    if host:
        nb = q.is_pinned()
        qd = q.to(dev, non_blocking=nb)
        kd = k.to(dev, non_blocking=nb)
        vd = v.to(dev, non_blocking=nb)
        qs = None if q_segment_ids is None else \
            q_segment_ids.to(dev, non_blocking=nb)
        ks = None if kv_segment_ids is None else \
            kv_segment_ids.to(dev, non_blocking=nb)
    else:
        qd, kd, vd, qs, ks = q, k, v, q_segment_ids, kv_segment_ids
    if mask_info is None:
        bits = None
        if dense_mask is not None:
            bits = pack_dense_mask(dense_mask.to(dev))
        mask_info = build_mask_info(mask_flags, B, Sq, Skv, block_q, block_kv,
                                    window, qs, ks, device=dev, stream=stream,
                                    dense_bits=bits)
    od = torch.empty((B, H, Sq, D), dtype=torch.bfloat16, device=dev) \
        if (host or out is None) else out
    ld = None
    if want_lse:
        ld = torch.empty((B, H, Sq), dtype=torch.float32, device=dev) \
            if (host or lse is None) else lse
    bsm_splash_fwd(qd, kd, vd, mask_info, qs, ks, scale, score, od, ld,
                   stream)
    if not host:
        return od, ld
    if out is None:
        out = torch.empty((B, H, Sq, D), dtype=torch.bfloat16,
                          pin_memory=True)
    out.copy_(od, non_blocking=True)
    if want_lse:
        if lse is None:
            lse = torch.empty((B, H, Sq), dtype=torch.float32,
                              pin_memory=True)
        lse.copy_(ld, non_blocking=True)
    if stream is None:
        torch.cuda.current_stream(dev).synchronize()
    else:
        stream.synchronize()
    return out, (lse if want_lse else None)
