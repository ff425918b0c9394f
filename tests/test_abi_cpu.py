"""C-ABI checks that need no GPU: the library builds for sm_103a, loads,
exports every function include/bsm.h declares, and rejects bad arguments
before it touches the device."""

import ctypes
import os
import re

import pytest

from block_sparse_masked_build_gb300 import build as bsm_build
from block_sparse_masked_build_gb300 import _lib
from block_sparse_masked_build_gb300._lib import MaskInfoStruct, MaskSpec, I64x3

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bsm.h")

INVALID = _lib.BSM_ERR_INVALID_ARG
UNSUPPORTED = _lib.BSM_ERR_UNSUPPORTED


@pytest.fixture(scope="module")
def lib():
    bsm_build.build()
    return _lib.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsm_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("bsm_mask_info_bytes", "bsm_build_mask_info", "bsm_splash_fwd",
              "bsm_splash_bwd", "bsm_splash_bwd_workspace_bytes",
              "bsm_device_status", "bsm_last_error", "bsm_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
    assert lib.bsm_version() == 302 == _lib.ABI_VERSION


def test_library_is_built_for_sm_103a(lib):
    # the cubin's target is recorded in the ELF notes; cuobjdump is not
    # needed: the build command carries exactly one -gencode for sm_103a
    assert bsm_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def _align(x, a=256):
    return (x + a - 1) // a * a


@pytest.mark.parametrize("flags,B,Sq,Skv,bq,bkv", [
    (1, 4, 2048, 2048, 128, 128), (5, 2, 8192, 8192, 128, 128),
    (3, 1, 32768, 32768, 128, 128), (1, 1, 256, 256, 64, 64),
    (4, 3, 700, 300, 64, 32), (4, 9, 262144, 256, 512, 512)])
def test_mask_info_bytes_layout(lib, flags, B, Sq, Skv, bq, bkv):
    T = B if flags & 4 else 1
    nq, nk = -(-Sq // bq), -(-Skv // bkv)
    cells = T * nq * nk
    seg_rows = B * Sq if flags & 4 else 0
    pairs = T * -(-Sq // 256)  # (table, 256-row super-tile) pairs
    want = (_align(cells) + _align(4 * cells) + _align(4 * (T * nq + 1))
            + _align(4 * cells) + _align(cells) + _align(8 * seg_rows)
            + _align(4 * (1 + (T if flags & 4 else 0)))
            + (_align(4 * pairs) if pairs <= 8192 else 0))
    if T * nq < 2 ** 24 and cells <= 2 ** 20:
        # one-launch build: uint16 staged row lists and the ticket word
        want += _align(2 * cells) + _align(8)
    spec = MaskSpec(flags, 4096 if flags & 2 else 0)
    assert lib.bsm_mask_info_bytes(ctypes.byref(spec), B, Sq, Skv, bq,
                                   bkv) == want


@pytest.mark.parametrize("flags,window,bq,bkv,Sq", [
    (1, 0, 100, 128, 256), (1, 0, 8, 128, 256), (1, 0, 128, 1024, 256),
    (2, 0, 128, 128, 256), (8, 0, 128, 128, 256), (1, 0, 128, 128, -1),
    (32, 0, 128, 128, 256)])
def test_mask_info_bytes_rejects(lib, flags, window, bq, bkv, Sq):
    spec = MaskSpec(flags, window)
    assert lib.bsm_mask_info_bytes(ctypes.byref(spec), 1, Sq, 256, bq,
                                   bkv) == 0


def _build(lib, spec, qs, ks, B, Sq, Skv, bq, bkv, buf, nbytes):
    info = MaskInfoStruct()
    return lib.bsm_build_mask_info(
        None if spec is None else ctypes.byref(spec), qs, ks, B, Sq, Skv, bq,
        bkv, buf, nbytes, ctypes.byref(info), None)


def test_dense_mask_needs_its_bits(lib):
    # an arbitrary mask without its bit array, or with rows shorter than
    # ceil(Skv / 32) words, is rejected before any device work
    spec = MaskSpec(16, 0)
    assert _build(lib, spec, None, None, 1, 256, 256, 64, 64, 0x100000,
                  1 << 20) == INVALID
    assert "dense" in _lib.last_error()
    spec.dense_bits = 0x200000
    spec.dense_row_words = 7  # 256 keys need 8 words
    assert _build(lib, spec, None, None, 1, 256, 256, 64, 64, 0x100000,
                  1 << 20) == INVALID


def test_build_mask_info_argument_errors(lib):
    ok = MaskSpec(1, 0)
    big = 1 << 30
    buf = 0x100000  # never dereferenced: every case fails validation first
    assert _build(lib, None, None, None, 1, 256, 256, 64, 64, buf, big) == INVALID
    assert _build(lib, MaskSpec(2, 0), None, None, 1, 256, 256, 64, 64, buf,
                  big) == INVALID
    assert "window" in _lib.last_error()
    # segment ids: both or neither (hstu_ops pointwise_splash_attention)
    assert _build(lib, MaskSpec(4, 0), 0x1000, None, 1, 256, 256, 64, 64, buf,
                  big) == INVALID
    assert _build(lib, ok, 0x1000, 0x2000, 1, 256, 256, 64, 64, buf,
                  big) == INVALID
    assert "SEGMENT" in _lib.last_error()
    assert _build(lib, ok, None, None, 1, 256, 256, 64, 64, 0x100010,
                  big) == INVALID
    assert "aligned" in _lib.last_error()
    assert _build(lib, ok, None, None, 1, 256, 256, 64, 64, buf, 16) == INVALID
    assert "too small" in _lib.last_error()
    assert _build(lib, ok, None, None, 1, 300000, 256, 64, 64, buf,
                  big) == UNSUPPORTED
    assert _build(lib, ok, None, None, 1, 256, 256, 48, 64, buf,
                  big) == INVALID


def _fwd(lib, info, B=1, H=2, Hkv=2, Sq=256, Skv=256, D=128, score=0,
         lse=None, seg=(None, None), strides=None, q=0x10000, ws=0x70000,
         wsb=256 + 256 * 2 * 3 * 2048 * 2):
    st = strides or (H * Sq * D, Sq * D, D)
    s3 = I64x3(*st)
    kv3 = I64x3(Hkv * Skv * D, Skv * D, D)
    return lib.bsm_splash_fwd(q, 0x20000, 0x30000, s3, kv3, kv3, s3, B, H,
                              Hkv, Sq, Skv, D, ctypes.byref(info), seg[0],
                              seg[1], 0.125, score, 0x40000, lse, ws, wsb,
                              None)


def _info(flags=1, Sq=256, Skv=256, bq=128, bkv=128, tables=1):
    i = MaskInfoStruct()
    i.flags, i.window, i.num_tables = flags, 0, tables
    i.Sq, i.Skv, i.block_q, i.block_kv = Sq, Skv, bq, bkv
    i.nq, i.nk = -(-Sq // bq), -(-Skv // bkv)
    i.num_super = -(-Sq // 256)
    i.block_mask = 0x50000
    return i


def test_splash_fwd_argument_errors(lib):
    info = _info()
    assert _fwd(lib, info, D=96) == UNSUPPORTED
    assert "head_dim" in _lib.last_error()
    assert _fwd(lib, info, H=3, Hkv=2) == INVALID
    assert _fwd(lib, info, score=1, lse=0x60000) == INVALID
    assert "logsumexp" in _lib.last_error()
    assert _fwd(lib, info, score=7) == INVALID
    assert _fwd(lib, _info(Sq=512)) == INVALID           # info for other Sq
    assert _fwd(lib, _info(flags=5, tables=1), B=2) == INVALID
    assert _fwd(lib, _info(flags=5, tables=1)) == INVALID  # no segment ids
    assert _fwd(lib, info, seg=(0x1000, 0x2000)) == INVALID
    assert _fwd(lib, info, strides=(2 * 256 * 128, 256 * 128, 100)) == INVALID
    assert "multiples of 8" in _lib.last_error()
    assert _fwd(lib, info, q=0x10004) == INVALID
    assert _fwd(lib, info, Sq=300000, Skv=300000) == UNSUPPORTED
    assert _fwd(lib, info, ws=None) == INVALID
    assert _fwd(lib, info, wsb=8) == INVALID
    assert "workspace" in _lib.last_error()
    assert lib.bsm_splash_fwd_workspace_bytes() == 256 + 256 * 2 * 3 * 2048 * 2
    # an arbitrary-mask info must carry its bits, with full rows
    dense = _info(flags=16)
    assert _fwd(lib, dense) == INVALID
    assert "dense" in _lib.last_error()
    dense.dense_bits, dense.dense_row_words = 0x80000, 7  # 256 keys: 8 words
    assert _fwd(lib, dense) == INVALID
    # mask info whose super-tile count does not match Sq
    bad = _info()
    bad.num_super = 3
    assert _fwd(lib, bad) == INVALID


def test_splash_fwd_empty_input_is_a_no_op(lib):
    # B = 0 or Sq = 0: nothing to do, nothing touched
    assert _fwd(lib, _info(), B=0) == 0
    assert _fwd(lib, _info(Sq=0, bq=128), Sq=0) == 0


def test_selftest_rejects_out_of_range_limits(lib):
    assert lib.bsm_selftest_wait_timeout(10, None) == INVALID
    assert lib.bsm_selftest_wait_timeout(10**12, None) == INVALID


def test_dense_packing_needs_cuda_tensors():
    # packing runs in the library's kernel only: CPU tensors are refused,
    # never packed on the host
    import pytest as _pytest
    import torch
    import block_sparse_masked_build_gb300 as bsm
    m = torch.zeros((4, 40), dtype=torch.bool)
    w = torch.zeros((4, 2), dtype=torch.int32)
    with _pytest.raises(ValueError):
        bsm.bsm_pack_dense_mask(m, w)


def test_pack_dense_mask_argument_checks(lib):
    # row_words below ceil(Skv / 32), a row stride below Skv, negative sizes
    assert lib.bsm_pack_dense_mask(None, 64, 4, 64, None, 1, None) == INVALID
    assert lib.bsm_pack_dense_mask(None, 32, 4, 64, None, 2, None) == INVALID
    assert lib.bsm_pack_dense_mask(None, 64, -1, 64, None, 2, None) == INVALID
    assert lib.bsm_pack_dense_mask(None, 64, 4, 64, None, 2, None) == INVALID
    # an empty mask is a no-op
    assert lib.bsm_pack_dense_mask(None, 0, 0, 0, None, 0, None) == 0


def test_bwd_workspace_bytes(lib):
    # the softmax backward keeps D_q = sum_d dO * out per row (f32), the
    # pointwise one needs no workspace
    assert lib.bsm_splash_bwd_workspace_bytes(2, 16, 8192, 0) == 2 * 16 * 8192 * 4
    assert lib.bsm_splash_bwd_workspace_bytes(1, 3, 100, 0) == 1280
    assert lib.bsm_splash_bwd_workspace_bytes(2, 16, 8192, 1) == 0
    assert lib.bsm_splash_bwd_workspace_bytes(-1, 16, 8192, 0) == 0


def test_host_entry_buffer_bytes(lib):
    # device copies of q, k, v, out, lse and the segment ids, the mask info
    # and the forward's workspace, each 256-aligned
    spec = MaskSpec(5, 0)
    B, H, Hkv, S, D = 2, 16, 4, 8192, 128
    mi = lib.bsm_mask_info_bytes(ctypes.byref(spec), B, S, S, 128, 128)
    ws = lib.bsm_splash_fwd_workspace_bytes()
    qo, kv = B * H * S * D * 2, B * Hkv * S * D * 2
    want = (2 * _align(qo) + 2 * _align(kv) + _align(B * H * S * 4)
            + 2 * _align(B * S * 4) + _align(mi) + _align(ws))
    got = lib.bsm_splash_fwd_host_bytes(ctypes.byref(spec), B, H, Hkv, S, S,
                                        D, 128, 128, 0)
    assert got == want
    # pointwise: no lse; no segment ids without SEGMENT
    causal = MaskSpec(1, 0)
    mi1 = lib.bsm_mask_info_bytes(ctypes.byref(causal), B, S, S, 128, 128)
    got = lib.bsm_splash_fwd_host_bytes(ctypes.byref(causal), B, H, Hkv, S,
                                        S, D, 128, 128, 1)
    assert got == 2 * _align(qo) + 2 * _align(kv) + _align(mi1) + _align(ws)
    # bad block size or negative size
    assert lib.bsm_splash_fwd_host_bytes(ctypes.byref(spec), B, H, Hkv, S, S,
                                         D, 100, 128, 0) == 0
    assert lib.bsm_splash_fwd_host_bytes(ctypes.byref(spec), -1, H, Hkv, S,
                                         S, D, 128, 128, 0) == 0


def _host(lib, flags=1, B=2, H=4, Hkv=4, S=256, D=128, score=0, q=0x10000,
          seg=(None, None), lse=0x30000, buf=0x100000, nbuf=None):
    spec = MaskSpec(flags, 0)
    if nbuf is None:
        nbuf = lib.bsm_splash_fwd_host_bytes(ctypes.byref(spec), max(B, 0),
                                             max(H, 0), max(Hkv, 1), max(S, 0),
                                             max(S, 0), 128, 128, 128, score)
    return lib.bsm_splash_fwd_host(
        ctypes.byref(spec), q, 0x20000, 0x20000, seg[0], seg[1], B, H, Hkv, S,
        S, D, 128, 128, 0.1, score, 0x40000, lse, buf, nbuf, 0, None)


def test_host_entry_argument_errors(lib):
    # every check below is made before anything touches the device
    assert _host(lib, D=96) == UNSUPPORTED
    assert "head_dim" in _lib.last_error()
    assert _host(lib, H=3, Hkv=2) == INVALID
    assert _host(lib, score=1) == INVALID               # pointwise with lse
    assert "logsumexp" in _lib.last_error()
    assert _host(lib, score=5) == INVALID
    assert _host(lib, flags=5) == INVALID               # SEGMENT, no ids
    assert _host(lib, seg=(0x50000, 0x60000)) == INVALID  # ids, no SEGMENT
    assert _host(lib, flags=5, seg=(0x50000, None)) == INVALID
    assert "segment" in _lib.last_error()
    assert _host(lib, q=None) == INVALID
    assert _host(lib, buf=None) == INVALID
    assert _host(lib, buf=0x100010) == INVALID           # not 256-aligned
    assert _host(lib, nbuf=1024) == INVALID
    assert "device buffer" in _lib.last_error()
    assert _host(lib, B=-1) == INVALID


def test_host_entry_empty_input_is_a_no_op(lib):
    assert _host(lib, B=0, q=None, lse=None) == 0
    assert _host(lib, S=0, q=None, lse=None) == 0
