"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/bea.h declares, and rejects bad arguments with the
documented status codes before touching CUDA."""

import ctypes
import os
import re

import pytest

from blockwise_exact_attention_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "bea.h")

OK, ARG, SHAPE, DTYPE, ALIGN, UNSUP, CUDA, TIMEOUT, WS = 0, -1, -2, -3, -4, -5, -6, -7, -8
BF16, F32 = 0, 1
FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced (validation fails first)


@pytest.fixture(scope="module")
def lib():
    from blockwise_exact_attention_gb300 import build
    build.build()
    return _lib.load()


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bea_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_header_symbol(lib):
    names = header_functions()
    assert len(names) >= 9
    assert sorted(_lib.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_strings(lib):
    assert lib.bea_version() == 1
    for code in (OK, ARG, SHAPE, DTYPE, ALIGN, UNSUP, CUDA, TIMEOUT, WS):
        assert lib.bea_status_string(code)
    assert lib.bea_status_string(12345) == b"unknown status"


def T(shape, dtype=BF16, ptr=FAKE, strides=None):
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    return _lib.describe(ptr, dtype, shape, strides)


def fwd(lib, q, k, v, o, l, scale=0.125, causal=0, wl=-1, wr=-1):
    r = ctypes.byref
    return lib.bea_flash_mha_fwd(r(q) if q else None, r(k), r(v), r(o), r(l), scale, causal, wl, wr, None)


def good(n=1, l=256, h=4, hkv=2, d=128, dt=BF16, lk=None):
    lk = l if lk is None else lk
    return (T([n, l, h, d], dt), T([n, lk, hkv, d], dt), T([n, lk, hkv, d], dt), T([n, l, h, d], dt),
            T([n, h, l], F32))


def test_fwd_rejects_bad_arguments(lib):
    q, k, v, o, l = good()
    assert fwd(lib, None, k, v, o, l) == ARG
    assert fwd(lib, q, k, v, o, l, scale=0.0) == ARG
    assert fwd(lib, q, k, v, o, l, scale=float("nan")) == ARG
    assert fwd(lib, q, k, v, o, l, causal=1, wr=4) == ARG
    assert fwd(lib, q, k, v, o, l, wl=-2) == ARG
    assert fwd(lib, q, k, v, o, l, causal=2) == ARG
    # shapes
    assert fwd(lib, *good(h=4, hkv=3)) == SHAPE
    # lq != lk under a mask is valid (bottom-right alignment); lengths of 2^30 or more are not
    q3, k3, v3, o3, l3 = good(l=1 << 30, lk=300)
    assert fwd(lib, q3, k3, v3, o3, l3, causal=1) == SHAPE
    q4, k4, v4, o4, l4 = good(l=256, lk=1 << 30)
    assert fwd(lib, q4, k4, v4, o4, l4, wl=16) == SHAPE
    assert fwd(lib, q, k, v, o, T([1, 4, 255], F32)) == SHAPE
    assert fwd(lib, q, k, v, T([1, 256, 4], BF16), l) == SHAPE
    assert fwd(lib, q, T([1, 256, 2, 64]), v, o, l) == SHAPE
    # dtypes
    assert fwd(lib, q, T([1, 256, 2, 128], F32), v, o, l) == DTYPE
    assert fwd(lib, q, k, v, o, T([1, 4, 256], BF16)) == DTYPE
    q3, k3, v3, o3, l3 = good(dt=F32)
    assert fwd(lib, q3, k3, v3, T([1, 256, 4, 128], BF16), l3) == DTYPE
    bad = T([1, 256, 4, 128])
    bad.dtype = 7
    assert fwd(lib, bad, k, v, o, l) == DTYPE
    # alignment and layout
    assert fwd(lib, T([1, 256, 4, 128], ptr=FAKE + 2), k, v, o, l) == ALIGN
    assert fwd(lib, T([1, 256, 4, 128], strides=[256 * 512, 512, 128, 2]), k, v, o, l) == ALIGN
    assert fwd(lib, T([1, 256, 4, 128], strides=[256 * 4 * 130, 4 * 130, 130, 1]), k, v, o, l) == ALIGN
    # head dims the tensor-core path does not implement
    assert fwd(lib, *good(d=96)) == UNSUP
    assert fwd(lib, *good(d=256)) == UNSUP
    assert fwd(lib, *good(d=132, dt=F32)) == UNSUP


def test_fwd_accepts_strided_chunk_views_in_validation(lib):
    # a chunk view keeps the parent's strides; validation must not reject it.
    # (a zero-size request passes validation and launches nothing)
    parent = [1, 16384, 16, 128]
    strides = [16384 * 16 * 128, 16 * 128, 128, 1]
    q = T([1, 0, 16, 128], strides=strides)
    k = T([1, 2048, 16, 128], strides=strides)
    o = T([1, 0, 16, 128], strides=strides)
    l = T([1, 16, 0], F32, strides=[16 * 16384, 16384, 1])
    assert fwd(lib, q, k, k, o, l) == OK
    assert parent


def test_bwd_rejects_bad_arguments(lib):
    q, k, v, o, l = good()
    do = T([1, 256, 4, 128])
    dq, dk, dv = T([1, 256, 4, 128], F32), T([1, 256, 2, 128], F32), T([1, 256, 2, 128], F32)
    need = lib.bea_flash_mha_bwd_workspace_size(1, 256, 4, 128)
    assert need == 1 * 4 * 256 * 128 * 4 + 2 * 1 * 4 * 256 * 4
    r = ctypes.byref

    def call(dq=dq, dk=dk, dv=dv, acc=0, ws=FAKE, wsb=need, do=do, out=o):
        return lib.bea_flash_mha_bwd(r(do), r(q), r(k), r(v), r(out), r(l), r(dq), r(dk), r(dv), 0.125, 1, -1, -1,
                                     acc, ws, wsb, None)

    assert call(wsb=need - 1) == WS
    assert call(ws=None) == WS
    assert call(ws=FAKE + 128) == WS
    assert call(acc=2) == ARG
    assert call(dq=T([1, 256, 4, 128], BF16), acc=1) == DTYPE
    assert call(do=T([1, 256, 4, 128], F32)) == DTYPE
    assert call(dk=T([1, 256, 4, 128], F32)) == SHAPE
    assert call(out=T([1, 256, 4, 128], F32), ws=FAKE + 8) == WS


def test_staged_bwd_rejects_bad_arguments(lib):
    q, k, v, o, l = good()
    do = T([1, 256, 4, 128])
    dq, dk, dv = T([1, 256, 4, 128], F32), T([1, 256, 2, 128], F32), T([1, 256, 2, 128], F32)
    need = lib.bea_flash_mha_bwd_workspace_size(1, 256, 4, 128)
    r = ctypes.byref

    def prep(do=do, out=o, lse=l, ws=FAKE, wsb=need):
        return lib.bea_flash_mha_bwd_prepare(r(do), r(out), r(lse), ws, wsb, None)

    def block(q=q, k=k, dk=dk, dv=dv, acc=1, ws=FAKE, wsb=need, causal=1, wr=-1):
        return lib.bea_flash_mha_bwd_kv_block(r(do), r(q), r(k), r(v), r(dk), r(dv), 0.125, causal, -1, wr, 0, acc,
                                              ws, wsb, None)

    def fin(dq=dq, acc=0, ws=FAKE, wsb=need, scale=0.125):
        return lib.bea_flash_mha_bwd_finish(r(dq), scale, acc, ws, wsb, None)

    assert prep(wsb=need - 1) == WS
    assert prep(ws=FAKE + 64) == WS
    assert prep(lse=T([1, 4, 255], F32)) == SHAPE
    assert prep(do=T([1, 256, 4, 128], F32), out=T([1, 256, 4, 128], F32)) == UNSUP
    assert prep(do=T([1, 256, 4, 96]), out=T([1, 256, 4, 96])) == UNSUP
    assert block(wsb=need - 1) == WS
    assert block(dk=T([1, 256, 2, 128], BF16)) == DTYPE        # accumulate needs f32
    assert block(dk=T([1, 256, 4, 128], F32)) == SHAPE
    assert block(acc=2) == ARG
    assert block(wr=3) == ARG                                  # causal with a right window
    assert block(q=T([1, 256, 4, 128], F32), k=T([1, 256, 2, 128], F32)) == DTYPE
    assert fin(acc=1, dq=T([1, 256, 4, 128], BF16)) == DTYPE
    assert fin(scale=0.0) == ARG
    assert fin(wsb=need - 1) == WS
    assert fin(dq=T([1, 256, 4, 64], F32), wsb=lib.bea_flash_mha_bwd_workspace_size(1, 256, 4, 64) - 1) == WS


def test_fwd_merge_rejects_bad_arguments(lib):
    q, k, v, o, l = good()
    r = ctypes.byref
    acc = T([1, 256, 4, 128], F32)

    def call(q=q, k=k, acc=acc, lse=l, fin=None, off=0):
        return lib.bea_flash_mha_fwd_merge(r(q), r(k), r(v), r(acc), r(lse), r(fin) if fin is not None else None,
                                           0.125, 1, -1, -1, off, None)

    assert call(acc=T([1, 256, 4, 128], BF16)) == DTYPE          # the accumulator is fp32
    assert call(acc=T([1, 255, 4, 128], F32)) == SHAPE
    assert call(lse=T([1, 4, 255], F32)) == SHAPE
    assert call(fin=T([1, 256, 4, 128], F32)) == DTYPE           # the final copy is bf16
    assert call(q=T([1, 256, 4, 128], F32), k=T([1, 256, 2, 128], F32)) == DTYPE  # v stays bf16
    assert call(acc=T([1, 256, 4, 128], F32, ptr=FAKE + 4)) == ALIGN
    assert call(off=(1 << 30) + 1) == ARG                        # key offset out of range


def test_merge_rejects_bad_arguments(lib):
    r = ctypes.byref
    acc, la = T([1, 64, 2, 128], F32), T([1, 2, 64], F32)
    blk, lb = T([1, 64, 2, 128], BF16), T([1, 2, 64], F32)
    assert lib.bea_ring_merge(r(T([1, 64, 2, 128], BF16)), r(la), r(blk), r(lb), None, None) == DTYPE
    assert lib.bea_ring_merge(r(acc), r(T([1, 2, 63], F32)), r(blk), r(lb), None, None) == SHAPE
    assert lib.bea_ring_merge(r(T([1, 64, 2, 96], F32)), r(la), r(T([1, 64, 2, 96])), r(lb), None, None) == UNSUP
    assert lib.bea_ring_merge(r(acc), r(la), r(blk), r(lb), r(T([1, 64, 2, 128], F32)), None) == DTYPE
    assert lib.bea_ring_merge(r(acc), r(la), r(T([1, 64, 2, 128], BF16, ptr=FAKE + 4)), r(lb), None, None) == ALIGN


def test_selftest_argument_range(lib):
    assert lib.bea_selftest_wait_timeout(0, None) == ARG
    assert lib.bea_selftest_wait_timeout(2000001, None) == ARG
    assert lib.bea_selftest_inject_abort(-2) == ARG
    assert lib.bea_selftest_inject_abort(3) == 0     # armed (one-shot) ...
    assert lib.bea_selftest_inject_abort(-1) == 0    # ... and disarmed again before any launch


def _bwd_args(n=1, l=256, h=4, hkv=2, d=128, dt=BF16, gdt=F32):
    q, k, v, o, lse = good(n=n, l=l, h=h, hkv=hkv, d=d, dt=dt)
    do = T([n, l, h, d], dt)
    return [do, q, k, v, o, lse, T([n, l, h, d], gdt), T([n, l, hkv, d], gdt), T([n, l, hkv, d], gdt)]


def noalloc(lib, args, scale=0.125, causal=1, wl=-1, wr=-1, acc=0):
    r = ctypes.byref
    return lib.bea_flash_mha_bwd_noalloc(*[r(a) if a is not None else None for a in args], scale, causal, wl, wr,
                                         acc, None)


def test_noalloc_checks_arguments_before_its_size(lib):
    """A malformed call gets the error bea_flash_mha_bwd would give, not the array-size error,
    even when its (malformed) shape would need more workspace than the array holds."""
    big = 1 << 20  # needs ~2 GiB of workspace at h = 4, d = 128
    args = _bwd_args(l=big)
    args[0] = None                                      # dout missing
    assert noalloc(lib, args) == ARG
    args = _bwd_args(l=big)
    args[6] = T([1, big, 4, 64], F32)                   # dq of the wrong shape
    assert noalloc(lib, args) == SHAPE
    assert noalloc(lib, _bwd_args(l=big), scale=-1.0) == ARG
    assert noalloc(lib, _bwd_args(l=big, gdt=BF16), acc=1) == DTYPE
    assert noalloc(lib, _bwd_args(l=big, h=4, hkv=3)) == SHAPE
    # well-formed but too large for the array: only now the size error
    assert noalloc(lib, _bwd_args(l=big)) == WS


def test_workspace_size_saturates(lib):
    huge = (1 << 31) - 1
    assert lib.bea_flash_mha_bwd_workspace_size(huge, huge, huge, 128) == (1 << 64) - 1
    assert lib.bea_flash_mha_bwd_workspace_size(1, 8192, 32, 128) == (
        1 * 32 * 8192 * 128 * 4 + 2 * 32 * 8192 * 4)
    # a tensor whose element count overflows 64 bits is rejected, not wrapped
    args = _bwd_args()
    args[1] = T([huge, huge, huge, 128], BF16, strides=[16, 16, 16, 1])
    assert noalloc(lib, args) != OK


def test_ring_calls_reject_bad_arguments(lib):
    r = ctypes.byref
    q, k, v, o, l = good(l=256)
    acc = T([1, 256, 4, 128], F32)

    def rf(q_=q, acc_=acc, fin=None, C=2, causal=1, wl=-1, wr=-1, lse=l):
        return lib.bea_ring_attention_fwd(r(q_), r(k), r(v), r(acc_), r(lse), r(fin) if fin else None, C, 0.1,
                                          causal, wl, wr, None)
    assert rf(C=3) == ARG                      # 256 rows do not split into 3 chunks
    assert rf(C=0) == ARG
    assert rf(acc_=T([1, 256, 4, 128], BF16)) == DTYPE
    assert rf(fin=T([1, 256, 4, 128], F32)) == DTYPE
    assert rf(causal=1, wr=5) == ARG
    qf, kf, vf, _, _ = good(l=256, dt=F32)
    assert lib.bea_ring_attention_fwd(r(qf), r(kf), r(vf), r(acc), r(l), None, 2, 0.1, 1, -1, -1, None) == UNSUP
    q2, k2, v2, _, _ = good(l=256, lk=128)   # ring chunks pair equal lengths only
    assert lib.bea_ring_attention_fwd(r(q2), r(k2), r(v2), r(acc), r(l), None, 2, 0.1, 0, -1, -1, None) == SHAPE
    # backward
    assert lib.bea_ring_attention_bwd_workspace_size(1, 256, 4, 128, 3) == 0
    ws_need = lib.bea_ring_attention_bwd_workspace_size(1, 16384, 16, 128, 8)
    assert ws_need == lib.bea_flash_mha_bwd_workspace_size(8, 2048, 16, 128)
    args = _bwd_args(l=256)
    ws = FAKE

    def rb(a=args, C=2, nbytes=1 << 30, wsp=ws):
        return lib.bea_ring_attention_bwd(*[r(x) for x in a], C, 0.1, 1, -1, -1, wsp, nbytes, None)
    assert rb(C=3) == ARG
    assert rb(nbytes=16) == WS
    assert rb(wsp=FAKE + 16) == WS            # not 256-byte aligned
    bad = list(args)
    bad[6] = T([1, 256, 4, 128], BF16)        # dq must be f32
    assert rb(a=bad) == DTYPE
