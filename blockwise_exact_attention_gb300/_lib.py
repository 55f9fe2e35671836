"""ctypes binding of libbea.so (the C ABI declared in include/bea.h).

Argument marshalling only: torch tensors are described to the library by
pointer, dtype, shape and strides, together with the current CUDA stream.
Nothing here computes; every step of the path runs in the library's
kernels. The library is loaded on first use and a missing build raises.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbea.so")

BEA_BF16 = 0
BEA_F32 = 1

STATUS = {
    0: "BEA_OK",
    -1: "BEA_ERR_ARG",
    -2: "BEA_ERR_SHAPE",
    -3: "BEA_ERR_DTYPE",
    -4: "BEA_ERR_ALIGN",
    -5: "BEA_ERR_UNSUPPORTED",
    -6: "BEA_ERR_CUDA",
    -7: "BEA_ERR_TIMEOUT",
    -8: "BEA_ERR_WORKSPACE",
}

# every symbol include/bea.h declares
EXPORTS = (
    "bea_flash_mha_fwd",
    "bea_flash_mha_fwd_merge",
    "bea_flash_mha_bwd_workspace_size",
    "bea_flash_mha_bwd",
    "bea_ring_merge",
    "bea_get_device_status",
    "bea_status_string",
    "bea_version",
    "bea_selftest_wait_timeout",
    "bea_selftest_inject_abort",
    "bea_last_launch_count",
    "bea_flash_mha_bwd_noalloc",
    "bea_flash_mha_bwd_prepare",
    "bea_flash_mha_bwd_kv_block",
    "bea_flash_mha_bwd_finish",
    "bea_ring_attention_fwd",
    "bea_ring_attention_bwd_workspace_size",
    "bea_ring_attention_bwd",
)


class BeaTensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("ndim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 4),
        ("stride", ctypes.c_int64 * 4),
    ]


class BeaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = load().bea_status_string(code).decode() if _LIB is not None else STATUS.get(code, "?")
        super().__init__(f"{where}: {STATUS.get(code, code)} ({msg})")


_LIB = None


def load() -> ctypes.CDLL:
    """Load libbea.so (built in-tree by ``blockwise_exact_attention_gb300.build``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(BeaTensor)
    vp, i, f, sz, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_int64
    lib.bea_flash_mha_fwd.argtypes = [P, P, P, P, P, f, i, i, i, vp]
    lib.bea_flash_mha_fwd.restype = i
    lib.bea_flash_mha_fwd_merge.argtypes = [P, P, P, P, P, P, f, i, i, i, i64, vp]
    lib.bea_flash_mha_fwd_merge.restype = i
    lib.bea_flash_mha_bwd_workspace_size.argtypes = [i64, i64, i64, i64]
    lib.bea_flash_mha_bwd_workspace_size.restype = sz
    lib.bea_flash_mha_bwd.argtypes = [P, P, P, P, P, P, P, P, P, f, i, i, i, i, vp, sz, vp]
    lib.bea_flash_mha_bwd.restype = i
    lib.bea_ring_merge.argtypes = [P, P, P, P, P, vp]
    lib.bea_ring_merge.restype = i
    lib.bea_get_device_status.argtypes = [vp]
    lib.bea_get_device_status.restype = i
    lib.bea_status_string.argtypes = [i]
    lib.bea_status_string.restype = ctypes.c_char_p
    lib.bea_version.argtypes = []
    lib.bea_version.restype = i
    lib.bea_selftest_wait_timeout.argtypes = [i, vp]
    lib.bea_selftest_wait_timeout.restype = i
    lib.bea_selftest_inject_abort.argtypes = [i]
    lib.bea_selftest_inject_abort.restype = i
    lib.bea_last_launch_count.argtypes = []
    lib.bea_last_launch_count.restype = i
    lib.bea_flash_mha_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, f, i, i, i, i, vp]
    lib.bea_flash_mha_bwd_noalloc.restype = i
    lib.bea_flash_mha_bwd_prepare.argtypes = [P, P, P, vp, sz, vp]
    lib.bea_flash_mha_bwd_prepare.restype = i
    lib.bea_flash_mha_bwd_kv_block.argtypes = [P, P, P, P, P, P, f, i, i, i, i64, i, vp, sz, vp]
    lib.bea_flash_mha_bwd_kv_block.restype = i
    lib.bea_flash_mha_bwd_finish.argtypes = [P, f, i, vp, sz, vp]
    lib.bea_flash_mha_bwd_finish.restype = i
    lib.bea_ring_attention_fwd.argtypes = [P, P, P, P, P, P, i, f, i, i, i, vp]
    lib.bea_ring_attention_fwd.restype = i
    lib.bea_ring_attention_bwd_workspace_size.argtypes = [i64, i64, i64, i64, i]
    lib.bea_ring_attention_bwd_workspace_size.restype = sz
    lib.bea_ring_attention_bwd.argtypes = [P, P, P, P, P, P, P, P, P, i, f, i, i, i, vp, sz, vp]
    lib.bea_ring_attention_bwd.restype = i
    _LIB = lib
    return lib


def describe(data_ptr: int, dtype_code: int, shape, strides) -> BeaTensor:
    t = BeaTensor()
    t.data = data_ptr
    t.dtype = dtype_code
    t.ndim = len(shape)
    for k, (s, st) in enumerate(zip(shape, strides)):
        t.shape[k] = int(s)
        t.stride[k] = int(st)
    return t


def check(code: int, where: str) -> None:
    if code != 0:
        raise BeaError(code, where)
