"""ctypes declarations of the C ABI in include/retention.h.

Loading fails loudly when libretention.so has not been built: there is no
fallback implementation anywhere in the package.
"""

from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libretention.so")

RET_OK, RET_EINVAL, RET_EUNSUPPORTED, RET_ECUDA, RET_ETIMEOUT, RET_EWORKSPACE = range(6)
RET_F32, RET_BF16 = 0, 1
RET_PATH_TC, RET_PATH_SIMT, RET_PATH_TC_SINGLE, RET_PATH_TC_CARRY = 1, 2, 3, 4
RET_NOALLOC_SCRATCH_BYTES = 32 << 20

STATUS_NAMES = {
    RET_OK: "RET_OK", RET_EINVAL: "RET_EINVAL", RET_EUNSUPPORTED: "RET_EUNSUPPORTED",
    RET_ECUDA: "RET_ECUDA", RET_ETIMEOUT: "RET_ETIMEOUT", RET_EWORKSPACE: "RET_EWORKSPACE",
}

# Every exported symbol and its (restype, argtypes).
_vp, _i, _i64, _f, _sz, _fp = C.c_void_p, C.c_int, C.c_int64, C.c_float, C.c_size_t, C.POINTER(C.c_float)


class RetGN(C.Structure):
    _fields_ = [("enabled", C.c_int), ("eps", C.c_float), ("weight", _vp), ("bias", _vp)]


_FORWARD = [_vp, _vp, _vp, _i, _fp, _fp, _i, _i, _i, _i, _i, _i64]
SIGNATURES = {
    "ret_chunkwise": (_i, _FORWARD + [_i, _vp, _vp, _vp, _i, C.POINTER(RetGN), _vp, _sz, _vp]),
    "ret_chunkwise_scan": (_i, _FORWARD + [_i, _vp, _vp, _vp, _i, C.POINTER(RetGN), _vp, _sz, _vp]),
    "ret_chunkwise_noalloc": (_i, _FORWARD + [_i, _vp, _vp, _vp, _i, C.POINTER(RetGN), _vp]),
    "ret_chunkwise_rowpos": (_i, _FORWARD[:-1] + [C.POINTER(_i64), _i, _vp, _vp, _vp, _i, C.POINTER(RetGN),
                                                  _vp, _sz, _vp]),
    "ret_parallel": (_i, _FORWARD + [_vp, _vp, _vp, _i, C.POINTER(RetGN), _vp, _sz, _vp]),
    "ret_chunkwise_backward": (_i, [_vp, _vp, _vp, _vp, _i, _fp, _fp, _i, _i, _i, _i, _i, _i64, _i,
                                    _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _sz, _vp]),
    "ret_chunkwise_backward_plan": (_i, [_i, _fp, _i, _i, _i, _i, _i, _i, C.POINTER(_i), C.POINTER(_sz)]),
    "ret_chunkwise_param_grads": (_i, [_vp, _vp, _vp, _vp, _i, _vp, _i, _vp, _vp, _vp, _i, _fp, _fp, _i,
                                       _i, _i, _i, _i, _i64, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "ret_chunkwise_param_grads_plan": (_i, [_i, _i, _i, _i, _i, C.POINTER(_sz)]),
    "ret_groupnorm": (_i, [_vp, _i, _vp, _i, _i, _i, _i, _i, C.POINTER(RetGN), _vp]),
    "ret_groupnorm_backward": (_i, [_vp, _vp, _i, _vp, _f, _i, _i, _i, _i, _vp, _i, _vp, _vp, _vp, _sz,
                                    _vp]),
    "ret_groupnorm_backward_plan": (_i, [_i, _i, _i, _i, C.POINTER(_sz)]),
    "ret_chunk_size": (_i, [_i, _fp, _i, _i, _i, _i]),
    "ret_chunkwise_plan": (_i, [_i, _fp, _i, _i, _i, _i, _i, _i, _i, _i, C.POINTER(_i), C.POINTER(_sz)]),
    "ret_chunkwise_plan_compact": (_i, [_i, _fp, _i, _i, _i, _i, _i, _i, _i, _i, C.POINTER(_i),
                                        C.POINTER(_sz)]),
    "ret_chunkwise_scan_plan": (_i, [_i, _fp, _i, _i, _i, _i, _i, _i, _i, _i, C.POINTER(_i), C.POINTER(_sz)]),
    "ret_parallel_plan": (_i, [_i, _fp, _i, _i, _i, _i, _i, _i, _i, _i, C.POINTER(_i), C.POINTER(_sz)]),
    "ret_matmul": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "ret_msr_block": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _fp, _fp, _i, _i, _i, _i, _i, _i, _i, _i64,
                           _vp, _vp, _vp, _i, _f, _vp, _sz, _vp]),
    "ret_msr_block_plan": (_i, [_fp, _i, _i, _i, _i, _i, _i, _i, C.POINTER(_sz)]),
    "ret_step": (_i, [_vp, _vp, _vp, _i, _fp, _fp, _i, _i, _i, _i, _i64, _vp, _vp, _i,
                      C.POINTER(RetGN), _vp]),
    "ret_rotate": (_i, [_vp, _i, _fp, _i, _i, _i, _i, _i64, _f, _vp, _i, _vp]),
    "ret_decay_row_norm": (_i, [_vp, _i, _fp, _i, _i, _i, _i, _i64, _vp]),
    "ret_sync_status": (_i, [_vp]),
    "ret_selftest_timeout": (_i, [_i, _vp]),
    "ret_force_path": (_i, [_i]),
    "ret_profile_begin": (_i, [_vp, _i]),
    "ret_profile_end": (_i, []),
    "ret_profile_kernel": (C.c_char_p, [_i]),
    "ret_status_string": (C.c_char_p, [_i]),
    "ret_abi_version": (_i, []),
}

_LIB = None


class RetentionError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")


def load(path: str = LIB_PATH):
    """Load libretention.so (after torch, so both share one CUDA runtime)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m linear_recurrent_sequence_prologue_b300.build`")
    import torch  # noqa: F401  (loads libcudart.so.13 first)
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def check(fn: str, status: int) -> None:
    if status != RET_OK:
        raise RetentionError(fn, status)
