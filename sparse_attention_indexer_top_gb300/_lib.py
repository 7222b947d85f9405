"""ctypes binding of libsai.so: loads the in-tree library and declares the
C signatures of include/sai.h. Argument marshalling only."""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsai.so")

_c_i64 = ctypes.c_int64
_c_i32 = ctypes.c_int32
_c_size = ctypes.c_size_t
_vp = ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/sai.h
SIGNATURES = {
    "sai_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "sai_last_error": (ctypes.c_char_p, []),
    "sai_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int), ctypes.c_int, _vp]),
    "sai_test_stall_next_fused": (None, [_c_i32]),
    "sai_topk_transform_workspace": (_c_size, [_c_i64, _c_i64, _c_i32]),
    "sai_topk_transform": (ctypes.c_int, [_vp, _c_i64, _c_i64, _vp, _vp, _vp, _c_i64, _c_i64, _vp, _c_i32, _c_i32,
                                          _vp, _vp, _c_i32, _vp, _vp, _vp, _c_size, _vp]),
    "sai_index_score_topk_workspace": (_c_size, [_c_i64, _c_i32, _c_i32, _c_i32]),
    "sai_index_score_topk": (ctypes.c_int, [_vp, _vp, _vp, _vp, _c_i64, _vp, _c_i64, _c_i64, _vp, _vp, _c_i64, _c_i32,
                                            _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _vp, _vp, _vp, _c_i32, _vp, _vp,
                                            _vp, _c_size, _vp]),
    "sai_index_score": (ctypes.c_int, [_vp, _vp, _vp, _vp, _c_i64, _vp, _c_i64, _c_i64, _vp, _vp, _c_i64, _c_i32, _c_i32,
                                       _c_i32, _c_i32, _c_i32, _vp, _c_i64, _vp]),
    "sai_index_score_topk_bf16": (ctypes.c_int, [_vp, _vp, _vp, _vp, _c_i64, _vp, _c_i64, _c_i64, _vp, _vp, _c_i64,
                                                 _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _vp, _vp, _vp,
                                                 _c_i32, _vp, _vp, _vp, _c_size, _vp]),
    "sai_index_score_bf16": (ctypes.c_int, [_vp, _vp, _vp, _vp, _c_i64, _vp, _c_i64, _c_i64, _vp, _vp, _c_i64, _c_i32,
                                            _c_i32, _c_i32, _c_i32, _c_i32, _vp, _c_i64, _vp]),
    "sai_index_score_topk_per_head_workspace": (_c_size, [_c_i64, _c_i32, _c_i32]),
    "sai_index_score_per_head": (ctypes.c_int, [_vp, _vp, _vp, _vp, _c_i64, _vp, _c_i64, _c_i64, _vp, _vp, _c_i64,
                                                _c_i32, _c_i32, _c_i32, _c_i32, _vp, _c_i64, _vp]),
    "sai_index_score_per_head_bf16": (ctypes.c_int, [_vp, _vp, _vp, _vp, _c_i64, _vp, _c_i64, _c_i64, _vp, _vp,
                                                     _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _vp, _c_i64, _vp]),
    "sai_index_score_topk_per_head": (ctypes.c_int, [_vp, _vp, _vp, _vp, _c_i64, _vp, _c_i64, _c_i64, _vp, _vp,
                                                     _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _vp, _vp, _vp,
                                                     _c_size, _vp]),
    "sai_index_score_topk_per_head_bf16": (ctypes.c_int, [_vp, _vp, _vp, _vp, _c_i64, _vp, _c_i64, _c_i64, _vp, _vp,
                                                          _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _vp, _vp,
                                                          _vp, _c_size, _vp]),
    "sai_topk_transform_noalloc": (ctypes.c_int, [_vp, _c_i64, _c_i64, _vp, _vp, _vp, _c_i64, _c_i64, _vp, _c_i32,
                                                  _c_i32, _vp, _vp, _vp]),
    "sai_sparse_blocks": (ctypes.c_int, [_vp, _c_i64, _c_i32, _c_i32, _vp, _vp, _vp]),
}

_lib = None


class SaiError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == -5:
            detail = " [" + load().sai_last_error().decode() + "]"
        super().__init__(f"{where}: {status_string(status)} (status {status}){detail}")


def load() -> ctypes.CDLL:
    """Load libsai.so once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with sparse_attention_indexer_top_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().sai_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != 0:
        raise SaiError(status, where)
