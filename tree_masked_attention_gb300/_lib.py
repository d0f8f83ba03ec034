"""ctypes loader of the in-tree C-ABI library ``libtreeattn.so`` (include/tree_attn.h).

There is no fallback: if the library is missing or fails to load, every call
raises. Build it with ``python -c "import __graft_entry__ as g; g.build()"`` or
``python tree_masked_attention_gb300/build.py``.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtreeattn.so")

STATUS = {
    0: "TREE_OK", 1: "TREE_ERR_INVALID_ARG", 2: "TREE_ERR_SHAPE", 3: "TREE_ERR_DTYPE",
    4: "TREE_ERR_ALIGNMENT", 5: "TREE_ERR_CUDA", 6: "TREE_ERR_TIMEOUT",
    7: "TREE_ERR_DEVICE_CHECK", 8: "TREE_ERR_WORKSPACE",
}

# Every exported symbol the header declares, with (restype, argtypes).
_i32p = C.POINTER(C.c_int32)
_i64p = C.POINTER(C.c_int64)
_f32p = C.POINTER(C.c_float)
_vp = C.c_void_p
_i64 = C.c_int64
_int = C.c_int
_f = C.c_float
_sz = C.c_size_t


class PackSizes(C.Structure):
    _fields_ = [("T", C.c_int64), ("n_nodes", C.c_int64), ("n_occ", C.c_int64),
                ("n_roots", C.c_int64), ("n_tokens", C.c_int64)]


class PackOut(C.Structure):
    _fields_ = [(n, _i32p) for n in ("packed_ids", "position_ids", "subtree_end", "path_count",
                                     "parent_row", "node_of_token", "node_start", "node_end",
                                     "node_parent", "token_rows", "occ_source_rows", "occ_targets",
                                     "occ_seq")] + \
               [("occ_weights", _f32p), ("occ_row_ptr", _i32p), ("occ_perm", _i32p)]


SIGNATURES = {
    "tree_pack_plan": (_int, [_i32p, _i64p, _i64, C.POINTER(_vp), C.POINTER(PackSizes)]),
    "tree_pack_emit": (_int, [_vp, _f32p, C.POINTER(PackOut)]),
    "tree_plan_free": (None, [_vp]),
    "tree_validate_subtree_end": (_int, [_i32p, _i64]),
    "tree_rope": (_int, [_vp, _vp, _vp, _i64, _int, _int, _int, _f, _int, _int, _vp]),
    "tree_attn_workspace_size": (_sz, [_i64, _int, _int, _int, _int]),
    "tree_attn_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _int, _int, _f,
                             _vp, _sz, _vp]),
    "tree_attn_fwd_noalloc": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _int, _int, _f, _vp]),
    "tree_attn_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int,
                             _int, _int, _f, _int, _vp, _sz, _vp]),
    "tree_kernel_timing": (_int, [_int]),
    "tree_policy_loss": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _f, _f, _vp, _vp, _vp, _vp]),
    "tree_selftest_exp2": (_int, [_vp, _vp, _i64, _vp]),
    "tree_attn_gateway_workspace_size": (_sz, [_i64, _i64, _int, _int, _int, _int]),
    "tree_attn_fwd_gateway": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _int, _f,
                                     _vp, _sz, _vp]),
    "tree_attn_bwd_gateway": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                     _int, _int, _int, _int, _f, _vp, _sz, _vp]),
    "tree_gdn_workspace_size": (_sz, [_i64, _i64, _int, _int, _int]),
    "tree_gdn_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _int, _vp,
                            _sz, _vp]),
    "tree_gdn_bwd_workspace_size": (_sz, [_i64, _i64, _int, _int, _int]),
    "tree_gdn_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                            _int, _int, _int, _int, _vp, _sz, _vp]),
    "tree_gdn_bwd_saved": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                  _i64, _int, _int, _int, _int, _vp, _sz, _vp]),
    "tree_gdn_test_withhold": (_int, [_i64, C.c_double]),
    "tree_conv1d_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _int, _vp]),
    "tree_conv1d_workspace_size": (_sz, [_i64, _int, _int]),
    "tree_conv1d_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _int, _vp, _sz,
                               _vp]),
    "tree_kernel_last_ms": (C.c_float, [_int]),
    "tree_attn_bwd_rope": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _int,
                                  _int, _int, _int, _f, _f, _int, _vp, _sz, _vp]),
    "tree_logprob_workspace_size": (_sz, [_i64, _i64, _i64, _i64, _int]),
    "tree_logprob_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _int,
                                _vp, _sz, _vp]),
    "tree_logprob_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp,
                                _vp, _int, _int, _vp, _sz, _vp]),
    "tree_check_device_status": (_int, [_vp]),
    "tree_last_error": (C.c_char_p, []),
    "tree_kernel_path": (_int, [_int, _int, _int]),
    "tree_launch_count": (C.c_uint64, []),
    "tree_version": (C.c_char_p, []),
}

_lib = None


class TreeError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {message}")
        self.status = status


def lib():
    """The loaded library (loaded once); raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def check(status: int, where: str):
    if status != 0:
        msg = lib().tree_last_error()
        raise TreeError(status, where, msg.decode() if msg else "")
