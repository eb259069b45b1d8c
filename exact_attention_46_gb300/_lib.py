"""ctypes loader for libattn46.so (the C ABI declared in include/attn46.h).

Loading fails loudly: there is no fallback implementation.  Build the library
with ``python -m exact_attention_46_gb300.build`` (``__graft_entry__.build()``).
"""

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn46.so")

# Functions exported by the library: name -> (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_LL = ctypes.c_longlong
_D = ctypes.c_double
_SZ = ctypes.c_size_t
SIGNATURES = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "attn_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_varlen_scale_blocks": (_I, [_I, _I]),
    "hadamard_rotate_quant_fp8_varlen": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "rope_hadamard_rotate_quant_fp8_varlen": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "attn_fwd_varlen_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_gqa_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "attn_decode": (_I, [_P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_decode_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_bwd_workspace_bytes": (_SZ, [_I, _I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _F, _P]),
    "attn_bwd_gqa": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "hadamard_rotate_quant_fp8": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "hadamard_rotate_quant_fp8_qkv": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "rope_cos_sin_table": (_I, [_P, _I, _I, _D, _P]),
    "rope_hadamard_rotate_quant_fp8": (_I, [_P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P]),
    "attn_get_last_error": (ctypes.c_char_p, []),
    "attn_check": (_I, [_P]),
    "attn_set_spin_limit": (None, [_LL]),
    "attn_set_key_split": (None, [_I]),
    "attn_key_split_plan": (_I, [_LL, _I, _I, _I, _P]),
    "attn_fwd_split": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "attn_fwd_split_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "attn_selftest_bounded_wait": (_I, [_LL, _P]),
    "attn_version": (_I, []),
}

STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
          4: "ATTN_ERR_TIMEOUT"}

_lib = None


def load():
    """The loaded library (cached).  Raises ImportError if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                "libattn46.so is not built (%s); run `python -m exact_attention_46_gb300.build`" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class AttnError(RuntimeError):
    """A non-OK status from the library; ``status`` holds the attn_status code."""

    def __init__(self, status, message):
        super().__init__("%s: %s" % (STATUS.get(status, status), message))
        self.status = status


def call(name, *args):
    """Call an entry point that returns an attn_status; raise AttnError unless ATTN_OK."""
    lib = load()
    rc = getattr(lib, name)(*args)
    if rc != 0:
        raise AttnError(rc, lib.attn_get_last_error().decode(errors="replace"))
    return rc
