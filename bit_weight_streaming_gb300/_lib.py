"""ctypes loader for libbws.so and the C signatures of include/bws.h."""
import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbws.so")

_lib = None

P = C.c_void_p
I = C.c_int
Z = C.c_size_t

SIGNATURES = {
    "bws_version": (I, []),
    "bws_last_error": (C.c_char_p, []),
    "bws_nvfp4_quantize_workspace_size": (Z, [I, I]),
    "bws_nvfp4_quantize": (I, [P, I, I, P, P, P, P, Z, P]),
    "bws_mxfp4_quantize": (I, [P, I, I, P, P, P]),
    "bws_fp8_rowwise_quantize": (I, [P, I, I, P, P, P]),
    "bws_gemv_workspace_size": (Z, [I, I, I]),
    "bws_nvfp4_gemv": (I, [P, P, P, P, I, I, I, P, P, Z, P]),
    "bws_nvfp4_prepare": (I, [P, I, I, I, P, Z, P]),
    "bws_nvfp4_gemv_prepared": (I, [P, P, P, I, I, I, P, P, Z, P]),
    "bws_nvfp4_gemv_noalloc": (I, [P, P, P, P, I, I, I, P, P]),
    "bws_nvfp4_gate_up_silu": (I, [P, P, P, P, P, P, P, I, I, I, P, P, Z, P]),
    "bws_fp8_lmhead_gemv": (I, [P, P, P, I, I, I, P, P, Z, P]),
    "bws_fp8_lmhead_argmax": (I, [P, P, P, I, I, I, P, P, P, P, Z, P]),
    "bws_mxfp4_moe_workspace_size": (Z, [P, I, I]),
    "bws_moe_router_workspace_size": (Z, [I, I]),
    "bws_mxfp8_quantize": (I, [P, I, I, P, P, P]),
    "bws_w4a8_workspace_size": (Z, [I, I, I]),
    "bws_mxfp4_w4a8_gemv": (I, [P, P, P, I, I, I, P, P, Z, P]),
    "bws_moe_router_topk": (I, [P, P, I, I, I, I, P, P, P, P, Z, P]),
    "bws_mxfp4_moe_gemv": (I, [P, P, P, I, I, P, P, P, Z, P]),
    "bws_mxfp4_moe_inspect": (I, [P, P, I, I, P, P, P, P, P]),
    "bws_decode_step_workspace_size": (Z, [P]),
    "bws_decode_step_plan_create": (I, [P, I, P]),
    "bws_decode_step_plan_destroy": (None, [P]),
    "bws_decode_step_stream": (I, [P, P, P, P, Z, P]),
    "bws_decode_step_greedy": (I, [P, P, P, P, P, P, Z, P]),
    "bws_decode_step_kernel_count": (I, [P]),
    "bws_decode_step_tap_size": (Z, [P]),
    "bws_decode_step_tap": (I, [P, P, P, P, Z, P, Z, P]),
    "bws_status_word": (I, [P, P, P]),
    "bws_debug_wait_flag": (I, [P, C.c_uint32, P, Z, P]),
    "bws_hbm_read_probe": (I, [P, Z, P, P]),
    "bws_l2_flush": (I, [P, Z, P]),
}


class BwsError(RuntimeError):
    pass


def lib():
    """The loaded library. Raises if libbws.so has not been built: there is
    no fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise BwsError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name, None)
            if f is None:
                continue
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def check(rc, what):
    if rc != 0:
        msg = lib().bws_last_error().decode(errors="replace")
        raise BwsError(f"{what} failed with status {rc}: {msg}")
