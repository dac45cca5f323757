"""ctypes declarations of libcg.so (include/cg.h).  Loading fails loudly when the
library has not been built; there is no other implementation to fall back on."""

from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libcg.so")

CG_OK = 0
CG_E_ARG, CG_E_SYNTAX, CG_E_UNSUPPORTED, CG_E_EMPTY, CG_E_UNDEFINED_RULE = -1, -2, -3, -4, -5
CG_E_LIMIT, CG_E_CUDA, CG_E_DEVICE, CG_E_NOMEM = -6, -7, -8, -9
CG_GBNF, CG_JSON_SCHEMA, CG_STRUCTURAL_TAG = 0, 1, 2
CG_F32, CG_BF16 = 0, 1
CG_DEAD = CG_NO_TOKEN = 0xFFFFFFFF
CG_FLAG_DONE, CG_FLAG_FORCED_NEXT, CG_FLAG_REJECTED, CG_FLAG_NO_TOKEN, CG_FLAG_CAPPED = 1, 2, 4, 8, 16
CG_FLAG_DRAFT_CUT = 32
CG_STATE_ACCEPT, CG_STATE_SINK, CG_STATE_FORCED_ONLY = 1, 2, 4
CG_SAMPLE_INPLACE = 1
CG_NOALLOC_MAX_ROWS = 64
CG_RESULT_CALC_TAG, CG_RESULT_JSON_ANSWER, CG_RESULT_STROP_TAG = 0, 1, 2
CG_PDA_MAX_DEPTH = 64

ERROR_NAMES = {CG_E_ARG: "CG_E_ARG", CG_E_SYNTAX: "CG_E_SYNTAX", CG_E_UNSUPPORTED: "CG_E_UNSUPPORTED",
               CG_E_EMPTY: "CG_E_EMPTY", CG_E_UNDEFINED_RULE: "CG_E_UNDEFINED_RULE", CG_E_LIMIT: "CG_E_LIMIT",
               CG_E_CUDA: "CG_E_CUDA", CG_E_DEVICE: "CG_E_DEVICE", CG_E_NOMEM: "CG_E_NOMEM"}


class cg_bounds(C.Structure):
    _fields_ = [("ws_max", C.c_uint32), ("max_len_default", C.c_uint32), ("depth_max", C.c_uint32),
                ("max_items_default", C.c_uint32), ("max_tokens", C.c_uint32)]


class cg_span_rule(C.Structure):
    _fields_ = [("span_open", C.c_void_p), ("span_open_len", C.c_size_t),
                ("span_close", C.c_void_p), ("span_close_len", C.c_size_t),
                ("result_format", C.c_int)]


# name -> (restype, argtypes); every symbol include/cg.h declares
SIGNATURES = {
    "cg_compile": (C.c_int, [C.c_char_p, C.c_size_t, C.c_int, C.POINTER(cg_bounds), C.POINTER(C.c_void_p),
                             C.c_char_p, C.c_size_t]),
    "cg_grammar_destroy": (None, [C.c_void_p]),
    "cg_grammar_info": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint32), C.POINTER(C.c_uint32), C.POINTER(C.c_uint32)]),
    "cg_grammar_export": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p]),
    "cg_try_input": (C.c_int, [C.c_void_p, C.c_char_p, C.c_size_t, C.c_void_p, C.POINTER(C.c_size_t),
                               C.POINTER(C.c_uint32), C.POINTER(C.c_int)]),
    "cg_live_states": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint32, C.POINTER(C.c_uint32)]),
    "cg_vocab_create": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint32, C.POINTER(C.c_void_p)]),
    "cg_vocab_destroy": (None, [C.c_void_p]),
    "cg_tokenize_greedy": (C.c_int, [C.c_void_p, C.c_char_p, C.c_size_t, C.c_void_p, C.c_size_t,
                                     C.POINTER(C.c_size_t)]),
    "cg_ctx_create": (C.c_int, [C.c_void_p, C.c_uint32, C.c_void_p, C.c_void_p, C.POINTER(C.c_void_p)]),
    "cg_ctx_destroy": (None, [C.c_void_p]),
    "cg_ctx_info": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint32), C.POINTER(C.c_uint64), C.POINTER(C.c_uint32),
                              C.POINTER(C.c_uint32)]),
    "cg_ctx_status": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint32)]),
    "cg_ctx_prefill": (C.c_int, [C.c_void_p]),
    "cg_ctx_cache_stats": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint64), C.POINTER(C.c_uint64),
                                     C.POINTER(C.c_uint32)]),
    "cg_fill_bitmask": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_uint32, C.c_void_p]),
    "cg_mask_and_sample": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_uint32, C.c_uint32, C.c_void_p,
                                     C.c_float, C.c_float, C.c_uint64, C.c_uint32, C.c_void_p, C.c_void_p,
                                     C.c_uint32]),
    "cg_mask_and_sample_noalloc": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_uint32, C.c_uint32, C.c_void_p,
                                             C.c_float, C.c_float, C.c_uint64, C.c_uint32, C.c_void_p, C.c_void_p,
                                             C.c_uint32]),
    "cg_mask_classes": (C.c_int, [C.c_void_p, C.c_uint32, C.c_uint32, C.c_void_p, C.c_uint32,
                                  C.POINTER(C.c_uint32), C.POINTER(C.c_uint32)]),
    "cg_self_test_wait_timeout": (C.c_int, [C.c_void_p]),
    "cg_accept_many": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_uint32,
                                 C.c_uint32, C.c_void_p, C.c_uint32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "cg_step_host": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_uint32, C.c_void_p, C.c_int,
                               C.c_uint32, C.c_float, C.c_float, C.c_uint64, C.c_uint32, C.c_void_p, C.c_uint32,
                               C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "cg_ctx_sync": (C.c_int, [C.c_void_p]),
    "cg_step": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_uint32, C.c_void_p, C.c_int, C.c_uint32,
                          C.c_float, C.c_float, C.c_uint64, C.c_uint32, C.c_void_p, C.c_uint32, C.c_void_p, C.c_void_p,
                          C.c_void_p, C.c_void_p]),
    "cg_accept": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_uint32, C.c_void_p,
                            C.c_uint32, C.c_void_p, C.c_void_p]),
    "cg_eval_strop": (C.c_int, [C.c_char_p, C.c_size_t, C.c_void_p, C.c_size_t, C.POINTER(C.c_size_t),
                                C.POINTER(C.c_int)]),
    "cg_eval_arith": (C.c_int, [C.c_char_p, C.c_size_t, C.c_int, C.c_void_p, C.c_size_t, C.POINTER(C.c_size_t),
                                C.POINTER(C.c_int)]),
    "cg_pda_compile": (C.c_int, [C.c_char_p, C.c_size_t, C.c_uint32, C.POINTER(C.c_void_p)]),
    "cg_pda_grammar_destroy": (None, [C.c_void_p]),
    "cg_pda_grammar_info": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint32), C.POINTER(C.c_uint32),
                                      C.POINTER(C.c_uint32), C.POINTER(C.c_uint32)]),
    "cg_pda_try_input": (C.c_int, [C.c_void_p, C.c_char_p, C.c_size_t, C.c_void_p, C.POINTER(C.c_size_t),
                                   C.POINTER(C.c_int), C.POINTER(C.c_uint32)]),
    "cg_pda_create": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(C.c_void_p)]),
    "cg_pda_destroy": (None, [C.c_void_p]),
    "cg_pda_info": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint32), C.POINTER(C.c_uint32), C.POINTER(C.c_uint64),
                              C.POINTER(C.c_uint32)]),
    "cg_pda_fill_bitmask": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint32, C.c_void_p, C.c_void_p]),
    "cg_pda_accept": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint32, C.c_void_p, C.c_void_p, C.c_void_p,
                                C.c_uint32, C.c_void_p]),
    "cg_pda_accept_many": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint32, C.c_void_p, C.c_void_p, C.c_void_p,
                                     C.c_uint32, C.c_void_p, C.c_uint32, C.c_void_p, C.c_void_p]),
    "cg_pda_step": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint32, C.c_void_p, C.c_int, C.c_uint32, C.c_float,
                              C.c_float, C.c_uint64, C.c_uint32, C.c_void_p, C.c_void_p, C.c_uint32, C.c_void_p,
                              C.c_void_p, C.c_void_p]),
    "cg_pda_accept_fill": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint32, C.c_void_p, C.c_void_p, C.c_void_p,
                                     C.c_uint32, C.c_void_p, C.c_void_p, C.c_void_p]),
    "cg_driver_create": (C.c_int, [C.c_void_p, C.c_uint32, C.c_void_p, C.POINTER(cg_span_rule), C.c_uint32,
                                   C.POINTER(C.c_void_p)]),
    "cg_driver_destroy": (None, [C.c_void_p]),
    "cg_driver_update": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                   C.POINTER(C.c_uint32)]),
}

_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libcg.so is not built ({LIB_PATH}); run "
                               "`python -m grammar_constrained_decoding_gb300.build`")
        handle = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class CgError(RuntimeError):
    def __init__(self, call: str, code: int, msg: str = ""):
        super().__init__(f"{call} failed: {ERROR_NAMES.get(code, code)}" + (f" ({msg})" if msg else ""))
        self.code = code


def check(call: str, rc: int, msg: str = "") -> None:
    if rc != CG_OK:
        raise CgError(call, rc, msg)
