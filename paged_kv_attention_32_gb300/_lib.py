"""ctypes declarations of the C ABI in ``include/pka.h``.

Loads the in-tree ``_lib/libpka.so``; there is no fallback: if the library is
missing or does not load, every call raises.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpka.so")

PKA_OK = 0
PKA_ERR_INVALID_ARG = -1
PKA_ERR_UNSUPPORTED = -2
PKA_ERR_WORKSPACE_TOO_SMALL = -3
PKA_ERR_CUDA = -4
PKA_ERR_DEVICE_BOUNDS = -5
PKA_ERR_DEVICE_TIMEOUT = -6

PKA_DTYPE_BF16, PKA_DTYPE_F16, PKA_DTYPE_F32 = 0, 1, 2
PKA_MASK_DENSE, PKA_MASK_CAUSAL, PKA_MASK_VARIABLE_WINDOW = 0, 1, 2
PKA_PLAN_HOST_ONLY = 1
PKA_KERNEL_CUDA_CORE, PKA_KERNEL_MMA = 0, 1

# every symbol include/pka.h declares
EXPORTED = (
    "pka_last_error", "pka_version",
    "paged_decode_plan", "paged_decode_plan_update", "paged_decode_plan_destroy",
    "paged_decode_plan_info",
    "paged_decode_plan_export", "paged_decode_run", "paged_decode_plan_check",
    "paged_decode_check_tables", "paged_decode_step_host",
    "paged_decode_run_noalloc",
    "attn_merge_lse",
    "batch_prefill_plan", "batch_prefill_plan_fixed", "batch_prefill_plan_destroy", "batch_prefill_plan_check",
    "batch_prefill_run",
    "paged_kv_gather", "pka_wait_timeout_probe",
)


class DecodeDesc(ctypes.Structure):
    _fields_ = [
        ("batch_size", ctypes.c_int32), ("num_qo_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
        ("num_pages", ctypes.c_int64), ("dtype", ctypes.c_int32), ("q_len", ctypes.c_int32),
        ("max_q_len", ctypes.c_int32), ("mask", ctypes.c_int32), ("window_left", ctypes.c_int32),
        ("scale", ctypes.c_float), ("bmm2_scale", ctypes.c_float),
        ("return_lse", ctypes.c_int32), ("freeze_seq_lens", ctypes.c_int32),
        ("num_sms", ctypes.c_int32), ("split_waves", ctypes.c_int32),
        ("min_chunk_tokens", ctypes.c_int32), ("mma_min_rows", ctypes.c_int32),
        ("flags", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("num_items", ctypes.c_int32), ("chunk_pages", ctypes.c_int32),
        ("num_split", ctypes.c_int32), ("partial_rows", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64), ("kernel", ctypes.c_int32),
        ("rows_per_cta", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("split_waves", ctypes.c_int32), ("min_chunk_tokens", ctypes.c_int32),
        ("total_q", ctypes.c_int32),
    ]


class DecodeHostIO(ctypes.Structure):
    _fields_ = [
        ("q_host", ctypes.c_void_p), ("block_tables_host", ctypes.c_void_p),
        ("seq_lens_kv_host", ctypes.c_void_p), ("qo_indptr_host", ctypes.c_void_p),
        ("out_host", ctypes.c_void_p), ("lse_host", ctypes.c_void_p),
        ("q_dev", ctypes.c_void_p), ("block_tables_dev", ctypes.c_void_p),
        ("seq_lens_kv_dev", ctypes.c_void_p), ("out_dev", ctypes.c_void_p),
        ("lse_dev", ctypes.c_void_p), ("bt_row_stride", ctypes.c_int64),
    ]


class PrefillDesc(ctypes.Structure):
    _fields_ = [
        ("batch_size", ctypes.c_int32), ("num_qo_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("mask", ctypes.c_int32), ("window_left", ctypes.c_int32),
        ("sm_scale", ctypes.c_float), ("output_scale", ctypes.c_float),
        ("return_lse", ctypes.c_int32), ("num_sms", ctypes.c_int32), ("flags", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
    ]


_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_pi32 = ctypes.POINTER(ctypes.c_int32)

_SIGS = {
    "pka_last_error": (ctypes.c_char_p, []),
    "pka_version": (ctypes.c_char_p, []),
    "paged_decode_plan": (ctypes.c_int, [ctypes.POINTER(_vp), ctypes.POINTER(DecodeDesc), _pi32,
                                         _pi32, ctypes.POINTER(_sz), _vp]),
    "paged_decode_plan_update": (ctypes.c_int, [_vp, _i32, _pi32, _pi32, ctypes.POINTER(_sz),
                                                _vp]),
    "paged_decode_plan_destroy": (None, [_vp]),
    "paged_decode_plan_info": (ctypes.c_int, [_vp, ctypes.POINTER(PlanInfo)]),
    "paged_decode_plan_export": (ctypes.c_int, [_vp, _pi32, _pi32, _pi32, _pi32, _pi32, _pi32]),
    "paged_decode_run": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i64, _i64, _vp, _i64,
                                        _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "paged_decode_plan_check": (ctypes.c_int, [_vp, _vp]),
    "paged_decode_check_tables": (ctypes.c_int, [_vp, _vp, _i64, _vp, _vp]),
    "paged_decode_step_host": (ctypes.c_int, [_vp, _i32, ctypes.POINTER(DecodeHostIO), _vp, _vp,
                                              _i64, _i64, _vp, _vp, _sz, ctypes.POINTER(_sz),
                                              _i32, _vp]),
    "paged_decode_run_noalloc": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i64, _i64, _vp,
                                                _i64, _vp, _vp, _vp, _vp, _vp]),
    "attn_merge_lse": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32, _vp, _vp]),
    "batch_prefill_plan": (ctypes.c_int, [ctypes.POINTER(_vp), ctypes.POINTER(PrefillDesc),
                                          _pi32, _pi32, ctypes.POINTER(_sz), _pi32, _vp]),
    "batch_prefill_plan_fixed": (ctypes.c_int, [ctypes.POINTER(_vp), ctypes.POINTER(PrefillDesc),
                                                _i32, _i32, _pi32, _pi32, ctypes.POINTER(_sz),
                                                _pi32, _vp]),
    "batch_prefill_plan_destroy": (None, [_vp]),
    "batch_prefill_plan_check": (ctypes.c_int, [_vp, _vp]),
    "batch_prefill_run": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i64, _i64, _vp, _vp,
                                         _vp, _sz, _vp]),
    "paged_kv_gather": (ctypes.c_int, [_vp, _i64, _i64, _i64, _i32, _i32, _i32, _vp, _i64, _i32,
                                       _i32, _i32, _i32, _vp, _vp]),
    "pka_wait_timeout_probe": (ctypes.c_int, [_vp, _vp, _i64, _vp]),
}

_lib = None


def lib():
    """The loaded ``libpka.so`` with argtypes set.  Raises if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m paged_kv_attention_32_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class PkaError(RuntimeError):
    def __init__(self, code, where):
        msg = lib().pka_last_error().decode(errors="replace")
        super().__init__(f"{where} failed with status {code}: {msg}")
        self.code = code


def check(code, where):
    if code != PKA_OK:
        raise PkaError(code, where)
    return code
