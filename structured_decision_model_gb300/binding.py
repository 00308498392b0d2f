"""ctypes binding of libclef_head.so: the C ABI's entry points under the same names.

Argument marshalling only: every step of the head runs in the library's CUDA
kernels.  If the library is missing this module raises; there is no fallback.
"""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libclef_head.so")

CLEF_OK = 0
STATUS = {
    0: "CLEF_OK", 1: "CLEF_ERR_INVALID_ARGUMENT", 2: "CLEF_ERR_WORKSPACE_TOO_SMALL",
    3: "CLEF_ERR_UNSUPPORTED_CONFIG", 4: "CLEF_ERR_CUDA", 5: "CLEF_ERR_DEVICE_BOUNDS",
    6: "CLEF_ERR_DEVICE_TIMEOUT",
}
EXPORTED = [
    "clef_weight_count", "clef_prepared_size", "clef_prepare_weights", "clef_workspace_size",
    "clef_head_forward", "clef_device_status", "clef_span_sums", "clef_gemm_bf16",
    "clef_kernel_launches", "clef_status_string", "clef_span_sums_noalloc", "clef_stream_begin",
    "clef_stream_rows", "clef_stream_finish", "clef_selftest_wait_timeout", "clef_stream_rows_f16",
    "clef_stream_finish_f16",
]

_i32, _i64, _vp, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t


class ClefError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class ClefConfig(ctypes.Structure):
    _fields_ = [("hidden", _i32), ("width", _i32), ("heads", _i32), ("ffn", _i32),
                ("n_route", _i32), ("n_joint", _i32), ("vocab", _i32)]


class ClefSchema(ctypes.Structure):
    _fields_ = [("B", _i32), ("Lpad", _i32), ("row_stride", _i64), ("lengths", _vp), ("Q", _i32),
                ("q_rec", _vp), ("q_type", _vp), ("q_span", _vp), ("q_opt_off", _vp), ("O", _i32),
                ("o_span", _vp)]


class ClefDebugOutputs(ctypes.Structure):
    _fields_ = [("pooled_u", _vp), ("pooled_c", _vp), ("pooled_x", _vp), ("global_g", _vp),
                ("option_final", _vp), ("field_final", _vp), ("events", _vp * 8), ("timeline", _vp),
                ("timeline_len", _i32), ("timeline_count", _vp), ("tail_mode", _i32), ("row_mu", _vp),
                ("row_rstd", _vp)]


_lib = None


def load():
    """Load libclef_head.so (built in-tree by ``build.build_library``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise FileNotFoundError(f"{LIB_PATH} is missing: build it with structured_decision_model_gb300.build")
    lib = ctypes.CDLL(LIB_PATH)
    lib.clef_weight_count.argtypes = [ctypes.POINTER(ClefConfig)]
    lib.clef_weight_count.restype = ctypes.c_int
    lib.clef_prepared_size.argtypes = [ctypes.POINTER(ClefConfig), ctypes.POINTER(_sz)]
    lib.clef_prepare_weights.argtypes = [ctypes.POINTER(ClefConfig), ctypes.POINTER(_vp), _vp, _sz, _vp]
    lib.clef_workspace_size.argtypes = [ctypes.POINTER(ClefConfig), ctypes.POINTER(ClefSchema), ctypes.POINTER(_sz)]
    lib.clef_head_forward.argtypes = [ctypes.POINTER(ClefConfig), ctypes.POINTER(_vp), _vp, ctypes.POINTER(ClefSchema),
                                      _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                      ctypes.POINTER(ClefDebugOutputs), _vp]
    lib.clef_device_status.argtypes = [_vp, _vp]
    lib.clef_selftest_wait_timeout.argtypes = [_vp, _i64, _vp]
    lib.clef_stream_begin.argtypes = [ctypes.POINTER(ClefConfig), ctypes.POINTER(ClefSchema), _vp, _sz, _vp]
    lib.clef_stream_rows.argtypes = [ctypes.POINTER(ClefConfig), _vp, ctypes.POINTER(ClefSchema), _vp, _i32, _i32,
                                     _i32, _vp, _sz, _vp]
    lib.clef_stream_finish.argtypes = lib.clef_head_forward.argtypes
    lib.clef_stream_rows_f16.argtypes = lib.clef_stream_rows.argtypes
    lib.clef_stream_finish_f16.argtypes = lib.clef_head_forward.argtypes
    lib.clef_span_sums.argtypes = [ctypes.POINTER(ClefConfig), ctypes.POINTER(ClefSchema), _vp, _vp, _vp, _vp, _vp,
                                   _vp, _vp, _sz, _vp]
    lib.clef_gemm_bf16.argtypes = [_vp, _i64, _vp, _i64, _vp, _vp, _i64, _i32, _i32, _i32, _vp, _vp]
    lib.clef_span_sums_noalloc.argtypes = [ctypes.POINTER(ClefConfig), ctypes.POINTER(ClefSchema), _vp, _vp, _vp,
                                           _vp, _vp, _vp, _vp]
    lib.clef_kernel_launches.argtypes = []
    lib.clef_kernel_launches.restype = ctypes.c_uint64
    lib.clef_status_string.argtypes = [ctypes.c_int]
    lib.clef_status_string.restype = ctypes.c_char_p
    for name in EXPORTED:
        if name not in ("clef_weight_count", "clef_status_string", "clef_kernel_launches"):
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status, where):
    if status != CLEF_OK:
        raise ClefError(status, where)


def make_config(H=4096, D=1024, heads=16, F=4096, n_route=2, n_joint=4, vocab=248320):
    return ClefConfig(H, D, heads, F, n_route, n_joint, vocab)


class Schema:
    """Host schema tables kept alive together with the C struct that points at them."""

    def __init__(self, B, Lpad, row_stride, lengths, q_rec, q_type, q_span, q_opt_off, o_span):
        c = lambda a: np.ascontiguousarray(a, dtype=np.int32)
        self.lengths, self.q_rec, self.q_type = c(lengths), c(q_rec), c(q_type)
        self.q_span, self.q_opt_off, self.o_span = c(q_span), c(q_opt_off), c(o_span)
        self.B, self.Lpad = int(B), int(Lpad)
        self.Q, self.O = int(self.q_type.shape[0]), int(self.o_span.reshape(-1, 2).shape[0])
        self.struct = ClefSchema(self.B, self.Lpad, int(row_stride), self.lengths.ctypes.data, self.Q,
                                 self.q_rec.ctypes.data, self.q_type.ctypes.data, self.q_span.ctypes.data,
                                 self.q_opt_off.ctypes.data, self.O, self.o_span.ctypes.data)


def clef_status_string(status):
    return load().clef_status_string(int(status)).decode()


def clef_weight_count(cfg):
    n = load().clef_weight_count(ctypes.byref(cfg))
    if n < 0:
        raise ClefError(3, "clef_weight_count")
    return n


def clef_prepared_size(cfg):
    out = _sz(0)
    _check(load().clef_prepared_size(ctypes.byref(cfg), ctypes.byref(out)), "clef_prepared_size")
    return out.value


def clef_prepare_weights(cfg, weight_ptrs, prepared_ptr, prepared_bytes, stream=0):
    arr = (_vp * len(weight_ptrs))(*weight_ptrs)
    _check(load().clef_prepare_weights(ctypes.byref(cfg), arr, prepared_ptr, prepared_bytes, stream),
           "clef_prepare_weights")


def clef_workspace_size(cfg, schema: Schema):
    out = _sz(0)
    _check(load().clef_workspace_size(ctypes.byref(cfg), ctypes.byref(schema.struct), ctypes.byref(out)),
           "clef_workspace_size")
    return out.value


def clef_head_forward(cfg, weight_ptrs, prepared_ptr, schema: Schema, hidden_ptr, token_ids_ptr, lexical_ptr,
                      logits_ptr, probs_ptr, q_value_ptr, q_conf_ptr, q_argmax_ptr, workspace_ptr, workspace_bytes,
                      debug=None, stream=0, check=True):
    arr = (_vp * len(weight_ptrs))(*weight_ptrs)
    dbg = ctypes.byref(debug) if debug is not None else None
    st = load().clef_head_forward(ctypes.byref(cfg), arr, prepared_ptr, ctypes.byref(schema.struct), hidden_ptr,
                                  token_ids_ptr, lexical_ptr, logits_ptr, probs_ptr, q_value_ptr, q_conf_ptr,
                                  q_argmax_ptr, workspace_ptr, workspace_bytes, dbg, stream)
    if check:
        _check(st, "clef_head_forward")
    return st


def clef_stream_begin(cfg, schema: Schema, workspace_ptr, workspace_bytes, stream=0):
    _check(load().clef_stream_begin(ctypes.byref(cfg), ctypes.byref(schema.struct), workspace_ptr, workspace_bytes,
                                    stream), "clef_stream_begin")


def clef_stream_rows(cfg, prepared_ptr, schema: Schema, hidden_ptr, record, row0, n_rows, workspace_ptr,
                     workspace_bytes, stream=0, check=True):
    st = load().clef_stream_rows(ctypes.byref(cfg), prepared_ptr, ctypes.byref(schema.struct), hidden_ptr, record, row0,
                                 n_rows, workspace_ptr, workspace_bytes, stream)
    if check:
        _check(st, "clef_stream_rows")
    return st


def clef_stream_finish(cfg, weight_ptrs, prepared_ptr, schema: Schema, hidden_ptr, token_ids_ptr, lexical_ptr,
                       logits_ptr, probs_ptr, q_value_ptr, q_conf_ptr, q_argmax_ptr, workspace_ptr, workspace_bytes,
                       debug=None, stream=0):
    arr = (_vp * len(weight_ptrs))(*weight_ptrs)
    dbg = ctypes.byref(debug) if debug is not None else None
    _check(load().clef_stream_finish(ctypes.byref(cfg), arr, prepared_ptr, ctypes.byref(schema.struct), hidden_ptr,
                                     token_ids_ptr, lexical_ptr, logits_ptr, probs_ptr, q_value_ptr, q_conf_ptr,
                                     q_argmax_ptr, workspace_ptr, workspace_bytes, dbg, stream), "clef_stream_finish")


def clef_stream_rows_f16(cfg, prepared_ptr, schema: Schema, hidden_ptr, record, row0, n_rows, workspace_ptr,
                         workspace_bytes, stream=0, check=True):
    st = load().clef_stream_rows_f16(ctypes.byref(cfg), prepared_ptr, ctypes.byref(schema.struct), hidden_ptr, record,
                                     row0, n_rows, workspace_ptr, workspace_bytes, stream)
    if check:
        _check(st, "clef_stream_rows_f16")
    return st


def clef_stream_finish_f16(cfg, weight_ptrs, prepared_ptr, schema: Schema, hidden_ptr, token_ids_ptr, lexical_ptr,
                           logits_ptr, probs_ptr, q_value_ptr, q_conf_ptr, q_argmax_ptr, workspace_ptr,
                           workspace_bytes, debug=None, stream=0):
    arr = (_vp * len(weight_ptrs))(*weight_ptrs)
    dbg = ctypes.byref(debug) if debug is not None else None
    _check(load().clef_stream_finish_f16(ctypes.byref(cfg), arr, prepared_ptr, ctypes.byref(schema.struct),
                                         hidden_ptr, token_ids_ptr, lexical_ptr, logits_ptr, probs_ptr, q_value_ptr,
                                         q_conf_ptr, q_argmax_ptr, workspace_ptr, workspace_bytes, dbg, stream),
           "clef_stream_finish_f16")


def clef_kernel_launches():
    return int(load().clef_kernel_launches())


def clef_device_status(workspace_ptr, stream=0):
    return load().clef_device_status(workspace_ptr, stream)


def clef_selftest_wait_timeout(workspace_ptr, limit_ns, stream=0, check=True):
    st = load().clef_selftest_wait_timeout(workspace_ptr, int(limit_ns), stream)
    if check:
        _check(st, "clef_selftest_wait_timeout")
    return st


def clef_span_sums(cfg, schema: Schema, hidden_ptr, token_ids_ptr, lexical_ptr, q_sum_ptr, o_sum_ptr, x_sum_ptr,
                   workspace_ptr, workspace_bytes, stream=0):
    _check(load().clef_span_sums(ctypes.byref(cfg), ctypes.byref(schema.struct), hidden_ptr, token_ids_ptr,
                                 lexical_ptr, q_sum_ptr, o_sum_ptr, x_sum_ptr, workspace_ptr, workspace_bytes,
                                 stream), "clef_span_sums")


def clef_span_sums_noalloc(cfg, schema: Schema, hidden_ptr, token_ids_ptr, lexical_ptr, q_sum_ptr, o_sum_ptr,
                           x_sum_ptr, stream=0):
    """Status of the allocation-free span sums (the call waits for ``stream``)."""
    return load().clef_span_sums_noalloc(ctypes.byref(cfg), ctypes.byref(schema.struct), hidden_ptr,
                                         token_ids_ptr, lexical_ptr, q_sum_ptr, o_sum_ptr, x_sum_ptr, stream)


def clef_gemm_bf16(A_ptr, lda, B_ptr, ldb, bias_ptr, C_ptr, ldc, M, N, K, flags_ptr, stream=0):
    _check(load().clef_gemm_bf16(A_ptr, lda, B_ptr, ldb, bias_ptr, C_ptr, ldc, M, N, K, flags_ptr, stream),
           "clef_gemm_bf16")
