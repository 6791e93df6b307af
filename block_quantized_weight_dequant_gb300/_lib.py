"""ctypes declarations for libbqgemv.so (include/bqgemv.h).

The library is loaded on first use; that use raises ImportError if the
library has not been built.  There is no CPU or PyTorch fallback for any
operation in this package.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbqgemv.so")

BQ_OK, BQ_ERR_NULL, BQ_ERR_SHAPE, BQ_ERR_ALIGN, BQ_ERR_QTYPE, BQ_ERR_CUDA, BQ_ERR_DEVICE = range(7)
BQ_Q4_0, BQ_Q8_0, BQ_Q4_K = 2, 8, 12
BQ_VERIFY_MAX_ROWS = 6

BQ_OP_GEMV, BQ_OP_GATE_UP_SILU = 0, 1

# every extern "C" symbol of include/bqgemv.h
EXPORTS = ("bq_version", "bq_status_str", "bq_packed_bytes", "bq_quantize_pack", "bq_gemv_q8_0",
           "bq_gemv_q4_0", "bq_gemv_q4_k", "bq_gemv_gate_up_silu", "bq_gemv_verify", "bq_gemv_qkv_bias",
           "bq_gemv_f16", "bq_gemv_f16_f16out", "bq_device_status",
           "bq_tree_lanes", "bq_stream_workspace_bytes", "bq_stream_plan_create",
           "bq_stream_plan_launch", "bq_stream_plan_tune", "bq_stream_plan_launches",
           "bq_stream_plan_destroy", "bq_stream_run_noalloc")
BQ_NOALLOC_MAX_OPS = 512


class BqOp(ctypes.Structure):
    """struct bq_op of include/bqgemv.h"""
    _fields_ = [("kind", ctypes.c_int32), ("stage", ctypes.c_int32), ("M", ctypes.c_int64),
                ("K", ctypes.c_int64), ("W", ctypes.c_void_p), ("W_up", ctypes.c_void_p),
                ("x", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("eps", ctypes.c_float),
                ("y", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


class BQError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: bq status {status} ({status_str(status)})")


def _declare(lib):
    i64, i32, vp, fp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
    sig = {
        "bq_version": (i32, []),
        "bq_status_str": (ctypes.c_char_p, [i32]),
        "bq_packed_bytes": (i64, [i32, i64, i64]),
        "bq_quantize_pack": (i32, [i32, vp, i64, i64, vp, vp]),
        "bq_gemv_q8_0": (i32, [vp, vp, vp, i64, i64, vp]),
        "bq_gemv_q4_0": (i32, [vp, vp, vp, i64, i64, vp]),
        "bq_gemv_q4_k": (i32, [vp, vp, vp, i64, i64, vp]),
        "bq_gemv_gate_up_silu": (i32, [i32, vp, vp, vp, vp, fp, vp, i64, i64, vp]),
        "bq_gemv_verify": (i32, [i32, vp, vp, vp, i32, i64, i64, vp]),
        "bq_gemv_qkv_bias": (i32, [i32, vp, vp, vp, vp, i64, i64, vp]),
        "bq_gemv_f16": (i32, [vp, vp, vp, i64, i64, vp]),
        "bq_gemv_f16_f16out": (i32, [vp, vp, vp, i64, i64, vp]),
        "bq_device_status": (i32, [ctypes.POINTER(ctypes.c_uint), i32]),
        "bq_tree_lanes": (i32, [i64]),
        "bq_stream_workspace_bytes": (i64, [i32, i32]),
        "bq_stream_plan_create": (i32, [i32, ctypes.POINTER(BqOp), i32, vp, i64,
                                        ctypes.POINTER(vp)]),
        "bq_stream_plan_launch": (i32, [vp, vp]),
        "bq_stream_plan_tune": (i32, [vp, i32, vp]),
        "bq_stream_plan_launches": (i32, [vp]),
        "bq_stream_plan_destroy": (i32, [vp]),
        "bq_stream_run_noalloc": (i32, [i32, ctypes.POINTER(BqOp), i32, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path=LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m block_quantized_weight_dequant_gb300.build`"
            " (or __graft_entry__.build()); this package has no fallback without it")
    return _declare(ctypes.CDLL(path))


_LIB = None


def get():
    """The loaded library (loaded on first use; ImportError if not built)."""
    global _LIB
    if _LIB is None:
        _LIB = load()
    return _LIB


class _LazyLib:
    def __getattr__(self, name):
        return getattr(get(), name)


lib = _LazyLib()


def status_str(status):
    return get().bq_status_str(int(status)).decode()


def check(status, what):
    if status != BQ_OK:
        raise BQError(status, what)
