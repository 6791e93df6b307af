"""The oracle: a plain CPU statement of block-quantized packing and the batch-1
dequant + GEMV, in C with fp64 accumulation (``bq_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference leg may import this package.  The
GPU library neither imports it nor shares code with it.

Every function takes and returns numpy arrays.  ``Oracle(lib_path)`` loads a
given build of the C source, which lets the tests run their pins against
deliberately broken copies of the source (mutants) as well as the real one.
"""
import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build


def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _row_ranges(M, parts):
    """[r0, r1) row ranges splitting M rows into at most `parts` near-equal pieces."""
    parts = max(1, min(parts, M))
    return [(M * i // parts, M * (i + 1) // parts) for i in range(parts)]

Q4_0 = 2
Q8_0 = 8
Q4_K = 12
# bytes per 32 weights (a Q4_K super-block is 144 bytes per 256 weights)
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18, Q4_K: 18}

_dp = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def _ptr(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct)) if a is not None else None


class Oracle:
    def __init__(self, lib_path=None):
        if lib_path is None:
            lib_path = _build.compile_oracle()
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.bqo_f32_to_f16_bits.restype = ctypes.c_uint16
        lib.bqo_f32_to_f16_bits.argtypes = [ctypes.c_float]
        lib.bqo_f16_bits_to_f64.restype = ctypes.c_double
        lib.bqo_f16_bits_to_f64.argtypes = [ctypes.c_uint16]
        lib.bqo_f32_to_f16_array.restype = None
        lib.bqo_f32_to_f16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i64]
        lib.bqo_packed_bytes.restype = i64
        lib.bqo_packed_bytes.argtypes = [i32, i64, i64]
        lib.bqo_quantize_pack.restype = i32
        lib.bqo_quantize_pack.argtypes = [i32, ctypes.c_void_p, i64, i64, ctypes.c_void_p]
        lib.bqo_dequant.restype = i32
        lib.bqo_dequant.argtypes = [i32, ctypes.c_void_p, i64, i64, ctypes.c_void_p]
        lib.bqo_gemv.restype = i32
        lib.bqo_gemv.argtypes = [i32, ctypes.c_void_p, i64, i64, ctypes.c_void_p,
                                 ctypes.c_void_p, ctypes.c_void_p]
        lib.bqo_q4_k_split_scale.restype = i32
        lib.bqo_q4_k_split_scale.argtypes = [ctypes.c_void_p, i64, i64, ctypes.c_void_p,
                                             ctypes.c_void_p]
        lib.bqo_gemv_bias.restype = i32
        lib.bqo_gemv_bias.argtypes = [i32, ctypes.c_void_p, i64, i64, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.bqo_gemv_f16.restype = i32
        lib.bqo_gemv_f16.argtypes = [ctypes.c_void_p, i64, i64, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p]
        lib.bqo_rmsnorm.restype = i32
        lib.bqo_rmsnorm.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i64, ctypes.c_double,
                                    ctypes.c_void_p]
        lib.bqo_silu.restype = ctypes.c_double
        lib.bqo_silu.argtypes = [ctypes.c_double]
        lib.bqo_gate_up_silu.restype = i32
        lib.bqo_gate_up_silu.argtypes = [i32, ctypes.c_void_p, ctypes.c_void_p, i64, i64,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        self.lib = lib

    # -- fp16 ---------------------------------------------------------------
    def f32_to_f16_bits(self, a):
        a = np.ascontiguousarray(a, dtype=np.float32)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.bqo_f32_to_f16_array(a.ctypes.data, out.ctypes.data, a.size)
        return out

    def f16_bits_to_f64(self, h):
        return self.lib.bqo_f16_bits_to_f64(int(h))

    # -- formats --------------------------------------------------------------
    def packed_bytes(self, qtype, M, K):
        return int(self.lib.bqo_packed_bytes(qtype, M, K))

    def quantize_pack(self, qtype, W):
        """fp32 [M, K] -> uint8 [M, (K/32)*block_bytes]."""
        W = np.ascontiguousarray(W, dtype=np.float32)
        M, K = W.shape
        out = np.empty((M, (K // 32) * BLOCK_BYTES[qtype]), dtype=np.uint8)
        rc = self.lib.bqo_quantize_pack(qtype, W.ctypes.data, M, K, out.ctypes.data)
        if rc:
            raise ValueError(f"oracle quantize_pack rejected qtype={qtype} shape={W.shape}")
        return out

    def dequant(self, qtype, Wq, M, K):
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        out = np.empty((M, K), dtype=np.float64)
        if self.lib.bqo_dequant(qtype, Wq.ctypes.data, M, K, out.ctypes.data):
            raise ValueError("oracle dequant: bad arguments")
        return out

    def gemv(self, qtype, Wq, M, K, x):
        """Returns (y, S): fp64 y = W x and S = sum_k |w_mk x_k|."""
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        x = np.ascontiguousarray(x, dtype=np.float64)
        assert x.shape == (K,)
        y = np.empty(M, dtype=np.float64)
        S = np.empty(M, dtype=np.float64)
        if self.lib.bqo_gemv(qtype, Wq.ctypes.data, M, K, x.ctypes.data, y.ctypes.data,
                             S.ctypes.data):
            raise ValueError("oracle gemv: bad arguments")
        return y, S

    def gemv_parallel(self, qtype, Wq, M, K, x, threads=None, with_S=True):
        """gemv() with the rows split among `threads` host threads (default:
        every host core).  Each thread runs the same scalar C routine on its own
        rows (the call releases the GIL), so every row's value is exactly the
        single-threaded one."""
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8).reshape(M, -1)
        x = np.ascontiguousarray(x, dtype=np.float64)
        assert x.shape == (K,)
        y = np.empty(M, dtype=np.float64)
        S = np.empty(M, dtype=np.float64) if with_S else None
        rb = Wq.shape[1] if M else 0

        def run(r):
            r0, r1 = r
            return self.lib.bqo_gemv(qtype, Wq.ctypes.data + r0 * rb, r1 - r0, K, x.ctypes.data,
                                     y.ctypes.data + 8 * r0,
                                     S.ctypes.data + 8 * r0 if with_S else None)

        with ThreadPoolExecutor(threads or host_cores()) as ex:
            if any(ex.map(run, _row_ranges(M, 4 * (threads or host_cores())))):
                raise ValueError("oracle gemv: bad arguments")
        return y, S

    def gemv_f16_parallel(self, W_bits, x, threads=None, with_S=True):
        """gemv_f16() with the rows split among host threads (same values)."""
        W_bits = np.ascontiguousarray(W_bits, dtype=np.uint16)
        M, K = W_bits.shape
        x = np.ascontiguousarray(x, dtype=np.float64)
        assert x.shape == (K,)
        y = np.empty(M, dtype=np.float64)
        S = np.empty(M, dtype=np.float64) if with_S else None

        def run(r):
            r0, r1 = r
            return self.lib.bqo_gemv_f16(W_bits.ctypes.data + 2 * r0 * K, r1 - r0, K,
                                         x.ctypes.data, y.ctypes.data + 8 * r0,
                                         S.ctypes.data + 8 * r0 if with_S else None)

        with ThreadPoolExecutor(threads or host_cores()) as ex:
            if any(ex.map(run, _row_ranges(M, 4 * (threads or host_cores())))):
                raise ValueError("oracle gemv_f16: bad arguments")
        return y, S

    def quantize_pack_parallel(self, qtype, W, threads=None):
        """quantize_pack() with the rows split among host threads; every block
        is packed by the same scalar routine, so the bytes are identical."""
        W = np.ascontiguousarray(W, dtype=np.float32)
        M, K = W.shape
        out = np.empty((M, (K // 32) * BLOCK_BYTES[qtype]), dtype=np.uint8)
        rb = out.shape[1]

        def run(r):
            r0, r1 = r
            return self.lib.bqo_quantize_pack(qtype, W.ctypes.data + 4 * r0 * K, r1 - r0, K,
                                              out.ctypes.data + r0 * rb)

        with ThreadPoolExecutor(threads or host_cores()) as ex:
            if any(ex.map(run, _row_ranges(M, 4 * (threads or host_cores())))):
                raise ValueError(f"oracle quantize_pack rejected qtype={qtype} shape={W.shape}")
        return out

    def q4_k_split_scale(self, Wq, M, K, x):
        """Q4_K rows: SK[m] = sum over sub-blocks of d*sc * sum|q x| +
        dmin*m * sum|x|, the scale of the GEMV bound for a product evaluated
        as d*sc * sum(q x) - dmin*m * sum(x) per sub-block (SK >= S)."""
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        x = np.ascontiguousarray(x, dtype=np.float64)
        assert x.shape == (K,)
        SK = np.empty(M, dtype=np.float64)
        if self.lib.bqo_q4_k_split_scale(Wq.ctypes.data, M, K, x.ctypes.data, SK.ctypes.data):
            raise ValueError("oracle q4_k_split_scale: bad arguments")
        return SK

    def q4_k_split_scale_parallel(self, Wq, M, K, x, threads=None):
        """q4_k_split_scale() with the rows split among host threads."""
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8).reshape(M, -1)
        x = np.ascontiguousarray(x, dtype=np.float64)
        SK = np.empty(M, dtype=np.float64)
        rb = Wq.shape[1] if M else 0

        def run(r):
            r0, r1 = r
            return self.lib.bqo_q4_k_split_scale(Wq.ctypes.data + r0 * rb, r1 - r0, K,
                                                 x.ctypes.data, SK.ctypes.data + 8 * r0)

        with ThreadPoolExecutor(threads or host_cores()) as ex:
            if any(ex.map(run, _row_ranges(M, 4 * (threads or host_cores())))):
                raise ValueError("oracle q4_k_split_scale: bad arguments")
        return SK

    def gemv_y_only(self, qtype, Wq, M, K, x, y):
        """The same product without S, into a caller-owned fp64 ``y``."""
        return self.lib.bqo_gemv(qtype, Wq.ctypes.data, M, K, x.ctypes.data, y.ctypes.data,
                                 None)

    def gemv_bias(self, qtype, Wq, M, K, x, bias):
        """Returns (y, S): fp64 y = W x + bias (the fused q|k|v + bias
        projection) and S = sum_k |w_mk x_k| + |bias_m|."""
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        x = np.ascontiguousarray(x, dtype=np.float64)
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
        assert x.shape == (K,) and (b is None or b.shape == (M,))
        y = np.empty(M, dtype=np.float64)
        S = np.empty(M, dtype=np.float64)
        if self.lib.bqo_gemv_bias(qtype, Wq.ctypes.data, M, K, x.ctypes.data,
                                  None if b is None else b.ctypes.data, y.ctypes.data,
                                  S.ctypes.data):
            raise ValueError("oracle gemv_bias: bad arguments")
        return y, S

    def gemv_f16(self, W_bits, x):
        """Unquantized fp16 weights (uint16 bits [M, K]): returns (y, S), fp64
        y = W x and S = sum_k |w_mk x_k|."""
        W_bits = np.ascontiguousarray(W_bits, dtype=np.uint16)
        M, K = W_bits.shape
        x = np.ascontiguousarray(x, dtype=np.float64)
        assert x.shape == (K,)
        y = np.empty(M, dtype=np.float64)
        S = np.empty(M, dtype=np.float64)
        if self.lib.bqo_gemv_f16(W_bits.ctypes.data, M, K, x.ctypes.data, y.ctypes.data,
                                 S.ctypes.data):
            raise ValueError("oracle gemv_f16: bad arguments")
        return y, S

    def rmsnorm(self, x, gamma, eps):
        x = np.ascontiguousarray(x, dtype=np.float64)
        g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float64)
        xn = np.empty_like(x)
        if self.lib.bqo_rmsnorm(x.ctypes.data, None if g is None else g.ctypes.data, x.size,
                                eps, xn.ctypes.data):
            raise ValueError("oracle rmsnorm: bad arguments")
        return xn

    def silu(self, z):
        return self.lib.bqo_silu(float(z))

    def gate_up_silu(self, qtype, Wg, Wu, M, K, xn):
        """Returns dict of fp64 arrays y, g, u, Sg, Su for y = silu(Wg xn) * (Wu xn)."""
        Wg = np.ascontiguousarray(Wg, dtype=np.uint8)
        Wu = np.ascontiguousarray(Wu, dtype=np.uint8)
        xn = np.ascontiguousarray(xn, dtype=np.float64)
        r = {k: np.empty(M, dtype=np.float64) for k in ("y", "g", "u", "Sg", "Su")}
        if self.lib.bqo_gate_up_silu(qtype, Wg.ctypes.data, Wu.ctypes.data, M, K,
                                     xn.ctypes.data, r["y"].ctypes.data, r["g"].ctypes.data,
                                     r["u"].ctypes.data, r["Sg"].ctypes.data,
                                     r["Su"].ctypes.data):
            raise ValueError("oracle gate_up_silu: bad arguments")
        return r


_default = None


def get():
    """The oracle built from ``oracle/bq_oracle.c`` (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
