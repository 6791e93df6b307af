"""Block-quantized weight dequant + batch-1 GEMV for GB300 (sm_103a).

A thin Python binding over libbqgemv.so (include/bqgemv.h).  Every function
here only marshals arguments: it checks tensor dtypes/devices, allocates
outputs with PyTorch when the caller passes none, and calls the C ABI on the
current CUDA stream.  All arithmetic runs in this package's CUDA kernels.

Packed weights are uint8 tensors of shape [M, (K/32) * block_bytes]
(34 bytes per 32 weights for Q8_0, 18 for Q4_0 and for Q4_K, whose 144-byte
super-blocks hold 256 weights), so M and K are read from the packed tensor's
shape.
"""
import ctypes

import torch

from . import _lib
from ._lib import BQ_Q4_0, BQ_Q4_K, BQ_Q8_0, BQ_VERIFY_MAX_ROWS, BQError, lib  # noqa: F401

Q8_0 = BQ_Q8_0
Q4_0 = BQ_Q4_0
Q4_K = BQ_Q4_K
# packed bytes per 32 weights (a Q4_K super-block is 144 bytes per 256 weights)
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18, Q4_K: 18}
QTYPES = {"q8_0": Q8_0, "q4_0": Q4_0, "q4_k": Q4_K}

__all__ = ["Q8_0", "Q4_0", "Q4_K", "BLOCK_BYTES", "BQError", "packed_bytes", "quantize_pack",
           "gemv", "gemv_q8_0", "gemv_q4_0", "gemv_q4_k", "gemv_gate_up_silu", "gemv_verify",
           "gemv_qkv_bias", "gemv_f16", "concat_packed",
           "device_status", "tree_lanes", "version", "StreamOp", "StreamPlan"]


def _qt(qtype):
    return QTYPES[qtype] if isinstance(qtype, str) else int(qtype)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need(t, dtype, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (this package has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _packed_shape(Wq, qtype):
    if Wq.dim() != 2:
        raise ValueError("packed weights must be 2-D [M, (K/32)*block_bytes]")
    bb = BLOCK_BYTES[qtype]
    M, rb = Wq.shape
    if rb % bb:
        raise ValueError(f"packed row of {rb} bytes is not whole {bb}-byte blocks")
    return M, (rb // bb) * 32


def version():
    return lib.bq_version()


def tree_lanes(K):
    """Lanes G of the fixed summation tree of a row of K weights."""
    return lib.bq_tree_lanes(int(K))


def packed_bytes(qtype, M, K):
    n = lib.bq_packed_bytes(_qt(qtype), int(M), int(K))
    if n < 0:
        raise ValueError(f"no packed size for qtype={qtype} M={M} K={K}")
    return n


def quantize_pack(W, qtype, out=None):
    """fp32 CUDA [M, K] -> packed uint8 [M, (K/32)*block_bytes]."""
    qt = _qt(qtype)
    _need(W, torch.float32, "W")
    if W.dim() != 2:
        raise ValueError("W must be 2-D [M, K]")
    M, K = W.shape
    if out is None:
        out = torch.empty((M, (K // 32) * BLOCK_BYTES[qt]), dtype=torch.uint8, device=W.device)
    _need(out, torch.uint8, "out")
    _lib.check(lib.bq_quantize_pack(qt, _ptr(W), M, K, _ptr(out), _stream(W)), "quantize_pack")
    return out


def gemv(qtype, Wq, x, y=None):
    """y = W x for packed weights Wq and fp32 x [K]."""
    qt = _qt(qtype)
    _need(Wq, torch.uint8, "Wq")
    _need(x, torch.float32, "x")
    M, K = _packed_shape(Wq, qt)
    if x.numel() != K:
        raise ValueError(f"x has {x.numel()} elements, weights have K={K}")
    if y is None:
        y = torch.empty(M, dtype=torch.float32, device=Wq.device)
    _need(y, torch.float32, "y")
    fn = {Q8_0: lib.bq_gemv_q8_0, Q4_0: lib.bq_gemv_q4_0, Q4_K: lib.bq_gemv_q4_k}[qt]
    _lib.check(fn(_ptr(Wq), _ptr(x), _ptr(y), M, K, _stream(Wq)), "gemv")
    return y


def gemv_q8_0(Wq, x, y=None):
    return gemv(Q8_0, Wq, x, y)


def gemv_q4_0(Wq, x, y=None):
    return gemv(Q4_0, Wq, x, y)


def gemv_q4_k(Wq, x, y=None):
    return gemv(Q4_K, Wq, x, y)


def gemv_gate_up_silu(qtype, Wg, Wu, x, gamma=None, eps=1e-6, y=None):
    """y = silu(Wg xn) * (Wu xn), xn = x * gamma / sqrt(mean(x^2) + eps)
    (xn = x when gamma is None)."""
    qt = _qt(qtype)
    _need(Wg, torch.uint8, "Wg")
    _need(Wu, torch.uint8, "Wu")
    _need(x, torch.float32, "x")
    if gamma is not None:
        _need(gamma, torch.float32, "gamma")
    M, K = _packed_shape(Wg, qt)
    if tuple(Wu.shape) != tuple(Wg.shape):
        raise ValueError("Wg and Wu must have the same shape")
    if x.numel() != K or (gamma is not None and gamma.numel() != K):
        raise ValueError("x and gamma must have K elements")
    if y is None:
        y = torch.empty(M, dtype=torch.float32, device=Wg.device)
    _need(y, torch.float32, "y")
    _lib.check(lib.bq_gemv_gate_up_silu(qt, _ptr(Wg), _ptr(Wu), _ptr(x), _ptr(gamma),
                                        float(eps), _ptr(y), M, K, _stream(Wg)),
               "gemv_gate_up_silu")
    return y


def concat_packed(mats):
    """Load-time concatenation of packed matrices with the same K (e.g. the
    q, k and v projections): a packed matrix is its rows back to back, so the
    rows are concatenated as they are.  No arithmetic."""
    if not mats:
        raise ValueError("no matrices")
    rb = mats[0].shape[1]
    for P in mats:
        _need(P, torch.uint8, "packed matrix")
        if P.dim() != 2 or P.shape[1] != rb:
            raise ValueError("packed matrices must share the row size (same K and format)")
    return torch.cat(list(mats), dim=0)


def gemv_qkv_bias(qtype, Wqkv, x, bias=None, y=None):
    """y = Wqkv x + bias over the concatenated q|k|v rows (concat_packed):
    the single-row GEMV's dot products, then one fp32 add of the bias."""
    qt = _qt(qtype)
    _need(Wqkv, torch.uint8, "Wqkv")
    _need(x, torch.float32, "x")
    M, K = _packed_shape(Wqkv, qt)
    if x.numel() != K:
        raise ValueError(f"x must have K={K} elements")
    if bias is not None:
        _need(bias, torch.float32, "bias")
        if bias.numel() != M:
            raise ValueError(f"bias must have M={M} elements")
    if y is None:
        y = torch.empty(M, dtype=torch.float32, device=Wqkv.device)
    _need(y, torch.float32, "y")
    _lib.check(lib.bq_gemv_qkv_bias(qt, _ptr(Wqkv), _ptr(x), _ptr(bias), _ptr(y), M, K,
                                    _stream(Wqkv)), "gemv_qkv_bias")
    return y


def gemv_f16(W, x, y=None, out_dtype=torch.float32):
    """y = W x for unquantized fp16 weights W [M, K] (K % 8 == 0) and fp32 x,
    on the fixed tree of bq_gemv_f16 (bit-reproducible).  y is fp32, or fp16
    (out_dtype=torch.float16, or a given fp16 y: bq_gemv_f16_f16out, the fp32
    result rounded to nearest even)."""
    _need(W, torch.float16, "W")
    _need(x, torch.float32, "x")
    if W.dim() != 2:
        raise ValueError("W must be [M, K]")
    M, K = W.shape
    if x.numel() != K:
        raise ValueError(f"x must have K={K} elements")
    if y is None:
        y = torch.empty(M, dtype=out_dtype, device=W.device)
    if not isinstance(y, torch.Tensor) or y.dtype not in (torch.float32, torch.float16):
        raise TypeError("y must be a torch.float32 or torch.float16 tensor")
    _need(y, y.dtype, "y")
    if y.numel() != M:
        raise ValueError(f"y must have M={M} elements")
    fn = lib.bq_gemv_f16 if y.dtype == torch.float32 else lib.bq_gemv_f16_f16out
    _lib.check(fn(_ptr(W), _ptr(x), _ptr(y), M, K, _stream(W)), "gemv_f16")
    return y


def gemv_verify(qtype, Wq, X, Y=None):
    """Y [R, M] = X [R, K] @ W^T with the weights streamed once; row r is
    bit-identical to gemv(qtype, Wq, X[r])."""
    qt = _qt(qtype)
    _need(Wq, torch.uint8, "Wq")
    _need(X, torch.float32, "X")
    M, K = _packed_shape(Wq, qt)
    if X.dim() != 2 or X.shape[1] != K:
        raise ValueError(f"X must be [R, {K}]")
    R = X.shape[0]
    if Y is None:
        Y = torch.empty((R, M), dtype=torch.float32, device=Wq.device)
    _need(Y, torch.float32, "Y")
    _lib.check(lib.bq_gemv_verify(qt, _ptr(Wq), _ptr(X), _ptr(Y), R, M, K, _stream(Wq)),
               "gemv_verify")
    return Y


def device_status(clear=True):
    """Device-side error word (0 = healthy); synchronises the device."""
    flags = ctypes.c_uint(0)
    st = lib.bq_device_status(ctypes.byref(flags), int(clear))
    if st not in (_lib.BQ_OK, _lib.BQ_ERR_DEVICE):
        raise BQError(st, "device_status")
    return flags.value


class StreamOp:
    """One op of a per-token stream: a GEMV (``W`` only, optional ``bias``
    added to its output: the fused q|k|v + bias projection) or a fused
    RMSNorm+gate+up+SiLU (``W`` = gate, ``W_up`` = up, optional ``gamma``).
    ``stage`` orders the ops: ops of one stage run concurrently, and an op may
    read the output ``y`` of an op of an earlier stage as its ``x``."""

    def __init__(self, stage, W, x, y, W_up=None, gamma=None, eps=1e-6, bias=None):
        self.stage, self.W, self.x, self.y = int(stage), W, x, y
        self.W_up, self.gamma, self.eps, self.bias = W_up, gamma, float(eps), bias


class StreamPlan:
    """A whole list of StreamOps run per call (bq_stream_plan_* of
    include/bqgemv.h): independent ops in one launch of the streaming kernel,
    dependent stages in one launch per stage (``launches``).  The descriptor
    workspace is a torch tensor this object owns; keep the op tensors alive as
    long as the plan.  ``launch()`` enqueues on the current stream and can be
    captured in a CUDA graph; creating the plan synchronises, so do it before
    capture."""

    def __init__(self, qtype, ops):
        qt = _qt(qtype)
        if not ops:
            raise ValueError("empty op list")
        arr = (_lib.BqOp * len(ops))()
        for i, op in enumerate(ops):
            _need(op.W, torch.uint8, "W")
            _need(op.x, torch.float32, "x")
            _need(op.y, torch.float32, "y")
            M, K = _packed_shape(op.W, qt)
            if op.x.numel() != K or op.y.numel() != M:
                raise ValueError(f"op {i}: x must have K={K} and y M={M} elements")
            a = arr[i]
            a.stage, a.M, a.K = op.stage, M, K
            a.W, a.x, a.y = op.W.data_ptr(), op.x.data_ptr(), op.y.data_ptr()
            if op.W_up is not None:
                _need(op.W_up, torch.uint8, "W_up")
                if tuple(op.W_up.shape) != tuple(op.W.shape):
                    raise ValueError(f"op {i}: W_up must match W")
                a.kind, a.W_up, a.eps = _lib.BQ_OP_GATE_UP_SILU, op.W_up.data_ptr(), op.eps
                if op.gamma is not None:
                    _need(op.gamma, torch.float32, "gamma")
                    a.gamma = op.gamma.data_ptr()
            else:
                a.kind = _lib.BQ_OP_GEMV
                if op.bias is not None:
                    _need(op.bias, torch.float32, "bias")
                    if op.bias.numel() != M:
                        raise ValueError(f"op {i}: bias must have M={M} elements")
                    a.bias = op.bias.data_ptr()
        nstages = len({op.stage for op in ops})
        nbytes = lib.bq_stream_workspace_bytes(len(ops), nstages)
        if nbytes < 0:
            raise ValueError("bad op/stage counts")
        dev = ops[0].W.device
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=dev)
        base = self.workspace.data_ptr()
        ws = ctypes.c_void_p((base + 255) // 256 * 256)
        self._ops = ops  # keep the tensors alive
        self._handle = ctypes.c_void_p()
        self.n_ops, self.n_stages = len(ops), nstages
        with torch.cuda.device(dev):
            _lib.check(lib.bq_stream_plan_create(qt, arr, len(ops), ws, nbytes,
                                                 ctypes.byref(self._handle)), "stream_plan_create")
        self.device = dev

    def launch(self):
        _lib.check(lib.bq_stream_plan_launch(self._handle, _stream(self._ops[0].W)),
                   "stream_plan_launch")

    @property
    def launches(self):
        """Kernel launches one ``launch()`` enqueues (bq_stream_plan_launches)."""
        return int(lib.bq_stream_plan_launches(self._handle))

    def tune(self, rounds=3):
        """Re-split the plan's tiles among CTAs by measured time
        (bq_stream_plan_tune): runs the plan a few times, overwriting the
        ops' outputs; synchronous, so call it before graph capture."""
        _lib.check(lib.bq_stream_plan_tune(self._handle, int(rounds), _stream(self._ops[0].W)),
                   "stream_plan_tune")

    def __del__(self):
        h = getattr(self, "_handle", None)
        if h is not None and h.value:
            lib.bq_stream_plan_destroy(h)
            self._handle = None
