"""The allocation-free stream executor entry point (bq_stream_run_noalloc).

Callers that cannot allocate device memory -- a server whose HBM is already
parcelled out to weight and KV-cache pools, a framework that forbids raw
cudaMalloc beside its own caching allocator, a latency-critical path that
cannot afford an allocation's device synchronisation -- use this entry point
instead of a plan with a caller-allocated workspace.  This test calls it
through the C ABI on a decode stream, chained (the stream executor) and with
independent inputs (the multi-op kernel), twice in a row (the second call must
clear the barrier counters the first left behind), and checks every output
against the workspace-based plan, which is the existing entry point:
bit for bit, and the final logits within the library's GEMV bound against the
oracle.  It lives in a file of its own that pytest collects last, and it
passes alone in a fresh process (its first call does the per-device set-up)
as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_quantized_weight_dequant_gb300 as bq
from block_quantized_weight_dequant_gb300 import _lib
from block_quantized_weight_dequant_gb300 import workloads as wl
from block_quantized_weight_dequant_gb300.decode import DecodeStream

import oracle
from tolerance import assert_gemv_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def chained_stream(qt, seed=11, chained=True):
    def packed(M, K, *tag):
        W = wl.normal_torch((M, K), wl.W_STD, seed=seed, stream=wl.stream_id(*tag), device=DEV)
        return bq.quantize_pack(W, qt)

    hidden, q_dim, kv, inter = 1024, 2048, 512, 3072
    layers = [dict(q=packed(q_dim, hidden, l, "q"), k=packed(kv, hidden, l, "k"),
                   v=packed(kv, hidden, l, "v"), o=packed(hidden, q_dim, l, "o"),
                   gate=packed(inter, hidden, l, "g"), up=packed(inter, hidden, l, "u"),
                   down=packed(hidden, inter, l, "d"),
                   gamma=wl.normal_torch(hidden, 0.1, seed=seed, stream=wl.stream_id(l, "gm"),
                                         device=DEV, mean=1.0))
              for l in range(2)]
    ds = DecodeStream(qt, layers, packed(5000, hidden, "lm"), chained=chained)
    ds.inputs.copy_(wl.normal_torch(ds.inputs.numel(), 1.0, seed=seed, stream=3, device=DEV))
    return ds


def op_array(ds):
    arr = (_lib.BqOp * len(ds.ops))()
    for i, op in enumerate(ds.ops):
        a = arr[i]
        a.stage, a.M, a.K = op.stage, op.y.numel(), op.x.numel()
        a.W, a.x, a.y = op.W.data_ptr(), op.x.data_ptr(), op.y.data_ptr()
        if op.W_up is None:
            a.kind = _lib.BQ_OP_GEMV
        else:
            a.kind, a.W_up, a.eps = _lib.BQ_OP_GATE_UP_SILU, op.W_up.data_ptr(), op.eps
            a.gamma = op.gamma.data_ptr() if op.gamma is not None else None
    return arr


@pytest.mark.parametrize("chained", [True, False], ids=["chained", "independent"])
@pytest.mark.parametrize("qt", ["q8_0", "q4_0", "q4_k"])
def test_noalloc_matches_workspace_plan_on_two_calls(qt, chained):
    """chained: the stream executor; independent: the multi-op kernel."""
    ds = chained_stream(qt, chained=chained)
    ds.run_plan()  # the existing entry point: caller-allocated workspace
    torch.cuda.synchronize()
    want = [op.y.clone() for op in ds.ops]
    arr = op_array(ds)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    lm = ds.ops[-1]
    x = lm.x.cpu().numpy().astype(np.float64)
    y_ref, S = oracle.get().gemv(bq.QTYPES[qt], lm.W.cpu().numpy(), lm.y.numel(), x.size, x)
    if qt == "q4_k":  # the bound's scale for the split super-block evaluation
        S = oracle.get().q4_k_split_scale(lm.W.cpu().numpy(), lm.y.numel(), x.size, x)
    for call in range(2):
        for op in ds.ops:
            op.y.fill_(float("nan"))
        rc = _lib.get().bq_stream_run_noalloc(bq.QTYPES[qt], arr, len(ds.ops), stream)
        assert rc == _lib.BQ_OK, _lib.status_str(rc)
        torch.cuda.synchronize()
        for i, (op, w) in enumerate(zip(ds.ops, want)):
            assert torch.equal(op.y.view(torch.int32), w.view(torch.int32)), \
                f"call {call}: op {i} differs from the workspace plan"
        assert_gemv_close(lm.y.cpu().numpy(), y_ref, S, f"noalloc call {call} logits")
    assert bq.device_status(clear=True) == 0


def test_noalloc_rejects_too_many_ops():
    ds = chained_stream("q8_0")
    arr = op_array(ds)
    big = (_lib.BqOp * (_lib.BQ_NOALLOC_MAX_OPS + 1))()
    for i in range(len(big)):
        big[i] = arr[0]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert _lib.get().bq_stream_run_noalloc(bq.Q8_0, big, len(big), stream) == _lib.BQ_ERR_SHAPE


@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
def test_noalloc_back_to_back_different_op_lists(qt):
    """Two calls with DIFFERENT op lists queued on one stream with no host
    synchronisation between them: each call's tables are staged in the same
    static host arrays, so the second call must not refill them before the
    first call's copies have read them.  Both outputs must equal the workspace
    plan's bit for bit."""
    a = chained_stream(qt, seed=21, chained=True)
    b = chained_stream(qt, seed=22, chained=False)
    want = []
    for ds in (a, b):
        ds.run_plan()
        torch.cuda.synchronize()
        want.append([op.y.clone() for op in ds.ops])
        for op in ds.ops:
            op.y.fill_(float("nan"))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    arr_a, arr_b = op_array(a), op_array(b)
    for _ in range(2):
        assert _lib.get().bq_stream_run_noalloc(bq.QTYPES[qt], arr_a, len(a.ops), stream) == _lib.BQ_OK
        assert _lib.get().bq_stream_run_noalloc(bq.QTYPES[qt], arr_b, len(b.ops), stream) == _lib.BQ_OK
    torch.cuda.synchronize()
    for name, ds, wnt in (("a", a, want[0]), ("b", b, want[1])):
        for i, (op, w) in enumerate(zip(ds.ops, wnt)):
            assert torch.equal(op.y.view(torch.int32), w.view(torch.int32)), f"list {name} op {i}"
    assert bq.device_status(clear=True) == 0
