"""Stream plans against the launch-per-op path: every output of every stage
bit-identical, on chained decode streams where each stage reads the previous
stage's output (run as one streaming-kernel launch per stage, or by the
cooperative executor in one launch), and on independent streams (one launch
of the streaming kernel); plus the oracle bound on the final outputs and
repeat-run determinism."""
import contextlib
import ctypes

import numpy as np
import pytest
import torch

import block_quantized_weight_dequant_gb300 as bq
from block_quantized_weight_dequant_gb300 import workloads as wl
from block_quantized_weight_dequant_gb300.decode import DecodeStream

import oracle
from tolerance import assert_gemv_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make_stream(qt, n_layers, hidden, q_dim, kv_dim, inter, vocab, seed=0, chained=True,
                fused_qkv=False):
    def packed(M, K, *tag):
        W = wl.normal_torch((M, K), wl.W_STD, seed=seed, stream=wl.stream_id(*tag), device=DEV)
        return bq.quantize_pack(W, qt)

    layers = []
    for l in range(n_layers):
        layers.append(dict(
            q=packed(q_dim, hidden, l, "q"), k=packed(kv_dim, hidden, l, "k"),
            v=packed(kv_dim, hidden, l, "v"), o=packed(hidden, q_dim, l, "o"),
            gate=packed(inter, hidden, l, "g"), up=packed(inter, hidden, l, "u"),
            down=packed(hidden, inter, l, "d"),
            gamma=wl.normal_torch(hidden, 0.1, seed=seed, stream=wl.stream_id(l, "gm"),
                                  device=DEV, mean=1.0)))
    if fused_qkv:
        for l, L in enumerate(layers):
            L["qkv"] = bq.concat_packed([L.pop("q"), L.pop("k"), L.pop("v")])
            L["qkv_bias"] = wl.normal_torch(L["qkv"].shape[0], 0.1, seed=seed,
                                            stream=wl.stream_id(l, "qkv_bias"), device=DEV)
    ds = DecodeStream(qt, layers, packed(vocab, hidden, "lm"), chained=chained,
                      fused_qkv=fused_qkv)
    ds.inputs.copy_(wl.normal_torch(ds.inputs.numel(), 1.0, seed=seed, stream=7, device=DEV))
    return ds


def snapshot(ds):
    return [op.y.clone() for op in ds.ops]


@contextlib.contextmanager
def plan_kind(kind):
    """Plans of dependent stages created inside run as `kind`: "staged" (one
    launch per stage), "executor" (one cooperative launch) or None (the
    library's default); a test hook outside the public header."""
    from block_quantized_weight_dequant_gb300 import _lib
    f = _lib.get().bq_internal_set_plan_kind
    f.argtypes = [ctypes.c_int]
    f.restype = None
    f({"staged": 1, "executor": 0, None: -1}[kind])
    try:
        yield
    finally:
        f(-1)


STREAMS = [
    ("q8_0", 3, 512, 512, 128, 1024, 3000),      # G = 4 and 8, whole rows per slot
    ("q8_0", 2, 1024, 2048, 512, 3072, 20000),   # Qwen3-0.6B layer shapes, chunked down
    ("q4_0", 2, 3584, 3584, 512, 18944, 4096),   # 7B layer shapes, G = 16, chunked down
    ("q4_0", 2, 256, 768, 256, 1280, 999),       # odd unit counts, ragged tiles
]


@pytest.mark.parametrize("qt,n_layers,hidden,q_dim,kv_dim,inter,vocab", STREAMS)
def test_tuned_plan_is_bitwise_the_same(qt, n_layers, hidden, q_dim, kv_dim, inter, vocab):
    """bq_stream_plan_tune moves tiles between CTAs by measured time; every
    output row keeps its arithmetic, so outputs stay bit-identical to the
    launch-per-op path, and a plan of dependent stages is left as it is."""
    ds = make_stream(qt, n_layers, hidden, q_dim, kv_dim, inter, vocab, chained=False)
    ds.run_per_op()
    want = snapshot(ds)
    plan = ds.plan()
    plan.tune(rounds=2)
    for op in ds.ops:
        op.y.fill_(float("nan"))
    ds.run_plan()
    for i, (g, w) in enumerate(zip(snapshot(ds), want)):
        assert torch.equal(g.view(torch.int32), w.view(torch.int32)), f"op {i} differs after tune"
    dc = make_stream(qt, 1, hidden, q_dim, kv_dim, inter, vocab, chained=True)
    dc.run_per_op()
    want_c = snapshot(dc)
    dc.plan().tune(rounds=1)
    dc.run_plan()
    for g, w in zip(snapshot(dc), want_c):
        assert torch.equal(g.view(torch.int32), w.view(torch.int32))
    with pytest.raises(bq.BQError):
        plan.tune(rounds=0)
    assert bq.device_status(clear=True) == 0


@pytest.mark.parametrize("mode", ["staged", "executor", "independent"])
@pytest.mark.parametrize("qt,n_layers,hidden,q_dim,kv_dim,inter,vocab", STREAMS)
def test_plan_matches_launch_per_op_bitwise(qt, n_layers, hidden, q_dim, kv_dim, inter, vocab,
                                            mode):
    """staged: chained stages, one streaming-kernel launch per stage (the
    default); executor: chained stages in one cooperative launch with
    grid-wide barriers; independent: one launch of the multi-op streaming
    kernel (the planner finds no dependence)."""
    chained = mode != "independent"
    ds = make_stream(qt, n_layers, hidden, q_dim, kv_dim, inter, vocab, chained=chained)
    ds.run_per_op()
    want = snapshot(ds)
    for op in ds.ops:
        op.y.fill_(float("nan"))
    with plan_kind(mode if chained else None):
        ds.plan()
    assert ds.plan().launches == (ds.n_stages if mode == "staged" else 1)
    ds.run_plan()
    got = snapshot(ds)
    for i, (g, w) in enumerate(zip(got, want)):
        assert torch.equal(g.view(torch.int32), w.view(torch.int32)), f"op {i} differs"
    # run again: the counters are reset per launch and the result repeats
    ds.run_plan()
    again = snapshot(ds)
    for g, w in zip(again, want):
        assert torch.equal(g.view(torch.int32), w.view(torch.int32))
    assert bq.device_status(clear=True) == 0


def test_plan_final_output_within_oracle_bound():
    qt = "q8_0"
    ds = make_stream(qt, 1, 512, 512, 128, 1024, 700)
    ds.run_plan()
    lm = ds.ops[-1]
    x = lm.x.cpu().numpy().astype(np.float64)
    y_ref, S = oracle.get().gemv(oracle.Q8_0, lm.W.cpu().numpy(), lm.W.shape[0], x.size, x)
    assert_gemv_close(lm.y.cpu().numpy(), y_ref, S, "plan lm_head")


@pytest.mark.parametrize("kind", ["staged", "executor"])
def test_plan_in_cuda_graph(kind):
    ds = make_stream("q8_0", 2, 512, 512, 128, 1024, 2000)
    ds.run_per_op()
    want = snapshot(ds)
    with plan_kind(kind):
        ds.plan()  # created before capture (it synchronises)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ds.run_plan()
    for op in ds.ops:
        op.y.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for g_, w in zip(snapshot(ds), want):
        assert torch.equal(g_.view(torch.int32), w.view(torch.int32))


def test_staged_plan_falls_back_to_the_executor():
    """A dependent stage whose input exceeds what the streaming kernel stages
    for one row (K = 34816 fp32, 136 KB, over its 128 KB limit) cannot run as
    a stage launch; the plan then runs on the cooperative executor in one
    launch (its Q4_0 rings leave room for that input), with the same bits as
    one call per op."""
    qt = "q4_0"

    def packed(M, K, tag):
        W = wl.normal_torch((M, K), wl.W_STD, seed=3, stream=wl.stream_id("fallback", tag), device=DEV)
        return bq.quantize_pack(W, qt)

    K0 = 34816
    W0, W1 = packed(256, K0, 0), packed(80, 256, 1)
    x = wl.normal_torch(K0, 1.0, seed=3, stream=wl.stream_id("fallback-x"), device=DEV)
    y0 = torch.empty(256, device=DEV)
    y1 = torch.empty(80, device=DEV)
    ops = [bq.StreamOp(0, W0, x, y0), bq.StreamOp(1, W1, y0, y1)]
    bq.gemv(qt, W0, x, y0)
    bq.gemv(qt, W1, y0, y1)
    want = [y0.clone(), y1.clone()]
    y0.fill_(float("nan"))
    y1.fill_(float("nan"))
    with plan_kind("staged"):
        plan = bq.StreamPlan(qt, ops)
    assert plan.launches == 1
    plan.launch()
    torch.cuda.synchronize()
    for g, w in zip((y0, y1), want):
        assert torch.equal(g.view(torch.int32), w.view(torch.int32))
    assert bq.device_status(clear=True) == 0


def test_plan_rejects_bad_ops():
    P = bq.quantize_pack(torch.zeros(64, 512, device=DEV), "q8_0")
    x = torch.zeros(512, device=DEV)
    y = torch.zeros(64, device=DEV)
    with pytest.raises(bq.BQError):  # first stage must be 0
        bq.StreamPlan("q8_0", [bq.StreamOp(1, P, x, y)])
    with pytest.raises(bq.BQError):  # stages may not skip
        bq.StreamPlan("q8_0", [bq.StreamOp(0, P, x, y), bq.StreamOp(2, P, x, y)])
    P2 = bq.quantize_pack(torch.zeros(64, 288, device=DEV), "q8_0")
    with pytest.raises(bq.BQError):  # K % 256 != 0 is not streamed
        bq.StreamPlan("q8_0", [bq.StreamOp(0, P2, torch.zeros(288, device=DEV), y)])


def test_unchained_stream_matches_launch_per_op_bitwise():
    """Independent inputs: the planner finds no dependence and the executor
    runs without grid-wide barriers; results still match op by op."""
    qt = "q8_0"

    def packed(M, K, *tag):
        W = wl.normal_torch((M, K), wl.W_STD, seed=5, stream=wl.stream_id(*tag), device=DEV)
        return bq.quantize_pack(W, qt)

    layers = [dict(q=packed(512, 512, l, "q"), k=packed(128, 512, l, "k"),
                   v=packed(128, 512, l, "v"), o=packed(512, 512, l, "o"),
                   gate=packed(1024, 512, l, "g"), up=packed(1024, 512, l, "u"),
                   down=packed(512, 1024, l, "d"),
                   gamma=wl.normal_torch(512, 0.1, seed=5, stream=l, device=DEV, mean=1.0))
              for l in range(3)]
    ds = DecodeStream(qt, layers, packed(3000, 512, "lm"), chained=False)
    ds.inputs.copy_(wl.normal_torch(ds.inputs.numel(), 1.0, seed=5, stream=9, device=DEV))
    ds.run_per_op()
    want = snapshot(ds)
    for op in ds.ops:
        op.y.fill_(float("nan"))
    ds.run_plan()
    for i, (g, w) in enumerate(zip(snapshot(ds), want)):
        assert torch.equal(g.view(torch.int32), w.view(torch.int32)), f"op {i} differs"


def test_plan_rejects_outputs_overlapping_weights_or_own_stage():
    P = bq.quantize_pack(torch.zeros(64, 512, device=DEV), "q8_0")
    x = torch.zeros(512, device=DEV)
    y = torch.zeros(64, device=DEV)
    # an output written over packed weights (weights are prefetched across stages)
    wy = P.view(torch.float32).view(-1)[:64]
    with pytest.raises(bq.BQError):
        bq.StreamPlan("q8_0", [bq.StreamOp(0, P, x, wy)])
    # an output that is an input of its own stage
    y2 = torch.zeros(512, device=DEV)
    P2 = bq.quantize_pack(torch.zeros(512, 512, device=DEV), "q8_0")
    with pytest.raises(bq.BQError):
        bq.StreamPlan("q8_0", [bq.StreamOp(0, P2, x, y2), bq.StreamOp(0, P, y2, y)])
    # ... which is fine one stage later (the planner inserts a barrier)
    bq.StreamPlan("q8_0", [bq.StreamOp(0, P2, x, y2), bq.StreamOp(1, P, y2, y)])


@pytest.mark.parametrize("mode", ["staged", "executor", "independent"])
@pytest.mark.parametrize("qt,n_layers,hidden,q_dim,kv_dim,inter,vocab", [
    ("q8_0", 2, 1024, 2048, 512, 3072, 7000),   # Qwen3-0.6B layer shapes
    ("q4_0", 2, 3584, 3584, 512, 18944, 3000),  # 7B layer shapes
])
def test_fused_qkv_bias_plan_matches_launch_per_op_bitwise(qt, n_layers, hidden, q_dim, kv_dim,
                                                           inter, vocab, mode):
    """One fused q|k|v + bias op per layer (4 ops per layer): the plan (one
    launch per stage, the stream executor, or the multi-op kernel) and one
    launch per op agree bit for bit."""
    chained = mode != "independent"
    ds = make_stream(qt, n_layers, hidden, q_dim, kv_dim, inter, vocab, chained=chained,
                     fused_qkv=True)
    assert len(ds.ops) == 4 * n_layers + 1
    ds.run_per_op()
    want = snapshot(ds)
    for op in ds.ops:
        op.y.fill_(float("nan"))
    with plan_kind(mode if chained else None):
        ds.plan()
    ds.run_plan()
    torch.cuda.synchronize()
    for i, (op, w) in enumerate(zip(ds.ops, want)):
        assert torch.equal(op.y.view(torch.int32), w.view(torch.int32)), f"op {i}"
    assert bq.device_status(clear=True) == 0


BQ_DEVERR_BARRIER_WAIT = 0x8


def test_stage_barrier_wait_runs_out_and_reports():
    """Failure detection without a fault.  A stage barrier told to wait for one
    arrival more than the grid's CTAs can never complete; with the bounded
    waits' limit set to 1 ms for that launch, every CTA gives up, records
    BQ_DEVERR_BARRIER_WAIT in the device error word and returns (its warps
    waiting on shared-memory phases see the CTA's abort flag and return too).
    The host reads the word through bq_device_status; the context stays
    usable, and the same plan run normally afterwards gives the launch-per-op
    bits."""
    from block_quantized_weight_dequant_gb300 import _lib
    lib = _lib.get()
    hook = lib.bq_internal_plan_barrier_extra
    hook.argtypes = [ctypes.c_void_p, ctypes.c_uint, ctypes.c_ulonglong]
    hook.restype = ctypes.c_int
    ds = make_stream("q8_0", 2, 512, 512, 128, 1024, 2000, chained=True)
    ds.run_per_op()
    want = snapshot(ds)
    assert bq.device_status(clear=True) == 0
    with plan_kind("executor"):
        plan = ds.plan()
    assert hook(plan._handle, 1, 1_000_000) == 0
    plan.launch()
    flags = ctypes.c_uint(0)
    assert lib.bq_device_status(ctypes.byref(flags), 1) == _lib.BQ_ERR_DEVICE
    assert flags.value & BQ_DEVERR_BARRIER_WAIT, hex(flags.value)
    assert bq.device_status(clear=True) == 0  # cleared
    # the same plan with its barriers intact
    assert hook(plan._handle, 0, 2_000_000_000) == 0
    for op in ds.ops:
        op.y.fill_(float("nan"))
    ds.run_plan()
    for i, (g, w) in enumerate(zip(snapshot(ds), want)):
        assert torch.equal(g.view(torch.int32), w.view(torch.int32)), f"op {i} differs after"
    assert bq.device_status(clear=True) == 0
    # plans of independent ops, and staged plans, have no stage barrier to break
    di = make_stream("q8_0", 1, 512, 512, 128, 1024, 2000, chained=False)
    assert hook(di.plan()._handle, 1, 1_000_000) == -1
    dst = make_stream("q8_0", 1, 512, 512, 128, 1024, 2000, chained=True)
    with plan_kind("staged"):
        assert hook(dst.plan()._handle, 1, 1_000_000) == -1
