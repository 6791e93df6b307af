"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times: the workloads are built by bench.py's own builders (the same seeded
weights, inputs and, for the token streams, the tuned one-launch plan), run
once, and their outputs compared with the oracle on sampled rows
(tests/sampled_parity.py: the oracle re-packs the seeded fp32 rows itself, the
GPU's packed rows must equal its bytes, and every checked output is within the
GEMV bound of the oracle's fp64 product).

- Q8_0 GEMV 3072x1024: every row of the first and the last rotated copy;
- Qwen3-0.6B-shaped Q8_0 token (28 layers + 151936-row LM head) and the
  7B-shaped token (28 layers + 152064-row LM head) in Q4_0 and in Q4_K: every
  row of every layer-0 matrix, and 4096 seeded rows (with the first and the
  last) of every other matrix;
- RMSNorm + gate/up + SiLU 3072x1024: every row of the first and last pair;
- Q4_0 verify 17408x5120 and 5120x17408, R = 1..6: 4096 sampled rows of every
  input row against the oracle, and every output row memcmp-equal to the
  single-row decode GEMV;
- fp16-weight LM head 151936x1024: 4096 sampled rows.
"""
import argparse

import pytest
import torch

import bench

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def args(config, **kw):
    a = dict(config=config, layers=0, qkv="separate", launch="plan", inputs="independent",
             rows=6, tune=True, other_inputs=False)
    a.update(kw)
    return argparse.Namespace(**a)


def run_once(w):
    torch.cuda.synchronize()
    w.run()
    torch.cuda.synchronize()


def assert_parity(p, what):
    assert p["pass"], f"{what}: {p}"
    assert p["skipped_matrices"] == 0, f"{what}: {p}"


def test_q8_0_gemv_3072x1024_every_row():
    w = bench.build_workload(args("cfg1"), DEV)
    run_once(w)
    w.checks = [w.checks[0], w.checks[-1]]
    p = bench.sampled_parity(w, 3072)
    assert p["rows"] == 2 * 3072
    assert_parity(p, "cfg1")


def test_gate_up_silu_3072x1024_every_row():
    w = bench.build_workload(args("cfg4"), DEV)
    run_once(w)
    w.checks = [w.checks[0], w.checks[-1]]
    p = bench.sampled_parity(w, 3072)
    assert p["rows"] == 2 * 3072
    assert_parity(p, "cfg4")


@pytest.mark.parametrize("config", ["cfg2", "cfg3", "cfg3k"])
def test_token_stream_full_size(config):
    """The whole tuned one-launch token stream; every row of layer 0 and 4096
    rows of every other matrix."""
    w = bench.build_workload(args(config), DEV)
    for op in w.stream_obj.ops:
        op.y.fill_(float("nan"))  # every output row must be written
    run_once(w)
    ops_per_layer = 6  # q, k, v, o, gate+up, down
    assert len(w.checks) == 28 * ops_per_layer + 1
    p = bench.sampled_parity(w, lambda i: 1 << 30 if i < ops_per_layer else 4096)
    assert_parity(p, config)
    import block_quantized_weight_dequant_gb300 as bq
    assert bq.device_status(clear=True) == 0


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6])
def test_verify_full_size(R):
    w = bench.build_verify(DEV, bench.wl_cfg5(), R, copies=1)
    run_once(w)
    p = bench.sampled_parity(w, 4096)
    assert p["verify_rows_differ_from_decode"] == 0
    assert_parity(p, f"cfg5 R={R}")
    # every output row, not only the sampled ones, equals the decode GEMV
    import block_quantized_weight_dequant_gb300 as bq
    for c in w.checks:
        for r in range(R):
            yd = bq.gemv(c["qt"], c["P"], c["X"][r].contiguous())
            assert torch.equal(c["Y"][r].view(torch.int32), yd.view(torch.int32)), (c["tag"], r)


def test_f16_lm_head_sampled_rows():
    w = bench.build_workload(args("f16"), DEV)
    run_once(w)
    p = bench.sampled_parity(w, 4096)
    assert p["rows"] == 4096
    assert_parity(p, "f16")
