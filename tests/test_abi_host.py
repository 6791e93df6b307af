"""The C-ABI library on the host, without a GPU: it loads, exports every
symbol include/bqgemv.h declares, and rejects bad arguments before touching
the device.  No compute call runs here."""
import ctypes
import os
import re
import subprocess

import pytest

import block_quantized_weight_dequant_gb300 as bq
from block_quantized_weight_dequant_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bqgemv.h")

# a well-aligned fake device address: validation must reject or accept calls
# on arguments alone, before any CUDA call could dereference it
FAKE = ctypes.c_void_p(0x10000)
MIS = ctypes.c_void_p(0x10004)  # 4-byte aligned only


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bq_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return _lib.get()


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (bq_\w+)", out))
    assert set(names) <= exported, set(names) - exported
    assert set(_lib.EXPORTS) == set(names)
    for n in names:
        assert getattr(lib, n) is not None


def test_version_and_status_strings(lib):
    assert lib.bq_version() >= 100
    for s in range(7):
        assert len(_lib.status_str(s)) >= 2
    assert _lib.status_str(99) == "unknown status"


def test_packed_bytes(lib):
    assert lib.bq_packed_bytes(bq.Q8_0, 3072, 1024) == 3072 * 32 * 34
    assert lib.bq_packed_bytes(bq.Q4_0, 152064, 3584) == 152064 * 112 * 18
    assert lib.bq_packed_bytes(bq.Q8_0, 0, 1024) == 0
    assert lib.bq_packed_bytes(bq.Q8_0, 5, 33) == -1
    assert lib.bq_packed_bytes(3, 5, 32) == -1
    assert lib.bq_packed_bytes(bq.Q4_0, -1, 32) == -1


def test_tree_lanes_rule(lib):
    # G = largest power of two <= 32 wasting <= 1/8 of G*ceil(units/G) slots
    for K in range(32, 40000, 32):
        nsc = (K // 32 + 7) // 8
        G = lib.bq_tree_lanes(K)
        assert G in (1, 2, 4, 8, 16, 32)
        slots = G * -(-nsc // G)
        assert (slots - nsc) * 8 <= slots
        if G < 32:
            G2 = 2 * G
            slots2 = G2 * -(-nsc // G2)
            assert (slots2 - nsc) * 8 > slots2, K
    assert [lib.bq_tree_lanes(k) for k in (1024, 2048, 3072, 3584, 5120, 17408, 18944)] == \
        [4, 8, 4, 16, 4, 8, 16]
    assert lib.bq_tree_lanes(0) == -1 and lib.bq_tree_lanes(48) == -1


def test_gemv_argument_validation(lib):
    for fn in (lib.bq_gemv_q8_0, lib.bq_gemv_q4_0):
        assert fn(None, FAKE, FAKE, 8, 256, None) == _lib.BQ_ERR_NULL
        assert fn(FAKE, None, FAKE, 8, 256, None) == _lib.BQ_ERR_NULL
        assert fn(FAKE, FAKE, None, 8, 256, None) == _lib.BQ_ERR_NULL
        assert fn(FAKE, FAKE, FAKE, 8, 48, None) == _lib.BQ_ERR_SHAPE
        assert fn(FAKE, FAKE, FAKE, 8, 0, None) == _lib.BQ_ERR_SHAPE
        assert fn(FAKE, FAKE, FAKE, 8, (1 << 18) + 32, None) == _lib.BQ_ERR_SHAPE
        assert fn(FAKE, FAKE, FAKE, -1, 256, None) == _lib.BQ_ERR_SHAPE
        assert fn(FAKE, FAKE, FAKE, 1 << 31, 256, None) == _lib.BQ_ERR_SHAPE
        assert fn(MIS, FAKE, FAKE, 8, 256, None) == _lib.BQ_ERR_ALIGN
        assert fn(FAKE, MIS, FAKE, 8, 256, None) == _lib.BQ_ERR_ALIGN
        assert fn(FAKE, FAKE, ctypes.c_void_p(0x10002), 8, 256, None) == _lib.BQ_ERR_ALIGN
        # M == 0 is an empty product: accepted, nothing launched, NULL allowed
        assert fn(FAKE, FAKE, FAKE, 0, 256, None) == _lib.BQ_OK
        assert fn(None, None, None, 0, 256, None) == _lib.BQ_OK
        assert fn(None, None, None, 0, 48, None) == _lib.BQ_ERR_SHAPE


def test_verify_and_gate_up_validation(lib):
    v = lib.bq_gemv_verify
    assert v(bq.Q4_0, FAKE, FAKE, FAKE, 0, 8, 256, None) == _lib.BQ_ERR_SHAPE
    assert v(bq.Q4_0, FAKE, FAKE, FAKE, 7, 8, 256, None) == _lib.BQ_ERR_SHAPE
    assert v(5, FAKE, FAKE, FAKE, 2, 8, 256, None) == _lib.BQ_ERR_QTYPE
    assert v(bq.Q8_0, FAKE, FAKE, FAKE, 6, 0, 256, None) == _lib.BQ_OK
    g = lib.bq_gemv_gate_up_silu
    assert g(bq.Q8_0, FAKE, None, FAKE, None, 1e-6, FAKE, 8, 256, None) == _lib.BQ_ERR_NULL
    assert g(bq.Q8_0, FAKE, FAKE, FAKE, MIS, 1e-6, FAKE, 8, 256, None) == _lib.BQ_ERR_ALIGN
    assert g(bq.Q8_0, FAKE, FAKE, FAKE, FAKE, -1.0, FAKE, 8, 256, None) == _lib.BQ_ERR_SHAPE
    assert g(bq.Q8_0, FAKE, FAKE, FAKE, FAKE, float("nan"), FAKE, 8, 256, None) == \
        _lib.BQ_ERR_SHAPE
    assert g(7, FAKE, FAKE, FAKE, None, 0.0, FAKE, 8, 256, None) == _lib.BQ_ERR_QTYPE
    assert g(bq.Q4_0, FAKE, FAKE, FAKE, FAKE, 1e-6, FAKE, 0, 256, None) == _lib.BQ_OK


def test_pack_validation(lib):
    p = lib.bq_quantize_pack
    assert p(bq.Q8_0, None, 4, 64, FAKE, None) == _lib.BQ_ERR_NULL
    assert p(bq.Q8_0, FAKE, 4, 64, None, None) == _lib.BQ_ERR_NULL
    assert p(bq.Q8_0, FAKE, 4, 40, FAKE, None) == _lib.BQ_ERR_SHAPE
    assert p(bq.Q8_0, ctypes.c_void_p(0x10001), 4, 64, FAKE, None) == _lib.BQ_ERR_ALIGN
    assert p(bq.Q8_0, FAKE, 4, 64, MIS, None) == _lib.BQ_ERR_ALIGN
    assert p(1, FAKE, 4, 64, FAKE, None) == _lib.BQ_ERR_QTYPE
    assert p(bq.Q4_0, FAKE, 0, 64, FAKE, None) == _lib.BQ_OK


def test_python_binding_refuses_cpu_tensors():
    import torch

    W = torch.zeros(4, 64)
    with pytest.raises(ValueError, match="CUDA"):
        bq.quantize_pack(W, "q8_0")
    with pytest.raises(TypeError):
        bq.gemv_q8_0(torch.zeros(4, 68, dtype=torch.int8), torch.zeros(64))


def test_noalloc_entry_rejects_before_touching_the_device(lib):
    ops = (_lib.BqOp * 2)()
    assert lib.bq_stream_run_noalloc(bq.Q8_0, ops, 0, None) == _lib.BQ_ERR_SHAPE
    assert lib.bq_stream_run_noalloc(bq.Q8_0, None, 1, None) == _lib.BQ_ERR_NULL
    assert lib.bq_stream_run_noalloc(3, ops, 1, None) == _lib.BQ_ERR_QTYPE
    big = (_lib.BqOp * (_lib.BQ_NOALLOC_MAX_OPS + 1))()
    assert lib.bq_stream_run_noalloc(bq.Q4_0, big, len(big), None) == _lib.BQ_ERR_SHAPE


def test_qkv_bias_validation(lib):
    f = lib.bq_gemv_qkv_bias
    assert f(bq.Q8_0, None, FAKE, FAKE, FAKE, 8, 256, None) == _lib.BQ_ERR_NULL
    assert f(bq.Q8_0, FAKE, None, FAKE, FAKE, 8, 256, None) == _lib.BQ_ERR_NULL
    assert f(bq.Q8_0, FAKE, FAKE, FAKE, None, 8, 256, None) == _lib.BQ_ERR_NULL
    assert f(bq.Q4_0, FAKE, FAKE, ctypes.c_void_p(0x10002), FAKE, 8, 256, None) == \
        _lib.BQ_ERR_ALIGN
    assert f(bq.Q4_0, FAKE, FAKE, FAKE, FAKE, 8, 40, None) == _lib.BQ_ERR_SHAPE
    assert f(6, FAKE, FAKE, FAKE, FAKE, 8, 256, None) == _lib.BQ_ERR_QTYPE
    assert f(bq.Q8_0, None, None, None, None, 0, 256, None) == _lib.BQ_OK


def test_stream_plan_rejects_bias_on_gate_up_and_misaligned_bias(lib):
    ops = (_lib.BqOp * 1)()
    o = ops[0]
    o.kind, o.stage, o.M, o.K = _lib.BQ_OP_GATE_UP_SILU, 0, 64, 256
    o.W, o.W_up, o.x, o.y, o.eps = 0x10000, 0x20000, 0x30000, 0x40000, 1e-6
    o.bias = 0x50000
    plan = ctypes.c_void_p()
    ws = ctypes.c_void_p(0x100000)
    assert lib.bq_stream_plan_create(bq.Q8_0, ops, 1, ws, 1 << 20, ctypes.byref(plan)) == \
        _lib.BQ_ERR_SHAPE
    o.kind, o.bias = _lib.BQ_OP_GEMV, 0x50002
    assert lib.bq_stream_plan_create(bq.Q8_0, ops, 1, ws, 1 << 20, ctypes.byref(plan)) == \
        _lib.BQ_ERR_ALIGN


def test_stream_plan_tune_validation(lib):
    """A null plan is rejected before any CUDA call; the round count is
    checked on a real plan in the GPU tests."""
    assert lib.bq_stream_plan_tune(None, 3, None) == _lib.BQ_ERR_NULL
    assert lib.bq_stream_workspace_bytes(169, 113) >= 169 * 64 + (1024 + 1) * 4 + 1024 * 8


def test_stream_workspace_covers_staged_plans(lib):
    """A plan of dependent stages runs one launch per stage: the workspace
    holds the op table and one CTA split (up to 1024 CTAs + 1 entries) per
    stage, so it grows with the stage count; bad counts are refused."""
    n_ops = 113
    small = lib.bq_stream_workspace_bytes(n_ops, 1)
    for n_stages in (2, 29, 113):
        need = lib.bq_stream_workspace_bytes(n_ops, n_stages)
        assert need >= n_stages * (1024 + 1) * 4
        assert need >= small
    assert lib.bq_stream_workspace_bytes(4, 5) == -1  # more stages than ops
    assert lib.bq_stream_workspace_bytes(0, 0) == -1
    lib.bq_stream_plan_launches.restype = ctypes.c_int
    lib.bq_stream_plan_launches.argtypes = [ctypes.c_void_p]
    assert lib.bq_stream_plan_launches(None) == -1


def test_f16_gemv_validation(lib):
    f = lib.bq_gemv_f16
    assert f(None, FAKE, FAKE, 8, 256, None) == _lib.BQ_ERR_NULL
    assert f(FAKE, None, FAKE, 8, 256, None) == _lib.BQ_ERR_NULL
    assert f(FAKE, FAKE, None, 8, 256, None) == _lib.BQ_ERR_NULL
    assert f(ctypes.c_void_p(0x10008), FAKE, FAKE, 8, 256, None) == _lib.BQ_ERR_ALIGN
    assert f(FAKE, ctypes.c_void_p(0x10004), FAKE, 8, 256, None) == _lib.BQ_ERR_ALIGN
    assert f(FAKE, FAKE, FAKE, 8, 260, None) == _lib.BQ_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, 8, 0, None) == _lib.BQ_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, 8, (1 << 18) + 8, None) == _lib.BQ_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, -1, 256, None) == _lib.BQ_ERR_SHAPE
    assert f(None, None, None, 0, 256, None) == _lib.BQ_OK


def test_f16_gemv_f16out_validation(lib):
    f = lib.bq_gemv_f16_f16out
    assert f(None, FAKE, FAKE, 8, 256, None) == _lib.BQ_ERR_NULL
    assert f(FAKE, None, FAKE, 8, 256, None) == _lib.BQ_ERR_NULL
    assert f(FAKE, FAKE, None, 8, 256, None) == _lib.BQ_ERR_NULL
    assert f(ctypes.c_void_p(0x10008), FAKE, FAKE, 8, 256, None) == _lib.BQ_ERR_ALIGN
    assert f(FAKE, ctypes.c_void_p(0x10004), FAKE, 8, 256, None) == _lib.BQ_ERR_ALIGN
    assert f(FAKE, FAKE, ctypes.c_void_p(0x10001), 8, 256, None) == _lib.BQ_ERR_ALIGN
    assert f(FAKE, FAKE, FAKE, 8, 260, None) == _lib.BQ_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, 8, 0, None) == _lib.BQ_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, 8, (1 << 18) + 8, None) == _lib.BQ_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, -1, 256, None) == _lib.BQ_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, 1 << 31, 256, None) == _lib.BQ_ERR_SHAPE
    assert f(None, None, None, 0, 256, None) == _lib.BQ_OK


def test_failure_detection_hooks_exist_and_reject_no_plan(lib):
    """The internal hooks a GPU test uses to make a stage barrier's bounded
    wait run out (not part of the public header)."""
    hook = lib.bq_internal_plan_barrier_extra
    hook.argtypes = [ctypes.c_void_p, ctypes.c_uint, ctypes.c_ulonglong]
    hook.restype = ctypes.c_int
    assert hook(None, 1, 1_000_000) == -1
    assert lib.bq_internal_set_wait_limit_ns is not None
