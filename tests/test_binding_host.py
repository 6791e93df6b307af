"""The Python binding has no CPU path: on the CPU (no GPU needed) every
compute function refuses CPU tensors before it touches the library, so a
missing GPU or extension can never turn into a silent fallback."""
import pytest
import torch

import block_quantized_weight_dequant_gb300 as bq


class Untouchable:
    """stands in for the loaded library: any use of it fails the test"""

    def __init__(self):
        self.used = []

    def __getattr__(self, name):
        self.used.append(name)
        raise AssertionError(f"library entry point {name} reached with CPU tensors")


@pytest.fixture
def no_lib(monkeypatch):
    u = Untouchable()
    monkeypatch.setattr(bq, "lib", u)
    return u


K, M = 64, 4
u8 = dict(dtype=torch.uint8)


def packed(qt):
    return torch.zeros(M, (K // 32) * bq.BLOCK_BYTES[qt], **u8)


CALLS = {
    "quantize_pack": lambda: bq.quantize_pack(torch.zeros(M, K), "q8_0"),
    "gemv_q8_0": lambda: bq.gemv_q8_0(packed(bq.Q8_0), torch.zeros(K)),
    "gemv_q4_0": lambda: bq.gemv_q4_0(packed(bq.Q4_0), torch.zeros(K)),
    "gemv_gate_up_silu": lambda: bq.gemv_gate_up_silu("q8_0", packed(bq.Q8_0), packed(bq.Q8_0),
                                                      torch.zeros(K), torch.ones(K)),
    "gemv_qkv_bias": lambda: bq.gemv_qkv_bias("q4_0", packed(bq.Q4_0), torch.zeros(K), torch.zeros(M)),
    "gemv_verify": lambda: bq.gemv_verify("q8_0", packed(bq.Q8_0), torch.zeros(3, K)),
    "gemv_f16": lambda: bq.gemv_f16(torch.zeros(M, K, dtype=torch.float16), torch.zeros(K)),
    "gemv_f16 fp16 out": lambda: bq.gemv_f16(torch.zeros(M, K, dtype=torch.float16), torch.zeros(K),
                                             out_dtype=torch.float16),
    "StreamPlan": lambda: bq.StreamPlan("q8_0", [bq.StreamOp(0, packed(bq.Q8_0), torch.zeros(K),
                                                             torch.zeros(M))]),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_cpu_tensors_are_refused_before_the_library(no_lib, name):
    with pytest.raises(ValueError, match="no CPU path"):
        CALLS[name]()
    assert no_lib.used == []


def test_wrong_dtypes_are_refused(no_lib):
    with pytest.raises(TypeError):
        bq.gemv_f16(torch.zeros(M, K), torch.zeros(K))  # fp32 weights
    with pytest.raises(TypeError):
        bq.gemv_q8_0(torch.zeros(M, 68, dtype=torch.int8), torch.zeros(K))
    assert no_lib.used == []


def test_parity_sources_check_rows_and_shapes_on_the_host():
    """The full-size parity check draws a matrix's fp32 rows again from its
    seeded source: a row index outside the source, or a source that does not
    describe the packed matrix, is refused on the host before any gather runs
    on a device (an out-of-range device gather would fault)."""
    import sampled_parity as sp

    src = sp.WeightSource((8, 64), 0.02, 0, 5)
    assert src.rows([0, 7], "cpu").shape == (2, 64)
    with pytest.raises(IndexError):
        src.rows([0, 8], "cpu")
    with pytest.raises(IndexError):
        sp._take(torch.zeros(4), [4])
    with pytest.raises(ValueError):
        sp._need_source(src, torch.zeros((12, 36), dtype=torch.uint8), 64)
    sp._need_source(src, torch.zeros((8, 36), dtype=torch.uint8), 64)
