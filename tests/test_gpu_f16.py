"""The unquantized fp16-weight GEMV (bq_gemv_f16) against the oracle: the
1e-5 * sum|w x| bound on random weights over shapes that span one and many
segment groups and ragged tails, exact results where every product and sum is
exact (dyadic weights with small-integer x, one-hot x, the identity, x = 0),
bit-reproducibility, sampled rows of an LM-head-sized matrix, the split-K
kernel against the warp-per-row kernel, and the fp16-output call
(bq_gemv_f16_f16out) against the rounding of the fp32 result."""
import numpy as np
import pytest
import torch

import block_quantized_weight_dequant_gb300 as bq
from block_quantized_weight_dequant_gb300 import workloads as wl

import oracle
from tolerance import assert_gemv_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def f16_weights(M, K, seed, stream):
    return wl.normal_np((M, K), wl.W_STD, seed=seed, stream=stream).astype(np.float16)


def run(W16, x):
    return bq.gemv_f16(torch.from_numpy(W16).to(DEV), torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)).cpu().numpy()


# K: one segment, a ragged tail, whole 256-element segments, one and several
# 16-segment groups with a tail, the largest K
SHAPES = [(1, 8), (3, 24), (7, 264), (33, 1000), (64, 1024), (129, 4104), (17, 18944),
          (5, 65544), (2, 262144)]


@pytest.mark.parametrize("M,K", SHAPES)
def test_f16_gemv_within_bound(M, K):
    o = oracle.get()
    W = f16_weights(M, K, 0, 61)
    x = wl.normal_np(K, 1.0, seed=0, stream=62)
    y = run(W, x)
    y_ref, S = o.gemv_f16(W.view(np.uint16), x.astype(np.float64))
    assert_gemv_close(y, y_ref, S, f"f16 gemv {M}x{K}")


@pytest.mark.parametrize("K", [40, 1024, 4104])
def test_f16_gemv_exact_cases(K):
    o = oracle.get()
    rng = np.random.default_rng(K)
    M = 23
    # dyadic weights k/8 and small-integer x: every product and partial sum
    # is exact in fp32, so the result equals the exact value
    ints = rng.integers(-40, 41, size=(M, K))
    W = (ints / 8.0).astype(np.float16)
    x = rng.integers(-3, 4, size=K).astype(np.float32)
    y = run(W, x)
    y_ref, _ = o.gemv_f16(W.view(np.uint16), x.astype(np.float64))
    assert np.array_equal(y.astype(np.float64), y_ref)
    Wr = f16_weights(M, K, 1, 63)
    for k in (0, K // 2, K - 1):
        e = np.zeros(K, dtype=np.float32)
        e[k] = 1.0
        assert np.array_equal(run(Wr, e), Wr[:, k].astype(np.float32)), f"column {k}"
    assert not run(Wr, np.zeros(K, dtype=np.float32)).any()
    I = np.eye(K, dtype=np.float16)
    xr = wl.normal_np(K, 1.0, seed=2, stream=64)
    assert np.array_equal(run(I, xr), xr)


def test_f16_gemv_is_bit_reproducible():
    W = torch.from_numpy(f16_weights(300, 3072, 3, 65)).to(DEV)
    x = torch.from_numpy(wl.normal_np(3072, 1.0, seed=3, stream=66)).to(DEV)
    a = bq.gemv_f16(W, x)
    b = bq.gemv_f16(W, x)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_f16_gemv_lm_head_sampled_rows():
    """A Qwen3-0.6B-shaped LM head kept in fp16 (151936 x 1024): every
    997th row plus the first and last, against the oracle row by row."""
    o = oracle.get()
    M, K = 151936, 1024
    W = (torch.randn(M, K, device=DEV, generator=torch.Generator(DEV).manual_seed(7)) *
         wl.W_STD).to(torch.float16)
    x = torch.from_numpy(wl.normal_np(K, 1.0, seed=4, stream=67)).to(DEV)
    y = bq.gemv_f16(W, x).cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(0, M, 997), [M - 1]]))
    Wr = W[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    y_ref, S = o.gemv_f16(Wr.view(np.uint16), x.cpu().numpy().astype(np.float64))
    assert_gemv_close(y[rows], y_ref, S, "f16 LM head rows")
    assert bq.device_status(clear=True) == 0


def test_f16_gemv_split_k_rows_match_warp_per_row_rows():
    """The launcher splits K across a CTA's warps when there are fewer than 16
    rows per SM and K spans two or more 4096-element groups.  Rows taken out
    of a matrix large enough for the warp-per-row kernel give the same bits
    on their own (split K), because the tree depends on K alone."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    M = nsm * 16 + 5
    for K in (4104, 20000, 262144):
        W = (torch.randn(M, K, device=DEV, generator=torch.Generator(DEV).manual_seed(K)) *
             wl.W_STD).to(torch.float16)
        x = torch.from_numpy(wl.normal_np(K, 1.0, seed=5, stream=68)).to(DEV)
        y_all = bq.gemv_f16(W, x)
        for r0, m in ((0, 7), (1000, 9), (M - 1, 1)):
            y = bq.gemv_f16(W[r0:r0 + m], x)
            assert torch.equal(y.view(torch.int32), y_all[r0:r0 + m].view(torch.int32)), (K, r0)
        o = oracle.get()
        y_ref, S = o.gemv_f16(W[:7].cpu().numpy().view(np.uint16), x.cpu().numpy().astype(np.float64))
        assert_gemv_close(y_all[:7].cpu().numpy(), y_ref, S, f"f16 gemv K={K}")
        del W
    assert bq.device_status(clear=True) == 0


@pytest.mark.parametrize("M,K", [(5, 1000), (40, 9000), (3000, 1024), (2600, 8200)])
def test_f16_output_is_the_fp32_result_rounded(M, K):
    """bq_gemv_f16_f16out: every output is the fp32 call's value rounded to
    nearest even in binary16 (numpy's conversion), for both kernels."""
    W = torch.from_numpy(f16_weights(M, K, 4, 69)).to(DEV)
    x = torch.from_numpy(wl.normal_np(K, 1.0, seed=6, stream=70)).to(DEV)
    y32 = bq.gemv_f16(W, x).cpu().numpy()
    y16 = bq.gemv_f16(W, x, out_dtype=torch.float16)
    assert y16.dtype == torch.float16
    assert np.array_equal(y16.cpu().numpy().view(np.uint16), y32.astype(np.float16).view(np.uint16))
    y16b = torch.empty(M, dtype=torch.float16, device=DEV)
    assert bq.gemv_f16(W, x, y16b) is y16b and torch.equal(y16b.view(torch.int16), y16.view(torch.int16))


def test_f16_output_rounding_edges():
    """Identity weights pass x through exactly in fp32; the fp16 output then
    shows the rounding: ties to even, the overflow threshold 65520 to inf,
    the largest finite value, subnormals, a half-subnormal tie to 0."""
    vals = np.array([65520.0, -65520.0, 65519.996, 65504.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                     2.0 ** -25, 3 * 2.0 ** -26, 1e-8, 1.0 / 3.0, -2.5e-5, 7.0], dtype=np.float32)
    K = 16
    x = np.zeros(K, dtype=np.float32)
    x[:len(vals)] = vals
    I = torch.eye(K, dtype=torch.float16, device=DEV)
    xd = torch.from_numpy(x).to(DEV)
    y32 = bq.gemv_f16(I, xd).cpu().numpy()
    assert np.array_equal(y32[:len(vals)], vals)
    y16 = bq.gemv_f16(I, xd, out_dtype=torch.float16).cpu().numpy()
    with np.errstate(over="ignore"):
        want = y32.astype(np.float16)
    assert np.array_equal(y16.view(np.uint16), want.view(np.uint16))
    assert np.isposinf(y16[0]) and np.isneginf(y16[1]) and y16[3] == 65504.0
    assert y16[4] == 1.0 and y16[5] == 1.0 + 2.0 ** -9 and y16[6] == 0.0
