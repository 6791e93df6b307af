"""GPU parity: the CUDA library (through its C ABI) against the oracle.

- packing: bit-exact bytes;
- GEMV, Q8_0 and Q4_0: |y - y_ref| <= 1e-5 * sum|w x| per row, and exactly
  equal wherever every partial sum is an exact dyadic (power-of-two scales
  with small-integer x, one-hot x, the worked examples);
- gate+up+SiLU: the propagated bound of tests/tolerance.py;
- verify: every row memcmp-equal to the single-row GEMV, and within the bound.
Shapes span several tiles with ragged tails, both kernels (K % 256 == 0 and
not), and the edge cases M = 0, M = 1, K = 32.
"""
import numpy as np
import pytest
import torch

import block_quantized_weight_dequant_gb300 as bq
from block_quantized_weight_dequant_gb300 import workloads as wl

import oracle
import oracle_checks as oc
from tolerance import assert_gate_up_close, assert_gemv_close

pytestmark = pytest.mark.gpu

QT = {"q8_0": oracle.Q8_0, "q4_0": oracle.Q4_0}
DEV = "cuda"

# (M, K): stream kernel (K % 256 == 0) with several tiles and ragged tails,
# and the generic kernel (K % 256 != 0)
SHAPES = [(1, 256), (7, 256), (33, 512), (64, 1024), (97, 1280), (300, 1024), (130, 2048),
          (40, 3072), (19, 3584), (9, 5120), (37, 17408), (5, 18944),
          (1, 32), (3, 96), (17, 288), (65, 544), (31, 1056), (2, 18976)]


def ora():
    return oracle.get()


def weights(M, K, seed, spread=True):
    """N(0, 0.02) weights; with `spread`, blocks scaled by 2^-30..2^7 (down to
    fp16-subnormal and zero scales), and one all-zero block."""
    w = wl.normal_np((M, K), wl.W_STD, seed=seed, stream=wl.stream_id("parity", M, K))
    if spread:
        rng = np.random.default_rng([seed, M, K])
        s = (2.0 ** rng.integers(-30, 8, size=(M, K // 32, 1))).astype(np.float32)
        w = (w.reshape(M, K // 32, 32) * s).reshape(M, K)
        w[0, :32] = 0.0
    return np.ascontiguousarray(w)


def xvec(K, seed, R=None):
    shape = (K,) if R is None else (R, K)
    return wl.normal_np(shape, wl.X_STD, seed=seed, stream=wl.stream_id("x", K, R))


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def gpu_pack(qt, W):
    return bq.quantize_pack(cuda(W), qt)


# ---------------------------------------------------------------------------
# packing
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("M,K", SHAPES)
def test_pack_bit_exact(qt, M, K):
    W = weights(M, K, seed=1)
    got = gpu_pack(qt, W).cpu().numpy()
    want = ora().quantize_pack(QT[qt], W)
    assert got.shape == want.shape
    bad = np.flatnonzero((got != want).any(axis=1))
    assert bad.size == 0, f"rows {bad[:5]} differ"


@pytest.mark.parametrize("name", oc.GOLDEN_FILES)
def test_pack_and_gemv_golden(name):
    g = oc.load_golden(name)
    qt = {oracle.Q8_0: "q8_0", oracle.Q4_0: "q4_0", oracle.Q4_K: "q4_k"}[g["qtype"]]
    P = gpu_pack(qt, g["w"])
    assert np.array_equal(P.cpu().numpy(), g["packed"])
    y = bq.gemv(qt, P, torch.ones(g["K"], device=DEV)).cpu().numpy()
    assert y.tolist() == g["x_ones_y"]


# ---------------------------------------------------------------------------
# GEMV
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("M,K", SHAPES)
def test_gemv_within_bound(qt, M, K):
    W = weights(M, K, seed=2)
    x = xvec(K, seed=2)
    P = gpu_pack(qt, W)
    y = torch.full((M,), float("nan"), device=DEV)  # every element must be written
    bq.gemv(qt, P, cuda(x), y)
    y_ref, S = ora().gemv(QT[qt], P.cpu().numpy(), M, K, x.astype(np.float64))
    assert_gemv_close(y.cpu().numpy(), y_ref, S, f"{qt} {M}x{K}")


# Large M: enough warp tiles per SM that single calls take the unit-per-lane
# path of the streaming kernel (the small shapes above take row mode).
LARGE = [(40000, 1024), (24000, 2048), (6000, 5120)]


@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("M,K", LARGE)
def test_gemv_large_m_within_bound(qt, M, K):
    W = weights(M, K, seed=12)
    x = xvec(K, seed=12)
    P = gpu_pack(qt, W)
    y = torch.full((M,), float("nan"), device=DEV)
    bq.gemv(qt, P, cuda(x), y)
    y_ref, S = ora().gemv(QT[qt], P.cpu().numpy(), M, K, x.astype(np.float64))
    assert_gemv_close(y.cpu().numpy(), y_ref, S, f"{qt} {M}x{K}")


@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
def test_large_and_small_calls_agree_bitwise(qt):
    """Rows evaluated by the unit-per-lane path (a large call) and by row
    mode (a call over a few of the same rows) give the same bits."""
    M, K = 40000, 1024
    P = gpu_pack(qt, weights(M, K, seed=13))
    x = cuda(xvec(K, seed=13))
    y = bq.gemv(qt, P, x)
    for r0 in (0, 777, M - 5):
        ys = bq.gemv(qt, P[r0:r0 + 5].contiguous(), x)
        assert torch.equal(ys.view(torch.int32), y[r0:r0 + 5].view(torch.int32)), f"rows {r0}.."


@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
def test_gate_up_large_m_within_bound(qt):
    M, K = 40000, 1024
    Wg, Wu = weights(M, K, seed=14, spread=False), weights(M, K, seed=15, spread=False)
    x = xvec(K, seed=14)
    gamma = wl.normal_np(K, 0.1, seed=14, stream=wl.stream_id("gamma", K), mean=1.0)
    Pg, Pu = gpu_pack(qt, Wg), gpu_pack(qt, Wu)
    y = bq.gemv_gate_up_silu(qt, Pg, Pu, cuda(x), cuda(gamma), 1e-6).cpu().numpy()
    o = ora()
    r = o.gate_up_silu(QT[qt], Pg.cpu().numpy(), Pu.cpu().numpy(), M, K, o.rmsnorm(x, gamma, 1e-6))
    assert_gate_up_close(y, r, f"{qt} {M}x{K} large")


@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("M,K", [(33, 256), (9, 288), (70, 1024), (5, 1056), (11, 2048)])
def test_gemv_exact_on_dyadic_inputs(qt, M, K):
    rng = np.random.default_rng([7, M, K])
    raw, dsel = oc._direct_blocks(rng, QT[qt], M, K)
    x = rng.integers(-2, 3, size=K).astype(np.float32)
    y = bq.gemv(qt, cuda(raw), cuda(x)).cpu().numpy().astype(np.float64)
    y_ref, _ = ora().gemv(QT[qt], raw, M, K, x.astype(np.float64))
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("K", [256, 1024, 1056])
def test_gemv_one_hot_gives_exact_columns(qt, K):
    M = 50
    P = gpu_pack(qt, weights(M, K, seed=3))
    deq = oc.dequant_independent(QT[qt], P.cpu().numpy(), M, K)
    for k in (0, 1, 33, K // 2 + 5, K - 1):
        x = torch.zeros(K, device=DEV)
        x[k] = 1.0
        y = bq.gemv(qt, P, x).cpu().numpy().astype(np.float64)
        assert np.array_equal(y, deq[:, k]), f"column {k}"


def test_gemv_empty_rows_is_noop():
    P = torch.zeros((0, 34 * 8), dtype=torch.uint8, device=DEV)
    y = torch.full((4,), 7.0, device=DEV)
    bq.gemv_q8_0(P, torch.ones(256, device=DEV), y[:0])
    torch.cuda.synchronize()
    assert y.tolist() == [7.0] * 4


# ---------------------------------------------------------------------------
# gate + up + SiLU
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("use_gamma", [True, False])
@pytest.mark.parametrize("M,K", [(3072, 1024), (77, 256), (130, 2048), (33, 3584), (13, 288),
                                 (5, 1056)])
def test_gate_up_silu_within_bound(qt, use_gamma, M, K):
    Wg, Wu = weights(M, K, seed=4, spread=False), weights(M, K, seed=5, spread=False)
    x = xvec(K, seed=4)
    gamma = wl.normal_np(K, 0.1, seed=4, stream=wl.stream_id("gamma", K), mean=1.0)
    Pg, Pu = gpu_pack(qt, Wg), gpu_pack(qt, Wu)
    y = bq.gemv_gate_up_silu(qt, Pg, Pu, cuda(x), cuda(gamma) if use_gamma else None,
                             1e-6).cpu().numpy()
    o = ora()
    xn = o.rmsnorm(x, gamma, 1e-6) if use_gamma else x.astype(np.float64)
    r = o.gate_up_silu(QT[qt], Pg.cpu().numpy(), Pu.cpu().numpy(), M, K, xn)
    assert_gate_up_close(y, r, f"{qt} {M}x{K} gamma={use_gamma}")


def test_gate_up_without_gamma_matches_plain_gemv_bits():
    """With no RMSNorm the gate/up operands are the plain GEMV's, bit for bit."""
    M, K = 200, 1024
    Pg, Pu = gpu_pack("q8_0", weights(M, K, 8)), gpu_pack("q8_0", weights(M, K, 9))
    x = cuda(xvec(K, 8))
    y = bq.gemv_gate_up_silu("q8_0", Pg, Pu, x, None).cpu().numpy()
    g = bq.gemv_q8_0(Pg, x).cpu().numpy()
    u = bq.gemv_q8_0(Pu, x).cpu().numpy()
    want = (torch.from_numpy(g) / (1 + torch.exp(-torch.from_numpy(g))) * torch.from_numpy(u))
    assert np.allclose(y, want.numpy(), rtol=2e-6, atol=0)


# ---------------------------------------------------------------------------
# fused q|k|v + bias
# ---------------------------------------------------------------------------
# (K, q rows, k = v rows): Qwen2.5-0.5B (K = 896 takes the generic kernel),
# Qwen3-0.6B-like, 7B-like, and a large concatenation (unit-per-lane path)
QKV = [(896, 896, 128), (1024, 2048, 512), (3584, 3584, 512), (1024, 38000, 1000)]


@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("K,Mq,Mkv", QKV)
def test_qkv_bias_is_gemv_plus_bias_and_within_bound(qt, K, Mq, Mkv):
    Ps = [gpu_pack(qt, weights(M, K, seed=21 + i, spread=False))
          for i, M in enumerate((Mq, Mkv, Mkv))]
    P = bq.concat_packed(Ps)
    M = Mq + 2 * Mkv
    x = xvec(K, seed=21)
    bias = wl.normal_np(M, 0.5, seed=21, stream=wl.stream_id("qkv_bias", M, K))
    xc, bc = cuda(x), cuda(bias)
    y = bq.gemv_qkv_bias(qt, P, xc, bc)
    # the single-row GEMV's dot products, then one IEEE fp32 add
    want = bq.gemv(qt, P, xc) + bc
    assert torch.equal(y.view(torch.int32), want.view(torch.int32))
    # concatenation changes nothing: each part is its own GEMV plus its bias
    r0 = 0
    for Pi in Ps:
        Mi = Pi.shape[0]
        yi = bq.gemv_qkv_bias(qt, Pi, xc, bc[r0:r0 + Mi].contiguous())
        assert torch.equal(yi.view(torch.int32), y[r0:r0 + Mi].view(torch.int32))
        r0 += Mi
    y_ref, S = ora().gemv_bias(QT[qt], P.cpu().numpy(), M, K, x.astype(np.float64),
                               bias.astype(np.float64))
    assert_gemv_close(y.cpu().numpy(), y_ref, S, f"qkv+bias {qt} K={K}")
    # no bias: the plain GEMV, bit for bit
    y0 = bq.gemv_qkv_bias(qt, P, xc, None)
    assert torch.equal(y0.view(torch.int32), bq.gemv(qt, P, xc).view(torch.int32))


# ---------------------------------------------------------------------------
# multi-row verify
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("qt", ["q4_0", "q8_0"])
@pytest.mark.parametrize("M,K", [(300, 1024), (97, 5120), (40, 17408), (17, 288), (9, 1056)])
@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6])
def test_verify_rows_memcmp_equal_to_decode(qt, M, K, R):
    P = gpu_pack(qt, weights(M, K, seed=6))
    X = xvec(K, seed=6, R=R)
    Y = bq.gemv_verify(qt, P, cuda(X)).cpu().numpy()
    Pn = P.cpu().numpy()
    for r in range(R):
        y1 = bq.gemv(qt, P, cuda(X[r])).cpu().numpy()
        assert Y[r].tobytes() == y1.tobytes(), f"row {r} differs from decode"
        y_ref, S = ora().gemv(QT[qt], Pn, M, K, X[r].astype(np.float64))
        assert_gemv_close(Y[r], y_ref, S, f"verify {qt} {M}x{K} R={R} row {r}")


@pytest.mark.parametrize("qt", ["q4_0", "q8_0"])
@pytest.mark.parametrize("R", [2, 3, 5])
def test_panel_verify_several_tiles_per_warp(qt, R):
    """An R x K input over the staging limit (128 KB of fp32) is cut into
    K-panels; with more tiles than the GPU holds warps, a warp walks several
    tiles through each panel and parks their partial sums in shared memory
    between panels.  Every row stays memcmp-equal to decode; sampled rows are
    within the oracle bound."""
    M, K = 10000, 17408
    P = gpu_pack(qt, weights(M, K, seed=35, spread=False))
    X = xvec(K, seed=35, R=R)
    Y = bq.gemv_verify(qt, P, cuda(X)).cpu().numpy()
    Pn = P.cpu().numpy()
    rng = np.random.default_rng([35, R])
    idx = np.unique(np.r_[0, M - 1, rng.choice(M, 30, replace=False)])
    Ps = np.ascontiguousarray(Pn[idx])
    for r in range(R):
        y1 = bq.gemv(qt, P, cuda(X[r])).cpu().numpy()
        assert Y[r].tobytes() == y1.tobytes(), f"row {r} differs from decode"
        y_ref, S = ora().gemv(QT[qt], Ps, len(idx), K, X[r].astype(np.float64))
        assert_gemv_close(Y[r][idx], y_ref, S, f"panel verify {qt} {M}x{K} R={R} row {r}")


# ---------------------------------------------------------------------------
# K beyond what the streaming kernel stages in shared memory for one input row
# (32768 fp32): the documented range goes to K = 2^18 for every quantized call
# ---------------------------------------------------------------------------
LONG_K = [33024, 65536, 1 << 18]


@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("K", LONG_K)
def test_long_k_gemv_and_qkv_bias(qt, K):
    M = 37
    P = gpu_pack(qt, weights(M, K, seed=31))
    x = xvec(K, seed=31)
    y = torch.full((M,), float("nan"), device=DEV)
    bq.gemv(qt, P, cuda(x), y)
    Pn = P.cpu().numpy()
    y_ref, S = ora().gemv(QT[qt], Pn, M, K, x.astype(np.float64))
    assert_gemv_close(y.cpu().numpy(), y_ref, S, f"{qt} gemv {M}x{K}")
    bias = wl.normal_np(M, 0.5, seed=31, stream=wl.stream_id("long-k bias", K))
    yb = bq.gemv_qkv_bias(qt, P, cuda(x), cuda(bias))
    assert torch.equal(yb.view(torch.int32), (y + cuda(bias)).view(torch.int32))
    y_ref, S = ora().gemv_bias(QT[qt], Pn, M, K, x.astype(np.float64), bias.astype(np.float64))
    assert_gemv_close(yb.cpu().numpy(), y_ref, S, f"{qt} qkv_bias {M}x{K}")


@pytest.mark.parametrize("qt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("K", LONG_K)
def test_long_k_gate_up_silu(qt, K):
    M = 21
    Pg = gpu_pack(qt, weights(M, K, seed=32, spread=False))
    Pu = gpu_pack(qt, weights(M, K, seed=33, spread=False))
    x = xvec(K, seed=32)
    gamma = wl.normal_np(K, 0.1, seed=32, stream=wl.stream_id("gamma", K), mean=1.0)
    o = ora()
    for g in (gamma, None):
        y = bq.gemv_gate_up_silu(qt, Pg, Pu, cuda(x), None if g is None else cuda(g),
                                 1e-6).cpu().numpy()
        xn = o.rmsnorm(x, g, 1e-6) if g is not None else x.astype(np.float64)
        r = o.gate_up_silu(QT[qt], Pg.cpu().numpy(), Pu.cpu().numpy(), M, K, xn)
        assert_gate_up_close(y, r, f"{qt} gate_up {M}x{K} gamma={g is not None}")


@pytest.mark.parametrize("qt", ["q4_0", "q8_0"])
@pytest.mark.parametrize("K", [65536, 1 << 18])
def test_long_k_verify_memcmp_equal_to_decode(qt, K):
    M = 19
    P = gpu_pack(qt, weights(M, K, seed=34))
    X = xvec(K, seed=34, R=6)
    Pn = P.cpu().numpy()
    for R in range(1, 7):
        Y = bq.gemv_verify(qt, P, cuda(X[:R])).cpu().numpy()
        for r in range(R):
            y1 = bq.gemv(qt, P, cuda(X[r])).cpu().numpy()
            assert Y[r].tobytes() == y1.tobytes(), f"R={R} row {r} differs from decode"
    for r in range(6):
        y_ref, S = ora().gemv(QT[qt], Pn, M, K, X[r].astype(np.float64))
        assert_gemv_close(Y[r], y_ref, S, f"verify {qt} {M}x{K} row {r}")


def test_no_device_errors_recorded():
    assert bq.device_status(clear=True) == 0
