"""GPU parity for the Q4_K super-block format (RunIT README kernel table,
gemv_q4k_f16; "Quantization" table, Q4_K_M; the layout read from the public
GGUF definition, as in the oracle):

- packing: the GPU packer's bytes equal the oracle's, on weights with zero,
  all-positive, all-negative and widely scaled sub-blocks, and on the
  hand-derived golden example;
- GEMV: |y - y_ref| <= 1e-5 * SK per row, SK the oracle's sum over
  sub-blocks of d*sc*sum|q x| + dmin*m*sum|x| (the kernels evaluate each
  super-block as d*sc*sum(q x) - dmin*m*sum(x)); exactly equal where every
  partial sum is an exact dyadic (power-of-two scales, small-integer x);
- the row-mode and unit-per-lane paths, verify rows (memcmp against decode),
  gate+up+SiLU, q|k|v + bias, and the one-launch stream plans.
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
DEV = "cuda"
QK = oracle.Q4_K

SHAPES = [(1, 256), (7, 512), (33, 1024), (300, 1024), (130, 2048), (19, 3584), (9, 5120),
          (5, 18944), (40000, 1024), (6000, 3584), (37, 33024), (11, 65536), (3, 1 << 18)]


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def weights(M, K, seed):
    return oc._q4k_weights(np.random.default_rng([seed, M, K]), M, K)


def xvec(K, seed, R=None):
    shape = (K,) if R is None else (R, K)
    return wl.normal_np(shape, 1.0, seed=seed, stream=wl.stream_id("q4k x", K, R))


def ref(Pn, M, K, x):
    o = oracle.get()
    x = x.astype(np.float64)
    y, _ = o.gemv_parallel(QK, Pn, M, K, x)
    return y, o.q4_k_split_scale_parallel(Pn, M, K, x)


@pytest.mark.parametrize("M,K", [(1, 256), (7, 512), (33, 1024), (19, 3584), (5, 18944),
                                 (300, 1024), (3, 33024)])
def test_q4k_pack_bit_exact(M, K):
    W = weights(M, K, 1)
    got = bq.quantize_pack(cuda(W), "q4_k").cpu().numpy()
    want = oracle.get().quantize_pack_parallel(QK, W)
    bad = np.flatnonzero((got != want).any(axis=1))
    assert bad.size == 0, f"rows {bad[:5]} differ"
    # and on plain N(0, 0.02) weights
    W = wl.normal_np((M, K), wl.W_STD, seed=2, stream=wl.stream_id("q4k", M, K))
    assert np.array_equal(bq.quantize_pack(cuda(W), "q4_k").cpu().numpy(),
                          oracle.get().quantize_pack_parallel(QK, W))


def test_q4k_golden_example():
    g = oc.load_golden("q4_k_example_c.txt")
    P = bq.quantize_pack(cuda(g["w"]), "q4_k")
    assert np.array_equal(P.cpu().numpy(), g["packed"])
    y = bq.gemv("q4_k", P, torch.ones(g["K"], device=DEV)).cpu().numpy()
    assert y.tolist() == g["x_ones_y"]


@pytest.mark.parametrize("M,K", SHAPES)
def test_q4k_gemv_within_bound(M, K):
    P = bq.quantize_pack(cuda(weights(M, K, 3)), "q4_k")
    x = xvec(K, 3)
    y = torch.full((M,), float("nan"), device=DEV)
    bq.gemv_q4_k(P, cuda(x), y)
    y_ref, SK = ref(P.cpu().numpy(), M, K, x)
    assert_gemv_close(y.cpu().numpy(), y_ref, SK, f"q4_k {M}x{K}")


@pytest.mark.parametrize("M,K", [(1, 256), (33, 256), (9, 512), (70, 512), (5000, 512)])
def test_q4k_gemv_exact_on_dyadic_inputs(M, K):
    rng = np.random.default_rng([17, M, K])
    raw, *_ = oc._q4k_direct(rng, M, K)
    x = rng.integers(-2, 3, size=K).astype(np.float32)
    y = bq.gemv("q4_k", cuda(raw), cuda(x)).cpu().numpy().astype(np.float64)
    y_ref, _ = oracle.get().gemv(QK, raw, M, K, x.astype(np.float64))
    assert np.array_equal(y, y_ref)


def test_q4k_large_and_small_calls_agree_bitwise():
    M, K = 40000, 1024
    P = bq.quantize_pack(cuda(weights(M, K, 4)), "q4_k")
    x = cuda(xvec(K, 4))
    y = bq.gemv("q4_k", P, x)
    for r0 in (0, 777, M - 5):
        ys = bq.gemv("q4_k", P[r0:r0 + 5].contiguous(), x)
        assert torch.equal(ys.view(torch.int32), y[r0:r0 + 5].view(torch.int32)), f"rows {r0}.."


@pytest.mark.parametrize("M,K", [(300, 1024), (97, 5120), (40, 17408), (9, 18944), (7, 65536)])
@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6])
def test_q4k_verify_rows_memcmp_equal_to_decode(M, K, R):
    P = bq.quantize_pack(cuda(weights(M, K, 5)), "q4_k")
    X = xvec(K, 5, R=R)
    Y = bq.gemv_verify("q4_k", P, cuda(X)).cpu().numpy()
    Pn = P.cpu().numpy()
    for r in range(R):
        y1 = bq.gemv("q4_k", P, cuda(X[r])).cpu().numpy()
        assert Y[r].tobytes() == y1.tobytes(), f"row {r} differs from decode"
        y_ref, SK = ref(Pn, M, K, X[r])
        assert_gemv_close(Y[r], y_ref, SK, f"verify q4_k {M}x{K} R={R} row {r}")


@pytest.mark.parametrize("use_gamma", [True, False])
@pytest.mark.parametrize("M,K", [(3072, 1024), (77, 256), (33, 3584), (40000, 1024), (9, 65536)])
def test_q4k_gate_up_silu_within_bound(use_gamma, M, K):
    Pg = bq.quantize_pack(cuda(weights(M, K, 6)), "q4_k")
    Pu = bq.quantize_pack(cuda(weights(M, K, 7)), "q4_k")
    x = xvec(K, 6)
    gamma = wl.normal_np(K, 0.1, seed=6, stream=wl.stream_id("gamma", K), mean=1.0)
    y = bq.gemv_gate_up_silu("q4_k", Pg, Pu, cuda(x), cuda(gamma) if use_gamma else None,
                             1e-6).cpu().numpy()
    o = oracle.get()
    xn = o.rmsnorm(x, gamma, 1e-6) if use_gamma else x.astype(np.float64)
    Pgn, Pun = Pg.cpu().numpy(), Pu.cpu().numpy()
    r = o.gate_up_silu(QK, Pgn, Pun, M, K, xn)
    # the bound's sums for the split evaluation of each product
    r["Sg"] = o.q4_k_split_scale_parallel(Pgn, M, K, xn)
    r["Su"] = o.q4_k_split_scale_parallel(Pun, M, K, xn)
    assert_gate_up_close(y, r, f"q4_k gate_up {M}x{K} gamma={use_gamma}")


def test_q4k_qkv_bias_is_gemv_plus_bias():
    K, M = 1024, 2048 + 2 * 512
    P = bq.quantize_pack(cuda(weights(M, K, 8)), "q4_k")
    x = cuda(xvec(K, 8))
    b = cuda(wl.normal_np(M, 0.5, seed=8, stream=wl.stream_id("q4k bias")))
    y = bq.gemv_qkv_bias("q4_k", P, x, b)
    assert torch.equal(y.view(torch.int32), (bq.gemv("q4_k", P, x) + b).view(torch.int32))


@pytest.mark.parametrize("chained", [True, False], ids=["chained", "independent"])
@pytest.mark.parametrize("hidden,q_dim,kv,inter,vocab", [(1024, 2048, 512, 3072, 5000),
                                                         (3584, 3584, 512, 18944, 3000)])
def test_q4k_stream_plan_matches_launch_per_op_bitwise(chained, hidden, q_dim, kv, inter, vocab):
    from block_quantized_weight_dequant_gb300.decode import DecodeStream

    def packed(M, K, *tag):
        W = wl.normal_torch((M, K), wl.W_STD, seed=9, stream=wl.stream_id("q4k", *tag), device=DEV)
        return bq.quantize_pack(W, "q4_k")

    layers = [dict(q=packed(q_dim, hidden, l, "q"), k=packed(kv, hidden, l, "k"),
                   v=packed(kv, hidden, l, "v"), o=packed(hidden, q_dim, l, "o"),
                   gate=packed(inter, hidden, l, "g"), up=packed(inter, hidden, l, "u"),
                   down=packed(hidden, inter, l, "d"),
                   gamma=wl.normal_torch(hidden, 0.1, seed=9, stream=wl.stream_id(l, "gm"),
                                         device=DEV, mean=1.0))
              for l in range(2)]
    ds = DecodeStream("q4_k", layers, packed(vocab, hidden, "lm"), chained=chained)
    ds.inputs.copy_(wl.normal_torch(ds.inputs.numel(), 1.0, seed=9, stream=5, device=DEV))
    ds.run_per_op()
    want = [op.y.clone() for op in ds.ops]
    for op in ds.ops:
        op.y.fill_(float("nan"))
    ds.plan()
    if not chained:
        ds.plan().tune(rounds=2)
    ds.run_plan()
    for i, (op, w) in enumerate(zip(ds.ops, want)):
        assert torch.equal(op.y.view(torch.int32), w.view(torch.int32)), f"op {i}"
    lm = ds.ops[-1]
    x = lm.x.cpu().numpy()
    y_ref, SK = ref(lm.W.cpu().numpy(), lm.y.numel(), x.size, x)
    assert_gemv_close(lm.y.cpu().numpy(), y_ref, SK, "q4_k stream lm head")
    assert bq.device_status(clear=True) == 0


def test_q4k_rejects_k_not_a_multiple_of_256():
    P = torch.zeros((4, 288 // 32 * 18), dtype=torch.uint8, device=DEV)
    with pytest.raises(bq.BQError):
        bq.gemv("q4_k", P, torch.zeros(288, device=DEV))
