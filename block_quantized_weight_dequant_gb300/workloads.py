"""Synthetic workloads: the shapes of the benchmark configurations and seeded
input generators.

This module holds none of the method's arithmetic.  It only draws fp32
N(mean, std) tensors from counter-seeded generators and lists matrix shapes,
so the tests, the benchmark and the oracle-side checks can all feed the same
inputs to the GPU library and to the oracle.

Shapes and value distributions stand in for the pages' real GGUF models
(Qwen3-0.6B Q8_0 in the EdgeRunner post, Qwen2.5-0.5B Q8_0 in the RunIT
README, a 27B 4-bit model in "We Wrote Our Own Inference Engine"), whose
weights are not available here: weights are N(0, 0.02), activations N(0, 1),
RMSNorm gains N(1, 0.1).
"""
import zlib

import numpy as np

W_STD = 0.02
X_STD = 1.0


def stream_id(*parts):
    """A stable 32-bit id for a named tensor, e.g. stream_id("cfg2", 3, "q")."""
    return zlib.crc32("/".join(str(p) for p in parts).encode())


def normal_np(shape, std=1.0, seed=0, stream=0, mean=0.0):
    """fp32 numpy N(mean, std) from a PCG64 generator keyed by (seed, stream)."""
    rng = np.random.default_rng([seed, stream])
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return a


def normal_torch(shape, std=1.0, seed=0, stream=0, mean=0.0, device="cuda"):
    """fp32 torch N(mean, std) drawn on `device` from a generator keyed by
    (seed, stream).  Used for full-size inputs too large to draw on the host."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed((seed * 0x9E3779B1 + stream) & 0x7FFFFFFFFFFFFFFF)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


# ---------------------------------------------------------------------------
# configurations
# ---------------------------------------------------------------------------
# 1. single Q8_0 GEMV
CFG1 = dict(name="q8_0 gemv 3072x1024", qtype="q8_0", M=3072, K=1024, seed=0)

# 2. Qwen3-0.6B-shaped per-token Q8_0 weight stream (28 layers + LM head)
QWEN3_0_6B = dict(name="qwen3-0.6b-shaped q8_0 token stream", qtype="q8_0", layers=28,
                  hidden=1024, mats=[("q", 2048, 1024), ("k", 512, 1024), ("v", 512, 1024),
                                     ("o", 1024, 2048), ("gate", 3072, 1024),
                                     ("up", 3072, 1024), ("down", 1024, 3072)],
                  lm_head=(151936, 1024))

# 3. 7B-shaped Q4_0 per-token stream
Q7B = dict(name="7b-shaped q4_0 token stream", qtype="q4_0", layers=28, hidden=3584,
           mats=[("q", 3584, 3584), ("k", 512, 3584), ("v", 512, 3584), ("o", 3584, 3584),
                 ("gate", 18944, 3584), ("up", 18944, 3584), ("down", 3584, 18944)],
           lm_head=(152064, 3584))

# 3k. the same 7B-shaped stream in the Q4_K super-block format (the RunIT
# README's Q4_K_M row; 0.5625 B per weight like Q4_0)
Q7B_K = dict(Q7B, name="7b-shaped q4_k token stream", qtype="q4_k")

# 4. RMSNorm input + gate/up + SiLU, Q8_0, 28 rotated pairs
CFG4 = dict(name="rmsnorm+gate_up_silu q8_0 3072x1024 x28", qtype="q8_0", M=3072, K=1024,
            pairs=28, eps=1e-6, gamma_mean=1.0, gamma_std=0.1)

# 5. 27B-scale Q4_0 multi-row verify
CFG5 = dict(name="q4_0 verify 17408x5120 + 5120x17408, R=1..6", qtype="q4_0",
            mats=[("a", 17408, 5120), ("b", 5120, 17408)], R=(1, 2, 3, 4, 5, 6))


# 6. Unquantized fp16-weight GEMV: a Qwen3-0.6B-shaped LM head kept in fp16
F16_LM = dict(name="fp16-weight gemv 151936x1024 (qwen3-0.6b-shaped lm head, unquantized)",
              M=151936, K=1024)


def token_stream_ops(cfg, fused_qkv=False):
    """Per-token op list in model order: ("gemv", name, M, K), ("gate_up",
    name, M, K) or, with fused_qkv, ("gemv_bias", name, M, K) for the q, k, v
    rows concatenated.  Gate and up share one fused RMSNorm+SiLU op."""
    ops = []
    mats = {name: (M, K) for name, M, K in cfg["mats"]}
    for layer in range(cfg["layers"]):
        if fused_qkv:
            K = mats["q"][1]
            ops.append(("gemv_bias", f"L{layer}.qkv", mats["q"][0] + mats["k"][0] + mats["v"][0], K))
        for name, M, K in cfg["mats"]:
            if name == "up" or (fused_qkv and name in ("q", "k", "v")):
                continue
            if name == "gate":
                ops.append(("gate_up", f"L{layer}.gate_up", M, K))
            else:
                ops.append(("gemv", f"L{layer}.{name}", M, K))
    M, K = cfg["lm_head"]
    ops.append(("gemv", "lm_head", M, K))
    return ops


def token_weight_shapes(cfg):
    """Every packed matrix of one token, in model order: (name, M, K)."""
    out = []
    for layer in range(cfg["layers"]):
        for name, M, K in cfg["mats"]:
            out.append((f"L{layer}.{name}", M, K))
    out.append(("lm_head",) + tuple(cfg["lm_head"]))
    return out
