#!/usr/bin/env python3
"""Benchmark: achieved HBM GB/s and per-token weight-stream tok/s at batch 1.

Default workload (a "step" = one token of the Qwen3-0.6B-shaped Q8_0 weight
stream): 28 layers of q 2048x1024, k 512x1024, v 512x1024, o 1024x2048,
gate+up 3072x1024 (fused RMSNorm+gate+up+SiLU), down 1024x3072, then the LM
head 151936x1024: 169 ops, 197 GEMVs, 602 MB of packed weights.  Every op
reads an N(0, 1) input of its own (--inputs independent), so the step is the
pure per-token weight stream; the whole step is one launch of the multi-op
streaming kernel, captured once in a CUDA graph and replayed.  The same
weights are also timed with each stage reading the previous stage's output
(113 dependent stages, one cooperative launch of the stream executor with
grid-wide barriers) and reported under "other_inputs"; --inputs chained swaps
the two.  --launch per_op: one launch per op instead.  Weights N(0, 0.02)
packed to Q8_0 on the GPU, inputs N(0, 1), RMSNorm gains N(1, 0.1), all
seeded and synthetic (the pages' real checkpoints are not available).  The
packed weights (602 MB) are larger than the 129 MB L2, so every step reads
them from HBM; no flush is needed.

Other workloads (--config): cfg1 (one Q8_0 GEMV 3072x1024, 96 rotated
copies), cfg3 (7B-shaped Q4_0 token stream), cfg4 (RMSNorm+gate+up+SiLU Q8_0
3072x1024, 28 rotated pairs), cfg5 (Q4_0 verify 17408x5120 + 5120x17408,
--rows R, 7 rotated copies of each).

Prints ONE JSON line (rank 0).  --impl reference times the oracle (the plain
C fp64 CPU statement of the same product) on the host cores instead.
Multi-GPU (torchrun): independent replicas, one per GPU, no collective on the
data path; value = bytes of all ranks / max time over ranks.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (% of GB300 peak) and per-token weight-stream tok/s, batch 1"
NOMINAL_HBM_GBS = 8000.0
CFG1_COPIES = 96   # rotated weight copies: 321 MB per sweep, 2.5x the 129 MB L2
CFG5_COPIES = 7    # of each verify matrix: 702 MB per sweep
FALLBACK_HBM_GBS = 6800.0
# per-token weight streams: cfg2 (Qwen3-0.6B-shaped Q8_0), cfg3 (7B-shaped
# Q4_0) and cfg3k (the 7B-shaped stream in Q4_K super-blocks)
TOKEN_CONFIGS = ("cfg2", "cfg3", "cfg3k")


def token_cfg(config):
    from block_quantized_weight_dequant_gb300 import workloads as wl
    return dict({"cfg2": wl.QWEN3_0_6B, "cfg3": wl.Q7B, "cfg3k": wl.Q7B_K}[config])


# ---------------------------------------------------------------------------
# helpers
# DRAM traffic per launch of the dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum) from one ncu capture of the same workload; the
# summaries under profiles/ give the commands.  An entry is reported only while
# the CUDA sources hash to the state that was captured; after any kernel change
# the traffic is null until it is captured again.
NCU_TRAFFIC = {
    # (config, inputs): (bytes per launch, csrc_digest() at capture, summary)
    ("cfg2", "independent"): (606428416, "d73de573e099ed1dd14718d2c225affa8268bb5f2576b7b49fda195b403af08b",
                              "profiles/multi_kernel_q8_0_qwen3_0.6b_stream.md"),
    # captured on 2 of the 28 layers (+ LM head) and scaled by algorithmic bytes
    ("cfg3", "independent"): (4006526862, "d73de573e099ed1dd14718d2c225affa8268bb5f2576b7b49fda195b403af08b",
                              "profiles/multi_kernel_q4_0_7b_stream.md"),
    ("cfg3k", "independent"): (4006904606, "d73de573e099ed1dd14718d2c225affa8268bb5f2576b7b49fda195b403af08b",
                               "profiles/multi_kernel_q4_k_7b_stream.md"),
}


# CUDA sources that no part of the streaming kernel or its planner is built
# from: changing them leaves the captured traffic valid
DIGEST_EXCLUDES = ("bq_f16.cu",)


def csrc_digest():
    """sha256 over the CUDA sources (names and contents, sorted by name) that
    the streaming kernel and its planner may be built from"""
    import hashlib
    d = os.path.join(ROOT, "block_quantized_weight_dequant_gb300", "csrc")
    h = hashlib.sha256()
    for n in sorted(os.listdir(d)):
        if n.endswith((".cu", ".cuh", ".h")) and n not in DIGEST_EXCLUDES:
            h.update(n.encode())
            with open(os.path.join(d, n), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def ncu_traffic(config, inputs):
    e = NCU_TRAFFIC.get((config, inputs if config in TOKEN_CONFIGS else None))
    if e is None or e[1] != csrc_digest():
        return None, None
    return e[0], e[2]


# ---------------------------------------------------------------------------
def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads on the GPU
# ---------------------------------------------------------------------------
class Workload:
    """A list of launches (closures over device tensors) forming one step."""

    def __init__(self):
        self.launches = []      # callables, each one call of ours
        self.kernels = []       # kernel launches each call enqueues
        self.kinds = []         # kernel family per launch
        self.bytes = []         # algorithmic bytes per launch
        self.x_dev = None       # concatenated per-step inputs (device)
        self.y_dev = None       # concatenated per-step outputs (device)
        self.desc = {}
        self.checks = []        # what the CPU leg compares with the oracle (sampled rows)

    def add(self, fn, kind, nbytes, kernels=1):
        self.launches.append(fn)
        self.kernels.append(int(kernels))
        self.kinds.append(kind)
        self.bytes.append(nbytes)

    @property
    def kernels_per_step(self):
        return sum(self.kernels)

    @property
    def step_bytes(self):
        return sum(self.bytes)

    def run(self):
        for fn in self.launches:
            fn()


# The seeded generator call behind a packed matrix travels with the tensor
# (attribute `bq_source`), so the CPU leg can draw the same fp32 rows again for
# the oracle.  A tensor made otherwise (the load-time q|k|v concatenation) has
# none, and its rows are not checked.
def _packed(bq, wl, qt, M, K, seed, tag, dev):
    src = dict(shape=(M, K), std=wl.W_STD, seed=seed, stream=wl.stream_id(*tag))
    W = wl.normal_torch(src["shape"], src["std"], seed=seed, stream=src["stream"], device=dev)
    P = bq.quantize_pack(W, qt)
    del W
    P.bq_source = src
    return P


def weight_source(P):
    return getattr(P, "bq_source", None)


def build_token_layers(cfg, dev, seed=0, fused_qkv=False):
    """Packed weights of one token's stream (every layer's matrices, RMSNorm
    gains and the LM head), drawn and packed on the GPU."""
    import block_quantized_weight_dequant_gb300 as bq
    from block_quantized_weight_dequant_gb300 import workloads as wl

    qt = cfg["qtype"]
    shapes = {n: (M, K) for n, M, K in cfg["mats"]}
    layers = []
    for l in range(cfg["layers"]):
        L = {n: _packed(bq, wl, qt, M, K, seed, (cfg["name"], l, n), dev)
             for n, (M, K) in shapes.items()}
        L["gamma"] = wl.normal_torch(cfg["hidden"], 0.1, seed=seed,
                                     stream=wl.stream_id(cfg["name"], l, "gamma"), device=dev,
                                     mean=1.0)
        layers.append(L)
    if fused_qkv:
        for l, L in enumerate(layers):
            L["qkv"] = bq.concat_packed([L.pop("q"), L.pop("k"), L.pop("v")])
            L["qkv_bias"] = wl.normal_torch(L["qkv"].shape[0], 0.1, seed=seed,
                                            stream=wl.stream_id(cfg["name"], l, "qkv_bias"),
                                            device=dev)
    M, K = cfg["lm_head"]
    lm = _packed(bq, wl, qt, M, K, seed, (cfg["name"], "lm_head"), dev)
    return layers, lm


def build_token_stream(cfg, dev, seed=0, mode="plan", chained=False, packed=None,
                       fused_qkv=False, tune=True):
    """One decode step's GEMV stream (block_quantized_weight_dequant_gb300.decode).
    chained=False (default): every op reads an N(0, 1) input of its own, the
    pure per-token weight stream; chained: every stage reads the previous
    stage's output (113 dependent stages, grid-wide barriers).  mode "plan":
    one launch per step; mode "per_op": one launch per op.  `packed`: layers
    from build_token_layers, shared between the two input modes.  tune: split
    the plan's tiles among CTAs by measured time (set-up, untimed)."""
    import torch
    import block_quantized_weight_dequant_gb300 as bq
    from block_quantized_weight_dequant_gb300 import workloads as wl
    from block_quantized_weight_dequant_gb300.decode import DecodeStream

    qt = cfg["qtype"]
    layers, lm = packed if packed is not None else build_token_layers(cfg, dev, seed, fused_qkv)
    ds = DecodeStream(qt, layers, lm, chained=chained, fused_qkv=fused_qkv)
    ds.inputs.copy_(wl.normal_torch(ds.inputs.numel(), 1.0, seed=seed, stream=wl.stream_id("x0"),
                                    device=dev))
    w = Workload()
    nbytes = ds.weight_bytes() + ds.activation_bytes()
    if mode == "plan":
        p = ds.plan()
        if tune and not chained:
            # 10 rounds (33 launches at set-up): measured about 1% faster than 3
            p.tune(rounds=10)
        # a chained plan runs one kernel per stage, an independent one a single kernel
        w.add(ds.run_plan, f"stream_plan_{qt}", nbytes, kernels=p.launches)
    else:
        for op in ds.ops:
            nb = op.W.numel() + (op.W_up.numel() if op.W_up is not None else 0) + \
                4 * (op.x.numel() + op.y.numel() + (op.gamma.numel() if op.gamma is not None else 0))
            nb += 4 * (op.bias.numel() if op.bias is not None else 0)
            if op.W_up is None and op.bias is not None:
                w.add(lambda op=op: bq.gemv_qkv_bias(qt, op.W, op.x, op.bias, op.y),
                      f"gemv_qkv_bias_{qt}", nb)
            elif op.W_up is None:
                w.add(lambda op=op: bq.gemv(qt, op.W, op.x, op.y), f"gemv_{qt}", nb)
            else:
                w.add(lambda op=op: bq.gemv_gate_up_silu(qt, op.W, op.W_up, op.x, op.gamma,
                                                         op.eps, op.y), f"gate_up_silu_{qt}", nb)
    w.x_dev = ds.inputs
    # the step's result read back each e2e step: the logits of a chained
    # token; every op's output (one buffer) of an independent one
    w.y_dev = ds.logits if chained else ds.outputs
    w.stream_obj = ds
    w.desc = token_desc(cfg, mode, chained, fused_qkv)
    if mode == "plan" and not chained:
        w.desc["cta_split"] = ("equal measured time (bq_stream_plan_tune, 10 rounds, set-up)"
                               if tune else "equal bytes")
    assert (w.desc["ops_per_step"], w.desc["weight_bytes_per_step"]) == \
        (len(ds.ops), ds.weight_bytes())
    assert w.desc["stages_per_step"] == (ds.n_stages if chained else 1)
    if not chained:
        # every op reads a seeded input: each can be checked against the oracle
        # (a chained op reads another op's output, which the oracle may not use)
        for i, op in enumerate(ds.ops):
            tag = ("cfg-token", cfg["name"], i)
            if op.W_up is not None:
                w.checks.append(dict(kind="gate_up", qt=qt, Pg=op.W, Pu=op.W_up, x=op.x,
                                     gamma=op.gamma, eps=op.eps, y=op.y, tag=tag,
                                     src_g=weight_source(op.W),
                                     src_u=weight_source(op.W_up)))
            else:
                w.checks.append(dict(kind="gemv", qt=qt, P=op.W, x=op.x, y=op.y, bias=op.bias,
                                     tag=tag, src=weight_source(op.W)))
    return w


def build_rotated_gemv(dev, qt, M, K, copies, seed=0, name="cfg1"):
    import torch
    import block_quantized_weight_dequant_gb300 as bq
    from block_quantized_weight_dequant_gb300 import workloads as wl
    w = Workload()
    w.x_dev = wl.normal_torch(copies * K, 1.0, seed=seed, stream=wl.stream_id(name, "x"),
                              device=dev)
    w.y_dev = torch.empty(copies * M, device=dev)
    for c in range(copies):
        P = _packed(bq, wl, qt, M, K, seed, (name, c), dev)
        x, y = w.x_dev[c * K:(c + 1) * K], w.y_dev[c * M:(c + 1) * M]
        w.add(lambda P=P, x=x, y=y: bq.gemv(qt, P, x, y), f"gemv_{qt}", P.numel() + 4 * (M + K))
        w.checks.append(dict(kind="gemv", qt=qt, P=P, x=x, y=y, bias=None, tag=(name, c),
                             src=weight_source(P)))
    w.desc = {"workload": f"{qt} gemv {M}x{K}, {copies} rotated copies", "M": M, "K": K}
    return w


def build_f16_gemv(dev, seed=0):
    """One fp16-weight GEMV per step over a 151936 x 1024 matrix (311 MB,
    larger than L2, so every step reads it from HBM)."""
    import torch
    import block_quantized_weight_dequant_gb300 as bq
    from block_quantized_weight_dequant_gb300 import workloads as wl
    c = wl.F16_LM
    M, K = c["M"], c["K"]
    w = Workload()
    src = dict(shape=(M, K), std=1.0, seed=seed, stream=wl.stream_id("f16", "W"),
               post_scale=wl.W_STD, dtype=torch.float16)
    W = (wl.normal_torch((M, K), 1.0, seed=seed, stream=src["stream"], device=dev) *
         wl.W_STD).to(torch.float16)
    w.x_dev = wl.normal_torch(K, 1.0, seed=seed, stream=wl.stream_id("f16", "x"), device=dev)
    w.y_dev = torch.empty(M, device=dev)
    w.add(lambda: bq.gemv_f16(W, w.x_dev, w.y_dev), "gemv_f16", 2 * M * K + 4 * (M + K))
    w.checks.append(dict(kind="f16", W=W, x=w.x_dev, y=w.y_dev, tag=("f16",), src=src))
    w.desc = {"workload": c["name"], "M": M, "K": K}
    return w


def build_rotated_gate_up(dev, cfg, seed=0):
    import torch
    import block_quantized_weight_dequant_gb300 as bq
    from block_quantized_weight_dequant_gb300 import workloads as wl
    qt, M, K, n = cfg["qtype"], cfg["M"], cfg["K"], cfg["pairs"]
    w = Workload()
    w.x_dev = wl.normal_torch(n * K, 1.0, seed=seed, stream=wl.stream_id("cfg4", "x"), device=dev)
    w.y_dev = torch.empty(n * M, device=dev)
    for c in range(n):
        Pg = _packed(bq, wl, qt, M, K, seed, ("cfg4", c, "g"), dev)
        Pu = _packed(bq, wl, qt, M, K, seed, ("cfg4", c, "u"), dev)
        g = wl.normal_torch(K, cfg["gamma_std"], seed=seed, stream=wl.stream_id("cfg4", c, "gm"),
                            device=dev, mean=cfg["gamma_mean"])
        x, y = w.x_dev[c * K:(c + 1) * K], w.y_dev[c * M:(c + 1) * M]
        w.add(lambda Pg=Pg, Pu=Pu, x=x, g=g, y=y:
              bq.gemv_gate_up_silu(qt, Pg, Pu, x, g, cfg["eps"], y), f"gate_up_silu_{qt}",
              Pg.numel() + Pu.numel() + 8 * K + 4 * M)
        w.checks.append(dict(kind="gate_up", qt=qt, Pg=Pg, Pu=Pu, x=x, gamma=g, eps=cfg["eps"],
                             y=y, tag=("cfg4", c), src_g=weight_source(Pg),
                             src_u=weight_source(Pu)))
    w.desc = {"workload": cfg["name"], "M": M, "K": K, "pairs": n}
    return w


def build_verify(dev, cfg, R, copies=7, seed=0):
    import torch
    import block_quantized_weight_dequant_gb300 as bq
    from block_quantized_weight_dequant_gb300 import workloads as wl
    qt = cfg["qtype"]
    w = Workload()
    xs = sum(R * K for _, M, K in cfg["mats"]) * copies
    ys = sum(R * M for _, M, K in cfg["mats"]) * copies
    w.x_dev = wl.normal_torch(xs, 1.0, seed=seed, stream=wl.stream_id("cfg5", "x", R), device=dev)
    w.y_dev = torch.empty(ys, device=dev)
    xo = yo = 0
    for c in range(copies):
        for name, M, K in cfg["mats"]:
            P = _packed(bq, wl, qt, M, K, seed, ("cfg5", name, c), dev)
            X = w.x_dev[xo:xo + R * K].view(R, K)
            Y = w.y_dev[yo:yo + R * M].view(R, M)
            xo += R * K
            yo += R * M
            w.add(lambda P=P, X=X, Y=Y: bq.gemv_verify(qt, P, X, Y), f"verify_{qt}_R{R}",
                  P.numel() + 4 * R * (M + K))
            w.checks.append(dict(kind="verify", qt=qt, P=P, X=X, Y=Y, tag=("cfg5", name, c, R),
                                 src=weight_source(P)))
    w.desc = {"workload": cfg["name"], "R": R, "copies": copies}
    return w


def wl_cfg5():
    from block_quantized_weight_dequant_gb300 import workloads as wl
    return wl.CFG5


def token_desc(cfg, mode, chained, fused_qkv=False):
    """Config entries of a token-stream step (no GPU needed)."""
    from block_quantized_weight_dequant_gb300 import workloads as wl
    bb = 34 if cfg["qtype"] == "q8_0" else 18
    wbytes = sum(M * K // 32 * bb for _, M, K in wl.token_weight_shapes(cfg))
    d = {"workload": cfg["name"], "layers": cfg["layers"],
         "ops_per_step": len(wl.token_stream_ops(cfg, fused_qkv)),
         # dependent stages (grid-wide barriers): none when every op reads an input of its own
         "stages_per_step": 4 * cfg["layers"] + 1 if chained else 1,
         "weight_bytes_per_step": wbytes, "weight_format": cfg["qtype"], "launch": mode,
         "inputs": "chained (each stage reads the previous stage's output)" if chained
         else "independent (each op reads an N(0,1) input of its own)"}
    if fused_qkv:
        d["qkv"] = "fused: q|k|v rows concatenated at load time, one op with an N(0,0.1) bias"
    return d


def workload_desc(args):
    """The step's config entries, identical in both arms (no GPU needed)."""
    from block_quantized_weight_dequant_gb300 import workloads as wl
    if args.config in TOKEN_CONFIGS:
        cfg = token_cfg(args.config)
        if args.layers:
            cfg["layers"] = args.layers
        return token_desc(cfg, args.launch, args.inputs == "chained", args.qkv == "fused")
    if args.config == "cfg1":
        c = wl.CFG1
        return {"workload": f"{c['qtype']} gemv {c['M']}x{c['K']}, {CFG1_COPIES} rotated copies",
                "M": c["M"], "K": c["K"]}
    if args.config == "cfg4":
        c = wl.CFG4
        return {"workload": c["name"], "M": c["M"], "K": c["K"], "pairs": c["pairs"]}
    if args.config == "f16":
        c = wl.F16_LM
        return {"workload": c["name"], "M": c["M"], "K": c["K"]}
    return {"workload": wl.CFG5["name"], "R": args.rows, "copies": CFG5_COPIES}


def step_bytes_static(args):
    """Algorithmic bytes of one step (packed weights + x read + y written
    (+ gamma)), computed from the shapes alone."""
    from block_quantized_weight_dequant_gb300 import workloads as wl
    if args.config in TOKEN_CONFIGS:
        cfg = token_cfg(args.config)
        if args.layers:
            cfg["layers"] = args.layers
        return token_bytes_cfg(cfg, args.qkv == "fused")
    if args.config == "cfg1":
        c = wl.CFG1
        return CFG1_COPIES * (c["M"] * c["K"] // 32 * 34 + 4 * (c["M"] + c["K"]))
    if args.config == "cfg4":
        c = wl.CFG4
        return c["pairs"] * (2 * c["M"] * c["K"] // 32 * 34 + 8 * c["K"] + 4 * c["M"])
    if args.config == "f16":
        c = wl.F16_LM
        return 2 * c["M"] * c["K"] + 4 * (c["M"] + c["K"])
    R = args.rows
    return CFG5_COPIES * sum(M * K // 32 * 18 + 4 * R * (M + K) for _, M, K in wl.CFG5["mats"])


def build_workload(args, dev):
    from block_quantized_weight_dequant_gb300 import workloads as wl
    chained = args.inputs == "chained"
    if args.config in TOKEN_CONFIGS:
        cfg = token_cfg(args.config)
        if args.layers:
            cfg["layers"] = args.layers
        fq = args.qkv == "fused"
        packed = build_token_layers(cfg, dev, fused_qkv=fq)
        w = build_token_stream(cfg, dev, mode=args.launch, chained=chained, packed=packed,
                               fused_qkv=fq, tune=args.tune)
        if args.other_inputs:
            w.other = build_token_stream(cfg, dev, mode=args.launch, chained=not chained,
                                         packed=packed, fused_qkv=fq, tune=args.tune)
        return w
    if args.config == "cfg1":
        c = wl.CFG1
        return build_rotated_gemv(dev, c["qtype"], c["M"], c["K"], copies=CFG1_COPIES)
    if args.config == "cfg4":
        return build_rotated_gate_up(dev, wl.CFG4)
    if args.config == "cfg5":
        return build_verify(dev, wl.CFG5, args.rows, copies=CFG5_COPIES)
    if args.config == "f16":
        return build_f16_gemv(dev)
    raise SystemExit(f"unknown config {args.config}")


def tokens_per_step(args):
    return 1.0 if args.config in TOKEN_CONFIGS else None


# ---------------------------------------------------------------------------
# timing
# ---------------------------------------------------------------------------
def time_graph(graph, stream, steps, dist_barrier):
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    dist_barrier()
    torch.cuda.synchronize()
    start_all = torch.cuda.Event(enable_timing=True)
    end_all = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start_all.record(stream)
        for s, e in ev:
            s.record(stream)
            graph.replay()
            e.record(stream)
        end_all.record(stream)
    torch.cuda.synchronize()
    dist_barrier()
    per = [s.elapsed_time(e) for s, e in ev]
    return start_all.elapsed_time(end_all), per


def hold_load(replay, sync, seconds, batch=16):
    """Replay the step back to back, `batch` replays between host syncs, for
    at least `seconds` of wall time; returns the number of replays.  Run just
    before the timed region while nvidia-smi samples, so that the clock
    samples see the GPU under this step's load, not idle."""
    n = 0
    t0 = time.perf_counter()
    while True:
        for _ in range(batch):
            replay()
        sync()
        n += batch
        if time.perf_counter() - t0 >= seconds:
            return n


def capture(w, stream, warmup):
    """Run the step once eagerly (module load, kernel attributes), capture it
    in a CUDA graph and replay it `warmup` times."""
    import torch
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        w.run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        w.run()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    return graph


# ---------------------------------------------------------------------------
# the CPU leg: the oracle on the host (cpu_baseline, --impl reference) and the
# sampled-row parity of the timed step.  This is the only part of bench.py
# that loads the oracle (test infrastructure under oracle/ and tests/).
# ---------------------------------------------------------------------------
def _oracle_modules():
    tests = os.path.join(ROOT, "tests")
    if tests not in sys.path:
        sys.path.insert(0, tests)
    import oracle
    return oracle


def oracle_jobs(config, rows=6, layers=0):
    """One step of the config as the oracle computes it: a list of GEMVs
    (format, M, K, input rows), the matrices in the step's order (gate and up
    of a fused op are two GEMVs; a verify call is R GEMVs of one matrix)."""
    from block_quantized_weight_dequant_gb300 import workloads as wl
    if config in TOKEN_CONFIGS:
        cfg = token_cfg(config)
        if layers:
            cfg["layers"] = layers
        return [(cfg["qtype"], M, K, 1) for _, M, K in wl.token_weight_shapes(cfg)]
    if config == "cfg1":
        c = wl.CFG1
        return [(c["qtype"], c["M"], c["K"], 1)] * CFG1_COPIES
    if config == "cfg4":
        c = wl.CFG4
        return [(c["qtype"], c["M"], c["K"], 1)] * (2 * c["pairs"])
    if config == "f16":
        return [("f16", wl.F16_LM["M"], wl.F16_LM["K"], 1)]
    return [(wl.CFG5["qtype"], M, K, rows) for _, M, K in wl.CFG5["mats"]] * CFG5_COPIES


def oracle_step_data(jobs, seed=0):
    """Host inputs for the oracle jobs: packed bytes drawn at random (every
    block scale a finite fp16 between 2^-9 and 2^-6; the scalar oracle's time
    does not depend on the values) and N(0, 1) inputs.  Distinct arrays per
    job, so the host caches hold no more of the step than a real one would."""
    import numpy as np
    rng = np.random.default_rng([seed, 0xB0])
    data = []
    for fmt, M, K, R in jobs:
        if fmt == "f16":
            W = (rng.standard_normal((M, K), dtype=np.float32) * np.float32(0.02)).astype(
                np.float16).view(np.uint16)
        else:
            bb = 34 if fmt == "q8_0" else 18
            W = np.frombuffer(rng.bytes(M * (K // 32) * bb), dtype=np.uint8).copy()
            # the high byte of every fp16 scale (Q4_K: d and dmin of each
            # 144-byte super-block)
            blk = W.reshape(-1, 144) if fmt == "q4_k" else W.reshape(-1, bb)
            for at in ((1, 3) if fmt == "q4_k" else (1,)):
                blk[:, at] = rng.integers(0x18, 0x24, size=blk.shape[0], dtype=np.uint8)
            W = W.reshape(M, (K // 32) * bb)
        X = rng.standard_normal((R, K))
        data.append((fmt, M, K, W, X))
    return data


def oracle_run(o, oracle, data, threads, budget_s, whole_steps):
    """Run the oracle over the step's jobs in order, on `threads` host threads
    (rows split among them), until `budget_s` has passed -- in whole steps
    (at least one) when `whole_steps`, else stopping after any job.  Returns
    (fraction of steps done, seconds)."""
    import numpy as np
    weights = sum(M * K * X.shape[0] for _, M, K, _, X in data)
    done = 0
    t0 = time.perf_counter()
    while True:
        for fmt, M, K, W, X in data:
            for x in X:
                if fmt == "f16":
                    o.gemv_f16_parallel(W, x, threads=threads, with_S=False)
                else:
                    qt = {"q8_0": oracle.Q8_0, "q4_0": oracle.Q4_0, "q4_k": oracle.Q4_K}[fmt]
                    o.gemv_parallel(qt, W, M, K, x, threads=threads, with_S=False)
                done += M * K
            if not whole_steps and time.perf_counter() - t0 >= budget_s:
                return done / weights, time.perf_counter() - t0
        if time.perf_counter() - t0 >= budget_s:
            return done / weights, time.perf_counter() - t0


def oracle_timing(args, budget_s, threads, whole_steps):
    """The oracle (plain C, fp64, scalar) over the config's step on `threads`
    host threads; GB/s counts the step's algorithmic bytes.  Returns (GB/s,
    seconds, bytes, description)."""
    oracle = _oracle_modules()
    o = oracle.get()
    jobs = oracle_jobs(args.config, getattr(args, "rows", 6), getattr(args, "layers", 0))
    data = oracle_step_data(jobs)
    frac, dt = oracle_run(o, oracle, data, threads, budget_s, whole_steps)
    nbytes = frac * step_bytes_static(args)
    desc = (f"the oracle over the whole step ({len(jobs)} GEMVs: "
            f"{sum(W.nbytes for _, _, _, W, _ in data) / 1e6:.0f} MB of weights drawn at random "
            f"with finite scales, N(0,1) inputs) on {threads} host thread(s), rows split among "
            f"them; {frac:.3g} steps in {dt:.1f} s")
    return nbytes / dt / 1e9, dt, nbytes, desc


def cpu_baseline(args, budget_s):
    """The oracle single-threaded (a bounded part of the step) and on every
    host core (whole steps)."""
    oracle = _oracle_modules()
    n = oracle.host_cores()
    g1, dt1, nb1, d1 = oracle_timing(args, budget_s, 1, whole_steps=False)
    gn, dtn, nbn, dn = oracle_timing(args, budget_s, n, whole_steps=True)
    out = {"value": round(gn, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": dn,
           "single_core": {"value": round(g1, 4), "cores": 1, "sample": d1}}
    if tokens_per_step(args):
        out["tok_per_s"] = round(gn * 1e9 / step_bytes_static(args), 4)
        out["single_core"]["tok_per_s"] = round(g1 * 1e9 / step_bytes_static(args), 4)
    return out


def sampled_parity(w, rows_per_matrix):
    """The timed step's outputs against the oracle on sampled rows of every
    matrix (tests/sampled_parity.py): the oracle packs the seeded fp32 rows
    itself (the GPU's packed rows must equal its bytes) and its fp64 product
    bounds the GPU's output.  Verify rows are also compared bit for bit with
    the single-row decode GEMV."""
    import torch
    _oracle_modules()
    import sampled_parity as sp
    import block_quantized_weight_dequant_gb300 as bq
    res, skipped, decode_differ = [], 0, 0
    per = rows_per_matrix if callable(rows_per_matrix) else (lambda i: rows_per_matrix)
    for i, c in enumerate(w.checks):
        rows_per_matrix = per(i)
        src = c.get("src")
        if c["kind"] == "gemv":
            if src is None:
                skipped += 1
                continue
            idx = sp.sample_rows(c["y"].numel(), rows_per_matrix, *c["tag"])
            res.append(sp.check_gemv(c["qt"], sp.WeightSource(**src), c["P"], c["x"], c["y"], idx,
                                     c["bias"]))
        elif c["kind"] == "gate_up":
            if c["src_g"] is None or c["src_u"] is None:
                skipped += 1
                continue
            idx = sp.sample_rows(c["y"].numel(), rows_per_matrix, *c["tag"])
            res.append(sp.check_gate_up(c["qt"], sp.WeightSource(**c["src_g"]),
                                        sp.WeightSource(**c["src_u"]), c["Pg"], c["Pu"], c["x"],
                                        c["gamma"], c["eps"], c["y"], idx))
        elif c["kind"] == "verify":
            X, Y = c["X"], c["Y"]
            idx = sp.sample_rows(Y.shape[1], rows_per_matrix, *c["tag"])
            ii = torch.as_tensor(idx, device=Y.device)
            for r in range(X.shape[0]):
                res.append(sp.check_gemv(c["qt"], sp.WeightSource(**src), c["P"], X[r], Y[r], idx))
                yd = bq.gemv(c["qt"], c["P"], X[r].contiguous())
                decode_differ += int((Y[r].index_select(0, ii).view(torch.int32) !=
                                      yd.index_select(0, ii).view(torch.int32)).sum().item())
        elif c["kind"] == "f16":
            idx = sp.sample_rows(c["y"].numel(), rows_per_matrix, *c["tag"])
            res.append(sp.check_f16(sp.WeightSource(**src), c["W"], c["x"], c["y"], idx))
    out = sp.merge(res)
    out["skipped_matrices"] = skipped
    if any(c["kind"] == "verify" for c in w.checks):
        out["verify_rows_differ_from_decode"] = decode_differ
        out["pass"] = out["pass"] and decode_differ == 0
    out["sample"] = (f"{per(0)} rows per matrix and input row (the first, the last and "
                     "seeded rows; every row of smaller matrices)")
    return out


def token_bytes_cfg(cfg, fused_qkv=False):
    bb = 34 if cfg["qtype"] == "q8_0" else 18
    from block_quantized_weight_dequant_gb300 import workloads as wl
    total = 0
    for kind, name, M, K in wl.token_stream_ops(cfg, fused_qkv):
        if kind == "gemv":
            total += M * K // 32 * bb + 4 * (M + K)
        elif kind == "gemv_bias":
            total += M * K // 32 * bb + 4 * (M + K) + 4 * M
        else:
            total += 2 * M * K // 32 * bb + 8 * K + 4 * M
    return total


# FMA pipe of GB300: 152 SMs x 128 fp32 lane-ops per clock x 2.07 GHz (max SM
# clock).  The packed FFMA2/FADD2 issue in two cycles, so they do not raise it.
FMA_LANE_OPS_PER_S = 152 * 128 * 2.07e9


def roofline(args, dom, n_launch, achieved, peak, peak_kind, traffic, traffic_src, total_ms):
    """The dominant kernel against its bound.  HBM for the streams and the
    decode GEMVs; for verify with R >= 2 the FMA pipe, since every weight then
    costs R fp32 FMAs plus one fp32 add of its exact code conversion."""
    hbm = {"bound": "hbm", "kernel": dom, "launches_per_step": n_launch,
           "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
           "frac": round(achieved / peak, 4), "traffic": traffic,
           "traffic_source": traffic_src, "peak_kind": peak_kind}
    if args.config != "cfg5" or args.rows < 2:
        return hbm
    from block_quantized_weight_dequant_gb300 import workloads as wl
    R = args.rows
    weights = CFG5_COPIES * sum(M * K for _, M, K in wl.CFG5["mats"])
    ops_per_s = weights * (R + 1) * args.steps / (total_ms * 1e-3)
    return {"bound": "alu", "kernel": dom, "launches_per_step": n_launch,
            "achieved": round(ops_per_s / 1e9, 1), "peak": round(FMA_LANE_OPS_PER_S / 1e9, 1),
            "unit": "G FMA-pipe lane-ops/s", "frac": round(ops_per_s / FMA_LANE_OPS_PER_S, 4),
            "ops_per_weight": R + 1, "traffic": traffic, "traffic_source": traffic_src,
            "peak_kind": "derived: 152 SMs x 128 lanes x 2.07 GHz", "hbm": hbm}


# ---------------------------------------------------------------------------
# ranks: independent replicas; the job's time is the slowest rank's
# ---------------------------------------------------------------------------
def max_over_ranks(v, device, world):
    """The largest of every rank's v (all ranks get it)."""
    if world <= 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(step_bytes, steps, ms, world):
    """Bytes that all `world` replicas processed over the slowest rank's time."""
    return world * step_bytes * steps / (ms * 1e-3) / 1e9


# ---------------------------------------------------------------------------
def run_reference(args):
    """The reference arm: the oracle (the pages publish no runnable code; the
    oracle is this repository's plain CPU statement of the same products) on
    every host core, one whole step per timed step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    oracle = _oracle_modules()
    o = oracle.get()
    n = oracle.host_cores()
    jobs = oracle_jobs(args.config, args.rows, args.layers)
    data = oracle_step_data(jobs)
    for _ in range(args.warmup):
        oracle_run(o, oracle, data, n, 0.0, True)
    per = []
    for _ in range(args.steps):
        frac, dt = oracle_run(o, oracle, data, n, 0.0, True)
        per.append(dt / frac)
    t_total = sum(per)
    value = step_bytes_static(args) * args.steps / t_total / 1e9
    desc = (f"the oracle over one whole step per timed step ({len(jobs)} GEMVs, weights drawn at "
            f"random with finite scales, N(0,1) inputs) on {n} host threads, rows split among them")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t_total / max(1, args.steps), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: random packed weights with finite scales, N(0,1) inputs",
            "config": dict(workload_desc(args), config=args.config, bytes_per_step=step_bytes_static(args),
                           parallelism="replicas1"),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    if tokens_per_step(args):
        line["tok_per_s"] = round(value * 1e9 / step_bytes_static(args), 4)
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=15)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="cfg2",
                    choices=["cfg1", "cfg2", "cfg3", "cfg3k", "cfg4", "cfg5", "f16"])
    ap.add_argument("--rows", type=int, default=6, help="R for cfg5")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work per cpu_baseline leg (0 disables)")
    ap.add_argument("--parity-rows", type=int, default=16,
                    help="rows per matrix of the timed step checked against the oracle (0: none)")
    ap.add_argument("--launch", choices=["plan", "per_op"], default="plan",
                    help="cfg2/cfg3: one cooperative launch per token, or one launch per op")
    ap.add_argument("--inputs", choices=["chained", "independent"], default="independent",
                    help="cfg2/cfg3: each op reads an input of its own (the per-token weight "
                         "stream), or each stage reads the previous stage's output")
    ap.add_argument("--qkv", choices=["separate", "fused"], default="separate",
                    help="cfg2/cfg3: q, k, v as three ops, or one fused q|k|v op with a bias")
    ap.add_argument("--layers", type=int, default=0,
                    help="cfg2/cfg3: fewer layers than the model's (smaller cases for profiling)")
    ap.add_argument("--no-tune", dest="tune", action="store_false",
                    help="cfg2/cfg3 plans: keep the planner's equal-bytes CTA split instead of "
                         "re-splitting by measured time at set-up")
    ap.add_argument("--no-other-inputs", dest="other_inputs", action="store_false",
                    help="cfg2/cfg3: skip timing the other input mode as a secondary figure")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist
    import block_quantized_weight_dequant_gb300 as bq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def barrier():
        if world > 1:
            dist.barrier()

    w = build_workload(args, dev)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)
    graph = capture(w, stream, args.warmup)

    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(stream):
        held = hold_load(graph.replay, stream.synchronize, 1.0)
    total_ms, per = time_graph(graph, stream, args.steps, barrier)
    clk = clocks.stop()
    if clk is not None:
        clk["window"] = (f"100 ms samples over {held} untimed replays of the step (1 s) "
                         "run just before the timed steps, and over the timed steps")
    other = None
    if getattr(w, "other", None) is not None:
        og = capture(w.other, stream, args.warmup)
        o_ms, o_per = time_graph(og, stream, args.steps, barrier)
        other = {"inputs": w.other.desc["inputs"], "stages_per_step": w.other.desc["stages_per_step"],
                 "launches_per_step": w.other.kernels_per_step,
                 "ms_per_step": round(o_ms / args.steps, 5),
                 "step_ms_median": round(statistics.median(o_per), 5),
                 "value": round(w.other.step_bytes * args.steps / (o_ms * 1e-3) / 1e9, 2),
                 "unit": "GB/s",
                 "tok_per_s": round(args.steps / (o_ms * 1e-3), 2)}
        del og

    total_ms = max_over_ranks(total_ms, dev, world)
    step_bytes = w.step_bytes
    assert step_bytes == step_bytes_static(args)
    value = whole_job_gbs(step_bytes, args.steps, total_ms, world)

    # e2e: the same step with host buffers: H2D of the step's inputs from
    # pinned memory, the step, D2H of the step's outputs, every step.  `e2e`
    # makes the step's calls through the public API (Python binding -> C ABI)
    # each step, as a user would; `e2e_graph` replays the captured graph.
    x_host = torch.empty(w.x_dev.shape, dtype=w.x_dev.dtype, pin_memory=True)
    x_host.copy_(w.x_dev.cpu())
    y_host = torch.empty(w.y_dev.shape, dtype=w.y_dev.dtype, pin_memory=True)

    def e2e_leg(step):
        barrier()
        torch.cuda.synchronize()
        e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e_s.record(stream)
            for _ in range(args.steps):
                w.x_dev.copy_(x_host, non_blocking=True)
                step()
                y_host.copy_(w.y_dev, non_blocking=True)
            e_e.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms = max_over_ranks(e_s.elapsed_time(e_e), dev, world)
        return whole_job_gbs(step_bytes, args.steps, ms, world)

    e2e_value = e2e_leg(w.run)
    e2e_graph_value = e2e_leg(graph.replay)

    # every step is one kernel family (the stream executor for cfg2/cfg3, one
    # GEMV family for the rotated configs), so the dominant kernel's launch
    # durations are the timed region's own per-launch CUDA-event times
    peak, peak_kind = measured_peak()
    kinds = sorted(set(w.kinds))
    dom = kinds[0] if len(kinds) == 1 else "+".join(kinds)
    n_launch = w.kernels_per_step
    achieved = (step_bytes / n_launch) / (total_ms * 1e-3 / args.steps / n_launch) / 1e9
    assert bq.device_status(clear=True) == 0, "device-side error recorded during the bench"

    if rank != 0:
        return 0
    ms_step = total_ms / args.steps
    traffic, traffic_src = ncu_traffic(args.config, args.inputs) \
        if not args.layers and args.launch == "plan" and args.qkv == "separate" else (None, None)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded N(0,0.02) weights packed on the GPU, N(0,1) inputs",
        "config": dict(w.desc, config=args.config,
                       l2="packed weights per step larger than the 129 MB L2 (no flush)",
                       bytes_per_step=step_bytes, parallelism=f"replicas{world}"),
        "pct_of_peak": {"measured": round(100 * value / world / peak, 2),
                        "nominal_8TBps": round(100 * value / world / NOMINAL_HBM_GBS, 2),
                        "peak_kind": peak_kind},
        "step_ms_median": round(statistics.median(per), 5),
        "step_ms_p10_p90": [round(sorted(per)[len(per) // 10], 5),
                            round(sorted(per)[(9 * len(per)) // 10], 5)],
        "roofline": roofline(args, dom, n_launch, achieved, peak, peak_kind, traffic, traffic_src,
                             total_ms),
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": x_host.numel() * 4, "d2h_bytes_per_step": y_host.numel() * 4,
                "calls": f"{len(w.launches)} public-API call(s) per step, no graph"},
        "e2e_graph": {"value": round(e2e_graph_value, 2), "unit": "GB/s",
                      "calls": "the step's calls captured once in a CUDA graph, replayed"},
        "clocks": clk,
        "gpu_launches": w.kernels_per_step * args.steps,
    }
    if other is not None:
        line["other_inputs"] = other
    if tokens_per_step(args):
        line["tok_per_s"] = round(value * 1e9 / step_bytes / world, 2)
        ds = w.stream_obj
        n_gemv = sum(2 if op.W_up is not None else 1 for op in ds.ops)
        line["gemvs_per_s"] = round(n_gemv * args.steps / (total_ms * 1e-3), 1)
    if args.parity_rows > 0:
        line["parity"] = sampled_parity(w, args.parity_rows)
    if args.cpu_budget > 0:
        line["cpu_baseline"] = cpu_baseline(args, args.cpu_budget)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
