"""Parity at full size on sampled rows: the GPU library's outputs against the
oracle, row by row, for workloads too large for the oracle to evaluate whole.

For each checked matrix the fp32 weights are drawn again from the same seeded
generator call that produced them (``WeightSource``), the sampled rows are
copied to the host, and the oracle packs them itself.  The GPU's packed rows
must equal the oracle's bytes, and the GPU's outputs on those rows must be
within the GEMV bound of the oracle's fp64 product of the ORACLE's packed rows
with the seeded input.  So no oracle input and no expected value comes from
the CUDA path: only the seeded generators serve both sides.

TEST INFRASTRUCTURE (it calls the oracle): used by ``tests/`` and by the CPU
leg of ``bench.py``.
"""
import numpy as np
import torch

import oracle
from tolerance import REL, gate_up_bound

QT = {"q8_0": oracle.Q8_0, "q4_0": oracle.Q4_0, "q4_k": oracle.Q4_K}


class WeightSource:
    """The seeded generator call of one weight matrix: fp32 N(mean, std) of
    `shape` from ``workloads.normal_torch`` (seed, stream), then an optional
    scale and cast (the fp16-weight GEMV's matrix)."""

    def __init__(self, shape, std, seed, stream, mean=0.0, post_scale=None, dtype=None):
        self.shape, self.std, self.seed, self.stream, self.mean = tuple(shape), std, seed, stream, mean
        self.post_scale, self.dtype = post_scale, dtype

    def draw(self, device):
        from block_quantized_weight_dequant_gb300 import workloads as wl
        t = wl.normal_torch(self.shape, self.std, seed=self.seed, stream=self.stream,
                            mean=self.mean, device=device)
        if self.post_scale is not None:
            t = t * self.post_scale
        if self.dtype is not None:
            t = t.to(self.dtype)
        return t

    def rows(self, idx, device):
        """The drawn matrix's rows `idx` (numpy) on the host.  The indices are
        checked here, on the host: an index past the matrix must never reach
        a device gather."""
        idx = np.asarray(idx)
        if idx.size and (idx.min() < 0 or idx.max() >= self.shape[0]):
            raise IndexError(f"rows {idx.min()}..{idx.max()} outside a {self.shape} source")
        i = torch.as_tensor(idx, device=device, dtype=torch.long)
        return self.draw(device).index_select(0, i).cpu().numpy()

    def matches(self, rows, K):
        """Whether this source drew a rows x K matrix."""
        return tuple(self.shape[:2]) == (int(rows), int(K))


def sample_rows(M, n, *tag, seed=0):
    """Sorted row indices: every row when M <= n, else the first and the last
    row and n - 2 distinct rows drawn from a generator keyed by `tag`."""
    if M <= n:
        return np.arange(M)
    from block_quantized_weight_dequant_gb300 import workloads as wl
    rng = np.random.default_rng([seed, wl.stream_id("parity-rows", *tag)])
    mid = rng.choice(np.arange(1, M - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, M - 1], mid]))


def _take(t, idx):
    idx = np.asarray(idx)
    if idx.size and (idx.min() < 0 or idx.max() >= t.shape[0]):
        raise IndexError(f"rows {idx.min()}..{idx.max()} outside a tensor of {t.shape[0]} rows")
    return t.index_select(0, torch.as_tensor(idx, device=t.device, dtype=torch.long))


def _need_source(src, P, K):
    if not src.matches(P.shape[0], K):
        raise ValueError(f"weight source {src.shape} does not describe a {P.shape[0]} x {K} matrix")


def _result(rows, pack_bad, err, bound, S=None):
    ok = np.isfinite(err)
    ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0), np.where(err > 0, np.inf, 0.0))
    r = {"rows": int(rows), "pack_rows_differ": int(pack_bad),
         "violations": int((~ok | (ratio > 1.0)).sum()),
         "max_err_over_bound": float(np.max(ratio)) if ratio.size else 0.0}
    if S is not None:
        q = np.where(S > 0, err / np.where(S > 0, S, 1.0), 0.0)
        r["max_err_over_S"] = float(np.max(q)) if q.size else 0.0
    return r


def oracle_packed_rows(qt, src, P, idx):
    """The oracle's packing of the sampled fp32 rows, and how many of them
    differ from the GPU's packed rows."""
    o = oracle.get()
    Pref = o.quantize_pack_parallel(QT[qt], src.rows(idx, P.device))
    bad = int((_take(P, idx).cpu().numpy() != Pref).any(axis=1).sum())
    return Pref, bad


def check_gemv(qt, src, P, x, y, idx, bias=None):
    """Rows idx of y = W x (+ bias) against the oracle; P the GPU's packed W."""
    o = oracle.get()
    _need_source(src, P, x.numel())
    Pref, bad = oracle_packed_rows(qt, src, P, idx)
    xh = x.detach().reshape(-1).cpu().numpy().astype(np.float64)
    y_ref, S = o.gemv_parallel(QT[qt], Pref, len(idx), xh.size, xh)
    if qt == "q4_k":
        # the bound's scale for the kernels' split evaluation d*sc*sum(q x) - dmin*m*sum(x)
        S = o.q4_k_split_scale_parallel(Pref, len(idx), xh.size, xh)
    if bias is not None:
        b = _take(bias, idx).cpu().numpy().astype(np.float64)
        y_ref, S = y_ref + b, S + np.abs(b)
    yg = _take(y.reshape(-1), idx).cpu().numpy().astype(np.float64)
    err = np.abs(yg - y_ref)
    # S == 0 demands an exact zero: any error is then a violation
    return _result(len(idx), bad, err, REL * S, S)


def check_gate_up(qt, src_g, src_u, Pg, Pu, x, gamma, eps, y, idx):
    """Rows idx of y = silu(Wg xn) * (Wu xn) against the oracle's fp64
    RMSNorm and gate+up, within the propagated bound of tolerance.py."""
    o = oracle.get()
    _need_source(src_g, Pg, x.numel())
    _need_source(src_u, Pu, x.numel())
    Pgr, bg = oracle_packed_rows(qt, src_g, Pg, idx)
    Pur, bu = oracle_packed_rows(qt, src_u, Pu, idx)
    xh = x.detach().reshape(-1).cpu().numpy().astype(np.float64)
    if gamma is not None:
        xn = o.rmsnorm(xh, gamma.detach().cpu().numpy().astype(np.float64), eps)
    else:
        xn = xh
    r = o.gate_up_silu(QT[qt], Pgr, Pur, len(idx), xh.size, xn)
    if qt == "q4_k":
        r["Sg"] = o.q4_k_split_scale_parallel(Pgr, len(idx), xh.size, xn)
        r["Su"] = o.q4_k_split_scale_parallel(Pur, len(idx), xh.size, xn)
    yg = _take(y.reshape(-1), idx).cpu().numpy().astype(np.float64)
    return _result(len(idx), bg + bu, np.abs(yg - r["y"]), gate_up_bound(r))


def check_f16(src, W, x, y, idx):
    """Rows idx of the fp16-weight GEMV against the oracle; the weights are
    drawn again and must equal the GPU's copy bit for bit."""
    o = oracle.get()
    _need_source(src, W, x.numel())
    Wr = src.rows(idx, W.device)
    bad = int((_take(W, idx).cpu().numpy().view(np.uint16) != Wr.view(np.uint16)).any(axis=1).sum())
    xh = x.detach().reshape(-1).cpu().numpy().astype(np.float64)
    y_ref, S = o.gemv_f16_parallel(Wr.view(np.uint16), xh)
    yg = _take(y.reshape(-1), idx).cpu().numpy().astype(np.float64)
    return _result(len(idx), bad, np.abs(yg - y_ref), REL * S, S)


def merge(results):
    """One summary over many checks."""
    out = {"rows": 0, "pack_rows_differ": 0, "violations": 0, "max_err_over_bound": 0.0}
    s = [r["max_err_over_S"] for r in results if "max_err_over_S" in r]
    for r in results:
        out["rows"] += r["rows"]
        out["pack_rows_differ"] += r["pack_rows_differ"]
        out["violations"] += r["violations"]
        out["max_err_over_bound"] = max(out["max_err_over_bound"], r["max_err_over_bound"])
    if s:
        out["max_err_over_S"] = max(s)
    out["checks"] = len(results)
    out["pass"] = out["violations"] == 0 and out["pack_rows_differ"] == 0
    return out
