"""Parity bounds between the GPU library and the oracle.

GEMV outputs: |y_gpu - y_ref| <= 1e-5 * S with S = sum_k |w_mk * x_k| (the
oracle's fp64 sum of absolute products), and y_gpu == 0 exactly where S == 0.
The kernels' fixed fp32 tree has at most ~10 (block) + 8 (unit) + 37 (lane)
+ 5 (fold) sequential roundings per row at the largest K here, about
60 * 2^-24 * S = 3.6e-6 * S in the worst case, inside 1e-5 * S.

gate+up+SiLU outputs y = silu(g) * u: first-order propagation of the g and u
bounds, with |silu'| <= 1.0999, plus the fp32 rounding of expf, the divide
and the product:
    |dy| <= 1e-5 * (1.1 * S_g * |u| + |silu(g)| * S_u) + 1.1e-10 * S_g * S_u
            + 1e-6 * |y|
"""
import numpy as np

REL = 1e-5


def gemv_violations(y_gpu, y_ref, S, rel=REL):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bad = err > rel * S
    zero = S == 0
    bad |= zero & (y_gpu != 0)
    bad |= ~np.isfinite(y_gpu)
    return bad


def assert_gemv_close(y_gpu, y_ref, S, what="", rel=REL):
    bad = gemv_violations(y_gpu, y_ref, S, rel)
    if bad.any():
        i = np.flatnonzero(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outside |dy| <= {rel}*S; rows {i.tolist()} "
            f"gpu={np.asarray(y_gpu)[i].tolist()} ref={y_ref[i].tolist()} S={S[i].tolist()}")


def silu(z):
    return z / (1.0 + np.exp(-z))


def gate_up_bound(r):
    g, u, Sg, Su, y = r["g"], r["u"], r["Sg"], r["Su"], r["y"]
    return (REL * (1.1 * Sg * np.abs(u) + np.abs(silu(g)) * Su) + 1.1e-10 * Sg * Su
            + 1e-6 * np.abs(y))


def assert_gate_up_close(y_gpu, r, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    bound = gate_up_bound(r)
    err = np.abs(y_gpu - r["y"])
    bad = (err > bound) | ~np.isfinite(y_gpu)
    if bad.any():
        i = np.flatnonzero(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outside the gate+up bound; rows {i.tolist()} "
            f"gpu={y_gpu[i].tolist()} ref={r['y'][i].tolist()} bound={bound[i].tolist()}")
