"""Host logic of the streaming kernel's planner, on the CPU (no GPU needed):
the per-op lane-order search, the CTA split by measured time, and the split
of a short op list in which every op has CTAs of its own.

The lane order decides which lane bits of a warp form the unit column l and
which the row rho.  Its contract, for 16-byte shared-memory loads on GB300:
every lane quad reads at most two distinct x chunks (the lanes of one unit
column read the same x chunk), and the 8 lanes of every quarter-warp read
weight chunks rho*S + l*U + k in 8 distinct bank groups (chunk mod 8).  The
split contract: contiguous ranges covering every tile, with equal estimated
time when every tile costs its bytes times its previous CTA's time per byte.
"""
import ctypes

import numpy as np
import pytest

from block_quantized_weight_dequant_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    L = ctypes.CDLL(_lib.LIB_PATH)
    i32, vp = ctypes.c_int, ctypes.c_void_p
    L.bq_internal_lane_order.restype = i32
    L.bq_internal_lane_order.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(i32),
                                         ctypes.POINTER(i32)]
    L.bq_internal_rebalance.restype = None
    L.bq_internal_rebalance.argtypes = [vp, ctypes.c_longlong, i32, vp, vp, vp]
    L.bq_internal_split_by_op.restype = None
    L.bq_internal_split_by_op.argtypes = [vp, vp, i32, i32, vp]
    return L


def pext(v, m):
    r = k = 0
    for b in range(5):
        if m >> b & 1:
            r |= (v >> b & 1) << k
            k += 1
    return r


def meets_contract(mask, G, S, U):
    if bin(mask).count("1") != G.bit_length() - 1:
        return False
    for q in range(4):
        groups = {(pext(ln, ~mask & 31) * S + pext(ln, mask) * U) % 8 for ln in range(8 * q, 8 * q + 8)}
        if len(groups) != 8:
            return False
    for q in range(8):
        if len({pext(ln, mask) for ln in range(4 * q, 4 * q + 4)}) > 2:
            return False
    return True


def candidates(G, rows_low):
    """the planner's candidate orders: rows in lane bits 0..2; row/unit/row;
    row/unit/unit (rows_low: the first only)"""
    ub = G.bit_length() - 1
    rb = 5 - ub
    out = []
    if rows_low or rb >= 3:
        out.append(((G - 1) << rb) & 31)
    if not rows_low and ub >= 1 and rb >= 2:
        out.append(0b00010 | (((1 << (ub - 1)) - 1) << 3))
    if not rows_low and ub >= 2 and rb >= 1:
        out.append((G - 1) << 1)
    return out


def lane_order(lib, G, S0, U, pad, rows_low=False):
    S, m = ctypes.c_int(), ctypes.c_int()
    ok = lib.bq_internal_lane_order(G, S0, U, int(pad), int(rows_low), ctypes.byref(S), ctypes.byref(m))
    return bool(ok), S.value, m.value


# (G, natural stride in chunks, unit chunks): the configured shapes' items
SHAPES = [(4, 68, 17), (8, 136, 17), (4, 204, 17), (2, 34, 17), (1, 17, 17),  # Q8_0
          (16, 126, 9), (16, 144, 9), (4, 36, 9), (8, 72, 9), (4, 180, 9)]    # Q4_0


@pytest.mark.parametrize("G,S0,U", SHAPES)
@pytest.mark.parametrize("rows_low", [False, True])
def test_lane_order_meets_the_load_contract(lib, G, S0, U, rows_low):
    ok, S, m = lane_order(lib, G, S0, U, pad=True, rows_low=rows_low)
    assert ok
    assert S0 <= S < S0 + 8
    assert meets_contract(m, G, S, U), (G, S, m)
    if rows_low:  # the Q4_0 decode instance computes rho = lane mod (32/G) by shifts
        rb = 5 - (G.bit_length() - 1)
        assert m == ((G - 1) << rb) & 31
    # the stride is the smallest at which a candidate order meets the contract
    for s in range(S0, S):
        assert not any(meets_contract(c, G, s, U) for c in candidates(G, rows_low))


@pytest.mark.parametrize("G,S0,U", SHAPES)
def test_lane_order_without_padding_keeps_the_stride(lib, G, S0, U):
    ok, S, m = lane_order(lib, G, S0, U, pad=False)
    assert ok == any(meets_contract(c, G, S0, U) for c in candidates(G, False))
    if ok:
        assert S == S0 and meets_contract(m, G, S, U)


def test_one_row_tiles_have_no_candidate(lib):
    # G = 32: every lane is a unit column of one row; the planner falls back
    # to 8 units per quarter-warp (its x loads then take 4 cycles)
    assert not lane_order(lib, 32, 544, 17, pad=True)[0]


def rebalance(lib, tb, ct, d):
    tb = np.ascontiguousarray(tb, dtype=np.float64)
    ct = np.ascontiguousarray(ct, dtype=np.int32)
    d = np.ascontiguousarray(d, dtype=np.float64)
    grid = len(ct) - 1
    out = np.zeros(grid + 1, dtype=np.int32)
    lib.bq_internal_rebalance(tb.ctypes.data, len(tb), grid, ct.ctypes.data, d.ctypes.data,
                              out.ctypes.data)
    return out


def owner_cost(tb, ct, d):
    """cost of every tile: its bytes times its CTA's time per byte"""
    cost = np.empty(len(tb))
    for c in range(len(ct) - 1):
        b = tb[ct[c]:ct[c + 1]].sum()
        cost[ct[c]:ct[c + 1]] = tb[ct[c]:ct[c + 1]] * (d[c] / b)
    return cost


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_rebalance_equalises_estimated_time(lib, seed):
    rng = np.random.default_rng(seed)
    n, grid = 5000, 37
    tb = rng.integers(1, 40, n).astype(np.float64) * 272.0
    # an equal-bytes start, and per-CTA times with up to 2x differences per byte
    cum = np.cumsum(tb)
    ct = np.concatenate([[0], np.searchsorted(cum, cum[-1] * np.arange(1, grid) / grid) + 1, [n]])
    d = np.array([tb[ct[c]:ct[c + 1]].sum() for c in range(grid)]) * rng.uniform(1.0, 2.0, grid)
    out = rebalance(lib, tb, ct, d)
    assert out[0] == 0 and out[-1] == n and np.all(np.diff(out) >= 0)
    cost = owner_cost(tb, ct, d)
    per = np.array([cost[out[c]:out[c + 1]].sum() for c in range(grid)])
    target = cost.sum() / grid
    assert np.all(np.abs(per - target) <= cost.max() + 1e-9 * target)
    # the slowest range of the new split beats the slowest CTA measured
    assert per.max() < d.max()


def test_rebalance_with_uniform_times_keeps_an_equal_bytes_split(lib):
    n, grid = 1200, 8
    tb = np.full(n, 1088.0)
    ct = np.arange(grid + 1, dtype=np.int32) * (n // grid)
    d = np.full(grid, 5.0)
    assert np.array_equal(rebalance(lib, tb, ct, d), ct)


def test_rebalance_gives_idle_ctas_the_mean_rate(lib):
    # CTAs that ran no tile (or report no time) take the mean time per byte
    tb = np.full(100, 10.0)
    ct = np.array([0, 50, 50, 100], dtype=np.int32)
    d = np.array([2.0, 0.0, 1.0])
    out = rebalance(lib, tb, ct, d)
    assert out[0] == 0 and out[-1] == 100 and np.all(np.diff(out) >= 0)
    cost = owner_cost(tb, ct[[0, 1, 3]], d[[0, 2]])
    per = [cost[out[c]:out[c + 1]].sum() for c in range(3)]
    assert max(per) - min(per) <= 2 * cost.max()


def split_by_op(lib, op_bytes, op_tiles, grid):
    ob = np.asarray(op_bytes, dtype=np.int64)
    ot = np.asarray(op_tiles, dtype=np.int32)
    out = np.zeros(grid + 1, dtype=np.int32)
    lib.bq_internal_split_by_op(ob.ctypes.data, ot.ctypes.data, len(ob), grid, out.ctypes.data)
    return out


@pytest.mark.parametrize("op_bytes,op_tiles,grid", [
    ([2048, 1024, 1024], [256, 128, 128], 152),      # a layer's q, k, v
    ([1, 1, 1, 10 ** 9], [4, 4, 4, 3000], 152),      # tiny ops beside a large one
    ([5, 7], [1, 1], 152),                            # fewer tiles than CTAs
    ([3] * 76, [9] * 76, 152),                        # half as many ops as CTAs
    ([1000, 1], [50, 50], 9),
])
def test_split_by_op_gives_every_op_its_own_ctas(lib, op_bytes, op_tiles, grid):
    out = split_by_op(lib, op_bytes, op_tiles, grid)
    bounds = np.concatenate([[0], np.cumsum(op_tiles)])
    assert out[0] == 0 and out[-1] == bounds[-1]
    assert np.all(np.diff(out) >= 0)  # contiguous ranges covering every tile
    # no CTA range crosses an op boundary, and every op has at least one CTA
    owner = np.searchsorted(bounds, out[:-1], side="right") - 1
    for c in range(grid):
        lo, hi = out[c], out[c + 1]
        if hi > lo:
            assert bounds[owner[c]] <= lo and hi <= bounds[owner[c] + 1], (c, lo, hi)
    ctas = np.bincount(owner[np.diff(out) >= 0], minlength=len(op_tiles))
    assert np.all(ctas >= 1)
    assert ctas.sum() == grid
    # within an op the tiles are split evenly (sizes differ by at most one)
    for i in range(len(op_tiles)):
        sizes = np.diff(out)[owner == i]
        assert sizes.max() - sizes.min() <= 1
    # CTAs follow the bytes: within one CTA of the proportional share
    share = grid * np.asarray(op_bytes, dtype=np.float64) / np.sum(op_bytes)
    assert np.all(np.abs(ctas - np.maximum(1, share)) <= len(op_tiles))
