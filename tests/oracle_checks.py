"""Pins for the oracle: checks against facts fixed outside the oracle itself.

Each ``check_*`` function takes an ``oracle.Oracle`` and raises AssertionError
on a mismatch.  The pins are (a) hand-derived worked examples stored under
``tests/golden/``, (b) an independent library routine (numpy's IEEE binary16
conversion, numpy's structured-dtype decoding of the bytes, scipy's logistic
function), (c) closed forms (all-ones and one-hot x, permutation matrices,
constant RMSNorm input) and (d) exact brute force: packed bytes built directly
with power-of-two scales and small-integer x, where every product and partial
sum is an exact dyadic rational, compared with Python integer arithmetic.

The same checks run against mutants of the oracle source in
``test_oracle_mutants.py``: every planted mistake must fail one of them.
"""
import os
from fractions import Fraction

import numpy as np

import oracle as _o

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

Q8_0, Q4_0, Q4_K = _o.Q8_0, _o.Q4_0, _o.Q4_K
QNAMES = {"q8_0": Q8_0, "q4_0": Q4_0, "q4_k": Q4_K}


# --------------------------------------------------------------------------
# independent decoding of the packed bytes (numpy structured dtypes)
# --------------------------------------------------------------------------
Q8_DT = np.dtype([("d", "<f2"), ("q", "i1", (32,))])
Q4_DT = np.dtype([("d", "<f2"), ("qs", "u1", (16,))])


def decode_independent(qtype, Wq, M, K):
    """(d [M, nb] float64, ints [M, K] int64) by reinterpreting the bytes."""
    nb = K // 32
    raw = np.ascontiguousarray(Wq, dtype=np.uint8).reshape(-1)
    if qtype == Q8_0:
        blk = raw.view(Q8_DT).reshape(M, nb)
        ints = blk["q"].astype(np.int64).reshape(M, K)
    else:
        blk = raw.view(Q4_DT).reshape(M, nb)
        qs = blk["qs"].astype(np.int64)
        ints = np.concatenate([qs & 0xF, qs >> 4], axis=-1).reshape(M, K) - 8
    return blk["d"].astype(np.float64), ints


def dequant_independent(qtype, Wq, M, K):
    if qtype == Q4_K:
        return q4k_dequant_independent(Wq, M, K)
    d, ints = decode_independent(qtype, Wq, M, K)
    return np.repeat(d, 32, axis=1) * ints


# Q4_K, the GGUF super-block as read in the oracle's header: 144 bytes per 256
# weights, decoded here with array slicing instead of per-element indexing
def q4k_decode_independent(Wq, M, K):
    """(d [M, ns], dmin [M, ns], sc [M, ns, 8], mn [M, ns, 8], q [M, ns, 8, 32])"""
    ns = K // 256
    sb = np.ascontiguousarray(Wq, dtype=np.uint8).reshape(M, ns, 144)
    d = sb[..., 0:2].copy().view("<f2")[..., 0].astype(np.float64)
    dmin = sb[..., 2:4].copy().view("<f2")[..., 0].astype(np.float64)
    s = sb[..., 4:16].astype(np.int64)
    sc = np.concatenate([s[..., 0:4] & 63, (s[..., 8:12] & 15) | ((s[..., 0:4] >> 6) << 4)], -1)
    mn = np.concatenate([s[..., 4:8] & 63, (s[..., 8:12] >> 4) | ((s[..., 4:8] >> 6) << 4)], -1)
    qs = sb[..., 16:].reshape(M, ns, 4, 32).astype(np.int64)
    q = np.stack([qs & 15, qs >> 4], axis=3).reshape(M, ns, 8, 32)
    return d, dmin, sc, mn, q


def q4k_dequant_independent(Wq, M, K):
    d, dmin, sc, mn, q = q4k_decode_independent(Wq, M, K)
    w = (d[..., None, None] * sc[..., None]) * q - (dmin[..., None] * mn)[..., None]
    return w.reshape(M, K)


def _round_away(v):
    """C roundf of fp32 values, in fp64 (exact for fp32 inputs)."""
    v = np.asarray(v, dtype=np.float64)
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


def q4k_quantize_independent(W):
    """The Q4_K packer's reading, vectorised in numpy fp32 (IEEE, correctly
    rounded divisions; float16 casts round to nearest even): per sub-block
    lo = min(0, min w), hi = max w, scale = (hi - lo)/15, min = -lo; d and
    dmin = fp16(max / 63) (+0 when every term is zero); sc, m, q rounded half
    away from zero and clamped."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    M, K = W.shape
    ns = K // 256
    f32 = np.float32
    w = W.reshape(M, ns, 8, 32)
    lo = np.minimum(w.min(-1), f32(0))
    hi = w.max(-1)
    scale = (hi - lo) / f32(15)
    mins = -lo
    smax = scale.max(-1) + f32(0)  # + 0 turns a -0 into +0
    mmax = mins.max(-1) + f32(0)
    dh = (smax / f32(63)).astype(np.float16)
    mh = (mmax / f32(63)).astype(np.float16)
    df, mf = dh.astype(f32), mh.astype(f32)
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(df[..., None] != 0, np.clip(_round_away(scale / df[..., None]), 0, 63), 0)
        mn = np.where(mf[..., None] != 0, np.clip(_round_away(mins / mf[..., None]), 0, 63), 0)
        sc, mn = sc.astype(np.int64), mn.astype(np.int64)
        D = df[..., None] * sc.astype(f32)
        Mf = mf[..., None] * mn.astype(f32)
        v = (w + Mf[..., None]) / D[..., None]
        q = np.where(D[..., None] != 0, np.clip(_round_away(v), 0, 15), 0).astype(np.int64)
    out = np.zeros((M, ns, 144), np.uint8)
    out[..., 0:2] = dh.view(np.uint8).reshape(M, ns, 2)
    out[..., 2:4] = mh.view(np.uint8).reshape(M, ns, 2)
    out[..., 4:8] = sc[..., :4] | ((sc[..., 4:] >> 4) << 6)
    out[..., 8:12] = mn[..., :4] | ((mn[..., 4:] >> 4) << 6)
    out[..., 12:16] = (sc[..., 4:] & 15) | ((mn[..., 4:] & 15) << 4)
    qq = q.reshape(M, ns, 4, 2, 32)
    out[..., 16:] = (qq[:, :, :, 0, :] | (qq[:, :, :, 1, :] << 4)).reshape(M, ns, 128)
    return out.reshape(M, ns * 144)


# --------------------------------------------------------------------------
# golden fixtures
# --------------------------------------------------------------------------
def load_golden(name):
    rec = {"w": [], "packed": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "qtype":
                rec["qtype"] = QNAMES[vals[0]]
            elif key in ("M", "K"):
                rec[key] = int(vals[0])
            elif key == "w":
                rec["w"].append([float(v) for v in vals])
            elif key == "packed":
                rec["packed"].append([int(v, 16) for v in vals])
            elif key == "x_ones_y":
                rec["x_ones_y"] = [float(v) for v in vals]
    rec["w"] = np.array(rec["w"], dtype=np.float32)
    rec["packed"] = np.array(rec["packed"], dtype=np.uint8)
    return rec


GOLDEN_FILES = ("q8_0_example_a.txt", "q4_0_example_b.txt", "q4_k_example_c.txt")


def check_golden(o):
    for name in GOLDEN_FILES:
        g = load_golden(name)
        got = o.quantize_pack(g["qtype"], g["w"])
        assert np.array_equal(got, g["packed"]), f"{name}: packed bytes differ\n{got}"
        y, S = o.gemv(g["qtype"], g["packed"], g["M"], g["K"], np.ones(g["K"]))
        assert list(y) == g["x_ones_y"], f"{name}: y={y} want {g['x_ones_y']}"
        # with x = ones, S is the sum of |dequantized weights|
        wdq = dequant_independent(g["qtype"], g["packed"], g["M"], g["K"])
        assert np.array_equal(S, np.abs(wdq).sum(axis=1)), f"{name}: S={S}"


# --------------------------------------------------------------------------
# fp16 conversion
# --------------------------------------------------------------------------
# (fp32 value, binary16 bits), derived by hand from IEEE-754 binary16
FP16_POINTS = [
    (0.0, 0x0000), (-0.0, 0x8000), (1.0, 0x3C00), (-2.0, 0xC000),
    (1.0 / 128, 0x2000), (1.0 / 64, 0x2400), (0.25, 0x3400), (0.125, 0x3000),
    (np.float32(1.0) / np.float32(127.0), 0x2008),  # 1/127 -> 2^-7*(1+8/1024)
    (65504.0, 0x7BFF), (65519.0, 0x7BFF), (65520.0, 0x7C00),  # 65520 is a tie -> even=Inf
    (2.0 ** -14, 0x0400), (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000),  # tie -> even 0
    (1.5 * 2.0 ** -25, 0x0001), (3.0 * 2.0 ** -25, 0x0002),  # 1.5 ulp tie -> even 2
    (1.0 + 2.0 ** -11, 0x3C00), (1.0 + 3 * 2.0 ** -11, 0x3C02),  # ties to even
    (float("inf"), 0x7C00), (float("-inf"), 0xFC00),
]


def check_fp16_points(o):
    for v, bits in FP16_POINTS:
        got = int(o.lib.bqo_f32_to_f16_bits(float(np.float32(v))))
        assert got == bits, f"f16({v!r}) = {got:#06x}, want {bits:#06x}"
    for bits, v in [(0x3C00, 1.0), (0x2008, 0.00787353515625), (0x0001, 2.0 ** -24),
                    (0x7BFF, 65504.0), (0x8400, -(2.0 ** -14)), (0x3555, 0.333251953125)]:
        assert o.f16_bits_to_f64(bits) == v, f"f16 bits {bits:#06x} -> {o.f16_bits_to_f64(bits)}"


def _compare_fp16(o, u32):
    f = u32.view(np.float32)
    with np.errstate(all="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    got = o.f32_to_f16_bits(f)
    nan = np.isnan(f)
    bad = (got != ref) & ~nan
    assert not bad.any(), (
        f"f16 mismatch at fp32 bits {u32[bad][:4]}: got {got[bad][:4]} want {ref[bad][:4]}")
    if nan.any():  # any NaN encoding is acceptable; it must stay a NaN
        g = got[nan]
        assert np.all(((g & 0x7C00) == 0x7C00) & ((g & 0x3FF) != 0)), "NaN lost"


def check_fp16_vs_numpy(o, exhaustive=True):
    """Against numpy's float32->float16 cast (IEEE RNE).  Exhaustive mode
    covers every positive fp32 whose exponent field is 100..143 (all inputs
    whose result is a nonzero finite half, or rounds across the zero or
    overflow boundary); everything else, and the negative half, by stride."""
    step = 1 if exhaustive else 997
    chunk = 1 << 23
    for be in range(100, 144):
        base = np.uint32(be << 23)
        u = np.arange(0, chunk, step, dtype=np.uint32) + base
        _compare_fp16(o, u)
        _compare_fp16(o, u[::13] | np.uint32(0x80000000))
    # the rest of the fp32 line: zero / subnormal-f32 / huge / Inf / NaN
    rest = np.arange(0, 1 << 32, 65521, dtype=np.uint64).astype(np.uint32)
    _compare_fp16(o, rest)
    _compare_fp16(o, np.array([0x7F800000, 0xFF800000, 0x7FC00000, 0x7F800001, 0x00000001,
                               0x33000000, 0x33000001, 0x387FE000, 0x387FF000],
                              dtype=np.uint32))


# --------------------------------------------------------------------------
# pack / dequant round trip
# --------------------------------------------------------------------------
def _random_weights(rng, M, K):
    w = rng.standard_normal((M, K)).astype(np.float32) * np.float32(0.02)
    # a spread of block magnitudes, down to fp16-subnormal scales, and a few
    # all-zero blocks
    scale = (2.0 ** rng.integers(-30, 8, size=(M, K // 32, 1))).astype(np.float32)
    w = (w.reshape(M, K // 32, 32) * scale).reshape(M, K)
    w[0, :32] = 0.0
    return np.ascontiguousarray(w)


def check_roundtrip(o, rng=None):
    rng = rng or np.random.default_rng(1)
    M, K = 37, 256
    W = _random_weights(rng, M, K)
    for qt in (Q8_0, Q4_0):
        P = o.quantize_pack(qt, W)
        d, ints = decode_independent(qt, P, M, K)
        df = np.repeat(d, 32, axis=1)
        deq = o.dequant(qt, P, M, K)
        assert np.array_equal(deq, df * ints), "dequant disagrees with byte decoding"
        err = np.abs(deq - W.astype(np.float64))
        blocks_amax = np.abs(W.reshape(M, -1, 32)).max(-1)
        # scale rule: d = fp16(amax / 127) or fp16(amax / 8), fp32 division
        div = np.float32(127.0) if qt == Q8_0 else np.float32(8.0)
        with np.errstate(all="ignore"):
            want_d = (blocks_amax.astype(np.float32) / div).astype(np.float16)
        assert np.array_equal(d.astype(np.float16), want_d), "scale rule"
        tol = df * (0.5 + 2.0 ** -16)
        w64 = W.astype(np.float64)
        # an fp16-subnormal scale can sit far from amax/127 (or amax/8), so
        # the clamp can bind beyond the usual +-127.5 d (or 7.5 d / -8.5 d)
        if qt == Q8_0:
            inside = np.abs(w64) <= 127.5 * df
            assert np.all(err[inside] <= tol[inside]), "Q8_0: |w' - w| > d/2"
            assert np.all(deq[~inside] == np.sign(w64[~inside]) * 127 * df[~inside]), \
                "Q8_0: clamp gives +-127 d"
            assert np.all(np.abs(ints) <= 127), "Q8_0 code outside [-127, 127]"
            normal = d >= 2.0 ** -14
            assert np.all(np.abs(ints).reshape(M, -1, 32).max(-1)[normal] == 127), \
                "Q8_0: the max-|w| element must map to +-127"
        else:
            hi, lo = w64 >= 7.5 * df, w64 < -8.5 * df
            inside = ~hi & ~lo
            assert np.all(err[inside] <= tol[inside]), "Q4_0: |w' - w| > d/2"
            assert np.all(deq[hi] == 7 * df[hi]), "Q4_0: clamp above 7.5d gives 7d"
            assert np.all(deq[lo] == -8 * df[lo]), "Q4_0: clamp below -8.5d gives -8d"
            assert np.all((ints >= -8) & (ints <= 7)), "Q4_0 code outside [-8, 7]"
        zero_blk = d == 0
        assert np.all(ints.reshape(M, -1, 32)[zero_blk] == 0), "d == 0 gives zero codes"
    # idempotence: Q8_0 always; Q4_0 for blocks that hold an n = 0 code
    P = o.quantize_pack(Q8_0, W)
    P2 = o.quantize_pack(Q8_0, o.dequant(Q8_0, P, M, K).astype(np.float32))
    d8, _ = decode_independent(Q8_0, P, M, K)
    keep = ((d8 >= 2.0 ** -14) | (d8 == 0)).reshape(-1)  # max code is +-127 there
    assert keep.sum() > 0.6 * keep.size
    assert np.array_equal(P.reshape(-1, 34)[keep], P2.reshape(-1, 34)[keep]), \
        "Q8_0 pack(dequant(pack(w))) != pack(w)"
    P = o.quantize_pack(Q4_0, W)
    P2 = o.quantize_pack(Q4_0, o.dequant(Q4_0, P, M, K).astype(np.float32))
    _, ints = decode_independent(Q4_0, P, M, K)
    has_min = (ints.reshape(M, -1, 32) == -8).any(-1).reshape(-1)
    b1 = P.reshape(-1, 18)[has_min]
    b2 = P2.reshape(-1, 18)[has_min]
    assert np.array_equal(b1, b2), "Q4_0 blocks with an n=0 code must repack identically"
    # the literal +amax rule is not idempotent: [2, 0, ...] -> 7d -> new scale
    one = np.zeros((1, 32), np.float32)
    one[0, 0] = 2.0
    p1 = o.quantize_pack(Q4_0, one)
    p2 = o.quantize_pack(Q4_0, o.dequant(Q4_0, p1, 1, 32).astype(np.float32))
    assert p1[0, :2].tolist() == [0x00, 0x34] and p2[0, :2].tolist() == [0x00, 0x33], \
        f"Q4_0 +amax clamp then repack: {p1[0, :3]} -> {p2[0, :3]}"


# --------------------------------------------------------------------------
# GEMV closed forms and brute force
# --------------------------------------------------------------------------
D_BITS = {0x3400: Fraction(1, 4), 0x3800: Fraction(1, 2), 0x3C00: Fraction(1),
          0x4000: Fraction(2), 0x4400: Fraction(4)}


def _direct_blocks(rng, qtype, M, K):
    """Packed bytes built without the packer: d in {2^-2..2^2}, codes over
    their full byte range (Q8_0 includes -128, which a decoder must accept)."""
    nb = K // 32
    dsel = rng.choice(list(D_BITS), size=(M, nb))
    if qtype == Q8_0:
        blk = np.zeros((M, nb), Q8_DT)
        blk["q"] = rng.integers(-128, 128, size=(M, nb, 32))
    else:
        blk = np.zeros((M, nb), Q4_DT)
        blk["qs"] = rng.integers(0, 256, size=(M, nb, 16))
    raw = blk.view(np.uint8).reshape(M, nb, -1)
    raw[:, :, 0] = dsel & 0xFF
    raw[:, :, 1] = dsel >> 8
    return np.ascontiguousarray(raw.reshape(M, -1)), dsel


def _exact_gemv(qtype, raw, dsel, M, K, x_int):
    """Python-integer statement: y_m = sum_b d_b * sum_j code_bj * x_j."""
    nb = K // 32
    out = []
    for m in range(M):
        acc = Fraction(0)
        for b in range(nb):
            body = raw[m, b * (raw.shape[1] // nb) + 2:(b + 1) * (raw.shape[1] // nb)]
            if qtype == Q8_0:
                codes = [int(v) - 256 if v >= 128 else int(v) for v in body]
            else:
                codes = [int(v) & 0xF for v in body] + [int(v) >> 4 for v in body]
                codes = [c - 8 for c in codes]
            acc += D_BITS[int(dsel[m, b])] * sum(c * int(x_int[32 * b + j])
                                                  for j, c in enumerate(codes))
        out.append(acc)
    return out


def check_bruteforce(o, rng=None):
    rng = rng or np.random.default_rng(2)
    for qt in (Q8_0, Q4_0):
        for M in (1, 2, 3, 7, 33):
            for K in (32, 64, 256, 288, 512):
                raw, dsel = _direct_blocks(rng, qt, M, K)
                x = rng.integers(-2, 3, size=K)
                y, _ = o.gemv(qt, raw, M, K, x.astype(np.float64))
                want = _exact_gemv(qt, raw, dsel, M, K, x)
                assert [Fraction(v) for v in y] == want, f"qt={qt} M={M} K={K}"
        # every (position, value) one-hot pattern on one block
        raw, dsel = _direct_blocks(rng, qt, 1, 32)
        for j in range(32):
            for v in (-2, -1, 1, 2):
                x = np.zeros(32, np.int64)
                x[j] = v
                y, S = o.gemv(qt, raw, 1, 32, x.astype(np.float64))
                want = _exact_gemv(qt, raw, dsel, 1, 32, x)[0]
                assert Fraction(y[0]) == want and Fraction(S[0]) == abs(want), \
                    f"qt={qt} one-hot j={j} v={v}"


def check_all_codes(o):
    """Every Q8_0 byte and every Q4_0 nibble against its integer meaning."""
    for dbits, d in D_BITS.items():
        blk = np.zeros((8, 34), np.uint8)
        blk[:, 0], blk[:, 1] = dbits & 0xFF, dbits >> 8
        blk[:, 2:] = np.arange(256, dtype=np.uint8).reshape(8, 32)
        deq = o.dequant(Q8_0, blk.reshape(-1), 8, 32)
        want = np.array([float(d) * (c - 256 if c >= 128 else c) for c in range(256)]).reshape(8, 32)
        assert np.array_equal(deq, want), "Q8_0 code table"
        blk = np.zeros((1, 18), np.uint8)
        blk[0, 0], blk[0, 1] = dbits & 0xFF, dbits >> 8
        blk[0, 2:] = [(lo | ((15 - lo) << 4)) for lo in range(16)]
        deq = o.dequant(Q4_0, blk.reshape(-1), 1, 32)
        want = [float(d) * (n - 8) for n in range(16)] + [float(d) * (7 - n) for n in range(16)]
        assert deq[0].tolist() == want, "Q4_0 nibble table (low = j, high = j+16)"


def check_closed_forms(o, rng=None):
    rng = rng or np.random.default_rng(3)
    M, K = 48, 288
    W = _random_weights(rng, M, K)
    for qt in (Q8_0, Q4_0):
        P = o.quantize_pack(qt, W)
        d, ints = decode_independent(qt, P, M, K)
        # all-ones x: y_m = sum_b d_b * (integer sum of the block's codes)
        y, _ = o.gemv(qt, P, M, K, np.ones(K))
        want = (d * ints.reshape(M, -1, 32).sum(-1)).sum(-1)
        assert np.allclose(y, want, rtol=1e-14, atol=0), "all-ones x"
        # one-hot x = e_k gives column k exactly
        deq = dequant_independent(qt, P, M, K)
        for k in (0, 1, 31, 32, 100, K - 1):
            e = np.zeros(K)
            e[k] = 1.0
            y, S = o.gemv(qt, P, M, K, e)
            assert np.array_equal(y, deq[:, k]) and np.array_equal(S, np.abs(deq[:, k])), \
                f"one-hot column {k}"
    # permutation matrix (not an involution, so a transposed operand shows)
    n = 96
    perm = np.roll(np.arange(n), 5)
    perm[:7] = perm[:7][::-1]
    Pm = np.zeros((n, n), np.float32)
    Pm[np.arange(n), perm] = 1.0
    x = rng.standard_normal(n).astype(np.float32)
    # Q8_0: d = fp16(1/127) = 0x2008 = 0.00787353515625, q = 127
    y, _ = o.gemv(Q8_0, o.quantize_pack(Q8_0, Pm), n, n, x.astype(np.float64))
    assert np.array_equal(y, 0.00787353515625 * 127 * x[perm].astype(np.float64)), "Q8_0 P x"
    # Q4_0: d = 1/8, +1 clamps to n=15 -> 7/8;  -1 -> n=0 -> exactly -1
    y, _ = o.gemv(Q4_0, o.quantize_pack(Q4_0, Pm), n, n, x.astype(np.float64))
    assert np.array_equal(y, 0.875 * x[perm].astype(np.float64)), "Q4_0 P x"
    y, _ = o.gemv(Q4_0, o.quantize_pack(Q4_0, -Pm), n, n, x.astype(np.float64))
    assert np.array_equal(y, -x[perm].astype(np.float64)), "Q4_0 -P x"


# --------------------------------------------------------------------------
# RMSNorm, SiLU, gate+up
# --------------------------------------------------------------------------
def check_norm_silu(o, rng=None):
    from scipy.special import expit
    rng = rng or np.random.default_rng(4)
    K = 256
    gamma = 1.0 + 0.1 * rng.standard_normal(K)
    for c, eps in ((0.5, 1e-6), (3.0, 0.0), (-2.0, 1e-2)):
        xn = o.rmsnorm(np.full(K, c), gamma, eps)
        want = gamma * c / np.sqrt(c * c + eps)
        assert np.allclose(xn, want, rtol=1e-15, atol=0), f"rmsnorm const c={c} eps={eps}"
    # alternating +-c: mean square is still c^2; gamma=None means ones
    xa = np.where(np.arange(K) % 2 == 0, 1.5, -1.5)
    assert np.allclose(o.rmsnorm(xa, None, 0.25), xa / np.sqrt(2.25 + 0.25), rtol=1e-15)
    # a two-level input: mean square (a^2 + b^2)/2
    xb = np.where(np.arange(K) < K // 2, 1.0, 3.0)
    assert np.allclose(o.rmsnorm(xb, None, 0.0), xb / np.sqrt(5.0), rtol=1e-15)
    for z in (-30.0, -4.5, -1.0, -1e-3, 0.0, 0.7, 2.4, 12.0):
        s = o.silu(z)
        assert abs(s - z * expit(z)) <= 1e-15 * max(1.0, abs(z)), f"silu({z})"
        assert abs((s - o.silu(-z)) - z) <= 1e-14 * max(1.0, abs(z)), "silu(z)-silu(-z)=z"
    # gate+up on permutation weights: g = c8 * xn[p], u = c8 * xn[q]
    n = 64
    p = np.roll(np.arange(n), 3)
    q = np.roll(np.arange(n), -9)
    Wg = np.zeros((n, n), np.float32)
    Wg[np.arange(n), p] = 1.0
    Wu = np.zeros((n, n), np.float32)
    Wu[np.arange(n), q] = 1.0
    x = rng.standard_normal(n)
    xn = o.rmsnorm(x, None, 1e-6)
    r = o.gate_up_silu(Q8_0, o.quantize_pack(Q8_0, Wg), o.quantize_pack(Q8_0, Wu), n, n, xn)
    c8 = 0.00787353515625 * 127
    g, u = c8 * xn[p], c8 * xn[q]
    assert np.array_equal(r["g"], g) and np.array_equal(r["u"], u), "gate/up operands"
    assert np.allclose(r["y"], g * expit(g) * u, rtol=1e-14, atol=0), "silu(g) * u"
    assert np.array_equal(r["Sg"], np.abs(g)) and np.array_equal(r["Su"], np.abs(u))


def check_bias(o, rng=None):
    """The q|k|v + bias projection: with x = 0 the output is the bias exactly
    (and S = |bias|); with no bias it is the plain GEMV; with power-of-two
    scales, small-integer x and integer biases every value is an exact dyadic
    rational, compared with Python's exact arithmetic row by row."""
    rng = rng or np.random.default_rng(41)
    for qt in (Q8_0, Q4_0):
        M, K = 7, 96
        raw, dsel = _direct_blocks(rng, qt, M, K)
        bias = rng.integers(-9, 10, size=M).astype(np.float64)
        y0, S0 = o.gemv_bias(qt, raw, M, K, np.zeros(K), bias)
        assert np.array_equal(y0, bias) and np.array_equal(S0, np.abs(bias)), "x = 0"
        x = rng.integers(-2, 3, size=K).astype(np.float64)
        yb, Sb = o.gemv_bias(qt, raw, M, K, x, None)
        yg, Sg = o.gemv(qt, raw, M, K, x)
        assert np.array_equal(yb, yg) and np.array_equal(Sb, Sg), "no bias"
        y, S = o.gemv_bias(qt, raw, M, K, x, bias)
        want = _exact_gemv(qt, raw, dsel, M, K, x.astype(np.int64))
        for m in range(M):
            assert Fraction(y[m]) == want[m] + Fraction(int(bias[m])), f"row {m}"
        assert np.array_equal(S, Sg + np.abs(bias)), "S includes |bias|"


def check_gemv_f16(o, rng=None):
    """The unquantized fp16-weight GEMV, anchored outside the oracle: weights
    k/8 (|k| <= 40, exact in fp16) against small-integer x compared with
    Python's exact arithmetic row by row (y and S); one-hot x = e_k returns
    column k as numpy's float16 decoder reads it (an independent decoder);
    the identity returns x; x = 0 returns zeros."""
    rng = rng or np.random.default_rng(51)
    M, K = 9, 40
    ints = rng.integers(-40, 41, size=(M, K))
    W = (ints / 8.0).astype(np.float16)
    x = rng.integers(-3, 4, size=K).astype(np.float64)
    y, S = o.gemv_f16(W.view(np.uint16), x)
    for m in range(M):
        terms = [Fraction(int(ints[m, k]), 8) * int(x[k]) for k in range(K)]
        assert Fraction(y[m]) == sum(terms), f"row {m}"
        assert Fraction(S[m]) == sum(abs(t) for t in terms), f"S row {m}"
    Wr = (rng.standard_normal((M, K)) * 0.02).astype(np.float16)
    for k in (0, 17, K - 1):
        e = np.zeros(K)
        e[k] = 1.0
        y, _ = o.gemv_f16(Wr.view(np.uint16), e)
        assert np.array_equal(y, Wr[:, k].astype(np.float64)), f"column {k}"
    xr = rng.standard_normal(K)
    y, _ = o.gemv_f16(np.eye(K, dtype=np.float16).view(np.uint16), xr)
    assert np.array_equal(y, xr), "identity"
    y, S = o.gemv_f16(Wr.view(np.uint16), np.zeros(K))
    assert not y.any() and not S.any(), "x = 0"


# --------------------------------------------------------------------------
# Q4_K
# --------------------------------------------------------------------------
def _q4k_weights(rng, M, K):
    """Weights that exercise the Q4_K packer: N(0, 0.02) scaled per sub-block
    by 2^-12..2^4, sub-blocks that are all positive, all negative, all zero,
    or hold -0.0, and a few ties."""
    w = rng.standard_normal((M, K)).astype(np.float32) * np.float32(0.02)
    sub = w.reshape(M, K // 32, 32)
    sub *= (2.0 ** rng.integers(-12, 5, size=(M, K // 32, 1))).astype(np.float32)
    kind = rng.integers(0, 8, size=(M, K // 32))
    sub[kind == 1] = np.abs(sub[kind == 1])
    sub[kind == 2] = -np.abs(sub[kind == 2])
    sub[kind == 3] = 0.0
    sub[kind == 4] = -0.0
    return np.ascontiguousarray(sub.reshape(M, K))


def check_q4k_independent(o, rng=None):
    """The oracle's Q4_K packing equals the independent numpy statement of
    the same reading byte for byte, and its dequant equals the independent
    decoder."""
    rng = rng or np.random.default_rng(11)
    for M, K in ((1, 256), (5, 512), (33, 1024), (3, 3584)):
        W = _q4k_weights(rng, M, K)
        P = o.quantize_pack(Q4_K, W)
        want = q4k_quantize_independent(W)
        bad = np.flatnonzero((P != want).any(axis=1))
        assert bad.size == 0, f"Q4_K pack {M}x{K}: rows {bad[:5]} differ"
        assert np.array_equal(o.dequant(Q4_K, P, M, K), q4k_dequant_independent(P, M, K)), \
            f"Q4_K dequant {M}x{K}"
    assert o.packed_bytes(Q4_K, 7, 512) == 7 * 2 * 144 and o.packed_bytes(Q4_K, 1, 288) == -1


def check_q4k_roundtrip(o, rng=None):
    """|dequant(pack(w)) - w| <= (d sc)/2 wherever the code is not clamped;
    a clamped code sits at the end of the range it was clamped to."""
    rng = rng or np.random.default_rng(12)
    M, K = 24, 1024
    W = _q4k_weights(rng, M, K)
    P = o.quantize_pack(Q4_K, W)
    d, dmin, sc, mn, q = q4k_decode_independent(P, M, K)
    D = (d[..., None] * sc)[..., None]
    Mf = (dmin[..., None] * mn)[..., None]
    w = W.reshape(M, K // 256, 8, 32).astype(np.float64)
    v = w + Mf  # the code's target times D
    err = np.abs(D * q - v)
    inside = (v >= -0.5 * D) & (v <= 15.5 * D)
    tol = 0.5 * D * (1 + 1e-6) + 1e-6 * np.abs(v)
    assert np.all(err[inside & (D > 0)] <= tol[inside & (D > 0)]), "Q4_K round trip"
    assert np.all(q[(v > 15.5 * D * (1 + 1e-6)) & (D > 0)] == 15), "Q4_K clamp at 15"
    assert np.all(q[(v < -0.5 * D * (1 + 1e-6)) & (D > 0)] == 0), "Q4_K clamp at 0"
    # the sub-block scales follow the data: the largest sub-block range takes sc = 63
    rng_w = w.max(-1) - np.minimum(w.min(-1), 0.0)
    big = rng_w == rng_w.max(-1, keepdims=True)
    assert np.all(sc[big & (rng_w > 0)] >= 62), "Q4_K scale of the widest sub-block"


Q4K_D = {0x3400: Fraction(1, 4), 0x3800: Fraction(1, 2), 0x3C00: Fraction(1), 0x2C00: Fraction(1, 16)}


def _q4k_direct(rng, M, K):
    """Q4_K bytes built without the packer (numpy bit assembly): d and dmin
    powers of two, 6-bit scales and mins and 4-bit codes over their full
    ranges.  Returns the bytes and their exact meaning as Fractions."""
    ns = K // 256
    keys = list(Q4K_D)
    dsel = rng.choice(keys, size=(M, ns))
    msel = rng.choice(keys, size=(M, ns))
    sc = rng.integers(0, 64, size=(M, ns, 8))
    mn = rng.integers(0, 64, size=(M, ns, 8))
    q = rng.integers(0, 16, size=(M, ns, 8, 32))
    out = np.zeros((M, ns, 144), np.uint8)
    out[..., 0], out[..., 1] = dsel & 0xFF, dsel >> 8
    out[..., 2], out[..., 3] = msel & 0xFF, msel >> 8
    out[..., 4:8] = sc[..., :4] | ((sc[..., 4:] >> 4) << 6)
    out[..., 8:12] = mn[..., :4] | ((mn[..., 4:] >> 4) << 6)
    out[..., 12:16] = (sc[..., 4:] & 15) | ((mn[..., 4:] & 15) << 4)
    qq = q.reshape(M, ns, 4, 2, 32)
    out[..., 16:] = (qq[:, :, :, 0, :] | (qq[:, :, :, 1, :] << 4)).reshape(M, ns, 128)
    return out.reshape(M, ns * 144), dsel, msel, sc, mn, q


def check_q4k_bruteforce(o, rng=None):
    """Exact Q4_K products: power-of-two d and dmin and small-integer x make
    every product and sum a dyadic rational, computed here with Fractions;
    y, S = sum|w x| and the split scale SK must equal them exactly."""
    rng = rng or np.random.default_rng(13)
    for M, K in ((1, 256), (3, 512), (2, 768)):
        raw, dsel, msel, sc, mn, q = _q4k_direct(rng, M, K)
        x = rng.integers(-2, 3, size=K)
        y, S = o.gemv(Q4_K, raw, M, K, x.astype(np.float64))
        SK = o.q4_k_split_scale(raw, M, K, x.astype(np.float64))
        for m in range(M):
            acc = s_abs = s_split = Fraction(0)
            for b in range(K // 256):
                d, dm = Q4K_D[int(dsel[m, b])], Q4K_D[int(msel[m, b])]
                for j in range(8):
                    for i in range(32):
                        xi = int(x[256 * b + 32 * j + i])
                        wv = d * int(sc[m, b, j]) * int(q[m, b, j, i]) - dm * int(mn[m, b, j])
                        acc += wv * xi
                        s_abs += abs(wv * xi)
                        s_split += d * int(sc[m, b, j]) * abs(int(q[m, b, j, i]) * xi) + \
                            dm * int(mn[m, b, j]) * abs(xi)
            assert Fraction(y[m]) == acc, f"Q4_K y {M}x{K} row {m}"
            assert Fraction(S[m]) == s_abs, f"Q4_K S {M}x{K} row {m}"
            assert Fraction(SK[m]) == s_split, f"Q4_K SK {M}x{K} row {m}"
    # one-hot x picks column k of the dequantized matrix exactly
    raw, *_ = _q4k_direct(rng, 4, 512)
    deq = q4k_dequant_independent(raw, 4, 512)
    for k in (0, 31, 32, 255, 256, 300, 511):
        e = np.zeros(512)
        e[k] = 1.0
        y, _ = o.gemv(Q4_K, raw, 4, 512, e)
        assert np.array_equal(y, deq[:, k]), f"Q4_K one-hot column {k}"


QUICK_CHECKS = (check_golden, check_fp16_points, check_roundtrip, check_bruteforce,
                check_all_codes, check_closed_forms, check_norm_silu, check_bias, check_gemv_f16,
                check_q4k_independent, check_q4k_roundtrip, check_q4k_bruteforce)


def run_quick(o):
    """Names of the quick checks that fail for oracle ``o``."""
    failed = []
    for chk in QUICK_CHECKS:
        try:
            chk(o)
        except AssertionError:
            failed.append(chk.__name__)
    try:
        check_fp16_vs_numpy(o, exhaustive=False)
    except AssertionError:
        failed.append("check_fp16_vs_numpy")
    return failed
