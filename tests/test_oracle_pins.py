"""The oracle against its pins (CPU only).  See ``oracle_checks`` for what
each pin is anchored to."""
import oracle

import oracle_checks as checks


def o():
    return oracle.get()


def test_golden_worked_examples():
    checks.check_golden(o())


def test_fp16_hand_points():
    checks.check_fp16_points(o())


def test_fp16_exhaustive_against_numpy():
    checks.check_fp16_vs_numpy(o(), exhaustive=True)


def test_pack_dequant_round_trip():
    checks.check_roundtrip(o())


def test_gemv_bruteforce_exact():
    checks.check_bruteforce(o())


def test_every_code_value():
    checks.check_all_codes(o())


def test_gemv_closed_forms():
    checks.check_closed_forms(o())


def test_rmsnorm_silu_gate_up():
    checks.check_norm_silu(o())


def test_qkv_bias():
    checks.check_bias(o())


def test_gemv_f16():
    checks.check_gemv_f16(o())


def test_packed_bytes_and_bad_args():
    ob = o()
    assert ob.packed_bytes(oracle.Q8_0, 3072, 1024) == 3072 * 32 * 34
    assert ob.packed_bytes(oracle.Q4_0, 3584, 18944) == 3584 * 592 * 18
    assert ob.packed_bytes(oracle.Q8_0, 1, 33) == -1
    assert ob.packed_bytes(5, 1, 32) == -1
