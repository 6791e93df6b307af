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


def test_q4_k_packing_against_an_independent_statement():
    checks.check_q4k_independent(o())


def test_q4_k_round_trip():
    checks.check_q4k_roundtrip(o())


def test_q4_k_exact_products():
    checks.check_q4k_bruteforce(o())


def test_packed_bytes_and_bad_args():
    ob = o()
    assert ob.packed_bytes(oracle.Q8_0, 3072, 1024) == 3072 * 32 * 34
    assert ob.packed_bytes(oracle.Q4_0, 3584, 18944) == 3584 * 592 * 18
    assert ob.packed_bytes(oracle.Q8_0, 1, 33) == -1
    assert ob.packed_bytes(5, 1, 32) == -1


def test_parallel_drivers_give_the_single_threaded_values():
    """The threaded drivers split rows among host threads and call the same
    scalar routines, so every value equals the single-threaded oracle's."""
    import numpy as np

    ob = o()
    rng = np.random.default_rng(5)
    for qt in (oracle.Q8_0, oracle.Q4_0):
        for M, K in ((1, 32), (7, 288), (333, 1024)):
            W = (rng.standard_normal((M, K)) * 0.02).astype(np.float32)
            P = ob.quantize_pack(qt, W)
            for threads in (1, 3, 8):
                assert np.array_equal(ob.quantize_pack_parallel(qt, W, threads), P)
                x = rng.standard_normal(K)
                y, S = ob.gemv(qt, P, M, K, x)
                yp, Sp = ob.gemv_parallel(qt, P, M, K, x, threads)
                assert np.array_equal(y, yp) and np.array_equal(S, Sp)
    Wh = (rng.standard_normal((97, 136)) * 0.02).astype(np.float16).view(np.uint16)
    x = rng.standard_normal(136)
    y, S = ob.gemv_f16(Wh, x)
    yp, Sp = ob.gemv_f16_parallel(Wh, x, 5)
    assert np.array_equal(y, yp) and np.array_equal(S, Sp)
