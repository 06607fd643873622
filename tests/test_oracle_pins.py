"""The oracle against facts outside itself (CPU only)."""
import numpy as np
import pytest

import oracle
import oracle_pins as P
from oracle import merge as om


def test_brute_force():
    P.pin_brute_force()


def test_worked_example(golden_dir):
    P.pin_worked_example(golden_dir)


def test_closed_forms():
    P.pin_closed_forms()


def test_invariants():
    P.pin_invariants()


def test_merge_algebra_and_blocks():
    P.pin_merge()


def test_ring_restatement_equals_single_pass():
    P.pin_ring()


def test_ring_backward_steps():
    P.pin_ring_backward()


def test_gradient_rows_match_whole_gradients():
    P.pin_gradient_rows()


def test_zigzag_map_and_step_cases(golden_dir):
    P.pin_zigzag_map(golden_dir)


def test_bf16_input_path_exact():
    """bf16 bit patterns widen exactly: the oracle on bf16 bits == the oracle on their f64 values."""
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 1, 2, 19, 8)).astype(np.float32)
    bits = oracle.f32_to_bf16_bits(x)
    wide = oracle.bf16_bits_to_f64(bits)
    o1, l1 = oracle.attention(bits[0], bits[1], bits[2], True, 0.25)
    o2, l2 = oracle.attention(wide[0], wide[1], wide[2], True, 0.25)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # round-to-nearest-even: 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> stays at 1 (even)
    t = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5], np.float32)
    assert list(oracle.bf16_bits_to_f64(oracle.f32_to_bf16_bits(t))) == [1.0, 1.0 + 2.0 ** -6, -2.5]


def test_sampled_rows_match_full():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((2, 4, 37, 8))
    k = rng.standard_normal((2, 2, 37, 8))
    v = rng.standard_normal((2, 2, 37, 8))
    o, l = oracle.attention(q, k, v, True, 0.4)
    rows = np.array([[0, 0, 0], [1, 3, 36], [0, 2, 17], [1, 1, 5]])
    os_, ls = oracle.attention(q, k, v, True, 0.4, rows=rows)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(os_[n], o[b, h, i]) and ls[n] == l[b, h, i]


def test_thread_count_does_not_change_result():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 3, 50, 16))
    k = rng.standard_normal((1, 3, 50, 16))
    v = rng.standard_normal((1, 3, 50, 16))
    a = oracle.attention(q, k, v, True, 0.25, nthreads=1)
    b = oracle.attention(q, k, v, True, 0.25, nthreads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bad_arguments_rejected():
    q = np.zeros((1, 3, 4, 2))
    with pytest.raises(ValueError):
        oracle.attention(q, np.zeros((1, 2, 4, 2)), np.zeros((1, 2, 4, 2)), False)
    with pytest.raises(ValueError):
        oracle.attention(q, q, q, False, rows=[[0, 5, 0]])
    with pytest.raises(TypeError):
        oracle.attention(q.astype(np.int32), q, q, False)


def test_merge_identity_both_forms():
    o = np.ones((2, 3))
    l = np.array([0.5, -np.inf])
    ident = (np.zeros((2, 3)), np.full(2, -np.inf))
    for f in (om.merge, om.merge_sigmoid):
        mo, ml = f(*ident, o, l)
        assert np.array_equal(ml, l)
        assert np.array_equal(mo[0], o[0])


def test_varlen_block_diagonal():
    P.pin_varlen()


def test_backward_oracle():
    P.pin_backward()


def test_ulysses_oracle():
    P.pin_ulysses()
