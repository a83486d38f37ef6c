"""The fp64 oracle against what the pages and the mathematics fix (see
tests/oracle_pins.py for what each pin rests on).  CPU only."""
import numpy as np
import pytest

import oracle
from tests.oracle_pins import ALL_PINS, CONV_PINS, ZOH_PINS


@pytest.mark.parametrize("name", sorted(ALL_PINS))
def test_oracle_pin(name):
    fn, tol = ALL_PINS[name]
    err = fn(oracle.selective_scan_fwd)
    assert err <= tol, f"{name}: error {err:.3e} > {tol:.1e}"


def test_oracle_lti_with_skip():
    from tests.oracle_pins import pin_lti_direct
    assert pin_lti_direct(oracle.selective_scan_fwd, seed=5, skip=True) <= 1e-9


def test_oracle_threaded_split_is_identical():
    rng = np.random.default_rng(9)
    from tests.oracle_pins import random_problem
    p = random_problem(rng, 2, 17, 11, 4)
    args = (p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"],
            p["softplus"])
    y1, h1 = oracle.selective_scan_fwd(*args)
    y4, h4 = oracle.selective_scan_fwd_threads(*args, threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(h1, h4)


def test_oracle_empty_and_degenerate_sizes():
    A = -np.ones((3, 2))
    for L in (0, 1):
        u = np.ones((2, L, 3)); B = np.ones((2, L, 2))
        y, h = oracle.selective_scan_fwd(u, u, A, B, B)
        assert y.shape == (2, L, 3) and h.shape == (2, 3, 2)
        if L == 0:
            assert not np.any(h)
    # zero batch / zero channels
    y, h = oracle.selective_scan_fwd(np.ones((0, 4, 3)), np.ones((0, 4, 3)), A,
                                     np.ones((0, 4, 2)), np.ones((0, 4, 2)))
    assert y.shape == (0, 4, 3)


def test_oracle_rejects_bad_arguments():
    lib = oracle.load()
    assert lib.ssm_oracle_fwd(None, None, None, None, None, None, None, None, 0,
                              None, None, 1, 1, 1, 1) == -1


def test_oracle_decode_step_is_the_scan_at_one_token():
    from tests.oracle_pins import random_problem
    rng = np.random.default_rng(11)
    p = random_problem(rng, 3, 4, 5, 6)
    h = rng.standard_normal((3, 5, 6))
    y_ref, h_ref = oracle.selective_scan_fwd(p["u"][:, :1], p["delta"][:, :1], p["A"],
                                             p["B"][:, :1], p["C"][:, :1], p["D"],
                                             p["z"][:, :1], p["delta_bias"], True, h0=h)
    y, hn = oracle.selective_scan_step(h, p["u"][:, 0], p["delta"][:, 0], p["A"], p["B"][:, 0],
                                       p["C"][:, 0], p["D"], p["z"][:, 0], p["delta_bias"], True)
    assert np.array_equal(y, y_ref[:, 0]) and np.array_equal(hn, h_ref)


@pytest.mark.parametrize("name", sorted(CONV_PINS))
def test_oracle_conv_pin(name):
    fn, tol = CONV_PINS[name]
    err = fn(oracle.causal_conv_silu)
    assert err <= tol, f"{name}: error {err:.3e} > {tol:.1e}"


@pytest.mark.parametrize("name", sorted(ZOH_PINS))
def test_oracle_zoh_pin(name):
    fn, tol = ZOH_PINS[name]
    err = fn(oracle.selective_scan_fwd)
    assert err <= tol, f"{name}: error {err:.3e} > {tol:.1e}"


def test_oracle_backward_loop_forward():
    from tests.oracle_pins import pin_bwd_loop_forward
    assert pin_bwd_loop_forward() <= 1e-13


def test_oracle_backward_finite_differences():
    from oracle.backward import selective_scan_bwd
    from tests.oracle_pins import pin_bwd_finite_differences
    assert pin_bwd_finite_differences(selective_scan_bwd) <= 1e-7


def test_oracle_backward_catches_a_wrong_gradient():
    """The finite-difference pin rejects a gradient with one term wrong."""
    from oracle.backward import selective_scan_bwd
    from tests.oracle_pins import pin_bwd_finite_differences

    def broken(*a):
        g = selective_scan_bwd(*a)
        g["B"] = g["B"] * 1.01
        return g
    assert pin_bwd_finite_differences(broken) > 1e-5


def test_backward_with_states_matches_finite_differences():
    from oracle.backward import selective_scan_bwd
    from tests.oracle_pins import pin_bwd_state_finite_differences
    assert pin_bwd_state_finite_differences(selective_scan_bwd) <= 1e-7


def test_backward_chains_through_the_state():
    from oracle.backward import selective_scan_bwd
    from tests.oracle_pins import pin_bwd_chaining
    assert pin_bwd_chaining(selective_scan_bwd) <= 1e-12


def test_state_finite_differences_reject_a_dropped_terminal_gradient():
    """A backward that ignores dh_last fails the pin."""
    from oracle.backward import selective_scan_bwd
    from tests.oracle_pins import pin_bwd_state_finite_differences

    def broken(*a, h0=None, dh_last=None):
        return selective_scan_bwd(*a, h0=h0)
    assert pin_bwd_state_finite_differences(broken) > 1e-3
