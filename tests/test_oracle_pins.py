"""The fp64 oracle against what the blog and mathematics fix (CPU only).

Pins: brute-force unrolled sum, the A = 0 linear-attention closed form, dt = 0
state invariance, chunked == sequential at several chunk sizes (ragged
included), split-sequence hand-off, causality, group mapping, a scalar
geometric closed form, hand-worked fixtures and the stage-1 ramp.
"""
import numpy as np
import pytest

import oracle_pins as pins

PIN_NAMES = [
    "brute_force_y", "brute_force_final", "a0_recurrence_y", "a0_recurrence_final",
    "a0_chunked_y", "a0_chunked_final", "dt0_rec_final", "dt0_rec_y", "dt0_chunked_final",
    "dt0_chunked_y", "chunked_vs_rec_y", "chunked_vs_rec_final", "chunked_vs_rec_chunk_states",
    "split_y", "split_final", "causality", "groups_repeat", "geometric_y", "geometric_final",
    "golden_scalar_geometric", "golden_two_by_two", "cumsum_ramp",
]


@pytest.fixture(scope="module")
def suite(oracle_mod):
    return pins.run_suite(oracle_mod)


def test_suite_covers_every_pin(suite):
    assert sorted(suite) == sorted(PIN_NAMES)


@pytest.mark.parametrize("name", PIN_NAMES)
def test_pin(suite, name):
    assert suite[name] <= pins.TOL, f"{name}: error {suite[name]:.3e}"


def test_pairs_subset_matches_full(oracle_mod):
    """Computing only some (batch, head) pairs gives those pairs bit-identically."""
    p = pins.random_problem(11, 3, 17, 4, 3, 5, 2)
    full = oracle_mod.ssd_recurrence(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], init=p["init"])
    sub = oracle_mod.ssd_recurrence(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], init=p["init"],
                                    pairs=[(2, 1), (0, 3)])
    for b, h in ((2, 1), (0, 3)):
        assert np.array_equal(sub["y"][b, :, h], full["y"][b, :, h])
        assert np.array_equal(sub["final_state"][b, h], full["final_state"][b, h])
    assert not sub["y"][1].any()


def test_thread_count_does_not_change_result(oracle_mod):
    p = pins.random_problem(12, 2, 19, 3, 4, 3, 1)
    a = oracle_mod.ssd_chunked(p["x"], p["dt"], p["A"], p["B"], p["C"], 4, D=p["D"], init=p["init"],
                               nthreads=1)
    b = oracle_mod.ssd_chunked(p["x"], p["dt"], p["A"], p["B"], p["C"], 4, D=p["D"], init=p["init"],
                               nthreads=5)
    for k in ("y", "final_state", "chunk_states", "G"):
        assert np.array_equal(a[k], b[k])


def test_empty_sequence_keeps_state(oracle_mod):
    p = pins.random_problem(13, 1, 0, 2, 3, 4, 1)
    r = oracle_mod.ssd_recurrence(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], init=p["init"])
    assert r["y"].shape == (1, 0, 2, 3)
    assert np.array_equal(r["final_state"], p["init"])


def test_rejects_bad_group_count(oracle_mod):
    p = pins.random_problem(14, 1, 4, 3, 2, 2, 1)
    with pytest.raises(ValueError):
        oracle_mod.ssd_recurrence(p["x"], p["dt"], p["A"], np.repeat(p["B"], 2, axis=2),
                                  np.repeat(p["C"], 2, axis=2))


def _step_slice(p, t):
    """Token t of a problem, in the decode step's layouts."""
    return p["x"][:, t], p["dt"][:, t], p["B"][:, t], p["C"][:, t]


def test_step_matches_brute_force(oracle_mod):
    """The decode step against the unrolled expansion on a one-token problem
    (groups, S != H, a carried state: a transposed or mis-grouped operand fails)."""
    p = pins.random_problem(15, 2, 1, 4, 3, 5, 2)
    y, h = oracle_mod.ssd_step(*_step_slice(p, 0)[:2], p["A"], *_step_slice(p, 0)[2:], state=p["init"],
                               D=p["D"])
    y_bf, h_bf = pins.brute_force(p)
    assert pins.rel_err(y, y_bf[:, 0]) <= pins.TOL
    assert pins.rel_err(h, h_bf) <= pins.TOL


def test_steps_compose_to_the_recurrence(oracle_mod):
    """K decode steps from a prefill state equal the recurrence over the whole
    sequence, bit for bit (the state hand-off of the blog's §Kernel 2)."""
    p = pins.random_problem(16, 2, 9, 4, 3, 5, 2)
    full = oracle_mod.ssd_recurrence(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], init=p["init"])
    pre = oracle_mod.ssd_recurrence(p["x"][:, :6], p["dt"][:, :6], p["A"], p["B"][:, :6], p["C"][:, :6],
                                    D=p["D"], init=p["init"])
    h = pre["final_state"]
    for t in range(6, 9):
        x, dt, B, C = _step_slice(p, t)
        y, h = oracle_mod.ssd_step(x, dt, p["A"], B, C, state=h, D=p["D"])
        assert np.array_equal(y, full["y"][:, t])
    assert np.array_equal(h, full["final_state"])


def test_step_scalar_closed_form(oracle_mod):
    """S = H = 1: h' = e^{A dt} h + dt b x and y = c h' + D x, by hand."""
    import math
    x, dt, A, b, c, D, h0 = 0.7, 0.25, -1.3, 1.9, -0.4, 0.6, 2.0
    y, h = oracle_mod.ssd_step(np.full((1, 1, 1), x), np.full((1, 1), dt), np.array([A]),
                               np.full((1, 1, 1), b), np.full((1, 1, 1), c), state=np.full((1, 1, 1, 1), h0),
                               D=np.array([D]))
    h_ref = math.exp(A * dt) * h0 + dt * b * x
    assert abs(h[0, 0, 0, 0] - h_ref) <= 1e-15 * abs(h_ref)
    assert abs(y[0, 0, 0] - (c * h_ref + D * x)) <= 1e-14
