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
