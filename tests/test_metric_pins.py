"""Pins for the two tolerance metrics every parity test goes through.

rel_err_rows(got, ref): max over rows (last axis) of ||got - ref||_inf / ||ref||_inf,
with a zero reference row measured in absolute terms.
rel_err_state(got, ref, axes): max over the leading index of max|got - ref| / max|ref|,
both maxima taken over `axes` (per head for a state [B, H, d, dv] with axes (2, 3)).

Each test builds arrays whose answer is known exactly by hand and checks the value
itself, not an upper bound, so that a slip in either metric (numerator and
denominator swapped, a wrong axis, one global normaliser instead of one per row or
head, a missing absolute value, the zero-row convention) changes a checked number."""
import numpy as np

import oracle


# ---------------------------------------------------------------- rel_err_rows

def test_rows_exact_value_per_row_normaliser():
    ref = np.array([[4.0, -2.0, 1.0],      # ||ref||_inf = 4
                    [0.5, 0.25, -0.5]])    # ||ref||_inf = 0.5
    got = ref.copy()
    got[0, 1] += 0.25                      # row 0: 0.25 / 4 = 1/16
    got[1, 2] -= 0.0625                    # row 1: 0.0625 / 0.5 = 1/8  (the maximum)
    assert oracle.rel_err_rows(got, ref) == 0.125
    # one global normaliser (max over everything = 4) would give 0.0625 / 4 = 1/64
    # and the swapped ratio ||ref|| / ||diff|| would give 8: both differ from 1/8


def test_rows_sign_of_the_difference_does_not_matter():
    ref = np.array([[2.0, 2.0]])
    assert oracle.rel_err_rows(ref + np.array([[0.0, -0.5]]), ref) == 0.25
    assert oracle.rel_err_rows(ref + np.array([[0.0, 0.5]]), ref) == 0.25
    # the reference's sign enters through its absolute value
    assert oracle.rel_err_rows(-ref + np.array([[0.5, 0.0]]), -ref) == 0.25


def test_rows_zero_reference_row_is_absolute():
    ref = np.array([[0.0, 0.0, 0.0], [8.0, 1.0, 1.0]])
    got = np.array([[0.0, 0.03125, 0.0], [8.0, 1.0, 1.0]])
    assert oracle.rel_err_rows(got, ref) == 0.03125


def test_rows_normalise_along_the_last_axis_only():
    # the largest entry of column 0 is in row 1; per-row normalisation must not see it
    ref = np.array([[1.0, 1.0], [64.0, 1.0]])
    got = ref.copy()
    got[0, 1] = 1.5                        # row 0: 0.5 / 1
    assert oracle.rel_err_rows(got, ref) == 0.5
    # column-wise normalisation (axis 0) would give 0.5 / 1 on column 1 as well, so
    # also plant a column-only case: row 1's error against its own row maximum
    got2 = ref.copy()
    got2[1, 1] = 5.0                       # row 1: 4 / 64 = 1/16; column 1 max is 1 -> 4
    assert oracle.rel_err_rows(got2, ref) == 0.0625


def test_rows_batched_leading_axes():
    ref = np.ones((2, 3, 4, 5))
    got = ref.copy()
    got[1, 2, 3, 4] = 1.0 + 2.0 ** -10     # one element of one row of one head
    assert oracle.rel_err_rows(got, ref) == 2.0 ** -10
    got[0, 0, 0, 0] = 1.0 - 2.0 ** -6
    assert oracle.rel_err_rows(got, ref) == 2.0 ** -6
    assert oracle.rel_err_rows(ref, ref) == 0.0


def test_rows_planted_one_percent_error():
    rng = np.random.default_rng(0)
    ref = rng.normal(size=(3, 7, 16))
    got = ref.copy()
    b, t = 1, 4
    j = int(np.abs(ref[b, t]).argmax())
    got[b, t, j] *= 1.01                   # 1% of the row's largest entry
    assert abs(oracle.rel_err_rows(got, ref) - 0.01) < 1e-12


# ---------------------------------------------------------------- rel_err_state

def test_state_per_head_normaliser():
    # [B=1, H=2, d=2, dv=2]: head 0 has max|M| = 8, head 1 has max|M| = 0.5
    ref = np.array([[[[8.0, 1.0], [2.0, -4.0]],
                     [[0.5, 0.25], [-0.125, 0.5]]]])
    got = ref.copy()
    got[0, 0, 1, 1] += 0.5                 # head 0: 0.5 / 8 = 1/16
    got[0, 1, 0, 1] -= 0.125               # head 1: 0.125 / 0.5 = 1/4 (the maximum)
    assert oracle.rel_err_state(got, ref, (2, 3)) == 0.25
    # a global normaliser (max over both heads = 8) would report 0.5 / 8 = 1/16


def test_state_axes_select_the_normalised_block():
    # [B=2, H=1, d=2]: z per head; the normaliser runs over d only
    ref = np.array([[[4.0, 1.0]], [[16.0, 16.0]]])
    got = ref.copy()
    got[0, 0, 1] = 2.0                     # (b=0): 1 / 4
    got[1, 0, 0] = 17.0                    # (b=1): 1 / 16
    assert oracle.rel_err_state(got, ref, (2,)) == 0.25
    # per-element normalisation (axes = ()) would report 1 / 1 for (b=0, i=1)
    assert oracle.rel_err_state(got, ref, ()) == 1.0


def test_state_wrong_axes_give_a_different_answer():
    # M [B=1, H=1, d=2, dv=2]: rows of very different size
    ref = np.array([[[[100.0, 100.0], [1.0, 1.0]]]])
    got = ref.copy()
    got[0, 0, 1, 0] = 2.0
    assert oracle.rel_err_state(got, ref, (2, 3)) == 0.01      # 1 / 100 over the whole head
    assert oracle.rel_err_state(got, ref, (3,)) == 1.0         # row by row: 1 / 1
    assert oracle.rel_err_state(got, ref, (2,)) == 0.01        # column by column: 1 / 100


def test_state_zero_reference_head_is_absolute():
    ref = np.zeros((1, 2, 3))
    ref[0, 1] = [2.0, 2.0, 2.0]
    got = ref.copy()
    got[0, 0, 2] = -0.0078125              # head 0 has a zero reference: absolute error
    assert oracle.rel_err_state(got, ref, (2,)) == 0.0078125


def test_state_planted_one_percent_error_in_one_head():
    rng = np.random.default_rng(1)
    ref = rng.normal(size=(2, 3, 8, 8))
    got = ref.copy()
    b, h = 1, 2
    i, j = np.unravel_index(np.abs(ref[b, h]).argmax(), (8, 8))
    got[b, h, i, j] *= 1.01
    assert abs(oracle.rel_err_state(got, ref, (2, 3)) - 0.01) < 1e-12
    # the same slip in another element of that head scales with that element
    got = ref.copy()
    got[b, h, 0, 0] += 0.01 * np.abs(ref[b, h]).max() / 2
    assert abs(oracle.rel_err_state(got, ref, (2, 3)) - 0.005) < 1e-12
