"""Pins for the float64 oracle: each test checks the oracle against something other
than itself (a hand-derived example, a closed form, a different formulation,
an invariant of the mathematics), so that a plausible slip in the oracle (a
dropped term, a wrong index, a transposed state, a missing +1 in phi) fails
at least one of them. test_planted_mistakes_are_caught shows that for six
planted mistakes."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _rand(seed, B, H, T, d, dv, scale=1.0, dtype="f32"):
    q = synthetic.normal(seed, 0, (B, H, T, d), scale, dtype)
    k = synthetic.normal(seed, 1, (B, H, T, d), scale, dtype)
    v = synthetic.normal(seed, 2, (B, H, T, dv), scale, dtype)
    return q, k, v


def _fr(s):
    return float(Fraction(s))


# --- phi -------------------------------------------------------------------

def test_phi_closed_forms():
    x = np.array([0.0, 1e-300, 0.5, 3.0, -1e-12, -math.log(2.0), -math.log(4.0), -700.0])
    y = oracle.phi(x)
    assert y[0] == 1.0                        # elu(0) + 1
    assert y[1] == 1.0 and y[2] == 1.5 and y[3] == 4.0   # x + 1 for x > 0
    assert abs(y[4] - 1.0) < 1e-11            # continuous at 0 from the left
    assert abs(y[5] - 0.5) < 1e-15 and abs(y[6] - 0.25) < 1e-15   # exp branch
    assert 0.0 < y[7] < 1e-300                # tends to 0, stays positive
    # slope 1 on both sides of 0 (elu is C1 at 0 for alpha = 1)
    h = 1e-7
    assert abs((oracle.phi(np.array([h]))[0] - 1.0) / h - 1.0) < 1e-6
    assert abs((1.0 - oracle.phi(np.array([-h]))[0]) / h - 1.0) < 1e-6


# --- hand-derived examples ---------------------------------------------------

def test_hand_worked_examples():
    cases = json.load(open(GOLDEN))["cases"]
    for case in cases:
        q = np.array(case["q"], dtype=np.float32)[None, None]
        k = np.array(case["k"], dtype=np.float32)[None, None]
        v = np.array(case["v"], dtype=np.float32)[None, None]
        for ec in case["eps_cases"]:
            out, M, z = oracle.causal_fwd(q, k, v, eps=ec["eps"])
            want = np.array([[_fr(s) for s in row] for row in ec["out"]])
            np.testing.assert_allclose(out[0, 0], want, rtol=1e-14, atol=1e-14)
            np.testing.assert_allclose(M[0, 0], [[_fr(s) for s in r] for r in case["M_final"]], rtol=0, atol=0)
            np.testing.assert_allclose(z[0, 0], [_fr(s) for s in case["z_final"]], rtol=0, atol=0)
            # the all-pairs form agrees on the same hand example
            np.testing.assert_allclose(oracle.brute_force(q, k, v, eps=ec["eps"])[0, 0], want,
                                       rtol=1e-14, atol=1e-14)
        if "decode" in case:
            dc = case["decode"]
            _, M, z = oracle.causal_fwd(q, k, v, eps=0.0)
            o, M2, z2 = oracle.decode_step(np.array(dc["q"], np.float32)[None, None],
                                           np.array(dc["k"], np.float32)[None, None],
                                           np.array(dc["v"], np.float32)[None, None],
                                           M, z, eps=dc["eps"])
            np.testing.assert_allclose(o[0, 0], [_fr(s) for s in dc["out"]], rtol=1e-14)
            np.testing.assert_allclose(M2[0, 0], [[_fr(s) for s in r] for r in dc["M_final"]], rtol=0)
            np.testing.assert_allclose(z2[0, 0], [_fr(s) for s in dc["z_final"]], rtol=0)


# --- closed forms ----------------------------------------------------------------

def test_single_token_closed_form():
    q, k, v = _rand(7, 2, 3, 1, 8, 5)
    eps = 0.25
    out, M, z = oracle.causal_fwd(q, k, v, eps=eps)
    fq = oracle.phi(q.astype(np.float64))
    fk = oracle.phi(k.astype(np.float64))
    a = (fq * fk).sum(-1)                                   # [B,H,1]
    np.testing.assert_allclose(out, v.astype(np.float64) * (a / (a + eps))[..., None], rtol=1e-14)
    np.testing.assert_allclose(M, fk[:, :, 0, :, None] * v.astype(np.float64)[:, :, 0, None, :], rtol=0)
    np.testing.assert_allclose(z, fk[:, :, 0], rtol=0)


def test_constant_values_closed_form():
    q, k, _ = _rand(11, 1, 2, 40, 6, 3)
    c = np.array([0.5, -2.0, 3.0], dtype=np.float32)
    v = np.broadcast_to(c, (1, 2, 40, 3)).copy()
    eps = 1e-3
    out, _, _ = oracle.causal_fwd(q, k, v, eps=eps)
    fq, fk = oracle.phi(q.astype(np.float64)), oracle.phi(k.astype(np.float64))
    D = np.einsum("bhtd,bhtd->bht", fq, np.cumsum(fk, axis=2)) + eps
    np.testing.assert_allclose(out, c[None, None, None, :] * ((D - eps) / D)[..., None], rtol=1e-13)


def test_identical_keys_give_running_mean():
    q, _, v = _rand(12, 1, 1, 30, 4, 4)
    k = np.broadcast_to(np.array([0.3, -0.7, 1.1, 0.0], np.float32), (1, 1, 30, 4)).copy()
    eps = 1e-2
    out, _, _ = oracle.causal_fwd(q, k, v, eps=eps)
    fq, fk = oracle.phi(q.astype(np.float64)), oracle.phi(k[0, 0, 0].astype(np.float64))
    t = np.arange(1, 31)
    a = fq[0, 0] @ fk
    mean = np.cumsum(v[0, 0].astype(np.float64), axis=0) / t[:, None]
    np.testing.assert_allclose(out[0, 0], mean * ((t * a) / (t * a + eps))[:, None], rtol=1e-13)


def test_zero_queries_weight_by_key_mass():
    _, k, v = _rand(13, 1, 1, 25, 5, 3)
    q = np.zeros((1, 1, 25, 5), np.float32)                 # phi(0) = 1 in every feature
    eps = 1e-6
    out, _, _ = oracle.causal_fwd(q, k, v, eps=eps)
    w = oracle.phi(k.astype(np.float64))[0, 0].sum(-1)       # sum_a phi(k_ia)
    num = np.cumsum(w[:, None] * v[0, 0].astype(np.float64), axis=0)
    np.testing.assert_allclose(out[0, 0], num / (np.cumsum(w) + eps)[:, None], rtol=1e-13)


# --- other formulations --------------------------------------------------------------

@pytest.mark.parametrize("B,H,T,d,dv", [(1, 1, 1, 4, 4), (2, 3, 37, 8, 5), (1, 2, 128, 16, 16), (1, 1, 200, 32, 8)])
def test_recurrence_matches_all_pairs_form(B, H, T, d, dv):
    q, k, v = _rand(100 + T, B, H, T, d, dv)
    out, _, _ = oracle.causal_fwd(q, k, v)
    assert oracle.rel_err_rows(out, oracle.brute_force(q, k, v)) < 1e-12


def test_recurrence_matches_all_pairs_form_with_initial_state_bf16():
    q, k, v = _rand(21, 2, 2, 64, 16, 8, scale=0.5, dtype="bf16")
    rng = np.random.default_rng(0)
    M0 = rng.normal(size=(2, 2, 16, 8))
    z0 = rng.uniform(0.5, 3.0, size=(2, 2, 16))
    out, _, _ = oracle.causal_fwd(q, k, v, M_in=M0, z_in=z0)
    assert oracle.rel_err_rows(out, oracle.brute_force(q, k, v, M_in=M0, z_in=z0)) < 1e-12


@pytest.mark.parametrize("chunk", [1, 7, 16, 64, 100, 256])
def test_chunk_invariance(chunk):
    q, k, v = _rand(31, 1, 2, 150, 16, 12)
    out, M, z = oracle.causal_fwd(q, k, v)
    co, cM, cz = oracle.chunked_form(q, k, v, chunk)
    assert oracle.rel_err_rows(co, out) < 1e-12
    assert oracle.rel_err_state(cM, M, (2, 3)) < 1e-12
    assert oracle.rel_err_state(cz, z, (2,)) < 1e-12


def test_segment_invariance():
    q, k, v = _rand(41, 2, 2, 300, 16, 16, scale=0.5, dtype="bf16")
    out, M, z = oracle.causal_fwd(q, k, v)
    M_c = z_c = None
    outs = []
    for s0, s1 in [(0, 64), (64, 65), (65, 200), (200, 300)]:
        o, M_c, z_c = oracle.causal_fwd(q[:, :, s0:s1], k[:, :, s0:s1], v[:, :, s0:s1], M_in=M_c, z_in=z_c)
        outs.append(o)
    assert oracle.rel_err_rows(np.concatenate(outs, axis=2), out) < 1e-13
    assert oracle.rel_err_state(M_c, M, (2, 3)) < 1e-13
    assert oracle.rel_err_state(z_c, z, (2,)) < 1e-13


def test_last_causal_output_equals_noncausal():
    q, k, v = _rand(51, 1, 3, 90, 16, 16)
    out, _, _ = oracle.causal_fwd(q, k, v)
    nc = oracle.noncausal(q, k, v)
    assert oracle.rel_err_rows(out[:, :, -1], nc[:, :, -1]) < 1e-13
    # and it differs from the non-causal output everywhere before the end
    assert oracle.rel_err_rows(out[:, :, 10], nc[:, :, 10]) > 1e-3


def test_prefill_equals_forward_state_and_last_output():
    q, k, v = _rand(61, 2, 2, 120, 16, 8, scale=0.5, dtype="bf16")
    out, M, z = oracle.causal_fwd(q, k, v)
    o_last, Mp, zp = oracle.prefill(q, k, v)
    np.testing.assert_array_equal(Mp, M)
    np.testing.assert_array_equal(zp, z)
    np.testing.assert_array_equal(o_last, out[:, :, -1])


def test_decode_step_equals_appended_forward():
    q, k, v = _rand(71, 3, 2, 51, 16, 16, scale=0.5, dtype="bf16")
    out_all, M_all, z_all = oracle.causal_fwd(q, k, v)
    _, M, z = oracle.causal_fwd(q[:, :, :50], k[:, :, :50], v[:, :, :50])
    o, M2, z2 = oracle.decode_step(q[:, :, 50], k[:, :, 50], v[:, :, 50], M, z)
    np.testing.assert_allclose(o, out_all[:, :, 50], rtol=1e-14, atol=0)
    np.testing.assert_allclose(M2, M_all, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(z2, z_all, rtol=1e-14)


# --- invariants ----------------------------------------------------------------

def test_causality_exact():
    q, k, v = _rand(81, 1, 2, 80, 8, 8)
    out, _, _ = oracle.causal_fwd(q, k, v)
    v2, k2, q2 = v.copy(), k.copy(), q.copy()
    v2[:, :, 41:] += 10.0
    k2[:, :, 41:] -= 3.0
    q2[:, :, 41:] *= -1.0
    out2, _, _ = oracle.causal_fwd(q2, k2, v2)
    np.testing.assert_array_equal(out2[:, :, :41], out[:, :, :41])
    assert np.abs(out2[:, :, 41:] - out[:, :, 41:]).max() > 1e-3


def test_linear_in_values():
    q, k, v1 = _rand(91, 1, 2, 60, 8, 6)
    _, _, v2 = _rand(92, 1, 2, 60, 8, 6)
    o1, _, _ = oracle.causal_fwd(q, k, v1)
    o2, _, _ = oracle.causal_fwd(q, k, v2)
    v3 = (2.0 * v1.astype(np.float64) - 0.5 * v2.astype(np.float64)).astype(np.float32)
    o3, _, _ = oracle.causal_fwd(q, k, v3)
    ref = 2.0 * o1 - 0.5 * o2
    # v3 was rounded to float32, so compare through the float32 rounding of v3
    o3_exact = oracle.brute_force(q, k, v3)
    assert oracle.rel_err_rows(o3, o3_exact) < 1e-12
    assert oracle.rel_err_rows(o3, ref) < 1e-6


def test_outputs_inside_value_hull():
    q, k, v = _rand(93, 2, 2, 200, 16, 16, scale=0.5, dtype="bf16")
    out, _, _ = oracle.causal_fwd(q, k, v)
    vmax = np.maximum.accumulate(np.abs(synthetic.to_f64(v)), axis=2)
    assert np.all(np.abs(out) <= vmax * (1 + 1e-12))


# --- the pins catch planted mistakes ---------------------------------------------

def _pins_pass(mutation):
    """Run a compact set of the pins above against a mutated oracle."""
    case = json.load(open(GOLDEN))["cases"][1]
    q = np.array(case["q"], dtype=np.float32)[None, None]
    k = np.array(case["k"], dtype=np.float32)[None, None]
    v = np.array(case["v"], dtype=np.float32)[None, None]
    for ec in case["eps_cases"]:
        out, _, _ = oracle.causal_fwd(q, k, v, eps=ec["eps"], mutation=mutation)
        want = np.array([[_fr(s) for s in row] for row in ec["out"]])
        if not np.allclose(out[0, 0], want, rtol=1e-12, atol=1e-12):
            return False
    q, k, v = _rand(5, 1, 2, 64, 8, 8)
    out, _, _ = oracle.causal_fwd(q, k, v, eps=0.1, mutation=mutation)
    if oracle.rel_err_rows(out, oracle.brute_force(q, k, v, eps=0.1)) > 1e-12:
        return False
    return True


@pytest.mark.parametrize("mutation", [1, 2, 3, 4, 5, 6])
def test_planted_mistakes_are_caught(mutation):
    assert _pins_pass(0)
    assert not _pins_pass(mutation)
