"""Pins for the oracle's training backward (oracle.causal_bwd). Each check compares
it with something other than itself: a hand-worked example with exact rational values
(tests/golden/hand_worked_bwd.json), central finite differences of a float64 forward
written out in this file, float64 autograd of the masked all-pairs form, the
single-token closed form, and the chaining of segment backwards through the state
gradient. test_planted_backward_mistakes_are_caught shows that each of six
planted mistakes (a dropped normaliser term, an off-by-one state, an ignored state
gradient, a token missing from its own key gradient, a wrong phi', a transposed
state) fails at least one of them."""
import numpy as np
import pytest
import torch

import oracle
import synthetic

EPS = 1e-6


def _inputs(seed, B, H, T, d, dv, dtype="f32", scale=1.0):
    q = synthetic.normal(seed, 0, (B, H, T, d), scale, dtype)
    k = synthetic.normal(seed, 1, (B, H, T, d), scale, dtype)
    v = synthetic.normal(seed, 2, (B, H, T, dv), scale, dtype)
    rng = np.random.default_rng(seed)
    M0 = rng.normal(size=(B, H, d, dv))
    z0 = rng.uniform(0.5, 2.0, size=(B, H, d))
    dout = rng.normal(size=(B, H, T, dv))
    dM = rng.normal(size=(B, H, d, dv))
    dz = rng.normal(size=(B, H, d))
    return q, k, v, M0, z0, dout, dM, dz


def _values(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _loss(Q, K, V, M0, z0, dout, dM, dz, eps=EPS):
    """L = sum(dout * out) + sum(dM * M_T) + sum(dz * z_T) of the masked all-pairs
    forward, float64, from raw (pre-phi) q and k."""
    fq = np.where(Q > 0, Q + 1.0, np.exp(np.minimum(Q, 0.0)))
    fk = np.where(K > 0, K + 1.0, np.exp(np.minimum(K, 0.0)))
    T = Q.shape[2]
    A = np.einsum("bhtd,bhsd->bhts", fq, fk) * np.tril(np.ones((T, T)))
    num = np.einsum("bhts,bhsv->bhtv", A, V) + np.einsum("bhtd,bhdv->bhtv", fq, M0)
    den = A.sum(-1) + np.einsum("bhtd,bhd->bht", fq, z0) + eps
    out = num / den[..., None]
    MT = M0 + np.einsum("bhsd,bhsv->bhdv", fk, V)
    zT = z0 + fk.sum(2)
    return float((dout * out).sum() + (dM * MT).sum() + (dz * zT).sum())


def _fd_grads(q, k, v, M0, z0, dout, dM, dz):
    """Central differences of _loss with respect to every element of q, k, v, M0, z0."""
    args = [_values(q), _values(k), _values(v), np.array(M0, dtype=np.float64), np.array(z0, dtype=np.float64)]
    grads = []
    for which in range(5):
        g = np.zeros_like(args[which])
        flat = args[which].reshape(-1)
        gf = g.reshape(-1)
        for i in range(flat.size):
            x0 = flat[i]
            h = 1e-6 * max(1.0, abs(x0))
            flat[i] = x0 + h
            lp = _loss(*args, dout, dM, dz)
            flat[i] = x0 - h
            lm = _loss(*args, dout, dM, dz)
            flat[i] = x0
            gf[i] = (lp - lm) / (2 * h)
        grads.append(g)
    return grads


def _close(a, b, rtol):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.abs(a - b).max()) <= rtol * max(1.0, float(np.abs(b).max()))


def _fd_pin(mutation, seed=11, shape=(1, 2, 6, 3, 3)):
    q, k, v, M0, z0, dout, dM, dz = _inputs(seed, *shape)
    assert np.abs(_values(q)).min() > 1e-3 and np.abs(_values(k)).min() > 1e-3  # away from phi's kink
    got = oracle.causal_bwd(q, k, v, dout, M0, z0, dM, dz, eps=EPS, mutation=mutation)
    ref = _fd_grads(q, k, v, M0, z0, dout, dM, dz)
    return all(_close(g, r, 1e-6) for g, r in zip(got, ref))


def _single_token_pin(mutation):
    """T = 1, zero state: out = v a / (a + eps) with a = phi(q) . phi(k)."""
    q, k, v, _, _, dout, _, _ = _inputs(5, 1, 1, 1, 4, 3)
    eps = 0.25  # large enough that the eps terms are not negligible
    Q, K, V, g_out = _values(q)[0, 0, 0], _values(k)[0, 0, 0], _values(v)[0, 0, 0], dout[0, 0, 0]
    fq = np.where(Q > 0, Q + 1, np.exp(Q))
    fk = np.where(K > 0, K + 1, np.exp(K))
    dfq = np.where(Q > 0, 1.0, np.exp(Q))
    dfk = np.where(K > 0, 1.0, np.exp(K))
    a = fq @ fk
    dL_da = (g_out @ V) * eps / (a + eps) ** 2
    exp_dv = g_out * a / (a + eps)
    exp_dq = dL_da * fk * dfq
    exp_dk = dL_da * fq * dfk
    exp_dM = np.outer(fq, g_out / (a + eps))
    exp_dz = -(g_out @ V) * a / (a + eps) ** 2 * fq
    dq, dk, dvv, dM, dz = oracle.causal_bwd(q, k, v, dout, eps=eps, mutation=mutation)
    return (_close(dq[0, 0, 0], exp_dq, 1e-12) and _close(dk[0, 0, 0], exp_dk, 1e-12)
            and _close(dvv[0, 0, 0], exp_dv, 1e-12) and _close(dM[0, 0], exp_dM, 1e-12)
            and _close(dz[0, 0], exp_dz, 1e-12))


def _chain_pin(mutation, T=24, cut=10):
    """Backward over [0, T) equals the backward of [cut, T) from the state after the first
    part, followed by the backward of [0, cut) with that part's state gradients."""
    q, k, v, M0, z0, dout, dM, dz = _inputs(9, 1, 2, T, 4, 4)
    full = oracle.causal_bwd(q, k, v, dout, M0, z0, dM, dz, mutation=mutation)
    s1, s2 = slice(0, cut), slice(cut, T)
    part = lambda a, s: np.ascontiguousarray(a[:, :, s])
    _, M1, z1 = oracle.causal_fwd(part(q, s1), part(k, s1), part(v, s1), M0, z0)
    dq2, dk2, dv2, dM1, dz1 = oracle.causal_bwd(part(q, s2), part(k, s2), part(v, s2), part(dout, s2), M1, z1, dM, dz,
                                                mutation=mutation)
    dq1, dk1, dv1, dM0, dz0 = oracle.causal_bwd(part(q, s1), part(k, s1), part(v, s1), part(dout, s1), M0, z0, dM1,
                                                dz1, mutation=mutation)
    pieces = [(np.concatenate([dq1, dq2], 2), full[0]), (np.concatenate([dk1, dk2], 2), full[1]),
              (np.concatenate([dv1, dv2], 2), full[2]), (dM0, full[3]), (dz0, full[4])]
    return all(_close(a, b, 1e-11) for a, b in pieces)


def test_backward_matches_finite_differences():
    assert _fd_pin(0)


def test_backward_matches_finite_differences_unequal_dims():
    assert _fd_pin(0, seed=12, shape=(1, 1, 7, 3, 2))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_matches_autograd_of_all_pairs_form(dtype):
    q, k, v, M0, z0, dout, dM, dz = _inputs(21, 2, 2, 40, 8, 5, dtype=dtype)
    t = lambda a: torch.tensor(_values(a) if isinstance(a, np.ndarray) and a.dtype in (np.uint16, np.float32)
                               else np.asarray(a, dtype=np.float64), dtype=torch.float64, requires_grad=True)
    Q, K, V, Mt, zt = t(q), t(k), t(v), t(M0), t(z0)
    fq = torch.where(Q > 0, Q + 1, torch.exp(torch.clamp(Q, max=0)))
    fk = torch.where(K > 0, K + 1, torch.exp(torch.clamp(K, max=0)))
    T = Q.shape[2]
    A = torch.einsum("bhtd,bhsd->bhts", fq, fk) * torch.tril(torch.ones(T, T, dtype=torch.float64))
    num = torch.einsum("bhts,bhsv->bhtv", A, V) + torch.einsum("bhtd,bhdv->bhtv", fq, Mt)
    den = A.sum(-1) + torch.einsum("bhtd,bhd->bht", fq, zt) + EPS
    out = num / den[..., None]
    MT = Mt + torch.einsum("bhsd,bhsv->bhdv", fk, V)
    zT = zt + fk.sum(2)
    L = (torch.tensor(dout) * out).sum() + (torch.tensor(dM) * MT).sum() + (torch.tensor(dz) * zT).sum()
    L.backward()
    got = oracle.causal_bwd(q, k, v, dout, M0, z0, dM, dz, eps=EPS)
    for g, r in zip(got, (Q.grad, K.grad, V.grad, Mt.grad, zt.grad)):
        assert _close(g, r.numpy(), 1e-10)


def test_backward_single_token_closed_form():
    assert _single_token_pin(0)


def test_backward_chains_across_segments():
    assert _chain_pin(0)


def test_backward_without_state_gradients_equals_zero_state_gradients():
    q, k, v, M0, z0, dout, _, _ = _inputs(3, 1, 2, 17, 4, 3)
    a = oracle.causal_bwd(q, k, v, dout, M0, z0)
    b = oracle.causal_bwd(q, k, v, dout, M0, z0, np.zeros((1, 2, 4, 3)), np.zeros((1, 2, 4)))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def _bwd_pins_pass(mutation):
    return _fd_pin(mutation) and _single_token_pin(mutation) and _chain_pin(mutation)


def test_backward_pins_pass_for_the_oracle():
    assert _bwd_pins_pass(0)


@pytest.mark.parametrize("mutation", [11, 12, 13, 14, 15, 16])
def test_planted_backward_mistakes_are_caught(mutation):
    assert not _bwd_pins_pass(mutation)


def test_backward_hand_worked_example():
    """tests/golden/hand_worked_bwd.json: T = 2, d = dv = 1, eps = 1, values derived by hand."""
    import json
    import os
    from fractions import Fraction
    with open(os.path.join(os.path.dirname(__file__), "golden", "hand_worked_bwd.json")) as f:
        g = json.load(f)
    x = g["inputs"]
    arr = lambda a, n: np.array(a, dtype=np.float32).reshape(1, 1, 2, n)
    q, k, v = arr(x["q"], 1), arr(x["k"], 1), arr(x["v"], 1)
    dout = np.array(x["dout"], dtype=np.float64).reshape(1, 1, 2, 1)
    dq, dk, dvv, dM, dz = oracle.causal_bwd(q, k, v, dout, eps=x["eps"])
    fr = lambda s: float(Fraction(s))
    e = g["expected"]
    for got, want in ((dq, e["dq"]), (dk, e["dk"]), (dvv, e["dv"])):
        assert np.allclose(got.reshape(-1), [fr(s) for s in want], rtol=1e-14, atol=0)
    assert abs(dM.item() - fr(e["dM_in"])) <= 1e-14 * abs(fr(e["dM_in"]))
    assert abs(dz.item() - fr(e["dz_in"])) <= 1e-14 * abs(fr(e["dz_in"]))
