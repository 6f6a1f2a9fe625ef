"""The oracle's pins have teeth: each test plants one plausible mistake in a
copy of the oracle's per-sequence forward or backward (on the CPU, through
monkeypatch) and checks that at least one pin of the oracle then fails
(a wrong value, or operands whose shapes no longer fit).

Pins exercised: the hand-computed two-key golden case, length-one
sequences (O = V, dQ = dK = 0, dV = dO), central finite differences of
sum(O * dO) on tiny inputs, and the backward invariants sum_j dK_j = 0 and
sum_j dV_j = sum_i dO_i.
"""

import json
import os

import numpy as np
import pytest

from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "two_keys.json")


def _rand(shape, rng):
    return rng.standard_normal(shape)


# ------------------------------------------------------------ the pin battery


def _pin_golden():
    g = json.load(open(GOLDEN))
    q, k, v, do = (np.asarray(g[n], dtype=np.float64) for n in ("q", "k", "v", "do"))
    o, lse = A.seq_fwd(q, k, v, g["scale"])
    np.testing.assert_allclose(o, g["o"], atol=1e-12)
    np.testing.assert_allclose(lse, g["lse"], atol=1e-12)
    for got, name in zip(A.seq_bwd(q, k, v, do, g["scale"]), ("dq", "dk", "dv")):
        np.testing.assert_allclose(got, g[name], atol=1e-12)


def _pin_length_one():
    rng = np.random.default_rng(31)
    q, k, v, do = (_rand((1, 6), rng) for _ in range(4))
    o, _ = A.seq_fwd(q, k, v, 0.4)
    np.testing.assert_allclose(o, v, atol=1e-12)
    dq, dk, dv = A.seq_bwd(q, k, v, do, 0.4)
    np.testing.assert_allclose(dq, 0.0, atol=1e-12)
    np.testing.assert_allclose(dk, 0.0, atol=1e-12)
    np.testing.assert_allclose(dv, do, atol=1e-12)


def _pin_finite_differences():
    rng = np.random.default_rng(32)
    Q, K, V, dO = (_rand((5, 3), rng) for _ in range(4))
    s, h = 0.6, 1e-6

    def loss(q, k, v):
        o, _ = A.seq_fwd(q, k, v, s)
        return float(np.sum(o * dO))

    grads = A.seq_bwd(Q, K, V, dO, s)
    for which, g in enumerate(grads):
        num = np.zeros_like(g)
        for idx in np.ndindex(g.shape):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            num[idx] = (lp - loss(*args)) / (2 * h)
        assert np.linalg.norm(num - g) <= 1e-6 * np.linalg.norm(num), which


def _pin_invariants():
    rng = np.random.default_rng(33)
    Q, K, V, dO = (_rand((9, 4), rng) for _ in range(4))
    _, dk, dv = A.seq_bwd(Q, K, V, dO, 0.5)
    np.testing.assert_allclose(dk.sum(0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(0), dO.sum(0), atol=1e-12)


PINS = (_pin_golden, _pin_length_one, _pin_finite_differences, _pin_invariants)


def test_unmodified_oracle_passes_every_pin():
    for pin in PINS:
        pin()


# --------------------------------------------------- mutated copies of the oracle


def _bwd_with(ds_rule=None, dq_rule=None, dk_rule=None, dv_rule=None):
    """A copy of the oracle's per-sequence backward with one step replaced;
    each rule gets every intermediate by name."""

    def seq_bwd(Q, K, V, dO, scale, O=None, window=None):  # window: unused by these pins
        Q, K, V, dO = (np.asarray(x, dtype=np.float64) for x in (Q, K, V, dO))
        if O is None:
            O, _ = A.seq_fwd(Q, K, V, scale)
        x = dict(Q=Q, K=K, V=V, dO=dO, O=O, s=scale)
        x["P"], _ = A.softmax_rows(scale * (Q @ K.T))
        x["dP"] = dO @ V.T
        x["Di"] = np.sum(dO * O, axis=1, keepdims=True)
        x["dS"] = ds_rule(x) if ds_rule else x["P"] * (x["dP"] - x["Di"])
        dV = dv_rule(x) if dv_rule else x["P"].T @ dO
        dQ = dq_rule(x) if dq_rule else scale * (x["dS"] @ K)
        dK = dk_rule(x) if dk_rule else scale * (x["dS"].T @ Q)
        return dQ, dK, dV

    return seq_bwd


def _fwd_with(scores=None, softmax_axis=1):
    """A copy of the oracle's per-sequence forward with one step replaced."""

    def seq_fwd(Q, K, V, scale, window=None):  # window: unused by these pins
        Q, K, V = (np.asarray(x, dtype=np.float64) for x in (Q, K, V))
        S = scores(Q, K, scale) if scores else scale * (Q @ K.T)
        m = S.max(axis=softmax_axis, keepdims=True)
        e = np.exp(S - m)
        l = e.sum(axis=softmax_axis, keepdims=True)
        P = e / l
        lse = (S.max(axis=1, keepdims=True) + np.log(np.exp(S - S.max(axis=1, keepdims=True)).sum(
            axis=1, keepdims=True)))[:, 0]
        return P @ V, lse

    return seq_fwd


BWD_MUTANTS = {
    "Di dropped": dict(ds_rule=lambda x: x["P"] * x["dP"]),
    "sign of Di flipped": dict(ds_rule=lambda x: x["P"] * (x["dP"] + x["Di"])),
    "dK from dO instead of Q": dict(dk_rule=lambda x: x["s"] * (x["dS"].T @ x["dO"])),
    "dV from P not transposed": dict(dv_rule=lambda x: x["P"] @ x["dO"]),
    "scale missing in dQ": dict(dq_rule=lambda x: x["dS"] @ x["K"]),
    "Di summed over the wrong axis": dict(ds_rule=lambda x: x["P"] * (
        x["dP"] - np.sum(x["dO"] * x["O"], axis=0, keepdims=True)[:, :1])),
}

FWD_MUTANTS = {
    "softmax over the query axis": dict(softmax_axis=0),
    "scores not scaled": dict(scores=lambda Q, K, s: Q @ K.T),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_backward_mutant_is_caught(monkeypatch, name):
    monkeypatch.setattr(A, "seq_bwd", _bwd_with(**BWD_MUTANTS[name]))
    failures = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError):  # a wrong value, or shapes that no longer fit
            failures += 1
    assert failures > 0, name


@pytest.mark.parametrize("name", sorted(FWD_MUTANTS))
def test_forward_mutant_is_caught(monkeypatch, name):
    monkeypatch.setattr(A, "seq_fwd", _fwd_with(**FWD_MUTANTS[name]))
    failures = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError):  # a wrong value, or shapes that no longer fit
            failures += 1
    assert failures > 0, name
