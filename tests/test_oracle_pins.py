"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test names the fact it checks. Together they are chosen so that a
dropped term, a wrong sign, a wrong scale, a transposed operand or a
softmax over the wrong axis in the oracle fails at least one of them:

* a hand-worked example with a closed form (tests/golden/two_keys.json);
* length-1 sequences (O = V, LSE = s q.k, dQ = dK = 0, dV = dO);
* constant scores (O = mean of V, LSE = ln Lk);
* jagged == padded dense attention through torch's float64
  scaled_dot_product_attention with a key mask (a library routine), forward
  and, through torch autograd, backward;
* central finite differences of sum(O * dO) on tiny inputs;
* invariants: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i per sequence/head;
  shift invariance of O under k_j -> k_j + c;
* block-diagonal == jagged with offsets at multiples of 64;
* broadcast-Q == library attention per sequence, dQ == sum of per-sequence
  autograd gradients.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng):
    return rng.standard_normal(shape)


def _offsets(lengths):
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    off[1:] = np.cumsum(lengths)
    return off


# ---------------------------------------------------------------- closed forms

def test_golden_two_keys():
    g = json.load(open(os.path.join(GOLDEN, "two_keys.json")))
    q, k, v, do = (np.array(g[n]) for n in ("q", "k", "v", "do"))
    O, lse = A.seq_fwd(q, k, v, g["scale"])
    np.testing.assert_allclose(O, g["o"], atol=1e-12)
    np.testing.assert_allclose(lse, g["lse"], atol=1e-12)
    dq, dk, dv = A.seq_bwd(q, k, v, do, g["scale"])
    np.testing.assert_allclose(dq, g["dq"], atol=1e-12)
    np.testing.assert_allclose(dk, g["dk"], atol=1e-12)
    np.testing.assert_allclose(dv, g["dv"], atol=1e-12)


def test_length_one_sequences():
    rng = np.random.default_rng(11)
    lengths = [1, 1, 3, 1]
    T, H, D = sum(lengths), 2, 8
    q, k, v, do = (_rand((T, H, D), rng) for _ in range(4))
    s = 1 / math.sqrt(D)
    off = _offsets(lengths)
    o, lse = A.jagged_fwd(q, k, v, off, s)
    dq, dk, dv = A.jagged_bwd(q, k, v, do, off, s)
    for b, L in enumerate(lengths):
        if L != 1:
            continue
        t = off[b]
        np.testing.assert_array_equal(o[t], v[t])
        np.testing.assert_allclose(lse[:, t], s * np.sum(q[t] * k[t], axis=-1), rtol=1e-14)
        # exact arithmetic gives 0; dP and Di are summed in different orders
        np.testing.assert_allclose(dq[t], 0.0, atol=1e-13)
        np.testing.assert_allclose(dk[t], 0.0, atol=1e-13)
        np.testing.assert_allclose(dv[t], do[t], rtol=1e-14)


def test_constant_scores_give_mean_of_v():
    rng = np.random.default_rng(12)
    Lk, D = 37, 16
    v = _rand((Lk, D), rng)
    # Q = 0: every score is 0.
    O, lse = A.seq_fwd(np.zeros((5, D)), _rand((Lk, D), rng), v, 0.125)
    np.testing.assert_allclose(O, np.broadcast_to(v.mean(0), O.shape), atol=1e-13)
    np.testing.assert_allclose(lse, math.log(Lk), atol=1e-13)
    # all keys equal: scores constant along each row.
    q = _rand((5, D), rng)
    krow = _rand((1, D), rng)
    O, lse = A.seq_fwd(q, np.repeat(krow, Lk, 0), v, 0.125)
    np.testing.assert_allclose(O, np.broadcast_to(v.mean(0), O.shape), atol=1e-13)
    np.testing.assert_allclose(lse, 0.125 * (q @ krow[0]) + math.log(Lk), atol=1e-12)


# ----------------------------------------------------------- library routines

def _padded_sdpa(q, k, v, do, offsets, scale):
    """Padded dense attention through torch's fp64 SDPA + autograd."""
    lengths = np.diff(offsets)
    B, Lmax = len(lengths), int(lengths.max())
    T, H, D = q.shape

    def pad(x):
        out = torch.zeros(B, H, Lmax, x.shape[-1], dtype=torch.float64)
        for b in range(B):
            s, e = offsets[b], offsets[b + 1]
            out[b, :, : e - s] = torch.from_numpy(x[s:e]).permute(1, 0, 2)
        return out

    Q, K, V, dO = (pad(x) for x in (q, k, v, do))
    mask = torch.zeros(B, 1, Lmax, Lmax, dtype=torch.bool)
    for b in range(B):
        mask[b, :, :, : lengths[b]] = True
    for t in (Q, K, V):
        t.requires_grad_(True)
    O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
    (O * dO).sum().backward()

    def unpad(x):
        out = np.zeros((T, H, x.shape[-1]))
        for b in range(B):
            s, e = offsets[b], offsets[b + 1]
            out[s:e] = x[b, :, : e - s].permute(1, 0, 2).detach().numpy()
        return out

    return unpad(O), unpad(Q.grad), unpad(K.grad), unpad(V.grad)


def test_jagged_equals_padded_dense_library():
    rng = np.random.default_rng(13)
    lengths = [5, 1, 17, 9, 30]
    T, H, D = sum(lengths), 3, 16
    q, k, v, do = (_rand((T, H, D), rng) for _ in range(4))
    off = _offsets(lengths)
    s = 1 / math.sqrt(D)
    O_ref, dq_ref, dk_ref, dv_ref = _padded_sdpa(q, k, v, do, off, s)
    o, _ = A.jagged_fwd(q, k, v, off, s)
    dq, dk, dv = A.jagged_bwd(q, k, v, do, off, s)
    np.testing.assert_allclose(o, O_ref, atol=1e-12)
    np.testing.assert_allclose(dq, dq_ref, atol=1e-12)
    np.testing.assert_allclose(dk, dk_ref, atol=1e-12)
    np.testing.assert_allclose(dv, dv_ref, atol=1e-12)


def test_lse_is_log_of_row_sum():
    rng = np.random.default_rng(14)
    q, k, v = _rand((9, 8), rng), _rand((13, 8), rng), _rand((13, 8), rng)
    _, lse = A.seq_fwd(q, k, v, 0.3)
    ref = torch.logsumexp(torch.from_numpy(0.3 * q @ k.T), dim=1).numpy()
    np.testing.assert_allclose(lse, ref, atol=1e-13)


def test_bcast_equals_library_attention_and_summed_dq():
    rng = np.random.default_rng(15)
    lengths = [4, 11, 1, 7]
    Lq, H, D = 6, 2, 8
    Tk = sum(lengths)
    q = _rand((Lq, H, D), rng)
    k, v = _rand((Tk, H, D), rng), _rand((Tk, H, D), rng)
    do = _rand((len(lengths), Lq, H, D), rng)
    off = _offsets(lengths)
    s = 0.4
    o, lse = A.bcastq_fwd(q, k, v, off, s)
    dq, dk, dv = A.bcastq_bwd(q, k, v, do, off, s)
    Q = torch.from_numpy(q).permute(1, 0, 2).clone().requires_grad_(True)
    dq_ref = np.zeros_like(q)
    for b in range(len(lengths)):
        a, e = off[b], off[b + 1]
        K = torch.from_numpy(k[a:e]).permute(1, 0, 2).clone().requires_grad_(True)
        V = torch.from_numpy(v[a:e]).permute(1, 0, 2).clone().requires_grad_(True)
        if Q.grad is not None:
            Q.grad = None
        O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=s)
        (O * torch.from_numpy(do[b]).permute(1, 0, 2)).sum().backward()
        np.testing.assert_allclose(o[b], O.detach().permute(1, 0, 2).numpy(), atol=1e-12)
        np.testing.assert_allclose(dk[a:e], K.grad.permute(1, 0, 2).numpy(), atol=1e-12)
        np.testing.assert_allclose(dv[a:e], V.grad.permute(1, 0, 2).numpy(), atol=1e-12)
        dq_ref += Q.grad.permute(1, 0, 2).numpy()
        ref_lse = torch.logsumexp(s * Q.detach() @ K.detach().transpose(1, 2), dim=-1).numpy()
        np.testing.assert_allclose(lse[b], ref_lse, atol=1e-12)
    np.testing.assert_allclose(dq, dq_ref, atol=1e-12)


def test_bcast_empty_sequence_reading():
    q = np.ones((3, 1, 4))
    k = np.ones((2, 1, 4))
    off = np.array([0, 0, 2])
    o, lse = A.bcastq_fwd(q, k, k, off, 0.5)
    np.testing.assert_array_equal(o[0], 0.0)
    assert np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


# ----------------------------------------------------------- finite differences

def _loss(q, k, v, do, off, s):
    o, _ = A.jagged_fwd(q, k, v, off, s)
    return float(np.sum(o * do))


def test_finite_differences_tiny():
    rng = np.random.default_rng(16)
    lengths = [3, 1, 7, 5]
    T, H, D = sum(lengths), 2, 4
    q, k, v, do = (_rand((T, H, D), rng) for _ in range(4))
    off = _offsets(lengths)
    s = 1 / math.sqrt(D)
    grads = A.jagged_bwd(q, k, v, do, off, s)
    h = 1e-6
    for which, g in zip(range(3), grads):
        num = np.zeros_like(g)
        for idx in np.ndindex(g.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = _loss(*args, do, off, s)
            args[which][idx] -= 2 * h
            lm = _loss(*args, do, off, s)
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(num - g) / np.linalg.norm(g)
        assert err < 1e-6, (which, err)


# ------------------------------------------------------------------ invariants

def test_backward_invariants():
    rng = np.random.default_rng(17)
    Q, K, V, dO = _rand((21, 8), rng), _rand((21, 8), rng), _rand((21, 8), rng), _rand((21, 8), rng)
    dq, dk, dv = A.seq_bwd(Q, K, V, dO, 0.35)
    np.testing.assert_allclose(dk.sum(0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(0), dO.sum(0), atol=1e-12)


def test_shift_invariance_of_keys():
    rng = np.random.default_rng(18)
    Q, K, V = _rand((12, 8), rng), _rand((12, 8), rng), _rand((12, 8), rng)
    c = _rand((1, 8), rng)
    O1, l1 = A.seq_fwd(Q, K, V, 0.35)
    O2, l2 = A.seq_fwd(Q, K + c, V, 0.35)
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, 0.35 * (Q @ c[0]), atol=1e-12)


def test_row_chunking_is_invisible(monkeypatch):
    rng = np.random.default_rng(19)
    Q, K, V, dO = (_rand((50, 8), rng) for _ in range(4))
    ref = A.seq_fwd(Q, K, V, 0.3), A.seq_bwd(Q, K, V, dO, 0.3)
    monkeypatch.setattr(A, "ROW_CHUNK", 7)
    got = A.seq_fwd(Q, K, V, 0.3), A.seq_bwd(Q, K, V, dO, 0.3)
    for a, b in zip(ref[0] + ref[1], got[0] + got[1]):
        np.testing.assert_allclose(a, b, atol=1e-13)


def test_blockdiag_equals_jagged_with_64_token_sequences():
    rng = np.random.default_rng(20)
    B, L, H, D = 2, 192, 2, 8
    q, k, v, do = (_rand((B, L, H, D), rng) for _ in range(4))
    s = 1 / math.sqrt(D)
    o = A.blockdiag_fwd(q, k, v, s)
    dq, dk, dv = A.blockdiag_bwd(q, k, v, do, s)
    off = np.arange(0, B * L + 1, 64)
    flat = lambda x: x.reshape(B * L, H, D)  # noqa: E731
    o_j, _ = A.jagged_fwd(flat(q), flat(k), flat(v), off, s)
    g_j = A.jagged_bwd(flat(q), flat(k), flat(v), flat(do), off, s)
    np.testing.assert_allclose(flat(o), o_j, atol=1e-12)
    for a, b in zip((dq, dk, dv), g_j):
        np.testing.assert_allclose(flat(a), b, atol=1e-12)
