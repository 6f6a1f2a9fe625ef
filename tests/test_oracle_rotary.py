"""Pins of the oracle's rotary block-diagonal attention (CPU only):

* zero angles (cos = 1, sin = 0) reduce it to plain block-diagonal attention;
* the rotation keeps every (i, i + D/2) pair's length and its transpose
  undoes it;
* with the usual tables (angle = position * base^(-2i/D)) a rotated score
  depends only on the distance between the two positions;
* the same attention written with torch complex numbers (pairs as
  x[i] + j x[i + D/2] multiplied by exp(j angle)) through torch's float64
  scaled_dot_product_attention with a block mask, forward and, by autograd,
  backward;
* central finite differences of sum(O * dO) on a tiny case;
* a planted mistake (the backward rotating forward instead of back) fails;
* the backward taken from the rotated q_r, k_r equals the one taken from q
  and k (with q_r, k_r the rotation of q, k).
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention as A


def _tables(L, D, base=10000.0):
    i = np.arange(D // 2)
    ang = np.arange(L)[:, None] * base ** (-2.0 * i / D)[None, :]
    return np.cos(ang), np.sin(ang)


def _rand(shape, rng):
    return rng.standard_normal(shape)


def test_zero_angles_reduce_to_plain_blockdiag():
    rng = np.random.default_rng(81)
    B, L, H, D = 2, 128, 2, 16
    q, k, v, do = (_rand((B, L, H, D), rng) for _ in range(4))
    c, s = np.ones((L, D // 2)), np.zeros((L, D // 2))
    np.testing.assert_allclose(A.blockdiag_rotary_fwd(q, k, v, c, s, 0.3),
                               A.blockdiag_fwd(q, k, v, 0.3), atol=1e-14)
    for a, b in zip(A.blockdiag_rotary_bwd(q, k, v, do, c, s, 0.3), A.blockdiag_bwd(q, k, v, do, 0.3)):
        np.testing.assert_allclose(a, b, atol=1e-13)


def test_rotation_is_orthogonal_and_transpose_inverts_it():
    rng = np.random.default_rng(82)
    L, D = 64, 8
    x = _rand((1, L, 3, D), rng)
    c, s = _tables(L, D)
    xr = A.rope(x, c, s)
    h = D // 2
    np.testing.assert_allclose(xr[..., :h] ** 2 + xr[..., h:] ** 2, x[..., :h] ** 2 + x[..., h:] ** 2,
                               rtol=1e-12)
    np.testing.assert_allclose(A.rope_transpose(xr, c, s), x, atol=1e-12)


def test_rotated_score_depends_on_distance_only():
    rng = np.random.default_rng(83)
    L, D = 96, 16
    c, s = _tables(L, D)
    qv, kv = _rand(D, rng), _rand(D, rng)
    x = np.zeros((1, L, 1, D))
    x[0, :, 0] = qv
    y = np.zeros((1, L, 1, D))
    y[0, :, 0] = kv
    qr, kr = A.rope(x, c, s)[0, :, 0], A.rope(y, c, s)[0, :, 0]
    for m, n, d in ((10, 3, 20), (40, 40, 50), (5, 60, 30)):
        assert abs(qr[m] @ kr[n] - qr[m + d] @ kr[n + d]) < 1e-10


def _complex_rope_torch(x, ang):
    h = x.shape[-1] // 2
    z = torch.complex(x[..., :h], x[..., h:]) * torch.exp(1j * ang)[None, :, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def test_equals_complex_rotation_with_library_attention():
    rng = np.random.default_rng(84)
    B, L, H, D = 2, 128, 2, 16
    q, k, v, do = (_rand((B, L, H, D), rng) for _ in range(4))
    i = np.arange(D // 2)
    ang = np.arange(L)[:, None] * 10000.0 ** (-2.0 * i / D)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    sc = 1 / math.sqrt(D)
    o = A.blockdiag_rotary_fwd(q, k, v, c, s, sc)
    grads = A.blockdiag_rotary_bwd(q, k, v, do, c, s, sc)
    tq, tk, tv = (torch.tensor(t, requires_grad=True) for t in (q, k, v))
    ta = torch.tensor(ang)
    qr, kr = _complex_rope_torch(tq, ta), _complex_rope_torch(tk, ta)
    blk = torch.arange(L) // 64
    mask = blk[:, None] == blk[None, :]
    to = torch.nn.functional.scaled_dot_product_attention(
        qr.transpose(1, 2), kr.transpose(1, 2), tv.transpose(1, 2), attn_mask=mask, scale=sc).transpose(1, 2)
    to.backward(torch.tensor(do))
    np.testing.assert_allclose(o, to.detach().numpy(), atol=1e-12)
    for a, t in zip(grads, (tq, tk, tv)):
        np.testing.assert_allclose(a, t.grad.numpy(), atol=1e-11)


def _fd_pin():
    rng = np.random.default_rng(85)
    B, L, H, D, h = 1, 64, 1, 4, 1e-6
    q, k, v, do = (_rand((B, L, H, D), rng) for _ in range(4))
    c, s = _tables(L, D, base=3.0)
    sc = 0.5
    grads = A.blockdiag_rotary_bwd(q, k, v, do, c, s, sc)
    for which, g in enumerate(grads):
        # a few sampled coordinates per tensor (the loss couples a whole block)
        for idx in ((0, 3, 0, 1), (0, 40, 0, 2), (0, 63, 0, 0)):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = float(np.sum(A.blockdiag_rotary_fwd(*args, c, s, sc) * do))
            args[which][idx] -= 2 * h
            lm = float(np.sum(A.blockdiag_rotary_fwd(*args, c, s, sc) * do))
            assert abs((lp - lm) / (2 * h) - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (which, idx)


def test_finite_differences():
    _fd_pin()


def test_planted_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(A, "rope_transpose", A.rope)  # backward rotates the wrong way
    with pytest.raises(AssertionError):
        _fd_pin()


def test_backward_from_rotated_inputs_equals_backward_from_unrotated():
    rng = np.random.default_rng(87)
    B, L, H, D = 2, 128, 2, 16
    q, k, v, do = (_rand((B, L, H, D), rng) for _ in range(4))
    c, s = _tables(L, D)
    ref = A.blockdiag_rotary_bwd(q, k, v, do, c, s, 0.3)
    got = A.blockdiag_rotary_bwd_from_rotated(A.rope(q, c, s), A.rope(k, c, s), v, do, c, s, 0.3)
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a, b, atol=1e-12)
    # and with unrelated q_r, k_r it is not the rotation-free backward
    plain = A.blockdiag_bwd(q, k, v, do, 0.3)
    dq_wrong = A.blockdiag_rotary_bwd_from_rotated(q, k, v, do, c, s, 0.3)[0]
    assert np.abs(dq_wrong - plain[0]).max() > 1e-3


def test_jagged_rotary_on_64_token_sequences_equals_block_diagonal_rotary():
    # Sequences of 64 tokens each: a row's position in its sequence is its
    # index mod 64 and attention never crosses a 64-token block, so the
    # jagged rotary forward and backward equal the block-diagonal ones.
    rng = np.random.default_rng(88)
    B, L, H, D = 3, 64, 2, 16
    q, k, v, do = (_rand((B, L, H, D), rng) for _ in range(4))
    c, s = _tables(L, D)
    offs = np.arange(B + 1) * L
    flat = lambda t: t.reshape(B * L, H, D)
    o_j, _ = A.jagged_rotary_fwd(flat(q), flat(k), flat(v), offs, c, s, 0.3)
    np.testing.assert_allclose(o_j, flat(A.blockdiag_rotary_fwd(q, k, v, c, s, 0.3)), atol=1e-12)
    qr, kr = A.rope(q, c, s), A.rope(k, c, s)
    np.testing.assert_allclose(A.jagged_rope(flat(q), offs, c, s), flat(qr), atol=1e-14)
    got = A.jagged_rotary_bwd_from_rotated(flat(qr), flat(kr), flat(v), flat(do), offs, c, s, 0.3)
    ref = A.blockdiag_rotary_bwd_from_rotated(qr, kr, v, do, c, s, 0.3)
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a, flat(b), atol=1e-12)


def test_jagged_rotary_backward_matches_finite_differences():
    # d/dq of sum(O * dO) with O = attention(rope(q), rope(k), v) on ragged
    # sequences (positions restart at every sequence start).
    rng = np.random.default_rng(89)
    lengths, H, D = [3, 5, 1], 1, 4
    offs = np.concatenate([[0], np.cumsum(lengths)])
    T = int(offs[-1])
    q, k, v, do = (_rand((T, H, D), rng) for _ in range(4))
    c, s = _tables(max(lengths), D)
    sc = 0.7
    grads = A.jagged_rotary_bwd_from_rotated(A.jagged_rope(q, offs, c, s), A.jagged_rope(k, offs, c, s),
                                             v, do, offs, c, s, sc)
    eps = 1e-6
    for which, g in ((0, grads[0]), (1, grads[1])):
        for idx in [(0, 0, 1), (4, 0, 3), (8, 0, 0)]:
            args = [q.copy(), k.copy(), v]
            args[which][idx] += eps
            lp = float(np.sum(A.jagged_rotary_fwd(*args, offs, c, s, sc)[0] * do))
            args[which][idx] -= 2 * eps
            lm = float(np.sum(A.jagged_rotary_fwd(*args, offs, c, s, sc)[0] * do))
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, fd, g[idx])
