"""Pins of the oracle's block-sparse attention and of the scheduler oracle's
block-sparse tiles and lists (CPU only). Each pin checks against something
other than the oracle's own formula:

* an all-ones block mask equals the unmasked varlen oracle;
* the identity block mask (each 128-row block sees only its own key block)
  equals jagged attention on 128-token sub-sequences;
* torch's float64 scaled_dot_product_attention with a boolean mask built by
  a Kronecker product of the block mask (a library routine and a different
  construction of the element mask), forward and, through autograd,
  backward, on cross attention with Lq != Lk;
* rows whose block row is empty get O = 0, LSE = -inf and no gradient;
* central finite differences of sum(O * dO);
* the scheduler's entries and works equal those counted by brute force from
  the element mask;
* a planted mistake (the block mask transposed) fails.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import sched as S


def _rand(shape, rng):
    return rng.standard_normal(shape)


def _masks(q_lengths, kv_lengths, rng, p=0.5):
    return [rng.random((-(-lq // 128), -(-lk // 128))) < p for lq, lk in zip(q_lengths, kv_lengths)]


def _offs(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)


def test_all_ones_mask_equals_unmasked():
    rng = np.random.default_rng(121)
    ql, kl, H, D = [300, 129, 5], [200, 260, 130], 2, 16
    q, do = _rand((sum(ql), H, D), rng), _rand((sum(ql), H, D), rng)
    k, v = _rand((sum(kl), H, D), rng), _rand((sum(kl), H, D), rng)
    masks = [np.ones((-(-a // 128), -(-b // 128)), bool) for a, b in zip(ql, kl)]
    o, lse = A.blocksparse_fwd(q, k, v, _offs(ql), _offs(kl), masks, 0.3)
    ro, rl = A.varlen_fwd(q, k, v, _offs(ql), _offs(kl), 0.3)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    np.testing.assert_allclose(lse, rl, atol=1e-12)
    for a, b in zip(A.blocksparse_bwd(q, k, v, do, _offs(ql), _offs(kl), masks, 0.3),
                    A.varlen_bwd(q, k, v, do, _offs(ql), _offs(kl), 0.3)):
        np.testing.assert_allclose(a, b, atol=1e-12)


def test_identity_mask_equals_jagged_on_128_token_pieces():
    rng = np.random.default_rng(122)
    lengths, H, D = [384, 256], 2, 8
    T = sum(lengths)
    q, k, v, do = (_rand((T, H, D), rng) for _ in range(4))
    masks = [np.eye(L // 128, dtype=bool) for L in lengths]
    offs = _offs(lengths)
    pieces = np.arange(0, T + 1, 128)
    o, lse = A.blocksparse_fwd(q, k, v, offs, offs, masks, 0.4)
    ro, rl = A.jagged_fwd(q, k, v, pieces, 0.4)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    np.testing.assert_allclose(lse, rl, atol=1e-12)
    for a, b in zip(A.blocksparse_bwd(q, k, v, do, offs, offs, masks, 0.4),
                    A.jagged_bwd(q, k, v, do, pieces, 0.4)):
        np.testing.assert_allclose(a, b, atol=1e-12)


def test_equals_library_attention_with_kronecker_mask():
    rng = np.random.default_rng(123)
    Lq, Lk, H, D = 300, 420, 2, 16
    q, do = _rand((Lq, H, D), rng), _rand((Lq, H, D), rng)
    k, v = _rand((Lk, H, D), rng), _rand((Lk, H, D), rng)
    mask = rng.random((3, 4)) < 0.6
    mask[:, 0] = True  # every row sees something
    sc = 0.25
    o, lse = A.blocksparse_fwd(q, k, v, [0, Lq], [0, Lk], [mask], sc)
    grads = A.blocksparse_bwd(q, k, v, do, [0, Lq], [0, Lk], [mask], sc)
    em = np.kron(mask, np.ones((128, 128), dtype=bool))[:Lq, :Lk]
    tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2), requires_grad=True) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.tensor(em),
                                                           scale=sc)
    ref.backward(torch.tensor(do.transpose(1, 0, 2)))
    np.testing.assert_allclose(o, ref.detach().numpy().transpose(1, 0, 2), atol=1e-12)
    for a, t in zip(grads, (tq, tk, tv)):
        np.testing.assert_allclose(a, t.grad.numpy().transpose(1, 0, 2), atol=1e-12)


def test_rows_with_an_empty_block_row_see_nothing():
    rng = np.random.default_rng(124)
    L, H, D = 300, 1, 8
    q, k, v, do = (_rand((L, H, D), rng) for _ in range(4))
    mask = np.ones((3, 3), dtype=bool)
    mask[1] = False
    o, lse = A.blocksparse_fwd(q, k, v, [0, L], [0, L], [mask], 0.3)
    dq, dk, dv = A.blocksparse_bwd(q, k, v, do, [0, L], [0, L], [mask], 0.3)
    assert np.all(o[128:256] == 0) and np.all(np.isneginf(lse[:, 128:256]))
    assert np.all(dq[128:256] == 0)
    # the keys still get gradients from the other rows; dV = P^T dO over those rows only
    S_ = 0.3 * q[:, 0] @ k[:, 0].T
    ok = np.ones((L, L), bool)
    ok[128:256] = False
    P, _ = A.masked_softmax_rows(S_, ok)
    np.testing.assert_allclose(dv[:, 0], P.T @ do[:, 0], atol=1e-12)


def test_finite_differences():
    rng = np.random.default_rng(125)
    Lq, Lk, H, D = 140, 260, 1, 4
    q, do = _rand((Lq, H, D), rng), _rand((Lq, H, D), rng)
    k, v = _rand((Lk, H, D), rng), _rand((Lk, H, D), rng)
    mask = np.array([[True, False, True], [False, True, True]])
    sc = 0.6
    grads = A.blocksparse_bwd(q, k, v, do, [0, Lq], [0, Lk], [mask], sc)
    eps = 1e-6
    for which, idx in ((0, (3, 0, 1)), (0, (135, 0, 2)), (1, (200, 0, 0)), (2, (5, 0, 3))):
        args = [q.copy(), k.copy(), v.copy()]
        args[which][idx] += eps
        lp = float(np.sum(A.blocksparse_fwd(*args, [0, Lq], [0, Lk], [mask], sc)[0] * do))
        args[which][idx] -= 2 * eps
        lm = float(np.sum(A.blocksparse_fwd(*args, [0, Lq], [0, Lk], [mask], sc)[0] * do))
        fd = (lp - lm) / (2 * eps)
        assert abs(fd - grads[which][idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx)


@pytest.mark.parametrize("op", ["fwd", "bwd"])
def test_sparse_tiles_equal_brute_force(op):
    rng = np.random.default_rng(126)
    ql, kl = [1, 300, 700, 129, 0, 513], [256, 5, 700, 300, 40, 513]
    masks = _masks(ql, kl, rng)
    tiles = S.sparse_tiles(ql, kl, 2, op, masks)
    for b, h, m, work, ent in tiles:
        em = A.block_visible(ql[b], kl[b], masks[b]) if ql[b] and kl[b] else np.zeros((ql[b], kl[b]), bool)
        if op == "fwd":
            rows = em[256 * m:256 * m + 256]
            want = []
            for j in range(-(-kl[b] // 128)):
                s0 = rows[:128, 128 * j:128 * j + 128].any() if rows.shape[0] else False
                s1 = rows[128:, 128 * j:128 * j + 128].any() if rows.shape[0] > 128 else False
                if s0 or s1:
                    want.append((j, bool(s0), bool(s1)))
            assert ent == want
            assert work == sum(min(kl[b], 128 * j + 128) - 128 * j for j, _, _ in want)
        else:
            cols = em[:, 128 * m:128 * m + 128]
            want = [qb for qb in range(-(-ql[b] // 64)) if cols[64 * qb:64 * qb + 64].any()]
            assert ent == want
            assert work == int(cols.any(axis=1).sum())


def test_transposed_mask_is_caught():
    # a planted mistake: the mask read as [key block, query block]
    rng = np.random.default_rng(127)
    L, H, D = 256, 1, 8
    q, k, v = (_rand((L, H, D), rng) for _ in range(3))
    mask = np.array([[True, True], [False, True]])
    o, _ = A.blocksparse_fwd(q, k, v, [0, L], [0, L], [mask], 0.3)
    o_t, _ = A.blocksparse_fwd(q, k, v, [0, L], [0, L], [mask.T], 0.3)
    em = np.kron(mask, np.ones((128, 128), bool))
    tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2)) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.tensor(em),
                                                           scale=0.3).numpy().transpose(1, 0, 2)
    np.testing.assert_allclose(o, ref, atol=1e-12)
    assert np.abs(o_t - ref).max() > 1e-3
