"""Pins of the oracle's band-masked and cross (separate q/kv offsets)
attention, and of the scheduler oracle's ranges under a mask (CPU only).

Each pin checks against something other than the oracle's own formula:

* causal self-attention == torch's float64 scaled_dot_product_attention
  with is_causal=True (a library routine), forward and, through autograd,
  backward;
* band windows == the library routine with a boolean mask built by
  torch.tril / torch.triu (a different construction of the band than the
  oracle's index comparison), including cross attention with Lq != Lk and
  the bottom-right alignment;
* closed forms: window (0, 0) lets a query see only its own key, so O = V,
  LSE = s q.k, dQ = dK = 0, dV = dO; a causal first row sees only key 0;
  rows that see no key give O = 0, LSE = -inf and no gradient anywhere;
* an unbounded window equals the unmasked jagged oracle;
* central finite differences of sum(O * dO) under a band mask;
* the backward invariants sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i over
  the rows that see some key;
* scheduler: the closed-form key / query ranges of a tile equal the union of
  visible positions counted from the mask by brute force.
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import sched as S


def _rand(shape, rng):
    return rng.standard_normal(shape)


def _offsets(lengths):
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    off[1:] = np.cumsum(lengths)
    return off


def _lib_mask(Lq, Lk, window):
    """Band mask [Lq, Lk] built with torch.tril / torch.triu: diagonal d of
    tril keeps j <= i + d, of triu keeps j >= i + d."""
    left, right = window
    shift = Lk - Lq
    m = torch.ones(Lq, Lk, dtype=torch.bool)
    if right >= 0:
        m = torch.tril(m, diagonal=shift + right)
    if left >= 0:
        m = torch.triu(m, diagonal=shift - left)
    return m


def _lib_attention(Q, K, V, dO, s, mask=None, causal=False):
    """Library forward and autograd backward for one sequence/head (fp64)."""
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
    o = torch.nn.functional.scaled_dot_product_attention(
        q[None, None], k[None, None], v[None, None], attn_mask=mask, is_causal=causal, scale=s)[0, 0]
    o.backward(torch.tensor(dO, dtype=torch.float64))
    return o.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def test_causal_self_attention_equals_library():
    rng = np.random.default_rng(51)
    lengths = [1, 7, 30, 64]
    H, D = 2, 16
    T = sum(lengths)
    q, k, v, do = (_rand((T, H, D), rng) for _ in range(4))
    off = _offsets(lengths)
    s = 1 / math.sqrt(D)
    o, lse = A.varlen_fwd(q, k, v, off, off, s, (-1, 0))
    dq, dk, dv = A.varlen_bwd(q, k, v, do, off, off, s, (-1, 0))
    for b in range(len(lengths)):
        a, e = off[b], off[b + 1]
        for h in range(H):
            ro, rq, rk, rv = _lib_attention(q[a:e, h], k[a:e, h], v[a:e, h], do[a:e, h], s,
                                            causal=True)
            np.testing.assert_allclose(o[a:e, h], ro, atol=1e-12)
            np.testing.assert_allclose(dq[a:e, h], rq, atol=1e-11)
            np.testing.assert_allclose(dk[a:e, h], rk, atol=1e-11)
            np.testing.assert_allclose(dv[a:e, h], rv, atol=1e-11)
            S_ = s * q[a:e, h] @ k[a:e, h].T
            want = torch.logsumexp(torch.tensor(S_).masked_fill(~_lib_mask(e - a, e - a, (-1, 0)),
                                                                 -math.inf), dim=1).numpy()
            np.testing.assert_allclose(lse[h, a:e], want, atol=1e-12)


@pytest.mark.parametrize("window", [(3, 0), (0, 2), (2, 5), (-1, 2), (4, -1), (0, 0)])
@pytest.mark.parametrize("Lq,Lk", [(20, 20), (9, 23), (23, 23)])
def test_band_windows_equal_library_masks(window, Lq, Lk):
    rng = np.random.default_rng(52)
    D = 8
    Q, dO = _rand((Lq, D), rng), _rand((Lq, D), rng)
    K, V = _rand((Lk, D), rng), _rand((Lk, D), rng)
    s = 0.4
    mask = _lib_mask(Lq, Lk, window)
    seen = mask.any(dim=1).numpy()
    assert seen.all()  # these shapes leave no query without a key
    o, lse = A.seq_fwd(Q, K, V, s, window)
    dq, dk, dv = A.seq_bwd(Q, K, V, dO, s, window=window)
    ro, rq, rk, rv = _lib_attention(Q, K, V, dO, s, mask=mask)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    np.testing.assert_allclose(dq, rq, atol=1e-11)
    np.testing.assert_allclose(dk, rk, atol=1e-11)
    np.testing.assert_allclose(dv, rv, atol=1e-11)


def test_cross_causal_rows_without_keys():
    # Lq > Lk with a causal (bottom-right) mask: the first Lq - Lk rows see no
    # key. They get O = 0 and LSE = -inf, and the other rows' results equal the
    # library on those rows alone (the keyless rows add nothing to dK, dV).
    rng = np.random.default_rng(53)
    Lq, Lk, D, s = 12, 5, 8, 0.5
    Q, dO = _rand((Lq, D), rng), _rand((Lq, D), rng)
    K, V = _rand((Lk, D), rng), _rand((Lk, D), rng)
    o, lse = A.seq_fwd(Q, K, V, s, (-1, 0))
    dq, dk, dv = A.seq_bwd(Q, K, V, dO, s, window=(-1, 0))
    dead = Lq - Lk
    np.testing.assert_array_equal(o[:dead], 0.0)
    assert np.all(np.isneginf(lse[:dead]))
    np.testing.assert_array_equal(dq[:dead], 0.0)
    mask = _lib_mask(Lq, Lk, (-1, 0))[dead:]
    ro, rq, rk, rv = _lib_attention(Q[dead:], K, V, dO[dead:], s, mask=mask)
    np.testing.assert_allclose(o[dead:], ro, atol=1e-12)
    np.testing.assert_allclose(dq[dead:], rq, atol=1e-11)
    np.testing.assert_allclose(dk, rk, atol=1e-11)
    np.testing.assert_allclose(dv, rv, atol=1e-11)


def test_varlen_cross_attention_equals_library_per_sequence():
    rng = np.random.default_rng(54)
    ql, kl = [3, 0, 17, 8], [11, 4, 17, 1]
    H, D, s = 2, 8, 0.3
    q, do = _rand((sum(ql), H, D), rng), _rand((sum(ql), H, D), rng)
    k, v = _rand((sum(kl), H, D), rng), _rand((sum(kl), H, D), rng)
    qo, ko = _offsets(ql), _offsets(kl)
    o, lse = A.varlen_fwd(q, k, v, qo, ko, s)
    dq, dk, dv = A.varlen_bwd(q, k, v, do, qo, ko, s)
    np.testing.assert_array_equal(dk[ko[1]:ko[2]], 0.0)  # sequence 1 has no queries
    for b in range(len(ql)):
        if ql[b] == 0:
            continue
        qa, qe, ka, ke = qo[b], qo[b + 1], ko[b], ko[b + 1]
        for h in range(H):
            ro, rq, rk, rv = _lib_attention(q[qa:qe, h], k[ka:ke, h], v[ka:ke, h], do[qa:qe, h], s)
            np.testing.assert_allclose(o[qa:qe, h], ro, atol=1e-12)
            np.testing.assert_allclose(dq[qa:qe, h], rq, atol=1e-11)
            np.testing.assert_allclose(dk[ka:ke, h], rk, atol=1e-11)
            np.testing.assert_allclose(dv[ka:ke, h], rv, atol=1e-11)


def test_window_zero_closed_form():
    rng = np.random.default_rng(55)
    L, D, s = 9, 6, 0.7
    Q, K, V, dO = (_rand((L, D), rng) for _ in range(4))
    o, lse = A.seq_fwd(Q, K, V, s, (0, 0))
    np.testing.assert_allclose(o, V, rtol=1e-14)
    np.testing.assert_allclose(lse, s * np.sum(Q * K, axis=1), rtol=1e-14)
    dq, dk, dv = A.seq_bwd(Q, K, V, dO, s, window=(0, 0))
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-13)
    np.testing.assert_allclose(dv, dO, rtol=1e-14)


def test_causal_first_row_sees_only_the_first_key():
    rng = np.random.default_rng(56)
    Q, K, V = (_rand((6, 4), rng) for _ in range(3))
    o, lse = A.seq_fwd(Q, K, V, 0.5, (-1, 0))
    np.testing.assert_allclose(o[0], V[0], rtol=1e-14)
    np.testing.assert_allclose(lse[0], 0.5 * Q[0] @ K[0], rtol=1e-14)


def test_unbounded_window_equals_unmasked_jagged():
    rng = np.random.default_rng(57)
    lengths = [5, 0, 33]
    T, H, D = sum(lengths), 2, 8
    q, k, v, do = (_rand((T, H, D), rng) for _ in range(4))
    off = _offsets(lengths)
    o1, l1 = A.jagged_fwd(q, k, v, off, 0.35)
    o2, l2 = A.varlen_fwd(q, k, v, off, off, 0.35, (-1, -1))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    for a, b in zip(A.jagged_bwd(q, k, v, do, off, 0.35), A.varlen_bwd(q, k, v, do, off, off, 0.35)):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("window", [(-1, 0), (2, 1), (1, -1)])
def test_finite_differences_with_band_mask(window):
    rng = np.random.default_rng(58)
    Lq, Lk, D, s, h = 5, 7, 3, 0.6, 1e-6
    Q, dO = _rand((Lq, D), rng), _rand((Lq, D), rng)
    K, V = _rand((Lk, D), rng), _rand((Lk, D), rng)

    def loss(q, k, v):
        o, _ = A.seq_fwd(q, k, v, s, window)
        return float(np.sum(o * dO))

    grads = A.seq_bwd(Q, K, V, dO, s, window=window)
    for which, g in enumerate(grads):
        num = np.zeros_like(g)
        for idx in np.ndindex(g.shape):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            num[idx] = (lp - loss(*args)) / (2 * h)
        assert np.linalg.norm(num - g) <= 1e-6 * max(np.linalg.norm(num), 1e-12), which


@pytest.mark.parametrize("window", [(-1, 0), (3, 2), (0, 0)])
def test_backward_invariants_with_band_mask(window):
    rng = np.random.default_rng(59)
    Lq, Lk, D = 11, 14, 5
    Q, dO = _rand((Lq, D), rng), _rand((Lq, D), rng)
    K, V = _rand((Lk, D), rng), _rand((Lk, D), rng)
    _, dk, dv = A.seq_bwd(Q, K, V, dO, 0.45, window=window)
    seen = A.band_visible(range(Lq), Lq, Lk, window).any(axis=1)
    np.testing.assert_allclose(dk.sum(0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(0), dO[seen].sum(0), atol=1e-12)


# ----------------------------------------------------------------- scheduler


@pytest.mark.parametrize("window", [(-1, -1), (-1, 0), (100, 0), (0, 0), (37, 260), (-1, 5), (300, -1)])
@pytest.mark.parametrize("Lq,Lk", [(1, 1), (300, 300), (130, 700), (700, 130), (513, 513)])
def test_tile_ranges_equal_brute_force_union(window, Lq, Lk):
    vis = A.band_visible(range(Lq), Lq, Lk, window)
    for m in range(-(-Lq // S.FWD_ROWS)):
        r0, r1 = m * S.FWD_ROWS, min(Lq, m * S.FWD_ROWS + S.FWD_ROWS)
        lo, hi = S.fwd_key_range(r0, r1, Lq, Lk, window)
        cols = np.flatnonzero(vis[r0:r1].any(axis=0))
        if cols.size == 0:
            assert hi - lo == 0 or not vis[r0:r1].any()
            continue
        assert lo <= cols[0] and hi >= cols[-1] + 1  # a superset always
        if vis[r0:r1].any(axis=1).all():  # every row sees a key: exactly the union
            assert (lo, hi) == (cols[0], cols[-1] + 1)
    for n in range(-(-Lk // S.BWD_ROWS)):
        k0, k1 = n * S.BWD_ROWS, min(Lk, n * S.BWD_ROWS + S.BWD_ROWS)
        lo, hi = S.bwd_query_range(k0, k1, Lq, Lk, window)
        rows = np.flatnonzero(vis[:, k0:k1].any(axis=1))
        if rows.size == 0:
            assert hi - lo == 0 or not vis[lo:hi, k0:k1].any()
            continue
        assert lo <= rows[0] and hi >= rows[-1] + 1
        if vis[:, k0:k1].any(axis=0).all():  # every key is seen: exactly the union
            assert (lo, hi) == (rows[0], rows[-1] + 1)


def test_unmasked_self_varlen_schedule_equals_jagged_schedule():
    rng = np.random.default_rng(60)
    lengths = list(rng.integers(0, 700, 40))
    for op, rows in (("fwd", S.FWD_ROWS), ("bwd", S.BWD_ROWS)):
        for zz in (True, False):
            a = S.schedule_varlen(lengths, lengths, 3, op, 7, zigzag=zz)
            b = S.schedule(lengths, 3, rows, 7, zigzag=zz)
            assert a == b


def test_causal_schedule_hand_worked():
    # One sequence of 600 tokens, causal, one head, three SMs, forward tiles of
    # 256 rows: m = 0 sees keys [0, 256), m = 1 [0, 512), m = 2 [0, 600).
    # Work 256, 512, 600 -> sorted m = 2, 1, 0 -> SM0, SM1, SM2.
    sm_ptr, tiles = S.schedule_varlen([600], [600], 1, "fwd", 3, window=(-1, 0))
    assert sm_ptr == [0, 1, 2, 3]
    assert tiles == [(0, 0, 2), (0, 0, 1), (0, 0, 0)]
    # Backward key tiles of 128: n = 0..4 are seen by rows [128 n, 600):
    # work 600, 472, 344, 216, 88 -> already in order -> SM0, 1, 2, then
    # pass 1 right to left: n = 3 -> SM2, n = 4 -> SM1.
    sm_ptr, tiles = S.schedule_varlen([600], [600], 1, "bwd", 3, window=(-1, 0))
    assert sm_ptr == [0, 1, 3, 5]
    assert tiles == [(0, 0, 0), (0, 0, 1), (0, 0, 4), (0, 0, 2), (0, 0, 3)]


# ----------------------------------------------------- the pins have teeth

def _band_mutant(kind):
    def band_visible(rows, Lq, Lk, window):
        left, right = window
        if kind == "left/right swapped":
            left, right = right, left
        shift = (Lq - Lk) if kind == "shift sign" else (Lk - Lq)
        if kind == "top-left alignment":
            shift = 0
        i = np.asarray(rows, dtype=np.int64)[:, None] + shift
        j = np.arange(Lk, dtype=np.int64)[None, :]
        ok = np.ones((i.shape[0], Lk), dtype=bool)
        if left >= 0:
            ok &= (j > i - left) if kind == "strict lower edge" else (j >= i - left)
        if right >= 0:
            ok &= j <= i + right
        return ok
    return band_visible


@pytest.mark.parametrize("kind", ["left/right swapped", "shift sign", "top-left alignment",
                                  "strict lower edge"])
def test_band_mutant_is_caught(monkeypatch, kind):
    monkeypatch.setattr(A, "band_visible", _band_mutant(kind))
    pins = [lambda: test_band_windows_equal_library_masks(w, lq, lk)
            for w in [(3, 0), (0, 2), (2, 5)] for lq, lk in [(20, 20), (9, 23)]]
    pins += [test_window_zero_closed_form, test_causal_first_row_sees_only_the_first_key]
    failures = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures > 0, kind
