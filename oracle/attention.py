"""fp64 NumPy oracle for exact softmax attention over packed (jagged) sequences.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA path never
imports this module and this module imports nothing from the CUDA path.

What is computed is the plain definition of softmax attention, written out
per sequence and per head, with no blocking, fusion or online rescaling:

* forward, for one sequence b and head h ([TLX-BA] section 2, the standard
  FlashAttention loop, which reaches this result tile by tile; [JFA-GEM]
  "Desarrollo de Jagged Flash Attention": FlashAttention run directly on the
  packed Q, K, V with an offsets tensor and no padding):

      S   = scale * Q K^T                      (Lq x Lk)
      P   = row-softmax(S)
      O   = P V
      LSE = max_j S_ij + ln sum_j exp(S_ij - max_j S_ij)   (natural log)

  [TLX-BA] section 2 stores L = m + log(l) for the backward pass; here it is
  expressed in natural-log units of the scaled score.

* backward, with the upstream gradient dO of the same shape as O
  ([TLX-BA] sections 2 and 4: P rebuilt from S, Di = rowsum(dO * O)):

      dV = P^T dO
      dP = dO V^T
      Di = sum_d dO_id O_id
      dS = P * (dP - Di)
      dQ = scale * dS K
      dK = scale * dS^T Q

* broadcast-Q ([JFA-GEM] "Optimización del proceso de Backward y dQ"): one
  dense Q is shared by every jagged K/V sequence; O and LSE are per
  sequence and dQ is the sum over sequences of each sequence's dQ.

* block-diagonal ([TLX-BA] sections 1-2): the sequence is cut into fixed
  64-token blocks and each query block attends only to its own key/value
  block, i.e. the definition above applied to every block independently.

* rotary block-diagonal attention ([TLX-BA] section 1: block attention with
  rotary embeddings fused in, forward and backward). The pages do not write
  the rotation out; the reading used is the usual "rotate half" form: with
  tables cos, sin of shape [L, D/2] indexed by a token's position in its
  sequence, a row x of q or k becomes

      x_r[i]       = x[i] cos[i] - x[i + D/2] sin[i]
      x_r[i + D/2] = x[i + D/2] cos[i] + x[i] sin[i]      (i < D/2),

  attention runs on (q_r, k_r, v), and the gradients of q and k are those of
  q_r and k_r rotated back by the transposed rotation (rotation by -angle).
  The backward is also given from q_r and k_r themselves (the rotary
  layer's saved output), the form whose rotary part the page fuses into the
  attention epilogue. The jagged form rotates each packed row at its
  position counted from the start of its own sequence.

* masked and cross (varlen) attention ([JFA-GEM] "Impacto en el desarrollo
  de modelos generativos": causal, sliding-window and block-sparse masks as
  the natural extensions of the jagged kernels; "Optimización del proceso de
  Backward y dQ": the peeled, masked last K/V block). The pages give no
  formula; the plain reading used here is the usual band mask. Query i of a
  sequence sees key j iff

      (left < 0  or  j >= i + shift - left)  and
      (right < 0 or  j <= i + shift + right),   shift = Lk - Lq,

  i.e. a window of `left` keys before and `right` keys after the key aligned
  with the query (bottom-right alignment, so a causal mask, left = -1 and
  right = 0, lets the last query see every key when Lq != Lk). Masked scores
  are -inf before the softmax; a query that sees no key gets O = 0 and
  LSE = -inf and contributes nothing to the gradients. Cross attention takes
  separate query and key/value offsets: sequence b pairs query rows
  q_offsets[b]:q_offsets[b+1] with key rows kv_offsets[b]:kv_offsets[b+1].

Inputs are NumPy arrays. Callers pass the bf16 values already widened to
float64 (exactly); all arithmetic here is float64. Query rows are processed
in chunks only to bound memory: every row's softmax is still taken over all
of its keys at once.

Layouts (shared with the library's documented ABI, so tests can compare):
packed tensors are [T, H, D] (token, head, dim); offsets is [B+1] with
offsets[0] = 0, non-decreasing, offsets[B] = T; jagged LSE is [H, T];
broadcast-Q O is [B, Lq, H, D] and its LSE is [B, H, Lq]; block-diagonal
tensors are [B, L, H, D].
"""

import numpy as np

ROW_CHUNK = 2048
BLOCK = 64  # [TLX-BA] section 2: fixed 64-token blocks


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def softmax_rows(S):
    """Row softmax of a 2-D fp64 score matrix and its natural-log LSE.

    Returns (P, lse). A row with no keys is not allowed here; callers
    handle empty key sets before calling.
    """
    m = S.max(axis=1, keepdims=True)
    e = np.exp(S - m)
    l = e.sum(axis=1, keepdims=True)
    return e / l, (m + np.log(l))[:, 0]


def band_visible(rows, Lq, Lk, window):
    """Boolean [len(rows), Lk]: which keys each query row of `rows` sees under
    the band mask `window` = (left, right) (see the module docstring; -1 is
    unbounded, (-1, -1) sees every key)."""
    left, right = window
    i = np.asarray(rows, dtype=np.int64)[:, None] + (Lk - Lq)
    j = np.arange(Lk, dtype=np.int64)[None, :]
    ok = np.ones((i.shape[0], Lk), dtype=bool)
    if left >= 0:
        ok &= j >= i - left
    if right >= 0:
        ok &= j <= i + right
    return ok


def masked_softmax_rows(S, ok):
    """Row softmax of S over the entries where `ok` holds; P is 0 elsewhere.
    Rows with no such entry get P = 0 and LSE = -inf."""
    S = np.where(ok, S, -np.inf)
    any_ = ok.any(axis=1)
    m = np.where(any_, S.max(axis=1), 0.0)[:, None]
    e = np.where(ok, np.exp(S - m), 0.0)
    l = e.sum(axis=1, keepdims=True)
    P = np.where(any_[:, None], e / np.where(l > 0, l, 1.0), 0.0)
    lse = np.where(any_, (m + np.log(np.where(l > 0, l, 1.0)))[:, 0], -np.inf)
    return P, lse


def seq_fwd(Q, K, V, scale, window=None):
    """Attention forward for one sequence and one head.

    Q [Lq, D], K [Lk, D], V [Lk, Dv] (fp64). Returns O [Lq, Dv] and
    LSE [Lq]. With Lk = 0 the output is 0 and the LSE is -inf (no keys:
    the empty sum), the reading used for broadcast-Q sequences of length 0.
    `window` = (left, right) applies the band mask of the module docstring.
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    Lq, Lk = Q.shape[0], K.shape[0]
    O = np.zeros((Lq, V.shape[1]))
    lse = np.full(Lq, -np.inf)
    if Lq == 0 or Lk == 0:
        return O, lse
    for r0 in range(0, Lq, ROW_CHUNK):
        r1 = min(Lq, r0 + ROW_CHUNK)
        S = scale * (Q[r0:r1] @ K.T)
        if window is None:
            P, lse[r0:r1] = softmax_rows(S)
        else:
            P, lse[r0:r1] = masked_softmax_rows(S, band_visible(range(r0, r1), Lq, Lk, window))
        O[r0:r1] = P @ V
    return O, lse


def seq_bwd(Q, K, V, dO, scale, O=None, window=None):
    """Attention backward for one sequence and one head.

    Q [Lq, D], K [Lk, D], V [Lk, D], dO [Lq, D] (fp64). O is the oracle's
    own forward output (recomputed when not given). Returns dQ, dK, dV.
    `window` = (left, right) applies the band mask of the module docstring.
    """
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    Lq, Lk = Q.shape[0], K.shape[0]
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    if Lq == 0 or Lk == 0:
        return dQ, dK, dV
    if O is None:
        O, _ = seq_fwd(Q, K, V, scale, window)
    for r0 in range(0, Lq, ROW_CHUNK):
        r1 = min(Lq, r0 + ROW_CHUNK)
        S = scale * (Q[r0:r1] @ K.T)
        if window is None:
            P, _ = softmax_rows(S)
        else:
            P, _ = masked_softmax_rows(S, band_visible(range(r0, r1), Lq, Lk, window))
        dV += P.T @ dO[r0:r1]
        dP = dO[r0:r1] @ V.T
        Di = np.sum(dO[r0:r1] * O[r0:r1], axis=1, keepdims=True)
        dS = P * (dP - Di)
        dQ[r0:r1] = scale * (dS @ K)
        dK += scale * (dS.T @ Q[r0:r1])
    return dQ, dK, dV


def _bounds(offsets):
    off = np.asarray(offsets, dtype=np.int64)
    return [(int(off[b]), int(off[b + 1])) for b in range(len(off) - 1)]


def jagged_fwd(q, k, v, offsets, scale):
    """Jagged self-attention forward over packed [T, H, D] tensors.

    Returns O [T, H, D] and LSE [H, T] (fp64).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, _ = q.shape
    o = np.zeros((T, H, v.shape[2]))
    lse = np.full((H, T), -np.inf)
    for s, e in _bounds(offsets):
        for h in range(H):
            o[s:e, h], lse[h, s:e] = seq_fwd(q[s:e, h], k[s:e, h], v[s:e, h], scale)
    return o, lse


def jagged_bwd(q, k, v, do, offsets, scale):
    """Jagged self-attention backward. Returns dQ, dK, dV [T, H, D] (fp64)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    H = q.shape[1]
    for s, e in _bounds(offsets):
        for h in range(H):
            dq[s:e, h], dk[s:e, h], dv[s:e, h] = seq_bwd(
                q[s:e, h], k[s:e, h], v[s:e, h], do[s:e, h], scale)
    return dq, dk, dv


def varlen_fwd(q, k, v, q_offsets, kv_offsets, scale, window=(-1, -1)):
    """Cross (or self) attention over packed sequences with separate query and
    key/value offsets and an optional band mask. q [Tq, H, D]; k, v [Tk, H, D].
    Returns O [Tq, H, D] and LSE [H, Tq] (fp64)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, H, _ = q.shape
    o = np.zeros((Tq, H, v.shape[2]))
    lse = np.full((H, Tq), -np.inf)
    for (qs, qe), (ks, ke) in zip(_bounds(q_offsets), _bounds(kv_offsets)):
        for h in range(H):
            o[qs:qe, h], lse[h, qs:qe] = seq_fwd(q[qs:qe, h], k[ks:ke, h], v[ks:ke, h], scale,
                                                 tuple(window))
    return o, lse


def varlen_bwd(q, k, v, do, q_offsets, kv_offsets, scale, window=(-1, -1)):
    """Backward of :func:`varlen_fwd`. Returns dQ [Tq, H, D], dK, dV [Tk, H, D]."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    H = q.shape[1]
    for (qs, qe), (ks, ke) in zip(_bounds(q_offsets), _bounds(kv_offsets)):
        for h in range(H):
            dq[qs:qe, h], dk[ks:ke, h], dv[ks:ke, h] = seq_bwd(
                q[qs:qe, h], k[ks:ke, h], v[ks:ke, h], do[qs:qe, h], scale, window=tuple(window))
    return dq, dk, dv


def bcastq_fwd(q, k, v, kv_offsets, scale):
    """Broadcast-Q forward: q [Lq, H, D] shared by every sequence of the
    packed k, v [Tk, H, D]. Returns O [B, Lq, H, D], LSE [B, H, Lq]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Lq, H, _ = q.shape
    bounds = _bounds(kv_offsets)
    o = np.zeros((len(bounds), Lq, H, v.shape[2]))
    lse = np.full((len(bounds), H, Lq), -np.inf)
    for b, (s, e) in enumerate(bounds):
        for h in range(H):
            o[b, :, h], lse[b, h] = seq_fwd(q[:, h], k[s:e, h], v[s:e, h], scale)
    return o, lse


def bcastq_bwd(q, k, v, do, kv_offsets, scale):
    """Broadcast-Q backward: do [B, Lq, H, D]. Returns dQ [Lq, H, D] summed
    over the B sequences, and dK, dV [Tk, H, D]."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    H = q.shape[1]
    dq = np.zeros_like(q)
    dk, dv = np.zeros_like(k), np.zeros_like(v)
    for b, (s, e) in enumerate(_bounds(kv_offsets)):
        for h in range(H):
            dq_b, dk[s:e, h], dv[s:e, h] = seq_bwd(
                q[:, h], k[s:e, h], v[s:e, h], do[b, :, h], scale)
            dq[:, h] += dq_b
    return dq, dk, dv


def _blocks(x, block):
    """View [B, L, H, D] as [B*L/block, block, H, D]."""
    B, L, H, D = x.shape
    return x.reshape(B * (L // block), block, H, D)


def blockdiag_fwd(q, k, v, scale, block=BLOCK):
    """Block-diagonal attention forward on [B, L, H, D]; L % block == 0.

    Each block of `block` tokens attends only within itself. Returns O
    [B, L, H, D] (no LSE: [TLX-BA] section 2, none is stored)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, L, H, D = q.shape
    assert L % block == 0
    qb, kb, vb = _blocks(q, block), _blocks(k, block), _blocks(v, block)
    o = np.zeros_like(qb)
    for h in range(H):
        S = scale * np.einsum("nid,njd->nij", qb[:, :, h], kb[:, :, h])
        m = S.max(axis=2, keepdims=True)
        e = np.exp(S - m)
        P = e / e.sum(axis=2, keepdims=True)
        o[:, :, h] = np.einsum("nij,njd->nid", P, vb[:, :, h])
    return o.reshape(B, L, H, v.shape[3])


def blockdiag_bwd(q, k, v, do, scale, block=BLOCK):
    """Block-diagonal attention backward on [B, L, H, D].

    Same formulas as :func:`seq_bwd`, per block, with Di = rowsum(dO * O)
    taken from the oracle's own fp64 O. Returns dQ, dK, dV [B, L, H, D]."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, L, H, D = q.shape
    assert L % block == 0
    qb, kb, vb, dob = (_blocks(x, block) for x in (q, k, v, do))
    dq, dk, dv = np.zeros_like(qb), np.zeros_like(kb), np.zeros_like(vb)
    for h in range(H):
        Q, K, V, dO = qb[:, :, h], kb[:, :, h], vb[:, :, h], dob[:, :, h]
        S = scale * np.einsum("nid,njd->nij", Q, K)
        m = S.max(axis=2, keepdims=True)
        e = np.exp(S - m)
        P = e / e.sum(axis=2, keepdims=True)
        O = np.einsum("nij,njd->nid", P, V)
        dv[:, :, h] = np.einsum("nij,nid->njd", P, dO)
        dP = np.einsum("nid,njd->nij", dO, V)
        Di = np.sum(dO * O, axis=2, keepdims=True)
        dS = P * (dP - Di)
        dq[:, :, h] = scale * np.einsum("nij,njd->nid", dS, K)
        dk[:, :, h] = scale * np.einsum("nij,nid->njd", dS, Q)
    shape = (B, L, H, D)
    return dq.reshape(shape), dk.reshape(shape), dv.reshape(shape)


def rope(x, cos, sin):
    """Rotary embedding of x [B, L, H, D] with tables cos, sin [L, D/2]
    (position = index along L), "rotate half" form (module docstring)."""
    x = _f64(x)
    h = x.shape[-1] // 2
    c = _f64(cos)[None, :, None, :]
    s = _f64(sin)[None, :, None, :]
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def rope_transpose(g, cos, sin):
    """The transposed rotation (rotation by -angle): maps the gradient of a
    rotated tensor to the gradient of the unrotated one."""
    g = _f64(g)
    h = g.shape[-1] // 2
    c = _f64(cos)[None, :, None, :]
    s = _f64(sin)[None, :, None, :]
    lo, hi = g[..., :h], g[..., h:]
    return np.concatenate([lo * c + hi * s, hi * c - lo * s], axis=-1)


def blockdiag_rotary_fwd(q, k, v, cos, sin, scale, block=BLOCK):
    """Block-diagonal attention on rotated q and k. Returns O [B, L, H, D]."""
    return blockdiag_fwd(rope(q, cos, sin), rope(k, cos, sin), v, scale, block)


def blockdiag_rotary_bwd(q, k, v, do, cos, sin, scale, block=BLOCK):
    """Backward of :func:`blockdiag_rotary_fwd` with respect to the
    unrotated q, k and v. Returns dQ, dK, dV [B, L, H, D]."""
    dqr, dkr, dv = blockdiag_bwd(rope(q, cos, sin), rope(k, cos, sin), v, do, scale, block)
    return rope_transpose(dqr, cos, sin), rope_transpose(dkr, cos, sin), dv


def blockdiag_rotary_bwd_from_rotated(q_r, k_r, v, do, cos, sin, scale, block=BLOCK):
    """The combined attention-and-rotary backward ([TLX-BA] section 1: the
    rotary backward fused into the attention backward), taken from the
    rotated q_r, k_r that a rotary layer saves: the block-diagonal attention
    backward on (q_r, k_r, v), then the gradients of q_r and k_r rotated back.
    Returns dQ, dK, dV [B, L, H, D] with respect to the unrotated q, k and v."""
    dqr, dkr, dv = blockdiag_bwd(q_r, k_r, v, do, scale, block)
    return rope_transpose(dqr, cos, sin), rope_transpose(dkr, cos, sin), dv


def jagged_rope(x, offsets, cos, sin):
    """Rotary embedding of packed rows x [T, H, D], each row at its position
    in its own sequence (row - offsets[b]); tables [L, D/2], L at least the
    longest sequence. The jagged form of :func:`rope`."""
    x = _f64(x)
    out = np.empty_like(x)
    for s, e in _bounds(offsets):
        out[s:e] = rope(x[s:e][None], _f64(cos)[:e - s], _f64(sin)[:e - s])[0]
    return out


def jagged_rope_transpose(g, offsets, cos, sin):
    """The transposed rotation of :func:`jagged_rope` (gradient of the rotated
    rows to gradient of the unrotated ones)."""
    g = _f64(g)
    out = np.empty_like(g)
    for s, e in _bounds(offsets):
        out[s:e] = rope_transpose(g[s:e][None], _f64(cos)[:e - s], _f64(sin)[:e - s])[0]
    return out


def jagged_rotary_fwd(q, k, v, offsets, cos, sin, scale):
    """Jagged attention on rotated q and k. Returns O, LSE."""
    return jagged_fwd(jagged_rope(q, offsets, cos, sin), jagged_rope(k, offsets, cos, sin), v,
                      offsets, scale)


def jagged_rotary_bwd_from_rotated(q_r, k_r, v, do, offsets, cos, sin, scale):
    """The combined attention-and-rotary backward on jagged sequences, taken
    from the rotated q_r, k_r: the jagged attention backward on (q_r, k_r, v),
    then the gradients of q_r and k_r rotated back. Returns dQ, dK, dV with
    respect to the unrotated q, k and v."""
    dqr, dkr, dv = jagged_bwd(q_r, k_r, v, do, offsets, scale)
    return (jagged_rope_transpose(dqr, offsets, cos, sin),
            jagged_rope_transpose(dkr, offsets, cos, sin), dv)


# ----------------------------------------------------------- block-sparse masks
SPARSE_BLOCK = 128  # query and key rows per mask block


def block_visible(Lq, Lk, mask):
    """Boolean [Lq, Lk] of a block mask ([JFA-GEM] "Impacto en el desarrollo
    de modelos generativos": sparse-block masks on the jagged kernels; reading
    used: mask[i // 128, j // 128] says whether query i of the sequence sees
    key j, blocks counted from the start of the query and key sequences)."""
    mask = np.asarray(mask, dtype=bool)
    nqb, nkb = -(-Lq // SPARSE_BLOCK), -(-Lk // SPARSE_BLOCK)
    assert mask.shape == (nqb, nkb), (mask.shape, nqb, nkb)
    rows = np.arange(Lq) // SPARSE_BLOCK
    cols = np.arange(Lk) // SPARSE_BLOCK
    return mask[rows][:, cols]


def _sparse_seq(Q, K, V, dO, scale, ok):
    """Forward (and backward when dO is given) of one sequence and head under
    the element mask `ok` [Lq, Lk]: the definitions of the module docstring
    with masked scores at -inf; rows that see no key get O = 0, LSE = -inf
    and no gradient."""
    S = scale * (Q @ K.T)
    P, lse = masked_softmax_rows(S, ok)
    O = P @ V
    if dO is None:
        return O, lse
    dV = P.T @ dO
    dP = dO @ V.T
    Di = np.sum(dO * O, axis=1, keepdims=True)
    dS = P * (dP - Di)
    return scale * dS @ K, scale * dS.T @ Q, dV


def blocksparse_fwd(q, k, v, q_offsets, kv_offsets, masks, scale):
    """Attention with a block mask per sequence (`masks[b]` of shape
    [ceil(Lq_b / 128), ceil(Lk_b / 128)]), separate query and key offsets.
    Returns O [Tq, H, D] and LSE [H, Tq]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, H, _ = q.shape
    o = np.zeros((Tq, H, v.shape[2]))
    lse = np.full((H, Tq), -np.inf)
    for b, ((qs, qe), (ks, ke)) in enumerate(zip(_bounds(q_offsets), _bounds(kv_offsets))):
        if qe == qs or ke == ks:
            continue
        ok = block_visible(qe - qs, ke - ks, masks[b])
        for h in range(H):
            o[qs:qe, h], lse[h, qs:qe] = _sparse_seq(q[qs:qe, h], k[ks:ke, h], v[ks:ke, h], None,
                                                     scale, ok)
    return o, lse


def blocksparse_bwd(q, k, v, do, q_offsets, kv_offsets, masks, scale):
    """Backward of :func:`blocksparse_fwd`. Returns dQ, dK, dV."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    H = q.shape[1]
    for b, ((qs, qe), (ks, ke)) in enumerate(zip(_bounds(q_offsets), _bounds(kv_offsets))):
        if qe == qs or ke == ks:
            continue
        ok = block_visible(qe - qs, ke - ks, masks[b])
        for h in range(H):
            dq[qs:qe, h], dk[ks:ke, h], dv[ks:ke, h] = _sparse_seq(
                q[qs:qe, h], k[ks:ke, h], v[ks:ke, h], do[qs:qe, h], scale, ok)
    return dq, dk, dv
