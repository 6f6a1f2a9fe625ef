"""GPU parity of the masked and cross (varlen) attention paths against the
fp64 oracle, through the C ABI: causal and sliding-window band masks on
jagged self-attention, separate query / key-value offsets (including
queries that see no key and keys that no query sees), and the
deterministic dQ reduction (bit-identical from run to run)."""

import math

import numpy as np
import pytest
import torch

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from oracle import attention as A
from tests._util import assert_close, assert_lse, f64

pytestmark = pytest.mark.gpu

RAGGED = [1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 513]


def _cross_inputs(q_lengths, kv_lengths, H, D, seed):
    q = W.jagged_inputs(q_lengths, H, D, seed, device="cuda")
    kv = W.jagged_inputs(kv_lengths, H, D, seed + 500, device="cuda")
    return {"q": q["q"], "do": q["do"], "k": kv["k"], "v": kv["v"]}


def _run(inp, q_lengths, kv_lengths, H, D, window, det=False, plan=None):
    qo = torch.from_numpy(W.offsets_of(q_lengths)).cuda()
    ko = torch.from_numpy(W.offsets_of(kv_lengths)).cuda()
    plan = plan or jfa.Plan(ko, H, D, kind="varlen", q_offsets=qo, window=window,
                            deterministic=det)
    o, lse = jfa.jfa_varlen_fwd(inp["q"], inp["k"], inp["v"], qo, ko, window=window, plan=plan)
    g = jfa.jfa_varlen_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], qo, ko, window=window,
                           deterministic=det, plan=plan)
    plan.check()
    return o, lse, g


def _check(inp, q_lengths, kv_lengths, D, window, got):
    o, lse, g = got
    s = 1 / math.sqrt(D)
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    qo, ko = W.offsets_of(q_lengths), W.offsets_of(kv_lengths)
    ro, rl = A.varlen_fwd(q, k, v, qo, ko, s, window)
    assert_close(o, ro, "O", bf16_out=True)
    assert_lse(lse, rl)
    for name, a, b in zip(("dQ", "dK", "dV"), g, A.varlen_bwd(q, k, v, do, qo, ko, s, window)):
        assert_close(a, b, name, bf16_out=True)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("window", [(-1, 0), (127, 0), (0, 0), (63, 64), (300, 5), (-1, 130)])
def test_band_masks_ragged(D, window):
    H = 2
    inp = W.jagged_inputs(RAGGED, H, D, 91, device="cuda")
    _check(inp, RAGGED, RAGGED, D, window, _run(inp, RAGGED, RAGGED, H, D, window))


def test_unmasked_varlen_self_equals_jfa():
    # Same kernel configuration as jfa_fwd / jfa_bwd: identical O, LSE, dK, dV.
    lengths, H, D = [300, 5, 700, 129], 2, 128
    inp = W.jagged_inputs(lengths, H, D, 92, device="cuda")
    o, lse, g = _run(inp, lengths, lengths, H, D, (-1, -1))
    off = torch.from_numpy(W.offsets_of(lengths)).cuda()
    o2, l2 = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off)
    g2 = jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], o2, l2, inp["do"], off)
    jfa.check_status()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    assert torch.equal(g[1], g2[1]) and torch.equal(g[2], g2[2])
    assert_close(g[0], g2[0], "dQ", atol=1e-2, rl2=1e-3)


@pytest.mark.parametrize("window", [(-1, -1), (-1, 0), (40, 10)])
def test_cross_attention(window):
    # Separate offsets: more queries than keys, fewer, none, and no keys at all;
    # with the causal mask the first Lq - Lk queries of a sequence see no key
    # (O = 0, LSE = -inf) and, with Lq < Lk, leading keys may see no query.
    ql = [130, 7, 0, 300, 64, 5]
    kl = [40, 200, 9, 300, 0, 513]
    H, D = 2, 128
    inp = _cross_inputs(ql, kl, H, D, 93)
    _check(inp, ql, kl, D, window, _run(inp, ql, kl, H, D, window))


@pytest.mark.parametrize("window", [(-1, -1), (-1, 0)])
def test_deterministic_dq_is_bit_identical(window):
    lengths, H, D = [700, 129, 2048, 64, 1], 2, 128
    inp = W.jagged_inputs(lengths, H, D, 94, device="cuda")
    qo = torch.from_numpy(W.offsets_of(lengths)).cuda()
    plan = jfa.Plan(qo, H, D, kind="varlen", window=window, deterministic=True)
    runs = [_run(inp, lengths, lengths, H, D, window, det=True, plan=plan) for _ in range(3)]
    for r in runs[1:]:
        assert torch.equal(r[2][0], runs[0][2][0]), "deterministic dQ changed between runs"
        assert torch.equal(r[2][1], runs[0][2][1]) and torch.equal(r[2][2], runs[0][2][2])
    _check(inp, lengths, lengths, D, window, runs[0])
    # dK, dV do not depend on the dQ mode; dQ agrees with the atomic reduction
    nd = _run(inp, lengths, lengths, H, D, window)
    assert torch.equal(nd[2][1], runs[0][2][1]) and torch.equal(nd[2][2], runs[0][2][2])
    assert_close(nd[2][0], runs[0][2][0], "dQ atomic vs ordered", atol=1e-2, rl2=1e-3)


def test_deterministic_cross_with_window():
    ql, kl = [300, 0, 77, 129], [129, 50, 300, 1000]
    H, D = 2, 64
    inp = _cross_inputs(ql, kl, H, D, 95)
    _check(inp, ql, kl, D, (100, 3), _run(inp, ql, kl, H, D, (100, 3), det=True))


def test_gem_causal_sampled():
    # The GEM-shaped batch with a causal mask, checked on sampled sequences
    # (every head), like the unmasked configuration test.
    L = W.lengths_for("gem")
    H, D = 4, 128
    inp = W.jagged_inputs(L, H, D, W.SEEDS["gem"], device="cuda")
    o, lse, g = _run(inp, L, L, H, D, (-1, 0))
    offs = W.offsets_of(L)
    rng = np.random.default_rng(96)
    pick = sorted(set(rng.choice(len(L), 6, replace=False).tolist()) | {int(np.argmax(L))})
    s = 1 / math.sqrt(D)
    for b in pick:
        a, e = int(offs[b]), int(offs[b + 1])
        for h in range(H):
            Q, K, V, dO = (f64(inp[n][a:e, h]) for n in ("q", "k", "v", "do"))
            ro, rl = A.seq_fwd(Q, K, V, s, (-1, 0))
            assert_close(o[a:e, h], ro, "O[b=%d,h=%d]" % (b, h))
            assert_lse(lse[h, a:e], rl, "LSE[b=%d,h=%d]" % (b, h))
            for name, got, r in zip(("dQ", "dK", "dV"), g, A.seq_bwd(Q, K, V, dO, s, window=(-1, 0))):
                assert_close(got[a:e, h], r, "%s[b=%d,h=%d]" % (name, b, h))


def test_gem_cross_sampled():
    # The GEM cross-attention batch at full size: GEM query lengths against
    # key/value lengths drawn the same way with their own seed (separate
    # offsets, no mask), in the bench's launch configuration; sampled
    # sequences (every head) against the oracle.
    Lq = W.lengths_for("gem")
    Lk = W.lengths_for("gem", seed=W.KV_SEEDS["gem_cross"])
    H, D = 4, 128
    inp = _cross_inputs(Lq, Lk, H, D, W.SEEDS["gem_cross"])
    o, lse, g = _run(inp, Lq, Lk, H, D, (-1, -1))
    qo, ko = W.offsets_of(Lq), W.offsets_of(Lk)
    rng = np.random.default_rng(97)
    pick = sorted(set(rng.choice(len(Lq), 6, replace=False).tolist()) |
                  {int(np.argmax(Lq)), int(np.argmax(Lk))})
    s = 1 / math.sqrt(D)
    for b in pick:
        qa, qe, ka, ke = int(qo[b]), int(qo[b + 1]), int(ko[b]), int(ko[b + 1])
        for h in range(H):
            Q, dO = f64(inp["q"][qa:qe, h]), f64(inp["do"][qa:qe, h])
            K, V = f64(inp["k"][ka:ke, h]), f64(inp["v"][ka:ke, h])
            ro, rl = A.seq_fwd(Q, K, V, s)
            assert_close(o[qa:qe, h], ro, "O[b=%d,h=%d]" % (b, h))
            assert_lse(lse[h, qa:qe], rl, "LSE[b=%d,h=%d]" % (b, h))
            rq, rk, rv = A.seq_bwd(Q, K, V, dO, s)
            assert_close(g[0][qa:qe, h], rq, "dQ[b=%d,h=%d]" % (b, h))
            assert_close(g[1][ka:ke, h], rk, "dK[b=%d,h=%d]" % (b, h))
            assert_close(g[2][ka:ke, h], rv, "dV[b=%d,h=%d]" % (b, h))


def test_long_sequence_sliding_window_sampled():
    # The stress batch (four 16384-token sequences) with a causal window of
    # 1024 keys; rows of one long sequence checked on every head.
    L = W.lengths_for("stress")
    H, D = 4, 128
    window = (1023, 0)
    inp = W.jagged_inputs(L, H, D, W.SEEDS["stress"], device="cuda")
    o, lse, g = _run(inp, L, L, H, D, window)
    offs = W.offsets_of(L)
    b = int(np.flatnonzero(L == 16384)[0])
    a = int(offs[b])
    s = 1 / math.sqrt(D)
    rows = np.arange(5000, 5000 + 256)  # far from the sequence start
    keys = slice(a + rows[0] - 1023, a + rows[-1] + 1)
    for h in range(H):
        # Within the key slice [r0 - 1023, r_last], row i sees keys [i, i + 1023]:
        # the same band with the slice's bottom-right alignment (shift = 1023).
        Q = f64(inp["q"][a + rows, h])
        K, V = f64(inp["k"][keys, h]), f64(inp["v"][keys, h])
        ro, rl = A.seq_fwd(Q, K, V, s, window)
        assert_close(o[a + rows, h], ro, "O[h=%d]" % h)
        assert_lse(lse[h, a + rows], rl, "LSE[h=%d]" % h)
    # gradients of the whole long sequence, one head
    h = 1
    e = int(offs[b + 1])
    Q, K, V, dO = (f64(inp[n][a:e, h]) for n in ("q", "k", "v", "do"))
    for name, got, r in zip(("dQ", "dK", "dV"), g, A.seq_bwd(Q, K, V, dO, s, window=window)):
        assert_close(got[a:e, h], r, "%s[h=%d]" % (name, h))
