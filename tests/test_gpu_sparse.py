"""GPU parity of block-sparse attention (jfa_sparse_fwd / jfa_sparse_bwd: a
128 x 128 block mask per sequence, separate query and key/value offsets)
against the fp64 oracle, through the C ABI; plus two exact pins against
other GPU paths that walk the same keys in the same order with the same
arithmetic: an all-ones mask equals the unmasked varlen kernels, and the
identity mask equals jagged attention on the 128-token pieces."""

import ctypes
import math

import numpy as np
import pytest
import torch

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from oracle import attention as A
from tests._util import assert_close, assert_lse, f64

pytestmark = pytest.mark.gpu

RAGGED = [1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 513, 0, 700]


def _cross_inputs(q_lengths, kv_lengths, H, D, seed):
    q = W.jagged_inputs(q_lengths, H, D, seed, device="cuda")
    kv = W.jagged_inputs(kv_lengths, H, D, seed + 500, device="cuda")
    return {"q": q["q"], "do": q["do"], "k": kv["k"], "v": kv["v"]}


def _offs(q_lengths, kv_lengths, dtype=np.int64):
    return (torch.from_numpy(W.offsets_of(q_lengths, dtype)).cuda(),
            torch.from_numpy(W.offsets_of(kv_lengths, dtype)).cuda())


def _run(inp, q_lengths, kv_lengths, H, D, masks, dtype=np.int64):
    qo, ko = _offs(q_lengths, kv_lengths, dtype)
    plan = jfa.Plan(ko, H, D, kind="sparse", q_offsets=qo, block_masks=masks)
    o, lse = jfa.jfa_sparse_fwd(inp["q"], inp["k"], inp["v"], qo, ko, plan=plan)
    g = jfa.jfa_sparse_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], qo, ko, plan=plan)
    plan.check()
    return o, lse, g


def _check(inp, q_lengths, kv_lengths, D, masks, got):
    o, lse, g = got
    s = 1 / math.sqrt(D)
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    qo, ko = W.offsets_of(q_lengths), W.offsets_of(kv_lengths)
    ro, rl = A.blocksparse_fwd(q, k, v, qo, ko, masks, s)
    assert_close(o, ro, "O", bf16_out=True)
    assert_lse(lse, rl)
    for name, a, b in zip(("dQ", "dK", "dV"), g, A.blocksparse_bwd(q, k, v, do, qo, ko, masks, s)):
        assert_close(a, b, name, bf16_out=True)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("density", [0.3, 0.7])
def test_random_masks_ragged_self(D, density):
    H = 2
    rng = np.random.default_rng(141)
    masks = [rng.random((-(-n // 128),) * 2) < density for n in RAGGED]
    inp = W.jagged_inputs(RAGGED, H, D, 142, device="cuda")
    _check(inp, RAGGED, RAGGED, D, masks, _run(inp, RAGGED, RAGGED, H, D, masks))


@pytest.mark.parametrize("D,dtype", [(64, np.int64), (128, np.int64), (128, np.int32)])
def test_block_causal_cross(D, dtype):
    # Lq != Lk, empty query and empty key sequences, block-causal masks
    H = 2
    ql = [300, 0, 129, 700, 64, 513, 5]
    kl = [129, 40, 0, 1000, 640, 513, 300]
    masks = W.block_masks(ql, kl, 143, density=0.5)
    inp = _cross_inputs(ql, kl, H, D, 144)
    _check(inp, ql, kl, D, masks, _run(inp, ql, kl, H, D, masks, dtype))


def test_empty_block_rows_and_columns_are_exact_zeros():
    # A query block row with no key block: O = 0, LSE = -inf, dQ = 0; a key
    # block column that no query block sees: dK = dV = 0.
    H, D = 2, 128
    lengths = [600, 300]
    m0 = np.ones((5, 5), bool)
    m0[1, :] = False   # rows 128..255 see nothing
    m0[:, 3] = False   # keys 384..511 are seen by nobody
    m1 = np.zeros((3, 3), bool)  # the whole second sequence sees nothing
    masks = [m0, m1]
    inp = W.jagged_inputs(lengths, H, D, 145, device="cuda")
    o, lse, (dq, dk, dv) = got = _run(inp, lengths, lengths, H, D, masks)
    assert bool((o[128:256] == 0).all()) and bool((o[600:] == 0).all())
    assert bool(torch.isneginf(lse[:, 128:256]).all()) and bool(torch.isneginf(lse[:, 600:]).all())
    assert bool((dq[128:256] == 0).all()) and bool((dq[600:] == 0).all())
    assert bool((dk[384:512] == 0).all()) and bool((dv[384:512] == 0).all())
    assert bool((dk[600:] == 0).all()) and bool((dv[600:] == 0).all())
    _check(inp, lengths, lengths, D, masks, got)


@pytest.mark.parametrize("D", [64, 128])
def test_all_ones_mask_equals_unmasked_varlen(D):
    # Every tile walks all of its keys (queries) in order: O, LSE, dK and dV
    # are bit-identical to the unmasked varlen kernels; dQ differs only by the
    # order of its reduce-adds.
    H = 2
    ql = [300, 129, 700, 1, 513]
    kl = [200, 640, 700, 129, 5]
    masks = [np.ones((-(-a // 128), -(-b // 128)), bool) for a, b in zip(ql, kl)]
    inp = _cross_inputs(ql, kl, H, D, 146)
    o, lse, g = _run(inp, ql, kl, H, D, masks)
    qo, ko = _offs(ql, kl)
    vo, vl = jfa.jfa_varlen_fwd(inp["q"], inp["k"], inp["v"], qo, ko)
    vg = jfa.jfa_varlen_bwd(inp["q"], inp["k"], inp["v"], vo, vl, inp["do"], qo, ko)
    assert torch.equal(o, vo) and torch.equal(lse, vl)
    assert torch.equal(g[1], vg[1]) and torch.equal(g[2], vg[2])
    assert_close(g[0], vg[0], "dQ (reduction order)", atol=1e-2, rl2=1e-3)


@pytest.mark.parametrize("D", [64, 128])
def test_identity_mask_equals_jagged_pieces(D):
    # The identity block mask is jagged attention over the 128-token pieces
    # of each sequence; each query block gets its dQ from one key block only,
    # so all outputs are bit-identical.
    H = 2
    lengths = [384, 256, 130, 1]
    masks = [np.eye(-(-n // 128), dtype=bool) for n in lengths]
    pieces = []
    for n in lengths:
        pieces += [min(128, n - s) for s in range(0, n, 128)]
    inp = W.jagged_inputs(lengths, H, D, 147, device="cuda")
    o, lse, g = _run(inp, lengths, lengths, H, D, masks)
    po = torch.from_numpy(W.offsets_of(pieces)).cuda()
    jo, jl = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], po)
    jg = jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], jo, jl, inp["do"], po)
    assert torch.equal(o, jo) and torch.equal(lse, jl)
    for a, b in zip(g, jg):
        assert torch.equal(a, b)


def test_gem_sparse_sampled():
    # The GEM batch with its block-causal masks, full size, in the launch
    # configuration the benchmark times; sampled sequences (every head)
    # against the oracle.
    L = W.lengths_for("gem")
    H, D = 4, 128
    masks = W.block_masks(L, L, W.MASK_SEEDS["gem_sparse"], density=0.5)
    inp = W.jagged_inputs(L, H, D, W.SEEDS["gem_sparse"], device="cuda")
    o, lse, g = _run(inp, L, L, H, D, masks)
    offs = W.offsets_of(L)
    rng = np.random.default_rng(148)
    pick = sorted(set(rng.choice(len(L), 6, replace=False).tolist()) | {int(np.argmax(L))})
    s = 1 / math.sqrt(D)
    for b in pick:
        a, e = int(offs[b]), int(offs[b + 1])
        sub = np.array([0, e - a])
        q, k, v, do = (f64(inp[n][a:e]) for n in ("q", "k", "v", "do"))
        ro, rl = A.blocksparse_fwd(q, k, v, sub, sub, [masks[b]], s)
        assert_close(o[a:e], ro, "O[b=%d]" % b, bf16_out=True)
        assert_lse(lse[:, a:e], rl)
        for name, got, r in zip(("dQ", "dK", "dV"), g,
                                A.blocksparse_bwd(q, k, v, do, sub, sub, [masks[b]], s)):
            assert_close(got[a:e], r, "%s[b=%d]" % (name, b), bf16_out=True)


def test_lists_of_another_batch_stay_inside_the_tensors():
    # The schedule and lists of a larger batch with the call's own (smaller)
    # offsets: listed blocks are clamped to each sequence and tiles past B are
    # skipped, so nothing past the call's rows is written (the outputs are
    # views at the start of larger buffers).
    H, D = 2, 128
    big, small = [300, 129, 700, 640], [70, 500]
    Tb, Ts = sum(big), sum(small)
    rng = np.random.default_rng(149)
    masks = [rng.random((-(-n // 128),) * 2) < 0.6 for n in big]
    ob = torch.from_numpy(W.offsets_of(big)).cuda()
    os_ = torch.from_numpy(W.offsets_of(small)).cuda()
    plan = jfa.Plan(ob, H, D, kind="sparse", block_masks=masks)
    inp = W.jagged_inputs(small, H, D, 150, device="cuda", with_grad=False)
    o = torch.full((Tb, H, D), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H * Tb,), 7.0, dtype=torch.float32, device="cuda")
    L, P = jfa.lib(), jfa._ptr
    sp, tl, lp, ent, meta = plan.fwd_sched
    ws = plan.workspace
    assert L.jfa_sparse_fwd(P(inp["q"]), P(inp["k"]), P(inp["v"]), P(os_), P(os_), jfa.JFA_I64, 2, Ts,
                            Ts, H, D, ctypes.c_float(D ** -0.5), P(sp), P(tl), P(lp), P(ent), P(meta),
                            plan.n_sms, P(o), P(lse), P(ws), ws.numel(), jfa._stream()) == 0, \
        L.jfa_last_error()
    plan.check()
    assert bool((o[Ts:] == 7.0).all()) and bool((lse[H * Ts:] == 7.0).all())
    assert bool(torch.isfinite(o[:Ts].float()).all())


def test_sparse_plan_refuses_a_window_or_deterministic_dq():
    off = torch.from_numpy(W.offsets_of([10])).cuda()
    m = [np.ones((1, 1), bool)]
    with pytest.raises(ValueError):
        jfa.Plan(off, 2, 64, kind="sparse", block_masks=m, window=(-1, 0))
    with pytest.raises(ValueError):
        jfa.Plan(off, 2, 64, kind="sparse", block_masks=m, deterministic=True)
    with pytest.raises(ValueError):
        jfa.Plan(off, 2, 64, kind="sparse")
