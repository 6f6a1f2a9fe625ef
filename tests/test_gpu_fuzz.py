"""Seeded random sweeps of the jagged, masked / cross, broadcast-Q,
block-sparse, block-diagonal and rotary paths against the fp64 oracle,
through the C ABI: batch sizes, lengths (zero,
one, every tile edge and random), head counts including odd ones, both head
dimensions, both offset index types and non-default softmax scales, drawn
per case from a fixed seed so that a failure names a reproducible case.

Unusual draws (a larger scale, hundreds of queries on a two-key sequence)
give gradients far above 1 in magnitude. Each output element is a sum of
products whose bf16 operands (P, dS and the inputs) carry a relative rounding
of up to 2^-9, so its error grows with the size of the terms: the absolute
bound here is the usual 2e-2 or 2^-7 (four such roundings) of the tensor's
largest reference magnitude, whichever is larger; the relative L2 bound stays
1e-2."""

import math

import numpy as np
import pytest
import torch

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from oracle import attention as A
from tests._util import ATOL, assert_close, assert_lse, f64

pytestmark = pytest.mark.gpu

EDGES = [0, 1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 384, 385, 511, 512, 513]


def _lengths(rng, lo_b=1, hi_b=12, cap=900):
    B = int(rng.integers(lo_b, hi_b + 1))
    pick_edge = rng.random(B) < 0.5
    return [int(rng.choice(EDGES)) if e else int(rng.integers(1, cap)) for e in pick_edge]


def _close(got, ref, name, bf16_out=True):
    atol = max(ATOL, 2.0 ** -7 * float(np.abs(f64(ref)).max(initial=0.0)))
    assert_close(got, ref, name, atol=atol, bf16_out=bf16_out)


def _case(seed):
    rng = np.random.default_rng(seed)
    H = int(rng.choice([1, 2, 3, 5]))
    D = int(rng.choice([64, 128]))
    idx = np.int32 if rng.random() < 0.5 else np.int64
    # the default 1/sqrt(D), or a larger or smaller one (a larger scale makes
    # the running maximum jump, so the lazy rescale of O runs)
    scale = None if rng.random() < 0.5 else float(rng.choice([0.02, 0.25, 0.5])) / math.sqrt(D) * 8
    return rng, H, D, idx, scale


@pytest.mark.parametrize("seed", range(16))
def test_jagged_random_batches(seed):
    rng, H, D, idx, scale = _case(1000 + seed)
    lengths = _lengths(rng)
    if sum(lengths) == 0:
        lengths[0] = 1
    s = scale if scale is not None else 1 / math.sqrt(D)
    inp = W.jagged_inputs(lengths, H, D, 2000 + seed, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths, idx)).cuda()
    plan = jfa.Plan(off, H, D)
    o, lse = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, scale=scale, plan=plan)
    g = jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, scale=scale, plan=plan)
    plan.check()
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    offs = W.offsets_of(lengths)
    ro, rl = A.jagged_fwd(q, k, v, offs, s)
    tag = "case %d (lengths %s, H=%d, D=%d, %s, scale %s)" % (seed, lengths, H, D, idx.__name__, scale)
    _close(o, ro, "O " + tag)
    assert_lse(lse, rl, "LSE " + tag)
    for name, a, b in zip(("dQ", "dK", "dV"), g, A.jagged_bwd(q, k, v, do, offs, s)):
        _close(a, b, name + " " + tag)


@pytest.mark.parametrize("seed", range(10))
def test_masked_cross_random_batches(seed):
    rng, H, D, idx, scale = _case(3000 + seed)
    ql = _lengths(rng, hi_b=8, cap=700)
    kl = [int(x) if rng.random() < 0.4 else int(rng.integers(0, 700)) for x in ql]
    if sum(ql) == 0:
        ql[0] = 1
    if sum(kl) == 0:
        kl[0] = 1
    window = (int(rng.choice([-1, 0, 5, 64, 200])), int(rng.choice([-1, 0, 3, 128])))
    s = scale if scale is not None else 1 / math.sqrt(D)
    qi = W.jagged_inputs(ql, H, D, 4000 + seed, device="cuda")
    ki = W.jagged_inputs(kl, H, D, 4500 + seed, device="cuda")
    q, do, k, v = qi["q"], qi["do"], ki["k"], ki["v"]
    qo = torch.from_numpy(W.offsets_of(ql, idx)).cuda()
    ko = torch.from_numpy(W.offsets_of(kl, idx)).cuda()
    plan = jfa.Plan(ko, H, D, kind="varlen", q_offsets=qo, window=window)
    o, lse = jfa.jfa_varlen_fwd(q, k, v, qo, ko, scale=scale, window=window, plan=plan)
    g = jfa.jfa_varlen_bwd(q, k, v, o, lse, do, qo, ko, scale=scale, window=window, plan=plan)
    plan.check()
    Q, K, V, dO = (f64(x) for x in (q, k, v, do))
    qoh, koh = W.offsets_of(ql), W.offsets_of(kl)
    tag = "case %d (q %s, kv %s, window %s, H=%d, D=%d)" % (seed, ql, kl, window, H, D)
    ro, rl = A.varlen_fwd(Q, K, V, qoh, koh, s, window)
    _close(o, ro, "O " + tag)
    assert_lse(lse, rl, "LSE " + tag)
    for name, a, b in zip(("dQ", "dK", "dV"), g, A.varlen_bwd(Q, K, V, dO, qoh, koh, s, window)):
        _close(a, b, name + " " + tag)


@pytest.mark.parametrize("seed", range(6))
def test_bcastq_random_batches(seed):
    rng, H, D, idx, scale = _case(5000 + seed)
    lengths = _lengths(rng, hi_b=10, cap=600)
    if sum(lengths) == 0:
        lengths[0] = 1
    Lq = int(rng.choice([1, 37, 128, 129, 256, 300]))
    s = scale if scale is not None else 1 / math.sqrt(D)
    inp = W.bcast_inputs(lengths, Lq, H, D, 6000 + seed, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths, idx)).cuda()
    plan = jfa.Plan(off, H, D, kind="bcast", Lq=Lq)
    o, lse = jfa.jfa_bcastq_fwd(inp["q"], inp["k"], inp["v"], off, scale=scale, plan=plan)
    g = jfa.jfa_bcastq_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, scale=scale,
                           plan=plan)
    plan.check()
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    offs = W.offsets_of(lengths)
    tag = "case %d (lengths %s, Lq=%d, H=%d, D=%d)" % (seed, lengths, Lq, H, D)
    ro, rl = A.bcastq_fwd(q, k, v, offs, s)
    _close(o, ro, "O " + tag)
    assert_lse(lse, rl, "LSE " + tag)
    rdq, rdk, rdv = A.bcastq_bwd(q, k, v, do, offs, s)
    _close(g[0], rdq, "dQ " + tag, bf16_out=False)  # fp32 output: no bf16 rounding slack
    _close(g[1], rdk, "dK " + tag)
    _close(g[2], rdv, "dV " + tag)


@pytest.mark.parametrize("seed", range(8))
def test_block_sparse_random_batches(seed):
    rng, H, D, idx, scale = _case(7000 + seed)
    ql = _lengths(rng, hi_b=8, cap=700)
    kl = [int(x) if rng.random() < 0.5 else int(rng.integers(0, 700)) for x in ql]
    if sum(ql) == 0:
        ql[0] = 1
    if sum(kl) == 0:
        kl[0] = 1
    masks = [rng.random((-(-a // 128), -(-b // 128))) < rng.uniform(0.1, 1.0) for a, b in zip(ql, kl)]
    s = scale if scale is not None else 1 / math.sqrt(D)
    qi = W.jagged_inputs(ql, H, D, 7500 + seed, device="cuda")
    ki = W.jagged_inputs(kl, H, D, 7800 + seed, device="cuda")
    q, do, k, v = qi["q"], qi["do"], ki["k"], ki["v"]
    qo = torch.from_numpy(W.offsets_of(ql, idx)).cuda()
    ko = torch.from_numpy(W.offsets_of(kl, idx)).cuda()
    plan = jfa.Plan(ko, H, D, kind="sparse", q_offsets=qo, block_masks=masks)
    o, lse = jfa.jfa_sparse_fwd(q, k, v, qo, ko, scale=scale, plan=plan)
    g = jfa.jfa_sparse_bwd(q, k, v, o, lse, do, qo, ko, scale=scale, plan=plan)
    plan.check()
    Q, K, V, dO = (f64(x) for x in (q, k, v, do))
    qoh, koh = W.offsets_of(ql), W.offsets_of(kl)
    tag = "case %d (q %s, kv %s, H=%d, D=%d)" % (seed, ql, kl, H, D)
    ro, rl = A.blocksparse_fwd(Q, K, V, qoh, koh, masks, s)
    _close(o, ro, "O " + tag)
    assert_lse(lse, rl, "LSE " + tag)
    for name, a, b in zip(("dQ", "dK", "dV"), g, A.blocksparse_bwd(Q, K, V, dO, qoh, koh, masks, s)):
        _close(a, b, name + " " + tag)


@pytest.mark.parametrize("seed", range(6))
def test_blockdiag_random_shapes(seed):
    rng, H, D, _, scale = _case(8000 + seed)
    B, L = int(rng.integers(1, 5)), 64 * int(rng.integers(1, 11))
    s = scale if scale is not None else 1 / math.sqrt(D)
    inp = W.blockdiag_inputs(B, L, H, D, 8100 + seed, device="cuda")
    o = jfa.blockdiag_fwd(inp["q"], inp["k"], inp["v"], scale=scale)
    g = jfa.blockdiag_bwd(inp["q"], inp["k"], inp["v"], inp["do"], scale=scale)
    jfa.check_status()
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    tag = "case %d (B=%d, L=%d, H=%d, D=%d)" % (seed, B, L, H, D)
    _close(o, A.blockdiag_fwd(q, k, v, s), "O " + tag)
    for name, a, b in zip(("dQ", "dK", "dV"), g, A.blockdiag_bwd(q, k, v, do, s)):
        _close(a, b, name + " " + tag)
    # the same shapes with rotary embeddings: the forward rotates q and k
    # itself; the backward takes the oracle's rotated rows, rounded to bf16
    cos, sin = W.rotary_tables(L, D, device="cuda")
    o_r = jfa.blockdiag_rotary_fwd(inp["q"], inp["k"], inp["v"], cos, sin, scale=scale)
    c, sn = f64(cos), f64(sin)
    _close(o_r, A.blockdiag_rotary_fwd(q, k, v, c, sn, s), "rotary O " + tag)
    qr64, kr64 = A.rope(q, c, sn), A.rope(k, c, sn)
    qr = torch.from_numpy(qr64).to(torch.bfloat16).cuda()
    kr = torch.from_numpy(kr64).to(torch.bfloat16).cuda()
    g_r = jfa.blockdiag_rotary_bwd(qr, kr, inp["v"], inp["do"], cos, sin, scale=scale)
    jfa.check_status()
    ref = A.blockdiag_rotary_bwd_from_rotated(f64(qr), f64(kr), v, do, c, sn, s)
    for name, a, b in zip(("dQ", "dK", "dV"), g_r, ref):
        _close(a, b, "rotary " + name + " " + tag)


@pytest.mark.parametrize("seed", range(4))
def test_jagged_rotary_random_batches(seed):
    rng, H, D, idx, scale = _case(9000 + seed)
    lengths = _lengths(rng, hi_b=8, cap=700)
    if sum(lengths) == 0:
        lengths[0] = 1
    s = scale if scale is not None else 1 / math.sqrt(D)
    offs = W.offsets_of(lengths)
    inp = W.jagged_inputs(lengths, H, D, 9100 + seed, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths, idx)).cuda()
    cos, sin = W.rotary_tables(max(lengths), D, device="cuda")
    c, sn = f64(cos), f64(sin)
    plan = jfa.Plan(off, H, D)
    tag = "case %d (lengths %s, H=%d, D=%d)" % (seed, lengths, H, D)
    q_rot = jfa.jfa_rope(inp["q"], off, cos, sin, plan=plan)
    _close(q_rot, A.jagged_rope(f64(inp["q"]), offs, c, sn), "q_rot " + tag)
    qr = torch.from_numpy(A.jagged_rope(f64(inp["q"]), offs, c, sn)).to(torch.bfloat16).cuda()
    kr = torch.from_numpy(A.jagged_rope(f64(inp["k"]), offs, c, sn)).to(torch.bfloat16).cuda()
    o, lse = jfa.jfa_fwd(qr, kr, inp["v"], off, scale=scale, plan=plan)
    g = jfa.jfa_rotary_bwd(qr, kr, inp["v"], o, lse, inp["do"], off, cos, sin, scale=scale, plan=plan)
    plan.check()
    ref = A.jagged_rotary_bwd_from_rotated(f64(qr), f64(kr), f64(inp["v"]), f64(inp["do"]), offs,
                                           c, sn, s)
    for name, a, b in zip(("dQ", "dK", "dV"), g, ref):
        _close(a, b, name + " " + tag)


@pytest.mark.parametrize("seed", range(6))
def test_schedules_and_modes_agree_random_batches(seed):
    # Every way of running the same batch walks each tile's keys in the same
    # order with the same arithmetic: O and LSE are bit-identical across the
    # static zigzag and naive deals, both dynamic orders and (D = 128) the
    # CTA-pair forward; dK and dV (fixed accumulation order) across the
    # deals; the deterministic dQ across two runs.
    rng, H, D, idx, scale = _case(9500 + seed)
    lengths = _lengths(rng)
    if sum(lengths) == 0:
        lengths[0] = 1
    tag = "case %d (lengths %s, H=%d, D=%d)" % (seed, lengths, H, D)
    inp = W.jagged_inputs(lengths, H, D, 9600 + seed, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths, idx)).cuda()
    q, k, v, do = (inp[n] for n in ("q", "k", "v", "do"))
    ref = None
    for zz in (True, False):
        plan = jfa.Plan(off, H, D, zigzag=zz)
        o, lse = jfa.jfa_fwd(q, k, v, off, scale=scale, plan=plan)
        g = jfa.jfa_bwd(q, k, v, o, lse, do, off, scale=scale, plan=plan)
        plan.check()
        if ref is None:
            ref = (o, lse, g)
        else:
            assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1]), "naive deal O/LSE " + tag
            assert torch.equal(g[1], ref[2][1]) and torch.equal(g[2], ref[2][2]), "naive deal dK/dV " + tag
    for order in ("device", "lpt"):
        dplan = jfa.DynamicPlan(off, H, D, order=order)
        o, lse = jfa.jfa_fwd_dynamic(q, k, v, off, scale=scale, plan=dplan)
        dplan.check()
        assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1]), "dynamic %s %s" % (order, tag)
    if D == 128:
        pplan = jfa.Plan(off, H, D, pair=True)
        o, lse = jfa.jfa_fwd(q, k, v, off, scale=scale, plan=pplan)
        pplan.check()
        assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1]), "pair " + tag
    dets = []
    for _ in range(2):
        vplan = jfa.Plan(off, H, D, kind="varlen", window=(-1, -1), deterministic=True)
        o, lse = jfa.jfa_varlen_fwd(q, k, v, off, off, scale=scale, plan=vplan)
        dets.append(jfa.jfa_varlen_bwd(q, k, v, o, lse, do, off, off, scale=scale, deterministic=True,
                                       plan=vplan))
        vplan.check()
    assert torch.equal(dets[0][0], dets[1][0]), "deterministic dQ differs between runs " + tag
    s = scale if scale is not None else 1 / math.sqrt(D)
    offs = W.offsets_of(lengths)
    Q, K, V, dO = (f64(x) for x in (q, k, v, do))
    for name, a, b in zip(("dQ", "dK", "dV"), dets[0], A.jagged_bwd(Q, K, V, dO, offs, s)):
        _close(a, b, "deterministic " + name + " " + tag)
