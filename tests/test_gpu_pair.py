"""GPU checks of the forward on CTA pairs (jfa_fwd_pair: two CTAs of a
cluster compute each product together, M = 256, each loading half of every
K and V tile). Each CTA row still gets exactly the single-CTA kernel's
arithmetic (the same products over the same keys in the same order), so O
and LSE must equal jfa_fwd's bit for bit; they are also compared with the
fp64 oracle, and the backward run on the pair forward's O and LSE must equal
the one run on jfa_fwd's."""

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

# ragged lengths around the 128-row halves, the 256-row products and the
# 512-row pair tiles, with empty sequences
RAGGED = [1, 0, 127, 128, 129, 255, 256, 257, 383, 384, 385, 511, 512, 513, 700, 0, 1024, 1500]


def _both(lengths, H, D, seed):
    inp = W.jagged_inputs(lengths, H, D, seed, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths)).cuda()
    out = {}
    for pair in (False, True):
        plan = jfa.Plan(off, H, D, pair=pair)
        o, lse = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan)
        plan.check()
        out[pair] = (o, lse, plan)
    return inp, off, out


def test_pair_ragged_equals_single_and_oracle():
    H, D = 2, 128
    inp, off, out = _both(RAGGED, H, D, 101)
    (o1, l1, _), (o2, l2, _) = out[False], out[True]
    assert torch.equal(o1, o2), "pair O differs from the single-CTA forward"
    assert torch.equal(l1, l2), "pair LSE differs from the single-CTA forward"
    q, k, v = (f64(inp[n]) for n in ("q", "k", "v"))
    ref_o, ref_lse = A.jagged_fwd(q, k, v, W.offsets_of(RAGGED), 1 / math.sqrt(D))
    assert_close(o2, ref_o, "O", bf16_out=True)
    assert_lse(l2, ref_lse)


def test_pair_backward_on_pair_forward_equals_single():
    H, D = 2, 128
    lengths = [700, 5, 1300, 256, 513]
    inp, off, out = _both(lengths, H, D, 102)
    o, lse, plan = out[True]
    g_pair = jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, plan=plan)
    plan.check()
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    for name, a, b in zip(("dQ", "dK", "dV"), g_pair,
                          A.jagged_bwd(q, k, v, do, W.offsets_of(lengths), 1 / math.sqrt(D))):
        assert_close(a, b, name, bf16_out=True)


@pytest.mark.parametrize("name", ["gem", "stress"])
def test_pair_full_configs_equal_single(name):
    # The full GEM and stress batches: bit-identical to the single-CTA forward,
    # which the configuration tests check against the oracle.
    L = W.lengths_for(name)
    H, D = 4, 128
    inp = W.jagged_inputs(L, H, D, W.SEEDS[name], device="cuda", with_grad=False)
    off = torch.from_numpy(W.offsets_of(L)).cuda()
    res = []
    for pair in (False, True):
        plan = jfa.Plan(off, H, D, pair=pair)
        res.append(jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan))
        plan.check()
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


def test_pair_guards_against_a_schedule_of_another_batch():
    # The pair tile list of a larger batch with the call's own offsets: tiles of
    # sequences past the call's B are skipped and rows are clamped to T, so the
    # results are right and nothing past the call's rows is written (the
    # outputs are views at the start of buffers as large as the larger batch).
    H, D = 2, 128
    big, small = [300, 129, 700, 640], [70, 500]  # each small sequence fits the tiles listed for it
    Tb, Ts = sum(big), sum(small)
    off_big = torch.from_numpy(W.offsets_of(big)).cuda()
    off_small = torch.from_numpy(W.offsets_of(small)).cuda()
    plan_big = jfa.Plan(off_big, H, D, pair=True)
    inp = W.jagged_inputs(small, H, D, 103, device="cuda", with_grad=False)
    o = torch.full((Tb, H, D), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H * Tb,), 7.0, dtype=torch.float32, device="cuda")
    L, P = jfa.lib(), jfa._ptr
    sp, tl = plan_big.fwd_sched
    ws = plan_big.workspace
    assert L.jfa_fwd_pair(P(inp["q"]), P(inp["k"]), P(inp["v"]), P(off_small), jfa.JFA_I64, 2, Ts, H,
                          D, ctypes.c_float(D ** -0.5), P(sp), P(tl), plan_big.n_pairs, P(o),
                          P(lse), P(ws), ws.numel(), jfa._stream()) == 0, L.jfa_last_error()
    plan_big.check()
    assert bool((o[Ts:] == 7.0).all()) and bool((lse[H * Ts:] == 7.0).all())
    q, k, v = (f64(inp[n]) for n in ("q", "k", "v"))
    ref_o, ref_lse = A.jagged_fwd(q, k, v, W.offsets_of(small), 1 / math.sqrt(D))
    assert_close(o[:Ts], ref_o, "O", bf16_out=True)
    assert_lse(lse[:H * Ts].view(H, Ts), ref_lse)


def test_pair_refuses_other_head_dims():
    off = torch.from_numpy(W.offsets_of([10])).cuda()
    with pytest.raises(ValueError):
        jfa.Plan(off, 2, 64, pair=True)
