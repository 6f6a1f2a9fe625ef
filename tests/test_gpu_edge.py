"""GPU edge cases of the jagged path: zero-length sequences between, before
and after non-empty ones (forward and backward against the fp64 oracle),
and a batch whose sequences are all empty (nothing to compute: empty
outputs, no error)."""

import math

import numpy as np
import pytest
import torch

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from oracle import attention as A
from tests._util import assert_close, assert_lse, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
def test_zero_length_sequences(D):
    lengths = [0, 5, 0, 0, 130, 64, 0, 257, 0]
    H = 2
    inp = W.jagged_inputs(lengths, H, D, 23, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths)).cuda()
    plan = jfa.Plan(off, H, D)
    o, lse = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan)
    grads = jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, plan=plan)
    plan.check()
    s = 1 / math.sqrt(D)
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    offs = off.cpu().numpy()
    ref_o, ref_lse = A.jagged_fwd(q, k, v, offs, s)
    assert_close(o, ref_o, "O", bf16_out=True)
    assert_lse(lse, ref_lse)
    for name, g, r in zip(("dQ", "dK", "dV"), grads, A.jagged_bwd(q, k, v, do, offs, s)):
        assert_close(g, r, name, bf16_out=True)


def test_all_empty_batch():
    lengths = [0, 0, 0]
    H, D = 2, 128
    inp = W.jagged_inputs(lengths, H, D, 24, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths, np.int32)).cuda()
    plan = jfa.Plan(off, H, D)
    assert plan.n_fwd_tiles == 0 and plan.n_bwd_tiles == 0
    o, lse = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan)
    dq, dk, dv = jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, plan=plan)
    plan.check()
    assert tuple(o.shape) == (0, H, D) and tuple(lse.shape) == (H, 0)
    assert all(tuple(t.shape) == (0, H, D) for t in (dq, dk, dv))


def test_bounded_wait_timeout_reported_and_context_usable():
    # A wait that nothing completes gives up after 2 ms and reports through the
    # status block; no fault, and the next computation on the GPU is correct.
    L = jfa.lib()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert L.jfa_selftest_wait_timeout(jfa._ptr(ws), 256, 2_000_000, jfa._stream()) == 0
    assert L.jfa_check_status(jfa._ptr(ws), jfa._stream()) == jfa.JFA_ERR_TIMEOUT
    assert b"site 99" in L.jfa_last_error()
    assert L.jfa_check_status(jfa._ptr(ws), jfa._stream()) == 0  # cleared by the first check
    lengths, H, D = [70, 200], 2, 128
    inp = W.jagged_inputs(lengths, H, D, 25, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths)).cuda()
    o, lse = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off)
    jfa.check_status()
    ref_o, ref_lse = A.jagged_fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), off.cpu().numpy(),
                                  1 / math.sqrt(D))
    assert_close(o, ref_o, "O", bf16_out=True)
    assert_lse(lse, ref_lse)


def test_dq_accumulator_clearing_in_every_call_order():
    # The jagged forward clears the backward's dQ accumulator when the
    # workspace holds one, and records how many bytes it cleared; the backward
    # clears it itself otherwise, and every backward marks it dirty again.
    # Each order below must give the oracle's gradients.
    H, D = 2, 128
    small, large = [70, 200, 5], [300, 129, 64, 250]
    runs = {}
    for name, lengths, seed in (("small", small, 26), ("large", large, 27)):
        inp = W.jagged_inputs(lengths, H, D, seed, device="cuda")
        off = torch.from_numpy(W.offsets_of(lengths)).cuda()
        ref = A.jagged_bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["do"]),
                           off.cpu().numpy(), 1 / math.sqrt(D))
        runs[name] = (inp, off, ref)
    big_plan = jfa.Plan(runs["large"][1], H, D)
    ws = big_plan.workspace
    plans = {"large": big_plan, "small": jfa.Plan(runs["small"][1], H, D, workspace=ws)}

    def fwd(name):
        inp, off, _ = runs[name]
        return jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=plans[name])

    def bwd_check(name, o, lse, tag):
        inp, off, ref = runs[name]
        got = jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, plan=plans[name])
        plans[name].check()
        for g, r, n in zip(got, ref, ("dQ", "dK", "dV")):
            assert_close(g, r, "%s %s" % (tag, n), bf16_out=True)

    o_s, l_s = fwd("small")
    bwd_check("small", o_s, l_s, "fwd then bwd")
    bwd_check("small", o_s, l_s, "second bwd without a forward")
    o_l, l_l = fwd("large")
    o_s, l_s = fwd("small")  # the last forward cleared fewer bytes than "large" needs
    bwd_check("large", o_l, l_l, "larger bwd after a smaller forward")
    bwd_check("small", o_s, l_s, "bwd after another batch's bwd")
