"""GPU edge cases of the jagged path: zero-length sequences between, before
and after non-empty ones (forward and backward against the fp64 oracle),
and a batch whose sequences are all empty (nothing to compute: empty
outputs, no error)."""

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


def test_pipelined_steps_sharing_a_workspace_match_single_calls():
    # The pattern of the end-to-end measurement: two device buffer sets, host
    # copies on their own streams, plans rebuilt every step on one shared
    # workspace (so each forward clears the accumulator the next backward uses).
    # Every step's outputs must equal a fresh single call on the same inputs
    # (dK, dV, O bit for bit; dQ up to the order of its atomic additions).
    H, D = 2, 128
    lengths = [70, 300, 5, 129]
    comp = torch.cuda.current_stream()
    batches = [W.jagged_inputs(lengths, H, D, 40 + n, device="cuda") for n in range(3)]
    host = [{k: v.cpu().pin_memory() for k, v in b.items()} for b in batches]
    off_host = W.offsets_of(lengths)
    h_off = torch.from_numpy(off_host).pin_memory()
    ws = jfa.Plan(torch.from_numpy(off_host).cuda(), H, D).workspace
    d_in = [{k: torch.empty_like(v) for k, v in batches[0].items()} for _ in range(2)]
    d_off = [torch.empty_like(h_off, device="cuda") for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    outs = []
    for n in range(3):
        b = n & 1
        with torch.cuda.stream(s_in):
            if n >= 2:
                s_in.wait_event(ev_comp[b])
            for k in d_in[b]:
                d_in[b][k].copy_(host[n][k], non_blocking=True)
            d_off[b].copy_(h_off, non_blocking=True)
        comp.wait_stream(s_in)
        x = d_in[b]
        plan = jfa.Plan(d_off[b], H, D, host_offsets=off_host, workspace=ws)
        o, lse = jfa.jfa_fwd(x["q"], x["k"], x["v"], d_off[b], plan=plan)
        g = jfa.jfa_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], d_off[b], plan=plan)
        ev_comp[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            outs.append([t.to("cpu", non_blocking=True) for t in (o,) + tuple(g)])
            for t in (o,) + tuple(g):
                t.record_stream(s_out)
    torch.cuda.synchronize()
    jfa.check_status(ws)
    off = torch.from_numpy(off_host).cuda()
    for n in range(3):
        x = batches[n]
        o, lse = jfa.jfa_fwd(x["q"], x["k"], x["v"], off)
        ref = (o,) + tuple(jfa.jfa_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], off))
        got = outs[n]
        assert torch.equal(got[0], ref[0].cpu()), "O differs at step %d" % n
        assert torch.equal(got[2], ref[2].cpu()) and torch.equal(got[3], ref[3].cpu()), n
        assert_close(got[1], ref[1], "dQ step %d" % n, atol=1e-2, rl2=1e-3)


def _raw_fwd_bwd(q, k, v, do, off_dev, idx, B, T, H, D, plan, o, lse, dq, dk, dv):
    """jfa_fwd then jfa_bwd through the C ABI with explicit sizes and the given
    plan's tile lists (bypassing the binding's plan validation)."""
    L, P, s = jfa.lib(), jfa._ptr, ctypes.c_float(D ** -0.5)
    ws = plan.workspace
    fsp, ftl = plan.fwd_sched
    bsp, btl = plan.bwd_sched
    assert L.jfa_fwd(P(q), P(k), P(v), P(off_dev), idx, B, T, H, D, s, P(fsp), P(ftl), plan.n_sms,
                     P(o), P(lse), P(ws), ws.numel(), jfa._stream()) == 0, L.jfa_last_error()
    assert L.jfa_bwd(P(q), P(k), P(v), P(o), P(lse), P(do), P(off_dev), idx, B, T, H, D, s, P(bsp),
                     P(btl), plan.n_sms, P(dq), P(dk), P(dv), P(ws), ws.numel(),
                     jfa._stream()) == 0, L.jfa_last_error()
    plan.check()


def test_mismatched_schedule_or_offsets_never_write_past_the_tensors():
    # The kernels skip tiles naming a sequence or head outside the call and
    # clamp every sequence to [0, T]. Outputs are views at the start of larger
    # buffers whose tails hold a sentinel: nothing may change it. Every access
    # stays inside allocated memory even if a guard were missing (the buffers
    # are as large as the larger batch), so no case here can fault.
    H, D = 2, 128
    big, small = [300, 129, 700, 64], [70, 200]
    Tb, Ts = sum(big), sum(small)
    off_big = torch.from_numpy(W.offsets_of(big)).cuda()
    off_small = torch.from_numpy(W.offsets_of(small)).cuda()
    plan_big = jfa.Plan(off_big, H, D)
    inp = W.jagged_inputs(small, H, D, 81, device="cuda")
    sentinel = 7.0

    def buffers():
        o = torch.full((Tb, H, D), sentinel, dtype=torch.bfloat16, device="cuda")
        lse = torch.full((H * Tb,), sentinel, dtype=torch.float32, device="cuda")
        g = [torch.full((Tb, H, D), sentinel, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
        return o, lse, g

    def untouched(o, lse, g):
        assert bool((o[Ts:] == sentinel).all()) and bool((lse[H * Ts:] == sentinel).all())
        for t in g:
            assert bool((t[Ts:] == sentinel).all())

    # (a) tile lists of a larger batch with the call's own offsets: tiles of
    # sequences 2 and 3 are skipped, and the ones the small batch needs are in
    # the list, so the results are also right.
    o, lse, g = buffers()
    _raw_fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], off_small, jfa.JFA_I64, 2, Ts, H, D,
                 plan_big, o, lse, *g)
    untouched(o, lse, g)
    s = 1 / math.sqrt(D)
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    offs = W.offsets_of(small)
    ref_o, ref_lse = A.jagged_fwd(q, k, v, offs, s)
    assert_close(o[:Ts], ref_o, "O", bf16_out=True)
    assert_lse(lse[:H * Ts].view(H, Ts), ref_lse)
    for name, got, r in zip(("dQ", "dK", "dV"), g, A.jagged_bwd(q, k, v, do, offs, s)):
        assert_close(got[:Ts], r, name, bf16_out=True)

    # (b) device offsets of the larger batch (ending past T) with the small
    # tensors: sequences are clamped to T, values are unspecified, but no row
    # at or past T is written and no kernel gives up.
    o, lse, g = buffers()
    _raw_fwd_bwd(inp["q"], inp["k"], inp["v"], inp["do"], off_big, jfa.JFA_I64, 4, Ts, H, D,
                 plan_big, o, lse, *g)
    untouched(o, lse, g)
