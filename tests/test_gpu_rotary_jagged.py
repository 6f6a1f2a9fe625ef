"""GPU parity of the jagged rotary path against the fp64 oracle, through the
C ABI: jfa_rope (each packed row rotated at its position in its sequence)
and jfa_rotary_bwd (the jagged backward taken from the rotated q and k, with
dQ and dK rotated back in the backward's closing cast pass).

The backward's rotated inputs are the oracle's own rotation of the seeded q
and k, rounded to bf16 by the test; the forward that supplies O and LSE runs
on those same rows."""

import math

import numpy as np
import pytest
import torch

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from oracle import attention as A
from tests._util import assert_close, f64

pytestmark = pytest.mark.gpu

RAGGED = [1, 63, 64, 65, 127, 128, 129, 255, 256, 0, 257, 300, 513]


def _rotated_bf16(x, offs, cos, sin):
    return torch.from_numpy(A.jagged_rope(f64(x), offs, f64(cos), f64(sin))).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("D", [64, 128])
def test_rope_rows_match_oracle(D):
    H = 2
    inp = W.jagged_inputs(RAGGED, H, D, 111, device="cuda", with_grad=False)
    off = torch.from_numpy(W.offsets_of(RAGGED)).cuda()
    cos, sin = W.rotary_tables(max(RAGGED), D, device="cuda")
    plan = jfa.Plan(off, H, D)
    q_rot = jfa.jfa_rope(inp["q"], off, cos, sin, plan=plan)
    ref = A.jagged_rope(f64(inp["q"]), W.offsets_of(RAGGED), f64(cos), f64(sin))
    assert_close(q_rot, ref, "q_rot", bf16_out=True)


@pytest.mark.parametrize("D", [64, 128])
def test_rotary_backward_matches_oracle(D):
    H = 2
    offs = W.offsets_of(RAGGED)
    inp = W.jagged_inputs(RAGGED, H, D, 112, device="cuda")
    off = torch.from_numpy(offs).cuda()
    cos, sin = W.rotary_tables(max(RAGGED), D, device="cuda")
    qr, kr = _rotated_bf16(inp["q"], offs, cos, sin), _rotated_bf16(inp["k"], offs, cos, sin)
    plan = jfa.Plan(off, H, D)
    o, lse = jfa.jfa_fwd(qr, kr, inp["v"], off, plan=plan)
    g = jfa.jfa_rotary_bwd(qr, kr, inp["v"], o, lse, inp["do"], off, cos, sin, plan=plan)
    plan.check()
    ref = A.jagged_rotary_bwd_from_rotated(f64(qr), f64(kr), f64(inp["v"]), f64(inp["do"]), offs,
                                           f64(cos), f64(sin), 1 / math.sqrt(D))
    for name, a, b in zip(("dQ", "dK", "dV"), g, ref):
        assert_close(a, b, name, bf16_out=True)


@pytest.mark.parametrize("D", [64, 128])
def test_rotary_zero_angles_equal_plain(D):
    # cos = 1, sin = 0: rope is the identity and the rotary backward is jfa_bwd, bit for bit
    H, lengths = 2, [300, 5, 700]
    inp = W.jagged_inputs(lengths, H, D, 113, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths)).cuda()
    cos = torch.ones(max(lengths), D // 2, dtype=torch.float32, device="cuda")
    sin = torch.zeros_like(cos)
    plan = jfa.Plan(off, H, D)
    assert torch.equal(jfa.jfa_rope(inp["q"], off, cos, sin, plan=plan), inp["q"])
    o, lse = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan)
    g1 = jfa.jfa_rotary_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, cos, sin, plan=plan)
    g0 = jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, plan=plan)
    plan.check()
    assert torch.equal(g1[1], g0[1]) and torch.equal(g1[2], g0[2])
    assert_close(g1[0], g0[0], "dQ (reduction order)", atol=1e-2, rl2=1e-3)


def test_rotary_tables_shorter_than_a_sequence_are_refused():
    H, D, lengths = 2, 64, [10, 70]
    inp = W.jagged_inputs(lengths, H, D, 114, device="cuda", with_grad=False)
    off = torch.from_numpy(W.offsets_of(lengths)).cuda()
    cos, sin = W.rotary_tables(64, D, device="cuda")
    with pytest.raises(ValueError):
        jfa.jfa_rope(inp["q"], off, cos, sin)


def test_gem_rotary_sampled():
    # The GEM batch: rotary layer (jfa_rope on q and k), forward, rotary
    # backward; sampled sequences (every head) against the oracle's rotation
    # of the same bf16 q and k.
    L = W.lengths_for("gem")
    H, D = 4, 128
    offs = W.offsets_of(L)
    inp = W.jagged_inputs(L, H, D, W.SEEDS["gem"], device="cuda")
    off = torch.from_numpy(offs).cuda()
    cos, sin = W.rotary_tables(int(max(L)), D, device="cuda")
    plan = jfa.Plan(off, H, D)
    qr = jfa.jfa_rope(inp["q"], off, cos, sin, plan=plan)
    kr = jfa.jfa_rope(inp["k"], off, cos, sin, plan=plan)
    o, lse = jfa.jfa_fwd(qr, kr, inp["v"], off, plan=plan)
    g = jfa.jfa_rotary_bwd(qr, kr, inp["v"], o, lse, inp["do"], off, cos, sin, plan=plan)
    plan.check()
    rng = np.random.default_rng(115)
    pick = sorted(set(rng.choice(len(L), 5, replace=False).tolist()) | {int(np.argmax(L))})
    c, s = f64(cos), f64(sin)
    sc = 1 / math.sqrt(D)
    for b in pick:
        a, e = int(offs[b]), int(offs[b + 1])
        sub = np.array([0, e - a])
        q, k, v, do = (f64(inp[n][a:e]) for n in ("q", "k", "v", "do"))
        ref_o, _ = A.jagged_rotary_fwd(q, k, v, sub, c, s, sc)
        assert_close(o[a:e], ref_o, "O[b=%d]" % b)
        ref = A.jagged_rotary_bwd_from_rotated(A.jagged_rope(q, sub, c, s), A.jagged_rope(k, sub, c, s),
                                               v, do, sub, c, s, sc)
        for name, got, r in zip(("dQ", "dK", "dV"), g, ref):
            assert_close(got[a:e], r, "%s[b=%d]" % (name, b))
