"""GPU parity of the 64-token block-diagonal kernels against the fp64
oracle, plus the cross-check against the jagged kernels on 64-token
sequences."""

import math

import numpy as np
import pytest
import torch

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from oracle import attention as A
from tests._util import assert_close, f64

pytestmark = pytest.mark.gpu


def _run(B, L, H, D, seed):
    inp = W.blockdiag_inputs(B, L, H, D, seed, device="cuda")
    o = jfa.blockdiag_fwd(inp["q"], inp["k"], inp["v"])
    dq, dk, dv = jfa.blockdiag_bwd(inp["q"], inp["k"], inp["v"], inp["do"])
    jfa.check_status()
    return inp, o, (dq, dk, dv)


@pytest.mark.parametrize("B,L,D", [(3, 192, 128), (2, 256, 64), (3, 64, 128), (1, 64, 64)])
def test_blockdiag_small(B, L, D):
    H = 2
    inp, o, g = _run(B, L, H, D, 41)
    s = 1 / math.sqrt(D)
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    assert_close(o, A.blockdiag_fwd(q, k, v, s), "O", bf16_out=True)
    for name, a, b in zip(("dQ", "dK", "dV"), g, A.blockdiag_bwd(q, k, v, do, s)):
        assert_close(a, b, name, bf16_out=True)


def test_blockdiag_equals_jagged_64_token_sequences():
    B, L, H, D = 2, 320, 2, 128
    inp, o, g = _run(B, L, H, D, 42)
    flat = {n: t.reshape(B * L, H, D) for n, t in inp.items()}
    off = torch.arange(0, B * L + 1, 64, dtype=torch.int32, device="cuda")
    plan = jfa.Plan(off, H, D)
    oj, lse = jfa.jfa_fwd(flat["q"], flat["k"], flat["v"], off, plan=plan)
    gj = jfa.jfa_bwd(flat["q"], flat["k"], flat["v"], oj, lse, flat["do"], off, plan=plan)
    plan.check()
    assert_close(o.reshape(B * L, H, D), oj, "O vs jagged", atol=1e-2, rl2=5e-3)
    for name, a, b in zip(("dQ", "dK", "dV"), g, gj):
        assert_close(a.reshape(B * L, H, D), b, name + " vs jagged", atol=1e-2, rl2=5e-3)


@pytest.mark.parametrize("D", [128, 64])
def test_blockdiag_config_sampled(D):
    B, L, H = 1152, 4096, 2
    inp, o, g = _run(B, L, H, D, W.SEEDS["blockdiag"])
    s = 1 / math.sqrt(D)
    rng = np.random.default_rng(7)
    n_blocks = B * L // 64
    picks = np.sort(rng.choice(n_blocks, 48, replace=False))
    picks = np.unique(np.concatenate([picks, [0, n_blocks - 1]]))
    flat = {n: t.reshape(B * L, H, D) for n, t in inp.items()}
    outs = [o.reshape(B * L, H, D)] + [t.reshape(B * L, H, D) for t in g]
    for blk in picks:
        r0 = int(blk) * 64
        sl = slice(r0, r0 + 64)
        q, k, v, do = (f64(flat[n][sl]).reshape(1, 64, H, D) for n in ("q", "k", "v", "do"))
        ro = A.blockdiag_fwd(q, k, v, s)[0]
        rg = A.blockdiag_bwd(q, k, v, do, s)
        assert_close(outs[0][sl], ro, "O[block %d]" % blk)
        for name, a, b in zip(("dQ", "dK", "dV"), outs[1:], rg):
            assert_close(a[sl], b[0], "%s[block %d]" % (name, blk))


def _rotated_bf16(x, cos, sin):
    """x rotated by the oracle (fp64), rounded to bf16 like the rows the
    forward writes: an input of the rotary backward."""
    return torch.from_numpy(A.rope(f64(x), f64(cos), f64(sin))).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("B,L,D", [(3, 192, 128), (2, 256, 64), (1, 64, 128), (2, 4096, 128)])
def test_blockdiag_rotary_small(B, L, D):
    H = 2
    inp = W.blockdiag_inputs(B, L, H, D, 43, device="cuda")
    cos, sin = W.rotary_tables(L, D, device="cuda")
    o, q_rot, k_rot = jfa.blockdiag_rotary_fwd(inp["q"], inp["k"], inp["v"], cos, sin,
                                               return_rotated=True)
    o_only = jfa.blockdiag_rotary_fwd(inp["q"], inp["k"], inp["v"], cos, sin)
    qr, kr = _rotated_bf16(inp["q"], cos, sin), _rotated_bf16(inp["k"], cos, sin)
    g = jfa.blockdiag_rotary_bwd(qr, kr, inp["v"], inp["do"], cos, sin)
    jfa.check_status()
    s = 1 / math.sqrt(D)
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    c, sn = f64(cos), f64(sin)
    assert torch.equal(o, o_only)
    assert_close(o, A.blockdiag_rotary_fwd(q, k, v, c, sn, s), "O", bf16_out=True)
    assert_close(q_rot, A.rope(q, c, sn), "q_rot", bf16_out=True)
    assert_close(k_rot, A.rope(k, c, sn), "k_rot", bf16_out=True)
    ref = A.blockdiag_rotary_bwd_from_rotated(f64(qr), f64(kr), v, do, c, sn, s)
    for name, a, b in zip(("dQ", "dK", "dV"), g, ref):
        assert_close(a, b, name, bf16_out=True)


@pytest.mark.parametrize("D", [128, 64])
def test_blockdiag_rotary_zero_angles_equal_plain(D):
    # cos = 1, sin = 0 leaves q and k unchanged: bit-identical to the plain kernels
    B, L, H = 2, 320, 2
    inp = W.blockdiag_inputs(B, L, H, D, 44, device="cuda")
    cos = torch.ones(L, D // 2, dtype=torch.float32, device="cuda")
    sin = torch.zeros_like(cos)
    o, q_rot, k_rot = jfa.blockdiag_rotary_fwd(inp["q"], inp["k"], inp["v"], cos, sin,
                                               return_rotated=True)
    g = jfa.blockdiag_rotary_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cos, sin)
    o2 = jfa.blockdiag_fwd(inp["q"], inp["k"], inp["v"])
    g2 = jfa.blockdiag_bwd(inp["q"], inp["k"], inp["v"], inp["do"])
    jfa.check_status()
    assert torch.equal(o, o2)
    assert torch.equal(q_rot, inp["q"]) and torch.equal(k_rot, inp["k"])
    for a, b in zip(g, g2):
        assert torch.equal(a, b)


def test_blockdiag_rotary_config_sampled():
    # The full rotary configuration: the forward (with the rotated rows
    # written) and the backward, checked on sampled 64-token blocks. The
    # backward's rotated inputs are the seeded q and k themselves (any bf16
    # values are valid rotated rows).
    B, L, H, D = 1152, 4096, 2, 128
    inp = W.blockdiag_inputs(B, L, H, D, W.SEEDS["blockdiag_rotary"], device="cuda")
    cos, sin = W.rotary_tables(L, D, device="cuda")
    o, q_rot, k_rot = jfa.blockdiag_rotary_fwd(inp["q"], inp["k"], inp["v"], cos, sin,
                                               return_rotated=True)
    # without the rotated rows the fused forward runs: the same O bit for bit
    assert torch.equal(o, jfa.blockdiag_rotary_fwd(inp["q"], inp["k"], inp["v"], cos, sin))
    g = jfa.blockdiag_rotary_bwd(inp["q"], inp["k"], inp["v"], inp["do"], cos, sin)
    jfa.check_status()
    s = 1 / math.sqrt(D)
    c, sn = f64(cos), f64(sin)
    rng = np.random.default_rng(8)
    n_blocks = B * L // 64
    picks = np.unique(np.concatenate([rng.choice(n_blocks, 32, replace=False), [0, n_blocks - 1]]))
    flat = {n: t.reshape(B * L, H, D) for n, t in inp.items()}
    outs = [t.reshape(B * L, H, D) for t in (o, q_rot, k_rot) + tuple(g)]
    for blk in picks:
        r0 = int(blk) * 64
        pos0 = r0 % L
        sl = slice(r0, r0 + 64)
        q, k, v, do = (f64(flat[n][sl]).reshape(1, 64, H, D) for n in ("q", "k", "v", "do"))
        cb, sb = c[pos0:pos0 + 64], sn[pos0:pos0 + 64]
        assert_close(outs[0][sl], A.blockdiag_rotary_fwd(q, k, v, cb, sb, s)[0], "O[block %d]" % blk)
        assert_close(outs[1][sl], A.rope(q, cb, sb)[0], "q_rot[block %d]" % blk, bf16_out=True)
        assert_close(outs[2][sl], A.rope(k, cb, sb)[0], "k_rot[block %d]" % blk, bf16_out=True)
        rg = A.blockdiag_rotary_bwd_from_rotated(q, k, v, do, cb, sb, s)
        for name, a, b in zip(("dQ", "dK", "dV"), outs[3:], rg):
            assert_close(a[sl], b[0], "%s[block %d]" % (name, blk))
