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
