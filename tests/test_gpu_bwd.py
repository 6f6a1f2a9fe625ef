"""GPU parity of the backward kernels (jagged and broadcast-Q) against the
fp64 oracle. The GPU backward consumes the GPU forward's O and LSE; the
oracle recomputes everything from Q, K, V, dO in fp64."""

import math

import numpy as np
import pytest
import torch

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from oracle import attention as A
from tests._util import assert_close, f64

pytestmark = pytest.mark.gpu

RAGGED = [1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 513]


def _run_jagged(lengths, H, D, seed, idx_dtype=np.int64):
    inp = W.jagged_inputs(lengths, H, D, seed, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths, idx_dtype)).cuda()
    plan = jfa.Plan(off, H, D)
    o, lse = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan)
    dq, dk, dv = jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, plan=plan)
    plan.check()
    return inp, off, (dq, dk, dv)


def _check_full(lengths, H, D, seed, idx_dtype=np.int64, bf16_out=True):
    inp, off, got = _run_jagged(lengths, H, D, seed, idx_dtype)
    ref = A.jagged_bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["do"]),
                       off.cpu().numpy(), 1 / math.sqrt(D))
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert_close(g, r, name, bf16_out=bf16_out)


def test_bwd_tiny_config():
    _check_full(W.lengths_for("tiny"), 2, 64, W.SEEDS["tiny"], np.int32, bf16_out=False)


@pytest.mark.parametrize("D", [64, 128])
def test_bwd_ragged_edges(D):
    _check_full(RAGGED, 2, D, 17)


def test_bwd_single_tokens_and_long():
    _check_full([1, 1, 2048, 3], 1, 128, 18)


def test_bwd_repeatable_within_tolerance():
    lengths = [300, 5, 700]
    inp, off, a = _run_jagged(lengths, 2, 128, 19)
    _, _, b = _run_jagged(lengths, 2, 128, 19)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])  # dK, dV: fixed order
    assert_close(a[0], b[0], "dQ rerun", atol=1e-2, rl2=1e-3)   # dQ: reduction order varies


def _sampled(name, picks, rows_cap=None):
    L = W.lengths_for(name)
    cfg = W.WORKLOADS[name]
    H, D = cfg["H"], cfg["D"]
    inp, off, got = _run_jagged(L, H, D, W.SEEDS[name])
    offs = W.offsets_of(L)
    s = 1 / math.sqrt(D)
    for b in picks(L):
        a, e = int(offs[b]), int(offs[b + 1])
        for h in range(H):  # every head of each picked sequence
            ref = A.seq_bwd(f64(inp["q"][a:e, h]), f64(inp["k"][a:e, h]), f64(inp["v"][a:e, h]),
                            f64(inp["do"][a:e, h]), s)
            for name_, g, r in zip(("dQ", "dK", "dV"), got, ref):
                assert_close(g[a:e, h], r, "%s[b=%d,h=%d]" % (name_, b, h))


def test_bwd_gem_config_sampled():
    def picks(L):
        rng = np.random.default_rng(5)
        return sorted(set(rng.choice(len(L), 8, replace=False).tolist())
                      | {int(np.argmax(L)), int(np.argmin(L))})
    _sampled("gem", picks)


def test_bwd_stress_config_sampled():
    def picks(L):
        long_ = int(np.flatnonzero(L == 16384)[0])
        short = np.flatnonzero(L < 256)[:3].tolist()
        return [long_] + short
    _sampled("stress", picks)


@pytest.mark.parametrize("Lq,D", [(256, 128), (100, 128), (300, 64)])
def test_bcastq_bwd_small(Lq, D):
    lengths = [64, 1, 0, 130, 1024, 257]
    H = 2
    inp = W.bcast_inputs(lengths, Lq, H, D, 31, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths)).cuda()
    plan = jfa.Plan(off, H, D, kind="bcast", Lq=Lq)
    o, lse = jfa.jfa_bcastq_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan)
    dq, dk, dv = jfa.jfa_bcastq_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, plan=plan)
    plan.check()
    ref = A.bcastq_bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["do"]),
                       off.cpu().numpy(), 1 / math.sqrt(D))
    assert_close(dq, ref[0], "dQ (fp32, summed)")  # fp32 output: no bf16 rounding slack
    assert_close(dk, ref[1], "dK", bf16_out=True)
    assert_close(dv, ref[2], "dV", bf16_out=True)


def test_bcastq_bwd_config_sampled():
    L = W.lengths_for("bcast")
    H, D, Lq = 4, 128, 256
    inp = W.bcast_inputs(L, Lq, H, D, W.SEEDS["bcast"], device="cuda")
    off = torch.from_numpy(W.offsets_of(L)).cuda()
    plan = jfa.Plan(off, H, D, kind="bcast", Lq=Lq)
    o, lse = jfa.jfa_bcastq_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan)
    dq, dk, dv = jfa.jfa_bcastq_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, plan=plan)
    plan.check()
    offs = W.offsets_of(L)
    s = 1 / math.sqrt(D)
    q, k, v, do = f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["do"])
    for h in range(H):  # dQ of a head is a sum over every sequence
        dq_ref = np.zeros((Lq, D))
        for b in range(len(L)):
            a, e = int(offs[b]), int(offs[b + 1])
            rq, rk, rv = A.seq_bwd(q[:, h], k[a:e, h], v[a:e, h], do[b, :, h], s)
            dq_ref += rq
            if b in (0, 3, 200, 511):
                assert_close(dk[a:e, h], rk, "dK[b=%d,h=%d]" % (b, h))
                assert_close(dv[a:e, h], rv, "dV[b=%d,h=%d]" % (b, h))
        assert_close(dq[:, h], dq_ref, "dQ[h=%d] (sum over 512 sequences)" % h)
