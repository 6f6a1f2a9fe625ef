"""GPU parity of the forward kernels (jagged and broadcast-Q) against the
fp64 oracle, through the C ABI (via the thin binding)."""

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


def _jagged(lengths, H, D, seed, idx_dtype=np.int64):
    inp = W.jagged_inputs(lengths, H, D, seed, device="cuda", with_grad=False)
    off = torch.from_numpy(W.offsets_of(lengths, idx_dtype)).cuda()
    return inp, off


def _check_fwd_full(lengths, H, D, seed, idx_dtype=np.int64, bf16_out=True):
    inp, off = _jagged(lengths, H, D, seed, idx_dtype)
    o, lse = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off)
    jfa.check_status()
    ref_o, ref_lse = A.jagged_fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]),
                                  off.cpu().numpy(), 1 / math.sqrt(D))
    assert_close(o, ref_o, "O", bf16_out=bf16_out)
    assert_lse(lse, ref_lse)


def test_fwd_tiny_config():
    L = W.lengths_for("tiny")
    _check_fwd_full(L, 2, 64, W.SEEDS["tiny"], np.int32, bf16_out=False)


@pytest.mark.parametrize("D", [64, 128])
def test_fwd_ragged_edges(D):
    _check_fwd_full(RAGGED, 2, D, 7)


def test_fwd_single_token_and_long():
    _check_fwd_full([1, 1, 2048, 3], 1, 128, 8)


def test_fwd_naive_schedule_same_result():
    lengths = [300, 5, 700, 129]
    inp, off = _jagged(lengths, 2, 128, 9)
    o1, l1 = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off)
    plan = jfa.Plan(off, 2, 128, zigzag=False)
    o2, l2 = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan)
    jfa.check_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def _sampled_check(name, n_seq=10, rows_cap=None):
    L = W.lengths_for(name)
    cfg = W.WORKLOADS[name]
    H, D = cfg["H"], cfg["D"]
    inp, off = _jagged(L, H, D, W.SEEDS[name])
    o, lse = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off)
    jfa.check_status()
    offs = W.offsets_of(L)
    rng = np.random.default_rng(123)
    pick = set(rng.choice(len(L), n_seq, replace=False).tolist())
    pick |= {int(np.argmax(L)), int(np.argmin(L))}
    s = 1 / math.sqrt(D)
    for b in sorted(pick):
        a, e = int(offs[b]), int(offs[b + 1])
        rows = np.arange(e - a)
        if rows_cap and rows.size > rows_cap:
            rows = np.sort(rng.choice(rows.size, rows_cap, replace=False))
        for h in range(H):  # every head of each picked sequence
            Q = f64(inp["q"][a:e, h])[rows]
            K, V = f64(inp["k"][a:e, h]), f64(inp["v"][a:e, h])
            ro, rl = A.seq_fwd(Q, K, V, s)
            assert_close(o[a:e, h][rows], ro, "O[b=%d,h=%d]" % (b, h))
            assert_lse(lse[h, a:e][rows], rl, "LSE[b=%d,h=%d]" % (b, h))


def test_fwd_gem_config_sampled():
    _sampled_check("gem")


def test_fwd_stress_config_sampled():
    _sampled_check("stress", n_seq=6, rows_cap=2048)


@pytest.mark.parametrize("Lq,D", [(256, 128), (100, 128), (300, 64)])
def test_bcastq_fwd_small(Lq, D):
    lengths = [64, 1, 0, 130, 1024, 257]
    H = 2
    inp = W.bcast_inputs(lengths, Lq, H, D, 21, device="cuda", with_grad=False)
    off = torch.from_numpy(W.offsets_of(lengths)).cuda()
    o, lse = jfa.jfa_bcastq_fwd(inp["q"], inp["k"], inp["v"], off)
    jfa.check_status()
    ro, rl = A.bcastq_fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), off.cpu().numpy(),
                          1 / math.sqrt(D))
    assert_close(o, ro, "O", bf16_out=True)
    assert_lse(lse, rl)


def test_bcastq_fwd_config_sampled():
    L = W.lengths_for("bcast")
    H, D, Lq = 4, 128, 256
    inp = W.bcast_inputs(L, Lq, H, D, W.SEEDS["bcast"], device="cuda", with_grad=False)
    off = torch.from_numpy(W.offsets_of(L)).cuda()
    o, lse = jfa.jfa_bcastq_fwd(inp["q"], inp["k"], inp["v"], off)
    jfa.check_status()
    offs = W.offsets_of(L)
    q = f64(inp["q"])
    for b in (0, 1, 77, 300, 511):
        a, e = int(offs[b]), int(offs[b + 1])
        for h in range(H):
            ro, rl = A.seq_fwd(q[:, h], f64(inp["k"][a:e, h]), f64(inp["v"][a:e, h]),
                               1 / math.sqrt(D))
            assert_close(o[b, :, h], ro, "O[b=%d,h=%d]" % (b, h))
            assert_lse(lse[b, h], rl)
