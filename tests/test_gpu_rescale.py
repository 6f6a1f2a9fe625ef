"""GPU parity of the forward's online-softmax correction, the step that
rescales the running output when a row's maximum grows ("TLX Block
Attention", section 2: alpha = exp(m_old - m_new), O = alpha O + ...).

The forward raises a row's running maximum, and rescales that row's O in
tensor memory, only when a K/V tile's maximum exceeds it by more than 8 in
log2 units. With N(0, 1) inputs at scale 1/sqrt(D) a row's maximum never
grows that much after its first 128 keys, so these tests build inputs that
make it grow: keys past the first 128 of each sequence are multiplied by 4,
and query rows by 1, 2 or 1/8 in turn (all powers of two, so the bf16
inputs stay exact). Rows scaled by 1 or 2 cross the threshold, rows scaled by
1/8 do not, so every 32-row warp holds both kinds and the warp-wide "any row
rescaled" branch runs with a mix of rescaled and untouched rows.

Each test first checks, from fp64 scores of the same inputs and the
kernel's threshold rule, that the inputs really do cross the threshold
(many rows, and mixed warps), so the test cannot silently stop covering the
branch; then it compares O, LSE and the backward's dQ, dK, dV (computed from
that O and LSE) with the fp64 oracle.

The enlarged keys make the gradients about ten times larger than with the
workload configurations' N(0, 1) inputs (max |dQ| 13.6 against 1.4), and the
fixed absolute tolerance is set for the latter. The backward is linear in dO,
so dO is scaled by 1/8 (exact in bf16), which brings the gradients back to
the configurations' magnitudes without changing anything the test covers.
"""

import math

import numpy as np
import pytest
import torch

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from oracle import attention as A
from tests._util import assert_close, assert_lse, f64

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634
THRESHOLD = 8.0  # log2 units: the forward's lazy-rescale rule
Q_FACTORS = (1.0, 2.0, 0.125)


def _scale_rows(t, factors):
    return (t.float() * factors.to(t.device)[:, None, None]).to(torch.bfloat16)


def _k_factors(lengths):
    f = []
    for L in lengths:
        f.extend([1.0] * min(L, 128) + [4.0] * max(0, L - 128))
    return torch.tensor(f, dtype=torch.float32)


def _q_factors(n):
    return torch.tensor([Q_FACTORS[i % 3] for i in range(n)], dtype=torch.float32)


def _rescale_rows(Q, K, scale):
    """Per query row: True where the kernel's rule rescales at least once
    (with a 0.25 margin both ways; None in the band around the threshold).
    Rows are taken in 128-key tiles in order, as the forward walks them."""
    S = (Q @ K.T) * (scale * LOG2E)
    n_kv = (K.shape[0] + 127) // 128
    m_run = S[:, :128].max(axis=1)
    fired = np.zeros(Q.shape[0], dtype=bool)
    near = np.zeros(Q.shape[0], dtype=bool)
    for j in range(1, n_kv):
        m_tile = S[:, j * 128:(j + 1) * 128].max(axis=1)
        d = m_tile - (m_run + THRESHOLD)
        near |= np.abs(d) < 0.25
        up = d > 0
        fired |= up
        m_run = np.where(up, m_tile, m_run)
    return np.where(near, None, fired)


def _assert_branch_covered(rows_per_group):
    """rows_per_group: list of arrays (each a 32-row warp's rows, True/False/None)."""
    n_fired = sum(int(np.sum(g == True)) for g in rows_per_group)  # noqa: E712
    n_total = sum(len(g) for g in rows_per_group)
    mixed = sum(1 for g in rows_per_group if np.any(g == True) and np.any(g == False))  # noqa: E712
    assert n_fired >= n_total // 4, "only %d of %d rows cross the rescale threshold" % (n_fired, n_total)
    assert mixed >= 4, "only %d warps mix rescaled and untouched rows" % mixed


@pytest.mark.parametrize("D", [64, 128])
def test_jagged_rescale_fwd_and_bwd(D):
    lengths = [129, 300, 2048, 40]
    H = 2
    s = 1 / math.sqrt(D)
    inp = W.jagged_inputs(lengths, H, D, 71, device="cuda")
    T = int(sum(lengths))
    inp["k"] = _scale_rows(inp["k"], _k_factors(lengths))
    inp["q"] = _scale_rows(inp["q"], _q_factors(T))
    inp["do"] = _scale_rows(inp["do"], torch.full((T,), 0.125))
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    offs = W.offsets_of(lengths)

    groups = []
    for b in range(len(lengths)):
        a, e = int(offs[b]), int(offs[b + 1])
        if e - a <= 128:
            continue
        for h in range(H):
            fired = _rescale_rows(q[a:e, h], k[a:e, h], s)
            groups += [fired[i:i + 32] for i in range(0, e - a, 32)]
    _assert_branch_covered(groups)

    off = torch.from_numpy(offs).cuda()
    plan = jfa.Plan(off, H, D)
    o, lse = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan)
    dq, dk, dv = jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, plan=plan)
    plan.check()
    ref_o, ref_lse = A.jagged_fwd(q, k, v, offs, s)
    assert_close(o, ref_o, "O", bf16_out=True)
    assert_lse(lse, ref_lse)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), A.jagged_bwd(q, k, v, do, offs, s)):
        assert_close(g, r, name, bf16_out=True)


def test_bcastq_rescale_fwd_and_bwd():
    lengths = [300, 129, 700, 64]
    Lq, H, D = 256, 2, 128
    s = 1 / math.sqrt(D)
    inp = W.bcast_inputs(lengths, Lq, H, D, 72, device="cuda")
    inp["k"] = _scale_rows(inp["k"], _k_factors(lengths))
    inp["q"] = _scale_rows(inp["q"], _q_factors(Lq))
    inp["do"] = (inp["do"].float() * 0.125).to(torch.bfloat16)
    q, k, v, do = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    offs = W.offsets_of(lengths)

    groups = []
    for b in range(len(lengths)):
        a, e = int(offs[b]), int(offs[b + 1])
        if e - a <= 128:
            continue
        for h in range(H):
            fired = _rescale_rows(q[:, h], k[a:e, h], s)
            groups += [fired[i:i + 32] for i in range(0, Lq, 32)]
    _assert_branch_covered(groups)

    off = torch.from_numpy(offs).cuda()
    plan = jfa.Plan(off, H, D, kind="bcast", Lq=Lq)
    o, lse = jfa.jfa_bcastq_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan)
    dq, dk, dv = jfa.jfa_bcastq_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, plan=plan)
    plan.check()
    ref_o, ref_lse = A.bcastq_fwd(q, k, v, offs, s)
    assert_close(o, ref_o, "O", bf16_out=True)
    assert_lse(lse, ref_lse)
    rq, rk, rv = A.bcastq_bwd(q, k, v, do, offs, s)
    assert_close(dq, rq, "dQ (fp32, summed)")
    assert_close(dk, rk, "dK", bf16_out=True)
    assert_close(dv, rv, "dV", bf16_out=True)
