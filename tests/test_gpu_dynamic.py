"""GPU checks of the forward with device-side dynamic tile scheduling
(persistent CTAs claiming tiles from a global counter): the result does not
depend on which CTA computes a tile, so O and LSE must equal the statically
scheduled forward bit for bit, on both claim orders (device enumeration and
the host's longest-first list), and match the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from oracle import attention as A
from tests._util import assert_close, assert_lse, f64

pytestmark = pytest.mark.gpu

RAGGED = [1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 513, 0, 2048]


def _both_orders(lengths, H, D, seed, idx_dtype=np.int64):
    inp = W.jagged_inputs(lengths, H, D, seed, device="cuda", with_grad=False)
    off = torch.from_numpy(W.offsets_of(lengths, idx_dtype)).cuda()
    o_ref, l_ref = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off)
    out = {}
    for order in ("device", "lpt"):
        plan = jfa.DynamicPlan(off, H, D, order=order)
        o, lse = jfa.jfa_fwd_dynamic(inp["q"], inp["k"], inp["v"], off, plan=plan)
        plan.check()
        assert torch.equal(o, o_ref), "O differs from the static schedule (%s)" % order
        assert torch.equal(lse, l_ref), "LSE differs from the static schedule (%s)" % order
        out[order] = (o, lse)
    jfa.check_status()
    return inp, off, out


@pytest.mark.parametrize("D", [64, 128])
def test_dynamic_ragged_equals_static_and_oracle(D):
    inp, off, out = _both_orders(RAGGED, 2, D, 101, np.int32)
    o, lse = out["device"]
    ro, rl = A.jagged_fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), off.cpu().numpy(),
                          1 / math.sqrt(D))
    assert_close(o, ro, "O", bf16_out=True)
    assert_lse(lse, rl)


@pytest.mark.parametrize("name", ["gem", "stress"])
def test_dynamic_full_configs_equal_static(name):
    L = W.lengths_for(name)
    _both_orders(L, 4, 128, W.SEEDS[name])


def test_dynamic_more_ctas_than_tiles_and_empty_batch():
    _both_orders([5, 0, 300], 1, 128, 102)
    inp = W.jagged_inputs([0, 0], 2, 128, 103, device="cuda", with_grad=False)
    off = torch.from_numpy(W.offsets_of([0, 0])).cuda()
    o, lse = jfa.jfa_fwd_dynamic(inp["q"], inp["k"], inp["v"], off)
    jfa.check_status()
    assert o.shape[0] == 0 and lse.shape[1] == 0
