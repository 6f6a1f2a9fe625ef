"""jfa_bwd_noalloc: the jagged backward for callers that cannot allocate
device memory when they call (for example a plug-in inside a framework that
owns all device memory through its own pool, or a latency-critical path that
must not call cudaMalloc). Its scratch is a static 64 MiB device array
instead of a caller workspace.

Checked through the C ABI against jfa_bwd on the same inputs, twice in a row
(the array keeps the previous call's contents, so the second call shows that
everything that must start at zero is cleared). The file sorts last so that a
run stopping at the first failure has run every other test before it; it also
passes on its own in a fresh process.
"""

import ctypes

import pytest
import torch

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from tests._util import assert_close

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(inp, o, lse, off, plan, H, D):
    dq, dk, dv = (torch.empty_like(inp[n]) for n in ("q", "k", "v"))
    T = inp["q"].shape[0]
    sp, tl = plan.bwd_sched
    code = jfa.lib().jfa_bwd_noalloc(
        _p(inp["q"]), _p(inp["k"]), _p(inp["v"]), _p(o), _p(lse), _p(inp["do"]), _p(off),
        plan.idx, plan.B, T, H, D, ctypes.c_float(D ** -0.5), _p(sp), _p(tl), plan.n_sms,
        _p(dq), _p(dk), _p(dv), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, jfa.lib().jfa_last_error().decode()
    torch.cuda.synchronize()
    return dq, dk, dv


def test_noalloc_matches_jfa_bwd_twice():
    lengths = [300, 5, 700, 129, 64, 1]
    H, D = 2, 128
    inp = W.jagged_inputs(lengths, H, D, 61, device="cuda")
    off = torch.from_numpy(W.offsets_of(lengths)).cuda()
    plan = jfa.Plan(off, H, D)
    o, lse = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=plan)
    ref = jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], off, plan=plan)
    plan.check()
    for _ in range(2):
        got = _noalloc(inp, o, lse, off, plan, H, D)
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert_close(g, r, name + " (no-alloc vs jfa_bwd)")
    # No kernel of either call gave up waiting: the static status block says so.
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert jfa.lib().jfa_noalloc_check_status(stream) == 0, jfa.lib().jfa_last_error().decode()


def test_noalloc_rejects_oversized_problem():
    # T * H * D beyond the static buffer: refused on the host, nothing launched.
    T, H, D = 40000, 4, 128

    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    code = jfa.lib().jfa_bwd_noalloc(*([_p(dummy)] * 7), 1, 1, T, H, D, ctypes.c_float(0.1),
                                      _p(dummy), _p(dummy), 1, _p(dummy), _p(dummy), _p(dummy),
                                      ctypes.c_void_p(0))
    assert code == 3  # JFA_ERR_WORKSPACE
    assert "static buffer" in jfa.lib().jfa_last_error().decode()
