"""Host side of block-sparse attention (no GPU): the C scheduler's tiles,
lists and per-half step ranges against the scheduler oracle, the all-ones
mask against the unmasked varlen scheduler, and the argument checks of the
scheduler and of the block-sparse entry points."""

import ctypes
import os

import numpy as np
import pytest

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from oracle import sched as S

IDX = (1 << 29) - 1


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(jfa.LIB_PATH):
        from jagged_flash_attention_flashattention_gb300 import build

        build.build()
    return jfa.lib()


def _null():
    return ctypes.c_void_p(0)


def _masks(ql, kl, rng, p):
    return [rng.random((-(-int(a) // 128), -(-int(b) // 128))) < p for a, b in zip(ql, kl)]


def _decode_fwd(ent):
    return [(int(x) & IDX, bool(int(x) >> 29 & 1), bool(int(x) >> 30 & 1)) for x in ent]


@pytest.mark.parametrize("p", [0.0, 0.3, 0.7, 1.0])
@pytest.mark.parametrize("op", [jfa.OP_FWD, jfa.OP_BWD])
@pytest.mark.parametrize("dtype", [np.int32, np.int64])
def test_c_sparse_scheduler_matches_oracle(L, p, op, dtype):
    rng = np.random.default_rng(131)
    ql = rng.integers(0, 1200, 40)
    kl = np.where(rng.random(40) < 0.5, ql, rng.integers(0, 1200, 40))
    masks = _masks(ql, kl, rng, p)
    name = "fwd" if op == jfa.OP_FWD else "bwd"
    for zz in (True, False):
        sp, tl, lp, ent, meta = jfa.schedule_sparse(W.offsets_of(ql).astype(dtype),
                                                    W.offsets_of(kl).astype(dtype), 3, op, 11,
                                                    masks, zz)
        rp, rt, rl = S.schedule_sparse(list(ql), list(kl), 3, name, 11, masks, zz)
        assert sp.tolist() == rp
        assert [tuple(t) for t in tl.tolist()] == rt
        assert lp[0] == 0 and lp[-1] == sum(len(x) for x in rl)
        for i, want in enumerate(rl):
            got = ent[lp[i]:lp[i + 1]]
            if op == jfa.OP_FWD:
                got = _decode_fwd(got)
                # meta: first and one-past-last step that each half sees
                for x in range(2):
                    steps = [s for s, e in enumerate(got) if e[1 + x]]
                    exp = (steps[0], steps[-1] + 1) if steps else (0, 0)
                    assert tuple(meta[i, 2 * x:2 * x + 2]) == exp
            else:
                got = [int(v) for v in got]
                assert meta is None
            assert got == want


@pytest.mark.parametrize("op", [jfa.OP_FWD, jfa.OP_BWD])
def test_all_ones_mask_deals_like_the_unmasked_varlen_schedule(L, op):
    # Work of a tile under an all-ones mask is the whole key (query) range, the
    # unmasked varlen work, so the LPT deal is the same tile for tile.
    rng = np.random.default_rng(132)
    ql = rng.integers(0, 2000, 50)
    kl = rng.integers(1, 2000, 50)
    masks = _masks(ql, kl, rng, 2.0)
    qo, ko = W.offsets_of(ql), W.offsets_of(kl)
    sp, tl, lp, ent, _ = jfa.schedule_sparse(qo, ko, 2, op, 13, masks)
    vp, vt = jfa.schedule_varlen(qo, ko, 2, op, 13)
    assert sp.tolist() == vp.tolist() and tl.tolist() == vt.tolist()
    for i, (b, h, m) in enumerate(tl.tolist()):
        n = lp[i + 1] - lp[i]
        if op == jfa.OP_FWD:
            assert n == (-(-int(kl[b]) // 128) if 256 * m < ql[b] else 0)
        else:
            assert n == -(-int(ql[b]) // 64)


def test_sparse_scheduler_rejects_bad_arguments(L):
    qo = np.array([0, 300, 500], dtype=np.int64)
    ko = np.array([0, 200, 600], dtype=np.int64)
    need = 3 * 2 + 2 * 4
    n, ne = ctypes.c_int64(0), ctypes.c_int64(0)
    m = np.ones(need, dtype=np.uint8)
    assert L.jfa_sched_size_sparse(2, 2, jfa.OP_FWD, qo.ctypes.data, ko.ctypes.data, 1, m.ctypes.data,
                                   need, ctypes.byref(n), ctypes.byref(ne)) == 0
    # sequence 0: two forward tiles of 2 key blocks each; sequence 1: one tile of 4
    assert n.value == 2 * (2 + 1) and ne.value == 2 * (2 + 2 + 4)
    code = L.jfa_sched_size_sparse(2, 2, jfa.OP_FWD, qo.ctypes.data, ko.ctypes.data, 1,
                                   m.ctypes.data, need - 1, ctypes.byref(n), ctypes.byref(ne))
    assert code == 1 and b"masks hold" in L.jfa_last_error()
    assert L.jfa_sched_size_sparse(2, 2, jfa.OP_FWD, qo.ctypes.data, ko.ctypes.data, 1, _null(),
                                   need, ctypes.byref(n), ctypes.byref(ne)) == 1
    assert L.jfa_sched_size_sparse(2, 2, jfa.OP_BCASTQ_FWD, qo.ctypes.data, ko.ctypes.data, 1,
                                   m.ctypes.data, need, ctypes.byref(n), ctypes.byref(ne)) == 1
    sm = np.zeros(4, dtype=np.int32)
    tl = np.zeros(3 * 6, dtype=np.int32)
    lp = np.zeros(7, dtype=np.int32)
    ent = np.zeros(16, dtype=np.int32)
    assert L.jfa_sched_build_sparse(2, 2, jfa.OP_FWD, 3, qo.ctypes.data, ko.ctypes.data, 1,
                                    m.ctypes.data, need, 1, sm.ctypes.data, tl.ctypes.data,
                                    lp.ctypes.data, ent.ctypes.data, _null()) == 1  # no meta
    meta = np.zeros(4 * 6, dtype=np.int32)
    assert L.jfa_sched_build_sparse(2, 2, jfa.OP_FWD, 3, qo.ctypes.data, ko.ctypes.data, 1,
                                    m.ctypes.data, need, 1, sm.ctypes.data, tl.ctypes.data,
                                    lp.ctypes.data, ent.ctypes.data, meta.ctypes.data) == 0
    assert lp[-1] == 16


def test_pack_block_masks_checks_shapes():
    qo, ko = W.offsets_of([300, 0]), W.offsets_of([129, 50])
    ok = [np.ones((3, 2), bool), np.ones((0, 1), bool)]
    assert jfa.pack_block_masks(ok, qo, ko).tolist() == [1] * 6
    with pytest.raises(ValueError):
        jfa.pack_block_masks([np.ones((3, 1), bool), np.ones((0, 1), bool)], qo, ko)
    with pytest.raises(ValueError):
        jfa.pack_block_masks(ok[:1], qo, ko)
    with pytest.raises(ValueError):
        jfa.pack_block_masks(np.ones(5, np.uint8), qo, ko)


def test_sparse_entry_points_reject_missing_lists_on_host(L):
    dummy = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(dummy, ctypes.c_void_p)
    code = L.jfa_sparse_fwd(p, p, p, p, p, 0, 1, 10, 10, 2, 64, 0.1, p, p, p, p, _null(), 1, p, p, p,
                            256, _null())
    assert code == 1 and b"meta" in L.jfa_last_error()
    code = L.jfa_sparse_bwd(p, p, p, p, p, p, p, p, 0, 1, 10, 10, 2, 64, 0.1, p, p, _null(), p, 1, p,
                            p, p, p, 1 << 20, _null())
    assert code == 1 and b"list_ptr" in L.jfa_last_error()
