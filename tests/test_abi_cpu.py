"""CPU tests of the C ABI: the library loads, exports every symbol that
include/jfa.h declares, rejects bad arguments on the host without touching a
device, and its host scheduler matches the scheduler oracle exactly."""

import ctypes
import os
import re

import numpy as np
import pytest

import jagged_flash_attention_flashattention_gb300 as jfa
from jagged_flash_attention_flashattention_gb300 import workloads as W
from oracle import sched as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(jfa.LIB_PATH):
        from jagged_flash_attention_flashattention_gb300 import build

        build.build()
    return jfa.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "jfa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:jfa_status|size_t|const char \*)\s*\**\s*(\w+)\(", src,
                                 flags=re.M)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 16, names
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(jfa.EXPORTS)


def test_status_strings(L):
    assert L.jfa_status_str(0) == b"JFA_OK"
    assert L.jfa_status_str(5) == b"JFA_ERR_TIMEOUT"


def _null():
    return ctypes.c_void_p(0)


def test_fwd_rejects_unsupported_head_dim(L):
    dummy = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(dummy, ctypes.c_void_p)
    code = L.jfa_fwd(p, p, p, p, 0, 1, 10, 2, 96, 0.1, p, p, 1, p, p, p, 256, _null())
    assert code == 2 and b"D = 96" in L.jfa_last_error()


def test_fwd_rejects_missing_workspace(L):
    dummy = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(dummy, ctypes.c_void_p)
    assert L.jfa_fwd(p, p, p, p, 0, 1, 10, 2, 64, 0.1, p, p, 1, p, p, _null(), 256, _null()) == 3
    assert L.jfa_fwd(p, p, p, p, 0, 1, 10, 2, 64, 0.1, p, p, 1, p, p, p, 16, _null()) == 3


def test_fwd_rejects_bad_scale_and_index_type(L):
    dummy = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(dummy, ctypes.c_void_p)
    assert L.jfa_fwd(p, p, p, p, 0, 1, 10, 2, 64, -1.0, p, p, 1, p, p, p, 256, _null()) == 1
    assert L.jfa_fwd(p, p, p, p, 7, 1, 10, 2, 64, 0.1, p, p, 1, p, p, p, 256, _null()) == 1


def test_bwd_rejects_small_workspace(L):
    dummy = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(dummy, ctypes.c_void_p)
    need = L.jfa_workspace_size(jfa.OP_BWD, 1000, 2, 64)
    assert need == 256 + 1000 * 2 * 64 * 4
    code = L.jfa_bwd(p, p, p, p, p, p, p, 0, 1, 1000, 2, 64, 0.1, p, p, 1, p, p, p, p, need - 1,
                     _null())
    assert code == 3


def test_blockdiag_rejects_length_not_multiple_of_64(L):
    dummy = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(dummy, ctypes.c_void_p)
    assert L.blockdiag_fwd(p, p, p, 2, 100, 2, 64, 0.1, p, p, 256, _null()) == 1
    assert b"multiple of 64" in L.jfa_last_error()


def test_tile_rows(L):
    assert jfa.tile_rows(jfa.OP_FWD, 128) == 256
    assert jfa.tile_rows(jfa.OP_BWD, 64) == 128


def test_sched_rejects_bad_offsets(L):
    off = np.array([0, 5, 3], dtype=np.int64)
    with pytest.raises(jfa.JFAError):
        jfa.schedule(off, 2, 128, 4)
    off = np.array([1, 5], dtype=np.int64)
    with pytest.raises(jfa.JFAError):
        jfa.schedule(off, 2, 128, 4)


@pytest.mark.parametrize("name,tile_rows,sms", [("tiny", 256, 3), ("gem", 256, 152),
                                                ("gem", 128, 148), ("stress", 128, 152),
                                                ("stress", 256, 7)])
def test_c_scheduler_matches_oracle(L, name, tile_rows, sms):
    lengths = W.lengths_for(name)
    H = W.WORKLOADS[name]["H"]
    for zz in (True, False):
        sp, tl = jfa.schedule(W.offsets_of(lengths), H, tile_rows, sms, zigzag=zz)
        rp, rt = S.schedule(list(lengths), H, tile_rows, sms, zigzag=zz)
        assert sp.tolist() == rp
        assert [tuple(t) for t in tl.tolist()] == rt


def test_c_scheduler_matches_oracle_bcast(L):
    lengths = W.lengths_for("bcast")
    off = W.offsets_of(lengths)
    sp, tl = jfa.schedule(off, 4, 256, 152, fixed_rows=256)
    rp, rt = S.schedule(list(lengths), 4, 256, 152, fixed_rows=256)
    assert sp.tolist() == rp and [tuple(t) for t in tl.tolist()] == rt
    sp, tl = jfa.schedule(off, 4, 128, 152, fixed_work=256)
    rp, rt = S.schedule(list(lengths), 4, 128, 152, fixed_work=256)
    assert sp.tolist() == rp and [tuple(t) for t in tl.tolist()] == rt


def test_c_scheduler_matches_oracle_on_both_sort_paths(L):
    # The deal's stable sort by work is a counting sort while the works stay
    # below 2^20 tokens and a merge sort beyond; a batch with a few
    # sequences of millions of tokens takes the second path, and many equal
    # works check that ties keep their enumeration order on both.
    rng = np.random.default_rng(21)
    lengths = [int(x) for x in rng.integers(1, 3000, 200)] + [1 << 21, 3 << 20, 1 << 21, 700]
    lengths += [512] * 40
    for sms in (152, 13):
        for lens in (lengths, lengths[:200] + lengths[-41:]):
            sp, tl = jfa.schedule(W.offsets_of(lens), 2, 256, sms)
            rp, rt = S.schedule(list(lens), 2, 256, sms)
            assert sp.tolist() == rp
            assert [tuple(t) for t in tl.tolist()] == rt


def test_c_scheduler_int32_offsets_and_empty(L):
    off = np.array([0, 0, 3, 3, 200], dtype=np.int32)
    sp, tl = jfa.schedule(off, 2, 64, 5)
    rp, rt = S.schedule([0, 3, 0, 197], 2, 64, 5)
    assert sp.tolist() == rp and [tuple(t) for t in tl.tolist()] == rt
    sp, tl = jfa.schedule(np.array([0], dtype=np.int64), 2, 64, 5)
    assert sp.tolist() == [0] * 6 and tl.shape[0] == 0


def test_selftest_rejects_bad_arguments(L):
    # argument checks happen before any launch (no GPU needed)
    assert L.jfa_selftest_wait_timeout(None, 256, 1_000_000, None) == jfa.JFA_ERR_WORKSPACE
    fake = ctypes.c_void_p(0x1000)
    assert L.jfa_selftest_wait_timeout(fake, 64, 1_000_000, None) == jfa.JFA_ERR_WORKSPACE
    assert L.jfa_selftest_wait_timeout(fake, 256, 10, None) == jfa.JFA_ERR_INVALID_ARG
    assert L.jfa_selftest_wait_timeout(fake, 256, 5_000_000_000, None) == jfa.JFA_ERR_INVALID_ARG


def test_bcastq_rejects_batches_past_32_bit_row_indices(L):
    # B * Lq rows of O / dO are addressed with 32-bit row indices in the kernels:
    # refused on the host, nothing launched.
    dummy = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(dummy, ctypes.c_void_p)
    B, Lq = 1 << 20, 1 << 12
    assert L.jfa_bcastq_fwd(p, p, p, p, 0, B, Lq, 10, 2, 64, 0.1, p, p, 1, p, p, p, 256,
                            _null()) == 1
    assert b"B * Lq too large" in L.jfa_last_error()
    assert L.jfa_bcastq_bwd(p, p, p, p, p, p, p, 0, B, Lq, 10, 2, 64, 0.1, p, p, 1, p, p, p, p,
                            256, _null()) == 1
    assert b"B * Lq too large" in L.jfa_last_error()


def test_noalloc_rejects_oversized_problem_on_host(L):
    # Refused before any CUDA call, so this runs without a device too.
    dummy = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(dummy, ctypes.c_void_p)
    code = L.jfa_bwd_noalloc(p, p, p, p, p, p, p, 0, 1, 40000, 4, 128, 0.1, p, p, 1, p, p, p,
                             _null())
    assert code == 3 and b"static buffer" in L.jfa_last_error()


def test_noalloc_check_status_without_a_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    # No device: the address lookup fails cleanly, nothing crashes.
    assert L.jfa_noalloc_check_status(_null()) == 4


class _FakePlan(jfa.Plan):
    def __init__(self, kind, B, T, H, D, Lq=0):  # no device work: only the fields validate() reads
        self.kind, self.B, self.T, self.H, self.D, self.Lq = kind, B, T, H, D, Lq


class _Off:
    def __init__(self, n):
        self.n = n

    def numel(self):
        return self.n


def test_plan_validate_rejects_another_batch_layout():
    plan = _FakePlan("jagged", 3, 100, 2, 128)
    plan.validate("jagged", _Off(4), 100, 2, 128)
    for args in ((_Off(5), 100, 2, 128), (_Off(4), 99, 2, 128), (_Off(4), 100, 4, 128),
                 (_Off(4), 100, 2, 64)):
        with pytest.raises(ValueError):
            plan.validate("jagged", *args)
    with pytest.raises(ValueError):
        plan.validate("bcast", _Off(4), 100, 2, 128, 256)
    bplan = _FakePlan("bcast", 3, 100, 2, 128, Lq=256)
    bplan.validate("bcast", _Off(4), 100, 2, 128, 256)
    with pytest.raises(ValueError):
        bplan.validate("bcast", _Off(4), 100, 2, 128, 255)


def test_host_offsets_checks():
    jfa.check_host_offsets(np.array([0, 3, 3, 9], dtype=np.int64), 4)
    jfa.check_host_offsets(np.array([0], dtype=np.int32), 1)
    for bad, n in ((np.array([0, 3, 2]), 3), (np.array([1, 3]), 2), (np.array([0, 3]), 3),
                   (np.array([[0, 3]]), 2), (np.array([0.0, 3.0]), 2)):
        with pytest.raises(ValueError):
            jfa.check_host_offsets(bad, n)


@pytest.mark.parametrize("window", [(-1, -1), (-1, 0), (255, 0), (0, 0), (100, 300), (-1, 7),
                                    (513, -1)])
@pytest.mark.parametrize("op", [jfa.OP_FWD, jfa.OP_BWD])
def test_c_varlen_scheduler_matches_oracle(L, window, op):
    rng = np.random.default_rng(71)
    ql = rng.integers(0, 900, 60)
    kl = np.where(rng.random(60) < 0.5, ql, rng.integers(0, 900, 60))  # self and cross mixed
    for zz in (True, False):
        sp, tl = jfa.schedule_varlen(W.offsets_of(ql), W.offsets_of(kl), 3, op, 11, window, zz)
        rp, rt = S.schedule_varlen(list(ql), list(kl), 3, "fwd" if op == jfa.OP_FWD else "bwd",
                                   11, window, zz)
        assert sp.tolist() == rp
        assert [tuple(t) for t in tl.tolist()] == rt


def test_c_varlen_scheduler_rejects_bad_arguments(L):
    off = np.array([0, 5, 9], dtype=np.int64)
    sm = np.zeros(4, dtype=np.int32)
    tl = np.zeros(30, dtype=np.int32)
    assert L.jfa_sched_build_varlen(2, 1, jfa.OP_FWD, 3, off.ctypes.data, off.ctypes.data, 1, -2, 0,
                                    1, sm.ctypes.data, tl.ctypes.data) == 1
    assert L.jfa_sched_build_varlen(2, 1, jfa.OP_BCASTQ_FWD, 3, off.ctypes.data, off.ctypes.data,
                                    1, -1, -1, 1, sm.ctypes.data, tl.ctypes.data) == 1
    bad = np.array([0, 5, 4], dtype=np.int64)
    assert L.jfa_sched_build_varlen(2, 1, jfa.OP_BWD, 3, bad.ctypes.data, off.ctypes.data, 1, -1,
                                    -1, 1, sm.ctypes.data, tl.ctypes.data) == 1


def test_varlen_workspace_sizes(L):
    qo = np.array([0, 100, 100, 400], dtype=np.int64)
    ko = np.array([0, 300, 301, 302], dtype=np.int64)
    sz = ctypes.c_size_t(0)
    assert L.jfa_varlen_workspace_size(3, qo.ctypes.data, ko.ctypes.data, 1, 2, 64, 0,
                                       ctypes.byref(sz)) == 0
    assert sz.value == 256 + 400 * 2 * 64 * 4
    assert L.jfa_varlen_workspace_size(3, qo.ctypes.data, ko.ctypes.data, 1, 2, 64, 1,
                                       ctypes.byref(sz)) == 0
    # partial rows: ceil(300/128)*round_up(100,64) + 1*0 + 1*round_up(300,64) = 3*128 + 320
    header = 256 + ((2 * 4 * 8 + 255) // 256) * 256
    assert sz.value == header + (3 * 128 + 320) * 2 * 64 * 4


def test_varlen_entry_points_reject_bad_windows_on_host(L):
    dummy = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(dummy, ctypes.c_void_p)
    code = L.jfa_varlen_fwd(p, p, p, p, p, 0, 1, 10, 10, 2, 64, 0.1, -3, 0, p, p, 1, p, p, p, 256,
                            _null())
    assert code == 1 and b"window" in L.jfa_last_error()
    code = L.jfa_varlen_bwd(p, p, p, p, p, p, p, p, 0, 1, 10, 10, 2, 64, 0.1, 0, -5, 0, p, p, 1, p, p,
                            p, p, 1 << 20, _null())
    assert code == 1 and b"window" in L.jfa_last_error()


def test_fwd_dynamic_rejects_bad_arguments(L):
    dummy = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(dummy, ctypes.c_void_p)
    need = L.jfa_fwd_dynamic_workspace_size(10)
    assert need == 256 + 256
    # device enumeration needs the tile table in the workspace
    assert L.jfa_fwd_dynamic(p, p, p, p, 0, 10, 100, 2, 64, 0.1, _null(), 0, 4, p, p, p, 256,
                             _null()) == 3
    assert L.jfa_fwd_dynamic(p, p, p, p, 0, 10, 100, 2, 64, 0.1, p, -1, 4, p, p, p, need,
                             _null()) == 1
