"""Jagged Flash Attention for GB300 (sm_103a): thin Python binding of libjfa.

Every step of the attention runs in libjfa's CUDA kernels behind the C ABI
declared in ``include/jfa.h``; this module only marshals arguments: it
allocates outputs and workspaces with torch, calls the host scheduler,
copies its tile lists to the device and passes raw pointers and the current
CUDA stream. There is no fallback: if ``libjfa.so`` is missing or the
tensors are not CUDA tensors, the calls raise.

Functions mirror the C entry points:

* :func:`jfa_fwd`, :func:`jfa_bwd` -- jagged self-attention over packed
  ``[T, H, D]`` bf16 tensors and an offsets tensor ``[B+1]``;
* :func:`jfa_bcastq_fwd`, :func:`jfa_bcastq_bwd` -- one dense Q
  ``[Lq, H, D]`` shared by every jagged K/V sequence;
* :func:`jfa_varlen_fwd`, :func:`jfa_varlen_bwd` -- separate query and
  key/value offsets (jagged cross attention), an optional band mask
  (causal, sliding window) and an optional deterministic dQ reduction;
* :func:`jfa_sparse_fwd`, :func:`jfa_sparse_bwd` -- block-sparse masks of
  128 x 128 blocks per sequence, with separate query and key/value offsets;
* :func:`blockdiag_fwd`, :func:`blockdiag_bwd` -- 64-token block-diagonal
  attention on ``[B, L, H, D]``;
* :func:`schedule` -- the host LPT + zigzag tile scheduler.
"""

import ctypes
import math
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libjfa.so")

JFA_I32, JFA_I64 = 0, 1
OP_FWD, OP_BWD, OP_BCASTQ_FWD, OP_BCASTQ_BWD, OP_BLOCKDIAG_FWD, OP_BLOCKDIAG_BWD, OP_FWD_PAIR = range(7)

(JFA_OK, JFA_ERR_INVALID_ARG, JFA_ERR_UNSUPPORTED, JFA_ERR_WORKSPACE, JFA_ERR_CUDA,
 JFA_ERR_TIMEOUT) = range(6)
_STATUS = {0: "JFA_OK", 1: "JFA_ERR_INVALID_ARG", 2: "JFA_ERR_UNSUPPORTED",
           3: "JFA_ERR_WORKSPACE", 4: "JFA_ERR_CUDA", 5: "JFA_ERR_TIMEOUT"}

EXPORTS = [
    "jfa_status_str", "jfa_last_error", "jfa_sched_size", "jfa_sched_build", "jfa_tile_rows",
    "jfa_num_sms", "jfa_workspace_size", "jfa_workspace_init", "jfa_check_status", "jfa_fwd",
    "jfa_bwd", "jfa_bcastq_fwd", "jfa_bcastq_bwd", "blockdiag_fwd", "blockdiag_bwd",
    "jfa_bwd_noalloc", "jfa_noalloc_check_status", "jfa_selftest_wait_timeout",
    "jfa_fwd_pair", "jfa_num_pairs", "jfa_rope", "jfa_rotary_bwd",
    "jfa_sched_size_varlen", "jfa_sched_build_varlen", "jfa_varlen_fwd", "jfa_varlen_bwd",
    "jfa_varlen_workspace_size", "jfa_fwd_dynamic", "jfa_fwd_dynamic_workspace_size",
    "blockdiag_rotary_fwd", "blockdiag_rotary_bwd",
    "jfa_sched_size_sparse", "jfa_sched_build_sparse", "jfa_sparse_fwd", "jfa_sparse_bwd",
]


class JFAError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("%s: %s" % (_STATUS.get(code, code), msg))
        self.code = code


_lib = None


def lib():
    """The loaded libjfa (ctypes), with argument types set. Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libjfa.so is not built (run __graft_entry__.build() or "
                           "python -m jagged_flash_attention_flashattention_gb300.build)")
    L = ctypes.CDLL(LIB_PATH)
    P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    sig = {
        "jfa_status_str": ([I], ctypes.c_char_p),
        "jfa_last_error": ([], ctypes.c_char_p),
        "jfa_sched_size": ([I64, I, I, P, I, I64, P], I),
        "jfa_sched_build": ([I64, I, I, I, P, I, I64, I64, I, P, P], I),
        "jfa_tile_rows": ([I, I, P], I),
        "jfa_num_sms": ([P], I),
        "jfa_workspace_size": ([I, I64, I, I], SZ),
        "jfa_workspace_init": ([P, SZ, P], I),
        "jfa_check_status": ([P, P], I),
        "jfa_fwd": ([P, P, P, P, I, I64, I64, I, I, F, P, P, I, P, P, P, SZ, P], I),
        "jfa_bwd": ([P, P, P, P, P, P, P, I, I64, I64, I, I, F, P, P, I, P, P, P, P, SZ, P], I),
        "jfa_bcastq_fwd": ([P, P, P, P, I, I64, I64, I64, I, I, F, P, P, I, P, P, P, SZ, P], I),
        "jfa_bcastq_bwd": ([P, P, P, P, P, P, P, I, I64, I64, I64, I, I, F, P, P, I, P, P, P, P,
                            SZ, P], I),
        "blockdiag_fwd": ([P, P, P, I64, I64, I, I, F, P, P, SZ, P], I),
        "blockdiag_bwd": ([P, P, P, P, I64, I64, I, I, F, P, P, P, P, SZ, P], I),
        "jfa_bwd_noalloc": ([P, P, P, P, P, P, P, I, I64, I64, I, I, F, P, P, I, P, P, P, P], I),
        "jfa_noalloc_check_status": ([P], I),
        "jfa_sched_size_varlen": ([I64, I, I, P, P, I, P], I),
        "jfa_sched_build_varlen": ([I64, I, I, I, P, P, I, I, I, I, P, P], I),
        "jfa_varlen_fwd": ([P, P, P, P, P, I, I64, I64, I64, I, I, F, I, I, P, P, I, P, P, P, SZ,
                            P], I),
        "jfa_varlen_bwd": ([P, P, P, P, P, P, P, P, I, I64, I64, I64, I, I, F, I, I, I, P, P, I, P,
                            P, P, P, SZ, P], I),
        "jfa_varlen_workspace_size": ([I64, P, P, I, I, I, I, P], I),
        "jfa_fwd_dynamic": ([P, P, P, P, I, I64, I64, I, I, F, P, I64, I, P, P, P, SZ, P], I),
        "jfa_fwd_dynamic_workspace_size": ([I64], SZ),
        "blockdiag_rotary_fwd": ([P, P, P, P, P, I64, I64, I, I, F, P, P, P, P, SZ, P], I),
        "blockdiag_rotary_bwd": ([P, P, P, P, P, P, I64, I64, I, I, F, P, P, P, P, SZ, P], I),
        "jfa_selftest_wait_timeout": ([P, SZ, ctypes.c_uint64, P], I),
        "jfa_fwd_pair": ([P, P, P, P, I, I64, I64, I, I, F, P, P, I, P, P, P, SZ, P], I),
        "jfa_num_pairs": ([P], I),
        "jfa_rope": ([P, P, I, I64, I64, I, I, P, P, I64, P, P], I),
        "jfa_rotary_bwd": ([P, P, P, P, P, P, P, I, I64, I64, I, I, F, P, P, I64, P, P, I, P, P, P,
                            P, SZ, P], I),
        "jfa_sched_size_sparse": ([I64, I, I, P, P, I, P, I64, P, P], I),
        "jfa_sched_build_sparse": ([I64, I, I, I, P, P, I, P, I64, I, P, P, P, P, P], I),
        "jfa_sparse_fwd": ([P, P, P, P, P, I, I64, I64, I64, I, I, F, P, P, P, P, P, I, P, P, P, SZ,
                            P], I),
        "jfa_sparse_bwd": ([P, P, P, P, P, P, P, P, I, I64, I64, I64, I, I, F, P, P, P, P, I, P, P,
                            P, P, SZ, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(code):
    if code != 0:
        raise JFAError(code, lib().jfa_last_error().decode())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")
        if t.dtype != torch.bfloat16:
            raise ValueError("tensors must be bf16")


def num_sms():
    n = ctypes.c_int(0)
    _check(lib().jfa_num_sms(ctypes.byref(n)))
    return n.value


def num_pairs():
    """Two-CTA clusters of the pair forward that fit on the device at once."""
    n = ctypes.c_int(0)
    _check(lib().jfa_num_pairs(ctypes.byref(n)))
    return n.value


def tile_rows(op, D):
    n = ctypes.c_int(0)
    _check(lib().jfa_tile_rows(op, D, ctypes.byref(n)))
    return n.value


def schedule(offsets_host, H, tile_rows_, n_sms, fixed_rows=0, fixed_work=0, zigzag=True):
    """Host LPT + zigzag schedule. Returns (sm_ptr [n_sms+1], tiles [n, 3]) int32 numpy."""
    off = np.ascontiguousarray(offsets_host)
    idx = JFA_I64 if off.dtype == np.int64 else JFA_I32
    if off.dtype not in (np.int32, np.int64):
        raise ValueError("offsets must be int32 or int64")
    B = off.size - 1
    n = ctypes.c_int64(0)
    L = lib()
    _check(L.jfa_sched_size(B, H, tile_rows_, off.ctypes.data, idx, fixed_rows, ctypes.byref(n)))
    sm_ptr = np.zeros(n_sms + 1, dtype=np.int32)
    tiles = np.zeros((max(n.value, 1), 3), dtype=np.int32)
    _check(L.jfa_sched_build(B, H, tile_rows_, n_sms, off.ctypes.data, idx, fixed_rows,
                             fixed_work, 1 if zigzag else 0, sm_ptr.ctypes.data,
                             tiles.ctypes.data))
    return sm_ptr, tiles[: n.value]


def check_host_offsets(host, n):
    """Raises unless `host` is a 1-D integer array of n >= 1 offsets starting at 0
    and non-decreasing (the host copy the scheduler reads must describe the
    device offsets the kernels read; at least its length is checked here)."""
    host = np.asarray(host)
    if host.ndim != 1 or host.size != n or host.size < 1:
        raise ValueError("host_offsets must be 1-D with as many entries as offsets (%d)" % n)
    if host.dtype not in (np.int32, np.int64):
        raise ValueError("offsets must be int32 or int64")
    if host[0] != 0 or np.any(np.diff(host.astype(np.int64)) < 0):
        raise ValueError("offsets must start at 0 and be non-decreasing")


def schedule_varlen(q_offsets_host, kv_offsets_host, H, op, n_sms, window=(-1, -1), zigzag=True):
    """Host LPT + zigzag schedule of the masked / cross attention tiles
    (op = OP_FWD or OP_BWD). Returns (sm_ptr, tiles) int32 numpy."""
    qo = np.ascontiguousarray(q_offsets_host)
    ko = np.ascontiguousarray(kv_offsets_host)
    if qo.dtype != ko.dtype or ko.dtype not in (np.int32, np.int64):
        raise ValueError("offsets must both be int32 or both int64")
    idx = JFA_I64 if ko.dtype == np.int64 else JFA_I32
    B = ko.size - 1
    n = ctypes.c_int64(0)
    L = lib()
    _check(L.jfa_sched_size_varlen(B, H, op, qo.ctypes.data, ko.ctypes.data, idx, ctypes.byref(n)))
    sm_ptr = np.zeros(n_sms + 1, dtype=np.int32)
    tiles = np.zeros((max(n.value, 1), 3), dtype=np.int32)
    _check(L.jfa_sched_build_varlen(B, H, op, n_sms, qo.ctypes.data, ko.ctypes.data, idx,
                                    int(window[0]), int(window[1]), 1 if zigzag else 0,
                                    sm_ptr.ctypes.data, tiles.ctypes.data))
    return sm_ptr, tiles[: n.value]


SPARSE_BLOCK = 128  # query and key rows per block of a block mask


def pack_block_masks(masks, q_offsets_host, kv_offsets_host):
    """The scheduler's mask array from one boolean (or 0/1) array per sequence,
    masks[b] of shape [ceil(Lq_b / 128), ceil(Lk_b / 128)] (row-major,
    concatenated, uint8), or a flat array already in that layout (checked
    for length)."""
    qo = np.asarray(q_offsets_host, dtype=np.int64)
    ko = np.asarray(kv_offsets_host, dtype=np.int64)
    nq = -(-np.diff(qo) // SPARSE_BLOCK)
    nk = -(-np.diff(ko) // SPARSE_BLOCK)
    need = int(np.sum(nq * nk))
    if isinstance(masks, np.ndarray) and masks.ndim == 1:
        # already packed: used as is when it is contiguous uint8 (any non-zero byte is a kept block)
        flat = masks if masks.dtype == np.uint8 else (masks != 0).astype(np.uint8)
        flat = np.ascontiguousarray(flat)
    else:
        if len(masks) != len(nq):
            raise ValueError("%d block masks for %d sequences" % (len(masks), len(nq)))
        arrs = [np.asarray(m) for m in masks]
        shapes = np.array([m.shape if m.ndim == 2 else (-1, -1) for m in arrs], dtype=np.int64)
        bad = np.flatnonzero((shapes[:, 0] != nq) | (shapes[:, 1] != nk)) if arrs else []
        if len(bad):
            b = int(bad[0])
            raise ValueError("block mask %d has shape %s, its sequence needs %s" % (
                b, arrs[b].shape, (int(nq[b]), int(nk[b]))))
        flat = (np.concatenate([m.ravel() for m in arrs]) != 0).view(np.uint8) if arrs \
            else np.zeros(0, np.uint8)
    if flat.size != need:
        raise ValueError("block masks hold %d blocks, the offsets need %d" % (flat.size, need))
    return flat


def schedule_sparse(q_offsets_host, kv_offsets_host, H, op, n_sms, masks, zigzag=True):
    """Host LPT + zigzag schedule of block-sparse tiles (op = OP_FWD or
    OP_BWD) and their lists. `masks`: as for :func:`pack_block_masks`.
    Returns (sm_ptr, tiles [n, 3], list_ptr [n + 1], entries, meta [n, 4] or
    None for the backward), int32 numpy."""
    qo = np.ascontiguousarray(q_offsets_host)
    ko = np.ascontiguousarray(kv_offsets_host)
    if qo.dtype != ko.dtype or ko.dtype not in (np.int32, np.int64):
        raise ValueError("offsets must both be int32 or both int64")
    idx = JFA_I64 if ko.dtype == np.int64 else JFA_I32
    flat = pack_block_masks(masks, qo, ko)
    B = ko.size - 1
    n, ne = ctypes.c_int64(0), ctypes.c_int64(0)
    L = lib()
    _check(L.jfa_sched_size_sparse(B, H, op, qo.ctypes.data, ko.ctypes.data, idx, flat.ctypes.data,
                                   flat.size, ctypes.byref(n), ctypes.byref(ne)))
    sm_ptr = np.zeros(n_sms + 1, dtype=np.int32)
    tiles = np.zeros((max(n.value, 1), 3), dtype=np.int32)
    list_ptr = np.zeros(n.value + 1, dtype=np.int32)
    entries = np.zeros(max(ne.value, 1), dtype=np.int32)
    meta = np.zeros((max(n.value, 1), 4), dtype=np.int32)
    _check(L.jfa_sched_build_sparse(B, H, op, n_sms, qo.ctypes.data, ko.ctypes.data, idx,
                                    flat.ctypes.data, flat.size, 1 if zigzag else 0,
                                    sm_ptr.ctypes.data, tiles.ctypes.data, list_ptr.ctypes.data,
                                    entries.ctypes.data, meta.ctypes.data))
    return (sm_ptr, tiles[: n.value], list_ptr, entries,
            meta[: n.value] if op == OP_FWD else None)


class Plan:
    """Schedules (on the device) and workspace for one batch layout.

    kind: "jagged" (offsets of the packed Q/K/V), "bcast" (offsets of the
    packed K/V, dense Q of length Lq) or "varlen" (`offsets` of the packed
    K/V and `q_offsets` of the packed queries, which may be the same tensor;
    band mask `window` = (left, right), -1 unbounded; `deterministic` sizes
    the workspace for the ordered dQ reduction). The scheduler runs on the
    host, so it reads host offsets: pass them as `host_offsets` /
    `host_q_offsets` (numpy) when the caller already has them, otherwise they
    are copied from the device once. Tile lists are copied to the device
    asynchronously from pinned memory. `workspace` (uint8 CUDA tensor) may be
    shared between plans; it is allocated when absent or too small.
    `pair` (jagged, D = 128): the forward runs on CTA pairs (jfa_fwd_pair,
    512-row tiles scheduled over jfa_num_pairs() slots); same results.
    kind "sparse": as "varlen" without a window, plus `block_masks` (one
    [ceil(Lq_b / 128), ceil(Lk_b / 128)] boolean array per sequence, see
    :func:`pack_block_masks`); the schedules then carry the per-tile block
    lists.
    """

    def __init__(self, offsets, H, D, kind="jagged", Lq=0, zigzag=True, host_offsets=None,
                 workspace=None, q_offsets=None, host_q_offsets=None, window=(-1, -1),
                 deterministic=False, pair=False, block_masks=None):
        if not offsets.is_cuda:
            raise ValueError("offsets must be a CUDA tensor")
        self.offsets = offsets
        self.idx = JFA_I64 if offsets.dtype == torch.int64 else JFA_I32
        host = np.asarray(host_offsets) if host_offsets is not None else offsets.cpu().numpy()
        check_host_offsets(host, offsets.numel())
        self.host_offsets = host
        self.B = host.size - 1
        self.T = int(host[-1])
        self.H, self.D, self.kind, self.Lq = H, D, kind, int(Lq)
        self.window = (int(window[0]), int(window[1]))
        self.deterministic = bool(deterministic)
        self.n_sms = num_sms()
        dev = offsets.device
        if kind in ("varlen", "sparse"):
            self.q_offsets = offsets if q_offsets is None else q_offsets
            if self.q_offsets.dtype != offsets.dtype:
                raise ValueError("q_offsets and offsets must have the same dtype")
            if host_q_offsets is not None:
                hq = np.asarray(host_q_offsets)
            elif q_offsets is None:
                hq = host
            else:
                hq = self.q_offsets.cpu().numpy()
            check_host_offsets(hq, self.q_offsets.numel())
            self.host_q_offsets = hq
            self.Tq = int(hq[-1])
        if kind == "sparse":
            if block_masks is None:
                raise ValueError("a sparse plan needs block_masks")
            if self.window != (-1, -1) or self.deterministic:
                raise ValueError("block masks take no window and no deterministic dQ")
            flat = pack_block_masks(block_masks, self.host_q_offsets, host)
            f = schedule_sparse(self.host_q_offsets, host, H, OP_FWD, self.n_sms, flat, zigzag)
            bwd = schedule_sparse(self.host_q_offsets, host, H, OP_BWD, self.n_sms, flat, zigzag)[:4]
            # (sm_ptr, tiles, list_ptr, entries, meta); meta keeps one row when there are no tiles
            fwd = f[:4] + (f[4] if f[4].size else np.zeros((1, 4), np.int32),)
        elif kind == "varlen":
            fwd = schedule_varlen(self.host_q_offsets, host, H, OP_FWD, self.n_sms, self.window,
                                  zigzag)
            bwd = schedule_varlen(self.host_q_offsets, host, H, OP_BWD, self.n_sms, self.window,
                                  zigzag)
        elif kind == "jagged":
            # pair: the forward runs on CTA pairs (jfa_fwd_pair, D = 128 only).
            self.pair = bool(pair)
            if self.pair and D != 128:
                raise ValueError("the CTA-pair forward takes D = 128")
            if self.pair:
                self.n_pairs = num_pairs()
                fwd = schedule(host, H, tile_rows(OP_FWD_PAIR, D), self.n_pairs, zigzag=zigzag)
            else:
                fwd = schedule(host, H, tile_rows(OP_FWD, D), self.n_sms, zigzag=zigzag)
            bwd = schedule(host, H, tile_rows(OP_BWD, D), self.n_sms, zigzag=zigzag)
        else:
            fwd = schedule(host, H, tile_rows(OP_BCASTQ_FWD, D), self.n_sms, fixed_rows=self.Lq,
                           zigzag=zigzag)
            bwd = schedule(host, H, tile_rows(OP_BCASTQ_BWD, D), self.n_sms, fixed_work=self.Lq,
                           zigzag=zigzag)
        # All the int32 lists go up in one pinned staging buffer and one copy,
        # each starting on a 16-byte boundary (the kernels read some as int4).
        arrs = [np.ascontiguousarray(a, dtype=np.int32) for a in fwd + bwd]
        starts, total = [], 0
        for a in arrs:
            starts.append(total)
            total += -(-a.size // 4) * 4
        staging = np.zeros(max(total, 4), dtype=np.int32)
        for a, s0 in zip(arrs, starts):
            staging[s0:s0 + a.size] = a.ravel()
        self._pinned = torch.from_numpy(staging).pin_memory()
        dbuf = self._pinned.to(dev, non_blocking=True)
        d = [dbuf[s0:s0 + a.size].view(a.shape) for a, s0 in zip(arrs, starts)]
        nf = len(fwd)
        self.fwd_sched, self.bwd_sched = tuple(d[:nf]), tuple(d[nf:])
        self.n_fwd_tiles, self.n_bwd_tiles = fwd[1].shape[0], bwd[1].shape[0]
        if kind in ("varlen", "sparse"):
            sz = ctypes.c_size_t(0)
            hq = np.ascontiguousarray(self.host_q_offsets)
            hk = np.ascontiguousarray(host)
            _check(lib().jfa_varlen_workspace_size(self.B, hq.ctypes.data, hk.ctypes.data, self.idx,
                                                   H, D, 1 if self.deterministic else 0,
                                                   ctypes.byref(sz)))
            nbytes = sz.value
        else:
            rows = self.T if kind == "jagged" else self.Lq
            op = OP_BWD if kind == "jagged" else OP_BCASTQ_BWD
            nbytes = lib().jfa_workspace_size(op, rows, H, D)
        if workspace is None or workspace.numel() < nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            _check(lib().jfa_workspace_init(_ptr(workspace), nbytes, _stream()))
        self.workspace = workspace

    def check(self):
        """Synchronises and raises if a kernel reported a timeout."""
        _check(lib().jfa_check_status(_ptr(self.workspace), _stream()))

    def validate(self, kind, offsets, rows, H, D, Lq=0):
        """Raises if this plan was built for another batch layout than the call's:
        kind, offsets tensor length, packed rows (T for jagged, Tk for
        broadcast-Q, which must equal the last offset), heads, head dim and
        broadcast length. The kernels also clamp every sequence to the tensors
        they are given, so a mismatch that got past this check could give wrong
        numbers but never touch memory outside the tensors."""
        want = (kind, offsets.numel() - 1, rows, H, D, int(Lq))
        have = (self.kind, self.B, self.T, self.H, self.D, self.Lq)
        if want != have:
            raise ValueError("plan built for (kind, B, T, H, D, Lq) = %s, call has %s" % (have, want))


def _check_varlen_plan(plan, q_offsets, kv_offsets, Tq, Tk, H, D, window):
    if plan.kind != "varlen":
        raise ValueError("a varlen call needs a plan of kind 'varlen'")
    if (plan.B, plan.T, plan.Tq, plan.H, plan.D) != (kv_offsets.numel() - 1, Tk, Tq, H, D):
        raise ValueError("plan built for (B, Tk, Tq, H, D) = %s, call has %s" % (
            (plan.B, plan.T, plan.Tq, plan.H, plan.D), (kv_offsets.numel() - 1, Tk, Tq, H, D)))
    if q_offsets.numel() != kv_offsets.numel():
        raise ValueError("q_offsets and kv_offsets must have the same length")
    if tuple(window) != plan.window:
        raise ValueError("plan built for window %s, call has %s" % (plan.window, tuple(window)))


def _scale(scale, D):
    return 1.0 / math.sqrt(D) if scale is None else float(scale)


def jfa_fwd(q, k, v, offsets, scale=None, plan=None):
    """Jagged forward. q, k, v: [T, H, D] bf16 CUDA; offsets [B+1] int32/int64 CUDA.
    Returns (o [T, H, D] bf16, lse [H, T] fp32)."""
    _need_cuda(q, k, v)
    T, H, D = q.shape
    plan = plan or Plan(offsets, H, D)
    plan.validate("jagged", offsets, T, H, D)
    o = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    sp, tl = plan.fwd_sched
    if getattr(plan, "pair", False):
        _check(lib().jfa_fwd_pair(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), plan.idx, plan.B, T, H,
                                  D, _scale(scale, D), _ptr(sp), _ptr(tl), plan.n_pairs, _ptr(o),
                                  _ptr(lse), _ptr(plan.workspace), plan.workspace.numel(), _stream()))
    else:
        _check(lib().jfa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), plan.idx, plan.B, T, H, D,
                             _scale(scale, D), _ptr(sp), _ptr(tl), plan.n_sms, _ptr(o), _ptr(lse),
                             _ptr(plan.workspace), plan.workspace.numel(), _stream()))
    return o, lse


def _check_rope_tables(cos, sin, D, plan):
    for t in (cos, sin):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.float32 and t.dim() == 2 and
                t.shape[1] == D // 2 and t.shape[0] == cos.shape[0]):
            raise ValueError("rotary tables must be contiguous fp32 CUDA tensors [L, D/2]")
    lmax = int(np.max(np.diff(plan.host_offsets))) if plan.B > 0 else 0
    if lmax > cos.shape[0]:
        raise ValueError("a sequence of %d tokens is longer than the rotary tables (%d rows)"
                         % (lmax, cos.shape[0]))


def jfa_rope(x, offsets, cos, sin, plan=None):
    """Rotary embedding of x [T, H, D] bf16 with each row at its position in its
    sequence (tables cos, sin [L, D/2] fp32): returns x_rot. The rotary forward
    of a layer whose attention then runs on the rotated q and k."""
    _need_cuda(x)
    T, H, D = x.shape
    plan = plan or Plan(offsets, H, D)
    plan.validate("jagged", offsets, T, H, D)
    _check_rope_tables(cos, sin, D, plan)
    y = torch.empty_like(x)
    _check(lib().jfa_rope(_ptr(x), _ptr(offsets), plan.idx, plan.B, T, H, D, _ptr(cos), _ptr(sin),
                          cos.shape[0], _ptr(y), _stream()))
    return y


def jfa_rotary_bwd(q_rot, k_rot, v, o, lse, do, offsets, cos, sin, scale=None, plan=None):
    """Jagged backward from the rotated q_rot, k_rot (as jfa_rope writes them),
    with the rotary backward fused in: returns (dq, dk, dv) with respect to the
    unrotated q, k and v (dQ and dK rotated back in the backward's closing
    cast of dQ)."""
    _need_cuda(q_rot, k_rot, v, o, do)
    T, H, D = q_rot.shape
    plan = plan or Plan(offsets, H, D)
    plan.validate("jagged", offsets, T, H, D)
    _check_rope_tables(cos, sin, D, plan)
    dq, dk, dv = torch.empty_like(q_rot), torch.empty_like(k_rot), torch.empty_like(v)
    sp, tl = plan.bwd_sched
    _check(lib().jfa_rotary_bwd(_ptr(q_rot), _ptr(k_rot), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                _ptr(offsets), plan.idx, plan.B, T, H, D, _scale(scale, D),
                                _ptr(cos), _ptr(sin), cos.shape[0], _ptr(sp), _ptr(tl), plan.n_sms,
                                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(plan.workspace),
                                plan.workspace.numel(), _stream()))
    return dq, dk, dv


def jfa_bwd(q, k, v, o, lse, do, offsets, scale=None, plan=None):
    """Jagged backward. Returns (dq, dk, dv), each [T, H, D] bf16."""
    _need_cuda(q, k, v, o, do)
    T, H, D = q.shape
    plan = plan or Plan(offsets, H, D)
    plan.validate("jagged", offsets, T, H, D)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    sp, tl = plan.bwd_sched
    _check(lib().jfa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(offsets),
                         plan.idx, plan.B, T, H, D, _scale(scale, D), _ptr(sp), _ptr(tl),
                         plan.n_sms, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(plan.workspace),
                         plan.workspace.numel(), _stream()))
    return dq, dk, dv


def jfa_varlen_fwd(q, k, v, q_offsets, kv_offsets, scale=None, window=(-1, -1), plan=None):
    """Masked / cross attention forward. q [Tq, H, D], k, v [Tk, H, D] bf16 CUDA;
    q_offsets, kv_offsets [B+1] (same dtype; the same tensor twice for
    self-attention); window = (left, right) band mask, (-1, -1) none, (-1, 0)
    causal. Returns (o [Tq, H, D] bf16, lse [H, Tq] fp32)."""
    _need_cuda(q, k, v)
    Tq, H, D = q.shape
    Tk = k.shape[0]
    plan = plan or Plan(kv_offsets, H, D, kind="varlen", q_offsets=q_offsets, window=window)
    _check_varlen_plan(plan, q_offsets, kv_offsets, Tq, Tk, H, D, window)
    o = torch.empty_like(q)
    lse = torch.empty((H, Tq), dtype=torch.float32, device=q.device)
    sp, tl = plan.fwd_sched
    # a deterministic plan's workspace holds no accumulator for the forward to clear
    ws_bytes = 256 if plan.deterministic else plan.workspace.numel()
    _check(lib().jfa_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(q_offsets), _ptr(kv_offsets),
                                plan.idx, plan.B, Tq, Tk, H, D, _scale(scale, D), int(window[0]),
                                int(window[1]), _ptr(sp), _ptr(tl), plan.n_sms, _ptr(o), _ptr(lse),
                                _ptr(plan.workspace), ws_bytes, _stream()))
    return o, lse


def jfa_varlen_bwd(q, k, v, o, lse, do, q_offsets, kv_offsets, scale=None, window=(-1, -1),
                   deterministic=False, plan=None):
    """Backward of :func:`jfa_varlen_fwd`. With deterministic=True the dQ
    reduction runs in a fixed order (bit-identical dQ from run to run); the
    plan must then be built with deterministic=True. Returns (dq, dk, dv) bf16."""
    _need_cuda(q, k, v, o, do)
    Tq, H, D = q.shape
    Tk = k.shape[0]
    plan = plan or Plan(kv_offsets, H, D, kind="varlen", q_offsets=q_offsets, window=window,
                        deterministic=deterministic)
    _check_varlen_plan(plan, q_offsets, kv_offsets, Tq, Tk, H, D, window)
    if deterministic and not plan.deterministic:
        raise ValueError("deterministic=True needs a plan built with deterministic=True")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    sp, tl = plan.bwd_sched
    _check(lib().jfa_varlen_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                _ptr(q_offsets), _ptr(kv_offsets), plan.idx, plan.B, Tq, Tk, H, D,
                                _scale(scale, D), int(window[0]), int(window[1]),
                                1 if deterministic else 0, _ptr(sp), _ptr(tl), plan.n_sms,
                                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(plan.workspace),
                                plan.workspace.numel(), _stream()))
    return dq, dk, dv


def _check_sparse_plan(plan, q_offsets, kv_offsets, Tq, Tk, H, D):
    if plan is None or plan.kind != "sparse":
        raise ValueError("a block-sparse call needs a plan of kind 'sparse' (it holds the masks)")
    if (plan.B, plan.T, plan.Tq, plan.H, plan.D) != (kv_offsets.numel() - 1, Tk, Tq, H, D):
        raise ValueError("plan built for (B, Tk, Tq, H, D) = %s, call has %s" % (
            (plan.B, plan.T, plan.Tq, plan.H, plan.D), (kv_offsets.numel() - 1, Tk, Tq, H, D)))
    if q_offsets.numel() != kv_offsets.numel():
        raise ValueError("q_offsets and kv_offsets must have the same length")


def jfa_sparse_fwd(q, k, v, q_offsets, kv_offsets, block_masks=None, scale=None, plan=None):
    """Block-sparse attention forward: query i of sequence b sees key j iff
    block_masks[b][i // 128, j // 128]. q [Tq, H, D], k, v [Tk, H, D] bf16
    CUDA; q_offsets, kv_offsets [B+1] (same dtype). Pass block_masks, or a
    plan of kind "sparse" built with them. Returns (o [Tq, H, D] bf16,
    lse [H, Tq] fp32); rows that see no key get O = 0, LSE = -inf."""
    _need_cuda(q, k, v)
    Tq, H, D = q.shape
    Tk = k.shape[0]
    if plan is None:
        plan = Plan(kv_offsets, H, D, kind="sparse", q_offsets=q_offsets, block_masks=block_masks)
    _check_sparse_plan(plan, q_offsets, kv_offsets, Tq, Tk, H, D)
    o = torch.empty_like(q)
    lse = torch.empty((H, Tq), dtype=torch.float32, device=q.device)
    sp, tl, lp, ent, meta = plan.fwd_sched
    _check(lib().jfa_sparse_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(q_offsets), _ptr(kv_offsets),
                                plan.idx, plan.B, Tq, Tk, H, D, _scale(scale, D), _ptr(sp), _ptr(tl),
                                _ptr(lp), _ptr(ent), _ptr(meta), plan.n_sms, _ptr(o), _ptr(lse),
                                _ptr(plan.workspace), plan.workspace.numel(), _stream()))
    return o, lse


def jfa_sparse_bwd(q, k, v, o, lse, do, q_offsets, kv_offsets, block_masks=None, scale=None,
                   plan=None):
    """Backward of :func:`jfa_sparse_fwd`. Returns (dq, dk, dv) bf16; keys that
    no query sees get dK = dV = 0."""
    _need_cuda(q, k, v, o, do)
    Tq, H, D = q.shape
    Tk = k.shape[0]
    if plan is None:
        plan = Plan(kv_offsets, H, D, kind="sparse", q_offsets=q_offsets, block_masks=block_masks)
    _check_sparse_plan(plan, q_offsets, kv_offsets, Tq, Tk, H, D)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    sp, tl, lp, ent = plan.bwd_sched
    _check(lib().jfa_sparse_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                _ptr(q_offsets), _ptr(kv_offsets), plan.idx, plan.B, Tq, Tk, H, D,
                                _scale(scale, D), _ptr(sp), _ptr(tl), _ptr(lp), _ptr(ent),
                                plan.n_sms, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(plan.workspace),
                                plan.workspace.numel(), _stream()))
    return dq, dk, dv


class DynamicPlan:
    """Workspace (and, for order="lpt", the longest-first tile list) of the
    forward with device-side dynamic tile scheduling. order="device": tiles
    enumerated on the device from the device offsets, no host work at all;
    order="lpt": the host sorts the tiles longest first and the CTAs claim
    them in that order (greedy LPT)."""

    def __init__(self, offsets, H, D, order="device", host_offsets=None):
        if order not in ("device", "lpt"):
            raise ValueError("order must be 'device' or 'lpt'")
        self.offsets, self.H, self.D, self.order = offsets, H, D, order
        self.idx = JFA_I64 if offsets.dtype == torch.int64 else JFA_I32
        self.B = offsets.numel() - 1
        self.n_ctas = num_sms()
        self.tiles, self.n_tiles = None, 0
        if order == "lpt":
            host = np.asarray(host_offsets) if host_offsets is not None else offsets.cpu().numpy()
            check_host_offsets(host, offsets.numel())
            _, tl = schedule(host, H, tile_rows(OP_FWD, D), 1, zigzag=True)
            self._pinned = torch.from_numpy(np.ascontiguousarray(tl)).pin_memory()
            self.tiles = self._pinned.to(offsets.device, non_blocking=True)
            self.n_tiles = tl.shape[0]
        nbytes = lib().jfa_fwd_dynamic_workspace_size(self.B)
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=offsets.device)

    def check(self):
        _check(lib().jfa_check_status(_ptr(self.workspace), _stream()))


def jfa_fwd_dynamic(q, k, v, offsets, scale=None, plan=None, order="device"):
    """Jagged forward whose persistent CTAs claim tiles at run time from a
    global counter (see :class:`DynamicPlan`). Returns (o, lse) like jfa_fwd."""
    _need_cuda(q, k, v)
    T, H, D = q.shape
    plan = plan or DynamicPlan(offsets, H, D, order=order)
    if (plan.B, plan.H, plan.D) != (offsets.numel() - 1, H, D):
        raise ValueError("dynamic plan built for another layout")
    o = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    _check(lib().jfa_fwd_dynamic(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), plan.idx, plan.B, T, H, D,
                                 _scale(scale, D), _ptr(plan.tiles), plan.n_tiles, plan.n_ctas, _ptr(o),
                                 _ptr(lse), _ptr(plan.workspace), plan.workspace.numel(), _stream()))
    return o, lse


def jfa_bcastq_fwd(q, k, v, kv_offsets, scale=None, plan=None):
    """Broadcast-Q forward. q [Lq, H, D]; k, v [Tk, H, D]; kv_offsets [B+1].
    Returns (o [B, Lq, H, D], lse [B, H, Lq])."""
    _need_cuda(q, k, v)
    Lq, H, D = q.shape
    plan = plan or Plan(kv_offsets, H, D, kind="bcast", Lq=Lq)
    plan.validate("bcast", kv_offsets, k.shape[0], H, D, Lq)
    Tk, B = k.shape[0], plan.B
    o = torch.empty((B, Lq, H, D), dtype=q.dtype, device=q.device)
    lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    sp, tl = plan.fwd_sched
    _check(lib().jfa_bcastq_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_offsets), plan.idx, B, Lq, Tk,
                                H, D, _scale(scale, D), _ptr(sp), _ptr(tl), plan.n_sms, _ptr(o),
                                _ptr(lse), _ptr(plan.workspace), plan.workspace.numel(),
                                _stream()))
    return o, lse


def jfa_bcastq_bwd(q, k, v, o, lse, do, kv_offsets, scale=None, plan=None):
    """Broadcast-Q backward. Returns (dq [Lq, H, D] fp32 summed over sequences,
    dk, dv [Tk, H, D] bf16)."""
    _need_cuda(q, k, v, o, do)
    Lq, H, D = q.shape
    plan = plan or Plan(kv_offsets, H, D, kind="bcast", Lq=Lq)
    plan.validate("bcast", kv_offsets, k.shape[0], H, D, Lq)
    Tk, B = k.shape[0], plan.B
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    sp, tl = plan.bwd_sched
    _check(lib().jfa_bcastq_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                _ptr(kv_offsets), plan.idx, B, Lq, Tk, H, D, _scale(scale, D),
                                _ptr(sp), _ptr(tl), plan.n_sms, _ptr(dq), _ptr(dk), _ptr(dv),
                                _ptr(plan.workspace), plan.workspace.numel(), _stream()))
    return dq, dk, dv


_ws_cache = {}


def _small_workspace(device):
    key = str(device)
    if key not in _ws_cache:
        _ws_cache[key] = torch.zeros(lib().jfa_workspace_size(OP_BLOCKDIAG_FWD, 0, 1, 64),
                                     dtype=torch.uint8, device=device)
    return _ws_cache[key]


def blockdiag_fwd(q, k, v, scale=None):
    """64-token block-diagonal forward on [B, L, H, D] bf16. Returns o."""
    _need_cuda(q, k, v)
    B, L, H, D = q.shape
    o = torch.empty_like(q)
    ws = _small_workspace(q.device)
    _check(lib().blockdiag_fwd(_ptr(q), _ptr(k), _ptr(v), B, L, H, D, _scale(scale, D), _ptr(o),
                               _ptr(ws), ws.numel(), _stream()))
    return o


def blockdiag_bwd(q, k, v, do, scale=None):
    """64-token block-diagonal backward. Returns (dq, dk, dv)."""
    _need_cuda(q, k, v, do)
    B, L, H, D = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = _small_workspace(q.device)
    _check(lib().blockdiag_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, L, H, D, _scale(scale, D),
                               _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream()))
    return dq, dk, dv


def _check_tables(cos, sin, L, D):
    for t in (cos, sin):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.float32 and
                tuple(t.shape) == (L, D // 2)):
            raise ValueError("rotary tables must be contiguous fp32 CUDA tensors [L, D/2]")


def blockdiag_rotary_fwd(q, k, v, cos, sin, scale=None, return_rotated=False):
    """64-token block-diagonal forward with q and k rotated in the kernel by the
    rotary tables cos, sin [L, D/2] (fp32). Returns o, or (o, q_rot, k_rot)
    with the rotated q and k the kernel wrote (bf16), which the backward takes."""
    _need_cuda(q, k, v)
    B, L, H, D = q.shape
    _check_tables(cos, sin, L, D)
    o = torch.empty_like(q)
    q_rot = torch.empty_like(q) if return_rotated else None
    k_rot = torch.empty_like(k) if return_rotated else None
    ws = _small_workspace(q.device)
    _check(lib().blockdiag_rotary_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cos), _ptr(sin), B, L, H, D,
                                      _scale(scale, D), _ptr(o),
                                      _ptr(q_rot) if return_rotated else None,
                                      _ptr(k_rot) if return_rotated else None,
                                      _ptr(ws), ws.numel(), _stream()))
    return (o, q_rot, k_rot) if return_rotated else o


def blockdiag_rotary_bwd(q_rot, k_rot, v, do, cos, sin, scale=None):
    """Backward of :func:`blockdiag_rotary_fwd` with the rotary backward fused
    into the epilogue: from the rotated q_rot, k_rot (as the forward writes
    them), v and do, returns (dq, dk, dv) with respect to the unrotated q, k
    and v."""
    _need_cuda(q_rot, k_rot, v, do)
    B, L, H, D = q_rot.shape
    _check_tables(cos, sin, L, D)
    dq, dk, dv = torch.empty_like(q_rot), torch.empty_like(k_rot), torch.empty_like(v)
    ws = _small_workspace(q_rot.device)
    _check(lib().blockdiag_rotary_bwd(_ptr(q_rot), _ptr(k_rot), _ptr(v), _ptr(do), _ptr(cos),
                                      _ptr(sin), B, L, H, D, _scale(scale, D), _ptr(dq), _ptr(dk),
                                      _ptr(dv), _ptr(ws), ws.numel(), _stream()))
    return dq, dk, dv


def check_status(workspace=None, device=None):
    """Synchronises the current stream and raises JFAError if a kernel gave up waiting."""
    ws = workspace if workspace is not None else _small_workspace(device or torch.device("cuda"))
    _check(lib().jfa_check_status(_ptr(ws), _stream()))
