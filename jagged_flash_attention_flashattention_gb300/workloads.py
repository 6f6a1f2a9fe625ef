"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA path.

This module draws random numbers and lays them out; it holds none of the
attention arithmetic. It is the one module that both the oracle checks and
the library's callers (tests, bench) use, so that both sides see identical
bf16 bytes.

Workloads (the shapes of the pages' GEM jagged attention, broadcast-Q and
block-diagonal cases; user-sequence data is proprietary, so these stand in):

===========  ====================================================  =====
name         lengths                                               H, D
===========  ====================================================  =====
tiny         B=4, uniform integers in [1, 128]                     2, 64
gem          B=1024, rint(exp(ln 256 + 0.8 z)) clipped to [1,2048]  4, 128
stress       4 x 16384 plus 252 uniform in [1, 256], shuffled       4, 128
bcast        Lq=256 dense Q; B=512 K/V lengths uniform [64, 1024]   4, 128
blockdiag    B=1152, L=4096 (64 blocks of 64 tokens)               2, 128
blockdiag64  same, D=64                                            2, 64
gem_sparse   the gem lengths with block masks (block_masks below)  4, 128
gem_cross    query lengths of gem; key/value lengths drawn the      4, 128
             same way with seed 6 (jagged cross attention)
===========  ====================================================  =====

Lengths come from ``numpy.random.default_rng(seed)``; values are N(0, 1)
drawn as fp32 by a seeded ``torch.Generator`` on the requested device and
rounded to bf16 (round to nearest even) by torch.
"""

import math

import numpy as np
import torch

SEEDS = {"tiny": 1, "gem": 2, "stress": 3, "bcast": 4, "blockdiag": 5, "blockdiag64": 5,
         "blockdiag_rotary": 5, "gem_rotary": 2, "gem_sparse": 2, "gem_cross": 2}
KV_SEEDS = {"gem_cross": 6}  # key/value lengths of the cross-attention workload
MASK_SEEDS = {"gem_sparse": 12}


def lengths_for(name, seed=None):
    """Sequence lengths (numpy int64) of a named jagged workload."""
    seed = SEEDS[name] if seed is None else seed
    rng = np.random.default_rng(seed)
    if name == "tiny":
        return rng.integers(1, 129, 4).astype(np.int64)
    if name == "gem":
        z = rng.standard_normal(1024)
        return np.clip(np.rint(np.exp(math.log(256.0) + 0.8 * z)), 1, 2048).astype(np.int64)
    if name == "stress":
        L = np.concatenate([np.full(4, 16384), rng.integers(1, 257, 252)]).astype(np.int64)
        return L[rng.permutation(L.size)]
    if name == "bcast":
        return rng.integers(64, 1025, 512).astype(np.int64)
    raise KeyError(name)


def offsets_of(lengths, dtype=np.int64):
    """Prefix sums [B+1] with offsets[0] = 0."""
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    off[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return off.astype(dtype)


def block_masks(q_lengths, kv_lengths, seed, density=0.5, causal=True):
    """One boolean mask of 128 x 128 blocks per sequence, shape
    [ceil(Lq / 128), ceil(Lk / 128)], drawn from numpy.random.default_rng(seed).
    causal=True: block-causal (block column j <= block row i, counted from the
    bottom-right corner when Lq != Lk) with the diagonal block kept and every
    other block below it kept with probability `density` (a local-plus-random
    pattern: every query sees its own block). causal=False: every block kept
    with probability `density`."""
    rng = np.random.default_rng(seed)
    out = []
    for lq, lk in zip(q_lengths, kv_lengths):
        nq, nk = -(-int(lq) // 128), -(-int(lk) // 128)
        keep = rng.random((nq, nk)) < density
        if causal:
            i = np.arange(nq)[:, None] + (nk - nq)
            j = np.arange(nk)[None, :]
            keep = (keep & (j < i)) | (j == i)
        out.append(keep)
    return out


def randn_bf16(shape, seed, device="cpu"):
    """N(0,1) fp32 from a seeded torch generator on `device`, rounded to bf16."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def jagged_inputs(lengths, H, D, seed, device="cpu", with_grad=True):
    """Packed q, k, v (and dO) [T, H, D] bf16 for the given lengths."""
    T = int(np.sum(lengths))
    names = ("q", "k", "v", "do") if with_grad else ("q", "k", "v")
    return {n: randn_bf16((T, H, D), seed * 1000 + i, device) for i, n in enumerate(names)}


def bcast_inputs(lengths, Lq, H, D, seed, device="cpu", with_grad=True):
    """q [Lq, H, D]; k, v [Tk, H, D]; dO [B, Lq, H, D] (bf16)."""
    Tk = int(np.sum(lengths))
    out = {
        "q": randn_bf16((Lq, H, D), seed * 1000 + 0, device),
        "k": randn_bf16((Tk, H, D), seed * 1000 + 1, device),
        "v": randn_bf16((Tk, H, D), seed * 1000 + 2, device),
    }
    if with_grad:
        out["do"] = randn_bf16((len(lengths), Lq, H, D), seed * 1000 + 3, device)
    return out


def blockdiag_inputs(B, L, H, D, seed, device="cpu", with_grad=True):
    """q, k, v (and dO) [B, L, H, D] bf16."""
    names = ("q", "k", "v", "do") if with_grad else ("q", "k", "v")
    return {n: randn_bf16((B, L, H, D), seed * 1000 + i, device) for i, n in enumerate(names)}


def rotary_tables(L, D, base=10000.0, device="cpu"):
    """The usual rotary tables: angle = position * base^(-2i/D) for i < D/2,
    computed in float64 and stored as fp32 [L, D/2] (cos, sin)."""
    i = np.arange(D // 2, dtype=np.float64)
    ang = np.arange(L, dtype=np.float64)[:, None] * base ** (-2.0 * i / D)[None, :]
    return (torch.from_numpy(np.cos(ang).astype(np.float32)).to(device),
            torch.from_numpy(np.sin(ang).astype(np.float32)).to(device))


WORKLOADS = {
    "tiny": dict(kind="jagged", H=2, D=64, offsets_dtype=np.int32),
    "gem": dict(kind="jagged", H=4, D=128, offsets_dtype=np.int64),
    # the GEM batch with a causal mask, and with the deterministic dQ reduction
    "gem_causal": dict(kind="varlen", lengths="gem", H=4, D=128, offsets_dtype=np.int64,
                       window=(-1, 0), deterministic=False),
    "gem_det": dict(kind="varlen", lengths="gem", H=4, D=128, offsets_dtype=np.int64,
                    window=(-1, -1), deterministic=True),
    "stress": dict(kind="jagged", H=4, D=128, offsets_dtype=np.int64),
    "bcast": dict(kind="bcast", H=4, D=128, Lq=256, offsets_dtype=np.int64),
    "blockdiag": dict(kind="blockdiag", B=1152, L=4096, H=2, D=128),
    "blockdiag64": dict(kind="blockdiag", B=1152, L=4096, H=2, D=64),
    # the GEM batch with rotary embeddings (rotary layer, forward, backward
    # with the rotary backward fused in)
    "gem_rotary": dict(kind="jagged", lengths="gem", H=4, D=128, offsets_dtype=np.int64,
                       rotary=True),
    # the block-diagonal configuration with rotary embeddings fused in
    "blockdiag_rotary": dict(kind="blockdiag", B=1152, L=4096, H=2, D=128, rotary=True),
    # jagged cross attention: GEM query lengths against independently drawn
    # GEM-distributed key/value lengths (separate offsets), no mask
    "gem_cross": dict(kind="varlen", lengths="gem", kv_seed=6, H=4, D=128, offsets_dtype=np.int64,
                      window=(-1, -1), deterministic=False),
    # the GEM batch with block-causal block-sparse masks (block_masks, density 0.5)
    "gem_sparse": dict(kind="sparse", lengths="gem", H=4, D=128, offsets_dtype=np.int64,
                       density=0.5),
}


def visible_pairs(Lq, Lk, window=(-1, -1)):
    """Number of (query, key) pairs of one sequence that a band mask
    (left, right) keeps (-1 = unbounded; query i is aligned with key
    i + Lk - Lq). Used to count useful FLOPs of masked workloads."""
    left, right = window
    i = np.arange(Lq, dtype=np.int64) + (Lk - Lq)
    lo = np.zeros(Lq, dtype=np.int64) if left < 0 else np.maximum(0, i - left)
    hi = np.full(Lq, Lk - 1, dtype=np.int64) if right < 0 else np.minimum(Lk - 1, i + right)
    return int(np.sum(np.maximum(0, hi - lo + 1)))


def masked_pairs(Lq, Lk, mask):
    """Number of (query, key) pairs of one sequence that a 128 x 128 block mask
    keeps (rows and columns of the last block clipped to the sequence)."""
    rows = np.minimum(128, Lq - 128 * np.arange(-(-Lq // 128)))
    cols = np.minimum(128, Lk - 128 * np.arange(-(-Lk // 128)))
    return int(rows @ np.asarray(mask, dtype=np.int64) @ cols) if rows.size and cols.size else 0


def useful_flops(name_or_kind, lengths=None, H=None, D=None, Lq=None, B=None, L=None, block=64,
                 window=(-1, -1), masks=None):
    """Useful (unpadded) forward FLOPs: 4 * H * D * sum_b Lq_b * Lk_b.

    The backward counts 2.5x this (five contractions against two).
    """
    if name_or_kind == "jagged":
        return 4.0 * H * D * float(np.sum(np.asarray(lengths, dtype=np.float64) ** 2))
    if name_or_kind == "varlen":  # self-attention lengths with a band mask
        return 4.0 * H * D * float(sum(visible_pairs(int(n), int(n), window) for n in lengths))
    if name_or_kind == "cross":  # separate query and key/value lengths, no mask
        return 4.0 * H * D * float(np.dot(np.asarray(lengths[0], np.float64), np.asarray(lengths[1], np.float64)))
    if name_or_kind == "sparse":  # self-attention lengths with block masks
        return 4.0 * H * D * float(sum(masked_pairs(int(n), int(n), m) for n, m in zip(lengths, masks)))
    if name_or_kind == "bcast":
        return 4.0 * H * D * Lq * float(np.sum(lengths))
    if name_or_kind == "blockdiag":
        return 4.0 * H * D * B * L * block
    raise KeyError(name_or_kind)
