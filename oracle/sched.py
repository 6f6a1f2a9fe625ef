"""Plain-Python oracle of the host tile scheduler (LPT sort + zigzag deal).

TEST INFRASTRUCTURE ONLY (see the package docstring).

[JFA-GEM] "Optimizaciones específicas para el flujo de trabajo de GEM" and
[PT-TLX] "Kevesebb kód, nagyobb teljesítmény": on the host, all tiles are
sorted by their KV workload in descending order and dealt to the SMs in a
zigzag (boustrophedon) pattern: even passes fill the SMs left to right, odd
passes right to left.

Readings where the pages are silent:

* a tile is (b, h, m): sequence b, head h, row block m of `tile_rows` rows;
  sequence b has ceil(rows_b / tile_rows) row blocks;
* rows_b is the sequence length unless `fixed_rows` > 0 (broadcast-Q forward
  tiles the dense Q of fixed length); work_b is the sequence length unless
  `fixed_work` > 0 (broadcast-Q backward: every KV tile walks the same Lq);
* the sort is stable, so equal-work tiles keep the enumeration order
  b, then h, then m;
* position i of the sorted list goes to pass p = i // S, slot j = i % S and
  SM j on even p, SM S-1-j on odd p;
* the "naive" order used as the A/B baseline deals the unsorted tiles
  round-robin (SM i % S).

Output is CSR: ``sm_ptr[S+1]`` and ``tiles`` as a list of (b, h, m), each
SM's tiles in the order they were dealt.

Masked and cross (varlen) attention (the band mask of ``oracle.attention``:
query i sees key j iff j - i - (Lk - Lq) lies in [-left, right], -1 meaning
unbounded) reuse the same sort and deal; only a tile's rows and work change:

* forward tile (b, h, m) covers query rows [256 m, min(Lq, 256 m + 256)) and
  its work is the length of the key range those rows can see,
  [max(0, r0 + shift - left), min(Lk, r1 - 1 + shift + right + 1)), or 0 when
  that range is empty (the tile still runs: its rows get O = 0);
* backward tile (b, h, n) covers keys [128 n, min(Lk, 128 n + 128)) and its
  work is the number of query rows that can see them,
  [max(0, k0 - shift - right), min(Lq, k1 - 1 - shift + left + 1)), or 0
  (the tile still runs: its keys get dK = dV = 0).

Without a mask and with equal offsets this is the jagged schedule above.
"""

import numpy as np


def enumerate_tiles(lengths, H, tile_rows, fixed_rows=0, fixed_work=0):
    """All tiles in enumeration order, each as (b, h, m, work)."""
    out = []
    for b, L in enumerate(lengths):
        rows = fixed_rows if fixed_rows > 0 else L
        work = fixed_work if fixed_work > 0 else L
        n_m = -(-rows // tile_rows)
        for h in range(H):
            for m in range(n_m):
                out.append((b, h, m, work))
    return out


def schedule(lengths, H, tile_rows, num_sms, fixed_rows=0, fixed_work=0, zigzag=True):
    """Returns (sm_ptr, tiles) as plain Python lists."""
    tiles = enumerate_tiles(lengths, H, tile_rows, fixed_rows, fixed_work)
    if zigzag:
        order = sorted(range(len(tiles)), key=lambda i: -tiles[i][3])  # stable
    else:
        order = list(range(len(tiles)))
    per_sm = [[] for _ in range(num_sms)]
    for i, t in enumerate(order):
        p, j = divmod(i, num_sms)
        sm = j if (not zigzag or p % 2 == 0) else num_sms - 1 - j
        per_sm[sm].append(tiles[t][:3])
    sm_ptr = [0]
    flat = []
    for lst in per_sm:
        flat.extend(lst)
        sm_ptr.append(len(flat))
    return sm_ptr, flat


def makespan(sm_ptr, tiles, lengths, fixed_work=0):
    """Largest per-SM sum of tile work (the quantity LPT balances)."""
    best = 0
    for s in range(len(sm_ptr) - 1):
        tot = 0
        for (b, _h, _m) in tiles[sm_ptr[s]:sm_ptr[s + 1]]:
            tot += fixed_work if fixed_work > 0 else lengths[b]
        best = max(best, tot)
    return best


FWD_ROWS, BWD_ROWS = 256, 128


def fwd_key_range(r0, r1, Lq, Lk, window):
    """Keys [lo, hi) that query rows [r0, r1) can see under the band mask."""
    left, right = window
    shift = Lk - Lq
    lo = 0 if left < 0 else max(0, r0 + shift - left)
    hi = Lk if right < 0 else min(Lk, r1 - 1 + shift + right + 1)
    return lo, max(lo, hi)


def bwd_query_range(k0, k1, Lq, Lk, window):
    """Query rows [lo, hi) that can see some key of [k0, k1) under the band mask."""
    left, right = window
    shift = Lk - Lq
    lo = 0 if right < 0 else max(0, k0 - shift - right)
    hi = Lq if left < 0 else min(Lq, k1 - 1 - shift + left + 1)
    return lo, max(lo, hi)


def enumerate_varlen_tiles(q_lengths, kv_lengths, H, op, window=(-1, -1)):
    """Tiles (b, h, m, work) of the masked / cross attention forward
    (op = "fwd") or backward (op = "bwd"), in enumeration order."""
    out = []
    for b, (Lq, Lk) in enumerate(zip(q_lengths, kv_lengths)):
        if op == "fwd":
            n_m = -(-Lq // FWD_ROWS)
            works = []
            for m in range(n_m):
                r0, r1 = m * FWD_ROWS, min(Lq, m * FWD_ROWS + FWD_ROWS)
                lo, hi = fwd_key_range(r0, r1, Lq, Lk, window)
                works.append(hi - lo)
        else:
            n_m = -(-Lk // BWD_ROWS)
            works = []
            for n in range(n_m):
                k0, k1 = n * BWD_ROWS, min(Lk, n * BWD_ROWS + BWD_ROWS)
                lo, hi = bwd_query_range(k0, k1, Lq, Lk, window)
                works.append(hi - lo)
        for h in range(H):
            for m in range(n_m):
                out.append((b, h, m, works[m]))
    return out


def schedule_varlen(q_lengths, kv_lengths, H, op, num_sms, window=(-1, -1), zigzag=True):
    """LPT + zigzag (or naive) deal of the varlen tiles. Returns (sm_ptr, tiles)."""
    return _deal(enumerate_varlen_tiles(q_lengths, kv_lengths, H, op, window), num_sms, zigzag)


def _deal(tiles, num_sms, zigzag):
    if zigzag:
        order = sorted(range(len(tiles)), key=lambda i: -tiles[i][3])  # stable
    else:
        order = list(range(len(tiles)))
    per_sm = [[] for _ in range(num_sms)]
    for i, t in enumerate(order):
        p, j = divmod(i, num_sms)
        sm = j if (not zigzag or p % 2 == 0) else num_sms - 1 - j
        per_sm[sm].append(tiles[t][:3])
    sm_ptr = [0]
    flat = []
    for lst in per_sm:
        flat.extend(lst)
        sm_ptr.append(len(flat))
    return sm_ptr, flat


# ----------------------------------------------------------- block-sparse masks
# Tiles of block-sparse attention (masks[b] [ceil(Lq/128), ceil(Lk/128)] of
# oracle.attention.block_visible) and the lists the kernels walk:
#
# * forward tile (b, h, m): query blocks 2m and 2m+1 (its two 128-row
#   halves); it walks the union of the key blocks either half sees, in
#   increasing order, each entry with a bit per half; its work is the number
#   of keys in those blocks;
# * backward tile (b, h, n): key block n; it walks the 64-row query blocks qb
#   (in increasing order) whose 128-row block qb // 2 sees it; its work is the
#   number of query rows in them.


def sparse_tiles(q_lengths, kv_lengths, H, op, masks):
    """(b, h, m, work, entries) in enumeration order; entries are
    (key block, sees0, sees1) for the forward, query blocks for the backward."""
    out = []
    for b, (Lq, Lk) in enumerate(zip(q_lengths, kv_lengths)):
        mask = np.asarray(masks[b], dtype=bool)
        nqb, nkb = -(-Lq // 128), -(-Lk // 128)
        if op == "fwd":
            n_m = -(-Lq // FWD_ROWS)
            per = []
            for m in range(n_m):
                ent = []
                for j in range(nkb):
                    s0 = bool(mask[2 * m, j]) if 2 * m < nqb else False
                    s1 = bool(mask[2 * m + 1, j]) if 2 * m + 1 < nqb else False
                    if s0 or s1:
                        ent.append((j, s0, s1))
                work = sum(min(Lk, 128 * j + 128) - 128 * j for j, _, _ in ent)
                per.append((work, ent))
        else:
            n_m = nkb
            per = []
            for n in range(n_m):
                ent = [qb for qb in range(-(-Lq // 64)) if mask[qb // 2, n]]
                work = sum(min(Lq, 64 * qb + 64) - 64 * qb for qb in ent)
                per.append((work, ent))
        for h in range(H):
            for m in range(n_m):
                out.append((b, h, m, per[m][0], per[m][1]))
    return out


def schedule_sparse(q_lengths, kv_lengths, H, op, num_sms, masks, zigzag=True):
    """LPT + zigzag deal of the block-sparse tiles. Returns (sm_ptr, tiles,
    lists): lists[i] are the entries of dealt tile i."""
    tiles = sparse_tiles(q_lengths, kv_lengths, H, op, masks)
    sm_ptr, flat = _deal([t[:4] for t in tiles], num_sms, zigzag)
    key = {t[:3]: t[4] for t in tiles}
    return sm_ptr, flat, [key[tuple(t)] for t in flat]
