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
"""


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
