"""Split-KV work partition, restated in plain Python (test infrastructure).

STAGE_D2.md ("Grid vs. Persistent Tile Scheduler") notes that a static grid
is enough for fixed-length decode but that variable sequence lengths want a
persistent scheduler that balances work over a fixed set of workers.  The
pages fix no rule, so this is the rule the library states and implements on
the GPU; this file writes it out one item and one part at a time so that the
device result can be compared with it integer for integer.

Rule
----
Work items.  The query rows of one sequence are packed head-fastest, row
r = t*H + h (STAGE_D2.md "Strategy A": heads folded into M; row order token
major).  Dense/causal: the rows of sequence b are cut into M tiles of up to
128 rows, item = (b, m_tile), ordered m-tile-major (item m_tile * B + b):
the M tiles of a sequence share its keys, and in this order the cost line
holds all first M tiles, then all second ones, so the parts that hold the
same tile range of a sequence's M tiles run at the same time and each page
comes from HBM once.  Top-k: each query token has its own key set, so
item = (b, t) with H rows, ordered b-major.

Key tiles.  An item's keys are cut into 64-key tiles (one 64-token page):
  dense   ceil(s_k / 64)
  causal  ceil(k / 64), k = clamp(s_k - T + t_last + 1, 0, s_k) where t_last
          is the last query token among the item's rows
  top-k   ceil(topk / 64)

Cost line.  Item i occupies the interval [C_i, C_i + F + n_i) of a line,
C_0 = 0, C_{i+1} = C_i + F + n_i, where F = FIXED_COST stands for the
per-item set-up (query load, epilogue).  Tile k of item i sits at coordinate
C_i + F + k.  With W = C_{items}, P parts and L = ceil(W / P), part p owns
the coordinates [p*L, min((p+1)*L, W)): every tile has exactly one owner, an
item's tiles go to consecutive parts, and an item without tiles (s_k = 0) is
owned by the part that owns its start C_i.

Outputs.
  tile_md[p] = (begin_item, begin_tile, last_item, end_tile, first_piece,
                begin_at_start, 0, 0)
      The part processes items begin_item..last_item; item begin_item from
      tile begin_tile, item last_item up to end_tile (exclusive), others in
      full.  first_piece = the index, among the parts that share it, of this
      part's piece of begin_item.  begin_at_start = 1 when p*L == C_begin
      (then an empty begin_item belongs to this part).  A part with no work
      has begin_item = items, last_item = items - 1.
  num_splits[i] = exclusive prefix over items of the number of parts that
      process item i (1 for an item without tiles); length items + 1.
"""
from __future__ import annotations

FIXED_COST = 4
TILE = 64
M_TILE = 128


def item_list(seqlens, H: int, T: int, topk: int = 0, causal: bool = False):
    """[(b, row_begin, row_count, n_tiles)] in schedule order."""
    items = []
    if topk > 0:
        for b in range(len(seqlens)):
            for t in range(T):
                items.append((b, t * H, H, -(-topk // TILE)))
        return items
    rows = T * H
    for r0 in range(0, rows, M_TILE):
        for b, sk in enumerate(seqlens):
            sk = int(sk)
            cnt = min(M_TILE, rows - r0)
            if causal:
                t_last = (r0 + cnt - 1) // H
                k = min(max(sk - T + t_last + 1, 0), sk)
            else:
                k = sk
            items.append((b, r0, cnt, -(-k // TILE)))
    return items


def schedule(seqlens, H: int, T: int, num_parts: int, topk: int = 0,
             causal: bool = False):
    """Returns (tile_md: list of 8-int lists, num_splits: list of ints)."""
    items = item_list(seqlens, H, T, topk, causal)
    n_items = len(items)
    ntiles = [it[3] for it in items]
    C = [0]
    for n in ntiles:
        C.append(C[-1] + FIXED_COST + n)
    W = C[-1]
    P = num_parts
    L = -(-W // P)

    def item_at(x):
        """Index i with C[i] <= x < C[i+1] (plain scan)."""
        for i in range(n_items):
            if C[i] <= x < C[i + 1]:
                return i
        raise AssertionError("coordinate outside the line")

    def clamp(v, lo, hi):
        return max(lo, min(v, hi))

    def owner(x):
        return x // L

    tile_md = []
    for p in range(P):
        lo = p * L
        hi = min((p + 1) * L, W)
        if lo >= W:
            tile_md.append([n_items, 0, n_items - 1, 0, 0, 0, 0, 0])
            continue
        a = item_at(lo)
        z = item_at(hi - 1)
        begin_tile = clamp(lo - C[a] - FIXED_COST, 0, ntiles[a])
        end_tile = clamp(hi - C[z] - FIXED_COST, 0, ntiles[z])
        first_piece = 0
        if ntiles[a] > 0:
            first_piece = p - owner(C[a] + FIXED_COST)
            if first_piece < 0:
                first_piece = 0
        tile_md.append([a, begin_tile, z, end_tile, first_piece,
                        1 if C[a] == lo else 0, 0, 0])

    num_splits = [0]
    for i in range(n_items):
        if ntiles[i] == 0:
            n = 1
        else:
            n = owner(C[i] + FIXED_COST + ntiles[i] - 1) - owner(C[i] + FIXED_COST) + 1
        num_splits.append(num_splits[-1] + n)
    return tile_md, num_splits


def pieces(tile_md, items):
    """Expand tile_md into the pieces each part processes:
    [(part, item, tile_begin, tile_end, piece_index)] (tile_end exclusive);
    a piece with tile_begin == tile_end is an item without tiles."""
    out = []
    for p, md in enumerate(tile_md):
        a, bt, z, et, fp, at_start = md[:6]
        for i in range(a, z + 1):
            n = items[i][3]
            t0 = bt if i == a else 0
            t1 = et if i == z else n
            if n == 0:
                if i > a or at_start:
                    out.append((p, i, 0, 0, 0))
                continue
            if t1 > t0:
                out.append((p, i, t0, t1, fp if i == a else 0))
    return out
