"""Block top-k selection -- TEST INFRASTRUCTURE ONLY.

Same rules as the rest of ``oracle/``: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg may import it; the product library never does.

What it computes (the MiniMax Sparse Attention notes, "MiniMax Sparse
Attention: paper algorithm and exact code correspondence", section 4.7,
Equation (7) TopK_b over a query's block scores, and the selector contract
quoted there and in section 5.3):

* input: block scores ``score[h, t, beta]`` as written by msa_index_score,
  fp32 ``[H, T, MBp]`` (one row per index head and query token);
* output: int32 ``[T, H, k]``: for each row, the k blocks with the highest
  score, listed by block index in ascending numeric order (not by score);
  rows with fewer than k valid blocks end in a tail of -1.

Readings where the pages are silent (listed in the design notes):

* a block is valid when ``beta < MB`` and its score is greater than -inf:
  -inf marks a block with no visible key, columns ``[MB, MBp)`` are
  padding, and a NaN score is never selected;
* equal scores are ranked by the smaller block index first;
* the forced blocks of the local mask need no special case: their scores
  (1e30 / 1e29) rank above every dot product, so they are kept whenever k is
  at least their number (section 4.7 asks for the query's local block to be
  in the selection; msa_index_score's local mask puts it there).

The selection is written as the definition: filter, sort by (score
descending, index ascending), cut at k, sort the cut by index.  A library
sort is the only primitive; no blocking or reordering beyond that.

Per-group selection (:func:`group_topk`), the same notes, section 4.3
(Equation (3): every query head of a GQA group uses the group's index set)
and the checklist of section 10 (items 7-9: one independent selection per
GQA group shared by its heads; each query's own block added and occupying a
slot; indices deduplicated, ascending, -1 only in the tail).  Readings where
the pages leave the step open (listed in the design notes):

* the group ranks blocks by its group score, the maximum over the group's g
  index heads of their block scores (the op computes one score row per index
  head; the paper's index branch has one index head per group, where this
  maximum is that head's own score);
* a query's own block is the block holding its position under the op's
  rightDownCausal alignment, ``q_pos = kv_len - Lq + i``; it exists when
  ``0 <= q_pos < kv_len`` (and its block is below MB).  With the local slot on,
  it is always selected and the other k - 1 slots take the best remaining
  blocks; without it the selection is the plain top-k of the group score.
"""
from __future__ import annotations

import numpy as np


def row_topk(row: np.ndarray, MB: int, k: int) -> np.ndarray:
    """Top-k block indices of one score row (ascending), -1 padded to k."""
    s = np.asarray(row, dtype=np.float32)[:MB]
    idx = np.arange(s.shape[0], dtype=np.int64)
    valid = s > np.float32(-np.inf)                 # False for -inf and NaN
    s, idx = s[valid], idx[valid]
    # primary key: score descending; secondary key: index ascending
    order = np.lexsort((idx, -s.astype(np.float64)))
    chosen = np.sort(idx[order[:k]])
    out = np.full(k, -1, dtype=np.int32)
    out[: chosen.shape[0]] = chosen
    return out


def block_topk(score, MB: int, k: int, rows=None) -> np.ndarray:
    """Selections for a whole score tensor ``[H, T, MBp]`` -> ``[T, H, k]``.

    ``rows`` (optional) limits the work to the listed flat rows ``h * T + t``;
    the others stay -1.
    """
    sc = score.detach().cpu().numpy() if hasattr(score, "detach") else np.asarray(score)
    H, T, _ = sc.shape
    out = np.full((T, H, k), -1, dtype=np.int32)
    it = range(H * T) if rows is None else rows
    for r in it:
        h, t = divmod(int(r), T)
        out[t, h] = row_topk(sc[h, t], MB, k)
    return out


def local_blocks_of(case) -> np.ndarray:
    """Each query token's own block (int64 ``[T]``, -1 where it has none)."""
    P, MB = int(case.P), int(case.MB)
    out = np.full(int(case.T), -1, dtype=np.int64)
    t = 0
    for Lq, L in zip(case.q_lens, case.kv_lens):
        for i in range(Lq):
            qpos = L - Lq + i
            if 0 <= qpos < L and qpos // P < MB:
                out[t + i] = qpos // P
        t += Lq
    return out


def group_topk(score, g: int, MB: int, k: int, local=None, rows=None) -> np.ndarray:
    """One selection per GQA group: ``[H, T, MBp]`` scores -> int32 ``[T, H // g, k]``.

    ``local`` (optional, ``[T]``): each token's own block (-1: none); when
    given, that block always takes one of the k slots.  ``rows`` (optional)
    limits the work to the flat rows ``r * T + t``; the others stay -1.
    """
    sc = score.detach().cpu().numpy() if hasattr(score, "detach") else np.asarray(score)
    H, T, MBp = sc.shape
    R = H // g
    gs = np.fmax.reduce(sc.reshape(R, g, T, MBp), axis=1)   # the group score: max over its heads
    out = np.full((T, R, k), -1, dtype=np.int32)
    it = range(R * T) if rows is None else rows
    for flat in it:
        r, t = divmod(int(flat), T)
        row = gs[r, t]
        loc = -1 if local is None else int(local[t])
        if loc < 0:
            out[t, r] = row_topk(row, MB, k)
            continue
        rest = np.array(row[:MB], dtype=np.float32, copy=True)
        rest[loc] = np.float32(-np.inf)              # the local block is not a candidate twice
        chosen = [c for c in row_topk(rest, MB, k - 1).tolist() if c >= 0] if k > 1 else []
        chosen = sorted(chosen + [loc])
        out[t, r, : len(chosen)] = chosen
    return out
