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
