"""Sparse main-branch attention over the selected blocks -- TEST INFRASTRUCTURE ONLY.

Same rules as the rest of ``oracle/``: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg may import it; the product library never does.

What it computes (MiniMax Sparse Attention notes, "MiniMax Sparse Attention:
paper algorithm and exact code correspondence", section 4.8 Equation (8): the
main branch's softmax restricted to the blocks the index branch selected,
shared by the heads of a GQA group, section 4.3 Equation (3)):

    O[t, h]   = sum_{j in S} softmax_j(s_j) * V[j, r]
    LSE[t, h] = log sum_{j in S} exp(s_j)
    s_j       = sm_scale * < Q[t, h], K[j, r] >,   r = h // g

where S holds the keys j of the blocks listed in ``sel[t, r, :]`` (logical
block indices of the token's request; -1 entries and blocks at or beyond
ceil(kv_len / P) are ignored) that are visible to t: j < kv_len and, for
sparse_mode 3, j <= q_pos = kv_len - Lq + i (the rightDownCausal alignment of
the block-score op).  ``sm_scale`` defaults to 1 / sqrt(D) (Equation (8)).

Readings (listed in the design notes): a token with no visible key in its
selected blocks gets O = 0 and LSE = -inf; the keys and values share one paged
(or packed) layout and one block table.

Written as the definition: for each (t, h), gather the visible keys of the
selected blocks, form the scores, and apply a plain softmax, all in float64
with numpy; no two-phase split, no blocking.  Only meant for small inputs or
sampled rows.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np
import torch


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def _key_rows(case, cache: torch.Tensor, b: int, js: np.ndarray, r: int) -> np.ndarray:
    """Rows of `cache` (same layout as case.key) at logical positions js of request b, head r."""
    layout = case.layout.upper()
    P = case.P
    if layout == "TND":
        base = int(case.cu_seqlens_k[b])
        return _f64(cache[torch.as_tensor(base + js), r])
    pages = case.block_table[b, torch.as_tensor(js // P)].to(torch.int64)
    off = torch.as_tensor(js % P)
    if layout == "BBND":
        return _f64(cache[pages, off, r])
    return _f64(cache[pages, r, off])                     # BNBD


def sparse_attention(case, value: torch.Tensor, sel: torch.Tensor,
                     sm_scale: Optional[float] = None, rows: Optional[Sequence[int]] = None):
    """O float64 ``[T, H_q, D]`` and LSE float64 ``[T, H_q]``.

    ``value`` has the key cache's layout and shape; ``sel`` is int ``[T, H_kv, k]``.
    ``rows`` (optional) limits the work to the flat rows ``t * H_q + h``; the
    others stay O = 0, LSE = nan.
    """
    T, H_q, D = case.T, case.H_q, case.D
    g = H_q // case.H_kv
    P, MB = case.P, case.MB
    scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    q = _f64(case.query)
    sel = sel.detach().cpu().to(torch.int64).numpy()
    O = np.zeros((T, H_q, D))
    LSE = np.full((T, H_q), np.nan)
    cu = case.cu_seqlens_q.tolist()
    req = np.zeros(T, dtype=np.int64)
    for b in range(len(cu) - 1):
        req[cu[b]:cu[b + 1]] = b
    todo = range(T * H_q) if rows is None else rows
    for flat in todo:
        t, h = divmod(int(flat), H_q)
        b = int(req[t])
        r = h // g
        Lq = cu[b + 1] - cu[b]
        if case.layout.upper() == "TND":
            L = int(case.cu_seqlens_k[b + 1] - case.cu_seqlens_k[b])
        else:
            L = int(case.kv_len[b])
        qpos = L - Lq + (t - cu[b])
        nb = -(-L // P)
        js = []
        for beta in sel[t, r]:
            if beta < 0 or beta >= MB or beta >= nb:
                continue
            for j in range(beta * P, beta * P + P):
                if j < L and (case.sparse_mode != 3 or j <= qpos):
                    js.append(j)
        if not js:
            O[t, h] = 0.0
            LSE[t, h] = -np.inf
            continue
        js = np.asarray(js, dtype=np.int64)
        kk = _key_rows(case, case.key, b, js, r)          # [n, D]
        vv = _key_rows(case, value, b, js, r)
        s = scale * (kk @ q[t, h])
        m = s.max()
        w = np.exp(s - m)
        O[t, h] = (w[:, None] * vv).sum(axis=0) / w.sum()
        LSE[t, h] = m + math.log(w.sum())
    return O, LSE
