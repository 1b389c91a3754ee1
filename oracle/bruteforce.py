"""Second, independent formulation of the block score -- TEST INFRASTRUCTURE ONLY.

It follows the mask-then-block-max definition in the "DSA / GQA forward"
notes (notes.kuangjux.top, section 3 "from token score to block selection"):
build the dense token-score matrix of each request, replace every invisible
position by -inf, reshape the key axis into blocks of P and take ``amax``.
The int8 case dequantises the keys first (k~ = cast(k) * scale, as the
"MsaIndexScore" feature request writes k~), which is the other side of the
identity Q.(K s) = (Q.cast K) s that the C oracle uses.  FP4 cases (E2M1
codes with E8M0 / E4M3 group scales) are dequantised here by a value table and
torch's decoding of the scale bytes, independently of the C oracle's decoders.

Everything is numpy float64; only meant for tiny inputs.  The local mask of
the torch API guide (sec. 2) is applied afterwards.  Returns float64 so the
caller can compare before the final rounding.
"""
from __future__ import annotations

import numpy as np
import torch


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


# FP4 E2M1 magnitudes by the 3 low bits of a code (OCP Microscaling formats:
# 1 sign, 2 exponent bits with bias 1, 1 mantissa bit; no infinities or NaN)
_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _fp4_dequant(packed: torch.Tensor, scales: torch.Tensor, fmt: str) -> np.ndarray:
    """Packed E2M1 rows [..., D/2] with group scales [..., D/G] -> float64 [..., D].

    The scale bytes are decoded by torch (E8M0 for MXFP4, E4M3 for NVFP4)."""
    b = packed.detach().cpu().numpy().astype(np.int64)
    codes = np.stack([b & 15, b >> 4], axis=-1).reshape(*b.shape[:-1], 2 * b.shape[-1])
    vals = np.where(codes & 8, -1.0, 1.0) * _E2M1[codes & 7]
    sdt = torch.float8_e8m0fnu if fmt == "mx" else torch.float8_e4m3fn
    sc = scales.detach().cpu().view(sdt).to(torch.float64).numpy()
    G = 32 if fmt == "mx" else 16
    return vals * np.repeat(sc, G, axis=-1)


def _gather_keys(case, b: int, L: int, NB: int) -> np.ndarray:
    """Dequantised keys of request b by logical position: [NB*P, H_kv, D] (rows >= L zero)."""
    P = case.P
    key = case.key
    layout = case.layout.upper()
    H_kv = case.H_kv
    D = case.D
    dense = np.zeros((max(NB, 0) * P, H_kv, D), dtype=np.float64)
    if L == 0:
        return dense
    fp4 = getattr(case, "fp4", None)
    if fp4:
        # dequantise first: E2M1 values times their group scales
        if layout == "TND":
            lo = int(case.cu_seqlens_k[b])
            dense[:L] = _fp4_dequant(key[lo:lo + L], case.k_scale[lo:lo + L], fp4)
            return dense
        for beta in range(NB):
            page = int(case.block_table[b, beta])
            blk = key[page]                                # BBND [P,H,D/2] / BNBD [H,P,D/2]
            if layout == "BNBD":
                blk = blk.transpose(0, 1)
            dq = _fp4_dequant(blk, case.k_scale[page].transpose(0, 1), fp4)   # scales [H,P,G] -> [P,H,G]
            dense[beta * P:(beta + 1) * P] = dq
        dense[L:] = 0.0
        return dense
    if layout == "TND":
        lo = int(case.cu_seqlens_k[b])
        rows = _f64(key[lo:lo + L])                         # [L, H_kv, D]
        if case.scale is not None:
            rows = rows * _f64(case.scale[lo:lo + L])[:, :, None]
        dense[:L] = rows
        return dense
    for beta in range(NB):
        page = int(case.block_table[b, beta])
        blk = key[page]                                    # BBND [P,H,D] / BNBD [H,P,D]
        if layout == "BNBD":
            blk = blk.transpose(0, 1)
        blk = _f64(blk)
        if case.scale is not None:
            blk = blk * _f64(case.scale[page]).T[:, :, None]   # scale [H,P] -> [P,H,1]
        dense[beta * P:(beta + 1) * P] = blk
    dense[L:] = 0.0
    return dense


def block_scores(case, fill_value: float = float("-inf")) -> np.ndarray:
    """Dense-then-amax block scores, float64 ``[H_q, T, RoundUp(MB,16)]``."""
    P = case.P
    H_q, T, MB = case.H_q, case.T, case.MB
    MBp = (MB + 15) // 16 * 16
    g = H_q // case.H_kv
    out = np.full((H_q, T, MBp), fill_value, dtype=np.float64)
    if getattr(case, "fp4", None):
        q_all = _fp4_dequant(case.query, case.q_scale, case.fp4)   # [T, H_q, D]
    else:
        q_all = _f64(case.query)                            # [T, H_q, D]
    cu = case.cu_seqlens_q.tolist()
    layout = case.layout.upper()
    for b in range(len(cu) - 1):
        t0, t1 = cu[b], cu[b + 1]
        Lq = t1 - t0
        if Lq == 0:
            continue
        if layout == "TND":
            L = int(case.cu_seqlens_k[b + 1] - case.cu_seqlens_k[b])
        else:
            L = int(case.kv_len[b])
        NB = -(-L // P)
        keys = _gather_keys(case, b, L, min(NB, MB))        # [nb*P, H_kv, D]
        nb_cols = keys.shape[0] // P
        # dense token scores r[i, h, j]
        kh = keys[:, np.arange(H_q) // g, :]                # [nbP, H_q, D]
        r = np.einsum("ihd,jhd->ihj", q_all[t0:t1], kh)     # [Lq, H_q, nbP]
        j = np.arange(nb_cols * P)[None, :]
        i = np.arange(Lq)[:, None]
        visible = j < L
        if case.sparse_mode == 3:
            visible = visible & (j <= (L - Lq + i))
        r = np.where(visible[:, None, :], r, -np.inf)
        blk = r.reshape(Lq, H_q, nb_cols, P).max(axis=-1) if nb_cols else \
            np.zeros((Lq, H_q, 0))
        blk = np.where(np.isneginf(blk), fill_value, blk)
        res = np.full((Lq, H_q, MBp), fill_value, dtype=np.float64)
        res[:, :, :nb_cols] = blk
        if L > 0 and (case.init_blocks > 0 or case.local_blocks > 0):
            res[:, :, :min(case.init_blocks, MB)] = 1e30
            sl = int(case.start_loc[b])
            lo = max(0, sl + 1 - case.local_blocks)
            hi = min(sl, MB - 1)
            if hi >= lo:
                res[:, :, lo:hi + 1] = 1e29
        out[:, t0:t1, :] = res.transpose(1, 0, 2)
    return out
