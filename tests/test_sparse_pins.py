"""Pins for the sparse main-branch oracle (no GPU).

oracle/sparse_attention.py follows the MiniMax Sparse Attention notes,
section 4.8 Equation (8) (softmax restricted to the selected blocks, GQA
groups sharing one selection, section 4.3 Equation (3)).  It is checked
against things other than itself:
  * torch's scaled_dot_product_attention (float64, explicit causal mask) when
    every block is selected: the restricted softmax is then plain attention
    (paged and packed keys; the default scale against torch's default);
  * a hand-worked example (P = 2, D = 2) in tests/golden/;
  * closed forms: one visible key gives O = v_j and LSE = s_j;
  * invariants: keys and values of blocks that are not selected, or of
    positions that are not visible, never matter; -1 entries are ignored.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle.sparse_attention import sparse_attention
from synth import make_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sparse_attention_hand_example.json")


def _value_like(case, seed):
    g = torch.Generator().manual_seed(seed)
    base = case.key
    return torch.randn(base.shape, generator=g, dtype=torch.float32).to(base.dtype)


def _all_blocks(case, k):
    T = case.T
    sel = torch.full((T, case.H_kv, k), -1, dtype=torch.int32)
    cu = case.cu_seqlens_q.tolist()
    for b in range(case.B):
        nb = -(-case.kv_lens[b] // case.P)
        for t in range(cu[b], cu[b + 1]):
            sel[t, :, :nb] = torch.arange(nb, dtype=torch.int32)
    return sel


def _dense(case, value, b):
    """Keys and values of request b by logical position, float64 [L, H_kv, D]."""
    L, P = case.kv_lens[b], case.P
    if case.layout == "TND":                               # packed rows from cu_seqlens_k[b]
        lo = int(case.cu_seqlens_k[b])
        return case.key[lo:lo + L].double(), value[lo:lo + L].double()
    ks, vs = [], []
    for j in range(L):
        page = int(case.block_table[b, j // P])
        off = j % P
        if case.layout == "BBND":
            ks.append(case.key[page, off]); vs.append(value[page, off])
        else:
            ks.append(case.key[page, :, off]); vs.append(value[page, :, off])
    return torch.stack(ks).double(), torch.stack(vs).double()


@pytest.mark.parametrize("layout", ["BBND", "BNBD", "TND"])
@pytest.mark.parametrize("mode", [3, 0])
def test_full_selection_is_plain_attention(layout, mode):
    case = make_case([5, 3, 1], [9, 20, 7], H_q=4, H_kv=2, P=4, D=8, layout=layout,
                     q_dtype=torch.bfloat16, MB=6, sparse_mode=mode, seed=70 + mode)
    value = _value_like(case, 71)
    O, LSE = sparse_attention(case, value, _all_blocks(case, 6), sm_scale=0.3)
    g = case.H_q // case.H_kv
    cu = case.cu_seqlens_q.tolist()
    for b in range(case.B):
        k, v = _dense(case, value, b)                     # [L, H_kv, D]
        q = case.query[cu[b]:cu[b + 1]].double()          # [Lq, H_q, D]
        Lq, L = q.shape[0], k.shape[0]
        kh = k[:, torch.arange(case.H_q) // g].permute(1, 0, 2)   # [H_q, L, D]
        vh = v[:, torch.arange(case.H_q) // g].permute(1, 0, 2)
        mask = torch.ones(Lq, L, dtype=torch.bool)
        if mode == 3:
            i = torch.arange(Lq)[:, None]
            j = torch.arange(L)[None, :]
            mask = j <= (L - Lq + i)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.permute(1, 0, 2), kh, vh, attn_mask=mask, scale=0.3)    # [H_q, Lq, D]
        scores = torch.einsum("hid,hjd->hij", q.permute(1, 0, 2), kh) * 0.3
        lse = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)   # [H_q, Lq]
        np.testing.assert_allclose(O[cu[b]:cu[b + 1]], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(LSE[cu[b]:cu[b + 1]], lse.T.numpy(), rtol=1e-12, atol=1e-12)


def test_default_scale_is_torchs_default():
    # sm_scale omitted: Equation (8)'s 1/sqrt(D), which is also the default of
    # torch's scaled_dot_product_attention
    case = make_case([4, 2], [11, 6], H_q=2, H_kv=1, P=4, D=16, layout="BBND",
                     q_dtype=torch.bfloat16, MB=3, sparse_mode=3, seed=78)
    value = _value_like(case, 79)
    O, _ = sparse_attention(case, value, _all_blocks(case, 3))
    cu = case.cu_seqlens_q.tolist()
    for b in range(case.B):
        k, v = _dense(case, value, b)
        q = case.query[cu[b]:cu[b + 1]].double().permute(1, 0, 2)   # [H_q, Lq, D]
        Lq, L = q.shape[1], k.shape[0]
        mask = torch.arange(L)[None, :] <= (L - Lq + torch.arange(Lq)[:, None])
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, k.permute(1, 0, 2).expand(2, L, 16), v.permute(1, 0, 2).expand(2, L, 16),
            attn_mask=mask)
        np.testing.assert_allclose(O[cu[b]:cu[b + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=1e-12, atol=1e-12)


def test_hand_example():
    spec = json.load(open(GOLDEN))
    case = make_case([1], [4], H_q=1, H_kv=1, P=2, D=2, layout="BBND", q_dtype=torch.bfloat16,
                     MB=2, permute_pages=False, sparse_mode=3, seed=0)
    case.query[0, 0] = torch.tensor(spec["q"], dtype=torch.bfloat16)
    value = torch.zeros_like(case.key)
    for j, (kr, vr) in enumerate(zip(spec["k"], spec["v"])):
        case.key[j // 2, j % 2, 0] = torch.tensor(kr, dtype=torch.bfloat16)
        value[j // 2, j % 2, 0] = torch.tensor(vr, dtype=torch.bfloat16)
    for name, sel in spec["selections"].items():
        O, LSE = sparse_attention(case, value, torch.tensor([[sel["blocks"]]], dtype=torch.int32),
                                  sm_scale=spec["sm_scale"])
        np.testing.assert_allclose(O[0, 0], sel["O"], rtol=1e-12, atol=1e-12, err_msg=name)
        np.testing.assert_allclose(LSE[0, 0], sel["LSE"], rtol=1e-12, atol=1e-12, err_msg=name)


def test_single_visible_key():
    # kv_len 1: the selected block holds one visible key
    case = make_case([1], [1], H_q=2, H_kv=1, P=4, D=8, layout="BNBD", q_dtype=torch.bfloat16,
                     MB=1, seed=72)
    value = _value_like(case, 73)
    O, LSE = sparse_attention(case, value, torch.tensor([[[0]]], dtype=torch.int32), sm_scale=0.5)
    page = int(case.block_table[0, 0])
    for h in range(2):
        k = case.key[page, 0, 0].double()
        v = value[page, 0, 0].double()
        assert np.allclose(O[0, h], v.numpy(), rtol=0, atol=1e-15)
        assert math.isclose(LSE[0, h], 0.5 * float(case.query[0, h].double() @ k), rel_tol=1e-14)


def test_invisible_and_unselected_keys_never_matter():
    case = make_case([6, 2], [40, 33], H_q=4, H_kv=2, P=8, D=8, layout="BBND",
                     q_dtype=torch.bfloat16, MB=5, seed=74)
    value = _value_like(case, 75)
    sel = torch.tensor([[[0, 2, -1], [1, 3, 4]]] * 8, dtype=torch.int32)
    O, LSE = sparse_attention(case, value, sel)
    # poison every key / value that is not in a selected block or not visible
    k2, v2 = case.key.clone(), value.clone()
    cu = case.cu_seqlens_q.tolist()
    for b in range(case.B):
        L, Lq = case.kv_lens[b], case.q_lens[b]
        first = L - Lq                                     # the earliest query's position
        for j in range(case.MB * case.P):
            beta = j // case.P
            page = int(case.block_table[b, beta]) if beta < -(-L // case.P) else None
            if page is None:
                continue
            for r in range(2):
                chosen = beta in sel[cu[b], r].tolist()
                if not chosen or j >= L:
                    k2[page, j % case.P, r] = 1e4
                    v2[page, j % case.P, r] = -1e4
    import dataclasses
    O2, LSE2 = sparse_attention(dataclasses.replace(case, key=k2), v2, sel)
    assert np.array_equal(O, O2) and np.array_equal(LSE, LSE2)
    # -1 entries and blocks past the request's last block are ignored
    sel3 = sel.clone()
    sel3[:, 0, 2] = 9
    O3, _ = sparse_attention(case, value, sel3)
    assert np.array_equal(O, O3)


def test_empty_selection_gives_zero_and_minus_inf():
    case = make_case([2], [50], H_q=2, H_kv=1, P=8, D=8, layout="BBND", q_dtype=torch.bfloat16,
                     MB=7, seed=76)
    value = _value_like(case, 77)
    O, LSE = sparse_attention(case, value, torch.full((2, 1, 4), -1, dtype=torch.int32))
    assert np.all(O == 0) and np.all(np.isneginf(LSE))


def test_row_subset_computes_the_listed_rows_only():
    # rows = flat t * H_q + h: those rows equal the full call's, the others stay O = 0, LSE = nan
    case = make_case([5, 3], [30, 12], H_q=4, H_kv=2, P=4, D=8, layout="BBND",
                     q_dtype=torch.bfloat16, MB=8, seed=80)
    value = _value_like(case, 81)
    sel = _all_blocks(case, 8)
    O, LSE = sparse_attention(case, value, sel)
    rows = [1, 14, 30]                                   # (t, h) = (0, 1), (3, 2), (7, 2)
    O2, LSE2 = sparse_attention(case, value, sel, rows=rows)
    for flat in range(case.T * case.H_q):
        t, h = divmod(flat, case.H_q)
        if flat in rows:
            assert np.array_equal(O2[t, h], O[t, h]) and LSE2[t, h] == LSE[t, h]
        else:
            assert np.all(O2[t, h] == 0) and np.isnan(LSE2[t, h])
