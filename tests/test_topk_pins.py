"""Pins for the block top-k oracle (no GPU).

Checked against things other than itself:
  * a hand-worked example (tests/golden/topk_hand_example.json) with ties,
    -inf, NaN, forced-block constants and a large value in a padding column,
  * torch.topk (an independent library routine) on rows without ties,
  * invariants the definition implies on rows full of ties: ascending order,
    the -1 tail, the count, the threshold property and the tie rule,
  * composition with the score oracle: the local mask's forced blocks are
    always selected when k covers them.

Definition: MiniMax Sparse Attention notes, section 4.7 (Equation (7) and
the selector contract) and section 5.3.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import topk as otk
from synth import make_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "topk_hand_example.json")


def _v(x):
    return {"-inf": -np.inf, "nan": np.nan}.get(x, x) if isinstance(x, str) else float(x)


def _golden():
    spec = json.load(open(GOLDEN))
    H, T, MB, MBp = spec["H"], spec["T"], spec["MB"], spec["MBp"]
    score = np.full((H, T, MBp), -np.inf, dtype=np.float32)
    for key, vals in spec["rows"].items():
        h, t = int(key[1]), int(key[3])
        score[h, t, :MB] = [_v(x) for x in vals]
    for key, cols in spec.get("padding_overrides", {}).items():
        h, t = int(key[1]), int(key[3])
        for c, v in cols.items():
            score[h, t, int(c)] = v
    return spec, score


def test_hand_example():
    spec, score = _golden()
    out = otk.block_topk(score, spec["MB"], spec["k"])
    assert out.shape == (spec["T"], spec["H"], spec["k"]) and out.dtype == np.int32
    for key, exp in spec["expect"].items():
        h, t = int(key[1]), int(key[3])
        assert out[t, h].tolist() == exp, key


@pytest.mark.parametrize("MB,k", [(1, 1), (7, 3), (64, 16), (300, 16), (1104, 32)])
def test_matches_torch_topk_without_ties(MB, k):
    g = torch.Generator().manual_seed(MB * 31 + k)
    H, T = 3, 5
    MBp = (MB + 15) // 16 * 16
    score = torch.full((H, T, MBp), float("-inf"))
    # distinct values: a random permutation of distinct floats per row
    for h in range(H):
        for t in range(T):
            score[h, t, :MB] = torch.randperm(MB, generator=g).float() * 0.5 - MB / 4
    out = otk.block_topk(score, MB, k)
    kk = min(k, MB)
    for h in range(H):
        for t in range(T):
            ref = torch.topk(score[h, t, :MB], kk).indices.sort().values.tolist()
            assert out[t, h, :kk].tolist() == ref
            assert (out[t, h, kk:] == -1).all()


@pytest.mark.parametrize("seed", range(6))
def test_invariants_with_ties(seed):
    rng = np.random.default_rng(seed)
    H, T, MB, k = 2, 7, int(rng.integers(1, 200)), int(rng.integers(1, 33))
    MBp = (MB + 15) // 16 * 16
    score = np.full((H, T, MBp), -np.inf, dtype=np.float32)
    score[:, :, :MB] = rng.integers(-3, 4, size=(H, T, MB)).astype(np.float32)   # many ties
    score[:, :, :MB][rng.random((H, T, MB)) < 0.3] = -np.inf
    score[:, :, MB:] = 1e30                                                       # padding must be ignored
    out = otk.block_topk(score, MB, k)
    for h in range(H):
        for t in range(T):
            row, sel = score[h, t, :MB], out[t, h]
            valid = np.nonzero(row > -np.inf)[0]
            n = min(k, valid.size)
            chosen = sel[:n]
            assert (sel[n:] == -1).all()
            assert (np.diff(chosen) > 0).all()                     # ascending, distinct
            assert set(chosen.tolist()) <= set(valid.tolist())
            if n and n < valid.size:
                rest = np.setdiff1d(valid, chosen)
                thr = row[chosen].min()
                assert row[rest].max() <= thr                       # threshold property
                tied_rest = rest[row[rest] == thr]
                tied_in = chosen[row[chosen] == thr]
                if tied_rest.size:
                    assert tied_in.max() < tied_rest.min()          # smaller index wins a tie


def test_forced_blocks_are_selected():
    case = make_case([3, 1], [1100, 700], H_q=4, H_kv=2, layout="BBND", q_dtype=torch.bfloat16,
                     MB=12, init_blocks=2, local_blocks=3, seed=7)
    score = oracle.oracle_full(case)
    H, T, MBp = score.shape
    out = otk.block_topk(score, case.MB, 8)
    for h in range(H):
        for t in range(T):
            row = score[h, t].numpy()
            forced = np.nonzero(row[: case.MB] >= 1e28)[0]
            assert forced.size and forced.size <= 8
            assert set(forced.tolist()) <= set(out[t, h].tolist())


# ---------------------------------------------------------------------------
# per-GQA-group selection (MiniMax Sparse Attention notes, section 4.3
# Equation (3), section 4.7 Equation (7), section 10 checklist items 7-9)

GROUP_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "group_topk_hand_example.json")


def _group_golden():
    spec = json.load(open(GROUP_GOLDEN))
    H, T, MB, MBp = spec["H"], spec["T"], spec["MB"], spec["MBp"]
    score = np.full((H, T, MBp), -np.inf, dtype=np.float32)
    for key, vals in spec["rows"].items():
        h, t = int(key[1]), int(key[3])
        score[h, t, :MB] = [_v(x) for x in vals]
    for key, cols in spec.get("padding_overrides", {}).items():
        h, t = int(key[1]), int(key[3])
        for c, v in cols.items():
            score[h, t, int(c)] = v
    return spec, score


def test_group_hand_example():
    spec, score = _group_golden()
    g, MB, k = spec["g"], spec["MB"], spec["k"]
    plain = otk.group_topk(score, g, MB, k)
    local = otk.group_topk(score, g, MB, k, local=np.array(spec["local"]))
    assert plain.shape == (spec["T"], spec["H"] // g, k)
    for key, exp in spec["expect_plain"].items():
        assert plain[int(key[3]), int(key[1])].tolist() == exp, key
    for key, exp in spec["expect_local"].items():
        assert local[int(key[3]), int(key[1])].tolist() == exp, key
    k4 = otk.group_topk(score, g, MB, 4)
    assert k4[1, 0].tolist() == spec["k4_plain_r0t1"]


@pytest.mark.parametrize("g", [1, 2, 8])
def test_group_selection_matches_torch_amax_then_topk(g):
    # the group score by torch.amax over the group's heads, the selection by
    # torch.topk: the same sets on rows without ties
    gen = torch.Generator().manual_seed(70 + g)
    R, T, MB, MBp, k = 3, 4, 200, 208, 16
    score = torch.randn(R * g, T, MBp, generator=gen)
    score[:, :, MB:] = 1e30                           # padding columns never count
    out = otk.group_topk(score.numpy(), g, MB, k)
    gs = score.reshape(R, g, T, MBp).amax(dim=1)[:, :, :MB]
    for r in range(R):
        for t in range(T):
            want = sorted(torch.topk(gs[r, t], k).indices.tolist())
            assert out[t, r].tolist() == want


def test_group_selection_ignores_head_order_inside_a_group():
    gen = torch.Generator().manual_seed(77)
    g, R, T, MBp = 4, 2, 3, 64
    score = torch.randn(R * g, T, MBp, generator=gen).numpy()
    perm = np.concatenate([r * g + np.random.default_rng(r).permutation(g) for r in range(R)])
    a = otk.group_topk(score, g, 60, 8)
    b = otk.group_topk(score[perm], g, 60, 8)
    assert np.array_equal(a, b)


def test_group_of_one_head_is_the_per_head_selection():
    gen = torch.Generator().manual_seed(78)
    score = torch.randn(5, 6, 48, generator=gen).numpy()
    assert np.array_equal(otk.group_topk(score, 1, 40, 7), otk.block_topk(score, 40, 7))


def test_local_slot_keeps_the_own_block_and_the_best_others():
    gen = torch.Generator().manual_seed(79)
    g, R, T, MB, MBp, k = 2, 2, 8, 90, 96, 16
    score = torch.randn(R * g, T, MBp, generator=gen)
    local = np.array([0, 5, 89, 44, 44, 3, 88, 17])
    out = otk.group_topk(score.numpy(), g, MB, k, local=local)
    gs = score.reshape(R, g, T, MBp).amax(dim=1)[:, :, :MB]
    for r in range(R):
        for t in range(T):
            row = out[t, r].tolist()
            assert row == sorted(set(row)) and len(row) == k      # ascending, no repeats
            assert int(local[t]) in row
            rest = gs[r, t].clone()
            rest[int(local[t])] = -float("inf")
            best = set(torch.topk(rest, k - 1).indices.tolist())
            assert set(row) == best | {int(local[t])}


def test_own_block_of_each_query_token():
    # rightDownCausal positions: q_pos = kv_len - Lq + i, block q_pos // P
    case = make_case([3, 1, 0, 2], [300, 129, 50, 1], H_q=2, H_kv=1, P=128, D=16,
                     layout="BBND", q_dtype=torch.float16, MB=4, seed=80)
    loc = otk.local_blocks_of(case).tolist()
    # request 0: q_pos 297, 298, 299 -> block 2; request 1: q_pos 128 -> block 1;
    # request 3: q_pos -1 (no key at or before it) and 0 -> none, block 0
    assert loc == [2, 2, 2, 1, -1, 0]


def test_row_subsets_select_the_listed_rows_only():
    # rows = flat h * T + t (block_topk) and r * T + t (group_topk); a subset
    # gives the full call's selections there and -1 everywhere else
    rng = np.random.default_rng(7)
    H, T, MB, k, g = 4, 6, 20, 5, 2
    score = rng.standard_normal((H, T, 32)).astype(np.float32)
    full = otk.block_topk(score, MB, k)
    rows = [1, 8, 23]                                    # (h, t) = (0, 1), (1, 2), (3, 5)
    part = otk.block_topk(score, MB, k, rows=rows)
    for r in range(H * T):
        h, t = divmod(r, T)
        want = full[t, h] if r in rows else np.full(k, -1)
        assert np.array_equal(part[t, h], want), (h, t)
    gfull = otk.group_topk(score, g, MB, k)
    grows = [2, 7]                                       # (r, t) = (0, 2), (1, 1)
    gpart = otk.group_topk(score, g, MB, k, rows=grows)
    for flat in range((H // g) * T):
        r, t = divmod(flat, T)
        want = gfull[t, r] if flat in grows else np.full(k, -1)
        assert np.array_equal(gpart[t, r], want), (r, t)
