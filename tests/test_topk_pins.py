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
