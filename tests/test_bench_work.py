"""The benchmark's algorithmic work (the numerators of its roofline fractions)
against brute-force counts on small cases (no GPU).

The score op's FLOPs are 2 * D per visible (query head, token, key) triple,
with visibility as the feature request "MsaIndexScore" defines it ("calculation":
j < kv_len and, in sparse_mode 3, j <= q_pos = kv_len - Lq + i); its key bytes
count every key some row of the request sees once per kv head, at the bytes a
stored key row takes (int8 rows add their fp32 scale, FP4 rows their group
scale bytes).  The sparse main branch's FLOPs are 4 * D per visible (query
head, token, key) of the selected blocks (S = Q K^T and O = P V; MiniMax Sparse
Attention notes, section 4.8 Equation (8)), and its K/V bytes count each
distinct selected (kv head, request, block) page once.
"""
import numpy as np
import pytest
import torch

import bench
from synth import make_case, make_fp4_case


def _visible(mode, L, Lq, i, j):
    return j < L and (mode != 3 or j <= L - Lq + i)


def _brute_score_work(case, row_bytes):
    triples, keys = 0, 0
    for Lq, L in zip(case.q_lens, case.kv_lens):
        seen = set()
        for i in range(Lq):
            for j in range(case.MB * case.P):
                if _visible(case.sparse_mode, L, Lq, i, j):
                    triples += 1
                    seen.add(j)
        keys += len(seen)
    return 2.0 * case.D * case.H_q * triples, keys * case.H_kv * row_bytes


CASES = {
    # q_lens, kv_lens (a request longer than its KV, an empty query, an empty KV)
    "mixed_mode3": ([5, 0, 9, 3, 1], [17, 40, 4, 0, 33], 3),
    "mixed_mode0": ([5, 0, 9, 3, 1], [17, 40, 4, 0, 33], 0),
    "decode": ([1, 1, 1], [1, 16, 31], 3),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("kdt", ["bf16", "int8"])
def test_score_work_matches_brute_force(name, kdt):
    q_lens, kv_lens, mode = CASES[name]
    k_dtype = torch.int8 if kdt == "int8" else None
    q_dtype = torch.float16 if kdt == "int8" else torch.bfloat16
    case = make_case(q_lens, kv_lens, H_q=4, H_kv=2, P=8, D=16, layout="BBND",
                     q_dtype=q_dtype, k_dtype=k_dtype, MB=6, sparse_mode=mode, seed=5)
    # bytes of one stored key row, from the tensors themselves
    row = case.key.shape[-1] * case.key.element_size()
    if case.scale is not None:
        row += case.scale.element_size()
    flops, kbytes = _brute_score_work(case, row)
    w = bench.algorithmic_work(case)
    assert w["flops"] == flops
    assert w["k_bytes"] == kbytes
    assert w["q_bytes"] == case.query.numel() * case.query.element_size()
    assert w["out_bytes"] == 4 * int(np.prod(case.out_shape))


@pytest.mark.parametrize("fmt", ["mx", "nv"])
def test_fp4_score_work_counts_codes_and_group_scales(fmt):
    case = make_fp4_case([3, 2], [20, 9], fmt=fmt, H_q=2, H_kv=1, P=8, MB=3, layout="BNBD",
                         seed=6)
    row = case.key.shape[-1] + case.k_scale.shape[-1]      # code bytes + scale bytes of a row
    flops, kbytes = _brute_score_work(case, row)
    w = bench.algorithmic_work(case)
    assert w["flops"] == flops and w["k_bytes"] == kbytes
    assert w["q_bytes"] == case.query.numel() + case.q_scale.numel()


@pytest.mark.parametrize("mode", [3, 0])
def test_sparse_work_matches_brute_force(mode):
    case = make_case([4, 3, 2], [30, 5, 19], H_q=4, H_kv=2, P=8, D=16, layout="BBND",
                     q_dtype=torch.bfloat16, MB=4, sparse_mode=mode, seed=8)
    # well-formed selections: distinct blocks of [0, MB) ascending, then a -1 tail
    rng = np.random.default_rng(9)
    sel = torch.full((case.T, case.H_kv, 3), -1, dtype=torch.int32)
    for t in range(case.T):
        for r in range(case.H_kv):
            n = int(rng.integers(0, 4))
            sel[t, r, :n] = torch.as_tensor(np.sort(rng.choice(case.MB, n, replace=False)))
    gq = case.H_q // case.H_kv
    cu = case.cu_seqlens_q.tolist()
    keys, pages = 0, set()
    for b in range(case.B):
        Lq, L = case.q_lens[b], case.kv_lens[b]
        for t in range(cu[b], cu[b + 1]):
            for r in range(case.H_kv):
                for beta in sel[t, r].tolist():
                    if beta < 0 or beta >= case.MB or beta * case.P >= L:
                        continue                           # -1, past the table, past the last block
                    pages.add((r, b, beta))
                    keys += sum(_visible(mode, L, Lq, t - cu[b], j)
                                for j in range(beta * case.P, (beta + 1) * case.P))
    flops, nbytes, nblocks = bench.sparse_work(case, sel)
    assert flops == 4.0 * case.D * gq * keys
    assert nblocks == len(pages)
    es = case.key.element_size()
    assert nbytes == (case.query.numel() * case.query.element_size()
                      + len(pages) * 2 * case.P * case.D * es + case.T * case.H_q * (case.D + 1) * 4)
