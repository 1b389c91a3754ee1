"""The seeded synthetic workloads follow their recipes (no GPU).

Each workload of the benchmark and of the full-size parity tests is drawn by
``synth.config(n)``; these tests hold the drawn inputs to the recipe's shapes,
length ranges, value ranges and table structure, so a change to the generator
cannot silently change what is measured.
"""
import pytest
import torch

import synth


def _cdiv(a, b):
    return -(-a // b)


def _check_table(case, whole_pool: bool):
    """Entries below ceil(kv_len / P) are distinct pages of [0, NP) (the pool in
    a random order when whole_pool); every other entry is -1."""
    NP = int(case.key.shape[0])
    used = []
    for b in range(case.B):
        nb = _cdiv(case.kv_lens[b], case.P)
        row = case.block_table[b].tolist()
        assert all(0 <= p < NP for p in row[:nb])
        assert all(p == -1 for p in row[nb:])
        used += row[:nb]
    assert len(set(used)) == len(used)
    if whole_pool:
        assert sorted(used) == list(range(NP))
        assert used != sorted(used)                     # permuted, not in pool order


def _check_lengths(case):
    cu = case.cu_seqlens_q.tolist()
    assert cu[0] == 0 and all(cu[b + 1] - cu[b] == case.q_lens[b] for b in range(case.B))
    assert cu[-1] == case.T
    if case.kv_len is not None:
        assert case.kv_len.tolist() == case.kv_lens


def test_tiny_paged_prefill():
    c = synth.config(1)
    assert (c.layout, c.query.dtype, c.key.dtype) == ("BBND", torch.float16, torch.float16)
    assert (c.B, c.T, c.H_q, c.H_kv, c.D, c.P) == (1, 32, 8, 1, 128, 128)
    assert int(c.key.shape[0]) == 8 and c.block_table.tolist() == [[0, 1]]
    assert c.kv_lens == [256] and c.cu_seqlens_q.tolist() == [0, 32]
    assert c.start_loc.tolist() == [1]
    assert (c.sparse_mode, c.init_blocks, c.local_blocks) == (3, 0, 1)
    assert c.out_shape == (8, 32, 16)


def test_batched_decode():
    c = synth.config(2)
    _check_lengths(c)
    assert (c.layout, c.query.dtype, c.key.dtype) == ("BBND", torch.bfloat16, torch.bfloat16)
    assert (c.B, c.T, c.H_q, c.H_kv, c.MB) == (64, 64, 16, 1, 512)
    assert c.q_lens == [1] * 64
    assert all(1024 <= L <= 65536 for L in c.kv_lens)
    assert int(c.key.shape[0]) == sum(_cdiv(L, 128) for L in c.kv_lens)
    _check_table(c, whole_pool=True)
    assert c.start_loc.tolist() == [_cdiv(L, 128) - 1 for L in c.kv_lens]
    assert (c.sparse_mode, c.init_blocks, c.local_blocks) == (3, 0, 1)
    assert 0.09 < float(c.key.float().std()) < 0.11          # randn * 0.1
    assert c.out_shape == (16, 64, 512)


def test_varlen_chunked_prefill():
    c = synth.config(3)
    _check_lengths(c)
    assert (c.layout, c.query.dtype, c.key.dtype) == ("BNBD", torch.bfloat16, torch.bfloat16)
    assert (c.B, c.H_q, c.H_kv, c.MB) == (6, 32, 4, 128)
    pairs = sorted(zip(c.q_lens, c.kv_lens))
    # one request with no query, one with no keys, four with q_len 2048 .. 8192
    # and kv_len = q_len + U[0, 8192]
    assert pairs[0][0] == 0 and 1 <= pairs[0][1] <= 8192
    assert pairs[1] == (256, 0)
    assert [q for q, _ in pairs[2:]] == [2048, 4096, 6144, 8192]
    assert all(0 <= L - q <= 8192 for q, L in pairs[2:])
    assert c.T == 20736
    assert c.q_lens != sorted(c.q_lens)                       # shuffled order
    _check_table(c, whole_pool=False)
    assert c.start_loc.tolist() == [max(_cdiv(L, 128) - 1, 0) for L in c.kv_lens]
    assert (c.sparse_mode, c.init_blocks, c.local_blocks) == (3, 1, 4)
    assert c.out_shape == (32, 20736, 128)


def test_int8_mixed():
    c = synth.config(4)
    _check_lengths(c)
    assert (c.layout, c.query.dtype, c.key.dtype) == ("BBND", torch.float16, torch.int8)
    assert (c.B, c.H_q, c.H_kv, c.MB) == (32, 16, 2, 256)
    assert sorted(c.q_lens) == [1] * 24 + [512] * 8
    assert c.q_lens != sorted(c.q_lens)
    assert all(8192 <= L <= 32768 for L in c.kv_lens)
    _check_table(c, whole_pool=False)
    k = c.key.to(torch.int16)
    assert int(k.min()) >= -127 and int(k.max()) <= 127
    assert tuple(c.scale.shape) == (int(c.key.shape[0]), 2, 128)
    assert 1e-3 <= float(c.scale.min()) and float(c.scale.max()) <= 2e-2
    assert c.start_loc.tolist() == [_cdiv(L, 128) - 1 for L in c.kv_lens]
    assert (c.sparse_mode, c.init_blocks, c.local_blocks) == (3, 0, 1)


def test_long_context_prefill():
    c = synth.config(5)
    _check_lengths(c)
    assert (c.layout, c.query.dtype, c.key.dtype) == ("BBND", torch.bfloat16, torch.bfloat16)
    assert (c.B, c.T, c.H_q, c.H_kv, c.MB) == (1, 16384, 64, 8, 1100)
    assert c.kv_lens == [131072] and int(c.key.shape[0]) == 1024
    _check_table(c, whole_pool=True)                         # columns 1024 .. 1099 are -1
    assert c.start_loc.tolist() == [1023]
    assert (c.sparse_mode, c.init_blocks, c.local_blocks) == (3, 4, 8)
    assert c.out_shape == (64, 16384, 1104)


@pytest.mark.parametrize("n", [1, 2, 4])
def test_workloads_are_seeded(n):
    a, b = synth.config(n), synth.config(n)
    assert a.kv_lens == b.kv_lens and a.q_lens == b.q_lens
    assert torch.equal(a.query, b.query) and torch.equal(a.key, b.key)
    assert torch.equal(a.block_table, b.block_table)
