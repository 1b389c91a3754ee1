"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself:
  * a hand-worked example (tests/golden/hand_example_p2d2.json),
  * closed forms whose value follows from the definition by inspection
    (one-hot queries against keys that encode their own position, head or
    scale), which fix the mask edges, the gather, the head map and the
    dequantisation order exactly,
  * the independent dense mask-then-amax formulation (oracle.bruteforce),
  * invariants the definition implies (invisible keys never matter, a
    permuted table with a permuted cache is the same input, the three
    layouts are the same data, gap pages are never read, and so on).

Definition: feature request "MsaIndexScore" (gitcode.com/cann/ops-transformer
issues/4117, "calculation"); local mask / shape / modes: torch API guide
"CANN ops-transformer ... msa_index_score", sec. 2, 4, 5.
"""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import bruteforce
from synth import MsaCase, make_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example_p2d2.json")
NEG_INF = float("-inf")


def _val(x):
    return NEG_INF if x == "-inf" else float(x)


def _golden_case(spec, c):
    P, D, H_q, H_kv = spec["P"], spec["D"], spec["H_q"], spec["H_kv"]
    q = torch.tensor(spec["query"], dtype=torch.float32).to(torch.float16)
    kdt = torch.int8 if c["k_dtype"] == "int8" else torch.float16
    key = torch.tensor(spec["key_pages_bbnd"], dtype=torch.float32).to(kdt)
    scale = (torch.tensor(spec["scale_pages"], dtype=torch.float32)
             if c["k_dtype"] == "int8" else None)
    return MsaCase(name=c["name"], query=q, key=key,
                   block_table=torch.tensor(spec["block_table"], dtype=torch.int32),
                   cu_seqlens_q=torch.tensor(spec["cu_seqlens_q"], dtype=torch.int32),
                   kv_len=torch.tensor(spec["kv_len"], dtype=torch.int32), cu_seqlens_k=None,
                   start_loc=torch.tensor(spec["start_loc"], dtype=torch.int32), scale=scale,
                   layout="BBND", sparse_mode=c["sparse_mode"], init_blocks=c["init_blocks"],
                   local_blocks=c["local_blocks"], MB=2, P=P,
                   q_lens=[2], kv_lens=spec["kv_len"])


def _golden_cases():
    with open(GOLDEN) as f:
        spec = json.load(f)
    return spec, spec["cases"]


@pytest.mark.parametrize("idx", range(4))
def test_hand_worked_example(idx):
    spec, cases = _golden_cases()
    c = cases[idx]
    case = _golden_case(spec, c)
    out = oracle.oracle_full(case)
    assert tuple(out.shape) == (2, 2, 16)
    for key, want in c["expect_first_two_cols"].items():
        h, t = int(key[1]), int(key[3])
        got = out[h, t, :2].tolist()
        assert got == [np.float32(_val(w)).item() for w in want], (c["name"], key, got, want)
        assert all(v == NEG_INF for v in out[h, t, 2:].tolist())
    # the second formulation reaches the same hand values
    bf = bruteforce.block_scores(case)
    assert np.array_equal(bf.astype(np.float32), out.numpy())


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def _position_coded_case(q_lens, kv_lens, *, H_q, H_kv, P, D, layout, mode,
                         init_blocks=0, local_blocks=0, start_loc=None, MB=None, seed=0,
                         permute=True):
    """Queries are e_0; key row at logical position j of request b holds j in dim 0.

    Then <q, k_j> = j, so the block score is the largest visible position in
    the block: min(beta*P + P - 1, lim) where lim = min(q_pos, kv_len - 1),
    or -inf when lim < beta*P.  Positions stay below 2048 (exact in fp16).
    """
    case = make_case(q_lens, kv_lens, H_q=H_q, H_kv=H_kv, P=P, D=D, layout=layout,
                     q_dtype=torch.float16, q_kind="onehot_d0", k_kind="randn",
                     sparse_mode=mode, init_blocks=init_blocks, local_blocks=local_blocks,
                     start_loc=start_loc, MB=MB, seed=seed, permute_pages=permute)
    key = case.key
    for b, L in enumerate(kv_lens):
        for j in range(L):
            if layout == "TND":
                row = int(case.cu_seqlens_k[b]) + j
                key[row, :, 0] = float(j)
            else:
                page = int(case.block_table[b, j // P])
                if layout == "BBND":
                    key[page, j % P, :, 0] = float(j)
                else:
                    key[page, :, j % P, 0] = float(j)
    return case


def _closed_form_position(case, q_lens, kv_lens, P):
    MBp = case.MBp
    T = sum(q_lens)
    exp = np.full((case.H_q, T, MBp), NEG_INF, dtype=np.float64)
    t = 0
    for b, (Lq, L) in enumerate(zip(q_lens, kv_lens)):
        for i in range(Lq):
            lim = L - 1 if case.sparse_mode == 0 else min(L - Lq + i, L - 1)
            for beta in range(case.MB):
                if lim >= beta * P:
                    exp[:, t, beta] = min(beta * P + P - 1, lim)
            if L > 0:
                exp[:, t, :min(case.init_blocks, case.MB)] = 1e30
                sl = int(case.start_loc[b])
                for beta in range(max(0, sl + 1 - case.local_blocks), min(sl, case.MB - 1) + 1):
                    exp[:, t, beta] = 1e29
            t += 1
    return exp.astype(np.float32)


@pytest.mark.parametrize("layout", ["BBND", "BNBD", "TND"])
@pytest.mark.parametrize("mode", [0, 3])
def test_closed_form_mask_edges(layout, mode):
    q_lens = [3, 0, 5, 1, 4]
    kv_lens = [9, 7, 4, 13, 0]
    P = 4
    case = _position_coded_case(q_lens, kv_lens, H_q=4, H_kv=2, P=P, D=8, layout=layout,
                                mode=mode, MB=5 if layout != "TND" else None, seed=3)
    out = oracle.oracle_full(case).numpy()
    exp = _closed_form_position(case, q_lens, kv_lens, P)
    assert np.array_equal(out, exp)


@pytest.mark.parametrize("layout", ["BBND", "TND"])
def test_closed_form_local_mask(layout):
    q_lens = [2, 3, 2]
    kv_lens = [17, 0, 6]
    P = 4
    case = _position_coded_case(q_lens, kv_lens, H_q=2, H_kv=1, P=P, D=4, layout=layout,
                                mode=3, init_blocks=2, local_blocks=3, start_loc=[3, 2, 0],
                                MB=6 if layout != "TND" else None, seed=5)
    out = oracle.oracle_full(case).numpy()
    exp = _closed_form_position(case, q_lens, kv_lens, P)
    assert np.array_equal(out, exp)
    # constants are the exact fp32 values; the request with kv_len == 0 stays all fill
    assert (out[:, 0, 0] == np.float32(1e30)).all()
    assert (out[:, 0, 1:4] == np.float32(1e29)).all()   # window [1,3] overrides init at 1
    assert np.isneginf(out[:, 2:5, :]).all()


def test_closed_form_gqa_head_map():
    """Key dim 1 holds 100*(h_kv+1); query e_1 -> score 100*(floor(h/g)+1) on visible blocks."""
    H_q, H_kv, P, D = 8, 2, 4, 4
    case = make_case([3], [10], H_q=H_q, H_kv=H_kv, P=P, D=D, layout="BBND",
                     q_dtype=torch.float16, q_kind="randn", k_kind="randn", sparse_mode=0,
                     init_blocks=0, local_blocks=0, seed=7)
    case.query.zero_()
    case.query[:, :, 1] = 1.0
    for hk in range(H_kv):
        case.key[:, :, hk, :] = 0.0
        case.key[:, :, hk, 1] = 100.0 * (hk + 1)
    out = oracle.oracle_full(case).numpy()
    g = H_q // H_kv
    for h in range(H_q):
        assert (out[h, :, :3] == 100.0 * (h // g + 1)).all(), h
        assert np.isneginf(out[h, :, 3:]).all()


def test_closed_form_int8_scale_index_and_order():
    """int8 keys: k[.,0] = s_sign, scale[page, hk, off] codes (page, hk, off).

    With positive keys the score is the largest scale among visible keys; with
    negative keys it is minus the smallest.  The scale is taken per column
    before the max (order DOT -> DEQUANT -> MASK -> MAX); a max-then-scale
    order gives a different value in the negative case.
    """
    P, D, H_q, H_kv = 4, 4, 2, 2
    for sign in (1, -1):
        case = make_case([2], [7], H_q=H_q, H_kv=H_kv, P=P, D=D, layout="BBND",
                         q_dtype=torch.float16, k_dtype=torch.int8, k_kind="int8_full",
                         sparse_mode=3, init_blocks=0, local_blocks=0, NP=4, seed=11)
        case.query.zero_()
        case.query[:, :, 0] = 1.0
        case.key.zero_()
        case.key[:, :, :, 0] = sign
        NP = case.key.shape[0]
        code = torch.zeros((NP, H_kv, P), dtype=torch.float32)
        for page in range(NP):
            for hk in range(H_kv):
                for off in range(P):
                    code[page, hk, off] = (1 + page * 64 + hk * 16 + off) / 1024.0
        case.scale = code
        out = oracle.oracle_full(case).numpy()
        table = case.block_table[0].tolist()
        # q_pos(t=0)=5, q_pos(t=1)=6; kv_len 7
        for t, lim in ((0, 5), (1, 6)):
            for h in range(H_q):
                hk = h  # g = 1
                for beta in range(2):
                    vis = [j for j in range(beta * P, beta * P + P) if j <= lim]
                    vals = [sign * code[table[j // P], hk, j % P].item() for j in vis]
                    assert out[h, t, beta] == np.float32(max(vals)), (sign, t, h, beta)


# ---------------------------------------------------------------------------
# second formulation
# ---------------------------------------------------------------------------

def _compare_with_bruteforce(case, exact=False):
    """Compare the C oracle with the dense formulation; returns the oracle's output."""
    out = oracle.oracle_full(case).numpy()
    bf = bruteforce.block_scores(case)
    assert out.shape == bf.shape
    inf_o, inf_b = np.isinf(out), np.isinf(bf.astype(np.float32))
    assert np.array_equal(inf_o, inf_b)
    assert np.array_equal(out[inf_o], bf.astype(np.float32)[inf_o])
    fin = ~inf_o
    if exact:
        assert np.array_equal(out[fin], bf[fin].astype(np.float32))
    else:
        # one rounding to fp32 of the same fp64 value (sums may differ in order)
        err = np.abs(out[fin].astype(np.float64) - bf[fin])
        assert (err <= np.abs(bf[fin]) * 2.0 ** -23 + 1e-30).all()
    return out


@pytest.mark.parametrize("layout", ["BBND", "BNBD", "TND"])
@pytest.mark.parametrize("kdt", ["fp16", "bf16", "int8"])
@pytest.mark.parametrize("mode", [0, 3])
def test_oracle_matches_dense_amax(layout, kdt, mode):
    qdt = torch.bfloat16 if kdt == "bf16" else torch.float16
    kdtype = {"fp16": torch.float16, "bf16": torch.bfloat16, "int8": torch.int8}[kdt]
    case = make_case([5, 0, 3, 9, 1], [21, 6, 0, 9, 33], H_q=6, H_kv=3, P=8, D=16,
                     layout=layout, q_dtype=qdt, k_dtype=kdtype,
                     k_kind="int8_full" if kdt == "int8" else "randn", sparse_mode=mode,
                     init_blocks=1, local_blocks=2, MB=6 if layout != "TND" else None,
                     seed=21 + mode)
    _compare_with_bruteforce(case)


@pytest.mark.parametrize("layout", ["BBND", "BNBD", "TND"])
def test_oracle_matches_dense_amax_full_size_blocks(layout):
    """P = D = 128 (the only shape the CUDA path takes), small lengths."""
    case = make_case([7, 2], [300, 129], H_q=4, H_kv=2, P=128, D=128, layout=layout,
                     q_dtype=torch.bfloat16, sparse_mode=3, init_blocks=0, local_blocks=1,
                     MB=4 if layout != "TND" else None, seed=5)
    _compare_with_bruteforce(case)


def test_integer_inputs_are_exact():
    case = make_case([6, 4], [200, 77], H_q=4, H_kv=1, P=128, D=128, layout="BBND",
                     q_dtype=torch.float16, q_kind="int_small", k_kind="int_small",
                     sparse_mode=3, seed=9, MB=3)
    _compare_with_bruteforce(case, exact=True)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

def test_empty_kv_gives_fill_everywhere():
    case = make_case([4, 2], [0, 0], H_q=2, H_kv=1, P=4, D=4, layout="BBND",
                     q_dtype=torch.float16, init_blocks=2, local_blocks=3, MB=3, seed=1)
    out = oracle.oracle_full(case).numpy()
    assert out.shape == (2, 6, 16)
    assert np.isneginf(out).all()


def test_invisible_keys_never_matter():
    """Overwrite every key with j > q_pos(last token) or j >= kv_len; nothing changes."""
    P = 4
    case = make_case([3, 2], [10, 5], H_q=2, H_kv=1, P=P, D=8, layout="BBND",
                     q_dtype=torch.float16, sparse_mode=3, MB=4, NP=8, seed=13)
    base = oracle.oracle_full(case).numpy()
    key = case.key.clone()
    used = set()
    for b, (Lq, L) in enumerate(zip(case.q_lens, case.kv_lens)):
        # rows of request b see at most j <= L-1 (q_pos of the last token)
        for beta in range(case.MB):
            page = int(case.block_table[b, beta])
            if page < 0:
                continue
            used.add(page)
            for off in range(P):
                j = beta * P + off
                if j >= L:
                    key[page, off] = 1.0e4
    for page in range(key.shape[0]):
        if page not in used:
            key[page] = -1.0e4
    case.key = key
    assert np.array_equal(base, oracle.oracle_full(case).numpy())


def test_future_keys_do_not_change_earlier_rows():
    """A row's score never depends on keys beyond its own q_pos."""
    P = 4
    case = make_case([6], [14], H_q=2, H_kv=1, P=P, D=8, layout="BBND",
                     q_dtype=torch.float16, sparse_mode=3, MB=4, seed=17)
    base = oracle.oracle_full(case).numpy()
    # q_pos(i) = 14 - 6 + i = 8 + i; perturb j = 11 (visible only to i >= 3)
    page = int(case.block_table[0, 11 // P])
    case.key[page, 11 % P] = 1.0e4
    out = oracle.oracle_full(case).numpy()
    assert np.array_equal(base[:, :3], out[:, :3])
    assert not np.array_equal(base[:, 3:], out[:, 3:])


def test_permuted_table_equals_contiguous_cache():
    a = make_case([4, 3], [11, 6], H_q=4, H_kv=2, P=4, D=8, layout="BBND",
                  q_dtype=torch.bfloat16, permute_pages=False, MB=4, seed=23)
    b = make_case([4, 3], [11, 6], H_q=4, H_kv=2, P=4, D=8, layout="BBND",
                  q_dtype=torch.bfloat16, permute_pages=True, MB=4, seed=23)
    # same logical keys: move a's pages to b's physical slots
    b.query = a.query.clone()
    key = torch.zeros_like(b.key)
    for r in range(2):
        for beta in range(4):
            pa, pb = int(a.block_table[r, beta]), int(b.block_table[r, beta])
            if pa >= 0:
                key[pb] = a.key[pa]
    b.key = key
    assert np.array_equal(oracle.oracle_full(a).numpy(), oracle.oracle_full(b).numpy())


def test_layouts_agree():
    bb = make_case([5, 2], [19, 8], H_q=4, H_kv=2, P=4, D=8, layout="BBND",
                   q_dtype=torch.float16, permute_pages=True, MB=5, seed=29,
                   init_blocks=1, local_blocks=1)
    bn = MsaCase(**{**bb.__dict__, "key": bb.key.permute(0, 2, 1, 3).contiguous(),
                    "layout": "BNBD"})
    # TND: gather logical rows per request
    rows = []
    for r, L in enumerate(bb.kv_lens):
        for j in range(L):
            rows.append(bb.key[int(bb.block_table[r, j // 4]), j % 4])
    tnd = MsaCase(**{**bb.__dict__, "key": torch.stack(rows), "layout": "TND",
                     "block_table": None, "kv_len": None,
                     "cu_seqlens_k": torch.tensor([0, 19, 27], dtype=torch.int32)})
    o1 = oracle.oracle_full(bb).numpy()
    assert np.array_equal(o1, oracle.oracle_full(bn).numpy())
    assert np.array_equal(o1, oracle.oracle_full(tnd).numpy())


def test_gap_pages_never_read():
    a = make_case([3, 4], [9, 12], H_q=2, H_kv=1, P=4, D=8, layout="BBND",
                  q_dtype=torch.float16, q_kind="abs_randn", MB=4, seed=31, page_gap=1)
    b = make_case([3, 4], [9, 12], H_q=2, H_kv=1, P=4, D=8, layout="BBND",
                  q_dtype=torch.float16, q_kind="abs_randn", MB=4, seed=31, page_gap=2,
                  poison=1.0e4)
    b.query = a.query.clone()
    b.key[:] = a.key          # same data in the used slots; gap slots keep poison
    assert b.key.stride(0) == 2 * a.key.stride(0)
    assert np.array_equal(oracle.oracle_full(a).numpy(), oracle.oracle_full(b).numpy())


def test_mode0_equals_mode3_for_single_token():
    a = make_case([1, 1, 1], [37, 5, 64], H_q=4, H_kv=1, P=8, D=8, layout="BBND",
                  q_dtype=torch.float16, sparse_mode=3, MB=8, seed=37)
    b = MsaCase(**{**a.__dict__, "sparse_mode": 0})
    assert np.array_equal(oracle.oracle_full(a).numpy(), oracle.oracle_full(b).numpy())


def test_prefill_row_equals_decode_call():
    """Row i of a prefill equals a one-token call with kv_len' = kv_len - Lq + i + 1."""
    Lq, L, P = 5, 23, 4
    pre = make_case([Lq], [L], H_q=2, H_kv=1, P=P, D=8, layout="BBND",
                    q_dtype=torch.float16, sparse_mode=3, MB=6, seed=41,
                    init_blocks=0, local_blocks=0)
    out = oracle.oracle_full(pre).numpy()
    for i in range(Lq):
        dec = MsaCase(**{**pre.__dict__,
                         "query": pre.query[i:i + 1].clone(),
                         "cu_seqlens_q": torch.tensor([0, 1], dtype=torch.int32),
                         "kv_len": torch.tensor([L - Lq + i + 1], dtype=torch.int32)})
        o = oracle.oracle_full(dec).numpy()
        assert np.array_equal(o[:, 0], out[:, i])


def test_output_shape_and_padding():
    case = make_case([2], [40], H_q=3, H_kv=1, P=4, D=4, layout="BBND",
                     q_dtype=torch.float16, MB=17, seed=43)
    out = oracle.oracle_full(case).numpy()
    assert out.shape == (3, 2, 32)
    assert np.isneginf(out[:, :, 17:]).all()
    assert np.isneginf(out[:, :, 10:]).all()   # blocks past ceil(40/4)=10 are empty


def test_fill_value_is_a_parameter():
    case = make_case([1], [3], H_q=1, H_kv=1, P=4, D=4, layout="BBND",
                     q_dtype=torch.float16, MB=2, seed=47, local_blocks=0)
    out = oracle.oracle_full(case, fill_value=-3.4028e38).numpy()
    assert out[0, 0, 1] == np.float32(-3.4028e38)


def test_row_sampling_matches_full():
    case = make_case([5, 3], [30, 12], H_q=4, H_kv=2, P=8, D=8, layout="BNBD",
                     q_dtype=torch.bfloat16, MB=4, seed=53)
    full = oracle.oracle_full(case).numpy()
    rows = [0, 5, 9, 17, 31]
    part = oracle.oracle_rows(case, rows).numpy()
    for i, r in enumerate(rows):
        assert np.array_equal(part[i], full[r // case.T, r % case.T])


# ---------------------------------------------------------------- FP8 inputs
# FP8 query and key of one type, no scale (torch API guide, sec. 4 and 7.2).

@pytest.mark.parametrize("dt", [torch.float8_e4m3fn, torch.float8_e5m2])
def test_fp8_decoding_matches_torch_for_every_bit_pattern(dt):
    bits = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = bits.view(dt).to(torch.float64).numpy()
    got = np.array([oracle.decode(dt, int(b)) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_fp16_decoding_matches_numpy_for_every_bit_pattern():
    # all 65,536 binary16 patterns, decoded by numpy's IEEE half type: pins the
    # normal, subnormal (exponent field 0), infinity and NaN branches
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.decode(torch.float16, int(b)) for b in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # the subnormal range on its own: m * 2^-24 for m in 1..1023, both signs
    m = np.arange(1, 1024)
    assert np.array_equal(got[m], m * 2.0 ** -24)
    assert np.array_equal(got[0x8000 + m], -m * 2.0 ** -24)


def test_bf16_decoding_matches_torch_for_every_bit_pattern():
    # all 65,536 bfloat16 patterns, decoded by torch's bfloat16 type
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode(torch.bfloat16, b & 0xFFFF) for b in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("layout", ["BBND", "BNBD", "TND"])
@pytest.mark.parametrize("dt", [torch.float8_e4m3fn, torch.float8_e5m2])
@pytest.mark.parametrize("mode", [0, 3])
def test_fp8_oracle_matches_dense_amax(layout, dt, mode):
    case = make_case([5, 0, 3, 9, 1], [21, 6, 0, 9, 33], H_q=6, H_kv=3, P=8, D=16,
                     layout=layout, q_dtype=dt, k_dtype=dt, sparse_mode=mode,
                     init_blocks=1, local_blocks=2, MB=6 if layout != "TND" else None,
                     seed=41 + mode)
    _compare_with_bruteforce(case)


def test_fp8_one_hot_reads_the_key_value():
    # q = e_0 (1.0 is exact in both formats): each score is the largest visible
    # k[j, 0] of the block, decoded by torch from the same bytes
    dt = torch.float8_e4m3fn
    case = make_case([1], [300], H_q=2, H_kv=1, P=128, D=128, layout="BBND",
                     q_dtype=dt, k_dtype=dt, q_kind="onehot_d0", sparse_mode=0,
                     init_blocks=0, local_blocks=0, MB=3, seed=3)
    out = oracle.oracle_full(case).numpy()
    keys = bruteforce._gather_keys(case, 0, 300, 3)      # [300, H_kv, D] fp64 via torch
    for beta in range(3):
        lo, hi = beta * 128, min(300, beta * 128 + 128)
        assert out[0, 0, beta] == np.float32(keys[lo:hi, 0, 0].max())


# ---------------------------------------------------------------------------
# FP4 inputs (MiniMax Sparse Attention notes, section 8.2: MXFP4 = E2M1 values
# with an E8M0 scale per 32 elements, NVFP4 = E2M1 values with an E4M3 scale
# per 16); formats as defined by the OCP Microscaling (MX) specification

# E2M1 by code 0..15: +0, 0.5, 1, 1.5, 2, 3, 4, 6, then the same negated
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_decoding_matches_the_format_table():
    got = [oracle.decode("e2m1", c) for c in range(16)]
    assert got == E2M1_TABLE
    assert [np.signbit(x) for x in got] == [c >= 8 for c in range(16)]


def test_e2m1_decoding_matches_torch_e4m3_of_the_same_value():
    # every E2M1 value is an E4M3 value: same sign, exponent e - 1 + 7, mantissa
    # bit m as the top of three (code 1, 0.5, is the normal E4M3 0.5); torch
    # decodes those bytes
    def as_e4m3(c):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        if e == 0:
            mag = 0 if m == 0 else (6 << 3)              # 0, or 0.5 = 2^(6-7)
        else:
            mag = ((e + 6) << 3) | (m << 2)
        return (s << 7) | mag
    b = torch.tensor([as_e4m3(c) for c in range(16)], dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    assert [oracle.decode("e2m1", c) for c in range(16)] == ref


def test_e8m0_decoding_matches_torch_for_every_bit_pattern():
    bits = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = bits.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([oracle.decode("e8m0", b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 1
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("layout", ["BBND", "BNBD", "TND"])
@pytest.mark.parametrize("fmt", ["mx", "nv"])
@pytest.mark.parametrize("mode", [0, 3])
def test_fp4_oracle_matches_dense_amax(layout, fmt, mode):
    from synth import make_fp4_case
    case = make_fp4_case([5, 0, 3, 9, 1], [900, 6, 0, 9, 1000], fmt=fmt, H_q=6, H_kv=3,
                         layout=layout, sparse_mode=mode, init_blocks=1, local_blocks=1,
                         MB=8 if layout != "TND" else None, seed=60 + mode)
    out = _compare_with_bruteforce(case)
    real = np.isfinite(out) & (np.abs(out) < 1e28)
    assert real.sum() > 100                       # most blocks are real scores, not forced


def test_fp4_with_unit_scales_equals_the_fp16_oracle_on_the_decoded_values():
    # E8M0 code 127 is 1.0: the block scores are those of the E2M1 values
    # themselves, which fp16 holds exactly, so the fp16 oracle must agree bit
    # for bit
    from synth import make_fp4_case
    case = make_fp4_case([7, 1], [400, 130], fmt="mx", H_q=4, H_kv=2, layout="BBND", MB=4,
                         scale_codes=(127, 127), seed=61)
    table = torch.tensor(E2M1_TABLE, dtype=torch.float16)

    def unpack(p):
        b = p.to(torch.int64)
        return table[torch.stack([b & 15, b >> 4], dim=-1).flatten(-2)]
    f16 = dataclasses.replace(case, query=unpack(case.query), key=unpack(case.key), fp4=None,
                              q_scale=None, k_scale=None)
    assert torch.equal(oracle.oracle_full(case), oracle.oracle_full(f16))


def test_fp4_group_scales_apply_to_their_own_elements():
    # query = +1 everywhere (code 2) with unit scales; key = +1 everywhere with
    # the scale of group gi of token j equal to 2^gi (MXFP4, 4 groups of 32):
    # every dot product is 32 * (1 + 2 + 4 + 8) = 480, and a wrong group or
    # element index would change it
    from synth import make_fp4_case
    case = make_fp4_case([3], [200], fmt="mx", H_q=2, H_kv=1, layout="BNBD", MB=2,
                         sparse_mode=0, init_blocks=0, local_blocks=0, seed=62)
    case.query.fill_(0x22)
    case.key.fill_(0x22)
    case.q_scale.fill_(127)
    case.k_scale.copy_(torch.tensor([127, 128, 129, 130], dtype=torch.uint8).expand_as(case.k_scale))
    out = oracle.oracle_full(case)
    assert torch.all(out[:, :, :2] == 480.0)
