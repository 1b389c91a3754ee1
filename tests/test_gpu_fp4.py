"""GPU parity of the FP4 index branch (msa_index_score_fp4) against the oracle.

FP4 inputs (MiniMax Sparse Attention notes, sec. 8.2): E2M1 codes with one
E8M0 scale per 32 elements (MXFP4) or one E4M3 scale per 16 (NVFP4), for the
query and the key cache alike.  The oracle dequantises every element exactly
and sums in fp64; the GPU dequantises exactly into 16-bit operands and sums in
fp32, so the scores agree within the 16-bit tolerance
|diff| <= 1e-3 + 1e-4 * |ref|, and bit for bit when every product and partial
sum is exact in fp32 (unit scales: E2M1 products are multiples of 1/4 up to
36, sums of 128 of them stay far below 2^24 quarters).
"""
import pytest
import torch

import oracle
import synth
from test_gpu_parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_score_gb300 as bs
    bs.load_library()
    return torch.device("cuda:0")


def run(case, dev):
    import block_score_gb300 as bs
    prep = bs.from_case(case, dev)
    out = prep().cpu()
    return out, prep.device_error()


MATRIX = [(layout, fmt) for layout in ("BBND", "BNBD", "TND") for fmt in ("mx", "nv")]


@pytest.mark.parametrize("layout,fmt", MATRIX)
@pytest.mark.parametrize("mode", [3, 0])
def test_fp4_layout_matrix_mixed_batch(dev, layout, fmt, mode):
    # prefill tiles, decode, q_len 0, kv_len 0, a tail, long KV, GQA g = 8
    case = synth.make_fp4_case([37, 1, 0, 4, 200, 1], [290, 1, 77, 0, 600, 4100], fmt=fmt,
                               H_q=16, H_kv=2, layout=layout, sparse_mode=mode,
                               MB=40 if layout != "TND" else None, init_blocks=1,
                               local_blocks=2, seed=400 + 10 * mode + (fmt == "nv"))
    out, err = run(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what=f"fp4 {fmt} {layout} mode {mode}")


@pytest.mark.parametrize("fmt,unit", [("mx", 127), ("nv", 0x38)])
def test_fp4_unit_scales_bit_exact(dev, fmt, unit):
    case = synth.make_fp4_case([70, 1, 3], [700, 5000, 129], fmt=fmt, H_q=8, H_kv=2,
                               layout="BBND", MB=40, scale_codes=(unit, unit),
                               init_blocks=0, local_blocks=0, seed=410)
    out, err = run(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), exact=True, what=f"fp4 {fmt} unit scales")


@pytest.mark.parametrize("fmt", ["mx", "nv"])
def test_fp4_wide_scale_range_and_gqa(dev, fmt):
    # scales over a wide range (MXFP4 2^-20 .. 2^20; NVFP4 E4M3 2^-6 .. 448)
    codes = (107, 147) if fmt == "mx" else (0x08, 0x7e)
    case = synth.make_fp4_case([17, 40], [300, 1000], fmt=fmt, H_q=32, H_kv=2, layout="BNBD",
                               MB=9, scale_codes=codes, sparse_mode=3, init_blocks=1,
                               local_blocks=2, seed=411)
    out, err = run(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what=f"fp4 {fmt} wide scales")


def test_fp4_strided_cache_with_poisoned_gaps(dev):
    case = synth.make_fp4_case([20, 3], [500, 260], fmt="nv", H_q=8, H_kv=1, layout="BBND",
                               MB=6, page_gap=2, poison=0.0, seed=412)
    # the gap pages hold codes that no correct read may see: all 0x77 (+6, +6)
    base = case.key
    while base._base is not None:
        base = base._base
    base[:, 1:] = 0x77
    out, err = run(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what="fp4 strided")


def test_fp4_validation(dev):
    import block_score_gb300 as bs
    case = synth.make_fp4_case([4], [300], fmt="mx", H_q=4, H_kv=1, layout="BBND", MB=3, seed=413)
    with pytest.raises(Exception):
        bs.from_case(synth.dataclasses.replace(case, q_scale=None), dev)
    # E2M1 through the 16-bit entry point is refused
    prep = bs.from_case(case, dev)
    lib = bs.load_library()
    st = lib.msa_index_score(bs.ctypes.byref(prep.call.args), prep.out.data_ptr(),
                             prep.workspace.data_ptr(), prep.ws_bytes, None)
    assert st == 1


@pytest.mark.parametrize("n", [2, 5])
def test_fp4_benchmark_workload_sampled(dev, n):
    case = synth.to_fp4(synth.config(n), "nv" if n == 2 else "mx")
    out, err = run(case, dev)
    assert err == 0
    import numpy as np
    rng = np.random.default_rng(n)
    rows = sorted(set(rng.integers(0, case.H_q * case.T, 256).tolist()))
    ref = oracle.oracle_rows(case, rows)
    got = out.reshape(-1, out.shape[2])[torch.tensor(rows)]
    assert_parity(got, ref, what=f"cfg{n} fp4 sampled")


@pytest.mark.parametrize("fmt", ["mx", "nv"])
@pytest.mark.parametrize("layout", ["BBND", "BNBD", "TND"])
@pytest.mark.parametrize("g,mode", [(1, 3), (8, 3), (8, 0), (32, 3)])
def test_fp4_short_query_requests(dev, fmt, layout, g, mode):
    # requests of at most 32 query rows (decode, speculative decode): the
    # short-query kernel dequantises each FP4 page once into tensor memory.
    # One-key and one-page requests, q_len 0, kv_len 0, a ragged tail and a
    # long request; with the host length bound the tile kernel is left out.
    import block_score_gb300 as bs
    qmax = 32 // g
    H_kv = 1 if g == 32 else 2
    case = synth.make_fp4_case([1, qmax, 0, 1, max(1, qmax // 2), 1], [1, 300, 50, 0, 129, 9000],
                               fmt=fmt, H_q=g * H_kv, H_kv=H_kv, layout=layout,
                               MB=80 if layout != "TND" else None, sparse_mode=mode,
                               init_blocks=1, local_blocks=2,
                               seed=430 + g + 2 * mode + (fmt == "nv") + 5 * len(layout))
    ref = oracle.oracle_full(case)
    for bound in (None, qmax):
        prep = bs.from_case(case, dev, max_seqlen_q=bound)
        out = prep().cpu()
        assert prep.device_error() == 0
        assert_parity(out, ref, what=f"fp4 short {fmt} {layout} g={g} mode {mode} bound={bound}")


@pytest.mark.parametrize("fmt,unit", [("mx", 127), ("nv", 0x38)])
def test_fp4_short_query_unit_scales_bit_exact(dev, fmt, unit):
    # decode only (g = 16, N = 16 rows, and q_len 2 -> 32 rows): bit-exact
    case = synth.make_fp4_case([1, 2, 1, 1], [5000, 700, 128, 33], fmt=fmt, H_q=16, H_kv=1,
                               layout="BNBD", MB=40, scale_codes=(unit, unit),
                               init_blocks=0, local_blocks=0, seed=450 + (fmt == "nv"))
    out, err = run(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), exact=True, what=f"fp4 short {fmt} unit scales")


def test_fp4_short_query_bad_block_table_entry_is_reported(dev):
    case = synth.make_fp4_case([1, 2], [300, 500], fmt="nv", H_q=8, H_kv=1, layout="BBND",
                               MB=4, seed=460)
    case.block_table[0, 1] = 10_000          # beyond NP, inside the needed range
    _, err = run(case, dev)
    assert err & 0x08
    case.block_table[0, 1] = -3
    _, err = run(case, dev)
    assert err & 0x08


@pytest.mark.parametrize("fmt", ["mx", "nv"])
@pytest.mark.parametrize("mirror", [True, False])
def test_fp4_mirror_and_converter_paths(dev, fmt, mirror):
    # a prefill-heavy call: with the full workspace the key pages are
    # dequantised once into the 16-bit mirror and scored by the 16-bit tile
    # kernel; with room for the plan and the query only, the converter warps
    # dequantise each page per query tile.  Unit scales: both bit-exact.
    import block_score_gb300 as bs
    unit = 127 if fmt == "mx" else 0x38
    case = synth.make_fp4_case([200, 1, 70], [900, 300, 4100], fmt=fmt, H_q=16, H_kv=2,
                               layout="BNBD", MB=33, scale_codes=(unit, unit),
                               init_blocks=1, local_blocks=2, seed=420 + (fmt == "nv"))
    prep = bs.from_case(case, dev)
    mirror_bytes = case.key.shape[0] * case.H_kv * case.P * case.D * 2
    assert prep.ws_bytes > mirror_bytes          # T * g >= 128 * B: the mirror is sized in
    if not mirror:
        prep.ws_bytes -= mirror_bytes
    out = prep().cpu()
    assert prep.device_error() == 0
    assert_parity(out, oracle.oracle_full(case), exact=True, what=f"fp4 {fmt} mirror={mirror}")
