"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerance (fp inputs): |gpu - oracle| <= 1e-3 + 1e-4 * |oracle| on finite
scores.  Fill (-inf), forced (1e30 / 1e29) and padding positions must match
bit for bit, and so must every score of the integer-valued cases, where all
products and sums are exact in fp32.

Case categories follow the reference op's test matrix (torch API guide,
sec. 9.2): fp16 / bf16 / int8 x BBND / BNBD / TND, mixed batches with
q_len = 0 / kv_len = 0, a strided paged cache whose gap pages hold poison,
wide block tables (257, 275), short decode (q4-kv4, q4-kv275), speculative
multi-token decode, long KV over many blocks and tiny-KV tails.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-3, 1e-4


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_score_gb300 as bs
    bs.load_library()
    return torch.device("cuda:0")


def run_gpu(case, dev):
    import block_score_gb300 as bs
    prep = bs.from_case(case, dev)
    out = prep()
    err = prep.device_error()
    return out.cpu(), err, prep


def assert_parity(out, ref, exact=False, what=""):
    assert tuple(out.shape) == tuple(ref.shape), what
    inf_r = torch.isinf(ref)
    inf_o = torch.isinf(out)
    bad = (inf_r != inf_o).nonzero()
    assert bad.numel() == 0, f"{what}: fill pattern differs at {bad[:8].tolist()}"
    assert torch.equal(out[inf_r], ref[inf_r]), f"{what}: sign of fill differs"
    forced = ref.abs() >= 1e28
    assert torch.equal(out[forced], ref[forced]), f"{what}: forced scores differ"
    fin = ~inf_r & ~forced
    if exact:
        neq = (out[fin] != ref[fin])
        assert not bool(neq.any()), f"{what}: {int(neq.sum())} inexact scores"
        return
    o, r = out[fin].double(), ref[fin].double()
    diff = (o - r).abs()
    tol = ATOL + RTOL * r.abs()
    if diff.numel():
        worst = int(torch.argmax(diff - tol))
        assert bool((diff <= tol).all()), (
            f"{what}: max excess {float((diff - tol).max()):.3e} "
            f"(gpu {float(o[worst])}, oracle {float(r[worst])})")


def test_tiny_paged_prefill_workload(dev):
    case = synth.config(1)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what="cfg1")


def test_integer_inputs_bit_exact(dev):
    # several tiles per request (g=4 -> 32 positions per tile), ragged tails,
    # diagonal blocks, GQA heads, permuted pages
    case = synth.make_case([70, 1, 0, 33, 129], [700, 130, 50, 33, 129], H_q=8, H_kv=2,
                           layout="BBND", q_dtype=torch.float16, q_kind="int_small",
                           k_kind="int_small", MB=7, init_blocks=0, local_blocks=0, seed=101)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), exact=True, what="int exact")


def test_integer_inputs_bit_exact_bf16_mode0(dev):
    case = synth.make_case([17, 40], [300, 1000], H_q=16, H_kv=1, layout="BNBD",
                           q_dtype=torch.bfloat16, q_kind="int_small", k_kind="int_small",
                           MB=9, sparse_mode=0, init_blocks=1, local_blocks=2, seed=102)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), exact=True, what="int exact mode0")


def test_int8_with_unit_scale_is_bit_exact(dev):
    # integer queries and int8 keys with scale 1: every product and sum is exact
    # in fp32, so the int8 path (convert, MMA, column scale, max) must match the
    # oracle bit for bit, including decode and prefill rows
    case = synth.make_case([1, 40, 1, 130], [5000, 700, 128, 1000], H_q=16, H_kv=2,
                           layout="BBND", q_dtype=torch.float16, k_dtype=torch.int8,
                           q_kind="int_small", k_kind="int8_full", scale_const=1.0, MB=40,
                           seed=105)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), exact=True, what="int8 unit scale")


MATRIX = []
for layout in ("BBND", "BNBD", "TND"):
    for kdt in ("fp16", "bf16", "int8"):
        MATRIX.append((layout, kdt))


@pytest.mark.parametrize("layout,kdt", MATRIX)
def test_dtype_layout_matrix_mixed_batch(dev, layout, kdt):
    qdt = torch.bfloat16 if kdt == "bf16" else torch.float16
    kdtype = {"fp16": torch.float16, "bf16": torch.bfloat16, "int8": torch.int8}[kdt]
    # mixed batch: prefill, decode, q_len=0, kv_len=0, tail, long kv
    q = [37, 1, 0, 4, 200, 1]
    kv = [290, 1, 77, 0, 600, 4100]
    case = synth.make_case(q, kv, H_q=16, H_kv=2, layout=layout, q_dtype=qdt, k_dtype=kdtype,
                           k_kind="int8_full" if kdt == "int8" else "randn",
                           MB=None if layout == "TND" else 40, init_blocks=1, local_blocks=2,
                           seed=200 + len(layout) + len(kdt))
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what=f"{layout}/{kdt}")


@pytest.mark.parametrize("mode", [0, 3])
def test_sparse_modes(dev, mode):
    case = synth.make_case([64, 9], [333, 129], H_q=8, H_kv=8, layout="BBND",
                           q_dtype=torch.float16, MB=5, sparse_mode=mode, seed=300 + mode)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what=f"mode{mode}")


# int8 keys without the causal bound (sparse_mode 0, torch API guide sec. 4;
# int8 path sec. 7.1): the short-query kernel (Lq * g <= 32 query rows) and the
# tile kernel each have a mode-0 branch of their own
INT8_MODE0 = [(layout, g) for layout in ("BBND", "TND") for g in (8, 4)]


@pytest.mark.parametrize("layout,g", INT8_MODE0)
def test_int8_keys_sparse_mode0(dev, layout, g):
    # g=8: Lq 2, 3, 4 are short-class requests (16, 24, 32 query rows), Lq 5
    # and 40 are tile-class; g=4 moves Lq 5..8 into the short class as well
    H_kv = 2
    q = [2, 3, 4, 1, 5, 40, 8, 0]
    kv = [700, 129, 4000, 1, 260, 1500, 128, 50]
    case = synth.make_case(q, kv, H_q=g * H_kv, H_kv=H_kv, layout=layout,
                           q_dtype=torch.float16, k_dtype=torch.int8, sparse_mode=0,
                           MB=40 if layout != "TND" else None, init_blocks=1,
                           local_blocks=2, seed=340 + g + (layout == "TND"))
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what=f"int8 mode0 {layout} g={g}")


@pytest.mark.parametrize("layout", ["BBND", "TND"])
def test_int8_unit_scale_bit_exact_mode0(dev, layout):
    # integer queries, int8 keys, scale 1: exact in fp32, so bit-exact in mode 0
    # for short-class (Lq 2..4 with g=8) and tile-class requests alike
    case = synth.make_case([2, 4, 3, 1, 70], [300, 4100, 128, 9, 900], H_q=16, H_kv=2,
                           layout=layout, q_dtype=torch.float16, k_dtype=torch.int8,
                           q_kind="int_small", k_kind="int8_full", scale_const=1.0,
                           sparse_mode=0, MB=33 if layout != "TND" else None,
                           init_blocks=0, local_blocks=0, seed=350 + (layout == "TND"))
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), exact=True, what=f"int8 exact mode0 {layout}")


@pytest.mark.parametrize("layout", ["BBND", "BNBD"])
def test_int8_converter_path_without_mirror(dev, layout):
    # a workspace with room for the plan only: query-tile requests convert each
    # int8 page per tile in the converter warps instead of reading the fp16
    # mirror; same bit-exact scores
    import block_score_gb300 as bs
    case = synth.make_case([2, 70, 1, 130], [300, 900, 128, 4100], H_q=16, H_kv=2,
                           layout=layout, q_dtype=torch.float16, k_dtype=torch.int8,
                           q_kind="int_small", k_kind="int8_full", scale_const=1.0,
                           MB=33, init_blocks=1, local_blocks=2, seed=360)
    prep = bs.from_case(case, dev)
    mirror = case.key.shape[0] * case.H_kv * case.P * case.D * 2
    assert prep.ws_bytes > mirror
    prep.ws_bytes -= mirror
    out = prep().cpu()
    assert prep.device_error() == 0
    assert_parity(out, oracle.oracle_full(case), exact=True, what=f"int8 converter path {layout}")


@pytest.mark.parametrize("layout", ["BBND", "BNBD"])
def test_int8_mirror_strided_cache(dev, layout):
    # int8 keys in a paged cache with a gap page after every page (dim0 stride
    # of two pages, the gaps filled with 127): the conversion into the fp16
    # mirror reads each page through the page stride; integer query, unit
    # scale, so the scores are exact
    case = synth.make_case([70, 1, 130], [900, 300, 4100], H_q=16, H_kv=2, layout=layout,
                           q_dtype=torch.float16, k_dtype=torch.int8, q_kind="int_small",
                           k_kind="int8_full", scale_const=1.0, MB=33, page_gap=2,
                           init_blocks=1, local_blocks=2, seed=370 + (layout == "BNBD"))
    assert case.key.stride(0) == 2 * case.key[0].numel()
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), exact=True, what=f"int8 mirror strided {layout}")


def test_strided_cache_poisoned_gaps(dev):
    case = synth.make_case([20, 3], [500, 260], H_q=8, H_kv=1, layout="BBND",
                           q_dtype=torch.float16, q_kind="abs_randn", MB=6, page_gap=2,
                           poison=1.0e4, seed=310)
    assert case.key.stride(0) == 2 * case.key[0].numel()
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    ref = oracle.oracle_full(case)
    assert_parity(out, ref, what="gap poison")
    assert float(out[torch.isfinite(out) & (out.abs() < 1e28)].max()) < 1.0e4


@pytest.mark.parametrize("width", [257, 275])
def test_wide_block_table(dev, width):
    case = synth.make_case([4, 2], [4, 275], H_q=8, H_kv=1, layout="BBND",
                           q_dtype=torch.float16, MB=width, seed=320 + width)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert out.shape[2] == (width + 15) // 16 * 16
    assert_parity(out, oracle.oracle_full(case), what=f"wide {width}")


def test_short_decode_and_speculative(dev):
    # q4-kv4, q4-kv275, q_len 3 speculative, single-token decode with g=16
    case = synth.make_case([4, 4, 3, 1, 1], [4, 275, 1000, 7000, 128], H_q=16, H_kv=1,
                           layout="BNBD", q_dtype=torch.bfloat16, MB=60, seed=330)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what="short decode")


def test_all_requests_empty(dev):
    case = synth.make_case([3, 5], [0, 0], H_q=4, H_kv=1, layout="BBND",
                           q_dtype=torch.float16, MB=3, init_blocks=1, seed=340)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert torch.isneginf(out).all()


@pytest.mark.parametrize("kdt", ["bf16", "int8"])
def test_batch_above_one_thousand_requests(dev, kdt):
    # more requests than the plan kernel has threads: the plan takes its
    # slice-by-slice path (and, for int8 keys, splits both request classes)
    rng = np.random.default_rng(77)
    B = 1100
    q = [int(x) for x in rng.integers(0, 4, size=B)]
    kv = [int(x) for x in rng.integers(0, 300, size=B)]
    kdtype = torch.int8 if kdt == "int8" else torch.bfloat16
    case = synth.make_case(q, kv, H_q=8, H_kv=2, layout="BBND",
                           q_dtype=torch.float16 if kdt == "int8" else torch.bfloat16,
                           k_dtype=kdtype, k_kind="int8_full" if kdt == "int8" else "randn",
                           MB=3, init_blocks=1, local_blocks=1, seed=378)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what=f"B=1100 {kdt}")


def test_group_size_not_a_power_of_two(dev):
    # g = 3: 42 positions x 3 heads = 126 of the 128 MMA rows are used
    case = synth.make_case([100, 50], [400, 90], H_q=6, H_kv=2, layout="BBND",
                           q_dtype=torch.float16, MB=4, seed=350)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what="g=3")


def test_plan_run_split_and_repeat_are_identical(dev):
    import block_score_gb300 as bs
    case = synth.make_case([50, 1], [900, 2000], H_q=16, H_kv=2, layout="BBND",
                           q_dtype=torch.bfloat16, MB=16, seed=360)
    prep = bs.from_case(case, dev)
    a = prep().clone()
    prep.out.fill_(7.0)
    prep.plan()
    b = prep.run().clone()
    c = prep().clone()
    assert torch.equal(a, b) and torch.equal(a, c)


def test_host_length_bound_skips_nothing_it_should_not(dev):
    # int8 decode batch (every request short): with the host bound the tile
    # kernel is not launched; the scores are the same bits as without it
    import block_score_gb300 as bs
    case = synth.make_case([1, 1, 2, 1], [700, 3000, 1500, 0], H_q=16, H_kv=2, layout="BBND",
                           q_dtype=torch.float16, k_dtype=torch.int8, k_kind="int8_full",
                           MB=30, init_blocks=1, local_blocks=2, seed=385)
    a = bs.from_case(case, dev)
    out_a = a().cpu()
    assert a.device_error() == 0
    b = bs.from_case(case, dev, max_seqlen_q=2)
    out_b = b().cpu()
    assert b.device_error() == 0
    assert torch.equal(out_a, out_b)
    assert_parity(out_b, oracle.oracle_full(case), what="host bound, int8 decode")
    # 16-bit keys have no short path: the bound changes nothing
    c16 = synth.make_case([1, 3], [900, 260], H_q=8, H_kv=1, layout="BNBD",
                          q_dtype=torch.bfloat16, MB=8, seed=386)
    o1 = bs.from_case(c16, dev)().cpu()
    o2 = bs.from_case(c16, dev, max_seqlen_q=3)().cpu()
    assert torch.equal(o1, o2)


def test_host_length_bound_that_is_broken_is_reported(dev):
    # a prefill request longer than the bound would have needed the tile kernel
    import block_score_gb300 as bs
    case = synth.make_case([1, 40], [700, 900], H_q=16, H_kv=2, layout="BBND",
                           q_dtype=torch.float16, k_dtype=torch.int8, k_kind="int8_full",
                           MB=8, seed=387)
    prep = bs.from_case(case, dev, max_seqlen_q=1)
    prep()
    assert prep.device_error() & 0x01


def test_bad_block_table_entry_is_reported_not_faulted(dev):
    case = synth.make_case([5], [300], H_q=4, H_kv=1, layout="BBND", q_dtype=torch.float16,
                           MB=4, seed=370)
    case.block_table[0, 1] = 10_000          # beyond NP, inside the needed range
    _, err, _ = run_gpu(case, dev)
    assert err & 0x08
    case.block_table[0, 1] = -3
    _, err, _ = run_gpu(case, dev)
    assert err & 0x08


def test_bad_lengths_are_reported(dev):
    case = synth.make_case([5], [300], H_q=4, H_kv=1, layout="BBND", q_dtype=torch.float16,
                           MB=4, seed=380)
    case.kv_len[0] = 600                      # needs 5 blocks, table has 4
    _, err, _ = run_gpu(case, dev)
    assert err & 0x02
    case.kv_len[0] = 300
    case.cu_seqlens_q[1] = 4                  # cu_q[B] != T
    _, err, _ = run_gpu(case, dev)
    assert err & 0x01


# ---------------------------------------------------------------------------
# the benchmark workloads at full size
# ---------------------------------------------------------------------------

def _sample_rows(case, n, seed):
    """Rows (h*T + t) spread over heads and tokens, plus each request's first/last token."""
    rng = np.random.default_rng(seed)
    T, H = case.T, case.H_q
    rows = set(int(x) for x in rng.integers(0, H * T, size=n))
    cu = case.cu_seqlens_q.tolist()
    for b in range(len(cu) - 1):
        if cu[b + 1] > cu[b]:
            for t in (cu[b], cu[b + 1] - 1):
                h = int(rng.integers(0, H))
                rows.add(h * T + t)
    return sorted(rows)


def _structural_checks(out, case):
    """Properties of the whole output that hold at any size."""
    MB, MBp, P = case.MB, case.MBp, case.P
    assert torch.isneginf(out[:, :, MB:]).all()
    cu = case.cu_seqlens_q.tolist()
    for b in range(len(cu) - 1):
        t0, t1 = cu[b], cu[b + 1]
        if t1 == t0:
            continue
        L = case.kv_lens[b]
        blk = out[:, t0:t1, :MB]
        if L == 0:
            assert torch.isneginf(blk).all()
            continue
        sl = int(case.start_loc[b])
        lo = max(0, sl + 1 - case.local_blocks)
        forced = torch.zeros(MB, dtype=torch.bool)
        forced[:min(case.init_blocks, MB)] = True
        if sl >= lo:
            forced[lo:min(sl, MB - 1) + 1] = True
        if case.init_blocks:
            init_cols = [c for c in range(min(case.init_blocks, MB)) if not (lo <= c <= sl)]
            if init_cols:
                assert (blk[:, :, init_cols] == np.float32(1e30)).all()
        if sl >= lo and lo < MB:
            assert (blk[:, :, lo:min(sl, MB - 1) + 1] == np.float32(1e29)).all()
        nb = -(-L // P)
        if nb < MB:
            tail = blk[:, :, nb:][:, :, ~forced[nb:]]
            assert torch.isneginf(tail).all()


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_benchmark_workload_sampled(dev, n):
    case = synth.config(n)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    _structural_checks(out, case)
    rows = _sample_rows(case, 512 if n != 5 else 256, seed=n)
    ref = oracle.oracle_rows(case, rows)
    got = out.reshape(-1, out.shape[2])[torch.tensor(rows)]
    assert_parity(got, ref, what=f"cfg{n} sampled")


def test_batched_decode_workload_full(dev):
    case = synth.config(2)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what="cfg2 full")


# ------------------------------------------------------------------ FP8 inputs
# FP8 query and key of one type, no scale (torch API guide, sec. 4 and 7.2),
# on tcgen05 kind::f8f6f4: the products are exact in fp32, so the scores stay
# within the fp16 path's tolerance of the fp64 oracle.

@pytest.mark.parametrize("layout", ["BBND", "BNBD", "TND"])
@pytest.mark.parametrize("dt", [torch.float8_e4m3fn, torch.float8_e5m2])
def test_fp8_layout_matrix_mixed_batch(dev, layout, dt):
    q = [37, 1, 0, 4, 200, 1]
    kv = [290, 1, 77, 0, 600, 4100]
    case = synth.make_case(q, kv, H_q=16, H_kv=2, layout=layout, q_dtype=dt, k_dtype=dt,
                           MB=None if layout == "TND" else 40, init_blocks=1, local_blocks=2,
                           seed=300 + len(layout) + (dt == torch.float8_e5m2))
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), what=f"{layout}/{dt}")


@pytest.mark.parametrize("g", [1, 8, 3])
def test_fp8_gqa_groups_and_modes(dev, g):
    dt = torch.float8_e4m3fn
    for mode in (0, 3):
        case = synth.make_case([130, 9, 1], [1000, 140, 333], H_q=2 * g, H_kv=2, layout="BBND",
                               q_dtype=dt, k_dtype=dt, sparse_mode=mode, MB=12, init_blocks=0,
                               local_blocks=1, seed=310 + g + mode)
        out, err, _ = run_gpu(case, dev)
        assert err == 0
        assert_parity(out, oracle.oracle_full(case), what=f"fp8 g={g} mode={mode}")


def test_fp8_integer_inputs_bit_exact(dev):
    # integers in [-8, 8] are exact in E4M3; products and 128-term sums are exact in fp32
    dt = torch.float8_e4m3fn
    case = synth.make_case([70, 1], [500, 260], H_q=8, H_kv=1, layout="BNBD", q_dtype=dt, k_dtype=dt,
                           q_kind="int_small", k_kind="int_small", MB=6, seed=320)
    out, err, _ = run_gpu(case, dev)
    assert err == 0
    assert_parity(out, oracle.oracle_full(case), exact=True, what="fp8 integers")


def test_fp8_validation():
    import block_score_gb300 as bs
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda:0")
    q = torch.zeros(4, 2, 128, device=d).to(torch.float8_e4m3fn)
    k = torch.zeros(2, 128, 1, 128, device=d).to(torch.float8_e5m2)
    args = dict(block_table=torch.zeros(1, 2, dtype=torch.int32, device=d),
                actual_seq_qlen=torch.tensor([0, 4], dtype=torch.int32, device=d),
                actual_seq_klen=torch.tensor([100], dtype=torch.int32, device=d))
    with pytest.raises(ValueError):   # mixed fp8 types
        bs.msa_index_score(q, k, torch.zeros(1, dtype=torch.int32, device=d), **args)
    with pytest.raises(ValueError):   # a scale with fp8
        bs.msa_index_score(q, k.to(torch.float32).to(torch.float8_e4m3fn),
                           torch.zeros(1, dtype=torch.int32, device=d),
                           scale=torch.ones(2, 1, 128, device=d), **args)
