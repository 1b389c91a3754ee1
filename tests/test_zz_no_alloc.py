"""The allocation-free entry point against the workspace entry point.

msa_index_score_noalloc serves callers that cannot allocate device memory
(its plan scratch is a fixed array inside the library).  It must give the
same scores as msa_index_score, call after call, although every call reuses
and overwrites the same array.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-3, 1e-4


def _close(a, b):
    inf = torch.isinf(b)
    assert torch.equal(torch.isinf(a), inf)
    assert torch.equal(a[inf], b[inf])
    fin = ~inf
    assert bool(((a[fin] - b[fin]).abs() <= ATOL + RTOL * b[fin].abs()).all())


KEYS = {
    "bf16": (torch.bfloat16, None),
    "int8": (torch.float16, torch.int8),          # tile and short-query kernels
    "e4m3": (torch.float8_e4m3fn, torch.float8_e4m3fn),
}


@pytest.mark.parametrize("keys", sorted(KEYS))
def test_noalloc_matches_workspace_entry_on_two_calls(keys):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_score_gb300 as bs
    lib = bs.load_library()
    dev = torch.device("cuda:0")
    q_dtype, k_dtype = KEYS[keys]
    # a mixed batch: prefill tiles, single-token decode, an empty request, forced blocks
    case = synth.make_case([37, 1, 0, 4, 130], [290, 3000, 77, 4, 900], H_q=16, H_kv=2,
                           layout="BBND", q_dtype=q_dtype, k_dtype=k_dtype, MB=24,
                           init_blocks=1, local_blocks=2, seed=901)
    prep = bs.from_case(case, dev)
    ref = prep().clone().cpu()
    stream = torch.cuda.current_stream(dev)
    for _ in range(2):
        out = torch.full(prep.shape, float("nan"), dtype=torch.float32, device=dev)
        st = lib.msa_index_score_noalloc(ctypes.byref(prep.call.args), out.data_ptr(),
                                         stream.cuda_stream)
        assert st == 0, lib.msa_last_error_message()
        torch.cuda.synchronize(dev)
        _close(out.cpu(), ref)


def test_noalloc_rejects_batches_above_its_limit():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_score_gb300 as bs
    lib = bs.load_library()
    case = synth.make_case([1, 1], [10, 10], H_q=4, H_kv=1, layout="BBND",
                           q_dtype=torch.float16, MB=1, seed=902)
    prep = bs.from_case(case, torch.device("cuda:0"))
    args = prep.call.args
    saved = args.B
    args.B = 1025
    try:
        st = lib.msa_index_score_noalloc(ctypes.byref(args), prep.out.data_ptr(), None)
    finally:
        args.B = saved
    assert st == 5
    assert b"at most 1024" in lib.msa_last_error_message()


def test_noalloc_back_to_back_calls_without_a_sync():
    # two different calls enqueued on one stream with nothing between them: the
    # second call's plan kernel rewrites the shared array while it is ordered
    # after the first call's score kernels on the stream; the int8 case runs the
    # plan -> tile -> short-query chain
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_score_gb300 as bs
    bs.load_library()
    dev = torch.device("cuda:0")
    a = synth.make_case([1, 1, 2, 130, 1], [9000, 300, 700, 1500, 4100], H_q=16, H_kv=2,
                        layout="BBND", q_dtype=torch.float16, k_dtype=torch.int8, MB=72,
                        init_blocks=1, local_blocks=2, seed=911)
    b = synth.make_case([64, 1, 0], [5000, 128, 10], H_q=8, H_kv=1, layout="BNBD",
                        q_dtype=torch.bfloat16, MB=48, seed=912)
    pa, pb = bs.from_case(a, dev), bs.from_case(b, dev)
    ref_a, ref_b = pa().clone().cpu(), pb().clone().cpu()
    stream = torch.cuda.current_stream(dev)
    for _ in range(2):
        oa = torch.full(pa.shape, float("nan"), dtype=torch.float32, device=dev)
        ob = torch.full(pb.shape, float("nan"), dtype=torch.float32, device=dev)
        torch.cuda.synchronize(dev)
        bs.msa_index_score_noalloc(pa, oa, stream)
        bs.msa_index_score_noalloc(pb, ob, stream)
        bs.msa_index_score_noalloc(pa, oa, stream)
        assert bs.noalloc_device_error(stream) == 0
        _close(oa.cpu(), ref_a)
        _close(ob.cpu(), ref_b)


def test_noalloc_device_error_word_is_readable():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_score_gb300 as bs
    bs.load_library()
    dev = torch.device("cuda:0")
    case = synth.make_case([5], [300], H_q=4, H_kv=1, layout="BBND", q_dtype=torch.float16,
                           MB=4, seed=913)
    case.block_table[0, 1] = 10_000          # beyond NP, inside the needed range
    prep = bs.from_case(case, dev)
    bs.msa_index_score_noalloc(prep)
    assert bs.noalloc_device_error() & 0x08
    # the next clean call clears the word
    good = bs.from_case(synth.make_case([5], [300], H_q=4, H_kv=1, layout="BBND",
                                        q_dtype=torch.float16, MB=4, seed=914), dev)
    bs.msa_index_score_noalloc(good)
    assert bs.noalloc_device_error() == 0


def test_noalloc_binding_checks_out():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_score_gb300 as bs
    bs.load_library()
    dev = torch.device("cuda:0")
    prep = bs.from_case(synth.make_case([3], [200], H_q=4, H_kv=1, layout="BBND",
                                        q_dtype=torch.float16, MB=2, seed=915), dev)
    small = torch.empty((4, 3, 8), dtype=torch.float32, device=dev)
    with pytest.raises(ValueError):
        bs.msa_index_score_noalloc(prep, small)
