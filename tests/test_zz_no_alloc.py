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
