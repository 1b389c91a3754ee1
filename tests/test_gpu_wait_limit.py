"""Bounded pipeline waits: a wait that runs out ends the call with an error
status instead of hanging the GPU, and the next call is clean.

The score kernels give every on-chip wait a wall-clock limit (default 4 s).
Here the watchdog's test stall makes the warp that feeds each CTA's
tensor-core issuer wait on a barrier that nothing completes, under a 20 ms
limit: the call must still return, the device error word must carry
MSA_DEVERR_TIMEOUT (0x10), the context must stay usable, and a call with the
default limit restored must match the oracle.
"""
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TIMEOUT = 0x10
ATOL, RTOL = 1e-3, 1e-4


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_score_gb300 as bs
    bs.load_library()
    return torch.device("cuda:0")


def _close(out, ref):
    inf = torch.isinf(ref)
    assert torch.equal(torch.isinf(out), inf)
    assert torch.equal(out[inf], ref[inf])
    fin = ~inf
    assert bool(((out[fin].double() - ref[fin].double()).abs()
                 <= ATOL + RTOL * ref[fin].double().abs()).all())


CASES = {
    # 16-bit keys: the tile kernel (scheduler, producer, MMA warp and helper, epilogue)
    "bf16_decode": dict(q=[1] * 12 + [40], kv=[9000, 20000, 31000, 4000, 15000, 26000,
                                               12000, 7000, 30000, 18000, 25000, 11000, 6000],
                        H_q=16, H_kv=1, q_dtype=torch.bfloat16, k_dtype=None, MB=256),
    # int8 keys: the tile kernel's converter warps and the short-query kernel
    "int8_mixed": dict(q=[1] * 10 + [200, 3], kv=[9000, 20000, 31000, 4000, 15000, 26000,
                                                  12000, 7000, 30000, 18000, 6000, 9000],
                       H_q=16, H_kv=2, q_dtype=torch.float16, k_dtype=torch.int8, MB=256),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_wait_that_runs_out_returns_an_error_and_the_next_call_is_clean(dev, name):
    import block_score_gb300 as bs
    lib = bs.load_library()
    c = CASES[name]
    case = synth.make_case(c["q"], c["kv"], H_q=c["H_q"], H_kv=c["H_kv"], layout="BBND",
                           q_dtype=c["q_dtype"], k_dtype=c["k_dtype"], MB=c["MB"],
                           init_blocks=1, local_blocks=2, seed=960)
    prep = bs.from_case(case, dev)
    torch.cuda.synchronize(dev)
    assert lib.msa_set_watchdog(20_000_000, 1) == 0
    try:
        prep()
        err = prep.device_error()          # synchronises: the kernels returned
    finally:
        lib.msa_set_watchdog(0, 0)
    assert err & TIMEOUT, f"error bits {err:#x}"
    torch.cuda.synchronize(dev)            # the context is still usable
    out = prep().cpu()
    assert prep.device_error() == 0
    _close(out, oracle.oracle_full(case))
