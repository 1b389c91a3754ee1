"""GPU parity of the sparse main branch (msa_sparse_attention) against the
oracle (oracle/sparse_attention.py: MiniMax Sparse Attention notes, sec. 4.8
Equation (8), in float64).

Tolerance, from the arithmetic, with u the unit roundoff of the input's 16-bit
type (2^-8 for bf16's 8-bit significand, 2^-11 for fp16's 11 bits): scores are
exact products of 16-bit values summed in fp32; the softmax weights p_j (fp32,
normalised per block by their fp32 sum l) are rounded to 16 bits before the
P V product, so a block's partial output is off by at most u * max_j |v_j|;
the partial is stored in the same 16-bit type, another u * max|V|; the merge
of the partials is a convex combination, so it adds nothing beyond its fp32
weights, which with the exp2 / log2 approximations are accurate to about
1e-6 relative.  The test allows |dO| <= 2 u max|V| + 1e-5 and
|dLSE| <= 1e-4 + 1e-5 * |LSE|; empty rows must be exactly O = 0, LSE = -inf.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import topk as otk
from oracle.sparse_attention import sparse_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_score_gb300 as bs
    bs.load_library()
    return torch.device("cuda:0")


def value_like(case, seed):
    g = torch.Generator().manual_seed(seed)
    k = case.key
    base = k
    while base._base is not None:
        base = base._base
    vb = torch.randn(base.shape, generator=g).to(k.dtype)
    return torch.as_strided(vb, k.shape, k.stride(), k.storage_offset())


def to_dev(view, dev):
    base = view
    while base._base is not None:
        base = base._base
    return torch.as_strided(base.to(dev), view.shape, view.stride(), view.storage_offset())


def random_selection(case, k, seed, beyond=True):
    """Ascending distinct blocks per (token, group), -1 tail; some rows select
    blocks past their last block (skipped by the op)."""
    rng = np.random.default_rng(seed)
    sel = np.full((case.T, case.H_kv, k), -1, dtype=np.int32)
    cu = case.cu_seqlens_q.tolist()
    for b in range(case.B):
        nb = -(-case.kv_lens[b] // case.P)
        top = min(case.MB, nb + (2 if beyond else 0))
        for t in range(cu[b], cu[b + 1]):
            for r in range(case.H_kv):
                n = int(rng.integers(0, min(k, top) + 1)) if top else 0
                if n:
                    sel[t, r, :n] = np.sort(rng.choice(top, n, replace=False))
    return torch.from_numpy(sel)


def check(case, dev, sel, value, sm_scale=0.0):
    import block_score_gb300 as bs
    prep = bs.from_case(case, dev)
    out, lse = prep.sparse_attention(to_dev(value, dev), sel.to(dev), sm_scale=sm_scale)
    assert prep.sparse_device_error() == 0
    O_ref, L_ref = sparse_attention(case, value, sel, sm_scale=sm_scale or None)
    out, lse = out.cpu().double().numpy(), lse.cpu().double().numpy()
    empty = np.isneginf(L_ref)
    assert np.array_equal(np.isneginf(lse), empty)
    assert np.all(out[empty] == 0)
    vmax = float(value.abs().max())
    u = 2.0 ** -8 if value.dtype == torch.bfloat16 else 2.0 ** -11
    dO = np.abs(out[~empty] - O_ref[~empty])
    assert dO.max(initial=0) <= 2 * u * vmax + 1e-5, f"max |dO| {dO.max():.3e} (vmax {vmax:.2f})"
    dL = np.abs(lse[~empty] - L_ref[~empty])
    assert (dL <= 1e-4 + 1e-5 * np.abs(L_ref[~empty])).all(), f"max |dLSE| {dL.max():.3e}"
    return out, lse


CASES = {
    # prefill and decode requests, GQA g = 8, BBND bf16
    "bf16_bbnd_g8": dict(q=[37, 1, 0, 4, 200, 1], kv=[290, 1, 77, 0, 900, 4100], H_q=16, H_kv=2,
                         layout="BBND", dt=torch.bfloat16, MB=40, mode=3),
    # fp16 BNBD, g = 1, no causal bound
    "f16_bnbd_g1_mode0": dict(q=[40, 3], kv=[700, 2000], H_q=4, H_kv=4, layout="BNBD",
                              dt=torch.float16, MB=20, mode=0),
    # packed TND keys and values, g = 16 (8 query positions per unit)
    "bf16_tnd_g16": dict(q=[70, 1, 5], kv=[1500, 600, 129], H_q=16, H_kv=1, layout="TND",
                         dt=torch.bfloat16, MB=None, mode=3),
    # g = 3 (42 positions x 3 heads = 126 rows per unit)
    "bf16_bbnd_g3": dict(q=[50, 9], kv=[800, 300], H_q=6, H_kv=2, layout="BBND",
                         dt=torch.bfloat16, MB=8, mode=3),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("k", [16, 3])
def test_sparse_attention_random_selection(dev, name, k):
    c = CASES[name]
    case = synth.make_case(c["q"], c["kv"], H_q=c["H_q"], H_kv=c["H_kv"], layout=c["layout"],
                           q_dtype=c["dt"], MB=c["MB"], sparse_mode=c["mode"],
                           seed=sum(map(ord, name)) + k)
    value = value_like(case, 500 + k)
    sel = random_selection(case, k, seed=k)
    check(case, dev, sel, value)


def test_sparse_attention_on_the_fused_selection(dev):
    # the index branch's fused per-group selection feeds the main branch
    import block_score_gb300 as bs
    case = synth.make_case([300, 1, 64], [2000, 5000, 900], H_q=16, H_kv=2, layout="BBND",
                           q_dtype=torch.bfloat16, MB=40, init_blocks=1, local_blocks=2, seed=520)
    prep = bs.from_case(case, dev)
    sel = prep.topk(16, local_slot=True, scores=False).cpu()
    value = value_like(case, 521)
    check(case, dev, sel, value, sm_scale=0.125)


def test_sparse_attention_strided_cache_and_full_selection(dev):
    # every block selected: plain causal attention over the request
    case = synth.make_case([20, 3], [500, 260], H_q=8, H_kv=1, layout="BBND",
                           q_dtype=torch.float16, MB=6, page_gap=2, seed=522)
    value = value_like(case, 523)
    sel = torch.full((case.T, 1, 8), -1, dtype=torch.int32)
    sel[:20, 0, :4] = torch.arange(4)
    sel[20:, 0, :3] = torch.arange(3)
    check(case, dev, sel, value)


def test_sparse_attention_reports_a_bad_selection(dev):
    import block_score_gb300 as bs
    case = synth.make_case([3], [500], H_q=4, H_kv=1, layout="BBND", q_dtype=torch.bfloat16,
                           MB=4, seed=524)
    prep = bs.from_case(case, dev)
    value = to_dev(value_like(case, 525), dev)
    sel = torch.tensor([[[2, 1, -1]], [[0, 0, -1]], [[1, 3, -1]]], dtype=torch.int32, device=dev)
    prep.sparse_attention(value, sel)
    assert prep.sparse_device_error() & 0x20


@pytest.mark.parametrize("n", [3, 5])
def test_sparse_attention_benchmark_workload_sampled(dev, n):
    # the bench's sparse record at full size (varlen prefill; long-context
    # prefill, T = 16384 at kv_len 131072): the fused top-16 selection of the
    # workload, random values in the key cache's layout, 256 sampled (token,
    # head) rows against the oracle
    import block_score_gb300 as bs
    case = synth.config(n)
    prep = bs.from_case(case, dev)
    sel = prep.topk(16, local_slot=True, scores=False)
    assert prep.select_device_error() == 0
    value = value_like(case, seed=90 + n)
    out, lse = prep.sparse_attention(to_dev(value, dev), sel)
    assert prep.sparse_device_error() == 0
    rng = np.random.default_rng(n)
    rows = np.sort(rng.choice(case.T * case.H_q, 256, replace=False))
    O_ref, L_ref = sparse_attention(case, value, sel.cpu(), rows=rows.tolist())
    t, h = rows // case.H_q, rows % case.H_q
    got_o = out.cpu().double().numpy()[t, h]
    got_l = lse.cpu().double().numpy()[t, h]
    ref_o, ref_l = O_ref[t, h], L_ref[t, h]
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(got_l), empty)
    assert np.all(got_o[empty] == 0)
    u = 2.0 ** -8 if value.dtype == torch.bfloat16 else 2.0 ** -11
    dO = np.abs(got_o[~empty] - ref_o[~empty])
    assert dO.max(initial=0) <= 2 * u * float(value.abs().max()) + 1e-5
    dL = np.abs(got_l[~empty] - ref_l[~empty])
    assert (dL <= 1e-4 + 1e-5 * np.abs(ref_l[~empty])).all()
