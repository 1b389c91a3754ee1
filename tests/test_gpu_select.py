"""GPU parity of the fused per-GQA-group block selection (msa_index_score_topk).

The selection is integer work on fp32 scores, so it is checked bit for bit:
the oracle's per-group selection (oracle/topk.py, group_topk: MiniMax Sparse
Attention notes, section 4.3 Equation (3), section 4.7 Equation (7), section
10 items 7-9) is applied to the scores of the same inputs computed by
msa_index_score, and must give exactly the fused call's indices.  The fused
call's own scores must equal msa_index_score's bit for bit, and without the
own-block slot the selection must equal msa_block_topk over the group maxima.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import topk as otk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_score_gb300 as bs
    bs.load_library()
    return torch.device("cuda:0")


def _check(case, dev, k, local_slot, g):
    import block_score_gb300 as bs
    prep = bs.from_case(case, dev)
    ref = prep().clone()
    assert prep.device_error() == 0
    # fused call that also stores the scores: same scores, bit for bit
    prep.out.fill_(float("nan"))
    idx = prep.topk(k, local_slot=local_slot, scores=True)
    assert prep.select_device_error() == 0
    assert torch.equal(prep.out, ref)
    # the selection on the oracle's side, from the same scores
    local = otk.local_blocks_of(case) if local_slot else None
    want = otk.group_topk(ref.cpu(), g, case.MB, k, local=local)
    got = idx.cpu().numpy()
    bad = np.argwhere((got != want).any(axis=2))
    assert bad.size == 0, f"{len(bad)} rows differ, first (t, group) {bad[:4].tolist()}: " \
                          f"gpu {got[tuple(bad[0])].tolist()} oracle {want[tuple(bad[0])].tolist()}"
    # without storing the scores: the same selection, the output untouched
    prep.out.fill_(float("nan"))
    idx2 = prep.topk(k, local_slot=local_slot, scores=False)
    assert torch.equal(idx2, idx)
    assert bool(torch.isnan(prep.out).all())
    if not local_slot:
        # the unfused selector over the group maxima gives the same indices
        H, T, MBp = ref.shape
        gmax = ref.reshape(H // g, g, T, MBp).amax(dim=1).contiguous()
        unf = bs.msa_block_topk(gmax, k=k, MB=case.MB)
        assert torch.equal(unf, idx)
    return idx


CASES = {
    # bf16 prefill: several query tiles per request, ragged tails, GQA g=8
    "bf16_prefill_g8": dict(q=[70, 1, 0, 33, 300], kv=[700, 130, 50, 33, 2000], H_q=16, H_kv=2,
                            layout="BBND", q_dtype=torch.bfloat16, k_dtype=None, MB=20),
    # decode batch: many KV chunks per request, g=16
    "bf16_decode_g16": dict(q=[1] * 9, kv=[30000, 128, 1, 5000, 64000, 17, 9000, 257, 40000],
                            H_q=16, H_kv=1, layout="BBND", q_dtype=torch.bfloat16, k_dtype=None,
                            MB=512),
    # fp16 BNBD, g=1 (one index head per group, the paper's layout), mode 0
    "fp16_bnbd_g1_mode0": dict(q=[40, 3, 1], kv=[900, 4000, 128], H_q=4, H_kv=4, layout="BNBD",
                               q_dtype=torch.float16, k_dtype=None, MB=40, sparse_mode=0),
    # int8 keys: tile kernel (Lq 200) and short-query kernel (Lq 1..4 with g=8)
    "int8_mixed_g8": dict(q=[1, 200, 2, 1, 4, 0], kv=[9000, 3000, 700, 1, 4100, 10],
                          H_q=16, H_kv=2, layout="BBND", q_dtype=torch.float16,
                          k_dtype=torch.int8, MB=80),
    # packed TND keys, g=4
    "fp16_tnd_g4": dict(q=[50, 1, 7], kv=[3000, 600, 129], H_q=8, H_kv=2, layout="TND",
                        q_dtype=torch.float16, k_dtype=None, MB=None),
    # FP8 E4M3, g=2
    "e4m3_g2": dict(q=[33, 1], kv=[5000, 2000], H_q=4, H_kv=2, layout="BBND",
                    q_dtype=torch.float8_e4m3fn, k_dtype=torch.float8_e4m3fn, MB=48),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("local_slot", [False, True])
def test_fused_group_selection(dev, name, local_slot):
    c = dict(CASES[name])
    g = c["H_q"] // c["H_kv"]
    case = synth.make_case(c.pop("q"), c.pop("kv"), init_blocks=2, local_blocks=3,
                           seed=sum(map(ord, name)), **c)
    for k in (16, 5):
        _check(case, dev, k, local_slot, g)


def test_fused_selection_k1_and_empty_rows(dev):
    # k = 1 with the own-block slot keeps only the own block; kv_len = 0 rows
    # select nothing
    case = synth.make_case([5, 3], [900, 0], H_q=8, H_kv=1, layout="BBND",
                           q_dtype=torch.float16, MB=8, init_blocks=0, local_blocks=0, seed=990)
    idx = _check(case, dev, 1, True, 8)
    assert idx[:5, 0, 0].tolist() == [6, 7, 7, 7, 7]   # q_pos 895..899 // 128
    assert (idx[5:] == -1).all()


def test_fused_selection_rejects_what_it_does_not_build(dev):
    import block_score_gb300 as bs
    case = synth.make_case([4], [300], H_q=6, H_kv=2, layout="BBND", q_dtype=torch.float16,
                           MB=3, seed=991)
    prep = bs.from_case(case, dev)
    with pytest.raises(Exception):
        prep.topk(4)                                    # g = 3 does not divide 32
    case = synth.make_case([4], [300], H_q=8, H_kv=2, layout="BBND", q_dtype=torch.float16,
                           MB=3, seed=992)
    prep = bs.from_case(case, dev)
    with pytest.raises(Exception):
        prep.topk(17)


@pytest.mark.parametrize("n", [2, 5])
def test_fused_selection_on_the_benchmark_workloads(dev, n):
    # batched decode: every row; long-context prefill: sampled tokens
    import block_score_gb300 as bs
    case = synth.config(n)
    g = case.H_q // case.H_kv
    prep = bs.from_case(case, dev)
    ref = prep()
    idx = prep.topk(16, local_slot=True, scores=False).cpu().numpy()
    assert prep.select_device_error() == 0
    local = otk.local_blocks_of(case)
    if n == 2:
        want = otk.group_topk(ref.cpu(), g, case.MB, 16, local=local)
        assert np.array_equal(idx, want)
        return
    rng = np.random.default_rng(5)
    ts = np.unique(np.concatenate([rng.integers(0, case.T, 64), [0, case.T - 1]]))
    sub = ref[:, torch.as_tensor(ts, device=ref.device), :].cpu()
    want = otk.group_topk(sub, g, case.MB, 16, local=local[ts])
    assert np.array_equal(idx[ts], want)
