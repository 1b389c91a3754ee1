"""C-ABI library checks that need no GPU: it builds, loads, exports every
declared entry point, and its host-side argument rules behave as documented."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa_index_score.h")


@pytest.fixture(scope="module")
def lib():
    from block_score_gb300 import _build
    _build.build()
    import block_score_gb300 as bs
    return bs.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w \*]*?\b(msa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for want in ("msa_index_score", "msa_index_score_plan", "msa_index_score_run",
                 "msa_index_score_out_shape", "msa_index_score_workspace_size",
                 "msa_get_device_error", "msa_status_string", "msa_last_error_message",
                 "msa_abi_version", "msa_block_topk"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_library_is_sm103a_only():
    from block_score_gb300 import _build
    assert "arch=compute_103a,code=sm_103a" in _build.ARCH


def test_abi_version(lib):
    assert lib.msa_abi_version() == 3


def _args(**over):
    import block_score_gb300 as bs
    a = bs._Args()
    base = dict(query=16, q_dtype=1, T=32, H_q=8, D=128, key_cache=16, k_dtype=1, layout=0, NP=8,
                P=128, H_kv=1, page_stride=128 * 128, block_table=16, B=1, MB=2,
                cu_seqlens_q=16, kv_len=16, cu_seqlens_k=None, start_loc=16, scale=None,
                sparse_mode=3, init_blocks=0, local_blocks=1)
    base.update(over)
    for k, v in base.items():
        setattr(a, k, v)
    return a


def _shape(lib, a):
    shape = (ctypes.c_int64 * 3)()
    st = lib.msa_index_score_out_shape(ctypes.byref(a), shape)
    return st, tuple(shape)


def test_out_shape_rounds_mb_to_16(lib):
    st, shape = _shape(lib, _args(MB=2))
    assert st == 0 and shape == (8, 32, 16)
    st, shape = _shape(lib, _args(MB=1100))
    assert st == 0 and shape == (8, 32, 1104)
    st, shape = _shape(lib, _args(MB=257))
    assert st == 0 and shape == (8, 32, 272)


def test_workspace_holds_the_int8_key_mirror(lib):
    # int8 paged keys: the plan plus an fp16 copy of the pages [NP, H_kv, P, D];
    # TND int8 keys and 16-bit keys: the plan only
    plan, i8, i8_tnd = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.msa_index_score_workspace_size(ctypes.byref(_args()), ctypes.byref(plan)) == 0
    a = _args(k_dtype=2, q_dtype=0, scale=16)
    assert lib.msa_index_score_workspace_size(ctypes.byref(a), ctypes.byref(i8)) == 0
    assert i8.value == plan.value + a.NP * a.H_kv * a.P * a.D * 2
    t = _args(k_dtype=2, q_dtype=0, scale=16, layout=2, block_table=None, kv_len=None,
              cu_seqlens_k=16, page_stride=128)
    assert lib.msa_index_score_workspace_size(ctypes.byref(t), ctypes.byref(i8_tnd)) == 0
    assert i8_tnd.value == plan.value


def test_workspace_size_grows_with_batch(lib):
    n1, n2 = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.msa_index_score_workspace_size(ctypes.byref(_args(B=1)), ctypes.byref(n1)) == 0
    assert lib.msa_index_score_workspace_size(ctypes.byref(_args(B=5000)), ctypes.byref(n2)) == 0
    assert n1.value >= 256 and n2.value > n1.value and n2.value % 256 == 0


@pytest.mark.parametrize("over,status", [
    (dict(layout=7), 1),                        # layout outside BBND/BNBD/TND
    (dict(sparse_mode=1), 1),                   # modes 0 and 3 only
    (dict(H_q=9, H_kv=2), 1),                   # H_q % H_kv
    (dict(D=64), 2),                            # scope of this library
    (dict(P=64, page_stride=64 * 128), 2),
    (dict(k_dtype=2, q_dtype=1, scale=16), 1),  # int8 keys need an fp16 query
    (dict(k_dtype=2, q_dtype=0, scale=None), 1),  # int8 keys need a scale
    (dict(scale=16), 1),                        # scale only with int8 keys
    (dict(k_dtype=0), 1),                       # key dtype must match query
    (dict(init_blocks=3), 1),                   # init_blocks <= MB
    (dict(local_blocks=-1), 1),
    (dict(layout=2, block_table=16, kv_len=None, cu_seqlens_k=16, page_stride=128), 1),
    (dict(layout=2, block_table=None, kv_len=16, cu_seqlens_k=None, page_stride=128), 1),
    (dict(page_stride=100), 1),                 # smaller than a compact page
    (dict(H_q=256, H_kv=1), 2),                 # GQA group above 128 rows
    (dict(query=17), 1),                        # TMA needs 16-byte aligned bases
    (dict(B=0, T=4), 1),
])
def test_host_validation(lib, over, status):
    st, _ = _shape(lib, _args(**over))
    assert st == status
    assert lib.msa_last_error_message()


def test_tnd_init_blocks_may_reach_padded_width(lib):
    # guide sec. 10: TND bounds init/local by the 16-aligned score width
    st, _ = _shape(lib, _args(layout=2, block_table=None, kv_len=None, cu_seqlens_k=16,
                              page_stride=128, MB=3, init_blocks=16))
    assert st == 0


def test_status_strings(lib):
    for s in range(6):
        assert lib.msa_status_string(s)


def test_python_binding_rejects_bad_layout_key():
    import block_score_gb300 as bs
    q = torch.zeros(4, 2, 128, dtype=torch.float16)
    k = torch.zeros(2, 128, 1, 128, dtype=torch.float16)
    with pytest.raises(ValueError):
        bs.msa_index_score_out_shape(q, k, torch.zeros(1, dtype=torch.int32),
                                     layout_key="bshd",
                                     actual_seq_qlen=torch.tensor([0, 4], dtype=torch.int32),
                                     actual_seq_klen=torch.tensor([10], dtype=torch.int32),
                                     block_table=torch.zeros(1, 1, dtype=torch.int32))


def test_python_binding_unsqueezes_3d_bbnd_key():
    import block_score_gb300 as bs
    q = torch.zeros(4, 2, 128, dtype=torch.float16)
    k = torch.zeros(2, 128, 128, dtype=torch.float16)   # [NP, P, D] -> N2 = 1
    shape = bs.msa_index_score_out_shape(
        q, k, torch.zeros(1, dtype=torch.int32), layout_key="bbnd",
        actual_seq_qlen=torch.tensor([0, 4], dtype=torch.int32),
        actual_seq_klen=torch.tensor([10], dtype=torch.int32),
        block_table=torch.zeros(1, 3, dtype=torch.int32))
    assert shape == (2, 4, 16)


@pytest.mark.parametrize("H,T,MBp,MB,k,status", [
    (2, 3, 16, 6, 0, 1),      # k below 1
    (2, 3, 16, 6, 33, 1),     # k above 32
    (2, 3, 16, 17, 4, 1),     # MB > MBp
    (-1, 3, 16, 6, 4, 1),     # negative size
    (0, 3, 16, 6, 4, 0),      # no rows: nothing to do, no launch
    (2, 0, 16, 6, 4, 0),
])
def test_block_topk_host_validation(lib, H, T, MBp, MB, k, status):
    assert lib.msa_block_topk(None, H, T, MBp, MB, k, None, None) == status


def test_fp4_host_rules(lib):
    # E2M1 (FP4) query and key: page_stride counts bytes (D/2 per row); the
    # output shape is the usual one; the 16-bit entry points refuse FP4 args
    fp4 = dict(q_dtype=5, k_dtype=5, page_stride=128 * 64)
    st, shape = _shape(lib, _args(**fp4))
    assert st == 0 and shape == (8, 32, 16)
    n = ctypes.c_size_t()
    assert lib.msa_index_score_fp4_workspace_size(ctypes.byref(_args(**fp4)), 1, ctypes.byref(n)) == 0
    plan = ctypes.c_size_t()
    assert lib.msa_index_score_workspace_size(ctypes.byref(_args()), ctypes.byref(plan)) == 0
    # + the dequantised query + (T * g >= 128 * B: a prefill-heavy call) the
    # 16-bit mirror of the key pages [NP, H_kv, P, D]
    assert n.value == plan.value + 32 * 8 * 128 * 2 + 8 * 1 * 128 * 128 * 2
    # a decode-heavy call (T * g < 128 * B): no mirror
    nd, pd = ctypes.c_size_t(), ctypes.c_size_t()
    dec = dict(fp4, T=2, B=2)
    assert lib.msa_index_score_fp4_workspace_size(ctypes.byref(_args(**dec)), 1, ctypes.byref(nd)) == 0
    assert lib.msa_index_score_workspace_size(ctypes.byref(_args(T=2, B=2)), ctypes.byref(pd)) == 0
    assert nd.value == pd.value + (2 * 8 * 128 * 2 + 255) // 256 * 256
    assert lib.msa_index_score_fp4_workspace_size(ctypes.byref(_args(**fp4)), 7, ctypes.byref(n)) == 1
    assert lib.msa_index_score_workspace_size(ctypes.byref(_args(**fp4)), ctypes.byref(n)) == 1
    # one side FP4 only, a scale, a stride below a compact FP4 page
    for over in (dict(q_dtype=5, k_dtype=1, page_stride=128 * 64), dict(fp4, scale=16),
                 dict(fp4, page_stride=100)):
        assert lib.msa_index_score_fp4_workspace_size(ctypes.byref(_args(**over)), 0,
                                                      ctypes.byref(n)) == 1


def _sparse(**over):
    import block_score_gb300 as bs
    sa = bs._SparseArgs()
    base = dict(value_cache=16, selection=16, k=16, sm_scale=0.0)
    base.update(over)
    for k, v in base.items():
        setattr(sa, k, v)
    return sa


def test_sparse_attention_host_rules(lib):
    n = ctypes.c_size_t()
    ok = _args()                                           # bf16 query and keys
    assert lib.msa_sparse_attention_workspace_size(ctypes.byref(ok), ctypes.byref(_sparse()),
                                                   ctypes.byref(n)) == 0
    small = n.value
    # the per-entry records (8 bytes) and unit descriptors (16) and the 16-bit
    # partials grow with T * H_kv * k
    big = _args(T=64)
    assert lib.msa_sparse_attention_workspace_size(ctypes.byref(big), ctypes.byref(_sparse()),
                                                   ctypes.byref(n)) == 0
    assert n.value > small
    cases = [
        (ok, dict(k=0), 1), (ok, dict(k=33), 1), (ok, dict(sm_scale=-1.0), 1),
        (ok, dict(value_cache=None), 1), (ok, dict(selection=None), 1),
        (_args(q_dtype=0, k_dtype=0), {}, 0),              # fp16 is fine too
        (_args(q_dtype=3, k_dtype=3), {}, 1),              # FP8: not for the sparse branch
        # a unit descriptor keeps the kv head in 15 bits, an entry record the
        # token in 27
        (_args(H_q=40000, H_kv=40000, page_stride=40000 * 128 * 128), {}, 2),
        (_args(T=1 << 27), {}, 2),
        (_args(T=(1 << 27) - 1), {}, 0),
    ]
    for a, over, status in cases:
        got = lib.msa_sparse_attention_workspace_size(ctypes.byref(a), ctypes.byref(_sparse(**over)),
                                                      ctypes.byref(n))
        assert got == status, (over, got, status)


def test_sparse_attention_binding_checks_the_arrays_it_indexes():
    # a selection, out or lse of another shape would make the kernels read or
    # write out of bounds: the binding refuses them before anything runs
    import block_score_gb300 as bs
    import synth
    case = synth.make_case([3, 2], [300, 40], H_q=4, H_kv=2, layout="BBND",
                           q_dtype=torch.bfloat16, MB=3, seed=1)
    prep = bs.from_case(case, torch.device("cpu"))
    value = torch.zeros_like(prep.call.key)
    good = torch.full((5, 2, 4), -1, dtype=torch.int32)
    for sel in (torch.full((4, 2, 4), -1, dtype=torch.int32),     # fewer tokens
                torch.full((5, 1, 4), -1, dtype=torch.int32),     # fewer groups
                good.to(torch.int64),                             # wrong dtype
                good.transpose(0, 1).contiguous().transpose(0, 1)):   # not contiguous
        with pytest.raises(ValueError, match="selection"):
            prep.sparse_attention(value, sel)
    with pytest.raises(ValueError, match="out"):
        prep.sparse_attention(value, good, out=torch.empty(5, 4, 64))
    with pytest.raises(ValueError, match="lse"):
        prep.sparse_attention(value, good, lse=torch.empty(5, 4, dtype=torch.float64))
    with pytest.raises(ValueError, match="value"):                # a CPU value cache
        prep.sparse_attention(value, good)


def test_binding_refuses_arrays_on_another_device():
    # a pointer of another device (or of host memory) would be dereferenced by
    # the kernels: every array must be on the query's device
    import block_score_gb300 as bs
    q = torch.zeros(4, 2, 128, dtype=torch.float16)
    k = torch.zeros(2, 128, 1, 128, dtype=torch.float16)
    args = dict(layout_key="BBND", actual_seq_qlen=torch.tensor([0, 4], dtype=torch.int32),
                actual_seq_klen=torch.tensor([10], dtype=torch.int32),
                block_table=torch.zeros(1, 1, dtype=torch.int32))
    assert bs.msa_index_score_out_shape(q, k, torch.zeros(1, dtype=torch.int32), **args)
    for name in ("block_table", "actual_seq_klen"):
        bad = dict(args, **{name: args[name].to("meta")})
        with pytest.raises(ValueError, match=name):
            bs.msa_index_score_out_shape(q, k, torch.zeros(1, dtype=torch.int32), **bad)
    with pytest.raises(ValueError, match="key"):
        bs.msa_index_score_out_shape(q, k.to("meta"), torch.zeros(1, dtype=torch.int32), **args)


@pytest.mark.parametrize("T,H_q,H_kv,k", [(32, 8, 1, 16), (1000, 16, 2, 3), (4096, 64, 8, 32)])
def test_workspaces_hold_what_the_kernels_write(lib, T, H_q, H_kv, k):
    # lower bounds from the header's description of each workspace: the sparse
    # branch's partials (T * H_q * k outputs of D 16-bit values and as many fp32
    # log-sum-exps) and the fused selection's partial lists (at least one part
    # per epilogue group: T * H_kv * 2 * k 64-bit keys)
    n = ctypes.c_size_t()
    a = _args(T=T, H_q=H_q, H_kv=H_kv, page_stride=128 * H_kv * 128)
    assert lib.msa_sparse_attention_workspace_size(ctypes.byref(a), ctypes.byref(_sparse(k=k)),
                                                   ctypes.byref(n)) == 0
    assert n.value >= T * H_q * k * (128 * 2 + 4)
    if 32 % (H_q // H_kv) == 0 and k <= 16:
        assert lib.msa_index_score_topk_workspace_size(ctypes.byref(a), k, ctypes.byref(n)) == 0
        assert n.value >= T * H_kv * 2 * k * 8
