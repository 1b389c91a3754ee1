"""Seeded synthetic inputs for the MSA index-branch block-score op.

This module only draws random tensors and lays them out the way a paged
(BBND / BNBD) or packed (TND) key cache stores them.  It holds none of the
operator's arithmetic: no dot products, no masks, no maxima.  Both the CPU
oracle (``oracle/``) and the CUDA path (``block_score_gb300``) take their
inputs from here, so the two sides see identical bytes.

Shapes follow the torch API described on "CANN ops-transformer ...
msa_index_score" (sec. 4, parameter table):

* ``query``        [T, H_q, D]            fp16 / bf16
* ``key`` (BBND)   [NP, P, H_kv, D]       fp16 / bf16 / int8, dim0 may be strided
* ``key`` (BNBD)   [NP, H_kv, P, D]
* ``key`` (TND)    [T2, H_kv, D]          contiguous
* ``block_table``  [B, MB] int32          (paged layouts only; unused entries -1)
* ``cu_seqlens_q`` [B+1] int32
* ``kv_len``       [B] int32 (paged)  /  ``cu_seqlens_k`` [B+1] int32 (TND)
* ``start_loc``    [B] int32               logical block index of the current query
* ``scale``        [NP, H_kv, P] fp32 (paged int8) / [T2, H_kv] fp32 (TND int8)

Every function takes an explicit seed and uses its own ``torch.Generator`` on
the CPU, so a case is reproducible byte for byte on any host.
"""
from __future__ import annotations

import dataclasses
import itertools
import math
from typing import List, Optional, Sequence

import torch

__all__ = [
    "MsaCase", "make_case", "make_fp4_case", "to_fp4", "config", "CONFIG_NAMES", "FILL_KINDS",
]

FILL_KINDS = ("randn", "randn01", "int_small", "int8_full", "onehot_d0",
              "abs_randn", "bytes")


@dataclasses.dataclass
class MsaCase:
    """One self-contained input set (CPU tensors)."""
    name: str
    query: torch.Tensor
    key: torch.Tensor
    block_table: Optional[torch.Tensor]
    cu_seqlens_q: torch.Tensor
    kv_len: Optional[torch.Tensor]
    cu_seqlens_k: Optional[torch.Tensor]
    start_loc: torch.Tensor
    scale: Optional[torch.Tensor]
    layout: str
    sparse_mode: int
    init_blocks: int
    local_blocks: int
    MB: int
    P: int
    # bookkeeping of what was drawn (host ints, for reports and sampling)
    q_lens: List[int] = dataclasses.field(default_factory=list)
    kv_lens: List[int] = dataclasses.field(default_factory=list)
    # FP4 inputs ("mx" / "nv"): query and key hold packed E2M1 codes (two per
    # byte, element 2i in the low nibble), with one scale byte per group
    fp4: Optional[str] = None
    q_scale: Optional[torch.Tensor] = None     # [T, H_q, D/G] uint8
    k_scale: Optional[torch.Tensor] = None     # paged [NP, H_kv, P, D/G]; TND [T2, H_kv, D/G]

    @property
    def T(self) -> int:
        return int(self.query.shape[0])

    @property
    def H_q(self) -> int:
        return int(self.query.shape[1])

    @property
    def D(self) -> int:
        return int(self.query.shape[2]) * (2 if self.fp4 else 1)

    @property
    def H_kv(self) -> int:
        if self.layout == "BBND":
            return int(self.key.shape[2])
        return int(self.key.shape[1])

    @property
    def B(self) -> int:
        return int(self.cu_seqlens_q.shape[0]) - 1

    @property
    def MBp(self) -> int:
        return ((self.MB + 15) // 16) * 16

    @property
    def out_shape(self):
        return (self.H_q, self.T, self.MBp)

    def kv_len_list(self) -> List[int]:
        return list(self.kv_lens)


def _draw(shape, kind: str, dtype: torch.dtype, gen: torch.Generator) -> torch.Tensor:
    """Draw a tensor of the given value distribution, then cast to ``dtype``."""
    if kind == "randn":
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
    elif kind == "randn01":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) * 0.1
    elif kind == "abs_randn":
        x = torch.randn(shape, generator=gen, dtype=torch.float32).abs()
    elif kind == "int_small":
        # integers in [-8, 8]: every product and every 128-term sum is exact in fp32
        x = torch.randint(-8, 9, shape, generator=gen, dtype=torch.int32).to(torch.float32)
    elif kind == "int8_full":
        x = torch.randint(-127, 128, shape, generator=gen, dtype=torch.int32).to(torch.float32)
    elif kind == "onehot_d0":
        x = torch.zeros(shape, dtype=torch.float32)
        x[..., 0] = 1.0
    elif kind == "bytes":
        # every byte pattern equally likely (packed FP4 codes: two per byte)
        return torch.randint(0, 256, shape, generator=gen, dtype=torch.int32).to(torch.uint8)
    else:
        raise ValueError(f"unknown value kind {kind!r}")
    if dtype == torch.int8:
        return x.round().clamp(-127, 127).to(torch.int8)
    return x.to(dtype)


def _cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


def make_case(
    q_lens: Sequence[int],
    kv_lens: Sequence[int],
    *,
    H_q: int,
    H_kv: int,
    D: int = 128,
    P: int = 128,
    layout: str = "BBND",
    q_dtype: torch.dtype = torch.float16,
    k_dtype: Optional[torch.dtype] = None,
    q_kind: str = "randn",
    k_kind: str = "randn",
    MB: Optional[int] = None,
    NP: Optional[int] = None,
    permute_pages: bool = True,
    page_gap: int = 1,
    poison: Optional[float] = None,
    sparse_mode: int = 3,
    init_blocks: int = 0,
    local_blocks: int = 1,
    start_loc: Optional[Sequence[int]] = None,
    scale_range=(1e-3, 2e-2),
    scale_const: Optional[float] = None,
    seed: int = 0,
    name: str = "case",
) -> MsaCase:
    """Build one case.

    ``q_lens`` / ``kv_lens`` give each request's query and visible KV length.
    ``page_gap`` > 1 stores the paged cache with a dim0 stride of ``page_gap``
    compact pages; the gap pages hold ``poison`` (a value no correct read may
    ever see).  ``start_loc`` defaults to the last logical block of each request
    (``max(ceil(kv_len/P) - 1, 0)``).
    """
    layout = layout.upper()
    if layout not in ("BBND", "BNBD", "TND"):
        raise ValueError(f"layout {layout!r}")
    k_dtype = k_dtype or q_dtype
    gen = torch.Generator().manual_seed(int(seed))
    B = len(q_lens)
    assert len(kv_lens) == B
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    nbs = [_cdiv(L, P) for L in kv_lens]
    T = sum(q_lens)
    cu_q = torch.tensor([0] + list(_prefix(q_lens)), dtype=torch.int32)
    query = _draw((T, H_q, D), q_kind, q_dtype, gen)
    if start_loc is None:
        start_loc = [max(nb - 1, 0) for nb in nbs]
    start = torch.tensor(list(start_loc), dtype=torch.int32)

    scale = None
    if layout == "TND":
        T2 = sum(kv_lens)
        key = _draw((T2, H_kv, D), k_kind, k_dtype, gen)
        cu_k = torch.tensor([0] + list(_prefix(kv_lens)), dtype=torch.int32)
        if k_dtype == torch.int8:
            if scale_const is not None:
                scale = torch.full((T2, H_kv), float(scale_const), dtype=torch.float32)
            else:
                scale = torch.empty((T2, H_kv), dtype=torch.float32).uniform_(
                    scale_range[0], scale_range[1], generator=gen)
        mb = MB if MB is not None else max(1, max(nbs) if nbs else 1)
        return MsaCase(name=name, query=query, key=key, block_table=None,
                       cu_seqlens_q=cu_q, kv_len=None, cu_seqlens_k=cu_k,
                       start_loc=start, scale=scale, layout=layout,
                       sparse_mode=sparse_mode, init_blocks=init_blocks,
                       local_blocks=local_blocks, MB=mb, P=P,
                       q_lens=q_lens, kv_lens=kv_lens)

    need = sum(nbs)
    NP = max(NP or 0, need, 1)
    mb = MB if MB is not None else max(1, max(nbs) if nbs else 1)
    if any(nb > mb for nb in nbs):
        raise ValueError("block_table width smaller than a request's block count")
    pages = (torch.randperm(NP, generator=gen) if permute_pages
             else torch.arange(NP)).to(torch.int32)
    table = torch.full((B, mb), -1, dtype=torch.int32)
    off = 0
    for b, nb in enumerate(nbs):
        table[b, :nb] = pages[off:off + nb]
        off += nb
    if layout == "BBND":
        page_shape = (P, H_kv, D)
    else:
        page_shape = (H_kv, P, D)
    store = _draw((NP, page_gap) + page_shape, k_kind, k_dtype, gen)
    if page_gap > 1:
        fill = poison if poison is not None else (127 if k_dtype == torch.int8 else 1.0e4)
        store[:, 1:] = torch.tensor(fill).to(k_dtype)
    key = store[:, 0]            # view: dim0 stride = page_gap compact pages
    if k_dtype == torch.int8:
        if scale_const is not None:
            scale = torch.full((NP, H_kv, P), float(scale_const), dtype=torch.float32)
        else:
            scale = torch.empty((NP, H_kv, P), dtype=torch.float32).uniform_(
                scale_range[0], scale_range[1], generator=gen)
    kv = torch.tensor(kv_lens, dtype=torch.int32)
    return MsaCase(name=name, query=query, key=key, block_table=table,
                   cu_seqlens_q=cu_q, kv_len=kv, cu_seqlens_k=None,
                   start_loc=start, scale=scale, layout=layout,
                   sparse_mode=sparse_mode, init_blocks=init_blocks,
                   local_blocks=local_blocks, MB=mb, P=P,
                   q_lens=q_lens, kv_lens=kv_lens)


def _prefix(xs):
    s = 0
    for x in xs:
        s += x
        yield s


# --------------------------------------------------------------------------
# The five benchmark workloads (seeded recipes; sizes from the op's spec of the
# decode / chunked-prefill / int8 / long-context use cases).
# --------------------------------------------------------------------------

CONFIG_NAMES = {
    1: "tiny_paged_prefill",
    2: "batched_decode_bbnd_bf16",
    3: "varlen_chunked_prefill_bnbd_bf16",
    4: "int8_mixed_decode_prefill",
    5: "long_context_prefill_131k",
}


def _randint(gen, lo, hi):
    """Uniform integer in [lo, hi] inclusive."""
    return int(torch.randint(lo, hi + 1, (1,), generator=gen).item())


def config(n: int, seed: Optional[int] = None, layout: Optional[str] = None,
           q_len: Optional[int] = None) -> MsaCase:
    """Workload ``n`` (1..5) with its default seed ``1234 + n``.

    ``layout`` (optional) stores the same lengths in another key layout
    (BBND, BNBD or packed TND; for TND, MB becomes the longest request's block
    count); the drawn values then differ, the shapes and lengths do not.
    ``q_len`` (workload 5 only) cuts the long prefill to its last ``q_len``
    query positions at the same kv_len (a smaller case of the same kernel, for
    profiler captures).
    """
    seed = 1234 + n if seed is None else seed
    g = torch.Generator().manual_seed(seed)
    name = CONFIG_NAMES[n]
    build = make_case
    if layout is not None:
        lay = layout.upper()

        def build(q, kv, **kw):   # the same builder with the layout replaced
            kw["layout"] = lay
            if lay == "TND":
                kw["MB"] = None
                kw.pop("NP", None)
                kw.pop("permute_pages", None)
            kw["name"] = kw.get("name", name) + "_" + lay.lower()
            return make_case(q, kv, **kw)
    if n == 1:
        # B=1, T=32, H_q=8, H_kv=1, kv_len=256, NP=8 pages, table = arange(2)
        return build([32], [256], H_q=8, H_kv=1, layout="BBND",
                         q_dtype=torch.float16, MB=2, NP=8, permute_pages=False,
                         sparse_mode=3, init_blocks=0, local_blocks=1,
                         start_loc=[1], seed=seed, name=name)
    if n == 2:
        kv = [_randint(g, 1024, 65536) for _ in range(64)]
        return build([1] * 64, kv, H_q=16, H_kv=1, layout="BBND",
                         q_dtype=torch.bfloat16, q_kind="randn01", k_kind="randn01",
                         MB=512, sparse_mode=3, init_blocks=0, local_blocks=1,
                         seed=seed + 1, name=name)
    if n == 3:
        # one request per query length 2048/4096/6144/8192 (T = 20480 + 256)
        reqs = []
        for lq in (2048, 4096, 6144, 8192):
            reqs.append((lq, lq + _randint(g, 0, 8192)))
        reqs.append((0, _randint(g, 1, 8192)))
        reqs.append((256, 0))
        order = torch.randperm(len(reqs), generator=g).tolist()
        reqs = [reqs[i] for i in order]
        return build([r[0] for r in reqs], [r[1] for r in reqs], H_q=32, H_kv=4,
                         layout="BNBD", q_dtype=torch.bfloat16, MB=128,
                         sparse_mode=3, init_blocks=1, local_blocks=4,
                         seed=seed + 1, name=name)
    if n == 4:
        reqs = [(1, _randint(g, 8192, 32768)) for _ in range(24)]
        reqs += [(512, _randint(g, 8192, 32768)) for _ in range(8)]
        order = torch.randperm(len(reqs), generator=g).tolist()
        reqs = [reqs[i] for i in order]
        return build([r[0] for r in reqs], [r[1] for r in reqs], H_q=16, H_kv=2,
                         layout="BBND", q_dtype=torch.float16, k_dtype=torch.int8,
                         k_kind="int8_full", MB=256, sparse_mode=3,
                         init_blocks=0, local_blocks=1, seed=seed + 1, name=name)
    if n == 5:
        return build([16384 if q_len is None else int(q_len)], [131072], H_q=64, H_kv=8,
                         layout="BBND",
                         q_dtype=torch.bfloat16, MB=1100, NP=1024, sparse_mode=3,
                         init_blocks=4, local_blocks=8, start_loc=[1023],
                         seed=seed + 1, name=name)
    raise ValueError(f"no workload {n}")


# scale bytes drawn for FP4 cases: E8M0 codes 2^-6 .. 2^6 (MXFP4) and E4M3
# values 0.25 .. 4.5 (NVFP4, codes 0x28 .. 0x49), per group of 32 / 16 elements
FP4_SCALE_CODES = {"mx": (121, 133), "nv": (0x28, 0x49)}
FP4_GROUP = {"mx": 32, "nv": 16}


def make_fp4_case(q_lens: Sequence[int], kv_lens: Sequence[int], *, fmt: str, H_q: int,
                  H_kv: int, D: int = 128, scale_codes=None, seed: int = 0,
                  name: str = "fp4_case", **kw) -> MsaCase:
    """An FP4 case: uniformly random packed E2M1 codes for the query and the
    key cache (any layout of ``make_case``), random group scale bytes.

    ``fmt`` is "mx" (E8M0 scale per 32 elements) or "nv" (E4M3 scale per 16).
    The key scales are kept in logical page order: paged [NP, H_kv, P, D/G],
    TND [T2, H_kv, D/G]; the query scales are [T, H_q, D/G].  ``scale_codes``
    (lo, hi) overrides the drawn scale byte range (inclusive).
    """
    if fmt not in FP4_GROUP:
        raise ValueError(f"fp4 format {fmt!r}")
    base = make_case(q_lens, kv_lens, H_q=H_q, H_kv=H_kv, D=D // 2, q_dtype=torch.uint8,
                     k_dtype=torch.uint8, q_kind="bytes", k_kind="bytes", seed=seed, name=name,
                     **kw)
    ng = D // FP4_GROUP[fmt]
    lo, hi = scale_codes if scale_codes is not None else FP4_SCALE_CODES[fmt]
    gen = torch.Generator().manual_seed(int(seed) + 7777)

    def codes(shape):
        return torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int32).to(torch.uint8)
    q_scale = codes((base.T, H_q, ng))
    if base.layout == "TND":
        k_scale = codes((int(base.key.shape[0]), H_kv, ng))
    else:
        k_scale = codes((int(base.key.shape[0]), H_kv, base.P, ng))
    return dataclasses.replace(base, fp4=fmt, q_scale=q_scale, k_scale=k_scale)


def to_fp4(case: MsaCase, fmt: str, seed: Optional[int] = None) -> MsaCase:
    """The same workload (lengths, table, layout, page order) with FP4 inputs:
    random packed E2M1 codes in place of the query and key values and random
    group scale bytes (see ``make_fp4_case``).  The key must be compact."""
    if fmt not in FP4_GROUP:
        raise ValueError(f"fp4 format {fmt!r}")
    gen = torch.Generator().manual_seed(4321 if seed is None else int(seed))
    D = case.D
    kshape = tuple(case.key.shape[:-1]) + (D // 2,)
    q = torch.randint(0, 256, (case.T, case.H_q, D // 2), generator=gen, dtype=torch.int32).to(torch.uint8)
    k = torch.randint(0, 256, kshape, generator=gen, dtype=torch.int32).to(torch.uint8)
    ng = D // FP4_GROUP[fmt]
    lo, hi = FP4_SCALE_CODES[fmt]

    def codes(shape):
        return torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int32).to(torch.uint8)
    if case.layout == "TND":
        k_scale = codes((kshape[0], case.H_kv, ng))
    else:
        k_scale = codes((kshape[0], case.H_kv, case.P, ng))
    return dataclasses.replace(case, query=q, key=k, scale=None, fp4=fmt,
                               q_scale=codes((case.T, case.H_q, ng)), k_scale=k_scale,
                               name=f"{case.name}_fp4{fmt}")


def decode_subset(case: MsaCase) -> MsaCase:
    """Requests of ``case`` with a single query token, re-packed as their own batch.

    Used to time the decode part of a mixed batch on its own.  The cache,
    table rows and scale are shared with ``case`` (no data is redrawn).
    """
    keep = [b for b, lq in enumerate(case.q_lens) if lq == 1]
    cu = case.cu_seqlens_q.tolist()
    rows = [cu[b] for b in keep]
    q = case.query[rows].contiguous()
    cu_q = torch.arange(len(keep) + 1, dtype=torch.int32)
    table = case.block_table[keep].contiguous() if case.block_table is not None else None
    kv = case.kv_len[keep].contiguous() if case.kv_len is not None else None
    key, scale, cu_k = case.key, case.scale, None
    if case.layout.upper() == "TND":
        # packed keys: the kept requests' rows, re-packed with their prefix sums
        ck = case.cu_seqlens_k.tolist()
        spans = [(ck[b], ck[b + 1]) for b in keep]
        key = torch.cat([case.key[a:e] for a, e in spans]).contiguous()
        if case.scale is not None:
            scale = torch.cat([case.scale[a:e] for a, e in spans]).contiguous()
        cu_k = torch.tensor([0] + list(itertools.accumulate(e - a for a, e in spans)), dtype=torch.int32)
    return MsaCase(name=case.name + "_decode_subset", query=q, key=key,
                   block_table=table, cu_seqlens_q=cu_q, kv_len=kv,
                   cu_seqlens_k=cu_k, start_loc=case.start_loc[keep].contiguous(),
                   scale=scale, layout=case.layout, sparse_mode=case.sparse_mode,
                   init_blocks=case.init_blocks, local_blocks=case.local_blocks,
                   MB=case.MB, P=case.P, q_lens=[1] * len(keep),
                   kv_lens=[case.kv_lens[b] for b in keep])
