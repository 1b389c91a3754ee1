"""Host logic of the benchmark that needs no GPU: the source hash that keeps a
recorded DRAM-traffic figure tied to the code it was measured on, the roofline
record (binding roof, peak of the operand type, fractions) and the kernel
launches per call that the bench line claims."""
import os
import shutil

import pytest

import bench


def test_code_only_drops_comments_and_keeps_literals():
    src = ('int a = 1;   // trailing\n'
           '/* block\n   comment */ const char* s = "// in a string /* too */";\n'
           '\n   \n'
           "char q = '\"'; char r = '\\''; // after\n"
           'asm volatile("add.s32 %0, %1, 2;" : "=r"(a) : "r"(a));\n')
    assert bench.code_only(src) == (
        'int a = 1;\n'
        '  const char* s = "// in a string /* too */";\n'
        "char q = '\"'; char r = '\\'';\n"
        'asm volatile("add.s32 %0, %1, 2;" : "=r"(a) : "r"(a));')


def _copy_sources(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "block_score_gb300", "csrc")
    dst = tmp_path / "block_score_gb300" / "csrc"
    dst.mkdir(parents=True)
    for names in bench.KERNEL_SOURCES.values():
        for name in names:
            shutil.copy(os.path.join(src, name), dst / name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return dst


def test_source_hash_ignores_comment_edits_but_not_code_edits(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path, monkeypatch)
    before = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    common = dst / "msa_common.cuh"
    text = common.read_text()
    common.write_text("// a new comment line\n" + text.replace("\n", "  \n", 3) + "\n/* and a block */\n")
    assert {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES} == before
    common.write_text(text + "\nconstexpr int kUnusedForTheTest = 1;\n")
    after = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert all(after[k] != before[k] for k in bench.KERNEL_SOURCES)
    # an edit to a file of one kernel alone leaves the other kernel's hash
    common.write_text(text)
    short = dst / "msa_short.cu"
    short.write_text(short.read_text() + "\nstatic int kUnusedForTheTest = 2;\n")
    assert bench.kernel_source_hash("tile_kernel") == before["tile_kernel"]
    assert bench.kernel_source_hash("short_kernel") != before["short_kernel"]


def test_recorded_traffic_needs_the_current_hash(tmp_path, monkeypatch):
    _copy_sources(tmp_path, monkeypatch)
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.kernel_source_hash("tile_kernel")
    (prof / "kernel_dram_traffic.txt").write_text(
        "# workload kernel bytes hash\n"
        f"cfgA tile_kernel 1000 {h}\n"
        "cfgB tile_kernel 2000 0000000000000000\n")
    assert bench.recorded_traffic("cfgA", "tile_kernel") == 1000.0
    assert bench.recorded_traffic("cfgB", "tile_kernel") is None
    assert bench.recorded_traffic("cfgA", "short_kernel") is None
    assert bench.recorded_traffic("cfgC", "tile_kernel") is None


# ---------------------------------------------------------------- roofline --
PEAKS = {"hbm_gbs": 1000.0, "bf16_tflops": 1.0, "bf16_tflops_sustained": 0.8, "source": "test"}


def _small(q_dtype, k_dtype=None, **kw):
    import torch
    from synth import make_case
    return make_case([3, 1], [40, 20], H_q=4, H_kv=2, P=8, D=16, layout="BBND",
                     q_dtype=q_dtype, k_dtype=k_dtype, MB=6, seed=3, **kw)


def test_roofline_fractions_and_binding_roof():
    import torch
    case = _small(torch.bfloat16)
    # 1.5 ms of HBM time against 2 ms of bf16 tensor time: tensor-bound
    roof = bench.roofline_of(case, {"bytes": 1.5e9, "flops": 2e9}, 4.0, PEAKS, None)
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert abs(roof["achieved"] - 0.5) < 1e-12 and abs(roof["frac"] - 0.5) < 1e-12
    assert abs(roof["frac_of_sustained"] - 0.5 / 0.8) < 1e-12
    assert roof["kernel_us"] == 4000.0 and roof["algorithmic_flops"] == 2e9
    # 2.5 ms of HBM time against 2 ms of tensor time: HBM-bound
    roof = bench.roofline_of(case, {"bytes": 2.5e9, "flops": 2e9}, 5.0, PEAKS, 3e9)
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["traffic"] == 3e9
    assert abs(roof["achieved"] - 500.0) < 1e-9 and abs(roof["frac"] - 0.5) < 1e-12


def test_fp8_is_judged_at_the_fp8_peak():
    import torch
    case = _small(torch.float8_e4m3fn, torch.float8_e4m3fn)
    # 1.5 ms of HBM time, 2 ms at the bf16 peak but 1 ms at the FP8 peak: HBM binds
    roof = bench.roofline_of(case, {"bytes": 1.5e9, "flops": 2e9}, 3.0, PEAKS, None)
    assert roof["bound"] == "hbm"
    roof = bench.roofline_of(case, {"bytes": 0.5e9, "flops": 2e9}, 2.0, PEAKS, None)
    assert roof["bound"] == "tensor" and roof["peak"] == 2.0
    assert abs(roof["frac"] - 0.5) < 1e-12
    assert bench.tensor_peak(case, PEAKS) == 2.0


def test_fp4_and_int8_use_the_16_bit_peak():
    import torch
    from synth import to_fp4
    for case in (to_fp4(_small(torch.bfloat16), "mx"), _small(torch.float16, torch.int8)):
        assert bench.tensor_peak(case, PEAKS) == 1.0
        roof = bench.roofline_of(case, {"bytes": 0.5e9, "flops": 2e9}, 4.0, PEAKS, None)
        assert roof["bound"] == "tensor" and roof["peak"] == 1.0
        assert "frac_of_sustained" in roof


# ------------------------------------------------------- launches per call --
# Kernels one call launches, as the ncu launch lists of the bench commands show
# them (profiles/launch_lists.md; the bench's top-k leg left out):
LAUNCHES = [
    # (workload, decode subset, fp8, fp4, kernels per call)
    (2, False, None, None, 2),       # plan, tile
    (4, False, None, None, 4),       # plan, int8 mirror, tile, short
    (4, True, None, None, 2),        # plan, short (the host bound leaves the tile kernel out)
    (2, False, "e4m3", None, 2),     # plan, tile
    (2, False, None, "nv", 3),       # query dequantisation, plan, short
    (3, False, None, "mx", 5),       # query dequantisation, plan, FP4 mirror, tile, short
]


@pytest.mark.parametrize("n,dsub,fp8,fp4,want", LAUNCHES)
def test_launches_per_call_match_the_launch_lists(n, dsub, fp8, fp4, want):
    import argparse
    args = argparse.Namespace(workload=n, decode_subset=dsub, layout=None, fp8=fp8, fp4=fp4,
                              q_len=None, steps=None)
    case = bench.make_workload(args)
    assert bench.launches_per_call(case) == want
    short = dsub or fp4 == "nv"
    assert bench.dominant_kernel(case) == ("short_kernel" if short else "tile_kernel")
