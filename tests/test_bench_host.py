"""Host logic of the benchmark that needs no GPU: the source hash that keeps a
recorded DRAM-traffic figure tied to the code it was measured on."""
import os
import shutil

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
